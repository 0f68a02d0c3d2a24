// Host block pool and iteration-level scheduler (pure C++, no GPU).
//
// The pool is a preallocated set of physical block ids with a free list used
// as a stack ("Project 17: Production Serving: Continuous Batching and
// PagedAttention", Step 4, BlockPool; "Build a pure-Python continuous batching
// LLM serving engine", Step 2).  The scheduler runs one engine step per call:
// running requests first (admission order), then FCFS admission, then the
// token accounting of the iteration with immediate retirement ("Project 17"
// Step 2; "Continuous Batching" §1, §4, §5).  It only builds block tables,
// slot mappings, context lengths and cu_seqlens; the rules are spelled out in
// include/pkv.h next to pkv_sched_step.
#include <algorithm>
#include <chrono>
#include <cstring>
#include <deque>
#include <new>
#include <string>
#include <unordered_map>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "pkv.h"

struct pkv_pool {
    int num_blocks = 0;
    std::vector<int32_t> free_list;   // stack: back() is popped first
    std::vector<uint8_t> is_free;
    int64_t alloc_calls = 0;
    int64_t fail_at = 0;              // absolute alloc call index that fails (0 = none)

    bool init(int n, const int32_t *order) {
        if (n <= 0) return false;
        num_blocks = n;
        free_list.resize(n);
        is_free.assign(n, 0);
        for (int i = 0; i < n; ++i) {
            int32_t b = order ? order[i] : i;
            if (b < 0 || b >= n || is_free[b]) return false;
            free_list[i] = b;
            is_free[b] = 1;
        }
        return true;
    }

    // All-or-nothing pop of n ids, appended to out in pop order.
    bool alloc(int n, std::vector<int32_t> &out) {
        ++alloc_calls;
        if (fail_at != 0 && alloc_calls == fail_at) {
            fail_at = 0;
            return false;
        }
        if (n < 0 || n > (int)free_list.size()) return false;
        for (int i = 0; i < n; ++i) {
            int32_t b = free_list.back();
            free_list.pop_back();
            is_free[b] = 0;
            out.push_back(b);
        }
        return true;
    }

    void release(const std::vector<int32_t> &ids) {
        for (int32_t b : ids) {
            free_list.push_back(b);
            is_free[b] = 1;
        }
    }
};

static pkv_pool *pool_create_impl(int num_blocks, const int32_t *initial_order) {
    pkv_pool *p = new (std::nothrow) pkv_pool();
    if (!p) return nullptr;
    if (!p->init(num_blocks, initial_order)) {
        delete p;
        return nullptr;
    }
    return p;
}

extern "C" void pkv_pool_destroy(pkv_pool *pool) { delete pool; }

static int pool_alloc_impl(pkv_pool *pool, int n, int32_t *out_ids) {
    if (!pool || n < 0 || (n > 0 && !out_ids)) return PKV_ERR_INVALID_ARG;
    std::vector<int32_t> got;
    got.reserve(n);
    if (!pool->alloc(n, got)) return PKV_ERR_OUT_OF_BLOCKS;
    std::copy(got.begin(), got.end(), out_ids);
    return PKV_OK;
}

static int pool_free_impl(pkv_pool *pool, const int32_t *ids, int n) {
    if (!pool || n < 0 || (n > 0 && !ids)) return PKV_ERR_INVALID_ARG;
    std::vector<uint8_t> seen(pool->num_blocks, 0);
    for (int i = 0; i < n; ++i) {
        int32_t b = ids[i];
        if (b < 0 || b >= pool->num_blocks || pool->is_free[b] || seen[b]) return PKV_ERR_INVALID_ARG;
        seen[b] = 1;
    }
    pool->release(std::vector<int32_t>(ids, ids + n));
    return PKV_OK;
}

extern "C" int pkv_pool_free_count(const pkv_pool *pool) {
    return pool ? (int)pool->free_list.size() : PKV_ERR_INVALID_ARG;
}

extern "C" int pkv_pool_free_list(const pkv_pool *pool, int32_t *out) {
    if (!pool || !out) return PKV_ERR_INVALID_ARG;
    std::copy(pool->free_list.begin(), pool->free_list.end(), out);
    return (int)pool->free_list.size();
}

extern "C" int pkv_pool_inject_failure(pkv_pool *pool, int64_t nth) {
    if (!pool || nth < 0) return PKV_ERR_INVALID_ARG;
    pool->fail_at = nth == 0 ? 0 : pool->alloc_calls + nth;
    return PKV_OK;
}

// ------------------------------------------------------------------ scheduler

namespace {

enum State { WAITING = 0, RUNNING = 1, FINISHED = 2 };

struct Request {
    int64_t rid;
    int prompt_len, max_tokens, eos_after;
    int generated = 0;
    int num_computed = 0;     // tokens whose K/V are in the cache
    State state = WAITING;
    std::vector<int32_t> blocks;
    std::vector<int32_t> tokens;   // prompt token ids (empty: no prefix sharing)
    int registered = 0;            // leading prompt pages registered in the prefix cache
    bool reg_stopped = false;      // a page of this prompt is held by another block
    std::vector<int32_t> slots;    // host slots holding its swapped-out blocks, in table order
    int length() const { return prompt_len + generated; }
};

inline int cdiv(int a, int b) { return (a + b - 1) / b; }

}  // namespace

struct pkv_sched {
    pkv_sched_config cfg{};
    pkv_pool pool;
    int max_blocks = 0;
    std::vector<Request> reqs;
    std::unordered_map<int64_t, int> index;
    std::vector<int> free_reqs;        // slots of forgotten requests, reused by add
    std::vector<int> running;          // request indices, admission order
    std::deque<int> waiting;
    pkv_sched_stats stats{};
    // prefix cache: page key -> block, and each block's key (empty: none);
    // reference count of each block = requests whose tables hold it
    std::unordered_map<std::string, int32_t> cache;
    std::vector<std::string> key_of;
    std::vector<int> ref;
    // swap space: free host slots (a stack) and slots freed this step, usable
    // from the next one; the step's copies
    std::vector<int32_t> swap_free, swap_free_next, swap_out_pairs, swap_in_pairs;

    bool caching() const { return cfg.prefix_caching != 0; }

    std::string page_key(int32_t parent, const int32_t *toks) const {
        std::string k(sizeof(int32_t) * (1 + cfg.block_size), '\0');
        std::memcpy(&k[0], &parent, sizeof(int32_t));
        std::memcpy(&k[sizeof(int32_t)], toks, sizeof(int32_t) * cfg.block_size);
        return k;
    }

    // fresh blocks: owned by one request
    bool alloc_blocks(int n, std::vector<int32_t> &got) {
        if (!pool.alloc(n, got)) return false;
        for (int32_t b : got) ref[b] = 1;
        return true;
    }

    // drop one holder of each block, in table order; a block nobody holds
    // goes back to the free list and out of the prefix cache
    void release_blocks(std::vector<int32_t> &blocks) {
        for (int32_t b : blocks) {
            if (--ref[b] > 0) continue;
            pool.release(std::vector<int32_t>(1, b));
            if (!key_of[b].empty()) {
                cache.erase(key_of[b]);
                key_of[b].clear();
            }
        }
        blocks.clear();
    }

    // the registered pages matching the start of r's prompt, at most
    // (prompt_len - 1) / block_size of them
    void prefix_match(const Request &r, std::vector<int32_t> &chain) const {
        chain.clear();
        if (!caching() || r.tokens.empty()) return;
        const int bs = cfg.block_size;
        const int pages = (r.prompt_len - 1) / bs;
        int32_t parent = -1;
        for (int k = 0; k < pages; ++k) {
            auto it = cache.find(page_key(parent, r.tokens.data() + (size_t)k * bs));
            if (it == cache.end()) break;
            chain.push_back(it->second);
            parent = it->second;
        }
    }

    // register r's prompt pages whose K/V are now computed
    void register_pages(Request &r) {
        if (!caching() || r.tokens.empty() || r.reg_stopped) return;
        const int bs = cfg.block_size;
        const int full = std::min(r.num_computed, r.prompt_len) / bs;
        while (r.registered < full) {
            const int k = r.registered;
            const int32_t parent = k == 0 ? -1 : r.blocks[k - 1];
            if (k > 0 && key_of[parent].empty()) {   // its prefix is not the registered one
                r.reg_stopped = true;
                return;
            }
            std::string key = page_key(parent, r.tokens.data() + (size_t)k * bs);
            auto it = cache.find(key);
            if (it == cache.end()) {
                cache.emplace(key, r.blocks[k]);
                key_of[r.blocks[k]] = std::move(key);
            } else if (it->second != r.blocks[k]) {  // another block holds this page
                r.reg_stopped = true;
                return;
            }
            ++r.registered;
        }
    }

    // emitted arrays (valid until the next step)
    std::vector<int64_t> seq_rids, slot_mapping, token_rids, finished_rids;
    std::vector<int32_t> q_lens, context_lens, cu_seqlens, block_tables, token_pos;

    void preempt(int idx) {
        Request &r = reqs[idx];
        const int keep = cdiv(r.num_computed, cfg.block_size);   // blocks holding computed tokens
        if (cfg.preemption == PKV_PREEMPT_SWAP && keep > 0 && keep <= (int)swap_free.size()) {
            // swap: copy the computed blocks to host slots, keep the progress
            for (int k = 0; k < keep; ++k) {
                const int32_t slot = swap_free.back();
                swap_free.pop_back();
                r.slots.push_back(slot);
                swap_out_pairs.push_back(r.blocks[k]);
                swap_out_pairs.push_back(slot);
            }
            stats.swapped_out_blocks += keep;
        } else {
            r.num_computed = 0;
        }
        release_blocks(r.blocks);
        r.registered = 0;
        r.reg_stopped = false;
        r.state = WAITING;
        running.erase(std::find(running.begin(), running.end(), idx));
        waiting.push_front(idx);
        ++stats.preemptions;
    }

    int step(pkv_step_meta *out);
    void emit(const std::vector<std::pair<int, int>> &scheduled, pkv_step_meta *out);
};

void pkv_sched::emit(const std::vector<std::pair<int, int>> &scheduled, pkv_step_meta *out) {
    std::vector<std::pair<int, int>> order;
    order.reserve(scheduled.size());
    for (auto &x : scheduled)
        if (x.second > 1) order.push_back(x);
    int num_prefill = (int)order.size();
    for (auto &x : scheduled)
        if (x.second == 1) order.push_back(x);
    const int S = (int)order.size();
    const int bs = cfg.block_size;
    seq_rids.resize(S);
    q_lens.resize(S);
    context_lens.resize(S);
    cu_seqlens.assign(S + 1, 0);
    block_tables.assign((size_t)S * max_blocks, -1);
    for (int s = 0; s < S; ++s) cu_seqlens[s + 1] = cu_seqlens[s] + order[s].second;
    const int T = cu_seqlens[S];
    slot_mapping.resize(T);
    token_rids.resize(T);
    token_pos.resize(T);
    for (int s = 0; s < S; ++s) {
        const Request &r = reqs[order[s].first];
        const int q = order[s].second;
        seq_rids[s] = r.rid;
        q_lens[s] = q;
        context_lens[s] = r.num_computed + q;
        std::copy(r.blocks.begin(), r.blocks.end(), block_tables.begin() + (size_t)s * max_blocks);
        for (int j = 0; j < q; ++j) {
            const int pos = r.num_computed + j;
            const int t = cu_seqlens[s] + j;
            slot_mapping[t] = (int64_t)r.blocks[pos / bs] * bs + pos % bs;
            token_rids[t] = r.rid;
            token_pos[t] = pos;
        }
    }
    out->num_seqs = S;
    out->num_prefill = num_prefill;
    out->num_tokens = T;
    out->max_blocks = max_blocks;
    out->seq_rids = seq_rids.data();
    out->q_lens = q_lens.data();
    out->context_lens = context_lens.data();
    out->cu_seqlens = cu_seqlens.data();
    out->block_tables = block_tables.data();
    out->slot_mapping = slot_mapping.data();
    out->token_rids = token_rids.data();
    out->token_pos = token_pos.data();
}

int pkv_sched::step(pkv_step_meta *out) {
    const int bs = cfg.block_size;
    // host slots freed by last step's swap-ins can be reused now
    swap_free.insert(swap_free.end(), swap_free_next.begin(), swap_free_next.end());
    swap_free_next.clear();
    swap_out_pairs.clear();
    swap_in_pairs.clear();
    int budget = cfg.max_num_batched_tokens;
    std::vector<std::pair<int, int>> scheduled;
    std::vector<int32_t> got;

    // 1. running requests, admission order
    size_t i = 0;
    while (i < running.size() && budget > 0) {
        const int idx = running[i];
        Request &r = reqs[idx];
        const int q = std::min(std::min(r.length() - r.num_computed, cfg.chunk), budget);
        const int need = cdiv(r.num_computed + q, bs) - (int)r.blocks.size();
        got.clear();
        bool ok = need <= 0 || alloc_blocks(need, got);
        bool self = false;
        while (!ok) {
            const int victim = running.back();
            preempt(victim);
            if (victim == idx) {
                self = true;
                break;
            }
            got.clear();
            ok = alloc_blocks(need, got);
        }
        if (self) continue;   // r was the last running request; the loop ends
        r.blocks.insert(r.blocks.end(), got.begin(), got.end());
        scheduled.emplace_back(idx, q);
        budget -= q;
        ++i;
    }
    // 2. admission, first come first served; under the static policy only
    // when nothing runs, and then a whole batch whatever the token budget
    // (its members' prefill chunks are scheduled as the budget allows)
    const bool is_static = cfg.policy == PKV_SCHED_STATIC;
    const bool may_admit = !is_static || running.empty();
    std::vector<int32_t> chain;
    while (may_admit && !waiting.empty() && (int)running.size() < cfg.max_batch && (is_static || budget > 0)) {
        const int idx = waiting.front();
        Request &r = reqs[idx];
        const bool swapped = !r.slots.empty();
        if (swapped)
            chain.clear();
        else
            prefix_match(r, chain);
        got.clear();
        if (!alloc_blocks(cdiv(r.length(), bs) - (int)chain.size(), got)) break;
        waiting.pop_front();
        for (int32_t b : chain) ++ref[b];
        r.blocks = chain;
        r.blocks.insert(r.blocks.end(), got.begin(), got.end());
        if (swapped) {
            // swap in: the host slots go back to the first blocks; the
            // computed length is the one it had
            for (size_t k = 0; k < r.slots.size(); ++k) {
                swap_in_pairs.push_back(r.slots[k]);
                swap_in_pairs.push_back(r.blocks[k]);
            }
            stats.swapped_in_blocks += (int64_t)r.slots.size();
            swap_free_next.insert(swap_free_next.end(), r.slots.begin(), r.slots.end());
            r.slots.clear();
            r.registered = 0;
        } else {
            r.num_computed = (int)chain.size() * bs;
            r.registered = (int)chain.size();
        }
        r.reg_stopped = false;
        stats.prefix_hit_blocks += (int64_t)chain.size();
        r.state = RUNNING;
        running.push_back(idx);
        ++stats.admitted;
        const int q = std::min(std::min(r.length() - r.num_computed, cfg.chunk), budget);
        if (q > 0) {
            scheduled.emplace_back(idx, q);
            budget -= q;
        }
    }
    stats.sum_running += (int64_t)running.size();
    if (!scheduled.empty()) {
        emit(scheduled, out);
    } else {
        std::memset(out, 0, sizeof(*out));
        out->max_blocks = max_blocks;
    }
    // 3. the iteration ran: account tokens, emit, retire
    finished_rids.clear();
    for (auto &x : scheduled) {
        Request &r = reqs[x.first];
        r.num_computed += x.second;
        stats.tokens += x.second;
        if (x.second > 1) stats.prefill_tokens += x.second;
        register_pages(r);
        if (r.num_computed == r.length()) {
            ++r.generated;
            if (r.generated >= r.eos_after || r.generated >= r.max_tokens ||
                r.length() >= cfg.max_model_len) {
                release_blocks(r.blocks);
                // a finished request keeps only its counters
                std::vector<int32_t>().swap(r.blocks);
                std::vector<int32_t>().swap(r.tokens);
                std::vector<int32_t>().swap(r.slots);
                r.state = FINISHED;
                running.erase(std::find(running.begin(), running.end(), x.first));
                ++stats.finished;
                finished_rids.push_back(r.rid);
            }
        }
    }
    out->num_finished = (int)finished_rids.size();
    out->finished_rids = finished_rids.data();
    out->num_swap_out = (int)swap_out_pairs.size() / 2;
    out->swap_out = swap_out_pairs.data();
    out->num_swap_in = (int)swap_in_pairs.size() / 2;
    out->swap_in = swap_in_pairs.data();
    ++stats.steps;
    return (int)scheduled.size();
}

static pkv_sched *sched_create_impl(const pkv_sched_config *config) {
    if (!config) return nullptr;
    const pkv_sched_config &c = *config;
    if (c.num_blocks <= 0 || c.block_size <= 0 || c.max_batch <= 0 || c.max_num_batched_tokens <= 0 ||
        c.chunk <= 0 || c.max_model_len <= 1 || (c.policy != PKV_SCHED_CONTINUOUS && c.policy != PKV_SCHED_STATIC) ||
        (c.prefix_caching != 0 && c.prefix_caching != 1) ||
        (c.preemption != PKV_PREEMPT_RECOMPUTE && c.preemption != PKV_PREEMPT_SWAP) || c.swap_blocks < 0)
        return nullptr;
    pkv_sched *s = new (std::nothrow) pkv_sched();
    if (!s) return nullptr;
    s->cfg = c;
    s->cfg.initial_order = nullptr;
    if (!s->pool.init(c.num_blocks, c.initial_order)) {
        delete s;
        return nullptr;
    }
    s->max_blocks = cdiv(c.max_model_len, c.block_size);
    s->key_of.assign(c.num_blocks, std::string());
    s->ref.assign(c.num_blocks, 0);
    // host slots popped from the end: slot 0 first
    for (int i = c.swap_blocks - 1; i >= 0; --i) s->swap_free.push_back(i);
    return s;
}

extern "C" void pkv_sched_destroy(pkv_sched *sched) { delete sched; }

static int sched_add_impl(pkv_sched *sched, int64_t rid, int prompt_len, int max_tokens,
                             int eos_after) {
    if (!sched || prompt_len < 1 || prompt_len >= sched->cfg.max_model_len || max_tokens < 1 ||
        eos_after < 1)
        return PKV_ERR_INVALID_ARG;
    if (sched->index.count(rid)) return PKV_ERR_INVALID_ARG;
    Request r;
    r.rid = rid;
    r.prompt_len = prompt_len;
    r.max_tokens = max_tokens;
    r.eos_after = eos_after;
    int idx;
    if (!sched->free_reqs.empty()) {
        idx = sched->free_reqs.back();
        sched->free_reqs.pop_back();
        sched->reqs[idx] = std::move(r);
    } else {
        idx = (int)sched->reqs.size();
        sched->reqs.push_back(std::move(r));
    }
    sched->index[rid] = idx;
    sched->waiting.push_back(idx);
    return PKV_OK;
}

static int sched_forget_impl(pkv_sched *sched, int64_t rid) {
    if (!sched) return PKV_ERR_INVALID_ARG;
    auto it = sched->index.find(rid);
    if (it == sched->index.end() || sched->reqs[it->second].state != FINISHED) return PKV_ERR_INVALID_ARG;
    sched->free_reqs.push_back(it->second);
    sched->index.erase(it);
    return PKV_OK;
}

static int sched_add_tokens_impl(pkv_sched *sched, int64_t rid, const int32_t *tokens, int prompt_len,
                                    int max_tokens, int eos_after) {
    if (!tokens) return PKV_ERR_INVALID_ARG;
    const int rc = sched_add_impl(sched, rid, prompt_len, max_tokens, eos_after);
    if (rc != PKV_OK) return rc;
    sched->reqs[sched->index[rid]].tokens.assign(tokens, tokens + prompt_len);
    return PKV_OK;
}

static int sched_step_impl(pkv_sched *sched, pkv_step_meta *out) {
    if (!sched || !out) return PKV_ERR_INVALID_ARG;
    nvtxRangePushA("pkv_sched_step");
    auto t0 = std::chrono::steady_clock::now();
    int n = sched->step(out);
    auto t1 = std::chrono::steady_clock::now();
    nvtxRangePop();
    sched->stats.host_ms += std::chrono::duration<double, std::milli>(t1 - t0).count();
    return n;
}

extern "C" int pkv_sched_get_stats(const pkv_sched *sched, pkv_sched_stats *out) {
    if (!sched || !out) return PKV_ERR_INVALID_ARG;
    *out = sched->stats;
    out->running = (int)sched->running.size();
    out->waiting = (int)sched->waiting.size();
    out->free_blocks = (int)sched->pool.free_list.size();
    out->cached_blocks = (int)sched->cache.size();
    out->free_swap_slots = (int)(sched->swap_free.size() + sched->swap_free_next.size());
    return PKV_OK;
}

extern "C" int pkv_sched_inject_alloc_failure(pkv_sched *sched, int64_t nth) {
    if (!sched) return PKV_ERR_INVALID_ARG;
    return pkv_pool_inject_failure(&sched->pool, nth);
}

extern "C" int pkv_sched_request_state(const pkv_sched *sched, int64_t rid, int *generated) {
    if (!sched) return PKV_ERR_INVALID_ARG;
    auto it = sched->index.find(rid);
    if (it == sched->index.end()) return -1;
    const Request &r = sched->reqs[it->second];
    if (generated) *generated = r.generated;
    return (int)r.state;
}

// ---------------------------------------------------------- C entry points
// The C ABI never lets a C++ exception out: an allocation failure inside
// returns PKV_ERR_NO_MEMORY (a null handle from the create calls); a
// scheduler that hit one mid-step should be destroyed.

extern "C" pkv_pool *pkv_pool_create(int num_blocks, const int32_t *initial_order) {
    try {
        return pool_create_impl(num_blocks, initial_order);
    } catch (const std::bad_alloc &) {
        return nullptr;
    }
}

extern "C" int pkv_pool_alloc(pkv_pool *pool, int n, int32_t *out_ids) {
    try {
        return pool_alloc_impl(pool, n, out_ids);
    } catch (const std::bad_alloc &) {
        return PKV_ERR_NO_MEMORY;
    }
}

extern "C" int pkv_pool_free(pkv_pool *pool, const int32_t *ids, int n) {
    try {
        return pool_free_impl(pool, ids, n);
    } catch (const std::bad_alloc &) {
        return PKV_ERR_NO_MEMORY;
    }
}

extern "C" pkv_sched *pkv_sched_create(const pkv_sched_config *config) {
    try {
        return sched_create_impl(config);
    } catch (const std::bad_alloc &) {
        return nullptr;
    }
}

extern "C" int pkv_sched_add(pkv_sched *sched, int64_t rid, int prompt_len, int max_tokens, int eos_after) {
    try {
        return sched_add_impl(sched, rid, prompt_len, max_tokens, eos_after);
    } catch (const std::bad_alloc &) {
        return PKV_ERR_NO_MEMORY;
    }
}

extern "C" int pkv_sched_forget(pkv_sched *sched, int64_t rid) {
    try {
        return sched_forget_impl(sched, rid);
    } catch (const std::bad_alloc &) {
        return PKV_ERR_NO_MEMORY;
    }
}

extern "C" int pkv_sched_add_tokens(pkv_sched *sched, int64_t rid, const int32_t *tokens, int prompt_len,
                                    int max_tokens, int eos_after) {
    try {
        return sched_add_tokens_impl(sched, rid, tokens, prompt_len, max_tokens, eos_after);
    } catch (const std::bad_alloc &) {
        return PKV_ERR_NO_MEMORY;
    }
}

extern "C" int pkv_sched_step(pkv_sched *sched, pkv_step_meta *out) {
    try {
        return sched_step_impl(sched, out);
    } catch (const std::bad_alloc &) {
        return PKV_ERR_NO_MEMORY;
    }
}
