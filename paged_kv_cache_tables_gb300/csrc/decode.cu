// K2 + K3: paged decode attention with split KV ranges and a log-sum-exp merge.
//
// What is computed: "Project 17: Production Serving: Continuous Batching and
// PagedAttention", Step 6 "Implement attention over paged storage" -- walk a
// sequence's page table, score every stored key against the query scaled by
// 1/sqrt(head_dim), softmax over the sequence, weighted sum of the stored
// values -- per query head, with query head h reading KV head h / G.
//
// How (GB300):
//  * Work = the flat list of (sequence, KV head, block) triples.  Every warp
//    of a persistent grid (one CTA of 8 warps per SM) starts on an equal
//    contiguous range of it and claims its blocks a few at a time with one
//    atomic add on its range word (begin and end packed in 64 bits).  The SMs
//    of one GPU do not stream at the same rate, so equal ranges finish at
//    different times: a warp that runs out of work steals the far half of the
//    unclaimed blocks of the busiest warp it can see, with one compare-and-
//    swap on the same word, and streams that piece too.  Owner and thief can
//    never both get a block.
//  * A (sequence, KV head) range processed in more than one piece leaves one
//    partial record (m, l, acc) per piece, in records the warp owns, and
//    registers it in the range's slot array (record, first block, block
//    count; pieces past the fourth go on a per-range list instead).  A
//    per-range counter word counts the pieces registered and the blocks
//    finished; the warp that finishes the range's last block notes the range
//    and, after its own work, reads the slots in one round trip and combines
//    the records by log-sum-exp, with the loads of several records in flight
//    together.  The counters and list
//    heads sit in a control region at the front of the workspace that a small
//    kernel zeroes just before every call, so nothing read from the workspace
//    depends on what the memory held before the call.
//  * The kernel checks its own bookkeeping: a merge verifies that its pieces
//    tile the range exactly (no gap, no overlap), and the last CTA to leave
//    compares the blocks consumed by all warps with the planned total; either
//    failure sets PKV_DEV_SPLIT in the status word.
//  * Each warp runs its own ring of STAGES shared-memory slots.  Lane 0 issues
//    2-D TMA loads (128-byte swizzle) of the K and V tiles of a block -- the
//    block id comes from the block table -- and the warp waits on the slot's
//    mbarrier (bounded wait, error bit on timeout).
//  * The GQA group is one MMA row tile: S = Q(16 padded heads x d) . K^T
//    (d x 16 tokens) with mma.m16n8k16 (K fragments by ldmatrix from the
//    swizzled tile), online softmax in fp32 with warp shuffles over the four
//    lanes of a row, then O^T(d x heads) += V^T . P^T (V fragments by
//    ldmatrix.trans).  P is fed to the MMA as a 16-bit pair (rounded value +
//    rounding residual), so the weights keep ~16 significant bits.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdlib>

#include "pkv.h"
#include "pkv_device.cuh"
#include "pkv_host.h"

namespace pkv {

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // a tile that has not landed in 2 s never will
constexpr int kDecodeWarps = 8;
constexpr int kClaimBatch = 4;      // blocks an owner claims per atomic add
constexpr int kStealMin = 10;       // unclaimed blocks a warp must hold to be robbed
// A step too small to give every warp a share uses fewer warps, each with at
// least clamp(ceil(longest range / kMaxPieces), 1, kMinWarpBlocks) blocks:
// short ranges spread over many warps (a small step is bound by latency, not
// bandwidth), while a long range is not cut into more pieces than its merge
// (a chain of dependent loads) is worth.
constexpr int kMaxPieces = 4;
constexpr int kMinWarpBlocks = 20;
// Pieces of a range registered in its slot array; later pieces go on the
// range's list.  A slot is one u64: record (bits 0-23), first block (24-43),
// block count (44-63).  A step of at most kManySlotsRanges ranges -- where
// long contexts are cut into many pieces -- gives each range kSlotsMax slots
// when the workspace holds them (a merge then finds up to 32 pieces with one
// load per lane); larger steps, whose ranges have few pieces, and the
// smallest accepted workspace use kSlots.
constexpr int kSlots = 4;
constexpr int kSlotsMax = 32;
constexpr int64_t kManySlotsRanges = 1024;
// Merges a warp owes, kept in shared memory and run after its work (at most
// this many; more are merged at once)
constexpr int kDefer = 8;
constexpr int kSlotRecBits = 24, kSlotBlkBits = 20;

// Control words, zeroed before every call (u32 each).
enum Ctl : int {
    kCtlReady = 0,      // CTAs that have published their warps' range words
    kCtlDrained = 3,    // 1 once a full scan found no warp worth robbing
    kCtlExited = 4,     // CTAs that have finished
    kCtlConsumed64 = 8, // u64 at words 8-9: blocks streamed by all warps (checked at exit)
    kCtlBytes = 256,
};

__device__ __forceinline__ unsigned long long slot_pack(uint32_t rec1, int j0, int n) {
    return (unsigned long long)rec1 | ((unsigned long long)j0 << kSlotRecBits) |
           ((unsigned long long)n << (kSlotRecBits + kSlotBlkBits));
}

struct DecodeParams {
    void *out;
    const void *q;
    const int32_t *block_tables;
    const int32_t *context_lens;
    // control region (zeroed before the call)
    uint32_t *ctl;                  // [kCtlBytes / 4]
    unsigned long long *seg_cnt;    // [S * Hkv]: (pieces registered << 32) | blocks finished in recorded pieces
    uint32_t *seg_list;             // [S * Hkv]: 1 + the range's last listed record (0: none)
    // written by the call before they are read
    unsigned long long *seg_slots;  // [S * Hkv][n_slots]: the first pieces' slot words
    unsigned long long *ranges;     // [total_warps]: (end << 32) | begin, offsets from the warp's range start
    long long *prefix;              // [S + 1]: blocks before sequence s (written by CTA 0)
    float *part;                    // [total_warps * rec_per_warp][rec_floats] partial records
    int *dev_status;
    int S, max_blocks, num_blocks, Hq, Hkv, G;
    float scale_log2;   // scale * log2(e): scores are kept in base-2 units
    int out_dtype;
    int total_warps;
    int rec_floats;     // m[G], l[G], acc[G][D], padding, then a 16-byte trailer:
                        // next record, first block, block count, unused
    int rec_per_warp;   // records each warp owns (its own range's two, two per steal)
    int steal;          // 0: no work stealing (the split is fixed by the contexts alone)
    int n_slots;        // slots per range: kSlots or kSlotsMax
    // fused append (null: none): row s of k_new / v_new [S][Hkv][D] is the
    // token at position context_lens[s] - 1 of sequence s
    const void *k_new, *v_new;
    void *k_cache, *v_cache;
};

template <int D, int NT>
struct DecodeShape {
    static constexpr int HALVES = D / 64;              // 64-element (128-byte) column halves
    static constexpr int HALF_BYTES = 64 * 16 * 2;     // one 16-row half tile
    static constexpr int TILE_BYTES = HALVES * HALF_BYTES;
    static constexpr int STAGE_BYTES = 2 * TILE_BYTES;  // K + V
    static constexpr int STAGES = D == 128 ? 3 : 6;
    static constexpr int HP = 8 * NT;                   // heads an MMA tile holds
    static constexpr int RING_BYTES = kDecodeWarps * STAGES * STAGE_BYTES;
    // per slot: the new token's K and V rows (fused append) and its block id
    static constexpr int ROW_BYTES = D * 2;
    static constexpr int SIDE_BYTES = 2 * ROW_BYTES + 16;
    static constexpr int SIDE_TOTAL = kDecodeWarps * STAGES * SIDE_BYTES;
    static constexpr int DEFER_BYTES = kDecodeWarps * kDefer * 16;
    static constexpr int SMEM_BYTES = 1024 + RING_BYTES + SIDE_TOTAL + kDecodeWarps * STAGES * 8 + 256 + DEFER_BYTES;
};

__device__ __forceinline__ int blocks_of(const int32_t *context_lens, int s, int max_blocks, int *dev_status,
                                         int *ctx_out) {
    int c = __ldg(context_lens + s);
    if (c < 0) {
        set_status(dev_status, PKV_DEV_BAD_CONTEXT);
        c = 0;
    }
    if (c > max_blocks * 16) {
        set_status(dev_status, PKV_DEV_BAD_CONTEXT);
        c = max_blocks * 16;
    }
    if (ctx_out) *ctx_out = c;
    return (c + 15) >> 4;
}

// Inclusive block-wide scan of v over kDecodeWarps warps; *total gets the sum.
__device__ __forceinline__ int64_t block_scan(int64_t v, int64_t *sh, int64_t *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        int64_t n = __shfl_up_sync(0xffffffffu, v, off);
        if (lane >= off) v += n;
    }
    if (lane == 31) sh[warp] = v;
    __syncthreads();
    int64_t add = 0, tot = 0;
#pragma unroll
    for (int w = 0; w < kDecodeWarps; ++w) {
        int64_t x = sh[w];
        if (w < warp) add += x;
        tot += x;
    }
    __syncthreads();
    *total = tot;
    return v + add;
}

__device__ __forceinline__ int64_t range_lo(int64_t w, int64_t total, int64_t nw) { return w * total / nw; }

// ---- range words: (end << 32) | begin, offsets from the warp's range start.
// The owner claims from the front with atomic adds on begin; a thief takes
// from the back with a compare-and-swap of the whole word.
__device__ __forceinline__ int rw_begin(unsigned long long w) { return (int)(uint32_t)w; }
__device__ __forceinline__ int rw_end(unsigned long long w) { return (int)(uint32_t)(w >> 32); }
__device__ __forceinline__ unsigned long long rw_make(int b, int e) {
    return ((unsigned long long)(uint32_t)e << 32) | (uint32_t)b;
}

__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long *p) {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ uint32_t ld_relaxed_u32(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// The sequence holding flat triple x (the last s with prefix[s] * Hkv <= x,
// which skips empty sequences), by a 32-way search of the prefix array.
__device__ __forceinline__ int locate_seq(const DecodeParams &p, int64_t x, int lane) {
    int lo = 0, hi = p.S;
    while (hi - lo > 1) {
        const int step = (hi - lo + 31) / 32;
        const int c = lo + lane * step;
        const bool le = c < hi && __ldcg(p.prefix + c) * p.Hkv <= x;
        const unsigned m = __ballot_sync(0xffffffffu, le);
        const int k = 31 - __clz(m);
        lo += k * step;
        hi = min(hi, lo + step);
    }
    return lo;
}

// Log-sum-exp combination of the npieces partial records of range (s, h),
// run by the warp that finished the range's last block.  Lane k takes piece
// k: the first n_slots come from the range's slot array (one load each, all at
// once), later ones from its list.  The pieces are taken in the order of
// their first block (not the order they registered), so a given split always
// combines to the same bits, and the sorted pieces must tile blocks [0, c_nb)
// exactly, else PKV_DEV_SPLIT is set.  Lane hh folds the (max, sum) pairs of
// head hh; then every lane accumulates its D/32 output columns of every head,
// the loads of several records in flight together.
template <typename T, int D, int NT, bool kBatch>
__device__ __forceinline__ void merge_range(const DecodeParams &p, int s, int h, int c_nb, int npieces, int lane) {
    constexpr int HP = 8 * NT, PER = D / 32;
    constexpr uint32_t kFull = 0xffffffffu;
    const int G = p.G;
    const int tr = p.rec_floats - 4;   // trailer: next, first block, block count
    const uint32_t seg = (uint32_t)s * (uint32_t)p.Hkv + (uint32_t)h;
    auto rec_of = [&](uint32_t idx1) { return p.part + (size_t)(idx1 - 1) * p.rec_floats; };
    uint32_t mine = 0u;
    int key = INT32_MAX, cnt = 0;
    const int nslot = min(npieces, p.n_slots);
    if (lane < nslot) {
        const unsigned long long e = __ldcg(p.seg_slots + (size_t)seg * p.n_slots + lane);
        mine = (uint32_t)(e & ((1u << kSlotRecBits) - 1u));
        key = (int)((e >> kSlotRecBits) & ((1u << kSlotBlkBits) - 1u));
        cnt = (int)(e >> (kSlotRecBits + kSlotBlkBits));
    }
    int n = nslot;
    uint32_t rest = 0u;   // pieces past the 32nd (not produced by the usual splits) follow in list order
    if (npieces > p.n_slots) {
        uint32_t r = ld_acquire_u32(p.seg_list + seg);
        while (r != 0u && n < 32) {
            if (lane == n) mine = r;
            r = __float_as_uint(__ldcg(rec_of(r) + tr));
            ++n;
        }
        rest = r;
        if (lane >= nslot && lane < n) {
            const float *rec = rec_of(mine);
            key = __float_as_int(__ldcg(rec + tr + 1));
            cnt = __float_as_int(__ldcg(rec + tr + 2));
        }
    }
    // bitonic sort of the 32 (first block, record, count) triples, ascending
#pragma unroll
    for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
        for (int j = k >> 1; j > 0; j >>= 1) {
            const int ok = __shfl_xor_sync(kFull, key, j);
            const uint32_t om = __shfl_xor_sync(kFull, mine, j);
            const int oc = __shfl_xor_sync(kFull, cnt, j);
            const bool up = (lane & k) == 0;
            const bool lower = (lane & j) == 0;
            const bool take = lower == up ? ok < key : ok > key;
            if (take) {
                key = ok;
                mine = om;
                cnt = oc;
            }
        }
    }
    // the pieces must tile [0, c_nb): sorted, each starts where the previous
    // one ended, the first at 0 and the last at the range's end
    const int pkey = __shfl_up_sync(kFull, key, 1), pcnt = __shfl_up_sync(kFull, cnt, 1);
    bool bad = false;
    if (lane < n) {
        bad = cnt <= 0 || (lane == 0 ? key != 0 : (rest == 0u && key != pkey + pcnt));
        if (lane == n - 1 && rest == 0u) bad |= key + cnt != c_nb;
    }
    int counted = cnt;   // with more than 32 pieces only the total is checked
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) counted += __shfl_xor_sync(kFull, counted, o);

    // ---- (max, sum) per head: lane hh < G folds the records in order, the
    // (m, l) loads of eight records in flight at a time
    float M = -INFINITY, L = 0.f;
    for (int k0 = 0; k0 < n; k0 += 8) {
        float mv[8], lv[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const uint32_t r = __shfl_sync(kFull, mine, (k0 + u) & 31);
            mv[u] = -INFINITY;
            lv[u] = 0.f;
            if (k0 + u < n && lane < G) {
                const float *rec = rec_of(r);
                mv[u] = __ldcg(rec + lane);
                lv[u] = __ldcg(rec + G + lane);
            }
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            if (k0 + u < n) {
                const float Mn = fmaxf(M, mv[u]);
                L = L * exp2_approx(M - Mn) + lv[u] * exp2_approx(mv[u] - Mn);
                M = Mn;
            }
        }
    }
    for (uint32_t walk = rest; walk != 0u;) {
        const float *rec = rec_of(walk);
        walk = __float_as_uint(__ldcg(rec + tr));
        counted += __float_as_int(__ldcg(rec + tr + 2));
        if (lane < G) {
            const float mv = __ldcg(rec + lane), lv = __ldcg(rec + G + lane);
            const float Mn = fmaxf(M, mv);
            L = L * exp2_approx(M - Mn) + lv * exp2_approx(mv - Mn);
            M = Mn;
        }
    }
    if (rest != 0u) bad |= counted != c_nb;
    if (__any_sync(kFull, bad) && lane == 0) set_status(p.dev_status, PKV_DEV_SPLIT);
    float Mh[HP], invL[HP], o[HP][PER];
#pragma unroll
    for (int hh = 0; hh < HP; ++hh) {
        Mh[hh] = __shfl_sync(kFull, M, hh);
        invL[hh] = 1.f / __shfl_sync(kFull, L, hh);
#pragma unroll
        for (int k = 0; k < PER; ++k) o[hh][k] = 0.f;
    }
    // ---- accumulators, a record at a time (its G x D/32 loads per lane in
    // flight together)
    auto add_record = [&](const float *rec) {
#pragma unroll
        for (int hh = 0; hh < HP; ++hh) {
            if (hh < G) {
                const float f = exp2_approx(__ldcg(rec + hh) - Mh[hh]) * invL[hh];
                const float *racc = rec + 2 * G + hh * D;
#pragma unroll
                for (int k2 = 0; k2 < PER; ++k2) o[hh][k2] += f * __ldcg(racc + lane + 32 * k2);
            }
        }
    };
    if constexpr (kBatch) {
        // two records' loads in flight together (outside the streaming loop
        // there are registers to spare)
        for (int k0 = 0; k0 < n; k0 += 2) {
            const bool two = k0 + 1 < n;
            const float *rec0 = rec_of(__shfl_sync(kFull, mine, k0 & 31));
            const float *rec1 = two ? rec_of(__shfl_sync(kFull, mine, (k0 + 1) & 31)) : rec0;
            float a0[HP][PER], a1[HP][PER], f0[HP], f1[HP];
#pragma unroll
            for (int hh = 0; hh < HP; ++hh) {
                if (hh < G) {
                    f0[hh] = __ldcg(rec0 + hh);
                    f1[hh] = __ldcg(rec1 + hh);
#pragma unroll
                    for (int k2 = 0; k2 < PER; ++k2) {
                        a0[hh][k2] = __ldcg(rec0 + 2 * G + hh * D + lane + 32 * k2);
                        a1[hh][k2] = __ldcg(rec1 + 2 * G + hh * D + lane + 32 * k2);
                    }
                }
            }
#pragma unroll
            for (int hh = 0; hh < HP; ++hh) {
                if (hh < G) {
                    const float g0 = exp2_approx(f0[hh] - Mh[hh]) * invL[hh];
                    const float g1 = two ? exp2_approx(f1[hh] - Mh[hh]) * invL[hh] : 0.f;
#pragma unroll
                    for (int k2 = 0; k2 < PER; ++k2) o[hh][k2] += g0 * a0[hh][k2] + g1 * a1[hh][k2];
                }
            }
        }
    } else {
        for (int k = 0; k < n; ++k) add_record(rec_of(__shfl_sync(kFull, mine, k)));
    }
    for (uint32_t walk = rest; walk != 0u;) {
        const float *rec = rec_of(walk);
        walk = __float_as_uint(__ldcg(rec + tr));
        add_record(rec);
    }
#pragma unroll
    for (int hh = 0; hh < HP; ++hh) {
        if (hh < G) {
            const int64_t ob = ((int64_t)s * p.Hq + (int64_t)h * G + hh) * D;
#pragma unroll
            for (int k = 0; k < PER; ++k) store_out<T>(p.out, p.out_dtype, ob + lane + 32 * k, o[hh][k]);
        }
    }
}

// PAIR (head_dim 64 only): one unit of work is a block of two adjacent KV
// heads, whose tiles lie next to each other in the cache (4 KB of K and 4 KB
// of V instead of 2 KB each), held in the registers and ring of the
// head_dim-128 form: the first KV head's 64 dimensions in the first 64-column
// half, the second's in the other.  p.Hkv and p.G then count KV-head pairs
// and the 2G query heads of a pair; the query rows of the first head are zero
// against the second half of K and the other way round, so the product S
// holds each head's own scores, and of O^T += V^T P^T a row only uses the
// half of its own KV head.  D is the register width (128), DO the head_dim.
template <typename T, int D, int NT, bool PAIR>
__global__ void __launch_bounds__(kDecodeWarps * 32, 1)
    paged_decode_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap tk,
                        const __grid_constant__ CUtensorMap tv) {
    static_assert(!PAIR || (D == 128 && NT == 1), "paired heads use the 128-wide single-tile form");
    using Sh = DecodeShape<D, NT>;
    constexpr int DO = PAIR ? 64 : D;   // head_dim of q, out, the caches' rows and the records
    constexpr int STAGES = Sh::STAGES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *ring = smem;
    uint8_t *side = smem + Sh::RING_BYTES;
    uint64_t *bars = reinterpret_cast<uint64_t *>(side + Sh::SIDE_TOTAL);
    int64_t *sh_scan = reinterpret_cast<int64_t *>(bars + kDecodeWarps * STAGES);
    int *plan_s = reinterpret_cast<int *>(sh_scan + kDecodeWarps);   // segment holding each warp's first block
    int *plan_off = plan_s + kDecodeWarps;
    int *sh_max = plan_off + kDecodeWarps;                           // per-warp longest sequence, in blocks
    int4 *defer = reinterpret_cast<int4 *>(reinterpret_cast<uint8_t *>(sh_scan) + 256);   // merges owed, per warp

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int Hkv = p.Hkv, G = p.G;
    // query row r of a unit is a real head, and (paired) register group x
    // (an mt or kk index) belongs to r's own KV head
    auto own_half = [&](int r, int x) { return r < G && (!PAIR || ((2 * r >= G) == (x >= D / 32))); };

    // The kernel may start while the clear of the control region still
    // waits for the kernel before it on the stream (which may be the last
    // call, still using this workspace).  A one-pass plan (a sequence per
    // thread) reads only context_lens and writes only shared memory before
    // it waits; a longer plan waits first, since it writes the prefix array
    // as it goes.
    pdl_launch_dependents();
    const bool one_pass = p.S <= (int)blockDim.x;
    if (!one_pass) pdl_wait_primary();

    // ---- plan: total blocks, this CTA's warp starts; CTA 0 publishes the
    // per-sequence block offsets that thieves search ----
    int64_t local = 0;
    int local_max = 0;
    if (tid < kDecodeWarps) plan_s[tid] = -1;   // (the scan's barriers order this before the plan)
    for (int s = tid; s < p.S; s += blockDim.x) {
        // (a bad context is reported after the wait when the plan runs before it)
        const int nb = blocks_of(p.context_lens, s, p.max_blocks, one_pass ? nullptr : p.dev_status, nullptr);
        local += nb;
        local_max = max(local_max, nb);
    }
    local_max = __reduce_max_sync(0xffffffffu, local_max);
    if (lane == 0) sh_max[warp] = local_max;
    int64_t total_nblk;
    const int64_t incl0 = block_scan(local, sh_scan, &total_nblk);
    const int64_t total = total_nblk * Hkv;
    // warps that get a share: all of them, unless the step is too small to
    // give each at least min_blocks blocks (the scan's barriers published sh_max)
    int max_nb = 0;
#pragma unroll
    for (int w = 0; w < kDecodeWarps; ++w) max_nb = max(max_nb, sh_max[w]);
    const int64_t min_blocks = min(kMinWarpBlocks, max(1, (max_nb + kMaxPieces - 1) / kMaxPieces));
    int64_t nw = (total + min_blocks - 1) / min_blocks;
    if (nw > p.total_warps) nw = p.total_warps;
    if (nw < 1) nw = 1;
    // sequence s holds flat triples [excl * Hkv, (excl + nb) * Hkv): note it as
    // the start of this CTA's warps whose first triple falls there
    auto place = [&](int s, int nb, int64_t excl) {
        if (blockIdx.x == 0 && s < p.S && !one_pass) p.prefix[s] = excl;
        if (nb > 0) {
#pragma unroll
            for (int w = 0; w < kDecodeWarps; ++w) {
                const int64_t ww = (int64_t)blockIdx.x * kDecodeWarps + w;
                const int64_t lo = range_lo(ww, total, nw);
                if (ww < nw && lo >= excl * Hkv && lo < (excl + nb) * Hkv) {
                    plan_s[w] = s;
                    plan_off[w] = (int)(lo - excl * Hkv);
                }
            }
        }
    };
    if (p.S <= (int)blockDim.x) {
        // one sequence per thread: the first scan already gave its offset
        if (tid < p.S) place(tid, (int)local, incl0 - local);
    } else {
        int64_t carry = 0;
        for (int base = 0; base < p.S; base += blockDim.x) {
            const int s = base + tid;
            const int nb = s < p.S ? blocks_of(p.context_lens, s, p.max_blocks, nullptr, nullptr) : 0;
            int64_t tile_total;
            const int64_t excl = carry + block_scan(nb, sh_scan, &tile_total) - nb;
            place(s, nb, excl);
            carry += tile_total;
        }
    }
    if (one_pass) {
        pdl_wait_primary();
        if (blockIdx.x == 0 && tid < p.S) {
            p.prefix[tid] = incl0 - local;
            blocks_of(p.context_lens, tid, p.max_blocks, p.dev_status, nullptr);
        }
    }
    if (blockIdx.x == 0 && tid == 0) p.prefix[p.S] = total_nblk;

    // sequences with an empty context get all-zero rows
    for (int s = blockIdx.x; s < p.S; s += gridDim.x) {
        if (blocks_of(p.context_lens, s, p.max_blocks, nullptr, nullptr) != 0) continue;
        for (int e = tid; e < p.Hq * DO; e += blockDim.x) store_out<T>(p.out, p.out_dtype, (int64_t)s * p.Hq * DO + e, 0.f);
    }

    // every warp publishes its range word; the CTA then counts itself ready
    // (thieves rob no warp before every CTA has published)
    const int64_t wg = (int64_t)blockIdx.x * kDecodeWarps + warp;
    const int64_t lo_w = wg < nw ? range_lo(wg, total, nw) : total;
    const int n_own = wg < nw ? (int)(range_lo(wg + 1, total, nw) - lo_w) : 0;
    if (lane == 0) p.ranges[wg] = rw_make(0, n_own);
    // publish: the barrier orders every thread's range word and prefix
    // stores before thread 0's fence, which makes them visible at GPU scope
    // before the ready count moves (only thread 0 waits for it)
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        atomicAdd(p.ctl + kCtlReady, 1u);
    }

    // ---- this warp's ring ----
    uint8_t *wring = ring + warp * STAGES * Sh::STAGE_BYTES;
    uint8_t *wside = side + warp * STAGES * Sh::SIDE_BYTES;
    uint64_t *wbar = bars + warp * STAGES;
    const bool fuse_append = p.k_new != nullptr;
    if (lane == 0) {
        for (int st = 0; st < STAGES; ++st) mbar_init(&wbar[st], 1);
        fence_mbar_init();
        if (warp == 0) {
            prefetch_tensormap(&tk);
            prefetch_tensormap(&tv);
        }
    }
    __syncwarp();
    const uint64_t policy = l2_policy_evict_first();

    const int g = lane >> 2, t4 = lane & 3;
    const int mi = lane >> 3;
    const int ld_row = ((mi >> 1) << 3) + (lane & 7);          // token row this lane addresses
    const int ld_sw = ld_row & 7;                               // 128-byte swizzle phase of that row
    const uint32_t ring_addr = smem_addr(wring);

    uint32_t slot_base = 0;     // ring slots used by earlier pieces of work (phases continue)
    bool seen_ready = false;    // every CTA has published its range words
    int rec_used = 0;           // records of this warp's own set taken so far
    uint32_t warp_blocks = 0;   // blocks this warp has streamed (checked against the plan at exit)
    int4 *wdefer = defer + warp * kDefer;
    int n_defer = 0;            // merges this warp owes (run after its work)

    // Work: first the warp's own range (claimed in batches), then stolen pieces.
    int64_t x0 = lo_w;          // flat start of the current work
    int len = n_own;            // its length in blocks
    bool own = true;
    int s0 = plan_s[warp], off0 = plan_off[warp];
    for (;;) {
        if (len > 0 && s0 >= 0) {
            // ---------------- stream [x0, x0 + len) ----------------
            auto next_seq = [&](int s, int &nb_out, int *ctx_out) {
                int nb;
                do {
                    ++s;
                    nb = blocks_of(p.context_lens, s, p.max_blocks, nullptr, ctx_out);
                } while (nb == 0);
                nb_out = nb;
                return s;
            };
            int cs = s0, c_ctx, c_nb, ch, cj;
            c_nb = blocks_of(p.context_lens, cs, p.max_blocks, nullptr, &c_ctx);
            ch = off0 / c_nb;
            cj = off0 % c_nb;
            int ps = cs, p_nb = c_nb, ph = ch, pj = cj;
            auto table_entry = [&]() { return __ldg(p.block_tables + (int64_t)ps * p.max_blocks + pj); };
            auto advance_producer = [&]() {
                if (++pj == p_nb) {
                    pj = 0;
                    if (++ph == Hkv) {
                        ph = 0;
                        ps = next_seq(ps, p_nb, nullptr);
                    }
                }
            };
            auto issue = [&](uint32_t slot, int blk) {
                if (lane == 0) {
                    // cache row of the tile (its first KV head's, when paired);
                    // past the end for a bad block id: the load fills zeros
                    const bool bad_blk = blk < 0 || blk >= p.num_blocks;
                    if (bad_blk) set_status(p.dev_status, PKV_DEV_BAD_BLOCK_ID);
                    const int row = ((bad_blk ? p.num_blocks : blk) * Hkv + (bad_blk ? 0 : ph)) * 16 * (PAIR ? 2 : 1);
                    const int stage = (int)(slot % STAGES);
                    uint64_t *bar = &wbar[stage];
                    // the last block of a range also brings the range's new
                    // token (fused append), with the block id it goes to
                    const bool with_row = fuse_append && pj == p_nb - 1;
                    mbar_arrive_expect_tx(bar, Sh::STAGE_BYTES + (with_row ? 2 * Sh::ROW_BYTES : 0));
                    uint8_t *kdst = wring + stage * Sh::STAGE_BYTES;
                    uint8_t *vdst = kdst + Sh::TILE_BYTES;
#pragma unroll
                    for (int hf = 0; hf < Sh::HALVES; ++hf) {
                        // a half is 64 columns of the tile, or (paired) the next KV head's 16 rows
                        const int x = PAIR ? 0 : hf * 64, y = PAIR ? row + 16 * hf : row;
                        tma_load_2d(kdst + hf * Sh::HALF_BYTES, &tk, x, y, bar, policy);
                        tma_load_2d(vdst + hf * Sh::HALF_BYTES, &tv, x, y, bar, policy);
                    }
                    if (with_row) {
                        uint8_t *sd = wside + stage * Sh::SIDE_BYTES;
                        const size_t src = ((size_t)ps * Hkv + ph) * Sh::ROW_BYTES;
                        bulk_load(sd, static_cast<const uint8_t *>(p.k_new) + src, Sh::ROW_BYTES, bar);
                        bulk_load(sd + Sh::ROW_BYTES, static_cast<const uint8_t *>(p.v_new) + src, Sh::ROW_BYTES,
                                  bar);
                        *reinterpret_cast<int *>(sd + 2 * Sh::ROW_BYTES) = blk;
                    }
                }
            };
            auto wait_slot = [&](uint32_t slot, uint64_t limit) {
                return mbar_wait(&wbar[slot % STAGES], (slot / STAGES) & 1u, limit);
            };

            // claims: blocks [0, limit) are this warp's; an own range asks for
            // kClaimBatch more with one atomic add, a batch ahead of use
            int limit = own ? 0 : len;
            bool more = own;
            unsigned long long claim = 0;
            if (own && lane == 0) claim = atomicAdd(p.ranges + wg, (unsigned long long)kClaimBatch);

            // prologue: fill the ring (loads run ahead of the claims; a load
            // of a block that turns out not to be ours is only waited out)
            int issued = 0;
            const int pro = len < STAGES ? len : STAGES;
            // the ring's first table entries are read by lanes 0..pro-1 at
            // once (lane l walks a copy of the cursor l blocks ahead), not one
            // dependent load after another
            int first_entries = 0;
            if (lane < pro) {
                int ls = ps, lnb = p_nb, lh = ph, lj = pj;
                for (int k = 0; k < lane; ++k) {
                    if (++lj == lnb) {
                        lj = 0;
                        if (++lh == Hkv) {
                            lh = 0;
                            ls = next_seq(ls, lnb, nullptr);
                        }
                    }
                }
                first_entries = __ldg(p.block_tables + (int64_t)ls * p.max_blocks + lj);
            }
            int pending = 0;
            for (; issued < pro; ++issued) {
                issue(slot_base + issued, __shfl_sync(0xffffffffu, first_entries, issued));
                if (issued + 1 < len) advance_producer();
            }
            if (issued < len) pending = table_entry();

            uint32_t qa[D / 16][4];
            float acc[D / 16][NT][4];
            float m_run[NT], l_run[NT];
            bool seg_fresh = true;
            int piece_j0 = cj, piece_n = 0;
            // a piece sure to leave a record (it starts inside its range, or
            // the work ends before the range does) takes its number within
            // the range when it starts, so the round trip overlaps its blocks
            bool early_no = false;
            unsigned long long early_word = 0;   // lane 0: the counter word before this piece's number

            // closes the piece of (cs, ch) that ends with block cj of this warp
            auto finish_piece = [&]() {
                warp_blocks += (uint32_t)piece_n;
                float lsum[NT];
#pragma unroll
                for (int pn = 0; pn < NT; ++pn) {
                    lsum[pn] = l_run[pn];
                    lsum[pn] += __shfl_xor_sync(0xffffffffu, lsum[pn], 1);
                    lsum[pn] += __shfl_xor_sync(0xffffffffu, lsum[pn], 2);
                }
                const int head0 = ch * G;
                if (piece_j0 == 0 && cj == c_nb - 1) {
                    // the whole range in this piece: normalise and store
#pragma unroll
                    for (int pn = 0; pn < NT; ++pn) {
                        const float inv_lo = 1.f / __shfl_sync(0xffffffffu, lsum[pn], 8 * t4);
                        const float inv_hi = 1.f / __shfl_sync(0xffffffffu, lsum[pn], 8 * t4 + 4);
                        const int ha = pn * 8 + 2 * t4, hb = ha + 1;
#pragma unroll
                        for (int mt = 0; mt < D / 16; ++mt) {
                            const int d0 = (PAIR ? (mt & 3) : mt) * 16 + g;
                            if (own_half(ha, mt)) {
                                const int64_t o = ((int64_t)cs * p.Hq + head0 + ha) * DO;
                                store_out<T>(p.out, p.out_dtype, o + d0, acc[mt][pn][0] * inv_lo);
                                store_out<T>(p.out, p.out_dtype, o + d0 + 8, acc[mt][pn][2] * inv_lo);
                            }
                            if (own_half(hb, mt)) {
                                const int64_t o = ((int64_t)cs * p.Hq + head0 + hb) * DO;
                                store_out<T>(p.out, p.out_dtype, o + d0, acc[mt][pn][1] * inv_hi);
                                store_out<T>(p.out, p.out_dtype, o + d0 + 8, acc[mt][pn][3] * inv_hi);
                            }
                        }
                    }
                    return;
                }
                // one piece of a range: leave (m, l, acc) in a record of
                // this warp's own set, register it, count its blocks
                const uint32_t seg = (uint32_t)cs * (uint32_t)Hkv + (uint32_t)ch;
                if (rec_used >= p.rec_per_warp) {
                    // cannot happen: a warp steals only while two records are left
                    if (lane == 0) set_status(p.dev_status, PKV_DEV_SPLIT);
                    return;
                }
                const uint32_t ri = (uint32_t)(wg * p.rec_per_warp + rec_used) + 1u;
                ++rec_used;
                // the piece's number within the range: taken when the piece
                // started, or now (a round trip that overlaps the record
                // stores below)
                unsigned long long before = early_word;
                if (!early_no && lane == 0) before = atomicAdd(p.seg_cnt + seg, 1ull << 32);
                float *rec = p.part + (size_t)(ri - 1) * p.rec_floats;
#pragma unroll
                for (int pn = 0; pn < NT; ++pn) {
                    const int hr = pn * 8 + g;
                    if (t4 == 0 && hr < G) {
                        rec[hr] = m_run[pn];
                        rec[G + hr] = lsum[pn];
                    }
                    float *racc = rec + 2 * G;
                    const int ha = pn * 8 + 2 * t4, hb = ha + 1;
#pragma unroll
                    for (int mt = 0; mt < D / 16; ++mt) {
                        const int d0 = (PAIR ? (mt & 3) : mt) * 16 + g;
                        if (own_half(ha, mt)) {
                            racc[ha * DO + d0] = acc[mt][pn][0];
                            racc[ha * DO + d0 + 8] = acc[mt][pn][2];
                        }
                        if (own_half(hb, mt)) {
                            racc[hb * DO + d0] = acc[mt][pn][1];
                            racc[hb * DO + d0 + 8] = acc[mt][pn][3];
                        }
                    }
                }
                if (lane == 0) {
                    float *trailer = rec + p.rec_floats - 4;
                    trailer[1] = __int_as_float(piece_j0);
                    trailer[2] = __int_as_float(piece_n);
                    const int k = (int)(before >> 32);
                    if (k < p.n_slots) {
                        p.seg_slots[(size_t)seg * p.n_slots + k] = slot_pack(ri, piece_j0, piece_n);
                    } else {
                        // past the slots: on the range's list
                        trailer[0] = __uint_as_float(atomicExch(p.seg_list + seg, ri));
                    }
                }
                // publish: every lane's stores, then lane 0 adds the piece's
                // blocks to the range's count (a release; the warp that
                // completes the count acquires)
                __threadfence();
                __syncwarp();
                unsigned long long after = 0;
                if (lane == 0) {
                    after = atomicAdd(p.seg_cnt + seg, (unsigned long long)piece_n) + (unsigned long long)piece_n;
                    __threadfence();
                    // a count past the range's blocks means a block was
                    // streamed twice (a merge may already have run short)
                    if ((uint32_t)after > (uint32_t)c_nb) set_status(p.dev_status, PKV_DEV_SPLIT);
                }
                after = __shfl_sync(0xffffffffu, after, 0);
                if ((uint32_t)after == (uint32_t)c_nb) {
                    // this piece completed the range: merge it after the
                    // warp's work, so the warp keeps streaming now (groups of
                    // more than 8 heads, or a full list, merge at once)
                    if (NT == 1 && n_defer < kDefer) {
                        if (lane == 0) wdefer[n_defer] = make_int4(cs, ch, c_nb, (int)(after >> 32));
                        ++n_defer;
                    } else {
                        __syncwarp();
                        merge_range<T, DO, NT, false>(p, cs, ch, c_nb, (int)(after >> 32), lane);
                    }
                }
            };

            bool timed_out = false;
            int i = 0;
            for (; i < len; ++i) {
                if (i == limit) {
                    if (!more) break;
                    // the batch claimed a batch ago: [b, min(b + batch, e)) is ours
                    const unsigned long long c = __shfl_sync(0xffffffffu, claim, 0);
                    const int b = rw_begin(c), e = rw_end(c);
                    const int got = max(0, min(kClaimBatch, e - b));
                    limit += got;
                    more = got == kClaimBatch && b + kClaimBatch < e;
                    if (more && lane == 0) claim = atomicAdd(p.ranges + wg, (unsigned long long)kClaimBatch);
                    if (got == 0) break;
                }
                if (seg_fresh) {
                    // query fragments of (cs, ch): rows = heads of the group (padded to 16)
                    const uint32_t *qbase = reinterpret_cast<const uint32_t *>(
                        static_cast<const T *>(p.q) + ((int64_t)cs * p.Hq + (int64_t)ch * G) * DO);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        // paired: a query row meets only its own KV head's half of K
                        const int c0 = ((PAIR ? (kk & 3) : kk) * 16 + 2 * t4) >> 1;
                        const bool use = own_half(g, kk);
                        qa[kk][0] = use ? __ldg(qbase + g * (DO / 2) + c0) : 0u;
                        qa[kk][2] = use ? __ldg(qbase + g * (DO / 2) + c0 + 4) : 0u;
                        if constexpr (NT == 1) {   // group of at most 8 heads: rows 8..15 are padding
                            qa[kk][1] = 0u;
                            qa[kk][3] = 0u;
                        } else {
                            qa[kk][1] = g + 8 < G ? __ldg(qbase + (g + 8) * (DO / 2) + c0) : 0u;
                            qa[kk][3] = g + 8 < G ? __ldg(qbase + (g + 8) * (DO / 2) + c0 + 4) : 0u;
                        }
                    }
#pragma unroll
                    for (int mt = 0; mt < D / 16; ++mt)
#pragma unroll
                        for (int pn = 0; pn < NT; ++pn)
#pragma unroll
                            for (int e = 0; e < 4; ++e) acc[mt][pn][e] = 0.f;
#pragma unroll
                    for (int pn = 0; pn < NT; ++pn) {
                        m_run[pn] = -INFINITY;
                        l_run[pn] = 0.f;
                    }
                    seg_fresh = false;
                    piece_j0 = cj;
                    piece_n = 0;
                    early_no = cj > 0 || len - i < c_nb - cj;
                    if (early_no && lane == 0)
                        early_word = atomicAdd(p.seg_cnt + (size_t)cs * Hkv + ch, 1ull << 32);
                }

                const uint32_t slot = slot_base + i;
                if (!__all_sync(0xffffffffu, wait_slot(slot, kWaitLimitNs))) {
                    timed_out = true;
                    break;
                }
                const uint32_t kbase = ring_addr + (slot % STAGES) * Sh::STAGE_BYTES;
                const uint32_t vbase = kbase + Sh::TILE_BYTES;
                if (fuse_append && cj == c_nb - 1) {
                    // fused append: the new token's rows replace row (ctx-1)%16
                    // of the tiles (which held the cache's old bytes) and go to
                    // the cache; one lane per 16-byte chunk of the K and V rows
                    constexpr int CH = D / 8;   // chunks per row
                    const uint8_t *sd = wside + (slot % STAGES) * Sh::SIDE_BYTES;
                    const int r = (c_ctx - 1) & 15;
                    if (lane < 2 * CH) {
                        const int which = lane / CH, c = lane % CH;
                        const uint4 val = *reinterpret_cast<const uint4 *>(sd + which * Sh::ROW_BYTES + c * 16);
                        const uint32_t dst = (which ? vbase : kbase) + (c >> 3) * Sh::HALF_BYTES + r * 128 +
                                             (((c & 7) ^ (r & 7)) << 4);
                        st_shared_v4(dst, val);
                        const int blk = *reinterpret_cast<const int *>(sd + 2 * Sh::ROW_BYTES);
                        if (blk >= 0 && blk < p.num_blocks) {
                            uint8_t *cache = static_cast<uint8_t *>(which ? p.v_cache : p.k_cache);
                            // paired: chunks 0-7 are the first KV head's row, 8-15 the second's
                            const size_t crow = PAIR ? ((size_t)blk * 2 * Hkv + 2 * ch + (c >> 3)) * 16 + r
                                                     : ((size_t)blk * Hkv + ch) * 16 + r;
                            const int ccol = PAIR ? (c & 7) : c;
                            *reinterpret_cast<uint4 *>(cache + crow * (DO * 2) + ccol * 16) = val;
                        }
                    }
                    __syncwarp();
                }

                // ---- pull the block's K and V fragments into registers, then
                // hand the slot straight back to the TMA engine ----
                uint32_t kf[D / 16][4], vf[D / 16][4];
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const int chunk = ((kk & 3) << 1) + (mi & 1);
                    const uint32_t off = (kk >> 2) * Sh::HALF_BYTES + ld_row * 128 + ((chunk ^ ld_sw) << 4);
                    ldsm_x4(kbase + off, kf[kk][0], kf[kk][1], kf[kk][2], kf[kk][3]);
                    ldsm_x4_t(vbase + off, vf[kk][0], vf[kk][1], vf[kk][2], vf[kk][3]);
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (issued < len) {
                    issue(slot_base + issued, pending);
                    if (issued + 1 < len) {
                        advance_producer();
                        pending = table_entry();
                    }
                    ++issued;
                }

                // ---- S = Q K^T over the 16 tokens of this block ----
                float sacc[2][4];
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) sacc[nt][e] = 0.f;
                // two accumulator chains per n-tile (even / odd k-steps) halve
                // the dependent MMA chain
                float sacc2[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
                for (int kk = 0; kk < D / 16; kk += 2) {
                    mma_16816<T>(sacc[0], qa[kk], kf[kk][0], kf[kk][1]);
                    mma_16816<T>(sacc[1], qa[kk], kf[kk][2], kf[kk][3]);
                    mma_16816<T>(sacc2[0], qa[kk + 1], kf[kk + 1][0], kf[kk + 1][1]);
                    mma_16816<T>(sacc2[1], qa[kk + 1], kf[kk + 1][2], kf[kk + 1][3]);
                }
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) sacc[nt][e] += sacc2[nt][e];

                // ---- mask, online softmax (base 2) ----
                const int lim = c_ctx - cj * 16;   // valid tokens in this block (>= 16: all)
                float pr[2][4];
                float alpha[NT];
#pragma unroll
                for (int pn = 0; pn < NT; ++pn) {
                    float x[2][2];
                    float mx = -INFINITY;
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const int tok = nt * 8 + 2 * t4 + e;
                            x[nt][e] = tok < lim ? sacc[nt][pn * 2 + e] * p.scale_log2 : -INFINITY;
                            mx = fmaxf(mx, x[nt][e]);
                        }
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
                    const float m_new = fmaxf(m_run[pn], mx);
                    alpha[pn] = exp2_approx(m_run[pn] - m_new);
                    m_run[pn] = m_new;
                    float rs = 0.f;
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            pr[nt][pn * 2 + e] = exp2_approx(x[nt][e] - m_new);
                            rs += pr[nt][pn * 2 + e];
                        }
                    l_run[pn] = l_run[pn] * alpha[pn] + rs;
                }

                // tokens beyond the context may hold anything (even NaN): clear
                // their V values in the fragments so 0-weight x garbage cannot
                // reach the accumulator.  Fragment registers 0/1 hold tokens
                // 2*t4 (low half) and 2*t4+1 (high half); registers 2/3 the same
                // tokens + 8.
                if (lim < 16) {
                    const uint32_t m01 = (2 * t4 < lim ? 0x0000ffffu : 0u) | (2 * t4 + 1 < lim ? 0xffff0000u : 0u);
                    const uint32_t m23 = (2 * t4 + 8 < lim ? 0x0000ffffu : 0u) | (2 * t4 + 9 < lim ? 0xffff0000u : 0u);
#pragma unroll
                    for (int mt = 0; mt < D / 16; ++mt) {
                        vf[mt][0] &= m01;
                        vf[mt][1] &= m01;
                        vf[mt][2] &= m23;
                        vf[mt][3] &= m23;
                    }
                }

                // ---- rescale the accumulator (skipped when no row max moved,
                // the common case once a range is under way), O^T += V^T P^T ----
                bool moved = false;
#pragma unroll
                for (int pn = 0; pn < NT; ++pn) moved |= alpha[pn] != 1.f;
                if (__any_sync(0xffffffffu, moved))
#pragma unroll
                    for (int pn = 0; pn < NT; ++pn) {
                        const float a_lo = __shfl_sync(0xffffffffu, alpha[pn], 8 * t4);
                        const float a_hi = __shfl_sync(0xffffffffu, alpha[pn], 8 * t4 + 4);
#pragma unroll
                        for (int mt = 0; mt < D / 16; ++mt) {
                            acc[mt][pn][0] *= a_lo;
                            acc[mt][pn][1] *= a_hi;
                            acc[mt][pn][2] *= a_lo;
                            acc[mt][pn][3] *= a_hi;
                        }
                    }
                uint32_t pb0[NT][2], pb1[NT][2];
#pragma unroll
                for (int pn = 0; pn < NT; ++pn) {
                    pack2_split<T>(pr[0][pn * 2], pr[0][pn * 2 + 1], pb0[pn][0], pb0[pn][1]);
                    pack2_split<T>(pr[1][pn * 2], pr[1][pn * 2 + 1], pb1[pn][0], pb1[pn][1]);
                }
#pragma unroll
                for (int mt = 0; mt < D / 16; ++mt) {
#pragma unroll
                    for (int pn = 0; pn < NT; ++pn) {
                        mma_16816<T>(acc[mt][pn], vf[mt], pb0[pn][0], pb1[pn][0]);
                        mma_16816<T>(acc[mt][pn], vf[mt], pb0[pn][1], pb1[pn][1]);
                    }
                }
                ++piece_n;

                // ---- end of a (sequence, head) range ----
                if (cj == c_nb - 1) {
                    finish_piece();
                    seg_fresh = true;
                }
                // advance the consumer cursor (the next block exists when it
                // is inside this work)
                if (i + 1 < len) {
                    if (++cj == c_nb) {
                        cj = 0;
                        if (++ch == Hkv) {
                            ch = 0;
                            cs = next_seq(cs, c_nb, &c_ctx);
                        }
                    }
                }
            }
            if (!timed_out && !seg_fresh && piece_n > 0) {
                // the work ended inside a range: cj was advanced past the last
                // block taken, so step back to it before closing the piece
                if (i < len) {
                    if (cj == 0) {
                        // cannot happen: a piece that ends at a range boundary
                        // was closed above
                    } else {
                        --cj;
                    }
                }
                finish_piece();
                seg_fresh = true;
            }
            // loads issued but not consumed (speculative, or after a timeout)
            // must land before their slots are reused or the warp leaves
            for (int k = i + (timed_out ? 1 : 0); k < issued; ++k)
                wait_slot(slot_base + k, timed_out ? kWaitLimitNs / 8 : kWaitLimitNs);
            slot_base += issued;
            if (timed_out) {
                set_status(p.dev_status, PKV_DEV_WAIT_TIMEOUT);
                break;
            }
        }

        // ---------------- steal the far half of a busy warp's blocks ----------------
        if (n_own == 0) break;   // a warp without a share of its own does not rob others
        // no share reaches kStealMin blocks (shares differ by at most one
        // block): no warp can ever be robbed in this call
        if ((total + nw - 1) / nw < kStealMin) break;
        // a steal can leave two records: stop when fewer are left
        if (!p.steal || rec_used + 2 > p.rec_per_warp) break;
        // nothing left to take: unclaimed work only shrinks, so once one full
        // scan found no warp worth robbing, none will be again in this call.
        // The drained word and the ready count are read side by side.
        const uint32_t drained = ld_relaxed_u32(p.ctl + kCtlDrained);
        uint32_t rdy = 0u;
        if (lane == 0 && !seen_ready) rdy = ld_acquire_u32(p.ctl + kCtlReady);
        if (drained != 0u) break;
        // thieves rob no warp before every CTA has published its words; the
        // other lanes' reads of range words and prefixes below come after
        // lane 0's acquire of the ready count
        if (lane == 0 && !seen_ready) seen_ready = rdy >= gridDim.x;
        __syncwarp();
        if (!__shfl_sync(0xffffffffu, seen_ready ? 1 : 0, 0)) break;
        bool got = false;
        for (int attempt = 0; attempt < 8 && !got; ++attempt) {
            // every lane reads its share of the range words, eight at a time
            int best = 0;
            int64_t best_v = -1;
            unsigned long long best_w = 0;
            for (int64_t k0 = 0; k0 * 32 < nw; k0 += 8) {
                unsigned long long w[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int64_t v = (k0 + u) * 32 + lane;
                    w[u] = v < nw ? ld_relaxed_u64(p.ranges + v) : 0ull;
                }
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int64_t v = (k0 + u) * 32 + lane;
                    const int rem = (v < nw && v != wg) ? rw_end(w[u]) - rw_begin(w[u]) : 0;
                    if (rem > best) {
                        best = rem;
                        best_v = v;
                        best_w = w[u];
                    }
                }
            }
            // thieves spread over victims: each first tries the best candidate
            // of a lane picked by its own index, and takes the overall best
            // only when that one is too small
            int top = best, top_lane = lane;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const int ob = __shfl_xor_sync(0xffffffffu, top, o);
                const int ol = __shfl_xor_sync(0xffffffffu, top_lane, o);
                if (ob > top || (ob == top && ol < top_lane)) {
                    top = ob;
                    top_lane = ol;
                }
            }
            const int pick = (int)((wg * 7 + attempt) & 31);
            const int picked = __shfl_sync(0xffffffffu, best, pick);
            if (top >= kStealMin && picked >= kStealMin) top_lane = pick;
            if (top < kStealMin) {
                if (lane == 0) atomicExch(p.ctl + kCtlDrained, 1u);
                break;
            }
            int start = 0, take = 0;
            if (lane == top_lane) {
                // the unclaimed blocks are [begin, end): take the far half
                take = (best + 1) / 2;
                start = rw_end(best_w) - take;
                if (atomicCAS(p.ranges + best_v, best_w, rw_make(rw_begin(best_w), start)) != best_w) take = 0;
            }
            take = __shfl_sync(0xffffffffu, take, top_lane);
            start = __shfl_sync(0xffffffffu, start, top_lane);
            const int64_t vv = __shfl_sync(0xffffffffu, best_v, top_lane);
            if (take > 0) {
                got = true;
                x0 = range_lo(vv, total, nw) + start;
                len = take;
            }
        }
        if (!got) break;
        own = false;
        s0 = locate_seq(p, x0, lane);
        off0 = (int)(x0 - __ldcg(p.prefix + s0) * Hkv);
    }

    // ---- the merges this warp owes ----
    __syncwarp();
    for (int k = 0; k < n_defer; ++k) {
        const int4 e = wdefer[k];
        merge_range<T, DO, NT, true>(p, e.x, e.y, e.z, e.w, lane);
    }

    // ---- exit: every block of the plan must have been streamed exactly once
    // (the last CTA out compares the warps' counts with the planned total) ----
    unsigned long long *consumed_ctr = reinterpret_cast<unsigned long long *>(p.ctl + kCtlConsumed64);
    if (lane == 0 && warp_blocks != 0u) atomicAdd(consumed_ctr, (unsigned long long)warp_blocks);
    __threadfence();
    __syncthreads();
    if (tid == 0 && atomicAdd(p.ctl + kCtlExited, 1u) == gridDim.x - 1) {
        __threadfence();
        const unsigned long long consumed = atomicAdd(consumed_ctr, 0ull);
        if ((int64_t)consumed != total) set_status(p.dev_status, PKV_DEV_SPLIT);
    }
}

// Zeroes the decode kernel's control region (n16 16-byte words) before a call.
// It waits for the previous kernel on the stream (which may be the previous
// call, still using the region) and lets the decode kernel launch at once.
__global__ void __launch_bounds__(256) decode_clear_kernel(uint4 *ctl, int n16) {
    pdl_launch_dependents();
    pdl_wait_primary();
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += gridDim.x * blockDim.x)
        ctl[i] = make_uint4(0u, 0u, 0u, 0u);
}

template <typename T, int D, int NT, bool PAIR = false>
static int launch_decode(DecodeParams prm, const CUtensorMap &tk, const CUtensorMap &tv, int grid,
                         size_t clear_bytes, cudaStream_t stream) {
    using Sh = DecodeShape<D, NT>;
    static unsigned long long attr_set = 0;   // per instantiation and device
    if (!done_on_device(&attr_set)) {
        cudaError_t e = cudaFuncSetAttribute(paged_decode_kernel<T, D, NT, PAIR>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, Sh::SMEM_BYTES);
        if (e != cudaSuccess) return cuda_fail(e);
        mark_done_on_device(&attr_set);
    }
    // the control region sits at the front of the workspace
    const int n16 = (int)(clear_bytes / 16);
    const int cgrid = std::min(64, (n16 + 255) / 256);
    cudaError_t e = launch_pdl(decode_clear_kernel, dim3(cgrid), dim3(256), 0, stream,
                               reinterpret_cast<uint4 *>(prm.ctl), n16);
    if (e == cudaSuccess)
        e = launch_pdl(paged_decode_kernel<T, D, NT, PAIR>, dim3(grid), dim3(kDecodeWarps * 32), Sh::SMEM_BYTES, stream,
                       prm, tk, tv);
    if (e == cudaSuccess) e = cudaGetLastError();
    return e == cudaSuccess ? PKV_OK : cuda_fail(e);
}

// ---- workspace ----------------------------------------------------------------
// Control region, zeroed before every call:
//   [control words 256 B][range counter words S*Hkv x 8][range list heads S*Hkv x 4]
// then, written by the call before it reads them:
//   [range slot arrays S*Hkv x n_slots x 8][range words, one per warp x 8]
//   [prefix (S+1) x 8][partial records, rec_per_warp per warp]
// each part 256-B aligned.  A partial record holds G maxima, G sums,
// G x head_dim accumulators and a trailer (link, first block, block count).

static size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

static int record_floats(int G, int head_dim) { return ((2 * G + G * head_dim + 3) & ~3) + 4; }

struct DecodeLayout {
    size_t ctl, seg_cnt, seg_list, clear_bytes, seg_slots, ranges, prefix, part, fixed;
};

static DecodeLayout decode_layout(int S, int Hkv, int total_warps, int n_slots) {
    DecodeLayout L;
    size_t o = 0;
    L.ctl = o;
    o += kCtlBytes;
    L.seg_cnt = o;
    o += align256((size_t)S * Hkv * 8);
    L.seg_list = o;
    o += align256((size_t)S * Hkv * 4);
    L.clear_bytes = o;
    L.seg_slots = o;
    o += align256((size_t)S * Hkv * n_slots * 8);
    L.ranges = o;
    o += align256((size_t)total_warps * 8);
    L.prefix = o;
    o += align256((size_t)(S + 1) * 8);
    L.part = o;
    L.fixed = o;
    return L;
}

// records per warp: two for its own range (the pieces at its ends) plus two
// per steal; the recommended size allows four steals per warp
constexpr int kRecordsMin = 2;
constexpr int kRecordsRecommended = 10;
static size_t records_min(int total_warps) { return (size_t)kRecordsMin * total_warps; }
static size_t records_recommended(int total_warps) { return (size_t)kRecordsRecommended * total_warps; }

// head_dim 64 with groups of at most 4 query heads and an even number of KV
// heads can run two adjacent KV heads as one unit (the kernel's PAIR form):
// the kernel then sees num_kv_heads / 2 units of 2G query heads each.  A unit
// then streams twice the bytes at twice the arithmetic, which pays while the
// warps have long shares (the step is bound by bandwidth), and costs in a
// small step, where each warp's few units are a chain of round trips.  So it
// is used from 256 sequence x KV-pair ranges on, or from 512 when the block
// tables are wider than 128 blocks: contexts past 2,048 tokens, whose long
// ranges a small step cuts into many pieces.
static bool pair_eligible(int num_q_heads, int num_kv_heads, int head_dim) {
    return head_dim == 64 && num_kv_heads % 2 == 0 && num_q_heads / num_kv_heads <= 4;
}

static bool pair_wanted(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim, int max_blocks_per_seq) {
    if (!pair_eligible(num_q_heads, num_kv_heads, head_dim)) return false;
    const int64_t ranges = (int64_t)num_seqs * (num_kv_heads / 2);
    return ranges >= (max_blocks_per_seq > 128 ? 512 : 256);
}

static int slots_for(int num_seqs, int units) {
    return (int64_t)num_seqs * units <= kManySlotsRanges ? kSlotsMax : kSlots;
}

static size_t workspace_bytes_for(int num_seqs, int num_q_heads, int units, int head_dim, int nw, size_t records,
                                  int n_slots) {
    return decode_layout(num_seqs, units, nw, n_slots).fixed +
           records * (size_t)record_floats(num_q_heads / units, head_dim) * sizeof(float);
}

// The smallest workspace a call accepts (the paired form falls back to the
// single-head one when its own layout does not fit).
size_t decode_workspace_min(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim) {
    if (num_seqs < 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0) return 0;
    int sms = 0;
    if (current_sm_count(&sms) != PKV_OK) return 0;
    const int nw = sms * kDecodeWarps;
    size_t need = workspace_bytes_for(num_seqs, num_q_heads, num_kv_heads, head_dim, nw, records_min(nw), kSlots);
    if (pair_eligible(num_q_heads, num_kv_heads, head_dim))
        need = std::min(need, workspace_bytes_for(num_seqs, num_q_heads, num_kv_heads / 2, head_dim, nw,
                                                  records_min(nw), kSlots));
    return need;
}

}  // namespace pkv

extern "C" size_t pkv_decode_workspace_size(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim) {
    using namespace pkv;
    if (num_seqs < 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0) return 0;
    int sms = 0;
    if (current_sm_count(&sms) != PKV_OK) return 0;
    const int nw = sms * kDecodeWarps;
    // large enough for either form
    size_t need = workspace_bytes_for(num_seqs, num_q_heads, num_kv_heads, head_dim, nw, records_recommended(nw),
                                      slots_for(num_seqs, num_kv_heads));
    if (pair_eligible(num_q_heads, num_kv_heads, head_dim))
        need = std::max(need, workspace_bytes_for(num_seqs, num_q_heads, num_kv_heads / 2, head_dim, nw,
                                                  records_recommended(nw), slots_for(num_seqs, num_kv_heads / 2)));
    return need;
}

namespace pkv {

// The decode entry point with the grid capped at max_sms CTAs (0: one per SM).
int decode_attention(void *out, const void *q, const void *k_cache, const void *v_cache,
                     const int32_t *block_tables, int max_blocks_per_seq, const int32_t *context_lens, int num_seqs,
                     int num_blocks, int num_q_heads, int num_kv_heads, int head_dim, int block_size, float scale,
                     int dtype, int out_dtype, void *workspace, size_t workspace_bytes, int *dev_status,
                     cudaStream_t stream, int max_sms, const void *k_new, const void *v_new) {
    if (num_seqs < 0 || num_blocks <= 0 || num_kv_heads <= 0 || num_q_heads <= 0 || max_blocks_per_seq <= 0)
        return PKV_ERR_INVALID_ARG;
    if (num_q_heads % num_kv_heads != 0) return PKV_ERR_INVALID_ARG;
    const int G = num_q_heads / num_kv_heads;
    if (G > 16 || block_size != 16 || (head_dim != 64 && head_dim != 128)) return PKV_ERR_UNSUPPORTED;
    if (dtype != PKV_DTYPE_F16 && dtype != PKV_DTYPE_BF16) return PKV_ERR_UNSUPPORTED;
    if (out_dtype != dtype && out_dtype != PKV_DTYPE_F32) return PKV_ERR_UNSUPPORTED;
    if (!std::isfinite(scale)) return PKV_ERR_INVALID_ARG;
    if ((int64_t)num_blocks * num_kv_heads * block_size >= (int64_t)1 << 31) return PKV_ERR_UNSUPPORTED;
    if ((int64_t)num_seqs * max_blocks_per_seq >= (int64_t)1 << 31) return PKV_ERR_UNSUPPORTED;
    // a range's first block and block count live in 20-bit fields of its slots
    if (max_blocks_per_seq >= (1 << kSlotBlkBits)) return PKV_ERR_UNSUPPORTED;
    if (num_seqs == 0) return PKV_OK;
    if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens || !workspace)
        return PKV_ERR_INVALID_ARG;
    if (!aligned(q, 4) || !aligned(out, 4) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
        !aligned(block_tables, 4) || !aligned(context_lens, 4))
        return PKV_ERR_INVALID_ARG;
    if (!aligned(workspace, 16)) return PKV_ERR_WORKSPACE;
    if ((k_new == nullptr) != (v_new == nullptr)) return PKV_ERR_INVALID_ARG;
    if (k_new && (!aligned(k_new, 16) || !aligned(v_new, 16))) return PKV_ERR_INVALID_ARG;
    int sms = 0;
    int rc = current_sm_count(&sms);
    if (rc != PKV_OK) return rc;
    // the kernel's units: KV heads, or pairs of adjacent KV heads
    bool pair = pair_wanted(num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq);
    int units = 0, Gu = 0, total_warps = 0, grid = 0;
    int64_t upper = 0;
    DecodeLayout lay;
    size_t rec_bytes = 0;
    for (;;) {
        units = pair ? num_kv_heads / 2 : num_kv_heads;
        Gu = num_q_heads / units;
        // enough warps for the largest possible total, at most one CTA per SM
        upper = (int64_t)num_seqs * units * max_blocks_per_seq;
        grid = (int)((upper + kDecodeWarps - 1) / kDecodeWarps);
        if (grid > sms) grid = sms;
        if (max_sms > 0 && grid > max_sms) grid = max_sms;
        if (grid < 1) grid = 1;
        total_warps = grid * kDecodeWarps;
        lay = decode_layout(num_seqs, units, total_warps, kSlots);
        rec_bytes = (size_t)record_floats(Gu, head_dim) * sizeof(float);
        // the paired form falls back to single heads when its layout does not fit
        if (pair && workspace_bytes < lay.fixed + records_min(total_warps) * rec_bytes) {
            pair = false;
            continue;
        }
        break;
    }
    // range offsets are 32-bit fields
    if (upper / total_warps + 1 >= ((int64_t)1 << 30)) return PKV_ERR_UNSUPPORTED;
    if (workspace_bytes < lay.fixed + records_min(total_warps) * rec_bytes) return PKV_ERR_WORKSPACE;
    // the full slot arrays for a step of few ranges, when they leave the
    // recommended records room
    int n_slots = kSlots;
    if (slots_for(num_seqs, units) == kSlotsMax) {
        const DecodeLayout big = decode_layout(num_seqs, units, total_warps, kSlotsMax);
        if (workspace_bytes >= big.fixed + records_recommended(total_warps) * rec_bytes) {
            lay = big;
            n_slots = kSlotsMax;
        }
    }
    // records per warp (record numbers live in 24-bit slot fields)
    size_t per_warp = (workspace_bytes - lay.fixed) / rec_bytes / total_warps;
    const size_t max_per_warp = (((size_t)1 << kSlotRecBits) - 2) / total_warps;
    if (per_warp > max_per_warp) per_warp = max_per_warp;

    CUtensorMap tk, tv;
    rc = encode_cache_map(&tk, k_cache, num_blocks, num_kv_heads, block_size, head_dim);
    if (rc != PKV_OK) return rc;
    rc = encode_cache_map(&tv, v_cache, num_blocks, num_kv_heads, block_size, head_dim);
    if (rc != PKV_OK) return rc;

    char *ws = static_cast<char *>(workspace);
    DecodeParams prm;
    prm.out = out;
    prm.q = q;
    prm.block_tables = block_tables;
    prm.context_lens = context_lens;
    prm.ctl = reinterpret_cast<uint32_t *>(ws + lay.ctl);
    prm.seg_cnt = reinterpret_cast<unsigned long long *>(ws + lay.seg_cnt);
    prm.seg_list = reinterpret_cast<uint32_t *>(ws + lay.seg_list);
    prm.seg_slots = reinterpret_cast<unsigned long long *>(ws + lay.seg_slots);
    prm.ranges = reinterpret_cast<unsigned long long *>(ws + lay.ranges);
    prm.prefix = reinterpret_cast<long long *>(ws + lay.prefix);
    prm.part = reinterpret_cast<float *>(ws + lay.part);
    prm.dev_status = dev_status;
    prm.S = num_seqs;
    prm.max_blocks = max_blocks_per_seq;
    prm.num_blocks = num_blocks;
    prm.Hq = num_q_heads;
    prm.Hkv = units;
    prm.G = Gu;
    prm.scale_log2 = scale * 1.4426950408889634f;
    prm.out_dtype = out_dtype;
    prm.total_warps = total_warps;
    prm.rec_floats = record_floats(Gu, head_dim);
    prm.rec_per_warp = (int)per_warp;
    // PKV_DETERMINISTIC=1: no stealing, so the split of every range is fixed
    // by the contexts alone and the output bits repeat from call to call
    const char *det = std::getenv("PKV_DETERMINISTIC");
    prm.steal = (det && det[0] == '1') ? 0 : 1;
    prm.n_slots = n_slots;
    prm.k_new = k_new;
    prm.v_new = v_new;
    prm.k_cache = const_cast<void *>(k_cache);
    prm.v_cache = const_cast<void *>(v_cache);
    cudaStream_t st = stream;
    const bool wide = G > 8;
    if (pair)
        return dtype == PKV_DTYPE_BF16 ? launch_decode<__nv_bfloat16, 128, 1, true>(prm, tk, tv, grid, lay.clear_bytes, st)
                                       : launch_decode<__half, 128, 1, true>(prm, tk, tv, grid, lay.clear_bytes, st);
    if (dtype == PKV_DTYPE_BF16) {
        if (head_dim == 128)
            return wide ? launch_decode<__nv_bfloat16, 128, 2>(prm, tk, tv, grid, lay.clear_bytes, st)
                        : launch_decode<__nv_bfloat16, 128, 1>(prm, tk, tv, grid, lay.clear_bytes, st);
        return wide ? launch_decode<__nv_bfloat16, 64, 2>(prm, tk, tv, grid, lay.clear_bytes, st)
                    : launch_decode<__nv_bfloat16, 64, 1>(prm, tk, tv, grid, lay.clear_bytes, st);
    }
    if (head_dim == 128)
        return wide ? launch_decode<__half, 128, 2>(prm, tk, tv, grid, lay.clear_bytes, st)
                    : launch_decode<__half, 128, 1>(prm, tk, tv, grid, lay.clear_bytes, st);
    return wide ? launch_decode<__half, 64, 2>(prm, tk, tv, grid, lay.clear_bytes, st)
                : launch_decode<__half, 64, 1>(prm, tk, tv, grid, lay.clear_bytes, st);
}

}  // namespace pkv

extern "C" int pkv_paged_decode_attention(void *out, const void *q, const void *k_cache, const void *v_cache,
                                          const int32_t *block_tables, int max_blocks_per_seq,
                                          const int32_t *context_lens, int num_seqs, int num_blocks,
                                          int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                          float scale, int dtype, int out_dtype, void *workspace,
                                          size_t workspace_bytes, int *dev_status, void *stream) {
    pkv::NvtxRange nvtx_range("pkv_paged_decode_attention");
    return pkv::decode_attention(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, num_seqs,
                                 num_blocks, num_q_heads, num_kv_heads, head_dim, block_size, scale, dtype, out_dtype,
                                 workspace, workspace_bytes, dev_status, static_cast<cudaStream_t>(stream), 0);
}

extern "C" int pkv_paged_decode_append_attention(void *out, const void *q, const void *k_new, const void *v_new,
                                                 void *k_cache, void *v_cache, const int32_t *block_tables,
                                                 int max_blocks_per_seq, const int32_t *context_lens, int num_seqs,
                                                 int num_blocks, int num_q_heads, int num_kv_heads, int head_dim,
                                                 int block_size, float scale, int dtype, int out_dtype,
                                                 void *workspace, size_t workspace_bytes, int *dev_status,
                                                 void *stream) {
    pkv::NvtxRange nvtx_range("pkv_paged_decode_append_attention");
    if (num_seqs > 0 && (!k_new || !v_new)) return PKV_ERR_INVALID_ARG;
    return pkv::decode_attention(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, num_seqs,
                                 num_blocks, num_q_heads, num_kv_heads, head_dim, block_size, scale, dtype, out_dtype,
                                 workspace, workspace_bytes, dev_status, static_cast<cudaStream_t>(stream), 0, k_new,
                                 v_new);
}
