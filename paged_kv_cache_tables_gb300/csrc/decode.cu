// K2 + K3: paged decode attention with a split KV range and a log-sum-exp merge.
//
// What is computed: "Project 17: Production Serving: Continuous Batching and
// PagedAttention", Step 6 "Implement attention over paged storage" -- walk a
// sequence's page table, score every stored key against the query scaled by
// 1/sqrt(head_dim), softmax over the sequence, weighted sum of the stored
// values -- per query head, with query head h reading KV head h / G.
//
// How (GB300):
//  * Work = the flat list of (sequence, KV head, block) triples, cut into equal
//    contiguous ranges, one per warp of a persistent grid (one CTA of 8 warps
//    per SM).  Every warp streams the same number of 16-token blocks, whatever
//    the context-length mix; a (sequence, head) range that crosses a warp
//    boundary leaves per-warp partials (m, l, acc), and the warp that finishes
//    the range's last piece combines them by log-sum-exp (an arrival counter
//    per range, tagged with the call's epoch, tells it that it is last).
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

#include <atomic>
#include <cmath>

#include "pkv.h"
#include "pkv_device.cuh"
#include "pkv_host.h"

namespace pkv {

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // a tile that has not landed in 2 s never will
constexpr int kDecodeWarps = 8;

struct DecodeParams {
    void *out;
    const void *q;
    const int32_t *block_tables;
    const int32_t *context_lens;
    float *part;        // [2 * total_warps][record] partial results
    unsigned long long *arrivals;   // [S * Hkv]: (epoch << 32) | pieces arrived
    int *dev_status;
    int S, max_blocks, num_blocks, Hq, Hkv, G;
    float scale_log2;   // scale * log2(e): scores are kept in base-2 units
    int out_dtype;
    int total_warps;
    uint32_t epoch;     // nonzero, different for every call
};

template <int D, int NT>
struct DecodeShape {
    static constexpr int HALVES = D / 64;              // 64-element (128-byte) column halves
    static constexpr int HALF_BYTES = 64 * 16 * 2;     // one 16-row half tile
    static constexpr int TILE_BYTES = HALVES * HALF_BYTES;
    static constexpr int STAGE_BYTES = 2 * TILE_BYTES;  // K + V
    static constexpr int STAGES = D == 128 ? 3 : 6;
    static constexpr int HP = 8 * NT;                   // heads held by a partial record
    static constexpr int REC = 2 * HP + HP * D;         // m[HP], l[HP], acc[HP][D]
    static constexpr int RING_BYTES = kDecodeWarps * STAGES * STAGE_BYTES;
    static constexpr int SMEM_BYTES = 1024 + RING_BYTES + kDecodeWarps * STAGES * 8 + 256;
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

// The warp whose range holds flat position x: the largest w with range_lo(w) <= x.
__device__ __forceinline__ int64_t owner_of(int64_t x, int64_t total, int64_t nw) {
    return ((x + 1) * nw + total - 1) / total - 1;
}

// Counts one more finished piece of a split (sequence, KV head) range and
// returns how many have finished in this call.  The counter carries the call's
// epoch in its high half, so a value left by an earlier call counts as zero
// and the workspace never needs clearing.  Returns 0 if the update kept losing
// races (not expected: at most a handful of warps share a range).
__device__ __forceinline__ uint32_t count_arrival(unsigned long long *ctr, uint32_t epoch) {
    unsigned long long cur = atomicAdd(ctr, 0ull);
    for (int it = 0; it < (1 << 16); ++it) {
        const unsigned long long want =
            (uint32_t)(cur >> 32) == epoch ? cur + 1ull : (((unsigned long long)epoch << 32) | 1ull);
        unsigned long long prev;
        asm volatile("atom.acq_rel.gpu.global.cas.b64 %0, [%1], %2, %3;"
                     : "=l"(prev)
                     : "l"(ctr), "l"(cur), "l"(want)
                     : "memory");
        if (prev == cur) return (uint32_t)(want & 0xffffffffull);
        cur = prev;
    }
    return 0;
}

// Log-sum-exp combination of the partial records of one split range, run by
// the warp that finished its last piece.  Records: warp w0 left its piece in
// slot 1 (range ended past its end), later warps in slot 0.  Lane hh folds the
// (max, sum) pairs of head hh over the pieces; then every lane accumulates its
// D/32 output columns of every head, with all loads of a piece independent.
template <typename T, int D, int NT>
__device__ __forceinline__ void merge_pieces(const DecodeParams &p, int64_t w0, int64_t w1, int64_t total,
                                             int64_t nw, int s, int h, int lane) {
    using Sh = DecodeShape<D, NT>;
    constexpr int HP = Sh::HP, PER = D / 32;
    const int G = p.G;
    auto rec_of = [&](int64_t w) { return p.part + (size_t)(w * 2 + (w == w0 ? 1 : 0)) * Sh::REC; };
    auto empty_range = [&](int64_t w) { return range_lo(w + 1, total, nw) == range_lo(w, total, nw); };
    float M = -INFINITY, L = 0.f;
    if (lane < G) {
        for (int64_t w = w0; w <= w1; ++w) {
            if (empty_range(w)) continue;
            const float *rec = rec_of(w);
            const float mv = __ldcg(rec + lane), lv = __ldcg(rec + HP + lane);
            const float Mn = fmaxf(M, mv);
            L = L * exp2_approx(M - Mn) + lv * exp2_approx(mv - Mn);
            M = Mn;
        }
    }
    float Mh[HP], invL[HP], o[HP][PER];
#pragma unroll
    for (int hh = 0; hh < HP; ++hh) {
        Mh[hh] = __shfl_sync(0xffffffffu, M, hh);
        invL[hh] = 1.f / __shfl_sync(0xffffffffu, L, hh);
#pragma unroll
        for (int k = 0; k < PER; ++k) o[hh][k] = 0.f;
    }
    for (int64_t w = w0; w <= w1; ++w) {
        if (empty_range(w)) continue;
        const float *rec = rec_of(w);
#pragma unroll
        for (int hh = 0; hh < HP; ++hh) {
            if (hh < G) {
                const float f = exp2_approx(__ldcg(rec + hh) - Mh[hh]) * invL[hh];
                const float *racc = rec + 2 * HP + hh * D;
#pragma unroll
                for (int k = 0; k < PER; ++k) o[hh][k] += f * __ldcg(racc + lane + 32 * k);
            }
        }
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

template <typename T, int D, int NT>
__global__ void __launch_bounds__(kDecodeWarps * 32, 1)
    paged_decode_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap tk,
                        const __grid_constant__ CUtensorMap tv) {
    using Sh = DecodeShape<D, NT>;
    constexpr int STAGES = Sh::STAGES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *ring = smem;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Sh::RING_BYTES);
    int64_t *sh_scan = reinterpret_cast<int64_t *>(bars + kDecodeWarps * STAGES);
    int *plan_s = reinterpret_cast<int *>(sh_scan + kDecodeWarps);   // segment holding each warp's first block
    int *plan_off = plan_s + kDecodeWarps;
    int *plan_s2 = plan_off + kDecodeWarps;                             // ... and its last block
    int *plan_off2 = plan_s2 + kDecodeWarps;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int Hkv = p.Hkv;

    // inputs may come from the previous kernel on the stream (the append)
    pdl_wait_primary();
    pdl_launch_dependents();

    // ---- plan: total blocks, this CTA's warp ranges, per-sequence offsets ----
    int64_t local = 0;
    for (int s = tid; s < p.S; s += blockDim.x) local += blocks_of(p.context_lens, s, p.max_blocks, p.dev_status, nullptr);
    int64_t total_nblk;
    block_scan(local, sh_scan, &total_nblk);
    const int64_t total = total_nblk * Hkv;
    const int64_t nw = p.total_warps;
    if (tid < kDecodeWarps) plan_s[tid] = -1;
    __syncthreads();
    int64_t carry = 0;
    for (int base = 0; base < p.S; base += blockDim.x) {
        const int s = base + tid;
        const int nb = s < p.S ? blocks_of(p.context_lens, s, p.max_blocks, nullptr, nullptr) : 0;
        int64_t tile_total;
        const int64_t excl = carry + block_scan(nb, sh_scan, &tile_total) - nb;
        if (nb > 0) {
#pragma unroll
            for (int w = 0; w < kDecodeWarps; ++w) {
                const int64_t lo = range_lo((int64_t)blockIdx.x * kDecodeWarps + w, total, nw);
                const int64_t last = range_lo((int64_t)blockIdx.x * kDecodeWarps + w + 1, total, nw) - 1;
                if (lo >= excl * Hkv && lo < (excl + nb) * Hkv) {
                    plan_s[w] = s;
                    plan_off[w] = (int)(lo - excl * Hkv);
                }
                if (last >= excl * Hkv && last < (excl + nb) * Hkv) {
                    plan_s2[w] = s;
                    plan_off2[w] = (int)(last - excl * Hkv);
                }
            }
        }
        carry += tile_total;
    }
    __syncthreads();

    // sequences with an empty context get all-zero rows
    for (int s = blockIdx.x; s < p.S; s += gridDim.x) {
        if (blocks_of(p.context_lens, s, p.max_blocks, nullptr, nullptr) != 0) continue;
        for (int e = tid; e < p.Hq * D; e += blockDim.x) store_out<T>(p.out, p.out_dtype, (int64_t)s * p.Hq * D + e, 0.f);
    }

    const int64_t wg = (int64_t)blockIdx.x * kDecodeWarps + warp;
    const int64_t lo_w = range_lo(wg, total, nw);
    const int n = (int)(range_lo(wg + 1, total, nw) - lo_w);
    if (n <= 0 || plan_s[warp] < 0) return;

    // ---- this warp's ring ----
    uint8_t *wring = ring + warp * STAGES * Sh::STAGE_BYTES;
    uint64_t *wbar = bars + warp * STAGES;
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

    // Block order inside the range: if the range's last (sequence, KV head)
    // segment continues into the next warp, that tail piece is streamed first,
    // then the range from its start.  Both pieces of a split segment are then
    // finished early in the kernel, so the warp that combines them does so
    // while the other warps keep HBM busy, not at the very end.
    const int s_head = plan_s[warp], off_head = plan_off[warp];
    const int nb_head = blocks_of(p.context_lens, s_head, p.max_blocks, nullptr, nullptr);
    const int s_last = plan_s2[warp];
    const int nb_last = blocks_of(p.context_lens, s_last, p.max_blocks, nullptr, nullptr);
    const int j_last = plan_off2[warp] % nb_last;
    const int64_t t_start = lo_w + n - 1 - j_last;                  // flat start of the last segment
    const int n_tail = (j_last < nb_last - 1 && t_start > lo_w) ? (int)(lo_w + n - t_start) : 0;

    auto next_seq = [&](int s, int &nb_out, int *ctx_out) {
        int nb;
        do {
            ++s;
            nb = blocks_of(p.context_lens, s, p.max_blocks, nullptr, ctx_out);
        } while (nb == 0);
        nb_out = nb;
        return s;
    };
    // consumer (c*) and producer (p*) cursors over (sequence, head, block)
    int cs, c_ctx, c_nb, ch, cj;
    auto seek_head = [&](int &s_, int &nb_, int &h_, int &j_, int *ctx_) {
        s_ = s_head;
        nb_ = blocks_of(p.context_lens, s_, p.max_blocks, nullptr, ctx_);
        h_ = off_head / nb_;
        j_ = off_head % nb_;
    };
    if (n_tail > 0) {
        cs = s_last;
        c_nb = blocks_of(p.context_lens, cs, p.max_blocks, nullptr, &c_ctx);
        ch = plan_off2[warp] / c_nb;
        cj = 0;
    } else {
        seek_head(cs, c_nb, ch, cj, &c_ctx);
    }
    int ps = cs, p_nb = c_nb, ph = ch, pj = cj;
    bool started_mid = n_tail == 0 && cj != 0;
    (void)nb_head;

    auto table_entry = [&]() { return __ldg(p.block_tables + (int64_t)ps * p.max_blocks + pj); };
    // move the producer from block k of the warp's order to block k + 1
    auto advance_producer = [&](int k) {
        if (k + 1 == n_tail) {
            seek_head(ps, p_nb, ph, pj, nullptr);
            return;
        }
        if (++pj == p_nb) {
            pj = 0;
            if (++ph == Hkv) {
                ph = 0;
                ps = next_seq(ps, p_nb, nullptr);
            }
        }
    };
    auto issue = [&](int stage, int blk) {
        if (lane == 0) {
            int row = (blk * Hkv + ph) * 16;
            if (blk < 0 || blk >= p.num_blocks) {
                set_status(p.dev_status, PKV_DEV_BAD_BLOCK_ID);
                row = p.num_blocks * Hkv * 16;   // past the end: the load fills zeros
            }
            uint64_t *bar = &wbar[stage];
            mbar_arrive_expect_tx(bar, Sh::STAGE_BYTES);
            uint8_t *kdst = wring + stage * Sh::STAGE_BYTES;
            uint8_t *vdst = kdst + Sh::TILE_BYTES;
#pragma unroll
            for (int hf = 0; hf < Sh::HALVES; ++hf) {
                tma_load_2d(kdst + hf * Sh::HALF_BYTES, &tk, hf * 64, row, bar, policy);
                tma_load_2d(vdst + hf * Sh::HALF_BYTES, &tv, hf * 64, row, bar, policy);
            }
        }
    };

    // prologue: fill the ring
    int pending = table_entry();
    const int pro = n < STAGES ? n : STAGES;
    for (int k = 0; k < pro; ++k) {
        issue(k, pending);
        if (k + 1 < n) {
            advance_producer(k);
            pending = table_entry();
        }
    }

    const int g = lane >> 2, t4 = lane & 3;
    const int mi = lane >> 3;
    const int ld_row = ((mi >> 1) << 3) + (lane & 7);          // token row this lane addresses
    const int ld_sw = ld_row & 7;                               // 128-byte swizzle phase of that row
    const uint32_t ring_addr = smem_addr(wring);

    uint32_t qa[D / 16][4];
    float acc[D / 16][NT][4];
    float m_run[NT], l_run[NT];
    bool seg_fresh = true;

    const int G = p.G;
    for (int i = 0; i < n; ++i) {
        if (seg_fresh) {
            // query fragments of (cs, ch): rows = heads of the group (padded to 16)
            const uint32_t *qbase = reinterpret_cast<const uint32_t *>(
                static_cast<const T *>(p.q) + ((int64_t)cs * p.Hq + (int64_t)ch * G) * D);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const int c0 = (kk * 16 + 2 * t4) >> 1;
                qa[kk][0] = g < G ? __ldg(qbase + g * (D / 2) + c0) : 0u;
                qa[kk][2] = g < G ? __ldg(qbase + g * (D / 2) + c0 + 4) : 0u;
                if constexpr (NT == 1) {   // group of at most 8 heads: rows 8..15 are padding
                    qa[kk][1] = 0u;
                    qa[kk][3] = 0u;
                } else {
                    qa[kk][1] = g + 8 < G ? __ldg(qbase + (g + 8) * (D / 2) + c0) : 0u;
                    qa[kk][3] = g + 8 < G ? __ldg(qbase + (g + 8) * (D / 2) + c0 + 4) : 0u;
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
        }

        const int stage = i % STAGES;
        const bool landed = mbar_wait(&wbar[stage], (uint32_t)((i / STAGES) & 1), kWaitLimitNs);
        if (!__all_sync(0xffffffffu, landed)) {
            set_status(p.dev_status, PKV_DEV_WAIT_TIMEOUT);
            // let the copies this warp still has in flight land before leaving
            for (int k = i + 1; k < n && k < i + STAGES; ++k)
                mbar_wait(&wbar[k % STAGES], (uint32_t)((k / STAGES) & 1), kWaitLimitNs / 8);
            return;
        }
        const uint32_t kbase = ring_addr + stage * Sh::STAGE_BYTES;
        const uint32_t vbase = kbase + Sh::TILE_BYTES;

        // ---- pull the block's K and V fragments into registers, then hand the
        // slot straight back to the TMA engine: the slot is held for the
        // ldmatrix reads only, not for the whole block's arithmetic ----
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
        if (i + STAGES < n) {
            issue(stage, pending);
            if (i + STAGES + 1 < n) {
                advance_producer(i + STAGES);
                pending = table_entry();
            }
        }

        // ---- S = Q K^T over the 16 tokens of this block ----
        float sacc[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) sacc[nt][e] = 0.f;
        // two accumulator chains per n-tile (even / odd k-steps) halve the
        // dependent MMA chain
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

        // tokens beyond the context may hold anything (even NaN): clear their
        // V values in the fragments so 0-weight x garbage cannot reach the
        // accumulator.  Fragment registers 0/1 hold tokens 2*t4 (low half)
        // and 2*t4+1 (high half); registers 2/3 the same tokens + 8.
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

        // ---- rescale the accumulator (skipped when no row max moved, the
        // common case once a range is under way), O^T += V^T P^T ----
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

        // ---- end of a (sequence, head) range in this warp ----
        const bool seg_done = cj == c_nb - 1;
        if (seg_done || i == n - 1 || i == n_tail - 1) {
            float lsum[NT];
#pragma unroll
            for (int pn = 0; pn < NT; ++pn) {
                lsum[pn] = l_run[pn];
                lsum[pn] += __shfl_xor_sync(0xffffffffu, lsum[pn], 1);
                lsum[pn] += __shfl_xor_sync(0xffffffffu, lsum[pn], 2);
            }
            const int head0 = ch * G;
            if (!started_mid && seg_done) {
                // whole range in this warp: normalise and store
#pragma unroll
                for (int pn = 0; pn < NT; ++pn) {
                    const float inv_lo = 1.f / __shfl_sync(0xffffffffu, lsum[pn], 8 * t4);
                    const float inv_hi = 1.f / __shfl_sync(0xffffffffu, lsum[pn], 8 * t4 + 4);
                    const int ha = pn * 8 + 2 * t4, hb = ha + 1;
#pragma unroll
                    for (int mt = 0; mt < D / 16; ++mt) {
                        const int d0 = mt * 16 + g;
                        if (ha < G) {
                            const int64_t o = ((int64_t)cs * p.Hq + head0 + ha) * D;
                            store_out<T>(p.out, p.out_dtype, o + d0, acc[mt][pn][0] * inv_lo);
                            store_out<T>(p.out, p.out_dtype, o + d0 + 8, acc[mt][pn][2] * inv_lo);
                        }
                        if (hb < G) {
                            const int64_t o = ((int64_t)cs * p.Hq + head0 + hb) * D;
                            store_out<T>(p.out, p.out_dtype, o + d0, acc[mt][pn][1] * inv_hi);
                            store_out<T>(p.out, p.out_dtype, o + d0 + 8, acc[mt][pn][3] * inv_hi);
                        }
                    }
                }
            } else {
                // part of a range shared with other warps: leave (m, l, acc)
                float *rec = p.part + (size_t)(wg * 2 + (started_mid ? 0 : 1)) * Sh::REC;
#pragma unroll
                for (int pn = 0; pn < NT; ++pn) {
                    if (t4 == 0) {
                        rec[pn * 8 + g] = m_run[pn];
                        rec[Sh::HP + pn * 8 + g] = lsum[pn];
                    }
                    float *racc = rec + 2 * Sh::HP;
                    const int ha = pn * 8 + 2 * t4, hb = ha + 1;
#pragma unroll
                    for (int mt = 0; mt < D / 16; ++mt) {
                        const int d0 = mt * 16 + g;
                        racc[ha * D + d0] = acc[mt][pn][0];
                        racc[hb * D + d0] = acc[mt][pn][1];
                        racc[ha * D + d0 + 8] = acc[mt][pn][2];
                        racc[hb * D + d0 + 8] = acc[mt][pn][3];
                    }
                }
                // the warp that finishes the last piece of the range combines
                // them; the counter update is a release (it publishes the
                // record the lanes wrote before the __syncwarp) and an acquire
                // (the last arriver then sees every other piece's record)
                __syncwarp();
                const int64_t flat = i < n_tail ? t_start + i : lo_w + (i - n_tail);
                const int64_t seg_lo = flat - cj, seg_hi = seg_lo + c_nb - 1;
                const int64_t w0 = owner_of(seg_lo, total, nw), w1 = owner_of(seg_hi, total, nw);
                uint32_t pieces = 0;
                for (int64_t w = w0; w <= w1; ++w) pieces += range_lo(w + 1, total, nw) > range_lo(w, total, nw);
                unsigned long long *ctr = p.arrivals + (size_t)cs * Hkv + ch;
                uint32_t arrived = 0;
                if (lane == 0) arrived = count_arrival(ctr, p.epoch);
                arrived = __shfl_sync(0xffffffffu, arrived, 0);
                if (arrived == pieces) {
                    __syncwarp();
                    merge_pieces<T, D, NT>(p, w0, w1, total, nw, cs, ch, lane);
                    if (lane == 0) atomicExch(ctr, 0ull);
                } else if (arrived == 0) {
                    set_status(p.dev_status, PKV_DEV_WAIT_TIMEOUT);
                }
            }
            started_mid = false;
            seg_fresh = true;
        }
        // advance the consumer cursor
        if (i + 1 == n_tail) {
            seek_head(cs, c_nb, ch, cj, &c_ctx);
            started_mid = cj != 0;
        } else if (i + 1 < n) {
            if (++cj == c_nb) {
                cj = 0;
                if (++ch == Hkv) {
                    ch = 0;
                    cs = next_seq(cs, c_nb, &c_ctx);
                }
            }
        }
    }
}

template <typename T, int D, int NT>
static int launch_decode(DecodeParams prm, const CUtensorMap &tk, const CUtensorMap &tv, int grid,
                         cudaStream_t stream) {
    using Sh = DecodeShape<D, NT>;
    static bool attr_set = false;   // per instantiation; idempotent if raced
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(paged_decode_kernel<T, D, NT>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, Sh::SMEM_BYTES);
        if (e != cudaSuccess) return cuda_fail(e);
        attr_set = true;
    }
    cudaError_t e = launch_pdl(paged_decode_kernel<T, D, NT>, dim3(grid), dim3(kDecodeWarps * 32), Sh::SMEM_BYTES,
                               stream, prm, tk, tv);
    if (e == cudaSuccess) e = cudaGetLastError();
    return e == cudaSuccess ? PKV_OK : cuda_fail(e);
}

static size_t decode_record_floats(int G, int head_dim) {
    const int HP = G > 8 ? 16 : 8;
    return (size_t)(2 * HP + HP * head_dim);
}

// Workspace: [arrival counters, S * Hkv x 8 B, padded to 256 B][partial records].
static size_t arrivals_bytes(int S, int Hkv) { return ((size_t)S * Hkv * 8 + 255) & ~size_t(255); }

static size_t workspace_bytes_for(int S, int Hkv, int G, int head_dim, int total_warps) {
    return arrivals_bytes(S, Hkv) + (size_t)2 * total_warps * decode_record_floats(G, head_dim) * sizeof(float);
}

static uint32_t next_epoch() {
    static std::atomic<uint32_t> epoch{0};
    uint32_t e = ++epoch;
    if (e == 0) e = ++epoch;
    return e;
}

}  // namespace pkv

extern "C" size_t pkv_decode_workspace_size(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim) {
    using namespace pkv;
    if (num_seqs < 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0) return 0;
    int sms = 0;
    if (current_sm_count(&sms) != PKV_OK) return 0;
    return workspace_bytes_for(num_seqs, num_kv_heads, num_q_heads / num_kv_heads, head_dim, sms * kDecodeWarps);
}

extern "C" int pkv_paged_decode_attention(void *out, const void *q, const void *k_cache, const void *v_cache,
                                          const int32_t *block_tables, int max_blocks_per_seq,
                                          const int32_t *context_lens, int num_seqs, int num_blocks,
                                          int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                          float scale, int dtype, int out_dtype, void *workspace,
                                          size_t workspace_bytes, int *dev_status, void *stream) {
    using namespace pkv;
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
    if (num_seqs == 0) return PKV_OK;
    if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens || !workspace)
        return PKV_ERR_INVALID_ARG;
    if (!aligned(q, 4) || !aligned(out, 4) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
        !aligned(block_tables, 4) || !aligned(context_lens, 4))
        return PKV_ERR_INVALID_ARG;
    if (!aligned(workspace, 16)) return PKV_ERR_WORKSPACE;
    int sms = 0;
    int rc = current_sm_count(&sms);
    if (rc != PKV_OK) return rc;
    // enough warps for the largest possible total, at most one CTA per SM
    const int64_t upper = (int64_t)num_seqs * num_kv_heads * max_blocks_per_seq;
    int grid = (int)((upper + kDecodeWarps - 1) / kDecodeWarps);
    if (grid > sms) grid = sms;
    if (grid < 1) grid = 1;
    const int total_warps = grid * kDecodeWarps;
    if (workspace_bytes < workspace_bytes_for(num_seqs, num_kv_heads, G, head_dim, total_warps))
        return PKV_ERR_WORKSPACE;

    CUtensorMap tk, tv;
    rc = encode_cache_map(&tk, k_cache, num_blocks, num_kv_heads, block_size, head_dim);
    if (rc != PKV_OK) return rc;
    rc = encode_cache_map(&tv, v_cache, num_blocks, num_kv_heads, block_size, head_dim);
    if (rc != PKV_OK) return rc;

    DecodeParams prm;
    prm.out = out;
    prm.q = q;
    prm.block_tables = block_tables;
    prm.context_lens = context_lens;
    prm.arrivals = static_cast<unsigned long long *>(workspace);
    prm.part = reinterpret_cast<float *>(static_cast<char *>(workspace) + arrivals_bytes(num_seqs, num_kv_heads));
    prm.dev_status = dev_status;
    prm.S = num_seqs;
    prm.max_blocks = max_blocks_per_seq;
    prm.num_blocks = num_blocks;
    prm.Hq = num_q_heads;
    prm.Hkv = num_kv_heads;
    prm.G = G;
    prm.scale_log2 = scale * 1.4426950408889634f;
    prm.out_dtype = out_dtype;
    prm.total_warps = total_warps;
    prm.epoch = next_epoch();
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const bool wide = G > 8;
    if (dtype == PKV_DTYPE_BF16) {
        if (head_dim == 128)
            return wide ? launch_decode<__nv_bfloat16, 128, 2>(prm, tk, tv, grid, st)
                        : launch_decode<__nv_bfloat16, 128, 1>(prm, tk, tv, grid, st);
        return wide ? launch_decode<__nv_bfloat16, 64, 2>(prm, tk, tv, grid, st)
                    : launch_decode<__nv_bfloat16, 64, 1>(prm, tk, tv, grid, st);
    }
    if (head_dim == 128)
        return wide ? launch_decode<__half, 128, 2>(prm, tk, tv, grid, st)
                    : launch_decode<__half, 128, 1>(prm, tk, tv, grid, st);
    return wide ? launch_decode<__half, 64, 2>(prm, tk, tv, grid, st)
                : launch_decode<__half, 64, 1>(prm, tk, tv, grid, st);
}
