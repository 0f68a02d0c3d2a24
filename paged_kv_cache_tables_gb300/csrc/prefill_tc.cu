// K4 on the 5th-generation tensor cores: paged prefill attention for chunked
// prefill with tcgen05.mma, accumulators and the probability tile in tensor
// memory.
//
// What is computed: "Continuous Batching" (infra.pidoku.co.in) §5 "Mixed
// batching (prefill + decode in one step)": chunk c's query row i sits at
// position ctx_c - q_len_c + i and attends every key at or before it, the
// keys and values gathered through the sequence's block table ("Project 17",
// Step 6).
//
// One CTA per (chunk, pair of query tiles, KV head).  A query tile is 128 MMA
// rows = 128 / G tokens x the G query heads that share the KV head
// (row = token * G + head), so each K/V tile feeds the whole group; the two
// tiles of a pair (adjacent tokens) share every K/V tile.  Warp roles:
//   warp 0     TMA: both query tiles once (3-D boxes, 128-byte swizzle), then
//              K and V tiles of 128 keys = 8 pages of 16 through the block
//              table (ids read one tile ahead) into 2-stage K and V rings
//              with their own barriers: a K slot frees after the second
//              Q.K^T of its tile, a V slot after the second P.V;
//   warp 1     allocates all 512 tensor-memory columns (S and O of each tile)
//              and issues every MMA from one thread, ping-ponging the tiles:
//              O_A += P_A V_j, S_A = Q_A K_{j+1}^T, O_B += P_B V_j,
//              S_B = Q_B K_{j+1}^T, ...;
//   warps 2-3  idle (they complete the first warpgroup, whose register
//              budget drops so that the softmax warpgroups can grow);
//   warps 4-7  softmax of tile A, warps 8-11 of tile B, one row per thread (the
//              tensor-memory lane of the row): one pass over S held in
//              registers (causal mask on diagonal tiles only, running max in
//              base 2 with lazy rescaling of O when the max grows by more
//              than 2^8, packed fp32x2 arithmetic), then P written back over S as
//              16-bit (rounded value, rounding residual) pairs, which the MMA
//              reads as its A operand straight from tensor memory.
// While one tile's softmax runs, the tensor core works on the other tile.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdio>

#include "pkv.h"
#include "pkv_device.cuh"
#include "pkv_host.h"
#include "pkv_tc.cuh"

namespace pkv {

constexpr int kTcThreads = 384;
// registers per thread: the launch gives every thread kTcLaunchRegs; the
// TMA/MMA warpgroup then drops to kTcLowRegs and the two softmax warpgroups
// rise to kTcHighRegs, which must not exceed what the drop frees
constexpr int kTcLaunchRegs = 168;
constexpr int kTcLowRegs = 88;
constexpr int kTcHighRegs = 208;
static_assert(128 * kTcLowRegs + 256 * kTcHighRegs <= kTcThreads * kTcLaunchRegs, "register split");
constexpr int kTcRows = 128;    // MMA rows = (token, head) pairs per query tile
constexpr int kTcKeys = 128;    // keys per K/V tile
constexpr int kTcStages = 2;
constexpr uint64_t kTcWaitNs = 2000000000ull;
constexpr uint32_t kTmemCols = 512;   // tile t: S/P at 256 t, O at 256 t + 128

struct PrefillTcParams {
    void *out;
    const int32_t *cu_seqlens;
    const int32_t *block_tables;
    const int32_t *context_lens;
    int *dev_status;
    int S, max_blocks, num_blocks, Hq, Hkv, G;
    int rtok, pairs_per_seq;
    float scale_log2;
    int out_dtype;
};

template <int D>
struct TcShape {
    static constexpr int HALVES = D / 64;
    static constexpr int Q_HALF = kTcRows * 128;            // 128 rows x 64 columns
    static constexpr int Q_BYTES = HALVES * Q_HALF;
    static constexpr int KV_HALF = kTcKeys * 128;           // 128 keys x 64 columns
    static constexpr int K_BYTES = HALVES * KV_HALF;
    static constexpr int STAGE_BYTES = 2 * K_BYTES;         // K then V
    static constexpr int OFF_Q = 0;                         // tile A, then tile B
    static constexpr int OFF_KV = 2 * Q_BYTES;
    static constexpr int OFF_BAR = OFF_KV + kTcStages * STAGE_BYTES;
    static constexpr int SMEM_BYTES = 1024 + OFF_BAR + 256;
};

template <typename T, int D>
__global__ void __launch_bounds__(kTcThreads, 1)
    paged_prefill_tc_kernel(const PrefillTcParams p, const __grid_constant__ CUtensorMap tk,
                            const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tq) {
    using Sh = TcShape<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + Sh::OFF_BAR);
    uint64_t *q_full = bars + 0;
    uint64_t *k_full = bars + 1;      // [stage]
    uint64_t *v_full = bars + 3;      // [stage]
    uint64_t *k_empty = bars + 5;     // [stage]
    uint64_t *v_empty = bars + 7;     // [stage]
    uint64_t *s_full = bars + 9;      // [tile]
    uint64_t *p_full = bars + 11;     // [tile]
    uint64_t *o_done = bars + 13;     // [tile]
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 15);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int Hkv = p.Hkv, G = p.G;
    // inputs may come from the previous kernel on the stream (the append)
    pdl_wait_primary();
    pdl_launch_dependents();
    // CTAs in launch order: chunk by chunk, and within a chunk its last tile
    // pair (the most keys) first.  The pairs of one chunk read the same
    // context pages, so running them side by side serves the repeats from L2.
    const int h = blockIdx.x % Hkv;
    const int rest = blockIdx.x / Hkv;
    const int pair = p.pairs_per_seq - 1 - rest % p.pairs_per_seq;
    const int c = rest / p.pairs_per_seq;
    const int q0 = __ldg(p.cu_seqlens + c);
    const int q_len = __ldg(p.cu_seqlens + c + 1) - q0;
    const int ctx = __ldg(p.context_lens + c);
    if (q_len < 0 || q_len > ctx) {
        if (tid == 0 && pair == 0) set_status(p.dev_status, PKV_DEV_BAD_CHUNK);
        return;
    }
    if (ctx > p.max_blocks * 16) {
        if (tid == 0 && pair == 0) set_status(p.dev_status, PKV_DEV_BAD_CONTEXT);
        return;
    }
    const int i0 = pair * 2 * p.rtok;
    if (i0 >= q_len) return;
    const int ntok = min(2 * p.rtok, q_len - i0);      // tokens of this pair (tile A first)
    const int prior = ctx - q_len;
    const int ntiles = (prior + i0 + ntok - 1) / kTcKeys + 1;
    const int nblk = (ctx + 15) / 16;

    if (tid == 0) {
        mbar_init(q_full, 1);
        for (int s = 0; s < kTcStages; ++s) {
            mbar_init(&k_full[s], 1);
            mbar_init(&v_full[s], 1);
            mbar_init(&k_empty[s], 1);
            mbar_init(&v_empty[s], 1);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(&s_full[t], 1);
            mbar_init(&p_full[t], 128);
            mbar_init(&o_done[t], 1);
        }
        fence_mbar_init();
    }
    if (warp == 1) {
        tc::tmem_alloc(tmem_slot, kTmemCols);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const uint32_t sbase = smem_addr(sm);

    if (warp < 4) {
      tc::setmaxnreg_dec<kTcLowRegs>();
      if (warp == 0) {
        // ---------------- TMA producer ----------------
        // lane 0 issues the copies; lanes 0-7 read the block ids of the next
        // tile's eight pages one tile ahead, so no table read sits between
        // a slot becoming free and its copies starting
        constexpr int kPages = kTcKeys / 16;
        const int32_t *row = p.block_tables + (int64_t)c * p.max_blocks;
        auto in_context = [&](int jt) { return lane < kPages && jt * kPages + lane < nblk; };
        auto fetch = [&](int jt) { return in_context(jt) ? __ldg(row + jt * kPages + lane) : 0; };
        int blk_next = fetch(0);
        if (lane == 0) {
            const int qrows = G * p.rtok;
            mbar_arrive_expect_tx(q_full, (uint32_t)(2 * Sh::HALVES * qrows * 128));
#pragma unroll
            for (int t = 0; t < 2; ++t)
#pragma unroll
                for (int hf = 0; hf < Sh::HALVES; ++hf)
                    tc::tma_load_3d(sm + Sh::OFF_Q + t * Sh::Q_BYTES + hf * Sh::Q_HALF, &tq, hf * 64, h * G,
                                    q0 + i0 + t * p.rtok, q_full);
        }
        const uint64_t policy = l2_policy_evict_first();
        for (int j = 0; j < ntiles; ++j) {
            const int blk = blk_next;
            if (j + 1 < ntiles) blk_next = fetch(j + 1);
            int y = p.num_blocks * Hkv * 16;               // past the pool: zero fill
            if (in_context(j)) {
                if (blk >= 0 && blk < p.num_blocks)
                    y = (blk * Hkv + h) * 16;
                else
                    set_status(p.dev_status, PKV_DEV_BAD_BLOCK_ID);
            }
            int ys[kPages];
#pragma unroll
            for (int pg = 0; pg < kPages; ++pg) ys[pg] = __shfl_sync(0xffffffffu, y, pg);
            const int st = j % kTcStages;
            const uint32_t par = (uint32_t)(((j - kTcStages) / kTcStages) & 1);
            bool ok = true;
            if (lane == 0) {
                // K of tile j - 2 is free once both S products of that tile are done
                if (j >= kTcStages) ok = mbar_wait(&k_empty[st], par, kTcWaitNs);
                if (ok) {
                    mbar_arrive_expect_tx(&k_full[st], Sh::K_BYTES);
                    uint8_t *kd = sm + Sh::OFF_KV + st * Sh::STAGE_BYTES;
#pragma unroll
                    for (int pg = 0; pg < kPages; ++pg)
#pragma unroll
                        for (int hf = 0; hf < Sh::HALVES; ++hf)
                            tma_load_2d(kd + hf * Sh::KV_HALF + pg * 2048, &tk, hf * 64, ys[pg], &k_full[st], policy);
                }
                // V of tile j - 2 is free once both P.V products of that tile are done
                if (ok && j >= kTcStages) ok = mbar_wait(&v_empty[st], par, kTcWaitNs);
                if (ok) {
                    mbar_arrive_expect_tx(&v_full[st], Sh::K_BYTES);
                    uint8_t *vd = sm + Sh::OFF_KV + st * Sh::STAGE_BYTES + Sh::K_BYTES;
#pragma unroll
                    for (int pg = 0; pg < kPages; ++pg)
#pragma unroll
                        for (int hf = 0; hf < Sh::HALVES; ++hf)
                            tma_load_2d(vd + hf * Sh::KV_HALF + pg * 2048, &tv, hf * 64, ys[pg], &v_full[st], policy);
                }
                if (!ok) set_status(p.dev_status, PKV_DEV_WAIT_TIMEOUT);
            }
            if (!__shfl_sync(0xffffffffu, ok, 0)) break;
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        // The whole warp walks the schedule, so the waits and the descriptor
        // arithmetic are warp-uniform; one elected lane issues each MMA and
        // commit.  Shared-memory descriptors are built once and moved by
        // adding (byte offset >> 4) to their address field: every operand
        // lies below 256 KB, so the 14-bit field never carries.
        const bool leader = tc::elect_one();
        constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
        constexpr uint32_t idesc_s = tc::idesc_f16(kBf16, false, false, kTcRows, kTcKeys);
        constexpr uint32_t idesc_o = tc::idesc_f16(kBf16, false, true, kTcRows, D);
        const uint64_t q_desc = tc::smem_desc_sw128(sbase + Sh::OFF_Q, 16, 1024);
        const uint64_t k_desc = tc::smem_desc_sw128(sbase + Sh::OFF_KV, 16, 1024);
        const uint64_t v_desc = tc::smem_desc_sw128(sbase + Sh::OFF_KV + Sh::K_BYTES, Sh::KV_HALF, 1024);
        auto issue_s = [&](int j, int t) {   // S_t = Q_t K_j^T
            const uint64_t kb = k_desc + (uint64_t)(((j % kTcStages) * Sh::STAGE_BYTES) >> 4);
            const uint64_t qb = q_desc + (uint64_t)((t * Sh::Q_BYTES) >> 4);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t qo = ((kk >> 2) * Sh::Q_HALF + (kk & 3) * 32) >> 4;
                const uint32_t ko = ((kk >> 2) * Sh::KV_HALF + (kk & 3) * 32) >> 4;
                if (leader) tc::mma_f16_ss(tmem + t * 256, qb + qo, kb + ko, idesc_s, kk > 0);
            }
            if (leader) tc::mma_commit(&s_full[t]);
        };
        auto issue_pv = [&](int j, int t) {   // O_t += P_t V_j, P_t from tensor memory
            const uint64_t vb = v_desc + (uint64_t)(((j % kTcStages) * Sh::STAGE_BYTES) >> 4);
#pragma unroll
            for (int kk = 0; kk < kTcKeys / 16; ++kk) {
                const uint32_t ph = tmem + t * 256 + 32 * (kk >> 1) + 8 * (kk & 1);
                if (leader) {
                    tc::mma_f16_ts(tmem + t * 256 + 128, ph, vb + (uint32_t)(kk * 2048 >> 4), idesc_o, j > 0 || kk > 0);
                    tc::mma_f16_ts(tmem + t * 256 + 128, ph + 16, vb + (uint32_t)(kk * 2048 >> 4), idesc_o, true);
                }
            }
            if (leader) tc::mma_commit(&o_done[t]);
        };
        auto wait_all = [&](uint64_t *bar, uint32_t parity) {
            return __all_sync(0xffffffffu, mbar_wait(bar, parity, kTcWaitNs));
        };
        bool ok = wait_all(q_full, 0) && wait_all(&k_full[0], 0);
        if (ok) {
            tc::fence_after_sync();
            issue_s(0, 0);
            issue_s(0, 1);
            if (leader) tc::mma_commit(&k_empty[0]);
        }
        for (int j = 0; ok && j < ntiles; ++j) {
            const bool more = j + 1 < ntiles;
            ok = wait_all(&p_full[0], (uint32_t)(j & 1)) &&
                 wait_all(&v_full[j % kTcStages], (uint32_t)((j / kTcStages) & 1));
            if (!ok) break;
            tc::fence_after_sync();
            issue_pv(j, 0);
            if (more) {
                ok = wait_all(&k_full[(j + 1) % kTcStages], (uint32_t)(((j + 1) / kTcStages) & 1));
                if (!ok) break;
                tc::fence_after_sync();
                issue_s(j + 1, 0);
            }
            ok = wait_all(&p_full[1], (uint32_t)(j & 1));
            if (!ok) break;
            tc::fence_after_sync();
            issue_pv(j, 1);
            if (leader) tc::mma_commit(&v_empty[j % kTcStages]);
            if (more) {
                issue_s(j + 1, 1);
                if (leader) tc::mma_commit(&k_empty[(j + 1) % kTcStages]);
            }
        }
        if (!ok && leader) set_status(p.dev_status, PKV_DEV_WAIT_TIMEOUT);
      }
    } else {
        tc::setmaxnreg_inc<kTcHighRegs>();
        // ---------------- softmax: tile t, one row per thread ----------------
        const int t = (warp - 4) >> 2;
        const int lane_base = 32 * (warp & 3);          // tensor-memory lanes this warp may touch
        const int r = lane_base + lane;                 // row within the tile
        const int tok = t * p.rtok + r / G, head = r % G;
        const bool valid = r < G * p.rtok && tok < ntok;
        const int pos = valid ? prior + i0 + tok : ctx - 1;   // padding rows see every key
        const uint32_t trow = tmem + ((uint32_t)lane_base << 16) + t * 256;
        float m_used = -INFINITY, l = 0.f;
        const uint64_t scale2 = f2_pack(p.scale_log2, p.scale_log2);
        bool ok = true;
        for (int j = 0; j < ntiles; ++j) {
            ok = mbar_wait(&s_full[t], (uint32_t)(j & 1), kTcWaitNs);
            if (!__all_sync(0xffffffffu, ok)) {
                ok = false;
                break;
            }
            tc::fence_after_sync();
            const int key0 = j * kTcKeys;
            // one pass: the whole row of 128 scores in registers
            float v[kTcKeys];
#pragma unroll
            for (int cc = 0; cc < kTcKeys / 32; ++cc)
                tc::tmem_ld32(trow + cc * 32, *reinterpret_cast<float(*)[32]>(v + cc * 32));
            tc::tmem_wait_ld();
            // causal mask, only on tiles that reach past some row's position
            const int lim = pos - key0;
            if (__any_sync(0xffffffffu, lim < kTcKeys - 1)) {
#pragma unroll
                for (int e = 0; e < kTcKeys; ++e)
                    if (e > lim) v[e] = -INFINITY;
            }
            // four independent chains of 3-input maxima over the 124 scores
            // after the first four
            float mx4[4] = {v[0], v[1], v[2], v[3]};
#pragma unroll
            for (int pr = 0; pr < (kTcKeys - 4) / 2; ++pr)
                mx4[pr & 3] = fmax3(mx4[pr & 3], v[4 + 2 * pr], v[5 + 2 * pr]);
            // scale_log2 > 0, so the scaled maximum is the maximum scaled
            const float mx = fmax3(fmaxf(mx4[0], mx4[1]), mx4[2], mx4[3]) * p.scale_log2;
            const bool first = m_used == -INFINITY;
            const float m_new = fmaxf(m_used, mx);
            const bool rescale = !first && m_new > m_used + 8.f;
            const float alpha = rescale ? exp2_approx(m_used - m_new) : 1.f;
            if (first || rescale) m_used = m_new;
            // O was last written by P_t V_{j-1}, which the tensor core finished
            // before S_t = Q_t K_j^T (issued after it) completed
            if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll 1
                for (int cc = 0; cc < D / 32; ++cc) {
                    float o[32];
                    tc::tmem_ld32(trow + 128 + cc * 32, o);
                    tc::tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] *= alpha;
                    tc::tmem_st32(trow + 128 + cc * 32, o);
                }
            }
            // P = 2^(x - m_used) over the same columns, 32 keys at a time: 16
            // columns of rounded pairs, then 16 of residual pairs
            const uint64_t negm2 = f2_pack(-m_used, -m_used);
            uint64_t sum2[2] = {f2_pack(0.f, 0.f), f2_pack(0.f, 0.f)};
#pragma unroll
            for (int cc = 0; cc < kTcKeys / 32; ++cc) {
                float w[32];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    float a, b;
                    f2_unpack(f2_fma(f2_pack(v[32 * cc + 2 * e], v[32 * cc + 2 * e + 1]), scale2, negm2), a, b);
                    a = exp2_approx(a);
                    b = exp2_approx(b);
                    const uint64_t ab = f2_pack(a, b);
                    sum2[e & 1] = f2_add(sum2[e & 1], ab);
                    uint32_t hi, lo;
                    pack2_split2<T>(ab, a, b, hi, lo);
                    w[e] = __uint_as_float(hi);
                    w[16 + e] = __uint_as_float(lo);
                }
                tc::tmem_st32(trow + cc * 32, w);
            }
            float s0, s1, s2, s3;
            f2_unpack(sum2[0], s0, s1);
            f2_unpack(sum2[1], s2, s3);
            l = l * alpha + ((s0 + s1) + (s2 + s3));
            // keys at or past the context in the last stored page may hold
            // anything: clear those V rows so 0 x garbage cannot reach O
            // (both tiles' warps write the same zeros before their product)
            const int zlo = max(ctx - key0, 0), zhi = min(kTcKeys, nblk * 16 - key0);
            if (zlo < zhi) {
                // V_j cannot be reloaded before this tile's P.V products,
                // so the phase waited for here is this tile's
                ok = mbar_wait(&v_full[j % kTcStages], (uint32_t)((j / kTcStages) & 1), kTcWaitNs);
                if (!__all_sync(0xffffffffu, ok)) {
                    ok = false;
                    break;
                }
                if (r >= zlo && r < zhi) {
                    uint8_t *vrow = sm + Sh::OFF_KV + (j % kTcStages) * Sh::STAGE_BYTES + Sh::K_BYTES + r * 128;
#pragma unroll
                    for (int hf = 0; hf < Sh::HALVES; ++hf)
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            *reinterpret_cast<uint4 *>(vrow + hf * Sh::KV_HALF + e * 16) =
                                make_uint4(0u, 0u, 0u, 0u);
                }
                fence_proxy_async_smem();
            }
            tc::tmem_wait_st();
            tc::fence_before_sync();
            tc::mbar_arrive_cta(&p_full[t]);
        }
        if (ok) {
            ok = mbar_wait(&o_done[t], (uint32_t)((ntiles - 1) & 1), kTcWaitNs);
            ok = __all_sync(0xffffffffu, ok);
        }
        if (ok) {
            tc::fence_after_sync();
            const float inv = 1.f / l;
            const int64_t ob = ((int64_t)(q0 + i0 + tok) * p.Hq + (int64_t)h * G + head) * D;
#pragma unroll 1
            for (int cc = 0; cc < D / 32; ++cc) {
                float v[32];
                tc::tmem_ld32(trow + 128 + cc * 32, v);
                tc::tmem_wait_ld();
                if (valid) {
                    if (p.out_dtype == PKV_DTYPE_F32) {
                        float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(p.out) + ob + cc * 32);
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            dst[e] = make_float4(v[4 * e] * inv, v[4 * e + 1] * inv, v[4 * e + 2] * inv,
                                                 v[4 * e + 3] * inv);
                    } else {
                        uint4 *dst = reinterpret_cast<uint4 *>(static_cast<T *>(p.out) + ob + cc * 32);
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            dst[e] = make_uint4(pack2<T>(v[8 * e] * inv, v[8 * e + 1] * inv),
                                                pack2<T>(v[8 * e + 2] * inv, v[8 * e + 3] * inv),
                                                pack2<T>(v[8 * e + 4] * inv, v[8 * e + 5] * inv),
                                                pack2<T>(v[8 * e + 6] * inv, v[8 * e + 7] * inv));
                    }
                }
            }
        } else {
            set_status(p.dev_status, PKV_DEV_WAIT_TIMEOUT);
        }
    }

    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
}

// 3-D TMA descriptor over q viewed as [total_q][Hq][head_dim]: box of 64
// columns x G heads x rtok tokens, 128-byte swizzle; rows past total_q read 0.
static int encode_q_map(CUtensorMap *map, const void *q, int total_q, int Hq, int head_dim, int G, int rtok) {
    const uint64_t dims[3] = {(uint64_t)head_dim, (uint64_t)Hq, (uint64_t)total_q};
    const uint64_t strides[2] = {(uint64_t)head_dim * 2, (uint64_t)Hq * head_dim * 2};
    const uint32_t box[3] = {64, (uint32_t)G, (uint32_t)rtok};
    return encode_tiled_map(map, q, 3, dims, strides, box);
}

template <typename T, int D>
int launch_prefill_tc(const PrefillTcParams &prm, const CUtensorMap &tk, const CUtensorMap &tv,
                      const CUtensorMap &tq, int grid, cudaStream_t stream) {
    using Sh = TcShape<D>;
    // the register split inside the kernel waits for registers that only
    // exist if the compiled count is the one it was sized for: check it
    // (once; the answer does not change) and refuse to launch otherwise
    static int regs_ok = 0;   // 0 unknown, 1 as sized, -1 not
    if (regs_ok == 0) {
        cudaFuncAttributes fa;
        cudaError_t e = cudaFuncGetAttributes(&fa, paged_prefill_tc_kernel<T, D>);
        if (e != cudaSuccess) return cuda_fail(e);
        regs_ok = fa.numRegs == kTcLaunchRegs ? 1 : -1;
        if (regs_ok < 0) {
            char msg[128];
            std::snprintf(msg, sizeof msg, "prefill kernel compiled to %d registers per thread, its split needs %d",
                          fa.numRegs, kTcLaunchRegs);
            set_error_message(msg);
        }
    }
    if (regs_ok < 0) return PKV_ERR_UNSUPPORTED;
    static unsigned long long attr_set = 0;   // per instantiation and device
    if (!done_on_device(&attr_set)) {
        cudaError_t e = cudaFuncSetAttribute(paged_prefill_tc_kernel<T, D>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, Sh::SMEM_BYTES);
        if (e != cudaSuccess) return cuda_fail(e);
        mark_done_on_device(&attr_set);
    }
    cudaError_t e = launch_pdl(paged_prefill_tc_kernel<T, D>, dim3(grid), dim3(kTcThreads), Sh::SMEM_BYTES, stream,
                               prm, tk, tv, tq);
    if (e == cudaSuccess) e = cudaGetLastError();
    return e == cudaSuccess ? PKV_OK : cuda_fail(e);
}

int prefill_tc(void *out, const void *q, const int32_t *cu_seqlens, int num_seqs, int max_q_len, int total_q,
               const void *k_cache, const void *v_cache, const int32_t *block_tables, int max_blocks_per_seq,
               const int32_t *context_lens, int num_blocks, int Hq, int Hkv, int head_dim, float scale, int dtype,
               int out_dtype, int *dev_status, cudaStream_t stream) {
    const int G = Hq / Hkv;
    const int rtok = kTcRows / G;
    const int pairs = (max_q_len + 2 * rtok - 1) / (2 * rtok);
    const int64_t grid64 = (int64_t)num_seqs * pairs * Hkv;
    if (grid64 >= ((int64_t)1 << 31)) return PKV_ERR_UNSUPPORTED;
    if (!aligned(out, 16)) return PKV_ERR_INVALID_ARG;
    CUtensorMap tk, tv, tq;
    int rc = encode_cache_map(&tk, k_cache, num_blocks, Hkv, 16, head_dim);
    if (rc != PKV_OK) return rc;
    rc = encode_cache_map(&tv, v_cache, num_blocks, Hkv, 16, head_dim);
    if (rc != PKV_OK) return rc;
    rc = encode_q_map(&tq, q, total_q, Hq, head_dim, G, rtok);
    if (rc != PKV_OK) return rc;
    PrefillTcParams prm;
    prm.out = out;
    prm.cu_seqlens = cu_seqlens;
    prm.block_tables = block_tables;
    prm.context_lens = context_lens;
    prm.dev_status = dev_status;
    prm.S = num_seqs;
    prm.max_blocks = max_blocks_per_seq;
    prm.num_blocks = num_blocks;
    prm.Hq = Hq;
    prm.Hkv = Hkv;
    prm.G = G;
    prm.rtok = rtok;
    prm.pairs_per_seq = pairs;
    prm.scale_log2 = scale * 1.4426950408889634f;
    prm.out_dtype = out_dtype;
    const int grid = (int)grid64;
    if (dtype == PKV_DTYPE_BF16)
        return head_dim == 128 ? launch_prefill_tc<__nv_bfloat16, 128>(prm, tk, tv, tq, grid, stream)
                               : launch_prefill_tc<__nv_bfloat16, 64>(prm, tk, tv, tq, grid, stream);
    return head_dim == 128 ? launch_prefill_tc<__half, 128>(prm, tk, tv, tq, grid, stream)
                           : launch_prefill_tc<__half, 64>(prm, tk, tv, tq, grid, stream);
}

}  // namespace pkv
