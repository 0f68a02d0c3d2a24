// K4: paged prefill attention for chunked prefill (varlen chunks, causal over
// prior context plus the chunk).
//
// What is computed: "Continuous Batching" (infra.pidoku.co.in) §5 "Mixed
// batching (prefill + decode in one step)": a prompt is processed in chunks
// that ride with the decode step; chunk c's query row i sits at position
// ctx_c - q_len_c + i and attends every key at or before that position,
// gathered through the sequence's block table ("Project 17", Step 6).
//
// How: one CTA per (chunk, tile of 128 / G query tokens, KV head).  The G
// query heads that share the KV head are packed into the MMA rows (row =
// token * G + head), so every K/V page is used by the whole group.  A producer
// warp streams the 16-token pages 0 .. last needed page through an 8-slot
// TMA ring (full/empty mbarriers); eight consumer warps each own 16 rows and
// run S = Q K^T and O += P V with mma.m16n8k16, an online base-2 softmax in
// fp32, and P fed as a rounded 16-bit value plus its rounding residual.
#include <cuda_runtime.h>

#include <cmath>

#include "pkv.h"
#include "pkv_device.cuh"
#include "pkv_host.h"

namespace pkv {

constexpr int kPfWarps = 8;                        // consumer warps
constexpr int kPfThreads = (kPfWarps + 1) * 32;    // + one producer warp
constexpr int kPfRows = kPfWarps * 16;             // (token, head) rows per CTA
constexpr int kPfStages = 8;
constexpr uint64_t kPfWaitLimitNs = 2000000000ull;

struct PrefillParams {
    void *out;
    const void *q;
    const int32_t *cu_seqlens;
    const int32_t *block_tables;
    const int32_t *context_lens;
    int *dev_status;
    int S, max_blocks, num_blocks, Hq, Hkv, G;
    int rtok;             // query tokens per CTA = kPfRows / G
    int tiles_per_seq;    // ceil(max_q_len / rtok)
    float scale_log2;
    int out_dtype;
};

template <int D>
struct PrefillShape {
    static constexpr int HALVES = D / 64;
    static constexpr int HALF_BYTES = 64 * 16 * 2;
    static constexpr int TILE_BYTES = HALVES * HALF_BYTES;
    static constexpr int STAGE_BYTES = 2 * TILE_BYTES;
    static constexpr int RING_BYTES = kPfStages * STAGE_BYTES;
    static constexpr int SMEM_BYTES = 1024 + RING_BYTES + 2 * kPfStages * 8;
};

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

template <typename T, int D>
__global__ void __launch_bounds__(kPfThreads, 1)
    paged_prefill_kernel(const PrefillParams p, const __grid_constant__ CUtensorMap tk,
                         const __grid_constant__ CUtensorMap tv) {
    using Sh = PrefillShape<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *ring = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(ring + Sh::RING_BYTES);
    uint64_t *empty = full + kPfStages;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int Hkv = p.Hkv, G = p.G;
    // work item; the last tiles of a chunk (the most keys) get the lowest ids
    const int h = blockIdx.x % Hkv;
    const int rest = blockIdx.x / Hkv;
    const int tile = p.tiles_per_seq - 1 - rest % p.tiles_per_seq;
    const int c = rest / p.tiles_per_seq;
    const int q0 = __ldg(p.cu_seqlens + c);
    const int q_len = __ldg(p.cu_seqlens + c + 1) - q0;
    const int ctx = __ldg(p.context_lens + c);
    if (q_len < 0 || q_len > ctx) {
        if (tid == 0 && tile == 0) set_status(p.dev_status, PKV_DEV_BAD_CHUNK);
        return;
    }
    if (ctx > p.max_blocks * 16) {
        if (tid == 0 && tile == 0) set_status(p.dev_status, PKV_DEV_BAD_CONTEXT);
        return;
    }
    const int i0 = tile * p.rtok;
    if (i0 >= q_len) return;
    const int ntok = min(p.rtok, q_len - i0);
    const int prior = ctx - q_len;
    const int npages = (prior + i0 + ntok - 1) / 16 + 1;

    if (tid == 0) {
        for (int s = 0; s < kPfStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kPfWarps);
        }
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == kPfWarps) {
        // ---------------- producer ----------------
        if (lane == 0) {
            const uint64_t policy = l2_policy_evict_first();
            const int32_t *row = p.block_tables + (int64_t)c * p.max_blocks;
            for (int pg = 0; pg < npages; ++pg) {
                const int st = pg % kPfStages;
                if (pg >= kPfStages) {
                    if (!mbar_wait(&empty[st], (uint32_t)(((pg / kPfStages) + 1) & 1), kPfWaitLimitNs)) {
                        set_status(p.dev_status, PKV_DEV_WAIT_TIMEOUT);
                        return;
                    }
                }
                int blk = __ldg(row + pg);
                int y = (blk * Hkv + h) * 16;
                if (blk < 0 || blk >= p.num_blocks) {
                    set_status(p.dev_status, PKV_DEV_BAD_BLOCK_ID);
                    y = p.num_blocks * Hkv * 16;
                }
                mbar_arrive_expect_tx(&full[st], Sh::STAGE_BYTES);
                uint8_t *kd = ring + st * Sh::STAGE_BYTES;
#pragma unroll
                for (int hf = 0; hf < Sh::HALVES; ++hf) {
                    tma_load_2d(kd + hf * Sh::HALF_BYTES, &tk, hf * 64, y, &full[st], policy);
                    tma_load_2d(kd + Sh::TILE_BYTES + hf * Sh::HALF_BYTES, &tv, hf * 64, y, &full[st], policy);
                }
            }
        }
        return;
    }

    // ---------------- consumers ----------------
    const int g = lane >> 2, t4 = lane & 3, mi = lane >> 3;
    const int ra = warp * 16 + g, rb = ra + 8;          // CTA rows held by this lane
    const int tok_a = ra / G, head_a = ra - tok_a * G;
    const int tok_b = rb / G, head_b = rb - tok_b * G;
    const bool va = tok_a < ntok, vb = tok_b < ntok;
    // padding rows see every key so their (discarded) state stays finite
    const int pos_a = va ? prior + i0 + tok_a : ctx - 1;
    const int pos_b = vb ? prior + i0 + tok_b : ctx - 1;
    const int warp_tok_lo = (warp * 16) / G;
    const bool warp_has_rows = warp_tok_lo < ntok;
    const int warp_tok_hi = min(ntok - 1, (warp * 16 + 15) / G);
    const int warp_max_pos = prior + i0 + warp_tok_hi;

    uint32_t qa[D / 16][4];
    {
        const uint32_t *qra = reinterpret_cast<const uint32_t *>(
            static_cast<const T *>(p.q) + ((int64_t)(q0 + i0 + tok_a) * p.Hq + h * G + head_a) * D);
        const uint32_t *qrb = reinterpret_cast<const uint32_t *>(
            static_cast<const T *>(p.q) + ((int64_t)(q0 + i0 + tok_b) * p.Hq + h * G + head_b) * D);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            const int c0 = kk * 8 + t4;
            qa[kk][0] = va ? __ldg(qra + c0) : 0u;
            qa[kk][2] = va ? __ldg(qra + c0 + 4) : 0u;
            qa[kk][1] = vb ? __ldg(qrb + c0) : 0u;
            qa[kk][3] = vb ? __ldg(qrb + c0 + 4) : 0u;
        }
    }
    float o[D / 8][4];
#pragma unroll
    for (int nt = 0; nt < D / 8; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) o[nt][e] = 0.f;
    float m_a = -INFINITY, m_b = -INFINITY, l_a = 0.f, l_b = 0.f;

    const uint32_t ring_addr = smem_addr(ring);
    const int k_row = ((mi >> 1) << 3) + (lane & 7);   // ldmatrix row for K (non-transposed)
    const int v_row = ((mi & 1) << 3) + (lane & 7);    // ldmatrix row for V (transposed)

    for (int pg = 0; pg < npages; ++pg) {
        const int st = pg % kPfStages;
        const bool landed = mbar_wait(&full[st], (uint32_t)((pg / kPfStages) & 1), kPfWaitLimitNs);
        if (!__all_sync(0xffffffffu, landed)) {
            set_status(p.dev_status, PKV_DEV_WAIT_TIMEOUT);
            return;
        }
        const int key0 = pg * 16;
        if (warp_has_rows && key0 <= warp_max_pos) {
            const uint32_t kbase = ring_addr + st * Sh::STAGE_BYTES;
            const uint32_t vbase = kbase + Sh::TILE_BYTES;
            float s[2][4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) s[nt][e] = 0.f;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const int chunk = ((kk & 3) << 1) + (mi & 1);
                const uint32_t addr = kbase + (kk >> 2) * Sh::HALF_BYTES + k_row * 128 + ((chunk ^ (k_row & 7)) << 4);
                uint32_t b00, b01, b10, b11;
                ldsm_x4(addr, b00, b01, b10, b11);
                mma_16816<T>(s[0], qa[kk], b00, b01);
                mma_16816<T>(s[1], qa[kk], b10, b11);
            }
            // causal mask and online softmax; rows a (regs 0,1) and b (regs 2,3)
            float mx_a = -INFINITY, mx_b = -INFINITY;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int key = key0 + nt * 8 + 2 * t4 + e;
                    s[nt][e] = key <= pos_a ? s[nt][e] * p.scale_log2 : -INFINITY;
                    s[nt][2 + e] = key <= pos_b ? s[nt][2 + e] * p.scale_log2 : -INFINITY;
                    mx_a = fmaxf(mx_a, s[nt][e]);
                    mx_b = fmaxf(mx_b, s[nt][2 + e]);
                }
            mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 1));
            mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 2));
            mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 1));
            mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 2));
            const float mn_a = fmaxf(m_a, mx_a), mn_b = fmaxf(m_b, mx_b);
            const float al_a = exp2_approx(m_a - mn_a), al_b = exp2_approx(m_b - mn_b);
            m_a = mn_a;
            m_b = mn_b;
            float sum_a = 0.f, sum_b = 0.f;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    s[nt][e] = exp2_approx(s[nt][e] - mn_a);
                    s[nt][2 + e] = exp2_approx(s[nt][2 + e] - mn_b);
                    sum_a += s[nt][e];
                    sum_b += s[nt][2 + e];
                }
            l_a = l_a * al_a + sum_a;
            l_b = l_b * al_b + sum_b;
#pragma unroll
            for (int nt = 0; nt < D / 8; ++nt) {
                o[nt][0] *= al_a;
                o[nt][1] *= al_a;
                o[nt][2] *= al_b;
                o[nt][3] *= al_b;
            }
            // keys at or past the context may hold anything: zero those V rows
            // (every warp that reads this page writes the same zeros)
            if (key0 + 16 > ctx) {
                const int first = ctx - key0;
                const int nbad = 16 - first;
                for (int idx = lane; idx < nbad * 8 * Sh::HALVES; idx += 32) {
                    const int hf = idx / (nbad * 8);
                    const int rem = idx - hf * nbad * 8;
                    uint4 *dst = reinterpret_cast<uint4 *>(ring + st * Sh::STAGE_BYTES + Sh::TILE_BYTES +
                                                           hf * Sh::HALF_BYTES + (first + (rem >> 3)) * 128 +
                                                           ((rem & 7) << 4));
                    *dst = make_uint4(0u, 0u, 0u, 0u);
                }
                __syncwarp();
            }
            // P as A operand: (rounded, residual) pairs
            uint32_t ph[4], pl[4];
            pack2_split<T>(s[0][0], s[0][1], ph[0], pl[0]);
            pack2_split<T>(s[0][2], s[0][3], ph[1], pl[1]);
            pack2_split<T>(s[1][0], s[1][1], ph[2], pl[2]);
            pack2_split<T>(s[1][2], s[1][3], ph[3], pl[3]);
#pragma unroll
            for (int dn = 0; dn < D / 16; ++dn) {
                const int chunk = ((dn & 3) << 1) + (mi >> 1);
                const uint32_t addr = vbase + (dn >> 2) * Sh::HALF_BYTES + v_row * 128 + ((chunk ^ (v_row & 7)) << 4);
                uint32_t b0a, b1a, b0b, b1b;
                ldsm_x4_t(addr, b0a, b1a, b0b, b1b);
                mma_16816<T>(o[2 * dn], ph, b0a, b1a);
                mma_16816<T>(o[2 * dn], pl, b0a, b1a);
                mma_16816<T>(o[2 * dn + 1], ph, b0b, b1b);
                mma_16816<T>(o[2 * dn + 1], pl, b0b, b1b);
            }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);
    }

    if (!warp_has_rows) return;
    l_a += __shfl_xor_sync(0xffffffffu, l_a, 1);
    l_a += __shfl_xor_sync(0xffffffffu, l_a, 2);
    l_b += __shfl_xor_sync(0xffffffffu, l_b, 1);
    l_b += __shfl_xor_sync(0xffffffffu, l_b, 2);
    const float inv_a = 1.f / l_a, inv_b = 1.f / l_b;
    const int64_t oa = ((int64_t)(q0 + i0 + tok_a) * p.Hq + h * G + head_a) * D;
    const int64_t ob = ((int64_t)(q0 + i0 + tok_b) * p.Hq + h * G + head_b) * D;
#pragma unroll
    for (int nt = 0; nt < D / 8; ++nt) {
        const int d0 = nt * 8 + 2 * t4;
        if (va) {
            store_out<T>(p.out, p.out_dtype, oa + d0, o[nt][0] * inv_a);
            store_out<T>(p.out, p.out_dtype, oa + d0 + 1, o[nt][1] * inv_a);
        }
        if (vb) {
            store_out<T>(p.out, p.out_dtype, ob + d0, o[nt][2] * inv_b);
            store_out<T>(p.out, p.out_dtype, ob + d0 + 1, o[nt][3] * inv_b);
        }
    }
}

template <typename T, int D>
static int launch_prefill(const PrefillParams &prm, const CUtensorMap &tk, const CUtensorMap &tv, int grid,
                          cudaStream_t stream) {
    using Sh = PrefillShape<D>;
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(paged_prefill_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             Sh::SMEM_BYTES);
        if (e != cudaSuccess) return cuda_fail(e);
        attr_set = true;
    }
    paged_prefill_kernel<T, D><<<grid, kPfThreads, Sh::SMEM_BYTES, stream>>>(prm, tk, tv);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? PKV_OK : cuda_fail(e);
}

}  // namespace pkv

extern "C" int pkv_paged_prefill_attention(void *out, const void *q, const int32_t *cu_seqlens, int num_seqs,
                                           int max_q_len, int total_q, const void *k_cache, const void *v_cache,
                                           const int32_t *block_tables, int max_blocks_per_seq,
                                           const int32_t *context_lens, int num_blocks, int num_q_heads,
                                           int num_kv_heads, int head_dim, int block_size, float scale, int dtype,
                                           int out_dtype, int *dev_status, void *stream) {
    using namespace pkv;
    if (num_seqs < 0 || max_q_len < 0 || total_q < 0 || num_blocks <= 0 || num_kv_heads <= 0 || num_q_heads <= 0 ||
        max_blocks_per_seq <= 0)
        return PKV_ERR_INVALID_ARG;
    if (num_q_heads % num_kv_heads != 0) return PKV_ERR_INVALID_ARG;
    const int G = num_q_heads / num_kv_heads;
    if (G > 16 || block_size != 16 || (head_dim != 64 && head_dim != 128)) return PKV_ERR_UNSUPPORTED;
    if (dtype != PKV_DTYPE_F16 && dtype != PKV_DTYPE_BF16) return PKV_ERR_UNSUPPORTED;
    if (out_dtype != dtype && out_dtype != PKV_DTYPE_F32) return PKV_ERR_UNSUPPORTED;
    if (!std::isfinite(scale)) return PKV_ERR_INVALID_ARG;
    if ((int64_t)num_blocks * num_kv_heads * block_size >= (int64_t)1 << 31) return PKV_ERR_UNSUPPORTED;
    if (num_seqs == 0 || max_q_len == 0 || total_q == 0) return PKV_OK;
    if (!out || !q || !cu_seqlens || !k_cache || !v_cache || !block_tables || !context_lens) return PKV_ERR_INVALID_ARG;
    if (!aligned(q, 4) || !aligned(out, 4) || !aligned(k_cache, 16) || !aligned(v_cache, 16)) return PKV_ERR_INVALID_ARG;
    const int rtok = kPfRows / G;
    const int tiles = (max_q_len + rtok - 1) / rtok;
    const int64_t grid64 = (int64_t)num_seqs * tiles * num_kv_heads;
    if (grid64 >= ((int64_t)1 << 31)) return PKV_ERR_UNSUPPORTED;

    CUtensorMap tk, tv;
    int rc = encode_cache_map(&tk, k_cache, num_blocks, num_kv_heads, block_size, head_dim);
    if (rc != PKV_OK) return rc;
    rc = encode_cache_map(&tv, v_cache, num_blocks, num_kv_heads, block_size, head_dim);
    if (rc != PKV_OK) return rc;

    PrefillParams prm;
    prm.out = out;
    prm.q = q;
    prm.cu_seqlens = cu_seqlens;
    prm.block_tables = block_tables;
    prm.context_lens = context_lens;
    prm.dev_status = dev_status;
    prm.S = num_seqs;
    prm.max_blocks = max_blocks_per_seq;
    prm.num_blocks = num_blocks;
    prm.Hq = num_q_heads;
    prm.Hkv = num_kv_heads;
    prm.G = G;
    prm.rtok = rtok;
    prm.tiles_per_seq = tiles;
    prm.scale_log2 = scale * 1.4426950408889634f;
    prm.out_dtype = out_dtype;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int grid = (int)grid64;
    if (dtype == PKV_DTYPE_BF16)
        return head_dim == 128 ? launch_prefill<__nv_bfloat16, 128>(prm, tk, tv, grid, st)
                               : launch_prefill<__nv_bfloat16, 64>(prm, tk, tv, grid, st);
    return head_dim == 128 ? launch_prefill<__half, 128>(prm, tk, tv, grid, st)
                           : launch_prefill<__half, 64>(prm, tk, tv, grid, st);
}
