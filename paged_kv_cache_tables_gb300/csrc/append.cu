// K1: append this step's new K/V rows into the paged cache by slot mapping.
//
// "Project 17: Production Serving: Continuous Batching and PagedAttention",
// Step 4 "Implement the paged KV cache": a token's key and value go to
// (physical page, slot in page).  The slot of every new token comes from the
// step's slot_mapping ("Continuous Batching" §6 "Under the hood").  A pure
// bit copy: each thread moves one 16-byte vector of K and the matching vector
// of V; a warp covers two (token, head) rows of head_dim 128, so reads and
// writes are whole 256-byte rows.
#include <cuda_runtime.h>

#include "pkv.h"
#include "pkv_device.cuh"
#include "pkv_host.h"

namespace pkv {

__global__ void __launch_bounds__(256) kv_append_kernel(const uint4 *__restrict__ k, const uint4 *__restrict__ v,
                                                        const int64_t *__restrict__ slot_mapping, int num_tokens,
                                                        uint4 *__restrict__ k_cache, uint4 *__restrict__ v_cache,
                                                        int num_blocks, int block_size, int num_kv_heads,
                                                        int vec_per_row, int *dev_status) {
    pdl_wait_primary();
    pdl_launch_dependents();
    const int64_t items = (int64_t)num_tokens * num_kv_heads * vec_per_row;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < items; i += stride) {
        const int64_t row = i / vec_per_row;           // (token, head)
        const int vec = (int)(i - row * vec_per_row);
        const int t = (int)(row / num_kv_heads);
        const int h = (int)(row - (int64_t)t * num_kv_heads);
        const int64_t slot = __ldg(slot_mapping + t);
        if (slot < 0) continue;
        const int64_t block = slot / block_size;
        const int off = (int)(slot - block * block_size);
        if (block >= num_blocks) {
            if (vec == 0 && h == 0) set_status(dev_status, PKV_DEV_BAD_SLOT);
            continue;
        }
        const int64_t dst = ((block * num_kv_heads + h) * block_size + off) * vec_per_row + vec;
        k_cache[dst] = __ldg(k + i);
        v_cache[dst] = __ldg(v + i);
    }
}

}  // namespace pkv

extern "C" int pkv_kv_append(const void *k, const void *v, const int64_t *slot_mapping, int num_tokens,
                             void *k_cache, void *v_cache, int num_blocks, int block_size, int num_kv_heads,
                             int head_dim, int dtype, int *dev_status, void *stream) {
    pkv::NvtxRange nvtx_range("pkv_kv_append");
    using namespace pkv;
    if (num_tokens < 0 || num_blocks <= 0 || num_kv_heads <= 0) return PKV_ERR_INVALID_ARG;
    if (dtype != PKV_DTYPE_F16 && dtype != PKV_DTYPE_BF16) return PKV_ERR_UNSUPPORTED;
    if (block_size != 16 || (head_dim != 64 && head_dim != 128)) return PKV_ERR_UNSUPPORTED;
    if (num_tokens == 0) return PKV_OK;
    if (!k || !v || !slot_mapping || !k_cache || !v_cache) return PKV_ERR_INVALID_ARG;
    if (!aligned(k, 16) || !aligned(v, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
        !aligned(slot_mapping, 8))
        return PKV_ERR_INVALID_ARG;
    int sms = 0;
    int rc = current_sm_count(&sms);
    if (rc != PKV_OK) return rc;
    const int vec_per_row = head_dim * 2 / 16;
    const int64_t items = (int64_t)num_tokens * num_kv_heads * vec_per_row;
    const int threads = 256;
    int64_t blocks = (items + threads - 1) / threads;
    if (blocks > (int64_t)sms * 8) blocks = (int64_t)sms * 8;
    cudaError_t e = launch_pdl(kv_append_kernel, dim3((unsigned)blocks), dim3(threads), 0,
                               static_cast<cudaStream_t>(stream), static_cast<const uint4 *>(k),
                               static_cast<const uint4 *>(v), slot_mapping, num_tokens, static_cast<uint4 *>(k_cache),
                               static_cast<uint4 *>(v_cache), num_blocks, block_size, num_kv_heads, vec_per_row,
                               dev_status);
    if (e == cudaSuccess) e = cudaGetLastError();
    return e == cudaSuccess ? PKV_OK : cuda_fail(e);
}

// ---------------------------------------------------------------- block copies

namespace pkv {

constexpr int kCopyUnroll = 8;

// One CTA per (src, dst) pair: copies block_vec 16-byte vectors from block
// pairs[2i] of src to block pairs[2i+1] of dst (device or pinned host memory:
// both are addressed directly).  Each thread issues kCopyUnroll loads before
// its stores, so that enough bytes are in flight to cover the latency of the
// host link.
__global__ void __launch_bounds__(256) copy_blocks_kernel(uint4 *__restrict__ dst, const uint4 *__restrict__ src,
                                                          const int32_t *__restrict__ pairs, int num_pairs,
                                                          int64_t block_vec, int64_t src_blocks, int64_t dst_blocks,
                                                          int *dev_status) {
    pdl_wait_primary();
    pdl_launch_dependents();
    for (int i = blockIdx.x; i < num_pairs; i += gridDim.x) {
        const int64_t s = __ldg(pairs + 2 * i), d = __ldg(pairs + 2 * i + 1);
        if (s < 0 || s >= src_blocks || d < 0 || d >= dst_blocks) {
            if (threadIdx.x == 0) set_status(dev_status, PKV_DEV_BAD_BLOCK_ID);
            continue;
        }
        const uint4 *from = src + s * block_vec;
        uint4 *to = dst + d * block_vec;
        for (int64_t v0 = threadIdx.x; v0 < block_vec; v0 += (int64_t)blockDim.x * kCopyUnroll) {
            uint4 r[kCopyUnroll];
#pragma unroll
            for (int j = 0; j < kCopyUnroll; ++j) {
                const int64_t v = v0 + (int64_t)j * blockDim.x;
                if (v < block_vec) r[j] = from[v];
            }
#pragma unroll
            for (int j = 0; j < kCopyUnroll; ++j) {
                const int64_t v = v0 + (int64_t)j * blockDim.x;
                if (v < block_vec) to[v] = r[j];
            }
        }
    }
}

}  // namespace pkv

extern "C" int pkv_copy_blocks(void *dst, int64_t dst_blocks, const void *src, int64_t src_blocks,
                               const int32_t *pairs, int num_pairs, int64_t block_bytes, int *dev_status,
                               void *stream) {
    pkv::NvtxRange nvtx_range("pkv_copy_blocks");
    using namespace pkv;
    if (num_pairs < 0 || block_bytes <= 0 || dst_blocks <= 0 || src_blocks <= 0) return PKV_ERR_INVALID_ARG;
    if (num_pairs == 0) return PKV_OK;
    if (!dst || !src || !pairs) return PKV_ERR_INVALID_ARG;
    if (block_bytes % 16 != 0 || !aligned(dst, 16) || !aligned(src, 16) || !aligned(pairs, 4))
        return PKV_ERR_INVALID_ARG;
    int sms = 0;
    int rc = current_sm_count(&sms);
    if (rc != PKV_OK) return rc;
    const int grid = num_pairs < sms * 4 ? num_pairs : sms * 4;
    cudaError_t e = launch_pdl(copy_blocks_kernel, dim3(grid), dim3(256), 0, static_cast<cudaStream_t>(stream),
                               static_cast<uint4 *>(dst), static_cast<const uint4 *>(src), pairs, num_pairs,
                               (int64_t)(block_bytes / 16), src_blocks, dst_blocks, dev_status);
    if (e == cudaSuccess) e = cudaGetLastError();
    return e == cudaSuccess ? PKV_OK : cuda_fail(e);
}
