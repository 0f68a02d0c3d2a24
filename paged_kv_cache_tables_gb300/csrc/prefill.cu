// C ABI entry of K4, paged prefill attention: host-side validation, then the
// tensor-core kernel in prefill_tc.cu.
#include <cuda_runtime.h>

#include <cmath>

#include "pkv.h"
#include "pkv_host.h"

namespace pkv {
int prefill_tc(void *out, const void *q, const int32_t *cu_seqlens, int num_seqs, int max_q_len, int total_q,
               const void *k_cache, const void *v_cache, const int32_t *block_tables, int max_blocks_per_seq,
               const int32_t *context_lens, int num_blocks, int Hq, int Hkv, int head_dim, float scale, int dtype,
               int out_dtype, int *dev_status, cudaStream_t stream);
}  // namespace pkv

extern "C" int pkv_paged_prefill_attention(void *out, const void *q, const int32_t *cu_seqlens, int num_seqs,
                                           int max_q_len, int total_q, const void *k_cache, const void *v_cache,
                                           const int32_t *block_tables, int max_blocks_per_seq,
                                           const int32_t *context_lens, int num_blocks, int num_q_heads,
                                           int num_kv_heads, int head_dim, int block_size, float scale, int dtype,
                                           int out_dtype, int *dev_status, void *stream) {
    pkv::NvtxRange nvtx_range("pkv_paged_prefill_attention");
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
    // the query tile is fetched by TMA and output rows are stored as 16-byte vectors
    if (!aligned(q, 16) || !aligned(out, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16))
        return PKV_ERR_INVALID_ARG;
    return prefill_tc(out, q, cu_seqlens, num_seqs, max_q_len, total_q, k_cache, v_cache, block_tables,
                      max_blocks_per_seq, context_lens, num_blocks, num_q_heads, num_kv_heads, head_dim, scale, dtype,
                      out_dtype, dev_status, static_cast<cudaStream_t>(stream));
}
