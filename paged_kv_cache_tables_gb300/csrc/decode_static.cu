// Decode attention for callers that cannot allocate device memory.
//
// pkv_paged_decode_attention needs a caller-provided workspace for its
// split-context partial results.  Some callers have no way to provide one:
// a serving engine that hands every free byte of HBM to its KV-cache pool up
// front and allows no allocation after start-up, a plugin whose host framework
// owns all device memory, or a latency-critical loop that must not call
// cudaMalloc because it can synchronise the device.  For them this file keeps
// one library-owned scratch array in device global memory and runs the
// existing entry point on it.  Nothing here allocates.
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "pkv.h"
#include "pkv_host.h"

namespace {

constexpr size_t kScratchBytes = (size_t)PKV_STATIC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

// The scratch itself.  Every GPU that loads the library holds it until the
// process exits.  Host code must not pass the symbol directly to a kernel: on
// the host it names a stand-in, not the device address.
__device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

std::mutex g_mu;
void *g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of g_decode_scratch on the current device, looked up once per
// device (with that device current) and cached.
int scratch_address(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        pkv::cuda_fail(e);
        return PKV_ERR_NO_DEVICE;
    }
    if (dev < 0 || dev >= kMaxDevices) return PKV_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_decode_scratch);
        if (e != cudaSuccess || !p) return pkv::cuda_fail(e == cudaSuccess ? cudaErrorInvalidSymbol : e);
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return PKV_OK;
}

}  // namespace

extern "C" int pkv_paged_decode_attention_static(void *out, const void *q, const void *k_cache,
                                                 const void *v_cache, const int32_t *block_tables,
                                                 int max_blocks_per_seq, const int32_t *context_lens,
                                                 int num_seqs, int num_blocks, int num_q_heads, int num_kv_heads,
                                                 int head_dim, int block_size, float scale, int dtype,
                                                 int out_dtype, int *dev_status, void *stream) {
    if (num_seqs > PKV_STATIC_MAX_SEQS) {
        pkv::set_error_message("pkv_paged_decode_attention_static: num_seqs exceeds PKV_STATIC_MAX_SEQS");
        return PKV_ERR_WORKSPACE;
    }
    void *scratch = nullptr;
    int rc = scratch_address(&scratch);
    if (rc != PKV_OK) return rc;
    // The existing entry point validates everything else; only the scratch
    // capacity is checked here.
    if (num_seqs > 0 && num_kv_heads > 0 && num_q_heads > 0 && num_q_heads % num_kv_heads == 0) {
        const size_t need = pkv::decode_workspace_min(num_seqs, num_q_heads, num_kv_heads, head_dim);
        if (need > kScratchBytes) {
            pkv::set_error_message("pkv_paged_decode_attention_static: shape needs more than PKV_STATIC_SCRATCH_BYTES");
            return PKV_ERR_WORKSPACE;
        }
    }
    return pkv_paged_decode_attention(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                                      num_seqs, num_blocks, num_q_heads, num_kv_heads, head_dim, block_size, scale,
                                      dtype, out_dtype, scratch, kScratchBytes, dev_status, stream);
}
