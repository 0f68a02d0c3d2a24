// Host-side helpers shared by the launchers: CUDA error capture, device
// properties, and TMA descriptor encoding for the paged caches.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <nvtx3/nvToolsExt.h>

#include <utility>

#include "pkv.h"

namespace pkv {

// NVTX range around a host call (named after the entry point), so profilers
// can filter and attribute the launches; costs a null check without a tool.
struct NvtxRange {
    explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange &) = delete;
    NvtxRange &operator=(const NvtxRange &) = delete;
};

// Records the CUDA error name for pkv_last_cuda_error() and returns PKV_ERR_CUDA.
int cuda_fail(cudaError_t err);
int cuda_fail_driver(int cu_result, const char *what);
// Records a message for pkv_last_cuda_error() (size-limit rejections).
void set_error_message(const char *msg);

// SM count of the current device (cached per device).  PKV_OK or an error.
int current_sm_count(int *num_sms);

// Per-device "done once" flags (kernel attributes are set per device):
// done_on_device tells whether mark_done_on_device has been called for the
// current device.  A caller marks only after its one-time work succeeded, so a
// concurrent caller either sees it done or repeats it (the attribute calls are
// idempotent).  Devices 0..63; beyond that the work is always repeated.
bool done_on_device(const unsigned long long *flag_bits);
void mark_done_on_device(unsigned long long *flag_bits);

// Smallest workspace pkv_paged_decode_attention accepts for this shape (two
// partial records per warp; no room left for stolen pieces).
size_t decode_workspace_min(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim);

// pkv_paged_decode_attention with its grid capped at max_sms CTAs (0: no cap);
// with k_new / v_new given, the append of each sequence's new token is fused
// in (pkv_paged_decode_append_attention).
int decode_attention(void *out, const void *q, const void *k_cache, const void *v_cache,
                     const int32_t *block_tables, int max_blocks_per_seq, const int32_t *context_lens, int num_seqs,
                     int num_blocks, int num_q_heads, int num_kv_heads, int head_dim, int block_size, float scale,
                     int dtype, int out_dtype, void *workspace, size_t workspace_bytes, int *dev_status,
                     cudaStream_t stream, int max_sms, const void *k_new = nullptr, const void *v_new = nullptr);

// Encodes a 2-D TMA descriptor over a paged cache viewed as
// [num_blocks * num_kv_heads * block_size rows][head_dim elements] of 16-bit
// elements, with a box of 64 elements x block_size rows and 128-byte swizzle.
// Out-of-range rows read as zeros.
int encode_cache_map(CUtensorMap *map, const void *base, int num_blocks, int num_kv_heads,
                     int block_size, int head_dim);

// Generic 2..5-D tiled TMA descriptor over 16-bit elements with 128-byte
// swizzle; strides in bytes for dims 1..rank-1.  Out-of-range boxes read 0.
int encode_tiled_map(CUtensorMap *map, const void *base, int rank, const uint64_t *dims, const uint64_t *strides,
                     const uint32_t *box);

// Launches `kernel` on `stream` allowing programmatic dependent launch: it may
// start while the previous kernel on the stream finishes, and waits for that
// kernel's results with griddepcontrol.wait before touching its inputs.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                              Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

inline bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace pkv
