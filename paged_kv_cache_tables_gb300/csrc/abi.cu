// Library-wide C ABI pieces: status strings, CUDA error capture, device
// queries and the TMA descriptor encoder used by the attention launchers.
#include <cudaTypedefs.h>

#include <cstdio>
#include <cstring>
#include <mutex>

#include "pkv.h"
#include "pkv_host.h"

namespace pkv {

static thread_local char g_last_error[256] = "no error";

int cuda_fail(cudaError_t err) {
    std::snprintf(g_last_error, sizeof g_last_error, "%s: %s", cudaGetErrorName(err),
                  cudaGetErrorString(err));
    return PKV_ERR_CUDA;
}

int cuda_fail_driver(int cu_result, const char *what) {
    std::snprintf(g_last_error, sizeof g_last_error, "%s failed with CUresult %d", what, cu_result);
    return PKV_ERR_CUDA;
}

void set_error_message(const char *msg) { std::snprintf(g_last_error, sizeof g_last_error, "%s", msg); }

bool done_on_device(const unsigned long long *flag_bits) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
    return (__atomic_load_n(flag_bits, __ATOMIC_ACQUIRE) >> dev) & 1ull;
}

void mark_done_on_device(unsigned long long *flag_bits) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return;
    __atomic_fetch_or(flag_bits, 1ull << dev, __ATOMIC_ACQ_REL);
}

int current_sm_count(int *num_sms) {
    static int cached[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        cuda_fail(e);
        return PKV_ERR_NO_DEVICE;
    }
    if (dev >= 0 && dev < 64) {
        const int c = __atomic_load_n(&cached[dev], __ATOMIC_RELAXED);
        if (c > 0) {
            *num_sms = c;
            return PKV_OK;
        }
    }
    int n = 0;
    e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) {
        cuda_fail(e);
        return PKV_ERR_NO_DEVICE;
    }
    if (dev >= 0 && dev < 64) __atomic_store_n(&cached[dev], n, __ATOMIC_RELAXED);
    *num_sms = n;
    return PKV_OK;
}

static PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

int encode_tiled_map(CUtensorMap *map, const void *base, int rank, const uint64_t *dims, const uint64_t *strides,
                     const uint32_t *box) {
    auto fn = get_encode_fn();
    if (!fn) return cuda_fail_driver(-1, "cuTensorMapEncodeTiled lookup");
    cuuint64_t d[5], st[4];
    cuuint32_t b[5], es[5];
    for (int i = 0; i < rank; ++i) {
        d[i] = dims[i];
        b[i] = box[i];
        es[i] = 1;
        if (i + 1 < rank) st[i] = strides[i];
    }
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, (cuuint32_t)rank, const_cast<void *>(base), d, st, b, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cuda_fail_driver((int)r, "cuTensorMapEncodeTiled");
    return PKV_OK;
}

int encode_cache_map(CUtensorMap *map, const void *base, int num_blocks, int num_kv_heads, int block_size,
                     int head_dim) {
    auto fn = get_encode_fn();
    if (!fn) return cuda_fail_driver(-1, "cuTensorMapEncodeTiled lookup");
    const cuuint64_t rows = (cuuint64_t)num_blocks * num_kv_heads * block_size;
    cuuint64_t dims[2] = {(cuuint64_t)head_dim, rows};
    cuuint64_t strides[1] = {(cuuint64_t)head_dim * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)block_size};
    cuuint32_t estrides[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void *>(base), dims, strides, box,
                    estrides, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cuda_fail_driver((int)r, "cuTensorMapEncodeTiled");
    return PKV_OK;
}

}  // namespace pkv

extern "C" const char *pkv_status_string(int status) {
    switch (status) {
        case PKV_OK: return "PKV_OK";
        case PKV_ERR_INVALID_ARG: return "PKV_ERR_INVALID_ARG";
        case PKV_ERR_UNSUPPORTED: return "PKV_ERR_UNSUPPORTED";
        case PKV_ERR_WORKSPACE: return "PKV_ERR_WORKSPACE";
        case PKV_ERR_CUDA: return "PKV_ERR_CUDA";
        case PKV_ERR_OUT_OF_BLOCKS: return "PKV_ERR_OUT_OF_BLOCKS";
        case PKV_ERR_NO_DEVICE: return "PKV_ERR_NO_DEVICE";
        case PKV_ERR_NO_MEMORY: return "PKV_ERR_NO_MEMORY";
        default: return "PKV_ERR_UNKNOWN";
    }
}

extern "C" const char *pkv_last_cuda_error(void) { return pkv::g_last_error; }

extern "C" const char *pkv_version(void) { return "pkv 0.1 sm_103a"; }
