// Synthetic input rows for the continuous-batching trace, generated on the
// GPU with the same counter-based hash as synth/trace.py (numpy).  Input
// generation only: no attention arithmetic lives here.
//
// Value of element e of the row of token (rid, pos) under tag:
//   base = H(H(H(seed ^ lo32(rid)) ^ pos) ^ tag),  h = H(base ^ e),
//   x = float(h >> 8) * 2^-24 * 4 - 2   (uniform on [-2, 2)),
// rounded to nearest even to bf16 or fp16, where H is Wellons' "lowbias32"
// integer hash (x ^= x>>16; x *= 0x7feb352d; x ^= x>>15; x *= 0x846ca68b;
// x ^= x>>16).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

__device__ __forceinline__ uint32_t lowbias32(uint32_t x) {
    x ^= x >> 16;
    x *= 0x7feb352du;
    x ^= x >> 15;
    x *= 0x846ca68bu;
    x ^= x >> 16;
    return x;
}

__global__ void fill_rows_kernel(uint16_t *out, const int64_t *rids, const int32_t *pos, int n, int width,
                                 uint32_t seed, uint32_t tag, int bf16) {
    const int64_t total = (int64_t)n * width;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int t = (int)(i / width);
        const uint32_t e = (uint32_t)(i - (int64_t)t * width);
        uint32_t b = lowbias32(seed ^ (uint32_t)rids[t]);
        b = lowbias32(b ^ (uint32_t)pos[t]);
        b = lowbias32(b ^ tag);
        const uint32_t h = lowbias32(b ^ e);
        const float x = (float)(h >> 8) * (1.0f / 16777216.0f) * 4.0f - 2.0f;
        if (bf16) {
            __nv_bfloat16 v = __float2bfloat16_rn(x);
            out[i] = *reinterpret_cast<uint16_t *>(&v);
        } else {
            __half v = __float2half_rn(x);
            out[i] = *reinterpret_cast<uint16_t *>(&v);
        }
    }
}

// One launch for a layer's Q, K and V rows: block (t, which) writes the row of
// token t in out_which; the row's base hash is computed once.
__device__ __forceinline__ uint16_t synth_value(uint32_t b, uint32_t e, int bf16) {
    const uint32_t h = lowbias32(b ^ e);
    const float x = (float)(h >> 8) * (1.0f / 16777216.0f) * 4.0f - 2.0f;
    if (bf16) {
        __nv_bfloat16 v = __float2bfloat16_rn(x);
        return *reinterpret_cast<uint16_t *>(&v);
    }
    __half v = __float2half_rn(x);
    return *reinterpret_cast<uint16_t *>(&v);
}

__global__ void fill_qkv_kernel(uint16_t *q, uint16_t *k, uint16_t *v, const int64_t *rids, const int32_t *pos,
                                int wq, int wkv, uint32_t seed, uint32_t tq, uint32_t tk, uint32_t tv, int bf16) {
    const int t = blockIdx.x, which = blockIdx.y;
    uint16_t *out = which == 0 ? q : (which == 1 ? k : v);
    const int width = which == 0 ? wq : wkv;
    const uint32_t tag = which == 0 ? tq : (which == 1 ? tk : tv);
    uint32_t b = lowbias32(seed ^ (uint32_t)rids[t]);
    b = lowbias32(b ^ (uint32_t)pos[t]);
    b = lowbias32(b ^ tag);
    uint16_t *row = out + (int64_t)t * width;
    for (int e = threadIdx.x; e < width; e += blockDim.x) row[e] = synth_value(b, (uint32_t)e, bf16);
}

}  // namespace

extern "C" int synth_fill_qkv(void *q, void *k, void *v, const int64_t *rids, const int32_t *pos, int n, int wq,
                              int wkv, uint32_t seed, uint32_t tq, uint32_t tk, uint32_t tv, int bf16, void *stream) {
    if (n <= 0) return 0;
    fill_qkv_kernel<<<dim3(n, 3), 256, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<uint16_t *>(q), static_cast<uint16_t *>(k), static_cast<uint16_t *>(v), rids, pos, wq, wkv, seed,
        tq, tk, tv, bf16);
    return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

extern "C" int synth_fill_rows(void *out, const int64_t *rids, const int32_t *pos, int n, int width, uint32_t seed,
                               uint32_t tag, int bf16, void *stream) {
    if (n <= 0) return 0;
    const int64_t total = (int64_t)n * width;
    int blocks = (int)((total + 255) / 256);
    if (blocks > 4096) blocks = 4096;
    fill_rows_kernel<<<blocks, 256, 0, static_cast<cudaStream_t>(stream)>>>(static_cast<uint16_t *>(out), rids, pos,
                                                                            n, width, seed, tag, bf16);
    return cudaGetLastError() == cudaSuccess ? 0 : -1;
}
