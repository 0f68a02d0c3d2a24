// The attention of one mixed engine step -- prefill chunks and decodes in one
// batch ("Continuous Batching" §5 "Mixed batching (prefill + decode in one
// step)") -- with the two kernels running side by side.
//
// Prefill is bound by the tensor cores and decode by HBM, so running them one
// after the other leaves each resource idle half the step.  Both kernels hold
// about 200 KB of shared memory per CTA, so they cannot share an SM; instead
// the persistent decode kernel is launched on `decode_sms` CTAs (its work
// stealing rebalances whatever SMs it gets) and the prefill CTAs cycle through
// the other SMs, on a side stream forked from and joined back into the
// caller's stream with events.  The split comes from a cost model of the two
// kernels when the caller passes host copies of the step's metadata.
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>

#include "pkv.h"
#include "pkv_host.h"

namespace pkv {
namespace {

// Per-SM rates of the two kernels on a GB300 (measured: prefill at ~1.1
// PFLOP/s of algorithmic work on 152 SMs, decode streaming ~55 GB/s per SM
// until HBM saturates near 6.2 TB/s).
constexpr double kPrefillFlopsPerSm = 7.0e12;
constexpr double kDecodeBytesPerSm = 55.0e9;
constexpr double kDecodeBytesTotal = 6.2e12;

struct SideStream {
    cudaStream_t stream = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
};

SideStream g_side[64];
std::mutex g_side_mu;   // also serialises the fork / launch / join sequence

// The current device's side stream and events, created on first use.  Call
// with g_side_mu held.
int side_stream(SideStream **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev < 0 || dev >= 64) return PKV_ERR_UNSUPPORTED;
    SideStream &s = g_side[dev];
    if (!s.stream) {
        SideStream n;
        e = cudaStreamCreateWithFlags(&n.stream, cudaStreamNonBlocking);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&n.fork, cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&n.join, cudaEventDisableTiming);
        if (e != cudaSuccess) {
            if (n.fork) cudaEventDestroy(n.fork);
            if (n.stream) cudaStreamDestroy(n.stream);
            return cuda_fail(e);
        }
        s = n;
    }
    *out = &s;
    return PKV_OK;
}

}  // namespace
}  // namespace pkv

extern "C" int pkv_mixed_split(int num_sms, const int32_t *cu_seqlens, int num_prefill,
                               const int32_t *context_lens, int num_decode, int num_q_heads, int num_kv_heads,
                               int head_dim, int elem_bytes) {
    using namespace pkv;
    if (num_sms < 2 || num_prefill < 0 || num_decode < 0 || !context_lens || (num_prefill > 0 && !cu_seqlens))
        return PKV_ERR_INVALID_ARG;
    if (num_prefill == 0) return num_sms;
    if (num_decode == 0) return 0;
    double flops = 0.0, bytes = 0.0;
    for (int c = 0; c < num_prefill; ++c) {
        const double q = cu_seqlens[c + 1] - cu_seqlens[c];
        const double prior = std::max(0.0, (double)context_lens[c] - q);
        flops += 4.0 * num_q_heads * head_dim * (q * prior + q * (q + 1.0) / 2.0);
    }
    for (int s = num_prefill; s < num_prefill + num_decode; ++s)
        bytes += (double)std::max(0, context_lens[s]) * 2.0 * num_kv_heads * head_dim * elem_bytes;
    // the split that balances the two kernels' times
    const int lo = std::max(1, num_sms / 16), hi = num_sms - lo;
    int best = lo;
    double best_t = 1e300;
    for (int d = lo; d <= hi; ++d) {
        const double t_pre = flops / ((num_sms - d) * kPrefillFlopsPerSm);
        const double t_dec = bytes / std::min(d * kDecodeBytesPerSm, kDecodeBytesTotal);
        const double t = std::max(t_pre, t_dec);
        if (t < best_t) {
            best_t = t;
            best = d;
        }
    }
    return best;
}

namespace pkv {
namespace {

// The mixed step's attention, and with k_new / v_new / slot_mapping given its
// append too: the prefill chunks' rows by slot mapping ahead of the prefill
// kernel (on the side stream when decodes run beside it), the decode rows
// inside the decode kernel.
int mixed_attention(void *out, const void *q, const void *k_new, const void *v_new, const int64_t *slot_mapping,
                    const int32_t *cu_seqlens, int num_prefill, int prefill_tokens, int max_q_len, int num_decode,
                    const void *k_cache, const void *v_cache, const int32_t *block_tables, int max_blocks_per_seq,
                    const int32_t *context_lens, int num_blocks, int num_q_heads, int num_kv_heads, int head_dim,
                    int block_size, float scale, int dtype, int out_dtype, void *workspace, size_t workspace_bytes,
                    const int32_t *cu_seqlens_host, const int32_t *context_lens_host, int decode_sms,
                    int *dev_status, cudaStream_t st) {
    if (num_prefill < 0 || num_decode < 0 || prefill_tokens < 0 || num_kv_heads <= 0 || num_q_heads <= 0)
        return PKV_ERR_INVALID_ARG;
    if (num_prefill == 0 && num_decode == 0) return PKV_OK;
    if (!out || !q || !block_tables || !context_lens) return PKV_ERR_INVALID_ARG;
    const bool append = k_new != nullptr;
    if (append && (!v_new || (num_prefill > 0 && !slot_mapping))) return PKV_ERR_INVALID_ARG;
    const size_t in_row = (size_t)num_q_heads * head_dim * 2;
    const size_t kv_row = (size_t)num_kv_heads * head_dim * 2;
    const size_t out_row = (size_t)num_q_heads * head_dim * (out_dtype == PKV_DTYPE_F32 ? 4 : 2);
    void *out_d = static_cast<char *>(out) + prefill_tokens * out_row;
    const void *q_d = static_cast<const char *>(q) + prefill_tokens * in_row;
    const int32_t *bt_d = block_tables + (size_t)num_prefill * max_blocks_per_seq;
    const int32_t *cl_d = context_lens + num_prefill;
    const void *k_d = append ? static_cast<const char *>(k_new) + prefill_tokens * kv_row : nullptr;
    const void *v_d = append ? static_cast<const char *>(v_new) + prefill_tokens * kv_row : nullptr;
    // the prefill part, on stream s: its rows appended first
    auto prefill = [&](cudaStream_t s) {
        if (append) {
            const int rc = pkv_kv_append(k_new, v_new, slot_mapping, prefill_tokens, const_cast<void *>(k_cache),
                                         const_cast<void *>(v_cache), num_blocks, block_size, num_kv_heads,
                                         head_dim, dtype, dev_status, s);
            if (rc != PKV_OK) return rc;
        }
        return pkv_paged_prefill_attention(out, q, cu_seqlens, num_prefill, max_q_len, prefill_tokens, k_cache,
                                           v_cache, block_tables, max_blocks_per_seq, context_lens, num_blocks,
                                           num_q_heads, num_kv_heads, head_dim, block_size, scale, dtype, out_dtype,
                                           dev_status, s);
    };
    // one kind of work only: no side stream
    if (num_decode == 0) return prefill(st);
    if (num_prefill == 0)
        return decode_attention(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                                num_decode, num_blocks, num_q_heads, num_kv_heads, head_dim, block_size, scale, dtype,
                                out_dtype, workspace, workspace_bytes, dev_status, st, 0, k_new, v_new);
    int sms = 0;
    int rc = current_sm_count(&sms);
    if (rc != PKV_OK) return rc;
    int d_sms = decode_sms;
    if (d_sms <= 0) {
        d_sms = (cu_seqlens_host && context_lens_host)
                    ? pkv_mixed_split(sms, cu_seqlens_host, num_prefill, context_lens_host, num_decode, num_q_heads,
                                      num_kv_heads, head_dim, 2)
                    : sms * 3 / 5;
    }
    d_sms = std::max(1, std::min(d_sms, sms - 1));
    std::lock_guard<std::mutex> lock(g_side_mu);
    SideStream *side = nullptr;
    rc = side_stream(&side);
    if (rc != PKV_OK) return rc;
    cudaError_t e = cudaEventRecord(side->fork, st);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(side->stream, side->fork, 0);
    if (e != cudaSuccess) return cuda_fail(e);
    // decode first, so that its persistent CTAs hold their SMs; the prefill
    // CTAs take the rest and keep cycling through them.  The two touch
    // different sequences' blocks (a shared prefix page is never written).
    rc = decode_attention(out_d, q_d, k_cache, v_cache, bt_d, max_blocks_per_seq, cl_d, num_decode, num_blocks,
                          num_q_heads, num_kv_heads, head_dim, block_size, scale, dtype, out_dtype, workspace,
                          workspace_bytes, dev_status, st, d_sms, k_d, v_d);
    const int rc2 = prefill(side->stream);
    // join, whatever happened, so the caller's stream never runs ahead of
    // work still queued on the side stream
    e = cudaEventRecord(side->join, side->stream);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(st, side->join, 0);
    if (e != cudaSuccess) return cuda_fail(e);
    return rc != PKV_OK ? rc : rc2;
}

}  // namespace
}  // namespace pkv

extern "C" int pkv_paged_mixed_attention(void *out, const void *q, const int32_t *cu_seqlens, int num_prefill,
                                         int prefill_tokens, int max_q_len, int num_decode, const void *k_cache,
                                         const void *v_cache, const int32_t *block_tables, int max_blocks_per_seq,
                                         const int32_t *context_lens, int num_blocks, int num_q_heads,
                                         int num_kv_heads, int head_dim, int block_size, float scale, int dtype,
                                         int out_dtype, void *workspace, size_t workspace_bytes,
                                         const int32_t *cu_seqlens_host, const int32_t *context_lens_host,
                                         int decode_sms, int *dev_status, void *stream) {
    pkv::NvtxRange nvtx_range("pkv_paged_mixed_attention");
    return pkv::mixed_attention(out, q, nullptr, nullptr, nullptr, cu_seqlens, num_prefill, prefill_tokens,
                                max_q_len, num_decode, k_cache, v_cache, block_tables, max_blocks_per_seq,
                                context_lens, num_blocks, num_q_heads, num_kv_heads, head_dim, block_size, scale,
                                dtype, out_dtype, workspace, workspace_bytes, cu_seqlens_host, context_lens_host,
                                decode_sms, dev_status, static_cast<cudaStream_t>(stream));
}

extern "C" int pkv_paged_mixed_append_attention(void *out, const void *q, const void *k_new, const void *v_new,
                                                const int64_t *slot_mapping, const int32_t *cu_seqlens,
                                                int num_prefill, int prefill_tokens, int max_q_len, int num_decode,
                                                void *k_cache, void *v_cache, const int32_t *block_tables,
                                                int max_blocks_per_seq, const int32_t *context_lens, int num_blocks,
                                                int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                                float scale, int dtype, int out_dtype, void *workspace,
                                                size_t workspace_bytes, const int32_t *cu_seqlens_host,
                                                const int32_t *context_lens_host, int decode_sms, int *dev_status,
                                                void *stream) {
    pkv::NvtxRange nvtx_range("pkv_paged_mixed_append_attention");
    if (!k_new || !v_new) return PKV_ERR_INVALID_ARG;
    return pkv::mixed_attention(out, q, k_new, v_new, slot_mapping, cu_seqlens, num_prefill, prefill_tokens,
                                max_q_len, num_decode, k_cache, v_cache, block_tables, max_blocks_per_seq,
                                context_lens, num_blocks, num_q_heads, num_kv_heads, head_dim, block_size, scale,
                                dtype, out_dtype, workspace, workspace_bytes, cu_seqlens_host, context_lens_host,
                                decode_sms, dev_status, static_cast<cudaStream_t>(stream));
}
