"""Paged KV-cache attention for one continuous-batching engine step on GB300.

The work happens in ``libpkv.so`` (CUDA kernels for sm_103a plus a C++ host
block pool and scheduler); this package only binds it.  Public names mirror
the C ABI in ``include/pkv.h``.
"""
from ._binding import (DTYPE_BF16, DTYPE_F16, DTYPE_F32, PREEMPT_RECOMPUTE, PREEMPT_SWAP, SCHED_CONTINUOUS,
                       SCHED_STATIC, BlockPool, PkvError, Scheduler, copy_blocks, decode_workspace_size, kv_append,
                       lib, mixed_split, paged_decode_append_attention, paged_decode_attention,
                       paged_mixed_append_attention, paged_mixed_attention, paged_prefill_attention)

__all__ = ["DTYPE_BF16", "DTYPE_F16", "DTYPE_F32", "PREEMPT_RECOMPUTE", "PREEMPT_SWAP", "SCHED_CONTINUOUS",
           "SCHED_STATIC", "BlockPool", "PkvError", "Scheduler", "copy_blocks", "decode_workspace_size", "kv_append",
           "lib", "mixed_split", "paged_decode_append_attention", "paged_decode_attention",
           "paged_mixed_append_attention", "paged_mixed_attention", "paged_prefill_attention"]
