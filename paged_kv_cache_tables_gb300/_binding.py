"""Thin ctypes binding over libpkv.so (argument marshalling only).

Every function here has the name of the C entry point it calls (without the
``pkv_`` prefix) and does nothing but check tensor placement/dtype/layout,
take pointers and sizes, and pass the current CUDA stream.  All arithmetic of
the attention path runs in the library's kernels; there is no fallback.  If
libpkv.so is missing the first call raises: build it with
``paged_kv_cache_tables_gb300.build.build()`` (``__graft_entry__.build()``).
"""
import ctypes
import math
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpkv.so")

PKV_OK = 0
DTYPE_F16, DTYPE_BF16, DTYPE_F32 = 0, 1, 2
DEV_BAD_BLOCK_ID, DEV_BAD_CONTEXT, DEV_WAIT_TIMEOUT, DEV_BAD_SLOT, DEV_BAD_CHUNK, DEV_SPLIT = 1, 2, 4, 8, 16, 32

_lib = None


class PkvError(RuntimeError):
    def __init__(self, func, status):
        self.status = status
        msg = "%s failed: %s" % (func, _lib.pkv_status_string(status).decode() if _lib else status)
        if _lib is not None and status == -4:
            msg += " (%s)" % _lib.pkv_last_cuda_error().decode()
        super().__init__(msg)


class StepMeta(ctypes.Structure):
    _fields_ = [("num_seqs", ctypes.c_int), ("num_prefill", ctypes.c_int), ("num_tokens", ctypes.c_int),
                ("max_blocks", ctypes.c_int), ("seq_rids", ctypes.POINTER(ctypes.c_int64)),
                ("q_lens", ctypes.POINTER(ctypes.c_int32)), ("context_lens", ctypes.POINTER(ctypes.c_int32)),
                ("cu_seqlens", ctypes.POINTER(ctypes.c_int32)), ("block_tables", ctypes.POINTER(ctypes.c_int32)),
                ("slot_mapping", ctypes.POINTER(ctypes.c_int64)), ("token_rids", ctypes.POINTER(ctypes.c_int64)),
                ("token_pos", ctypes.POINTER(ctypes.c_int32)), ("num_finished", ctypes.c_int),
                ("finished_rids", ctypes.POINTER(ctypes.c_int64)), ("num_swap_out", ctypes.c_int),
                ("swap_out", ctypes.POINTER(ctypes.c_int32)), ("num_swap_in", ctypes.c_int),
                ("swap_in", ctypes.POINTER(ctypes.c_int32))]


class SchedConfig(ctypes.Structure):
    _fields_ = [("num_blocks", ctypes.c_int), ("block_size", ctypes.c_int), ("max_batch", ctypes.c_int),
                ("max_num_batched_tokens", ctypes.c_int), ("chunk", ctypes.c_int), ("max_model_len", ctypes.c_int),
                ("initial_order", ctypes.POINTER(ctypes.c_int32)), ("policy", ctypes.c_int),
                ("prefix_caching", ctypes.c_int), ("preemption", ctypes.c_int), ("swap_blocks", ctypes.c_int)]


SCHED_CONTINUOUS, SCHED_STATIC = 0, 1
PREEMPT_RECOMPUTE, PREEMPT_SWAP = 0, 1


class SchedStats(ctypes.Structure):
    _fields_ = [("steps", ctypes.c_int64), ("preemptions", ctypes.c_int64), ("admitted", ctypes.c_int64),
                ("finished", ctypes.c_int64), ("sum_running", ctypes.c_int64), ("tokens", ctypes.c_int64),
                ("prefill_tokens", ctypes.c_int64), ("running", ctypes.c_int), ("waiting", ctypes.c_int),
                ("free_blocks", ctypes.c_int), ("host_ms", ctypes.c_double), ("prefix_hit_blocks", ctypes.c_int64),
                ("cached_blocks", ctypes.c_int), ("swapped_out_blocks", ctypes.c_int64),
                ("swapped_in_blocks", ctypes.c_int64), ("free_swap_slots", ctypes.c_int)]


def lib():
    """Load libpkv.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError("libpkv.so is not built (%s); run paged_kv_cache_tables_gb300.build.build()" % LIB_PATH)
    L = ctypes.CDLL(LIB_PATH)
    P, I, I64, F, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
    sig = {
        "pkv_status_string": ([I], ctypes.c_char_p),
        "pkv_last_cuda_error": ([], ctypes.c_char_p),
        "pkv_version": ([], ctypes.c_char_p),
        "pkv_kv_append": ([P, P, P, I, P, P, I, I, I, I, I, P, P], I),
        "pkv_decode_workspace_size": ([I, I, I, I], SZ),
        "pkv_paged_decode_attention": ([P, P, P, P, P, I, P, I, I, I, I, I, I, F, I, I, P, SZ, P, P], I),
        "pkv_paged_decode_append_attention": ([P, P, P, P, P, P, P, I, P, I, I, I, I, I, I, F, I, I, P, SZ, P, P], I),
        "pkv_paged_prefill_attention": ([P, P, P, I, I, I, P, P, P, I, P, I, I, I, I, I, F, I, I, P, P], I),
        "pkv_paged_decode_attention_static": ([P, P, P, P, P, I, P, I, I, I, I, I, I, F, I, I, P, P], I),
        "pkv_paged_mixed_attention": ([P, P, P, I, I, I, I, P, P, P, I, P, I, I, I, I, I, F, I, I, P, SZ, P, P, I, P, P],
                                      I),
        "pkv_paged_mixed_append_attention": ([P, P, P, P, P, P, I, I, I, I, P, P, P, I, P, I, I, I, I, I, F, I, I, P,
                                              SZ, P, P, I, P, P], I),
        "pkv_mixed_split": ([I, P, I, P, I, I, I, I, I], I),
        "pkv_copy_blocks": ([P, I64, P, I64, P, I, I64, P, P], I),
        "pkv_pool_create": ([I, P], P),
        "pkv_pool_destroy": ([P], None),
        "pkv_pool_alloc": ([P, I, P], I),
        "pkv_pool_free": ([P, P, I], I),
        "pkv_pool_free_count": ([P], I),
        "pkv_pool_free_list": ([P, P], I),
        "pkv_pool_inject_failure": ([P, I64], I),
        "pkv_sched_create": ([ctypes.POINTER(SchedConfig)], P),
        "pkv_sched_destroy": ([P], None),
        "pkv_sched_add": ([P, I64, I, I, I], I),
        "pkv_sched_add_tokens": ([P, I64, P, I, I, I], I),
        "pkv_sched_step": ([P, ctypes.POINTER(StepMeta)], I),
        "pkv_sched_get_stats": ([P, ctypes.POINTER(SchedStats)], I),
        "pkv_sched_inject_alloc_failure": ([P, I64], I),
        "pkv_sched_request_state": ([P, I64, ctypes.POINTER(ctypes.c_int)], I),
        "pkv_sched_forget": ([P, I64], I),
    }
    for name, (args, res) in sig.items():
        fn = getattr(L, name)
        fn.argtypes = args
        fn.restype = res
    _lib = L
    return L


def _check(func, status):
    if status != PKV_OK:
        raise PkvError(func, status)


# ------------------------------------------------------------ device entry points

def _dtype_code(t):
    import torch
    return {torch.float16: DTYPE_F16, torch.bfloat16: DTYPE_BF16, torch.float32: DTYPE_F32}[t.dtype]


def _dev(t, name, dtype=None, ndim=None):
    import torch
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError("%s must be a CUDA tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if dtype is not None and t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if ndim is not None and t.dim() != ndim:
        raise ValueError("%s must have %d dims" % (name, ndim))
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _status_ptr(dev_status):
    import torch
    if dev_status is None:
        return None
    return _dev(dev_status, "dev_status", torch.int32)


def kv_append(k, v, slot_mapping, k_cache, v_cache, dev_status=None, stream=None):
    """pkv_kv_append: k, v [T, Hkv, d]; slot_mapping int64 [T]; caches [NB, Hkv, 16, d]."""
    import torch
    L = lib()
    T, Hkv, d = k.shape
    NB, _, bs, _ = k_cache.shape
    st = L.pkv_kv_append(_dev(k, "k", ndim=3), _dev(v, "v", k.dtype, 3), _dev(slot_mapping, "slot_mapping", torch.int64),
                         T, _dev(k_cache, "k_cache", k.dtype, 4), _dev(v_cache, "v_cache", k.dtype, 4), NB, bs, Hkv, d,
                         _dtype_code(k), _status_ptr(dev_status), _stream(stream))
    _check("pkv_kv_append", st)


def decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim):
    return int(lib().pkv_decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim))


def paged_decode_attention(out, q, k_cache, v_cache, block_tables, context_lens, scale=None, workspace=None,
                           dev_status=None, stream=None):
    """pkv_paged_decode_attention: q/out [S, Hq, d]; block_tables int32 [S, max_blocks];
    context_lens int32 [S].  workspace: uint8 CUDA tensor (allocated here if None)."""
    import torch
    L = lib()
    S, Hq, d = q.shape
    NB, Hkv, bs, _ = k_cache.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if workspace is None:
        workspace = torch.empty(max(16, decode_workspace_size(S, Hq, Hkv, d)), dtype=torch.uint8, device=q.device)
    st = L.pkv_paged_decode_attention(
        _dev(out, "out", ndim=3), _dev(q, "q", ndim=3), _dev(k_cache, "k_cache", q.dtype, 4),
        _dev(v_cache, "v_cache", q.dtype, 4), _dev(block_tables, "block_tables", torch.int32, 2),
        block_tables.shape[1], _dev(context_lens, "context_lens", torch.int32, 1), S, NB, Hq, Hkv, d, bs,
        float(scale), _dtype_code(q), _dtype_code(out), _dev(workspace, "workspace"), workspace.numel(),
        _status_ptr(dev_status), _stream(stream))
    _check("pkv_paged_decode_attention", st)


def paged_decode_append_attention(out, q, k_new, v_new, k_cache, v_cache, block_tables, context_lens, scale=None,
                                  workspace=None, dev_status=None, stream=None):
    """pkv_paged_decode_append_attention: kv_append of k_new/v_new [S, Hkv, d]
    at position context_lens[s] - 1 of each sequence, then decode attention, in
    one launch."""
    import torch
    L = lib()
    S, Hq, d = q.shape
    NB, Hkv, bs, _ = k_cache.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if workspace is None:
        workspace = torch.empty(max(16, decode_workspace_size(S, Hq, Hkv, d)), dtype=torch.uint8, device=q.device)
    st = L.pkv_paged_decode_append_attention(
        _dev(out, "out", ndim=3), _dev(q, "q", ndim=3), _dev(k_new, "k_new", q.dtype, 3),
        _dev(v_new, "v_new", q.dtype, 3), _dev(k_cache, "k_cache", q.dtype, 4), _dev(v_cache, "v_cache", q.dtype, 4),
        _dev(block_tables, "block_tables", torch.int32, 2), block_tables.shape[1],
        _dev(context_lens, "context_lens", torch.int32, 1), S, NB, Hq, Hkv, d, bs, float(scale), _dtype_code(q),
        _dtype_code(out), _dev(workspace, "workspace"), workspace.numel(), _status_ptr(dev_status), _stream(stream))
    _check("pkv_paged_decode_append_attention", st)


def paged_prefill_attention(out, q, cu_seqlens, max_q_len, k_cache, v_cache, block_tables, context_lens, scale=None,
                            dev_status=None, stream=None):
    """pkv_paged_prefill_attention: q/out [total_q, Hq, d]; cu_seqlens int32 [S+1]."""
    import torch
    L = lib()
    total_q, Hq, d = q.shape
    NB, Hkv, bs, _ = k_cache.shape
    S = cu_seqlens.shape[0] - 1
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    st = L.pkv_paged_prefill_attention(
        _dev(out, "out", ndim=3), _dev(q, "q", ndim=3), _dev(cu_seqlens, "cu_seqlens", torch.int32, 1), S,
        int(max_q_len), total_q, _dev(k_cache, "k_cache", q.dtype, 4), _dev(v_cache, "v_cache", q.dtype, 4),
        _dev(block_tables, "block_tables", torch.int32, 2), block_tables.shape[1],
        _dev(context_lens, "context_lens", torch.int32, 1), NB, Hq, Hkv, d, bs, float(scale), _dtype_code(q),
        _dtype_code(out), _status_ptr(dev_status), _stream(stream))
    _check("pkv_paged_prefill_attention", st)


def paged_mixed_attention(out, q, cu_seqlens, num_prefill, max_q_len, k_cache, v_cache, block_tables, context_lens,
                          scale=None, workspace=None, cu_seqlens_host=None, context_lens_host=None, decode_sms=0,
                          dev_status=None, stream=None):
    """pkv_paged_mixed_attention: rows [0, cu_seqlens[num_prefill]) of q/out are
    the prefill chunks, the rest one decode row each; block_tables and
    context_lens hold the prefill sequences first.  Host copies of cu_seqlens
    and context_lens (numpy int32) let the library pick the SM split."""
    import torch
    L = lib()
    T, Hq, d = q.shape
    NB, Hkv, bs, _ = k_cache.shape
    S = context_lens.shape[0]
    num_decode = S - num_prefill
    if cu_seqlens_host is not None:
        cu_seqlens_host = np.ascontiguousarray(cu_seqlens_host, dtype=np.int32)
        prefill_tokens = int(cu_seqlens_host[num_prefill])
    else:
        prefill_tokens = T - num_decode
    if context_lens_host is not None:
        context_lens_host = np.ascontiguousarray(context_lens_host, dtype=np.int32)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if workspace is None:
        workspace = torch.empty(max(16, decode_workspace_size(num_decode, Hq, Hkv, d)), dtype=torch.uint8,
                                device=q.device)
    hp = lambda a: None if a is None else a.ctypes.data_as(ctypes.c_void_p)
    st = L.pkv_paged_mixed_attention(
        _dev(out, "out", ndim=3), _dev(q, "q", ndim=3), _dev(cu_seqlens, "cu_seqlens", torch.int32, 1), num_prefill,
        prefill_tokens, int(max_q_len), num_decode, _dev(k_cache, "k_cache", q.dtype, 4),
        _dev(v_cache, "v_cache", q.dtype, 4), _dev(block_tables, "block_tables", torch.int32, 2),
        block_tables.shape[1], _dev(context_lens, "context_lens", torch.int32, 1), NB, Hq, Hkv, d, bs, float(scale),
        _dtype_code(q), _dtype_code(out), _dev(workspace, "workspace"), workspace.numel(), hp(cu_seqlens_host),
        hp(context_lens_host), int(decode_sms), _status_ptr(dev_status), _stream(stream))
    _check("pkv_paged_mixed_attention", st)


def paged_mixed_append_attention(out, q, k_new, v_new, slot_mapping, cu_seqlens, num_prefill, max_q_len, k_cache,
                                 v_cache, block_tables, context_lens, scale=None, workspace=None, cu_seqlens_host=None,
                                 context_lens_host=None, decode_sms=0, dev_status=None, stream=None):
    """pkv_paged_mixed_append_attention: the append of k_new/v_new (rows as q;
    prefill rows by slot_mapping, int64 [prefill tokens]; decode rows at
    position context_lens - 1) and the mixed step's attention in one call."""
    import torch
    L = lib()
    T, Hq, d = q.shape
    NB, Hkv, bs, _ = k_cache.shape
    S = context_lens.shape[0]
    num_decode = S - num_prefill
    if cu_seqlens_host is not None:
        cu_seqlens_host = np.ascontiguousarray(cu_seqlens_host, dtype=np.int32)
        prefill_tokens = int(cu_seqlens_host[num_prefill])
    else:
        prefill_tokens = T - num_decode
    if context_lens_host is not None:
        context_lens_host = np.ascontiguousarray(context_lens_host, dtype=np.int32)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if workspace is None:
        workspace = torch.empty(max(16, decode_workspace_size(num_decode, Hq, Hkv, d)), dtype=torch.uint8,
                                device=q.device)
    hp = lambda a: None if a is None else a.ctypes.data_as(ctypes.c_void_p)
    st = L.pkv_paged_mixed_append_attention(
        _dev(out, "out", ndim=3), _dev(q, "q", ndim=3), _dev(k_new, "k_new", q.dtype, 3),
        _dev(v_new, "v_new", q.dtype, 3), _dev(slot_mapping, "slot_mapping", torch.int64, 1),
        _dev(cu_seqlens, "cu_seqlens", torch.int32, 1), num_prefill, prefill_tokens, int(max_q_len), num_decode,
        _dev(k_cache, "k_cache", q.dtype, 4), _dev(v_cache, "v_cache", q.dtype, 4),
        _dev(block_tables, "block_tables", torch.int32, 2), block_tables.shape[1],
        _dev(context_lens, "context_lens", torch.int32, 1), NB, Hq, Hkv, d, bs, float(scale), _dtype_code(q),
        _dtype_code(out), _dev(workspace, "workspace"), workspace.numel(), hp(cu_seqlens_host),
        hp(context_lens_host), int(decode_sms), _status_ptr(dev_status), _stream(stream))
    _check("pkv_paged_mixed_append_attention", st)


def copy_blocks(dst, src, pairs, dev_status=None, stream=None):
    """pkv_copy_blocks: dst, src [blocks, ...] tensors (CUDA or pinned CPU) with
    equal block shapes; pairs int32 [n, 2] (source block, destination block),
    on the device or pinned."""
    import torch
    if dst.shape[1:] != src.shape[1:] or dst.dtype != src.dtype:
        raise ValueError("dst and src must hold blocks of one shape and dtype")
    for name, t in (("dst", dst), ("src", src), ("pairs", pairs)):
        if not t.is_contiguous() or not (t.is_cuda or t.is_pinned()):
            raise ValueError("%s must be contiguous, on the GPU or pinned" % name)
    if pairs.dtype != torch.int32 or pairs.dim() != 2 or pairs.shape[1] != 2:
        raise ValueError("pairs must be int32 [n, 2]")
    block_bytes = dst[0].numel() * dst.element_size()
    st = lib().pkv_copy_blocks(ctypes.c_void_p(dst.data_ptr()), dst.shape[0], ctypes.c_void_p(src.data_ptr()),
                               src.shape[0], ctypes.c_void_p(pairs.data_ptr()), pairs.shape[0], block_bytes,
                               _status_ptr(dev_status), _stream(stream))
    _check("pkv_copy_blocks", st)


def mixed_split(num_sms, cu_seqlens, num_prefill, context_lens, num_q_heads, num_kv_heads, head_dim, elem_bytes=2):
    """pkv_mixed_split on host arrays: the SMs the decode kernel gets."""
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    r = lib().pkv_mixed_split(num_sms, cu.ctypes.data_as(ctypes.c_void_p), num_prefill,
                              cl.ctypes.data_as(ctypes.c_void_p), len(cl) - num_prefill, num_q_heads, num_kv_heads,
                              head_dim, elem_bytes)
    if r < 0:
        raise PkvError("pkv_mixed_split", r)
    return r


# ------------------------------------------------------------ host pool / scheduler

class BlockPool:
    """pkv_pool_*: LIFO free list of physical block ids (host only)."""

    def __init__(self, num_blocks, initial_order=None):
        L = lib()
        self._keep = None
        ptr = None
        if initial_order is not None:
            self._keep = np.ascontiguousarray(initial_order, dtype=np.int32)
            ptr = self._keep.ctypes.data_as(ctypes.c_void_p)
        self._h = L.pkv_pool_create(num_blocks, ptr)
        if not self._h:
            raise ValueError("pkv_pool_create rejected its arguments")

    def __del__(self):
        if getattr(self, "_h", None) and _lib is not None:
            _lib.pkv_pool_destroy(self._h)
            self._h = None

    def alloc(self, n):
        out = np.empty(max(n, 1), dtype=np.int32)
        st = lib().pkv_pool_alloc(self._h, n, out.ctypes.data_as(ctypes.c_void_p))
        _check("pkv_pool_alloc", st)
        return out[:n].tolist()

    def free(self, ids):
        a = np.ascontiguousarray(ids, dtype=np.int32)
        _check("pkv_pool_free", lib().pkv_pool_free(self._h, a.ctypes.data_as(ctypes.c_void_p), a.size))

    def free_count(self):
        return lib().pkv_pool_free_count(self._h)

    def free_list(self):
        out = np.empty(max(self.free_count(), 1), dtype=np.int32)
        n = lib().pkv_pool_free_list(self._h, out.ctypes.data_as(ctypes.c_void_p))
        return out[:n].tolist()

    def inject_failure(self, nth):
        _check("pkv_pool_inject_failure", lib().pkv_pool_inject_failure(self._h, nth))


class Scheduler:
    """pkv_sched_*: the native iteration-level scheduler (host only)."""

    def __init__(self, num_blocks, block_size=16, max_batch=256, max_num_batched_tokens=8192, chunk=512,
                 max_model_len=8192, initial_order=None, policy=SCHED_CONTINUOUS, prefix_caching=False,
                 preemption=PREEMPT_RECOMPUTE, swap_blocks=0):
        L = lib()
        self._keep = None
        cfg = SchedConfig(num_blocks, block_size, max_batch, max_num_batched_tokens, chunk, max_model_len, None,
                          policy, 1 if prefix_caching else 0, preemption, swap_blocks)
        if initial_order is not None:
            self._keep = np.ascontiguousarray(initial_order, dtype=np.int32)
            cfg.initial_order = self._keep.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))
        self._h = L.pkv_sched_create(ctypes.byref(cfg))
        if not self._h:
            raise ValueError("pkv_sched_create rejected its configuration")
        self.max_blocks = -(-max_model_len // block_size)

    def __del__(self):
        if getattr(self, "_h", None) and _lib is not None:
            _lib.pkv_sched_destroy(self._h)
            self._h = None

    def add(self, rid, prompt_len, max_tokens, eos_after, tokens=None):
        if tokens is None:
            _check("pkv_sched_add", lib().pkv_sched_add(self._h, rid, prompt_len, max_tokens, eos_after))
            return
        t = np.ascontiguousarray(tokens, dtype=np.int32)
        if t.shape != (prompt_len,):
            raise ValueError("tokens must hold prompt_len ids")
        _check("pkv_sched_add_tokens", lib().pkv_sched_add_tokens(self._h, rid, t.ctypes.data_as(ctypes.c_void_p),
                                                                  prompt_len, max_tokens, eos_after))

    def step_raw(self):
        """One step; returns the raw StepMeta (arrays valid until the next step)."""
        meta = StepMeta()
        n = lib().pkv_sched_step(self._h, ctypes.byref(meta))
        if n < 0:
            raise PkvError("pkv_sched_step", n)
        return meta

    def step(self):
        """One step; returns a dict of numpy copies of the metadata, or None
        when nothing was scheduled or copied."""
        m = self.step_raw()
        if m.num_seqs == 0 and m.num_swap_out == 0 and m.num_swap_in == 0:
            return None
        S, T, MB = m.num_seqs, m.num_tokens, m.max_blocks

        def arr(ptr, n, dt):
            if n == 0:   # nothing scheduled (a step that only swapped): the pointers may be null
                return np.zeros(0, dt)
            return np.ctypeslib.as_array(ptr, shape=(n,)).astype(dt, copy=True)

        return {
            "seq_rids": arr(m.seq_rids, S, np.int64), "q_lens": arr(m.q_lens, S, np.int32),
            "context_lens": arr(m.context_lens, S, np.int32), "cu_seqlens": arr(m.cu_seqlens, S + 1, np.int32),
            "block_tables": arr(m.block_tables, S * MB, np.int32).reshape(S, MB),
            "slot_mapping": arr(m.slot_mapping, T, np.int64), "token_rids": arr(m.token_rids, T, np.int64),
            "token_pos": arr(m.token_pos, T, np.int32), "num_prefill": m.num_prefill,
            "finished_rids": arr(m.finished_rids, m.num_finished, np.int64) if m.num_finished else
            np.zeros(0, np.int64),
            "swap_out": arr(m.swap_out, 2 * m.num_swap_out, np.int32).reshape(-1, 2) if m.num_swap_out else
            np.zeros((0, 2), np.int32),
            "swap_in": arr(m.swap_in, 2 * m.num_swap_in, np.int32).reshape(-1, 2) if m.num_swap_in else
            np.zeros((0, 2), np.int32),
        }

    def stats(self):
        s = SchedStats()
        _check("pkv_sched_get_stats", lib().pkv_sched_get_stats(self._h, ctypes.byref(s)))
        return {f: getattr(s, f) for f, _ in SchedStats._fields_}

    def inject_alloc_failure(self, nth):
        _check("pkv_sched_inject_alloc_failure", lib().pkv_sched_inject_alloc_failure(self._h, nth))

    def request_state(self, rid):
        g = ctypes.c_int(0)
        st = lib().pkv_sched_request_state(self._h, rid, ctypes.byref(g))
        return st, g.value

    def forget(self, rid):
        """pkv_sched_forget: drop a finished request's record."""
        _check("pkv_sched_forget", lib().pkv_sched_forget(self._h, rid))
