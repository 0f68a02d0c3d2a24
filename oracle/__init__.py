"""FP64 CPU oracle for paged KV-cache attention and for the host scheduler.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  It shares no code
with the CUDA path (``paged_kv_cache_tables_gb300``) and imports nothing from
it; the two meet only through the seeded input generators in ``synth``.

The attention functions wrap ``oracle.c`` (plain scalar loops in double
precision) through ctypes; the scheduler restatement lives in
``oracle/sched.py``.  16-bit tensors are passed as numpy ``uint16`` bit
patterns with a dtype name ("fp16" or "bf16").
"""
import ctypes
import math
import os

import numpy as np

from . import build as _build

_DT = {"fp16": 0, "bf16": 1}
_lib = None


def _open(path):
    """Open a compiled oracle library and declare its C signatures."""
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    I = ctypes.c_int
    D = ctypes.c_double
    L = ctypes.c_int64
    lib.oracle_decode_bits.argtypes = [P, L, I, P]
    lib.oracle_decode_bits.restype = None
    lib.oracle_append.argtypes = [P, P, P, I, P, P, I, I, I, I]
    lib.oracle_append.restype = L
    lib.oracle_decode.argtypes = [P, P, P, P, I, P, I, I, I, I, I, D, I, P]
    lib.oracle_decode.restype = I
    lib.oracle_decode_range.argtypes = [P, P, P, P, I, I, I, I, I, I, D, I, P, P, P]
    lib.oracle_decode_range.restype = I
    lib.oracle_merge.argtypes = [I, P, P, P, I, P]
    lib.oracle_merge.restype = None
    lib.oracle_prefill.argtypes = [P, P, I, P, P, P, I, P, I, I, I, I, D, I, P]
    lib.oracle_prefill.restype = I
    lib.oracle_dense.argtypes = [P, P, P, I, I, I, I, D, I, P]
    lib.oracle_dense.restype = I
    return lib


def _load():
    global _lib
    if _lib is None:
        _lib = _open(_build.build())
    return _lib


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a, a.ctypes.data_as(ctypes.c_void_p)


def default_scale(d: int) -> float:
    """1/sqrt(head_dim), the scale of Project 17 Step 6."""
    return 1.0 / math.sqrt(d)


def to_double(bits, dtype: str) -> np.ndarray:
    """Exact decode of fp16/bf16 bit patterns to float64 (same shape)."""
    lib = _load()
    b, pb = _c(bits, np.uint16)
    out = np.empty(b.shape, dtype=np.float64)
    lib.oracle_decode_bits(pb, b.size, _DT[dtype], out.ctypes.data_as(ctypes.c_void_p))
    return out


def append(k, v, slot_mapping, k_cache, v_cache, block_size: int) -> int:
    """Write k[t], v[t] ([T, Hkv, d] uint16 bits) into the caches in place
    ([NB, Hkv, bs, d] uint16 bits) at slot_mapping[t]; negative slots skip.
    Returns the number of (token, head) rows written."""
    lib = _load()
    T, Hkv, d = k.shape
    NB = k_cache.shape[0]
    assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
    assert k_cache.dtype == np.uint16 and v_cache.dtype == np.uint16
    k, pk = _c(k, np.uint16)
    v, pv = _c(v, np.uint16)
    sm, ps = _c(slot_mapping, np.int64)
    n = lib.oracle_append(pk, pv, ps, T, k_cache.ctypes.data_as(ctypes.c_void_p),
                          v_cache.ctypes.data_as(ctypes.c_void_p), NB, block_size, Hkv, d)
    if n < 0:
        raise ValueError("slot outside the pool")
    return int(n)


def copy_blocks(src, dst, pairs) -> None:
    """Preemption by swap ("Continuous Batching" §5 "Preemption"): block
    pairs[i][0] of src is copied whole into block pairs[i][1] of dst, in
    order (a block is [Hkv][block_size][d] of one cache)."""
    for s, d in np.asarray(pairs).reshape(-1, 2):
        dst[int(d)] = src[int(s)]


def decode(q, k_cache, v_cache, block_tables, context_lens, dtype: str, scale=None) -> np.ndarray:
    """Paged decode attention; q [S, Hq, d] bits, caches [NB, Hkv, bs, d] bits,
    block_tables [S, max_blocks] int32, context_lens [S] int32 -> float64 [S, Hq, d]."""
    lib = _load()
    S, Hq, d = q.shape
    _, Hkv, bs, _ = k_cache.shape
    scale = default_scale(d) if scale is None else float(scale)
    q, pq = _c(q, np.uint16)
    kc, pk = _c(k_cache, np.uint16)
    vc, pv = _c(v_cache, np.uint16)
    bt, pb = _c(block_tables, np.int32)
    cl, pc = _c(context_lens, np.int32)
    out = np.zeros((S, Hq, d), dtype=np.float64)
    rc = lib.oracle_decode(pq, pk, pv, pb, bt.shape[1] if bt.ndim == 2 else 0, pc, S, Hq, Hkv, d, bs,
                           scale, _DT[dtype], out.ctypes.data_as(ctypes.c_void_p))
    if rc != 0:
        raise ValueError("oracle_decode: bad shapes")
    return out


def decode_range(q_s, k_cache, v_cache, block_row, t0: int, t1: int, dtype: str, scale=None):
    """Partial attention of one sequence's query heads q_s [Hq, d] over logical
    tokens [t0, t1): returns (m [Hq], l [Hq], acc [Hq, d]), natural-log domain."""
    lib = _load()
    Hq, d = q_s.shape
    _, Hkv, bs, _ = k_cache.shape
    scale = default_scale(d) if scale is None else float(scale)
    q_s, pq = _c(q_s, np.uint16)
    kc, pk = _c(k_cache, np.uint16)
    vc, pv = _c(v_cache, np.uint16)
    br, pb = _c(block_row, np.int32)
    m = np.empty(Hq, np.float64)
    l = np.empty(Hq, np.float64)
    acc = np.empty((Hq, d), np.float64)
    rc = lib.oracle_decode_range(pq, pk, pv, pb, t0, t1, Hq, Hkv, d, bs, scale, _DT[dtype],
                                 m.ctypes.data_as(ctypes.c_void_p), l.ctypes.data_as(ctypes.c_void_p),
                                 acc.ctypes.data_as(ctypes.c_void_p))
    if rc != 0:
        raise ValueError("oracle_decode_range: bad shapes")
    return m, l, acc


def merge(m, l, acc) -> np.ndarray:
    """Log-sum-exp merge of partials m [n], l [n], acc [n, d] -> [d]."""
    lib = _load()
    m, pm = _c(m, np.float64)
    l, pl = _c(l, np.float64)
    acc, pa = _c(acc, np.float64)
    n, d = acc.shape
    out = np.empty(d, np.float64)
    lib.oracle_merge(n, pm, pl, pa, d, out.ctypes.data_as(ctypes.c_void_p))
    return out


def prefill(q, cu_seqlens, k_cache, v_cache, block_tables, context_lens, dtype: str,
            scale=None) -> np.ndarray:
    """Paged prefill attention, causal over prior context plus the chunk.
    q [total_q, Hq, d] bits; cu_seqlens [S+1]; returns float64 [total_q, Hq, d]."""
    lib = _load()
    total, Hq, d = q.shape
    _, Hkv, bs, _ = k_cache.shape
    S = len(cu_seqlens) - 1
    scale = default_scale(d) if scale is None else float(scale)
    q, pq = _c(q, np.uint16)
    cu, pcu = _c(cu_seqlens, np.int32)
    kc, pk = _c(k_cache, np.uint16)
    vc, pv = _c(v_cache, np.uint16)
    bt, pb = _c(block_tables, np.int32)
    cl, pc = _c(context_lens, np.int32)
    out = np.zeros((total, Hq, d), dtype=np.float64)
    rc = lib.oracle_prefill(pq, pcu, S, pk, pv, pb, bt.shape[1], pc, Hq, Hkv, d, bs, scale,
                            _DT[dtype], out.ctypes.data_as(ctypes.c_void_p))
    if rc != 0:
        raise ValueError("oracle_prefill: bad shapes or q_len > ctx")
    return out


def dense(q_s, k, v, dtype: str, scale=None) -> np.ndarray:
    """Attention of q_s [Hq, d] over contiguous k, v [ctx, Hkv, d] (no table)."""
    lib = _load()
    Hq, d = q_s.shape
    ctx, Hkv, _ = k.shape
    scale = default_scale(d) if scale is None else float(scale)
    q_s, pq = _c(q_s, np.uint16)
    k, pk = _c(k, np.uint16)
    v, pv = _c(v, np.uint16)
    out = np.empty((Hq, d), np.float64)
    rc = lib.oracle_dense(pq, pk, pv, ctx, Hq, Hkv, d, scale, _DT[dtype],
                          out.ctypes.data_as(ctypes.c_void_p))
    if rc != 0:
        raise ValueError("oracle_dense: bad shapes")
    return out
