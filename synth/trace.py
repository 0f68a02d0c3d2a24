"""Seeded continuous-batching trace and counter-based synthetic token rows.

Input generation only (no attention arithmetic).  The trace: requests arrive
as a Poisson process of `rate` per engine step; prompt lengths are
lognormal with mean `prompt_mean` (sigma 1, mu = ln(mean) - sigma^2 / 2)
rounded and clipped to [8, 4096]; output lengths (the step at which the
request emits EOS) are geometric with mean `out_mean`, at least 1.

Token rows: K, V and Q of token (request, position) are a pure function of
(request, position, tag, element), so any token can be regenerated anywhere
-- on the GPU by synth/csrc/synth_fill.cu while the trace runs, and here in
numpy to rebuild what the cache must hold for the oracle.  The hash is
Wellons' "lowbias32"; values are uniform on [-2, 2) rounded to nearest even.
K/V rows of a layer depend on the physical cache that layer writes (tag), so
every layer that shares a cache stores the same rows.
"""
import ctypes
import os

import numpy as np

from . import rne_bits

HASH_SEED = 0x5EED1234
_M1, _M2 = np.uint32(0x7FEB352D), np.uint32(0x846CA68B)


def lowbias32(x: np.ndarray) -> np.ndarray:
    x = np.asarray(x, dtype=np.uint32).copy()
    with np.errstate(over="ignore"):
        x ^= x >> np.uint32(16)
        x *= _M1
        x ^= x >> np.uint32(15)
        x *= _M2
        x ^= x >> np.uint32(16)
    return x


def kv_tag(cache_id: int, which: str) -> int:
    """Tag of K ("k") or V ("v") rows stored in physical cache cache_id."""
    return (cache_id << 2) | (0 if which == "k" else 1)


def q_tag(layer: int) -> int:
    return (layer << 2) | 2


def token_rows(rids, pos, tag: int, width: int, dtype: str = "bf16") -> np.ndarray:
    """uint16 bit patterns [n, width] of the rows of tokens (rids[i], pos[i])."""
    rids = np.asarray(rids, dtype=np.int64)
    pos = np.asarray(pos, dtype=np.int64)
    b = lowbias32(np.uint32(HASH_SEED) ^ (rids & 0xFFFFFFFF).astype(np.uint32))
    b = lowbias32(b ^ (pos & 0xFFFFFFFF).astype(np.uint32))
    b = lowbias32(b ^ np.uint32(tag))
    e = np.arange(width, dtype=np.uint32)
    h = lowbias32(b[:, None] ^ e[None, :])
    x = (h >> np.uint32(8)).astype(np.float32) * np.float32(1.0 / 16777216.0) * np.float32(4.0) - np.float32(2.0)
    return rne_bits(x, dtype)


def make_requests(seed: int, n: int = 1000, rate: float = 20.0, prompt_mean: float = 512.0,
                  sigma: float = 1.0, out_mean: float = 256.0, pmin: int = 8, pmax: int = 4096,
                  outputs: str = "geometric"):
    """Returns arrival_step, prompt_len, eos_after (int64 arrays of length n).
    Output lengths are geometric with mean out_mean, or (outputs="lognormal")
    lognormal with mean out_mean and the prompts' sigma, at least 1."""
    rng = np.random.Generator(np.random.PCG64(seed))
    arrival = np.empty(n, dtype=np.int64)
    k, step = 0, 0
    while k < n:
        m = int(rng.poisson(rate))
        take = min(m, n - k)
        arrival[k:k + take] = step
        k += take
        step += 1
    mu = np.log(prompt_mean) - sigma * sigma / 2
    prompt = np.clip(np.rint(rng.lognormal(mu, sigma, size=n)), pmin, pmax).astype(np.int64)
    if outputs == "geometric":
        eos = rng.geometric(1.0 / out_mean, size=n).astype(np.int64)
    elif outputs == "lognormal":
        mo = np.log(out_mean) - sigma * sigma / 2
        eos = np.maximum(np.rint(rng.lognormal(mo, sigma, size=n)), 1).astype(np.int64)
    else:
        raise ValueError(outputs)
    return arrival, prompt, eos


GROUP_KEY_BASE = 0x80000000   # content keys of shared prompt heads (request ids stay below)


def make_shared_requests(seed: int, n: int = 1000, rate: float = 20.0, groups: int = 8,
                         head_mean: float = 1024.0, tail_mean: float = 128.0, sigma: float = 1.0,
                         out_mean: float = 256.0, bs: int = 16, pmax: int = 4096):
    """A sharing-heavy trace: every request belongs to one of `groups` groups
    whose prompts start with the same head (lognormal length with mean
    head_mean, rounded down to whole pages of bs tokens, at least one page),
    followed by the request's own tail (lognormal, mean tail_mean, at least 1
    token); prompts clipped to pmax.  Returns arrival, prompt_len, eos_after,
    tokens (list of int32 arrays), head_len and group (int64 arrays)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    arrival = np.empty(n, dtype=np.int64)
    k, step = 0, 0
    while k < n:
        m = int(rng.poisson(rate))
        take = min(m, n - k)
        arrival[k:k + take] = step
        k += take
        step += 1
    mh = np.log(head_mean) - sigma * sigma / 2
    heads_len = np.maximum(np.floor(rng.lognormal(mh, sigma, size=groups) / bs), 1).astype(np.int64) * bs
    heads_len = np.minimum(heads_len, (pmax // 2) // bs * bs)
    heads = [rng.integers(1, 1 << 20, size=int(h), dtype=np.int64).astype(np.int32) for h in heads_len]
    group = rng.integers(0, groups, size=n).astype(np.int64)
    mt = np.log(tail_mean) - sigma * sigma / 2
    tail = np.maximum(np.rint(rng.lognormal(mt, sigma, size=n)), 1).astype(np.int64)
    eos = rng.geometric(1.0 / out_mean, size=n).astype(np.int64)
    tokens, prompt, head_len = [], np.empty(n, np.int64), np.empty(n, np.int64)
    for i in range(n):
        t = min(int(tail[i]), pmax - int(heads_len[group[i]]))
        own = rng.integers(1 << 20, 1 << 30, size=t, dtype=np.int64).astype(np.int32)
        tokens.append(np.concatenate([heads[group[i]], own]))
        prompt[i] = len(tokens[-1])
        head_len[i] = heads_len[group[i]]
    return arrival, prompt, eos, tokens, head_len, group


def content_keys(rids, pos, head_len, group):
    """Key of the row of token (rids[i], pos[i]): inside its request's shared
    head the group's key (the same prefix has the same K/V whichever request
    computed it), else the request id."""
    rids = np.asarray(rids, dtype=np.int64)
    pos = np.asarray(pos, dtype=np.int64)
    return np.where(pos < head_len[rids], GROUP_KEY_BASE + group[rids], rids)


# ---------------------------------------------------------------- GPU generator

_lib = None


def _gpu_lib():
    global _lib
    if _lib is None:
        path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libsynth.so")
        if not os.path.exists(path):
            raise RuntimeError("synth/libsynth.so is not built; run synth.build.build()")
        L = ctypes.CDLL(path)
        L.synth_fill_rows.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                                      ctypes.c_uint32, ctypes.c_uint32, ctypes.c_int, ctypes.c_void_p]
        L.synth_fill_rows.restype = ctypes.c_int
        L.synth_fill_qkv.argtypes = [ctypes.c_void_p] * 5 + [ctypes.c_int] * 3 + [ctypes.c_uint32] * 4 + \
            [ctypes.c_int, ctypes.c_void_p]
        L.synth_fill_qkv.restype = ctypes.c_int
        _lib = L
    return _lib


def fill_rows_gpu(out, rids, pos, tag: int, stream=None) -> None:
    """Fill CUDA tensor out [n, ...] (bf16/fp16) with token_rows(rids, pos, tag)."""
    import torch
    n = out.shape[0]
    width = out.numel() // max(n, 1)
    s = stream if stream is not None else torch.cuda.current_stream()
    rc = _gpu_lib().synth_fill_rows(ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(rids.data_ptr()),
                                    ctypes.c_void_p(pos.data_ptr()), n, width, HASH_SEED, tag,
                                    1 if out.dtype == torch.bfloat16 else 0, ctypes.c_void_p(s.cuda_stream))
    if rc != 0:
        raise RuntimeError("synth_fill_rows failed")


def fill_qkv_gpu(q, k, v, rids, pos, tq: int, tk: int, tv: int, stream=None) -> None:
    """fill_rows_gpu of q, k and v (tags tq, tk, tv) in one launch."""
    import torch
    n = q.shape[0]
    s = stream if stream is not None else torch.cuda.current_stream()
    rc = _gpu_lib().synth_fill_qkv(ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()),
                                   ctypes.c_void_p(v.data_ptr()), ctypes.c_void_p(rids.data_ptr()),
                                   ctypes.c_void_p(pos.data_ptr()), n, q.numel() // max(n, 1),
                                   k.numel() // max(n, 1), HASH_SEED, tq, tk, tv,
                                   1 if q.dtype == torch.bfloat16 else 0, ctypes.c_void_p(s.cuda_stream))
    if rc != 0:
        raise RuntimeError("synth_fill_qkv failed")


def make_fill():
    """Per-layer filler for PagedEngine.step: Q rows tagged by layer, K/V rows
    by the physical cache the layer writes (one launch per layer)."""
    def fill(layer, cid, q, k, v, trids, tpos):
        fill_qkv_gpu(q, k, v, trids, tpos, q_tag(layer), kv_tag(cid, "k"), kv_tag(cid, "v"))
    return fill


def pick_rows(info, rng, n_decode=2, n_prefill=1):
    """Samples (output row, request id, position) from one step's metadata:
    a few decode rows and prefill-chunk rows."""
    S, P, cu, ctx, rids = info["S"], info["P"], info["cu_seqlens"], info["context_lens"], info["seq_rids"]
    out = []
    if S > P:
        for s in rng.choice(np.arange(P, S), size=min(n_decode, S - P), replace=False):
            out.append((int(cu[s]), int(rids[s]), int(ctx[s]) - 1))
    if P:
        for s in rng.choice(np.arange(P), size=min(n_prefill, P), replace=False):
            ql = int(cu[s + 1] - cu[s])
            i = int(rng.integers(0, ql))
            out.append((int(cu[s]) + i, int(rids[s]), int(ctx[s]) - ql + i))
    return out
