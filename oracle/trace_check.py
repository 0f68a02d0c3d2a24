"""Oracle values for sampled rows of the continuous-batching trace.

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).  Rebuilds, from the
counter-based generator in synth.trace, the K/V rows that layer 0's cache
must hold for one request and runs the FP64 oracle for one query position
over keys 0..pos (for a decode row pos = ctx - 1; for a prefill-chunk row the
causal bound is the row's own position).
"""
import numpy as np

from synth import NAN_BITS
from synth.trace import kv_tag, q_tag, token_rows

from . import decode


def layer0_inputs(rid, pos, Hq, Hkv, d, dtype="bf16", keys=None):
    """The oracle's inputs for one sampled row: (q, k_cache, v_cache,
    block_table, context_len) of that row alone, its layer-0 K/V rebuilt from
    the generator.  keys(positions) -> the row keys of the request's tokens
    (default: the request id; a shared prompt head uses its group's key)."""
    n = pos + 1
    nb = -(-n // 16)
    kk = np.full(n, rid) if keys is None else keys(np.arange(n))
    ks = token_rows(kk, np.arange(n), kv_tag(0, "k"), Hkv * d, dtype).reshape(n, Hkv, d)
    vs = token_rows(kk, np.arange(n), kv_tag(0, "v"), Hkv * d, dtype).reshape(n, Hkv, d)
    kc = np.full((nb * 16, Hkv, d), NAN_BITS[dtype], np.uint16)
    vc = kc.copy()
    kc[:n], vc[:n] = ks, vs
    kc = kc.reshape(nb, 16, Hkv, d).transpose(0, 2, 1, 3).copy()
    vc = vc.reshape(nb, 16, Hkv, d).transpose(0, 2, 1, 3).copy()
    qk = np.array([rid]) if keys is None else keys(np.array([pos]))
    q = token_rows(qk, np.array([pos]), q_tag(0), Hq * d, dtype).reshape(1, Hq, d)
    return q, kc, vc, np.arange(nb, dtype=np.int32)[None], np.array([n], np.int32)


def layer0_row(rid, pos, Hq, Hkv, d, dtype="bf16", keys=None):
    """The FP64 oracle's output [Hq, d] for one sampled row."""
    return decode(*layer0_inputs(rid, pos, Hq, Hkv, d, dtype, keys), dtype)[0]
