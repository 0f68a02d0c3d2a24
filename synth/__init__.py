"""Seeded synthetic inputs for paged KV-cache attention steps.

This module only makes inputs: random 16-bit values, context lengths, block
assignments from a shuffled pool, and the per-step metadata arrays that point
at them.  It holds none of the attention arithmetic, and both the CUDA path's
tests/benchmark and the oracle consume exactly the arrays it returns.

Value recipe: fp32 draws from N(0, 1) (numpy PCG64), rounded to fp16 with
numpy's IEEE round-to-nearest-even cast, or to bfloat16 by round-to-nearest-
even on the fp32 bit pattern.  Pool slots that hold no token (free blocks, the
tail of a sequence's last block) are filled with a NaN bit pattern so that any
stray read shows up.

Workloads (seed = 1000 + index unless given):
  tiny     2 decode sequences, prior contexts 17 and 14 (the prompt lengths of
           tiny-vllm's queue), one new token each -> attended 18 and 15;
           4 query = 4 KV heads, head_dim 64, 16-token blocks, 64-block pool
           assigned by a seeded permutation, fp16.
  llama1b  64 decode sequences, context ~ U{128..2048}, 32/8 heads, d 64,
           16k-block pool, blocks drawn at random, bf16.
  llama8b  256 decode sequences, context = clip(rint(exp(ln 1024 + z)), 32,
           8192) with z ~ N(0, 1), 32/8 heads, d 128, 64k-block pool popped
           from a seeded shuffled free list, bf16.
  mixed    8 prefill chunks of 512 tokens with prior context ~ U{0..4096}
           plus 248 decode sequences with context ~ U{256..4096}; 32/8 heads,
           d 128, 64k-block pool, bf16; all 4344 new tokens appended by
           slot mapping.
"""
from dataclasses import dataclass, field
from typing import Optional

import numpy as np

BLOCK_SIZE = 16
NAN_BITS = {"fp16": np.uint16(0x7E00), "bf16": np.uint16(0x7FC0)}


def rne_bits(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round float32 values to fp16/bf16 (nearest, ties to even); uint16 bits."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    if dtype == "fp16":
        return x.astype(np.float16).view(np.uint16)
    if dtype == "bf16":
        u = x.view(np.uint32)
        bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
        return ((u + bias) >> np.uint32(16)).astype(np.uint16)
    raise ValueError(dtype)


def bits_to_float32(bits: np.ndarray, dtype: str) -> np.ndarray:
    """Widen fp16/bf16 bit patterns to float32 (exact)."""
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    if dtype == "fp16":
        return bits.view(np.float16).astype(np.float32)
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)


@dataclass
class Step:
    """One engine step's inputs.  New tokens are ordered prefill chunks first
    (sequences 0 .. n_prefill-1), then decode sequences (one token each)."""
    name: str
    dtype: str
    Hq: int
    Hkv: int
    d: int
    bs: int
    NB: int
    context_lens: np.ndarray          # int32 [S], includes this step's new tokens
    q_lens: np.ndarray                # int32 [S], new tokens per sequence
    block_tables: np.ndarray          # int32 [S, max_blocks], -1 padded
    slot_mapping: np.ndarray          # int64 [T]
    cu_seqlens: np.ndarray            # int32 [S+1], prefix sum of q_lens
    q: np.ndarray                     # uint16 [T, Hq, d]
    k_new: np.ndarray                 # uint16 [T, Hkv, d]
    v_new: np.ndarray                 # uint16 [T, Hkv, d]
    k_cache: np.ndarray               # uint16 [NB, Hkv, bs, d], prior tokens filled
    v_cache: np.ndarray
    n_prefill: int = 0
    meta: dict = field(default_factory=dict)

    @property
    def S(self) -> int:
        return int(self.context_lens.shape[0])

    @property
    def T(self) -> int:
        return int(self.slot_mapping.shape[0])

    @property
    def max_blocks(self) -> int:
        return int(self.block_tables.shape[1])

    def decode_part(self):
        """Views of the decode sequences: (q, block_tables, context_lens)."""
        p = self.n_prefill
        t0 = int(self.cu_seqlens[p])
        return self.q[t0:], self.block_tables[p:], self.context_lens[p:]

    def prefill_part(self):
        """Views of the prefill chunks: (q, cu_seqlens, block_tables, context_lens)."""
        p = self.n_prefill
        t1 = int(self.cu_seqlens[p])
        return self.q[:t1], self.cu_seqlens[: p + 1], self.block_tables[:p], self.context_lens[:p]


def build_step(name: str, rng: np.random.Generator, *, ctx, q_lens, Hq: int, Hkv: int, d: int,
               NB: int, dtype: str, pool_order: np.ndarray, bs: int = BLOCK_SIZE,
               n_prefill: int = 0, max_blocks: Optional[int] = None,
               chunk_blocks: int = 2048) -> Step:
    """Generic step builder.  Sequence s attends ctx[s] tokens of which the last
    q_lens[s] are new this step (written by append); its blocks are the next
    ceil(ctx/bs) ids of pool_order."""
    ctx = np.asarray(ctx, dtype=np.int64)
    q_lens = np.asarray(q_lens, dtype=np.int64)
    S = ctx.shape[0]
    assert np.all(q_lens <= ctx) and np.all(q_lens >= 0)
    nblk = (ctx + bs - 1) // bs
    total_blocks = int(nblk.sum())
    if total_blocks > NB:
        raise ValueError("pool too small: need %d blocks, have %d" % (total_blocks, NB))
    if max_blocks is None:
        max_blocks = max(1, int(nblk.max()) if S else 1)
    ids = np.asarray(pool_order[:total_blocks], dtype=np.int32)
    block_tables = np.full((S, max_blocks), -1, dtype=np.int32)
    starts = np.zeros(S + 1, dtype=np.int64)
    starts[1:] = np.cumsum(nblk)
    for s in range(S):
        block_tables[s, : nblk[s]] = ids[starts[s]: starts[s + 1]]

    cu = np.zeros(S + 1, dtype=np.int32)
    cu[1:] = np.cumsum(q_lens)
    T = int(cu[-1])
    # positions of the new tokens and their slots
    slot_mapping = np.empty(T, dtype=np.int64)
    for s in range(S):
        pos = np.arange(ctx[s] - q_lens[s], ctx[s], dtype=np.int64)
        slot_mapping[cu[s]: cu[s + 1]] = block_tables[s, pos // bs].astype(np.int64) * bs + pos % bs

    q = rne_bits(rng.standard_normal((T, Hq, d), dtype=np.float32), dtype)
    k_new = rne_bits(rng.standard_normal((T, Hkv, d), dtype=np.float32), dtype)
    v_new = rne_bits(rng.standard_normal((T, Hkv, d), dtype=np.float32), dtype)

    nan = NAN_BITS[dtype]
    k_cache = np.full((NB, Hkv, bs, d), nan, dtype=np.uint16)
    v_cache = np.full((NB, Hkv, bs, d), nan, dtype=np.uint16)
    # logical index and owner of every assigned block, in pool order
    owner = np.repeat(np.arange(S), nblk)
    logical = np.arange(total_blocks) - starts[owner]
    prior = (ctx - q_lens)[owner]
    offs = np.arange(bs)
    for b0 in range(0, total_blocks, chunk_blocks):
        b1 = min(total_blocks, b0 + chunk_blocks)
        n = b1 - b0
        # positions at or beyond the prior context are not yet stored
        keep = (logical[b0:b1, None] * bs + offs[None, :]) < prior[b0:b1, None]   # [n, bs]
        for cache in (k_cache, v_cache):
            vals = rne_bits(rng.standard_normal((n, Hkv, bs, d), dtype=np.float32), dtype)
            vals = np.where(keep[:, None, :, None], vals, nan)
            cache[ids[b0:b1]] = vals
    return Step(name=name, dtype=dtype, Hq=Hq, Hkv=Hkv, d=d, bs=bs, NB=NB,
                context_lens=ctx.astype(np.int32), q_lens=q_lens.astype(np.int32),
                block_tables=block_tables, slot_mapping=slot_mapping, cu_seqlens=cu, q=q,
                k_new=k_new, v_new=v_new, k_cache=k_cache, v_cache=v_cache, n_prefill=n_prefill)


SEEDS = {"tiny": 1000, "llama1b": 1001, "llama8b": 1002, "mixed": 1003, "trace": 1004}


def llama8b_context_lens(rng: np.random.Generator, S: int) -> np.ndarray:
    z = rng.standard_normal(S)
    return np.clip(np.rint(np.exp(np.log(1024.0) + z)), 32, 8192).astype(np.int64)


def make_step(name: str, seed: Optional[int] = None, **over) -> Step:
    """One of the named workloads (see the module docstring)."""
    seed = SEEDS[name] if seed is None else seed
    rng = np.random.Generator(np.random.PCG64(seed))
    if name == "tiny":
        prior = np.array(over.pop("prior", [17, 14]), dtype=np.int64)
        ctx = prior + 1
        NB = 64
        order = rng.permutation(NB)
        return build_step(name, rng, ctx=ctx, q_lens=np.ones_like(ctx), Hq=4, Hkv=4, d=64, NB=NB,
                          dtype="fp16", pool_order=order, **over)
    if name == "llama1b":
        S = over.pop("S", 64)
        ctx = rng.integers(128, 2048, size=S, endpoint=True)
        NB = 16384
        order = rng.permutation(NB)
        return build_step(name, rng, ctx=ctx, q_lens=np.ones_like(ctx), Hq=32, Hkv=8, d=64, NB=NB,
                          dtype="bf16", pool_order=order, **over)
    if name == "llama8b":
        S = over.pop("S", 256)
        NB = over.pop("NB", 65536)
        ctx = llama8b_context_lens(rng, S)
        # seeded shuffled free list, popped from the end per sequence
        order = rng.permutation(NB)[::-1]
        return build_step(name, rng, ctx=ctx, q_lens=np.ones_like(ctx), Hq=32, Hkv=8, d=128, NB=NB,
                          dtype="bf16", pool_order=order, **over)
    if name == "mixed":
        n_chunks = over.pop("n_chunks", 8)
        chunk = over.pop("chunk", 512)
        n_dec = over.pop("n_decode", 248)
        NB = over.pop("NB", 65536)
        prior_p = rng.integers(0, 4096, size=n_chunks, endpoint=True)
        fixed = over.pop("prior_fixed", None)
        if fixed is not None:   # profiling case: every chunk behind the same prior context
            prior_p = np.full(n_chunks, int(fixed), dtype=prior_p.dtype)
        ctx_d = rng.integers(256, 4096, size=n_dec, endpoint=True)
        ctx = np.concatenate([prior_p + chunk, ctx_d])
        q_lens = np.concatenate([np.full(n_chunks, chunk), np.ones(n_dec, dtype=np.int64)])
        order = rng.permutation(NB)
        return build_step(name, rng, ctx=ctx, q_lens=q_lens, Hq=32, Hkv=8, d=128, NB=NB,
                          dtype="bf16", pool_order=order, n_prefill=n_chunks, **over)
    raise ValueError(name)
