"""Plain Python restatement of the iteration-level scheduler and block pool.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).  The native scheduler in
the product library must emit exactly the same metadata, step by step, for the
same request trace.  This file is written for readability, not speed.

Sources and the reading taken where they differ:

* Block pool: a preallocated set of physical block ids and a free list used as
  a stack (pop from the end, push freed ids back on the end) -- "Project 17",
  Step 4 "Implement the paged KV cache" (BlockPool), and the free-list-as-stack
  of "Build a pure-Python continuous batching LLM serving engine", Step 2.
  Allocation of n blocks is all-or-nothing; failure is reported, never a crash.
* Step order -- retire, admit, run one iteration -- from "Project 17" Step 2
  (Scheduler.step) and "Continuous Batching" §4 (Engine.Step).
* Admission is first-come-first-served and stops at the first request that does
  not fit ("Continuous Batching" §4: break on allocation failure), with
  optimistic allocation: blocks for the tokens known now, grown as the
  sequence grows (§5 "Admission policy").  A recomputed request needs blocks
  for prompt + generated tokens, not the prompt alone.
* Per-step token budget max_num_batched_tokens and prefill chunks of at most
  `chunk` tokens riding with decodes (§5 "Mixed batching").
* Preemption by recompute: free the victim's blocks, push it to the FRONT of
  the waiting queue, re-prefill prompt + generated later (§4 preempt, §5
  "Preemption").  Victim: the most recently admitted running request (LIFO,
  §5 "Victim selection"); if that is the request that needs the block, it
  preempts itself (matching §4, where the request that needs the block is
  the one re-queued).
* Retire on EOS (a pre-drawn output length here), on max_tokens, or when the
  total length reaches max_model_len (tiny-vllm part 7 "Termination and
  returning blocks"); blocks are freed immediately (§1 lifecycle diagram).
* Context length of a scheduled sequence counts its tokens appended this step
  (tiny-vllm part 7 "Uploading the active arrays to the GPU").
* Prefix caching ("Project 17" Step 8, PrefixCache.find_prefix_match: the
  longest page-aligned prefix of the prompt found in the cache, its pages'
  reference counts raised).  Readings where the page is silent: a full prompt
  page is registered once its K/V are computed, keyed by (block of the
  preceding page, its own tokens) -- the same prefix identity as the page's
  tuple of all tokens up to it -- and only if that preceding page is the
  registered one; a match covers at most prompt_len - 1 tokens, so one prompt
  token is always computed and no request writes into a shared page; a block
  is freed when no request holds it, and leaves the cache then.
* Preemption by swap ("Continuous Batching" §5 "Preemption", SWAP: copy the
  victim's KV blocks to CPU memory, free the GPU blocks, copy back later).
  Readings: only the blocks holding computed tokens are copied, to host slots
  taken from a stack; a victim they do not fit is recomputed instead; the
  swapped request keeps its computed length and waits at the front of the
  queue; when admitted again it gets fresh blocks (no prefix match) and its
  slots are copied back into the first of them; a slot freed by a swap-in is
  reused from the next step on (the step's copies run swap-outs first).

Emitted per step: prefill chunks (more than one new token) first, then decode
sequences (exactly one new token), each group in scheduling order.
"""
from collections import deque
from dataclasses import dataclass, field
from typing import List, Optional

import numpy as np


class OutOfBlocks(Exception):
    pass


class BlockPool:
    def __init__(self, num_blocks: int, initial_order=None):
        self.num_blocks = num_blocks
        if initial_order is None:
            self.free_list = list(range(num_blocks))
        else:
            self.free_list = [int(x) for x in initial_order]
            assert sorted(self.free_list) == list(range(num_blocks))
        self.fail_at = None      # fault injection: fail the n-th alloc call (1-based)
        self.alloc_calls = 0

    def free_count(self) -> int:
        return len(self.free_list)

    def alloc(self, n: int) -> List[int]:
        self.alloc_calls += 1
        if self.fail_at is not None and self.alloc_calls == self.fail_at:
            raise OutOfBlocks("injected")
        if n > len(self.free_list):
            raise OutOfBlocks("need %d, free %d" % (n, len(self.free_list)))
        return [self.free_list.pop() for _ in range(n)]

    def free(self, ids) -> None:
        for i in ids:
            self.free_list.append(int(i))


@dataclass
class Request:
    rid: int
    prompt_len: int
    max_tokens: int
    eos_after: int                 # output length at which the request emits EOS
    generated: int = 0
    num_computed: int = 0          # tokens whose K/V are in the cache
    blocks: List[int] = field(default_factory=list)
    tokens: Optional[list] = None  # prompt token ids (None: no prefix sharing)
    registered: int = 0            # leading prompt pages registered in the prefix cache
    reg_stopped: bool = False
    slots: List[int] = field(default_factory=list)   # host slots of its swapped-out blocks
    state: str = "waiting"         # waiting | running | finished
    arrival_step: int = 0
    finish_step: int = -1
    preemptions: int = 0

    @property
    def length(self) -> int:
        return self.prompt_len + self.generated


@dataclass
class StepMeta:
    seq_rids: np.ndarray           # int64 [S]
    q_lens: np.ndarray             # int32 [S]
    context_lens: np.ndarray       # int32 [S]
    cu_seqlens: np.ndarray         # int32 [S+1]
    block_tables: np.ndarray       # int32 [S, max_blocks], -1 padded
    slot_mapping: np.ndarray       # int64 [T]
    token_rids: np.ndarray         # int64 [T]
    token_pos: np.ndarray          # int32 [T]
    num_prefill: int
    finished_rids: np.ndarray = None   # int64: requests retired at the end of this step
    swap_out: np.ndarray = None        # int32 [n, 2]: device block -> host slot, before the kernels
    swap_in: np.ndarray = None         # int32 [n, 2]: host slot -> device block, after the swap-outs


def cdiv(a: int, b: int) -> int:
    return -(-a // b)


class Scheduler:
    def __init__(self, num_blocks: int, block_size: int = 16, max_batch: int = 256,
                 max_num_batched_tokens: int = 8192, chunk: int = 512, max_model_len: int = 8192,
                 initial_order=None, policy: str = "continuous", prefix_caching: bool = False,
                 preemption: str = "recompute", swap_blocks: int = 0):
        assert policy in ("continuous", "static")
        assert preemption in ("recompute", "swap")
        self.policy = policy
        self.preemption = preemption
        self.swap_free = list(range(swap_blocks - 1, -1, -1))   # a stack: slot 0 first
        self.swap_free_next = []
        self.swap_out_pairs, self.swap_in_pairs = [], []
        self.swapped_out_blocks = self.swapped_in_blocks = 0
        self.prefix_caching = prefix_caching
        self.cache = {}          # (block of the preceding page or -1, page tokens) -> block
        self.key_of = {}         # block -> its cache key
        self.refcount = {}       # block -> number of requests holding it
        self.prefix_hit_blocks = 0
        self.bs = block_size
        self.pool = BlockPool(num_blocks, initial_order)
        self.max_batch = max_batch
        self.budget = max_num_batched_tokens
        self.chunk = chunk
        self.max_model_len = max_model_len
        self.max_blocks = cdiv(max_model_len, block_size)
        self.waiting = deque()
        self.running: List[Request] = []
        self.finished: List[Request] = []
        self.step_no = 0
        self.n_preemptions = 0
        self.sum_running = 0

    def add(self, rid: int, prompt_len: int, max_tokens: int, eos_after: int, tokens=None) -> None:
        # A request that needs more blocks than the pool holds is accepted but
        # never admitted (it stays at the head of the queue).
        if prompt_len < 1 or prompt_len >= self.max_model_len or max_tokens < 1 or eos_after < 1:
            raise ValueError("bad request")
        if tokens is not None:
            tokens = [int(t) for t in tokens]
            assert len(tokens) == prompt_len
        self.waiting.append(Request(rid, prompt_len, max_tokens, eos_after, tokens=tokens,
                                    arrival_step=self.step_no))

    # ---- blocks with reference counts, and the prefix cache
    def _alloc(self, n: int):
        got = self._try_alloc(n)
        if got is not None:
            for b in got:
                self.refcount[b] = 1
        return got

    def _release(self, r: Request) -> None:
        for b in r.blocks:
            self.refcount[b] -= 1
            if self.refcount[b] == 0:
                del self.refcount[b]
                self.pool.free([b])
                if b in self.key_of:
                    del self.cache[self.key_of.pop(b)]
        r.blocks = []

    def _page(self, r: Request, k: int):
        return tuple(r.tokens[k * self.bs:(k + 1) * self.bs])

    def find_prefix_match(self, r: Request) -> list:
        """Blocks of the longest chain of registered pages matching r's
        prompt, covering at most prompt_len - 1 tokens."""
        if not self.prefix_caching or r.tokens is None:
            return []
        chain, parent = [], -1
        for k in range((r.prompt_len - 1) // self.bs):
            b = self.cache.get((parent, self._page(r, k)))
            if b is None:
                break
            chain.append(b)
            parent = b
        return chain

    def _register(self, r: Request) -> None:
        if not self.prefix_caching or r.tokens is None or r.reg_stopped:
            return
        full = min(r.num_computed, r.prompt_len) // self.bs
        while r.registered < full:
            k = r.registered
            parent = -1 if k == 0 else r.blocks[k - 1]
            if k > 0 and parent not in self.key_of:
                r.reg_stopped = True
                return
            key = (parent, self._page(r, k))
            if key not in self.cache:
                self.cache[key] = r.blocks[k]
                self.key_of[r.blocks[k]] = key
            elif self.cache[key] != r.blocks[k]:
                r.reg_stopped = True
                return
            r.registered += 1

    def _preempt(self, r: Request) -> None:
        keep = cdiv(r.num_computed, self.bs)        # blocks holding computed tokens
        if self.preemption == "swap" and 0 < keep <= len(self.swap_free):
            for k in range(keep):
                slot = self.swap_free.pop()
                r.slots.append(slot)
                self.swap_out_pairs.append((r.blocks[k], slot))
            self.swapped_out_blocks += keep
        else:
            r.num_computed = 0
        self._release(r)
        r.registered = 0
        r.reg_stopped = False
        r.state = "waiting"
        r.preemptions += 1
        self.running.remove(r)
        self.waiting.appendleft(r)
        self.n_preemptions += 1

    def _try_alloc(self, n: int):
        try:
            return self.pool.alloc(n)
        except OutOfBlocks:
            return None

    def step(self) -> Optional[StepMeta]:
        budget = self.budget
        self.swap_free.extend(self.swap_free_next)
        self.swap_free_next = []
        self.swap_out_pairs, self.swap_in_pairs = [], []
        scheduled = []
        # running requests first, in admission order
        i = 0
        while i < len(self.running) and budget > 0:
            r = self.running[i]
            q = min(r.length - r.num_computed, self.chunk, budget)
            need = cdiv(r.num_computed + q, self.bs) - len(r.blocks)
            got = [] if need <= 0 else self._alloc(need)
            preempted_self = False
            while got is None:
                victim = self.running[-1]
                self._preempt(victim)
                if victim is r:
                    preempted_self = True
                    break
                got = self._alloc(need)
            if preempted_self:
                continue
            r.blocks.extend(got)
            scheduled.append((r, q))
            budget -= q
            i += 1
        # admit waiting requests, first come first served.  Static batching
        # ("Continuous Batching", opening section): a new batch only when
        # nothing runs, filled to max_batch whatever the token budget; the
        # members' prefill chunks then take the budget step by step.
        static = self.policy == "static"
        may_admit = not static or not self.running
        while may_admit and self.waiting and len(self.running) < self.max_batch and (static or budget > 0):
            r = self.waiting[0]
            swapped = bool(r.slots)
            chain = [] if swapped else self.find_prefix_match(r)
            got = self._alloc(cdiv(r.length, self.bs) - len(chain))
            if got is None:
                break
            self.waiting.popleft()
            for b in chain:
                self.refcount[b] += 1
            r.blocks = chain + got
            if swapped:
                # the host slots go back into the first blocks
                self.swap_in_pairs.extend(zip(r.slots, r.blocks))
                self.swapped_in_blocks += len(r.slots)
                self.swap_free_next.extend(r.slots)
                r.slots = []
                r.registered = 0
            else:
                r.num_computed = len(chain) * self.bs
                r.registered = len(chain)
            r.reg_stopped = False
            self.prefix_hit_blocks += len(chain)
            r.state = "running"
            self.running.append(r)
            q = min(r.length - r.num_computed, self.chunk, budget)
            if q > 0:
                scheduled.append((r, q))
                budget -= q
        self.sum_running += len(self.running)
        meta = self._emit(scheduled) if scheduled else None
        # the iteration ran: advance, emit a token where the context caught up, retire
        done = []
        for r, q in scheduled:
            r.num_computed += q
            self._register(r)
            if r.num_computed == r.length:
                r.generated += 1
                if (r.generated >= r.eos_after or r.generated >= r.max_tokens
                        or r.length >= self.max_model_len):
                    self._release(r)
                    r.state = "finished"
                    r.finish_step = self.step_no
                    self.running.remove(r)
                    self.finished.append(r)
                    done.append(r.rid)
        if meta is None and (self.swap_out_pairs or self.swap_in_pairs):
            meta = self._emit([])
        if meta is not None:
            meta.finished_rids = np.array(done, dtype=np.int64)
            meta.swap_out = np.array(self.swap_out_pairs, dtype=np.int32).reshape(-1, 2)
            meta.swap_in = np.array(self.swap_in_pairs, dtype=np.int32).reshape(-1, 2)
        self.step_no += 1
        return meta

    def _emit(self, scheduled) -> StepMeta:
        order = [x for x in scheduled if x[1] > 1] + [x for x in scheduled if x[1] == 1]
        S = len(order)
        q_lens = np.array([q for _, q in order], dtype=np.int32)
        cu = np.zeros(S + 1, dtype=np.int32)
        cu[1:] = np.cumsum(q_lens)
        tables = np.full((S, self.max_blocks), -1, dtype=np.int32)
        ctx = np.zeros(S, dtype=np.int32)
        T = int(cu[-1])
        slots = np.zeros(T, dtype=np.int64)
        trid = np.zeros(T, dtype=np.int64)
        tpos = np.zeros(T, dtype=np.int32)
        for s, (r, q) in enumerate(order):
            ctx[s] = r.num_computed + q
            tables[s, : len(r.blocks)] = r.blocks
            for j in range(q):
                pos = r.num_computed + j
                t = cu[s] + j
                slots[t] = r.blocks[pos // self.bs] * self.bs + pos % self.bs
                trid[t] = r.rid
                tpos[t] = pos
        return StepMeta(seq_rids=np.array([r.rid for r, _ in order], dtype=np.int64), q_lens=q_lens,
                        context_lens=ctx, cu_seqlens=cu, block_tables=tables, slot_mapping=slots,
                        token_rids=trid, token_pos=tpos,
                        num_prefill=sum(1 for _, q in order if q > 1))

    def idle(self) -> bool:
        return not self.running and not self.waiting

    def stats(self) -> dict:
        return {
            "steps": self.step_no,
            "free_blocks": self.pool.free_count(),
            "running": len(self.running),
            "waiting": len(self.waiting),
            "finished": len(self.finished),
            "preemptions": self.n_preemptions,
            "sum_running": self.sum_running,
            "prefix_hit_blocks": self.prefix_hit_blocks,
            "cached_blocks": len(self.cache),
            "swapped_out_blocks": self.swapped_out_blocks,
            "swapped_in_blocks": self.swapped_in_blocks,
            "free_swap_slots": len(self.swap_free) + len(self.swap_free_next),
        }
