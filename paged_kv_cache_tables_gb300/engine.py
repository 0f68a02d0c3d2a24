"""A minimal engine loop over the library: the native scheduler builds each
step's metadata, one upload carries it to the device, and every layer runs
append -> prefill chunks -> decode on the paged caches.

Orchestration only: the scheduling rules live in libpkv.so's scheduler and
all arithmetic in its kernels.  Per-layer Q/K/V rows of the step's new tokens
come from a caller-supplied `fill(layer, cache_id, q, k, v, token_rids,
token_pos)` (the model would produce them; benchmarks and tests pass a
synthetic generator).

Layers share one block table per sequence ("tiny-vllm part 7" keeps one per
layer and re-uploads all of them every layer; here the step's metadata goes
up once).  `num_caches` physical K/V caches are rotated over the layers
(layer l uses cache l % num_caches) so that a many-layer trace fits in HBM;
every layer still streams its own full context.

With preemption by swap ("Continuous Batching" §5 "Preemption") each
physical K and V cache has a pinned host mirror of `swap_blocks` blocks; the
scheduler names, per step, which device blocks go out to which host slots and
which come back, and the step runs those copies (one pkv_copy_blocks launch
per cache array and direction, out before in) ahead of its layers.
"""
import ctypes
import time

import numpy as np

from . import _binding as B


class PagedEngine:
    def __init__(self, num_blocks, num_layers=32, num_caches=4, Hq=32, Hkv=8, d=128, dtype="bf16",
                 max_batch=256, max_num_batched_tokens=8192, chunk=512, max_model_len=8192, initial_order=None,
                 device="cuda", policy=B.SCHED_CONTINUOUS, prefix_caching=False, row_keys=None,
                 preemption=B.PREEMPT_RECOMPUTE, swap_blocks=0, forget_finished=True):
        import torch
        self.torch = torch
        self.L, self.R = num_layers, num_caches
        self.Hq, self.Hkv, self.d, self.bs = Hq, Hkv, d, 16
        self.NB = num_blocks
        self.tdt = torch.bfloat16 if dtype == "bf16" else torch.float16
        self.sched = B.Scheduler(num_blocks, 16, max_batch, max_num_batched_tokens, chunk, max_model_len,
                                 initial_order=initial_order, policy=policy, prefix_caching=prefix_caching,
                                 preemption=preemption, swap_blocks=swap_blocks)
        self.forget_finished = forget_finished
        # row_keys(token_rids, token_pos) -> int64 keys handed to `fill` in
        # place of the request ids (a caller whose rows depend on content)
        self.row_keys = row_keys
        self.max_blocks = self.sched.max_blocks
        self.max_T = max_num_batched_tokens
        self.max_S = max_batch
        dev = torch.device(device)
        shape = (num_blocks, Hkv, 16, d)
        self.k_cache = [torch.zeros(shape, dtype=self.tdt, device=dev) for _ in range(num_caches)]
        self.v_cache = [torch.zeros(shape, dtype=self.tdt, device=dev) for _ in range(num_caches)]
        # host mirrors of the caches for swapped-out blocks (the GPU reads and
        # writes pinned memory directly)
        self.swap_blocks = swap_blocks if preemption == B.PREEMPT_SWAP else 0
        hshape = (self.swap_blocks,) + shape[1:]
        self.k_swap = [torch.empty(hshape, dtype=self.tdt).pin_memory() for _ in range(num_caches)] \
            if self.swap_blocks else []
        self.v_swap = [torch.empty(hshape, dtype=self.tdt).pin_memory() for _ in range(num_caches)] \
            if self.swap_blocks else []
        self.swap_bytes = 0
        T, S = self.max_T, self.max_S
        self.q = torch.empty((T, Hq, d), dtype=self.tdt, device=dev)
        self.k = torch.empty((T, Hkv, d), dtype=self.tdt, device=dev)
        self.v = torch.empty((T, Hkv, d), dtype=self.tdt, device=dev)
        self.out = torch.empty((T, Hq, d), dtype=self.tdt, device=dev)
        self.work = torch.empty(max(16, B.decode_workspace_size(S, Hq, Hkv, d)), dtype=torch.uint8, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        # one pinned staging area and one device area for the step's metadata
        self.n_i64 = 3 * T                       # slot_mapping, token_rids, (spare)
        self.n_i32 = T + 2 * S + 1 + S * self.max_blocks + 4 * self.swap_blocks   # + swap pairs
        # two pinned staging areas used alternately: the host may only rewrite
        # one after the device has finished copying it (the GPU can be a step
        # behind the host)
        self.h_i64 = [torch.empty(self.n_i64, dtype=torch.int64).pin_memory() for _ in range(2)]
        self.h_i32 = [torch.empty(self.n_i32, dtype=torch.int32).pin_memory() for _ in range(2)]
        self.copied = [torch.cuda.Event() for _ in range(2)]
        self.nstep = 0
        self.d_i64 = torch.empty(self.n_i64, dtype=torch.int64, device=dev)
        self.d_i32 = torch.empty(self.n_i32, dtype=torch.int32, device=dev)
        self.stream = torch.cuda.current_stream()
        self.host_ms = 0.0      # host work per step, without waiting for the device
        self.wait_ms = 0.0      # host time spent waiting for a staging buffer
        self.upload_bytes = 0

    def add(self, rid, prompt_len, max_tokens, eos_after, tokens=None):
        self.sched.add(rid, prompt_len, max_tokens, eos_after, tokens=tokens)

    def _swap(self, o, n_out, n_in):
        """The step's block copies: device -> host slots for preempted
        sequences, then host slots -> device for re-admitted ones (a block
        swapped out may be the destination of a swap-in of the same step)."""
        L = B.lib()
        blk = self.k_cache[0][0].numel() * self.k_cache[0].element_size()
        pst, pstream = self.status.data_ptr(), self.stream.cuda_stream
        pairs_out = self.d_i32.data_ptr() + o * 4
        pairs_in = pairs_out + 2 * n_out * 4
        for dev, host in zip(self.k_cache + self.v_cache, self.k_swap + self.v_swap):
            if n_out:
                rc = L.pkv_copy_blocks(host.data_ptr(), self.swap_blocks, dev.data_ptr(), self.NB, pairs_out, n_out,
                                       blk, pst, pstream)
                if rc != B.PKV_OK:
                    raise B.PkvError("swap out", rc)
        for dev, host in zip(self.k_cache + self.v_cache, self.k_swap + self.v_swap):
            if n_in:
                rc = L.pkv_copy_blocks(dev.data_ptr(), self.NB, host.data_ptr(), self.swap_blocks, pairs_in, n_in,
                                       blk, pst, pstream)
                if rc != B.PKV_OK:
                    raise B.PkvError("swap in", rc)
        self.swap_bytes += (n_out + n_in) * blk * 2 * self.R

    def step(self, fill, on_layer_done=None, time_layers=False):
        """One engine step.  Returns None when nothing was scheduled, else a
        dict with the step's metadata (numpy) and device views.  With
        time_layers, events around each layer's attention call let the caller
        separate the attention's device time from the rows' generation."""
        torch = self.torch
        t0 = time.perf_counter()
        m = self.sched.step_raw()
        S, T, P = m.num_seqs, m.num_tokens, m.num_prefill
        n_out, n_in = m.num_swap_out, m.num_swap_in
        arr = lambda ptr, n: np.ctypeslib.as_array(ptr, shape=(n,)) if n else np.zeros(0, np.int64)
        if S == 0 and not (n_out or n_in):
            self.host_ms += (time.perf_counter() - t0) * 1e3
            return None
        MB = m.max_blocks
        # stage: i64 = [slot_mapping T][token_rids T];
        #        i32 = [token_pos T][ctx S][cu S+1][tables S*MB][swap_out 2*n_out][swap_in 2*n_in]
        buf = self.nstep & 1
        self.nstep += 1
        tw = time.perf_counter()
        self.copied[buf].synchronize()    # the device is at most one step behind
        waited = (time.perf_counter() - tw) * 1e3
        self.wait_ms += waited
        h64, h32 = self.h_i64[buf].numpy(), self.h_i32[buf].numpy()
        h64[:T] = arr(m.slot_mapping, T)
        h64[T:2 * T] = (arr(m.token_rids, T) if self.row_keys is None
                        else self.row_keys(arr(m.token_rids, T), arr(m.token_pos, T)))
        o = 0
        if S:
            h32[o:o + T] = arr(m.token_pos, T); o += T
            h32[o:o + S] = arr(m.context_lens, S); o += S
            h32[o:o + S + 1] = arr(m.cu_seqlens, S + 1); o += S + 1
            h32[o:o + S * MB] = arr(m.block_tables, S * MB); o += S * MB
        o_swap = o
        h32[o:o + 2 * n_out] = arr(m.swap_out, 2 * n_out); o += 2 * n_out
        h32[o:o + 2 * n_in] = arr(m.swap_in, 2 * n_in); o += 2 * n_in
        n32 = o
        self.d_i64[:2 * T].copy_(self.h_i64[buf][:2 * T], non_blocking=True)
        self.d_i32[:n32].copy_(self.h_i32[buf][:n32], non_blocking=True)
        self.copied[buf].record(self.stream)
        self.upload_bytes += 2 * T * 8 + n32 * 4
        ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
        ev[0].record(self.stream)
        if n_out or n_in:
            self._swap(o_swap, n_out, n_in)
        if S == 0:
            self.host_ms += (time.perf_counter() - t0) * 1e3 - waited
            return None
        slots, trids = self.d_i64[:T], self.d_i64[T:2 * T]
        o = 0
        tpos = self.d_i32[o:o + T]; o += T
        ctx = self.d_i32[o:o + S]; o += S
        cu = self.d_i32[o:o + S + 1]; o += S + 1
        tables = self.d_i32[o:o + S * MB].view(S, MB)
        cu_h = arr(m.cu_seqlens, S + 1)
        t1 = int(cu_h[P])
        max_q = int(np.diff(cu_h[:P + 1]).max()) if P else 0
        q, k, v, out = self.q[:T], self.k[:T], self.v[:T], self.out[:T]
        info = {"S": S, "T": T, "P": P, "t1": t1, "seq_rids": arr(m.seq_rids, S).copy(),
                "context_lens": arr(m.context_lens, S).copy(), "cu_seqlens": cu_h.copy(),
                "q_lens": arr(m.q_lens, S).copy(),
                "finished": arr(m.finished_rids, m.num_finished).copy() if m.num_finished else np.zeros(0, np.int64)}
        if self.forget_finished:
            # the scheduler keeps a finished request's counters until told to
            # drop them; a serving loop learns of the finish here
            for rid in info["finished"]:
                self.sched.forget(int(rid))
        # the step's device pointers are resolved once; every layer then calls
        # the C ABI directly (the same entry points the binding wraps)
        L = B.lib()
        esz = 2
        row_q = self.Hq * self.d * esz
        pq, pk, pv, pout = q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr()
        pslots, pcu, pctx, ptab = slots.data_ptr(), cu.data_ptr(), ctx.data_ptr(), tables.data_ptr()
        pst, pstream = self.status.data_ptr(), self.stream.cuda_stream
        pwork, nwork = self.work.data_ptr(), self.work.numel()
        dt = B.DTYPE_BF16 if self.tdt == torch.bfloat16 else B.DTYPE_F16
        scale = 1.0 / float(np.sqrt(self.d))
        # host copies of cu_seqlens and context lengths (the scheduler's arrays,
        # valid until its next step) let the library split the SMs
        hcu = ctypes.cast(m.cu_seqlens, ctypes.c_void_p) if P else None
        hctx = ctypes.cast(m.context_lens, ctypes.c_void_p) if P else None
        kc = [t.data_ptr() for t in self.k_cache]
        vc = [t.data_ptr() for t in self.v_cache]
        NB, Hq, Hkv, d = self.NB, self.Hq, self.Hkv, self.d
        self.host_ms += (time.perf_counter() - t0) * 1e3 - waited
        layer_events = []
        for layer in range(self.L):
            cid = layer % self.R
            fill(layer, cid, q, k, v, trids, tpos)
            if time_layers:
                layer_events.append((torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)))
                layer_events[-1][0].record(self.stream)
            # the layer's append and attention in one call: prefill chunks
            # (their rows appended by slot) beside the decodes on split SMs,
            # each decode's row appended inside the decode kernel
            rc = L.pkv_paged_mixed_append_attention(pout, pq, pk, pv, pslots, pcu, P, t1, max_q, S - P, kc[cid],
                                                    vc[cid], ptab, MB, pctx, NB, Hq, Hkv, d, 16, scale, dt, dt, pwork,
                                                    nwork, hcu, hctx, 0, pst, pstream)
            if rc != B.PKV_OK:
                raise B.PkvError("engine step, layer %d" % layer, rc)
            if time_layers:
                layer_events[-1][1].record(self.stream)
            if on_layer_done is not None:
                on_layer_done(layer, info, out)
        ev[1].record(self.stream)
        info["events"] = ev
        info["layer_events"] = layer_events
        return info


def run_trace(engine, arrival, prompt, eos, max_tokens, fill, sample_every=0, pick=None, max_steps=1000000,
              tokens=None, time_layers_every=0):
    """Drive `engine` through a request trace: request i is added at engine
    step arrival[i]; steps run until every request has finished.  On every
    `sample_every`-th engine step, pick(info) names (output row, rid,
    position) samples whose layer-0 outputs are copied back for checking.
    Every `time_layers_every`-th step also times its attention calls alone
    (events around each; they break the overlap of a layer's launches with
    the row generation before them, so only a sample of steps is timed).
    Returns per-step records, finish steps, timings and the sampled rows."""
    torch = engine.torch
    n = len(arrival)
    order = np.argsort(arrival, kind="stable")
    nxt = 0
    finish_step = {}
    steps = []
    samples = []
    state = {"sample": False}

    def on_layer(layer, info, out):
        if layer == 0 and state["sample"]:
            rows = pick(info)
            if rows:
                idx = torch.tensor([r[0] for r in rows], device=out.device)
                samples.append((rows, out.index_select(0, idx).float().to("cpu")))

    first_token = {}
    t_wall = time.perf_counter()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    ev0.record(engine.stream)
    for step in range(max_steps):
        while nxt < n and arrival[order[nxt]] <= step:
            i = int(order[nxt])
            engine.add(i, int(prompt[i]), int(max_tokens), int(eos[i]), tokens=None if tokens is None else tokens[i])
            nxt += 1
        state["sample"] = bool(sample_every) and pick is not None and len(steps) % sample_every == 0
        timed = bool(time_layers_every) and len(steps) % time_layers_every == 0
        info = engine.step(fill, on_layer_done=on_layer, time_layers=timed)
        if info is not None:
            for rid in info["finished"]:
                finish_step[int(rid)] = step
            # a request emits its first token after the step in which its
            # context first covers the whole prompt
            for rid, c in zip(info["seq_rids"], info["context_lens"]):
                rid = int(rid)
                if rid not in first_token and c >= prompt[rid]:
                    first_token[rid] = step
            steps.append({"step": step, "S": info["S"], "T": info["T"], "P": info["P"],
                          "context_lens": info["context_lens"], "q_lens": info["q_lens"], "events": info["events"],
                          "layer_events": info["layer_events"]})
        if nxt >= n and len(finish_step) == n:
            break
    ev1.record(engine.stream)
    torch.cuda.synchronize()
    for s in steps:   # device time of each step's layer launches (and of their attention calls alone)
        e = s.pop("events")
        s["device_ms"] = e[0].elapsed_time(e[1])
        le = s.pop("layer_events")
        if le:
            s["attention_ms"] = sum(a.elapsed_time(b) for a, b in le)
    return {"steps": steps, "finish_step": finish_step, "first_token_step": first_token, "wall_s": time.perf_counter() - t_wall,
            "stream_ms": ev0.elapsed_time(ev1), "samples": samples}
