"""Benchmark: one engine step of paged decode attention on the Llama-3-8B-shaped
workload (256 sequences, 32 query / 8 KV heads, head_dim 128, 16-token blocks,
lognormal contexts with median 1024 clipped to 32..8192, bf16, 64k-block pool).

A step = append of the 256 new tokens' K/V, then paged decode attention over
every sequence's whole context, in one call: a small kernel that zeroes the
call's control region of the workspace, then the split-KV decode kernel with
the append fused in (the same step as separate append and decode calls is
timed beside it).
Prints ONE JSON line (rank 0).  `--impl reference` times the FP64 CPU oracle
on a bounded sample of the same workload instead.

Metric: algorithmic bytes of the step / step time, where the bytes are every
attended token's K and V once per KV head, Q in, O out, the block-table
entries in use, the context lengths, plus the append's reads and writes.
"""
import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged decode-attention KV GB/s (% of ~8 TB/s HBM) and attended tokens/s"
WORKLOAD = "llama8b-decode"


def decode_bytes(ctx, Hq, Hkv, d, esize=2, bs=16):
    ctx = np.asarray(ctx, np.int64)
    S = ctx.shape[0]
    kv = int(ctx.sum()) * 2 * Hkv * d * esize
    return kv + S * Hq * d * esize * 2 + int(((ctx + bs - 1) // bs).sum()) * 4 + 4 * S


# DRAM traffic of one full-size decode launch (the default 256-sequence step,
# append fused): dram__bytes_read.sum + dram__bytes_write.sum from one ncu
# capture of that launch, valid for the decode source with this SHA-1 and
# reported as null once it changes (or for another workload).
DECODE_TRAFFIC_BYTES = 1454636544 + 4925696
DECODE_TRAFFIC_SHA1 = "9d5df3620f33531e1f5fc04ecfd5f2408b0c6255"


# launches per decode call: the control-region clear and the decode kernel
LAUNCHES_PER_DECODE_CALL = 2


def clear_bytes(S, Hkv):
    """Bytes a decode call zeroes before its kernel: control words (256),
    per-range counter words (8 B) and list heads (4 B), each array 256-B
    aligned."""
    a = lambda x: (x + 255) // 256 * 256
    return 256 + a(8 * S * Hkv) + a(4 * S * Hkv)


def decode_traffic(default_workload):
    import hashlib
    src = os.path.join(os.path.dirname(os.path.abspath(__file__)), "paged_kv_cache_tables_gb300", "csrc", "decode.cu")
    with open(src, "rb") as f:
        if hashlib.sha1(f.read()).hexdigest() != DECODE_TRAFFIC_SHA1:
            return None
    return DECODE_TRAFFIC_BYTES if default_workload else None


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            pk = json.load(f)
        return float(pk["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def load_tensor_peak():
    """bf16 dense peak for a kernel timed inside a long step (sustained)."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            pk = json.load(f)
        return float(pk["bf16_tflops_sustained"]), "measured (sustained)"
    except Exception:
        return 1700.0, "fallback (sustained)"


def prefill_flops(ctx, q_lens, Hq, d):
    """Algorithmic FLOPs of causal chunked prefill: query i of a chunk of q_len
    attends prior + i + 1 keys; QK^T and PV each take 2*d FLOPs per (query
    head, key)."""
    total = 0
    for c, q in zip(ctx, q_lens):
        q = int(q)
        prior = int(c) - q
        keys = q * prior + q * (q + 1) // 2
        total += 4 * Hq * d * keys
    return total


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""
    Q = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.Q,
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            # the timed region starts once nvidia-smi is up and sampling (its
            # start-up on a fresh machine can take seconds)
            t_end = time.time() + 15.0
            while not self.lines and time.time() < t_end and self.proc.poll() is None:
                time.sleep(0.05)
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 6:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[2:6]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_setup(args):
    import torch
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, ws):
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def to_dev_bits(a, dtype):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16))
    return t.view(torch.bfloat16 if dtype == "bf16" else torch.float16).cuda()


def oracle_sample_size(st, budget_s):
    """Number k of leading sequences whose oracle decode takes about budget_s
    on this host (calibrated on the first sequence)."""
    import oracle
    t0 = time.perf_counter()
    oracle.decode(st.q[:1], st.k_cache, st.v_cache, st.block_tables[:1], st.context_lens[:1], st.dtype)
    per_tok = (time.perf_counter() - t0) / max(1, int(st.context_lens[0]))
    k, acc = 0, 0.0
    while k < st.S and acc + per_tok * int(st.context_lens[k]) <= budget_s:
        acc += per_tok * int(st.context_lens[k])
        k += 1
    return max(k, 1)


def cpu_oracle_run(st, k, min_seconds=0.0):
    """Time the oracle (as it stands: one thread, FP64) on the first k
    sequences, repeated until at least min_seconds of work have been timed."""
    import oracle
    cl = st.context_lens[:k]
    reps, dt = 0, 0.0
    while reps == 0 or dt < min_seconds:
        t0 = time.perf_counter()
        oracle.decode(st.q[:k], st.k_cache, st.v_cache, st.block_tables[:k], cl, st.dtype)
        dt += time.perf_counter() - t0
        reps += 1
    nbytes = decode_bytes(cl, st.Hq, st.Hkv, st.d) * reps
    return {"value": nbytes / dt / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": "first %d of %d sequences of the step (%d attended tokens), decode only, %d pass%s, %.2f s"
                      % (k, st.S, int(cl.sum()), reps, "" if reps == 1 else "es", dt),
            "seconds": dt / reps}


def _oracle_worker(args):
    """One worker of the all-cores CPU baseline: the oracle, as it stands, on
    a slice of the step's sequences, reading the caches from shared memory."""
    from multiprocessing import shared_memory
    import oracle
    names, shapes, dtype, lo, hi, passes = args
    shms = [shared_memory.SharedMemory(name=n) for n in names]
    try:
        arrs = [np.ndarray(sh, dtype=dt, buffer=m.buf) for m, (sh, dt) in zip(shms, shapes)]
        q, kc, vc, bt, cl = arrs
        t0 = time.perf_counter()
        for _ in range(passes):
            oracle.decode(q[lo:hi], kc, vc, bt[lo:hi], cl[lo:hi], dtype)
        return time.perf_counter() - t0
    finally:
        del arrs
        for m in shms:
            m.close()


class OraclePool:
    """The oracle on every host core: the step's sequences split into slices
    of about equal attended tokens, one spawned process per slice (spawned,
    not forked: the parent may hold a CUDA context), the caches in shared
    memory rather than copied.  run(passes) times `passes` decodes of the
    whole step, as wall time until the slowest slice is done."""

    def __init__(self, st):
        import multiprocessing as mp
        from multiprocessing import shared_memory
        self.st = st
        cores = len(os.sched_getaffinity(0))
        arrays = [st.q, st.k_cache, st.v_cache, st.block_tables, st.context_lens]
        # shared memory lives in /dev/shm; writing past a small tmpfs there
        # would kill the process (SIGBUS), so check its room first
        need = sum(a.nbytes for a in arrays)
        vfs = os.statvfs("/dev/shm")
        if vfs.f_bavail * vfs.f_frsize < need * 1.25:
            raise RuntimeError("/dev/shm has %.1f GB free, %.1f GB needed" % (vfs.f_bavail * vfs.f_frsize / 1e9,
                                                                              need * 1.25 / 1e9))
        self.shms, names, shapes = [], [], []
        try:
            for a in arrays:
                m = shared_memory.SharedMemory(create=True, size=max(1, a.nbytes))
                self.shms.append(m)
                np.ndarray(a.shape, dtype=a.dtype, buffer=m.buf)[...] = a
                names.append(m.name)
                shapes.append((a.shape, a.dtype.str))
            cum = np.concatenate([[0], np.cumsum(st.context_lens.astype(np.int64))])
            cuts = [int(np.searchsorted(cum, cum[-1] * k / cores)) for k in range(cores + 1)]
            cuts[0], cuts[-1] = 0, st.S
            self.slices = [(names, shapes, st.dtype, cuts[k], cuts[k + 1]) for k in range(cores)
                           if cuts[k + 1] > cuts[k]]
            self.pool = mp.get_context("spawn").Pool(len(self.slices))
        except Exception:
            self.close()
            raise
        self.cores = len(self.slices)

    def run(self, passes):
        t0 = time.perf_counter()
        times = self.pool.map(_oracle_worker, [sl + (passes,) for sl in self.slices])
        return time.perf_counter() - t0, max(times)

    def close(self):
        if getattr(self, "pool", None) is not None:
            self.pool.close()
            self.pool.join()
            self.pool = None
        for m in self.shms:
            m.close()
            m.unlink()
        self.shms = []


def cpu_oracle_all_cores(st, budget_s, one_pass_s):
    """cpu_baseline on every host core: OraclePool, the whole step repeated to
    fill about budget_s."""
    op = OraclePool(st)
    try:
        op.run(1)   # process start and first touch of the shared caches
        passes = max(1, int(budget_s / max(one_pass_s / op.cores, 1e-3)))
        wall, slowest = op.run(passes)
    finally:
        op.close()
    nbytes = decode_bytes(st.context_lens, st.Hq, st.Hkv, st.d) * passes
    return {"value": nbytes / wall / 1e9, "unit": "GB/s", "cores": op.cores, "kind": "oracle",
            "sample": "the whole decode step, %d pass%s, split over %d spawned processes (%.2f s wall, slowest "
                      "slice %.2f s)" % (passes, "" if passes == 1 else "es", op.cores, wall, slowest)}


def step_config(st, ws):
    """The `config` of the decode-step line (both arms)."""
    dbytes = decode_bytes(st.context_lens, st.Hq, st.Hkv, st.d)
    return {"workload": WORKLOAD, "seqs_per_gpu": st.S, "q_heads": st.Hq, "kv_heads": st.Hkv, "head_dim": st.d,
            "block_size": st.bs, "pool_blocks": st.NB, "mean_context": round(float(st.context_lens.mean()), 1),
            "step": "kv_append(256 tokens) + paged_decode_attention, fused in one launch "
                    "(pkv_paged_decode_append_attention)",
            "l2": "inputs larger than L2 (%.2f GB of KV per step vs 129 MB L2), no flush" % (dbytes / 1e9),
            "parallelism": "dp%d" % ws}


def run_reference(args):
    ws, rank, _ = dist_setup(args)
    if rank != 0:
        return
    from synth import make_step
    st = make_step("llama8b")
    # each step: one decode of the whole step by the oracle on every host
    # core (a few tenths of a second on a 16-core host); one core if the
    # host cannot start the worker processes
    try:
        op = OraclePool(st)
    except Exception as e:
        op, why = None, "%s: %s" % (type(e).__name__, e)
    vals = []
    try:
        for i in range(args.warmup + args.steps):
            if op is not None:
                wall, _ = op.run(1)
            else:
                wall = cpu_oracle_run(st, st.S)["seconds"]
            if i >= args.warmup:
                vals.append(wall)
    finally:
        if op is not None:
            op.close()
    sec = statistics.median(vals)
    v = decode_bytes(st.context_lens, st.Hq, st.Hkv, st.d) / sec / 1e9
    cores = op.cores if op is not None else 1
    sample = ("the whole decode step (%d sequences, %d attended tokens) per step, split over %d spawned processes"
              % (st.S, int(st.context_lens.sum()), cores) if op is not None else
              "the whole decode step per step on one core (%s)" % why)
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": step_config(st, args.gpus),
            "cpu_baseline": {"value": v, "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def run_e2e(args, ws, st, q, kn, vn, bt, cl, out, kc, vc, work, status, stream, scale, step_bytes, K):
    """Same step through the public API with inputs in pinned host memory:
    every step copies its inputs host->device and its output device->host.
    As a serving engine would, the transfers run on a copy stream and overlap
    the neighbouring steps' kernels: each step's inputs (one packed pinned
    buffer, one copy, on an input-copy stream) go into one of two device input
    sets, its kernels wait for them, and its output (one of two) is read back
    on an output-copy stream once they are done."""
    import torch
    import paged_kv_cache_tables_gb300 as pkv
    parts = [q, kn, vn, bt, cl]
    nbytes = [t.numel() * t.element_size() for t in parts]
    offs = [0]
    for n in nbytes:
        offs.append((offs[-1] + n + 255) // 256 * 256)
    total = offs[-1]
    h_in = torch.empty(total, dtype=torch.uint8).pin_memory()
    for t, o, n in zip(parts, offs, nbytes):
        h_in[o:o + n].copy_(t.contiguous().view(-1).view(torch.uint8).cpu())
    h2d = sum(nbytes)
    d2h = out.numel() * out.element_size()

    def views(buf):
        return [buf[o:o + n].view(t.dtype).view(t.shape) for t, o, n in zip(parts, offs, nbytes)]
    d_in = [torch.empty(total, dtype=torch.uint8, device="cuda") for _ in range(2)]
    d_views = [views(b) for b in d_in]
    d_out = [torch.empty_like(out) for _ in range(2)]
    h_out = [torch.empty_like(out, device="cpu").pin_memory() for _ in range(2)]
    copy_in, copy_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]     # inputs of the set are on the device
    ev_done = [torch.cuda.Event() for _ in range(2)]   # kernels of the set have finished
    ev_back = [torch.cuda.Event() for _ in range(2)]   # output of the set is back on the host
    for e in ev_done + ev_back:
        e.record(stream)

    def e2e_step(k):
        i = k & 1
        # inputs: the set's previous kernels must be done with it
        copy_in.wait_event(ev_done[i])
        with torch.cuda.stream(copy_in):
            d_in[i].copy_(h_in, non_blocking=True)
        ev_in[i].record(copy_in)
        # kernels: after their inputs, and after the previous read-back of this output
        stream.wait_event(ev_in[i])
        stream.wait_event(ev_back[i])
        d_q, d_kn, d_vn, d_bt, d_cl = d_views[i]
        pkv.paged_decode_append_attention(d_out[i], d_q, d_kn, d_vn, kc, vc, d_bt, d_cl, scale=scale,
                                          workspace=work, dev_status=status, stream=stream)
        ev_done[i].record(stream)
        # result back to the host (a stream of its own, so that the next
        # step's input copy does not queue behind it)
        copy_out.wait_event(ev_done[i])
        with torch.cuda.stream(copy_out):
            h_out[i].copy_(d_out[i], non_blocking=True)
        ev_back[i].record(copy_out)

    for k in range(args.warmup):
        e2e_step(k)
    torch.cuda.synchronize()
    barrier(ws)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for k in range(K):
        e2e_step(k)
    # the timed region ends when the last result is on the host
    stream.wait_event(ev_back[(K - 1) & 1])
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), ws) / K
    e2e_value = step_bytes * ws / (e2e_ms * 1e-3) / 1e9
    # the read-back is the step's real output
    if not torch.equal(h_out[(K - 1) & 1], d_out[(K - 1) & 1].cpu()):
        raise RuntimeError("e2e: output read back differs from the device copy")
    return e2e_value, e2e_ms, h2d, d2h


def run_mixed(args):
    """The mixed step: append 4344 tokens, prefill 8 chunks of 512 (prior
    context U{0..4096}), decode 248 sequences, on one stream."""
    import torch
    import paged_kv_cache_tables_gb300 as pkv
    from synth import make_step
    over = {"n_chunks": args.mixed_chunks} if args.mixed_chunks else {}
    if args.mixed_prior >= 0:
        over["prior_fixed"] = args.mixed_prior
    if args.pool:
        over["NB"] = args.pool
    st = make_step("mixed", **over)
    p = st.n_prefill
    t1 = int(st.cu_seqlens[p])
    q = to_dev_bits(st.q, st.dtype)
    kn, vn = to_dev_bits(st.k_new, st.dtype), to_dev_bits(st.v_new, st.dtype)
    kc, vc = to_dev_bits(st.k_cache, st.dtype), to_dev_bits(st.v_cache, st.dtype)
    slots = torch.from_numpy(st.slot_mapping).cuda()
    bt = torch.from_numpy(st.block_tables).cuda()
    cl = torch.from_numpy(st.context_lens).cuda()
    cu = torch.from_numpy(st.cu_seqlens).cuda()
    out = torch.empty((st.T, st.Hq, st.d), dtype=torch.bfloat16, device="cuda")
    work = torch.empty(pkv.decode_workspace_size(st.S - p, st.Hq, st.Hkv, st.d), dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()
    q_p, q_d, o_p, o_d = q[:t1], q[t1:], out[:t1], out[t1:]
    bt_p, bt_d, cl_p, cl_d, cu_p = bt[:p], bt[p:], cl[:p], cl[p:], cu[:p + 1]
    max_q = int(st.q_lens[:p].max())

    def step(ev=None):
        if ev:
            ev[0].record(stream)
        pkv.kv_append(kn, vn, slots, kc, vc, dev_status=status, stream=stream)
        if ev:
            ev[1].record(stream)
        pkv.paged_prefill_attention(o_p, q_p, cu_p, max_q, kc, vc, bt_p, cl_p, dev_status=status, stream=stream)
        if ev:
            ev[2].record(stream)
        pkv.paged_decode_attention(o_d, q_d, kc, vc, bt_d, cl_d, workspace=work, dev_status=status, stream=stream)
        if ev:
            ev[3].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    K = args.mixed_steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    for k in range(K):
        step(evs[k])
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError("device status %d in the mixed step" % int(status.item()))
    ms = lambda a, b: statistics.mean(evs[k][a].elapsed_time(evs[k][b]) for k in range(K))
    step_ms, app_ms, pre_ms, dec_ms = ms(0, 3), ms(0, 1), ms(1, 2), ms(2, 3)

    # the same step through the mixed entry point: prefill and decode side by
    # side on split SMs (the split picked from the host copies of the metadata)
    out2 = torch.empty_like(out)
    cu_h, cl_h = st.cu_seqlens[:p + 1].astype(np.int32), st.context_lens.astype(np.int32)
    d_sms = pkv.mixed_split(torch.cuda.get_device_properties(0).multi_processor_count, cu_h, p, cl_h, st.Hq,
                            st.Hkv, st.d)

    def fused():
        pkv.kv_append(kn, vn, slots, kc, vc, dev_status=status, stream=stream)
        pkv.paged_mixed_attention(out2, q, cu_p, p, max_q, kc, vc, bt, cl, workspace=work, cu_seqlens_host=cu_h,
                                  context_lens_host=cl_h, dev_status=status, stream=stream)
    for _ in range(args.warmup):
        fused()
    torch.cuda.synchronize()
    fe = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    for a, b in fe:
        a.record(stream)
        fused()
        b.record(stream)
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError("device status %d in the side-by-side mixed step" % int(status.item()))
    fused_ms = statistics.mean(a.elapsed_time(b) for a, b in fe)

    # the whole step in one call: the prefill rows appended on the side stream
    # ahead of the prefill kernel, each decode row inside the decode kernel
    def one_call():
        pkv.paged_mixed_append_attention(out2, q, kn, vn, slots[:t1], cu_p, p, max_q, kc, vc, bt, cl, workspace=work,
                                         cu_seqlens_host=cu_h, context_lens_host=cl_h, dev_status=status,
                                         stream=stream)
    for _ in range(args.warmup):
        one_call()
    torch.cuda.synchronize()
    for a, b in fe:
        a.record(stream)
        one_call()
        b.record(stream)
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError("device status %d in the one-call mixed step" % int(status.item()))
    one_ms = statistics.mean(a.elapsed_time(b) for a, b in fe)
    sweep = {}
    for dn in [int(x) for x in args.mixed_decode_sms.split(",") if x]:
        def forced(dn=dn):
            pkv.kv_append(kn, vn, slots, kc, vc, dev_status=status, stream=stream)
            pkv.paged_mixed_attention(out2, q, cu_p, p, max_q, kc, vc, bt, cl, workspace=work, decode_sms=dn,
                                      dev_status=status, stream=stream)
        for _ in range(args.warmup):
            forced()
        for a, b in fe:
            a.record(stream)
            forced()
            b.record(stream)
        torch.cuda.synchronize()
        sweep[dn] = round(statistics.mean(a.elapsed_time(b) for a, b in fe), 4)
    flops = prefill_flops(st.context_lens[:p], st.q_lens[:p], st.Hq, st.d)
    dbytes = decode_bytes(st.context_lens[p:], st.Hq, st.Hkv, st.d)
    tpeak, tkind = load_tensor_peak()
    hpeak, hkind = load_peaks()
    tfl = flops / (pre_ms * 1e-3) / 1e12
    return {
        "workload": "mixed: %d prefill chunks x 512 (prior %s) + 248 decodes (ctx U{256..4096}), 32/8 heads, "
                    "d 128, bf16; append of %d tokens first"
                    % (p, "U{0..4096}" if args.mixed_prior < 0 else args.mixed_prior, st.T),
        "steps": K, "ms_per_step": round(one_ms, 4),
        "one_call": {"ms_per_step": round(one_ms, 4),
                     "note": "pkv_paged_mixed_append_attention: the append of the prefill rows on the side stream "
                             "before the prefill kernel, the decode rows inside the decode kernel"},
        "sequential_ms_per_step": round(step_ms, 4),
        "side_by_side": {"ms_per_step": round(fused_ms, 4), "decode_sms": d_sms,
                         "note": "append, then pkv_paged_mixed_attention: decode on decode_sms SMs, prefill on the "
                                 "rest, concurrently; the kernel timings below are the sequential run"},
        **({"decode_sms_sweep_ms": sweep} if sweep else {}),
        "kv_append_ms": round(app_ms, 4),
        "prefill": {"ms": round(pre_ms, 4), "gflop": round(flops / 1e9, 2), "tflops": round(tfl, 1),
                    "executed_tflops": round(tfl * 1.5, 1),
                    "executed_note": "tensor-core work actually issued: Q.K^T once and P.V twice (the rounded "
                                     "16-bit P and its rounding residual), 1.5 x the algorithmic FLOPs",
                    "roofline": {"bound": "tensor", "achieved": round(tfl, 1), "peak": tpeak, "unit": "TFLOP/s",
                                 "frac": round(tfl / tpeak, 4), "traffic": None, "peak_source": tkind}},
        "decode": {"ms": round(dec_ms, 4), "bytes": dbytes,
                   "roofline": {"bound": "hbm", "achieved": round(dbytes / (dec_ms * 1e-3) / 1e9, 1), "peak": hpeak,
                                "unit": "GB/s", "frac": round(dbytes / (dec_ms * 1e-3) / 1e9 / hpeak, 4),
                                "traffic": None, "peak_source": hkind}},
    }


def warm_up_kernels():
    """One small call of every entry point the engine uses (module loading,
    kernel attributes, the side stream, the tensor-map encoder) and of the
    torch ops of the row sampling, so that a trace's first step is not
    charged for them."""
    import torch
    import paged_kv_cache_tables_gb300 as pkv
    from synth.trace import fill_qkv_gpu
    NB, Hq, Hkv, d = 64, 32, 8, 128
    kc = torch.zeros((NB, Hkv, 16, d), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    cl = torch.tensor([200, 17, 40], dtype=torch.int32, device="cuda")
    bt = torch.arange(3 * 16, dtype=torch.int32, device="cuda").view(3, 16)
    cu = torch.tensor([0, 128], dtype=torch.int32, device="cuda")
    q = torch.zeros((130, Hq, d), dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(q)
    new = torch.zeros((130, Hkv, d), dtype=torch.bfloat16, device="cuda")
    rid = torch.zeros(130, dtype=torch.int64, device="cuda")
    pos = torch.arange(130, dtype=torch.int32, device="cuda")
    fill_qkv_gpu(q, new, new.clone(), rid, pos, 2, 0, 1)
    pkv.kv_append(new, new, torch.arange(130, dtype=torch.int64, device="cuda"), kc, vc)
    pkv.paged_prefill_attention(out[:128], q[:128], cu, 128, kc, vc, bt[:1], cl[:1])
    pkv.paged_decode_append_attention(out[128:], q[128:], new[128:], new[128:], kc, vc, bt[1:], cl[1:])
    pkv.paged_mixed_attention(out, q, cu, 1, 128, kc, vc, bt, cl, cu_seqlens_host=np.array([0, 128], np.int32),
                              context_lens_host=np.array([200, 17, 40], np.int32))
    # and the torch ops that copy sampled rows back (their kernels load lazily:
    # seconds on a machine whose first process this is)
    out.index_select(0, torch.tensor([0, 129], device="cuda")).float().to("cpu")
    torch.cuda.synchronize()


def trace_line(args, n, NB, policy="continuous", outputs="geometric", shared=False, caching=False, swap_blocks=0):
    """The continuous-batching trace: n requests, Poisson(20) arrivals per
    step, prompts lognormal (mean 512, sigma 1, clipped 8..4096), outputs
    geometric (or lognormal) with mean 256, max batch 256, 8192-token budget,
    512-token prefill chunks, a pool of NB 16-token blocks, preemption by
    recompute; every step runs append + prefill chunks + decode for 32 layers
    of the 8B shape.  The 32 layers rotate over 4 physical caches so the trace
    fits in HBM; every layer still streams its full context."""
    import torch
    from paged_kv_cache_tables_gb300 import _binding
    from paged_kv_cache_tables_gb300.engine import PagedEngine, run_trace
    from synth import SEEDS
    from synth.trace import content_keys, make_fill, make_requests, make_shared_requests, pick_rows
    torch.cuda.set_device(0)
    seed = SEEDS["trace"]
    L, R = args.trace_layers, args.trace_caches
    tokens, row_keys = None, None
    if shared:
        arrival, prompt, eos, tokens, head_len, group = make_shared_requests(seed, n=n)
        row_keys = lambda r, p: content_keys(r, p, head_len, group)
    else:
        arrival, prompt, eos = make_requests(seed, n=n, outputs=outputs)
    pol = {"continuous": _binding.SCHED_CONTINUOUS, "static": _binding.SCHED_STATIC}[policy]
    eng = PagedEngine(NB, num_layers=L, num_caches=R, initial_order=np.random.default_rng(seed).permutation(NB),
                      policy=pol, prefix_caching=caching, row_keys=row_keys,
                      preemption=_binding.PREEMPT_SWAP if swap_blocks else _binding.PREEMPT_RECOMPUTE,
                      swap_blocks=swap_blocks)
    rng = np.random.default_rng(seed + 1)
    warm_up_kernels()
    torch.cuda.synchronize()
    clk = ClockSampler(0)
    with clk:
        res = run_trace(eng, arrival, prompt, eos, max_tokens=4096, fill=make_fill(), sample_every=50,
                        pick=lambda info: pick_rows(info, rng, n_decode=1, n_prefill=1), tokens=tokens,
                        time_layers_every=8)
    if int(eng.status.item()) != 0:
        raise RuntimeError("device status %d in the trace" % int(eng.status.item()))
    st = eng.sched.stats()
    steps = res["steps"]
    if args.steps_jsonl:
        # one record per engine step: batch shape, KV bytes per layer, device time
        with open(args.steps_jsonl, "a") as f:
            for s_ in steps:
                ctx_ = s_["context_lens"]
                f.write(json.dumps({"policy": policy, "caching": caching, "swap_blocks": swap_blocks,
                                    "step": s_["step"], "seqs": int(s_["S"]), "tokens": int(s_["T"]),
                                    "prefill_chunks": int(s_["P"]), "context_tokens": int(ctx_.sum()),
                                    "kv_bytes_per_layer": int(ctx_.sum()) * 2 * 8 * 128 * 2,
                                    "device_ms": round(s_["device_ms"], 4)}) + "\n")
    Hq, Hkv, d = 32, 8, 128
    dec_tokens = pre_keys = kv_bytes = 0
    big_bytes, big_ms, big_steps, dev_ms = 0, 0.0, 0, 0.0
    # the steps whose attention calls were timed alone: their KV bytes and times
    t_bytes, t_attn_ms, t_dev_ms, tb_bytes, tb_attn_ms = 0, 0.0, 0.0, 0, 0.0
    l2_bytes = 129e6
    for s in steps:
        ctx, ql = s["context_lens"], s["q_lens"]
        dmask = ql == 1
        dec_tokens += int(ctx[dmask].sum())
        for c, q in zip(ctx[~dmask], ql[~dmask]):
            c, q = int(c), int(q)
            pre_keys += q * (c - q) + q * (q + 1) // 2
        layer_bytes = int(ctx.sum()) * 2 * Hkv * d * 2
        kv_bytes += layer_bytes
        dev_ms += s["device_ms"]
        if "attention_ms" in s:
            t_bytes += layer_bytes * L
            t_attn_ms += s["attention_ms"]
            t_dev_ms += s["device_ms"]
        # steps whose per-layer working set is more than 4x L2: no layer can
        # be served from the previous layer's cached pages
        if layer_bytes > 4 * l2_bytes:
            big_bytes += layer_bytes * L
            big_ms += s["device_ms"]
            big_steps += 1
            if "attention_ms" in s:
                tb_bytes += layer_bytes * L
                tb_attn_ms += s["attention_ms"]
    gen = sum(min(int(eos[i]), 4096, 8192 - int(prompt[i])) for i in range(n))
    lat = np.array([res["finish_step"][i] - int(arrival[i]) for i in range(n)])
    # time to first token: in engine steps, and in device time from the start
    # of the arrival step to the end of the first token's step
    step_ms = np.zeros(max(s["step"] for s in steps) + 1)
    for s_ in steps:
        step_ms[s_["step"]] = s_["device_ms"]
    cum = np.concatenate([[0.0], np.cumsum(step_ms)])
    ft = res["first_token_step"]
    ttft_steps = np.array([ft[i] - int(arrival[i]) for i in range(n)], dtype=np.float64)
    ttft_ms = np.array([cum[ft[i] + 1] - cum[int(arrival[i])] for i in range(n)])
    dev_s = res["stream_ms"] / 1e3
    # oracle check of the sampled layer-0 rows, and the oracle's own time on them
    import oracle
    from oracle.trace_check import layer0_inputs
    worst, checked, t_or, keys = 0.0, 0, 0.0, 0
    for rows, vals in res["samples"]:
        for (row, rid, pos), got in zip(rows, vals.numpy()):
            inputs = layer0_inputs(rid, pos, Hq, Hkv, d, keys=None if row_keys is None else
                                   (lambda ps, r=rid: row_keys(np.full(len(ps), r), ps)))
            # the oracle's attention alone is timed (not the regeneration of its inputs)
            t0 = time.perf_counter()
            ref = oracle.decode(*inputs, "bf16")[0]
            t_or += time.perf_counter() - t0
            keys += pos + 1
            err = np.abs(got.astype(np.float64) - ref)
            bound = np.maximum(2e-3, np.exp2(np.floor(np.log2(np.maximum(np.abs(ref), 1e-30))) - 8) + 1e-4)
            if np.any(err > bound):
                raise RuntimeError("trace sample rid %d pos %d off by %g" % (rid, pos, float(err.max())))
            worst = max(worst, float(err.max()))
            checked += 1
    line = {
        "metric": "continuous-batching trace: output tokens/s and aggregate paged-attention KV GB/s",
        "workload": "trace: %d requests, Poisson(20)/step, prompt lognormal mean 512 clip 8-4096, output %s "
                    "mean 256, max batch 256, budget 8192, chunk 512, pool %d blocks, %d layers (8B shape) over %d "
                    "physical caches, %s batching" % (n, outputs, NB, L, R, policy),
        "engine_steps": len(steps), "wall_s": round(res["wall_s"], 3), "stream_s": round(dev_s, 3),
        "host_sched_ms_per_step": round(st["host_ms"] / max(1, st["steps"]), 4),
        "host_ms_per_step": round(eng.host_ms / max(1, len(steps)), 4),
        "host_wait_ms_per_step": round(eng.wait_ms / max(1, len(steps)), 4),
        "output_tokens": gen, "output_tokens_per_s": round(gen / res["wall_s"], 1),
        "attended_tokens_per_s": round((dec_tokens + pre_keys) * L / res["wall_s"], 1),
        "kv_gbs": round(kv_bytes * L / res["wall_s"] / 1e9, 1),
        "device_s": round(dev_ms / 1e3, 3),
        "kv_gbs_device": round(kv_bytes * L / (dev_ms * 1e-3) / 1e9, 1),
        "kv_gbs_steps_over_4x_l2": {"steps": big_steps, "gbs": round(big_bytes / max(big_ms * 1e-3, 1e-12) / 1e9, 1),
                                    "attention_gbs": round(tb_bytes / max(tb_attn_ms * 1e-3, 1e-12) / 1e9, 1),
                                    "note": "KV bytes / device time of the steps whose per-layer working set "
                                            "exceeds 4 x 129 MB (append, prefill and decode of all layers); "
                                            "attention_gbs: the same over the library calls' own time on the "
                                            "sampled steps (every 8th) timed layer by layer, without the "
                                            "generation of the layers' synthetic Q/K/V rows"},
        "attention_share_of_device_time": round(t_attn_ms / max(t_dev_ms, 1e-12), 4),
        "kv_gbs_attention": round(t_bytes / max(t_attn_ms * 1e-3, 1e-12) / 1e9, 1),
        "preemptions": st["preemptions"], "preemption_rate": round(st["preemptions"] / max(1, st["steps"]), 4),
        "avg_running_batch": round(st["sum_running"] / max(1, st["steps"]), 2),
        "latency_steps_p50": float(np.percentile(lat, 50)), "latency_steps_p99": float(np.percentile(lat, 99)),
        "ttft_steps_mean": round(float(ttft_steps.mean()), 2), "ttft_ms_mean": round(float(ttft_ms.mean()), 3),
        "prefill_tokens": st["prefill_tokens"], "prefix_hit_blocks": st["prefix_hit_blocks"],
        "swapped_out_blocks": st["swapped_out_blocks"], "swapped_in_blocks": st["swapped_in_blocks"],
        "swap_bytes": int(eng.swap_bytes),
        "upload_bytes_per_step": int(eng.upload_bytes / max(1, len(steps))),
        "oracle_check": {"rows": checked, "max_abs_err": worst, "every": "50th engine step, layer 0",
                         "oracle_s": round(t_or, 2), "oracle_keys_per_s": round(keys / max(t_or, 1e-9), 1)},
        "clocks": clk.summary(),
    }
    return line


def run_trace_bench(args):
    print(json.dumps(trace_line(args, args.trace_requests, args.trace_pool)))


def prefix_summary(args):
    """Prefix caching on a sharing-heavy trace: 1000 requests in 8 groups whose
    prompts share a head (lognormal, mean 1024 tokens, whole pages) followed by
    their own tail (lognormal, mean 128), outputs geometric with mean 256; the
    same engine with and without the prefix cache."""
    n = args.trace_requests
    off = trace_line(args, n, args.trace_pool, shared=True, caching=False)
    on = trace_line(args, n, args.trace_pool, shared=True, caching=True)
    keep = ["engine_steps", "wall_s", "output_tokens", "output_tokens_per_s", "prefill_tokens", "prefix_hit_blocks",
            "avg_running_batch", "ttft_steps_mean", "ttft_ms_mean", "latency_steps_p50", "latency_steps_p99",
            "preemptions", "oracle_check", "clocks"]
    return {
        "metric": "prefix caching: output tokens/s, prefill tokens and mean time to first token",
        "workload": "%d requests in 8 groups sharing a prompt head (lognormal mean 1024, whole pages) + own tail "
                    "(lognormal mean 128), outputs geometric mean 256, Poisson(20)/step, max batch 256, budget 8192, "
                    "chunk 512, pool %d blocks, %d layers (8B shape)" % (n, args.trace_pool, args.trace_layers),
        "no_cache": {k: off[k] for k in keep}, "cache": {k: on[k] for k in keep},
        "throughput_ratio": round(on["output_tokens_per_s"] / off["output_tokens_per_s"], 3),
        "prefill_token_ratio": round(off["prefill_tokens"] / max(1, on["prefill_tokens"]), 3),
        "ttft_ratio_no_cache_over_cache": round(off["ttft_ms_mean"] / on["ttft_ms_mean"], 3),
    }


def run_prefix_bench(args):
    print(json.dumps(prefix_summary(args)))


def swap_copy_rates(NB=8192, n=4096, reps=5):
    """Device <-> pinned host block copies of the 8B shape (32 KB per block and
    cache array) through pkv_copy_blocks: GB/s each way, CUDA events."""
    import torch
    import paged_kv_cache_tables_gb300 as pkv
    cache = torch.empty((NB, 8, 16, 128), dtype=torch.bfloat16, device="cuda").normal_()
    host = torch.empty((n, 8, 16, 128), dtype=torch.bfloat16).pin_memory()
    rng = np.random.default_rng(1)
    pairs_out = torch.from_numpy(np.stack([rng.choice(NB, n, replace=False), rng.permutation(n)], 1)
                                 .astype(np.int32)).cuda()
    pairs_in = torch.from_numpy(np.stack([rng.permutation(n), rng.choice(NB, n, replace=False)], 1)
                                .astype(np.int32)).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    nbytes = n * cache[0].numel() * 2
    res = {}
    for name, fn in (("device_to_host", lambda: pkv.copy_blocks(host, cache, pairs_out, dev_status=status)),
                     ("host_to_device", lambda: pkv.copy_blocks(cache, host, pairs_in, dev_status=status))):
        fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        res[name] = round(nbytes * reps / (e0.elapsed_time(e1) * 1e-3) / 1e9, 1)
    if int(status.item()) != 0:
        raise RuntimeError("device status %d in the swap copies" % int(status.item()))
    res["bytes_per_call"] = nbytes
    # the copy engines on one contiguous buffer of the same size: the bound
    # for the gather above
    flat_d, flat_h = cache[:n].view(-1), host.view(-1)
    for name, (dst, src) in (("memcpy_device_to_host", (flat_h, flat_d)), ("memcpy_host_to_device", (flat_d, flat_h))):
        dst.copy_(src, non_blocking=True)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            dst.copy_(src, non_blocking=True)
        e1.record()
        torch.cuda.synchronize()
        res[name] = round(nbytes * reps / (e0.elapsed_time(e1) * 1e-3) / 1e9, 1)
    return res


def preempt_summary(args):
    """Preemption by recompute against preemption by swap on the trace with a
    pool small enough to preempt: the same requests, engine and kernels; only
    what happens to a victim's blocks differs (freed and recomputed, or copied
    to pinned host memory and back)."""
    import torch
    NB = args.trace_pool if args.trace_pool != 200000 else 6250
    swap = args.swap_blocks or 2 * NB
    n = args.trace_requests
    rec = trace_line(args, n, NB)
    sw = trace_line(args, n, NB, swap_blocks=swap)
    torch.cuda.synchronize()
    rates = swap_copy_rates() if not args.no_copy_rates else None
    keep = ["engine_steps", "wall_s", "output_tokens", "output_tokens_per_s", "prefill_tokens", "preemptions",
            "swapped_out_blocks", "swapped_in_blocks", "swap_bytes", "avg_running_batch", "ttft_ms_mean",
            "latency_steps_p50", "latency_steps_p99", "oracle_check", "clocks"]
    return {
        "metric": "preemption by recompute vs by swap: output tokens/s, prefill tokens and swapped bytes",
        "workload": "%d requests as in the trace, pool %d blocks, %d layers (8B shape) over %d caches; swap space "
                    "%d blocks per cache array in pinned host memory" % (n, NB, args.trace_layers,
                                                                        args.trace_caches, swap),
        "recompute": {k: rec[k] for k in keep}, "swap": {k: sw[k] for k in keep},
        "throughput_ratio_swap_over_recompute": round(sw["output_tokens_per_s"] / rec["output_tokens_per_s"], 3),
        "swap_copy_gbs": rates,
    }


def run_preempt_bench(args):
    import torch
    if args.copy_rates_only:
        torch.cuda.set_device(0)
        print(json.dumps({"swap_copy_gbs": swap_copy_rates()}))
        return
    print(json.dumps(preempt_summary(args)))


def batching_summary(args):
    """Static against continuous batching on one synthetic trace: 500 requests
    with lognormal output lengths, the rest as in the trace workload.  Both runs
    use the same engine, kernels and pool; only the admission policy differs."""
    n = args.trace_requests if args.trace_requests != 1000 else 500
    st = trace_line(args, n, args.trace_pool, policy="static", outputs="lognormal")
    co = trace_line(args, n, args.trace_pool, policy="continuous", outputs="lognormal")
    keep = ["engine_steps", "wall_s", "output_tokens", "output_tokens_per_s", "avg_running_batch", "ttft_steps_mean",
            "ttft_ms_mean", "latency_steps_p50", "latency_steps_p99", "preemptions", "oracle_check", "clocks"]
    return {
        "metric": "static vs continuous batching: output tokens/s and mean time to first token",
        "workload": "%d requests, Poisson(20)/step, prompt lognormal mean 512, output lognormal mean 256 (sigma 1), "
                    "max batch 256, budget 8192, chunk 512, pool %d blocks, %d layers (8B shape)"
                    % (n, args.trace_pool, args.trace_layers),
        "static": {k: st[k] for k in keep}, "continuous": {k: co[k] for k in keep},
        "throughput_ratio": round(co["output_tokens_per_s"] / st["output_tokens_per_s"], 3),
        "ttft_ratio_static_over_continuous": round(st["ttft_ms_mean"] / co["ttft_ms_mean"], 3),
    }


def run_batching_bench(args):
    print(json.dumps(batching_summary(args)))



def llama1b_line(args, K, with_cpu=True):
    """The Llama-3.2-1B-shaped decode step: 64 sequences, contexts U{128..2048},
    32 query / 8 KV heads, head_dim 64, 16,384-block pool, append fused, one
    call per step.  A step streams about 143 MB of K/V, close to the 129 MB
    L2, so R = 8 independent instances (own caches, tables, queries and new
    rows; seeds apart) are stepped in turn: a step's data was last touched
    eight steps (over 1.1 GB of traffic) earlier."""
    import torch
    import paged_kv_cache_tables_gb300 as pkv
    from synth import SEEDS, make_step
    torch.cuda.set_device(0)
    R = 8
    inst = []
    for r in range(R):
        st = make_step("llama1b", seed=SEEDS["llama1b"] + 1000 * (r + 1))
        inst.append({
            "st": st, "q": to_dev_bits(st.q, st.dtype), "kn": to_dev_bits(st.k_new, st.dtype),
            "vn": to_dev_bits(st.v_new, st.dtype), "kc": to_dev_bits(st.k_cache, st.dtype),
            "vc": to_dev_bits(st.v_cache, st.dtype), "bt": torch.from_numpy(st.block_tables).cuda(),
            "cl": torch.from_numpy(st.context_lens).cuda(),
            "out": torch.empty((st.S, st.Hq, st.d), dtype=torch.bfloat16, device="cuda"),
            "work": torch.empty(pkv.decode_workspace_size(st.S, st.Hq, st.Hkv, st.d), dtype=torch.uint8,
                                device="cuda"),
            # the decode bytes of the method plus the new rows read and written
            "bytes": decode_bytes(st.context_lens, st.Hq, st.Hkv, st.d) + st.T * 2 * st.Hkv * st.d * 2 * 2,
        })
    st0 = inst[0]["st"]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()
    scale = 1.0 / math.sqrt(st0.d)

    def step(k):
        x = inst[k % R]
        pkv.paged_decode_append_attention(x["out"], x["q"], x["kn"], x["vn"], x["kc"], x["vc"], x["bt"], x["cl"],
                                          scale=scale, workspace=x["work"], dev_status=status, stream=stream)

    warm = max(args.warmup, R)
    for k in range(warm):
        step(k)
    torch.cuda.synchronize()
    with ClockSampler(0) as clk:
        torch.cuda.synchronize()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for k in range(K):
            step(k)
        t1.record(stream)
        torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError("device status %d during the benchmark" % int(status.item()))
    ms = t0.elapsed_time(t1) / K
    total_bytes = sum(inst[k % R]["bytes"] for k in range(K))
    attended = sum(float(inst[k % R]["st"].context_lens.sum()) for k in range(K))
    value = total_bytes / (ms * K * 1e-3) / 1e9
    peak, peak_kind = load_peaks()
    ctx_all = np.concatenate([x["st"].context_lens for x in inst])
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "steps": K, "warmup": warm,
        "ms_per_step": round(ms, 4),
        "config": {"workload": "llama1b-decode", "seqs_per_gpu": st0.S, "q_heads": st0.Hq, "kv_heads": st0.Hkv,
                   "head_dim": st0.d, "block_size": 16, "pool_blocks": int(st0.k_cache.shape[0]),
                   "mean_context": round(float(ctx_all.mean()), 1), "instances": R,
                   "l2": "%d instances stepped in turn, %.2f GB of K/V between two visits of one"
                         % (R, sum(x["bytes"] for x in inst) / 1e9),
                   "append": "fused (pkv_paged_decode_append_attention)", "parallelism": "dp1"},
        "attended_tokens_per_s": round(attended / (ms * K * 1e-3), 1),
        "pct_of_8tbs": round(100 * value / 8000.0, 2),
        "roofline": {"bound": "hbm", "achieved": round(value, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(value / peak, 4), "traffic": None, "peak_source": peak_kind,
                     "kernel": "paged_decode_kernel<bf16, 64, 1> with the append fused, one call (control-region "
                               "clear + decode kernel) per step"},
        "gpu_launches": LAUNCHES_PER_DECODE_CALL * K,
        "clocks": clk.summary(),
    }
    if with_cpu:
        cb = cpu_oracle_run(st0, st0.S, min_seconds=min(args.cpu_budget, 4.0))
        cb.pop("seconds")
        line["cpu_baseline"] = cb
    return line


def run_llama1b(args):
    line = llama1b_line(args, args.steps)
    out = {"metric": METRIC, "value": line["value"], "unit": "GB/s", "n_gpus": 1, "steps": line["steps"],
           "warmup": line["warmup"], "ms_per_step": line["ms_per_step"], "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic"}
    out.update({k: v for k, v in line.items() if k not in out})
    print(json.dumps(out))


def tiny_line(args, K=1000):
    """The tiny correctness step (2 sequences, contexts 18 and 15 after the
    append, 4/4 heads, head_dim 64, fp16): append fused into decode, K calls
    back to back.  Launch-bound; reported for completeness, with the oracle's
    time on the same step."""
    import torch
    import paged_kv_cache_tables_gb300 as pkv
    from synth import make_step
    import oracle
    st = make_step("tiny")
    dv = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.float16).cuda()
    q, kn, vn, kc, vc = dv(st.q), dv(st.k_new), dv(st.v_new), dv(st.k_cache), dv(st.v_cache)
    bt = torch.from_numpy(st.block_tables).cuda()
    cl = torch.from_numpy(st.context_lens).cuda()
    out = torch.empty((st.S, st.Hq, st.d), dtype=torch.float32, device="cuda")
    work = torch.empty(pkv.decode_workspace_size(st.S, st.Hq, st.Hkv, st.d), dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()
    step = lambda: pkv.paged_decode_append_attention(out, q, kn, vn, kc, vc, bt, cl, workspace=work,
                                                     dev_status=status, stream=stream)
    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(K):
        step()
    b.record(stream)
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError("device status %d in the tiny step" % int(status.item()))
    ms = a.elapsed_time(b) / K
    k_ref, v_ref = st.k_cache.copy(), st.v_cache.copy()
    oracle.append(st.k_new, st.v_new, st.slot_mapping, k_ref, v_ref, st.bs)
    t0 = time.perf_counter()
    reps = 0
    while reps == 0 or time.perf_counter() - t0 < 0.5:
        ref = oracle.decode(st.q, k_ref, v_ref, st.block_tables, st.context_lens, st.dtype)
        reps += 1
    or_ms = (time.perf_counter() - t0) / reps * 1e3
    err = float(np.abs(out.cpu().numpy().astype(np.float64) - ref).max())
    nbytes = decode_bytes(st.context_lens, st.Hq, st.Hkv, st.d) + st.T * 2 * st.Hkv * st.d * 2 * 2
    return {"workload": "tiny: 2 sequences, contexts 18 and 15 after the append, 4/4 heads, d 64, fp16, "
                        "64-block pool", "steps": K, "ms_per_step": round(ms, 5),
            "value": round(nbytes / (ms * 1e-3) / 1e9, 3), "unit": "GB/s",
            "note": "launch-bound (one call: control-region clear + decode kernel); a correctness config",
            "max_abs_err_fp32_out": err, "gpu_launches": LAUNCHES_PER_DECODE_CALL * K,
            "cpu_baseline": {"value": round(nbytes / (or_ms * 1e-3) / 1e9, 4), "unit": "GB/s", "cores": 1,
                             "kind": "oracle", "sample": "the whole step, %d passes, %.3f ms each" % (reps, or_ms)}}


def trace_summary(args, n, NB, big_steps_only=True):
    """The trace line condensed for the default bench line, with the oracle's
    time on the sampled rows extrapolated to every attended key of the trace
    (one host core) as its CPU baseline.  The roofline is taken over the steps
    whose per-layer working set exceeds 4 x L2, or (big_steps_only False, for a
    pool too small to hold such a step) over every step."""
    t = trace_line(args, n, NB)
    oc = t["oracle_check"]
    keys_total = t["attended_tokens_per_s"] * t["wall_s"]
    keep = ["workload", "engine_steps", "wall_s", "stream_s", "device_s", "attention_share_of_device_time",
            "output_tokens_per_s",
            "attended_tokens_per_s", "kv_gbs", "kv_gbs_device", "kv_gbs_attention", "kv_gbs_steps_over_4x_l2",
            "preemptions",
            "preemption_rate", "avg_running_batch", "latency_steps_p50", "latency_steps_p99", "ttft_ms_mean",
            "host_ms_per_step", "oracle_check", "clocks"]
    out = {k: t[k] for k in keep}
    peak, peak_kind = load_peaks()
    if big_steps_only:
        big = t["kv_gbs_steps_over_4x_l2"]["attention_gbs"]
        what = ("the attention calls (append, prefill and decode) of the steps whose per-layer working set exceeds "
                "4 x L2, KV bytes over their device time")
    else:
        big = t["kv_gbs_attention"]
        what = ("the attention calls (append, prefill and decode) of every step, KV bytes over their device time; "
                "the pool caps a layer's working set near 3 x L2, so some bytes may come from L2")
    out["roofline"] = {"bound": "hbm", "achieved": big, "peak": peak, "unit": "GB/s", "frac": round(big / peak, 4),
                       "traffic": None, "peak_source": peak_kind, "kernel": what}
    out["cpu_baseline"] = {"value": round(oc["oracle_keys_per_s"], 1), "unit": "attended tokens/s (per query head "
                           "group, one layer)", "cores": 1, "kind": "oracle",
                           "sample": "%d sampled layer-0 rows, %.2f s; the whole trace (%.3g attended keys x %d "
                                     "layers) would take ~%.0f s on one core (extrapolated)"
                                     % (oc["rows"], oc["oracle_s"], keys_total / args.trace_layers,
                                        args.trace_layers, keys_total / max(oc["oracle_keys_per_s"], 1e-9))}
    return out


def run_pkv(args):
    import torch
    import paged_kv_cache_tables_gb300 as pkv
    from synth import SEEDS, make_step

    ws, rank, local = dist_setup(args)
    dev_index = local if ws > 1 else 0
    # weak scaling: each rank runs its own 256-sequence step (its own seed)
    over = {}
    if args.seqs:
        over["S"] = args.seqs
    if args.pool:
        over["NB"] = args.pool
    st = make_step("llama8b", seed=SEEDS["llama8b"] + rank, **over)
    S, Hq, Hkv, d = st.S, st.Hq, st.Hkv, st.d
    q = to_dev_bits(st.q, st.dtype)
    kn, vn = to_dev_bits(st.k_new, st.dtype), to_dev_bits(st.v_new, st.dtype)
    kc, vc = to_dev_bits(st.k_cache, st.dtype), to_dev_bits(st.v_cache, st.dtype)
    slots = torch.from_numpy(st.slot_mapping).cuda()
    bt = torch.from_numpy(st.block_tables).cuda()
    cl = torch.from_numpy(st.context_lens).cuda()
    out = torch.empty((S, Hq, d), dtype=torch.bfloat16, device="cuda")
    ws_bytes = pkv.decode_workspace_size(S, Hq, Hkv, d)
    work = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()
    scale = 1.0 / math.sqrt(d)

    # the step: append of the 256 new tokens and decode attention, in one
    # launch (pkv_paged_decode_append_attention)
    def step():
        pkv.paged_decode_append_attention(out, q, kn, vn, kc, vc, bt, cl, scale=scale, workspace=work,
                                          dev_status=status, stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    K = args.steps
    barrier(ws)
    with ClockSampler(dev_index) as clk:
        torch.cuda.synchronize()
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        t_start.record(stream)
        for k in range(K):
            step()
        t_end.record(stream)
        torch.cuda.synchronize()
    barrier(ws)
    total_ms = max_over_ranks(t_start.elapsed_time(t_end), ws)
    ms_step = total_ms / K
    # one call per step and nothing else in the region: the call's two
    # launches (control-region clear, then the decode kernel) average the
    # region's time over K, gaps included -- the decode kernel's own time is
    # at most this
    fused_ms = t_start.elapsed_time(t_end) / K
    if int(status.item()) != 0:
        raise RuntimeError("device status %d during the benchmark" % int(status.item()))

    # the same step as two launches (pkv_kv_append, then
    # pkv_paged_decode_attention), for comparison
    for _ in range(args.warmup):
        pkv.kv_append(kn, vn, slots, kc, vc, dev_status=status, stream=stream)
        pkv.paged_decode_attention(out, q, kc, vc, bt, cl, scale=scale, workspace=work, dev_status=status,
                                   stream=stream)
    torch.cuda.synchronize()
    K2 = min(K, 200)
    ev2 = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K2)]
    for k in range(K2):
        ev2[k][0].record(stream)
        pkv.kv_append(kn, vn, slots, kc, vc, dev_status=status, stream=stream)
        ev2[k][1].record(stream)
        pkv.paged_decode_attention(out, q, kc, vc, bt, cl, scale=scale, workspace=work, dev_status=status,
                                   stream=stream)
        ev2[k][2].record(stream)
    torch.cuda.synchronize()
    app_ms = statistics.mean(ev2[k][0].elapsed_time(ev2[k][1]) for k in range(K2))
    dec_ms = statistics.mean(ev2[k][1].elapsed_time(ev2[k][2]) for k in range(K2))
    two_ms = statistics.mean(ev2[k][0].elapsed_time(ev2[k][2]) for k in range(K2))
    if int(status.item()) != 0:
        raise RuntimeError("device status %d in the two-launch step" % int(status.item()))

    dbytes = decode_bytes(st.context_lens, Hq, Hkv, d)
    # the fused append reads the new K/V rows and writes them to the cache
    step_bytes = dbytes + st.T * 2 * Hkv * d * 2 * 2
    value = step_bytes * ws / (ms_step * 1e-3) / 1e9
    attended = float(st.context_lens.sum())

    # ---- end to end through the public API with host buffers ----
    if args.no_e2e:
        e2e_value, e2e_ms, h2d, d2h = None, None, 0, 0
    else:
        e2e_value, e2e_ms, h2d, d2h = run_e2e(args, ws, st, q, kn, vn, bt, cl, out, kc, vc, work, status,
                                              stream, scale, step_bytes, K)
    if rank != 0:
        return
    peak, peak_kind = load_peaks()
    achieved = step_bytes / (fused_ms * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": ws, "steps": K, "warmup": args.warmup,
        "ms_per_step": round(ms_step, 4), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": step_config(st, ws),
        "attended_tokens_per_s": round(attended * ws / (ms_step * 1e-3), 1),
        "attended_q_head_tokens_per_s": round(attended * Hq * ws / (ms_step * 1e-3), 1),
        # bytes the kernel touches: whole 16-token blocks, so the masked tail
        # of each sequence's last block counts too
        "touched_bytes_per_step": int(step_bytes + (((st.context_lens + 15) // 16 * 16 - st.context_lens).sum())
                                      * 2 * Hkv * d * 2),
        "pct_of_8tbs": round(100 * value / 8000.0, 2),
        "kernels_ms": {"paged_decode_append_attention (clear + decode kernels)": round(fused_ms, 4)},
        "two_launch_step": {"ms_per_step": round(two_ms, 4), "kv_append_ms": round(app_ms, 4),
                            "paged_decode_attention_ms": round(dec_ms, 4), "steps": K2,
                            "decode_gbs": round(dbytes / (dec_ms * 1e-3) / 1e9, 1)},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": decode_traffic(not (args.seqs or args.pool)),
                     "peak_source": peak_kind,
                     "kernel": "paged_decode_kernel with the append fused (split-KV, in-kernel merge), "
                               "bytes %d per launch; timed together with the control-region clear launched "
                               "before it (%d bytes zeroed)" % (step_bytes, clear_bytes(S, Hkv)),
                     "traffic_source": "ncu dram__bytes_read.sum + dram__bytes_write.sum of one full-size "
                                       "launch of this decode source (profiles/paged_decode_llama8b_launches.md)"},
        "e2e": None if e2e_value is None else {
            "value": round(e2e_value, 1), "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": round(e2e_ms, 4)},
        "gpu_launches": LAUNCHES_PER_DECODE_CALL * K,
        "clocks": clk.summary(),
    }
    if not args.no_mixed:
        line["mixed_step"] = run_mixed(args)
    if not args.no_more_configs and ws == 1:
        # the other configurations of the workload family, each with its
        # own roofline fraction and oracle baseline
        line["llama1b_step"] = llama1b_line(args, min(K, 1000))
        line["trace"] = trace_summary(args, args.trace_requests, args.trace_pool)
        line["trace_small_pool"] = trace_summary(args, args.trace_requests, 6250, big_steps_only=False)
        line["tiny_step"] = tiny_line(args)
        # the NEXT rows on the same engine: static against continuous
        # batching, prefix caching, preemption by swap against recompute
        # (the pages' batching gains are context, not targets)
        line["next"] = {"static_vs_continuous": batching_summary(args), "prefix_caching": prefix_summary(args),
                        "swap_vs_recompute": preempt_summary(args)}
    if not args.no_cpu_baseline and ws == 1:
        k = oracle_sample_size(st, args.cpu_budget)
        cb = cpu_oracle_run(st, k, min_seconds=args.cpu_budget)
        # one pass over the whole step, from the timed sample
        one_pass = cb.pop("seconds") * float(st.context_lens.sum()) / float(st.context_lens[:k].sum())
        try:
            cb["all_cores"] = cpu_oracle_all_cores(st, args.cpu_budget / 2, one_pass)
        except Exception as e:   # a host without shared memory or process start: the one-core figure stands
            cb["all_cores"] = {"unavailable": "%s: %s" % (type(e).__name__, e)}
        line["cpu_baseline"] = cb
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="pkv", choices=["pkv", "reference"])
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-mixed", action="store_true", help="skip the mixed prefill + decode step")
    ap.add_argument("--no-more-configs", action="store_true",
                    help="skip the 1B-shaped step and the two traces in the default line")
    ap.add_argument("--mixed-steps", type=int, default=50)
    ap.add_argument("--mixed-chunks", type=int, default=0, help="override the prefill chunk count (profiling)")
    ap.add_argument("--mixed-prior", type=int, default=-1,
                    help="give every prefill chunk this prior context instead of U{0..4096} (profiling)")
    ap.add_argument("--only-mixed", action="store_true", help="run only the mixed step (profiling)")
    ap.add_argument("--mixed-decode-sms", default="",
                    help="comma-separated decode SM counts at which to time the side-by-side mixed step too")
    ap.add_argument("--workload", default="llama8b",
                    choices=["llama8b", "llama1b", "trace", "batching", "prefix", "preempt"],
                    help="llama1b: the Llama-3.2-1B-shaped decode step (8 instances in turn); "
                         "trace: the continuous-batching trace; batching: static vs continuous on one trace; "
                         "prefix: with and without the prefix cache on a sharing-heavy trace; preempt: recompute "
                         "vs swap on the trace with a small pool")
    ap.add_argument("--swap-blocks", type=int, default=0, help="host swap slots for --workload preempt")
    ap.add_argument("--steps-jsonl", default="", help="trace workloads: append one JSON record per engine step here")
    ap.add_argument("--copy-rates-only", action="store_true", help="--workload preempt: only the block copy rates")
    ap.add_argument("--no-copy-rates", action="store_true")
    ap.add_argument("--trace-requests", type=int, default=1000)
    ap.add_argument("--trace-layers", type=int, default=32)
    ap.add_argument("--trace-caches", type=int, default=4)
    ap.add_argument("--trace-pool", type=int, default=200000)
    ap.add_argument("--seqs", type=int, default=0, help="override the sequence count (profiling cases)")
    ap.add_argument("--pool", type=int, default=0, help="override the pool size in blocks (profiling cases)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.workload == "llama1b":
        run_llama1b(args)
        return
    if args.workload == "trace":
        run_trace_bench(args)
        return
    if args.workload == "batching":
        run_batching_bench(args)
        return
    if args.workload == "prefix":
        run_prefix_bench(args)
        return
    if args.workload == "preempt":
        run_preempt_bench(args)
        return
    if args.only_mixed:
        import torch
        torch.cuda.set_device(0)
        args.warmup = max(args.warmup, 3)
        print(json.dumps({"mixed_step": run_mixed(args)}))
        return
    if args.impl == "reference":
        # each reference step is a bounded oracle sample sized so the run takes a few minutes
        run_reference(args)
    else:
        run_pkv(args)


if __name__ == "__main__":
    main()
