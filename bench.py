#!/usr/bin/env python
"""Benchmark of split-KV MLA decode (partial + LSE combine) on GB300.

Default workload: dense MLA decode, batch 1, H=16, d_c=512 + d_r=64, context
T=8192, bf16 N(0,1) inputs, scale 1/sqrt(576).  One *step* is one pass of the
hot path over every cache copy: the copies (distinct caches, as the layers of
a model would be) together exceed 3x the L2, so every call reads its cache
from HBM.  The calls of one step are captured as one CUDA graph and replayed.

Prints ONE JSON line: metric/value (achieved HBM GB/s of the whole call,
algorithmic bytes / time per call), us_per_call, the roofline of the partial
kernel (live CUDA-event timing), the end-to-end number through the C ABI with
host buffers, the oracle timed on the host cores (all threads and one), the SM
clocks seen during the timed region, a `sweep` of the five workloads and the
context sweep at H=16 (us per call, the partial kernel alone, fractions of the
roofline), a PDL on/off A/B (`pdl_ab`) and the `floor` (what a call costs with
no decode work: empty kernels, a bare bulk read, a bare row gather, beside
the calls).  ``--impl reference`` times the fp64
CPU oracle instead.  ``--details PATH`` also writes a longer table (split sweep,
E4M3 cache, fused step, projection) to PATH.

Multi-GPU: replicas only (each rank runs its own copy of the workload; no
collective on the data path; max time over ranks).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

import workloads  # noqa: E402

METRIC = "MLA decode µs/call and achieved HBM GB/s (fraction of roofline) on 1 GB300"
ROW_BYTES = 1152
FLOP_PER_ROW_HEAD = 2 * (576 + 512)


# --------------------------------------------------------------------------- utils
def log(*a):
    print(*a, file=sys.stderr, flush=True)


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# the sources each kernel is compiled from (its traffic counters stay valid while they are unchanged)
KERNEL_SOURCES = {
    "mla_partial_mma_kernel": ("mla_partial_mma.cu", "tc_utils.cuh", "device_utils.cuh", "mla_internal.h",
                               "slicing.cuh"),
    "mla_partial_tc_kernel": ("mla_partial_tc.cu", "tc_utils.cuh", "device_utils.cuh", "mla_internal.h",
                              "slicing.cuh"),
    "mla_combine_kernel": ("mla_combine.cu", "device_utils.cuh", "mla_internal.h"),
}


def kernel_source_hash(kernel):
    h = hashlib.sha256()
    for fn in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "decode_attention_mla_gb300", "csrc", fn), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def ncu_traffic(kernel, workload):
    """Per-launch DRAM bytes of `kernel` from the committed ncu summary, or None
    if the kernel source changed since the counters were taken."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    e = d.get(kernel, {}).get(workload)
    if not e or kernel not in KERNEL_SOURCES or e.get("source_sha256") != kernel_source_hash(kernel):
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi SM clocks and throttle reasons sampled every 200 ms."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.out = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()
        return False

    def summary(self):
        if not self.out:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# --------------------------------------------------------------------------- workloads
class DenseBench:
    """Dense decode over `copies` distinct caches of T rows (B=1)."""

    def __init__(self, T, H, copies, splits, pdl, seed=0, variant=0, fp8=False):
        import decode_attention_mla_gb300 as mla
        self.mla = mla
        d = torch.device("cuda")
        self.T, self.H, self.copies = T, H, copies
        x = workloads.dense(1, H, T, seed=seed)
        self.host = x
        self.kv_scale = 1.0
        kv0 = x.kv
        if fp8:
            # the same draws as an E4M3 cache with one scale (576-byte rows)
            kv0, self.kv_scale = workloads.to_e4m3(x.kv)
        # copy 0 is the seeded workload; the others are shifted versions (distinct bytes, same distribution)
        self.kv = [kv0.to(d)]
        for c in range(1, copies):
            self.kv.append(torch.roll(self.kv[0], shifts=c * 37, dims=0))
        self.q = [x.q.to(d) for _ in range(copies)]
        self.d_pos = x.d_pos.to(d)
        self.out = [torch.empty(1, H, 512, device=d) for _ in range(copies)]
        self.lse = [torch.empty(1, H, device=d) for _ in range(copies)]
        self.plan = mla.plan(batch=1, heads=H, max_ctx=T, scale=x.scale, splits=splits, pdl=pdl, variant=variant,
                             kv_fp8=fp8)
        self.scratch = mla.alloc_scratch(self.plan)
        self.args = [mla.make_args(self.q[c], self.kv[c], self.out[c], self.lse[c], d_pos=self.d_pos,
                                   kv_scale=self.kv_scale) for c in range(copies)]
        row_bytes = ROW_BYTES // 2 if fp8 else ROW_BYTES
        self.alg_bytes = T * row_bytes + H * 576 * 2 + 4 + H * 512 * 4 + H * 4
        self.flops = T * H * FLOP_PER_ROW_HEAD

    def call(self, c, stream=None):
        self.mla.forward_args(self.plan, self.args[c], self.scratch, stream)

    def partial(self, c, stream=None):
        self.mla.run(self.plan, self.args[c], self.scratch, stream)

    def replan(self, pdl):
        """The same plan (split count, kernel) launched with or without PDL."""
        self.plan = self.mla.plan(batch=1, heads=self.H, max_ctx=self.T, scale=self.host.scale,
                                  splits=self.plan.splits, pdl=pdl, variant=self.plan.variant,
                                  kv_fp8=bool(self.plan.shape.kv_fp8))


class SparseBench:
    """Sparse decode; `copies` distinct caches when one cache is below 3x L2."""

    def __init__(self, name, copies, splits, pdl, seed=0, variant=0, device_cache=False):
        import decode_attention_mla_gb300 as mla
        self.mla = mla
        d = torch.device("cuda")
        if device_cache:
            # timing only: the recipe's lengths, offsets, queries and index lists,
            # with the cache rows drawn N(0,1) bf16 on the device (drawing ~5 GB on
            # the host takes tens of seconds); the parity tests use the host draw
            x = sparse_recipe_without_cache(name, seed)
            total = int(x.cache_len.to(torch.int64).sum())
            gen = torch.Generator(device=d).manual_seed(seed)
            kv0 = torch.empty(total, 576, dtype=torch.bfloat16, device=d)
            for r0 in range(0, total, 1 << 20):
                r1 = min(total, r0 + (1 << 20))
                kv0[r0:r1] = torch.randn(r1 - r0, 576, generator=gen, device=d).to(torch.bfloat16)
        else:
            x = workloads.make(name, seed=seed)
            kv0 = x.kv.to(d)
        self.host = x
        B, H, _ = x.q.shape
        topk = x.indices.shape[1]
        self.copies = copies
        self.kv = [kv0]
        for c in range(1, copies):
            self.kv.append(torch.roll(self.kv[0], shifts=c * 37, dims=0))
        self.q = x.q.to(d)
        self.idx = x.indices.to(d)
        self.len = x.cache_len.to(d)
        self.off = x.row_offset.to(d)
        self.out = [torch.empty(B, H, 512, device=d) for _ in range(copies)]
        self.lse = [torch.empty(B, H, device=d) for _ in range(copies)]
        self.plan = mla.plan(batch=B, heads=H, sparse=True, topk=topk, scale=x.scale, splits=splits, pdl=pdl,
                             variant=variant)
        self.scratch = mla.alloc_scratch(self.plan)
        self.args = [mla.make_args(self.q, self.kv[c], self.out[c], self.lse[c], indices=self.idx,
                                   cache_len=self.len, row_offset=self.off) for c in range(copies)]
        valid = int(((x.indices >= 0) & (x.indices < x.cache_len[:, None])).sum())
        self.alg_bytes = valid * ROW_BYTES + B * H * 576 * 2 + B * topk * 4 + B * 12 + B * H * 512 * 4 + B * H * 4
        self.flops = valid * H * FLOP_PER_ROW_HEAD

    def call(self, c, stream=None):
        self.mla.forward_args(self.plan, self.args[c], self.scratch, stream)

    def partial(self, c, stream=None):
        self.mla.run(self.plan, self.args[c], self.scratch, stream)



def sparse_recipe_without_cache(name, seed):
    """The sparse workload's lengths, offsets, queries and index lists as the
    input recipe draws them, with an empty cache (rows drawn elsewhere)."""
    w = workloads.WORKLOADS[name]
    B, H, topk = w["B"], w["H"], w["topk"]
    if "cache" in w:
        lens = torch.full((B,), w["cache"], dtype=torch.int32)
    else:
        lens = workloads.ragged_lengths(B, w["len_lo"], w["len_hi"], seed=seed)
    offs = torch.zeros(B, dtype=torch.int64)
    if B > 1:
        offs[1:] = torch.cumsum(lens.to(torch.int64), 0)[:-1]
    q = workloads.randn_bf16(B * H, 576, seed=seed, stream=1).view(B, H, 576)
    idx = torch.stack([workloads.unique_indices(int(lens[b]), topk, seed=seed, stream=3, chunk=b) for b in range(B)])
    return workloads.SparseInputs(q=q, kv=torch.empty(0, 576, dtype=torch.bfloat16), indices=idx.contiguous(),
                                  cache_len=lens, row_offset=offs)


class GraphBench:
    """Multi-step dense decode, H=128, start context T0, `steps` steps per graph.
    `layers` distinct caches (as the layers of a model) share one d_pos: each
    step appends a row to every layer's cache, runs partial + combine per layer,
    then advances d_pos once.  The layers together exceed 3x L2."""

    def __init__(self, H, T0, steps, layers, splits, pdl, seed=0, variant=0, fused=False):
        import decode_attention_mla_gb300 as mla
        self.mla = mla
        self.fused = fused
        d = torch.device("cuda")
        g = workloads.graph(H, T0, steps, seed=seed)
        self.g, self.H, self.T0, self.steps, self.copies = g, H, T0, steps, layers
        base = g.kv.to(d)
        self.kv = [base] + [torch.roll(base, shifts=c * 37, dims=0) for c in range(1, layers)]
        self.kv_init = [k.clone() for k in self.kv] if layers * base.numel() * 2 < (8 << 30) else None
        rows = g.new_rows.to(d)
        self.new_rows = [rows] + [torch.roll(rows, shifts=c, dims=0) for c in range(1, layers)]
        self.q = g.q_steps.to(d)
        self.d_pos = torch.tensor([T0], dtype=torch.int32, device=d)
        self.d_pos0 = self.d_pos.clone()
        self.out = [torch.empty(steps, 1, H, 512, device=d) for _ in range(layers)]
        self.lse = [torch.empty(steps, 1, H, device=d) for _ in range(layers)]
        self.plan = mla.plan(batch=1, heads=H, max_ctx=T0 + steps, scale=g.scale, splits=splits, pdl=pdl,
                             variant=variant)
        self.scratch = mla.alloc_scratch(self.plan)
        self.args = [[mla.make_args(self.q[k], self.kv[l], self.out[l][k], self.lse[l][k], d_pos=self.d_pos)
                      for k in range(steps)] for l in range(layers)]
        self.g_scale = g.scale
        mean_rows = T0 + 1 + (steps - 1) / 2.0
        self.alg_bytes = mean_rows * ROW_BYTES + H * 576 * 2 + H * 512 * 4 + H * 4 + 2 * ROW_BYTES + 8
        self.flops = mean_rows * H * FLOP_PER_ROW_HEAD
        self.calls = steps * layers

    def replan(self, pdl):
        self.plan = self.mla.plan(batch=1, heads=self.H, max_ctx=self.T0 + self.steps, scale=self.g_scale,
                                  splits=self.plan.splits, pdl=pdl, variant=self.plan.variant)

    def loop(self, _c=0, stream=None):
        mla = self.mla
        self.d_pos.copy_(self.d_pos0)
        for k in range(self.steps):
            for l in range(self.copies):
                if self.fused:
                    # append, partial + combine and (after the last layer) the advance in two launches
                    mla.forward_step_args(self.plan, self.args[l][k], self.scratch, self.new_rows[l][k:k + 1],
                                          advance=l == self.copies - 1)
                else:
                    mla.append(self.kv[l], self.new_rows[l][k:k + 1], self.d_pos)
                    mla.forward_args(self.plan, self.args[l][k], self.scratch)
            if not self.fused:
                mla.advance(self.d_pos)


def capture(fn, n):
    """CUDA graph of fn(0..n-1) on a side stream (warmed up eagerly first)."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for c in range(n):
            fn(c)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for c in range(n):
            fn(c)
    torch.cuda.synchronize()
    return g


def time_graph(g, reps, warmup):
    for _ in range(warmup):
        g.replay()
    torch.cuda.synchronize()
    st = torch.cuda.current_stream()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(st)
    for _ in range(reps):
        g.replay()
    e1.record(st)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / 1e3          # seconds


def per_rep_times(g, reps):
    """Individual replay times (seconds), for the spread."""
    st = torch.cuda.current_stream()
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(reps + 1)]
    evs[0].record(st)
    for r in range(reps):
        g.replay()
        evs[r + 1].record(st)
    torch.cuda.synchronize()
    return [evs[r].elapsed_time(evs[r + 1]) / 1e3 for r in range(reps)]


def l2_bytes():
    return int(getattr(torch.cuda.get_device_properties(0), "L2_cache_size", 128 << 20))


def copies_for(bytes_per_cache):
    return max(1, math.ceil(3 * l2_bytes() / bytes_per_cache))


# --------------------------------------------------------------------------- oracle timing
def oracle_time_dense(x, budget_s, threads=0):
    import oracle
    n = 0
    t0 = time.perf_counter()
    while True:
        oracle.decode(x.q, x.kv, scale=x.scale, d_pos=x.d_pos, n_threads=threads)
        n += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            return el / n, n


def cpu_model():
    """The host CPU's model name (x86 'model name', else lscpu's, else the Arm part id)."""
    try:
        with open("/proc/cpuinfo") as f:
            text = f.read()
    except OSError:
        text = ""
    for line in text.splitlines():
        if line.lower().startswith("model name"):
            return line.split(":", 1)[1].strip()
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    parts = [line.split(":", 1)[1].strip() for line in text.splitlines()
             if line.lower().startswith(("cpu implementer", "cpu part"))][:2]
    return "implementer/part " + "/".join(parts) if parts else "unknown"


def cpu_baseline(bench, budget_s):
    """The oracle on the host cores, on the bench's own dense workload: all
    hardware threads (parallel over request and head) and one thread."""
    import oracle
    threads = oracle.hardware_threads()
    per_call, n = oracle_time_dense(bench.host, budget_s, threads)
    per_call_1, n1 = oracle_time_dense(bench.host, budget_s / 2, 1)
    return {"value": bench.alg_bytes / per_call / 1e9, "unit": "GB/s", "cores": threads, "kind": "oracle",
            "cpu_model": cpu_model(), "nproc": os.cpu_count(),
            "us_per_call": per_call * 1e6,
            "single_thread": {"value": bench.alg_bytes / per_call_1 / 1e9, "unit": "GB/s", "cores": 1,
                              "us_per_call": per_call_1 * 1e6, "calls": n1},
            "sample": f"{n} full calls of the dense T={bench.T} H={bench.H} workload (fp64 oracle, "
                      f"{threads} threads), {per_call * 1e3:.1f} ms/call; single thread: {n1} calls, "
                      f"{per_call_1 * 1e3:.1f} ms/call"}


# --------------------------------------------------------------------------- e2e
def e2e_dense(bench, calls):
    """Through the public C ABI with host buffers, the way a graph-resident
    decode loop runs it: per call, one replay of a CUDA graph that holds the
    H2D copies of q and d_pos from pinned memory, partial + combine, and the
    D2H copies of out and lse, then a host synchronisation to read the result.
    The same per-call work issued eagerly (four copies and two launches from
    Python, no graph) is reported beside it as `eager_us_per_call`."""
    mla = bench.mla
    H = bench.H
    q_h = bench.host.q.pin_memory()
    dpos_h = bench.host.d_pos.pin_memory()
    out_h = torch.empty(1, H, 512).pin_memory()
    lse_h = torch.empty(1, H).pin_memory()
    q_d = torch.empty_like(bench.q[0])
    dpos_d = torch.empty_like(bench.d_pos)
    out_d = torch.empty(1, H, 512, device="cuda")
    lse_d = torch.empty(1, H, device="cuda")
    st = torch.cuda.current_stream()
    args = [mla.make_args(q_d, bench.kv[c], out_d, lse_d, d_pos=dpos_d) for c in range(bench.copies)]

    def work(c):
        q_d.copy_(q_h, non_blocking=True)
        dpos_d.copy_(dpos_h, non_blocking=True)
        mla.forward_args(bench.plan, args[c % bench.copies], bench.scratch)
        out_h.copy_(out_d, non_blocking=True)
        lse_h.copy_(lse_d, non_blocking=True)

    def timed(one):
        for c in range(20):
            one(c)
        t0 = time.perf_counter()
        for c in range(calls):
            one(c)
        return (time.perf_counter() - t0) / calls

    def eager(c):
        work(c)
        st.synchronize()

    per_eager = timed(eager)
    graphs = [capture(lambda _c, c=c: work(c), 1) for c in range(bench.copies)]

    def replay(c):
        graphs[c % bench.copies].replay()
        st.synchronize()

    per = timed(replay)
    # the last replay's result really came back to the host
    if not (torch.equal(out_h, out_d.cpu()) and torch.equal(lse_h, lse_d.cpu()) and torch.isfinite(out_h).all()):
        raise RuntimeError("end-to-end loop: host copies of out/lse do not match the device")
    h2d = q_h.numel() * 2 + 4
    d2h = out_h.numel() * 4 + lse_h.numel() * 4
    return {"value": bench.alg_bytes / per / 1e9, "unit": "GB/s", "us_per_call": per * 1e6,
            "h2d_bytes_per_step": h2d * bench.copies, "d2h_bytes_per_step": d2h * bench.copies,
            "calls": calls, "eager_us_per_call": per_eager * 1e6,
            "how": "per call: one CUDA-graph replay (H2D q, d_pos; partial + combine; D2H out, lse) + host sync"}


# --------------------------------------------------------------------------- replicas
def max_over_ranks(elapsed: float, world: int) -> float:
    """The slowest rank's time (every rank gets it); identity at world 1."""
    if world <= 1:
        return elapsed
    import torch.distributed as dist
    t = torch.tensor([elapsed], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(alg_bytes_per_call: int, calls_per_rank: int, world: int, elapsed_max: float) -> float:
    """Algorithmic bytes all ranks moved / the slowest rank's time, in GB/s."""
    return world * alg_bytes_per_call * calls_per_rank / elapsed_max / 1e9


# --------------------------------------------------------------------------- main arms
class CpuSide:
    """What the oracle timing needs of a bench (its host inputs and sizes)."""

    def __init__(self, bench):
        self.host, self.T, self.H, self.alg_bytes = bench.host, bench.T, bench.H, bench.alg_bytes


def workload_config(world):
    """The timed workload, the same keys in both arms."""
    return {"workload": "dense_t8192", "batch": 1, "heads": 16, "d_latent": 512, "d_rope": 64, "context": 8192,
            "l2": "inputs larger than L2: every step reads distinct caches totalling more than 3x L2",
            "parallelism": f"replicas x{world}"}


def run_ours(args, rank, world):
    import decode_attention_mla_gb300 as mla
    from decode_attention_mla_gb300 import build as mla_build
    mla_build.build()
    dev_index = int(os.environ.get("LOCAL_RANK", 0))
    torch.cuda.set_device(dev_index)
    P = peaks()
    T = 8192
    H = 16
    copies = copies_for(T * ROW_BYTES)
    bench = DenseBench(T, H, copies, args.splits, bool(args.pdl), variant=args.variant)
    g = capture(bench.call, copies)
    gp = capture(bench.partial, copies)
    # choose K for ~2 s of timed work unless given
    t_one = time_graph(g, 20, 3) / 20
    steps = args.steps if args.steps > 0 else max(10, int(2.0 / max(t_one, 1e-6)))
    warm = max(3, args.warmup)

    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(dev_index) as clk:
        elapsed = time_graph(g, steps, warm)
    torch.cuda.synchronize()
    elapsed = max_over_ranks(elapsed, world)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    calls = steps * copies
    us_call = elapsed / calls * 1e6
    value = whole_job_gbs(bench.alg_bytes, calls, world, elapsed)

    # dominant kernel (split partial): live CUDA-event time per launch, same copies
    t_part = time_graph(gp, max(10, steps // 2), warm) / (max(10, steps // 2) * copies)
    part_bytes = T * ROW_BYTES + H * 576 * 2 + 4      # KV rows + q + d_pos read by the partial kernel
    achieved = part_bytes / t_part / 1e9
    kname = "mla_partial_mma_kernel" if bench.plan.variant == 1 else "mla_partial_tc_kernel"
    traffic = ncu_traffic(kname, "dense_t8192")
    reps = per_rep_times(g, 20)
    per_call_reps = [r / copies * 1e6 for r in reps]
    cpu_bench = CpuSide(bench)
    clocks = clk.summary()

    result = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": steps,
        "warmup": warm, "ms_per_step": round(elapsed / steps * 1e3, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": workload_config(world),
        "launch": {"splits": bench.plan.splits, "pdl": bool(args.pdl),
                   "kernel": KERNEL_NAMES.get(bench.plan.variant, str(bench.plan.variant)),
                   "calls_per_step": copies,
                   "l2_detail": f"{copies} distinct caches x {T * ROW_BYTES / 1e6:.2f} MB "
                                f"= {copies * T * ROW_BYTES / 1e6:.0f} MB per step (> 3x L2 {l2_bytes() / 1e6:.0f} MB)"},
        "us_per_call": round(us_call, 4),
        "us_per_call_reps": [round(x, 4) for x in per_call_reps],
        "us_per_call_sd": round(statistics.pstdev(per_call_reps), 4),
        "roofline_us": round(bench.alg_bytes / (P["hbm_gbs"] * 1e9) * 1e6, 4),
        "frac_of_roofline": round(bench.alg_bytes / (P["hbm_gbs"] * 1e9) / (us_call * 1e-6), 4),
        "frac_of_roofline_8tbs": round(bench.alg_bytes / 8e12 / (us_call * 1e-6), 4),
        "alg_bytes_per_call": bench.alg_bytes,
        "roofline": {"kernel": kname, "bound": "hbm", "achieved": round(achieved, 1),
                     "peak": P["hbm_gbs"], "peak_source": P["source"] + " (burst copy)", "unit": "GB/s",
                     "frac": round(achieved / P["hbm_gbs"], 4), "traffic": traffic,
                     "alg_bytes_per_launch": part_bytes, "us_per_launch": round(t_part * 1e6, 4)},
        "gpu_launches": 2 * calls,
        "clocks": clocks,
    }
    if rank == 0:
        result["e2e"] = e2e_dense(bench, calls=2000)
        del g, gp, bench
        torch.cuda.empty_cache()
        if not args.no_sweep:
            t0 = time.perf_counter()
            result["sweep"] = sweep_rows(args, P)
            result["pdl_ab"] = pdl_ab(args, P)
            result["floor"] = floor_rows(args, P)
            result["sweep_seconds"] = round(time.perf_counter() - t0, 1)
        if not args.no_cpu_baseline:
            result["cpu_baseline"] = cpu_baseline(cpu_bench, args.cpu_seconds)
        if args.details:
            result["details_file"] = args.details
            write_details(args, P)
    return result


def run_reference(args):
    import oracle
    T, H = 8192, 16
    x = workloads.dense(1, H, T, seed=0)
    alg = T * ROW_BYTES + H * 576 * 2 + 4 + H * 512 * 4 + H * 4
    threads = oracle.hardware_threads()
    steps = args.steps if args.steps > 0 else 10
    for _ in range(max(1, min(args.warmup, 3))):
        oracle.decode(x.q, x.kv, scale=x.scale, d_pos=x.d_pos, n_threads=threads)
    t0 = time.perf_counter()
    for _ in range(steps):
        oracle.decode(x.q, x.kv, scale=x.scale, d_pos=x.d_pos, n_threads=threads)
    el = time.perf_counter() - t0
    value = alg * steps / el / 1e9
    return {"metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": 1, "steps": steps,
            "warmup": args.warmup, "ms_per_step": round(el / steps * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": workload_config(int(os.environ.get("WORLD_SIZE", "1"))),
            "us_per_call": round(el / steps * 1e6, 1),
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                             "cpu_model": cpu_model(), "nproc": os.cpu_count(),
                             "sample": f"{steps} full calls of dense T={T} H={H}"},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


# --------------------------------------------------------------------------- details (all workloads)
def time_bench(bench, reps=200, warm=5):
    g = capture(bench.call, bench.copies)
    gp = capture(bench.partial, bench.copies)
    el = time_graph(g, reps, warm)
    elp = time_graph(gp, reps, warm)
    rep_list = per_rep_times(g, 20)
    us = el / (reps * bench.copies) * 1e6
    return us, elp / (reps * bench.copies) * 1e6, [r / bench.copies * 1e6 for r in rep_list]


def time_graph_bench(gb, reps=10, warm=3):
    g = capture(gb.loop, 1)
    el = time_graph(g, reps, warm)
    rep_list = per_rep_times(g, 5)
    us = el / (reps * gb.calls) * 1e6
    return us, None, [r / gb.calls * 1e6 for r in rep_list]


def project_timing(H, V, reps=50):
    """mla_decode_project on one merged latent [1, H, 512] with distinct bf16
    wv_b copies [H, V, 512] (together > 3x L2), captured as one graph."""
    import decode_attention_mla_gb300 as mla
    d = torch.device("cuda")
    g = torch.Generator().manual_seed(5)
    wbytes = H * V * 512 * 2
    copies = copies_for(wbytes)
    w0 = (torch.randn(H, V, 512, generator=g) / 512 ** 0.5).to(torch.bfloat16).to(d)
    ws = [w0] + [torch.roll(w0, shifts=c, dims=2) for c in range(1, copies)]
    lat = torch.randn(1, H, 512, generator=g).to(d)
    y = torch.empty(1, H, V, device=d)
    gr = capture(lambda c: mla.project(lat, ws[c], y, pdl=True), copies)
    el = time_graph(gr, reps, 3)
    us = el / (reps * copies) * 1e6
    del ws
    torch.cuda.empty_cache()
    return {"us": us, "copies": copies, "bytes": wbytes + H * 512 * 4 + H * V * 4}


KERNEL_NAMES = {1: "warp-mma", 2: "tcgen05-16", 3: "tcgen05-32", 4: "tcgen05-64", 5: "warp-mma-tcgen05-pv"}


def sweep_row(name, bench, us, us_part, reps, P, per="call", tensor_bound=False):
    """One workload's figures: us per call (partial + combine), the partial
    kernel alone, and both against the roofline (the slower of the bytes at
    the measured HBM copy bandwidth and, where it binds, the flops at the
    sustained bf16 tensor rate)."""
    hbm_us = bench.alg_bytes / (P["hbm_gbs"] * 1e9) * 1e6
    tensor_us = bench.flops / (P["bf16_tflops_sustained"] * 1e12) * 1e6
    roof_us = max(hbm_us, tensor_us) if tensor_bound else hbm_us
    r = {"workload": name, "per": per, "kernel": KERNEL_NAMES.get(bench.plan.variant, str(bench.plan.variant)),
         "splits": bench.plan.splits, "copies": bench.copies,
         "us_per_call": round(us, 3), "us_per_call_sd": round(statistics.pstdev(reps), 3),
         "alg_bytes": int(bench.alg_bytes), "gbs": round(bench.alg_bytes / (us * 1e-6) / 1e9, 1),
         "roofline_us": round(roof_us, 3), "frac": round(roof_us / us, 4),
         "frac_8tbs": round(bench.alg_bytes / 8e12 / (us * 1e-6), 4)}
    if getattr(bench.plan, "flat_ranges", 0):
        r["flat_ranges"] = bench.plan.flat_ranges
    if tensor_bound:
        r["roofline_us_hbm"] = round(hbm_us, 3)
        r["roofline_us_tensor_sustained"] = round(tensor_us, 3)
    if us_part is not None:
        r["us_partial"] = round(us_part, 3)
        r["partial_gbs"] = round(bench.alg_bytes / (us_part * 1e-6) / 1e9, 1)
        r["partial_frac"] = round(hbm_us / us_part, 4)
    return r


def sweep_rows(args, P):
    """The five workloads and the context sweep at H = 16, timed the way the
    headline is (CUDA graphs of back-to-back calls over distinct inputs that
    together exceed 3x L2; CUDA events on the launching stream)."""
    rows = []
    pdl = bool(args.pdl)
    for T in (256, 8192, 32768, 65536, 131072):
        b = DenseBench(T, 16, copies_for(T * ROW_BYTES), args.splits, pdl, variant=args.variant)
        us, usp, reps = time_bench(b, reps=100 if T <= 8192 else 40)
        rows.append(sweep_row(f"dense_h16_t{T}", b, us, usp, reps, P))
        del b
    torch.cuda.empty_cache()
    b = SparseBench("sparse_k2048", copies_for(2048 * ROW_BYTES), args.splits, pdl, variant=args.variant)
    us, usp, reps = time_bench(b, reps=100)
    rows.append(sweep_row("sparse_k2048", b, us, usp, reps, P))
    del b
    b = SparseBench("sparse_b64", copies_for(64 * 2048 * ROW_BYTES), args.splits, pdl, variant=args.variant,
                    device_cache=True)
    us, usp, reps = time_bench(b, reps=30)
    rows.append(sweep_row("sparse_b64", b, us, usp, reps, P))
    del b
    torch.cuda.empty_cache()
    gb = GraphBench(128, 32768, 64, copies_for((32768 + 64) * ROW_BYTES), args.splits, pdl, variant=args.variant)
    us, _, reps = time_graph_bench(gb, reps=5)
    rows.append(sweep_row("graph_h128", gb, us, None, reps, P, per="decode step per layer (append, partial, "
                          "combine, advance; 64 steps in one graph)", tensor_bound=True))
    del gb
    torch.cuda.empty_cache()
    # the same steps with the append and the advance folded into the two kernels
    gb = GraphBench(128, 32768, 64, copies_for((32768 + 64) * ROW_BYTES), args.splits, pdl, variant=args.variant,
                    fused=True)
    us, _, reps = time_graph_bench(gb, reps=5)
    rows.append(sweep_row("graph_h128_fused_step", gb, us, None, reps, P, per="decode step per layer "
                          "(mla_decode_forward_step: two launches; 64 steps in one graph)", tensor_bound=True))
    del gb
    torch.cuda.empty_cache()
    return rows


def alternate(graphs, calls, reps, inner):
    """Time each graph `reps` times, the arms alternating; us per call, mean and sem per arm."""
    out = {k: [] for k in graphs}
    for g in graphs.values():
        time_graph(g, 3, 2)
    for _ in range(reps):
        for k, g in graphs.items():
            out[k].append(time_graph(g, inner, 1) / (inner * calls) * 1e6)
    res = {}
    for k, v in out.items():
        res[k] = {"us_per_call": round(statistics.mean(v), 3),
                  "sem": round(statistics.pstdev(v) / math.sqrt(len(v)), 4), "reps": len(v)}
    return res


def pdl_ab(args, P, reps=12):
    """Programmatic dependent launch on and off, same plan and inputs, arms
    alternating in one process: the timing half of the PDL leave-one-out."""
    rows = []
    b = DenseBench(8192, 16, copies_for(8192 * ROW_BYTES), args.splits, True, variant=args.variant)
    g_on = capture(b.call, b.copies)
    b.replan(False)
    g_off = capture(b.call, b.copies)
    r = alternate({"pdl_on": g_on, "pdl_off": g_off}, b.copies, reps, 20)
    rows.append({"workload": "dense_h16_t8192", "splits": b.plan.splits, **r,
                 "pdl_saves_us": round(r["pdl_off"]["us_per_call"] - r["pdl_on"]["us_per_call"], 3)})
    del b, g_on, g_off
    gb = GraphBench(128, 32768, 64, copies_for((32768 + 64) * ROW_BYTES), args.splits, True, variant=args.variant)
    g_on = capture(gb.loop, 1)
    gb.replan(False)
    g_off = capture(gb.loop, 1)
    r = alternate({"pdl_on": g_on, "pdl_off": g_off}, gb.calls, reps, 1)
    rows.append({"workload": "graph_h128", "per": "decode step per layer", "splits": gb.plan.splits, **r,
                 "pdl_saves_us": round(r["pdl_off"]["us_per_call"] - r["pdl_on"]["us_per_call"], 3)})
    del gb, g_on, g_off
    torch.cuda.empty_cache()
    return rows


# the combine kernel reserves this much shared memory per CTA when its grid
# fits the GPU (one CTA per SM), which its empty stand-in copies
COMBINE_SPREAD_SMEM = 120 * 1024


def floor_rows(args, P, reps=12):
    """What a dense T = 8192 call costs with no decode work in it, timed like
    the calls (graphs over the same distinct caches, arms alternating):
    two empty kernels with the partial and combine kernels' launch shapes
    (PDL on and off), one kernel that only reads a call's cache rows with
    bulk copies (over every SM and over the partial's grid), and that read
    followed by the real combine kernel."""
    import decode_attention_mla_gb300 as mla
    d = torch.device("cuda")
    b = DenseBench(8192, 16, copies_for(8192 * ROW_BYTES), args.splits, True, variant=args.variant)
    pl = b.plan
    part = (pl.grid_x, pl.block, pl.smem_bytes)
    cgrid = pl.combine_grid_x * pl.combine_grid_y
    comb = (cgrid, pl.combine_block, COMBINE_SPREAD_SMEM if cgrid <= pl.num_sms else 0)
    nbytes = 8192 * ROW_BYTES
    sms = pl.num_sms
    sink = torch.zeros(max(sms, pl.grid_x), dtype=torch.int32, device=d)
    status = torch.zeros(1, dtype=torch.int32, device=d)
    graphs = {
        "empty_pair": capture(lambda c: mla.floor_empty_pair(part, comb, pdl=True), b.copies),
        "empty_pair_no_pdl": capture(lambda c: mla.floor_empty_pair(part, comb, pdl=False), b.copies),
        "read_all_sms": capture(lambda c: mla.floor_read(b.kv[c], nbytes, sms, sink, status), b.copies),
        "read_partial_grid": capture(lambda c: mla.floor_read(b.kv[c], nbytes, pl.grid_x, sink, status),
                                     b.copies),
    }

    def read_then_combine(c):
        mla.floor_read(b.kv[c], nbytes, pl.grid_x, sink, status)
        mla.combine(pl, b.args[c], b.scratch)

    graphs["read_then_combine"] = capture(read_then_combine, b.copies)
    graphs["call"] = capture(b.call, b.copies)
    r = alternate(graphs, b.copies, reps, 20)
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError("floor read kernel reported a wait timeout")
    out = {"workload": "dense_h16_t8192", "read_bytes": nbytes, "partial_launch": list(part),
           "combine_launch": list(comb)}
    for k, v in r.items():
        out[k] = v
    for k in ("read_all_sms", "read_partial_grid"):
        out[k]["gbs"] = round(nbytes / (r[k]["us_per_call"] * 1e-6) / 1e9, 1)
    del b, graphs
    torch.cuda.empty_cache()
    out["stream_t131072"] = stream_floor(131072, args, reps)
    out["gather"] = [gather_floor(name, args, reps) for name in ("sparse_k2048", "sparse_b64")]
    return out


def stream_floor(T, args, reps):
    """A long dense call's cache rows read by the bulk-copy kernel over every
    SM, beside the partial kernel alone and the whole call, same caches."""
    import decode_attention_mla_gb300 as mla
    d = torch.device("cuda")
    b = DenseBench(T, 16, copies_for(T * ROW_BYTES), args.splits, True, variant=args.variant)
    nbytes = T * ROW_BYTES
    sink = torch.zeros(b.plan.num_sms, dtype=torch.int32, device=d)
    status = torch.zeros(1, dtype=torch.int32, device=d)
    graphs = {"read": capture(lambda c: mla.floor_read(b.kv[c], nbytes, b.plan.num_sms, sink, status), b.copies),
              "partial": capture(b.partial, b.copies), "call": capture(b.call, b.copies)}
    r = alternate(graphs, b.copies, reps, 5)
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError("floor read kernel reported a wait timeout")
    res = {"workload": f"dense_h16_t{T}", "read_bytes": nbytes, **r}
    res["read"]["gbs"] = round(nbytes / (r["read"]["us_per_call"] * 1e-6) / 1e9, 1)
    del b, graphs
    torch.cuda.empty_cache()
    return res


def gather_floor(name, args, reps):
    """The sparse workload's listed rows gathered by a kernel that computes
    nothing (one bulk copy per row, over the partial's grid), beside the
    sparse call itself, on the same caches and index lists."""
    import decode_attention_mla_gb300 as mla
    d = torch.device("cuda")
    if name == "sparse_b64":
        b = SparseBench(name, copies_for(64 * 2048 * ROW_BYTES), args.splits, True, variant=args.variant,
                        device_cache=True)
    else:
        b = SparseBench(name, copies_for(2048 * ROW_BYTES), args.splits, True, variant=args.variant)
    idx, ln, off = b.idx.to(torch.int64), b.len.to(torch.int64), b.off
    valid = (idx >= 0) & (idx < ln[:, None])
    rows = (off[:, None] + idx)[valid].contiguous()
    ctas = b.plan.grid_x
    sink = torch.zeros(ctas, dtype=torch.int32, device=d)
    status = torch.zeros(1, dtype=torch.int32, device=d)
    graphs = {"gather": capture(lambda c: mla.floor_gather(b.kv[c], rows, ctas, sink, status), b.copies),
              "call": capture(b.call, b.copies)}
    r = alternate(graphs, b.copies, reps, 5 if name == "sparse_b64" else 20)
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError("floor gather kernel reported a wait timeout")
    nbytes = int(rows.numel()) * ROW_BYTES
    res = {"workload": name, "rows": int(rows.numel()), "ctas": ctas, "gather_bytes": nbytes, **r}
    res["gather"]["gbs"] = round(nbytes / (r["gather"]["us_per_call"] * 1e-6) / 1e9, 1)
    del b, graphs, rows
    torch.cuda.empty_cache()
    return res


def write_details(args, P):
    rows = []

    def entry(name, bench, us, us_part, reps, extra=None):
        r = {"workload": name, "splits": bench.plan.splits, "copies": bench.copies, "us_per_call": us,
             "us_partial": us_part, "sd_us": statistics.pstdev(reps), "alg_bytes": bench.alg_bytes,
             "gbs": bench.alg_bytes / (us * 1e-6) / 1e9,
             "frac_hbm": bench.alg_bytes / (P["hbm_gbs"] * 1e9) / (us * 1e-6),
             "frac_8tbs": bench.alg_bytes / 8e12 / (us * 1e-6),
             "tflops": bench.flops / (us * 1e-6) / 1e12}
        r.update(extra or {})
        rows.append(r)
        log(json.dumps(r))

    for T in (256, 8192, 16384, 32768, 65536, 131072):
        b = DenseBench(T, 16, copies_for(T * ROW_BYTES), args.splits, bool(args.pdl), variant=args.variant)
        us, usp, reps = time_bench(b)
        entry(f"dense_h16_t{T}", b, us, usp, reps)
        del b
    # the same workloads over an E4M3 cache (576-byte rows, one scale)
    for T in (8192, 32768, 131072):
        b = DenseBench(T, 16, copies_for(T * ROW_BYTES // 2), args.splits, bool(args.pdl), fp8=True)
        us, usp, reps = time_bench(b)
        entry(f"dense_fp8_h16_t{T}", b, us, usp, reps)
        del b
    torch.cuda.empty_cache()
    for s in (1, 2, 4, 8, 16, 32, 64, 128):
        b = DenseBench(8192, 16, copies_for(8192 * ROW_BYTES), s, bool(args.pdl), variant=args.variant)
        us, usp, reps = time_bench(b)
        entry("dense_t8192_split_sweep", b, us, usp, reps)
        del b
    # a call touches only its gathered rows: enough distinct caches that those exceed 3x L2
    b = SparseBench("sparse_k2048", copies_for(2048 * ROW_BYTES), args.splits, bool(args.pdl), variant=args.variant)
    us, usp, reps = time_bench(b)
    entry("sparse_k2048", b, us, usp, reps)
    del b
    torch.cuda.empty_cache()
    b = SparseBench("sparse_b64", copies_for(64 * 2048 * ROW_BYTES), args.splits, bool(args.pdl),
                    variant=args.variant)
    us, usp, reps = time_bench(b, reps=50)
    entry("sparse_b64", b, us, usp, reps)
    del b
    torch.cuda.empty_cache()
    gb = GraphBench(128, 32768, 64, copies_for((32768 + 64) * ROW_BYTES), args.splits, bool(args.pdl),
                    variant=args.variant)
    us, _, reps = time_graph_bench(gb)
    tensor_us = gb.flops / (P["bf16_tflops_sustained"] * 1e12) * 1e6
    entry("graph_h128", gb, us, None, reps,
          {"per": "decode step per layer", "layers": gb.copies,
           "roofline_us_hbm": gb.alg_bytes / (P["hbm_gbs"] * 1e9) * 1e6, "roofline_us_tensor": tensor_us,
           "frac_roofline": max(gb.alg_bytes / (P["hbm_gbs"] * 1e9) * 1e6, tensor_us) / us})
    del gb
    torch.cuda.empty_cache()
    # the same steps with the append and the advance folded into the two kernels
    gb = GraphBench(128, 32768, 64, copies_for((32768 + 64) * ROW_BYTES), args.splits, bool(args.pdl),
                    variant=args.variant, fused=True)
    us, _, reps = time_graph_bench(gb)
    entry("graph_h128_fused_step", gb, us, None, reps,
          {"per": "decode step per layer", "layers": gb.copies, "launches_per_layer_step": 2,
           "frac_roofline": max(gb.alg_bytes / (P["hbm_gbs"] * 1e9) * 1e6, tensor_us) / us})
    del gb
    torch.cuda.empty_cache()
    # wv_b projection of the merged latent (H heads, v_dim = 128), one weight copy per call
    for H in (16, 128):
        pr = project_timing(H, 128)
        r = {"workload": f"project_h{H}_v128", "copies": pr["copies"], "us_per_call": pr["us"],
             "alg_bytes": pr["bytes"], "gbs": pr["bytes"] / (pr["us"] * 1e-6) / 1e9,
             "frac_hbm": pr["bytes"] / (P["hbm_gbs"] * 1e9) / (pr["us"] * 1e-6)}
        rows.append(r)
        log(json.dumps(r))
    with open(args.details, "w") as f:
        json.dump({"peaks": P, "rows": rows}, f, indent=1)


def ncu_case(args):
    """A few eager calls on distinct caches (together larger than L2), for ncu."""
    from decode_attention_mla_gb300 import build as mla_build
    mla_build.build()
    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
    if args.ncu_case.startswith("dense_fp8_"):
        # dense_fp8_t<T>: the E4M3 cache, H = 16
        T = int(args.ncu_case[len("dense_fp8_t"):])
        b = DenseBench(T, 16, copies_for(T * ROW_BYTES // 2), args.splits, bool(args.pdl), fp8=True)
    elif args.ncu_case.startswith("dense_"):
        # dense_t<T> (16 heads) or dense_h<H>_t<T>
        fields = dict((f[0], int(f[1:])) for f in args.ncu_case[len("dense_"):].split("_"))
        T, H = fields["t"], fields.get("h", 16)
        b = DenseBench(T, H, copies_for(T * ROW_BYTES), args.splits, bool(args.pdl), variant=args.variant)
    elif args.ncu_case.startswith("project_h"):
        # project_h<H>: the wv_b projection (v_dim 128) over distinct weight copies
        import decode_attention_mla_gb300 as mla
        H = int(args.ncu_case[len("project_h"):])
        d = torch.device("cuda")
        g = torch.Generator().manual_seed(5)
        w0 = (torch.randn(H, 128, 512, generator=g) / 512 ** 0.5).to(torch.bfloat16).to(d)
        ws = [w0] + [torch.roll(w0, shifts=c, dims=2) for c in range(1, copies_for(H * 128 * 512 * 2))]
        lat = torch.randn(1, H, 512, generator=g).to(d)
        y = torch.empty(1, H, 128, device=d)
        for c in range(args.calls):
            mla.project(lat, ws[c % len(ws)], y, pdl=True)
        torch.cuda.synchronize()
        log(f"ncu case {args.ncu_case}: {args.calls} calls over {len(ws)} weight copies")
        return
    elif args.ncu_case.startswith("step_"):
        # step_h<H>_t<T>: the fused decode step (append + partial + combine, no
        # advance, so every call attends the same rows) over distinct caches
        fields = dict((f[0], int(f[1:])) for f in args.ncu_case[len("step_"):].split("_"))
        T, H = fields["t"], fields.get("h", 16)
        b = DenseBench(T, H, copies_for(T * ROW_BYTES), args.splits, bool(args.pdl), variant=args.variant)
        rows = workloads.randn_bf16(1, 576, seed=9, stream=4).to(torch.device("cuda"))
        for c in range(args.calls):
            b.mla.forward_step_args(b.plan, b.args[c % b.copies], b.scratch, rows, advance=False)
        torch.cuda.synchronize()
        log(f"ncu case {args.ncu_case}: {args.calls} fused steps, splits {b.plan.splits}, variant {b.plan.variant}")
        return
    elif args.ncu_case.startswith("loop_"):
        # loop_h<H>_t<T>: one eager pass of the multi-step loop (two steps of
        # append, partial + combine per layer, advance) over distinct caches
        fields = dict((f[0], int(f[1:])) for f in args.ncu_case[len("loop_"):].split("_"))
        T, H = fields["t"], fields.get("h", 128)
        gb = GraphBench(H, T, 2, copies_for((T + 2) * ROW_BYTES), args.splits, bool(args.pdl), variant=args.variant)
        for _ in range(max(1, args.calls // (2 * gb.copies))):
            gb.loop()
        torch.cuda.synchronize()
        log(f"ncu case {args.ncu_case}: {gb.copies} layers x 2 steps, splits {gb.plan.splits}")
        return
    elif args.ncu_case.startswith("floor_t"):
        # floor_t<T>: the floor probes on a T-row dense call's caches (the read
        # kernel over every SM, then the empty pair with the plan's launch shapes)
        import decode_attention_mla_gb300 as mla
        T = int(args.ncu_case[len("floor_t"):])
        b = DenseBench(T, 16, copies_for(T * ROW_BYTES), args.splits, True, variant=args.variant)
        pl = b.plan
        cgrid = pl.combine_grid_x * pl.combine_grid_y
        comb = (cgrid, pl.combine_block, COMBINE_SPREAD_SMEM if cgrid <= pl.num_sms else 0)
        sink = torch.zeros(pl.num_sms, dtype=torch.int32, device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        for c in range(args.calls):
            mla.floor_read(b.kv[c % b.copies], T * ROW_BYTES, pl.num_sms, sink, status)
            mla.floor_empty_pair((pl.grid_x, pl.block, pl.smem_bytes), comb)
        torch.cuda.synchronize()
        if int(status.item()) != 0:
            raise RuntimeError("floor read kernel reported a wait timeout")
        log(f"ncu case {args.ncu_case}: {args.calls} reads of {T * ROW_BYTES} B over {pl.num_sms} CTAs + empty pairs")
        return
    elif args.ncu_case == "floor_gather_k2048":
        # the gather floor probe on config 3's index list (8 cache copies)
        import decode_attention_mla_gb300 as mla
        b = SparseBench("sparse_k2048", 8, args.splits, True, variant=args.variant)
        idx, ln = b.idx.to(torch.int64), b.len.to(torch.int64)
        rows = (b.off[:, None] + idx)[(idx >= 0) & (idx < ln[:, None])].contiguous()
        sink = torch.zeros(b.plan.grid_x, dtype=torch.int32, device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        for c in range(args.calls):
            mla.floor_gather(b.kv[c % b.copies], rows, b.plan.grid_x, sink, status)
        torch.cuda.synchronize()
        if int(status.item()) != 0:
            raise RuntimeError("floor gather kernel reported a wait timeout")
        log(f"ncu case {args.ncu_case}: {args.calls} gathers of {rows.numel()} rows over {b.plan.grid_x} CTAs")
        return
    elif args.ncu_case == "sparse_k2048":
        b = SparseBench("sparse_k2048", min(32, copies_for(2048 * ROW_BYTES)), args.splits, bool(args.pdl),
                        variant=args.variant)
    else:
        b = SparseBench("sparse_b64", 1, args.splits, bool(args.pdl), variant=args.variant)
    for c in range(args.calls):
        b.call(c % b.copies)
    torch.cuda.synchronize()
    log(f"ncu case {args.ncu_case}: {args.calls} calls, splits {b.plan.splits}, copies {b.copies}")


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=0, help="timed steps (0 = about 2 s of work)")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--splits", type=int, default=int(os.environ.get("MLA_DECODE_SPLITS", "0")))
    ap.add_argument("--pdl", type=int, default=int(os.environ.get("MLA_DECODE_PDL", "1")))
    ap.add_argument("--variant", type=int, default=int(os.environ.get("MLA_DECODE_VARIANT", "0")),
                    help="0 = the planner's choice (warp-MMA for this shape), 1 = warp-MMA kernel, "
                         "2 / 3 / 4 = tcgen05 kernel with 16 / 32 / 64 heads per CTA, 5 = warp-MMA scores "
                         "with P . V on tcgen05")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sweep", action="store_true", help="skip the per-workload sweep, the PDL A/B and the floor")
    ap.add_argument("--details", default=None)
    ap.add_argument("--ncu-case", default=None,
                    help="profiling helper: dense_t<T> | dense_h<H>_t<T> | dense_fp8_t<T> | sparse_k2048 | sparse_b64 | "
                         "project_h<H> | step_h<H>_t<T> | loop_h<H>_t<T> | floor_t<T> | floor_gather_k2048: run --calls eager calls of "
                         "that workload and exit (no JSON)")
    ap.add_argument("--calls", type=int, default=20)
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    if args.ncu_case:
        ncu_case(args)
        return

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
    res = run_ours(args, rank, world)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
