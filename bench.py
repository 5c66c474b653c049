#!/usr/bin/env python
"""Benchmark of the GB300 Q4_0 dequant-matmul path.

Default workload (``--workload decode_sweep_7b``): one decode token through a
7B-like model's Q4_0 weights, M = 1, fp32 activations: 32 layers x
{4 x (K=4096, N=4096), 2 x (4096, 11008), 1 x (11008, 4096)} GEMVs, 224 in all,
3,642,753,024 bytes of weights, each GEMV with its own fresh input.  One step =
one pass of the 224 GEMVs, run as one persistent launch (q4_gemv_seq_run)
captured in a CUDA graph.  Metric: weight bytes streamed per second.  The
line also carries the same sweep with a decoder layer's ordering and as a
graph of 224 separate launches (``sweep_variants``), every other configuration
of the benchmark as a short nested run (``records``: one 4096 x 4096 GEMV, the
batched 5120 x 12288 decode at M = 1, 4, 8, 64, the routed experts at T = 1
and 32, the M = 2048 prefill GEMM), and two CPU baselines: the oracle
(``cpu_baseline``) and the pages' fused fp32 loop with OpenMP on every
physical core (``cpu_baseline_openmp``).

Other workloads (``--workload``), each printing its own line: ``gemv`` (one
GEMV, fp32 A, default K = N = 4096, --m/--k/--n), ``batched`` (K = 5120,
N = 12288, bf16 A with --m rows), ``moe`` (top-6 of 160 experts, H = 5120,
I = 1536, --tokens), ``moe_block`` (router + shared expert + routed experts
of the same block, --tokens), ``quantize`` (the Q4_0 encoder on a fp32
--k x --n matrix; GB/s of input plus output), ``host_stream`` (the decode
sweep with its weights in pinned host memory, copied into --slots device slots
while earlier GEMVs run; roofline: the host-to-device copy rate measured in
the same run), ``prefill`` (M = 2048, K = 5120, N = 12288, bf16 A and C on the
tensor cores; metric TFLOP/s).  Weight copies or routings rotate so
that each pass reads at least four times the L2 capacity.

``--impl reference`` times the fp64 CPU oracle on the host cores on a bounded
sample of the same workload and prints the same JSON line with
``"impl": "reference"``.

Prints exactly one JSON line (rank 0).  Under torchrun (N > 1) every rank runs
an independent replica on its own GPU (the path has no exchange step); the
reported value is the work of all ranks divided by the slowest rank's time.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import seeded_inputs as si  # noqa: E402

METRIC = "Q4_0 dequant-matmul weight GB/s (% HBM peak) at M=1; TFLOP/s at M=2048"


# Nominal figures beside the measured ones: HBM3e 8.0 TB/s (the workload's
# stated target denominator) and the sustained bf16 rate.
NOMINAL_HBM_GBS = 8000.0


def sustained_bf16_tflops():
    """MEASURED_PEAKS.json's seconds-long bf16 rate under the power cap, or None."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        return json.load(f).get("bf16_tflops_sustained")


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d.get("hbm_gbs", 6800.0), d.get("bf16_tflops", 1900.0), "measured"
    return 6800.0, 1900.0, "fallback"


# dram__bytes_read.sum + dram__bytes_write.sum per launch of the dominant kernel,
# from an ncu capture, keyed by the hash of the kernel sources it was taken on.
# A changed source hash makes the figure stale and the bench reports null.
TRAFFIC = {
    # mean per launch over the sweep's 4:2:1 shape mix
    "d74610c072511ba9": 16312210,
}


# The same for the persistent decode-sequence kernel (q4_gemv_seq_kernel), per
# launch of the whole 32-layer sweep, keyed by the hash of the kernel's own
# sources and the plan's buffer size (which counts its units of work: the
# partial sums they write and read back are the traffic beyond the weights).
SEQ_SOURCES = ("q4_gemv_seq.cu", "q4_gemv_core.cuh", "q4_device.cuh")
TRAFFIC_SEQ = {
    # captured on the 32-layer launch itself (one pass per launch)
    "7d1a784ef69b6a66/7454208": 3783943680,
}


# The same for the prefill GEMM kernel (q4_gemm_tc_kernel), one launch of
# M = 2048, K = 5120, N = 12288.
TRAFFIC_GEMM = {
    # the last round's K steps shared over the grid (fp32 partial tiles)
    "caa0687ce8c057d2": 99115776,
}


def kernel_source_hash(names=("q4_gemv.cu", "q4_device.cuh", "q4_kernels.h")) -> str:
    h = hashlib.sha256()
    for name in names:
        with open(os.path.join(ROOT, "quantized_weight_q4_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.gpu), "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            time.sleep(0.3)
        except (OSError, ValueError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# distributed plumbing (replicas only)
# ---------------------------------------------------------------------------
def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(ws, x: float) -> float:
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# workloads
# ---------------------------------------------------------------------------
def sweep_plan(layers, block_bytes=18):
    shapes = si.sweep_shapes(layers)
    wbytes = sum(K * si.nblocks(N) * block_bytes for K, N in shapes)
    return shapes, wbytes


def device_weights(torch, q4, dev, K, N, fmt, seed, stream):
    """(weights on the device, their Q4_LAYOUT_* code) for a seeded K x N
    matrix: Q4_0 or Q8_0 blocks, or Q4_0 blocks repacked once, on the GPU and
    before any timing, into the planar layout."""
    gen = si.q8_weights if fmt == "q8_0" else si.q4_weights
    B = torch.from_numpy(gen(K, N, seed=seed, stream=stream)).to(dev)
    if fmt == "q8_0":
        return B, q4.Q4_LAYOUT_Q8_0
    if fmt == "q4_0_planar":
        P = torch.empty(q4.q4_planar_bytes(K, N), dtype=torch.uint8, device=dev)
        q4.q4_repack(P, B, K, N)
        return P, q4.Q4_LAYOUT_PLANAR
    return B, q4.Q4_LAYOUT_BLOCKS


def build_sweep(torch, dev, layers, seed=0, fmt="q4_0"):
    """Device weights, one contiguous A buffer and one contiguous C buffer."""
    import quantized_weight_q4_gb300 as q4
    from quantized_weight_q4_gb300.graph import MatmulSequence
    q8 = fmt == "q8_0"
    shapes, wbytes = sweep_plan(layers, 34 if q8 else 18)
    a_off, c_off, oa, oc = [], [], 0, 0
    for K, N in shapes:
        a_off.append(oa)
        c_off.append(oc)
        oa += (K + 3) // 4 * 4
        oc += (N + 3) // 4 * 4
    dA = torch.empty(oa, dtype=torch.float32, device=dev)
    dC = torch.empty(oc, dtype=torch.float32, device=dev)
    hA = torch.empty(oa, dtype=torch.float32).pin_memory()
    hC = torch.empty(oc, dtype=torch.float32).pin_memory()
    calls = []
    weights = []
    layout = q4.Q4_LAYOUT_BLOCKS
    for i, (K, N) in enumerate(shapes):
        B, layout = device_weights(torch, q4, dev, K, N, fmt, seed, 100 + i)
        weights.append(B)
        hA[a_off[i]:a_off[i] + K] = torch.from_numpy(si.activations_f32(1, K, seed, 10000 + i)[0])
        calls.append((dC[c_off[i]:c_off[i] + N].view(1, N), dA[a_off[i]:a_off[i] + K].view(1, K),
                      B, 1, N, K))
    dA.copy_(hA)
    torch.cuda.synchronize()
    seq = MatmulSequence(calls, b_layout=layout)
    return dict(seq=seq, dA=dA, dC=dC, hA=hA, hC=hC, weights=weights, shapes=shapes,
                wbytes=wbytes, launches_per_step=len(shapes))


def sweep_deps(n, kind):
    """Dependency lists of the sweep's ops (7 per layer: q, k, v, o, gate, up,
    down).  'none': every op has its own fresh input; 'layer': a decoder
    layer's ordering (q, k, v after the previous down; o after q, k, v; gate
    and up after o; down after gate and up); 'chain': each op after the one
    before it."""
    out = []
    for i in range(n):
        if kind == "none":
            out.append([])
        elif kind == "chain":
            out.append([i - 1] if i else [])
        else:
            j, base = i % 7, i - i % 7
            if j < 3:
                out.append([base - 1] if base else [])
            elif j == 3:
                out.append([base, base + 1, base + 2])
            elif j < 6:
                out.append([base + 3])
            else:
                out.append([base + 4, base + 5])
    return out


DEPS_TEXT = {
    "none": "every GEMV has its own fresh input, no ordering",
    "layer": "a decoder layer's ordering: q, k, v after the previous layer's down; o after "
             "q, k, v; gate and up after o; down after gate and up",
    "chain": "every GEMV reads its input only after the previous GEMV has completed",
}


class SeqGraph:
    """A decode sequence plan (one persistent launch per step), its run
    captured once into a CUDA graph and replayed."""

    def __init__(self, torch, q4, calls, deps, slice_rows=0):
        ops = [(C.view(-1), A.view(-1), B, N, K, d) for (C, A, B, M, N, K), d in zip(calls, deps)]
        self.plan = q4.GemvSequence(ops, slice_rows=slice_rows)
        self.stream = torch.cuda.Stream()
        with torch.cuda.stream(self.stream):
            self.plan.run(stream=self.stream)
        self.stream.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph, stream=self.stream):
            self.plan.run(stream=self.stream)

    def capture(self):
        return self

    def replay(self):
        self.graph.replay()


def pipelined_e2e(torch, q4, w, seq, deps, slice_rows):
    """Steps of the decode sequence from pinned host A to pinned host C, two
    in flight: step i uses buffer set i % 2 (device A and C, its plan, host
    C); its A copy (copy-in stream) waits for step i - 2's kernel, its kernel
    (compute stream) for its A copy, its C copy (copy-out stream) for its
    kernel; before issuing step i the host waits for step i - 2's C copy.
    Returns run(n), which runs n steps and returns once the last result is
    on the host."""
    dA, dC = w["dA"], w["dC"]
    dA2, dC2 = torch.empty_like(dA), torch.empty_like(dC)
    hC2 = torch.empty_like(w["hC"]).pin_memory()

    def remap(t, base, other):   # the same view of the other buffer
        off = (t.data_ptr() - base.data_ptr()) // t.element_size()
        return other[off:off + t.numel()].view(t.shape)

    ops2 = [(remap(C, dC, dC2).view(-1), remap(A, dA, dA2).view(-1), B, N, K, d)
            for (C, A, B, M, N, K), d in zip(w["seq"].calls, deps)]
    plan2 = q4.GemvSequence(ops2, slice_rows=slice_rows)
    sets = [(dA, dC, w["hC"], seq.plan), (dA2, dC2, hC2, plan2)]
    s_in, s_k, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev = {(kind, b): torch.cuda.Event() for kind in ("in", "k", "out") for b in (0, 1)}

    def run(n):
        for i in range(n):
            b = i & 1
            a_dev, c_dev, c_host, plan = sets[b]
            if i >= 2:
                ev[("out", b)].synchronize()   # step i - 2's C is on the host
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(ev[("k", b)])
                a_dev.copy_(w["hA"], non_blocking=True)
                ev[("in", b)].record(s_in)
            with torch.cuda.stream(s_k):
                s_k.wait_event(ev[("in", b)])
                plan.run(stream=s_k)                    # q4_gemv_seq_run
                ev[("k", b)].record(s_k)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev[("k", b)])
                c_host.copy_(c_dev, non_blocking=True)
                ev[("out", b)].record(s_out)
        s_out.synchronize()
    return run


# Per-step times (ms) of the last timed region: an event after every replay,
# on the replaying stream, so that the median and the minimum step can be
# reported beside the aggregate.
_STEP_MS = []


def _timed_replays(torch, stream, replay, steps):
    """The timed region: `steps` replays between two events (the value).  A
    second, separate pass of up to 100 replays with an event after each
    gives the per-step median and minimum, so that the extra events do not
    touch the reported aggregate."""
    s = torch.cuda.Event(enable_timing=True)
    e = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        s.record()
        for _ in range(steps):
            replay()
        e.record()
    e.synchronize()
    total = s.elapsed_time(e) / 1e3
    n = min(steps, 100)
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(n + 1)]
    with torch.cuda.stream(stream):
        evs[0].record()
        for i in range(n):
            replay()
            evs[i + 1].record()
    evs[-1].synchronize()
    _STEP_MS[:] = [evs[i].elapsed_time(evs[i + 1]) for i in range(n)]
    return total


def step_summary():
    """Median and minimum step (ms) of the per-step pass after the last timed region."""
    if not _STEP_MS:
        return None
    v = sorted(_STEP_MS)
    n = len(v)
    med = v[n // 2] if n % 2 else 0.5 * (v[n // 2 - 1] + v[n // 2])
    return {"median_ms": round(med, 5), "min_ms": round(v[0], 5), "steps": n}


def time_graph(torch, seq, steps, warmup):
    seq.capture()
    for _ in range(warmup):
        seq.replay()
    torch.cuda.synchronize()
    return _timed_replays(torch, seq.stream, seq.graph.replay, steps)


def cpu_baseline_sweep(layers_sample, seed=0, fmt="q4_0"):
    """The oracle, single-threaded, on the first `layers_sample` layers."""
    import oracle
    shapes, _ = sweep_plan(layers_sample)
    total_bytes, total_t = 0, 0.0
    q8 = fmt == "q8_0"
    for i, (K, N) in enumerate(shapes):
        B = (si.q8_weights if q8 else si.q4_weights)(K, N, seed=seed, stream=100 + i)
        A = si.activations_f32(1, K, seed, 10000 + i)
        t = time.perf_counter()
        (oracle.q8_matmul if q8 else oracle.matmul)(A, B, 1, N, K, with_abs=False)
        total_t += time.perf_counter() - t
        total_bytes += B.nbytes
    return total_bytes, total_t


def cpu_openmp_sweep(layers_sample, budget_s=6.0, seed=0):
    """The engine page's fused fp32 loop with OpenMP over column blocks
    (cpu_baseline/), one thread per physical core, on the first
    `layers_sample` layers of the sweep, repeated for about `budget_s`."""
    import cpu_baseline
    cores = cpu_baseline.physical_cores()
    shapes, _ = sweep_plan(layers_sample)
    mats = [(si.activations_f32(1, K, seed, 10000 + i), si.q4_weights(K, N, seed=seed, stream=100 + i),
             N, K) for i, (K, N) in enumerate(shapes)]
    for A, B, N, K in mats[:2]:
        cpu_baseline.matmul(A, B, 1, N, K, cores)   # build and warm up
    nbytes, t, passes = 0, 0.0, 0
    while t < budget_s and passes < 50:
        for A, B, N, K in mats:
            t0 = time.perf_counter()
            cpu_baseline.matmul(A, B, 1, N, K, cores)
            t += time.perf_counter() - t0
            nbytes += B.nbytes
        passes += 1
    return {"value": round(nbytes / t / 1e9, 3), "unit": "GB/s", "cores": cores,
            "kind": "fused fp32 Q4_0 loop (engine page §3.2-§3.4), OpenMP schedule(static) "
                    "over column blocks, one thread per physical core",
            "sample": f"first {layers_sample} of 32 layers ({7 * layers_sample} GEMVs), "
                      f"{passes} passes, {nbytes} weight bytes in {t:.1f} s"}


def summarize(line):
    """The fields of a bench line that a nested record keeps."""
    keep = ("value", "unit", "ms_per_step", "step_ms", "steps", "warmup", "config", "roofline",
            "clocks", "gpu_launches", "launches_per_step")
    return {k: line[k] for k in keep if k in line}


def nested_records(args, ws, rank, local, torch, q4, dev, hbm_peak, peak_src):
    """Every configuration of the benchmark besides the decode sweep, each a
    short run of its own workload: one 4096 x 4096 GEMV, the batched
    5120 x 12288 decode at M = 1, 4, 8, 64, the routed experts at T = 1 and
    32, and the M = 2048 prefill GEMM."""
    base = dict(vars(args))
    recs = {}
    plan = [("gemv_4096x4096", dict(workload="gemv", m=1, k=4096, n=4096, steps=200)),
            ("batched_m1", dict(workload="batched", m=1, k=0, n=0, steps=100)),
            ("batched_m4", dict(workload="batched", m=4, k=0, n=0, steps=100)),
            ("batched_m8", dict(workload="batched", m=8, k=0, n=0, steps=100)),
            ("batched_m64", dict(workload="batched", m=64, k=0, n=0, steps=100)),
            ("moe_t1", dict(workload="moe", tokens=1, steps=50)),
            ("moe_t32", dict(workload="moe", tokens=32, steps=10)),
            ("prefill_m2048", dict(workload="prefill", m=2048, k=0, n=0, steps=20))]
    for name, kw in plan:
        a = argparse.Namespace(**{**base, "format": "q4_0", "warmup": 5, **kw})
        recs[name] = summarize(run_other(a, ws, rank, local, torch, q4, dev, hbm_peak, peak_src))
    return recs


def run_ours(args, ws, rank, local):
    import torch
    import __graft_entry__
    __graft_entry__.build()
    import quantized_weight_q4_gb300 as q4
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    hbm_peak, bf16_peak, peak_src = measured_peaks()

    if args.workload != "decode_sweep_7b":
        return run_other(args, ws, rank, local, torch, q4, dev, hbm_peak, peak_src)

    # CPU baseline first (rank 0 at N = 1 only), while the GPU is idle
    cpu = cpu_omp = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        nbytes, t = cpu_baseline_sweep(args.cpu_layers, fmt=args.format)
        cpu = {"value": nbytes / t / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
               "sample": f"first {args.cpu_layers} of 32 layers ({7 * args.cpu_layers} GEMVs, "
                         f"{nbytes} weight bytes), fp64 oracle, 1 thread, {t:.1f} s"}
        if args.format == "q4_0":
            try:
                cpu_omp = cpu_openmp_sweep(4)
            except (OSError, subprocess.CalledProcessError) as e:
                cpu_omp = {"unavailable": f"the OpenMP baseline did not build or load: {e}"}

    w = build_sweep(torch, dev, args.layers, fmt=args.format)
    use_seq = args.launch == "seq" and args.format == "q4_0"
    if use_seq:
        seq = SeqGraph(torch, q4, w["seq"].calls, sweep_deps(len(w["shapes"]), args.deps),
                       args.slice_rows)
        w["launches_per_step"] = 1
    else:
        seq = w["seq"]
    torch.cuda.synchronize()

    # device-resident timing (inputs already in HBM)
    barrier(ws)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        elapsed = time_graph(torch, seq, args.steps, args.warmup)
        steps_main = step_summary()
    torch.cuda.synchronize()
    barrier(ws)
    elapsed = max_over_ranks(ws, elapsed)
    status = q4.q4_get_device_status()
    if status != q4.Q4_OK:
        raise SystemExit(f"device status {status} after the timed region")

    # end to end: pinned host A -> device, the public call (through the C
    # ABI: host-side checks and launches on the clock, no graph), device C ->
    # pinned host.  The sequence form pipelines the steps as a serving loop
    # would: two sets of device A and C (two plans over the same weights) and
    # host C, so that one step's copies overlap the other step's kernel; the
    # host waits for step i - 2's result before it issues step i.
    e2e_steps = max(10, args.steps // 4)
    if use_seq:
        e2e_run = pipelined_e2e(torch, q4, w, seq, sweep_deps(len(w["shapes"]), args.deps),
                                args.slice_rows)
    else:
        stream = seq.stream
        def e2e_run(n):
            for _ in range(n):
                with torch.cuda.stream(stream):
                    w["dA"].copy_(w["hA"], non_blocking=True)
                    w["seq"].run_eager(stream=stream)       # one q4_matmul_ex per GEMV
                    w["hC"].copy_(w["dC"], non_blocking=True)
                stream.synchronize()
    e2e_run(max(3, args.warmup))
    barrier(ws)
    t0 = time.perf_counter()
    e2e_run(e2e_steps)
    e2e_t = time.perf_counter() - t0
    barrier(ws)
    e2e_t = max_over_ranks(ws, e2e_t)

    # the same sweep with other launch structures (same weights and inputs)
    variants = {}
    if use_seq and not args.no_records:
        vsteps = min(args.steps, 100)
        for name, make in (
                ("layer_ordered", lambda: SeqGraph(torch, q4, w["seq"].calls,
                                                   sweep_deps(len(w["shapes"]), "layer"),
                                                   args.slice_rows)),
                ("serial_launches", lambda: w["seq"])):
            g = make()
            with ClockSampler(local) as vclk:
                vt = time_graph(torch, g, vsteps, args.warmup)
            vt = max_over_ranks(ws, vt)
            variants[name] = {
                "value": round(ws * w["wbytes"] * vsteps / vt / 1e9, 2), "unit": "GB/s",
                "ms_per_step": round(vt / vsteps * 1e3, 5), "steps": vsteps, "warmup": args.warmup,
                "launch": ("one persistent launch per step, dependencies: " + DEPS_TEXT["layer"]
                           if name == "layer_ordered" else
                           "one CUDA graph of 224 GEMV launches (q4_matmul_ex, split-K GEMV) "
                           "with programmatic dependent launch"),
                "gpu_launches": vsteps * (1 if name == "layer_ordered" else len(w["shapes"])),
                "clocks": vclk.summary()}
        status = q4.q4_get_device_status()
        if status != q4.Q4_OK:
            raise SystemExit(f"device status {status} after the sweep variants")
    records = None
    if not args.no_records and args.format == "q4_0":
        records = nested_records(args, ws, rank, local, torch, q4, dev, hbm_peak, peak_src)

    wbytes = w["wbytes"]
    value = ws * wbytes * args.steps / elapsed / 1e9
    per_launch_bytes = wbytes / w["launches_per_step"]
    avg_launch_s = elapsed / (args.steps * w["launches_per_step"])
    achieved = per_launch_bytes / avg_launch_s / 1e9
    if use_seq:
        h = f"{kernel_source_hash(SEQ_SOURCES)}/{seq.plan.buf.numel()}"
        traffic = TRAFFIC_SEQ.get(h)
    else:
        h = kernel_source_hash()
        traffic = TRAFFIC.get(h) if args.format == "q4_0" else None
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(elapsed / args.steps * 1e3, 5),
        "step_ms": steps_main,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic (seeded: q ~ U{0..15}, d = fp16(U[0.001, 0.01]), A ~ N(0,1))",
        "config": {
            "workload": "decode_sweep_7b",
            "format": args.format,
            "layers": args.layers,
            "gemvs_per_step": w["launches_per_step"],
            "shapes_per_layer": "4x(K=4096,N=4096) 2x(4096,11008) 1x(11008,4096)",
            "M": 1, "a_dtype": "f32", "c_dtype": "f32",
            "weight_bytes_per_step": wbytes,
            "launch": (f"one persistent launch per step (q4_gemv_seq_run: counter clear + "
                       f"{seq.plan.grid} resident CTAs taking units of 512 columns x 512..4096 "
                       f"rows in op order), "
                       f"captured in a CUDA graph" if use_seq else
                       "one CUDA graph of 224 GEMV launches with programmatic dependent launch"),
            "deps": (args.deps + ": " + DEPS_TEXT[args.deps]) if use_seq else "serial launches",
            "slice_rows": (args.slice_rows or "library's choice") if use_seq else None,
            "l2": "no flush: each step streams 3.64 GB of weights, > 28x the 129 MB L2",
            "parallelism": f"replicas x{ws}",
            "pct_of_hbm_peak": round(100.0 * value / ws / hbm_peak, 2),
        },
        "roofline": {
            "bound": "hbm",
            "kernel": ("q4_gemv_seq_kernel (persistent: 36 KB TMA stages, 8 consumer warps, "
                       "2 CTAs per SM; all 224 GEMVs in one launch)" if use_seq else
                       "q4_gemv_kernel (GEMV, one row of A, 2 blocks per thread, 32-row stages"
                       + {"q8_0": ", Q8_0 blocks)", "q4_0_planar": ", planar Q4_0)"}.get(args.format, ")")),
            "kernel_source_hash": h,
            "achieved": round(achieved, 2),
            "peak": hbm_peak,
            "unit": "GB/s",
            "frac": round(achieved / hbm_peak, 4),
            "frac_of_nominal_8000": round(achieved / NOMINAL_HBM_GBS, 4),
            "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)" if peak_src == "measured" else "fallback",
            "algorithmic_bytes_per_launch": round(per_launch_bytes),
            "traffic": traffic,
        },
        "cpu_baseline": cpu,
        "e2e": {
            "value": round(ws * wbytes * e2e_steps / e2e_t / 1e9, 2),
            "unit": "GB/s",
            "h2d_bytes_per_step": int(w["hA"].numel() * 4),
            "d2h_bytes_per_step": int(w["hC"].numel() * 4),
            "steps": e2e_steps,
            "note": ("per step: pinned A -> device, the C-ABI call (q4_gemv_seq_run), "
                     "C -> pinned host; two steps in flight on two buffer sets (copies of "
                     "one overlap the other's kernel), the host waiting for step i-2's C "
                     "before issuing step i" if use_seq else
                     "per step: pinned A -> device, the C-ABI calls (224 x q4_matmul_ex), "
                     "C -> pinned host, stream sync"),
        },
        "gpu_launches": args.steps * w["launches_per_step"],
        "clocks": clk.summary(),
        "cpu_baseline_openmp": cpu_omp,
        "sweep_variants": variants or None,
        "records": records,
    }
    return line


# ---------------------------------------------------------------------------
# other workloads: one GEMV, batched decode, routed experts
# ---------------------------------------------------------------------------
class GraphOf:
    """A list of callables captured once into a CUDA graph."""

    def __init__(self, torch, fns):
        self.torch, self.fns = torch, fns
        self.stream = torch.cuda.Stream()
        with torch.cuda.stream(self.stream):
            for f in fns:
                f()
        self.stream.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph, stream=self.stream):
            for f in fns:
                f()

    def time(self, steps, warmup):
        torch = self.torch
        with torch.cuda.stream(self.stream):
            for _ in range(warmup):
                self.graph.replay()
        torch.cuda.synchronize()
        return _timed_replays(torch, self.stream, self.graph.replay, steps)


_MOE = {}


def moe_device_weights(to_dev, E, H, I):
    """The seeded expert stacks on the device, generated once per process."""
    key = (E, H, I)
    if key not in _MOE:
        _MOE[key] = tuple(to_dev(a) for a in si.moe_weights(E, H, I, seed=0))
    return _MOE[key]


# kernels one call of a workload launches (routed experts: gate/up, down and the
# slot combine; MoE block: router, shared expert, routed experts)
KERNELS_PER_CALL = {"gemv": 1, "batched": 1, "moe": 3, "quantize": 1, "prefill": 1,
                    "moe_block": 6}


def run_other(args, ws, rank, local, torch, q4, dev, hbm_peak, peak_src):
    l2 = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 128 << 20)
    to_dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    if args.workload in ("gemv", "batched"):
        M = args.m if args.workload == "gemv" else args.m
        K = args.k if args.k else (4096 if args.workload == "gemv" else 5120)
        N = args.n if args.n else (4096 if args.workload == "gemv" else 12288)
        q8 = args.format == "q8_0"
        wbytes = K * si.nblocks(N) * (34 if q8 else 18)
        copies = max(1, -(-4 * l2 // wbytes))   # >= 4x L2 of distinct weights per pass
        bf16 = args.workload == "batched"
        fns, keep = [], []
        # one zeroed workspace for the calls' K-slice partials (the calls run
        # one after another on one stream), so that the captured calls take
        # the same kernels as eager ones
        wsb = q4.q4_matmul_workspace_size(M, N, K) if bf16 else 0
        wspace = torch.zeros(max(wsb, 16), dtype=torch.uint8, device=dev) if wsb else None
        for i in range(copies):
            B, layout = device_weights(torch, q4, dev, K, N, args.format, 0, 500 + i)
            A = si.activations_bf16(M, K, 0, 600 + i) if bf16 else si.activations_f32(M, K, 0, 600 + i)
            A = to_dev(A.view(np.int16)).view(torch.bfloat16) if bf16 else to_dev(A)
            C = torch.empty((M, N), dtype=torch.float32, device=dev)
            keep += [A, B, C]
            fns.append(lambda C=C, A=A, B=B: q4.q4_matmul_ex(C, A, B, M, N, K, workspace=wspace,
                                                             b_layout=layout))
        g = GraphOf(torch, fns)
        barrier(ws)
        with ClockSampler(local) as clk:
            t = g.time(args.steps, args.warmup)
        barrier(ws)
        t = max_over_ranks(ws, t)
        per_launch = t / (args.steps * copies)
        value = ws * wbytes / per_launch / 1e9
        flops = 2.0 * M * K * N
        cfg = {"workload": args.workload, "format": args.format, "M": M, "K": K, "N": N,
               "a_dtype": "bf16" if bf16 else "f32", "c_dtype": "f32",
               "weight_bytes_per_launch": wbytes, "weight_copies_rotated": copies,
               "l2": f"{copies} distinct weight copies per pass ({copies * wbytes} B >= 4x L2)",
               "parallelism": f"replicas x{ws}", "tflops": round(flops / per_launch / 1e12, 3)}
        units = copies
    elif args.workload == "moe":
        T, E, H, I, topk = args.tokens, 160, 5120, 1536, 6
        dWg, dWu, dWd = moe_device_weights(to_dev, E, H, I)
        R = args.routings
        fns, keep, uniq = [], [], 0
        per_expert = (2 * H * si.nblocks(I) + I * si.nblocks(H)) * 18
        wsz = q4.q4_moe_workspace_size(T, topk, E, H, I)
        wspace = torch.zeros(wsz, dtype=torch.uint8, device=dev)
        for r in range(R):
            idx, w = si.routing(T, E, topk, seed=r)
            x = si.activations_bf16(T, H, seed=r)
            uniq += len(set(idx.reshape(-1).tolist())) * per_expert
            dx = to_dev(x.view(np.int16)).view(torch.bfloat16)
            di, dw = to_dev(idx), to_dev(w)
            out = torch.empty((T, H), dtype=torch.float32, device=dev)
            keep += [dx, di, dw, out]
            fns.append(lambda out=out, dx=dx, di=di, dw=dw: q4.q4_moe_experts_ex(
                out, dx, dWg, dWu, dWd, di, dw, T, topk, E, H, I, workspace=wspace))
        g = GraphOf(torch, fns)
        barrier(ws)
        with ClockSampler(local) as clk:
            t = g.time(args.steps, args.warmup)
        barrier(ws)
        t = max_over_ranks(ws, t)
        per_call = t / (args.steps * R)
        wbytes = uniq / R
        value = ws * wbytes / per_call / 1e9
        cfg = {"workload": "moe", "T": T, "E": E, "H": H, "I": I, "topk": topk,
               "routings_rotated": R, "unique_expert_bytes_per_call": round(wbytes),
               "l2": f"{R} seeded routings rotate over 160 experts (2.12 GB of weights)",
               "parallelism": f"replicas x{ws}"}
        units = R
    elif args.workload == "quantize":
        # the Q4_0 encoder on a fp32 matrix (HBM-bound: read W, write blocks)
        K = args.k if args.k else 5120
        N = args.n if args.n else 12288
        nbytes = K * N * 4 + K * si.nblocks(N) * 18
        copies = max(1, -(-4 * l2 // nbytes))
        fns, keep = [], []
        for i in range(copies):
            W = to_dev((si.rng(0, 900 + i).standard_normal((K, N)) * 0.02).astype(np.float32))
            B = torch.empty((K, si.nblocks(N) * 18), dtype=torch.uint8, device=dev)
            keep += [W, B]
            fns.append(lambda B=B, W=W: q4.q4_quantize(B, W, K, N))
        g = GraphOf(torch, fns)
        barrier(ws)
        with ClockSampler(local) as clk:
            t = g.time(args.steps, args.warmup)
        barrier(ws)
        t = max_over_ranks(ws, t)
        per_launch = t / (args.steps * copies)
        wbytes = nbytes
        value = ws * nbytes / per_launch / 1e9
        cfg = {"workload": "quantize", "K": K, "N": N, "w_dtype": "f32",
               "bytes_per_launch": nbytes, "copies_rotated": copies,
               "l2": f"{copies} distinct inputs per pass ({copies * nbytes} B >= 4x L2)",
               "parallelism": f"replicas x{ws}", "us_per_launch": round(per_launch * 1e6, 2)}
        units = copies
    elif args.workload == "moe_block":
        # router + shared expert + routed experts of one DeepSeek-V2-sized block
        T, E, H, I, topk, Is = args.tokens, 160, 5120, 1536, 6, 3072
        Wg, Wu, Wd = si.moe_weights(E, H, I, seed=0)
        dWg, dWu, dWd = to_dev(Wg), to_dev(Wu), to_dev(Wd)
        del Wg, Wu, Wd
        Sg, Su, Sd = (to_dev(a[0]) for a in si.moe_weights(1, H, Is, seed=100))
        R = args.routings
        fns, keep, uniq = [], [], 0
        per_expert = (2 * H * si.nblocks(I) + I * si.nblocks(H)) * 18
        shared_bytes = (2 * H * si.nblocks(Is) + Is * si.nblocks(H)) * 18
        wsz = q4.q4_moe_block_workspace_size(T, topk, E, H, I, Is)
        wspace = torch.zeros(wsz, dtype=torch.uint8, device=dev)
        for r in range(R):
            logits = si.router_logits(T, E, seed=r)
            order = np.argsort(-logits, axis=1, kind="stable")[:, :topk]
            uniq += len(set(order.reshape(-1).tolist())) * per_expert + shared_bytes
            dx = to_dev(si.activations_bf16(T, H, seed=r).view(np.int16)).view(torch.bfloat16)
            dl = to_dev(logits)
            out = torch.empty((T, H), dtype=torch.float32, device=dev)
            keep += [dx, dl, out]
            fns.append(lambda out=out, dx=dx, dl=dl: q4.q4_moe_block(
                out, dx, dl, dWg, dWu, dWd, T, topk, E, H, I, Sg, Su, Sd, Is, workspace=wspace))
        g = GraphOf(torch, fns)
        barrier(ws)
        with ClockSampler(local) as clk:
            t = g.time(args.steps, args.warmup)
        barrier(ws)
        t = max_over_ranks(ws, t)
        per_call = t / (args.steps * R)
        wbytes = uniq / R
        value = ws * wbytes / per_call / 1e9
        cfg = {"workload": "moe_block", "T": T, "E": E, "H": H, "I": I, "topk": topk,
               "shared_I": Is, "routings_rotated": R,
               "weight_bytes_per_call": round(wbytes),
               "note": "router on the GPU, shared expert (two of I=1536 run as one of 3072), "
                       "routed experts; the chosen experts' bytes plus the shared expert's",
               "l2": f"{R} seeded router-logit sets rotate over 160 experts",
               "parallelism": f"replicas x{ws}", "us_per_call": round(per_call * 1e6, 2)}
        units = R
    elif args.workload == "host_stream":
        return run_host_stream(args, ws, local, torch, q4, dev)
    elif args.workload == "prefill":
        M = args.m if args.m > 64 else 2048
        K = args.k if args.k else 5120
        N = args.n if args.n else 12288
        wbytes = K * si.nblocks(N) * 18
        per_copy = wbytes + M * K * 2 + M * N * 2
        copies = max(1, -(-4 * l2 // per_copy))   # >= 4x L2 of distinct A, B and C per pass
        fns, keep = [], []
        # the workspace carries the last round's shared-K partial tiles (one
        # workspace serves the calls in turn: each leaves its tickets zero)
        wsz = q4.q4_matmul_workspace_size(M, N, K)
        wspace = torch.zeros(max(wsz, 1), dtype=torch.uint8, device=dev)
        for i in range(copies):
            B = to_dev(si.q4_weights(K, N, seed=0, stream=700 + i))
            A = to_dev(si.activations_bf16(M, K, 0, 800 + i).view(np.int16)).view(torch.bfloat16)
            C = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
            keep += [A, B, C]
            fns.append(lambda C=C, A=A, B=B: q4.q4_matmul_ex(C, A, B, M, N, K, workspace=wspace))
        g = GraphOf(torch, fns)
        barrier(ws)
        with ClockSampler(local) as clk:
            t = g.time(args.steps, args.warmup)
        barrier(ws)
        t = max_over_ranks(ws, t)
        per_launch = t / (args.steps * copies)
        flops = 2.0 * M * K * N
        value = ws * flops / per_launch / 1e12
        status = q4.q4_get_device_status()
        if status != q4.Q4_OK:
            raise SystemExit(f"device status {status} after the timed region")
        tf_peak = measured_peaks()[1]
        tf_sustained = sustained_bf16_tflops()
        ghash = kernel_source_hash(("q4_gemm_sm103.cu", "q4_tc_core.cuh", "q4_device.cuh", "q4_kernels.h"))
        return {
            "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(t / args.steps * 1e3, 5), "step_ms": step_summary(),
            "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic (seeded)",
            "config": {"workload": "prefill", "M": M, "K": K, "N": N, "a_dtype": "bf16",
                       "c_dtype": "bf16", "flops_per_launch": flops,
                       "weight_bytes_per_launch": wbytes, "copies_rotated": copies,
                       "l2": f"{copies} distinct (A, B, C) sets per pass ({copies * per_copy} B >= 4x L2)",
                       "parallelism": f"replicas x{ws}",
                       "weight_gbs": round(wbytes / per_launch / 1e9, 2)},
            "roofline": {"bound": "tensor", "achieved": round(value / ws, 2), "peak": tf_peak,
                         "unit": "TFLOP/s", "frac": round(value / ws / tf_peak, 4),
                         "frac_of_sustained": (round(value / ws / tf_sustained, 4)
                                               if tf_sustained else None),
                         "peak_source": peak_src + " (bf16 burst)",
                         "kernel": "q4_gemm_tc_kernel", "kernel_source_hash": ghash,
                         "traffic": TRAFFIC_GEMM.get(ghash)},
            "gpu_launches": args.steps * copies, "clocks": clk.summary(),
            "launches_per_step": copies,
        }
    else:
        raise SystemExit(f"unknown workload {args.workload}")
    status = q4.q4_get_device_status()
    if status != q4.Q4_OK:
        raise SystemExit(f"device status {status} after the timed region")
    return {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(t / args.steps * 1e3, 5), "step_ms": step_summary(),
        "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic (seeded)", "config": cfg,
        "roofline": {"bound": "hbm", "achieved": round(value / ws, 2), "peak": hbm_peak,
                     "unit": "GB/s", "frac": round(value / ws / hbm_peak, 4),
                     "frac_of_nominal_8000": round(value / ws / NOMINAL_HBM_GBS, 4),
                     "peak_source": peak_src, "traffic": None},
        "gpu_launches": args.steps * units * (8 if args.workload == "moe_block" and args.tokens > 1
                                              else KERNELS_PER_CALL.get(args.workload, 1)),
        "clocks": clk.summary(), "launches_per_step": units,
    }


def run_host_stream(args, ws, local, torch, q4, dev):
    """The decode sweep with its weights in pinned host memory: each GEMV's
    blocks cross the host link into a ring of device slots while earlier GEMVs
    run (q4_matmul_host_stream), the whole sequence captured in a CUDA graph.
    The roofline is the host-to-device copy rate measured in the same run."""
    shapes, wbytes = sweep_plan(args.layers)
    ops, keep = [], []
    for i, (K, N) in enumerate(shapes):
        Bh = torch.from_numpy(si.q4_weights(K, N, seed=0, stream=100 + i)).pin_memory()
        A = torch.from_numpy(si.activations_f32(1, K, 0, 10000 + i)).to(dev)
        C = torch.empty((1, N), dtype=torch.float32, device=dev)
        ops.append((C, A, Bh, 1, N, K))
        keep += [A, C]
    slots = args.slots
    staging = torch.empty(q4.q4_host_stream_slot_bytes(ops) * slots, dtype=torch.uint8, device=dev)
    st, cp = torch.cuda.Stream(), torch.cuda.Stream()
    # the link alone: pinned host -> device copies of the same bytes, back to back
    big = max(K * si.nblocks(N) * 18 for K, N in shapes)
    src = torch.empty(big, dtype=torch.uint8).pin_memory()
    dst = torch.empty(big, dtype=torch.uint8, device=dev)
    n_copy = max(8, (1 << 30) // big)
    for _ in range(3):
        dst.copy_(src, non_blocking=True)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(cp):
        e0.record()
        for _ in range(n_copy):
            dst.copy_(src, non_blocking=True)
        e1.record()
    e1.synchronize()
    link_gbs = big * n_copy / (e0.elapsed_time(e1) / 1e3) / 1e9
    # the sequence, captured once and replayed
    q4.q4_matmul_host_stream(ops, staging, slots, stream=st, copy_stream=cp)
    st.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=st):
        q4.q4_matmul_host_stream(ops, staging, slots, stream=st, copy_stream=cp)
    for _ in range(args.warmup):
        g.replay()
    torch.cuda.synchronize()
    barrier(ws)
    with ClockSampler(local) as clk:
        with torch.cuda.stream(st):
            e0.record()
            for _ in range(args.steps):
                g.replay()
            e1.record()
        e1.synchronize()
    t = max_over_ranks(ws, e0.elapsed_time(e1) / 1e3)
    barrier(ws)
    status = q4.q4_get_device_status()
    if status != q4.Q4_OK:
        raise SystemExit(f"device status {status} after the timed region")
    value = ws * wbytes * args.steps / t / 1e9
    return {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(t / args.steps * 1e3, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic (seeded)",
        "config": {"workload": "host_stream", "layers": args.layers, "gemvs_per_step": len(shapes),
                   "weight_bytes_per_step": wbytes, "weights": "pinned host memory",
                   "slots": slots, "slot_bytes": q4.q4_host_stream_slot_bytes(ops),
                   "launch": "one CUDA graph: per GEMV a host-to-device copy on a copy stream "
                             "and the GEMV from its slot, ordered by events",
                   "l2": "no flush: each step copies 3.64 GB from the host",
                   "parallelism": f"replicas x{ws}"},
        "roofline": {"bound": "host link", "achieved": round(value / ws, 2),
                     "peak": round(link_gbs, 2), "unit": "GB/s",
                     "frac": round(value / ws / link_gbs, 4),
                     "peak_source": f"measured in this run: {n_copy} pinned host-to-device "
                                    f"copies of {big} B on one stream",
                     "traffic": None},
        "gpu_launches": args.steps * len(shapes), "clocks": clk.summary(),
        "launches_per_step": len(shapes),
    }


# ---------------------------------------------------------------------------
# reference arm: the oracle on the host cores
# ---------------------------------------------------------------------------
def run_reference(args, ws, rank):
    if rank != 0:
        return None
    import oracle
    oracle.build()
    # a bounded sample per step: the first `rows` rows of the sweep's first matrix
    K, N = si.SWEEP_LAYER[0]
    rows = args.ref_rows
    B = si.q4_weights(K, N, seed=0, stream=100)[:rows].copy()
    A = si.activations_f32(1, K, 0, 10000)[:, :rows].copy()
    for _ in range(args.warmup):
        oracle.matmul(A, B, 1, N, rows, with_abs=False)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.matmul(A, B, 1, N, rows, with_abs=False)
    t = time.perf_counter() - t0
    value = B.nbytes * args.steps / t / 1e9
    sample = (f"per step: rows 0..{rows - 1} of the sweep's first 4096x4096 Q4_0 matrix "
              f"({B.nbytes} weight bytes), fp64 oracle, 1 thread")
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 4),
        "unit": "GB/s",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(t / args.steps * 1e3, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded, same generator as the GPU arm)",
        "config": {"workload": "decode_sweep_7b", "sampled": True},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="decode_sweep_7b")
    ap.add_argument("--layers", type=int, default=32)
    ap.add_argument("--launch", choices=("seq", "graph"), default="seq",
                    help="decode sweep: one persistent launch per step (seq) or a graph of "
                         "one launch per GEMV (graph)")
    ap.add_argument("--deps", choices=("none", "layer", "chain"), default="none",
                    help="decode sweep with --launch seq: the ops' dependency structure")
    ap.add_argument("--slice-rows", type=int, default=0,
                    help="decode sweep with --launch seq: rows per unit of work (0: the "
                         "library's choice)")
    ap.add_argument("--cpu-layers", type=int, default=24)
    ap.add_argument("--ref-rows", type=int, default=512)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-records", action="store_true",
                    help="decode sweep: skip the nested records of the other configurations")
    ap.add_argument("--slots", type=int, default=4, help="host_stream: device weight slots")
    ap.add_argument("--format", choices=("q4_0", "q8_0", "q4_0_planar"), default="q4_0",
                    help="weight format (decode sweep, gemv, batched); q4_0_planar: the Q4_0 "
                         "blocks repacked once into the planar layout before timing")
    ap.add_argument("--m", type=int, default=1, help="rows of A (gemv, batched)")
    ap.add_argument("--k", type=int, default=0)
    ap.add_argument("--n", type=int, default=0)
    ap.add_argument("--tokens", type=int, default=1, help="tokens (moe)")
    ap.add_argument("--routings", type=int, default=32, help="seeded routings rotated (moe)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    ws, rank, local = dist_setup()
    if args.impl == "reference":
        line = run_reference(args, ws, rank)
    else:
        line = run_ours(args, ws, rank, local)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
