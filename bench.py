"""Benchmark of the trellis-quantized linear layer on GB300.

Headline workload: the decode-shaped gate_proj geometry (K=5120, N=17408,
bits=4), one step = four exl3_linear calls at M = 1, 4, 8, 16 (fp16 in,
fp16 out), weights resident in HBM. Metric: weight GB/s = trellis bytes read
per step / step time. Twelve rotating weight copies (535 MB, > 4x L2) keep
every call's weights out of L2. The timed loop replays CUDA graphs of one
step each. The end-to-end figure (`e2e`) times the same step through the
public API with host buffers: one H2D of the step's inputs from pinned
memory, the four calls, one D2H of the outputs, the whole step captured
once as a CUDA graph and replayed (the eager, Python-issued figure is
reported beside it).

Also measured in the same run (reported as sub-objects of the JSON line):
  prefill   - the prefill-shaped call on the same geometry at M=2048
              (TFLOP/s = 2*M*K*N / call time, reconstruct and Hadamards
              included), with the reconstruct / GEMM split;
  crossover - both paths timed at M in {64 .. 4096} on both MLP geometries;
  logits    - the odd-vocab masked logits call at M in {1, 16, 2048};
  mlp_stack - 64 dense MLP layers (gate, up, SiLU*up, down) at M=2048,
              bits 4 and 3: ms per pass and the reconstruct/GEMM split;
  decode_stack - the same 64-layer stack as one decode step at M = 1 and
              16 (bits 4), run eagerly and as one captured CUDA graph.

--impl reference times the CPU oracle (test infrastructure) on the host's
cores on a bounded sample of the same workload, as the reference arm.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
       [--quick] [--no-extras] [--extras a,b,...]
       python bench.py --profile-call K,N,BITS,M[,REPS]   (profiling aid, no JSON)
"""
from __future__ import annotations

import argparse
import datetime
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

import synthetic  # noqa: E402

METRIC = "EXL3 linear: decode weight GB/s, prefill TFLOP/s, both as % roofline"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
WEIGHT_COPIES = 12
L2_BYTES = 129 * 10**6


# ---------------------------------------------------------------------------
# plumbing
# ---------------------------------------------------------------------------

def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20000)
    p.add_argument("--warmup", type=int, default=200)
    p.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    p.add_argument("--quick", action="store_true", help="smaller extras (for profiling runs)")
    p.add_argument("--no-extras", action="store_true", help="headline workload only")
    p.add_argument("--profile-call", default=None, metavar="K,N,BITS,M[,REPS[,THRESHOLD]]",
                   help="profiling aid: run exl3_linear REPS (default 4) times on one seeded matrix of that shape "
                        "with that m_threshold (default 0: decode-shaped) and exit (no JSON line)")
    p.add_argument("--extras", default="prefill,prefill_fused,crossover,logits,mlp_stack,decode_stack",
                   help="comma-separated sub-measurements to run after the headline")
    return p.parse_args()


def dist_info():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def reduce_max(torch, value: float, device) -> float:
    """Max of `value` over all ranks (identity when not distributed)."""
    if not (torch.distributed.is_available() and torch.distributed.is_initialized()):
        return float(value)
    t = torch.tensor([float(value)], device=device, dtype=torch.float64)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: float, world: int, seconds_max: float) -> float:
    """Whole-job throughput of N independent replicas: the units all ranks
    processed divided by the slowest rank's time."""
    return units_per_rank * world / seconds_max


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": FALLBACK_BF16_TFLOPS,
                "bf16_tflops_sustained": 1700.0, "source": "fallback"}


class ClockSampler:
    """nvidia-smi samples every 200 ms; keeps those inside [t0, t1]."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            threading.Thread(target=self._read, daemon=True).start()
        except Exception:
            self.proc = None
        time.sleep(0.6)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def stop(self):
        time.sleep(0.25)
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=2)
        except Exception:
            self.proc.kill()
        inside, allv = [], []
        for ln in self.lines:
            parts = [s.strip() for s in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rec = (ts, float(parts[1]), float(parts[2]), parts[4:9])
            except ValueError:
                continue
            allv.append(rec)
            if self.t0 is not None and self.t0 - 0.25 <= ts <= (self.t1 or ts) + 0.25:
                inside.append(rec)
        use = inside if inside else allv[-3:]
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        names = ["active", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in use:
            for n, v in zip(names[1:], r[3][1:]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(r[1] for r in use), "sm_max_mhz": max(r[2] for r in use),
                "reasons": sorted(reasons), "samples": len(inside)}


DECODE_SOURCES = ("trellis_quantized_linear_gb300/csrc/exl3_decode_gemm.cu",
                  "trellis_quantized_linear_gb300/csrc/exl3_common.cuh",
                  "trellis_quantized_linear_gb300/csrc/exl3_bounds.cuh")


def source_hash(*rel):
    h = hashlib.sha256()
    for r in rel:
        with open(os.path.join(ROOT, r), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel_files, summary: str):
    """DRAM bytes per launch from a committed ncu summary, or None when the
    kernel's sources (its file and the device header it inlines) changed
    since the counters were taken."""
    path = os.path.join(ROOT, "profiles", summary)
    try:
        with open(path) as f:
            text = f.read()
    except OSError:
        return None
    want = source_hash(*kernel_files)
    rec_hash, traffic = None, None
    for line in text.splitlines():
        if line.startswith("source_sha256_16:"):
            rec_hash = line.split(":", 1)[1].strip()
        if line.startswith("dram_bytes_per_launch:"):
            traffic = float(line.split(":", 1)[1].strip())
    return traffic if rec_hash == want else None


# ---------------------------------------------------------------------------
# device helpers
# ---------------------------------------------------------------------------

def _dev(torch, a):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).cuda()


class DevMatrix:
    def __init__(self, torch, mat, n_gemm=None):
        self.K, self.n_stored, self.bits = mat.K, mat.n_stored, mat.bits
        self.n_gemm = mat.n_stored if n_gemm is None else n_gemm
        self.trellis = _dev(torch, mat.trellis)
        self.su = _dev(torch, mat.su)
        self.sv = _dev(torch, mat.sv)
        self.nbytes = mat.trellis.nbytes


def make_ws(torch, tql, M_max, K, n_gemm, bits, thr):
    n = tql.exl3_linear_workspace_bytes(M_max, K, n_gemm, bits, thr)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    tql.exl3_workspace_init(ws)
    return ws


def call_linear(tql, x, M, mat, y, thr, ws, y_dtype):
    tql.exl3_linear(x, M, mat.K, mat.trellis, mat.bits, mat.n_stored, mat.n_gemm, mat.su, mat.sv, y, y_dtype,
                    thr, ws)


def time_fn(torch, fn, iters, warmup=2):
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record()
    for _ in range(iters):
        fn()
    e.record()
    torch.cuda.synchronize()
    return s.elapsed_time(e) / iters


def graph_time(torch, fns, reps=5, warm=2):
    """ms per call of the closures in `fns`, captured once (in order) as one
    CUDA graph on a side stream and replayed `warm` + `reps` times; CUDA
    events on the replay stream bracket the timed replays."""
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for fn in fns:  # eager pass: nothing lazy happens inside the capture
            fn()
        stream.synchronize()
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=stream):
            for fn in fns:
                fn()
        for _ in range(warm):
            gr.replay()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        for _ in range(reps):
            gr.replay()
        e.record(stream)
    torch.cuda.synchronize()
    ms = s.elapsed_time(e) / (reps * len(fns))
    del gr
    return ms


def copies_for(nbytes: int) -> int:
    """Distinct weight copies whose calls in a row stream more than 4x the L2
    (129 MB on GB300), at least 2."""
    return max(2, min(WEIGHT_COPIES, -(-4 * L2_BYTES // nbytes)))


# ---------------------------------------------------------------------------
# CPU oracle baselines for the sub-lines (test infrastructure, host cores)
# ---------------------------------------------------------------------------

def oracle_call_time(K, N, bits, M, seed, x_scale=1.0, rows=None, cols=None, matrix_index=0):
    """Seconds the oracle takes for an M-row call of the K x N layer. With
    `rows` (< M) the oracle runs on that many seeded rows and, with `cols`
    (< N), on output columns [0, cols); the full-call time is then the
    sample's time scaled by (M/rows) * (N/cols): labelled extrapolated."""
    import oracle
    oracle.build()
    mat = synthetic.make_matrix(K, N, bits, seed=seed, matrix_index=matrix_index)
    r = M if rows is None else min(rows, M)
    c = N if cols is None else min(cols, N)
    x = synthetic.make_activations(r, K, seed=seed, x_scale=x_scale)
    t0 = time.perf_counter()
    oracle.linear(x, mat.trellis, bits, K, N, mat.su, mat.sv, 0, c)
    dt = time.perf_counter() - t0
    scale = (M / r) * (N / c)
    return {"s": dt * scale, "extrapolated": scale != 1.0, "sample": f"{r} rows x {c} columns, {dt:.2f} s",
            "cores": oracle.num_threads()}


def oracle_line(ms_gpu, cpu):
    """The CPU oracle's time beside a GPU time, and their ratio."""
    return {"oracle_ms": round(cpu["s"] * 1e3, 2), "extrapolated": cpu["extrapolated"], "sample": cpu["sample"],
            "cores": cpu["cores"], "kind": "oracle", "gpu_speedup": round(cpu["s"] * 1e3 / ms_gpu, 1)}


# ---------------------------------------------------------------------------
# headline: decode-shaped gate_proj
# ---------------------------------------------------------------------------

def bench_decode(args, torch, tql, peaks, dist):
    world, rank, local = dist
    g = synthetic.GATE_DECODE
    K, N, bits, Ms = g["K"], g["N"], g["bits"], g["Ms"]
    mats = [DevMatrix(torch, synthetic.make_matrix(K, N, bits, seed=g["seed"], matrix_index=j))
            for j in range(WEIGHT_COPIES)]
    xs = {M: _dev(torch, synthetic.make_activations(M, K, seed=g["seed"], x_scale=g["x_scale"])) for M in Ms}
    ys = {M: torch.empty((M, N), dtype=torch.float16, device="cuda") for M in Ms}
    thr = 128
    ws = make_ws(torch, tql, max(Ms), K, N, bits, 0)
    wbytes = mats[0].nbytes
    per_step_bytes = wbytes * len(Ms)

    stream = torch.cuda.Stream()
    graphs = []
    n_graphs = WEIGHT_COPIES // len(Ms)
    with torch.cuda.stream(stream):
        # eager warm-up of every shape before capture
        for i, M in enumerate(Ms):
            call_linear(tql, xs[M], M, mats[i], ys[M], thr, ws, tql.EXL3_F16)
        torch.cuda.synchronize()
        for gi in range(n_graphs):
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gr, stream=stream):
                for i, M in enumerate(Ms):
                    call_linear(tql, xs[M], M, mats[gi * len(Ms) + i], ys[M], thr, ws, tql.EXL3_F16)
            graphs.append(gr)
    torch.cuda.synchronize()

    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            graphs[i % n_graphs].replay()
    torch.cuda.synchronize()

    clocks = ClockSampler(local)
    clocks.start()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.mark_start()
    with torch.cuda.stream(stream):
        start.record(stream)
        for i in range(args.steps):
            graphs[i % n_graphs].replay()
        end.record(stream)
    torch.cuda.synchronize()
    clocks.mark_end()
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop()
    ms = reduce_max(torch, start.elapsed_time(end), "cuda")
    ms_per_step = ms / args.steps
    value = whole_job_rate(per_step_bytes, world, ms_per_step * 1e-3) / 1e9

    # per-M kernel durations (graph of 12 back-to-back launches of one shape)
    per_m = {}
    for M in Ms:
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(gr, stream=stream):
                for j in range(WEIGHT_COPIES):
                    call_linear(tql, xs[M], M, mats[j], ys[M], thr, ws, tql.EXL3_F16)
            t_ms = time_fn(torch, gr.replay, 50, 5) / WEIGHT_COPIES
        per_m[str(M)] = {"us_per_call": round(t_ms * 1e3, 3),
                         "weight_gbs": round(wbytes / (t_ms * 1e-3) / 1e9, 1)}
        if rank == 0 and not args.no_extras:
            per_m[str(M)]["cpu_baseline"] = oracle_line(t_ms, oracle_call_time(K, N, bits, M, g["seed"],
                                                                                x_scale=g["x_scale"]))
    launch_us = ms_per_step * 1e3 / len(Ms)  # the step is exactly len(Ms) decode-GEMM launches
    achieved = wbytes / (launch_us * 1e-6) / 1e9
    return {
        "value": value, "ms_per_step": ms_per_step, "clocks": clk, "per_m": per_m,
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": round(achieved / peaks["hbm_gbs"], 4),
                     "traffic": profiled_traffic(DECODE_SOURCES, "decode_gemm_gate_k5120_n17408_b4.md"),
                     "peak_kind": f"of {peaks['source']} (burst copy)", "kernel": "decode_gemm_kernel<4,*>",
                     "bytes_per_launch": wbytes},
        # each decode-shaped call launches three kernels: input rotation,
        # decode GEMM, slot reduction
        "gpu_launches": args.steps * len(Ms) * 3,
        "weights_per_step_bytes": per_step_bytes,
        "mats": mats, "xs": xs, "ws": ws,
    }


def bench_e2e(args, torch, tql, state):
    """Same metric through the public API with host buffers: per step, one
    H2D of every call's x from pinned memory, the exl3_linear calls, and the
    D2H of every call's y into pinned memory; the step ends with all results
    on the host, and steps do not overlap one another. In the graph each
    call's y is copied down on a side stream right after that call (so it
    overlaps the calls that follow; only the last call's copy is exposed);
    issued eagerly, one D2H of all y follows the calls (the extra stream
    switches would cost more host time than they hide). Timed two ways: the step captured once
    in CUDA graphs (copies and calls as graph nodes, replayed; how a serving
    loop would issue it, the headline) and issued eagerly from Python (bound
    by host launch overhead)."""
    g = synthetic.GATE_DECODE
    K, N, Ms = g["K"], g["N"], g["Ms"]
    mats, ws = state["mats"], state["ws"]
    # the step's inputs (and outputs) for all its calls in one pinned host
    # buffer each: one copy up and one copy down per step
    rows = sum(Ms)
    hx = torch.cat([torch.from_numpy(synthetic.make_activations(M, K, seed=g["seed"], x_scale=g["x_scale"]))
                    for M in Ms]).pin_memory()
    hy = torch.empty((rows, N), dtype=torch.float16).pin_memory()
    dx = torch.empty((rows, K), dtype=torch.float16, device="cuda")
    dy = torch.empty((rows, N), dtype=torch.float16, device="cuda")
    offs = [sum(Ms[:j]) for j in range(len(Ms))]
    h2d = hx.numel() * 2
    d2h = hy.numel() * 2
    steps = max(20, min(args.steps // 20, 2000))

    side = torch.cuda.Stream()

    def issue(i, overlap):
        main = torch.cuda.current_stream()
        dx.copy_(hx, non_blocking=True)
        for j, M in enumerate(Ms):
            o = offs[j]
            call_linear(tql, dx[o:o + M], M, mats[(i * len(Ms) + j) % len(mats)], dy[o:o + M], 128, ws,
                        tql.EXL3_F16)
            if overlap:  # this call's y is ready: copy it down while the next calls run
                side.wait_stream(main)
                with torch.cuda.stream(side):
                    hy[o:o + M].copy_(dy[o:o + M], non_blocking=True)
        if overlap:
            main.wait_stream(side)
        else:
            hy.copy_(dy, non_blocking=True)

    def step(i):
        issue(i, False)
        torch.cuda.current_stream().synchronize()

    def timed(fn):
        for i in range(10):
            fn(i)
        t0 = time.perf_counter()
        for i in range(steps):
            fn(i)
        return (time.perf_counter() - t0) / steps

    dt_eager = timed(step)
    # one graph per group of len(Ms) weight copies, so that consecutive steps
    # still stream different weights (the copies exceed L2 together)
    ngraphs = max(1, len(mats) // len(Ms))
    stream = torch.cuda.Stream()
    graphs = []
    with torch.cuda.stream(stream):
        for k in range(ngraphs):
            issue(k, True)
        stream.synchronize()
        for k in range(ngraphs):
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gr, stream=stream):
                issue(k, True)
            graphs.append(gr)
    torch.cuda.synchronize()

    def gstep(i):
        graphs[i % ngraphs].replay()
        torch.cuda.current_stream().synchronize()

    dt = timed(gstep)
    wb = state["weights_per_step_bytes"]
    return {"value": round(wb / dt / 1e9, 1), "unit": "GB/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(dt * 1e3, 4),
            "steps": steps, "mode": "cuda_graph (step captured once: copies + calls, each D2H overlapping the later calls, replayed)",
            "eager": {"value": round(wb / dt_eager / 1e9, 1), "ms_per_step": round(dt_eager * 1e3, 4)}}


# ---------------------------------------------------------------------------
# extras: prefill, crossover, logits
# ---------------------------------------------------------------------------

def bench_prefill(args, torch, tql, peaks):
    """Prefill-shaped gate_proj at M=2048. Every timing replays a CUDA graph
    of calls over distinct weight copies (more than 4x L2 in total), so each
    call reads its trellis from HBM; the input rotation is timed over as many
    distinct activation copies."""
    K, N, bits, M = 5120, 17408, 4, 2048
    nc = copies_for(K * N * bits // 8)
    mats = [DevMatrix(torch, synthetic.make_matrix(K, N, bits, seed=synthetic.PREFILL_SEED, matrix_index=j))
            for j in range(nc)]
    mat = mats[0]
    x = _dev(torch, synthetic.make_activations(M, K, seed=synthetic.PREFILL_SEED))
    y = torch.empty((M, N), dtype=torch.float16, device="cuda")
    ws = make_ws(torch, tql, M, K, N, bits, 128)
    reps = 2 if args.quick else 5
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    clocks.mark_start()
    t_call = graph_time(torch, [lambda m=m: call_linear(tql, x, M, m, y, 128, ws, tql.EXL3_F16) for m in mats], reps)
    clocks.mark_end()
    clk = clocks.stop()
    xs = [x] + [torch.randn((M, K), device="cuda").half() for _ in range(nc - 1)]
    xr = torch.empty((M, K), dtype=torch.float16, device="cuda")
    t_had = graph_time(torch, [lambda xx=xx: tql.exl3_hadamard128(xx, xr, mat.su) for xx in xs], reps)
    del xs
    wt = torch.empty((N, K), dtype=torch.float16, device="cuda")
    t_rec = graph_time(torch, [lambda m=m: tql.exl3_reconstruct(m.trellis, bits, K, N, 0, N, wt, tql.EXL3_LAYOUT_NK)
                               for m in mats], reps)
    flops = 2.0 * M * K * N
    tflops = flops / (t_call * 1e-3) / 1e12
    t_gemm = max(t_call - t_had - t_rec, 1e-6)
    peak = peaks["bf16_tflops"]  # fp16 and bf16 share the tensor-core rate
    # weight-side rotation variant on the same call: rotated reconstruct + plain GEMM
    wsr = torch.empty(tql.exl3_weight_rotated_workspace_bytes(K, N), dtype=torch.uint8, device="cuda")
    t_wr = graph_time(torch, [lambda m=m: tql.exl3_linear_weight_rotated(x, M, K, m.trellis, bits, N, N, m.su, m.sv,
                                                                         y, tql.EXL3_F16, wsr) for m in mats], reps)
    t_rr = graph_time(torch, [lambda m=m: tql.exl3_reconstruct_rotated(m.trellis, bits, K, N, 0, N, m.su, m.sv, wt,
                                                                       tql.EXL3_LAYOUT_NK) for m in mats], reps)
    weight_rotated = {"ms_per_call": round(t_wr, 4), "tflops": round(flops / (t_wr * 1e-3) / 1e12, 1),
                      "frac": round(flops / (t_wr * 1e-3) / 1e12 / peak, 4),
                      "reconstruct_rotated_ms": round(t_rr, 4),
                      "reconstruct_rotated_gbs": round((mat.nbytes + N * K * 2) / (t_rr * 1e-3) / 1e9, 1)}
    del wsr, mats
    cpu = oracle_call_time(K, N, bits, M, synthetic.PREFILL_SEED, rows=128)
    return {"geometry": "K=5120 N=17408 bits=4 M=2048", "ms_per_call": round(t_call, 4),
            "weight_rotated": weight_rotated,
            "tflops": round(tflops, 1), "peak_tflops": peak, "frac": round(tflops / peak, 4),
            "peak_kind": f"of {peaks['source']} (cuBLAS bf16 burst; fp16 same rate)",
            "frac_sustained": round(tflops / peaks["bf16_tflops_sustained"], 4), "clocks": clk,
            "split_ms": {"hadamard": round(t_had, 4), "reconstruct": round(t_rec, 4), "gemm": round(t_gemm, 4)},
            "gemm_tflops": round(flops / (t_gemm * 1e-3) / 1e12, 1),
            "reconstruct_gbs": round((mat.nbytes + N * K * 2) / (t_rec * 1e-3) / 1e9, 1),
            "timing": f"CUDA graph replays over {nc} weight copies ({nc * mat.nbytes / 1e6:.0f} MB > 4x L2)",
            "cpu_baseline": oracle_line(t_call, cpu)}


def bench_prefill_fused(args, torch, tql, peaks):
    """Prefill-shaped gate_proj at M=512, the largest M at which exl3_linear
    takes the fused prefill kernel (the trellis decoded into the MMA operand,
    no reconstructed weight). Graph replays over distinct weight copies (more
    than 4x L2 in total), whole call including the input rotation."""
    K, N, bits, M = 5120, 17408, 4, 512
    nc = copies_for(K * N * bits // 8)
    mats = [DevMatrix(torch, synthetic.make_matrix(K, N, bits, seed=synthetic.PREFILL_SEED, matrix_index=j))
            for j in range(nc)]
    x = _dev(torch, synthetic.make_activations(M, K, seed=synthetic.PREFILL_SEED))
    y = torch.empty((M, N), dtype=torch.float16, device="cuda")
    ws = make_ws(torch, tql, M, K, N, bits, 128)
    reps = 2 if args.quick else 5
    t_call = graph_time(torch, [lambda m=m: call_linear(tql, x, M, m, y, 128, ws, tql.EXL3_F16) for m in mats], reps)
    nbytes = mats[0].nbytes
    del mats
    flops = 2.0 * M * K * N
    tflops = flops / (t_call * 1e-3) / 1e12
    peak = peaks["bf16_tflops"]
    cpu = oracle_call_time(K, N, bits, M, synthetic.PREFILL_SEED, rows=128)
    return {"geometry": "K=5120 N=17408 bits=4 M=512", "path": "fused prefill (decode into the MMA operand)",
            "ms_per_call": round(t_call, 4), "tflops": round(tflops, 1), "peak_tflops": peak,
            "frac": round(tflops / peak, 4),
            "peak_kind": f"of {peaks['source']} (cuBLAS bf16 burst; fp16 same rate)",
            "timing": f"CUDA graph replays over {nc} weight copies ({nc * nbytes / 1e6:.0f} MB > 4x L2)",
            "cpu_baseline": oracle_line(t_call, cpu)}


def bench_crossover(args, torch, tql):
    """Both paths at every M on both MLP geometries. Each (M, path) time
    replays a CUDA graph of calls over distinct weight copies (> 4x L2 in
    total), so no call finds its trellis in L2. The CPU oracle runs in full
    for the configured M up to 1024 and on 128 seeded rows above."""
    out = {}
    Ms = (16, 32, 64, 128) if args.quick else tuple(sorted(set((16, 32, 48, 384, 512, 768) + synthetic.PREFILL_MS)))
    reps = 2 if args.quick else 3
    for gm in synthetic.PREFILL_GEOMS:
        K, N, bits = gm["K"], gm["N"], 4
        nc = copies_for(K * N * bits // 8)
        mats = [DevMatrix(torch, synthetic.make_matrix(K, N, bits, seed=synthetic.PREFILL_SEED, matrix_index=j))
                for j in range(nc)]
        ws = make_ws(torch, tql, max(Ms), K, N, bits, 1)
        rows = []
        mx = None
        for M in Ms:
            x = _dev(torch, synthetic.make_activations(M, K, seed=synthetic.PREFILL_SEED))
            y = torch.empty((M, N), dtype=torch.float16, device="cuda")
            td = graph_time(torch, [lambda m=m: call_linear(tql, x, M, m, y, 0, ws, tql.EXL3_F16) for m in mats], reps)
            tp = graph_time(torch, [lambda m=m: call_linear(tql, x, M, m, y, 1, ws, tql.EXL3_F16) for m in mats], reps)
            row = {"M": M, "decode_ms": round(td, 4), "prefill_ms": round(tp, 4)}
            if M in synthetic.PREFILL_MS and not args.quick:
                cpu = oracle_call_time(K, N, bits, M, synthetic.PREFILL_SEED, rows=None if M <= 1024 else 128)
                row["cpu_baseline"] = oracle_line(min(td, tp), cpu)
            rows.append(row)
            if mx is None and tp < td:
                mx = M
            del x, y
        out[gm["name"]] = {"rows": rows, "crossover_M": mx,
                           "timing": f"CUDA graph replays over {nc} weight copies "
                                     f"({nc * mats[0].nbytes / 1e6:.0f} MB > 4x L2)"}
        del ws, mats
        torch.cuda.empty_cache()
    return out


def bench_logits(args, torch, tql, peaks):
    """Odd-vocab masked logits (the weight alone, 953 MB, is > 4x L2).
    Times replay a CUDA graph of calls."""
    c = synthetic.LOGITS
    K, ns, ng, nd, bits = c["K"], c["n_stored"], c["n_gemm"], c["n_decodable"], c["bits"]
    mat = DevMatrix(torch, synthetic.make_matrix(K, ns, bits, seed=c["seed"]), n_gemm=ng)
    res = {}
    Ms = (1, 16) if args.quick else c["Ms"]
    ws = make_ws(torch, tql, max(Ms), K, ng, bits, 128)
    wbytes = K * ng * bits // 8
    for M in Ms:
        x = _dev(torch, synthetic.make_activations(M, K, seed=c["seed"]))
        lg = torch.empty((M, ng), dtype=torch.float32, device="cuda")
        am = torch.empty((M,), dtype=torch.int32, device="cuda")
        fn = lambda: tql.exl3_logits_masked(x, M, K, mat.trellis, bits, ns, ng, nd, mat.su, mat.sv, lg, am, 128, ws)
        t = graph_time(torch, [fn] * (2 if M >= 2048 else 4), 3 if M >= 2048 else 10)
        r = {"ms": round(t, 4), "path": "prefill" if M >= 128 else "decode"}
        if M >= 128:
            r["tflops"] = round(2.0 * M * K * ng / (t * 1e-3) / 1e12, 1)
        else:
            r["weight_gbs"] = round(wbytes / (t * 1e-3) / 1e9, 1)
            r["frac_hbm"] = round(r["weight_gbs"] / peaks["hbm_gbs"], 4)
        if not args.quick:
            # oracle on one reconstruct chunk's columns (and 128 rows at M=2048), scaled to the call
            cpu = oracle_call_time(K, ns, bits, M, c["seed"], rows=None if M <= 16 else 128, cols=32768)
            r["cpu_baseline"] = oracle_line(t, cpu)
        res[str(M)] = r
        del x, lg, am
    res["timing"] = "CUDA graph replays; the 953 MB weight alone exceeds 4x L2"
    return res


def bench_mlp_stack(args, torch, tql, peaks):
    """64 layers of gate/up (5120->17408), SiLU(gate)*up, down (17408->5120)
    at M=2048 on the prefill path, for bits 4 and 3. Weights are drawn on the
    device (timing only); the per-layer parity of this geometry is covered by
    the test suite with the host generator. Every layer reads the same input
    x0: chained through random weights with no normalisation, SiLU(gate)*up
    grows the activations quadratically and overflows fp16 within a few
    layers, and inf/NaN operands draw less power than real data. The call
    sequence and work per layer are those of a chained stack."""
    st = synthetic.MLP_STACK
    L, d, f, M = st["layers"], st["d_model"], st["d_ff"], st["M"]
    if args.quick:
        L = 8
    out = {}
    thr = 128
    for bits in st["bits"]:
        layers = []
        for l in range(L):
            mats = []
            for j, (K, N) in enumerate(((d, f), (d, f), (f, d))):
                tr, su, sv = synthetic.make_matrix_device(K, N, bits, seed=st["seed_base"] + l, matrix_index=j)
                mats.append(dict(K=K, N=N, tr=tr, su=su, sv=sv))
            layers.append(mats)
        ws = torch.empty(max(tql.exl3_linear_workspace_bytes(M, d, f, bits, thr),
                             tql.exl3_linear_workspace_bytes(M, f, d, bits, thr)), dtype=torch.uint8, device="cuda")
        tql.exl3_workspace_init(ws)
        x0 = _dev(torch, synthetic.make_activations(M, d, seed=st["seed_base"]))
        g = torch.empty((M, f), dtype=torch.float16, device="cuda")
        u = torch.empty_like(g)
        h = torch.empty_like(g)
        xa = torch.empty((M, d), dtype=torch.float16, device="cuda")

        def lin(xin, m, yout):
            tql.exl3_linear(xin, M, m["K"], m["tr"], bits, m["N"], m["N"], m["su"], m["sv"], yout, tql.EXL3_F16,
                            thr, ws)

        def one_pass(check=False):
            first_bad = None
            for l, (mg, mu, md) in enumerate(layers):
                lin(x0, mg, g)
                lin(x0, mu, u)
                tql.exl3_silu_mul(g, u, h)
                lin(h, md, xa)
                if check and first_bad is None and not bool(torch.isfinite(xa).all()):
                    first_bad = l
            return first_bad

        first_bad = one_pass(check=True)
        torch.cuda.synchronize()
        clocks = ClockSampler(torch.cuda.current_device())
        clocks.start()
        clocks.mark_start()
        ms = time_fn(torch, one_pass, 8, 1)
        clocks.mark_end()
        clk = clocks.stop()
        # split from component timings of each geometry
        split = {"hadamard": 0.0, "reconstruct": 0.0, "gemm": 0.0}
        for (K, N), times in (((d, f), 2), ((f, d), 1)):
            m = layers[0][0 if K == d else 2]
            xin = x0 if K == d else h
            yv = g if K == d else xa
            t_call = time_fn(torch, lambda: lin(xin, m, yv), 5, 2)
            xr = torch.empty((M, K), dtype=torch.float16, device="cuda")
            t_had = time_fn(torch, lambda: tql.exl3_hadamard128(xin, xr, m["su"]), 5, 2)
            wt = torch.empty((N, K), dtype=torch.float16, device="cuda")
            t_rec = time_fn(torch, lambda: tql.exl3_reconstruct(m["tr"], bits, K, N, 0, N, wt, tql.EXL3_LAYOUT_NK),
                            5, 2)
            split["hadamard"] += L * times * t_had
            split["reconstruct"] += L * times * t_rec
            split["gemm"] += L * times * (t_call - t_had - t_rec)
            del xr, wt
        flops = 2.0 * M * (2 * d * f + f * d) * L
        cpu_s, samples = 0.0, []
        if not args.quick:
            # oracle: layer 0's three projections on 128 seeded rows, scaled to M rows and L layers
            for j, (K, N) in enumerate(((d, f), (d, f), (f, d))):
                c1 = oracle_call_time(K, N, bits, M, st["seed_base"], rows=128, matrix_index=j)
                cpu_s += c1["s"] * L
                samples.append(c1["sample"])
        out[f"bits{bits}"] = {"layers": L, "ms_per_pass": round(ms, 3), "tok_per_s": round(M / (ms * 1e-3), 1),
                              "tflops": round(flops / (ms * 1e-3) / 1e12, 1),
                              "frac_sustained": round(flops / (ms * 1e-3) / 1e12 / peaks["bf16_tflops_sustained"], 4),
                              "split_ms": {k: round(v, 3) for k, v in split.items()},
                              "first_nonfinite_layer": first_bad, "clocks": clk,
                              "cpu_baseline": oracle_line(ms, {"s": cpu_s, "extrapolated": True,
                                                               "sample": "layer 0 gate, up, down on 128 rows each: "
                                                                         + "; ".join(samples) + f"; x {L} layers",
                                                               "cores": c1["cores"]}) if samples else None,
                              "trellis_gb": round(sum(m["tr"].numel() * 2 for lay in layers for m in lay) / 1e9, 2)}
        del layers, ws
        torch.cuda.empty_cache()
    return out


def bench_decode_stack(args, torch, tql, peaks):
    """One decode step of the 64-layer MLP stack (gate, up 5120->17408;
    SiLU(gate)*up; down 17408->5120; bits 4) at M = 1 and 16: 192 linear
    calls and 64 glue calls, timed eagerly (one host launch per kernel) and
    replayed as one captured CUDA graph. Weights (8.56 GB) are drawn on the
    device (timing only); every weight byte comes from HBM once per step."""
    st = synthetic.MLP_STACK
    L, d, f, bits = st["layers"], st["d_model"], st["d_ff"], 4
    if args.quick:
        L = 8
    layers = []
    for l in range(L):
        mats = []
        for j, (K, N) in enumerate(((d, f), (d, f), (f, d))):
            tr, su, sv = synthetic.make_matrix_device(K, N, bits, seed=st["seed_base"] + l, matrix_index=j)
            mats.append(dict(K=K, N=N, tr=tr, su=su, sv=sv))
        layers.append(mats)
    wbytes = sum(m["tr"].numel() * 2 for lay in layers for m in lay)
    Mmax = 16
    ws = torch.empty(max(tql.exl3_linear_workspace_bytes(Mmax, d, f, bits, 0),
                         tql.exl3_linear_workspace_bytes(Mmax, f, d, bits, 0)), dtype=torch.uint8, device="cuda")
    tql.exl3_workspace_init(ws)
    out = {"layers": L, "bits": bits, "trellis_gb": round(wbytes / 1e9, 2)}
    stream = torch.cuda.Stream()
    for M in (1, 16):
        x0 = _dev(torch, synthetic.make_activations(M, d, seed=st["seed_base"], x_scale=0.05))
        g = torch.empty((M, f), dtype=torch.float16, device="cuda")
        u = torch.empty_like(g)
        h = torch.empty_like(g)
        xa = torch.empty((M, d), dtype=torch.float16, device="cuda")

        def one_step():
            xin = x0
            for mg, mu, md in layers:
                for m, yout in ((mg, g), (mu, u)):
                    tql.exl3_linear(xin, M, m["K"], m["tr"], bits, m["N"], m["N"], m["su"], m["sv"], yout,
                                    tql.EXL3_F16, 0, ws)
                tql.exl3_silu_mul(g, u, h)
                tql.exl3_linear(h, M, md["K"], md["tr"], bits, md["N"], md["N"], md["su"], md["sv"], xa,
                                tql.EXL3_F16, 0, ws)
                xin = xa

        with torch.cuda.stream(stream):
            eager_ms = time_fn(torch, one_step, 5, 2)
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gr, stream=stream):
                one_step()
            graph_ms = time_fn(torch, gr.replay, 20, 3)
        cpu = None
        if not args.quick:
            cpu_s, samples = 0.0, []
            for j, (K, N) in enumerate(((d, f), (d, f), (f, d))):
                c1 = oracle_call_time(K, N, bits, M, st["seed_base"], x_scale=0.05, matrix_index=j)
                cpu_s += c1["s"] * L
                samples.append(c1["sample"])
            cpu = oracle_line(graph_ms, {"s": cpu_s, "extrapolated": True, "cores": c1["cores"],
                                         "sample": "layer 0 gate, up, down in full: " + "; ".join(samples)
                                                   + f"; x {L} layers"})
        out[f"M{M}"] = {"eager_ms": round(eager_ms, 3), "graph_ms": round(graph_ms, 3), "cpu_baseline": cpu,
                        "graph_speedup": round(eager_ms / graph_ms, 3),
                        "graph_weight_gbs": round(wbytes / (graph_ms * 1e-3) / 1e9, 1),
                        "graph_frac_hbm": round(wbytes / (graph_ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
                        "us_per_linear": round(graph_ms * 1e3 / (3 * L), 2)}
        del gr
    del layers, ws
    torch.cuda.empty_cache()
    return out


# ---------------------------------------------------------------------------
# CPU oracle: baseline leg and reference arm
# ---------------------------------------------------------------------------

def oracle_sample(budget_s: float, total_s: float = 0.0):
    """Times the oracle on a column sample of the decode workload (M=16
    rows, full K), doubling the sample until one call takes >= budget_s (or
    covers all columns), then repeating that call until total_s seconds of
    CPU work have run."""
    import oracle
    oracle.build()
    g = synthetic.GATE_DECODE
    K, N, bits = g["K"], g["N"], g["bits"]
    mat = synthetic.make_matrix(K, N, bits, seed=g["seed"])
    x = synthetic.make_activations(16, K, seed=g["seed"], x_scale=g["x_scale"])
    cols = 256
    while True:
        t0 = time.perf_counter()
        oracle.linear(x, mat.trellis, bits, K, N, mat.su, mat.sv, 0, cols)
        dt = time.perf_counter() - t0
        if dt >= budget_s or cols >= N:
            break
        cols = min(N, cols * 2)
    calls, total = 1, dt
    while total < total_s:
        t0 = time.perf_counter()
        oracle.linear(x, mat.trellis, bits, K, N, mat.su, mat.sv, 0, cols)
        total += time.perf_counter() - t0
        calls += 1
    bytes_ = K * cols * bits // 8
    return {"value": bytes_ * calls / total / 1e9, "unit": "GB/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{calls} M=16 calls over columns [0, {cols}) of K=5120 N=17408 bits=4 "
                      f"({bytes_} trellis bytes each), {total:.1f} s", "cols": cols, "seconds": dt}


def profile_call(spec: str):
    """Runs exl3_linear a few times at one shape (decode-shaped unless a
    threshold <= M is given), for capturing its kernels under a profiler."""
    import torch
    import trellis_quantized_linear_gb300 as tql
    vals = [int(v) for v in spec.split(",")]
    K, N, bits, M = vals[:4]
    reps = vals[4] if len(vals) > 4 else 4
    thr = vals[5] if len(vals) > 5 else 0
    torch.cuda.set_device(0)
    tql.build()
    tql.exl3_init(0)
    mat = DevMatrix(torch, synthetic.make_matrix(K, N, bits, seed=synthetic.PREFILL_SEED))
    x = _dev(torch, synthetic.make_activations(M, K, seed=synthetic.PREFILL_SEED))
    y = torch.empty((M, N), dtype=torch.float16, device="cuda")
    ws = make_ws(torch, tql, M, K, N, bits, thr)
    for _ in range(reps):
        call_linear(tql, x, M, mat, y, thr, ws, tql.EXL3_F16)
    torch.cuda.synchronize()


def headline_config(world: int) -> dict:
    """The workload both arms measure (the GB300 arm and the oracle arm),
    with the GPU arm's L2 rule: its timed calls rotate over weight copies
    that together exceed L2 (no flush needed)."""
    g = synthetic.GATE_DECODE
    wbytes = g["K"] * g["N"] * g["bits"] // 8
    return {"workload": g["name"], "step": "exl3_linear at M=1,4,8,16 (fp16 out)",
            "parallelism": f"replicas x{world}",
            "l2": f"inputs larger than L2: {WEIGHT_COPIES} rotating weight copies "
                  f"({WEIGHT_COPIES * wbytes / 1e6:.0f} MB > 129 MB)"}


def run_reference(args, dist, budget_s: float = 150.0):
    """Reference arm: the CPU oracle on the host cores, on the headline step
    (the four calls at M = 1, 4, 8, 16), exactly --warmup untimed and --steps
    timed steps. Each step covers output columns [0, cols) of every call,
    with cols (a multiple of 128, at most N) sized so that the whole run
    stays within about budget_s seconds."""
    world, rank, _ = dist
    if rank != 0:
        return
    import oracle
    oracle.build()
    g = synthetic.GATE_DECODE
    K, N, bits, Ms = g["K"], g["N"], g["bits"], g["Ms"]
    mat = synthetic.make_matrix(K, N, bits, seed=g["seed"])
    xs = {M: synthetic.make_activations(M, K, seed=g["seed"], x_scale=g["x_scale"]) for M in Ms}

    def step(cols):
        for M in Ms:
            oracle.linear(xs[M], mat.trellis, bits, K, N, mat.su, mat.sv, 0, cols)

    t128 = float("inf")
    for _ in range(2):
        t0 = time.perf_counter()
        step(128)
        t128 = min(t128, time.perf_counter() - t0)
    n_steps = max(1, args.steps + args.warmup)
    cols = int(max(1, min(N // 128, budget_s / n_steps / t128))) * 128
    for _ in range(args.warmup):
        step(cols)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step(cols)
    dt = (time.perf_counter() - t0) / max(1, args.steps)
    bytes_ = len(Ms) * K * cols * bits // 8
    v = bytes_ / dt / 1e9
    sample = f"each step the four calls (M = 1, 4, 8, 16, full K) over output columns [0, {cols}) of {N}"
    line = {"impl": "reference", "metric": METRIC, "value": round(v, 4), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": headline_config(world),
            "cpu_baseline": {"value": round(v, 4), "unit": "GB/s", "cores": oracle.num_threads(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(v, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------

def main():
    args = parse_args()
    dist = dist_info()
    world, rank, local = dist
    if args.impl == "reference":
        run_reference(args, dist)
        return
    if args.profile_call:
        profile_call(args.profile_call)
        return
    import torch
    import trellis_quantized_linear_gb300 as tql
    if world > 1:
        torch.distributed.init_process_group(backend="nccl")
    torch.cuda.set_device(local)
    tql.build()
    tql.exl3_init(local)
    peaks = load_peaks()

    dec = bench_decode(args, torch, tql, peaks, dist)
    e2e = bench_e2e(args, torch, tql, dec)
    extras = {}
    if not args.no_extras and rank == 0:
        wanted = set(args.extras.split(","))
        for name, fn in (("prefill", lambda: bench_prefill(args, torch, tql, peaks)),
                         ("prefill_fused", lambda: bench_prefill_fused(args, torch, tql, peaks)),
                         ("crossover", lambda: bench_crossover(args, torch, tql)),
                         ("logits", lambda: bench_logits(args, torch, tql, peaks)),
                         ("mlp_stack", lambda: bench_mlp_stack(args, torch, tql, peaks)),
                         ("decode_stack", lambda: bench_decode_stack(args, torch, tql, peaks))):
            if name not in wanted:
                continue
            try:
                extras[name] = fn()
            except Exception as ex:  # report, never hide
                extras[name] = {"error": repr(ex)}
            torch.cuda.empty_cache()
    status = tql.exl3_get_device_status()
    cpu = None
    if rank == 0 and world == 1:
        cpu = oracle_sample(1.0, 10.0)
        cpu = {k: (round(v, 4) if isinstance(v, float) else v) for k, v in cpu.items() if k not in ("cols", "seconds")}
    if rank == 0:
        line = {
            "metric": METRIC, "value": round(dec["value"], 1), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dec["ms_per_step"], 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
            "data": "synthetic",
            "config": headline_config(world),
            "timing": {"method": "CUDA graph replays, CUDA events on the launching stream"},
            "roofline": dec["roofline"], "clocks": dec["clocks"], "e2e": e2e,
            "gpu_launches": dec["gpu_launches"], "per_m": dec["per_m"], "cpu_baseline": cpu,
            "device_status": status,
        }
        line.update(extras)
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
