#!/usr/bin/env python3
"""Benchmark of the ternary-weight linear layer's training step on GB300.

One step = one pass of the whole hot path over one batch of synthetic input:
  tern_materialize (q -> 2-bit tiles + bf16 operand planes)
  tern_linear_fwd  (Y = scale * (X T))
  tern_linear_bwd  (dX = dY W_eff^T; gq and sgrad from the fused G epilogue)
  adamw_step       (AdamW on the per-column scales, gradient sgrad)
on the large single projection X [32768 x 4096], q [4096 x 12288],
dY [32768 x 12288] (inputs larger than L2).  `value` is the credited work of
the layer, 6*M*K*N flops per step, in TFLOP/s over the device-timed step.

Extra keys: per-kernel times, the roofline of the dominant kernel, the end-to-end
figure through the C ABI with the step's inputs copied from pinned host memory
(and a second one that also reads every output back), the CPU oracle timed on a
bounded sample (every host core, and one), the clocks seen during the timed
region, AdamW / multi-tensor AdamW / ternarise bandwidth sweeps, and under
`workloads` the RWKV-style block (six projections at M = 8192) and the wide FFN
chain (2048 -> 6144 -> 2048 at M = 16384), each run in a fresh child process.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun (N > 1) every rank runs an independent replica of the step
(the layer's step has no exchange on one GPU); rank 0 prints the line.
"""
from __future__ import annotations

import argparse
import faulthandler
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import tern_synth as syn  # noqa: E402

METRIC = "ternary-linear fwd+bwd TFLOP/s (% bf16 TC peak); AdamW/ternarise HBM GB/s"
WORKLOADS = {
    "large_single_projection": dict(M=32768, K=4096, N=12288, scale_lo=0.005, scale_hi=0.05, zero_prob=0.0),
    "tiny": dict(M=64, K=128, N=128, scale_lo=0.01, scale_hi=0.1, zero_prob=0.0),
    # the large projection's weight with a quarter of its tokens: a profiling case whose
    # operands still exceed L2 (dY 201 MB) while the device holds under 1 GB
    "profile_quarter_tokens": dict(M=8192, K=4096, N=12288, scale_lo=0.005, scale_hi=0.05, zero_prob=0.0),
    # not a layer: the HBM-bound kernels alone (AdamW, ternarise, materialise, SR4, panel)
    "hbm_kernels": None,
    # the six projections of the RWKV-style block, M = 8192 (a child process of the default run)
    "rwkv_block": None,
    # the two-layer ternary FFN chain, M = 16384: 2048 -> 6144 -> 2048, layer 1's output
    # rounded to bf16 as layer 2's input (a child process of the default run)
    "wide_ffn_chain": None,
}
ADAM_HP = dict(lr=1e-3, b1=0.9, b2=0.95, eps=1e-8, wd=0.1)
# GB300 nominal dense bf16 tensor-core peak (without 2:4 sparsity), TFLOP/s
SPEC_BF16_TFLOPS = 2250.0


_T0 = time.perf_counter()


_PHASE = ["start"]


def progress(msg):
    """One line per bench phase on stderr (the JSON line alone goes to stdout)."""
    _PHASE[0] = msg
    print(f"[bench {time.perf_counter() - _T0:7.1f} s] {msg}", file=sys.stderr, flush=True)


class Watchdog:
    """Ends the process if the extra measurements stall: after `limit_s` it writes
    every thread's stack to stderr, prints the headline line (when given) with the
    stalled phase named, and exits.  The process exit releases the GPU context."""

    def __init__(self, limit_s, line, extra=None, diag=None):
        self.line = line
        self.extra = extra if extra is not None else {}
        self.diag = diag
        self.timer = threading.Timer(limit_s, self._fire, args=(limit_s,))
        self.timer.daemon = True
        self.timer.start()

    def _fire(self, limit_s):
        phase = _PHASE[0]
        faulthandler.dump_traceback(file=sys.stderr, all_threads=True)
        progress(f"watchdog: the extra lines did not finish within {limit_s:.0f} s (phase '{phase}')")
        # the line first: a CUDA call from this thread may block behind the stuck one
        if self.line is not None:
            self.line.update(self.extra)
            self.line["stalled"] = {"phase": phase, "limit_s": limit_s,
                                    "note": "the headline and e2e were complete; the extra lines were cut"}
            print(json.dumps(self.line), flush=True)
        if self.diag is not None:   # device-side records, twice: are GEMM CTAs still finishing?
            reads = []

            def read():
                for _ in range(2):
                    try:
                        reads.append(self.diag())
                    except Exception as e:   # noqa: BLE001 - report whatever the read says
                        reads.append(str(e))
                    time.sleep(2.0)
            t = threading.Thread(target=read, daemon=True)
            t.start()
            t.join(timeout=10.0)
            print(f"[bench] device diagnostics: {reads if reads else 'no answer within 10 s'}", file=sys.stderr,
                  flush=True)
        os._exit(0)

    def cancel(self):
        self.timer.cancel()


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm=float(d["hbm_gbs"]), bf16=float(d["bf16_tflops"]),
                    bf16_sus=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), src="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, src="fallback")


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(value, device=None):
    """The largest `value` over all ranks (the slowest replica sets the job time)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(flops_per_step, ms_per_step_max, world_size):
    """Whole-job TFLOP/s: every replica's work over the slowest replica's time."""
    return flops_per_step * world_size / (ms_per_step_max * 1e-3) / 1e12


# --------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms while running."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.idx = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.th = threading.Thread(target=self._read, daemon=True)
            self.th.start()
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append(ln.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# --------------------------------------------------------------------------- CPU oracle leg

def oracle_family_times(inp, budget_s, nthreads, seed=7):
    """Seconds per output of each output family of the layer (Y, dX, gq with sgrad),
    from the CPU oracle as it stands, run on blocks of whole rows with the oracle's
    own pthreads row split (nthreads threads; 1 = single-threaded) for about
    budget_s seconds in all.

    A Y row costs K*N multiply-adds, a dX row N*K and a gq row (G over every token,
    with its sgrad terms) M*N, so each family's time per output extrapolates to the
    whole layer.  Returns (per-family seconds per output, outputs sampled, threads)."""
    import oracle
    M, K, N = inp.M, inp.K, inp.N
    rng = np.random.default_rng(seed)
    rows = max(1, nthreads)
    fam = {"Y": [0.0, 0], "dX": [0.0, 0], "gq": [0.0, 0]}
    start = time.perf_counter()
    while time.perf_counter() - start < budget_s or min(v[1] for v in fam.values()) == 0:
        m0 = int(rng.integers(0, max(1, M - rows)))
        r0 = int(rng.integers(0, max(1, K - rows)))
        xs = np.ascontiguousarray(inp.X[m0:m0 + rows])
        dys = np.ascontiguousarray(inp.dY[m0:m0 + rows])
        xcols = np.ascontiguousarray(inp.X[:, r0:r0 + rows])
        qrows = np.ascontiguousarray(inp.q[r0:r0 + rows])
        t0 = time.perf_counter()
        oracle.fwd(xs, inp.q, inp.scale, nthreads=nthreads)
        t1 = time.perf_counter()
        oracle.dx(dys, inp.q, inp.scale, nthreads=nthreads)
        t2 = time.perf_counter()
        oracle.dw(xcols, inp.dY, qrows, inp.scale, nthreads=nthreads)
        t3 = time.perf_counter()
        for k, dt, n in (("Y", t1 - t0, xs.shape[0] * N), ("dX", t2 - t1, dys.shape[0] * K),
                         ("gq", t3 - t2, xcols.shape[1] * N)):
            fam[k][0] += dt
            fam[k][1] += n
    per = {k: v[0] / v[1] for k, v in fam.items()}
    return per, {k: v[1] for k, v in fam.items()}, nthreads


def oracle_baseline(inp, budget_s, nthreads):
    """The CPU oracle's throughput on the layer, extrapolated from sampled whole rows
    of each output family: (TFLOP/s, description, threads used)."""
    M, K, N = inp.M, inp.K, inp.N
    per, counts, nt = oracle_family_times(inp, budget_s, nthreads)
    full_s = per["Y"] * M * N + per["dX"] * M * K + per["gq"] * K * N
    tflops = 6.0 * M * K * N / full_s / 1e12
    desc = (f"{counts['Y'] // N} Y rows, {counts['dX'] // K} dX rows and {counts['gq'] // N} gq rows (with their "
            f"sgrad terms) of the same layer, fp64 dot products over K, N and M, on {nt} thread(s) by the "
            f"oracle's own row split; time per output extrapolated to all M*N + M*K + K*N outputs")
    return tflops, desc, nt


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_baseline_line(inp, budget_s):
    """cpu_baseline: the oracle on every host core (the value) and on one core."""
    nproc = host_cores()
    v1, d1, _ = oracle_baseline(inp, budget_s * 0.35, 1)
    vn, dn, nt = oracle_baseline(inp, budget_s * 0.65, nproc)
    return {"value": vn, "unit": "TFLOP/s", "cores": nt, "nproc": nproc, "kind": "oracle", "sample": dn,
            "single_thread": {"value": v1, "cores": 1, "sample": d1}}


def make_inputs(wl):
    c = WORKLOADS[wl]
    return syn.linear_inputs(c["M"], c["K"], c["N"], seed=0, scale_lo=c["scale_lo"], scale_hi=c["scale_hi"],
                             zero_prob=c["zero_prob"])


# --------------------------------------------------------------------------- reference arm

def large_config(M, K, N, ws=1):
    """The `config` object of the large-projection line (both arms)."""
    return {"workload": "large_single_projection", "M": M, "K": K, "N": N, "theta": 2, "q_clamp": 7,
            "step": "materialise + fwd + bwd (dX, gq, sgrad) + AdamW on scale",
            "flops_per_step": 6.0 * M * K * N, "l2": "inputs larger than L2 (X 268 MB, dY 805 MB)",
            "parallelism": f"replicas x{ws}"}


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    inp = make_inputs(args.workload)
    total = args.steps + args.warmup
    per_step = max(1.0, min(6.0, 150.0 / max(total, 1)))
    nproc = host_cores()
    for _ in range(args.warmup):
        oracle_baseline(inp, per_step / 4, nproc)
    vals, desc, cores = [], "", nproc
    t0 = time.perf_counter()
    for _ in range(args.steps):
        v, desc, cores = oracle_baseline(inp, per_step, nproc)
        vals.append(v)
    wall = time.perf_counter() - t0
    value = statistics.median(vals)
    M, K, N = inp.M, inp.K, inp.N
    cfg = large_config(M, K, N, ws) if args.workload == "large_single_projection" else \
        {"workload": args.workload, "M": M, "K": K, "N": N}
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 6.0 * M * K * N / (value * 1e12) * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": cfg,
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "nproc": nproc, "kind": "oracle",
                         "sample": f"per step: {desc}; {args.steps} steps in {wall:.1f} s"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# --------------------------------------------------------------------------- our arm

def code_hash(src_files):
    """Hash of the sources' code: comments, trailing blanks and empty lines removed, so
    that a comment edit does not count as a kernel change."""
    h = hashlib.sha256()
    for f in src_files:
        text = open(f, encoding="utf-8").read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        lines = [re.sub(r"//.*$", "", ln).rstrip() for ln in text.splitlines()]
        h.update("\n".join(ln for ln in lines if ln).encode())
    return h.hexdigest()[:16]


def traffic_from_profiles(kernel, src_files):
    """dram bytes per launch committed under profiles/, if the kernel code is unchanged since."""
    p = os.path.join(ROOT, "profiles", "traffic.md")
    if not os.path.exists(p):
        return None
    digest = code_hash(src_files)
    for ln in open(p):
        m = re.match(r"^\|\s*(\w+)\s*\|\s*([0-9.eE+]+)\s*\|\s*(\w+)\s*\|", ln)
        if m and m.group(1) == kernel and m.group(3) == digest:
            return float(m.group(2))
    return None


def rwkv_block(bl, dev, stream, steps):
    """The six projections of the RWKV-style block at M = 8192 tokens (receptance, key,
    value, output 512 x 512; channel-mixing key 512 x 2048 and value 2048 x 512), each
    with its own seeded X, dY, q and scale.  One step materialises the six weights,
    runs every forward and backward (dX, gq, sgrad) and AdamW on the six scales, under
    three launch schedules:
      independent   the six layers as one group per GEMM kind (one forward launch,
                    one dX and one G launch, their reduces), which the workload's six
                    independent inputs allow;
      dependency    the order a block's data flow imposes: r, k, v as one group, then
                    the output projection, the channel-mixing key and value one after
                    another (and the reverse in the backward);
      per_layer     the single-layer calls.
    independent_2bit_T is the independent schedule with the forward reading T as the 2-bit
    codes (materialise then skips the bf16 T plane).  Each is timed eager and replayed as
    one CUDA graph.  The grouped schedules use the
    prepared calls (arguments marshalled once); per_layer uses the plain functions."""
    import torch
    M = 8192
    shapes = syn.RWKV_SHAPES

    def bf(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)

    layers = []
    for i, (K, N) in enumerate(shapes):
        inp = syn.linear_inputs(M, K, N, seed=1, scale_lo=0.01, scale_hi=0.1,
                                tids=(10 * i + 1, 10 * i + 2, 10 * i + 3, 10 * i + 4))
        L = dict(K=K, N=N, X=bf(inp.X), dY=bf(inp.dY), q=torch.from_numpy(inp.q).to(dev),
                 scale=torch.from_numpy(inp.scale).to(dev), tiles=bl.Tiles.empty(K, N, device=dev),
                 Y=torch.empty(M, N, device=dev), dX=torch.empty(M, K, device=dev),
                 gq=torch.empty(K, N, device=dev), sgrad=torch.empty(N, device=dev),
                 ws=bl.workspace_for(M, K, N, device=dev), m=torch.zeros(N, device=dev),
                 v=torch.zeros(N, device=dev))
        layers.append(L)
    adam_scalars = torch.tensor([ADAM_HP["lr"], 1 - ADAM_HP["b1"], 1 - ADAM_HP["b2"], 1.0], device=dev)

    # the grouped schedules call the library through prepared calls (arguments marshalled
    # once), as a training loop repeating the step on the same buffers does, and materialise
    # the six weights in one grouped call
    adam_all = bl.MultiAdamW([L["scale"] for L in layers], [L["sgrad"] for L in layers], [L["m"] for L in layers],
                             [L["v"] for L in layers], adam_scalars, ADAM_HP["b1"], ADAM_HP["b2"], ADAM_HP["eps"],
                             ADAM_HP["wd"])

    def per_layer():
        for L in layers:
            bl.tern_materialize(L["q"], L["scale"], L["tiles"], 2, 7)
            bl.tern_linear_fwd(L["X"], L["tiles"], L["scale"], L["Y"])
            bl.tern_linear_bwd(L["X"], L["dY"], L["tiles"], L["scale"], L["dX"], L["gq"], L["sgrad"], L["ws"])
            bl.adamw_step(L["scale"], L["sgrad"], L["m"], L["v"], 1, **ADAM_HP)

    def grouped(fwd_groups, bwd_groups, packed_t=False):
        # packed_t: the forward reads T as the 2-bit codes and materialise skips the bf16 T plane
        tl = [bl.Tiles(L["K"], L["N"], packed=L["tiles"].packed, whi_bf16=L["tiles"].whi_bf16,
                       wlo_bf16=L["tiles"].wlo_bf16) if packed_t else L["tiles"] for L in layers]
        mat_all = bl.MaterializeGrouped([dict(q=L["q"], scale=L["scale"], tiles=t_) for L, t_ in zip(layers, tl)],
                                        2, 7)
        fwds = [bl.GroupedForward([dict(X=layers[i]["X"], tiles=tl[i], scale=layers[i]["scale"],
                                        Y=layers[i]["Y"]) for i in gr]) for gr in fwd_groups]
        bwds = []
        for gr in bwd_groups:
            ws_ = torch.empty(bl.tern_linear_bwd_grouped_workspace([(M, layers[i]["K"], layers[i]["N"]) for i in gr])
                              // 4, device=dev)
            bwds.append(bl.GroupedBackward([dict(X=layers[i]["X"], dY=layers[i]["dY"], tiles=tl[i],
                                                 scale=layers[i]["scale"], dX=layers[i]["dX"], gq=layers[i]["gq"],
                                                 sgrad=layers[i]["sgrad"]) for i in gr], ws_))

        def step():
            mat_all()
            for f_ in fwds:
                f_()
            for b_ in bwds:
                b_()
            adam_all()
        return step

    schedules = {
        "independent": grouped([[0, 1, 2, 3, 4, 5]], [[0, 1, 2, 3, 4, 5]]),
        "independent_2bit_T": grouped([[0, 1, 2, 3, 4, 5]], [[0, 1, 2, 3, 4, 5]], packed_t=True),
        "dependency": grouped([[0, 1, 2], [3], [4], [5]], [[5], [4], [3], [0, 1, 2]]),
        "per_layer": per_layer,
    }
    launches = {"independent": 1 + 1 + 4 + 1, "independent_2bit_T": 1 + 1 + 4 + 1, "dependency": 1 + 4 + 4 * 3 + 1,
                "per_layer": 6 * 6}
    flops = 6.0 * M * sum(K * N for K, N in shapes)
    reps = max(20, min(steps, 200))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def checked(fn, what):
        fn()
        st = bl.tern_device_status()
        if st != bl.TERN_OK:
            raise RuntimeError(f"RWKV block, {what}: {bl.strerror(st)}")

    def eager(fn):
        checked(fn, "first eager step")
        for _ in range(4):
            fn()
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(reps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / reps

    def graphed(fn):
        g = torch.cuda.CUDAGraph()
        s2 = torch.cuda.Stream()
        s2.wait_stream(stream)
        with torch.cuda.graph(g, stream=s2):
            fn()
        torch.cuda.synchronize()
        checked(g.replay, "first graph replay")
        for _ in range(2):
            g.replay()
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / reps

    def rate(ms):
        return {"ms": ms, "tflops": flops / (ms * 1e-3) / 1e12}

    out = {"M": M, "shapes": [list(x) for x in shapes], "flops_per_step": flops, "timing":
           f"{reps} steps per figure, CUDA events on the launching stream; eager launches and one CUDA-graph replay "
           "per step", "schedules": {}}
    for name, fn in schedules.items():
        progress(f"RWKV block: {name}, eager")
        em = eager(fn)
        progress(f"RWKV block: {name}, graph")
        gm = graphed(fn)
        out["schedules"][name] = {"eager": rate(em), "graph": rate(gm), "launches_per_step_approx": launches[name]}
    st = bl.tern_device_status()
    if st != bl.TERN_OK:
        raise RuntimeError(f"RWKV block: {bl.strerror(st)}")
    best = out["schedules"]["independent"]["eager"]
    out["tflops"], out["ms"] = best["tflops"], best["ms"]
    out["headline"] = "independent schedule, eager"
    return out


def wide_chain(bl, dev, stream, steps):
    """Two chained projections, (M, K1, N1) = (16384, 2048, 6144) then (16384, 6144, 2048),
    40% of q forced to zero: materialise both (one grouped call), fwd 1 writes its output in bf16 only
    (layer 2's input), fwd 2, bwd 2 writes its input gradient in bf16 only (layer 1's
    dY), bwd 1, then AdamW of both scales in one launch."""
    import torch
    c = syn.WIDE
    M, K1, N1 = c["M"], c["K"], c["N"]

    def bf(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)

    a = syn.linear_inputs(M, K1, N1, seed=3, scale_lo=c["scale_lo"], scale_hi=c["scale_hi"],
                          zero_prob=c["zero_prob"], tids=(31, 33, 34, 32))
    b = syn.linear_inputs(M, N1, K1, seed=3, scale_lo=c["scale_lo"], scale_hi=c["scale_hi"],
                          zero_prob=c["zero_prob"], tids=(41, 43, 44, 42))
    X = bf(a.X)
    dY2 = bf(b.dY)
    q1, q2 = torch.from_numpy(a.q).to(dev), torch.from_numpy(b.q).to(dev)
    s1, s2 = torch.from_numpy(a.scale).to(dev), torch.from_numpy(b.scale).to(dev)
    t1, t2 = bl.Tiles.empty(K1, N1, device=dev), bl.Tiles.empty(N1, K1, device=dev)
    X2 = torch.empty(M, N1, dtype=torch.bfloat16, device=dev)
    Y2 = torch.empty(M, K1, device=dev)
    dY1 = torch.empty(M, N1, dtype=torch.bfloat16, device=dev)
    dX1 = torch.empty(M, K1, device=dev)
    gq1, gq2 = torch.empty(K1, N1, device=dev), torch.empty(N1, K1, device=dev)
    sg1, sg2 = torch.empty(N1, device=dev), torch.empty(K1, device=dev)
    m1, v1, m2, v2 = (torch.zeros(n, device=dev) for n in (N1, N1, K1, K1))
    ws1 = torch.empty(bl.tern_linear_bwd_grouped_workspace([(M, K1, N1)]) // 4, device=dev)
    ws2 = torch.empty(bl.tern_linear_bwd_grouped_workspace([(M, N1, K1)]) // 4, device=dev)
    adam_scalars = torch.tensor([ADAM_HP["lr"], 1 - ADAM_HP["b1"], 1 - ADAM_HP["b2"], 1.0], device=dev)
    names = ["materialize", "fwd1", "fwd2", "bwd2", "bwd1", "adamw"]
    mat = bl.MaterializeGrouped([dict(q=q1, scale=s1, tiles=t1), dict(q=q2, scale=s2, tiles=t2)], 2, 7)

    def step(ev=None):
        def mark(i):
            if ev is not None:
                ev[i].record(stream)
        mark(0)
        mat()
        mark(1)
        bl.tern_linear_fwd_grouped([dict(X=X, tiles=t1, scale=s1, Y_bf16=X2)])
        mark(2)
        bl.tern_linear_fwd_grouped([dict(X=X2, tiles=t2, scale=s2, Y=Y2)])
        mark(3)
        bl.tern_linear_bwd_grouped([dict(X=X2, dY=dY2, tiles=t2, scale=s2, dX_bf16=dY1, gq=gq2, sgrad=sg2)], ws2)
        mark(4)
        bl.tern_linear_bwd_grouped([dict(X=X, dY=dY1, tiles=t1, scale=s1, dX=dX1, gq=gq1, sgrad=sg1)], ws1)
        mark(5)
        bl.adamw_step_multi([s1, s2], [sg1, sg2], [m1, m2], [v1, v2], adam_scalars, ADAM_HP["b1"], ADAM_HP["b2"],
                            ADAM_HP["eps"], ADAM_HP["wd"])
        mark(6)

    flops = 6.0 * M * (K1 * N1 + N1 * K1)
    reps = max(10, min(steps, 100))
    for _ in range(5):
        step()
    torch.cuda.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(7)] for _ in range(reps)]
    for i in range(reps):
        step(evs[i])
    torch.cuda.synchronize()
    if bl.tern_device_status() != bl.TERN_OK:
        raise RuntimeError("a kernel gave up on a bounded wait in the FFN chain")
    ms = evs[0][0].elapsed_time(evs[-1][6]) / reps
    per = {n: statistics.mean(e[j].elapsed_time(e[j + 1]) for e in evs) for j, n in enumerate(names)}
    gemm_flops = {"fwd1": 2.0 * M * K1 * N1, "fwd2": 2.0 * M * K1 * N1, "bwd2": 4.0 * M * K1 * N1,
                  "bwd1": 4.0 * M * K1 * N1}
    return {"M": M, "layers": [[K1, N1], [N1, K1]], "q_zero_fraction": c["zero_prob"], "flops_per_step": flops,
            "ms": ms, "tflops": flops / (ms * 1e-3) / 1e12,
            "parts_ms": per, "parts_tflops": {n: f / (per[n] * 1e-3) / 1e12 for n, f in gemm_flops.items()},
            "timing": f"{reps} eager steps, CUDA events on the launching stream"}


def graph_bw(torch, fn, nbytes, reps, warm, stream, peak_gbs):
    """Device time per call of `fn` over `reps` calls captured in one CUDA graph."""
    for _ in range(warm):
        fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.graph(g, stream=side):
        for _ in range(reps):
            fn()
    torch.cuda.synchronize()
    g.replay()                     # warm replay
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    g.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / reps
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"ms": ms, "gbs": gbs, "frac": gbs / peak_gbs, "timing": f"{reps} calls in one CUDA graph"}


def hbm_kernels(args):
    """The HBM-bound kernels alone at profiling sizes (each input over L2, a few GB in
    all): AdamW on 1e8 elements, packed ternarisation of 1e9 weights, the full
    materialise, the SR4 step and the panel of the large projection's weight, the fp16 +
    e4m3 dX planes and the split dX call (whose dY split is the HBM-bound part).
    Prints one line of GB/s per kernel; a case for ncu, not a bench line."""
    import torch
    torch.cuda.set_device(0)
    import __graft_entry__
    __graft_entry__._builder().build()
    import bit_linear_gb300 as bl
    dev = torch.device("cuda")
    pk = peaks()
    stream = torch.cuda.current_stream()

    def loop(fn, nbytes, reps):
        return graph_bw(torch, fn, nbytes, reps, args.warmup, stream, pk["hbm"])

    out = {}
    n = 100_000_000
    w, g = torch.empty(n, device=dev).normal_(0, 0.02), torch.empty(n, device=dev).normal_(0, 1e-3)
    m, v = torch.zeros(n, device=dev), torch.zeros(n, device=dev)
    out["adamw_1e8"] = loop(lambda: bl.adamw_step(w, g, m, v, 1, **ADAM_HP), 28 * n, args.steps)
    del w, g, m, v
    Kt, Nt = 65536, 15264
    qt = torch.randint(-7, 8, (Kt, Nt), dtype=torch.int8, device=dev)
    tt = bl.Tiles(Kt, Nt, packed=torch.empty((Kt, Nt // 16), dtype=torch.int32, device=dev))
    out["ternarise_1e9"] = loop(lambda: bl.tern_materialize(qt, None, tt, 2, 7), 1.25 * Kt * Nt, args.steps)
    del qt, tt
    K, N = 4096, 12288
    q = torch.randint(-7, 8, (K, N), dtype=torch.int8, device=dev)
    scale = torch.empty(N, device=dev).uniform_(0.005, 0.05)
    tiles = bl.Tiles.empty(K, N)
    out["materialise_all_planes"] = loop(lambda: bl.tern_materialize(q, scale, tiles, 2, 7), 7.25 * K * N, args.steps)
    gq = torch.empty(K, N, device=dev).normal_(0, 1e-3)
    ws = torch.empty(bl.tern_sr4_workspace(K * N) // 4 + 4, device=dev)
    out["sr4_step"] = loop(lambda: bl.tern_sr4_step(q, gq, ws, target_step=0.003), 10.0 * K * N, args.steps)
    counts = torch.zeros(6, dtype=torch.int64, device=dev)
    stats = torch.zeros(3, dtype=torch.float64, device=dev)
    out["sr4_panel"] = loop(lambda: bl.tern_sr4_panel(q, scale, counts, stats, packed_prev=tiles.packed),
                            1.25 * K * N, args.steps)
    # the fp16 + e4m3 dX planes alone (1 B of q read, 2 + 1 B written per weight), and the
    # split of dY at the profiling case's M = 8192 (2 B read, 3 B written per element; the
    # call also runs the split GEMM, so this is a case for ncu's per-kernel counters)
    t8 = bl.Tiles(K, N, whi_f16=torch.empty((K, N), dtype=torch.float16, device=dev),
                  wlo_e4m3=torch.empty((K, N), dtype=torch.uint8, device=dev))
    out["split8_planes"] = loop(lambda: bl.tern_materialize(q, scale, t8, 2, 7), 4.0 * K * N, args.steps)
    Mq = 8192
    X = torch.empty(Mq, K, device=dev).normal_().to(torch.bfloat16)
    dY = torch.empty(Mq, N, device=dev).normal_(0, 0.01).to(torch.bfloat16)
    dX = torch.empty(Mq, K, device=dev)
    ws8 = torch.empty(bl.tern_linear_bwd_workspace_ex(Mq, K, N, bl.TERN_BWD_DX_SPLIT8) // 4, device=dev)
    out["split8_dx_call"] = loop(lambda: bl.tern_linear_bwd(X, dY, t8, scale, dX, None, None, ws8, split8=True),
                                 5.0 * Mq * N, args.steps)
    print(json.dumps({"hbm_kernels": out, "peak_hbm_gbs": pk["hbm"]}), flush=True)
    return 0


def run_ours(args):
    import torch

    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    import __graft_entry__
    __graft_entry__._builder().build()
    import bit_linear_gb300 as bl
    bl.tern_device_diagnostics()   # creates its stream and buffer while the device is healthy

    pk = peaks()
    progress(f"generating inputs ({args.workload})")
    inp = make_inputs(args.workload)
    M, K, N = inp.M, inp.K, inp.N
    dev = torch.device("cuda")

    def bf(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)

    X_h, dY_h = bf(inp.X).pin_memory(), bf(inp.dY).pin_memory()
    X, dY = X_h.to(dev), dY_h.to(dev)
    q = torch.from_numpy(inp.q).to(dev)
    scale0 = torch.from_numpy(inp.scale).to(dev)
    scale = scale0.clone()
    ms, vs = torch.zeros(N, device=dev), torch.zeros(N, device=dev)
    # the forward's T operand: bf16 planes (t_operand "bf16") or the 2-bit codes expanded
    # inside the GEMM ("packed": the materialise pass then skips the bf16 T plane)
    tiles = bl.Tiles.empty(K, N, t=(args.t_operand == "bf16"))
    Y = torch.empty(M, N, device=dev)
    dX = torch.empty(M, K, device=dev)
    gq = torch.empty(K, N, device=dev)
    sgrad = torch.empty(N, device=dev)
    wsp = bl.workspace_for(M, K, N)
    stream = torch.cuda.current_stream()
    names = ["materialize", "fwd", "dx", "dw", "adamw"]
    step_no = [0]

    def step(ev=None, Xs=None, dYs=None, tl=None, ws8=None, wsd=None):
        Xs = X if Xs is None else Xs
        dYs = dY if dYs is None else dYs
        tl = tiles if tl is None else tl
        step_no[0] += 1
        if ev is not None:
            ev[0].record(stream)
        bl.tern_materialize(q, scale, tl, 2, 7)
        if ev is not None:
            ev[1].record(stream)
        bl.tern_linear_fwd(Xs, tl, scale, Y)
        if ev is not None:
            ev[2].record(stream)
        if ws8 is None:   # dX from the 2-bit codes takes a workspace for its s_hi / s_lo table
            bl.tern_linear_bwd(Xs, dYs, tl, scale, dX, None, None, wsd)
        else:   # dX from the fp16 + e4m3 split: dY is split into ws8 first
            bl.tern_linear_bwd(Xs, dYs, tl, scale, dX, None, None, ws8, split8=True)
        if ev is not None:
            ev[3].record(stream)
        bl.tern_linear_bwd(Xs, dYs, tl, scale, None, gq, sgrad, wsp)
        if ev is not None:
            ev[4].record(stream)
        bl.adamw_step(scale, sgrad, ms, vs, step_no[0], **ADAM_HP)
        if ev is not None:
            ev[5].record(stream)

    # materialise, fwd, dX, G, sgrad reduce, AdamW; plus the split G tail and its reduce when the
    # last wave of G tiles is partial (768 pair tiles on 76 pairs at the large shape)
    units = torch.cuda.get_device_properties(dev).multi_processor_count // 2
    g_tiles = ((K + 255) // 256) * ((N + 255) // 256)
    launches_per_step = 6 + (2 if g_tiles % units else 0)

    progress("warm-up steps")
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    progress("timed steps")
    if bl.tern_device_status() != bl.TERN_OK:
        raise RuntimeError("a kernel gave up on a bounded wait during warm-up")

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(args.steps)]
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        for i in range(args.steps):
            step(evs[i])
        torch.cuda.synchronize()
    if ws > 1:
        torch.distributed.barrier()
    st = bl.tern_device_status()
    if st != bl.TERN_OK:
        raise RuntimeError(f"device status: {bl.strerror(st)}")
    total_ms = evs[0][0].elapsed_time(evs[-1][5])
    per = {n: statistics.mean(e[j].elapsed_time(e[j + 1]) for e in evs) for j, n in enumerate(names)}
    total_ms = max_over_ranks(total_ms, dev)
    ms_step = total_ms / args.steps
    flops = 6.0 * M * K * N
    value = job_throughput(flops, ms_step, ws)

    # kernel rooflines: credited flops per launch / average launch time.  The timed
    # region is a short burst of steps (well under a second), so the measured burst
    # bf16 peak is the denominator; the sustained one is given beside it.
    credited = {"fwd": 2.0 * M * K * N, "dx": 2.0 * M * K * N, "dw": 2.0 * M * K * N}
    kern = {}
    for n in names:
        kern[n] = {"ms": per[n]}
    for n, f in credited.items():
        kern[n]["tflops"] = f / (per[n] * 1e-3) / 1e12
        kern[n]["frac_of_measured_burst"] = kern[n]["tflops"] / pk["bf16"]
    # dX runs two bf16 passes (W_hi and W_lo) into one accumulator: 4*M*K*N executed
    kern["dx"]["executed_tflops"] = 2.0 * kern["dx"]["tflops"]
    mat_bytes = K * N * (1 + 0.25 + (2 if args.t_operand == "bf16" else 0) + 2 + 2) + N * 4
    kern["materialize"]["gbs"] = mat_bytes / (per["materialize"] * 1e-3) / 1e9
    kern["materialize"]["frac_of_measured_hbm"] = kern["materialize"]["gbs"] / pk["hbm"]
    dom = max(credited, key=lambda n: per[n])
    kname = {"fwd": "tern_fwd_gemm", "dx": "tern_dx_gemm", "dw": "tern_dw_gemm"}[dom]
    gemm_src = [os.path.join(ROOT, "bit_linear_gb300", "csrc", f) for f in ("gemm.cu", "common.cuh")]
    traffic = traffic_from_profiles(kname, gemm_src)
    roof = {"kernel": kname, "bound": "tensor", "achieved": kern[dom]["tflops"], "peak": pk["bf16"],
            "unit": "TFLOP/s", "frac": kern[dom]["tflops"] / pk["bf16"], "traffic": traffic,
            "peak_kind": f"{pk['src']} burst bf16 (torch.matmul 8192^3); the timed region is "
                         f"{total_ms / 1e3:.2f} s of steps",
            "frac_of_measured_sustained": kern[dom]["tflops"] / pk["bf16_sus"],
            "credited": "2*M*K*N per launch" + (" (the kernel executes twice that: two bf16 passes)"
                                                if dom == "dx" else "")}

    # ---- the same step with the forward's other T operand (bf16 plane or 2-bit codes)
    progress("step with the other forward operand")
    other = "packed" if args.t_operand == "bf16" else "bf16"
    tiles_o = bl.Tiles.empty(K, N, t=(other == "bf16"))
    for _ in range(3):
        step(tl=tiles_o)
    torch.cuda.synchronize()
    evo = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(args.steps)]
    for i in range(args.steps):
        step(evo[i], tl=tiles_o)
    torch.cuda.synchronize()
    if bl.tern_device_status() != bl.TERN_OK:
        raise RuntimeError("a kernel gave up on a bounded wait (other forward operand)")
    per_o = {n: statistics.mean(e[j].elapsed_time(e[j + 1]) for e in evo) for j, n in enumerate(names)}
    ms_o = evo[0][0].elapsed_time(evo[-1][5]) / args.steps
    variant = {"t_operand": other, "ms_per_step": ms_o, "tflops": flops / (ms_o * 1e-3) / 1e12,
               "kernels_ms": per_o, "fwd_tflops": 2.0 * M * K * N / (per_o["fwd"] * 1e-3) / 1e12,
               "materialize_bytes_per_weight": 1 + 0.25 + (2 if other == "bf16" else 0) + 4}
    del tiles_o

    # ---- the same step with dX's W_hi / W_lo expanded from the 2-bit codes inside the GEMM
    #      (materialise then writes no hi/lo planes: 3.25 instead of 7.25 B per weight)
    progress("step with dX from the 2-bit codes")
    tiles_c = bl.Tiles.empty(K, N, t=(args.t_operand == "bf16"), hi_lo=False)
    wsc = torch.empty(max(bl.tern_linear_bwd_workspace(M, K, N) // 4, N), device=dev)
    for _ in range(3):
        step(tl=tiles_c, wsd=wsc)
    torch.cuda.synchronize()
    evc = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(args.steps)]
    for i in range(args.steps):
        step(evc[i], tl=tiles_c, wsd=wsc)
    torch.cuda.synchronize()
    if bl.tern_device_status() != bl.TERN_OK:
        raise RuntimeError("a kernel gave up on a bounded wait (dX from the 2-bit codes)")
    per_c = {n: statistics.mean(e[j].elapsed_time(e[j + 1]) for e in evc) for j, n in enumerate(names)}
    ms_c = evc[0][0].elapsed_time(evc[-1][5]) / args.steps
    dxc = {"ms_per_step": ms_c, "tflops": flops / (ms_c * 1e-3) / 1e12, "kernels_ms": per_c,
           "dx_tflops_credited": 2.0 * M * K * N / (per_c["dx"] * 1e-3) / 1e12,
           "dx_ms_includes": "the s_hi / s_lo table (N columns) and the GEMM",
           "materialize_bytes_per_weight": 1 + 0.25 + (2 if args.t_operand == "bf16" else 0)}
    del tiles_c, wsc

    # ---- the same step with dX from the fp16 + e4m3 split (TERN_BWD_DX_SPLIT8): one
    #      binary16 and one e4m3 pass (1.5 bf16-pass equivalents executed) after a split of dY
    progress("step with dX from the fp16 + e4m3 split")
    tiles_8 = bl.Tiles.empty(K, N, t=(args.t_operand == "bf16"), hi_lo=False, split8=True)
    ws8 = torch.empty(bl.tern_linear_bwd_workspace_ex(M, K, N, bl.TERN_BWD_DX_SPLIT8) // 4, device=dev)
    for _ in range(3):
        step(tl=tiles_8, ws8=ws8)
    torch.cuda.synchronize()
    ev8 = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(args.steps)]
    for i in range(args.steps):
        step(ev8[i], tl=tiles_8, ws8=ws8)
    torch.cuda.synchronize()
    if bl.tern_device_status() != bl.TERN_OK:
        raise RuntimeError("a kernel gave up on a bounded wait (dX from the fp16 + e4m3 split)")
    per_8 = {n: statistics.mean(e[j].elapsed_time(e[j + 1]) for e in ev8) for j, n in enumerate(names)}
    ms_8 = ev8[0][0].elapsed_time(ev8[-1][5]) / args.steps
    dx8 = {"ms_per_step": ms_8, "tflops": flops / (ms_8 * 1e-3) / 1e12, "kernels_ms": per_8,
           "dx_tflops_credited": 2.0 * M * K * N / (per_8["dx"] * 1e-3) / 1e12,
           "dx_executed": "2*M*K*N binary16 + 2*M*K*N e4m3 (1.5 bf16-pass equivalents), after the dY split",
           "dx_ms_includes": "the dY split (binary16 and e4m3 copies, per-row exponents) and the GEMM",
           "materialize_bytes_per_weight": 1 + 0.25 + (2 if args.t_operand == "bf16" else 0) + 3,
           "error_bound": "6.3e-5*sum|term| + 4.3e-9*max_c|dY*scale|*nnz(T row), against 1e-4*sum|term|"}
    del tiles_8, ws8

    # ---- end to end through the C ABI: every step's inputs X and dY copied from
    #      pinned host memory and the step's result (updated scales and their
    #      gradient) read back.  The upload of step i+1 runs on a copy stream into
    #      the other of two input buffers while step i computes (double buffering).
    progress("end to end")
    e2e_steps = min(args.steps, 50)
    res_h = torch.empty(2, N, dtype=torch.float32).pin_memory()
    Xb, dYb = [X, torch.empty_like(X)], [dY, torch.empty_like(dY)]
    copy_streams = [torch.cuda.Stream(), torch.cuda.Stream()]   # X and dY on separate copy engines
    copied = [[torch.cuda.Event(), torch.cuda.Event()] for _ in range(2)]
    consumed = [torch.cuda.Event(), torch.cuda.Event()]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def upload(i):
        b = i % 2
        for cs, dst, src, ev in zip(copy_streams, (Xb[b], dYb[b]), (X_h, dY_h), copied[b]):
            cs.wait_event(consumed[b] if i >= 2 else e0)
            with torch.cuda.stream(cs):
                dst.copy_(src, non_blocking=True)
            ev.record(cs)

    torch.cuda.synchronize()
    e0.record(stream)
    upload(0)
    for i in range(e2e_steps):
        if i + 1 < e2e_steps:
            upload(i + 1)
        b = i % 2
        for ev in copied[b]:
            stream.wait_event(ev)
        step(None, Xb[b], dYb[b])
        consumed[b].record(stream)
        res_h[0].copy_(scale, non_blocking=True)
        res_h[1].copy_(sgrad, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    h2d = X.numel() * 2 + dY.numel() * 2
    d2h = 2 * N * 4
    # the host -> device rate alone (X and dY on their two copy streams, no compute):
    # the end-to-end step is copy-bound when h2d / rate exceeds the device step
    c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    c0.record(stream)
    for cs in copy_streams:
        cs.wait_event(c0)
    for _ in range(3):
        for cs, dst, src in zip(copy_streams, (Xb[0], dYb[0]), (X_h, dY_h)):
            with torch.cuda.stream(cs):
                dst.copy_(src, non_blocking=True)
    for cs in copy_streams:
        done = torch.cuda.Event()
        done.record(cs)
        stream.wait_event(done)
    c1.record(stream)
    torch.cuda.synchronize()
    h2d_gbs = 3 * h2d / (c0.elapsed_time(c1) * 1e-3) / 1e9
    del Xb, dYb

    # ---- the same, with every output of the layer brought back to the host each step
    #      (Y, dX, gq, sgrad and the updated scale): one stream, no overlap of the copies
    progress("end to end, every output read back")
    all_steps = 5
    outs_h = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in (Y, dX, gq, sgrad, scale)]
    torch.cuda.synchronize()
    a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a0.record(stream)
    for _ in range(all_steps):
        X.copy_(X_h, non_blocking=True)
        dY.copy_(dY_h, non_blocking=True)
        step()
        for h, d in zip(outs_h, (Y, dX, gq, sgrad, scale)):
            h.copy_(d, non_blocking=True)
    a1.record(stream)
    torch.cuda.synchronize()
    all_ms = a0.elapsed_time(a1) / all_steps
    d2h_all = sum(t.numel() * t.element_size() for t in outs_h)
    del outs_h

    line = None
    if rank == 0:
        cpu = None
        if ws == 1 and not args.skip_cpu:
            progress("CPU oracle sample")
            cpu = cpu_baseline_line(inp, args.cpu_budget)
        csum = clk.summary()
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": dict(large_config(M, K, N, ws), t_operand=args.t_operand),
            "other_t_operand": variant,
            "dx_split8": dx8,
            "dx_from_codes": dxc,
            "frac_of_peak": {"spec_dense_bf16_2250": value / ws / SPEC_BF16_TFLOPS,
                             "measured_burst": value / ws / pk["bf16"],
                             "measured_sustained": value / ws / pk["bf16_sus"],
                             "note": f"spec = GB300 nominal dense bf16, {SPEC_BF16_TFLOPS:.0f} TFLOP/s; measured = "
                                     f"{pk['src']} torch.matmul bf16 8192^3 on this pool ({pk['bf16']:.0f} burst, "
                                     f"{pk['bf16_sus']:.0f} sustained)"},
            "roofline": roof,
            "kernels": kern,
            "cpu_baseline": cpu,
            "e2e": {"value": flops / (e2e_ms * 1e-3) / 1e12 * ws, "unit": "TFLOP/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                    "steps": e2e_steps, "inputs": "X, dY uploaded from pinned host memory every step, "
                                                  "double-buffered on two copy streams",
                    "returned": "the updated scale and its gradient sgrad (the step's parameter update)",
                    "resident": "Y, dX and gq stay on the device: in training the next layer reads Y, the "
                                "layer before reads dX and the q-update reads gq",
                    "h2d_gbs_alone": h2d_gbs, "h2d_ms_per_step_alone": h2d / h2d_gbs / 1e6},
            "e2e_all_outputs": {"value": flops / (all_ms * 1e-3) / 1e12 * ws, "unit": "TFLOP/s",
                                "ms_per_step": all_ms, "steps": all_steps, "h2d_bytes_per_step": h2d,
                                "d2h_bytes_per_step": d2h_all,
                                "how": "X, dY uploaded, the step, then Y, dX, gq, sgrad and scale copied to pinned "
                                       "host memory, all on one stream (no overlap)"},
            "gpu_launches": launches_per_step * args.steps,
            "clocks": csum,
        }

    # The extra lines below run after the headline is complete.  Should one of them
    # stall, a watchdog prints the headline line with the stalled phase named (and
    # every thread's stack on stderr) and ends the process.
    extra = {}
    dog = Watchdog(args.extras_limit, line if rank == 0 else None, extra, bl.tern_device_diagnostics)

    def bw_loop(fn, nbytes, reps=10, warm=3):
        # the reps run as one captured CUDA graph: a short kernel (tens of microseconds)
        # would otherwise wait on the host's launch rate between reps
        return graph_bw(torch, fn, nbytes, reps, warm, stream, pk["hbm"])

    if not args.skip_bandwidth and args.workload == "large_single_projection":
        progress("AdamW and ternarise bandwidth sweeps")
        del Y
        torch.cuda.empty_cache()
        sweep = []
        n_max = 400_000_000
        w_ = torch.empty(n_max, device=dev).normal_(0, 0.02)
        g_ = torch.empty(n_max, device=dev).normal_(0, 1e-3)
        m_, v_ = torch.zeros(n_max, device=dev), torch.zeros(n_max, device=dev)
        for n_ad in (10_000, 100_000, 1_000_000, 10_000_000, 100_000_000, n_max):
            tcount = [0]

            def ad(n_ad=n_ad, tcount=tcount):
                tcount[0] += 1
                bl.adamw_step(w_[:n_ad], g_[:n_ad], m_[:n_ad], v_[:n_ad], tcount[0], **ADAM_HP)
            sweep.append(dict(n=n_ad, **bw_loop(ad, 28 * n_ad, reps=10 if n_ad > 1e7 else 50)))
        extra["adamw"] = dict(bytes_per_elem=28, **sweep[-1])
        extra["adamw_sweep"] = sweep
        # many small tensors: one multi-tensor launch against one launch per tensor
        multi = []
        sc = torch.tensor([ADAM_HP["lr"], 1 - ADAM_HP["b1"], 1 - ADAM_HP["b2"], 1.0], device=dev)
        for n_tot in (10_000, 100_000, 1_000_000):
            nt = bl.TERN_ADAM_MAX_TENSORS
            per_t = max(4, (n_tot // nt) // 4 * 4)
            sl = [slice(i * per_t, (i + 1) * per_t) for i in range(nt)]
            W, G, Mm, V = ([t[x] for x in sl] for t in (w_, g_, m_, v_))
            tot = per_t * nt
            one = bw_loop(lambda: bl.adamw_step_multi(W, G, Mm, V, sc, ADAM_HP["b1"], ADAM_HP["b2"], ADAM_HP["eps"],
                                                      ADAM_HP["wd"]), 28 * tot, reps=50)

            def each():
                for a_, b_, c_, d_ in zip(W, G, Mm, V):
                    bl.adamw_step(a_, b_, c_, d_, 1, **ADAM_HP)
            sep = bw_loop(each, 28 * tot, reps=10)
            multi.append({"n": tot, "tensors": nt, "multi_tensor": one, "one_launch_per_tensor": sep})
        extra["adamw_multi_sweep"] = multi
        del w_, g_, m_, v_
        torch.cuda.empty_cache()
        sweep = []
        for Kt, Nt in ((122, 8192), (1221, 8192), (12207, 8192), (65536, 15264)):
            qt = torch.randint(-7, 8, (Kt, Nt), dtype=torch.int8, device=dev)
            tt = bl.Tiles(Kt, Nt, packed=torch.empty((Kt, Nt // 16), dtype=torch.int32, device=dev))
            sweep.append(dict(n=Kt * Nt, **bw_loop(lambda: bl.tern_materialize(qt, None, tt, 2, 7), 1.25 * Kt * Nt,
                                                   reps=10 if Kt * Nt > 1e7 else 50)))
            del qt, tt
        extra["ternarise"] = dict(bytes_per_elem=1.25, **sweep[-1])
        extra["ternarise_sweep"] = sweep
        # the step's own materialise (all four encodings, 7.25 B per weight) timed alone as
        # graph-replayed calls: the in-step figure above also holds the launch and event gaps
        ma = bl.Tiles.empty(K, N)
        extra["materialise_all_planes_alone"] = dict(
            bytes_per_elem=7.25, n=K * N, **bw_loop(lambda: bl.tern_materialize(q, scale, ma, 2, 7), 7.25 * K * N,
                                                    reps=20))
        del ma
        torch.cuda.empty_cache()
    dog.cancel()

    if ws > 1:
        torch.distributed.destroy_process_group()
    # The other layer workloads (the RWKV-style block, the wide FFN chain) run each in a
    # fresh child process of this script, after this process's GPU work is done.
    if rank == 0 and not args.skip_workloads and args.workload == "large_single_projection":
        wl = {}
        for name in ("rwkv_block", "wide_ffn_chain"):
            progress(f"workload {name} (child process)")
            wl[name] = child_workload(name, args)
        extra["workloads"] = wl
    if rank == 0:
        line.update(extra)
        print(json.dumps(line), flush=True)
    return 0


def child_workload(name, args):
    """Run `bench.py --workload name` in a fresh process (own CUDA context) and return its
    result object; a child that does not finish within --workload-limit seconds is
    killed with its process group and reported as such."""
    cmd = [sys.executable, os.path.abspath(__file__), "--workload", name, "--steps", str(args.steps),
           "--warmup", str(args.warmup)]
    t0 = time.perf_counter()
    p = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True, start_new_session=True,
                         cwd=ROOT)
    try:
        out, err = p.communicate(timeout=args.workload_limit)
    except subprocess.TimeoutExpired:
        try:
            os.killpg(p.pid, 9)
        except OSError:
            pass
        out, err = p.communicate()
        sys.stderr.write(err[-4000:])
        return {"stalled": {"limit_s": args.workload_limit, "note": "killed; see stderr"}}
    sys.stderr.write(err)
    for ln in reversed(out.strip().splitlines()):
        try:
            d = json.loads(ln)
        except ValueError:
            continue
        if name in d:
            d[name]["wall_s"] = time.perf_counter() - t0
            return d[name]
    return {"failed": {"rc": p.returncode, "stderr_tail": err[-800:]}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="large_single_projection")
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of CPU oracle sampling")
    ap.add_argument("--skip-cpu", action="store_true")
    ap.add_argument("--skip-bandwidth", action="store_true")
    ap.add_argument("--extras-limit", type=float, default=300.0,
                    help="seconds after which the bandwidth sweeps are cut (the headline line is printed)")
    ap.add_argument("--skip-workloads", action="store_true", help="leave out the RWKV block and the FFN chain")
    ap.add_argument("--t-operand", choices=["bf16", "packed"], default="bf16",
                    help="the forward's T operand: the bf16 plane, or the 2-bit codes expanded inside the GEMM")
    ap.add_argument("--workload-limit", type=float, default=300.0,
                    help="seconds after which a child workload process is killed")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.workload == "hbm_kernels":
        return hbm_kernels(args)
    if args.workload in ("rwkv_block", "wide_ffn_chain"):
        import torch
        torch.cuda.set_device(0)
        import __graft_entry__
        __graft_entry__._builder().build()
        import bit_linear_gb300 as bl
        fn = rwkv_block if args.workload == "rwkv_block" else wide_chain
        with ClockSampler(0) as clk:
            out = fn(bl, torch.device("cuda"), torch.cuda.current_stream(), args.steps)
        out["clocks"] = clk.summary()
        print(json.dumps({args.workload: out}), flush=True)
        return 0
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
