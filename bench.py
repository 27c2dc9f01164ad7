"""Benchmark of the parallel Newton forward of the diagonal-mix GRU.

python bench.py [--gpus N] [--steps K] [--warmup W] [--workload I] [--algo A]
                [--impl ours|reference]

A step is one Newton forward over one batch of the workload: K iterations of
cell + Jacobian + residual + affine scan and the final residual gate
(nrnn_newton_forward), preactivations resident in HBM.  The default workload
is the largest single-GPU configuration (diagonal GRU, bf16 storage with fp32
math, B16 T16384 d_in = d_h = 1024, K = 3; the ragged N262144 d512 fp32 pack
moves the same bytes and is timed beside it under ``other_workloads``).  The
input projection is timed beside the forward (``with_projection``).  Prints
one JSON line on rank 0.

Under torchrun each rank runs its own replica of the workload on its own GPU
(the batch rows are independent; there is no collective on the data path):
weak scaling, value = tokens of all ranks / max over ranks of the time.

``--impl reference`` times the float64 CPU oracle's sequential unroll (the
definition the Newton forward must reproduce) on a bounded sample of the same
workload on the host cores, rank 0 only.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synthetic as syn  # noqa: E402

METRIC = "Newton forward tokens/s and achieved HBM GB/s vs GB300 peak (1 GPU)"
L2_FLUSH_BYTES = 512 << 20


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            d = json.load(fh)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d.get("bf16_tflops", 1900.0), "src": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "src": "fallback"}


def max_over_ranks(ms, world, device):
    """Slowest rank's time (all ranks call this)."""
    import torch
    if world <= 1:
        return ms
    t = torch.tensor([float(ms)], device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def tokens_all_ranks(tokens_per_rank, world):
    """Weak scaling: every rank runs a full replica of the workload."""
    return tokens_per_rank * world


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            if self.thread is not None:
                self.thread.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


def workload_bytes(w, algo):
    """Algorithmic HBM bytes per launch of one Newton forward."""
    s = 2 if w.dtype == "bf16" else 4
    tok = w.B * w.T
    if algo == "per_iter":
        # iteration 1: read P, write H; later ones: read P and H^(k-1), write H^(k);
        # the last launch evaluates the residual in-kernel (no extra pass)
        return [4 * w.d_h * s * tok] + [5 * w.d_h * s * tok] * (w.K - 1)
    return [4 * w.d_h * s * tok]          # fused: read P once, write H once


# Special-function (MUFU) work per cell evaluation in the Newton kernels: for
# fp32 storage three ex2 (one per gate) and two rcp (one for r, one shared by
# z and the tanh); for bf16 storage three tanh.approx.  The roof is the SM's
# measured MUFU rate (nrnn_probe_xu_rates, run live): an rcp or tanh occupies
# the unit for ex2_rate / its rate ex2 slots, so the work is counted in
# ex2-equivalent operations.
MUFU_PER_EVAL = {"f32": {"ex2": 3, "rcp": 2}, "bf16": {"tanh": 3}}
SM_MAX_MHZ = 2070.0
DEFAULT_WORKLOAD = 3
CPU_SAMPLE_BYTES = 256 << 20


def mhz_of(clocks):
    return clocks.get("sm_mhz") or clocks.get("sm_max_mhz") or SM_MAX_MHZ


def xu_work(w, rates):
    """ex2-equivalent MUFU operations of one fused forward."""
    mix = MUFU_PER_EVAL[w.dtype]
    per_eval = sum(n * rates["ex2"] / rates[op] for op, n in mix.items())
    return per_eval * (w.K + 1) * w.B * w.T * w.d_h


def segments_of(inp):
    """Segments of a workload's cu_seqlens pack (0: no pack): the workspace then
    has room for segment-aligned chunks."""
    return 0 if inp["cu_seqlens"] is None else len(inp["cu_seqlens"]) - 1


def time_workload(torch, nr, w, args, dev, flush, stream, xu_rates, props, mhz):
    """Fused and per-iteration forward of workload w (CUDA-graph replays, L2
    flushed between steps): ms, tokens/s, the fused kernel's MUFU fraction and
    the per-iteration kernel's HBM fraction."""
    P = syn.preact_uniform_torch(w, device=dev)
    inp = syn.make_inputs(w, with_x=False)
    prm = nr.params_tensor(inp["params"], w.d_h, dev)
    cu = None if inp["cu_seqlens"] is None else nr.DeviceCuSeqlens(inp["cu_seqlens"], w.T, dev)
    tdt = P.dtype
    H = torch.empty((w.B, w.T, w.d_h), dtype=tdt, device=dev)
    ws = torch.empty(max(nr.workspace_bytes(w.B, w.T, w.d_h, tdt, w.K, a, num_segments=segments_of(inp))
                         for a in ("fused", "per_iter")),
                     dtype=torch.uint8, device=dev)
    res = {"B": w.B, "T": w.T, "d_h": w.d_h, "K": w.K, "dtype": w.dtype,
           "input": "preact drawn directly, U(-1, 1)"}
    rates = dict(zip(("ex2", "rcp", "tanh"), xu_rates))
    pk = peaks()
    for algo in ("fused", "per_iter"):
        def call(a=algo):
            return nr.newton_forward(P, prm, cu_seqlens=cu, K=w.K, algo=a, check=False, out=H,
                                     workspace=ws)
        call()
        torch.cuda.synchronize()
        if args.graph:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                call()
            step = g.replay
        else:
            step = call
        for _ in range(args.warmup):
            flush()
            step()
        ms_l, _ = time_steps(torch, step, max(3, min(args.steps, 10)), flush, stream, nvtx=False)
        ms = sum(ms_l) / len(ms_l)
        entry = {"ms": ms, "tokens_per_s": w.B * w.T / (ms * 1e-3)}
        if algo == "fused":
            peak = rates["ex2"] * props.multi_processor_count * mhz * 1e6 / 1e9
            entry["alu_frac"] = xu_work(w, rates) / (ms * 1e-3) / 1e9 / peak
            entry["hbm_frac"] = sum(workload_bytes(w, algo)) / (ms * 1e-3) / 1e9 / pk["hbm_gbs"]
        else:
            b = workload_bytes(w, algo)
            entry["hbm_frac"] = (sum(b) / len(b)) / (ms / len(b) * 1e-3) / 1e9 / pk["hbm_gbs"]
        res[algo] = entry
    if not args.skip_routes:
        res["routes_to_tau"] = routes_to_tau(torch, nr, w, P, prm, cu, args, flush, stream)
    del P, H, ws
    return res


def time_graph(torch, fn, args, flush, stream):
    """Median ms of fn as a CUDA-graph replay (eager launches with --no-graph),
    L2 flushed between steps."""
    fn()
    torch.cuda.synchronize()
    step = fn
    if args.graph:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        step = g.replay
    for _ in range(args.warmup):
        flush()
        step()
    ms, _ = time_steps(torch, step, max(3, min(args.steps, 10)), flush, stream, nvtx=False)
    return statistics.median(ms)


def routes_to_tau(torch, nr, w, P, prm, cu, args, flush, stream):
    """Two routes past the configured K's method error (FAQs, "How many Newton
    iterations should I use?"): one more Newton iteration, or two Picard
    sweeps and then K Newton iterations from their result.  ms of each; their
    max-abs against the float64 unroll is checked by the GPU tests."""
    H = torch.empty((w.B, w.T, w.d_h), dtype=P.dtype, device=P.device)
    k1 = time_graph(torch, lambda: nr.newton_forward(P, prm, cu_seqlens=cu, K=w.K + 1,
                                                     check=False, out=H), args, flush, stream)
    pk = time_graph(torch, lambda: nr.newton_forward(P, prm, cu_seqlens=cu, K=w.K, check=False,
                                                     out=H, picard_iters=2), args, flush, stream)
    return {f"newton_K{w.K + 1}_ms": k1, f"picard2_newton_K{w.K}_ms": pk}


def bench_config(w, args, world):
    """The workload and launch configuration (identical in both arms' lines)."""
    return {"workload": w.name, "B": w.B, "T": w.T, "d_in": w.d_in, "d_h": w.d_h,
            "K": w.K, "segments": w.segments, "algo": args.algo,
            "parallelism": f"replica x{world}",
            "launch": "CUDA graph replay of one forward" if args.graph else "eager launches",
            "l2": f"flushed between steps ({L2_FLUSH_BYTES >> 20} MiB write, then "
                  f"{L2_FLUSH_BYTES >> 20} MiB read; untimed)"}


class L2Flush:
    """Empties L2 between timed steps, outside the timed region: writes a buffer
    larger than L2, then reads another one, so that the step starts with a
    cold L2 holding clean lines only (dirty lines of the write alone would be
    written back during the timed step)."""

    def __init__(self, torch, dev):
        self.torch = torch
        self.w = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        self.r = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        self.out = torch.empty((), dtype=torch.float32, device=dev)

    def __call__(self):
        self.w.fill_(1.0)
        self.torch.sum(self.r, 0, out=self.out)


def time_steps(torch, fn, steps, flush, stream, nvtx=True):
    """Per-step device time (ms) with CUDA events; L2 flushed between steps, untimed."""
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    out = None
    for i in range(steps):
        flush()
        if nvtx:
            torch.cuda.nvtx.range_push("nrnn_step")
        ev[i][0].record(stream)
        out = fn()
        ev[i][1].record(stream)
        if nvtx:
            torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in ev], out


def run_ours(args, w, rank, world, local):
    import torch
    import nonlinear_rnn_gb300 as nr

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    props = torch.cuda.get_device_properties(dev)
    inp = syn.make_inputs(w)
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    x = torch.from_numpy(inp["x"]).to(dev).to(tdt)
    W = torch.from_numpy(inp["W_x"]).to(dev).to(tdt)
    prm = nr.params_tensor(inp["params"], w.d_h, dev)
    cu = None if inp["cu_seqlens"] is None else nr.DeviceCuSeqlens(inp["cu_seqlens"], w.T, dev)
    P = nr.input_projection(x, W)
    H = torch.empty((w.B, w.T, w.d_h), dtype=tdt, device=dev)
    algo = args.algo
    ws = torch.empty(max(nr.workspace_bytes(w.B, w.T, w.d_h, tdt, w.K, a, num_segments=segments_of(inp))
                         for a in ("fused", "per_iter")),
                     dtype=torch.uint8, device=dev)
    flush = L2Flush(torch, dev)
    stream = torch.cuda.current_stream(dev)

    def newton_call(a=algo):
        return nr.newton_forward(P, prm, cu_seqlens=cu, K=w.K, algo=a, check=False,
                                 out=H, workspace=ws)

    def graphed(a):
        """The forward (the per-call clear kernel + the Newton kernels) captured once as a
        CUDA graph."""
        newton_call(a)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            res = newton_call(a)
        return lambda: (g.replay(), res)[1]

    newton = graphed(algo) if args.graph else newton_call

    def replay_of(fn):
        """fn captured once as a CUDA graph (so that the timed region holds the
        device work, not the binding's host-side argument handling)."""
        if not args.graph:
            return fn
        fn()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        return g.replay
    xu_rates = nr.probe_xu_rates(dev)   # live denominator of the fused kernel's ALU roof

    for _ in range(args.warmup):
        flush()
        newton()
    torch.cuda.synchronize()

    with ClockSampler(local) as clk:
        # keep the GPU busy while the sampler starts, so that its samples cover
        # the load the timed steps run under (untimed)
        t_pre = time.perf_counter()
        while time.perf_counter() - t_pre < args.preroll_s:
            for _ in range(20):
                flush()
                newton()
            torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        t_wall = time.perf_counter()
        step_ms, (_, rho) = time_steps(torch, newton, args.steps, flush, stream)
        t_wall = time.perf_counter() - t_wall
    ms = max_over_ranks(sum(step_ms) / len(step_ms), world, dev)
    if world > 1:
        torch.distributed.barrier()

    tokens = w.B * w.T
    pk = peaks()
    clocks = clk.summary()
    fused = algo != "per_iter"
    byts = workload_bytes(w, algo)
    launches = len(byts) if w.K > 0 else 1
    per_launch_ms = ms / launches
    hbm_achieved = (sum(byts) / len(byts)) / (per_launch_ms * 1e-3) / 1e9
    kname = "k_newton<%s,%s>" % ("bf16" if w.dtype == "bf16" else "float",
                                 "fused" if fused else "per_iter")
    hbm = {"bound": "hbm", "achieved": hbm_achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
           "frac": hbm_achieved / pk["hbm_gbs"], "traffic": load_traffic(w, algo),
           "kernel": kname, "algorithmic_bytes_per_launch": sum(byts) / len(byts),
           "peak_src": pk["src"] + " (MEASURED_PEAKS.json hbm_gbs)"}
    if fused:
        # one launch runs K iterations plus the residual evaluation
        rates = dict(zip(("ex2", "rcp", "tanh"), xu_rates))
        mix = MUFU_PER_EVAL[w.dtype]
        per_eval = sum(n * rates["ex2"] / rates[op] for op, n in mix.items())
        ex2_rate = rates["ex2"]
        xu_ops = per_eval * (w.K + 1) * tokens * w.d_h
        xu_achieved = xu_ops / (ms * 1e-3) / 1e9
        # the SM clock the timed steps ran at (median of the samples taken
        # during them), else the maximum clock
        mhz = clocks.get("sm_mhz") or clocks.get("sm_max_mhz") or SM_MAX_MHZ
        xu_peak = ex2_rate * props.multi_processor_count * mhz * 1e6 / 1e9
        roof = {"bound": "alu", "achieved": xu_achieved, "peak": xu_peak,
                "unit": "Gop/s (MUFU, ex2-equivalent)",
                "frac": xu_achieved / xu_peak, "traffic": load_traffic(w, algo), "kernel": kname,
                "algorithmic_ops_per_launch": xu_ops,
                "peak_src": "measured " + ", ".join(f"{rates[k]:.2f} {k}" for k in rates)
                            + f" results/clk/SM (nrnn_probe_xu_rates) x {props.multi_processor_count} "
                            f"SMs x {mhz:.0f} MHz (median sampled SM clock); per evaluation "
                            + " + ".join(f"{n} {op}" for op, n in mix.items()),
                "hbm": {k: hbm[k] for k in ("achieved", "peak", "unit", "frac",
                                            "algorithmic_bytes_per_launch")}}
    else:
        roof = hbm

    # the per-iteration kernel's HBM roofline, timed the same way
    per_iter = None
    if fused and w.K > 0 and not args.skip_per_iter:
        per_iter_step = graphed("per_iter") if args.graph else (lambda: newton_call("per_iter"))
        for _ in range(args.warmup):
            per_iter_step()
        pms, _ = time_steps(torch, per_iter_step, args.steps, flush, stream, nvtx=False)
        pb = workload_bytes(w, "per_iter")
        pl = (sum(pms) / len(pms)) / len(pb)
        pa = (sum(pb) / len(pb)) / (pl * 1e-3) / 1e9
        per_iter = {"bound": "hbm", "achieved": pa, "peak": pk["hbm_gbs"], "unit": "GB/s",
                    "frac": pa / pk["hbm_gbs"], "ms_per_step": sum(pms) / len(pms),
                    "launches_per_step": len(pb), "traffic": load_traffic(w, "per_iter"),
                    "kernel": kname.replace("fused", "per_iter"),
                    "algorithmic_bytes_per_launch": sum(pb) / len(pb)}

    # projection and the GPU sequential unroll beside it
    pws = torch.empty(max(1, nr.projection_workspace_bytes(tdt, w.d_in, w.d_h)), dtype=torch.uint8,
                      device=dev)
    proj_ms, _ = time_steps(torch, replay_of(lambda: nr.input_projection(x, W, out=P, workspace=pws)),
                            max(3, min(args.steps, 10)),
                            flush, stream, nvtx=False)
    seq_ms, _ = time_steps(torch, replay_of(lambda: nr.sequential_forward(P, prm, cu_seqlens=cu, out=H)), 3,
                           flush, stream, nvtx=False)

    # end to end through the C-ABI calls on host buffers, copies overlapped
    # block by block (blocks of rows or segments) with the kernels:
    # nrnn_newton_forward_x_host takes x (W_x resident on the device, each
    # block projected there), nrnn_newton_forward_host the preactivations
    x_host = x.cpu().pin_memory()
    P_host = P.cpu().pin_memory()
    H_host = torch.empty(H.shape, dtype=H.dtype).pin_memory()
    cu_host = None if inp["cu_seqlens"] is None else inp["cu_seqlens"]
    staging = torch.empty(max(nr.x_host_staging_bytes(w.B, w.T, w.d_in, w.d_h, tdt, w.K, cu_seqlens=cu_host),
                              nr.host_staging_bytes(w.B, w.T, w.d_h, tdt, w.K, cu_seqlens=cu_host)),
                          dtype=torch.uint8, device=dev)

    def e2e_x_step():
        nr.newton_forward_x_host(x_host, W, prm, cu_seqlens=cu_host, K=w.K, out=H_host,
                                 staging=staging, check=False)

    def e2e_p_step():
        nr.newton_forward_host(P_host, prm, cu_seqlens=cu_host, K=w.K, out=H_host,
                               staging=staging, device=dev, check=False)
    e2e_ms = {}
    for name, fn in (("x", e2e_x_step), ("preact", e2e_p_step)):
        fn()
        t_e2e, _ = time_steps(torch, fn, max(3, min(args.steps, 10)), flush, stream, nvtx=False)
        e2e_ms[name] = statistics.median(t_e2e)
    del P_host, x_host

    proj = statistics.median(proj_ms)

    # NEXT rows, each against the HBM roof: the backward (adjoint) scan at the
    # forward's trajectory (reads P, H, dL/dH, writes dL/dP: 8 d_h s bytes per
    # token) and one decode step for a batch of slots (reads P and h, writes h':
    # 5 d_h s per slot; fused projection: x and h in, h' out, W_x once)
    s_el = 2 if w.dtype == "bf16" else 4
    nxt = {}
    if not args.skip_next:
        gH = H.clone()
        bw_ms, _ = time_steps(torch, replay_of(lambda: nr.newton_backward(P, prm, H, gH, cu_seqlens=cu)), 3,
                              flush, stream, nvtx=False)
        bw = statistics.median(bw_ms)
        bw_bytes = 8 * w.d_h * s_el * tokens
        nxt["backward"] = {"ms": bw, "bytes": bw_bytes, "achieved_gbs": bw_bytes / (bw * 1e-3) / 1e9,
                           "frac": bw_bytes / (bw * 1e-3) / 1e9 / pk["hbm_gbs"]}
        del gH
        # two Picard sweeps (the warm start of NEXT row f1): P read twice, G written
        # twice, read once: 9 d_h s bytes per token
        Gp = torch.empty_like(H)
        pc_ms, _ = time_steps(torch, replay_of(lambda: nr.picard(P, prm, 2, cu_seqlens=cu, out=Gp)), 3,
                              flush, stream, nvtx=False)
        pc = statistics.median(pc_ms)
        pc_bytes = 9 * w.d_h * s_el * tokens
        nxt["picard2"] = {"ms": pc, "bytes": pc_bytes, "achieved_gbs": pc_bytes / (pc * 1e-3) / 1e9,
                          "frac": pc_bytes / (pc * 1e-3) / 1e9 / pk["hbm_gbs"]}
        del Gp
        def decode_leg(name, slots, with_x):
            Pd = P.reshape(-1, 3 * w.d_h)[:slots]
            hd = H.reshape(-1, w.d_h)[:slots]
            xd = x.reshape(-1, w.d_in)[:slots]
            hout = torch.empty_like(hd)
            if with_x:   # W_x read once; x and h in, h' out
                fn = lambda: nr.decode_step(prm, hd, x=xd, W_x=W, out=hout)
                nbytes = (w.d_in + 2 * w.d_h) * s_el * slots + 3 * w.d_h * w.d_in * s_el
            else:
                fn = lambda: nr.decode_step(prm, hd, preact=Pd, out=hout)
                nbytes = 5 * w.d_h * s_el * slots
            dms, _ = time_steps(torch, replay_of(fn), 5, flush, stream, nvtx=False)
            dm = statistics.median(dms)
            nxt[name] = {"slots": slots, "ms": dm, "bytes": nbytes,
                         "achieved_gbs": nbytes / (dm * 1e-3) / 1e9,
                         "frac": nbytes / (dm * 1e-3) / 1e9 / pk["hbm_gbs"]}
            if with_x:
                # the step's projection x W_x^T is a GEMM of 2 slots 3 d_h d_in
                # flops: against the tensor roof of the storage type (bf16
                # measured; fp32 runs three TF32 products at half that rate)
                flops = 2.0 * slots * 3 * w.d_h * w.d_in * (3 if w.dtype == "f32" else 1)
                tf = pk["bf16_tflops"] * (0.5 if w.dtype == "f32" else 1.0)
                nxt[name]["tensor"] = {"flops": flops, "achieved_tflops": flops / (dm * 1e-3) / 1e12,
                                       "peak_tflops": tf, "frac": flops / (dm * 1e-3) / 1e12 / tf}

        # a step for every token of the workload as a slot (P and h far larger
        # than L2: the kernel's bandwidth), then the batch sizes of serving;
        # small steps sit near the event-timing floor of a few microseconds
        decode_leg("decode_all_tokens", tokens, False)
        big = min(8192, tokens)
        decode_leg("decode", big, False)
        decode_leg("decode_x", big, True)                       # projection, then the step
        decode_leg("decode_x_small", min(64, tokens), True)     # fused kernel

    # bf16: the projection fused into the Newton kernel (P never written)
    fused_x = None
    if w.dtype == "bf16" and w.K > 0:
        def fx():
            return nr.newton_forward_x(x, W, prm, cu_seqlens=cu, K=w.K, check=False, out=H,
                                       workspace=ws)
        fx()
        torch.cuda.synchronize()
        if args.graph:
            gx = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gx):
                fx()
            fx_step = gx.replay
        else:
            fx_step = fx
        for _ in range(args.warmup):
            fx_step()
        fx_ms, _ = time_steps(torch, fx_step, max(3, min(args.steps, 10)), flush, stream, nvtx=False)
        fused_x = {"ms": statistics.median(fx_ms),
                   "tokens_per_s": tokens * world / (statistics.median(fx_ms) * 1e-3)}
    routes = None if args.skip_routes else routes_to_tau(torch, nr, w, P, prm, cu, args, flush,
                                                         stream)

    # the other multi-megabyte workloads, timed the same way on preactivations
    # drawn directly on the device (U(-1, 1), the variance of x W_x^T)
    others = {}
    if not args.skip_others:
        for oi in args.others:
            if oi == args.workload:
                continue
            others[syn.WORKLOADS[oi].name] = time_workload(
                torch, nr, syn.WORKLOADS[oi], args, dev, flush, stream, xu_rates, props, mhz_of(clocks))

    out = {
        "metric": METRIC,
        "value": tokens_all_ranks(tokens, world) / (ms * 1e-3),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": w.dtype,
        "data": "synthetic (seeded SplitMix64: x~N(0,1), W_x~U(+-1/sqrt(d_in)), a~U(+-1), b=0)",
        "config": bench_config(w, args, world),
        "roofline": roof,
        "per_iter_roofline": per_iter,
        "e2e": {"value": tokens * world / (e2e_ms["x"] * 1e-3), "unit": "tokens/s",
                "h2d_bytes_per_step": x.numel() * x.element_size(),
                "d2h_bytes_per_step": H.numel() * H.element_size() + 4,
                "ms_per_step": e2e_ms["x"],
                "call": "nrnn_newton_forward_x_host (x on the host, W_x on the device, "
                        "projection and forward per block)",
                "from_preactivations": {
                    "value": tokens * world / (e2e_ms["preact"] * 1e-3), "unit": "tokens/s",
                    "h2d_bytes_per_step": P.numel() * P.element_size(),
                    "d2h_bytes_per_step": H.numel() * H.element_size() + 4,
                    "ms_per_step": e2e_ms["preact"], "call": "nrnn_newton_forward_host"}},
        # per step: the clear kernel of the call's workspace, then the Newton launch(es)
        "gpu_launches": (launches + 1) * args.steps,
        "with_projection": {"projection_ms": proj,
                            "tokens_per_s": tokens * world / ((ms + proj) * 1e-3),
                            "fused_in_kernel": fused_x},
        "sequential_gpu": {"ms": statistics.median(seq_ms),
                           "tokens_per_s": tokens / (statistics.median(seq_ms) * 1e-3)},
        "next_rows": nxt or None,
        "routes_to_tau": routes,
        "other_workloads": others or None,
        "residual": float(rho.item()),
        "wall_s": t_wall,
        "clocks": clocks,
    }
    return out


# Sources whose change invalidates the recorded DRAM counters of the Newton kernel.
TRAFFIC_SOURCES = ("nonlinear_rnn_gb300/csrc/newton.cu", "nonlinear_rnn_gb300/csrc/nrnn_device.cuh",
                   "nonlinear_rnn_gb300/csrc/nrnn_internal.h")


def kernel_sources_digest():
    import hashlib
    h = hashlib.sha256()
    for rel in TRAFFIC_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def load_traffic(w, algo):
    """DRAM bytes per launch of the dominant kernel from the committed ncu summary,
    or None when there is none or the kernel sources changed since it was taken."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as fh:
        d = json.load(fh)
    if d.get("_kernel_sources_sha256") != kernel_sources_digest():
        return None
    return d.get(f"{w.name}|{algo}")


def cpu_baseline(w, budget_s=10.0, steps=1):
    """Times the float64 oracle's sequential unroll h_t = f(h_{t-1}, P_t) (the
    definition the Newton forward must reproduce; numerics contract,
    "Invariant") as it stands, on all host cores, on a bounded sample of the
    workload: whole rows of T steps (every segment of a pack, each from h = 0)
    for a subset of hidden units, which are independent, as many rows and
    units as fit in about budget_s per pass.  Returns tokens/s scaled to full
    tokens (d_h units per token)."""
    import oracle

    cores = os.cpu_count() or 1
    inp = syn.make_inputs(w, with_x=False)
    prm = oracle.pack_params(inp["params"])
    cu = inp["cu_seqlens"]
    n0 = min(w.d_h, cores)
    units = np.arange(n0)
    Pc = syn.preact_uniform_columns(w, units, rows=[0]).astype(np.float64)
    t = time.perf_counter()
    oracle.sequential(Pc, prm[:, units], cu_seqlens=cu, threads=cores)
    t_unit_row = max(time.perf_counter() - t, 1e-4)     # one unit per core, one row
    waves = lambda n: -(-n // cores)                      # noqa: E731
    # sample: whole rows, at most SAMPLE_BYTES of float64 preactivations
    n_units, n_rows = w.d_h, w.B
    fits = lambda nu, nr: (t_unit_row * waves(nu) * nr <= budget_s and        # noqa: E731
                           nu * nr * w.T * 3 * 8 <= CPU_SAMPLE_BYTES)
    while n_rows > 1 and not fits(n_units, n_rows):
        n_rows -= 1
    while n_units > 1 and not fits(n_units, n_rows):
        n_units = max(1, n_units // 2)
    units = np.arange(n_units)
    rows = list(range(n_rows))
    Pc = syn.preact_uniform_columns(w, units, rows=rows).astype(np.float64)
    pp = prm[:, units]
    reps = max(1, int(budget_s / max(t_unit_row * waves(n_units) * n_rows, 1e-3)))
    threads = min(cores, n_units)
    times = []
    for _ in range(steps):
        t = time.perf_counter()
        for _ in range(reps):
            oracle.sequential(Pc, pp, cu_seqlens=cu, threads=threads)
        times.append((time.perf_counter() - t) / reps)
    sec = statistics.mean(times)
    unit_tokens = n_units * n_rows * w.T
    return {"value": unit_tokens / w.d_h / sec, "unit": "tokens/s", "cores": threads,
            "kind": "oracle",
            "sample": f"oracle.sequential (float64 unroll) on {n_units} of {w.d_h} units x "
                      f"{n_rows} of {w.B} rows x T={w.T} (uniform preact), {threads} threads, "
                      f"{sec:.3f} s per pass, {reps} passes per step",
            "seconds": sec}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", type=int, default=DEFAULT_WORKLOAD)
    ap.add_argument("--algo", default="auto", choices=["auto", "fused", "per_iter"])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--preroll-s", type=float, default=1.0)
    ap.add_argument("--skip-next", action="store_true",
                    help="skip the backward and decode legs")
    ap.add_argument("--skip-per-iter", action="store_true")
    ap.add_argument("--skip-routes", action="store_true",
                    help="skip the K+1 and Picard-warm-start timings")
    ap.add_argument("--skip-others", action="store_true",
                    help="skip the fused / per-iteration timings of the other workloads")
    ap.add_argument("--others", type=int, nargs="*", default=[1, 2, 3, 4],
                    help="workloads timed under other_workloads (the headline one is skipped)")
    ap.add_argument("--no-graph", dest="graph", action="store_false",
                    help="launch each forward eagerly instead of replaying a CUDA graph")
    ap.add_argument("--batch", type=int, default=0,
                    help="override the workload's batch rows (smaller profiling captures)")
    ap.add_argument("--segments", type=int, default=0,
                    help="pack workloads: that many segments over proportionally fewer tokens "
                         "(smaller profiling captures)")
    args = ap.parse_args()
    w = syn.WORKLOADS[args.workload]
    if args.batch > 0:
        import dataclasses
        w = dataclasses.replace(w, B=args.batch, name=w.name.replace(f"B{w.B} ", f"B{args.batch} "))
    if args.segments > 0 and w.segments > 0:
        import dataclasses
        T = w.T * args.segments // w.segments
        w = dataclasses.replace(w, T=T, segments=args.segments,
                                name=w.name.replace(f"N{w.T} S{w.segments} ", f"N{T} S{args.segments} "))
    rank, world, local = dist_env()

    if args.impl == "reference":
        if rank != 0:
            return
        cb = cpu_baseline(w, budget_s=max(1.0, 60.0 / max(args.steps, 1)), steps=args.steps)
        out = {"impl": "reference", "metric": METRIC, "value": cb["value"], "unit": "tokens/s",
               "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
               "ms_per_step": 1e3 * w.B * w.T / cb["value"], "higher_is_better": True,
               "scaling": "weak", "vs_baseline": None, "dtype": "f64",
               "data": "synthetic (seeded SplitMix64)",
               "config": bench_config(w, args, world),
               "cpu_baseline": {k: cb[k] for k in ("value", "unit", "cores", "kind", "sample")},
               "e2e": {"value": cb["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                       "d2h_bytes_per_step": 0}}
        print(json.dumps(out))
        return

    import torch
    if world > 1:
        torch.distributed.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    out = run_ours(args, w, rank, world, local)
    if rank == 0 and not args.no_cpu_baseline:
        cb = cpu_baseline(w)
        out["cpu_baseline"] = {k: cb[k] for k in ("value", "unit", "cores", "kind", "sample")}
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
    if rank == 0:
        print(json.dumps(out))


if __name__ == "__main__":
    main()
