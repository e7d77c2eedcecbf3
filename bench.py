"""Benchmark of the NVFP4 quantizer hot path on one GB300 (or N replicas).

A step is one pass of the whole hot path over one tensor: nvfp4_amax (tensor
amax per copy) then nvfp4_quantize (scale, round, pack; rowwise + transposed
columnwise outputs).  The default workload is the recipe's activation tensor,
8192 x 5120 bf16 with outlier channels, 4/6 with MAE selection, both copies.

Metric: NVFP4 quantize GB/s = (bf16 bytes read + code bytes + scale bytes
written) per step / step time.  The timed steps rotate over several input and
output sets whose combined size exceeds the L2, so every step reads from HBM.
The roofline entry is for the dominant kernel (quantize), timed with CUDA
events on its own stream inside the same rotating stream of steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]
  python bench.py --report | --error-analysis | --once

Under torchrun (N > 1) every rank runs an independent replica (the path needs
no exchange for independent tensors) and rank 0 prints the JSON line with the
max step time over ranks.  --impl reference times the CPU oracle on the host
cores instead (a bounded row sample of the same workload).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synthetic  # noqa: E402

METRIC = "NVFP4 quantize GB/s (bf16 in + fp4/scales out), % of GB300 HBM peak"
UNIT = "GB/s"


# DRAM bytes (read + written) of one quantize launch, from one ncu capture of
# the current kernel on that workload (cold cache; outputs partly still in L2
# at kernel end).  Keyed by (workload, flags, selection); absent -> null.
QUANTIZE_TRAFFIC_BYTES = {
    ("act_46mae_8192x5120", 67, 0): 83_940_864 + 10_233_856,
}


def max_over_ranks(value: float, world: int, device=None) -> float:
    """The largest `value` over all ranks (the slowest rank sets the job time)."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def algorithmic_bytes(M: int, N: int, flags: int) -> int:
    """bf16 read + per copy (codes N*M/2 + scales N*M/16)."""
    copies = (1 if flags & 1 else 0) + (1 if flags & 2 else 0)
    return 2 * M * N + copies * (M * N // 2 + M * N // 16)


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 50 ms."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            out, _ = self.proc.communicate(timeout=5)
            self.lines = [ln for ln in out.splitlines() if ln.strip()]
        return False

    def summary(self, skip_first: bool = True):
        """Median SM clock and the throttle reasons seen; the first reading
        (taken as the sampler starts, before the load) is left out."""
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines[1 if skip_first else 0:]:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax = float(f[2])
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


def run_ours(args, rank: int, world: int):
    import torch
    import torch.distributed as dist

    import nvfp4_bit_block_gb300 as nv

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    nv.build() if rank == 0 else None
    if world > 1:
        dist.barrier()
    nv.lib()
    flags, sel = workload_config(args)
    bits = synthetic.workload(args.workload)
    M, N = bits.shape
    x_host = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).pin_memory()
    # Several input/output sets used in rotation, so that the bytes touched
    # between two uses of the same set exceed the 129 MB L2: every step reads
    # its input from HBM and the previous steps' outputs are written back
    # during later steps, as in a steady stream of tensors.
    per_set = algorithmic_bytes(M, N, flags)
    nsets = max(2, -(-3 * 128 * 2**20 // per_set))
    stream = torch.cuda.Stream(device=dev)
    xs = [x_host.to(dev) for _ in range(nsets)]
    amaxs = [torch.empty(2, dtype=torch.float32, device=dev) for _ in range(nsets)]
    outs = [nv.nvfp4_quantize(xs[i], nv.nvfp4_amax(xs[i], flags, synthetic.RHT_SEED), flags, sel)
            for i in range(nsets)]
    torch.cuda.synchronize()
    x, amax, out = xs[0], amaxs[0], outs[0]

    def step(i):
        nv.nvfp4_amax(xs[i], flags, synthetic.RHT_SEED, out=amaxs[i], stream=stream)
        nv.nvfp4_quantize(xs[i], amaxs[i], flags, sel, synthetic.SR_SEED, synthetic.RHT_SEED, 0, out=outs[i],
                          stream=stream)

    with torch.cuda.stream(stream):
        for k in range(max(args.warmup, nsets)):
            step(k % nsets)
    torch.cuda.synchronize()

    # the step (amax then quantize) as one CUDA graph per set: no host launch gaps
    graphs = []
    for i in range(nsets):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            step(i)
        graphs.append(g)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for k in range(args.warmup):
            graphs[k % nsets].replay()
    torch.cuda.synchronize()

    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    # the timed steps last milliseconds, shorter than the sampling interval, so
    # the sampler also covers an untimed half second of the same steps run
    # right before them: the clocks reported are the clocks under this load
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for k in range(max(1, 2 * nsets)):
            graphs[k % nsets].replay()
    torch.cuda.synchronize()
    per_step_s = max((time.perf_counter() - t0) / max(1, 2 * nsets), 1e-6)
    load_steps = int(min(20000, max(1, 0.5 / per_step_s)))
    with ClockSampler(dev.index) as clocks:
        time.sleep(0.06)  # the sampler's first reading precedes the load
        with torch.cuda.stream(stream):
            for k in range(load_steps):
                graphs[k % nsets].replay()
            ev0.record(stream)
            for k in range(args.steps):
                graphs[k % nsets].replay()
            ev1.record(stream)
        torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    total_ms = max_over_ranks(ev0.elapsed_time(ev1), world, dev)

    # per-kernel durations inside the same rotating stream of steps, launched
    # directly with an event between the two kernels, for the roofline of the
    # dominant kernel
    kev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    with torch.cuda.stream(stream):
        for k in range(args.steps):
            i = k % nsets
            kev[k][0].record(stream)
            nv.nvfp4_amax(xs[i], flags, synthetic.RHT_SEED, out=amaxs[i], stream=stream)
            kev[k][1].record(stream)
            nv.nvfp4_quantize(xs[i], amaxs[i], flags, sel, synthetic.SR_SEED, synthetic.RHT_SEED, 0, out=outs[i],
                              stream=stream)
            kev[k][2].record(stream)
    torch.cuda.synchronize()
    amax_ms = [e[0].elapsed_time(e[1]) for e in kev]
    quant_ms = [e[1].elapsed_time(e[2]) for e in kev]
    for o in outs:
        status = int(o.status.item())
        assert status == 0, f"quantize reported status {status}"

    # End to end through the public API: every step copies its input from
    # pinned host memory to the device, runs amax + quantize and copies all
    # outputs back to pinned host memory.  Steps are pipelined the way a
    # stream of tensors would be: copy-in, compute and copy-out run on their
    # own streams, ordered by events, over two device buffer sets (the input
    # and output of set i are reused two steps later).
    e2e_steps = max(4, min(args.steps, 12))
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    dev_outs = [[t_ for t_ in (o.q_row, o.s_row, o.q_col, o.s_col, o.alpha) if t_ is not None] for o in outs[:2]]
    host_outs = [[torch.empty(t_.shape, dtype=t_.dtype, pin_memory=True) for t_ in d] for d in dev_outs]
    x_hosts = [x_host, x_host.clone().pin_memory()]
    ev_in = [torch.cuda.Event() for _ in range(e2e_steps + 2)]
    ev_comp = [torch.cuda.Event() for _ in range(e2e_steps + 2)]
    ev_out = [torch.cuda.Event() for _ in range(e2e_steps + 2)]
    torch.cuda.synchronize()

    def e2e_step(k):
        i = k % 2
        with torch.cuda.stream(s_in):
            if k >= 2:
                s_in.wait_event(ev_comp[k - 2])     # set i's input no longer read
            xs[i].copy_(x_hosts[i], non_blocking=True)
            ev_in[k].record(s_in)
        with torch.cuda.stream(stream):
            stream.wait_event(ev_in[k])
            if k >= 2:
                stream.wait_event(ev_out[k - 2])    # set i's outputs copied out
            step(i)
            ev_comp[k].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_comp[k])
            for h, d in zip(host_outs[i], dev_outs[i]):
                h.copy_(d, non_blocking=True)
            ev_out[k].record(s_out)

    for k in range(2):
        e2e_step(k)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for k in range(2, 2 + e2e_steps):
        e2e_step(k)
    torch.cuda.synchronize()
    e2e_s = (time.perf_counter() - t0) / e2e_steps
    d2h = sum(t_.numel() * t_.element_size() for t_ in dev_outs[0])

    nbytes = algorithmic_bytes(M, N, flags)
    value = nbytes * args.steps / (total_ms * 1e-3) / 1e9 * world
    peak, peak_kind = measured_peaks()
    quant_avg_ms = statistics.mean(quant_ms)
    achieved = nbytes / (quant_avg_ms * 1e-3) / 1e9
    res = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(total_ms / args.steps, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16->nvfp4 (fp32 arithmetic)",
        "data": "synthetic",
        "config": {"workload": args.workload, "M": M, "N": N, "flags": flags, "selection": sel,
                   "elements": M * N, "bytes_per_step": nbytes,
                   "l2": f"inputs larger than L2: {nsets} input/output sets of {per_set / 1e6:.0f} MB in rotation",
                   "parallelism": f"replicas{world}" if world > 1 else "single GPU"},
        "kernels_ms": {"amax": round(statistics.mean(amax_ms), 5), "quantize": round(quant_avg_ms, 5)},
        "elements_per_s": round(M * N * args.steps * world / (total_ms * 1e-3), 1),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4),
                     "traffic": QUANTIZE_TRAFFIC_BYTES.get((args.workload, flags, sel)), "peak_kind": peak_kind,
                     "kernel": "quantize"},
        "step_frac_of_peak": round(value / world / peak, 4),
        "e2e": {"value": round(nbytes / e2e_s / 1e9 * world, 1), "unit": UNIT,
                "h2d_bytes_per_step": 2 * M * N, "d2h_bytes_per_step": d2h},
        "gpu_launches": 2 * args.steps,
        "step": "CUDA graph replay of nvfp4_amax (memset + kernel) then nvfp4_quantize",
        "clocks": clocks.summary(),
    }
    return res


def workload_config(args):
    flags, sel = synthetic.workload_flags(args.workload)
    if getattr(args, "flags", None) is not None:
        flags = args.flags
    if getattr(args, "sel", None) is not None:
        sel = args.sel
    return flags, sel


def run_once(args):
    """Three amax + quantize passes on one workload, nothing timed: the
    command the ncu captures under profiles/ run."""
    import torch

    import nvfp4_bit_block_gb300 as nv

    nv.lib()
    flags, sel = workload_config(args)
    bits = synthetic.workload(args.workload)
    x = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()
    for _ in range(3):
        amax = nv.nvfp4_amax(x, flags, synthetic.RHT_SEED)
        out = nv.nvfp4_quantize(x, amax, flags, sel, synthetic.SR_SEED, synthetic.RHT_SEED)
    torch.cuda.synchronize()
    assert int(out.status.item()) == 0
    print(json.dumps({"once": args.workload, "flags": flags, "selection": sel}))


def _time_kernels(nv, torch, xs, flags, sel, reps):
    """Average durations (ms) of nvfp4_amax alone, nvfp4_quantize alone and the
    step (both), each measured over `reps` CUDA-graph replays that rotate over
    the input sets `xs` (no host launch gaps inside the timed region)."""
    stream = torch.cuda.Stream()
    am = [nv.nvfp4_amax(x, flags, synthetic.RHT_SEED) for x in xs]
    outs = [nv.nvfp4_quantize(x, a, flags, sel, synthetic.SR_SEED, synthetic.RHT_SEED) for x, a in zip(xs, am)]
    torch.cuda.synchronize()
    graphs = {"amax": [], "quantize": [], "step": []}
    for i, x in enumerate(xs):
        for kind in graphs:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                if kind in ("amax", "step"):
                    nv.nvfp4_amax(x, flags, synthetic.RHT_SEED, out=am[i])
                if kind in ("quantize", "step"):
                    nv.nvfp4_quantize(x, am[i], flags, sel, synthetic.SR_SEED, synthetic.RHT_SEED, out=outs[i])
            graphs[kind].append(g)
    torch.cuda.synchronize()
    res = {}
    with torch.cuda.stream(stream):
        for kind, gl in graphs.items():
            for r in range(len(gl)):
                gl[r].replay()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for r in range(reps):
                gl[r % len(gl)].replay()
            e1.record(stream)
            e1.synchronize()
            res[kind] = e0.elapsed_time(e1) / reps
    torch.cuda.synchronize()
    for o in outs:
        assert int(o.status.item()) == 0
    return res["amax"], res["quantize"], res["step"]


def _report_line(kind, name, M, N, flags, sel, amax_ms, quant_ms, step_ms, peak):
    nb = algorithmic_bytes(M, N, flags)
    q_gbs = nb / (quant_ms * 1e-3) / 1e9
    step_gbs = nb / (step_ms * 1e-3) / 1e9
    return {"report": kind, "name": name, "M": M, "N": N, "flags": flags, "selection": sel,
            "amax_us": round(amax_ms * 1e3, 2), "quantize_us": round(quant_ms * 1e3, 2),
            "step_us": round(step_ms * 1e3, 2),
            "quantize_GBs": round(q_gbs, 1), "quantize_frac_of_measured_peak": round(q_gbs / peak, 4),
            "step_GBs": round(step_gbs, 1), "step_frac_of_measured_peak": round(step_gbs / peak, 4),
            "quantize_elements_per_s": round(M * N / (quant_ms * 1e-3), 1)}


def run_report(args):
    """One JSON line per measurement: every recipe workload, the 4/6, RHT and
    SR ablations, and the size sweep of the activation (X) path from 2^20 to
    2^30 elements.  Input/output sets rotate so that each step reads from HBM.
    amax_us / quantize_us time each call alone (its input cold in L2);
    step_us times amax then quantize, where quantize finds X in L2."""
    import torch

    import nvfp4_bit_block_gb300 as nv

    nv.lib()
    peak, _ = measured_peaks()
    reps = max(5, args.steps)

    def sets_of(bits_or_tensor, M, N, flags):
        per_set = algorithmic_bytes(M, N, flags)
        nsets = max(2, -(-3 * 128 * 2**20 // per_set))
        if isinstance(bits_or_tensor, np.ndarray):
            x0 = torch.from_numpy(bits_or_tensor.view(np.int16)).view(torch.bfloat16).cuda()
        else:
            x0 = bits_or_tensor
        return [x0] + [x0.clone() for _ in range(nsets - 1)]

    cache = {}
    for name in synthetic.WORKLOADS:
        flags, sel = synthetic.workload_flags(name)
        bits = synthetic.workload(name)
        M, N = bits.shape
        xs = sets_of(bits, M, N, flags)
        a, q, st = _time_kernels(nv, torch, xs, flags, sel, reps)
        print(json.dumps(_report_line("workload", name, M, N, flags, sel, a, q, st, peak)), flush=True)
        if name in ("act_46mae_8192x5120", "grad_rht_sr_16384x5120", "weight_2d_5120x20480"):
            cache[name] = xs
        else:
            del xs
    ablations = [("act_46mae_8192x5120", "RN rowwise+columnwise", 3, 0),
                 ("act_46mae_8192x5120", "4/6 MAE", 67, 0), ("act_46mae_8192x5120", "4/6 MSE", 67, 1),
                 ("act_46mae_8192x5120", "4/6 MAXERR", 67, 2), ("act_46mae_8192x5120", "RN rowwise only", 1, 0),
                 ("act_46mae_8192x5120", "4/6 MAE rowwise only", 65, 0),
                 ("grad_rht_sr_16384x5120", "RN", 3, 0), ("grad_rht_sr_16384x5120", "RHT(col)", 19, 0),
                 ("grad_rht_sr_16384x5120", "SR", 35, 0), ("grad_rht_sr_16384x5120", "RHT(col)+SR", 51, 0),
                 ("weight_2d_5120x20480", "1D RN", 3, 0), ("weight_2d_5120x20480", "2D RN", 7, 0),
                 ("weight_2d_5120x20480", "2D 4/6 MAE", 71, 0)]
    for wl, label, flags, sel in ablations:
        xs = cache[wl]
        M, N = xs[0].shape
        a, q, st = _time_kernels(nv, torch, xs, flags, sel, reps)
        print(json.dumps(_report_line("ablation", f"{wl}: {label}", M, N, flags, sel, a, q, st, peak)), flush=True)
    cache.clear()
    # size sweep of the X path (4/6-MSE, both copies), N = 4096, inputs drawn on the GPU
    flags, sel = 67, 1
    N = 4096
    g = torch.Generator(device="cuda")
    for k in range(20, 31):
        M = (1 << k) // N
        g.manual_seed(synthetic.DATA_SEED_BASE + 100 + k)
        mult = torch.ones(N, device="cuda")
        mult[torch.randperm(N, generator=g, device="cuda")[:2]] = 30.0
        x0 = (torch.randn(M, N, generator=g, device="cuda") * mult).to(torch.bfloat16)
        xs = sets_of(x0, M, N, flags)
        a, q, st = _time_kernels(nv, torch, xs, flags, sel, reps)
        print(json.dumps(_report_line("sweep", f"x_path_2^{k}", M, N, flags, sel, a, q, st, peak)), flush=True)
        del xs, x0
        torch.cuda.empty_cache()


def run_error_analysis(args, nbins: int = 24):
    """Where the rounding error sits within the blocks of the workload's
    rowwise copy: standard NVFP4 (block max at 6, alpha over 6*448) against
    4/6 with each selection rule.  One JSON line per variant with, per bin of
    v = 6|x|/b (b = block max), the count, the mean and the RMS of
    e = 6|x - x^|/b, plus the means over v in [4, 6] (the 4-6 gap) and over all
    elements, and the time of the histogram kernel."""
    import torch
    import nvfp4_bit_block_gb300 as nv
    nv.build()
    bits = synthetic.workload(args.workload)
    M, N = bits.shape
    x = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()
    lo = int(4 * nbins / 6)
    variants = [("standard (max 6, 448)", nv.ROWWISE, 0), ("4/6 MAE", nv.ROWWISE | nv.FOUR_SIX, 0),
                ("4/6 MSE", nv.ROWWISE | nv.FOUR_SIX, 1), ("4/6 MAXERR", nv.ROWWISE | nv.FOUR_SIX, 2)]
    for label, flags, sel in variants:
        amax = nv.nvfp4_amax(x, flags)
        out = nv.nvfp4_quantize(x, amax, flags, sel)
        h = nv.nvfp4_error_histogram(x, out.q_row, out.s_row, out.alpha[:1], nbins)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        h2 = torch.zeros_like(h)
        e0.record()
        nv.nvfp4_error_histogram(x, out.q_row, out.s_row, out.alpha[:1], nbins, out=h2)
        e1.record()
        torch.cuda.synchronize()
        hist = h.cpu().numpy().astype(np.float64)
        cnt, se, see = hist[0], hist[1] / 2.0 ** 24, hist[2] / 2.0 ** 32
        with np.errstate(invalid="ignore", divide="ignore"):
            mean = np.where(cnt > 0, se / cnt, 0.0)
            rms = np.sqrt(np.where(cnt > 0, see / cnt, 0.0))
        bins = [[round(6 * i / nbins, 4), round(6 * (i + 1) / nbins, 4), int(cnt[i]), round(float(mean[i]), 5),
                 round(float(rms[i]), 5)] for i in range(nbins)]
        print(json.dumps({
            "analysis": "error_histogram", "workload": args.workload, "M": M, "N": N, "variant": label,
            "flags": flags, "selection": sel, "copy": "rowwise",
            "bins [v_lo, v_hi, count, mean e, rms e]": bins,
            "mean_e_v_4_to_6": round(float(se[lo:].sum() / max(cnt[lo:].sum(), 1)), 5),
            "mean_e_all": round(float(se.sum() / max(cnt.sum(), 1)), 5),
            "rms_e_all": round(float(np.sqrt(see.sum() / max(cnt.sum(), 1))), 5),
            "histogram_kernel_ms": round(e0.elapsed_time(e1), 4)}), flush=True)


def run_oracle_sample(args, max_seconds: float = 20.0, bits=None):
    """Time the CPU oracle (as it stands) on a bounded row sample of the
    workload (`bits`: the workload's tensor if already drawn)."""
    import oracle

    flags, sel = workload_config(args)
    if bits is None:
        bits = synthetic.workload(args.workload)
    M, N = bits.shape
    t0 = time.perf_counter()
    st, am = oracle.amax(bits, flags, synthetic.RHT_SEED)
    t_amax = time.perf_counter() - t0
    rows = 16
    outs = oracle.output_buffers(M, N, flags)
    elapsed = 0.0
    done = 0
    while elapsed < max_seconds / 2 and done < M:
        n = min(rows, M - done)
        t0 = time.perf_counter()
        oracle.quantize(bits, N, am, flags, sel=sel, sr_seed=synthetic.SR_SEED, rht_seed=synthetic.RHT_SEED,
                        row0=done, row1=done + n, outs=outs)
        elapsed += time.perf_counter() - t0
        done += n
        rows = min(rows * 2, 1024)
    frac = done / M
    t_step = t_amax + elapsed / frac           # full-tensor estimate: amax + scaled quantize
    nbytes = algorithmic_bytes(M, N, flags)
    return {"value": round(nbytes / t_step / 1e9, 4), "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"amax over the full {M}x{N} tensor ({t_amax:.2f} s) + quantize of the first "
                      f"{done} rows ({elapsed:.2f} s), scaled to the full tensor"}


def _oracle_stripe_worker(shm_name, shape, r0, r1, flags, sel, amax_parts, amax_all, idx, b_start, b_amax,
                         b_quant, times):
    """One process of the all-cores oracle run: amax of rows [r0, r1), then (after
    the parent has reduced the stripes' maxima) the quantize of the same rows."""
    from multiprocessing import shared_memory
    import oracle
    shm = shared_memory.SharedMemory(name=shm_name)
    try:
        bits = np.ndarray(shape, dtype=np.uint16, buffer=shm.buf)
        M, N = shape
        outs = oracle.output_buffers(M, N, flags)
        b_start.wait()
        t0 = time.monotonic()
        st, am = oracle.amax(bits[r0:r1], flags, synthetic.RHT_SEED)
        amax_parts[2 * idx], amax_parts[2 * idx + 1] = float(am[0]), float(am[1])
        b_amax.wait()
        b_quant.wait()
        am = np.array([amax_all[0], amax_all[1]], dtype=np.float32)
        oracle.quantize(bits, N, am, flags, sel=sel, sr_seed=synthetic.SR_SEED, rht_seed=synthetic.RHT_SEED,
                        row0=r0, row1=r1, outs=outs)
        times[2 * idx], times[2 * idx + 1] = t0, time.monotonic()
        del bits
    finally:
        shm.close()


def run_oracle_all_cores(args):
    """The oracle as it stands, run on every host core at once: the workload's
    rows split into one stripe (a multiple of 16 rows) per process; each process
    takes its stripe's amax, the parent reduces them, and each process then
    quantizes its stripe.  Time = first start to last finish."""
    import multiprocessing as mp
    from multiprocessing import shared_memory
    import oracle

    oracle.build()
    flags, sel = workload_config(args)
    bits = np.ascontiguousarray(synthetic.workload(args.workload).view(np.uint16))
    M, N = bits.shape
    n = max(1, min(len(os.sched_getaffinity(0)), M // 16))
    blocks = M // 16
    bounds = [16 * (blocks * i // n) for i in range(n)] + [M]
    ctx = mp.get_context("spawn")
    shm = shared_memory.SharedMemory(create=True, size=bits.nbytes)
    try:
        np.ndarray(bits.shape, dtype=np.uint16, buffer=shm.buf)[:] = bits
        amax_parts = ctx.Array("f", 2 * n, lock=False)
        amax_all = ctx.Array("f", 2, lock=False)
        times = ctx.Array("d", 2 * n, lock=False)
        b_start, b_amax, b_quant = ctx.Barrier(n + 1), ctx.Barrier(n + 1), ctx.Barrier(n + 1)
        procs = [ctx.Process(target=_oracle_stripe_worker,
                             args=(shm.name, bits.shape, bounds[i], bounds[i + 1], flags, sel, amax_parts, amax_all,
                                   i, b_start, b_amax, b_quant, times)) for i in range(n)]
        for p in procs:
            p.start()
        try:
            b_start.wait(timeout=120)
            b_amax.wait(timeout=120)
            parts = np.frombuffer(amax_parts, dtype=np.float32).reshape(n, 2)
            # NaN-propagating maximum, as a whole-tensor amax would give
            amax_all[0], amax_all[1] = (float(np.max(parts[:, k])) for k in range(2))
            b_quant.wait(timeout=120)
        except threading.BrokenBarrierError:
            pass
        for p in procs:
            p.join(timeout=120)
            if p.exitcode is None:
                p.kill()
                p.join()
        if any(p.exitcode != 0 for p in procs):
            return None
        t = np.frombuffer(times, dtype=np.float64).reshape(n, 2)
        wall = float(t[:, 1].max() - t[:, 0].min())
    finally:
        shm.close()
        shm.unlink()
    nbytes = algorithmic_bytes(M, N, flags)
    return {"value": round(nbytes / wall / 1e9, 4), "unit": UNIT, "cores": n, "kind": "oracle",
            "sample": f"the full {M}x{N} tensor (amax + quantize) in {n} processes over 16-row-aligned "
                      f"row stripes, {wall:.2f} s"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="act_46mae_8192x5120", choices=list(synthetic.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--flags", type=int, default=None, help="override the workload's flags")
    ap.add_argument("--sel", type=int, default=None, help="override the workload's 4/6 selection rule")
    ap.add_argument("--once", action="store_true",
                    help="run amax + quantize three times on the workload and exit (for profilers)")
    ap.add_argument("--report", action="store_true",
                    help="print one JSON line per workload, ablation and X-path size (2^20..2^30)")
    ap.add_argument("--error-analysis", action="store_true",
                    help="print the rowwise error histogram over the scaled value, standard vs 4/6")
    args = ap.parse_args()
    if args.error_analysis:
        run_error_analysis(args)
        return
    if args.once:
        run_once(args)
        return
    if args.report:
        run_report(args)
        return
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))

    if args.impl == "reference":
        if rank != 0:
            return
        per_step = []
        cb = None
        bits = synthetic.workload(args.workload)  # drawn once; the steps time the oracle only
        for _ in range(args.warmup + args.steps):
            cb = run_oracle_sample(args, max_seconds=4.0, bits=bits)
            per_step.append(cb["value"])
        v = round(statistics.mean(per_step[args.warmup:]) if args.steps else per_step[-1], 5)
        flags, sel = workload_config(args)
        _, M, N = synthetic.WORKLOADS[args.workload][:3]
        print(json.dumps({
            "impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": 0,
            "steps": args.steps, "warmup": args.warmup, "higher_is_better": True,
            "config": {"workload": args.workload, "M": M, "N": N, "flags": flags, "selection": sel},
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": cb["sample"]},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        }))
        return

    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    res = run_ours(args, rank, world)
    if rank == 0:
        if not args.no_cpu_baseline:
            res["cpu_baseline"] = run_oracle_sample(args)
            allc = run_oracle_all_cores(args)
            if allc is not None:
                res["cpu_baseline_all_cores"] = allc
        print(json.dumps(res))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
