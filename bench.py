"""Benchmark of the NVFP4 quantizer hot path on one GB300 (or N replicas).

A step is one pass of the whole hot path over every tensor of the workload:
for each tensor nvfp4_amax (tensor amax per copy) then nvfp4_quantize (scale,
round, pack; rowwise + transposed columnwise outputs).  The default workload
is the recipe's full linear layer (its largest configuration):

  X  16384 x 5120  activation, 1x16 blocks, 4/6 with MSE selection, both copies
  W  5120 x 20480  weight, 16x16 2D blocks, both copies
  dY 16384 x 20480 gradient, Hadamard on the columnwise copy, stochastic
                   rounding on both copies

The single tensors (the 256x1024 rowwise case, the 8192x5120 activation, the
weight, the 16384x5120 gradient, and each linear-layer tensor alone) are
available with --workload.

Metric: NVFP4 quantize GB/s = (bf16 bytes read + code bytes + scale bytes
written) per step / step time.  The timed steps rotate over input/output sets
whose combined size exceeds the L2, so every step reads from HBM.  Every kernel
is also timed alone inside the same rotating stream (CUDA events on its own
stream); the roofline entry is for the kernel that takes the most time: HBM
bandwidth for the codec kernels, and for the stochastic-rounding kernels
(one Philox4x32-10 call per element, bound by 32x32->64-bit integer products)
Philox calls per second against the SMs' wide-multiply rate.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]
  python bench.py --report | --error-analysis | --once | --gemm

Under torchrun (N > 1) every rank runs an independent replica (the path needs
no exchange for independent tensors) and rank 0 prints the JSON line with the
max step time over ranks.  --impl reference times the CPU oracle on the host
cores instead (a bounded row sample of the same workload).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synthetic  # noqa: E402

METRIC = "NVFP4 quantize GB/s (bf16 in + fp4/scales out), % of GB300 HBM peak"
UNIT = "GB/s"

# Workloads made of several tensors quantized in one step.
COMPOSITES = {
    "linear_layer": ["linear_x_16384x5120", "linear_w_5120x20480", "linear_dy_16384x20480"],
}
DEFAULT_WORKLOAD = "linear_layer"
WORKLOAD_CHOICES = list(COMPOSITES) + list(synthetic.WORKLOADS)

# Integer-multiply roofline of the stochastic-rounding kernels: a Philox4x32-10
# call takes ten rounds of two 32x32->64-bit products; with the counter's
# upper words zero, the first round's second product is a product with zero,
# the second round's first product depends only on the counter's high word
# (shared by every element of a block) and the last round's first product
# feeds only the unused words 2 and 3, so 17 products per call depend on the
# element.  A 64-bit-result integer multiply issues at a quarter of the 128
# lanes per clock of an SM (measured: 28.7-29.7 products per clock per SM for
# mul.wide.u32 and mul.hi.u32).
PHILOX_PRODUCTS_PER_CALL = 17
WIDE_PRODUCTS_PER_CLK_PER_SM = 32

# DRAM bytes (read + written) of one launch of a kernel from an ncu capture,
# keyed by (tensor, kernel) with the hash of that kernel's sources
# (KERNEL_SOURCES) when the capture was taken; a stale hash reports null.  Captured with
#   ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum --clock-control none \
#       -k regex:quant1d_sr -c 1 python bench.py --once --workload <tensor>
# (one pass; a cold single launch, so outputs still in L2 at its end are not
# counted as written).
TRAFFIC = {
    ("linear_dy_16384x20480", "quantize_sr"): (689_250_000 + 362_170_000, "561874a1ea1c2cb6"),
    ("grad_rht_sr_16384x5120", "quantize_sr"): (167_877_888 + 56_236_544, "561874a1ea1c2cb6"),
}
CSRC = os.path.join(ROOT, "nvfp4_bit_block_gb300", "csrc")


# The CUDA sources each kernel of the step is built from (a traffic capture
# stays valid while these are unchanged).
KERNEL_SOURCES = {
    "quantize": ["api.cu", "tmap.cu", "quant1d.cu", "quant1d_46mae.cu", "quant1d_46mse.cu", "quant1d_46max.cu",
                 "quant1d_common.cuh", "quant1d_kernel.cuh", "quant1d_sr.cu", "quant1d_sr_kernel.cuh", "quant2d.cu",
                 "tile_pipeline.cuh", "tma.cuh", "nvfp4_device.cuh", "nvfp4_internal.h"],
    # the kernel that quantizes with SR on both copies, without 4/6, 2D or a
    # rowwise transform (quant1d_sr_kernel)
    "quantize_sr": ["api.cu", "tmap.cu", "quant1d_common.cuh", "quant1d_sr.cu", "quant1d_sr_kernel.cuh",
                    "tile_pipeline.cuh", "tma.cuh", "nvfp4_device.cuh", "nvfp4_internal.h"],
    "amax": ["api.cu", "amax.cu", "tile_pipeline.cuh", "nvfp4_device.cuh", "nvfp4_internal.h"],
}


def source_hash(kernel: str = "quantize") -> str:
    """Hash of the CUDA sources `kernel` is built from (16 hex digits)."""
    h = hashlib.sha256()
    for name in sorted(KERNEL_SOURCES[kernel]):
        with open(os.path.join(CSRC, name), "rb") as f:
            h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


def sources_of(kernel: str, flags: int) -> str:
    """The KERNEL_SOURCES key of the kernel that runs `kernel` with `flags`."""
    sr_both = flags & 32 and flags & 1 and flags & 2 and not flags & (4 | 8 | 64)  # SR, R + C; no 2D, RHT_ROW, 4/6
    return "quantize_sr" if kernel == "quantize" and sr_both else kernel


def traffic_of(part: str, kernel: str):
    entry = TRAFFIC.get((part, kernel))
    if entry is None or entry[1] != source_hash(kernel):
        return None
    return entry[0]


def parts_of(workload: str):
    return COMPOSITES.get(workload, [workload])


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
    """(HBM GB/s, kind, SM max MHz) from MEASURED_PEAKS.json, else the fallback."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured", float(d.get("sm_max_mhz", 2070.0))
    return 6800.0, "fallback", 2070.0


def philox_peak_gcalls(sms: int, sm_mhz: float) -> float:
    """Philox calls per second (G) at the SMs' wide-multiply rate."""
    return sms * WIDE_PRODUCTS_PER_CLK_PER_SM / PHILOX_PRODUCTS_PER_CALL * sm_mhz * 1e6 / 1e9


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


def workload_config(args, part: str):
    """(flags, selection) of one tensor of the workload (--flags/--sel override)."""
    flags, sel = synthetic.workload_flags(part)
    if getattr(args, "flags", None) is not None:
        flags = args.flags
    if getattr(args, "sel", None) is not None:
        sel = args.sel
    return flags, sel


def _kernel_roofline(part, kernel, flags, M, N, ms, hbm_peak, peak_kind, sms, sm_mhz):
    """Roofline record of one kernel launch that took `ms` on average."""
    if kernel == "amax":
        nbytes = 2 * M * N
        rec = {"bound": "hbm", "achieved": nbytes / (ms * 1e-3) / 1e9, "peak": hbm_peak, "unit": "GB/s",
               "algorithmic": f"{nbytes} bytes (bf16 read)"}
    elif flags & 32:  # stochastic rounding: one Philox4x32-10 call per element
        calls = M * N
        rec = {"bound": "alu", "achieved": calls / (ms * 1e-3) / 1e9, "peak": round(philox_peak_gcalls(sms, sm_mhz), 1),
               "unit": "G Philox calls/s",
               "algorithmic": f"{calls} Philox4x32-10 calls x {PHILOX_PRODUCTS_PER_CALL} wide products",
               "peak_basis": f"{sms} SMs x {WIDE_PRODUCTS_PER_CLK_PER_SM} 32x32->64 products/clk / "
                             f"{PHILOX_PRODUCTS_PER_CALL} per call x {sm_mhz:.0f} MHz",
               "hbm_gbs": round(algorithmic_bytes(M, N, flags) / (ms * 1e-3) / 1e9, 1)}
    else:
        nbytes = algorithmic_bytes(M, N, flags)
        rec = {"bound": "hbm", "achieved": nbytes / (ms * 1e-3) / 1e9, "peak": hbm_peak, "unit": "GB/s",
               "algorithmic": f"{nbytes} bytes (bf16 read + codes + scales)"}
    rec["achieved"] = round(rec["achieved"], 1)
    rec["frac"] = round(rec["achieved"] / rec["peak"], 4)
    rec["peak_kind"] = peak_kind if rec["bound"] == "hbm" else "derived from the SM count, the measured " \
                                                                 "multiply rate and the maximum SM clock"
    t = traffic_of(part, sources_of(kernel, flags))
    rec["traffic"] = t
    if t is not None:
        rec["dram_gbs"] = round(t / (ms * 1e-3) / 1e9, 1)
    rec.update({"kernel": kernel, "tensor": part, "ms": round(ms, 5)})
    return rec


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
    parts = parts_of(args.workload)
    cfg = []
    for p in parts:
        flags, sel = workload_config(args, p)
        bits = synthetic.workload(p)
        M, N = bits.shape
        host = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).pin_memory()
        cfg.append(dict(part=p, flags=flags, sel=sel, M=M, N=N, host=host, nbytes=algorithmic_bytes(M, N, flags)))
        del bits
    nbytes = sum(c["nbytes"] for c in cfg)
    # Several input/output sets used in rotation, so that the bytes touched
    # between two uses of the same set exceed the 129 MB L2: every step reads
    # its inputs from HBM and the previous steps' outputs are written back
    # during later steps, as in a steady stream of tensors.
    nsets = max(2, -(-3 * 128 * 2**20 // nbytes))
    stream = torch.cuda.Stream(device=dev)
    sets = []
    for i in range(nsets):
        s = []
        for c in cfg:
            x = c["host"].to(dev)
            am = torch.empty(2, dtype=torch.float32, device=dev)
            out = nv.nvfp4_quantize(x, nv.nvfp4_amax(x, c["flags"], synthetic.RHT_SEED), c["flags"], c["sel"])
            s.append((x, am, out))
        sets.append(s)
    torch.cuda.synchronize()

    def step(i, events=None, single_pass=False):
        for j, c in enumerate(cfg):
            x, am, out = sets[i][j]
            if events is not None:
                events[j][0].record(stream)
            if not single_pass:
                nv.nvfp4_amax(x, c["flags"], synthetic.RHT_SEED, out=am, stream=stream)
            if events is not None:
                events[j][1].record(stream)
            nv.nvfp4_quantize(x, am, c["flags"], c["sel"], synthetic.SR_SEED, synthetic.RHT_SEED, 0, out=out,
                              stream=stream)
            if events is not None:
                events[j][2].record(stream)

    with torch.cuda.stream(stream):
        for k in range(max(args.warmup, nsets)):
            step(k % nsets)
    torch.cuda.synchronize()

    # the step (every amax and quantize) as one CUDA graph per set: no host launch gaps
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

    def timed_interval(nsteps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for k in range(nsteps):
                graphs[k % nsets].replay()
            e1.record(stream)
        e1.synchronize()
        return e0.elapsed_time(e1)

    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    # The sampler also covers untimed steps run right before the timed ones
    # (at least half a second), so the clocks reported are the clocks under
    # this load even when the timed region is shorter than its interval.
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for k in range(max(1, 2 * nsets)):
            graphs[k % nsets].replay()
    torch.cuda.synchronize()
    per_step_s = max((time.perf_counter() - t0) / max(1, 2 * nsets), 1e-6)
    load_steps = int(min(20000, max(1, 0.5 / per_step_s)))
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
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
        # further intervals of the same length, for the spread of the figure
        repeats = [timed_interval(args.steps) for _ in range(5)]
    # Single pass (delayed scaling): the same step with each tensor's amax
    # supplied by the caller -- here the amax each set already holds -- so
    # only the quantize kernels run.
    graphs_sp = []
    for i in range(nsets):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            step(i, single_pass=True)
        graphs_sp.append(g)
    with torch.cuda.stream(stream):
        for k in range(max(args.warmup, nsets)):
            graphs_sp[k % nsets].replay()
        e_sp0, e_sp1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e_sp0.record(stream)
        for k in range(args.steps):
            graphs_sp[k % nsets].replay()
        e_sp1.record(stream)
    e_sp1.synchronize()
    sp_ms = max_over_ranks(e_sp0.elapsed_time(e_sp1), world, dev) / args.steps
    if world > 1:
        dist.barrier()
    total_ms = max_over_ranks(ev0.elapsed_time(ev1), world, dev)

    # Every kernel timed alone inside the same rotating stream of steps:
    # the calls are launched directly with an event between any two.
    kev = [[[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in cfg] for _ in range(args.steps)]
    with torch.cuda.stream(stream):
        for k in range(args.steps):
            step(k % nsets, kev[k])
    torch.cuda.synchronize()
    for s in sets:
        for _, _, out in s:
            status = int(out.status.item())
            assert status == 0, f"quantize reported status {status}"

    # End to end through the public API: every step copies its inputs from
    # pinned host memory to the device, runs amax + quantize on each and copies
    # all outputs back to pinned host memory.  Steps are pipelined the way a
    # stream of tensors would be: copy-in, compute and copy-out run on their
    # own streams, ordered by events, over two device buffer sets (the inputs
    # and outputs of set i are reused two steps later).
    e2e_steps = max(4, min(args.steps, 8))
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    dev_outs = [[t_ for (_, _, o) in sets[i] for t_ in (o.q_row, o.s_row, o.q_col, o.s_col, o.alpha) if t_ is not None]
                for i in range(2)]
    host_outs = [[torch.empty(t_.shape, dtype=t_.dtype, pin_memory=True) for t_ in d] for d in dev_outs]
    x_hosts = [[c["host"] for c in cfg], [c["host"].clone().pin_memory() for c in cfg]]
    e2e_reps = 3  # several intervals: a host link shared with other processes varies
    e2e_warm = 4
    ev_in = [torch.cuda.Event() for _ in range(e2e_reps * e2e_steps + e2e_warm)]
    ev_comp = [torch.cuda.Event() for _ in range(e2e_reps * e2e_steps + e2e_warm)]
    ev_out = [torch.cuda.Event() for _ in range(e2e_reps * e2e_steps + e2e_warm)]
    torch.cuda.synchronize()

    def e2e_step(k):
        i = k % 2
        with torch.cuda.stream(s_in):
            if k >= 2:
                s_in.wait_event(ev_comp[k - 2])     # set i's inputs no longer read
            for j in range(len(cfg)):
                sets[i][j][0].copy_(x_hosts[i][j], non_blocking=True)
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

    for k in range(e2e_warm):
        e2e_step(k)
    torch.cuda.synchronize()
    e2e_times = []
    for r in range(e2e_reps):
        t0 = time.perf_counter()
        for k in range(e2e_warm + r * e2e_steps, e2e_warm + (r + 1) * e2e_steps):
            e2e_step(k)
        torch.cuda.synchronize()
        e2e_times.append((time.perf_counter() - t0) / e2e_steps)
    e2e_s = statistics.median(e2e_times)
    d2h = sum(t_.numel() * t_.element_size() for t_ in dev_outs[0])
    h2d = sum(2 * c["M"] * c["N"] for c in cfg)

    hbm_peak, peak_kind, sm_max_mhz = measured_peaks()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    kernels = []
    for j, c in enumerate(cfg):
        am_ms = statistics.mean(e[j][0].elapsed_time(e[j][1]) for e in kev)
        q_ms = statistics.mean(e[j][1].elapsed_time(e[j][2]) for e in kev)
        kernels.append(_kernel_roofline(c["part"], "amax", c["flags"], c["M"], c["N"], am_ms, hbm_peak, peak_kind,
                                        sms, sm_max_mhz))
        kernels.append(_kernel_roofline(c["part"], "quantize", c["flags"], c["M"], c["N"], q_ms, hbm_peak, peak_kind,
                                        sms, sm_max_mhz))
    dominant = max(kernels, key=lambda r: r["ms"])
    value = nbytes * args.steps / (total_ms * 1e-3) / 1e9 * world
    clk = clocks.summary()
    ms_per_step = total_ms / args.steps
    if len(parts) == 1:
        c = cfg[0]
        config = {"workload": parts[0], "M": c["M"], "N": c["N"], "flags": c["flags"], "selection": c["sel"]}
    else:
        config = {"workload": args.workload,
                  "tensors": [{"name": c["part"], "M": c["M"], "N": c["N"], "flags": c["flags"], "selection": c["sel"]}
                              for c in cfg]}
    config.update({"elements": sum(c["M"] * c["N"] for c in cfg), "bytes_per_step": nbytes,
                   "l2": f"inputs larger than L2: {nsets} input/output sets of {nbytes / 1e6:.0f} MB in rotation",
                   "parallelism": f"replicas{world}" if world > 1 else "single GPU"})
    reps = sorted(r / args.steps for r in repeats)
    res = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded, the recipe's shapes and value distributions)",
        "config": config,
        "kernels_ms": {f"{r['tensor']}:{r['kernel']}": r["ms"] for r in kernels},
        "elements_per_s": round(config["elements"] * args.steps * world / (total_ms * 1e-3), 1),
        "roofline": {k: dominant[k] for k in ("bound", "achieved", "peak", "unit", "frac", "traffic")},
        "roofline_detail": dominant,
        "kernels": kernels,
        "step_frac_of_hbm_peak": round(value / world / hbm_peak, 4),
        "repeat_intervals": {"count": len(reps), "ms_per_step_median": round(statistics.median(reps), 5),
                             "ms_per_step_min": round(reps[0], 5), "ms_per_step_max": round(reps[-1], 5)},
        "e2e": {"value": round(nbytes / e2e_s / 1e9 * world, 1), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "intervals": {"count": e2e_reps, "steps_each": e2e_steps,
                              "GBs_min": round(nbytes / max(e2e_times) / 1e9 * world, 1),
                              "GBs_max": round(nbytes / min(e2e_times) / 1e9 * world, 1)}},
        "gpu_launches": 2 * len(cfg) * args.steps,
        "step": "CUDA graph replay of nvfp4_amax (memset + kernel) then nvfp4_quantize for each tensor",
        "single_pass": {"value": round(nbytes / (sp_ms * 1e-3) / 1e9 * world, 1), "unit": UNIT,
                        "ms_per_step": round(sp_ms, 5),
                        "step": "the same step with the amax supplied by the caller (delayed scaling): "
                                "nvfp4_quantize only"},
        "clocks": clk,
    }
    if clk.get("sm_mhz"):
        res["ms_x_sm_mhz"] = round(ms_per_step * clk["sm_mhz"], 2)
    return res


def run_once(args):
    """Three amax + quantize passes over each tensor of the workload, nothing
    timed: the command the ncu captures under profiles/ run."""
    import torch

    import nvfp4_bit_block_gb300 as nv

    nv.lib()
    for p in parts_of(args.workload):
        flags, sel = workload_config(args, p)
        bits = synthetic.workload(p)
        x = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()
        del bits
        for _ in range(3):
            amax = nv.nvfp4_amax(x, flags, synthetic.RHT_SEED)
            out = nv.nvfp4_quantize(x, amax, flags, sel, synthetic.SR_SEED, synthetic.RHT_SEED)
        torch.cuda.synchronize()
        assert int(out.status.item()) == 0
        print(json.dumps({"once": p, "flags": flags, "selection": sel}))
        del x, out
        torch.cuda.empty_cache()


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
    """One JSON line per measurement: every recipe tensor, the 4/6, RHT and
    SR ablations, and the size sweep of the activation (X) path from 2^20 to
    2^30 elements.  Input/output sets rotate so that each step reads from HBM.
    amax_us / quantize_us time each call alone (its input cold in L2);
    step_us times amax then quantize, where quantize finds X in L2."""
    import torch

    import nvfp4_bit_block_gb300 as nv

    nv.lib()
    peak = measured_peaks()[0]
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
                 ("act_46mae_8192x5120", "RN columnwise only", 2, 0),
                 ("act_46mae_8192x5120", "4/6 MAE columnwise only", 66, 0),
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


def fp4_peak_tflops():
    """Dense FP4 tensor peak: the measured bf16 GEMM peak x 6, the nominal
    FP4 / BF16 ratio (13.5 / 2.25 PFLOP/s dense)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return 6.0 * float(json.load(f)["bf16_tflops"]), "measured bf16 x 6 (nominal FP4/BF16 ratio)"
    return 6.0 * 1900.0, "fallback bf16 x 6"


def run_gemm(args):
    """The linear layer's three NVFP4 GEMMs on the quantizer's own outputs
    (tiled scales): fprop Y = X W (A = X rowwise, B = W columnwise), dgrad
    dX = dY W^T (A = dY rowwise, B = W rowwise), wgrad dW = X^T dY (A = X
    columnwise, B = dY columnwise).  One JSON line per GEMM: CUDA-event time
    averaged over --steps launches after --warmup, TFLOP/s (2MNK) and the
    fraction of the dense FP4 tensor peak."""
    import torch

    import nvfp4_bit_block_gb300 as nv

    nv.lib()
    q = {}
    for p in parts_of("linear_layer"):
        flags, sel = synthetic.workload_flags(p)
        bits = synthetic.workload(p)
        x = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()
        del bits
        am = nv.nvfp4_amax(x, flags, synthetic.RHT_SEED)
        q[p] = nv.nvfp4_quantize(x, am, flags | nv.SF_SWIZZLED, sel, synthetic.SR_SEED, synthetic.RHT_SEED)
        del x
    torch.cuda.synchronize()
    X, W, dY = (q[p] for p in parts_of("linear_layer"))
    gemms = [("fprop Y = X W", X.q_row, X.s_row, X.alpha[0:1], W.q_col, W.s_col, W.alpha[1:2]),
             ("dgrad dX = dY W^T", dY.q_row, dY.s_row, dY.alpha[0:1], W.q_row, W.s_row, W.alpha[0:1]),
             ("wgrad dW = X^T dY", X.q_col, X.s_col, X.alpha[1:2], dY.q_col, dY.s_col, dY.alpha[1:2])]
    peak, peak_kind = fp4_peak_tflops()
    out_dtype = torch.bfloat16 if args.gemm_out == "bf16" else torch.float32
    for name, qa, sa, aa, qb, sb, ab in gemms:
        M, N, K = qa.shape[0], qb.shape[0], 2 * qa.shape[1]
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        out = torch.empty((M, N), dtype=out_dtype, device="cuda")
        for _ in range(max(3, args.warmup)):
            nv.nvfp4_gemm(qa, sa, aa, qb, sb, ab, out=out, status=status)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(args.steps):
            nv.nvfp4_gemm(qa, sa, aa, qb, sb, ab, out=out, status=status)
        e1.record()
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        ms = e0.elapsed_time(e1) / args.steps
        tflops = 2.0 * M * N * K / (ms * 1e-3) / 1e12
        print(json.dumps({"gemm": name, "M": M, "N": N, "K": K, "out": args.gemm_out, "ms": round(ms, 4),
                          "TFLOP/s": round(tflops, 1),
                          "roofline": {"bound": "tensor", "achieved": round(tflops, 1), "peak": round(peak, 1),
                                       "unit": "TFLOP/s", "frac": round(tflops / peak, 4), "peak_kind": peak_kind},
                          "steps": args.steps, "warmup": args.warmup}), flush=True)


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
    name = parts_of(args.workload)[0] if args.workload in COMPOSITES else args.workload
    bits = synthetic.workload(name)
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
            "analysis": "error_histogram", "workload": name, "M": M, "N": N, "variant": label,
            "flags": flags, "selection": sel, "copy": "rowwise",
            "bins [v_lo, v_hi, count, mean e, rms e]": bins,
            "mean_e_v_4_to_6": round(float(se[lo:].sum() / max(cnt[lo:].sum(), 1)), 5),
            "mean_e_all": round(float(se.sum() / max(cnt.sum(), 1)), 5),
            "rms_e_all": round(float(np.sqrt(see.sum() / max(cnt.sum(), 1))), 5),
            "histogram_kernel_ms": round(e0.elapsed_time(e1), 4)}), flush=True)


def run_oracle_sample(args, max_seconds: float = 20.0, bits_by_part=None):
    """The CPU oracle (as it stands, one thread) on a bounded row sample of
    every tensor of the workload, scaled to the whole step: per tensor the
    amax over a leading row stripe and the quantize of a growing number of
    leading rows, each scaled by the tensor's row count.  `bits_by_part`: the
    tensors if already drawn."""
    import oracle

    parts = parts_of(args.workload)
    total_bytes = 0
    t_step = 0.0
    notes = []
    for p in parts:
        flags, sel = workload_config(args, p)
        bits = bits_by_part[p] if bits_by_part else synthetic.workload(p)
        M, N = bits.shape
        nb = algorithmic_bytes(M, N, flags)
        total_bytes += nb
        budget = max_seconds * nb / sum(algorithmic_bytes(*synthetic.WORKLOADS[q][1:3], workload_config(args, q)[0])
                                        for q in parts)
        arows = min(M, 256)
        t0 = time.perf_counter()
        st, _ = oracle.amax(bits[:arows], flags, synthetic.RHT_SEED)
        t_amax = (time.perf_counter() - t0) * M / arows
        st, am = oracle.amax(bits[:arows], flags, synthetic.RHT_SEED)  # the sample's amax scales the sample
        outs = oracle.output_buffers(M, N, flags)
        elapsed, done, rows = 0.0, 0, 16
        while elapsed < budget / 2 and done < M:
            n = min(rows, M - done)
            t0 = time.perf_counter()
            oracle.quantize(bits, N, am, flags, sel=sel, sr_seed=synthetic.SR_SEED, rht_seed=synthetic.RHT_SEED,
                            row0=done, row1=done + n, outs=outs)
            elapsed += time.perf_counter() - t0
            done += n
            rows = min(rows * 2, 1024)
        t_step += t_amax + elapsed * M / done
        notes.append(f"{p}: amax of {arows} rows, quantize of {done} rows of {M}")
        del outs
    return {"value": round(total_bytes / t_step / 1e9, 4), "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": "; ".join(notes) + "; each scaled to the whole tensor"}


def run_oracle_all_cores(args):
    """The oracle as it stands, run on every host core at once over the whole
    workload: each tensor's rows split into one stripe (a multiple of 16 rows)
    per process, each process takes its stripe's amax, the parent reduces
    them, and each process then quantizes its stripe.  Time = the amax and
    quantize phases of every tensor, first start to last finish."""
    from oracle.parallel import amax_parallel, quantize_parallel

    total_bytes, wall, procs = 0, 0.0, 0
    for p in parts_of(args.workload):
        flags, sel = workload_config(args, p)
        bits = np.ascontiguousarray(synthetic.workload(p).view(np.uint16))
        M, N = bits.shape
        t0 = time.monotonic()
        st, am = amax_parallel(bits, flags, synthetic.RHT_SEED)
        t_amax = time.monotonic() - t0
        if st != 0:
            return None
        r = quantize_parallel(bits, flags, sel, synthetic.SR_SEED, synthetic.RHT_SEED, amax2=am)
        if r["status"] != 0:
            return None
        wall += t_amax + r["seconds"]
        procs = max(procs, r["procs"])
        total_bytes += algorithmic_bytes(M, N, flags)
        del bits, r
    return {"value": round(total_bytes / wall / 1e9, 4), "unit": UNIT, "cores": procs, "kind": "oracle",
            "sample": f"the whole workload ({', '.join(parts_of(args.workload))}): amax and quantize in {procs} "
                      f"processes over 16-row-aligned row stripes, {wall:.2f} s"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=WORKLOAD_CHOICES)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--flags", type=int, default=None, help="override the flags (single-tensor workloads)")
    ap.add_argument("--sel", type=int, default=None, help="override the 4/6 selection rule (single-tensor workloads)")
    ap.add_argument("--once", action="store_true",
                    help="run amax + quantize three times on each tensor and exit (for profilers)")
    ap.add_argument("--report", action="store_true",
                    help="print one JSON line per tensor, ablation and X-path size (2^20..2^30)")
    ap.add_argument("--error-analysis", action="store_true",
                    help="print the rowwise error histogram over the scaled value, standard vs 4/6")
    ap.add_argument("--gemm", action="store_true",
                    help="time the linear layer's three NVFP4 GEMMs (fprop, dgrad, wgrad) on the tensor cores")
    ap.add_argument("--gemm-out", default="bf16", choices=["bf16", "fp32"], help="output type of --gemm")
    args = ap.parse_args()
    if args.workload in COMPOSITES and (args.flags is not None or args.sel is not None):
        ap.error("--flags / --sel apply to single-tensor workloads")
    if args.error_analysis:
        run_error_analysis(args)
        return
    if args.once:
        run_once(args)
        return
    if args.gemm:
        run_gemm(args)
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
        drawn = {p: synthetic.workload(p) for p in parts_of(args.workload)}  # drawn once; the steps time the oracle
        for _ in range(args.warmup + args.steps):
            cb = run_oracle_sample(args, max_seconds=4.0, bits_by_part=drawn)
            per_step.append(cb["value"])
        v = round(statistics.mean(per_step[args.warmup:]) if args.steps else per_step[-1], 5)
        parts = parts_of(args.workload)
        if len(parts) == 1:
            flags, sel = workload_config(args, parts[0])
            _, M, N = synthetic.WORKLOADS[parts[0]][:3]
            config = {"workload": parts[0], "M": M, "N": N, "flags": flags, "selection": sel}
        else:
            config = {"workload": args.workload,
                      "tensors": [{"name": p, "M": synthetic.WORKLOADS[p][1], "N": synthetic.WORKLOADS[p][2],
                                   "flags": workload_config(args, p)[0], "selection": workload_config(args, p)[1]}
                                  for p in parts]}
        print(json.dumps({
            "impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "higher_is_better": True,
            "config": config,
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
