"""Benchmark of the NVFP4 W4A4 MoE expert forward on GB300.

One step = one moe_expert_forward call (route, permute + amax + quantise,
FC1 + SwiGLU + requantise, FC2 + router-weighted scatter, unpermute reduce)
over the Qwen3-30B-A3B-shaped layer (T = 65536 tokens = 16 x 4096, d = 2048,
E = 128, top-8, d_ff = 768, uniform router logits), inputs resident in HBM.
The timed steps are replays of one CUDA-graph capture of the forward.
Prints one JSON line: the headline, each kernel against its roofline (CUDA
events around each launch), the other Qwen-shaped and small workloads, the
built next rows, end-to-end throughput with host buffers, and the CPU
oracle.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...    # the CPU oracle as the reference arm

Multi-GPU (torchrun, one rank per GPU): token data parallelism, each rank
runs its own batch of T tokens with replicated weights; no collective on the
data path; timing is the max over ranks (weak scaling).
"""
from __future__ import annotations

import argparse
import ctypes
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

METRIC = "NVFP4 MoE expert-forward tokens/s at 1 GB300; % FP4 tensor peak, % HBM BW"
UNIT = "tokens/s"
# Dense FP4 (NVFP4 block-scaled) tensor peak derived from the measured bf16
# cuBLAS peak times the nominal fp4:bf16 ratio (13.5 / 2.25 = 6).
FP4_PER_BF16 = 6.0
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# The seven launches of the forward, in order.
KERNELS = ["route_kernel", "scan_kernel", "pad_rows_kernel", "permute_quant_kernel", "fc1_swiglu_kernel",
           "fc2_scatter_kernel", "unpermute_reduce_kernel"]

# DRAM traffic per launch of the dominant kernel (dram__bytes_read.sum +
# dram__bytes_write.sum from one ncu capture), keyed to the hash of the
# device code it was captured on and to the workload; reported as null once
# either differs.
NCU_TRAFFIC = {"fc1": {"src_sha": "3df75dfdc6085eb0", "bytes_per_launch": 976925312 + 481038592, "workload": "qwen64k"}}
# Host code follows this line in a source file; it is left out of the hash,
# so a launcher edit keeps a capture of unchanged device code valid.
HOST_MARKER = "// host launchers"


def src_sha(*names):
    """Hash of the sources' device code: everything up to a line holding
    HOST_MARKER, with // comments, trailing blanks and blank lines left out,
    so comment and host-code edits keep a capture valid and any change of
    device code invalidates it."""
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "nvfp4_w4a4_moe_top_gb300", "csrc", n), encoding="utf-8") as f:
            for line in f:
                if HOST_MARKER in line:
                    break
                code = re.sub(r"//.*", "", line).rstrip()
                if code:
                    h.update(code.encode() + b"\n")
    return h.hexdigest()[:16]


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# --------------------------------------------------------------------------
# distributed harness (testable on CPU with gloo)
# --------------------------------------------------------------------------
def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def shard_seed(base_seed, rank):
    """Each rank draws its own token batch (data parallel); weights are
    shared (seeded by the base seed only)."""
    return base_seed + 1000003 * rank


def max_over_ranks(value, world, device=None):
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(tokens_per_rank_step, steps, world, seconds_max):
    """Whole-job throughput: all ranks' tokens over the slowest rank's time."""
    return tokens_per_rank_step * steps * world / seconds_max


# --------------------------------------------------------------------------
# clocks
# --------------------------------------------------------------------------
# NVML clock-event reason bits (nvml.h)
NVML_REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
                0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}


class ClockSampler:
    """SM clock and clock-event reasons of the GPU sampled during the timed
    region: through NVML (read-only queries, every `period` seconds, in a
    thread), else nvidia-smi at its fastest interval."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index, uuid=None, period=0.002):
        self.index, self.uuid, self.period = index, uuid, period
        self.samples, self.max_mhz, self.source = [], None, None
        self.proc = None
        self.stop = threading.Event()

    def _nvml_open(self):
        nv = ctypes.CDLL("libnvidia-ml.so.1")
        if nv.nvmlInit_v2() != 0:
            return None
        h = ctypes.c_void_p()
        ok = False
        if self.uuid:
            ok = nv.nvmlDeviceGetHandleByUUID(("GPU-" + self.uuid).encode(), ctypes.byref(h)) == 0
        if not ok:
            ok = nv.nvmlDeviceGetHandleByIndex_v2(self.index, ctypes.byref(h)) == 0
        if not ok:
            return None
        mx = ctypes.c_uint()
        if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:  # NVML_CLOCK_SM
            self.max_mhz = float(mx.value)
        self.reason_fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            nv.nvmlDeviceGetCurrentClocksThrottleReasons
        return nv, h

    def _poll(self, nv, h):
        clk, rs = ctypes.c_uint(), ctypes.c_ulonglong()
        while not self.stop.is_set():
            if nv.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0 and self.reason_fn(h, ctypes.byref(rs)) == 0:
                self.samples.append((float(clk.value), int(rs.value)))
            time.sleep(self.period)

    def __enter__(self):
        try:
            opened = self._nvml_open()
        except OSError:
            opened = None
        if opened:
            self.source = "nvml"
            self.thread = threading.Thread(target=self._poll, args=opened, daemon=True)
            self.thread.start()
            return self
        self.path = os.path.join("/tmp", "moe_clocks_%d_%d.csv" % (os.getpid(), self.index))
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
            self.source = "nvidia-smi"
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.source == "nvml":
            self.stop.set()
            self.thread.join(timeout=5)
        elif self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()
            names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
            bits = {"hw_slowdown": 0x8, "hw_thermal_slowdown": 0x40, "sw_thermal_slowdown": 0x20,
                    "sw_power_cap": 0x4}
            with open(self.path) as f:
                for line in f:
                    parts = [p.strip() for p in line.split(",")]
                    if len(parts) < 9:
                        continue
                    try:
                        sm = float(parts[1])
                        self.max_mhz = float(parts[2])
                    except ValueError:
                        continue
                    r = 0
                    for n, v in zip(names, parts[5:9]):
                        if v.lower().startswith("active"):
                            r |= bits[n]
                    self.samples.append((sm, r))
            os.unlink(self.path)

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": ["no clock samples"], "samples": 0,
                    "source": self.source}
        reasons = set()
        for _, r in self.samples:
            for bit, name in NVML_REASONS.items():
                if r & bit:
                    reasons.add(name)
        return {"sm_mhz": statistics.median(s for s, _ in self.samples), "sm_max_mhz": self.max_mhz,
                "reasons": sorted(reasons), "samples": len(self.samples), "source": self.source}


# --------------------------------------------------------------------------
# workload
# --------------------------------------------------------------------------
def make_inputs(lay, seed_rank):
    import synth
    rank_lay = synth.layer(lay.name, seed=seed_rank)
    return rank_lay.x(), rank_lay.logits()


def algorithmic(T, d, E, k, F):
    """Algorithmic work of one forward per kernel: routed rows only (no pad
    rows), the method's own dataflow (x read once, codes written k times)."""
    R = T * k
    fp4 = lambda rows, K: rows * (K / 2 + K / 16)            # codes + block scales
    w1 = fp4(E * 2 * F, d) + E * 2 * F * 4
    w2 = fp4(E * d, F) + E * d * 4
    return dict(
        fc1_flops=2.0 * R * d * 2 * F,
        fc2_flops=2.0 * R * F * d,
        bytes_route=T * E * 4 + R * 12,                          # logits in; ids, weights, ranks out
        bytes_quant=T * d * 2 + fp4(R, d) + R * 4,               # x in once, k copies of codes, scales, g out
        bytes_fc1=fp4(R, d) + R * 4 + w1 + fp4(R, F) + R * 4,    # A in, W1 in, h out
        bytes_fc2=fp4(R, F) + R * 4 + w2 + R * d * 2,            # h in, W2 in, slots out
        bytes_reduce=R * d * 2 + T * d * 2)                      # slots in, out


class Forward:
    """One workload's device buffers and its forward (eager, timed with
    per-launch events, or captured once in a CUDA graph)."""

    def __init__(self, M, dev, x, lg, T, E, k, d, F, w1q, w2q, stream):
        import torch
        self.M, self.dev, self.x, self.lg = M, dev, x, lg
        self.T, self.E, self.k, self.d, self.F = T, E, k, d, F
        self.w1q, self.w2q, self.stream = w1q, w2q, stream
        self.out = torch.empty((T, d), dtype=torch.int16, device=dev)
        self.ws = M.forward_workspace(T, E, k, d, F, dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.graph = None

    def args(self):
        return (self.x, self.lg, self.T, self.E, self.k, self.d, self.F, self.w1q["codes"], self.w1q["sf"],
                self.w1q["g"], self.w2q["codes"], self.w2q["sf"], self.w2q["g"], self.out, self.ws)

    def eager(self):
        self.M.moe_expert_forward(*self.args(), self.status, self.stream)

    def timed(self, events):
        self.M.moe_expert_forward_timed(*self.args(), self.status, self.stream, events)

    def capture(self):
        import torch
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=self.stream):
            self.eager()
        self.graph = g

    def replay(self):
        self.graph.replay()

    def check(self):
        import torch
        torch.cuda.synchronize()
        if int(self.status.item()) != 0:
            raise RuntimeError("device status %#x" % int(self.status.item()))


def graph_median_ms(fwd, reps):
    """Median over `reps` graph replays, each between its own pair of
    events on the launching stream."""
    import torch
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    with torch.cuda.stream(fwd.stream):
        for a, b in ev:
            a.record(fwd.stream)
            fwd.replay()
            b.record(fwd.stream)
    torch.cuda.synchronize()
    return statistics.median(a.elapsed_time(b) for a, b in ev)


def per_kernel_ms(fwd, reps):
    """Mean device time of each of the forward's seven launches: events
    recorded by the library before the first launch and after each one."""
    import torch
    sets = [[torch.cuda.Event(enable_timing=True) for _ in range(8)] for _ in range(reps)]
    for evs in sets:
        fwd.timed(evs)
    torch.cuda.synchronize()
    return [statistics.fmean(evs[i].elapsed_time(evs[i + 1]) for evs in sets) for i in range(7)]


def kernel_rooflines(ms, alg, peaks, fp4_peak):
    """Each launch against the roofline that bounds it (achieved from the
    algorithmic bytes or FLOPs of one launch over its mean duration)."""
    hbm = peaks["hbm_gbs"]
    out = {}
    for name, t in zip(KERNELS, ms):
        out[name] = {"ms": round(t, 4)}
    def mem(name, nbytes):
        gbs = nbytes / (out[name]["ms"] * 1e-3) / 1e9
        out[name].update(bound="hbm", achieved_gbs=round(gbs, 1), frac_hbm=round(gbs / hbm, 4),
                         algorithmic_bytes=int(nbytes))
    def flops(name, f):
        tf = f / (out[name]["ms"] * 1e-3) / 1e12
        out[name].update(achieved_tflops=round(tf, 1), frac_fp4_peak=round(tf / fp4_peak, 4),
                         algorithmic_flops=int(f))
    mem("route_kernel", alg["bytes_route"])
    out["scan_kernel"]["bound"] = "latency"
    out["pad_rows_kernel"]["bound"] = "latency"
    mem("permute_quant_kernel", alg["bytes_quant"])
    flops("fc1_swiglu_kernel", alg["fc1_flops"])
    out["fc1_swiglu_kernel"]["bound"] = "tensor"
    mem("fc2_scatter_kernel", alg["bytes_fc2"])
    flops("fc2_scatter_kernel", alg["fc2_flops"])
    mem("unpermute_reduce_kernel", alg["bytes_reduce"])
    return out


def tiny_latency(dev, reps=200):
    """Per-forward latency of the tiny layer (T=256, d=256, E=8, top-2,
    d_ff=128), launch-bound: eager calls against one CUDA-graph replay per
    forward (the forward is captured once)."""
    import numpy as np
    import torch

    import nvfp4_w4a4_moe_top_gb300 as M
    import synth
    lay = synth.layer("tiny")
    T, E, k, d, F = lay.T, lay.E, lay.k, lay.d, lay.d_ff

    def to_dev(a):
        a = np.ascontiguousarray(a)
        return torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).to(dev)

    w1q, w2q = M.quantize_weights(to_dev(lay.w1())), M.quantize_weights(to_dev(lay.w2()))
    s = torch.cuda.Stream(dev)
    fwd = Forward(M, dev, to_dev(lay.x()), to_dev(lay.logits()), T, E, k, d, F, w1q, w2q, s)

    def per_call(fn):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        for _ in range(10):
            fn()
        e0.record(s)
        for _ in range(reps):
            fn()
        e1.record(s)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) * 1e3 / reps

    with torch.cuda.stream(s):
        fwd.eager()
    torch.cuda.synchronize()
    eager = per_call(fwd.eager)
    fwd.capture()
    with torch.cuda.stream(s):  # replay() launches on the current stream
        graph = per_call(fwd.replay)
    fwd.check()
    return {"workload": "tiny", "eager_us": round(eager, 2), "graph_us": round(graph, 2), "launches": 7}


def other_config(M, dev, name, seed, rank, reps, w1q=None, w2q=None):
    """Tokens/s of another workload (median of `reps` graph replays) with
    its per-kernel times; Qwen-shaped workloads reuse the headline's
    quantised weights (the same seeded weights)."""
    import numpy as np
    import torch

    import synth
    lay = synth.layer(name, seed=seed)
    T, E, k, d, F = lay.T, lay.E, lay.k, lay.d, lay.d_ff

    def to_dev(a):
        a = np.ascontiguousarray(a)
        return torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).to(dev)

    if w1q is None:
        w1q = M.quantize_weights(to_dev(lay.w1()))
        w2q = M.quantize_weights(to_dev(lay.w2()))
    x_np, lg_np = make_inputs(lay, shard_seed(seed, rank))
    s = torch.cuda.current_stream(dev)
    fwd = Forward(M, dev, to_dev(x_np), to_dev(lg_np), T, E, k, d, F, w1q, w2q, s)
    for _ in range(3):
        fwd.eager()
    fwd.check()
    fwd.capture()
    med = graph_median_ms(fwd, reps)
    ms = per_kernel_ms(fwd, max(5, reps // 5))
    fwd.check()
    counts = M.forward_views(fwd.ws, T, E, k, d, F)["counts"].cpu().numpy()
    alg = algorithmic(T, d, E, k, F)
    return {"workload": name, "T": T, "d": d, "E": E, "k": k, "d_ff": F,
            "value": round(T / (med * 1e-3), 1), "unit": UNIT, "ms_median_graph": round(med, 4),
            "forward_tflops": round((alg["fc1_flops"] + alg["fc2_flops"]) / (med * 1e-3) / 1e12, 1),
            "kernel_ms": {n: round(t, 4) for n, t in zip(KERNELS, ms)},
            "empty_experts": int((counts == 0).sum()), "max_group_rows": int(counts.max())}


def native(args):
    import numpy as np
    import torch

    import nvfp4_w4a4_moe_top_gb300 as M
    import synth
    from nvfp4_w4a4_moe_top_gb300 import build as B

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    # one non-default stream for all the work (graph capture needs one)
    torch.cuda.set_stream(torch.cuda.Stream(dev))
    B.build()
    lay = synth.layer(args.workload, seed=args.seed)
    T, E, k, d, F = lay.T, lay.E, lay.k, lay.d, lay.d_ff

    def to_dev(a):
        a = np.ascontiguousarray(a)
        if a.dtype == np.uint16:
            a = a.view(np.int16)
        return torch.from_numpy(a).to(dev)

    W1 = torch.stack([to_dev(lay.w1_expert(e)) for e in range(E)])
    W2 = torch.stack([to_dev(lay.w2_expert(e)) for e in range(E)])
    w1q, w2q = M.quantize_weights(W1), M.quantize_weights(W2)
    w1e, w2e = M.quantize_weights_per_expert(W1), M.quantize_weights_per_expert(W2)
    x_np, lg_np = make_inputs(lay, shard_seed(args.seed, rank))
    x, lg = to_dev(x_np), to_dev(lg_np)
    stream = torch.cuda.current_stream(dev)
    fwd = Forward(M, dev, x, lg, T, E, k, d, F, w1q, w2q, stream)
    out, ws, status = fwd.out, fwd.ws, fwd.status

    for _ in range(args.warmup):
        fwd.eager()
    fwd.check()
    fwd.capture()
    for _ in range(3):
        fwd.replay()
    fwd.check()

    # ---- headline: K graph replays of the forward on resident inputs,
    # device-timed on the launching stream ----
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
    except (AttributeError, RuntimeError):
        uuid = None
    with ClockSampler(local, uuid) as clk:
        ev0.record(stream)
        for _ in range(args.steps):
            fwd.replay()
        ev1.record(stream)
        torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    sec = ev0.elapsed_time(ev1) / 1e3
    sec_max = max_over_ranks(sec, world, dev)
    value = aggregate(T, args.steps, world, sec_max)
    clocks = clk.summary()
    fwd.check()
    median_ms = graph_median_ms(fwd, max(50, min(args.steps, 200)))

    # ---- each launch of the forward against its roofline ----
    peaks, peak_kind = load_peaks()
    fp4_peak = peaks["bf16_tflops"] * FP4_PER_BF16
    alg = algorithmic(T, d, E, k, F)
    kms = per_kernel_ms(fwd, max(10, min(args.steps, 50)))
    fwd.check()
    kernels = kernel_rooflines(kms, alg, peaks, fp4_peak)
    t_fc1 = kms[KERNELS.index("fc1_swiglu_kernel")] * 1e-3
    fc1_tflops = alg["fc1_flops"] / t_fc1 / 1e12
    sha = src_sha("gemm.cu", "common.cuh", "swiglu.cuh")
    tr = NCU_TRAFFIC.get("fc1")
    # ncu's DRAM bytes of one launch, valid only for the device code and the
    # workload they were captured on
    traffic = (tr["bytes_per_launch"] if tr and tr.get("src_sha") == sha and tr.get("workload") == args.workload
               else None)
    roofline = {"kernel": "fc1_swiglu_kernel", "bound": "tensor", "achieved": round(fc1_tflops, 1),
                "peak": round(fp4_peak, 1), "unit": "TFLOP/s", "frac": round(fc1_tflops / fp4_peak, 4),
                "traffic": traffic, "ms_per_launch": round(t_fc1 * 1e3, 4), "src_sha": sha,
                "algorithmic_bytes": int(alg["bytes_fc1"]),
                "peak_source": "%s bf16 burst x %g (nominal fp4:bf16)" % (peak_kind, FP4_PER_BF16)}
    fwd_sec = sec_max / args.steps
    forward = {"tflops": round((alg["fc1_flops"] + alg["fc2_flops"]) / fwd_sec / 1e12, 1),
               "frac_fp4_peak": round((alg["fc1_flops"] + alg["fc2_flops"]) / fwd_sec / 1e12 / fp4_peak, 4),
               "algorithmic_gb": round(sum(alg[n] for n in ["bytes_route", "bytes_quant", "bytes_fc1", "bytes_fc2",
                                                           "bytes_reduce"]) / 1e9, 3),
               "hbm_gbs_of_algorithmic_bytes": round(sum(alg[n] for n in ["bytes_route", "bytes_quant", "bytes_fc1",
                                                                        "bytes_fc2", "bytes_reduce"])
                                                    / fwd_sec / 1e9, 1)}

    # ---- the other workloads of the layer ----
    configs = {}
    if args.workload == "qwen64k":
        configs["qwen16k"] = other_config(M, dev, "qwen16k", args.seed, rank, 50, w1q, w2q)
    configs["small"] = other_config(M, dev, "small", args.seed, rank, 50)

    # ---- weight quantisation (once per optimizer step, outside the forward):
    # the per-row recipe and the per-expert recipe, W1 and W2 each call ----
    reps = max(5, min(args.steps, 50))

    def timed(fn):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        fn()
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(reps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / 1e3 / reps

    def quant_rows():
        M.moe_nvfp4_quantize_weights(W1, w1q["codes"], w1q["sf"], w1q["g"], status, stream)
        M.moe_nvfp4_quantize_weights(W2, w2q["codes"], w2q["sf"], w2q["g"], status, stream)

    def quant_expert():
        M.moe_nvfp4_quantize_weights_per_expert(W1, w1e["codes"], w1e["sf"], w1e["g"], w1e["amax_e"], status,
                                                 stream)
        M.moe_nvfp4_quantize_weights_per_expert(W2, w2e["codes"], w2e["sf"], w2e["g"], w2e["amax_e"], status,
                                                 stream)

    t_wq_row, t_wq_exp = timed(quant_rows), timed(quant_expert)
    wq_bytes = sum(W.numel() * 2 + W.numel() // 2 + W.numel() // 16 + W.shape[0] * W.shape[1] * 4 for W in (W1, W2))
    t_fwd_exp = timed(lambda: M.moe_expert_forward(x, lg, T, E, k, d, F, w1e["codes"], w1e["sf"], w1e["g"],
                                                   w2e["codes"], w2e["sf"], w2e["g"], out, ws, status, stream))
    t_fwd_gather = timed(lambda: M.moe_expert_forward_gather(x, lg, T, E, k, d, F, w1q["codes"], w1q["sf"], w1q["g"],
                                                             w2q["codes"], w2q["sf"], w2q["g"], out, ws, status,
                                                             stream))
    # ---- forward + straight-through BF16 backward of the layer (training
    # step; weights quantised beforehand, as for the forward) ----
    mc = M.m_cap(T, E, k)
    su = torch.empty((mc, 2 * F), dtype=torch.int16, device=dev)
    sh = torch.empty((mc, F), dtype=torch.int16, device=dev)
    dY = to_dev(synth.layer(args.workload, seed=shard_seed(args.seed, rank)).grad_out())
    gx = torch.empty((T, d), dtype=torch.float32, device=dev)
    gW1 = torch.empty((E, 2 * F, d), dtype=torch.float32, device=dev)
    gW2 = torch.empty((E, d, F), dtype=torch.float32, device=dev)
    gl = torch.empty((T, E), dtype=torch.float32, device=dev)
    gw = torch.empty((T, k), dtype=torch.float32, device=dev)
    bws = torch.empty(M.backward_workspace_bytes(T, E, k, d, F), dtype=torch.uint8, device=dev)
    fv = M.forward_views(ws, T, E, k, d, F)

    def fwd_train():
        M.moe_expert_forward_train(x, lg, T, E, k, d, F, w1q["codes"], w1q["sf"], w1q["g"], w2q["codes"], w2q["sf"],
                                   w2q["g"], out, ws, su, sh, status, stream)

    def bwd():
        M.moe_expert_backward(dY, x, T, E, k, d, F, W1, W2, w2q["codes"], w2q["sf"], w2q["g"], fv["topk_ids"],
                              fv["topk_w"], fv["offsets"], fv["row_to_token"], fv["token_slot_row"], su, sh,
                              fv["h_codes"], fv["h_sf"], fv["h_g"], gx, gW1, gW2, gl, gw, bws, status, stream)

    t_ftrain = timed(fwd_train)
    t_bwd = timed(bwd)
    t_fb = timed(lambda: (fwd_train(), bwd()))
    bwd_flops = 2.0 * (alg["fc1_flops"] + alg["fc2_flops"])  # dgrad + wgrad of both GEMMs
    del W1, W2, su, sh, bws, gW1, gW2
    latency = tiny_latency(dev)
    fb = {"value": round(T / t_fb, 1), "unit": UNIT, "ms_per_step": round(t_fb * 1e3, 4),
          "forward_train_ms": round(t_ftrain * 1e3, 4), "backward_ms": round(t_bwd * 1e3, 4),
          "backward_gemm_tflop": round(bwd_flops / 1e12, 3),
          "backward_bf16_tflops": round(bwd_flops / t_bwd / 1e12, 1),
          "backward_frac_of_bf16_peak": round(bwd_flops / t_bwd / 1e12 / peaks["bf16_tflops"], 4),
          "launches": 14, "workload": "forward with saved values + BF16 backward, dY ~ N(0, 1e-3)"}
    wq = lambda t: {"ms": round(t * 1e3, 4), "achieved": round(wq_bytes / t / 1e9, 1), "unit": "GB/s",
                    "frac": round(wq_bytes / t / 1e9 / peaks["hbm_gbs"], 4)}
    next_rows = {"weight_quant_per_row": dict(wq(t_wq_row), launches=4,
                                              note="per tensor: the encode, then the fix-up pass for rows with "
                                                   "extreme outer scales"),
                 "weight_quant_per_expert": dict(wq(t_wq_exp), launches=6,
                                                 note="two passes over W: expert amax, then encode (and the "
                                                      "fix-up pass)"),
                 "forward_per_expert_weights": {"value": round(T / t_fwd_exp, 1), "unit": UNIT,
                                                "ms_per_step": round(t_fwd_exp * 1e3, 4)},
                 "forward_gather_on_load": {"value": round(T / t_fwd_gather, 1), "unit": UNIT,
                                            "ms_per_step": round(t_fwd_gather * 1e3, 4),
                                            "note": "codes quantised once per token, FC1 A rows by tile::gather4"},
                 "algorithmic_bytes_weight_quant": int(wq_bytes), "forward_backward": fb}

    # ---- end to end through the public call with host buffers ----
    xh = torch.from_numpy(x_np.view(np.int16)).pin_memory()
    lgh = torch.from_numpy(lg_np).pin_memory()
    outh = torch.empty((T, d), dtype=torch.int16).pin_memory()
    e2e_steps = max(3, min(args.steps, 100))  # the pipeline's fill and drain (about 3 ms) spread over the steps

    def e2e_step():
        x.copy_(xh, non_blocking=True)
        lg.copy_(lgh, non_blocking=True)
        fwd.eager()
        outh.copy_(out, non_blocking=True)

    e2e_step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_serial_sec = e0.elapsed_time(e1) / 1e3
    # the public pipelined call: each step's copies overlap its neighbours'
    # forwards (host wall clock around submit ... synchronize)
    pipe = M.Pipeline(T, E, k, d, F, depth=2, device=dev)
    for _ in range(2):
        pipe.submit(xh, lgh, outh, w1q, w2q, status)
    pipe.synchronize()
    if world > 1:
        torch.distributed.barrier()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        pipe.submit(xh, lgh, outh, w1q, w2q, status)
    pipe.synchronize()
    e2e_sec = max_over_ranks(time.perf_counter() - t0, world, dev)
    pipe.close()
    e2e = {"value": round(aggregate(T, e2e_steps, world, e2e_sec), 1), "unit": UNIT,
           "api": "moe_pipeline_submit (copy-in, forward, copy-out on three streams, depth 2)",
           "serial_value": round(aggregate(T, e2e_steps, world, max_over_ranks(e2e_serial_sec, world, dev)), 1),
           "h2d_bytes_per_step": int(xh.numel() * 2 + lgh.numel() * 4), "d2h_bytes_per_step": int(outh.numel() * 2),
           "steps": e2e_steps}
    fwd.check()

    line = {"metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(sec_max / args.steps * 1e3, 4),
            "ms_median_graph": round(median_ms, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "nvfp4 (e2m1 x e2m1, fp32 accumulate, bf16 out)",
            "data": "synthetic (seeded; shapes and distributions of the Qwen3-30B-A3B expert layer)",
            "config": config_of(args.workload, lay, world),
            "gpu_launches": 7 * args.steps, "roofline": roofline, "kernels": kernels, "forward": forward,
            "clocks": clocks, "e2e": e2e, "configs": configs, "next_rows": next_rows, "latency_tiny": latency}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(lay, args)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def config_of(workload, lay, world):
    return {"workload": workload, "T": lay.T, "d": lay.d, "E": lay.E, "k": lay.k, "d_ff": lay.d_ff,
            "parallelism": "token data parallel x%d" % world,
            "l2": "inputs larger than L2 (no flush)", "timing": "CUDA-graph replays, CUDA events"}


# --------------------------------------------------------------------------
# the oracle on the host cores
# --------------------------------------------------------------------------
def oracle_weights(lay):
    import numpy as np
    import oracle
    w1 = [oracle.quantize_weights(lay.w1_expert(e)[None]) for e in range(lay.E)]
    w2 = [oracle.quantize_weights(lay.w2_expert(e)[None]) for e in range(lay.E)]
    cat = lambda qs: (np.concatenate([q[0] for q in qs]), np.concatenate([q[1] for q in qs]),
                      np.concatenate([q[2] for q in qs]))
    return cat(w1), cat(w2)


def cpu_baseline(lay, args, tokens=None):
    import oracle
    tokens = tokens or args.cpu_tokens
    w1q, w2q = oracle_weights(lay)
    x = lay.x_rows(range(tokens))
    lg = lay.logits_rows(range(tokens))
    t0 = time.perf_counter()
    oracle.moe_forward(x, lg, w1q, w2q, lay.k, lay.d_ff)
    sec = time.perf_counter() - t0
    return {"value": round(tokens / sec, 2), "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
            "sample": "first %d tokens of the %s workload, one oracle forward (weights quantised beforehand)"
                      % (tokens, args.workload),
            "single_thread": oracle_single_thread(args)}


def oracle_single_thread(args, tokens=256):
    """The oracle on one host thread, on the tiny and small layers (the first
    `tokens` tokens of each, weights quantised beforehand): the per-core
    figure beside the all-cores baseline."""
    import oracle
    import synth
    out = {}
    n0 = oracle.num_threads()
    for name in ("tiny", "small"):
        lay = synth.layer(name, seed=args.seed)
        w1q, w2q = oracle_weights(lay)
        n = min(tokens, lay.T)
        x, lg = lay.x_rows(range(n)), lay.logits_rows(range(n))
        oracle.set_num_threads(1)
        try:
            t0 = time.perf_counter()
            oracle.moe_forward(x, lg, w1q, w2q, lay.k, lay.d_ff)
            sec = time.perf_counter() - t0
        finally:
            oracle.set_num_threads(n0)
        out[name] = {"value": round(n / sec, 2), "unit": UNIT, "cores": 1,
                     "sample": "first %d tokens of the %s workload" % (n, name)}
    return out


def reference(args):
    """The oracle as the reference arm: W untimed + K timed steps, each step a
    bounded sample (n consecutive tokens) of the same workload.  n is the
    cpu_baseline's 1024 tokens unless the whole run would then pass about
    three minutes and a half, in which case it shrinks to fit (not below 256)."""
    import oracle
    import synth
    rank, world, _ = dist_env()
    if rank != 0:
        return
    lay = synth.layer(args.workload, seed=args.seed)
    w1q, w2q = oracle_weights(lay)

    def step(i, n):
        t0 = (i * n) % lay.T
        toks = [(t0 + j) % lay.T for j in range(n)]
        oracle.moe_forward(lay.x_rows(toks), lay.logits_rows(toks), w1q, w2q, lay.k, lay.d_ff)

    n = args.ref_tokens
    if n is None:
        per_tok = float("inf")
        for _ in range(2):  # the first call also pays the thread pool's start-up
            t0 = time.perf_counter()
            step(0, 256)
            per_tok = min(per_tok, (time.perf_counter() - t0) / 256)
        n = int(max(256, min(1024, 200.0 / max(per_tok, 1e-9) / (args.steps + args.warmup))))
        n = min(n, lay.T)
    for i in range(args.warmup):
        step(i, n)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(args.warmup + i, n)
    sec = time.perf_counter() - t0
    value = n * args.steps / sec
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(sec / args.steps * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "fp32 (oracle)",
            "data": "synthetic (seeded)", "config": config_of(args.workload, lay, world),
            "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "cores": oracle.num_threads(),
                             "kind": "oracle", "sample": "%d consecutive tokens per step" % n},
            "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--workload", default="qwen64k")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--cpu-tokens", type=int, default=1024)
    ap.add_argument("--ref-tokens", type=int, default=None,
                    help="tokens per reference step (default: 1024, fewer if the run would be long)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        reference(args)
    else:
        native(args)


if __name__ == "__main__":
    main()
