#!/usr/bin/env python3
"""MoE-layer throughput of the token-dispatch hot path on GB300.

One step = one pass of the whole layer over one batch: route -> permute ->
grouped FFN (gate/up + SwiGLU, then down) -> combine, every kernel this
library's.  Default workload: the OLMoE-shaped decode layer (hidden 2048,
64 experts, top-8, intermediate 1024, bf16) at T=64 tokens, with T=1 and
T=8 reported beside it.  Inputs are seeded synthetic tensors; expert
weights (805 MB) exceed the 129 MB L2 and L2 is flushed between steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME]

Prints one JSON line (rank 0).  With --gpus N > 1 (launched by torchrun)
every rank runs an independent replica on its own batch (the layer has no
cross-GPU exchange on one GPU per expert set), value = all tokens / max
rank time.  --impl reference times the CPU oracle on the host cores.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE-layer tokens/s and µs/layer at T=1..2048; % of HBM BW (decode) / tensor peak"
UNIT = "tokens/s"
L2_FLUSH_BYTES = 256 << 20

# name -> (shape config, T, routing, extra T values measured beside it)
WORKLOADS = {
    "olmoe_decode_t64": ("olmoe", 64, "uniform", (1, 8)),
    "olmoe_decode_t8": ("olmoe", 8, "uniform", ()),
    "olmoe_decode_t1": ("olmoe", 1, "uniform", ()),
    "olmoe_t2048": ("olmoe", 2048, "uniform", (128, 512)),
    "deepseek_t2048": ("deepseek", 2048, "uniform", (1, 16, 128, 512)),
    "deepseek_t2048_zipf": ("deepseek", 2048, "zipf", (1, 16, 128, 512)),
}
DEFAULT_WORKLOAD = "olmoe_decode_t64"

CLOCK_FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


# ----------------------------------------------------------------- helpers

def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def reduce_max(value: float, world: int, device=None) -> float:
    """Max of a per-rank float over all ranks (identity at world size 1)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def aggregate_value(tokens_per_rank: float, world: int, max_seconds: float) -> float:
    """Whole-job tokens/s: tokens of every rank over the slowest rank's time."""
    return tokens_per_rank * world / max_seconds


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return dict(hbm_gbs=float(p["hbm_gbs"]), bf16_tflops=float(p["bf16_tflops"]),
                    bf16_tflops_sustained=float(p.get("bf16_tflops_sustained",
                                                      p["bf16_tflops"])), source="measured")
    except (OSError, KeyError, ValueError):
        return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0,
                    source="fallback")


# The CUDA sources behind each kernel named in a roofline object (with the
# headers they include): a committed traffic figure is used only while these
# are unchanged since the counters were taken.
KERNEL_SOURCES = {
    "tc_grouped_gemm_swiglu": ("gemm_tc.cu", "gemm_tc_pair.cu", "tc_common.cuh", "tc_pair.cuh",
                               "common.cuh"),
    "tc_grouped_gemm_dec_w8": ("gemm_tc_dec_w8.cu", "gemm_tc_w8.cu", "gemm_tc.cu", "tc_w8.cuh",
                               "tc_common.cuh", "common.cuh"),
    "decode_layer_kernel": ("decode_layer.cu", "gemv_tasks.cuh", "route_token.cuh",
                            "common.cuh"),
    "gemv_gateup_bf16": ("gemv.cu", "gemv_tasks.cuh", "common.cuh"),
}


def kernel_source_hash(kernel: str) -> str:
    """Hash of the CUDA sources of `kernel` (every source if it is not listed)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "grouped_expert_gemm_moe_gb300", "csrc")
    names = KERNEL_SOURCES.get(kernel) or sorted(
        f for f in os.listdir(csrc) if f.endswith((".cu", ".cuh")))
    for f in names:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode())
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel: str, workload: str):
    """dram bytes per launch from the committed ncu summary, if it was taken
    on the current sources of that kernel; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        e = d[f"{kernel}@{workload}"]
        if e.get("source_hash") != kernel_source_hash(kernel):
            return None
        return float(e["dram_bytes_per_launch"])
    except (OSError, KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons every 100 ms; stop(t0, t1)
    keeps the samples taken inside the wall-clock window [t0, t1]."""

    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_index: int):
        import tempfile
        self.proc = None
        self.fh = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={gpu_index}", f"--query-gpu={CLOCK_FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.fh,
                stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    @staticmethod
    def _ts(text):
        import datetime
        for fmt in ("%Y/%m/%d %H:%M:%S.%f", "%Y/%m/%d %H:%M:%S"):
            try:
                return datetime.datetime.strptime(text, fmt).timestamp()
            except ValueError:
                pass
        return None

    def stop(self, t0: float, t1: float):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        rows = []
        with open(self.fh.name) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 10:
                    rows.append(parts)
        os.remove(self.fh.name)
        inside = [r for r in rows if (ts := self._ts(r[0])) is not None and t0 <= ts <= t1]
        use = inside if inside else rows

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [v for r in use if (v := num(r[2])) is not None]
        mx = [v for r in use if (v := num(r[3])) is not None]
        reasons = sorted({self.REASONS[i] for r in use for i in range(4)
                          if r[6 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(use), "samples_in_timed_region": len(inside)}


class NvmlSampler:
    """SM clock, max SM clock and clock-event reasons every ~1 ms from a
    host thread through NVML's C API (the driver's libnvidia-ml.so.1, loaded
    with ctypes), so that a timed region of a few milliseconds still holds
    samples; stop(t0, t1) keeps the samples inside the wall-clock window.
    `ok` is False when NVML cannot be used (ClockSampler is used then)."""

    # nvmlClocksEventReasons bits
    BITS = {"sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20,
            "hw_thermal_slowdown": 0x40}

    def __init__(self, gpu_index: int, period_s: float = 0.001):
        import ctypes
        import threading
        self.ok = False
        self.samples = []
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                return
            h = ctypes.c_void_p()
            if nv.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(gpu_index), ctypes.byref(h)) != 0:
                return
            reasons_fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                getattr(nv, "nvmlDeviceGetCurrentClocksThrottleReasons")
        except (OSError, AttributeError):
            return
        self.nv, self.h, self.reasons_fn = nv, h, reasons_fn
        mx = ctypes.c_uint(0)
        self.max_mhz = (float(mx.value) if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx))
                        == 0 else None)
        self.period = period_s
        self.stop_flag = threading.Event()
        self.thread = threading.Thread(target=self._run, daemon=True)
        self.ok = True
        self.thread.start()

    def _run(self):
        import ctypes
        mhz = ctypes.c_uint(0)
        rs = ctypes.c_ulonglong(0)
        while not self.stop_flag.is_set():
            t = time.time()
            a = self.nv.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(mhz))   # NVML_CLOCK_SM
            b = self.reasons_fn(self.h, ctypes.byref(rs))
            if a == 0 and b == 0:
                self.samples.append((t, float(mhz.value), int(rs.value)))
            time.sleep(self.period)

    def stop(self, t0: float, t1: float):
        if not self.ok:
            return None
        self.stop_flag.set()
        self.thread.join(timeout=5)
        inside = [x for x in self.samples if t0 <= x[0] <= t1]
        use = inside if inside else self.samples
        sm = [x[1] for x in use]
        reasons = sorted({name for x in use for name, bit in self.BITS.items() if x[2] & bit})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": self.max_mhz,
                "reasons": reasons, "samples": len(use), "samples_in_timed_region": len(inside),
                "source": "NVML, ~1 ms period"}


# ------------------------------------------------------------ workload

def build_workload(name, device, seed):
    from grouped_expert_gemm_moe_gb300 import workloads as W
    from grouped_expert_gemm_moe_gb300.layer import MoELayer
    cfg, T, routing, extra = WORKLOADS[name]
    shape = W.CONFIGS[cfg]
    inp = W.make_layer(shape, T, routing, seed=seed, device=device)
    layer = MoELayer(shape.H, shape.E, shape.k, shape.I, shape.S, shape.renormalize,
                     w_gu=inp.w_gu, w_down=inp.w_down, device=device)
    return shape, T, routing, extra, inp, layer


def extra_batch(shape, T, routing, seed, device, inp):
    """Another batch (x, logits) for the same layer weights."""
    import torch
    from grouped_expert_gemm_moe_gb300 import workloads as W
    g = W.make_generator(seed + 7919 * T, device)
    x = torch.randn((T, shape.H), generator=g, device=device).to(torch.bfloat16)
    return x, W.router_logits_input(x, inp.w_r, inp.bias)


class Phases:
    """One layer step recorded as three CUDA graphs -- [route, permute],
    [gate/up] (bf16 experts; the whole FFN for int8 experts, whose two GEMMs
    are one call), [down, combine] -- so the dominant kernel can be timed
    with events between graph launches inside the timed region."""

    def __init__(self, layer, x, logits, kind):
        import torch
        self.layer, self.kind = layer, kind
        b = self.b = layer.buffers(x.shape[0])

        def pre():
            layer.route_permute(logits, x, b)

        def mid():
            if layer.int8:
                layer.ffn(b, kind)
            else:
                layer.gate_up(b, kind)

        def post():
            if not layer.int8:
                layer.down(b, kind)
            layer.combine(b, b.out)

        self.graphs = []
        for fn in (pre, mid, post):
            fn()                                   # eager pass: attributes set outside capture
        torch.cuda.synchronize()
        for fn in (pre, mid, post):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, capture_error_mode="thread_local"):
                fn()
            self.graphs.append(g)
        torch.cuda.synchronize()

    def run(self, ev=None):
        g0, g1, g2 = self.graphs
        if ev is None:
            g0.replay(); g1.replay(); g2.replay()
            return
        s, k0, k1, e = ev
        s.record()
        g0.replay()
        k0.record()
        g1.replay()
        k1.record()
        g2.replay()
        e.record()


def kernels_per_step(layer, T, kind="auto"):
    """Kernels of one layer step: the single-launch decode layer is 1;
    otherwise route + permute (1 fused launch for small batches; else the
    routing kernel plus 1 permute kernel up to 1024 slots or 3 above), then
    gate/up, down and combine."""
    if kind == "decode":
        return 1
    if layer.fused_route_permute_ok(T):
        rp = 1
    else:
        rp = 1 + (1 if T * layer.k <= 1024 else 3)
    return rp + 3


def touched_groups(layer, b):
    import numpy as np
    off = b.offsets.cpu().numpy()
    return int(np.count_nonzero(np.diff(off) > 0))


def time_graph(cap, K, W, flush):
    """W warm-up steps, then K timed steps of a captured forward pass, L2
    flushed before each step; per-step device times (ms)."""
    import torch
    for _ in range(W):
        flush.zero_()
        cap.replay()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(K)]
    for a, b in evs:
        flush.zero_()
        a.record()
        cap.replay()
        b.record()
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in evs]


def time_steps(phases, K, W, flush):
    """W warm-up steps, then K timed steps, L2 flushed before each step.
    Returns per-step and per-gate/up-launch device times (ms)."""
    import torch
    for _ in range(W):
        flush.zero_()
        phases.run()
    torch.cuda.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    for i in range(K):
        flush.zero_()
        phases.run(evs[i])
    torch.cuda.synchronize()
    step = [e[0].elapsed_time(e[3]) for e in evs]
    gate_up = [e[1].elapsed_time(e[2]) for e in evs]
    return step, gate_up


def weight_bytes_per_group(shape, int8: bool) -> int:
    """Algorithmic weight bytes of one served group: bf16 3*H*I*2; int8
    3*H*I plus the fp32 scales of its 2I + H output rows."""
    H, I = shape.H, shape.I
    return 3 * H * I + (2 * I + H) * 4 if int8 else 3 * H * I * 2


def layer_roofline(shape, T, n_groups, peaks, int8=False):
    """Ideal layer time: max(FLOPs / bf16 peak, algorithmic bytes / HBM BW).
    Bytes: weights of served groups + x in + out (T*H*2 each); FLOPs:
    6*H*I per served row (routed slots + shared rows)."""
    H, I = shape.H, shape.I
    bytes_ = n_groups * weight_bytes_per_group(shape, int8) + 2 * T * H * 2
    flops = 6.0 * H * I * shape.rows(T)
    t_mem = bytes_ / (peaks["hbm_gbs"] * 1e9)
    t_flop = flops / (peaks["bf16_tflops"] * 1e12)
    return dict(bytes=bytes_, flops=flops, t_roof_us=max(t_mem, t_flop) * 1e6,
                bound="hbm" if t_mem >= t_flop else "tensor")


def kernel_roofline(shape, T, n_groups, gate_up_ms, peaks, kind, workload, int8=False):
    """Roofline of the dominant kernel.  bf16: the gate/up GEMM, whose
    algorithmic bytes are the gate and up weights of the served groups
    (2*I*H*2 per group) and whose FLOPs are 4*H*I per served row.  int8:
    the whole FFN (both GEMMs are one call), bytes as weight_bytes_per_group,
    FLOPs 6*H*I per served row.  Both fractions are given; `bound` names the
    one the roofline says limits it."""
    H, I = shape.H, shape.I
    if int8:
        bytes_ = n_groups * weight_bytes_per_group(shape, True)
        flops = 6.0 * H * I * shape.rows(T)
        name = "tc_grouped_gemm_dec_w8" if kind == "gemm" else "gemv_gateup_w8"
    else:
        bytes_ = n_groups * 2 * I * H * 2
        flops = 4.0 * H * I * shape.rows(T)
        name = "tc_grouped_gemm_swiglu" if kind == "gemm" else "gemv_gateup_bf16"
    sec = gate_up_ms / 1e3
    t_mem = bytes_ / (peaks["hbm_gbs"] * 1e9)
    t_flop = flops / (peaks["bf16_tflops"] * 1e12)
    traffic = profiled_traffic(name, workload)
    gbs = bytes_ / sec / 1e9
    tfs = flops / sec / 1e12
    both = {"hbm_frac": round(gbs / peaks["hbm_gbs"], 4),
            "tensor_frac": round(tfs / peaks["bf16_tflops"], 4),
            "hbm_frac_of_nominal_8tbs": round(gbs / 8000.0, 4)}
    if t_mem >= t_flop:
        return {"kernel": name, "bound": "hbm", "achieved": round(gbs, 1),
                "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": both["hbm_frac"],
                "traffic": traffic, "algorithmic_bytes": bytes_, **both,
                "avg_launch_us": round(gate_up_ms * 1e3, 2),
                "peak_source": f"{peaks['source']} (STREAM copy, burst)"}
    return {"kernel": name, "bound": "tensor", "achieved": round(tfs, 1),
            "peak": peaks["bf16_tflops"], "unit": "TFLOP/s", "frac": both["tensor_frac"],
            "traffic": traffic, "algorithmic_flops": flops, "algorithmic_bytes": bytes_,
            **both, "avg_launch_us": round(gate_up_ms * 1e3, 2),
            "peak_source": f"{peaks['source']} (cuBLAS bf16, burst)"}


def measure_T(layer, shape, T, x, logits, K, W, flush, peaks, workload, ffn="auto"):
    """Layer time from K steps of the whole forward pass captured in one
    CUDA graph; the dominant kernel's time from K further steps recorded as
    three graphs with events around it.  ffn: "auto" (the layer's own
    choice) or a forced "decode", "gemv" or "gemm"."""
    kind = layer.choose_path(T, x.dtype) if ffn == "auto" else ffn
    if kind == "decode" and not layer.decode_layer_ok(T, x.dtype):
        raise SystemExit(f"--ffn decode: T={T} is outside the fused decode layer's limits")
    cap = layer.capture(x, logits, ffn=kind)
    step = time_graph(cap, K, W, flush)
    ms = statistics.fmean(step)
    if kind == "decode":
        # one kernel is the whole layer: its roofline is the layer's
        b = layer.buffers(T)
        layer.route(logits, b)
        layer.permute(x, b)
        n_groups = touched_groups(layer, b)
        roof = layer_roofline(shape, T, n_groups, peaks)
        return dict(kind=kind, step_ms=step, gate_up_ms=ms, ms=ms, n_groups=n_groups, roof=roof,
                    kroof=decode_kernel_roofline(shape, T, n_groups, ms, peaks, workload))
    ph = Phases(layer, x, logits, kind)
    _, gu = time_steps(ph, K, W, flush)
    n_groups = touched_groups(layer, ph.b)
    roof = layer_roofline(shape, T, n_groups, peaks, layer.int8)
    return dict(kind=kind, step_ms=step, gate_up_ms=statistics.fmean(gu), ms=ms,
                n_groups=n_groups, roof=roof,
                kroof=kernel_roofline(shape, T, n_groups, statistics.fmean(gu), peaks, kind,
                                      workload, layer.int8))


def decode_kernel_roofline(shape, T, n_groups, step_ms, peaks, workload):
    """Roofline of the single-launch decode layer: its algorithmic bytes are
    all weights of the served groups (3*H*I*2 each) plus x in and out; the
    step time is the kernel's (plus a 4-byte memset node)."""
    H, I = shape.H, shape.I
    bytes_ = n_groups * 3 * H * I * 2 + 2 * T * H * 2
    ach = bytes_ / (step_ms / 1e3) / 1e9
    return {"kernel": "decode_layer_kernel", "bound": "hbm", "achieved": round(ach, 1),
            "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": round(ach / peaks["hbm_gbs"], 4),
            "hbm_frac": round(ach / peaks["hbm_gbs"], 4),
            "hbm_frac_of_nominal_8tbs": round(ach / 8000.0, 4),
            "traffic": profiled_traffic("decode_layer_kernel", workload),
            "algorithmic_bytes": bytes_, "avg_launch_us": round(step_ms * 1e3, 2),
            "peak_source": f"{peaks['source']} (STREAM copy, burst)"}


def e2e_measure(layer, shape, T, inp, K, W, flush, ffn="auto"):
    """End to end through the public API: pinned host x and logits copied in,
    the forward pass, the output copied back, every step -- one CUDA graph
    (MoELayer.capture_host) holding the copies and the kernels."""
    import torch
    x_host = inp.x.detach().cpu().pin_memory()
    l_host = inp.logits.detach().cpu().pin_memory()
    cap = layer.capture_host(x_host, l_host, ffn=ffn)

    for _ in range(W):
        flush.zero_()
        cap.replay()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(K)]
    for i in range(K):
        flush.zero_()
        evs[i][0].record()
        cap.replay()
        evs[i][1].record()
    torch.cuda.synchronize()
    ms = statistics.fmean(a.elapsed_time(b) for a, b in evs)
    h2d = x_host.numel() * x_host.element_size() + l_host.numel() * l_host.element_size()
    d2h = cap.out_host.numel() * cap.out_host.element_size()
    return ms, h2d, d2h, cap.out_host.clone()


# The sweep of other_rows: (row prefix, shape config, routing, token counts,
# int8 experts).  The token counts are the configs' own: OLMoE decode 1/8/64
# (and the 2048-token prefill), DeepSeek 1..2048 under uniform and zipf
# routing, OLMoE int8 at 7 token counts under both routings, and the DeepSeek
# shapes in int8 as the secondary sweep.
SWEEP = (
    ("olmoe", "olmoe", "uniform", (1, 8, 64, 2048), False),
    ("deepseek", "deepseek", "uniform", (1, 16, 128, 512, 2048), False),
    ("deepseek_zipf", "deepseek", "zipf", (1, 16, 128, 512, 2048), False),
    ("olmoe_int8", "olmoe", "uniform", (1, 8, 16, 64, 128, 512, 2048), True),
    ("olmoe_int8_zipf", "olmoe", "zipf", (1, 8, 16, 64, 128, 512, 2048), True),
    ("deepseek_int8", "deepseek", "uniform", (1, 16, 128, 512, 2048), True),
    ("deepseek_int8_zipf", "deepseek", "zipf", (1, 16, 128, 512, 2048), True),
)


def row_of(m, T):
    """One table row from measure_T's result."""
    kr = m["kroof"]
    row = {"us_per_layer": round(m["ms"] * 1e3, 2),
           "tokens_per_s": round(T / (m["ms"] / 1e3), 1), "ffn": m["kind"],
           "groups": m["n_groups"], "layer_bound": m["roof"]["bound"],
           "layer_t_roof_us": round(m["roof"]["t_roof_us"], 2),
           "layer_roofline_frac": round(m["roof"]["t_roof_us"] / (m["ms"] * 1e3), 4)}
    label = ("layer" if m["kind"] == "decode" else
             "ffn" if kr["kernel"].endswith("_w8") else "gate_up")
    row[f"{label}_us"] = kr["avg_launch_us"]
    row[f"{label}_hbm_frac"] = kr.get("hbm_frac", kr["frac"])
    row[f"{label}_hbm_frac_of_nominal_8tbs"] = kr.get("hbm_frac_of_nominal_8tbs")
    if "tensor_frac" in kr:
        row[f"{label}_tensor_frac"] = kr["tensor_frac"]
    return row


def sweep_rows(dev, K, W, flush, peaks):
    """Every (layer, routing, T) of SWEEP: the layer built once per shape and
    weight type (seed 0), a fresh seeded batch per T, each T timed like the
    headline (whole layer in one graph; the dominant kernel by events around
    its own graph).  Steps capped at 100 per row."""
    import torch

    from grouped_expert_gemm_moe_gb300 import binding as B
    from grouped_expert_gemm_moe_gb300 import workloads as WL
    from grouped_expert_gemm_moe_gb300.layer import MoELayer
    rows = {}
    K2 = max(3, min(K, 100))
    built = {}
    for prefix, cfg, routing, Ts, int8 in SWEEP:
        key = (cfg, int8)
        if key not in built:
            built.clear()
            torch.cuda.empty_cache()
            sh = WL.CONFIGS[cfg]
            inp = WL.make_layer(sh, 1, "uniform", seed=0, device=dev)
            if int8:
                q_gu, s_gu = B.moe_quantize_w8(inp.w_gu)
                q_down, s_down = B.moe_quantize_w8(inp.w_down)
                layer = MoELayer(sh.H, sh.E, sh.k, sh.I, sh.S, sh.renormalize,
                                 q_gu=q_gu.to(dev), s_gu=s_gu.to(dev), q_down=q_down.to(dev),
                                 s_down=s_down.to(dev), device=dev)
                inp.w_gu = inp.w_down = None
            else:
                layer = MoELayer(sh.H, sh.E, sh.k, sh.I, sh.S, sh.renormalize, w_gu=inp.w_gu,
                                 w_down=inp.w_down, device=dev)
            built[key] = (sh, inp, layer)
        sh, inp, layer = built[key]
        bias = WL.routing_bias(sh, routing)
        for T in Ts:
            g = WL.make_generator(1000 + T, dev)
            x = torch.randn((T, sh.H), generator=g, device=dev).to(torch.bfloat16)
            logits = WL.router_logits_input(x, inp.w_r, None if bias is None else bias.to(dev))
            m = measure_T(layer, sh, T, x, logits, K2, W, flush, peaks, f"{prefix}_t{T}")
            layer.check()
            rows[f"{prefix}_t{T}"] = {**row_of(m, T), "steps": K2}
        layer._bufs.clear()
    built.clear()
    torch.cuda.empty_cache()
    return rows


def other_rows(dev, K, W, flush, peaks):
    """The capacity-limited (token-dropping) layer at the pages' 4x load
    skew (T=2048, dropless / CF 2.0 / CF 1.0) and the 16-layer OLMoE-shaped
    stack (skewed routing, T=64 and T=2048), each captured in one CUDA graph
    and timed like the main workload: W warm-up steps, then K (capped for the
    long stack steps) timed steps with L2 flushed before each.  Rooflines:
    weight bytes of the served groups at HBM bandwidth vs FLOPs at the bf16
    peak (sustained for the stack, whose steps run for milliseconds), per
    layer, summed over the stack."""
    import numpy as np
    import torch

    from grouped_expert_gemm_moe_gb300 import workloads as WL
    from grouped_expert_gemm_moe_gb300.layer import MoELayer, MoEStack
    rows = {}
    bw = peaks["hbm_gbs"] * 1e9

    # token dropping at the pages' load skew (busiest expert ~4x the mean),
    # OLMoE layer, T=2048: dropless vs capacity factors 2.0 and 1.0
    sh = WL.OLMOE
    T = 2048
    inp = WL.make_layer(sh, T, "skew4", seed=0, device=dev)
    for cf in (None, 2.0, 1.0):
        layer = MoELayer(sh.H, sh.E, sh.k, sh.I, 0, False, w_gu=inp.w_gu, w_down=inp.w_down,
                         device=dev, capacity_factor=cf)
        cap = layer.capture(inp.x, inp.logits, ffn="gemm")
        K2 = max(3, min(K, 200))
        ms = statistics.fmean(time_graph(cap, K2, W, flush))
        layer.check()
        b = layer.buffers(T)
        off = b.offsets.cpu().numpy()
        served = int(off[sh.E])
        ng = int(np.count_nonzero(np.diff(off[:sh.E + 1]) > 0))
        H, I = sh.H, sh.I
        bytes_ = ng * 3 * H * I * 2 + 2 * T * H * 2
        flops = 6.0 * H * I * served
        t_roof = max(bytes_ / bw, flops / (peaks["bf16_tflops"] * 1e12)) * 1e6
        rows[f"capacity_{'dropless' if cf is None else f'cf{cf:g}'}_t2048_skew4"] = {
            "us_per_layer": round(ms * 1e3, 2), "tokens_per_s": round(T / (ms / 1e3), 1),
            "capacity": b.capacity, "dropped_slots": int(b.dropped.item()) if cf else 0,
            "dropped_frac": round((T * sh.k - served) / (T * sh.k), 4), "steps": K2,
            "t_roof_us": round(t_roof, 2), "roofline_frac": round(t_roof / (ms * 1e3), 4)}
        del layer, cap
    del inp
    torch.cuda.empty_cache()

    sh = WL.OLMOE_STACK
    for T, K2 in ((64, min(K, 200)), (2048, min(K, 20))):
        K2 = max(K2, 3)
        x0, layers_w, bias = WL.make_stack(sh, T, "skew4", seed=0, device=dev)
        layers = [MoELayer(sh.H, sh.E, sh.k, sh.I, 0, False, w_gu=wg, w_down=wd, device=dev)
                  for (_, wg, wd) in layers_w]
        stack = MoEStack(layers, [wr for (wr, _, _) in layers_w], bias)
        cap = stack.capture(x0)
        ms = statistics.fmean(time_graph(cap, K2, W, flush))
        for ly in layers:
            ly.check()
        H, I, E, k = sh.H, sh.I, sh.E, sh.k
        t_roof = 0.0
        groups = []
        for ly in layers:
            ng = touched_groups(ly, ly.buffers(T))
            groups.append(ng)
            b_l = ng * 3 * H * I * 2 + 3 * T * H * 2 + E * H * 2
            f_l = 6.0 * H * I * T * k + 2.0 * T * H * E
            t_roof += max(b_l / bw, f_l / (peaks["bf16_tflops_sustained"] * 1e12))
        t_roof *= 1e6
        rows[f"stack16_t{T}"] = {
            "us_per_step": round(ms * 1e3, 1), "us_per_layer": round(ms * 1e3 / sh.layers, 2),
            "tokens_per_s": round(T / (ms / 1e3), 1), "steps": K2,
            "groups_per_layer": groups, "t_roof_us": round(t_roof, 1),
            "roofline_frac": round(t_roof / (ms * 1e3), 4)}
        del stack, layers, layers_w, cap
        torch.cuda.empty_cache()
    return rows


# ------------------------------------------------------------ oracle legs

def oracle_sample(inp, tokens):
    """The oracle's view of the given tokens: fp32 logits and x (fp32, or
    bf16 bit patterns)."""
    import numpy as np
    import torch

    from grouped_expert_gemm_moe_gb300 import workloads as W
    logits = inp.logits.detach().cpu().numpy()[tokens]
    xb = inp.x.detach().cpu()
    x = xb.numpy()[tokens] if xb.dtype == torch.float32 else W.bf16_bits(xb)[tokens]
    return dict(logits=np.ascontiguousarray(logits), x=np.ascontiguousarray(x))


def run_oracle_tokens(inp, host, tokens, wbits, nthreads=0):
    import oracle
    sh = inp.shape
    ids, w = oracle.route(host["logits"], sh.k, sh.renormalize)
    oracle.permute(ids, sh.E, sh.S)
    return oracle.moe_layer(host["x"], ids, w, sh.E, sh.S, wbits[0], wbits[1],
                            nthreads=nthreads)


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo), for the record."""
    import subprocess
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu part")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def cpu_baseline(inp, gpu_out, min_seconds=10.0, min_seconds_1_thread=2.0):
    """The oracle, as it stands, on the host cores: route + permute + layer
    of every token of the batch, repeated until at least min_seconds of
    work have run; also the parity gate of the bench: a GPU result that
    disagrees with it (on any token) is not timed."""
    import numpy as np

    import oracle
    from grouped_expert_gemm_moe_gb300 import workloads as W
    T = inp.T
    tokens = np.arange(T)
    host = oracle_sample(inp, tokens)
    wbits = (W.bf16_bits(inp.w_gu), W.bf16_bits(inp.w_down))
    t0 = time.perf_counter()
    y = run_oracle_tokens(inp, host, tokens, wbits)
    sec = time.perf_counter() - t0
    reps = 1
    while sec < min_seconds:
        t0 = time.perf_counter()
        run_oracle_tokens(inp, host, tokens, wbits)
        sec += time.perf_counter() - t0
        reps += 1
    got = gpu_out.float().cpu().numpy().astype(np.float64)[tokens]
    rel = float(np.linalg.norm(got - y) / np.linalg.norm(y))
    mx = float(np.abs(got - y).max() / np.abs(y).max())
    cores = min(len(tokens), oracle.num_threads())
    # the same oracle on one thread, for scale (a few tokens, repeated)
    t1 = tokens[:min(len(tokens), 4)]
    h1 = oracle_sample(inp, t1)
    sec1, reps1 = 0.0, 0
    while sec1 < min_seconds_1_thread:
        t0 = time.perf_counter()
        run_oracle_tokens(inp, h1, t1, wbits, nthreads=1)
        sec1 += time.perf_counter() - t0
        reps1 += 1
    return dict(value=round(reps * len(tokens) / sec, 3), unit=UNIT, cores=cores, kind="oracle",
                cpu=cpu_model(),
                sample=f"route+permute+layer of all {len(tokens)} tokens of the timed batch, "
                       f"{reps} times ({sec:.1f} s)",
                value_1_thread=round(reps1 * len(t1) / sec1, 3),
                sample_1_thread=f"tokens 0..{len(t1) - 1} on one thread, {reps1} times "
                                f"({sec1:.1f} s)",
                parity={"rel_frobenius": rel, "max_rel": mx, "ok": rel <= 5e-3 and mx <= 2e-2})


# ------------------------------------------------------------------ arms

def run_ours(args):
    import torch
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    peaks = load_peaks()
    shape, T, routing, extra, inp, layer = build_workload(args.workload, dev, seed=rank)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    # correctness first: one pass, checked against the oracle before timing
    out0 = layer.forward(inp.x, inp.logits, ffn=args.ffn).clone()
    layer.check()
    base = None
    if rank == 0 and world == 1:
        base = cpu_baseline(inp, out0)
        if not base["parity"]["ok"]:
            print(json.dumps({"error": "GPU result disagrees with the oracle; not timed",
                              "parity": base["parity"]}))
            sys.exit(1)

    sampler = None
    if rank == 0:
        sampler = NvmlSampler(local)
        if not sampler.ok:
            sampler = ClockSampler(local)
            time.sleep(0.5)                     # let nvidia-smi start sampling
    barrier(world)
    torch.cuda.synchronize()
    t_wall0 = time.time()
    m = measure_T(layer, shape, T, inp.x, inp.logits, args.steps, args.warmup, flush, peaks,
                  args.workload, args.ffn)
    torch.cuda.synchronize()
    barrier(world)
    t_wall1 = time.time()
    clocks = sampler.stop(t_wall0, t_wall1) if sampler is not None else None
    layer.check()

    sec = reduce_max(sum(m["step_ms"]) / 1e3, world, dev)
    value = aggregate_value(T * args.steps, world, sec)
    ms_per_step = sec * 1e3 / args.steps

    per_T = {}
    for t2 in extra:
        x2, l2 = extra_batch(shape, t2, routing, rank, dev, inp)
        m2 = measure_T(layer, shape, t2, x2, l2, args.steps, args.warmup, flush, peaks,
                       args.workload)
        per_T[str(t2)] = {"us_per_layer": round(m2["ms"] * 1e3, 2),
                          "tokens_per_s": round(t2 / (m2["ms"] / 1e3), 1), "ffn": m2["kind"],
                          "roofline_frac": round(m2["roof"]["t_roof_us"] / (m2["ms"] * 1e3), 4),
                          "gate_up_frac": m2["kroof"]["frac"], "groups": m2["n_groups"]}
    layer.check()

    rows = sweep = None
    if world == 1 and not args.no_rows:
        sweep = sweep_rows(dev, args.steps, args.warmup, flush, peaks)
        rows = other_rows(dev, args.steps, args.warmup, flush, peaks)

    e2e_ms, h2d, d2h, out_e2e = e2e_measure(layer, shape, T, inp, args.steps, args.warmup, flush,
                                            m["kind"])
    layer.check()
    e2e_sec = reduce_max(e2e_ms * args.steps / 1e3, world, dev)
    if not torch.equal(out_e2e.to(dev), out0):
        print(json.dumps({"error": "end-to-end output differs from the first pass"}))
        sys.exit(1)

    if rank == 0:
        roof = m["roof"]
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0,1) activations, N(0,0.02) bf16 expert weights)",
            "impl": "ours",
            "config": {"workload": args.workload, "layer": shape.name, "T": T,
                       "H": shape.H, "E": shape.E, "k": shape.k, "I": shape.I, "S": shape.S,
                       "routing": routing, "ffn": m["kind"], "served_groups": m["n_groups"],
                       "l2": "flushed between steps (256 MiB write, outside the timed events)",
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                       "timing": "CUDA events around each step on the launch stream; a step "
                                 "is one CUDA graph of the whole layer; the gate/up kernel is "
                                 "timed over K more steps recorded as three graphs "
                                 "[route+permute][gate/up][down+combine]"},
            "us_per_layer": round(m["ms"] * 1e3, 2),
            "layer_roofline": {"t_roof_us": round(roof["t_roof_us"], 2), "bound": roof["bound"],
                               "frac": round(roof["t_roof_us"] / (m["ms"] * 1e3), 4),
                               "algorithmic_bytes": roof["bytes"],
                               "peak_source": peaks["source"]},
            "roofline": m["kroof"],
            "per_T": per_T,
            "sweep": sweep,
            "other_rows": rows,
            "e2e": {"value": round(aggregate_value(T * args.steps, world, e2e_sec), 1),
                    "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "us_per_step": round(e2e_ms * 1e3, 2),
                    "path": "pinned host x+logits -> device -> forward -> pinned host out, "
                            "copies and kernels in one CUDA graph (MoELayer.capture_host)"},
            "gpu_launches": (1 if m["kind"] == "decode" else 2) * kernels_per_step(
                layer, T, m["kind"]) * args.steps,           # every timed pass
            "clocks": clocks,
        }
        if base is not None:
            line["cpu_baseline"] = {k: base[k] for k in ("value", "unit", "cores", "kind",
                                                         "cpu", "sample", "value_1_thread",
                                                         "sample_1_thread")}
            line["parity_vs_oracle"] = base["parity"]
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_reference(args):
    """The CPU oracle as the reference arm: each step is the route + permute
    + layer of a bounded sample of the workload's tokens (as many tokens as
    the host has cores, round robin over the batch), on the host cores."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import numpy as np
    import torch

    import oracle
    from grouped_expert_gemm_moe_gb300 import workloads as W
    cfg, T, routing, _ = WORKLOADS[args.workload]
    shape = W.CONFIGS[cfg]
    inp = W.make_layer(shape, T, routing, seed=0, device="cpu")
    wbits = (W.bf16_bits(inp.w_gu), W.bf16_bits(inp.w_down))
    per = max(1, min(T, oracle.num_threads()))
    def step(i):
        tok = (np.arange(per) + i * per) % T
        host = oracle_sample(inp, tok)
        run_oracle_tokens(inp, host, tok, wbits)
    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(args.warmup + i)
    sec = time.perf_counter() - t0
    value = per * args.steps / sec
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(sec * 1e3 / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "impl": "reference",
        "config": {"workload": args.workload, "layer": shape.name, "T": T, "H": shape.H,
                   "E": shape.E, "k": shape.k, "I": shape.I, "S": shape.S, "routing": routing},
        "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "cores": per, "kind": "oracle",
                         "cpu": cpu_model(),
                         "sample": f"per step: route+permute+layer of {per} of the {T} tokens"},
        "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default=DEFAULT_WORKLOAD)
    ap.add_argument("--ffn", choices=("auto", "decode", "gemv", "gemm"), default="auto",
                    help="FFN path of the workload's layer: the layer's own choice, or "
                         "forced (to time or profile one path)")
    ap.add_argument("--no-rows", action="store_true",
                    help="skip the sweep over every config and the capacity and 16-layer "
                         "stack measurements of other_rows")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.steps < 1:
        ap.error("--steps must be at least 1")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
