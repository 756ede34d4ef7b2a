"""Benchmark of the int8 quantized linear layer on GB300: forward + backward
to the input (and bias) of every layer of a workload, throughput in TOPS.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference]

One step = every layer of the workload: quantize the activations (outlier
detection, row quantization, outlier weight columns), the int8 GEMM with its
fused dequant/outlier/bias epilogue, the grad_output prepass (grad_bias) and
the dequantizing backward GEMM.  Inputs are resident in HBM and larger than
L2 (so no flush is needed between steps).  Under torchrun every rank runs its
own replica of the workload (no collective on the data path): weak scaling.

``--impl reference`` times the CPU oracle on the host cores instead, on a
bounded row sample of the same workload, and prints the same metric.
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
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "Int8 linear fwd+bwd TOPS on one GB300, % of int8/fp16 tensor-core peak"
DEFAULT_WORKLOAD = "proj_8192x28672"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# DRAM bytes per launch of the GEMMs on the default workload, from the one-pass
# ncu capture summarised in profiles/gemm_dram_proj_8192x28672.md, valid
# while the kernel sources are the ones captured (sha256 below).
MEASURED_TRAFFIC = {
    "workload": "proj_8192x28672",
    "sources": {"int8_quantized_linear_i8lt_gb300/csrc/i8lt_gemm.cu":
                "db72aec6e1193a23043428cf17ce2e294e8fb2466bc09ac14163773552107a15",
                "int8_quantized_linear_i8lt_gb300/csrc/i8lt_common.cuh":
                "cc2fb6fa161ef5430ebd36ed4e9af7f9a5113376b51d4738964ca1dbdcce7d42"},
    "bytes_per_launch": {"fwd_gemm": 8.07e9, "bwd_gemm": 5.64e9},
}


def measured_traffic(workload, kernel, bwd_schedule):
    """DRAM bytes per launch of ``kernel`` from the committed capture, or None
    when the workload, the schedule or the kernel sources differ."""
    import hashlib
    if workload != MEASURED_TRAFFIC["workload"] or (kernel == "bwd_gemm" and bwd_schedule != "fused"):
        return None
    for rel, digest in MEASURED_TRAFFIC["sources"].items():
        p = os.path.join(ROOT, rel)
        if not os.path.exists(p) or hashlib.sha256(open(p, "rb").read()).hexdigest() != digest:
            return None
    return MEASURED_TRAFFIC["bytes_per_launch"].get(kernel)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ---------------------------------------------------------------------------
# distributed plumbing (replicas: timing only, no data-path collective)
# ---------------------------------------------------------------------------

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def reduce_max(value: float, device) -> float:
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def reduce_sum(value: float, device) -> float:
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (FileNotFoundError, OSError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

class Layer:
    """Device-resident tensors of one layer of the workload."""

    def __init__(self, wl, li, seed, device):
        import int8_quantized_linear_i8lt_gb300 as I
        spec = wl.layers[li]
        self.spec = spec
        gen_dev = device                      # draw on the GPU: same recipe, fast
        torch.manual_seed(seed * 1000 + li)
        A = torch.randn(spec.M, spec.K, device=gen_dev, dtype=torch.float32)
        heavy = W.heavy_columns(spec.K, spec.heavy_frac, seed + li * W.OFF_LAYER2 + W.OFF_HEAVY).to(device)
        if len(heavy):
            A[:, heavy] *= spec.heavy_factor
        self.A = A.to(spec.dtype)
        del A
        wdt = wl.w_dtype or spec.dtype
        Wf = (torch.randn(spec.N, spec.K, device=gen_dev) * spec.w_std).to(wdt)
        self.CB, self.SCB = I.quantize_weight(Wf)
        self.W = Wf                           # the float weight of the trainable-weight mode
        self.bias = (torch.randn(spec.N, device=gen_dev) * (spec.bias_std or 0.0)).to(wdt)
        self.G = torch.randn(spec.M, spec.N, device=gen_dev).to(spec.dtype)
        cap = I.default_max_outliers(spec.K)
        self.cap = cap
        self.out = torch.empty(spec.M, spec.N, dtype=spec.dtype, device=device)
        self.ws_f = I.functional.forward_workspace(spec.M, spec.K, spec.N, cap, device)
        # fused backward schedule (the fp16 weight rebuilt inside the GEMM, never
        # stored); the larger workspace selects the materialized schedule
        self.ws_b = I.functional.backward_workspace(spec.M, spec.N, spec.dtype, device)
        self.ws_b_dq = I.functional.backward_workspace(spec.M, spec.N, spec.dtype, device, K=spec.K)
        self.grad_A = torch.empty(spec.M, spec.K, dtype=spec.dtype, device=device)
        self.grad_bias = torch.empty(spec.N, dtype=wdt, device=device)

    def ops(self):
        s = self.spec
        return 4.0 * s.M * s.N * s.K        # 2MNK forward + 2MNK backward-to-input


def _launch_layer(L, stream_ptr, materialized=False):
    """One layer through the C ABI: forward, then backward to the input and
    the bias (fused backward schedule unless ``materialized``)."""
    from int8_quantized_linear_i8lt_gb300 import _lib
    from int8_quantized_linear_i8lt_gb300.functional import DTYPE_CODE
    s = L.spec
    dt = DTYPE_CODE[s.dtype]
    bt = DTYPE_CODE[L.bias.dtype]
    st = _lib.i8lt_forward(L.A.data_ptr(), dt, s.M, s.K, L.CB.data_ptr(), L.SCB.data_ptr(), s.N,
                           L.bias.data_ptr(), bt, s.threshold, None, L.out.data_ptr(), L.ws_f.data_ptr(),
                           L.ws_f.numel(), L.cap, stream=stream_ptr)
    assert st == 0, _lib.i8lt_status_string(st)
    wsb = L.ws_b_dq if materialized else L.ws_b
    st = _lib.i8lt_backward_input(L.G.data_ptr(), dt, s.M, s.N, L.CB.data_ptr(), L.SCB.data_ptr(), s.K, None,
                                  L.grad_A.data_ptr(), L.grad_bias.data_ptr(), bt, wsb.data_ptr(),
                                  wsb.numel(), stream_ptr)
    assert st == 0, _lib.i8lt_status_string(st)


def kernel_flops(L, name):
    """Algorithmic work of one launch of a GEMM kernel: 2*M*N*K."""
    s = L.spec
    return 2.0 * s.M * s.N * s.K if name in ("fwd_gemm", "bwd_gemm") else 0.0


def fused_quantize(spec) -> bool:
    """Whether the forward quantizes the activations in one launch (column
    maxima, outlier set and row quantization: 16-bit A, K a multiple of 8,
    rows up to 32768 columns), as the library decides."""
    kp = (spec.K + 15) // 16 * 16
    return spec.dtype in (torch.float16, torch.bfloat16) and spec.K % 8 == 0 and kp <= 32768


def _threshold_on(spec) -> bool:
    import math
    return math.isfinite(spec.threshold) and spec.threshold > 0


def kernel_bytes(L, name):
    """Algorithmic HBM bytes of one launch of a memory-bound kernel."""
    s = L.spec
    a = {torch.float16: 2, torch.bfloat16: 2, torch.float32: 4}[s.dtype]
    cnt = getattr(L, "found", 0)
    cap_pad = (min(cnt, s.K) + 63) // 64 * 64
    kp = (s.K + 15) // 16 * 16
    # the one-launch activation quantization reads A twice (the column maxima
    # must be complete before any row's scale) when the outliers are on
    reads = 2 if (fused_quantize(s) and _threshold_on(s)) else 1
    return {
        "colmax": s.M * s.K * a + s.K * 4,
        # the codes count as int8, one byte each, whatever form the kernel stores
        "row_quantize": reads * s.M * s.K * a + s.M * kp + s.M * 4 + s.M * cap_pad * 2,
        # it runs where the GEMM needs an fp16 copy of G: reads G, writes the copy
        "gradout_prepass": s.M * s.N * a + s.M * ((s.N + 7) // 8 * 8) * 2,
        "build_subB": s.N * cap_pad * 3,
        "widen_codes": s.N * kp * 3,
        "dequant_weight": s.N * kp + kp * ((s.N + 7) // 8 * 8) * 2 + s.N * 4,
    }.get(name, 0.0)


def run_ours(args):
    import int8_quantized_linear_i8lt_gb300 as I  # noqa: F401  (fails loudly without the library)
    from int8_quantized_linear_i8lt_gb300 import _lib
    _lib.load()
    ws, rank, local = dist_env()
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
    wl = W.WORKLOADS[args.workload]
    layers = [Layer(wl, li, 1234 + rank, device) for li in range(len(wl.layers))]
    stream = torch.cuda.current_stream(device)
    sp = stream.cuda_stream
    mat = args.bwd_schedule == "materialized"
    for _ in range(args.warmup):
        for L in layers:
            _launch_layer(L, sp, mat)
    torch.cuda.synchronize()
    for L in layers:
        st, found = I.device_status(L.ws_f)
        assert st == 0, _lib.i8lt_status_string(st)
        L.found = found
    # --- timed region: K steps, every kernel launch bracketed by CUDA events
    barrier()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    _lib.i8lt_profile_start(1 << 20)
    with ClockSampler(local) as clk:
        t_wall = time.perf_counter()
        step_ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps - 1)]
        ev0.record(stream)
        for k in range(args.steps):
            for L in layers:
                _launch_layer(L, sp, mat)
            if k < args.steps - 1:
                step_ev[k].record(stream)
        ev1.record(stream)
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall
    bounds = [ev0, *step_ev, ev1]
    step_ms = sorted(a.elapsed_time(b) for a, b in zip(bounds, bounds[1:]))
    pst, recs, n_launches = _lib.i8lt_profile_stop(1 << 20)
    assert pst == 0
    barrier()
    ms_total = reduce_max(ev0.elapsed_time(ev1), device)
    ops_step = sum(L.ops() for L in layers)
    ms_step = ms_total / args.steps
    units = reduce_sum(ops_step * args.steps, device)
    value = units / (ms_total * 1e-3) / 1e12

    # --- per-kernel totals from the records (launch order repeats per step)
    per_step = len(recs) // args.steps
    kern = {}
    per_layer = [{"fwd_ms": 0.0, "bwd_ms": 0.0, "fwd_gemm_ms": 0.0, "bwd_gemm_ms": 0.0} for _ in layers]
    for i, (name, ms) in enumerate(recs):
        li = _layer_of(i % per_step, layers, mat)
        L = layers[li]
        d = kern.setdefault(name, {"launches": 0, "ms": 0.0, "flops": 0.0, "bytes": 0.0})
        d["launches"] += 1
        d["ms"] += ms
        d["flops"] += kernel_flops(L, name)
        d["bytes"] += kernel_bytes(L, name)
        side = "bwd" if name in ("gradout_prepass", "grad_bias_finalize", "dequant_weight", "bwd_gemm") else "fwd"
        per_layer[li][side + "_ms"] += ms
        if name in ("fwd_gemm", "bwd_gemm"):
            per_layer[li][name + "_ms"] += ms
    total_k_ms = sum(d["ms"] for d in kern.values())
    dom = max(kern, key=lambda k: kern[k]["ms"])
    peaks, peak_src = load_peaks()
    peak_t = float(peaks.get("bf16_tflops_sustained", peaks.get("bf16_tflops")))
    peak_t_burst = float(peaks.get("bf16_tflops", peak_t))
    peak_b = float(peaks.get("hbm_gbs"))
    d = kern[dom]
    if d["flops"] > 0:
        achieved = d["flops"] / (d["ms"] * 1e-3) / 1e12
        # the GEMMs run inside a seconds-long loop of steps under the power
        # cap, so the headline fraction is against the sustained peak; the
        # burst fraction is given beside it
        roof = {"kernel": dom, "bound": "tensor", "achieved": round(achieved, 1), "peak": peak_t,
                "unit": "TFLOP/s", "frac": round(achieved / peak_t, 4),
                "peak_source": f"{peak_src} bf16 sustained (fp16 runs at the bf16 rate; kind::f16 is the "
                               "only tensor path of these GEMMs, sm_103a has no int8 tcgen05 MMA)",
                "peak_burst": peak_t_burst, "frac_burst": round(achieved / peak_t_burst, 4),
                "headline_peak": "sustained"}
    else:
        achieved = d["bytes"] / (d["ms"] * 1e-3) / 1e9
        roof = {"kernel": dom, "bound": "hbm", "achieved": round(achieved, 1), "peak": peak_b, "unit": "GB/s",
                "frac": round(achieved / peak_b, 4), "peak_source": f"{peak_src} hbm copy"}
    roof["launch_ms"] = round(d["ms"] / d["launches"], 4)
    traffic = measured_traffic(wl.name, dom, args.bwd_schedule)
    roof["traffic"] = traffic
    if traffic is not None:
        roof["traffic_unit"] = "bytes per launch (ncu dram__bytes_read.sum + dram__bytes_write.sum)"
        roof["traffic_gbs"] = round(traffic / (roof["launch_ms"] * 1e-3) / 1e9, 1)
    kernels = {}
    for k, v in sorted(kern.items(), key=lambda kv: -kv[1]["ms"]):
        e = {"launches": v["launches"], "ms_per_launch": round(v["ms"] / v["launches"], 4),
             "share": round(v["ms"] / total_k_ms, 4)}
        if v["flops"]:
            t = v["flops"] / (v["ms"] * 1e-3) / 1e12
            e.update(tflops=round(t, 1), frac_tensor=round(t / peak_t, 4), frac_tensor_burst=round(t / peak_t_burst, 4))
        elif v["bytes"]:
            g = v["bytes"] / (v["ms"] * 1e-3) / 1e9
            e.update(gbs=round(g, 1), frac_hbm=round(g / peak_b, 4))
        kernels[k] = e
    # --- per layer: forward and backward (all their kernels) against the fp16 tensor peak.  The
    # forward's int8 products run on the fp16 tensor cores (kind::f16, exact integer operands):
    # sm_103a has no int8 tcgen05 MMA, so the kind::f16 rate is the forward's ceiling.  The int8
    # rate the installed libraries reach through the legacy path is measured beside it as context.
    int8_peak = measure_int8_peak(device)
    layers_out = []
    for L, pl in zip(layers, per_layer):
        s_ = L.spec
        w = 2.0 * s_.M * s_.N * s_.K * args.steps
        f_t = w / (pl["fwd_ms"] * 1e-3) / 1e12
        b_t = w / (pl["bwd_ms"] * 1e-3) / 1e12
        entry = {"shape": [s_.M, s_.K, s_.N], "fwd_ms": round(pl["fwd_ms"] / args.steps, 4),
                 "bwd_ms": round(pl["bwd_ms"] / args.steps, 4), "fwd_tops": round(f_t, 1),
                 "bwd_tflops": round(b_t, 1), "fwd_bwd_tops": round(2 * w / ((pl["fwd_ms"] + pl["bwd_ms"]) * 1e-3) / 1e12, 1),
                 "fwd_frac_fp16_peak": round(f_t / peak_t, 4), "bwd_frac_fp16_peak": round(b_t / peak_t, 4)}
        if int8_peak.get("tops"):
            entry["fwd_vs_library_int8_rate"] = round(f_t / int8_peak["tops"], 2)
        layers_out.append(entry)
    # --- end to end through host buffers (pinned), inputs and results copied each
    # step, over as many steps as the device-timed region (the first step's
    # input copies and the last one's read-backs have nothing to overlap)
    e2e = run_e2e(layers, stream, max(2, args.steps), device)
    # --- the trainable-weight mode on the same layers (context, not the headline)
    trainable = time_trainable(layers, stream, max(2, min(args.steps, 10)), device)
    # --- the same step with the other backward schedule (context, not the headline)
    alt = time_schedule(layers, stream, max(2, min(args.steps, 10)), device, not mat)
    # --- the step replayed from a CUDA graph (context, not the headline)
    graph = time_graph(layers, max(3, min(args.steps, 20)), device)
    # --- the 4-bit weight-only layers (another workload: context, not the headline); FP4 runs the
    # same matmul kernels with another level table
    nf4 = time_nf4(stream, max(2, min(args.steps, 10)), device)
    fp4 = time_nf4(stream, max(2, min(args.steps, 10)), device, fmt="fp4", materialized_too=False)

    clocks = clk.summary()
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "TOPS", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
        "step_ms": {"median": round(step_ms[len(step_ms) // 2], 4), "best": round(step_ms[0], 4),
                    "worst": round(step_ms[-1], 4)},
        "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int8 codes (exact fp16 on tcgen05 kind::f16, int32 sums) + f16",
        "data": "synthetic (seeded N(0,1) activations with heavy outlier columns, N(0,std) weights)",
        "config": {"workload": wl.name, "layers": [[s.M, s.K, s.N, str(s.dtype).replace("torch.", "")]
                                                   for s in wl.layers],
                   "threshold": wl.layers[0].threshold, "outlier_columns": [L.found for L in layers],
                   "l2": "inputs larger than L2 (126 MB); no flush", "parallelism": f"replicas x{ws}"},
        "roofline": roof,
        "kernels": kernels,
        "per_layer": layers_out,
        "int8_tensor_peak": int8_peak,
        "e2e": e2e,
        "bwd_schedule": args.bwd_schedule,
        **({"mlp_chain": time_mlp_chain(wl, layers, stream, max(2, min(args.steps, 10)), device)}
           if wl.kind == "mlp" and len(layers) == 2 else {}),
        "trainable_mode": trainable,
        ("bwd_fused" if mat else "bwd_materialized"): alt,
        "cuda_graph": graph,
        "nf4_weight_only": nf4,
        "fp4_weight_only": fp4,
        "gpu_launches": n_launches,
        "gemm_launch": {k: dict(zip(("status", "ctas", "threads", "smem"), _lib.i8lt_gemm_launch_info(k)))
                        for k in ("fwd_gemm", "bwd_gemm")},
        "clocks": clocks,
        "wall_s": round(t_wall, 3),
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, budget_s=args.cpu_budget)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


class ShardLayer:
    """One rank's share of a layer of a token-sharded batch: the weight is the
    same on every rank (drawn from the layer's seed), the rank holds rows
    [r0, r0 + M_r) of the batch's activations and grad_output (drawn from the
    rank's own seed: the same recipe and shapes)."""

    def __init__(self, wl, li, seed, rank, world, device):
        import dataclasses

        import int8_quantized_linear_i8lt_gb300 as I
        spec = wl.layers[li]
        M_r = spec.M // world + (1 if rank < spec.M % world else 0)
        self.spec = dataclasses.replace(spec, M=M_r)
        self.full_M = spec.M
        s = self.spec
        wdt = wl.w_dtype or spec.dtype
        torch.manual_seed(seed * 1000 + li)                     # the weight: same on every rank
        Wf = (torch.randn(s.N, s.K, device=device) * s.w_std).to(wdt)
        self.CB, self.SCB = I.quantize_weight(Wf)
        del Wf
        self.bias = (torch.randn(s.N, device=device) * (s.bias_std or 0.0)).to(wdt)
        torch.manual_seed(seed * 1000 + li + 7919 * (rank + 1))  # this rank's rows
        A = torch.randn(M_r, s.K, device=device, dtype=torch.float32)
        heavy = W.heavy_columns(s.K, s.heavy_frac, seed + li * W.OFF_LAYER2 + W.OFF_HEAVY).to(device)
        if len(heavy):
            A[:, heavy] *= s.heavy_factor
        self.A = A.to(s.dtype)
        del A
        self.G = torch.randn(M_r, s.N, device=device).to(s.dtype)
        self.cap = I.default_max_outliers(s.K)
        self.out = torch.empty(M_r, s.N, dtype=s.dtype, device=device)
        self.ws_f = I.functional.forward_workspace(M_r, s.K, s.N, self.cap, device)
        self.colmax = I.functional.colmax_region(self.ws_f, M_r, s.K, s.N, s.threshold)
        self.ws_b = I.functional.backward_workspace(M_r, s.N, s.dtype, device)
        self.grad_A = torch.empty(M_r, s.K, dtype=s.dtype, device=device)
        self.grad_bias = torch.empty(s.N, dtype=wdt, device=device)

    def ops(self):
        s = self.spec
        return 4.0 * s.M * s.N * s.K


def _launch_sharded_layer(L, stream, merge, ev=None):
    """One rank's share of a layer: column maxima of its rows, the exchange
    (``merge``: an all-reduce MAX of the K maxima, or nothing on one rank),
    the rest of the forward, then the backward to the input and the bias."""
    from int8_quantized_linear_i8lt_gb300 import _lib
    from int8_quantized_linear_i8lt_gb300.functional import DTYPE_CODE
    s = L.spec
    dt, bt, sp = DTYPE_CODE[s.dtype], DTYPE_CODE[L.bias.dtype], stream.cuda_stream
    st = _lib.i8lt_forward_colmax(L.A.data_ptr(), dt, s.M, s.K, s.N, L.ws_f.data_ptr(), L.ws_f.numel(), L.cap,
                                  stream=sp)
    assert st == 0, _lib.i8lt_status_string(st)
    if ev is not None:
        ev[0].record(stream)
    merge(L.colmax)
    if ev is not None:
        ev[1].record(stream)
    st = _lib.i8lt_forward_from_colmax(L.A.data_ptr(), dt, s.M, s.K, L.CB.data_ptr(), L.SCB.data_ptr(), s.N,
                                       L.bias.data_ptr(), bt, s.threshold, None, L.out.data_ptr(), L.ws_f.data_ptr(),
                                       L.ws_f.numel(), L.cap, stream=sp)
    assert st == 0, _lib.i8lt_status_string(st)
    st = _lib.i8lt_backward_input(L.G.data_ptr(), dt, s.M, s.N, L.CB.data_ptr(), L.SCB.data_ptr(), s.K, None,
                                  L.grad_A.data_ptr(), L.grad_bias.data_ptr(), bt, L.ws_b.data_ptr(), L.ws_b.numel(),
                                  sp)
    assert st == 0, _lib.i8lt_status_string(st)


def run_sharded(args):
    """``--shard tokens``: one batch of the workload split over the ranks by
    tokens (strong scaling).  The outlier columns are a property of the whole
    batch, so every layer's forward exchanges its K column maxima with one
    all-reduce MAX between the column-maxima pass and the rest; after that
    every row is independent.  On one rank the exchange is empty and the
    output equals the unsharded forward bit for bit (checked here)."""
    import int8_quantized_linear_i8lt_gb300 as I
    from int8_quantized_linear_i8lt_gb300 import _lib
    _lib.load()
    world, rank, local = dist_env()
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
        merge = I.functional.allreduce_colmax()
    else:
        merge = lambda t: None  # noqa: E731  (one rank: its maxima are the batch's)
    wl = W.WORKLOADS[args.workload]
    layers = [ShardLayer(wl, li, 1234, rank, world, device) for li in range(len(wl.layers))]
    stream = torch.cuda.current_stream(device)
    for _ in range(args.warmup):
        for L in layers:
            _launch_sharded_layer(L, stream, merge)
    torch.cuda.synchronize()
    identical = None
    if world == 1:
        identical = True
        for L in layers:
            ref, _ = I.forward(L.A, L.CB, L.SCB, L.spec.K, L.bias, L.spec.threshold, max_outliers=L.cap)
            identical = identical and bool(torch.equal(ref.view(torch.uint8), L.out.view(torch.uint8)))
            del ref
    barrier()
    torch.cuda.synchronize()
    ex_ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in layers]
             for _ in range(args.steps)]
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        ev0.record(stream)
        for k in range(args.steps):
            for L, ev in zip(layers, ex_ev[k]):
                _launch_sharded_layer(L, stream, merge, ev)
        ev1.record(stream)
        torch.cuda.synchronize()
    barrier()
    ms_total = reduce_max(ev0.elapsed_time(ev1), device)
    ex_ms = reduce_max(sum(a.elapsed_time(b) for step in ex_ev for a, b in step), device)
    units = reduce_sum(sum(L.ops() for L in layers) * args.steps, device)
    value = units / (ms_total * 1e-3) / 1e12
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "TOPS", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_total / args.steps, 4), "higher_is_better": True,
        "scaling": "strong", "vs_baseline": None,
        "dtype": "int8 codes (exact fp16 on tcgen05 kind::f16, int32 sums) + f16",
        "data": "synthetic (seeded N(0,1) activations with heavy outlier columns, N(0,std) weights)",
        "config": {"workload": wl.name, "layers": [[s.M, s.K, s.N, str(s.dtype).replace("torch.", "")]
                                                   for s in wl.layers],
                   "rows_per_rank": [L.spec.M for L in layers], "threshold": wl.layers[0].threshold,
                   "l2": "inputs larger than L2 (126 MB); no flush", "parallelism": f"tokens sharded x{world}"},
        "exchange": {"what": "all-reduce MAX of each layer's K column maxima (int32), between the column-maxima "
                             "pass and the rest of the forward",
                     "ms_per_step": round(ex_ms / args.steps, 4), "share": round(ex_ms / ms_total, 5),
                     "bytes_per_step": sum(4 * L.spec.K for L in layers)},
        "bit_identical_to_unsharded": identical,
        "e2e": None,
        "clocks": clk.summary(),
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def measure_int8_peak(device, n=8192, iters=10):
    """The int8 tensor rate of this GPU as the CUDA libraries reach it
    (torch._int_mm, cuBLASLt int8 x int8 -> int32, n^3).  sm_103a offers no
    int8 tcgen05 MMA, so this is the legacy int8 tensor path and not a
    ceiling of the forward, which runs the int8 codes on the fp16 tensor
    cores.  Context only, off the timed region."""
    try:
        a = torch.randint(-127, 128, (n, n), dtype=torch.int8, device=device)
        b = torch.randint(-127, 128, (n, n), dtype=torch.int8, device=device)
        for _ in range(3):
            torch._int_mm(a, b.t())
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(iters):
            torch._int_mm(a, b.t())
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / iters
        return {"tops": round(2.0 * n ** 3 / (ms * 1e-3) / 1e12, 1), "how": f"torch._int_mm {n}^3, best path of "
                "the installed cuBLASLt, mean of 10 after 3 warm-up",
                "note": "context only, not a roofline: the legacy int8 tensor path of the libraries; sm_103a has no "
                        "int8 tcgen05 MMA, so the forward runs its exact int8 products on the fp16 tensor cores "
                        "and is judged against the fp16 peak (per_layer[*].fwd_frac_fp16_peak)"}
    except Exception as exc:   # no int8 GEMM in this build of the libraries
        return {"tops": None, "how": f"torch._int_mm unavailable: {type(exc).__name__}: {exc}"[:200]}


def _layer_of(i, layers, materialized=False):
    """Index of the layer that launch ``i`` (within one step) belongs to."""
    n = 0
    for li, L in enumerate(layers):
        n += launches_per_layer(L, materialized)
        if i < n:
            return li
    return len(layers) - 1


def launches_per_layer(L, materialized=False) -> int:
    """Our kernels per layer and step: the activation quantization (one
    launch for 16-bit rows of a multiple of 8 columns, else colmax and the
    outlier index (outliers on) and row quantize), subB (outliers on),
    weight-code widening, accumulation plan, forward GEMM; then (weight
    dequantization when materialized,) the
    backward GEMM and the grad_bias finalize -- with a grad_output prepass
    first when G is not fp16 with N a multiple of 8 (the GEMM reads fp16 G
    as it is and reduces grad_bias from it itself)."""
    if _threshold_on(L.spec):
        # column maxima + outlier index + row quantization, or the one launch
        # that does all three; subB; widening; plan; GEMM
        fwd = 5 if fused_quantize(L.spec) else 7
    else:
        fwd = 4
    prepass = 0 if (L.spec.dtype == torch.float16 and L.spec.N % 8 == 0) else 1
    return fwd + 2 + prepass + (1 if materialized else 0)


def time_trainable(layers, stream, steps, device):
    """The trainable-weight mode (has_fp16_weights=True) on the same layers:
    per layer and step the weight is quantized afresh, then the forward,
    grad_A (fused schedule), grad_bias and grad_W (int8 column-wise
    product).  Ops counted: 6 M N K per layer (three GEMMs)."""
    from int8_quantized_linear_i8lt_gb300 import _lib
    from int8_quantized_linear_i8lt_gb300.functional import DTYPE_CODE
    sp = stream.cuda_stream
    extra = []
    for L in layers:
        s = L.spec
        gW = torch.empty(s.N, s.K, dtype=L.W.dtype, device=device)
        wsw = torch.empty(_lib.i8lt_grad_weight_workspace_size(s.M, s.N, s.K), dtype=torch.uint8, device=device)
        extra.append((gW, wsw))

    def step():
        for L, (gW, wsw) in zip(layers, extra):
            s = L.spec
            st = _lib.i8lt_quantize_weight(L.W.data_ptr(), DTYPE_CODE[L.W.dtype], s.N, s.K, L.CB.data_ptr(),
                                           L.SCB.data_ptr(), sp)
            assert st == 0, _lib.i8lt_status_string(st)
            _launch_layer(L, sp)
            st = _lib.i8lt_grad_weight(L.G.data_ptr(), DTYPE_CODE[s.dtype], L.A.data_ptr(), DTYPE_CODE[s.dtype], s.M,
                                       s.N, s.K, gW.data_ptr(), DTYPE_CODE[L.W.dtype], wsw.data_ptr(), wsw.numel(), sp)
            assert st == 0, _lib.i8lt_status_string(st)

    step()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    _lib.i8lt_profile_start(1 << 16)
    ev0.record(stream)
    for _ in range(steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize()
    _, recs, _ = _lib.i8lt_profile_stop(1 << 16)
    ms = reduce_max(ev0.elapsed_time(ev1), device)
    ops = reduce_sum(sum(6.0 * L.spec.M * L.spec.N * L.spec.K for L in layers) * steps, device)
    wg_ms = sum(t for n, t in recs if n == "wgrad_gemm")
    cq_ms = sum(t for n, t in recs if n == "col_quantize")
    qw_ms = sum(t for n, t in recs if n == "quantize_weight")
    flops = sum(2.0 * L.spec.M * L.spec.N * L.spec.K for L in layers) * steps
    peaks, _ = load_peaks()
    peak_t = float(peaks.get("bf16_tflops_sustained", peaks.get("bf16_tflops")))
    wg_tf = flops / (wg_ms * 1e-3) / 1e12 if wg_ms else None
    return {"value": round(ops / (ms * 1e-3) / 1e12, 2), "unit": "TOPS", "ms_per_step": round(ms / steps, 3),
            "steps": steps, "wgrad_gemm_tflops": round(wg_tf, 1) if wg_tf else None,
            "wgrad_gemm_frac_tensor": round(wg_tf / peak_t, 4) if wg_tf else None,
            "col_quantize_ms_per_step": round(cq_ms / steps, 4), "quantize_weight_ms_per_step": round(qw_ms / steps, 4)}


def time_nf4(stream, steps, device, warmup=3, fmt="nf4", materialized_too=True):
    """The 4-bit NormalFloat weight-only layers (QLoRA fine-tuning: frozen
    NF4 weights, bf16 compute) of the qlora_mlp_7b_nf4 workload: per layer
    and step the forward and the input gradient, each a tensor-core matmul
    that decodes the 4-bit weight tile by tile.  FLOPs counted: 4 M N K per
    layer.  The weights are quantized once, outside the timed region (they
    are frozen)."""
    import int8_quantized_linear_i8lt_gb300 as I
    from int8_quantized_linear_i8lt_gb300 import _lib
    from int8_quantized_linear_i8lt_gb300.functional import DTYPE_CODE
    wl = W.NF4_WORKLOADS["qlora_mlp_7b_nf4"]
    sp = stream.cuda_stream
    fwd_fn = getattr(_lib, f"i8lt_{fmt}_forward")
    bwd_fn = getattr(_lib, f"i8lt_{fmt}_backward_input")
    ws = torch.empty(_lib.i8lt_nf4_workspace_size(), dtype=torch.uint8, device=device)
    lay = []
    for li, spec in enumerate(wl.layers):
        Wf, _, G = W.layer_tensors(wl, li, 4321, device)
        A = W.layer_input(wl, li, 4321, device)
        packed, absmax = I.quantize_4bit(Wf, fmt)
        out = torch.empty(spec.M, spec.N, dtype=spec.dtype, device=device)
        gA = torch.empty(spec.M, spec.K, dtype=spec.dtype, device=device)
        lay.append((spec, A, G, packed, absmax, out, gA))
        del Wf

    ws_dq = torch.empty(max(_lib.i8lt_nf4_workspace_size_dq(s_.K, s_.N) for s_ in wl.layers), dtype=torch.uint8,
                        device=device) if materialized_too else None

    # the double-quantized storage of each layer's absmax (the -dq option) and
    # a buffer its decoded values go to on every step
    dq = [(I.double_quantize_absmax(absmax), torch.empty_like(absmax)) for (_, _, _, _, absmax, _, _) in lay]

    def step(w, double_quant=False):
        for li, (spec, A, G, packed, absmax, out, gA) in enumerate(lay):
            dt = DTYPE_CODE[spec.dtype]
            if double_quant:
                (q, a2, off), absmax = dq[li]
                st = _lib.i8lt_absmax8_dequantize(q.data_ptr(), a2.data_ptr(), off.data_ptr(), q.numel(),
                                                  absmax.data_ptr(), sp)
                assert st == 0, _lib.i8lt_status_string(st)
            st = fwd_fn(A.data_ptr(), dt, spec.M, spec.K, packed.data_ptr(), absmax.data_ptr(), spec.N,
                        None, 0, out.data_ptr(), w.data_ptr(), w.numel(), sp)
            assert st == 0, _lib.i8lt_status_string(st)
            st = bwd_fn(G.data_ptr(), dt, spec.M, spec.N, packed.data_ptr(), absmax.data_ptr(),
                        spec.K, gA.data_ptr(), None, 0, w.data_ptr(), w.numel(), sp)
            assert st == 0, _lib.i8lt_status_string(st)

    def timed(w, double_quant=False):
        for _ in range(warmup):
            step(w, double_quant)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        _lib.i8lt_profile_start(1 << 16)
        e0.record(stream)
        for _ in range(steps):
            step(w, double_quant)
        e1.record(stream)
        torch.cuda.synchronize()
        _, r, n = _lib.i8lt_profile_stop(1 << 16)
        return reduce_max(e0.elapsed_time(e1), device), r, n

    ms, recs, n_launches = timed(ws)          # fused: the weight decoded inside the GEMM
    flops = sum(4.0 * spec.M * spec.N * spec.K for spec, *_ in lay) * steps
    half = flops / 2
    peaks, src = load_peaks()
    peak_t = float(peaks.get("bf16_tflops_sustained", peaks.get("bf16_tflops")))
    res = {"workload": wl.name, "format": fmt,
           "layers": [[s.M, s.K, s.N, str(s.dtype).replace("torch.", "")] for s in wl.layers],
           "value": round(reduce_sum(flops, device) / (ms * 1e-3) / 1e12, 1), "unit": "TFLOP/s",
           "ms_per_step": round(ms / steps, 4), "steps": steps, "gpu_launches": n_launches}
    for name in ("nf4_gemm_fwd", "nf4_gemm_bwd"):
        k_ms = sum(t for n, t in recs if n == name)
        if k_ms:
            tf = half / (k_ms * 1e-3) / 1e12
            res[name] = {"tflops": round(tf, 1), "frac_tensor": round(tf / peak_t, 4),
                         "ms_per_launch": round(k_ms / (steps * len(lay)), 4)}
    if materialized_too:
        ms_dq, recs_dq, _ = timed(ws_dq)      # materialized: dequantized weight in the workspace
        res["materialized"] = {"value": round(reduce_sum(flops, device) / (ms_dq * 1e-3) / 1e12, 1),
                               "unit": "TFLOP/s", "ms_per_step": round(ms_dq / steps, 4),
                               "dequantize_ms_per_step": round(sum(t for n, t in recs_dq if n == "nf4_dequantize")
                                                               / steps, 4)}
        for name in ("nf4_gemm_fwd", "nf4_gemm_bwd"):
            k_ms = sum(t for n, t in recs_dq if n == name)
            if k_ms:
                tf = half / (k_ms * 1e-3) / 1e12
                res["materialized"][name] = {"tflops": round(tf, 1), "frac_tensor": round(tf / peak_t, 4)}
    ms_q, recs_q, _ = timed(ws, double_quant=True)   # fused, absmax stored in 8 bits and decoded per step
    res["double_quant"] = {"value": round(reduce_sum(flops, device) / (ms_q * 1e-3) / 1e12, 1), "unit": "TFLOP/s",
                           "ms_per_step": round(ms_q / steps, 4),
                           "absmax8_ms_per_step": round(sum(t for n, t in recs_q if n == "absmax8") / steps, 4),
                           "absmax_bytes_per_layer": [int(q.numel() + 4 * a2.numel() + 4)
                                                      for ((q, a2, _), _) in dq]}
    res["peak"] = peak_t
    res["peak_source"] = f"{src} bf16 sustained"
    return res


def time_mlp_chain(wl, layers, stream, steps, device):
    """An MLP workload run as one block (fc1 -> SiLU -> fc2, then the
    backward of both), fused -- fc1's epilogue applies the SiLU and writes
    fc2's column maxima -- and unfused (separate SiLU kernel and column-maxima
    pass).  Same results bit for bit; both timed with CUDA events."""
    import int8_quantized_linear_i8lt_gb300 as I
    F = I.functional
    L1, L2 = layers
    s1, s2 = L1.spec, L2.spec
    thr = s1.threshold
    x, G = L1.A, L2.G
    M, K, H, N2 = s1.M, s1.K, s1.N, s2.N
    cap2 = F._capacity(H, thr, None)
    ws2 = F.forward_workspace(M, H, N2, cap2, device)
    colmax = F.colmax_region(ws2, M, H, N2, thr)

    def block(fused):
        if fused:
            h, a, _ = F.forward_silu(x, L1.CB, L1.SCB, K, L1.bias, thr, act_colmax=colmax)
            y, _ = I.forward(a, L2.CB, L2.SCB, H, L2.bias, thr, ws=ws2, colmax_ready=True)
        else:
            h, _ = I.forward(x, L1.CB, L1.SCB, K, L1.bias, thr)
            a = F.silu(h)
            y, _ = I.forward(a, L2.CB, L2.SCB, H, L2.bias, thr, ws=ws2)
        ga, _ = I.backward_input(G, L2.CB, L2.SCB, H, bias_dtype=L2.bias.dtype)
        gh = F.silu_backward(ga, h)
        gx, _ = I.backward_input(gh, L1.CB, L1.SCB, K, bias_dtype=L1.bias.dtype)
        return y, gx

    out = {}
    for fused in (True, False):
        block(fused)
        torch.cuda.synchronize()
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        for _ in range(steps):
            block(fused)
        ev1.record(stream)
        torch.cuda.synchronize()
        ms = reduce_max(ev0.elapsed_time(ev1), device) / steps
        ops = 4.0 * M * K * H + 4.0 * M * H * N2
        out["fused" if fused else "unfused"] = {"ms_per_step": round(ms, 4),
                                                "value": round(ops / (ms * 1e-3) / 1e12, 2), "unit": "TOPS"}
    y1, g1 = block(True)
    y2, g2 = block(False)
    out["bit_identical"] = bool(torch.equal(y1.view(torch.uint8), y2.view(torch.uint8))
                                and torch.equal(g1.view(torch.uint8), g2.view(torch.uint8)))
    out["steps"] = steps
    return out


def time_schedule(layers, stream, steps, device, materialized):
    """The step with the given backward schedule.  Materialized: a prepass
    writes the dequantized weight (K x N fp16) to the workspace, then a
    TMA-fed fp16 GEMM reads it; fused: the weight is rebuilt inside the GEMM.
    Same results either way; the one not timed as the headline is reported
    as context."""
    from int8_quantized_linear_i8lt_gb300 import _lib
    sp = stream.cuda_stream
    for L in layers:
        _launch_layer(L, sp, materialized)
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    _lib.i8lt_profile_start(1 << 16)
    ev0.record(stream)
    for _ in range(steps):
        for L in layers:
            _launch_layer(L, sp, materialized)
    ev1.record(stream)
    torch.cuda.synchronize()
    pst, recs, _ = _lib.i8lt_profile_stop(1 << 16)
    ms = reduce_max(ev0.elapsed_time(ev1), device)
    ops = reduce_sum(sum(L.ops() for L in layers) * steps, device)
    bwd_ms = sum(t for n, t in recs if n == "bwd_gemm")
    dq_ms = sum(t for n, t in recs if n == "dequant_weight")
    bwd_flops = sum(2.0 * L.spec.M * L.spec.N * L.spec.K for L in layers) * steps
    return {"value": round(ops / (ms * 1e-3) / 1e12, 2), "unit": "TOPS", "ms_per_step": round(ms / steps, 3),
            "steps": steps, "bwd_gemm_tflops": round(bwd_flops / (bwd_ms * 1e-3) / 1e12, 1) if bwd_ms else None,
            "dequant_weight_ms_per_step": round(dq_ms / steps, 4)}


def time_graph(layers, steps, device):
    """The same step captured once in a CUDA graph and replayed: every launch
    of the library goes through the caller's stream, so a captured step
    replays with no host work per kernel.  For the large workloads this
    matches the eager step; for the tiny MLP it removes the launch latency."""
    side = torch.cuda.Stream(device)
    side.wait_stream(torch.cuda.current_stream(device))
    with torch.cuda.stream(side):
        for L in layers:                      # warm-up outside the capture (attributes, caches)
            _launch_layer(L, side.cuda_stream)
    torch.cuda.current_stream(device).wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        sp = torch.cuda.current_stream(device).cuda_stream
        for L in layers:
            _launch_layer(L, sp)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream(device)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(steps):
        g.replay()
    ev1.record(stream)
    torch.cuda.synchronize()
    ms = reduce_max(ev0.elapsed_time(ev1), device)
    ops = reduce_sum(sum(L.ops() for L in layers) * steps, device)
    return {"value": round(ops / (ms * 1e-3) / 1e12, 4), "unit": "TOPS", "ms_per_step": round(ms / steps, 4),
            "us_per_step": round(1e3 * ms / steps, 2), "steps": steps}


def run_e2e(layers, stream, steps, device):
    """The metric through the public C ABI with host buffers: every step copies
    A and grad_output of every layer from pinned host memory and reads out,
    grad_A and grad_bias back, inside the timed region.

    The copies run on two copy streams (host to device, device to host) and
    overlap the kernels of other layers and steps: each layer has two sets of
    device buffers used by alternate steps, and CUDA events order every copy
    against the kernels that produce or consume its buffer.  The timed region
    opens on the compute stream before the first copy and closes after the
    last read-back of the last step."""
    host_in = [(torch.empty_like(L.A, device="cpu").pin_memory(), torch.empty_like(L.G, device="cpu").pin_memory())
               for L in layers]
    host_out = [(torch.empty_like(L.out, device="cpu").pin_memory(),
                 torch.empty_like(L.grad_A, device="cpu").pin_memory(),
                 torch.empty_like(L.grad_bias, device="cpu").pin_memory()) for L in layers]
    for (hA, hG), L in zip(host_in, layers):
        hA.copy_(L.A)
        hG.copy_(L.G)
    # buffer set 0 is the layer's own tensors, set 1 a copy of their shapes
    names = ("A", "G", "out", "grad_A", "grad_bias")
    bufs = [[{n: getattr(L, n) for n in names}, {n: torch.empty_like(getattr(L, n)) for n in names}]
            for L in layers]
    h2d_s = torch.cuda.Stream(device)
    d2h_s = torch.cuda.Stream(device)
    ev = lambda: torch.cuda.Event()  # noqa: E731
    ev_h2d = [[ev(), ev()] for _ in layers]
    ev_comp = [[ev(), ev()] for _ in layers]
    ev_d2h = [[ev(), ev()] for _ in layers]
    used = [[False, False] for _ in layers]
    sp = stream.cuda_stream
    h2d = sum(hA.numel() * hA.element_size() + hG.numel() * hG.element_size() for hA, hG in host_in)
    d2h = sum(sum(t.numel() * t.element_size() for t in ho) for ho in host_out)
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    h2d_s.wait_event(ev0)
    for step in range(steps):
        b = step % 2
        for li, ((hA, hG), (ho, hga, hgb), L) in enumerate(zip(host_in, host_out, layers)):
            B = bufs[li][b]
            with torch.cuda.stream(h2d_s):
                if used[li][b]:
                    h2d_s.wait_event(ev_d2h[li][b])     # step - 2 has read back and consumed this set
                B["A"].copy_(hA, non_blocking=True)
                B["G"].copy_(hG, non_blocking=True)
                ev_h2d[li][b].record(h2d_s)
            stream.wait_event(ev_h2d[li][b])
            for n in names:
                setattr(L, n, B[n])
            _launch_layer(L, sp)
            ev_comp[li][b].record(stream)
            with torch.cuda.stream(d2h_s):
                d2h_s.wait_event(ev_comp[li][b])
                ho.copy_(B["out"], non_blocking=True)
                hga.copy_(B["grad_A"], non_blocking=True)
                hgb.copy_(B["grad_bias"], non_blocking=True)
                ev_d2h[li][b].record(d2h_s)
            used[li][b] = True
    stream.wait_stream(d2h_s)
    ev1.record(stream)
    torch.cuda.synchronize()
    for li, L in enumerate(layers):
        for n in names:
            setattr(L, n, bufs[li][0][n])
    ms = reduce_max(ev0.elapsed_time(ev1), device)
    ops = reduce_sum(sum(L.ops() for L in layers) * steps, device)
    return {"value": round(ops / (ms * 1e-3) / 1e12, 2), "unit": "TOPS", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": round(ms / steps, 3), "steps": steps,
            "overlap": "copy streams, two buffer sets per layer"}


# ---------------------------------------------------------------------------
# CPU oracle (baseline / reference arm)
# ---------------------------------------------------------------------------

def _blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [d.get("num_threads") for d in threadpool_info() if d.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return os.cpu_count()


def oracle_sample_step(wl, rows_per_layer, seed=0):
    """One bounded oracle step: for every layer, the forward and the backward
    to the input on ``rows_per_layer`` rows (the outlier columns taken over
    those rows), with the weight quantized beforehand (off the step path).
    Returns (seconds, ops done)."""
    import oracle as O
    ops, secs = 0.0, 0.0
    for li, spec in enumerate(wl.layers):
        rows = np.arange(min(rows_per_layer, spec.M))
        sub = W.LayerSpec(len(rows), spec.K, spec.N, spec.dtype, spec.w_std, spec.bias_std, spec.heavy_frac,
                          spec.heavy_factor, spec.threshold)
        A = W.activation(sub, seed + li * W.OFF_LAYER2)
        g = torch.Generator().manual_seed(seed + li)
        wdt = wl.w_dtype or spec.dtype
        Wf = (torch.randn(spec.N, spec.K, generator=g) * spec.w_std).to(wdt)
        b = (torch.randn(spec.N, generator=g) * (spec.bias_std or 0.0)).to(wdt)
        G = torch.randn(len(rows), spec.N, generator=g).to(spec.dtype)
        odt = {torch.float16: O.F16, torch.bfloat16: O.BF16, torch.float32: O.F32}

        def np_(t):
            t = t.contiguous()
            return t.view(torch.int16).numpy().view(np.uint16) if t.dtype == torch.bfloat16 else t.numpy()

        CB, SCB = O.quantize_weight(np_(Wf), odt[wdt])
        A_np, b_np, G_np = np_(A), np_(b), np_(G)
        t0 = time.perf_counter()
        O.forward(A_np, odt[spec.dtype], CB, SCB, b_np, odt[wdt], spec.threshold)
        O.backward_input(G_np, odt[spec.dtype], CB, SCB)
        O.grad_bias(G_np, odt[spec.dtype], odt[wdt])
        secs += time.perf_counter() - t0
        ops += 4.0 * len(rows) * spec.N * spec.K
    return secs, ops


def cpu_baseline(wl, budget_s=20.0):
    """The oracle on a bounded row sample: the sample doubles until one
    measurement takes at least half of ``budget_s`` seconds (or holds every
    row, or 4096 rows)."""
    rows = 16
    secs, ops = oracle_sample_step(wl, rows)
    cap = min(4096, max(16, max(s.M for s in wl.layers)))
    while secs < budget_s / 2 and rows < cap:
        rows = min(cap, rows * 2 if secs > budget_s / 8 else rows * 4)
        secs, ops = oracle_sample_step(wl, rows)
    return {"value": round(ops / secs / 1e12, 6), "unit": "TOPS", "cores": _blas_threads(), "kind": "oracle",
            "sample": f"{rows} rows of every layer of {wl.name}: forward + backward to the input + grad_bias, "
                      f"weights pre-quantized; {secs:.1f} s of CPU time"}


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    wl = W.WORKLOADS[args.workload]
    rows = max(16, min(256, int(args.ref_rows)))
    for _ in range(args.warmup):
        oracle_sample_step(wl, 16)
    secs_total, ops_total = 0.0, 0.0
    for k in range(args.steps):
        s, o = oracle_sample_step(wl, rows, seed=k)
        secs_total += s
        ops_total += o
    value = ops_total / secs_total / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TOPS", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * secs_total / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64 (oracle)",
        "data": "synthetic", "config": {"workload": wl.name, "sample_rows_per_layer": rows},
        "cpu_baseline": {"value": round(value, 6), "unit": "TOPS", "cores": _blas_threads(), "kind": "oracle",
                         "sample": f"{rows} rows of every layer per step"},
        "e2e": {"value": round(value, 6), "unit": "TOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_aux_kernels(args):
    """The library's kernels that the bench step does not launch, each on an
    input larger than L2 (where it streams one): the quantization paths for
    fp32 activations and for rows longer than the one-launch kernel takes, the
    16-bit copy of a bf16 grad_output, the materialized schedules' prepasses,
    the SiLU of the MLP block, the 4-bit quantize and dequantize kernels, the
    absmax double quantization, the weight gradient's column passes and the
    fallback weight quantization.  Each case builds its inputs, runs once
    untimed and once with the library's CUDA-event records, and frees them
    (so that an ncu capture holds at most about a GB on the device): one JSON
    line of milliseconds per kernel and case."""
    import int8_quantized_linear_i8lt_gb300 as I
    from int8_quantized_linear_i8lt_gb300 import _lib
    _lib.load()
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    F = I.functional
    g = torch.Generator(device=device).manual_seed(11)

    def rnd(shape, dtype, std=1.0):
        return (torch.randn(shape, generator=g, device=device) * std).to(dtype)

    def weight(N, K):
        return I.quantize_weight(rnd((N, K), torch.float16, 0.02))

    def fwd(M, K, N, dt):
        A = rnd((M, K), dt)
        A[:, :16] *= 20.0                                 # outlier columns
        CB, SCB = weight(N, K)
        return lambda: F.forward(A, CB, SCB, K, None, 6.0)

    def bwd_bf16():
        G = rnd((16384, 8192), torch.bfloat16)
        CB, SCB = weight(8192, 1024)
        return lambda: F.backward_input(G, CB, SCB, 1024, bias_dtype=torch.bfloat16)

    def bwd_materialized():
        G = rnd((256, 16384), torch.float16)
        CB, SCB = weight(16384, 8192)
        ws = F.backward_workspace(256, 16384, torch.float16, device, K=8192)
        return lambda: F.backward_input(G, CB, SCB, 8192, ws=ws, fused=False)

    def silu_fwd():
        H = rnd((16384, 8192), torch.float16)
        return lambda: F.silu(H)

    def silu_bwd():
        H = rnd((16384, 8192), torch.float16)
        Gs = rnd((16384, 8192), torch.float16)
        return lambda: F.silu_backward(Gs, H)

    def nf4(kind):
        W4 = rnd((8192, 16384), torch.bfloat16, 0.02)
        if kind == "quantize":
            return lambda: I.nf4_quantize(W4)
        packed, absmax = I.nf4_quantize(W4)
        del W4
        if kind == "forward":
            A4 = rnd((256, 16384), torch.bfloat16)
            return lambda: F.nf4_forward(A4, packed, absmax, 16384, materialized=True)
        if kind == "input_grad":
            G4 = rnd((256, 8192), torch.bfloat16)
            return lambda: F.nf4_backward_input(G4, packed, absmax, 16384, materialized=True)
        if kind == "dq":
            return lambda: F.double_quantize_absmax(absmax)
        dq = F.double_quantize_absmax(absmax)
        return lambda: F.dequantize_absmax(*dq)

    def wgrad():
        Gw = rnd((8192, 8192), torch.float16)
        Aw = rnd((8192, 8192), torch.float16)
        return lambda: F.grad_weight(Gw, Aw)

    def wq32():
        W32 = rnd((8192, 8192), torch.float32, 0.02)
        return lambda: I.quantize_weight(W32)

    cases = [
        ("fp32 activations 8192 x 8192 (separate quantization kernels, bulk rows)",
         lambda: fwd(8192, 8192, 256, torch.float32)),
        ("fp32 activations 2048 x 32768 (staged rows)", lambda: fwd(2048, 32768, 256, torch.float32)),
        ("fp16 activations 2048 x 57344 (rows past the staged kernel)", lambda: fwd(2048, 57344, 256, torch.float16)),
        ("bf16 grad_output 16384 x 8192 (fp16 copy and grad_bias sums)", bwd_bf16),
        ("materialized backward, weight 16384 x 8192 (dequantized weight prepass)", bwd_materialized),
        ("SiLU forward 16384 x 8192", silu_fwd),
        ("SiLU backward 16384 x 8192", silu_bwd),
        ("NF4 quantize 8192 x 16384", lambda: nf4("quantize")),
        ("NF4 forward, materialized (dequantize 8192 x 16384)", lambda: nf4("forward")),
        ("NF4 input gradient, materialized (transposed dequantize 8192 x 16384)", lambda: nf4("input_grad")),
        ("absmax double quantization (8192 x 256 values)", lambda: nf4("dq")),
        ("absmax decode (8192 x 256 values)", lambda: nf4("decode")),
        ("weight gradient 8192 x 8192 x 8192 (column maxima, column quantization, tile maxima)", wgrad),
        ("fp32 weight quantization 8192 x 8192 (bulk rows)", wq32),
    ]
    out = []
    for name, make in cases:
        fn = make()
        fn()
        torch.cuda.synchronize()
        _lib.i8lt_profile_start(1 << 12)
        fn()
        torch.cuda.synchronize()
        _, recs, _ = _lib.i8lt_profile_stop(1 << 12)
        ms = {}
        for n, t in recs:
            ms[n] = round(ms.get(n, 0.0) + t, 4)
        out.append({"case": name, "ms": ms})
        del fn
        torch.cuda.empty_cache()
    print(json.dumps({"aux_kernels": out, "device": torch.cuda.get_device_name(device)}), flush=True)


def run_nf4_only(args):
    """The NF4 section of the bench line on its own (profiling runs of the
    4-bit matmuls): W warm-up steps, then K timed steps."""
    import int8_quantized_linear_i8lt_gb300 as I  # noqa: F401  (fails loudly without the library)
    from int8_quantized_linear_i8lt_gb300 import _lib
    _lib.load()
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    res = time_nf4(torch.cuda.current_stream(device), args.steps, device, warmup=args.warmup)
    print(json.dumps({"nf4_weight_only": res}), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=60)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(W.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=20.0)
    ap.add_argument("--ref-rows", type=int, default=64)
    ap.add_argument("--bwd-schedule", default="fused", choices=["fused", "materialized"],
                    help="backward schedule of the timed steps (the other one is timed beside it)")
    ap.add_argument("--shard", default="none", choices=["none", "tokens"],
                    help="tokens: one batch split over the ranks by tokens, with the column-maxima all-reduce "
                         "(strong scaling); none: every rank runs its own replica (weak scaling)")
    ap.add_argument("--nf4-only", action="store_true",
                    help="time only the NF4 weight-only layers (qlora_mlp_7b_nf4) and print their line")
    ap.add_argument("--aux-kernels", action="store_true",
                    help="run each kernel outside the bench step once, on inputs larger than L2 (for ncu)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    if args.aux_kernels:
        run_aux_kernels(args)
    elif args.nf4_only:
        run_nf4_only(args)
    elif args.impl == "reference":
        run_reference(args)
    elif args.shard == "tokens":
        run_sharded(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
