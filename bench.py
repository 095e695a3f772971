"""Benchmark of the binarized linear / conv2d forward on GB300.

One step = one forward over one batch of synthetic input: shift + sign +
pack of the activations, the packed contraction and the fused scale + cast
epilogue. Weights are packed once, before timing (bitorch-engine packs
weights offline, in generate_quantized_weight / w_pack). Default workload: the
largest configuration, the 8192 x 4096 x 11008 bf16 linear layer; after it,
`all_configs` records every configuration with each code the library has.

Prints ONE JSON line on rank 0. Under torchrun every rank runs its own
replica of the workload (its shard of a batch N times larger; no collective
on the data path) and the max-over-ranks time gives the whole-job value.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                  [--impl reference]
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

import numpy as np
import torch

import workloads

ROOT = os.path.dirname(os.path.abspath(__file__))
L2_BYTES = 129 * 1024 * 1024


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default="large_linear", choices=sorted(workloads.NAMED))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--algo", default="auto", choices=["auto", "popc", "e4m3", "e2m1"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-tune", action="store_true",
                    help="skip the measured selection (bt_tune_linear / bt_tune_conv2d) and take the planner's shape")
    ap.add_argument("--tune-reps", type=int, default=10, help="timed calls per candidate launch shape or plan")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the record of every configuration (all_configs) after the headline")
    ap.add_argument("--config-steps", type=int, default=20, help="timed steps per configuration and code")
    ap.add_argument("--no-graph", action="store_true",
                    help="launch the headline steps one call at a time instead of replaying them as a CUDA graph")
    ap.add_argument("--pass", dest="pass_", default="forward",
                    choices=["forward", "backward", "w8a8", "w8a8-smooth", "tune-survey"],
                    help="backward: the straight-through backward (all three gradients); w8a8[-smooth]: the W8A8 "
                         "im2col + gemm convolution of a conv workload (with SmoothQuant); tune-survey: the "
                         "measured selection over ResNet conv layers and LLM projection shapes")
    return ap.parse_args()


# ---------------------------------------------------------------------------
# distributed plumbing (barrier + max over ranks only)
# ---------------------------------------------------------------------------

def dist_init(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() and args.impl == "ours" else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        dist.init_process_group(backend)
    return rank, world


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v: float, world: int) -> float:
    if world == 1:
        return v
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    """SM clock and clock-event reasons sampled every millisecond during the
    timed region, through NVML (the driver's library, read-only queries);
    falls back to `nvidia-smi -lms` when NVML cannot be loaded."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, device_index: int):
        self.dev = device_index
        self.samples = []
        self.max_mhz = None
        self._stop = threading.Event()
        self._thread = None
        self._nvml = None
        self._handle = None
        self._smi = None

    def _open_nvml(self):
        import ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        handle = ctypes.c_void_p()
        props = torch.cuda.get_device_properties(self.dev)
        bus = None
        if all(hasattr(props, a) for a in ("pci_domain_id", "pci_bus_id", "pci_device_id")):
            bus = f"{props.pci_domain_id:08X}:{props.pci_bus_id:02X}:{props.pci_device_id:02X}.0"
        if bus is None or lib.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(handle)) != 0:
            if lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(self.dev), ctypes.byref(handle)) != 0:
                raise OSError("no NVML handle")
        self._nvml, self._handle = lib, handle
        mx = ctypes.c_uint()
        if lib.nvmlDeviceGetMaxClockInfo(handle, 1, ctypes.byref(mx)) == 0:
            self.max_mhz = float(mx.value)
        self._reason_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons")

    def _run(self):
        import ctypes
        mhz, reasons = ctypes.c_uint(), ctypes.c_ulonglong()
        while not self._stop.is_set():
            if self._nvml.nvmlDeviceGetClockInfo(self._handle, 1, ctypes.byref(mhz)) == 0:
                r = reasons.value if self._reason_fn(self._handle, ctypes.byref(reasons)) == 0 else 0
                self.samples.append((float(mhz.value), int(r)))
            time.sleep(0.001)

    def __enter__(self):
        try:
            self._open_nvml()
            self._thread = threading.Thread(target=self._run, daemon=True)
            self._thread.start()
        except (OSError, AttributeError):
            self._nvml = None
            try:
                self._smi = subprocess.Popen(
                    ["nvidia-smi", "-i", str(self.dev), "--query-gpu=clocks.sm,clocks.max.sm,clocks_event_reasons.active",
                     "--format=csv,noheader,nounits", "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                    text=True)
            except OSError:
                self._smi = None
        return self

    def __exit__(self, *exc):
        if self._thread is not None:
            self._stop.set()
            self._thread.join(timeout=5)
        if self._smi is not None:
            self._smi.terminate()
            try:
                out, _ = self._smi.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self._smi.kill()
                out = ""
            for line in out.splitlines():
                parts = [p.strip() for p in line.split(",")]
                try:
                    self.samples.append((float(parts[0]), int(parts[2], 16)))
                    self.max_mhz = float(parts[1])
                except (ValueError, IndexError):
                    continue

    def summary(self):
        if not self.samples:
            return None
        mhz = [m for m, _ in self.samples]
        seen = 0
        for _, r in self.samples:
            seen |= r
        return {"sm_mhz": statistics.median(mhz), "sm_min_mhz": min(mhz), "sm_max_mhz": self.max_mhz,
                "reasons": sorted(n for b, n in self.REASONS.items() if seen & b), "samples": len(mhz),
                "source": "nvml" if self._nvml is not None else "nvidia-smi"}


# ---------------------------------------------------------------------------
# peaks
# ---------------------------------------------------------------------------

def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        return json.load(open(p)), "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "sm_max_mhz": 2070.0}, "fallback"


# nominal dense tensor rates (PFLOP/s) for the ratio to the measured bf16 peak
NOMINAL_PF = {"bf16": 2.25, "e4m3": 4.5, "e2m1": 13.5}
# 32-bit population counts per clock per SM: the per-SM issue rate the CUDA
# programming guide's arithmetic-throughput table gives for the popc
# instruction on recent compute capabilities, and what a standalone probe on a
# GB300 (a loop of XOR + POPC on every SM, not part of this repository) reached;
# the denominator of the popcount path's ALU roofline.
POPC_PER_CLK_PER_SM = 16
SM_COUNT_GB300 = 152


def roofline_peak(algo: str, peaks: dict, sms: int):
    if algo == "popc":
        # each 32-bit popcount of a XOR retires 32 multiply-adds = 64 binary ops
        tops = sms * POPC_PER_CLK_PER_SM * 64 * peaks.get("sm_max_mhz", 2070.0) * 1e6 / 1e12
        return "alu", tops, "TOP/s", f"{sms} SMs x {POPC_PER_CLK_PER_SM} POPC/clk x 64 ops x max SM clock"
    tflops = peaks["bf16_tflops"] * NOMINAL_PF[algo] / NOMINAL_PF["bf16"]
    return "tensor", tflops, "TFLOP/s", f"measured bf16 x nominal {algo}/bf16 ratio"


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

ALGO_NAME = {0: "popc", 1: "e4m3", 2: "e2m1"}


CODE_OF = {"popc": 0, "e4m3": 1, "e2m1": 2}


class ForwardSetup:
    """One forward step of a workload as a user's stream runs it: the pack call
    (shift + sign + pack of x), then the contraction call (packed contraction
    + fused scale and cast), over input and output buffers that rotate so that
    one pass over them exceeds L2. Weights are packed once, here, outside any
    timing (bitorch-engine packs them offline)."""

    def __init__(self, bt, wl, code: int, algo: int, dev):
        self.bt, self.wl, self.code, self.algo = bt, wl, code, algo
        M, N, K = wl.gemm_shape()
        self.M, self.N, self.K = M, N, K
        self.out_t = {"f32": torch.float32, "bf16": torch.bfloat16}[wl.out_dtype]
        if wl.kind == "linear":
            self.wp = bt.bt_pack_sign(wl.w.to(dev), code)
        else:
            self.wp = bt.bt_pack_sign(wl.w.to(dev), code, bt.BT_LAYOUT_NCHW_TO_NHWC)
        self.bias = None if wl.bias is None else wl.bias.to(dev)
        self.x_bytes = wl.x.numel() * wl.x.element_size()
        self.out_bytes = M * N * torch.tensor([], dtype=self.out_t).element_size()
        self.nbuf = max(1, -(-2 * L2_BYTES // (self.x_bytes + self.out_bytes)))
        self.xs = [wl.x.to(dev) for _ in range(self.nbuf)]
        self.single_pass = False
        self.fused = False
        self.ws_rows = None
        if wl.kind == "linear":
            self.outs = [torch.empty((M, N), dtype=self.out_t, device=dev) for _ in range(self.nbuf)]
            self.ws = torch.empty(bt.bt_binary_linear_workspace(M, K, bt.BT_BF16, code), dtype=torch.uint8,
                                  device=dev)
            xp_shape = (M, bt.bt_packed_row_bytes(K, code))
        else:
            B, C, H, W = wl.x.shape
            k = wl.w.shape[2]
            self.C, self.k = C, k
            Ho = bt.conv2d_out_size(H, k, wl.stride, wl.padding, wl.dilation)
            Wo = bt.conv2d_out_size(W, k, wl.stride, wl.padding, wl.dilation)
            self.im2col_hw = (B, H, W)
            self.outs = [torch.empty((B, N, Ho, Wo), dtype=self.out_t, device=dev) for _ in range(self.nbuf)]
            geom = (B, C, H, W, k, wl.stride, wl.padding, wl.dilation)
            self.ws = torch.empty(max(1, bt.bt_binary_conv2d_workspace(*geom, bt.BT_BF16, code)), dtype=torch.uint8,
                                  device=dev)
            # the public calls that split the library's own path for this shape:
            # one call on x (the convolution packs x itself), or pack + contraction
            mode = bt.bt_conv2d_single_pass(
                *geom, {torch.float32: bt.BT_F32, torch.bfloat16: bt.BT_BF16, torch.float16: bt.BT_F16}[wl.x.dtype],
                code)
            self.fused = mode == 2
            self.single_pass = mode == 1
            if self.fused:
                xp_shape = (1,)
            elif not self.single_pass:
                # packed NHWC pixels; the contraction call unfolds them (where it
                # needs rows) or contracts them in place
                xp_shape = (B, H, W, bt.bt_packed_row_bytes(C, code))
                ws_rows_bytes = bt.bt_binary_conv2d_workspace(*geom, bt.BT_PACKED, code)
                self.ws_rows = torch.empty(ws_rows_bytes, dtype=torch.uint8, device=dev) if ws_rows_bytes else None
            else:
                # im2col rows of packed codes (one pass from x), contracted with the weights
                xp_shape = (B * Ho * Wo, k * k * bt.bt_packed_row_bytes(C, code))
        self.xp = torch.empty(xp_shape, dtype=torch.uint8, device=dev)
        # kernels per step: the pack, then the contraction; a contraction call
        # that unfolds packed pixels into rows first adds one
        unfolds = wl.kind == "conv" and not self.single_pass and self.ws_rows is not None
        self.launches_per_step = 1 if self.fused else (3 if unfolds else 2)

    def step(self, i, ev=None):
        bt, wl = self.bt, self.wl
        x, out = self.xs[i % self.nbuf], self.outs[i % self.nbuf]
        if ev is not None:
            ev[0].record(torch.cuda.current_stream())
        if wl.kind == "linear":
            bt.bt_pack_sign(x, self.code, bt.BT_LAYOUT_ROWS, self.bias, out=self.xp)
        elif self.fused:
            pass                                  # the convolution call packs x itself
        elif not self.single_pass:
            bt.bt_pack_sign(x, self.code, bt.BT_LAYOUT_NCHW_TO_NHWC, self.bias, out=self.xp)
        else:
            bt.bt_pack_im2col(x, self.code, self.k, wl.stride, wl.padding, wl.dilation, self.bias, out=self.xp)
        if ev is not None:
            ev[1].record(torch.cuda.current_stream())
        if wl.kind == "linear":
            bt.bt_binary_linear(self.xp, self.wp, self.code, self.K, wl.scale_a, wl.scale_w, out=out,
                                out_dtype=self.out_t, algo=self.algo, x_packed=True)
        elif self.fused:
            bt.bt_binary_conv2d(x, self.wp, self.code, self.C, self.k, wl.stride, wl.padding, wl.dilation,
                                wl.scale_a, wl.scale_w, self.bias, out=out, out_dtype=self.out_t, algo=self.algo)
        elif not self.single_pass:
            bt.bt_binary_conv2d(self.xp, self.wp, self.code, self.C, self.k, wl.stride, wl.padding, wl.dilation,
                                wl.scale_a, wl.scale_w, out=out, out_dtype=self.out_t, algo=self.algo,
                                x_packed=True, workspace=self.ws_rows)
        else:
            bt.bt_binary_conv2d(self.xp, self.wp, self.code, self.C, self.k, wl.stride, wl.padding, wl.dilation,
                                wl.scale_a, wl.scale_w, out=out, out_dtype=self.out_t, algo=self.algo,
                                x_im2col_hw=self.im2col_hw)
        if ev is not None:
            ev[2].record(torch.cuda.current_stream())

    def capture(self, steps: int, use_graph: bool):
        """The K steps captured once into a CUDA graph (each public call's
        kernels as nodes, nothing between the two calls of a step), or None
        when capture is off or unsupported; and a note saying which."""
        if not use_graph:
            return None, "off (--no-graph)"
        try:
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                for i in range(steps):
                    self.step(i)
            graph.replay()
            torch.cuda.synchronize()
            return graph, f"one CUDA graph of the {steps} steps, replayed"
        except RuntimeError as e:                       # capture unsupported: launch eagerly
            torch.cuda.synchronize()
            return None, f"off (capture failed: {str(e).splitlines()[0][:80]})"

    def run_steps(self, graph, steps: int, world: int = 1) -> float:
        """Milliseconds of `steps` back-to-back steps (device events on the
        launching stream, barrier and synchronize on both sides)."""
        stream = torch.cuda.current_stream()
        barrier(world)
        torch.cuda.synchronize()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        if graph is not None:
            graph.replay()
        else:
            for i in range(steps):
                self.step(i)
        t1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        return t0.elapsed_time(t1)

    def split(self, steps: int):
        """Mean milliseconds of the pack call and of the contraction call, from
        events around each on the launching stream (they serialise the two and
        add each launch's latency to its kernel)."""
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
        for i in range(steps):
            self.step(i, evs[i])
        torch.cuda.synchronize()
        return (statistics.mean(e[0].elapsed_time(e[1]) for e in evs),
                statistics.mean(e[1].elapsed_time(e[2]) for e in evs))


def step_bytes(wl) -> float:
    """Algorithmic bytes of one forward step: x read once, the weights packed
    to one bit per element, the output written once."""
    M, N, K = wl.gemm_shape()
    out_b = 4 if wl.out_dtype == "f32" else 2
    return wl.x.numel() * wl.x.element_size() + N * K / 8 + M * N * out_b


def contraction_bytes(wl, code, bt) -> float:
    """Least bytes the contraction call moves: the packed activations (rows of
    a linear layer; the packed pixels of a convolution, each read once by an
    implicit im2col; x itself where the convolution packs it), the packed
    weights, the output."""
    out_b = 4 if wl.out_dtype == "f32" else 2
    if wl.kind == "linear":
        M, K = wl.x.shape
        N = wl.w.shape[0]
        rb = bt.bt_packed_row_bytes(K, code)
        return (M + N) * rb + M * N * out_b
    B, C, H, W = wl.x.shape
    O, k = wl.w.shape[0], wl.w.shape[2]
    Ho = bt.conv2d_out_size(H, k, wl.stride, wl.padding, wl.dilation)
    Wo = bt.conv2d_out_size(W, k, wl.stride, wl.padding, wl.dilation)
    rbc = bt.bt_packed_row_bytes(C, code)
    if conv_mode(wl, code, bt) == 2:
        return wl.x.numel() * wl.x.element_size() + O * k * k * rbc + B * O * Ho * Wo * out_b
    return B * H * W * rbc + O * k * k * rbc + B * O * Ho * Wo * out_b


def conv_mode(wl, code, bt) -> int:
    """bt_conv2d_single_pass for the workload's convolution: 2 one kernel from
    x, 1 one-pass im2col rows + contraction, 0 NHWC pack + contraction."""
    B, C, H, W = wl.x.shape
    k = wl.w.shape[2]
    dt = {torch.float32: bt.BT_F32, torch.bfloat16: bt.BT_BF16, torch.float16: bt.BT_F16}[wl.x.dtype]
    return bt.bt_conv2d_single_pass(B, C, H, W, k, wl.stride, wl.padding, wl.dilation, dt, code)


def roofline_of(ops: float, nbytes: float, ms: float, algo_name: str, peaks: dict, sms: int) -> dict:
    """Roofline of `ops` binary ops moving `nbytes` in `ms`: bound by the pipe
    of the code used (tensor fp4 / fp8, or the POPC ALU) when the ops per byte
    exceed that pipe's ridge point (peak ops / measured HBM bandwidth), by HBM
    otherwise; frac = achieved / peak of that bound."""
    bound, peak, unit, how = roofline_peak(algo_name, peaks, sms)
    intensity = ops / nbytes
    ridge = peak * 1e12 / (peaks["hbm_gbs"] * 1e9)
    if intensity < ridge:
        bound, unit, peak = "hbm", "GB/s", peaks["hbm_gbs"]
        how = f"measured copy bandwidth; {intensity:.0f} ops/B < ridge {ridge:.0f}"
        achieved = nbytes / (ms / 1e3) / 1e9
    else:
        achieved = ops / (ms / 1e3) / 1e12
    return {"bound": bound, "achieved": round(achieved, 2), "peak": round(peak, 1), "unit": unit,
            "frac": round(achieved / peak, 4), "algorithmic_bytes": int(nbytes), "ops_per_byte": round(intensity, 1),
            "peak_how": how}


# every configuration the workloads module names, in the order of the table
CONFIG_ORDER = ["tiny_linear", "llm_linear", "resnet_conv", "downsample_conv", "downsample_conv_d2",
                "large_linear", "ragged_linear"]


def tune_linear(bt, wl, dev, reps: int) -> dict:
    """The measured "ADAPTIVE" selection of a linear workload, before any
    warm-up or timing: bt_tune_linear times the whole forward call on x (the
    pack, then the contraction: the kernels of a step, back to back) in every
    candidate launch shape of each tensor-core code, and the popcount kernel,
    keeping the fastest shape per code; bt_plan then names the fastest code
    for the size."""
    M, N, K = wl.gemm_shape()
    out_t = {"f32": torch.float32, "bf16": torch.bfloat16}[wl.out_dtype]
    xd = wl.x.to(dev)
    bias = None if wl.bias is None else wl.bias.to(dev)
    per = {}
    for code in (2, 1, 0):
        if code != 0 and K > 16384:
            continue
        wp = bt.bt_pack_sign(wl.w.to(dev), code)
        r = bt.bt_tune_linear(xd, wp, code, K, wl.scale_a, wl.scale_w, bias, out_dtype=out_t,
                              reps=reps if code != 0 else max(1, reps // 5))
        shape = (f"{'pair' if r['pair'] else 'single'} bn{r['bn']} d{r['slices_per_stage']} "
                 f"epi{r['epilogue_warps']}" if code != 0 else "popcount kernel")
        per[ALGO_NAME[code]] = {"us": round(r["us"], 2), "us_cost_model_shape": round(r["us_model"], 2),
                                "kept": shape, "candidates": r["candidates"]}
        del wp
    del xd
    torch.cuda.empty_cache()
    code, _ = bt.bt_plan(bt.BT_OP_LINEAR, M, N, K)
    return {"code": ALGO_NAME[code], "per_code": per,
            "how": "bt_tune_linear on x: mean of the timed forward calls (pack + contraction) per launch shape "
                   "(CUDA events), a shape replacing the cost model's only when > 1 % faster; bt_plan names the "
                   "code with the shortest"}


def tune_conv(bt, wl, dev, reps: int) -> dict:
    """The same for a convolution: bt_tune_conv2d times the whole call on x
    (the NHWC pack, then the implicit-im2col contraction; or the convolution
    packing x itself) in every candidate plan of each tensor-core code, and
    the popcount route, keeping the fastest plan per code; bt_plan then names
    the fastest code."""
    M, N, K = wl.gemm_shape()
    out_t = {"f32": torch.float32, "bf16": torch.bfloat16}[wl.out_dtype]
    B, C, H, W = wl.x.shape
    k = wl.w.shape[2]
    xd = wl.x.to(dev)
    bias = None if wl.bias is None else wl.bias.to(dev)
    per = {}
    for code in (2, 1, 0):
        wp = bt.bt_pack_sign(wl.w.to(dev), code, bt.BT_LAYOUT_NCHW_TO_NHWC)
        r = bt.bt_tune_conv2d(xd, wp, code, C, k, wl.stride, wl.padding, wl.dilation, wl.scale_a, wl.scale_w, bias,
                              out_dtype=out_t, reps=reps if code != 0 else max(1, reps // 5))
        plan = (f"{'pair' if r['pair'] else 'single'} {'resident' if r['weights_resident'] else 'streamed'} "
                f"weights, {r['pixel_stages']} pixel stage(s), {r['band_split']}x the planner's bands, "
                f"{'packs x itself' if r['fused'] else 'after the NHWC pack'}" if code != 0 else "popcount route")
        per[ALGO_NAME[code]] = {"us": round(r["us"], 2), "us_planner_plan": round(r["us_model"], 2), "kept": plan,
                                "candidates": r["candidates"]}
        del wp
    del xd
    torch.cuda.empty_cache()
    code, _ = bt.bt_plan(bt.BT_OP_CONV2D, M, N, K)
    return {"code": ALGO_NAME[code], "per_code": per,
            "how": "bt_tune_conv2d on x: mean of the timed calls per plan (CUDA events), a plan replacing the "
                   "planner's only when > 1 % faster; bt_plan names the code with the shortest"}


def tune(bt, wl, dev, args):
    if args.no_tune:
        return None
    return (tune_linear if wl.kind == "linear" else tune_conv)(bt, wl, dev, args.tune_reps)


def sweep_configs(bt, dev, peaks, peak_src, sms, args) -> dict:
    """Every configuration, each code the library has (the planner's choice
    first): graph-replayed step time, the pack / contraction split, and the
    rooflines of the step (its algorithmic bytes) and of the contraction call.
    The per-code step times show whether the planner ("ADAPTIVE") picks the
    fastest code for each shape."""
    steps, warm = args.config_steps, 3
    out = {}
    for name in CONFIG_ORDER:
        wl = workloads.NAMED[name]()
        M, N, K = wl.gemm_shape()
        ops = wl.binary_ops()
        op = bt.BT_OP_LINEAR if wl.kind == "linear" else bt.BT_OP_CONV2D
        sel = tune(bt, wl, dev, args)
        plan_code, _ = bt.bt_plan(op, M, N, K)
        codes = [plan_code] + [c for c in (2, 1, 0) if c != plan_code]
        per_code, rec = {}, None
        for code in codes:
            if code != 0 and K > 16384:
                continue
            su = ForwardSetup(bt, wl, code, bt.BT_ALGO_AUTO, dev)
            n = steps if code != 0 else max(3, steps // 4)         # the popcount path is the slow one
            for i in range(warm):
                su.step(i)
            torch.cuda.synchronize()
            graph, _ = su.capture(n, not args.no_graph)
            ms = su.run_steps(graph, n) / n
            pack_ms, gemm_ms = su.split(n)
            del graph
            per_code[ALGO_NAME[code]] = round(ms * 1e3, 2)
            if code == plan_code:
                an = ALGO_NAME[code]
                rec = {"M": M, "N": N, "K": K, "x_dtype": wl.x_dtype, "out_dtype": wl.out_dtype, "code": an,
                       "step_us": round(ms * 1e3, 2), "pack_us": round(pack_ms * 1e3, 2),
                       "contraction_us": round(gemm_ms * 1e3, 2), "gops": round(ops / (ms / 1e3) / 1e9, 1),
                       "step_roofline": roofline_of(ops, step_bytes(wl), ms, an, peaks, sms),
                       "contraction_roofline": roofline_of(ops, contraction_bytes(wl, code, bt), gemm_ms, an, peaks,
                                                           sms),
                       "steps": n}
            del su
            torch.cuda.empty_cache()
        if bt.bt_device_status() != 0:
            raise RuntimeError(f"device status after {name}")
        if sel is not None:
            rec["selection"] = sel
        rec["step_us_per_code"] = per_code
        rec["fastest_code"] = min(per_code, key=per_code.get)
        rec["planner_picks_fastest"] = rec["fastest_code"] == rec["code"]
        out[wl.name] = rec
    return {"peak_source": peak_src, "how": "graph-replayed steps per code (planner's code for the rooflines); "
            "step roofline on x + 1-bit W + out bytes, contraction roofline on packed activations + packed W + out",
            "configs": out}


def run_ours(args, rank, world):
    import xnor_popcount_gemm_gb300 as bt

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    wl = workloads.NAMED[args.workload]()
    M, N, K = wl.gemm_shape()
    ops = wl.binary_ops()
    op = bt.BT_OP_LINEAR if wl.kind == "linear" else bt.BT_OP_CONV2D
    selection = tune(bt, wl, dev, args)
    if args.algo == "auto":
        code, algo = bt.bt_plan(op, M, N, K)
    else:
        code = CODE_OF[args.algo]
        algo = bt.BT_ALGO_AUTO
    algo_name = ALGO_NAME[code]
    su = ForwardSetup(bt, wl, code, algo, dev)

    for i in range(args.warmup):
        su.step(i)
    torch.cuda.synchronize()
    assert bt.bt_device_status() == 0

    # headline: K steps back to back, nothing between the two calls of a step
    # (so a step's contraction may start as its pack drains, as in a user's
    # stream), replayed from one CUDA graph so that the host's per-call overhead
    # does not set the pace of small steps; then the same K steps again with
    # events around each call for the split and the roofline
    graph, graph_note = su.capture(args.steps, not args.no_graph)
    with ClockSampler(dev.index) as clk:
        ms_total = max_over_ranks(su.run_steps(graph, args.steps, world), world)
        pack_ms, gemm_ms = su.split(args.steps)
    status = bt.bt_device_status()
    if status != 0:
        raise RuntimeError(f"device status {bt.bt_status_string(status)}")
    ms_step = ms_total / args.steps
    value = ops * world * args.steps / (ms_total / 1e3) / 1e9

    # end to end through the public API from pinned host buffers: every step
    # copies its input in, runs the forward and copies its output back. Steps
    # are independent batches, so the copies of neighbouring steps overlap the
    # forward (three streams, two device slots); host buffers rotate over more
    # than the host's last-level cache so each copy reads and writes memory.
    e2e_ms, nh = e2e_pipelined(wl, bt, code, algo, su.wp, su.bias, su.out_t, su.ws, su.xs, su.outs,
                               torch.cuda.current_stream(), args, world)

    peaks, peak_src = measured_peaks()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    roof = roofline_of(ops, contraction_bytes(wl, code, bt), gemm_ms, algo_name, peaks, sms)
    roof.update({"traffic": load_traffic(wl.name, algo_name, wl.kind),
                 "traffic_unit": "DRAM bytes per launch of the contraction kernel (ncu, this kernel source)",
                 "peak_source": f"{peak_src}: {roof.pop('peak_how')}", "kernel": "contraction"})
    pack_b = pack_bytes(wl, code, bt)
    line = {
        "metric": "binary GOPS (2*M*N*K/s)",
        "value": round(value, 1),
        "unit": "GOPS",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": {"popc": "b1 (xor+popc, int32 acc)", "e4m3": "fp8 e4m3 +-1 (fp32 acc, exact)",
                  "e2m1": "fp4 e2m1 +-1 (fp32 acc, exact)"}[algo_name],
        "data": "synthetic (seeded; shapes of binarized LLM linear and ResNet conv layers)",
        "config": {"workload": wl.name, "M": M, "N": N, "K": K, "x_dtype": wl.x_dtype,
                   "out_dtype": wl.out_dtype, "code": algo_name, "weights": "pre-packed outside timing",
                   "l2": f"inputs+outputs rotate over {su.nbuf} buffers "
                         f"({su.nbuf * (su.x_bytes + su.out_bytes) / 1e6:.0f} MB > L2)",
                   "parallelism": f"replicas x{world}", "launch": graph_note},
        "kernel_ms": {"pack": round(pack_ms, 5), "contraction": round(gemm_ms, 5),
                      "how": "second pass of the same steps, CUDA events around each call on its stream"},
        "roofline": roof,
        "step_roofline": roofline_of(ops, step_bytes(wl), ms_step, algo_name, peaks, sms),
        "pack_roofline": ({"bound": "hbm", "achieved": round(pack_b / (pack_ms / 1e3) / 1e9, 1),
                           "peak": peaks["hbm_gbs"], "unit": "GB/s",
                           "frac": round(pack_b / (pack_ms / 1e3) / 1e9 / peaks["hbm_gbs"], 4)}
                          if pack_b > 0 else "none: the convolution kernel packs x itself"),
        "e2e": {"value": round(ops * world / (e2e_ms / 1e3) / 1e9, 1), "unit": "GOPS",
                "h2d_bytes_per_step": int(su.x_bytes), "d2h_bytes_per_step": int(su.out_bytes),
                "ms_per_step": round(e2e_ms, 4),
                "how": f"pinned host buffers (x{nh} rotating); copy-in, forward, copy-out on three streams, "
                       "neighbouring steps overlapped"},
        "selection": selection if selection is not None else
        "not measured (--no-tune): the planner's launch shape, or the one the environment forces",
        "gpu_launches": su.launches_per_step * args.steps,
        "clocks": clk.summary(),
    }
    del graph, su
    torch.cuda.empty_cache()
    if world == 1 and not args.no_configs:
        line["all_configs"] = sweep_configs(bt, dev, peaks, peak_src, sms, args)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl)
    return line


HOST_LLC_BYTES = 256 << 20     # rotate host buffers over more than this


def e2e_pipelined(wl, bt, code, algo, wp, bias, out_t, ws, xs, outs, stream, args, world):
    """Milliseconds per step of host x -> forward -> host y through the public
    calls, steady state over max(5, steps // 2) steps, and the number of host
    buffers each side rotates over."""
    dev = xs[0].device
    x_bytes = wl.x.numel() * wl.x.element_size()
    nh = min(64, max(2, -(-HOST_LLC_BYTES // x_bytes)))
    x_hosts = []
    for _ in range(nh):
        h = torch.empty(wl.x.shape, dtype=wl.x.dtype).pin_memory()
        h.copy_(wl.x)
        x_hosts.append(h)
    y_hosts = [torch.empty(outs[0].shape, dtype=out_t).pin_memory() for _ in range(nh)]
    xdev = [xs[0], xs[1] if len(xs) > 1 else torch.empty_like(xs[0])]
    ydev = [outs[0], outs[1] if len(outs) > 1 else torch.empty_like(outs[0])]
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    comp_done = [None, None]    # forward of the slot's last step (frees x slot, fills y slot)
    out_done = [None, None]     # copy-out of the slot's last step (frees y slot)

    def forward(x, y):
        if wl.kind == "linear":
            bt.bt_binary_linear(x, wp, code, wl.x.shape[1], wl.scale_a, wl.scale_w, bias, out=y,
                                out_dtype=out_t, algo=algo, workspace=ws, stream=stream)
        else:
            C, k = wl.x.shape[1], wl.w.shape[2]
            bt.bt_binary_conv2d(x, wp, code, C, k, wl.stride, wl.padding, wl.dilation, wl.scale_a,
                                wl.scale_w, bias, out=y, out_dtype=out_t, algo=algo, workspace=ws,
                                stream=stream)

    def e2e_step(i):
        slot = i & 1
        in_done = torch.cuda.Event()
        with torch.cuda.stream(s_in):
            if comp_done[slot] is not None:
                s_in.wait_event(comp_done[slot])
            xdev[slot].copy_(x_hosts[i % nh], non_blocking=True)
            in_done.record(s_in)
        stream.wait_event(in_done)
        if out_done[slot] is not None:
            stream.wait_event(out_done[slot])
        forward(xdev[slot], ydev[slot])
        comp_done[slot] = torch.cuda.Event()
        comp_done[slot].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(comp_done[slot])
            y_hosts[i % nh].copy_(ydev[slot], non_blocking=True)
            out_done[slot] = torch.cuda.Event()
            out_done[slot].record(s_out)

    def join():
        for e in out_done:
            if e is not None:
                stream.wait_event(e)

    for i in range(max(3, args.warmup)):
        e2e_step(i)
    join()
    torch.cuda.synchronize()
    n = max(5, args.steps // 2)
    barrier(world)
    a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a0.record(stream)
    s_in.wait_event(a0)
    for i in range(n):
        e2e_step(i)
    join()
    a1.record(stream)
    torch.cuda.synchronize()
    return max_over_ranks(a0.elapsed_time(a1), world) / n, nh


def pack_bytes(wl, code, bt):
    """Algorithmic bytes of the activation pack: read x once, write it packed
    (a tensor-core convolution's pack writes its im2col rows)."""
    if wl.kind == "linear":
        M, K = wl.x.shape
        return wl.x.numel() * wl.x.element_size() + M * bt.bt_packed_row_bytes(K, code)
    B, C, H, W = wl.x.shape
    k = wl.w.shape[2]
    mode = conv_mode(wl, code, bt)
    if mode == 2:
        return 0.0                              # no pack call: the convolution packs x itself
    if mode == 0:
        return wl.x.numel() * wl.x.element_size() + B * H * W * bt.bt_packed_row_bytes(C, code)
    # one pass: x read once, the im2col rows written
    Ho = bt.conv2d_out_size(H, k, wl.stride, wl.padding, wl.dilation)
    Wo = bt.conv2d_out_size(W, k, wl.stride, wl.padding, wl.dilation)
    return wl.x.numel() * wl.x.element_size() + B * Ho * Wo * k * k * bt.bt_packed_row_bytes(C, code)


def kernel_source_hash(kind: str = "linear") -> str:
    """First 16 hex digits of the sha256 of the contraction kernel's sources:
    tc_gemm.cu then tc_ptx.cuh (linear); tc_conv_kernel.cuh, tc_conv.cu,
    tc_ptx.cuh, then sign_pack.cuh (implicit-im2col convolution)."""
    h = hashlib.sha256()
    files = ("tc_gemm.cu", "tc_ptx.cuh") if kind == "linear" else \
        ("tc_conv_kernel.cuh", "tc_conv.cu", "tc_ptx.cuh", "sign_pack.cuh")
    for f in files:
        with open(os.path.join(ROOT, "xnor_popcount_gemm_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def load_traffic(workload: str, algo: str, kind: str = "linear"):
    """DRAM bytes per contraction launch from the committed ncu summary, if one
    exists for this workload and for the kernel source as it is now."""
    p = os.path.join(ROOT, "profiles", "contraction_dram_traffic.txt")
    if not os.path.exists(p):
        return None
    try:
        src = kernel_source_hash(kind)
        for line in open(p):
            parts = line.split()
            if len(parts) == 3 and not line.startswith("#") and parts[0] == f"{workload}/{algo}" and parts[2] == src:
                return int(parts[1])
    except (ValueError, OSError):
        return None
    return None


# ---------------------------------------------------------------------------
# backward pass (straight-through estimator) of a linear workload
# ---------------------------------------------------------------------------

def run_backward(args, rank, world):
    """K steps of the straight-through backward (the input gradient with its
    fused mask and grad_scale_a, and the weight gradient) on the workload's x
    and W with a synthetic bf16 upstream gradient; sign(W)^T is prepared once
    outside timing, as the forward's packed weight is."""
    import xnor_popcount_gemm_gb300 as bt

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    wl = workloads.NAMED[args.workload]()
    M, N, K = wl.gemm_shape()
    conv = wl.kind == "conv"
    if conv:
        B, C, H, W = wl.x.shape
        O, k = wl.w.shape[0], wl.w.shape[2]
        Ho = bt.conv2d_out_size(H, k, wl.stride, wl.padding, wl.dilation)
        Wo = bt.conv2d_out_size(W, k, wl.stride, wl.padding, wl.dilation)
        g_shape = (B, O, Ho, Wo)
        if O % 8:
            raise SystemExit("--pass backward needs O a multiple of 8")
    else:
        g_shape = (M, N)
        if N % 8 or K % 8:
            raise SystemExit("--pass backward needs N and K multiples of 8")
    if conv and bt.bt_conv2d_backward_implicit(B, C, H, W, O, k, wl.stride, wl.padding, wl.dilation):
        dgrad_label = "the input-gradient call (g per pixel, codes of x, one implicit GEMM with the mask in its epilogue)"
    elif conv:
        dgrad_label = "the input-gradient call (g per pixel, product over the unfolded taps, gather with the mask)"
    else:
        dgrad_label = "the input-gradient call (product with the mask fused in its epilogue)"
    stream = torch.cuda.current_stream()
    gen = torch.Generator().manual_seed(1000)
    g_host = (torch.randn(*g_shape, generator=gen) * 0.01).to(torch.bfloat16)
    x_host = wl.x if wl.x.dtype in (torch.bfloat16, torch.float32) else wl.x.float()
    wst = bt.bt_sign_transpose(wl.w.reshape(wl.w.shape[0], -1).to(dev))
    gw_shape = tuple(wl.w.shape)
    per = x_host.numel() * x_host.element_size() + g_host.numel() * 2 + (x_host.numel() + wl.w.numel()) * 2
    nbuf = max(1, -(-2 * L2_BYTES // per))
    xs = [x_host.to(dev) for _ in range(nbuf)]
    gs = [g_host.to(dev) for _ in range(nbuf)]
    gxs = [torch.empty(x_host.shape, dtype=torch.bfloat16, device=dev) for _ in range(nbuf)]
    gws = [torch.empty(gw_shape, dtype=torch.bfloat16, device=dev) for _ in range(nbuf)]
    gsa = torch.empty((), dtype=torch.float32, device=dev)
    if conv:
        ws = torch.empty(bt.bt_binary_conv2d_backward_workspace(B, C, H, W, O, k, wl.stride, wl.padding, wl.dilation),
                         dtype=torch.uint8, device=dev)
    else:
        ws = torch.empty(bt.bt_binary_linear_backward_workspace(M, N, K, True), dtype=torch.uint8, device=dev)
    flops = 2 * (2.0 * M * N * K)

    def step(i, which="both"):
        j = i % nbuf
        kw = dict(grad_input=which in ("both", "input"),
                  grad_weight_dtype=torch.bfloat16 if which in ("both", "weight") else None,
                  grad_x=gxs[j], grad_scale_a=gsa, grad_w=gws[j], workspace=ws)
        if conv:
            bt.bt_binary_conv2d_backward(xs[j], wst, gs[j], O, k, wl.stride, wl.padding, wl.dilation, wl.scale_a,
                                         wl.scale_w, **kw)
        else:
            bt.bt_binary_linear_backward(xs[j], wst, gs[j], wl.scale_a, wl.scale_w, **kw)

    def timed(which, n):
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(world)
        torch.cuda.synchronize()
        a0.record(stream)
        for i in range(n):
            step(i, which)
        a1.record(stream)
        torch.cuda.synchronize()
        return max_over_ranks(a0.elapsed_time(a1), world) / n

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    assert bt.bt_device_status() == 0
    with ClockSampler(dev.index) as clk:
        ms = timed("both", args.steps)
        ms_in = timed("input", args.steps)
        ms_w = timed("weight", args.steps)
    if bt.bt_device_status() != 0:
        raise RuntimeError("device status")
    peaks, peak_src = measured_peaks()
    achieved = 2.0 * M * N * K / (ms_in / 1e3) / 1e12
    launches = (6 if not conv else 7) * args.steps
    line = {
        "metric": "backward TFLOP/s (grad_input + grad_weight, 2 x 2*M*N*K / s)",
        "value": round(flops * world / (ms / 1e3) / 1e12, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16 x bf16 (fp32 acc)",
        "data": "synthetic (the workload's x and W; upstream gradient N(0, 0.01) in bf16)",
        "config": {"workload": wl.name, "pass": "backward", "M": M, "N": N, "K": K,
                   "x_dtype": str(x_host.dtype).replace("torch.", ""),
                   "weights": "sign(W)^T prepared outside timing",
                   "l2": f"inputs+outputs rotate over {nbuf} buffers", "parallelism": f"replicas x{world}"},
        "kernel_ms": {"grad_input_call": round(ms_in, 5), "grad_weight_call": round(ms_w, 5),
                      "how": "the same call asking for one gradient only, K steps each"},
        "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": peaks["bf16_tflops"],
                     "unit": "TFLOP/s", "frac": round(achieved / peaks["bf16_tflops"], 4), "traffic": None,
                     "peak_source": f"{peak_src}: cuBLAS bf16 burst",
                     "kernel": dgrad_label},
        "gpu_launches": launches,
        "clocks": clk.summary(),
    }
    return line


# layers of the measured-selection survey: ResNet convolutions (B, C, H = W, O,
# k, s, p, d, x dtype) and LLM projections (M, N, K; bf16 x)
SURVEY_CONVS = [
    (64, 64, 56, 64, 3, 1, 1, 1, torch.bfloat16), (64, 64, 56, 128, 3, 2, 1, 1, torch.bfloat16),
    (128, 128, 28, 128, 3, 1, 1, 1, torch.bfloat16), (128, 128, 28, 256, 3, 2, 1, 1, torch.bfloat16),
    (128, 256, 14, 256, 3, 1, 1, 1, torch.bfloat16), (128, 256, 14, 512, 3, 2, 1, 1, torch.bfloat16),
    (256, 512, 7, 512, 3, 1, 1, 1, torch.bfloat16), (128, 256, 14, 256, 3, 1, 1, 1, torch.float32),
    (256, 128, 28, 256, 3, 2, 1, 1, torch.bfloat16), (32, 512, 7, 2048, 1, 1, 0, 1, torch.bfloat16),
]
SURVEY_LINEARS = [(256, 4096, 4096), (1024, 4096, 4096), (2048, 11008, 4096), (4096, 4096, 11008),
                  (8192, 11008, 4096), (512, 14336, 4096), (16384, 4096, 4096), (4096, 1024, 4096)]


def run_tune_survey(args, rank, world):
    """bt_tune_conv2d / bt_tune_linear on each survey layer (seeded random
    inputs on the device): per layer the kept plan or shape, its time per call
    and the planner's, with --tune-reps timed calls per candidate."""
    import xnor_popcount_gemm_gb300 as bt

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    g = torch.Generator(device=dev).manual_seed(0)
    rows = []
    for (B, C, H, O, k, s, p, d, dt) in SURVEY_CONVS:
        x = torch.randn(B, C, H, H, device=dev, generator=g).to(dt)
        w = torch.randn(O, C, k, k, device=dev, generator=g).to(dt)
        wp = bt.bt_pack_sign(w, bt.BT_CODE_E2M1, bt.BT_LAYOUT_NCHW_TO_NHWC)
        bt.bt_tune_reset()
        r = bt.bt_tune_conv2d(x, wp, bt.BT_CODE_E2M1, C, k, s, p, d, 1.0, 1.0, reps=args.tune_reps)
        rows.append({"layer": f"conv [{B},{C},{H},{H}] -> {O}, {k}x{k} s{s} p{p} d{d}, {str(dt)[6:]} x",
                     "kept": f"{'pairs' if r['pair'] else 'single'}, {'resident' if r['weights_resident'] else 'streamed'}"
                             f", {r['pixel_stages']} stage(s), {r['band_split']}x bands"
                             f"{', packs x itself' if r['fused'] else ''}",
                     "candidates": r["candidates"], "us": round(r["us"], 2), "us_planner": round(r["us_model"], 2)})
        del x, w, wp
    for (M, N, K) in SURVEY_LINEARS:
        x = torch.randn(M, K, device=dev, generator=g).to(torch.bfloat16)
        w = torch.randn(N, K, device=dev, generator=g).to(torch.bfloat16)
        for code in (bt.BT_CODE_E2M1, bt.BT_CODE_E4M3):
            wp = bt.bt_pack_sign(w, code)
            bt.bt_tune_reset()
            r = bt.bt_tune_linear(x, wp, code, K, 1.0, 1.0, reps=args.tune_reps)
            rows.append({"layer": f"linear {M}x{N}x{K} {ALGO_NAME[code]}",
                         "kept": f"{'pairs' if r['pair'] else 'single'}, BN {r['bn']}, {r['slices_per_stage']} "
                                 f"slice(s) per stage, {r['epilogue_warps']} epilogue warps",
                         "candidates": r["candidates"], "us": round(r["us"], 2), "us_planner": round(r["us_model"], 2),
                         "gops": round(2.0 * M * N * K / r["us"] / 1e3, 1)})
            del wp
        del x, w
    bt.bt_tune_reset()
    if bt.bt_device_status() != 0:
        raise RuntimeError("device status after the survey")
    return {"metric": "measured selection survey", "pass": "tune-survey", "n_gpus": 1, "reps": args.tune_reps,
            "how": "whole public calls on x timed per candidate with CUDA events; a candidate replaces the "
                   "planner's choice only when > 1 % faster", "layers": rows}


def run_w8a8(args, rank, world):
    """K steps of the W8A8 im2col + gemm convolution on the workload's x and W
    (quantization of both sides inside every step)."""
    import xnor_popcount_gemm_gb300 as bt

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    wl = workloads.NAMED[args.workload]()
    if wl.kind != "conv":
        raise SystemExit("--pass w8a8 covers the conv workloads")
    smooth = args.pass_ == "w8a8-smooth"
    M, N, K = wl.gemm_shape()
    B, C, H, W = wl.x.shape
    O, k = wl.w.shape[0], wl.w.shape[2]
    stream = torch.cuda.current_stream()
    x_host = wl.x if wl.x.dtype in (torch.bfloat16, torch.float32) else wl.x.float()
    w = wl.w.to(x_host.dtype).to(dev)
    Ho = bt.conv2d_out_size(H, k, wl.stride, wl.padding, wl.dilation)
    Wo = bt.conv2d_out_size(W, k, wl.stride, wl.padding, wl.dilation)
    out_t = torch.float32
    per = x_host.numel() * x_host.element_size() + B * O * Ho * Wo * 4
    nbuf = max(1, -(-2 * L2_BYTES // per))
    xs = [x_host.to(dev) for _ in range(nbuf)]
    outs = [torch.empty(B, O, Ho, Wo, dtype=out_t, device=dev) for _ in range(nbuf)]
    ws = torch.empty(bt.bt_w8a8_conv2d_workspace(B, C, H, W, O, k, wl.stride, wl.padding, wl.dilation),
                     dtype=torch.uint8, device=dev)

    def step(i):
        j = i % nbuf
        bt.bt_w8a8_conv2d(xs[j], w, wl.stride, wl.padding, wl.dilation, smooth=smooth, out=outs[j], workspace=ws)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    assert bt.bt_device_status() == 0
    with ClockSampler(dev.index) as clk:
        barrier(world)
        torch.cuda.synchronize()
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        for i in range(args.steps):
            step(i)
        a1.record(stream)
        torch.cuda.synchronize()
    ms = max_over_ranks(a0.elapsed_time(a1), world) / args.steps
    if bt.bt_device_status() != 0:
        raise RuntimeError("device status")
    peaks, peak_src = measured_peaks()
    ops = 2.0 * M * N * K
    return {
        "metric": "W8A8 conv GOPS (2*M*N*K/s, quantization included)",
        "value": round(ops * world / (ms / 1e3) / 1e9, 1),
        "unit": "GOPS", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms, 5), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "int8 x int8 as bf16 on the tensor cores (exact fp32 K splits, double sum)",
        "data": "synthetic (the workload's x and W)",
        "config": {"workload": wl.name, "pass": args.pass_, "M": M, "N": N, "K": K,
                   "l2": f"inputs+outputs rotate over {nbuf} buffers", "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "tensor", "achieved": round(ops / (ms / 1e3) / 1e12, 2), "peak": peaks["bf16_tflops"],
                     "unit": "TFLOP/s", "frac": round(ops / (ms / 1e3) / 1e12 / peaks["bf16_tflops"], 4),
                     "traffic": None, "peak_source": f"{peak_src}: cuBLAS bf16 burst", "kernel": "whole call"},
        "gpu_launches": 9 * args.steps,
        "clocks": clk.summary(),
    }


# ---------------------------------------------------------------------------
# the oracle on the host cores
# ---------------------------------------------------------------------------

def oracle_forward(wl, rows: int):
    import oracle
    if wl.kind == "linear":
        return oracle.binary_linear(wl.x[:rows], wl.w, wl.scale_a, wl.scale_w, wl.bias, wl.out_dtype)
    return oracle.binary_conv2d(wl.x[:rows], wl.w, wl.scale_a, wl.scale_w, wl.stride, wl.padding,
                                wl.dilation, wl.bias, wl.out_dtype)


def sample_rows(wl, budget_ops: float) -> int:
    """Rows (linear) or images (conv) of the workload whose forward is about
    `budget_ops` binary ops."""
    total = wl.x.shape[0]
    per = wl.binary_ops() / total
    return int(max(1, min(total, budget_ops // per)))


def cpu_baseline(wl, budget_ops: float = 1.5e11):
    rows = sample_rows(wl, budget_ops)
    ops = wl.binary_ops() * rows / wl.x.shape[0]
    t = time.perf_counter()
    oracle_forward(wl, rows)
    dt = time.perf_counter() - t
    return {"value": round(ops / dt / 1e9, 3), "unit": "GOPS", "cores": len(os.sched_getaffinity(0)),
            "kind": "oracle", "seconds": round(dt, 2),
            "sample": f"first {rows} of {wl.x.shape[0]} {'rows' if wl.kind == 'linear' else 'images'} "
                      f"of {wl.name} (binarize + nested-loop dot + epilogue)"}


def run_reference(args, rank, world):
    wl = workloads.NAMED[args.workload]()
    rows = sample_rows(wl, 2.0e10)
    ops = wl.binary_ops() * rows / wl.x.shape[0]
    for _ in range(args.warmup):
        oracle_forward(wl, rows)
    t = time.perf_counter()
    for _ in range(args.steps):
        oracle_forward(wl, rows)
    dt = (time.perf_counter() - t) / args.steps
    value = ops / dt / 1e9
    cores = len(os.sched_getaffinity(0))
    sample = f"first {rows} of {wl.x.shape[0]} rows/images of {wl.name} per step"
    return {"impl": "reference", "metric": "binary GOPS (2*M*N*K/s)", "value": round(value, 3), "unit": "GOPS",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int8 +-1 (int32 acc)",
            "data": "synthetic (seeded; shapes of binarized LLM linear and ResNet conv layers)",
            "config": {"workload": wl.name, "sample_rows": rows},
            "cpu_baseline": {"value": round(value, 3), "unit": "GOPS", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 3), "unit": "GOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    args = parse()
    if args.impl == "reference":
        # rank 0 alone times the oracle on the host cores; other ranks exit
        rank, world = int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1"))
        if rank != 0:
            return
        print(json.dumps(run_reference(args, rank, world)), flush=True)
        return
    rank, world = dist_init(args)
    if args.pass_ == "backward":
        line = run_backward(args, rank, world)
    elif args.pass_ == "tune-survey":
        line = run_tune_survey(args, rank, world)
    elif args.pass_.startswith("w8a8"):
        line = run_w8a8(args, rank, world)
    else:
        line = run_ours(args, rank, world)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
