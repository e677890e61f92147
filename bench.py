#!/usr/bin/env python
"""Benchmark of the stencil library on one GB300 (or N replicas under torchrun).

Headline workload: AvgPool3d(k3, s2, p1, count_include_pad) on x fp32
[16,32,128,128,256] (the Kimi-K2.6__l1_p46 task).  A step is one pass of the
op over one batch; `value` is outputs/s of the whole job with the input
resident in HBM (8.59 GB, larger than L2, so no flush is needed).  The line
also carries:
  * roofline -- algorithmic bytes per launch (input read once + output written
    once) / the kernel's average CUDA-event duration on its launch stream,
    against the measured copy bandwidth in MEASURED_PEAKS.json;
  * e2e -- the same metric through the C ABI with host buffers: every step
    copies the input from pinned host memory, runs the op and reads the output
    back, all inside the timed region;
  * cpu_baseline -- the fp64 oracle on the host cores, on a bounded sample of
    (n, c) planes of the same workload, with the CPU model and thread count;
  * clocks -- nvidia-smi samples taken during the timed region;
  * per_config (the last key, kept compact) -- every other workload and kernel
    path: per entry the time per launch, outputs/s, the roofline (bound,
    achieved, fraction of the binding peak, DRAM traffic per launch from the
    committed ncu summary of that kernel's source) and the oracle's outputs/s
    on a sample of the same workload on the host cores.

`--impl reference` times the oracle itself (the only other leg that runs
oracle code) on the same workload and prints the same line shape.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
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

METRIC = "outputs/s and % of binding roofline (HBM GB/s or FP32/TF32 FLOP/s) per config"
HEADLINE_CFG = 1
SMS = 152
FP32_LANES_PER_SM = 128


def parse_args():
    return parse_args_from(sys.argv[1:])


def parse_args_from(argv):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--e2e-steps", type=int, default=8, help="0 skips the e2e leg")
    ap.add_argument("--workload", type=int, default=HEADLINE_CFG,
                    help="workload of the headline line (default: the avgpool workload)")
    ap.add_argument("--precision", choices=["fp32", "tf32", "tf32x3", "fp32_fma"],
                    default="fp32",
                    help="ConvTranspose1d precision of the headline workload (fp32: the "
                         "library's choice at the fp32 bound; fp32_fma: the FP32 pipe)")
    ap.add_argument("--x-shape", type=str, default=None,
                    help="override the input shape of the headline workload (profiling "
                         "runs on small cases), e.g. 2,32,128,128,256")
    ap.add_argument("--no-per-config", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="target CPU time of the oracle sample")
    ap.add_argument("--cpu-seconds-per-config", type=float, default=2.0,
                    help="target CPU time of each per-config oracle sample")
    ap.add_argument("--only", type=str, default=None,
                    help="comma-separated per-config keys to run (default: all)")
    return ap.parse_args(argv)


# ----------------------------------------------------------------- helpers
def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "sm_max_mhz": 2070.0}, "fallback"


def fp32_peak_tflops(mhz):
    """FP32 FMA peak: 152 SMs x 128 lanes x 2 FLOP per clock."""
    return SMS * FP32_LANES_PER_SM * 2 * mhz * 1e6 / 1e12


def numel(shape):
    return int(math.prod(shape))


def convt_pairs(L, L_out, K, s, p, d):
    """Number of (i, k) pairs whose output index i*s - p + k*d lands in range
    (the in-range taps of a transposed convolution, per channel pair)."""
    n = 0
    for k in range(K):
        lo = max(0, -((k * d - p) // s))          # ceil((p - k*d) / s)
        hi = min(L - 1, (L_out - 1 + p - k * d) // s)
        n += max(0, hi - lo + 1)
    return n


def pooled_cells(L, P_out, K, s, p, d, q):
    """Input cells read, summed over the pooled outputs of one dim: pooled output P
    covers pre-pool positions [qP, qP + q), whose taps read inputs (o + p - d*k)/s
    where that is an integer in [0, L); each distinct input counts once (the
    collapsed weights of the fused op)."""
    n = 0
    for P in range(P_out):
        cells = {(o + p - d * k) // s for o in range(q * P, q * P + q) for k in range(K)
                 if (o + p - d * k) % s == 0 and 0 <= (o + p - d * k) // s < L}
        n += len(cells)
    return n


class ClockSampler:
    """nvidia-smi samples of the SM clock and throttle reasons, in the background."""
    FIELDS = ["timestamp", "clocks.sm", "clocks.max.sm", "power.draw",
              "clocks_event_reasons.active", "clocks_event_reasons.hw_slowdown",
              "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, index, interval_ms=100):
        self.samples = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(index), "--query-gpu=" + ",".join(self.FIELDS),
                 "--format=csv,noheader,nounits", "-lms", str(interval_ms)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) == len(self.FIELDS):
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        sel = [p for (t, p) in self.samples if t0 <= t <= t1 + 0.15]
        if not sel:
            sel = [p for (_, p) in self.samples[-3:]]
        if not sel:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"]}
        mhz = [float(p[1]) for p in sel if re.match(r"^[\d.]+$", p[1])]
        mx = [float(p[2]) for p in sel if re.match(r"^[\d.]+$", p[2])]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in sel for i in range(4) if p[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(mhz) if mhz else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(sel)}


def traffic_from_profile(kernel_file, profile_name, key):
    """DRAM bytes per launch of per-config workload `key`, recorded in
    profiles/<profile_name> as `traffic_bytes_per_launch[key]: <bytes>` beside the
    sha256 prefix of the kernel source it was measured on.  Returns the bytes,
    "stale" when the source has changed since, or None when nothing is recorded."""
    prof = os.path.join(ROOT, "profiles", profile_name)
    src = os.path.join(ROOT, "average_pooling_stencil_gb300", "csrc", kernel_file)
    if not (os.path.exists(prof) and os.path.exists(src)):
        return None
    text = open(prof).read()
    m = re.search(r"traffic_bytes_per_launch\[" + re.escape(key) + r"\]:\s*([0-9.eE+]+)", text)
    h = re.search(r"source_sha256_16:\s*([0-9a-f]{16})", text)
    if not (m and h):
        return None
    cur = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    return float(m.group(1)) if cur == h.group(1) else "stale"


# kernel source and committed ncu summary behind each measured workload (the
# summary holds that kernel's DRAM bytes per launch, keyed by workload)
PROFILE_OF = {
    "avgpool": ("avgpool3d.cu", "avgpool3d_k3s2p1_tma.md"),
    "avgpool_nopad": ("avgpool3d.cu", "avgpool3d_k3s2p1_tma.md"),
    "avgpool_k2": ("avgpool3d.cu", "avgpool3d_k2s2_vec.md"),
    "fused": ("ct3d_pool_tc.cu", "ct3d_pool2_tc_fused.md"),
    "fused_cin8": ("ct3d_pool_tc.cu", "ct3d_pool2_tc_chunked_cin8.md"),
    "fused_op1": ("ct3d_pool_tc.cu", "ct3d_pool2_tc_fused.md"),
    "fused_k4": ("ct3d_pool_gen.cu", "ct3d_pool_gen_k4.md"),
    "fused_w30": ("ct3d_pool.cu", "ct3d_pool2_fast_fused_w30.md"),
    "convt1d": ("convt1d.cu", "convt1d_tiled_fp32.md"),
    "convt1d_strided": ("convt1d.cu", "convt1d_tiled_fp32.md"),
    "convt1d_tf32": ("convt1d_tc.cu", "convt1d_tf32.md"),
    "convt1d_strided_tf32": ("convt1d_tc.cu", "convt1d_tf32.md"),
    "convt1d_tf32x3": ("convt1d_tc.cu", "convt1d_tf32x3.md"),
    "convt1d_strided_tf32x3": ("convt1d_tc.cu", "convt1d_tf32x3.md"),
    "convt3d": ("convt3d_tc.cu", "convt3d_tc_k3s2p1.md"),
    "convt3d_cin8": ("convt3d_tc.cu", "convt3d_tc_k3s2p1_cin8.md"),
    "convt3d_w64": ("convt3d_tc.cu", "convt3d_tc_k3s2p1_w64.md"),
}

# per-config workloads: key, workload id, ConvTranspose1d precision (the C ABI's value:
# 0 fp32 as the library routes it, 1 tf32, 2 3xTF32, 3 fp32 on the FP32 pipe), timing mode
PER_CONFIG = [
    ("fused_tiny", 0, 0, "graph"),
    ("fused", 2, 0, "rotate"),
    ("fused_cin8", 6, 0, "rotate"),
    ("fused_op1", 7, 0, "rotate"),
    ("fused_k4", 11, 0, "rotate"),
    ("fused_w30", 13, 0, "rotate"),
    ("avgpool_nopad", 8, 0, "plain"),
    ("avgpool_k2", 9, 0, "plain"),
    ("convt1d", 3, 3, "plain"),
    ("convt1d_tf32", 3, 1, "plain"),
    ("convt1d_tf32x3", 3, 2, "plain"),
    ("convt1d_strided", 4, 3, "plain"),
    ("convt1d_strided_tf32", 4, 1, "plain"),
    ("convt1d_strided_tf32x3", 4, 2, "plain"),
    ("convt3d", 5, 0, "plain"),
    ("convt3d_cin8", 10, 0, "plain"),
    ("convt3d_w64", 12, 0, "plain"),
]


def sig(v, n=4):
    """`v` rounded to n significant digits (keeps the JSON line short)."""
    if v is None or isinstance(v, str) or v == 0 or not math.isfinite(v):
        return v
    return float(f"{v:.{n}g}")


def compact_json(obj):
    """json.dumps without spaces, integer-valued floats of 7+ digits in exponent
    form (4.426e11 rather than 442600000000.0): the line stays short enough that
    the per-config block at its end survives a tail of a few KB."""
    s = json.dumps(obj, separators=(",", ":"))

    def exp(m):
        import numpy as np   # shortest exact scientific form
        t = np.format_float_scientific(float(m.group(2)), unique=True, trim="-")
        return m.group(1) + t.replace("e+", "e")
    return re.sub(r"([:\[,])(\d{7,})\.0(?=[,}\]])", exp, s)


def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the platform)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu model")):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.processor() or platform.machine()


# --------------------------------------------------------------- workloads
def workload_desc(wl):
    shp = "x".join(map(str, wl.tensors["x"][0]))
    p = wl.params
    if wl.op == "avgpool3d":
        g = "k{}{}{} s{}{}{} p{}{}{}".format(*p["k"], *p["stride"], *p["pad"])
        g = re.sub(r"([kps])(\d)\2\2", r"\1\2", g)
        cip = "count_include_pad" if p["count_include_pad"] else "count_include_pad=False"
        return f"avgpool3d {g} {cip} x[{shp}] fp32"
    if wl.op == "ct3d_scale_pool_bias":
        op = "" if not any(p["out_pad"]) else ",op{}".format(p["out_pad"][0])
        return (f"convtranspose3d(k3,s2,p1{op})+x{p['scale1']}+avgpool3d(2)+bias+x{p['scale2']} "
                f"x[{shp}] fp32")
    if wl.op == "convtranspose3d":
        return (f"convtranspose3d k3 s2 p1 d1 op0 x[{shp}] -> C_out {p['c_out']} "
                f"(the pre-pool tensor) fp32")
    return (f"convtranspose1d K{p['k']} s{p['stride']} p{p['pad']} d{p['dil']} "
            f"op{p['out_pad']} x[{shp}] -> C_out {p['c_out']} fp32")


def line_config(wl, ws):
    """The `config` object of a bench line (the same for both arms)."""
    in_bytes = 4 * numel(wl.tensors["x"][0])
    return {"workload": workload_desc(wl), "seed": wl.seed,
            "l2": (f"input larger than L2 ({in_bytes / 1e9:.2f} GB read per step), no flush"
                   if in_bytes > 2 * 129e6 else "input may stay in L2 (small case)"),
            "parallelism": f"replicas{ws}" if ws > 1 else "single GPU"}


_HOST = {}


def host_tensor(torch, wl, name, pin=False):
    """The workload tensor `name` in (optionally pinned) host memory, generated once
    per (seed, recipe, shape) in this process and shared by the cases that use it."""
    shape, dist, stream = wl.tensors[name]
    key = (wl.seed, stream, tuple(shape), tuple(dist))
    h = _HOST.get(key)
    if h is None or (pin and not h.is_pinned()):
        h = torch.empty(shape, dtype=torch.float32, pin_memory=pin)
        wl.generate(name, out=h.numpy())
        _HOST[key] = h
    return h


def release_host(keep=()):
    """Drops the cached host tensors other than `keep`."""
    for k in [k for k, v in _HOST.items() if not any(v is t for t in keep)]:
        del _HOST[k]


class GpuCase:
    """Device-resident inputs/outputs of one workload plus its launch closure."""

    def __init__(self, cfg, torch, aps, with_host=False, x_shape=None, precision=0):
        from average_pooling_stencil_gb300 import workloads
        self.cfg = cfg
        self.precision = precision
        self.kind = None          # ConvTranspose1d: the precision the library actually ran
        self.wl = wl = workloads.get(cfg)
        if x_shape is not None:
            self.wl = wl = wl.with_input_shape(x_shape)
        self.torch = torch
        p = wl.params
        dev = torch.device("cuda")
        names = [n for n in ("x", "w", "conv_bias", "bias") if n in wl.tensors]
        self.host = {}
        self.d = {}
        for n in names:
            h = host_tensor(torch, wl, n, pin=with_host and n == "x")
            self.host[n] = h
            self.d[n] = h.to(dev, non_blocking=False)
        x = self.d["x"]
        self.tc = False
        self.chunked = False
        self.tensor_passes = 0
        if wl.op == "avgpool3d":
            st, oshape = aps.binding.aps_avgpool3d_out_shape(x.shape, p["k"], p["stride"],
                                                             p["pad"], p["ceil_mode"])
            self.flops = numel(p["k"]) * numel(oshape)        # window adds
            self.bound = "hbm"
        elif wl.op == "ct3d_scale_pool_bias":
            st, oshape = aps.binding.aps_ct3d_scale_pool_bias_out_shape(
                x.shape, p["c_out"], p["k"], p["stride"], p["pad"], p["out_pad"], p["dil"],
                p["pool_k"])
            cin = x.shape[1]
            fast = (tuple(p["k"]) == (3, 3, 3) and tuple(p["stride"]) == (2, 2, 2)
                    and tuple(p["pad"]) == (1, 1, 1) and all(o <= 1 for o in p["out_pad"])
                    and tuple(p["dil"]) == (1, 1, 1) and p["pool_k"] == 2
                    and p["c_out"] == 16 and 1 <= cin <= 8)
            if fast:
                self.flops = 2 * 8 * cin * numel(oshape)      # 8 collapsed taps per ci
            else:
                # the collapsed form of any geometry: per pooled output and input
                # channel, one multiply-add per input cell its window reads
                cells = 1
                for i in range(3):
                    cells *= pooled_cells(x.shape[2 + i], oshape[2 + i], p["k"][i],
                                          p["stride"][i], p["pad"][i], p["dil"][i],
                                          p["pool_k"])
                self.flops = 2 * x.shape[0] * cin * p["c_out"] * cells
            # 16-byte input rows run on the tensor cores (3xTF32, three MMA passes;
            # C_in 4..8 in chunks of <= 3 channels), bound by HBM; otherwise on the
            # FP32 pipe
            self.tc = fast and x.shape[4] % 4 == 0
            self.chunked = self.tc and cin > 3
            self.tensor_passes = 3 if self.tc else 0
            self.bound = "hbm" if self.tc else "hbm+alu"
        elif wl.op == "convtranspose3d":
            st, oshape = aps.binding.aps_convtranspose3d_out_shape(
                x.shape, p["c_out"], p["k"], p["stride"], p["pad"], p["dil"], p["out_pad"])
            pairs = 1
            for i in range(3):   # in-range taps, per dim
                pairs *= convt_pairs(x.shape[2 + i], oshape[2 + i], p["k"][i], p["stride"][i],
                                     p["pad"][i], p["dil"][i])
            self.flops = 2 * x.shape[0] * x.shape[1] * p["c_out"] * pairs
            self.tc = x.shape[1] <= 8 and x.shape[4] % 4 == 0
            self.tensor_passes = 3 if self.tc else 0
            self.bound = "hbm" if self.tc else "hbm+alu"
        else:
            st, oshape = aps.binding.aps_convtranspose1d_out_shape(
                x.shape, p["c_out"], p["k"], p["stride"], p["pad"], p["dil"], p["out_pad"])
            pairs = convt_pairs(x.shape[2], oshape[2], p["k"], p["stride"], p["pad"], p["dil"])
            self.flops = 2 * x.shape[0] * x.shape[1] * p["c_out"] * pairs
        assert st == 0
        self.oshape = oshape
        self.y = torch.empty(oshape, device=dev, dtype=torch.float32)
        if wl.op == "convtranspose1d":
            # APS_PREC_FP32 runs the 3xTF32 kernel where it takes the shape, else
            # the FP32 pipe: one 3xTF32 launch tells which
            self.kind = precision
            if precision == 0:
                bias = self.d["bias"].data_ptr() if "bias" in self.d else 0
                st = aps.binding.aps_convtranspose1d(
                    self.d["x"].data_ptr(), x.shape, self.d["w"].data_ptr(), bias, p["c_out"],
                    p["k"], p["stride"], p["pad"], p["dil"], p["out_pad"], 2,
                    self.y.data_ptr(), torch.cuda.current_stream().cuda_stream)
                self.kind = 2 if st == 0 else 3
            # the FP32-pipe kernels are bound by the FP32 pipe, the tensor-core ones by HBM
            self.bound = "alu" if self.kind == 3 else "hbm"
            self.tensor_passes = {3: 0, 1: 1, 2: 3}[self.kind]
        self.bytes = 4 * (sum(numel(t.shape) for t in self.d.values()) + numel(oshape))
        self.outputs = numel(oshape)
        self.aps = aps
        self.stream = torch.cuda.current_stream()
        if with_host:
            self.yh = torch.empty(oshape, dtype=torch.float32, pin_memory=True)

    def launch(self):
        B = self.aps.binding
        p = self.wl.params
        d = self.d
        s = self.stream.cuda_stream
        if self.wl.op == "avgpool3d":
            st = B.aps_avgpool3d(d["x"].data_ptr(), d["x"].shape, p["k"], p["stride"], p["pad"],
                                 p["count_include_pad"], p["ceil_mode"], self.y.data_ptr(), s)
        elif self.wl.op == "ct3d_scale_pool_bias":
            st = B.aps_ct3d_scale_pool_bias(
                d["x"].data_ptr(), d["x"].shape, d["w"].data_ptr(), d["conv_bias"].data_ptr(),
                d["bias"].data_ptr(), p["c_out"], p["k"], p["stride"], p["pad"], p["out_pad"],
                p["dil"], p["pool_k"], p["scale1"], p["scale2"], self.y.data_ptr(), s)
        elif self.wl.op == "convtranspose3d":
            st = B.aps_convtranspose3d(d["x"].data_ptr(), d["x"].shape, d["w"].data_ptr(),
                                       d["bias"].data_ptr(), p["c_out"], p["k"], p["stride"],
                                       p["pad"], p["dil"], p["out_pad"], self.y.data_ptr(), s)
        else:
            bias = d["bias"].data_ptr() if "bias" in d else 0
            st = B.aps_convtranspose1d(d["x"].data_ptr(), d["x"].shape, d["w"].data_ptr(), bias,
                                       p["c_out"], p["k"], p["stride"], p["pad"], p["dil"],
                                       p["out_pad"], self.precision, self.y.data_ptr(), s)
        if st != 0:
            raise RuntimeError(f"launch failed: {B.status_string(st)}")

    def e2e_step(self):
        """Host x -> device, op, device y -> host, on the launch stream."""
        self.d["x"].copy_(self.host["x"], non_blocking=True)
        self.launch()
        self.yh.copy_(self.y, non_blocking=True)


class E2EPipeline:
    """The e2e steps as a stream: step k's host -> device copy, op and device -> host
    read on three streams, with two device copies of x and y, so that the copy of step
    k+1's input overlaps step k's op and the read of its result (the host link carries
    both directions at once).  Every step still moves its own input and result."""

    def __init__(self, torch, case):
        self.torch, self.case = torch, case
        self.x = [case.d["x"], torch.empty_like(case.d["x"])]
        self.y = [case.y, torch.empty_like(case.y)]
        self.yh = [case.yh, torch.empty_like(case.yh).pin_memory()]
        self.s_in, self.s_out = torch.cuda.Stream(), torch.cuda.Stream()
        self.s_op = case.stream
        ev = lambda: torch.cuda.Event()
        self.x_ready, self.x_free = [ev(), ev()], [ev(), ev()]
        self.y_ready, self.y_free = [ev(), ev()], [ev(), ev()]
        self.k = 0

    def step(self):
        b = self.k & 1
        c = self.case
        if self.k >= 2:
            self.s_in.wait_event(self.x_free[b])        # op k-2 has read x[b]
        with self.torch.cuda.stream(self.s_in):
            self.x[b].copy_(c.host["x"], non_blocking=True)
        self.x_ready[b].record(self.s_in)
        self.s_op.wait_event(self.x_ready[b])
        if self.k >= 2:
            self.s_op.wait_event(self.y_free[b])        # y[b] of step k-2 is read back
        c.d["x"], c.y = self.x[b], self.y[b]
        c.launch()
        self.x_free[b].record(self.s_op)
        self.y_ready[b].record(self.s_op)
        self.s_out.wait_event(self.y_ready[b])
        with self.torch.cuda.stream(self.s_out):
            self.yh[b].copy_(self.y[b], non_blocking=True)
        self.y_free[b].record(self.s_out)
        self.k += 1

    def restore(self):
        self.case.d["x"], self.case.y = self.x[0], self.y[0]


def time_launches(torch, case, reps, flush=None):
    """Average device time of one launch (CUDA events on the launch stream)."""
    st = case.stream
    if flush is None:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(st)
        for _ in range(reps):
            case.launch()
        e1.record(st)
        e1.synchronize()
        return e0.elapsed_time(e1) / 1e3 / reps
    tot = 0.0
    for _ in range(reps):
        flush.add_(1.0)   # a write larger than L2 between launches, outside the events
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(st)
        case.launch()
        e1.record(st)
        e1.synchronize()
        tot += e0.elapsed_time(e1) / 1e3
    return tot / reps


def time_rotating(torch, cases, reps):
    """Average device time of one launch over back-to-back launches that rotate
    through several input/output sets (all on one stream) whose total is well
    above L2, so that no launch finds its data in L2 and no flush kernel runs
    between them."""
    st = cases[0].stream
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(st)
    for i in range(reps):
        cases[i % len(cases)].launch()
    e1.record(st)
    e1.synchronize()
    return e0.elapsed_time(e1) / 1e3 / reps


def time_graph(torch, case, per_graph=100, reps=20):
    """Launch-latency-bound workload: average launch time inside a CUDA graph."""
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        case.stream = s
        case.launch()
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=s):
            for _ in range(per_graph):
                case.launch()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(s):
        g.replay()
        e0.record(s)
        for _ in range(reps):
            g.replay()
        e1.record(s)
    e1.synchronize()
    case.stream = torch.cuda.current_stream()
    return e0.elapsed_time(e1) / 1e3 / (reps * per_graph)


def measure_fma_ceilings(torch, aps, sms, iters=4096, reps=5):
    """FP32 FMA rate this GPU sustains (TFLOP/s), scalar and packed fp32x2,
    from the library's register-only probe at 64 warps per SM."""
    B = aps.binding
    sink = torch.zeros(1, device="cuda")
    st = torch.cuda.current_stream()
    blocks = sms * 8
    out = {}
    for packed in (0, 1):
        for _ in range(2):
            assert B.aps_fp32_fma_probe(packed, blocks, iters, sink.data_ptr(), st.cuda_stream) == 0
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(st)
        for _ in range(reps):
            B.aps_fp32_fma_probe(packed, blocks, iters, sink.data_ptr(), st.cuda_stream)
        e1.record(st)
        e1.synchronize()
        t = e0.elapsed_time(e1) / 1e3
        flops = 64.0 * iters * blocks * B.APS_PROBE_THREADS * reps
        out["packed" if packed else "scalar"] = flops / t / 1e12
    return out


def measure_tf32_ceiling(torch, n=8192, reps=5):
    """Dense TF32 tensor-core rate (TFLOP/s) of the vendor GEMM (cuBLAS through
    torch.matmul with TF32 allowed) on n x n x n: a ceiling for the tensor work
    of the TF32 paths, measured only, never on an op's path."""
    prev = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = True
    try:
        a = torch.randn(n, n, device="cuda")
        b = torch.randn(n, n, device="cuda")
        for _ in range(2):
            c = a @ b
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            c = a @ b
        e1.record()
        e1.synchronize()
        del a, b, c
        return 2.0 * n ** 3 * reps / (e0.elapsed_time(e1) / 1e3) / 1e12
    finally:
        torch.backends.cuda.matmul.allow_tf32 = prev


def roofline_for(case, t, peaks, src, clock_mhz):
    hbm = float(peaks["hbm_gbs"])
    gbs = case.bytes / t / 1e9
    tfl = case.flops / t / 1e12
    fp32 = fp32_peak_tflops(float(peaks.get("sm_max_mhz", 2070.0)))
    if case.bound == "hbm":
        r = {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s", "frac": gbs / hbm,
             "peak_source": src}
        tc = peaks.get("tf32_measured")
        passes = getattr(case, "tensor_passes", 0)
        if passes and tc:
            # tensor work: one MMA product per FLOP pair, three for 3xTF32
            work = case.flops * passes / t / 1e12
            r["tensor_tflops"] = work
            r["tensor_ceiling"] = tc
            r["tensor_frac_of_ceiling"] = work / tc
            r["tensor_ceiling_source"] = "cuBLAS TF32 GEMM 8192^3 timed in this run"
        return r
    if case.bound == "alu":
        r = {"bound": "alu", "achieved": tfl, "peak": fp32, "unit": "TFLOP/s",
             "frac": tfl / fp32,
             "peak_source": "152 SMs x 128 FP32 lanes x 2 FLOP x max SM clock "
                            f"{peaks.get('sm_max_mhz', 2070.0)} MHz"}
        fma = peaks.get("fma_measured")
        if fma:
            r["measured_ceiling"] = fma["packed"]
            r["frac_of_measured_ceiling"] = tfl / fma["packed"]
            r["measured_ceiling_source"] = (
                "packed fp32x2 FMA probe (aps_fp32_fma_probe, 64 warps/SM) timed in this run; "
                f"scalar FMA {fma['scalar']:.1f} TFLOP/s")
        return r
    floor = max(case.bytes / (hbm * 1e9), case.flops / (fp32 * 1e12))
    return {"bound": "hbm" if case.bytes / (hbm * 1e9) >= case.flops / (fp32 * 1e12) else "alu",
            "achieved": gbs, "unit": "GB/s", "peak": hbm, "frac": floor / t,
            "achieved_tflops": tfl, "peak_tflops": fp32,
            "note": "frac = max(HBM floor, FP32 floor) / measured time", "peak_source": src}


# ------------------------------------------------------------------ oracle
def oracle_sample(wl, seconds, host=None, whole=False):
    """Time the oracle (as it stands) on a bounded sample of output planes of
    workload `wl`, sized to about `seconds` of CPU time (`whole`: every plane).
    `host` maps tensor names to the workload's arrays already in host memory
    (generated from the workload's seed if absent).  Returns (outputs/s,
    threads, description, outputs, seconds)."""
    import numpy as np

    import oracle
    p = wl.params
    xs = tuple(wl.tensors["x"][0])
    N, C = xs[0], xs[1]
    threads = oracle.threads()
    host = host or {}
    tens = {n: (np.asarray(host[n]).reshape(wl.tensors[n][0]) if n in host else wl.generate(n))
            for n in wl.tensors}
    x = tens["x"]
    if wl.op == "avgpool3d":
        units = [(n, c) for n in range(N) for c in range(C)]

        def run(planes):
            t0 = time.perf_counter()
            y = oracle.avgpool3d(x, p["k"], p["stride"], p["pad"], p["count_include_pad"],
                                 p["ceil_mode"], sel=planes)
            return time.perf_counter() - t0, y.size
    else:
        units = [(n, co) for n in range(N) for co in range(p["c_out"])]

        def run(planes):
            t0 = time.perf_counter()
            if wl.op == "ct3d_scale_pool_bias":
                y = oracle.ct3d_scale_pool_bias(x, tens["w"], tens["conv_bias"], tens["bias"],
                                                p["stride"], p["pad"], p["out_pad"], p["dil"],
                                                p["pool_k"], p["scale1"], p["scale2"], sel=planes)
            else:
                y = oracle.convt(x, tens["w"], tens.get("bias"), p["stride"], p["pad"], p["dil"],
                                 p["out_pad"], sel=planes)
            return time.perf_counter() - t0, y.size
    if whole:
        sample = units
    else:
        # calibrate on one plane per thread, then size the sample to `seconds`
        k = min(len(units), max(1, threads))
        t, _ = run(units[:k])
        m = int(min(len(units), max(k, round(seconds * k / max(t, 1e-6)))))
        step = max(1, len(units) // m)
        sample = units[::step][:m]
    t, cnt = run(sample)
    desc = f"{len(sample)} of {len(units)} (n, c) output planes of {workload_desc(wl)}"
    return cnt / t, threads, desc, cnt, t


# ------------------------------------------------------------------- legs
def max_over_ranks(dist, value, device):
    """The largest `value` over all ranks (the job's time), or `value` itself
    when the run is not distributed."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(world_size, units_per_rank_step, steps, t_max):
    """Units all ranks processed per second: every rank runs the same full
    workload (weak scaling) and the job takes as long as its slowest rank."""
    return world_size * units_per_rank_step * steps / t_max


def sm_count_of(torch):
    return torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    from average_pooling_stencil_gb300 import workloads
    wl = workloads.get(HEADLINE_CFG)
    oracle.build()
    x = wl.generate("x")
    per_step = max(1.0, min(args.cpu_seconds, 60.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_sample(wl, per_step, {"x": x})
    vals, times, desc, threads = [], [], "", 1
    for _ in range(args.steps):
        v, threads, desc, cnt, t = oracle_sample(wl, per_step, {"x": x})
        vals.append(v)
        times.append(t)
    value = sum(times) and sum(v * t for v, t in zip(vals, times)) / sum(times)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "outputs/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * statistics.mean(times), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": line_config(wl, ws),
        "cpu_baseline": {"value": value, "unit": "outputs/s", "cores": threads, "kind": "oracle",
                         "model": cpu_model(), "sample": f"per step: {desc}"},
        "e2e": {"value": value, "unit": "outputs/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line))
    return 0


# per_config columns: the driver keeps only the last 1500 characters of the
# output, so each workload is one array in this order
PER_CONFIG_COLS = ["us", "out_s", "frac", "bound", "dram_B", "cpu_out_s"]


def per_config_entry(key, c, t, peaks, peak_src, cpu_out_s):
    """One per_config entry, in PER_CONFIG_COLS order: time per launch (us),
    outputs/s, fraction of the binding roofline, its kind ("hbm": measured copy
    peak; "alu": FP32 unit peak), DRAM bytes per launch from the kernel's profile
    (or "stale" / None) and the oracle's outputs/s on the host cores."""
    r = roofline_for(c, t, peaks, peak_src, None)
    src = PROFILE_OF.get(key)
    return [sig(1e6 * t), sig(c.outputs / t, 3), sig(r["frac"], 3), r["bound"],
            sig(traffic_from_profile(src[0], src[1], key), 3) if src else None,
            sig(cpu_out_s, 3)]


def run_native(args):
    import torch

    import average_pooling_stencil_gb300 as aps
    from average_pooling_stencil_gb300 import build as aps_build
    ws, rank, local = dist_env()
    dist = None
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    aps_build.build()
    peaks, peak_src = load_peaks()
    # measured FP32 FMA ceilings (outside every timed region), for the FMA-bound lines
    peaks = dict(peaks)
    peaks["fma_measured"] = measure_fma_ceilings(torch, aps, sm_count_of(torch))
    peaks["tf32_measured"] = measure_tf32_ceiling(torch)
    dev_index = local if ws > 1 else 0

    def barrier():
        if dist:
            dist.barrier()
        torch.cuda.synchronize()

    # ---- headline: each rank runs its own full workload (weak scaling)
    x_shape = tuple(int(v) for v in args.x_shape.split(",")) if args.x_shape else None
    case = GpuCase(args.workload, torch, aps, with_host=args.e2e_steps > 0, x_shape=x_shape,
                   precision={"fp32": 0, "tf32": 1, "tf32x3": 2, "fp32_fma": 3}[args.precision])
    for _ in range(max(3, args.warmup)):
        case.launch()
    barrier()
    sampler = ClockSampler(dev_index, 50)
    time.sleep(0.6)   # nvidia-smi start-up
    st = case.stream
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    t_wall0 = time.time()
    e0.record(st)
    for _ in range(args.steps):
        case.launch()
    e1.record(st)
    barrier()
    t_wall1 = time.time()
    sampler.stop()
    t_dev = e0.elapsed_time(e1) / 1e3
    t_max = max_over_ranks(dist, t_dev, "cuda")
    per_launch = t_dev / args.steps
    value = whole_job_rate(ws, case.outputs, args.steps, t_max)

    # ---- e2e through the ABI with host buffers: the steps streamed (the headline
    # e2e), and the same steps one after another on one stream (for reference)
    e2e = None
    if args.e2e_steps > 0:
        e2e_steps = args.e2e_steps
        for _ in range(2):
            case.e2e_step()
        barrier()
        f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        f0.record(st)
        for _ in range(e2e_steps):
            case.e2e_step()
        f1.record(st)
        barrier()
        t_serial = max_over_ranks(dist, f0.elapsed_time(f1) / 1e3, "cuda")
        pipe = E2EPipeline(torch, case)
        for _ in range(2):
            pipe.step()
        torch.cuda.synchronize()
        barrier()
        p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        p0.record(pipe.s_in)
        for _ in range(e2e_steps):
            pipe.step()
        pipe.s_out.wait_stream(pipe.s_in)
        pipe.s_out.wait_stream(pipe.s_op)
        p1.record(pipe.s_out)
        p1.synchronize()
        barrier()
        t_e2e = max_over_ranks(dist, p0.elapsed_time(p1) / 1e3, "cuda")
        pipe.restore()
        e2e = {"value": whole_job_rate(ws, case.outputs, e2e_steps, t_e2e), "unit": "outputs/s",
               "h2d_bytes_per_step": 4 * numel(case.host["x"].shape),
               "d2h_bytes_per_step": 4 * case.outputs, "steps": e2e_steps,
               "ms_per_step": 1e3 * t_e2e / e2e_steps,
               "how": ("steps streamed: step k+1's host->device copy overlaps step k's op and "
                       "device->host read (three streams, two device buffers each for x and y)"),
               "serial_ms_per_step": 1e3 * t_serial / e2e_steps}

    clocks = sampler.summary(t_wall0, t_wall1)
    roof = roofline_for(case, per_launch, peaks, peak_src, clocks.get("sm_mhz"))
    kernel_of = {"avgpool3d": "avgpool3d_k3s2p1_tma_kernel",
                 "ct3d_scale_pool_bias": ("ct3d_pool2_tc_chunked_kernel" if case.chunked
                                          else "ct3d_pool2_tc_kernel" if case.tc
                                          else "ct3d_pool2_fast_kernel"),
                 "convtranspose3d": "convt3d_tc_kernel" if case.tc else "convt3d_direct_kernel",
                 "convtranspose1d": ("convt1d_tiled_kernel" if case.kind == 3
                                     else "convt1d_tf32_kernel")}
    roof["kernel"] = kernel_of[case.wl.op]
    roof["algorithmic_bytes_per_launch"] = case.bytes
    hkey = case.wl.name + {None: "", 3: "", 1: "_tf32", 2: "_tf32x3"}[case.kind]
    src = PROFILE_OF.get(hkey)
    traffic = (traffic_from_profile(src[0], src[1], hkey)
               if src is not None and x_shape is None else None)
    roof["traffic"] = None if traffic == "stale" else traffic
    if traffic == "stale":
        roof["traffic_note"] = "kernel source changed since its ncu capture"

    st_code, bits = aps.binding.aps_device_status(clear=True)
    if st_code != 0 or bits != 0:
        raise RuntimeError(f"device status {st_code} bits {bits}")

    line = {
        "metric": METRIC, "value": value, "unit": "outputs/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t_max / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic", "config": line_config(case.wl, ws),
        "roofline": roof, "e2e": e2e, "gpu_launches": args.steps, "clocks": clocks,
        "fma_ceilings_tflops": {k: sig(v) for k, v in peaks["fma_measured"].items()},
        "tf32_gemm_ceiling_tflops": sig(peaks["tf32_measured"]),
    }
    headline_host = {"x": case.host["x"].numpy()} if x_shape is None else None
    headline_wl = case.wl
    del case
    torch.cuda.empty_cache()

    # ---- CPU baseline: the oracle on the host cores (rank 0, N = 1 only)
    model = cpu_model()
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        v, threads, desc, cnt, t = oracle_sample(headline_wl, args.cpu_seconds, headline_host)
        line["cpu_baseline"] = {"value": v, "unit": "outputs/s", "cores": threads,
                                "kind": "oracle", "model": model, "sample": desc,
                                "seconds": sig(t)}

    # ---- per-config breakdown (rank 0), the last key of the line
    if rank == 0 and not args.no_per_config:
        import oracle
        only = set(args.only.split(",")) if args.only else None
        want_cpu = ws == 1 and not args.no_cpu_baseline
        per = {"_cols": PER_CONFIG_COLS,
               "_peaks": {"hbm_GB_s": peaks["hbm_gbs"],
                          "fp32_TF_s": sig(fp32_peak_tflops(float(peaks.get("sm_max_mhz",
                                                                             2070.0)))),
                          "fp32_meas_TF_s": sig(peaks["fma_measured"]["packed"]),
                          "tf32_gemm_TF_s": sig(peaks["tf32_measured"])}}
        if want_cpu:
            per["_cpu"] = {"model": model, "threads": oracle.threads()}
        flush = torch.empty(64 * 1024 * 1024, device="cuda")   # 256 MB > L2
        cpu_of = {}                                               # oracle outputs/s per workload
        for key, cfg, prec, mode in PER_CONFIG:
            if only is not None and key not in only:
                continue
            c = GpuCase(cfg, torch, aps, precision=prec)
            for _ in range(3):
                c.launch()
            torch.cuda.synchronize()
            t_flushed = None
            if mode == "graph":
                t = time_graph(torch, c)
            elif mode == "rotate":
                # steady state over 4 sets of buffers launched back to back in
                # rotation (their total is well above L2); and, for the fused op,
                # one launch after a 256 MB flush
                sets = [c] + [GpuCase(cfg, torch, aps, precision=prec) for _ in range(3)]
                for o in sets[1:]:
                    o.launch()
                torch.cuda.synchronize()
                t = time_rotating(torch, sets, 40)
                if key == "fused":
                    t_flushed = time_launches(torch, c, 30, flush)
                del sets
            else:
                t = time_launches(torch, c, 20)
            if want_cpu and c.wl.name not in cpu_of:
                host = {n: h.numpy() for n, h in c.host.items()}
                cpu_of[c.wl.name] = oracle_sample(c.wl, args.cpu_seconds_per_config, host,
                                                  whole=(mode == "graph"))[0]
            e = per_config_entry(key, c, t, peaks, peak_src, cpu_of.get(c.wl.name))
            if mode == "graph":
                e[2], e[3] = None, "launch"
            if t_flushed is not None:
                per["_fused_us_after_flush"] = sig(1e6 * t_flushed)
            per[key] = e
            if want_cpu and mode == "graph":
                # the tiny workload on one host thread as well
                oracle.set_threads(1)
                try:
                    _, _, _, cnt, t1 = oracle_sample(c.wl, 0, None, whole=True)
                finally:
                    oracle.set_threads(per["_cpu"]["threads"])
                per["_cpu"][key + "_1thread_s"] = sig(t1)
                per["_cpu"][key + "_1thread_out_s"] = sig(cnt / t1, 3)
            del c
            torch.cuda.empty_cache()
        release_host()
        line["per_config"] = per
    if rank == 0:
        print(compact_json(line))
    if dist:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def main():
    args = parse_args()
    if args.impl == "reference":
        return run_reference(args)
    return run_native(args)


if __name__ == "__main__":
    sys.exit(main())
