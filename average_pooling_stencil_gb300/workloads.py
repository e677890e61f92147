"""The synthetic workloads: input shapes, value distributions, op parameters and
seeds.  Nothing here computes any part of the ops (output shapes come from the
library's shape queries on one side and from the oracle on the other).

Each workload mirrors one task traced on the Kimi-K2.6 pages:
  * ``fused_tiny`` / ``fused``  -- Kimi-K2.6__l2_p50: ConvTranspose3d(3->16, k3, s2,
    p1) with conv bias, x0.5, AvgPool3d(2), + bias[16,1,1,1], x1.0.
  * ``avgpool``                 -- Kimi-K2.6__l1_p46: AvgPool3d(k3, s2, p1),
    count_include_pad, on [16,32,128,128,256].
  * ``convt1d``                 -- Kimi-K2.6__l1_p74: ConvTranspose1d(32->64, K5,
    s1, p0, d3), no bias, on [32,32,131072].
  * ``convt1d_strided``         -- the strided variant (64->64, K4, s2, p1, op1, d2,
    with bias) that exercises per-parity tap selection.
  * ``convt3d``                 -- the first stage of l2_p50's unfused chain: its
    ConvTranspose3d(3->16, k3, s2, p1) with conv bias alone, on the fused
    workload's input, emitting the full [128,16,31,63,63] tensor.
Initialiser bounds are the usual 1/sqrt(fan) uniform ones: fan = C_out*prod(k)
for the transposed-conv weights (432 = 16*27, 320 = 64*5, 256 = 64*4).

Variants that send the same ops down their other kernels or code paths
(measured beside the workloads above):
  * ``fused_cin8`` / ``convt3d_cin8`` -- the fused op and the standalone
    ConvTranspose3d with 8 input channels (the fused op's product in channel
    chunks; the ConvTranspose3d outputs stored from registers).
  * ``fused_op1``  -- the fused op with output_padding 1 (pre-pool
    [32,64,64], pooled [16,32,32]; the last pooled position of each dim
    reads one input past the end as zero).
  * ``fused_k4``   -- the fused op with 4-tap kernels (a general geometry:
    the tiled 3x3x3 form of the general kernel).
  * ``convt3d_w64`` -- the standalone ConvTranspose3d on rows of 64 (units of
    two input rows).
  * ``fused_w30``  -- the fused op on rows of 30 floats, which are not 16-byte
    strided: no TMA box can read them, so it takes the FP32-pipe kernel with
    element copies.
  * ``avgpool_nopad`` -- the avgpool workload with count_include_pad off.
  * ``avgpool_k2``    -- AvgPool3d(k2, s2, p0), the pool of l2_p50's chain,
    alone on the avgpool workload's input (the vectorised k2 s2 kernel).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

from . import synth

STREAM_X, STREAM_W, STREAM_CONV_BIAS, STREAM_BIAS = 0, 1, 2, 3


@dataclass
class Workload:
    name: str
    op: str                      # "ct3d_scale_pool_bias" | "avgpool3d" | "convtranspose1d"
                                 # | "convtranspose3d"
    seed: int
    tensors: dict                # name -> (shape, dist, stream)
    params: dict = field(default_factory=dict)

    def generate(self, name: str, out=None, threads=None):
        shape, dist, stream = self.tensors[name]
        return synth.generate(dist, shape, self.seed, stream, out=out, threads=threads)

    def generate_range(self, name: str, start: int, stop: int):
        shape, dist, stream = self.tensors[name]
        return synth.generate_range(dist, self.seed, stream, start, stop)

    def numel(self, name: str) -> int:
        return int(math.prod(self.tensors[name][0]))

    def with_input_shape(self, shape, name: str | None = None) -> "Workload":
        """Same recipe with a different activation shape (for small parity cases)."""
        t = dict(self.tensors)
        s, d, st = t["x"]
        t["x"] = (tuple(shape), d, st)
        return Workload(name or f"{self.name}@{'x'.join(map(str, shape))}", self.op,
                        self.seed, t, dict(self.params))


def _u(b):
    return ("uniform", -b, b)


def _fused(name, xshape, seed, out_pad=(0, 0, 0), k=(3, 3, 3)):
    # U(+-1/sqrt(fan)), fan = C_out * prod(k) (432 for the pages' k = 3)
    b = 1.0 / math.sqrt(16.0 * k[0] * k[1] * k[2])
    cin = xshape[1]
    return Workload(
        name, "ct3d_scale_pool_bias", seed,
        {
            "x": (tuple(xshape), ("uniform", -1.0, 1.0), STREAM_X),
            "w": ((cin, 16) + tuple(k), _u(b), STREAM_W),
            "conv_bias": ((16,), _u(b), STREAM_CONV_BIAS),
            "bias": ((16,), ("normal", 0.02), STREAM_BIAS),
        },
        dict(c_out=16, k=tuple(k), stride=(2, 2, 2), pad=(1, 1, 1), out_pad=tuple(out_pad),
             dil=(1, 1, 1), pool_k=2, scale1=0.5, scale2=1.0),
    )


def _convt3d(name, xshape, seed):
    b = 1.0 / math.sqrt(432.0)
    return Workload(
        name, "convtranspose3d", seed,
        {
            "x": (tuple(xshape), ("uniform", -1.0, 1.0), STREAM_X),
            "w": ((xshape[1], 16, 3, 3, 3), _u(b), STREAM_W),
            "bias": ((16,), _u(b), STREAM_CONV_BIAS),
        },
        dict(c_out=16, k=(3, 3, 3), stride=(2, 2, 2), pad=(1, 1, 1), out_pad=(0, 0, 0),
             dil=(1, 1, 1), has_bias=True),
    )


def _avgpool(name, k, s, p, cip):
    return Workload(
        name, "avgpool3d", 1,
        {"x": ((16, 32, 128, 128, 256), ("normal", 1.0), STREAM_X)},
        dict(k=k, stride=s, pad=p, count_include_pad=cip, ceil_mode=0),
    )


WORKLOADS = {
    0: _fused("fused_tiny", (2, 3, 8, 16, 16), 0),
    1: _avgpool("avgpool", (3, 3, 3), (2, 2, 2), (1, 1, 1), 1),
    2: _fused("fused", (128, 3, 16, 32, 32), 2),
    3: Workload(
        "convt1d", "convtranspose1d", 3,
        {
            "x": ((32, 32, 131072), ("normal", 1.0), STREAM_X),
            "w": ((32, 64, 5), _u(1.0 / math.sqrt(320.0)), STREAM_W),
        },
        dict(c_out=64, k=5, stride=1, pad=0, dil=3, out_pad=0, has_bias=False),
    ),
    4: Workload(
        "convt1d_strided", "convtranspose1d", 4,
        {
            "x": ((16, 64, 65536), ("normal", 1.0), STREAM_X),
            "w": ((64, 64, 4), _u(1.0 / 16.0), STREAM_W),
            "bias": ((64,), _u(1.0 / 16.0), STREAM_BIAS),
        },
        dict(c_out=64, k=4, stride=2, pad=1, dil=2, out_pad=1, has_bias=True),
    ),
    5: _convt3d("convt3d", (128, 3, 16, 32, 32), 5),
    6: _fused("fused_cin8", (128, 8, 16, 32, 32), 6),
    7: _fused("fused_op1", (128, 3, 16, 32, 32), 7, out_pad=(1, 1, 1)),
    8: _avgpool("avgpool_nopad", (3, 3, 3), (2, 2, 2), (1, 1, 1), 0),
    9: _avgpool("avgpool_k2", (2, 2, 2), (2, 2, 2), (0, 0, 0), 1),
    10: _convt3d("convt3d_cin8", (128, 8, 16, 32, 32), 10),
    11: _fused("fused_k4", (128, 3, 16, 32, 32), 11, k=(4, 4, 4)),
    12: _convt3d("convt3d_w64", (64, 3, 16, 32, 64), 12),
    13: _fused("fused_w30", (128, 3, 16, 32, 30), 13),
}


def get(cfg) -> Workload:
    if isinstance(cfg, str):
        for w in WORKLOADS.values():
            if w.name == cfg:
                return w
        raise KeyError(cfg)
    return WORKLOADS[int(cfg)]
