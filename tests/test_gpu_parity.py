"""CUDA path (through the C ABI) against the fp64 oracle, element by element.

Tolerance (fp32 FMA kernels): |gpu - oracle| <= 1e-5 * (1 + |oracle|) for every
output, output shapes exact.  Small cases span several tiles and ragged tails
and cover every kernel variant; the full-size workloads are compared on sampled
(n, c) planes, which the oracle computes one by one.
"""
import numpy as np
import pytest

import __graft_entry__
import oracle as ora

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from average_pooling_stencil_gb300 import binding as B  # noqa: E402
from average_pooling_stencil_gb300 import workloads  # noqa: E402

TOL = 1e-5


@pytest.fixture(scope="module", autouse=True)
def built():
    __graft_entry__.build()
    assert torch.cuda.is_available()
    torch.cuda.set_device(0)
    B.aps_device_status(clear=True)
    yield
    st, bits = B.aps_device_status(clear=True)
    assert st == 0 and bits == 0, f"device status word {bits}"


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def assert_close(got, want, tol=TOL, what=""):
    got = np.asarray(got, dtype=np.float64)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    assert np.isfinite(got).all(), what
    err = np.abs(got - want)
    bound = tol * (1.0 + np.abs(want))
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err / bound), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())}/{err.size} outputs off; worst at {i}: "
                             f"gpu {got[i]!r} oracle {want[i]!r}")


def rng_inputs(seed, *shapes, lo=-1.0, hi=1.0):
    r = np.random.default_rng(seed)
    return [r.uniform(lo, hi, s).astype(np.float32) for s in shapes]


# ------------------------------------------------------------------ avgpool3d
FAST_POOL_SHAPES = [(2, 3, 9, 20, 68), (1, 2, 4, 17, 132), (1, 1, 2, 2, 4), (3, 2, 7, 5, 8),
                    (1, 1, 1, 1, 4), (2, 1, 3, 33, 260), (1, 3, 6, 16, 256)]


@pytest.mark.parametrize("cip", [1, 0])
@pytest.mark.parametrize("shape", FAST_POOL_SHAPES)
def test_avgpool_k3s2p1_tma_path(shape, cip):
    """The TMA kernel, count_include_pad on (divisor 27) and off (divisor = cells in
    range: odd extents also clip the last window at the high end)."""
    x = workloads.get(1).with_input_shape(shape).generate("x")
    y = B.avgpool3d(dev(x), 3, 2, 1, bool(cip))
    assert_close(y.cpu().numpy(), ora.avgpool3d(x, 3, 2, 1, cip, 0),
                 what=f"avgpool {shape} cip {cip}")


@pytest.mark.parametrize("shape", [(2, 3, 9, 20, 67), (1, 1, 5, 6, 7), (1, 2, 3, 3, 2)])
def test_avgpool_k3s2p1_direct_path(shape):
    x, = rng_inputs(1, shape)
    y = B.avgpool3d(dev(x), 3, 2, 1)
    assert_close(y.cpu().numpy(), ora.avgpool3d(x, 3, 2, 1, 1, 0), what=f"avgpool {shape}")


def test_avgpool_unaligned_input_takes_direct_path():
    x, = rng_inputs(2, (1 * 2 * 5 * 6 * 8 + 1,))
    xt = dev(x)[1:].view(1, 2, 5, 6, 8)
    assert xt.data_ptr() % 16 != 0
    y = B.avgpool3d(xt, 3, 2, 1)
    ref = ora.avgpool3d(x[1:].reshape(1, 2, 5, 6, 8), 3, 2, 1, 1, 0)
    assert_close(y.cpu().numpy(), ref, what="unaligned avgpool")


@pytest.mark.parametrize("k,s,p,cip,ceil", [
    ((2, 3, 4), (1, 2, 3), (1, 1, 2), 1, 0), ((3, 3, 3), (2, 2, 2), (1, 1, 1), 0, 0),
    ((3, 3, 3), (2, 2, 2), (1, 1, 1), 1, 1), ((3, 3, 3), (2, 2, 2), (1, 1, 1), 0, 1),
    ((5, 2, 3), (3, 2, 1), (2, 0, 1), 0, 1), ((1, 1, 1), (1, 1, 1), (0, 0, 0), 1, 0),
    # cubic windows of 2 and 3 take the unrolled-window kernel
    ((2, 2, 2), (2, 2, 2), (0, 0, 0), 1, 0), ((2, 2, 2), (1, 2, 3), (1, 1, 0), 0, 1),
    ((2, 2, 2), (3, 1, 2), (1, 0, 1), 1, 1), ((3, 3, 3), (1, 3, 2), (0, 1, 1), 1, 0)])
def test_avgpool_general_windows(k, s, p, cip, ceil):
    x, = rng_inputs(3, (2, 2, 7, 9, 10))
    y = B.avgpool3d(dev(x), k, s, p, bool(cip), bool(ceil))
    assert_close(y.cpu().numpy(), ora.avgpool3d(x, k, s, p, cip, ceil),
                 what=f"avgpool {k} {s} {p} {cip} {ceil}")


# k2 s2 p0 with whole windows and 16-byte rows: the vectorised pair kernel (odd D and H
# leave their last plane and row unused; rows of 4 give one pair per row); and the same
# with rows of 10 (not 16-byte), which takes the unrolled-window kernel
@pytest.mark.parametrize("shape", [(2, 3, 6, 8, 16), (1, 2, 7, 9, 20), (3, 1, 2, 2, 4),
                                   (1, 2, 5, 6, 10)])
def test_avgpool_k2s2_pairs(shape):
    x, = rng_inputs(4, shape)
    for cip in (1, 0):
        y = B.avgpool3d(dev(x), 2, 2, 0, bool(cip))
        assert_close(y.cpu().numpy(), ora.avgpool3d(x, 2, 2, 0, cip, 0), what=f"avgpool k2 {shape}")


def test_avgpool_repeatable_bitwise():
    x = dev(workloads.get(1).with_input_shape((2, 4, 10, 34, 132)).generate("x"))
    a = B.avgpool3d(x, 3, 2, 1)
    b = B.avgpool3d(x, 3, 2, 1)
    assert torch.equal(a, b)


_FULL_POOL_X = {}


# the avgpool workload (cfg 1), the same input with count_include_pad off (cfg 8) and
# AvgPool3d(k2, s2) on it (cfg 9, the general kernel), as the bench launches them
@pytest.mark.slow
@pytest.mark.parametrize("cfg", [1, 8, 9])
def test_avgpool_full_workload_sampled_planes(cfg):
    wl = workloads.get(cfg)
    p = wl.params
    if "x" not in _FULL_POOL_X:
        _FULL_POOL_X["x"] = wl.generate("x")               # [16,32,128,128,256], 8.6 GB
    x = _FULL_POOL_X["x"]
    xd = dev(x)
    y = B.avgpool3d(xd, p["k"], p["stride"], p["pad"], bool(p["count_include_pad"]))
    torch.cuda.synchronize()
    sel = [(0, 0), (0, 31), (7, 13), (15, 0), (15, 31), (9, 22)]
    ref = ora.avgpool3d(x, p["k"], p["stride"], p["pad"], p["count_include_pad"], 0, sel=sel)
    got = np.stack([y[n, c].cpu().numpy() for n, c in sel])
    assert_close(got, ref, what=f"avgpool full workload cfg {cfg}")
    assert torch.isfinite(y).all()
    del xd, y
    torch.cuda.empty_cache()
    if cfg == 9:
        _FULL_POOL_X.clear()


# ------------------------------------------------------- ct3d_scale_pool_bias
def fused_ref(wl, x, w, cb, b, **over):
    p = dict(wl.params, **over)
    return ora.ct3d_scale_pool_bias(x, w, cb, b, p["stride"], p["pad"], p["out_pad"], p["dil"],
                                    p["pool_k"], p["scale1"], p["scale2"])


def fused_gpu(x, w, cb, b, p):
    return B.ct3d_scale_pool_bias(dev(x), dev(w), None if cb is None else dev(cb), dev(b),
                                  p["stride"], p["pad"], p["out_pad"], p["dil"], p["pool_k"],
                                  p["scale1"], p["scale2"]).cpu().numpy()


# the tiny and full workloads, and the full one with 8 input channels (cfg 6, the
# tensor-core kernel in channel chunks), with output_padding 1 (cfg 7), with 4-tap kernels
# (cfg 11, the general kernel) and on rows of 30 floats (cfg 13, the FP32-pipe kernel)
@pytest.mark.parametrize("cfg", [0, 2, 6, 7, 11, 13])
def test_fused_workloads_all_outputs(cfg):
    wl = workloads.get(cfg)
    x, w, cb, b = (wl.generate(n) for n in ("x", "w", "conv_bias", "bias"))
    assert_close(fused_gpu(x, w, cb, b, wl.params), fused_ref(wl, x, w, cb, b),
                 what=f"fused cfg {cfg}")


# C_in <= 3 with W % 4 == 0 runs on the tensor cores (C_in 1, 2, 3; staged rows of 32
# columns or a run-time width; Ho = 32 exactly; several row and column blocks); the rest on
# the FP32 pipe (C_in 4..8, rows that are not 16-byte strided)
@pytest.mark.parametrize("shape", [(1, 3, 5, 7, 9), (2, 1, 2, 2, 2), (3, 8, 4, 6, 33),
                                   (1, 2, 3, 40, 40), (2, 3, 4, 8, 32), (1, 5, 2, 3, 1030),
                                   (1, 3, 3, 70, 20), (2, 1, 3, 9, 12), (1, 2, 5, 33, 8),
                                   (1, 1, 2, 2, 4), (3, 3, 2, 17, 68)])
def test_fused_fast_path_shapes(shape):
    base = workloads.get(0)
    wl = workloads.Workload(base.name, base.op, 5, dict(base.tensors), dict(base.params))
    wl.tensors["x"] = (shape, ("uniform", -1.0, 1.0), 0)
    wl.tensors["w"] = ((shape[1], 16, 3, 3, 3), base.tensors["w"][1], 1)
    x, w, cb, b = (wl.generate(n) for n in ("x", "w", "conv_bias", "bias"))
    assert_close(fused_gpu(x, w, cb, b, wl.params), fused_ref(wl, x, w, cb, b),
                 what=f"fused {shape}")


# output_padding 1 in some dims keeps the fast path: the extra pooled position of such a
# dim reads input offset 1 past the end of x, which the TMA box (tensor cores, FP32 pipe)
# or the element copies (rows that are not 16-byte strided) fill with zeros.  Whole rows of
# 32 (a 36-column staged window), several row and column blocks, C_in 1..8
@pytest.mark.parametrize("shape,op", [
    ((2, 3, 4, 8, 32), (1, 1, 1)), ((1, 2, 3, 9, 12), (0, 1, 1)), ((2, 3, 5, 7, 8), (1, 0, 0)),
    ((1, 1, 3, 40, 40), (0, 0, 1)), ((1, 3, 2, 33, 36), (1, 1, 0)), ((1, 5, 3, 6, 20), (1, 1, 0)),
    ((1, 4, 3, 5, 7), (1, 1, 1)), ((2, 8, 2, 9, 33), (0, 1, 1)), ((1, 3, 2, 2, 4), (1, 1, 1))])
def test_fused_fast_path_with_output_padding(shape, op):
    x, = rng_inputs(47, shape)
    w, cb, b = rng_inputs(48, (shape[1], 16, 3, 3, 3), (16,), (16,), lo=-0.2, hi=0.2)
    one = (1, 1, 1)
    prm = dict(stride=(2, 2, 2), pad=one, out_pad=op, dil=one, pool_k=2, scale1=0.5, scale2=1.25)
    ref = ora.ct3d_scale_pool_bias(x, w, cb, b, (2, 2, 2), one, op, one, 2, 0.5, 1.25)
    assert ref.shape[2:] == tuple(shape[2 + i] - 1 + op[i] for i in range(3))
    assert_close(fused_gpu(x, w, cb, b, prm), ref, what=f"fused op {op} {shape}")


def test_fused_unaligned_input_takes_the_fp32_kernel():
    """An input that is not 16-byte aligned cannot be a TMA source: the op then runs the
    FP32-pipe kernel with element copies, on the same shape the tensor cores take."""
    base = workloads.get(0)
    x, = rng_inputs(41, (2, 3, 4, 8, 32))
    w, cb, b = (base.generate(n) for n in ("w", "conv_bias", "bias"))
    store = torch.empty(x.size + 1, device="cuda", dtype=torch.float32)
    xd = store[1:].view(x.shape)
    xd.copy_(dev(x))
    assert xd.data_ptr() % 16 != 0
    y = B.ct3d_scale_pool_bias(xd, dev(w), dev(cb), dev(b), scale1=base.params["scale1"],
                               scale2=base.params["scale2"])
    assert_close(y.cpu().numpy(), fused_ref(base, x, w, cb, b), what="fused unaligned x")


class skip_tensor_cores:
    """Within the block every op passes over its tensor-core kernels (the library's test
    hook), so that its FP32-pipe fallbacks run on shapes the tensor cores take."""

    def __enter__(self):
        B.aps_debug_skip_tensor_cores(True)

    def __exit__(self, *exc):
        B.aps_debug_skip_tensor_cores(False)


FUSED_FAST = dict(stride=(2, 2, 2), pad=(1, 1, 1), out_pad=(0, 0, 0), dil=(1, 1, 1), pool_k=2,
                  scale1=0.5, scale2=1.0)


def fused_fast_ref(x, w, cb, b, op=(0, 0, 0)):
    return ora.ct3d_scale_pool_bias(x, w, cb, b, (2, 2, 2), (1, 1, 1), op, (1, 1, 1), 2, 0.5, 1.0)


# many small units: every CTA of the FP32-pipe kernel's persistent grid takes several, so
# its double-buffered input ring goes round (and its barrier phases flip) many times; W = 4
# stages the input by TMA (the tensor cores passed over), W = 5 by element copies
@pytest.mark.parametrize("shape", [(80, 5, 33, 3, 4), (80, 4, 33, 3, 5)])
def test_fused_fp32_kernel_many_units_per_cta(shape):
    x, = rng_inputs(45, shape)
    w, cb, b = rng_inputs(46, (shape[1], 16, 3, 3, 3), (16,), (16,), lo=-0.2, hi=0.2)
    with skip_tensor_cores():
        got = fused_gpu(x, w, cb, b, FUSED_FAST)
    assert_close(got, fused_fast_ref(x, w, cb, b), what=f"fused fp32 many units {shape}")


# the FP32-pipe kernel on shapes the tensor cores take (16-byte rows): C_in 1..8, whole
# rows of 32 and a 36-column window, ragged row blocks, output padding
@pytest.mark.parametrize("shape,op", [((2, 3, 4, 8, 32), (0, 0, 0)), ((1, 8, 3, 33, 36), (1, 1, 0)),
                                      ((2, 1, 3, 9, 12), (0, 1, 1)), ((1, 6, 5, 6, 20), (1, 0, 1))])
def test_fused_fp32_fallback_on_tensor_core_shapes(shape, op):
    x, = rng_inputs(49, shape)
    w, cb, b = rng_inputs(50, (shape[1], 16, 3, 3, 3), (16,), (16,), lo=-0.2, hi=0.2)
    with skip_tensor_cores():
        got = fused_gpu(x, w, cb, b, dict(FUSED_FAST, out_pad=op))
    assert_close(got, fused_fast_ref(x, w, cb, b, op), what=f"fused fp32 fallback {shape} op {op}")


# C_in 4..8 on the tensor cores: each tile's product in chunks of <= 3 channels through two
# alternating A slots (2 chunks for C_in 4..6, 3 for 7..8).  Whole rows of 32 (3 stages at
# C_in 8), a 36-column window in two column blocks, ragged row blocks, output padding, and
# many units per CTA (the stage ring and the slot barriers go round many times)
@pytest.mark.parametrize("shape,op", [
    ((3, 4, 5, 9, 12), (0, 0, 0)), ((2, 5, 4, 40, 36), (0, 0, 0)), ((1, 7, 3, 33, 64), (1, 1, 1)),
    ((2, 8, 6, 32, 32), (0, 0, 0)), ((2, 8, 3, 9, 32), (1, 1, 1)), ((1, 6, 2, 17, 8), (0, 1, 0)),
    ((160, 8, 9, 3, 4), (0, 0, 0)), ((96, 5, 9, 3, 8), (1, 0, 1)),
    # 33 staged rows of 36 columns at C_in 8: a 76 KB stage, so the ring holds two
    ((1, 8, 2, 33, 36), (0, 0, 0)), ((2, 8, 3, 34, 36), (1, 0, 1))])
def test_fused_tensor_core_chunked_channels(shape, op):
    x, = rng_inputs(51, shape)
    w, cb, b = rng_inputs(52, (shape[1], 16, 3, 3, 3), (16,), (16,), lo=-0.2, hi=0.2)
    got = fused_gpu(x, w, cb, b, dict(FUSED_FAST, out_pad=op))
    assert_close(got, fused_fast_ref(x, w, cb, b, op), what=f"fused chunked {shape} op {op}")


def test_fused_without_conv_bias_and_other_scales():
    wl = workloads.get(0)
    x, w, b = (wl.generate(n) for n in ("x", "w", "bias"))
    p = dict(wl.params, scale1=1.75, scale2=-0.3)
    assert_close(fused_gpu(x, w, None, b, p), fused_ref(wl, x, w, None, b, scale1=1.75, scale2=-0.3),
                 what="fused no conv bias")


@pytest.mark.parametrize("cout,k,s,p,op,d,q", [
    (5, (3, 2, 4), (1, 2, 3), (0, 1, 1), (0, 1, 2), (1, 2, 1), 3),
    (16, (3, 3, 3), (2, 2, 2), (1, 1, 1), (0, 0, 0), (1, 1, 1), 3),
    (16, (3, 3, 3), (2, 2, 2), (1, 1, 1), (1, 1, 1), (1, 1, 1), 2),
    (12, (3, 3, 3), (2, 2, 2), (1, 1, 1), (0, 0, 0), (1, 1, 1), 2),
    (4, (2, 2, 2), (2, 2, 2), (0, 0, 0), (0, 0, 0), (1, 1, 1), 1)])
def test_fused_general_geometry(cout, k, s, p, op, d, q):
    x, = rng_inputs(7, (2, 3, 4, 5, 6))
    w, cb, b = rng_inputs(8, (3, cout) + k, (cout,), (cout,), lo=-0.2, hi=0.2)
    prm = dict(stride=s, pad=p, out_pad=op, dil=d, pool_k=q, scale1=0.5, scale2=1.5)
    ref = ora.ct3d_scale_pool_bias(x, w, cb, b, s, p, op, d, q, 0.5, 1.5)
    assert_close(fused_gpu(x, w, cb, b, prm), ref, what=f"fused general {k} {s} {p} {op} {d} {q}")


# the general kernel's per-dim phase tables: pool sizes that are not multiples of the
# stride (3 and 2 phases per dim), stride 4 with pool 1 (two of the four phases reached
# by no tap: bias only), several 16-channel output blocks with a ragged last one; and,
# past the tables' limits (9 input offsets per phase with dilation 3; 9 phases), the
# per-output direct kernel
@pytest.mark.parametrize("xs,cout,k,s,p,op,d,q", [
    ((2, 5, 5, 7, 41), 20, (3, 3, 4), (3, 2, 4), (1, 0, 2), (0, 1, 3), (1, 1, 1), 2),
    ((3, 3, 4, 6, 33), 33, (3, 3, 3), (2, 2, 2), (1, 1, 1), (1, 1, 1), (1, 1, 1), 2),
    ((1, 2, 3, 4, 37), 6, (2, 2, 2), (1, 1, 4), (0, 0, 1), (0, 0, 0), (1, 1, 1), 1),
    ((1, 2, 6, 5, 9), 7, (2, 3, 3), (2, 1, 3), (0, 2, 1), (1, 0, 2), (2, 3, 1), 3),
    ((1, 2, 3, 4, 5), 6, (2, 2, 3), (1, 1, 9), (0, 0, 1), (0, 0, 0), (1, 1, 1), 1),
    # at most 3 input offsets per phase in every dim: the unrolled 3 x 3 x 3 cells (4-tap
    # kernels, a 4-tap dim beside 3-tap ones, 5 taps with padding 2, dilation 2), and one
    # with 4 offsets in a dim (run-time loops)
    ((2, 3, 5, 6, 7), 16, (4, 4, 4), (2, 2, 2), (1, 1, 1), (0, 0, 0), (1, 1, 1), 2),
    ((1, 2, 4, 5, 9), 20, (3, 4, 3), (2, 2, 2), (1, 1, 1), (1, 0, 1), (1, 1, 1), 2),
    ((1, 3, 3, 7, 10), 7, (5, 5, 3), (2, 2, 2), (2, 2, 1), (0, 0, 0), (1, 1, 1), 2),
    ((2, 2, 4, 6, 8), 16, (3, 3, 3), (2, 2, 2), (1, 1, 1), (0, 0, 0), (2, 1, 1), 2),
    ((1, 2, 4, 5, 6), 9, (4, 4, 2), (2, 2, 1), (1, 2, 0), (0, 1, 0), (1, 1, 1), 3),
    # one phase per dim, pool = stride, 3 offsets in some dim, 16-byte rows: the tiled
    # 3 x 3 x 3 kernel (a TMA box whose x origin is rounded down to 4; two and a ragged
    # output-channel block; several row and column blocks; 8 input channels; a plain
    # stride-1 3 x 3 x 3 convolution with pool 1)
    ((2, 3, 5, 6, 8), 16, (4, 4, 4), (2, 2, 2), (1, 1, 1), (0, 0, 0), (1, 1, 1), 2),
    ((1, 2, 4, 5, 36), 20, (3, 4, 3), (2, 2, 2), (1, 1, 1), (1, 0, 1), (1, 1, 1), 2),
    ((1, 3, 3, 7, 40), 7, (5, 5, 3), (2, 2, 2), (2, 2, 1), (0, 0, 0), (1, 1, 1), 2),
    ((2, 4, 3, 18, 68), 16, (3, 3, 3), (1, 1, 1), (1, 1, 1), (0, 0, 0), (1, 1, 1), 1),
    ((1, 8, 2, 3, 4), 16, (4, 4, 4), (2, 2, 2), (1, 1, 1), (1, 1, 1), (1, 1, 1), 2)])
def test_fused_general_geometry_tables(xs, cout, k, s, p, op, d, q):
    x, = rng_inputs(9, xs)
    w, cb, b = rng_inputs(10, (xs[1], cout) + k, (cout,), (cout,), lo=-0.2, hi=0.2)
    prm = dict(stride=s, pad=p, out_pad=op, dil=d, pool_k=q, scale1=0.75, scale2=-1.25)
    ref = ora.ct3d_scale_pool_bias(x, w, cb, b, s, p, op, d, q, 0.75, -1.25)
    assert_close(fused_gpu(x, w, cb, b, prm), ref,
                 what=f"fused general {xs} {k} {s} {p} {op} {d} {q}")


# ------------------------------------------------------------ convtranspose3d
CONVT3D_CASES = [  # (x shape, C_out, k, s, p, d, op, bias)
    # W > 32: units of 2 rows of up to 64 columns or 1 row of up to 128 (C_in <= 3: staged
    # runs; C_in 4..8: outputs from registers), and 128-column blocks of wider rows
    # (outputs from registers; the last block partial); output padding
    ((1, 3, 4, 19, 36), 16, (3, 3, 3), (2, 2, 2), (1, 1, 1), (1, 1, 1), (0, 0, 0), True),
    ((1, 8, 3, 9, 40), 16, (3, 3, 3), (2, 2, 2), (1, 1, 1), (1, 1, 1), (1, 1, 1), False),
    ((1, 5, 2, 7, 36), 16, (3, 3, 3), (2, 2, 2), (1, 1, 1), (1, 1, 1), (0, 1, 0), True),
    ((1, 3, 2, 2, 68), 16, (3, 3, 3), (2, 2, 2), (1, 1, 1), (1, 1, 1), (1, 0, 1), True),
    ((2, 2, 3, 5, 64), 16, (3, 3, 3), (2, 2, 2), (1, 1, 1), (1, 1, 1), (0, 0, 0), True),
    ((1, 1, 2, 3, 128), 16, (3, 3, 3), (2, 2, 2), (1, 1, 1), (1, 1, 1), (1, 1, 1), True),
    ((1, 3, 2, 4, 100), 16, (3, 3, 3), (2, 2, 2), (1, 1, 1), (1, 1, 1), (0, 1, 1), False),
    ((1, 3, 2, 3, 260), 16, (3, 3, 3), (2, 2, 2), (1, 1, 1), (1, 1, 1), (0, 0, 1), True),
    ((1, 8, 2, 2, 136), 16, (3, 3, 3), (2, 2, 2), (1, 1, 1), (1, 1, 1), (1, 0, 0), True),
    # W <= 32: the tensor-core kernel, C_in 1..3 with staged output runs and C_in 4..8
    # with outputs from registers (output padding in every dim, H not a multiple of 4, a
    # single input plane, no bias)
    ((2, 3, 5, 9, 12), 16, (3, 3, 3), (2, 2, 2), (1, 1, 1), (1, 1, 1), (0, 0, 0), True),
    ((2, 8, 3, 17, 8), 16, (3, 3, 3), (2, 2, 2), (1, 1, 1), (1, 1, 1), (1, 1, 1), False),
    ((1, 1, 6, 6, 4), 16, (3, 3, 3), (2, 2, 2), (1, 1, 1), (1, 1, 1), (0, 1, 0), True),
    ((1, 5, 3, 6, 32), 16, (3, 3, 3), (2, 2, 2), (1, 1, 1), (1, 1, 1), (0, 0, 1), True),
    ((2, 4, 4, 9, 20), 16, (3, 3, 3), (2, 2, 2), (1, 1, 1), (1, 1, 1), (1, 0, 0), True),
    ((1, 7, 2, 5, 12), 16, (3, 3, 3), (2, 2, 2), (1, 1, 1), (1, 1, 1), (0, 0, 0), False),
    ((3, 2, 3, 9, 16), 16, (3, 3, 3), (2, 2, 2), (1, 1, 1), (1, 1, 1), (1, 1, 1), True),
    ((1, 3, 1, 7, 32), 16, (3, 3, 3), (2, 2, 2), (1, 1, 1), (1, 1, 1), (0, 0, 0), False),
    ((2, 1, 4, 4, 28), 16, (3, 3, 3), (2, 2, 2), (1, 1, 1), (1, 1, 1), (1, 0, 1), True),
    # W % 4 != 0 (no TMA) and other geometries: the direct kernel
    ((2, 3, 4, 5, 10), 16, (3, 3, 3), (2, 2, 2), (1, 1, 1), (1, 1, 1), (0, 0, 0), True),
    ((1, 2, 3, 4, 5), 5, (2, 3, 4), (1, 2, 3), (0, 1, 2), (2, 1, 1), (1, 1, 2), True),
    ((2, 4, 3, 3, 3), 7, (1, 1, 1), (1, 1, 1), (0, 0, 0), (1, 1, 1), (0, 0, 0), False),
    ((1, 3, 5, 4, 4), 16, (3, 3, 3), (2, 2, 2), (1, 1, 1), (2, 2, 2), (1, 1, 1), True),
]


@pytest.mark.parametrize("xs,cout,k,s,p,d,op,has_bias", CONVT3D_CASES)
def test_convt3d_cases(xs, cout, k, s, p, d, op, has_bias):
    x, = rng_inputs(31, xs)
    w, b = rng_inputs(32, (xs[1], cout) + tuple(k), (cout,), lo=-0.3, hi=0.3)
    b = b if has_bias else None
    y = B.convtranspose3d(dev(x), dev(w), None if b is None else dev(b), s, p, d, op)
    assert_close(y.cpu().numpy(), ora.convt(x, w, b, s, p, d, op),
                 what=f"convt3d {xs} k{k} s{s} p{p} d{d} op{op}")


# ~1500 units, several per CTA of the persistent grid, so the input ring wraps many
# times: C_in 8 at W 4 (outputs from registers), C_in 3 and 8 at W 36 (units of 2 rows of
# up to 64 columns; staged runs for C_in 3)
@pytest.mark.parametrize("xs", [(48, 8, 16, 3, 4), (24, 3, 16, 3, 36), (12, 8, 16, 3, 36)])
def test_convt3d_many_units_per_cta(xs):
    x, = rng_inputs(47, xs)
    w, b = rng_inputs(48, (xs[1], 16, 3, 3, 3), (16,), lo=-0.3, hi=0.3)
    args = ((2, 2, 2), (1, 1, 1), (1, 1, 1), (0, 0, 0))
    y = B.convtranspose3d(dev(x), dev(w), dev(b), *args)
    assert_close(y.cpu().numpy(), ora.convt(x, w, b, *args), what=f"convt3d many units {xs}")


# a seeded sweep over the fast path's shapes: C_in 1..8, ragged sizes, 16-byte rows or not,
# output padding per dim (every kernel of the fast path, with its ring and block counts)
def _fused_sweep(n, seed=20261202):
    r = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        cin = int(r.integers(1, 9))
        w = int(r.choice([4, 8, 12, 20, 28, 32, 36, 44, 64, 13, 30]))
        out.append(((int(r.integers(1, 4)), cin, int(r.integers(2, 7)), int(r.integers(2, 40)), w),
                    tuple(int(v) for v in r.integers(0, 2, 3))))
    return out


@pytest.mark.parametrize("shape,op", _fused_sweep(16))
def test_fused_fast_path_seeded_sweep(shape, op):
    x, = rng_inputs(57, shape)
    w, cb, b = rng_inputs(58, (shape[1], 16, 3, 3, 3), (16,), (16,), lo=-0.2, hi=0.2)
    got = fused_gpu(x, w, cb, b, dict(FUSED_FAST, out_pad=op))
    assert_close(got, fused_fast_ref(x, w, cb, b, op), what=f"fused sweep {shape} op {op}")


# a seeded sweep over the ConvTranspose3d fast path: C_in 1..8 (the ring depth the staging
# leaves), widths for units of 4 / 2 / 1 rows and 128-column blocks, 16-byte rows or not
def _convt3d_sweep(n, seed=20261203):
    r = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        w = int(r.choice([4, 12, 28, 32, 36, 60, 64, 100, 128, 132, 30, 66]))
        out.append(((int(r.integers(1, 3)), int(r.integers(1, 9)), int(r.integers(1, 5)),
                     int(r.integers(1, 12)), w), tuple(int(v) for v in r.integers(0, 2, 3))))
    return out


@pytest.mark.parametrize("xs,op", _convt3d_sweep(12))
def test_convt3d_fast_path_seeded_sweep(xs, op):
    x, = rng_inputs(59, xs)
    w, b = rng_inputs(60, (xs[1], 16, 3, 3, 3), (16,), lo=-0.3, hi=0.3)
    args = ((2, 2, 2), (1, 1, 1), (1, 1, 1), op)
    y = B.convtranspose3d(dev(x), dev(w), dev(b), *args)
    assert_close(y.cpu().numpy(), ora.convt(x, w, b, *args), what=f"convt3d sweep {xs} op {op}")


# the direct kernel on shapes the tensor cores take (the tensor cores passed over)
@pytest.mark.parametrize("xs,op", [((2, 3, 3, 8, 16), (0, 0, 0)), ((1, 8, 2, 5, 36), (1, 1, 1))])
def test_convt3d_direct_fallback_on_tensor_core_shapes(xs, op):
    x, = rng_inputs(53, xs)
    w, b = rng_inputs(54, (xs[1], 16, 3, 3, 3), (16,), lo=-0.3, hi=0.3)
    args = ((2, 2, 2), (1, 1, 1), (1, 1, 1), op)
    with skip_tensor_cores():
        y = B.convtranspose3d(dev(x), dev(w), dev(b), *args)
    assert_close(y.cpu().numpy(), ora.convt(x, w, b, *args), what=f"convt3d direct fallback {xs}")


def test_convt3d_unaligned_input_takes_the_direct_kernel():
    """An input that is not 16-byte aligned cannot be a TMA source: the op then runs
    the direct kernel, on a shape the tensor cores take when aligned."""
    xs = (2, 3, 3, 8, 16)
    x, = rng_inputs(43, xs)
    w, b = rng_inputs(44, (3, 16, 3, 3, 3), (16,), lo=-0.3, hi=0.3)
    store = torch.empty(x.size + 1, device="cuda", dtype=torch.float32)
    xd = store[1:].view(x.shape)
    xd.copy_(dev(x))
    assert xd.data_ptr() % 16 != 0
    y = B.convtranspose3d(xd, dev(w), dev(b), (2, 2, 2), (1, 1, 1), (1, 1, 1), (0, 0, 0))
    assert_close(y.cpu().numpy(), ora.convt(x, w, b, (2, 2, 2), (1, 1, 1), (1, 1, 1), (0, 0, 0)),
                 what="convt3d unaligned x")


@pytest.mark.parametrize("cfg", [5, 10, 12])
def test_convt3d_full_workload_sampled_planes(cfg):
    wl = workloads.get(cfg)
    p = wl.params
    x, w, b = wl.generate("x"), wl.generate("w"), wl.generate("bias")
    y = B.convtranspose3d(dev(x), dev(w), dev(b), p["stride"], p["pad"], p["dil"], p["out_pad"])
    torch.cuda.synchronize()
    N, C = y.shape[0], y.shape[1]
    sel = [(0, 0), (N - 1, C - 1), (N // 2, 7), (5, 12)]
    ref = ora.convt(x, w, b, p["stride"], p["pad"], p["dil"], p["out_pad"], sel=sel)
    got = np.stack([y[n, c].cpu().numpy() for n, c in sel])
    assert_close(got, ref, what=f"convt3d full workload cfg {cfg}")
    assert torch.isfinite(y).all()


# ------------------------------------------------------------ back-to-back ops
def test_an_op_sees_what_the_kernel_before_it_wrote():
    """The convolution kernels are launched as programmatic dependents of the
    kernel before them on the stream.  A direct ConvTranspose3d writes x1 and the
    fused tensor-core kernel reads it at once, with no synchronisation between."""
    x0, = rng_inputs(51, (4, 3, 9, 33, 64))
    w0, = rng_inputs(52, (3, 3, 1, 1, 1), lo=-0.8, hi=0.8)
    w, cb, b = rng_inputs(53, (3, 16, 3, 3, 3), (16,), (16,), lo=-0.2, hi=0.2)
    one, zero = (1, 1, 1), (0, 0, 0)
    x1 = B.convtranspose3d(dev(x0), dev(w0), None, one, zero, one, zero)
    y = B.ct3d_scale_pool_bias(x1, dev(w), dev(cb), dev(b), scale1=0.5, scale2=1.0)
    torch.cuda.synchronize()
    x1h = x1.cpu().numpy()
    assert_close(x1h, ora.convt(x0, w0, None, one, zero, one, zero), what="producer")
    ref = ora.ct3d_scale_pool_bias(x1h, w, cb, b, (2, 2, 2), (1, 1, 1), zero, one, 2, 0.5, 1.0)
    assert_close(y.cpu().numpy(), ref, what="consumer of the previous kernel's output")


def test_an_op_does_not_overwrite_what_the_kernel_before_it_reads():
    """A ConvTranspose1d reads x; the next op on the stream writes its output over
    x.  The first must still see the original x everywhere."""
    x, = rng_inputs(54, (4, 32, 65536))
    w, = rng_inputs(55, (32, 64, 5), lo=-0.06, hi=0.06)
    z, w2 = rng_inputs(56, (4, 64, 65532), (64, 32, 5), lo=-0.5, hi=0.5)
    xd, zd, w2d = dev(x), dev(z), dev(w2)
    torch.cuda.synchronize()
    y = B.convtranspose1d(xd, dev(w), None, 1, 0, 3, 0)
    B.convtranspose1d(zd, w2d, None, 1, 0, 1, 0, out=xd)      # overwrites x
    torch.cuda.synchronize()
    sel = [(0, 0), (1, 40), (2, 63), (3, 5)]
    got = np.stack([y[n, c].cpu().numpy() for n, c in sel])
    assert_close(got, ora.convt(x, w, None, 1, 0, 3, 0, sel=sel), what="reader of the overwritten x")


def test_dependent_ops_in_a_cuda_graph_and_across_streams():
    """The same producer -> consumer pair (a direct ConvTranspose3d writing x1, the
    fused tensor-core op reading it) captured in a CUDA graph and replayed, and run on
    two streams joined by an event: both give the result of the plain sequence."""
    x0, = rng_inputs(57, (2, 3, 5, 17, 32))
    w0, = rng_inputs(58, (3, 3, 1, 1, 1), lo=-0.8, hi=0.8)
    w, cb, b = rng_inputs(59, (3, 16, 3, 3, 3), (16,), (16,), lo=-0.2, hi=0.2)
    one, zero = (1, 1, 1), (0, 0, 0)
    xd, w0d, wd, cbd, bd = dev(x0), dev(w0), dev(w), dev(cb), dev(b)
    x1h = ora.convt(x0, w0, None, one, zero, one, zero).astype(np.float32)
    ref = ora.ct3d_scale_pool_bias(x1h, w, cb, b, (2, 2, 2), (1, 1, 1), zero, one, 2, 0.5, 1.0)

    x1 = B.convtranspose3d(xd, w0d, None, one, zero, one, zero)
    y = B.ct3d_scale_pool_bias(x1, wd, cbd, bd, scale1=0.5, scale2=1.0)
    torch.cuda.synchronize()
    plain = y.cpu().numpy()
    assert_close(plain, ref, what="plain sequence")

    # CUDA graph: capture both calls on a side stream, replay twice with fresh input
    x1.zero_(); y.zero_()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            B.convtranspose3d(xd, w0d, None, one, zero, one, zero, out=x1)
            B.ct3d_scale_pool_bias(x1, wd, cbd, bd, scale1=0.5, scale2=1.0, out=y)
    torch.cuda.synchronize()
    for _ in range(2):
        y.zero_()
        g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(y.cpu().numpy(), plain), "graph replay differs from the plain sequence"

    # two streams: the producer on s1, the consumer on s2 after an event
    x1.zero_(); y.zero_()
    torch.cuda.synchronize()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    with torch.cuda.stream(s1):
        B.convtranspose3d(xd, w0d, None, one, zero, one, zero, out=x1)
        ev = torch.cuda.Event()
        ev.record(s1)
    s2.wait_event(ev)
    with torch.cuda.stream(s2):
        B.ct3d_scale_pool_bias(x1, wd, cbd, bd, scale1=0.5, scale2=1.0, out=y)
    torch.cuda.synchronize()
    assert np.array_equal(y.cpu().numpy(), plain), "two-stream run differs from the plain sequence"


# ------------------------------------------------------------ convtranspose1d
CONVT_CASES = [  # (s, K, d, p, op, Cin, Cout, L, bias)
    (1, 5, 3, 0, 0, 32, 64, 1000, False),
    (1, 5, 3, 2, 0, 3, 16, 77, True),
    (2, 4, 2, 1, 1, 64, 64, 513, True),
    (2, 4, 2, 3, 1, 9, 24, 100, True),
    (1, 3, 1, 1, 0, 17, 72, 300, False),
    (2, 4, 1, 1, 1, 5, 8, 64, True),
    (2, 3, 1, 1, 1, 6, 16, 50, False),
    (1, 5, 1, 4, 0, 8, 8, 9, True),
    (3, 2, 1, 1, 2, 4, 8, 30, True),
    (1, 5, 3, 0, 0, 4, 12, 40, True),
    (1, 1, 1, 0, 0, 1, 8, 1, True),
    (4, 3, 5, 2, 3, 2, 3, 11, True),
    # 16-channel chunks through three window stages (resident weights with room to
    # spare), with a ragged last chunk
    (2, 4, 1, 1, 1, 40, 32, 200, True),
    (1, 5, 3, 0, 0, 24, 64, 333, True),
    # weight slabs too large to stay resident: staged with each input chunk
    (2, 4, 2, 1, 1, 128, 64, 300, True),
    (1, 5, 3, 0, 0, 96, 64, 700, False),
    (1, 3, 1, 1, 0, 150, 16, 200, True),
]


# APS_PREC_FP32_FMA: the FP32-pipe kernels; APS_PREC_FP32: the library's choice (the
# 3xTF32 tensor-core kernel where it takes the shape, else the FP32 pipe), at the same bound
@pytest.mark.parametrize("prec", [3, 0])
@pytest.mark.parametrize("s,K,d,p,op,cin,cout,L,has_bias", CONVT_CASES)
def test_convt1d_cases(s, K, d, p, op, cin, cout, L, has_bias, prec):
    x, = rng_inputs(11, (2, cin, L))
    w, b = rng_inputs(12, (cin, cout, K), (cout,), lo=-0.3, hi=0.3)
    b = b if has_bias else None
    y = B.convtranspose1d(dev(x), dev(w), None if b is None else dev(b), s, p, d, op,
                          precision=prec)
    assert_close(y.cpu().numpy(), ora.convt(x, w, b, s, p, d, op),
                 what=f"convt1d s{s} K{K} d{d} p{p} op{op} {cin}->{cout} L{L} prec {prec}")


def test_convt1d_unaligned_output():
    x, = rng_inputs(13, (2, 8, 129))
    w, = rng_inputs(14, (8, 16, 5), lo=-0.3, hi=0.3)
    L_out = 129 + 12
    buf = torch.empty(2 * 16 * L_out + 1, device="cuda")
    out = buf[1:].view(2, 16, L_out)
    B.convtranspose1d(dev(x), dev(w), None, 1, 0, 3, 0, out=out,
                      precision=B.APS_PREC_FP32_FMA)
    assert_close(out.cpu().numpy(), ora.convt(x, w, None, 1, 0, 3, 0), what="unaligned out")


@pytest.mark.parametrize("cfg", [3, 4])
@pytest.mark.slow
def test_convt1d_full_workload_sampled_planes(cfg):
    wl = workloads.get(cfg)
    p = wl.params
    x, w = wl.generate("x"), wl.generate("w")
    b = wl.generate("bias") if p["has_bias"] else None
    y = B.convtranspose1d(dev(x), dev(w), None if b is None else dev(b), p["stride"], p["pad"],
                          p["dil"], p["out_pad"], precision=B.APS_PREC_FP32_FMA)
    torch.cuda.synchronize()
    N, C = y.shape[0], y.shape[1]
    sel = [(0, 0), (N - 1, C - 1), (N // 2, 17), (3, C // 2), (N - 1, 0)]
    ref = ora.convt(x, w, b, p["stride"], p["pad"], p["dil"], p["out_pad"], sel=sel)
    got = np.stack([y[n, c].cpu().numpy() for n, c in sel])
    assert_close(got, ref, what=f"convt1d cfg {cfg}")
    assert torch.isfinite(y).all()
    if cfg == 4:  # no tap reaches an even output: exactly the bias
        assert torch.equal(y[:, :, 0::2], dev(b).view(1, -1, 1).expand_as(y[:, :, 0::2]))


# ------------------------------------------- convtranspose1d, tf32 tensor cores
def assert_frobenius(got, want, tol=5e-3, what=""):
    got = np.asarray(got, dtype=np.float64)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    assert np.isfinite(got).all(), what
    rel = np.linalg.norm(got - want) / max(np.linalg.norm(want), 1e-300)
    assert rel <= tol, f"{what}: relative Frobenius error {rel:.3e} > {tol}"
    return rel


TF32_CASES = [  # (s, K, d, p, op, Cin, Cout, L, bias)
    (1, 5, 3, 0, 0, 32, 64, 1000, False),
    (2, 4, 2, 1, 1, 64, 64, 516, True),
    (1, 3, 1, 1, 0, 8, 32, 300, True),
    (2, 4, 1, 1, 1, 16, 32, 64, True),
    (3, 2, 1, 1, 2, 8, 32, 32, True),
    (1, 2, 1, 0, 0, 32, 256, 200, True),
    (2, 3, 3, 2, 1, 96, 64, 124, False),
    (1, 3, 2, 1, 0, 64, 128, 160, True),
    (1, 1, 1, 0, 0, 24, 64, 4, True),
]


@pytest.mark.parametrize("s,K,d,p,op,cin,cout,L,has_bias", TF32_CASES)
def test_convt1d_tf32_cases(s, K, d, p, op, cin, cout, L, has_bias):
    x, = rng_inputs(21, (3, cin, L))
    w, b = rng_inputs(22, (cin, cout, K), (cout,), lo=-0.3, hi=0.3)
    b = b if has_bias else None
    y = B.convtranspose1d(dev(x), dev(w), None if b is None else dev(b), s, p, d, op,
                          precision=B.APS_PREC_TF32)
    assert_frobenius(y.cpu().numpy(), ora.convt(x, w, b, s, p, d, op),
                     what=f"tf32 s{s} K{K} d{d} p{p} op{op} {cin}->{cout} L{L}")


def test_convt1d_with_tensor_cores_passed_over():
    """With the tensor cores passed over, APS_PREC_FP32 on a shape 3xTF32 takes runs the
    FP32-pipe kernel (the same bits as APS_PREC_FP32_FMA), and the explicit tensor-core
    precisions are refused without a launch."""
    x, = rng_inputs(55, (2, 32, 400))
    w, b = rng_inputs(56, (32, 64, 5), (64,), lo=-0.3, hi=0.3)
    args = (dev(x), dev(w), dev(b), 1, 0, 3, 0)
    with skip_tensor_cores():
        y = B.convtranspose1d(*args, precision=B.APS_PREC_FP32)
        for prec in (B.APS_PREC_TF32, B.APS_PREC_TF32X3):
            with pytest.raises(B.ApsError) as e:
                B.convtranspose1d(*args, precision=prec)
            assert e.value.status == B.APS_ERR_UNSUPPORTED
    fma = B.convtranspose1d(*args, precision=B.APS_PREC_FP32_FMA)
    assert torch.equal(y, fma)
    assert_close(y.cpu().numpy(), ora.convt(x, w, b, 1, 0, 3, 0), what="convt1d fp32 fallback")
    assert not torch.equal(B.convtranspose1d(*args, precision=B.APS_PREC_FP32), fma)


# 3xTF32 (APS_PREC_TF32X3): the fp32 elementwise bound, on the tensor cores
TF32X3_CASES = [  # (s, K, d, p, op, Cin, Cout, L, bias)
    (1, 5, 3, 0, 0, 32, 64, 1000, False),
    (2, 4, 2, 1, 1, 64, 64, 516, True),     # hi+lo weights 128 KB: 16-channel chunks
    (1, 3, 1, 1, 0, 8, 32, 300, True),
    (2, 4, 1, 1, 1, 16, 32, 64, True),
    (3, 2, 1, 1, 2, 8, 32, 32, True),
    (1, 2, 1, 0, 0, 32, 256, 200, True),   # 2 x C_out > 256: three MMAs per product
    (1, 1, 1, 0, 0, 24, 64, 4, True),
    (1, 3, 1, 1, 0, 16, 128, 200, True),   # paired hi | lo weights: one N = 256 MMA
    (2, 4, 1, 1, 1, 16, 64, 132, True),    # two classes, paired: N = 128, two accumulators
    # stride 2 with the one class on even outputs (odd L_out: direct stores; L_out a
    # multiple of 4: TMA stores)
    (2, 2, 2, 0, 0, 32, 64, 200, True),
    (2, 2, 4, 0, 1, 32, 64, 200, False),
]


@pytest.mark.parametrize("s,K,d,p,op,cin,cout,L,has_bias", TF32X3_CASES)
def test_convt1d_tf32x3_cases_meet_fp32_bound(s, K, d, p, op, cin, cout, L, has_bias):
    x, = rng_inputs(25, (3, cin, L))
    w, b = rng_inputs(26, (cin, cout, K), (cout,), lo=-0.3, hi=0.3)
    b = b if has_bias else None
    y = B.convtranspose1d(dev(x), dev(w), None if b is None else dev(b), s, p, d, op,
                          precision=B.APS_PREC_TF32X3)
    assert_close(y.cpu().numpy(), ora.convt(x, w, b, s, p, d, op),
                 what=f"tf32x3 s{s} K{K} d{d} p{p} op{op} {cin}->{cout} L{L}")


def test_convt1d_tf32x3_rejects_weights_too_large_for_shared_memory():
    # hi + lo weights of 3 x 64 x 128 taps = 196 KB: no pipeline fits beside them
    x, = rng_inputs(27, (1, 64, 160))
    w, = rng_inputs(28, (64, 128, 3))
    with pytest.raises(B.ApsError) as e:
        B.convtranspose1d(dev(x), dev(w), None, 1, 1, 2, 0, precision=B.APS_PREC_TF32X3)
    assert e.value.status == B.APS_ERR_UNSUPPORTED


@pytest.mark.parametrize("cfg", [3, 4])
@pytest.mark.slow
def test_convt1d_tf32x3_full_workload_sampled_planes(cfg):
    wl = workloads.get(cfg)
    p = wl.params
    x, w = wl.generate("x"), wl.generate("w")
    b = wl.generate("bias") if p["has_bias"] else None
    y = B.convtranspose1d(dev(x), dev(w), None if b is None else dev(b), p["stride"], p["pad"],
                          p["dil"], p["out_pad"], precision=B.APS_PREC_TF32X3)
    torch.cuda.synchronize()
    N, C = y.shape[0], y.shape[1]
    sel = [(0, 0), (N - 1, C - 1), (N // 2, 17), (3, C // 2), (N - 1, 0)]
    ref = ora.convt(x, w, b, p["stride"], p["pad"], p["dil"], p["out_pad"], sel=sel)
    got = np.stack([y[n, c].cpu().numpy() for n, c in sel])
    assert_close(got, ref, what=f"tf32x3 cfg {cfg}")


@pytest.mark.parametrize("cin,cout,L", [(12, 32, 64), (32, 48, 64), (32, 64, 66), (40, 64, 64),
                                        (64, 256, 64)])
def test_convt1d_tf32_unsupported_shapes(cin, cout, L):
    x, = rng_inputs(23, (1, cin, L))
    w, = rng_inputs(24, (cin, cout, 3))
    with pytest.raises(B.ApsError) as e:
        B.convtranspose1d(dev(x), dev(w), None, 1, 0, 1, 0, precision=B.APS_PREC_TF32)
    assert e.value.status == B.APS_ERR_UNSUPPORTED


@pytest.mark.parametrize("cfg", [3, 4])
@pytest.mark.slow
def test_convt1d_tf32_full_workload_sampled_planes(cfg):
    wl = workloads.get(cfg)
    p = wl.params
    x, w = wl.generate("x"), wl.generate("w")
    b = wl.generate("bias") if p["has_bias"] else None
    y = B.convtranspose1d(dev(x), dev(w), None if b is None else dev(b), p["stride"], p["pad"],
                          p["dil"], p["out_pad"], precision=B.APS_PREC_TF32)
    torch.cuda.synchronize()
    N, C = y.shape[0], y.shape[1]
    sel = [(0, 0), (N - 1, C - 1), (N // 2, 17), (3, C // 2), (N - 1, 0)]
    ref = ora.convt(x, w, b, p["stride"], p["pad"], p["dil"], p["out_pad"], sel=sel)
    got = np.stack([y[n, c].cpu().numpy() for n, c in sel])
    assert_frobenius(got, ref, what=f"tf32 cfg {cfg}")
    assert torch.isfinite(y).all()


def test_kernel_smem_limit_survives_smaller_launches():
    """A launch that needs less dynamic shared memory must not lower the limit
    a later, larger launch of the same kernel relies on."""
    big = (1, 3, 3, 70, 20)     # fused tile > 48 KB of shared memory
    small = (1, 3, 2, 3, 4)
    base = workloads.get(0)
    for shape in (big, small, big):
        x, = rng_inputs(31, shape)
        w, cb, b = (base.generate(n) for n in ("w", "conv_bias", "bias"))
        assert_close(fused_gpu(x, w, cb, b, base.params), fused_ref(base, x, w, cb, b),
                     what=f"fused {shape}")
    for cin, cout, L in ((32, 64, 400), (8, 32, 64), (32, 64, 400)):
        x, = rng_inputs(32, (2, cin, L))
        w, = rng_inputs(33, (cin, cout, 5), lo=-0.3, hi=0.3)
        y = B.convtranspose1d(dev(x), dev(w), None, 1, 0, 3, 0, precision=B.APS_PREC_TF32)
        assert_frobenius(y.cpu().numpy(), ora.convt(x, w, None, 1, 0, 3, 0), what="tf32 order")


# ------------------------------------------------------------ degenerate inputs
def test_empty_batch_every_op():
    """N = 0: a zero-element output, no launch, no error (the data pointers of
    empty tensors may be NULL)."""
    y = B.avgpool3d(torch.empty((0, 3, 8, 8, 8), device="cuda"), 3, 2, 1)
    assert tuple(y.shape) == (0, 3, 4, 4, 4)
    w3, cb, b = (dev(a) for a in rng_inputs(41, (3, 16, 3, 3, 3), (16,), (16,)))
    y = B.ct3d_scale_pool_bias(torch.empty((0, 3, 8, 8, 8), device="cuda"), w3, cb, b)
    assert tuple(y.shape) == (0, 16, 7, 7, 7)
    y = B.convtranspose3d(torch.empty((0, 3, 4, 4, 4), device="cuda"), w3, b, 2, 1, 1, 0)
    assert tuple(y.shape) == (0, 16, 7, 7, 7)
    w1, b1 = (dev(a) for a in rng_inputs(42, (32, 64, 5), (64,)))
    for prec in (B.APS_PREC_FP32, B.APS_PREC_TF32, B.APS_PREC_TF32X3, B.APS_PREC_FP32_FMA):
        y = B.convtranspose1d(torch.empty((0, 32, 100), device="cuda"), w1, b1, 1, 0, 3, 0,
                              precision=prec)
        assert tuple(y.shape) == (0, 64, 112)


def test_zero_input_channels_give_the_bias():
    """C_in = 0: every output is the (folded) bias, at every precision."""
    b1, = rng_inputs(43, (8,))
    x1, w1 = np.zeros((2, 0, 9), np.float32), np.zeros((0, 8, 3), np.float32)
    want = ora.convt(x1, w1, b1, 2, 1, 1, 0)
    for prec in (B.APS_PREC_FP32, B.APS_PREC_TF32, B.APS_PREC_TF32X3, B.APS_PREC_FP32_FMA):
        y = B.convtranspose1d(torch.empty((2, 0, 9), device="cuda"),
                              torch.empty((0, 8, 3), device="cuda"), dev(b1), 2, 1, 1, 0,
                              precision=prec)
        assert_close(y.cpu().numpy(), want, what=f"convt1d C_in 0 prec {prec}")
    b3, cb = rng_inputs(44, (16,), (16,))
    x3, w3 = np.zeros((1, 0, 3, 4, 4), np.float32), np.zeros((0, 16, 3, 3, 3), np.float32)
    y = B.convtranspose3d(torch.empty((1, 0, 3, 4, 4), device="cuda"),
                          torch.empty((0, 16, 3, 3, 3), device="cuda"), dev(b3), 2, 1, 1, 0)
    assert_close(y.cpu().numpy(), ora.convt(x3, w3, b3, 2, 1, 1, 0), what="convt3d C_in 0")
    y = B.ct3d_scale_pool_bias(torch.empty((1, 0, 3, 4, 4), device="cuda"),
                               torch.empty((0, 16, 3, 3, 3), device="cuda"), dev(cb), dev(b3),
                               scale1=0.5, scale2=2.0)
    assert_close(y.cpu().numpy(), ora.ct3d_scale_pool_bias(x3, w3, cb, b3, 2, 1, 0, 1, 2, 0.5,
                                                           2.0), what="fused C_in 0")


def test_launches_on_a_side_stream_are_ordered_on_it():
    wl = workloads.get(3).with_input_shape((2, 32, 700))
    p = wl.params
    x, w = wl.generate("x"), wl.generate("w")
    s = torch.cuda.Stream()
    xd, wd = dev(x), dev(w)
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        y = B.convtranspose1d(xd, wd, None, p["stride"], p["pad"], p["dil"], p["out_pad"],
                              precision=B.APS_PREC_TF32X3, stream=s)
    s.synchronize()
    assert_close(y.cpu().numpy(), ora.convt(x, w, None, p["stride"], p["pad"], p["dil"],
                                            p["out_pad"]), what="side stream")


def test_no_kernel_recorded_a_timeout():
    """Every bounded wait in every launch so far completed in time."""
    torch.cuda.synchronize()
    st, bits = B.aps_device_status(clear=False)
    assert st == B.APS_OK and bits == 0, (st, bits)


def test_fp32_fma_probe_reports_a_sane_rate():
    """The FMA-rate probe behind the roofline of the FMA-bound kernels: its
    packed form beats its scalar form and both lie below the unit-count peak
    (152 SMs x 128 lanes x 2 FLOP x 2.07 GHz = 80.5 TFLOP/s)."""
    import bench
    r = bench.measure_fma_ceilings(torch, __import__("average_pooling_stencil_gb300"),
                                   bench.sm_count_of(torch), iters=1024, reps=3)
    assert 10.0 < r["scalar"] < r["packed"] < 82.0, r


# ------------------------------------------------------------ guard canaries
# Every op writes into a view in the middle of a larger buffer whose other words hold a
# sentinel no kernel writes (a NaN bit pattern): the words around the view must survive, at a
# 256-byte-aligned start and at a start one float off (which sends the paths that need an
# aligned output to their fallbacks and gives the bulk-copy runs every head/tail split).
GUARD = 64
SENTINEL = 0x7FA5A5A5


def _canary_cases():
    base0, base3, base4, base5 = (workloads.get(i) for i in (0, 3, 4, 5))
    cases = {}

    def pool(shape, k, s, p):
        x, = rng_inputs(51, shape)
        want = ora.avgpool3d(x, k, s, p, 1, 0)
        return want, lambda out: B.avgpool3d(dev(x), k, s, p, out=out), 1e-5
    cases["avgpool_tma"] = lambda: pool((2, 3, 9, 20, 68), (3, 3, 3), (2, 2, 2), (1, 1, 1))
    cases["avgpool_direct"] = lambda: pool((1, 2, 5, 7, 9), (2, 3, 2), (1, 2, 2), (1, 1, 0))

    def fused(shape, k=(3, 3, 3), s=(2, 2, 2), p=(1, 1, 1)):
        x, = rng_inputs(52, shape)
        w, cb, b = rng_inputs(53, (shape[1], 16) + k, (16,), (16,), lo=-0.3, hi=0.3)
        want = ora.ct3d_scale_pool_bias(x, w, cb, b, s, p, (0, 0, 0), (1, 1, 1), 2, 0.5, 1.25)
        return want, lambda out: B.ct3d_scale_pool_bias(
            dev(x), dev(w), dev(cb), dev(b), s, p, 0, 1, 2, 0.5, 1.25, out=out), 1e-5
    cases["fused_tc"] = lambda: fused((2, 3, 4, 8, 32))
    cases["fused_fp32"] = lambda: fused((1, 5, 3, 6, 20))
    cases["fused_direct"] = lambda: fused((1, 2, 3, 5, 6), k=(2, 2, 2), s=(2, 2, 2), p=(0, 0, 0))

    def convt1d(wl, shape, prec, tol):
        x, = rng_inputs(54, shape)
        w, = rng_inputs(55, (shape[1], 64, wl.params["k"]), lo=-0.1, hi=0.1)
        b, = rng_inputs(56, (64,))
        p = wl.params
        want = ora.convt(x, w, b, p["stride"], p["pad"], p["dil"], p["out_pad"])
        return want, lambda out: B.convtranspose1d(
            dev(x), dev(w), dev(b), p["stride"], p["pad"], p["dil"], p["out_pad"],
            precision=prec, out=out), tol
    cases["convt1d_fp32"] = lambda: convt1d(base4, (2, 64, 300), B.APS_PREC_FP32_FMA, 1e-5)
    cases["convt1d_tf32"] = lambda: convt1d(base3, (2, 32, 400), B.APS_PREC_TF32, None)
    cases["convt1d_tf32x3"] = lambda: convt1d(base3, (2, 32, 400), B.APS_PREC_TF32X3, 1e-5)

    def convt3d(shape, k=(3, 3, 3), s=(2, 2, 2), p=(1, 1, 1), op=(0, 0, 0)):
        x, = rng_inputs(57, shape)
        w, b = rng_inputs(58, (shape[1], 16) + k, (16,), lo=-0.3, hi=0.3)
        want = ora.convt(x, w, b, s, p, (1, 1, 1), op)
        return want, lambda out: B.convtranspose3d(dev(x), dev(w), dev(b), s, p, (1, 1, 1), op,
                                                   out=out), 1e-5
    cases["convt3d_tc"] = lambda: convt3d((2, 3, 5, 9, 12), op=(1, 0, 1))
    cases["convt3d_fp32"] = lambda: convt3d((1, 8, 3, 7, 36))
    cases["convt3d_direct"] = lambda: convt3d((1, 2, 3, 4, 5), k=(2, 3, 2), s=(1, 2, 3),
                                              p=(0, 1, 1))
    del base0, base5
    return cases


CANARY = _canary_cases()


@pytest.mark.parametrize("offset", [GUARD, GUARD + 1])
@pytest.mark.parametrize("name", sorted(CANARY))
def test_outputs_stay_inside_their_buffer(name, offset):
    want, run, tol = CANARY[name]()
    n = want.size
    buf = torch.empty(n + 2 * GUARD, device="cuda", dtype=torch.float32)
    buf.view(torch.int32).fill_(SENTINEL)
    out = buf[offset:offset + n].view(want.shape)
    run(out)
    torch.cuda.synchronize()
    raw = buf.view(torch.int32).cpu().numpy()
    outside = np.concatenate([raw[:offset], raw[offset + n:]])
    assert (outside == SENTINEL).all(), f"{name}: {int((outside != SENTINEL).sum())} guard words written"
    got = out.cpu().numpy()
    if tol is None:
        assert_frobenius(got, want, what=name)
    else:
        assert_close(got, want, tol=tol, what=name)


# ------------------------------------------------------------ error propagation
@pytest.mark.parametrize("name", ["avgpool_tma", "fused_tc", "fused_fp32", "convt1d_fp32",
                                  "convt1d_tf32x3", "convt3d_tc", "convt3d_direct"])
def test_a_rejected_launch_reaches_the_caller(name):
    """With the test hook set, the next launch reports APS_ERR_LAUNCH: the op returns it
    and the binding raises it; the following call runs normally."""
    want, run, tol = CANARY[name]()
    out = torch.empty(want.shape, device="cuda", dtype=torch.float32)
    B.aps_debug_fail_launches(1)
    try:
        with pytest.raises(B.ApsError) as e:
            run(out)
        assert e.value.status == B.APS_ERR_LAUNCH
    finally:
        B.aps_debug_fail_launches(0)
    run(out)
    assert_close(out.cpu().numpy(), want, tol=tol, what=name)


def test_a_pipeline_wait_that_runs_out_is_recorded_and_the_context_stays_usable():
    """A wait made to run out on the host's request (one input box withheld, its barrier
    still expecting the bytes, a 50 ms limit): the launch returns, the kernel records
    APS_DEVERR_TIMEOUT in the status word instead of hanging, and the next launch on the
    same context is normal and correct."""
    x = workloads.get(1).with_input_shape((2, 3, 9, 20, 68)).generate("x")
    xd = dev(x)
    st, _ = B.aps_device_status(clear=True)
    assert st == 0
    B.aps_debug_stall_next_pool(50_000_000)
    B.avgpool3d(xd, 3, 2, 1)
    torch.cuda.synchronize()
    st, bits = B.aps_device_status(clear=True)
    assert st == 0 and bits & B.APS_DEVERR_TIMEOUT, bits
    y = B.avgpool3d(xd, 3, 2, 1)
    assert_close(y.cpu().numpy(), ora.avgpool3d(x, 3, 2, 1, 1, 0), what="after a timed-out launch")
    st, bits = B.aps_device_status(clear=True)
    assert st == 0 and bits == 0
