"""The C ABI without a GPU: the library loads, exports every symbol the header
declares, answers shape queries like the pages' closed forms, and rejects bad
arguments before touching CUDA."""
import ctypes
import os
import re

import pytest

import __graft_entry__
import oracle as ora
import pins
from average_pooling_stencil_gb300 import binding as B
from average_pooling_stencil_gb300 import workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "aps.h")


@pytest.fixture(scope="module", autouse=True)
def built():
    __graft_entry__.build()


def header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(aps_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_binding_exports():
    assert header_functions() == sorted(B.EXPORTS)


def test_header_constants_match_the_binding():
    text = open(HEADER).read()
    defines = dict(re.findall(r"#define\s+(APS_PREC_[A-Z0-9_]+)\s+(\d+)", text))
    assert set(defines) == {"APS_PREC_FP32", "APS_PREC_TF32", "APS_PREC_TF32X3",
                            "APS_PREC_FP32_FMA"}
    for name, v in defines.items():
        assert getattr(B, name) == int(v), name
    for name, v in re.findall(r"\b(APS_(?:OK|ERR_[A-Z]+))\s*=\s*(-?\d+)", text):
        assert getattr(B, name) == int(v), name


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(B.LIB_PATH)
    for name in header_functions():
        assert hasattr(lib, name), name
    assert B.aps_abi_version() == 1


def test_status_strings():
    for code in range(0, -7, -1):
        s = B.status_string(code)
        assert s and "unknown" not in s
    assert "unknown" in B.status_string(-99)


def test_printed_sizes_through_shape_queries():
    """The sizes the pages print (golden/output_sizes.txt) via the ABI's queries."""
    for op, L, prm, want in pins.load_sizes():
        if op == "convt":
            st, out = B.aps_convtranspose1d_out_shape((1, 1, L), 1, prm["k"], prm["s"], prm["p"],
                                                      prm["d"], prm["op"])
            assert st == 0 and out[2] == want
        else:
            st, out = B.aps_avgpool3d_out_shape((1, 1, L, L, L), prm["k"], prm["s"], prm["p"])
            assert st == 0 and out[2:] == (want, want, want)


def test_workload_output_shapes():
    """Output shapes of the workloads (cfg 4 has 131076 outputs: the
    closed form (65536-1)*2 - 2 + 2*3 + 1 + 1; cfg 5 is l2_p50's pre-pool
    tensor, (16-1)*2 - 2 + 3 = 31 and (32-1)*2 - 2 + 3 = 63; cfg 7's
    output_padding 1 makes the pre-pool sizes 32 and 64, pooled 16 and 32, and so do
    cfg 11's 4-tap kernels: (16-1)*2 - 2 + 4 = 32)."""
    want = {0: (2, 16, 7, 15, 15), 1: (16, 32, 64, 64, 128), 2: (128, 16, 15, 31, 31),
            3: (32, 64, 131084), 4: (16, 64, 131076), 5: (128, 16, 31, 63, 63),
            6: (128, 16, 15, 31, 31), 7: (128, 16, 16, 32, 32), 8: (16, 32, 64, 64, 128),
            9: (16, 32, 64, 64, 128), 10: (128, 16, 31, 63, 63), 11: (128, 16, 16, 32, 32),
            12: (64, 16, 31, 63, 127), 13: (128, 16, 15, 31, 29)}
    for cfg, shape in want.items():
        wl = workloads.get(cfg)
        p = wl.params
        xs = wl.tensors["x"][0]
        if wl.op == "ct3d_scale_pool_bias":
            st, out = B.aps_ct3d_scale_pool_bias_out_shape(xs, p["c_out"], p["k"], p["stride"],
                                                           p["pad"], p["out_pad"], p["dil"],
                                                           p["pool_k"])
        elif wl.op == "avgpool3d":
            st, out = B.aps_avgpool3d_out_shape(xs, p["k"], p["stride"], p["pad"], p["ceil_mode"])
        elif wl.op == "convtranspose3d":
            st, out = B.aps_convtranspose3d_out_shape(xs, p["c_out"], p["k"], p["stride"],
                                                      p["pad"], p["dil"], p["out_pad"])
        else:
            st, out = B.aps_convtranspose1d_out_shape(xs, p["c_out"], p["k"], p["stride"],
                                                      p["pad"], p["dil"], p["out_pad"])
        assert st == 0 and out == shape, (cfg, st, out)


def test_shape_queries_agree_with_oracle_sizes():
    import itertools
    for L, k, s, p, d in itertools.product((1, 2, 7, 16), (1, 2, 3, 5), (1, 2, 3), (0, 1, 2),
                                           (1, 2, 3)):
        for op in range(max(s, d)):
            want = ora.convt_len(L, k, s, p, d, op)
            st, out = B.aps_convtranspose1d_out_shape((2, 3, L), 4, k, s, p, d, op)
            if want <= 0:
                assert st == B.APS_ERR_SHAPE
            else:
                assert st == 0 and out == (2, 4, want)
    for L, k, s, p, c in itertools.product((1, 3, 6, 9), (1, 2, 3, 4), (1, 2, 3), (0, 1, 2),
                                           (0, 1)):
        if 2 * p > k:
            continue
        want = ora.pool_len(L, k, s, p, c)
        st, out = B.aps_avgpool3d_out_shape((1, 2, L, L, L), k, s, p, c)
        if want <= 0:
            assert st == B.APS_ERR_SHAPE
        else:
            assert st == 0 and out == (1, 2, want, want, want), (L, k, s, p, c)


FAKE = 0x10000  # never dereferenced: every call below returns before any CUDA call


def test_null_pointers_rejected():
    assert B.aps_avgpool3d(0, (1, 1, 4, 4, 4), 3, 2, 1, 1, 0, FAKE) == B.APS_ERR_NULL
    assert B.aps_avgpool3d(FAKE, (1, 1, 4, 4, 4), 3, 2, 1, 1, 0, 0) == B.APS_ERR_NULL
    assert B.aps_ct3d_scale_pool_bias(FAKE, (1, 3, 4, 4, 4), FAKE, 0, 0, 16, 3, 2, 1, 0, 1, 2,
                                      0.5, 1.0, FAKE) == B.APS_ERR_NULL
    assert B.aps_convtranspose1d(FAKE, (1, 2, 8), 0, 0, 4, 3, 1, 0, 1, 0, 0, FAKE) == B.APS_ERR_NULL
    st = B.lib().aps_avgpool3d_out_shape(None, None, None, None, 0, None)
    assert st == B.APS_ERR_NULL


def test_bad_parameters_rejected():
    E = B.APS_ERR_SHAPE
    assert B.aps_avgpool3d(FAKE, (1, 1, 4, 4, 4), 3, 2, 2, 1, 0, FAKE) == E      # 2p > k
    assert B.aps_avgpool3d(FAKE, (1, 1, 4, 4, 4), 3, 0, 1, 1, 0, FAKE) == E      # stride 0
    assert B.aps_avgpool3d(FAKE, (1, 1, 1, 4, 4), 5, 1, 0, 1, 0, FAKE) == E      # empty output
    assert B.aps_avgpool3d(FAKE, (-1, 1, 4, 4, 4), 3, 2, 1, 1, 0, FAKE) == E     # negative dim
    assert B.aps_ct3d_scale_pool_bias(FAKE, (1, 3, 4, 4, 4), FAKE, 0, FAKE, 16, 3, 2, 1, 2, 1, 2,
                                      0.5, 1.0, FAKE) == E                       # op >= max(s,d)
    assert B.aps_ct3d_scale_pool_bias(FAKE, (1, 3, 4, 4, 4), FAKE, 0, FAKE, 16, 3, 2, 1, 0, 1, 0,
                                      0.5, 1.0, FAKE) == E                       # pool_k 0
    assert B.aps_ct3d_scale_pool_bias(FAKE, (1, 3, 1, 1, 1), FAKE, 0, FAKE, 16, 1, 1, 0, 0, 1, 2,
                                      0.5, 1.0, FAKE) == E                       # pooled size 0
    assert B.aps_convtranspose1d(FAKE, (1, 2, 8), FAKE, 0, 4, 3, 1, 0, 1, 1, 0, FAKE) == E
    assert B.aps_convtranspose1d(FAKE, (1, 2, 1), FAKE, 0, 4, 1, 1, 1, 1, 0, 0, FAKE) == E
    assert B.aps_convtranspose1d(FAKE, (1, 2, 8), FAKE, 0, 0, 3, 1, 0, 1, 0, 0, FAKE) == E
    assert B.aps_convtranspose1d(FAKE, (1, 2, 8), FAKE, 0, 4, 3, 1, 0, 1, 0, 7, FAKE) == E
    huge = 1 << 40
    assert B.aps_avgpool3d(FAKE, (huge, huge, 4, 4, 4), 3, 2, 1, 1, 0, FAKE) == E


def test_misaligned_pointers_rejected():
    A = B.APS_ERR_ALIGN
    assert B.aps_avgpool3d(FAKE + 2, (1, 1, 4, 4, 4), 3, 2, 1, 1, 0, FAKE) == A
    assert B.aps_avgpool3d(FAKE, (1, 1, 4, 4, 4), 3, 2, 1, 1, 0, FAKE + 1) == A
    assert B.aps_ct3d_scale_pool_bias(FAKE, (1, 3, 4, 4, 4), FAKE + 2, 0, FAKE, 16, 3, 2, 1, 0, 1,
                                      2, 0.5, 1.0, FAKE) == A
    assert B.aps_convtranspose1d(FAKE, (1, 2, 8), FAKE, FAKE + 3, 4, 3, 1, 0, 1, 0, 0, FAKE) == A


def test_empty_tensors_are_noops():
    """N = 0 (or C = 0 for the pool) is valid and launches nothing."""
    assert B.aps_avgpool3d(FAKE, (0, 3, 4, 4, 4), 3, 2, 1, 1, 0, FAKE) == B.APS_OK
    assert B.aps_avgpool3d(FAKE, (2, 0, 4, 4, 4), 3, 2, 1, 1, 0, FAKE) == B.APS_OK
    assert B.aps_ct3d_scale_pool_bias(FAKE, (0, 3, 4, 4, 4), FAKE, 0, FAKE, 16, 3, 2, 1, 0, 1, 2,
                                      0.5, 1.0, FAKE) == B.APS_OK
    assert B.aps_convtranspose1d(FAKE, (0, 2, 8), FAKE, 0, 4, 3, 1, 0, 1, 0, 0, FAKE) == B.APS_OK


def test_skip_tensor_cores_hook_refuses_the_explicit_tensor_core_precisions_before_cuda():
    """With the hook on, APS_PREC_TF32 / APS_PREC_TF32X3 are refused by a host check (no CUDA
    call: this runs without a GPU); validation still comes first; the hook turns off again."""
    B.aps_debug_skip_tensor_cores(True)
    try:
        for prec in (B.APS_PREC_TF32, B.APS_PREC_TF32X3):
            assert B.aps_convtranspose1d(FAKE, (1, 32, 64), FAKE, 0, 64, 5, 1, 0, 3, 0, prec,
                                         FAKE) == B.APS_ERR_UNSUPPORTED
            assert B.aps_convtranspose1d(0, (1, 32, 64), FAKE, 0, 64, 5, 1, 0, 3, 0, prec,
                                         FAKE) == B.APS_ERR_NULL
            assert B.aps_convtranspose1d(FAKE, (0, 32, 64), FAKE, 0, 64, 5, 1, 0, 3, 0, prec,
                                         FAKE) == B.APS_OK
    finally:
        B.aps_debug_skip_tensor_cores(False)


def test_tensor_api_requires_cuda_tensors():
    import torch
    with pytest.raises(TypeError):
        B.avgpool3d(torch.zeros(1, 1, 4, 4, 4))


def test_convtranspose3d_shape_query_matches_closed_form_and_rejects_bad_params():
    """O = (I-1)*s - 2p + d*(k-1) + op + 1 per dim; out_pad must be < max(s, d)."""
    cases = [((1, 2, 4, 5, 6), (3, 3, 3), (2, 2, 2), (1, 1, 1), (1, 1, 1), (0, 1, 0)),
             ((2, 1, 3, 3, 3), (2, 3, 4), (1, 2, 3), (0, 1, 2), (2, 1, 1), (1, 1, 2))]
    for xs, k, s, p, d, op in cases:
        st, out = B.aps_convtranspose3d_out_shape(xs, 7, k, s, p, d, op)
        want = tuple((xs[2 + i] - 1) * s[i] - 2 * p[i] + d[i] * (k[i] - 1) + op[i] + 1
                     for i in range(3))
        assert st == 0 and out == (xs[0], 7) + want, (st, out, want)
    st, _ = B.aps_convtranspose3d_out_shape((1, 1, 4, 4, 4), 2, (3, 3, 3), (2, 2, 2),
                                            (1, 1, 1), (1, 1, 1), (2, 0, 0))
    assert st == B.APS_ERR_SHAPE
    st, _ = B.aps_convtranspose3d_out_shape((1, 1, 4, 4, 4), 0, (3, 3, 3), (2, 2, 2),
                                            (1, 1, 1), (1, 1, 1), (0, 0, 0))
    assert st == B.APS_ERR_SHAPE
    st = B.aps_convtranspose3d(0, (1, 1, 4, 4, 4), 0, 0, 2, (3, 3, 3), (2, 2, 2), (1, 1, 1),
                               (1, 1, 1), (0, 0, 0), 0)
    assert st == B.APS_ERR_NULL


def test_extents_beyond_the_launch_limits_are_unsupported_before_any_cuda_call():
    """Channel counts and spatial sizes of 2^30 or more (and an avgpool output plane of
    2^31 cells or more) are valid shapes the launches decline: APS_ERR_UNSUPPORTED, decided
    on the host (this machine has no GPU, so any CUDA call would fail differently)."""
    U = B.APS_ERR_UNSUPPORTED
    big = 1 << 30
    assert B.aps_avgpool3d(FAKE, (1, 1, 4, 4, big), 3, 2, 1, 1, 0, FAKE) == U
    # each output size below 2^30, but 2^31 cells in a plane
    assert B.aps_avgpool3d(FAKE, (1, 1, 2, 1 << 16, 1 << 16), 1, 1, 0, 1, 0, FAKE) == U
    # W = 2^29 + 1: pre-pool width 2^30 + 1, pooled width 2^29 (pool_k times it is 2^30)
    assert B.aps_ct3d_scale_pool_bias(FAKE, (1, 3, 4, 4, big // 2 + 1), FAKE, 0, FAKE, 16, 3,
                                      2, 1, 0, 1, 2, 0.5, 1.0, FAKE) == U
    assert B.aps_convtranspose3d(FAKE, (1, 1, 4, 4, big // 2 + 1), FAKE, 0, 2, (3, 3, 3), (2, 2, 2),
                                 (1, 1, 1), (1, 1, 1), (0, 0, 0), FAKE) == U
    for prec in (0, 1, 2):
        assert B.aps_convtranspose1d(FAKE, (1, 2, big), FAKE, 0, 4, 3, 1, 0, 1, 0, prec,
                                     FAKE) == U
        assert B.aps_convtranspose1d(FAKE, (1, big, 8), FAKE, 0, 4, 3, 1, 0, 1, 0, prec,
                                     FAKE) == U
    # the shape queries still answer for such shapes
    st, out = B.aps_convtranspose1d_out_shape((1, 2, big), 4, 3, 1, 0, 1, 0)
    assert st == 0 and out == (1, 4, big + 2)
