"""fp64 CPU oracle for the stencil ops (ctypes wrapper around oracle.c).

TEST INFRASTRUCTURE ONLY: tests/, __graft_entry__.smoke() and bench.py's
cpu_baseline / reference leg are the only callers.  The CUDA library and its
Python binding never import this package, and it imports nothing from them.

What each function computes is written out in oracle.c: the scatter definition
of transposed convolution, the explicit average pool, and the Kimi-K2.6__l2_p50
chain (convT + conv bias, x scale1, AvgPool3d(pool_k), + bias, x scale2) in
that literal order.  Parity status: every function here is pinned by
tests/test_oracle_pins.py against facts the pages fix (output-size closed
forms, the printed transposed-matrix examples, the 27-tap table of the fused
pool window, the constant 27 divisor) and against independent brute force
(dense forward-convolution matrices, adjoint identity, separable window sums).
The ceil_mode branch of the pool is pinned against its closed-form window
count only (the pages never use ceil mode).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None

_I64P = ctypes.POINTER(ctypes.c_int64)
_IP = ctypes.POINTER(ctypes.c_int)
_FP = ctypes.POINTER(ctypes.c_float)
_DP = ctypes.POINTER(ctypes.c_double)


def build(force: bool = False, src: str | None = None, out: str | None = None) -> str:
    """Compile oracle.c (or ``src``) into a shared library with gcc."""
    src = src or _SRC
    out = out or _LIB
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(src)):
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fPIC",
           "-shared", src, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _bind(lib):
    lib.ora_max_threads.restype = ctypes.c_int
    lib.ora_set_threads.argtypes = [ctypes.c_int]
    lib.ora_convt_len.restype = ctypes.c_int64
    lib.ora_convt_len.argtypes = [ctypes.c_int64] + [ctypes.c_int] * 5
    lib.ora_pool_len.restype = ctypes.c_int64
    lib.ora_pool_len.argtypes = [ctypes.c_int64] + [ctypes.c_int] * 4
    lib.ora_convt_planes.restype = ctypes.c_int
    lib.ora_convt_planes.argtypes = [_FP, _I64P, _FP, _FP, ctypes.c_int64, _IP, _IP, _IP,
                                     _IP, _IP, _I64P, ctypes.c_int64, _DP]
    lib.ora_avgpool_planes.restype = ctypes.c_int
    lib.ora_avgpool_planes.argtypes = [_FP, _I64P, _IP, _IP, _IP, ctypes.c_int,
                                       ctypes.c_int, _I64P, ctypes.c_int64, _DP]
    lib.ora_ct3d_scale_pool_bias_planes.restype = ctypes.c_int
    lib.ora_ct3d_scale_pool_bias_planes.argtypes = [
        _FP, _I64P, _FP, _FP, _FP, ctypes.c_int64, _IP, _IP, _IP, _IP, _IP, ctypes.c_int,
        ctypes.c_double, ctypes.c_double, _I64P, ctypes.c_int64, _DP]
    return lib


def load(path: str | None = None):
    """Load (building first if needed) the oracle library."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    if _lib is None:
        build()
        _lib = _bind(ctypes.CDLL(_LIB))
    return _lib


def _f32(a):
    a = np.ascontiguousarray(a, dtype=np.float32)
    return a, a.ctypes.data_as(_FP)


def _i64(v):
    a = np.ascontiguousarray(v, dtype=np.int64)
    return a, a.ctypes.data_as(_I64P)


def _i32(v):
    a = np.ascontiguousarray(v, dtype=np.int32)
    return a, a.ctypes.data_as(_IP)


def _triple(v, fill):
    """Scalar -> the same value in all three dims; shorter sequence -> left-padded."""
    if not hasattr(v, "__len__"):
        return [int(v)] * 3
    v = [int(t) for t in v]
    return [fill] * (3 - len(v)) + v


def _sel(sel):
    if sel is None:
        return None, None, 0
    s = np.ascontiguousarray(np.asarray(sel, dtype=np.int64).reshape(-1, 2))
    return s, s.ctypes.data_as(_I64P), s.shape[0]


def threads() -> int:
    return load().ora_max_threads()


def set_threads(n: int) -> None:
    load().ora_set_threads(int(n))


def convt_len(L, k, s, p, d, op) -> int:
    return int(load().ora_convt_len(int(L), int(k), int(s), int(p), int(d), int(op)))


def pool_len(L, k, s, p, ceil_mode=0) -> int:
    return int(load().ora_pool_len(int(L), int(k), int(s), int(p), int(ceil_mode)))


def _spatial5(x):
    """Shape [N, C, *spatial] padded with unit dims on the left to 3 spatial dims."""
    sh = list(x.shape)
    nd = len(sh) - 2
    if not 1 <= nd <= 3:
        raise ValueError("expected 1 to 3 spatial dims")
    return sh[:2] + [1] * (3 - nd) + sh[2:], nd


def convt(x, w, b, stride, pad, dil, out_pad, sel=None, backend=None):
    """Transposed convolution (scatter form) for 1-3 spatial dims.

    x [N, Cin, *L], w [Cin, Cout, *k], b [Cout] or None.  Returns fp64
    [N, Cout, *O], or [len(sel), *O] when ``sel`` lists (n, co) planes."""
    lib = backend or load()
    in5, nd = _spatial5(x)
    cout = int(w.shape[1])
    k = [1] * (3 - nd) + list(w.shape[2:])
    st, pd, dl, op = (_triple(stride, 1), _triple(pad, 0), _triple(dil, 1), _triple(out_pad, 0))
    st = [1] * (3 - nd) + st[3 - nd:]
    pd = [0] * (3 - nd) + pd[3 - nd:]
    dl = [1] * (3 - nd) + dl[3 - nd:]
    op = [0] * (3 - nd) + op[3 - nd:]
    O = [int(lib.ora_convt_len(in5[2 + i], k[i], st[i], pd[i], dl[i], op[i])) for i in range(3)]
    xa, xp = _f32(x)
    wa, wp = _f32(w)
    ba, bp = (None, None) if b is None else _f32(b)
    sa, sp, ns = _sel(sel)
    nplanes = ns if sel is not None else in5[0] * cout
    y = np.empty((nplanes, O[0], O[1], O[2]), dtype=np.float64)
    keep = [_i64(in5), _i32(k), _i32(st), _i32(pd), _i32(dl), _i32(op)]
    rc = lib.ora_convt_planes(xp, keep[0][1], wp, bp, cout, keep[1][1], keep[2][1], keep[3][1],
                              keep[4][1], keep[5][1], sp, ns, y.ctypes.data_as(_DP))
    if rc != 0:
        raise ValueError("oracle convt: bad arguments")
    osp = O[3 - nd:]
    if sel is not None:
        return y.reshape([nplanes] + osp)
    return y.reshape([in5[0], cout] + osp)


def avgpool3d(x, k, stride, pad, count_include_pad=1, ceil_mode=0, sel=None, backend=None):
    """AvgPool3d on x [N, C, D, H, W]; fp64 [N, C, *P] (or [len(sel), *P])."""
    lib = backend or load()
    if x.ndim != 5:
        raise ValueError("x must be [N, C, D, H, W]")
    k, st, pd = _triple(k, 1), _triple(stride, 1), _triple(pad, 0)
    P = [int(lib.ora_pool_len(x.shape[2 + i], k[i], st[i], pd[i], int(ceil_mode)))
         for i in range(3)]
    if min(P) <= 0:
        raise ValueError("oracle avgpool: empty output")
    xa, xp = _f32(x)
    sa, sp, ns = _sel(sel)
    nplanes = ns if sel is not None else x.shape[0] * x.shape[1]
    y = np.empty((nplanes, *P), dtype=np.float64)
    keep = [_i64(x.shape), _i32(k), _i32(st), _i32(pd)]
    rc = lib.ora_avgpool_planes(xp, keep[0][1], keep[1][1], keep[2][1], keep[3][1],
                                int(count_include_pad), int(ceil_mode), sp, ns,
                                y.ctypes.data_as(_DP))
    if rc != 0:
        raise ValueError("oracle avgpool: bad arguments")
    if sel is not None:
        return y
    return y.reshape(x.shape[0], x.shape[1], *P)


def ct3d_scale_pool_bias(x, w, conv_bias, bias, stride, pad, out_pad, dil, pool_k,
                         scale1, scale2, sel=None, backend=None):
    """The l2_p50 chain on x [N, Cin, D, H, W], w [Cin, Cout, kD, kH, kW]."""
    lib = backend or load()
    if x.ndim != 5 or w.ndim != 5:
        raise ValueError("expected 3 spatial dims")
    cout = int(w.shape[1])
    k = list(w.shape[2:])
    st, pd, op, dl = _triple(stride, 1), _triple(pad, 0), _triple(out_pad, 0), _triple(dil, 1)
    O = [int(lib.ora_convt_len(x.shape[2 + i], k[i], st[i], pd[i], dl[i], op[i]))
         for i in range(3)]
    P = [int(lib.ora_pool_len(O[i], pool_k, pool_k, 0, 0)) for i in range(3)]
    if min(P) <= 0:
        raise ValueError("oracle fused: empty output")
    xa, xp = _f32(x)
    wa, wp = _f32(w)
    ca, cp = (None, None) if conv_bias is None else _f32(conv_bias)
    ba, bp = _f32(bias)
    sa, sp, ns = _sel(sel)
    nplanes = ns if sel is not None else x.shape[0] * cout
    y = np.empty((nplanes, *P), dtype=np.float64)
    keep = [_i64(x.shape), _i32(k), _i32(st), _i32(pd), _i32(dl), _i32(op)]
    rc = lib.ora_ct3d_scale_pool_bias_planes(
        xp, keep[0][1], wp, cp, bp, cout, keep[1][1], keep[2][1], keep[3][1], keep[4][1],
        keep[5][1], int(pool_k), float(scale1), float(scale2), sp, ns, y.ctypes.data_as(_DP))
    if rc != 0:
        raise ValueError("oracle fused: bad arguments")
    if sel is not None:
        return y
    return y.reshape(x.shape[0], cout, *P)
