"""Python binding of libaps.so (include/aps.h): argument marshalling only.

Every computation runs in the library's CUDA kernels.  If the library has not
been built, or no CUDA device is present, calls raise instead of computing
anything another way.

Two layers:
  * ``aps_*`` functions mirror the C ABI one to one (device pointers as ints,
    shapes as sequences, stream as a cudaStream_t handle int) and return the
    aps_status code.
  * ``avgpool3d``, ``ct3d_scale_pool_bias`` and ``convtranspose1d`` take torch
    CUDA tensors, allocate the output with torch (or use ``out``), call the
    ABI on the current (or given) stream, and raise ApsError on a non-zero
    status.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libaps.so")

APS_OK = 0
APS_ERR_NULL = -1
APS_ERR_SHAPE = -2
APS_ERR_UNSUPPORTED = -3
APS_ERR_ALIGN = -4
APS_ERR_LAUNCH = -5
APS_ERR_CUDA = -6
APS_DEVERR_TIMEOUT = 1
APS_PREC_FP32 = 0
APS_PREC_TF32 = 1
APS_PREC_TF32X3 = 2
APS_PREC_FP32_FMA = 3

# Every symbol include/aps.h declares.
EXPORTS = [
    "aps_abi_version", "aps_status_string", "aps_avgpool3d_out_shape", "aps_avgpool3d",
    "aps_ct3d_scale_pool_bias_out_shape", "aps_ct3d_scale_pool_bias",
    "aps_convtranspose3d_out_shape", "aps_convtranspose3d",
    "aps_convtranspose1d_out_shape", "aps_convtranspose1d", "aps_device_status",
    "aps_fp32_fma_probe", "aps_debug_fail_launches", "aps_debug_stall_next_pool",
    "aps_debug_skip_tensor_cores",
]

_lib = None
_I64_5 = ctypes.c_int64 * 5
_I64_3 = ctypes.c_int64 * 3
_I32_3 = ctypes.c_int * 3
_VP = ctypes.c_void_p


class ApsError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


def lib():
    """The loaded library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                "(python -c 'import __graft_entry__ as g; g.build()')")
        L = ctypes.CDLL(LIB_PATH)
        L.aps_abi_version.restype = ctypes.c_int
        L.aps_status_string.restype = ctypes.c_char_p
        L.aps_status_string.argtypes = [ctypes.c_int]
        L.aps_avgpool3d_out_shape.argtypes = [_VP, _VP, _VP, _VP, ctypes.c_int, _VP]
        L.aps_avgpool3d.argtypes = [_VP, _VP, _VP, _VP, _VP, ctypes.c_int, ctypes.c_int, _VP, _VP]
        L.aps_ct3d_scale_pool_bias_out_shape.argtypes = [_VP, ctypes.c_int64, _VP, _VP, _VP, _VP,
                                                         _VP, ctypes.c_int, _VP]
        L.aps_ct3d_scale_pool_bias.argtypes = [_VP, _VP, _VP, _VP, _VP, ctypes.c_int64, _VP, _VP,
                                               _VP, _VP, _VP, ctypes.c_int, ctypes.c_float,
                                               ctypes.c_float, _VP, _VP]
        L.aps_convtranspose3d_out_shape.argtypes = [_VP, ctypes.c_int64, _VP, _VP, _VP, _VP, _VP,
                                                    _VP]
        L.aps_convtranspose3d.argtypes = [_VP, _VP, _VP, _VP, ctypes.c_int64, _VP, _VP, _VP, _VP,
                                          _VP, _VP, _VP]
        L.aps_convtranspose1d_out_shape.argtypes = [_VP, ctypes.c_int64] + [ctypes.c_int] * 5 + [_VP]
        L.aps_convtranspose1d.argtypes = [_VP, _VP, _VP, _VP, ctypes.c_int64] + \
            [ctypes.c_int] * 6 + [_VP, _VP]
        L.aps_device_status.argtypes = [ctypes.POINTER(ctypes.c_uint), ctypes.c_int]
        L.aps_fp32_fma_probe.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, _VP, _VP]
        L.aps_debug_fail_launches.argtypes = [ctypes.c_int]
        L.aps_debug_fail_launches.restype = None
        L.aps_debug_stall_next_pool.argtypes = [ctypes.c_ulonglong]
        L.aps_debug_stall_next_pool.restype = None
        L.aps_debug_skip_tensor_cores.argtypes = [ctypes.c_int]
        L.aps_debug_skip_tensor_cores.restype = None
        for name in EXPORTS:
            if name not in ("aps_status_string", "aps_abi_version", "aps_debug_fail_launches",
                            "aps_debug_stall_next_pool", "aps_debug_skip_tensor_cores"):
                getattr(L, name).restype = ctypes.c_int
        _lib = L
    return _lib


def status_string(status: int) -> str:
    try:
        return lib().aps_status_string(int(status)).decode()
    except RuntimeError:
        return f"status {status}"


def _i3(v):
    v = list(v) if hasattr(v, "__len__") else [v] * 3
    if len(v) != 3:
        raise ValueError("expected 3 values")
    return _I32_3(*[int(t) for t in v])


# ------------------------------------------------------------- raw ABI mirror
def aps_abi_version() -> int:
    return lib().aps_abi_version()


def aps_avgpool3d_out_shape(in_ncdhw, k, stride, pad, ceil_mode=0):
    out = _I64_5()
    st = lib().aps_avgpool3d_out_shape(_I64_5(*in_ncdhw), _i3(k), _i3(stride), _i3(pad),
                                       int(ceil_mode), out)
    return st, tuple(out)


def aps_avgpool3d(x_ptr, in_ncdhw, k, stride, pad, count_include_pad, ceil_mode, y_ptr,
                  stream=0) -> int:
    return lib().aps_avgpool3d(_VP(x_ptr), _I64_5(*in_ncdhw), _i3(k), _i3(stride), _i3(pad),
                               int(count_include_pad), int(ceil_mode), _VP(y_ptr), _VP(stream))


def aps_ct3d_scale_pool_bias_out_shape(in_ncdhw, c_out, k, stride, pad, out_pad, dil, pool_k):
    out = _I64_5()
    st = lib().aps_ct3d_scale_pool_bias_out_shape(_I64_5(*in_ncdhw), int(c_out), _i3(k),
                                                  _i3(stride), _i3(pad), _i3(out_pad),
                                                  _i3(dil), int(pool_k), out)
    return st, tuple(out)


def aps_ct3d_scale_pool_bias(x_ptr, in_ncdhw, w_ptr, conv_bias_ptr, bias_ptr, c_out, k, stride,
                             pad, out_pad, dil, pool_k, scale1, scale2, y_ptr, stream=0) -> int:
    return lib().aps_ct3d_scale_pool_bias(
        _VP(x_ptr), _I64_5(*in_ncdhw), _VP(w_ptr), _VP(conv_bias_ptr), _VP(bias_ptr),
        int(c_out), _i3(k), _i3(stride), _i3(pad), _i3(out_pad), _i3(dil), int(pool_k),
        float(scale1), float(scale2), _VP(y_ptr), _VP(stream))


def aps_convtranspose3d_out_shape(in_ncdhw, c_out, k, stride, pad, dil, out_pad):
    out = _I64_5()
    st = lib().aps_convtranspose3d_out_shape(_I64_5(*in_ncdhw), int(c_out), _i3(k), _i3(stride),
                                             _i3(pad), _i3(dil), _i3(out_pad), out)
    return st, tuple(out)


def aps_convtranspose3d(x_ptr, in_ncdhw, w_ptr, bias_ptr, c_out, k, stride, pad, dil, out_pad,
                        y_ptr, stream=0) -> int:
    return lib().aps_convtranspose3d(_VP(x_ptr), _I64_5(*in_ncdhw), _VP(w_ptr), _VP(bias_ptr),
                                     int(c_out), _i3(k), _i3(stride), _i3(pad), _i3(dil),
                                     _i3(out_pad), _VP(y_ptr), _VP(stream))


def aps_convtranspose1d_out_shape(in_ncl, c_out, k, stride, pad, dil, out_pad):
    out = _I64_3()
    st = lib().aps_convtranspose1d_out_shape(_I64_3(*in_ncl), int(c_out), int(k), int(stride),
                                             int(pad), int(dil), int(out_pad), out)
    return st, tuple(out)


def aps_convtranspose1d(x_ptr, in_ncl, w_ptr, bias_ptr, c_out, k, stride, pad, dil, out_pad,
                        precision, y_ptr, stream=0) -> int:
    return lib().aps_convtranspose1d(_VP(x_ptr), _I64_3(*in_ncl), _VP(w_ptr), _VP(bias_ptr),
                                     int(c_out), int(k), int(stride), int(pad), int(dil),
                                     int(out_pad), int(precision), _VP(y_ptr), _VP(stream))


def aps_device_status(clear: bool = False):
    bits = ctypes.c_uint(0)
    st = lib().aps_device_status(ctypes.byref(bits), int(bool(clear)))
    return st, bits.value


# --------------------------------------------------------- torch-level calls
APS_PROBE_THREADS = 256


def aps_debug_fail_launches(n: int) -> None:
    """Test hook: the next n launches report APS_ERR_LAUNCH (the kernels still run)."""
    lib().aps_debug_fail_launches(int(n))


def aps_debug_stall_next_pool(wait_limit_ns: int) -> None:
    """Test hook: the next TMA-path avgpool launch withholds one input box and its
    waits give up after wait_limit_ns (0 clears)."""
    lib().aps_debug_stall_next_pool(int(wait_limit_ns))


def aps_debug_skip_tensor_cores(on: bool) -> None:
    """Test hook: while on, every op passes over its tensor-core kernels (its FP32-pipe
    fallbacks run; explicit tf32 / 3xTF32 ConvTranspose1d requests are refused)."""
    lib().aps_debug_skip_tensor_cores(int(bool(on)))


def aps_fp32_fma_probe(packed, blocks, iters, sink_ptr, stream=0) -> int:
    return lib().aps_fp32_fma_probe(int(bool(packed)), int(blocks), int(iters), _VP(sink_ptr),
                                    _VP(stream))


def _stream(stream):
    import torch
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _check_tensor(t, name):
    import torch
    if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dtype != torch.float32:
        raise TypeError(f"{name} must be a CUDA float32 tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _ptr(t):
    return 0 if t is None else t.data_ptr()


def avgpool3d(x, kernel_size=3, stride=2, padding=1, count_include_pad=True, ceil_mode=False,
              out=None, stream=None):
    import torch
    _check_tensor(x, "x")
    st, oshape = aps_avgpool3d_out_shape(x.shape, kernel_size, stride, padding, ceil_mode)
    if st != APS_OK:
        raise ApsError(st, "aps_avgpool3d_out_shape")
    y = out if out is not None else torch.empty(oshape, device=x.device, dtype=torch.float32)
    _check_tensor(y, "out")
    if tuple(y.shape) != oshape:
        raise ValueError(f"out has shape {tuple(y.shape)}, expected {oshape}")
    st = aps_avgpool3d(x.data_ptr(), x.shape, kernel_size, stride, padding,
                       int(bool(count_include_pad)), int(bool(ceil_mode)), y.data_ptr(),
                       _stream(stream))
    if st != APS_OK:
        raise ApsError(st, "aps_avgpool3d")
    return y


def ct3d_scale_pool_bias(x, weight, conv_bias, bias, stride=2, padding=1, output_padding=0,
                         dilation=1, pool_k=2, scale1=0.5, scale2=1.0, out=None, stream=None):
    import torch
    _check_tensor(x, "x")
    _check_tensor(weight, "weight")
    _check_tensor(bias, "bias")
    if conv_bias is not None:
        _check_tensor(conv_bias, "conv_bias")
    if x.dim() != 5 or weight.dim() != 5:
        raise ValueError("x and weight must be 5-D")
    c_out = weight.shape[1]
    k = tuple(weight.shape[2:])
    st, oshape = aps_ct3d_scale_pool_bias_out_shape(x.shape, c_out, k, stride, padding,
                                                    output_padding, dilation, pool_k)
    if st != APS_OK:
        raise ApsError(st, "aps_ct3d_scale_pool_bias_out_shape")
    if weight.shape[0] != x.shape[1] or bias.numel() != c_out or (
            conv_bias is not None and conv_bias.numel() != c_out):
        raise ValueError("weight / bias shapes do not match x and C_out")
    y = out if out is not None else torch.empty(oshape, device=x.device, dtype=torch.float32)
    _check_tensor(y, "out")
    if tuple(y.shape) != oshape:
        raise ValueError(f"out has shape {tuple(y.shape)}, expected {oshape}")
    st = aps_ct3d_scale_pool_bias(x.data_ptr(), x.shape, weight.data_ptr(), _ptr(conv_bias),
                                  bias.data_ptr(), c_out, k, stride, padding, output_padding,
                                  dilation, pool_k, scale1, scale2, y.data_ptr(), _stream(stream))
    if st != APS_OK:
        raise ApsError(st, "aps_ct3d_scale_pool_bias")
    return y


def convtranspose3d(x, weight, bias=None, stride=2, padding=1, dilation=1, output_padding=0,
                    out=None, stream=None):
    """ConvTranspose3d on device tensors through the C ABI; returns (or fills)
    y [N, C_out, Do, Ho, Wo]."""
    import torch
    _check_tensor(x, "x")
    _check_tensor(weight, "weight")
    if bias is not None:
        _check_tensor(bias, "bias")
    if x.dim() != 5 or weight.dim() != 5:
        raise ValueError("x and weight must be 5-D")
    c_out = weight.shape[1]
    k = tuple(weight.shape[2:])
    st, oshape = aps_convtranspose3d_out_shape(x.shape, c_out, k, stride, padding, dilation,
                                               output_padding)
    if st != APS_OK:
        raise ApsError(st, "aps_convtranspose3d_out_shape")
    if weight.shape[0] != x.shape[1] or (bias is not None and bias.numel() != c_out):
        raise ValueError("weight / bias shapes do not match x and C_out")
    y = out if out is not None else torch.empty(oshape, device=x.device, dtype=torch.float32)
    _check_tensor(y, "out")
    if tuple(y.shape) != oshape:
        raise ValueError(f"out has shape {tuple(y.shape)}, expected {oshape}")
    st = aps_convtranspose3d(x.data_ptr(), x.shape, weight.data_ptr(), _ptr(bias), c_out, k,
                             stride, padding, dilation, output_padding, y.data_ptr(),
                             _stream(stream))
    if st != APS_OK:
        raise ApsError(st, "aps_convtranspose3d")
    return y


def convtranspose1d(x, weight, bias=None, stride=1, padding=0, dilation=1, output_padding=0,
                    precision=APS_PREC_FP32, out=None, stream=None):
    import torch
    _check_tensor(x, "x")
    _check_tensor(weight, "weight")
    if bias is not None:
        _check_tensor(bias, "bias")
    if x.dim() != 3 or weight.dim() != 3:
        raise ValueError("x and weight must be 3-D")
    c_out, k = weight.shape[1], weight.shape[2]
    st, oshape = aps_convtranspose1d_out_shape(x.shape, c_out, k, stride, padding, dilation,
                                               output_padding)
    if st != APS_OK:
        raise ApsError(st, "aps_convtranspose1d_out_shape")
    if weight.shape[0] != x.shape[1] or (bias is not None and bias.numel() != c_out):
        raise ValueError("weight / bias shapes do not match x and C_out")
    y = out if out is not None else torch.empty(oshape, device=x.device, dtype=torch.float32)
    _check_tensor(y, "out")
    if tuple(y.shape) != oshape:
        raise ValueError(f"out has shape {tuple(y.shape)}, expected {oshape}")
    st = aps_convtranspose1d(x.data_ptr(), x.shape, weight.data_ptr(), _ptr(bias), c_out, k,
                             stride, padding, dilation, output_padding, precision, y.data_ptr(),
                             _stream(stream))
    if st != APS_OK:
        raise ApsError(st, "aps_convtranspose1d")
    return y
