"""GB300-native (sm_103a) CUDA library for fp32 stencil ops: fused
ConvTranspose3d -> scale -> AvgPool3d -> bias -> scale, AvgPool3d,
ConvTranspose1d, and the standalone ConvTranspose3d.  The kernels and the C ABI live in csrc/ and include/aps.h;
``binding`` is the ctypes layer.  Importing the package loads nothing; the
library is loaded (and must have been built) on first use.
"""
from .binding import (APS_OK, APS_PREC_FP32, APS_PREC_FP32_FMA, APS_PREC_TF32,  # noqa: F401
                      APS_PREC_TF32X3, ApsError, avgpool3d, convtranspose1d, convtranspose3d,
                      ct3d_scale_pool_bias)

__all__ = ["avgpool3d", "ct3d_scale_pool_bias", "convtranspose1d", "convtranspose3d",
           "ApsError", "APS_OK", "APS_PREC_FP32", "APS_PREC_TF32", "APS_PREC_TF32X3",
           "APS_PREC_FP32_FMA"]
