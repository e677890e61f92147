"""GB300-native (sm_103a) CUDA library for three fp32 stencil ops:
fused ConvTranspose3d -> scale -> AvgPool3d -> bias -> scale, AvgPool3d, and
ConvTranspose1d.  The kernels and the C ABI live in csrc/ and include/aps.h;
``binding`` is the ctypes layer.  Importing the package loads nothing; the
library is loaded (and must have been built) on first use.
"""
from .binding import (APS_OK, APS_PREC_FP32, APS_PREC_TF32, ApsError, avgpool3d,  # noqa: F401
                      convtranspose1d, ct3d_scale_pool_bias)

__all__ = ["avgpool3d", "ct3d_scale_pool_bias", "convtranspose1d", "ApsError",
           "APS_OK", "APS_PREC_FP32", "APS_PREC_TF32"]
