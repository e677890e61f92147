// aps_internal.h -- host-side declarations shared by the library's translation
// units (not part of the public ABI).
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>   // PFN_cuTensorMapEncodeTiled (type only)
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/aps.h"

namespace aps {

// Device address of the current device's status word (see aps_device_status).
unsigned int *status_word();

// Number of SMs of the current device (cached per device).
int sm_count();

// Resident CTAs per SM of `func` at `threads` threads and `smem` bytes of
// dynamic shared memory on the current device; raises the kernel's dynamic
// shared-memory limit to `smem` first.  Cached per (device, kernel, config).
// Returns 0 if the attribute cannot be set.
int resident_ctas(const void *func, int threads, int smem);

// cuTensorMapEncodeTiled obtained through the runtime's driver entry point
// (no link-time dependency on libcuda).  Returns false if unavailable.
bool encode_tiled(CUtensorMap *map, CUtensorMapDataType type, uint32_t rank, void *base,
                  const cuuint64_t *dims, const cuuint64_t *strides_bytes,
                  const cuuint32_t *box, const cuuint32_t *elem_strides);

// Maps the launch's own result to APS_OK / APS_ERR_LAUNCH.  A failed launch's
// error is also taken off the runtime's last-error slot, so that the caller's
// next cudaGetLastError does not report it again; a successful launch leaves
// that slot (and any error the caller left in it) untouched.
aps_status launch_status(cudaError_t launch_result);

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Opt-in dynamic shared memory of one CTA on sm_103a (bytes).
constexpr size_t kMaxSmemPerCta = 227 * 1024;

// Launches `kern` on `st` as a programmatic dependent of the kernel before it
// on the stream (the kernel calls pdl_wait before touching global memory), so
// that its launch and on-chip setup overlap the previous kernel's tail.
// Returns the runtime's result for the launch itself.
template <typename... P, typename... A>
inline cudaError_t launch_pdl(void (*kern)(P...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t st, A &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<P>(args)...);
}

// Plain launch (no programmatic dependency); returns the launch's own result.
template <typename... P, typename... A>
inline cudaError_t launch_plain(void (*kern)(P...), dim3 grid, dim3 block, size_t smem,
                                cudaStream_t st, A &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cfg.attrs = nullptr;
    cfg.numAttrs = 0;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<P>(args)...);
}

// ------------------------------------------------------------ launchers
// Each launcher assumes validated arguments and a non-empty output.

// AvgPool3d k3/s2/p1, floor mode, count_include_pad on or off; W % 4 == 0, x
// 16-byte and y 8-byte aligned.  Returns APS_ERR_UNSUPPORTED if the tensor map
// cannot be built (the caller then uses the direct kernel).
aps_status launch_avgpool3d_k3s2p1_tma(const float *x, const int64_t in[5], float *y,
                                       const int64_t out[5], int count_include_pad,
                                       cudaStream_t st);

aps_status launch_avgpool3d_direct(const float *x, const int64_t in[5], const int k[3],
                                   const int s[3], const int p[3], int count_include_pad,
                                   float *y, const int64_t out[5], cudaStream_t st);

// Fused transposed conv (k3 s2 p1, pool 2, C_out = 16, C_in <= 8).  Returns
// APS_ERR_UNSUPPORTED when the tile does not fit (the caller then uses the
// direct kernel).
aps_status launch_ct3d_pool2_fast(const float *x, const int64_t in[5], const float *w,
                                  const float *conv_bias, const float *bias, float scale1,
                                  float scale2, float *y, const int64_t out[5],
                                  cudaStream_t st);

// The same fused op on the tensor cores (3xTF32: fp32 accuracy), for
// C_in <= 3 and input rows of a multiple of 16 bytes; APS_ERR_UNSUPPORTED
// otherwise (the caller then uses launch_ct3d_pool2_fast).
aps_status launch_ct3d_pool2_tc(const float *x, const int64_t in[5], const float *w,
                                const float *conv_bias, const float *bias, float scale1,
                                float scale2, float *y, const int64_t out[5], cudaStream_t st);

// The fused op for any geometry whose per-dim phase tables fit (at most 8
// phases and 8 input offsets per phase per dim, kernels of at most 32 taps per
// dim, collapsed weights of at most 96 KB); APS_ERR_UNSUPPORTED otherwise (the
// caller then uses launch_ct3d_pool_direct).
aps_status launch_ct3d_pool_gen(const float *x, const int64_t in[5], const float *w,
                                const float *conv_bias, const float *bias, int64_t c_out,
                                const int k[3], const int s[3], const int p[3], const int d[3],
                                int pool_k, float scale1, float scale2, float *y,
                                const int64_t out[5], cudaStream_t st);

aps_status launch_ct3d_pool_direct(const float *x, const int64_t in[5], const float *w,
                                   const float *conv_bias, const float *bias, int64_t c_out,
                                   const int k[3], const int s[3], const int p[3],
                                   const int d[3], int pool_k, float scale1, float scale2,
                                   float *y, const int64_t out[5], cudaStream_t st);

// Standalone ConvTranspose3d k3 s2 p1 on the tensor cores (3xTF32: fp32
// accuracy) for C_in <= 8 and 16-byte input rows (W % 4 == 0; rows wider than 32
// in 32-column blocks); APS_ERR_UNSUPPORTED otherwise (the caller then uses
// launch_convt3d_direct).
aps_status launch_convt3d_tc(const float *x, const int64_t in[5], const float *w,
                             const float *bias, float *y, const int64_t out[5], cudaStream_t st);

// ConvTranspose3d, fp32, any geometry: one thread per output.
aps_status launch_convt3d_direct(const float *x, const int64_t in[5], const float *w,
                                 const float *bias, int64_t c_out, const int k[3],
                                 const int s[3], const int p[3], const int d[3], float *y,
                                 const int64_t out[5], cudaStream_t st);

// ConvTranspose1d, fp32.  The tiled kernel covers the (stride, taps,
// dilation, padding mod stride) combinations compiled in and C_out % 8 == 0;
// it returns APS_ERR_UNSUPPORTED otherwise.
aps_status launch_convt1d_tiled(const float *x, const int64_t in[3], const float *w,
                                const float *bias, int64_t c_out, int k, int s, int p,
                                int d, float *y, int64_t l_out, cudaStream_t st);

// ConvTranspose1d on the tensor cores (tf32 operands, fp32 accumulation).
// Needs C_in % 8 == 0 (and C_in % 32 == 0 above 32), C_out % 32 == 0,
// C_out <= 256, L % 4 == 0, x 16-byte aligned, at most 4 output classes with
// taps; returns APS_ERR_UNSUPPORTED otherwise.
aps_status launch_convt1d_tf32(const float *x, const int64_t in[3], const float *w,
                               const float *bias, int64_t c_out, int k, int s, int p, int d,
                               float *y, int64_t l_out, bool split, cudaStream_t st);

aps_status launch_convt1d_direct(const float *x, const int64_t in[3], const float *w,
                                 const float *bias, int64_t c_out, int k, int s, int p,
                                 int d, float *y, int64_t l_out, cudaStream_t st);

}  // namespace aps
