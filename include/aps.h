/*
 * aps.h -- C ABI of the average_pooling_stencil GB300 library (libaps.so).
 *
 * Three fp32 stencil ops on contiguous NC(D)HW / NCL tensors, and the
 * standalone transposed convolution of the first (aps_convtranspose3d, the
 * pre-pool tensor of the page's unfused chain), each computed by hand-written
 * CUDA kernels for sm_103a:
 *
 *   aps_ct3d_scale_pool_bias  ConvTranspose3d -> x scale1 -> AvgPool3d(pool_k)
 *                             -> + bias[c] -> x scale2, fused so that the
 *                             pre-pool tensor is never written
 *                             (page Kimi-K2.6__l2_p50, the fused model and its
 *                             27-term / 8-neighbour decomposition).
 *   aps_avgpool3d             AvgPool3d with zero padding
 *                             (page Kimi-K2.6__l1_p46: kernel 3, stride 2,
 *                             padding 1, count_include_pad, divisor 27).
 *   aps_convtranspose1d       ConvTranspose1d with stride, padding, dilation
 *                             and output padding
 *                             (page Kimi-K2.6__l1_p74: the gather formula
 *                             y[o] = sum_k x[(o + p - d*k)/s] * w[k], taken only
 *                             where the quotient is an integer in range).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Tensors are fp32, dense, C-contiguous.  Activations are [N, C, D, H, W]
 *    (3-D) or [N, C, L] (1-D).  Transposed-convolution weights are
 *    [C_in, C_out, k...] (the PyTorch ConvTranspose layout); biases are [C_out].
 *  - Shapes are passed as int64 arrays; kernel sizes, strides, paddings,
 *    dilations and output paddings as int arrays (one entry per spatial dim).
 *  - Output sizes: transposed convolution (L - 1)*s - 2p + d*(k - 1) + op + 1;
 *    pooling floor((L + 2p - k)/s) + 1 (ceil mode: ceil instead of floor, and a
 *    last window that would start inside the right padding is dropped).
 *  - All tensor pointers are DEVICE pointers on the current CUDA device.  The
 *    caller owns all memory: the library never allocates, frees or
 *    synchronises.  Outputs must not overlap inputs.  Pointers must be at
 *    least 4-byte aligned; 16-byte alignment (plus the shape conditions stated
 *    per op) selects the fastest kernels, never changes results beyond the
 *    stated tolerance, and is not required.
 *  - Launches are asynchronous and ordered on `stream` (a cudaStream_t; NULL is
 *    the legacy default stream).  A status other than APS_OK means nothing
 *    was launched, except APS_ERR_LAUNCH, which reports the error the CUDA
 *    runtime gave for the launch itself.  A tensor with zero elements (N or C
 *    equal to 0) is valid: the call returns APS_OK and launches nothing.
 *    The convolution ops launch their kernel as a programmatic dependent of
 *    the work before it on `stream` (its launch and on-chip set-up overlap
 *    that work's tail; it touches no global memory until that work has
 *    completed), so stream order holds exactly as for a plain launch.
 *  - Shape queries are pure host functions; they need no GPU and no CUDA
 *    context.
 *  - Size limits of the launches (the shape queries accept larger shapes):
 *    every channel count and every spatial size of the input and of the
 *    output must be below 2^30 (for aps_ct3d_scale_pool_bias also pool_k
 *    times each pooled size), and for aps_avgpool3d the product of the three
 *    output spatial sizes below 2^31.  A larger request with elements returns
 *    APS_ERR_UNSUPPORTED before any CUDA call; within them every valid
 *    request runs (at APS_PREC_FP32 for aps_convtranspose1d).
 *  - Kernels contain no unbounded waits.  A pipeline wait that exceeds its
 *    time limit makes the kernel stop early and record APS_DEVERR_TIMEOUT in a
 *    per-device status word read by aps_device_status().
 */
#ifndef APS_H
#define APS_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t, declared without CUDA headers. */
struct CUstream_st;
typedef struct CUstream_st *aps_stream_t;

typedef enum {
    APS_OK = 0,
    APS_ERR_NULL = -1,        /* a shape array, or the data pointer of an array
                                 with elements, is NULL (a pointer to an array of
                                 zero elements may be NULL: nothing touches it) */
    APS_ERR_SHAPE = -2,       /* a dimension or parameter is out of range, or
                                 the output would be empty in a spatial dim */
    APS_ERR_UNSUPPORTED = -3, /* a valid request no kernel here implements */
    APS_ERR_ALIGN = -4,       /* a tensor pointer is not 4-byte aligned */
    APS_ERR_LAUNCH = -5,      /* the CUDA runtime rejected the launch */
    APS_ERR_CUDA = -6         /* another CUDA runtime call failed */
} aps_status;

/* Bits of the per-device status word (see aps_device_status). */
#define APS_DEVERR_TIMEOUT 1u

/* Precision choices of aps_convtranspose1d. */
#define APS_PREC_FP32 0   /* fp32 accuracy: max |y - exact| <= 1e-5 * (1 + |exact|);
                             runs as APS_PREC_TF32X3 where that form accepts the shape
                             (3-4x the speed at the same bound), else as
                             APS_PREC_FP32_FMA */
#define APS_PREC_TF32 1   /* tcgen05 tensor cores, tf32 operands, fp32 accumulate;
                             ||y - exact||_F <= 5e-3 * ||exact||_F */
#define APS_PREC_TF32X3 2 /* tensor cores, each operand split v = hi + lo (tf32) and
                             each product summed as lo*hi + hi*lo + hi*hi (3xTF32);
                             max |y - exact| <= 1e-5 * (1 + |exact|), as fp32 */
#define APS_PREC_FP32_FMA 3 /* fp32 FMAs on the FP32 pipe only (no tensor cores);
                               max |y - exact| <= 1e-5 * (1 + |exact|) */

/* Version of this ABI (bumped on any incompatible change). */
int aps_abi_version(void);

/* Human-readable name of a status code (static string, never NULL). */
const char *aps_status_string(int status);

/* ---------------------------------------------------------------- avgpool3d
 * y[n,c,i,j,l] = (1/div) * sum over the kD x kH x kW window starting at
 * (i*sD - pD, j*sH - pH, l*sW - pW) of x, cells outside the input counting as
 * zero.  div = kD*kH*kW when count_include_pad is non-zero (the window clipped
 * at the end of the right padding in ceil mode), otherwise the number of
 * window cells inside the input.  Kimi-K2.6__l1_p46 fixes k = 3, s = 2, p = 1,
 * count_include_pad, floor mode, where the divisor is always 27.
 *
 * x: [N, C, D, H, W] device fp32.  y: [N, C, Do, Ho, Wo] device fp32 (shape
 * from aps_avgpool3d_out_shape).  Requires k >= 1, s >= 1, 0 <= 2p <= k.
 * Fast path: k = 3, s = 2, p = 1 in all dims, floor mode, count_include_pad
 * on or off, W % 4 == 0, x 16-byte and y 8-byte aligned (TMA-tiled kernel).
 * k = 2, s = 2, p = 0 with whole windows, W % 4 == 0, x 16-byte and y 8-byte
 * aligned: a vectorised kernel (two outputs per thread).  Other cubic windows
 * of 2 or 3: an unrolled window kernel; every other valid request: a
 * direct-window kernel.
 */
aps_status aps_avgpool3d_out_shape(const int64_t in_ncdhw[5], const int k[3],
                                   const int stride[3], const int pad[3],
                                   int ceil_mode, int64_t out_ncdhw[5]);

aps_status aps_avgpool3d(const float *x, const int64_t in_ncdhw[5], const int k[3],
                         const int stride[3], const int pad[3], int count_include_pad,
                         int ceil_mode, float *y, aps_stream_t stream);

/* ----------------------------------------------------- ct3d_scale_pool_bias
 * y = ((AvgPool3d_q(convT3d(x, w) + conv_bias) * scale1) + bias[c]) * scale2,
 * written in the order of Kimi-K2.6__l2_p50's model: transposed convolution
 * with conv_bias, multiply by scale1, average pool with kernel = stride =
 * pool_k (no padding, floor mode), add bias[c], multiply by scale2.  Only the
 * pooled result is written.
 *
 * x: [N, C_in, D, H, W]; w: [C_in, C_out, kD, kH, kW]; conv_bias: [C_out] or
 * NULL (treated as zeros); bias: [C_out]; y: [N, C_out, Do, Ho, Wo] (shape from
 * aps_ct3d_scale_pool_bias_out_shape).  Requires k, s, dil >= 1, pad >= 0,
 * 0 <= out_pad < max(s, dil), pool_k >= 1.
 * Fast path: k = 3, s = 2, p = 1, out_pad 0 or 1 (per dim), dil = 1, pool_k = 2,
 * C_out = 16, 1 <= C_in <= 8: the pooled output then equals a 2x2x2 correlation of x
 * (zero past the input's end, which only the last pooled position of a dim with
 * out_pad 1 reaches) with 8 collapsed weights per (ci, co) plus a folded bias (the page's
 * grouping of the 27 taps by input neighbour), computed in one kernel whose
 * CTAs collapse the weights themselves.  With W % 4 == 0 and x 16-byte
 * aligned that kernel runs the correlation on the tensor cores as 3xTF32
 * (each operand split v = hi + lo, each product summed as lo*hi + hi*lo +
 * hi*hi in fp32; C_in 4..8 in chunks of up to 3 input channels); otherwise,
 * or where the tensor-core kernel cannot be made resident, on the FP32 pipe.
 * Both meet
 * max |y - exact| <= 1e-5 * (1 + |exact|).  Every other valid geometry runs on
 * per-phase collapsed weights while its per-dim phase tables fit (at most 8
 * phases and 8 input offsets per phase per dim, at most 32 taps per dim, at
 * most 96 KB of collapsed weights), else on a direct per-output kernel.
 */
aps_status aps_ct3d_scale_pool_bias_out_shape(const int64_t in_ncdhw[5], int64_t c_out,
                                              const int k[3], const int stride[3],
                                              const int pad[3], const int out_pad[3],
                                              const int dil[3], int pool_k,
                                              int64_t out_ncdhw[5]);

aps_status aps_ct3d_scale_pool_bias(const float *x, const int64_t in_ncdhw[5],
                                    const float *w, const float *conv_bias,
                                    const float *bias, int64_t c_out, const int k[3],
                                    const int stride[3], const int pad[3],
                                    const int out_pad[3], const int dil[3], int pool_k,
                                    float scale1, float scale2, float *y,
                                    aps_stream_t stream);

/* -------------------------------------------------------- convtranspose3d
 * The transposed convolution alone, emitting the full-resolution tensor (the
 * first stage of Kimi-K2.6__l2_p50's unfused chain, "approach 1" there):
 *   y[n,co,o] = bias[co] + sum_ci sum_k w[ci,co,k] * x[n,ci,(o + p - d*k)/s],
 * per spatial dim a term existing only where o + p - d*k is a non-negative
 * multiple of s whose quotient is inside the input; weights are not flipped.
 *
 * x: [N, C_in, D, H, W]; w: [C_in, C_out, kD, kH, kW]; bias: [C_out] or NULL
 * (no bias); y: [N, C_out, Do, Ho, Wo] with O = (I-1)*s - 2p + d*(k-1) + op + 1
 * (shape from aps_convtranspose3d_out_shape).  Requires k, s, d >= 1,
 * p >= 0, 0 <= out_pad < max(s, d).
 * Fast path: k = 3, s = 2, p = 1, d = 1 in all dims (out_pad 0 or 1),
 * C_out = 16, 1 <= C_in <= 8, W % 4 == 0 and x 16-byte aligned (per-parity
 * tap sets, TMA-staged input): on the tensor cores as 3xTF32 (each operand
 * split v = hi + lo, each product summed as lo*hi + hi*lo + hi*hi in fp32),
 * meeting max |y - exact| <= 1e-5 * (1 + |exact|).  Every other valid
 * request, and a fast-path one whose tensor-core kernel cannot be made
 * resident (shared memory or tensor memory unavailable), runs a direct
 * per-output kernel on the FP32 pipe at the same bound.
 */
aps_status aps_convtranspose3d_out_shape(const int64_t in_ncdhw[5], int64_t c_out,
                                         const int k[3], const int stride[3],
                                         const int pad[3], const int dil[3],
                                         const int out_pad[3], int64_t out_ncdhw[5]);

aps_status aps_convtranspose3d(const float *x, const int64_t in_ncdhw[5], const float *w,
                               const float *bias, int64_t c_out, const int k[3],
                               const int stride[3], const int pad[3], const int dil[3],
                               const int out_pad[3], float *y, aps_stream_t stream);

/* -------------------------------------------------------- convtranspose1d
 * y[n,co,o] = bias[co] + sum_ci sum_k w[ci,co,k] * x[n,ci,(o + p - d*k)/s], each
 * term taken only when o + p - d*k is a multiple of s and the quotient lies in
 * [0, L) (Kimi-K2.6__l1_p74's gather formula; weights are NOT flipped).
 *
 * x: [N, C_in, L]; w: [C_in, C_out, K]; bias: [C_out] or NULL (no bias);
 * y: [N, C_out, L_out] (shape from aps_convtranspose1d_out_shape).  Requires
 * K, s, d >= 1, p >= 0, 0 <= out_pad < max(s, d).  precision: APS_PREC_FP32,
 * APS_PREC_TF32, APS_PREC_TF32X3 or APS_PREC_FP32_FMA (tolerances above).  The
 * two explicit tensor-core precisions return APS_ERR_UNSUPPORTED
 * (nothing launched) unless: C_in % 8 == 0 and, above 32, C_in % 32 == 0;
 * C_out % 32 == 0 and (number of output residues mod s that some tap reaches)
 * x C_out <= 256; L % 4 == 0 and x 16-byte aligned; s <= 8, at most 4
 * reached residues with at most 8 taps each; the tap span d*(K-1)/s <= 124;
 * K * C_in <= 2048 (the per-tile MMA descriptor table);
 * and the weights (K*C_in*C_out*4 bytes, twice that for APS_PREC_TF32X3, which
 * also holds two copies of each converted stage and may stage 16 channels at a
 * time) plus the staging buffers fit in one CTA's 227 KB of shared memory.
 * APS_PREC_FP32 and APS_PREC_FP32_FMA accept every valid shape within the size
 * limits above.
 */
aps_status aps_convtranspose1d_out_shape(const int64_t in_ncl[3], int64_t c_out, int k,
                                         int stride, int pad, int dil, int out_pad,
                                         int64_t out_ncl[3]);

aps_status aps_convtranspose1d(const float *x, const int64_t in_ncl[3], const float *w,
                               const float *bias, int64_t c_out, int k, int stride,
                               int pad, int dil, int out_pad, int precision, float *y,
                               aps_stream_t stream);

/* ------------------------------------------------------------ diagnostics
 * Reads (and, if clear != 0, resets) the status word of the current device:
 * a bitwise OR of APS_DEVERR_* recorded by kernels since the last reset.
 * Synchronous: it waits for all prior work on the device, then reads and
 * clears the word in one atomic step on the GPU (a one-thread kernel on the
 * legacy default stream), so a bit that a kernel still running on another
 * stream sets meanwhile is reported by this call or the next, never lost.
 */
aps_status aps_device_status(unsigned int *bits, int clear);

/* FP32 FMA-rate probe (not part of any op): launches `blocks` CTAs of
 * APS_PROBE_THREADS threads, each thread running `iters` rounds of 32
 * independent fp32 multiply-adds on registers -- scalar FMA, or (packed != 0)
 * the packed fp32x2 FMA in 16 pairs.  FLOPs per launch =
 * 64 * iters * blocks * APS_PROBE_THREADS.  The caller times the launch on
 * `stream`; sink (one device float) is written only under a condition that
 * never holds.  Returns APS_ERR_NULL without sink, APS_ERR_SHAPE for
 * blocks < 1 or iters < 1.  Asynchronous, allocates nothing. */
#define APS_PROBE_THREADS 256
aps_status aps_fp32_fma_probe(int packed, int blocks, int iters, float *sink,
                              aps_stream_t stream);

/* Test hook for the error path (not part of any op): the next n kernel
 * launches of this process report APS_ERR_LAUNCH, as if the CUDA runtime had
 * rejected them, although the kernels still run; n <= 0 clears it.  Lets a
 * test check that every entry point returns the launch status and that
 * callers see it.  Host-only, thread-safe. */
void aps_debug_fail_launches(int n);

/* Test hook for the fallback kernels (not part of any op): while on != 0,
 * every entry point passes over its tensor-core kernels, as if they could not
 * be made resident on this device -- the fused op and aps_convtranspose3d then
 * run their FP32-pipe kernels, aps_convtranspose1d with APS_PREC_FP32 runs as
 * APS_PREC_FP32_FMA, and APS_PREC_TF32 / APS_PREC_TF32X3 return
 * APS_ERR_UNSUPPORTED.  Results stay within each op's stated bound.  Lets a
 * test reach the fallbacks on shapes the tensor cores take.  Host-only,
 * process-wide, thread-safe; on = 0 restores the normal dispatch. */
void aps_debug_skip_tensor_cores(int on);

/* Test hook for a wait that runs out (not part of any op): the next
 * aps_avgpool3d launch that takes the TMA-tiled kernel withholds the first
 * input box of its first CTA -- the box's barrier still expects its bytes --
 * and every pipeline wait of that launch gives up after wait_limit_ns instead
 * of the usual 2 s.  The consumers of that CTA then record APS_DEVERR_TIMEOUT
 * in the status word and return; its producer waits (bounded) for the boxes it
 * did issue and returns; the other CTAs finish normally, and the CUDA context
 * stays usable.  wait_limit_ns = 0 clears a pending stall.  Host-only,
 * thread-safe; the CTA's outputs of that launch are left unwritten. */
void aps_debug_stall_next_pool(unsigned long long wait_limit_ns);

#ifdef __cplusplus
}
#endif

#endif /* APS_H */
