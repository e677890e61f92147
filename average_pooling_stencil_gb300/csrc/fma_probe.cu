// fma_probe.cu -- diagnostic: the FP32 FMA rate this GPU sustains, for the
// roofline of the FMA-bound kernels.  Every thread runs `iters` rounds of 32
// independent fp32 multiply-adds on registers (scalar fmaf, or the packed
// fp32x2 form in 16 pairs); nothing is loaded, and the result is written only
// under a condition that never holds, so the time is the FMA pipe's alone.  The
// caller times the launch (CUDA events on `stream`); FLOPs per launch =
// 2 * 32 * iters * threads, threads = blocks * APS_PROBE_THREADS.
#include "aps_dev.cuh"
#include "aps_internal.h"

namespace aps {
namespace fp {
constexpr int THREADS = 256;
constexpr int CHAINS = 32;   // independent fp32 accumulators per thread
}  // namespace fp

__global__ void __launch_bounds__(fp::THREADS)
    fma_probe_scalar_kernel(float *sink, int iters, float a, float b) {
    float acc[fp::CHAINS];
#pragma unroll
    for (int i = 0; i < fp::CHAINS; ++i) acc[i] = threadIdx.x * 1e-3f + i;
#pragma unroll 1
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int i = 0; i < fp::CHAINS; ++i) acc[i] = fmaf(acc[i], a, b);
    }
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < fp::CHAINS; ++i) s += acc[i];
    if (s == 1.2345e-30f) sink[0] = s;   // never true: keeps the chains alive
}

__global__ void __launch_bounds__(fp::THREADS)
    fma_probe_packed_kernel(float *sink, int iters, float a, float b) {
    float2 acc[fp::CHAINS / 2];
#pragma unroll
    for (int i = 0; i < fp::CHAINS / 2; ++i) acc[i] = make_float2(threadIdx.x * 1e-3f + i, 0.5f * i);
    const float2 a2 = make_float2(a, a), b2 = make_float2(b, b);
#pragma unroll 1
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int i = 0; i < fp::CHAINS / 2; ++i) acc[i] = __ffma2_rn(acc[i], a2, b2);
    }
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < fp::CHAINS / 2; ++i) s += acc[i].x + acc[i].y;
    if (s == 1.2345e-30f) sink[0] = s;
}

}  // namespace aps

extern "C" aps_status aps_fp32_fma_probe(int packed, int blocks, int iters, float *sink,
                                         aps_stream_t stream) {
    using namespace aps;
    if (!sink) return APS_ERR_NULL;
    if (blocks < 1 || iters < 1 || blocks > (1 << 24)) return APS_ERR_SHAPE;
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    const cudaError_t e =
        packed ? launch_plain(fma_probe_packed_kernel, dim3(blocks), dim3(fp::THREADS), 0, cs,
                              sink, iters, 0.999f, 1e-3f)
               : launch_plain(fma_probe_scalar_kernel, dim3(blocks), dim3(fp::THREADS), 0, cs,
                              sink, iters, 0.999f, 1e-3f);
    return launch_status(e);
}
