// convt3d.cu -- standalone ConvTranspose3d in fp32 for any geometry, emitting
// the full-resolution (pre-pool) tensor: the first stage of Kimi-K2.6__l2_p50's
// unfused chain ("approach 1" on that page, there done by the vendor library).
//
// Operation (the page's scatter definition, written as a gather):
//   y[n,co,o] = bias[co] + sum_ci sum_k w[ci,co,k] * x[n,ci,(o + p - d*k)/s]
// per spatial dim, a term existing only where o + p - d*k is a non-negative
// multiple of s whose quotient is inside the input.
//
// Which kernel runs: the k3 s2 p1 d1 geometry with C_out = 16, C_in <= 8 and
// 16-byte input rows takes the tensor-core kernel (convt3d_tc.cu).  This file
// holds the direct kernel for every other request: one thread per output
// evaluating the gather formula as written, for any (k, s, p, d,
// output_padding) and channel counts.
#include <algorithm>

#include "aps_dev.cuh"
#include "aps_internal.h"

namespace aps {
// ------------------------------------------------------------ direct kernel
__global__ void convt3d_direct_kernel(const float *__restrict__ x, const float *__restrict__ w,
                                      const float *__restrict__ bias, float *__restrict__ y,
                                      long long total, int Cin, int Cout, int D, int H, int W,
                                      int Do, int Ho, int Wo, int kd, int kh, int kw, int sd,
                                      int sh, int sw, int pd, int ph, int pw, int dd, int dh,
                                      int dw) {
    pdl_trigger();
    pdl_wait();
    for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        const int ow = (int)(idx % Wo);
        long long t = idx / Wo;
        const int oh = (int)(t % Ho);
        t /= Ho;
        const int od = (int)(t % Do);
        t /= Do;
        const int co = (int)(t % Cout);
        const long long n = t / Cout;
        float acc = bias ? __ldg(bias + co) : 0.f;
        for (int ci = 0; ci < Cin; ++ci) {
            const float *xp = x + (n * Cin + ci) * (long long)D * H * W;
            const float *wp = w + ((long long)ci * Cout + co) * kd * kh * kw;
            for (int a = 0; a < kd; ++a) {
                const long long nd = (long long)od + pd - (long long)a * dd;
                if (nd < 0 || nd % sd) continue;
                const long long id = nd / sd;
                if (id >= D) continue;
                for (int b = 0; b < kh; ++b) {
                    const long long nh = (long long)oh + ph - (long long)b * dh;
                    if (nh < 0 || nh % sh) continue;
                    const long long ih = nh / sh;
                    if (ih >= H) continue;
                    for (int c = 0; c < kw; ++c) {
                        const long long nw = (long long)ow + pw - (long long)c * dw;
                        if (nw < 0 || nw % sw) continue;
                        const long long iw = nw / sw;
                        if (iw >= W) continue;
                        acc = fmaf(__ldg(xp + (id * H + ih) * W + iw),
                                   __ldg(wp + (a * kh + b) * kw + c), acc);
                    }
                }
            }
        }
        y[idx] = acc;
    }
}

aps_status launch_convt3d_direct(const float *x, const int64_t in[5], const float *w,
                                 const float *bias, int64_t c_out, const int k[3],
                                 const int s[3], const int p[3], const int d[3], float *y,
                                 const int64_t out[5], cudaStream_t st) {
    for (int i = 2; i < 5; ++i)
        if (in[i] >= (1 << 30) || out[i] >= (1 << 30)) return APS_ERR_UNSUPPORTED;
    if (c_out >= (1 << 30) || in[1] >= (1 << 30)) return APS_ERR_UNSUPPORTED;
    const long long total = out[0] * out[1] * out[2] * out[3] * out[4];
    const int threads = 256;
    const long long blocks =
        std::min<long long>(ceil_div(total, threads), (long long)sm_count() * 16);
    const cudaError_t e = launch_pdl(convt3d_direct_kernel, dim3((unsigned)blocks), dim3(threads), 0, st, x, w, bias, y,
               total, (int)in[1], (int)c_out, (int)in[2], (int)in[3], (int)in[4], (int)out[2],
               (int)out[3], (int)out[4], k[0], k[1], k[2], s[0], s[1], s[2], p[0], p[1], p[2], d[0],
               d[1], d[2]);
    return launch_status(e);
}

}  // namespace aps
