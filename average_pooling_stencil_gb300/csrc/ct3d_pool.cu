// ct3d_pool.cu -- fused ConvTranspose3d -> x scale1 -> AvgPool3d(pool_k) ->
// + bias -> x scale2 (the model of Kimi-K2.6__l2_p50).
//
// Fast path (k3, s2, p1, output_padding 0, dilation 1, pool 2, C_out = 16):
// per dimension an even pre-pool position 2d takes input d with tap 1 and an
// odd one 2d+1 takes input d with tap 2 and input d+1 with tap 0 (the page's
// per-parity analysis).  Averaging the 2x2x2 window therefore touches only the
// 8 inputs (d+a, h+b, w+c), a,b,c in {0,1}, and input offset 0 in a dim pairs
// with taps {1,2}, offset 1 with tap {0} (the page's grouping of the 27 terms,
// counts 8/4/4/4/2/2/2/1).  Summing the taps of each group gives 8 effective
// weights per (ci, co):
//     Weff[ci,co,a,b,c] = scale1*scale2/8 * sum_{kd in T(a), kh in T(b), kw in T(c)} w
//     beff[co]          = (conv_bias[co]*scale1 + bias[co]) * scale2
// and the pooled output is the 2x2x2 valid correlation
//     y[n,co,d,h,w] = beff[co] + sum_ci sum_abc x[n,ci,d+a,h+b,w+c] * Weff[ci,co,a,b,c],
// with pooled size = input size - 1 in each dim.  This equals the literal
// chain in exact arithmetic; in fp32 it differs by rounding only (the page
// argues the reassociation is far inside an fp32 tolerance).
//
// Design (GB300): every CTA collapses the weights itself (C_in*16*27 loads,
// computed in double, rounded once) into shared memory, so the op is one
// kernel with no scratch buffer and no host access to the weights.  The
// output rows of all (n, d) planes form one flat range that is split evenly
// across a persistent grid; a CTA walks its range in segments of <= TH rows of
// one plane.  A segment's input (C_in x 2 planes x (rows+1) x W) is staged in
// shared memory with cp.async, double-buffered so the next segment loads while
// this one computes.  Each thread owns up to 4 output points of the segment
// (strided by the block size, so every store instruction of a warp writes 32
// consecutive floats) and all 16 output channels: per input channel it reads
// the 8 neighbours of each point once and applies them to 16 channels with
// broadcast float4 weight reads (16 FMAs per shared-memory load).
//
// General path: one thread per pooled output evaluates the literal chain with
// the gather form of the transposed convolution, tap k taken where
// (o + pad - dil*k) is a non-negative multiple of the stride below the input
// size in each dim.
#include <algorithm>

#include "aps_dev.cuh"
#include "aps_internal.h"

namespace aps {
namespace ct3 {
constexpr int COUT = 16;
constexpr int CIN_MAX = 8;
constexpr int THREADS = 256;
constexpr int P = 4;                          // output points per thread
constexpr int MAX_PTS = THREADS * P;          // points per segment
constexpr int XTILE_MAX = 12288;              // floats per staged segment (48 KB)
}  // namespace ct3

// One segment of rows of one (n, d) output plane from the staged input xt
// ([C_in][2 planes][PT floats], rows of W): PJ points per thread (strided by
// the block size, so each store instruction of a warp covers 32 consecutive
// outputs) x all 16 channels.  CIN_T / W_T fix C_in / W at compile time (0:
// run time) so that every neighbour offset folds into an immediate.
template <int PJ, int CIN_T, int W_T>
__device__ __forceinline__ void fused_segment(const float *__restrict__ xt,
                                              const float *__restrict__ wsm,
                                              const float *__restrict__ bsm, float *yt,
                                              long long cstride, int npts, int Cin_rt, int W_rt,
                                              int PT) {
    using namespace ct3;
    const int Cin = CIN_T ? CIN_T : Cin_rt;
    const int W = W_T ? W_T : W_rt;
    const int Wo = W - 1;
    const int tid = threadIdx.x;
    int base[PJ];
    bool valid[PJ];
#pragma unroll
    for (int j = 0; j < PJ; ++j) {
        const int s = tid + j * THREADS;
        valid[j] = s < npts;
        const int ss = valid[j] ? s : 0;
        const int ohl = ss / Wo;
        base[j] = ohl * W + (ss - ohl * Wo);
    }
    float acc[COUT][PJ];
#pragma unroll
    for (int co = 0; co < COUT; ++co)
#pragma unroll
        for (int j = 0; j < PJ; ++j) acc[co][j] = bsm[co];

#pragma unroll 1
    for (int ci = 0; ci < Cin; ++ci) {
        float xv[PJ][8];
        const float *x0 = xt + (ci * 2) * PT;
        const float *x1 = x0 + PT;
#pragma unroll
        for (int j = 0; j < PJ; ++j) {
            xv[j][0] = x0[base[j]];
            xv[j][1] = x0[base[j] + 1];
            xv[j][2] = x0[base[j] + W];
            xv[j][3] = x0[base[j] + W + 1];
            xv[j][4] = x1[base[j]];
            xv[j][5] = x1[base[j] + 1];
            xv[j][6] = x1[base[j] + W];
            xv[j][7] = x1[base[j] + W + 1];
        }
        const float4 *wq = reinterpret_cast<const float4 *>(wsm + ci * COUT * 8);
#pragma unroll
        for (int co = 0; co < COUT; ++co) {
            const float4 wl = wq[2 * co], wh = wq[2 * co + 1];
#pragma unroll
            for (int j = 0; j < PJ; ++j) {
                float t = acc[co][j];
                t = fmaf(xv[j][0], wl.x, t);
                t = fmaf(xv[j][1], wl.y, t);
                t = fmaf(xv[j][2], wl.z, t);
                t = fmaf(xv[j][3], wl.w, t);
                t = fmaf(xv[j][4], wh.x, t);
                t = fmaf(xv[j][5], wh.y, t);
                t = fmaf(xv[j][6], wh.z, t);
                t = fmaf(xv[j][7], wh.w, t);
                acc[co][j] = t;
            }
        }
    }
#pragma unroll
    for (int co = 0; co < COUT; ++co) {
        float *yc = yt + co * cstride;
#pragma unroll
        for (int j = 0; j < PJ; ++j)
            if (valid[j]) yc[j * THREADS] = acc[co][j];
    }
}

template <int CIN_T, int W_T>
__global__ void __launch_bounds__(ct3::THREADS, 2)
    ct3d_pool2_fast_kernel(const float *__restrict__ x, const float *__restrict__ w,
                           const float *__restrict__ conv_bias, const float *__restrict__ bias,
                           float scale1, float scale2, float *__restrict__ y, int Cin_rt, int D,
                           int H, int W_rt, int TH, int PT, long long total_rows, int vec16) {
    using namespace ct3;
    const int Cin = CIN_T ? CIN_T : Cin_rt;
    const int W = W_T ? W_T : W_rt;
    extern __shared__ __align__(16) float sm[];
    float *wsm = sm;                               // [Cin][16][8]
    float *bsm = sm + CIN_MAX * COUT * 8;          // [16]
    const int tile_floats = Cin * 2 * PT;
    float *xs0 = bsm + COUT;                       // two staging buffers
    float *xs1 = xs0 + ((tile_floats + 3) & ~3);
    const int Do = D - 1, Ho = H - 1, Wo = W - 1;
    const int tid = threadIdx.x;

    // ---- collapsed weights and folded bias (the page's 8-group sums), fp32
    const float wscale = scale1 * scale2 * 0.125f;
    for (int i = tid; i < Cin * COUT * 8; i += THREADS) {
        const int ci = i / (COUT * 8), co = (i / 8) % COUT, g = i % 8;
        const int a = g >> 2, b = (g >> 1) & 1, c = g & 1;
        const float *wp = w + (size_t)(ci * COUT + co) * 27;
        float acc = 0.f;
        for (int kd = a ? 0 : 1; kd <= (a ? 0 : 2); ++kd)
            for (int kh = b ? 0 : 1; kh <= (b ? 0 : 2); ++kh)
                for (int kw = c ? 0 : 1; kw <= (c ? 0 : 2); ++kw)
                    acc += __ldg(wp + kd * 9 + kh * 3 + kw);
        wsm[i] = acc * wscale;
    }
    if (tid < COUT) {
        const float cb = conv_bias ? __ldg(conv_bias + tid) : 0.f;
        bsm[tid] = fmaf(cb, scale1, __ldg(bias + tid)) * scale2;
    }

    // ---- this CTA's range of output rows
    const long long r_begin = total_rows * blockIdx.x / gridDim.x;
    const long long r_end = total_rows * (blockIdx.x + 1) / gridDim.x;

    // Stage segment (plane, oh0, rows) into dst: for each (ci, a) the input
    // rows oh0 .. oh0+rows of plane od+a, which are contiguous in memory.
    auto stage = [&](long long plane, int oh0, int rows, float *dst) {
        const long long n = plane / Do;
        const int od = (int)(plane - n * Do);
        const int count = (rows + 1) * W;
        for (int ci = 0; ci < Cin; ++ci)
            for (int a = 0; a < 2; ++a) {
                const float *src = x + ((((n * Cin + ci) * D + od + a) * H) + oh0) * (long long)W;
                float *d = dst + (ci * 2 + a) * PT;
                if (vec16) {
                    for (int e = tid * 4; e < count; e += THREADS * 4) cp_async_16(d + e, src + e);
                } else {
                    for (int e = tid; e < count; e += THREADS) cp_async_4(d + e, src + e);
                }
            }
    };
    auto next_segment = [&](long long r, int &rows) {
        const int oh0 = (int)(r % Ho);
        const int cap = TH < Ho - oh0 ? TH : Ho - oh0;
        rows = (long long)cap < r_end - r ? cap : (int)(r_end - r);
    };

    long long r = r_begin;
    int rows = 0;
    if (r < r_end) {
        next_segment(r, rows);
        stage(r / Ho, (int)(r % Ho), rows, xs0);
    }
    cp_async_commit();
    int buf = 0;
    const long long plane_out = (long long)Ho * Wo;
    const long long cstride = (long long)Do * plane_out;
    while (r < r_end) {
        const long long rn = r + rows;
        int rows_n = 0;
        if (rn < r_end) {
            next_segment(rn, rows_n);
            stage(rn / Ho, (int)(rn % Ho), rows_n, buf ? xs0 : xs1);
        }
        cp_async_commit();
        cp_async_wait<1>();
        __syncthreads();

        // ---- compute segment (plane, oh0, rows) from buffer `buf`
        const float *xt = buf ? xs1 : xs0;
        const long long plane = r / Ho;
        const int oh0 = (int)(r % Ho);
        const int npts = rows * Wo;
        const long long n = plane / Do;
        const long long od = plane - n * Do;
        float *yt = y + ((n * COUT) * Do + od) * plane_out + (long long)oh0 * Wo + tid;
        // only as many point slots per thread as the segment needs (block-uniform)
        switch ((npts + THREADS - 1) / THREADS) {
            case 1: fused_segment<1, CIN_T, W_T>(xt, wsm, bsm, yt, cstride, npts, Cin, W, PT); break;
            case 2: fused_segment<2, CIN_T, W_T>(xt, wsm, bsm, yt, cstride, npts, Cin, W, PT); break;
            case 3: fused_segment<3, CIN_T, W_T>(xt, wsm, bsm, yt, cstride, npts, Cin, W, PT); break;
            default: fused_segment<4, CIN_T, W_T>(xt, wsm, bsm, yt, cstride, npts, Cin, W, PT); break;
        }
        __syncthreads();   // buffer `buf` is restaged two segments later
        r = rn;
        rows = rows_n;
        buf ^= 1;
    }
    cp_async_wait<0>();
}

template <int CIN_T, int W_T>
static aps_status launch_fused_fast(const float *x, const int64_t in[5], const float *w,
                                    const float *conv_bias, const float *bias, float scale1,
                                    float scale2, float *y, const int64_t out[5], cudaStream_t st) {
    using namespace ct3;
    const int64_t N = in[0], Cin = in[1], D = in[2], H = in[3], W = in[4];
    const int64_t Do = out[2], Ho = out[3], Wo = out[4];
    int64_t TH = std::min<int64_t>(Ho, MAX_PTS / Wo);
    TH = std::min<int64_t>(TH, XTILE_MAX / (Cin * 2 * W) - 1);
    if (TH < 1) return APS_ERR_UNSUPPORTED;
    // staged floats per (ci, input plane): fixed at compile time for a fixed W
    const int64_t PT = W_T ? (MAX_PTS / (W_T - 1) + 1) * W_T : (TH + 1) * W;
    if (Cin * 2 * PT > XTILE_MAX) return APS_ERR_UNSUPPORTED;
    const int64_t tile_floats = Cin * 2 * PT;
    const int smem = (int)((CIN_MAX * COUT * 8 + COUT + 2 * ((tile_floats + 3) & ~3)) * 4);
    const auto kern = ct3d_pool2_fast_kernel<CIN_T, W_T>;
    const int per_sm = resident_ctas((const void *)kern, THREADS, smem);
    if (per_sm < 1) return APS_ERR_CUDA;
    const long long total_rows = N * Do * Ho;
    const long long pts = total_rows * Wo;
    long long grid = std::min<long long>((long long)sm_count() * per_sm, ceil_div(pts, THREADS));
    grid = std::max<long long>(grid, 1);
    const int vec16 = (W % 4 == 0) && (reinterpret_cast<uintptr_t>(x) % 16 == 0);
    kern<<<(unsigned)grid, THREADS, smem, st>>>(x, w, conv_bias, bias, scale1, scale2, y,
                                                (int)Cin, (int)D, (int)H, (int)W, (int)TH,
                                                (int)PT, total_rows, vec16);
    return launch_status();
}

aps_status launch_ct3d_pool2_fast(const float *x, const int64_t in[5], const float *w,
                                  const float *conv_bias, const float *bias, float scale1,
                                  float scale2, float *y, const int64_t out[5],
                                  cudaStream_t st) {
    using namespace ct3;
    const int64_t Cin = in[1], D = in[2], H = in[3], W = in[4];
    if (Cin < 1 || Cin > CIN_MAX || D < 2 || H < 2 || W < 2 || W > MAX_PTS) return APS_ERR_UNSUPPORTED;
    // the pages' shapes (3 input channels, rows of 32 and 16) run fully specialised
    if (Cin == 3 && W == 32)
        return launch_fused_fast<3, 32>(x, in, w, conv_bias, bias, scale1, scale2, y, out, st);
    if (Cin == 3 && W == 16)
        return launch_fused_fast<3, 16>(x, in, w, conv_bias, bias, scale1, scale2, y, out, st);
    return launch_fused_fast<0, 0>(x, in, w, conv_bias, bias, scale1, scale2, y, out, st);
}

// ------------------------------------------------------------ direct kernel
__global__ void ct3d_pool_direct_kernel(const float *__restrict__ x, const float *__restrict__ w,
                                        const float *__restrict__ conv_bias,
                                        const float *__restrict__ bias, float scale1,
                                        float scale2, float *__restrict__ y, long long total,
                                        int Cin, int Cout, int D, int H, int W, int Do, int Ho,
                                        int Wo, int kd, int kh, int kw, int sd, int sh, int sw,
                                        int pd, int ph, int pw, int dd, int dh, int dw, int q) {
    for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        const int pw_ = (int)(idx % Wo);
        long long t = idx / Wo;
        const int ph_ = (int)(t % Ho);
        t /= Ho;
        const int pd_ = (int)(t % Do);
        t /= Do;
        const int co = (int)(t % Cout);
        const long long n = t / Cout;
        const float cb = conv_bias ? conv_bias[co] : 0.f;
        float pool = 0.f;
        for (int qa = 0; qa < q; ++qa)
            for (int qb = 0; qb < q; ++qb)
                for (int qc = 0; qc < q; ++qc) {
                    const int od = pd_ * q + qa, oh = ph_ * q + qb, ow = pw_ * q + qc;
                    float v = 0.f;
                    for (int ci = 0; ci < Cin; ++ci) {
                        const float *xp = x + (n * Cin + ci) * (long long)D * H * W;
                        const float *wp = w + ((long long)ci * Cout + co) * kd * kh * kw;
                        for (int a = 0; a < kd; ++a) {
                            const int nd = od + pd - a * dd;
                            if (nd < 0 || nd % sd) continue;
                            const int id = nd / sd;
                            if (id >= D) continue;
                            for (int b = 0; b < kh; ++b) {
                                const int nh = oh + ph - b * dh;
                                if (nh < 0 || nh % sh) continue;
                                const int ih = nh / sh;
                                if (ih >= H) continue;
                                for (int c = 0; c < kw; ++c) {
                                    const int nw = ow + pw - c * dw;
                                    if (nw < 0 || nw % sw) continue;
                                    const int iw = nw / sw;
                                    if (iw >= W) continue;
                                    v = fmaf(__ldg(xp + ((long long)id * H + ih) * W + iw),
                                             __ldg(wp + (a * kh + b) * kw + c), v);
                                }
                            }
                        }
                    }
                    pool += (v + cb) * scale1;
                }
        y[idx] = (pool / (float)(q * q * q) + bias[co]) * scale2;
    }
}

aps_status launch_ct3d_pool_direct(const float *x, const int64_t in[5], const float *w,
                                   const float *conv_bias, const float *bias, int64_t c_out,
                                   const int k[3], const int s[3], const int p[3],
                                   const int d[3], int pool_k, float scale1, float scale2,
                                   float *y, const int64_t out[5], cudaStream_t st) {
    for (int i = 2; i < 5; ++i)
        if (in[i] >= (1 << 30) || out[i] * pool_k >= (1 << 30)) return APS_ERR_UNSUPPORTED;
    if (c_out >= (1 << 30) || in[1] >= (1 << 30)) return APS_ERR_UNSUPPORTED;
    const long long total = out[0] * out[1] * out[2] * out[3] * out[4];
    const int threads = 256;
    const long long blocks =
        std::min<long long>(ceil_div(total, threads), (long long)sm_count() * 16);
    ct3d_pool_direct_kernel<<<(unsigned)blocks, threads, 0, st>>>(
        x, w, conv_bias, bias, scale1, scale2, y, total, (int)in[1], (int)c_out, (int)in[2],
        (int)in[3], (int)in[4], (int)out[2], (int)out[3], (int)out[4], k[0], k[1], k[2], s[0],
        s[1], s[2], p[0], p[1], p[2], d[0], d[1], d[2], pool_k);
    return launch_status();
}

}  // namespace aps
