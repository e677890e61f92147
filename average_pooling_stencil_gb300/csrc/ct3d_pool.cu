// ct3d_pool.cu -- fused ConvTranspose3d -> x scale1 -> AvgPool3d(pool_k) ->
// + bias -> x scale2 (the model of Kimi-K2.6__l2_p50).
//
// Fast path (k3, s2, p1, output_padding 0 or 1, dilation 1, pool 2, C_out = 16):
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
// with pooled size = input size - 1 in a dim with output_padding 0 and = input
// size with output_padding 1: the extra pooled position averages pre-pool
// positions 2D-2 and 2D-1, the latter the output_padding row, whose input
// offset 1 lies past the end of x and counts as zero.  This equals the literal
// chain in exact arithmetic; in fp32 it differs by rounding only (the page
// argues the reassociation is far inside an fp32 tolerance).
//
// Which kernel runs: C_in <= 3 with 16-byte input rows takes the tensor-core
// kernel (ct3d_pool_tc.cu); this FP32-pipe kernel serves the rest of the fast
// path (C_in 4..8, inputs a TMA box cannot read).
//
// Design (GB300): a persistent grid of 8-warp CTAs (2 per SM).  Each CTA
// collapses the weights once (C_in*16*27 loads) into shared memory, so the op
// is one kernel with no scratch buffer and no host access to the weights.  A
// unit is up to 32 output rows x 32 output columns of one (n, od) plane; units
// are dealt to the CTAs round-robin, so at any time the grid works on a narrow
// window of the output.  A unit's input -- C_in channels x 2 planes x 33 rows
// x (32 or 36) columns -- arrives by one 4-D TMA box (zero-filled outside the
// tensor), double-buffered behind mbarriers with bounded waits, or by 4-byte
// cp.async when the rows are not 16-byte strided.  Lane l owns output column
// l and warp w output rows 4w..4w+3 of the unit, all 16 channels: per input
// channel a thread reads its 2 x 5 x 2 input window once (32 consecutive
// words per warp load: no bank conflicts) and applies each of the 8 taps to
// its 4 rows with broadcast float4 weight reads.  Accumulators are channel
// pairs updated with the packed fp32x2 FMA (two exactly rounded fp32 FMAs per
// instruction).  Outputs are staged per channel in shared memory at their
// destination's float offset mod 4; when the unit spans whole output rows a
// channel's outputs are one contiguous run of y, whose 16-byte-aligned middle
// leaves by one cp.async.bulk copy (head and tail floats by plain stores), so
// the stores overlap the next unit's math.
//
// General path: one thread per pooled output evaluates the literal chain with
// the gather form of the transposed convolution, tap k taken where
// (o + pad - dil*k) is a non-negative multiple of the stride below the input
// size in each dim.
#include <algorithm>
#include <cstring>

#include "aps_dev.cuh"
#include "aps_internal.h"

namespace aps {
namespace ct3 {
constexpr int COUT = 16;
constexpr int CIN_MAX = 8;
constexpr int WARPS = 8;
constexpr int THREADS = 32 * WARPS;
constexpr int RPT = 4;                 // output rows per thread
constexpr int TOH = WARPS * RPT;       // output rows per unit (at most)
constexpr int TOW = 32;                // output columns per unit (one per lane)
constexpr int SLACK = 64;              // floats after a stage: lanes past the last column read on
// Floats one stage occupies: the staged window plus the rows a warp whose
// rows end inside the unit may still read (up to row 4*WARPS), plus slack.
__host__ __device__ inline int stage_stride_of(int Cin, int XR, int BW) {
    return (Cin * 2 * XR * BW + (TOH + 1 - XR) * BW + SLACK + 31) & ~31;
}
// Floats of one channel's output staging: a unit's RB x WB outputs, 16-byte
// aligned, plus 3 for the shift that gives the run the alignment of its
// destination.
__host__ __device__ inline int chan_stride_of(int RB, int WB) {
    return ((RB * WB + 3) & ~3) + 4;
}
}  // namespace ct3

// BW_T: staged row length (columns) fixed at compile time (0: run time), so
// that every window offset folds into an immediate.
template <int BW_T>
__global__ void __launch_bounds__(ct3::THREADS, BW_T ? 2 : 1)
    ct3d_pool2_fast_kernel(const __grid_constant__ CUtensorMap xmap, int use_tma,
                           const float *__restrict__ x, const float *__restrict__ w,
                           const float *__restrict__ conv_bias, const float *__restrict__ bias,
                           float scale1, float scale2, float *__restrict__ y, int Cin, int D,
                           int H, int W, int Do, int Ho, int Wo, int BW_rt, int XR, int RB, int WB, int n_ohb,
                           int n_owb, long long n_units, unsigned int *status) {
    pdl_trigger();
    pdl_wait();
    using namespace ct3;
    const int BW = BW_T ? BW_T : BW_rt;
    extern __shared__ __align__(128) float sm[];
    const int stage_floats = Cin * 2 * XR * BW;
    const int stage_stride = stage_stride_of(Cin, XR, BW);   // 128-byte aligned stages
    float *xs = sm;                                  // [2][Cin][2][XR][BW]
    const int CH = chan_stride_of(RB, WB);
    float *ost = xs + 2 * stage_stride;              // [16][CH] output staging
    float *wsm = ost + ((COUT * CH + 31) & ~31);     // [Cin][8][16]
    float *bsm = wsm + Cin * 8 * COUT;               // [16]
    uint64_t *bar = reinterpret_cast<uint64_t *>(bsm + COUT);   // [2], 8-byte aligned
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    struct Unit {
        long long n;
        int od, oh0, ow0, rows, cols;
    };
    auto unit = [&](long long u) {
        Unit g;
        const int owb = (int)(u % n_owb);
        long long t = u / n_owb;
        const int ohb = (int)(t % n_ohb);
        t /= n_ohb;
        g.od = (int)(t % Do);
        g.n = t / Do;
        g.oh0 = ohb * RB;
        g.ow0 = owb * WB;
        g.rows = Ho - g.oh0 < RB ? Ho - g.oh0 : RB;
        g.cols = Wo - g.ow0 < WB ? Wo - g.ow0 : WB;
        return g;
    };
    // input window of a unit into stage b: TMA box (thread 0), or element
    // copies with zero fill (all threads)
    auto stage = [&](const Unit &g, int b) {
        float *dst = xs + b * stage_stride;
        if (use_tma) {
            if (tid == 0) {
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                mbar_arrive_expect_tx(&bar[b], (uint32_t)stage_floats * 4u);
                tma_load_4d(dst, &xmap, &bar[b], g.ow0, g.oh0, g.od, (int)(g.n * Cin));
            }
        } else {
            for (int e = tid; e < stage_floats; e += THREADS) {
                const int col = e % BW;
                int t = e / BW;
                const int r = t % XR;
                t /= XR;
                const int a = t & 1, ci = t >> 1;
                const int ih = g.oh0 + r, iw = g.ow0 + col;
                const bool in = g.od + a < D && ih < H && iw < W;
                const float *src =
                    in ? x + (((g.n * Cin + ci) * D + g.od + a) * (long long)H + ih) * W + iw : x;
                asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(
                                 smem_u32(dst + e)),
                             "l"(src), "r"(in ? 4 : 0)
                             : "memory");
            }
            cp_async_commit();
        }
    };

    if (tid == 0 && use_tma) {
        mbar_init(&bar[0], 1);
        mbar_init(&bar[1], 1);
        mbar_fence_init();
    }
    __syncthreads();
    Unit cur{};
    if ((long long)blockIdx.x < n_units) {
        cur = unit(blockIdx.x);
        stage(cur, 0);
    }

    // ---- collapsed weights [ci][a*4+b*2+c][co] and folded bias, once per CTA
    const float wscale = scale1 * scale2 * 0.125f;
    for (int i = tid; i < Cin * 8 * COUT; i += THREADS) {
        // one collapsed tap of one (ci, co): its (up to 8) weights by
        // independent loads, summed in ascending (kd, kh, kw)
        const int co = i % COUT, g = (i / COUT) % 8, ci = i / (8 * COUT);
        wsm[i] = collapse_tap_ldg(w + (size_t)(ci * COUT + co) * 27, g) * wscale;
    }
    if (tid < COUT) {
        const float cb = conv_bias ? __ldg(conv_bias + tid) : 0.f;
        bsm[tid] = fmaf(cb, scale1, __ldg(bias + tid)) * scale2;
    }
    __syncthreads();

    const long long plane = (long long)Ho * Wo;
    const long long cstride = (long long)Do * plane;   // between output channels
    long long k = 0;
    // units are dealt round-robin, so at any time the grid works on a narrow,
    // contiguous window of the output
    for (long long u = blockIdx.x; u < n_units; u += gridDim.x, ++k) {
        const int b = (int)(k & 1);
        // prefetch the next unit into the other stage (freed by the barrier
        // that ended the previous iteration)
        const bool more = u + gridDim.x < n_units;
        if (more) stage(unit(u + gridDim.x), b ^ 1);
        bool ok = true;
        if (use_tma) {
            ok = mbar_wait(&bar[b], (uint32_t)(k >> 1) & 1u);
        } else {
            if (more)
                cp_async_wait<1>();
            else
                cp_async_wait<0>();
        }
        if (__syncthreads_or(!ok)) {
            // a copy never landed: note it, let the prefetch (if any) and the
            // output copies finish or time out, and stop
            if (tid == 0) {
                record_error(status, APS_DEVERR_TIMEOUT);
                if (use_tma && more) mbar_wait(&bar[b ^ 1], (uint32_t)((k + 1) >> 1) & 1u);
                bulk_wait<0>();
            }
            return;
        }

        // ---- 4 rows x 16 channels per thread
        float2 acc[COUT / 2][RPT];
#pragma unroll
        for (int c2 = 0; c2 < COUT / 2; ++c2) {
            const float2 bv = make_float2(bsm[2 * c2], bsm[2 * c2 + 1]);
#pragma unroll
            for (int i = 0; i < RPT; ++i) acc[c2][i] = bv;
        }
        const float *xb = xs + b * stage_stride;
        const int nci = RPT * warp < cur.rows ? Cin : 0;   // warps past the unit's rows idle
#pragma unroll 1
        for (int ci = 0; ci < nci; ++ci) {
            const float *xp = xb + (ci * 2 * XR + RPT * warp) * BW + lane;
            float xv[2][RPT + 1][2];
#pragma unroll
            for (int a = 0; a < 2; ++a)
#pragma unroll
                for (int rr = 0; rr <= RPT; ++rr)
#pragma unroll
                    for (int c = 0; c < 2; ++c) xv[a][rr][c] = xp[(a * XR + rr) * BW + c];
            const float4 *wq = reinterpret_cast<const float4 *>(wsm + ci * 8 * COUT);
#pragma unroll
            for (int g = 0; g < 8; ++g) {
                const int a = g >> 2, bb = (g >> 1) & 1, c = g & 1;
                const float4 w0 = wq[4 * g], w1 = wq[4 * g + 1], w2 = wq[4 * g + 2],
                             w3 = wq[4 * g + 3];
                const float2 wp[COUT / 2] = {make_float2(w0.x, w0.y), make_float2(w0.z, w0.w),
                                             make_float2(w1.x, w1.y), make_float2(w1.z, w1.w),
                                             make_float2(w2.x, w2.y), make_float2(w2.z, w2.w),
                                             make_float2(w3.x, w3.y), make_float2(w3.z, w3.w)};
#pragma unroll
                for (int i = 0; i < RPT; ++i) {
                    const float xg = xv[a][i + bb][c];
#pragma unroll
                    for (int c2 = 0; c2 < COUT / 2; ++c2)
                        acc[c2][i] = __ffma2_rn(make_float2(xg, xg), wp[c2], acc[c2][i]);
                }
            }
        }

        // ---- outputs.  With whole output rows in the unit (WB == Wo) the unit's
        // outputs of channel co are one run, contiguous in y; it is staged at
        // ost + co*CH + off (off = its destination's float offset mod 4, so
        // both sides share 16-byte alignment), its aligned middle leaves by one
        // bulk copy and the at most 3 + 3 head and tail floats by plain stores.
        // Otherwise the staging rows are WB long and rows leave by plain stores.
        const bool runs = WB == Wo;
        const float *y_unit = y + ((cur.n * COUT) * Do + cur.od) * plane + (long long)cur.oh0 * Wo;
        const uint32_t a0 = runs ? (uint32_t)(reinterpret_cast<uintptr_t>(y_unit) >> 2) & 3u : 0u;
        const uint32_t ac = runs ? (uint32_t)cstride & 3u : 0u;
        // the bulk copies of the previous unit have read the staging block
        if (tid == 0) bulk_wait_read<0>();
        __syncthreads();
        if (lane < cur.cols) {
#pragma unroll
            for (int i = 0; i < RPT; ++i) {
                const int row = RPT * warp + i;
                if (row >= cur.rows) break;
#pragma unroll
                for (int c2 = 0; c2 < COUT / 2; ++c2) {
                    const int c0 = 2 * c2, c1 = 2 * c2 + 1;
                    ost[c0 * CH + ((a0 + c0 * ac) & 3u) + row * WB + lane] = acc[c2][i].x;
                    ost[c1 * CH + ((a0 + c1 * ac) & 3u) + row * WB + lane] = acc[c2][i].y;
                }
            }
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncthreads();
        if (runs) {
            const int run = cur.rows * Wo;
            if (tid == 0) {
                for (int co = 0; co < COUT; ++co) {
                    const uint32_t off = (a0 + co * ac) & 3u, h = (4u - off) & 3u;
                    const int mid = run > (int)h ? (run - (int)h) & ~3 : 0;
                    if (mid > 0)
                        bulk_store(const_cast<float *>(y_unit) + co * cstride + h,
                                   ost + co * CH + off + h, (uint32_t)mid * 4u);
                }
                bulk_commit();
            }
            for (int co = warp; co < COUT; co += WARPS) {
                const uint32_t off = (a0 + co * ac) & 3u, h = (4u - off) & 3u;
                const int head = run < (int)h ? run : (int)h;
                const int mid = run > (int)h ? (run - (int)h) & ~3 : 0;
                const int tail0 = head + mid;
                float *yc = const_cast<float *>(y_unit) + co * cstride;
                const float *sc = ost + co * CH + off;
                if (lane < head) yc[lane] = sc[lane];
                if (tail0 + lane < run) yc[tail0 + lane] = sc[tail0 + lane];
            }
        } else {
            for (int co = warp; co < COUT; co += WARPS) {
                float *yc = const_cast<float *>(y_unit) + co * cstride;
                const float *sc = ost + co * CH;
                if (lane < cur.cols)
                    for (int r = 0; r < cur.rows; ++r)
                        yc[(long long)r * Wo + cur.ow0 + lane] = sc[r * WB + lane];
            }
        }
        if (more) cur = unit(u + gridDim.x);
    }
    // the output copies are complete before the CTA exits
    if (tid == 0) bulk_wait<0>();
}

aps_status launch_ct3d_pool2_fast(const float *x, const int64_t in[5], const float *w,
                                  const float *conv_bias, const float *bias, float scale1,
                                  float scale2, float *y, const int64_t out[5],
                                  cudaStream_t st) {
    using namespace ct3;
    const int64_t N = in[0], Cin = in[1], D = in[2], H = in[3], W = in[4];
    if (Cin < 1 || Cin > CIN_MAX || D < 2 || H < 2 || W < 2 || D >= (1 << 30) ||
        H >= (1 << 30) || W >= (1 << 30) || N * Cin >= (1ll << 31))
        return APS_ERR_UNSUPPORTED;
    const int64_t Do = out[2], Ho = out[3], Wo = out[4];
    // a unit: up to 32 output rows x 32 output columns of one (n, od) plane
    const int RB = (int)std::min<int64_t>(Ho, TOH), WB = (int)std::min<int64_t>(Wo, TOW);
    const int64_t n_ohb = ceil_div(Ho, RB), n_owb = ceil_div(Wo, WB);
    const long long n_units = N * Do * n_ohb * n_owb;
    // staged input: rows RB+1, columns WB+1 rounded up to a multiple of 4
    const int XR = RB + 1;
    const int BW = (WB + 1 + 3) & ~3;
    const int use_tma = (W % 4 == 0) && (reinterpret_cast<uintptr_t>(x) % 16 == 0);
    CUtensorMap map;
    if (use_tma) {
        const cuuint64_t dims[4] = {(cuuint64_t)W, (cuuint64_t)H, (cuuint64_t)D,
                                    (cuuint64_t)(N * Cin)};
        const cuuint64_t strides[3] = {(cuuint64_t)(W * 4), (cuuint64_t)(H * W * 4),
                                       (cuuint64_t)(D * H * W * 4)};
        const cuuint32_t box[4] = {(cuuint32_t)BW, (cuuint32_t)XR, 2, (cuuint32_t)Cin};
        const cuuint32_t estr[4] = {1, 1, 1, 1};
        if (!encode_tiled(&map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<float *>(x), dims,
                          strides, box, estr))
            return APS_ERR_UNSUPPORTED;
    } else {
        std::memset(&map, 0, sizeof(map));
    }
    const int64_t stage_stride = stage_stride_of((int)Cin, XR, BW);
    const int64_t ost_floats = (COUT * chan_stride_of(RB, WB) + 31) & ~31;
    const size_t smem =
        (size_t)(2 * stage_stride + ost_floats + Cin * 8 * COUT + COUT) * 4 + 16;
    const auto kern = BW == 32 ? ct3d_pool2_fast_kernel<32>
                    : BW == 36 ? ct3d_pool2_fast_kernel<36>
                    : BW == 16 ? ct3d_pool2_fast_kernel<16>
                               : ct3d_pool2_fast_kernel<0>;
    const int per_sm = resident_ctas((const void *)kern, THREADS, (int)smem);
    if (per_sm < 1) return APS_ERR_UNSUPPORTED;
    const long long grid = std::min<long long>((long long)per_sm * sm_count(), n_units);
    const cudaError_t e = launch_pdl(kern, dim3((unsigned)grid), dim3(THREADS), smem, st, map, use_tma, x, w, conv_bias,
               bias, scale1, scale2, y, (int)Cin, (int)D, (int)H, (int)W, (int)Do, (int)Ho,
               (int)Wo, BW, XR, RB, WB,
               (int)n_ohb, (int)n_owb, n_units, status_word());
    return launch_status(e);
}

// ------------------------------------------------------------ direct kernel
__global__ void ct3d_pool_direct_kernel(const float *__restrict__ x, const float *__restrict__ w,
                                        const float *__restrict__ conv_bias,
                                        const float *__restrict__ bias, float scale1,
                                        float scale2, float *__restrict__ y, long long total,
                                        int Cin, int Cout, int D, int H, int W, int Do, int Ho,
                                        int Wo, int kd, int kh, int kw, int sd, int sh, int sw,
                                        int pd, int ph, int pw, int dd, int dh, int dw, int q) {
    pdl_trigger();
    pdl_wait();
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
    const cudaError_t e = launch_pdl(ct3d_pool_direct_kernel, dim3((unsigned)blocks), dim3(threads), 0, st, x, w,
               conv_bias, bias, scale1, scale2, y, total, (int)in[1], (int)c_out, (int)in[2],
               (int)in[3], (int)in[4], (int)out[2], (int)out[3], (int)out[4], k[0], k[1], k[2],
               s[0], s[1], s[2], p[0], p[1], p[2], d[0], d[1], d[2], pool_k);
    return launch_status(e);
}

}  // namespace aps
