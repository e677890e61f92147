// convt3d.cu -- standalone ConvTranspose3d in fp32, emitting the full-resolution
// (pre-pool) tensor: the first stage of Kimi-K2.6__l2_p50's unfused chain
// ("approach 1" on that page, there done by the vendor library).
//
// Operation (the page's scatter definition, written as a gather):
//   y[n,co,o] = bias[co] + sum_ci sum_k w[ci,co,k] * x[n,ci,(o + p - d*k)/s]
// per spatial dim, a term existing only where o + p - d*k is a non-negative
// multiple of s whose quotient is inside the input.
//
// Which kernel runs: C_in <= 3 with W <= 32 and 16-byte input rows takes the
// tensor-core kernel (convt3d_tc.cu); this FP32-pipe kernel serves the rest of
// the fast path (C_in 4..8, W > 32).
//
// Fast kernel (k3, s2, p1, d1, output_padding 0 or 1, C_out = 16, C_in <= 8):
// per dim an output o = 2m + r takes, for r = 0, input m with tap 1 and, for
// r = 1, input m+1 with tap 0 and input m with tap 2 (the page's per-parity
// analysis).  A thread owns one input position (mh, mw) of a plane and the 2x2
// outputs (2mh + rh, 2mw + rw) around it; per input channel it reads the
// inputs (mh+b, mw+c) of each input plane the output plane's parity needs
// (one for an even od, two for an odd one) and applies each to the outputs it
// reaches: 9 (kh, kw) products per plane for 4 outputs, i.e. 1.5 taps per dim
// per output and no zero taps.  A CTA of 8 warps owns a unit of 16 output rows
// x 64 output columns of one (n, od) plane: warp w takes input rows
// mh0 + 4*(w%2) + 0..3 and channels 4*(w/2) .. +3 (each broadcast weight
// read serves four input rows), lane l input column mw0 + l.  The unit's
// input -- C_in x 2 planes x 9 rows x 36 columns -- is one 4-D TMA box,
// double-buffered behind mbarriers with bounded waits; units are dealt to a
// persistent grid round-robin.  Accumulators are channel pairs updated with
// the packed fp32x2 FMA.  Outputs are staged per channel in shared memory; when
// the unit spans whole output rows a channel's outputs are one contiguous run
// in y, and its 16-byte-aligned middle leaves by one bulk copy (its head and
// tail by plain stores), overlapping the next unit's math.
//
// Direct kernel: one thread per output evaluating the gather formula as
// written, for any (k, s, p, d, output_padding) and channel counts.
#include <algorithm>
#include <cstring>

#include "aps_dev.cuh"
#include "aps_internal.h"

namespace aps {
namespace c3 {
constexpr int COUT = 16;
constexpr int CIN_MAX = 8;
constexpr int WARPS = 8;
constexpr int THREADS = 32 * WARPS;
constexpr int MH = WARPS;              // input rows per unit (one per warp)
constexpr int MW = 32;                 // input columns per unit (one per lane)
constexpr int XR = MH + 1;             // staged input rows
constexpr int XC = MW + 4;             // staged input columns (33 used)
constexpr int OR = 2 * MH;             // output rows per unit
constexpr int OC = 2 * MW;             // output columns per unit
constexpr int SLACK = 64;
constexpr int R = 4;                   // input rows per thread (4: 251 us, 2: 258, 1: 300 on
                                       // the [128,3,16,32,32] workload)
constexpr int CPW = COUT / R;          // output channels per thread
static_assert(MH % R == 0 && CPW % 4 == 0, "rows per warp and channel groups");

__host__ __device__ inline int stage_stride_of(int Cin) {
    return (Cin * 2 * XR * XC + SLACK + 31) & ~31;
}
// floats of one channel's output staging: OR x min(OC, Wo) outputs, 16-byte
// aligned, plus 3 for the shift that gives a run its destination's alignment
__host__ __device__ inline int chan_stride_of(int WB) { return ((OR * WB + 3) & ~3) + 4; }
}  // namespace c3

__global__ void __launch_bounds__(c3::THREADS, 2)
    convt3d_k3s2p1_kernel(const __grid_constant__ CUtensorMap xmap, const float *__restrict__ w,
                          const float *__restrict__ bias, float *__restrict__ y, int Cin,
                          int D, int H, int W, int Do, int Ho, int Wo, int WB, int n_mhb,
                          int n_mwb, long long n_units, unsigned int *status) {
    pdl_trigger();
    pdl_wait();
    using namespace c3;
    extern __shared__ __align__(128) float sm[];
    const int stage_stride = stage_stride_of(Cin);
    const int CH = chan_stride_of(WB);
    float *xs = sm;                                   // [2][Cin][2][XR][XC]
    float *ost = xs + 2 * stage_stride;               // [16][CH]
    float *wsm = ost + ((COUT * CH + 31) & ~31);      // [Cin][27][16]
    float *bsm = wsm + Cin * 27 * COUT;               // [16]
    uint64_t *bar = reinterpret_cast<uint64_t *>(bsm + COUT);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int stage_floats = Cin * 2 * XR * XC;

    struct Unit {
        long long n;
        int od, mh0, mw0;
    };
    auto unit = [&](long long u) {
        Unit g;
        g.mw0 = (int)(u % n_mwb) * MW;
        long long t = u / n_mwb;
        g.mh0 = (int)(t % n_mhb) * MH;
        t /= n_mhb;
        g.od = (int)(t % Do);
        g.n = t / Do;
        return g;
    };
    // input planes md = od/2 and md+1, rows mh0.., columns mw0..; zero outside
    auto stage = [&](const Unit &g, int b) {
        if (tid == 0) {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            mbar_arrive_expect_tx(&bar[b], (uint32_t)stage_floats * 4u);
            tma_load_4d(xs + b * stage_stride, &xmap, &bar[b], g.mw0, g.mh0, g.od >> 1,
                        (int)(g.n * Cin));
        }
    };

    if (tid == 0) {
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
    // weights [ci][kd*9+kh*3+kw][co] (channel-contiguous for float4 broadcast reads)
    for (int i = tid; i < Cin * 27 * COUT; i += THREADS) {
        const int co = i % COUT, t = (i / COUT) % 27, ci = i / (27 * COUT);
        wsm[i] = __ldg(w + ((size_t)(ci * COUT + co)) * 27 + t);
    }
    if (tid < COUT) bsm[tid] = bias ? __ldg(bias + tid) : 0.f;
    __syncthreads();

    const long long plane = (long long)Ho * Wo;
    const long long cstride = (long long)Do * plane;
    long long k = 0;
    for (long long u = blockIdx.x; u < n_units; u += gridDim.x, ++k) {
        const int b = (int)(k & 1);
        const bool more = u + gridDim.x < n_units;
        if (more) stage(unit(u + gridDim.x), b ^ 1);
        const bool ok = mbar_wait(&bar[b], (uint32_t)(k >> 1) & 1u);
        if (__syncthreads_or(!ok)) {
            if (tid == 0) {
                record_error(status, APS_DEVERR_TIMEOUT);
                if (more) mbar_wait(&bar[b ^ 1], (uint32_t)((k + 1) >> 1) & 1u);
            }
            if (lane == 0) bulk_wait<0>();
            return;
        }

        // ---- R input rows x 2x2 outputs x CPW channels per thread: warp w
        // takes input rows mh0 + R*(w % (MH/R)) + 0..R-1 and channels
        // CPW*(w / (MH/R)) .. +CPW-1, so each weight read serves R input rows
        const int rsel = warp % (MH / R), cgrp = warp / (MH / R);
        float2 acc[CPW / 2][R][2][2];   // [channel pair][input row r][rh][rw]
#pragma unroll
        for (int c2 = 0; c2 < CPW / 2; ++c2) {
            const float2 bv =
                make_float2(bsm[CPW * cgrp + 2 * c2], bsm[CPW * cgrp + 2 * c2 + 1]);
#pragma unroll
            for (int r = 0; r < R; ++r)
#pragma unroll
                for (int rh = 0; rh < 2; ++rh)
#pragma unroll
                    for (int rw = 0; rw < 2; ++rw) acc[c2][r][rh][rw] = bv;
        }
        const int pd = cur.od & 1;   // even plane: input plane md with tap 1; odd:
                                     // md+1 with tap 0 and md with tap 2
        const float *xb = xs + b * stage_stride + R * rsel * XC + lane;
#pragma unroll 1
        for (int ci = 0; ci < Cin; ++ci) {
#pragma unroll 1
            for (int dt = 0; dt <= pd; ++dt) {
                const int a = pd ? (dt == 0 ? 1 : 0) : 0;            // staged plane
                const int kd = pd ? (dt == 0 ? 0 : 2) : 1;
                const float *xp = xb + (ci * 2 + a) * XR * XC;
                float v[R + 1][2];   // input rows R*rsel + 0..R, columns lane + 0..1
#pragma unroll
                for (int rr = 0; rr <= R; ++rr)
#pragma unroll
                    for (int c = 0; c < 2; ++c) v[rr][c] = xp[rr * XC + c];
                const float4 *wq =
                    reinterpret_cast<const float4 *>(wsm + (ci * 27 + kd * 9) * COUT + CPW * cgrp);
                // (input row b, column c) reaches output (rh, rw) with tap
                // kh = rh ? (b ? 0 : 2) : 1 (b = 0 only), likewise kw
#pragma unroll
                for (int t = 0; t < 9; ++t) {
                    // t / 3 = kh, t % 3 = kw; kh 1 -> (rh 0, b 0), kh 2 -> (rh 1, b 0),
                    // kh 0 -> (rh 1, b 1); the same for kw
                    const int rh = (t / 3) == 1 ? 0 : 1, bb = (t / 3) == 0 ? 1 : 0;
                    const int rw = (t % 3) == 1 ? 0 : 1, cc = (t % 3) == 0 ? 1 : 0;
                    float2 wp[CPW / 2];
#pragma unroll
                    for (int q = 0; q < CPW / 4; ++q) {
                        const float4 w4 = wq[(COUT / 4) * t + q];
                        wp[2 * q] = make_float2(w4.x, w4.y);
                        wp[2 * q + 1] = make_float2(w4.z, w4.w);
                    }
#pragma unroll
                    for (int r = 0; r < R; ++r) {
                        const float2 vv = make_float2(v[r + bb][cc], v[r + bb][cc]);
#pragma unroll
                        for (int c2 = 0; c2 < CPW / 2; ++c2)
                            acc[c2][r][rh][rw] = __ffma2_rn(vv, wp[c2], acc[c2][r][rh][rw]);
                    }
                }
            }
        }

        // ---- outputs (the fused kernel's scheme): staged per channel at the
        // destination's float offset mod 4; whole-row units leave as one run per
        // channel by a bulk copy of its aligned middle plus plain head/tail stores
        const int oh0 = 2 * cur.mh0, ow0 = 2 * cur.mw0;
        const int rows = Ho - oh0 < OR ? Ho - oh0 : OR;
        const int cols = Wo - ow0 < WB ? Wo - ow0 : WB;
        const bool runs = WB == Wo;
        float *y_unit = y + ((cur.n * COUT) * Do + cur.od) * plane + (long long)oh0 * Wo;
        const uint32_t a0 = runs ? (uint32_t)(reinterpret_cast<uintptr_t>(y_unit) >> 2) & 3u : 0u;
        const uint32_t ac = runs ? (uint32_t)cstride & 3u : 0u;
        if (tid == 0) bulk_wait_read<0>();
        __syncthreads();
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int rh = 0; rh < 2; ++rh) {
                const int row = 2 * (R * rsel + r) + rh;
                if (row >= rows) continue;
#pragma unroll
                for (int rw = 0; rw < 2; ++rw) {
                    const int col = 2 * lane + rw;
                    if (col >= cols) continue;
#pragma unroll
                    for (int c2 = 0; c2 < CPW / 2; ++c2) {
                        const int c0 = CPW * cgrp + 2 * c2, c1 = c0 + 1;
                        ost[c0 * CH + ((a0 + c0 * ac) & 3u) + row * WB + col] = acc[c2][r][rh][rw].x;
                        ost[c1 * CH + ((a0 + c1 * ac) & 3u) + row * WB + col] = acc[c2][r][rh][rw].y;
                    }
                }
            }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncthreads();
        if (runs) {
            const int run = rows * Wo;
            if (tid == 0) {
                for (int co = 0; co < COUT; ++co) {
                    const uint32_t off = (a0 + co * ac) & 3u, h = (4u - off) & 3u;
                    const int mid = run > (int)h ? (run - (int)h) & ~3 : 0;
                    if (mid > 0)
                        bulk_store(y_unit + co * cstride + h, ost + co * CH + off + h,
                                   (uint32_t)mid * 4u);
                }
                bulk_commit();
            }
            for (int co = warp; co < COUT; co += WARPS) {
                const uint32_t off = (a0 + co * ac) & 3u, h = (4u - off) & 3u;
                const int head = run < (int)h ? run : (int)h;
                const int mid = run > (int)h ? (run - (int)h) & ~3 : 0;
                const int tail0 = head + mid;
                float *yc = y_unit + co * cstride;
                const float *sc = ost + co * CH + off;
                if (lane < head) yc[lane] = sc[lane];
                if (tail0 + lane < run) yc[tail0 + lane] = sc[tail0 + lane];
            }
        } else {
            for (int co = warp; co < COUT; co += WARPS) {
                float *yc = y_unit + co * cstride + ow0;
                const float *sc = ost + co * CH;
                for (int e = lane; e < rows * cols; e += 32) {
                    const int r = e / cols, c = e - r * cols;
                    yc[(long long)r * Wo + c] = sc[r * WB + c];
                }
            }
        }
        if (more) cur = unit(u + gridDim.x);
    }
    if (tid == 0) bulk_wait<0>();
}

aps_status launch_convt3d_k3s2p1(const float *x, const int64_t in[5], const float *w,
                                 const float *bias, float *y, const int64_t out[5],
                                 cudaStream_t st) {
    using namespace c3;
    const int64_t N = in[0], Cin = in[1], D = in[2], H = in[3], W = in[4];
    const int64_t Do = out[2], Ho = out[3], Wo = out[4];
    if (Cin < 1 || Cin > CIN_MAX || W % 4 != 0 || reinterpret_cast<uintptr_t>(x) % 16 != 0 ||
        D >= (1 << 30) || H >= (1 << 30) || W >= (1 << 30) || N * Cin >= (1ll << 31))
        return APS_ERR_UNSUPPORTED;
    const int WB = (int)std::min<int64_t>(Wo, OC);
    const int64_t n_mhb = ceil_div(ceil_div(Ho, 2), MH), n_mwb = ceil_div(ceil_div(Wo, 2), MW);
    const long long n_units = N * Do * n_mhb * n_mwb;
    CUtensorMap map;
    const cuuint64_t dims[4] = {(cuuint64_t)W, (cuuint64_t)H, (cuuint64_t)D, (cuuint64_t)(N * Cin)};
    const cuuint64_t strides[3] = {(cuuint64_t)(W * 4), (cuuint64_t)(H * W * 4),
                                   (cuuint64_t)(D * H * W * 4)};
    const cuuint32_t box[4] = {(cuuint32_t)XC, (cuuint32_t)XR, 2, (cuuint32_t)Cin};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    if (!encode_tiled(&map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<float *>(x), dims,
                      strides, box, estr))
        return APS_ERR_UNSUPPORTED;
    const size_t smem = (size_t)(2 * stage_stride_of((int)Cin) +
                                 ((COUT * chan_stride_of(WB) + 31) & ~31) + Cin * 27 * COUT +
                                 COUT) * 4 + 16;
    const int per_sm = resident_ctas((const void *)convt3d_k3s2p1_kernel, THREADS, (int)smem);
    if (per_sm < 1) return APS_ERR_UNSUPPORTED;
    const long long grid = std::min<long long>((long long)per_sm * sm_count(), n_units);
    const cudaError_t e = launch_pdl(convt3d_k3s2p1_kernel, dim3((unsigned)grid), dim3(THREADS), smem, st, map, w, bias,
               y, (int)Cin, (int)D, (int)H, (int)W, (int)Do, (int)Ho, (int)Wo, WB, (int)n_mhb,
               (int)n_mwb, n_units, status_word());
    return launch_status(e);
}

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
