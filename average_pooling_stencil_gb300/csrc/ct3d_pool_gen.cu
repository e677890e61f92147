// ct3d_pool_gen.cu -- the fused ConvTranspose3d -> x scale1 -> AvgPool3d(q) ->
// + bias -> x scale2 op for any geometry (kernel, stride, padding, dilation,
// output padding per dim; any pool size q; any channel counts).
//
// Kimi-K2.6__l2_p50 derives, for its k3 s2 p1 / pool 2 model, that a pooled
// output reads a fixed 2x2x2 neighbourhood of the input with 8 collapsed
// weights (the 27 taps grouped by the input cell they read), and sketches the
// same idea for other geometries.  Written out per dim: pooled output P covers
// the pre-pool positions o in [qP, qP + q); tap k of o reads input
// i = (o + p - d*k) / s where that quotient is an integer.  The (i - base, k)
// pattern repeats every T = s / gcd(q, s) pooled outputs (the window moves by
// lcm(q, s) pre-pool positions, i.e. by q*T/s inputs), so per dim and phase
// phi = P mod T there is a short list of input offsets delta, each with the set
// of taps that reaches it.  The pooled output is then
//   y[n,co,P] = bias' + sum_ci sum_delta x[n,ci,base(P) + delta] * Weff[phi][ci][co][delta]
// with Weff the sum of w over each delta's taps (per dim, the product of the
// three dims' tap sets) times scale1*scale2/q^3, and bias' = (conv_bias*scale1 +
// bias)*scale2.  Input cells outside the tensor contribute nothing (they are
// the transposed convolution's missing terms, not zero padding of x).
//
// Tiled kernel: geometries with one phase per dim, the window moving one input
// per pooled output and at most 3 offsets per dim (some dim with 3) -- e.g. 4-tap
// kernels at stride 2 with pool 2 -- run as a tiled 3x3x3 correlation (below).
//
// Kernel: each CTA builds Weff for all phase combinations in shared memory
// (host-built per-dim tables come in the launch parameters), then each thread
// takes one pooled position and accumulates 16 output channels at a time in
// registers: one input load feeds 16 FMAs whose weights are a broadcast
// 16-float shared-memory read when the warp's threads share a phase (always
// for q a multiple of s).  Threads run along the pooled W axis, so input and
// output accesses are coalesced.  Geometries whose tables exceed the limits
// below fall back to the per-output direct kernel in ct3d_pool.cu.
#include <algorithm>

#include "aps_dev.cuh"
#include "aps_internal.h"

namespace aps {
namespace gen {
constexpr int MAX_PHASE = 8;    // T = s / gcd(q, s)
constexpr int MAX_DELTA = 8;    // input offsets per phase
constexpr int MAX_TAPS = 32;    // kernel size per dim (tap sets are bit masks)
constexpr int CO_T = 16;        // output channels per register block
constexpr int THREADS = 128;
constexpr int MAX_WEFF_BYTES = 96 * 1024;

struct Dim {
    int T;                               // phases
    int step;                            // input advance per T pooled outputs
    int md;                              // max offsets over the phases
    int nd[MAX_PHASE];                   // offsets of each phase
    int i0[MAX_PHASE];                   // first input of phase phi at P = phi
    uint32_t kmask[MAX_PHASE][MAX_DELTA];  // taps reaching each offset
};
struct Geom {
    Dim d[3];
};

// Sum of w[ci][co][kd][kh][kw] over the three tap sets (bit masks).
__device__ __forceinline__ float tap_set_sum(const float *__restrict__ wp, int kH, int kW,
                                             uint32_t md, uint32_t mh, uint32_t mw) {
    float acc = 0.f;
    for (uint32_t a = md; a; a &= a - 1) {
        const int kd = __ffs(a) - 1;
        for (uint32_t b = mh; b; b &= b - 1) {
            const int kh = __ffs(b) - 1;
            for (uint32_t c = mw; c; c &= c - 1) {
                const int kw = __ffs(c) - 1;
                acc += __ldg(wp + (kd * kH + kh) * kW + kw);
            }
        }
    }
    return acc;
}
}  // namespace gen

// ND > 0: every phase of every dim reads at most ND input offsets; the cell
// loops are unrolled and the loads of one input channel (ND^3 of them) are all
// in flight before their FMAs.  ND == 0: any count, run-time loops.
template <int ND>
__global__ void __launch_bounds__(gen::THREADS)
    ct3d_pool_gen_kernel(const float *__restrict__ x, const float *__restrict__ w,
                         const float *__restrict__ conv_bias, const float *__restrict__ bias,
                         float wscale, float scale1, float scale2, float *__restrict__ y,
                         long long n_pos, int Cin, int Cout, int COP, int D, int H, int W,
                         int Do, int Ho, int Wo, int kD, int kH, int kW,
                         const __grid_constant__ gen::Geom g) {
    using namespace gen;
    pdl_trigger();
    pdl_wait();
    extern __shared__ __align__(16) float weff[];   // [combo][ci][dd][dh][dw][COP]
    const Dim &GD = g.d[0], &GH = g.d[1], &GW = g.d[2];
    const int MD = GD.md, MH = GH.md, MW = GW.md;
    const int taps = MD * MH * MW;
    const int combos = GD.T * GH.T * GW.T;
    // ---- collapsed weights (scaled by scale1 * scale2 / q^3)
    const long long total = (long long)combos * Cin * taps * COP;
    for (long long e = threadIdx.x; e < total; e += blockDim.x) {
        long long t = e;
        const int co = (int)(t % COP);
        t /= COP;
        const int tw = (int)(t % MW);
        t /= MW;
        const int th = (int)(t % MH);
        t /= MH;
        const int td = (int)(t % MD);
        t /= MD;
        const int ci = (int)(t % Cin);
        const int combo = (int)(t / Cin);
        const int fw = combo % GW.T, fh = (combo / GW.T) % GH.T, fd = combo / (GW.T * GH.T);
        float v = 0.f;
        if (co < Cout && td < GD.nd[fd] && th < GH.nd[fh] && tw < GW.nd[fw])
            v = tap_set_sum(w + ((long long)ci * Cout + co) * kD * kH * kW, kH, kW,
                            GD.kmask[fd][td], GH.kmask[fh][th], GW.kmask[fw][tw]) *
                wscale;
        weff[e] = v;
    }
    __syncthreads();

    const long long in_plane = (long long)D * H * W;
    const long long out_plane = (long long)Do * Ho * Wo;
    for (long long pos = blockIdx.x * (long long)blockDim.x + threadIdx.x; pos < n_pos;
         pos += (long long)gridDim.x * blockDim.x) {
        const int pw = (int)(pos % Wo);
        long long t = pos / Wo;
        const int ph = (int)(t % Ho);
        t /= Ho;
        const int pd = (int)(t % Do);
        const long long n = t / Do;
        const int fd = pd % GD.T, fh = ph % GH.T, fw = pw % GW.T;
        const int bd = (pd / GD.T) * GD.step + GD.i0[fd];
        const int bh = (ph / GH.T) * GH.step + GH.i0[fh];
        const int bw = (pw / GW.T) * GW.step + GW.i0[fw];
        // offsets of this position that land inside the input
        const int d0 = max(0, -bd), d1 = min(GD.nd[fd], D - bd);
        const int h0 = max(0, -bh), h1 = min(GH.nd[fh], H - bh);
        const int w0 = max(0, -bw), w1 = min(GW.nd[fw], W - bw);
        const int combo = (fd * GH.T + fh) * GW.T + fw;
        const float *xn = x + n * Cin * in_plane;
        float *yp = y + n * Cout * out_plane + ((long long)pd * Ho + ph) * Wo + pw;
        // ND > 0: the cells of this position (offsets within an input plane and
        // whether they lie inside it) once, for every channel block and input
        // channel
        constexpr int NC = ND > 0 ? ND * ND * ND : 1;
        int coff[NC];
        unsigned cin_mask = 0;
        if constexpr (ND > 0) {
#pragma unroll
            for (int a = 0; a < ND; ++a)
#pragma unroll
                for (int b = 0; b < ND; ++b)
#pragma unroll
                    for (int c = 0; c < ND; ++c) {
                        const int e = (a * ND + b) * ND + c;
                        const bool in = a >= d0 && a < d1 && b >= h0 && b < h1 && c >= w0 &&
                                        c < w1;
                        coff[e] = in ? ((bd + a) * H + (bh + b)) * W + (bw + c) : 0;
                        cin_mask |= (in ? 1u : 0u) << e;
                    }
        }
        for (int co0 = 0; co0 < Cout; co0 += CO_T) {
            float acc[CO_T];
#pragma unroll
            for (int j = 0; j < CO_T; ++j) acc[j] = 0.f;
            if constexpr (ND > 0) {
                // channel pairs by the packed fp32x2 FMA (two exactly rounded FMAs
                // per instruction)
                float2 acc2[CO_T / 2];
#pragma unroll
                for (int j = 0; j < CO_T / 2; ++j) acc2[j] = make_float2(0.f, 0.f);
                // the cells of input channel ci + 1 load while channel ci's FMAs
                // run (two register sets, the loop unrolled by two)
                auto load = [&](float (&xv)[NC], int ci) {
                    const float *xc = xn + ci * in_plane;
#pragma unroll
                    for (int e = 0; e < NC; ++e)
                        xv[e] = (cin_mask >> e) & 1u ? __ldg(xc + coff[e]) : 0.f;
                };
                auto fma = [&](const float (&xv)[NC], int ci) {
                    const float *wc = weff + ((long long)(combo * Cin + ci) * NC) * COP + co0;
#pragma unroll
                    for (int e = 0; e < NC; ++e) {
                        const float4 *w4 = reinterpret_cast<const float4 *>(wc + e * COP);
                        const float2 xx = make_float2(xv[e], xv[e]);
#pragma unroll
                        for (int j = 0; j < CO_T / 4; ++j) {
                            const float4 q4 = w4[j];
                            acc2[2 * j] = __ffma2_rn(xx, make_float2(q4.x, q4.y), acc2[2 * j]);
                            acc2[2 * j + 1] =
                                __ffma2_rn(xx, make_float2(q4.z, q4.w), acc2[2 * j + 1]);
                        }
                    }
                };
                float xa[NC], xb[NC];
                if (Cin > 0) load(xa, 0);
                for (int ci = 0; ci < Cin; ci += 2) {
                    if (ci + 1 < Cin) load(xb, ci + 1);
                    fma(xa, ci);
                    if (ci + 1 >= Cin) break;
                    if (ci + 2 < Cin) load(xa, ci + 2);
                    fma(xb, ci + 1);
                }
#pragma unroll
                for (int j = 0; j < CO_T / 2; ++j) {
                    acc[2 * j] = acc2[j].x;
                    acc[2 * j + 1] = acc2[j].y;
                }
            } else {
                for (int ci = 0; ci < Cin; ++ci) {
                    const float *xc = xn + ci * in_plane;
                    const float *wc = weff + ((long long)(combo * Cin + ci) * taps) * COP + co0;
                    for (int a = d0; a < d1; ++a)
                        for (int b = h0; b < h1; ++b) {
                            const float *xr = xc + ((long long)(bd + a) * H + (bh + b)) * W + bw;
                            const float *wr = wc + ((a * MH + b) * MW) * COP;
                            for (int c = w0; c < w1; ++c) {
                                const float xv = __ldg(xr + c);
                                const float4 *w4 = reinterpret_cast<const float4 *>(wr + c * COP);
#pragma unroll
                                for (int j = 0; j < CO_T / 4; ++j) {
                                    const float4 q4 = w4[j];
                                    acc[4 * j + 0] = fmaf(xv, q4.x, acc[4 * j + 0]);
                                    acc[4 * j + 1] = fmaf(xv, q4.y, acc[4 * j + 1]);
                                    acc[4 * j + 2] = fmaf(xv, q4.z, acc[4 * j + 2]);
                                    acc[4 * j + 3] = fmaf(xv, q4.w, acc[4 * j + 3]);
                                }
                            }
                        }
                }
            }
#pragma unroll
            for (int j = 0; j < CO_T; ++j) {
                const int co = co0 + j;
                if (co < Cout) {
                    const float cb = conv_bias ? __ldg(conv_bias + co) : 0.f;
                    yp[(long long)co * out_plane] =
                        acc[j] + (cb * scale1 + __ldg(bias + co)) * scale2;
                }
            }
        }
    }
}

// ---------------------------------------------------------------- tiled form
// Geometries with one phase per dim and the window moving one input per pooled
// output (pool size = stride), at most 3 input offsets per dim: the pooled
// output is a plain 3x3x3 correlation of the input (zero outside it) from its
// origin P + i0, so it is tiled like the pages' k3 s2 p1 geometry.  A CTA of 8
// warps takes units of 16 pooled rows x 32 pooled columns of one (n, pd) plane
// and one 16-channel output block; the unit's input -- C_in channels x 3 planes
// x 18 rows x 40 columns from the origin, its x coordinate rounded down to a
// multiple of 4 (a TMA box must start 16-byte aligned) -- is one 4-D TMA box,
// double-buffered behind mbarriers with bounded waits.  Warp w owns pooled rows
// 2w, 2w+1 and lane l pooled column l, all 16 channels of the block: per input
// channel a thread reads its 3 x 4 x 3 window once and applies the 27 taps with
// broadcast float4 weight reads and packed fp32x2 FMAs.  Outputs leave by
// whole-warp stores of 32 consecutive columns per channel row.
namespace gent {
constexpr int WARPS = 8, THREADS = 32 * WARPS;
constexpr int RB = 2 * WARPS;       // pooled rows per unit
constexpr int WB = 32;              // pooled columns per unit
constexpr int XR = RB + 2;          // staged rows
constexpr int BW = 40;              // staged columns: 32 + 2, shifted by up to 3
constexpr int NT = 27;              // taps (3 x 3 x 3)
constexpr int CO_T = 16;
__host__ __device__ inline int stage_stride_of(int Cin) { return (Cin * 3 * XR * BW + 31) & ~31; }
}  // namespace gent

__global__ void __launch_bounds__(gent::THREADS, 2)
    ct3d_pool_gen_tiled_kernel(const __grid_constant__ CUtensorMap xmap,
                               const float *__restrict__ w, const float *__restrict__ conv_bias,
                               const float *__restrict__ bias, float wscale, float scale1,
                               float scale2, float *__restrict__ y, int Cin, int Cout, int COP,
                               int Do, int Ho, int Wo, int kD, int kH, int kW, int i0d, int i0h,
                               int i0w, int n_cob, int n_hb, int n_wb, long long n_units,
                               const __grid_constant__ gen::Geom g, unsigned int *status) {
    using namespace gent;
    pdl_trigger();
    pdl_wait();
    extern __shared__ __align__(128) float smt[];
    const int stage_stride = stage_stride_of(Cin);
    float *xs = smt;                                  // [2][Cin][3][XR][BW]
    float *wsm = xs + 2 * stage_stride;               // [Cin][27][COP]
    float *bsm = wsm + (size_t)Cin * NT * COP;        // [COP]
    uint64_t *bar = reinterpret_cast<uint64_t *>(bsm + COP);   // [2]
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t stage_bytes = (uint32_t)(Cin * 3 * XR * BW) * 4u;

    struct Unit {
        long long n;
        int cob, pd, ph0, pw0;
    };
    auto unit = [&](long long u) {
        Unit t;
        t.cob = (int)(u % n_cob);
        long long r = u / n_cob;
        t.pw0 = (int)(r % n_wb) * WB;
        r /= n_wb;
        t.ph0 = (int)(r % n_hb) * RB;
        r /= n_hb;
        t.pd = (int)(r % Do);
        t.n = r / Do;
        return t;
    };
    // the box origin's x rounded down to a multiple of 4; the thread then reads
    // from column (origin - rounded) + lane
    auto stage = [&](const Unit &t, int b) {
        if (tid == 0) {
            const int x0 = (t.pw0 + i0w) & ~3;
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            mbar_arrive_expect_tx(&bar[b], stage_bytes);
            tma_load_4d(xs + b * stage_stride, &xmap, &bar[b], x0, t.ph0 + i0h, t.pd + i0d,
                        (int)(t.n * Cin));
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
    // ---- collapsed weights [ci][tap][co] (scaled) and the folded bias, once per CTA
    const gen::Dim &GD = g.d[0], &GH = g.d[1], &GW = g.d[2];
    for (int e = tid; e < Cin * NT * COP; e += THREADS) {
        const int co = e % COP, tap = (e / COP) % NT, ci = e / (COP * NT);
        const int a = tap / 9, b = (tap / 3) % 3, c = tap % 3;
        float v = 0.f;
        if (co < Cout && a < GD.nd[0] && b < GH.nd[0] && c < GW.nd[0])
            v = gen::tap_set_sum(w + ((long long)ci * Cout + co) * kD * kH * kW, kH, kW,
                                 GD.kmask[0][a], GH.kmask[0][b], GW.kmask[0][c]) * wscale;
        wsm[e] = v;
    }
    for (int co = tid; co < COP; co += THREADS) {
        const float cb = co < Cout && conv_bias ? __ldg(conv_bias + co) : 0.f;
        bsm[co] = co < Cout ? (cb * scale1 + __ldg(bias + co)) * scale2 : 0.f;
    }
    __syncthreads();

    const long long plane = (long long)Ho * Wo;
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
            return;
        }
        const int co0 = cur.cob * CO_T;
        float2 acc[CO_T / 2][2];
#pragma unroll
        for (int c2 = 0; c2 < CO_T / 2; ++c2) {
            const float2 bv = make_float2(bsm[co0 + 2 * c2], bsm[co0 + 2 * c2 + 1]);
            acc[c2][0] = bv;
            acc[c2][1] = bv;
        }
        const int shift = (cur.pw0 + i0w) - ((cur.pw0 + i0w) & ~3);
        const float *xb = xs + b * stage_stride + (2 * warp) * BW + shift + lane;
#pragma unroll 1
        for (int ci = 0; ci < Cin; ++ci) {
            float xv[3][4][3];
#pragma unroll
            for (int a = 0; a < 3; ++a)
#pragma unroll
                for (int rr = 0; rr < 4; ++rr)
#pragma unroll
                    for (int c = 0; c < 3; ++c)
                        xv[a][rr][c] = xb[((ci * 3 + a) * XR + rr) * BW + c];
            const float4 *wq = reinterpret_cast<const float4 *>(wsm + (size_t)ci * NT * COP + co0);
#pragma unroll
            for (int tap = 0; tap < NT; ++tap) {
                const int a = tap / 9, bb = (tap / 3) % 3, c = tap % 3;
                const float4 *wt = wq + tap * (COP / 4);
                const float4 w0 = wt[0], w1 = wt[1], w2 = wt[2], w3 = wt[3];
                const float2 wp[CO_T / 2] = {make_float2(w0.x, w0.y), make_float2(w0.z, w0.w),
                                             make_float2(w1.x, w1.y), make_float2(w1.z, w1.w),
                                             make_float2(w2.x, w2.y), make_float2(w2.z, w2.w),
                                             make_float2(w3.x, w3.y), make_float2(w3.z, w3.w)};
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const float xg = xv[a][i + bb][c];
#pragma unroll
                    for (int c2 = 0; c2 < CO_T / 2; ++c2)
                        acc[c2][i] = __ffma2_rn(make_float2(xg, xg), wp[c2], acc[c2][i]);
                }
            }
        }
        // ---- outputs: per channel and row, one whole-warp store of 32 columns
        const int pw = cur.pw0 + lane;
        float *yb = y + ((cur.n * Cout) * Do + cur.pd) * plane;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int ph = cur.ph0 + 2 * warp + i;
            if (ph < Ho && pw < Wo) {
                float *yr = yb + (long long)ph * Wo + pw;
#pragma unroll
                for (int c2 = 0; c2 < CO_T / 2; ++c2) {
                    const int co = co0 + 2 * c2;
                    if (co < Cout) yr[(long long)co * Do * plane] = acc[c2][i].x;
                    if (co + 1 < Cout) yr[(long long)(co + 1) * Do * plane] = acc[c2][i].y;
                }
            }
        }
        // every thread is done with stage b before the next iteration refills it
        __syncthreads();
        if (more) cur = unit(u + gridDim.x);
    }
}

namespace {
int gcd_i(int a, int b) {
    while (b) {
        const int t = a % b;
        a = b;
        b = t;
    }
    return a;
}
int floordiv_i(int a, int b) { return a >= 0 ? a / b : -((-a + b - 1) / b); }

// Per-dim phase tables; false if the geometry exceeds the table limits.
bool build_dim(int K, int s, int p, int d, int q, gen::Dim &t) {
    using namespace gen;
    if (K > MAX_TAPS) return false;
    const int g = gcd_i(q, s);
    t = gen::Dim{};
    t.T = s / g;
    t.step = q / g;
    if (t.T > MAX_PHASE) return false;
    t.md = 0;
    for (int f = 0; f < t.T; ++f) {
        int lo = 1 << 30, hi = -(1 << 30);
        for (int o = q * f; o < q * f + q; ++o)
            for (int k = 0; k < K; ++k) {
                const long long num = (long long)o + p - (long long)d * k;
                if (((num % s) + s) % s) continue;
                const int i = floordiv_i((int)num, s);
                lo = std::min(lo, i);
                hi = std::max(hi, i);
            }
        if (lo > hi) {   // no tap reaches this phase: bias only
            t.nd[f] = 0;
            t.i0[f] = 0;
            continue;
        }
        if (hi - lo + 1 > MAX_DELTA) return false;
        t.nd[f] = hi - lo + 1;
        t.i0[f] = lo;
        t.md = std::max(t.md, t.nd[f]);
        for (int o = q * f; o < q * f + q; ++o)
            for (int k = 0; k < K; ++k) {
                const long long num = (long long)o + p - (long long)d * k;
                if (((num % s) + s) % s) continue;
                t.kmask[f][floordiv_i((int)num, s) - lo] |= 1u << k;
            }
    }
    if (t.md == 0) t.md = 1;
    return true;
}
}  // namespace

aps_status launch_ct3d_pool_gen(const float *x, const int64_t in[5], const float *w,
                                const float *conv_bias, const float *bias, int64_t c_out,
                                const int k[3], const int s[3], const int p[3], const int d[3],
                                int pool_k, float scale1, float scale2, float *y,
                                const int64_t out[5], cudaStream_t st) {
    using namespace gen;
    if (pool_k > 64) return APS_ERR_UNSUPPORTED;   // o and the tap loops stay small
    // cell offsets within an input plane in 32 bits
    if (in[2] * in[3] * in[4] >= ((int64_t)1 << 31)) return APS_ERR_UNSUPPORTED;
    gen::Geom g;
    for (int i = 0; i < 3; ++i)
        if (!build_dim(k[i], s[i], p[i], d[i], pool_k, g.d[i])) return APS_ERR_UNSUPPORTED;
    const int COP = (int)((c_out + CO_T - 1) / CO_T) * CO_T;
    // one phase per dim, the window moving one input per pooled output, at most 3
    // input offsets per dim: the tiled 3x3x3 form (TMA-staged, 16-byte input rows)
    bool tiled = in[1] <= 8 && in[4] % 4 == 0 && reinterpret_cast<uintptr_t>(x) % 16 == 0 &&
                 in[0] * in[1] < ((int64_t)1 << 31) && (int64_t)COP * in[1] * gent::NT * 4 <= 32768;
    for (int i = 0; i < 3; ++i)
        tiled = tiled && g.d[i].T == 1 && g.d[i].step == 1 && g.d[i].md <= 3 && g.d[i].nd[0] > 0;
    // (at most 2 offsets in every dim: the unrolled 2 x 2 x 2 kernel below does a third
    // of the multiply-adds)
    tiled = tiled && (g.d[0].md == 3 || g.d[1].md == 3 || g.d[2].md == 3);
    if (tiled) {
        const int Cin = (int)in[1];
        const size_t smem_t = ((size_t)2 * gent::stage_stride_of(Cin) +
                               (size_t)Cin * gent::NT * COP + COP) * 4 + 16;
        const int per_sm_t = resident_ctas((const void *)ct3d_pool_gen_tiled_kernel, gent::THREADS,
                                           (int)smem_t);
        CUtensorMap map;
        const cuuint64_t dims[4] = {(cuuint64_t)in[4], (cuuint64_t)in[3], (cuuint64_t)in[2],
                                    (cuuint64_t)(in[0] * in[1])};
        const cuuint64_t strides[3] = {(cuuint64_t)(in[4] * 4), (cuuint64_t)(in[3] * in[4] * 4),
                                       (cuuint64_t)(in[2] * in[3] * in[4] * 4)};
        const cuuint32_t box[4] = {(cuuint32_t)gent::BW, (cuuint32_t)gent::XR, 3, (cuuint32_t)Cin};
        const cuuint32_t estr[4] = {1, 1, 1, 1};
        if (per_sm_t >= 1 && encode_tiled(&map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4,
                                          const_cast<float *>(x), dims, strides, box, estr)) {
            const int n_cob = COP / gent::CO_T;
            const int64_t n_hb = ceil_div(out[3], (int64_t)gent::RB);
            const int64_t n_wb = ceil_div(out[4], (int64_t)gent::WB);
            const long long n_units = out[0] * out[2] * n_hb * n_wb * n_cob;
            const long long grid = std::min<long long>((long long)per_sm_t * sm_count(), n_units);
            const float q3 = (float)pool_k * pool_k * pool_k;
            const cudaError_t e = launch_pdl(
                ct3d_pool_gen_tiled_kernel, dim3((unsigned)grid), dim3(gent::THREADS), smem_t, st,
                map, w, conv_bias, bias, scale1 * scale2 / q3, scale1, scale2, y, Cin, (int)c_out,
                COP, (int)out[2], (int)out[3], (int)out[4], k[0], k[1], k[2], g.d[0].i0[0],
                g.d[1].i0[0], g.d[2].i0[0], n_cob, (int)n_hb, (int)n_wb, n_units, g,
                status_word());
            return launch_status(e);
        }
    }
    // offsets per phase at most 2 in every dim (the pages' geometry and its
    // pool variants), or at most 3 (4-tap kernels at stride 2, pool 2): unrolled
    // cells, Weff laid out ND x ND x ND per (ci, phase); the rest run-time loops
    int nd = 0;
    if (g.d[0].md <= 2 && g.d[1].md <= 2 && g.d[2].md <= 2)
        nd = 2;
    else if (g.d[0].md <= 3 && g.d[1].md <= 3 && g.d[2].md <= 3)
        nd = 3;
    if (nd)
        for (int i = 0; i < 3; ++i) g.d[i].md = nd;
    const long long weff_floats = (long long)g.d[0].T * g.d[1].T * g.d[2].T * in[1] * g.d[0].md *
                            g.d[1].md * g.d[2].md * COP;
    if (weff_floats * 4 > MAX_WEFF_BYTES) return APS_ERR_UNSUPPORTED;
    const int smem = (int)std::max<long long>(16, weff_floats * 4);
    const auto kern = nd == 2 ? ct3d_pool_gen_kernel<2>
                    : nd == 3 ? ct3d_pool_gen_kernel<3>
                              : ct3d_pool_gen_kernel<0>;
    const int per_sm = resident_ctas((const void *)kern, THREADS, smem);
    if (per_sm < 1) return APS_ERR_UNSUPPORTED;
    const long long n_pos = out[0] * out[2] * out[3] * out[4];
    const long long grid =
        std::max<long long>(1, std::min<long long>(ceil_div(n_pos, THREADS),
                                                   (long long)sm_count() * per_sm));
    const float q3 = (float)pool_k * pool_k * pool_k;
    const float wscale = scale1 * scale2 / q3;
    const cudaError_t e = launch_pdl(
        kern, dim3((unsigned)grid), dim3(THREADS), (size_t)smem, st, x, w,
        conv_bias, bias, wscale, scale1, scale2, y, n_pos, (int)in[1], (int)c_out, COP,
        (int)in[2], (int)in[3], (int)in[4], (int)out[2], (int)out[3], (int)out[4], k[0], k[1],
        k[2], g);
    return launch_status(e);
}

}  // namespace aps
