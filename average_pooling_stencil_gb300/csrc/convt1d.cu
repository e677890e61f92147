// convt1d.cu -- ConvTranspose1d in fp32.
//
// Operation (Kimi-K2.6__l1_p74, its gather formula): y[n,co,o] = bias[co] +
// sum_ci sum_k w[ci,co,k] * x[n,ci,(o + p - d*k)/s], a term existing only when
// o + p - d*k is a non-negative multiple of s whose quotient is below L; the
// weights are not flipped.
//
// Per-parity tap sets instead of zero insertion: write o = s*m + r and
// p = s*ph + pl (0 <= r, pl < s).  Tap k reaches class r iff
// (r + pl - d*k) mod s == 0, and then reads input i = m + ph + e(r,k) with
// e(r,k) = (r + pl - d*k)/s.  With (s, K, d, pl) fixed at compile time every
// tap set and offset is a constant, so each class is a dense, stride-1,
// K'-tap correlation over m with no divisibility tests and no wasted FMAs
// (with stride 2, dilation 2 and odd padding the even class has no taps at
// all and is just the bias).
//
// Tiled kernel (GB300): a CTA computes 64 output channels x 32*Q positions of m
// (all s classes, i.e. 32*Q*s consecutive outputs) per unit, where Q is 8
// divided by the number of classes that have taps; it is persistent and walks
// (batch row, m-tile) units.  A warp owns 8 output channels and each lane Q
// consecutive m.  Input channels stream through shared memory in chunks of 8
// (16, through three stages, where the resident weights leave room) with one
// continuous cp.async pipeline over the CTA's (unit, chunk) sequence: warp w
// stages channels w, w + 8 of the chunk's window (32*Q + span samples, zero
// outside [0, L)).  Window rows are padded by one
// word per Q samples, so lane l's j-th window register sits at row offset
// (Q+1)*l + j + j/Q -- an immediate per j -- and, Q+1 being odd, the 32 lanes
// hit 32 different banks.  The weights, stored [ci][k][co] so a warp's 8
// channels are two float4 broadcast reads, are either resident for the whole
// CTA (loaded once) or, when the CTA's [C_in][K][64] slab is too large, staged
// with each chunk.  Accumulators are kept in channel pairs and updated with the
// packed fp32x2 FMA (two exactly rounded fp32 FMAs per instruction), which
// halves the FMA issue slots.  Results leave as 128-bit stores of Q*s
// consecutive outputs per channel.
//
// Direct kernel: one thread per output evaluating the formula as written, for
// any (s, K, d, p).
#include <algorithm>

#include "aps_dev.cuh"
#include "aps_internal.h"

namespace aps {
namespace ct1 {
constexpr int THREADS = 256;
constexpr int WARPS = THREADS / 32;
constexpr int CO_T = 8;                 // output channels per warp
constexpr int CO_B = WARPS * CO_T;      // 64 output channels per CTA
constexpr int CI_C = WARPS;             // input channels per staged chunk (one per warp)
// "wide" staging: 16 channels per chunk through 3 window stages (one CTA barrier
// per chunk instead of two, half as many chunks), used when the resident weights
// leave room for it: 1720 -> 1632 us on the stride-1 K5 workload; the strided K4
// workload's weights leave no room (staging its weights per chunk was slower)
constexpr int CI_W = 2 * WARPS;
constexpr int NB_W = 3;
// Resident weights while the CTA's shared memory stays within this, so that
// two CTAs share an SM.
constexpr int RESIDENT_SMEM = 110 * 1024;

__host__ __device__ constexpr int floordiv(int a, int b) {
    return (a >= 0) ? a / b : -((-a + b - 1) / b);
}
__host__ __device__ constexpr int posmod(int a, int b) { return ((a % b) + b) % b; }

template <int S, int K, int DIL, int PL>
struct Taps {
    __host__ __device__ static constexpr bool has(int r, int k) { return posmod(r + PL - DIL * k, S) == 0; }
    __host__ __device__ static constexpr int e(int r, int k) { return floordiv(r + PL - DIL * k, S); }
    __host__ __device__ static constexpr bool class_has_taps(int r) {
        for (int k = 0; k < K; ++k)
            if (has(r, k)) return true;
        return false;
    }
    __host__ __device__ static constexpr int emin() {
        int v = 1 << 30;
        for (int r = 0; r < S; ++r)
            for (int k = 0; k < K; ++k)
                if (has(r, k) && e(r, k) < v) v = e(r, k);
        return v;
    }
    __host__ __device__ static constexpr int emax() {
        int v = -(1 << 30);
        for (int r = 0; r < S; ++r)
            for (int k = 0; k < K; ++k)
                if (has(r, k) && e(r, k) > v) v = e(r, k);
        return v;
    }
    __host__ __device__ static constexpr bool any() { return emin() <= emax(); }
    __host__ __device__ static constexpr int nclasses() {
        int c = 0;
        for (int r = 0; r < S; ++r) c += class_has_taps(r) ? 1 : 0;
        return c;
    }
    // m positions per lane: 8 accumulators per channel whatever the stride
    static constexpr int Q = nclasses() > 1 ? 8 / nclasses() : 8;
    static constexpr int TM = 32 * Q;                    // m positions per CTA unit
    static constexpr int E_MIN = any() ? emin() : 0;
    static constexpr int SPAN = any() ? emax() - emin() : 0;
    static constexpr int XW = TM + SPAN;                 // window samples per channel
    static constexpr int XP = XW + XW / Q + 1;           // padded row (one word per Q)
    static constexpr int XS = CI_C * XP;                 // floats per window stage
    static constexpr int WC = CI_C * K * CO_B;           // floats of one chunk's weights
    static constexpr int XS_W = CI_W * XP;               // ... with wide staging
};
}  // namespace ct1

template <int S, int K, int DIL, int PL, bool RES, bool WIDE>
__global__ void __launch_bounds__(ct1::THREADS, 2)
    convt1d_tiled_kernel(const float *__restrict__ x, const float *__restrict__ w,
                         const float *__restrict__ bias, float *__restrict__ y, int Cin,
                         int Cout, int L, int L_out, int ph, int n_mtiles, long long n_units,
                         int vec_store) {
    pdl_trigger();
    pdl_wait();
    using namespace ct1;
    using T = Taps<S, K, DIL, PL>;
    static_assert(RES || !WIDE, "wide staging keeps the weights resident");
    constexpr int CIC = WIDE ? CI_W : CI_C;   // channels per chunk
    constexpr int NB = WIDE ? NB_W : 2;       // window stages
    constexpr int XW = T::XW, XP = T::XP, XS = CIC * XP, WC = T::WC;
    constexpr int SPAN = T::SPAN, E_MIN = T::E_MIN, Q = T::Q, TM = T::TM;
    extern __shared__ __align__(16) float sm[];
    // resident: ws = [Cin][K][CO_B]; staged: ws = [2][CI_C][K][CO_B]
    float *ws = sm;
    float *xs = sm + (RES ? (size_t)Cin * K * CO_B : (size_t)2 * WC);   // [NB][CIC][XP]

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int co_base = blockIdx.y * CO_B;
    const int nchunks = (Cin + CIC - 1) / CIC;

    // weights of input channels c0 .. c0+nci-1: global [ci][co][k] -> shared
    // [ci - c0][k][co] (zeros for channels past C_out)
    auto load_w = [&](int c0, int nci, float *dst, bool async) {
        for (int e = tid; e < nci * CO_B * K; e += THREADS) {
            const int cl = e / (CO_B * K), rem = e - cl * (CO_B * K);
            const int col = rem / K, k = rem - col * K;
            const int co = co_base + col;
            const bool in = co < Cout;
            const float *src = in ? w + ((long long)(c0 + cl) * Cout + co) * K + k : w;
            float *d = dst + (cl * K + k) * CO_B + col;
            if (async)
                asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(smem_u32(d)),
                             "l"(src), "r"(in ? 4 : 0)
                             : "memory");
            else
                *d = in ? __ldg(src) : 0.f;
        }
    };
    if (RES) load_w(0, Cin, ws, false);

    // Stage chunk c0 of a unit into buffer b: warp w copies channel c0 + w of
    // the window.  The unit is given by its batch row's first input channel
    // (xn) and its window start i_lo; samples j in [j_lo, j_hi) lie inside
    // [0, L), the rest are zeros.
    auto stage = [&](const float *xn, long long i_lo, int c0, int b) {
        if (!RES) load_w(c0, min(CIC, Cin - c0), ws + b * WC, true);
        const long long rem = (long long)L - i_lo;   // samples left in the row
        const int j_lo = i_lo >= 0 ? 0 : (-i_lo < XW ? (int)-i_lo : XW);
        const int j_hi = rem <= 0 ? 0 : (rem < XW ? (int)rem : XW);
        for (int cw = warp; cw < CIC; cw += WARPS) {
            const bool chan = c0 + cw < Cin;
            const float *src = xn + (long long)(chan ? c0 + cw : 0) * L + i_lo + lane;
            const uint32_t dst = smem_u32(xs + b * XS + cw * XP + lane + lane / Q);
#pragma unroll 3
            for (int j = lane, t = 0; j < XW; j += 32, ++t) {
                const bool in = chan && j >= j_lo && j < j_hi;
                asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(
                                 dst + 4u * (uint32_t)(t * (32 + 32 / Q))),
                             "l"(in ? src + 32 * t : x), "r"(in ? 4 : 0)
                             : "memory");
            }
        }
    };
    auto unit_origin = [&](long long u, const float *&xn, long long &i_lo) {
        const long long n = u / n_mtiles;
        xn = x + n * Cin * (long long)L;
        i_lo = (u - n * n_mtiles) * TM + ph + E_MIN;
    };

    // accumulators in channel pairs: one packed FMA updates channels 2c2 and
    // 2c2+1 of one position
    float2 acc[CO_T / 2][Q][S];
    long long u = blockIdx.x;
    int ch = 0, b = 0;
    const float *xn = x, *xn_next = x;
    long long i_lo = 0, i_lo_next = 0;
    if (u < n_units) {
        unit_origin(u, xn, i_lo);
        stage(xn, i_lo, 0, 0);
    }
    cp_async_commit();
    while (u < n_units) {
        long long un = u;
        int chn = ch + 1;
        xn_next = xn;
        i_lo_next = i_lo;
        if (chn == nchunks) {
            chn = 0;
            un = u + gridDim.x;
            if (un < n_units) unit_origin(un, xn_next, i_lo_next);
        }
        const int bn = b + 1 == NB ? 0 : b + 1;
        if (un < n_units) stage(xn_next, i_lo_next, chn * CIC, bn);
        cp_async_commit();
        cp_async_wait<1>();
        __syncthreads();
        if (ch == 0) {
#pragma unroll
            for (int c2 = 0; c2 < CO_T / 2; ++c2)
#pragma unroll
                for (int q = 0; q < Q; ++q)
#pragma unroll
                    for (int r = 0; r < S; ++r) acc[c2][q][r] = make_float2(0.f, 0.f);
        }
        const float *xl = xs + b * XS + (Q + 1) * lane;
        const float *wb = (RES ? ws + (size_t)ch * CIC * K * CO_B : ws + b * WC) + warp * CO_T;
        const int nci = min(CIC, Cin - ch * CIC);
#pragma unroll 1
        for (int cl = 0; cl < nci; ++cl) {
            float xr[Q + SPAN];
#pragma unroll
            for (int j = 0; j < Q + SPAN; ++j) xr[j] = xl[cl * XP + j + j / Q];
#pragma unroll
            for (int k = 0; k < K; ++k) {
                const float4 wa = *reinterpret_cast<const float4 *>(wb + (cl * K + k) * CO_B);
                const float4 wc = *reinterpret_cast<const float4 *>(wb + (cl * K + k) * CO_B + 4);
                const float2 wp[CO_T / 2] = {make_float2(wa.x, wa.y), make_float2(wa.z, wa.w),
                                             make_float2(wc.x, wc.y), make_float2(wc.z, wc.w)};
#pragma unroll
                for (int r = 0; r < S; ++r) {
                    if (!T::has(r, k)) continue;
                    const int off = T::e(r, k) - E_MIN;
#pragma unroll
                    for (int c2 = 0; c2 < CO_T / 2; ++c2)
#pragma unroll
                        for (int q = 0; q < Q; ++q)
                            acc[c2][q][r] = __ffma2_rn(make_float2(xr[q + off], xr[q + off]),
                                                       wp[c2], acc[c2][q][r]);
                }
            }
        }
        // buffer b is free for the stage issued next iteration (with three stages,
        // the next stage goes to the buffer every warp left before this
        // iteration's barrier)
        if (NB == 2) __syncthreads();
        if (ch == nchunks - 1) {
            // ---- epilogue: bias, then Q*S consecutive outputs per channel
            const long long n = u / n_mtiles;
            const long long m0 = (u - n * n_mtiles) * TM;
            const long long o0 = (m0 + (long long)lane * Q) * S;
#pragma unroll
            for (int c = 0; c < CO_T; ++c) {
                const int co = co_base + warp * CO_T + c;
                if (co >= Cout) break;
                const float bv = bias ? __ldg(bias + co) : 0.f;
                float v[Q * S];
#pragma unroll
                for (int q = 0; q < Q; ++q)
#pragma unroll
                    for (int r = 0; r < S; ++r) {
                        const float a = (c & 1) ? acc[c / 2][q][r].y : acc[c / 2][q][r].x;
                        v[q * S + r] = T::class_has_taps(r) ? a + bv : bv;
                    }
                float *yp = y + (n * Cout + co) * (long long)L_out + o0;
                if (vec_store && o0 + Q * S <= L_out) {
#pragma unroll
                    for (int t = 0; t < Q * S; t += 4)
                        *reinterpret_cast<float4 *>(yp + t) =
                            make_float4(v[t], v[t + 1], v[t + 2], v[t + 3]);
                } else {
#pragma unroll
                    for (int t = 0; t < Q * S; ++t)
                        if (o0 + t < L_out) yp[t] = v[t];
                }
            }
        }
        u = un;
        ch = chn;
        b = bn;
        xn = xn_next;
        i_lo = i_lo_next;
    }
    cp_async_wait<0>();
}

template <int S, int K, int DIL, int PL>
static aps_status launch_tiled(const float *x, const int64_t in[3], const float *w,
                               const float *bias, int64_t c_out, int p, float *y,
                               int64_t l_out, cudaStream_t st) {
    using namespace ct1;
    using T = Taps<S, K, DIL, PL>;
    const int64_t M = ceil_div(l_out, S);
    const int64_t gy = ceil_div(c_out, CO_B), n_mtiles = ceil_div(M, T::TM);
    if (gy > 65535 || n_mtiles >= ((int64_t)1 << 31)) return APS_ERR_UNSUPPORTED;
    const long long n_units = (long long)in[0] * n_mtiles;
    const int vec = (l_out % 4 == 0) && (reinterpret_cast<uintptr_t>(y) % 16 == 0);
    // resident weights when the CTA's slab and two window stages leave room for
    // two CTAs per SM, otherwise weights staged with each chunk
    const int64_t wsmem = (in[1] * K * CO_B + NB_W * T::XS_W) * 4;
    const int64_t rsmem = (in[1] * K * CO_B + 2 * T::XS) * 4;
    const int ssmem = (2 * T::WC + 2 * T::XS) * 4;
    const bool wide = wsmem <= RESIDENT_SMEM && in[1] >= CI_W;
    const bool res = rsmem <= RESIDENT_SMEM;
    const auto kern = wide ? convt1d_tiled_kernel<S, K, DIL, PL, true, true>
                    : res  ? convt1d_tiled_kernel<S, K, DIL, PL, true, false>
                           : convt1d_tiled_kernel<S, K, DIL, PL, false, false>;
    const int smem = wide ? (int)wsmem : res ? (int)rsmem : ssmem;
    const int per_sm = resident_ctas((const void *)kern, THREADS, smem);
    if (per_sm < 1) return APS_ERR_CUDA;
    const long long slots = std::max<long long>(1, (long long)per_sm * sm_count() / gy);
    const long long gx = std::min<long long>(n_units, slots);
    const cudaError_t e = launch_pdl(kern, dim3((unsigned)gx, (unsigned)gy, 1), dim3(THREADS), (size_t)smem, st, x, w,
               bias, y, (int)in[1], (int)c_out, (int)in[2], (int)l_out, (p - PL) / S, (int)n_mtiles,
               n_units, vec);
    return launch_status(e);
}

aps_status launch_convt1d_tiled(const float *x, const int64_t in[3], const float *w,
                                const float *bias, int64_t c_out, int k, int s, int p, int d,
                                float *y, int64_t l_out, cudaStream_t st) {
    if (c_out % 8 != 0 || in[1] >= (1 << 30) || in[2] >= (1 << 30) || l_out >= (1 << 30) ||
        c_out >= (1 << 20))
        return APS_ERR_UNSUPPORTED;
    const int pl = p % s;
    // (stride, taps, dilation, padding mod stride) combinations compiled in.
    if (s == 1 && k == 5 && d == 3) return launch_tiled<1, 5, 3, 0>(x, in, w, bias, c_out, p, y, l_out, st);
    if (s == 1 && k == 3 && d == 1) return launch_tiled<1, 3, 1, 0>(x, in, w, bias, c_out, p, y, l_out, st);
    if (s == 1 && k == 5 && d == 1) return launch_tiled<1, 5, 1, 0>(x, in, w, bias, c_out, p, y, l_out, st);
    if (s == 2 && k == 4 && d == 2 && pl == 1) return launch_tiled<2, 4, 2, 1>(x, in, w, bias, c_out, p, y, l_out, st);
    if (s == 2 && k == 4 && d == 1 && pl == 1) return launch_tiled<2, 4, 1, 1>(x, in, w, bias, c_out, p, y, l_out, st);
    if (s == 2 && k == 3 && d == 1 && pl == 1) return launch_tiled<2, 3, 1, 1>(x, in, w, bias, c_out, p, y, l_out, st);
    return APS_ERR_UNSUPPORTED;
}

// ------------------------------------------------------------ direct kernel
__global__ void convt1d_direct_kernel(const float *__restrict__ x, const float *__restrict__ w,
                                      const float *__restrict__ bias, float *__restrict__ y,
                                      long long total, int Cin, int Cout, int L, int L_out, int K,
                                      int s, int p, int d) {
    pdl_trigger();
    pdl_wait();
    for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        const int o = (int)(idx % L_out);
        const long long t = idx / L_out;
        const int co = (int)(t % Cout);
        const long long n = t / Cout;
        float acc = bias ? __ldg(bias + co) : 0.f;
        for (int ci = 0; ci < Cin; ++ci) {
            const float *xp = x + (n * Cin + ci) * (long long)L;
            const float *wp = w + ((long long)ci * Cout + co) * K;
            for (int k = 0; k < K; ++k) {
                const long long num = (long long)o + p - (long long)d * k;
                if (num < 0 || num % s) continue;
                const long long i = num / s;
                if (i >= L) continue;
                acc = fmaf(__ldg(xp + i), __ldg(wp + k), acc);
            }
        }
        y[idx] = acc;
    }
}

aps_status launch_convt1d_direct(const float *x, const int64_t in[3], const float *w,
                                 const float *bias, int64_t c_out, int k, int s, int p, int d,
                                 float *y, int64_t l_out, cudaStream_t st) {
    if (in[1] >= (1 << 30) || in[2] >= (1 << 30) || l_out >= (1 << 30) || c_out >= (1 << 30))
        return APS_ERR_UNSUPPORTED;
    const long long total = in[0] * c_out * l_out;
    const int threads = 256;
    const long long blocks =
        std::min<long long>(ceil_div(total, threads), (long long)sm_count() * 16);
    const cudaError_t e = launch_pdl(convt1d_direct_kernel, dim3((unsigned)blocks), dim3(threads), 0, st, x, w, bias, y,
               total, (int)in[1], (int)c_out, (int)in[2], (int)l_out, k, s, p, d);
    return launch_status(e);
}

}  // namespace aps
