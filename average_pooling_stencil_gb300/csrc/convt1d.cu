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
// (all s classes, i.e. 32*Q*s consecutive outputs) for one batch row, where Q
// is 8 divided by the number of classes that have taps (8 for stride 1 and
// for the stride-2, dilation-2 case).  Input
// channels stream through shared memory in chunks of 8 with double-buffered
// cp.async: the x window of the chunk (256 + span samples, zero-filled outside
// [0, L)) and its weights, stored [ci][k][co] so a thread's 8 channels are two
// float4 broadcast reads.  A warp owns 8 output channels and each lane Q
// consecutive m: per input channel the lane loads its window (Q + span samples,
// shared-memory rows padded by one word per 32 so the stride-8 lane pattern is
// conflict-free) into registers and does 8 x Q x K' FMAs per class from it.
// Results leave as 128-bit stores of Q*s consecutive outputs per channel.
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
constexpr int CI_C = 8;                 // input channels per staged chunk

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
    static constexpr int TM = 32 * Q;                    // m positions per CTA
    static constexpr int E_MIN = any() ? emin() : 0;
    static constexpr int SPAN = any() ? emax() - emin() : 0;
    static constexpr int XW = TM + SPAN;                 // window samples per channel
    static constexpr int XW_PAD = XW + XW / 32 + 1;      // padded row length
};

__device__ __forceinline__ int padidx(int j) { return j + (j >> 5); }
}  // namespace ct1

template <int S, int K, int DIL, int PL>
__global__ void __launch_bounds__(ct1::THREADS, 2)
    convt1d_tiled_kernel(const float *__restrict__ x, const float *__restrict__ w,
                         const float *__restrict__ bias, float *__restrict__ y, int Cin,
                         int Cout, int L, int L_out, int ph, int vec_store) {
    using namespace ct1;
    using T = Taps<S, K, DIL, PL>;
    constexpr int XW = T::XW, XW_PAD = T::XW_PAD, SPAN = T::SPAN, E_MIN = T::E_MIN;
    constexpr int Q = T::Q, TM = T::TM;
    constexpr int XS = CI_C * XW_PAD;             // floats per x stage
    constexpr int WS = CI_C * K * CO_B;           // floats per w stage
    extern __shared__ __align__(16) float sm[];
    float *xs = sm;                 // [2][CI_C][XW_PAD]
    float *ws = sm + 2 * XS;        // [2][CI_C][K][CO_B]

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const long long m0 = (long long)blockIdx.x * TM;
    const int co_base = blockIdx.y * CO_B;
    const long long n = blockIdx.z;
    const long long i_lo = m0 + ph + E_MIN;       // input index of window sample 0
    const float *xn = x + n * (long long)Cin * L;

    auto stage = [&](int c0, int b) {
        float *xd = xs + b * XS;
        float *wd = ws + b * WS;
        const int nci = min(CI_C, Cin - c0);
        for (int e = tid; e < CI_C * XW; e += THREADS) {
            const int cl = e / XW, j = e - cl * XW;
            const long long i = i_lo + j;
            const bool in = cl < nci && i >= 0 && i < L;
            const float *src = in ? xn + (long long)(c0 + cl) * L + i : x;
            float *dst = xd + cl * XW_PAD + padidx(j);
            asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(smem_u32(dst)),
                         "l"(src), "r"(in ? 4 : 0)
                         : "memory");
        }
        for (int e = tid; e < CI_C * CO_B * K; e += THREADS) {
            // global order [ci][co][k]; shared order [ci][k][co]
            const int cl = e / (CO_B * K), rem = e - cl * (CO_B * K);
            const int col = rem / K, k = rem - col * K;
            const int co = co_base + col;
            const bool in = cl < nci && co < Cout;
            const float *src = in ? w + ((long long)(c0 + cl) * Cout + co) * K + k : w;
            float *dst = wd + (cl * K + k) * CO_B + col;
            asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(smem_u32(dst)),
                         "l"(src), "r"(in ? 4 : 0)
                         : "memory");
        }
    };

    float acc[CO_T][Q][S];
#pragma unroll
    for (int c = 0; c < CO_T; ++c)
#pragma unroll
        for (int q = 0; q < Q; ++q)
#pragma unroll
            for (int r = 0; r < S; ++r) acc[c][q][r] = 0.f;

    const int nchunks = (Cin + CI_C - 1) / CI_C;
    stage(0, 0);
    cp_async_commit();
    for (int ch = 0; ch < nchunks; ++ch) {
        const int b = ch & 1;
        if (ch + 1 < nchunks) stage((ch + 1) * CI_C, b ^ 1);
        cp_async_commit();
        cp_async_wait<1>();
        __syncthreads();
        const float *xb = xs + b * XS;
        const float *wb = ws + b * WS + warp * CO_T;
        const int nci = min(CI_C, Cin - ch * CI_C);
#pragma unroll 1
        for (int cl = 0; cl < nci; ++cl) {
            float xr[Q + SPAN];
            const float *xrow = xb + cl * XW_PAD;
#pragma unroll
            for (int j = 0; j < Q + SPAN; ++j) xr[j] = xrow[padidx(lane * Q + j)];
#pragma unroll
            for (int k = 0; k < K; ++k) {
                const float4 wa = *reinterpret_cast<const float4 *>(wb + (cl * K + k) * CO_B);
                const float4 wc = *reinterpret_cast<const float4 *>(wb + (cl * K + k) * CO_B + 4);
                const float wv[CO_T] = {wa.x, wa.y, wa.z, wa.w, wc.x, wc.y, wc.z, wc.w};
#pragma unroll
                for (int r = 0; r < S; ++r) {
                    if (!T::has(r, k)) continue;
                    const int off = T::e(r, k) - E_MIN;
#pragma unroll
                    for (int q = 0; q < Q; ++q)
#pragma unroll
                        for (int c = 0; c < CO_T; ++c)
                            acc[c][q][r] = fmaf(xr[q + off], wv[c], acc[c][q][r]);
                }
            }
        }
        __syncthreads();
    }
    cp_async_wait<0>();

    // ---- epilogue: bias, then 8*S consecutive outputs per channel
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
            for (int r = 0; r < S; ++r)
                v[q * S + r] = T::class_has_taps(r) ? acc[c][q][r] + bv : bv;
        float *yp = y + (n * Cout + co) * (long long)L_out + o0;
        if (vec_store && o0 + Q * S <= L_out) {
#pragma unroll
            for (int t = 0; t < Q * S; t += 4)
                *reinterpret_cast<float4 *>(yp + t) = make_float4(v[t], v[t + 1], v[t + 2], v[t + 3]);
        } else {
#pragma unroll
            for (int t = 0; t < Q * S; ++t)
                if (o0 + t < L_out) yp[t] = v[t];
        }
    }
}

template <int S, int K, int DIL, int PL>
static aps_status launch_tiled(const float *x, const int64_t in[3], const float *w,
                               const float *bias, int64_t c_out, int p, float *y,
                               int64_t l_out, cudaStream_t st) {
    using namespace ct1;
    using T = Taps<S, K, DIL, PL>;
    const int smem = (2 * CI_C * T::XW_PAD + 2 * CI_C * K * CO_B) * 4;
    const auto kern = convt1d_tiled_kernel<S, K, DIL, PL>;
    if (resident_ctas((const void *)kern, THREADS, smem) < 1) return APS_ERR_CUDA;
    const int64_t M = ceil_div(l_out, S);
    const int64_t gx = ceil_div(M, T::TM), gy = ceil_div(c_out, CO_B), gz = in[0];
    if (gx >= ((int64_t)1 << 31) || gy > 65535 || gz > 65535) return APS_ERR_UNSUPPORTED;
    const int vec = (l_out % 4 == 0) && (reinterpret_cast<uintptr_t>(y) % 16 == 0);
    kern<<<dim3((unsigned)gx, (unsigned)gy, (unsigned)gz), THREADS, smem, st>>>(
        x, w, bias, y, (int)in[1], (int)c_out, (int)in[2], (int)l_out, (p - PL) / S, vec);
    return launch_status();
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
    convt1d_direct_kernel<<<(unsigned)blocks, threads, 0, st>>>(
        x, w, bias, y, total, (int)in[1], (int)c_out, (int)in[2], (int)l_out, k, s, p, d);
    return launch_status();
}

}  // namespace aps
