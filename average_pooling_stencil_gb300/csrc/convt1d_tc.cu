// convt1d_tc.cu -- ConvTranspose1d as a TF32 implicit GEMM on the tcgen05
// tensor cores (APS_PREC_TF32).
//
// Operation (Kimi-K2.6__l1_p74, its gather formula): y[n,co,o] = bias[co] +
// sum_ci sum_k w[ci,co,k] * x[n,ci,(o + p - d*k)/s], where a term exists only
// when o + p - d*k is a non-negative multiple of s whose quotient is below L.
// With o = s*m + r, every output class r is a sum over its tap set of shifted
// products  Y_r[m, co] += X[m + ph + e(r,k), ci] * W_k[ci, co], i.e. one GEMM per
// (class, tap) with M = positions m, N = C_out, K = C_in, all accumulating
// into the class's tile (the implicit-GEMM form the page sketches, without
// an im2col buffer and without inserting zeros).
//
// Kernel structure (one persistent CTA per SM, warp-specialised):
//  * warp 0, lane 0  -- TMA producer: for each (n, 128-position tile, 32-channel
//    chunk) one 3-D box x[n, ci0:ci0+32, a0:a0+BW] (BW = 128 + tap span, start
//    rounded down to 16 bytes; out-of-range cells arrive as zeros) into a
//    4-stage ring.  Warp 0 also owns the tensor-memory allocation.
//  * warps 2, 3, 8, 9 -- converters: transpose each raw box into the K-major,
//    no-swizzle operand layout (8-row x 16-byte core matrices; rows = window
//    positions, 4 channels per 16 bytes, one block of rows per 4 channels) and
//    round to tf32 (cvt.rna).  Because rows are 16 bytes apart, the operand of
//    tap k is the same buffer with its start moved by 16 bytes per row of tap
//    offset: one transposed copy serves every tap of every class.
//  * warp 1, lane 0  -- MMA issuer: per chunk and (class, tap), CK/8 tcgen05.mma
//    kind::tf32 of 128 x C_out x 8 into the class's accumulator in tensor memory
//    (double-buffered across tiles), then tcgen05.commit to release the
//    operand stage and, after the last chunk, to hand the tile to the epilogue.
//  * warps 4..7 -- epilogue: tcgen05.ld of their 32 accumulator rows, + bias,
//    and stores of s consecutive outputs per channel (classes without taps are
//    the bias alone), 32 lanes writing consecutive positions.
// Weights are rounded to tf32 once per CTA into shared memory in the same
// K-major layout, one [C_in/4][C_out][4] block per tap.  Every wait is bounded;
// a wait that times out records APS_DEVERR_TIMEOUT, the CTA drains what it has
// in flight and frees its tensor memory before returning.
#include <algorithm>

#include "aps_dev.cuh"
#include "aps_internal.h"

namespace aps {
namespace tc1 {
constexpr int BM = 128;           // positions per tile (MMA M)
constexpr int CK = 32;            // input channels per staged chunk (MMA K per chunk)
constexpr int RAW_STAGES = 4;
constexpr int XT_STAGES = 3;
constexpr int MAX_CLASSES = 4;
constexpr int MAX_TAPS = 8;       // taps per class
constexpr int THREADS = 320;      // 10 warps
constexpr int W_PRODUCER = 0, W_MMA = 1, W_EPI0 = 4;

struct Taps {
    int nclass;                        // classes (output residues) with taps
    int cls_r[MAX_CLASSES];            // residue of each such class
    int ntaps[MAX_CLASSES];
    int tap_k[MAX_CLASSES][MAX_TAPS];  // weight tap index
    int tap_row[MAX_CLASSES][MAX_TAPS];// first window row used by tile position 0
};

__device__ __forceinline__ int converter_id(int warp) {
    return warp == 2 ? 0 : warp == 3 ? 1 : warp - 6;   // warps 2, 3, 8, 9
}

__device__ __forceinline__ uint32_t to_tf32(float v) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(v));
    return r;
}

// tcgen05 shared-memory matrix descriptor, K-major, no swizzle.
__device__ __forceinline__ uint64_t umma_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFF);
    d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
    d |= (uint64_t)1 << 46;   // descriptor version of sm_100-class tensor cores
    return d;
}

__device__ __forceinline__ void umma_tf32(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate));
}

__device__ __forceinline__ void umma_commit(uint64_t *bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 32 lanes x 32 columns of 32-bit accumulator, one column per register.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
        "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
}  // namespace tc1

__global__ void __launch_bounds__(tc1::THREADS, 1)
    convt1d_tf32_kernel(const __grid_constant__ CUtensorMap xmap, const float *__restrict__ w,
                        const float *__restrict__ bias, float *__restrict__ y, int Cin, int Cout,
                        int K, int S, int L_out, int n_mtiles, long long n_units, int win0, int BW,
                        int tmem_cols, const __grid_constant__ tc1::Taps taps,
                        unsigned int *status) {
    using namespace tc1;
    extern __shared__ __align__(1024) unsigned char smem[];
    const int CKr = Cin < CK ? Cin : CK;          // channels per chunk
    const int nchunks = Cin / CKr;
    const uint32_t LBO_X = (uint32_t)BW * 16 + 16;   // 16-byte pad: conflict-free transposes
    const uint32_t XT_BYTES = (uint32_t)(CKr / 4) * LBO_X;
    const uint32_t XT_STRIDE = (XT_BYTES + 1023) & ~1023u;
    const uint32_t RAW_BYTES = (uint32_t)CKr * BW * 4;
    const uint32_t RAW_STRIDE = (RAW_BYTES + 1023) & ~1023u;
    unsigned char *xt = smem;
    unsigned char *raw = xt + XT_STAGES * XT_STRIDE;
    float *wt = reinterpret_cast<float *>(raw + RAW_STAGES * RAW_STRIDE);   // [K][Cin/4][Cout][4]
    float *bs = wt + (size_t)K * Cin * Cout;
    uint64_t *bars = reinterpret_cast<uint64_t *>(bs + ((Cout + 1) & ~1));
    uint64_t *raw_full = bars, *raw_empty = raw_full + RAW_STAGES;
    uint64_t *xt_full = raw_empty + RAW_STAGES, *xt_empty = xt_full + XT_STAGES;
    uint64_t *acc_full = xt_empty + XT_STAGES, *acc_empty = acc_full + 2;
    uint64_t *drain = acc_empty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    __shared__ volatile int abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // ---- set-up: barriers, tensor memory, tf32 weights, bias
    if (threadIdx.x == 0) {
        for (int s = 0; s < RAW_STAGES; ++s) {
            mbar_init(&raw_full[s], 1);
            mbar_init(&raw_empty[s], 4);
        }
        for (int s = 0; s < XT_STAGES; ++s) {
            mbar_init(&xt_full[s], 4);
            mbar_init(&xt_empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_empty[b], 4);
        }
        mbar_init(drain, 1);
        abort_flag = 0;
        mbar_fence_init();
    }
    __syncwarp();
    if (warp == W_PRODUCER) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"(tmem_cols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    {
        const int total = K * Cin * Cout;
        uint32_t *wtu = reinterpret_cast<uint32_t *>(wt);
        for (int e = threadIdx.x; e < total; e += THREADS) {
            // destination order [k][ci/4][co][ci%4]
            const int j = e & 3;
            int t = e >> 2;
            const int co = t % Cout;
            t /= Cout;
            const int cb = t % (Cin / 4);
            const int k = t / (Cin / 4);
            const int ci = cb * 4 + j;
            wtu[e] = to_tf32(__ldg(w + ((size_t)ci * Cout + co) * K + k));
        }
        for (int c = threadIdx.x; c < Cout; c += THREADS) bs[c] = bias ? __ldg(bias + c) : 0.f;
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    tc1::tc_fence_before();
    __syncthreads();
    tc1::tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == W_PRODUCER) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            tma_prefetch_desc(&xmap);
            uint32_t it = 0;
            bool ok = true;
            for (long long u = blockIdx.x; ok && u < n_units; u += gridDim.x) {
                const int n = (int)(u / n_mtiles);
                const int mt = (int)(u - (long long)n * n_mtiles);
                const int a0 = mt * BM + win0;
                for (int ch = 0; ch < nchunks; ++ch, ++it) {
                    const uint32_t s = it % RAW_STAGES;
                    if (it >= (uint32_t)RAW_STAGES &&
                        !mbar_wait(&raw_empty[s], ((it / RAW_STAGES) & 1u) ^ 1u)) {
                        record_error(status, APS_DEVERR_TIMEOUT);
                        abort_flag = 1;
                        ok = false;
                        break;
                    }
                    if (abort_flag) { ok = false; break; }
                    mbar_arrive_expect_tx(&raw_full[s], RAW_BYTES);
                    tma_load_3d(raw + s * RAW_STRIDE, &xmap, &raw_full[s], a0, ch * CKr, n);
                }
            }
            // boxes still in flight land before the CTA goes on to exit
            const uint32_t first = it > (uint32_t)RAW_STAGES ? it - RAW_STAGES : 0u;
            for (uint32_t j = first; j < it; ++j)
                if (!mbar_wait(&raw_full[j % RAW_STAGES], (j / RAW_STAGES) & 1u)) break;
        }
    } else if (warp == W_MMA) {
        // ------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idesc = (1u << 4) | (2u << 7) | (2u << 10) |
                                   ((uint32_t)(Cout >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);
            const uint32_t xt_addr = smem_u32(xt);
            const uint32_t wt_addr = smem_u32(wt);
            const uint32_t LBO_W = (uint32_t)Cout * 16;
            uint32_t it = 0, tile = 0;
            bool issued = false;
            for (long long u = blockIdx.x; u < n_units && !abort_flag; u += gridDim.x, ++tile) {
                const uint32_t b = tile & 1u;
                if (tile >= 2 && !mbar_wait(&acc_empty[b], ((tile >> 1) & 1u) ^ 1u)) {
                    record_error(status, APS_DEVERR_TIMEOUT);
                    abort_flag = 1;
                    break;
                }
                tc1::tc_fence_after();
                bool fail = false;
                for (int ch = 0; ch < nchunks; ++ch, ++it) {
                    const uint32_t s = it % XT_STAGES;
                    if (!mbar_wait(&xt_full[s], (it / XT_STAGES) & 1u)) {
                        record_error(status, APS_DEVERR_TIMEOUT);
                        abort_flag = 1;
                        fail = true;
                        break;
                    }
                    tc1::tc_fence_after();
                    const uint32_t xs = xt_addr + s * XT_STRIDE;
                    for (int c = 0; c < taps.nclass; ++c) {
                        const uint32_t d = tmem_base + (b * taps.nclass + c) * (uint32_t)Cout;
                        for (int t = 0; t < taps.ntaps[c]; ++t) {
                            const uint32_t arow = xs + (uint32_t)taps.tap_row[c][t] * 16;
                            const uint32_t wk = wt_addr + (uint32_t)taps.tap_k[c][t] * (Cin / 4) * LBO_W;
                            for (int j = 0; j < CKr / 8; ++j) {
                                const uint64_t ad = tc1::umma_desc(arow + 2 * j * LBO_X, LBO_X, 128);
                                const uint32_t cb = (uint32_t)(ch * CKr + 8 * j) / 4;
                                const uint64_t bd = tc1::umma_desc(wk + cb * LBO_W, LBO_W, 128);
                                tc1::umma_tf32(d, ad, bd, idesc, (ch | t | j) ? 1u : 0u);
                                issued = true;
                            }
                        }
                    }
                    tc1::umma_commit(&xt_empty[s]);
                }
                if (fail) break;
                tc1::umma_commit(&acc_full[b]);
            }
            if (issued) {
                // everything issued has completed before tensor memory is freed
                tc1::umma_commit(drain);
                mbar_wait(drain, 0);
            }
        }
    } else if (warp >= W_EPI0 && warp < W_EPI0 + 4) {
        // ------------------------------------------------------ epilogue
        const int q = warp - W_EPI0;   // tensor-memory lane quadrant (= warp % 4)
        const int row = q * 32 + lane;
        uint32_t tile = 0;
        for (long long u = blockIdx.x; u < n_units && !abort_flag; u += gridDim.x, ++tile) {
            const uint32_t b = tile & 1u;
            if (!mbar_wait(&acc_full[b], (tile >> 1) & 1u)) {
                record_error(status, APS_DEVERR_TIMEOUT);
                abort_flag = 1;
                break;
            }
            tc1::tc_fence_after();
            const int n = (int)(u / n_mtiles);
            const int mt = (int)(u - (long long)n * n_mtiles);
            const long long o_base = (long long)(mt * BM + row) * S;   // output of residue 0
            const bool any = o_base < L_out;
            float *yn = y + (long long)n * Cout * L_out;
            for (int c0 = 0; c0 < Cout; c0 += 32) {
                float v[MAX_CLASSES][32];
#pragma unroll
                for (int c = 0; c < MAX_CLASSES; ++c) {
                    if (c < taps.nclass) {
                        uint32_t r[32];
                        tc1::tmem_ld32(tmem_base + ((uint32_t)(q * 32) << 16) +
                                           (b * taps.nclass + c) * (uint32_t)Cout + c0,
                                       r);
#pragma unroll
                        for (int j = 0; j < 32; ++j) v[c][j] = __uint_as_float(r[j]);
                    }
                }
                if (!any) continue;
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const int co = c0 + j;
                    const float bv = bs[co];
                    float *yp = yn + (long long)co * L_out + o_base;
                    if (S == 1) {
                        yp[0] = v[0][j] + bv;
                    } else {
                        for (int r = 0; r < S; ++r) {
                            if (o_base + r >= L_out) break;
                            float val = bv;
#pragma unroll
                            for (int c = 0; c < MAX_CLASSES; ++c)
                                if (c < taps.nclass && taps.cls_r[c] == r) val += v[c][j];
                            yp[r] = val;
                        }
                    }
                }
            }
            tc1::tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[b]);
        }
    } else {
        // ------------------------------------------------------ converters
        const int ctid = converter_id(warp) * 32 + lane;
        const int pblocks = BW / 4;
        const int nblocks = (CKr / 4) * pblocks;
        uint32_t it = 0;
        for (long long u = blockIdx.x; u < n_units && !abort_flag; u += gridDim.x) {
            bool fail = false;
            for (int ch = 0; ch < nchunks; ++ch, ++it) {
                const uint32_t rs = it % RAW_STAGES, xs = it % XT_STAGES;
                if (!mbar_wait(&raw_full[rs], (it / RAW_STAGES) & 1u) ||
                    (it >= (uint32_t)XT_STAGES &&
                     !mbar_wait(&xt_empty[xs], ((it / XT_STAGES) & 1u) ^ 1u))) {
                    record_error(status, APS_DEVERR_TIMEOUT);
                    abort_flag = 1;
                    fail = true;
                    break;
                }
                const float *src = reinterpret_cast<const float *>(raw + rs * RAW_STRIDE);
                unsigned char *dst = xt + xs * XT_STRIDE;
                for (int blk = ctid; blk < nblocks; blk += 128) {
                    const int cb = blk / pblocks, pb = blk - cb * pblocks;
                    const float *s0 = src + (size_t)(4 * cb) * BW + 4 * pb;
                    const float4 r0 = *reinterpret_cast<const float4 *>(s0);
                    const float4 r1 = *reinterpret_cast<const float4 *>(s0 + BW);
                    const float4 r2 = *reinterpret_cast<const float4 *>(s0 + 2 * BW);
                    const float4 r3 = *reinterpret_cast<const float4 *>(s0 + 3 * BW);
                    const float a[4][4] = {{r0.x, r0.y, r0.z, r0.w}, {r1.x, r1.y, r1.z, r1.w},
                                           {r2.x, r2.y, r2.z, r2.w}, {r3.x, r3.y, r3.z, r3.w}};
                    unsigned char *d0 = dst + cb * LBO_X + (size_t)(4 * pb) * 16;
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj) {
                        const int j = (jj + pb) & 3;   // rotate to spread banks
                        uint4 v;
                        v.x = tc1::to_tf32(a[0][j]);
                        v.y = tc1::to_tf32(a[1][j]);
                        v.z = tc1::to_tf32(a[2][j]);
                        v.w = tc1::to_tf32(a[3][j]);
                        *reinterpret_cast<uint4 *>(d0 + j * 16) = v;
                    }
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&raw_empty[rs]);
                    mbar_arrive(&xt_full[xs]);
                }
            }
            if (fail) break;
        }
    }

    // ---- teardown: every role is done (or has drained after a timeout)
    tc1::tc_fence_before();
    __syncthreads();
    if (warp == W_PRODUCER) {
        tc1::tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                     "r"(tmem_cols)
                     : "memory");
    }
}

namespace {
int floordiv_h(int a, int b) { return (a >= 0) ? a / b : -((-a + b - 1) / b); }
}  // namespace

aps_status launch_convt1d_tf32(const float *x, const int64_t in[3], const float *w,
                               const float *bias, int64_t c_out, int k, int s, int p, int d,
                               float *y, int64_t l_out, cudaStream_t st) {
    using namespace tc1;
    const int64_t N = in[0], Cin = in[1], L = in[2];
    if (Cin % 8 != 0 || (Cin > CK && Cin % CK != 0) || c_out % 32 != 0 || c_out > 256 ||
        L % 4 != 0 || (reinterpret_cast<uintptr_t>(x) % 16) != 0 || N >= (1 << 30) ||
        L >= ((int64_t)1 << 31) || l_out >= ((int64_t)1 << 31) || s > 8)
        return APS_ERR_UNSUPPORTED;
    // classes and taps: o = s*m + r reads input i = m + ph + e(r,k) where
    // e(r,k) = (r + pl - d*k)/s for the taps with (r + pl - d*k) % s == 0.
    const int pl = p % s, ph = p / s;
    Taps taps{};
    int emin = 1 << 30, emax = -(1 << 30);
    int ce[MAX_CLASSES][MAX_TAPS];
    for (int r = 0; r < s; ++r) {
        int nt = 0, ks[64], es[64];
        for (int kk = 0; kk < k; ++kk) {
            const int v = r + pl - d * kk;
            if (((v % s) + s) % s == 0 && nt < 64) {
                ks[nt] = kk;
                es[nt] = floordiv_h(v, s);
                ++nt;
            }
        }
        if (!nt) continue;
        if (taps.nclass == MAX_CLASSES || nt > MAX_TAPS) return APS_ERR_UNSUPPORTED;
        const int c = taps.nclass++;
        taps.cls_r[c] = r;
        taps.ntaps[c] = nt;
        for (int t = 0; t < nt; ++t) {
            taps.tap_k[c][t] = ks[t];
            ce[c][t] = es[t];
            emin = std::min(emin, es[t]);
            emax = std::max(emax, es[t]);
        }
    }
    if (taps.nclass == 0) return APS_ERR_UNSUPPORTED;
    // window of a tile at m0: inputs m0 + ph + emin .. m0 + 127 + ph + emax, start
    // rounded down to a multiple of 4 (16-byte TMA coordinate)
    const int lo = ph + emin;
    const int win0 = floordiv_h(lo, 4) * 4;
    const int off = lo - win0;
    const int BW = ((off + BM + (emax - emin)) + 3) & ~3;
    if (BW > 256) return APS_ERR_UNSUPPORTED;
    for (int c = 0; c < taps.nclass; ++c)
        for (int t = 0; t < taps.ntaps[c]; ++t) taps.tap_row[c][t] = ph + ce[c][t] - win0;
    int cols = 32;
    while (cols < 2 * taps.nclass * (int)c_out) cols *= 2;
    if (cols > 512) return APS_ERR_UNSUPPORTED;

    const int CKr = Cin < CK ? (int)Cin : CK;
    const uint32_t LBO_X = (uint32_t)BW * 16 + 16;
    const uint32_t XT_STRIDE = ((uint32_t)(CKr / 4) * LBO_X + 1023) & ~1023u;
    const uint32_t RAW_STRIDE = ((uint32_t)CKr * BW * 4 + 1023) & ~1023u;
    const size_t w_bytes = (size_t)k * Cin * c_out * 4;
    const size_t smem = XT_STAGES * XT_STRIDE + RAW_STAGES * RAW_STRIDE + w_bytes +
                        ((c_out + 1) & ~1) * 4 + (2 * RAW_STAGES + 2 * XT_STAGES + 5) * 8 + 16;
    if (smem > 227 * 1024) return APS_ERR_UNSUPPORTED;

    CUtensorMap map;
    const cuuint64_t dims[3] = {(cuuint64_t)L, (cuuint64_t)Cin, (cuuint64_t)N};
    const cuuint64_t strides[2] = {(cuuint64_t)(L * 4), (cuuint64_t)(Cin * L * 4)};
    const cuuint32_t box[3] = {(cuuint32_t)BW, (cuuint32_t)CKr, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    if (!encode_tiled(&map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float *>(x), dims,
                      strides, box, estr))
        return APS_ERR_UNSUPPORTED;

    const int per_sm = resident_ctas((const void *)convt1d_tf32_kernel, THREADS, (int)smem);
    if (per_sm < 1) return APS_ERR_UNSUPPORTED;
    const int64_t M = ceil_div(l_out, s);
    const int n_mtiles = (int)ceil_div(M, BM);
    const long long n_units = (long long)N * n_mtiles;
    const long long grid = std::min<long long>(n_units, (long long)sm_count());
    convt1d_tf32_kernel<<<(unsigned)grid, THREADS, smem, st>>>(
        map, w, bias, y, (int)Cin, (int)c_out, k, s, (int)l_out, n_mtiles, n_units, win0, BW,
        cols, taps, status_word());
    return launch_status();
}

}  // namespace aps
