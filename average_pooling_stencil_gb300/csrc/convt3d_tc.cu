// convt3d_tc.cu -- standalone ConvTranspose3d(k3, s2, p1) on the tensor cores,
// emitting the full-resolution (pre-pool) tensor of Kimi-K2.6__l2_p50's
// unfused chain.
//
// Per dim an output o = 2m + r takes, for r = 0, input m with tap 1 and, for
// r = 1, input m with tap 2 and input m+1 with tap 0 (the page's per-parity
// analysis).  So the 8 outputs (2m + r), r in {0,1}^3, around an input
// position m read only its 2x2x2 neighbourhood m + (a, b, c): per position a
// dot product of the K = 8*C_in neighbourhood values with a K x 128 matrix
// whose column (r, co) holds w[ci][co][k(r_d,a)][k(r_h,b)][k(r_w,c)], and 0
// where a parity does not reach a neighbour (r = 0 with offset 1).  128
// positions x K x 128 is one M128 N128 MMA chain.
//
// Precision (3xTF32), as in the fused kernel: hi = v with the low 13 mantissa
// bits cleared, lo = v - hi; each product accumulated as lo(x)hi(w) +
// hi(x)lo(w) + hi(x)hi(w) in fp32.
//
// Design (GB300): one persistent CTA per SM, two groups of four warps and a
// TMA warp.  A unit is 128 input positions of one (n, md) input plane: 4 rows of
// up to 32 columns, 2 rows of up to 64 or 1 row of up to 128 (each row spread over
// 1, 2 or 4 warps of a group) -- outputs: planes 2md, 2md+1, twice the unit's rows,
// all columns -- or, for rows wider than 128, a 128-column block of one row (box
// origin 128*mwb, 128-byte aligned), whose outputs leave straight from registers.
// CTA-local unit k goes to group k % 2 and stage k % nst of a ring the TMA
// warp fills (one 4-D box per unit: C_in x 2 planes x (rows + 1) x (columns + 1,
// rounded up to 4), zero-filled outside the tensor).  Warp q of a group owns
// tensor-memory lanes 32q..32q+31, one position of the unit per lane.  Per
// unit a thread reads its 8*C_in inputs, writes its hi and lo A row into its
// lane (tcgen05.st); after a group barrier the group's MMA thread issues 9
// MMAs (M 128, N 128, K 8; A in tensor memory, B = the parity-tap matrix in
// shared memory) and commits.  The epilogue loads the 128 accumulator columns
// in four tcgen05.ld of 32 (one (r_d, r_h) pair and both r_w each), adds the
// bias and writes the group's staging block, where output plane r_d, channel
// co is one run of up to 2 x rows x Wo floats at an offset congruent to its
// destination mod 16 bytes.  Each run then leaves by one cp.async.bulk issued by
// its own lane (head and tail by plain stores); a group restages only after
// its previous copies have read the block, while the other group computes.
// Every wait is bounded; the group barrier also carries each warp's go-on
// vote, so that a group whose wait ran out leaves together, drains what it
// issued and frees the tensor memory.
// C_in 4..8: the A row grows to 16*C_in columns (the accumulator then starts
// at column 128 of the group's 256) and B to 8 KB per input channel, so the
// staging blocks fit only beside a shorter input ring (the launcher takes the
// most stages that fit, down to one per group).  Where they do not fit at all,
// and for blocks of wider rows, the epilogue writes each thread's outputs
// straight from registers (for each channel, its two r_w outputs; a warp's 32
// lanes cover 64 consecutive outputs of one row).
#include <algorithm>
#include <cstring>

#include "aps_dev.cuh"
#include "aps_internal.h"
#include "aps_tc.cuh"

namespace aps {
namespace c3t {
constexpr int COUT = 16;
constexpr int NCOL = 8 * COUT;             // MMA N: 8 parity classes x 16 channels
constexpr int CIN_MAX = 8;
constexpr int GROUPS = 2;
constexpr int WORKERS = 4 * GROUPS;        // warps 0..7
constexpr int W_FILL = WORKERS;            // warp 8: the TMA loads of the input ring
constexpr int THREADS = 32 * (WORKERS + 1);   // 288
// A unit is 128 input positions: 4 rows of up to 32 columns, 2 of up to 64 or 1 of
// up to 128 (lgw = 0, 1, 2: each input row spread over 1 << lgw warps of a group),
// or a 128-column block of a wider row.
constexpr int STAGES = 4 * GROUPS;         // input ring: up to four units in flight per group
constexpr int TMEM_COLS = 512;
constexpr int GROUP_COLS = TMEM_COLS / GROUPS;   // 256
// accumulator: 128 columns after A hi + lo (16 * C_in columns)
__host__ __device__ constexpr int d_col_of(int cin) { return 16 * cin <= 64 ? 64 : 128; }
// Fixed head of the dynamic shared memory (bytes); stages and staging follow.
constexpr int OFF_FULL = 0;                // uint64 [STAGES]
constexpr int OFF_EMPTY = 64;              // uint64 [STAGES]
constexpr int OFF_DFULL = 128;             // uint64 [GROUPS]: the group's MMAs of a unit are done
constexpr int OFF_TMEM = 144;              // uint32
constexpr int OFF_ABORT = 148;             // int
constexpr int OFF_SLOT = 192;              // Slot [STAGES]
constexpr int OFF_BIAS = 448;              // float [16]
constexpr int OFF_B = 512;                 // B, hi then lo: [C_in][2][128][4] words each
constexpr int B_CI_BYTES = 2 * NCOL * 16;  // one input channel's K-step of 8: 4096 bytes
__host__ __device__ constexpr int head_bytes_of(int cin) { return OFF_B + 2 * cin * B_CI_BYTES; }
static_assert(head_bytes_of(1) % 128 == 0, "stages start 128-byte aligned");
static_assert(d_col_of(CIN_MAX) >= 16 * CIN_MAX && d_col_of(CIN_MAX) + NCOL <= GROUP_COLS,
              "tile buffer layout");
static_assert(STAGES % GROUPS == 0, "a group's units always use the same stages");
// stages of a launch: nst, a multiple of GROUPS in [GROUPS, STAGES]

struct Slot {
    long long n;
    int md, mh0, mw0, pad[3];
};
static_assert(sizeof(Slot) * STAGES <= OFF_BIAS - OFF_SLOT, "slots fit");

// Floats of one stage: the box (C_in x 2 planes x XRu rows x BW columns), plus the
// columns a lane past the last input column may read on (at most UW).
__host__ __device__ inline int stage_stride_of(int Cin, int XRu, int BW, int UW) {
    return (Cin * 2 * XRu * BW + UW + 32 + 31) & ~31;
}
// Output staging of one group: run (r_d, co) at r_d*RDS + co*CH + a0, where
// CH = the channel step of y mod 4 and RDS = the plane step of y mod 4 (both
// mod 4), so that one shift a0 per unit gives every run the alignment of its
// destination; each run holds up to orows x Wo floats after a shift of <= 3.
__host__ __device__ inline int chan_stride_of(int Wo, int ac, int orows) {
    return ((orows * Wo + 6) & ~3) + ac;
}
__host__ __device__ inline int plane_stride_of(int Wo, int ac, int ap, int orows) {
    return ((COUT * chan_stride_of(Wo, ac, orows) + 3) & ~3) + ap;
}
__host__ __device__ inline int staging_floats_of(int Wo, int ac, int ap, int orows) {
    return (2 * plane_stride_of(Wo, ac, ap, orows) + 31) & ~31;
}
}  // namespace c3t

// 32 lanes x 8 columns from registers (the caller waits with tmem_st_wait).
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t *v) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
        : "memory");
}

// CIN: input channels (1..8); NST: stages of the input ring at compile time (0: the
// run-time nst)
template <int CIN, int NST>
__global__ void __launch_bounds__(c3t::THREADS, 1)
    convt3d_tc_kernel(const __grid_constant__ CUtensorMap xmap, const float *__restrict__ w,
                      const float *__restrict__ bias, float *__restrict__ y, int D, int H, int W,
                      int BW, int Do, int Ho, int Wo, int n_mhb, int n_mwb, int lgw,
                      int direct_rt, int nst, long long n_units, unsigned int *status) {
    pdl_trigger();
    pdl_wait();
    using namespace c3t;
    constexpr int D_COL = d_col_of(CIN), HEAD_BYTES = head_bytes_of(CIN);
    // outputs from registers (the launcher's choice): 128-column blocks of wider
    // rows, whose runs are not whole rows, and where the staging blocks do not fit
    const bool DIRECT = direct_rt != 0;
    extern __shared__ __align__(128) unsigned char smraw[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smraw + OFF_FULL);
    uint64_t *empty = reinterpret_cast<uint64_t *>(smraw + OFF_EMPTY);
    uint64_t *dfull = reinterpret_cast<uint64_t *>(smraw + OFF_DFULL);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smraw + OFF_TMEM);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smraw + OFF_ABORT);
    Slot *slot = reinterpret_cast<Slot *>(smraw + OFF_SLOT);
    float *bsm = reinterpret_cast<float *>(smraw + OFF_BIAS);
    uint32_t *bop = reinterpret_cast<uint32_t *>(smraw + OFF_B);
    const int MR = 4 >> lgw, XRu = MR + 1, UW = 32 << lgw;   // unit rows, staged rows, width
    const int orows = 2 * MR;                                   // output rows per unit
    const int stage_stride = stage_stride_of(CIN, XRu, BW, UW);
    float *xs = reinterpret_cast<float *>(smraw + HEAD_BYTES);   // [nst][C_in][2][XRu][BW]
    const long long plane = (long long)Ho * Wo;
    const long long cstride = (long long)Do * plane;              // between output channels
    const int ac = (int)(cstride & 3), ap = (int)(plane & 3);
    const int CH = chan_stride_of(Wo, ac, orows), RDS = plane_stride_of(Wo, ac, ap, orows);
    float *ost = xs + (NST ? NST : nst) * stage_stride;            // [GROUPS][2][16][CH]
    const uint32_t ust = NST ? (uint32_t)NST : (uint32_t)nst;
    const int stage_floats = CIN * 2 * XRu * BW;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    if (tid == 0) {
        for (int s = 0; s < (int)ust; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 4);   // the four warps of the unit's group
        }
        for (int g = 0; g < GROUPS; ++g) mbar_init(&dfull[g], 1);
        *abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == 0) tc::tmem_alloc(tmem_slot, TMEM_COLS);
    __syncthreads();

    // ---- B: word (ci, kc, n, e) holds column n = r*16 + co, row ci*8 + 4*kc + e
    // (neighbour e = a*4 + b*2 + c): w[ci][co][k(rd,a)][k(rh,b)][k(rw,c)] with,
    // per dim, k(0,0) = 1, k(1,0) = 2, k(1,1) = 0 and 0 for (r = 0, offset 1)
    for (int i = tid; i < CIN * 8 * NCOL; i += THREADS) {
        const int n = i % NCOL, e = (i / NCOL) % 8, ci = i / (8 * NCOL);
        const int r = n >> 4, co = n & 15;
        const int rd = r >> 2, rh = (r >> 1) & 1, rw = r & 1;
        const int a = e >> 2, b = (e >> 1) & 1, c = e & 1;
        const int kd = rd ? (a ? 0 : 2) : (a ? -1 : 1);
        const int kh = rh ? (b ? 0 : 2) : (b ? -1 : 1);
        const int kw = rw ? (c ? 0 : 2) : (c ? -1 : 1);
        const float v = (kd < 0 || kh < 0 || kw < 0)
                            ? 0.f
                            : __ldg(w + ((size_t)(ci * COUT + co) * 3 + kd) * 9 + kh * 3 + kw);
        const uint32_t hi = __float_as_uint(v) & 0xFFFFE000u;
        const int word = ((ci * 2 + (e >> 2)) * NCOL + n) * 4 + (e & 3);
        bop[word] = hi;
        bop[CIN * 8 * NCOL + word] = __float_as_uint(v - __uint_as_float(hi));
    }
    if (tid < COUT) bsm[tid] = bias ? __ldg(bias + tid) : 0.f;
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // B is read by the tensor core
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == W_FILL) {
        // -------------------------------------------------- input ring (lane 0)
        // CTA-local unit k goes to stage k % nst, which held unit k - nst of
        // the same group (units alternate between the groups, nst is even),
        // once that group is done with it.
        if (lane == 0) {
            tma_prefetch_desc(&xmap);
            uint32_t k = 0;
            for (long long u = blockIdx.x; u < n_units; u += gridDim.x, ++k) {
                const int s = (int)(k % ust);
                if (*abort_flag) break;
                if (k >= ust && !mbar_wait(&empty[s], ((k - ust) / ust) & 1u)) {
                    record_error(status, APS_DEVERR_TIMEOUT);
                    *abort_flag = 1;
                    break;
                }
                const int mwb = (int)(u % n_mwb);
                long long t = u / n_mwb;
                const int mhb = (int)(t % n_mhb);
                t /= n_mhb;
                const int md = (int)(t % D);
                const long long n = t / D;
                slot[s].n = n;
                slot[s].md = md;
                slot[s].mh0 = MR * mhb;
                slot[s].mw0 = UW * mwb;
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                mbar_arrive_expect_tx(&full[s], (uint32_t)stage_floats * 4u);
                tma_load_4d(xs + s * stage_stride, &xmap, &full[s], UW * mwb, MR * mhb, md,
                            (int)(n * CIN));
            }
            // the loads in flight land before the CTA exits (the latest of each stage)
            for (uint32_t j = k > ust ? k - ust : 0; j < k; ++j)
                mbar_wait(&full[j % ust], (j / ust) & 1u);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ workers
        const int grp = warp >> 2, q = warp & 3;
        // this thread's input position in the unit: row mr, column mc (tensor-memory
        // lane 32q + lane = mr * UW + mc)
        const int mr = q >> lgw, mc = ((q & ((1 << lgw) - 1)) << 5) + lane;
        const uint32_t lane_q = (uint32_t)(32 * q) << 16;   // this warp's tensor-memory lanes
        const uint32_t gcol = (uint32_t)(grp * GROUP_COLS); // the group's tile buffer
        const int gbar = 1 + grp;                            // the group's barrier (0 is __syncthreads)
        constexpr uint32_t IDESC = tc::idesc_tf32(128, NCOL);
        const uint32_t b_hi = smem_u32(bop), b_lo = b_hi + CIN * B_CI_BYTES;
        float *og = ost + grp * staging_floats_of(Wo, ac, ap, orows);   // the group's staging block
        float bias_r[COUT];
#pragma unroll
        for (int co = 0; co < COUT; ++co) bias_r[co] = bsm[co];
        uint32_t j = 0, ncommit = 0;   // units this group has taken; MMA commits (MMA thread)
        bool fail = false;
        // C_in <= 3: whether the group's next box has landed and whether another
        // thread has aborted are asked a unit early (a non-blocking barrier test, a
        // plain load), as every shared-memory access waits behind the gathers and the
        // tensor core (183.8 -> 181.0 us on the C_in 3 workload; 256 -> 263 us with
        // C_in 8, whose longer gather hides the waits already)
        constexpr bool EARLY = CIN <= 3;
        bool full_ready = false;
        int abort_seen = 0;
        for (long long kk = grp;; kk += GROUPS, ++j) {
            const long long u = blockIdx.x + kk * gridDim.x;
            if (u >= n_units) break;
            const uint32_t kq = (uint32_t)kk;   // CTA-local unit (< 2^32: the launcher checks)
            const int s = (int)(kq % ust);
            bool ok = !fail && !(EARLY ? abort_seen : *abort_flag);
            if (ok && !full_ready && !mbar_wait(&full[s], (kq / ust) & 1u)) {
                record_error(status, APS_DEVERR_TIMEOUT);
                *abort_flag = 1;
                ok = false;
            }
            ok = __all_sync(0xffffffffu, ok);

            // ---- the A row of input position (mh0 + mr, mw0 + mc): hi and lo of
            // its 8*C_in neighbourhood values
            if constexpr (CIN > 3) {
              if (ok) {
                // one input channel at a time: its 8 hi and 8 lo columns
                const float *xp = xs + s * stage_stride + mr * BW + mc;
#pragma unroll
                for (int ci = 0; ci < CIN; ++ci) {
                    uint32_t hv[8], lv[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int a = e >> 2, b = (e >> 1) & 1, c = e & 1;
                        const float v = xp[((ci * 2 + a) * XRu + b) * BW + c];
                        hv[e] = __float_as_uint(v) & 0xFFFFE000u;
                        lv[e] = __float_as_uint(v - __uint_as_float(hv[e]));
                    }
                    tmem_st8(tmem + lane_q + gcol + 8 * ci, hv);
                    tmem_st8(tmem + lane_q + gcol + 8 * CIN + 8 * ci, lv);
                }
                tc::tmem_st_wait();
              }
            } else if (ok) {
                const float *xp = xs + s * stage_stride + mr * BW + mc;
                uint32_t av[16 * CIN];   // hi[0 .. 8*CIN), then lo
#pragma unroll
                for (int ci = 0; ci < CIN; ++ci)
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int a = e >> 2, b = (e >> 1) & 1, c = e & 1;
                        const float v = xp[((ci * 2 + a) * XRu + b) * BW + c];
                        const uint32_t hi = __float_as_uint(v) & 0xFFFFE000u;
                        av[ci * 8 + e] = hi;
                        av[8 * CIN + ci * 8 + e] = __float_as_uint(v - __uint_as_float(hi));
                    }
#pragma unroll
                for (int r = 0; r < CIN; ++r) tc::tmem_st16(tmem + lane_q + gcol + 16 * r, av + 16 * r);
                tc::tmem_st_wait();
            }
            tc::tc_fence_before();
            __syncwarp();
            // hand the tile to the group's MMA thread; the group decides together
            // whether to go on, so that no warp is left at its barrier
            if (tc::named_bar_or(gbar, 128, !ok)) break;
            if (q == 0 && lane == 0) {
                tc::tc_fence_after();
                const uint32_t d = tmem + gcol + D_COL;
#pragma unroll
                for (int ci = 0; ci < CIN; ++ci) {
                    const uint32_t ahi = tmem + gcol + 8 * ci, alo = ahi + 8 * CIN;
                    const uint64_t bh = tc::umma_desc(b_hi + ci * B_CI_BYTES, NCOL * 16, 128);
                    const uint64_t bl = tc::umma_desc(b_lo + ci * B_CI_BYTES, NCOL * 16, 128);
                    tc::umma_tf32_ts(d, alo, bh, IDESC, ci > 0 ? 1u : 0u);   // lo(x) hi(w)
                    tc::umma_tf32_ts(d, ahi, bl, IDESC, 1u);                 // hi(x) lo(w)
                    tc::umma_tf32_ts(d, ahi, bh, IDESC, 1u);                 // hi(x) hi(w)
                }
                tc::umma_commit(&dfull[grp]);
                ++ncommit;
            }
            __syncwarp();

            // where the outputs go, read before the stage and its slot are released
            const long long gn = slot[s].n;
            const int gmd = slot[s].md, gmh0 = slot[s].mh0, gmw0 = slot[s].mw0;
            const bool in_w = gmw0 + mc < W;   // this thread's input column exists
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
            if (EARLY) {
                const uint32_t kn = kq + GROUPS;
                full_ready = mbar_test(&full[kn % ust], (kn / ust) & 1u);
                abort_seen = *abort_flag;
            }

            // ---- epilogue: the 128 accumulator columns, 32 at a time (one
            // (r_d, r_h) and both r_w), + bias -> the group's staging block
            bool okd = mbar_wait(&dfull[grp], j & 1u);
            if (!okd) {
                record_error(status, APS_DEVERR_TIMEOUT);
                *abort_flag = 1;
            }
            okd = __all_sync(0xffffffffu, okd);
            if (DIRECT) {
                if (tc::named_bar_or(gbar, 128, !okd)) break;
                // outputs straight from registers: the thread holds output columns
                // 2(mw0 + mc) and 2(mw0 + mc) + 1 of every channel of its (r_d, r_h) row
                const int oh0 = 2 * gmh0;
                const int nrows = Ho - oh0 < orows ? Ho - oh0 : orows;
                float *y0 = y + ((gn * COUT) * Do + 2 * gmd) * plane + (long long)oh0 * Wo + 2 * gmw0;
                tc::tc_fence_after();
#pragma unroll 1
                for (int c = 0; c < 4; ++c) {
                    const int rd = c >> 1, rh = c & 1;
                    uint32_t v[32];   // v[rw*16 + co]
                    tc::tmem_ld32(tmem + lane_q + gcol + D_COL + 32 * c, v);
                    const int row = 2 * mr + rh;
                    if (2 * gmd + rd < Do && row < nrows && in_w) {
                        float *yp = y0 + rd * plane + (long long)row * Wo + 2 * mc;
                        const bool w1 = 2 * (gmw0 + mc) + 1 < Wo;
#pragma unroll
                        for (int co = 0; co < COUT; ++co) {
                            yp[0] = __uint_as_float(v[co]) + bias_r[co];
                            if (w1) yp[1] = __uint_as_float(v[16 + co]) + bias_r[co];
                            yp += cstride;
                        }
                    }
                }
                // the accumulator is read: the next unit's MMAs may overwrite it
                tc::tc_fence_before();
                continue;
            } else {
                // the group's previous copies (each issued by its own lane) have
                // read its staging block before this unit's epilogue rewrites it:
                // they had this unit's gather and MMAs to do so
                bulk_wait_read<0>();
                __syncwarp();
                if (tc::named_bar_or(gbar, 128, !okd)) break;
                const int oh0 = 2 * gmh0;
                const int nrows = Ho - oh0 < orows ? Ho - oh0 : orows;
                float *y0 = y + ((gn * COUT) * Do + 2 * gmd) * plane + (long long)oh0 * Wo;
                const int a0 = (int)((reinterpret_cast<uintptr_t>(y0) >> 2) & 3u);
                {
                    tc::tc_fence_after();
    #pragma unroll 1
                    for (int c = 0; c < 4; ++c) {
                        const int rd = c >> 1, rh = c & 1;
                        uint32_t v[32];   // v[rw*16 + co]
                        tc::tmem_ld32(tmem + lane_q + gcol + D_COL + 32 * c, v);
                        const int row = 2 * mr + rh;
                        if (2 * gmd + rd < Do && row < nrows && in_w) {
                            float *sp = og + rd * RDS + a0 + row * Wo + 2 * mc;
                            const bool w1 = 2 * mc + 1 < Wo;
    #pragma unroll
                            for (int co = 0; co < COUT; ++co) {
                                sp[0] = __uint_as_float(v[co]) + bias_r[co];
                                if (w1) sp[1] = __uint_as_float(v[16 + co]) + bias_r[co];
                                sp += CH;
                            }
                        }
                    }
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                tc::named_bar(gbar, 128);   // the staging block is complete

                // ---- each (r_d, co) run: its 16-byte-aligned middle by one bulk copy,
                // the at most 3 + 3 head and tail floats by plain stores.  Warp q takes
                // channels 4q..4q+3 of both planes; lane i < 8 issues run i's copy.
                const int run = nrows * Wo;
                {
                    const int i = lane & 7;
                    const int rd = i >> 2, co = 4 * q + (i & 3);
                    const uint32_t off = (uint32_t)(a0 + co * ac + rd * ap) & 3u;
                    const int hd = (int)((4u - off) & 3u);
                    const int mid = run > hd ? (run - hd) & ~3 : 0;
                    float *yc = y0 + co * cstride + rd * plane;
                    const float *sc = og + rd * RDS + co * CH + a0;
                    if (lane < 8 && 2 * gmd + rd < Do && mid > 0) {
                        bulk_store(yc + hd, sc + hd, (uint32_t)mid * 4u);
                        bulk_commit();
                    }
    #pragma unroll 1
                    for (int r = 0; r < 8; ++r) {   // head and tail of run r of this warp
                        const int rd2 = r >> 2, co2 = 4 * q + (r & 3);
                        if (2 * gmd + rd2 >= Do) break;
                        const uint32_t off2 = (uint32_t)(a0 + co2 * ac + rd2 * ap) & 3u;
                        const int hd2 = (int)((4u - off2) & 3u);
                        const int head = run < hd2 ? run : hd2;
                        const int mid2 = run > hd2 ? (run - hd2) & ~3 : 0;
                        const int tail0 = head + mid2;
                        float *yc2 = y0 + co2 * cstride + rd2 * plane;
                        const float *sc2 = og + rd2 * RDS + co2 * CH + a0;
                        if (lane < head) yc2[lane] = sc2[lane];
                        if (tail0 + lane < run) yc2[tail0 + lane] = sc2[tail0 + lane];
                    }
                }
            }
        }
        // the group's last MMAs and its output copies are done before the
        // tensor memory and the shared memory go
        if (q == 0 && lane == 0 && ncommit > 0) mbar_wait(&dfull[grp], (ncommit - 1) & 1u);
        bulk_wait<0>();   // every lane's own copies
        __syncwarp();
    }

    // ---- teardown: every role is done (or has drained after a timeout)
    tc::tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, TMEM_COLS);
    }
}

aps_status launch_convt3d_tc(const float *x, const int64_t in[5], const float *w,
                             const float *bias, float *y, const int64_t out[5], cudaStream_t st) {
    using namespace c3t;
    const int64_t N = in[0], Cin = in[1], D = in[2], H = in[3], W = in[4];
    const int64_t Do = out[2], Ho = out[3], Wo = out[4];
    // the TMA box needs 16-byte rows
    if (Cin < 1 || Cin > CIN_MAX || W % 4 != 0 ||
        reinterpret_cast<uintptr_t>(x) % 16 != 0 || D >= (1 << 30) || H >= (1 << 30) ||
        N * Cin >= (1ll << 31) || N * D >= (1ll << 40))
        return APS_ERR_UNSUPPORTED;
    // unit: 128 positions -- 4 rows of <= 32 columns, 2 of <= 64, 1 of <= 128, or a
    // 128-column block of a wider row; staged columns: the unit's and one more (past
    // W it reads as zero), a multiple of 4
    const int lgw = W <= 32 ? 0 : W <= 64 ? 1 : 2;
    const int MR = 4 >> lgw, UW = 32 << lgw;
    const int BW = (int)((std::min<int64_t>(W, UW) + 1 + 3) & ~3);
    const int64_t n_mhb = ceil_div(H, (int64_t)MR), n_mwb = ceil_div(W, (int64_t)UW);
    const long long n_units = N * D * n_mhb * n_mwb;
    const long long grid = std::min<long long>(sm_count(), n_units);
    if (n_units / grid >= (1ll << 31)) return APS_ERR_UNSUPPORTED;   // CTA-local unit counters
    // staged runs leaving by bulk copies where the staging blocks fit beside B and
    // the input ring; outputs from registers for blocks of wider rows (whose runs
    // are not whole rows) and where the staging does not fit.  The ring has four
    // stages per group; for C_in > 3 (B of 8 KB per channel) as many as fit beside
    // the staging, down to one per group (C_in <= 3 keeps its ring at compile time)
    const int ac = (int)((Do * Ho * Wo) & 3), ap = (int)((Ho * Wo) & 3);
    const size_t stage_bytes = (size_t)stage_stride_of((int)Cin, MR + 1, BW, UW) * 4;
    const size_t staging_bytes = (size_t)GROUPS * staging_floats_of((int)Wo, ac, ap, 2 * MR) * 4;
    auto fits = [&](int ns) {
        return head_bytes_of((int)Cin) + ns * stage_bytes + staging_bytes <= kMaxSmemPerCta;
    };
    int direct = n_mwb > 1, nst = STAGES;
    if (!direct) {
        while (Cin > 3 && nst > GROUPS && !fits(nst)) nst -= GROUPS;
        if (!fits(nst)) {
            direct = 1;
            nst = STAGES;
        }
    }
    CUtensorMap map;
    const cuuint64_t dims[4] = {(cuuint64_t)W, (cuuint64_t)H, (cuuint64_t)D, (cuuint64_t)(N * Cin)};
    const cuuint64_t strides[3] = {(cuuint64_t)(W * 4), (cuuint64_t)(H * W * 4),
                                   (cuuint64_t)(D * H * W * 4)};
    const cuuint32_t box[4] = {(cuuint32_t)BW, (cuuint32_t)(MR + 1), 2, (cuuint32_t)Cin};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    if (!encode_tiled(&map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<float *>(x), dims,
                      strides, box, estr))
        return APS_ERR_UNSUPPORTED;
    const size_t smem = head_bytes_of((int)Cin) + nst * stage_bytes + (direct ? 0 : staging_bytes);
    void (*const kerns[CIN_MAX])(const CUtensorMap, const float *, const float *, float *, int,
                                 int, int, int, int, int, int, int, int, int, int, int, long long,
                                 unsigned int *) = {
        convt3d_tc_kernel<1, STAGES>, convt3d_tc_kernel<2, STAGES>, convt3d_tc_kernel<3, STAGES>,
        convt3d_tc_kernel<4, 0>,      convt3d_tc_kernel<5, 0>,      convt3d_tc_kernel<6, 0>,
        convt3d_tc_kernel<7, 0>,      convt3d_tc_kernel<8, 0>};
    const auto kern = kerns[Cin - 1];
    // one CTA per SM: each holds all 512 tensor-memory columns
    if (resident_ctas((const void *)kern, THREADS, (int)smem) < 1) return APS_ERR_UNSUPPORTED;
    const cudaError_t e = launch_pdl(kern, dim3((unsigned)grid), dim3(THREADS), smem, st, map, w, bias, y, (int)D, (int)H,
               (int)W, BW, (int)Do, (int)Ho, (int)Wo, (int)n_mhb, (int)n_mwb, lgw, direct,
               nst, n_units, status_word());
    return launch_status(e);
}

}  // namespace aps
