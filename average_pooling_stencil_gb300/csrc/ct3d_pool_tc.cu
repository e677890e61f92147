// ct3d_pool_tc.cu -- the fused ConvTranspose3d(k3, s2, p1) -> x scale1 ->
// AvgPool3d(2) -> + bias -> x scale2 of Kimi-K2.6__l2_p50 on the tensor cores.
//
// The chain collapses (the page's per-parity grouping of the 27 taps; see
// ct3d_pool.cu) to a 2x2x2 valid correlation with collapsed weights:
//     y[n,co,d,h,w] = beff[co] + sum_{ci,a,b,c} x[n,ci,d+a,h+b,w+c] * Weff[ci,co,a,b,c].
// Per output position that is a dot product of length K = 8*C_in for each of
// the 16 output channels: a (positions x K) x (K x 16) matrix product whose
// A row is the position's 2x2x2 x C_in input neighbourhood.  On the FP32 pipe
// it costs 24 FMAs per output plus the loads and moves around them, and the
// instruction issue, not HBM, bounds it.  Here the tensor core does the
// product and the SM only gathers A and stores y.
//
// Precision (3xTF32): every operand v is split as hi = v with the low 13 bits
// of its fp32 pattern cleared (exactly a tf32) and lo = v - hi (exact in fp32;
// the tensor core reads its leading tf32 bits), and each product is
// accumulated as lo(x)hi(w) + hi(x)lo(w) + hi(x)hi(w) in fp32.  The terms
// left out are below 2^-21 of each product.
//
// Design (GB300): one persistent CTA per SM holding all 512 tensor-memory
// columns, 16 warps in 4 groups of 4.  A unit is up to 32 output rows x 32
// output columns of one (n, od) plane; units are dealt round-robin.  Thread 0
// keeps a 4-stage ring of units in flight, one 4-D TMA box each (C_in
// channels x 2 input planes x 33 rows x 32/36 columns, zero-filled outside
// the tensor) behind full/empty mbarriers, and writes each unit's coordinates
// into its stage's slot.  An M-tile is 4 output rows x 32 columns = 128
// positions; group g takes tiles g and g+4 of each unit (its tile 0 and tile
// 1, through tile buffers 0 and 1), warp q of the group row q of a tile
// (tensor-memory lanes 32q..32q+31, the lanes a warp may address), lane l
// column l.  Per tile each thread reads its 8*C_in inputs from shared memory
// (32 consecutive words per warp load), splits them and writes its hi and lo
// A row into its lane with tcgen05.st; a group barrier then hands the tile to
// its MMA thread (lane 0 of the group's warp 0 for tile 0, warp 1 for tile 1),
// which issues the tile's 3*C_in MMAs (M 128, N 16, K 8, A from tensor
// memory, B = the collapsed weights in shared memory) and commits to the
// buffer's barrier.  The epilogue of a buffer -- wait for the commit, load the
// accumulator row, add the folded bias, one whole-warp store per channel row
// -- runs one step behind: per unit a group gathers tile 0, issues it, stores
// the previous unit's tile 1, gathers tile 1, releases the stage, issues
// tile 1 and stores tile 0, so that each MMA chain runs while the group
// works on the other buffer.  Every wait is bounded; each group barrier also
// carries each warp's "go on" vote, so that a group whose wait ran out leaves
// together, drains what it issued and frees the tensor memory.  The kernel is
// launched as a programmatic dependent of the one before it on the stream:
// barrier set-up and the tensor-memory allocation overlap that kernel's tail.
// That is the kernel for C_in <= 3; C_in 4..8, whose A rows do not fit a tile
// buffer, runs ct3d_pool2_tc_chunked_kernel below (the same units and groups,
// each tile's product in chunks of up to 3 input channels).
#include <algorithm>
#include <cstring>
#include <type_traits>

#include "aps_dev.cuh"
#include "aps_internal.h"
#include "aps_tc.cuh"

namespace aps {
namespace ctc {
constexpr int COUT = 16;
constexpr int CIN_MAX = 3;                 // K = 8*C_in <= 24: A hi + lo fit 48 columns
constexpr int GROUPS = 4;
constexpr int WARPS = 4 * GROUPS;
constexpr int THREADS = 32 * WARPS;        // 512
constexpr int TILE_ROWS = 4;               // 4 rows x 32 columns = MMA M 128
constexpr int UNIT_ROWS = 32;
constexpr int UNIT_COLS = 32;
constexpr int TILES_PER_GROUP = UNIT_ROWS / TILE_ROWS / GROUPS;   // 2
constexpr int STAGES = 4;                  // input ring: units in flight ahead of the math
constexpr int TMEM_COLS = 512;
constexpr int GROUP_COLS = TMEM_COLS / GROUPS;                    // 128: two tile buffers
constexpr int BUF_COLS = GROUP_COLS / TILES_PER_GROUP;            // 64: A hi, A lo, D
constexpr int D_COL = 48;                                         // accumulator, 16 columns
constexpr int SLACK = 64;                  // floats after a stage: lanes past the last column read on
// Fixed head of the dynamic shared memory (bytes); the stages follow.
constexpr int OFF_FULL = 0;                // uint64 [STAGES]
constexpr int OFF_EMPTY = 32;              // uint64 [STAGES]
constexpr int OFF_DFULL = 64;              // uint64 [GROUPS][2]: a tile buffer's MMAs are done
constexpr int OFF_TMEM = 128;              // uint32: tensor-memory base
constexpr int OFF_ABORT = 132;             // int
constexpr int OFF_SLOT = 144;              // UnitSlot [STAGES]
constexpr int OFF_BIAS = 320;              // float [16]
constexpr int OFF_B = 384;                 // B operand, hi then lo: [C_in][2][16][4] words each
constexpr int B_CI_BYTES = 2 * COUT * 16;  // one input channel's K-step of 8: 512 bytes
constexpr int HEAD_BYTES = OFF_B + 2 * CIN_MAX * B_CI_BYTES;      // 3456, a multiple of 128
static_assert(HEAD_BYTES % 128 == 0, "stages start 128-byte aligned");
static_assert(OFF_EMPTY - OFF_FULL >= 8 * STAGES && OFF_DFULL - OFF_EMPTY >= 8 * STAGES &&
                  OFF_TMEM - OFF_DFULL >= 16 * GROUPS,
              "barrier arrays fit");
static_assert(D_COL + COUT <= BUF_COLS && 16 * CIN_MAX <= D_COL, "tile buffer layout");

struct UnitSlot {
    long long n;
    int od, oh0, ow0, rows, cols, pad;
};
static_assert(sizeof(UnitSlot) * STAGES <= OFF_BIAS - OFF_SLOT, "slots fit");

// C_in 4..8 (the chunked kernel): the head holds B for up to 8 channels
constexpr int CIN_CHUNKED_MAX = 8;
constexpr int HEAD_BYTES_CHUNKED = OFF_B + 2 * CIN_CHUNKED_MAX * B_CI_BYTES;   // 8576
static_assert(HEAD_BYTES_CHUNKED % 128 == 0, "stages start 128-byte aligned");

// B = collapsed weights, split hi / lo, K-major: word (ci, kc, co, e) holds
// Weff[ci][co][tap 4*kc+e] (tap = a*4 + b*2 + c), so that input channel ci is
// one K-step of 8 and its core matrices (8 co x 4 taps) lie 128 bytes apart
// along N and 256 bytes apart along K; lo follows hi after CIN*512 bytes.  The
// folded bias goes to bsm.  Each collapsed tap of one (ci, co) sums its (up to
// 8) weights, read by independent loads, in ascending (kd, kh, kw).
template <int CIN>
__device__ __forceinline__ void build_collapsed_b(uint32_t *bop, float *bsm,
                                                  const float *__restrict__ w,
                                                  const float *__restrict__ conv_bias,
                                                  const float *__restrict__ bias, float scale1,
                                                  float scale2, int tid) {
    const float wscale = scale1 * scale2 * 0.125f;
    for (int i = tid; i < CIN * 8 * COUT; i += THREADS) {
        const int co = i % COUT, t = (i / COUT) % 8, ci = i / (8 * COUT);
        const float v = collapse_tap_ldg(w + (size_t)(ci * COUT + co) * 27, t) * wscale;
        const uint32_t hi = __float_as_uint(v) & 0xFFFFE000u;
        const int word = ((ci * 2 + (t >> 2)) * COUT + co) * 4 + (t & 3);
        bop[word] = hi;
        bop[CIN * 8 * COUT + word] = __float_as_uint(v - __uint_as_float(hi));
    }
    if (tid < COUT) {
        const float cb = conv_bias ? __ldg(conv_bias + tid) : 0.f;
        bsm[tid] = fmaf(cb, scale1, __ldg(bias + tid)) * scale2;
    }
}

// Decodes unit u (a block of up to RB output rows x WB output columns of one
// (n, od) plane) into slot g and loads its input window -- C_in channels x 2
// planes from (od, oh0, ow0), zero-filled outside the tensor -- into dst by one
// 4-D TMA box behind barrier bar.  Issued by one thread.
__device__ __forceinline__ void fill_unit(UnitSlot &g, uint64_t *bar, float *dst,
                                          const CUtensorMap *xmap, long long u, int n_owb,
                                          int n_ohb, int Do, int Ho, int Wo, int RB, int WB,
                                          int cin, uint32_t bytes) {
    const int owb = (int)(u % n_owb);
    long long t = u / n_owb;
    const int ohb = (int)(t % n_ohb);
    t /= n_ohb;
    const int od = (int)(t % Do);
    const long long n = t / Do;
    const int oh0 = ohb * RB, ow0 = owb * WB;
    g.n = n;
    g.od = od;
    g.oh0 = oh0;
    g.ow0 = ow0;
    g.rows = Ho - oh0 < RB ? Ho - oh0 : RB;
    g.cols = Wo - ow0 < WB ? Wo - ow0 : WB;
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    mbar_arrive_expect_tx(bar, bytes);
    tma_load_4d(dst, xmap, bar, ow0, oh0, od, (int)(n * cin));
}

// Calls f(std::integral_constant<int, I>) for I = 0 .. N-1, unrolled.
template <int N, int I = 0, class F>
__device__ __forceinline__ void static_for(F &&f) {
    if constexpr (I < N) {
        f(std::integral_constant<int, I>{});
        static_for<N, I + 1>(f);
    }
}

// Floats one stage occupies: the staged window plus the rows the last tile
// may still read (up to row UNIT_ROWS), plus slack.
__host__ __device__ inline int stage_stride_of(int Cin, int XR, int BW) {
    return (Cin * 2 * XR * BW + (UNIT_ROWS + 1 - XR) * BW + SLACK + 31) & ~31;
}
}  // namespace ctc

// CIN: input channels (1..3); BW_T: staged row length fixed at compile time
// (0: run time).
template <int CIN, int BW_T>
__global__ void __launch_bounds__(ctc::THREADS, 1)
    ct3d_pool2_tc_kernel(const __grid_constant__ CUtensorMap xmap, const float *__restrict__ w,
                         const float *__restrict__ conv_bias, const float *__restrict__ bias,
                         float scale1, float scale2, float *__restrict__ y, int Do, int Ho, int Wo,
                         int BW_rt, int XR, int RB, int WB, int n_ohb, int n_owb,
                         long long n_units, unsigned int *status) {
    using namespace ctc;
    const int BW = BW_T ? BW_T : BW_rt;
    extern __shared__ __align__(128) unsigned char smraw[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smraw + OFF_FULL);
    uint64_t *empty = reinterpret_cast<uint64_t *>(smraw + OFF_EMPTY);
    uint64_t *dfull = reinterpret_cast<uint64_t *>(smraw + OFF_DFULL);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smraw + OFF_TMEM);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smraw + OFF_ABORT);
    UnitSlot *slot = reinterpret_cast<UnitSlot *>(smraw + OFF_SLOT);
    float *bsm = reinterpret_cast<float *>(smraw + OFF_BIAS);
    uint32_t *bop = reinterpret_cast<uint32_t *>(smraw + OFF_B);
    float *xs = reinterpret_cast<float *>(smraw + HEAD_BYTES);   // [STAGES][C_in][2][XR][BW]
    const int stage_floats = CIN * 2 * XR * BW;
    const int stage_stride = stage_stride_of(CIN, XR, BW);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int grp = warp >> 2, q = warp & 3;

    // decode unit u into the slot of stage b and load its input window
    auto fill = [&](long long u, int b) {
        fill_unit(slot[b], &full[b], xs + b * stage_stride, &xmap, u, n_owb, n_ohb, Do, Ho, Wo, RB,
                  WB, CIN, (uint32_t)stage_floats * 4u);
    };

    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], WARPS);
        }
        for (int g = 0; g < 2 * GROUPS; ++g) mbar_init(&dfull[g], 1);
        *abort_flag = 0;
        mbar_fence_init();
    }
    // barrier set-up and the tensor-memory allocation overlap the kernel
    // before this one on the stream; global memory waits for it
    pdl_trigger();
    if (warp == 0) tc::tmem_alloc(tmem_slot, TMEM_COLS);
    __syncthreads();
    pdl_wait();
    uint32_t issued = 0;   // units thread 0 has filled
    if (tid == 0) {
        tma_prefetch_desc(&xmap);
        for (; issued < STAGES - 1 && (long long)blockIdx.x + (long long)issued * gridDim.x < n_units;
             ++issued)
            fill(blockIdx.x + (long long)issued * gridDim.x, (int)issued);
    }

    // ---- B = collapsed weights (hi, lo) and the folded bias
    build_collapsed_b<CIN>(bop, bsm, w, conv_bias, bias, scale1, scale2, tid);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // B is read by the tensor core
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    const long long plane = (long long)Ho * Wo;
    const int cs = (int)(Do * plane);                    // between output channels (< 2^27)
    constexpr uint32_t IDESC = tc::idesc_tf32(128, COUT);
    const uint32_t b_hi = smem_u32(bop), b_lo = b_hi + CIN * B_CI_BYTES;
    const uint32_t lane_q = (uint32_t)(32 * q) << 16;   // this warp's tensor-memory lanes
    const uint32_t gcol = (uint32_t)(grp * GROUP_COLS); // the group's two tile buffers
    const int gbar = 1 + grp;                            // the group's barrier (0 is __syncthreads)
    float bias_r[COUT];
#pragma unroll
    for (int co = 0; co < COUT; ++co) bias_r[co] = bsm[co];
    uint32_t k = 0;                                      // units this CTA has taken
    bool fail = false;
    uint64_t *dfb = dfull + 2 * grp;                     // its two buffers' MMA-done barriers
    // tile j of a unit goes through buffer j; buffer 1's epilogue runs one
    // step later, so that each MMA chain runs under the other buffer's
    // epilogue and gather
    auto gather = [&](const float *xb, int j) {
        const int h = TILE_ROWS * (grp + GROUPS * j) + q;
        uint32_t av[16 * CIN];   // hi[0 .. 8*CIN), then lo
#pragma unroll
        for (int ci = 0; ci < CIN; ++ci)
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                const int a = t >> 2, bb = (t >> 1) & 1, c = t & 1;
                const float v = xb[((ci * 2 + a) * XR + h + bb) * BW + lane + c];
                const uint32_t hi = __float_as_uint(v) & 0xFFFFE000u;
                av[ci * 8 + t] = hi;
                av[8 * CIN + ci * 8 + t] = __float_as_uint(v - __uint_as_float(hi));
            }
        const uint32_t col = gcol + (uint32_t)(j * BUF_COLS);
#pragma unroll
        for (int s = 0; s < CIN; ++s) tc::tmem_st16(tmem + lane_q + col + 16 * s, av + 16 * s);
        tc::tmem_st_wait();
    };
    auto issue = [&](int j, int rows) {
        if (q == j && lane == 0) {
            tc::tc_fence_after();
            if (TILE_ROWS * (grp + GROUPS * j) < rows) {
                const uint32_t col = gcol + (uint32_t)(j * BUF_COLS);
                const uint32_t d = tmem + col + D_COL;
#pragma unroll
                for (int ci = 0; ci < CIN; ++ci) {
                    const uint32_t ahi = tmem + col + 8 * ci, alo = ahi + 8 * CIN;
                    const uint64_t bh = tc::umma_desc(b_hi + ci * B_CI_BYTES, 256, 128);
                    const uint64_t bl = tc::umma_desc(b_lo + ci * B_CI_BYTES, 256, 128);
                    tc::umma_tf32_ts(d, alo, bh, IDESC, ci > 0 ? 1u : 0u);   // lo(x) hi(w)
                    tc::umma_tf32_ts(d, ahi, bl, IDESC, 1u);                 // hi(x) lo(w)
                    tc::umma_tf32_ts(d, ahi, bh, IDESC, 1u);                 // hi(x) hi(w)
                }
            }
            tc::umma_commit(&dfb[j]);
        }
        __syncwarp();
    };
    // wait for buffer j's MMAs of the unit taken k-th; then its accumulator
    // row + bias -> 16 whole-warp row stores
    auto epilogue = [&](int j, uint32_t kk, float *yb, int rows, bool ready) {
        if (!ready && !mbar_wait(&dfb[j], kk & 1u)) {
            record_error(status, APS_DEVERR_TIMEOUT);
            *abort_flag = 1;
            fail = true;
        }
        fail = __any_sync(0xffffffffu, fail);
        if (fail) return;
        tc::tc_fence_after();
        uint32_t d[COUT];
        tc::tmem_ld16(tmem + lane_q + gcol + (uint32_t)(j * BUF_COLS) + D_COL, d);
        const int h = TILE_ROWS * (grp + GROUPS * j) + q;
        if (h < rows && yb) {
            float *yr = yb + h * Wo;
#pragma unroll
            for (int co = 0; co < COUT; ++co) yr[co * cs] = __uint_as_float(d[co]) + bias_r[co];
        }
    };
    float *prev_y = nullptr;   // the previous unit's output corner (this lane's column)
    int prev_rows = 0;
    uint32_t c0 = 0, c1 = 0;         // commits to each buffer's barrier
    // Each shared-memory access here waits behind the gathers' and the tensor
    // core's traffic, so whether the next unit's box has landed, the previous
    // unit's tile-1 MMAs are done and another thread has aborted are asked early
    // (a non-blocking barrier test, a plain load) and answered while this unit's
    // work runs.
    bool full_ready = false;         // early answers for the next unit
    int abort_seen = 0;
    for (long long u = blockIdx.x; u < n_units; u += gridDim.x, ++k) {
        const int b = (int)(k % STAGES);
        const long long ahead = u + (long long)(STAGES - 1) * gridDim.x;
        if (tid == 0 && !abort_seen && ahead < n_units) {
            const int nb = (int)((k + STAGES - 1) % STAGES);
            if (k >= 1 && !mbar_wait(&empty[nb], ((k - 1) / STAGES) & 1u)) {
                record_error(status, APS_DEVERR_TIMEOUT);
                *abort_flag = 1;
            } else {
                fill(ahead, nb);
                ++issued;
            }
        }
        bool ok = !fail && !abort_seen;
        if (ok && !full_ready && !mbar_wait(&full[b], (k / STAGES) & 1u)) {
            record_error(status, APS_DEVERR_TIMEOUT);
            *abort_flag = 1;
            ok = false;
        }
        ok = __all_sync(0xffffffffu, ok);
        // the previous unit's tile-1 MMAs: asked now, needed after this unit's tile 0
        const bool d1_ready = k > 0 && mbar_test(&dfb[1], (k - 1) & 1u);
        const int grows = ok ? slot[b].rows : 0;
        const float *xb = xs + b * stage_stride;
        if (ok && TILE_ROWS * grp < grows) gather(xb, 0);
        tc::tc_fence_before();
        __syncwarp();
        if (tc::named_bar_or(gbar, 128, !ok)) break;
        issue(0, grows);
        ++c0;
        if (k > 0) epilogue(1, k - 1, prev_y, prev_rows, d1_ready);
        if (!fail && TILE_ROWS * (grp + GROUPS) < grows) gather(xb, 1);
        const long long gn = slot[b].n;
        const int god = slot[b].od, goh0 = slot[b].oh0, gow0 = slot[b].ow0, gcols = slot[b].cols;
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[b]);
        tc::tc_fence_before();
        __syncwarp();
        if (tc::named_bar_or(gbar, 128, fail)) break;
        issue(1, grows);
        ++c1;
        // the next unit's box and the abort flag, answered during the epilogue below
        full_ready = mbar_test(&full[(k + 1) % STAGES], ((k + 1) / STAGES) & 1u);
        abort_seen = *abort_flag;
        float *ycur = lane < gcols
            ? y + ((gn * COUT) * Do + god) * plane + (long long)goh0 * Wo + gow0 + lane : nullptr;
        epilogue(0, k, ycur, grows, false);
        prev_y = ycur;
        prev_rows = grows;
    }
    // the last unit's buffer-1 tiles
    if (__all_sync(0xffffffffu, c1 > 0 && c1 == k && !fail && !*abort_flag))
        epilogue(1, c1 - 1, prev_y, prev_rows, false);

    // ---- leave nothing in flight: each buffer's last MMAs (their wait may
    // have run out), the fills no warp consumed; then free the tensor memory
    if (q < 2 && lane == 0) {
        const uint32_t c = q ? c1 : c0;
        if (c > 0) mbar_wait(&dfb[q], (c - 1) & 1u);
    }
    if (tid == 0)
        for (uint32_t j = k; j < issued; ++j) mbar_wait(&full[j % STAGES], (j / STAGES) & 1u);
    tc::tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, TMEM_COLS);
    }
}

// C_in 4..8: K = 8*C_in does not fit a tile buffer, so each tile's product runs
// as NCH chunks of at most 3 input channels.  A group's 128 tensor-memory
// columns hold two A slots (hi + lo of one chunk, 48 columns each) and the
// accumulators of its two tiles (16 columns each).  Chunk steps alternate the
// A slots: a step's gather waits for the MMAs of the step two before it, so
// that it overlaps the MMAs of the step just before.  Lane 0 of one warp of
// the group (warp g of group g, so that the four issuers sit on four
// schedulers) issues every step and commits it to its slot's barrier; one
// thread issuing makes each commit cover all the group's earlier MMAs, so a
// tile is done when its last step's commit arrives.  The stage ring holds nst (2..4)
// units, as many as shared memory takes.
template <int CIN, int BW_T>
__global__ void __launch_bounds__(ctc::THREADS, 1)
    ct3d_pool2_tc_chunked_kernel(const __grid_constant__ CUtensorMap xmap,
                                 const float *__restrict__ w,
                                 const float *__restrict__ conv_bias,
                                 const float *__restrict__ bias, float scale1, float scale2,
                                 float *__restrict__ y, int Do, int Ho, int Wo, int BW_rt, int XR,
                                 int RB, int WB, int n_ohb, int n_owb, long long n_units, int nst,
                                 unsigned int *status) {
    using namespace ctc;
    constexpr int NCH = (CIN + 2) / 3;                  // chunks per tile
    constexpr int CH = (CIN + NCH - 1) / NCH;           // channels per chunk (the last: fewer)
    constexpr int A_COLS = 16 * CH;                     // one A slot: hi + lo
    constexpr int ACC_COL = 2 * A_COLS;                 // the two accumulators follow
    static_assert(CIN <= CIN_CHUNKED_MAX && CH <= 3 && ACC_COL + 2 * COUT <= GROUP_COLS,
                  "chunk buffers fit a group's columns");
    const int BW = BW_T ? BW_T : BW_rt;
    extern __shared__ __align__(128) unsigned char smraw[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smraw + OFF_FULL);
    uint64_t *empty = reinterpret_cast<uint64_t *>(smraw + OFF_EMPTY);
    uint64_t *dslot = reinterpret_cast<uint64_t *>(smraw + OFF_DFULL);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smraw + OFF_TMEM);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smraw + OFF_ABORT);
    UnitSlot *slot = reinterpret_cast<UnitSlot *>(smraw + OFF_SLOT);
    float *bsm = reinterpret_cast<float *>(smraw + OFF_BIAS);
    uint32_t *bop = reinterpret_cast<uint32_t *>(smraw + OFF_B);
    float *xs = reinterpret_cast<float *>(smraw + HEAD_BYTES_CHUNKED);
    const int stage_floats = CIN * 2 * XR * BW;
    const int stage_stride = stage_stride_of(CIN, XR, BW);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int grp = warp >> 2, q = warp & 3;
    const uint32_t ust = (uint32_t)nst;

    auto fill = [&](long long u, int b) {
        fill_unit(slot[b], &full[b], xs + b * stage_stride, &xmap, u, n_owb, n_ohb, Do, Ho, Wo, RB,
                  WB, CIN, (uint32_t)stage_floats * 4u);
    };

    if (tid == 0) {
        for (int s = 0; s < nst; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], WARPS);
        }
        for (int g = 0; g < 2 * GROUPS; ++g) mbar_init(&dslot[g], 1);
        *abort_flag = 0;
        mbar_fence_init();
    }
    pdl_trigger();
    if (warp == 0) tc::tmem_alloc(tmem_slot, TMEM_COLS);
    __syncthreads();
    pdl_wait();
    uint32_t issued = 0;
    if (tid == 0) {
        tma_prefetch_desc(&xmap);
        for (; issued + 1 < ust && (long long)blockIdx.x + (long long)issued * gridDim.x < n_units;
             ++issued)
            fill(blockIdx.x + (long long)issued * gridDim.x, (int)issued);
    }
    build_collapsed_b<CIN>(bop, bsm, w, conv_bias, bias, scale1, scale2, tid);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    const long long plane = (long long)Ho * Wo;
    const int cs = (int)(Do * plane);
    constexpr uint32_t IDESC = tc::idesc_tf32(128, COUT);
    const uint32_t b_hi = smem_u32(bop), b_lo = b_hi + CIN * B_CI_BYTES;
    const uint32_t lane_q = (uint32_t)(32 * q) << 16;
    const uint32_t gcol = (uint32_t)(grp * GROUP_COLS);
    const int gbar = 1 + grp;
    float bias_r[COUT];
#pragma unroll
    for (int co = 0; co < COUT; ++co) bias_r[co] = bsm[co];
    uint64_t *dsb = dslot + 2 * grp;   // the group's two A-slot barriers
    // the group's issuing warp: warp q of a group runs on scheduler q, so the four
    // groups' issuers take one scheduler each (all on one: 86.7 -> 79.0 us at C_in 8)
    const int iq = grp & 3;
    bool fail = false, stopped = false;

    // waits (bounded) for the MMAs of chunk step st; false (warp-uniform) on a timeout
    auto step_done = [&](uint32_t st) {
        if (!fail && !mbar_wait(&dsb[st & 1u], (st >> 1) & 1u)) {
            record_error(status, APS_DEVERR_TIMEOUT);
            *abort_flag = 1;
            fail = true;
        }
        fail = __any_sync(0xffffffffu, fail);
        return !fail;
    };
    // chunk c of tile j: this thread's 8 inputs per channel, split, into A slot sl
    auto gather = [&](const float *xb, int j, auto cc, uint32_t sl) {
        constexpr int C0 = decltype(cc)::value * CH;
        constexpr int NC = CIN - C0 < CH ? CIN - C0 : CH;
        const int h = TILE_ROWS * (grp + GROUPS * j) + q;
        uint32_t av[16 * NC];   // hi[0 .. 8*NC), then lo
#pragma unroll
        for (int i = 0; i < NC; ++i)
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                const int a = t >> 2, bb = (t >> 1) & 1, c = t & 1;
                const float v = xb[(((C0 + i) * 2 + a) * XR + h + bb) * BW + lane + c];
                const uint32_t hi = __float_as_uint(v) & 0xFFFFE000u;
                av[i * 8 + t] = hi;
                av[8 * NC + i * 8 + t] = __float_as_uint(v - __uint_as_float(hi));
            }
        const uint32_t col = gcol + sl * (uint32_t)A_COLS;
#pragma unroll
        for (int s2 = 0; s2 < NC; ++s2)
            tc::tmem_st16(tmem + lane_q + col + 16 * s2, av + 16 * s2);
        tc::tmem_st_wait();
    };
    auto issue = [&](int j, auto cc, uint32_t sl, bool active) {
        constexpr int c = decltype(cc)::value;
        constexpr int C0 = c * CH;
        constexpr int NC = CIN - C0 < CH ? CIN - C0 : CH;
        if (q == iq && lane == 0) {
            tc::tc_fence_after();
            if (active) {
                const uint32_t a = tmem + gcol + sl * (uint32_t)A_COLS;
                const uint32_t d = tmem + gcol + ACC_COL + 16 * j;
#pragma unroll
                for (int i = 0; i < NC; ++i) {
                    const uint32_t ahi = a + 8 * i, alo = a + 8 * NC + 8 * i;
                    const uint64_t bh = tc::umma_desc(b_hi + (C0 + i) * B_CI_BYTES, 256, 128);
                    const uint64_t bl = tc::umma_desc(b_lo + (C0 + i) * B_CI_BYTES, 256, 128);
                    tc::umma_tf32_ts(d, alo, bh, IDESC, (c > 0 || i > 0) ? 1u : 0u);
                    tc::umma_tf32_ts(d, ahi, bl, IDESC, 1u);
                    tc::umma_tf32_ts(d, ahi, bh, IDESC, 1u);
                }
            }
            tc::umma_commit(&dsb[sl]);
        }
        __syncwarp();
    };
    // tile j's accumulator (done with chunk step st) + bias -> 16 whole-warp row stores
    auto epilogue = [&](int j, uint32_t st, float *yb, int rows) {
        if (!step_done(st)) return;
        tc::tc_fence_after();
        uint32_t d[COUT];
        tc::tmem_ld16(tmem + lane_q + gcol + ACC_COL + 16 * j, d);
        const int h = TILE_ROWS * (grp + GROUPS * j) + q;
        if (h < rows && yb) {
            float *yr = yb + h * Wo;
#pragma unroll
            for (int co = 0; co < COUT; ++co) yr[co * cs] = __uint_as_float(d[co]) + bias_r[co];
        }
    };

    float *prev_y = nullptr;
    int prev_rows = 0;
    uint32_t k = 0, s = 0;   // units taken, chunk steps issued
    for (long long u = blockIdx.x; u < n_units; u += gridDim.x, ++k) {
        const uint32_t b = k % ust;
        const long long ahead = u + (long long)(nst - 1) * gridDim.x;
        if (tid == 0 && !*abort_flag && ahead < n_units) {
            const uint32_t nb = (k + ust - 1) % ust;
            if (k >= 1 && !mbar_wait(&empty[nb], ((k - 1) / ust) & 1u)) {
                record_error(status, APS_DEVERR_TIMEOUT);
                *abort_flag = 1;
            } else {
                fill(ahead, (int)nb);
                ++issued;
            }
        }
        bool ok = !fail && !*abort_flag;
        if (ok && !mbar_wait(&full[b], (k / ust) & 1u)) {
            record_error(status, APS_DEVERR_TIMEOUT);
            *abort_flag = 1;
            ok = false;
        }
        ok = __all_sync(0xffffffffu, ok);
        int grows = 0, gcols = 0, god = 0, goh0 = 0, gow0 = 0;
        long long gn = 0;
        if (ok) {
            grows = slot[b].rows;
            gcols = slot[b].cols;
            gn = slot[b].n;
            god = slot[b].od;
            goh0 = slot[b].oh0;
            gow0 = slot[b].ow0;
        }
        float *ycur = ok && lane < gcols
            ? y + ((gn * COUT) * Do + god) * plane + (long long)goh0 * Wo + gow0 + lane : nullptr;
        const float *xb = xs + b * stage_stride;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const bool active = TILE_ROWS * (grp + GROUPS * j) < grows;
            static_for<NCH>([&](auto cc) {
                constexpr int c = decltype(cc)::value;
                if (stopped) return;
                const uint32_t sl = s & 1u;
                // the slot's last readers: the MMAs of step s - 2
                const bool free = s < 2 || step_done(s - 2);
                if (free && ok && active) {
                    tc::tc_fence_after();
                    gather(xb, j, cc, sl);
                }
                if (j == 1 && c == NCH - 1) {   // the unit's input is no longer read
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&empty[b]);
                }
                tc::tc_fence_before();
                __syncwarp();
                if (tc::named_bar_or(gbar, 128, !ok || fail)) {
                    stopped = true;
                    return;
                }
                issue(j, cc, sl, active);
                ++s;
                if (c == 0) {
                    // the tile before this one (its last step is s - 2) is stored
                    // while this tile's remaining chunks are gathered
                    if (j == 0 && k > 0) epilogue(1, s - 2, prev_y, prev_rows);
                    if (j == 1) epilogue(0, s - 2, ycur, grows);
                }
            });
        }
        if (stopped) break;
        prev_y = ycur;
        prev_rows = grows;
    }
    // the last unit's tile 1
    if (__all_sync(0xffffffffu, !stopped && k > 0 && !fail && !*abort_flag))
        epilogue(1, s - 1, prev_y, prev_rows);

    // ---- leave nothing in flight: the group's last commit (it covers all its
    // MMAs), the fills no warp consumed; then free the tensor memory
    if (q == iq && lane == 0 && s > 0) mbar_wait(&dsb[(s - 1) & 1u], ((s - 1) >> 1) & 1u);
    if (tid == 0)
        for (uint32_t j = k; j < issued; ++j) mbar_wait(&full[j % ust], (j / ust) & 1u);
    tc::tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, TMEM_COLS);
    }
}

aps_status launch_ct3d_pool2_tc(const float *x, const int64_t in[5], const float *w,
                                const float *conv_bias, const float *bias, float scale1,
                                float scale2, float *y, const int64_t out[5], cudaStream_t st) {
    using namespace ctc;
    const int64_t N = in[0], Cin = in[1], D = in[2], H = in[3], W = in[4];
    // the TMA box needs 16-byte rows; C_in 4..8 runs in chunks of <= 3 channels
    if (Cin < 1 || Cin > CIN_CHUNKED_MAX || D < 2 || H < 2 || W < 2 || W % 4 != 0 ||
        reinterpret_cast<uintptr_t>(x) % 16 != 0 || D >= (1 << 30) || H >= (1 << 30) ||
        W >= (1 << 30) || N * Cin >= (1ll << 31))
        return APS_ERR_UNSUPPORTED;
    const int64_t Do = out[2], Ho = out[3], Wo = out[4];
    if (Do * Ho * Wo >= (1ll << 27)) return APS_ERR_UNSUPPORTED;   // channel offsets in 32 bits
    const int RB = (int)std::min<int64_t>(Ho, UNIT_ROWS), WB = (int)std::min<int64_t>(Wo, UNIT_COLS);
    const int64_t n_ohb = ceil_div(Ho, RB), n_owb = ceil_div(Wo, WB);
    const long long n_units = N * Do * n_ohb * n_owb;
    const int XR = RB + 1;                  // staged rows
    const int BW = (WB + 1 + 3) & ~3;       // staged columns, a multiple of 4
    CUtensorMap map;
    const cuuint64_t dims[4] = {(cuuint64_t)W, (cuuint64_t)H, (cuuint64_t)D, (cuuint64_t)(N * Cin)};
    const cuuint64_t strides[3] = {(cuuint64_t)(W * 4), (cuuint64_t)(H * W * 4),
                                   (cuuint64_t)(D * H * W * 4)};
    const cuuint32_t box[4] = {(cuuint32_t)BW, (cuuint32_t)XR, 2, (cuuint32_t)Cin};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    if (!encode_tiled(&map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<float *>(x), dims,
                      strides, box, estr))
        return APS_ERR_UNSUPPORTED;
    if (Cin > CIN_MAX) {
        // as many stages (2..4) as shared memory takes
        const size_t stage = (size_t)stage_stride_of((int)Cin, XR, BW) * 4;
        int nst = STAGES;
        while (nst > 2 && HEAD_BYTES_CHUNKED + nst * stage > kMaxSmemPerCta) --nst;
        const size_t smem = HEAD_BYTES_CHUNKED + nst * stage;
        if (smem > kMaxSmemPerCta) return APS_ERR_UNSUPPORTED;
        using KernC = void (*)(CUtensorMap, const float *, const float *, const float *, float,
                               float, float *, int, int, int, int, int, int, int, int, int,
                               long long, int, unsigned int *);
        static const KernC k32[5] = {
            ct3d_pool2_tc_chunked_kernel<4, 32>, ct3d_pool2_tc_chunked_kernel<5, 32>,
            ct3d_pool2_tc_chunked_kernel<6, 32>, ct3d_pool2_tc_chunked_kernel<7, 32>,
            ct3d_pool2_tc_chunked_kernel<8, 32>};
        static const KernC krt[5] = {
            ct3d_pool2_tc_chunked_kernel<4, 0>, ct3d_pool2_tc_chunked_kernel<5, 0>,
            ct3d_pool2_tc_chunked_kernel<6, 0>, ct3d_pool2_tc_chunked_kernel<7, 0>,
            ct3d_pool2_tc_chunked_kernel<8, 0>};
        const KernC kern = (BW == 32 ? k32 : krt)[Cin - 4];
        if (resident_ctas((const void *)kern, THREADS, (int)smem) < 1) return APS_ERR_UNSUPPORTED;
        const long long grid = std::min<long long>(sm_count(), n_units);
        const cudaError_t e = launch_pdl(kern, dim3((unsigned)grid), dim3(THREADS), smem, st, map,
                                         w, conv_bias, bias, scale1, scale2, y, (int)Do, (int)Ho,
                                         (int)Wo, BW, XR, RB, WB, (int)n_ohb, (int)n_owb, n_units,
                                         nst, status_word());
        return launch_status(e);
    }
    const size_t smem = (size_t)HEAD_BYTES + (size_t)STAGES * stage_stride_of((int)Cin, XR, BW) * 4;
    using Kern = void (*)(CUtensorMap, const float *, const float *, const float *, float, float,
                          float *, int, int, int, int, int, int, int, int, int, long long,
                          unsigned int *);
    Kern kern;
    if (BW == 32)
        kern = Cin == 1 ? ct3d_pool2_tc_kernel<1, 32>
             : Cin == 2 ? ct3d_pool2_tc_kernel<2, 32>
                        : ct3d_pool2_tc_kernel<3, 32>;
    else
        kern = Cin == 1 ? ct3d_pool2_tc_kernel<1, 0>
             : Cin == 2 ? ct3d_pool2_tc_kernel<2, 0>
                        : ct3d_pool2_tc_kernel<3, 0>;
    // one CTA per SM: each holds all 512 tensor-memory columns
    if (resident_ctas((const void *)kern, THREADS, (int)smem) < 1) return APS_ERR_UNSUPPORTED;
    const long long grid = std::min<long long>(sm_count(), n_units);
    const cudaError_t e = launch_pdl(kern, dim3((unsigned)grid), dim3(THREADS), smem, st, map, w, conv_bias, bias,
               scale1, scale2, y, (int)Do, (int)Ho, (int)Wo, BW, XR, RB, WB, (int)n_ohb,
               (int)n_owb, n_units, status_word());
    return launch_status(e);
}

}  // namespace aps
