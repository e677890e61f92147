// convt1d_tc.cu -- ConvTranspose1d as a TF32 implicit GEMM on the tcgen05
// tensor cores (APS_PREC_TF32), and its 3xTF32 form at fp32 accuracy
// (APS_PREC_TF32X3: the MODE_X3 and MODE_X3_PAIRED instantiations, described
// at the end).
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
//  * warp 0, lane 0  -- TMA producer: for each (n, 128-position tile, chunk
//    of 32 (or, split, 16) channels) one 3-D box x[n, ci0:ci0+CKr, a0:a0+BW]
//    (BW = 128 + tap span, start rounded down to 16 bytes; out-of-range cells
//    arrive as zeros) into a ring of up to 4 stages, and an L2 prefetch of the
//    box 4 steps ahead (one CTA per SM holds few stages; the prefetch keeps
//    bytes in flight; 4 measured fastest of 0..24).
//    Warp 0 also owns the tensor-memory allocation.
//  * warps 2, 3, 12..17 -- converters (one per 4 channels): transpose each raw
//    box into the K-major,
//    no-swizzle operand layout (8-row x 16-byte core matrices; rows = window
//    positions, 4 channels per 16 bytes, one block of rows per 4 channels); for
//    tf32 the words go in as they are (the MMA reads their leading 19 bits), for
//    3xTF32 split into hi and lo.  Because rows are 16 bytes apart, the operand of
//    tap k is the same buffer with its start moved by 16 bytes per row of tap
//    offset: one transposed copy serves every tap of every class.
//  * warp 1, lane 0  -- MMA issuer: walks a per-CTA table of descriptors (held in
//    registers for the one-chunk, 20-entry stride-1 K5 geometry) and, per chunk and
//    (class, tap), issues CKr/8 tcgen05.mma
//    kind::tf32 of 128 x C_out x 8 into the class's accumulator in tensor memory
//    (a ring of up to 8 tiles' accumulators, as many as 512 columns hold, so the
//    epilogue's latency never stalls the MMAs), then tcgen05.commit to release the
//    operand stage and, after the last chunk, to hand the tile to the epilogue.
//  * warps 4..11 -- epilogue, two groups of four taking alternate slabs:
//    tcgen05.ld of their 32 accumulator rows, + bias,
//    into shared-memory slabs laid out like the output (class r of position
//    m at s*m + r; residues no tap reaches hold the bias).  With stride <= 2
//    each 16 KB slab leaves by one TMA tensor store (2 per group in flight);
//    otherwise by 128-bit coalesced stores of each channel's s*128 outputs.
// Weights are rounded to tf32 once per CTA into shared memory in the same
// K-major layout, one [C_in/4][C_out][4] block per tap.  Every wait is bounded;
// a wait that times out records APS_DEVERR_TIMEOUT, the CTA drains what it has
// in flight and frees its tensor memory before returning.
// 3xTF32: weights and every converted stage are held twice.  Weights: hi =
// tf32(w) (round to nearest) and lo = tf32(w - hi); inputs: hi = the raw word,
// which the MMA truncates to tf32, and lo = v - trunc_tf32(v).  Each table entry
// issues hi(x)[hi(w) | lo(w)] as one MMA of twice C_out columns and lo(x)hi(w)
// into the first half of the same accumulator (the epilogue adds the halves;
// where 2*C_out is no valid N, the three products go to one accumulator as three
// C_out-wide MMAs).  The dropped lo(x)lo(w) term is below 2^-21 of each product
// and the truncation of lo(x) below 2^-20.  The launcher picks the deepest
// pipeline that fits 227 KB: 32- then 16-channel chunks, 3 then 2 converted
// stages.  Only two converter warps convert in this form, each taking every second
// 4-channel block (hi + lo stores from eight warps at once slowed the MMAs by 3-4 %;
// the strided K4 workload's short chunks run the same with 2, 4 or 8).
#include <algorithm>
#include <type_traits>

#include "aps_dev.cuh"
#include "aps_internal.h"
#include "aps_tc.cuh"

namespace aps {
namespace tc1 {
constexpr int BM = 128;           // positions per tile (MMA M)
constexpr int CK = 32;            // input channels per staged chunk (at most; MMA K per chunk)
constexpr int RAW_STAGES = 4;    // at most; the launcher may use fewer to fit smem
constexpr int XT_STAGES = 3;      // converted-operand stages (at most; the launcher may use 2)
constexpr int MAX_CLASSES = 4;
constexpr int MAX_TAPS = 8;       // taps per class
constexpr int NBUF = 4;           // TMA-store staging slabs in flight (at most; 2 if smem is short)
constexpr int MAX_ACC = 8;        // accumulator buffers in tensor memory (at most)
constexpr int PREFETCH = 4;       // input boxes prefetched into L2 ahead of the loads
                                  // (swept 0..24 on the box: 4 is fastest; 12 cost 9 %
                                  // on the strided workload)
constexpr int THREADS = 576;      // 18 warps
constexpr int CONVERTERS = 8;     // converter warps: 2, 3, 12..17
constexpr int EPI_WARPS = 8;      // two epilogue groups of four warps: 4..7 and 8..11
constexpr int MAX_MMA_TAB = 256;  // (chunk, class, tap, k-step) entries of one tile
constexpr int W_PRODUCER = 0, W_MMA = 1, W_EPI0 = 4;

// Operand forms of the kernel: plain tf32; 3xTF32 with three C_out-wide MMAs per
// product; 3xTF32 with the hi and lo weights side by side in one 2*C_out-wide B (two
// MMAs per product: M128 N2C_out K8 + M128 N_Cout K8 instead of three M128 N_Cout K8,
// 64 + 48 cycles against 3 x 48 at C_out = 64).
constexpr int MODE_TF32 = 0, MODE_X3 = 1, MODE_X3_PAIRED = 2;

struct Taps {
    int nclass;                        // classes (output residues) with taps
    int cls_r[MAX_CLASSES];            // residue of each such class
    int ntaps[MAX_CLASSES];
    int tap_k[MAX_CLASSES][MAX_TAPS];  // weight tap index
    int tap_row[MAX_CLASSES][MAX_TAPS];// first window row used by tile position 0
    int nempty;                        // residues no tap reaches (bias only)
    int empty_r[8];
};

__device__ __forceinline__ int converter_id(int warp) {
    return warp == 2 ? 0 : warp == 3 ? 1 : warp - 10;   // warps 2, 3, 12..17
}

using namespace tc;   // named_bar, to_tf32, umma_*, tc_fence_*, tmem_ld*

// One chunk's MMAs.  Table entry e: A offset (16-byte units) | class << 16 | bit 31 on the
// class's first entry; its B descriptor.  NE > 0: exactly NE entries, UNROLL per turn of
// the loop, so that the table loads go ahead of the MMAs and the MMAs issue back to back;
// the issuing thread's loads and address arithmetic, not the tensor core, set the pace of
// a loop of 2 or 4 entries per turn.  Measured on the stride-1 K5 workload (20 entries):
// fully unrolled 318 / 566 us (TF32 / 3xTF32) against 348 / 675.  The strided K4 workload
// (16 entries) keeps the loop: fully unrolled it was 1.5 % (TF32) and 2 % (3xTF32)
// slower, and 8 per turn for 3xTF32 was 276 against 302 us in one comparison but 312 in
// the bench.  NE == 0: any count, 4 (TF32) or 2 (3xTF32) per turn.
// MODE: MODE_TF32, MODE_X3 (three C_out-wide MMAs per entry) or MODE_X3_PAIRED (hi and lo
// weights side by side as one 2*C_out-wide B: hi(x) [hi(w) | lo(w)], then lo(x) hi(w)).
// `acc_cols`: accumulator columns per class (C_out, or 2*C_out when paired).
// The MMAs of one table entry: its A offset word `ae` and B descriptor `bw`.
template <int MODE>
__device__ __forceinline__ void issue_entry(uint32_t ae, uint64_t bw, uint64_t abase, uint32_t dbase,
                                            uint32_t acc_cols, uint32_t idesc, uint32_t idesc_pair,
                                            bool first_chunk, uint32_t a_lo, uint32_t b_lo) {
    const uint32_t acc = (!first_chunk || !(ae >> 31)) ? 1u : 0u;
    const uint32_t d = dbase + ((ae >> 16) & 0xFFu) * acc_cols;
    const uint64_t a = abase + (ae & 0xFFFFu);
    if (MODE == MODE_X3_PAIRED) {
        umma_tf32(d, a, bw, idesc_pair, acc);     // hi(x) [hi(w) | lo(w)]
        umma_tf32(d, a + a_lo, bw, idesc, 1u);    // lo(x) hi(w)
    } else if (MODE == MODE_X3) {
        umma_tf32(d, a + a_lo, bw, idesc, acc);   // lo(x) hi(w)
        umma_tf32(d, a, bw + b_lo, idesc, 1u);    // hi(x) lo(w)
        umma_tf32(d, a, bw, idesc, 1u);           // hi(x) hi(w)
    } else {
        umma_tf32(d, a, bw, idesc, acc);
    }
}

// A tile's MMAs (one chunk) from a table held in registers: `ra` the A words and
// `rb` the low words of the B descriptors, whose high words (SBO and version) are
// the same for every entry: `bhi`.
template <int NE, int MODE>
__device__ __forceinline__ void issue_chunk_reg(const uint32_t (&ra)[NE], const uint32_t (&rb)[NE],
                                                uint32_t bhi, uint64_t abase, uint32_t dbase,
                                                uint32_t acc_cols, uint32_t idesc,
                                                uint32_t idesc_pair, uint32_t a_lo, uint32_t b_lo) {
#pragma unroll
    for (int e = 0; e < NE; ++e)
        issue_entry<MODE>(ra[e], ((uint64_t)bhi << 32) | rb[e], abase, dbase, acc_cols, idesc,
                          idesc_pair, true, a_lo, b_lo);
}

template <int NE, int UNROLL, int MODE>
__device__ __forceinline__ void issue_chunk(const uint32_t *tab_a, const uint64_t *bt, int n_ent,
                                            uint64_t abase, uint32_t dbase, uint32_t acc_cols,
                                            uint32_t idesc, uint32_t idesc_pair, bool first_chunk,
                                            uint32_t a_lo, uint32_t b_lo) {
    auto one = [&](int e) {
        issue_entry<MODE>(tab_a[e], bt[e], abase, dbase, acc_cols, idesc, idesc_pair, first_chunk,
                          a_lo, b_lo);
    };
    if constexpr (NE > 0) {
#pragma unroll UNROLL
        for (int e = 0; e < NE; ++e) one(e);
    } else if constexpr (MODE != MODE_TF32) {
#pragma unroll 2
        for (int e = 0; e < n_ent; ++e) one(e);
    } else {
#pragma unroll 4
        for (int e = 0; e < n_ent; ++e) one(e);
    }
}
}  // namespace tc1

// MODE != MODE_TF32: 3xTF32 (operands split into tf32 hi + lo).
template <int MODE>
__global__ void __launch_bounds__(tc1::THREADS, 1)
    convt1d_tf32_kernel(const __grid_constant__ CUtensorMap xmap,
                        const __grid_constant__ CUtensorMap ymap, const float *__restrict__ w,
                        const float *__restrict__ bias, float *__restrict__ y, int Cin, int Cout,
                        int K, int S, int L_out, int n_mtiles, long long n_units, int win0, int BW,
                        int tmem_cols, int nacc, int RS, int nbuf, int dgroups, int vec_store,
                        int tma_store, int CKr, int XTS, int nconv,
                        const __grid_constant__ tc1::Taps taps, unsigned int *status) {
    pdl_trigger();
    pdl_wait();
    using namespace tc1;
    constexpr bool split = MODE != tc1::MODE_TF32;
    constexpr bool paired = MODE == tc1::MODE_X3_PAIRED;
    // accumulator columns per class: the paired form keeps hi(w) and lo(w) products in
    // two halves, summed by the epilogue
    const uint32_t acc_cols = (uint32_t)Cout * (paired ? 2u : 1u);
    extern __shared__ __align__(1024) unsigned char smem[];
    // CKr: channels per chunk; XTS: converted-operand stages.  split: operands
    // are split as v = hi + lo (both tf32) and each product is accumulated as
    // lo(x)*hi(w) + hi(x)*lo(w) + hi(x)*hi(w) (3xTF32, fp32-level accuracy);
    // the lo halves sit XT_LO bytes after a stage's hi half and W_LO bytes
    // after the hi weights.
    const int nchunks = Cin / CKr;
    const uint32_t LBO_X = (uint32_t)BW * 16 + 16;   // 16-byte pad: conflict-free transposes
    const uint32_t XT_BYTES = (uint32_t)(CKr / 4) * LBO_X;
    const uint32_t XT_LO = split ? ((XT_BYTES + 127u) & ~127u) : 0u;
    const uint32_t XT_STRIDE = (XT_LO + XT_BYTES + 1023) & ~1023u;
    const uint32_t RAW_BYTES = (uint32_t)CKr * BW * 4;
    const uint32_t RAW_STRIDE = (RAW_BYTES + 1023) & ~1023u;
    unsigned char *xt = smem;
    unsigned char *raw = xt + XTS * XT_STRIDE;
    // weights: [K][Cin/4][Cout][4] (hi; the 3xTF32 lo copy W_LO bytes after it), or,
    // paired, [K][Cin/4][hi, lo][Cout][4]
    float *wt = reinterpret_cast<float *>(raw + RS * RAW_STRIDE);
    const uint32_t W_LO = (split && !paired) ? (uint32_t)K * Cin * Cout * 4u : 0u;
    float *bs = wt + (size_t)K * Cin * Cout * (split ? 2 : 1);
    const int OROW = BM * S + 4;                   // staged output row (one channel)
    const int SLAB = S == 1 ? 32 : 16;             // channels per TMA-stored slab
    // epilogue staging, 1 KB aligned (offset from the shared array so the
    // compiler keeps shared-memory stores): NBUF dense [SLAB][BM*S] slabs for
    // TMA stores, or one [32][OROW] block
    const uint32_t ost_off =
        ((uint32_t)(reinterpret_cast<unsigned char *>(bs + Cout) - smem) + 1023u) & ~1023u;
    float *ost = reinterpret_cast<float *>(smem + ost_off);
    const int ost_floats = tma_store ? nbuf * SLAB * BM * S : dgroups * 32 * OROW;
    uint64_t *bars = reinterpret_cast<uint64_t *>(ost + ost_floats);
    uint64_t *raw_full = bars, *raw_empty = raw_full + RAW_STAGES;
    uint64_t *xt_full = raw_empty + RAW_STAGES, *xt_empty = xt_full + XT_STAGES;
    uint64_t *acc_full = xt_empty + XT_STAGES, *acc_empty = acc_full + MAX_ACC;
    uint64_t *drain = acc_empty + MAX_ACC;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    // MMA descriptor tables: B descriptors per (chunk, entry); per entry the A
    // offset (16-byte units, low 16 bits), class (bits 16..23) and a flag (bit
    // 31) for the first MMA of its class, which overwrites the accumulator
    uint64_t *tab_b = reinterpret_cast<uint64_t *>(tmem_slot + 2);
    uint32_t *tab_a = reinterpret_cast<uint32_t *>(tab_b + MAX_MMA_TAB);
    __shared__ volatile int abort_flag;
    __shared__ volatile int epi_ok[2][4];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // ---- set-up: barriers, tensor memory, tf32 weights, bias
    if (threadIdx.x == 0) {
        for (int s = 0; s < RS; ++s) {
            mbar_init(&raw_full[s], 1);
            mbar_init(&raw_empty[s], CONVERTERS);
        }
        for (int s = 0; s < XTS; ++s) {
            mbar_init(&xt_full[s], CONVERTERS);
            mbar_init(&xt_empty[s], 1);
        }
        for (int b = 0; b < nacc; ++b) {
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_empty[b], EPI_WARPS);
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
            const float v = __ldg(w + ((size_t)ci * Cout + co) * K + k);
            const uint32_t hi = to_tf32(v);
            if (paired) {
                // block (k, cb) holds Cout hi rows, then Cout lo rows
                const int blk = (e >> 2) / Cout;   // k * (Cin / 4) + cb
                const int at = blk * 2 * Cout * 4 + co * 4 + j;
                wtu[at] = hi;
                wtu[at + Cout * 4] = to_tf32(v - __uint_as_float(hi));
            } else {
                wtu[e] = hi;
                if (split) wtu[total + e] = to_tf32(v - __uint_as_float(hi));
            }
        }
        for (int c = threadIdx.x; c < Cout; c += THREADS) bs[c] = bias ? __ldg(bias + c) : 0.f;
    }
    int n_ent = 0;   // MMAs per chunk
    for (int c = 0; c < taps.nclass; ++c) n_ent += taps.ntaps[c] * (CKr / 8);
    if (warp == W_MMA && lane == 0) {
        const uint32_t LBO_W = (uint32_t)Cout * 16 * (paired ? 2u : 1u);
        const uint32_t wt_addr = smem_u32(wt);
        int e = 0;
        for (int c = 0; c < taps.nclass; ++c)
            for (int t = 0; t < taps.ntaps[c]; ++t)
                for (int j = 0; j < CKr / 8; ++j, ++e) {
                    const uint32_t aoff = ((uint32_t)taps.tap_row[c][t] * 16 + 2 * j * LBO_X) >> 4;
                    tab_a[e] = aoff | ((uint32_t)c << 16) | ((t == 0 && j == 0) ? 0x80000000u : 0u);
                    for (int ch = 0; ch < nchunks; ++ch) {
                        const uint32_t cb = (uint32_t)(ch * CKr + 8 * j) / 4;
                        const uint32_t wk =
                            wt_addr + (uint32_t)taps.tap_k[c][t] * (Cin / 4) * LBO_W + cb * LBO_W;
                        tab_b[ch * n_ent + e] = tc1::umma_desc(wk, LBO_W, 128);
                    }
                }
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
            // L2 prefetch runs PREFETCH boxes ahead of the loads, so the smem
            // ring's few stages are refilled from L2 rather than from HBM.
            auto prefetch = [&](uint32_t j) {
                const long long pu = blockIdx.x + (long long)(j / nchunks) * gridDim.x;
                if (pu >= n_units) return;
                const int pn = (int)(pu / n_mtiles);
                const int pmt = (int)(pu - (long long)pn * n_mtiles);
                tma_prefetch_3d(&xmap, pmt * BM + win0, (int)(j % nchunks) * CKr, pn);
            };
            for (uint32_t j = 0; j < (uint32_t)PREFETCH; ++j) prefetch(j);
            uint32_t it = 0;
            bool ok = true;
            for (long long u = blockIdx.x; ok && u < n_units; u += gridDim.x) {
                const int n = (int)(u / n_mtiles);
                const int mt = (int)(u - (long long)n * n_mtiles);
                const int a0 = mt * BM + win0;
                for (int ch = 0; ch < nchunks; ++ch, ++it) {
                    prefetch(it + PREFETCH);
                    const uint32_t s = it % RS;
                    if (it >= (uint32_t)RS && !mbar_wait(&raw_empty[s], ((it / RS) & 1u) ^ 1u)) {
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
            const uint32_t first = it > (uint32_t)RS ? it - RS : 0u;
            for (uint32_t j = first; j < it; ++j)
                if (!mbar_wait(&raw_full[j % RS], (j / RS) & 1u)) break;
        }
    } else if (warp == W_MMA) {
        // ------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idesc = tc::idesc_tf32(BM, Cout);
            const uint32_t idesc_pair = tc::idesc_tf32(BM, 2 * Cout);   // paired form only
            uint64_t a_stage[XT_STAGES];
            for (int st = 0; st < XT_STAGES; ++st)
                a_stage[st] = tc1::umma_desc(smem_u32(xt) + st * XT_STRIDE, LBO_X, 128);
            // lo halves: the same descriptors with the start address moved
            const uint32_t a_lo = XT_LO >> 4, b_lo = W_LO >> 4;
            bool issued = false;
            if (n_ent == 20 && nchunks == 1) {
                // The stride-1 K5 geometry at 32-channel chunks: one chunk of 20 entries
                // per tile.  Every shared-memory access of this thread waits behind the
                // tensor core's operand reads (about 150 cycles, even a wait on a phase
                // that has long completed), so this loop makes few: the table (the same
                // for every tile) sits in registers, the loop condition reads no shared
                // flag, and for tf32 the waits for the next stage and accumulator are
                // asked early with a non-blocking test, answered while this tile's MMAs
                // issue.  Measured per tile (3xTF32, per-role clock stamps on the box):
                // 3948 -> 3608 cycles; 452 -> 398 us (3xTF32) and 318 -> 283 us (tf32)
                // against the table loop below, which the other geometries keep (the
                // strided K4 one ran 3 % slower in this form).  The early test costs the
                // 3xTF32 form more than it saves (406 against 398 us).
                constexpr bool EARLY = MODE == tc1::MODE_TF32;
                uint32_t ra[20], rb[20];
#pragma unroll
                for (int e = 0; e < 20; ++e) {
                    ra[e] = tab_a[e];
                    rb[e] = (uint32_t)tab_b[e];
                }
                const uint32_t bhi = (uint32_t)(tab_b[0] >> 32);
                uint32_t tile = 0, b = 0;
                uint32_t xs_i = 0, xs_ph = 0;   // converted stage and its phase parity
                bool acc_ready = false, xt_ready = false;   // early answers (tf32)
                for (long long u = blockIdx.x; u < n_units; u += gridDim.x, ++tile) {
                    const uint32_t s = xs_i;
                    if ((tile >= (uint32_t)nacc && !acc_ready &&
                         !mbar_wait(&acc_empty[b], ((tile / nacc) & 1u) ^ 1u)) ||
                        (!xt_ready && !mbar_wait(&xt_full[s], xs_ph))) {
                        record_error(status, APS_DEVERR_TIMEOUT);
                        abort_flag = 1;
                        break;
                    }
                    tc1::tc_fence_after();
                    const uint32_t dbase = tmem_base + b * taps.nclass * acc_cols;
                    const uint32_t bn = b + 1 == (uint32_t)nacc ? 0u : b + 1;
                    const uint32_t ns = s + 1 == (uint32_t)XTS ? 0u : s + 1;
                    const uint32_t nph = s + 1 == (uint32_t)XTS ? xs_ph ^ 1u : xs_ph;
                    if (EARLY) {
                        xt_ready = mbar_test(&xt_full[ns], nph);
                        acc_ready = tile + 1 < (uint32_t)nacc ||
                                    mbar_test(&acc_empty[bn], (((tile + 1) / nacc) & 1u) ^ 1u);
                    }
                    const uint64_t abase = s == 0 ? a_stage[0] : (s == 1 ? a_stage[1] : a_stage[2]);
                    tc1::issue_chunk_reg<20, MODE>(ra, rb, bhi, abase, dbase, acc_cols, idesc,
                                                   idesc_pair, a_lo, b_lo);
                    issued = true;
                    tc1::umma_commit(&xt_empty[s]);
                    tc1::umma_commit(&acc_full[b]);
                    xs_i = ns;
                    xs_ph = nph;
                    b = bn;
                }
            } else if (n_ent == 8 && nchunks == 4) {
                // Four chunks per tile (the strided K4 workload in 3xTF32: 16-channel
                // chunks of 8 entries): chunk 0's table in registers, chunk ch's B words
                // chunk 0's plus ch times a fixed step (the weights of the next channels
                // start one step further on): 249 -> 230 us.  The same for the tf32 form's
                // two 16-entry chunks ran slower (167 against 154 us), so that keeps the
                // table loop.
                auto reg_loop = [&](auto ne_c) {
                    constexpr int NE = decltype(ne_c)::value;
                    uint32_t ra[NE], rb[NE];
#pragma unroll
                    for (int e = 0; e < NE; ++e) {
                        ra[e] = tab_a[e];
                        rb[e] = (uint32_t)tab_b[e];
                    }
                    const uint32_t bhi = (uint32_t)(tab_b[0] >> 32);
                    const uint32_t bstep = (uint32_t)tab_b[NE] - rb[0];
                    uint32_t tile = 0;
                    uint32_t xs_i = 0, xs_ph = 0;
                    for (long long u = blockIdx.x; u < n_units; u += gridDim.x, ++tile) {
                        const uint32_t b = tile % (uint32_t)nacc;
                        if (tile >= (uint32_t)nacc &&
                            !mbar_wait(&acc_empty[b], ((tile / nacc) & 1u) ^ 1u)) {
                            record_error(status, APS_DEVERR_TIMEOUT);
                            abort_flag = 1;
                            break;
                        }
                        tc1::tc_fence_after();
                        const uint32_t dbase = tmem_base + b * taps.nclass * acc_cols;
                        bool fail = false;
#pragma unroll 1
                        for (int ch = 0; ch < nchunks; ++ch) {
                            const uint32_t s = xs_i;
                            if (!mbar_wait(&xt_full[s], xs_ph)) {
                                record_error(status, APS_DEVERR_TIMEOUT);
                                abort_flag = 1;
                                fail = true;
                                break;
                            }
                            tc1::tc_fence_after();
                            const uint64_t abase =
                                s == 0 ? a_stage[0] : (s == 1 ? a_stage[1] : a_stage[2]);
                            const uint32_t bdel = (uint32_t)ch * bstep;
#pragma unroll
                            for (int e = 0; e < NE; ++e)
                                tc1::issue_entry<MODE>(ra[e], ((uint64_t)bhi << 32) | (rb[e] + bdel),
                                                       abase, dbase, acc_cols, idesc, idesc_pair,
                                                       ch == 0, a_lo, b_lo);
                            issued = true;
                            tc1::umma_commit(&xt_empty[s]);
                            if (++xs_i == (uint32_t)XTS) {
                                xs_i = 0;
                                xs_ph ^= 1u;
                            }
                        }
                        if (fail) break;
                        tc1::umma_commit(&acc_full[b]);
                    }
                };
                reg_loop(std::integral_constant<int, 8>{});
            } else {
                uint32_t tile = 0;
                uint32_t xs_i = 0, xs_ph = 0;   // converted stage and its phase parity
                for (long long u = blockIdx.x; u < n_units && !abort_flag; u += gridDim.x, ++tile) {
                    const uint32_t b = tile % (uint32_t)nacc;
                    if (tile >= (uint32_t)nacc &&
                        !mbar_wait(&acc_empty[b], ((tile / nacc) & 1u) ^ 1u)) {
                        record_error(status, APS_DEVERR_TIMEOUT);
                        abort_flag = 1;
                        break;
                    }
                    tc1::tc_fence_after();
                    const uint32_t dbase = tmem_base + b * taps.nclass * acc_cols;
                    bool fail = false;
                    for (int ch = 0; ch < nchunks; ++ch) {
                        const uint32_t s = xs_i;
                        if (!mbar_wait(&xt_full[s], xs_ph)) {
                            record_error(status, APS_DEVERR_TIMEOUT);
                            abort_flag = 1;
                            fail = true;
                            break;
                        }
                        tc1::tc_fence_after();
                        const uint64_t abase = s == 0 ? a_stage[0] : (s == 1 ? a_stage[1] : a_stage[2]);
                        const uint64_t *bt = tab_b + ch * n_ent;
                        if (n_ent == 20)
                            tc1::issue_chunk<20, 20, MODE>(tab_a, bt, n_ent, abase, dbase, acc_cols,
                                                           idesc, idesc_pair, ch == 0, a_lo, b_lo);
                        else
                            tc1::issue_chunk<0, 1, MODE>(tab_a, bt, n_ent, abase, dbase, acc_cols,
                                                         idesc, idesc_pair, ch == 0, a_lo, b_lo);
                        issued = true;
                        tc1::umma_commit(&xt_empty[s]);
                        if (++xs_i == (uint32_t)XTS) {
                            xs_i = 0;
                            xs_ph ^= 1u;
                        }
                    }
                    if (fail) break;
                    tc1::umma_commit(&acc_full[b]);
                }
            }
            if (issued) {
                // everything issued has completed before tensor memory is freed
                tc1::umma_commit(drain);
                mbar_wait(drain, 0);
            }
        }
    } else if (warp >= W_EPI0 && warp < W_EPI0 + EPI_WARPS) {
        // ------------------------------------------------------ epilogue
        // Two independent groups of four warps (one warp per tensor-memory lane
        // quadrant each) take alternate slabs of a tile, so two slabs are in
        // flight at once.  Per slab: each class's accumulator columns (+ bias)
        // go to their residue slots of a dense [SLAB][BM*S] staging block, the
        // bias-only residues are filled in, and the block leaves by one TMA
        // store (or, when the output rows are not 16-byte strided or s > 2, by
        // 128-bit coalesced stores from group 0).
        const int g = (warp - W_EPI0) >> 2;    // epilogue group
        const int q = warp & 3;                // tensor-memory lane quadrant
        const int row = q * 32 + lane;
        const int gtid = q * 32 + lane;        // thread index within the group
        const int bar_id = 1 + g;
        const int span = BM * S;               // outputs of one channel in a tile
        const int nslab = tma_store ? Cout / SLAB : Cout / 32;
        const int nbg = nbuf / 2;              // staging slabs per group (1 or 2)
        auto release = [&](uint32_t b) {       // this warp is done reading the accumulator
            tc1::tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[b]);
        };
        uint32_t tile = 0, gs = 0;
        for (long long u = blockIdx.x; u < n_units; u += gridDim.x, ++tile) {
            const uint32_t b = tile % (uint32_t)nacc;
            // The group's warps meet at named barriers below, so they must agree
            // on whether to go on: each posts its wait result, all read all four.
            const bool ok = mbar_wait(&acc_full[b], (tile / nacc) & 1u);
            if (lane == 0) epi_ok[g][q] = ok ? 1 : 0;
            named_bar(bar_id, 128);
            const bool all_ok = epi_ok[g][0] && epi_ok[g][1] && epi_ok[g][2] && epi_ok[g][3];
            named_bar(bar_id, 128);
            if (!all_ok) {
                record_error(status, APS_DEVERR_TIMEOUT);
                abort_flag = 1;
                break;
            }
            tc1::tc_fence_after();
            const int n = (int)(u / n_mtiles);
            const int mt = (int)(u - (long long)n * n_mtiles);
            const long long o0 = (long long)mt * span;
            if (tma_store) {
                for (int i = g; i < nslab; i += 2, ++gs) {
                    const int c0 = i * SLAB;
                    float *st_buf = ost + (g * nbg + gs % nbg) * (SLAB * span);
                    // the store issued from this buffer nbg slabs ago has read it
                    if (gtid == 0) {
                        if (nbg >= 2)
                            bulk_wait_read<1>();
                        else
                            bulk_wait_read<0>();
                    }
                    named_bar(bar_id, 128);
                    for (int c = 0; c < taps.nclass; ++c) {
                        const uint32_t col = tmem_base + ((uint32_t)(q * 32) << 16) +
                                             (b * taps.nclass + c) * acc_cols + c0;
                        float *dst = st_buf + S * row + taps.cls_r[c];
                        const float4 *b4 = reinterpret_cast<const float4 *>(bs + c0);
                        if (SLAB == 32) {
                            uint32_t r[32];
                            tc1::tmem_ld32(col, r);
                            if (paired) {   // + the lo(w) half
                                uint32_t r2[32];
                                tc1::tmem_ld32(col + (uint32_t)Cout, r2);
#pragma unroll
                                for (int j = 0; j < 32; ++j)
                                    r[j] = __float_as_uint(__uint_as_float(r[j]) +
                                                           __uint_as_float(r2[j]));
                            }
#pragma unroll
                            for (int j = 0; j < 32; j += 4) {
                                const float4 bv = b4[j / 4];
                                dst[(j + 0) * span] = __uint_as_float(r[j + 0]) + bv.x;
                                dst[(j + 1) * span] = __uint_as_float(r[j + 1]) + bv.y;
                                dst[(j + 2) * span] = __uint_as_float(r[j + 2]) + bv.z;
                                dst[(j + 3) * span] = __uint_as_float(r[j + 3]) + bv.w;
                            }
                        } else {
                            uint32_t r[16];
                            tc1::tmem_ld16(col, r);
                            if (paired) {   // + the lo(w) half
                                uint32_t r2[16];
                                tc1::tmem_ld16(col + (uint32_t)Cout, r2);
#pragma unroll
                                for (int j = 0; j < 16; ++j)
                                    r[j] = __float_as_uint(__uint_as_float(r[j]) +
                                                           __uint_as_float(r2[j]));
                            }
#pragma unroll
                            for (int j = 0; j < 16; j += 4) {
                                const float4 bv = b4[j / 4];
                                dst[(j + 0) * span] = __uint_as_float(r[j + 0]) + bv.x;
                                dst[(j + 1) * span] = __uint_as_float(r[j + 1]) + bv.y;
                                dst[(j + 2) * span] = __uint_as_float(r[j + 2]) + bv.z;
                                dst[(j + 3) * span] = __uint_as_float(r[j + 3]) + bv.w;
                            }
                        }
                    }
                    for (int e = 0; e < taps.nempty; ++e) {
                        float *dst = st_buf + S * row + taps.empty_r[e];
                        for (int j = 0; j < SLAB; ++j) dst[j * span] = bs[c0 + j];
                    }
                    if (i + 2 >= nslab) release(b);   // last slab of this group
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    named_bar(bar_id, 128);
                    if (gtid == 0) {
                        tma_store_3d(&ymap, st_buf, (int)o0, c0, n);
                        bulk_commit();
                    }
                }
                if (g >= nslab) release(b);           // no slab for this group
                continue;
            }
            // direct stores: group g (of dgroups, 1 or 2 as shared memory allows)
            // stages 32-channel slabs i = g, g+dgroups, ... in its own [32][OROW]
            // block and writes them with 128-bit stores
            float *yn = y + (long long)n * Cout * L_out;
            float *gst = ost + g * 32 * OROW;
            for (int i = g; i < nslab && g < dgroups; i += dgroups) {
                const int c0 = i * 32;
                for (int c = 0; c < taps.nclass; ++c) {
                    uint32_t r[32];
                    const uint32_t col = tmem_base + ((uint32_t)(q * 32) << 16) +
                                         (b * taps.nclass + c) * acc_cols + c0;
                    tc1::tmem_ld32(col, r);
                    if (paired) {   // + the lo(w) half
                        uint32_t r2[32];
                        tc1::tmem_ld32(col + (uint32_t)Cout, r2);
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            r[j] = __float_as_uint(__uint_as_float(r[j]) + __uint_as_float(r2[j]));
                    }
                    float *dst = gst + S * row + taps.cls_r[c];
#pragma unroll
                    for (int j = 0; j < 32; ++j) dst[j * OROW] = __uint_as_float(r[j]) + bs[c0 + j];
                }
                for (int e = 0; e < taps.nempty; ++e) {
                    float *dst = gst + S * row + taps.empty_r[e];
#pragma unroll
                    for (int j = 0; j < 32; ++j) dst[j * OROW] = bs[c0 + j];
                }
                if (i + dgroups >= nslab) release(b);
                named_bar(bar_id, 128);
                if (vec_store) {
                    const int per_row = span / 4;
                    for (int idx = gtid; idx < 32 * per_row; idx += 128) {
                        const int cl = idx / per_row, qv = idx - cl * per_row;
                        const long long o = o0 + 4 * qv;
                        if (o >= L_out) continue;
                        const float4 v = *reinterpret_cast<const float4 *>(gst + cl * OROW + 4 * qv);
                        float *yp = yn + (long long)(c0 + cl) * L_out + o;
                        if (o + 4 <= L_out) {
                            *reinterpret_cast<float4 *>(yp) = v;
                        } else {
                            yp[0] = v.x;
                            if (o + 1 < L_out) yp[1] = v.y;
                            if (o + 2 < L_out) yp[2] = v.z;
                        }
                    }
                } else {
                    for (int idx = gtid; idx < 32 * span; idx += 128) {
                        const int cl = idx / span, t = idx - cl * span;
                        if (o0 + t < L_out) yn[(long long)(c0 + cl) * L_out + o0 + t] = gst[cl * OROW + t];
                    }
                }
                named_bar(bar_id, 128);
            }
            if (g >= nslab || g >= dgroups) release(b);
        }
        // stores issued from shared memory complete before the CTA exits
        if (tma_store && gtid == 0) bulk_wait<0>();
    } else {
        // ------------------------------------------------------ converters
        // converter warp cb owns channels 4cbx..4cbx+3 of every chunk, cbx = cb,
        // cb + ACTIVE, ... (ACTIVE = `nconv`, from the launcher).  The split form
        // writes twice the bytes per channel, and its shared-memory stores then slow
        // the tensor core's operand reads: two busy converters (the rest only arrive)
        // leave the MMA more of the port.
        const int cb = converter_id(warp);
        const int ACTIVE = nconv;
        uint32_t it = 0;
        uint32_t xs_i = 0, xs_ph = 0;   // converted stage and its phase parity
        for (long long u = blockIdx.x; u < n_units && !abort_flag; u += gridDim.x) {
            bool fail = false;
            for (int ch = 0; ch < nchunks; ++ch, ++it) {
                const uint32_t rs = it % RS, xs = xs_i;
                if (!mbar_wait(&raw_full[rs], (it / RS) & 1u) ||
                    (it >= (uint32_t)XTS && !mbar_wait(&xt_empty[xs], xs_ph ^ 1u))) {
                    record_error(status, APS_DEVERR_TIMEOUT);
                    abort_flag = 1;
                    fail = true;
                    break;
                }
                for (int cbx = cb; cb < ACTIVE && cbx < CKr / 4; cbx += ACTIVE) {
                    const float *s0 = reinterpret_cast<const float *>(raw + rs * RAW_STRIDE) +
                                      (size_t)(4 * cbx) * BW;
                    // lane -> positions lane, lane+32, ...: the four channel reads
                    // and the 16-byte row writes of a warp are each contiguous, so
                    // neither has bank conflicts
                    uint4 *d0 = reinterpret_cast<uint4 *>(xt + xs * XT_STRIDE + cbx * LBO_X);
                    if constexpr (split) {
                        // hi: the raw words (the MMA reads their leading tf32 bits,
                        // i.e. truncates); lo = v - trunc_tf32(v), exact in fp32 (the
                        // MMA truncates it in turn).  Two integer/fp operations per
                        // value instead of two tf32 conversions: 268 -> 249 us on the
                        // strided K4 workload, unchanged on the stride-1 K5 one.
                        uint4 *d1 = reinterpret_cast<uint4 *>(reinterpret_cast<unsigned char *>(d0) + XT_LO);
                        auto lo = [](float t) {
                            return __float_as_uint(t - __uint_as_float(__float_as_uint(t) & 0xFFFFE000u));
                        };
#pragma unroll 2
                        for (int pos = lane; pos < BW; pos += 32) {
                            const float v0 = s0[pos], v1 = s0[BW + pos], v2 = s0[2 * BW + pos],
                                        v3 = s0[3 * BW + pos];
                            d0[pos] = make_uint4(__float_as_uint(v0), __float_as_uint(v1),
                                                 __float_as_uint(v2), __float_as_uint(v3));
                            d1[pos] = make_uint4(lo(v0), lo(v1), lo(v2), lo(v3));
                        }
                    } else {
                        // plain tf32: the MMA reads the leading 19 bits of each fp32
                        // word, so the values go in unrounded (truncated to tf32)
#pragma unroll 2
                        for (int pos = lane; pos < BW; pos += 32)
                            d0[pos] = make_uint4(__float_as_uint(s0[pos]), __float_as_uint(s0[BW + pos]),
                                                 __float_as_uint(s0[2 * BW + pos]),
                                                 __float_as_uint(s0[3 * BW + pos]));
                    }
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&raw_empty[rs]);
                    mbar_arrive(&xt_full[xs]);
                }
                if (++xs_i == (uint32_t)XTS) {
                    xs_i = 0;
                    xs_ph ^= 1u;
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
                               float *y, int64_t l_out, bool split, cudaStream_t st) {
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
    for (int r = 0; r < s; ++r) {
        bool has = false;
        for (int c = 0; c < taps.nclass; ++c) has = has || taps.cls_r[c] == r;
        if (!has) taps.empty_r[taps.nempty++] = r;
    }
    // window of a tile at m0: inputs m0 + ph + emin .. m0 + 127 + ph + emax, start
    // rounded down to a multiple of 4 (16-byte TMA coordinate)
    const int lo = ph + emin;
    const int win0 = floordiv_h(lo, 4) * 4;
    const int off = lo - win0;
    const int BW = ((off + BM + (emax - emin)) + 3) & ~3;
    if (BW > 256) return APS_ERR_UNSUPPORTED;
    for (int c = 0; c < taps.nclass; ++c)
        for (int t = 0; t < taps.ntaps[c]; ++t) taps.tap_row[c][t] = ph + ce[c][t] - win0;
    // 3xTF32 pairs the hi and lo weights in one 2*C_out-wide MMA where that width is a
    // valid N (<= 256) and two accumulator sets still fit; otherwise three MMAs
    const bool paired = split && 2 * c_out <= 256 && taps.nclass * 4 * (int)c_out <= 512;
    const int acc_cols = (int)c_out * (paired ? 2 : 1);
    // as many accumulator buffers as fit in the 512 tensor-memory columns (>= 2)
    int nacc = 512 / (taps.nclass * acc_cols);
    if (nacc > MAX_ACC) nacc = MAX_ACC;
    if (nacc < 2) return APS_ERR_UNSUPPORTED;
    int cols = 32;
    while (cols < nacc * taps.nclass * acc_cols) cols *= 2;

    const uint32_t LBO_X = (uint32_t)BW * 16 + 16;
    // split (3xTF32): hi and lo copies of the weights and of each converted stage
    const size_t w_bytes = (size_t)k * Cin * c_out * 4 * (split ? 2 : 1);
    // the output leaves by TMA store when a tile's outputs form a <= 256-wide box
    // and y and its rows are 16-byte aligned; otherwise by the direct stores
    const int tma_store =
        (s <= 2 && l_out % 4 == 0 && reinterpret_cast<uintptr_t>(y) % 16 == 0) ? 1 : 0;
    // the CTA's shared memory, less the 1 KB of static shared memory the kernel declares
    const size_t budget = kMaxSmemPerCta - 1024;
    // Deepest pipeline that fits, trying in order: chunks of 32 channels then
    // (split only) 16; 3 converted stages then 2; then, as before, 4 staging
    // slabs if the raw ring can still hold 2 stages, otherwise 2 (for direct
    // stores: two epilogue groups' staging blocks, else one).
    int CKr = 0, XTS = 0, RS = 0, nbuf = 0, dgroups = 0;
    size_t smem = budget + 1;
    const int ck_try[2] = {Cin < CK ? (int)Cin : CK, (split && Cin >= 16) ? 16 : 0};
    for (int ci = 0; ci < 2 && smem > budget; ++ci) {
        const int ck = ck_try[ci];
        if (ck == 0 || (ci == 1 && ck == ck_try[0]) || Cin % ck != 0) continue;
        int n_ent = 0;   // MMAs per chunk; the descriptor table holds them for every chunk
        for (int c = 0; c < taps.nclass; ++c) n_ent += taps.ntaps[c] * (ck / 8);
        if (n_ent * (int)(Cin / ck) > MAX_MMA_TAB) continue;
        const uint32_t xt_bytes = (uint32_t)(ck / 4) * LBO_X;
        const uint32_t xt_lo = split ? ((xt_bytes + 127u) & ~127u) : 0u;
        const uint32_t XT_STRIDE = (xt_lo + xt_bytes + 1023) & ~1023u;
        const uint32_t RAW_STRIDE = ((uint32_t)ck * BW * 4 + 1023) & ~1023u;
        for (int xts = XT_STAGES; xts >= (split ? 2 : XT_STAGES) && smem > budget; --xts) {
            int rs = RAW_STAGES, nb = tma_store ? NBUF : 0, dg = tma_store ? 0 : 2;
            for (;;) {
                const size_t ost_bytes = tma_store ? (size_t)nb * (s == 1 ? 32 : 16) * BM * s * 4
                                                   : (size_t)dg * 32 * (BM * s + 4) * 4;
                const size_t fixed = xts * XT_STRIDE + w_bytes + (size_t)c_out * 4 + 1024 +
                                     ost_bytes +
                                     (2 * RAW_STAGES + 2 * XT_STAGES + 2 * MAX_ACC + 1) * 8 +
                                     16 + MAX_MMA_TAB * 8 + MAX_MMA_TAB * 4;
                rs = RAW_STAGES;
                while (rs > 2 && fixed + rs * RAW_STRIDE > budget) --rs;
                const size_t need = fixed + rs * RAW_STRIDE;
                if (need <= budget) {
                    CKr = ck, XTS = xts, RS = rs, nbuf = nb, dgroups = dg, smem = need;
                    break;
                }
                if (tma_store && nb == 4) {
                    nb = 2;
                } else if (!tma_store && dg == 2) {
                    dg = 1;
                } else {
                    break;
                }
            }
        }
    }
    if (smem > budget) return APS_ERR_UNSUPPORTED;

    CUtensorMap map;
    const cuuint64_t dims[3] = {(cuuint64_t)L, (cuuint64_t)Cin, (cuuint64_t)N};
    const cuuint64_t strides[2] = {(cuuint64_t)(L * 4), (cuuint64_t)(Cin * L * 4)};
    const cuuint32_t box[3] = {(cuuint32_t)BW, (cuuint32_t)CKr, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    if (!encode_tiled(&map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float *>(x), dims,
                      strides, box, estr))
        return APS_ERR_UNSUPPORTED;

    CUtensorMap ymap;
    if (tma_store) {
        const cuuint64_t ydims[3] = {(cuuint64_t)l_out, (cuuint64_t)c_out, (cuuint64_t)N};
        const cuuint64_t ystr[2] = {(cuuint64_t)(l_out * 4), (cuuint64_t)(c_out * l_out * 4)};
        const cuuint32_t ybox[3] = {(cuuint32_t)(BM * s), (cuuint32_t)(s == 1 ? 32 : 16), 1};
        if (!encode_tiled(&ymap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, y, ydims, ystr, ybox, estr))
            return APS_ERR_UNSUPPORTED;
    } else {
        ymap = map;   // unused
    }
    const auto kern = paired  ? convt1d_tf32_kernel<MODE_X3_PAIRED>
                      : split ? convt1d_tf32_kernel<MODE_X3>
                              : convt1d_tf32_kernel<MODE_TF32>;
    const int per_sm = resident_ctas((const void *)kern, THREADS, (int)smem);
    if (per_sm < 1) return APS_ERR_UNSUPPORTED;
    const int64_t M = ceil_div(l_out, s);
    const int n_mtiles = (int)ceil_div(M, BM);
    const long long n_units = (long long)N * n_mtiles;
    const long long grid = std::min<long long>(n_units, (long long)sm_count());
    const int vec = (l_out % 4 == 0) && (reinterpret_cast<uintptr_t>(y) % 16 == 0);
    const cudaError_t e = launch_pdl(kern, dim3((unsigned)grid), dim3(THREADS), smem, st, map, ymap, w, bias, y, (int)Cin,
               (int)c_out, k, s, (int)l_out, n_mtiles, n_units, win0, BW, cols, nacc, RS, nbuf,
               dgroups, vec, tma_store, CKr, XTS, split ? 2 : CONVERTERS, taps, status_word());
    return launch_status(e);
}

}  // namespace aps
