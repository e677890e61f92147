// avgpool3d.cu -- AvgPool3d kernels.
//
// Operation (Kimi-K2.6__l1_p46): y[n,c,i,j,l] = (1/27) * sum of the 3x3x3 input
// window starting at (2i-1, 2j-1, 2l-1), cells outside the input counting as
// zero (count_include_pad, so the divisor is always 27).  Every input cell is
// read by at most 2x2x2 windows; the page's tiling estimate is 42.8 B of
// traffic per output for a shared-memory halo tile against 108 B for a
// per-output gather.  The kernel below moves each input byte from HBM once
// (plus an L2-resident one-row / one-float4 halo per tile).
//
// Design (GB300):
//  * A tile is 16 output rows x 64 output columns of one (n, c) plane; the CTA
//    walks it through all output depths.  Per output depth i it needs input
//    planes 2i-1, 2i, 2i+1; plane 2i-1 was already summed at step i-1, so each
//    step fetches just planes 2i and 2i+1: one 4-D TMA box of 132 x 33 x 2 x 1
//    cells (columns 2*l0-4 .. 2*l0+127, rows 2*j0-1 .. 2*j0+31).  TMA fills
//    cells outside the tensor with zeros, which is exactly the zero padding,
//    so there is no boundary code.  The column origin is moved 3 cells left of
//    the halo so that it stays 16-byte aligned.
//  * One producer warp issues the boxes into a 2-stage mbarrier ring; sixteen
//    consumer warps each own one output row.  Two CTAs share an SM (registers
//    allow no third), so four boxes, 139 KB, are in flight per SM.  Against
//    8-row tiles with a 4-stage ring the taller tile halves the boxes per
//    output and the re-read row halo (33/32 rows instead of 17/16) and gives
//    each SM 32 consumer warps instead of 24: 7.0 TB/s instead of 6.4.  A lane reads one float4 per
//    input row (128-bit, conflict-free), sums the three rows of its window
//    (H direction), gets the left neighbour column by a warp shuffle and forms
//    two W-direction window sums; the D direction is a running carry in
//    registers (sum of plane 2i+1 carried into step i+1).  The two outputs are
//    stored as one float2 (each warp writes 256 contiguous bytes).
//  * The grid is persistent: one CTA per (SM x resident CTAs), tiles dealt
//    round-robin, so the ring stays full across tile boundaries.
//  * With count_include_pad off (CIP = false) the same sums are divided by
//    the number of window cells inside the input instead (the page's "18 at a
//    face": 27 inside, 18 / 12 / 8 on a face / edge / corner, fewer where the
//    last window of an odd extent also reaches past the high end).  Per dim
//    the count is 3, less one at output 0 and less one where 2i + 1 is past
//    the end; a thread takes the reciprocals of its products once per tile.
#include <atomic>

#include "aps_dev.cuh"
#include "aps_internal.h"

namespace aps {
// aps_debug_stall_next_pool: the wait limit (ns) of the next TMA pool launch, which
// also withholds its first input box; 0 = no stall.
static std::atomic<unsigned long long> g_stall_next_pool{0};

namespace pool {
constexpr int TW = 64;               // output columns per tile (2 per lane)
constexpr int TH = 16;               // output rows per tile (1 per consumer warp)
constexpr int BOX_W = 2 * TW + 4;    // 132 input columns from 2*l0 - 4
constexpr int BOX_H = 2 * TH + 1;    // 33 input rows from 2*j0 - 1
constexpr int BOX_D = 2;             // input planes 2i, 2i + 1
constexpr int STAGE_BYTES = BOX_W * BOX_H * BOX_D * 4;             // 34848
constexpr int STAGE_STRIDE = ((STAGE_BYTES + 127) / 128) * 128;    // 34944
constexpr int STAGES = 2;
constexpr int CONSUMERS = TH;
constexpr int THREADS = (CONSUMERS + 1) * 32;
constexpr int SMEM_BYTES = STAGES * STAGE_STRIDE + 2 * STAGES * 8;
static_assert((BOX_W * 4) % 16 == 0, "TMA box rows must be a multiple of 16 bytes");
}  // namespace pool

// In-range cells of a k3 s2 p1 window at output i along a dim of input length L.
__device__ __forceinline__ int k3s2p1_cells(int i, int L) {
    return 3 - (i == 0 ? 1 : 0) - (2 * i + 1 >= L ? 1 : 0);
}

template <bool CIP>
__global__ void __launch_bounds__(pool::THREADS)
    avgpool3d_k3s2p1_tma_kernel(const __grid_constant__ CUtensorMap xmap, float *__restrict__ y,
                                int D, int H, int W, int Do, int Ho, int Wo, int n_ht, int n_wt,
                                long long n_units, unsigned int *status,
                                unsigned long long wait_ns, int withhold_first_box) {
    using namespace pool;
    extern __shared__ __align__(1024) unsigned char smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + STAGES * STAGE_STRIDE);
    uint64_t *empty = full + STAGES;
    __shared__ volatile int abort_flag;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], CONSUMERS);
        }
        abort_flag = 0;
        mbar_fence_init();
    }
    __syncthreads();

    if (warp == CONSUMERS) {
        // ------------------------------------------------------ producer
        if (lane == 0) {
            tma_prefetch_desc(&xmap);
            uint32_t it = 0;
            bool ok = true;
            for (long long u = blockIdx.x; ok && u < n_units; u += gridDim.x) {
                const int wt = (int)(u % n_wt);
                const long long r = u / n_wt;
                const int ht = (int)(r % n_ht);
                const int nc = (int)(r / n_ht);
                const int c0 = 2 * wt * TW - 4;
                const int c1 = 2 * ht * TH - 1;
                for (int od = 0; od < Do; ++od, ++it) {
                    const uint32_t slot = it % STAGES;
                    if (it >= (uint32_t)STAGES &&
                        !mbar_wait_for(&empty[slot], ((it / STAGES) & 1u) ^ 1u, wait_ns)) {
                        record_error(status, APS_DEVERR_TIMEOUT);
                        abort_flag = 1;
                        ok = false;
                        break;
                    }
                    if (abort_flag) { ok = false; break; }
                    mbar_arrive_expect_tx(&full[slot], STAGE_BYTES);
                    // the test hook's withheld box: its barrier expects bytes that never come
                    if (withhold_first_box && blockIdx.x == 0 && it == 0) continue;
                    tma_load_4d(smem + slot * STAGE_STRIDE, &xmap, &full[slot], c0, c1, 2 * od,
                                nc);
                }
            }
            if (!ok) {
                // Let every box still in flight land before the CTA exits (a box
                // whose wait runs out does not end the waits for the others).
                const uint32_t first = it > (uint32_t)STAGES ? it - STAGES : 0u;
                for (uint32_t j = first; j < it; ++j)
                    mbar_wait_for(&full[j % STAGES], (j / STAGES) & 1u, wait_ns);
            }
        }
        return;
    }

    // ---------------------------------------------------------- consumers
    const float inv27 = 1.0f / 27.0f;
    const long long plane_out = (long long)Ho * Wo;
    uint32_t it = 0;
    for (long long u = blockIdx.x; u < n_units; u += gridDim.x) {
        const int wt = (int)(u % n_wt);
        const long long r = u / n_wt;
        const int ht = (int)(r % n_ht);
        const long long nc = r / n_ht;
        const int oh = ht * TH + warp;
        const int ow = wt * TW + 2 * lane;
        const bool active = oh < Ho && ow < Wo;
        float *yp = y + ((nc * Do) * Ho + oh) * (long long)Wo + ow;
        float carry0 = 0.f, carry1 = 0.f;   // window sums of input plane 2i-1
        // CIP off: 1 / (cells in range) for the two columns, by the D count 1..3
        float rdiv0[3], rdiv1[3];
        if (!CIP) {
            const int ch = k3s2p1_cells(oh, H);
            const int c0 = ch * k3s2p1_cells(ow, W), c1 = ch * k3s2p1_cells(ow + 1, W);
#pragma unroll
            for (int cd = 1; cd <= 3; ++cd) {
                rdiv0[cd - 1] = 1.0f / (float)(cd * c0);
                rdiv1[cd - 1] = 1.0f / (float)(cd * c1);
            }
        }
        for (int od = 0; od < Do; ++od, ++it) {
            const uint32_t slot = it % STAGES;
            if (!mbar_wait_for(&full[slot], (it / STAGES) & 1u, wait_ns)) {
                record_error(status, APS_DEVERR_TIMEOUT);
                abort_flag = 1;
                return;
            }
            const float *buf = reinterpret_cast<const float *>(smem + slot * STAGE_STRIDE);
            float s0[2], s1[2];
#pragma unroll
            for (int pl = 0; pl < 2; ++pl) {
                const float *r0 = buf + (pl * BOX_H + 2 * warp) * BOX_W;
                const float4 a = *reinterpret_cast<const float4 *>(r0 + 4 + 4 * lane);
                const float4 b = *reinterpret_cast<const float4 *>(r0 + BOX_W + 4 + 4 * lane);
                const float4 c = *reinterpret_cast<const float4 *>(r0 + 2 * BOX_W + 4 + 4 * lane);
                // column sums over the three input rows of this output row
                const float hx = a.x + b.x + c.x, hy = a.y + b.y + c.y;
                const float hz = a.z + b.z + c.z, hw = a.w + b.w + c.w;
                float hl = __shfl_up_sync(0xffffffffu, hw, 1);   // column 4*lane - 1
                if (lane == 0) hl = r0[3] + r0[BOX_W + 3] + r0[2 * BOX_W + 3];
                s0[pl] = hl + hx + hy;   // output column 2*lane
                s1[pl] = hy + hz + hw;   // output column 2*lane + 1
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);
            float r0 = inv27, r1 = inv27;
            if (!CIP) {
                const int cd = k3s2p1_cells(od, D);
                r0 = cd == 3 ? rdiv0[2] : (cd == 2 ? rdiv0[1] : rdiv0[0]);
                r1 = cd == 3 ? rdiv1[2] : (cd == 2 ? rdiv1[1] : rdiv1[0]);
            }
            const float o0 = (carry0 + s0[0] + s0[1]) * r0;
            const float o1 = (carry1 + s1[0] + s1[1]) * r1;
            carry0 = s0[1];
            carry1 = s1[1];
            if (active) *reinterpret_cast<float2 *>(yp + od * plane_out) = make_float2(o0, o1);
        }
    }
}

aps_status launch_avgpool3d_k3s2p1_tma(const float *x, const int64_t in[5], float *y,
                                       const int64_t out[5], int count_include_pad,
                                       cudaStream_t st) {
    using namespace pool;
    const int64_t N = in[0], C = in[1], D = in[2], H = in[3], W = in[4];
    const int64_t NC = N * C;
    // TMA coordinates are 32-bit; strides must stay below 2^40 bytes.
    if (NC >= ((int64_t)1 << 31) || D >= ((int64_t)1 << 30) || H >= ((int64_t)1 << 30) ||
        W >= ((int64_t)1 << 30) || D * H * W * 4 >= ((int64_t)1 << 40))
        return APS_ERR_UNSUPPORTED;
    CUtensorMap map;
    const cuuint64_t dims[4] = {(cuuint64_t)W, (cuuint64_t)H, (cuuint64_t)D, (cuuint64_t)NC};
    const cuuint64_t strides[3] = {(cuuint64_t)(W * 4), (cuuint64_t)(H * W * 4),
                                   (cuuint64_t)(D * H * W * 4)};
    const cuuint32_t box[4] = {BOX_W, BOX_H, BOX_D, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    if (!encode_tiled(&map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<float *>(x), dims,
                      strides, box, estr))
        return APS_ERR_UNSUPPORTED;

    const int Do = (int)out[2], Ho = (int)out[3], Wo = (int)out[4];
    const int n_ht = (int)ceil_div(Ho, TH), n_wt = (int)ceil_div(Wo, TW);
    const long long n_units = (long long)NC * n_ht * n_wt;

    const auto kern = count_include_pad ? avgpool3d_k3s2p1_tma_kernel<true>
                                        : avgpool3d_k3s2p1_tma_kernel<false>;
    const int per_sm = resident_ctas((const void *)kern, THREADS, SMEM_BYTES);
    if (per_sm < 1) return APS_ERR_CUDA;
    const long long grid = std::min<long long>(n_units, (long long)sm_count() * per_sm);
    // the test hook (aps_debug_stall_next_pool) applies to one launch
    const unsigned long long stall = g_stall_next_pool.exchange(0);
    const cudaError_t e = launch_plain(
        kern, dim3((unsigned)grid), dim3(THREADS), (size_t)SMEM_BYTES, st, map, y, (int)D, (int)H,
        (int)W, Do, Ho, Wo, n_ht, n_wt, n_units, status_word(),
        (unsigned long long)(stall ? stall : kWaitLimitNs), stall ? 1 : 0);
    return launch_status(e);
}

// ------------------------------------------------------------ direct kernel
// Any window, stride and padding; count_include_pad on or off; floor or ceil
// mode (the output shape fixes which).  One thread per output, grid-stride.
__global__ void avgpool3d_direct_kernel(const float *__restrict__ x, float *__restrict__ y,
                                        long long total, int D, int H, int W, int Do, int Ho,
                                        int Wo, int kd, int kh, int kw, int sd, int sh, int sw,
                                        int pd, int ph, int pw, int count_include_pad) {
    const long long in_plane = (long long)D * H * W;
    for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        const int ow = (int)(idx % Wo);
        long long t = idx / Wo;
        const int oh = (int)(t % Ho);
        t /= Ho;
        const int od = (int)(t % Do);
        const long long nc = t / Do;
        int d0 = od * sd - pd, h0 = oh * sh - ph, w0 = ow * sw - pw;
        int d1 = min(d0 + kd, D + pd), h1 = min(h0 + kh, H + ph), w1 = min(w0 + kw, W + pw);
        const long long padded = (long long)(d1 - d0) * (h1 - h0) * (w1 - w0);
        d0 = max(d0, 0); h0 = max(h0, 0); w0 = max(w0, 0);
        d1 = min(d1, D); h1 = min(h1, H); w1 = min(w1, W);
        const float *xp = x + nc * in_plane;
        float sum = 0.f;
        for (int a = d0; a < d1; ++a)
            for (int b = h0; b < h1; ++b) {
                const float *row = xp + ((long long)a * H + b) * W;
                for (int c = w0; c < w1; ++c) sum += __ldg(row + c);
            }
        const long long inside = (long long)(d1 - d0) * (h1 - h0) * (w1 - w0);
        const long long div = count_include_pad ? padded : inside;
        y[idx] = div > 0 ? sum / (float)div : 0.f;
    }
}

// Small windows known at compile time (2x2x2 and 3x3x3, any stride and
// padding, count_include_pad on or off, floor or ceil mode): the same
// definition as above with the window unrolled, so that all its loads are in
// flight at once, and 32-bit index arithmetic (the launcher checks that every
// index fits).  One thread per output, consecutive threads on consecutive
// output columns.
template <int K>
__global__ void __launch_bounds__(256)
    avgpool3d_win_kernel(const float *__restrict__ x, float *__restrict__ y, unsigned total,
                         int D, int H, int W, int Do, int Ho, int Wo, int sd, int sh, int sw,
                         int pd, int ph, int pw, int count_include_pad) {
    const unsigned in_plane = (unsigned)D * H * W;
    for (unsigned idx = blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += gridDim.x * blockDim.x) {
        const int ow = (int)(idx % (unsigned)Wo);
        unsigned t = idx / (unsigned)Wo;
        const int oh = (int)(t % (unsigned)Ho);
        t /= (unsigned)Ho;
        const int od = (int)(t % (unsigned)Do);
        const unsigned nc = t / (unsigned)Do;
        const int d0 = od * sd - pd, h0 = oh * sh - ph, w0 = ow * sw - pw;
        const float *xp = x + (size_t)nc * in_plane;
        float sum = 0.f;
#pragma unroll
        for (int a = 0; a < K; ++a)
#pragma unroll
            for (int b = 0; b < K; ++b)
#pragma unroll
                for (int c = 0; c < K; ++c) {
                    const int id = d0 + a, ih = h0 + b, iw = w0 + c;
                    const bool in = (unsigned)id < (unsigned)D && (unsigned)ih < (unsigned)H &&
                                    (unsigned)iw < (unsigned)W;
                    sum += in ? __ldg(xp + ((unsigned)id * H + ih) * W + iw) : 0.f;
                }
        int div;
        if (count_include_pad) {
            // the window clipped at the end of the right padding (ceil mode)
            div = (min(d0 + K, D + pd) - d0) * (min(h0 + K, H + ph) - h0) *
                  (min(w0 + K, W + pw) - w0);
        } else {
            div = (min(d0 + K, D) - max(d0, 0)) * (min(h0 + K, H) - max(h0, 0)) *
                  (min(w0 + K, W) - max(w0, 0));
        }
        y[idx] = div > 0 ? sum / (float)div : 0.f;
    }
}

// k2 s2 p0 with whole windows (floor mode) and 16-byte rows: a thread takes two
// adjacent outputs, i.e. one 16-byte run of each of the window's four input rows
// (4 x LDG.128; a warp reads 512 contiguous bytes of each row), sums each window
// in the (d, h, w) order of the kernel above and stores the pair with one 8-byte
// store.  64-bit plane offsets; the pair index fits 32 bits.
__global__ void __launch_bounds__(256)
    avgpool3d_k2s2_vec_kernel(const float *__restrict__ x, float *__restrict__ y,
                              unsigned pairs, int D, int H, int W, int Do, int Ho, int Wo) {
    const unsigned half = (unsigned)Wo >> 1;   // output pairs per row
    const size_t hw = (size_t)H * W;
    for (unsigned idx = blockIdx.x * blockDim.x + threadIdx.x; idx < pairs;
         idx += gridDim.x * blockDim.x) {
        const unsigned pw = idx % half;
        unsigned t = idx / half;
        const unsigned oh = t % (unsigned)Ho;
        t /= (unsigned)Ho;
        const unsigned od = t % (unsigned)Do;
        const unsigned nc = t / (unsigned)Do;
        const float *p0 = x + ((size_t)nc * D + 2 * od) * hw + (size_t)(2 * oh) * W + 4 * pw;
        const float4 a = __ldg(reinterpret_cast<const float4 *>(p0));
        const float4 b = __ldg(reinterpret_cast<const float4 *>(p0 + W));
        const float4 c = __ldg(reinterpret_cast<const float4 *>(p0 + hw));
        const float4 e = __ldg(reinterpret_cast<const float4 *>(p0 + hw + W));
        float s0 = 0.f, s1 = 0.f;
        s0 += a.x; s0 += a.y; s0 += b.x; s0 += b.y; s0 += c.x; s0 += c.y; s0 += e.x; s0 += e.y;
        s1 += a.z; s1 += a.w; s1 += b.z; s1 += b.w; s1 += c.z; s1 += c.w; s1 += e.z; s1 += e.w;
        float2 *yp = reinterpret_cast<float2 *>(
            y + (((size_t)nc * Do + od) * Ho + oh) * (size_t)Wo + 2 * pw);
        *yp = make_float2(s0 / 8.f, s1 / 8.f);
    }
}

aps_status launch_avgpool3d_direct(const float *x, const int64_t in[5], const int k[3],
                                   const int s[3], const int p[3], int count_include_pad,
                                   float *y, const int64_t out[5], cudaStream_t st) {
    if (in[2] >= (1 << 30) || in[3] >= (1 << 30) || in[4] >= (1 << 30) ||
        out[2] * out[3] * out[4] >= ((int64_t)1 << 31))
        return APS_ERR_UNSUPPORTED;
    const long long total = out[0] * out[1] * out[2] * out[3] * out[4];
    const int threads = 256;
    const long long blocks =
        std::min<long long>(ceil_div(total, threads), (long long)sm_count() * 16);
    const bool cube = k[0] == k[1] && k[1] == k[2] && (k[0] == 2 || k[0] == 3);
    // k2 s2 p0, every window whole, 16-byte input rows and 8-byte output pairs
    if (cube && k[0] == 2 && s[0] == 2 && s[1] == 2 && s[2] == 2 && p[0] == 0 && p[1] == 0 &&
        p[2] == 0 && out[2] == in[2] / 2 && out[3] == in[3] / 2 && out[4] == in[4] / 2 &&
        in[4] % 4 == 0 && reinterpret_cast<uintptr_t>(x) % 16 == 0 &&
        reinterpret_cast<uintptr_t>(y) % 8 == 0 && total / 2 < ((int64_t)1 << 31)) {
        const long long pairs = total / 2;
        const int sms = sm_count();
        const long long blocks2 =
            std::max<long long>(1, std::min<long long>(ceil_div(pairs, threads), (long long)sms * 8));
        const cudaError_t e = launch_plain(
            avgpool3d_k2s2_vec_kernel, dim3((unsigned)blocks2), dim3(threads), 0, st, x, y,
            (unsigned)pairs, (int)in[2], (int)in[3], (int)in[4], (int)out[2], (int)out[3],
            (int)out[4]);
        return launch_status(e);
    }
    // 32-bit output index (with headroom for the grid stride) and plane offsets
    if (cube && total <= ((int64_t)1 << 31) && in[2] * in[3] * in[4] < ((int64_t)1 << 31)) {
        const auto kern = k[0] == 2 ? avgpool3d_win_kernel<2> : avgpool3d_win_kernel<3>;
        const cudaError_t e = launch_plain(
            kern, dim3((unsigned)blocks), dim3(threads), 0, st, x, y, (unsigned)total, (int)in[2],
            (int)in[3], (int)in[4], (int)out[2], (int)out[3], (int)out[4], s[0], s[1], s[2], p[0],
            p[1], p[2], count_include_pad);
        return launch_status(e);
    }
    const cudaError_t e = launch_plain(
        avgpool3d_direct_kernel, dim3((unsigned)blocks), dim3(threads), 0, st, x, y, total,
        (int)in[2], (int)in[3], (int)in[4], (int)out[2], (int)out[3], (int)out[4], k[0], k[1],
        k[2], s[0], s[1], s[2], p[0], p[1], p[2], count_include_pad);
    return launch_status(e);
}

}  // namespace aps

extern "C" void aps_debug_stall_next_pool(unsigned long long wait_limit_ns) {
    aps::g_stall_next_pool.store(wait_limit_ns);
}
