// aps_api.cu -- the C ABI declared in include/aps.h: argument validation,
// output shapes, kernel selection and the per-device status word.  Every
// accepted request runs on the GPU; nothing here computes on the host.
#include <atomic>
#include <mutex>

#include "aps_internal.h"

namespace aps {

// ------------------------------------------------------------ status word
static __device__ unsigned int g_status_word;
// aps_device_status's copy of the word, taken and (optionally) cleared in one
// atomic step on the GPU, so that a bit set meanwhile by a kernel on another
// stream is either in this read or left for the next one.
static __device__ unsigned int g_status_snapshot;

__global__ void status_exchange_kernel(int clear) {
    g_status_snapshot = clear ? atomicExch(&g_status_word, 0u) : atomicOr(&g_status_word, 0u);
}

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_mutex;
unsigned int *g_status_ptr[kMaxDevices];
int g_sms[kMaxDevices];

int current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
    return dev;
}
}  // namespace

unsigned int *status_word() {
    const int dev = current_device();
    if (dev < 0) return nullptr;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_status_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
        g_status_ptr[dev] = static_cast<unsigned int *>(p);
    }
    return g_status_ptr[dev];
}

int sm_count() {
    const int dev = current_device();
    if (dev < 0) return 1;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_sms[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            n <= 0)
            n = 1;
        g_sms[dev] = n;
    }
    return g_sms[dev];
}

namespace {
struct OccEntry {
    const void *func;
    int dev, threads, smem, n;
};
struct SmemLimit {
    const void *func;
    int dev, bytes;
};
constexpr int kOccEntries = 256;
OccEntry g_occ[kOccEntries];
int g_occ_used = 0;
SmemLimit g_limit[kOccEntries];
int g_limit_used = 0;

// Raises (never lowers) a kernel's dynamic shared-memory limit on `dev`; the
// limit is per kernel and device, and a call needing less must not undo it.
bool raise_smem_limit(const void *func, int dev, int smem) {
    int i = 0;
    for (; i < g_limit_used; ++i)
        if (g_limit[i].func == func && g_limit[i].dev == dev) break;
    if (i < g_limit_used && g_limit[i].bytes >= smem) return true;
    if (cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
        cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    if (i < g_limit_used) {
        g_limit[i].bytes = smem;
    } else if (g_limit_used < kOccEntries) {
        g_limit[g_limit_used++] = SmemLimit{func, dev, smem};
    }
    return true;
}
}  // namespace

int resident_ctas(const void *func, int threads, int smem) {
    const int dev = current_device();
    if (dev < 0) return 0;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (smem > 48 * 1024 && !raise_smem_limit(func, dev, smem)) return 0;
    for (int i = 0; i < g_occ_used; ++i) {
        const OccEntry &e = g_occ[i];
        if (e.func == func && e.dev == dev && e.threads == threads && e.smem == smem) return e.n;
    }
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, func, threads, smem) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    if (g_occ_used < kOccEntries) g_occ[g_occ_used++] = OccEntry{func, dev, threads, smem, n};
    return n;
}

namespace {
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;
}  // namespace

bool encode_tiled(CUtensorMap *map, CUtensorMapDataType type, uint32_t rank, void *base,
                  const cuuint64_t *dims, const cuuint64_t *strides_bytes,
                  const cuuint32_t *box, const cuuint32_t *elem_strides) {
    std::call_once(g_encode_once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    if (!g_encode) return false;
    return g_encode(map, type, rank, base, dims, strides_bytes, box, elem_strides,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Launches still to report as rejected (aps_debug_fail_launches).
static std::atomic<int> g_fail_launches{0};
// Set: dispatch passes over the tensor-core kernels (aps_debug_skip_tensor_cores).
static std::atomic<int> g_skip_tc{0};
static bool tensor_cores_on() { return g_skip_tc.load(std::memory_order_relaxed) == 0; }

aps_status launch_status(cudaError_t launch_result) {
    if (launch_result != cudaSuccess) {
        cudaGetLastError();   // the launch's own error; the caller sees it as our status
        return APS_ERR_LAUNCH;
    }
    if (g_fail_launches.load(std::memory_order_relaxed) > 0 &&
        g_fail_launches.fetch_sub(1, std::memory_order_relaxed) > 0)
        return APS_ERR_LAUNCH;
    return APS_OK;
}

}  // namespace aps

using namespace aps;

namespace {

int64_t convt_len(int64_t L, int k, int s, int p, int d, int op) {
    return (L - 1) * s - 2 * (int64_t)p + (int64_t)d * (k - 1) + op + 1;
}

// Pool output length; 0 when the window does not fit.
int64_t pool_len(int64_t L, int k, int s, int p, int ceil_mode) {
    const int64_t span = L + 2 * (int64_t)p - k;
    if (span < 0) return 0;
    if (!ceil_mode) return span / s + 1;
    int64_t n = (span + s - 1) / s + 1;
    if ((n - 1) * s >= L + p) --n;
    return n;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Sizes past this bound would overflow 64-bit index arithmetic somewhere.
constexpr int64_t kMaxElems = (int64_t)1 << 46;

bool dims_ok(const int64_t *d, int n) {
    int64_t prod = 1;
    for (int i = 0; i < n; ++i) {
        if (d[i] < 0 || d[i] > kMaxElems) return false;
        if (d[i] && prod > kMaxElems / d[i]) return false;
        prod *= d[i] ? d[i] : 1;
    }
    return true;
}

// Extents the general kernels address with 32-bit positions: every channel
// count and every spatial size of input and output below 2^30 (and, for the
// fused op, each pre-pool size pool_k * out).  Larger requests are
// APS_ERR_UNSUPPORTED, decided here on the host before any CUDA call.
constexpr int64_t kMaxExtent = (int64_t)1 << 30;

bool extents_ok(const int64_t *in, const int64_t *out, int n, int64_t pool_k = 1) {
    if (in[1] >= kMaxExtent || out[1] >= kMaxExtent) return false;
    for (int i = 2; i < n; ++i)
        if (in[i] >= kMaxExtent || out[i] >= kMaxExtent || out[i] * pool_k >= kMaxExtent)
            return false;
    return true;
}

int64_t numel(const int64_t *d, int n) {
    int64_t p = 1;
    for (int i = 0; i < n; ++i) p *= d[i];
    return p;
}

aps_status conv_params_ok(const int k[3], const int s[3], const int p[3], const int op[3],
                          const int d[3], int nd) {
    for (int i = 0; i < nd; ++i) {
        if (k[i] < 1 || s[i] < 1 || d[i] < 1 || p[i] < 0 || op[i] < 0) return APS_ERR_SHAPE;
        if (op[i] >= (s[i] > d[i] ? s[i] : d[i])) return APS_ERR_SHAPE;
        if (k[i] > 4096 || s[i] > 4096 || d[i] > 4096 || p[i] > (1 << 20)) return APS_ERR_SHAPE;
    }
    return APS_OK;
}

}  // namespace

extern "C" {

int aps_abi_version(void) { return 1; }

const char *aps_status_string(int status) {
    switch (status) {
        case APS_OK: return "APS_OK";
        case APS_ERR_NULL: return "APS_ERR_NULL: a required pointer or shape array is NULL";
        case APS_ERR_SHAPE: return "APS_ERR_SHAPE: a dimension or parameter is out of range";
        case APS_ERR_UNSUPPORTED: return "APS_ERR_UNSUPPORTED: no kernel implements this request";
        case APS_ERR_ALIGN: return "APS_ERR_ALIGN: a tensor pointer is not 4-byte aligned";
        case APS_ERR_LAUNCH: return "APS_ERR_LAUNCH: the CUDA runtime rejected the launch";
        case APS_ERR_CUDA: return "APS_ERR_CUDA: a CUDA runtime call failed";
        default: return "unknown aps_status";
    }
}

// ---------------------------------------------------------------- avgpool3d
aps_status aps_avgpool3d_out_shape(const int64_t in[5], const int k[3], const int s[3],
                                   const int p[3], int ceil_mode, int64_t out[5]) {
    if (!in || !k || !s || !p || !out) return APS_ERR_NULL;
    if (!dims_ok(in, 5)) return APS_ERR_SHAPE;
    for (int i = 0; i < 3; ++i) {
        if (k[i] < 1 || s[i] < 1 || p[i] < 0 || 2 * (int64_t)p[i] > k[i] || k[i] > 4096 ||
            s[i] > 4096)
            return APS_ERR_SHAPE;
    }
    int64_t o[5] = {in[0], in[1], 0, 0, 0};
    for (int i = 0; i < 3; ++i) {
        o[2 + i] = pool_len(in[2 + i], k[i], s[i], p[i], ceil_mode);
        if (o[2 + i] <= 0) return APS_ERR_SHAPE;
    }
    for (int i = 0; i < 5; ++i) out[i] = o[i];
    return APS_OK;
}

// A data pointer may be NULL exactly when its array has no elements (nothing
// is read from or written to it).
static bool present(const void *ptr, int64_t elems) { return elems == 0 || ptr != nullptr; }

aps_status aps_avgpool3d(const float *x, const int64_t in[5], const int k[3], const int s[3],
                         const int p[3], int count_include_pad, int ceil_mode, float *y,
                         aps_stream_t stream) {
    int64_t out[5];
    aps_status st = aps_avgpool3d_out_shape(in, k, s, p, ceil_mode, out);
    if (st != APS_OK) return st;
    if (!present(x, numel(in, 5)) || !present(y, numel(out, 5))) return APS_ERR_NULL;
    if (!aligned(x, 4) || !aligned(y, 4)) return APS_ERR_ALIGN;
    if (numel(out, 5) == 0) return APS_OK;
    // the general kernel also numbers an output plane's cells in 32 bits
    if (!extents_ok(in, out, 5) || out[2] * out[3] * out[4] >= ((int64_t)1 << 31))
        return APS_ERR_UNSUPPORTED;
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    const bool k3s2p1 = k[0] == 3 && k[1] == 3 && k[2] == 3 && s[0] == 2 && s[1] == 2 &&
                        s[2] == 2 && p[0] == 1 && p[1] == 1 && p[2] == 1;
    if (k3s2p1 && !ceil_mode && in[4] % 4 == 0 && aligned(x, 16) && aligned(y, 8)) {
        st = launch_avgpool3d_k3s2p1_tma(x, in, y, out, count_include_pad ? 1 : 0, cs);
        if (st != APS_ERR_UNSUPPORTED) return st;
    }
    return launch_avgpool3d_direct(x, in, k, s, p, count_include_pad ? 1 : 0, y, out, cs);
}

// ----------------------------------------------------- ct3d_scale_pool_bias
aps_status aps_ct3d_scale_pool_bias_out_shape(const int64_t in[5], int64_t c_out,
                                              const int k[3], const int s[3], const int p[3],
                                              const int op[3], const int d[3], int pool_k,
                                              int64_t out[5]) {
    if (!in || !k || !s || !p || !op || !d || !out) return APS_ERR_NULL;
    if (!dims_ok(in, 5) || c_out < 1 || c_out > kMaxElems || pool_k < 1 || pool_k > 4096)
        return APS_ERR_SHAPE;
    aps_status st = conv_params_ok(k, s, p, op, d, 3);
    if (st != APS_OK) return st;
    int64_t o[5] = {in[0], c_out, 0, 0, 0};
    for (int i = 0; i < 3; ++i) {
        if (in[2 + i] < 1) return APS_ERR_SHAPE;
        const int64_t t = convt_len(in[2 + i], k[i], s[i], p[i], d[i], op[i]);
        if (t <= 0) return APS_ERR_SHAPE;
        o[2 + i] = pool_len(t, pool_k, pool_k, 0, 0);
        if (o[2 + i] <= 0) return APS_ERR_SHAPE;
    }
    if (!dims_ok(o, 5)) return APS_ERR_SHAPE;
    for (int i = 0; i < 5; ++i) out[i] = o[i];
    return APS_OK;
}

aps_status aps_ct3d_scale_pool_bias(const float *x, const int64_t in[5], const float *w,
                                    const float *conv_bias, const float *bias, int64_t c_out,
                                    const int k[3], const int s[3], const int p[3],
                                    const int op[3], const int d[3], int pool_k, float scale1,
                                    float scale2, float *y, aps_stream_t stream) {
    int64_t out[5];
    aps_status st = aps_ct3d_scale_pool_bias_out_shape(in, c_out, k, s, p, op, d, pool_k, out);
    if (st != APS_OK) return st;
    if (!present(x, numel(in, 5)) || !present(w, in[1]) || !present(y, numel(out, 5)) ||
        !present(bias, numel(out, 5)))
        return APS_ERR_NULL;
    if (!aligned(x, 4) || !aligned(w, 4) || !aligned(bias, 4) || !aligned(y, 4) ||
        (conv_bias && !aligned(conv_bias, 4)))
        return APS_ERR_ALIGN;
    if (numel(out, 5) == 0) return APS_OK;  // C_in == 0 alone still has bias-only outputs
    if (!extents_ok(in, out, 5, pool_k)) return APS_ERR_UNSUPPORTED;
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    bool fast = pool_k == 2 && c_out == 16 && in[1] >= 1 && in[1] <= 8;
    for (int i = 0; i < 3; ++i)
        fast = fast && k[i] == 3 && s[i] == 2 && p[i] == 1 && op[i] <= 1 && d[i] == 1;
    if (fast) {
        // tensor cores (16-byte input rows), else the FP32-pipe kernel
        st = tensor_cores_on()
            ? launch_ct3d_pool2_tc(x, in, w, conv_bias, bias, scale1, scale2, y, out, cs)
            : APS_ERR_UNSUPPORTED;
        if (st != APS_ERR_UNSUPPORTED) return st;
        st = launch_ct3d_pool2_fast(x, in, w, conv_bias, bias, scale1, scale2, y, out, cs);
        if (st != APS_ERR_UNSUPPORTED) return st;
    }
    // any other geometry: collapsed per-phase weights, else one thread per output
    st = launch_ct3d_pool_gen(x, in, w, conv_bias, bias, c_out, k, s, p, d, pool_k, scale1,
                              scale2, y, out, cs);
    if (st != APS_ERR_UNSUPPORTED) return st;
    return launch_ct3d_pool_direct(x, in, w, conv_bias, bias, c_out, k, s, p, d, pool_k,
                                   scale1, scale2, y, out, cs);
}

// -------------------------------------------------------- convtranspose3d
aps_status aps_convtranspose3d_out_shape(const int64_t in[5], int64_t c_out, const int k[3],
                                         const int s[3], const int p[3], const int d[3],
                                         const int op[3], int64_t out[5]) {
    if (!in || !k || !s || !p || !d || !op || !out) return APS_ERR_NULL;
    if (!dims_ok(in, 5) || c_out < 1 || c_out > kMaxElems) return APS_ERR_SHAPE;
    aps_status st = conv_params_ok(k, s, p, op, d, 3);
    if (st != APS_OK) return st;
    int64_t o[5] = {in[0], c_out, 0, 0, 0};
    for (int i = 0; i < 3; ++i) {
        if (in[2 + i] < 1) return APS_ERR_SHAPE;
        o[2 + i] = convt_len(in[2 + i], k[i], s[i], p[i], d[i], op[i]);
        if (o[2 + i] <= 0) return APS_ERR_SHAPE;
    }
    if (!dims_ok(o, 5)) return APS_ERR_SHAPE;
    for (int i = 0; i < 5; ++i) out[i] = o[i];
    return APS_OK;
}

aps_status aps_convtranspose3d(const float *x, const int64_t in[5], const float *w,
                               const float *bias, int64_t c_out, const int k[3],
                               const int s[3], const int p[3], const int d[3], const int op[3],
                               float *y, aps_stream_t stream) {
    int64_t out[5];
    aps_status st = aps_convtranspose3d_out_shape(in, c_out, k, s, p, d, op, out);
    if (st != APS_OK) return st;
    if (!present(x, numel(in, 5)) || !present(w, in[1]) || !present(y, numel(out, 5)))
        return APS_ERR_NULL;
    if (!aligned(x, 4) || !aligned(w, 4) || !aligned(y, 4) || (bias && !aligned(bias, 4)))
        return APS_ERR_ALIGN;
    if (numel(out, 5) == 0) return APS_OK;
    if (!extents_ok(in, out, 5)) return APS_ERR_UNSUPPORTED;
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    bool fast = c_out == 16 && in[1] >= 1 && in[1] <= 8;
    for (int i = 0; i < 3; ++i)
        fast = fast && k[i] == 3 && s[i] == 2 && p[i] == 1 && d[i] == 1 && op[i] <= 1;
    if (fast && tensor_cores_on()) {
        // tensor cores (16-byte input rows)
        st = launch_convt3d_tc(x, in, w, bias, y, out, cs);
        if (st != APS_ERR_UNSUPPORTED) return st;
    }
    return launch_convt3d_direct(x, in, w, bias, c_out, k, s, p, d, y, out, cs);
}

// -------------------------------------------------------- convtranspose1d
aps_status aps_convtranspose1d_out_shape(const int64_t in[3], int64_t c_out, int k, int s,
                                         int p, int d, int op, int64_t out[3]) {
    if (!in || !out) return APS_ERR_NULL;
    if (!dims_ok(in, 3) || c_out < 1 || c_out > kMaxElems || in[2] < 1) return APS_ERR_SHAPE;
    const int kk[3] = {k, 1, 1}, ss[3] = {s, 1, 1}, pp[3] = {p, 0, 0}, oo[3] = {op, 0, 0},
              dd[3] = {d, 1, 1};
    aps_status st = conv_params_ok(kk, ss, pp, oo, dd, 1);
    if (st != APS_OK) return st;
    const int64_t L = convt_len(in[2], k, s, p, d, op);
    if (L <= 0) return APS_ERR_SHAPE;
    const int64_t o[3] = {in[0], c_out, L};
    if (!dims_ok(o, 3)) return APS_ERR_SHAPE;
    for (int i = 0; i < 3; ++i) out[i] = o[i];
    return APS_OK;
}

aps_status aps_convtranspose1d(const float *x, const int64_t in[3], const float *w,
                               const float *bias, int64_t c_out, int k, int s, int p, int d,
                               int op, int precision, float *y, aps_stream_t stream) {
    int64_t out[3];
    aps_status st = aps_convtranspose1d_out_shape(in, c_out, k, s, p, d, op, out);
    if (st != APS_OK) return st;
    if (!present(x, numel(in, 3)) || !present(w, in[1]) || !present(y, numel(out, 3)))
        return APS_ERR_NULL;
    if (precision != APS_PREC_FP32 && precision != APS_PREC_TF32 &&
        precision != APS_PREC_TF32X3 && precision != APS_PREC_FP32_FMA)
        return APS_ERR_SHAPE;
    if (!aligned(x, 4) || !aligned(w, 4) || !aligned(y, 4) || (bias && !aligned(bias, 4)))
        return APS_ERR_ALIGN;
    if (numel(out, 3) == 0) return APS_OK;
    if (!extents_ok(in, out, 3)) return APS_ERR_UNSUPPORTED;
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    // no input channels: every output is its bias (exact at any precision)
    if (in[1] == 0) return launch_convt1d_direct(x, in, w, bias, c_out, k, s, p, d, y, out[2], cs);
    if (precision == APS_PREC_TF32 || precision == APS_PREC_TF32X3)
        return !tensor_cores_on() ? APS_ERR_UNSUPPORTED : launch_convt1d_tf32(x, in, w, bias, c_out, k, s, p, d, y, out[2],
                                   precision == APS_PREC_TF32X3, cs);
    if (precision == APS_PREC_FP32 && tensor_cores_on()) {
        // fp32 accuracy: 3xTF32 on the tensor cores where the shape allows
        st = launch_convt1d_tf32(x, in, w, bias, c_out, k, s, p, d, y, out[2], true, cs);
        if (st != APS_ERR_UNSUPPORTED) return st;
    }
    if (in[1] >= 1) {
        st = launch_convt1d_tiled(x, in, w, bias, c_out, k, s, p, d, y, out[2], cs);
        if (st != APS_ERR_UNSUPPORTED) return st;
    }
    return launch_convt1d_direct(x, in, w, bias, c_out, k, s, p, d, y, out[2], cs);
}

// ------------------------------------------------------------ diagnostics
aps_status aps_device_status(unsigned int *bits, int clear) {
    if (!bits) return APS_ERR_NULL;
    if (!status_word()) return APS_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mutex);   // one snapshot at a time
    if (cudaDeviceSynchronize() != cudaSuccess) return APS_ERR_CUDA;
    const cudaError_t e = launch_plain(status_exchange_kernel, dim3(1), dim3(1), 0,
                                       (cudaStream_t)0, clear ? 1 : 0);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return APS_ERR_CUDA;
    }
    unsigned int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_status_snapshot, sizeof(v)) != cudaSuccess) return APS_ERR_CUDA;
    *bits = v;
    return APS_OK;
}

}  // extern "C"

extern "C" void aps_debug_fail_launches(int n) {
    aps::g_fail_launches.store(n > 0 ? n : 0, std::memory_order_relaxed);
}

extern "C" void aps_debug_skip_tensor_cores(int on) {
    aps::g_skip_tc.store(on ? 1 : 0, std::memory_order_relaxed);
}
