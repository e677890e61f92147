// aps_dev.cuh -- device-side helpers shared by the kernels: mbarrier and TMA
// inline PTX for sm_103a, bounded waits, and the per-device status word.
#pragma once

#include <cuda.h>          // CUtensorMap (type only; no driver library is linked)
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/aps.h"

namespace aps {

// ------------------------------------------------------------ status word
// Kernels OR APS_DEVERR_* bits into this word (one per device, defined in
// aps_api.cu; launchers pass its device address).  A pipeline wait that runs
// past its limit records APS_DEVERR_TIMEOUT and the kernel stops early.
__device__ __forceinline__ void record_error(unsigned int *status, unsigned int bits) {
    if (status) atomicOr(status, bits);
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Time limit of any single wait inside a kernel.  Every kernel here finishes
// in milliseconds; a wait this long means a copy never landed.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

// ------------------------------------------------------------ launch overlap
// The convolution kernels are launched as programmatic dependents of the
// kernel before them on the stream; the AvgPool3d kernels are not (launched
// that way, the streaming pool ran 5 % slower back to back with the trigger at
// its start, and no faster with the trigger at its end).
// pdl_trigger lets the next launch begin once every CTA of this grid has
// started (its CTAs take SMs as this grid's CTAs leave them); pdl_wait holds
// the calling thread until the grids before this one have completed and their
// writes are visible.  Each thread calls pdl_wait before its first
// global-memory access, so the overlap covers only launch and on-chip set-up.
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ------------------------------------------------------------ mbarriers
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

// Makes initialised barriers visible to the async (TMA) proxy.
__device__ __forceinline__ void mbar_fence_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

// One poll; the thread may be suspended (and is woken when the phase
// completes) for up to kSuspendHintNs, which keeps waiting warps off the issue
// slots of the warps doing work.
constexpr uint32_t kSuspendHintNs = 20000;
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(kSuspendHintNs)
        : "memory");
    return ok != 0;
}

// Waits for the phase with the given parity to complete.  Returns false if it
// has not completed within limit_ns.
__device__ __forceinline__ bool mbar_wait_for(uint64_t *bar, uint32_t parity, uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 15u) == 0 && globaltimer_ns() - t0 > limit_ns) return false;
    }
}
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity) {
    return mbar_wait_for(bar, parity, kWaitLimitNs);
}

// Non-blocking test of the same condition (never suspends the thread): lets a
// thread ask early and use the answer later, off its critical path.
__device__ __forceinline__ bool mbar_test(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// ------------------------------------------------------------------ TMA
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 4-D tiled load of one box into shared memory, completing on `bar`.
// Coordinates are element indices, innermost first; out-of-range cells
// (including negative coordinates) are filled with zeros.
__device__ __forceinline__ void tma_load_4d(void *dst, const CUtensorMap *map, uint64_t *bar,
                                            int c0, int c1, int c2, int c3) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2),
        "r"(c3)
        : "memory");
}

// 3-D tiled load (same rules as tma_load_4d).
__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, uint64_t *bar,
                                            int c0, int c1, int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

// Prefetch of one 3-D box into L2 (no shared memory, no completion signal);
// out-of-range cells are ignored.
__device__ __forceinline__ void tma_prefetch_3d(const CUtensorMap *map, int c0, int c1, int c2) {
    asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(c0), "r"(c1), "r"(c2)
                 : "memory");
}

// 3-D tiled store of one box from shared memory (bulk-group completion).  The
// box's cells outside the tensor are not written.  The source must have been
// made visible to the async proxy (fence.proxy.async) first.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap *map, const void *src, int c0,
                                             int c1, int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(smem_u32(src)), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}
// Untiled bulk copy of `bytes` from shared to global memory (bulk-group
// completion).  Both addresses 16-byte aligned, bytes a multiple of 16; the
// source must have been made visible to the async proxy first.
__device__ __forceinline__ void bulk_store(void *gdst, const void *ssrc, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(
                     reinterpret_cast<uint64_t>(gdst)),
                 "r"(smem_u32(ssrc)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Waits until at most N committed bulk groups of this thread still read smem.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// Waits until at most N committed bulk groups of this thread are incomplete.
template <int N>
__device__ __forceinline__ void bulk_wait() {
    asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

// ---------------------------------- k3 s2 p1 + pool 2: the collapsed taps
// Collapsed tap g = a*4 + b*2 + c of the weights wp[kd*9 + kh*3 + kw] of one
// (ci, co): the sum over kd in T(a), kh in T(b), kw in T(c), where input
// offset 0 takes taps {1, 2} and offset 1 tap {0} (the page's grouping of the
// 27 terms), in ascending (kd, kh, kw).  The loads are unrolled and
// predicated, so that they are all in flight at once.
__device__ __forceinline__ float collapse_tap_ldg(const float *__restrict__ wp, int g) {
    const int a = g >> 2, b = (g >> 1) & 1, c = g & 1;
    float v[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        // e-th term of a 2x2x2 enumeration; terms outside the tap sets are 0
        const int od = e >> 2, oh = (e >> 1) & 1, ow = e & 1;
        const int kd = a ? 0 : 1 + od, kh = b ? 0 : 1 + oh, kw = c ? 0 : 1 + ow;
        const bool in = !(a && od) && !(b && oh) && !(c && ow);
        v[e] = in ? __ldg(wp + kd * 9 + kh * 3 + kw) : 0.f;
    }
    float acc = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e)
        if (!(a && (e >> 2)) && !(b && ((e >> 1) & 1)) && !(c && (e & 1))) acc += v[e];
    return acc;
}

// ------------------------------------------------------------- cp.async
__device__ __forceinline__ void cp_async_4(void *dst, const void *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_16(void *dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

}  // namespace aps
