// PTX wrappers and device-status helpers shared by the decode kernels.
// Internal to the library (included by its .cu files only).
#pragma once

#include <cuda_bf16.h>

#include "oxd_internal.h"

namespace oxd {
namespace {

constexpr int kDeviceBadPage = 1;
constexpr int kDevicePlanMismatch = 2;
constexpr int kDeviceWaitTimeout = 3;
constexpr float kLn2 = 0.693147180559945309f;

// ------------------------------------------------------------------ PTX wrappers

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// ---- thread-block clusters (a cluster merge of split pieces)

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Every thread of every CTA of the cluster (all threads of each warp).
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// The same barrier, arriving without release semantics (this thread's
// earlier writes need no ordering before the other CTAs pass it).
__device__ __forceinline__ void cluster_sync_relaxed_arrive() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Arrive on the mbarrier at the same shared-memory offset in CTA `rank` of
// the cluster; release at cluster scope (orders this thread's earlier
// writes, and those it has seen through a barrier, before the arrival).
__device__ __forceinline__ void mbar_arrive_remote(uint64_t* bar, uint32_t rank) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_addr(bar)), "r"(rank));
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(remote)
                 : "memory");
}

// Bounded wait for phase `parity` of a local mbarrier with acquire at
// cluster scope (writes released by the cluster's arrivals are then seen).
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity,
                                                  long long limit_ns) {
    uint64_t t0 = 0;
    for (int i = 0;; ++i) {
        uint32_t done;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(done)
            : "r"(smem_addr(bar)), "r"(parity)
            : "memory");
        if (done) return true;
        uint64_t t;
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
        if (i == 0) t0 = t;
        else if (t - t0 > static_cast<uint64_t>(limit_ns)) return false;
    }
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Non-blocking test of the phase (never suspends the thread).
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// Limits below this are polled with test_wait: try_wait may suspend the
// thread for a hardware-chosen time, longer than such a limit.
constexpr long long kPolledWaitNs = 1000000LL;  // 1 ms

// Waits for the phase with `parity` to complete. Gives up (returns false)
// after limit_ns, or early once *abort is set by another warp. Pipeline
// waits take the run's limit (DecodeParams / PrefillParams wait_ns); the
// waits for copies and MMAs already in flight before a CTA leaves take
// kWaitTimeoutNs, whatever the run's limit, so no CTA exits while the
// asynchronous units still write its shared memory.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity,
                                          const volatile int* abort, long long limit_ns) {
    if (limit_ns < kPolledWaitNs) {
        const uint64_t t0 = global_ns();
        while (true) {
            if (mbar_test_wait(bar, parity)) return true;
            if (abort != nullptr && *abort) return false;
            if (global_ns() - t0 > static_cast<uint64_t>(limit_ns)) return false;
        }
    }
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (abort != nullptr && *abort) return false;
        if (global_ns() - t0 > static_cast<uint64_t>(limit_ns)) return false;
    }
}

// The same wait without the polled form, for the tcgen05 kernels: their MMA
// thread checks the limit itself on every idle poll, so a short limit runs
// out there; their other waits honour it to within try_wait's suspension.
// (The polled branch cost their step about 0.5 us in 53, A/B.)
__device__ __forceinline__ bool mbar_wait_tc(uint64_t* bar, uint32_t parity,
                                             const volatile int* abort, long long limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (abort != nullptr && *abort) return false;
        if (global_ns() - t0 > static_cast<uint64_t>(limit_ns)) return false;
    }
}

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, uint64_t* bar,
                                            int c0, int c1, int c2, int c3) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_addr(bar)), "r"(c0), "r"(c1), "r"(c2),
        "r"(c3)
        : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint64_t* bar,
                                            int c0, int c1, int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_addr(bar)), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint64_t* bar,
                                            int c0, int c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_addr(bar)), "r"(c0), "r"(c1)
        : "memory");
}

// Contiguous global -> shared copy (16-byte aligned, size a multiple of 16).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(dst), "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// Waits until the grids this one depends on programmatically have completed
// and their memory operations are visible (a no-op for a plain launch).
__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Packed f32x2 arithmetic and a three-input max (sm_100-class): half the
// issue slots of the scalar forms for the softmax's bulk work, same results
// (each lane rounds as the scalar instruction does).
__device__ __forceinline__ float max3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// (a, b) * (s, s) + (c, c)
__device__ __forceinline__ void fma2(float a, float b, float s, float c, float& x, float& y) {
    asm("{\n\t.reg .b64 u, v, w, r;\n\t"
        "mov.b64 u, {%2, %3};\n\tmov.b64 v, {%4, %4};\n\tmov.b64 w, {%5, %5};\n\t"
        "fma.rn.f32x2 r, u, v, w;\n\tmov.b64 {%0, %1}, r;\n\t}"
        : "=f"(x), "=f"(y)
        : "f"(a), "f"(b), "f"(s), "f"(c));
}

// (x, y) += (a, b)
__device__ __forceinline__ void add2(float& x, float& y, float a, float b) {
    asm("{\n\t.reg .b64 u, v, r;\n\t"
        "mov.b64 u, {%0, %1};\n\tmov.b64 v, {%2, %3};\n\t"
        "add.rn.f32x2 r, u, v;\n\tmov.b64 {%0, %1}, r;\n\t}"
        : "+f"(x), "+f"(y)
        : "f"(a), "f"(b));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}


// The status word is {run epoch : 32, code : 32}. The first error of a run
// replaces whatever an older run left there; later errors of the same run
// keep it. Only error paths touch the word, so nothing has to reset it.
__device__ __forceinline__ void record_status(unsigned long long* st, uint32_t epoch, int code) {
    const unsigned long long want =
        (static_cast<unsigned long long>(epoch) << 32) | static_cast<uint32_t>(code);
    unsigned long long old = *reinterpret_cast<volatile unsigned long long*>(st);
    for (int tries = 0; tries < 4096; ++tries) {
        if ((old >> 32) == epoch && static_cast<uint32_t>(old) != 0u) return;
        const unsigned long long prev = atomicCAS(st, old, want);
        if (prev == old) return;
        old = prev;
    }
}

}  // namespace
}  // namespace oxd
