// tma.cuh -- mbarrier, 1-D bulk async copy (the TMA engine) and bounded-wait
// helpers for sm_103a, as inline PTX.
//
// Every wait here is bounded: it polls mbarrier.try_wait (which itself parks
// the thread for a hardware-chosen interval) and gives up after kWaitLimitNs of
// %globaltimer time, or as soon as another thread of the CTA has raised the
// CTA's abort flag.  A kernel that gives up records a code in the library's
// device error word, stops issuing copies, waits (again bounded) for the
// copies it already issued, and returns.
#pragma once

#include <stdint.h>

namespace osd {

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

// device error codes (low byte: which wait gave up)
constexpr unsigned kErrFullWait = 1u;   // waiting for a bulk copy to land
constexpr unsigned kErrEmptyWait = 2u;  // waiting for consumers to release a stage
constexpr unsigned kErrPeerWait = 3u;   // waiting for a cluster peer's partial statistics

__device__ __forceinline__ uint32_t smem_u32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ uint64_t global_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Make barrier initialisation visible to the other threads and to the async
// (bulk-copy) proxy.
__device__ __forceinline__ void mbar_init_fence()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(bar),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase of parity `parity` to complete.  false: gave up (time
// limit, or *abort raised by another thread when check_abort is set).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, const volatile int *abort,
                                          bool check_abort = true, uint64_t limit_ns = kWaitLimitNs)
{
    if (mbar_try(bar, parity))
        return true;
    const uint64_t t0 = global_ns();
    for (uint32_t n = 1;; n++) {
        if (mbar_try(bar, parity))
            return true;
        if ((n & 15u) == 0) {
            if (check_abort && *abort)
                return false;
            if (global_ns() - t0 > limit_ns)
                return false;
        }
    }
}

// Wait with cluster-scope acquire (the phase was completed by arrivals of
// other CTAs of the cluster); bounded like mbar_wait.
__device__ __forceinline__ bool mbar_try_cluster(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity, const volatile int *abort)
{
    if (mbar_try_cluster(bar, parity))
        return true;
    const uint64_t t0 = global_ns();
    for (uint32_t n = 1;; n++) {
        if (mbar_try_cluster(bar, parity))
            return true;
        if ((n & 15u) == 0) {
            if (*abort)
                return false;
            if (global_ns() - t0 > kWaitLimitNs)
                return false;
        }
    }
}

// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa(uint32_t addr, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

// Store two floats into a (possibly remote) CTA's shared memory.
__device__ __forceinline__ void st_cluster_f32x2(uint32_t raddr, float a, float b)
{
    asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(raddr), "f"(a), "f"(b) : "memory");
}

// Arrive on a (possibly remote) CTA's mbarrier, releasing this thread's prior
// writes at cluster scope.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t raddr)
{
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(raddr) : "memory");
}

__device__ __forceinline__ uint32_t cluster_ctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_nctarank()
{
    uint32_t n;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(n));
    return n;
}

// Full-cluster barrier (every thread of every CTA of the cluster).
__device__ __forceinline__ void cluster_sync_all()
{
    asm volatile("barrier.cluster.arrive.aligned;\n\tbarrier.cluster.wait.aligned;" ::: "memory");
}

// 1-D bulk copy global -> shared, completion counted on `bar` in bytes.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

__device__ __forceinline__ uint4 lds_chunk(uint32_t addr)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}

// Named barrier over `threads` threads (a multiple of 32).
__device__ __forceinline__ void named_sync(uint32_t id, uint32_t threads)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Named barrier that also ANDs a predicate over the participating threads.
__device__ __forceinline__ bool named_and(uint32_t id, uint32_t threads, bool pred)
{
    uint32_t out;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.and.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(out)
        : "r"((uint32_t)pred), "r"(id), "r"(threads)
        : "memory");
    return out != 0;
}

}  // namespace osd
