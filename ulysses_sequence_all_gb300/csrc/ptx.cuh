// ptx.cuh -- inline-PTX wrappers for the sm_103a data movers: mbarrier, bulk async copies
// (cp.async.bulk global<->shared, the TMA unit's non-tensor form), bulk groups, global timer.
#pragma once
#include <cstdint>

namespace uly {

// Every wait in these kernels gives up after this many nanoseconds of the global timer, records
// an error in the device status word and lets the kernel return.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

// Shared memory of one SM (GB300): 228 KiB per SM, 1 KiB of it reserved per resident CTA, and at
// most 227 KiB of dynamic shared memory for one CTA.
constexpr int kSmemPerSm = 228 * 1024;
constexpr int kSmemReservedPerCta = 1024;
constexpr int kSmemPerCtaMax = 227 * 1024;

// Bits of the device status word.
constexpr unsigned kStatusWaitTimeout = 1u;
constexpr unsigned kStatusDrainTimeout = 2u;

// Non-negative a / b (b > 0), in 32-bit arithmetic when both fit, which is the common case.
__device__ __forceinline__ int64_t div_fast(int64_t a, int64_t b)
{
    if (((a | b) >> 32) == 0) return int64_t(uint32_t(a) / uint32_t(b));
    return a / b;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

// Makes the initialised barriers visible to the async proxy (the bulk-copy unit).
__device__ __forceinline__ void fence_barrier_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(
                     smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar)
{
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// Suspend-time hint (ns) for a try_wait that finds the phase incomplete: the warp may sleep up to
// this long in hardware instead of returning at once (0 = the implementation's default).
#ifndef ULY_WAIT_HINT_NS
#define ULY_WAIT_HINT_NS 0
#endif

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity)
{
    uint32_t done;
#if ULY_WAIT_HINT_NS > 0
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity), "n"(ULY_WAIT_HINT_NS)
        : "memory");
#else
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
#endif
    return done != 0;
}

// Waits for the barrier phase with the given parity to complete; false after limit_ns.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  uint64_t limit_ns = kWaitLimitNs)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_timer_ns() - t0 > limit_ns) return false;
    }
    return true;
}

// The same with a suspend-time hint: a waiting thread may be parked by the hardware for up to
// HINT_NS nanoseconds (woken early when the phase completes) instead of polling, which leaves
// issue slots to the warps doing the work.
template <uint32_t HINT_NS>
__device__ __forceinline__ bool mbar_try_wait_hint(uint64_t* bar, uint32_t parity)
{
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity), "n"(HINT_NS)
        : "memory");
    return done != 0;
}

template <uint32_t HINT_NS>
__device__ __forceinline__ bool mbar_wait_bounded_hint(uint64_t* bar, uint32_t parity,
                                                       uint64_t limit_ns = kWaitLimitNs)
{
    if (mbar_try_wait_hint<HINT_NS>(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait_hint<HINT_NS>(bar, parity)) {
        if (global_timer_ns() - t0 > limit_ns) return false;
    }
    return true;
}

// Bulk copy global -> shared; completion is signalled as transaction bytes on `bar`.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst_smem, const void* src_gmem, uint32_t bytes,
                                         uint64_t* bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_u32(dst_smem)),
        "l"(src_gmem), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// Tiled tensor copy global -> shared of one box of a 3-D tensor map at coordinates (c0, c1, c2)
// (elements; c0 counts the innermost dimension); completion is signalled as transaction bytes (the
// whole box, out-of-range elements included) on `bar`. `map` is the address of a CUtensorMap in
// parameter, constant or global memory; dst 128-byte aligned.
__device__ __forceinline__ void tensor_g2s_3d(void* dst_smem, const void* map, int c0, int c1,
                                              int c2, uint64_t* bar)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst_smem)),
        "l"(map), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
        : "memory");
}

// The same for a 4-D map: coordinates (c0, c1, c2, c3), c0 the innermost.
__device__ __forceinline__ void tensor_g2s_4d(void* dst_smem, const void* map, int c0, int c1,
                                              int c2, int c3, uint64_t* bar)
{
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(smem_u32(dst_smem)),
        "l"(map), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_u32(bar))
        : "memory");
}

// Tiled tensor copy shared -> global of one box, tracked by this thread's bulk async-groups; the
// parts of the box outside the tensor's extent are not written.
__device__ __forceinline__ void tensor_s2g_3d(const void* map, int c0, int c1, int c2,
                                              const void* src_smem)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
            map),
        "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(src_smem))
        : "memory");
}

// The same for a 4-D map: coordinates (c0, c1, c2, c3), c0 the innermost.
__device__ __forceinline__ void tensor_s2g_4d(const void* map, int c0, int c1, int c2, int c3,
                                              const void* src_smem)
{
    asm volatile(
        "cp.async.bulk.tensor.4d.global.shared::cta.tile.bulk_group [%0, {%1, %2, %3, %4}], [%5];" ::"l"(
            map),
        "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_u32(src_smem))
        : "memory");
}

// Bulk copy shared -> global, tracked by this thread's bulk async-groups.
__device__ __forceinline__ void bulk_s2g(void* dst_gmem, const void* src_smem, uint32_t bytes)
{
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst_gmem),
                 "r"(smem_u32(src_smem)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Wait until at most N of this thread's bulk groups still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read()
{
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// Wait until at most N of this thread's bulk groups are incomplete (writes visible).
template <int N>
__device__ __forceinline__ void bulk_wait()
{
    asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

// 16-byte global load that bypasses L1 (data is read once) and 16-byte store.
__device__ __forceinline__ uint4 ld_stream_v4(const void* p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ void st_v4(void* p, const uint4& v)
{
    asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ void st_v2(void* p, uint32_t a, uint32_t b)
{
    asm volatile("st.global.v2.u32 [%0], {%1, %2};" ::"l"(p), "r"(a), "r"(b) : "memory");
}

__device__ __forceinline__ void st_shared_v4(void* p, const uint4& v)
{
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(smem_u32(p)), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}

// Orders this thread's earlier generic-proxy shared-memory writes before later async-proxy
// (bulk copy) reads of the same memory, once a barrier has passed between them.
__device__ __forceinline__ void fence_proxy_async_shared()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void st_shared_v2(void* p, uint32_t a, uint32_t b)
{
    asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(smem_u32(p)), "r"(a), "r"(b) : "memory");
}

__device__ __forceinline__ uint2 ld_shared_v2(const void* p)
{
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(smem_u32(p)));
    return v;
}

__device__ __forceinline__ uint4 ld_shared_v4(const void* p)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(smem_u32(p)));
    return v;
}

}  // namespace uly
