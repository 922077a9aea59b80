// Bulk-copy (TMA) and mbarrier helpers for sm_103a, written as inline PTX.
//
// Every wait is bounded: after kWaitPolls unsuccessful polls the caller gets
// `false`, records S3D8_ERR_TIMEOUT in the library's device status word and
// stops, instead of spinning forever.
#pragma once

#include <stdint.h>

namespace s3d8 {

constexpr int kWaitPolls = 1 << 22;
constexpr int kStatusTimeout = -5;  // S3D8_ERR_TIMEOUT
constexpr int kStatusBounds = -7;   // S3D8_ERR_BOUNDS

// In-kernel bounds check of the debug build (S3D8_DEBUG_CHECKS): a failed
// check records S3D8_ERR_BOUNDS in the device status word and returns false, so
// that the caller skips the access; nothing traps.  In the normal build it is
// `true` and costs nothing.
#ifdef S3D8_DEBUG_CHECKS
__device__ __forceinline__ bool dcheck(int *status, bool ok)
{
    if (!ok && status)
        atomicExch(status, kStatusBounds);
    return ok;
}
#else
__device__ __forceinline__ bool dcheck(int *, bool)
{
    return true;
}
#endif

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

// Polls the phase with parity `parity` of the mbarrier; false after the poll budget.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity)
{
    for (int i = 0; i < kWaitPolls; ++i) {
        uint32_t done;
        asm volatile(
            "{\n.reg .pred p;\n"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
            "selp.u32 %0, 1, 0, p;\n}\n"
            : "=r"(done)
            : "r"(bar), "r"(parity)
            : "memory");
        if (done)
            return true;
    }
    return false;
}

// 1-D bulk copy global -> shared, completion signalled on `bar` (tx bytes).
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// L2 cache policy that marks lines as the first to evict: for weight bytes that
// a launch reads exactly once, so that they do not push activations, scales and
// outputs (read again by every block, or by the next kernel) out of L2.
__device__ __forceinline__ uint64_t l2_evict_first_policy()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// As bulk_load, with an L2 cache policy for the source lines.
__device__ __forceinline__ void bulk_load_hint(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar,
                                               uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
        "%4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

// Orders this thread's earlier generic-proxy shared-memory accesses before
// later async-proxy (bulk copy) accesses to the same memory.
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ uint4 lds_v4(uint32_t addr)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}

__device__ __forceinline__ void record_timeout(int *status)
{
    if (status)
        atomicExch(status, kStatusTimeout);
}

}  // namespace s3d8
