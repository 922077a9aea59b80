// Diagnostics: exercise the bounded-wait failure path without any fault.
#include "launch.h"
#include "tma.cuh"

namespace s3d8 {

// One warp waits on an mbarrier that nothing will complete, with a small poll
// budget; on expiry it records S3D8_ERR_TIMEOUT exactly as the streaming
// kernels do, and returns.
__global__ void wait_timeout_kernel(int polls, int *status)
{
    __shared__ __align__(8) unsigned long long bar;
    const uint32_t b = static_cast<uint32_t>(__cvta_generic_to_shared(&bar));
    if (threadIdx.x == 0)
        mbar_init(b, 1);
    __syncwarp();
    bool done = false;
    for (int i = 0; i < polls && !done; ++i) {
        uint32_t ok;
        asm volatile(
            "{\n.reg .pred p;\n"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
            "selp.u32 %0, 1, 0, p;\n}\n"
            : "=r"(ok)
            : "r"(b), "r"(0u)
            : "memory");
        done = ok != 0;
    }
    if (!done && threadIdx.x == 0)
        record_timeout(status);
}

cudaError_t launch_wait_timeout(int polls, int *status, cudaStream_t stream)
{
    wait_timeout_kernel<<<1, 32, 0, stream>>>(polls, status);
    return cudaGetLastError();
}

}  // namespace s3d8
