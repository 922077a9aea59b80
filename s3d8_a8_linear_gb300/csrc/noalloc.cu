// s3d8_linear_tc_noalloc: the tensor-core linear for callers that cannot
// allocate device memory.  The kernel itself is the one s3d8_linear_ex runs with
// S3D8_ALGO_TC; only the scratch differs.  That path needs M * K * 2 bytes of
// device workspace for the bf16 copy of the activation codes (the operand the
// tensor cores read), and its callers pass workspace they allocated.  Some
// callers cannot: code that runs where cudaMalloc is off limits (inside a
// custom allocator or memory-pool callback, in a real-time loop that must not
// block on the driver's allocator, or in a host that owns all device memory and
// hands out nothing).  For them the scratch lives in a fixed array in this
// library's device image.
#include "../../include/s3d8.h"
#include "launch.h"

#include <cuda_runtime.h>

#include <mutex>

namespace s3d8 {

// Every GPU that loads the library holds this array until the process exits.
// Calls share it and it keeps the last call's contents; each call overwrites
// the part it reads before reading it, so nothing needs clearing between calls.
static __device__ __align__(256) unsigned char g_noalloc_scratch[S3D8_NOALLOC_SCRATCH_BYTES];

static constexpr int kMaxScratchDevices = 64;

// Device address of g_noalloc_scratch on the current device.  In host code the
// array's name is only a host-side stand-in, so the address must come from the
// runtime; it is looked up once per device, with that device current.
static cudaError_t noalloc_scratch(void **ptr)
{
    static std::mutex mu;
    static void *cached[kMaxScratchDevices] = {nullptr};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= kMaxScratchDevices)
        return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (!cached[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess)
            return e;
        cached[dev] = p;
    }
    *ptr = cached[dev];
    return cudaSuccess;
}

}  // namespace s3d8

using namespace s3d8;

int s3d8_linear_tc_noalloc(const uint8_t *packed, const int8_t *centroids, const void *chan_scale_bf16,
                           const int8_t *xq, const float *xscale, int64_t M, int64_t N, int64_t K,
                           void *out_bf16, void *stream)
{
    if (K < 16 || (K % 16) != 0 || K > S3D8_MAX_K || M < 0 || N < 0 || M > S3D8_MAX_M ||
        N > S3D8_MAX_N)
        return S3D8_ERR_INVALID_ARG;
    if (M == 0 || N == 0)
        return S3D8_OK;
    if (!packed || !centroids || !chan_scale_bf16 || !xq || !xscale || !out_bf16)
        return S3D8_ERR_INVALID_ARG;
    if (((uintptr_t)packed & 15) || ((uintptr_t)xq & 15) || ((uintptr_t)chan_scale_bf16 & 1) ||
        ((uintptr_t)xscale & 3) || ((uintptr_t)out_bf16 & 1))
        return S3D8_ERR_ALIGNMENT;
    if (prefill_workspace_bytes((int)M, (int)N, (int)K, kTcOneSm) > (size_t)S3D8_NOALLOC_SCRATCH_BYTES)
        return S3D8_ERR_WORKSPACE;

    void *scratch = nullptr;
    if (noalloc_scratch(&scratch) != cudaSuccess)
        return S3D8_ERR_CUDA;
    LinearArgs a;
    a.packed = packed;
    a.C = centroids;
    a.cs = static_cast<const __nv_bfloat16 *>(chan_scale_bf16);
    a.xq = xq;
    a.xscale = xscale;
    a.M = (int)M;
    a.N = (int)N;
    a.K = (int)K;
    a.out = static_cast<__nv_bfloat16 *>(out_bf16);
    a.acc = nullptr;
    a.ws = scratch;
    a.ws_bytes = S3D8_NOALLOC_SCRATCH_BYTES;
    a.status = device_status_ptr();
    if (!a.status)
        return S3D8_ERR_CUDA;
    return launch_prefill_tc(a, kTcOneSm, static_cast<cudaStream_t>(stream)) == cudaSuccess ? S3D8_OK : S3D8_ERR_CUDA;
}
