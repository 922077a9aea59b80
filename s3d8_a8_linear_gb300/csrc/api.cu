// C ABI of the S3D8 library: argument checks, algorithm choice, launches.
// Every check runs before the first CUDA call so that a rejected call touches
// neither the device nor any memory.
#include "../../include/s3d8.h"
#include "launch.h"

#include <cuda_runtime.h>

#include <atomic>

namespace s3d8 {

__device__ int g_device_status;  // sticky S3D8_ERR_TIMEOUT set by bounded waits

static constexpr int kMaxDevices = 64;

// Both caches below are filled on first use per device; threads that race on
// the first call store the same value, and the atomics make that well defined.
int device_sm_count()
{
    static std::atomic<int> cached[kMaxDevices];   // zero-initialised (static storage)
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return 148;
    int n = cached[dev].load(std::memory_order_relaxed);
    if (n == 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            n = 148;
        cached[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

int *device_status_ptr()
{
    static std::atomic<int *> cached[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return nullptr;
    int *ptr = cached[dev].load(std::memory_order_relaxed);
    if (!ptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess)
            return nullptr;
        ptr = static_cast<int *>(p);
        cached[dev].store(ptr, std::memory_order_relaxed);
    }
    return ptr;
}

}  // namespace s3d8

using namespace s3d8;

static bool aligned(const void *p, size_t a)
{
    return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}

static int check_k(int64_t K)
{
    if (K < 16 || (K % 16) != 0 || K > S3D8_MAX_K)
        return S3D8_ERR_INVALID_ARG;
    return S3D8_OK;
}

static int check_mn(int64_t M, int64_t N)
{
    if (M < 0 || N < 0 || M > S3D8_MAX_M || N > S3D8_MAX_N)
        return S3D8_ERR_INVALID_ARG;
    return S3D8_OK;
}

static int cuda_status(cudaError_t e)
{
    return e == cudaSuccess ? S3D8_OK : S3D8_ERR_CUDA;
}

extern "C" {

int s3d8_version(void) { return 100; }

const char *s3d8_status_string(int status)
{
    switch (status) {
    case S3D8_OK: return "ok";
    case S3D8_ERR_INVALID_ARG: return "invalid argument";
    case S3D8_ERR_ALIGNMENT: return "misaligned pointer";
    case S3D8_ERR_UNSUPPORTED: return "unsupported algorithm for this shape or device";
    case S3D8_ERR_CUDA: return "CUDA error";
    case S3D8_ERR_TIMEOUT: return "device-side wait timed out";
    case S3D8_ERR_WORKSPACE: return "workspace missing or too small";
    case S3D8_ERR_BOUNDS: return "in-kernel bounds check failed (debug build)";
    default: return "unknown status";
    }
}

int s3d8_quantize_act(const void *x_bf16, int64_t M, int64_t K, int8_t *xq, float *xscale,
                      void *stream)
{
    int st = check_k(K);
    if (st == S3D8_OK)
        st = check_mn(M, 1);
    if (st != S3D8_OK)
        return st;
    if (M == 0)
        return S3D8_OK;
    if (!x_bf16 || !xq || !xscale)
        return S3D8_ERR_INVALID_ARG;
    if (!aligned(x_bf16, 16) || !aligned(xq, 16) || !aligned(xscale, 4))
        return S3D8_ERR_ALIGNMENT;
    return cuda_status(launch_quantize_act(static_cast<const __nv_bfloat16 *>(x_bf16), (int)M,
                                           (int)K, xq, xscale, static_cast<cudaStream_t>(stream)));
}

int s3d8_decode(const uint8_t *packed, const int8_t *centroids, int64_t N, int64_t K, int8_t *w,
                void *stream)
{
    int st = check_k(K);
    if (st == S3D8_OK)
        st = check_mn(0, N);
    if (st != S3D8_OK)
        return st;
    if (N == 0)
        return S3D8_OK;
    if (!packed || !centroids || !w)
        return S3D8_ERR_INVALID_ARG;
    if (!aligned(packed, 16) || !aligned(w, 16))
        return S3D8_ERR_ALIGNMENT;
    return cuda_status(launch_decode(packed, centroids, (int)N, (int)K, w,
                                     static_cast<cudaStream_t>(stream)));
}

int s3d8_encode(const void *w_bf16, const int8_t *centroids, int64_t N, int64_t K,
                uint8_t *packed, void *chan_scale_bf16, void *workspace, size_t workspace_bytes,
                void *stream)
{
    int st = check_k(K);
    if (st == S3D8_OK)
        st = check_mn(0, N);
    if (st != S3D8_OK)
        return st;
    if (N == 0)
        return S3D8_OK;
    if (!w_bf16 || !centroids || !packed || !chan_scale_bf16)
        return S3D8_ERR_INVALID_ARG;
    if (!aligned(w_bf16, 16) || !aligned(packed, 8) || !aligned(chan_scale_bf16, 2))
        return S3D8_ERR_ALIGNMENT;
    if (!workspace || workspace_bytes < S3D8_ENCODE_WORKSPACE_BYTES)
        return S3D8_ERR_WORKSPACE;
    if (!aligned(workspace, 16))
        return S3D8_ERR_ALIGNMENT;
    return cuda_status(launch_encode(static_cast<const __nv_bfloat16 *>(w_bf16), centroids, (int)N,
                                     (int)K, packed, static_cast<__nv_bfloat16 *>(chan_scale_bf16),
                                     workspace, static_cast<cudaStream_t>(stream)));
}

size_t s3d8_fit_workspace_size(int64_t N, int64_t K)
{
    if (N <= 0 || K <= 0 || N > S3D8_MAX_N || K > S3D8_MAX_K || K % 16 != 0)
        return 0;
    return fit_workspace_bytes(N, K);
}

int s3d8_fit_centroids(const void *w_bf16, int64_t N, int64_t K, const uint32_t *draws,
                       int32_t iters, float *centroids_f32, int8_t *centroids, void *workspace,
                       size_t workspace_bytes, void *stream)
{
    int st = check_k(K);
    if (st == S3D8_OK)
        st = check_mn(0, N);
    if (st != S3D8_OK)
        return st;
    if (N == 0 || iters < 0 || iters > S3D8_FIT_MAX_ITERS)
        return S3D8_ERR_INVALID_ARG;
    if (!w_bf16 || !draws || !centroids_f32 || !centroids)
        return S3D8_ERR_INVALID_ARG;
    if (!aligned(w_bf16, 16) || !aligned(draws, 4) || !aligned(centroids_f32, 4))
        return S3D8_ERR_ALIGNMENT;
    if (!workspace || workspace_bytes < fit_workspace_bytes(N, K))
        return S3D8_ERR_WORKSPACE;
    if (!aligned(workspace, 256))
        return S3D8_ERR_ALIGNMENT;
    return cuda_status(launch_fit(static_cast<const __nv_bfloat16 *>(w_bf16), (int)N, (int)K, draws,
                                  iters, centroids_f32, centroids, workspace,
                                  static_cast<cudaStream_t>(stream)));
}

int s3d8_fake_quant(const void *w_bf16, const int8_t *centroids, int64_t N, int64_t K,
                    void *w_hat_bf16, void *chan_scale_bf16, void *workspace,
                    size_t workspace_bytes, void *stream)
{
    int st = check_k(K);
    if (st == S3D8_OK)
        st = check_mn(0, N);
    if (st != S3D8_OK)
        return st;
    if (N == 0)
        return S3D8_OK;
    if (!w_bf16 || !centroids || !w_hat_bf16 || !chan_scale_bf16)
        return S3D8_ERR_INVALID_ARG;
    if (!aligned(w_bf16, 16) || !aligned(w_hat_bf16, 16) || !aligned(chan_scale_bf16, 2))
        return S3D8_ERR_ALIGNMENT;
    if (!workspace || workspace_bytes < S3D8_ENCODE_WORKSPACE_BYTES)
        return S3D8_ERR_WORKSPACE;
    if (!aligned(workspace, 16))
        return S3D8_ERR_ALIGNMENT;
    return cuda_status(launch_fake_quant(static_cast<const __nv_bfloat16 *>(w_bf16), centroids,
                                         (int)N, (int)K, static_cast<__nv_bfloat16 *>(w_hat_bf16),
                                         static_cast<__nv_bfloat16 *>(chan_scale_bf16), workspace,
                                         static_cast<cudaStream_t>(stream)));
}

int s3d8_selftest_scaled_abs(const void *x_bf16, const void *alpha_bf16, int64_t n, float *out,
                             void *stream)
{
    if (n < 0)
        return S3D8_ERR_INVALID_ARG;
    if (n == 0)
        return S3D8_OK;
    if (!x_bf16 || !alpha_bf16 || !out)
        return S3D8_ERR_INVALID_ARG;
    if (!aligned(x_bf16, 2) || !aligned(alpha_bf16, 2) || !aligned(out, 4))
        return S3D8_ERR_ALIGNMENT;
    return cuda_status(launch_selftest_scaled_abs(static_cast<const __nv_bfloat16 *>(x_bf16),
                                                  static_cast<const __nv_bfloat16 *>(alpha_bf16),
                                                  n, out, static_cast<cudaStream_t>(stream)));
}

// The algorithm AUTO runs (measured on GB300 on the 11B layer's shapes): the
// bulk-copy dp4a GEMV up to 4 tokens; the tcgen05 GEMM with the weights
// decoded into tensor memory for 5..32 tokens, and up to 64 while its 128-row
// tiles fit in one wave;
// the tcgen05 GEMM on shared-memory tiles otherwise.
static int resolve_algo(int64_t M, int64_t N, int64_t K, int algo)
{
    if (algo != S3D8_ALGO_AUTO)
        return algo;
    if (tmem_preferred((int)M, (int)N, (int)K))
        return S3D8_ALGO_TMEM;
    if (M <= 8)
        return S3D8_ALGO_GEMV;
    return S3D8_ALGO_TC;
}

size_t s3d8_linear_workspace_size(int64_t M, int64_t N, int64_t K, int algo)
{
    if (M <= 0 || K <= 0 || M > S3D8_MAX_M || K > S3D8_MAX_K)
        return 0;
    const int r = resolve_algo(M, N, K, algo);
    if (r == S3D8_ALGO_TC)
        return prefill_workspace_bytes((int)M, (int)N, (int)K, prefill_kind((int)M, (int)K));
    if (r == S3D8_ALGO_TMEM && tmem_supported((int)M))
        return tmem_workspace_bytes((int)M, (int)N, (int)K);
    return 0;
}

static int linear_common(const uint8_t *packed, const int8_t *centroids, const void *chan_scale,
                         const int8_t *xq, const float *xscale, int64_t M, int64_t N, int64_t K,
                         void *out_bf16, int32_t *acc, void *workspace, size_t workspace_bytes,
                         int algo, void *stream)
{
    int st = check_k(K);
    if (st == S3D8_OK)
        st = check_mn(M, N);
    if (st != S3D8_OK)
        return st;
    if (algo < S3D8_ALGO_AUTO || algo > S3D8_ALGO_TMEM)
        return S3D8_ERR_INVALID_ARG;
    if (M == 0 || N == 0)
        return S3D8_OK;
    if (!packed || !centroids || !xq)
        return S3D8_ERR_INVALID_ARG;
    if (acc) {
        if (!aligned(acc, 4))
            return S3D8_ERR_ALIGNMENT;
    } else {
        if (!chan_scale || !xscale || !out_bf16)
            return S3D8_ERR_INVALID_ARG;
        if (!aligned(chan_scale, 2) || !aligned(xscale, 4) || !aligned(out_bf16, 2))
            return S3D8_ERR_ALIGNMENT;
    }
    if (!aligned(packed, 16) || !aligned(xq, 16))
        return S3D8_ERR_ALIGNMENT;
    const size_t need = s3d8_linear_workspace_size(M, N, K, algo);
    if (need > 0 && (!workspace || workspace_bytes < need))
        return S3D8_ERR_WORKSPACE;
    algo = resolve_algo(M, N, K, algo);
    if (algo == S3D8_ALGO_SKINNY)   // retired: slower than TMEM at every size it took
        return S3D8_ERR_UNSUPPORTED;
    if (algo == S3D8_ALGO_TMEM && !tmem_supported((int)M))
        return S3D8_ERR_UNSUPPORTED;

    LinearArgs a;
    a.packed = packed;
    a.C = centroids;
    a.cs = static_cast<const __nv_bfloat16 *>(chan_scale);
    a.xq = xq;
    a.xscale = xscale;
    a.M = (int)M;
    a.N = (int)N;
    a.K = (int)K;
    a.out = static_cast<__nv_bfloat16 *>(out_bf16);
    a.acc = acc;
    a.ws = workspace;
    a.ws_bytes = workspace_bytes;
    a.status = device_status_ptr();
    cudaStream_t strm = static_cast<cudaStream_t>(stream);
    if (algo == S3D8_ALGO_TC)
        return cuda_status(launch_prefill_tc(a, prefill_kind(a.M, a.K), strm));
    if (algo == S3D8_ALGO_TMEM)
        return cuda_status(launch_tmem(a, strm));
    if (gemv_tma_supported(a.M, a.K))
        return cuda_status(launch_gemv_tma(a, strm));
    return cuda_status(launch_gemv(a, strm));
}

int s3d8_linear(const uint8_t *packed, const int8_t *centroids, const void *chan_scale_bf16,
                const int8_t *xq, const float *xscale, int64_t M, int64_t N, int64_t K,
                void *out_bf16, void *workspace, size_t workspace_bytes, void *stream)
{
    return linear_common(packed, centroids, chan_scale_bf16, xq, xscale, M, N, K, out_bf16,
                         nullptr, workspace, workspace_bytes, S3D8_ALGO_AUTO, stream);
}

int s3d8_linear_ex(const uint8_t *packed, const int8_t *centroids, const void *chan_scale_bf16,
                   const int8_t *xq, const float *xscale, int64_t M, int64_t N, int64_t K,
                   void *out_bf16, void *workspace, size_t workspace_bytes, int algo, void *stream)
{
    return linear_common(packed, centroids, chan_scale_bf16, xq, xscale, M, N, K, out_bf16,
                         nullptr, workspace, workspace_bytes, algo, stream);
}

int s3d8_linear_acc_i32(const uint8_t *packed, const int8_t *centroids, const int8_t *xq,
                        int64_t M, int64_t N, int64_t K, int32_t *acc, void *workspace,
                        size_t workspace_bytes, int algo, void *stream)
{
    if (!acc) {
        int st = check_k(K);
        if (st == S3D8_OK)
            st = check_mn(M, N);
        if (st != S3D8_OK)
            return st;
        return (M == 0 || N == 0) ? S3D8_OK : S3D8_ERR_INVALID_ARG;
    }
    return linear_common(packed, centroids, nullptr, xq, nullptr, M, N, K, nullptr, acc,
                         workspace, workspace_bytes, algo, stream);
}

int s3d8_linear_batch(const s3d8_linear_job *jobs, int count, int64_t M, void *stream)
{
    if (count < 0 || count > S3D8_MAX_BATCH || M < 0 || M > S3D8_MAX_M)
        return S3D8_ERR_INVALID_ARG;
    if (count == 0 || M == 0)
        return S3D8_OK;
    if (!jobs)
        return S3D8_ERR_INVALID_ARG;
    if (M > 8)
        return S3D8_ERR_UNSUPPORTED;
    GroupArgs g = {};
    g.M = (int)M;
    g.njobs = 0;
    for (int i = 0; i < count; ++i) {
        const s3d8_linear_job &j = jobs[i];
        int st = check_k(j.K);
        if (st == S3D8_OK)
            st = check_mn(M, j.N);
        if (st != S3D8_OK)
            return st;
        if (j.N == 0)
            continue;
        const bool fused = j.x_bf16 != nullptr;
        if (!j.packed || !j.centroids || (fused == (j.xq != nullptr)))
            return S3D8_ERR_INVALID_ARG;
        if (!j.acc && (!j.chan_scale_bf16 || !j.out_bf16))
            return S3D8_ERR_INVALID_ARG;
        if (!fused && !j.acc && !j.xscale)
            return S3D8_ERR_INVALID_ARG;
        if (!aligned(j.packed, 16) || (j.acc && !aligned(j.acc, 4)) ||
            (j.out_bf16 && !aligned(j.out_bf16, 2)) || (j.chan_scale_bf16 && !aligned(j.chan_scale_bf16, 2)))
            return S3D8_ERR_ALIGNMENT;
        if (fused && (!aligned(j.x_bf16, 16) || (j.xq_out && !aligned(j.xq_out, 16)) ||
                      (j.xscale_out && !aligned(j.xscale_out, 4))))
            return S3D8_ERR_ALIGNMENT;
        if (!fused && (!aligned(j.xq, 16) || (j.xscale && !aligned(j.xscale, 4))))
            return S3D8_ERR_ALIGNMENT;
        if (!gemv_group_job_ok((int)M, (int)j.K, fused))
            return S3D8_ERR_UNSUPPORTED;
        GroupJob &d = g.jobs[g.njobs++];
        d.packed = j.packed;
        d.C = j.centroids;
        d.cs = static_cast<const __nv_bfloat16 *>(j.chan_scale_bf16);
        d.x = static_cast<const __nv_bfloat16 *>(j.x_bf16);
        d.xq = j.xq;
        d.xscale = j.xscale;
        d.xq_out = fused ? j.xq_out : nullptr;
        d.xscale_out = fused ? j.xscale_out : nullptr;
        d.out = static_cast<__nv_bfloat16 *>(j.out_bf16);
        d.acc = j.acc;
        d.N = (int)j.N;
        d.K = (int)j.K;
    }
    if (g.njobs == 0)
        return S3D8_OK;
    g.status = device_status_ptr();
    return cuda_status(launch_gemv_group(g, static_cast<cudaStream_t>(stream)));
}

int s3d8_selftest_wait_timeout(int64_t polls, void *stream)
{
    if (polls < 1 || polls > (1 << 24))
        return S3D8_ERR_INVALID_ARG;
    int *st = device_status_ptr();
    if (!st)
        return S3D8_ERR_CUDA;
    return cuda_status(launch_wait_timeout((int)polls, st, static_cast<cudaStream_t>(stream)));
}

int s3d8_device_status(void *stream)
{
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess)
        return S3D8_ERR_CUDA;
    int *p = device_status_ptr();
    if (!p)
        return S3D8_ERR_CUDA;
    int v = 0;
    if (cudaMemcpy(&v, p, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess)
        return S3D8_ERR_CUDA;
    if (v != 0) {
        const int zero = 0;
        if (cudaMemcpy(p, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess)
            return S3D8_ERR_CUDA;
    }
    return v == 0 ? S3D8_OK : v;
}

}  // extern "C"
