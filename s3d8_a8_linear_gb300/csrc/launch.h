// Internal launcher interface between the C ABI (api.cu) and the kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace s3d8 {

struct LinearArgs {
    const uint8_t *packed;      // [G, K]
    const int8_t *C;            // [32 * 3]
    const __nv_bfloat16 *cs;    // [N]            (unused when acc != nullptr)
    const int8_t *xq;           // [M, K]
    const float *xscale;        // [M]            (unused when acc != nullptr)
    int M, N, K;
    __nv_bfloat16 *out;         // [M, N] bf16 output, or
    int32_t *acc;               // [M, N] int32 accumulators (test entry)
    void *ws;                   // device workspace
    size_t ws_bytes;
    int *status;                // device status word
};

// One linear of a grouped launch (see s3d8_linear_job in include/s3d8.h).
struct GroupJob {
    const uint8_t *packed;
    const int8_t *C;
    const __nv_bfloat16 *cs;
    const __nv_bfloat16 *x;     // bf16 activations to quantise in-kernel, or nullptr
    const int8_t *xq;           // pre-quantised codes (when x == nullptr)
    const float *xscale;
    int8_t *xq_out;             // optional copies of the in-kernel codes / scales
    float *xscale_out;
    __nv_bfloat16 *out;
    int32_t *acc;
    int N, K;
};

constexpr int kMaxJobs = 8;

struct GroupArgs {
    GroupJob jobs[kMaxJobs];
    int njobs;
    int M;
    int cta_begin[kMaxJobs + 1];   // filled by the launcher
    int *status;
};

int device_sm_count();
void *tensor_map_encoder_fn();   // cuTensorMapEncodeTiled, or nullptr
int *device_status_ptr();   // this device's sticky status word, or nullptr

cudaError_t launch_quantize_act(const __nv_bfloat16 *x, int M, int K, int8_t *xq, float *xscale,
                                cudaStream_t stream);
cudaError_t launch_encode(const __nv_bfloat16 *w, const int8_t *C, int N, int K, uint8_t *packed,
                          __nv_bfloat16 *chan_scale, void *workspace, cudaStream_t stream);
cudaError_t launch_fake_quant(const __nv_bfloat16 *w, const int8_t *C, int N, int K,
                              __nv_bfloat16 *w_hat, __nv_bfloat16 *chan_scale, void *workspace,
                              cudaStream_t stream);
size_t fit_workspace_bytes(int64_t N, int64_t K);
cudaError_t launch_fit(const __nv_bfloat16 *w, int N, int K, const uint32_t *r, int iters,
                       float *cf, int8_t *C, void *workspace, cudaStream_t stream);
cudaError_t launch_selftest_scaled_abs(const __nv_bfloat16 *x, const __nv_bfloat16 *alpha,
                                       int64_t n, float *out, cudaStream_t stream);
cudaError_t launch_decode(const uint8_t *packed, const int8_t *C, int N, int K, int8_t *w,
                          cudaStream_t stream);
cudaError_t launch_gemv(const LinearArgs &a, cudaStream_t stream);
bool gemv_tma_supported(int M, int K);
cudaError_t launch_wait_timeout(int polls, int *status, cudaStream_t stream);
bool gemv_group_job_ok(int M, int K, bool fused);
cudaError_t launch_gemv_group(GroupArgs &g, cudaStream_t stream);
cudaError_t launch_gemv_tma(const LinearArgs &a, cudaStream_t stream);
// Tensor-core path, three kernels: one SM per tile (decoding packed tiles
// itself), SM pairs decoding packed tiles themselves, or SM pairs on weights
// expanded to bf16 in the workspace first.  prefill_kind(M, K) picks by token
// count and row length.
constexpr int kTcOneSm = 0, kTcPairFused = 1, kTcPairExpanded = 2;
int prefill_kind(int M, int K);
size_t prefill_workspace_bytes(int M, int N, int K, int kind);
cudaError_t launch_prefill_tc(const LinearArgs &a, int kind, cudaStream_t stream);
cudaError_t launch_prefill_pair(const LinearArgs &a, const __nv_bfloat16 *act, const __nv_bfloat16 *wdec,
                                int32_t *part, int nsplit, int kbps, cudaStream_t stream);
cudaError_t launch_prefill_fused(const LinearArgs &a, const uint16_t *act_f16, int32_t *part, int nsplit, int kbps,
                                 int g2, cudaStream_t stream);
// Split-K finish shared by the tensor-core paths: sums int32 partials
// [nsplit][M][N] into a.out (epilogue) or a.acc.
cudaError_t launch_splitk_finalize(const int32_t *part, int nsplit, const LinearArgs &a, cudaStream_t stream);
// tcgen05 GEMM with the weights decoded into tensor memory (decode_tmem.cu):
// 1..64 tokens.
bool tmem_supported(int M);
// AUTO takes it for 5..32 tokens, and up to 64 when its tiles fit in one wave
// (not with more 128-row tiles than SMs).
bool tmem_preferred(int M, int N, int K);
size_t tmem_workspace_bytes(int M, int N, int K);
cudaError_t launch_tmem(const LinearArgs &a, cudaStream_t stream);

}  // namespace s3d8
