/*
 * s3d8.h - C ABI of the GB300 (sm_103a) S3D8 W2.7A8 linear-layer library.
 *
 * The layer (Llama-Mobile: Efficient 2.7-Bit Quantization of VLMs, section 3.4,
 * Eq. 1, and section 4.3 for Y = X W^T) is
 *
 *     out[m, n] = bf16( xscale[m] * chan_scale[n] * sum_k xq[m, k] * Wq[n, k] )
 *
 * where Wq[n, k] = s * C[q][n mod 3] is decoded on the fly from one packed byte
 * per (n / 3, k).  Byte layout ("11 billion parameters on a phone", Graphcore
 * Research blog, section "Bit layout"): bit 0 = S0, bits 1..5 = Q (Q0 in bit
 * 1), bit 6 = S1, bit 7 = S2 xor S0; a selector of 0 is +, 1 is -.  Selector
 * S_d and table column d belong to output channel 3g + d of packed row g
 * (blog, "Output channel packing").
 *
 * Conventions shared by every entry point
 *   - Every pointer is caller-owned DEVICE memory unless stated otherwise.  The
 *     library allocates nothing per call and keeps no state except one device
 *     status word (see s3d8_device_status) and the fixed scratch array of
 *     s3d8_linear_tc_noalloc.
 *   - Calls are asynchronous on `stream` (a cudaStream_t passed as void*; NULL
 *     is the legacy default stream).  They neither synchronise nor read device
 *     memory from the host.
 *   - Arguments are checked before anything is launched; a failed check returns
 *     a negative s3d8_status and touches no memory.  A launch failure returns
 *     S3D8_ERR_CUDA.
 *   - Shapes: M tokens, N output channels, K input columns.  G = ceil(N / 3)
 *     packed rows.  M == 0 or N == 0 is a valid empty call (returns S3D8_OK and
 *     launches nothing).  K must be a positive multiple of 16 (the pages' fused
 *     kernel steps K by 16) and at most S3D8_MAX_K, so that every int32
 *     accumulator is exact (127 * 127 * K < 2^31).
 *   - Not checked, for speed: centroid values must lie in 0..127 and the bf16
 *     inputs must be finite.
 *   - The decode-regime kernels (s3d8_linear_batch, and s3d8_linear* for
 *     M <= 8) use programmatic dependent launch: when the kernel before them on
 *     the stream allows an early start (this library's kernels do), they read
 *     the packed weights and centroid tables while that kernel is still
 *     finishing, and everything else only after it has completed.  So packed
 *     weights and centroids must not be outputs of the kernel launched
 *     immediately before on the same stream; activations and scales may be.
 */
#ifndef S3D8_H
#define S3D8_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define S3D8_MAX_K 133144
#define S3D8_MAX_M (1 << 24)
#define S3D8_MAX_N (1 << 26)

typedef enum {
    S3D8_OK = 0,
    S3D8_ERR_INVALID_ARG = -1, /* null pointer, bad shape, K % 16 != 0, K too large */
    S3D8_ERR_ALIGNMENT = -2,   /* a pointer misses its required alignment         */
    S3D8_ERR_UNSUPPORTED = -3, /* algorithm not available for this shape/device   */
    S3D8_ERR_CUDA = -4,        /* a CUDA call or kernel launch failed             */
    S3D8_ERR_TIMEOUT = -5,     /* a bounded device-side wait ran out (sticky)     */
    S3D8_ERR_WORKSPACE = -6,   /* workspace missing or smaller than required      */
    S3D8_ERR_BOUNDS = -7       /* debug build only: an in-kernel bounds check failed (sticky) */
} s3d8_status;

/* Algorithm choice for s3d8_linear_ex.  AUTO picks by shape: GEMV up to 4
 * tokens; TMEM for 5..32 tokens, and up to 64
 * tokens while its tiles fit in one wave on the device; TC otherwise.  The value
 * 2 (a register-fragment mma.sync path, slower than TMEM at every size it took)
 * is retired and stays reserved: it returns S3D8_ERR_UNSUPPORTED. */
typedef enum {
    S3D8_ALGO_AUTO = 0,
    S3D8_ALGO_GEMV = 1,    /* CUDA-core table decode + dp4a; bulk-copy rings up to 8 tokens      */
    S3D8_ALGO_SKINNY = 2,  /* retired: S3D8_ERR_UNSUPPORTED                                      */
    S3D8_ALGO_TC = 3,      /* tcgen05 16-bit tensor-core GEMM with exact chunked int32 sums    */
    S3D8_ALGO_TMEM = 4     /* tcgen05 fp16 GEMM, weights decoded into tensor memory, 1..64 tokens */
} s3d8_algo;

/*
 * Per-token INT8 activation quantisation (the pages fix channel-scaled INT8
 * activations with one float scale per activation vector; the absmax/127 rule
 * follows the paper's channel scale alpha_i = max_j |W_ij| / 127, section 3.4).
 *   x_bf16 : [M, K] bfloat16, row-major, 16-byte aligned
 *   xq     : [M, K] int8 output, row-major, 16-byte aligned
 *   xscale : [M] fp32 output, xscale[m] = absmax_k |x[m,k]| / 127 (IEEE division)
 * xq[m,k] = clamp(round_half_even(x[m,k] / xscale[m]), -127, 127) with IEEE fp32
 * division; an all-zero row gives xscale 0 and codes 0.
 */
int s3d8_quantize_act(const void *x_bf16, int64_t M, int64_t K, int8_t *xq, float *xscale,
                      void *stream);

/*
 * Standalone S3D8 -> INT8 unpack (the pages' dequantisation kernel, blog
 * section "Fast? How fast?"; paper section 4.3).
 *   packed    : [G, K] uint8, row-major, 16-byte aligned
 *   centroids : [32 * 3] int8, row-major C[q][d] (any alignment)
 *   w         : [N, K] int8 output, row-major, 16-byte aligned; row n is
 *               component n % 3 of packed row n / 3.  Padded rows are not written.
 */
int s3d8_decode(const uint8_t *packed, const int8_t *centroids, int64_t N, int64_t K, int8_t *w,
                void *stream);

/*
 * Direct-cast encoder: bf16 weights -> channel scales and packed S3D8 bytes,
 * with the centroid table held fixed (paper section 3.4, "Quantization": the
 * forward assignment; the byte layout of blog section "Bit layout").
 *   w_bf16     : [N, K] bfloat16, row-major, 16-byte aligned
 *   centroids  : [32 * 3] int8, row-major C[q][d], values 0..127 (any alignment)
 *   packed     : [G, K] uint8 output, row-major, 8-byte aligned
 *   chan_scale : [N] bfloat16 output, 2-byte aligned
 *   workspace  : device scratch of S3D8_ENCODE_WORKSPACE_BYTES, 16-byte
 *                aligned, caller-owned, not shared by calls that overlap on
 *                the GPU (S3D8_ERR_WORKSPACE when missing or smaller)
 * chan_scale[n] = bf16_rn(max_k |W[n,k]| / 127) (fp32 IEEE division).  For
 * packed row g and column k, with alpha the stored scale of each channel:
 * W'_d = |W[3g+d,k]| / alpha (IEEE fp32; 0 when alpha is 0 and for the padded
 * channels 3g+d >= N); the selector of channel d is 0 (+) where W >= 0,
 * including -0, and 1 elsewhere (0 for padded channels); Q is the first index
 * l minimising ((C_l0 - W'_0)^2 + (C_l1 - W'_1)^2) + (C_l2 - W'_2)^2 evaluated
 * in fp32, every operation rounded to nearest.  Two launches: scales and a
 * per-call candidate table (in the workspace), then the assignment.
 */
#define S3D8_ENCODE_WORKSPACE_BYTES 16384u
int s3d8_encode(const void *w_bf16, const int8_t *centroids, int64_t N, int64_t K,
                uint8_t *packed, void *chan_scale_bf16, void *workspace, size_t workspace_bytes,
                void *stream);

/*
 * QAT fake-quant forward (paper section 3.4, "Quantization": in QAT the weight
 * is quantised in the forward pass with the centroids frozen and rebuilt by
 * Eq. 1): w_hat[n,k] = bf16_rn(s * alpha_n * C[q][n mod 3]) with alpha, s and q
 * exactly as s3d8_encode chooses them (the product alpha C is exact in fp32).
 * The straight-through backward passes the gradient of w_hat to w unchanged
 * (no clipping: every weight is inside the absmax range), so it needs no call.
 *   w_bf16     : [N, K] bfloat16, row-major, 16-byte aligned
 *   centroids  : [32 * 3] int8, row-major C[q][d], values 0..127
 *   w_hat_bf16 : [N, K] bfloat16 output, row-major, 16-byte aligned
 *   chan_scale : [N] bfloat16 output (alpha), 2-byte aligned
 *   workspace  : as for s3d8_encode (S3D8_ENCODE_WORKSPACE_BYTES, 16-byte aligned)
 */
int s3d8_fake_quant(const void *w_bf16, const int8_t *centroids, int64_t N, int64_t K,
                    void *w_hat_bf16, void *chan_scale_bf16, void *workspace,
                    size_t workspace_bytes, void *stream);

/*
 * Centroid fit (paper section 3.4, "Quantization": C = Round(Lloyd-Max(W'))
 * with k-means++ initialisation, Arthur and Vassilvitskii, SODA 2007), on the
 * ceil(N/3) K points W'_p = (|W[3g+d,k]| / alpha_{3g+d})_{d=0..2}, with
 * alpha and W' exactly as in s3d8_encode (padded channels are 0).
 *   w_bf16        : [N, K] bfloat16, row-major, 16-byte aligned
 *   draws         : [32] uint32 random draws (device), 4-byte aligned
 *   iters         : Lloyd iterations, 0..S3D8_FIT_MAX_ITERS (0: k-means++ only)
 *   centroids_f32 : [32 * 3] fp32 output, the fitted centroids before Round
 *   centroids     : [32 * 3] int8 output, the table: rint (ties to even) of
 *                   centroids_f32 clamped to 0..127
 *   workspace     : s3d8_fit_workspace_size(N, K) bytes, 256-byte aligned,
 *                   caller-owned, not shared by calls that overlap on the GPU
 *                   (about 16 bytes per point)
 * k-means++: centre 0 is point floor(draws[0] Np / 2^32); centre t >= 1 is
 * the first point whose inclusive prefix sum of w_p = floor(D2_p 2^20) exceeds
 * floor(draws[t] S / 2^32), S = sum w_p, D2_p the fp32 squared distance to the
 * nearest chosen centre (point floor(draws[t] Np / 2^32) when S = 0).
 * Lloyd: nearest centroid per point in fp32 (lowest index on a tie); each
 * nonempty cluster's centroid becomes float(RN(sum_p floor(W'_p 2^20) / n)
 * 2^-20) per component (fp64 division); empty clusters stay.  All sums are
 * exact integers, so the result does not depend on the order of summation.
 * 2 + 63 + 2 iters + 1 launches; N == 0 is rejected (no points).
 */
#define S3D8_FIT_MAX_ITERS 10000
size_t s3d8_fit_workspace_size(int64_t N, int64_t K);
int s3d8_fit_centroids(const void *w_bf16, int64_t N, int64_t K, const uint32_t *draws,
                       int32_t iters, float *centroids_f32, int8_t *centroids, void *workspace,
                       size_t workspace_bytes, void *stream);

/*
 * Self-test of the encoder's scaled magnitude: out[i] = |x[i]| / alpha[i]
 * through the same device code the encoder uses (a correction step on a
 * per-channel reciprocal, IEEE division outside its range).  Must equal the
 * IEEE fp32 quotient for every finite x and alpha > 0 with |x| <= 2^20 alpha
 * (the encoder only meets |x| <= 128 alpha); alpha = 0 gives 0.  x, alpha:
 * [n] bfloat16; out: [n] fp32.
 */
int s3d8_selftest_scaled_abs(const void *x_bf16, const void *alpha_bf16, int64_t n, float *out,
                             void *stream);

/* Bytes of device workspace s3d8_linear_ex needs for this shape and algorithm
 * (0 when none).  Host function; the tensor-core algorithm's size depends on
 * the current device's SM count (how far a small M splits K). */
size_t s3d8_linear_workspace_size(int64_t M, int64_t N, int64_t K, int algo);

/*
 * The S3D8 linear layer, Y = X W^T (paper section 4.3, Eq. 1; blog fused
 * matrix-vector example for the epilogue order and dtypes):
 *   out[m,n] = bf16_rn( (xscale[m] * float(acc[m,n])) * float(chan_scale[n]) )
 * with acc the exact int32 sum over k of xq[m,k] * Wq[n,k].
 *   packed     : [G, K] uint8, row-major (k contiguous), 16-byte aligned
 *   centroids  : [32 * 3] int8, row-major C[q][d]
 *   chan_scale : [N] bfloat16, 2-byte aligned
 *   xq         : [M, K] int8, row-major, 16-byte aligned
 *   xscale     : [M] fp32, 4-byte aligned
 *   out_bf16   : [M, N] bfloat16 output, row-major, 2-byte aligned
 *   workspace  : device scratch of s3d8_linear_workspace_size(M, N, K, AUTO)
 *                bytes (may be NULL when that size is 0); caller-owned, must
 *                not be shared by calls that overlap on the GPU.
 */
int s3d8_linear(const uint8_t *packed, const int8_t *centroids, const void *chan_scale_bf16,
                const int8_t *xq, const float *xscale, int64_t M, int64_t N, int64_t K,
                void *out_bf16, void *workspace, size_t workspace_bytes, void *stream);

/* As s3d8_linear with an explicit algorithm (s3d8_algo).  Returns
 * S3D8_ERR_UNSUPPORTED when that algorithm cannot run the shape. */
int s3d8_linear_ex(const uint8_t *packed, const int8_t *centroids, const void *chan_scale_bf16,
                   const int8_t *xq, const float *xscale, int64_t M, int64_t N, int64_t K,
                   void *out_bf16, void *workspace, size_t workspace_bytes, int algo,
                   void *stream);

/*
 * The exact integer part of the layer alone: acc[m, n] = sum_k xq[m,k] * Wq[n,k]
 * as int32 [M, N] row-major (4-byte aligned), through the same kernels as
 * s3d8_linear_ex with `algo`.  Exists so that the accumulators can be checked
 * bit for bit.
 */
int s3d8_linear_acc_i32(const uint8_t *packed, const int8_t *centroids, const int8_t *xq,
                        int64_t M, int64_t N, int64_t K, int32_t *acc, void *workspace,
                        size_t workspace_bytes, int algo, void *stream);

/*
 * One linear of a grouped call (s3d8_linear_batch).  All pointers are device
 * memory and follow the layouts of s3d8_linear.  Exactly one of x_bf16 and xq
 * is given:
 *   x_bf16      [M, K] bfloat16 activations, quantised inside the kernel with
 *               the s3d8_quantize_act rule (16-byte aligned; M * K <= 28672);
 *   xq, xscale  [M, K] int8 codes and [M] fp32 scales, already quantised.
 * xq_out / xscale_out (optional, used only with x_bf16) receive the codes and
 * scales the kernel computed.  out_bf16 receives the layer output unless acc is
 * given, in which case acc receives the exact int32 accumulators instead.
 */
typedef struct {
    const uint8_t *packed;
    const int8_t *centroids;
    const void *chan_scale_bf16;
    const void *x_bf16;
    const int8_t *xq;
    const float *xscale;
    int8_t *xq_out;
    float *xscale_out;
    void *out_bf16;
    int32_t *acc;
    int64_t N;
    int64_t K;
} s3d8_linear_job;

#define S3D8_MAX_BATCH 8

/*
 * Several independent S3D8 linears (the same token count M, 1 <= M <= 8) in one
 * launch: the GPU's SMs are divided among the jobs in proportion to their
 * packed bytes and every job streams its weights concurrently.  With x_bf16 the
 * activation quantisation is fused into the launch (each CTA quantises the
 * activation row(s) it needs).  This is the decode-step form of the layer: for
 * example the q, k and v projections of one token, or the seven projections of
 * a decoder layer when their inputs are available together.
 * Up to S3D8_MAX_BATCH jobs; each job's K must satisfy the s3d8_linear rules and
 * K <= 65536.  Returns S3D8_ERR_UNSUPPORTED for M > 8.
 */
int s3d8_linear_batch(const s3d8_linear_job *jobs, int count, int64_t M, void *stream);

/* Synchronises `stream`, then returns and clears the sticky device status word
 * (S3D8_OK or S3D8_ERR_TIMEOUT), or S3D8_ERR_CUDA if the synchronisation fails. */
int s3d8_device_status(void *stream);

/*
 * Failure-path self-test (no fault, no hang): launches one warp that waits on an
 * mbarrier nothing completes, for `polls` polls (1..2^24), then records
 * S3D8_ERR_TIMEOUT in the device status word exactly as the streaming kernels'
 * bounded waits do.  s3d8_device_status then returns (and clears) the timeout.
 * Covers the bounded-wait design of the kernels; the pages have no counterpart.
 */
int s3d8_selftest_wait_timeout(int64_t polls, void *stream);

/* Size of the fixed device scratch behind s3d8_linear_tc_noalloc (32 MiB). */
#define S3D8_NOALLOC_SCRATCH_BYTES (32u << 20)

/*
 * The tensor-core linear, with the same results, argument layouts and alignment
 * rules as s3d8_linear_ex with S3D8_ALGO_TC (the int32 sums are exact on both,
 * and the bf16 epilogue is the same), for callers that cannot allocate device
 * memory: code inside an allocator or memory-pool callback, a real-time loop
 * that must never wait on the driver's allocator, or a host that owns all
 * device memory itself.  It calls no cudaMalloc or cudaFree and no allocating
 * library routine.  Instead of caller workspace it uses a fixed scratch array of
 * S3D8_NOALLOC_SCRATCH_BYTES compiled into the library, which every GPU that
 * loads the library holds until the process exits.  The paper has no
 * counterpart; this is a deployment convenience.
 *   - Kernel: always the one-SM tensor-core GEMM that decodes the packed weight
 *     tiles itself (S3D8_ALGO_TC takes it below 384 tokens); it never expands
 *     the weights into scratch, so its scratch need does not grow with N.
 *   - Scratch need: the bf16 copy of the activation codes, 2 * M * K + 256
 *     bytes, plus int32 partial sums (nsplit * M * N * 4 bytes) when the output
 *     tiles cannot fill the GPU and K is split.  Shapes beyond
 *     S3D8_NOALLOC_SCRATCH_BYTES are rejected with S3D8_ERR_WORKSPACE before any
 *     launch; without a K split that is M <= 4095 at K = 4096.
 *   - The first call on a device looks up the scratch array's device address
 *     (once per device, with that device current); make that first call before
 *     any stream capture.
 *   - All calls on a device share the one array, which keeps the last call's
 *     contents (each call overwrites what it reads).  Calls that overlap on the
 *     GPU (on different streams, or from several threads without ordering) race
 *     on it and give wrong results; order them on one stream.
 * Inputs and outputs are still the caller's device memory, as in s3d8_linear.
 */
int s3d8_linear_tc_noalloc(const uint8_t *packed, const int8_t *centroids,
                           const void *chan_scale_bf16, const int8_t *xq, const float *xscale,
                           int64_t M, int64_t N, int64_t K, void *out_bf16, void *stream);

/* Static English text for a status code. */
const char *s3d8_status_string(int status);

/* Library version, major * 10000 + minor * 100 + patch. */
int s3d8_version(void);

#ifdef __cplusplus
}
#endif

#endif /* S3D8_H */
