// Activation quantisation and the standalone S3D8 -> INT8 unpack.
#include "common.cuh"
#include "launch.h"

namespace s3d8 {

// Two fp32 lanes in one 64-bit register, and the packed fp32 operations on
// them: mul.rn / add.rn / sub.rn .f32x2 round each lane exactly as the scalar
// instruction does (no flush to zero), at one issue slot per two values.
__device__ __forceinline__ uint64_t f32x2_pack(float lo, float hi)
{
    uint64_t d;
    asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(lo), "f"(hi));
    return d;
}
__device__ __forceinline__ void f32x2_unpack(uint64_t v, float &lo, float &hi)
{
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f32x2_mul(uint64_t a, uint64_t b)
{
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f32x2_add(uint64_t a, uint64_t b)
{
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f32x2_sub(uint64_t a, uint64_t b)
{
    uint64_t d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// As quant_chunk8, with the multiply and the two rounding steps on value pairs
// (f32x2): the same result bit for bit, in fewer issue slots.  The standalone
// quantisation kernels use it (measured 26.5 -> 25.6 us on bf16 [2048, 14336]);
// the GEMV's fused prologue keeps the scalar form, which measured 1% faster
// there.
static __device__ __forceinline__
uint2 quant_chunk8_x2(uint4 v, float s, float r)
{
    if (s == 0.0f)
        return make_uint2(0u, 0u);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    const uint64_t r2 = f32x2_pack(r, r), m2 = f32x2_pack(kRoundMagic, kRoundMagic);
    float x[8];
    uint32_t b[8];
    bool redo = s < kTinyScale;
#pragma unroll
    for (int j = 0; j < 4; ++j) {   // values 2j and 2j + 1 (the two halves of word j) as one pair
        x[2 * j] = __uint_as_float(w[j] << 16);
        x[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
        const uint64_t t2 = f32x2_mul(f32x2_pack(x[2 * j], x[2 * j + 1]), r2);
        const uint64_t y2 = f32x2_add(t2, m2);
        const uint64_t d2 = f32x2_sub(t2, f32x2_sub(y2, m2));   // t - rint(t), per lane
        float d0, d1, y0, y1;
        f32x2_unpack(d2, d0, d1);
        f32x2_unpack(y2, y0, y1);
        redo |= fabsf(d0) > kTieFloor;
        redo |= fabsf(d1) > kTieFloor;
        b[2 * j] = __float_as_uint(y0);
        b[2 * j + 1] = __float_as_uint(y1);
    }
    if (redo) {
#pragma unroll
        for (int e = 0; e < 8; ++e)
            b[e] = (uint32_t)quant_code(x[e], s, r);
    }
    const uint32_t lo = prmt(prmt(b[0], b[1], 0x0040), prmt(b[2], b[3], 0x0040), 0x5410);
    const uint32_t hi = prmt(prmt(b[4], b[5], 0x0040), prmt(b[6], b[7], 0x0040), 0x5410);
    return make_uint2(lo, hi);
}


// ---------------------------------------------------------------------------
// Per-token absmax INT8 quantisation.  Rows of more than 16384 columns: one CTA
// per row (grid-stride over rows), 16-byte vector loads, two passes over the row
// (the second hits L1/L2).  Shorter rows: quantize_act_rows_kernel below.
// xscale = absmax / 127 with IEEE division; q = rint(x / xscale), ties to even,
// clamped to +-127 (quant_code: one multiply by RN(1/xscale), exact division
// only near ties); a zero row gives scale 0 and codes 0.
// ---------------------------------------------------------------------------
constexpr int kQuantThreads = 256;

__global__ __launch_bounds__(kQuantThreads) void quantize_act_kernel(
    const __nv_bfloat16 *__restrict__ x, int M, int K, int8_t *__restrict__ xq,
    float *__restrict__ xscale)
{
    __shared__ float red[kQuantThreads / 32];
    const int chunks = K / 8;  // 8 bf16 per 16 bytes; K % 16 == 0
    for (int m = blockIdx.x; m < M; m += gridDim.x) {
        const uint4 *row = reinterpret_cast<const uint4 *>(x + (size_t)m * K);
        uint32_t m2 = 0u;
        for (int c = threadIdx.x; c < chunks; c += kQuantThreads)
            m2 = absmax_bf16x8(__ldg(row + c), m2);
        float amax = absmax_bf16x2_value(m2);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        if ((threadIdx.x & 31) == 0)
            red[threadIdx.x >> 5] = amax;
        __syncthreads();
        amax = red[0];
#pragma unroll
        for (int i = 1; i < kQuantThreads / 32; ++i)
            amax = fmaxf(amax, red[i]);
        __syncthreads();  // red is reused by the next row
        const float s = __fdiv_rn(amax, 127.0f);
        const float r = s > 0.0f ? __frcp_rn(s) : 0.0f;
        if (threadIdx.x == 0)
            xscale[m] = s;
        uint2 *qrow = reinterpret_cast<uint2 *>(xq + (size_t)m * K);
        for (int c = threadIdx.x; c < chunks; c += kQuantThreads) {
            const uint4 v = __ldg(row + c);
            qrow[c] = quant_chunk8_x2(v, s, r);
        }
    }
}

// Rows of at most NS * kQuantThreads 16-byte chunks (K <= 2048 NS): one CTA per
// row, the whole row held in registers.  Every load of a thread leaves before
// the first is used, so a row costs one memory latency, and the block scheduler
// deals rows to SMs as they free up (no grid-stride tail).  Same arithmetic as
// quantize_act_kernel.
template <int NS>
__global__ __launch_bounds__(kQuantThreads) void quantize_act_rows_kernel(
    const __nv_bfloat16 *__restrict__ x, int K, int8_t *__restrict__ xq, float *__restrict__ xscale)
{
    __shared__ float red[kQuantThreads / 32];
    const int chunks = K / 8;
    const size_t m = blockIdx.x;
    const uint4 *row = reinterpret_cast<const uint4 *>(x + m * K);
    uint4 v[NS];
#pragma unroll
    for (int i = 0; i < NS; ++i) {
        const int c = threadIdx.x + i * kQuantThreads;
        v[i] = c < chunks ? ldg_stream_v4(row + c) : make_uint4(0u, 0u, 0u, 0u);
    }
    uint32_t m2 = 0u;
#pragma unroll
    for (int i = 0; i < NS; ++i)
        m2 = absmax_bf16x8(v[i], m2);
    float amax = absmax_bf16x2_value(m2);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if ((threadIdx.x & 31) == 0)
        red[threadIdx.x >> 5] = amax;
    __syncthreads();
    amax = red[0];
#pragma unroll
    for (int i = 1; i < kQuantThreads / 32; ++i)
        amax = fmaxf(amax, red[i]);
    const float s = __fdiv_rn(amax, 127.0f);
    const float r = s > 0.0f ? __frcp_rn(s) : 0.0f;
    if (threadIdx.x == 0)
        xscale[m] = s;
    uint2 *qrow = reinterpret_cast<uint2 *>(xq + m * K);
#pragma unroll
    for (int i = 0; i < NS; ++i) {
        const int c = threadIdx.x + i * kQuantThreads;
        if (c < chunks)
            qrow[c] = quant_chunk8_x2(v[i], s, r);
    }
}

cudaError_t launch_quantize_act(const __nv_bfloat16 *x, int M, int K, int8_t *xq, float *xscale,
                                cudaStream_t stream)
{
    const int chunks = K / 8;
    if (chunks <= kQuantThreads)
        quantize_act_rows_kernel<1><<<M, kQuantThreads, 0, stream>>>(x, K, xq, xscale);
    else if (chunks <= 2 * kQuantThreads)
        quantize_act_rows_kernel<2><<<M, kQuantThreads, 0, stream>>>(x, K, xq, xscale);
    else if (chunks <= 4 * kQuantThreads)
        quantize_act_rows_kernel<4><<<M, kQuantThreads, 0, stream>>>(x, K, xq, xscale);
    else if (chunks <= 8 * kQuantThreads)
        quantize_act_rows_kernel<8><<<M, kQuantThreads, 0, stream>>>(x, K, xq, xscale);
    else {
        const int grid = M < device_sm_count() * 8 ? M : device_sm_count() * 8;
        quantize_act_kernel<<<grid, kQuantThreads, 0, stream>>>(x, M, K, xq, xscale);
    }
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Standalone unpack: packed[G, K] -> w[N, K] int8.  Each thread takes one
// 16-byte chunk of a packed row, looks every byte up once in the expanded
// table and writes 16 bytes to each of the (up to) three output rows.
// Persistent grid so that the 32 KiB table build is amortised.
// ---------------------------------------------------------------------------
constexpr int kDecodeThreads = 256;

__global__ __launch_bounds__(kDecodeThreads) void decode_kernel(const uint8_t *__restrict__ packed,
                                                                const int8_t *__restrict__ C,
                                                                int N, int K,
                                                                int8_t *__restrict__ w)
{
    extern __shared__ __align__(16) unsigned char smem[];
    uint32_t *lut = reinterpret_cast<uint32_t *>(smem);
    uint32_t *stage = lut + kLutWords;
    build_lut(lut, stage, C);
    const uint32_t lane_base = smem_addr(lut) + 4u * (threadIdx.x & 31);
    const int G = (N + 2) / 3;
    const int chunks_per_row = K / 16;
    const long long total = (long long)G * chunks_per_row;
    for (long long i = (long long)blockIdx.x * kDecodeThreads + threadIdx.x; i < total;
         i += (long long)gridDim.x * kDecodeThreads) {
        const int g = (int)(i / chunks_per_row);
        const int k = (int)(i % chunks_per_row) * 16;
        const uint4 p = ldg_stream_v4(packed + (size_t)g * K + k);
        uint32_t V[3][4];
        decode_quad(p.x, lane_base, V[0][0], V[1][0], V[2][0]);
        decode_quad(p.y, lane_base, V[0][1], V[1][1], V[2][1]);
        decode_quad(p.z, lane_base, V[0][2], V[1][2], V[2][2]);
        decode_quad(p.w, lane_base, V[0][3], V[1][3], V[2][3]);
#pragma unroll
        for (int d = 0; d < 3; ++d) {
            const int n = 3 * g + d;
            if (n < N)
                *reinterpret_cast<uint4 *>(w + (size_t)n * K + k) =
                    make_uint4(V[d][0], V[d][1], V[d][2], V[d][3]);
        }
    }
}

cudaError_t launch_decode(const uint8_t *packed, const int8_t *C, int N, int K, int8_t *w,
                          cudaStream_t stream)
{
    const size_t smem = (size_t)(kLutWords + kLutStageWords) * 4;
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(decode_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess)
            return e;
        attr_set = true;
    }
    const long long G = (N + 2) / 3;
    const long long work = G * (K / 16);
    long long grid = (work + kDecodeThreads - 1) / kDecodeThreads;
    const long long cap = (long long)device_sm_count() * 4;
    if (grid > cap)
        grid = cap;
    decode_kernel<<<(int)grid, kDecodeThreads, smem, stream>>>(packed, C, N, K, w);
    return cudaGetLastError();
}

}  // namespace s3d8
