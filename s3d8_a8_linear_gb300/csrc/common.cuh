// Shared device helpers of the S3D8 CUDA library (sm_103a).
//
// Decoding follows "11 billion parameters on a phone" (Graphcore Research
// blog), sections "Bit layout" and "Format decoding on Arm CPUs": each column
// of the 32 x 3 absolute-value centroid table is expanded over both signs into
// a 64-entry signed table (components 0 and 2 in sign-minor order, component 1
// in sign-major order), and the three lookup indices come from the byte by
//   I0 = b & 0x3F,  I1 = (b >> 1) & 0x3F,  I2 = I0 ^ (b >> 7).
// On the GPU the three lookups are folded once per CTA into one 256-entry
// table of 32-bit words [w0, w1, w2, 0] (one signed byte per output channel
// of the group), so that a packed byte costs one shared-memory load.  The
// table is replicated once per lane (word index = byte * 32 + lane), which
// makes every warp-wide lookup conflict-free whatever the byte values.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace s3d8 {

constexpr int kLutEntries = 256;
constexpr int kLutWords = kLutEntries * 32;     // lane-replicated
constexpr int kLutBytes = kLutWords * 4;        // 32 KiB
constexpr int kLutStageWords = kLutEntries;     // one unreplicated copy

__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint32_t lds_u32(uint32_t addr)
{
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}

__device__ __forceinline__ uint4 ldg_stream_v4(const void *p)
{
    // Read-only, streamed once: bypass L1 allocation.
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel)
{
    return __byte_perm(a, b, sel);
}

// Signed value of one of the blog's 64-entry tables.
//   sign-minor (components 0 and 2): index = 2 q + s
//   sign-major (component 1):        index = 32 s + q
__device__ __forceinline__ int signed_minor(const int8_t *C, int d, uint32_t idx)
{
    int c = C[(idx >> 1) * 3 + d];
    return (idx & 1) ? -c : c;
}
__device__ __forceinline__ int signed_major(const int8_t *C, int d, uint32_t idx)
{
    int c = C[(idx & 31) * 3 + d];
    return (idx >> 5) ? -c : c;
}

// Expanded table word for packed byte b: bytes 0..2 = decoded weights of
// components 0..2, byte 3 = 0.
__device__ __forceinline__ uint32_t expanded_entry(const int8_t *C, uint32_t b)
{
    const uint32_t i0 = b & 0x3Fu;
    const uint32_t i1 = (b >> 1) & 0x3Fu;
    const uint32_t i2 = i0 ^ (b >> 7);
    const int w0 = signed_minor(C, 0, i0);
    const int w1 = signed_major(C, 1, i1);
    const int w2 = signed_minor(C, 2, i2);
    return (uint32_t)(uint8_t)w0 | ((uint32_t)(uint8_t)w1 << 8) | ((uint32_t)(uint8_t)w2 << 16);
}

// Builds the lane-replicated table in shared memory.  `stage` holds 256 words.
// Every thread of the block must call it; it ends with __syncthreads().
__device__ __forceinline__ void build_lut(uint32_t *lut, uint32_t *stage, const int8_t *C_global)
{
    __shared__ int8_t Cs[96];
    for (int i = threadIdx.x; i < 96; i += blockDim.x)
        Cs[i] = C_global[i];
    __syncthreads();
    for (int b = threadIdx.x; b < kLutEntries; b += blockDim.x)
        stage[b] = expanded_entry(Cs, (uint32_t)b);
    __syncthreads();
    for (int w = threadIdx.x; w < kLutWords; w += blockDim.x)
        lut[w] = stage[w >> 5];
    __syncthreads();
}

// Four packed bytes of one group (consecutive k) -> the three per-channel
// k-quads V[d] = [w_d(k0), w_d(k1), w_d(k2), w_d(k3)], ready for dp4a / IMMA.
// `lane_base` = shared address of lut + 4 * lane.
__device__ __forceinline__ void decode_quad(uint32_t word, uint32_t lane_base, uint32_t &V0,
                                            uint32_t &V1, uint32_t &V2)
{
    const uint32_t L0 = lds_u32(lane_base + ((word & 0xFFu) << 7));
    const uint32_t L1 = lds_u32(lane_base + (((word >> 8) & 0xFFu) << 7));
    const uint32_t L2 = lds_u32(lane_base + (((word >> 16) & 0xFFu) << 7));
    const uint32_t L3 = lds_u32(lane_base + ((word >> 24) << 7));
    const uint32_t T01 = prmt(L0, L1, 0x5140);   // [w0k0 w0k1 w1k0 w1k1]
    const uint32_t T23 = prmt(L2, L3, 0x5140);   // [w0k2 w0k3 w1k2 w1k3]
    const uint32_t U01 = prmt(L0, L1, 0x0062);   // [w2k0 w2k1 . .]
    const uint32_t U23 = prmt(L2, L3, 0x0062);   // [w2k2 w2k3 . .]
    V0 = prmt(T01, T23, 0x5410);
    V1 = prmt(T01, T23, 0x7632);
    V2 = prmt(U01, U23, 0x5410);
}

__device__ __forceinline__ __nv_bfloat16 epilogue_bf16(int acc, float xs, __nv_bfloat16 cs)
{
    // (x_s * float(acc)) * W_s, rounded once to bf16 (blog, fused matrix-vector example)
    const float a = __fmul_rn(xs, __int2float_rn(acc));
    return __float2bfloat16_rn(__fmul_rn(a, __bfloat162float(cs)));
}

// ---------------------------------------------------------------------------
// Activation code q = clamp(rint(RN(x / s)), -127, 127) without a division per
// element.  With r = RN(1/s) and t = RN(x * r):
//   |t - x/s| <= |x/s| (2^-23 + 2^-48)  and  |RN(x/s) - x/s| <= |x/s| 2^-24,
// so for |x/s| <= 127.5 the two quotients differ by less than 2.3e-5.  Unless t
// lies within kTieMargin of a half-integer, rint(t) == rint(RN(x/s)); otherwise
// (and for scales below 2^-100, where 1/s could overflow) the exact IEEE
// quotient decides.  Parity with the division-based rule is tested bit for bit.
// ---------------------------------------------------------------------------
constexpr float kTieMargin = 1.0e-4f;
constexpr float kTinyScale = 7.8886090522101181e-31f;   // 2^-100

// The rare exact path, kept out of line so that the common path stays small.
static __device__ __noinline__ float exact_quotient(float x, float s)
{
    return __fdiv_rn(x, s);
}

__device__ __forceinline__ int quant_code(float x, float s, float r)
{
    if (s == 0.0f)
        return 0;
    float t = __fmul_rn(x, r);
    const float f = t - floorf(t);                         // exact for |t| < 2^23
    if (s < kTinyScale || fabsf(f - 0.5f) < kTieMargin)
        t = exact_quotient(x, s);
    return max(-127, min(127, __float2int_rn(t)));
}

// Per-lane unsigned 16-bit maximum of two packed pairs.
__device__ __forceinline__ uint32_t max_u16x2(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("max.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// Absolute maximum of the eight bf16 values of a 16-byte chunk, folded into m
// (two 16-bit lanes of bf16 bit patterns, start from 0).  With the sign bits
// cleared, the bit patterns of finite bf16 values order like their magnitudes,
// so a per-lane unsigned maximum is exact and needs no conversion to fp32.
__device__ __forceinline__ uint32_t absmax_bf16x8(uint4 v, uint32_t m)
{
    m = max_u16x2(m, v.x & 0x7FFF7FFFu);
    m = max_u16x2(m, v.y & 0x7FFF7FFFu);
    m = max_u16x2(m, v.z & 0x7FFF7FFFu);
    return max_u16x2(m, v.w & 0x7FFF7FFFu);
}

// The fp32 value of the larger of m's two lanes.
__device__ __forceinline__ float absmax_bf16x2_value(uint32_t m)
{
    return __uint_as_float(max(m >> 16, m & 0xFFFFu) << 16);
}

// Eight bf16 values (one 16-byte chunk) -> eight codes (8 bytes), for values of
// a row whose absmax a gives s = RN(a / 127).  The common path is branch-free
// over the eight values and uses only full-rate FP32 multiplies and adds:
// t = RN(x * r) is rounded to the nearest integer (ties to even) by adding
// 1.5 * 2^23, whose float encoding then holds the two's-complement code in its
// low byte.  No clamp is needed: |x| <= a, so |t| <= 127 (1 + 2^-24)^2 /
// (1 - 2^-24) < 127.5 and rint(t) is already within +-127.  t - rint(t), exact
// in fp32, flags the rare near-ties, which are redone with the exact quotient
// afterwards (quant_code, which clamps).
constexpr float kRoundMagic = 12582912.0f;   // 1.5 * 2^23
// |t - rint(t)| <= 0.5, so t lies within kTieMargin of a half-integer exactly
// when |t - rint(t)| > 0.5 - kTieMargin: one compare per value.
constexpr float kTieFloor = 0.5f - kTieMargin;

#ifdef S3D8_QUANT_NOINLINE
static __device__ __noinline__
#else
static __device__ __forceinline__
#endif
uint2 quant_chunk8(uint4 v, float s, float r)
{
    if (s == 0.0f)
        return make_uint2(0u, 0u);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    float x[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        x[2 * j] = __uint_as_float(w[j] << 16);
        x[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
    }
    uint32_t b[8];
    bool redo = s < kTinyScale;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        const float t = __fmul_rn(x[e], r);
        const float y = __fadd_rn(t, kRoundMagic);
        const float d = __fsub_rn(t, __fsub_rn(y, kRoundMagic));   // t - rint(t)
        redo |= fabsf(d) > kTieFloor;
        b[e] = __float_as_uint(y);
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

__device__ __forceinline__ int warp_sum(int v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}


// ---------------------------------------------------------------------------
// Wide-stride table for the streaming kernels: entry b of lane l sits at
// lut_win + 256 b + 4 l, with lut_win a multiple of 64 KiB in the shared
// window.  A single PRMT then forms the lookup address: byte 0 from the lane
// offset, byte 1 = the packed byte, bytes 2..3 from lut_win.
// ---------------------------------------------------------------------------
constexpr uint32_t kWideLutBytes = 0x10000;

__device__ __forceinline__ uint32_t wide_lut_window(uint32_t dyn_base)
{
    return (dyn_base + 0xFFFFu) & ~0xFFFFu;
}

// Fills the wide table (all threads of the block; ends with __syncthreads()).
__device__ __forceinline__ void build_wide_lut(unsigned char *lut_ptr, uint32_t *stage,
                                               const int8_t *C_global)
{
    __shared__ int8_t Cw[96];
    for (int i = threadIdx.x; i < 96; i += blockDim.x)
        Cw[i] = C_global[i];
    __syncthreads();
    for (int b = threadIdx.x; b < kLutEntries; b += blockDim.x)
        stage[b] = expanded_entry(Cw, (uint32_t)b);
    __syncthreads();
    uint32_t *w = reinterpret_cast<uint32_t *>(lut_ptr);
    for (int i = threadIdx.x; i < kLutEntries * 32; i += blockDim.x)
        w[(i >> 5) * 64 + (i & 31)] = stage[i >> 5];
    __syncthreads();
}

// As build_wide_lut, with the 96 table bytes already loaded: thread t < 96
// passes C[t] in `cval`.
__device__ __forceinline__ void build_wide_lut_from(unsigned char *lut_ptr, uint32_t *stage, int8_t cval)
{
    __shared__ int8_t Cv[96];
    if (threadIdx.x < 96)
        Cv[threadIdx.x] = cval;
    __syncthreads();
    for (int b = threadIdx.x; b < kLutEntries; b += blockDim.x)
        stage[b] = expanded_entry(Cv, (uint32_t)b);
    __syncthreads();
    uint32_t *w = reinterpret_cast<uint32_t *>(lut_ptr);
    for (int i = threadIdx.x; i < kLutEntries * 32; i += blockDim.x)
        w[(i >> 5) * 64 + (i & 31)] = stage[i >> 5];
    __syncthreads();
}

__device__ __forceinline__ uint32_t lds_u32_nv(uint32_t addr)
{
    uint32_t v;
    asm("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}

__device__ __forceinline__ uint32_t mad_lo_u32(uint32_t a, uint32_t b, uint32_t c)
{
    uint32_t d;
    asm("mad.lo.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// As decode_quad, against the wide table (`lane_base` = lut_win | 4 lane).
// The third channel is merged on the FMA pipe (U01 + U23 * 2^16; both halves
// are zero-padded because byte 3 of every table entry is 0).
__device__ __forceinline__ void decode_quad_wide(uint32_t word, uint32_t lane_base, uint32_t &V0,
                                                 uint32_t &V1, uint32_t &V2)
{
    const uint32_t L0 = lds_u32_nv(prmt(word, lane_base, 0x7604));
    const uint32_t L1 = lds_u32_nv(prmt(word, lane_base, 0x7614));
    const uint32_t L2 = lds_u32_nv(prmt(word, lane_base, 0x7624));
    const uint32_t L3 = lds_u32_nv(prmt(word, lane_base, 0x7634));
    const uint32_t T01 = prmt(L0, L1, 0x5140);   // [w0k0 w0k1 w1k0 w1k1]
    const uint32_t T23 = prmt(L2, L3, 0x5140);
    const uint32_t U01 = prmt(L0, L1, 0x3362);   // [w2k0 w2k1 0 0]
    const uint32_t U23 = prmt(L2, L3, 0x3362);
    V0 = prmt(T01, T23, 0x5410);
    V1 = prmt(T01, T23, 0x7632);
    V2 = mad_lo_u32(U23, 65536u, U01);
}

// Sum over the warp of P values per lane (P a power of two, 2..32), returned
// transposed: afterwards every lane of group j (lanes j * 32/P .. +32/P - 1)
// holds the full sum of value j.  Costs P - 1 + log2(32/P) shuffles.
template <int P>
__device__ __forceinline__ int warp_reduce_transposed(int (&v)[P], int lane)
{
#pragma unroll
    for (int n = P, o = 16; n > 1; n >>= 1, o >>= 1) {
        const bool upper = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < n / 2; ++i) {
            const int keep = upper ? v[i + n / 2] : v[i];
            const int send = upper ? v[i] : v[i + n / 2];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
    }
    int r = v[0];
#pragma unroll
    for (int o = 16 / P; o > 0; o >>= 1)
        r += __shfl_xor_sync(0xffffffffu, r, o);
    return r;
}

}  // namespace s3d8
