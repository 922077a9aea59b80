// Direct-cast encoder: bf16 weights W[N, K] and a fixed 32 x 3 centroid table
// -> per-channel bf16 scales and packed S3D8 bytes [ceil(N/3), K].
//
// Llama-Mobile: Efficient 2.7-Bit Quantization of VLMs, section 3.4
// "Quantization" (the forward assignment with frozen centroids):
//   alpha_n = max_k |W[n,k]| / 127                      -> stored as bf16
//   W'      = |W| / alpha (the stored alpha), per 3-vector of channels 3g..3g+2
//   s       = + where W >= 0, - elsewhere
//   q       = the nearest centroid to W' in L2, the lowest index on a tie.
// The byte follows "11 billion parameters on a phone" (Graphcore Research
// blog), section "Bit layout": bit 0 = S0, bits 1..5 = Q, bit 6 = S1,
// bit 7 = S2 xor S0.
//
// Every decision is taken in fp32 with IEEE rounding and no contraction: the
// division, then t_d = C_d - W'_d, then ((t0 t0 + t1 t1) + t2 t2), compared
// with "<" in index order.  Padded channels (3g + d >= N) enter as W'_d = 0
// with a + selector; a channel whose alpha is 0 gives W' = 0.
#include "common.cuh"
#include "launch.h"

namespace s3d8 {

// ---------------------------------------------------------------------------
// Channel scales.  One warp per row (stride over the row CTAs), 16-byte loads, four in
// flight per lane.  For finite bf16 values |a| <= |b| exactly when the low
// 15 bits compare that way, so the row maximum is a packed 16-bit integer max
// of the masked words; it is converted back to fp32 once per row.
// ---------------------------------------------------------------------------
constexpr int kScaleThreads = 256;

// Packed per-half maximum of |x| (as 15-bit magnitudes) over 8 bf16 values.
__device__ __forceinline__ uint32_t absmax_word(const uint4 v)
{
    const uint32_t a = __vmaxu2(v.x & 0x7FFF7FFFu, v.y & 0x7FFF7FFFu);
    const uint32_t b = __vmaxu2(v.z & 0x7FFF7FFFu, v.w & 0x7FFF7FFFu);
    return __vmaxu2(a, b);
}
constexpr int kScaleRowsPerCta = kScaleThreads / 32;

__device__ __forceinline__ void scale_rows(const __nv_bfloat16 *__restrict__ w, int N, int K,
                                           int ctas, __nv_bfloat16 *__restrict__ chan_scale)
{
    const int lane = threadIdx.x & 31;
    const int chunks = K / 8;
    for (int n = blockIdx.x * kScaleRowsPerCta + (threadIdx.x >> 5); n < N;
         n += ctas * kScaleRowsPerCta) {
        const uint4 *row = reinterpret_cast<const uint4 *>(w + (size_t)n * K);
        uint32_t m = 0;
        int c = lane;
        for (; c + 96 < chunks; c += 128) {
            const uint4 v0 = __ldg(row + c), v1 = __ldg(row + c + 32);
            const uint4 v2 = __ldg(row + c + 64), v3 = __ldg(row + c + 96);
            m = __vmaxu2(m, absmax_word(v0));
            m = __vmaxu2(m, absmax_word(v1));
            m = __vmaxu2(m, absmax_word(v2));
            m = __vmaxu2(m, absmax_word(v3));
        }
        for (; c < chunks; c += 32)
            m = __vmaxu2(m, absmax_word(__ldg(row + c)));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            m = __vmaxu2(m, __shfl_xor_sync(0xffffffffu, m, o));
        if (lane == 0) {
            const uint32_t hi = m >> 16, lo = m & 0xFFFFu;
            const float amax = __uint_as_float((hi > lo ? hi : lo) << 16);
            chan_scale[n] = __float2bfloat16_rn(__fdiv_rn(amax, 127.0f));
        }
    }
}

// ---------------------------------------------------------------------------
// Candidate masks.  The cube [0, 128)^3 of scaled magnitudes W' is cut into
// 16^3 cells of side 8, indexed i0 + 16 i1 + 256 i2 with i_d = floor(W'_d / 8).
// Bit l of a cell's mask is cleared when some centroid j is nearer than l by
// more than a margin of 1 everywhere in the closed cell.  D_l(x) - D_j(x) =
// |C_l|^2 - |C_j|^2 - 2 x.(C_l - C_j) is linear in x, so its minimum over the
// box is at a corner: each axis takes lo or hi, whichever gives the larger
// x_d (C_l - C_j)_d.  All of these are integers below 2^24 (corners are
// multiples of 8 up to 128, centroids 0..127), exact in fp32.  The fp32 value
// of a point's squared distance differs from the real one by less than 0.025
// (relative error below 6 units of 2^-24 on values below 2^16), so a centroid
// that can be the fp32 minimum anywhere in the cell, ties included, keeps its
// bit; the centroid nearest to any point of the cell always does.
// One warp per cell, lane l testing centroid l against all j; a ballot forms
// the mask.
// ---------------------------------------------------------------------------
constexpr int kCellBits = 4;
constexpr int kCells = 1 << (3 * kCellBits);   // 4096
constexpr float kCellSide = 8.0f;

// ctab[l] = (C_l0, C_l1, C_l2, |C_l|^2)
__device__ __forceinline__ uint32_t cell_mask(const float4 *ctab, int cell, int lane)
{
    float lo[3], hi[3];
#pragma unroll
    for (int d = 0; d < 3; ++d) {
        lo[d] = kCellSide * (float)((cell >> (kCellBits * d)) & ((1 << kCellBits) - 1));
        hi[d] = lo[d] + kCellSide;
    }
    const float4 me = ctab[lane];
    bool keep = true;
    for (int j = 0; j < 32; ++j) {
        const float4 o = ctab[j];
        const float d0 = me.x - o.x, d1 = me.y - o.y, d2 = me.z - o.z;
        const float mx = fmaxf(lo[0] * d0, hi[0] * d0) + fmaxf(lo[1] * d1, hi[1] * d1) +
                         fmaxf(lo[2] * d2, hi[2] * d2);
        const float mn = (me.w - o.w) - 2.0f * mx;
        keep = keep && !(mn > 1.0f);
    }
    return __ballot_sync(0xFFFFFFFFu, keep);
}

// The channel-scale kernel's trailing CTAs build the masks, one cell per warp.
constexpr int kMaskCtas = kCells / (kScaleThreads / 32);

__global__ __launch_bounds__(kScaleThreads) void encode_prepare_kernel(
    const __nv_bfloat16 *__restrict__ w, const int8_t *__restrict__ C, int N, int K,
    int row_ctas, __nv_bfloat16 *__restrict__ chan_scale, uint32_t *__restrict__ masks)
{
    if ((int)blockIdx.x >= row_ctas) {
        __shared__ float4 ctab[32];
        if (threadIdx.x < 32) {
            const float c0 = (float)C[3 * threadIdx.x], c1 = (float)C[3 * threadIdx.x + 1];
            const float c2 = (float)C[3 * threadIdx.x + 2];
            ctab[threadIdx.x] = make_float4(c0, c1, c2, c0 * c0 + c1 * c1 + c2 * c2);
        }
        __syncthreads();
        const int cell = ((int)blockIdx.x - row_ctas) * (kScaleThreads / 32) + (threadIdx.x >> 5);
        const uint32_t m = cell_mask(ctab, cell, threadIdx.x & 31);
        if ((threadIdx.x & 31) == 0)
            masks[cell] = m;
        return;
    }
    scale_rows(w, N, K, row_ctas, chan_scale);
}

// ---------------------------------------------------------------------------
// Scaled magnitude q = RN(a / alpha) for a = |x| >= 0.  With r = RN(1/alpha)
// computed once per channel, q0 = RN(a r) is within one unit in the last place
// of a / alpha, the remainder a - alpha q0 is then exact in one fused
// multiply-add, and RN(q0 + rem r) is the correctly rounded quotient
// (P. Markstein, "Computation of elementary functions on the IBM RISC
// System/6000 processor", IBM J. Res. Dev. 34(1), 1990, the division theorem).
// The argument needs every intermediate far from underflow and overflow: the
// fast path runs for alpha in [2^-50, 2^50] and a = 0 or a >= alpha 2^-30,
// with a <= 2^20 alpha (the encoder meets a <= 128 alpha: alpha is the row's
// absmax / 127 rounded to bf16).  A nonzero a below alpha 2^-30, or any
// nonzero a when alpha is outside the range, takes the IEEE division.
// alpha = 0 gives 0.  The test "a is 0 or a >= lo" is one unsigned compare
// of (bits(a) - 1) against lo_m1 = bits(lo) - 1.
// ---------------------------------------------------------------------------
struct ChanDiv {
    float alpha, r;
    uint32_t lo_m1;
};

__device__ __forceinline__ ChanDiv chan_div(float alpha)
{
    ChanDiv c;
    c.alpha = alpha;
    if (alpha == 0.0f) {
        c.r = 0.0f;                  // q0 = 0, rem = a, q = 0 for every finite a
        c.lo_m1 = 0u;
    } else if (alpha >= 0x1p-50f && alpha <= 0x1p50f) {
        c.r = __frcp_rn(alpha);
        c.lo_m1 = __float_as_uint(alpha * 0x1p-30f) - 1u;   // exact power-of-two scaling
    } else {
        c.r = 0.0f;                  // a = 0 still gives 0 on the fast path
        c.lo_m1 = 0xFFFFFFFFu;
    }
    return c;
}

__device__ __forceinline__ float scaled_abs_fast(float a, const ChanDiv &c)
{
    const float q0 = __fmul_rn(a, c.r);
    const float rem = __fmaf_rn(-q0, c.alpha, a);
    return __fmaf_rn(rem, c.r, q0);
}

__device__ __forceinline__ bool needs_ieee_div(float a, const ChanDiv &c)
{
    return __float_as_uint(a) - 1u < c.lo_m1;
}

__device__ __forceinline__ float scaled_abs(float a, const ChanDiv &c)
{
    return needs_ieee_div(a, c) ? __fdiv_rn(a, c.alpha) : scaled_abs_fast(a, c);
}

__global__ void selftest_scaled_abs_kernel(const __nv_bfloat16 *__restrict__ x,
                                           const __nv_bfloat16 *__restrict__ alpha, int64_t n,
                                           float *__restrict__ out)
{
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x)
        out[i] = scaled_abs(fabsf(__bfloat162float(x[i])), chan_div(__bfloat162float(alpha[i])));
}

cudaError_t launch_selftest_scaled_abs(const __nv_bfloat16 *x, const __nv_bfloat16 *alpha,
                                       int64_t n, float *out, cudaStream_t stream)
{
    const int64_t want = (n + 255) / 256;
    const int grid = (int)(want < 4096 ? want : 4096);
    selftest_scaled_abs_kernel<<<grid, 256, 0, stream>>>(x, alpha, n, out);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Assignment.  Persistent CTAs; a thread takes one packed row g and 8
// consecutive k per item: three 16-byte loads (rows 3g, 3g+1, 3g+2), 8 output
// bytes.  Per code, the cell's mask from shared memory lists the candidates.
// The warp walks them in lockstep for as many steps as its largest candidate
// count: at each step a lane takes its highest remaining index l (as
// c = clz(mask) = 31 - l) and clears it; a lane with none left gets c = 32.
// The table is stored by c (entry c = centroid 31 - c) with a far-away dummy
// at c = 32, so that lane's distance is +inf and never wins.  A centroid
// whose distance is <= the best so far replaces it; walking indices downward,
// that leaves the lowest index among equal distances, the answer of a 0..31
// scan with a strict "<".
// The table is stored eight times, entry c of copy j at float4 8 c + j, and
// lane t reads copy t mod 8: the eight lanes of a 128-bit access phase then
// touch distinct bank groups whatever entries they want.
// Finite inputs give W' <= 127.25 (alpha >= absmax/127 (1 - 2^-9)), inside the
// cell grid; the cell index is masked to 12 bits in any case.
// ---------------------------------------------------------------------------
constexpr int kEncodeThreads = 256;
constexpr int kEncodeCtasPerSm = 4;
constexpr int kTabEntries = 33;

__device__ __forceinline__ float dist2(const float4 c, float w0, float w1, float w2)
{
    const float t0 = __fsub_rn(c.x, w0);
    const float t1 = __fsub_rn(c.y, w1);
    const float t2 = __fsub_rn(c.z, w2);
    return __fadd_rn(__fadd_rn(__fmul_rn(t0, t0), __fmul_rn(t1, t1)), __fmul_rn(t2, t2));
}

// floor(v / 8) + 2^23 for 0 <= v < 2^26, rounded toward -inf in one fused
// multiply-add (v / 8 is exact); the low 4 bits are the cell coordinate.
__device__ __forceinline__ uint32_t cell_coord(float v)
{
    return __float_as_uint(__fmaf_rd(v, 0.125f, 8388608.0f)) & 15u;
}

// |x| of element e (0..7) of an 8-element bf16 chunk held as 4 words, in fp32.
__device__ __forceinline__ float elem_abs(const uint32_t (&u)[4], int e)
{
    const uint32_t word = u[e >> 1];
    return __uint_as_float(((e & 1) ? (word & 0xFFFF0000u) : (word << 16)) & 0x7FFFFFFFu);
}

// Negative-selector flags of the two bf16 in a word, at bits 15 and 31: the
// sign bit, unless the magnitude is 0 (-0 takes the + selector).
__device__ __forceinline__ uint32_t neg_flags(uint32_t u)
{
    const uint32_t nz = (u & 0x7FFF7FFFu) + 0x7FFF7FFFu;  // bit 15 / 31 set iff magnitude != 0
    return u & nz & 0x80008000u;
}

// DENSE = false writes the packed bytes; DENSE = true writes the fake-quant
// reconstruction w_hat[n, k] = bf16_rn(s alpha_n C[q][n mod 3]) instead (the
// product of a bf16 alpha and an integer below 128 is exact in fp32).
template <bool DENSE>
__global__ __launch_bounds__(kEncodeThreads, DENSE ? kEncodeCtasPerSm - 1 : kEncodeCtasPerSm) void
encode_assign_kernel(
    const __nv_bfloat16 *__restrict__ w, const int8_t *__restrict__ C,
    const __nv_bfloat16 *__restrict__ chan_scale, const uint32_t *__restrict__ masks_g, int N,
    int K, int G, uint8_t *__restrict__ packed, __nv_bfloat16 *__restrict__ w_hat)
{
    __shared__ __align__(16) uint32_t masks[kCells];
    __shared__ float4 tab[kTabEntries * 8];
    for (int i = threadIdx.x; i < kCells / 4; i += kEncodeThreads)
        reinterpret_cast<uint4 *>(masks)[i] = __ldg(reinterpret_cast<const uint4 *>(masks_g) + i);
    for (int i = threadIdx.x; i < kTabEntries * 8; i += kEncodeThreads) {
        const int c = i >> 3;
        tab[i] = c < 32 ? make_float4((float)C[3 * (31 - c)], (float)C[3 * (31 - c) + 1],
                                      (float)C[3 * (31 - c) + 2], 0.0f)
                        : make_float4(1.0e30f, 1.0e30f, 1.0e30f, 0.0f);
    }
    __syncthreads();
    const float4 *mytab = tab + (threadIdx.x & 7);

    const int chunks = K / 8;
    const int64_t items = (int64_t)G * chunks;
    // The loop runs per warp (the walk below is a warp collective); lanes past
    // the end work on zeros and store nothing.
    for (int64_t base = (int64_t)blockIdx.x * kEncodeThreads + (threadIdx.x & ~31); base < items;
         base += (int64_t)gridDim.x * kEncodeThreads) {
        const int64_t it = base + (threadIdx.x & 31);
        const bool live = it < items;
        const int g = live ? (int)(it / chunks) : 0;
        const int c = live ? (int)(it - (int64_t)g * chunks) : 0;
        uint32_t u[3][4];
        ChanDiv dv[3];
#pragma unroll
        for (int d = 0; d < 3; ++d) {
            const int n = 3 * g + d;
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            float alpha = 0.0f;
            if (live && n < N) {
                v = __ldg(reinterpret_cast<const uint4 *>(w + (size_t)n * K) + c);
                alpha = __bfloat162float(chan_scale[n]);
            }
            u[d][0] = v.x;
            u[d][1] = v.y;
            u[d][2] = v.z;
            u[d][3] = v.w;
            dv[d] = chan_div(alpha);
        }
        // selectors: byte e of out[e / 4] gets S0 at bit 0, S1 at bit 6 and
        // S2 xor S0 at bit 7; the flags of codes 4o..4o+3 sit at bits 15 and 31
        // of words 2o and 2o+1, gathered to bit 7 of each byte by one permute
        uint32_t out[2];
        uint32_t hat[3][4] = {{0u, 0u, 0u, 0u}, {0u, 0u, 0u, 0u}, {0u, 0u, 0u, 0u}};
#pragma unroll
        for (int o = 0; o < 2; ++o) {
            const uint32_t f0 = __byte_perm(neg_flags(u[0][2 * o]), neg_flags(u[0][2 * o + 1]), 0x7531);
            const uint32_t f1 = __byte_perm(neg_flags(u[1][2 * o]), neg_flags(u[1][2 * o + 1]), 0x7531);
            const uint32_t f2 = __byte_perm(neg_flags(u[2][2 * o]), neg_flags(u[2][2 * o + 1]), 0x7531);
            out[o] = (f0 >> 7) | (f1 >> 1) | (f2 ^ f0);
        }
        // Two halves of 4 codes: the 12 scaled magnitudes of a half, then its
        // walks.  One branch per half sends the (never seen in practice)
        // elements outside the fast division's range to the IEEE division.
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            float wp[3][4];
            bool slow = false;
#pragma unroll
            for (int d = 0; d < 3; ++d)
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    slow |= needs_ieee_div(elem_abs(u[d], 4 * h + e), dv[d]);
            if (slow) {
#pragma unroll
                for (int d = 0; d < 3; ++d)
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        wp[d][e] = scaled_abs(elem_abs(u[d], 4 * h + e), dv[d]);
            } else {
#pragma unroll
                for (int d = 0; d < 3; ++d)
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        wp[d][e] = scaled_abs_fast(elem_abs(u[d], 4 * h + e), dv[d]);
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float w0 = wp[0][e], w1 = wp[1][e], w2 = wp[2][e];
                const uint32_t cell = cell_coord(w0) + 16u * cell_coord(w1) + 256u * cell_coord(w2);
                uint32_t cand = masks[cell];
                const uint32_t steps = __reduce_max_sync(0xFFFFFFFFu, (uint32_t)__popc(cand));
                float bestd = 3.0e38f;
                uint32_t best = 31;   // centroid 0 if nothing compares (only NaN inputs)
                // two candidates per trip; a lane with none left reads the dummy
                for (uint32_t i = 0; i < steps; i += 2) {
                    const uint32_t k0 = __clz(cand);                 // 32 when none is left
                    cand ^= __funnelshift_rc(0x80000000u, 0u, k0);   // clears it; 0 for k = 32
                    const uint32_t k1 = __clz(cand);
                    cand ^= __funnelshift_rc(0x80000000u, 0u, k1);
                    const float d0 = dist2(mytab[8 * k0], w0, w1, w2);
                    const float d1 = dist2(mytab[8 * k1], w0, w1, w2);
                    if (d0 <= bestd) {
                        bestd = d0;
                        best = k0;
                    }
                    if (d1 <= bestd) {
                        bestd = d1;
                        best = k1;
                    }
                }
                out[h] += (31u - best) << (1 + 8 * e);
                if (DENSE) {
                    const float4 cq = mytab[8 * best];
                    const float cd[3] = {cq.x, cq.y, cq.z};
#pragma unroll
                    for (int d = 0; d < 3; ++d) {
                        const uint32_t word = u[d][(4 * h + e) >> 1];
                        const bool neg = neg_flags(word) & (((4 * h + e) & 1) ? 0x80000000u : 0x8000u);
                        // the decoded weight is an integer: a zero table entry is
                        // +0 whatever the selector (-0 + 0 = +0)
                        const float wq = __fadd_rn(neg ? -cd[d] : cd[d], 0.0f);
                        const float v = __fmul_rn(dv[d].alpha, wq);
                        const uint32_t b = __bfloat16_as_ushort(__float2bfloat16_rn(v));
                        hat[d][(4 * h + e) >> 1] |= ((4 * h + e) & 1) ? (b << 16) : b;
                    }
                }
            }
        }
        if (!DENSE && live)
            reinterpret_cast<uint2 *>(packed + (size_t)g * K)[c] = make_uint2(out[0], out[1]);
        if (DENSE && live) {
#pragma unroll
            for (int d = 0; d < 3; ++d)
                if (3 * g + d < N)
                    reinterpret_cast<uint4 *>(w_hat + (size_t)(3 * g + d) * K)[c] =
                        make_uint4(hat[d][0], hat[d][1], hat[d][2], hat[d][3]);
        }
    }
}

static cudaError_t launch_encode_impl(const __nv_bfloat16 *w, const int8_t *C, int N, int K,
                                      uint8_t *packed, __nv_bfloat16 *w_hat,
                                      __nv_bfloat16 *chan_scale, void *workspace,
                                      cudaStream_t stream)
{
    const int sms = device_sm_count();
    uint32_t *masks = static_cast<uint32_t *>(workspace);
    const int rows_ctas = (N + kScaleRowsPerCta - 1) / kScaleRowsPerCta;
    const int g1 = rows_ctas < sms * 8 ? rows_ctas : sms * 8;
    encode_prepare_kernel<<<g1 + kMaskCtas, kScaleThreads, 0, stream>>>(w, C, N, K, g1, chan_scale,
                                                                         masks);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return e;
    const int G = (N + 2) / 3;
    const int64_t items = (int64_t)G * (K / 8);
    const int64_t want = (items + kEncodeThreads - 1) / kEncodeThreads;
    const int64_t cap = (int64_t)sms * (w_hat ? kEncodeCtasPerSm - 1 : kEncodeCtasPerSm);
    const int g2 = (int)(want < cap ? want : cap);
    if (w_hat)
        encode_assign_kernel<true><<<g2, kEncodeThreads, 0, stream>>>(w, C, chan_scale, masks, N, K,
                                                                      G, nullptr, w_hat);
    else
        encode_assign_kernel<false><<<g2, kEncodeThreads, 0, stream>>>(w, C, chan_scale, masks, N,
                                                                       K, G, packed, nullptr);
    return cudaGetLastError();
}

cudaError_t launch_encode(const __nv_bfloat16 *w, const int8_t *C, int N, int K, uint8_t *packed,
                          __nv_bfloat16 *chan_scale, void *workspace, cudaStream_t stream)
{
    return launch_encode_impl(w, C, N, K, packed, nullptr, chan_scale, workspace, stream);
}

cudaError_t launch_fake_quant(const __nv_bfloat16 *w, const int8_t *C, int N, int K,
                              __nv_bfloat16 *w_hat, __nv_bfloat16 *chan_scale, void *workspace,
                              cudaStream_t stream)
{
    return launch_encode_impl(w, C, N, K, nullptr, w_hat, chan_scale, workspace, stream);
}

// ===========================================================================
// Centroid fit (paper section 3.4, "Quantization": C = Round(Lloyd-Max(W'))
// with k-means++ initialisation, Arthur and Vassilvitskii, SODA 2007).
//
// Points: p = g K + k, W'_p = (|W[3g+d,k]| / alpha_{3g+d})_d exactly as in the
// encoder, stored as three fp32 arrays (structure of arrays).  Draws are 32
// caller-supplied 32-bit integers r[t].  Every sum is an exact integer on a
// 2^-20 grid (floor), so the order in which the GPU adds is immaterial:
//   k-means++: centre 0 = point floor(r[0] Np / 2^32); for t >= 1, with
//     w_p = floor(D2_p 2^20) (D2_p the fp32 squared distance to the nearest
//     chosen centre) and S = sum w_p, centre t = the first point whose
//     inclusive prefix sum of w exceeds floor(r[t] S / 2^32) (point
//     floor(r[t] Np / 2^32) when S = 0);
//   Lloyd: `iters` times, nearest centroid per point (fp32, lowest index on a
//     tie), then each nonempty cluster's centroid becomes, per component,
//     float(RN(sum floor(W' 2^20) / n) 2^-20) with the division in fp64; an
//     empty cluster keeps its centroid;
//   Round: to nearest, ties to even, clamped to 0..127.
// ===========================================================================
constexpr int kFitThreads = 256;
constexpr int kKppSelectThreads = 1024;

struct FitSpace {
    __nv_bfloat16 *alpha;   // [N]
    float *P[3];            // [Np] each
    float *D2;              // [Np]
    unsigned long long *bsum;  // [blocks] k-means++ block sums of w
    unsigned long long *acc;   // [32][4] Lloyd sums (x, y, z) and counts
};

constexpr size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// k-means++ point blocks: 4 per SM, at most one per thread of the select kernel.
static int fit_blocks()
{
    const int b = device_sm_count() * 4;
    return b < kKppSelectThreads ? b : kKppSelectThreads;
}

// Byte offsets of the workspace parts; total returned.
static size_t fit_layout(int64_t N, int64_t K, int blocks, size_t off[6])
{
    const int64_t Np = (N + 2) / 3 * K;
    size_t o = 0;
    off[0] = o;  o = align_up(o + (size_t)N * 2, 256);
    for (int d = 0; d < 3; ++d) {
        off[1 + d] = o;
        o = align_up(o + (size_t)Np * 4, 256);
    }
    off[4] = o;  o = align_up(o + (size_t)Np * 4, 256);
    off[5] = o;  o = align_up(o + (size_t)blocks * 8 + 32 * 4 * 8, 256);
    return o;
}

size_t fit_workspace_bytes(int64_t N, int64_t K)
{
    size_t off[6];
    return fit_layout(N, K, fit_blocks(), off);
}

static FitSpace fit_space(void *ws, int64_t N, int64_t K, int blocks)
{
    size_t off[6];
    fit_layout(N, K, blocks, off);
    char *b = static_cast<char *>(ws);
    FitSpace f;
    f.alpha = reinterpret_cast<__nv_bfloat16 *>(b + off[0]);
    for (int d = 0; d < 3; ++d)
        f.P[d] = reinterpret_cast<float *>(b + off[1 + d]);
    f.D2 = reinterpret_cast<float *>(b + off[4]);
    f.bsum = reinterpret_cast<unsigned long long *>(b + off[5]);
    f.acc = f.bsum + blocks;
    return f;
}

// Scaled magnitudes of all points, 8 consecutive k of one packed row per thread.
__global__ __launch_bounds__(kFitThreads) void fit_points_kernel(
    const __nv_bfloat16 *__restrict__ w, const __nv_bfloat16 *__restrict__ alpha, int N, int K,
    int G, float *__restrict__ P0, float *__restrict__ P1, float *__restrict__ P2)
{
    const int chunks = K / 8;
    const int64_t items = (int64_t)G * chunks;
    float *const P[3] = {P0, P1, P2};
    for (int64_t it = (int64_t)blockIdx.x * kFitThreads + threadIdx.x; it < items;
         it += (int64_t)gridDim.x * kFitThreads) {
        const int g = (int)(it / chunks);
        const int c = (int)(it - (int64_t)g * chunks);
#pragma unroll
        for (int d = 0; d < 3; ++d) {
            const int n = 3 * g + d;
            uint32_t u[4] = {0u, 0u, 0u, 0u};
            float a = 0.0f;
            if (n < N) {
                const uint4 v = __ldg(reinterpret_cast<const uint4 *>(w + (size_t)n * K) + c);
                u[0] = v.x;
                u[1] = v.y;
                u[2] = v.z;
                u[3] = v.w;
                a = __bfloat162float(alpha[n]);
            }
            const ChanDiv dv = chan_div(a);
            float q[8];
#pragma unroll
            for (int e = 0; e < 8; ++e)
                q[e] = scaled_abs(elem_abs(u, e), dv);
            float4 *dst = reinterpret_cast<float4 *>(P[d] + (size_t)it * 8);
            dst[0] = make_float4(q[0], q[1], q[2], q[3]);
            dst[1] = make_float4(q[4], q[5], q[6], q[7]);
        }
    }
}

// floor(r x / 2^32) for r < 2^32 and x < 2^62.
__device__ __forceinline__ unsigned long long scale_draw(uint32_t r, unsigned long long x)
{
    return (unsigned long long)r * (x >> 32) + (((unsigned long long)r * (x & 0xFFFFFFFFull)) >> 32);
}

// floor(x 2^20) for 0 <= x < 2^23 without a float-to-integer conversion (those
// run on the FP64 pipe here): ip = floor(x) and floor(frac(x) 2^20) each come
// from the low bits of an add of 2^23 rounded toward zero; x - ip is exact.
__device__ __forceinline__ unsigned long long fixed20(float x)
{
    const float t = __fadd_rz(x, 8388608.0f);                 // 2^23 + floor(x)
    const float fr = __fsub_rn(x, __fsub_rn(t, 8388608.0f));  // x - floor(x), exact
    const float u = __fadd_rz(__fmul_rn(fr, 1048576.0f), 8388608.0f);
    return ((unsigned long long)(__float_as_uint(t) & 0x7FFFFFu) << 20) |
           (__float_as_uint(u) & 0xFFFFFu);
}

__device__ __forceinline__ unsigned long long d2_weight(float d2)
{
    return fixed20(d2);   // d2 < 2^17
}

// Block b of `blocks` covers points [b per, min((b + 1) per, Np)), per a
// multiple of 4 (Np is a multiple of 16), so that blocks start on whole quads.
__device__ __forceinline__ void block_range(int64_t Np, int blocks, int b, int64_t &lo, int64_t &hi)
{
    const int64_t per = ((Np + blocks - 1) / blocks + 3) / 4 * 4;
    lo = (int64_t)b * per;
    hi = lo + per < Np ? lo + per : Np;
    if (lo > Np)
        lo = Np;
}

// D2 update against centre t, and per-block sums of the weights.
__global__ __launch_bounds__(kFitThreads) void kpp_update_kernel(
    const float *__restrict__ P0, const float *__restrict__ P1, const float *__restrict__ P2,
    float *__restrict__ D2, int64_t Np, const float *__restrict__ cf, int t,
    unsigned long long *__restrict__ bsum)
{
    __shared__ unsigned long long red[kFitThreads / 32];
    int64_t lo, hi;
    block_range(Np, gridDim.x, blockIdx.x, lo, hi);
    const float4 c = make_float4(cf[3 * t], cf[3 * t + 1], cf[3 * t + 2], 0.0f);
    unsigned long long sum = 0;
    for (int64_t q = lo / 4 + threadIdx.x; q < hi / 4; q += kFitThreads) {
        const float4 x = reinterpret_cast<const float4 *>(P0)[q];
        const float4 y = reinterpret_cast<const float4 *>(P1)[q];
        const float4 z = reinterpret_cast<const float4 *>(P2)[q];
        float4 d = make_float4(dist2(c, x.x, y.x, z.x), dist2(c, x.y, y.y, z.y),
                               dist2(c, x.z, y.z, z.z), dist2(c, x.w, y.w, z.w));
        if (t > 0) {
            const float4 o = reinterpret_cast<const float4 *>(D2)[q];
            d = make_float4(fminf(d.x, o.x), fminf(d.y, o.y), fminf(d.z, o.z), fminf(d.w, o.w));
        }
        reinterpret_cast<float4 *>(D2)[q] = d;
        sum += d2_weight(d.x) + d2_weight(d.y) + d2_weight(d.z) + d2_weight(d.w);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        sum += __shfl_xor_sync(0xFFFFFFFFu, sum, o);
    if ((threadIdx.x & 31) == 0)
        red[threadIdx.x >> 5] = sum;
    __syncthreads();
    if (threadIdx.x == 0) {
        unsigned long long s2 = 0;
        for (int i = 0; i < kFitThreads / 32; ++i)
            s2 += red[i];
        bsum[blockIdx.x] = s2;
    }
}

// Inclusive prefix sum over the CTA (blockDim.x a multiple of 32, at most 1024).
__device__ unsigned long long block_inclusive_scan(unsigned long long v,
                                                   unsigned long long *warp_tot)
{
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long n = __shfl_up_sync(0xFFFFFFFFu, v, o);
        if (lane >= o)
            v += n;
    }
    if (lane == 31)
        warp_tot[wid] = v;
    __syncthreads();
    if (wid == 0) {
        const int nw = blockDim.x >> 5;
        unsigned long long t = lane < nw ? warp_tot[lane] : 0ull;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned long long n = __shfl_up_sync(0xFFFFFFFFu, t, o);
            if (lane >= o)
                t += n;
        }
        if (lane < nw)
            warp_tot[lane] = t;
    }
    __syncthreads();
    const unsigned long long before = wid > 0 ? warp_tot[wid - 1] : 0ull;
    __syncthreads();   // warp_tot may be reused by the caller's next scan
    return v + before;
}

// Choose centre t (one CTA): uniform for t = 0 or when every weight is 0,
// otherwise the D^2 draw by a two-level prefix search (block sums, then the
// chosen block's points in per-thread chunks).
__global__ __launch_bounds__(kKppSelectThreads) void kpp_select_kernel(
    const float *__restrict__ P0, const float *__restrict__ P1, const float *__restrict__ P2,
    const float *__restrict__ D2, int64_t Np, const unsigned long long *__restrict__ bsum,
    int blocks, const uint32_t *__restrict__ r, int t, float *__restrict__ cf)
{
    __shared__ unsigned long long warp_tot[32];
    __shared__ unsigned long long sh_target, sh_excl;
    __shared__ int sh_block;
    __shared__ long long sh_idx;
    const uint32_t draw = r[t];
    if (threadIdx.x == 0) {
        sh_idx = -1;
        sh_block = -1;
    }
    unsigned long long incl = 0, mine = 0;
    if (t > 0) {
        mine = (int)threadIdx.x < blocks ? bsum[threadIdx.x] : 0ull;
        incl = block_inclusive_scan(mine, warp_tot);
        // the total is the last thread's inclusive sum
        if (threadIdx.x == blockDim.x - 1)
            sh_target = incl;
        __syncthreads();
        const unsigned long long S = sh_target;
        __syncthreads();
        if (S != 0) {
            const unsigned long long target = scale_draw(draw, S);
            if (incl > target && incl - mine <= target) {
                sh_block = (int)threadIdx.x;
                sh_target = target;
                sh_excl = incl - mine;
            }
        }
    }
    __syncthreads();
    if (sh_block < 0) {
        if (threadIdx.x == 0)
            sh_idx = (long long)scale_draw(draw, (unsigned long long)Np);
    } else {
        // Within the chosen block: each warp sums a contiguous run of the block's
        // points in coalesced rows of 32; a scan of the 32 warp sums finds the
        // warp holding the crossing, which walks its rows with a warp scan.
        int64_t lo, hi;
        block_range(Np, blocks, sh_block, lo, hi);
        const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
        const int nw = kKppSelectThreads / 32;
        const int64_t per_w = ((hi - lo + nw - 1) / nw + 31) / 32 * 32;
        const int64_t w0 = lo + (int64_t)wid * per_w;
        const int64_t w1 = w0 + per_w < hi ? w0 + per_w : hi;
        unsigned long long s = 0;
        for (int64_t p = w0 + lane; p < w1; p += 32)
            s += d2_weight(D2[p]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            s += __shfl_xor_sync(0xFFFFFFFFu, s, o);
        const unsigned long long wincl = block_inclusive_scan(lane == 0 ? s : 0ull, warp_tot);
        // wincl of lane 0 of warp w is the inclusive sum up to warp w
        const unsigned long long incl_w = __shfl_sync(0xFFFFFFFFu, wincl, 0);
        const unsigned long long want = sh_target - sh_excl;   // residual within the block
        if (incl_w > want && incl_w - s <= want) {
            unsigned long long run = incl_w - s;
            for (int64_t r0 = w0; r0 < w1; r0 += 32) {
                const int64_t p = r0 + lane;
                unsigned long long v = p < w1 ? d2_weight(D2[p]) : 0ull;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const unsigned long long n = __shfl_up_sync(0xFFFFFFFFu, v, o);
                    if (lane >= o)
                        v += n;
                }
                const uint32_t hit = __ballot_sync(0xFFFFFFFFu, run + v > want);
                if (hit) {
                    if (lane == 0)
                        sh_idx = r0 + (__ffs(hit) - 1);
                    break;
                }
                run += __shfl_sync(0xFFFFFFFFu, v, 31);
            }
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        // the block and point sums come from the same D2 values, so a point is
        // always found; the guard only keeps the read in bounds
        const long long i = sh_idx >= 0 && sh_idx < Np ? sh_idx : 0;
        cf[3 * t] = P0[i];
        cf[3 * t + 1] = P1[i];
        cf[3 * t + 2] = P2[i];
    }
}

// Lloyd assignment: nearest centroid per point, sums into per-warp shared bins,
// then one global add per bin and CTA.  Np is a multiple of 16 (K is), so every
// thread takes 4 whole points.  A point's fixed-point coordinate v < 2^27 goes
// into a warp bin as two 32-bit atomic adds, v mod 2^16 and v / 2^16; the
// launch keeps every warp at no more than 2^16 points (kLloydMaxWarpPoints),
// so neither part can wrap, and the CTA recombines them exactly in 64 bits.
constexpr int kLloydMaxWarpPoints = 1 << 16;
// x lo, x hi, y lo, y hi, z lo, z hi, count, and 2 unused words: a stride of 9
// words puts the 32 bins of a warp on 32 different banks
constexpr int kBinWords = 9;

__global__ __launch_bounds__(kFitThreads) void lloyd_assign_kernel(
    const float *__restrict__ P0, const float *__restrict__ P1, const float *__restrict__ P2,
    int64_t Np, const float *__restrict__ cf, unsigned long long *__restrict__ acc)
{
    __shared__ float4 cen[32];
    __shared__ uint32_t bins[kFitThreads / 32][32][kBinWords];
    if (threadIdx.x < 32)
        cen[threadIdx.x] = make_float4(cf[3 * threadIdx.x], cf[3 * threadIdx.x + 1],
                                       cf[3 * threadIdx.x + 2], 0.0f);
    for (int i = threadIdx.x; i < (kFitThreads / 32) * 32 * kBinWords; i += kFitThreads)
        (&bins[0][0][0])[i] = 0u;
    __syncthreads();
    uint32_t(*mybins)[kBinWords] = bins[threadIdx.x >> 5];
    const int64_t quads = Np / 4;
    for (int64_t q = (int64_t)blockIdx.x * kFitThreads + threadIdx.x; q < quads;
         q += (int64_t)gridDim.x * kFitThreads) {
        const float4 x = reinterpret_cast<const float4 *>(P0)[q];
        const float4 y = reinterpret_cast<const float4 *>(P1)[q];
        const float4 z = reinterpret_cast<const float4 *>(P2)[q];
        const float px[4] = {x.x, x.y, x.z, x.w}, py[4] = {y.x, y.y, y.z, y.w},
                    pz[4] = {z.x, z.y, z.z, z.w};
        float bestd[4];
        int best[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            bestd[j] = dist2(cen[0], px[j], py[j], pz[j]);
            best[j] = 0;
        }
#pragma unroll 4
        for (int l = 1; l < 32; ++l) {
            const float4 c = cen[l];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float d = dist2(c, px[j], py[j], pz[j]);
                if (d < bestd[j]) {
                    bestd[j] = d;
                    best[j] = l;
                }
            }
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            uint32_t *bin = mybins[best[j]];
            const uint32_t vx = (uint32_t)fixed20(px[j]), vy = (uint32_t)fixed20(py[j]),
                           vz = (uint32_t)fixed20(pz[j]);
            atomicAdd(bin + 0, vx & 0xFFFFu);
            atomicAdd(bin + 1, vx >> 16);
            atomicAdd(bin + 2, vy & 0xFFFFu);
            atomicAdd(bin + 3, vy >> 16);
            atomicAdd(bin + 4, vz & 0xFFFFu);
            atomicAdd(bin + 5, vz >> 16);
            atomicAdd(bin + 6, 1u);
        }
    }
    __syncthreads();
    if (threadIdx.x < 128) {
        const int l = threadIdx.x >> 2, j = threadIdx.x & 3;
        unsigned long long s = 0;
        for (int wi = 0; wi < kFitThreads / 32; ++wi) {
            if (j < 3)
                s += (unsigned long long)bins[wi][l][2 * j] +
                     ((unsigned long long)bins[wi][l][2 * j + 1] << 16);
            else
                s += bins[wi][l][6];
        }
        if (s)
            atomicAdd(&acc[4 * l + j], s);
    }
}

// New centroids from the sums (empty clusters stay), then the sums are cleared.
__global__ void lloyd_update_kernel(unsigned long long *__restrict__ acc, float *__restrict__ cf)
{
    const int i = threadIdx.x;
    if (i < 96) {
        const int l = i / 3, d = i - 3 * (i / 3);
        const unsigned long long n = acc[4 * l + 3];
        if (n != 0)
            cf[i] = (float)(((double)acc[4 * l + d] / (double)n) * 0x1p-20);
    }
    __syncthreads();
    if (i < 128)
        acc[i] = 0ull;
}

__global__ void fit_round_kernel(const float *__restrict__ cf, int8_t *__restrict__ C)
{
    const int i = threadIdx.x;
    if (i < 96) {
        int v = __float2int_rn(cf[i]);
        v = v < 0 ? 0 : (v > 127 ? 127 : v);
        C[i] = (int8_t)v;
    }
}

cudaError_t launch_fit(const __nv_bfloat16 *w, int N, int K, const uint32_t *r, int iters,
                       float *cf, int8_t *C, void *workspace, cudaStream_t stream)
{
    const int sms = device_sm_count();
    const int blocks = fit_blocks();
    const FitSpace f = fit_space(workspace, N, K, blocks);
    const int G = (N + 2) / 3;
    const int64_t Np = (int64_t)G * K;
    const int rows_ctas = (N + kScaleRowsPerCta - 1) / kScaleRowsPerCta;
    const int g1 = rows_ctas < sms * 8 ? rows_ctas : sms * 8;
    encode_prepare_kernel<<<g1, kScaleThreads, 0, stream>>>(w, nullptr, N, K, g1, f.alpha, nullptr);
    const int64_t items = (int64_t)G * (K / 8);
    const int64_t want = (items + kFitThreads - 1) / kFitThreads;
    const int gp = (int)(want < (int64_t)sms * 8 ? want : (int64_t)sms * 8);
    fit_points_kernel<<<gp, kFitThreads, 0, stream>>>(w, f.alpha, N, K, G, f.P[0], f.P[1], f.P[2]);
    kpp_select_kernel<<<1, kKppSelectThreads, 0, stream>>>(f.P[0], f.P[1], f.P[2], f.D2, Np, f.bsum,
                                                          blocks, r, 0, cf);
    for (int t = 1; t < 32; ++t) {
        kpp_update_kernel<<<blocks, kFitThreads, 0, stream>>>(f.P[0], f.P[1], f.P[2], f.D2, Np, cf,
                                                              t - 1, f.bsum);
        kpp_select_kernel<<<1, kKppSelectThreads, 0, stream>>>(f.P[0], f.P[1], f.P[2], f.D2, Np,
                                                              f.bsum, blocks, r, t, cf);
    }
    cudaError_t e = cudaMemsetAsync(f.acc, 0, 32 * 4 * sizeof(unsigned long long), stream);
    if (e != cudaSuccess)
        return e;
    const int64_t quads = Np / 4;
    const int64_t wantq = (quads + kFitThreads - 1) / kFitThreads;
    // at least enough CTAs that no warp takes more than kLloydMaxWarpPoints points:
    // a warp's lanes take quads q, q + grid * 256, ..., 4 points each
    const int64_t min_grid = (quads + (int64_t)kFitThreads * (kLloydMaxWarpPoints / 4 / 32) - 1) /
                             ((int64_t)kFitThreads * (kLloydMaxWarpPoints / 4 / 32));
    int64_t ga64 = wantq < (int64_t)sms * 4 ? wantq : (int64_t)sms * 4;
    if (ga64 < min_grid)
        ga64 = min_grid;
    const int ga = (int)ga64;
    for (int it = 0; it < iters; ++it) {
        lloyd_assign_kernel<<<ga, kFitThreads, 0, stream>>>(f.P[0], f.P[1], f.P[2], Np, cf, f.acc);
        lloyd_update_kernel<<<1, 128, 0, stream>>>(f.acc, cf);
    }
    fit_round_kernel<<<1, 128, 0, stream>>>(cf, C);
    return cudaGetLastError();
}

}  // namespace s3d8
