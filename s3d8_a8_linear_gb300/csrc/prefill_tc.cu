// Prefill-regime S3D8 linear on the 5th-generation tensor cores (tcgen05).
//
// sm_103a has no tcgen05 integer MMA, and its legacy INT8 tensor rate is about a
// thirteenth of bf16, so the product runs as bf16 x bf16 -> fp32 with an exact
// integer result: int8 codes and int8 weights are exact in bf16, every product
// is an integer below 2^14, and each K-chunk of at most 1024 columns keeps every
// partial sum below 127 * 127 * 1024 < 2^24, where fp32 holds integers exactly.
// After each chunk the fp32 accumulator is drained into int32 registers.
//
// This file holds the one-SM kernel that decodes packed weight tiles itself
// (below 384 tokens) and the host side of the three tensor-core kernels: from
// 384 tokens the SM-pair kernel that decodes the packed tiles itself
// (prefill_fused.cu, fp16 operands), and from 1537 tokens (2049 on rows longer
// than 8192 columns) the SM-pair kernel on weights expanded to bf16 once per
// call (prefill_pair.cu).
//
// Tile: 128 tokens (MMA M) x 240 output channels (MMA N; 80 whole packed groups)
// per CTA, K in blocks of 64.  Sixteen warps in four warpgroups:
//   warp 0      bulk tensor copies (TMA) of the bf16 activation tile (from the
//               workspace) and of the 80 x 64 packed-byte tile;
//   warp 1      TMEM allocation and the MMA issuer (one thread);
//   warps 2-15  decode: packed bytes -> bf16 weights, written straight into the
//               128-byte-swizzled K-major layout the MMA descriptor reads;
//   warps 8-15  also drain the fp32 accumulator per K-chunk into int32 registers
//               (between decode steps) and write the epilogue (x_s * acc) * W_s
//               as bf16 (or the raw int32).
// Warpgroups 0-1 give registers up (setmaxnreg 80) so that the drain warps can
// hold 120 int32 sums each (setmaxnreg 176): 128 x (80+80+176+176) = 65536.
// TMEM holds two accumulator buffers (columns 0 and 256) so that the MMA fills
// one chunk while the other drains.  Every mbarrier wait is bounded.
#include "tcgen05.cuh"

#include <atomic>


namespace s3d8 {

namespace tc {

// The weight tile is decoded from packed bytes in shared memory by warps 2-15.
__global__ __launch_bounds__(THREADS, 1) void prefill_kernel(const __grid_constant__ CUtensorMap tm_act,
                                                             const __grid_constant__ CUtensorMap tm_pk,
                                                             Params p)
{
    constexpr int LST = LSTAGES;
    constexpr int BST = BSTAGES;
    constexpr int O_B = OFF_B;
    constexpr int O_BARS = OFF_BARS;
    constexpr int NB = NBARS;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    unsigned char *smem = smem_raw + (base - raw);
    const uint32_t lut = base + OFF_LUT;
    const uint32_t bars = base + O_BARS;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + O_BARS + NB * 8);
    // barriers: l_full[L] (TMA bytes of the slot), l_empty[L] (MMA done with the
    //           slot), b_full[B] (decoded tile written), b_empty[B] (MMA done with
    //           the decoded tile), acc_full[2] (chunk in TMEM), acc_empty[2]
    const uint32_t l_full = bars, l_empty = l_full + 8 * LST;
    const uint32_t b_full = l_empty + 8 * LST, b_empty = b_full + 8 * BST;
    const uint32_t acc_full = b_empty + 8 * BST, acc_empty = acc_full + 16;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // Persistent: CTA b takes output tiles b, b + gridDim.x, ...  A tile is
    // (128 tokens, 240 channels, one K split); consecutive tile indices share the
    // channel tile, so the CTAs working at one time reuse its weights from L2.
    const int mtiles = (p.M + BM - 1) / BM;
    const int ntiles = ((p.N + 2) / 3 + GROUPS - 1) / GROUPS;
    const int nk_all = (p.K + BK - 1) / BK;
    const int total = mtiles * ntiles * p.nsplit;
    struct Tile {
        int m0, nt, split, kbase, nk;
    };
    auto tile_of = [&](int t) {
        Tile T;
        const int mt = t % mtiles, rest = t / mtiles;
        T.nt = rest % ntiles;
        T.split = rest / ntiles;
        T.m0 = mt * BM;
        T.kbase = T.split * p.kb_per_split;
        T.nk = min(p.kb_per_split, nk_all - T.kbase);
        return T;
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < LST; ++s) {
            mbar_init(l_full + 8 * s, 1);
            mbar_init(l_empty + 8 * s, 1);
        }
        for (int s = 0; s < BST; ++s) {
            mbar_init(b_full + 8 * s, DECODERS / 32);
            mbar_init(b_empty + 8 * s, 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(acc_full + 8 * i, 1);
            mbar_init(acc_empty + 8 * i, 8);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(
                         smem_addr(tmem_slot))
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    // decode table: byte -> [bf16 w0 | bf16 w1 << 16, bf16 w2], 16 copies (one per
    // half-warp lane) so that 8-byte lookups never conflict.
    {
        __shared__ int8_t Cs[96];
        for (int i = threadIdx.x; i < 96; i += THREADS)
            Cs[i] = p.C[i];
        __syncthreads();
        uint2 *t = reinterpret_cast<uint2 *>(smem + OFF_LUT);
        for (int i = threadIdx.x; i < kLutEntries * LUT_COPIES; i += THREADS) {
            const uint32_t e = expanded_entry(Cs, (uint32_t)(i / LUT_COPIES));
            const int w0 = (int8_t)(e & 0xFF), w1 = (int8_t)((e >> 8) & 0xFF), w2 = (int8_t)((e >> 16) & 0xFF);
            t[i] = make_uint2(bf16_bits_of(w0) | (bf16_bits_of(w1) << 16), bf16_bits_of(w2));
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    bool timed_out = false;
    pdl_launch_dependents();   // the split-K finish may be scheduled; it waits for this grid

    if (warp < DRAIN_WARP0) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 80;");
    if (warp == 0) {
        // ---- bulk tensor copies (whole warp; one elected lane issues) --------------
        {
            pdl_wait();       // the activation codes come from the previous kernel
            int issued = 0;   // k-blocks issued by this CTA over all its tiles
            for (int t = blockIdx.x; t < total && !timed_out; t += gridDim.x) {
                const Tile T = tile_of(t);
                for (int kb = 0; kb < T.nk; ++kb) {
                    const int s = issued % LST;
                    if (issued >= LST && !warp_wait(l_empty + 8 * s, ((issued / LST) - 1) & 1)) {
                        timed_out = true;
                        break;
                    }
                    mbar_arrive_expect_tx_elect(l_full + 8 * s, A_BYTES + P_BYTES);
                    tma_2d_elect(base + OFF_A + s * A_BYTES, &tm_act, (T.kbase + kb) * BK, T.m0, l_full + 8 * s);
                    tma_2d_elect(base + OFF_P + s * P_BYTES, &tm_pk, (T.kbase + kb) * BK, T.nt * GROUPS,
                                 l_full + 8 * s);
                    ++issued;
                }
            }
            // never leave with copies in flight: wait (bounded) for the last ones
            for (int v = issued - LST < 0 ? 0 : issued - LST; v < issued; ++v)
                if (!warp_wait(l_full + 8 * (v % LST), (v / LST) & 1))
                    timed_out = true;
        }
    } else if (warp == 1) {
        // ---- MMA issuer: the whole warp runs the loop so that the descriptors stay
        // warp-uniform; one elected lane issues --------------------------------------
        {
            int g = 0;    // k-blocks consumed by this CTA over all its tiles
            int gc = 0;   // chunks started by this CTA over all its tiles
            const uint32_t idesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) |
                                   ((uint32_t)(BM >> 4) << 24);
            for (int t = blockIdx.x; t < total && !timed_out; t += gridDim.x) {
                const Tile T = tile_of(t);
                for (int kb = 0; kb < T.nk; ++kb) {
                    const int s = g % LST, bs = g % BSTAGES;
                    const int c = gc + kb / CHUNK_BLOCKS, kin = kb % CHUNK_BLOCKS;
                    const uint32_t d = tmem + (uint32_t)((c & 1) * 256);
                    if (kin == 0 && c >= 2 && !warp_wait(acc_empty + 8 * (c & 1), ((c >> 1) - 1) & 1)) {
                        timed_out = true;
                        break;
                    }
                    if (!warp_wait(l_full + 8 * s, (g / LST) & 1) || !warp_wait(b_full + 8 * bs, (g / BSTAGES) & 1)) {
                        timed_out = true;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a = base + OFF_A + s * A_BYTES, b = base + O_B + bs * B_BYTES;
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk)
                        mma_bf16_elect(d, sw128_desc(a + kk * 32), sw128_desc(b + kk * 32), idesc,
                                       (kin | kk) ? 1u : 0u);
                    mma_commit_elect(l_empty + 8 * s);
                    mma_commit_elect(b_empty + 8 * bs);
                    if (kin == CHUNK_BLOCKS - 1 || kb == T.nk - 1)
                        mma_commit_elect(acc_full + 8 * (c & 1));
                    ++g;
                }
                gc += (T.nk + CHUNK_BLOCKS - 1) / CHUNK_BLOCKS;
            }
            // the tensor core must be done with TMEM and shared memory before exit
            if (g > 0 && !warp_wait(l_empty + 8 * ((g - 1) % LST), ((g - 1) / LST) & 1))
                timed_out = true;
        }
    } else {
        // ---- decode packed bytes into the swizzled bf16 weight tile -------------
        const int tid = threadIdx.x - 64;
        const uint32_t lut_lane = lut + (uint32_t)((lane & (LUT_COPIES - 1)) * 8);
        int g = 0;
        for (int t = blockIdx.x; t < total && !timed_out; t += gridDim.x) {
            const Tile T = tile_of(t);
            for (int kb = 0; kb < T.nk; ++kb, ++g) {
                const int s = g % LSTAGES, bs = g % BSTAGES;
                if (!mbar_wait_bounded(l_full + 8 * s, (g / LSTAGES) & 1) ||
                    (g >= BSTAGES && !mbar_wait_bounded(b_empty + 8 * bs, ((g / BSTAGES) - 1) & 1))) {
                    timed_out = true;
                    break;
                }
                decode_tile(base + OFF_P + s * P_BYTES, base + OFF_B + bs * B_BYTES, lut_lane, tid, DECODERS);
                fence_proxy_async_smem();   // generic writes -> visible to the tensor core
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(b_full + 8 * bs);
            }
        }
    }
    } else {
        // ---- drain chunks into int32, then the epilogue ---------------------------
        asm volatile("setmaxnreg.inc.sync.aligned.u32 176;");
        const int q = warp & 3;                 // TMEM lane quadrant of this warp
        const int h = (warp - DRAIN_WARP0) >> 2; // which half of the 240 columns
        int32_t acc[HALF];
        // fp32 chunk c in TMEM -> int32 registers; then release its buffer
        auto drain = [&](int c) {
            tc_fence_after();
            const uint32_t ta = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)((c & 1) * 256 + h * HALF);
#pragma unroll
            for (int gg = 0; gg < HALF / 24; ++gg) {
                float v[3][8];
#pragma unroll
                for (int i = 0; i < 3; ++i)
                    tmem_ld8(ta + (gg * 3 + i) * 8, v[i]);
                asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
                for (int i = 0; i < 3; ++i)
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        acc[(gg * 3 + i) * 8 + j] += __float2int_rn(v[i][j]);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(acc_empty + 8 * (c & 1));
        };
        // Between chunk drains these warps decode too.  A finished
        // chunk is drained before the next K block is decoded, so the MMA never
        // waits on a buffer these warps have not released while they wait on it.
        const int tid = threadIdx.x - 64;
        const uint32_t lut_lane = lut + (uint32_t)((lane & (LUT_COPIES - 1)) * 8);
        int g = 0;    // decoded k-blocks over all tiles
        int gc = 0;   // first chunk of the current tile
        for (int t = blockIdx.x; t < total && !timed_out; t += gridDim.x) {
            const Tile T = tile_of(t);
            const int nch = (T.nk + CHUNK_BLOCKS - 1) / CHUNK_BLOCKS;
#pragma unroll
            for (int i = 0; i < HALF; ++i)
                acc[i] = 0;
            int cn = gc;   // next chunk to drain
            for (int kb = 0; kb < T.nk && !timed_out; ++kb, ++g) {
                while (cn < gc + nch) {
                    const bool ready =
                        __shfl_sync(0xffffffffu, (int)mbar_test(acc_full + 8 * (cn & 1), (cn >> 1) & 1), 0) != 0;
                    if (!ready)
                        break;
                    drain(cn++);
                }
                const int s = g % LSTAGES, bs = g % BSTAGES;
                if (!mbar_wait_bounded(l_full + 8 * s, (g / LSTAGES) & 1) ||
                    (g >= BSTAGES && !mbar_wait_bounded(b_empty + 8 * bs, ((g / BSTAGES) - 1) & 1))) {
                    timed_out = true;
                    break;
                }
                decode_tile(base + OFF_P + s * P_BYTES, base + OFF_B + bs * B_BYTES, lut_lane, tid, DECODERS);
                fence_proxy_async_smem();   // generic writes -> visible to the tensor core
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(b_full + 8 * bs);
            }
            for (; cn < gc + nch && !timed_out; ++cn) {
                if (!mbar_wait_bounded(acc_full + 8 * (cn & 1), (cn >> 1) & 1)) {
                    timed_out = true;
                    break;
                }
                drain(cn);
            }
            gc += nch;
            const int row = T.m0 + 32 * q + lane;
            if (!timed_out && row < p.M)
                store_tile_row(p, T.split, row, T.nt * BN + h * HALF, acc);
        }
    }
    if (timed_out)
        record_timeout(p.status);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem) : "memory");
}

// int8 codes -> bf16 (exact), the tensor-core A operand, without int-to-float
// conversions: with b = code ^ 0x80 = v + 128 (0..255), one byte permute builds
// the float 0x4B4000bb = 1.5 * 2^23 + b, one FP32 add of -(1.5 * 2^23 + 128)
// leaves v exactly, and its upper 16 bits are v's bf16 (|v| <= 128 needs 8
// significant bits); one more permute packs two of them.
__device__ __forceinline__ void codes16_to_bf16(uint4 v, uint4 *dst)
{
    const uint32_t w[4] = {v.x ^ 0x80808080u, v.y ^ 0x80808080u, v.z ^ 0x80808080u, v.w ^ 0x80808080u};
    constexpr uint32_t kMagic = 0x4B400000u;
    constexpr float kOff = -12583040.0f;   // -(1.5 * 2^23 + 128)
    uint32_t o[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        float f[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
            f[i] = __fadd_rn(__uint_as_float(prmt(w[j], kMagic, 0x7650u | (uint32_t)i)), kOff);
        o[2 * j] = prmt(__float_as_uint(f[0]), __float_as_uint(f[1]), 0x7632u);
        o[2 * j + 1] = prmt(__float_as_uint(f[2]), __float_as_uint(f[3]), 0x7632u);
    }
    dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
    dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
}

__global__ void codes_to_bf16_kernel(const int8_t *__restrict__ xq, __nv_bfloat16 *__restrict__ a, long n16)
{
    pdl_launch_dependents();   // the GEMM may set up meanwhile; it waits before reading a
    const uint4 *src = reinterpret_cast<const uint4 *>(xq);
    uint4 *dst = reinterpret_cast<uint4 *>(a);
    const long stride = (long)gridDim.x * blockDim.x;
    for (long i = (long)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += 2 * stride) {
        const uint4 v0 = __ldg(src + i);
        const bool two = i + stride < n16;
        const uint4 v1 = two ? __ldg(src + i + stride) : make_uint4(0u, 0u, 0u, 0u);
        codes16_to_bf16(v0, dst + 2 * i);
        if (two)
            codes16_to_bf16(v1, dst + 2 * (i + stride));
    }
}

// int8 codes -> fp16 (exact), the A operand of the fused SM-pair kernel: with
// b = code ^ 0x80 = v + 128, one byte permute builds the fp16 pair 0x64bb
// (1024 + b) for two codes, and one packed fp16 subtract of 1152 leaves v
// (fp16 holds every integer of magnitude up to 2048).
__device__ __forceinline__ void codes16_to_f16(uint4 v, uint4 *dst)
{
    const uint32_t w[4] = {v.x ^ 0x80808080u, v.y ^ 0x80808080u, v.z ^ 0x80808080u, v.w ^ 0x80808080u};
    uint32_t o[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        o[2 * j] = f16x2_sub(prmt(w[j], 0x64646464u, 0x5140u), 0x64806480u);
        o[2 * j + 1] = f16x2_sub(prmt(w[j], 0x64646464u, 0x7362u), 0x64806480u);
    }
    dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
    dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
}

__global__ void codes_to_f16_kernel(const int8_t *__restrict__ xq, uint16_t *__restrict__ a, long n16)
{
    pdl_launch_dependents();   // the GEMM may set up meanwhile; it waits before reading a
    const uint4 *src = reinterpret_cast<const uint4 *>(xq);
    uint4 *dst = reinterpret_cast<uint4 *>(a);
    const long stride = (long)gridDim.x * blockDim.x;
    for (long i = (long)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += stride)
        codes16_to_f16(__ldg(src + i), dst + 2 * i);
}

// Weights expanded to bf16 [N, K] (row n = component n % 3 of packed row n / 3),
// the B operand of the SM-pair kernel (prefill_pair.cu).  One thread per 16
// packed bytes; the 16-copy table of bf16 triples is the kernel's own.
__global__ __launch_bounds__(256) void decode_bf16_kernel(const uint8_t *__restrict__ packed,
                                                          const int8_t *__restrict__ C, int N, int K,
                                                          __nv_bfloat16 *__restrict__ w)
{
    pdl_launch_dependents();   // the GEMM may set up meanwhile; it waits before reading w
    __shared__ int8_t Cs[96];
    __shared__ uint2 lut[kLutEntries * LUT_COPIES];
    for (int i = threadIdx.x; i < 96; i += blockDim.x)
        Cs[i] = C[i];
    __syncthreads();
    for (int i = threadIdx.x; i < kLutEntries * LUT_COPIES; i += blockDim.x) {
        const uint32_t e = expanded_entry(Cs, (uint32_t)(i / LUT_COPIES));
        const int w0 = (int8_t)(e & 0xFF), w1 = (int8_t)((e >> 8) & 0xFF), w2 = (int8_t)((e >> 16) & 0xFF);
        lut[i] = make_uint2(bf16_bits_of(w0) | (bf16_bits_of(w1) << 16), bf16_bits_of(w2));
    }
    __syncthreads();
    const int G = (N + 2) / 3, kc = K / 16;
    const uint2 *mylut = lut + (threadIdx.x & (LUT_COPIES - 1));
    for (long u = (long)blockIdx.x * blockDim.x + threadIdx.x; u < (long)G * kc; u += (long)gridDim.x * blockDim.x) {
        const int g = (int)(u / kc), c = (int)(u - (long)g * kc);
        const uint4 v = __ldg(reinterpret_cast<const uint4 *>(packed + (size_t)g * K) + c);
        const uint32_t pw[4] = {v.x, v.y, v.z, v.w};
        uint32_t o[3][8];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            uint2 e[4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
                e[i] = mylut[((pw[q] >> (8 * i)) & 0xFFu) * LUT_COPIES];
            o[0][2 * q] = prmt(e[0].x, e[1].x, 0x5410);
            o[0][2 * q + 1] = prmt(e[2].x, e[3].x, 0x5410);
            o[1][2 * q] = prmt(e[0].x, e[1].x, 0x7632);
            o[1][2 * q + 1] = prmt(e[2].x, e[3].x, 0x7632);
            o[2][2 * q] = prmt(e[0].y, e[1].y, 0x5410);
            o[2][2 * q + 1] = prmt(e[2].y, e[3].y, 0x5410);
        }
#pragma unroll
        for (int d = 0; d < 3; ++d) {
            const int n = 3 * g + d;
            if (n < N) {
                uint4 *dst = reinterpret_cast<uint4 *>(w + (size_t)n * K + (size_t)c * 16);
                dst[0] = make_uint4(o[d][0], o[d][1], o[d][2], o[d][3]);
                dst[1] = make_uint4(o[d][4], o[d][5], o[d][6], o[d][7]);
            }
        }
    }
}

// Split-K finish: out[m, n] (or acc) from the sum of the nsplit int32 partials.
// Integer sums, so the order of the splits does not matter.
// Split-K finish: sums the int32 partials [nsplit][M][N] and writes the raw
// int32 result or the bf16 epilogue.  Threads take 4 consecutive columns of a row
// (16-byte partial loads when N % 4 == 0), rows by grid stride: no division per
// element.
__global__ void finalize_kernel(const int32_t *__restrict__ part, int nsplit, int M, int N,
                                const float *__restrict__ xscale, const __nv_bfloat16 *__restrict__ cs,
                                __nv_bfloat16 *__restrict__ out, int32_t *__restrict__ acc, int vec_in,
                                int vec_out)
{
    // The next kernel may set up meanwhile (it waits for this grid before it
    // reads or writes anything this kernel touches).
    pdl_launch_dependents();
    pdl_wait();   // the partials are the previous kernel's output
    const size_t plane = (size_t)M * N;
    const int quads = (N + 3) / 4;
    for (int m = blockIdx.y; m < M; m += gridDim.y) {
        const size_t row = (size_t)m * N;
        for (int qd = blockIdx.x * blockDim.x + threadIdx.x; qd < quads; qd += gridDim.x * blockDim.x) {
            const int n0 = 4 * qd;
            int32_t v[4] = {0, 0, 0, 0};
            if (vec_in) {
                // eight partials' loads in flight at once, not one L2 round trip each
                for (int sp0 = 0; sp0 < nsplit; sp0 += 8) {
                    int4 t[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        t[j] = sp0 + j < nsplit
                                   ? __ldg(reinterpret_cast<const int4 *>(part + (sp0 + j) * plane + row + n0))
                                   : make_int4(0, 0, 0, 0);
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        v[0] += t[j].x;
                        v[1] += t[j].y;
                        v[2] += t[j].z;
                        v[3] += t[j].w;
                    }
                }
            } else {
                for (int sp = 0; sp < nsplit; ++sp)
                    for (int j = 0; j < 4; ++j)
                        if (n0 + j < N)
                            v[j] += __ldg(part + sp * plane + row + n0 + j);
            }
            if (acc) {
                if (vec_out)
                    *reinterpret_cast<int4 *>(acc + row + n0) = make_int4(v[0], v[1], v[2], v[3]);
                else
                    for (int j = 0; j < 4; ++j)
                        if (n0 + j < N)
                            acc[row + n0 + j] = v[j];
            } else {
                const float xs = __ldg(xscale + m);
                __nv_bfloat16 o[4];
                for (int j = 0; j < 4; ++j)
                    o[j] = epilogue_bf16(v[j], xs, cs[n0 + j < N ? n0 + j : 0]);
                if (vec_out) {
                    const uint32_t lo = (uint32_t)__bfloat16_as_ushort(o[0]) | ((uint32_t)__bfloat16_as_ushort(o[1]) << 16);
                    const uint32_t hi = (uint32_t)__bfloat16_as_ushort(o[2]) | ((uint32_t)__bfloat16_as_ushort(o[3]) << 16);
                    *reinterpret_cast<uint2 *>(out + row + n0) = make_uint2(lo, hi);
                } else {
                    for (int j = 0; j < 4; ++j)
                        if (n0 + j < N)
                            out[row + n0 + j] = o[j];
                }
            }
        }
    }
}

}  // namespace tc

// K split of the tensor-core GEMM when its output tiles alone cannot fill the
// GPU: the number of 64-column blocks per split that minimises
// waves x (blocks per CTA + a per-CTA fixed cost of about 4 blocks), for
// `tiles` CTAs per K range.  Returns that cost.
static double split_plan(long tiles, int nk, int sms, int &nsplit, int &kb_per_split)
{
    nsplit = 1;
    kb_per_split = nk;
    if (tiles >= sms)
        return (double)((tiles + sms - 1) / sms) * (nk + 4);
    double best = 1e30;
    for (int s = 1; s <= 16 && s <= nk; ++s) {
        const int kbps = (nk + s - 1) / s;
        const int real = (nk + kbps - 1) / kbps;   // no empty splits
        const long ctas = tiles * real;
        const double cost = (double)((ctas + sms - 1) / sms) * (kbps + 4);
        if (cost < best - 1e-9) {
            best = cost;
            nsplit = real;
            kb_per_split = kbps;
        }
    }
    return best;
}

// Packed rows per CTA of the fused SM-pair kernel's tile: 40 (256 tokens x 240
// channels) or 32 (256 x 192), whichever gives the lower split-plan cost times
// the tile's measured time per K block.  On gate/up at 512 tokens 40 makes 120
// pair tiles for 76 SM pairs (two rounds for 1.6 rounds of work), 32 makes 150
// (two rounds of shorter tiles).
int fused_tile_groups(int M, int N, int K, int sms)
{
    const long mt = (M + 255) / 256;
    const long G = (N + 2) / 3;
    const int nk = (K + tc::BK - 1) / tc::BK;
    // time per K block of one pair tile, relative, as measured on GB300 at 512
    // tokens (gate/up: 0.483 us per block with 32 packed rows per CTA, 0.548 us
    // with 40; a 24-row tile with three decoder warps, 0.385 us, lost on rounds
    // at every size and was dropped)
    const int g2s[2] = {40, 32};
    const double block_cost[2] = {910.0, 800.0};
    int best_g2 = 40;
    double best = 1e30;
    for (int i = 0; i < 2; ++i) {
        const int g2 = g2s[i];
        int ns, kb;
        const double c = split_plan(2 * mt * ((G + 2 * g2 - 1) / (2 * g2)), nk, sms, ns, kb) * block_cost[i];
        if (c < best - 1e-9) {
            best = c;
            best_g2 = g2;
        }
    }
    return best_g2;
}

// CTAs per K range: 128 x 240 tiles on one SM, 256 x 240 or 256 x 192 tiles on
// two (fused), or 256 x 256 tiles on two (expanded weights).
static void tc_plan(int M, int N, int K, int sms, int kind, int &nsplit, int &kb_per_split)
{
    const long G = (N + 2) / 3;
    long tiles;
    if (kind == kTcPairExpanded) {
        tiles = 2L * ((M + 255) / 256) * ((N + 255) / 256);
    } else if (kind == kTcPairFused) {
        const int g2 = fused_tile_groups(M, N, K, sms);
        tiles = 2L * ((M + 255) / 256) * ((G + 2 * g2 - 1) / (2 * g2));
    } else {
        tiles = (long)((M + tc::BM - 1) / tc::BM) * ((G + tc::GROUPS - 1) / tc::GROUPS);
    }
    split_plan(tiles, (K + tc::BK - 1) / tc::BK, sms, nsplit, kb_per_split);
}

static size_t align256(size_t v)
{
    return (v + 255) & ~(size_t)255;
}

// The kernel for M tokens of K columns.  From 384 tokens the SM pairs'
// 256-token tiles decode each packed weight tile once per 256 tokens instead of
// once per 128.  Expanding the weights to bf16 once per call pays off once the
// fused kernel needs a seventh row of 256-token tiles on rows of up to 8192
// columns (from 1537 tokens); on longer rows, whose expanded tiles (activation
// and weight rows of 2 K bytes each) overflow L2 when the SM pairs stream them
// at once, the fused kernel was faster at every size measured, up to 2048
// tokens.  Measured on GB300 on the 11B shapes (us, fused / expanded): gate/up
// (K 4096) 1024: 105.9 / 107.9, 1536: 148.8 / 150.5, 1792: 173.8 / 168.0,
// 2048: 199.4 / 172.6; down (K 14336) 1536: 162.7 / 177.1, 2048: 181.8 /
// 187.7.
constexpr int kPairsMinM = 384;
constexpr int kExpandMinMShortK = 1537;
constexpr int kExpandMinMLongK = 2049;
constexpr int kLongK = 8192;

int prefill_kind(int M, int K)
{
    const int expand_min = K > kLongK ? kExpandMinMLongK : kExpandMinMShortK;
    return M >= expand_min ? kTcPairExpanded : M >= kPairsMinM ? kTcPairFused : kTcOneSm;
}

// Workspace: the bf16 copy of the activation codes, then the split-K partials,
// then (expanded kind only) the bf16 weights [N, K].
size_t prefill_workspace_bytes(int M, int N, int K, int kind)
{
    int nsplit, kbps;
    tc_plan(M, N, K, device_sm_count(), kind, nsplit, kbps);
    size_t bytes = align256((size_t)M * K * 2) + 256;
    if (nsplit > 1)
        bytes += align256((size_t)nsplit * M * N * 4);
    if (kind == kTcPairExpanded)
        bytes += align256((size_t)N * K * 2);
    return bytes;
}

cudaError_t launch_splitk_finalize(const int32_t *part, int nsplit, const LinearArgs &a, cudaStream_t stream)
{
    const int quads = (a.N + 3) / 4;
    const int vec_in = (a.N & 3) == 0 && ((uintptr_t)part & 15) == 0;
    const int vec_out = (a.N & 3) == 0 && (a.acc ? ((uintptr_t)a.acc & 15) == 0 : ((uintptr_t)a.out & 7) == 0);
    const int bx = (quads + 127) / 128;
    const long rows_per = (long)device_sm_count() * 16 / (bx > 0 ? bx : 1);
    const int by = (int)(a.M < rows_per ? a.M : (rows_per > 0 ? rows_per : 1));
    return tc::launch_pdl(tc::finalize_kernel, dim3((unsigned)bx, (unsigned)by), dim3(128), 0, stream, part, nsplit,
                          a.M, a.N, a.xscale, a.cs, a.out, a.acc, vec_in, vec_out);
}

static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder()
{
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(tensor_map_encoder_fn());
}

// The driver's cuTensorMapEncodeTiled, looked up through the runtime until a
// lookup succeeds, then cached (racing threads store the same pointer).
void *tensor_map_encoder_fn()
{
    static std::atomic<void *> fn{nullptr};
    void *f = fn.load(std::memory_order_relaxed);
    if (!f) {
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        fn.store(f, std::memory_order_relaxed);
    }
    return f;
}

cudaError_t launch_prefill_tc(const LinearArgs &a, int kind, cudaStream_t stream)
{
    using namespace tc;
    if (!a.ws || a.ws_bytes < prefill_workspace_bytes(a.M, a.N, a.K, kind))
        return cudaErrorInvalidValue;
    const bool pre = kind == kTcPairExpanded;
    int nsplit, kbps;
    tc_plan(a.M, a.N, a.K, device_sm_count(), kind, nsplit, kbps);
    auto encode = tensor_map_encoder();
    if (!encode)
        return cudaErrorNotSupported;
    __nv_bfloat16 *act = reinterpret_cast<__nv_bfloat16 *>(((uintptr_t)a.ws + 255) & ~(uintptr_t)255);
    unsigned char *after_act = reinterpret_cast<unsigned char *>(act) + align256((size_t)a.M * a.K * 2);
    int32_t *part = nsplit > 1 ? reinterpret_cast<int32_t *>(after_act) : nullptr;
    __nv_bfloat16 *wdec = reinterpret_cast<__nv_bfloat16 *>(
        after_act + (nsplit > 1 ? align256((size_t)nsplit * a.M * a.N * 4) : 0));
    const long n16 = (long)a.M * a.K / 16;
    const int sms = device_sm_count();
    int cgrid = (int)((n16 + 511) / 512);
    if (cgrid > sms * 16)
        cgrid = sms * 16;
    // the fused SM-pair kernel multiplies fp16 operands, the others bf16
    if (kind == kTcPairFused)
        tc::codes_to_f16_kernel<<<cgrid, 256, 0, stream>>>(a.xq, reinterpret_cast<uint16_t *>(act), n16);
    else
        tc::codes_to_bf16_kernel<<<cgrid, 256, 0, stream>>>(a.xq, act, n16);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return e;
    if (pre) {
        const long units = (long)((a.N + 2) / 3) * (a.K / 16);
        long dgrid = (units + 255) / 256;
        if (dgrid > (long)sms * 8)
            dgrid = (long)sms * 8;
        tc::decode_bf16_kernel<<<(unsigned)dgrid, 256, 0, stream>>>(a.packed, a.C, a.N, a.K, wdec);
        e = cudaGetLastError();
        if (e != cudaSuccess)
            return e;
    }

    if (kind != kTcOneSm) {
        // the SM-pair kernels (256-token tiles on two SMs)
        e = pre ? launch_prefill_pair(a, act, wdec, part, nsplit, kbps, stream)
                : launch_prefill_fused(a, reinterpret_cast<const uint16_t *>(act), part, nsplit, kbps,
                                       fused_tile_groups(a.M, a.N, a.K, device_sm_count()), stream);
        if (e != cudaSuccess || nsplit == 1)
            return e;
        return launch_splitk_finalize(part, nsplit, a, stream);
    }

    const int G = (a.N + 2) / 3;
    CUtensorMap tm_act, tm_pk;
    const cuuint64_t dA[2] = {(cuuint64_t)a.K, (cuuint64_t)a.M};
    const cuuint64_t sA[1] = {(cuuint64_t)a.K * 2};
    const cuuint32_t boxA[2] = {BK, BM}, es[2] = {1, 1};
    const cuuint64_t dP[2] = {(cuuint64_t)a.K, (cuuint64_t)G};
    const cuuint64_t sP[1] = {(cuuint64_t)a.K};
    const cuuint32_t boxP[2] = {BK, GROUPS};
    if (encode(&tm_act, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, act, dA, sA, boxA, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    if (encode(&tm_pk, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(a.packed), dP, sP, boxP, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;

    const int smem_bytes = SMEM_BYTES;
    e = cudaFuncSetAttribute(tc::prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
    if (e != cudaSuccess)
        return e;
    tc::Params p = tc::make_params(a, nsplit, kbps, part);
    const long tiles = (long)((a.M + BM - 1) / BM) * (long)((G + GROUPS - 1) / GROUPS) * nsplit;
    if (tiles > 0x7FFFFFFFL)
        return cudaErrorInvalidValue;
    const long ctas = tiles < sms ? tiles : sms;   // persistent CTAs walk the tiles
    e = tc::launch_pdl(tc::prefill_kernel, dim3((unsigned)ctas), dim3(THREADS), (size_t)smem_bytes, stream, tm_act,
                       tm_pk, p);
    if (e != cudaSuccess || nsplit == 1)
        return e;
    return launch_splitk_finalize(part, nsplit, a, stream);
}

}  // namespace s3d8
