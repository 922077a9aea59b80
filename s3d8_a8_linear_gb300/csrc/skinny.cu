// Batched-decode S3D8 linear for 5..32 tokens: the weights are decoded straight
// into register fragments of mma.sync m16n8k16 (bf16 in, fp32 accumulate).
//
// Why not the tcgen05 kernel: at a few tokens every weight byte is used for
// only a few multiply-adds, and that kernel's expansion of packed bytes into a
// shared-memory bf16 tile (table read, tile store, tensor-core read: ~28 shared
// bytes per packed byte) bounds it far below HBM speed.  Here a packed byte is
// read once from a bulk-copied ring, looked up once in a lane-replicated table
// and never stored: the lookup's bf16 triple is permuted into B fragments.
//
// Operands: D[tokens x channels] += A[tokens x k] * B[k x channels].  A warp owns
// 8 packed rows (24 channels = three n8 tiles: tile d holds channel d of the 8
// groups); B fragment b0 of lane (g, t) needs weights of group g at two k-slots
// and b1 at two more.  Mapping the MMA's k-slots (2t, 2t+1, 2t+8, 2t+9) to the
// actual columns 4t..4t+3 of each 16-column step makes the four weights one
// packed word, and the same permutation of A (activation codes, staged once
// per CTA in fragment order in shared memory) keeps the product unchanged.
//
// Exactness: each CTA covers at most 1024 columns of K, so every fp32 partial
// sum of integer products stays below 127 * 127 * 1024 < 2^24 and is exact; the
// K splits' int32 partials are summed by the split-K finish kernel.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "launch.h"
#include "tma.cuh"

namespace s3d8 {

namespace sk {

constexpr int WARPS = 16;
constexpr int THREADS = WARPS * 32;
constexpr int GPW = 8;                     // packed rows (groups) per warp
constexpr int ROWS_PER_CTA = WARPS * GPW;  // 128
constexpr int STAGE_K = 256;               // packed bytes per row per ring stage
constexpr int BOX_K = 128;                 // one bulk tensor copy: 8 rows x 128 bytes, 128-byte swizzle
constexpr int STAGE_BYTES = GPW * STAGE_K; // two 1 KiB swizzle atoms
constexpr int DEPTH = 2;
constexpr int RING_BYTES = DEPTH * STAGE_BYTES;
constexpr int MAX_KCTA = 1024;             // fp32 partial sums stay exact
constexpr int MAX_MT = 2;                  // up to two m16 token tiles (32 tokens)
constexpr int ACT_BYTES = (MAX_KCTA / 16) * MAX_MT * 512;
constexpr int DYN_SMEM = 232448 - 4096;

struct Args {
    const uint8_t *packed;
    const int8_t *C;
    const __nv_bfloat16 *cs;
    const int8_t *xq;
    const float *xscale;
    int M, N, K;
    int R;        // row ranges (CTAs along N)
    int kcta;     // K columns per CTA (a multiple of STAGE_K, at most MAX_KCTA)
    __nv_bfloat16 *out;
    int32_t *acc;
    int32_t *part;   // int32 partials [splits][M][N] when K is split, else nullptr
    int *status;
};

__device__ __forceinline__ uint32_t bf16_pair(int lo, int hi)
{
    return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn((float)lo)) |
           ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn((float)hi)) << 16);
}

__device__ __forceinline__ void tma_box(uint32_t dst, const CUtensorMap *map, int x, int y, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            dst),
        "l"((uint64_t)map), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void mma16816(float (&d)[4], const uint4 &a, uint32_t b0, uint32_t b1)
{
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a.x), "r"(a.y), "r"(a.z), "r"(a.w), "r"(b0), "r"(b1));
}

template <int MT>
__global__ __launch_bounds__(THREADS, 1) void skinny_kernel(const __grid_constant__ CUtensorMap tm_pk, Args a)
{
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ int8_t Cv[96];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const int rr = (int)(blockIdx.x % (unsigned)a.R), sp = (int)(blockIdx.x / (unsigned)a.R);
    const int G = (a.N + 2) / 3;
    const int row0 = rr * ROWS_PER_CTA + warp * GPW;   // this warp's first packed row
    const int k0 = sp * a.kcta;
    const int klen = min(a.kcta, a.K - k0);
    const int nst = (klen + STAGE_K - 1) / STAGE_K;

    // ---- shared layout: 64 KiB-aligned table window, rings below it where they
    // fit, the rest of the rings and the activation fragments above it --------
    const uint32_t dyn = smem_addr(smem);
    const uint32_t bars = (dyn + 7) & ~7u;                       // WARPS * DEPTH barriers
    const uint32_t lo = (bars + WARPS * DEPTH * 8 + 1023) & ~1023u;   // swizzle atoms: 1 KiB aligned
    const uint32_t lut = wide_lut_window(lo);
    const int fit = lut > lo ? (int)((lut - lo) / RING_BYTES) : 0;
    const int nbelow = fit < WARPS ? fit : WARPS;
    const uint32_t hi = lut + kWideLutBytes;
    const uint32_t ring = warp < nbelow ? lo + warp * RING_BYTES : hi + (warp - nbelow) * RING_BYTES;
    const uint32_t act = hi + (WARPS - nbelow) * RING_BYTES;
    if (act + ACT_BYTES > dyn + DYN_SMEM || lo + nbelow * RING_BYTES > lut) {   // host never asks for this
        if (threadIdx.x == 0 && a.status)
            atomicExch(a.status, -3);
        return;
    }
    const uint32_t bar0 = bars + warp * DEPTH * 8;

    // Global loads first, all in flight together: the table bytes and this
    // thread's activation codes (converted to fragments below).
    int8_t cval = 0;
    if (threadIdx.x < 96)
        cval = a.C[threadIdx.x];
    constexpr int PER_THREAD = (MAX_KCTA / 16) * MT * 32 / THREADS;
    const int nsteps = (klen + 15) / 16;
    uint32_t xa[PER_THREAD], xb[PER_THREAD];
#pragma unroll
    for (int j = 0; j < PER_THREAD; ++j) {
        const int i = threadIdx.x + j * THREADS;
        const int l = i & 31, mt = (i >> 5) % MT, s = (i >> 5) / MT;
        const int k = k0 + 16 * s + 4 * (l & 3);
        const int ra = 16 * mt + (l >> 2), rb = ra + 8;
        const bool ok = s < nsteps && k < a.K;   // K % 16 == 0: the four columns are in range
        xa[j] = (ok && ra < a.M) ? __ldg(reinterpret_cast<const unsigned int *>(a.xq + (size_t)ra * a.K + k)) : 0u;
        xb[j] = (ok && rb < a.M) ? __ldg(reinterpret_cast<const unsigned int *>(a.xq + (size_t)rb * a.K + k)) : 0u;
    }
    if (lane == 0)
        for (int s = 0; s < DEPTH; ++s)
            mbar_init(bar0 + s * 8, 1);
    if (threadIdx.x < 96)
        Cv[threadIdx.x] = cval;
    fence_proxy_async_smem();
    __syncthreads();

    // ---- ring: stage st holds columns [k0 + 256 st, +256) of the warp's 8 rows as
    // two 128-byte-swizzled boxes (rows past G and columns past K read as zero) --
    auto issue_stage = [&](int st) {
        if (lane == 0) {
            const int slot = st % DEPTH;
            const uint32_t b = bar0 + slot * 8;
            fence_proxy_async_smem();
            mbar_arrive_expect_tx(b, STAGE_BYTES);
            const int kk = k0 + st * STAGE_K;
            tma_box(ring + slot * STAGE_BYTES, &tm_pk, kk, row0, b);
            tma_box(ring + slot * STAGE_BYTES + GPW * BOX_K, &tm_pk, kk + BOX_K, row0, b);
        }
    };
    for (int st = 0; st < DEPTH && st < nst; ++st)
        issue_stage(st);

    // ---- wide table of bf16 triples: entry b of lane l at lut + 256 b + 8 l ----
    for (int i = threadIdx.x; i < kLutEntries * 2; i += THREADS) {
        const int e = i >> 1, half = i & 1;   // each thread: 16 lane copies of one entry
        const uint32_t w = expanded_entry(Cv, (uint32_t)e);
        const int w0 = (int8_t)(w & 0xFF), w1 = (int8_t)((w >> 8) & 0xFF), w2 = (int8_t)((w >> 16) & 0xFF);
        const uint32_t x = bf16_pair(w0, w1), y = bf16_pair(w2, 0);
#pragma unroll
        for (int pr = 0; pr < 8; ++pr)
            asm volatile("st.shared.v4.u32 [%0], {%1, %2, %1, %2};" ::"r"(lut + (uint32_t)e * 256u +
                                                                           (uint32_t)(half * 8 + pr) * 16u),
                         "r"(x), "r"(y)
                         : "memory");
    }
    // ---- activation fragments in k-permuted order: for step s and token tile mt,
    // lane (g, t) holds {a0, a1, a2, a3} = tokens (16mt + g, 16mt + g + 8) at
    // columns k0 + 16 s + 4t .. + 3 as bf16 pairs --------------------------------
#pragma unroll
    for (int j = 0; j < PER_THREAD; ++j) {
        const int i = threadIdx.x + j * THREADS;
        const uint4 v = make_uint4(bf16_pair((int8_t)(xa[j] & 0xFF), (int8_t)((xa[j] >> 8) & 0xFF)),
                                   bf16_pair((int8_t)(xb[j] & 0xFF), (int8_t)((xb[j] >> 8) & 0xFF)),
                                   bf16_pair((int8_t)((xa[j] >> 16) & 0xFF), (int8_t)(xa[j] >> 24)),
                                   bf16_pair((int8_t)((xb[j] >> 16) & 0xFF), (int8_t)(xb[j] >> 24)));
        asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(act + (uint32_t)i * 16u), "r"(v.x),
                     "r"(v.y), "r"(v.z), "r"(v.w)
                     : "memory");
    }
    __syncthreads();

    // ---- stream ------------------------------------------------------------------
    float d[MT][3][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int c = 0; c < 3; ++c)
#pragma unroll
            for (int j = 0; j < 4; ++j)
                d[mt][c][j] = 0.0f;
    const uint32_t lane_base = lut | (uint32_t)(lane << 3);
    bool timed_out = false;
    int st = 0;
    for (; st < nst; ++st) {
        const int slot = st % DEPTH;
        if (!mbar_wait_bounded(bar0 + slot * 8, (uint32_t)((st / DEPTH) & 1))) {
            timed_out = true;
            break;
        }
        // Plain C++ loads from shared memory (stage words, activation fragments) stay
        // behind the barrier wait above, and, like the table loads and the MMAs
        // (no volatile), can be interleaved across steps by the compiler.
        const unsigned char *stage = smem + (ring - dyn) + slot * STAGE_BYTES + g * BOX_K + t * 4;
        const uint4 *actp = reinterpret_cast<const uint4 *>(smem + (act - dyn)) + lane;
        const int steps = min(16, (klen - st * STAGE_K + 15) / 16);
#pragma unroll
        for (int s = 0; s < 16; ++s) {
            if (s < steps) {
                // row g, columns 16 s + 4t .. + 3 inside the swizzled atoms
                const uint32_t word =
                    *reinterpret_cast<const uint32_t *>(stage + (s >> 3) * (GPW * BOX_K) + (((s & 7) ^ g) << 4));
                uint32_t e[4][2];
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    asm("ld.shared.v2.u32 {%0, %1}, [%2];"
                        : "=r"(e[i][0]), "=r"(e[i][1])
                        : "r"(prmt(word, lane_base, 0x7604u | ((uint32_t)i << 4))));
                const uint32_t b0[3] = {prmt(e[0][0], e[1][0], 0x5410), prmt(e[0][0], e[1][0], 0x7632),
                                        prmt(e[0][1], e[1][1], 0x5410)};
                const uint32_t b1[3] = {prmt(e[2][0], e[3][0], 0x5410), prmt(e[2][0], e[3][0], 0x7632),
                                        prmt(e[2][1], e[3][1], 0x5410)};
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                    const uint4 af = actp[((st * 16 + s) * MT + mt) * 32];
#pragma unroll
                    for (int c = 0; c < 3; ++c)
                        mma16816(d[mt][c], af, b0[c], b1[c]);
                }
            }
        }
        __syncwarp();
        if (st + DEPTH < nst)
            issue_stage(st + DEPTH);
    }
    if (timed_out) {
        // never leave with copies in flight: the stages issued and not consumed
        for (int v = st; v < nst && v < st + DEPTH; ++v)
            mbar_wait_bounded(bar0 + (v % DEPTH) * 8, (uint32_t)((v / DEPTH) & 1));
        if (lane == 0)
            record_timeout(a.status);
        return;
    }

    // ---- epilogue: exact fp32 sums -> int32 -> partials or the output ---------------
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int c = 0; c < 3; ++c)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int tok = 16 * mt + g + ((j & 2) ? 8 : 0);
                const int grp = row0 + 2 * t + (j & 1);
                const int ch = 3 * grp + c;
                if (tok >= a.M || grp >= G || ch >= a.N)
                    continue;
                const int v = __float2int_rn(d[mt][c][j]);
                const size_t idx = (size_t)tok * a.N + ch;
                if (a.part)
                    a.part[(size_t)sp * a.M * a.N + idx] = v;
                else if (a.acc)
                    a.acc[idx] = v;
                else
                    a.out[idx] = epilogue_bf16(v, a.xscale[tok], a.cs[ch]);
            }
}

}  // namespace sk

// K split: at most 1024 columns per CTA (exactness), a multiple of the 256-column
// ring stage, and enough splits for the row ranges to fill the GPU.
static void skinny_plan(int N, int K, int sms, int &R, int &kcta, int &splits)
{
    const int G = (N + 2) / 3;
    R = (G + sk::ROWS_PER_CTA - 1) / sk::ROWS_PER_CTA;
    int want = sms / R;
    if (want < 1)
        want = 1;
    const int min_splits = (K + sk::MAX_KCTA - 1) / sk::MAX_KCTA;
    if (want < min_splits)
        want = min_splits;
    kcta = (K + want - 1) / want;
    kcta = (kcta + sk::STAGE_K - 1) / sk::STAGE_K * sk::STAGE_K;
    if (kcta > sk::MAX_KCTA)
        kcta = sk::MAX_KCTA;
    splits = (K + kcta - 1) / kcta;
}

bool skinny_supported(int M)
{
    return M >= 1 && M <= 16 * sk::MAX_MT;
}

size_t skinny_workspace_bytes(int M, int N, int K)
{
    int R, kcta, splits;
    skinny_plan(N, K, device_sm_count(), R, kcta, splits);
    return splits > 1 ? (size_t)splits * M * N * 4 + 256 : 0;
}

cudaError_t launch_skinny(const LinearArgs &a, cudaStream_t stream)
{
    if (!skinny_supported(a.M))
        return cudaErrorInvalidValue;
    auto encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(tensor_map_encoder_fn());
    if (!encode)
        return cudaErrorNotSupported;
    CUtensorMap tm_pk;
    const cuuint64_t dims[2] = {(cuuint64_t)a.K, (cuuint64_t)((a.N + 2) / 3)};
    const cuuint64_t strides[1] = {(cuuint64_t)a.K};
    const cuuint32_t box[2] = {sk::BOX_K, sk::GPW}, es[2] = {1, 1};
    if (encode(&tm_pk, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(a.packed), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    const int sms = device_sm_count();
    int R, kcta, splits;
    skinny_plan(a.N, a.K, sms, R, kcta, splits);
    int32_t *part = nullptr;
    if (splits > 1) {
        if (!a.ws || a.ws_bytes < skinny_workspace_bytes(a.M, a.N, a.K))
            return cudaErrorInvalidValue;
        part = reinterpret_cast<int32_t *>(((uintptr_t)a.ws + 255) & ~(uintptr_t)255);
    }
    sk::Args k;
    k.packed = a.packed;
    k.C = a.C;
    k.cs = a.cs;
    k.xq = a.xq;
    k.xscale = a.xscale;
    k.M = a.M;
    k.N = a.N;
    k.K = a.K;
    k.R = R;
    k.kcta = kcta;
    k.out = a.out;
    k.acc = a.acc;
    k.part = part;
    k.status = a.status;
    const long ctas = (long)R * splits;
    if (ctas > 0x7FFFFFFFL)
        return cudaErrorInvalidValue;
    cudaError_t e;
    if (a.M <= 16) {
        e = cudaFuncSetAttribute(sk::skinny_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, sk::DYN_SMEM);
        if (e != cudaSuccess)
            return e;
        sk::skinny_kernel<1><<<(unsigned)ctas, sk::THREADS, sk::DYN_SMEM, stream>>>(tm_pk, k);
    } else {
        e = cudaFuncSetAttribute(sk::skinny_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, sk::DYN_SMEM);
        if (e != cudaSuccess)
            return e;
        sk::skinny_kernel<2><<<(unsigned)ctas, sk::THREADS, sk::DYN_SMEM, stream>>>(tm_pk, k);
    }
    e = cudaGetLastError();
    if (e != cudaSuccess || splits == 1)
        return e;
    return launch_splitk_finalize(part, splits, a, stream);
}

}  // namespace s3d8
