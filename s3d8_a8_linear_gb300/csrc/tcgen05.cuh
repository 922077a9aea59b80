// tcgen05 / bulk-tensor-copy building blocks and tile constants shared by the
// tensor-core linear kernels (one-SM tiles in prefill_tc.cu, SM-pair tiles in
// prefill_pair.cu), written as inline PTX for sm_103a.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "launch.h"
#include "tma.cuh"

namespace s3d8 {

namespace tc {

constexpr int BM = 128;                  // tokens per tile
constexpr int GROUPS = 80;               // packed rows per tile
constexpr int BN = 3 * GROUPS;           // 240 channels per tile
constexpr int BK = 64;                   // K per block (128 bytes of bf16)
constexpr int LSTAGES = 6;               // ring of loaded tiles (A + packed bytes)
constexpr int BSTAGES = 2;               // ring of decoded weight tiles
constexpr int CHUNK_BLOCKS = 16;         // 16 x 64 = 1024 columns per exact chunk
constexpr int A_BYTES = BM * BK * 2;     // 16 KiB
constexpr int B_BYTES = BN * BK * 2;     // 30 KiB
constexpr int P_BYTES = GROUPS * BK;     // 5 KiB packed bytes
constexpr int LUT_COPIES = 16;
constexpr int LUT_BYTES = kLutEntries * LUT_COPIES * 8;   // 32 KiB
constexpr int OFF_A = 0;
constexpr int OFF_B = OFF_A + LSTAGES * A_BYTES;
constexpr int OFF_P = OFF_B + BSTAGES * B_BYTES;
constexpr int OFF_LUT = OFF_P + LSTAGES * P_BYTES;
constexpr int OFF_BARS = OFF_LUT + LUT_BYTES;
constexpr int NBARS = 2 * LSTAGES + 2 * BSTAGES + 4;
constexpr int SMEM_BYTES = 1024 + OFF_BARS + NBARS * 8 + 16;
constexpr int THREADS = 16 * 32;
constexpr int DECODERS = 14 * 32;   // warps 2-15 all decode (8-15 also drain)
constexpr int DRAIN_WARP0 = 8;
constexpr int HALF = BN / 2;             // 120 columns per epilogue thread

static_assert(A_BYTES % 1024 == 0 && B_BYTES % 1024 == 0 && OFF_B % 1024 == 0,
              "swizzled tiles must stay 1024-aligned");
static_assert(OFF_P % 128 == 0 && P_BYTES % 128 == 0, "packed tiles 128-byte aligned");
static_assert(SMEM_BYTES + 1024 <= 232448, "shared memory budget");

__device__ __forceinline__ uint64_t sw128_desc(uint32_t a)
{
    // tcgen05 shared-memory descriptor: start >> 4, LBO 16 B (unused for swizzled
    // K-major), SBO 1024 B between 8-row atoms, version 1, 128-byte swizzle.
    return (uint64_t)((a & 0x3FFFFu) >> 4) | (1ull << 16) | ((uint64_t)(1024 >> 4) << 32) |
           (1ull << 46) | (2ull << 61);
}

// Warp-wide forms: the whole warp executes them convergently (so operands built
// from warp-uniform values can stay in uniform registers) and one lane, chosen
// by elect.sync, performs the operation.
__device__ __forceinline__ void mma_bf16_elect(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc)
{
    asm volatile(
        "{\n.reg .pred p, e;\nsetp.ne.b32 p, %4, 0;\nelect.sync _|e, 0xffffffff;\n"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}

__device__ __forceinline__ void mma_commit_elect(uint32_t bar)
{
    asm volatile(
        "{\n.reg .pred e;\nelect.sync _|e, 0xffffffff;\n"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n}\n" ::"r"(bar)
        : "memory");
}

__device__ __forceinline__ void tma_2d_elect(uint32_t dst, const CUtensorMap *map, int x, int y, uint32_t bar)
{
    asm volatile(
        "{\n.reg .pred e;\nelect.sync _|e, 0xffffffff;\n"
        "@e cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];\n}\n" ::"r"(dst),
        "l"((uint64_t)map), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx_elect(uint32_t bar, uint32_t bytes)
{
    asm volatile(
        "{\n.reg .pred e;\nelect.sync _|e, 0xffffffff;\n"
        "@e mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n}\n" ::"r"(bar),
        "r"(bytes)
        : "memory");
}

// Programmatic dependent launch: let the next kernel on the stream be scheduled,
// and wait until the kernel before this one has completed (its memory visible).
__device__ __forceinline__ void pdl_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void pdl_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Bounded wait taken by a whole warp: true only if every lane saw the phase.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity)
{
    return __all_sync(0xffffffffu, mbar_wait_bounded(bar, parity));
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float (&v)[8])
{
    uint32_t r[8];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
                   "=r"(r[7])
                 : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 8; ++i)
        v[i] = __uint_as_float(r[i]);
}

// bf16 bits of a small integer (exact: |v| <= 127 needs 7 significant bits).
__device__ __forceinline__ uint32_t bf16_bits_of(int v)
{
    return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn((float)v));
}

// Expands this thread's share of an NG x 64 packed tile (units u = t, t + nthr, ...;
// one unit = one group's 8 bytes at one 16-byte column chunk) into the
// 128-byte-swizzled K-major bf16 tile: element (n, k) at n * 128 +
// ((k / 8) ^ (n % 8)) * 16 + (k % 8) * 2.
// The table holds COPIES copies of each 8-byte entry side by side (entry b of
// copy c at 8 (COPIES b + c)); `lut_lane` = table + 8 (lane % COPIES).
template <int NG = GROUPS, int COPIES = LUT_COPIES>
__device__ __forceinline__ void decode_tile(uint32_t ptile, uint32_t btile, uint32_t lut_lane, int t, int nthr)
{
    for (int u = t; u < NG * 8; u += nthr) {
        const int gl = u >> 3, j = u & 7;   // group, 16-byte chunk (8 k)
        uint32_t pk0, pk1;
        asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(pk0), "=r"(pk1) : "r"(ptile + gl * 64 + j * 8));
        uint2 e[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t byte = ((i < 4 ? pk0 : pk1) >> (8 * (i & 3))) & 0xFFu;
            asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];"
                         : "=r"(e[i].x), "=r"(e[i].y)
                         : "r"(lut_lane + byte * (COPIES * 8)));
        }
        uint32_t w[3][4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            w[0][q] = prmt(e[2 * q].x, e[2 * q + 1].x, 0x5410);
            w[1][q] = prmt(e[2 * q].x, e[2 * q + 1].x, 0x7632);
            w[2][q] = prmt(e[2 * q].y, e[2 * q + 1].y, 0x5410);
        }
#pragma unroll
        for (int d = 0; d < 3; ++d) {
            const int n = 3 * gl + d;
            const uint32_t addr = btile + n * 128 + (((uint32_t)j ^ (uint32_t)(n & 7)) << 4);
            asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(w[d][0]), "r"(w[d][1]),
                         "r"(w[d][2]), "r"(w[d][3])
                         : "memory");
        }
    }
}

// Packed fp16 subtract a - b (two lanes), round to nearest.
__device__ __forceinline__ uint32_t f16x2_sub(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity)
{
    uint32_t done;
    asm volatile(
        "{\n.reg .pred p;\n"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        "selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}

struct Params {
    int M, N, K;
    const int8_t *C;
    const __nv_bfloat16 *cs;
    const float *xscale;
    __nv_bfloat16 *out;
    int32_t *acc;
    int *status;
    int vec_out;        // out / acc rows may be written with 16-byte stores
    int nsplit;         // K is split into nsplit ranges of kb_per_split 64-column blocks
    int kb_per_split;
    int32_t *part;      // with nsplit > 1: int32 partial sums [nsplit][M][N]
    int vec_part;       // partial rows may be written with 16-byte stores
};

// Writes one accumulator row segment of a tile: the int32 sums (to the split-K
// partials or the raw int32 output) or the bf16 epilogue (x_s * acc) * W_s.
// Columns nbase .. nbase + W - 1 of row `row`; columns >= N are skipped.
// With a width `w` < W only the first w columns are written.
template <int W = HALF>
__device__ __forceinline__ void store_tile_row(const Params &p, int split, int row, int nbase,
                                               const int32_t (&acc)[W], int w = W)
{
    static_assert(W % 8 == 0, "vector stores take 8 columns");
    if (!dcheck(p.status, row >= 0 && row < p.M && nbase >= 0 && (p.part == nullptr || split < p.nsplit)))
        return;
    // whole 8-column groups inside N take the vector stores (w is a multiple of 8
    // for every tile width the kernels use; narrower tiles skip the groups >= w)
    const bool full = w % 8 == 0 && nbase + w <= p.N;
    int32_t *accp = p.part ? p.part + (size_t)split * p.M * p.N : p.acc;
    const bool vec_acc = p.part ? p.vec_part : p.vec_out;
    if (accp) {
        int32_t *dst = accp + (size_t)row * p.N + nbase;
        if (full && vec_acc) {
#pragma unroll
            for (int i = 0; i < W; i += 4)
                if (i < w)
                    *reinterpret_cast<int4 *>(dst + i) = make_int4(acc[i], acc[i + 1], acc[i + 2], acc[i + 3]);
        } else {
#pragma unroll
            for (int i = 0; i < W; ++i)
                if (i < w && nbase + i < p.N)
                    dst[i] = acc[i];
        }
        return;
    }
    const float xs = p.xscale[row];
    __nv_bfloat16 *dst = p.out + (size_t)row * p.N + nbase;
    if (full && p.vec_out) {
#pragma unroll
        for (int i = 0; i < W; i += 8) {
            if (i >= w)
                break;
            uint32_t o[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const __nv_bfloat16 lo = epilogue_bf16(acc[i + 2 * j], xs, p.cs[nbase + i + 2 * j]);
                const __nv_bfloat16 hi = epilogue_bf16(acc[i + 2 * j + 1], xs, p.cs[nbase + i + 2 * j + 1]);
                o[j] = (uint32_t)__bfloat16_as_ushort(lo) | ((uint32_t)__bfloat16_as_ushort(hi) << 16);
            }
            *reinterpret_cast<uint4 *>(dst + i) = make_uint4(o[0], o[1], o[2], o[3]);
        }
    } else {
#pragma unroll
        for (int i = 0; i < W; ++i)
            if (i < w && nbase + i < p.N)
                dst[i] = epilogue_bf16(acc[i], xs, p.cs[nbase + i]);
    }
}

// Launches `kernel` with programmatic stream serialization: it may be scheduled
// while the previous kernel on the stream finishes, and must call pdl_wait()
// before touching anything that kernel writes.
template <typename Kernel, typename... Args>
inline cudaError_t launch_pdl(Kernel kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                              Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// ---- SM-pair (cluster of two CTAs) building blocks, shared by the two pair
// kernels (prefill_pair.cu, prefill_fused.cu) ---------------------------------

__device__ __forceinline__ uint32_t cluster_rank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// shared::cluster address of the same shared-memory offset in CTA `rank`
__device__ __forceinline__ uint32_t map_to_rank(uint32_t addr, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

__device__ __forceinline__ void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Arrive on a barrier of another CTA of the cluster (default release semantics
// at CTA scope, as for a local arrive; the tensor-core side is ordered by the
// tcgen05 fences around it).
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr)
{
    asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// Warp-wide pair forms (see the one-SM forms in tcgen05.cuh): the MMA with
// M = 256 across the pair; the commit arrives on the barrier at offset `bar` in
// both CTAs; the tensor copy completes on `bar`, which may be the barrier of the
// other CTA of the pair.
// tcgen05.mma.cta_group::2.kind::f16 (bf16 or fp16 operands, as the
// instruction descriptor says) issued by one elected lane of the warp.
__device__ __forceinline__ void mma_f16_pair_elect(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc)
{
    asm volatile(
        "{\n.reg .pred p, e;\nsetp.ne.b32 p, %4, 0;\nelect.sync _|e, 0xffffffff;\n"
        "@e tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}

__device__ __forceinline__ void mma_commit_pair_elect(uint32_t bar)
{
    const uint16_t mask = 0x3;
    asm volatile(
        "{\n.reg .pred e;\nelect.sync _|e, 0xffffffff;\n"
        "@e tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;\n}\n" ::"r"(
            bar),
        "h"(mask)
        : "memory");
}

__device__ __forceinline__ void tma_2d_pair_elect(uint32_t dst, const CUtensorMap *map, int x, int y, uint32_t bar)
{
    asm volatile(
        "{\n.reg .pred e;\nelect.sync _|e, 0xffffffff;\n"
        "@e cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, "
        "{%2, %3}], [%4];\n}\n" ::"r"(dst),
        "l"((uint64_t)map), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

inline Params make_params(const LinearArgs &a, int nsplit, int kbps, int32_t *part)
{
    Params p;
    p.M = a.M;
    p.N = a.N;
    p.K = a.K;
    p.C = a.C;
    p.cs = a.cs;
    p.xscale = a.xscale;
    p.out = a.out;
    p.acc = a.acc;
    p.status = a.status;
    p.vec_out = a.acc ? ((a.N & 3) == 0 && ((uintptr_t)a.acc & 15) == 0)
                      : ((a.N & 7) == 0 && ((uintptr_t)a.out & 15) == 0);
    p.nsplit = nsplit;
    p.kb_per_split = kbps;
    p.part = part;
    p.vec_part = (a.N & 3) == 0;
    return p;
}

}  // namespace tc

void *tensor_map_encoder_fn();

}  // namespace s3d8
