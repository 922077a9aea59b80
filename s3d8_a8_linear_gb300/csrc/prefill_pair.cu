// Prefill-regime S3D8 linear on SM pairs: tcgen05.mma.cta_group::2.
//
// Same exact scheme as the one-SM kernel in prefill_tc.cu (bf16 x bf16 -> fp32
// per 1024-column chunk, drained into int32; weights pre-expanded to bf16 [N, K]),
// but a cluster of two CTAs on two SMs computes a 256-token x 256-channel tile
// (the weights are bf16 rows here, so the tile need not hold whole packed
// groups): CTA r of the pair holds activation rows 128 r .. 128 r + 127 and
// weight rows 128 r .. 128 r + 127 of the tile in its shared memory, the even
// CTA issues M = 256, N = 256 MMAs that read both CTAs' halves, and each CTA's
// tensor memory receives its own 128 rows of the accumulator.  Per SM and K
// block the bulk copies bring 32 KB, where a one-SM 128 x 256 tile would need 48.
//
// Roles (16 warps per CTA):
//   warp 0       bulk tensor copies of this CTA's halves into a 7-stage ring (32 KB stages),
//                completing on the even CTA's barrier (cta_group::2 copies);
//   warp 1       TMEM allocation for the pair (both CTAs, cta_group::2); in the
//                even CTA the MMA issuer (one thread);
//   warps 8-15   drain this CTA's accumulator rows per chunk into int32 (setmaxnreg
//                176) and write the epilogue; they release the TMEM buffer to
//                the even CTA's MMA issuer (16 arrivals: 8 warps x 2 CTAs).
// MMA completion is committed to the barriers of both CTAs at once (multicast).
// Every mbarrier wait is bounded; both CTAs reach the closing cluster barrier on
// every path, so neither leaves while the other may still touch its memory.
#include "tcgen05.cuh"

namespace s3d8 {

namespace tc {

constexpr int PAIR_STAGES = 7;
constexpr int PAIR_BM = 2 * BM;                    // 256 tokens per pair tile
constexpr int PAIR_BN = 256;                       // channels per pair tile at most (bf16 rows: no group alignment)
constexpr int B_HALF = PAIR_BN / 2;                // weight rows per CTA at most
constexpr int B_HALF_BYTES = B_HALF * BK * 2;      // 16 KiB stage slot
constexpr int PH = PAIR_BN / 2;                    // accumulator columns per drain thread at most

struct PairParams {
    Params p;
    int bn;   // channels per tile: 128, 192 or 256
};
constexpr int PAIR_OFF_B = PAIR_STAGES * A_BYTES;
constexpr int PAIR_OFF_BARS = PAIR_OFF_B + PAIR_STAGES * B_HALF_BYTES;
constexpr int PAIR_NBARS = 2 * PAIR_STAGES + 4;
constexpr int PAIR_SMEM_BYTES = 1024 + PAIR_OFF_BARS + PAIR_NBARS * 8 + 16;
static_assert(B_HALF_BYTES % 1024 == 0 && PAIR_OFF_B % 1024 == 0, "swizzled tiles 1024-aligned");
static_assert(PAIR_SMEM_BYTES + 1024 <= 232448, "shared memory budget");
static_assert(B_HALF % 8 == 0 && PAIR_BN % 16 == 0 && PAIR_BN <= 256, "M = 256 MMAs need N a multiple of 16");

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(THREADS, 1)
    prefill_pair_kernel(const __grid_constant__ CUtensorMap tm_act, const __grid_constant__ CUtensorMap tm_w,
                        PairParams pp)
{
    const Params &p = pp.p;
    const int bn = pp.bn, bh = bn / 2;   // tile channels; per CTA and per drain thread
    constexpr int S = PAIR_STAGES;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    unsigned char *smem = smem_raw + (base - raw);
    const uint32_t bars = base + PAIR_OFF_BARS;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + PAIR_OFF_BARS + PAIR_NBARS * 8);
    // l_full[S] (even CTA: both CTAs' copies of the stage landed), l_empty[S] (the
    // pair's MMAs are done with the stage), acc_full[2] (chunk in TMEM),
    // acc_empty[2] (even CTA: both CTAs drained it)
    const uint32_t l_full = bars, l_empty = l_full + 8 * S;
    const uint32_t acc_full = l_empty + 8 * S, acc_empty = acc_full + 16;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();
    const int cid = (int)blockIdx.x >> 1, nclusters = (int)gridDim.x >> 1;
    const int mtiles = (p.M + PAIR_BM - 1) / PAIR_BM;
    const int ntiles = (p.N + bn - 1) / bn;
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
        T.m0 = mt * PAIR_BM;
        T.kbase = T.split * p.kb_per_split;
        T.nk = min(p.kb_per_split, nk_all - T.kbase);
        return T;
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(l_full + 8 * s, 1);
            mbar_init(l_empty + 8 * s, 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(acc_full + 8 * i, 1);
            mbar_init(acc_empty + 8 * i, 16);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(
                         smem_addr(tmem_slot))
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    cluster_sync();   // both CTAs' barriers initialised, the pair's TMEM allocated
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    bool timed_out = false;
    pdl_launch_dependents();   // the split-K finish may be scheduled; it waits for this grid

    if (warp < DRAIN_WARP0) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 80;");
        if (warp == 0) {
            // ---- this CTA's halves of every K block, by bulk tensor copy; both CTAs'
            // copies complete on the even CTA's l_full, which expects both halves
            {
                pdl_wait();   // the activation codes and bf16 weights come from earlier kernels
                const uint32_t full0 = map_to_rank(l_full, 0);
                int issued = 0;
                for (int t = cid; t < total && !timed_out; t += nclusters) {
                    const Tile T = tile_of(t);
                    for (int kb = 0; kb < T.nk; ++kb) {
                        const int s = issued % S;
                        if (issued >= S && !warp_wait(l_empty + 8 * s, ((issued / S) - 1) & 1)) {
                            timed_out = true;
                            break;
                        }
                        if (rank == 0)
                            mbar_arrive_expect_tx_elect(l_full + 8 * s, 2 * (A_BYTES + bh * BK * 2));
                        const int kx = (T.kbase + kb) * BK;
                        tma_2d_pair_elect(base + s * A_BYTES, &tm_act, kx, T.m0 + (int)rank * BM, full0 + 8 * s);
                        tma_2d_pair_elect(base + PAIR_OFF_B + s * B_HALF_BYTES, &tm_w, kx,
                                          T.nt * bn + (int)rank * bh, full0 + 8 * s);
                        ++issued;
                    }
                }
                // never leave with copies in flight: the last stages' MMAs (which
                // needed every copy) have completed
                for (int v = issued - S < 0 ? 0 : issued - S; v < issued; ++v)
                    if (!warp_wait(l_empty + 8 * (v % S), (v / S) & 1))
                        timed_out = true;
            }
        } else if (warp == 1 && rank == 0) {
            // ---- MMA issuer of the pair: the whole warp runs the loop so that the
            // descriptors stay warp-uniform; one elected lane issues -----------------
            {
                int g = 0, gc = 0;
                const uint32_t idesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(bn >> 3) << 17) |
                                       ((uint32_t)(PAIR_BM >> 4) << 24);
                for (int t = cid; t < total && !timed_out; t += nclusters) {
                    const Tile T = tile_of(t);
                    for (int kb = 0; kb < T.nk; ++kb) {
                        const int s = g % S;
                        const int c = gc + kb / CHUNK_BLOCKS, kin = kb % CHUNK_BLOCKS;
                        const uint32_t d = tmem + (uint32_t)((c & 1) * 256);
                        if (kin == 0 && c >= 2 && !warp_wait(acc_empty + 8 * (c & 1), ((c >> 1) - 1) & 1)) {
                            timed_out = true;
                            break;
                        }
                        if (!warp_wait(l_full + 8 * s, (g / S) & 1)) {
                            timed_out = true;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t a = base + s * A_BYTES, b = base + PAIR_OFF_B + s * B_HALF_BYTES;
#pragma unroll
                        for (int kk = 0; kk < BK / 16; ++kk)
                            mma_f16_pair_elect(d, sw128_desc(a + kk * 32), sw128_desc(b + kk * 32), idesc,
                                                (kin | kk) ? 1u : 0u);
                        mma_commit_pair_elect(l_empty + 8 * s);
                        if (kin == CHUNK_BLOCKS - 1 || kb == T.nk - 1)
                            mma_commit_pair_elect(acc_full + 8 * (c & 1));
                        ++g;
                    }
                    gc += (T.nk + CHUNK_BLOCKS - 1) / CHUNK_BLOCKS;
                }
                // the tensor core must be done with both CTAs' memory before exit
                if (g > 0 && !warp_wait(l_empty + 8 * ((g - 1) % S), ((g - 1) / S) & 1))
                    timed_out = true;
            }
        }
    } else {
        // ---- drain this CTA's accumulator rows, then the epilogue -----------------
        asm volatile("setmaxnreg.inc.sync.aligned.u32 176;");
        const int q = warp & 3;
        const int h = (warp - DRAIN_WARP0) >> 2;
        const uint32_t release = rank == 0 ? acc_empty : map_to_rank(acc_empty, 0);
        int32_t acc[PH];
        int gc = 0;
        for (int t = cid; t < total && !timed_out; t += nclusters) {
            const Tile T = tile_of(t);
            const int nch = (T.nk + CHUNK_BLOCKS - 1) / CHUNK_BLOCKS;
#pragma unroll
            for (int i = 0; i < PH; ++i)
                acc[i] = 0;
            for (int c = gc; c < gc + nch; ++c) {
                if (!mbar_wait_bounded(acc_full + 8 * (c & 1), (c >> 1) & 1)) {
                    timed_out = true;
                    break;
                }
                tc_fence_after();
                const uint32_t ta = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)((c & 1) * 256 + h * bh);
#pragma unroll
                for (int i = 0; i < PH / 32; ++i) {
                    if (i * 32 < bh) {   // bh is uniform and a multiple of 32: the warp loads together
                        float v[4][8];
#pragma unroll
                        for (int u = 0; u < 4; ++u)
                            tmem_ld8(ta + i * 32 + u * 8, v[u]);
                        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
                        for (int u = 0; u < 4; ++u)
#pragma unroll
                            for (int j = 0; j < 8; ++j)
                                acc[i * 32 + u * 8 + j] += __float2int_rn(v[u][j]);
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive_remote(release + 8 * (c & 1));
            }
            gc += nch;
            const int row = T.m0 + (int)rank * BM + 32 * q + lane;
            if (!timed_out && row < p.M)
                store_tile_row<PH>(p, T.split, row, T.nt * bn + h * bh, acc, bh);
        }
    }
    if (timed_out)
        record_timeout(p.status);
    tc_fence_before();
    cluster_sync();   // no CTA leaves while its pair may still signal or read it
    tc_fence_after();
    if (warp == 1)
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, 512;" ::"r"(tmem) : "memory");
}

}  // namespace tc

// Channels per pair tile: 256, 192 or 128 (each CTA's half then drains in whole
// groups of 32 columns), the one that minimises the rounds of tiles the SM
// pairs run, time per tile taken as proportional to the width plus a fixed 192
// columns' worth, the widest on a tie.  (With 64 columns' worth the model chose
// 192-channel tiles for gate/up at 1536 and 1792 tokens, measured 4% slower
// than 256; with 192 it picks the faster width on both 11B shapes at 1280,
// 1536 and 1792 tokens.)
static int pair_tile_n(int M, int N, int nsplit)
{
    const long pairs = device_sm_count() / 2 > 0 ? device_sm_count() / 2 : 1;
    const long mt = (long)((M + tc::PAIR_BM - 1) / tc::PAIR_BM) * nsplit;
    int best = tc::PAIR_BN;
    long best_cost = -1;
    for (int bn = tc::PAIR_BN; bn >= 128; bn -= 64) {
        const long tiles = mt * ((N + bn - 1) / bn);
        const long cost = (tiles + pairs - 1) / pairs * (bn + 192);
        if (best_cost < 0 || cost < best_cost) {
            best = bn;
            best_cost = cost;
        }
    }
    return best;
}

// SM-pair tensor-core GEMM on pre-expanded bf16 weights: act is the bf16 copy of
// the activation codes [M, K], wdec the bf16 weights [N, K] (both in the
// workspace), part the split-K partials or null.
cudaError_t launch_prefill_pair(const LinearArgs &a, const __nv_bfloat16 *act, const __nv_bfloat16 *wdec,
                                int32_t *part, int nsplit, int kbps, cudaStream_t stream)
{
    using namespace tc;
    auto encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(tensor_map_encoder_fn());
    if (!encode)
        return cudaErrorNotSupported;
    CUtensorMap tm_act, tm_w;
    const cuuint32_t es[2] = {1, 1};
    const cuuint64_t dA[2] = {(cuuint64_t)a.K, (cuuint64_t)a.M};
    const cuuint64_t sA[1] = {(cuuint64_t)a.K * 2};
    const cuuint32_t boxA[2] = {BK, BM};
    const cuuint64_t dW[2] = {(cuuint64_t)a.K, (cuuint64_t)a.N};
    const cuuint64_t sW[1] = {(cuuint64_t)a.K * 2};
    const int bn = pair_tile_n(a.M, a.N, nsplit);
    const cuuint32_t boxW[2] = {BK, (cuuint32_t)(bn / 2)};
    if (encode(&tm_act, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<__nv_bfloat16 *>(act), dA, sA, boxA, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS ||
        encode(&tm_w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<__nv_bfloat16 *>(wdec), dW, sW, boxW, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(prefill_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         PAIR_SMEM_BYTES);
    if (e != cudaSuccess)
        return e;
    PairParams pp;
    pp.p = make_params(a, nsplit, kbps, part);
    pp.bn = bn;
    const long tiles = (long)((a.M + PAIR_BM - 1) / PAIR_BM) * (long)((a.N + bn - 1) / bn) * nsplit;
    if (tiles > 0x7FFFFFFFL)
        return cudaErrorInvalidValue;
    long pairs = device_sm_count() / 2;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(2 * pairs));
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = PAIR_SMEM_BYTES;
    int fit = 0;   // pairs the GPU can hold at once (not every SM may find a partner)
    if (cudaOccupancyMaxActiveClusters(&fit, prefill_pair_kernel, &cfg) == cudaSuccess && fit > 0 && fit < pairs)
        pairs = fit;
    (void)cudaGetLastError();
    const long clusters = tiles < pairs ? tiles : pairs;
    return launch_pdl(prefill_pair_kernel, dim3((unsigned)(2 * clusters)), dim3(THREADS), (size_t)PAIR_SMEM_BYTES,
                      stream, tm_act, tm_w, pp);
}

}  // namespace s3d8
