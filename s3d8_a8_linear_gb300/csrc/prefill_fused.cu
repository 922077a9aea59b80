// Prefill-regime S3D8 linear on SM pairs with the S3D8 unpack inside the GEMM:
// tcgen05.mma.cta_group::2 kind::f16 on fp16 operands (every int8 value is an
// fp16 value) with exact fp32 chunks, like the one-SM kernel in prefill_tc.cu,
// and no 16-bit copy of the weights anywhere.
//
// A cluster of two CTAs on two SMs computes a 256-token x 240-channel tile:
// CTA r of the pair holds activation rows 128 r .. 128 r + 127 of the tile (by
// bulk tensor copy from the fp16 copy of the codes) and decodes packed rows
// 40 r .. 40 r + 39 of the tile's 80 (channels 120 r .. 120 r + 119) from
// packed bytes into its half of the fp16 weight tile; the even CTA issues
// M = 256, N = 240 MMAs that read both CTAs' halves, and each CTA's tensor
// memory receives its own 128 rows of the accumulator.  Per SM and K block the
// bulk copies bring 16 KiB of activations and 2.5 KiB of packed bytes.
//
// Roles (16 warps per CTA):
//   warp 0       bulk tensor copies, per K block, of this CTA's packed half
//                (completing on its own barrier) and activation half (cta_group::2
//                copy, completing on the even CTA's full barrier) into a ring of
//                6 or 5 stages (32 or 40 packed rows per CTA);
//   warp 1       TMEM allocation for the pair (both CTAs, cta_group::2); in the
//                even CTA the MMA issuer (one elected lane);
//   warps 3-6    decode (3-7 with 40 packed rows per CTA): two 8-byte units (one packed row, 8 columns) each per K block,
//                written into the 128-byte-swizzled K-major fp16 half of the
//                stage (one 4-byte lookup per packed byte in a lane-replicated
//                table of biased weights, a byte permute and a packed fp16
//                subtract per two weights); then a proxy fence (generic writes ->
//                the tensor core's async proxy) and an arrive on the even CTA's
//                full barrier, which completes with 1 + 2 x decoder warps
//                arrivals (the even CTA's copy-issuing lane, the decoders of
//                both CTAs) and both activation copies' bytes, so that the MMA
//                issuer waits and commits once per K block.  A decoder warp waits
//                on one barrier (the packed half landed) and arrives on one per
//                block: at ~100 cycles per barrier operation for a warp that has
//                nothing else to overlap them with, the earlier separate packed
//                ring (a wait for the packed half, a wait for the stage, two
//                arrives) spent ~460 of the ~780 cycles each block took;
//   warps 8-15   drain this CTA's accumulator rows per chunk into int32
//                (setmaxnreg 176) and write the epilogue.  They release the TMEM
//                buffer to the even CTA's MMA issuer (16 arrivals: 8 warps x 2
//                CTAs).  (Decoding in these warps too, between drains, made them
//                the slowest decoders: the 120 sums they hold leave the decode
//                too few registers.)
// MMA completion is committed to the barriers of both CTAs at once
// (multicast).  Every mbarrier wait is bounded; both CTAs reach the closing
// cluster barrier on every path, so neither leaves while the other may still
// touch its memory.
#include "tcgen05.cuh"

namespace s3d8 {

namespace tc {

constexpr int FUSED_LUT_BYTES = kLutEntries * 32 * 4;  // 32 KiB: one 4-byte entry per byte and lane
constexpr int FUSED_BM = 2 * BM;                      // 256 tokens per pair tile

// The pair tile for G2 packed rows per CTA: 40 (256 tokens x 240 channels, five
// decoder warps, 120 columns per drain thread) or 32 (256 x 192, four decoder
// warps, 96 columns), whichever covers the matrix in fewer rounds of tiles
// over the SM pairs (fused_tile_groups).
template <int G2>
struct FusedTile {
    static constexpr int TILE_GROUPS = 2 * G2;                 // packed rows per pair tile
    static constexpr int BH = 3 * G2;                          // weight rows (channels) per CTA
    static constexpr int BN = 2 * BH;                          // channels per pair tile
    static constexpr int P_BYTES = G2 * BK;                    // packed bytes per stage
    static constexpr int B_BYTES = BH * BK * 2;                // decoded half tile
    static constexpr int DEC_WARPS = G2 / 8;                   // two 8-byte units per thread and K block
    static constexpr int DECODERS = DEC_WARPS * 32;
    // ring stages of activation half + packed half + decoded weight half, as
    // many as fit beside the table
    static constexpr int STAGES = G2 == 32 ? 6 : 5;
    __device__ static int decoder_index(int w) { return w >= 3 && w < 3 + DEC_WARPS ? w - 3 : -1; }
    static constexpr int NBARS = 3 * STAGES + 4;
    static constexpr int OFF_A = 0;
    static constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
    static constexpr int OFF_P = OFF_B + STAGES * B_BYTES;
    static constexpr int OFF_LUT = OFF_P + STAGES * P_BYTES;
    static constexpr int OFF_BARS = OFF_LUT + FUSED_LUT_BYTES;
    static constexpr int SMEM_BYTES = 1024 + OFF_BARS + NBARS * 8 + 16;
    static_assert(B_BYTES % 1024 == 0 && OFF_B % 1024 == 0 && A_BYTES % 1024 == 0, "swizzled tiles 1024-aligned");
    static_assert(OFF_P % 128 == 0 && P_BYTES % 128 == 0 && OFF_LUT % 16 == 0, "packed tiles aligned");
    static_assert(SMEM_BYTES + 1024 <= 232448, "shared memory budget");
    static_assert(BH % 24 == 0 && BN % 16 == 0 && BN <= 256, "M = 256 MMAs need N a multiple of 16");
    static_assert(2 * DECODERS == G2 * 8, "two decode units per decoder thread and K block");
    static_assert(DEC_WARPS >= 4 && DEC_WARPS <= 5, "four or five decoder warps (warps 3..7)");
};

// Decodes the units t and t + nthr (8-byte units: packed row u / 8, columns
// 8 (u % 8) .. + 7 of the K block) of a packed half into fp16 weights.  Each of
// the unit's 8 bytes is one table lookup [w0 + 128, w1 + 128, w2 + 128, 0x64];
// a byte permute of two lookups forms the fp16 pair 0x64xx (1024 + xx) of one
// channel for two adjacent columns, and a packed subtract of 1152 leaves the
// weights.  The 16 bytes of channel d (row n = 3 g + d of the half tile) are one
// 16-byte chunk of the 128-byte-swizzled K-major tile.
__device__ __forceinline__ void decode_units_f16(uint32_t ptile, uint32_t btile, uint32_t lut_lane, int t, int nthr)
{
    uint32_t pk[2][2];
    int gl[2], j[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int u = t + h * nthr;
        gl[h] = u >> 3;
        j[h] = u & 7;
        asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];"
                     : "=r"(pk[h][0]), "=r"(pk[h][1])
                     : "r"(ptile + gl[h] * 64 + j[h] * 8));
    }
    uint32_t L[2][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const uint32_t byte = prmt(pk[h][i >> 2], 0u, 0x4440u | (uint32_t)(i & 3));
            L[h][i] = lds_u32_nv(mad_lo_u32(byte, 128u, lut_lane));
        }
    constexpr uint32_t kBias = 0x64806480u;   // fp16 (1152, 1152)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        uint32_t w[3][4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            w[0][q] = f16x2_sub(prmt(L[h][2 * q], L[h][2 * q + 1], 0x7430u), kBias);
            w[1][q] = f16x2_sub(prmt(L[h][2 * q], L[h][2 * q + 1], 0x7531u), kBias);
            w[2][q] = f16x2_sub(prmt(L[h][2 * q], L[h][2 * q + 1], 0x7632u), kBias);
        }
#pragma unroll
        for (int d = 0; d < 3; ++d) {
            const int n = 3 * gl[h] + d;
            const uint32_t addr = btile + n * 128 + (((uint32_t)j[h] ^ (uint32_t)(n & 7)) << 4);
            asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(w[d][0]), "r"(w[d][1]),
                         "r"(w[d][2]), "r"(w[d][3])
                         : "memory");
        }
    }
}

template <int G2>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(THREADS, 1)
    prefill_fused_kernel(const __grid_constant__ CUtensorMap tm_act, const __grid_constant__ CUtensorMap tm_pk,
                        Params p)
{
    using F = FusedTile<G2>;
    constexpr int S = F::STAGES;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    unsigned char *smem = smem_raw + (base - raw);
    const uint32_t lut = base + F::OFF_LUT;
    const uint32_t bars = base + F::OFF_BARS;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + F::OFF_BARS + F::NBARS * 8);
    // full[S] (even CTA: both CTAs' activation halves of the stage landed and
    // both CTAs' decoded halves written: 1 + 2 x decoder warps arrivals and the
    // copies' bytes), empty[S] (the pair's MMAs are done with the stage; both
    // CTAs), p_full[S] (this CTA's packed half of the stage landed: its copy is
    // issued after empty, so the stage's decoded half is free too), acc_full[2]
    // (chunk in TMEM), acc_empty[2] (even CTA: both CTAs drained it).  The MMA
    // issuer waits and commits once per K block, a decoder warp waits once and
    // arrives once.
    const uint32_t full = bars, empty = full + 8 * S, p_full = empty + 8 * S;
    const uint32_t acc_full = p_full + 8 * S, acc_empty = acc_full + 16;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();
    const int cid = (int)blockIdx.x >> 1, nclusters = (int)gridDim.x >> 1;
    const int mtiles = (p.M + FUSED_BM - 1) / FUSED_BM;
    const int ntiles = ((p.N + 2) / 3 + F::TILE_GROUPS - 1) / F::TILE_GROUPS;
    const int nk_all = (p.K + BK - 1) / BK;
    const int total = mtiles * ntiles * p.nsplit;
    struct Tile {
        int m0, nt, split, kbase, nk;
    };
    // consecutive tile indices share the channel tile, so the pairs working at
    // one time read its packed bytes from L2
    auto tile_of = [&](int t) {
        Tile T;
        const int mt = t % mtiles, rest = t / mtiles;
        T.nt = rest % ntiles;
        T.split = rest / ntiles;
        T.m0 = mt * FUSED_BM;
        T.kbase = T.split * p.kb_per_split;
        T.nk = min(p.kb_per_split, nk_all - T.kbase);
        return T;
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full + 8 * s, 1 + 2 * F::DEC_WARPS);
            mbar_init(empty + 8 * s, 1);
            mbar_init(p_full + 8 * s, 1);
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
    // decode table: byte -> [w0 + 128, w1 + 128, w2 + 128, 0x64], one copy per
    // lane (entry b of lane l at lut + 128 b + 4 l), so that a warp's lookups
    // fall in 32 different banks whatever the bytes
    {
        __shared__ int8_t Cs[96];
        for (int i = threadIdx.x; i < 96; i += THREADS)
            Cs[i] = p.C[i];
        __syncthreads();
        for (int i = threadIdx.x; i < kLutEntries * 8; i += THREADS) {
            const uint32_t e = (expanded_entry(Cs, (uint32_t)(i >> 3)) ^ 0x00808080u) | 0x64000000u;
            asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(lut + (uint32_t)(i >> 3) * 128u +
                                                                           (uint32_t)(i & 7) * 16u),
                         "r"(e)
                         : "memory");
        }
    }
    tc_fence_before();
    cluster_sync();   // both CTAs' barriers initialised, the pair's TMEM allocated, tables built
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    bool timed_out = false;
    pdl_launch_dependents();   // the split-K finish may be scheduled; it waits for this grid

    // decode of K block g (this CTA's half) into the decoded half of stage g % S,
    // once its packed bytes have landed (copied after the MMAs were done with the
    // stage's last use); the warp then signals the even CTA
    const uint32_t lut_lane = lut + (uint32_t)lane * 4u;
    const uint32_t full0 = map_to_rank(full, 0);
    // The next block's packed half is tested (without blocking) before this
    // block's decode, so that the test's latency hides behind the decode; when it
    // has landed the next call skips its wait.  The phase tested cannot be an
    // older one (that completed with the other parity) nor a later one (that
    // needs this warp's decode of the next block first).
    bool next_landed = false;
    auto decode_block = [&](int g) -> bool {
        const int s = g % S;
        if (!dcheck(p.status, s < S) || (!next_landed && !mbar_wait_bounded(p_full + 8 * s, (g / S) & 1)))
            return false;
        next_landed = mbar_test(p_full + 8 * ((g + 1) % S), ((g + 1) / S) & 1);
        decode_units_f16(base + F::OFF_P + s * F::P_BYTES, base + F::OFF_B + s * F::B_BYTES, lut_lane,
                         32 * F::decoder_index(warp) + lane, F::DECODERS);
        fence_proxy_async_smem();   // generic writes -> visible to the tensor core
        __syncwarp();
        if (lane == 0)
            mbar_arrive_remote(full0 + 8 * s);
        return true;
    };

    if (warp < DRAIN_WARP0) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 80;");
        if (warp == 0) {
            // ---- this CTA's packed half and activation half of every K block, by
            // bulk tensor copy: the packed half completes on this CTA's p_full,
            // both CTAs' activation halves on the even CTA's full barrier (which
            // expects both halves' bytes).  Packed weights are never outputs of
            // the kernel before, so the first stages' packed halves are requested
            // before the grid-dependency wait.
            auto issue_packed = [&](int s, const Tile &T, int kb) {
                mbar_arrive_expect_tx_elect(p_full + 8 * s, F::P_BYTES);
                tma_2d_elect(base + F::OFF_P + s * F::P_BYTES, &tm_pk, (T.kbase + kb) * BK,
                             T.nt * F::TILE_GROUPS + (int)rank * G2, p_full + 8 * s);
            };
            int early = 0;   // packed halves issued before the wait (blocks 0 .. early - 1)
            for (int t = cid; t < total && early < S; t += nclusters) {
                const Tile T = tile_of(t);
                for (int kb = 0; kb < T.nk && early < S; ++kb)
                    issue_packed(early++, T, kb);
            }
            pdl_wait();   // the fp16 activation codes come from the kernel before
            int issued = 0;
            for (int t = cid; t < total && !timed_out; t += nclusters) {
                const Tile T = tile_of(t);
                for (int kb = 0; kb < T.nk; ++kb) {
                    const int s = issued % S;
                    if (issued >= S && !warp_wait(empty + 8 * s, ((issued / S) - 1) & 1)) {
                        timed_out = true;
                        break;
                    }
                    if (issued >= early)
                        issue_packed(s, T, kb);
                    if (rank == 0)
                        mbar_arrive_expect_tx_elect(full + 8 * s, 2 * A_BYTES);
                    tma_2d_pair_elect(base + F::OFF_A + s * A_BYTES, &tm_act, (T.kbase + kb) * BK,
                                      T.m0 + (int)rank * BM, full0 + 8 * s);
                    ++issued;
                }
            }
            // never leave with copies in flight: the last stages' MMAs (which
            // needed every copy of both CTAs) have completed; packed halves issued
            // early for blocks the loop never reached (a timeout) have landed
            for (int v = issued - S < 0 ? 0 : issued - S; v < issued; ++v)
                if (!warp_wait(empty + 8 * (v % S), (v / S) & 1))
                    timed_out = true;
            for (int v = issued; v < early; ++v)
                if (!warp_wait(p_full + 8 * v, 0))
                    timed_out = true;
        } else if (warp == 1) {
            if (rank == 0) {
                // ---- MMA issuer of the pair: the whole warp runs the loop so that
                // the descriptors stay warp-uniform; one elected lane issues -------
                int g = 0, gc = 0;
                // fp32 accumulator, fp16 A and B (format 0), K-major, N and M
                const uint32_t idesc = (1u << 4) | ((uint32_t)(F::BN >> 3) << 17) |
                                       ((uint32_t)(FUSED_BM >> 4) << 24);
                for (int t = cid; t < total && !timed_out; t += nclusters) {
                    const Tile T = tile_of(t);
                    for (int kb = 0; kb < T.nk; ++kb) {
                        const int s = g % S;
                        const int c = gc + kb / CHUNK_BLOCKS, kin = kb % CHUNK_BLOCKS;
                        const uint32_t d = tmem + (uint32_t)((c & 1) * 256);
                        if ((kin == 0 && c >= 2 && !warp_wait(acc_empty + 8 * (c & 1), ((c >> 1) - 1) & 1)) ||
                            !warp_wait(full + 8 * s, (g / S) & 1)) {
                            timed_out = true;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t a = base + F::OFF_A + s * A_BYTES;
                        const uint32_t b = base + F::OFF_B + s * F::B_BYTES;
#pragma unroll
                        for (int kk = 0; kk < BK / 16; ++kk)
                            mma_f16_pair_elect(d, sw128_desc(a + kk * 32), sw128_desc(b + kk * 32), idesc,
                                                (kin | kk) ? 1u : 0u);
                        mma_commit_pair_elect(empty + 8 * s);
                        if (kin == CHUNK_BLOCKS - 1 || kb == T.nk - 1)
                            mma_commit_pair_elect(acc_full + 8 * (c & 1));
                        ++g;
                    }
                    gc += (T.nk + CHUNK_BLOCKS - 1) / CHUNK_BLOCKS;
                }
                // the tensor core must be done with both CTAs' memory before exit
                if (g > 0 && !warp_wait(empty + 8 * ((g - 1) % S), ((g - 1) / S) & 1))
                    timed_out = true;
            }
        } else if (F::decoder_index(warp) >= 0) {
            // ---- decode ---------------------------------------------------------------
            int g = 0;
            for (int t = cid; t < total && !timed_out; t += nclusters) {
                const int nk = tile_of(t).nk;
                for (int kb = 0; kb < nk; ++kb, ++g)
                    if (!decode_block(g)) {
                        timed_out = true;
                        break;
                    }
            }
        }
    } else {
        // ---- drain this CTA's accumulator rows (warps 8-15), then the epilogue
        asm volatile("setmaxnreg.inc.sync.aligned.u32 176;");
        const int q = warp & 3;
        const int h = (warp - DRAIN_WARP0) >> 2;   // which 120 of the 240 columns
        const uint32_t release = rank == 0 ? acc_empty : map_to_rank(acc_empty, 0);
        int32_t acc[F::BH];
        // fp32 chunk c in TMEM -> int32 registers; then release its buffer
        auto drain = [&](int c) {
            tc_fence_after();
            const uint32_t ta = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)((c & 1) * 256 + h * F::BH);
#pragma unroll
            for (int gg = 0; gg < F::BH / 24; ++gg) {
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
                mbar_arrive_remote(release + 8 * (c & 1));
        };
        int gc = 0;   // first chunk of the current tile
        for (int t = cid; t < total && !timed_out; t += nclusters) {
            const Tile T = tile_of(t);
            const int nch = (T.nk + CHUNK_BLOCKS - 1) / CHUNK_BLOCKS;
#pragma unroll
            for (int i = 0; i < F::BH; ++i)
                acc[i] = 0;
            int cn = gc;   // next chunk to drain
            for (; cn < gc + nch && !timed_out; ++cn) {
                if (!mbar_wait_bounded(acc_full + 8 * (cn & 1), (cn >> 1) & 1)) {
                    timed_out = true;
                    break;
                }
                drain(cn);
            }
            gc += nch;
            const int row = T.m0 + (int)rank * BM + 32 * q + lane;
            if (!timed_out && row < p.M)
                store_tile_row<F::BH>(p, T.split, row, T.nt * F::BN + h * F::BH, acc);
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

template <int G2>
static cudaError_t launch_fused_tile(const LinearArgs &a, const uint16_t *act_f16, int32_t *part, int nsplit,
                                     int kbps, cudaStream_t stream)
{
    using namespace tc;
    using F = FusedTile<G2>;
    auto encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(tensor_map_encoder_fn());
    if (!encode)
        return cudaErrorNotSupported;
    const int G = (a.N + 2) / 3;
    CUtensorMap tm_act, tm_pk;
    const cuuint32_t es[2] = {1, 1};
    const cuuint64_t dA[2] = {(cuuint64_t)a.K, (cuuint64_t)a.M};
    const cuuint64_t sA[1] = {(cuuint64_t)a.K * 2};
    const cuuint32_t boxA[2] = {BK, BM};
    const cuuint64_t dP[2] = {(cuuint64_t)a.K, (cuuint64_t)G};
    const cuuint64_t sP[1] = {(cuuint64_t)a.K};
    const cuuint32_t boxP[2] = {BK, G2};
    if (encode(&tm_act, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<uint16_t *>(act_f16), dA, sA, boxA, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS ||
        encode(&tm_pk, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(a.packed), dP, sP, boxP, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(prefill_fused_kernel<G2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         F::SMEM_BYTES);
    if (e != cudaSuccess)
        return e;
    const Params p = make_params(a, nsplit, kbps, part);
    const long tiles = (long)((a.M + FUSED_BM - 1) / FUSED_BM) * (long)((G + F::TILE_GROUPS - 1) / F::TILE_GROUPS) *
                       nsplit;
    if (tiles > 0x7FFFFFFFL)
        return cudaErrorInvalidValue;
    long pairs = device_sm_count() / 2;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(2 * pairs));
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = F::SMEM_BYTES;
    int fit = 0;   // pairs the GPU can hold at once (not every SM may find a partner)
    if (cudaOccupancyMaxActiveClusters(&fit, prefill_fused_kernel<G2>, &cfg) == cudaSuccess && fit > 0 &&
        fit < pairs)
        pairs = fit;
    (void)cudaGetLastError();
    const long clusters = tiles < pairs ? tiles : pairs;
    return launch_pdl(prefill_fused_kernel<G2>, dim3((unsigned)(2 * clusters)), dim3(THREADS),
                      (size_t)F::SMEM_BYTES, stream, tm_act, tm_pk, p);
}

// SM-pair tensor-core GEMM on packed weights: act_f16 is the fp16 copy of the
// activation codes [M, K] (in the workspace), part the split-K partials or null;
// g2 = packed rows per CTA of the tile (fused_tile_groups).
cudaError_t launch_prefill_fused(const LinearArgs &a, const uint16_t *act_f16, int32_t *part, int nsplit, int kbps,
                                 int g2, cudaStream_t stream)
{
    if (g2 == 32)
        return launch_fused_tile<32>(a, act_f16, part, nsplit, kbps, stream);
    if (g2 == 40)
        return launch_fused_tile<40>(a, act_f16, part, nsplit, kbps, stream);
    return cudaErrorInvalidValue;
}

}  // namespace s3d8
