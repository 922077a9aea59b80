// Streaming S3D8 GEMV for the decode regime (M <= 4 tokens), GB300 design.
//
// Per CTA (one per SM, 16 warps):
//   * the 64 KiB wide decode table (one PRMT per lookup address, see
//     common.cuh), built once;
//   * one private ring of kDepth stages per warp in shared memory, filled by
//     1-D bulk copies (cp.async.bulk + mbarrier complete_tx).  Each warp
//     refills the stage it has just consumed, so HBM keeps streaming while the
//     same warp decodes, and the bytes in flight do not occupy registers;
//   * the activations of the warp's fixed K-slice live in registers.
// Work: the CTA owns a contiguous range of packed rows.  A row's K is split
// into T slices of CC x 512 bytes; warp w always handles slice w % T of rows
// r0 + w / T, r0 + w / T + 16 / T, ...  A warp spans 512 contiguous bytes per
// step (16 per lane), so each bulk copy is one contiguous row slice.
// The three partial channel sums (per token) of a row slice are reduced across
// the warp with a transposed butterfly; with T > 1 the slices of a row are
// combined with shared-memory atomics and written after a CTA barrier.
// Output: bf16 epilogue (x_s * acc) * W_s, or the raw int32 accumulators.
#include "common.cuh"
#include "launch.h"
#include "tma.cuh"

namespace s3d8 {

constexpr int kTmaWarps = 16;
constexpr int kTmaThreads = kTmaWarps * 32;
constexpr int kDepth = 2;
constexpr int kMaxRangeRows = 512;      // rows per CTA pass (bounds the T > 1 accumulator)
constexpr int kTmaDynSmem = 232448 - 4096;

__host__ __device__ constexpr int pow2_at_least(int v)
{
    return v <= 1 ? 1 : v <= 2 ? 2 : v <= 4 ? 4 : v <= 8 ? 8 : v <= 16 ? 16 : 32;
}

struct TmaLayout {
    uint32_t lut;        // wide table (64 KiB, window-aligned)
    uint32_t bars;       // kTmaWarps * kDepth mbarriers
    uint32_t acc;        // kMaxRangeRows * 3 * MT ints
    uint32_t ring;       // this warp's ring
    bool ok;
};

// Carves the dynamic shared window [base, base + size) around the 64 KiB-aligned
// table.  Small blocks and rings go below the table first, then above it.
__device__ __forceinline__ TmaLayout tma_layout(uint32_t base, uint32_t size, uint32_t ring_bytes,
                                                uint32_t acc_bytes, int warp)
{
    TmaLayout L;
    L.lut = wide_lut_window(base);
    const uint32_t end = base + size;
    uint32_t lo = base, hi = L.lut + kWideLutBytes;
    auto take = [&](uint32_t bytes, uint32_t align) -> uint32_t {
        uint32_t a = (lo + align - 1) & ~(align - 1);
        if (a + bytes <= L.lut) {
            lo = a + bytes;
            return a;
        }
        uint32_t b = (hi + align - 1) & ~(align - 1);
        hi = b + bytes;
        return b;
    };
    L.bars = take(kTmaWarps * kDepth * 8, 8);
    L.acc = take(acc_bytes, 16);
    L.ring = 0;
    for (int w = 0; w < kTmaWarps; ++w) {
        const uint32_t r = take(ring_bytes, 128);
        if (w == warp)
            L.ring = r;
    }
    L.ok = hi <= end && L.lut + kWideLutBytes <= end;
    return L;
}

template <int MT, int CC>
__global__ __launch_bounds__(kTmaThreads, 1) void gemv_tma_kernel(LinearArgs a, int T, int smem_size)
{
    constexpr int STAGE = CC * 512;
    constexpr int NV = 3 * MT;
    constexpr int P = pow2_at_least(NV);
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ uint32_t stage_tab[kLutEntries];

    const uint32_t dyn = smem_addr(smem);
    const TmaLayout L = tma_layout(dyn, (uint32_t)smem_size, kDepth * STAGE,
                                   kMaxRangeRows * NV * 4, (int)(threadIdx.x >> 5));
    if (!L.ok) {  // cannot happen for the sizes the host requests; never silently wrong
        if (threadIdx.x == 0 && a.status)
            atomicExch(a.status, -3);
        return;
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int *sacc = reinterpret_cast<int *>(smem + (L.acc - dyn));
    for (int i = threadIdx.x; i < kMaxRangeRows * NV; i += kTmaThreads)
        sacc[i] = 0;
    if (lane == 0)
        for (int s = 0; s < kDepth; ++s)
            mbar_init(L.bars + (warp * kDepth + s) * 8, 1);
    fence_proxy_async_smem();
    build_wide_lut(smem + (L.lut - dyn), stage_tab, a.C);   // ends with __syncthreads()

    const int G = (a.N + 2) / 3;
    const int sets = kTmaWarps / T;
    const int rs = warp / T, t = warp - rs * T;
    const bool active = rs < sets;
    const uint32_t lane_base = L.lut | (uint32_t)(lane << 2);
    const int slice_off = t * STAGE;
    const int slice_len = max(0, min(STAGE, a.K - slice_off));
    const uint32_t ring = L.ring;
    const uint32_t bar0 = L.bars + warp * kDepth * 8;

    // activations of this warp's K-slice, per token (zero beyond K or M)
    uint32_t xr[MT][CC][4];
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int j = 0; j < CC; ++j) {
            const int k = slice_off + j * 512 + lane * 16;
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (m < a.M && k < a.K)
                v = __ldg(reinterpret_cast<const uint4 *>(a.xq + (size_t)m * a.K + k));
            xr[m][j][0] = v.x;
            xr[m][j][1] = v.y;
            xr[m][j][2] = v.z;
            xr[m][j][3] = v.w;
        }

    bool timed_out = false;
    int consumed = 0;   // uses of this warp's ring so far (identical in all lanes)
    int issued = 0;     // bulk copies issued into it so far
    // Contiguous row partition over the grid, cut into ranges of kMaxRangeRows rows.
    const int per_cta = (G + gridDim.x - 1) / gridDim.x;
    const int cta_beg = blockIdx.x * per_cta;
    const int cta_end = min(G, cta_beg + per_cta);
    for (int r0 = cta_beg; r0 < cta_end; r0 += kMaxRangeRows) {
        const int nrow = min(kMaxRangeRows, cta_end - r0);
        const int nmine = (active && !timed_out) ? max(0, (nrow - rs + sets - 1) / sets) : 0;
        for (int i = 0; i < kDepth && i < nmine; ++i) {
            if (lane == 0) {
                const uint32_t bar = bar0 + (issued % kDepth) * 8;
                mbar_arrive_expect_tx(bar, (uint32_t)slice_len);
                bulk_load(ring + (issued % kDepth) * STAGE,
                          a.packed + (size_t)(r0 + rs + i * sets) * a.K + slice_off,
                          (uint32_t)slice_len, bar);
            }
            ++issued;
        }
        for (int i = 0; i < nmine; ++i) {
            const int u = consumed;          // global use index of this warp's ring
            const int s = u % kDepth;
            const uint32_t bar = bar0 + s * 8;
            if (!mbar_wait_bounded(bar, (uint32_t)((u / kDepth) & 1))) {
                timed_out = true;
                break;
            }
            ++consumed;
            const uint32_t st = ring + s * STAGE + lane * 16;
            int acc[MT][3];
#pragma unroll
            for (int m = 0; m < MT; ++m)
                acc[m][0] = acc[m][1] = acc[m][2] = 0;
#pragma unroll
            for (int j = 0; j < CC; ++j) {
                const uint4 p = lds_v4(st + j * 512);
                const uint32_t pw[4] = {p.x, p.y, p.z, p.w};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    uint32_t V0, V1, V2;
                    decode_quad_wide(pw[q], lane_base, V0, V1, V2);
#pragma unroll
                    for (int m = 0; m < MT; ++m) {
                        acc[m][0] = __dp4a((int)V0, (int)xr[m][j][q], acc[m][0]);
                        acc[m][1] = __dp4a((int)V1, (int)xr[m][j][q], acc[m][1]);
                        acc[m][2] = __dp4a((int)V2, (int)xr[m][j][q], acc[m][2]);
                    }
                }
            }
            __syncwarp();
            if (i + kDepth < nmine) {
                if (lane == 0) {
                    fence_proxy_async_smem();   // our reads of stage s before the refill
                    mbar_arrive_expect_tx(bar, (uint32_t)slice_len);
                    bulk_load(ring + s * STAGE,
                              a.packed + (size_t)(r0 + rs + (i + kDepth) * sets) * a.K + slice_off,
                              (uint32_t)slice_len, bar);
                }
                ++issued;
            }
            int v[P];
#pragma unroll
            for (int e = 0; e < P; ++e)
                v[e] = e < NV ? acc[e / 3][e % 3] : 0;
            const int sum = warp_reduce_transposed<P>(v, lane);
            const int idx = lane / (32 / P);
            const bool leader = (lane & (32 / P - 1)) == 0;
            const int row = r0 + rs + i * sets;
            if (leader && idx < NV) {
                const int m = idx / 3, n = 3 * row + (idx - 3 * m);
                if (T == 1) {
                    if (m < a.M && n < a.N) {
                        if (a.acc)
                            a.acc[(size_t)m * a.N + n] = sum;
                        else
                            a.out[(size_t)m * a.N + n] = epilogue_bf16(sum, a.xscale[m], a.cs[n]);
                    }
                } else {
                    atomicAdd(&sacc[(row - r0) * NV + idx], sum);
                }
            }
        }
        if (T > 1) {
            __syncthreads();
            for (int e = threadIdx.x; e < nrow * NV; e += kTmaThreads) {
                const int rl = e / NV, idx = e - rl * NV;
                const int m = idx / 3, n = 3 * (r0 + rl) + (idx - 3 * m);
                if (m < a.M && n < a.N) {
                    if (a.acc)
                        a.acc[(size_t)m * a.N + n] = sacc[e];
                    else
                        a.out[(size_t)m * a.N + n] = epilogue_bf16(sacc[e], a.xscale[m], a.cs[n]);
                }
                sacc[e] = 0;
            }
            __syncthreads();
        }
    }
    if (timed_out) {
        // drain the copies still in flight into this warp's ring (bounded), then leave
        for (int u = consumed + 1; u < issued; ++u)
            mbar_wait_bounded(bar0 + (u % kDepth) * 8, (uint32_t)((u / kDepth) & 1));
        if (lane == 0)
            record_timeout(a.status);
    }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------

template <int MT, int CC>
static cudaError_t launch_tma_mt_cc(const LinearArgs &a, int T, int grid, cudaStream_t stream)
{
    cudaError_t e = cudaFuncSetAttribute(gemv_tma_kernel<MT, CC>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kTmaDynSmem);
    if (e != cudaSuccess)
        return e;
    gemv_tma_kernel<MT, CC><<<grid, kTmaThreads, kTmaDynSmem, stream>>>(a, T, kTmaDynSmem);
    return cudaGetLastError();
}

// Worst-case layout check on the host (the table window starts at 64 KiB; the
// dynamic region may begin anywhere up to 4 KiB into the window).
static bool tma_layout_fits(int CC, int MT)
{
    const long ring = (long)kDepth * CC * 512;
    const long below = 0x10000 - 0x1000 - kTmaWarps * kDepth * 8 - (long)kMaxRangeRows * 3 * MT * 4;
    const long above = (long)kTmaDynSmem + 0x400 - 0x20000;
    const long rings_below = below > 0 ? below / ring : 0;
    const long rings_above = above / (ring + 128);
    return rings_below + rings_above >= kTmaWarps;
}

// Chooses the slice width (CC chunks of 512 bytes) for a shape: the widest
// that still gives every warp of every CTA work and wastes little of K.
static int choose_cc(int G, int K, int ctas, int MT)
{
    // first choice: wide slices that keep every warp busy and waste < 1/8 of K;
    // second choice: any slice width that fits the 16 warps and the layout
    const int options_mt1[] = {8, 7, 4, 2, 1};
    const int options_mt2[] = {4, 2, 1};
    const int options_mt4[] = {2, 1};
    const int *opts = MT == 1 ? options_mt1 : MT == 2 ? options_mt2 : options_mt4;
    const int nopts = MT == 1 ? 5 : MT == 2 ? 3 : 2;
    const int rows_per_cta = (G + ctas - 1) / ctas;
    for (int i = 0; i < nopts; ++i) {
        const int cc = opts[i];
        const int T = (K + cc * 512 - 1) / (cc * 512);
        if (T > kTmaWarps || (kTmaWarps % T != 0 && T != 1))
            continue;
        const long waste = (long)T * cc * 512 - K;
        if (waste * 8 > (long)K && cc > 1)
            continue;
        if ((long)rows_per_cta * T < kTmaWarps && cc > 1)
            continue;
        if (!tma_layout_fits(cc, MT))
            continue;
        return cc;
    }
    for (int i = nopts - 1; i >= 0; --i) {
        const int cc = opts[i];
        const int T = (K + cc * 512 - 1) / (cc * 512);
        if (T <= kTmaWarps && tma_layout_fits(cc, MT))
            return cc;
    }
    return 0;
}

static int tma_token_block(int M)
{
    return M <= 1 ? 1 : M <= 2 ? 2 : 4;
}

bool gemv_tma_supported(int M, int K)
{
    if (M < 1 || M > 4)
        return false;
    const int widest = M <= 1 ? 8 : M <= 2 ? 4 : 2;
    return K <= kTmaWarps * 512 * widest;
}

cudaError_t launch_gemv_tma(const LinearArgs &a, cudaStream_t stream)
{
    const int MT = tma_token_block(a.M);
    const int G = (a.N + 2) / 3;
    const int sms = device_sm_count();
    const int cc = choose_cc(G, a.K, sms, MT);
    if (cc == 0)
        return cudaErrorInvalidValue;
    const int T = (a.K + cc * 512 - 1) / (cc * 512);
    if (T > kTmaWarps)
        return cudaErrorInvalidValue;
    // enough CTAs to cover the rows, at most one per SM
    const int items = G * T;
    int grid = (items + kTmaWarps - 1) / kTmaWarps;
    grid = grid < 1 ? 1 : grid > sms ? sms : grid;
#define S3D8_TMA_CASE(mt, c)                                                                      \
    if (MT == mt && cc == c)                                                                      \
        return launch_tma_mt_cc<mt, c>(a, T, grid, stream);
    S3D8_TMA_CASE(1, 8)
    S3D8_TMA_CASE(1, 7)
    S3D8_TMA_CASE(1, 4)
    S3D8_TMA_CASE(1, 2)
    S3D8_TMA_CASE(1, 1)
    S3D8_TMA_CASE(2, 4)
    S3D8_TMA_CASE(2, 2)
    S3D8_TMA_CASE(2, 1)
    S3D8_TMA_CASE(4, 2)
    S3D8_TMA_CASE(4, 1)
#undef S3D8_TMA_CASE
    return cudaErrorInvalidValue;
}

}  // namespace s3d8
