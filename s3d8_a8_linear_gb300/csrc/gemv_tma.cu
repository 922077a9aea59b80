// Streaming S3D8 GEMV for the decode regime (M <= 8 tokens), grouped form.
//
// One launch runs up to kMaxJobs independent linears.  The CTAs (one per SM,
// 16 warps) are divided among the jobs in proportion to their packed bytes, so
// every CTA works on exactly one matrix and all matrices stream concurrently.
// Per CTA:
//   * the 64 KiB wide decode table (one PRMT builds each lookup address, see
//     common.cuh), built once for the CTA's matrix;
//   * one private ring of kDepth stages per warp in shared memory, filled by
//     1-D bulk copies (cp.async.bulk + mbarrier complete_tx).  A warp refills
//     the stage it has just consumed, so HBM keeps streaming while the same warp
//     decodes and the bytes in flight occupy no registers;
//   * the int8 activations of the warp's fixed K-slice in registers.  With bf16
//     activations the CTA first quantises the whole row into shared memory
//     (per-token absmax / 127 with IEEE division, round-half-even), so that no
//     separate quantisation launch is needed.
// Work inside a job: a contiguous range of packed rows per CTA.  A row's K is
// cut into T slices of 4 KiB (the last may be shorter); warp w always takes
// slice w % T of rows r0 + w / T + i * (16 / T).  (Dealing rows out in stripes
// across CTAs, so that all warps of a job read one moving window of HBM, was
// measured slower on GB300.)  A warp covers 512 contiguous
// bytes per step (16 per lane), so each bulk copy is one contiguous row slice.
// The channel sums of a row slice are reduced with a transposed butterfly; with
// T > 1 the slices of a row meet in shared-memory atomics, written out after a
// CTA barrier.  Output: bf16 epilogue (x_s * acc) * W_s, or raw int32 sums.
//
// Programmatic dependent launch: the kernel lets the next grid launch early.
// Before griddepcontrol.wait it touches only weights (centroid table, the wide
// decode table, the first bulk copies of packed rows), which are parameters and
// never outputs of the preceding kernel; the activations (and everything
// written) come after the wait.
#include "common.cuh"
#include "launch.h"
#include "tma.cuh"

namespace s3d8 {

constexpr int kTmaWarps = 16;
constexpr int kTmaThreads = kTmaWarps * 32;
constexpr int kDepth = 2;    // row slices per warp ring
constexpr int kHalves = 2;   // each slice arrives as two bulk copies with their own barriers
constexpr int kBarsPerWarp = kDepth * kHalves;
#ifndef S3D8_PREWAIT_SLICES
#define S3D8_PREWAIT_SLICES 1
#endif
// Row slices a warp requests before the grid dependency wait; the rest of the
// ring is filled after the activation loads have been issued, so that their
// replies do not queue behind a whole ring of weight bytes.
constexpr int kPrewaitSlices = S3D8_PREWAIT_SLICES;
// 512-byte chunks per slice: 8 (4 KiB) for up to 2 tokens, 4 for 3..4 tokens and
// 2 for 5..8 tokens, so that the activations of the slice still fit in registers.
__host__ __device__ constexpr int chunks_for(int MT)
{
    return MT <= 2 ? 8 : MT <= 4 ? 4 : 2;
}
constexpr int kUnionBytes = 28672;               // fused activations, then T > 1 sums
constexpr int kTmaDynSmem = 232448 - 4096;

__host__ __device__ constexpr int pow2_at_least(int v)
{
    return v <= 1 ? 1 : v <= 2 ? 2 : v <= 4 ? 4 : v <= 8 ? 8 : v <= 16 ? 16 : 32;
}

struct TmaLayout {
    uint32_t lut;    // wide table (64 KiB, window-aligned)
    uint32_t bars;   // kTmaWarps * kBarsPerWarp mbarriers
    uint32_t uni;    // kUnionBytes: quantised activations, later the T > 1 sums
    uint32_t ring;   // this warp's ring
    bool ok;
};

// Carves the dynamic shared window [base, base + size) around the 64 KiB-aligned
// table: the mbarriers and the union buffer go first, then as many rings as fit
// below the table, the rest above it.
__device__ __forceinline__ TmaLayout tma_layout(uint32_t base, uint32_t size, int warp, uint32_t stage)
{
    TmaLayout L;
    L.lut = wide_lut_window(base);
    const uint32_t end = base + size;
    const uint32_t ring_bytes = kDepth * stage;
    uint32_t lo = (base + 7) & ~7u;
    uint32_t hi = L.lut + kWideLutBytes;
    const uint32_t small = kTmaWarps * kBarsPerWarp * 8 + 16 + kUnionBytes;
    uint32_t small_at;
    if (lo + small <= L.lut) {
        small_at = lo;
        lo += small;
    } else {
        small_at = hi;
        hi += small;
    }
    L.bars = small_at;
    L.uni = (small_at + kTmaWarps * kBarsPerWarp * 8 + 15) & ~15u;
    lo = (lo + 127) & ~127u;
    hi = (hi + 127) & ~127u;
    const uint32_t below = L.lut > lo ? (L.lut - lo) / ring_bytes : 0;
    const uint32_t n_below = below < (uint32_t)kTmaWarps ? below : (uint32_t)kTmaWarps;
    L.ring = (uint32_t)warp < n_below ? lo + warp * ring_bytes : hi + (warp - n_below) * ring_bytes;
    L.ok = hi + (kTmaWarps - n_below) * ring_bytes <= end && L.lut + kWideLutBytes <= end;
    return L;
}

__device__ __forceinline__ void pdl_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Per-token absmax quantisation of x[M, K] (bf16, M * K <= kUnionBytes) into
// shared int8 codes and shared fp32 scales, by the whole CTA.  Same rule as the
// standalone kernel.  The row is read once into registers (stage 1, issued
// before the bulk weight copies so that it does not queue behind them) and
// quantised from there (stage 2).  Instantiated for NS = 1, 2, 4 and 7 chunks
// per thread, so that a short row runs a short prologue.
constexpr int kActChunksPerThread = kUnionBytes / 8 / kTmaThreads;   // 16-byte chunks

template <int NS>
struct ActRegs {
    uint4 v[NS];
};

// Token (row of x) that 16-byte chunk c belongs to, for rows of per_row chunks:
// compares instead of an integer division.
template <int MT>
__device__ __forceinline__ int chunk_token(int c, int per_row)
{
    int m = 0;
#pragma unroll
    for (int t = 1; t < MT; ++t)
        m += c >= t * per_row ? 1 : 0;
    return m;
}

// Volatile loads: all chunks leave at once, here, instead of being sunk one by
// one to their first use (which would serialise their latencies).
template <int NS>
__device__ __forceinline__ void act_load(const __nv_bfloat16 *__restrict__ x, int M, int K, ActRegs<NS> &r)
{
    const int chunks = M * K / 8;
#pragma unroll
    for (int i = 0; i < NS; ++i) {
        const int c = threadIdx.x + i * kTmaThreads;
        r.v[i] = c < chunks ? ldg_stream_v4(reinterpret_cast<const uint4 *>(x) + c)
                            : make_uint4(0u, 0u, 0u, 0u);
    }
}

// Phase A of the fused quantisation: per-warp absmax of each token's row part
// held in `r`, written to red[warp * MT + m].
template <int MT, int NS>
__device__ __forceinline__ void act_amax_partial(const ActRegs<NS> &r, int M, int K, float *red)
{
    const int chunks = M * K / 8;
    const int per_row = K / 8;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float amax[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m)
        amax[m] = 0.0f;
#pragma unroll
    for (int i = 0; i < NS; ++i) {
        const int c = threadIdx.x + i * kTmaThreads;
        if (c < chunks) {
            const int m = chunk_token<MT>(c, per_row);
            const float a = absmax_bf16x2_value(absmax_bf16x8(r.v[i], 0u));
#pragma unroll
            for (int mm = 0; mm < MT; ++mm)
                if (mm == m)
                    amax[mm] = fmaxf(amax[mm], a);
        }
    }
#pragma unroll
    for (int m = 0; m < MT; ++m) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            amax[m] = fmaxf(amax[m], __shfl_xor_sync(0xffffffffu, amax[m], o));
        if (lane == 0)
            red[warp * MT + m] = amax[m];
    }
}

// Phase B: every thread folds the warp maxima into the per-token scale
// (absmax / 127, IEEE division) and writes the codes of its own chunks into
// the shared row `xs`.  Thread 0 also publishes the scales.
template <int MT, int NS>
__device__ __forceinline__ void act_codes(const ActRegs<NS> &r, int M, int K, const float *red, int8_t *xs,
                                          float *scale_s)
{
    const int chunks = M * K / 8;
    const int per_row = K / 8;
    float sc[MT], rcp[MT];
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int m = 0; m < MT; ++m) {
        // fold the kTmaWarps warp maxima across the lanes: one load, five shuffles
        float a = lane < kTmaWarps ? red[lane * MT + m] : 0.0f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
        sc[m] = __fdiv_rn(a, 127.0f);
        rcp[m] = sc[m] > 0.0f ? __frcp_rn(sc[m]) : 0.0f;
        if (threadIdx.x == 0)
            scale_s[m] = sc[m];
    }
#pragma unroll
    for (int i = 0; i < NS; ++i) {
        const int c = threadIdx.x + i * kTmaThreads;
        if (c < chunks) {
            const int m = chunk_token<MT>(c, per_row);
            float s = 0.0f, inv = 0.0f;
#pragma unroll
            for (int mm = 0; mm < MT; ++mm)
                if (mm == m) {
                    s = sc[mm];
                    inv = rcp[mm];
                }
            reinterpret_cast<uint2 *>(xs)[c] = quant_chunk8(r.v[i], s, inv);
        }
    }
}

// The fused quantisation with NS chunks per thread: loads x, runs issue_rest()
// (the rest of the bulk copies, queued behind x), publishes the warp maxima,
// then writes the codes and scales into shared memory.  Contains two CTA
// barriers, the first of which also publishes the decode table.
template <int MT, int NS, typename F>
__device__ __forceinline__ void fused_quant(const __nv_bfloat16 *x, int M, int K, float *red, int8_t *xs,
                                            float *scale_s, F issue_rest)
{
    ActRegs<NS> act;
    act_load<NS>(x, M, K, act);
    issue_rest();
    act_amax_partial<MT, NS>(act, M, K, red);
    __syncthreads();
    act_codes<MT, NS>(act, M, K, red, xs, scale_s);
    __syncthreads();
}

template <int MT, int CH>
struct SliceCompute {
    // Decodes chunks [J0, J1) (512 bytes each, at st + 512 j) of a staged slice,
    // only those below `nch` unless FULL, and accumulates all tokens.
    template <bool FULL, int J0, int J1>
    __device__ __forceinline__ static void run(uint32_t st, int nch, uint32_t lane_base,
                                               const uint32_t (&xr)[MT][CH][4], int (&acc)[MT][3])
    {
#pragma unroll
        for (int j = J0; j < J1; ++j) {
            if (FULL || j < nch) {
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
        }
    }
};

template <int MT>
__global__ __launch_bounds__(kTmaThreads, 1) void gemv_group_kernel(GroupArgs g, int smem_size)
{
    constexpr int CH = chunks_for(MT);
    constexpr int kStage = CH * 512;
    constexpr int NV = 3 * MT;
    constexpr int P = pow2_at_least(NV);
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ float red[kTmaWarps * MT];
    __shared__ float scale_s[MT];

    // ---- which job, which rows ------------------------------------------------
    int jb = 0;
#pragma unroll
    for (int j = 1; j < kMaxJobs; ++j)
        jb += (j < g.njobs && (int)blockIdx.x >= g.cta_begin[j]) ? 1 : 0;
    const GroupJob job = g.jobs[jb];
    const int nctas = g.cta_begin[jb + 1] - g.cta_begin[jb];
    const int b = (int)blockIdx.x - g.cta_begin[jb];
    const int M = g.M, N = job.N, K = job.K;
    const int G = (N + 2) / 3;
    const int T = (K + kStage - 1) / kStage;
    const int sets = kTmaWarps / T;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rs = warp / T, t = warp - rs * T;
    const bool active = rs < sets;
    const int slice_off = t * kStage;
    const int slice_len = max(0, min(kStage, K - slice_off));
    const int nch = (slice_len + 511) / 512;
    const int per_cta = (G + nctas - 1) / nctas;
    const int row0 = b * per_cta;                       // first packed row of this CTA
    const int nloc = max(0, min(G, row0 + per_cta) - row0);

    const uint32_t dyn = smem_addr(smem);
    const TmaLayout L = tma_layout(dyn, (uint32_t)smem_size, warp, kStage);
    if (!L.ok) {   // the host never requests a size this can happen for
        if (threadIdx.x == 0 && g.status)
            atomicExch(g.status, -3);
        return;
    }
    const uint32_t ring = L.ring;
    const uint32_t bar0 = L.bars + warp * kBarsPerWarp * 8;
    int8_t *xs = reinterpret_cast<int8_t *>(smem + (L.uni - dyn));
    int *sacc = reinterpret_cast<int *>(smem + (L.uni - dyn));
    const int range_rows = kUnionBytes / (4 * NV);

    // ---- before the grid dependency: weights only (table, first bulk copies) --
    // The packed bytes and the centroid table are parameters, never outputs of
    // the preceding kernel, so they are read while that kernel drains.
    __shared__ int8_t Cv[96];
    if (lane == 0)
        for (int s = 0; s < kBarsPerWarp; ++s)
            mbar_init(bar0 + s * 8, 1);
    if (threadIdx.x < 96) {
        short t;
        asm volatile("ld.global.nc.s8 %0, [%1];" : "=h"(t) : "l"(job.C + threadIdx.x));
        Cv[threadIdx.x] = (int8_t)t;
    }
    fence_proxy_async_smem();
    __syncthreads();
    // A warp's ring holds kDepth row slices; slice u of this warp sits in slot
    // u % kDepth and arrives as two halves (bytes [0, len0) and [len0, len)),
    // each with its own barrier, so that the first half of a slot can be
    // refilled while the second half is still being decoded.
    constexpr int kHalfBytes = kStage / kHalves;
    const int len0 = min(slice_len, kHalfBytes), len1 = slice_len - len0;
    const uint64_t wpol = l2_evict_first_policy();   // packed bytes are read once per launch
    auto issue_slice = [&](int slot, int row) {
        if (lane == 0 && dcheck(g.status, slot >= 0 && slot < kDepth && row >= 0 && row < G &&
                                               slice_off + slice_len <= K &&
                                               ring + (uint32_t)((slot + 1) * kStage) <= dyn + (uint32_t)smem_size)) {
            const uint8_t *src = job.packed + (size_t)row * K + slice_off;
            const uint32_t dst = ring + slot * kStage;
            const uint32_t b = bar0 + slot * kHalves * 8;
            fence_proxy_async_smem();   // this warp's earlier reads of the slot precede the refill
            mbar_arrive_expect_tx(b, (uint32_t)len0);
            bulk_load_hint(dst, src, (uint32_t)len0, b, wpol);
            if (len1 > 0) {
                mbar_arrive_expect_tx(b + 8, (uint32_t)len1);
                bulk_load_hint(dst + kHalfBytes, src + kHalfBytes, (uint32_t)len1, b + 8, wpol);
            }
        }
    };
    int issued = 0, consumed = 0;
    const int nrow0 = min(range_rows, nloc);
    const int nmine0 = active ? max(0, (nrow0 - rs + sets - 1) / sets) : 0;
    for (int i = 0; i < kPrewaitSlices && i < nmine0; ++i)
        issue_slice(issued++ % kDepth, row0 + rs + i * sets);
    // wide table: entry b's 32 lane copies are 128 contiguous bytes at lut + 256 b
    {
        const uint32_t lut = L.lut;
#pragma unroll
        for (int i = 0; i < kLutEntries * 8 / kTmaThreads; ++i) {
            const int q = threadIdx.x + i * kTmaThreads;
            const uint32_t e = expanded_entry(Cv, (uint32_t)(q >> 3));
            asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(lut + (uint32_t)(q >> 3) * 256u +
                                                                           (uint32_t)(q & 7) * 16u),
                         "r"(e)
                         : "memory");
        }
    }
    pdl_launch_dependents();
    pdl_wait();   // activations may come from the previous grid: read them only now

    // ---- activations -------------------------------------------------------------
    const bool fused = job.x != nullptr;
    uint32_t xr[MT][CH][4];
    auto issue_rest = [&]() {   // rest of the ring, behind the activation loads
        for (int i = kPrewaitSlices; i < kDepth && i < nmine0; ++i)
            issue_slice(issued++ % kDepth, row0 + rs + i * sets);
    };
    if (fused) {
        const int ns = (M * K / 8 + kTmaThreads - 1) / kTmaThreads;   // 16-byte chunks per thread
        if (ns <= 1)
            fused_quant<MT, 1>(job.x, M, K, red, xs, scale_s, issue_rest);
        else if (ns <= 2)
            fused_quant<MT, 2>(job.x, M, K, red, xs, scale_s, issue_rest);
        else if (ns <= 4)
            fused_quant<MT, 4>(job.x, M, K, red, xs, scale_s, issue_rest);
        else
            fused_quant<MT, kActChunksPerThread>(job.x, M, K, red, xs, scale_s, issue_rest);
    } else {
#pragma unroll
        for (int m = 0; m < MT; ++m)
#pragma unroll
            for (int j = 0; j < CH; ++j) {
                const int k = slice_off + j * 512 + lane * 16;
                uint4 v = make_uint4(0u, 0u, 0u, 0u);
                if (m < M && k < K && j * 512 < slice_len)
                    v = ldg_stream_v4(job.xq + (size_t)m * K + k);
                xr[m][j][0] = v.x;
                xr[m][j][1] = v.y;
                xr[m][j][2] = v.z;
                xr[m][j][3] = v.w;
            }
        issue_rest();
        if (threadIdx.x < MT)   // scales are read only for the bf16 output (none on the int32 path)
            scale_s[threadIdx.x] =
                ((int)threadIdx.x < M && job.xscale != nullptr) ? job.xscale[threadIdx.x] : 0.0f;
        __syncthreads();   // table written; scales published
    }
    if (fused) {
        if (b == 0) {   // optional copies of the codes and scales for the caller
            if (job.xq_out)
                for (int c = threadIdx.x; c < M * K / 16; c += kTmaThreads)
                    reinterpret_cast<uint4 *>(job.xq_out)[c] = reinterpret_cast<const uint4 *>(xs)[c];
            if (job.xscale_out && (int)threadIdx.x < M)
                job.xscale_out[threadIdx.x] = scale_s[threadIdx.x];
        }
#pragma unroll
        for (int m = 0; m < MT; ++m)
#pragma unroll
            for (int j = 0; j < CH; ++j) {
                const int k = slice_off + j * 512 + lane * 16;
                uint4 v = make_uint4(0u, 0u, 0u, 0u);
                if (m < M && k < K && j * 512 < slice_len)
                    v = *reinterpret_cast<const uint4 *>(xs + (size_t)m * K + k);
                xr[m][j][0] = v.x;
                xr[m][j][1] = v.y;
                xr[m][j][2] = v.z;
                xr[m][j][3] = v.w;
            }
    }
    if (T > 1) {
        if (fused)
            __syncthreads();   // every warp holds its codes: the union buffer is free
        for (int i = threadIdx.x; i < nrow0 * NV; i += kTmaThreads)
            sacc[i] = 0;
        __syncthreads();
    }
    float xsc[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m)
        xsc[m] = scale_s[m];

    // ---- stream ---------------------------------------------------------------
    const uint32_t lane_base = L.lut | (uint32_t)(lane << 2);
    bool timed_out = false;
    bool pending0 = false;   // a first-half refill issued for a slice not yet counted in `issued`
    for (int r0 = 0; r0 < nloc; r0 += range_rows) {
        const int nrow = min(range_rows, nloc - r0);
        const int nmine = (active && !timed_out) ? max(0, (nrow - rs + sets - 1) / sets) : 0;
        if (r0 != 0)   // the first range's copies were issued above
            for (int i = 0; i < kDepth && i < nmine; ++i)
                issue_slice(issued++ % kDepth, row0 + r0 + rs + i * sets);
        for (int i = 0; i < nmine; ++i) {
            const int u = consumed;
            const int s = u % kDepth;
            const uint32_t par = (uint32_t)((u / kDepth) & 1);
            const uint32_t b = bar0 + s * kHalves * 8;
            const bool refill = i + kDepth < nmine;
            const int next_row = row0 + r0 + rs + (i + kDepth) * sets;
            int acc[MT][3];
#pragma unroll
            for (int m = 0; m < MT; ++m)
                acc[m][0] = acc[m][1] = acc[m][2] = 0;
            const uint32_t st = ring + s * kStage + lane * 16;
            if (!mbar_wait_bounded(b, par)) {
                timed_out = true;
                break;
            }
            if (slice_len == kStage)
                SliceCompute<MT, CH>::template run<true, 0, CH / 2>(st, nch, lane_base, xr, acc);
            else
                SliceCompute<MT, CH>::template run<false, 0, CH / 2>(st, nch, lane_base, xr, acc);
            __syncwarp();
            if (refill && lane == 0 && dcheck(g.status, next_row < G)) {   // first half of the slot is free: refill it
                const uint8_t *src = job.packed + (size_t)next_row * K + slice_off;
                fence_proxy_async_smem();
                mbar_arrive_expect_tx(b, (uint32_t)len0);
                bulk_load_hint(ring + s * kStage, src, (uint32_t)len0, b, wpol);
            }
            if (len1 > 0) {
                if (!mbar_wait_bounded(b + 8, par)) {
                    timed_out = true;
                    pending0 = refill;
                    break;
                }
                if (slice_len == kStage)
                    SliceCompute<MT, CH>::template run<true, CH / 2, CH>(st, nch, lane_base, xr, acc);
                else
                    SliceCompute<MT, CH>::template run<false, CH / 2, CH>(st, nch, lane_base, xr, acc);
                __syncwarp();
                if (refill && lane == 0 && dcheck(g.status, next_row < G)) {
                    const uint8_t *src = job.packed + (size_t)next_row * K + slice_off + kHalfBytes;
                    fence_proxy_async_smem();
                    mbar_arrive_expect_tx(b + 8, (uint32_t)len1);
                    bulk_load_hint(ring + s * kStage + kHalfBytes, src, (uint32_t)len1, b + 8, wpol);
                }
            }
            ++consumed;
            if (refill)
                ++issued;
            int v[P];
#pragma unroll
            for (int e = 0; e < P; ++e)
                v[e] = e < NV ? acc[e / 3][e % 3] : 0;
            const int sum = warp_reduce_transposed<P>(v, lane);
            const int idx = lane / (32 / P);
            const bool leader = (lane & (32 / P - 1)) == 0;
            const int lrow = r0 + rs + i * sets, row = row0 + lrow;
            if (leader && idx < NV) {
                const int m = idx / 3, n = 3 * row + (idx - 3 * m);
                if (T == 1) {
                    if (m < M && n < N && dcheck(g.status, row < G)) {
                        if (job.acc)
                            job.acc[(size_t)m * N + n] = sum;
                        else
                            job.out[(size_t)m * N + n] = epilogue_bf16(sum, xsc[m], job.cs[n]);
                    }
                } else if (dcheck(g.status, (lrow - r0) * NV + idx < range_rows * NV)) {
                    atomicAdd(&sacc[(lrow - r0) * NV + idx], sum);
                }
            }
        }
        if (T > 1) {
            __syncthreads();
            for (int e = threadIdx.x; e < nrow * NV; e += kTmaThreads) {
                const int rl = e / NV, idx = e - rl * NV;
                const int m = idx / 3, n = 3 * (row0 + r0 + rl) + (idx - 3 * m);
                if (m < M && n < N && dcheck(g.status, row0 + r0 + rl < G)) {
                    if (job.acc)
                        job.acc[(size_t)m * N + n] = sacc[e];
                    else
                        job.out[(size_t)m * N + n] = epilogue_bf16(sacc[e], xsc[m], job.cs[n]);
                }
                sacc[e] = 0;
            }
            __syncthreads();
        }
    }
    if (timed_out) {
        // never leave with copies in flight: wait (bounded) for both halves of
        // every issued slice not yet consumed, and for an early first-half refill
        for (int v = consumed; v < issued; ++v) {
            const uint32_t b = bar0 + (v % kDepth) * kHalves * 8;
            mbar_wait_bounded(b, (uint32_t)((v / kDepth) & 1));
            if (len1 > 0)
                mbar_wait_bounded(b + 8, (uint32_t)((v / kDepth) & 1));
        }
        if (pending0)
            mbar_wait_bounded(bar0 + (issued % kDepth) * kHalves * 8, (uint32_t)((issued / kDepth) & 1));
        if (lane == 0)
            record_timeout(g.status);
    }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------

static int tma_token_block(int M)
{
    return M <= 1 ? 1 : M <= 2 ? 2 : M <= 4 ? 4 : 8;
}

static int stage_bytes(int M)
{
    return chunks_for(tma_token_block(M)) * 512;
}

bool gemv_group_job_ok(int M, int K, bool fused)
{
    if (M < 1 || M > 8)
        return false;
    if ((K + stage_bytes(M) - 1) / stage_bytes(M) > kTmaWarps)
        return false;
    if (fused && (long)M * K > kUnionBytes)
        return false;
    return true;
}

bool gemv_tma_supported(int M, int K)
{
    return gemv_group_job_ok(M, K, false);
}

// Splits `ctas` CTAs over the jobs in proportion to their cost (largest
// remainder), at least one CTA per job and never more CTAs than rows x slices.
// Cost = packed bytes, plus for jobs that quantise their activations in-kernel
// the longer prologue of a long row, in bytes a CTA would have streamed in that
// time (measured on GB300: about 1.2 us more at K = 14336 than at K = 4096, at
// about 32 KB per microsecond per SM), times 1.08 for rows cut into several
// slices (their CTAs streamed ~8% fewer bytes per microsecond in a per-CTA
// timeline of the 11B layer: shorter last slices and the shared-memory row
// sums; with the factor the layer step went from 19.41 to 19.24 us).
static void split_ctas(const GroupArgs &g, int ctas, int *cta_begin)
{
    const int kStage = stage_bytes(g.M);
    double total = 0.0;
    double bytes[kMaxJobs];
    int cap[kMaxJobs];
    double raw = 0.0;
    for (int j = 0; j < g.njobs; ++j)
        raw += (double)((g.jobs[j].N + 2) / 3) * g.jobs[j].K;
    for (int j = 0; j < g.njobs; ++j) {
        const long G = (g.jobs[j].N + 2) / 3;
        const long T = (g.jobs[j].K + kStage - 1) / kStage;
        bytes[j] = (double)G * g.jobs[j].K;
        if (g.jobs[j].x && g.jobs[j].K > 4096 && raw > 0) {
            const double est_ctas = ctas * bytes[j] / raw;
            bytes[j] += est_ctas * 1.2 * (g.jobs[j].K - 4096) / 10240.0 * 32768.0;
        }
        if (T > 1)
            bytes[j] *= 1.08;
        cap[j] = (int)(G * T < ctas ? G * T : ctas);
        total += bytes[j];
    }
    int count[kMaxJobs];
    double frac[kMaxJobs];
    int used = 0;
    for (int j = 0; j < g.njobs; ++j) {
        const double want = total > 0 ? ctas * bytes[j] / total : 1.0;
        count[j] = (int)want;
        if (count[j] < 1)
            count[j] = 1;
        if (count[j] > cap[j])
            count[j] = cap[j];
        frac[j] = want - (int)want;
        used += count[j];
    }
    while (used < ctas) {
        int best = -1;
        for (int j = 0; j < g.njobs; ++j)
            if (count[j] < cap[j] && (best < 0 || frac[j] > frac[best]))
                best = j;
        if (best < 0)
            break;
        ++count[best];
        frac[best] = -1.0;
        ++used;
    }
    cta_begin[0] = 0;
    for (int j = 0; j < g.njobs; ++j)
        cta_begin[j + 1] = cta_begin[j] + count[j];
}

template <int MT>
static cudaError_t launch_group_mt(const GroupArgs &g, int grid, cudaStream_t stream)
{
    cudaError_t e = cudaFuncSetAttribute(gemv_group_kernel<MT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kTmaDynSmem);
    if (e != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kTmaThreads);
    cfg.dynamicSmemBytes = kTmaDynSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, gemv_group_kernel<MT>, g, (int)kTmaDynSmem);
}

cudaError_t launch_gemv_group(GroupArgs &g, cudaStream_t stream)
{
    if (g.njobs < 1 || g.njobs > kMaxJobs)
        return cudaErrorInvalidValue;
    const int sms = device_sm_count();
    const int kStage = stage_bytes(g.M);
    // jobs with the longest rows first: their CTAs take the SMs that free up
    // first while the preceding grid drains, since their prologue is longest
    for (int a = 1; a < g.njobs; ++a)
        for (int c = a; c > 0 && g.jobs[c].K > g.jobs[c - 1].K; --c) {
            const GroupJob tmp = g.jobs[c];
            g.jobs[c] = g.jobs[c - 1];
            g.jobs[c - 1] = tmp;
        }
    long items = 0;
    for (int j = 0; j < g.njobs; ++j)
        items += (long)((g.jobs[j].N + 2) / 3) * ((g.jobs[j].K + kStage - 1) / kStage);
    int ctas = items < sms ? (int)items : sms;
    if (ctas < g.njobs)
        ctas = g.njobs;
    split_ctas(g, ctas, g.cta_begin);
    const int grid = g.cta_begin[g.njobs];
    switch (tma_token_block(g.M)) {
    case 1: return launch_group_mt<1>(g, grid, stream);
    case 2: return launch_group_mt<2>(g, grid, stream);
    case 4: return launch_group_mt<4>(g, grid, stream);
    default: return launch_group_mt<8>(g, grid, stream);
    }
}

cudaError_t launch_gemv_tma(const LinearArgs &a, cudaStream_t stream)
{
    GroupArgs g = {};
    g.njobs = 1;
    g.M = a.M;
    g.status = a.status;
    GroupJob &j = g.jobs[0];
    j.packed = a.packed;
    j.C = a.C;
    j.cs = a.cs;
    j.x = nullptr;
    j.xq = a.xq;
    j.xscale = a.xscale;
    j.xq_out = nullptr;
    j.xscale_out = nullptr;
    j.out = a.out;
    j.acc = a.acc;
    j.N = a.N;
    j.K = a.K;
    return launch_gemv_group(g, stream);
}

}  // namespace s3d8
