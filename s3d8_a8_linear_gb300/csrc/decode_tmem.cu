// S3D8 linear for a few tokens (1..64) on the tcgen05 tensor cores, with the
// weights decoded straight into tensor memory as the MMA's A operand.
//
// For 128 packed rows g and the three channels d = 0, 1, 2 of each row
// (channel 3g + d), D_d[g, t] = sum_k A_d[g, k] * X[t, k]: A_d holds channel
// 3g + d's weights, X the activation codes of token t, both as fp16 (every
// int8 value and every product is exact; each fp32 partial sum of at most 1024
// columns stays below 127^2 * 1024 < 2^24, so each 1024-column chunk's sum is
// exact, and chunks are added as int32).  The MMA is
// tcgen05.mma.cta_group::1.kind::f16 with M = 128 packed rows, N = the tokens
// rounded up to 16, K = 16; A comes from tensor memory, X from shared memory.
//
// Per CTA (one SM, 16 warps):
//   warp 0      bulk tensor copies: per 64-column block, the packed tile
//               (128 rows x 64 bytes, 64-byte swizzle) and the int8 codes tile
//               (N rows x 64 bytes) into an 8-stage ring;
//   warps 1-3   issue the MMAs, warp 1 + d those of channel d (one elected
//               lane each; warp 1 also allocates tensor memory): 4 per block
//               and warp, after one wait for the block's decoded weights (one
//               issuing warp for all 12 MMAs of a block was slower);
//   warps 4-15  three decoder teams of four warps; warp w owns tensor-memory
//               lanes 32 (w % 4) .. + 31, i.e. packed rows 32 (w % 4) + lane.
//               Team t decodes the blocks t, t + 3, ...: it first turns the
//               block's int8 codes tile into the fp16 B operand (128-byte
//               swizzle) in the same stage, then each thread reads its
//               row's 64 packed bytes, looks each up in a lane-replicated table
//               of biased weights [w0 + 128, w1 + 128, w2 + 128, 0x64], and
//               builds fp16 pairs with one byte permute (0x64xx is the fp16
//               value 1024 + xx) and one packed subtract of 1152; tcgen05.st
//               writes them into the team's A stage.  Every team drains its own
//               channel d = t of every 1024-column chunk: it adds the fp32 sums
//               into int32 sums (in tensor memory, or with 48..64 tokens in
//               shared memory beside a 4-stage ring, where tensor memory has no
//               room for them), and at the end of the tile writes them as int32
//               partials [split][M][N].
// The partials of the K splits are summed, and the epilogue applied, by the
// split-K finish kernel.  Handing the MMA warp whole blocks matters: with one
// handoff per 16-column step the issuing warp, sharing its scheduler with
// three decoder warps, spent ~830 cycles per step on bookkeeping and waits.
//
// Tensor memory (512 columns): D_d at columns d * NT; int32 sums at 3 NT + d * NT
// when a tile spans more than one chunk and they fit; then team t's A stage, 96 columns, at
// a_col + 96 t (step kk, channel d at + 24 kk + 8 d; 8 columns = 16 fp16 values,
// row r in lane r, column c holding elements 2c (low half) and 2c + 1).
#include <cuda_fp16.h>

#include "tcgen05.cuh"

namespace s3d8 {

namespace wt {

constexpr int ROWS = 128;                        // packed rows per tile (the MMA's M)
constexpr int BK = 64;                           // columns per k-block
constexpr int PK_BYTES = ROWS * BK;              // 8 KiB packed tile
constexpr int MAX_NT = 64;                       // tokens per MMA (N), a multiple of 16
constexpr int ACT_BYTES = MAX_NT * BK * 2;       // 8 KiB fp16 codes tile (the MMA's B operand)
constexpr int ACT8_BYTES = MAX_NT * BK;          // 4 KiB int8 codes tile, as copied
constexpr int STAGE = PK_BYTES + ACT_BYTES + ACT8_BYTES;
constexpr int MAX_LST = 8;                       // ring stages (4 when the chunk sums live in shared memory)
constexpr int LUT_BYTES = kLutEntries * 32 * 4;  // 32 KiB, one copy per lane

constexpr int TEAMS = 3;
constexpr int NBARS = 2 * MAX_LST + TEAMS + 2;
constexpr int THREADS = 512;
constexpr int DEC_WARP0 = 4;
constexpr int DEC_WARPS = TEAMS * 4;
constexpr int CHUNK_BLOCKS = 16;                 // 1024 columns per exact fp32 chunk
constexpr int A_STAGE_COLS = 24;                 // 3 channels x 8 columns

static_assert(STAGE % 1024 == 0 && PK_BYTES % 1024 == 0 && ACT_BYTES % 1024 == 0, "swizzled tiles 1024-aligned");

static_assert(3 * MAX_NT + TEAMS * 4 * A_STAGE_COLS <= 512, "tensor memory");

struct Params {
    int M, N, K, G;
    int nt;        // tokens per MMA: M rounded up to 16
    int rtiles;    // 128-row tiles
    int nsplit;    // K ranges of kbps 64-column blocks
    int kbps;
    int s_col;     // int32 sums at s_col + d * nt (tiles of more than one chunk)
    int a_col;     // team t's A stage (one 64-column block) at a_col + 96 t
    int s_smem;    // chunk sums in shared memory (48..64 tokens, tiles of several chunks)
    const int8_t *C;
    int32_t *part; // [nsplit][M][N]
    int *status;
};

// Position of this CTA in its sequence of 64-column blocks: tile (row tile,
// K split) and block kb inside the tile.
struct Walk {
    int tile, rt, split, kbase, nk;
    int kb;
    int gkb;      // blocks of this CTA before the current one
    int gchunk;   // 1024-column chunks of this CTA before the current one
    bool valid;
};

__device__ __forceinline__ void walk_set_tile(const Params &p, int nkb, Walk &w)
{
    const int total = p.rtiles * p.nsplit;
    w.valid = w.tile < total;
    if (!w.valid)
        return;
    w.rt = w.tile % p.rtiles;
    w.split = w.tile / p.rtiles;
    w.kbase = w.split * p.kbps;
    w.nk = min(p.kbps, nkb - w.kbase);
    w.kb = 0;
}

__device__ __forceinline__ Walk walk_begin(const Params &p, int nkb)
{
    Walk w;
    w.tile = blockIdx.x;
    w.gkb = 0;
    w.gchunk = 0;
    walk_set_tile(p, nkb, w);
    return w;
}

__device__ __forceinline__ void walk_next(const Params &p, int nkb, Walk &w)
{
    ++w.kb;
    ++w.gkb;
    if (w.kb % CHUNK_BLOCKS == 0 || w.kb == w.nk)
        ++w.gchunk;
    if (w.kb == w.nk) {
        w.tile += gridDim.x;
        walk_set_tile(p, nkb, w);
    }
}

// Advances to the first block of the next chunk.
__device__ __forceinline__ void walk_next_chunk(const Params &p, int nkb, Walk &w)
{
    const int c = w.gchunk;
    while (w.valid && w.gchunk == c)
        walk_next(p, nkb, w);
}

__device__ __forceinline__ bool walk_chunk_last_block(const Walk &w)
{
    return w.kb % CHUNK_BLOCKS == CHUNK_BLOCKS - 1 || w.kb == w.nk - 1;
}

__device__ __forceinline__ void mma_f16_tmem_a_elect(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc,
                                                     uint32_t acc)
{
    asm volatile(
        "{\n.reg .pred p, e;\nsetp.ne.b32 p, %4, 0;\nelect.sync _|e, 0xffffffff;\n"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d),
        "r"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}

__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&v)[8])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr),
                 "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
                 : "memory");
}

__device__ __forceinline__ void tmem_ld8u(uint32_t taddr, uint32_t (&r)[8])
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
                   "=r"(r[7])
                 : "r"(taddr));
}

__device__ __forceinline__ uint4 lds128(uint32_t addr)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}

__device__ __forceinline__ uint32_t hsub2(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// Decodes this thread's 16 packed bytes of one 16-column step into the three
// channels' fp16 pairs: a[d][c] holds the weights of columns 2c and 2c + 1.
// The packed tile row `row` (64 bytes) sits at tile + 64 row with its 16-byte
// units permuted by the 64-byte swizzle (unit u at u ^ ((row >> 1) & 3)).
__device__ __forceinline__ void decode_step(uint32_t tile, int row, int kk, uint32_t lut_lane,
                                            uint32_t (&a)[3][8])
{
    const uint4 v = lds128(tile + (uint32_t)row * 64u + ((((uint32_t)kk) ^ (((uint32_t)row >> 1) & 3u)) << 4));
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t L[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const uint32_t byte = prmt(w[i >> 2], 0u, 0x4440u | (uint32_t)(i & 3));
        L[i] = lds_u32_nv(mad_lo_u32(byte, 128u, lut_lane));
    }
    constexpr uint32_t kBias = 0x64806480u;   // fp16 (1152, 1152)
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        a[0][c] = hsub2(prmt(L[2 * c], L[2 * c + 1], 0x7430u), kBias);
        a[1][c] = hsub2(prmt(L[2 * c], L[2 * c + 1], 0x7531u), kBias);
        a[2][c] = hsub2(prmt(L[2 * c], L[2 * c + 1], 0x7632u), kBias);
    }
}

// 2-D bulk tensor copy with an L2 cache policy (whole warp; one elected lane).
__device__ __forceinline__ void tma_2d_hint_elect(uint32_t dst, const CUtensorMap *map, int x, int y, uint32_t bar,
                                                  uint64_t policy)
{
    asm volatile(
        "{\n.reg .pred e;\nelect.sync _|e, 0xffffffff;\n"
        "@e cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], "
        "[%1, {%2, %3}], [%4], %5;\n}\n" ::"r"(dst),
        "l"((uint64_t)map), "r"(x), "r"(y), "r"(bar), "l"(policy)
        : "memory");
}

// The stage's int8 codes tile (nt rows x 64 bytes, as copied) -> the fp16 B
// operand tile (nt rows x 128 bytes, 128-byte swizzle: 16-byte chunk j of row r
// at r * 128 + (j ^ (r % 8)) * 16), by the 128 threads of a decoder team (thread
// i takes 8-code chunks i, i + 128, ...).  Exact without int-to-float
// conversions: with b = code ^ 0x80 = v + 128, one byte permute builds the fp16
// pair 0x64bb (1024 + b) for two codes, and one packed subtract of 1152 leaves v.
__device__ __forceinline__ void codes_tile_to_f16(uint32_t act8, uint32_t act16, int nt, int i)
{
    for (int c = i; c < nt * 8; c += 128) {
        const int r = c >> 3, j = c & 7;
        uint32_t v0, v1;
        asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v0), "=r"(v1) : "r"(act8 + (uint32_t)(c * 8)));
        const uint32_t w[2] = {v0 ^ 0x80808080u, v1 ^ 0x80808080u};
        uint32_t o[4];
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            o[2 * q] = hsub2(prmt(w[q], 0x64646464u, 0x5140u), 0x64806480u);
            o[2 * q + 1] = hsub2(prmt(w[q], 0x64646464u, 0x7362u), 0x64806480u);
        }
        asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(act16 + (uint32_t)(r * 128) +
                                                                       (((uint32_t)j ^ (uint32_t)(r & 7)) << 4)),
                     "r"(o[0]), "r"(o[1]), "r"(o[2]), "r"(o[3])
                     : "memory");
    }
}

// LST: ring stages (8, or 4 when the chunk sums live in shared memory); a
// compile-time constant so that stage indices cost no division.
template <int LST>
__global__ __launch_bounds__(THREADS, 1) void tmem_a_kernel(const __grid_constant__ CUtensorMap tm_act,
                                                            const __grid_constant__ CUtensorMap tm_pk, Params p)
{
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    unsigned char *smem = smem_raw + (base - raw);
    // shared memory: ring, int32 chunk sums (s_smem only), table, barriers
    constexpr bool SSUM = LST != MAX_LST;   // the 4-stage form keeps the chunk sums in shared memory
    const int off_s = LST * STAGE;
    const int off_lut = off_s + (SSUM ? 3 * p.nt * ROWS * 4 : 0);
    const int off_bars = off_lut + LUT_BYTES;
    const uint32_t lut = base + (uint32_t)off_lut;
    const uint32_t bars = base + (uint32_t)off_bars;
    int32_t *ssum = reinterpret_cast<int32_t *>(smem + off_s);   // [channel][token][row]
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + off_bars + NBARS * 8);
    // full/empty: the ring's stages; a_full: each team's A stage is written;
    // acc_full: a chunk's sums are in D; acc_empty: D has been drained
    const uint32_t full = bars, empty = full + 8 * MAX_LST;
    const uint32_t a_full = empty + 8 * MAX_LST;
    const uint32_t acc_full = a_full + 8 * TEAMS, acc_empty = acc_full + 8;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nkb = (p.K + BK - 1) / BK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < LST; ++s) {
            mbar_init(full + 8 * s, 1);
            mbar_init(empty + 8 * s, 4 + 3);   // the block's team, and the three MMA warps
        }
        for (int t = 0; t < TEAMS; ++t) {
            mbar_init(a_full + 8 * t, 4);
        }
        mbar_init(acc_full, 3);
        mbar_init(acc_empty, DEC_WARPS);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    // The copy warp starts the first stages' packed tiles at once, while the
    // table is built: packed weights are never outputs of the kernel before
    // this one (the codes tiles follow after the grid dependency).
    const uint32_t tx = (uint32_t)PK_BYTES + (uint32_t)p.nt * BK;
    int pre = 0;
    // packed bytes are read once: evict them first, keeping the codes tiles
    // (read by every row tile of a K range) in L2
    const uint64_t wpol = l2_evict_first_policy();
    if (warp == 0) {
        __syncwarp();   // lane 0's barrier initialisation
        for (Walk w = walk_begin(p, nkb); w.valid && pre < LST; walk_next(p, nkb, w), ++pre) {
            const uint32_t st = base + (uint32_t)(pre * STAGE);
            tc::mbar_arrive_expect_tx_elect(full + 8 * pre, tx);
            tma_2d_hint_elect(st, &tm_pk, (w.kbase + w.kb) * BK, w.rt * ROWS, full + 8 * pre, wpol);
        }
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(
                         smem_addr(tmem_slot))
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    // table: byte -> [w0 + 128, w1 + 128, w2 + 128, 0x64], one copy per lane
    // (entry b of lane l at lut + 128 b + 4 l)
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
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    bool timed_out = false;
    tc::pdl_launch_dependents();   // the split-K finish may be scheduled; it waits for this grid

    if (warp == 0) {
        // ---- bulk tensor copies: packed tile + int8 codes tile per 64-column block
        tc::pdl_wait();   // the codes may be written by the kernel before this one
        int issued = 0;
        for (Walk w = walk_begin(p, nkb); w.valid; walk_next(p, nkb, w), ++issued) {
            const int s = w.gkb % LST;
            if (w.gkb >= LST && !tc::warp_wait(empty + 8 * s, ((w.gkb / LST) - 1) & 1)) {
                timed_out = true;
                break;
            }
            const uint32_t st = base + (uint32_t)(s * STAGE);
            const int x = (w.kbase + w.kb) * BK;
            if (w.gkb >= pre) {
                tc::mbar_arrive_expect_tx_elect(full + 8 * s, tx);
                tma_2d_hint_elect(st, &tm_pk, x, w.rt * ROWS, full + 8 * s, wpol);
            }
            tc::tma_2d_elect(st + PK_BYTES + ACT_BYTES, &tm_act, x, 0, full + 8 * s);
        }
        // never leave with copies in flight (only possible after a timeout)
        const int hi = issued > pre ? issued : pre;
        for (int v = hi - LST < 0 ? 0 : hi - LST; v < hi; ++v)
            if (!tc::warp_wait(full + 8 * (v % LST), (v / LST) & 1))
                timed_out = true;
    } else if (warp >= 1 && warp <= 3) {
        // ---- MMA issuers: warp 1 + d issues channel d's MMAs into D_d (whole
        // warp, one elected lane); the three accumulators are independent, so the
        // warps need no ordering among themselves.  Block b belongs to team b % 3.
        const int d = warp - 1;
        const uint32_t idesc = (1u << 4) | ((uint32_t)(p.nt >> 3) << 17) | ((uint32_t)(ROWS >> 4) << 24);
        for (Walk w = walk_begin(p, nkb); w.valid; walk_next(p, nkb, w)) {
            const int s = w.gkb % LST, t = w.gkb % TEAMS, use = w.gkb / TEAMS;
            const bool first = w.kb % CHUNK_BLOCKS == 0;
            // (no wait for the ring stage here: the team signals a_full only after
            // it has seen the stage's bulk copies complete)
            if ((first && w.gchunk >= 1 && !tc::warp_wait(acc_empty, (w.gchunk - 1) & 1)) ||
                !tc::warp_wait(a_full + 8 * t, use & 1)) {
                timed_out = true;
                break;
            }
            tc::tc_fence_after();
            const uint32_t acol = tmem + (uint32_t)(p.a_col + t * 4 * A_STAGE_COLS);
            const uint32_t act = base + (uint32_t)(s * STAGE + PK_BYTES);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_f16_tmem_a_elect(tmem + (uint32_t)(d * p.nt), acol + (uint32_t)(kk * A_STAGE_COLS + 8 * d),
                                     tc::sw128_desc(act + kk * 32), idesc, (first && kk == 0) ? 0u : 1u);
            tc::mma_commit_elect(empty + 8 * s);
            if (walk_chunk_last_block(w))
                tc::mma_commit_elect(acc_full);
        }
    } else if (warp >= DEC_WARP0) {
        // ---- decoder teams: team t decodes blocks t, t + 3, ...; every team
        // drains its channel of every chunk, before its first block of a later
        // chunk (or at the end)
        const int t = (warp - DEC_WARP0) / 4, q = warp & 3;
        const int row = 32 * q + lane;
        const uint32_t lut_lane = lut + (uint32_t)lane * 4u;
        const uint32_t lane_off = (uint32_t)(32 * q) << 16;
        const uint32_t acol = tmem + lane_off + (uint32_t)(p.a_col + t * 4 * A_STAGE_COLS);
        Walk w = walk_begin(p, nkb);
        for (int i = 0; i < t && w.valid; ++i)
            walk_next(p, nkb, w);
        Walk cw = walk_begin(p, nkb);   // the next chunk to drain
        int drained = 0;
        while (!timed_out) {
            const int upto = w.gchunk;   // chunks before the current block's (all of them at the end)
            while (drained < upto) {
                const bool first_chunk = cw.kb < CHUNK_BLOCKS;
                const bool last_chunk = cw.kb / CHUNK_BLOCKS == (cw.nk - 1) / CHUNK_BLOCKS;
                if (!tc::warp_wait(acc_full, drained & 1)) {
                    timed_out = true;
                    break;
                }
                tc::tc_fence_after();
                const int g = cw.rt * ROWS + row;
                for (int cb = 0; cb < p.nt / 8; ++cb) {
                    float v[8];
                    uint32_t s8[8];
                    tc::tmem_ld8(tmem + lane_off + (uint32_t)(t * p.nt + cb * 8), v);
                    if (!first_chunk && !SSUM)
                        tmem_ld8u(tmem + lane_off + (uint32_t)(p.s_col + t * p.nt + cb * 8), s8);
                    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
                    // sums in shared memory: entry (channel t, token, row), so a
                    // warp's 32 rows are 32 consecutive words
                    int32_t *srow = ssum + ((size_t)t * p.nt + cb * 8) * ROWS + row;
                    if (!first_chunk && SSUM) {
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            s8[e] = (uint32_t)srow[e * ROWS];
                    }
                    uint32_t sum[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        sum[e] = (uint32_t)(__float2int_rn(v[e]) + (first_chunk ? 0 : (int)s8[e]));
                    if (last_chunk) {
                        const int n = 3 * g + t;
                        if (g < p.G && n < p.N && dcheck(p.status, cw.split < p.nsplit)) {
#pragma unroll
                            for (int e = 0; e < 8; ++e) {
                                const int tok = cb * 8 + e;
                                if (tok < p.M)
                                    p.part[((size_t)cw.split * p.M + tok) * p.N + n] = (int32_t)sum[e];
                            }
                        }
                    } else if (SSUM) {
                        if (dcheck(p.status, (t * p.nt + cb * 8 + 7) * ROWS + row < 3 * p.nt * ROWS)) {
#pragma unroll
                            for (int e = 0; e < 8; ++e)
                                srow[e * ROWS] = (int32_t)sum[e];
                        }
                    } else if (dcheck(p.status, p.s_col + t * p.nt + cb * 8 + 8 <= 512)) {
                        tmem_st8(tmem + lane_off + (uint32_t)(p.s_col + t * p.nt + cb * 8), sum);
                    }
                }
                if (!last_chunk && !SSUM)
                    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
                tc::tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    tc::mbar_arrive(acc_empty);
                walk_next_chunk(p, nkb, cw);
                ++drained;
            }
            if (timed_out || !w.valid)
                break;
            // the team's A stage is free once its previous block (3 back) has been
            // released by the MMAs: that block's ring-stage barrier completes only
            // with the MMAs' commit, and its next phase cannot complete before this
            // wait (it needs this block's MMAs first)
            const int s = w.gkb % LST, use = w.gkb / TEAMS;
            const int prev = w.gkb - TEAMS;
            if ((use >= 1 && !tc::warp_wait(empty + 8 * (prev % LST), (prev / LST) & 1)) ||
                !tc::warp_wait(full + 8 * s, (w.gkb / LST) & 1)) {
                timed_out = true;
                break;
            }
            const uint32_t pk = base + (uint32_t)(s * STAGE);
            if (!dcheck(p.status, s < LST && p.a_col + t * 4 * A_STAGE_COLS + 4 * A_STAGE_COLS <= 512 &&
                                      p.nt <= MAX_NT)) {
                timed_out = true;
                break;
            }
            // the block's codes as the fp16 B operand, for the async proxy (the MMAs)
            codes_tile_to_f16(pk + PK_BYTES + ACT_BYTES, pk + PK_BYTES, p.nt, row);
            fence_proxy_async_smem();
#pragma unroll 1
            for (int kk = 0; kk < 4; ++kk) {
                uint32_t a[3][8];
                decode_step(pk, row, kk, lut_lane, a);
#pragma unroll
                for (int d = 0; d < 3; ++d)
                    tmem_st8(acol + (uint32_t)(kk * A_STAGE_COLS + 8 * d), a[d]);
            }
            asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
            tc::tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                tc::mbar_arrive(a_full + 8 * t);
                tc::mbar_arrive(empty + 8 * s);   // this team's packed bytes of the block are read
            }
            for (int i = 0; i < TEAMS && w.valid; ++i)
                walk_next(p, nkb, w);
        }
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    if (warp == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem) : "memory");
    if (timed_out && lane == 0)
        record_timeout(p.status);
}

}  // namespace wt

static size_t wt_align(size_t v)
{
    return (v + 255) & ~(size_t)255;
}

// 128-row tiles, and K split into ranges so that row tiles x ranges fills the
// SMs without a second wave.
static void wt_plan(int M, int N, int K, int sms, int &rtiles, int &nsplit, int &kbps)
{
    const int G = (N + 2) / 3;
    rtiles = (G + wt::ROWS - 1) / wt::ROWS;
    const int nkb = (K + wt::BK - 1) / wt::BK;
    int s = sms / rtiles;
    if (s < 1)
        s = 1;
    if (s > nkb)
        s = nkb;
    kbps = (nkb + s - 1) / s;
    nsplit = (nkb + kbps - 1) / kbps;
}

bool tmem_supported(int M)
{
    return M >= 1 && M <= wt::MAX_NT;
}

bool tmem_preferred(int M, int N, int K)
{
    // from 5 tokens the grouped GEMV runs its 8-token form, whose dp4a work per
    // byte is the largest; this path is faster there on both 11B shapes (graph-
    // timed on GB300 at 5, 6 and 8 tokens: gate/up 14.4 against 16.8-17.1 us,
    // down 16.3-16.8 against 18.0-18.1 us)
    if (M < 5 || M > wt::MAX_NT)
        return false;
    if (M <= 32)
        return true;
    const int sms = device_sm_count();
    int rtiles, nsplit, kbps;
    wt_plan(M, N, K, sms, rtiles, nsplit, kbps);
    return (long)rtiles * nsplit <= sms;   // one wave of tiles (all but the widest matrices)
}

size_t tmem_workspace_bytes(int M, int N, int K)
{
    int rtiles, nsplit, kbps;
    wt_plan(M, N, K, device_sm_count(), rtiles, nsplit, kbps);
    return 256 + wt_align((size_t)nsplit * M * N * 4);
}

cudaError_t launch_tmem(const LinearArgs &a, cudaStream_t stream)
{
    using namespace wt;
    if (!tmem_supported(a.M))
        return cudaErrorInvalidValue;
    if (!a.ws || a.ws_bytes < tmem_workspace_bytes(a.M, a.N, a.K))
        return cudaErrorInvalidValue;
    auto encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(tensor_map_encoder_fn());
    if (!encode)
        return cudaErrorNotSupported;
    const int sms = device_sm_count();
    int rtiles, nsplit, kbps;
    wt_plan(a.M, a.N, a.K, sms, rtiles, nsplit, kbps);
    const int G = (a.N + 2) / 3;
    const int nt = (a.M + 15) / 16 * 16;
    int32_t *part = reinterpret_cast<int32_t *>(((uintptr_t)a.ws + 255) & ~(uintptr_t)255);

    // the int8 codes [M, K] themselves: the decoder teams turn each block's tile
    // into the fp16 operand in shared memory
    CUtensorMap tm_act, tm_pk;
    const cuuint64_t dA[2] = {(cuuint64_t)a.K, (cuuint64_t)a.M};
    const cuuint64_t sA[1] = {(cuuint64_t)a.K};
    const cuuint32_t boxA[2] = {BK, (cuuint32_t)nt}, es[2] = {1, 1};
    const cuuint64_t dP[2] = {(cuuint64_t)a.K, (cuuint64_t)G};
    const cuuint64_t sP[1] = {(cuuint64_t)a.K};
    const cuuint32_t boxP[2] = {BK, ROWS};
    if (encode(&tm_act, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<int8_t *>(a.xq), dA, sA, boxA, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS ||
        encode(&tm_pk, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(a.packed), dP, sP, boxP, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    static_assert(1024 + MAX_LST * STAGE + LUT_BYTES + NBARS * 8 + 16 <= 232448 - 1024, "shared memory");
    static_assert(1024 + 4 * STAGE + 3 * MAX_NT * ROWS * 4 + LUT_BYTES + NBARS * 8 + 16 <= 232448 - 1024,
                  "shared memory");
    Params p;
    p.M = a.M;
    p.N = a.N;
    p.K = a.K;
    p.G = G;
    p.nt = nt;
    p.rtiles = rtiles;
    p.nsplit = nsplit;
    p.kbps = kbps;
    // tensor memory: D, then the int32 chunk sums if a tile spans several chunks
    // and they fit beside the three teams' A stages, then the A stages; with 48
    // or 64 tokens the sums go to shared memory instead, next to a 4-stage ring
    const bool multi = kbps > CHUNK_BLOCKS;
    p.s_smem = multi && 6 * nt + TEAMS * 4 * A_STAGE_COLS > 512;
    p.s_col = 3 * nt;
    p.a_col = multi && !p.s_smem ? 6 * nt : 3 * nt;
    if (p.a_col + TEAMS * 4 * A_STAGE_COLS > 512)
        return cudaErrorInvalidValue;
    p.C = a.C;
    p.part = part;
    p.status = a.status;
    const long tiles = (long)rtiles * nsplit;
    const long ctas = tiles < sms ? tiles : sms;   // persistent CTAs walk the tiles
    const int lst = p.s_smem ? 4 : MAX_LST;
    const int need = 1024 + lst * STAGE + (p.s_smem ? 3 * nt * ROWS * 4 : 0) + LUT_BYTES + NBARS * 8 + 16;
    auto kernel = p.s_smem ? tmem_a_kernel<4> : tmem_a_kernel<MAX_LST>;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, need);
    if (e != cudaSuccess)
        return e;
    e = tc::launch_pdl(kernel, dim3((unsigned)ctas), dim3(THREADS), (size_t)need, stream, tm_act, tm_pk, p);
    if (e != cudaSuccess)
        return e;
    return launch_splitk_finalize(part, nsplit, a, stream);
}

}  // namespace s3d8
