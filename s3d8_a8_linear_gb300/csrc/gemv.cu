// CUDA-core S3D8 GEMV / small-M GEMM: decode each packed byte once with the
// expanded shared-memory table and accumulate with dp4a.
//
// One warp owns one packed row g (three output channels) at a time and walks
// the whole of K with 16 bytes per lane per step; the tokens of the current
// block (MT of them) sit in shared memory.  The three k-quads decoded from
// each 4 packed bytes are reused for all MT tokens.  Rows are spread over
// all warps of a persistent grid.  Tokens beyond MT are processed in further
// passes over the weights.
#include "common.cuh"
#include "launch.h"

namespace s3d8 {

constexpr int kGemvThreads = 256;

template <int MT>
__global__ __launch_bounds__(kGemvThreads) void gemv_kernel(
    const uint8_t *__restrict__ packed, const int8_t *__restrict__ C,
    const __nv_bfloat16 *__restrict__ cs, const int8_t *__restrict__ xq,
    const float *__restrict__ xscale, int M, int N, int K, __nv_bfloat16 *__restrict__ out,
    int32_t *__restrict__ acc_out)
{
    extern __shared__ __align__(16) unsigned char smem[];
    uint32_t *lut = reinterpret_cast<uint32_t *>(smem);
    uint32_t *stage = lut + kLutWords;
    int8_t *xs = reinterpret_cast<int8_t *>(stage + kLutStageWords);
    build_lut(lut, stage, C);

    const int lane = threadIdx.x & 31;
    const int warps = kGemvThreads / 32;
    const int gwarp = blockIdx.x * warps + (threadIdx.x >> 5);
    const int nwarps = gridDim.x * warps;
    const int G = (N + 2) / 3;
    const uint32_t lane_base = smem_addr(lut) + 4u * lane;
    const int kchunks = K / 16;

    for (int m0 = 0; m0 < M; m0 += MT) {
        __syncthreads();
        for (int i = threadIdx.x; i < MT * kchunks; i += kGemvThreads) {
            const int t = i / kchunks;
            const int kc = (i - t * kchunks) * 16;
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (m0 + t < M)
                v = __ldg(reinterpret_cast<const uint4 *>(xq + (size_t)(m0 + t) * K + kc));
            *reinterpret_cast<uint4 *>(xs + (size_t)t * K + kc) = v;
        }
        __syncthreads();

        for (int g = gwarp; g < G; g += nwarps) {
            int acc[MT][3];
#pragma unroll
            for (int t = 0; t < MT; ++t)
                acc[t][0] = acc[t][1] = acc[t][2] = 0;
            const uint8_t *prow = packed + (size_t)g * K;
#pragma unroll 2
            for (int k = lane * 16; k < K; k += 512) {
                const uint4 p = ldg_stream_v4(prow + k);
                uint32_t V[4][3];
                decode_quad(p.x, lane_base, V[0][0], V[0][1], V[0][2]);
                decode_quad(p.y, lane_base, V[1][0], V[1][1], V[1][2]);
                decode_quad(p.z, lane_base, V[2][0], V[2][1], V[2][2]);
                decode_quad(p.w, lane_base, V[3][0], V[3][1], V[3][2]);
#pragma unroll
                for (int t = 0; t < MT; ++t) {
                    const uint4 xv = *reinterpret_cast<const uint4 *>(xs + (size_t)t * K + k);
                    const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
#pragma unroll
                        for (int d = 0; d < 3; ++d)
                            acc[t][d] = __dp4a((int)V[q][d], (int)xw[q], acc[t][d]);
                    }
                }
            }
            int mine = 0;
#pragma unroll
            for (int t = 0; t < MT; ++t) {
#pragma unroll
                for (int d = 0; d < 3; ++d) {
                    const int s = warp_sum(acc[t][d]);
                    if (lane == t * 3 + d)
                        mine = s;
                }
            }
            if (lane < 3 * MT) {
                const int t = lane / 3;
                const int d = lane - 3 * t;
                const int m = m0 + t;
                const int n = 3 * g + d;
                if (m < M && n < N) {
                    if (acc_out)
                        acc_out[(size_t)m * N + n] = mine;
                    else
                        out[(size_t)m * N + n] = epilogue_bf16(mine, xscale[m], cs[n]);
                }
            }
        }
    }
}

template <int MT>
static cudaError_t launch_gemv_mt(const LinearArgs &a, cudaStream_t stream)
{
    const size_t smem = (size_t)(kLutWords + kLutStageWords) * 4 + (size_t)MT * a.K;
    cudaError_t e = cudaFuncSetAttribute(gemv_kernel<MT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, gemv_kernel<MT>, kGemvThreads, smem);
    if (e != cudaSuccess)
        return e;
    if (per_sm < 1)
        per_sm = 1;
    const int G = (a.N + 2) / 3;
    const int want = (G + kGemvThreads / 32 - 1) / (kGemvThreads / 32);
    const int cap = device_sm_count() * per_sm;
    const int grid = want < cap ? want : cap;
    gemv_kernel<MT><<<grid, kGemvThreads, smem, stream>>>(a.packed, a.C, a.cs, a.xq, a.xscale, a.M,
                                                          a.N, a.K, a.out, a.acc);
    return cudaGetLastError();
}

// Largest token block whose activations fit next to the table in shared memory.
static int gemv_token_block(int M, int K)
{
    const size_t budget = 190 * 1024 - (size_t)(kLutWords + kLutStageWords) * 4;
    int mt = 8;
    while (mt > 1 && (size_t)mt * K > budget)
        mt >>= 1;
    while (mt > 1 && mt / 2 >= M)
        mt >>= 1;
    return mt;
}

cudaError_t launch_gemv(const LinearArgs &a, cudaStream_t stream)
{
    switch (gemv_token_block(a.M, a.K)) {
    case 1: return launch_gemv_mt<1>(a, stream);
    case 2: return launch_gemv_mt<2>(a, stream);
    case 4: return launch_gemv_mt<4>(a, stream);
    default: return launch_gemv_mt<8>(a, stream);
    }
}

}  // namespace s3d8
