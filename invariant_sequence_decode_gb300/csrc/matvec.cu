// matvec.cu - narrow-batch q8_0 x q8_0 matvec (1..16 rows), HBM-streaming.
//
// "antirez/ds4 pull 604", Commit walkthrough: each 32-weight block is read
// once and dotted against every token of the batch.  "exact 4-slot
// concurrent serving", How it stays exact: a 4-row batch must use the same
// arithmetic as one row.
//
// Work split: one warp owns G consecutive output rows n and sweeps the whole
// K extent; lane l owns the blocks b = l, l + 32, l + 64, ... of those rows.
// Per block the lane loads the 32 weights (two 16-byte streaming loads, L1
// bypassed) and the fp16 scale once, then for each of the T activation rows
// (L1-resident, shared by all warps) forms the exact int32 block dot with
// eight dp4a and folds it into that row's partial:
//     acc[t] = fma(fp16(wd) * ad[t][b], (float)sumi, acc[t])
// The 32 lane partials are then summed by an xor butterfly (16, 8, 4, 2, 1).
// The order of every floating-point operation on y[t][n] depends only on K:
// not on T, G, the unroll depth U or the grid, so any launch gives the same
// bits for a row as a launch of that row alone.
#include "common.cuh"
#include "kernels.h"

namespace luce {

template <int T, int G, int U>
__global__ void __launch_bounds__(256)
q8_matvec_kernel(const int8_t* __restrict__ wq, const __half* __restrict__ wd, int N, int K,
                 const int8_t* __restrict__ aq, const float* __restrict__ ad,
                 float* y, int64_t ldy, const float* resid, int64_t ldr)
{
    const int lane = threadIdx.x & 31;
    const int warp = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int n0 = warp * G;
    if (n0 >= N) return;
    const int nb = K >> 5;

    const int8_t* wrow[G];
    const __half* drow[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        const int n = min(n0 + g, N - 1);
        wrow[g] = wq + (size_t)n * (size_t)K;
        drow[g] = wd + (size_t)n * (size_t)nb;
    }

    float acc[G][T];
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
        for (int t = 0; t < T; ++t) acc[g][t] = 0.0f;

    for (int b0 = lane; b0 < nb; b0 += 32 * U) {
        int4 w0[U][G], w1[U][G];
        float dw[U][G];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int b = b0 + 32 * u;
            if (b < nb) {
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    const int8_t* p = wrow[g] + (size_t)b * 32;
                    w0[u][g] = ld_stream_v4(p);
                    w1[u][g] = ld_stream_v4(p + 16);
                    dw[u][g] = __half2float(__ushort_as_half(ld_stream_u16(drow[g] + b)));
                }
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int b = b0 + 32 * u;
            if (b < nb) {
#pragma unroll
                for (int t = 0; t < T; ++t) {
                    const int4* pa = reinterpret_cast<const int4*>(aq + (size_t)t * K + (size_t)b * 32);
                    const int4 a0 = __ldg(pa);
                    const int4 a1 = __ldg(pa + 1);
                    const float da = __ldg(ad + (size_t)t * nb + b);
#pragma unroll
                    for (int g = 0; g < G; ++g) {
                        const int s = block_dot(w0[u][g], w1[u][g], a0, a1);
                        acc[g][t] = __fmaf_rn(__fmul_rn(dw[u][g], da), (float)s, acc[g][t]);
                    }
                }
            }
        }
    }

    // Butterfly over the 32 lane partials, then lane (g*T + t) stores y[t][n0+g].
    float mine = 0.0f;
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
        for (int t = 0; t < T; ++t) {
            const float v = warp_sum_butterfly(acc[g][t]);
            if (lane == g * T + t) mine = v;
        }
    if (lane < G * T) {
        const int g = lane / T, t = lane - (lane / T) * T;
        const int n = n0 + g;
        if (n < N) {
            float out = mine;
            if (resid) out = __fadd_rn(resid[(size_t)t * ldr + n], mine);
            y[(size_t)t * ldy + n] = out;
        }
    }
}

template <int T, int G, int U>
static cudaError_t launch_t(const int8_t* wq, const __half* wd, int N, int K, const int8_t* aq,
                            const float* ad, float* y, int64_t ldy, const float* resid, int64_t ldr,
                            cudaStream_t s)
{
    const int warps = (N + G - 1) / G;
    const int blocks = (warps + 7) / 8;
    q8_matvec_kernel<T, G, U><<<blocks, 256, 0, s>>>(wq, wd, N, K, aq, ad, y, ldy, resid, ldr);
    count_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_matvec(const int8_t* wq, const __half* wd, int N, int K, const int8_t* aq,
                          const float* ad, int T, float* y, int64_t ldy, const float* resid,
                          int64_t ldr, cudaStream_t s)
{
    // G (rows per warp) and U (blocks in flight per lane) only shape the
    // memory pipeline; neither changes any row's arithmetic.
    switch (T) {
#define LUCE_MV(TT, GG, UU) \
    case TT: return launch_t<TT, GG, UU>(wq, wd, N, K, aq, ad, y, ldy, resid, ldr, s);
        LUCE_MV(1, 2, 4)
        LUCE_MV(2, 2, 4)
        LUCE_MV(3, 2, 4)
        LUCE_MV(4, 2, 4)
        LUCE_MV(5, 2, 2)
        LUCE_MV(6, 2, 2)
        LUCE_MV(7, 2, 2)
        LUCE_MV(8, 2, 2)
        LUCE_MV(9, 1, 2)
        LUCE_MV(10, 1, 2)
        LUCE_MV(11, 1, 2)
        LUCE_MV(12, 1, 2)
        LUCE_MV(13, 1, 2)
        LUCE_MV(14, 1, 2)
        LUCE_MV(15, 1, 2)
        LUCE_MV(16, 1, 2)
#undef LUCE_MV
        default: return cudaErrorInvalidValue;
    }
}

// ------------------------------------------------------------ block dots

__global__ void q8_block_dots_kernel(const int8_t* __restrict__ wq, int N, int K,
                                     const int8_t* __restrict__ aq, int T, int32_t* __restrict__ out)
{
    const int nb = K >> 5;
    const int64_t total = (int64_t)T * N * nb;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int b = (int)(i % nb);
        const int64_t tn = i / nb;
        const int n = (int)(tn % N);
        const int t = (int)(tn / N);
        const int4* pw = reinterpret_cast<const int4*>(wq + (size_t)n * K + (size_t)b * 32);
        const int4* pa = reinterpret_cast<const int4*>(aq + (size_t)t * K + (size_t)b * 32);
        out[i] = block_dot(pw[0], pw[1], pa[0], pa[1]);
    }
}

cudaError_t launch_block_dots(const int8_t* wq, int N, int K, const int8_t* aq, int T, int32_t* out,
                              cudaStream_t s)
{
    const int64_t total = (int64_t)T * N * (K >> 5);
    const int blocks = (int)((total + 255) / 256 < 65536 ? (total + 255) / 256 : 65536);
    q8_block_dots_kernel<<<blocks, 256, 0, s>>>(wq, N, K, aq, T, out);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace luce
