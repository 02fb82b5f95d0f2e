// elementwise.cu - activation quantization and the per-row layer glue:
// RMSNorm -> q8_0, SwiGLU -> q8_0, argmax.
//
// Activation quantization follows "#1209 ... fix QFUSE", What changed and
// why, item 2: a fused producer must quantize with exactly the consumer's
// division and rounding convention.  Here the fused kernels (RMSNorm +
// quantize, SwiGLU + quantize) call the very same per-lane routine as the
// standalone quantizer, on the same fp32 value they also store, so their
// codes equal a standalone quantization of their fp32 output bit for bit.
#include <cooperative_groups.h>

#include "common.cuh"
#include "kernels.h"

namespace cg = cooperative_groups;

namespace luce {

// One warp per 32-value block; lane i quantizes element i.  HALF: the
// scales are stored as binary16 (q8_quantize_lane_h).
template <bool HALF>
__global__ void __launch_bounds__(256)
quantize_kernel(const float* __restrict__ x, int T, int K, int64_t ldx, int8_t* __restrict__ q, void* d)
{
    pdl_trigger();
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int nb = K >> 5;
    const int64_t blk = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (blk >= (int64_t)T * nb) return;
    const int t = (int)(blk / nb), b = (int)(blk - (int64_t)t * nb);
    const float v = x[(size_t)t * ldx + (size_t)b * 32 + lane];
    const int code = q8_quantize_store<HALF>(v, d, (size_t)t * nb + b, lane == 0);
    q[(size_t)t * K + (size_t)b * 32 + lane] = (int8_t)code;
}

cudaError_t launch_quantize(const float* x, int T, int K, int64_t ldx, int8_t* q, void* d, bool half_scale,
                            cudaStream_t s)
{
    const int64_t blocks = (int64_t)T * (K >> 5);
    const dim3 grid((unsigned)((blocks + 7) / 8));
    const cudaError_t e = half_scale ? launch_pdl(quantize_kernel<true>, grid, dim3(256), s, x, T, K, ldx, q, d)
                                     : launch_pdl(quantize_kernel<false>, grid, dim3(256), s, x, T, K, ldx, q, d);
    count_launches(1);
    return e;
}

// RMSNorm of one row by a cluster of kNormCtas CTAs (128 threads each), then
// q8_0 quantization of the normalised row.  CTA c of the row owns the
// 32-value blocks [c*bpc, (c+1)*bpc), bpc = ceil((H/32) / kNormCtas); its warp
// w the blocks c*bpc + w, c*bpc + w + 4, ... and lane l element 32b + l of
// each, read once and kept in registers (gamma is read before the wait on the
// previous kernel).  Sum of squares, in an order that depends on H only: each
// thread adds its elements' squares with fma in ascending b; warp partials by
// butterfly; thread 0 adds its CTA's 4 warp sums in warp order; every thread
// then adds the kNormCtas CTA sums in rank order, read from the CTAs' shared
// memory, so all CTAs of the row hold the same r = 1 / sqrt(ss / H + eps)
// (IEEE division and square root).
constexpr int kNormCtas = 8;
constexpr int kNormThreads = 128;
constexpr int kNormMaxPerThread = 16;  // blocks per warp on the register path: H <= 16384

template <bool REG, bool HALF>
__global__ void __launch_bounds__(kNormThreads)
rmsnorm_quant_kernel(const float* __restrict__ x, int H, const float* __restrict__ gamma, float eps,
                     float* __restrict__ xn, int8_t* __restrict__ q, void* d)
{
    constexpr int NW = kNormThreads / 32;
    __shared__ float red[NW];
    __shared__ float part;
    cg::cluster_group cluster = cg::this_cluster();
    pdl_trigger();
    const int c = (int)cluster.block_rank();
    const int t = blockIdx.y;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nb = H >> 5;
    const int bpc = (nb + kNormCtas - 1) / kNormCtas;
    const int b0 = c * bpc, b1 = min(nb, b0 + bpc);
    const float* xr = x + (size_t)t * H;
    float v[kNormMaxPerThread], gv[kNormMaxPerThread];
    if (REG) {
#pragma unroll
        for (int k = 0; k < kNormMaxPerThread; ++k) {
            const int b = b0 + warp + NW * k;
            gv[k] = b < b1 ? gamma[b * 32 + lane] : 0.0f;
        }
    }
    pdl_wait();
    float ss = 0.0f;
    if (REG) {
#pragma unroll
        for (int k = 0; k < kNormMaxPerThread; ++k) {
            const int b = b0 + warp + NW * k;
            v[k] = b < b1 ? xr[b * 32 + lane] : 0.0f;
        }
#pragma unroll
        for (int k = 0; k < kNormMaxPerThread; ++k)
            if (b0 + warp + NW * k < b1) ss = __fmaf_rn(v[k], v[k], ss);
    } else {
        for (int b = b0 + warp; b < b1; b += NW) {
            const float e = xr[b * 32 + lane];
            ss = __fmaf_rn(e, e, ss);
        }
    }
    ss = warp_sum_butterfly(ss);
    if (lane == 0) red[warp] = ss;
    __syncthreads();
    if (tid == 0) {
        float s = red[0];
        for (int w = 1; w < NW; ++w) s = __fadd_rn(s, red[w]);
        part = s;
    }
    cluster.sync();  // every CTA's sum is in place
    float tot = *cluster.map_shared_rank(&part, 0);
    for (int cc = 1; cc < kNormCtas; ++cc) tot = __fadd_rn(tot, *cluster.map_shared_rank(&part, cc));
    // done reading the other CTAs' sums: arrive now, wait only before leaving
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    const float r = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(tot, (float)H), eps)));
#pragma unroll
    for (int k = 0; k < (REG ? kNormMaxPerThread : 1); ++k) {
        for (int b = b0 + warp + NW * k; b < b1; b += (REG ? nb : NW)) {
            const int i = b * 32 + lane;
            const float e = REG ? v[k] : xr[i];
            const float vn = __fmul_rn(__fmul_rn(e, r), REG ? gv[k] : gamma[i]);
            xn[(size_t)t * H + i] = vn;
            const int code = q8_quantize_store<HALF>(vn, d, (size_t)t * nb + b, lane == 0);
            q[(size_t)t * H + i] = (int8_t)code;
        }
    }
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");  // no CTA leaves while another may still read its sum
}

template <bool HALF>
static cudaError_t launch_rmsnorm_quant_t(const float* x, int T, int H, const float* gamma, float eps, float* xn,
                                         int8_t* q, void* d, cudaStream_t s)
{
    const int bpc = ((H >> 5) + kNormCtas - 1) / kNormCtas;
    const dim3 grid(kNormCtas, T);
    return bpc <= (kNormThreads / 32) * kNormMaxPerThread
               ? launch_pdl_cluster(rmsnorm_quant_kernel<true, HALF>, grid, dim3(kNormThreads), kNormCtas, s, x, H,
                                    gamma, eps, xn, q, d)
               : launch_pdl_cluster(rmsnorm_quant_kernel<false, HALF>, grid, dim3(kNormThreads), kNormCtas, s, x, H,
                                    gamma, eps, xn, q, d);
}

cudaError_t launch_rmsnorm_quant(const float* x, int T, int H, const float* gamma, float eps, float* xn, int8_t* q,
                                 void* d, bool half_scale, cudaStream_t s)
{
    const cudaError_t e = half_scale ? launch_rmsnorm_quant_t<true>(x, T, H, gamma, eps, xn, q, d, s)
                                     : launch_rmsnorm_quant_t<false>(x, T, H, gamma, eps, xn, q, d, s);
    count_launches(1);
    return e;
}

// SwiGLU of the concatenated gate||up row (gate first), then q8_0.
template <bool HALF>
__global__ void __launch_bounds__(256)
swiglu_quant_kernel(const float* __restrict__ gu, int T, int F, float* __restrict__ h, int8_t* __restrict__ q,
                    void* d)
{
    pdl_trigger();
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int nb = F >> 5;
    const int64_t blk = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (blk >= (int64_t)T * nb) return;
    const int t = (int)(blk / nb), b = (int)(blk - (int64_t)t * nb);
    const int i = b * 32 + lane;
    const float g = gu[(size_t)t * 2 * F + i];
    const float u = gu[(size_t)t * 2 * F + F + i];
    const float v = silu_mul(g, u);
    h[(size_t)t * F + i] = v;
    const int code = q8_quantize_store<HALF>(v, d, (size_t)t * nb + b, lane == 0);
    q[(size_t)t * F + i] = (int8_t)code;
}

cudaError_t launch_swiglu_quant(const float* gu, int T, int F, float* h, int8_t* q, void* d, bool half_scale,
                                cudaStream_t s)
{
    const int64_t blocks = (int64_t)T * (F >> 5);
    const dim3 grid((unsigned)((blocks + 7) / 8));
    const cudaError_t e = half_scale ? launch_pdl(swiglu_quant_kernel<true>, grid, dim3(256), s, gu, T, F, h, q, d)
                                     : launch_pdl(swiglu_quant_kernel<false>, grid, dim3(256), s, gu, T, F, h, q, d);
    count_launches(1);
    return e;
}

// Argmax of each row, lowest index on ties, NaN never chosen (all-NaN -> 0).
// The (value, index) winner is unique, so the reduction order is free.
__device__ __forceinline__ void better(float& bv, int& bi, float v, int i)
{
    if (v != v) return;
    if (bi < 0 || v > bv || (v == bv && i < bi)) {
        bv = v;
        bi = i;
    }
}

__global__ void __launch_bounds__(1024)
argmax_kernel(const float* __restrict__ x, int V, int32_t* __restrict__ out)
{
    __shared__ float sv[32];
    __shared__ int si[32];
    pdl_trigger();
    pdl_wait();
    const int t = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const float* r = x + (size_t)t * V;
    float bv = 0.0f;
    int bi = -1;
    for (int i = tid; i < V; i += blockDim.x) better(bv, bi, r[i], i);
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
        if (oi >= 0) better(bv, bi, ov, oi);
    }
    if (lane == 0) {
        sv[warp] = bv;
        si[warp] = bi;
    }
    __syncthreads();
    if (tid == 0) {
        float fv = 0.0f;
        int fi = -1;
        for (int w = 0; w < (int)(blockDim.x >> 5); ++w)
            if (si[w] >= 0) better(fv, fi, sv[w], si[w]);
        out[t] = fi < 0 ? 0 : fi;
    }
}

cudaError_t launch_argmax(const float* x, int T, int V, int32_t* out, cudaStream_t s)
{
    const cudaError_t e = launch_pdl(argmax_kernel, dim3(T), dim3(1024), s, x, V, out);
    count_launches(1);
    return e;
}

}  // namespace luce
