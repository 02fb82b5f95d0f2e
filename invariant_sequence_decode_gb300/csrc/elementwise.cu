// elementwise.cu - activation quantization and the per-row layer glue:
// RMSNorm -> q8_0, SwiGLU -> q8_0, argmax.
//
// Activation quantization follows "#1209 ... fix QFUSE", What changed and
// why, item 2: a fused producer must quantize with exactly the consumer's
// division and rounding convention.  Here the fused kernels (RMSNorm +
// quantize, SwiGLU + quantize) call the very same per-lane routine as the
// standalone quantizer, on the same fp32 value they also store, so their
// codes equal a standalone quantization of their fp32 output bit for bit.
#include "common.cuh"
#include "kernels.h"

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

// RMSNorm of one row, then q8_0 quantization of the normalised row.  The
// order of the sum of squares depends on H only: the row's 32-value blocks
// are cut into kNormSlices slices, slice c = blocks [c*bpc, (c+1)*bpc), bpc =
// ceil((H/32) / kNormSlices); 4 chains per slice, chain w of slice c taking
// the blocks c*bpc + w, c*bpc + w + 4, ... with lane l adding element 32b + l
// (its square, by fma, in ascending b), the chain's 32 lane partials meeting
// in a butterfly; a slice's sum is its 4 chains added in chain order, the
// row's sum the slice sums in slice order, and r = 1 / sqrt(ss / H + eps)
// (IEEE division and square root).
// Launch: kNormCtasPerRow CTAs of 8 warps per row; warp p of CTA k runs the
// chains p + 8 ((k / 2 + j) % 4), j = 0..3 (chain v = 4c + w), so every CTA
// forms the row's sum in full, and then normalises and quantizes every second
// block (from block k % 2) of its first chain, 8 (k / 2) + p, which spreads
// the per-element divisions over several SMs with few registers per CTA.  gamma
// is read before the wait on the previous kernel, x once.  xcopy (nullable):
// each CTA also stores the raw x values of the blocks it normalises there, so
// the CTAs of a row together copy the row (the decode step reads its input
// rows straight from mapped host memory this way).
constexpr int kNormSlices = 8;
constexpr int kNormChains = 4 * kNormSlices;
constexpr int kNormCtasPerRow = 8;
constexpr int kNormThreads = 256;
static_assert(kNormChains * 2 == kNormCtasPerRow * (kNormThreads / 32), "half a chain per warp");

template <int MAXK, bool HALF>  // MAXK: blocks per chain held in registers (0: loop over x)
__global__ void __launch_bounds__(kNormThreads)
rmsnorm_quant_kernel(const float* __restrict__ x, int H, const float* __restrict__ gamma, float eps,
                     float* __restrict__ xn, int8_t* __restrict__ q, void* d, float* __restrict__ xcopy)
{
    constexpr int NJ = kNormChains / (kNormThreads / 32);  // chains per warp
    constexpr int KR = MAXK > 0 ? MAXK : 1;
    __shared__ float red[kNormChains];
    __shared__ float rs;
    pdl_trigger();
    const int t = blockIdx.y, k = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, p = tid >> 5;
    const int nb = H >> 5;
    const int bpc = (nb + kNormSlices - 1) / kNormSlices;
    auto first = [&](int v) { return (v >> 2) * bpc + (v & 3); };     // first block of chain v
    auto end = [&](int v) { return min(nb, ((v >> 2) + 1) * bpc); };  // its slice's end
    auto chain = [&](int j) { return p + 8 * (((k >> 1) + j) & 3); };
    const int vo = chain(0), half = k & 1;  // this warp normalises blocks half, half + 2, ... of chain vo
    const float* xr = x + (size_t)t * H;
    float gv[KR];
    if (MAXK > 0) {
#pragma unroll
        for (int m = 0; m < KR; ++m) {
            const int b = first(vo) + 4 * m;
            gv[m] = ((m & 1) == half && b < end(vo)) ? gamma[b * 32 + lane] : 0.0f;
        }
    }
    pdl_wait();
    float xv[NJ][KR];
    if (MAXK > 0) {
#pragma unroll
        for (int j = 0; j < NJ; ++j)
#pragma unroll
            for (int m = 0; m < KR; ++m) {
                const int v = chain(j), b = first(v) + 4 * m;
                xv[j][m] = b < end(v) ? xr[b * 32 + lane] : 0.0f;
            }
#pragma unroll
        for (int j = 0; j < NJ; ++j) {
            const int v = chain(j);
            float ss = 0.0f;
#pragma unroll
            for (int m = 0; m < KR; ++m)
                if (first(v) + 4 * m < end(v)) ss = __fmaf_rn(xv[j][m], xv[j][m], ss);
            ss = warp_sum_butterfly(ss);
            if (lane == 0) red[v] = ss;

        }
    } else {
        for (int j = 0; j < NJ; ++j) {
            const int v = chain(j);
            float ss = 0.0f;
            for (int b = first(v); b < end(v); b += 4) {
                const float e = xr[b * 32 + lane];
                ss = __fmaf_rn(e, e, ss);
            }
            ss = warp_sum_butterfly(ss);
            if (lane == 0) red[v] = ss;
        }
    }
    __syncthreads();
    if (tid == 0) {
        float tot = 0.0f;
        for (int c = 0; c < kNormSlices; ++c) {
            float sl = red[4 * c];
            for (int w = 1; w < 4; ++w) sl = __fadd_rn(sl, red[4 * c + w]);
            tot = c == 0 ? sl : __fadd_rn(tot, sl);
        }
        rs = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(tot, (float)H), eps)));
    }
    __syncthreads();
    const float r = rs;
    if (MAXK > 0) {
        // every owned block's quantization computed branch-free (the shuffles
        // and divisions of the blocks interleave), the stores predicated
        constexpr int KH = (KR + 1) / 2;
        float vn[KH], raw[KH];
        Q8Lane qz[KH];
#pragma unroll
        for (int h = 0; h < KH; ++h) {
            // block 2h + half of the chain, picked without indexing by half
            constexpr int dummy = 0;
            const int m1 = 2 * h + 1 < KR ? 2 * h + 1 : dummy;
            const float e = half ? (2 * h + 1 < KR ? xv[0][m1] : 0.0f) : xv[0][2 * h];
            const float g = half ? (2 * h + 1 < KR ? gv[m1] : 0.0f) : gv[2 * h];
            raw[h] = e;
            vn[h] = __fmul_rn(__fmul_rn(e, r), g);
        }
#pragma unroll
        for (int h = 0; h < KH; ++h) qz[h] = q8_quantize_value<HALF>(vn[h]);
#pragma unroll
        for (int h = 0; h < KH; ++h) {
            const int m = 2 * h + half, b = first(vo) + 4 * m;
            if (m < KR && b < end(vo)) {
                const int i = b * 32 + lane;
                if (xcopy) xcopy[(size_t)t * H + i] = raw[h];
                xn[(size_t)t * H + i] = vn[h];
                q[(size_t)t * H + i] = (int8_t)qz[h].code;
                if (lane == 0) q8_store_scale<HALF>(d, (size_t)t * nb + b, qz[h].s);
            }
        }
    } else {
        for (int b = first(vo) + 4 * half; b < end(vo); b += 8) {
            const int i = b * 32 + lane;
            const float e = xr[i];
            if (xcopy) xcopy[(size_t)t * H + i] = e;
            const float vn = __fmul_rn(__fmul_rn(e, r), gamma[i]);
            xn[(size_t)t * H + i] = vn;
            const int code = q8_quantize_store<HALF>(vn, d, (size_t)t * nb + b, lane == 0);
            q[(size_t)t * H + i] = (int8_t)code;
        }
    }
}

template <bool HALF>
static cudaError_t launch_rmsnorm_quant_t(const float* x, int T, int H, const float* gamma, float eps, float* xn,
                                         int8_t* q, void* d, float* xcopy, cudaStream_t s)
{
    const int bpc = ((H >> 5) + kNormSlices - 1) / kNormSlices;
    const int per_chain = (bpc + 3) / 4;
    const dim3 grid(kNormCtasPerRow, T), block(kNormThreads);
    if (per_chain <= 8)
        return launch_pdl(rmsnorm_quant_kernel<8, HALF>, grid, block, s, x, H, gamma, eps, xn, q, d, xcopy);
    if (per_chain <= 16)
        return launch_pdl(rmsnorm_quant_kernel<16, HALF>, grid, block, s, x, H, gamma, eps, xn, q, d, xcopy);
    return launch_pdl(rmsnorm_quant_kernel<0, HALF>, grid, block, s, x, H, gamma, eps, xn, q, d, xcopy);
}

cudaError_t launch_rmsnorm_quant(const float* x, int T, int H, const float* gamma, float eps, float* xn, int8_t* q,
                                 void* d, bool half_scale, cudaStream_t s, float* xcopy)
{
    const cudaError_t e = half_scale ? launch_rmsnorm_quant_t<true>(x, T, H, gamma, eps, xn, q, d, xcopy, s)
                                     : launch_rmsnorm_quant_t<false>(x, T, H, gamma, eps, xn, q, d, xcopy, s);
    count_launches(1);
    return e;
}

// The step's results to the host through mapped (page-locked, device-visible)
// memory: x [n] floats to x_out and am [T] to am_out (either nullable), with
// plain stores that cross the host link inside the kernel.
__global__ void __launch_bounds__(256)
rows_to_host_kernel(const float4* __restrict__ x, int n4, float4* __restrict__ x_out, const int32_t* __restrict__ am,
                    int T, int32_t* __restrict__ am_out)
{
    pdl_trigger();
    pdl_wait();
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (x_out && i < n4) x_out[i] = x[i];
    if (am_out && i < T) am_out[i] = am[i];
}

cudaError_t launch_rows_to_host(const float* x, int64_t n, float* x_out, const int32_t* am, int T, int32_t* am_out,
                                cudaStream_t s)
{
    const int n4 = (int)(n / 4);
    const int work = n4 > T ? n4 : T;
    const cudaError_t e = launch_pdl(rows_to_host_kernel, dim3((unsigned)((work + 255) / 256)), dim3(256), s,
                                     reinterpret_cast<const float4*>(x), n4, reinterpret_cast<float4*>(x_out), am, T,
                                     am_out);
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
