// common.cuh - device helpers shared by the kernels of libluce.
//
// Every floating-point step below is an explicit round-to-nearest intrinsic
// (__fmaf_rn, __fmul_rn, __fadd_rn, __fdiv_rn, __fsqrt_rn), so the compiler
// can neither contract nor reorder it.  That, plus reduction orders that
// depend only on the problem's own sizes, is what makes every row of a
// batched launch bit-identical to a launch of that row alone.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#define LUCE_QK 32

namespace luce {

constexpr int kQK = 32;
constexpr int kHeadDim = 128;
constexpr int kMaxRows = 16;
constexpr int kMaxSeq = 4;
constexpr int kAttnChunk = 256;

// ---------------------------------------------------------------- loads

// 16-byte streaming load for data read exactly once (weights): bypass L1 so
// the activations that every warp re-reads keep the L1.
__device__ __forceinline__ int4 ld_stream_v4(const void* p)
{
    int4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.s32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ unsigned short ld_stream_u16(const void* p)
{
    unsigned short r;
    asm volatile("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(r) : "l"(p));
    return r;
}

// ---------------------------------------------------------------- q8_0

// Integer dot of one 32-value block held as two 16-byte vectors per side.
// Exact: |result| <= 32 * 127 * 127 < 2^24.
__device__ __forceinline__ int block_dot(const int4 w0, const int4 w1, const int4 a0, const int4 a1)
{
    int s = __dp4a(w0.x, a0.x, 0);
    s = __dp4a(w0.y, a0.y, s);
    s = __dp4a(w0.z, a0.z, s);
    s = __dp4a(w0.w, a0.w, s);
    s = __dp4a(w1.x, a1.x, s);
    s = __dp4a(w1.y, a1.y, s);
    s = __dp4a(w1.z, a1.z, s);
    s = __dp4a(w1.w, a1.w, s);
    return s;
}

// One quantization code: q = round-half-away(x / d) clamped to [-127, 127];
// 0 when d == 0 or the quotient is NaN.
__device__ __forceinline__ int q8_code(float x, float d)
{
    if (d == 0.0f) return 0;
    float r = __fdiv_rn(x, d);
    if (r != r) return 0;
    r = roundf(r);
    r = fminf(fmaxf(r, -127.0f), 127.0f);
    return (int)r;
}

// Warp-cooperative quantization of one 32-value block: lane i holds x_i.
// Returns lane i's code; *d_out receives the block scale on every lane.
// amax uses fmaxf (NaN operands are dropped), an order-free reduction.
__device__ __forceinline__ int q8_quantize_lane(float x, float* d_out)
{
    float a = fabsf(x);
    float amax = (a == a) ? a : 0.0f;
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    float d = __fdiv_rn(amax, 127.0f);
    *d_out = d;
    return q8_code(x, d);
}

// Pairwise xor-butterfly sum over the 32 lanes (offsets 16, 8, 4, 2, 1).
// Both lanes of a pair add the same two values, so all lanes end equal.
__device__ __forceinline__ float warp_sum_butterfly(float v)
{
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, off));
    return v;
}

__device__ __forceinline__ float warp_max(float v)
{
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
    return v;
}

// ---------------------------------------------------------------- RoPE

// Rotation of one (x0, x1) pair by (c, s) in fp32, no contraction.
__device__ __forceinline__ void rope_rotate(float& x0, float& x1, float c, float s)
{
    const float a = __fsub_rn(__fmul_rn(x0, c), __fmul_rn(x1, s));
    const float b = __fadd_rn(__fmul_rn(x0, s), __fmul_rn(x1, c));
    x0 = a;
    x1 = b;
}

// cos/sin of pos * theta^(-2i/D), evaluated in double and rounded to fp32.
__device__ __forceinline__ float2 rope_cs(int pos, int i, int D, double theta)
{
    const double inv = pow(theta, -2.0 * (double)i / (double)D);
    const double ang = (double)pos * inv;
    double s, c;
    sincos(ang, &s, &c);
    return make_float2((float)c, (float)s);
}

// ---------------------------------------------------------------- SwiGLU

__device__ __forceinline__ float silu_mul(float g, float u)
{
    const float e = expf(-g);
    const float sg = __fdiv_rn(g, __fadd_rn(1.0f, e));
    return __fmul_rn(sg, u);
}

}  // namespace luce
