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
#include <string.h>

#include <vector>

#define LUCE_QK 32

namespace luce {

// ---------------------------------------------------------------- launch

// Programmatic dependent launch: every kernel lets the next kernel of the
// stream start as soon as all of its own CTAs are running (pdl_trigger at
// entry); the next kernel does only work that reads nothing the previous
// kernel writes (weight loads, L2 prefetches) before pdl_wait, which returns
// once the previous kernel has completed and its writes are visible.  Both
// are no-ops for a launch without the attribute.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// A launch written down instead of issued.  While a thread's t_launch_log is
// set, launch_pdl_smem appends the kernel, its shape and a copy of its
// arguments (each at its own alignment, the gaps zeroed, so two records of
// equal launches compare equal byte for byte) to the log, and the host-device
// copies of the decode step go there too; the step graph (api.cu) builds a
// CUDA graph from such a log and refreshes its nodes from the next one.
struct LaunchRec {
    static constexpr int kMaxArgs = 24;
    static constexpr int kArgBytes = 3072;
    LaunchRec() {}  // fields are set by the recorder; the argument bytes are never zero-filled in bulk
    bool copy;  // a cudaMemcpyAsync (dst, src, bytes, dir), not a kernel
    const void* func;
    dim3 grid, block;
    size_t smem;
    int nargs, nbytes;
    uint16_t off[kMaxArgs];
    void* dst;
    const void* src;
    size_t bytes;
    cudaMemcpyKind dir;
    alignas(64) unsigned char args[kArgBytes];
};

struct LaunchLog {
    std::vector<LaunchRec> recs;
    bool overflow = false;  // a launch had more arguments or bytes than a record holds
};

extern thread_local LaunchLog* t_launch_log;

template <typename A>
static inline bool rec_put(LaunchRec& r, int& off, const A& a)
{
    const int at = (off + (int)alignof(A) - 1) & ~((int)alignof(A) - 1);
    if (r.nargs >= LaunchRec::kMaxArgs || at + (int)sizeof(A) > LaunchRec::kArgBytes) return false;
    memset(r.args + off, 0, (size_t)(at - off));
    memcpy(r.args + at, &a, sizeof(A));
    r.off[r.nargs++] = (uint16_t)at;
    off = at + (int)sizeof(A);
    return true;
}

template <typename... KArgs>
static inline cudaError_t rec_kernel(LaunchLog* log, void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                     const KArgs&... args)
{
    log->recs.emplace_back();
    LaunchRec& r = log->recs.back();
    r.copy = false;
    r.func = reinterpret_cast<const void*>(kernel);
    r.grid = grid;
    r.block = block;
    r.smem = smem;
    r.nargs = 0;
    r.dst = nullptr;
    r.src = nullptr;
    r.bytes = 0;
    r.dir = cudaMemcpyDefault;
    int off = 0;
    bool ok = true;
    ((ok = ok && rec_put(r, off, args)), ...);
    r.nbytes = off;
    if (!ok) {
        log->overflow = true;
        return cudaErrorInvalidValue;
    }
    return cudaSuccess;
}

template <typename... KArgs, typename... Args>
static inline cudaError_t launch_pdl_smem(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                          cudaStream_t s, Args... args)
{
    if (LaunchLog* log = t_launch_log)
        return rec_kernel<KArgs...>(log, kernel, grid, block, smem, static_cast<KArgs>(args)...);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

template <typename... KArgs, typename... Args>
static inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, cudaStream_t s,
                                     Args... args)
{
    return launch_pdl_smem(kernel, grid, block, 0, s, args...);
}

constexpr int kHeadDim = 128;
constexpr int kAttnChunk = 256;  // largest split-K chunk (keys)

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

// 32-byte loads (one whole q8_0 block per lane); the address must be 32-byte
// aligned.  Streaming variant for weights, L1-cached variant for activations
// that every warp of the CTA re-reads.
__device__ __forceinline__ void ld_stream_v8(const void* p, uint32_t (&v)[8])
{
    asm volatile("ld.global.nc.L1::no_allocate.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7])
                 : "l"(p));
}

__device__ __forceinline__ void ld_cached_v8(const void* p, uint32_t (&v)[8])
{
    asm volatile("ld.global.nc.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7])
                 : "l"(p));
}

// Ask the memory system to stage `bytes` (multiple of 16, 16-byte aligned
// address) into L2 ahead of use.
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// ---------------------------------------------------------------- q8_0

// Integer dot of one 32-value block held as 8 words per side, as two
// independent dp4a chains (integer sums are exact in any order).
// Exact: |result| <= 32 * 127 * 127 < 2^24.
__device__ __forceinline__ int block_dot8(const uint32_t (&w)[8], const uint32_t (&a)[8])
{
    int s0 = __dp4a((int)w[0], (int)a[0], 0);
    int s1 = __dp4a((int)w[4], (int)a[4], 0);
    s0 = __dp4a((int)w[1], (int)a[1], s0);
    s1 = __dp4a((int)w[5], (int)a[5], s1);
    s0 = __dp4a((int)w[2], (int)a[2], s0);
    s1 = __dp4a((int)w[6], (int)a[6], s1);
    s0 = __dp4a((int)w[3], (int)a[3], s0);
    s1 = __dp4a((int)w[7], (int)a[7], s1);
    return s0 + s1;
}

// The same dot returned as a float, exactly: one dp4a chain seeded with the
// bits of 1.5 * 2^23, so the int32 result is the float 1.5 * 2^23 + dot
// (|dot| <= 516,128 < 2^22 keeps it inside that binade), and one exact
// subtraction leaves (float)dot without an integer-to-float conversion.
__device__ __forceinline__ float block_dot8_f(const uint32_t (&w)[8], const uint32_t (&a)[8])
{
    int s = __dp4a((int)w[0], (int)a[0], 0x4B400000);
#pragma unroll
    for (int i = 1; i < 8; ++i) s = __dp4a((int)w[i], (int)a[i], s);
    return __fsub_rn(__int_as_float(s), 12582912.0f);
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

// The half-scale form of the same quantizer: the block scale is stored as
// binary16.  d = amax / 127 (fp32, IEEE division) is rounded to the nearest
// binary16; a scale that overflows binary16 is replaced by the largest finite
// half, 65504, so the stored scale is always finite; the codes are taken
// against the stored scale, q = round(x / float(d16)) with the division and
// rounding of q8_code (a stored scale of zero gives all-zero codes).  Returns
// lane i's code; *d_out receives the scale's binary16 bits on every lane.
__device__ __forceinline__ int q8_quantize_lane_h(float x, uint16_t* d_out)
{
    float a = fabsf(x);
    float amax = (a == a) ? a : 0.0f;
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    __half h = __float2half_rn(__fdiv_rn(amax, 127.0f));
    if (__hisinf(h)) h = __ushort_as_half((unsigned short)0x7BFF);
    *d_out = __half_as_ushort(h);
    return q8_code(x, __half2float(h));
}

// One lane's quantization in either form; the scale goes to d (fp32 or
// binary16 bits) at block index bi when write_scale.
template <bool HALF>
__device__ __forceinline__ int q8_quantize_store(float x, void* d, size_t bi, bool write_scale)
{
    if (HALF) {
        uint16_t dh;
        const int code = q8_quantize_lane_h(x, &dh);
        if (write_scale) static_cast<uint16_t*>(d)[bi] = dh;
        return code;
    }
    float dd;
    const int code = q8_quantize_lane(x, &dd);
    if (write_scale) static_cast<float*>(d)[bi] = dd;
    return code;
}

// The same quantization with the scale returned instead of stored: s holds
// the fp32 bits (or the binary16 bits when HALF) for q8_store_scale.
struct Q8Lane {
    int code;
    uint32_t s;
};
template <bool HALF>
__device__ __forceinline__ Q8Lane q8_quantize_value(float x)
{
    Q8Lane r;
    if (HALF) {
        uint16_t dh;
        r.code = q8_quantize_lane_h(x, &dh);
        r.s = dh;
    } else {
        float dd;
        r.code = q8_quantize_lane(x, &dd);
        r.s = __float_as_uint(dd);
    }
    return r;
}

template <bool HALF>
__device__ __forceinline__ void q8_store_scale(void* d, size_t bi, uint32_t s)
{
    if (HALF)
        static_cast<uint16_t*>(d)[bi] = (uint16_t)s;
    else
        static_cast<float*>(d)[bi] = __uint_as_float(s);
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

// The 32 chain values of one (row, token), combined by the xor butterfly's
// pairings: v[i] += v[i + off] for off = 16, 8, 4, 2, 1.
__device__ __forceinline__ float q8_butterfly(const float* __restrict__ part)
{
    float v[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = part[i];
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1)
#pragma unroll
        for (int i = 0; i < off; ++i) v[i] = __fadd_rn(v[i], v[i + off]);
    return v[0];
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

// cos/sin of the angle pos * inv_freq (inv_freq = theta^(-2i/D), evaluated
// in double on the host).  The angle is formed in double and reduced modulo
// 2*pi by Cody-Waite with a two-term 2*pi (the remainder keeps ~1e-12
// absolute accuracy up to position 32767 and far beyond), then rounded to
// fp32 (|r| <= pi, error <= 2e-7) for sincosf.
__device__ __forceinline__ float2 rope_cs(int pos, double inv_freq)
{
    const double ang = (double)pos * inv_freq;
    const double k = rint(ang * 0.15915494309189535);
    double r = fma(-k, 6.283185307179586, ang);
    r = fma(-k, 2.4492935982947064e-16, r);
    float s, c;
    sincosf((float)r, &s, &c);
    return make_float2(c, s);
}

// ---------------------------------------------------------------- SwiGLU

__device__ __forceinline__ float silu_mul(float g, float u)
{
    const float e = expf(-g);
    const float sg = __fdiv_rn(g, __fadd_rn(1.0f, e));
    return __fmul_rn(sg, u);
}

}  // namespace luce
