// matvec.cu - narrow-batch q8_0 x q8_0 matvec (1..16 rows), HBM-streaming.
//
// "antirez/ds4 pull 604", Commit walkthrough: each 32-weight block is read
// once and dotted against every token of the batch.  "exact 4-slot
// concurrent serving", How it stays exact: a 4-row batch must use the same
// arithmetic as one row.
//
// Reduction order (a function of K only): the blocks b of a weight row feed
// 32 partial sums ("chains"), block b into chain b mod 32; each chain adds
// its blocks in ascending order, acc = fma(fp16(wd) * ad[t], (float)sumi, acc),
// where sumi is the block's exact int32 dot; the 32 chain values are then
// summed pairwise as an xor butterfly over offsets 16, 8, 4, 2, 1.  Nothing
// in that order depends on the number of activation rows T, on the other
// rows or on the launch shape, so a row of any launch equals the same row
// launched alone, bit for bit.
//
// Work split (GB300): a CTA has 32/KL warps and owns RC = G * 32/KL
// consecutive weight rows.  Lane (r = lane / KL, kb = lane % KL) of warp w runs
// chain c = kb + KL*w of the G rows r, r + 32/KL, ..., so each warp
// instruction reads KL consecutive 32-byte blocks of each of 32/KL rows
// (KL*32 contiguous bytes per row, one 32-byte load per lane, L1 bypassed).
// Each activation block is loaded once per lane and reused for its G rows,
// and is one address shared by the 32/KL lanes of a kb column, which keeps
// the L1-to-register traffic per weight block at (G*32 + T*36)/G bytes (the
// limit of a first version with one row per warp).  A lane keeps the next
// stage of its G rows in flight while it computes the current one; the
// chain values meet in shared memory, where one thread per (row, token)
// applies the butterfly's pairings in the same order.  The int32 block dot
// reaches fp32 either by conversion or through an exact biased dp4a chain;
// the two give the same value.  The decode step's q|k|v projection uses the
// same chains with a RoPE / K/V-append epilogue (q8_qkv_rope_kernel).
#include "common.cuh"
#include "kernels.h"

#ifndef QKV_MMA_MIN
#define QKV_MMA_MIN 9  // measured: the one-layer step at 4 slots x 3 rows 159 -> 145 us, x 4 rows 161 -> 153 us; equal at 2 rows
#endif

namespace luce {

// The chains of lane (r, kb) of warp w (c = kb + KL*w) for the G weight rows
// rows[g]: acc[g][t] = chain c of row rows[g] against token t.  The first
// weight stage is loaded before the wait on the previous kernel.
template <int T, int KL, int G, bool BIAS>
__device__ __forceinline__ void q8_chains(const int8_t* __restrict__ wq, const __half* __restrict__ wd, int K,
                                          const int (&rows)[G], int c, const int8_t* __restrict__ aq,
                                          const float* __restrict__ ad, float (&acc)[G][T])
{
    const int nb = K >> 5;
    const int8_t* wp[G];
    const __half* dp[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        wp[g] = wq + (size_t)rows[g] * K + (size_t)c * 32;
        dp[g] = wd + (size_t)rows[g] * nb + c;
    }
    const int nj = (nb - c + 31) >> 5;  // blocks of this chain (>= 0)
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
        for (int t = 0; t < T; ++t) acc[g][t] = 0.0f;

    auto load = [&](uint32_t (&wv)[G][8], float (&sv)[G], int j) {
#pragma unroll
        for (int g = 0; g < G; ++g) {
            ld_stream_v8(wp[g] + (size_t)j * 1024, wv[g]);
            sv[g] = __half2float(__ushort_as_half(ld_stream_u16(dp[g] + j * 32)));
        }
    };
    auto compute = [&](const uint32_t (&wv)[G][8], const float (&sv)[G], int j) {
        const int b = c + 32 * j;
#pragma unroll
        for (int t = 0; t < T; ++t) {
            uint32_t av[8];
            ld_cached_v8(aq + (size_t)t * K + (size_t)b * 32, av);
            const float da = __ldg(ad + (size_t)t * nb + b);
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const float s = BIAS ? block_dot8_f(wv[g], av) : (float)block_dot8(wv[g], av);
                acc[g][t] = __fmaf_rn(__fmul_rn(sv[g], da), s, acc[g][t]);
            }
        }
    };
    uint32_t wa[G][8], wb[G][8];
    float sa[G], sb[G];
    if (nj > 0) load(wa, sa, 0);  // weights do not depend on the previous kernel
    pdl_wait();                   // activations and the residual do
    for (int j = 0; j < nj; j += 2) {
        if (j + 1 < nj) load(wb, sb, j + 1);
        compute(wa, sa, j);
        if (j + 2 < nj) load(wa, sa, j + 2);
        if (j + 1 < nj) compute(wb, sb, j + 1);
    }
}

template <int T, int KL, int G, bool BIAS>
__global__ void __launch_bounds__(32 * (32 / KL))
q8_matvec_kernel(const int8_t* __restrict__ wq, const __half* __restrict__ wd, int N, int K,
                 const int8_t* __restrict__ aq, const float* __restrict__ ad,
                 float* y, int64_t ldy, const float* resid, int64_t ldr)
{
    constexpr int RW = 32 / KL;
    constexpr int RC = RW * G;
    __shared__ float part[RC][T][33];
    pdl_trigger();
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int r = lane / KL, kb = lane - (lane / KL) * KL;
    const int c = kb + KL * w;
    const int row0 = blockIdx.x * RC;
    int rows[G];
#pragma unroll
    for (int g = 0; g < G; ++g) rows[g] = min(row0 + r + RW * g, N - 1);
    float acc[G][T];
    q8_chains<T, KL, G, BIAS>(wq, wd, K, rows, c, aq, ad, acc);
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
        for (int t = 0; t < T; ++t) part[r + RW * g][t][c] = acc[g][t];
    __syncthreads();
    for (int idx = threadIdx.x; idx < RC * T; idx += blockDim.x) {
        const int rr = idx / T, t = idx - (idx / T) * T;
        const int n = row0 + rr;
        if (n < N) {
            float out = q8_butterfly(part[rr][t]);
            if (resid) out = __fadd_rn(resid[(size_t)t * ldr + n], out);
            y[(size_t)t * ldy + n] = out;
        }
    }
}

template <int T, int KL, int G, bool BIAS>
static cudaError_t launch_t(const int8_t* wq, const __half* wd, int N, int K, const int8_t* aq,
                            const float* ad, float* y, int64_t ldy, const float* resid, int64_t ldr,
                            cudaStream_t s)
{
    constexpr int RC = (32 / KL) * G;
    const cudaError_t e = launch_pdl(q8_matvec_kernel<T, KL, G, BIAS>, dim3((N + RC - 1) / RC),
                                     dim3(32 * (32 / KL)), s, wq, wd, N, K, aq, ad, y, ldy, resid, ldr);
    count_launches(1);
    return e;
}

static cudaError_t launch_matvec_register(const int8_t* wq, const __half* wd, int N, int K, const int8_t* aq,
                                          const float* ad, int T, float* y, int64_t ldy, const float* resid,
                                          int64_t ldr, cudaStream_t s)
{
    // KL (lanes per row), G (rows per lane) and the form of the int-to-float
    // step (conversion, or the exact biased chain) only shape the pipeline;
    // none of them changes any row's arithmetic.
    switch (T) {
#define LUCE_MV(TT, KK, GG, BB) \
    case TT: return launch_t<TT, KK, GG, BB>(wq, wd, N, K, aq, ad, y, ldy, resid, ldr, s);
        LUCE_MV(1, 8, 1, true)
        LUCE_MV(2, 8, 2, false)
        LUCE_MV(3, 8, 3, false)
        LUCE_MV(4, 8, 4, false)
        LUCE_MV(5, 8, 4, true)
        LUCE_MV(6, 8, 4, true)
        LUCE_MV(7, 8, 4, true)
        LUCE_MV(8, 8, 4, true)
        LUCE_MV(9, 8, 2, false)
        LUCE_MV(10, 8, 2, false)
        LUCE_MV(11, 8, 2, false)
        LUCE_MV(12, 8, 3, false)
        LUCE_MV(13, 8, 2, false)
        LUCE_MV(14, 8, 2, false)
        LUCE_MV(15, 8, 2, false)
        LUCE_MV(16, 8, 2, false)
#undef LUCE_MV
        default: return cudaErrorInvalidValue;
    }
}

// Rows from which the tensor-core kernel (matvec_mma.cu) takes over from the
// dp4a TMA ring (measured), for the plain matvec and for the step's q|k|v
// projection (which the dp4a ring serves with RoPE fused at 1..8 rows).
constexpr int kMmaMinRows = 5;
constexpr int kMmaQkvMinRows = QKV_MMA_MIN;
// Rows from which the step's q|k|v runs on the tensor-core ring with RoPE and
// the K/V append fused (measured: one-layer step at 4 slots x 2 rows 103.4 ->
// 99.3 us, 2 x 3 rows 101.4 -> 99.3 us against the fused dp4a ring).
constexpr int kMmaQkvFusedMinRows = 5;

cudaError_t launch_matvec_path(int path, const int8_t* wq, const __half* wd, int N, int K, const int8_t* aq,
                               const float* ad, int T, float* y, int64_t ldy, const float* resid, int64_t ldr,
                               cudaStream_t s)
{
    switch (path) {
        case kMatvecRegister: return launch_matvec_register(wq, wd, N, K, aq, ad, T, y, ldy, resid, ldr, s);
        case kMatvecRing: return launch_matvec_tma(wq, wd, N, K, aq, ad, T, y, ldy, resid, ldr, s);
        case kMatvecMma: return launch_matvec_mma(wq, wd, N, K, aq, ad, T, y, ldy, resid, ldr, s);
        default: break;
    }
    // The library's choice: from kMmaMinRows rows the tensor-core ring, below
    // it the dp4a ring (K a multiple of 256, 16-byte aligned operands), else
    // the register-pipelined kernel.  All give the same bits.
    if (T >= kMmaMinRows) {
        const cudaError_t e = launch_matvec_mma(wq, wd, N, K, aq, ad, T, y, ldy, resid, ldr, s);
        if (e != cudaErrorNotSupported) return e;
    }
    const cudaError_t e = launch_matvec_tma(wq, wd, N, K, aq, ad, T, y, ldy, resid, ldr, s);
    if (e != cudaErrorNotSupported) return e;
    return launch_matvec_register(wq, wd, N, K, aq, ad, T, y, ldy, resid, ldr, s);
}

cudaError_t launch_matvec(const int8_t* wq, const __half* wd, int N, int K, const int8_t* aq,
                          const float* ad, int T, float* y, int64_t ldy, const float* resid,
                          int64_t ldr, cudaStream_t s)
{
    return launch_matvec_path(kMatvecAuto, wq, wd, N, K, aq, ad, T, y, ldy, resid, ldr, s);
}

// ------------------------------------------------------------ q|k|v + RoPE + K/V append
//
// The decode step's q|k|v projection with the RoPE rotation and the K/V
// append done by the CTA that computes the rows ("antirez/ds4 pull 604",
// Commit walkthrough: RoPE per row at the row's position, K/V appended per
// sequence).  The CTA's RC = 8G weight rows are P = RC/2 rotation pairs of one
// head: CTA b serves head h = b / (64/P), pair group q = b % (64/P), and local
// row s is dim q*P + s (s < P) or 64 + q*P + (s - P) of the head.  Each row's
// value is the same chain-and-butterfly result as the plain kernel's; the
// pair then takes exactly the rotation and conversion of the standalone RoPE
// and append kernels (rope_cs, rope_rotate, round-to-nearest binary16), and
// the unrotated q|k|v row is written too.
template <int T, int G, bool BIAS>
__global__ void __launch_bounds__(128)
q8_qkv_rope_kernel(const int8_t* __restrict__ wq, const __half* __restrict__ wd, int K,
                   const int8_t* __restrict__ aq, const float* __restrict__ ad, float* __restrict__ qkv, int Hq,
                   int Hkv, RowPos pos, RopeFreq f, float* __restrict__ q_rot, KvRows kv)
{
    constexpr int KL = 8, RW = 4, RC = RW * G, P = RC / 2, GROUPS = (kHeadDim / 2) / P;
    static_assert((kHeadDim / 2) % P == 0, "rotation pairs must tile the half head");
    __shared__ float part[RC][T][33];
    pdl_trigger();
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int r = lane / KL, kb = lane - (lane / KL) * KL;
    const int c = kb + KL * w;
    const int h = blockIdx.x / GROUPS, q0 = (blockIdx.x % GROUPS) * P;
    auto dim_of = [&](int s) { return s < P ? q0 + s : kHeadDim / 2 + q0 + (s - P); };
    static_assert(P * T <= 128, "one (pair, token) per thread");
    int rows[G];
#pragma unroll
    for (int g = 0; g < G; ++g) rows[g] = h * kHeadDim + dim_of(r + RW * g);
    // thread idx < P*T finishes pair p = idx / T of token t = idx % T; its
    // cos/sin depend only on the position, so they are formed first
    const int idx = threadIdx.x;
    const int p = idx / T, t = idx - (idx / T) * T;
    const int i = q0 + p;
    const bool fin = idx < P * T;
    const float2 cs = (fin && h < Hq + Hkv) ? rope_cs(pos.pos[t], f.inv[i]) : make_float2(1.0f, 0.0f);
    float acc[G][T];
    q8_chains<T, KL, G, BIAS>(wq, wd, K, rows, c, aq, ad, acc);
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
        for (int tt = 0; tt < T; ++tt) part[r + RW * g][tt][c] = acc[g][tt];
    __syncthreads();
    const int ldq = (Hq + 2 * Hkv) * kHeadDim;
    if (fin) {
        float x0 = q8_butterfly(part[p][t]);
        float x1 = q8_butterfly(part[p + P][t]);
        float* yr = qkv + (size_t)t * ldq + (size_t)h * kHeadDim;
        yr[i] = x0;
        yr[i + kHeadDim / 2] = x1;
        const KvRow kr = kv.row[t];
        if (h < Hq + Hkv) rope_rotate(x0, x1, cs.x, cs.y);
        if (h < Hq) {
            float* dst = q_rot + (size_t)t * Hq * kHeadDim + (size_t)h * kHeadDim;
            dst[i] = x0;
            dst[i + kHeadDim / 2] = x1;
        } else {
            __half* dst = (h < Hq + Hkv ? kr.k + (h - Hq) * kr.head_stride : kr.v + (h - Hq - Hkv) * kr.head_stride);
            dst[i] = __float2half_rn(x0);
            dst[i + kHeadDim / 2] = __float2half_rn(x1);
        }
    }
}

template <int T, int G, bool BIAS>
static cudaError_t launch_qkv_t(const int8_t* wq, const __half* wd, int K, const int8_t* aq, const float* ad,
                                float* qkv, int Hq, int Hkv, const RowPos& pos, const RopeFreq& f, float* q_rot,
                                const KvRows& kv, cudaStream_t s)
{
    constexpr int P = 4 * G / 2;
    const cudaError_t e = launch_pdl(q8_qkv_rope_kernel<T, G, BIAS>, dim3((Hq + 2 * Hkv) * ((kHeadDim / 2) / P)),
                                     dim3(128), s, wq, wd, K, aq, ad, qkv, Hq, Hkv, pos, f, q_rot, kv);
    count_launches(1);
    return e;
}

cudaError_t launch_qkv_rope(const int8_t* wq, const __half* wd, int K, const int8_t* aq, const float* ad, int T,
                            float* qkv, int Hq, int Hkv, const RowPos& pos, const RopeFreq& f, float* q_rot,
                            const KvRows& kv, cudaStream_t s)
{
    // From kMmaQkvFusedMinRows rows: the tensor-core ring with RoPE and the
    // K/V append in its epilogue; for shapes it does not take, from
    // kMmaQkvMinRows rows the tensor-core matvec and then RoPE and the append
    // as a launch of their own (the same rotation and rounding either way).
    // Otherwise 1..8 and 13..16 rows on the TMA ring when the shapes allow
    // (matvec_tma.cu), else the plain kernel's launch shapes, except G = 4
    // where the plain kernel takes G = 3 (T = 3, 12): the rotation pairs
    // P = 2G must tile 64
    if (T >= kMmaQkvFusedMinRows) {
        const cudaError_t e = launch_qkv_rope_mma(wq, wd, K, aq, ad, T, qkv, Hq, Hkv, pos, f, q_rot, kv, s);
        if (e != cudaErrorNotSupported) return e;
    }
    if (T >= kMmaQkvMinRows) {
        const int N = (Hq + 2 * Hkv) * kHeadDim;
        const cudaError_t e = launch_matvec_mma(wq, wd, N, K, aq, ad, T, qkv, N, nullptr, 0, s);
        if (e != cudaErrorNotSupported) {
            if (e != cudaSuccess) return e;
            return launch_qkv_rope_kv(qkv, T, Hq, Hkv, pos, f, q_rot, kv, s);
        }
    }
    {
        const cudaError_t e = launch_qkv_rope_tma(wq, wd, K, aq, ad, T, qkv, Hq, Hkv, pos, f, q_rot, kv, s);
        if (e != cudaErrorNotSupported) return e;
    }
    switch (T) {
#define LUCE_QKV(TT, GG, BB) \
    case TT: return launch_qkv_t<TT, GG, BB>(wq, wd, K, aq, ad, qkv, Hq, Hkv, pos, f, q_rot, kv, s);
        LUCE_QKV(1, 1, true)
        LUCE_QKV(2, 2, false)
        LUCE_QKV(3, 4, false)
        LUCE_QKV(4, 4, false)
        LUCE_QKV(5, 4, true)
        LUCE_QKV(6, 4, true)
        LUCE_QKV(7, 4, true)
        LUCE_QKV(8, 4, true)
        LUCE_QKV(9, 2, false)
        LUCE_QKV(10, 2, false)
        LUCE_QKV(11, 2, false)
        LUCE_QKV(12, 4, false)
        LUCE_QKV(13, 2, false)
        LUCE_QKV(14, 2, false)
        LUCE_QKV(15, 2, false)
        LUCE_QKV(16, 2, false)
#undef LUCE_QKV
        default: return cudaErrorInvalidValue;
    }
}

// ------------------------------------------------------------ block dots

__global__ void q8_block_dots_kernel(const int8_t* __restrict__ wq, int N, int K,
                                     const int8_t* __restrict__ aq, int T, int32_t* __restrict__ out)
{
    pdl_trigger();
    pdl_wait();
    const int nb = K >> 5;
    const int64_t total = (int64_t)T * N * nb;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int b = (int)(i % nb);
        const int64_t tn = i / nb;
        const int n = (int)(tn % N);
        const int t = (int)(tn / N);
        uint32_t wv[8], av[8];
        ld_stream_v8(wq + (size_t)n * K + (size_t)b * 32, wv);
        ld_cached_v8(aq + (size_t)t * K + (size_t)b * 32, av);
        out[i] = block_dot8(wv, av);
    }
}

cudaError_t launch_block_dots(const int8_t* wq, int N, int K, const int8_t* aq, int T, int32_t* out,
                              cudaStream_t s)
{
    const int64_t total = (int64_t)T * N * (K >> 5);
    const int blocks = (int)((total + 255) / 256 < 65536 ? (total + 255) / 256 : 65536);
    const cudaError_t e = launch_pdl(q8_block_dots_kernel, dim3(blocks), dim3(256), s, wq, N, K, aq, T, out);
    count_launches(1);
    return e;
}

}  // namespace luce
