// matvec_tma.cu - the q8_0 matvec for 1..4 activation rows, with the weights
// streamed through shared memory by the tensor memory accelerator (TMA).
//
// Arithmetic: the same as q8_matvec_kernel (matvec.cu).  Block b of a weight
// row feeds chain b mod 32; each chain adds its blocks in ascending order,
// acc = fma(fp16(wd) * ad[t], (float)sumi, acc); the 32 chain values meet in
// the xor butterfly over offsets 16, 8, 4, 2, 1.  Only the way the bytes reach
// the lanes differs, so both kernels give the same bits and the choice between
// them never shows in an output ("exact 4-slot concurrent serving", How it
// stays exact).
//
// Work split (GB300): persistent CTAs, three per SM, each owning a contiguous
// range of 4-row quads of W.  A CTA walks its rows in groups of 16 (4 quads).
// A stage is one kilobyte of K of a group: block c of stage j is block
// 32j + c, one block for each of the 32 chains.  One producer thread keeps a
// two-slot ring of stages in flight with tensor copies (W viewed as
// [N][K/256][256], one 4-row x 1 KB box per quad; the group's scales, the
// activation rows' 32 blocks and their scales as one box each), the arrival
// of a slot signalled on an mbarrier by the copies' byte count.  Four consumer
// warps read the slot from shared memory: lane (r = lane / 8, kb = lane % 8)
// of warp w runs chain c = kb + 8w of rows r, r + 4, r + 8 and r + 12 of the
// group, releases the slot once its operands are in registers, then does the
// dp4a work.  The copy engine fills boxes past the end of W or of the
// activations (rows >= N, blocks >= K/32) with zeros; the lanes that own such
// blocks skip them and rows past the CTA's range are never written.
//
// Why: the register-pipelined kernel keeps one stage of weights in flight per
// warp while it computes the other, and at 162 registers (12 warps per SM) that
// left ~30 % of the HBM stream idle at 4 rows; here the ring keeps copies in
// flight during the dp4a work and the consumers need ~125 registers.
//
// Every wait is bounded (about one second on the global timer); a wait that
// expires adds one to a device counter (luce_wait_timeouts) and the CTA stops
// consuming, leaving its remaining outputs unwritten.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace luce {

__device__ unsigned int g_wait_timeouts;

namespace {

constexpr int kRingG = 4;              // rows per lane (quads per group)
constexpr int kRingRows = 4 * kRingG;  // rows per group
constexpr int kRingSlots = 2;
constexpr int kRingCtasPerSm = 3;
constexpr int kRingThreads = 160;  // 4 consumer warps + 1 producer warp

template <int T>
struct RingLayout {
    static constexpr int W = kRingRows * 1024;  // [16 rows][1024 B]
    static constexpr int D = kRingRows * 64;    // [16 rows][32 fp16 scales]
    static constexpr int A = T * 1024;          // [T][1024 B]
    static constexpr int AD = T * 128;          // [T][32 fp32 scales]
    static constexpr int STAGE = W + D + A + AD;  // a multiple of 128
    static constexpr int PART = 2 * kRingRows * T * 33 * 4;
    static constexpr int SMEM = 128 + kRingSlots * STAGE + PART + 2 * kRingSlots * 8;
};

__device__ __forceinline__ uint32_t smem_addr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint64_t* b, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(b)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* b, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(b)), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* b)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(b)) : "memory");
}

__device__ __forceinline__ bool mbar_try(uint64_t* b, uint32_t parity)
{
    uint32_t done;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
        : "=r"(done)
        : "r"(smem_addr(b)), "r"(parity)
        : "memory");
    return done != 0;
}

__device__ __forceinline__ uint64_t global_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for the phase of parity `parity` to complete, for about a second at
// most; false (and one more timeout counted) if it did not.
__device__ __forceinline__ bool mbar_wait(uint64_t* b, uint32_t parity)
{
    if (mbar_try(b, parity)) return true;
    const uint64_t t0 = global_ns();
    while (!mbar_try(b, parity))
        if (global_ns() - t0 > 1000000000ull) {
            atomicAdd(&g_wait_timeouts, 1u);
            return false;
        }
    return true;
}

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* m, int x, int y, int z, uint64_t* bar)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
        "[%5];" ::"r"(smem_addr(dst)),
        "l"(m), "r"(x), "r"(y), "r"(z), "r"(smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* m, int x, int y, uint64_t* bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];" ::"r"(smem_addr(dst)),
        "l"(m), "r"(x), "r"(y), "r"(smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ uint4 lds128(const void* p)
{
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(smem_addr(p)));
    return v;
}

// Exact int32 dot of one block held as two 16-byte halves per side (x pairs
// with ax, y with ay), returned as a float: either one dp4a chain seeded with
// the bits of 1.5 * 2^23 and one exact subtraction, or two chains and a
// conversion.  Integer sums are exact in any order, so the value is the same
// as block_dot8's.
template <bool BIAS>
__device__ __forceinline__ float block_dot_halves(uint4 x, uint4 y, uint4 ax, uint4 ay)
{
    if (BIAS) {
        int s = __dp4a((int)x.x, (int)ax.x, 0x4B400000);
        s = __dp4a((int)x.y, (int)ax.y, s);
        s = __dp4a((int)x.z, (int)ax.z, s);
        s = __dp4a((int)x.w, (int)ax.w, s);
        s = __dp4a((int)y.x, (int)ay.x, s);
        s = __dp4a((int)y.y, (int)ay.y, s);
        s = __dp4a((int)y.z, (int)ay.z, s);
        s = __dp4a((int)y.w, (int)ay.w, s);
        return __fsub_rn(__int_as_float(s), 12582912.0f);
    } else {
        int s0 = __dp4a((int)x.x, (int)ax.x, 0), s1 = __dp4a((int)y.x, (int)ay.x, 0);
        s0 = __dp4a((int)x.y, (int)ax.y, s0);
        s1 = __dp4a((int)y.y, (int)ay.y, s1);
        s0 = __dp4a((int)x.z, (int)ax.z, s0);
        s1 = __dp4a((int)y.z, (int)ay.z, s1);
        s0 = __dp4a((int)x.w, (int)ax.w, s0);
        s1 = __dp4a((int)y.w, (int)ay.w, s1);
        return (float)(s0 + s1);
    }
}

}  // namespace

// mw: W as uint8 [N][K/256][256], box {256, 4, 4};  md: scales fp16 [N][K/32],
// box {32, 16};  ma: activations uint8 [T][K/256][256], box {256, 4, T};
// mad: activation scales fp32 [T][K/32], box {32, T}.
template <int T, bool BIAS>
__global__ void __launch_bounds__(kRingThreads)
q8_matvec_tma_kernel(const __grid_constant__ CUtensorMap mw, const __grid_constant__ CUtensorMap md,
                     const __grid_constant__ CUtensorMap ma, const __grid_constant__ CUtensorMap mad, int N, int K,
                     float* y, int64_t ldy, const float* resid, int64_t ldr)
{
    using L = RingLayout<T>;
    constexpr int G = kRingG, S = kRingSlots;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = smem_raw + ((128u - (smem_addr(smem_raw) & 127u)) & 127u);  // tensor copies land 128-aligned
    float* part = reinterpret_cast<float*>(sm + S * L::STAGE);
    uint64_t* full = reinterpret_cast<uint64_t*>(sm + S * L::STAGE + L::PART);
    uint64_t* empty = full + S;
    pdl_trigger();
    const int nb = K >> 5, nj = (nb + 31) >> 5;
    const int nq = (N + 3) >> 2;
    const int q0 = (int)((int64_t)blockIdx.x * nq / gridDim.x);
    const int q1 = (int)((int64_t)(blockIdx.x + 1) * nq / gridDim.x);
    const int ngrp = (q1 - q0 + G - 1) / G;
    const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);   // the producer's arrival + the copies' bytes
            mbar_init(&empty[s], 4);  // one arrival per consumer warp
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    if (w == 4) {
        // producer: stage it = (group it / nj, K-kilobyte it % nj) goes to slot it % S
        if (lane != 0) return;
        const int total = ngrp * nj;
        auto quads_of = [&](int it) { return min(G, q1 - (q0 + (it / nj) * G)); };
        auto bytes_of = [&](int it) { return (uint32_t)(quads_of(it) * 4096 + L::D + L::A + L::AD); };
        auto load_weights = [&](int it) {
            const int s = it % S, j = it % nj, qa = q0 + (it / nj) * G, nqv = quads_of(it);
            uint8_t* slot = sm + s * L::STAGE;
            for (int qq = 0; qq < nqv; ++qq) tma_load_3d(slot + qq * 4096, &mw, 0, 4 * j, 4 * (qa + qq), &full[s]);
            tma_load_2d(slot + L::W, &md, 32 * j, 4 * qa, &full[s]);
        };
        auto load_acts = [&](int it) {
            const int s = it % S, j = it % nj;
            uint8_t* slot = sm + s * L::STAGE;
            tma_load_3d(slot + L::W + L::D, &ma, 0, 4 * j, 0, &full[s]);
            tma_load_2d(slot + L::W + L::D + L::A, &mad, 32 * j, 0, &full[s]);
        };
        const int pre = min(S, total);
        for (int it = 0; it < pre; ++it) {  // weights do not depend on the previous kernel
            mbar_expect_tx(&full[it], bytes_of(it));
            load_weights(it);
        }
        pdl_wait();  // the activations do
        for (int it = 0; it < pre; ++it) load_acts(it);
        for (int it = pre; it < total; ++it) {
            const int s = it % S;
            if (!mbar_wait(&empty[s], ((it / S) - 1) & 1)) break;
            mbar_expect_tx(&full[s], bytes_of(it));
            load_weights(it);
            load_acts(it);
        }
        return;
    }

    pdl_wait();  // the residual and y may be touched by earlier kernels
    const int r = lane >> 3, kb = lane & 7, c = kb + 8 * w;
    const int h0 = (kb >> 2) & 1;  // which 16-byte half first: 8 lanes of a phase hit 8 distinct bank quads
    bool bad = false;
    int it = 0;
    for (int gi = 0; gi < ngrp; ++gi) {
        const int gr0 = 4 * (q0 + gi * G), gr1 = min(4 * q1, N);
        float acc[G][T];
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
            for (int t = 0; t < T; ++t) acc[g][t] = 0.0f;
        for (int j = 0; j < nj; ++j, ++it) {
            const int s = it % S;
            if (!bad && !mbar_wait(&full[s], (it / S) & 1)) bad = true;
            if (bad) continue;
            const uint8_t* slot = sm + s * L::STAGE;
            const bool has = 32 * j + c < nb;
            uint4 wx[G], wy[G], ax[T], ay[T];
            float sw[G], sa[T];
            if (has) {
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    const uint8_t* p = slot + (r + 4 * g) * 1024 + c * 32;
                    wx[g] = lds128(p + 16 * h0);
                    wy[g] = lds128(p + 16 * (h0 ^ 1));
                    sw[g] = __half2float(*reinterpret_cast<const __half*>(slot + L::W + (r + 4 * g) * 64 + c * 2));
                }
#pragma unroll
                for (int t = 0; t < T; ++t) {
                    const uint8_t* p = slot + L::W + L::D + t * 1024 + c * 32;
                    ax[t] = lds128(p + 16 * h0);
                    ay[t] = lds128(p + 16 * (h0 ^ 1));
                    sa[t] = *reinterpret_cast<const float*>(slot + L::W + L::D + L::A + t * 128 + c * 4);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);  // operands are in registers: the slot may refill
            if (has) {
#pragma unroll
                for (int t = 0; t < T; ++t)
#pragma unroll
                    for (int g = 0; g < G; ++g) {
                        const float sd = block_dot_halves<BIAS>(wx[g], wy[g], ax[t], ay[t]);
                        acc[g][t] = __fmaf_rn(__fmul_rn(sw[g], sa[t]), sd, acc[g][t]);
                    }
            }
        }
        // the 32 chains of each (row, token) meet in shared memory; two
        // buffers, so one barrier per group separates writers and readers
        float* pp = part + (gi & 1) * (kRingRows * T * 33);
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
            for (int t = 0; t < T; ++t) pp[((r + 4 * g) * T + t) * 33 + c] = acc[g][t];
        asm volatile("bar.sync 1, 128;" ::: "memory");
        for (int idx = tid; idx < kRingRows * T; idx += 128) {
            const int rr = idx / T, t = idx - (idx / T) * T;
            const int n = gr0 + rr;
            if (n < gr1 && !bad) {
                float out = q8_butterfly(pp + (rr * T + t) * 33);
                if (resid) out = __fadd_rn(resid[(size_t)t * ldr + n], out);
                y[(size_t)t * ldy + n] = out;
            }
        }
    }
}

namespace {

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder()
{
    static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return (PFN_cuTensorMapEncodeTiled_v12000) nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }();
    return fn;
}

// A tiled tensor map of `rank` dims (dims[0] innermost, strides in bytes for
// dims 1..rank-1), no swizzle, zero fill outside the tensor.
bool encode_map(CUtensorMap* m, CUtensorMapDataType dt, int rank, const void* base, const cuuint64_t* dims,
                const cuuint64_t* strides, const cuuint32_t* box)
{
    const PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint32_t es[3] = {1, 1, 1};
    return enc(m, dt, (cuuint32_t)rank, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count()
{
    static int counts[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (counts[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        counts[dev] = n;
    }
    return counts[dev];
}

template <int T, bool BIAS>
cudaError_t launch_tma_t(const CUtensorMap& mw, const CUtensorMap& md, const CUtensorMap& ma, const CUtensorMap& mad,
                         int N, int K, float* y, int64_t ldy, const float* resid, int64_t ldr, int sms,
                         cudaStream_t s)
{
    using L = RingLayout<T>;
    static std::once_flag once;
    static cudaError_t attr = cudaSuccess;
    std::call_once(once, [] {
        attr = cudaFuncSetAttribute(q8_matvec_tma_kernel<T, BIAS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    L::SMEM);
    });
    if (attr != cudaSuccess) return attr;
    const int nq = (N + 3) / 4;
    const int grid = min(kRingCtasPerSm * sms, (nq + kRingG - 1) / kRingG);
    const cudaError_t e = launch_pdl_smem(q8_matvec_tma_kernel<T, BIAS>, dim3(grid), dim3(kRingThreads), L::SMEM, s,
                                          mw, md, ma, mad, N, K, y, ldy, resid, ldr);
    count_launches(1);
    return e;
}

}  // namespace

cudaError_t launch_matvec_tma(const int8_t* wq, const __half* wd, int N, int K, const int8_t* aq, const float* ad,
                              int T, float* y, int64_t ldy, const float* resid, int64_t ldr, cudaStream_t s)
{
    auto al16 = [](const void* p) { return ((uintptr_t)p & 15) == 0; };
    if (T < 1 || T > 4 || K % 256 != 0 || !al16(wq) || !al16(wd) || !al16(aq) || !al16(ad))
        return cudaErrorNotSupported;
    const int sms = sm_count();
    if (sms <= 0) return cudaErrorNotSupported;
    const cuuint64_t nb = (cuuint64_t)K / 32;
    const cuuint64_t wdim[3] = {256, (cuuint64_t)K / 256, (cuuint64_t)N}, wstr[2] = {256, (cuuint64_t)K};
    const cuuint32_t wbox[3] = {256, 4, 4};
    const cuuint64_t ddim[2] = {nb, (cuuint64_t)N}, dstr[1] = {nb * 2};
    const cuuint32_t dbox[2] = {32, (cuuint32_t)kRingRows};
    const cuuint64_t adim[3] = {256, (cuuint64_t)K / 256, (cuuint64_t)T}, astr[2] = {256, (cuuint64_t)K};
    const cuuint32_t abox[3] = {256, 4, (cuuint32_t)T};
    const cuuint64_t addim[2] = {nb, (cuuint64_t)T}, adstr[1] = {nb * 4};
    const cuuint32_t adbox[2] = {32, (cuuint32_t)T};
    CUtensorMap mw, md, ma, mad;
    if (!encode_map(&mw, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, wq, wdim, wstr, wbox) ||
        !encode_map(&md, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, wd, ddim, dstr, dbox) ||
        !encode_map(&ma, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, aq, adim, astr, abox) ||
        !encode_map(&mad, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, ad, addim, adstr, adbox))
        return cudaErrorNotSupported;
    switch (T) {
        case 1: return launch_tma_t<1, true>(mw, md, ma, mad, N, K, y, ldy, resid, ldr, sms, s);
        case 2: return launch_tma_t<2, false>(mw, md, ma, mad, N, K, y, ldy, resid, ldr, sms, s);
        case 3: return launch_tma_t<3, false>(mw, md, ma, mad, N, K, y, ldy, resid, ldr, sms, s);
        default: return launch_tma_t<4, false>(mw, md, ma, mad, N, K, y, ldy, resid, ldr, sms, s);
    }
}

cudaError_t read_wait_timeouts(uint32_t* count, bool reset)
{
    cudaError_t e = cudaMemcpyFromSymbol(count, g_wait_timeouts, sizeof(uint32_t));
    if (e == cudaSuccess && reset) {
        const uint32_t zero = 0;
        e = cudaMemcpyToSymbol(g_wait_timeouts, &zero, sizeof(uint32_t));
    }
    return e;
}

}  // namespace luce
