// matvec_tma.cu - the q8_0 matvec for 1..8 activation rows (13..16 in two
// launches), with the weights streamed through shared memory by the tensor
// memory accelerator (TMA); also the fused q|k|v + RoPE + K/V-append form.
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
// range of 4-row quads of W.  A CTA walks its rows in groups of G quads (4G
// rows; G = 4 up to 4 activation rows, 2 for 5..8).  A stage is one kilobyte
// of K of a group: block c of stage j is block 32j + c, one block for each of
// the 32 chains.  One producer thread keeps a ring of three stages in flight
// with tensor copies (W viewed as [N][K/256][256], one
// 4-row x 1 KB box per quad; the group's scales, the activation rows' 32
// blocks and their scales as one box each), the arrival of a slot signalled on
// an mbarrier by the copies' byte count.  Four consumer warps read the slot
// from shared memory: lane (r = lane / 8, kb = lane % 8) of warp w runs chain
// c = kb + 8w of rows r, r + 4, ..., r + 4(G-1) of the group, releases the slot
// once its operands are in registers, then does the dp4a work.  The copy
// engine fills boxes past the end of W or of the activations (rows >= N,
// blocks >= K/32) with zeros; the lanes that own such blocks skip them and
// rows past the CTA's range are never written.
//
// Why: the register-pipelined kernel keeps one stage of weights in flight per
// warp while it computes the other, and at 162 registers (12 warps per SM) that
// left ~30 % of the HBM stream idle at 4 rows; here the ring keeps copies in
// flight during the dp4a work and the consumers need ~125 registers.
//
// Every wait is bounded (about one second on the global timer, 2^26 polls);
// a wait that expires adds one to a device counter (luce_wait_timeouts) and
// the CTA stops consuming, leaving its remaining outputs unwritten; the
// producer drains its last stages' copies (ring_drain, bounded) before it
// returns.
#include <string.h>

#include <atomic>
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "ring.cuh"

namespace luce {

__device__ unsigned int g_wait_timeouts;

namespace {

constexpr int kRingCtasPerSm = 3;      // 1..4 rows
constexpr int kRingCtasPerSmWide = 3;  // 5..8 rows (larger activation boxes)
constexpr int kRingSlotsWide = 3;
constexpr int kRingSlotsNarrow = 3;    // 1..4 rows
constexpr int kRingThreads = 160;  // 4 consumer warps + 1 producer warp
// Consumer warps of the fused gate||up kernel at T rows (two CTAs per SM):
// 8 at one row, where more warps hide more latency, 4 from two rows on, where
// each lane's 4 rows give the dp4a chains more independent work (measured).
__host__ __device__ constexpr int gateup_warps(int T) { return T == 1 ? 8 : 4; }

// Shape of a ring: T activation rows, G rows per lane (a group is G quads,
// 4G rows), S slots.
template <int T, int G, int S>
struct RingLayout {
    static constexpr int ROWS = 4 * G;
    static constexpr int W = ROWS * 1024;  // [4G rows][1024 B]
    static constexpr int D = ROWS * 64;    // [4G rows][32 fp16 scales]
    static constexpr int A = T * 1024;          // [T][1024 B]
    static constexpr int AD = T * 128;          // [T][32 fp32 scales]
    static constexpr int STAGE = W + D + A + AD;  // a multiple of 128
    // chain buffers: two (one barrier per group) unless three CTAs per SM
    // would then not fit in the SM's 228 KB, then one (two barriers per group)
    static constexpr int PART1 = ROWS * T * 33 * 4;
    static constexpr int PB = 3 * (128 + S * STAGE + 2 * PART1 + 2 * S * 8 + 1024) <= 233472 ? 2 : 1;
    static constexpr int PART = PB * PART1;
    static constexpr int SMEM = 128 + S * STAGE + PART + 2 * S * 8;
};

// Exercises the expiry path: one thread waits, for limit_ns, on a barrier
// that expects one arrival nobody makes (no copy is issued), so the wait
// runs out, is counted, and the kernel returns normally.
__global__ void wait_expiry_kernel(uint64_t limit_ns)
{
    __shared__ uint64_t bar;
    if (threadIdx.x != 0) return;
    mbar_init(&bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    mbar_wait(&bar, 0, &g_wait_timeouts, limit_ns);
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

namespace {

// Shared-memory carve-up of a ring CTA: 128-aligned slots, the chain values,
// the slot barriers.
template <int T, int G, int S>
struct RingSmem {
    uint8_t* slots;
    float* part;
    uint64_t* full;   // slot filled: the producer's arrival + the copies' bytes
    uint64_t* empty;  // slot released: one arrival per consumer warp
    __device__ explicit RingSmem(uint8_t* raw)
    {
        using L = RingLayout<T, G, S>;
        slots = raw + ((128u - (smem_addr(raw) & 127u)) & 127u);  // tensor copies land 128-aligned
        part = reinterpret_cast<float*>(slots + S * L::STAGE);
        full = reinterpret_cast<uint64_t*>(slots + S * L::STAGE + L::PART);
        empty = full + S;
    }
    __device__ void init(int consumer_warps = 4) const
    {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], consumer_warps);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
};

// The producer thread: stage it (group it / nj, K-kilobyte it % nj) of
// `total` goes to slot it % S.  load_weights(it, slot, bar) issues the
// group's weight and scale boxes, weight_bytes(it) counts them; the
// activation boxes of the kilobyte follow.  The first S stages' weights go
// before the wait on the previous kernel, which the activations need.
template <int T, int G, int S, typename LoadW, typename BytesW>
__device__ __forceinline__ void ring_produce(const RingSmem<T, G, S>& R, int total, int nj, const CUtensorMap* ma,
                                             const CUtensorMap* mad, LoadW load_weights, BytesW weight_bytes)
{
    using L = RingLayout<T, G, S>;
    auto load_acts = [&](int it) {
        uint8_t* slot = R.slots + (it % S) * L::STAGE;
        const int j = it % nj;
        tma_load_3d(slot + L::W + L::D, ma, 0, 4 * j, 0, &R.full[it % S]);
        tma_load_2d(slot + L::W + L::D + L::A, mad, 32 * j, 0, &R.full[it % S]);
    };
    const int pre = min(S, total);
    for (int it = 0; it < pre; ++it) {
        mbar_expect_tx(&R.full[it], (uint32_t)(weight_bytes(it) + L::A + L::AD));
        load_weights(it, R.slots + it * L::STAGE, &R.full[it]);
    }
    pdl_wait();
    for (int it = 0; it < pre; ++it) load_acts(it);
    int issued = pre;
    for (; issued < total; ++issued) {
        const int it = issued, s = it % S;
        if (!mbar_wait(&R.empty[s], ((it / S) - 1) & 1, &g_wait_timeouts)) break;
        mbar_expect_tx(&R.full[s], (uint32_t)(weight_bytes(it) + L::A + L::AD));
        load_weights(it, R.slots + s * L::STAGE, &R.full[s]);
        load_acts(it);
    }
    ring_drain<S>(R.full, issued, &g_wait_timeouts);
}

// A consumer lane's chains for one group: stages it .. it + nj - 1 (it
// advances), lane (r, kb) of warp w, chain c = kb + 8w, rows r + 4g of the
// group, g < GL (GL = G: all the group's rows; fewer when several warps share
// the chains, r then carrying the row offset of this warp's share).
// acc[g][t] = chain c of row r + 4g against token t.  ok turns false when a
// wait expires; from then on the lane waits for nothing more and the caller
// writes nothing.
template <int T, int G, int S, bool BIAS, int GL = G>
__device__ __forceinline__ void ring_chains(const RingSmem<T, G, S>& R, int& it, int nj, int nb, int r, int c, int lane,
                                            float (&acc)[GL][T], bool& ok)
{
    using L = RingLayout<T, G, S>;
    const int h0 = ((lane & 7) >> 2) & 1;  // which 16-byte half first: a phase's 8 lanes hit 8 distinct bank quads
#pragma unroll
    for (int g = 0; g < GL; ++g)
#pragma unroll
        for (int t = 0; t < T; ++t) acc[g][t] = 0.0f;
    for (int j = 0; j < nj; ++j, ++it) {
        const int s = it % S;
        if (ok && !mbar_wait(&R.full[s], (it / S) & 1, &g_wait_timeouts)) ok = false;
        if (!ok) continue;
        const uint8_t* slot = R.slots + s * L::STAGE;
        const bool has = 32 * j + c < nb;
        uint4 wx[GL], wy[GL], ax[T], ay[T];
        float sw[GL], sa[T];
        if (has) {
#pragma unroll
            for (int g = 0; g < GL; ++g) {
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
        if (lane == 0) mbar_arrive(&R.empty[s]);  // operands are in registers: the slot may refill
        if (has) {
#pragma unroll
            for (int t = 0; t < T; ++t)
#pragma unroll
                for (int g = 0; g < GL; ++g) {
                    const float sd = block_dot_halves<BIAS>(wx[g], wy[g], ax[t], ay[t]);
                    acc[g][t] = __fmaf_rn(__fmul_rn(sw[g], sa[t]), sd, acc[g][t]);
                }
        }
    }
}

// Chain values of local row rr = r + 4g, token t, chain c into a [4G][T][33] buffer.
template <int T, int G>
__device__ __forceinline__ void store_chains(float* pp, int r, int c, const float (&acc)[G][T])
{
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
        for (int t = 0; t < T; ++t) pp[((r + 4 * g) * T + t) * 33 + c] = acc[g][t];
}

}  // namespace

// mw: W as uint8 [N][K/256][256], box {256, 4, 4};  md: scales fp16 [N][K/32],
// box {32, 16};  ma: activations uint8 [T][K/256][256], box {256, 4, T};
// mad: activation scales fp32 [T][K/32], box {32, T}.  Persistent: CTA b owns
// quads [b*nq/grid, (b+1)*nq/grid) of the nq = ceil(N/4) quads, in groups of G
// (md's box is 4G rows).
template <int T, int G, int S, bool BIAS>
__global__ void __launch_bounds__(kRingThreads)
q8_matvec_tma_kernel(const __grid_constant__ CUtensorMap mw, const __grid_constant__ CUtensorMap md,
                     const __grid_constant__ CUtensorMap ma, const __grid_constant__ CUtensorMap mad, int N, int K,
                     float* y, int64_t ldy, const float* resid, int64_t ldr)
{
    using L = RingLayout<T, G, S>;
    extern __shared__ uint8_t smem_raw[];
    const RingSmem<T, G, S> R(smem_raw);
    pdl_trigger();
    const int nb = K >> 5, nj = (nb + 31) >> 5;
    const int nq = (N + 3) >> 2;
    const int q0 = (int)((int64_t)blockIdx.x * nq / gridDim.x);
    const int q1 = (int)((int64_t)(blockIdx.x + 1) * nq / gridDim.x);
    const int ngrp = (q1 - q0 + G - 1) / G;
    const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
    if (tid == 0) R.init();
    __syncthreads();

    if (w == 4) {
        if (lane != 0) return;
        auto quads = [&](int it) { return min(G, q1 - (q0 + (it / nj) * G)); };
        ring_produce<T, G, S>(
            R, ngrp * nj, nj, &ma, &mad,
            [&](int it, uint8_t* slot, uint64_t* bar) {
                const int j = it % nj, qa = q0 + (it / nj) * G, nqv = quads(it);
                for (int qq = 0; qq < nqv; ++qq) tma_load_3d(slot + qq * 4096, &mw, 0, 4 * j, 4 * (qa + qq), bar);
                tma_load_2d(slot + L::W, &md, 32 * j, 4 * qa, bar);
            },
            [&](int it) { return quads(it) * 4096 + L::D; });
        return;
    }

    pdl_wait();  // the residual and y may be touched by earlier kernels
    const int r = lane >> 3, c = (lane & 7) + 8 * w;
    bool ok = true;
    int it = 0;
    for (int gi = 0; gi < ngrp; ++gi) {
        const int gr0 = 4 * (q0 + gi * G), gr1 = min(4 * q1, N);
        float acc[G][T];
        ring_chains<T, G, S, BIAS>(R, it, nj, nb, r, c, lane, acc, ok);
        // two chain buffers, so one barrier per group separates writers and readers
        float* pp = R.part + (L::PB == 2 ? (gi & 1) * (L::ROWS * T * 33) : 0);
        if (L::PB == 1 && gi > 0) asm volatile("bar.sync 1, 128;" ::: "memory");  // last group's readers are done
        store_chains<T, G>(pp, r, c, acc);
        asm volatile("bar.sync 1, 128;" ::: "memory");
        for (int idx = tid; idx < L::ROWS * T; idx += 128) {
            const int rr = idx / T, t = idx - (idx / T) * T;
            const int n = gr0 + rr;
            if (n < gr1 && ok) {
                float out = q8_butterfly(pp + (rr * T + t) * 33);
                if (resid) out = __fadd_rn(resid[(size_t)t * ldr + n], out);
                y[(size_t)t * ldy + n] = out;
            }
        }
    }
}

// The decode step's q|k|v projection with the RoPE rotation and the K/V
// append in the epilogue ("antirez/ds4 pull 604", Commit walkthrough): the
// same chains, one group per CTA, the group being the P = 2G rotation pairs
// (i, i + 64) for i in [q0, q0 + P) of head h = b / (64/P), q0 = P (b % (64/P)).
// Quads [0, G/2) are rows h*128 + q0 + [0, P), quads [G/2, G) rows
// h*128 + 64 + q0 + [0, P); mdp is the scale map with a P-row box.  Thread
// idx < P*T finishes pair p = idx / T of token t = idx % T exactly as
// q8_qkv_rope_kernel does.
template <int T, int G, int S, bool BIAS>
__global__ void __launch_bounds__(kRingThreads)
q8_qkv_rope_tma_kernel(const __grid_constant__ CUtensorMap mw, const __grid_constant__ CUtensorMap mdp,
                       const __grid_constant__ CUtensorMap ma, const __grid_constant__ CUtensorMap mad, int K,
                       float* __restrict__ qkv, int Hq, int Hkv, const __grid_constant__ RowPos pos,
                       const __grid_constant__ RopeFreq f, float* __restrict__ q_rot, const __grid_constant__ KvRows kv)
{
    constexpr int P = 2 * G, GROUPS = (kHeadDim / 2) / P;
    using L = RingLayout<T, G, S>;
    static_assert(P * T <= 128, "one (pair, token) per consumer thread");
    extern __shared__ uint8_t smem_raw[];
    const RingSmem<T, G, S> R(smem_raw);
    pdl_trigger();
    const int nb = K >> 5, nj = (nb + 31) >> 5;
    const int h = blockIdx.x / GROUPS, q0 = (blockIdx.x % GROUPS) * P;
    const int row0 = h * kHeadDim + q0, row1 = h * kHeadDim + kHeadDim / 2 + q0;
    const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
    if (tid == 0) R.init();
    __syncthreads();

    if (w == 4) {
        if (lane != 0) return;
        ring_produce<T, G, S>(
            R, nj, nj, &ma, &mad,
            [&](int it, uint8_t* slot, uint64_t* bar) {
                const int j = it % nj;
#pragma unroll
                for (int qq = 0; qq < G; ++qq)
                    tma_load_3d(slot + qq * 4096, &mw, 0, 4 * j,
                                (qq < G / 2 ? row0 + 4 * qq : row1 + 4 * (qq - G / 2)), bar);
                tma_load_2d(slot + L::W, &mdp, 32 * j, row0, bar);
                tma_load_2d(slot + L::W + P * 64, &mdp, 32 * j, row1, bar);
            },
            [&](int) { return G * 4096 + L::D; });
        return;
    }

    // thread idx < P*T finishes pair p = idx / T of token t = idx % T; its
    // cos/sin depend only on the position, so they are formed first
    const int p = tid / T, t = tid - (tid / T) * T;
    const int i = q0 + p;
    const bool fin = tid < P * T;
    const float2 cs = (fin && h < Hq + Hkv) ? rope_cs(pos.pos[t], f.inv[i]) : make_float2(1.0f, 0.0f);
    pdl_wait();  // the K/V caches and outputs may be touched by earlier kernels
    const int r = lane >> 3, c = (lane & 7) + 8 * w;
    int it = 0;
    float acc[G][T];
    bool ok = true;
    ring_chains<T, G, S, BIAS>(R, it, nj, nb, r, c, lane, acc, ok);
    store_chains<T, G>(R.part, r, c, acc);
    asm volatile("bar.sync 1, 128;" ::: "memory");
    if (fin && ok) {
        float x0 = q8_butterfly(R.part + (p * T + t) * 33);
        float x1 = q8_butterfly(R.part + ((p + P) * T + t) * 33);
        const int ldq = (Hq + 2 * Hkv) * kHeadDim;
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

// The decode step's gate||up projection (gate rows [0, F), up rows [F, 2F)
// of W) with SwiGLU and its q8_0 quantization in the epilogue, 1..4
// activation rows: the same chains.  A unit is the 32 features f0 .. f0 + 31
// (f0 = 32u) and its four groups hold gate rows f0 + 8i .. f0 + 8i + 7
// (quads 0, 1) and the up rows F + the same features (quads 2, 3), i = 0..3,
// so the CTA that finishes a feature holds its gate and its up value: it
// stores both to gu as the plain projection would, h = silu(g) * u, and once
// the unit's 32 features are in, warp t quantizes token t's block of h -
// exactly swiglu_quant_kernel's arithmetic.  Persistent: CTA b owns units
// [b*U/grid, (b+1)*U/grid) of the U = F/32; mdp has an 8-row scale box.
// Shared memory allows two CTAs per SM; at one row a CTA has 8 consumer
// warps (the gate and the up rows of a group in two sets of 4, each lane 2
// rows), else 4 (each lane 4 rows: 2 gate, 2 up).
template <int T, int S, bool BIAS>
__global__ void __launch_bounds__(32 * (gateup_warps(T) + 1), 2)
q8_gateup_swiglu_tma_kernel(const __grid_constant__ CUtensorMap mw, const __grid_constant__ CUtensorMap mdp,
                            const __grid_constant__ CUtensorMap ma, const __grid_constant__ CUtensorMap mad, int F,
                            int K, float* __restrict__ gu, float* __restrict__ h, int8_t* __restrict__ hq,
                            float* __restrict__ hd)
{
    constexpr int G = 4;
    using L = RingLayout<T, G, S>;
    extern __shared__ uint8_t smem_raw[];
    const RingSmem<T, G, S> R(smem_raw);
    __shared__ float hb[T][32];  // the unit's h values, token by token
    pdl_trigger();
    const int nb = K >> 5, nj = (nb + 31) >> 5;
    const int U = F >> 5;
    const int u0 = (int)((int64_t)blockIdx.x * U / gridDim.x);
    const int u1 = (int)((int64_t)(blockIdx.x + 1) * U / gridDim.x);
    const int ngrp = 4 * (u1 - u0);
    constexpr int CW = gateup_warps(T), GL = 16 / CW;  // consumer warps, rows per lane
    const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
    if (tid == 0) R.init(CW);
    __syncthreads();

    if (w == CW) {
        if (lane != 0) return;
        ring_produce<T, G, S>(
            R, ngrp * nj, nj, &ma, &mad,
            [&](int it, uint8_t* slot, uint64_t* bar) {
                const int j = it % nj, gi = it / nj;
                const int f = 32 * (u0 + gi / 4) + 8 * (gi % 4);
                tma_load_3d(slot, &mw, 0, 4 * j, f, bar);
                tma_load_3d(slot + 4096, &mw, 0, 4 * j, f + 4, bar);
                tma_load_3d(slot + 2 * 4096, &mw, 0, 4 * j, F + f, bar);
                tma_load_3d(slot + 3 * 4096, &mw, 0, 4 * j, F + f + 4, bar);
                tma_load_2d(slot + L::W, &mdp, 32 * j, f, bar);
                tma_load_2d(slot + L::W + 8 * 64, &mdp, 32 * j, F + f, bar);
            },
            [&](int) { return G * 4096 + L::D; });
        return;
    }

    pdl_wait();  // gu, h and the codes may be touched by earlier kernels
    // with 8 consumer warps, warps 0-3 take the gate rows 0-7 of a group and
    // warps 4-7 the up rows 8-15; lane (r, kb) of warp w runs chain
    // c = kb + 8 (w % 4) of rows r + 8 (w / 4) + 4g, g < GL
    const int r = (lane >> 3) + 8 * (w >> 2), c = (lane & 7) + 8 * (w & 3);
    bool ok = true;
    int it = 0;
    for (int gi = 0; gi < ngrp; ++gi) {
        float acc[GL][T];
        ring_chains<T, G, S, BIAS, GL>(R, it, nj, nb, r, c, lane, acc, ok);
        // two chain buffers, so one barrier per group separates writers and readers
        float* pp = R.part + (L::PB == 2 ? (gi & 1) * (L::ROWS * T * 33) : 0);
        if (L::PB == 1 && gi > 0) asm volatile("bar.sync 1, %0;" ::"n"(32 * CW) : "memory");  // readers are done
        store_chains<T, GL>(pp, r, c, acc);
        asm volatile("bar.sync 1, %0;" ::"n"(32 * CW) : "memory");
        const int fu = 32 * (u0 + gi / 4), i = gi % 4;
        if (tid < 8 * T && ok) {  // feature fu + 8i + p of token t: local rows p (gate) and 8 + p (up)
            const int p = tid / T, t = tid - (tid / T) * T;
            const float g = q8_butterfly(pp + (p * T + t) * 33);
            const float u = q8_butterfly(pp + ((8 + p) * T + t) * 33);
            gu[(size_t)t * 2 * F + fu + 8 * i + p] = g;
            gu[(size_t)t * 2 * F + F + fu + 8 * i + p] = u;
            hb[t][8 * i + p] = silu_mul(g, u);
        }
        if (i == 3) {  // the unit's 32 features are in: warp t quantizes token t's block
            asm volatile("bar.sync 1, %0;" ::"n"(32 * CW) : "memory");
            if (w < T && ok) {
                const float v = hb[w][lane];
                h[(size_t)w * F + fu + lane] = v;
                const int code = q8_quantize_store<false>(v, hd, (size_t)w * U + (fu >> 5), lane == 0);
                hq[(size_t)w * F + fu + lane] = (int8_t)code;
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

// The inputs of one tiled tensor map; a map is a pure function of them, so
// maps are kept in a small table and encoded once per distinct key (the
// step's weights and workspace give the same keys every call).
struct MapKey {
    uint64_t base, dims[3], strides[2];
    uint32_t box[3], dt, rank, swizzle;
    bool operator==(const MapKey& o) const { return memcmp(this, &o, sizeof(MapKey)) == 0; }
};

struct MapCache {
    static constexpr int kSlots = 512;
    std::mutex mu;
    MapKey key[kSlots];
    CUtensorMap map[kSlots];
    bool used[kSlots] = {};
};

MapCache& map_cache()
{
    static MapCache c;
    return c;
}

}  // namespace

bool encode_map(CUtensorMap* m, CUtensorMapDataType dt, int rank, const void* base, const cuuint64_t* dims,
                const cuuint64_t* strides, const cuuint32_t* box, CUtensorMapSwizzle swizzle)
{
    MapKey k;
    memset(&k, 0, sizeof k);
    k.base = (uint64_t)(uintptr_t)base;
    k.dt = (uint32_t)dt;
    k.rank = (uint32_t)rank;
    k.swizzle = (uint32_t)swizzle;
    for (int i = 0; i < rank; ++i) {
        k.dims[i] = dims[i];
        k.box[i] = box[i];
        if (i + 1 < rank) k.strides[i] = strides[i];
    }
    uint64_t h = 1469598103934665603ull;  // FNV-1a over the key's bytes
    for (size_t i = 0; i < sizeof k; ++i) h = (h ^ reinterpret_cast<const uint8_t*>(&k)[i]) * 1099511628211ull;
    MapCache& c = map_cache();
    const int slot = (int)(h % MapCache::kSlots);
    {
        std::lock_guard<std::mutex> lock(c.mu);
        if (c.used[slot] && c.key[slot] == k) {
            *m = c.map[slot];
            return true;
        }
    }
    const PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint32_t es[3] = {1, 1, 1};
    if (enc(m, dt, (cuuint32_t)rank, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
    std::lock_guard<std::mutex> lock(c.mu);
    c.key[slot] = k;
    c.map[slot] = *m;
    c.used[slot] = true;
    return true;
}

int current_device()
{
    int dev = 0;
    return (cudaGetDevice(&dev) == cudaSuccess && dev >= 0 && dev < kMaxDevices) ? dev : -1;
}

int sm_count()
{
    static std::atomic<int> counts[kMaxDevices];
    const int dev = current_device();
    if (dev < 0) return 0;
    int n = counts[dev].load(std::memory_order_relaxed);
    if (n == 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        counts[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

namespace {

template <int T, int G, int S, bool BIAS>
cudaError_t launch_tma_t(const CUtensorMap& mw, const CUtensorMap& md, const CUtensorMap& ma, const CUtensorMap& mad,
                         int N, int K, float* y, int64_t ldy, const float* resid, int64_t ldr, int ctas,
                         cudaStream_t s)
{
    using L = RingLayout<T, G, S>;
    static std::atomic<bool> done[kMaxDevices];
    const cudaError_t attr = set_smem_once(q8_matvec_tma_kernel<T, G, S, BIAS>, L::SMEM, done);
    if (attr != cudaSuccess) return attr;
    const int nq = (N + 3) / 4;
    const int grid = min(ctas, (nq + G - 1) / G);
    const cudaError_t e = launch_pdl_smem(q8_matvec_tma_kernel<T, G, S, BIAS>, dim3(grid), dim3(kRingThreads), L::SMEM,
                                          s, mw, md, ma, mad, N, K, y, ldy, resid, ldr);
    count_launches(1);
    return e;
}

template <int T, int G, int S, bool BIAS>
cudaError_t launch_qkv_tma_t(const CUtensorMap& mw, const CUtensorMap& mdp, const CUtensorMap& ma,
                             const CUtensorMap& mad, int K, float* qkv, int Hq, int Hkv, const RowPos& pos,
                             const RopeFreq& f, float* q_rot, const KvRows& kv, cudaStream_t s)
{
    using L = RingLayout<T, G, S>;
    static std::atomic<bool> done[kMaxDevices];
    const cudaError_t attr = set_smem_once(q8_qkv_rope_tma_kernel<T, G, S, BIAS>, L::SMEM, done);
    if (attr != cudaSuccess) return attr;
    const int groups = (Hq + 2 * Hkv) * ((kHeadDim / 2) / (2 * G));
    const cudaError_t e = launch_pdl_smem(q8_qkv_rope_tma_kernel<T, G, S, BIAS>, dim3(groups), dim3(kRingThreads),
                                          L::SMEM, s, mw, mdp, ma, mad, K, qkv, Hq, Hkv, pos, f, q_rot, kv);
    count_launches(1);
    return e;
}

// The four maps of a ring launch; false when the shapes or alignments do not
// allow one (the caller then takes the register-pipelined kernels).
bool ring_maps(const int8_t* wq, const __half* wd, int N, int K, const int8_t* aq, const float* ad, int T,
               int scale_box_rows, CUtensorMap* mw, CUtensorMap* md, CUtensorMap* ma, CUtensorMap* mad)
{
    auto al16 = [](const void* p) { return ((uintptr_t)p & 15) == 0; };
    if (T < 1 || T > 8 || K % 256 != 0 || !al16(wq) || !al16(wd) || !al16(aq) || !al16(ad)) return false;
    const cuuint64_t nb = (cuuint64_t)K / 32;
    const cuuint64_t wdim[3] = {256, (cuuint64_t)K / 256, (cuuint64_t)N}, wstr[2] = {256, (cuuint64_t)K};
    const cuuint32_t wbox[3] = {256, 4, 4};
    const cuuint64_t ddim[2] = {nb, (cuuint64_t)N}, dstr[1] = {nb * 2};
    const cuuint32_t dbox[2] = {32, (cuuint32_t)scale_box_rows};
    const cuuint64_t adim[3] = {256, (cuuint64_t)K / 256, (cuuint64_t)T}, astr[2] = {256, (cuuint64_t)K};
    const cuuint32_t abox[3] = {256, 4, (cuuint32_t)T};
    const cuuint64_t addim[2] = {nb, (cuuint64_t)T}, adstr[1] = {nb * 4};
    const cuuint32_t adbox[2] = {32, (cuuint32_t)T};
    return encode_map(mw, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, wq, wdim, wstr, wbox) &&
           encode_map(md, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, wd, ddim, dstr, dbox) &&
           encode_map(ma, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, aq, adim, astr, abox) &&
           encode_map(mad, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, ad, addim, adstr, adbox);
}

}  // namespace

// One ring launch of T <= 8 rows, three slots: groups of 16 rows up to 4
// rows, groups of 8 rows for 5..8 (shared memory for the larger activation
// boxes).
static cudaError_t launch_ring_rows(const int8_t* wq, const __half* wd, int N, int K, const int8_t* aq,
                                    const float* ad, int T, float* y, int64_t ldy, const float* resid, int64_t ldr,
                                    int sms, cudaStream_t s)
{
    CUtensorMap mw, md, ma, mad;
    if (!ring_maps(wq, wd, N, K, aq, ad, T, T <= 4 ? 16 : 8, &mw, &md, &ma, &mad)) return cudaErrorNotSupported;
    const int narrow = kRingCtasPerSm * sms, wide = kRingCtasPerSmWide * sms;
    constexpr int SW = kRingSlotsWide, SN = kRingSlotsNarrow;
    switch (T) {
        case 1: return launch_tma_t<1, 4, SN, true>(mw, md, ma, mad, N, K, y, ldy, resid, ldr, narrow, s);
        case 2: return launch_tma_t<2, 4, SN, false>(mw, md, ma, mad, N, K, y, ldy, resid, ldr, narrow, s);
        case 3: return launch_tma_t<3, 4, SN, false>(mw, md, ma, mad, N, K, y, ldy, resid, ldr, narrow, s);
        case 4: return launch_tma_t<4, 4, SN, false>(mw, md, ma, mad, N, K, y, ldy, resid, ldr, narrow, s);
        case 5: return launch_tma_t<5, 2, SW, false>(mw, md, ma, mad, N, K, y, ldy, resid, ldr, wide, s);
        case 6: return launch_tma_t<6, 2, SW, false>(mw, md, ma, mad, N, K, y, ldy, resid, ldr, wide, s);
        case 7: return launch_tma_t<7, 2, SW, false>(mw, md, ma, mad, N, K, y, ldy, resid, ldr, wide, s);
        default: return launch_tma_t<8, 2, SW, false>(mw, md, ma, mad, N, K, y, ldy, resid, ldr, wide, s);
    }
}

cudaError_t launch_matvec_tma(const int8_t* wq, const __half* wd, int N, int K, const int8_t* aq, const float* ad,
                              int T, float* y, int64_t ldy, const float* resid, int64_t ldr, cudaStream_t s)
{
    // 1..8 rows: one launch.  13..16 rows: rows 0..7, then rows 8..T-1 - the
    // weights stream twice, which still beats the register kernel there;
    // 9..12 rows stay on the register kernel (measured faster).
    const int sms = sm_count();
    if (sms <= 0 || T < 1 || (T > 8 && T < 13) || T > 16) return cudaErrorNotSupported;
    if (T <= 8) return launch_ring_rows(wq, wd, N, K, aq, ad, T, y, ldy, resid, ldr, sms, s);
    CUtensorMap probe[4];
    if (!ring_maps(wq, wd, N, K, aq + (size_t)8 * K, ad + (size_t)8 * (K / 32), T - 8, 8, &probe[0], &probe[1],
                   &probe[2], &probe[3]))
        return cudaErrorNotSupported;  // both halves take the ring or neither does
    cudaError_t e = launch_ring_rows(wq, wd, N, K, aq, ad, 8, y, ldy, resid, ldr, sms, s);
    if (e != cudaSuccess) return e;
    return launch_ring_rows(wq, wd, N, K, aq + (size_t)8 * K, ad + (size_t)8 * (K / 32), T - 8, y + 8 * ldy, ldy,
                            resid ? resid + 8 * ldr : nullptr, ldr, sms, s);
}

// One fused launch of T <= 8 rows, three slots: 8 rotation pairs per group up
// to 4 rows, 4 pairs for 5..8.
static cudaError_t qkv_ring_rows(const int8_t* wq, const __half* wd, int K, const int8_t* aq, const float* ad, int T,
                                 float* qkv, int Hq, int Hkv, const RowPos& pos, const RopeFreq& f, float* q_rot,
                                 const KvRows& kv, cudaStream_t s)
{
    const int N = (Hq + 2 * Hkv) * kHeadDim;
    CUtensorMap mw, mdp, ma, mad;
    if (!ring_maps(wq, wd, N, K, aq, ad, T, T <= 4 ? 8 : 4, &mw, &mdp, &ma, &mad)) return cudaErrorNotSupported;
    constexpr int SW = kRingSlotsWide, SN = kRingSlotsNarrow;
    switch (T) {
        case 1: return launch_qkv_tma_t<1, 4, SN, true>(mw, mdp, ma, mad, K, qkv, Hq, Hkv, pos, f, q_rot, kv, s);
        case 2: return launch_qkv_tma_t<2, 4, SN, false>(mw, mdp, ma, mad, K, qkv, Hq, Hkv, pos, f, q_rot, kv, s);
        case 3: return launch_qkv_tma_t<3, 4, SN, false>(mw, mdp, ma, mad, K, qkv, Hq, Hkv, pos, f, q_rot, kv, s);
        case 4: return launch_qkv_tma_t<4, 4, SN, false>(mw, mdp, ma, mad, K, qkv, Hq, Hkv, pos, f, q_rot, kv, s);
        case 5: return launch_qkv_tma_t<5, 2, SW, false>(mw, mdp, ma, mad, K, qkv, Hq, Hkv, pos, f, q_rot, kv, s);
        case 6: return launch_qkv_tma_t<6, 2, SW, false>(mw, mdp, ma, mad, K, qkv, Hq, Hkv, pos, f, q_rot, kv, s);
        case 7: return launch_qkv_tma_t<7, 2, SW, false>(mw, mdp, ma, mad, K, qkv, Hq, Hkv, pos, f, q_rot, kv, s);
        default: return launch_qkv_tma_t<8, 2, SW, false>(mw, mdp, ma, mad, K, qkv, Hq, Hkv, pos, f, q_rot, kv, s);
    }
}

cudaError_t launch_qkv_rope_tma(const int8_t* wq, const __half* wd, int K, const int8_t* aq, const float* ad, int T,
                                float* qkv, int Hq, int Hkv, const RowPos& pos, const RopeFreq& f, float* q_rot,
                                const KvRows& kv, cudaStream_t s)
{
    // 1..8 rows: one launch; 13..16 rows: rows 0..7, then rows 8..T-1 (their
    // positions and K/V destinations shifted down); 9..12 rows: not taken
    if (T < 1 || (T > 8 && T < 13) || T > 16) return cudaErrorNotSupported;
    if (T <= 8) return qkv_ring_rows(wq, wd, K, aq, ad, T, qkv, Hq, Hkv, pos, f, q_rot, kv, s);
    const int N = (Hq + 2 * Hkv) * kHeadDim;
    CUtensorMap probe[4];
    if (!ring_maps(wq, wd, N, K, aq + (size_t)8 * K, ad + (size_t)8 * (K / 32), T - 8, 4, &probe[0], &probe[1],
                   &probe[2], &probe[3]))
        return cudaErrorNotSupported;  // both halves take the ring or neither does
    RowPos pos_hi{};
    KvRows kv_hi{};
    pos_hi.n_rows = kv_hi.n_rows = T - 8;
    for (int t = 8; t < T; ++t) {
        pos_hi.pos[t - 8] = pos.pos[t];
        kv_hi.row[t - 8] = kv.row[t];
    }
    const cudaError_t e = qkv_ring_rows(wq, wd, K, aq, ad, 8, qkv, Hq, Hkv, pos, f, q_rot, kv, s);
    if (e != cudaSuccess) return e;
    return qkv_ring_rows(wq, wd, K, aq + (size_t)8 * K, ad + (size_t)8 * (K / 32), T - 8, qkv + (size_t)8 * N, Hq, Hkv,
                         pos_hi, f, q_rot + (size_t)8 * Hq * kHeadDim, kv_hi, s);
}

namespace {

constexpr int kGateUpSlots = 4;  // two CTAs per SM at most, so one more slot than the plain ring

template <int T, bool BIAS>
cudaError_t launch_gateup_t(const CUtensorMap& mw, const CUtensorMap& mdp, const CUtensorMap& ma,
                            const CUtensorMap& mad, int F, int K, float* gu, float* h, int8_t* hq, float* hd,
                            int grid, cudaStream_t s)
{
    using L = RingLayout<T, 4, kGateUpSlots>;
    static std::atomic<bool> done[kMaxDevices];
    cudaError_t e = set_smem_once(q8_gateup_swiglu_tma_kernel<T, kGateUpSlots, BIAS>, L::SMEM, done);
    if (e == cudaSuccess)
        e = launch_pdl_smem(q8_gateup_swiglu_tma_kernel<T, kGateUpSlots, BIAS>, dim3(grid),
                            dim3(32 * (gateup_warps(T) + 1)),
                            L::SMEM, s, mw, mdp, ma, mad, F, K, gu, h, hq, hd);
    count_launches(1);
    return e;
}

}  // namespace

// The fused gate||up + SwiGLU + q8_0 launch for 1..4 rows: four slots, the
// units spread so that every CTA gets the same number (a grid of U/k CTAs, k
// the smallest count that keeps three CTAs per SM or fewer).  Not taken (the
// caller then launches the projection and the SwiGLU kernel) for other row
// counts, shapes the ring does not take or F not a multiple of 32.
cudaError_t launch_gateup_swiglu_tma(const int8_t* wq, const __half* wd, int F, int K, const int8_t* aq,
                                     const float* ad, int T, float* gu, float* h, int8_t* hq, float* hd,
                                     cudaStream_t s)
{
    const int sms = sm_count();
    if (sms <= 0 || T < 1 || T > 4 || F % 32 != 0 || F < 32) return cudaErrorNotSupported;
    CUtensorMap mw, mdp, ma, mad;
    if (!ring_maps(wq, wd, 2 * F, K, aq, ad, T, 8, &mw, &mdp, &ma, &mad)) return cudaErrorNotSupported;
    const int U = F / 32;
    const int k = (U + kRingCtasPerSm * sms - 1) / (kRingCtasPerSm * sms);
    const int grid = (U + k - 1) / k;
    switch (T) {
        case 1: return launch_gateup_t<1, true>(mw, mdp, ma, mad, F, K, gu, h, hq, hd, grid, s);
        case 2: return launch_gateup_t<2, false>(mw, mdp, ma, mad, F, K, gu, h, hq, hd, grid, s);
        case 3: return launch_gateup_t<3, false>(mw, mdp, ma, mad, F, K, gu, h, hq, hd, grid, s);
        default: return launch_gateup_t<4, false>(mw, mdp, ma, mad, F, K, gu, h, hq, hd, grid, s);
    }
}

cudaError_t launch_wait_expiry(uint64_t limit_ns, cudaStream_t s)
{
    wait_expiry_kernel<<<1, 32, 0, s>>>(limit_ns);
    count_launches(1);
    return cudaGetLastError();
}

cudaError_t read_wait_timeouts(uint32_t* count, bool reset)
{
    uint32_t mine = 0, mma = 0, attn = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&mine, g_wait_timeouts, sizeof(uint32_t));
    if (e == cudaSuccess && reset) {
        const uint32_t zero = 0;
        e = cudaMemcpyToSymbol(g_wait_timeouts, &zero, sizeof(uint32_t));
    }
    if (e == cudaSuccess) e = read_mma_wait_timeouts(&mma, reset);
    if (e == cudaSuccess) e = read_attn_wait_timeouts(&attn, reset);
    if (e == cudaSuccess) *count = mine + mma + attn;
    return e;
}

}  // namespace luce
