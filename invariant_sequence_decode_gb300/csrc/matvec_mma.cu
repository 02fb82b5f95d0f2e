// matvec_mma.cu - the q8_0 matvec for wide verify batches (up to 16
// activation rows) with the block dots on the tensor cores, weights streamed
// through a TMA ring in shared memory.
//
// "#1209 Speed up concurrent generation, fix QFUSE ...", What changed and
// why, item 1: wide verify batches of 8/12/16 rows exist to reuse the
// weights across requests, so every weight byte must cross HBM once for all
// rows; "exact 4-slot concurrent serving", How it stays exact: a row's
// result may not depend on how many rows share the launch.
//
// Arithmetic: identical to q8_matvec_kernel (matvec.cu) and the dp4a ring
// (matvec_tma.cu).  Block b of a weight row feeds chain b mod 32; each chain
// adds its blocks in ascending order, acc = fma(fp16(wd) * ad[t], dot, acc),
// where dot is the block's exact integer dot; the 32 chain values meet in the
// xor butterfly over offsets 16, 8, 4, 2, 1.  Only the way dot is formed
// differs: the int8 values are converted to binary16 exactly (the weights
// with a bias of 1152, removed through the accumulator) and multiplied by
// mma.sync m16n8k16 with fp32 accumulation; every product, partial sum and
// accumulator value of a block is an integer of magnitude below 2^24, exact
// in fp32, so the result is the exact dot, the value the dp4a kernels form.
//
// Why tensor cores here: at 16 rows a dp4a kernel issues 128 dp4a per
// 32-weight block, more than GB300's dp4a rate allows at HBM speed (measured
// ~60 per SM per clock), and int8 mma.sync is slower still on this part
// (~0.15 POPS); f16 mma.sync (~0.6 PFLOP/s) leaves headroom.
//
// Work split (GB300): one persistent CTA per SM, CW consumer warps and one
// producer warp.  A CTA owns a contiguous range of 16-row tiles of W and walks
// it in groups of TL tiles.  A stage is one kilobyte of K of a group: block c
// of stage j is block 32j + c, one block for each chain.  The producer keeps
// a ring of S stages in flight with tensor copies: W viewed as
// [K/128][N][128 B] (one 16-row x 1 KB box per tile), the activations as
// [K/128][T][128 B] (a box of 8 or 16 token rows, rows past T zero-filled),
// both with the 128-byte swizzle so that ldmatrix reads them without bank
// conflicts, and the weight and activation scales as one box each.  Warp w
// owns chains w + CW p: for each it loads the block's activation fragments
// (ldmatrix) and converts them once, forms -1152 times each token's block
// sum with two MMAs against a constant operand, then for each tile loads the
// weight fragments, converted with a bias (each weight w becomes the exact
// half w + 1152), and runs two MMAs (k = 2 x 16) per 8 tokens starting from
// that -1152 sum, which removes the bias exactly, followed by the fp32 chain
// update.  The k order inside a block is permuted the same way in both
// operands (thread quarter q holds bytes 4q..4q+3 of each 16-byte half),
// which leaves the integer dot unchanged.  At the end of a group a warp's
// chains meet in the butterfly's first levels in registers, the remaining
// levels across warps through shared memory.  Rows past N and blocks past K
// are zero-filled by the copy engine and never stored or counted.
//
// Every wait is bounded (about one second, ring.cuh); an expired wait adds one
// to this file's device counter (read by luce_wait_timeouts) and the CTA
// writes no further outputs.  The producer drains its last stages' copies
// (ring_drain, bounded) before it returns.
#include <string.h>

#include <atomic>
#include <type_traits>

#include "common.cuh"
#include "kernels.h"
#include "ring.cuh"

namespace luce {

namespace {

__device__ unsigned int g_mma_wait_timeouts;

constexpr int kTileRows = 16;
constexpr int kTileBytes = kTileRows * 1024;   // one tile's kilobyte of K

// Shape of a ring: NT token tiles of 8 (T <= 8 NT), groups of TL 16-row
// tiles, S slots, CW consumer warps in H halves (H = 2: each half serves one
// of two token tiles; H = 1: every warp serves all NT).
template <int NT, int TL, int S, int CW, int H>
struct MmaRing {
    static constexpr int TOK = 8 * NT;
    static constexpr int ROWS = TL * kTileRows;
    static constexpr int WH = CW / H;                   // warps sharing one token tile
    static constexpr int NTL = NT / H;                  // token tiles per warp
    static constexpr int CP = 32 / WH;                  // chains per consumer warp
    static constexpr int THREADS = 32 * (CW + 1);       // consumer warps + the producer warp
    static constexpr int W = TL * kTileBytes;           // [tile][8 lines][16 rows][128 B], swizzled
    static constexpr int A = TOK * 1024;                // [8 lines][TOK][128 B], swizzled
    static constexpr int WD = ROWS * 64;                // [ROWS][32 fp16]
    static constexpr int AD = TOK * 128;                // [TOK][32 fp32]
    static constexpr int STAGE = W + A + WD + AD;       // a multiple of 1024
    static constexpr int RED = (WH / 2) * ROWS * TOK;   // floats of the reduction buffer
    static constexpr int SMEM = 1024 + S * STAGE + RED * 4 + 2 * S * 8 + 16;
    static_assert(WH == 8 || WH == 16, "chains split evenly, butterfly levels split at a power of two");
    static_assert(H == 1 || (H == 2 && NT == 2), "halves split two token tiles");
    static_assert(STAGE % 1024 == 0, "slots stay 1024-byte aligned (the swizzle's period)");
    static_assert(SMEM <= 232448, "one CTA per SM");
};

// Byte offset of 16-byte chunk `chunk` of line `line` in a region written by
// a tensor copy with the 128-byte swizzle (chunk index xor line mod 8).
__device__ __forceinline__ uint32_t swz(int line, int chunk) { return line * 128 + ((chunk ^ (line & 7)) << 4); }

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4])
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t& r0, uint32_t& r1)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(addr));
}

// Four int8 values (bytes 0..3 of x) as two binary16 pairs lo = (x0, x1),
// hi = (x2, x3), each value v as the half 1024 + (v + 128) = v + 1152, exact
// (v ^ 0x80 placed under the exponent of 1024).
__device__ __forceinline__ void i8x4_to_h2_biased(uint32_t x, uint32_t& lo, uint32_t& hi)
{
    const uint32_t u = x ^ 0x80808080u;
    lo = __byte_perm(u, 0x64646464u, 0x7170);
    hi = __byte_perm(u, 0x64646464u, 0x7372);
}

// The same values without the bias (1152 subtracted, exact).
__device__ __forceinline__ void i8x4_to_h2(uint32_t x, uint32_t& lo, uint32_t& hi)
{
    i8x4_to_h2_biased(x, lo, hi);
    asm("sub.rn.f16x2 %0, %0, %1;" : "+r"(lo) : "r"(0x64806480u));
    asm("sub.rn.f16x2 %0, %0, %1;" : "+r"(hi) : "r"(0x64806480u));
}

constexpr uint32_t kMinus1152x2 = 0xE480E480u;  // (-1152, -1152) as binary16

// d = A(16x16) B(16x8) (+ d when ACC), f16 operands, fp32 accumulation.
template <bool ACC>
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    if (ACC)
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
            "{%0,%1,%2,%3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    else
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
            "{%10,%10,%10,%10};"
            : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(0.0f));
}

// d = A(16x16) B(16x8) + c, c a separate operand (no register copies).
__device__ __forceinline__ void mma16816c(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1,
                                          const float (&c)[4])
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%10,%11,%12,%13};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]), "f"(c[2]), "f"(c[3]));
}

// Two fp32 lanes in one 64-bit register: the packed (f32x2) multiply and
// fused multiply-add of sm_100 and later round each lane exactly as the
// scalar mul.rn / fma.rn do, in half the instructions.
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi)
{
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}

__device__ __forceinline__ void f2_unpack(uint64_t v, float& lo, float& hi)
{
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b)
{
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c)
{
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}

// Shared-memory carve-up: S 1024-aligned slots, the reduction buffer, the
// slot barriers and a failure flag.
template <int NT, int TL, int S, int CW, int H>
struct MmaSmem {
    uint8_t* slots;
    float* red;
    uint64_t* full;   // slot filled: the producer's arrival + the copies' bytes
    uint64_t* empty;  // slot released: one arrival per consumer warp
    volatile int* failed;
    __device__ explicit MmaSmem(uint8_t* raw)
    {
        using L = MmaRing<NT, TL, S, CW, H>;
        slots = raw + ((1024u - (smem_addr(raw) & 1023u)) & 1023u);
        red = reinterpret_cast<float*>(slots + S * L::STAGE);
        full = reinterpret_cast<uint64_t*>(red + L::RED);
        empty = full + S;
        failed = reinterpret_cast<volatile int*>(empty + S);
    }
};

// The producer thread: stage it (group it / nj, K-kilobyte it % nj) of
// `total` goes to slot it % S; the group's first tile is t0 + TL (it / nj) and
// it has min(TL, t1 - that) tiles.  The first S stages' weights go before the
// wait on the previous kernel, which the activations need.
// PAIRED (the q|k|v projection with RoPE): tile v holds rows 8a .. 8a + 7
// and 64 + 8a .. 64 + 8a + 7 of head v / 8 (a = v % 8), two 8-row boxes each
// (mw and md with 8-row boxes), so rows r and r + 8 of a tile are the
// rotation pair (8a + r, 8a + r + 64) and meet in one thread's fragment.
__device__ __forceinline__ int paired_row(int v, int half) { return (v >> 3) * kHeadDim + 8 * (v & 7) + 64 * half; }

template <int NT, int TL, int S, int CW, int H, bool PAIRED = false>
__device__ __forceinline__ void mma_produce(const MmaSmem<NT, TL, S, CW, H>& R, int total, int nj, int t0, int t1,
                                            const CUtensorMap* mw, const CUtensorMap* md, const CUtensorMap* ma,
                                            const CUtensorMap* mad)
{
    using L = MmaRing<NT, TL, S, CW, H>;
    auto tiles = [&](int it) { return min(TL, t1 - (t0 + TL * (it / nj))); };
    auto load_w = [&](int it) {
        const int s = it % S, j = it % nj, tile0 = t0 + TL * (it / nj), nt = tiles(it);
        uint8_t* slot = R.slots + s * L::STAGE;
        if (PAIRED) {
            for (int i = 0; i < nt; ++i)
                for (int hf = 0; hf < 2; ++hf) {
                    const int row = paired_row(tile0 + i, hf);
                    tma_load_3d(slot + i * kTileBytes + hf * (kTileBytes / 2), mw, 0, row, 8 * j, &R.full[s]);
                    tma_load_2d(slot + L::W + L::A + (16 * i + 8 * hf) * 64, md, 32 * j, row, &R.full[s]);
                }
        } else {
            for (int i = 0; i < nt; ++i)
                tma_load_3d(slot + i * kTileBytes, mw, 0, kTileRows * (tile0 + i), 8 * j, &R.full[s]);
            tma_load_2d(slot + L::W + L::A, md, 32 * j, kTileRows * tile0, &R.full[s]);
        }
    };
    auto load_a = [&](int it) {
        const int s = it % S, j = it % nj;
        uint8_t* slot = R.slots + s * L::STAGE;
        tma_load_3d(slot + L::W, ma, 0, 0, 8 * j, &R.full[s]);
        tma_load_2d(slot + L::W + L::A + L::WD, mad, 32 * j, 0, &R.full[s]);
    };
    auto bytes = [&](int it) {
        return (uint32_t)(tiles(it) * kTileBytes + L::A + (PAIRED ? tiles(it) * kTileRows * 64 : L::WD) + L::AD);
    };
    const int pre = min(S, total);
    for (int it = 0; it < pre; ++it) {
        mbar_expect_tx(&R.full[it], bytes(it));
        load_w(it);
    }
    pdl_wait();
    for (int it = 0; it < pre; ++it) load_a(it);
    int issued = pre;
    for (; issued < total; ++issued) {
        const int it = issued, s = it % S;
        if (!mbar_wait(&R.empty[s], ((it / S) - 1) & 1, &g_mma_wait_timeouts)) break;
        mbar_expect_tx(&R.full[s], bytes(it));
        load_w(it);
        load_a(it);
    }
    ring_drain<S>(R.full, issued, &g_mma_wait_timeouts);
}

// A consumer warp's chains for one group: stages it .. it + nj - 1 (it
// advances).  Warp w = nh WH + wl serves token tiles nh NTL .. nh NTL + NTL - 1
// and chains wl + WH p.  acc[p][i][n][e] = chain wl + WH p of tile i, local
// token tile n, element e of the m16n8 fragment (rows gr, gr + 8; tokens
// 2tq, 2tq + 1).  ok turns false when a wait expires; from then on the warp
// waits for nothing more.
template <int NT, int TL, int S, int CW, int H, bool PAIRED = false>
__device__ __forceinline__ void mma_chains(const MmaSmem<NT, TL, S, CW, H>& R, int& it, int nj, int nb, int nt, int w,
                                           int lane, float (&acc)[32 / (CW / H)][TL][NT / H][4], bool& ok)
{
    using L = MmaRing<NT, TL, S, CW, H>;
    constexpr int CP = L::CP, NTL = L::NTL, WH = L::WH;
    const int wl = w % WH, nh = w / WH;
    const int gr = lane >> 2, tq = lane & 3;
    const int mi = lane >> 3, rr = lane & 7;  // ldmatrix: the matrix and row this lane addresses
    const uint32_t bias[4] = {kMinus1152x2, kMinus1152x2, kMinus1152x2, kMinus1152x2};
#pragma unroll
    for (int p = 0; p < CP; ++p)
#pragma unroll
        for (int i = 0; i < TL; ++i)
#pragma unroll
            for (int n = 0; n < NTL; ++n)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[p][i][n][e] = 0.0f;
    for (int j = 0; j < nj; ++j, ++it) {
        const int s = it % S;
        if (ok && !mbar_wait(&R.full[s], (it / S) & 1, &g_mma_wait_timeouts)) {
            ok = false;
            *R.failed = 1;
        }
        if (!ok) continue;
        const uint8_t* slot = R.slots + s * L::STAGE;
        const uint32_t s_w = smem_addr(slot), s_a = s_w + L::W;
        const __half* wd = reinterpret_cast<const __half*>(slot + L::W + L::A);
        const float* ad = reinterpret_cast<const float*>(slot + L::W + L::A + L::WD);
        // with two token tiles, a stage whose 32 blocks all exist, of a group
        // of TL tiles, runs without the per-chain and per-tile guards, so that
        // the chains and tiles of the stage form one block of straight-line
        // code (9-16 rows: 3.43 -> 3.77 TB/s over the 27B layer's projections;
        // with one token tile the 16 warps' register cap makes it slower)
        auto stage = [&](auto full) {
            constexpr bool FULL = decltype(full)::value;
#pragma unroll
            for (int p = 0; p < CP; ++p) {
                const int c = wl + WH * p;
                if (FULL || 32 * j + c < nb) {
                    const int z = c >> 2, ch = 2 * (c & 3);
                    // activation fragments of block c: b[n][k-step][0..1], exact
                    uint32_t b[NTL][2][2];
                    if (NTL == 2) {
                        const int line = z * 16 + rr + 8 * (mi & 1);
                        uint32_t r[4];
                        ldsm_x4(s_a + swz(line, ch + (mi >> 1)), r);
                        i8x4_to_h2(r[0], b[0][0][0], b[0][0][1]);
                        i8x4_to_h2(r[2], b[0][1][0], b[0][1][1]);
                        i8x4_to_h2(r[1], b[NTL - 1][0][0], b[NTL - 1][0][1]);
                        i8x4_to_h2(r[3], b[NTL - 1][1][0], b[NTL - 1][1][1]);
                    } else {
                        const int line = z * L::TOK + 8 * nh + rr;
                        uint32_t r0, r1;
                        ldsm_x2(s_a + swz(line, ch + (mi & 1)), r0, r1);
                        i8x4_to_h2(r0, b[0][0][0], b[0][0][1]);
                        i8x4_to_h2(r1, b[0][1][0], b[0][1][1]);
                    }
                    // -1152 times each token's block sum: the accumulator start
                    // that cancels the weights' bias
                    float c0[NTL][4];
                    float sav[NTL][2];
#pragma unroll
                    for (int n = 0; n < NTL; ++n) {
                        mma16816<false>(c0[n], bias, b[n][0][0], b[n][0][1]);
                        mma16816<true>(c0[n], bias, b[n][1][0], b[n][1][1]);
                        const int t0 = 8 * (nh * NTL + n) + 2 * tq;
                        sav[n][0] = ad[t0 * 32 + c];
                        sav[n][1] = ad[(t0 + 1) * 32 + c];
                    }
#pragma unroll
                    for (int i = 0; i < TL; ++i) {
                        if (FULL || i < nt) {
                            uint32_t r[4], a[2][4];
                            if (PAIRED)  // rows 0-7 and 8-15 of the tile are two 8-row boxes
                                ldsm_x4(s_w + i * kTileBytes + (mi & 1) * (kTileBytes / 2) + swz(z * 8 + rr, ch + (mi >> 1)),
                                        r);
                            else
                                ldsm_x4(s_w + i * kTileBytes + swz(z * 16 + rr + 8 * (mi & 1), ch + (mi >> 1)), r);
                            i8x4_to_h2_biased(r[0], a[0][0], a[0][2]);  // row gr, bytes 4tq..4tq+3 of the first half
                            i8x4_to_h2_biased(r[1], a[0][1], a[0][3]);  // row gr + 8
                            i8x4_to_h2_biased(r[2], a[1][0], a[1][2]);  // the second half
                            i8x4_to_h2_biased(r[3], a[1][1], a[1][3]);
                            const float w0 = __half2float(wd[(16 * i + gr) * 32 + c]);
                            const float w1 = __half2float(wd[(16 * i + gr + 8) * 32 + c]);
#pragma unroll
                            for (int n = 0; n < NTL; ++n) {
                                float d[4];
                                mma16816c(d, a[0], b[n][0][0], b[n][0][1], c0[n]);
                                mma16816<true>(d, a[1], b[n][1][0], b[n][1][1]);
                                // q[e] = fma(w(row) * sav(token), d[e], q[e]),
                                // the two tokens of a row as one packed pair
                                float* q = acc[p][i][n];
                                const uint64_t sa = f2_pack(sav[n][0], sav[n][1]);
                                const uint64_t q01 = f2_fma(f2_mul(f2_pack(w0, w0), sa), f2_pack(d[0], d[1]),
                                                            f2_pack(q[0], q[1]));
                                const uint64_t q23 = f2_fma(f2_mul(f2_pack(w1, w1), sa), f2_pack(d[2], d[3]),
                                                            f2_pack(q[2], q[3]));
                                f2_unpack(q01, q[0], q[1]);
                                f2_unpack(q23, q[2], q[3]);
                            }
                        }
                    }
                }
            }
        };
        if (NT == 2 && 32 * j + 32 <= nb && nt == TL)
            stage(std::true_type{});
        else
            stage(std::false_type{});
        __syncwarp();
        if (lane == 0) mbar_arrive(&R.empty[s]);
    }
}

// Butterfly levels over the n values v[0..n): for off = n/2, ..., 1:
// v[i] += v[i + off] (i < off); the result is v[0].
template <int NV>
__device__ __forceinline__ float butterfly(float (&v)[NV])
{
#pragma unroll
    for (int off = NV / 2; off >= 1; off >>= 1)
#pragma unroll
        for (int i = 0; i < off; ++i) v[i] = __fadd_rn(v[i], v[i + off]);
    return v[0];
}

// The butterfly over one group's chains.  Chain index c = wl + WH p, so the
// levels with offsets 16 .. WH pair chains of one thread (p with p + CP/2,
// ...) and are taken in registers; level WH/2 (warp wl with wl + WH/2 of the
// same half) meets in a [WH/2][16 TL rows][TOK] buffer: the upper warps of
// each half write, the lower ones add their values in place; the levels
// below are taken by the thread that writes the (row, token) output
// (mma_finish).  Barriers: one before the writes (the last group's readers
// are done), one after each phase.
template <int NT, int TL, int CW, int H>
__device__ __forceinline__ void mma_reduce(float* rb, int w, int lane, bool later_group,
                                           const float (&acc)[32 / (CW / H)][TL][NT / H][4])
{
    constexpr int TOK = 8 * NT, ROWS = TL * kTileRows, WH = CW / H, CP = 32 / WH, NTL = NT / H;
    const int gr = lane >> 2, tq = lane & 3, wl = w % WH, nh = w / WH;
    float v[TL][NTL][4];
#pragma unroll
    for (int i = 0; i < TL; ++i)
#pragma unroll
        for (int n = 0; n < NTL; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                float u[CP];
#pragma unroll
                for (int p = 0; p < CP; ++p) u[p] = acc[p][i][n][e];
                v[i][n][e] = butterfly<CP>(u);
            }
    auto at = [&](int i, int n, int e) {
        const int row = 16 * i + gr + 8 * (e >> 1), tok = 8 * (nh * NTL + n) + 2 * tq + (e & 1);
        return ((wl % (WH / 2)) * ROWS + row) * TOK + tok;
    };
    if (later_group) asm volatile("bar.sync 1, %0;" ::"n"(32 * CW) : "memory");
    if (wl >= WH / 2) {
#pragma unroll
        for (int i = 0; i < TL; ++i)
#pragma unroll
            for (int n = 0; n < NTL; ++n)
#pragma unroll
                for (int e = 0; e < 4; ++e) rb[at(i, n, e)] = v[i][n][e];
    }
    asm volatile("bar.sync 1, %0;" ::"n"(32 * CW) : "memory");
    if (wl < WH / 2) {
#pragma unroll
        for (int i = 0; i < TL; ++i)
#pragma unroll
            for (int n = 0; n < NTL; ++n)
#pragma unroll
                for (int e = 0; e < 4; ++e) rb[at(i, n, e)] = __fadd_rn(v[i][n][e], rb[at(i, n, e)]);
    }
    asm volatile("bar.sync 1, %0;" ::"n"(32 * CW) : "memory");
}

// The butterfly's levels below WH/2 for one (row, token): over the WH/2
// values the lower warps left at idx, stride apart.
template <int WH>
__device__ __forceinline__ float mma_finish(const float* rb, int idx, int stride)
{
    float u[WH / 2];
#pragma unroll
    for (int k = 0; k < WH / 2; ++k) u[k] = rb[k * stride + idx];
    return butterfly<WH / 2>(u);
}

}  // namespace

// mw: W as uint8 [K/128][N][128], box {128, 16, 8}, 128-byte swizzle;
// md: scales fp16 [N][K/32], box {32, 16 TL}; ma: activations uint8
// [K/128][T][128], box {128, 8 NT, 8}, 128-byte swizzle; mad: activation
// scales fp32 [T][K/32], box {32, 8 NT}.  Persistent: CTA b owns tiles
// [b*ntl/grid, (b+1)*ntl/grid) of the ntl = ceil(N/16) tiles.
template <int NT, int TL, int S, int CW, int H>
__global__ void __launch_bounds__(32 * (CW + 1), 1)
q8_matvec_mma_kernel(const __grid_constant__ CUtensorMap mw, const __grid_constant__ CUtensorMap md,
                     const __grid_constant__ CUtensorMap ma, const __grid_constant__ CUtensorMap mad, int N, int K,
                     int T, float* y, int64_t ldy, const float* resid, int64_t ldr)
{
    using L = MmaRing<NT, TL, S, CW, H>;
    extern __shared__ uint8_t smem_raw[];
    const MmaSmem<NT, TL, S, CW, H> R(smem_raw);
    pdl_trigger();
    const int nb = K >> 5, nj = (nb + 31) >> 5;
    const int ntl = (N + kTileRows - 1) / kTileRows;
    const int t0 = (int)((int64_t)blockIdx.x * ntl / gridDim.x);
    const int t1 = (int)((int64_t)(blockIdx.x + 1) * ntl / gridDim.x);
    const int ngrp = (t1 - t0 + TL - 1) / TL;
    const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&R.full[s], 1);
            mbar_init(&R.empty[s], CW);
        }
        *R.failed = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    if (w == CW) {
        if (lane == 0) mma_produce<NT, TL, S, CW, H>(R, ngrp * nj, nj, t0, t1, &mw, &md, &ma, &mad);
        return;
    }

    pdl_wait();  // the residual and y may be touched by earlier kernels
    bool ok = true;
    int it = 0;
    for (int gi = 0; gi < ngrp; ++gi) {
        const int tile0 = t0 + TL * gi, nt = min(TL, t1 - tile0);
        float acc[L::CP][TL][L::NTL][4];
        mma_chains<NT, TL, S, CW, H>(R, it, nj, nb, nt, w, lane, acc, ok);
        mma_reduce<NT, TL, CW, H>(R.red, w, lane, gi > 0, acc);
        if (*R.failed) continue;
        for (int idx = tid; idx < L::ROWS * L::TOK; idx += 32 * CW) {
            const int row = idx / L::TOK, tok = idx - (idx / L::TOK) * L::TOK;
            const int n = kTileRows * tile0 + row;
            if (row < kTileRows * nt && n < N && tok < T) {
                float out = mma_finish<L::WH>(R.red, idx, L::ROWS * L::TOK);
                if (resid) out = __fadd_rn(resid[(size_t)tok * ldr + n], out);
                y[(size_t)tok * ldy + n] = out;
            }
        }
    }
}

// The decode step's q|k|v projection at wide verify batches with the RoPE
// rotation and the K/V append in the epilogue ("antirez/ds4 pull 604",
// Commit walkthrough): the tiles are PAIRED (mma_produce), so the thread that
// finishes row 8a + p of a head also finishes row 8a + p + 64, and it stores
// both to qkv, rotates them (q and k heads) by the token's position and
// writes q_rot, or rounds them to binary16 at the token's K/V destination -
// the rotation and conversion of qkv_rope_kv_kernel, so the same bits.
// mw: W as [K/128][N][128] with an 8-row box; md: scales with an 8-row box.
template <int NT, int TL, int S, int CW, int H>
__global__ void __launch_bounds__(32 * (CW + 1), 1)
q8_qkv_rope_mma_kernel(const __grid_constant__ CUtensorMap mw, const __grid_constant__ CUtensorMap md,
                       const __grid_constant__ CUtensorMap ma, const __grid_constant__ CUtensorMap mad, int K, int T,
                       float* __restrict__ qkv, int Hq, int Hkv, const __grid_constant__ RowPos pos,
                       const __grid_constant__ RopeFreq f, float* __restrict__ q_rot, const __grid_constant__ KvRows kv)
{
    using L = MmaRing<NT, TL, S, CW, H>;
    extern __shared__ uint8_t smem_raw[];
    const MmaSmem<NT, TL, S, CW, H> R(smem_raw);
    pdl_trigger();
    const int N = (Hq + 2 * Hkv) * kHeadDim;
    const int nb = K >> 5, nj = (nb + 31) >> 5;
    const int ntl = N / kTileRows;
    const int t0 = (int)((int64_t)blockIdx.x * ntl / gridDim.x);
    const int t1 = (int)((int64_t)(blockIdx.x + 1) * ntl / gridDim.x);
    const int ngrp = (t1 - t0 + TL - 1) / TL;
    const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&R.full[s], 1);
            mbar_init(&R.empty[s], CW);
        }
        *R.failed = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    if (w == CW) {
        if (lane == 0) mma_produce<NT, TL, S, CW, H, true>(R, ngrp * nj, nj, t0, t1, &mw, &md, &ma, &mad);
        return;
    }

    pdl_wait();  // the K/V caches and outputs may be touched by earlier kernels
    bool ok = true;
    int it = 0;
    const int ldq = N;
    for (int gi = 0; gi < ngrp; ++gi) {
        const int tile0 = t0 + TL * gi, nt = min(TL, t1 - tile0);
        float acc[L::CP][TL][L::NTL][4];
        mma_chains<NT, TL, S, CW, H, true>(R, it, nj, nb, nt, w, lane, acc, ok);
        mma_reduce<NT, TL, CW, H>(R.red, w, lane, gi > 0, acc);
        if (*R.failed) continue;
        // (tile i, pair p, token tok): rows p and 8 + p of tile i
        for (int idx = tid; idx < nt * 8 * L::TOK; idx += 32 * CW) {
            const int i = idx / (8 * L::TOK), rem = idx - i * 8 * L::TOK;
            const int p = rem / L::TOK, tok = rem - p * L::TOK;
            if (tok >= T) continue;
            const int v = tile0 + i, h = v >> 3, d = 8 * (v & 7) + p;  // the pair (d, d + 64) of head h
            float x0 = mma_finish<L::WH>(R.red, (16 * i + p) * L::TOK + tok, L::ROWS * L::TOK);
            float x1 = mma_finish<L::WH>(R.red, (16 * i + 8 + p) * L::TOK + tok, L::ROWS * L::TOK);
            float* yr = qkv + (size_t)tok * ldq + (size_t)h * kHeadDim;
            yr[d] = x0;
            yr[d + kHeadDim / 2] = x1;
            const bool rot = h < Hq + Hkv;
            if (rot) {
                const float2 cs = rope_cs(pos.pos[tok], f.inv[d]);
                rope_rotate(x0, x1, cs.x, cs.y);
            }
            if (h < Hq) {
                float* dst = q_rot + ((size_t)tok * Hq + h) * kHeadDim;
                dst[d] = x0;
                dst[d + kHeadDim / 2] = x1;
            } else {
                const KvRow kr = kv.row[tok];
                __half* dst = rot ? kr.k + (h - Hq) * kr.head_stride : kr.v + (h - Hq - Hkv) * kr.head_stride;
                dst[d] = __float2half_rn(x0);
                dst[d + kHeadDim / 2] = __float2half_rn(x1);
            }
        }
    }
}

namespace {

template <int NT, int TL, int S, int CW, int H>
cudaError_t launch_mma_t(const CUtensorMap& mw, const CUtensorMap& md, const CUtensorMap& ma, const CUtensorMap& mad,
                         int N, int K, int T, float* y, int64_t ldy, const float* resid, int64_t ldr, int ctas,
                         cudaStream_t s)
{
    using L = MmaRing<NT, TL, S, CW, H>;
    static std::atomic<bool> done[kMaxDevices];
    const cudaError_t attr = set_smem_once(q8_matvec_mma_kernel<NT, TL, S, CW, H>, L::SMEM, done);
    if (attr != cudaSuccess) return attr;
    const int ntl = (N + kTileRows - 1) / kTileRows;
    const int grid = min(ctas, ntl);
    const cudaError_t e = launch_pdl_smem(q8_matvec_mma_kernel<NT, TL, S, CW, H>, dim3(grid), dim3(L::THREADS), L::SMEM,
                                          s, mw, md, ma, mad, N, K, T, y, ldy, resid, ldr);
    count_launches(1);
    return e;
}

// The four maps of a launch; false when the shapes or alignments do not allow
// one (K a multiple of 256, 16-byte aligned operands, a driver that encodes it).
bool mma_maps(const int8_t* wq, const __half* wd, int N, int K, const int8_t* aq, const float* ad, int T, int tok_box,
              int scale_rows, CUtensorMap* mw, CUtensorMap* md, CUtensorMap* ma, CUtensorMap* mad,
              int w_rows = kTileRows)
{
    auto al16 = [](const void* p) { return ((uintptr_t)p & 15) == 0; };
    if (T < 1 || T > 16 || K % 256 != 0 || !al16(wq) || !al16(wd) || !al16(aq) || !al16(ad)) return false;
    const cuuint64_t nb = (cuuint64_t)K / 32, lines = (cuuint64_t)K / 128;
    // x = byte of a 128-byte line of K, y = row, z = line: rows of one line
    // land 128 bytes apart, which the swizzle spreads over all banks
    const cuuint64_t wdim[3] = {128, (cuuint64_t)N, lines}, wstr[2] = {(cuuint64_t)K, 128};
    const cuuint32_t wbox[3] = {128, (cuuint32_t)w_rows, 8};
    const cuuint64_t ddim[2] = {nb, (cuuint64_t)N}, dstr[1] = {nb * 2};
    const cuuint32_t dbox[2] = {32, (cuuint32_t)scale_rows};
    const cuuint64_t adim[3] = {128, (cuuint64_t)T, lines}, astr[2] = {(cuuint64_t)K, 128};
    const cuuint32_t abox[3] = {128, (cuuint32_t)tok_box, 8};
    const cuuint64_t addim[2] = {nb, (cuuint64_t)T}, adstr[1] = {nb * 4};
    const cuuint32_t adbox[2] = {32, (cuuint32_t)tok_box};
    return encode_map(mw, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, wq, wdim, wstr, wbox, CU_TENSOR_MAP_SWIZZLE_128B) &&
           encode_map(md, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, wd, ddim, dstr, dbox) &&
           encode_map(ma, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, aq, adim, astr, abox, CU_TENSOR_MAP_SWIZZLE_128B) &&
           encode_map(mad, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, ad, addim, adstr, adbox);
}

#ifndef MMA_TL
#define MMA_TL 3
#define MMA_S1 3
#define MMA_S2 3
#define MMA_CW1 16
#define MMA_CW2 8
#define MMA_H2 1
#endif
// Group size, ring depth and consumer warps per token tile count, measured
// on the 27B-shaped layer's four projections: groups of 3 tiles (48 rows)
// and 3 slots; 16 consumer warps up to 8 rows (8 at 9..16 rows, where 16
// warps leave 96 registers a thread and room for only 2 slots); the token
// tiles shared by all warps (splitting them across warp halves converts
// each weight fragment twice).
constexpr int kMmaTiles = MMA_TL, kMmaWarps1 = MMA_CW1, kMmaWarps2 = MMA_CW2, kMmaHalves2 = MMA_H2;
constexpr int kMmaSlots1 = MMA_S1, kMmaSlots2 = MMA_S2;

}  // namespace

cudaError_t launch_matvec_mma(const int8_t* wq, const __half* wd, int N, int K, const int8_t* aq, const float* ad,
                              int T, float* y, int64_t ldy, const float* resid, int64_t ldr, cudaStream_t s)
{
    const int sms = sm_count();
    if (sms <= 0 || T < 1 || T > 16) return cudaErrorNotSupported;
    CUtensorMap mw, md, ma, mad;
    if (!mma_maps(wq, wd, N, K, aq, ad, T, T <= 8 ? 8 : 16, kMmaTiles * kTileRows, &mw, &md, &ma, &mad))
        return cudaErrorNotSupported;
    if (T <= 8)
        return launch_mma_t<1, kMmaTiles, kMmaSlots1, kMmaWarps1, 1>(mw, md, ma, mad, N, K, T, y, ldy, resid, ldr,
                                                                      sms, s);
    return launch_mma_t<2, kMmaTiles, kMmaSlots2, kMmaWarps2, kMmaHalves2>(mw, md, ma, mad, N, K, T, y, ldy, resid,
                                                                           ldr, sms, s);
}

namespace {

template <int NT, int TL, int S, int CW, int H>
cudaError_t launch_qkv_mma_t(const CUtensorMap& mw, const CUtensorMap& md, const CUtensorMap& ma,
                             const CUtensorMap& mad, int K, int T, float* qkv, int Hq, int Hkv, const RowPos& pos,
                             const RopeFreq& f, float* q_rot, const KvRows& kv, int ctas, cudaStream_t s)
{
    using L = MmaRing<NT, TL, S, CW, H>;
    static std::atomic<bool> done[kMaxDevices];
    const cudaError_t attr = set_smem_once(q8_qkv_rope_mma_kernel<NT, TL, S, CW, H>, L::SMEM, done);
    if (attr != cudaSuccess) return attr;
    const int ntl = (Hq + 2 * Hkv) * kHeadDim / kTileRows;
    const cudaError_t e =
        launch_pdl_smem(q8_qkv_rope_mma_kernel<NT, TL, S, CW, H>, dim3(min(ctas, ntl)), dim3(L::THREADS), L::SMEM, s,
                        mw, md, ma, mad, K, T, qkv, Hq, Hkv, pos, f, q_rot, kv);
    count_launches(1);
    return e;
}

}  // namespace

cudaError_t launch_qkv_rope_mma(const int8_t* wq, const __half* wd, int K, const int8_t* aq, const float* ad, int T,
                                float* qkv, int Hq, int Hkv, const RowPos& pos, const RopeFreq& f, float* q_rot,
                                const KvRows& kv, cudaStream_t s)
{
    const int sms = sm_count();
    if (sms <= 0 || T < 1 || T > 16) return cudaErrorNotSupported;
    const int N = (Hq + 2 * Hkv) * kHeadDim;
    CUtensorMap mw, md, ma, mad;
    if (!mma_maps(wq, wd, N, K, aq, ad, T, T <= 8 ? 8 : 16, 8, &mw, &md, &ma, &mad, 8)) return cudaErrorNotSupported;
    if (T <= 8)
        return launch_qkv_mma_t<1, kMmaTiles, kMmaSlots1, kMmaWarps1, 1>(mw, md, ma, mad, K, T, qkv, Hq, Hkv, pos, f,
                                                                          q_rot, kv, sms, s);
    return launch_qkv_mma_t<2, kMmaTiles, kMmaSlots2, kMmaWarps2, kMmaHalves2>(mw, md, ma, mad, K, T, qkv, Hq, Hkv,
                                                                               pos, f, q_rot, kv, sms, s);
}

cudaError_t read_mma_wait_timeouts(uint32_t* count, bool reset)
{
    cudaError_t e = cudaMemcpyFromSymbol(count, g_mma_wait_timeouts, sizeof(uint32_t));
    if (e == cudaSuccess && reset) {
        const uint32_t zero = 0;
        e = cudaMemcpyToSymbol(g_mma_wait_timeouts, &zero, sizeof(uint32_t));
    }
    return e;
}

}  // namespace luce
