// attn.cu - multi-sequence GQA decode attention, split-K over each row's own
// f16 cache with an exact, ordered log-sum-exp merge.
//
// "antirez/ds4 pull 604", Commit walkthrough: one query token per sequence,
// each attending to its own cache, per-sequence views passed by value (max 4);
// section 2: one multi-sequence attention launch with no position limit.
//
// A row's keys are cut into chunks of CH keys, CH = attn_chunk_keys(row's key
// count) (128 up to 16,384 keys, else 256: small contexts get smaller chunks
// so the GPU has enough independent work).  One CTA of 256 threads (8 warps)
// per (row unit, chunk, KV head g) serves all GQ = Hq/Hkv query heads of g,
// so each K/V byte is read once.  Both contractions run on the tensor cores
// with f16 operands and fp32 accumulation.  f16 holds K and V exactly; q and
// the probabilities are fp32, so each is split into two f16 parts, x = hi +
// lo with hi = f16(x) and lo = f16(x - hi), and both parts are multiplied in.
// Keys are taken 128 at a time (a tile):
//   scores   (mma.sync m16n8k16) warp w owns keys 16w..16w+15 of the tile and
//            loads their K rows straight into its A fragments: lane quarter
//            t holds dims 32t..32t+31, and step s = 0..7 contracts dims
//            32t+4s..32t+4s+3 of every quarter t (q is laid out the same
//            way); per step the q_hi, then the q_lo product is accumulated;
//            s_h = scale * dot;
//   softmax  warp h owns head h: m = max_j s_hj, p_hj = exp(s_hj - m),
//            l = sum p_hj (lane-serial over j = lane + 32i, then butterfly);
//   values   the tile's V rows are staged in shared memory by cp.async while
//            the scores and the softmax run, then p.V:
//            - rows with 128-key chunks (attn_slot_kernel): consecutive rows
//              on one cache (a slot's verify rows) share one CTA, each row
//              taking its scores and softmax in turn, and p.V of all of them
//              is one tcgen05.mma pass: D[dim][n] = sum over the chunk's keys
//              of V[key][dim] P[n][key], A = the V tile (MN-major), B = the
//              rows' hi and lo probabilities (K-major), D in tensor memory
//              (lane = dim), out = D[hi] + D[lo]; each output column depends
//              on its own probability row only, so a row gives the same bits
//              alone, with its slot's other rows or as a single decode row;
//              the MMAs' completion wait is bounded and counts in
//              luce_wait_timeouts;
//            - rows past 16,384 keys (256-key chunks, two tiles through one V
//              buffer; attn_kernel): mma.sync, warp w owns dims 16w..16w+15
//              and for each step of 16 keys in key order accumulates
//              p_hi.V, then p_lo.V (A = the tile read transposed).
//   -> scratch (o_h[128], m_h, l_h) per row and chunk.
// A further kernel, launched behind with programmatic dependent launch (its
// wait returns once every chunk is written), merges each (row, query head)
// over the row's chunks, one CTA per pair and one thread per dim:
//   M = max_c m_c, w_c = e^(m_c - M), L = sum_c l_c w_c, O = sum_c o_c w_c,
//   out = O / L  (O sequential over c; L lane-serial over c = lane + 32i,
//   then a butterfly),
// and optionally quantizes out to q8_0 blocks (the Wo projection's input).
// Every chunking and reduction order, and which kernel serves a row, depends
// only on the row's own key count, never on the other rows, on which CTA
// merges or on the grid.
// A row's cache is flat or paged: pages hold 128 keys, one tile, so only the
// address of a tile's first key comes from the page table and a paged cache
// gives the flat cache's bits.
// The split of q assumes |q| < 65504 (the f16 range); larger entries make
// the row's scores non-finite.
#include <math.h>

#include "common.cuh"
#include "kernels.h"
#include "ring.cuh"

namespace luce {

constexpr int kPartStride = 132;  // o[128], m, l, 2 pad floats per (chunk, head)
constexpr int kAttnThreads = 256;
constexpr int kTileKeys = 128;    // keys staged in shared memory at a time
// Row stride of the probabilities: 264 = 8 (mod 32) words, so the value loads
// of 4 heads x 4 key pairs in one half-warp hit 16 distinct bank pairs.
constexpr int kPStride = kAttnChunk + 8;
constexpr int kAttnMaxGroupRows = 4;  // rows of one slot served by one CTA

size_t attn_part_floats(int total_chunks, int Hq) { return (size_t)total_chunks * Hq * kPartStride; }

int attn_chunk_keys(int len) { return len <= 16384 ? 128 : 256; }

template <int GQ>
struct AttnSmem {
    __half vt[kTileKeys * kHeadDim];  // staged V tile (32 KB)
    uint4 qf[8][32];                  // q as B fragments per step and lane: hi b0, hi b1, lo b0, lo b1
    float p[GQ][kPStride];            // scores, then probabilities, of the chunk
};

// Offset (in halves) of 16-byte piece c (8 dims) of key j in a staged tile.
__device__ __forceinline__ int tile_off(int j, int c) { return j * kHeadDim + ((c ^ (j & 7)) << 3); }

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// Stage keys [j0, j0 + 128) of a chunk (their rows tok_stride halves apart
// from src, the tile's first key) in a tile; keys at or past nvalid are
// zero-filled without a read.
__device__ __forceinline__ void stage_tile(__half* dst, const __half* src, int64_t tok_stride, int j0, int nvalid)
{
    const uint32_t d = (uint32_t)__cvta_generic_to_shared(dst);
#pragma unroll
    for (int i = threadIdx.x; i < kTileKeys * 16; i += kAttnThreads) {
        const int j = i >> 4, c = i & 15;
        const bool ok = j0 + j < nvalid;
        cp_async16(d + 2 * tile_off(j, c), ok ? src + (int64_t)j * tok_stride + c * 8 : src, ok ? 16 : 0);
    }
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t a, uint32_t (&r)[4])
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(a));
}

// c += A(16x16, row-major fragment) * B(16x8, column fragment b0, b1)
__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                 "{%0,%1,%2,%3};"
                 : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Two fp32 values as f16 pairs: x = hi + lo, hi = f16(x), lo = f16(x - hi);
// the first value in the low half of each word.
__device__ __forceinline__ void split2(float x0, float x1, uint32_t& hi, uint32_t& lo)
{
    const __half h0 = __float2half_rn(x0), h1 = __float2half_rn(x1);
    const __half l0 = __float2half_rn(__fsub_rn(x0, __half2float(h0)));
    const __half l1 = __float2half_rn(__fsub_rn(x1, __half2float(h1)));
    hi = (uint32_t)__half_as_ushort(h0) | ((uint32_t)__half_as_ushort(h1) << 16);
    lo = (uint32_t)__half_as_ushort(l0) | ((uint32_t)__half_as_ushort(l1) << 16);
}

__device__ unsigned int g_attn_wait_timeouts;

// Shared memory of a slot CTA (dynamic, the tiles 1024-byte aligned):
//   vt  the V tile, 128 keys x 128 dims f16 in the canonical 128-byte-swizzle
//       layout of an MN-major operand: [dim half][key][64 dims], 16-byte
//       piece p of key j's 128-byte row at p ^ (j & 7);
//   pt  the probabilities as the p.V MMA's B operand (K-major, 128-byte
//       swizzle): row n = (served row i, part hi/lo, head h) = 2 GQ i + GQ lo
//       + h, [key block of 64][n][64 keys], piece p of row n at p ^ (n & 7);
//   qf  q as mma.sync B fragments; p the chunk's fp32 scores/probabilities.
template <int GQ, int MRS>
struct AttnSlotLayout {
    static constexpr int MR = MRS;                                // rows served (at most)
    static constexpr int NP = ((MR * 2 * GQ + 15) / 16) * 16;     // N of the p.V MMA
    static constexpr int KEYS = kTileKeys;                        // key columns of pt (one 128-key chunk)
    static constexpr int VT = kTileKeys * kHeadDim * 2;
    static constexpr int PT = NP * KEYS * 2;
    static constexpr int QF = 8 * 32 * 16;
    static constexpr int PF = GQ * kPStride * 4;
    static constexpr int TCOLS = NP <= 32 ? 32 : (NP <= 64 ? 64 : 128);  // tensor-memory columns
    static constexpr int SMEM = 1024 + VT + PT + QF + PF + 16;
    static_assert(NP <= 256 && NP % 16 == 0, "N of a 128-row MMA");
};

// Byte offset of 16-byte piece c (dims 8c .. 8c + 7) of key j in the V tile.
__device__ __forceinline__ uint32_t vt_off(int j, int c)
{
    return (uint32_t)((c >> 3) * (kTileKeys * 128) + j * 128 + (((c & 7) ^ (j & 7)) << 4));
}

// Byte offset of key j in row n of the probability tile of NP rows.
__device__ __forceinline__ uint32_t pt_off(int NP, int n, int j)
{
    return (uint32_t)((j >> 6) * (NP * 128) + n * 128 + ((((j & 63) >> 3) ^ (n & 7)) << 4) + (j & 7) * 2);
}

// tcgen05 shared-memory matrix descriptor, 128-byte swizzle: start address,
// leading and stride byte offsets (>> 4), the fixed version bit.
__device__ __forceinline__ uint64_t umma_desc(uint32_t addr, uint32_t lbo, uint32_t sbo)
{
    return (uint64_t)((addr >> 4) & 0x3FFF) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | (1ull << 46) | (2ull << 61);
}

// D[128 dims][NP] (+)= Vt (A: MN-major, two 64-dim halves 16 KB apart, 8-key
// groups 1 KB apart) x P (B: K-major, 8-row groups 1 KB apart) over the 128
// keys of one tile; issued by one thread.
__device__ __forceinline__ void pv_mma(uint32_t tmem, uint32_t vt, uint32_t pt, int NP, int key_block0, bool accumulate)
{
    // kind::f16: D f32, A and B f16, A MN-major, B K-major, N = NP, M = 128
    const uint32_t idesc = (1u << 4) | (1u << 15) | ((uint32_t)(NP >> 3) << 17) | ((128u >> 4) << 24);
#pragma unroll
    for (int ks = 0; ks < kTileKeys / 16; ++ks) {
        const uint64_t a = umma_desc(vt + 2048 * ks, kTileKeys * 128, 1024);
        const uint64_t b = umma_desc(pt + (key_block0 + (ks >> 2)) * (NP * 128) + 32 * (ks & 3), 16, 1024);
        const uint32_t acc = (accumulate || ks > 0) ? 1u : 0u;
        asm volatile("{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
                     " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem),
                     "l"(a), "l"(b), "r"(idesc), "r"(acc));
    }
}

__device__ __forceinline__ void tc_commit(uint64_t* bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 16 columns of this warp's 32 tensor-memory lanes.
__device__ __forceinline__ void tmem_ld16(uint32_t addr, float (&v)[16])
{
    uint32_t r[16];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, "
                 "[%16];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                   "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
                   "=r"(r[15])
                 : "r"(addr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Stage keys [0, 128) of a 128-key chunk (rows tok_stride halves apart from
// src) in the slot kernel's V tile at shared address d (layout of vt_off);
// keys at or past nvalid are zero-filled without a read.
__device__ __forceinline__ void stage_tile_tc(uint32_t d, const __half* src, int64_t tok_stride, int nvalid)
{
#pragma unroll
    for (int i = threadIdx.x; i < kTileKeys * 16; i += kAttnThreads) {
        const int j = i >> 4, c = i & 15;
        const bool ok = j < nvalid;
        cp_async16(d + vt_off(j, c), ok ? src + (int64_t)j * tok_stride + c * 8 : src, ok ? 16 : 0);
    }
}

// The rows a chunk kernel serves: unit u is rows first[u] .. first[u] +
// count[u] - 1 (one cache) and owns the launch's chunk indices from
// chunk_begin[u] on.
struct AttnGroups {
    int first[16];
    int count[16];
    int chunk_begin[16];  // the group's first chunk index in the grid
    int n_groups;
};

// 4 CTAs per SM: a 4 x 2,051-key grid runs in one wave
template <int GQ>
__global__ void __launch_bounds__(kAttnThreads, 4)
attn_kernel(const float* __restrict__ q, int64_t ldq, AttnRows rows, AttnGroups units, int Hq, int Hkv, float scale,
            float* __restrict__ part)
{
    __shared__ __align__(128) AttnSmem<GQ> sm;
    pdl_trigger();
    const int g = blockIdx.y;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int gr = lane >> 2, tq = lane & 3;  // mma fragment: row group, thread in group
    const int mi = lane >> 3, mr = lane & 7;  // ldmatrix: the matrix and row this lane addresses

    // the row this CTA serves (one of the launch's single rows) and its chunk
    int ui = 0;
#pragma unroll 1
    for (int i = 1; i < units.n_groups; ++i)
        if ((int)blockIdx.x >= units.chunk_begin[i]) ui = i;
    const int r0 = units.first[ui], c = blockIdx.x - units.chunk_begin[ui];
    const AttnRow row = rows.row[r0];
    const int CH = row.chunk;
    const int key0 = c * CH;
    const int nvmax = min(CH, row.len - key0);                 // keys of the chunk
    const int ntile = (nvmax + kTileKeys - 1) / kTileKeys;     // tiles of this chunk: 1 or 2
    const int h0 = g * GQ;
    // the first key of tile t (keys key0 + 128t ..) of KV head g: tiles
    // never straddle a page, so within a tile keys are tok_stride apart
    auto tile_base = [&](const __half* base, int t) -> const __half* {
        const int key = key0 + kTileKeys * t;
        return row.pages ? base + (int64_t)__ldg(row.pages + (key >> 7)) * row.page_stride + g * row.head_stride
                         : base + g * row.head_stride + (int64_t)key * row.tok_stride;
    };
    const __half* kbase = tile_base(row.k, 0);
    const __half* vbase = tile_base(row.v, 0);
    if (tid == 0) {
        // stage the first tile's K and V rows in L2 while the previous kernel
        // ends (a cache hint only: the rows it writes are read after pdl_wait)
        const uint32_t span = (uint32_t)(((int64_t)(min(nvmax, kTileKeys) - 1) * row.tok_stride + kHeadDim) * 2);
        prefetch_l2(kbase, span);
        prefetch_l2(vbase, span);
    }
    pdl_wait();
    stage_tile(sm.vt, vbase, row.tok_stride, 0, nvmax);
    cp_async_commit();

    // K rows of keys j0 + 16w + gr (ka) and + 8 (kb): dims 32tq .. 32tq + 31,
    // read once with L1 bypassed: whole 32-byte sectors per load when the
    // row's rows start on 32-byte boundaries, else 16-byte loads
    const bool k32 = ((reinterpret_cast<uintptr_t>(kbase) | (uintptr_t)(row.tok_stride * 2)) & 31) == 0;
    uint32_t ka[16], kb[16];
    auto load_row = [&](const __half* p, bool ok, uint32_t (&w)[16]) {
        if (!ok) {
#pragma unroll
            for (int e = 0; e < 16; ++e) w[e] = 0u;
        } else if (k32) {
            ld_stream_v8(p, *reinterpret_cast<uint32_t(*)[8]>(&w[0]));
            ld_stream_v8(p + 16, *reinterpret_cast<uint32_t(*)[8]>(&w[8]));
        } else {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int4 v = ld_stream_v4(p + 8 * i);
                w[4 * i] = (uint32_t)v.x;
                w[4 * i + 1] = (uint32_t)v.y;
                w[4 * i + 2] = (uint32_t)v.z;
                w[4 * i + 3] = (uint32_t)v.w;
            }
        }
    };
    auto load_k = [&](const __half* kt, int j0) {
        const int ja = j0 + 16 * warp + gr, jb = ja + 8;
        load_row(kt + (int64_t)(ja - j0) * row.tok_stride + 32 * tq, ja < nvmax, ka);
        load_row(kt + (int64_t)(jb - j0) * row.tok_stride + 32 * tq, jb < nvmax, kb);
    };
    load_k(kbase, 0);
    // this thread's q slice for the B fragments: step s = warp, lane (head
    // n = lane / 4, t = lane % 4) holds q[n][32t + 4s .. 32t + 4s + 3] (heads
    // past the group are zero), loaded with the first K/V rows
    float4 qv = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    if ((lane >> 2) < GQ)
        qv = *reinterpret_cast<const float4*>(q + (size_t)r0 * ldq + (size_t)(h0 + (lane >> 2)) * kHeadDim +
                                              32 * (lane & 3) + 4 * warp);
    const int r = r0, nvalid = nvmax;

    // q as B fragments (hi, lo)
    {
        uint4 f;
        split2(qv.x, qv.y, f.x, f.z);
        split2(qv.z, qv.w, f.y, f.w);
        sm.qf[warp][lane] = f;
    }
    __syncthreads();

    // ---- scores of keys j0 + 16w .. j0 + 16w + 15
    auto scores = [&](int j0) {
        float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
        for (int s = 0; s < 8; ++s) {
            const uint32_t a[4] = {ka[2 * s], kb[2 * s], ka[2 * s + 1], kb[2 * s + 1]};
            const uint4 f = sm.qf[s][lane];
            mma16816(acc, a, f.x, f.y);
            mma16816(acc, a, f.z, f.w);
        }
        // acc: keys ja (c0, c1) and ja + 8 (c2, c3); heads 2tq (c0, c2) and 2tq + 1
        const int ja = j0 + 16 * warp + gr, jb = ja + 8, h = 2 * tq;
        if (h < GQ) {
            sm.p[h][ja] = ja < nvalid ? __fmul_rn(acc[0], scale) : -INFINITY;
            sm.p[h][jb] = jb < nvalid ? __fmul_rn(acc[2], scale) : -INFINITY;
        }
        if (h + 1 < GQ) {
            sm.p[h + 1][ja] = ja < nvalid ? __fmul_rn(acc[1], scale) : -INFINITY;
            sm.p[h + 1][jb] = jb < nvalid ? __fmul_rn(acc[3], scale) : -INFINITY;
        }
    };
    scores(0);
    if (ntile == 2) {  // a 256-key chunk
        load_k(tile_base(row.k, 1), kTileKeys);
        scores(kTileKeys);
    }
    __syncthreads();

    // ---- chunk softmax statistics, warp h per head
    float* pout = part + ((size_t)(rows.row[r].chunk0 + c) * Hq + h0) * kPartStride;
    for (int h = warp; h < GQ; h += 8) {
        float sv[kAttnChunk / 32];
        float m = -INFINITY;
#pragma unroll
        for (int i = 0; i < kAttnChunk / 32; ++i) {
            const int j = lane + 32 * i;
            sv[i] = (32 * i < CH && j < nvalid) ? sm.p[h][j] : -INFINITY;
            m = fmaxf(m, sv[i]);
        }
        m = warp_max(m);
        float l = 0.0f;
#pragma unroll
        for (int i = 0; i < kAttnChunk / 32; ++i) {
            const int j = lane + 32 * i;
            if (32 * i < CH) {
                const float p = j < nvalid ? expf(__fsub_rn(sv[i], m)) : 0.0f;
                sm.p[h][j] = p;
                l = __fadd_rn(l, p);
            }
        }
        l = warp_sum_butterfly(l);
        if (lane == 0) {
            pout[(size_t)h * kPartStride + 128] = m;
            pout[(size_t)h * kPartStride + 129] = l;
        }
    }
    cp_async_wait_all();
    __syncthreads();

    // ---- p . V for dims 16w .. 16w + 15, 16 keys per step: D[dim][head]
    // += V^T (A: the tile's rows read transposed) times P^T (B: the
    // probabilities of heads gr, split hi + lo)
    float o[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    const uint32_t vt = (uint32_t)__cvta_generic_to_shared(sm.vt);
    auto values = [&](int j0) {
#pragma unroll 2
        for (int ks = 0; ks < kTileKeys / 16; ++ks) {
            float2 x = make_float2(0.0f, 0.0f), y = make_float2(0.0f, 0.0f);
            if (gr < GQ) {
                x = *reinterpret_cast<const float2*>(&sm.p[gr][j0 + 16 * ks + 2 * tq]);
                y = *reinterpret_cast<const float2*>(&sm.p[gr][j0 + 16 * ks + 2 * tq + 8]);
            }
            uint32_t bh0, bl0, bh1, bl1;
            split2(x.x, x.y, bh0, bl0);
            split2(y.x, y.y, bh1, bl1);
            uint32_t a[4];  // (keys 0-7 | 8-15 of the step) x (dims 0-7 | 8-15 of the warp)
            ldsm_x4_trans(vt + 2 * tile_off(16 * ks + 8 * (mi >> 1) + mr, 2 * warp + (mi & 1)), a);
            mma16816(o, a, bh0, bh1);
            mma16816(o, a, bl0, bl1);
        }
    };
    values(0);
    if (ntile == 2) {
        __syncthreads();  // every warp is done with the first V tile
        stage_tile(sm.vt, tile_base(row.v, 1), row.tok_stride, kTileKeys, nvalid);
        cp_async_commit();
        cp_async_wait_all();
        __syncthreads();
        values(kTileKeys);
    }
    // o: dims 16w + gr (o0, o1) and 16w + gr + 8 (o2, o3); heads 2tq (o0, o2) and 2tq + 1
    const int d = 16 * warp + gr, h = 2 * tq;
    if (h < GQ) {
        pout[(size_t)h * kPartStride + d] = o[0];
        pout[(size_t)h * kPartStride + d + 8] = o[2];
    }
    if (h + 1 < GQ) {
        pout[(size_t)(h + 1) * kPartStride + d] = o[1];
        pout[(size_t)(h + 1) * kPartStride + d + 8] = o[3];
    }
}

// The slot form: one CTA per (row group, 128-key chunk, KV head) serves the
// group's rows (a slot's verify rows, one cache); scores and softmax per row
// as in attn_kernel, then p . V of all of them in one tcgen05.mma pass:
// D[dim][n] = sum over the chunk's keys of V[key][dim] P[n][key] with A = the
// V tile (MN-major), B = the probability tile (K-major), D in tensor memory
// (lane = dim, column = n), and out[row][head][dim] = D[.][hi] + D[.][lo].
// Each output column depends on its own probability row only, so a row gives
// the bits it gives alone in this form.  4 CTAs per SM.
template <int GQ, int MRS>
__global__ void __launch_bounds__(kAttnThreads, 4)
attn_slot_kernel(const float* __restrict__ q, int64_t ldq, AttnRows rows, AttnGroups groups, int Hq, int Hkv,
                 float scale, float* __restrict__ part)
{
    using LA = AttnSlotLayout<GQ, MRS>;
    extern __shared__ uint8_t attn_smem[];
    uint8_t* base = attn_smem + ((1024u - (smem_addr(attn_smem) & 1023u)) & 1023u);
    const uint32_t s_vt = smem_addr(base), s_pt = s_vt + LA::VT;
    uint8_t* pt = base + LA::VT;
    uint4 (*qf)[32] = reinterpret_cast<uint4 (*)[32]>(base + LA::VT + LA::PT);
    float (*sp)[kPStride] = reinterpret_cast<float (*)[kPStride]>(base + LA::VT + LA::PT + LA::QF);
    __shared__ uint64_t mbar;     // the p.V MMAs' completion
    __shared__ uint32_t tmem_at;  // the tensor-memory columns of D
    pdl_trigger();
    const int g = blockIdx.y;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int gr = lane >> 2, tq = lane & 3;  // mma fragment: row group, thread in group
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(&tmem_at)),
                     "r"((uint32_t)LA::TCOLS));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    if (tid == 0) {
        mbar_init(&mbar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    // probability rows no served row writes stay zero
    for (int i = tid; i < LA::PT / 16; i += kAttnThreads) reinterpret_cast<uint4*>(pt)[i] = make_uint4(0u, 0u, 0u, 0u);

    // the rows this CTA serves: r0 .. r0 + R - 1, sharing row r0's cache
    int gi = 0;
#pragma unroll 1
    for (int i = 1; i < groups.n_groups; ++i)
        if ((int)blockIdx.x >= groups.chunk_begin[i]) gi = i;
    const int r0 = groups.first[gi], R = groups.count[gi], c = blockIdx.x - groups.chunk_begin[gi];
    const AttnRow row = rows.row[r0];
    const int CH = row.chunk;
    const int key0 = c * CH;
    int len_max = row.len;
    for (int i = 1; i < R; ++i) len_max = max(len_max, rows.row[r0 + i].len);
    const int nvmax = min(CH, len_max - key0);  // keys of the chunk any row sees (CH = 128: one tile)
    const int h0 = g * GQ;
    // the first key of tile t (keys key0 + 128t ..) of KV head g: tiles
    // never straddle a page, so within a tile keys are tok_stride apart
    auto tile_base = [&](const __half* base, int t) -> const __half* {
        const int key = key0 + kTileKeys * t;
        return row.pages ? base + (int64_t)__ldg(row.pages + (key >> 7)) * row.page_stride + g * row.head_stride
                         : base + g * row.head_stride + (int64_t)key * row.tok_stride;
    };
    const __half* kbase = tile_base(row.k, 0);
    const __half* vbase = tile_base(row.v, 0);
    if (tid == 0) {
        // stage the first tile's K and V rows in L2 while the previous kernel
        // ends (a cache hint only: the rows it writes are read after pdl_wait)
        const uint32_t span = (uint32_t)(((int64_t)(min(nvmax, kTileKeys) - 1) * row.tok_stride + kHeadDim) * 2);
        prefetch_l2(kbase, span);
        prefetch_l2(vbase, span);
    }
    pdl_wait();
    stage_tile_tc(s_vt, vbase, row.tok_stride, nvmax);
    cp_async_commit();
    tc_fence_before();
    __syncthreads();  // the tensor-memory address, the barrier and the zeroed rows are in place
    tc_fence_after();
    const uint32_t tmem = tmem_at;

    // K rows of keys j0 + 16w + gr (ka) and + 8 (kb): dims 32tq .. 32tq + 31,
    // read once with L1 bypassed: whole 32-byte sectors per load when the
    // row's rows start on 32-byte boundaries, else 16-byte loads
    const bool k32 = ((reinterpret_cast<uintptr_t>(kbase) | (uintptr_t)(row.tok_stride * 2)) & 31) == 0;
    uint32_t ka[16], kb[16];
    auto load_row = [&](const __half* p, bool ok, uint32_t (&w)[16]) {
        if (!ok) {
#pragma unroll
            for (int e = 0; e < 16; ++e) w[e] = 0u;
        } else if (k32) {
            ld_stream_v8(p, *reinterpret_cast<uint32_t(*)[8]>(&w[0]));
            ld_stream_v8(p + 16, *reinterpret_cast<uint32_t(*)[8]>(&w[8]));
        } else {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int4 v = ld_stream_v4(p + 8 * i);
                w[4 * i] = (uint32_t)v.x;
                w[4 * i + 1] = (uint32_t)v.y;
                w[4 * i + 2] = (uint32_t)v.z;
                w[4 * i + 3] = (uint32_t)v.w;
            }
        }
    };
    auto load_k = [&](const __half* kt, int j0) {
        const int ja = j0 + 16 * warp + gr, jb = ja + 8;
        load_row(kt + (int64_t)(ja - j0) * row.tok_stride + 32 * tq, ja < nvmax, ka);
        load_row(kt + (int64_t)(jb - j0) * row.tok_stride + 32 * tq, jb < nvmax, kb);
    };
    load_k(kbase, 0);
    // every row's q slice this thread turns into B fragments: step s = warp,
    // lane (head n = lane / 4, t = lane % 4) holds q[n][32t + 4s .. 32t + 4s + 3]
    // (heads past the group are zero), loaded with the first K/V rows
    constexpr int MR = MRS;
    float4 qv[MR];
    {
        const int n = lane >> 2, t = lane & 3;
#pragma unroll
        for (int ri = 0; ri < MR; ++ri) {
            qv[ri] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            if (ri < R && n < GQ)
                qv[ri] = *reinterpret_cast<const float4*>(q + (size_t)(r0 + ri) * ldq + (size_t)(h0 + n) * kHeadDim +
                                                          32 * t + 4 * warp);
        }
    }

#pragma unroll
    for (int ri = 0; ri < MR; ++ri) {
        if (ri >= R) break;
        const int r = r0 + ri;
        const int len = rows.row[r].len;
        if (key0 >= len) continue;  // this row's keys end before the chunk (the same for every thread)
        const int nvalid = min(CH, len - key0);
        if (ri > 0) __syncthreads();  // the previous row is done with the q fragments and probabilities

        // q as B fragments (hi, lo)
        {
            uint4 f;
            split2(qv[ri].x, qv[ri].y, f.x, f.z);
            split2(qv[ri].z, qv[ri].w, f.y, f.w);
            qf[warp][lane] = f;
        }
        __syncthreads();

        // ---- scores of keys j0 + 16w .. j0 + 16w + 15
        auto scores = [&](int j0) {
            float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
            for (int s = 0; s < 8; ++s) {
                const uint32_t a[4] = {ka[2 * s], kb[2 * s], ka[2 * s + 1], kb[2 * s + 1]};
                const uint4 f = qf[s][lane];
                mma16816(acc, a, f.x, f.y);
                mma16816(acc, a, f.z, f.w);
            }
            // acc: keys ja (c0, c1) and ja + 8 (c2, c3); heads 2tq (c0, c2) and 2tq + 1
            const int ja = j0 + 16 * warp + gr, jb = ja + 8, h = 2 * tq;
            if (h < GQ) {
                sp[h][ja] = ja < nvalid ? __fmul_rn(acc[0], scale) : -INFINITY;
                sp[h][jb] = jb < nvalid ? __fmul_rn(acc[2], scale) : -INFINITY;
            }
            if (h + 1 < GQ) {
                sp[h + 1][ja] = ja < nvalid ? __fmul_rn(acc[1], scale) : -INFINITY;
                sp[h + 1][jb] = jb < nvalid ? __fmul_rn(acc[3], scale) : -INFINITY;
            }
        };
        scores(0);
        __syncthreads();

        // ---- chunk softmax statistics, warp h per head; the probabilities,
        // split hi + lo as for q, go to rows 2 GQ ri + h (hi) and
        // 2 GQ ri + GQ + h (lo) of the p.V MMA's B tile
        float* pout = part + ((size_t)(rows.row[r].chunk0 + c) * Hq + h0) * kPartStride;
        for (int h = warp; h < GQ; h += 8) {
            float sv[kAttnChunk / 32];
            float m = -INFINITY;
#pragma unroll
            for (int i = 0; i < kAttnChunk / 32; ++i) {
                const int j = lane + 32 * i;
                sv[i] = (32 * i < CH && j < nvalid) ? sp[h][j] : -INFINITY;
                m = fmaxf(m, sv[i]);
            }
            m = warp_max(m);
            float l = 0.0f;
            const int nhi = 2 * GQ * ri + h, nlo = nhi + GQ;
#pragma unroll
            for (int i = 0; i < kAttnChunk / 32; ++i) {
                const int j = lane + 32 * i;
                if (32 * i < CH && 32 * i < LA::KEYS) {  // (the launch gives the tile CH key columns)
                    const float p = j < nvalid ? expf(__fsub_rn(sv[i], m)) : 0.0f;
                    l = __fadd_rn(l, p);
                    const __half ph = __float2half_rn(p);
                    *reinterpret_cast<__half*>(pt + pt_off(LA::NP, nhi, j)) = ph;
                    *reinterpret_cast<__half*>(pt + pt_off(LA::NP, nlo, j)) =
                        __float2half_rn(__fsub_rn(p, __half2float(ph)));
                }
            }
            l = warp_sum_butterfly(l);
            if (lane == 0) {
                pout[(size_t)h * kPartStride + 128] = m;
                pout[(size_t)h * kPartStride + 129] = l;
            }
        }
    }

    // ---- p . V of every served row at once on the tensor cores:
    // D[dim][n] = sum over the chunk's 128 keys of V[key][dim] P[n][key],
    // in tensor memory (lane = dim, column = n); one thread issues the MMAs
    cp_async_wait_all();
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // V tile and probabilities: visible to the MMAs
    __syncthreads();
    tc_fence_after();
    if (tid == 0) {
        pv_mma(tmem, s_vt, s_pt, LA::NP, 0, false);
        tc_commit(&mbar);
    }
    bool ok = mbar_wait(&mbar, 0, &g_attn_wait_timeouts);
    ok = __syncthreads_and(ok);  // one expired wait and no warp reads the accumulator
    tc_fence_after();

    // ---- the partial outputs: warp w < 4 reads dims 32w .. 32w + 31 (its
    // lanes of tensor memory); out = hi part + lo part
    if (ok && warp < 4) {
        float o[LA::MR][GQ];
#pragma unroll
        for (int k = 0; k < LA::NP / 16; ++k) {
            float v[16];
            tmem_ld16(tmem + ((uint32_t)(32 * warp) << 16) + 16 * k, v);
#pragma unroll
            for (int ri = 0; ri < LA::MR; ++ri)
#pragma unroll
                for (int h = 0; h < GQ; ++h) {
                    const int chi = 2 * GQ * ri + h, clo = chi + GQ;
                    if (chi >= 16 * k && chi < 16 * k + 16) o[ri][h] = v[chi - 16 * k];
                    if (clo >= 16 * k && clo < 16 * k + 16) o[ri][h] = __fadd_rn(o[ri][h], v[clo - 16 * k]);
                }
        }
        const int d = 32 * warp + lane;
#pragma unroll
        for (int ri = 0; ri < LA::MR; ++ri) {
            if (ri >= R) break;
            const AttnRow& rr = rows.row[r0 + ri];
            if (key0 >= rr.len) continue;
            float* pout = part + ((size_t)(rr.chunk0 + c) * Hq + h0) * kPartStride;
#pragma unroll
            for (int h = 0; h < GQ; ++h) pout[(size_t)h * kPartStride + d] = o[ri][h];
        }
    }
    // after an expired wait the MMAs may still be writing the accumulator:
    // wait once more (bounded) before its tensor memory is freed
    if (!ok && tid == 0) mbar_wait(&mbar, 0, &g_attn_wait_timeouts);
    tc_fence_before();
    __syncthreads();  // every read of the accumulator is done
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"((uint32_t)LA::TCOLS));
}

// Merge of one (row, query head h) over the row's chunks, one thread per dim
// d (CTA of 128), after the chunk kernel has completed:
//   M = max_c m_c, w_c = e^(m_c - M), L = sum_c l_c w_c, O_d = sum_c o_c,d w_c,
//   out_d = O_d / L;  L lane-serial over c = lane + 32i then a butterfly, O_d
//   sequential over c; optionally q8_0 blocks of out (one warp per block).
__global__ void __launch_bounds__(kHeadDim)
attn_merge_kernel(AttnRows rows, int Hq, const float* __restrict__ part, float* __restrict__ out, int64_t ldo,
                  int8_t* __restrict__ out_q, float* __restrict__ out_d)
{
    __shared__ float wts[kAttnMaxChunksPerRow];
    __shared__ float lsum[kAttnMaxChunksPerRow];
    __shared__ float Lsh;
    pdl_trigger();
    const int h = blockIdx.x, r = blockIdx.y;
    const int d = threadIdx.x, lane = d & 31;
    const AttnRow row = rows.row[r];
    const int nch = (row.len + row.chunk - 1) / row.chunk;
    const size_t cstride = (size_t)Hq * kPartStride;
    const float* bh = part + ((size_t)row.chunk0 * Hq + h) * kPartStride;
    pdl_wait();
    constexpr int kPre = 32;  // chunk outputs loaded while the statistics are gathered
    float ov[kPre];
#pragma unroll
    for (int u = 0; u < kPre; ++u) ov[u] = u < nch ? __ldcg(bh + u * cstride + d) : 0.0f;
    if (d < 32) {
        // every chunk's (m, l) up to 128 chunks requested at once (one L2 round
        // trip), then the rest; the maximum is order-free
        constexpr int kStatPre = 4;
        float mp[kStatPre], lp[kStatPre];
#pragma unroll
        for (int i = 0; i < kStatPre; ++i) {
            const int cc = lane + 32 * i;
            mp[i] = cc < nch ? __ldcg(bh + cc * cstride + 128) : -INFINITY;
            lp[i] = cc < nch ? __ldcg(bh + cc * cstride + 129) : 0.0f;
        }
        float M = -INFINITY;
#pragma unroll
        for (int i = 0; i < kStatPre; ++i) {
            const int cc = lane + 32 * i;
            if (cc < nch) {
                wts[cc] = mp[i];
                lsum[cc] = lp[i];
                M = fmaxf(M, mp[i]);
            }
        }
        for (int cc = lane + 32 * kStatPre; cc < nch; cc += 32) {
            const float m = __ldcg(bh + cc * cstride + 128);
            wts[cc] = m;
            lsum[cc] = __ldcg(bh + cc * cstride + 129);
            M = fmaxf(M, m);
        }
        M = warp_max(M);
        float L = 0.0f;
        for (int cc = lane; cc < nch; cc += 32) {
            const float w = expf(__fsub_rn(wts[cc], M));
            wts[cc] = w;
            L = __fmaf_rn(lsum[cc], w, L);
        }
        L = warp_sum_butterfly(L);
        if (lane == 0) Lsh = L;
    }
    __syncthreads();
    float O = 0.0f;
#pragma unroll
    for (int u = 0; u < kPre; ++u)
        if (u < nch) O = __fmaf_rn(ov[u], wts[u], O);
    int cc = kPre;
    for (; cc + 32 <= nch; cc += 32) {
        float ob[32];
#pragma unroll
        for (int u = 0; u < 32; ++u) ob[u] = __ldcg(bh + (cc + u) * cstride + d);
#pragma unroll
        for (int u = 0; u < 32; ++u) O = __fmaf_rn(ob[u], wts[cc + u], O);
    }
    for (; cc + 16 <= nch; cc += 16) {
        float ob[16];
#pragma unroll
        for (int u = 0; u < 16; ++u) ob[u] = __ldcg(bh + (cc + u) * cstride + d);
#pragma unroll
        for (int u = 0; u < 16; ++u) O = __fmaf_rn(ob[u], wts[cc + u], O);
    }
    for (; cc < nch; ++cc) O = __fmaf_rn(__ldcg(bh + cc * cstride + d), wts[cc], O);
    const float val = __fdiv_rn(O, Lsh);
    const size_t oi = (size_t)r * ldo + (size_t)h * kHeadDim + d;
    out[oi] = val;
    if (out_q) {
        float dd;
        const int code = q8_quantize_lane(val, &dd);
        out_q[oi] = (int8_t)code;
        if (lane == 0) out_d[oi / 32] = dd;
    }
}

template <int GQ>
static cudaError_t launch_g(const float* q, int64_t ldq, const AttnRows& rows, int Hq, int Hkv, float scale,
                            float* part, float* out, int64_t ldo, int8_t* out_q, float* out_d, cudaStream_t s)
{
    // A row's form follows its own key count only: rows with 128-key chunks
    // (up to 16,384 keys) take attn_slot_kernel, consecutive ones on one
    // cache (a slot's verify rows, at most kAttnMaxGroupRows) served together
    // by one CTA per (chunk, KV head), a single one by the one-row
    // instantiation, which gives the same bits per row; rows past 16,384 keys
    // (256-key chunks) take attn_kernel, one CTA per row chunk.  A launch with
    // several kinds runs each kernel (each behind the previous one), then the
    // merge.
    AttnGroups multi{}, one{}, wide{};
    int cm = 0, co = 0, cw = 0;
    for (int r = 0; r < rows.n_rows;) {
        const AttnRow& a = rows.row[r];
        int cnt = 1, len_max = a.len;
        while (r + cnt < rows.n_rows && cnt < kAttnMaxGroupRows) {
            const AttnRow& b = rows.row[r + cnt];
            if (b.k != a.k || b.v != a.v || b.head_stride != a.head_stride || b.tok_stride != a.tok_stride ||
                b.pages != a.pages || b.page_stride != a.page_stride || a.chunk != kTileKeys || b.chunk != kTileKeys)
                break;
            len_max = max(len_max, b.len);
            ++cnt;
        }
        AttnGroups& u = cnt > 1 ? multi : (a.chunk == kTileKeys ? one : wide);
        int& chunks = cnt > 1 ? cm : (a.chunk == kTileKeys ? co : cw);
        u.first[u.n_groups] = r;
        u.count[u.n_groups] = cnt;
        u.chunk_begin[u.n_groups] = chunks;
        ++u.n_groups;
        chunks += (len_max + a.chunk - 1) / a.chunk;
        r += cnt;
    }
    cudaError_t e = cudaSuccess;
    if (wide.n_groups > 0) {
        e = launch_pdl(attn_kernel<GQ>, dim3(cw, Hkv), dim3(kAttnThreads), s, q, ldq, rows, wide, Hq, Hkv, scale,
                       part);
        count_launches(1);
        if (e != cudaSuccess) return e;
    }
    if (one.n_groups > 0) {
        static std::atomic<bool> done[kMaxDevices];
        e = set_smem_once(attn_slot_kernel<GQ, 1>, AttnSlotLayout<GQ, 1>::SMEM, done);
        if (e == cudaSuccess)
            e = launch_pdl_smem(attn_slot_kernel<GQ, 1>, dim3(co, Hkv), dim3(kAttnThreads),
                                AttnSlotLayout<GQ, 1>::SMEM, s, q, ldq, rows, one, Hq, Hkv, scale, part);
        count_launches(1);
        if (e != cudaSuccess) return e;
    }
    if (multi.n_groups > 0) {
        static std::atomic<bool> done[kMaxDevices];
        e = set_smem_once(attn_slot_kernel<GQ, kAttnMaxGroupRows>, AttnSlotLayout<GQ, kAttnMaxGroupRows>::SMEM, done);
        if (e == cudaSuccess)
            e = launch_pdl_smem(attn_slot_kernel<GQ, kAttnMaxGroupRows>, dim3(cm, Hkv), dim3(kAttnThreads),
                                AttnSlotLayout<GQ, kAttnMaxGroupRows>::SMEM, s, q, ldq, rows, multi, Hq, Hkv, scale,
                                part);
        count_launches(1);
        if (e != cudaSuccess) return e;
    }
    e = launch_pdl(attn_merge_kernel, dim3(Hq, rows.n_rows), dim3(kHeadDim), s, rows, Hq, (const float*)part, out,
                   ldo, out_q, out_d);
    count_launches(1);
    return e;
}

cudaError_t launch_attention(const float* q, int64_t ldq, const AttnRows& rows, int Hq, int Hkv, float scale,
                             float* part, float* out, int64_t ldo, int8_t* out_q, float* out_d, cudaStream_t s)
{
    switch (Hq / Hkv) {
#define LUCE_AT(G) \
    case G: return launch_g<G>(q, ldq, rows, Hq, Hkv, scale, part, out, ldo, out_q, out_d, s);
        LUCE_AT(1)
        LUCE_AT(2)
        LUCE_AT(3)
        LUCE_AT(4)
        LUCE_AT(5)
        LUCE_AT(6)
        LUCE_AT(7)
        LUCE_AT(8)
#undef LUCE_AT
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t read_attn_wait_timeouts(uint32_t* count, bool reset)
{
    cudaError_t e = cudaMemcpyFromSymbol(count, g_attn_wait_timeouts, sizeof(uint32_t));
    if (e == cudaSuccess && reset) {
        const uint32_t zero = 0;
        e = cudaMemcpyToSymbol(g_attn_wait_timeouts, &zero, sizeof(uint32_t));
    }
    return e;
}

}  // namespace luce
