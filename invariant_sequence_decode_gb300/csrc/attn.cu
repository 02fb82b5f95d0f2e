// attn.cu - multi-sequence GQA decode attention, split-K over each row's own
// f16 cache with an exact, ordered log-sum-exp merge.
//
// "antirez/ds4 pull 604", Commit walkthrough: one query token per sequence,
// each attending to its own cache, per-sequence views passed by value (max 4);
// section 2: one multi-sequence attention launch with no position limit.
//
// A row's keys are cut into chunks of CH keys, CH = attn_chunk_keys(row's key
// count) (128 up to 16,384 keys, else 256: small contexts get smaller chunks
// so the GPU has enough independent work).  One CTA of 256 threads per (row, chunk, KV
// head g) serves all Hq/Hkv query heads of g, so each K/V byte is read once:
//   scores   P = 512/CH threads per key pair (j, j + CH/2); thread part p
//            covers dims [p*128/P, (p+1)*128/P) of both keys: fma over its
//            dims ascending, then the P partial dots of a key are summed by an
//            xor butterfly (1, 2, ...); s_h = scale * dot;
//   softmax  warp h owns head h: m = max_j s_h, p_j = exp(s_h - m),
//            l = sum p_j (lane-serial over j = lane + 32i, then butterfly);
//   values   warp w owns keys w, w+8, ... and lane l dims 4l..4l+3:
//            o_h += p_hj * v_j (fma, keys ascending); the 8 warp partials are
//            added in warp order.
//   -> scratch (o_h[128], m_h, l_h) for the chunk.
// The CTA that finishes last for its (row, g) (an atomic ticket; nobody
// waits) merges the row's chunks in chunk order:
//   M = max_c m_c, w_c = e^(m_c - M), L = sum_c l_c w_c, O = sum_c o_c w_c,
//   out = O / L  (the sums sequential over c),
// and optionally quantizes out to q8_0 blocks (the Wo projection's input).
// Every chunking and reduction order depends only on the row's own key
// count, never on the other rows, on which CTA merges or on the grid.
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace luce {

constexpr int kPartStride = 132;  // o[128], m, l, 2 pad floats per (chunk, head)

size_t attn_part_floats(int total_chunks, int Hq) { return (size_t)total_chunks * Hq * kPartStride; }

int attn_chunk_keys(int len) { return len <= 16384 ? 128 : 256; }

// q row of head h in shared memory: dim d at qpad(d) = d + 4*(d/32), so the
// up-to-4 threads of a key (dims 32 apart) hit different banks and four
// consecutive dims are one aligned 16-byte load.
constexpr int kQStride = kHeadDim + 16;
__device__ __forceinline__ int qpad(int d) { return d + 4 * (d >> 5); }

template <int GQ>
struct AttnSmem {
    float q[GQ][kQStride];
    float p[GQ][kAttnChunk];
    float red[8][GQ][kHeadDim];  // also the merge's scratch
    int last;
};

// Scores, softmax statistics and p.V of one chunk of CH keys.
template <int GQ, int CH>
__device__ __forceinline__ void attn_chunk(AttnSmem<GQ>& sm, const __half* kbase, const __half* vbase,
                                           int64_t tok_stride, int nvalid, float scale, float* pout)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    // ---- scores: each thread computes 2 keys (j, j + CH/2) over DPT dims, so
    // every q load from shared memory serves 8 fma
    {
        constexpr int PARTS = 512 / CH;       // threads per key pair
        constexpr int DPT2 = kHeadDim / PARTS;
        const int j = tid / PARTS, part = tid % PARTS;
        float dot0[GQ], dot1[GQ];
#pragma unroll
        for (int h = 0; h < GQ; ++h) dot0[h] = dot1[h] = 0.0f;
        const bool v0 = j < nvalid, v1 = j + CH / 2 < nvalid;
        const int4* kp0 = reinterpret_cast<const int4*>(kbase + (int64_t)j * tok_stride + part * DPT2);
        const int4* kp1 = reinterpret_cast<const int4*>(kbase + (int64_t)(j + CH / 2) * tok_stride + part * DPT2);
        int4 ka[DPT2 / 8], kc[DPT2 / 8];
#pragma unroll
        for (int i = 0; i < DPT2 / 8; ++i) {
            ka[i] = v0 ? __ldg(kp0 + i) : make_int4(0, 0, 0, 0);
            kc[i] = v1 ? __ldg(kp1 + i) : make_int4(0, 0, 0, 0);
        }
#pragma unroll
        for (int i = 0; i < DPT2 / 8; ++i) {
            const __half2* ha = reinterpret_cast<const __half2*>(&ka[i]);
            const __half2* hc = reinterpret_cast<const __half2*>(&kc[i]);
#pragma unroll
            for (int e = 0; e < 4; e += 2) {
                const float2 a01 = __half22float2(ha[e]), a23 = __half22float2(ha[e + 1]);
                const float2 c01 = __half22float2(hc[e]), c23 = __half22float2(hc[e + 1]);
                const int dq = qpad(part * DPT2 + i * 8 + e * 2);
#pragma unroll
                for (int h = 0; h < GQ; ++h) {
                    const float4 qv = *reinterpret_cast<const float4*>(&sm.q[h][dq]);
                    dot0[h] = __fmaf_rn(qv.x, a01.x, dot0[h]);
                    dot0[h] = __fmaf_rn(qv.y, a01.y, dot0[h]);
                    dot0[h] = __fmaf_rn(qv.z, a23.x, dot0[h]);
                    dot0[h] = __fmaf_rn(qv.w, a23.y, dot0[h]);
                    dot1[h] = __fmaf_rn(qv.x, c01.x, dot1[h]);
                    dot1[h] = __fmaf_rn(qv.y, c01.y, dot1[h]);
                    dot1[h] = __fmaf_rn(qv.z, c23.x, dot1[h]);
                    dot1[h] = __fmaf_rn(qv.w, c23.y, dot1[h]);
                }
            }
        }
#pragma unroll
        for (int h = 0; h < GQ; ++h) {
#pragma unroll
            for (int off = 1; off < PARTS; off <<= 1) {
                dot0[h] = __fadd_rn(dot0[h], __shfl_xor_sync(0xffffffffu, dot0[h], off));
                dot1[h] = __fadd_rn(dot1[h], __shfl_xor_sync(0xffffffffu, dot1[h], off));
            }
        }
        if (part == 0) {
#pragma unroll
            for (int h = 0; h < GQ; ++h) {
                sm.p[h][j] = v0 ? __fmul_rn(dot0[h], scale) : -INFINITY;
                sm.p[h][j + CH / 2] = v1 ? __fmul_rn(dot1[h], scale) : -INFINITY;
            }
        }
    }
    __syncthreads();

    // ---- chunk softmax statistics, warp h per head
    for (int h = warp; h < GQ; h += 8) {
        float sv[CH / 32];
        float m = -INFINITY;
#pragma unroll
        for (int i = 0; i < CH / 32; ++i) {
            sv[i] = sm.p[h][lane + 32 * i];
            m = fmaxf(m, sv[i]);
        }
        m = warp_max(m);
        float l = 0.0f;
#pragma unroll
        for (int i = 0; i < CH / 32; ++i) {
            const int j = lane + 32 * i;
            const float p = (j < nvalid) ? expf(__fsub_rn(sv[i], m)) : 0.0f;
            sm.p[h][j] = p;
            l = __fadd_rn(l, p);
        }
        l = warp_sum_butterfly(l);
        if (lane == 0) {
            pout[(size_t)h * kPartStride + 128] = m;
            pout[(size_t)h * kPartStride + 129] = l;
        }
    }
    __syncthreads();

    // ---- p . V  (keys w, w+8, ...; all of this warp's loads issued first)
    {
        float o[GQ][4];
#pragma unroll
        for (int h = 0; h < GQ; ++h)
#pragma unroll
            for (int e = 0; e < 4; ++e) o[h][e] = 0.0f;
        const __half* vl = vbase + lane * 4;
        constexpr int KPW = CH / 8;  // keys per warp
        constexpr int UB = KPW < 8 ? KPW : 8;
#pragma unroll 1
        for (int u0 = 0; u0 < KPW; u0 += UB) {
            uint2 raw[UB];
#pragma unroll
            for (int u = 0; u < UB; ++u) {
                const int j = warp + 8 * (u0 + u);
                if (j < nvalid) raw[u] = __ldg(reinterpret_cast<const uint2*>(vl + (int64_t)j * tok_stride));
            }
#pragma unroll
            for (int u = 0; u < UB; ++u) {
                const int j = warp + 8 * (u0 + u);
                if (j < nvalid) {
                    const float2 v01 = __half22float2(*reinterpret_cast<const __half2*>(&raw[u].x));
                    const float2 v23 = __half22float2(*reinterpret_cast<const __half2*>(&raw[u].y));
#pragma unroll
                    for (int h = 0; h < GQ; ++h) {
                        const float p = sm.p[h][j];
                        o[h][0] = __fmaf_rn(p, v01.x, o[h][0]);
                        o[h][1] = __fmaf_rn(p, v01.y, o[h][1]);
                        o[h][2] = __fmaf_rn(p, v23.x, o[h][2]);
                        o[h][3] = __fmaf_rn(p, v23.y, o[h][3]);
                    }
                }
            }
        }
#pragma unroll
        for (int h = 0; h < GQ; ++h)
            *reinterpret_cast<float4*>(&sm.red[warp][h][lane * 4]) = make_float4(o[h][0], o[h][1], o[h][2], o[h][3]);
    }
    __syncthreads();
    for (int i = tid; i < GQ * kHeadDim; i += 256) {
        const int h = i / kHeadDim, d = i % kHeadDim;
        float s = sm.red[0][h][d];
#pragma unroll
        for (int w = 1; w < 8; ++w) s = __fadd_rn(s, sm.red[w][h][d]);
        pout[(size_t)h * kPartStride + d] = s;
    }
}

template <int GQ>
__global__ void __launch_bounds__(256)
attn_kernel(const float* __restrict__ q, int64_t ldq, AttnRows rows, int Hq, int Hkv, float scale,
            float* __restrict__ part, int* __restrict__ tickets, float* __restrict__ out, int64_t ldo,
            int8_t* __restrict__ out_q, float* __restrict__ out_d)
{
    __shared__ __align__(16) AttnSmem<GQ> sm;  // q rows stay 16-byte aligned: kQStride % 4 == 0
    pdl_trigger();
    const int chunk = blockIdx.x, g = blockIdx.y;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    int r = 0;
#pragma unroll 1
    for (int i = 1; i < rows.n_rows; ++i)
        if (chunk >= rows.row[i].chunk0) r = i;
    const AttnRow row = rows.row[r];
    const int CH = row.chunk;
    const int c = chunk - row.chunk0;
    const int nch = (row.len + CH - 1) / CH;
    const int key0 = c * CH;
    const int nvalid = min(CH, row.len - key0);
    const int h0 = g * GQ;
    const __half* kbase = row.k + g * row.head_stride + (int64_t)key0 * row.tok_stride;
    const __half* vbase = row.v + g * row.head_stride + (int64_t)key0 * row.tok_stride;
    if (tid == 0) {
        // stage the chunk's K and V rows in L2 while the previous kernel ends
        // (a cache hint only: the rows it writes are read after pdl_wait)
        const uint32_t span = (uint32_t)(((int64_t)(nvalid - 1) * row.tok_stride + kHeadDim) * 2);
        prefetch_l2(kbase, span);
        prefetch_l2(vbase, span);
    }
    pdl_wait();
    for (int i = tid; i < GQ * kHeadDim; i += 256)
        sm.q[i / kHeadDim][qpad(i % kHeadDim)] = q[(size_t)r * ldq + (size_t)(h0 + i / kHeadDim) * kHeadDim + i % kHeadDim];
    __syncthreads();

    float* pout = part + ((size_t)chunk * Hq + h0) * kPartStride;
    if (CH == 64)
        attn_chunk<GQ, 64>(sm, kbase, vbase, row.tok_stride, nvalid, scale, pout);
    else if (CH == 128)
        attn_chunk<GQ, 128>(sm, kbase, vbase, row.tok_stride, nvalid, scale, pout);
    else
        attn_chunk<GQ, 256>(sm, kbase, vbase, row.tok_stride, nvalid, scale, pout);

    // ---- the last CTA of (row, g) merges the row's chunks
    __threadfence();
    __syncthreads();
    if (tid == 0) sm.last = (atomicAdd(&tickets[r * Hkv + g], 1) == nch - 1);
    __syncthreads();
    if (!sm.last) return;
    __threadfence();
    const float* base = part + ((size_t)row.chunk0 * Hq + h0) * kPartStride;
    const size_t cstride = (size_t)Hq * kPartStride;
    // chunk weights w[h][c] = e^(m_c - M_h), the chunk sums l[h][c] and L_h,
    // in the reduction scratch; every load of the chunk statistics is issued
    // lane-parallel, only the sum over c is sequential (in chunk order).
    float* wts = &sm.red[0][0][0];                // [GQ][nch]
    float* lsum = &sm.red[0][0][0] + GQ * nch;    // [GQ][nch]
    float* Ls = &sm.red[0][0][0] + 2 * GQ * nch;  // [GQ]
    for (int h = warp; h < GQ; h += 8) {
        const float* bh = base + (size_t)h * kPartStride;
        float M = -INFINITY;
        for (int cc = lane; cc < nch; cc += 32) {
            const float m = __ldcg(bh + cc * cstride + 128);
            wts[h * nch + cc] = m;
            lsum[h * nch + cc] = __ldcg(bh + cc * cstride + 129);
            M = fmaxf(M, m);
        }
        M = warp_max(M);
        for (int cc = lane; cc < nch; cc += 32) wts[h * nch + cc] = expf(__fsub_rn(wts[h * nch + cc], M));
        __syncwarp();
        if (lane == 0) {
            float L = 0.0f;
            for (int cc = 0; cc < nch; ++cc) L = __fmaf_rn(lsum[h * nch + cc], wts[h * nch + cc], L);
            Ls[h] = L;
        }
    }
    __syncthreads();
    for (int blk = warp; blk < GQ * (kHeadDim / 32); blk += 8) {
        const int h = blk / (kHeadDim / 32), d = (blk % (kHeadDim / 32)) * 32 + lane;
        const float* bh = base + (size_t)h * kPartStride + d;
        const float* wh = wts + h * nch;
        float O = 0.0f;
        int cc = 0;
        for (; cc + 16 <= nch; cc += 16) {
            float ov[16];
#pragma unroll
            for (int u = 0; u < 16; ++u) ov[u] = __ldcg(bh + (cc + u) * cstride);
#pragma unroll
            for (int u = 0; u < 16; ++u) O = __fmaf_rn(ov[u], wh[cc + u], O);
        }
        for (; cc < nch; ++cc) O = __fmaf_rn(__ldcg(bh + cc * cstride), wh[cc], O);
        const float val = __fdiv_rn(O, Ls[h]);
        const size_t oi = (size_t)r * ldo + (size_t)(h0 + h) * kHeadDim + d;
        out[oi] = val;
        if (out_q) {
            float dd;
            const int code = q8_quantize_lane(val, &dd);
            out_q[oi] = (int8_t)code;
            if (lane == 0) out_d[oi / 32] = dd;
        }
    }
    if (tid == 0) tickets[r * Hkv + g] = 0;  // ready for the next launch
}

template <int GQ>
static void launch_g(const float* q, int64_t ldq, const AttnRows& rows, int Hq, int Hkv, float scale, float* part,
                     int* tickets, float* out, int64_t ldo, int8_t* out_q, float* out_d, cudaStream_t s)
{
    launch_pdl(attn_kernel<GQ>, dim3(rows.total_chunks, Hkv), dim3(256), s, q, ldq, rows, Hq, Hkv, scale, part, tickets,
               out, ldo, out_q, out_d);
    count_launches(1);
}

cudaError_t launch_attention(const float* q, int64_t ldq, const AttnRows& rows, int Hq, int Hkv, float scale,
                             float* part, int* tickets, float* out, int64_t ldo, int8_t* out_q, float* out_d,
                             cudaStream_t s)
{
    switch (Hq / Hkv) {
#define LUCE_AT(G) \
    case G: launch_g<G>(q, ldq, rows, Hq, Hkv, scale, part, tickets, out, ldo, out_q, out_d, s); break;
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
    return cudaGetLastError();
}

}  // namespace luce
