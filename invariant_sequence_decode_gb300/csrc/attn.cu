// attn.cu - multi-sequence GQA decode attention, split-K over each row's own
// f16 cache with an exact, ordered log-sum-exp merge.
//
// "antirez/ds4 pull 604", Commit walkthrough: one query token per sequence,
// each attending to its own cache, per-sequence views passed by value (max 4);
// section 2: one multi-sequence attention launch with no position limit.
//
// Pass 1 (one CTA per (row, chunk of 256 keys, KV head g)): the CTA serves
// all Hq/Hkv query heads of g, so each K/V byte is read once per row.
//   scores   thread j owns key j of the chunk: 16 x 16-byte loads of its K row,
//            s_h = scale * (q_h . k_j) with fma over d = 0..127 ascending;
//   softmax  warp h owns head h: m = max_j s_h, p_j = exp(s_h - m),
//            l = sum p_j (lane-serial over j = lane + 32i, then butterfly);
//   values   warp w owns keys w, w+8, ... and lane l dims 4l..4l+3:
//            o_h += p_hj * v_j (fma, keys ascending); the 8 warp partials are
//            added in warp order.
//   -> scratch (o_h[128], m_h, l_h) for the chunk.
// Pass 2 (one CTA per (row, q head), thread = dim): M = max_c m_c,
//   L = sum_c l_c e^(m_c - M), O = sum_c o_c e^(m_c - M) in chunk order,
//   out = O / L.
// The chunking and every reduction order depend only on the row's own key
// count, never on the other rows or on the grid.
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace luce {

constexpr int kPartStride = 132;  // o[128], m, l, 2 pad floats per (chunk, head)

size_t attn_part_floats(int total_chunks, int Hq) { return (size_t)total_chunks * Hq * kPartStride; }

template <int GQ>
__global__ void __launch_bounds__(256)
attn_partial_kernel(const float* __restrict__ q, int64_t ldq, AttnRows rows, int Hq, float scale,
                    float* __restrict__ part)
{
    __shared__ __align__(16) float q_s[GQ][kHeadDim];
    __shared__ float p_s[GQ][kAttnChunk];
    __shared__ __align__(16) float red[8][GQ][kHeadDim];

    const int chunk = blockIdx.x, g = blockIdx.y;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    int r = 0;
#pragma unroll 1
    for (int i = 1; i < rows.n_rows; ++i)
        if (chunk >= rows.row[i].chunk0) r = i;
    const AttnRow row = rows.row[r];
    const int c = chunk - row.chunk0;
    const int key0 = c * kAttnChunk;
    const int nvalid = min(kAttnChunk, row.len - key0);
    const int h0 = g * GQ;

    for (int i = tid; i < GQ * kHeadDim; i += 256)
        q_s[i / kHeadDim][i % kHeadDim] = q[(size_t)r * ldq + (size_t)(h0 + i / kHeadDim) * kHeadDim + i % kHeadDim];
    __syncthreads();

    // ---- scores
    {
        float dot[GQ];
#pragma unroll
        for (int h = 0; h < GQ; ++h) dot[h] = 0.0f;
        const int j = tid;
        if (j < nvalid) {
            const int4* kp = reinterpret_cast<const int4*>(row.k + g * row.head_stride + (int64_t)(key0 + j) * row.tok_stride);
            int4 kv[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) kv[i] = __ldg(kp + i);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const __half2* hp = reinterpret_cast<const __half2*>(&kv[i]);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 kf = __half22float2(hp[e]);
                    const int d = i * 8 + e * 2;
#pragma unroll
                    for (int h = 0; h < GQ; ++h) {
                        dot[h] = __fmaf_rn(q_s[h][d], kf.x, dot[h]);
                        dot[h] = __fmaf_rn(q_s[h][d + 1], kf.y, dot[h]);
                    }
                }
            }
        }
#pragma unroll
        for (int h = 0; h < GQ; ++h) p_s[h][j] = (j < nvalid) ? __fmul_rn(dot[h], scale) : -INFINITY;
    }
    __syncthreads();

    // ---- chunk softmax statistics, warp h per head
    float* pout = part + ((size_t)chunk * Hq + h0) * kPartStride;
    for (int h = warp; h < GQ; h += 8) {
        float sv[kAttnChunk / 32];
        float m = -INFINITY;
#pragma unroll
        for (int i = 0; i < kAttnChunk / 32; ++i) {
            sv[i] = p_s[h][lane + 32 * i];
            m = fmaxf(m, sv[i]);
        }
        m = warp_max(m);
        float l = 0.0f;
#pragma unroll
        for (int i = 0; i < kAttnChunk / 32; ++i) {
            const int j = lane + 32 * i;
            const float p = (j < nvalid) ? expf(__fsub_rn(sv[i], m)) : 0.0f;
            p_s[h][j] = p;
            l = __fadd_rn(l, p);
        }
        l = warp_sum_butterfly(l);
        if (lane == 0) {
            pout[(size_t)h * kPartStride + 128] = m;
            pout[(size_t)h * kPartStride + 129] = l;
        }
    }
    __syncthreads();

    // ---- p . V
    {
        float o[GQ][4];
#pragma unroll
        for (int h = 0; h < GQ; ++h)
#pragma unroll
            for (int e = 0; e < 4; ++e) o[h][e] = 0.0f;
        const __half* vbase = row.v + g * row.head_stride + (int64_t)key0 * row.tok_stride + lane * 4;
        for (int j = warp; j < nvalid; j += 8) {
            const uint2 raw = __ldg(reinterpret_cast<const uint2*>(vbase + (int64_t)j * row.tok_stride));
            const float2 v01 = __half22float2(*reinterpret_cast<const __half2*>(&raw.x));
            const float2 v23 = __half22float2(*reinterpret_cast<const __half2*>(&raw.y));
#pragma unroll
            for (int h = 0; h < GQ; ++h) {
                const float p = p_s[h][j];
                o[h][0] = __fmaf_rn(p, v01.x, o[h][0]);
                o[h][1] = __fmaf_rn(p, v01.y, o[h][1]);
                o[h][2] = __fmaf_rn(p, v23.x, o[h][2]);
                o[h][3] = __fmaf_rn(p, v23.y, o[h][3]);
            }
        }
#pragma unroll
        for (int h = 0; h < GQ; ++h)
            *reinterpret_cast<float4*>(&red[warp][h][lane * 4]) = make_float4(o[h][0], o[h][1], o[h][2], o[h][3]);
    }
    __syncthreads();
    for (int i = tid; i < GQ * kHeadDim; i += 256) {
        const int h = i / kHeadDim, d = i % kHeadDim;
        float s = red[0][h][d];
#pragma unroll
        for (int w = 1; w < 8; ++w) s = __fadd_rn(s, red[w][h][d]);
        pout[(size_t)h * kPartStride + d] = s;
    }
}

__global__ void __launch_bounds__(128)
attn_merge_kernel(AttnRows rows, int Hq, const float* __restrict__ part, float* __restrict__ out, int64_t ldo)
{
    const int r = blockIdx.x / Hq, h = blockIdx.x - (blockIdx.x / Hq) * Hq;
    const int d = threadIdx.x;
    const AttnRow row = rows.row[r];
    const int nch = (row.len + kAttnChunk - 1) / kAttnChunk;
    const float* base = part + ((size_t)row.chunk0 * Hq + h) * kPartStride;
    const size_t cstride = (size_t)Hq * kPartStride;
    float M = -INFINITY;
    for (int c = 0; c < nch; ++c) M = fmaxf(M, base[c * cstride + 128]);
    float L = 0.0f, O = 0.0f;
    for (int c = 0; c < nch; ++c) {
        const float* pc = base + c * cstride;
        const float w = expf(__fsub_rn(pc[128], M));
        L = __fmaf_rn(pc[129], w, L);
        O = __fmaf_rn(pc[d], w, O);
    }
    out[(size_t)r * ldo + (size_t)h * kHeadDim + d] = __fdiv_rn(O, L);
}

template <int GQ>
static void launch_partial(const float* q, int64_t ldq, const AttnRows& rows, int Hq, int Hkv, float scale,
                           float* part, cudaStream_t s)
{
    dim3 grid(rows.total_chunks, Hkv);
    attn_partial_kernel<GQ><<<grid, 256, 0, s>>>(q, ldq, rows, Hq, scale, part);
    count_launches(1);
}

cudaError_t launch_attention(const float* q, int64_t ldq, const AttnRows& rows, int Hq, int Hkv,
                             float scale, float* part, float* out, int64_t ldo, cudaStream_t s)
{
    switch (Hq / Hkv) {
        case 1: launch_partial<1>(q, ldq, rows, Hq, Hkv, scale, part, s); break;
        case 2: launch_partial<2>(q, ldq, rows, Hq, Hkv, scale, part, s); break;
        case 3: launch_partial<3>(q, ldq, rows, Hq, Hkv, scale, part, s); break;
        case 4: launch_partial<4>(q, ldq, rows, Hq, Hkv, scale, part, s); break;
        case 5: launch_partial<5>(q, ldq, rows, Hq, Hkv, scale, part, s); break;
        case 6: launch_partial<6>(q, ldq, rows, Hq, Hkv, scale, part, s); break;
        case 7: launch_partial<7>(q, ldq, rows, Hq, Hkv, scale, part, s); break;
        case 8: launch_partial<8>(q, ldq, rows, Hq, Hkv, scale, part, s); break;
        default: return cudaErrorInvalidValue;
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    attn_merge_kernel<<<rows.n_rows * Hq, kHeadDim, 0, s>>>(rows, Hq, part, out, ldo);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace luce
