// rope_kv.cu - pos-vector RoPE and the per-sequence K/V append.
//
// "antirez/ds4 pull 604", Commit walkthrough: decode tokens of different
// sequences sit at arbitrary positions, so RoPE takes a position per row and
// its per-element math is that of a single-token launch at that position;
// section 2: KV append runs per sequence with the single-token helpers.
//
// Pairing: dims (i, i + 64) of a 128-dim head rotate by pos * theta^(-i/64).
// cos/sin come from a double-precision evaluation rounded to fp32 (so the
// angle carries no fp32 error even at position 32767); the rotation is fp32.
#include "common.cuh"
#include "kernels.h"

namespace luce {

// Standalone RoPE: one CTA per row; 64 threads evaluate the row's cos/sin.
__global__ void __launch_bounds__(256)
rope_posvec_kernel(float* __restrict__ x, int n_heads, int64_t ldx, const int32_t* __restrict__ pos,
                   double theta)
{
    __shared__ float2 cs[kHeadDim / 2];
    const int t = blockIdx.x;
    if (threadIdx.x < kHeadDim / 2) cs[threadIdx.x] = rope_cs(pos[t], threadIdx.x, kHeadDim, theta);
    __syncthreads();
    float* xr = x + (size_t)t * ldx;
    for (int idx = threadIdx.x; idx < n_heads * (kHeadDim / 2); idx += blockDim.x) {
        const int h = idx >> 6, i = idx & 63;
        float* p = xr + h * kHeadDim + i;
        float x0 = p[0], x1 = p[kHeadDim / 2];
        rope_rotate(x0, x1, cs[i].x, cs[i].y);
        p[0] = x0;
        p[kHeadDim / 2] = x1;
    }
}

cudaError_t launch_rope_posvec(float* x, int T, int n_heads, int64_t ldx, const int32_t* pos,
                               double theta, cudaStream_t s)
{
    rope_posvec_kernel<<<T, 256, 0, s>>>(x, n_heads, ldx, pos, theta);
    count_launches(1);
    return cudaGetLastError();
}

// Per-step cos/sin table [T][64] (float2), positions by value.
__global__ void rope_table_kernel(RowPos pos, double theta, float2* __restrict__ cs)
{
    const int t = blockIdx.x, i = threadIdx.x;
    cs[t * (kHeadDim / 2) + i] = rope_cs(pos.pos[t], i, kHeadDim, theta);
}

cudaError_t launch_rope_table(const RowPos& pos, double theta, float2* cs, cudaStream_t s)
{
    rope_table_kernel<<<pos.n_rows, kHeadDim / 2, 0, s>>>(pos, theta, cs);
    count_launches(1);
    return cudaGetLastError();
}

// Standalone K/V append: one CTA per row; fp32 -> binary16 round-to-nearest.
__global__ void __launch_bounds__(256)
kv_append_kernel(const float* __restrict__ k, const float* __restrict__ v, int64_t ld, int Hkv, KvRows rows)
{
    const int t = blockIdx.x;
    const KvRow r = rows.row[t];
    for (int idx = threadIdx.x; idx < Hkv * kHeadDim; idx += blockDim.x) {
        const int g = idx >> 7, dd = idx & 127;
        r.k[g * r.head_stride + dd] = __float2half_rn(k[(size_t)t * ld + idx]);
        r.v[g * r.head_stride + dd] = __float2half_rn(v[(size_t)t * ld + idx]);
    }
}

cudaError_t launch_kv_append(const float* k, const float* v, int64_t ld, int Hkv, const KvRows& rows,
                             cudaStream_t s)
{
    kv_append_kernel<<<rows.n_rows, 256, 0, s>>>(k, v, ld, Hkv, rows);
    count_launches(1);
    return cudaGetLastError();
}

// Decode-step glue, one CTA per row: rotate the row's q heads into q_rot,
// rotate its k heads and append k and v to the row's cache position.  Uses
// the same rotation and conversion as the standalone kernels above.
__global__ void __launch_bounds__(256)
rope_kv_kernel(const float* __restrict__ qkv, int Hq, int Hkv, const float2* __restrict__ cs_tab,
               float* __restrict__ q_rot, KvRows rows)
{
    __shared__ float2 cs[kHeadDim / 2];
    const int t = blockIdx.x;
    const int ld = (Hq + 2 * Hkv) * kHeadDim;
    if (threadIdx.x < kHeadDim / 2) cs[threadIdx.x] = cs_tab[t * (kHeadDim / 2) + threadIdx.x];
    __syncthreads();
    const float* row = qkv + (size_t)t * ld;
    // q and k heads: (Hq + Hkv) heads x 64 pairs
    for (int idx = threadIdx.x; idx < (Hq + Hkv) * (kHeadDim / 2); idx += blockDim.x) {
        const int h = idx >> 6, i = idx & 63;
        float x0 = row[h * kHeadDim + i], x1 = row[h * kHeadDim + i + 64];
        rope_rotate(x0, x1, cs[i].x, cs[i].y);
        if (h < Hq) {
            q_rot[(size_t)t * Hq * kHeadDim + h * kHeadDim + i] = x0;
            q_rot[(size_t)t * Hq * kHeadDim + h * kHeadDim + i + 64] = x1;
        } else {
            const KvRow r = rows.row[t];
            __half* dst = r.k + (h - Hq) * r.head_stride;
            dst[i] = __float2half_rn(x0);
            dst[i + 64] = __float2half_rn(x1);
        }
    }
    const KvRow r = rows.row[t];
    const float* vrow = row + (Hq + Hkv) * kHeadDim;
    for (int idx = threadIdx.x; idx < Hkv * kHeadDim; idx += blockDim.x) {
        const int g = idx >> 7, dd = idx & 127;
        r.v[g * r.head_stride + dd] = __float2half_rn(vrow[idx]);
    }
}

cudaError_t launch_rope_kv(const float* qkv, int T, int Hq, int Hkv, const float2* cs, float* q_rot,
                           const KvRows& rows, cudaStream_t s)
{
    rope_kv_kernel<<<T, 256, 0, s>>>(qkv, Hq, Hkv, cs, q_rot, rows);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace luce
