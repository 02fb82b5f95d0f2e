// rope_kv.cu - pos-vector RoPE and the per-sequence K/V append.
//
// "antirez/ds4 pull 604", Commit walkthrough: decode tokens of different
// sequences sit at arbitrary positions, so RoPE takes a position per row and
// its per-element math is that of a single-token launch at that position;
// section 2: KV append runs per sequence with the single-token helpers.
//
// Pairing: dims (i, i + 64) of a 128-dim head rotate by pos * theta^(-i/64).
// theta^(-i/64) is evaluated in double on the host; the angle is formed and
// reduced in double on the device and only the reduced angle goes through
// fp32 sincosf (see rope_cs), so even position 32767 carries no fp32 angle
// error.  The rotation is fp32 with explicit rounding.  One CTA of 64 threads
// per (row, head): thread i owns pair i.  The decode step applies the same
// rotation and append in the epilogue of its q|k|v projection (matvec.cu).
#include "common.cuh"
#include "kernels.h"

namespace luce {

__global__ void __launch_bounds__(64)
rope_posvec_kernel(float* __restrict__ x, int64_t ldx, const int32_t* __restrict__ pos, RopeFreq f)
{
    pdl_trigger();
    pdl_wait();
    const int t = blockIdx.x, h = blockIdx.y, i = threadIdx.x;
    const float2 cs = rope_cs(pos[t], f.inv[i]);
    float* p = x + (size_t)t * ldx + (size_t)h * kHeadDim + i;
    float x0 = p[0], x1 = p[kHeadDim / 2];
    rope_rotate(x0, x1, cs.x, cs.y);
    p[0] = x0;
    p[kHeadDim / 2] = x1;
}

cudaError_t launch_rope_posvec(float* x, int T, int n_heads, int64_t ldx, const int32_t* pos,
                               const RopeFreq& f, cudaStream_t s)
{
    const cudaError_t e = launch_pdl(rope_posvec_kernel, dim3(T, n_heads), dim3(64), s, x, ldx, pos, f);
    count_launches(1);
    return e;
}

// RoPE and the K/V append of the decode step from a q|k|v projection already
// in memory (the wide-verify path, where the projection runs on the tensor
// cores without an epilogue): one 64-thread CTA per (row t, head h of the
// q|k|v output), thread i owning the pair (i, i + 64).  q and k heads rotate
// by the row's position, q heads go to q_rot [T][Hq][128], k and v heads are
// rounded to binary16 at the row's K/V destination.  These are the rotation
// and conversion of the fused q|k|v epilogue (rope_cs, rope_rotate, round to
// nearest), so either path gives the same bits; cos/sin are formed before the
// wait on the projection.
__global__ void __launch_bounds__(64)
qkv_rope_kv_kernel(const float* __restrict__ qkv, int Hq, int Hkv, RowPos pos, RopeFreq f, float* __restrict__ q_rot,
                   KvRows kv)
{
    pdl_trigger();
    const int t = blockIdx.x, h = blockIdx.y, i = threadIdx.x;
    const bool rot = h < Hq + Hkv;
    const float2 cs = rot ? rope_cs(pos.pos[t], f.inv[i]) : make_float2(1.0f, 0.0f);
    pdl_wait();
    const float* src = qkv + (size_t)t * (Hq + 2 * Hkv) * kHeadDim + (size_t)h * kHeadDim;
    float x0 = src[i], x1 = src[i + kHeadDim / 2];
    if (rot) rope_rotate(x0, x1, cs.x, cs.y);
    if (h < Hq) {
        float* dst = q_rot + ((size_t)t * Hq + h) * kHeadDim;
        dst[i] = x0;
        dst[i + kHeadDim / 2] = x1;
    } else {
        const KvRow r = kv.row[t];
        __half* dst = rot ? r.k + (h - Hq) * r.head_stride : r.v + (h - Hq - Hkv) * r.head_stride;
        dst[i] = __float2half_rn(x0);
        dst[i + kHeadDim / 2] = __float2half_rn(x1);
    }
}

cudaError_t launch_qkv_rope_kv(const float* qkv, int T, int Hq, int Hkv, const RowPos& pos, const RopeFreq& f,
                               float* q_rot, const KvRows& kv, cudaStream_t s)
{
    const cudaError_t e =
        launch_pdl(qkv_rope_kv_kernel, dim3(T, Hq + 2 * Hkv), dim3(kHeadDim / 2), s, qkv, Hq, Hkv, pos, f, q_rot, kv);
    count_launches(1);
    return e;
}

// Standalone K/V append: one CTA per row; fp32 -> binary16 round-to-nearest.
__global__ void __launch_bounds__(256)
kv_append_kernel(const float* __restrict__ k, const float* __restrict__ v, int64_t ld, int Hkv, KvRows rows)
{
    pdl_trigger();
    pdl_wait();
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
    const cudaError_t e = launch_pdl(kv_append_kernel, dim3(rows.n_rows), dim3(256), s, k, v, ld, Hkv, rows);
    count_launches(1);
    return e;
}

}  // namespace luce
