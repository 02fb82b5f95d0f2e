// kernels.h - host-side launchers of the libluce kernels (internal).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace luce {

// Counts kernel launches (bumped by every launcher below).
void count_launches(int n);

// Per-row destination of a K/V append: element (g, d) of the row goes to
// k[g * head_stride + d] (the pointers already point at the row's position).
struct KvRow {
    __half* k;
    __half* v;
    int64_t head_stride;
};
struct KvRows {
    KvRow row[16];
    int n_rows;
};

// One query row of decode attention over keys j < len; chunk0 is the index
// of its first split-K chunk in the scratch.  Flat cache (pages == nullptr):
// element d of key j of KV head g is k[g*head_stride + j*tok_stride + d].
// Paged cache: key j lives in page pages[j / 128] at
// k[pages[j / 128]*page_stride + g*head_stride + (j % 128)*tok_stride + d].
struct AttnRow {
    const __half* k;
    const __half* v;
    int64_t head_stride;
    int64_t tok_stride;
    int len;
    int chunk0;
    int chunk;  // keys per split-K chunk of this row: attn_chunk_keys(len)
    const int32_t* pages;  // device page table (128 keys per page) or nullptr
    int64_t page_stride;
};
struct AttnRows {
    AttnRow row[16];
    int n_rows;
    int total_chunks;
};

// Positions of up to 16 rows, passed by value.
struct RowPos {
    int pos[16];
    int n_rows;
};

// RoPE inverse frequencies theta^(-2i/128), i < 64, evaluated in double on
// the host and passed by value.
struct RopeFreq {
    double inv[64];
};
RopeFreq rope_freq(double theta);

// d: fp32 [T][K/32] scales, or binary16 bits when half_scale.
cudaError_t launch_quantize(const float* x, int T, int K, int64_t ldx, int8_t* q, void* d, bool half_scale,
                            cudaStream_t s);

cudaError_t launch_matvec(const int8_t* wq, const __half* wd, int N, int K, const int8_t* aq,
                          const float* ad, int T, float* y, int64_t ldy, const float* resid,
                          int64_t ldr, cudaStream_t s);

// The TMA-ring matvec (1..8 rows in one launch, 13..16 in two):
// cudaErrorNotSupported, with nothing launched, for 9..12 rows, K % 256 != 0,
// an operand not 16-byte aligned or no tensor-map encoder.
cudaError_t launch_matvec_tma(const int8_t* wq, const __half* wd, int N, int K, const int8_t* aq, const float* ad,
                              int T, float* y, int64_t ldy, const float* resid, int64_t ldr, cudaStream_t s);

// The tensor-core matvec (1..16 rows, one launch; matvec_mma.cu):
// cudaErrorNotSupported, with nothing launched, when K % 256 != 0, an operand
// is not 16-byte aligned or no tensor-map encoder is available.
cudaError_t launch_matvec_mma(const int8_t* wq, const __half* wd, int N, int K, const int8_t* aq, const float* ad,
                              int T, float* y, int64_t ldy, const float* resid, int64_t ldr, cudaStream_t s);

// The matvec through one named kernel (kMatvecPath*); cudaErrorNotSupported,
// with nothing launched, when that kernel does not serve the shape.
// (the values of LUCE_MATVEC_AUTO .. LUCE_MATVEC_TENSOR in luce.h)
enum { kMatvecAuto = 0, kMatvecRegister = 1, kMatvecRing = 2, kMatvecMma = 3 };
cudaError_t launch_matvec_path(int path, const int8_t* wq, const __half* wd, int N, int K, const int8_t* aq,
                               const float* ad, int T, float* y, int64_t ldy, const float* resid, int64_t ldr,
                               cudaStream_t s);

// The fused q|k|v + RoPE + K/V-append projection on the TMA ring (1..8 rows
// in one launch, 13..16 in two); cudaErrorNotSupported, with nothing
// launched, otherwise.
// The step's gate||up projection (W = [gate; up], 2F x K) with SwiGLU and
// its q8_0 codes (fp32 scales) in the epilogue: gu [T][2F] as the plain
// projection, h [T][F], hq [T][F], hd [T][F/32] as swiglu_quant_kernel.
// cudaErrorNotSupported when the fused ring does not take the shape (the
// caller then runs the two launches).
cudaError_t launch_gateup_swiglu_tma(const int8_t* wq, const __half* wd, int F, int K, const int8_t* aq,
                                     const float* ad, int T, float* gu, float* h, int8_t* hq, float* hd,
                                     cudaStream_t s);
cudaError_t launch_qkv_rope_tma(const int8_t* wq, const __half* wd, int K, const int8_t* aq, const float* ad, int T,
                                float* qkv, int Hq, int Hkv, const RowPos& pos, const RopeFreq& f, float* q_rot,
                                const KvRows& kv, cudaStream_t s);

// Bounded waits that expired on the current device (synchronous; the dp4a
// ring's, the tensor-core ring's and the slot attention's counters summed);
// reset clears the counters.
cudaError_t read_wait_timeouts(uint32_t* count, bool reset);
cudaError_t read_mma_wait_timeouts(uint32_t* count, bool reset);
cudaError_t read_attn_wait_timeouts(uint32_t* count, bool reset);

// One bounded wait that nothing completes (limit_ns), counted as expired.
cudaError_t launch_wait_expiry(uint64_t limit_ns, cudaStream_t s);

// The step's q|k|v projection (N = (Hq + 2*Hkv) * 128 rows) with RoPE of the
// q and k heads at each row's position, q heads to q_rot [T][Hq][128], k and v
// heads appended as binary16 at rows' K/V destinations; qkv [T][N] also written.
cudaError_t launch_qkv_rope(const int8_t* wq, const __half* wd, int K, const int8_t* aq, const float* ad, int T,
                            float* qkv, int Hq, int Hkv, const RowPos& pos, const RopeFreq& f, float* q_rot,
                            const KvRows& kv, cudaStream_t s);

// RoPE of the q and k heads and the K/V append from a q|k|v projection in
// qkv [T][(Hq + 2 Hkv) 128] (the epilogue of launch_qkv_rope as its own launch).
// The step's q|k|v projection on the tensor-core ring with RoPE and the K/V
// append in its epilogue (1..16 rows; the same bits as launch_matvec_mma +
// launch_qkv_rope_kv).  cudaErrorNotSupported when the ring does not take
// the shapes.
cudaError_t launch_qkv_rope_mma(const int8_t* wq, const __half* wd, int K, const int8_t* aq, const float* ad, int T,
                                float* qkv, int Hq, int Hkv, const RowPos& pos, const RopeFreq& f, float* q_rot,
                                const KvRows& kv, cudaStream_t s);
cudaError_t launch_qkv_rope_kv(const float* qkv, int T, int Hq, int Hkv, const RowPos& pos, const RopeFreq& f,
                               float* q_rot, const KvRows& kv, cudaStream_t s);

cudaError_t launch_block_dots(const int8_t* wq, int N, int K, const int8_t* aq, int T, int32_t* out,
                              cudaStream_t s);

cudaError_t launch_rope_posvec(float* x, int T, int n_heads, int64_t ldx, const int32_t* pos,
                               const RopeFreq& f, cudaStream_t s);

cudaError_t launch_kv_append(const float* k, const float* v, int64_t ld, int Hkv, const KvRows& rows,
                             cudaStream_t s);

// Scratch floats for `total_chunks` chunks of Hq heads.
size_t attn_part_floats(int total_chunks, int Hq);

// Keys per split-K chunk for a row with `len` keys (a function of len only).
int attn_chunk_keys(int len);
constexpr int kAttnMaxChunksPerRow = 511;  // the merge keeps two floats per chunk in shared memory

// part: attn_part_floats(total_chunks, Hq) floats of split-K scratch.
// out_q / out_d (nullable): q8_0 codes and scales of out (requires ldo == Hq*128).
// Two launches: the chunks, then their merge.
cudaError_t launch_attention(const float* q, int64_t ldq, const AttnRows& rows, int Hq, int Hkv,
                             float scale, float* part, float* out, int64_t ldo,
                             int8_t* out_q, float* out_d, cudaStream_t s);

// xcopy (nullable): the CTAs also copy the rows of x there (x may then be a
// mapped host pointer).
cudaError_t launch_rmsnorm_quant(const float* x, int T, int H, const float* gamma, float eps, float* xn, int8_t* q,
                                 void* d, bool half_scale, cudaStream_t s, float* xcopy = nullptr);
// x [n] (n a multiple of 4, 16-byte aligned) to x_out and am [T] to am_out,
// both mapped host memory (either nullable).
cudaError_t launch_rows_to_host(const float* x, int64_t n, float* x_out, const int32_t* am, int T, int32_t* am_out,
                                cudaStream_t s);

cudaError_t launch_swiglu_quant(const float* gu, int T, int F, float* h, int8_t* q, void* d, bool half_scale,
                                cudaStream_t s);

cudaError_t launch_argmax(const float* x, int T, int V, int32_t* out, cudaStream_t s);

}  // namespace luce
