/*
 * luce.h - C ABI of the batch-invariant concurrent decode step for GB300 (sm_103a).
 *
 * One decode step serves 1..4 sequences ("slots"); each slot contributes 1..4
 * rows (1 for plain decode, up to 4 when it verifies draft tokens), at most 16
 * rows in all.  Every projection reads the q8_0 weights once for all rows,
 * and every row comes out bit-identical to the same slot run alone: no
 * reduction order anywhere depends on the number of rows, on the other rows,
 * on their order or on the launch grid.
 *
 * Sources, cited by page title and section:
 *   [exact-4-slot]  "feat(qwen4exp): exact 4-slot concurrent serving",
 *                   sections "What" and "How it stays exact".
 *   [qfuse]         "#1209 Speed up concurrent generation, fix QFUSE, and
 *                   improve prefill monitoring", "What changed and why".
 *   [ds4-604]       antirez/ds4 pull 604, section 2 ("Single-GPU decode
 *                   batches don't scale") and "Commit walkthrough".
 *
 * Conventions for every entry point:
 *   - Pointers marked (device) are CUDA device pointers; (host) are host
 *     pointers read during the call only.  The caller allocates and owns
 *     every buffer; the library allocates nothing and never synchronises the
 *     host.  Work is enqueued on `stream` (a cudaStream_t; NULL = the legacy
 *     default stream) and is complete when that stream is.
 *   - Return value: LUCE_OK (0) or a negative luce_status.  On error nothing
 *     has been enqueued, except LUCE_ECUDA from a failed launch.
 *     luce_last_error() gives a message for the calling thread's last error.
 *   - binary16 data (fp16 weight scales, the K/V cache) is passed as uint16_t
 *     payloads.  q8_0 weights are stored as int8 wq[N][K] (row-major) plus
 *     binary16 wd[N][K/32]: 32 weights per block share one scale, 34 bytes
 *     per block in all.
 *   - Alignment: int8 weight and activation arrays start on 32-byte
 *     boundaries (each q8_0 block is fetched as one 32-byte load); K/V
 *     cache rows on 16-byte boundaries.
 */
#ifndef LUCE_H
#define LUCE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum luce_status {
    LUCE_OK = 0,
    LUCE_EINVAL = -1,       /* a null/misaligned pointer or an out-of-range size */
    LUCE_EUNSUPPORTED = -2, /* a shape the kernels do not serve (e.g. head_dim != 128) */
    LUCE_ECUDA = -3,        /* a CUDA launch failed */
    LUCE_ENOSPACE = -4      /* the workspace is smaller than required */
} luce_status;

#define LUCE_QK 32               /* q8_0 block length [ds4-604, Commit walkthrough] */
#define LUCE_MAX_SEQ 4           /* slots per step; more are refused [exact-4-slot, What] */
#define LUCE_MAX_ROWS_PER_SEQ 4  /* rows per slot (1 decode + up to 3 drafts) */
#define LUCE_MAX_ROWS 16         /* 8/12/16-row verify capacities [qfuse, item 1] */
#define LUCE_HEAD_DIM 128
#define LUCE_MAX_KEYS 130816     /* keys one attention row may see (511 chunks of 256) */

/* Message of the calling thread's last non-OK status ("" if none). */
const char* luce_last_error(void);

/* ABI version (major * 10000 + minor * 100 + patch). */
int luce_version(void);

/* Number of kernel launches this library has enqueued since it was loaded
 * (all threads).  A diagnostic for counting the work a call submits. */
uint64_t luce_launch_count(void);

/*
 * Bounded waits that expired on the current device.  The kernels that stream
 * weights through a ring of shared-memory stages filled by tensor copies (the
 * dp4a ring matvec, which luce_q8_matvec_batch takes at 1..4 rows; the
 * tensor-core ring matvec, at 5..16 rows; the fused q|k|v + RoPE + K/V-append
 * projection of the decode step on either ring) wait on shared-memory
 * barriers for those copies, and the attention that serves a slot's verify
 * rows together waits on one for its tcgen05 MMAs.  Every such wait gives up
 * after about one second and adds one to this device counter, so a stalled
 * copy engine or tensor core surfaces here instead of as a hung stream.  A
 * healthy run reads 0 (an attention CTA whose wait expired writes none of its
 * partial outputs).
 *
 * A non-zero count means the device context is suspect, not that some
 * outputs were merely skipped: the CTA whose wait expired stops writing;
 * before it exits it waits once more, again for about one second, for the
 * tensor copies it issued (and an attention CTA for its MMAs, before it
 * frees their tensor memory), and if that wait expires too (counted again)
 * a late copy can land in shared memory that later belongs to another CTA.
 * Treat every result computed since the last zero reading as untrusted and
 * recreate the context.  The decode step entry points return LUCE_OK
 * without looking at this counter (reading it synchronises the device):
 * callers that need the guarantee poll it after their steps.
 *   count (host) receives the counter; reset != 0 clears it afterwards.
 * Synchronises the device (it copies from device memory).  Returns LUCE_OK,
 * LUCE_EINVAL (null count) or LUCE_ECUDA.
 */
int luce_wait_timeouts(uint32_t* count, int reset);

/*
 * Test hook for the expiry path above: enqueues one kernel whose single
 * bounded wait (limit_ns, 1 us .. 1 s) is on a shared-memory barrier that
 * nothing completes, so the wait runs out, adds one to the counter and the
 * kernel returns; the context stays usable.  Returns LUCE_OK, LUCE_EINVAL or
 * LUCE_ECUDA.
 */
int luce_test_wait_expiry(int64_t limit_ns, void* stream);

/*
 * Activation quantization to q8_0 blocks [qfuse, item 2: the consumer's
 * division and rounding convention; ds4-604, Commit walkthrough].
 * For each row t and block b of 32 values: amax = max|x| (NaN skipped),
 * d = amax / 127 (fp32, IEEE division), q = round(x / d) with an IEEE fp32
 * division and rounding half away from zero, clamped to [-127, 127]; a block
 * with d == 0 gives all-zero codes and a NaN quotient gives 0.
 *   x  (device) fp32 [T][ldx], first K columns used (ldx >= K)
 *   q  (device) int8 [T][K], 16-byte aligned
 *   d  (device) fp32 [T][K/32]
 * 1 <= T <= LUCE_MAX_ROWS (any T >= 1 is accepted), K % 32 == 0.
 */
int luce_q8_quantize_act(const float* x, int T, int K, int64_t ldx, int8_t* q, float* d, void* stream);

/*
 * luce_q8_quantize_act with the block scale stored as binary16, the form a
 * fused producer must reproduce exactly [qfuse, item 2: match the consuming
 * quantizer's finite-half guards and division/rounding convention].  The
 * pages name the guards without stating them; read as: d = amax / 127 (fp32,
 * IEEE division) rounded to the nearest binary16; a scale that overflows
 * binary16 (amax / 127 >= 65520) is stored as the largest finite half, 65504,
 * so no stored scale is infinite; the codes are taken against the stored
 * scale, q = round(x / float(d)) with the IEEE fp32 division and rounding
 * half away from zero, clamped to [-127, 127]; a stored scale of zero (also
 * when amax / 127 underflows binary16) gives all-zero codes; a NaN quotient
 * gives 0.  float(d) is exact in fp32, so (q, float(d)) feeds
 * luce_q8_matvec_batch unchanged.
 *   x (device) fp32 [T][ldx];  q (device) int8 [T][K];  d (device) binary16 [T][K/32]
 */
int luce_q8_quantize_act_f16(const float* x, int T, int K, int64_t ldx, int8_t* q, uint16_t* d, void* stream);

/*
 * The decode step's fused producers of q8_0 activations, as entry points of
 * their own.  Each writes its fp32 output and that output's q8_0 codes and
 * scales with the very per-lane routine of luce_q8_quantize_act (half_scale
 * == 0: d is fp32 [T][K/32]) or of luce_q8_quantize_act_f16 (half_scale != 0:
 * d is binary16 [T][K/32]), so the codes equal a standalone quantization of
 * the fp32 output bit for bit [qfuse, item 2].
 *   luce_rmsnorm_q8: xn[t] = x[t] / sqrt(mean(x[t]^2) + eps) * gamma, the sum
 *     of squares in a fixed order that depends on H only (8 slices of the
 *     row's blocks, each summed per lane in ascending order, lanes by an xor
 *     butterfly, warps in order, then the slices in order); x, xn fp32 [T][H],
 *     gamma fp32 [H], q int8 [T][H]; 1 <= T <= LUCE_MAX_ROWS, H % 32 == 0.
 *   luce_swiglu_q8: h[t][i] = silu(gu[t][i]) * gu[t][F + i] (gate half first),
 *     silu(z) = z / (1 + e^-z); gu fp32 [T][2F], h fp32 [T][F], q int8 [T][F];
 *     F % 32 == 0.
 * All pointers (device).
 */
int luce_rmsnorm_q8(const float* x, int T, int H, const float* gamma, float eps, float* xn, int8_t* q, void* d,
                    int half_scale, void* stream);
int luce_swiglu_q8(const float* gu, int T, int F, float* h, int8_t* q, void* d, int half_scale, void* stream);

/*
 * Narrow-batch q8_0 matvec [ds4-604, Commit walkthrough: each 32-weight
 * block read once and dotted against all tokens; exact-4-slot, How it stays
 * exact: the same arithmetic for 1 row as for 4]:
 *   y[t][n] = sum_b (wd[n][b] * ad[t][b]) * sum_i wq[n][32b+i] * aq[t][32b+i]
 * The per-block sum is an exact int32.  The fp32 combine of a row uses a fixed
 * order that depends on K only: block b feeds partial sum (b mod 32), each
 * partial adds its blocks in ascending order with fused multiply-adds, and the
 * 32 partials are summed pairwise by an xor butterfly over offsets
 * 16, 8, 4, 2, 1.  Hence y[t][.] is bitwise independent of T, of the other
 * rows and of the launch shape.
 *   wq (device) int8 [N][K], 32-byte aligned;  wd (device) binary16 [N][K/32]
 *   aq (device) int8 [T][K], 32-byte aligned;  ad (device) fp32 [T][K/32]
 *   y  (device) fp32 [T][ldy] (ldy >= N)
 * 1 <= T <= LUCE_MAX_ROWS, K % 32 == 0, N >= 1.
 */
int luce_q8_matvec_batch(const int8_t* wq, const uint16_t* wd, int N, int K,
                         const int8_t* aq, const float* ad, int T, float* y, int64_t ldy, void* stream);

/*
 * luce_q8_matvec_batch through one named kernel (a diagnostic for tests and
 * benchmarks).  Every kernel computes the same chains and butterfly, so all
 * give the same bits:
 *   LUCE_MATVEC_AUTO      the library's choice (luce_q8_matvec_batch);
 *   LUCE_MATVEC_REGISTER  register-pipelined dp4a loads (any shape);
 *   LUCE_MATVEC_RING      dp4a on a TMA ring in shared memory (1..8 rows in
 *                         one launch, 13..16 in two; K % 256 == 0, 16-byte
 *                         aligned operands);
 *   LUCE_MATVEC_TENSOR    block dots on the tensor cores from a TMA ring
 *                         (1..16 rows in one launch; K % 256 == 0, 16-byte
 *                         aligned operands).
 * Arguments and errors as luce_q8_matvec_batch, plus LUCE_EUNSUPPORTED
 * (nothing launched) when the named kernel does not serve the shape.
 */
#define LUCE_MATVEC_AUTO 0
#define LUCE_MATVEC_REGISTER 1
#define LUCE_MATVEC_RING 2
#define LUCE_MATVEC_TENSOR 3
int luce_q8_matvec_batch_path(const int8_t* wq, const uint16_t* wd, int N, int K, const int8_t* aq, const float* ad,
                              int T, float* y, int64_t ldy, int path, void* stream);

/*
 * Per-block integer dots out[t][n][b] = sum_i wq[n][32b+i] * aq[t][32b+i],
 * computed with the register-pipelined matvec kernel's dp4a routine (exposed
 * so the exactness of the integer stage can be checked against the oracle).
 * The other matvec kernels form the same integers differently (a biased dp4a
 * chain, or f16 tensor-core products); that they agree is checked through
 * their outputs, which equal the register kernel's bit for bit.
 * out (device) int32 [T][N][K/32].
 */
int luce_q8_block_dots(const int8_t* wq, int N, int K, const int8_t* aq, int T, int32_t* out, void* stream);

/*
 * Pos-vector RoPE [ds4-604, Commit walkthrough: decode tokens of different
 * sequences sit at arbitrary positions; a row equals a single-row launch at
 * its own position].  Dims (i, i + D/2) of every head of row t rotate by
 * pos[t] * theta^(-2i/D).  The cosine and sine are evaluated in double
 * precision (theta^(-2i/D) and the angle in double, reduced modulo 2*pi before
 * an fp32 sincos) and rounded to fp32; the rotation itself is fp32.
 *   x   (device) fp32, element (t, h, d) at t*ldx + h*D + d, rotated in place
 *   pos (device) int32 [T]
 * D == 128, 1 <= T <= LUCE_MAX_ROWS (any T >= 1 is accepted), n_heads >= 1,
 * ldx >= n_heads * D.
 */
int luce_rope_posvec(float* x, int T, int n_heads, int D, int64_t ldx, const int32_t* pos,
                     double theta, void* stream);

/*
 * A sequence's view of its K/V cache for one layer [ds4-604, Commit
 * walkthrough: per-sequence view passed by value, max 4].  Element (g, j, d)
 * of K (and V) is at k[g*head_stride + j*tok_stride + d], binary16.
 * `len` counts the keys including this step's n_q rows: row j (0..n_q-1) of
 * the sequence is at position len - n_q + j and attends to keys
 * [0, len - n_q + j].  Its query/output row is row0 + j.
 */
typedef struct luce_seqview {
    uint16_t* k;          /* (device) */
    uint16_t* v;          /* (device) */
    int32_t len;
    int32_t n_q;          /* 1..LUCE_MAX_ROWS_PER_SEQ */
    int32_t row0;
    int32_t cap;          /* positions the view holds (len <= cap) */
    int64_t head_stride;  /* elements, multiple of 8 */
    int64_t tok_stride;   /* elements, multiple of 8, >= D */
} luce_seqview;

/*
 * Per-sequence KV append [ds4-604, section 2: KV append runs per sequence
 * with the single-token helpers].  Row row0 + j of k and v (fp32, element
 * (t, g, d) at t*ldkv + g*D + d) is rounded to binary16 (nearest even) and
 * written at position len - n_q + j of that view's cache.
 *   views (host) [n_seq], 1 <= n_seq <= LUCE_MAX_SEQ.
 */
int luce_kv_append(const float* k, const float* v, int64_t ldkv, int Hkv, int D,
                   const luce_seqview* views, int n_seq, void* stream);

/*
 * Multi-sequence decode attention [ds4-604, Commit walkthrough: one query
 * token per sequence against its own cache; here up to 4 causal rows per
 * sequence].  For row r of view s and query head h (KV head g = h / (Hq/Hkv)):
 *   out[r][h] = sum_j softmax_j(scale * q[r][h] . K[g][j]) V[g][j]
 * over the row's keys.  The keys are split into chunks of 128 keys (rows with
 * at most 16,384 keys) or 256 (more): a function of the row's own key count
 * only; each chunk yields (max, sum, unnormalised
 * output) and the chunks are merged in order by the exact log-sum-exp rule.
 * No output depends on the other rows.
 *   q   (device) fp32 [T][Hq][D] with T = max(row0 + n_q)
 *   out (device) fp32 [T][Hq][D]
 *   ws  (device) scratch of at least luce_decode_attn_workspace_size(...)
 *       bytes, 16-byte aligned (the chunk partials; no initial contents).
 * The chunks run on the tensor cores: rows with 128-key chunks in one kernel
 * (a view's rows share one CTA per (chunk, KV head), so the view's cache is
 * read once; scores on mma.sync, p.V on tcgen05.mma into tensor memory, whose
 * bounded wait counts in luce_wait_timeouts), rows with 256-key chunks in
 * another (mma.sync); which serves a row depends on its own key count only,
 * and a row gives the same bits alone or with its view's other rows.  Their
 * merge is launched behind them on the same stream (it starts once every
 * chunk is written): two launches, or three when both kinds of rows are
 * present.  No kernel waits on another CTA and nothing needs zeroing between
 * calls.
 * D == 128, Hq % Hkv == 0, Hq / Hkv <= 8, 1 <= n_seq <= LUCE_MAX_SEQ,
 * 1 <= len - n_q + 1, len <= cap, len <= LUCE_MAX_KEYS.
 */
int luce_decode_attn_multiseq(const float* q, const luce_seqview* views, int n_seq,
                              int Hq, int Hkv, int D, float scale, float* out,
                              void* ws, size_t ws_bytes, void* stream);

/* Bytes of scratch luce_decode_attn_multiseq needs for n_rows rows whose key
 * counts are at most max_len. */
size_t luce_decode_attn_workspace_size(int n_rows, int Hq, int D, int max_len);

/*
 * A sequence's K/V for one layer held in fixed pages of LUCE_PAGE_KEYS keys
 * [the per-sequence fallback beyond a flat cache: the pages' attention keeps
 * its per-sequence views, here each view names its pages].  Page p of a pool
 * is binary16 [Hkv][LUCE_PAGE_KEYS][D]; key j of the sequence is in pool page
 * table[j / LUCE_PAGE_KEYS] at row j % LUCE_PAGE_KEYS, so element (g, j, d) of
 * K is k_pool[(table[j / 128] * Hkv + g) * 128 * 128 + (j % 128) * 128 + d].
 * The page size equals the attention's key tile, so chunking and every sum
 * are those of the flat cache: a paged sequence gives the flat sequence's
 * bits.  table (device) holds ceil(len / 128) entries in [0, n_pages).
 */
#define LUCE_PAGE_KEYS 128
typedef struct luce_pagedview {
    const uint16_t* k_pool;  /* (device) [n_pages][Hkv][128][128], 16-byte aligned */
    const uint16_t* v_pool;  /* (device) same layout */
    const int32_t* table;    /* (device) page of each 128-key span */
    int32_t len;             /* keys including this step's n_q rows */
    int32_t n_q;             /* 1..LUCE_MAX_ROWS_PER_SEQ */
    int32_t row0;
} luce_pagedview;

/*
 * luce_decode_attn_multiseq over paged views (same rows, outputs, workspace
 * size and errors).  The table entries are device data the call cannot see:
 * the caller guarantees they lie in [0, n_pages) of their pool.
 */
int luce_decode_attn_paged(const float* q, const luce_pagedview* views, int n_seq, int Hq, int Hkv, int D,
                           float scale, float* out, void* ws, size_t ws_bytes, void* stream);

/*
 * luce_decode_attn_multiseq without a caller workspace.  The pages have no
 * counterpart: this entry point exists for callers that cannot allocate
 * device memory themselves (a serving loop that must not call cudaMalloc
 * once it is running, or a host runtime whose device allocator is not
 * reachable from C).  Arguments, results and numerics are those of
 * luce_decode_attn_multiseq; only the scratch differs.
 *
 * The scratch is one fixed array of luce_decode_attn_noalloc_max_bytes()
 * bytes (16 MiB) in the library's device memory; every GPU that loads the
 * library holds it until the process exits.  The call needs
 * (sum over rows of its chunk count) * Hq * 528 bytes of it (chunks as in
 * luce_decode_attn_multiseq) and returns LUCE_ENOSPACE, launching nothing,
 * when that exceeds the array (at Hq = 40: 4 rows of up to 32,768 keys, or
 * 16 rows of up to 2,051 keys, fit).  It allocates nothing: no cudaMalloc,
 * cudaFree or allocating library routine.  Nothing in the array needs to
 * start at zero: every chunk writes its partials before the merge reads
 * them, so the call clears nothing.
 *
 * The first call on each device (the calling thread's current device) looks
 * up the array's device address with cudaGetSymbolAddress; make that first
 * call before any stream capture.  All calls share the one array and it
 * keeps the last call's contents, so calls that can overlap on the GPU
 * (different streams without ordering between them) race: order them.
 */
int luce_decode_attn_multiseq_noalloc(const float* q, const luce_seqview* views, int n_seq,
                                      int Hq, int Hkv, int D, float scale, float* out, void* stream);

/* Size in bytes of the fixed scratch array of luce_decode_attn_multiseq_noalloc. */
size_t luce_decode_attn_noalloc_max_bytes(void);

/* ---------------------------------------------------------------- decode step */

/* One pre-norm decoder layer, all projections q8_0 (device pointers). */
typedef struct luce_layer {
    const float* attn_norm;                          /* [hidden] */
    const int8_t* wqkv_q; const uint16_t* wqkv_d;    /* [(Hq + 2 Hkv) D][hidden]: q rows, k rows, v rows */
    const int8_t* wo_q;   const uint16_t* wo_d;      /* [hidden][Hq D] */
    const float* ffn_norm;                           /* [hidden] */
    const int8_t* wgu_q;  const uint16_t* wgu_d;     /* [2 ffn][hidden]: gate rows first, then up */
    const int8_t* wdown_q; const uint16_t* wdown_d;  /* [hidden][ffn] */
} luce_layer;

typedef struct luce_model {
    int32_t n_layers, hidden, n_q_heads, n_kv_heads, head_dim, ffn, vocab; /* vocab 0: no head */
    float rms_eps;
    double rope_theta;
    const luce_layer* layers;                        /* (host) [n_layers] */
    const float* final_norm;                         /* (device) [hidden], when vocab > 0 */
    const int8_t* head_q; const uint16_t* head_d;    /* (device) [vocab][hidden], when vocab > 0 */
} luce_model;

/* A slot's K/V cache for all layers: binary16 [n_layers][n_kv_heads][cap][head_dim]. */
typedef struct luce_slot {
    uint16_t* k;    /* (device) */
    uint16_t* v;    /* (device) */
    int32_t len;    /* tokens already cached before this step */
    int32_t cap;
} luce_slot;

/* Byte offsets of the step's intermediates inside its workspace (the last
 * layer's values remain there after the call; useful for inspection). */
typedef struct luce_step_layout {
    size_t xn, xn_q, xn_d, qkv, q_rot, part, attn, attn_q, attn_d, x1,
           xn2, xn2_q, xn2_d, gu, h, h_q, h_d, xf, xf_q, xf_d, total;
} luce_step_layout;

/* Workspace layout for n_rows rows and caches of at most max_ctx positions. */
int luce_decode_step_layout(const luce_model* m, int n_rows, int max_ctx, luce_step_layout* out);

/*
 * One batched decode step through every layer [ds4-604, section 2: the dense
 * projections run once on the shared batch workspace with n_tokens = count,
 * KV append per sequence, one multi-sequence attention launch; logits land
 * one row per sequence].  slots (host) [n_seq] and rows_per_slot (host)
 * [n_seq]: slot s owns rows_per_slot[s] consecutive rows of x, in call order,
 * its row j at position slots[s].len + j.  For each layer:
 *   x1 = x + Wo . attn(rope(Wq . q8(norm(x))), cache)     (K/V rows appended)
 *   x  = x1 + Wdown . q8(silu(Wgate . q8(norm(x1))) * (Wup . q8(norm(x1))))
 * then, when vocab > 0 and logits/argmax are given, logits = Whead .
 * q8(norm(x)) and argmax (lowest index on ties).
 *   x      (device) fp32 [T][hidden], in: this step's hidden rows; out: the
 *          hidden state after the last layer
 *   logits (device) fp32 [T][vocab] or NULL;  argmax (device) int32 [T] or NULL
 * The cache rows [len, len + rows) of every listed slot are written; slots
 * are not otherwise touched and `len` is not updated (the caller commits the
 * accepted prefix).  1 <= n_seq <= LUCE_MAX_SEQ (5 or more is refused),
 * rows per slot 1..LUCE_MAX_ROWS_PER_SEQ, len + rows <= cap <= max_ctx of ws.
 */
int luce_decode_step(const luce_model* m, const luce_slot* slots, const int32_t* rows_per_slot,
                     int n_seq, float* x, float* logits, int32_t* argmax,
                     void* ws, size_t ws_bytes, void* stream);

/*
 * luce_decode_step with the rows' hidden states exchanged with the host, all
 * on the stream and without waiting: x_in (host, fp32 [T][hidden]) is copied
 * to x (device, the step's in/out rows), the step runs, then x is copied to
 * x_out (host, nullable) and argmax to argmax_out (host, nullable; needs
 * argmax).  A host buffer that is page-locked memory mapped into the device's
 * address space (cudaPointerGetAttributes gives a device address for all of
 * it; 16-byte aligned for x_out) is not copied by the copy engine: the first
 * RMSNorm reads x_in through the mapping (and fills x), and one kernel after
 * the last layer stores x_out and argmax_out through it.  Other buffers take
 * cudaMemcpyAsync (pageable ones then wait for the host).  Either way the
 * caller synchronises the stream before reading x_out.
 * Validation is luce_decode_step's (plus a non-null x_in); a refused call
 * enqueues nothing.
 */
int luce_decode_step_host(const luce_model* m, const luce_slot* slots, const int32_t* rows_per_slot, int n_seq,
                          const float* x_in, float* x, float* x_out, float* logits, int32_t* argmax,
                          int32_t* argmax_out, void* ws, size_t ws_bytes, void* stream);

/*
 * The step of luce_decode_step_host as one CUDA graph, for repeated steps over
 * the same slots and buffers [ds4-604, section 2; the step's launches are
 * the same ones].  A host call that issues the step's 9 or more launches
 * one by one costs tens of microseconds on the host per step; a graph is
 * started with one call.
 *
 * luce_step_graph_create binds the model, the slots' caches (k, v, cap; len
 * is taken per run), rows_per_slot, and the buffers of luce_decode_step_host
 * (x_in host, x device, x_out host or NULL, logits/argmax device or NULL,
 * argmax_out host or NULL, ws), validating them as luce_decode_step_host
 * would at the slots' given lengths; it makes no CUDA call.  All of them must
 * stay valid, unchanged and unmoved until luce_step_graph_destroy; *out is
 * the new object (NULL on error).
 *
 * luce_step_graph_run (lens: host int32 [n_seq], each slot's current length)
 * enqueues on the stream exactly what luce_decode_step_host would with those
 * lengths - every layer, with x_in read and x_out / argmax_out written through
 * their mapping - with the same kernels and arguments, hence the same bits.
 * The host buffers must be page-locked and mapped (else LUCE_EUNSUPPORTED,
 * checked at the first run).  The first run captures the
 * launches into a graph on a private stream; a later run whose launches form
 * the same sequence refreshes only the kernel nodes whose arguments changed
 * (positions, K/V destinations, attention rows and grids), otherwise it
 * captures anew.  Validation is luce_decode_step_host's; a refused run
 * enqueues nothing.  One object serves one thread at a time; runs on
 * different streams are not ordered with each other.
 *
 * luce_step_graph_stats: how many captures and node refreshes the object has
 * made, and the kernel nodes of its graph (each pointer nullable).
 * luce_step_graph_destroy releases the graph (NULL is accepted); the caller
 * first waits for the runs it enqueued.
 */
typedef struct luce_step_graph luce_step_graph;

int luce_step_graph_create(const luce_model* m, const luce_slot* slots, const int32_t* rows_per_slot, int n_seq,
                           const float* x_in, float* x, float* x_out, float* logits, int32_t* argmax,
                           int32_t* argmax_out, void* ws, size_t ws_bytes, luce_step_graph** out);
int luce_step_graph_run(luce_step_graph* g, const int32_t* lens, void* stream);
int luce_step_graph_stats(const luce_step_graph* g, int64_t* captures, int64_t* node_updates, int32_t* kernels);
int luce_step_graph_destroy(luce_step_graph* g);

/*
 * A slot whose K/V lives in pages of LUCE_PAGE_KEYS tokens: pool page p holds
 * binary16 [n_layers][n_kv_heads][128][head_dim], so token j's K in layer l,
 * KV head g is k_pool[((table[j / 128] * n_layers + l) * n_kv_heads + g)
 * * 128 * 128 + (j % 128) * 128 + d].  The table is given twice, identical:
 * on the device (read by attention) and on the host (where the step's rows
 * are appended).  n_table >= ceil((len + rows) / 128) entries, each in
 * [0, n_pages); the pages that receive this step's rows are referenced by no
 * other slot of the call.
 */
typedef struct luce_paged_slot {
    uint16_t* k_pool;              /* (device) [n_pages][n_layers][Hkv][128][128] */
    uint16_t* v_pool;              /* (device) */
    const int32_t* table;          /* (device) [n_table] */
    const int32_t* table_host;     /* (host)   [n_table], equal to table */
    int32_t n_table;
    int32_t n_pages;
    int32_t len;                   /* tokens already cached before this step */
} luce_paged_slot;

/*
 * luce_decode_step over paged slots: the same rows, outputs and bits as the
 * flat step over caches holding the same tokens.  ws is sized by
 * luce_decode_step_layout with max_ctx >= every len + rows.
 */
int luce_decode_step_paged(const luce_model* m, const luce_paged_slot* slots, const int32_t* rows_per_slot,
                           int n_seq, float* x, float* logits, int32_t* argmax,
                           void* ws, size_t ws_bytes, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* LUCE_H */
