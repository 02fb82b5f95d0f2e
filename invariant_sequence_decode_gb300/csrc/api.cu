// api.cu - the C ABI of libluce (see include/luce.h for the contract).
//
// Every entry point validates all of its arguments on the host before it
// enqueues anything; a refused call returns a negative status and leaves the
// stream untouched.  Nothing here allocates device memory or synchronises.
#include <math.h>
#include <stdarg.h>
#include <stdio.h>

#include <algorithm>
#include <atomic>
#include <mutex>
#include <new>
#include <string>

#include "../../include/luce.h"
#include "common.cuh"
#include "kernels.h"

using namespace luce;

static std::atomic<uint64_t> g_launches{0};
thread_local LaunchLog* luce::t_launch_log = nullptr;

// A recorded launch is not a launch: the step graph counts its kernel nodes
// when it launches the graph.
void luce::count_launches(int n)
{
    if (!t_launch_log) g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed);
}

RopeFreq luce::rope_freq(double theta)
{
    RopeFreq f;
    for (int i = 0; i < kHeadDim / 2; ++i) f.inv[i] = pow(theta, -2.0 * (double)i / (double)kHeadDim);
    return f;
}

namespace {

thread_local std::string g_err;

int fail(int code, const char* fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_err = buf;
    return code;
}

int ok()
{
    g_err.clear();
    return LUCE_OK;
}

int cuda_status(cudaError_t e, const char* what)
{
    if (e != cudaSuccess) return fail(LUCE_ECUDA, "%s: %s", what, cudaGetErrorString(e));
    return ok();
}

bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

#define REQUIRE(cond, code, ...) \
    do {                         \
        if (!(cond)) return fail(code, __VA_ARGS__); \
    } while (0)

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

constexpr int kPageKeys = LUCE_PAGE_KEYS;

int chunks_of(int len)
{
    const int ch = attn_chunk_keys(len);
    return (len + ch - 1) / ch;
}

// Largest chunk count of any row with at most max_len keys.
int max_chunks_upto(int max_len)
{
    int m = chunks_of(std::min(max_len, 16384));
    if (max_len > 16384) m = std::max(m, chunks_of(max_len));
    return m;
}

constexpr int kMaxKeys = 256 * kAttnMaxChunksPerRow;

}  // namespace

extern "C" {

const char* luce_last_error(void) { return g_err.c_str(); }

int luce_version(void) { return 10000; }

uint64_t luce_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

int luce_wait_timeouts(uint32_t* count, int reset)
{
    REQUIRE(count, LUCE_EINVAL, "wait_timeouts: null count");
    return cuda_status(read_wait_timeouts(count, reset != 0), "wait_timeouts");
}

int luce_test_wait_expiry(int64_t limit_ns, void* stream)
{
    REQUIRE(limit_ns >= 1000 && limit_ns <= 1000000000, LUCE_EINVAL,
            "test_wait_expiry: limit_ns=%lld outside 1 us .. 1 s", (long long)limit_ns);
    return cuda_status(launch_wait_expiry((uint64_t)limit_ns, (cudaStream_t)stream), "test_wait_expiry");
}

int luce_q8_quantize_act(const float* x, int T, int K, int64_t ldx, int8_t* q, float* d, void* stream)
{
    REQUIRE(x && q && d, LUCE_EINVAL, "quantize_act: null pointer");
    REQUIRE(T >= 1, LUCE_EINVAL, "quantize_act: T=%d must be >= 1", T);
    REQUIRE(K >= 32 && K % 32 == 0, LUCE_EINVAL, "quantize_act: K=%d must be a positive multiple of 32", K);
    REQUIRE(ldx >= K, LUCE_EINVAL, "quantize_act: ldx=%lld < K", (long long)ldx);
    REQUIRE(aligned(x, 4) && aligned(d, 4), LUCE_EINVAL, "quantize_act: x and d must be 4-byte aligned");
    return cuda_status(launch_quantize(x, T, K, ldx, q, d, false, (cudaStream_t)stream), "quantize_act");
}

int luce_q8_quantize_act_f16(const float* x, int T, int K, int64_t ldx, int8_t* q, uint16_t* d, void* stream)
{
    REQUIRE(x && q && d, LUCE_EINVAL, "quantize_act_f16: null pointer");
    REQUIRE(T >= 1, LUCE_EINVAL, "quantize_act_f16: T=%d must be >= 1", T);
    REQUIRE(K >= 32 && K % 32 == 0, LUCE_EINVAL, "quantize_act_f16: K=%d must be a positive multiple of 32", K);
    REQUIRE(ldx >= K, LUCE_EINVAL, "quantize_act_f16: ldx=%lld < K", (long long)ldx);
    REQUIRE(aligned(x, 4) && aligned(d, 2), LUCE_EINVAL, "quantize_act_f16: x must be 4- and d 2-byte aligned");
    return cuda_status(launch_quantize(x, T, K, ldx, q, d, true, (cudaStream_t)stream), "quantize_act_f16");
}

int luce_rmsnorm_q8(const float* x, int T, int H, const float* gamma, float eps, float* xn, int8_t* q, void* d,
                    int half_scale, void* stream)
{
    REQUIRE(x && gamma && xn && q && d, LUCE_EINVAL, "rmsnorm_q8: null pointer");
    REQUIRE(T >= 1 && T <= LUCE_MAX_ROWS, LUCE_EINVAL, "rmsnorm_q8: T=%d outside 1..%d", T, LUCE_MAX_ROWS);
    REQUIRE(H >= 32 && H % 32 == 0, LUCE_EINVAL, "rmsnorm_q8: H=%d must be a positive multiple of 32", H);
    REQUIRE(eps >= 0 && isfinite(eps), LUCE_EINVAL, "rmsnorm_q8: eps must be >= 0");
    REQUIRE(aligned(x, 4) && aligned(gamma, 4) && aligned(xn, 4) && aligned(d, half_scale ? 2 : 4), LUCE_EINVAL,
            "rmsnorm_q8: misaligned");
    return cuda_status(launch_rmsnorm_quant(x, T, H, gamma, eps, xn, q, d, half_scale != 0, (cudaStream_t)stream),
                       "rmsnorm_q8");
}

int luce_swiglu_q8(const float* gu, int T, int F, float* h, int8_t* q, void* d, int half_scale, void* stream)
{
    REQUIRE(gu && h && q && d, LUCE_EINVAL, "swiglu_q8: null pointer");
    REQUIRE(T >= 1, LUCE_EINVAL, "swiglu_q8: T=%d must be >= 1", T);
    REQUIRE(F >= 32 && F % 32 == 0, LUCE_EINVAL, "swiglu_q8: F=%d must be a positive multiple of 32", F);
    REQUIRE(aligned(gu, 4) && aligned(h, 4) && aligned(d, half_scale ? 2 : 4), LUCE_EINVAL, "swiglu_q8: misaligned");
    return cuda_status(launch_swiglu_quant(gu, T, F, h, q, d, half_scale != 0, (cudaStream_t)stream), "swiglu_q8");
}

static int check_matvec(const int8_t* wq, const uint16_t* wd, int N, int K, const int8_t* aq, const float* ad,
                        int T, const void* y, int64_t ldy, const char* who)
{
    REQUIRE(wq && wd && aq && ad && y, LUCE_EINVAL, "%s: null pointer", who);
    REQUIRE(N >= 1, LUCE_EINVAL, "%s: N=%d must be >= 1", who, N);
    REQUIRE(K >= 32 && K % 32 == 0, LUCE_EINVAL, "%s: K=%d must be a positive multiple of 32", who, K);
    REQUIRE(T >= 1 && T <= LUCE_MAX_ROWS, LUCE_EINVAL, "%s: T=%d outside 1..%d", who, T, LUCE_MAX_ROWS);
    REQUIRE(ldy >= N, LUCE_EINVAL, "%s: ldy=%lld < N", who, (long long)ldy);
    REQUIRE(aligned(wq, 32) && aligned(aq, 32), LUCE_EINVAL, "%s: wq and aq must be 32-byte aligned", who);
    REQUIRE(aligned(wd, 2) && aligned(ad, 4) && aligned(y, 4), LUCE_EINVAL, "%s: misaligned wd/ad/y", who);
    REQUIRE((int64_t)N * K < ((int64_t)1 << 40), LUCE_EINVAL, "%s: N*K too large", who);
    return LUCE_OK;
}

int luce_q8_matvec_batch(const int8_t* wq, const uint16_t* wd, int N, int K, const int8_t* aq, const float* ad,
                         int T, float* y, int64_t ldy, void* stream)
{
    int rc = check_matvec(wq, wd, N, K, aq, ad, T, y, ldy, "q8_matvec_batch");
    if (rc) return rc;
    return cuda_status(launch_matvec(wq, reinterpret_cast<const __half*>(wd), N, K, aq, ad, T, y, ldy, nullptr, 0,
                                     (cudaStream_t)stream),
                       "q8_matvec_batch");
}

int luce_q8_matvec_batch_path(const int8_t* wq, const uint16_t* wd, int N, int K, const int8_t* aq, const float* ad,
                              int T, float* y, int64_t ldy, int path, void* stream)
{
    int rc = check_matvec(wq, wd, N, K, aq, ad, T, y, ldy, "q8_matvec_batch_path");
    if (rc) return rc;
    REQUIRE(path >= LUCE_MATVEC_AUTO && path <= LUCE_MATVEC_TENSOR, LUCE_EINVAL, "q8_matvec_batch_path: path=%d",
            path);
    const cudaError_t e = launch_matvec_path(path, wq, reinterpret_cast<const __half*>(wd), N, K, aq, ad, T, y, ldy,
                                             nullptr, 0, (cudaStream_t)stream);
    REQUIRE(e != cudaErrorNotSupported, LUCE_EUNSUPPORTED,
            "q8_matvec_batch_path: kernel %d does not serve T=%d, K=%d at these alignments", path, T, K);
    return cuda_status(e, "q8_matvec_batch_path");
}

int luce_q8_block_dots(const int8_t* wq, int N, int K, const int8_t* aq, int T, int32_t* out, void* stream)
{
    REQUIRE(wq && aq && out, LUCE_EINVAL, "q8_block_dots: null pointer");
    REQUIRE(N >= 1 && T >= 1 && T <= LUCE_MAX_ROWS, LUCE_EINVAL, "q8_block_dots: bad N=%d or T=%d", N, T);
    REQUIRE(K >= 32 && K % 32 == 0, LUCE_EINVAL, "q8_block_dots: K=%d must be a positive multiple of 32", K);
    REQUIRE(aligned(wq, 32) && aligned(aq, 32) && aligned(out, 4), LUCE_EINVAL, "q8_block_dots: misaligned");
    return cuda_status(launch_block_dots(wq, N, K, aq, T, out, (cudaStream_t)stream), "q8_block_dots");
}

int luce_rope_posvec(float* x, int T, int n_heads, int D, int64_t ldx, const int32_t* pos, double theta,
                     void* stream)
{
    REQUIRE(x && pos, LUCE_EINVAL, "rope_posvec: null pointer");
    REQUIRE(D == LUCE_HEAD_DIM, LUCE_EUNSUPPORTED, "rope_posvec: head_dim %d (only %d)", D, LUCE_HEAD_DIM);
    REQUIRE(T >= 1 && n_heads >= 1, LUCE_EINVAL, "rope_posvec: T=%d n_heads=%d", T, n_heads);
    REQUIRE(ldx >= (int64_t)n_heads * D, LUCE_EINVAL, "rope_posvec: ldx too small");
    REQUIRE(theta > 0 && isfinite(theta), LUCE_EINVAL, "rope_posvec: theta must be positive");
    REQUIRE(aligned(x, 4) && aligned(pos, 4), LUCE_EINVAL, "rope_posvec: misaligned");
    return cuda_status(launch_rope_posvec(x, T, n_heads, ldx, pos, rope_freq(theta), (cudaStream_t)stream),
                       "rope_posvec");
}

// Validates views and returns the number of rows they cover (rows 0..T-1,
// each exactly once).
static int check_views(const luce_seqview* views, int n_seq, int Hkv, int D, int* T_out, const char* who)
{
    REQUIRE(views, LUCE_EINVAL, "%s: null views", who);
    REQUIRE(n_seq >= 1 && n_seq <= LUCE_MAX_SEQ, LUCE_EINVAL,
            "%s: n_seq=%d outside 1..%d (more than %d sequences are refused)", who, n_seq, LUCE_MAX_SEQ,
            LUCE_MAX_SEQ);
    REQUIRE(D == LUCE_HEAD_DIM, LUCE_EUNSUPPORTED, "%s: head_dim %d (only %d)", who, D, LUCE_HEAD_DIM);
    int covered[LUCE_MAX_ROWS] = {0};
    int T = 0;
    for (int s = 0; s < n_seq; ++s) {
        const luce_seqview& v = views[s];
        REQUIRE(v.k && v.v, LUCE_EINVAL, "%s: view %d has a null cache pointer", who, s);
        REQUIRE(aligned(v.k, 16) && aligned(v.v, 16), LUCE_EINVAL, "%s: view %d cache not 16-byte aligned", who, s);
        REQUIRE(v.n_q >= 1 && v.n_q <= LUCE_MAX_ROWS_PER_SEQ, LUCE_EINVAL, "%s: view %d n_q=%d outside 1..%d", who,
                s, v.n_q, LUCE_MAX_ROWS_PER_SEQ);
        REQUIRE(v.len >= v.n_q && v.len <= v.cap, LUCE_EINVAL, "%s: view %d len=%d outside [n_q, cap=%d]", who, s,
                v.len, v.cap);
        REQUIRE(v.len <= kMaxKeys, LUCE_EUNSUPPORTED, "%s: view %d has %d keys (at most %d)", who, s, v.len, kMaxKeys);
        REQUIRE(v.tok_stride >= D && v.tok_stride % 8 == 0 && v.head_stride % 8 == 0, LUCE_EINVAL,
                "%s: view %d strides must be multiples of 8 with tok_stride >= D", who, s);
        REQUIRE(v.head_stride >= (int64_t)v.cap * v.tok_stride || Hkv == 1, LUCE_EINVAL,
                "%s: view %d head_stride overlaps heads", who, s);
        REQUIRE(v.row0 >= 0 && v.row0 + v.n_q <= LUCE_MAX_ROWS, LUCE_EINVAL, "%s: view %d rows out of range", who, s);
        for (int j = 0; j < v.n_q; ++j) {
            REQUIRE(!covered[v.row0 + j], LUCE_EINVAL, "%s: row %d claimed twice", who, v.row0 + j);
            covered[v.row0 + j] = 1;
        }
        T = std::max(T, v.row0 + v.n_q);
    }
    for (int r = 0; r < T; ++r) REQUIRE(covered[r], LUCE_EINVAL, "%s: row %d belongs to no view", who, r);
    *T_out = T;
    return LUCE_OK;
}

int luce_kv_append(const float* k, const float* v, int64_t ldkv, int Hkv, int D, const luce_seqview* views,
                   int n_seq, void* stream)
{
    REQUIRE(k && v, LUCE_EINVAL, "kv_append: null k/v");
    REQUIRE(Hkv >= 1 && ldkv >= (int64_t)Hkv * D, LUCE_EINVAL, "kv_append: bad Hkv=%d or ldkv", Hkv);
    int T = 0;
    int rc = check_views(views, n_seq, Hkv, D, &T, "kv_append");
    if (rc) return rc;
    KvRows rows{};
    rows.n_rows = T;
    for (int s = 0; s < n_seq; ++s)
        for (int j = 0; j < views[s].n_q; ++j) {
            const int64_t p = views[s].len - views[s].n_q + j;
            KvRow& r = rows.row[views[s].row0 + j];
            r.k = reinterpret_cast<__half*>(views[s].k) + p * views[s].tok_stride;
            r.v = reinterpret_cast<__half*>(views[s].v) + p * views[s].tok_stride;
            r.head_stride = views[s].head_stride;
        }
    return cuda_status(launch_kv_append(k, v, ldkv, Hkv, rows, (cudaStream_t)stream), "kv_append");
}

// Attention scratch: the chunk partials (o[128], m, l per chunk and head).
size_t luce_decode_attn_workspace_size(int n_rows, int Hq, int D, int max_len)
{
    if (n_rows < 1 || Hq < 1 || D != LUCE_HEAD_DIM || max_len < 1) return 0;
    return attn_part_floats(n_rows * max_chunks_upto(max_len), Hq) * sizeof(float);
}

static void build_attn_rows(const luce_seqview* views, int n_seq, AttnRows& rows, int T)
{
    rows.n_rows = T;
    for (int s = 0; s < n_seq; ++s)
        for (int j = 0; j < views[s].n_q; ++j) {
            AttnRow& r = rows.row[views[s].row0 + j];
            r.k = reinterpret_cast<const __half*>(views[s].k);
            r.v = reinterpret_cast<const __half*>(views[s].v);
            r.head_stride = views[s].head_stride;
            r.tok_stride = views[s].tok_stride;
            r.len = views[s].len - views[s].n_q + 1 + j;
            r.chunk = attn_chunk_keys(r.len);
        }
    int c = 0;
    for (int r = 0; r < T; ++r) {
        rows.row[r].chunk0 = c;
        c += chunks_of(rows.row[r].len);
    }
    rows.total_chunks = c;
}

int luce_decode_attn_multiseq(const float* q, const luce_seqview* views, int n_seq, int Hq, int Hkv, int D,
                              float scale, float* out, void* ws, size_t ws_bytes, void* stream)
{
    REQUIRE(q && out && ws, LUCE_EINVAL, "decode_attn: null q/out/ws");
    REQUIRE(Hkv >= 1 && Hq >= Hkv && Hq % Hkv == 0, LUCE_EINVAL, "decode_attn: Hq=%d must be a multiple of Hkv=%d",
            Hq, Hkv);
    REQUIRE(Hq / Hkv <= 8, LUCE_EUNSUPPORTED, "decode_attn: group size %d > 8", Hq / Hkv);
    REQUIRE(isfinite(scale), LUCE_EINVAL, "decode_attn: scale must be finite");
    REQUIRE(aligned(q, 16) && aligned(out, 4) && aligned(ws, 16), LUCE_EINVAL, "decode_attn: misaligned q/out/ws");
    int T = 0;
    int rc = check_views(views, n_seq, Hkv, D, &T, "decode_attn");
    if (rc) return rc;
    AttnRows rows{};
    build_attn_rows(views, n_seq, rows, T);
    const size_t need = attn_part_floats(rows.total_chunks, Hq) * sizeof(float);
    REQUIRE(ws_bytes >= need, LUCE_ENOSPACE, "decode_attn: workspace %zu bytes < %zu needed", ws_bytes, need);
    return cuda_status(launch_attention(q, (int64_t)Hq * D, rows, Hq, Hkv, scale, (float*)ws, out, (int64_t)Hq * D,
                                        nullptr, nullptr, (cudaStream_t)stream),
                       "decode_attn");
}

int luce_decode_attn_paged(const float* q, const luce_pagedview* views, int n_seq, int Hq, int Hkv, int D,
                           float scale, float* out, void* ws, size_t ws_bytes, void* stream)
{
    const char* who = "decode_attn_paged";
    REQUIRE(q && out && ws && views, LUCE_EINVAL, "%s: null q/out/ws/views", who);
    REQUIRE(Hkv >= 1 && Hq >= Hkv && Hq % Hkv == 0, LUCE_EINVAL, "%s: Hq=%d must be a multiple of Hkv=%d", who, Hq,
            Hkv);
    REQUIRE(Hq / Hkv <= 8, LUCE_EUNSUPPORTED, "%s: group size %d > 8", who, Hq / Hkv);
    REQUIRE(D == LUCE_HEAD_DIM, LUCE_EUNSUPPORTED, "%s: head_dim %d (only %d)", who, D, LUCE_HEAD_DIM);
    REQUIRE(isfinite(scale), LUCE_EINVAL, "%s: scale must be finite", who);
    REQUIRE(aligned(q, 16) && aligned(out, 4) && aligned(ws, 16), LUCE_EINVAL, "%s: misaligned q/out/ws", who);
    REQUIRE(n_seq >= 1 && n_seq <= LUCE_MAX_SEQ, LUCE_EINVAL,
            "%s: n_seq=%d outside 1..%d (more than %d sequences are refused)", who, n_seq, LUCE_MAX_SEQ,
            LUCE_MAX_SEQ);
    int covered[LUCE_MAX_ROWS] = {0};
    int T = 0;
    AttnRows rows{};
    for (int s = 0; s < n_seq; ++s) {
        const luce_pagedview& v = views[s];
        REQUIRE(v.k_pool && v.v_pool && aligned(v.k_pool, 16) && aligned(v.v_pool, 16), LUCE_EINVAL,
                "%s: view %d pool null or not 16-byte aligned", who, s);
        REQUIRE(v.table && aligned(v.table, 4), LUCE_EINVAL, "%s: view %d table null", who, s);
        REQUIRE(v.n_q >= 1 && v.n_q <= LUCE_MAX_ROWS_PER_SEQ, LUCE_EINVAL, "%s: view %d n_q=%d outside 1..%d", who,
                s, v.n_q, LUCE_MAX_ROWS_PER_SEQ);
        REQUIRE(v.len >= v.n_q, LUCE_EINVAL, "%s: view %d len=%d < n_q", who, s, v.len);
        REQUIRE(v.len <= kMaxKeys, LUCE_EUNSUPPORTED, "%s: view %d has %d keys (at most %d)", who, s, v.len, kMaxKeys);
        REQUIRE(v.row0 >= 0 && v.row0 + v.n_q <= LUCE_MAX_ROWS, LUCE_EINVAL, "%s: view %d rows out of range", who, s);
        for (int j = 0; j < v.n_q; ++j) {
            REQUIRE(!covered[v.row0 + j], LUCE_EINVAL, "%s: row %d claimed twice", who, v.row0 + j);
            covered[v.row0 + j] = 1;
            AttnRow& r = rows.row[v.row0 + j];
            r.k = reinterpret_cast<const __half*>(v.k_pool);
            r.v = reinterpret_cast<const __half*>(v.v_pool);
            r.head_stride = (int64_t)kPageKeys * D;
            r.tok_stride = D;
            r.len = v.len - v.n_q + 1 + j;
            r.chunk = attn_chunk_keys(r.len);
            r.pages = v.table;
            r.page_stride = (int64_t)Hkv * kPageKeys * D;
        }
        T = std::max(T, v.row0 + v.n_q);
    }
    for (int r = 0; r < T; ++r) REQUIRE(covered[r], LUCE_EINVAL, "%s: row %d belongs to no view", who, r);
    rows.n_rows = T;
    int c = 0;
    for (int r = 0; r < T; ++r) {
        rows.row[r].chunk0 = c;
        c += chunks_of(rows.row[r].len);
    }
    rows.total_chunks = c;
    const size_t need = attn_part_floats(rows.total_chunks, Hq) * sizeof(float);
    REQUIRE(ws_bytes >= need, LUCE_ENOSPACE, "%s: workspace %zu bytes < %zu needed", who, ws_bytes, need);
    return cuda_status(launch_attention(q, (int64_t)Hq * D, rows, Hq, Hkv, scale, (float*)ws, out, (int64_t)Hq * D,
                                        nullptr, nullptr, (cudaStream_t)stream),
                       who);
}

// ------------------------------------------------------------ attention, no allocation
//
// For callers that cannot allocate device memory themselves (a real-time
// serving loop that must not call cudaMalloc after start-up, an embedding
// runtime whose allocator is not reachable from C): the split-K scratch lives
// in this fixed, file-scope device array instead of a caller workspace.  The
// host-side name of the array is only a stand-in; its device address is
// looked up once per device with cudaGetSymbolAddress.

static constexpr size_t kNoAllocScratchBytes = (size_t)16 << 20;
static constexpr int kNoAllocMaxDevices = 64;
static __device__ __align__(256) unsigned char g_attn_noalloc_scratch[kNoAllocScratchBytes];
static std::mutex g_noalloc_mu;
static void* g_noalloc_ptr[kNoAllocMaxDevices] = {};

static int noalloc_scratch(void** out)
{
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_status(e, "decode_attn_noalloc: cudaGetDevice");
    REQUIRE(dev >= 0 && dev < kNoAllocMaxDevices, LUCE_EUNSUPPORTED, "decode_attn_noalloc: device %d >= %d", dev,
            kNoAllocMaxDevices);
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_attn_noalloc_scratch);
        if (e != cudaSuccess) return cuda_status(e, "decode_attn_noalloc: cudaGetSymbolAddress");
        REQUIRE(p != nullptr, LUCE_ECUDA, "decode_attn_noalloc: null scratch address");
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return LUCE_OK;
}

size_t luce_decode_attn_noalloc_max_bytes(void) { return kNoAllocScratchBytes; }

int luce_decode_attn_multiseq_noalloc(const float* q, const luce_seqview* views, int n_seq, int Hq, int Hkv, int D,
                                      float scale, float* out, void* stream)
{
    const char* who = "decode_attn_noalloc";
    REQUIRE(q && out, LUCE_EINVAL, "%s: null q/out", who);
    REQUIRE(Hkv >= 1 && Hq >= Hkv && Hq % Hkv == 0, LUCE_EINVAL, "%s: Hq=%d must be a multiple of Hkv=%d", who, Hq,
            Hkv);
    REQUIRE(Hq / Hkv <= 8, LUCE_EUNSUPPORTED, "%s: group size %d > 8", who, Hq / Hkv);
    REQUIRE(isfinite(scale), LUCE_EINVAL, "%s: scale must be finite", who);
    REQUIRE(aligned(q, 16) && aligned(out, 4), LUCE_EINVAL, "%s: misaligned q/out", who);
    int T = 0;
    int rc = check_views(views, n_seq, Hkv, D, &T, who);
    if (rc) return rc;
    AttnRows rows{};
    build_attn_rows(views, n_seq, rows, T);
    const size_t need = attn_part_floats(rows.total_chunks, Hq) * sizeof(float);
    REQUIRE(need <= kNoAllocScratchBytes, LUCE_ENOSPACE,
            "%s: needs %zu bytes of scratch, more than the fixed %zu-byte array (fewer rows, shorter contexts or "
            "fewer heads fit)",
            who, need, kNoAllocScratchBytes);
    void* scratch = nullptr;
    rc = noalloc_scratch(&scratch);
    if (rc) return rc;
    return cuda_status(launch_attention(q, (int64_t)Hq * D, rows, Hq, Hkv, scale, (float*)scratch, out,
                                        (int64_t)Hq * D, nullptr, nullptr, (cudaStream_t)stream),
                       who);
}

// ------------------------------------------------------------ decode step

static int check_model(const luce_model* m, const char* who)
{
    REQUIRE(m, LUCE_EINVAL, "%s: null model", who);
    REQUIRE(m->n_layers >= 0 && m->hidden >= 32 && m->hidden % 32 == 0, LUCE_EINVAL,
            "%s: hidden=%d must be a positive multiple of 32", who, m->hidden);
    REQUIRE(m->head_dim == LUCE_HEAD_DIM, LUCE_EUNSUPPORTED, "%s: head_dim %d (only %d)", who, m->head_dim,
            LUCE_HEAD_DIM);
    REQUIRE(m->n_kv_heads >= 1 && m->n_q_heads % m->n_kv_heads == 0 && m->n_q_heads / m->n_kv_heads <= 8,
            LUCE_EUNSUPPORTED, "%s: heads %d/%d (need Hq %% Hkv == 0, group <= 8)", who, m->n_q_heads,
            m->n_kv_heads);
    REQUIRE(m->ffn >= 32 && m->ffn % 32 == 0, LUCE_EINVAL, "%s: ffn=%d must be a positive multiple of 32", who,
            m->ffn);
    REQUIRE(m->vocab >= 0, LUCE_EINVAL, "%s: vocab < 0", who);
    REQUIRE(m->n_layers == 0 || m->layers, LUCE_EINVAL, "%s: null layer table", who);
    REQUIRE(m->rope_theta > 0 && isfinite(m->rope_theta), LUCE_EINVAL, "%s: rope_theta must be positive", who);
    REQUIRE(m->rms_eps >= 0 && isfinite(m->rms_eps), LUCE_EINVAL, "%s: rms_eps must be >= 0", who);
    return LUCE_OK;
}

static void layout_of(const luce_model* m, int T, int max_ctx, luce_step_layout* L)
{
    const size_t H = m->hidden, Hq = m->n_q_heads, Hkv = m->n_kv_heads, D = m->head_dim, F = m->ffn;
    size_t o = 0;
    auto take = [&](size_t bytes) {
        size_t at = o;
        o = align_up(o + bytes, 256);
        return at;
    };
    L->xn = take(T * H * 4);
    L->xn_q = take(T * H);
    L->xn_d = take(T * H / 32 * 4);
    L->qkv = take(T * (Hq + 2 * Hkv) * D * 4);
    L->q_rot = take(T * Hq * D * 4);
    L->attn = take(T * Hq * D * 4);
    L->attn_q = take(T * Hq * D);
    L->attn_d = take(T * Hq * D / 32 * 4);
    L->x1 = take(T * H * 4);
    L->xn2 = take(T * H * 4);
    L->xn2_q = take(T * H);
    L->xn2_d = take(T * H / 32 * 4);
    L->gu = take(T * 2 * F * 4);
    L->h = take(T * F * 4);
    L->h_q = take(T * F);
    L->h_d = take(T * F / 32 * 4);
    L->xf = take(T * H * 4);
    L->xf_q = take(T * H);
    L->xf_d = take(T * H / 32 * 4);
    // The split-K scratch comes last so that the offsets above do not depend
    // on the context bound.
    L->part = take(attn_part_floats(T * max_chunks_upto(std::max(max_ctx, 1)), (int)Hq) * 4);
    L->total = o;
}

int luce_decode_step_layout(const luce_model* m, int n_rows, int max_ctx, luce_step_layout* out)
{
    int rc = check_model(m, "decode_step_layout");
    if (rc) return rc;
    REQUIRE(out, LUCE_EINVAL, "decode_step_layout: null out");
    REQUIRE(n_rows >= 1 && n_rows <= LUCE_MAX_ROWS, LUCE_EINVAL, "decode_step_layout: n_rows=%d outside 1..%d",
            n_rows, LUCE_MAX_ROWS);
    REQUIRE(max_ctx >= 1, LUCE_EINVAL, "decode_step_layout: max_ctx=%d", max_ctx);
    layout_of(m, n_rows, max_ctx, out);
    return ok();
}

// A slot as the step addresses it: a flat cache [n_layers][Hkv][cap][D], or
// pages of kPageKeys tokens [n_pages][n_layers][Hkv][kPageKeys][D] named by
// a table (device copy for attention, host copy for the appends).
struct StepSlot {
    __half* k;
    __half* v;
    int len;
    int cap;
    const int32_t* table;       // nullptr for a flat cache
    const int32_t* table_host;
};

// A host<->device copy of the step: issued on the stream, or written to the
// launch log while one is being recorded.
static cudaError_t step_copy(void* dst, const void* src, size_t bytes, cudaMemcpyKind dir, cudaStream_t st)
{
    if (LaunchLog* log = t_launch_log) {
        log->recs.emplace_back();
        LaunchRec& r = log->recs.back();
        r.copy = true;
        r.func = nullptr;
        r.grid = r.block = dim3(0, 0, 0);
        r.smem = 0;
        r.nargs = r.nbytes = 0;
        r.dst = dst;
        r.src = src;
        r.bytes = bytes;
        r.dir = dir;
        return cudaSuccess;
    }
    return cudaMemcpyAsync(dst, src, bytes, dir, st);
}

// Host buffers of luce_decode_step_host (all nullable): the step's input rows,
// and where its output rows and argmax are copied back.  The *_dev members
// are their device addresses when the buffers are page-locked memory mapped
// into the device's address space (resolve_io): the step's kernels then read
// x_in and write x_out / argmax_out directly, over the host link, in place of
// copy-engine transfers.
struct HostIO {
    const float* x_in;
    float* x_out;
    int32_t* argmax_out;
    const float* x_in_dev = nullptr;
    float* x_out_dev = nullptr;
    int32_t* argmax_out_dev = nullptr;
    bool outputs_resolved = false;  // else the step looks the output views up after its launches
};

// The device address of host buffer [p, p + bytes) when all of it is mapped
// page-locked memory and that address is `align`-aligned, else nullptr.
static void* device_view(const void* p, size_t bytes, size_t align)
{
    if (!p || bytes == 0) return nullptr;
    cudaPointerAttributes a0, a1;
    if (cudaPointerGetAttributes(&a0, p) != cudaSuccess ||
        cudaPointerGetAttributes(&a1, (const char*)p + bytes - 1) != cudaSuccess) {
        (void)cudaGetLastError();
        return nullptr;
    }
    if (a0.type != cudaMemoryTypeHost || a1.type != cudaMemoryTypeHost || !a0.devicePointer || !a1.devicePointer)
        return nullptr;
    if ((const char*)a1.devicePointer - (const char*)a0.devicePointer != (ptrdiff_t)(bytes - 1)) return nullptr;
    if ((uintptr_t)a0.devicePointer % align != 0) return nullptr;
    return a0.devicePointer;
}

static void resolve_input(HostIO* io, int T, int H)
{
    io->x_in_dev = (const float*)device_view(io->x_in, (size_t)T * H * sizeof(float), 4);
}

static void resolve_outputs(HostIO* io, int T, int H)
{
    io->x_out_dev = (float*)device_view(io->x_out, (size_t)T * H * sizeof(float), 16);
    io->argmax_out_dev = (int32_t*)device_view(io->argmax_out, (size_t)T * sizeof(int32_t), 4);
    io->outputs_resolved = true;
}

// The step's own argument checks (the slots are checked by the callers):
// buffers, weights, row count and workspace size.  On success *L is the
// workspace layout and *T the row count.
static int check_step(const luce_model* m, const StepSlot* slots, const int32_t* rows_per_slot, int n_seq, float* x,
                      float* logits, int32_t* argmax, void* ws, size_t ws_bytes, const char* who, const HostIO& io,
                      luce_step_layout* L, int* T_out)
{
    REQUIRE(x && ws, LUCE_EINVAL, "%s: null x/ws", who);
    REQUIRE(aligned(x, 16) && aligned(ws, 256), LUCE_EINVAL, "%s: x must be 16-byte and ws 256-byte aligned", who);
    REQUIRE(!(logits || argmax) || (m->vocab > 0 && m->final_norm && m->head_q && m->head_d), LUCE_EINVAL,
            "%s: logits/argmax need vocab > 0 and the head weights", who);
    REQUIRE(!argmax || logits, LUCE_EINVAL, "%s: argmax needs the logits buffer", who);
    REQUIRE(!io.argmax_out || argmax, LUCE_EINVAL, "%s: argmax_out needs the argmax buffer", who);
    int T = 0, max_len = 1;
    for (int s = 0; s < n_seq; ++s) {
        T += rows_per_slot[s];
        max_len = std::max(max_len, slots[s].len + rows_per_slot[s]);
    }
    REQUIRE(T <= LUCE_MAX_ROWS, LUCE_EINVAL, "%s: %d rows > %d", who, T, LUCE_MAX_ROWS);
    for (int l = 0; l < m->n_layers; ++l) {
        const luce_layer& w = m->layers[l];
        REQUIRE(w.attn_norm && w.wqkv_q && w.wqkv_d && w.wo_q && w.wo_d && w.ffn_norm && w.wgu_q && w.wgu_d &&
                    w.wdown_q && w.wdown_d,
                LUCE_EINVAL, "%s: layer %d has a null weight", who, l);
        REQUIRE(aligned(w.wqkv_q, 32) && aligned(w.wo_q, 32) && aligned(w.wgu_q, 32) && aligned(w.wdown_q, 32),
                LUCE_EINVAL, "%s: layer %d int8 weights must be 32-byte aligned", who, l);
    }
    REQUIRE(!logits || aligned(m->head_q, 32), LUCE_EINVAL, "%s: head weights must be 32-byte aligned", who);

    layout_of(m, T, max_len, L);
    REQUIRE(ws_bytes >= L->total, LUCE_ENOSPACE, "%s: workspace %zu bytes < %zu needed", who, ws_bytes, L->total);
    *T_out = T;
    return LUCE_OK;
}

static int decode_step_impl(const luce_model* m, const StepSlot* slots, const int32_t* rows_per_slot, int n_seq,
                            float* x, float* logits, int32_t* argmax, void* ws, size_t ws_bytes, void* stream,
                            const char* who, const HostIO& io = HostIO{nullptr, nullptr, nullptr})
{
    luce_step_layout L;
    int T = 0;
    const int rc = check_step(m, slots, rows_per_slot, n_seq, x, logits, argmax, ws, ws_bytes, who, io, &L, &T);
    if (rc) return rc;
    const int H = m->hidden, Hq = m->n_q_heads, Hkv = m->n_kv_heads, D = m->head_dim, F = m->ffn;

    char* wsb = (char*)ws;
    float* xn = (float*)(wsb + L.xn);
    int8_t* xn_q = (int8_t*)(wsb + L.xn_q);
    float* xn_d = (float*)(wsb + L.xn_d);
    float* qkv = (float*)(wsb + L.qkv);
    float* q_rot = (float*)(wsb + L.q_rot);
    float* part = (float*)(wsb + L.part);
    float* attn = (float*)(wsb + L.attn);
    int8_t* attn_q = (int8_t*)(wsb + L.attn_q);
    float* attn_d = (float*)(wsb + L.attn_d);
    float* x1 = (float*)(wsb + L.x1);
    float* xn2 = (float*)(wsb + L.xn2);
    int8_t* xn2_q = (int8_t*)(wsb + L.xn2_q);
    float* xn2_d = (float*)(wsb + L.xn2_d);
    float* gu = (float*)(wsb + L.gu);
    float* hh = (float*)(wsb + L.h);
    int8_t* h_q = (int8_t*)(wsb + L.h_q);
    float* h_d = (float*)(wsb + L.h_d);
    cudaStream_t st = (cudaStream_t)stream;

    // Row bookkeeping (host): positions, K/V destinations, attention rows.
    RowPos pos{};
    pos.n_rows = T;
    int slot_of[LUCE_MAX_ROWS];
    {
        int r = 0;
        for (int s = 0; s < n_seq; ++s)
            for (int j = 0; j < rows_per_slot[s]; ++j, ++r) {
                slot_of[r] = s;
                pos.pos[r] = slots[s].len + j;
            }
    }
    // the 64 inverse frequencies of the model's theta, formed once per thread and theta
    thread_local double freq_theta = -1.0;
    thread_local RopeFreq freq;
    if (freq_theta != m->rope_theta) {
        freq = rope_freq(m->rope_theta);
        freq_theta = m->rope_theta;
    }
    cudaError_t e = cudaSuccess;
    // input rows: read from mapped host memory by the first RMSNorm (which
    // copies them into x), else copied in first
    const bool in_mapped = io.x_in && io.x_in_dev;
    if (io.x_in && !in_mapped &&
        (e = step_copy(x, io.x_in, (size_t)T * H * sizeof(float), cudaMemcpyHostToDevice, st)))
        return cuda_status(e, who);

    const float scale = (float)(1.0 / sqrt((double)D));
    const int64_t page_elems = (int64_t)Hkv * kPageKeys * D;   // one layer of one page
    const int64_t page_stride = (int64_t)m->n_layers * page_elems;
    for (int l = 0; l < m->n_layers; ++l) {
        const luce_layer& w = m->layers[l];
        KvRows kv{};
        AttnRows ar{};
        kv.n_rows = ar.n_rows = T;
        for (int r = 0; r < T; ++r) {
            const StepSlot& sl = slots[slot_of[r]];
            const int p = pos.pos[r];
            if (sl.table) {
                const int64_t at = (int64_t)sl.table_host[p / kPageKeys] * page_stride + (int64_t)l * page_elems +
                                   (int64_t)(p % kPageKeys) * D;
                kv.row[r].k = sl.k + at;
                kv.row[r].v = sl.v + at;
                kv.row[r].head_stride = (int64_t)kPageKeys * D;
                ar.row[r].k = sl.k + (int64_t)l * page_elems;
                ar.row[r].v = sl.v + (int64_t)l * page_elems;
                ar.row[r].head_stride = (int64_t)kPageKeys * D;
                ar.row[r].pages = sl.table;
                ar.row[r].page_stride = page_stride;
            } else {
                const int64_t head_stride = (int64_t)sl.cap * D;
                const int64_t layer_off = (int64_t)l * Hkv * head_stride;
                __half* kb = sl.k + layer_off;
                __half* vb = sl.v + layer_off;
                kv.row[r].k = kb + (int64_t)p * D;
                kv.row[r].v = vb + (int64_t)p * D;
                kv.row[r].head_stride = head_stride;
                ar.row[r].k = kb;
                ar.row[r].v = vb;
                ar.row[r].head_stride = head_stride;
                ar.row[r].pages = nullptr;
                ar.row[r].page_stride = 0;
            }
            ar.row[r].tok_stride = D;
            ar.row[r].len = p + 1;
            ar.row[r].chunk = attn_chunk_keys(ar.row[r].len);
        }
        int c = 0;
        for (int r = 0; r < T; ++r) {
            ar.row[r].chunk0 = c;
            c += chunks_of(ar.row[r].len);
        }
        ar.total_chunks = c;

        const bool from_host = l == 0 && in_mapped;
        if ((e = launch_rmsnorm_quant(from_host ? io.x_in_dev : x, T, H, w.attn_norm, m->rms_eps, xn, xn_q, xn_d,
                                      false, st, from_host ? x : nullptr)))
            break;
        if ((e = launch_qkv_rope(w.wqkv_q, (const __half*)w.wqkv_d, H, xn_q, xn_d, T, qkv, Hq, Hkv, pos, freq, q_rot,
                                 kv, st)))
            break;
        if ((e = launch_attention(q_rot, (int64_t)Hq * D, ar, Hq, Hkv, scale, part, attn, (int64_t)Hq * D,
                                  attn_q, attn_d, st)))
            break;
        if ((e = launch_matvec(w.wo_q, (const __half*)w.wo_d, H, Hq * D, attn_q, attn_d, T, x1, H, x, H, st)))
            break;
        if ((e = launch_rmsnorm_quant(x1, T, H, w.ffn_norm, m->rms_eps, xn2, xn2_q, xn2_d, false, st))) break;
        // gate||up with SwiGLU and its codes in one launch where the fused ring
        // takes the shape, else the projection and then the SwiGLU kernel
        e = launch_gateup_swiglu_tma(w.wgu_q, (const __half*)w.wgu_d, F, H, xn2_q, xn2_d, T, gu, hh, h_q, h_d, st);
        if (e == cudaErrorNotSupported) {
            (void)cudaGetLastError();
            if ((e = launch_matvec(w.wgu_q, (const __half*)w.wgu_d, 2 * F, H, xn2_q, xn2_d, T, gu, 2 * F, nullptr, 0,
                                   st)))
                break;
            e = launch_swiglu_quant(gu, T, F, hh, h_q, h_d, false, st);
        }
        if (e) break;
        if ((e = launch_matvec(w.wdown_q, (const __half*)w.wdown_d, H, F, h_q, h_d, T, x, H, x1, H, st))) break;
    }
    if (e != cudaSuccess) return cuda_status(e, who);

    if (logits) {
        float* xf = (float*)(wsb + L.xf);
        int8_t* xf_q = (int8_t*)(wsb + L.xf_q);
        float* xf_d = (float*)(wsb + L.xf_d);
        if ((e = launch_rmsnorm_quant(x, T, H, m->final_norm, m->rms_eps, xf, xf_q, xf_d, false, st)))
            return cuda_status(e, who);
        if ((e = launch_matvec(m->head_q, (const __half*)m->head_d, m->vocab, H, xf_q, xf_d, T, logits, m->vocab,
                               nullptr, 0, st)))
            return cuda_status(e, who);
        if (argmax && (e = launch_argmax(logits, T, m->vocab, argmax, st))) return cuda_status(e, who);
    }
    // results: stored into mapped host memory by one kernel, else copied back
    HostIO out = io;
    if (!out.outputs_resolved) resolve_outputs(&out, T, H);  // off the path to the first launch
    float* xo = out.x_out ? out.x_out_dev : nullptr;
    int32_t* ao = out.argmax_out ? out.argmax_out_dev : nullptr;
    if ((xo || ao) && (e = launch_rows_to_host(x, (int64_t)T * H, xo, argmax, T, ao, st))) return cuda_status(e, who);
    if (io.x_out && !xo &&
        (e = step_copy(io.x_out, x, (size_t)T * H * sizeof(float), cudaMemcpyDeviceToHost, st)))
        return cuda_status(e, who);
    if (io.argmax_out && !ao &&
        (e = step_copy(io.argmax_out, argmax, (size_t)T * sizeof(int32_t), cudaMemcpyDeviceToHost, st)))
        return cuda_status(e, who);
    return ok();
}

static int check_rows(const int32_t* rows_per_slot, int s, const char* who)
{
    const int n = rows_per_slot[s];
    REQUIRE(n >= 1 && n <= LUCE_MAX_ROWS_PER_SEQ, LUCE_EINVAL, "%s: slot %d has %d rows (1..%d)", who, s, n,
            LUCE_MAX_ROWS_PER_SEQ);
    return LUCE_OK;
}

// Validates flat slots into ss; LUCE_OK or the refusal.
static int flat_slots(const luce_model* m, const luce_slot* slots, const int32_t* rows_per_slot, int n_seq,
                      StepSlot* ss, const char* who)
{
    int rc = check_model(m, who);
    if (rc) return rc;
    REQUIRE(slots && rows_per_slot, LUCE_EINVAL, "%s: null slots/rows", who);
    REQUIRE(n_seq >= 1 && n_seq <= LUCE_MAX_SEQ, LUCE_EINVAL,
            "%s: n_seq=%d outside 1..%d (more than %d slots are refused)", who, n_seq, LUCE_MAX_SEQ, LUCE_MAX_SEQ);
    for (int s = 0; s < n_seq; ++s) {
        const luce_slot& sl = slots[s];
        if ((rc = check_rows(rows_per_slot, s, who))) return rc;
        const int n = rows_per_slot[s];
        REQUIRE(sl.k && sl.v && aligned(sl.k, 16) && aligned(sl.v, 16), LUCE_EINVAL,
                "%s: slot %d cache null or not 16-byte aligned", who, s);
        REQUIRE(sl.len >= 0 && sl.cap >= 1 && (int64_t)sl.len + n <= sl.cap, LUCE_EINVAL,
                "%s: slot %d len=%d + rows=%d exceeds cap=%d", who, s, sl.len, n, sl.cap);
        REQUIRE(sl.len + n <= kMaxKeys, LUCE_EUNSUPPORTED, "%s: slot %d would hold %d keys (at most %d)", who, s,
                sl.len + n, kMaxKeys);
        ss[s] = StepSlot{reinterpret_cast<__half*>(sl.k), reinterpret_cast<__half*>(sl.v), sl.len, sl.cap, nullptr,
                         nullptr};
    }
    // Every K and V cache of the call is a byte range [base, base + extent)
    // with extent = n_layers * Hkv * cap * D binary16 values; no two of them
    // (two slots, or one slot's K and V) may overlap, or one slot's appends
    // would land in another's keys and break the untouched-slot guarantee.
    struct Range {
        uintptr_t lo, hi;
        int slot;
        char which;
    } r[2 * LUCE_MAX_SEQ];
    for (int s = 0; s < n_seq; ++s) {
        const uint64_t extent = (uint64_t)m->n_layers * m->n_kv_heads * (uint64_t)slots[s].cap * m->head_dim * 2;
        r[2 * s] = Range{(uintptr_t)slots[s].k, (uintptr_t)slots[s].k + extent, s, 'K'};
        r[2 * s + 1] = Range{(uintptr_t)slots[s].v, (uintptr_t)slots[s].v + extent, s, 'V'};
    }
    for (int a = 0; a < 2 * n_seq; ++a)
        for (int b = 0; b < a; ++b)
            REQUIRE(r[a].hi <= r[b].lo || r[b].hi <= r[a].lo || r[a].lo == r[a].hi || r[b].lo == r[b].hi,
                    LUCE_EINVAL, "%s: the %c cache of slot %d overlaps the %c cache of slot %d", who, r[a].which,
                    r[a].slot, r[b].which, r[b].slot);
    return LUCE_OK;
}

int luce_decode_step(const luce_model* m, const luce_slot* slots, const int32_t* rows_per_slot, int n_seq,
                     float* x, float* logits, int32_t* argmax, void* ws, size_t ws_bytes, void* stream)
{
    const char* who = "decode_step";
    StepSlot ss[LUCE_MAX_SEQ];
    const int rc = flat_slots(m, slots, rows_per_slot, n_seq, ss, who);
    if (rc) return rc;
    return decode_step_impl(m, ss, rows_per_slot, n_seq, x, logits, argmax, ws, ws_bytes, stream, who);
}

int luce_decode_step_host(const luce_model* m, const luce_slot* slots, const int32_t* rows_per_slot, int n_seq,
                          const float* x_in, float* x, float* x_out, float* logits, int32_t* argmax,
                          int32_t* argmax_out, void* ws, size_t ws_bytes, void* stream)
{
    const char* who = "decode_step_host";
    REQUIRE(x_in, LUCE_EINVAL, "%s: null x_in", who);
    StepSlot ss[LUCE_MAX_SEQ];
    const int rc = flat_slots(m, slots, rows_per_slot, n_seq, ss, who);
    if (rc) return rc;
    HostIO io{x_in, x_out, argmax_out};
    int T = 0;
    for (int s = 0; s < n_seq; ++s) T += rows_per_slot[s];
    resolve_input(&io, T, m->hidden);
    return decode_step_impl(m, ss, rows_per_slot, n_seq, x, logits, argmax, ws, ws_bytes, stream, who, io);
}

// ------------------------------------------------------------ step graph
//
// The step's launches and copies, recorded (not issued) by decode_step_impl,
// become the nodes of one CUDA graph: built once by capturing the recorded
// launches on a private stream, then, for every later step whose record has
// the same sequence of nodes (the same kernel count and copies), refreshed
// node by node - only the kernel nodes whose function, grid, block or
// argument bytes changed (the positions, K/V destinations and attention rows
// follow the slots' lengths) - and launched with one call.  A record with a
// different sequence (an attention kind appearing or leaving) is captured
// anew.  The graph's kernels are the very kernels, with the very arguments,
// that luce_decode_step_host would launch, so the outputs are its bits.

}  // extern "C"

struct luce_step_graph {
    const luce_model* m;
    luce_slot slots[LUCE_MAX_SEQ];
    int32_t rows[LUCE_MAX_SEQ];
    int n_seq;
    float* x;
    float* logits;
    int32_t* argmax;
    void* ws;
    size_t ws_bytes;
    HostIO io;
    bool io_resolved = false;    // io's device views are looked up at the first run
    cudaStream_t cap = nullptr;  // private capture stream
    cudaGraph_t graph = nullptr;
    cudaGraphExec_t exec = nullptr;
    std::vector<cudaGraphNode_t> nodes;  // graph nodes in launch order
    LaunchLog live;                      // the record the executable graph holds
    LaunchLog next;                      // this step's record
    int kernels = 0;
    int64_t captures = 0, node_updates = 0;
};

namespace {

void release_graph(luce_step_graph* g)
{
    if (g->exec) cudaGraphExecDestroy(g->exec);
    if (g->graph) cudaGraphDestroy(g->graph);
    g->exec = nullptr;
    g->graph = nullptr;
    g->nodes.clear();
}

bool same_kernel(const LaunchRec& a, const LaunchRec& b)
{
    return a.func == b.func && a.grid.x == b.grid.x && a.grid.y == b.grid.y && a.grid.z == b.grid.z &&
           a.block.x == b.block.x && a.block.y == b.block.y && a.block.z == b.block.z && a.smem == b.smem &&
           a.nargs == b.nargs && a.nbytes == b.nbytes && memcmp(a.off, b.off, sizeof(uint16_t) * a.nargs) == 0 &&
           memcmp(a.args, b.args, (size_t)a.nbytes) == 0;
}

// The same sequence of nodes: equal length, kernels where kernels were, and
// the same copies.
bool same_nodes(const LaunchLog& a, const LaunchLog& b)
{
    if (a.recs.size() != b.recs.size()) return false;
    for (size_t i = 0; i < a.recs.size(); ++i) {
        const LaunchRec &x = a.recs[i], &y = b.recs[i];
        if (x.copy != y.copy) return false;
        if (x.copy && (x.dst != y.dst || x.src != y.src || x.bytes != y.bytes || x.dir != y.dir)) return false;
    }
    return true;
}

void argv_of(LaunchRec& r, void** argv)
{
    for (int i = 0; i < r.nargs; ++i) argv[i] = r.args + r.off[i];
}

// Capture g->next into a new executable graph (the old one is released
// first); the nodes are then listed by walking the chain from its root.
cudaError_t capture(luce_step_graph* g)
{
    release_graph(g);
    cudaError_t e = cudaSuccess;
    if (!g->cap && (e = cudaStreamCreateWithFlags(&g->cap, cudaStreamNonBlocking))) return e;
    if ((e = cudaStreamBeginCapture(g->cap, cudaStreamCaptureModeThreadLocal))) return e;
    cudaError_t le = cudaSuccess;
    for (LaunchRec& r : g->next.recs) {
        if (r.copy) {
            le = cudaMemcpyAsync(r.dst, r.src, r.bytes, r.dir, g->cap);
        } else {
            void* argv[LaunchRec::kMaxArgs];
            argv_of(r, argv);
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = r.grid;
            cfg.blockDim = r.block;
            cfg.dynamicSmemBytes = r.smem;
            cfg.stream = g->cap;
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
            attr[0].val.programmaticStreamSerializationAllowed = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            le = cudaLaunchKernelExC(&cfg, r.func, argv);
        }
        if (le) break;
    }
    cudaGraph_t graph = nullptr;
    e = cudaStreamEndCapture(g->cap, &graph);
    if (le || e) {
        if (graph) cudaGraphDestroy(graph);
        return le ? le : e;
    }
    g->graph = graph;
    size_t n = 1;
    cudaGraphNode_t node = nullptr;
    if ((e = cudaGraphGetRootNodes(graph, &node, &n))) return e;
    while (n == 1 && node) {
        g->nodes.push_back(node);
        cudaGraphNode_t dep[2] = {nullptr, nullptr};
        cudaGraphEdgeData ed[2];
        n = 2;
        if ((e = cudaGraphNodeGetDependentNodes(node, dep, ed, &n))) return e;
        node = n == 1 ? dep[0] : nullptr;
    }
    if (n > 1 || g->nodes.size() != g->next.recs.size()) return cudaErrorInvalidValue;
    for (size_t i = 0; i < g->nodes.size(); ++i) {
        cudaGraphNodeType t;
        if ((e = cudaGraphNodeGetType(g->nodes[i], &t))) return e;
        if (t != (g->next.recs[i].copy ? cudaGraphNodeTypeMemcpy : cudaGraphNodeTypeKernel))
            return cudaErrorInvalidValue;
    }
    if ((e = cudaGraphInstantiate(&g->exec, graph, 0))) return e;
    g->kernels = 0;
    for (const LaunchRec& r : g->next.recs) g->kernels += r.copy ? 0 : 1;
    ++g->captures;
    return cudaSuccess;
}

// Refresh the executable graph from g->next, node by node; false when a node
// refused the new parameters (the caller then captures anew).
bool refresh(luce_step_graph* g)
{
    for (size_t i = 0; i < g->next.recs.size(); ++i) {
        LaunchRec& r = g->next.recs[i];
        if (r.copy || same_kernel(r, g->live.recs[i])) continue;
        void* argv[LaunchRec::kMaxArgs];
        argv_of(r, argv);
        cudaKernelNodeParams p = {};
        p.func = const_cast<void*>(r.func);
        p.gridDim = r.grid;
        p.blockDim = r.block;
        p.sharedMemBytes = (unsigned)r.smem;
        p.kernelParams = argv;
        p.extra = nullptr;
        if (cudaGraphExecKernelNodeSetParams(g->exec, g->nodes[i], &p) != cudaSuccess) {
            (void)cudaGetLastError();
            return false;
        }
        ++g->node_updates;
    }
    return true;
}

}  // namespace

extern "C" {

int luce_step_graph_create(const luce_model* m, const luce_slot* slots, const int32_t* rows_per_slot, int n_seq,
                           const float* x_in, float* x, float* x_out, float* logits, int32_t* argmax,
                           int32_t* argmax_out, void* ws, size_t ws_bytes, luce_step_graph** out)
{
    const char* who = "step_graph_create";
    REQUIRE(out, LUCE_EINVAL, "%s: null out", who);
    *out = nullptr;
    REQUIRE(x_in, LUCE_EINVAL, "%s: null x_in", who);
    StepSlot ss[LUCE_MAX_SEQ];
    int rc = flat_slots(m, slots, rows_per_slot, n_seq, ss, who);
    if (rc) return rc;
    luce_step_layout L;
    int T = 0;
    if ((rc = check_step(m, ss, rows_per_slot, n_seq, x, logits, argmax, ws, ws_bytes, who,
                         HostIO{x_in, x_out, argmax_out}, &L, &T)))
        return rc;
    luce_step_graph* g = new (std::nothrow) luce_step_graph();
    REQUIRE(g, LUCE_ENOSPACE, "%s: out of host memory", who);
    g->m = m;
    for (int s = 0; s < n_seq; ++s) {
        g->slots[s] = slots[s];
        g->rows[s] = rows_per_slot[s];
    }
    g->n_seq = n_seq;
    g->x = x;
    g->logits = logits;
    g->argmax = argmax;
    g->ws = ws;
    g->ws_bytes = ws_bytes;
    g->io = HostIO{x_in, x_out, argmax_out};
    const size_t per_step = 4 + 12 * (size_t)m->n_layers;
    g->live.recs.reserve(per_step);
    g->next.recs.reserve(per_step);
    *out = g;
    return ok();
}

int luce_step_graph_run(luce_step_graph* g, const int32_t* lens, void* stream)
{
    const char* who = "step_graph_run";
    REQUIRE(g && lens, LUCE_EINVAL, "%s: null graph/lens", who);
    luce_slot sl[LUCE_MAX_SEQ];
    for (int s = 0; s < g->n_seq; ++s) {
        sl[s] = g->slots[s];
        sl[s].len = lens[s];
    }
    StepSlot ss[LUCE_MAX_SEQ];
    int rc = flat_slots(g->m, sl, g->rows, g->n_seq, ss, who);
    if (rc) return rc;
    if (!g->io_resolved) {
        int T = 0;
        for (int s = 0; s < g->n_seq; ++s) T += g->rows[s];
        resolve_input(&g->io, T, g->m->hidden);
        resolve_outputs(&g->io, T, g->m->hidden);
        g->io_resolved = true;
    }
    REQUIRE((!g->io.x_in || g->io.x_in_dev) && (!g->io.x_out || g->io.x_out_dev) &&
                (!g->io.argmax_out || g->io.argmax_out_dev),
            LUCE_EUNSUPPORTED, "%s: the host buffers must be page-locked memory mapped into the device's space",
            who);
    g->next.recs.clear();
    g->next.overflow = false;
    t_launch_log = &g->next;
    rc = decode_step_impl(g->m, ss, g->rows, g->n_seq, g->x, g->logits, g->argmax, g->ws, g->ws_bytes, stream, who,
                          g->io);
    t_launch_log = nullptr;
    REQUIRE(!g->next.overflow, LUCE_EUNSUPPORTED, "%s: a launch has more arguments than a record holds", who);
    if (rc) return rc;
    cudaError_t e = cudaSuccess;
    if (!g->exec || !same_nodes(g->live, g->next) || !refresh(g)) {
        if ((e = capture(g))) {
            release_graph(g);
            return cuda_status(e, who);
        }
    }
    std::swap(g->live, g->next);
    if ((e = cudaGraphLaunch(g->exec, (cudaStream_t)stream))) return cuda_status(e, who);
    count_launches(g->kernels);
    return ok();
}

int luce_step_graph_stats(const luce_step_graph* g, int64_t* captures, int64_t* node_updates, int32_t* kernels)
{
    REQUIRE(g, LUCE_EINVAL, "step_graph_stats: null graph");
    if (captures) *captures = g->captures;
    if (node_updates) *node_updates = g->node_updates;
    if (kernels) *kernels = g->kernels;
    return ok();
}

int luce_step_graph_destroy(luce_step_graph* g)
{
    if (!g) return ok();
    release_graph(g);
    if (g->cap) cudaStreamDestroy(g->cap);
    delete g;
    return ok();
}

int luce_decode_step_paged(const luce_model* m, const luce_paged_slot* slots, const int32_t* rows_per_slot,
                           int n_seq, float* x, float* logits, int32_t* argmax, void* ws, size_t ws_bytes,
                           void* stream)
{
    const char* who = "decode_step_paged";
    int rc = check_model(m, who);
    if (rc) return rc;
    REQUIRE(slots && rows_per_slot, LUCE_EINVAL, "%s: null slots/rows", who);
    REQUIRE(n_seq >= 1 && n_seq <= LUCE_MAX_SEQ, LUCE_EINVAL,
            "%s: n_seq=%d outside 1..%d (more than %d slots are refused)", who, n_seq, LUCE_MAX_SEQ, LUCE_MAX_SEQ);
    StepSlot ss[LUCE_MAX_SEQ];
    for (int s = 0; s < n_seq; ++s) {
        const luce_paged_slot& sl = slots[s];
        if ((rc = check_rows(rows_per_slot, s, who))) return rc;
        const int n = rows_per_slot[s];
        REQUIRE(sl.k_pool && sl.v_pool && aligned(sl.k_pool, 16) && aligned(sl.v_pool, 16), LUCE_EINVAL,
                "%s: slot %d pool null or not 16-byte aligned", who, s);
        REQUIRE(sl.table && sl.table_host && aligned(sl.table, 4), LUCE_EINVAL, "%s: slot %d table null", who, s);
        REQUIRE(sl.len >= 0 && sl.len + n <= kMaxKeys, LUCE_EINVAL, "%s: slot %d len=%d + rows=%d outside 0..%d",
                who, s, sl.len, n, kMaxKeys);
        const int need = (sl.len + n + kPageKeys - 1) / kPageKeys;
        REQUIRE(sl.n_pages >= 1 && sl.n_table >= need, LUCE_EINVAL, "%s: slot %d table has %d entries, needs %d",
                who, s, sl.n_table, need);
        for (int i = 0; i < need; ++i)
            REQUIRE(sl.table_host[i] >= 0 && sl.table_host[i] < sl.n_pages, LUCE_EINVAL,
                    "%s: slot %d table[%d]=%d outside [0, %d)", who, s, i, sl.table_host[i], sl.n_pages);
        ss[s] = StepSlot{reinterpret_cast<__half*>(sl.k_pool), reinterpret_cast<__half*>(sl.v_pool), sl.len,
                         need * kPageKeys, sl.table, sl.table_host};
    }
    // pages written by this step belong to their slot alone within the call
    for (int s = 0; s < n_seq; ++s) {
        const luce_paged_slot& a = slots[s];
        for (int pg = a.len / kPageKeys; pg <= (a.len + rows_per_slot[s] - 1) / kPageKeys; ++pg)
            for (int o = 0; o < n_seq; ++o) {
                const luce_paged_slot& b = slots[o];
                if (b.k_pool != a.k_pool && b.v_pool != a.v_pool) continue;
                const int nb = (b.len + rows_per_slot[o] + kPageKeys - 1) / kPageKeys;
                for (int i = 0; i < nb; ++i)
                    REQUIRE(o == s ? (i == pg || b.table_host[i] != a.table_host[pg])
                                   : b.table_host[i] != a.table_host[pg],
                            LUCE_EINVAL, "%s: page %d written for slot %d is also referenced by slot %d", who,
                            a.table_host[pg], s, o);
            }
    }
    return decode_step_impl(m, ss, rows_per_slot, n_seq, x, logits, argmax, ws, ws_bytes, stream, who);
}

}  // extern "C"
