"""GPU parity of each kernel against the CPU oracle, plus batched == solo.

Tolerances: quantized activations and per-block int32 dots bit-exact; fp32
matvec rows within 1e-5 of the row's L2 norm; attention within 2e-3 absolute
(fp32 accumulation over an f16 cache); RoPE within 1e-6 of each pair's norm
(fp32 rotation by double-evaluated cos/sin); batched vs solo bitwise.
"""
import math

import numpy as np
import pytest

import oracle
from invariant_sequence_decode_gb300 import synth, workloads as wl

torch = pytest.importorskip("torch")
import invariant_sequence_decode_gb300 as luce  # noqa: E402

pytestmark = pytest.mark.gpu

SENTINEL = np.uint32(0x7FC0DEAD)


@pytest.fixture(scope="module", autouse=True)
def _built():
    from invariant_sequence_decode_gb300 import build
    build.build()
    luce.load_library()


def cuda(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    torch.cuda.synchronize()
    return t.cpu().numpy()


def rel_row_err(y, ref):
    return np.max(np.abs(y - ref), axis=1) / np.maximum(np.linalg.norm(ref, axis=1), 1e-30)


# ------------------------------------------------------------ quantizer

def crafted_rows(K):
    ties = np.array([127.0, -126.5, 126.5, 63.5, -63.5, 2.5, -2.5, 0.5, -0.5, 1.5] + [0.25] * 22, np.float32)
    rows = np.zeros((4, K), np.float32)
    rows[0, :32] = ties
    rows[1, :32] = 3.0                       # constant block -> all 127
    rows[1, 32:64] = 0.0                     # zero block -> d = 0
    rows[2, :32] = np.linspace(-1, 1, 32)
    rows[2, 5] = np.nan                      # NaN entry -> 0, ignored by amax
    rows[3, :32] = np.float32(1e-40) * np.arange(32)  # subnormal block
    return rows


@pytest.mark.parametrize("T,K", [(1, 32), (4, 1024), (3, 5120), (16, 17408)])
def test_quantize_bit_exact(T, K):
    x = wl.acts(0, T, K) * np.float32(3.0)
    x = np.concatenate([x, crafted_rows(K)])
    q, d = luce.luce_q8_quantize_act(cuda(x))
    qo, do = oracle.quantize_act(x)
    assert np.array_equal(host(q), qo)
    assert np.array_equal(host(d).view(np.uint32), do.view(np.uint32))


# ------------------------------------------------------------ block dots / matvec

# K % 256 == 0 with T <= 4 runs the TMA-ring kernel: (37, 1280) has a partial
# last kilobyte stage and a partial quad of rows, (100, 256) a K shorter than
# one stage, (2049, 768) stages of 24 blocks over many CTAs, (1, 512) and
# (5, 256) a single group mostly past the end of W
MV_SHAPES = [(1024, 1024), (1000, 1056), (33, 96), (7, 32), (301, 5120), (64, 17408), (37, 1280), (100, 256),
             (2049, 768), (1, 512), (5, 256)]


def mv_inputs(N, K, T, seed=0):
    wq, wd = wl.q8_weights(seed, wl.tid(wl.W_MAT, N % 4096, K % 16), N, K)
    aq, ad = oracle.quantize_act(wl.acts(seed, T, K, sub=3))
    return wq, wd, aq, ad


@pytest.mark.parametrize("N,K", MV_SHAPES)
def test_block_dots_bit_exact(N, K):
    wq, wd, aq, ad = mv_inputs(N, K, 3)
    got = host(luce.luce_q8_block_dots(cuda(wq), cuda(aq)))
    assert np.array_equal(got, oracle.block_dots(wq, aq))


def test_block_dots_extremes():
    wq = np.full((2, 64), -127, np.int8)
    wq[1] = 127
    aq = np.full((1, 64), -127, np.int8)
    got = host(luce.luce_q8_block_dots(cuda(wq), cuda(aq)))
    assert got[0, 0].tolist() == [516128, 516128] and got[0, 1].tolist() == [-516128, -516128]


@pytest.mark.parametrize("T", list(range(1, 17)))
def test_matvec_full_scale_blocks_exact(T):
    """Every block dot at its extreme, +-32*127*127 = +-516,128, in every launch
    shape: with unit scales each output is 32 * 516,128 = 16,516,096 (< 2^24),
    exact in fp32 whatever the form of the int-to-float step."""
    N, K = 40, 1024
    wq = np.full((N, K), 127, np.int8)
    wq[1::2] = -127
    aq = np.full((T, K), 127, np.int8)
    aq[1::2] = -127
    wd = np.ones((N, K // 32), np.float16)
    ad = np.ones((T, K // 32), np.float32)
    y = host(luce.luce_q8_matvec_batch(cuda(wq), cuda(wd), cuda(aq), cuda(ad)))
    sign = np.where(np.arange(T)[:, None] % 2 == np.arange(N)[None, :] % 2, 1.0, -1.0)
    assert np.array_equal(y, (sign * 32 * 516128).astype(np.float32))


@pytest.mark.parametrize("N,K", MV_SHAPES)
@pytest.mark.parametrize("T", [1, 2, 3, 4, 5, 8, 12, 16])
def test_matvec_parity(N, K, T):
    wq, wd, aq, ad = mv_inputs(N, K, T)
    y = host(luce.luce_q8_matvec_batch(cuda(wq), cuda(wd), cuda(aq), cuda(ad)))
    ref = oracle.matvec(wq, wd, aq, ad)
    assert np.all(rel_row_err(y.astype(np.float64), ref) <= 1e-5)


@pytest.mark.parametrize("N,K", [(1024, 1024), (1000, 1056), (33, 96), (301, 5120)])
def test_matvec_batched_equals_solo_bitwise(N, K):
    wq, wd, aq, ad = mv_inputs(N, K, 16, seed=2)
    W, D = cuda(wq), cuda(wd)
    solo = [host(luce.luce_q8_matvec_batch(W, D, cuda(aq[t:t + 1]), cuda(ad[t:t + 1])))[0] for t in range(16)]
    for T in range(1, 17):
        yb = host(luce.luce_q8_matvec_batch(W, D, cuda(aq[:T]), cuda(ad[:T])))
        for t in range(T):
            assert np.array_equal(yb[t].view(np.uint32), solo[t].view(np.uint32)), (T, t)
    perm = synth.permutation(2, 77, 16)
    yp = host(luce.luce_q8_matvec_batch(W, D, cuda(aq[perm]), cuda(ad[perm])))
    for i, t in enumerate(perm):
        assert np.array_equal(yp[i].view(np.uint32), solo[t].view(np.uint32))


@pytest.mark.parametrize("N,K", [(301, 5120), (37, 1280), (100, 256), (64, 17408)])
def test_matvec_tma_and_register_kernels_agree_bitwise(N, K):
    """Scales stored 2 bytes past a 16-byte boundary send every launch to the
    register-pipelined kernel instead of the TMA ring (1..8 rows in one launch,
    13..16 in two); the bits match at every row count."""
    wq, wd, aq, ad = mv_inputs(N, K, 16, seed=5)
    W, D = cuda(wq), cuda(wd)
    buf = torch.zeros(wd.size + 8, dtype=torch.float16, device="cuda")
    buf[1:1 + wd.size] = D.flatten()
    D_odd = buf[1:1 + wd.size].view(wd.shape)
    assert D_odd.data_ptr() % 16 == 2
    for T in range(1, 17):
        A, Ad = cuda(aq[:T]), cuda(ad[:T])
        ring = host(luce.luce_q8_matvec_batch(W, D, A, Ad))
        reg = host(luce.luce_q8_matvec_batch(W, D_odd, A, Ad))
        assert np.array_equal(ring.view(np.uint32), reg.view(np.uint32)), T
    assert luce.wait_timeouts() == 0


@pytest.mark.parametrize("N,K", [(301, 5120), (37, 1280), (100, 256), (64, 17408), (1, 512), (5, 2048),
                                 (1000, 1024), (17, 768)])
def test_matvec_three_kernels_agree_bitwise_and_match_the_oracle(N, K):
    """The register-pipelined dp4a kernel, the dp4a TMA ring and the
    tensor-core ring, each named explicitly, at every row count 1..16: the
    same bits (same chains, same butterfly; the tensor cores form each block
    dot exactly), and the tensor-core rows within 1e-5 of the oracle.  Ragged
    N (a 16-row tile mostly past W at N = 1, 5, 17), K shorter than one
    kilobyte stage (256, 512, 768) and K % 1024 != 0 (1280)."""
    wq, wd, aq, ad = mv_inputs(N, K, 16, seed=7)
    W, D = cuda(wq), cuda(wd)
    for T in range(1, 17):
        A, Ad = cuda(aq[:T]), cuda(ad[:T])
        reg = host(luce.luce_q8_matvec_batch_path(W, D, A, Ad, luce.MATVEC_REGISTER))
        tc = host(luce.luce_q8_matvec_batch_path(W, D, A, Ad, luce.MATVEC_TENSOR))
        assert np.array_equal(tc.view(np.uint32), reg.view(np.uint32)), ("tensor", T)
        if 9 <= T <= 12:
            with pytest.raises(luce.LuceError):
                luce.luce_q8_matvec_batch_path(W, D, A, Ad, luce.MATVEC_RING)
        else:
            ring = host(luce.luce_q8_matvec_batch_path(W, D, A, Ad, luce.MATVEC_RING))
            assert np.array_equal(ring.view(np.uint32), reg.view(np.uint32)), ("ring", T)
        auto = host(luce.luce_q8_matvec_batch_path(W, D, A, Ad, luce.MATVEC_AUTO))
        assert np.array_equal(auto.view(np.uint32), reg.view(np.uint32)), ("auto", T)
        ref = oracle.matvec(wq, wd, aq[:T], ad[:T])
        assert np.all(rel_row_err(tc.astype(np.float64), ref) <= 1e-5), T
    assert luce.wait_timeouts() == 0


def test_tensor_core_matvec_writes_only_its_outputs():
    """Rows past N of the last 16-row tile and tokens past T of the 16-token
    activation box are computed on zeros and never stored."""
    N, K = 21, 512
    for T in (3, 9, 16):
        wq, wd, aq, ad = mv_inputs(N, K, T, seed=8)
        buf = np.full((T + 1, N + 12), SENTINEL, np.uint32).view(np.float32)
        yb = cuda(buf)
        rc = luce.load_library().luce_q8_matvec_batch_path(
            cuda(wq).data_ptr(), cuda(wd).data_ptr(), N, K, cuda(aq).data_ptr(), cuda(ad).data_ptr(), T,
            yb.data_ptr(), N + 12, luce.MATVEC_TENSOR, torch.cuda.current_stream().cuda_stream)
        assert rc == 0
        out = host(yb).view(np.uint32)
        assert np.all(out[:T, N:] == SENTINEL) and np.all(out[T] == SENTINEL)
        assert not np.any(out[:T, :N] == SENTINEL)


@pytest.mark.parametrize("K", [2048, 4096, 5120, 8192])
def test_matvec_invariance_sweep_full_sizes(K):
    """Batch-invariance sweep at the sweep's sizes: n_tok 1..4 x N in
    {4096, 8192, 17408, 32768} (weights drawn on the device from a seeded
    generator): every row of every launch, and of a launch with the rows
    permuted, equals the row launched alone, bit for bit; rows past the
    launch's are never written; sampled outputs match the oracle."""
    gen = torch.Generator(device="cuda")
    gen.manual_seed(2000 + K)
    x = torch.randn((4, K), generator=gen, device="cuda")
    aq, ad = luce.luce_q8_quantize_act(x)
    for N in (4096, 8192, 17408, 32768):
        W = torch.randint(-127, 128, (N, K), generator=gen, device="cuda", dtype=torch.int8)
        D = (torch.rand((N, K // 32), generator=gen, device="cuda") * 2e-4 + 1e-5).to(torch.float16)
        solo = [host(luce.luce_q8_matvec_batch(W, D, aq[t:t + 1], ad[t:t + 1]))[0] for t in range(4)]
        for T in range(1, 5):
            buf = torch.full((5, N), float("nan"), device="cuda")
            luce.luce_q8_matvec_batch(W, D, aq[:T], ad[:T], buf[:T])
            yb = host(buf)
            for t in range(T):
                assert np.array_equal(yb[t].view(np.uint32), solo[t].view(np.uint32)), (N, T, t)
            assert np.all(np.isnan(yb[T:]))
        perm = synth.permutation(K, N, 4)
        yp = host(luce.luce_q8_matvec_batch(W, D, aq[perm], ad[perm]))
        for i, t in enumerate(perm):
            assert np.array_equal(yp[i].view(np.uint32), solo[t].view(np.uint32)), (N, "perm", i)
        rows = np.sort(synth.permutation(K, N + 1, N)[:48])
        idx = torch.from_numpy(rows).cuda()
        ref = oracle.matvec(host(W[idx]), host(D[idx].view(torch.int16)).view(np.float16), host(aq), host(ad))
        got = np.stack(solo)[:, rows].astype(np.float64)
        assert np.all(rel_row_err(got, ref) <= 1e-5), (N, K)
        del W, D


def test_matvec_writes_only_its_outputs():
    N, K, T = 100, 256, 3
    wq, wd, aq, ad = mv_inputs(N, K, T)
    buf = np.full((T + 1, N + 12), SENTINEL, np.uint32).view(np.float32)
    yb = cuda(buf)
    y = yb[:T, :N]
    luce.load_library()
    rc = luce.load_library().luce_q8_matvec_batch(cuda(wq).data_ptr(), cuda(wd).data_ptr(), N, K,
                                                  cuda(aq).data_ptr(), cuda(ad).data_ptr(), T, y.data_ptr(),
                                                  N + 12, torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    out = host(yb).view(np.uint32)
    assert np.all(out[:T, N:] == SENTINEL) and np.all(out[T] == SENTINEL)
    assert not np.any(out[:T, :N] == SENTINEL)


# ------------------------------------------------------------ RoPE

def test_rope_parity_and_rows_match_single_row_launches():
    T, Hq = 16, 40
    x = wl.qvec(2, T, Hq, sub=1)
    pos = wl.positions(2, T)
    pos[0], pos[1] = 0, 32767
    xg = cuda(x)
    luce.luce_rope_posvec(xg, cuda(pos), 1e6)
    y = host(xg).astype(np.float64)
    ref = oracle.rope(x, pos, 1e6)
    pair = np.sqrt(ref[..., :64] ** 2 + ref[..., 64:] ** 2)
    err = np.maximum(np.abs(y[..., :64] - ref[..., :64]), np.abs(y[..., 64:] - ref[..., 64:]))
    assert np.all(err <= 1e-6 * pair + 1e-30)
    assert np.array_equal(y[0], x[0].astype(np.float64))  # position 0 is the identity
    for t in range(T):
        x1 = cuda(x[t:t + 1])
        luce.luce_rope_posvec(x1, cuda(pos[t:t + 1]), 1e6)
        assert np.array_equal(host(x1)[0].view(np.uint32), host(xg)[t].view(np.uint32))


# ------------------------------------------------------------ KV append

def test_kv_append_bit_exact_and_in_place():
    Hkv, cap, D = 2, 64, 128
    k = wl.qvec(3, 4, Hkv, sub=2) * np.float32(7.0)
    v = wl.qvec(3, 4, Hkv, sub=3)
    kc = [cuda(np.full((Hkv, cap, D), 0x7E00, np.uint16).view(np.float16)) for _ in range(2)]
    vc = [cuda(np.full((Hkv, cap, D), 0x7E00, np.uint16).view(np.float16)) for _ in range(2)]
    views = [luce.SeqView(kc[0], vc[0], len=10, n_q=1, row0=0), luce.SeqView(kc[1], vc[1], len=40, n_q=3, row0=1)]
    luce.luce_kv_append(cuda(k), cuda(v), views)
    for s, (pos0, rows) in enumerate([(9, [0]), (37, [1, 2, 3])]):
        kh = host(kc[s]).view(np.uint16)
        vh = host(vc[s]).view(np.uint16)
        for j, r in enumerate(rows):
            assert np.array_equal(kh[:, pos0 + j], oracle.float_to_half_bits(k[r]).reshape(Hkv, D))
            assert np.array_equal(vh[:, pos0 + j], oracle.float_to_half_bits(v[r]).reshape(Hkv, D))
        mask = np.ones(cap, bool)
        mask[pos0:pos0 + len(rows)] = False
        assert np.all(kh[:, mask] == 0x7E00) and np.all(vh[:, mask] == 0x7E00)


# ------------------------------------------------------------ attention

def attn_case(seed, lens, nq, Hq, Hkv, cap=None):
    D = 128
    views, caches = [], []
    row0 = 0
    for s, (L, n) in enumerate(zip(lens, nq)):
        c = cap or L
        k, v = wl.cache_host(seed, s, 0, wl.Dims(0, Hq, Hkv, D, 0), c, L)
        caches.append((k, v))
        views.append((L, n, row0))
        row0 += n
    q = wl.qvec(seed, row0, Hq, sub=4)
    return q, caches, views


def run_attn(q, caches, views, Hkv, scale):
    dev = [(cuda(k), cuda(v)) for k, v in caches]
    sv = [luce.SeqView(k, v, L, n, r0) for (k, v), (L, n, r0) in zip(dev, views)]
    return host(luce.luce_decode_attn_multiseq(cuda(q), sv, Hkv, scale))


def oracle_attn(q, caches, views, Hkv, scale):
    out = np.empty(q.shape, np.float64)
    for (k, v), (L, n, r0) in zip(caches, views):
        for j in range(n):
            out[r0 + j] = oracle.attention_row(q[r0 + j], k, v, L - n + 1 + j, Hkv, scale)
    return out


@pytest.mark.parametrize("lens,nq,Hq,Hkv", [
    (wl.TINY_ATTN_LENS, [1, 1, 1, 1], 8, 2),          # the tiny decode slice
    ([1, 255, 256, 257], [1, 1, 1, 1], 8, 2),          # chunk edges
    ([2051, 2051, 2051, 2051], [1, 1, 1, 1], 40, 8),   # the 27B layer's attention
    ([1030, 1800, 2051, 1500], [4, 3, 2, 4], 40, 8),   # verify rows (causal)
    ([600], [4], 4, 4),
    ([1100, 300, 130, 2051], [4, 2, 1, 3], 64, 8),  # 8 query heads per KV head: the widest slot form
])
def test_attention_parity(lens, nq, Hq, Hkv):
    scale = np.float32(1 / math.sqrt(128))
    q, caches, views = attn_case(5, lens, nq, Hq, Hkv)
    got = run_attn(q, caches, views, Hkv, float(scale))
    ref = oracle_attn(q, caches, views, Hkv, float(scale))
    assert np.max(np.abs(got - ref)) <= 2e-3


def test_attention_long_context_parity():
    lens = wl.lens(3, 4, 16384, 32768)
    scale = float(np.float32(1 / math.sqrt(128)))
    q, caches, views = attn_case(3, lens, [1] * 4, 32, 8)
    got = run_attn(q, caches, views, 8, scale)
    ref = oracle_attn(q, caches, views, 8, scale)
    assert np.max(np.abs(got - ref)) <= 2e-3


def test_attention_strided_unaligned_cache_bitwise():
    """A cache whose rows start 16 (not 32) bytes into a padded row of 136
    halves gives the same bits as a packed, aligned cache: only how K is
    loaded differs."""
    lens, nq, Hkv = [1030, 257, 2051, 130], [2, 1, 1, 3], 8
    q, caches, views = attn_case(11, lens, nq, 40, Hkv)
    packed = run_attn(q, caches, views, Hkv, 0.08838834764831845)
    sv = []
    for (k, v), (L, n, r0) in zip(caches, views):
        cap = k.shape[1]
        pads = []
        for a in (k, v):
            flat = torch.zeros(8 + Hkv * cap * 136, dtype=torch.float16, device="cuda")
            t = flat[8:].view(Hkv, cap, 136)[:, :, :128]
            t.copy_(torch.from_numpy(a))
            pads.append(t)
        assert pads[0].data_ptr() % 32 == 16 and pads[0].stride(1) == 136
        sv.append(luce.SeqView(pads[0], pads[1], L, n, r0))
    got = host(luce.luce_decode_attn_multiseq(cuda(q), sv, Hkv, 0.08838834764831845))
    assert np.array_equal(got.view(np.uint32), packed.view(np.uint32))


def test_attention_batched_equals_solo_bitwise():
    lens, nq = [1030, 1800, 2051, 700], [4, 3, 2, 1]
    q, caches, views = attn_case(7, lens, nq, 40, 8)
    batched = run_attn(q, caches, views, 8, 0.08838834764831845)
    for s, (L, n, r0) in enumerate(views):
        solo = run_attn(q[r0:r0 + n], [caches[s]], [(L, n, 0)], 8, 0.08838834764831845)
        assert np.array_equal(solo.view(np.uint32), batched[r0:r0 + n].view(np.uint32))
    # sequences in another order
    order = [2, 0, 3, 1]
    vv, qq, r0 = [], [], 0
    for s in order:
        L, n, old = views[s]
        vv.append((L, n, r0))
        qq.append(q[old:old + n])
        r0 += n
    perm = run_attn(np.concatenate(qq), [caches[s] for s in order], vv, 8, 0.08838834764831845)
    for (L, n, newr0), s in zip(vv, order):
        old = views[s][2]
        assert np.array_equal(perm[newr0:newr0 + n].view(np.uint32), batched[old:old + n].view(np.uint32))


def test_attention_slot_rows_with_chunk_edges():
    """A slot's verify rows on 128-key chunks are served together (one CTA per
    (chunk, KV head), p.V on tcgen05), a single such row by the one-row form
    of the same kernel, rows past 16,384 keys one CTA per row chunk.  Rows
    whose key counts end in different chunks (127..130 keys), a 27B-shaped
    slot, rows on both sides of the 16,384-key chunk-size switch and a single
    row: within the oracle's tolerance, bit for bit the same rows served one
    by one (each on a cache of its own), and a slot's rows keep their bits
    when the other slots of the launch change."""
    scale = 0.08838834764831845
    lens, nq = [130, 2051, 16386, 1], [4, 4, 4, 1]
    q, caches, views = attn_case(13, lens, nq, 40, 8)
    grouped = run_attn(q, caches, views, 8, scale)
    ref = oracle_attn(q, caches, views, 8, scale)
    assert np.max(np.abs(grouped - ref)) <= 2e-3
    rows = []  # (cache, key count, row) of every row, each row on a cache of its own
    for (k, v), (L, n, r0) in zip(caches, views):
        for j in range(n):
            rows.append(((cuda(k), cuda(v)), L - n + 1 + j, r0 + j))
    separate = np.empty_like(grouped)
    for i in range(0, len(rows), 4):  # at most 4 views per call
        part = rows[i:i + 4]
        sv = [luce.SeqView(kk, vv, L, 1, j) for j, ((kk, vv), L, _) in enumerate(part)]
        got = host(luce.luce_decode_attn_multiseq(cuda(q[[r for _, _, r in part]]), sv, 8, scale))
        for j, (_, _, r) in enumerate(part):
            separate[r] = got[j]
    assert np.array_equal(grouped.view(np.uint32), separate.view(np.uint32))
    # the 130-key slot with other company: its rows keep their bits
    q2, caches2, views2 = attn_case(21, [700, 130], [1, 4], 40, 8)
    caches2[1] = caches[0]
    q2[1:5] = q[0:4]
    other = run_attn(q2, caches2, views2, 8, scale)
    assert np.array_equal(other[1:5].view(np.uint32), grouped[0:4].view(np.uint32))


def test_bounded_wait_expires_counts_and_leaves_the_context_usable():
    """A wait on a barrier that nothing completes gives up after its limit,
    is counted by luce_wait_timeouts, and the next launches run normally."""
    lib = luce.load_library()
    luce.wait_timeouts(reset=True)
    assert lib.luce_test_wait_expiry(5_000_000, torch.cuda.current_stream().cuda_stream) == 0
    torch.cuda.synchronize()
    assert luce.wait_timeouts(reset=True) == 1
    wq, wd, aq, ad = mv_inputs(301, 5120, 4, seed=8)
    y = host(luce.luce_q8_matvec_batch(cuda(wq), cuda(wd), cuda(aq), cuda(ad)))
    ref = oracle.matvec(wq, wd, aq, ad)
    assert np.all(rel_row_err(y.astype(np.float64), ref) <= 1e-5)
    assert luce.wait_timeouts() == 0
    assert lib.luce_test_wait_expiry(10, None) == luce.LUCE_EINVAL
