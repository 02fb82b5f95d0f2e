"""The composed decode step on the GPU against the oracle.

Staged parity: every stage of a layer is checked against the oracle fed the
GPU's own input to that stage (read from the step's workspace), because a
1-ulp difference upstream can legitimately flip one int8 activation code.
Free-running parity then bounds the end-to-end difference.  Invariance:
batched rows and cache writes equal solo runs bit for bit, in any slot
order, and slots outside the batch are untouched.
"""
import math

import numpy as np
import pytest

import oracle
from invariant_sequence_decode_gb300 import workloads as wl

torch = pytest.importorskip("torch")
import invariant_sequence_decode_gb300 as luce  # noqa: E402

pytestmark = pytest.mark.gpu

F16_NAN = 0x7E00
LAYER_FIELDS = ["attn_norm", "wqkv_q", "wqkv_d", "wo_q", "wo_d", "ffn_norm", "wgu_q", "wgu_d", "wdown_q", "wdown_d"]


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


class Case:
    def __init__(self, seed, dims, n_layers, lens, rows, cap, vocab=0):
        self.seed, self.dims, self.n_layers, self.lens, self.rows, self.cap = seed, dims, n_layers, lens, rows, cap
        self.layers_h = [wl.layer_host(seed, l, dims) for l in range(n_layers)]
        layers_d = [luce.LayerTensors(*[cuda(getattr(L, f)) for f in LAYER_FIELDS]) for L in self.layers_h]
        self.head_h = wl.head_host(seed, dims, vocab) if vocab else None
        hd = [cuda(a) for a in self.head_h] if vocab else [None, None, None]
        self.model = luce.Model(layers_d, dims.hidden, dims.n_q_heads, dims.n_kv_heads, dims.ffn,
                                rms_eps=dims.rms_eps, rope_theta=dims.rope_theta,
                                final_norm=hd[0], head_q=hd[1], head_d=hd[2])
        self.vocab = vocab
        # host caches [L][Hkv][cap][D] as fp16; positions >= len hold NaN sentinels
        self.k_h, self.v_h = [], []
        for s, ln in enumerate(lens):
            ks, vs = [], []
            for l in range(n_layers):
                k, v = wl.cache_host(seed, s, l, dims, cap, ln)
                k = k.copy()
                v = v.copy()
                k.view(np.uint16)[:, ln:] = F16_NAN
                v.view(np.uint16)[:, ln:] = F16_NAN
                ks.append(k)
                vs.append(v)
            self.k_h.append(np.stack(ks))
            self.v_h.append(np.stack(vs))
        self.x = wl.acts(seed, sum(rows), dims.hidden, sub=9)

    def slots(self, idx):
        return [luce.Slot(cuda(self.k_h[s]), cuda(self.v_h[s]), self.lens[s]) for s in idx]

    def run(self, idx=None, want_logits=True):
        idx = list(range(len(self.lens))) if idx is None else idx
        rows = [self.rows[s] for s in idx]
        starts = np.cumsum([0] + self.rows)
        x = cuda(np.concatenate([self.x[starts[s]:starts[s] + self.rows[s]] for s in idx]))
        T = sum(rows)
        slots = self.slots(idx)
        ws = self.model.workspace(T, self.cap)
        logits = argmax = None
        if self.vocab and want_logits:
            logits = torch.empty((T, self.vocab), dtype=torch.float32, device="cuda")
            argmax = torch.empty(T, dtype=torch.int32, device="cuda")
        luce.luce_decode_step(self.model, slots, rows, x, ws, logits, argmax)
        return dict(x=host(x), ws=ws, slots=slots, logits=None if logits is None else host(logits),
                    argmax=None if argmax is None else host(argmax), T=T, rows=rows, idx=idx)


def ws_view(ws, off, shape, dtype):
    n = int(np.prod(shape)) * np.dtype(dtype).itemsize
    return host(ws[off:off + n]).view(dtype).reshape(shape)


def rel_err(y, ref):
    return np.max(np.abs(y - ref), axis=1) / np.maximum(np.linalg.norm(ref, axis=1), 1e-30)


def staged_layer_check(case, out, layer=0):
    d = case.dims
    H, Hq, Hkv, D, F = d.hidden, d.n_q_heads, d.n_kv_heads, d.head_dim, d.ffn
    T = out["T"]
    lay = case.model.layout(T, case.cap)
    ws = out["ws"]
    L = case.layers_h[layer]
    x_in = case.x.astype(np.float64) if case.n_layers == 1 else None
    pos = oracle.row_positions([case.lens[s] for s in out["idx"]], out["rows"])

    xn = ws_view(ws, lay["xn"], (T, H), np.float32)
    if x_in is not None:
        ref = oracle.rmsnorm(x_in, L.attn_norm, d.rms_eps)
        assert np.all(rel_err(xn.astype(np.float64), ref) <= 1e-5)
    q, dd = oracle.quantize_act(xn)
    assert np.array_equal(ws_view(ws, lay["xn_q"], (T, H), np.int8), q)
    assert np.array_equal(ws_view(ws, lay["xn_d"], (T, H // 32), np.float32), dd)

    qkv = ws_view(ws, lay["qkv"], (T, (Hq + 2 * Hkv) * D), np.float32)
    assert np.all(rel_err(qkv.astype(np.float64), oracle.matvec(L.wqkv_q, L.wqkv_d, q, dd)) <= 1e-5)

    q_rot = ws_view(ws, lay["q_rot"], (T, Hq, D), np.float32)
    ref = oracle.rope(qkv[:, :Hq * D].reshape(T, Hq, D), pos, d.rope_theta)
    pair = np.sqrt(ref[..., :64] ** 2 + ref[..., 64:] ** 2)
    assert np.all(np.abs(q_rot[..., :64] - ref[..., :64]) <= 1e-6 * pair + 1e-30)
    assert np.all(np.abs(q_rot[..., 64:] - ref[..., 64:]) <= 1e-6 * pair + 1e-30)
    k_ref = oracle.rope(qkv[:, Hq * D:(Hq + Hkv) * D].reshape(T, Hkv, D), pos, d.rope_theta)
    v_new = qkv[:, (Hq + Hkv) * D:].reshape(T, Hkv, D)

    # cache rows this step wrote; attention against the GPU's cache
    attn_ref = np.empty((T, Hq, D))
    r = 0
    for s, n in zip(out["idx"], out["rows"]):
        slot = out["slots"][out["idx"].index(s)]
        kc = host(slot.k)[layer]
        vc = host(slot.v)[layer]
        ln = case.lens[s]
        for j in range(n):
            got_k = kc[:, ln + j].astype(np.float64)
            want_k = k_ref[r + j].astype(np.float16).astype(np.float64)
            ulp = np.abs(np.spacing(k_ref[r + j].astype(np.float16))).astype(np.float64)
            assert np.all(np.abs(got_k - want_k) <= ulp)
            assert np.array_equal(vc[:, ln + j].view(np.uint16), oracle.float_to_half_bits(v_new[r + j]).reshape(Hkv, D))
            attn_ref[r + j] = oracle.attention_row(q_rot[r + j], kc.view(np.uint16), vc.view(np.uint16), ln + j + 1,
                                                   Hkv, 1 / math.sqrt(D))
        r += n
    attn = ws_view(ws, lay["attn"], (T, Hq, D), np.float32)
    assert np.max(np.abs(attn - attn_ref)) <= 2e-3

    aq, ad = oracle.quantize_act(attn.reshape(T, Hq * D))
    assert np.array_equal(ws_view(ws, lay["attn_q"], (T, Hq * D), np.int8), aq)
    assert np.array_equal(ws_view(ws, lay["attn_d"], (T, Hq * D // 32), np.float32), ad)
    x1 = ws_view(ws, lay["x1"], (T, H), np.float32)
    o_ref = oracle.matvec(L.wo_q, L.wo_d, aq, ad)
    if x_in is not None:
        x1_ref = x_in + o_ref
        assert np.all(np.max(np.abs(x1 - x1_ref), axis=1) <= 1e-5 * (np.linalg.norm(o_ref, axis=1) +
                                                                     np.linalg.norm(x_in, axis=1)))

    xn2 = ws_view(ws, lay["xn2"], (T, H), np.float32)
    assert np.all(rel_err(xn2.astype(np.float64), oracle.rmsnorm(x1, L.ffn_norm, d.rms_eps)) <= 1e-5)
    fq, fd = oracle.quantize_act(xn2)
    assert np.array_equal(ws_view(ws, lay["xn2_q"], (T, H), np.int8), fq)
    gu = ws_view(ws, lay["gu"], (T, 2 * F), np.float32)
    assert np.all(rel_err(gu.astype(np.float64), oracle.matvec(L.wgu_q, L.wgu_d, fq, fd)) <= 1e-5)
    h = ws_view(ws, lay["h"], (T, F), np.float32)
    assert np.all(rel_err(h.astype(np.float64), oracle.swiglu(gu)) <= 1e-5)
    hq, hd = oracle.quantize_act(h)
    assert np.array_equal(ws_view(ws, lay["h_q"], (T, F), np.int8), hq)
    assert np.array_equal(ws_view(ws, lay["h_d"], (T, F // 32), np.float32), hd)
    if layer == case.n_layers - 1:
        dn = oracle.matvec(L.wdown_q, L.wdown_d, hq, hd)
        x2 = out["x"]
        assert np.all(np.max(np.abs(x2 - (x1 + dn)), axis=1) <= 1e-5 * (np.linalg.norm(dn, axis=1) +
                                                                        np.linalg.norm(x1, axis=1)))
    if case.vocab and layer == case.n_layers - 1:
        fn, wq, wd = case.head_h
        xf = ws_view(ws, lay["xf"], (T, H), np.float32)
        assert np.all(rel_err(xf.astype(np.float64), oracle.rmsnorm(out["x"], fn, d.rms_eps)) <= 1e-5)
        xq, xd = oracle.quantize_act(xf)
        assert np.array_equal(ws_view(ws, lay["xf_q"], (T, H), np.int8), xq)
        assert np.all(rel_err(out["logits"].astype(np.float64), oracle.matvec(wq, wd, xq, xd)) <= 1e-5)
        assert np.array_equal(out["argmax"], oracle.argmax(out["logits"]))


def test_tiny_layer_staged_parity():
    case = Case(11, wl.TINY_LAYER, 1, [5, 17, 300, 1000], [1, 2, 3, 4], cap=1024, vocab=1000)
    staged_layer_check(case, case.run())


def test_tiny_stack_free_running_parity():
    case = Case(12, wl.TINY_LAYER, 3, [0, 40, 257, 600], [2, 1, 4, 3], cap=640, vocab=500)
    out = case.run()
    d = case.dims
    x = case.x.astype(np.float64)
    starts = np.cumsum([0] + case.rows)
    oslots = [[oracle.Slot(case.k_h[s][l].view(np.uint16).copy(), case.v_h[s][l].view(np.uint16).copy(),
                           case.lens[s]) for s in range(4)] for l in range(case.n_layers)]
    for l in range(case.n_layers):
        L = case.layers_h[l]
        lw = oracle.LayerWeights(*[getattr(L, f) for f in LAYER_FIELDS])
        x = oracle.decode_layer(x, lw, oracle.Dims(d.hidden, d.n_q_heads, d.n_kv_heads, d.head_dim, d.ffn),
                                oslots[l], case.rows)
    err = rel_err(out["x"].astype(np.float64), x)
    # A few +-1 code flips at the layers' quantization points (a 1-ulp fp32
    # difference straddling a rounding tie) move a row by ~1/(127 sqrt(K)) of
    # its norm each; 2e-3 leaves room for several per row across 3 layers.
    assert np.all(err <= 2e-3), err
    fn, wq, wd = case.head_h
    lref = oracle.lm_head(x, fn, wq, wd, d.rms_eps)
    assert np.all(rel_err(out["logits"].astype(np.float64), lref) <= 5e-3)
    staged_layer_check(case, out, layer=case.n_layers - 1)


def same_bits(a, b):
    return np.array_equal(np.ascontiguousarray(a).view(np.uint8), np.ascontiguousarray(b).view(np.uint8))


@pytest.mark.parametrize("dims,lens,rows,cap,vocab,n_layers", [
    (wl.TINY_LAYER, [5, 17, 300, 1000], [1, 2, 3, 4], 1024, 1000, 2),
    (wl.TINY_LAYER, [0, 1, 255, 256], [4, 4, 4, 4], 512, 300, 2),
])
def test_batched_equals_solo_bitwise(dims, lens, rows, cap, vocab, n_layers):
    case = Case(13, dims, n_layers, lens, rows, cap, vocab)
    b = case.run()
    r0 = 0
    for s in range(len(lens)):
        so = case.run([s])
        n = rows[s]
        assert same_bits(so["x"], b["x"][r0:r0 + n])
        assert same_bits(so["logits"], b["logits"][r0:r0 + n])
        assert np.array_equal(so["argmax"], b["argmax"][r0:r0 + n])
        assert same_bits(host(so["slots"][0].k), host(b["slots"][s].k))
        assert same_bits(host(so["slots"][0].v), host(b["slots"][s].v))
        r0 += n
    # slot order permuted
    order = [3, 1, 0, 2]
    p = case.run(order)
    starts = np.cumsum([0] + rows)
    pr = 0
    for s in order:
        n = rows[s]
        assert same_bits(p["x"][pr:pr + n], b["x"][starts[s]:starts[s] + n])
        assert same_bits(p["logits"][pr:pr + n], b["logits"][starts[s]:starts[s] + n])
        pr += n
    # cache: only rows [len, len + rows) changed, everything else byte-identical
    for s in range(len(lens)):
        kc = host(b["slots"][s].k).view(np.uint16)
        before = case.k_h[s].view(np.uint16)
        changed = np.any(kc != before, axis=(1, 3))  # [L][cap]
        for l in range(n_layers):
            idx = np.nonzero(changed[l])[0]
            assert set(idx.tolist()) <= set(range(lens[s], lens[s] + rows[s]))


def test_untouched_slot_isolation():
    # All four caches live side by side in one allocation; a step over slots
    # 0, 2, 3 must leave slot 1's bytes (and every unwritten row) unchanged.
    case = Case(14, wl.TINY_LAYER, 2, [30, 60, 90, 120], [1, 1, 1, 1], 256, 0)
    kall = cuda(np.stack(case.k_h))
    vall = cuda(np.stack(case.v_h))
    k0, v0 = host(kall).view(np.uint16).copy(), host(vall).view(np.uint16).copy()
    idx = [0, 2, 3]
    slots = [luce.Slot(kall[s], vall[s], case.lens[s]) for s in idx]
    x = cuda(case.x[idx])
    ws = case.model.workspace(3, case.cap)
    luce.luce_decode_step(case.model, slots, [1, 1, 1], x, ws)
    k1, v1 = host(kall).view(np.uint16), host(vall).view(np.uint16)
    assert np.array_equal(k1[1], k0[1]) and np.array_equal(v1[1], v0[1])
    for s in idx:
        ch = np.nonzero(np.any(k1[s] != k0[s], axis=(0, 1, 3)))[0].tolist()
        assert ch == [case.lens[s]]
        chv = np.nonzero(np.any(v1[s] != v0[s], axis=(0, 1, 3)))[0].tolist()
        assert chv == [case.lens[s]]


def test_identical_rows_give_identical_outputs():
    # "identical" phase: every slot holds the same history and the same input
    case = Case(15, wl.TINY_LAYER, 2, [64, 64, 64, 64], [1, 1, 1, 1], 128, 200)
    for s in range(1, 4):
        case.k_h[s] = case.k_h[0].copy()
        case.v_h[s] = case.v_h[0].copy()
    case.x[1:] = case.x[0]
    out = case.run()
    for s in range(1, 4):
        assert same_bits(out["x"][s], out["x"][0]) and same_bits(out["logits"][s], out["logits"][0])


@pytest.mark.parametrize("n_seq", [1, 4])
def test_27b_layer_staged_parity(n_seq):
    case = Case(1, wl.LAYER27B, 1, [2050] * n_seq, [1] * n_seq, cap=2051)
    staged_layer_check(case, case.run())


def test_27b_layer_batched_equals_solo():
    case = Case(1, wl.LAYER27B, 1, [2050] * 4, [1] * 4, cap=2051)
    b = case.run()
    for k in (1, 2, 3):
        sub = case.run(list(range(k)))
        assert same_bits(sub["x"], b["x"][:k])


@pytest.mark.parametrize("dims,n_seq,rows", [(wl.LAYER27B, 4, 1), (wl.LAYER27B, 1, 1), (wl.TINY_LAYER, 3, 1),
                                             (wl.TINY_LAYER, 2, 2), (wl.TINY_LAYER, 2, 3)])
def test_fused_gate_up_swiglu_equals_the_two_launches_bitwise(dims, n_seq, rows):
    """At 1-4 rows the step computes gate||up, SwiGLU and its q8_0 codes in one
    launch; its gu, h and codes equal the standalone projection followed by the
    standalone SwiGLU quantizer on the same activations, bit for bit (at 5-8
    rows the step runs those two launches itself)."""
    cap = 2051 if dims is wl.LAYER27B else 160
    case = Case(5, dims, 1, [cap - rows] * n_seq, [rows] * n_seq, cap=cap)
    out = case.run()
    T, H, F = out["T"], dims.hidden, dims.ffn
    lay = case.model.layout(T, case.cap)
    ws = out["ws"]
    L = case.layers_h[0]
    aq = cuda(ws_view(ws, lay["xn2_q"], (T, H), np.int8))
    ad = cuda(ws_view(ws, lay["xn2_d"], (T, H // 32), np.float32))
    gu = luce.luce_q8_matvec_batch(cuda(L.wgu_q), cuda(L.wgu_d), aq, ad)
    h, hq, hd = luce.luce_swiglu_q8(gu)
    assert same_bits(ws_view(ws, lay["gu"], (T, 2 * F), np.float32), host(gu))
    assert same_bits(ws_view(ws, lay["h"], (T, F), np.float32), host(h))
    assert np.array_equal(ws_view(ws, lay["h_q"], (T, F), np.int8), host(hq))
    assert same_bits(ws_view(ws, lay["h_d"], (T, F // 32), np.float32), host(hd))


@pytest.mark.parametrize("dims,n_seq,rows", [(wl.LAYER27B, 4, 2), (wl.LAYER27B, 4, 4), (wl.TINY_LAYER, 2, 3),
                                             (wl.TINY_LAYER, 4, 4)])
def test_wide_qkv_rope_epilogue_equals_the_separate_kernels_bitwise(dims, n_seq, rows):
    """From 5 rows the step's q|k|v runs on the tensor-core ring with RoPE and
    the K/V append in its epilogue; its qkv, q_rot and cache rows equal the
    standalone projection, then the standalone RoPE, then binary16 rounding,
    bit for bit."""
    cap = 2051 if dims is wl.LAYER27B else 160
    case = Case(7, dims, 1, [cap - rows] * n_seq, [rows] * n_seq, cap=cap)
    out = case.run()
    T, H, Hq, Hkv, D = out["T"], dims.hidden, dims.n_q_heads, dims.n_kv_heads, dims.head_dim
    lay = case.model.layout(T, case.cap)
    ws = out["ws"]
    L = case.layers_h[0]
    aq = cuda(ws_view(ws, lay["xn_q"], (T, H), np.int8))
    ad = cuda(ws_view(ws, lay["xn_d"], (T, H // 32), np.float32))
    qkv = luce.luce_q8_matvec_batch(cuda(L.wqkv_q), cuda(L.wqkv_d), aq, ad)
    assert same_bits(ws_view(ws, lay["qkv"], (T, (Hq + 2 * Hkv) * D), np.float32), host(qkv))
    heads = qkv.view(T, Hq + 2 * Hkv, D)
    qk = heads[:, :Hq + Hkv].contiguous()
    pos = torch.tensor([cap - rows + j for _ in range(n_seq) for j in range(rows)], dtype=torch.int32, device="cuda")
    luce.luce_rope_posvec(qk, pos, dims.rope_theta)
    assert same_bits(ws_view(ws, lay["q_rot"], (T, Hq, D), np.float32), host(qk[:, :Hq]))
    k_ref = host(qk[:, Hq:]).astype(np.float16)
    v_ref = host(heads[:, Hq + Hkv:]).astype(np.float16)
    for t in range(T):
        s, j = divmod(t, rows)
        p = cap - rows + j
        sl = out["slots"][s]
        assert same_bits(host(sl.k[0, :, p, :]), k_ref[t]), t
        assert same_bits(host(sl.v[0, :, p, :]), v_ref[t]), t
