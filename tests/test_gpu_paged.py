"""Paged K/V caches give the flat cache's bits.

Pages hold 128 keys, the attention's key tile, so chunking and every sum are
unchanged; only where a tile's rows are read from (and where the step appends
its rows) differs.  Pools are filled from flat caches through shuffled page
tables, and several sequences share one pool.
"""
import math

import numpy as np
import pytest

from invariant_sequence_decode_gb300 import synth, workloads as wl

torch = pytest.importorskip("torch")
import invariant_sequence_decode_gb300 as luce  # noqa: E402

pytestmark = pytest.mark.gpu
PK = luce.PAGE_KEYS


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


def bits(a):
    return np.ascontiguousarray(a).view(np.uint8)


def page_tables(seed, spans):
    """Disjoint pages of one pool for sequences needing `spans` pages each, shuffled."""
    total = sum(spans) + 3  # a few pages nobody uses
    perm = synth.permutation(seed, 1, total)
    out, at = [], 0
    for n in spans:
        out.append(perm[at:at + n].astype(np.int32))
        at += n
    return out, total


@pytest.mark.parametrize("lens,nq,Hq,Hkv", [
    ([17, 128, 129, 2051], [1, 1, 2, 4], 40, 8),
    ([1, 300, 16385, 20000], [1, 3, 1, 2], 32, 8),   # 256-key chunks span two pages
    ([640], [4], 8, 2),
])
def test_paged_attention_equals_flat_bitwise(lens, nq, Hq, Hkv):
    d = wl.Dims(0, Hq, Hkv, 128, 0)
    spans = [-(-L // PK) for L in lens]
    tables, n_pages = page_tables(5, spans)
    kpool = np.zeros((n_pages, Hkv, PK, 128), np.float16)
    vpool = np.zeros_like(kpool)
    flat, row0 = [], 0
    for s, L in enumerate(lens):
        k, v = wl.cache_host(6, s, 0, d, spans[s] * PK, L)
        for p, pg in enumerate(tables[s]):
            kpool[pg] = k[:, p * PK:(p + 1) * PK]
            vpool[pg] = v[:, p * PK:(p + 1) * PK]
        flat.append(luce.SeqView(cuda(k), cuda(v), L, nq[s], row0))
        row0 += nq[s]
    q = cuda(wl.qvec(6, row0, Hq))
    scale = 1.0 / math.sqrt(128)
    ref = host(luce.luce_decode_attn_multiseq(q, flat, Hkv, scale))
    kp, vp = cuda(kpool), cuda(vpool)
    views, row0 = [], 0
    for s, L in enumerate(lens):
        views.append(luce.PagedView(kp, vp, cuda(tables[s]), L, nq[s], row0))
        row0 += nq[s]
    got = host(luce.luce_decode_attn_paged(q, views, Hkv, scale))
    assert np.array_equal(bits(got), bits(ref))


LAYER_FIELDS = ["attn_norm", "wqkv_q", "wqkv_d", "wo_q", "wo_d", "ffn_norm", "wgu_q", "wgu_d", "wdown_q", "wdown_d"]


@pytest.mark.parametrize("rws", [[1, 2, 3, 4], [2, 2, 2, 2], [4, 4, 4, 4]])  # 10, 8 and 16 rows
def test_paged_step_equals_flat_step_bitwise(rws):
    D, NL, VOCAB = wl.TINY_LAYER, 2, 250
    layers = [luce.LayerTensors(*[cuda(getattr(wl.layer_host(31, l, D), f)) for f in LAYER_FIELDS])
              for l in range(NL)]
    fn, hq, hd = wl.head_host(31, D, VOCAB)
    model = luce.Model(layers, D.hidden, D.n_q_heads, D.n_kv_heads, D.ffn, rms_eps=D.rms_eps,
                       rope_theta=D.rope_theta, final_norm=cuda(fn), head_q=cuda(hq), head_d=cuda(hd))
    lens = [5, 127, 128, 300]   # rows of slots 1 and 2 cross or start a page
    cap = 512
    spans = [-(-(L + n) // PK) for L, n in zip(lens, rws)]
    tables, n_pages = page_tables(7, spans)
    Hkv = D.n_kv_heads
    kpool = np.zeros((n_pages, NL, Hkv, PK, 128), np.float16)
    vpool = np.zeros_like(kpool)
    flat_k, flat_v = [], []
    for s, L in enumerate(lens):
        ks, vs = zip(*[wl.cache_host(32, s, l, D, cap, L) for l in range(NL)])
        k, v = np.stack(ks), np.stack(vs)                      # [NL][Hkv][cap][128]
        flat_k.append(k)
        flat_v.append(v)
        for p, pg in enumerate(tables[s]):
            kpool[pg] = k[:, :, p * PK:(p + 1) * PK]
            vpool[pg] = v[:, :, p * PK:(p + 1) * PK]
    x_h = wl.acts(33, sum(rws), D.hidden, sub=2)
    T = sum(rws)

    def run(paged):
        x = cuda(x_h)
        logits = torch.empty((T, VOCAB), dtype=torch.float32, device="cuda")
        am = torch.empty(T, dtype=torch.int32, device="cuda")
        ws = model.workspace(T, cap)
        if paged:
            kp, vp = cuda(kpool), cuda(vpool)
            slots = [luce.PagedSlot(kp, vp, tables[s], lens[s]) for s in range(4)]
            luce.luce_decode_step_paged(model, slots, rws, x, ws, logits, am)
            return host(x), host(logits), host(am), host(kp), host(vp)
        slots = [luce.Slot(cuda(flat_k[s]), cuda(flat_v[s]), lens[s]) for s in range(4)]
        luce.luce_decode_step(model, slots, rws, x, ws, logits, am)
        return host(x), host(logits), host(am), [host(sl.k) for sl in slots], [host(sl.v) for sl in slots]

    xf, lf, af, kf, vf = run(False)
    xp, lp, ap, kp, vp = run(True)
    assert np.array_equal(bits(xp), bits(xf)) and np.array_equal(bits(lp), bits(lf)) and np.array_equal(ap, af)
    # the appended rows landed in the right pages, equal to the flat cache's
    for s, (L, n) in enumerate(zip(lens, rws)):
        for j in range(L, L + n):
            pg, off = tables[s][j // PK], j % PK
            assert np.array_equal(kp[pg, :, :, off].view(np.uint16), kf[s][:, :, j].view(np.uint16))
            assert np.array_equal(vp[pg, :, :, off].view(np.uint16), vf[s][:, :, j].view(np.uint16))
    # pages no slot owns are untouched
    owned = set(np.concatenate(tables).tolist())
    for pg in range(n_pages):
        if pg not in owned:
            assert not np.any(kp[pg].view(np.uint16)) and not np.any(vp[pg].view(np.uint16))
