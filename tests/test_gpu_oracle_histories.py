"""Slot lifecycles, paged caches and wide composed steps against the oracle.

The lifecycle and paged tests elsewhere compare the GPU with other GPU runs
(bit for bit).  Here the same histories run through the oracle as well:

  * "feat(qwen4exp): exact 4-slot concurrent serving", Tests: a verify step
    whose accepted prefix is committed, then the next step; a cancelled slot
    reset and reused for a new sequence.  The oracle runs the same history
    (its own caches, the same commits) over both layers and the head; the
    GPU's hidden rows and logits stay within the free-running tolerances,
    and every step's last layer is checked stage by stage against the oracle
    fed the GPU's own stage inputs.
  * Paged K/V: each paged sequence's pages gathered into a flat array on the
    host and attended by the oracle (2e-3 absolute), and a paged step checked
    stage by stage against the oracle over the gathered caches.
  * Composed steps at 8 and 12 rows (4 slots x 2 and x 3 rows), where every
    projection runs on the tensor-core matvec and the q|k|v projection
    applies RoPE and appends K/V in its epilogue: stage by stage against the
    oracle, on the small stack and on the 27B-shaped layer.
"""
import math
import os

import numpy as np
import pytest

import oracle
from invariant_sequence_decode_gb300 import workloads as wl

torch = pytest.importorskip("torch")
import invariant_sequence_decode_gb300 as luce  # noqa: E402
from test_gpu_paged import page_tables  # noqa: E402
from test_gpu_step import LAYER_FIELDS, Case, rel_err, staged_layer_check  # noqa: E402

pytestmark = pytest.mark.gpu

D = wl.TINY_LAYER
N_LAYERS, CAP, VOCAB = 2, 160, 300
PK = luce.PAGE_KEYS
oracle.set_threads(os.cpu_count() or 1)  # the same bits on any thread count, faster


def cuda(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    torch.cuda.synchronize()
    return t.cpu().numpy()


class Stack:
    """The small 2-layer model with a head, on the device and on the host."""

    def __init__(self, seed=21):
        self.dims = D
        self.n_layers = N_LAYERS
        self.cap = CAP
        self.vocab = VOCAB
        self.layers_h = [wl.layer_host(seed, l, D) for l in range(N_LAYERS)]
        self.head_h = wl.head_host(seed, D, VOCAB)
        fn, hq, hd = [cuda(a) for a in self.head_h]
        self.model = luce.Model([luce.LayerTensors(*[cuda(getattr(L, f)) for f in LAYER_FIELDS])
                                 for L in self.layers_h], D.hidden, D.n_q_heads, D.n_kv_heads, D.ffn,
                                rms_eps=D.rms_eps, rope_theta=D.rope_theta, final_norm=fn, head_q=hq, head_d=hd)
        self.odims = oracle.Dims(D.hidden, D.n_q_heads, D.n_kv_heads, D.head_dim, D.ffn)
        self.lw = [oracle.LayerWeights(*[getattr(L, f) for f in LAYER_FIELDS]) for L in self.layers_h]


@pytest.fixture(scope="module")
def stack():
    from invariant_sequence_decode_gb300 import build
    build.build()
    luce.load_library()
    return Stack()


def caches(slot_seed, length):
    """Host K, V [L][Hkv][CAP][128] (fp16) with `length` cached rows."""
    ks, vs = zip(*[wl.cache_host(slot_seed, 0, l, D, CAP, length) for l in range(N_LAYERS)])
    return np.stack(ks), np.stack(vs)


class Seq:
    """One sequence followed on both sides: device caches and the oracle's."""

    def __init__(self, k, v, length):
        self.k, self.v = cuda(k), cuda(v)
        self.ok = [k[l].view(np.uint16).copy() for l in range(N_LAYERS)]
        self.ov = [v[l].view(np.uint16).copy() for l in range(N_LAYERS)]
        self.len = length


class View:
    """What staged_layer_check reads of a run: the model, its sizes and the slots' lengths."""

    def __init__(self, st, lens):
        self.__dict__.update(st.__dict__)
        self.lens = lens


def step_both(st, seqs, x_rows, n_rows):
    """One step on the GPU and in the oracle over the same history.  Returns
    the GPU run (for staged checks) and the oracle's hidden rows and logits."""
    x = np.concatenate(x_rows).astype(np.float32)
    T = x.shape[0]
    xd = cuda(x)
    logits = torch.empty((T, VOCAB), dtype=torch.float32, device="cuda")
    am = torch.empty(T, dtype=torch.int32, device="cuda")
    ws = st.model.workspace(T, CAP)
    slots = [luce.Slot(s.k, s.v, s.len) for s in seqs]
    luce.luce_decode_step(st.model, slots, n_rows, xd, ws, logits, am)
    out = dict(x=host(xd), ws=ws, slots=slots, logits=host(logits), argmax=host(am), T=T, rows=list(n_rows),
               idx=list(range(len(seqs))))
    xo = x.astype(np.float64)
    for l in range(N_LAYERS):
        osl = [oracle.Slot(s.ok[l], s.ov[l], s.len) for s in seqs]
        xo = oracle.decode_layer(xo, st.lw[l], st.odims, osl, n_rows)
    fn, wq, wd = st.head_h
    lo = oracle.lm_head(xo, fn, wq, wd, D.rms_eps)
    return out, xo, lo


def check(st, seqs, out, xo, lo):
    # free-running tolerances of the 3-layer test (a few +-1 code flips at the
    # quantization points move a row by ~1/(127 sqrt(K)) of its norm each)
    assert np.all(rel_err(out["x"].astype(np.float64), xo) <= 2e-3)
    assert np.all(rel_err(out["logits"].astype(np.float64), lo) <= 5e-3)
    staged_layer_check(View(st, [s.len for s in seqs]), out, layer=N_LAYERS - 1)


def test_accepted_prefix_history_matches_the_oracle(stack):
    L = 40
    seq = Seq(*caches(7, L), L)
    draft = wl.acts(1, 4, D.hidden, sub=5)
    out, xo, lo = step_both(stack, [seq], [draft], [4])           # verify 4 rows at [L, L + 4)
    check(stack, [seq], out, xo, lo)
    seq.len = L + 2                                               # accept 2
    nxt = wl.acts(2, 1, D.hidden, sub=5)
    out, xo, lo = step_both(stack, [seq], [nxt], [1])             # the next row at L + 2
    check(stack, [seq], out, xo, lo)
    seq.len = L + 3
    out, xo, lo = step_both(stack, [seq], [wl.acts(3, 2, D.hidden, sub=5)], [2])  # and a 2-row verify after it
    check(stack, [seq], out, xo, lo)


def test_cancelled_and_reused_slot_matches_the_oracle(stack):
    # slot 0's cache held a 120-token sequence; it is cancelled (len reset to
    # 0) and reused for a new sequence with its stale bytes in place, while
    # slot 1 keeps decoding.  The oracle runs the new sequence on a cache
    # that never held the old one.
    old_k, old_v = caches(8, 120)
    fresh_k, fresh_v = caches(9, 0)
    reused = Seq(old_k, old_v, 0)
    reused.ok = [fresh_k[l].view(np.uint16).copy() for l in range(N_LAYERS)]
    reused.ov = [fresh_v[l].view(np.uint16).copy() for l in range(N_LAYERS)]
    other = Seq(*caches(10, 33), 33)
    new_rows, other_rows = wl.acts(3, 3, D.hidden, sub=6), wl.acts(4, 3, D.hidden, sub=6)
    for i in range(3):
        out, xo, lo = step_both(stack, [reused, other], [new_rows[i:i + 1], other_rows[i:i + 1]], [1, 1])
        check(stack, [reused, other], out, xo, lo)
        reused.len += 1
        other.len += 1


@pytest.mark.parametrize("lens,nq,Hq,Hkv", [
    ([17, 128, 129, 2051], [1, 1, 2, 4], 40, 8),
    ([1, 300, 16385], [1, 3, 1], 32, 8),
])
def test_paged_attention_matches_the_oracle(lens, nq, Hq, Hkv):
    d = wl.Dims(0, Hq, Hkv, 128, 0)
    spans = [-(-L // PK) for L in lens]
    tables, n_pages = page_tables(15, spans)
    kpool = np.zeros((n_pages, Hkv, PK, 128), np.float16)
    vpool = np.zeros_like(kpool)
    for s, L in enumerate(lens):
        k, v = wl.cache_host(16, s, 0, d, spans[s] * PK, L)
        for p, pg in enumerate(tables[s]):
            kpool[pg] = k[:, p * PK:(p + 1) * PK]
            vpool[pg] = v[:, p * PK:(p + 1) * PK]
    T = sum(nq)
    q = wl.qvec(16, T, Hq)
    kp, vp = cuda(kpool), cuda(vpool)
    views, row0 = [], 0
    for s, L in enumerate(lens):
        views.append(luce.PagedView(kp, vp, cuda(tables[s]), L, nq[s], row0))
        row0 += nq[s]
    scale = 1.0 / math.sqrt(128)
    got = host(luce.luce_decode_attn_paged(cuda(q), views, Hkv, scale))
    r = 0
    for s, L in enumerate(lens):
        # the sequence's pages gathered in table order into a flat [Hkv][L][128] cache
        flat_k = np.concatenate([kpool[pg] for pg in tables[s]], axis=1)
        flat_v = np.concatenate([vpool[pg] for pg in tables[s]], axis=1)
        for j in range(nq[s]):
            ref = oracle.attention_row(q[r], flat_k, flat_v, L - nq[s] + 1 + j, Hkv, scale)
            assert np.max(np.abs(got[r] - ref)) <= 2e-3, (s, j)
            r += 1


class GatheredSlot:
    """A paged slot's pages gathered into flat [L][Hkv][cap][128] device caches."""

    def __init__(self, k, v):
        self.k, self.v = k, v


def test_paged_step_matches_the_oracle_stage_by_stage(stack):
    rws = [1, 2, 3, 4]
    lens = [5, 127, 128, 300]
    spans = [-(-(L + n) // PK) for L, n in zip(lens, rws)]
    tables, n_pages = page_tables(17, spans)
    Hkv = D.n_kv_heads
    kpool = np.zeros((n_pages, N_LAYERS, Hkv, PK, 128), np.float16)
    vpool = np.zeros_like(kpool)
    for s, L in enumerate(lens):
        ks, vs = zip(*[wl.cache_host(18, s, l, D, spans[s] * PK, L) for l in range(N_LAYERS)])
        k, v = np.stack(ks), np.stack(vs)
        for p, pg in enumerate(tables[s]):
            kpool[pg] = k[:, :, p * PK:(p + 1) * PK]
            vpool[pg] = v[:, :, p * PK:(p + 1) * PK]
    T = sum(rws)
    x = cuda(wl.acts(19, T, D.hidden, sub=2))
    logits = torch.empty((T, VOCAB), dtype=torch.float32, device="cuda")
    am = torch.empty(T, dtype=torch.int32, device="cuda")
    ws = stack.model.workspace(T, max(spans) * PK)
    kp, vp = cuda(kpool), cuda(vpool)
    luce.luce_decode_step_paged(stack.model, [luce.PagedSlot(kp, vp, tables[s], lens[s]) for s in range(4)], rws,
                                x, ws, logits, am)
    kh, vh = host(kp), host(vp)
    gathered = []
    for s in range(4):
        gk = np.concatenate([kh[pg] for pg in tables[s]], axis=2)   # [L][Hkv][spans*128][128]
        gv = np.concatenate([vh[pg] for pg in tables[s]], axis=2)
        gathered.append(GatheredSlot(cuda(gk), cuda(gv)))
    out = dict(x=host(x), ws=ws, slots=gathered, logits=host(logits), argmax=host(am), T=T, rows=rws,
               idx=[0, 1, 2, 3])
    view = View(stack, lens)
    view.cap = max(spans) * PK
    staged_layer_check(view, out, layer=N_LAYERS - 1)


@pytest.mark.parametrize("rows_per_slot", [2, 3])
def test_wide_step_small_stack_stages_match_the_oracle(rows_per_slot):
    """8 and 12 rows through two layers and the head."""
    case = Case(41 + rows_per_slot, wl.TINY_LAYER, 2, [3, 60, 129, 250], [rows_per_slot] * 4, cap=256, vocab=400)
    staged_layer_check(case, case.run(), layer=1)


@pytest.mark.parametrize("rows_per_slot", [2, 3])
def test_wide_step_27b_layer_stages_match_the_oracle(rows_per_slot):
    """8 and 12 rows through the 27B-shaped layer (every projection on the
    tensor-core matvec, the q|k|v projection with RoPE and the K/V append in
    its epilogue)."""
    case = Case(1, wl.LAYER27B, 1, [2050 - rows_per_slot] * 4, [rows_per_slot] * 4, cap=2050)
    staged_layer_check(case, case.run())
