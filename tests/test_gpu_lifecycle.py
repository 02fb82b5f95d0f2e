"""Slot lifecycle through the composed decode step, bit for bit.

"feat(qwen4exp): exact 4-slot concurrent serving", How it stays exact and
Tests: a slot's output depends only on its own history (accepted tokens),
whatever the other slots do; the step writes K/V rows at [len, len + n) and
the caller commits the accepted prefix by advancing len.  Checked here:
  * verify rows with an accepted prefix equal decoding the accepted tokens
    one step at a time, and the next step after the commit is identical too;
  * a cancelled slot reused for a new sequence (len reset, stale cache
    bytes left in place) behaves exactly like a fresh cache;
  * over several steps of mixed row counts and commits, every slot of the
    batched step equals the same slot run alone, and two slots in an
    identical phase stay identical.
"""
import numpy as np
import pytest

from invariant_sequence_decode_gb300 import synth, workloads as wl

torch = pytest.importorskip("torch")
import invariant_sequence_decode_gb300 as luce  # noqa: E402

pytestmark = pytest.mark.gpu

LAYER_FIELDS = ["attn_norm", "wqkv_q", "wqkv_d", "wo_q", "wo_d", "ffn_norm", "wgu_q", "wgu_d", "wdown_q", "wdown_d"]
D = wl.TINY_LAYER
N_LAYERS, CAP, VOCAB = 2, 160, 300


@pytest.fixture(scope="module")
def model():
    from invariant_sequence_decode_gb300 import build
    build.build()
    luce.load_library()
    layers = [luce.LayerTensors(*[cuda(getattr(wl.layer_host(21, l, D), f)) for f in LAYER_FIELDS])
              for l in range(N_LAYERS)]
    fn, hq, hd = wl.head_host(21, D, VOCAB)
    return luce.Model(layers, D.hidden, D.n_q_heads, D.n_kv_heads, D.ffn, rms_eps=D.rms_eps,
                      rope_theta=D.rope_theta, final_norm=cuda(fn), head_q=cuda(hq), head_d=cuda(hd))


def cuda(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    torch.cuda.synchronize()
    return t.cpu().numpy()


def bits(a):
    return np.ascontiguousarray(a).view(np.uint8)


def cache(slot_seed, length):
    """Device K, V [L][Hkv][CAP][128] with `length` cached rows and filler past them."""
    ks, vs = zip(*[wl.cache_host(slot_seed, 0, l, D, CAP, length) for l in range(N_LAYERS)])
    return cuda(np.stack(ks)), cuda(np.stack(vs))


def rows(seed, n):
    return wl.acts(seed, n, D.hidden, sub=5)


def step(model, slots, x_rows, n_rows):
    """One step; slots are (k, v, len).  Returns (hidden rows, logits, argmax)."""
    x = cuda(np.concatenate(x_rows))
    T = x.shape[0]
    logits = torch.empty((T, VOCAB), dtype=torch.float32, device="cuda")
    am = torch.empty(T, dtype=torch.int32, device="cuda")
    ws = model.workspace(T, CAP)
    luce.luce_decode_step(model, [luce.Slot(k, v, ln) for k, v, ln in slots], n_rows, x, ws, logits, am)
    return host(x), host(logits), host(am)


def test_accepted_prefix_then_next_step_equal_one_token_at_a_time(model):
    L = 40
    draft = rows(1, 4)   # four speculative rows
    nxt = rows(2, 1)     # the row after accepting two of them
    # verify history: 4 rows at [L, L + 4), accept 2, then one more step at L + 2
    k1, v1 = cache(7, L)
    hv, lv, av = step(model, [(k1, v1, L)], [draft], [4])
    hn, ln, an = step(model, [(k1, v1, L + 2)], [nxt], [1])
    # sequential history: the two accepted rows one step each, then the same next row
    k2, v2 = cache(7, L)
    hs, ls, as_ = [], [], []
    for j in range(2):
        h, lg, a = step(model, [(k2, v2, L + j)], [draft[j:j + 1]], [1])
        hs.append(h)
        ls.append(lg)
        as_.append(a)
    hn2, ln2, an2 = step(model, [(k2, v2, L + 2)], [nxt], [1])
    for j in range(2):
        assert np.array_equal(bits(hv[j:j + 1]), bits(hs[j])) and np.array_equal(bits(lv[j:j + 1]), bits(ls[j]))
        assert av[j] == as_[j][0]
    assert np.array_equal(bits(hn), bits(hn2)) and np.array_equal(bits(ln), bits(ln2)) and an[0] == an2[0]
    # the committed prefix [0, L + 3) of both caches is identical; the verify
    # history also holds the rejected draft row at L + 3 (scratch, never read)
    for a, b in ((k1, k2), (v1, v2)):
        ha, hb = host(a).view(np.uint16), host(b).view(np.uint16)
        assert np.array_equal(ha[:, :, :L + 3], hb[:, :, :L + 3])
        changed = np.nonzero(np.any(ha != hb, axis=(0, 1, 3)))[0].tolist()
        assert changed == [L + 3]


def test_cancelled_slot_reused_like_a_fresh_cache(model):
    # slot 0 ran a long sequence; it is cancelled (len reset to 0) and reused
    # for a new one while slot 1 keeps decoding; its stale bytes stay in place
    k_old, v_old = cache(8, 120)
    k_new, v_new = cache(9, 0)   # a fresh cache for the same new sequence
    kb, vb = cache(10, 33)       # the other slot, two copies (one per history)
    kb2, vb2 = cache(10, 33)
    new_rows = rows(3, 3)
    other = rows(4, 3)
    for i in range(3):
        hr, lr, ar = step(model, [(k_old, v_old, i), (kb, vb, 33 + i)], [new_rows[i:i + 1], other[i:i + 1]], [1, 1])
        hf, lf, af = step(model, [(k_new, v_new, i), (kb2, vb2, 33 + i)], [new_rows[i:i + 1], other[i:i + 1]],
                          [1, 1])
        assert np.array_equal(bits(hr), bits(hf)) and np.array_equal(bits(lr), bits(lf))
        assert np.array_equal(ar, af)
    # the reused cache holds the new sequence's rows at [0, 3) exactly
    for a, b in ((k_old, k_new), (v_old, v_new)):
        assert np.array_equal(host(a)[:, :, :3].view(np.uint16), host(b)[:, :, :3].view(np.uint16))


def test_phase_soak_batched_equals_solo_and_identical_phases_stay_identical(model):
    # 4 slots over 6 steps with varying row counts and accepted prefixes;
    # slots 0 and 1 share their history and inputs (identical phase)
    lens = [20, 20, 57, 90]
    seeds = [11, 11, 12, 13]
    batched = [cache(s, ln) for s, ln in zip(seeds, lens)]
    solo = [cache(s, ln) for s, ln in zip(seeds, lens)]
    for it in range(6):
        n_rows = [1 + (it + s) % 4 for s in range(4)]
        n_rows[1] = n_rows[0]
        xr = [rows(100 + 10 * it + s, n_rows[s]) for s in range(4)]
        xr[1] = xr[0]
        hb, lb, ab = step(model, [(k, v, ln) for (k, v), ln in zip(batched, lens)], xr, n_rows)
        r0 = 0
        for s in range(4):
            n = n_rows[s]
            hs, ls, as_ = step(model, [(solo[s][0], solo[s][1], lens[s])], [xr[s]], [n])
            assert np.array_equal(bits(hb[r0:r0 + n]), bits(hs)), (it, s)
            assert np.array_equal(bits(lb[r0:r0 + n]), bits(ls)) and np.array_equal(ab[r0:r0 + n], as_)
            r0 += n
        assert np.array_equal(bits(hb[:n_rows[0]]), bits(hb[n_rows[0]:2 * n_rows[0]]))
        # accept a prefix of each slot's rows (at least one), the same for 0 and 1
        acc = [1 + int(synth.int_uniform(500 + it, s, 1, 0, n_rows[s] - 1)[0]) for s in range(4)]
        acc[1] = acc[0]
        lens = [ln + a for ln, a in zip(lens, acc)]
    for s in range(4):
        for a, b in zip(batched[s], solo[s]):
            assert np.array_equal(host(a)[:, :, :lens[s]].view(np.uint16), host(b)[:, :, :lens[s]].view(np.uint16))


def test_host_buffer_step_equals_device_step_bitwise(model):
    """luce_decode_step_host: pinned host rows in, the same step, rows and
    argmax copied back on the stream - the same bits as the device-buffer step."""
    L = 37
    xr = rows(9, 3)
    k1, v1 = cache(14, L)
    hd, ld, ad = step(model, [(k1, v1, L)], [xr], [3])
    k2, v2 = cache(14, L)
    x_in = torch.from_numpy(np.ascontiguousarray(xr)).pin_memory()
    x_out = torch.empty_like(x_in).pin_memory()
    am_out = torch.empty(3, dtype=torch.int32).pin_memory()
    x = torch.empty(x_in.shape, dtype=torch.float32, device="cuda")
    logits = torch.empty((3, VOCAB), dtype=torch.float32, device="cuda")
    am = torch.empty(3, dtype=torch.int32, device="cuda")
    ws = model.workspace(3, CAP)
    luce.luce_decode_step_host(model, [luce.Slot(k2, v2, L)], [3], x_in, x, ws, x_out=x_out, logits=logits,
                               argmax=am, argmax_out=am_out)
    torch.cuda.synchronize()
    assert np.array_equal(bits(x_out.numpy()), bits(hd)) and np.array_equal(am_out.numpy(), ad)
    assert np.array_equal(bits(host(logits)), bits(ld))
    assert np.array_equal(host(k1).view(np.uint16), host(k2).view(np.uint16))
    # the prepared form: the same call twice (slot len advanced by 3 in between)
    k3, v3 = cache(14, L)
    sl = luce.Slot(k3, v3, L)
    plan = luce.HostStep(model, [sl], [3], x_in, x, ws, x_out=x_out, logits=logits, argmax=am, argmax_out=am_out)
    plan()
    torch.cuda.synchronize()
    assert np.array_equal(bits(x_out.numpy()), bits(hd)) and np.array_equal(am_out.numpy(), ad)
    sl.len = L + 3
    plan()
    k4, v4 = cache(14, L)
    step(model, [(k4, v4, L)], [xr], [3])
    h2, _, a2 = step(model, [(k4, v4, L + 3)], [xr], [3])
    torch.cuda.synchronize()
    assert np.array_equal(bits(x_out.numpy()), bits(h2)) and np.array_equal(am_out.numpy(), a2)


def test_prepared_device_step_equals_the_plain_call_bitwise(model):
    """DeviceStep (luce_decode_step with its arguments marshalled once) gives
    the plain call's bits, and follows the slot's len from call to call."""
    L = 37
    xr = rows(11, 3)
    k1, v1 = cache(15, L)
    h1, l1, a1 = step(model, [(k1, v1, L)], [xr], [3])
    h2, l2, a2 = step(model, [(k1, v1, L + 3)], [xr], [3])
    k2, v2 = cache(15, L)
    x = cuda(xr)
    logits = torch.empty((3, VOCAB), dtype=torch.float32, device="cuda")
    am = torch.empty(3, dtype=torch.int32, device="cuda")
    sl = luce.Slot(k2, v2, L)
    ds = luce.DeviceStep(model, [sl], [3], x, model.workspace(3, CAP), logits=logits, argmax=am)
    ds()
    assert np.array_equal(bits(host(x)), bits(h1)) and np.array_equal(bits(host(logits)), bits(l1))
    assert np.array_equal(host(am), a1)
    x.copy_(cuda(xr))
    sl.len = L + 3
    ds()
    assert np.array_equal(bits(host(x)), bits(h2)) and np.array_equal(host(am), a2)
    assert np.array_equal(host(k1).view(np.uint16), host(k2).view(np.uint16))
    assert np.array_equal(host(v1).view(np.uint16), host(v2).view(np.uint16))
