"""Pins of the CPU oracle against things other than itself.

Each check uses a library routine, a closed form, an invariant, a hand-worked
fixture or brute force, chosen so that a plausible slip in the oracle (a
dropped term, a wrong sign or index, a transposed operand, a wrong pairing)
fails at least one of them.  CPU only.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
rng = np.random.default_rng(1234)


def rand_w(N, K):
    wq = rng.integers(-127, 128, size=(N, K), dtype=np.int64).astype(np.int8)
    wd = (np.abs(rng.normal(0, 0.02, size=(N, K // 32))) / 127).astype(np.float16)
    return wq, wd


# ----------------------------------------------------------- binary16

def test_half_decode_all_bit_patterns_match_numpy():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = oracle.half_to_double(bits)
    fin = np.isfinite(ref)
    assert np.array_equal(got[fin], ref[fin])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(np.isinf(got) & (got > 0), np.isinf(ref) & (ref > 0))


def test_float_to_half_rounding_matches_numpy():
    x = np.concatenate([rng.normal(0, 3, 4000), rng.normal(0, 1e-5, 2000), [65504.0, 65519.0, 65520.0,
                       6.1e-5, 5.96e-8, 2.98e-8, 2.99e-8, -0.0, 0.0, 1.0 + 2 ** -11, 1.0 + 3 * 2 ** -11]]).astype(np.float32)
    got = oracle.float_to_half_bits(x)
    ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, ref)


# ----------------------------------------------------------- quantizer

def test_quantize_hand_worked_ties():
    rows = [l.split() for l in open(os.path.join(HERE, "golden", "q8_ties.txt")) if l.strip() and not l.startswith("#")]
    x = np.array([float(a) for a, _ in rows], np.float32)
    want = np.array([int(b) for _, b in rows], np.int8)
    assert x.size == 32 and np.max(np.abs(x)) == 127.0
    q, d = oracle.quantize_act(x[None])
    assert d[0, 0] == np.float32(1.0)
    assert np.array_equal(q[0], want)


def test_quantize_constant_and_zero_blocks():
    x = np.zeros((3, 64), np.float32)
    x[0, :32] = 5.0
    x[1, 32:] = -0.125
    q, d = oracle.quantize_act(x)
    assert np.all(q[0, :32] == 127) and d[0, 0] == np.float32(5.0) / np.float32(127.0)
    assert np.all(q[1, 32:] == -127)
    assert d[0, 1] == 0 and np.all(q[0, 32:] == 0)
    assert np.all(q[2] == 0) and np.all(d[2] == 0)


def test_quantize_nearest_code_and_extremes_on_random_blocks():
    x = (rng.normal(0, 1, (8, 1024)) * rng.uniform(1e-3, 1e3, (8, 1))).astype(np.float32)
    q, d = oracle.quantize_act(x)
    xb = x.reshape(8, 32, 32).astype(np.float64)
    qb = q.reshape(8, 32, 32).astype(np.float64)
    db = d.astype(np.float64)[..., None]
    # every code is the nearest multiple of d (within fp32 rounding of x / d)
    assert np.all(np.abs(xb - qb * db) <= db * (0.5 + 1e-6))
    # the largest magnitude maps to +-127 and signs are kept
    i = np.argmax(np.abs(xb), axis=2)
    ext = np.take_along_axis(qb, i[..., None], 2)[..., 0]
    sg = np.sign(np.take_along_axis(xb, i[..., None], 2)[..., 0])
    assert np.all(ext == 127 * sg)
    assert np.all((np.sign(qb) == np.sign(xb)) | (qb == 0))
    assert np.all(np.abs(qb) <= 127)


def test_quantize_nan_entry_is_zero_and_ignored_by_amax():
    x = np.linspace(-2, 2, 32).astype(np.float32)
    q0, d0 = oracle.quantize_act(x[None])
    x2 = x.copy()
    x2[5] = np.nan
    q1, d1 = oracle.quantize_act(x2[None])
    assert d1[0, 0] == d0[0, 0]
    assert q1[0, 5] == 0
    keep = np.arange(32) != 5
    assert np.array_equal(q1[0, keep], q0[0, keep])


# ----------------------------------------------------------- block dots / matvec

def test_block_dots_match_numpy_int64_einsum():
    wq, _ = rand_w(7, 96)
    aq = rng.integers(-127, 128, size=(3, 96)).astype(np.int8)
    got = oracle.block_dots(wq, aq)
    ref = np.einsum("nbi,tbi->tnb", wq.reshape(7, 3, 32).astype(np.int64), aq.reshape(3, 3, 32).astype(np.int64))
    assert np.array_equal(got, ref)


def test_block_dot_extreme_magnitude_is_exact():
    wq = np.full((1, 32), -127, np.int8)
    aq = np.full((1, 32), -127, np.int8)
    assert oracle.block_dots(wq, aq)[0, 0, 0] == 32 * 127 * 127


def test_matvec_equals_dequantize_then_dot():
    N, K, T = 40, 256, 4
    wq, wd = rand_w(N, K)
    x = rng.normal(0, 1, (T, K)).astype(np.float32)
    aq, ad = oracle.quantize_act(x)
    y = oracle.matvec(wq, wd, aq, ad)
    W = wq.astype(np.float64) * np.repeat(wd.astype(np.float64), 32, axis=1)
    A = aq.astype(np.float64) * np.repeat(ad.astype(np.float64), 32, axis=1)
    ref = A @ W.T
    assert y.shape == (T, N)
    assert np.max(np.abs(y - ref)) <= 1e-12 * np.max(np.abs(ref))


def test_matvec_one_hot_activation_selects_a_scaled_weight():
    N, K = 9, 128
    wq, wd = rand_w(N, K)
    for k in (0, 31, 32, 77, 127):
        aq = np.zeros((1, K), np.int8)
        ad = np.zeros((1, K // 32), np.float32)
        aq[0, k] = 1
        ad[0, k // 32] = 1.0
        y = oracle.matvec(wq, wd, aq, ad)[0]
        assert np.array_equal(y, wd[:, k // 32].astype(np.float64) * wq[:, k].astype(np.float64))


def test_matvec_rows_are_independent_of_batch_and_order():
    N, K = 16, 160
    wq, wd = rand_w(N, K)
    x = rng.normal(0, 1, (4, K)).astype(np.float32)
    aq, ad = oracle.quantize_act(x)
    yb = oracle.matvec(wq, wd, aq, ad)
    perm = np.array([2, 0, 3, 1])
    yp = oracle.matvec(wq, wd, aq[perm], ad[perm])
    assert np.array_equal(yp, yb[perm])
    for t in range(4):
        assert np.array_equal(oracle.matvec(wq, wd, aq[t:t + 1], ad[t:t + 1])[0], yb[t])


# ----------------------------------------------------------- RMSNorm

def test_rmsnorm_closed_forms():
    H = 64
    g = np.ones(H, np.float32)
    c = 3.0
    y = oracle.rmsnorm(np.full((1, H), c), g, 1e-6)
    assert np.allclose(y, c / math.sqrt(c * c + 1e-6), rtol=0, atol=1e-15)
    x = rng.normal(0, 2, (3, H))
    y0 = oracle.rmsnorm(x, g, 0.0)
    assert np.allclose(np.sqrt(np.mean(y0 ** 2, axis=1)), 1.0, atol=1e-14)
    assert np.allclose(oracle.rmsnorm(7.5 * x, g, 0.0), y0, atol=1e-14)
    gam = rng.normal(1, 0.1, H).astype(np.float32)
    assert np.allclose(oracle.rmsnorm(x, gam, 0.0), y0 * gam.astype(np.float64), atol=1e-14)


# ----------------------------------------------------------- RoPE

def test_rope_position_zero_is_identity():
    x = rng.normal(0, 1, (2, 3, 128))
    assert np.array_equal(oracle.rope(x, np.zeros(2, np.int32), 1e6), x)


def test_rope_preserves_pair_norms_and_composes():
    x = rng.normal(0, 1, (3, 2, 128))
    p1 = np.array([5, 1000, 32767], np.int32)
    y = oracle.rope(x, p1, 1e6)
    n0 = x[..., :64] ** 2 + x[..., 64:] ** 2
    n1 = y[..., :64] ** 2 + y[..., 64:] ** 2
    assert np.allclose(n0, n1, rtol=1e-13)
    p2 = np.array([7, 3, 11], np.int32)
    assert np.allclose(oracle.rope(y, p2, 1e6), oracle.rope(x, p1 + p2, 1e6), atol=1e-9)


def test_rope_pairs_half_split_dims_and_first_pair_turns_by_pos_radians():
    D = 128
    for i in (0, 5, 63):
        x = np.zeros((1, 1, D))
        x[0, 0, i] = 1.0
        pos = 3
        y = oracle.rope(x, np.array([pos], np.int32), 1e6)[0, 0]
        nz = set(np.nonzero(np.abs(y) > 1e-15)[0].tolist())
        assert nz <= {i, i + 64}
        ang = pos * (1e6 ** (-2.0 * i / D))
        assert math.isclose(y[i], math.cos(ang), abs_tol=1e-15)
        assert math.isclose(y[i + 64], math.sin(ang), abs_tol=1e-15)


def test_rope_scores_depend_only_on_relative_position():
    q = rng.normal(0, 1, (1, 1, 128))
    k = rng.normal(0, 1, (1, 1, 128))
    def score(pq, pk):
        return float(np.sum(oracle.rope(q, np.array([pq], np.int32), 1e6) * oracle.rope(k, np.array([pk], np.int32), 1e6)))
    assert math.isclose(score(10, 3), score(1010, 1003), rel_tol=1e-9, abs_tol=1e-9)
    assert not math.isclose(score(10, 3), score(10, 4), rel_tol=1e-6)


# ----------------------------------------------------------- attention

def f16(a):
    return np.asarray(a, np.float64).astype(np.float16)


def test_attention_single_key_returns_its_value():
    Hq, Hkv, D = 4, 2, 128
    q = rng.normal(0, 1, (Hq, D))
    k = f16(rng.normal(0, 1, (Hkv, 5, D)))
    v = f16(rng.normal(0, 1, (Hkv, 5, D)))
    out = oracle.attention_row(q, k, v, 1, Hkv, 1 / math.sqrt(D))
    for h in range(Hq):
        assert np.array_equal(out[h], v[h // 2, 0].astype(np.float64))


def test_attention_equal_keys_and_zero_query_give_mean_value():
    Hq, Hkv, D, L = 4, 1, 128, 37
    kk = f16(rng.normal(0, 1, (Hkv, 1, D)))
    k = np.repeat(kk, L, axis=1)
    v = f16(rng.normal(0, 1, (Hkv, L, D)))
    mean = v.astype(np.float64).mean(axis=1)[0]
    out = oracle.attention_row(rng.normal(0, 1, (Hq, D)), k, v, L, Hkv, 1 / math.sqrt(D))
    assert np.allclose(out, mean[None], atol=1e-13)
    k2 = f16(rng.normal(0, 1, (Hkv, L, D)))
    out0 = oracle.attention_row(np.zeros((Hq, D)), k2, v, L, Hkv, 1 / math.sqrt(D))
    assert np.allclose(out0, mean[None], atol=1e-13)


def test_attention_gqa_maps_query_head_to_kv_head_by_integer_division():
    Hq, Hkv, D, L = 8, 2, 128, 9
    v = np.zeros((Hkv, L, D), np.float16)
    v[0] = 1.0
    v[1] = -2.0
    k = f16(rng.normal(0, 1, (Hkv, L, D)))
    out = oracle.attention_row(rng.normal(0, 1, (Hq, D)), k, v, L, Hkv, 1 / math.sqrt(D))
    for h in range(Hq):
        assert np.allclose(out[h], 1.0 if h < 4 else -2.0, atol=1e-13)


def test_attention_matches_library_softmax_and_ignores_keys_past_len():
    from scipy.special import softmax
    Hq, Hkv, D, cap, L = 4, 2, 128, 50, 33
    q = rng.normal(0, 1, (Hq, D))
    k = f16(rng.normal(0, 1, (Hkv, cap, D)))
    v = f16(rng.normal(0, 1, (Hkv, cap, D)))
    sc = 1 / math.sqrt(D)
    out = oracle.attention_row(q, k, v, L, Hkv, sc)
    for h in range(Hq):
        g = h // 2
        K = k[g, :L].astype(np.float64)
        V = v[g, :L].astype(np.float64)
        ref = softmax(sc * (K @ q[h])) @ V
        assert np.allclose(out[h], ref, atol=1e-12)
    k2, v2 = k.copy(), v.copy()
    k2[:, L:] = 100.0
    v2[:, L:] = -100.0
    assert np.array_equal(oracle.attention_row(q, k2, v2, L, Hkv, sc), out)


def test_attention_dominant_key_selects_its_value():
    Hq, Hkv, D, L = 2, 1, 128, 20
    q = np.zeros((Hq, D))
    q[:, 0] = 1.0
    k = np.zeros((Hkv, L, D), np.float16)
    k[0, 13, 0] = 60000.0
    v = f16(rng.normal(0, 1, (Hkv, L, D)))
    out = oracle.attention_row(q, k, v, L, Hkv, 1 / math.sqrt(D))
    assert np.allclose(out, v[0, 13].astype(np.float64)[None], atol=1e-12)


# ----------------------------------------------------------- SwiGLU / argmax

def test_swiglu_identities_and_gate_first_order():
    g = rng.normal(0, 3, (2, 50))
    one = np.ones_like(g)
    h_pos = oracle.swiglu(np.concatenate([g, one], axis=1))
    h_neg = oracle.swiglu(np.concatenate([-g, one], axis=1))
    assert np.allclose(h_pos - h_neg, g, atol=1e-13)  # silu(x) - silu(-x) = x
    assert np.all(oracle.swiglu(np.concatenate([np.zeros_like(g), g], axis=1)) == 0)
    big = oracle.swiglu(np.array([[40.0, -40.0, 2.0, 3.0]]))
    assert math.isclose(big[0, 0], 80.0, rel_tol=1e-15) and abs(big[0, 1]) < 1e-15


def test_argmax_lowest_index_on_ties_and_skips_nan():
    x = np.array([[1, 3, 3, 2], [np.nan, -1, -1, -5], [0, 0, 0, 0]], np.float32)
    assert oracle.argmax(x).tolist() == [1, 1, 0]
    r = rng.normal(0, 1, (5, 1000)).astype(np.float32)
    assert np.array_equal(oracle.argmax(r), np.argmax(r, axis=1))


# ----------------------------------------------------------- the layer

def tiny_layer(seed=0, H=128, Hq=4, Hkv=2, D=128, F=192):
    r = np.random.default_rng(seed)
    def w(n, k):
        return (r.integers(-127, 128, size=(n, k)).astype(np.int8),
                (np.abs(r.normal(0, 0.02, (n, k // 32))) / 127).astype(np.float16))
    qkv = w((Hq + 2 * Hkv) * D, H)
    wo = w(H, Hq * D)
    gu = w(2 * F, H)
    dn = w(H, F)
    lw = oracle.LayerWeights(r.normal(1, 0.1, H).astype(np.float32), *qkv, *wo,
                             r.normal(1, 0.1, H).astype(np.float32), *gu, *dn)
    return lw, oracle.Dims(H, Hq, Hkv, D, F)


def make_slot(r, dims, length, cap=64):
    k = r.normal(0, 1, (dims.n_kv_heads, cap, dims.head_dim)).astype(np.float16).view(np.uint16)
    v = r.normal(0, 1, (dims.n_kv_heads, cap, dims.head_dim)).astype(np.float16).view(np.uint16)
    return oracle.Slot(k, v, length)


def clone(s):
    return oracle.Slot(s.k.copy(), s.v.copy(), s.len)


def test_layer_with_zero_output_scales_is_the_identity():
    lw, dims = tiny_layer()
    lw.wo_d[:] = 0
    lw.wdown_d[:] = 0
    r = np.random.default_rng(5)
    x = r.normal(0, 1, (2, dims.hidden)).astype(np.float32)
    out = oracle.decode_layer(x, lw, dims, [make_slot(r, dims, 3), make_slot(r, dims, 9)], [1, 1])
    assert np.array_equal(out, x.astype(np.float64))


def test_layer_first_token_attends_to_itself_only():
    lw, dims = tiny_layer()
    r = np.random.default_rng(6)
    x = r.normal(0, 1, (1, dims.hidden)).astype(np.float32)
    tr = {}
    oracle.decode_layer(x, lw, dims, [make_slot(r, dims, 0)], [1], trace=tr)
    v16 = tr["v"][0].astype(np.float16).astype(np.float64)  # [Hkv][D]
    for h in range(dims.n_q_heads):
        assert np.array_equal(tr["attn"][0, h], v16[h // 2])


def test_layer_batched_equals_solo_permutation_and_isolation():
    lw, dims = tiny_layer(seed=3)
    r = np.random.default_rng(7)
    slots = [make_slot(r, dims, L) for L in (5, 17, 30)]
    rows = [2, 1, 3]
    x = r.normal(0, 1, (6, dims.hidden)).astype(np.float32)
    bs = [clone(s) for s in slots]
    yb = oracle.decode_layer(x, lw, dims, bs, rows)
    r0 = 0
    for i, (s, n) in enumerate(zip(slots, rows)):
        ss = clone(s)
        ys = oracle.decode_layer(x[r0:r0 + n], lw, dims, [ss], [n])
        assert np.array_equal(ys, yb[r0:r0 + n])
        assert np.array_equal(ss.k, bs[i].k) and np.array_equal(ss.v, bs[i].v)
        r0 += n
    # slot order permuted: rows move with their slot, values unchanged
    order = [2, 0, 1]
    starts = np.cumsum([0] + rows)
    xp = np.concatenate([x[starts[i]:starts[i] + rows[i]] for i in order])
    yp = oracle.decode_layer(xp, lw, dims, [clone(slots[i]) for i in order], [rows[i] for i in order])
    assert np.array_equal(yp, np.concatenate([yb[starts[i]:starts[i] + rows[i]] for i in order]))
    # a slot left out of the batch is untouched
    bystander = clone(slots[1])
    before = (bystander.k.copy(), bystander.v.copy())
    oracle.decode_layer(x[:2], lw, dims, [clone(slots[0])], [2])
    assert np.array_equal(bystander.k, before[0]) and np.array_equal(bystander.v, before[1])


def test_layer_verify_rows_are_causal():
    lw, dims = tiny_layer(seed=4)
    r = np.random.default_rng(8)
    s = make_slot(r, dims, 11)
    x = r.normal(0, 1, (4, dims.hidden)).astype(np.float32)
    y = oracle.decode_layer(x, lw, dims, [clone(s)], [4])
    x2 = x.copy()
    x2[3] += 1.0
    y2 = oracle.decode_layer(x2, lw, dims, [clone(s)], [4])
    assert np.array_equal(y[:3], y2[:3]) and not np.array_equal(y[3], y2[3])
    x3 = x.copy()
    x3[0] += 1.0
    y3 = oracle.decode_layer(x3, lw, dims, [clone(s)], [4])
    assert all(not np.array_equal(y[j], y3[j]) for j in range(4))


# ----------------------------------------------------------- the half-scale quantizer

def half_bits_of(v):
    return int(np.array([v], np.float16).view(np.uint16)[0])


def test_quantize_f16_equals_the_fp32_form_when_the_scale_is_a_half():
    # amax = 127 * (a binary16 value): amax / 127 is exact in fp32 and in
    # binary16, so both forms must give the same codes and the same scale
    r = np.random.default_rng(41)
    halves = [1.0, 0.5, 3.0, 1024.0, 65504.0, 2.0 ** -14, 2.0 ** -20, 1.5 * 2.0 ** -17]
    x = r.uniform(-1, 1, (len(halves), 32)).astype(np.float32)
    for i, h in enumerate(halves):
        x[i] *= np.float32(127 * h) / np.max(np.abs(x[i]))
        x[i, i] = np.float32(127 * h) * (1 if i % 2 else -1)
    assert np.all(np.max(np.abs(x), axis=1) == np.float32(127) * np.array(halves, np.float32))
    q16, d16 = oracle.quantize_act_f16(x)
    q32, d32 = oracle.quantize_act(x)
    assert np.array_equal(q16, q32)
    assert np.array_equal(d16[:, 0], np.array([half_bits_of(h) for h in halves], np.uint16))
    assert np.array_equal(d16.view(np.float16).astype(np.float32), d32)


def test_quantize_f16_hand_worked_ties():
    rows = [l.split() for l in open(os.path.join(HERE, "golden", "q8_ties.txt")) if l.strip() and not l.startswith("#")]
    x = np.array([float(a) for a, _ in rows], np.float32)
    want = np.array([int(b) for _, b in rows], np.int8)
    q, d = oracle.quantize_act_f16(x[None])
    assert d[0, 0] == half_bits_of(1.0) and np.array_equal(q[0], want)


def test_quantize_f16_overflow_is_stored_as_the_largest_finite_half():
    x = np.zeros((4, 32), np.float32)
    x[0, :] = np.float32(127.0 * 65504.0)          # exactly the largest half: no guard needed
    x[1, :] = np.float32(127.0 * 65520.0)          # amax / 127 rounds to inf in binary16
    x[1, 3] = -np.float32(127.0 * 65520.0)
    x[2, :] = np.float32(1.0)
    x[2, 7] = np.float32(np.inf)                   # an infinite entry
    x[3, :] = np.float32(127.0 * 65519.0)          # just below the rounding boundary: rounds to 65504
    q, d = oracle.quantize_act_f16(x)
    assert np.all(d[:, 0] == 0x7BFF)
    assert np.all(q[0] == 127)
    assert np.all(q[1][np.arange(32) != 3] == 127) and q[1, 3] == -127
    assert q[2, 7] == 127 and np.all(q[2][np.arange(32) != 7] == 0)   # 1 / 65504 rounds to 0
    assert np.all(q[3] == 127)
    assert np.all(np.isfinite(d.view(np.float16)))


def test_quantize_f16_subnormal_and_underflowing_scales():
    x = np.zeros((3, 32), np.float32)
    x[0] = np.float32(127.0 * 2.0 ** -20) * np.linspace(-1, 1, 32, dtype=np.float32)   # subnormal half scale
    x[1] = np.float32(127.0 * 2.0 ** -26)                                           # rounds to zero
    x[2] = np.float32(127.0 * 1.5 * 2.0 ** -25)                                     # rounds up to 2^-24
    q, d = oracle.quantize_act_f16(x)
    assert d[0, 0] == 0x0010                                    # 2^-20 = 16 * 2^-24
    s0 = np.float32(2.0 ** -20)
    want0 = np.clip(np.sign(x[0]) * np.floor(np.abs(x[0] / s0) + np.float32(0.5)), -127, 127)
    assert np.array_equal(q[0], want0.astype(np.int8))
    assert d[1, 0] == 0 and np.all(q[1] == 0)
    assert d[2, 0] == 0x0001
    assert np.all(q[2] == 95)                                    # 127 * 1.5 * 2^-25 / 2^-24 = 95.25 -> 95


# ----------------------------------------------------------- hand compositions (numpy, float64)
#
# The layer and the head written out again from their definitions with numpy
# only (the quantizer, pinned above, is the one oracle routine they call):
# RMSNorm x / sqrt(mean(x^2) + eps) * gamma; every projection is the q8_0
# activation quantization of its fp32 input followed by the dequantized
# float64 product; silu(g) * u with the gate half first.


def np_rmsnorm(x, gamma, eps):
    x = np.asarray(x, np.float64)
    return x / np.sqrt(np.mean(x * x, axis=1, keepdims=True) + eps) * gamma.astype(np.float64)


def np_q8_project(x32, wq, wd):
    """q8_0 activations of fp32 rows x32 times q8_0 weights, dequantized, float64."""
    aq, ad = oracle.quantize_act(x32)
    a = aq.astype(np.float64) * np.repeat(ad.astype(np.float64), 32, axis=1)
    w = wq.astype(np.float64) * np.repeat(wd.astype(np.float64), 32, axis=1)
    return a @ w.T


def np_ffn(x1, lw, eps):
    xn2 = np_rmsnorm(x1, lw.ffn_norm, eps).astype(np.float32)
    gu = np_q8_project(xn2, lw.wgu_q, lw.wgu_d)
    F = gu.shape[1] // 2
    g, u = gu[:, :F], gu[:, F:]
    h = (g / (1.0 + np.exp(-g)) * u).astype(np.float32)
    return x1 + np_q8_project(h, lw.wdown_q, lw.wdown_d)


def np_first_token_layer(x, lw, dims):
    """decode_layer for rows that are each the first token of their slot: a
    row's only key is its own, so attention returns its own f16-rounded v."""
    H, Hq, Hkv, D = dims.hidden, dims.n_q_heads, dims.n_kv_heads, dims.head_dim
    xn = np_rmsnorm(x, lw.attn_norm, dims.rms_eps).astype(np.float32)
    qkv = np_q8_project(xn, lw.wqkv_q, lw.wqkv_d)
    v = qkv[:, (Hq + Hkv) * D:].reshape(-1, Hkv, D).astype(np.float16).astype(np.float64)
    attn = np.repeat(v, Hq // Hkv, axis=1).reshape(-1, Hq * D).astype(np.float32)
    x1 = np.asarray(x, np.float64) + np_q8_project(attn, lw.wo_q, lw.wo_d)
    return np_ffn(x1, lw, dims.rms_eps)


def rel(a, b):
    return float(np.max(np.abs(a - b) / np.maximum(np.linalg.norm(b, axis=1, keepdims=True), 1e-300)))


def test_lm_head_matches_numpy_norm_quantize_and_dequantized_product():
    r = np.random.default_rng(11)
    H, V = 256, 300
    x = r.normal(0, 1, (3, H))
    x[1] *= 1e-3        # mean(x^2) ~ 1e-6: the eps term matters here
    x[2] *= 40.0
    gamma = r.normal(1, 0.3, H).astype(np.float32)
    wq, wd = rand_w(V, H)
    got = oracle.lm_head(x, gamma, wq, wd, 1e-6)
    want = np_q8_project(np_rmsnorm(x, gamma, 1e-6).astype(np.float32), wq, wd)
    assert got.shape == (3, V)
    assert rel(got, want) <= 1e-12
    # a different eps changes the small row's logits beyond round-off
    other = np_q8_project(np_rmsnorm(x, gamma, 1e-5).astype(np.float32), wq, wd)
    assert rel(got[1:2], other[1:2]) > 1e-3


def test_lm_head_scales_with_the_final_norm_and_vanishes_with_zero_weight_scales():
    r = np.random.default_rng(12)
    H, V = 128, 64
    x = r.normal(0, 1, (2, H))
    gamma = r.normal(1, 0.2, H).astype(np.float32)
    wq, wd = rand_w(V, H)
    base = oracle.lm_head(x, gamma, wq, wd, 1e-6)
    # a power-of-two scale of gamma passes exactly through the fp32 cast, the
    # quantizer (codes unchanged, scales doubled) and the product
    assert np.array_equal(oracle.lm_head(x, gamma * np.float32(2), wq, wd, 1e-6), 2 * base)
    # any other constant c scales the logits by c up to the quantization step
    assert rel(oracle.lm_head(x, gamma * np.float32(3), wq, wd, 1e-6), 3 * base) < 2e-2
    assert np.all(oracle.lm_head(x, gamma, wq, np.zeros_like(wd), 1e-6) == 0)


def test_layer_ffn_branch_uses_ffn_norm_on_its_own_input():
    # Wo silenced (x1 = x) with attn_norm and ffn_norm far apart: the output
    # is x plus the FFN branch normalised by ffn_norm
    lw, dims = tiny_layer(seed=21)
    lw.attn_norm[:] = np.random.default_rng(1).normal(3, 1, dims.hidden).astype(np.float32)
    lw.wo_d[:] = 0
    r = np.random.default_rng(22)
    x = r.normal(0, 1, (2, dims.hidden)).astype(np.float32)
    got = oracle.decode_layer(x, lw, dims, [make_slot(r, dims, 4), make_slot(r, dims, 0)], [1, 1])
    want = np_ffn(x.astype(np.float64), lw, dims.rms_eps)
    assert rel(got, want) <= 1e-9


def test_layer_matches_hand_composition_for_first_tokens():
    # Wo live: the FFN must normalise x1 = x + Wo . attn, not x; each row is
    # the first token of its slot, so its attention is its own value row
    lw, dims = tiny_layer(seed=23)
    lw.wo_d[:] = lw.wo_d * np.float16(32)                  # a branch of the size of x
    r = np.random.default_rng(24)
    x = r.normal(0, 1, (3, dims.hidden)).astype(np.float32)
    slots = [make_slot(r, dims, 0) for _ in range(3)]
    tr = {}
    got = oracle.decode_layer(x, lw, dims, slots, [1, 1, 1], trace=tr)
    assert rel(tr["x1"], x.astype(np.float64)) > 1e-1      # the attention branch is not negligible
    assert rel(got, np_first_token_layer(x, lw, dims)) <= 1e-9


def test_page_limits_fixture_is_consistent():
    lim = json.load(open(os.path.join(HERE, "golden", "page_limits.json")))
    assert lim["max_concurrent_slots"]["value"] * 4 == max(lim["verify_row_capacities"]["value"])
    assert lim["q8_block"]["value"] == oracle.QK
