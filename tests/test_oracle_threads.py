"""The oracle gives the same bits on any number of host threads.

Its loops over independent outputs (rows, heads, blocks) are spread over
threads; every output is still computed by one thread with the serial code,
so a run on all host cores must equal the single-threaded run bit for bit.
CPU only.
"""
import os

import numpy as np

import oracle
from test_oracle_pins import make_slot, tiny_layer, clone


def run_all(seed):
    r = np.random.default_rng(seed)
    out = {}
    x = (r.normal(0, 1, (5, 1024)) * r.uniform(0.1, 10, (5, 1))).astype(np.float32)
    q, d = oracle.quantize_act(x)
    out["q"], out["d"] = q, d
    wq = r.integers(-127, 128, size=(300, 1024)).astype(np.int8)
    wd = (np.abs(r.normal(0, 0.02, (300, 32))) / 127).astype(np.float16)
    out["dots"] = oracle.block_dots(wq, q)
    out["mv"] = oracle.matvec(wq, wd, q, d)
    out["norm"] = oracle.rmsnorm(x.astype(np.float64), r.normal(1, 0.1, 1024).astype(np.float32), 1e-6)
    out["rope"] = oracle.rope(r.normal(0, 1, (3, 6, 128)), np.array([0, 77, 32767], np.int32), 1e6)
    k = r.normal(0, 1, (2, 700, 128)).astype(np.float16)
    v = r.normal(0, 1, (2, 700, 128)).astype(np.float16)
    out["attn"] = oracle.attention_row(r.normal(0, 1, (8, 128)), k, v, 651, 2, 1 / np.sqrt(128))
    out["swiglu"] = oracle.swiglu(r.normal(0, 2, (4, 384)))
    lw, dims = tiny_layer(seed=31)
    rr = np.random.default_rng(seed + 1)
    slots = [make_slot(rr, dims, L) for L in (0, 9, 30)]
    xl = rr.normal(0, 1, (6, dims.hidden)).astype(np.float32)
    s2 = [clone(s) for s in slots]
    out["layer"] = oracle.decode_layer(xl, lw, dims, s2, [1, 2, 3])
    out["cache_k"] = np.stack([s.k for s in s2])
    return out


def test_all_host_threads_equal_one_thread_bitwise():
    assert oracle.parallel(), "the oracle should be built with OpenMP"
    prev = oracle.set_threads(1)
    try:
        one = run_all(5)
        oracle.set_threads(max(2, os.cpu_count() or 2))
        many = run_all(5)
    finally:
        oracle.set_threads(prev)
    for key in one:
        a, b = np.ascontiguousarray(one[key]), np.ascontiguousarray(many[key])
        assert a.dtype == b.dtype and a.shape == b.shape, key
        assert np.array_equal(a.view(np.uint8), b.view(np.uint8)), key
