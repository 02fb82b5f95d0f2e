"""The half-scale q8_0 activations and the fused producers that emit them.

"#1209 Speed up concurrent generation, fix QFUSE ...", What changed and why,
item 2: a fused quantizer must match the consuming quantizer's finite-half
guards and division/rounding convention; Validation: the isolated
quantization fix restored 150/150 full-vocabulary positions byte for byte.
Here:
  * the standalone half-scale quantizer equals the oracle's, bit for bit, on
    random rows and on the edges (ties, binary16 overflow, subnormal and
    underflowing scales, NaN, infinity);
  * the fused producers (RMSNorm -> q8_0, SwiGLU -> q8_0), in both scale
    forms, equal a standalone quantization of their own fp32 output byte for
    byte over 1,024+ blocks whose magnitudes are steered across the edges;
  * half-scale activations feed the matvec unchanged (float(d) is exact).
"""
import numpy as np
import pytest

import oracle
from invariant_sequence_decode_gb300 import workloads as wl

torch = pytest.importorskip("torch")
import invariant_sequence_decode_gb300 as luce  # noqa: E402

pytestmark = pytest.mark.gpu


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


def edge_rows(K):
    rows = np.zeros((8, K), np.float32)
    ties = np.array([127.0, -126.5, 126.5, 63.5, -63.5, 2.5, -2.5, 0.5, -0.5, 1.5] + [0.25] * 22, np.float32)
    rows[0, :32] = ties                                         # scale 1: exact ties
    rows[1, :32] = np.float32(127.0 * 65520.0)                  # scale overflows binary16
    rows[1, 32:64] = np.float32(127.0 * 65504.0)                # largest finite scale
    rows[2, :32] = np.float32(127.0 * 2.0 ** -20) * np.linspace(-1, 1, 32, dtype=np.float32)  # subnormal scale
    rows[2, 32:64] = np.float32(127.0 * 2.0 ** -26)             # scale underflows to zero
    rows[3, :32] = np.linspace(-1, 1, 32, dtype=np.float32)
    rows[3, 5] = np.nan                                         # NaN entry
    rows[3, 32:64] = 1.0
    rows[3, 40] = np.inf                                        # infinite entry
    rows[4] = wl.acts(7, 1, K)[0] * np.float32(1e6)
    rows[5] = wl.acts(8, 1, K)[0] * np.float32(1e-6)
    rows[6] = wl.acts(9, 1, K)[0]
    rows[7] = wl.acts(10, 1, K)[0] * np.float32(3e-3)
    return rows


@pytest.mark.parametrize("K", [64, 1024, 5120])
def test_half_scale_quantizer_equals_the_oracle(K):
    x = np.concatenate([wl.acts(3, 4, K) * np.float32(5.0), edge_rows(K)])
    q, d = luce.luce_q8_quantize_act_f16(cuda(x))
    qo, do = oracle.quantize_act_f16(x)
    assert np.array_equal(host(q), qo)
    assert np.array_equal(host(d).view(np.uint16), do)
    assert np.all(np.isfinite(host(d)))


def steering_gamma(H, seed):
    """Per-block magnitudes from 1e-12 to 1e9 (scales that underflow,
    subnormal, normal, and overflow binary16) plus plain N(1, 0.1) blocks."""
    g = wl.acts(seed, 1, H)[0] * np.float32(0.1) + np.float32(1.0)
    mags = np.array([1e-12, 1e-9, 3e-7, 1e-5, 1e-3, 1.0, 10.0, 1e3, 1e5, 1e7, 1e8, 1e9], np.float32)
    for b in range(H // 32):
        if b % 3:
            g[32 * b:32 * b + 32] *= mags[b % len(mags)]
    return g


@pytest.mark.parametrize("half", [False, True])
def test_fused_rmsnorm_codes_equal_the_standalone_quantizer(half):
    T, H = 16, 2048                                           # 1,024 blocks
    x = wl.acts(11, T, H) * np.float32(2.0)
    x[3] *= np.float32(1e-20)                                 # a row where eps dominates
    gamma = steering_gamma(H, 12)
    xn, q, d = luce.luce_rmsnorm_q8(cuda(x), cuda(gamma), 1e-6, half_scale=half)
    xn_h = host(xn)
    qs, ds = (luce.luce_q8_quantize_act_f16 if half else luce.luce_q8_quantize_act)(xn)
    assert np.array_equal(host(q), host(qs))
    assert np.array_equal(bits(host(d)), bits(host(ds)))
    # and the codes are the oracle's quantization of the fused output
    qo, do = (oracle.quantize_act_f16 if half else oracle.quantize_act)(xn_h)
    assert np.array_equal(host(q), qo)
    assert np.array_equal(bits(host(d)), bits(do))
    if half:
        assert np.any(host(d).view(np.uint16) == 0x7BFF) and np.any(host(d).view(np.uint16) == 0)
        assert np.any((host(d).view(np.uint16) > 0) & (host(d).view(np.uint16) < 0x0400))  # subnormal scales


@pytest.mark.parametrize("half", [False, True])
def test_fused_swiglu_codes_equal_the_standalone_quantizer(half):
    T, F = 16, 2048
    gu = wl.acts(13, T, 2 * F) * np.float32(3.0)
    gu[:, F:] *= steering_gamma(F, 14)[None, :]               # the up half steers the magnitudes
    h, q, d = luce.luce_swiglu_q8(cuda(gu), half_scale=half)
    qs, ds = (luce.luce_q8_quantize_act_f16 if half else luce.luce_q8_quantize_act)(h)
    assert np.array_equal(host(q), host(qs))
    assert np.array_equal(bits(host(d)), bits(host(ds)))
    qo, do = (oracle.quantize_act_f16 if half else oracle.quantize_act)(host(h))
    assert np.array_equal(host(q), qo) and np.array_equal(bits(host(d)), bits(do))
    assert np.all(np.abs(host(h).astype(np.float64) - oracle.swiglu(gu.astype(np.float64))) <=
                  1e-5 * np.abs(oracle.swiglu(gu.astype(np.float64))) + 1e-30)


def test_half_scale_activations_feed_the_matvec():
    N, K, T = 300, 1024, 6
    wq, wd = wl.q8_weights(15, wl.tid(wl.W_MAT, 3), N, K)
    x = wl.acts(16, T, K)
    q, d = luce.luce_q8_quantize_act_f16(cuda(x))
    y = host(luce.luce_q8_matvec_batch(cuda(wq), cuda(wd), q, d.float()))
    ref = oracle.matvec(wq, wd, host(q), host(d).astype(np.float32))
    err = np.max(np.abs(y - ref), axis=1) / np.linalg.norm(ref, axis=1)
    assert np.all(err <= 1e-5)
