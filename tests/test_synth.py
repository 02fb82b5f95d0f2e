"""The C input generator against its numpy restatement and plain-Python SplitMix64."""
import numpy as np

from invariant_sequence_decode_gb300 import synth

M64 = (1 << 64) - 1


def py_mix(z):
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & M64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & M64
    return z ^ (z >> 31)


def test_splitmix_stream_matches_plain_python():
    seed, tid, n = 7, 3, 50
    key = py_mix(py_mix((seed * synth.GAMMA + 0x243F6A8885A308D3) & M64) ^ ((tid * 0xD1B54A32D192ED03) & M64))
    ref = [py_mix((key + (i + 1) * synth.GAMMA) & M64) for i in range(n)]
    assert synth.u64(seed, tid, n).tolist() == ref
    assert synth.np_u64(seed, tid, n).tolist() == ref


def test_c_generators_match_numpy_restatement_bitwise():
    for seed, tid in [(0, 1), (1, 99), (4, 2 ** 20 + 5)]:
        n = 20000
        assert np.array_equal(synth.int8_uniform(seed, tid, n), synth.np_int8_uniform(seed, tid, n))
        a = synth.normal_f64(seed, tid, n, 1.0, 0.1)
        assert np.array_equal(a, synth.np_normal_f64(seed, tid, n, 1.0, 0.1))
        assert np.array_equal(synth.normal_f32(seed, tid, n), synth.np_normal_f64(seed, tid, n).astype(np.float32))
        assert np.array_equal(synth.normal_f16(seed, tid, n).view(np.uint16),
                              synth.np_normal_f64(seed, tid, n).astype(np.float16).view(np.uint16))
        assert np.array_equal(synth.q8_scale_f16(seed, tid, n).view(np.uint16),
                              synth.np_q8_scale_f16(seed, tid, n).view(np.uint16))


def test_offsets_are_counter_based():
    full = synth.int8_uniform(3, 4, 1000)
    assert np.array_equal(synth.int8_uniform(3, 4, 300, off=700), full[700:])


def test_distributions_have_the_requested_shape():
    w = synth.int8_uniform(0, 0, 1 << 20)
    assert w.min() == -127 and w.max() == 127 and abs(w.mean()) < 0.5
    z = synth.normal_f64(0, 1, 1 << 20)
    assert abs(z.mean()) < 5e-3 and abs(z.std() - 1) < 5e-3 and np.max(np.abs(z)) <= 2 * np.sqrt(3) + 1e-12
    s = synth.q8_scale_f16(0, 2, 1 << 16).astype(np.float64)
    assert s.min() >= 0 and abs(s.mean() - 0.02 * np.sqrt(2 / np.pi) / 127) < 2e-6
    u = synth.int_uniform(0, 3, 10000, 16384, 32768)
    assert u.min() >= 16384 and u.max() <= 32768
    p = synth.permutation(0, 4, 100)
    assert sorted(p.tolist()) == list(range(100))
