"""Seeded, counter-based synthetic inputs (weights, scales, activations, KV).

Only inputs come from here: nothing in this module computes any step of the
decode path, so the CUDA library and the CPU oracle can both be fed from it.
The fast generator is ``synth.c`` (built into ``libsynth.so``); the ``np_*``
functions restate the same definitions in numpy for small sizes and are what
the tests pin the C generator against.

Generator: SplitMix64 (Steele, Lea & Flood, OOPSLA 2014).  Element ``i`` of a
tensor is ``mix(key + (i + 1) * gamma)`` with ``key = synth_key(seed, id)``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_SO = os.path.join(_HERE, "libsynth.so")

GAMMA = 0x9E3779B97F4A7C15
M64 = (1 << 64) - 1
SQRT3 = 1.7320508075688772


def build(force: bool = False) -> str:
    """Compile synth.c into libsynth.so next to it (gcc, OpenMP when present)."""
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= os.path.getmtime(_SRC):
        return _SO
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", _SRC, "-o", _SO]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True)
    return _SO


_lib = None


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_SO)
        u64, i64, dbl, vp = ctypes.c_uint64, ctypes.c_int64, ctypes.c_double, ctypes.c_void_p
        lib.synth_key.argtypes = [u64, u64]
        lib.synth_key.restype = u64
        lib.synth_u64.argtypes = [u64, u64, u64, i64, vp]
        lib.synth_int8.argtypes = [u64, u64, u64, i64, vp]
        lib.synth_normal_f64.argtypes = [u64, u64, u64, i64, dbl, dbl, vp]
        lib.synth_normal_f32.argtypes = [u64, u64, u64, i64, dbl, dbl, vp]
        lib.synth_normal_f16.argtypes = [u64, u64, u64, i64, dbl, dbl, vp]
        lib.synth_q8_scale_f16.argtypes = [u64, u64, u64, i64, dbl, vp]
        lib.synth_int_uniform.argtypes = [u64, u64, u64, i64, i64, i64, vp]
        _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


# ---------------------------------------------------------------- fast (C)

def u64(seed: int, tid: int, n: int, off: int = 0) -> np.ndarray:
    out = np.empty(n, np.uint64)
    _load().synth_u64(seed, tid, off, n, _ptr(out))
    return out


def int8_uniform(seed: int, tid: int, n: int, off: int = 0) -> np.ndarray:
    """int8 uniform on [-127, 127]."""
    out = np.empty(n, np.int8)
    _load().synth_int8(seed, tid, off, n, _ptr(out))
    return out


def normal_f64(seed, tid, n, mu=0.0, sigma=1.0, off=0) -> np.ndarray:
    out = np.empty(n, np.float64)
    _load().synth_normal_f64(seed, tid, off, n, mu, sigma, _ptr(out))
    return out


def normal_f32(seed, tid, n, mu=0.0, sigma=1.0, off=0) -> np.ndarray:
    out = np.empty(n, np.float32)
    _load().synth_normal_f32(seed, tid, off, n, mu, sigma, _ptr(out))
    return out


def normal_f16(seed, tid, n, mu=0.0, sigma=1.0, off=0) -> np.ndarray:
    out = np.empty(n, np.float16)
    _load().synth_normal_f16(seed, tid, off, n, mu, sigma, _ptr(out))
    return out


def q8_scale_f16(seed, tid, n, sigma=0.02, off=0) -> np.ndarray:
    """q8_0 weight scales: fp16(|N(0, sigma)| / 127)."""
    out = np.empty(n, np.float16)
    _load().synth_q8_scale_f16(seed, tid, off, n, sigma, _ptr(out))
    return out


def int_uniform(seed, tid, n, lo, hi, off=0) -> np.ndarray:
    """Integers uniform on [lo, hi] (inclusive)."""
    out = np.empty(n, np.int64)
    _load().synth_int_uniform(seed, tid, off, n, lo, hi, _ptr(out))
    return out


def permutation(seed, tid, n) -> np.ndarray:
    """A seeded permutation of range(n): stable argsort of the raw stream."""
    return np.argsort(u64(seed, tid, n), kind="stable")


# ------------------------------------------------- numpy restatement (small n)

def np_mix(z: np.ndarray) -> np.ndarray:
    z = z.astype(np.uint64)
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)
    return z ^ (z >> np.uint64(31))


def np_key(seed: int, tid: int) -> int:
    a = int(np_mix(np.array([(seed * GAMMA + 0x243F6A8885A308D3) & M64], np.uint64))[0])
    b = (tid * 0xD1B54A32D192ED03) & M64
    return int(np_mix(np.array([a ^ b], np.uint64))[0])


def np_u64(seed, tid, n, off=0) -> np.ndarray:
    key = np.uint64(np_key(seed, tid))
    i = np.arange(off + 1, off + n + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return np_mix(key + i * np.uint64(GAMMA))


def np_z(h: np.ndarray) -> np.ndarray:
    m = np.uint64(0xFFFF)
    s = ((h & m).astype(np.int64) + ((h >> np.uint64(16)) & m).astype(np.int64)
         + ((h >> np.uint64(32)) & m).astype(np.int64) + (h >> np.uint64(48)).astype(np.int64))
    return ((s - 131070).astype(np.float64) / 65536.0) * SQRT3


def np_int8_uniform(seed, tid, n, off=0):
    h = np_u64(seed, tid, n, off)
    return ((h >> np.uint64(32)) % np.uint64(255)).astype(np.int64).__sub__(127).astype(np.int8)


def np_normal_f64(seed, tid, n, mu=0.0, sigma=1.0, off=0):
    return mu + sigma * np_z(np_u64(seed, tid, n, off))


def np_q8_scale_f16(seed, tid, n, sigma=0.02, off=0):
    return (np.abs(sigma * np_z(np_u64(seed, tid, n, off))) / 127.0).astype(np.float16)
