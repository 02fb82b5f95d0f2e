"""CPU oracle of the batched q8_0 decode step (TEST INFRASTRUCTURE).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It is independent of the CUDA library:
the arithmetic lives in ``oracle.c`` (plain loops, double precision) and in
the short compositions below; nothing here loads, calls or shares code with
``invariant_sequence_decode_gb300``.

Pages followed (cited by title and section):
  * "feat(qwen4exp): exact 4-slot concurrent serving", "How it stays exact":
    a batched decode row must equal the same sequence decoded alone.
  * "#1209 Speed up concurrent generation, fix QFUSE ...", "What changed and
    why" item 2: the activation quantizer's division/rounding convention.
  * "antirez/ds4 pull 604", section 2 (dense projections run once on the
    shared batch workspace; per-sequence KV append; one multi-sequence
    attention launch) and "Commit walkthrough" (q8_0 narrow-batch matmul,
    multi-sequence decode attention, pos-vector RoPE, logits one row per
    sequence).

Readings where the pages are silent:
  q8_0 weights stored as int8 [N][K] + binary16 scales [N][K/32]; activation
  scale stored in fp32, d = amax/127, q = round-half-away(x/d) (or, in the
  half-scale form, d rounded to binary16 with overflow stored as 65504 and
  the codes taken against the stored d); RoPE pairs
  (i, i + D/2) at angle pos * theta^(-2i/D); GQA head h -> h // (Hq/Hkv);
  pre-norm layer without biases, SwiGLU with the gate rows first; row j of a
  slot with cached length ``len`` sits at position ``len + j`` and attends to
  keys ``[0, len + j]``.

Parity pins: every function here is pinned in ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass, field
from typing import List, Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_SO = os.path.join(_HERE, "liboracle.so")
QK = 32


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (gcc, no fast-math, no contraction)."""
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= os.path.getmtime(_SRC):
        return _SO
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                    "-fno-fast-math", "-fopenmp", _SRC, "-o", _SO, "-lm"], check=True)
    return _SO


_lib = None


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_SO)
        vp, i32, i64, dbl = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double
        lib.orc_half_to_double.argtypes = [ctypes.c_uint16]
        lib.orc_half_to_double.restype = dbl
        lib.orc_float_to_half.argtypes = [ctypes.c_float]
        lib.orc_float_to_half.restype = ctypes.c_uint16
        lib.orc_double_to_half.argtypes = [dbl]
        lib.orc_double_to_half.restype = ctypes.c_uint16
        lib.orc_quantize_act.argtypes = [vp, i32, i32, i64, vp, vp]
        lib.orc_quantize_act_f16.argtypes = [vp, i32, i32, i64, vp, vp]
        lib.orc_block_dots.argtypes = [vp, i32, i32, vp, i32, vp]
        lib.orc_matvec.argtypes = [vp, vp, i32, i32, vp, vp, i32, vp]
        lib.orc_rmsnorm.argtypes = [vp, i32, i32, vp, dbl, vp]
        lib.orc_rope.argtypes = [vp, i32, i32, i32, vp, dbl]
        lib.orc_attention_row.argtypes = [vp, vp, vp, i32, i32, i32, i32, i64, i64, dbl, vp]
        lib.orc_swiglu.argtypes = [vp, i32, i32, vp]
        lib.orc_argmax.argtypes = [vp, i32, i32, vp]
        lib.orc_set_threads.argtypes = [i32]
        lib.orc_set_threads.restype = i32
        lib.orc_parallel.restype = i32
        _lib = lib
    return _lib


def set_threads(n: int) -> int:
    """Host threads the oracle's loops use (1 by default); returns the previous
    count.  Results do not depend on it: each output is computed by one thread
    with the same serial code."""
    return int(_load().orc_set_threads(int(n)))


def parallel() -> bool:
    """Whether the oracle library was built with OpenMP."""
    return bool(_load().orc_parallel())


def _c(a: np.ndarray, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


def _p(a: np.ndarray) -> int:
    return a.ctypes.data


# ------------------------------------------------------------ primitives

def half_bits(a) -> np.ndarray:
    """binary16 payload as uint16 (accepts float16 arrays or uint16 bits)."""
    a = np.asarray(a)
    if a.dtype == np.float16:
        return np.ascontiguousarray(a).view(np.uint16)
    return _c(a, np.uint16)


def half_to_double(bits) -> np.ndarray:
    lib = _load()
    b = half_bits(bits).ravel()
    return np.array([lib.orc_half_to_double(int(v)) for v in b], np.float64)


def float_to_half_bits(x) -> np.ndarray:
    lib = _load()
    x = _c(x, np.float32).ravel()
    return np.array([lib.orc_float_to_half(float(v)) for v in x], np.uint16)


def quantize_act(x: np.ndarray):
    """fp32 [T][K] -> (int8 [T][K], fp32 scales [T][K/32])."""
    x = _c(x, np.float32)
    if x.ndim == 1:
        x = x[None]
    T, K = x.shape
    assert K % QK == 0
    q = np.empty((T, K), np.int8)
    d = np.empty((T, K // QK), np.float32)
    _load().orc_quantize_act(_p(x), T, K, K, _p(q), _p(d))
    return q, d


def quantize_act_f16(x: np.ndarray):
    """The half-scale form: fp32 [T][K] -> (int8 [T][K], binary16 bits [T][K/32] as uint16)."""
    x = _c(x, np.float32)
    if x.ndim == 1:
        x = x[None]
    T, K = x.shape
    assert K % QK == 0
    q = np.empty((T, K), np.int8)
    d = np.empty((T, K // QK), np.uint16)
    _load().orc_quantize_act_f16(_p(x), T, K, K, _p(q), _p(d))
    return q, d


def block_dots(wq: np.ndarray, aq: np.ndarray) -> np.ndarray:
    """int32 [T][N][K/32] per-block integer dots."""
    wq = _c(wq, np.int8)
    aq = _c(aq, np.int8)
    N, K = wq.shape
    T = aq.shape[0]
    out = np.empty((T, N, K // QK), np.int32)
    _load().orc_block_dots(_p(wq), N, K, _p(aq), T, _p(out))
    return out


def matvec(wq, wd, aq, ad) -> np.ndarray:
    """q8_0 weights x q8_0 activations -> float64 [T][N]."""
    wq = _c(wq, np.int8)
    wd = half_bits(wd)
    aq = _c(aq, np.int8)
    ad = _c(ad, np.float32)
    N, K = wq.shape
    T = aq.shape[0]
    assert wd.shape == (N, K // QK) and aq.shape == (T, K) and ad.shape == (T, K // QK)
    y = np.empty((T, N), np.float64)
    _load().orc_matvec(_p(wq), _p(wd), N, K, _p(aq), _p(ad), T, _p(y))
    return y


def rmsnorm(x, gamma, eps) -> np.ndarray:
    x = _c(x, np.float64)
    if x.ndim == 1:
        x = x[None]
    T, H = x.shape
    g = _c(gamma, np.float32)
    y = np.empty_like(x)
    _load().orc_rmsnorm(_p(x), T, H, _p(g), float(eps), _p(y))
    return y


def rope(x, pos, theta) -> np.ndarray:
    """x [T][n_heads][D] (any float dtype) -> rotated float64 copy."""
    x = np.array(x, dtype=np.float64, copy=True, order="C")
    T, nh, D = x.shape
    p = _c(pos, np.int32)
    assert p.shape == (T,)
    _load().orc_rope(_p(x), T, nh, D, _p(p), float(theta))
    return x


def attention_row(q, k, v, L, Hkv, scale) -> np.ndarray:
    """One query row.  q [Hq][D]; k, v binary16 [Hkv][cap][D] (first L keys)."""
    q = _c(q, np.float64)
    Hq, D = q.shape
    k = half_bits(k)
    v = half_bits(v)
    assert k.shape == v.shape and k.shape[0] == Hkv and k.shape[2] == D and L <= k.shape[1]
    out = np.empty((Hq, D), np.float64)
    _load().orc_attention_row(_p(q), _p(k), _p(v), int(L), Hq, Hkv, D,
                              k.shape[1] * D, D, float(scale), _p(out))
    return out


def swiglu(gu) -> np.ndarray:
    gu = _c(gu, np.float64)
    T, F2 = gu.shape
    F = F2 // 2
    h = np.empty((T, F), np.float64)
    _load().orc_swiglu(_p(gu), T, F, _p(h))
    return h


def argmax(x) -> np.ndarray:
    x = _c(x, np.float32)
    T, V = x.shape
    out = np.empty(T, np.int32)
    _load().orc_argmax(_p(x), T, V, _p(out))
    return out


# ------------------------------------------------------------ composition

@dataclass
class LayerWeights:
    """One pre-norm decoder layer; every projection is q8_0 (int8 + fp16 scales)."""
    attn_norm: np.ndarray          # fp32 [H]
    wqkv_q: np.ndarray             # int8 [(Hq + 2 Hkv) D][H]
    wqkv_d: np.ndarray             # f16  [(Hq + 2 Hkv) D][H/32]
    wo_q: np.ndarray               # int8 [H][Hq D]
    wo_d: np.ndarray
    ffn_norm: np.ndarray           # fp32 [H]
    wgu_q: np.ndarray              # int8 [2F][H], gate rows first
    wgu_d: np.ndarray
    wdown_q: np.ndarray            # int8 [H][F]
    wdown_d: np.ndarray


@dataclass
class Dims:
    hidden: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    ffn: int
    rms_eps: float = 1e-6
    rope_theta: float = 1e6


@dataclass
class Slot:
    """A sequence's cache for one layer: binary16 bits (uint16) [Hkv][cap][D] K and V, ``len`` keys
    already cached.  ``decode_layer`` writes this step's rows at len..len+n-1."""
    k: np.ndarray
    v: np.ndarray
    len: int


def row_positions(lens: Sequence[int], rows_per_slot: Sequence[int]) -> np.ndarray:
    """Row j of slot s sits at position lens[s] + j; rows are grouped by slot."""
    return np.array([lens[s] + j for s in range(len(lens)) for j in range(rows_per_slot[s])], np.int32)


def decode_layer(x, w: LayerWeights, dims: Dims, slots: List[Slot], rows_per_slot: Sequence[int],
                 trace: Optional[dict] = None) -> np.ndarray:
    """One decode step of one layer over the batch; returns x_out (float64 [T][H]).

    The dense projections see all T rows at once [ds4 pull 604, section 2], but
    every row's arithmetic is its own: nothing here mixes rows, which is the
    batch-invariance contract ["exact 4-slot concurrent serving", "How it
    stays exact"].  Slot caches are updated in place (f16 K/V rows appended).
    """
    H, Hq, Hkv, D, F = dims.hidden, dims.n_q_heads, dims.n_kv_heads, dims.head_dim, dims.ffn
    x = np.asarray(x, np.float64)
    T = x.shape[0]
    assert T == sum(rows_per_slot) and len(slots) == len(rows_per_slot)
    pos = row_positions([s.len for s in slots], rows_per_slot)

    xn = rmsnorm(x, w.attn_norm, dims.rms_eps).astype(np.float32)
    aq, ad = quantize_act(xn)
    qkv = matvec(w.wqkv_q, w.wqkv_d, aq, ad)
    q = rope(qkv[:, :Hq * D].reshape(T, Hq, D), pos, dims.rope_theta)
    k = rope(qkv[:, Hq * D:(Hq + Hkv) * D].reshape(T, Hkv, D), pos, dims.rope_theta)
    v = qkv[:, (Hq + Hkv) * D:].reshape(T, Hkv, D)

    attn = np.empty((T, Hq, D), np.float64)
    r = 0
    scale = 1.0 / np.sqrt(D)
    for s, n in zip(slots, rows_per_slot):
        for j in range(n):
            p = s.len + j
            assert p < s.k.shape[1], "cache capacity exceeded"
            s.k[:, p, :] = k[r + j].astype(np.float16).view(np.uint16)
            s.v[:, p, :] = v[r + j].astype(np.float16).view(np.uint16)
        for j in range(n):
            attn[r + j] = attention_row(q[r + j], s.k, s.v, s.len + j + 1, Hkv, scale)
        r += n

    a32 = attn.reshape(T, Hq * D).astype(np.float32)
    oq, od = quantize_act(a32)
    x1 = x + matvec(w.wo_q, w.wo_d, oq, od)

    xn2 = rmsnorm(x1, w.ffn_norm, dims.rms_eps).astype(np.float32)
    fq, fd = quantize_act(xn2)
    gu = matvec(w.wgu_q, w.wgu_d, fq, fd)
    h = swiglu(gu).astype(np.float32)
    hq, hd = quantize_act(h)
    x2 = x1 + matvec(w.wdown_q, w.wdown_d, hq, hd)
    if trace is not None:
        trace.update(xn=xn, qkv=qkv, q=q, k=k, v=v, attn=attn, x1=x1, xn2=xn2, gu=gu, h=h, x2=x2)
    return x2


def lm_head(x, final_norm, head_q, head_d, eps) -> np.ndarray:
    """Final RMSNorm, q8_0 activation quantization and the q8_0 output head:
    one logits row per batch row [ds4 pull 604, Commit walkthrough]."""
    xn = rmsnorm(x, final_norm, eps).astype(np.float32)
    aq, ad = quantize_act(xn)
    return matvec(head_q, head_d, aq, ad)
