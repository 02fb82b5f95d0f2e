"""Seeded synthetic workloads for the decode step (inputs only, host numpy).

Every tensor comes from ``synth`` under a (seed, tensor id) pair, so the CUDA
path and the CPU oracle see identical bits.  Shapes and value distributions:

  weights   int8 uniform on [-127, 127]; fp16 scale |N(0, 0.02)| / 127
  acts      fp32 N(0, 1)                   K/V   fp16 N(0, 1)
  norms     fp32 N(1, 0.1)                 (N(mu, s) is the 4-term Irwin-Hall
                                            approximation described in synth)

Named workloads:
  TINY      1024x1024 q8_0 matvec at n_tok 1..4; decode attention for 4
            sequences, 8 query / 2 KV heads, head_dim 128, contexts
            {17, 100, 513, 1000}, RoPE theta 1e6 at position len-1.
  LAYER27B  one dense decoder layer: hidden 5120, 40 query / 8 KV heads,
            head_dim 128, SwiGLU FFN 17408, n_seq 1..4, 2,051 keys per slot.
  SWEEP     matvec n_tok 1..4 x K {2048, 4096, 5120, 8192} x N {4096, 8192,
            17408, 32768}; RoPE positions uniform on [0, 32767].
  LONGCTX   4 sequences, contexts uniform on [16384, 32768], 32 query / 8 KV
            heads, one query row each.
  VERIFY    4 slots x 2/3/4 rows through 64 LAYER27B layers plus a
            151,936 x 5120 q8_0 head, cache lengths uniform on [1024, 2051].
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import List

import numpy as np

from . import synth

# tensor ids: (kind << 20) | (layer << 4) | sub
W_QKV, W_O, W_GU, W_DOWN, W_HEAD, W_MAT = 1, 2, 3, 4, 5, 6
N_ATTN, N_FFN, N_FINAL = 7, 8, 9
ACT, KCACHE, VCACHE, QVEC, LENS, POS, PERM = 10, 11, 12, 13, 14, 15, 16


def tid(kind: int, layer: int = 0, sub: int = 0) -> int:
    return (kind << 20) | (layer << 4) | sub


def q8_weights(seed: int, t: int, N: int, K: int):
    """(int8 [N][K], fp16 [N][K/32]) q8_0 weights."""
    wq = synth.int8_uniform(seed, t, N * K).reshape(N, K)
    wd = synth.q8_scale_f16(seed, t | 0x8, N * (K // 32), 0.02).reshape(N, K // 32)
    return wq, wd


def acts(seed: int, T: int, K: int, sub: int = 0) -> np.ndarray:
    return synth.normal_f32(seed, tid(ACT, 0, sub), T * K).reshape(T, K)


@dataclass
class Dims:
    hidden: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    ffn: int
    rms_eps: float = 1e-6
    rope_theta: float = 1e6


LAYER27B = Dims(5120, 40, 8, 128, 17408)
TINY_LAYER = Dims(256, 4, 2, 128, 512)
VOCAB = 151936


@dataclass
class LayerHost:
    attn_norm: np.ndarray
    wqkv_q: np.ndarray
    wqkv_d: np.ndarray
    wo_q: np.ndarray
    wo_d: np.ndarray
    ffn_norm: np.ndarray
    wgu_q: np.ndarray
    wgu_d: np.ndarray
    wdown_q: np.ndarray
    wdown_d: np.ndarray


def layer_host(seed: int, layer: int, d: Dims) -> LayerHost:
    H, Hq, Hkv, D, F = d.hidden, d.n_q_heads, d.n_kv_heads, d.head_dim, d.ffn
    return LayerHost(
        synth.normal_f32(seed, tid(N_ATTN, layer), H, 1.0, 0.1),
        *q8_weights(seed, tid(W_QKV, layer), (Hq + 2 * Hkv) * D, H),
        *q8_weights(seed, tid(W_O, layer), H, Hq * D),
        synth.normal_f32(seed, tid(N_FFN, layer), H, 1.0, 0.1),
        *q8_weights(seed, tid(W_GU, layer), 2 * F, H),
        *q8_weights(seed, tid(W_DOWN, layer), H, F),
    )


def head_host(seed: int, d: Dims, vocab: int):
    wq, wd = q8_weights(seed, tid(W_HEAD), vocab, d.hidden)
    return synth.normal_f32(seed, tid(N_FINAL), d.hidden, 1.0, 0.1), wq, wd


def cache_host(seed: int, slot: int, layer: int, d: Dims, cap: int, length: int):
    """fp16 K, V [Hkv][cap][D]; positions >= length hold N(0,1) filler too (never read)."""
    n = d.n_kv_heads * cap * d.head_dim
    k = synth.normal_f16(seed, tid(KCACHE, layer, slot), n).reshape(d.n_kv_heads, cap, d.head_dim)
    v = synth.normal_f16(seed, tid(VCACHE, layer, slot), n).reshape(d.n_kv_heads, cap, d.head_dim)
    return k, v


TINY_ATTN_LENS = [17, 100, 513, 1000]


def lens(seed: int, n: int, lo: int, hi: int, sub: int = 0) -> List[int]:
    return [int(v) for v in synth.int_uniform(seed, tid(LENS, 0, sub), n, lo, hi)]


def positions(seed: int, n: int, lo: int = 0, hi: int = 32767, sub: int = 0) -> np.ndarray:
    return synth.int_uniform(seed, tid(POS, 0, sub), n, lo, hi).astype(np.int32)


def qvec(seed: int, T: int, Hq: int, D: int = 128, sub: int = 0) -> np.ndarray:
    return synth.normal_f32(seed, tid(QVEC, 0, sub), T * Hq * D).reshape(T, Hq, D)
