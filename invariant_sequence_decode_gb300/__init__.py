"""Batch-invariant concurrent decode step for GB300 (sm_103a).

Thin Python binding over ``libluce.so`` (the C ABI declared in
``include/luce.h``).  Functions take torch CUDA tensors, check dtypes and
layouts, and pass raw pointers and the current CUDA stream to the library:
argument marshalling only, every step of the path runs in the library's CUDA
kernels.  There is no fallback: a missing library raises.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import List, Optional, Sequence

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libluce.so")

QK = 32
MAX_SEQ = 4
MAX_ROWS_PER_SEQ = 4
MAX_ROWS = 16
HEAD_DIM = 128
MAX_KEYS = 130816

LUCE_OK, LUCE_EINVAL, LUCE_EUNSUPPORTED, LUCE_ECUDA, LUCE_ENOSPACE = 0, -1, -2, -3, -4


class LuceError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"luce status {status}: {msg}")
        self.status = status


# ------------------------------------------------------------ ctypes mirror of luce.h

class SeqViewC(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("len", ctypes.c_int32),
                ("n_q", ctypes.c_int32), ("row0", ctypes.c_int32), ("cap", ctypes.c_int32),
                ("head_stride", ctypes.c_int64), ("tok_stride", ctypes.c_int64)]


class LayerC(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "attn_norm", "wqkv_q", "wqkv_d", "wo_q", "wo_d", "ffn_norm", "wgu_q", "wgu_d", "wdown_q", "wdown_d")]


class ModelC(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int32), ("hidden", ctypes.c_int32), ("n_q_heads", ctypes.c_int32),
                ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("ffn", ctypes.c_int32),
                ("vocab", ctypes.c_int32), ("rms_eps", ctypes.c_float), ("rope_theta", ctypes.c_double),
                ("layers", ctypes.POINTER(LayerC)), ("final_norm", ctypes.c_void_p),
                ("head_q", ctypes.c_void_p), ("head_d", ctypes.c_void_p)]


class SlotC(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("len", ctypes.c_int32), ("cap", ctypes.c_int32)]


class PagedViewC(ctypes.Structure):
    _fields_ = [("k_pool", ctypes.c_void_p), ("v_pool", ctypes.c_void_p), ("table", ctypes.c_void_p),
                ("len", ctypes.c_int32), ("n_q", ctypes.c_int32), ("row0", ctypes.c_int32)]


class PagedSlotC(ctypes.Structure):
    _fields_ = [("k_pool", ctypes.c_void_p), ("v_pool", ctypes.c_void_p), ("table", ctypes.c_void_p),
                ("table_host", ctypes.POINTER(ctypes.c_int32)), ("n_table", ctypes.c_int32),
                ("n_pages", ctypes.c_int32), ("len", ctypes.c_int32)]


_LAYOUT_FIELDS = ("xn", "xn_q", "xn_d", "qkv", "q_rot", "part", "attn", "attn_q", "attn_d", "x1",
                  "xn2", "xn2_q", "xn2_d", "gu", "h", "h_q", "h_d", "xf", "xf_q", "xf_d", "total")


class StepLayoutC(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in _LAYOUT_FIELDS]


EXPORTS = ("luce_last_error", "luce_version", "luce_launch_count", "luce_q8_quantize_act", "luce_q8_matvec_batch",
           "luce_q8_block_dots", "luce_rope_posvec", "luce_kv_append", "luce_decode_attn_multiseq",
           "luce_decode_attn_workspace_size", "luce_decode_step_layout", "luce_decode_step",
           "luce_decode_attn_multiseq_noalloc", "luce_decode_attn_noalloc_max_bytes", "luce_decode_attn_paged",
           "luce_decode_step_paged", "luce_wait_timeouts", "luce_decode_step_host",
           "luce_test_wait_expiry", "luce_q8_matvec_batch_path", "luce_q8_quantize_act_f16", "luce_rmsnorm_q8",
           "luce_swiglu_q8", "luce_step_graph_create", "luce_step_graph_run", "luce_step_graph_stats",
           "luce_step_graph_destroy")

_lib = None


def load_library(path: str = LIB_PATH):
    """Load libluce.so (built by ``invariant_sequence_decode_gb300.build``).  Raises if missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is not built; run `python -m invariant_sequence_decode_gb300.build`")
    lib = ctypes.CDLL(path)
    vp, i32, i64, sz, f32, f64 = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t,
                                  ctypes.c_float, ctypes.c_double)
    lib.luce_last_error.restype = ctypes.c_char_p
    lib.luce_last_error.argtypes = []
    lib.luce_version.restype = i32
    lib.luce_launch_count.restype = ctypes.c_uint64
    lib.luce_launch_count.argtypes = []
    lib.luce_q8_quantize_act.argtypes = [vp, i32, i32, i64, vp, vp, vp]
    lib.luce_q8_quantize_act_f16.argtypes = [vp, i32, i32, i64, vp, vp, vp]
    lib.luce_rmsnorm_q8.argtypes = [vp, i32, i32, vp, f32, vp, vp, vp, i32, vp]
    lib.luce_swiglu_q8.argtypes = [vp, i32, i32, vp, vp, vp, i32, vp]
    lib.luce_q8_matvec_batch.argtypes = [vp, vp, i32, i32, vp, vp, i32, vp, i64, vp]
    lib.luce_q8_matvec_batch_path.argtypes = [vp, vp, i32, i32, vp, vp, i32, vp, i64, i32, vp]
    lib.luce_q8_block_dots.argtypes = [vp, i32, i32, vp, i32, vp, vp]
    lib.luce_rope_posvec.argtypes = [vp, i32, i32, i32, i64, vp, f64, vp]
    lib.luce_kv_append.argtypes = [vp, vp, i64, i32, i32, ctypes.POINTER(SeqViewC), i32, vp]
    lib.luce_decode_attn_multiseq.argtypes = [vp, ctypes.POINTER(SeqViewC), i32, i32, i32, i32, f32, vp, vp, sz, vp]
    lib.luce_decode_attn_workspace_size.argtypes = [i32, i32, i32, i32]
    lib.luce_decode_attn_workspace_size.restype = sz
    lib.luce_decode_step_layout.argtypes = [ctypes.POINTER(ModelC), i32, i32, ctypes.POINTER(StepLayoutC)]
    lib.luce_decode_step.argtypes = [ctypes.POINTER(ModelC), ctypes.POINTER(SlotC), ctypes.POINTER(ctypes.c_int32),
                                     i32, vp, vp, vp, vp, sz, vp]
    lib.luce_decode_attn_multiseq_noalloc.argtypes = [vp, ctypes.POINTER(SeqViewC), i32, i32, i32, i32, f32, vp, vp]
    lib.luce_decode_attn_noalloc_max_bytes.argtypes = []
    lib.luce_decode_attn_paged.argtypes = [vp, ctypes.POINTER(PagedViewC), i32, i32, i32, i32, f32, vp, vp, sz, vp]
    lib.luce_decode_step_paged.argtypes = [ctypes.POINTER(ModelC), ctypes.POINTER(PagedSlotC),
                                           ctypes.POINTER(ctypes.c_int32), i32, vp, vp, vp, vp, sz, vp]
    lib.luce_decode_attn_noalloc_max_bytes.restype = sz
    lib.luce_wait_timeouts.argtypes = [ctypes.POINTER(ctypes.c_uint32), i32]
    lib.luce_test_wait_expiry.argtypes = [i64, vp]
    lib.luce_decode_step_host.argtypes = [ctypes.POINTER(ModelC), ctypes.POINTER(SlotC), ctypes.POINTER(ctypes.c_int32),
                                          i32, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.luce_step_graph_create.argtypes = [ctypes.POINTER(ModelC), ctypes.POINTER(SlotC),
                                           ctypes.POINTER(ctypes.c_int32), i32, vp, vp, vp, vp, vp, vp, vp, sz,
                                           ctypes.POINTER(vp)]
    lib.luce_step_graph_run.argtypes = [vp, ctypes.POINTER(ctypes.c_int32), vp]
    lib.luce_step_graph_stats.argtypes = [vp, ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_int64),
                                          ctypes.POINTER(ctypes.c_int32)]
    lib.luce_step_graph_destroy.argtypes = [vp]
    for name in EXPORTS:
        if name not in ("luce_last_error", "luce_version", "luce_launch_count", "luce_decode_attn_workspace_size",
                        "luce_decode_attn_noalloc_max_bytes"):
            getattr(lib, name).restype = i32
    _lib = lib
    return lib


def launch_count() -> int:
    """Kernel launches the library has enqueued so far (all threads)."""
    return int(load_library().luce_launch_count())


def wait_timeouts(reset: bool = False) -> int:
    """Bounded device waits that expired on the current device (0 on a healthy run)."""
    n = ctypes.c_uint32(0)
    _check(load_library().luce_wait_timeouts(ctypes.byref(n), 1 if reset else 0))
    return int(n.value)


def _check(rc: int):
    if rc != LUCE_OK:
        raise LuceError(rc, load_library().luce_last_error().decode())


def _stream(stream=None) -> int:
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _need(t, dtype, name):
    import torch
    if not isinstance(t, torch.Tensor) or t.dtype != dtype or not t.is_cuda:
        raise TypeError(f"{name}: expected a CUDA {dtype} tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")


# ------------------------------------------------------------ kernels

def luce_q8_quantize_act(x, q=None, d=None, stream=None):
    """fp32 [T][K] -> (int8 [T][K], fp32 [T][K/32]) q8_0 activation blocks."""
    import torch
    _need(x, torch.float32, "x")
    T, K = x.shape
    q = torch.empty((T, K), dtype=torch.int8, device=x.device) if q is None else q
    d = torch.empty((T, K // QK), dtype=torch.float32, device=x.device) if d is None else d
    _check(load_library().luce_q8_quantize_act(x.data_ptr(), T, K, K, q.data_ptr(), d.data_ptr(), _stream(stream)))
    return q, d


def luce_q8_quantize_act_f16(x, q=None, d=None, stream=None):
    """fp32 [T][K] -> (int8 [T][K], binary16 scales as float16 [T][K/32]): the half-scale form."""
    import torch
    _need(x, torch.float32, "x")
    T, K = x.shape
    q = torch.empty((T, K), dtype=torch.int8, device=x.device) if q is None else q
    d = torch.empty((T, K // QK), dtype=torch.float16, device=x.device) if d is None else d
    _check(load_library().luce_q8_quantize_act_f16(x.data_ptr(), T, K, K, q.data_ptr(), d.data_ptr(),
                                                   _stream(stream)))
    return q, d


def luce_rmsnorm_q8(x, gamma, eps: float, half_scale: bool = False, stream=None):
    """RMSNorm of fp32 rows [T][H] and its q8_0 blocks: (xn fp32, q int8, d fp32 or float16)."""
    import torch
    _need(x, torch.float32, "x")
    _need(gamma, torch.float32, "gamma")
    T, H = x.shape
    xn = torch.empty_like(x)
    q = torch.empty((T, H), dtype=torch.int8, device=x.device)
    d = torch.empty((T, H // QK), dtype=torch.float16 if half_scale else torch.float32, device=x.device)
    _check(load_library().luce_rmsnorm_q8(x.data_ptr(), T, H, gamma.data_ptr(), float(eps), xn.data_ptr(),
                                          q.data_ptr(), d.data_ptr(), 1 if half_scale else 0, _stream(stream)))
    return xn, q, d


def luce_swiglu_q8(gu, half_scale: bool = False, stream=None):
    """SwiGLU of gate||up rows [T][2F] and its q8_0 blocks: (h fp32, q int8, d fp32 or float16)."""
    import torch
    _need(gu, torch.float32, "gu")
    T, F2 = gu.shape
    F = F2 // 2
    h = torch.empty((T, F), dtype=torch.float32, device=gu.device)
    q = torch.empty((T, F), dtype=torch.int8, device=gu.device)
    d = torch.empty((T, F // QK), dtype=torch.float16 if half_scale else torch.float32, device=gu.device)
    _check(load_library().luce_swiglu_q8(gu.data_ptr(), T, F, h.data_ptr(), q.data_ptr(), d.data_ptr(),
                                         1 if half_scale else 0, _stream(stream)))
    return h, q, d


def luce_q8_matvec_batch(wq, wd, aq, ad, y=None, stream=None):
    """q8_0 weights (int8 [N][K], fp16 [N][K/32]) x q8_0 activations -> fp32 [T][N]."""
    import torch
    _need(wq, torch.int8, "wq")
    _need(aq, torch.int8, "aq")
    _need(ad, torch.float32, "ad")
    if wd.dtype not in (torch.float16, torch.int16, torch.uint16):
        raise TypeError("wd: expected fp16 scales")
    N, K = wq.shape
    T = aq.shape[0]
    y = torch.empty((T, N), dtype=torch.float32, device=wq.device) if y is None else y
    _check(load_library().luce_q8_matvec_batch(wq.data_ptr(), wd.data_ptr(), N, K, aq.data_ptr(), ad.data_ptr(),
                                               T, y.data_ptr(), y.stride(0), _stream(stream)))
    return y


MATVEC_AUTO, MATVEC_REGISTER, MATVEC_RING, MATVEC_TENSOR = 0, 1, 2, 3


def luce_q8_matvec_batch_path(wq, wd, aq, ad, path: int, y=None, stream=None):
    """luce_q8_matvec_batch through one named kernel (MATVEC_*); raises LuceError
    (LUCE_EUNSUPPORTED) when that kernel does not serve the shape."""
    import torch
    _need(wq, torch.int8, "wq")
    _need(aq, torch.int8, "aq")
    _need(ad, torch.float32, "ad")
    N, K = wq.shape
    T = aq.shape[0]
    y = torch.empty((T, N), dtype=torch.float32, device=wq.device) if y is None else y
    _check(load_library().luce_q8_matvec_batch_path(wq.data_ptr(), wd.data_ptr(), N, K, aq.data_ptr(), ad.data_ptr(),
                                                    T, y.data_ptr(), y.stride(0), int(path), _stream(stream)))
    return y


def luce_q8_block_dots(wq, aq, stream=None):
    import torch
    N, K = wq.shape
    T = aq.shape[0]
    out = torch.empty((T, N, K // QK), dtype=torch.int32, device=wq.device)
    _check(load_library().luce_q8_block_dots(wq.data_ptr(), N, K, aq.data_ptr(), T, out.data_ptr(), _stream(stream)))
    return out


def luce_rope_posvec(x, pos, theta: float, stream=None):
    """In-place RoPE of fp32 x [T][n_heads][128] at per-row positions pos (int32 [T])."""
    import torch
    _need(x, torch.float32, "x")
    _need(pos, torch.int32, "pos")
    T, nh, D = x.shape
    _check(load_library().luce_rope_posvec(x.data_ptr(), T, nh, D, nh * D, pos.data_ptr(), float(theta),
                                           _stream(stream)))
    return x


@dataclass
class SeqView:
    """A sequence's cache for one layer (fp16 [Hkv][cap][128] K and V) with ``len``
    keys including this step's ``n_q`` rows, which are rows row0.. of q/out."""
    k: object
    v: object
    len: int
    n_q: int = 1
    row0: int = 0

    def c(self) -> SeqViewC:
        Hkv, cap, D = self.k.shape
        return SeqViewC(self.k.data_ptr(), self.v.data_ptr(), self.len, self.n_q, self.row0, cap,
                        self.k.stride(0), self.k.stride(1))


def _views(views: Sequence[SeqView]):
    arr = (SeqViewC * max(1, len(views)))()
    for i, v in enumerate(views):
        arr[i] = v.c()
    return arr


def luce_kv_append(k, v, views: Sequence[SeqView], stream=None):
    """Append fp32 rows k, v ([T][Hkv][128]) as fp16 at each view's positions."""
    import torch
    _need(k, torch.float32, "k")
    _need(v, torch.float32, "v")
    T, Hkv, D = k.shape
    _check(load_library().luce_kv_append(k.data_ptr(), v.data_ptr(), Hkv * D, Hkv, D, _views(views), len(views),
                                         _stream(stream)))


def luce_decode_attn_workspace_size(n_rows: int, Hq: int, D: int, max_len: int) -> int:
    return int(load_library().luce_decode_attn_workspace_size(n_rows, Hq, D, max_len))


def luce_decode_attn_multiseq(q, views: Sequence[SeqView], n_kv_heads: int, scale: float, out=None, ws=None,
                              stream=None):
    """Decode attention of fp32 q [T][Hq][128] against each row's own fp16 cache."""
    import torch
    _need(q, torch.float32, "q")
    T, Hq, D = q.shape
    out = torch.empty_like(q) if out is None else out
    if ws is None:
        max_len = max(v.len for v in views)
        ws = torch.empty(luce_decode_attn_workspace_size(T, Hq, D, max_len), dtype=torch.uint8, device=q.device)
    _check(load_library().luce_decode_attn_multiseq(q.data_ptr(), _views(views), len(views), Hq, n_kv_heads, D,
                                                    float(scale), out.data_ptr(), ws.data_ptr(), ws.numel(),
                                                    _stream(stream)))
    return out


PAGE_KEYS = 128


@dataclass
class PagedView:
    """A sequence's K/V for one layer in pages: pools fp16 [n_pages][Hkv][128][128],
    ``table`` (device int32) the pool page of each 128-key span; ``len`` keys
    including this step's ``n_q`` rows, which are rows row0.. of q/out."""
    k_pool: object
    v_pool: object
    table: object
    len: int
    n_q: int = 1
    row0: int = 0


def luce_decode_attn_paged(q, views: Sequence[PagedView], n_kv_heads: int, scale: float, out=None, ws=None,
                           stream=None):
    """luce_decode_attn_multiseq over paged caches (the same bits as a flat cache)."""
    import torch
    _need(q, torch.float32, "q")
    T, Hq, D = q.shape
    out = torch.empty_like(q) if out is None else out
    if ws is None:
        max_len = max(v.len for v in views)
        ws = torch.empty(luce_decode_attn_workspace_size(T, Hq, D, max_len), dtype=torch.uint8, device=q.device)
    vc = (PagedViewC * len(views))(*[PagedViewC(v.k_pool.data_ptr(), v.v_pool.data_ptr(), v.table.data_ptr(), v.len,
                                                v.n_q, v.row0) for v in views])
    _check(load_library().luce_decode_attn_paged(q.data_ptr(), vc, len(views), Hq, n_kv_heads, D, float(scale),
                                                 out.data_ptr(), ws.data_ptr(), ws.numel(), _stream(stream)))
    return out


def luce_decode_attn_multiseq_noalloc(q, views: Sequence[SeqView], n_kv_heads: int, scale: float, out=None,
                                      stream=None):
    """luce_decode_attn_multiseq using the library's fixed scratch array instead
    of a workspace, for callers that cannot allocate device memory.  Calls that
    can overlap on the GPU share that array and must be ordered."""
    import torch
    _need(q, torch.float32, "q")
    T, Hq, D = q.shape
    out = torch.empty_like(q) if out is None else out
    _check(load_library().luce_decode_attn_multiseq_noalloc(q.data_ptr(), _views(views), len(views), Hq, n_kv_heads,
                                                            D, float(scale), out.data_ptr(), _stream(stream)))
    return out


# ------------------------------------------------------------ decode step

@dataclass
class LayerTensors:
    attn_norm: object
    wqkv_q: object
    wqkv_d: object
    wo_q: object
    wo_d: object
    ffn_norm: object
    wgu_q: object
    wgu_d: object
    wdown_q: object
    wdown_d: object


class Model:
    """Device weights of a decoder stack plus the C struct that points at them."""

    def __init__(self, layers: List[LayerTensors], hidden: int, n_q_heads: int, n_kv_heads: int, ffn: int,
                 head_dim: int = HEAD_DIM, rms_eps: float = 1e-6, rope_theta: float = 1e6,
                 final_norm=None, head_q=None, head_d=None):
        self.layers = layers
        self.hidden, self.n_q_heads, self.n_kv_heads, self.ffn, self.head_dim = hidden, n_q_heads, n_kv_heads, ffn, head_dim
        self.rms_eps, self.rope_theta = rms_eps, rope_theta
        self.final_norm, self.head_q, self.head_d = final_norm, head_q, head_d
        self.vocab = 0 if head_q is None else head_q.shape[0]
        self._layers_c = (LayerC * max(1, len(layers)))()
        for i, L in enumerate(layers):
            self._layers_c[i] = LayerC(*[getattr(L, n).data_ptr() for n, _ in LayerC._fields_])
        self.c = ModelC(len(layers), hidden, n_q_heads, n_kv_heads, head_dim, ffn, self.vocab, rms_eps, rope_theta,
                        self._layers_c, _ptr(final_norm), _ptr(head_q), _ptr(head_d))

    def layout(self, n_rows: int, max_ctx: int) -> dict:
        out = StepLayoutC()
        _check(load_library().luce_decode_step_layout(ctypes.byref(self.c), n_rows, max_ctx, ctypes.byref(out)))
        return {n: getattr(out, n) for n in _LAYOUT_FIELDS}

    def workspace(self, n_rows: int, max_ctx: int, device="cuda"):
        import torch
        return torch.empty(self.layout(n_rows, max_ctx)["total"], dtype=torch.uint8, device=device)


@dataclass
class Slot:
    """A sequence's K/V cache for every layer: fp16 [n_layers][Hkv][cap][128] each,
    with ``len`` tokens already cached."""
    k: object
    v: object
    len: int

    @property
    def cap(self) -> int:
        return self.k.shape[2]


@dataclass
class PagedSlot:
    """A slot in pages of 128 tokens: pools fp16 [n_pages][n_layers][Hkv][128][128];
    ``table`` lists the pool page of each 128-token span (kept as a host int32
    array and mirrored on the device)."""
    k_pool: object
    v_pool: object
    table: object  # numpy int32
    len: int

    def __post_init__(self):
        import numpy as np
        import torch
        self.table = np.ascontiguousarray(self.table, dtype=np.int32)
        self.table_dev = torch.from_numpy(self.table).to(self.k_pool.device)


def luce_decode_step_paged(model: "Model", slots: Sequence[PagedSlot], rows_per_slot: Sequence[int], x, ws,
                           logits=None, argmax=None, stream=None):
    """luce_decode_step over paged slots (the same bits as flat caches)."""
    import torch
    _need(x, torch.float32, "x")
    n = len(slots)
    sc = (PagedSlotC * max(1, n))()
    for i, s in enumerate(slots):
        sc[i] = PagedSlotC(s.k_pool.data_ptr(), s.v_pool.data_ptr(), s.table_dev.data_ptr(),
                           s.table.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), len(s.table),
                           s.k_pool.shape[0], s.len)
    rows = (ctypes.c_int32 * max(1, n))(*rows_per_slot)
    _check(load_library().luce_decode_step_paged(ctypes.byref(model.c), sc, rows, n, x.data_ptr(), _ptr(logits),
                                                 _ptr(argmax), ws.data_ptr(), ws.numel(), _stream(stream)))
    return x


def luce_decode_step(model: Model, slots: Sequence[Slot], rows_per_slot: Sequence[int], x, ws,
                     logits=None, argmax=None, stream=None):
    """One batched decode step (all layers, optional head) over the given slots.
    x: fp32 [T][hidden] in/out.  The slots' caches get this step's K/V rows."""
    import torch
    _need(x, torch.float32, "x")
    n = len(slots)
    sc = (SlotC * max(1, n))()
    for i, s in enumerate(slots):
        sc[i] = SlotC(s.k.data_ptr(), s.v.data_ptr(), s.len, s.cap)
    rows = (ctypes.c_int32 * max(1, n))(*rows_per_slot)
    _check(load_library().luce_decode_step(ctypes.byref(model.c), sc, rows, n, x.data_ptr(), _ptr(logits),
                                           _ptr(argmax), ws.data_ptr(), ws.numel(), _stream(stream)))
    return x


def luce_decode_step_host(model: Model, slots: Sequence[Slot], rows_per_slot: Sequence[int], x_in, x, ws,
                          x_out=None, logits=None, argmax=None, argmax_out=None, stream=None):
    """luce_decode_step with host rows: x_in (CPU fp32 [T][hidden], ideally
    pinned) is copied to x (device) on the stream, the step runs, and x (and
    argmax) are copied back to x_out (and argmax_out) when given.  Nothing
    waits: synchronise the stream before reading x_out."""
    import torch
    _need(x, torch.float32, "x")
    if x_in.device.type != "cpu" or x_in.dtype != torch.float32 or not x_in.is_contiguous():
        raise TypeError("x_in: expected a contiguous CPU float32 tensor")
    if x_in.shape != x.shape or (x_out is not None and x_out.shape != x.shape):
        raise ValueError("x_in, x and x_out must have the same shape")
    n = len(slots)
    sc = (SlotC * max(1, n))()
    for i, s in enumerate(slots):
        sc[i] = SlotC(s.k.data_ptr(), s.v.data_ptr(), s.len, s.cap)
    rows = (ctypes.c_int32 * max(1, n))(*rows_per_slot)
    _check(load_library().luce_decode_step_host(ctypes.byref(model.c), sc, rows, n, x_in.data_ptr(), x.data_ptr(),
                                                _ptr(x_out), _ptr(logits), _ptr(argmax), _ptr(argmax_out),
                                                ws.data_ptr(), ws.numel(), _stream(stream)))
    return x_out


class DeviceStep:
    """luce_decode_step with its arguments marshalled once, for repeated steps
    over the same slots and buffers (x on the device): each call copies the
    slots' current ``len`` into the prepared slot array and makes the C call
    (nothing else is re-checked).  The stream is the one given, or the current
    stream at construction."""

    def __init__(self, model: Model, slots: Sequence[Slot], rows_per_slot: Sequence[int], x, ws, logits=None,
                 argmax=None, stream=None):
        import torch
        _need(x, torch.float32, "x")
        self.slots = list(slots)
        n = len(self.slots)
        self._sc = (SlotC * max(1, n))()
        for i, s in enumerate(self.slots):
            self._sc[i] = SlotC(s.k.data_ptr(), s.v.data_ptr(), s.len, s.cap)
        self._rows = (ctypes.c_int32 * max(1, n))(*rows_per_slot)
        self._keep = (model, x, ws, logits, argmax)
        self._fn = load_library().luce_decode_step
        self._args = (ctypes.byref(model.c), self._sc, self._rows, n, x.data_ptr(), _ptr(logits), _ptr(argmax),
                      ws.data_ptr(), ws.numel(), _stream(stream))

    def __call__(self):
        sc = self._sc
        for i, s in enumerate(self.slots):
            sc[i].len = s.len
        _check(self._fn(*self._args))


class HostStep:
    """luce_decode_step_host with its arguments marshalled once, for repeated
    steps over the same slots and buffers: each call copies the slots' current
    ``len`` into the prepared slot array and makes the C call (nothing else is
    re-checked).  The stream is the one given, or the current stream at
    construction.  Synchronise the stream before reading x_out."""

    def __init__(self, model: Model, slots: Sequence[Slot], rows_per_slot: Sequence[int], x_in, x, ws,
                 x_out=None, logits=None, argmax=None, argmax_out=None, stream=None):
        import torch
        _need(x, torch.float32, "x")
        if x_in.device.type != "cpu" or x_in.dtype != torch.float32 or not x_in.is_contiguous():
            raise TypeError("x_in: expected a contiguous CPU float32 tensor")
        if x_in.shape != x.shape or (x_out is not None and x_out.shape != x.shape):
            raise ValueError("x_in, x and x_out must have the same shape")
        self.slots = list(slots)
        n = len(self.slots)
        self._sc = (SlotC * max(1, n))()
        for i, s in enumerate(self.slots):
            self._sc[i] = SlotC(s.k.data_ptr(), s.v.data_ptr(), s.len, s.cap)
        self._rows = (ctypes.c_int32 * max(1, n))(*rows_per_slot)
        self._keep = (model, x_in, x, ws, x_out, logits, argmax, argmax_out)
        self._fn = load_library().luce_decode_step_host
        self._args = (ctypes.byref(model.c), self._sc, self._rows, n, x_in.data_ptr(), x.data_ptr(), _ptr(x_out),
                      _ptr(logits), _ptr(argmax), _ptr(argmax_out), ws.data_ptr(), ws.numel(), _stream(stream))

    def __call__(self):
        sc = self._sc
        for i, s in enumerate(self.slots):
            sc[i].len = s.len
        _check(self._fn(*self._args))


class StepGraph:
    """luce_step_graph: the step of HostStep (same arguments) kept as one CUDA
    graph.  Each call passes the slots' current ``len`` to luce_step_graph_run,
    which refreshes the graph's changed nodes (or captures it anew) and
    launches it on the stream given at construction (else the current stream).
    Synchronise the stream before reading x_out.  close() (or garbage
    collection) releases the graph once the stream has finished its runs."""

    def __init__(self, model: Model, slots: Sequence[Slot], rows_per_slot: Sequence[int], x_in, x, ws,
                 x_out=None, logits=None, argmax=None, argmax_out=None, stream=None):
        import torch
        _need(x, torch.float32, "x")
        if x_in.device.type != "cpu" or x_in.dtype != torch.float32 or not x_in.is_contiguous():
            raise TypeError("x_in: expected a contiguous CPU float32 tensor")
        if x_in.shape != x.shape or (x_out is not None and x_out.shape != x.shape):
            raise ValueError("x_in, x and x_out must have the same shape")
        self.slots = list(slots)
        n = len(self.slots)
        sc = (SlotC * max(1, n))()
        for i, s in enumerate(self.slots):
            sc[i] = SlotC(s.k.data_ptr(), s.v.data_ptr(), s.len, s.cap)
        rows = (ctypes.c_int32 * max(1, n))(*rows_per_slot)
        self._lens = (ctypes.c_int32 * max(1, n))()
        self._keep = (model, x_in, x, ws, x_out, logits, argmax, argmax_out)
        self._lib = load_library()
        self._stream = _stream(stream)
        h = ctypes.c_void_p()
        _check(self._lib.luce_step_graph_create(ctypes.byref(model.c), sc, rows, n, x_in.data_ptr(), x.data_ptr(),
                                                _ptr(x_out), _ptr(logits), _ptr(argmax), _ptr(argmax_out),
                                                ws.data_ptr(), ws.numel(), ctypes.byref(h)))
        self._h = h

    def __call__(self):
        lens = self._lens
        for i, s in enumerate(self.slots):
            lens[i] = s.len
        _check(self._lib.luce_step_graph_run(self._h, lens, self._stream))

    def stats(self) -> dict:
        """Captures and node refreshes so far, and the graph's kernel nodes."""
        c, u, k = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int32()
        _check(self._lib.luce_step_graph_stats(self._h, ctypes.byref(c), ctypes.byref(u), ctypes.byref(k)))
        return {"captures": c.value, "node_updates": u.value, "kernels": k.value}

    def close(self):
        if getattr(self, "_h", None) and self._h.value:
            self._lib.luce_step_graph_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
