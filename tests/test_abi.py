"""The C ABI on the host: the library loads, exports every entry point the
header declares, and refuses invalid calls with a status before it touches
the GPU (these calls need no device: validation precedes every launch)."""
import ctypes
import os
import re

import pytest

import invariant_sequence_decode_gb300 as luce
from invariant_sequence_decode_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# Fake, aligned, never-dereferenced device addresses: every call below fails
# validation before any launch.
P = 0x10000


@pytest.fixture(scope="module")
def lib():
    build.build()
    return luce.load_library()


def header_functions():
    text = open(os.path.join(ROOT, "include", "luce.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(luce_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_five_path_entry_points():
    names = header_functions()
    for n in ("luce_q8_quantize_act", "luce_q8_matvec_batch", "luce_rope_posvec", "luce_decode_attn_multiseq",
              "luce_decode_step"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in header_functions() if not hasattr(lib, n)]
    assert not missing, missing
    assert set(luce.EXPORTS) <= set(header_functions())
    assert lib.luce_version() >= 10000


def status_msg(lib):
    return lib.luce_last_error().decode()


@pytest.mark.parametrize("N,K,T,wq,err", [
    (16, 33, 1, P, luce.LUCE_EINVAL),      # K not a multiple of 32
    (16, 64, 17, P, luce.LUCE_EINVAL),     # more rows than the 16-row capacity
    (16, 64, 0, P, luce.LUCE_EINVAL),
    (0, 64, 1, P, luce.LUCE_EINVAL),
    (16, 64, 1, P + 8, luce.LUCE_EINVAL),  # weights not 16-byte aligned
    (16, 64, 1, 0, luce.LUCE_EINVAL),      # null
])
def test_matvec_refuses_bad_shapes(lib, N, K, T, wq, err):
    rc = lib.luce_q8_matvec_batch(wq, P, N, K, P, P, T, P, max(N, 1), None)
    assert rc == err and status_msg(lib)


def test_matvec_ldy_smaller_than_n(lib):
    assert lib.luce_q8_matvec_batch(P, P, 64, 64, P, P, 1, P, 32, None) == luce.LUCE_EINVAL


def test_half_scale_and_fused_producer_refusals(lib):
    assert lib.luce_q8_quantize_act_f16(P, 1, 33, 33, P, P, None) == luce.LUCE_EINVAL       # K not a multiple of 32
    assert lib.luce_q8_quantize_act_f16(None, 1, 32, 32, P, P, None) == luce.LUCE_EINVAL
    assert lib.luce_q8_quantize_act_f16(P, 1, 64, 32, P, P, None) == luce.LUCE_EINVAL       # ldx < K
    assert lib.luce_rmsnorm_q8(P, 17, 64, P, 1e-6, P, P, P, 0, None) == luce.LUCE_EINVAL    # more than 16 rows
    assert lib.luce_rmsnorm_q8(P, 1, 48, P, 1e-6, P, P, P, 1, None) == luce.LUCE_EINVAL     # H not a multiple of 32
    assert lib.luce_rmsnorm_q8(P, 1, 64, P, -1.0, P, P, P, 0, None) == luce.LUCE_EINVAL     # negative eps
    assert lib.luce_rmsnorm_q8(P, 1, 64, P, 1e-6, P, P, P + 2, 0, None) == luce.LUCE_EINVAL  # fp32 scales misaligned
    assert lib.luce_swiglu_q8(P, 1, 33, P, P, P, 0, None) == luce.LUCE_EINVAL
    assert lib.luce_swiglu_q8(P, 0, 64, P, P, P, 1, None) == luce.LUCE_EINVAL
    assert lib.luce_swiglu_q8(P, 1, 64, None, P, P, 1, None) == luce.LUCE_EINVAL


def test_quantize_and_rope_refusals(lib):
    assert lib.luce_q8_quantize_act(P, 1, 40, 40, P, P, None) == luce.LUCE_EINVAL
    assert lib.luce_q8_quantize_act(P, 1, 64, 32, P, P, None) == luce.LUCE_EINVAL
    assert lib.luce_rope_posvec(P, 1, 4, 64, 256, P, 1e6, None) == luce.LUCE_EUNSUPPORTED
    assert lib.luce_rope_posvec(P, 1, 4, 128, 256, P, 1e6, None) == luce.LUCE_EINVAL  # ldx < heads*D
    assert lib.luce_rope_posvec(P, 1, 4, 128, 512, P, -1.0, None) == luce.LUCE_EINVAL


def views(specs):
    arr = (luce.SeqViewC * len(specs))()
    for i, (ln, nq, row0) in enumerate(specs):
        arr[i] = luce.SeqViewC(P, P + 0x100000, ln, nq, row0, 4096, 4096 * 128, 128)
    return arr


def test_attention_refusals(lib):
    ws = 1 << 30
    # five sequences are refused, not clamped ("more than 4 is refused")
    v5 = views([(10, 1, i) for i in range(5)])
    assert lib.luce_decode_attn_multiseq(P, v5, 5, 8, 2, 128, 0.1, P, P, ws, None) == luce.LUCE_EINVAL
    assert "refused" in status_msg(lib)
    v = views([(10, 1, 0), (10, 1, 0)])  # a row claimed twice
    assert lib.luce_decode_attn_multiseq(P, v, 2, 8, 2, 128, 0.1, P, P, ws, None) == luce.LUCE_EINVAL
    v = views([(10, 1, 1)])  # row 0 uncovered
    assert lib.luce_decode_attn_multiseq(P, v, 1, 8, 2, 128, 0.1, P, P, ws, None) == luce.LUCE_EINVAL
    v = views([(10, 5, 0)])  # five rows for one sequence
    assert lib.luce_decode_attn_multiseq(P, v, 1, 8, 2, 128, 0.1, P, P, ws, None) == luce.LUCE_EINVAL
    v = views([(5000, 1, 0)])  # len beyond cap
    assert lib.luce_decode_attn_multiseq(P, v, 1, 8, 2, 128, 0.1, P, P, ws, None) == luce.LUCE_EINVAL
    v = views([(10, 1, 0)])
    assert lib.luce_decode_attn_multiseq(P, v, 1, 18, 2, 128, 0.1, P, P, ws, None) == luce.LUCE_EUNSUPPORTED
    assert lib.luce_decode_attn_multiseq(P, v, 1, 9, 2, 128, 0.1, P, P, ws, None) == luce.LUCE_EINVAL
    assert lib.luce_decode_attn_multiseq(P, v, 1, 8, 2, 128, 0.1, P, P, 16, None) == luce.LUCE_ENOSPACE
    assert lib.luce_decode_attn_workspace_size(4, 8, 128, 1000) == 4 * 8 * 8 * 132 * 4


def fake_model(n_layers=2, vocab=0, head_dim=128, hidden=256, hq=4, hkv=2, ffn=512):
    layers = (luce.LayerC * n_layers)()
    for i in range(n_layers):
        layers[i] = luce.LayerC(*([P] * 10))
    m = luce.ModelC(n_layers, hidden, hq, hkv, head_dim, ffn, vocab, 1e-6, 1e6, layers,
                    P if vocab else None, P if vocab else None, P if vocab else None)
    return m, layers


def slots(specs):
    arr = (luce.SlotC * len(specs))()
    for i, (ln, cap) in enumerate(specs):
        arr[i] = luce.SlotC(P + i * 0x1000000, P + i * 0x1000000 + 0x800000, ln, cap)
    return arr


def rows(r):
    return (ctypes.c_int32 * len(r))(*r)


def test_decode_step_refusals(lib):
    m, _keep = fake_model()
    big = 1 << 40
    step = lib.luce_decode_step
    s5 = slots([(3, 64)] * 5)
    assert step(ctypes.byref(m), s5, rows([1] * 5), 5, P, None, None, P, big, None) == luce.LUCE_EINVAL
    assert "refused" in status_msg(lib)
    s = slots([(3, 64), (3, 64)])
    assert step(ctypes.byref(m), s, rows([1, 5]), 2, P, None, None, P, big, None) == luce.LUCE_EINVAL
    assert step(ctypes.byref(m), slots([(62, 64)]), rows([3]), 1, P, None, None, P, big, None) == luce.LUCE_EINVAL
    assert step(ctypes.byref(m), s, rows([1, 1]), 2, P, None, None, P, 1024, None) == luce.LUCE_ENOSPACE
    # two slots may not share one cache
    same = (luce.SlotC * 2)(luce.SlotC(P, P + 64, 3, 64), luce.SlotC(P, P + 128, 3, 64))
    assert step(ctypes.byref(m), same, rows([1, 1]), 2, P, None, None, P, big, None) == luce.LUCE_EINVAL
    # ... nor overlap at an offset: each cache here spans 2 layers x 2 heads x 64 positions x 128 halves = 64 KiB
    ext = 2 * 2 * 64 * 128 * 2
    apart = (luce.SlotC * 2)(luce.SlotC(P, P + 0x800000, 3, 64), luce.SlotC(P + ext, P + 0x900000, 3, 64))
    # adjacent caches pass the overlap check (shown by the later workspace refusal; nothing is launched)
    assert step(ctypes.byref(m), apart, rows([1, 1]), 2, P, None, None, P, 1024, None) == luce.LUCE_ENOSPACE
    offset = (luce.SlotC * 2)(luce.SlotC(P, P + 0x800000, 3, 64), luce.SlotC(P + ext - 256, P + 0x900000, 3, 64))
    assert step(ctypes.byref(m), offset, rows([1, 1]), 2, P, None, None, P, big, None) == luce.LUCE_EINVAL
    assert "overlaps" in status_msg(lib)
    kv_alias = (luce.SlotC * 1)(luce.SlotC(P, P + ext // 2, 3, 64))
    assert step(ctypes.byref(m), kv_alias, rows([1]), 1, P, None, None, P, big, None) == luce.LUCE_EINVAL
    assert "overlaps" in status_msg(lib)
    # logits without a head
    assert step(ctypes.byref(m), s, rows([1, 1]), 2, P, P, None, P, big, None) == luce.LUCE_EINVAL
    m64, _k2 = fake_model(head_dim=64)
    assert step(ctypes.byref(m64), s, rows([1, 1]), 2, P, None, None, P, big, None) == luce.LUCE_EUNSUPPORTED
    mh, _k3 = fake_model(hidden=250)
    assert step(ctypes.byref(mh), s, rows([1, 1]), 2, P, None, None, P, big, None) == luce.LUCE_EINVAL


def test_decode_step_host_refusals(lib):
    """The host-buffer step validates like the device step, plus its own
    buffers, and enqueues nothing (no copy either) when it refuses."""
    m, _keep = fake_model()
    big = 1 << 40
    host = lib.luce_decode_step_host
    s = slots([(3, 64), (3, 64)])
    xin = (ctypes.c_float * 16)()
    # null x_in
    assert host(ctypes.byref(m), s, rows([1, 1]), 2, None, P, None, None, None, None, P, big, None) == luce.LUCE_EINVAL
    # the device step's refusals apply: 5 slots, a row count above 4, too small a workspace
    assert host(ctypes.byref(m), slots([(3, 64)] * 5), rows([1] * 5), 5, xin, P, None, None, None, None, P, big,
                None) == luce.LUCE_EINVAL
    assert host(ctypes.byref(m), s, rows([1, 5]), 2, xin, P, None, None, None, None, P, big, None) == luce.LUCE_EINVAL
    assert host(ctypes.byref(m), s, rows([1, 1]), 2, xin, P, None, None, None, None, P, 1024, None) == luce.LUCE_ENOSPACE
    # argmax_out without the argmax buffer
    out = (ctypes.c_int32 * 2)()
    assert host(ctypes.byref(m), s, rows([1, 1]), 2, xin, P, None, None, None, out, P, big, None) == luce.LUCE_EINVAL


def test_step_graph_create_validates_and_makes_no_cuda_call(lib):
    """luce_step_graph_create checks what luce_decode_step_host checks and
    touches no device; run refuses bad lengths before any CUDA call; destroy
    of a never-run object (and of NULL) needs no device either."""
    m, _keep = fake_model()
    big = 1 << 40
    create = lib.luce_step_graph_create
    s = slots([(3, 64), (3, 64)])
    xin = (ctypes.c_float * 16)()
    h = ctypes.c_void_p()
    assert create(ctypes.byref(m), s, rows([1, 1]), 2, None, P, None, None, None, None, P, big,
                  ctypes.byref(h)) == luce.LUCE_EINVAL and not h.value
    assert create(ctypes.byref(m), s, rows([1, 5]), 2, xin, P, None, None, None, None, P, big,
                  ctypes.byref(h)) == luce.LUCE_EINVAL
    assert create(ctypes.byref(m), s, rows([1, 1]), 2, xin, P, None, None, None, None, P, 1024,
                  ctypes.byref(h)) == luce.LUCE_ENOSPACE
    assert create(ctypes.byref(m), s, rows([1, 1]), 2, xin, P, None, P, None, None, P, big,
                  ctypes.byref(h)) == luce.LUCE_EINVAL  # logits without a head
    assert create(ctypes.byref(m), s, rows([1, 1]), 2, xin, P, None, None, None, None, P, big, None) == luce.LUCE_EINVAL
    assert create(ctypes.byref(m), s, rows([1, 1]), 2, xin, P, None, None, None, None, P, big,
                  ctypes.byref(h)) == luce.LUCE_OK and h.value
    c, u, k = ctypes.c_int64(-1), ctypes.c_int64(-1), ctypes.c_int32(-1)
    assert lib.luce_step_graph_stats(h, ctypes.byref(c), ctypes.byref(u), ctypes.byref(k)) == luce.LUCE_OK
    assert (c.value, u.value, k.value) == (0, 0, 0)
    run = lib.luce_step_graph_run
    assert run(h, None, None) == luce.LUCE_EINVAL
    assert run(h, (ctypes.c_int32 * 2)(3, 64), None) == luce.LUCE_EINVAL  # len + rows > cap
    assert "exceeds cap" in status_msg(lib)
    assert run(h, (ctypes.c_int32 * 2)(-1, 3), None) == luce.LUCE_EINVAL
    assert lib.luce_step_graph_stats(h, ctypes.byref(c), None, None) == luce.LUCE_OK and c.value == 0
    assert lib.luce_step_graph_destroy(h) == luce.LUCE_OK
    assert lib.luce_step_graph_destroy(None) == luce.LUCE_OK
    assert lib.luce_step_graph_stats(None, None, None, None) == luce.LUCE_EINVAL


def test_step_layout_is_monotone_and_part_is_last(lib):
    m, _keep = fake_model()
    lay = luce.StepLayoutC()
    assert lib.luce_decode_step_layout(ctypes.byref(m), 4, 2051, ctypes.byref(lay)) == 0
    lay2 = luce.StepLayoutC()
    assert lib.luce_decode_step_layout(ctypes.byref(m), 4, 32768, ctypes.byref(lay2)) == 0
    assert lay2.total > lay.total and lay2.xf_d == lay.xf_d and lay.part >= lay.xf_d
    assert all(getattr(lay, n) % 256 == 0 for n, _ in luce.StepLayoutC._fields_)


def paged_slots(specs):
    """specs: (len, table list, n_pages, pool id); keeps the tables alive."""
    arr = (luce.PagedSlotC * len(specs))()
    keep = []
    for i, (ln, table, n_pages, pool) in enumerate(specs):
        t = (ctypes.c_int32 * max(1, len(table)))(*table)
        keep.append(t)
        arr[i] = luce.PagedSlotC(P + pool * 0x1000000, P + pool * 0x1000000 + 0x800000, P + 0x40000 * (i + 1),
                                 t, len(table), n_pages, ln)
    return arr, keep


def test_decode_step_paged_refusals(lib):
    m, _keep = fake_model()
    big = 1 << 40
    step = lib.luce_decode_step_paged
    ok, k1 = paged_slots([(100, [3, 1], 4, 0), (5, [0], 4, 1)])
    # a table entry outside the pool
    bad, k2 = paged_slots([(200, [3, 9], 4, 0)])
    assert step(ctypes.byref(m), bad, rows([1]), 1, P, None, None, P, big, None) == luce.LUCE_EINVAL
    assert "outside" in status_msg(lib)
    # too few table entries for len + rows (130 keys need 2 pages)
    short, k3 = paged_slots([(127, [2], 4, 0)])
    assert step(ctypes.byref(m), short, rows([3]), 1, P, None, None, P, big, None) == luce.LUCE_EINVAL
    # two slots of one pool writing / reading the same page
    clash, k4 = paged_slots([(10, [2], 4, 0), (20, [2], 4, 0)])
    assert step(ctypes.byref(m), clash, rows([1, 1]), 2, P, None, None, P, big, None) == luce.LUCE_EINVAL
    assert "also referenced" in status_msg(lib)
    # more than four slots, too many rows, workspace too small
    five, k5 = paged_slots([(3, [i], 8, i) for i in range(5)])
    assert step(ctypes.byref(m), five, rows([1] * 5), 5, P, None, None, P, big, None) == luce.LUCE_EINVAL
    assert step(ctypes.byref(m), ok, rows([1, 5]), 2, P, None, None, P, big, None) == luce.LUCE_EINVAL
    assert step(ctypes.byref(m), ok, rows([1, 1]), 2, P, None, None, P, 1024, None) == luce.LUCE_ENOSPACE


def test_decode_attn_paged_refusals(lib):
    ws = 1 << 30
    def pv(specs):
        arr = (luce.PagedViewC * len(specs))()
        for i, (ln, nq, r0) in enumerate(specs):
            arr[i] = luce.PagedViewC(P, P + 0x800000, P + 0x100000, ln, nq, r0)
        return arr
    f = lib.luce_decode_attn_paged
    assert f(P, pv([(10, 1, 0)] * 5), 5, 8, 2, 128, 0.1, P, P, ws, None) == luce.LUCE_EINVAL
    assert f(P, pv([(10, 1, 1)]), 1, 8, 2, 128, 0.1, P, P, ws, None) == luce.LUCE_EINVAL   # row 0 uncovered
    assert f(P, pv([(2, 3, 0)]), 1, 8, 2, 128, 0.1, P, P, ws, None) == luce.LUCE_EINVAL    # len < n_q
    assert f(P, pv([(10, 1, 0)]), 1, 8, 2, 64, 0.1, P, P, ws, None) == luce.LUCE_EUNSUPPORTED
    assert f(P, pv([(10, 1, 0)]), 1, 8, 2, 128, 0.1, P, P, 16, None) == luce.LUCE_ENOSPACE
    assert f(P, pv([(200000, 1, 0)]), 1, 8, 2, 128, 0.1, P, P, ws, None) == luce.LUCE_EUNSUPPORTED


def test_wait_counter_and_expiry_hook_refusals(lib):
    """The timeout counter needs somewhere to write; the expiry hook takes a
    limit between 1 us and 1 s.  Both refuse before touching the device."""
    assert lib.luce_wait_timeouts(None, 0) == luce.LUCE_EINVAL
    assert "null count" in status_msg(lib)
    for bad in (0, 999, 1_000_000_001, -5):
        assert lib.luce_test_wait_expiry(bad, None) == luce.LUCE_EINVAL
