"""The attention entry point that allocates nothing.

luce_decode_attn_multiseq_noalloc serves callers that cannot allocate device
memory (it uses the library's fixed scratch array instead of a caller
workspace).  Checked through the C ABI against luce_decode_attn_multiseq on
two calls in a row (the second reuses the scratch the first left behind),
and for its refusal of work that does not fit the array.  This file is
collected last so that a run stopping at the first failure has already run
every other test.
"""
import ctypes
import math

import numpy as np
import pytest

from invariant_sequence_decode_gb300 import workloads as wl

torch = pytest.importorskip("torch")
import invariant_sequence_decode_gb300 as luce  # noqa: E402

pytestmark = pytest.mark.gpu

TOL = 2e-3  # the attention tolerance of the other GPU tests


@pytest.fixture(scope="module")
def lib():
    from invariant_sequence_decode_gb300 import build
    build.build()
    return luce.load_library()


def cuda(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def case(seed, lens, nq, Hq, Hkv):
    d = wl.Dims(0, Hq, Hkv, 128, 0)
    views, row0 = [], 0
    for s, (L, n) in enumerate(zip(lens, nq)):
        k, v = wl.cache_host(seed, s, 0, d, L, L)
        views.append(luce.SeqView(cuda(k), cuda(v), L, n, row0))
        row0 += n
    return cuda(wl.qvec(seed, row0, Hq, sub=4)), views


def call_noalloc(lib, q, views, Hkv, scale):
    out = torch.full_like(q, float("nan"))
    T, Hq, D = q.shape
    rc = lib.luce_decode_attn_multiseq_noalloc(q.data_ptr(), luce._views(views), len(views), Hq, Hkv, D,
                                               float(scale), out.data_ptr(),
                                               torch.cuda.current_stream().cuda_stream)
    return rc, out


def test_noalloc_matches_workspace_entry_point_twice(lib):
    scale = 1 / math.sqrt(128)
    cases = [(case(21, [17, 100, 513, 1000], [1, 1, 1, 1], 8, 2), 2),
             (case(22, [1030, 1800, 2051, 700], [4, 3, 2, 1], 40, 8), 8)]
    for (q, views), Hkv in cases:
        ref = luce.luce_decode_attn_multiseq(q, views, Hkv, scale)
        rc, got = call_noalloc(lib, q, views, Hkv, scale)
        assert rc == 0, lib.luce_last_error().decode()
        torch.cuda.synchronize()
        a, b = got.cpu().numpy(), ref.cpu().numpy()
        assert np.max(np.abs(a - b)) <= TOL
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def test_noalloc_refuses_work_beyond_its_scratch(lib):
    Hq, Hkv, L = 64, 8, 32768
    need = 4 * math.ceil(L / 256) * Hq * 528  # 4 rows of 256-key chunks, 528 bytes per chunk and head
    assert need > lib.luce_decode_attn_noalloc_max_bytes()
    kv = torch.zeros((Hkv, L, 128), dtype=torch.float16, device="cuda")
    views = [luce.SeqView(kv, kv, L, 1, s) for s in range(4)]
    q = torch.zeros((4, Hq, 128), dtype=torch.float32, device="cuda")
    rc, out = call_noalloc(lib, q, views, Hkv, 0.1)
    assert rc == luce.LUCE_ENOSPACE
    assert "scratch" in lib.luce_last_error().decode()
    torch.cuda.synchronize()
    assert torch.isnan(out).all()  # nothing was launched
