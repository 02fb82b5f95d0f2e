"""The step graph (luce_step_graph) against the host-buffer step, bit for bit.

The graph holds the launches luce_decode_step_host makes, with the same
arguments, so over a run of consecutive steps - the slots' lengths growing
across split-K chunk edges, which changes attention grids and arguments, and
across the 16,384-key edge where a row's chunks change kernel, which changes
the graph's nodes - its copied-back rows, argmax, logits and K/V appends equal
the host step's bit for bit; its refreshes and captures are counted, and its
kernel nodes equal the launches the host step makes.  Page-locked host
buffers are read and written by the step's kernels through their mapping;
pageable ones go through copies: both give the same bits.
"""
import numpy as np
import pytest

from invariant_sequence_decode_gb300 import workloads as wl

torch = pytest.importorskip("torch")
import invariant_sequence_decode_gb300 as luce  # noqa: E402

pytestmark = pytest.mark.gpu

LAYER_FIELDS = ["attn_norm", "wqkv_q", "wqkv_d", "wo_q", "wo_d", "ffn_norm", "wgu_q", "wgu_d", "wdown_q", "wdown_d"]
D = wl.TINY_LAYER
N_LAYERS, VOCAB = 2, 300


@pytest.fixture(scope="module")
def model():
    from invariant_sequence_decode_gb300 import build
    build.build()
    luce.load_library()
    layers = [luce.LayerTensors(*[cuda(getattr(wl.layer_host(31, l, D), f)) for f in LAYER_FIELDS])
              for l in range(N_LAYERS)]
    fn, hq, hd = wl.head_host(31, D, VOCAB)
    return luce.Model(layers, D.hidden, D.n_q_heads, D.n_kv_heads, D.ffn, rms_eps=D.rms_eps,
                      rope_theta=D.rope_theta, final_norm=cuda(fn), head_q=cuda(hq), head_d=cuda(hd))


def cuda(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def bits(t):
    return np.ascontiguousarray(t.cpu().numpy() if isinstance(t, torch.Tensor) else t).view(np.uint8)


def caches(seed, cap, length):
    ks, vs = zip(*[wl.cache_host(seed, 0, l, D, cap, length) for l in range(N_LAYERS)])
    return np.stack(ks), np.stack(vs)


class Arm:
    """One way of running the steps: 'host' (HostStep) or 'graph' (StepGraph),
    on its own copy of the caches and buffers."""

    def __init__(self, kind, model, cache_h, lens, rows_per_slot, cap, pinned=True):
        T = sum(rows_per_slot)
        self.slots = [luce.Slot(cuda(k), cuda(v), ln) for (k, v), ln in zip(cache_h, lens)]
        pin = (lambda t: t.pin_memory()) if pinned else (lambda t: t)
        self.x_in = pin(torch.empty((T, D.hidden), dtype=torch.float32))
        self.x_out = pin(torch.empty((T, D.hidden), dtype=torch.float32))
        self.am_out = pin(torch.empty(T, dtype=torch.int32))
        self.x = torch.empty((T, D.hidden), dtype=torch.float32, device="cuda")
        self.logits = torch.empty((T, VOCAB), dtype=torch.float32, device="cuda")
        self.am = torch.empty(T, dtype=torch.int32, device="cuda")
        self.ws = model.workspace(T, cap)
        cls = luce.StepGraph if kind == "graph" else luce.HostStep
        self.step = cls(model, self.slots, rows_per_slot, self.x_in, self.x, self.ws, x_out=self.x_out,
                        logits=self.logits, argmax=self.am, argmax_out=self.am_out)

    def run(self, x_rows):
        self.x_in.copy_(torch.from_numpy(x_rows))
        before = luce.launch_count()
        self.step()
        torch.cuda.synchronize()
        return luce.launch_count() - before


def run_both(model, lens, rows_per_slot, cap, n_steps, seed, arms=(("host", True), ("graph", True))):
    """Steps through two arms (kind, page-locked buffers?) compared bit for bit;
    the second arm's graph statistics when it is a graph."""
    cache_h = [caches(seed + s, cap, ln) for s, ln in enumerate(lens)]
    host, graph = (Arm(k, model, cache_h, lens, rows_per_slot, cap, p) for k, p in arms)
    T = sum(rows_per_slot)
    for i in range(n_steps):
        xr = wl.acts(seed + 100 + i, T, D.hidden, sub=5)
        n_host = host.run(xr)
        n_graph = graph.run(xr)
        if arms[1][0] == "graph":
            assert n_graph == n_host == graph.step.stats()["kernels"], (i, n_host, n_graph)
        assert np.array_equal(bits(graph.x_out), bits(host.x_out)), i
        assert np.array_equal(graph.am_out.numpy(), host.am_out.numpy()), i
        assert np.array_equal(bits(graph.logits), bits(host.logits)), i
        for a, b in zip(graph.slots, host.slots):
            end = a.len + max(rows_per_slot)
            assert np.array_equal(bits(a.k[:, :, :end]), bits(b.k[:, :, :end])), i
            assert np.array_equal(bits(a.v[:, :, :end]), bits(b.v[:, :, :end])), i
        for arm in (host, graph):
            for s, sl in enumerate(arm.slots):
                sl.len += rows_per_slot[s]
    return graph.step.stats() if arms[1][0] == "graph" else None


def test_graph_equals_host_step_across_chunk_edges(model):
    # lengths cross the 128-key chunk edges at 128 and 384 during the run:
    # grids and attention arguments change, the node sequence does not
    stats = run_both(model, lens=[124, 126, 380], rows_per_slot=[1, 2, 1], cap=420, n_steps=6, seed=41)
    assert stats["captures"] == 1 and stats["node_updates"] > 0, stats


def test_graph_recaptures_when_an_attention_kind_appears(model):
    # slot 0 passes 16,384 keys after two steps: its chunks move to the
    # 256-key kernel, a third attention launch per layer, so the graph is
    # captured anew once and then refreshed again
    stats = run_both(model, lens=[16382, 90], rows_per_slot=[1, 1], cap=16400, n_steps=4, seed=43)
    assert stats["captures"] == 2 and stats["node_updates"] > 0, stats


def test_graph_refuses_bad_lengths_and_enqueues_nothing(model):
    cache_h = [caches(45, 64, 10)]
    arm = Arm("graph", model, cache_h, [10], [2], 64)
    arm.x_in.copy_(torch.from_numpy(wl.acts(46, 2, D.hidden, sub=5)))
    arm.slots[0].len = 63  # 63 + 2 rows > cap 64
    before = luce.launch_count()
    with pytest.raises(luce.LuceError):
        arm.step()
    assert luce.launch_count() == before and arm.step.stats()["captures"] == 0


def test_pageable_host_buffers_give_the_bits_of_page_locked_ones(model):
    # pageable buffers take copy-engine transfers, page-locked ones the mapped
    # reads and writes of the first and last kernels
    run_both(model, lens=[60, 200], rows_per_slot=[2, 1], cap=256, n_steps=2, seed=47,
             arms=(("host", False), ("host", True)))


def test_graph_refuses_pageable_host_buffers(model):
    arm = Arm("graph", model, [caches(48, 64, 10)], [10], [1], 64, pinned=False)
    before = luce.launch_count()
    with pytest.raises(luce.LuceError):
        arm.step()
    assert luce.launch_count() == before and arm.step.stats()["captures"] == 0
