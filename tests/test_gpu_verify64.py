"""Wide speculative verify at full size: 4 slots x 2/3/4 rows (8/12/16 rows)
through 64 distinct layers of the 27B-shaped layer plus a 151,936 x 5120 q8_0
head, cache lengths uniform on [1024, 2051].

Checked: every slot's rows, logits, argmax and cache bytes equal the slot run
alone (bitwise); the last layer and the head stage by stage against the
oracle (its inputs taken from the GPU's own stage inputs, see
test_gpu_step); cache rows other than the ones the step writes unchanged.
"""
import numpy as np
import pytest

from invariant_sequence_decode_gb300 import workloads as wl

torch = pytest.importorskip("torch")
import invariant_sequence_decode_gb300 as luce  # noqa: E402
from test_gpu_step import LAYER_FIELDS, same_bits, staged_layer_check  # noqa: E402

pytestmark = pytest.mark.gpu

N_LAYERS = 64
SEED = 4


def cuda(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


class Stack:
    """The 64-layer model on the device (generated and uploaded layer by layer)."""

    def __init__(self):
        d = wl.LAYER27B
        self.dims = d
        self.n_layers = N_LAYERS
        self.layers_d = []
        self.layers_h = {}
        for l in range(N_LAYERS):
            h = wl.layer_host(SEED, l, d)
            self.layers_d.append(luce.LayerTensors(*[cuda(getattr(h, f)) for f in LAYER_FIELDS]))
            if l == N_LAYERS - 1:
                self.layers_h[l] = h
        self.head_h = wl.head_host(SEED, d, wl.VOCAB)
        fn, hq, hd = [cuda(a) for a in self.head_h]
        self.vocab = wl.VOCAB
        self.model = luce.Model(self.layers_d, d.hidden, d.n_q_heads, d.n_kv_heads, d.ffn,
                                final_norm=fn, head_q=hq, head_d=hd)


@pytest.fixture(scope="module")
def stack():
    from invariant_sequence_decode_gb300 import build
    build.build()
    luce.load_library()
    return Stack()


class VerifyCase:
    def __init__(self, stack, rows_per_slot):
        d = stack.dims
        self.__dict__.update(stack.__dict__)
        self.lens = wl.lens(SEED, 4, 1024, 2051, sub=rows_per_slot)
        self.rows = [rows_per_slot] * 4
        self.cap = 2051 + 4
        # caches [L][Hkv][cap][D], generated on the device side by slot and layer
        self.k_d, self.v_d = [], []
        for s, ln in enumerate(self.lens):
            kk = torch.empty((N_LAYERS, d.n_kv_heads, self.cap, d.head_dim), dtype=torch.float16, device="cuda")
            vv = torch.empty_like(kk)
            for l in range(N_LAYERS):
                k, v = wl.cache_host(SEED, s, l, d, self.cap, ln)
                kk[l].copy_(torch.from_numpy(k))
                vv[l].copy_(torch.from_numpy(v))
            self.k_d.append(kk)
            self.v_d.append(vv)
        self.x = wl.acts(SEED, sum(self.rows), d.hidden, sub=20 + rows_per_slot)

    def run(self, idx):
        rows = [self.rows[s] for s in idx]
        starts = np.cumsum([0] + self.rows)
        x = cuda(np.concatenate([self.x[starts[s]:starts[s] + self.rows[s]] for s in idx]))
        T = sum(rows)
        slots = [luce.Slot(self.k_d[s].clone(), self.v_d[s].clone(), self.lens[s]) for s in idx]
        ws = self.model.workspace(T, self.cap)
        logits = torch.empty((T, self.vocab), dtype=torch.float32, device="cuda")
        am = torch.empty(T, dtype=torch.int32, device="cuda")
        luce.luce_decode_step(self.model, slots, rows, x, ws, logits, am)
        torch.cuda.synchronize()
        return dict(x=x.cpu().numpy(), ws=ws, slots=slots, logits=logits.cpu().numpy(), argmax=am.cpu().numpy(),
                    T=T, rows=rows, idx=idx)


@pytest.mark.parametrize("rows_per_slot", [2, 3, 4])
def test_verify64_batched_equals_solo_and_stages_match_oracle(stack, rows_per_slot):
    case = VerifyCase(stack, rows_per_slot)
    b = case.run([0, 1, 2, 3])
    assert b["T"] == 4 * rows_per_slot
    assert np.all(np.isfinite(b["logits"]))
    r0 = 0
    for s in range(4):
        so = case.run([s])
        n = rows_per_slot
        assert same_bits(so["x"], b["x"][r0:r0 + n])
        assert same_bits(so["logits"], b["logits"][r0:r0 + n])
        assert np.array_equal(so["argmax"], b["argmax"][r0:r0 + n])
        kb, ks = b["slots"][s].k, so["slots"][0].k
        vb, vs = b["slots"][s].v, so["slots"][0].v
        assert torch.equal(kb.view(torch.int16), ks.view(torch.int16))
        assert torch.equal(vb.view(torch.int16), vs.view(torch.int16))
        # only positions [len, len + n) of every layer changed
        ch = (kb.view(torch.int16) != case.k_d[s].view(torch.int16)).any(dim=3).any(dim=1).any(dim=0)
        changed = torch.nonzero(ch).flatten().tolist()
        assert set(changed) <= set(range(case.lens[s], case.lens[s] + n))
        r0 += n
    if rows_per_slot == 4:
        staged_layer_check(case, b, layer=N_LAYERS - 1)
