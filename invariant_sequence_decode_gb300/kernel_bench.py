"""Per-kernel microbenchmark (CUDA events, L2 flushed between launches).

  python -m invariant_sequence_decode_gb300.kernel_bench matvec --N 34816 --K 5120 --T 4
  python -m invariant_sequence_decode_gb300.kernel_bench attn --lens 2051,2051,2051,2051 --hq 40 --hkv 8
  python -m invariant_sequence_decode_gb300.kernel_bench step --nseq 4
  python -m invariant_sequence_decode_gb300.kernel_bench layer --T 4

Prints one JSON line per case with the launch time (mean, and median where a
single launch is timed) and the algorithmic GB/s (weights N*K*34/32 +
activations + outputs for the matvec; K/V bytes for attention).  `--reps` launches are timed; use a small `--reps` under a
profiler.
"""
from __future__ import annotations

import argparse
import json
import statistics

import numpy as np


class L2Flush:
    """Write one 256 MiB buffer, then read a second one: the write evicts
    whatever the L2 held, and the read (twice the L2's size) writes the dirty
    lines back and leaves the L2 holding clean lines of unrelated data, so the
    next launch pays neither hits nor write-backs it did not cause.  (Reading
    back the buffer just written would leave its last lines dirty in L2.)"""

    def __init__(self, torch):
        self.torch = torch
        self.buf = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
        self.clean = torch.zeros(256 << 20, dtype=torch.uint8, device="cuda")
        self.sink = torch.empty(1, dtype=torch.int64, device="cuda")

    def __call__(self):
        self.buf.fill_(1)
        self.sink.copy_(self.clean.view(self.torch.int64).sum().view(1))


def time_launches(torch, fn, flush, reps: int):
    st = torch.cuda.current_stream()
    out = []
    for _ in range(reps):
        if flush:
            flush()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(st)
        fn()
        b.record(st)
        out.append((a, b))
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in out]


def main(argv=None):
    import torch
    import invariant_sequence_decode_gb300 as luce
    from invariant_sequence_decode_gb300 import build, workloads as wl

    ap = argparse.ArgumentParser()
    ap.add_argument("kernel", choices=["matvec", "attn", "step", "layer"])
    ap.add_argument("--N", type=int, default=34816)
    ap.add_argument("--K", type=int, default=5120)
    ap.add_argument("--T", default="4")
    ap.add_argument("--lens", default="2051,2051,2051,2051")
    ap.add_argument("--hq", type=int, default=40)
    ap.add_argument("--hkv", type=int, default=8)
    ap.add_argument("--nseq", type=int, default=4)
    ap.add_argument("--rows", type=int, default=1, help="step: rows per slot (1 decode, 2..4 verify)")
    ap.add_argument("--reps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--no-flush", action="store_true")
    ap.add_argument("--path", type=int, default=0,
                    help="matvec kernel: 0 library choice, 1 register dp4a, 2 dp4a TMA ring, 3 tensor-core ring")
    a = ap.parse_args(argv)
    build.build()
    luce.load_library()
    flush = None if a.no_flush else L2Flush(torch)
    cu = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()

    if a.kernel == "matvec":
        wq, wd = wl.q8_weights(0, wl.tid(wl.W_MAT, 1), a.N, a.K)
        W, D = cu(wq), cu(wd)
        for T in [int(t) for t in a.T.split(",")]:
            aq, ad = luce.luce_q8_quantize_act(cu(wl.acts(0, T, a.K)))
            y = torch.empty((T, a.N), dtype=torch.float32, device="cuda")
            fn = lambda: luce.luce_q8_matvec_batch_path(W, D, aq, ad, a.path, y)
            for _ in range(a.warmup):
                fn()
            ms = time_launches(torch, fn, flush, a.reps)
            b = a.N * a.K * 34 // 32 + T * a.K + T * (a.K // 32) * 4 + T * a.N * 4
            m = statistics.mean(ms)
            print(json.dumps({"kernel": "q8_matvec", "path": a.path, "N": a.N, "K": a.K, "T": T,
                              "us_mean": round(m * 1e3, 2), "us_median": round(statistics.median(ms) * 1e3, 2),
                              "us_min": round(min(ms) * 1e3, 2), "gbps": round(b / m / 1e6, 1)}))
    elif a.kernel == "layer":
        # the four q8_0 projections of the 27B-shaped layer (qkv, o, gate||up, down)
        d = wl.LAYER27B
        shapes = [((d.n_q_heads + 2 * d.n_kv_heads) * d.head_dim, d.hidden), (d.hidden, d.n_q_heads * d.head_dim),
                  (2 * d.ffn, d.hidden), (d.hidden, d.ffn)]
        mats = [tuple(cu(m) for m in wl.q8_weights(1, wl.tid(wl.W_MAT, 8 + i), N, K)) for i, (N, K) in enumerate(shapes)]
        for T in [int(t) for t in a.T.split(",")]:
            tot_b, tot_ms, fns, per = 0, 0.0, [], []
            for (N, K), (W, D) in zip(shapes, mats):
                aq, ad = luce.luce_q8_quantize_act(cu(wl.acts(0, T, K)))
                y = torch.empty((T, N), dtype=torch.float32, device="cuda")
                fn = (lambda W=W, D=D, aq=aq, ad=ad, y=y: luce.luce_q8_matvec_batch_path(W, D, aq, ad, a.path, y))
                fns.append(fn)
                for _ in range(a.warmup):
                    fn()
                m = statistics.mean(time_launches(torch, fn, flush, a.reps))
                b = N * K * 34 // 32 + T * K + T * (K // 32) * 4 + T * N * 4
                per.append(round(m * 1e3, 2))
                tot_b += b
                tot_ms += m

            def layer():
                for f in fns:
                    f()
            mb = statistics.mean(time_launches(torch, layer, flush, a.reps))
            print(json.dumps({"kernel": "q8_matvec x4 (27B layer)", "path": a.path, "T": T,
                              "us_alone": per, "us_sum": round(tot_ms * 1e3, 2),
                              "us_back_to_back": round(mb * 1e3, 2), "bytes": tot_b,
                              "gbps_alone": round(tot_b / tot_ms / 1e6, 1), "gbps": round(tot_b / mb / 1e6, 1)}))
    elif a.kernel == "attn":
        lens = [int(x) for x in a.lens.split(",")]
        d = wl.Dims(0, a.hq, a.hkv, 128, 0)
        views = []
        for s, L in enumerate(lens):
            k, v = wl.cache_host(0, s, 0, d, L, L)
            views.append(luce.SeqView(cu(k), cu(v), L, 1, s))
        q = cu(wl.qvec(0, len(lens), a.hq))
        out = torch.empty_like(q)
        ws = torch.empty(luce.luce_decode_attn_workspace_size(len(lens), a.hq, 128, max(lens)), dtype=torch.uint8,
                         device="cuda")
        fn = lambda: luce.luce_decode_attn_multiseq(q, views, a.hkv, 0.08838834764831845, out, ws)
        for _ in range(a.warmup):
            fn()
        ms = time_launches(torch, fn, flush, a.reps)
        b = sum(lens) * a.hkv * 128 * 2 * 2
        m = statistics.mean(ms)
        med = statistics.median(ms)
        print(json.dumps({"kernel": "decode_attn", "lens": lens, "hq": a.hq, "hkv": a.hkv,
                          "us_mean": round(m * 1e3, 2), "us_median": round(med * 1e3, 2),
                          "gbps_median": round(b / med / 1e6, 1)}))
    else:
        d = wl.LAYER27B
        fields = ["attn_norm", "wqkv_q", "wqkv_d", "wo_q", "wo_d", "ffn_norm", "wgu_q", "wgu_d", "wdown_q",
                  "wdown_d"]
        Lh = wl.layer_host(1, 0, d)
        model = luce.Model([luce.LayerTensors(*[cu(getattr(Lh, f)) for f in fields])], d.hidden, d.n_q_heads,
                           d.n_kv_heads, d.ffn)
        slots = []
        cap = 2050 + a.rows
        for s in range(a.nseq):
            k, v = wl.cache_host(1, s, 0, d, cap, 2050)
            slots.append(luce.Slot(cu(k[None]), cu(v[None]), 2050))
        T = a.nseq * a.rows
        x = cu(wl.acts(1, T, d.hidden))
        ws = model.workspace(T, cap)
        fn = lambda: luce.luce_decode_step(model, slots, [a.rows] * a.nseq, x, ws)
        for _ in range(a.warmup):
            fn()
        ms = time_launches(torch, fn, flush, a.reps)
        m = statistics.mean(ms)
        med = statistics.median(ms)
        print(json.dumps({"kernel": "decode_step", "nseq": a.nseq, "rows_per_slot": a.rows,
                          "us_mean": round(m * 1e3, 2), "us_median": round(med * 1e3, 2),
                          "tok_s_median": round(T / (med / 1e3), 1)}))


if __name__ == "__main__":
    main()
