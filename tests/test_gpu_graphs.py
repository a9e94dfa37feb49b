"""The C-ABI calls inside CUDA graphs: a captured sequence replays to the
same bits as the same calls made eagerly (every entry point only enqueues
kernels and memsets on the caller's stream, so it can be captured)."""
import numpy as np
import pytest
import torch

import gradient_compression_sgd_gc_gb300 as gc
from gradient_compression_sgd_gc_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _replay_equals_eager(make_state, run):
    """run(state) enqueues the calls; the graph's replay and an eager run from
    the same starting state must leave identical buffers."""
    eager = make_state()
    run(eager)
    torch.cuda.synchronize()
    graphed = make_state()
    start = [t.clone() for t in graphed]
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        run(graphed)                      # warm-up on a side stream (loads the library, no capture)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    for t, s0 in zip(graphed, start):
        t.copy_(s0)
    with torch.cuda.graph(g):
        run(graphed)
    for t, s0 in zip(graphed, start):     # capture does not execute: reset and replay
        t.copy_(s0)
    g.replay()
    torch.cuda.synchronize()
    for a, b in zip(eager, graphed):
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))


def test_twobit_steps_in_a_graph():
    n, W, t, lr, steps = 100_003, 4, 2e-3, 0.1, 3
    grads = [[wl.normal(n, 1e-3, 100 * s + w, device=DEV) for w in range(W)] for s in range(steps)]

    def make():
        res = [torch.zeros(n, device=DEV) for _ in range(W)]
        codes = [torch.zeros(gc.code_words(n), dtype=torch.int32, device=DEV) for _ in range(W)]
        return res + codes + [wl.uniform(n, 0.05, 7, device=DEV)]

    def run(st):
        res, codes, wt = st[:W], st[W:2 * W], st[2 * W]
        for s in range(steps):
            gc.gc_2bit_quantize_batched(grads[s], res, codes, t)
            gc.gc_2bit_dequant_sum_update(codes, n, t, gc.GC_UPD_SGD, lr=lr, weights=wt)

    _replay_equals_eager(make, run)


def test_qsgd_step_elias_and_dequant_in_a_graph():
    n, W, d, s = 70_001, 3, 512, 127
    cfg = wl.scaled(wl.QSGD_S127, n)
    vs = [wl.qsgd_grad(cfg, w, device=DEV) for w in range(W)]
    nb, cb = gc.qsgd_num_buckets(n, d), gc.qsgd_code_bytes(n, s)
    cap = gc.qsgd_elias_max_words(n, d, s)

    def make():
        return ([torch.zeros(nb, device=DEV) for _ in range(W)]
                + [torch.zeros(cb, dtype=torch.uint8, device=DEV) for _ in range(W)]
                + [torch.zeros(n, device=DEV), torch.zeros(cap, dtype=torch.int32, device=DEV),
                   torch.zeros(nb + 1, dtype=torch.int32, device=DEV),
                   torch.zeros(gc.qsgd_elias_workspace_bytes(n, d), dtype=torch.uint8, device=DEV),
                   torch.zeros(cb, dtype=torch.uint8, device=DEV), torch.zeros(nb, device=DEV),
                   torch.zeros(n, device=DEV)])

    def run(st):
        norms, codes = st[:W], st[W:2 * W]
        out, words, offs, ws, dc, dn, total = st[2 * W:]
        gc.qsgd_step(vs, d, s, 9, norms, codes, 1.0 / W, out)
        gc.qsgd_elias_encode(codes[0], norms[0], n, d, s, words, offs, ws)
        gc.qsgd_elias_decode(words, offs, n, d, s, dc, dn)
        gc.qsgd_dequant_sum(codes, norms, n, d, s, 1.0, total)

    _replay_equals_eager(make, run)


def test_saps_rounds_in_a_graph():
    n, W, p = 60_001, 8, 0.01
    base = [wl.normal(n, 0.05, 40 + w, device=DEV) for w in range(W)]
    c0 = wl.saps_initial_center(base)
    seeds = [gc.saps_round_seed(3, r) for r in range(3)]
    pairs = [gc.saps_matching(sd, W) for sd in seeds]

    def make():
        return ([b.clone() for b in base] + [c0.clone(), torch.zeros(n, dtype=torch.int32, device=DEV)]
                + [torch.zeros(n, device=DEV) for _ in range(W)]
                + [torch.zeros(1, dtype=torch.int64, device=DEV),
                   torch.zeros(gc.saps_workspace_bytes(n), dtype=torch.uint8, device=DEV),
                   torch.zeros(1, dtype=torch.int32, device=DEV)])

    def run(st):
        models, center, idx = st[:W], st[W], st[W + 1]
        vals = st[W + 2:2 * W + 2]
        cnt, ws, status = st[2 * W + 2:]
        for r in range(3):
            gc.saps_round(n, p, seeds[r], models, pairs[r], 0.9, 0.9, center, idx, vals, cnt, ws, status)

    _replay_equals_eager(make, run)
