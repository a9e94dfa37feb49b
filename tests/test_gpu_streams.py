"""Entry points on several CUDA streams at once: the library keeps no state
between calls (every buffer, the compaction's look-back workspace included,
belongs to the caller), so independent calls may overlap on the GPU.  Two
copies of each workload run concurrently on separate streams and must equal
the same calls run one after another on the default stream."""
import pytest
import torch

import gradient_compression_sgd_gc_gb300 as gc
from gradient_compression_sgd_gc_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _twobit(state, grads, stream=None):
    res, codes, w = state
    gc.gc_2bit_quantize_batched(grads, res, codes, 2e-3, stream=stream)
    gc.gc_2bit_dequant_sum_update(codes, w.numel(), 2e-3, gc.GC_UPD_SGD, lr=0.1, weights=w, stream=stream)


def _saps(state, seed_t, stream=None):
    models, center, idx, vals, cnt, ws, st = state
    pairs = gc.saps_matching(seed_t, len(models))
    gc.saps_mask_compact(center.numel(), 0.01, seed_t, models, idx, vals, cnt, ws, st, stream=stream)
    gc.saps_average_easgd_step(models, vals, cnt, pairs, 0.9, 0.9, center, ws, stream=stream)


def _qsgd(state, vs, stream=None):
    norms, codes, out = state
    gc.qsgd_step(vs, 512, 7, 3, norms, codes, 0.25, out, stream=stream)


def test_independent_calls_overlap_on_streams():
    n = 300_007
    W = 4
    grads = [[wl.normal(n, 1e-3, 50 * c + w, device=DEV) for w in range(W)] for c in range(2)]
    qv = [[wl.qsgd_grad(wl.scaled(wl.QSGD_S7, n), 10 * c + w, device=DEV) for w in range(W)] for c in range(2)]
    base = [[wl.normal(n, 0.05, 600 + 30 * c + w, device=DEV) for w in range(W)] for c in range(2)]

    def fresh(c):
        tb = ([torch.zeros(n, device=DEV) for _ in range(W)],
              [torch.zeros(gc.code_words(n), dtype=torch.int32, device=DEV) for _ in range(W)],
              wl.uniform(n, 0.05, 70 + c, device=DEV))
        cap = n // 50
        sp = ([b.clone() for b in base[c]], wl.saps_initial_center(base[c]),
              torch.zeros(cap, dtype=torch.int32, device=DEV), [torch.zeros(cap, device=DEV) for _ in range(W)],
              torch.zeros(1, dtype=torch.int64, device=DEV),
              torch.zeros(gc.saps_workspace_bytes(n), dtype=torch.uint8, device=DEV),
              torch.zeros(1, dtype=torch.int32, device=DEV))
        nb, cb = gc.qsgd_num_buckets(n, 512), gc.qsgd_code_bytes(n, 7)
        qs = ([torch.zeros(nb, device=DEV) for _ in range(W)],
              [torch.zeros(cb, dtype=torch.uint8, device=DEV) for _ in range(W)], torch.zeros(n, device=DEV))
        return tb, sp, qs

    def flat(st):
        tb, sp, qs = st
        return (tb[0] + tb[1] + [tb[2]] + sp[0] + [sp[1], sp[2]] + sp[3] + [sp[4], sp[6]]
                + qs[0] + qs[1] + [qs[2]])

    seq = [fresh(c) for c in range(2)]
    for c in range(2):
        for step in range(3):
            _twobit(seq[c][0], grads[c])
            _saps(seq[c][1], gc.saps_round_seed(9 + c, step))
            _qsgd(seq[c][2], qv[c])
    torch.cuda.synchronize()

    par = [fresh(c) for c in range(2)]
    torch.cuda.synchronize()
    streams = [[torch.cuda.Stream() for _ in range(3)] for _ in range(2)]
    for step in range(3):
        for c in range(2):
            _twobit(par[c][0], grads[c], streams[c][0])
            _saps(par[c][1], gc.saps_round_seed(9 + c, step), streams[c][1])
            _qsgd(par[c][2], qv[c], streams[c][2])
    torch.cuda.synchronize()
    for c in range(2):
        for a, b in zip(flat(seq[c]), flat(par[c])):
            assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))
