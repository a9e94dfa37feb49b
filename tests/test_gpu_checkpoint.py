"""Checkpoint / resume: all state of the compression path lives in
caller-owned buffers (residuals, weights, the EASGD center), so saving them to
host memory and restoring them into fresh device buffers resumes the run
bit-for-bit: 10 steps straight == 5 steps + save/restore + 5 steps."""
import numpy as np
import pytest
import torch

import gradient_compression_sgd_gc_gb300 as gc
from gradient_compression_sgd_gc_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _twobit_run(state, steps, first_step, n, W, cfg):
    res, w = state
    codes = [torch.empty(gc.code_words(n), dtype=torch.int32, device=DEV) for _ in range(W)]
    for step in range(first_step, first_step + steps):
        grads = [wl.normal(n, cfg.grad_std, cfg.grad_seed(step, q), device=DEV) for q in range(W)]
        gc.gc_2bit_quantize_batched(grads, res, codes, cfg.threshold)
        gc.gc_2bit_dequant_sum_update(codes, n, cfg.threshold, gc.GC_UPD_SGD, lr=cfg.lr, weights=w)
    return res, w


def test_twobit_resume_is_bitwise():
    cfg = wl.scaled(wl.TWOBIT_DQ_SGD, 200_003)
    n, W = cfg.n, cfg.workers
    fresh = lambda: ([torch.zeros(n, device=DEV) for _ in range(W)], wl.twobit_weights(cfg, device=DEV))
    a = _twobit_run(fresh(), 10, 0, n, W, cfg)
    b = _twobit_run(fresh(), 5, 0, n, W, cfg)
    torch.cuda.synchronize()
    saved = ([r.cpu().numpy().copy() for r in b[0]], b[1].cpu().numpy().copy())
    del b
    restored = ([torch.from_numpy(r).to(DEV) for r in saved[0]], torch.from_numpy(saved[1]).to(DEV))
    b = _twobit_run(restored, 5, 5, n, W, cfg)
    torch.cuda.synchronize()
    for q in range(W):
        assert torch.equal(a[0][q].view(torch.int32), b[0][q].view(torch.int32))
    assert torch.equal(a[1].view(torch.int32), b[1].view(torch.int32))


def test_saps_resume_is_bitwise():
    cfg = wl.scaled(wl.SAPS_P01, 100_003)
    n, W = cfg.n, cfg.workers

    def run(models, center, first, rounds):
        idx = torch.empty(n, dtype=torch.int32, device=DEV)
        vals = [torch.empty(n, device=DEV) for _ in range(W)]
        cnt = torch.zeros(1, dtype=torch.int64, device=DEV)
        ws = torch.empty(gc.saps_workspace_bytes(n), dtype=torch.uint8, device=DEV)
        st = torch.zeros(1, dtype=torch.int32, device=DEV)
        for t in range(first, first + rounds):
            seed_t = gc.saps_round_seed(cfg.base_seed, t)
            gc.saps_mask_compact(n, cfg.p, seed_t, models, idx, vals, cnt, ws, st)
            gc.saps_average_easgd_step(models, vals, cnt, gc.saps_matching(seed_t, W), cfg.alpha, cfg.beta,
                                       center, ws)
        return models, center

    m0 = wl.saps_models(cfg, device=DEV)
    c0 = wl.saps_initial_center(m0)
    a = run([m.clone() for m in m0], c0.clone(), 0, 10)
    b = run([m.clone() for m in m0], c0.clone(), 0, 5)
    torch.cuda.synchronize()
    saved = ([m.cpu().numpy().copy() for m in b[0]], b[1].cpu().numpy().copy())
    b = run([torch.from_numpy(m).to(DEV) for m in saved[0]], torch.from_numpy(saved[1]).to(DEV), 5, 5)
    torch.cuda.synchronize()
    for q in range(W):
        assert torch.equal(a[0][q].view(torch.int32), b[0][q].view(torch.int32))
    assert torch.equal(a[1].view(torch.int32), b[1].view(torch.int32))
