"""Seeded random configurations of every kernel against the oracle.

Each case draws its sizes and parameters from a fixed seed (sizes up to a
few hundred thousand elements, ragged tails, every bucket size, s from 1 to
127, worker counts, mask densities), so that combinations the hand-picked
parity cases miss still meet the same bar: integer outputs bit-exact, floats
within the float tolerance, QSGD levels equal except at rounding boundaries.
"""
import numpy as np
import pytest
import torch

import gradient_compression_sgd_gc_gb300 as gc
from gradient_compression_sgd_gc_gb300 import workloads as wl
import oracle
from gpu_helpers import (assert_close, check_guard, compare_codes, guarded, host_bf16_bits, host_f32,
                         host_u32, qsgd_sum_reference)

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _rng(case, salt):
    return np.random.default_rng(1000 * salt + case)


@pytest.mark.parametrize("case", range(12))
def test_twobit_quantize_and_dequant_random(case):
    rng = _rng(case, 1)
    n = int(rng.integers(1, 200_000))
    W = int(rng.integers(1, 10))
    t = float(10 ** rng.uniform(-4, -1))
    bf16 = bool(rng.integers(0, 2))
    dt = torch.bfloat16 if bf16 else torch.float32
    scale = float(10 ** rng.uniform(-4, -1))
    grads = [wl.normal(n, scale, 5000 + 31 * case + w, device=DEV, dtype=dt) for w in range(W)]
    res = [wl.normal(n, t, 6000 + 31 * case + w, device=DEV) for w in range(W)]
    r_ref = [host_f32(r).copy() for r in res]
    codes = [guarded(gc.code_words(n), torch.int32) for _ in range(W)]
    gc.gc_2bit_quantize_batched(grads, res, [c[:gc.code_words(n)] for c in codes], t)
    w0 = wl.uniform(n, 0.05, 7000 + case, device=DEV)
    w_ref = host_f32(w0).astype(np.float64)
    lr = float(rng.uniform(0.01, 1.0))
    gc.gc_2bit_dequant_sum_update([c[:gc.code_words(n)] for c in codes], n, t, gc.GC_UPD_SGD, lr=lr, weights=w0)
    torch.cuda.synchronize()
    c_ref = []
    for w in range(W):
        g = host_bf16_bits(grads[w]) if bf16 else host_f32(grads[w])
        c_ref.append(oracle.twobit_quantize(g, r_ref[w], t))
        np.testing.assert_array_equal(host_u32(codes[w][:gc.code_words(n)]), c_ref[w])
        np.testing.assert_array_equal(host_f32(res[w]).view(np.uint32), r_ref[w].view(np.uint32))
        check_guard(codes[w], gc.code_words(n))
    sc = np.abs(w_ref) + lr * t
    oracle.twobit_dequant_sum_update(c_ref, n, t, oracle.KIND_SGD, lr=lr, weights=w_ref)
    assert_close(host_f32(w0), w_ref, sc, what="weights")


@pytest.mark.parametrize("case", range(12))
def test_qsgd_random(case):
    rng = _rng(case, 2)
    d = int(rng.choice([128, 256, 512, 1024, 2048]))
    n = int(rng.integers(1, 150_000))
    s = int(rng.integers(1, 128))
    W = int(rng.integers(1, 6))
    seed = int(rng.integers(0, 2 ** 63))
    cfg = wl.scaled(wl.QSGD_S7, n, seed=int(rng.integers(0, 10_000)))
    vs = [wl.qsgd_grad(cfg, w, device=DEV) for w in range(W)]
    nb, cb = gc.qsgd_num_buckets(n, d), gc.qsgd_code_bytes(n, s)
    norms = [torch.empty(nb, device=DEV) for _ in range(W)]
    codes = [guarded(cb, torch.uint8) for _ in range(W)]
    out = torch.empty(n, device=DEV)
    gc.qsgd_step(vs, d, s, seed, norms, [c[:cb] for c in codes], 1.0 / W, out)
    torch.cuda.synchronize()
    rcs, rns = [], []
    for w in range(W):
        vh = host_f32(vs[w])
        rn, rc = oracle.qsgd_quantize(vh, d, s, seed, w)
        assert_close(host_f32(norms[w]), rn, np.abs(rn), what="norms")
        compare_codes(codes[w][:cb].cpu().numpy(), rc, vh, n, d, s, seed, w)
        check_guard(codes[w], cb)
        rcs.append(rc)
        rns.append(rn)
    ref, terms = qsgd_sum_reference([c[:cb].cpu().numpy() for c in codes], [host_f32(x) for x in norms],
                                    n, d, s, 1.0 / W)
    assert_close(host_f32(out), ref, terms, what="average")
    # the Elias stream of worker 0's codes (oracle codes in, so the stream is
    # compared word for word)
    ref_w, ref_off = oracle.qsgd_elias_encode(rcs[0], rns[0], n, d, s)
    words = torch.empty(gc.qsgd_elias_max_words(n, d, s), dtype=torch.int32, device=DEV)
    offs = torch.empty(nb + 1, dtype=torch.int32, device=DEV)
    ws = torch.empty(gc.qsgd_elias_workspace_bytes(n, d), dtype=torch.uint8, device=DEV)
    gc.qsgd_elias_encode(torch.from_numpy(rcs[0]).to(DEV), torch.from_numpy(rns[0]).to(DEV), n, d, s,
                         words, offs, ws)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(host_u32(offs), ref_off)
    np.testing.assert_array_equal(host_u32(words[:ref_w.size]), ref_w)


@pytest.mark.parametrize("case", range(10))
def test_saps_round_random(case):
    rng = _rng(case, 3)
    n = int(rng.integers(1, 120_000))
    W = int(rng.choice([2, 4, 6, 8, 16]))
    p = float(rng.choice([0.001, 0.01, 0.05, 0.2, 1.0]))
    alpha, beta = float(rng.uniform(0.1, 1.0)), float(rng.uniform(0.1, 1.0))
    models = [wl.normal(n, 0.05, 8000 + 37 * case + w, device=DEV) for w in range(W)]
    center = wl.saps_initial_center(models)
    ref = [host_f32(m).astype(np.float64) for m in models]
    rc = host_f32(center).astype(np.float64)
    scale = np.max(np.abs(np.stack(ref)), axis=0) + np.abs(rc)
    seed_t = gc.saps_round_seed(int(rng.integers(0, 2 ** 32)), case)
    pairs = gc.saps_matching(seed_t, W)
    idx = guarded(n, torch.int32)
    vals = [guarded(n, torch.float32) for _ in range(W)]
    cnt = torch.zeros(1, dtype=torch.int64, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    ws = torch.empty(gc.saps_workspace_bytes(n), dtype=torch.uint8, device=DEV)
    gc.saps_round(n, p, seed_t, models, pairs, alpha, beta, center, idx[:n], [v[:n] for v in vals], cnt, ws, st)
    torch.cuda.synchronize()
    K, ridx, rvals = oracle.saps_mask_compact(n, p, seed_t, ref)
    assert int(cnt.item()) == K and int(st.item()) == 0
    np.testing.assert_array_equal(host_u32(idx[:K]), ridx)
    for w in range(W):
        # the gathered values are the pre-round fp32 models: exact
        np.testing.assert_array_equal(host_f32(vals[w][:K]).astype(np.float64), rvals[w])
        check_guard(vals[w], n)
    oracle.saps_peer_average(ref, rvals, ridx, np.array(pairs, np.int32))
    oracle.easgd_step(ref, alpha, beta, rc)
    for w in range(W):
        assert_close(host_f32(models[w]), ref[w], scale, what=f"model {w}")
    assert_close(host_f32(center), rc, scale, what="center")
    check_guard(idx, n)
