"""GPU parity of the SAPS round through the C ABI: seeded mask + decoupled
look-back compaction (count, indices and gathered values bit-exact), peer
averaging over the seeded perfect matching, and the EASGD elastic step
(floats within rel 1e-5 of the fp64 oracle)."""
import numpy as np
import pytest
import torch

import gradient_compression_sgd_gc_gb300 as gc
from gradient_compression_sgd_gc_gb300 import workloads as wl
import oracle
from gpu_helpers import assert_close, check_guard, guarded, host_f32, host_u32

pytestmark = pytest.mark.gpu
DEV = "cuda"


class Compactor:
    """Device buffers for one saps_mask_compact call."""

    def __init__(self, n, W, capacity):
        self.n, self.W, self.capacity = n, W, capacity
        self.idx = guarded(capacity, torch.int32)
        self.vals = [guarded(capacity, torch.float32) for _ in range(W)]
        self.count = torch.zeros(2, dtype=torch.int64, device=DEV)
        self.ws = torch.empty(gc.saps_workspace_bytes(n), dtype=torch.uint8, device=DEV)
        self.status = torch.zeros(1, dtype=torch.int32, device=DEV)

    def run(self, p, seed_t, models):
        gc.saps_mask_compact(self.n, p, seed_t, models, self.idx[:self.capacity],
                             [v[:self.capacity] for v in self.vals], self.count[:1], self.ws,
                             self.status)

    def result(self):
        torch.cuda.synchronize()
        K = int(self.count[0].item())
        kept = min(K, self.capacity)
        return (K, host_u32(self.idx[:kept]), [host_f32(v[:kept]) for v in self.vals],
                int(self.status.item()))


@pytest.mark.parametrize("n", [1, 100, 4095, 4096, 4097, 3 * 4096 + 5, 1_000_003])
@pytest.mark.parametrize("p", [0.001, 0.01, 0.25, 0.5, 1.0])
def test_mask_compact_parity(n, p):
    """p = 0.25 puts about half the 4096-element tiles above the 1024 entries
    a tile stages for its deferred write (the rest take their prefix at once),
    so both paths alternate in one launch."""
    W = 3
    models = [wl.normal(n, 0.05, 4000 + w, device=DEV) for w in range(W)]
    seed_t = oracle.round_seed(5, n % 7)
    comp = Compactor(n, W, n)
    comp.run(p, seed_t, models)
    K, idx, vals, status = comp.result()
    rK, ridx, rvals = oracle.saps_mask_compact(n, p, seed_t, [host_f32(m).astype(np.float64)
                                                              for m in models])
    assert status == 0
    assert K == rK
    np.testing.assert_array_equal(idx, ridx)
    for w in range(W):
        np.testing.assert_array_equal(vals[w].astype(np.float64), rvals[w])
    check_guard(comp.idx, n)
    for v in comp.vals:
        check_guard(v, n)


def test_mask_compact_sixteen_workers_and_repeat_calls():
    n, W = 300_007, 16
    models = [wl.normal(n, 0.05, 4000 + w, device=DEV) for w in range(W)]
    comp = Compactor(n, W, 6000)
    hm = [host_f32(m).astype(np.float64) for m in models]
    for t in range(3):       # the workspace is reused: every call clears it first
        seed_t = oracle.round_seed(5, t)
        comp.run(0.01, seed_t, models)
        K, idx, vals, status = comp.result()
        rK, ridx, rvals = oracle.saps_mask_compact(n, 0.01, seed_t, hm)
        assert status == 0 and K == rK
        np.testing.assert_array_equal(idx, ridx)
        for w in range(W):
            np.testing.assert_array_equal(vals[w].astype(np.float64), rvals[w])


def test_compaction_under_each_l2_fetch_granularity():
    """The L2 fetch-granularity hint changes what the gather moves, never what
    it returns: the compaction equals the oracle at 32, 64 and 128 bytes, and
    the previous setting comes back."""
    n, W = 300_007, 4
    models = [wl.normal(n, 0.05, 4100 + w, device=DEV) for w in range(W)]
    hm = [host_f32(m).astype(np.float64) for m in models]
    comp = Compactor(n, W, 20_000)
    seed_t = oracle.round_seed(5, 7)
    rK, ridx, rvals = oracle.saps_mask_compact(n, 0.01, seed_t, hm)
    torch.cuda.synchronize()
    first = gc.gc_l2_fetch_granularity(32)
    try:
        for g in (32, 64, 128):
            torch.cuda.synchronize()
            gc.gc_l2_fetch_granularity(g)
            comp.run(0.01, seed_t, models)
            K, idx, vals, status = comp.result()
            assert status == 0 and K == rK
            np.testing.assert_array_equal(idx, ridx)
            for w in range(W):
                np.testing.assert_array_equal(vals[w].astype(np.float64), rvals[w])
    finally:
        torch.cuda.synchronize()
        assert gc.gc_l2_fetch_granularity(first) == 128
    with pytest.raises(gc.GcError, match="GC_ERR_INVALID"):
        gc.gc_l2_fetch_granularity(256)


@pytest.mark.parametrize("p,cap", [(0.1, 100), (0.5, 100), (0.5, 3000), (0.25, 1500)])
def test_capacity_overflow_reports_and_truncates(p, cap):
    """The capacity cut lands inside a staged tile (p = 0.1), inside a dense
    tile written at once (p = 0.5), or where both kinds alternate."""
    n, W = 50_000, 2
    models = [wl.normal(n, 1.0, w, device=DEV) for w in range(W)]
    comp = Compactor(n, W, cap)
    comp.run(p, 99, models)
    K, idx, vals, status = comp.result()
    rK, ridx, rvals = oracle.saps_mask_compact(n, p, 99, [host_f32(m).astype(np.float64) for m in models])
    assert K == rK > cap
    assert status == gc.GC_ERR_CAPACITY
    np.testing.assert_array_equal(idx, ridx[:cap])
    for w in range(W):
        np.testing.assert_array_equal(vals[w].astype(np.float64), rvals[w][:cap])
    check_guard(comp.idx, cap)
    for v in comp.vals:
        check_guard(v, cap)


def test_saps_rounds_chain():
    """Ten full SAPS rounds on 16 workers (mask, compaction, pair average,
    elastic step) against the oracle's fp64 chain.  The fp32 chain's rounding
    errors are bounded by ulps of the largest magnitudes an element has taken
    in any round, so the tolerance scale is that running maximum."""
    n, W, p, alpha, beta = 200_003, 16, 0.01, 0.9, 0.9
    cfg = wl.scaled(wl.SAPS_P01, n)
    models = wl.saps_models(cfg, device=DEV)
    center = wl.saps_initial_center(models)
    ref = [host_f32(m).astype(np.float64) for m in models]
    rc = host_f32(center).astype(np.float64)
    comp = Compactor(n, W, n)
    scale = np.max(np.abs(np.stack(ref)), axis=0) + np.abs(rc)
    for t in range(10):
        seed_t = gc.saps_round_seed(cfg.base_seed, t)
        pairs = gc.saps_matching(seed_t, W)
        comp.run(p, seed_t, models)
        gc.saps_peer_average(models, [v[:n] for v in comp.vals], comp.idx[:n], comp.count[:1], pairs)
        gc.easgd_step(models, alpha, beta, center)
        rK, ridx, rvals = oracle.saps_mask_compact(n, p, seed_t, ref)
        assert pairs == oracle.saps_matching(seed_t, W).tolist()
        oracle.saps_peer_average(ref, rvals, ridx, np.array(pairs, np.int32))
        oracle.easgd_step(ref, alpha, beta, rc)
        torch.cuda.synchronize()
        assert int(comp.count[0].item()) == rK
        scale = np.maximum(scale, np.max(np.abs(np.stack(ref)), axis=0) + np.abs(rc))
        for w in range(W):
            assert_close(host_f32(models[w]), ref[w], scale, what=f"model {w} round {t}")
        assert_close(host_f32(center), rc, scale, what=f"center round {t}")
        assert int(comp.status.item()) == 0


def test_peer_average_is_exact_mean_of_pairs():
    n, W = 40_000, 4
    models = [wl.normal(n, 1.0, 10 + w, device=DEV) for w in range(W)]
    before = [host_f32(m) for m in models]
    comp = Compactor(n, W, n)
    seed_t = 1234
    comp.run(0.2, seed_t, models)
    pairs = gc.saps_matching(seed_t, W)
    gc.saps_peer_average(models, [v[:n] for v in comp.vals], comp.idx[:n], comp.count[:1], pairs)
    K, idx, _, _ = comp.result()
    mask = np.zeros(n, bool)
    mask[idx] = True
    after = [host_f32(m) for m in models]
    for q in range(W // 2):
        a, b = pairs[2 * q], pairs[2 * q + 1]
        mean = ((before[a].astype(np.float64) + before[b]) / 2).astype(np.float32)
        np.testing.assert_array_equal(after[a][mask], mean[mask])
        np.testing.assert_array_equal(after[b][mask], mean[mask])
    for w in range(W):
        np.testing.assert_array_equal(after[w][~mask], before[w][~mask])


@pytest.mark.parametrize("W", [1, 2, 4, 5, 16, 17, 64])
@pytest.mark.parametrize("n", [1, 3, 4, 1001, 65_539])
def test_easgd_step_parity(W, n):
    models = [wl.normal(n, 0.05, 50 + w, device=DEV) for w in range(W)]
    center = wl.normal(n, 0.05, 7, device=DEV)
    ref = [host_f32(m).astype(np.float64) for m in models]
    rc = host_f32(center).astype(np.float64)
    scale = np.max(np.abs(np.stack(ref)), axis=0) + np.abs(rc)
    gc.easgd_step(models, 0.9, 0.5, center)
    oracle.easgd_step(ref, 0.9, 0.5, rc)
    torch.cuda.synchronize()
    for w in range(W):
        assert_close(host_f32(models[w]), ref[w], scale, what=f"model {w}")
    assert_close(host_f32(center), rc, scale, what="center")


@pytest.mark.parametrize("W", [2, 4, 16, 18])
@pytest.mark.parametrize("n,p,cap", [(1, 0.5, None), (33, 0.5, None), (4097, 0.01, None),
                                     (100_003, 0.01, None), (100_003, 0.25, None), (100_003, 0.3, 5000)])
def test_fused_average_easgd_is_bitwise_the_two_calls(W, n, p, cap):
    """saps_average_easgd_step == saps_peer_average then easgd_step, bit for
    bit, including a capacity overflow (entries beyond capacity not averaged)."""
    capacity = cap or n
    base = [wl.normal(n, 0.05, 900 + w, device=DEV) for w in range(W)]
    c0 = wl.saps_initial_center(base)
    ma = [b.clone() for b in base]
    mb = [b.clone() for b in base]
    ca, cb = c0.clone(), c0.clone()
    seed_t = gc.saps_round_seed(11, n)
    pairs = gc.saps_matching(seed_t, W)
    comp = Compactor(n, W, capacity)
    comp.run(p, seed_t, ma)
    vals = [v[:capacity] for v in comp.vals]
    gc.saps_peer_average(ma, vals, comp.idx[:capacity], comp.count[:1], pairs)
    gc.easgd_step(ma, 0.9, 0.7, ca)
    gc.saps_average_easgd_step(mb, vals, comp.count[:1], pairs, 0.9, 0.7, cb, comp.ws)
    torch.cuda.synchronize()
    for w in range(W):
        assert torch.equal(ma[w].view(torch.int32), mb[w].view(torch.int32)), f"worker {w}"
    assert torch.equal(ca.view(torch.int32), cb.view(torch.int32))


def test_saps_rounds_chain_fused():
    """Six SAPS rounds with the fused pair-average + elastic step against the
    oracle's fp64 chain."""
    n, W, p, alpha, beta = 150_011, 16, 0.01, 0.9, 0.9
    cfg = wl.scaled(wl.SAPS_P01, n)
    models = wl.saps_models(cfg, device=DEV)
    center = wl.saps_initial_center(models)
    ref = [host_f32(m).astype(np.float64) for m in models]
    rc = host_f32(center).astype(np.float64)
    comp = Compactor(n, W, n)
    scale = np.max(np.abs(np.stack(ref)), axis=0) + np.abs(rc)
    for t in range(6):
        seed_t = gc.saps_round_seed(cfg.base_seed, t)
        pairs = gc.saps_matching(seed_t, W)
        comp.run(p, seed_t, models)
        gc.saps_average_easgd_step(models, [v[:n] for v in comp.vals], comp.count[:1], pairs, alpha, beta,
                                   center, comp.ws)
        rK, ridx, rvals = oracle.saps_mask_compact(n, p, seed_t, ref)
        oracle.saps_peer_average(ref, rvals, ridx, np.array(pairs, np.int32))
        oracle.easgd_step(ref, alpha, beta, rc)
        torch.cuda.synchronize()
        scale = np.maximum(scale, np.max(np.abs(np.stack(ref)), axis=0) + np.abs(rc))
        for w in range(W):
            assert_close(host_f32(models[w]), ref[w], scale, what=f"model {w} round {t}")
        assert_close(host_f32(center), rc, scale, what=f"center round {t}")


@pytest.mark.parametrize("one_pass", [False, True], ids=["public", "one-pass-kernel"])
@pytest.mark.parametrize("W", [2, 4, 16, 18])
@pytest.mark.parametrize("n,p", [(1, 0.5), (33, 1.0), (4097, 0.01), (100_003, 0.01), (100_003, 0.001),
                                 (3 * 4096 + 5, 0.3), (50_001, 0.9), (40_000, 0.09)])
def test_one_pass_round_is_bitwise_the_three_calls(one_pass, W, n, p):
    """saps_round == saps_mask_compact + saps_peer_average + easgd_step, bit for
    bit: count, idx, vals, models and center.  With the one-pass kernel forced,
    p = 0.09, 0.3 and 0.9 fill a tile's stash (the mid-tile prefix path)."""
    if one_pass and W > 16:
        pytest.skip("the one-pass kernel takes W <= 16")
    base = [wl.normal(n, 0.05, 700 + w, device=DEV) for w in range(W)]
    c0 = wl.saps_initial_center(base)
    ma = [b.clone() for b in base]
    mb = [b.clone() for b in base]
    ca, cb = c0.clone(), c0.clone()
    seed_t = gc.saps_round_seed(13, n + W)
    pairs = gc.saps_matching(seed_t, W)
    comp = Compactor(n, W, n)
    comp.run(p, seed_t, ma)
    gc.saps_peer_average(ma, [v[:n] for v in comp.vals], comp.idx[:n], comp.count[:1], pairs)
    gc.easgd_step(ma, 0.9, 0.6, ca)
    K, idx, vals, st = comp.result()
    r = Compactor(n, W, n)
    gc.saps_round(n, p, seed_t, mb, pairs, 0.9, 0.6, cb, r.idx[:n], [v[:n] for v in r.vals], r.count[:1],
                  r.ws, r.status, _one_pass=one_pass)
    K2, idx2, vals2, st2 = r.result()
    assert (K2, st2) == (K, st) == (K, 0)
    np.testing.assert_array_equal(idx2, idx)
    for w in range(W):
        np.testing.assert_array_equal(vals2[w].view(np.uint32), vals[w].view(np.uint32))
        assert torch.equal(ma[w].view(torch.int32), mb[w].view(torch.int32)), f"worker {w}"
    assert torch.equal(ca.view(torch.int32), cb.view(torch.int32))
    check_guard(r.idx, n)
    for v in r.vals:
        check_guard(v, n)


@pytest.mark.parametrize("p", [0.05, 0.2])
def test_one_pass_round_capacity_overflow(p):
    """More masked entries than capacity: GC_ERR_CAPACITY, the true count, and
    the first `capacity` entries of idx/vals as the compaction writes them."""
    n, W, cap = 60_000, 4, 1000
    base = [wl.normal(n, 0.05, 300 + w, device=DEV) for w in range(W)]
    seed_t = gc.saps_round_seed(2, 9)
    pairs = gc.saps_matching(seed_t, W)
    comp = Compactor(n, W, cap)
    comp.run(p, seed_t, [b.clone() for b in base])
    K, idx, vals, st = comp.result()
    r = Compactor(n, W, cap)
    center = wl.saps_initial_center(base)
    gc.saps_round(n, p, seed_t, [b.clone() for b in base], pairs, 0.9, 0.9, center, r.idx[:cap],
                  [v[:cap] for v in r.vals], r.count[:1], r.ws, r.status, _one_pass=True)
    K2, idx2, vals2, st2 = r.result()
    assert K2 == K > cap and st2 == gc.GC_ERR_CAPACITY
    np.testing.assert_array_equal(idx2, idx)
    for w in range(W):
        np.testing.assert_array_equal(vals2[w].view(np.uint32), vals[w].view(np.uint32))
    check_guard(r.idx, cap)


def test_one_pass_rounds_chain_against_oracle():
    """Six rounds of saps_round on 16 workers against the oracle's fp64 chain."""
    n, W, p, alpha, beta = 150_011, 16, 0.01, 0.9, 0.9
    cfg = wl.scaled(wl.SAPS_P01, n)
    models = wl.saps_models(cfg, device=DEV)
    center = wl.saps_initial_center(models)
    ref = [host_f32(m).astype(np.float64) for m in models]
    rc = host_f32(center).astype(np.float64)
    r = Compactor(n, W, n)
    scale = np.max(np.abs(np.stack(ref)), axis=0) + np.abs(rc)
    for t in range(6):
        seed_t = gc.saps_round_seed(cfg.base_seed, t)
        pairs = gc.saps_matching(seed_t, W)
        gc.saps_round(n, p, seed_t, models, pairs, alpha, beta, center, r.idx[:n], [v[:n] for v in r.vals],
                      r.count[:1], r.ws, r.status)
        rK, ridx, rvals = oracle.saps_mask_compact(n, p, seed_t, ref)
        oracle.saps_peer_average(ref, rvals, ridx, np.array(pairs, np.int32))
        oracle.easgd_step(ref, alpha, beta, rc)
        K, idx, vals, st = r.result()
        assert K == rK and st == 0
        np.testing.assert_array_equal(idx, ridx)
        scale = np.maximum(scale, np.max(np.abs(np.stack(ref)), axis=0) + np.abs(rc))
        for w in range(W):
            assert_close(host_f32(models[w]), ref[w], scale, what=f"model {w} round {t}")
        assert_close(host_f32(center), rc, scale, what=f"center round {t}")
