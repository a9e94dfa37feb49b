"""GPU side of the multi-process exchange: the two per-rank kernels against
the oracle, and the exchange classes on a world-size-1 NCCL group through the
library's kernels (the collectives degenerate to copies on one GPU; the
multi-rank exchange itself is covered over gloo in test_dist_exchange.py)."""
import numpy as np
import pytest
import torch

import gradient_compression_sgd_gc_gb300 as gc
from gradient_compression_sgd_gc_gb300 import workloads as wl
import oracle
from gpu_helpers import assert_close, check_guard, guarded, host_f32

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.mark.parametrize("n,p", [(1, 1.0), (4097, 0.3), (1_000_003, 0.01)])
def test_pair_average_remote_equals_the_pair_average(n, p):
    """Worker a's side of a pair whose partner b is another process: its
    model gets fl(fl(mine + peer) * 0.5) at the masked coordinates, the value
    saps_peer_average writes for the pair (a, b), and nothing else changes."""
    models = [wl.normal(n, 0.05, 700 + k, device=DEV) for k in range(2)]
    seed_t = gc.saps_round_seed(3, 1)
    cap = n
    idx = torch.empty(cap, dtype=torch.int32, device=DEV)
    vals = [torch.empty(cap, device=DEV) for _ in range(2)]
    cnt = torch.zeros(1, dtype=torch.int64, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    ws = torch.empty(gc.saps_workspace_bytes(n), dtype=torch.uint8, device=DEV)
    gc.saps_mask_compact(n, p, seed_t, models, idx, vals, cnt, ws, st)
    ref = [m.clone() for m in models]
    gc.saps_peer_average(ref, vals, idx, cnt, [0, 1])
    a = guarded(n, torch.float32)
    a[:n].copy_(models[0])
    gc.saps_pair_average_remote(a[:n], idx, cnt, vals[0], vals[1])
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(a[:n].view(torch.int32), ref[0].view(torch.int32))
    check_guard(a, n)
    # against the oracle too
    hm = [host_f32(m).astype(np.float64) for m in models]
    K, ridx, rvals = oracle.saps_mask_compact(n, p, seed_t, hm)
    oracle.saps_peer_average(hm, rvals, ridx, np.array([0, 1], np.int32))
    assert_close(host_f32(a[:n]), hm[0], np.abs(hm[0]), what="pair average")


@pytest.mark.parametrize("n,W", [(3, 2), (4099, 4), (1_000_003, 16)])
def test_easgd_from_sum_against_oracle(n, W):
    """Given the sum of all W models, each worker's elastic step and the
    center equal the all-worker EASGD step (the oracle's, within the float
    tolerance; the sum here is formed in worker order as the all-worker
    kernel does, so the GPU results are bit-identical to easgd_step too)."""
    models = [wl.normal(n, 0.05, 800 + k, device=DEV) for k in range(W)]
    center = wl.normal(n, 0.05, 899, device=DEV)
    total = models[0].clone()
    for k in range(1, W):
        total = total + models[k]
    ref_m = [m.clone() for m in models]
    ref_c = center.clone()
    gc.easgd_step(ref_m, 0.9, 0.9, ref_c)
    hm = [host_f32(m).astype(np.float64) for m in models]
    hc = host_f32(center).astype(np.float64)
    # the terms of w - alpha (w - c): w, alpha w, alpha c; and of
    # c + beta (sum / W - c): c, beta |w_k| / W summed, beta c
    scale = [np.abs(m) + 0.9 * (np.abs(m) + np.abs(hc)) for m in hm]
    cscale = np.abs(hc) + 0.9 * (sum(np.abs(m) for m in hm) / W + np.abs(hc))
    oracle.easgd_step(hm, 0.9, 0.9, hc)
    for k in range(W):
        m, c = models[k].clone(), center.clone()
        gc.easgd_step_from_sum(m, total, W, 0.9, 0.9, c)
        torch.cuda.synchronize()
        assert torch.equal(m.view(torch.int32), ref_m[k].view(torch.int32))
        assert torch.equal(c.view(torch.int32), ref_c.view(torch.int32))
        assert_close(host_f32(m), hm[k], scale[k], what="model")
    assert_close(host_f32(ref_c), hc, cscale, what="center")


@pytest.fixture
def nccl_group():
    import torch.distributed as dist
    if not dist.is_nccl_available():
        pytest.skip("NCCL not available")
    store = dist.HashStore()
    dist.init_process_group("nccl", store=store, rank=0, world_size=1, device_id=torch.device("cuda", 0))
    yield dist.group.WORLD
    dist.destroy_process_group()


def test_exchange_world_one_nccl_equals_direct_calls(nccl_group):
    """TwoBitExchange and QSGDExchange on a one-rank NCCL group run the real
    kernels around NCCL collectives; the results equal the direct calls."""
    from gradient_compression_sgd_gc_gb300 import dist as gdist
    n, t = 100_003, 2e-3
    g = wl.normal(n, 1e-3, 901, device=DEV)
    r1, r2 = torch.zeros(n, device=DEV), torch.zeros(n, device=DEV)
    w1 = wl.uniform(n, 0.05, 7, device=DEV)
    w2 = w1.clone()
    ex = gdist.TwoBitExchange(n, t, DEV)
    ex.step(g, r1, weights=w1, lr=0.1)
    codes = torch.empty(gc.code_words(n), dtype=torch.int32, device=DEV)
    gc.gc_2bit_quantize(g, r2, codes, t)
    gc.gc_2bit_dequant_sum_update([codes], n, t, gc.GC_UPD_SGD, lr=0.1, weights=w2)
    torch.cuda.synchronize()
    assert torch.equal(ex.gathered[0], codes)
    assert torch.equal(w1.view(torch.int32), w2.view(torch.int32))
    assert torch.equal(r1.view(torch.int32), r2.view(torch.int32))

    d, s = 512, 127
    v = wl.qsgd_grad(wl.scaled(wl.QSGD_S127, n), 0, device=DEV)
    q = gdist.QSGDExchange(n, d, s, 42, DEV)
    o1 = torch.empty(n, device=DEV)
    q.step(v, o1)
    nm = torch.empty(gc.qsgd_num_buckets(n, d), device=DEV)
    cd = torch.empty(gc.qsgd_code_bytes(n, s), dtype=torch.uint8, device=DEV)
    gc.qsgd_quantize(v, d, s, 42, 0, nm, cd)
    o2 = torch.empty(n, device=DEV)
    gc.qsgd_dequant_sum([cd], [nm], n, d, s, 1.0, o2)
    torch.cuda.synchronize()
    assert torch.equal(o1.view(torch.int32), o2.view(torch.int32))
