"""The key-value compression front end: parameter rules of "2bit gradient
compression" (MXNet PR #8662, "Usage": a dict {'type', 'threshold'}; no
default threshold; switching compression off after use is an error) on the
host, and on the GPU its calls against the oracle."""
import numpy as np
import pytest
import torch

from gradient_compression_sgd_gc_gb300.compression import GradientCompression
import gradient_compression_sgd_gc_gb300 as gc
from gradient_compression_sgd_gc_gb300 import workloads as wl
import oracle


def test_params_rules():
    with pytest.raises(ValueError):
        GradientCompression({"type": "2bit"})                      # no default threshold
    with pytest.raises(ValueError):
        GradientCompression({"type": "2bit", "threshold": 0.0})
    with pytest.raises(ValueError):
        GradientCompression({"type": "2bit", "threshold": float("nan")})
    with pytest.raises(ValueError):
        GradientCompression({"type": "1bit", "threshold": 0.5})
    with pytest.raises(ValueError):
        GradientCompression({"type": "2bit", "threshold": 0.5, "bits": 2})
    with pytest.raises(TypeError):
        GradientCompression("2bit")
    c = GradientCompression({"type": "2bit", "threshold": 0.5})
    assert c.params == {"type": "2bit", "threshold": 0.5}
    c.set_params({"type": "2bit", "threshold": 0.25})             # allowed at any time
    assert c.threshold == 0.25
    c.set_params({"type": "none"})                                 # never used yet: allowed
    assert c.params == {"type": "none"}
    g = torch.ones(3)
    assert c.compress("w", g) is g                                 # untouched
    with pytest.raises(ValueError):
        c.decompress([g], 3)


@pytest.mark.gpu
def test_keys_against_oracle_and_no_switch_off_after_use():
    dev = "cuda"
    n, W, t, lr = 70_001, 3, 2e-3, 0.1
    comp = GradientCompression({"type": "2bit", "threshold": t})
    grads = [wl.normal(n, 1e-3, 300 + w, device=dev) for w in range(W)]
    codes = [comp.compress(("layer0", w), grads[w]) for w in range(W)]
    avg = comp.decompress(codes, n)
    weights = wl.uniform(n, 0.05, 3, device=dev)
    w_ref = weights.cpu().numpy().astype(np.float64)
    comp.apply(codes, weights, lr)
    torch.cuda.synchronize()
    r_ref = [np.zeros(n, np.float32) for _ in range(W)]
    c_ref = [oracle.twobit_quantize(grads[w].cpu().numpy(), r_ref[w], t) for w in range(W)]
    for w in range(W):
        np.testing.assert_array_equal(codes[w].cpu().numpy().view(np.uint32), c_ref[w])
        np.testing.assert_array_equal(comp.residual(("layer0", w)).cpu().numpy().view(np.uint32),
                                      r_ref[w].view(np.uint32))
    a_ref = oracle.twobit_dequant_sum_update(c_ref, n, t, oracle.KIND_NONE)
    np.testing.assert_allclose(avg.cpu().numpy(), a_ref, rtol=0, atol=1e-5 * t)
    oracle.twobit_dequant_sum_update(c_ref, n, t, oracle.KIND_SGD, lr=lr, weights=w_ref)
    np.testing.assert_allclose(weights.cpu().numpy(), w_ref, rtol=1e-5, atol=1e-5 * lr * t)
    with pytest.raises(ValueError):
        comp.set_params({"type": "none"})
    # the fused step keeps the same per-key residuals
    weights2 = wl.uniform(n, 0.05, 4, device=dev)
    comp.step([("layer0", w) for w in range(W)], grads, weights2, lr)
    torch.cuda.synchronize()
    c2 = [oracle.twobit_quantize(grads[w].cpu().numpy(), r_ref[w], t) for w in range(W)]
    for w in range(W):
        np.testing.assert_array_equal(comp.residual(("layer0", w)).cpu().numpy().view(np.uint32),
                                      r_ref[w].view(np.uint32))


@pytest.mark.gpu
def test_qsgd_front_end_round_trip():
    from gradient_compression_sgd_gc_gb300.compression import QSGD
    dev = "cuda"
    n, W = 100_003, 3
    q = QSGD(n, W, bucket=512, s=22, seed=5)
    cfg = wl.scaled(wl.QSGD_S127, n)
    grads = [wl.qsgd_grad(cfg, w, device=dev) for w in range(W)]
    out = torch.empty(n, device=dev)
    q.step(grads, out)
    n1 = [x.clone() for x in q.norms]
    c1 = [x.clone() for x in q.codes]
    words, offsets = q.encode(1)
    q.codes[1].zero_()
    q.norms[1].zero_()
    q.decode(words, offsets, 1)
    torch.cuda.synchronize()
    assert torch.equal(q.norms[1], n1[1])
    lv = lambda c: c & 127
    assert torch.equal(lv(q.codes[1]), lv(c1[1]))
    ref = torch.empty(n, device=dev)
    gc.qsgd_dequant_sum(c1, n1, n, 512, 22, 1.0 / W, ref)
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
    # every worker's stream decoded in one launch
    streams = [q.encode(w) for w in range(W)]
    for x in q.codes + q.norms:
        x.zero_()
    q.decode_all(streams)
    torch.cuda.synchronize()
    for w in range(W):
        assert torch.equal(q.norms[w], n1[w])
        assert torch.equal(lv(q.codes[w]), lv(c1[w]))


@pytest.mark.gpu
def test_saps_front_end_rounds_equal_the_calls():
    from gradient_compression_sgd_gc_gb300.compression import SAPSGossip
    dev = "cuda"
    n, W, p = 60_001, 4, 0.01
    base = [wl.normal(n, 0.05, 70 + w, device=dev) for w in range(W)]
    c0 = wl.saps_initial_center(base)
    ga = SAPSGossip([b.clone() for b in base], c0.clone(), p, 0.9, 0.9, base_seed=11)
    mb, cb = [b.clone() for b in base], c0.clone()
    idx = torch.empty(n, dtype=torch.int32, device=dev)
    vals = [torch.empty(n, device=dev) for _ in range(W)]
    cnt = torch.zeros(1, dtype=torch.int64, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = torch.empty(gc.saps_workspace_bytes(n), dtype=torch.uint8, device=dev)
    for t in range(3):
        pairs = ga.round(t)
        seed_t = gc.saps_round_seed(11, t)
        assert pairs == gc.saps_matching(seed_t, W)
        gc.saps_mask_compact(n, p, seed_t, mb, idx, vals, cnt, ws, st)
        gc.saps_peer_average(mb, vals, idx, cnt, pairs)
        gc.easgd_step(mb, 0.9, 0.9, cb)
    torch.cuda.synchronize()
    for w in range(W):
        assert torch.equal(ga.models[w], mb[w])
    assert torch.equal(ga.center, cb)
    assert int(ga.status.item()) == 0


def test_cdsgd_rules():
    from gradient_compression_sgd_gc_gb300.compression import CDSGD
    for kw in ({"k": 0}, {"k": 2.5}, {"threshold": 0.0}, {"threshold": float("nan")},
               {"workers": 0}, {"workers": 65}, {"lr": float("inf")}, {"local_lr": float("nan")}):
        args = {"n": 10, "workers": 2, "threshold": 1e-3, "lr": 0.01, "device": "cpu"}
        args.update(kw)
        with pytest.raises(ValueError):
            CDSGD(**args)
    c = CDSGD(10, 2, 1e-3, 0.01, k=4, local_lr=0.1, device="cpu")
    # Algorithm 1 with the counter starting at 1: steps 4 and 8 are full precision
    assert [t for t in range(1, 9) if c.is_correction(t)] == [4, 8]
    with pytest.raises(ValueError):
        c.step([torch.zeros(10)], torch.zeros(10))                 # one gradient for two workers
    with pytest.raises(ValueError):
        c.step([torch.zeros(10)] * 2, torch.zeros(10))              # local_lr set, no local weights
    assert c.t == 0


@pytest.mark.gpu
@pytest.mark.parametrize("dtype,k", [(torch.float32, 4), (torch.bfloat16, 4), (torch.float32, 3), (torch.float32, 1)])
def test_cdsgd_eight_steps_against_oracle(dtype, k):
    """k = 4: steps 1-3 and 5-7 compressed (with eq. 11 local weights),
    steps 4 and 8 residual-compensated full precision (k = 3: steps 3 and 6;
    k = 1: every step); codes and residuals bit-exact, weights and local
    weights within the float tolerance."""
    from gradient_compression_sgd_gc_gb300.compression import CDSGD
    dev = "cuda"
    n, W, t, lr, llr = 70_001, 3, 1e-3, 0.01, 0.1
    cd = CDSGD(n, W, t, lr, k=k, local_lr=llr, device=dev)
    weights = wl.uniform(n, 0.05, 11, device=dev)
    w_ref = weights.cpu().numpy().astype(np.float64)
    r_ref = [np.zeros(n, np.float32) for _ in range(W)]
    local = [torch.empty(n, device=dev) for _ in range(W)]
    for step in range(1, 9):
        grads = [wl.normal(n, 5e-4, 100 * step + w, device=dev, dtype=dtype) for w in range(W)]
        hg = [(g.view(torch.int16).cpu().numpy().view(np.uint16) if dtype == torch.bfloat16 else g.cpu().numpy())
              for g in grads]
        w_before = w_ref.copy()
        corr = cd.step(grads, weights, local)
        torch.cuda.synchronize()
        assert corr == (step % k == 0)
        if corr:
            oracle.compensated_sum_update(hg, r_ref, lr, w_ref)
            for w in range(W):
                assert not cd.residuals[w].any()
        else:
            c_ref = [oracle.twobit_quantize(hg[w], r_ref[w], t) for w in range(W)]
            for w in range(W):
                np.testing.assert_array_equal(cd.codes[w].cpu().numpy().view(np.uint32), c_ref[w])
                loc = oracle.cdsgd_local_update(hg[w], w_before, llr)
                got = local[w].cpu().numpy()
                assert np.max(np.abs(got - loc) / (np.abs(loc) + llr * 1e-3)) < 1e-5
            oracle.twobit_dequant_sum_update(c_ref, n, t, oracle.KIND_SGD, lr=lr, weights=w_ref)
        for w in range(W):
            np.testing.assert_array_equal(cd.residuals[w].cpu().numpy().view(np.uint32), r_ref[w].view(np.uint32))
        got = weights.cpu().numpy()
        assert np.max(np.abs(got - w_ref) / (np.abs(w_ref) + lr * t)) < 1e-5, f"weights after step {step}"
