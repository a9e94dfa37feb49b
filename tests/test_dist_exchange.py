"""The multi-process exchange (``gradient_compression_sgd_gc_gb300.dist``) over
gloo on CPU, world sizes 2 and 4: one worker per rank, the methods' exchange
steps as collectives, and each step's arithmetic done by the oracle (injected
in place of the library's CUDA kernels, which a CPU process cannot run).

What is checked is the exchange: that what each rank gathers, sends and
reduces puts in front of the arithmetic exactly the data a single process
holding all W workers has, so the per-rank results equal the single-process
oracle run over the W workers -- bit for bit for 2-bit and QSGD (the same
arithmetic on the same codes; any world size, odd ones included), and to
rounding for SAPS + EASGD (the all-reduce sums the models in its own order;
even world sizes, as a perfect matching needs).
"""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


class OracleOps:
    """The exchange's operations done by the oracle on CPU tensors (fp64
    weights, models and centers; fp32 gradients and residuals)."""

    @staticmethod
    def quantize_2bit(grad, residual, codes, t):
        import oracle
        c = oracle.twobit_quantize(grad.numpy(), residual.numpy(), t)
        codes.copy_(torch.from_numpy(c.view(np.int32)))

    @staticmethod
    def dequant_sum_update_2bit(codes, n, t, kind, lr=0.0, alpha=0.0, center=None, weights=None, out=None):
        import oracle
        res = oracle.twobit_dequant_sum_update([c.numpy().view(np.uint32) for c in codes], n, t, kind, lr=lr,
                                               alpha=alpha, center=None if center is None else center.numpy(),
                                               weights=None if weights is None else weights.numpy())
        if out is not None:
            out.copy_(torch.from_numpy(res))

    @staticmethod
    def qsgd_quantize(v, bucket, s, seed, worker, norms, codes):
        import oracle
        rn, rc = oracle.qsgd_quantize(v.numpy(), bucket, s, seed, worker)
        norms.copy_(torch.from_numpy(rn))
        codes.copy_(torch.from_numpy(rc))

    @staticmethod
    def qsgd_dequant_sum(codes, norms, n, bucket, s, scale, out):
        import oracle
        out.copy_(torch.from_numpy(oracle.qsgd_dequant_sum([c.numpy() for c in codes], [x.numpy() for x in norms],
                                                           n, bucket, s, scale)))

    @staticmethod
    def saps_mask_compact(n, p, seed_t, models, idx, vals, count, ws, status):
        import oracle
        K, ridx, rvals = oracle.saps_mask_compact(n, p, seed_t, [m.numpy() for m in models],
                                                  capacity=idx.numel())
        idx[:K].copy_(torch.from_numpy(ridx.view(np.int32)))
        for v, r in zip(vals, rvals):
            v[:K].copy_(torch.from_numpy(r[:K]))
        count.fill_(K)

    @staticmethod
    def saps_pair_average_remote(model, idx, count, mine, peer):
        import oracle
        K = int(count.item())
        dummy = np.zeros(model.numel())
        oracle.saps_peer_average([model.numpy(), dummy], [mine.numpy()[:K], peer.numpy()[:K]],
                                 idx.numpy()[:K].view(np.uint32), np.array([0, 1], np.int32))

    @staticmethod
    def easgd_step_from_sum(model, model_sum, W, alpha, beta, center):
        import oracle
        oracle.easgd_step_from_sum(model.numpy(), model_sum.numpy(), W, alpha, beta, center.numpy())


def _grad(n, seed, scale):
    return torch.from_numpy(np.random.default_rng(seed).normal(0, scale, n).astype(np.float32))


def _rank_main(rank, world, port, case, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import torch.distributed as dist
    from gradient_compression_sgd_gc_gb300 import dist as gdist
    import gradient_compression_sgd_gc_gb300 as gc
    dist.init_process_group("gloo", rank=rank, world_size=world)
    from test_dist_exchange import OracleOps
    try:
        if case == "2bit":
            n, t, lr = 5 * 512 + 37, 2e-3, 0.1
            ex = gdist.TwoBitExchange(n, t, "cpu", ops=OracleOps)
            res = torch.zeros(n)
            w = torch.from_numpy(np.random.default_rng(7).uniform(-0.05, 0.05, n))
            codes = []
            for step in range(3):
                g = ex.step(_grad(n, 1000 * step + rank, 1e-3), res, weights=w, lr=lr)
                codes.append(g.clone().numpy())
            out[rank] = (w.numpy().copy(), res.numpy().copy(), codes)
        elif case == "qsgd":
            n, d, s = 3 * 512 + 100, 512, 7
            ex = gdist.QSGDExchange(n, d, s, 42, "cpu", ops=OracleOps)
            o = torch.zeros(n, dtype=torch.float64)
            ex.step(_grad(n, 2000 + rank, 1e-2), o)
            out[rank] = (o.numpy().copy(), ex.g_codes.numpy().copy(), ex.g_norms.numpy().copy())
        else:
            n, p = 20_011, 0.05
            bandwidth = case == "saps_bw"
            if bandwidth:
                B = np.random.default_rng(77).uniform(1.0, 10.0, (world, world))
                R = np.full((world, world), gc.NEVER, np.int64)
            ex = gdist.SAPSExchange(n, p, 5, 0.9, 0.9, "cpu", ops=OracleOps)
            rng = np.random.default_rng(4000 + rank)
            model = torch.from_numpy(rng.normal(0, 0.05, n).astype(np.float32).astype(np.float64))
            centers = [np.random.default_rng(4000 + k).normal(0, 0.05, n).astype(np.float32).astype(np.float64)
                       for k in range(world)]
            center = torch.from_numpy(sum(centers) / world)
            for t in range(3):
                seed_t = gc.saps_round_seed(5, t)
                if bandwidth:   # every rank runs the coordinator's selection on its own copy of R
                    pairs = gc.saps_matching_bandwidth(B, 5.0, R, t, 2, seed_t)
                else:
                    pairs = gc.saps_matching(seed_t, world)
                ex.round(t, model, center, pairs)
            out[rank] = (model.numpy().copy(), center.numpy().copy())
    finally:
        dist.destroy_process_group()


def _run(world, case):
    port = _free_port()
    with mp.Manager() as man:
        out = man.dict()
        mp.spawn(_rank_main, args=(world, port, case, out), nprocs=world, join=True)
        return dict(out)


@pytest.mark.parametrize("world", [2, 3, 4])
def test_two_bit_exchange_equals_single_process(world):
    import oracle
    got = _run(world, "2bit")
    n, t, lr = 5 * 512 + 37, 2e-3, 0.1
    w = np.random.default_rng(7).uniform(-0.05, 0.05, n)
    res = [np.zeros(n, np.float32) for _ in range(world)]
    for step in range(3):
        codes = [oracle.twobit_quantize(_grad(n, 1000 * step + r, 1e-3).numpy(), res[r], t) for r in range(world)]
        oracle.twobit_dequant_sum_update(codes, n, t, oracle.KIND_SGD, lr=lr, weights=w)
        for r in range(world):
            np.testing.assert_array_equal(got[r][2][step].view(np.uint32), np.stack(codes))
    for r in range(world):
        np.testing.assert_array_equal(got[r][0], w)               # every replica, bit for bit
        np.testing.assert_array_equal(got[r][1], res[r])


@pytest.mark.parametrize("world", [2, 3, 4])
def test_qsgd_exchange_equals_single_process(world):
    import oracle
    got = _run(world, "qsgd")
    n, d, s = 3 * 512 + 100, 512, 7
    q = [oracle.qsgd_quantize(_grad(n, 2000 + r, 1e-2).numpy(), d, s, 42, r) for r in range(world)]
    ref = oracle.qsgd_dequant_sum([c for _, c in q], [nm for nm, _ in q], n, d, s, 1.0 / world)
    for r in range(world):
        np.testing.assert_array_equal(got[r][0], ref)
        np.testing.assert_array_equal(got[r][1], np.stack([c for _, c in q]))
        np.testing.assert_array_equal(got[r][2], np.stack([nm for nm, _ in q]))


@pytest.mark.parametrize("world,case", [(2, "saps"), (4, "saps"), (4, "saps_bw")])
def test_saps_exchange_equals_single_process(world, case):
    """SAPS rounds across ranks with the seeded uniform matching, and (saps_bw)
    with the bandwidth-aware selection of Algorithm 3 run on every rank."""
    import oracle
    import gradient_compression_sgd_gc_gb300 as gc
    got = _run(world, case)
    n, p = 20_011, 0.05
    models = [np.random.default_rng(4000 + k).normal(0, 0.05, n).astype(np.float32).astype(np.float64)
              for k in range(world)]
    center = sum(models) / world
    if case == "saps_bw":
        B = np.random.default_rng(77).uniform(1.0, 10.0, (world, world))
        R = np.full((world, world), gc.NEVER, np.int64)
    for t in range(3):
        seed_t = gc.saps_round_seed(5, t)
        if case == "saps_bw":
            pairs = np.array(gc.saps_matching_bandwidth(B, 5.0, R, t, 2, seed_t), np.int32)
        else:
            pairs = np.array(gc.saps_matching(seed_t, world), np.int32)
        K, idx, vals = oracle.saps_mask_compact(n, p, seed_t, models)
        oracle.saps_peer_average(models, vals, idx, pairs)
        oracle.easgd_step(models, 0.9, 0.9, center)
    for r in range(world):
        np.testing.assert_allclose(got[r][0], models[r], rtol=1e-12, atol=1e-15)
        np.testing.assert_allclose(got[r][1], center, rtol=1e-12, atol=1e-15)


def test_peer_of_reads_the_matching():
    from gradient_compression_sgd_gc_gb300 import dist as gdist
    pairs = [3, 0, 2, 1]
    assert [gdist.peer_of(pairs, r) for r in range(4)] == [3, 2, 1, 0]
    with pytest.raises(ValueError):
        gdist.peer_of(pairs, 4)
