"""Parity at the workloads' full sizes, on sampled outputs.

Every output element's chain depends only on that element's inputs (2-bit,
CD-SGD, EASGD), on its bucket (QSGD) or on its index's mask bit and the round's
matching (SAPS), so the oracle runs on sampled chunks -- bucket-aligned,
including the first and the ragged last one -- while the GPU runs the whole
workload in the launch configuration bench.py times.  The SAPS counts are
also checked against the oracle's full-size mask every round.
"""
import numpy as np
import pytest
import torch

import gradient_compression_sgd_gc_gb300 as gc
from gradient_compression_sgd_gc_gb300 import workloads as wl
import oracle
from gpu_helpers import (assert_close, compare_codes, host_bf16_bits, host_f32, host_u32,
                         qsgd_sum_reference, sample_chunks)

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.mark.parametrize("one_pass", [False, True], ids=["separate", "one_pass"])
@pytest.mark.parametrize("cfg", [wl.QSGD_S7, wl.QSGD_S127], ids=lambda c: c.name)
def test_qsgd_full_size_sampled(cfg, one_pass):
    """4 workers x 61,100,840, bucket 512: every worker quantised and the
    average dequantised, by the separate calls or by qsgd_step in one pass;
    sampled chunks against the oracle (norms, codes up to boundary cases, the
    average of the GPU's own codes on every element of the chunks)."""
    n, W, d, s = cfg.n, cfg.workers, cfg.bucket, cfg.s
    nb, cb = gc.qsgd_num_buckets(n, d), gc.qsgd_code_bytes(n, s)
    vs = [wl.qsgd_grad(cfg, w, device=DEV) for w in range(W)]
    norms = [torch.empty(nb, device=DEV) for _ in range(W)]
    codes = [torch.empty(cb, dtype=torch.uint8, device=DEV) for _ in range(W)]
    out = torch.empty(n, device=DEV)
    if one_pass:
        gc.qsgd_step(vs, d, s, cfg.seed, norms, codes, 1.0 / W, out)
    else:
        for w in range(W):
            gc.qsgd_quantize(vs[w], d, s, cfg.seed, w, norms[w], codes[w])
        gc.qsgd_dequant_sum(codes, norms, n, d, s, 1.0 / W, out)
    torch.cuda.synchronize()
    chunks = sample_chunks(n, 40, 4 * d, align=d, seed=11)
    assert chunks[-1][1] == n and (n - chunks[-1][0]) % d == 296 % d
    hn = [host_f32(x) for x in norms]
    hc = [x.cpu().numpy() for x in codes]
    ho = host_f32(out)
    mism = 0
    for lo, hi in chunks:
        gcs, gns = [], []
        for w in range(W):
            v = host_f32(vs[w][lo:hi])
            rn, rc = oracle.qsgd_quantize(v, d, s, cfg.seed, w, i0=lo)
            gn = hn[w][lo // d:(hi + d - 1) // d]
            assert_close(gn, rn, np.abs(rn), what="norms")
            if s <= 7:
                gcodes = hc[w][lo // 2:(hi + 1) // 2]
            else:
                gcodes = hc[w][lo:hi]
            mism += compare_codes(gcodes, rc, v, hi - lo, d, s, cfg.seed, w, i0=lo)[0]
            gcs.append(np.ascontiguousarray(gcodes))
            gns.append(np.ascontiguousarray(gn))
        ref, terms = qsgd_sum_reference(gcs, gns, hi - lo, d, s, 1.0 / W)
        assert_close(ho[lo:hi], ref, terms, what="dequant-sum")
    print(f"{cfg.name}: level mismatches at boundaries in {len(chunks)} sampled chunks: {mism}")


@pytest.mark.parametrize("one_pass", [False, True], ids=["separate", "one_pass"])
def test_cdsgd_full_size_sampled(one_pass):
    """4 workers x 1.3e9 bf16, 8 steps, k = 4: steps 1-3 and 5-7 quantise each
    worker and apply the averaged dequantised sum (the batched quantiser and
    the dequant-sum, or gc_2bit_step in one pass), steps 4 and 8 apply the
    residual-compensated full-precision average."""
    cfg = wl.CDSGD
    n, W, t, lr, k = cfg.n, cfg.workers, cfg.threshold, cfg.lr, cfg.correction_every
    res = [torch.zeros(n, device=DEV) for _ in range(W)]
    codes = [torch.empty(gc.code_words(n), dtype=torch.int32, device=DEV) for _ in range(W)]
    wts = wl.twobit_weights(cfg, device=DEV, seed=8)
    chunks = sample_chunks(n, 24, 8192, align=16, seed=5)
    w_ref = {c: host_f32(wts[c[0]:c[1]]).astype(np.float64) for c in chunks}
    scale = {c: np.abs(w_ref[c]).copy() for c in chunks}
    r_ref = {(c, q): np.zeros(c[1] - c[0], np.float32) for c in chunks for q in range(W)}
    for step in range(1, 9):
        grads = [wl.twobit_grad(cfg, step, q, device=DEV) for q in range(W)]
        gh = {(c, q): host_bf16_bits(grads[q][c[0]:c[1]]) for c in chunks for q in range(W)}
        if step % k and one_pass:
            gc.gc_2bit_step(grads, res, codes, t, gc.GC_UPD_SGD, lr=lr, weights=wts)
        elif step % k:
            gc.gc_2bit_quantize_batched(grads, res, codes, t)
            gc.gc_2bit_dequant_sum_update(codes, n, t, gc.GC_UPD_SGD, lr=lr, weights=wts)
        else:
            gc.gc_compensated_sum_update(grads, res, lr, wts)
        torch.cuda.synchronize()
        hc = codes
        for c in chunks:
            lo, hi = c
            if step % k:
                cr = [oracle.twobit_quantize(gh[(c, q)], r_ref[(c, q)], t) for q in range(W)]
                oracle.twobit_dequant_sum_update(cr, hi - lo, t, oracle.KIND_SGD, lr=lr, weights=w_ref[c])
                scale[c] += lr * t
                for q in range(W):
                    np.testing.assert_array_equal(host_u32(hc[q][lo // 16:(hi + 15) // 16]), cr[q])
            else:
                mag = sum(np.abs(r_ref[(c, q)].astype(np.float64))
                          + np.abs((gh[(c, q)].astype(np.uint32) << 16).view(np.float32)) for q in range(W))
                oracle.compensated_sum_update([gh[(c, q)] for q in range(W)],
                                              [r_ref[(c, q)] for q in range(W)], lr, w_ref[c])
                scale[c] += lr * mag / W
        del grads
    for c in chunks:
        lo, hi = c
        for q in range(W):
            np.testing.assert_array_equal(host_f32(res[q][lo:hi]).view(np.uint32),
                                          r_ref[(c, q)].view(np.uint32))
        assert_close(host_f32(wts[lo:hi]), w_ref[c], scale[c], what=f"weights {c}")


@pytest.mark.parametrize("cfg", [wl.SAPS_P01, wl.SAPS_P001], ids=lambda c: c.name)
def test_saps_full_size_50_rounds_sampled(cfg):
    """16 workers x 25,557,032, 50 rounds of mask + compaction, fused pair
    average + elastic step, against the oracle on sampled chunks; the masked
    count of every round against the oracle's full-size mask."""
    n, W = cfg.n, cfg.workers
    models = wl.saps_models(cfg, device=DEV)
    center = wl.saps_initial_center(models)
    cap = int(n * cfg.p * 1.2 + 10_000)
    idx = torch.empty(cap, dtype=torch.int32, device=DEV)
    vals = [torch.empty(cap, device=DEV) for _ in range(W)]
    cnt = torch.zeros(1, dtype=torch.int64, device=DEV)
    ws = torch.empty(gc.saps_workspace_bytes(n), dtype=torch.uint8, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    chunks = sample_chunks(n, 16, 4096, align=32, seed=9)
    ref = {c: [host_f32(m[c[0]:c[1]]).astype(np.float64) for m in models] for c in chunks}
    rc = {c: host_f32(center[c[0]:c[1]]).astype(np.float64) for c in chunks}
    scale = {c: np.max(np.abs(np.stack(ref[c])), axis=0) + np.abs(rc[c]) for c in chunks}
    for t in range(cfg.rounds):
        seed_t = gc.saps_round_seed(cfg.base_seed, t)
        pairs = gc.saps_matching(seed_t, W)
        gc.saps_mask_compact(n, cfg.p, seed_t, models, idx, vals, cnt, ws, st)
        gc.saps_average_easgd_step(models, vals, cnt, pairs, cfg.alpha, cfg.beta, center, ws)
        for c in chunks:
            lo, hi = c
            Kc, ridx, rvals = oracle.saps_mask_compact(hi - lo, cfg.p, seed_t, ref[c], i0=lo)
            oracle.saps_peer_average(ref[c], rvals, ridx - np.uint32(lo), np.array(pairs, np.int32))
            oracle.easgd_step(ref[c], cfg.alpha, cfg.beta, rc[c])
            scale[c] = np.maximum(scale[c], np.max(np.abs(np.stack(ref[c])), axis=0) + np.abs(rc[c]))
        if t in (0, cfg.rounds - 1):
            torch.cuda.synchronize()
            Kfull = _full_mask_count(n, cfg.p, seed_t)
            assert int(cnt.item()) == Kfull and int(st.item()) == 0
    torch.cuda.synchronize()
    for c in chunks:
        lo, hi = c
        for w in range(W):
            assert_close(host_f32(models[w][lo:hi]), ref[c][w], scale[c], what=f"model {w} {c}")
        assert_close(host_f32(center[lo:hi]), rc[c], scale[c], what=f"center {c}")


def _full_mask_count(n, p, seed_t):
    """The oracle's masked count over all n indices (one worker of zeros)."""
    K, _, _ = oracle.saps_mask_compact(n, p, seed_t, [np.zeros(n)], capacity=0)
    return K


def test_indices_beyond_two_to_the_32():
    """64-bit indexing: 2^32 + 3000 elements (17 GB per fp32 buffer).  The QSGD
    buckets and the 2-bit words just below and above element 2^32, and the last
    ones, equal the oracle's at their global indices (the hash keys' high words
    change there)."""
    n = (1 << 32) + 3000
    free, _ = torch.cuda.mem_get_info()
    if free < (48 << 30):
        pytest.skip("needs about 48 GB of free device memory")
    v = torch.empty(n, device=DEV)
    chunk = 1 << 28
    for i, c0 in enumerate(range(0, n, chunk)):
        c1 = min(n, c0 + chunk)
        wl.normal(c1 - c0, 1e-2, 9000 + i, device=DEV, out=v[c0:c1])
    d, s, seed, worker = 512, 127, 77, 1
    nb, cb = gc.qsgd_num_buckets(n, d), gc.qsgd_code_bytes(n, s)
    norms = torch.empty(nb, device=DEV)
    codes = torch.empty(cb, dtype=torch.uint8, device=DEV)
    gc.qsgd_quantize(v, d, s, seed, worker, norms, codes)
    torch.cuda.synchronize()
    for b0 in ((1 << 32) // d - 3, nb - 4):
        lo, hi = b0 * d, min(n, (b0 + 6) * d)
        vh = host_f32(v[lo:hi])
        rn, rc = oracle.qsgd_quantize(vh, d, s, seed, worker, i0=lo)
        np.testing.assert_array_equal(host_f32(norms[b0:b0 + rn.size]).view(np.uint32), rn.view(np.uint32))
        compare_codes(codes[lo:hi].cpu().numpy(), rc, vh, hi - lo, d, s, seed, worker, i0=lo)
    del norms, codes
    t = 1e-2
    res = torch.zeros(n, device=DEV)
    words = torch.empty(gc.code_words(n), dtype=torch.int32, device=DEV)
    gc.gc_2bit_quantize(v, res, words, t)
    torch.cuda.synchronize()
    ranges = (((1 << 32) - 1024, (1 << 32) + 1024), (n - 1000 - (n - 1000) % 16, n))
    refs = []
    for lo, hi in ranges:
        r_ref = np.zeros(hi - lo, np.float32)
        c_ref = oracle.twobit_quantize(host_f32(v[lo:hi]), r_ref, t)
        np.testing.assert_array_equal(host_u32(words[lo // 16:lo // 16 + c_ref.size]), c_ref)
        np.testing.assert_array_equal(host_f32(res[lo:hi]).view(np.uint32), r_ref.view(np.uint32))
        refs.append(c_ref)
    del v
    # the dequantised values (one worker) into the residual buffer
    gc.gc_2bit_dequant_sum_update([words], n, t, gc.GC_UPD_NONE, out=res)
    torch.cuda.synchronize()
    for (lo, hi), c_ref in zip(ranges, refs):
        a_ref = oracle.twobit_dequant_sum_update([c_ref], hi - lo, t, oracle.KIND_NONE)
        assert_close(host_f32(res[lo:hi]), a_ref, np.full(hi - lo, t), what="dequantised")
    del res, words
    torch.cuda.empty_cache()


def test_saps_mask_at_the_largest_n():
    """n = 2^32 - 1, the largest count uint32 indices allow (two workers of
    17 GB): indices stay ascending and below n, and every sampled range --
    the first, the last and ones in between -- holds exactly the oracle's
    indices and gathered values for that range."""
    n, W, p = (1 << 32) - 1, 2, 1e-4
    free, _ = torch.cuda.mem_get_info()
    if free < (40 << 30):
        pytest.skip("needs about 40 GB of free device memory")
    models = [torch.empty(n, device=DEV) for _ in range(W)]
    chunk = 1 << 28
    for w in range(W):
        for i, c0 in enumerate(range(0, n, chunk)):
            c1 = min(n, c0 + chunk)
            wl.normal(c1 - c0, 0.05, 7000 + 100 * w + i, device=DEV, out=models[w][c0:c1])
    cap = int(n * p * 1.2) + 10_000
    idx = torch.empty(cap, dtype=torch.int32, device=DEV)
    vals = [torch.empty(cap, device=DEV) for _ in range(W)]
    cnt = torch.zeros(1, dtype=torch.int64, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    ws = torch.empty(gc.saps_workspace_bytes(n), dtype=torch.uint8, device=DEV)
    seed_t = gc.saps_round_seed(11, 3)
    gc.saps_mask_compact(n, p, seed_t, models, idx, vals, cnt, ws, st)
    torch.cuda.synchronize()
    K = int(cnt.item())
    assert int(st.item()) == 0 and 0 < K <= cap
    gi = host_u32(idx[:K]).astype(np.int64)
    assert np.all(np.diff(gi) > 0) and gi[-1] < n
    gv = [host_f32(v[:K]) for v in vals]
    for lo, hi in sample_chunks(n, 6, 1 << 22, align=4096, seed=5):
        ref = [host_f32(m[lo:hi]).astype(np.float64) for m in models]
        Kc, ridx, rvals = oracle.saps_mask_compact(hi - lo, p, seed_t, ref, i0=lo)
        a, b = np.searchsorted(gi, lo), np.searchsorted(gi, hi)
        assert b - a == Kc
        np.testing.assert_array_equal(gi[a:b], ridx.astype(np.int64))
        for w in range(W):
            np.testing.assert_array_equal(gv[w][a:b].astype(np.float64), rvals[w])
    del models, idx, vals, ws
    torch.cuda.empty_cache()


def test_elias_beyond_two_to_the_32():
    """The Elias codec on 2^32 + 3000 QSGD s=7 coordinates: offsets stay
    32-bit word indices; sampled buckets' words equal the oracle's encoding
    of the same codes; the decode gives the levels back everywhere."""
    n, d, s = (1 << 32) + 3000, 512, 7
    free, _ = torch.cuda.mem_get_info()
    if free < (40 << 30):
        pytest.skip("needs about 40 GB of free device memory")
    nb, cb = gc.qsgd_num_buckets(n, d), gc.qsgd_code_bytes(n, s)
    codes = torch.empty(cb, dtype=torch.uint8, device=DEV)
    norms = torch.empty(nb, device=DEV)
    v = torch.empty(1 << 28, device=DEV)
    for i, c0 in enumerate(range(0, n, 1 << 28)):       # quantise in slices: v is not kept whole
        c1 = min(n, c0 + (1 << 28))
        wl.normal(c1 - c0, 1e-2, 9500 + i, device=DEV, out=v[:c1 - c0])
        gc.qsgd_quantize(v[:c1 - c0], d, s, 5, 0, norms[c0 // d:(c1 + d - 1) // d], codes[c0 // 2:(c1 + 1) // 2])
    del v
    cap = gc.qsgd_elias_max_words(n, d, s)
    words = torch.empty(cap, dtype=torch.int32, device=DEV)
    offs = torch.empty(nb + 1, dtype=torch.int32, device=DEV)
    ws = torch.empty(gc.qsgd_elias_workspace_bytes(n, d), dtype=torch.uint8, device=DEV)
    gc.qsgd_elias_encode(codes, norms, n, d, s, words, offs, ws)
    torch.cuda.synchronize()
    ho = host_u32(offs).astype(np.int64)
    assert np.all(np.diff(ho) >= 2)
    for b0 in (0, (1 << 32) // d - 2, nb - 3):
        b1 = min(nb, b0 + 3)
        lo, hi = b0 * d, min(n, b1 * d)
        rc = codes[lo // 2:(hi + 1) // 2].cpu().numpy()
        rn = host_f32(norms[b0:b1])
        ref_w, ref_off = oracle.qsgd_elias_encode(rc, rn, hi - lo, d, s)
        np.testing.assert_array_equal(ho[b0:b1 + 1] - ho[b0], ref_off.astype(np.int64))
        np.testing.assert_array_equal(host_u32(words[int(ho[b0]):int(ho[b1])]), ref_w)
    dc = torch.empty_like(codes)
    dn = torch.empty_like(norms)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    gc.qsgd_elias_decode(words, offs, n, d, s, dc, dn, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(dn, norms)
    assert torch.equal(dc & 0x77, codes & 0x77)          # levels; a level-0 code comes back with sign 0
    del codes, norms, words, offs, ws, dc, dn
    torch.cuda.empty_cache()


@pytest.mark.parametrize("cfg", [wl.QSGD_S7, wl.QSGD_S127], ids=lambda c: c.name)
def test_elias_sparse_full_size_sampled(cfg):
    """The sparse-regime Elias stream of one worker's codes on the configured
    61,100,840 coordinates: 48 sampled buckets (the first and the ragged last
    among them) word for word against the oracle's encoding of the same
    bucket, and the whole stream decoded back to the codes."""
    n, d, s = cfg.n, cfg.bucket, cfg.s
    v = wl.qsgd_grad(cfg, 0, device=DEV)
    nb, cb = gc.qsgd_num_buckets(n, d), gc.qsgd_code_bytes(n, s)
    norms = torch.empty(nb, device=DEV)
    codes = torch.empty(cb, dtype=torch.uint8, device=DEV)
    gc.qsgd_quantize(v, d, s, cfg.seed, 0, norms, codes)
    cap = gc.qsgd_elias_sparse_max_words(n, d)
    words = torch.empty(cap, dtype=torch.int32, device=DEV)
    offs = torch.empty(nb + 1, dtype=torch.int32, device=DEV)
    ws = torch.empty(gc.qsgd_elias_workspace_bytes(n, d), dtype=torch.uint8, device=DEV)
    gc.qsgd_elias_encode_sparse(codes, norms, n, d, s, words, offs, ws)
    dc = torch.empty_like(codes)
    dn = torch.empty_like(norms)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    gc.qsgd_elias_decode_sparse(words, offs, n, d, s, dc, dn, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    hc, hn = codes.cpu().numpy(), host_f32(norms)
    ho, hw = host_u32(offs), host_u32(words)
    rng = np.random.default_rng(9)
    picks = sorted({0, nb - 1} | {int(b) for b in rng.integers(0, nb, 46)})
    for b in picks:
        lo = b * d
        ln = min(d, n - lo)
        cs = hc[lo // 2:(lo + ln + 1) // 2] if s <= 7 else hc[lo:lo + ln]
        rw, ro = oracle.qsgd_elias_encode_sparse(np.ascontiguousarray(cs), hn[b:b + 1].copy(), ln, d, s)
        np.testing.assert_array_equal(hw[ho[b]:ho[b + 1]], rw)
    if s <= 7:
        nib = np.stack([hc >> 4, hc & 15], axis=1).reshape(-1)
        nib = np.where((nib & 7) == 0, 0, nib)
        canon = ((nib[0::2] << 4) | nib[1::2]).astype(np.uint8)
    else:
        canon = np.where((hc & 127) == 0, 0, hc).astype(np.uint8)
    np.testing.assert_array_equal(dc.cpu().numpy(), canon)
    assert torch.equal(dn.view(torch.int32), norms.view(torch.int32))
