"""GPU parity of the 2-bit path through the C ABI: quantise + residual (fp32
and bf16 gradients), dequantise-sum + NONE/SGD/EASGD update, and the CD-SGD
correction step, element by element against the CPU oracle.

Bar: packed codes and residuals bit-exact; float outputs within the relative
1e-5 of ``gpu_helpers.assert_close``.  Sizes span one to many warp tiles and
every ragged tail (n mod 16, n mod 512); buffers carry sentinel tails that must
survive every call.
"""
import numpy as np
import pytest
import torch

import gradient_compression_sgd_gc_gb300 as gc
from gradient_compression_sgd_gc_gb300 import workloads as wl
import oracle
from gpu_helpers import (assert_close, check_guard, guarded, host_bf16_bits, host_f32, host_u32)

pytestmark = pytest.mark.gpu
DEV = "cuda"

SIZES = [1, 15, 16, 17, 255, 511, 512, 513, 1031, 3 * 512 + 40, 100_008, 262_147]


def _grad_host(g: torch.Tensor) -> np.ndarray:
    return host_bf16_bits(g) if g.dtype == torch.bfloat16 else host_f32(g)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("n", SIZES)
def test_quantize_bit_exact_over_steps(n, dtype):
    t = 0.5
    r = guarded(n, torch.float32)
    r[:n].zero_()
    codes = guarded(gc.code_words(n), torch.int32)
    r_ref = np.zeros(n, np.float32)
    for step in range(4):
        g = wl.normal(n, 0.7, seed=100 + step, device=DEV, dtype=dtype)
        gc.gc_2bit_quantize(g, r[:n], codes[:gc.code_words(n)], t)
        c_ref = oracle.twobit_quantize(_grad_host(g), r_ref, t)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(host_u32(codes[:gc.code_words(n)]), c_ref)
        np.testing.assert_array_equal(host_f32(r[:n]).view(np.uint32), r_ref.view(np.uint32))
    check_guard(r, n)
    check_guard(codes, gc.code_words(n))


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_quantize_many_tiles(dtype):
    """10,240 full tiles (many more than there are resident warps) and a
    ragged tail of 23 elements."""
    n = 5 * 1024 * 1024 + 23
    t = 1e-3
    r = torch.zeros(n, dtype=torch.float32, device=DEV)
    codes = torch.empty(gc.code_words(n), dtype=torch.int32, device=DEV)
    r_ref = np.zeros(n, np.float32)
    for step in range(3):
        g = wl.normal(n, 5e-4, seed=7 + step, device=DEV, dtype=dtype)
        gc.gc_2bit_quantize(g, r, codes, t)
        c_ref = oracle.twobit_quantize(_grad_host(g), r_ref, t)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(host_u32(codes), c_ref)
        np.testing.assert_array_equal(host_f32(r).view(np.uint32), r_ref.view(np.uint32))


def test_quantize_threshold_ties_and_special_values():
    t = np.float32(0.25)
    below = np.nextafter(t, np.float32(0))
    vals = np.array([t, -t, below, -below, 0.0, -0.0, 2 * t, -2 * t, 1e-30, -1e-30,
                     3.0, -3.0, 0.125, -0.125, t, -t, 7 * t], np.float32)
    n = vals.size
    g = torch.from_numpy(vals).to(DEV)
    r = torch.zeros(n, device=DEV)
    codes = torch.empty(gc.code_words(n), dtype=torch.int32, device=DEV)
    r_ref = np.zeros(n, np.float32)
    for _ in range(3):
        gc.gc_2bit_quantize(g, r, codes, float(t))
        c_ref = oracle.twobit_quantize(vals, r_ref, float(t))
        torch.cuda.synchronize()
        np.testing.assert_array_equal(host_u32(codes), c_ref)
        np.testing.assert_array_equal(host_f32(r).view(np.uint32), r_ref.view(np.uint32))


def test_printed_example_word_on_gpu():
    grad = torch.tensor([0.5, 2.0, -1.0, -2.5, 3.0, 1.9, -1.9, -2.0], device=DEV)
    r = torch.zeros(8, device=DEV)
    codes = torch.empty(1, dtype=torch.int32, device=DEV)
    gc.gc_2bit_quantize(grad, r, codes, 2.0)
    torch.cuda.synchronize()
    assert int(host_u32(codes)[0]) == 0x32C20000


def test_config_twobit_w1_ten_steps():
    """2-bit, one worker, 2^20 elements, t = 0.5, g ~ N(0,1) seeded by step,
    10 steps with the residual carried; each step dequantised (W = 1)."""
    cfg = wl.TWOBIT_W1
    n = cfg.n
    r = torch.zeros(n, device=DEV)
    codes = torch.empty(gc.code_words(n), dtype=torch.int32, device=DEV)
    out = torch.empty(n, device=DEV)
    r_ref = np.zeros(n, np.float32)
    for step in range(cfg.steps):
        g = wl.twobit_grad(cfg, step, 0, device=DEV)
        gc.gc_2bit_quantize(g, r, codes, cfg.threshold)
        gc.gc_2bit_dequant_sum_update([codes], n, cfg.threshold, gc.GC_UPD_NONE, out=out)
        c_ref = oracle.twobit_quantize(host_f32(g), r_ref, cfg.threshold)
        o_ref = oracle.twobit_dequant_sum_update([c_ref], n, cfg.threshold, oracle.KIND_NONE)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(host_u32(codes), c_ref)
        np.testing.assert_array_equal(host_f32(r).view(np.uint32), r_ref.view(np.uint32))
        np.testing.assert_array_equal(host_f32(out).astype(np.float64), o_ref)


def _random_words(nw, rng):
    return rng.integers(0, 2 ** 32, nw, dtype=np.uint64).astype(np.uint32)


@pytest.mark.parametrize("W", [1, 2, 7, 8, 9, 64])
@pytest.mark.parametrize("n", [1, 100, 513, 70_001])
def test_dequant_sum_update_all_kinds(W, n):
    rng = np.random.default_rng(W * 1000 + n)
    t, lr, alpha = 2e-3, 0.1, 0.9
    nw = gc.code_words(n)
    words = [_random_words(nw, rng) for _ in range(W)]
    # the tail bits beyond n are zero in any code buffer the quantiser writes
    if n % 16:
        for w in words:
            w[-1] &= np.uint32((0xFFFFFFFF << (32 - 2 * (n % 16))) & 0xFFFFFFFF)
    dcodes = [torch.from_numpy(w.view(np.int32)).to(DEV) for w in words]
    w0 = rng.uniform(-0.05, 0.05, n).astype(np.float32)
    c0 = rng.uniform(-0.05, 0.05, n).astype(np.float32)
    center = torch.from_numpy(c0).to(DEV)
    # NONE
    out = guarded(n, torch.float32)
    gc.gc_2bit_dequant_sum_update(dcodes, n, t, gc.GC_UPD_NONE, out=out[:n])
    o_ref = oracle.twobit_dequant_sum_update(words, n, t, oracle.KIND_NONE)
    torch.cuda.synchronize()
    assert_close(host_f32(out[:n]), o_ref, np.float32(t), what="dequant NONE")
    check_guard(out, n)
    # SGD
    wt = guarded(n, torch.float32)
    wt[:n].copy_(torch.from_numpy(w0))
    gc.gc_2bit_dequant_sum_update(dcodes, n, t, gc.GC_UPD_SGD, lr=lr, weights=wt[:n])
    w_ref = w0.astype(np.float64)
    oracle.twobit_dequant_sum_update(words, n, t, oracle.KIND_SGD, lr=lr, weights=w_ref)
    torch.cuda.synchronize()
    assert_close(host_f32(wt[:n]), w_ref, np.abs(w0) + lr * t, what="dequant SGD")
    check_guard(wt, n)
    # EASGD
    wt = torch.from_numpy(w0.copy()).to(DEV)
    gc.gc_2bit_dequant_sum_update(dcodes, n, t, gc.GC_UPD_EASGD, lr=lr, alpha=alpha,
                                  center=center, weights=wt)
    w_ref = w0.astype(np.float64)
    oracle.twobit_dequant_sum_update(words, n, t, oracle.KIND_EASGD, lr=lr, alpha=alpha,
                                     center=c0.astype(np.float64), weights=w_ref)
    torch.cuda.synchronize()
    assert_close(host_f32(wt), w_ref, np.abs(w0) + lr * t + alpha * (np.abs(w0) + np.abs(c0)),
                 what="dequant EASGD")


def test_dequant_lr_zero_leaves_weights_bitwise():
    n = 10_000
    rng = np.random.default_rng(3)
    words = [torch.from_numpy(_random_words(gc.code_words(n), rng).view(np.int32)).to(DEV)
             for _ in range(4)]
    w0 = torch.randn(n, device=DEV)
    w = w0.clone()
    gc.gc_2bit_dequant_sum_update(words, n, 0.5, gc.GC_UPD_SGD, lr=0.0, weights=w)
    torch.cuda.synchronize()
    assert torch.equal(w.view(torch.int32), w0.view(torch.int32))


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("n", [1, 255, 256, 257, 100_003])
def test_cdsgd_chain_k4(n, dtype):
    """Eight CD-SGD steps with k = 4: compressed steps (quantise every worker,
    dequantise-sum + SGD) and full-precision correction steps 4 and 8."""
    W, t, lr, k = 4, 1e-3, 0.01, 4
    res = [torch.zeros(n, device=DEV) for _ in range(W)]
    codes = [torch.empty(gc.code_words(n), dtype=torch.int32, device=DEV) for _ in range(W)]
    w = wl.uniform(n, 0.05, seed=8, device=DEV)
    res_ref = [np.zeros(n, np.float32) for _ in range(W)]
    w_ref = host_f32(w).astype(np.float64)
    scale = np.abs(w_ref).copy()
    for step in range(1, 9):
        grads = [wl.normal(n, 5e-4, 3000 + 10 * step + q, device=DEV, dtype=dtype) for q in range(W)]
        gh = [_grad_host(g) for g in grads]
        if step % k:
            for q in range(W):
                gc.gc_2bit_quantize(grads[q], res[q], codes[q], t)
            gc.gc_2bit_dequant_sum_update(codes, n, t, gc.GC_UPD_SGD, lr=lr, weights=w)
            c_ref = [oracle.twobit_quantize(gh[q], res_ref[q], t) for q in range(W)]
            oracle.twobit_dequant_sum_update(c_ref, n, t, oracle.KIND_SGD, lr=lr, weights=w_ref)
            scale += lr * t
            torch.cuda.synchronize()
            for q in range(W):
                np.testing.assert_array_equal(host_u32(codes[q]), c_ref[q])
        else:
            msg = np.sum([np.abs(res_ref[q].astype(np.float64))
                          + np.abs(gh[q].astype(np.float32) if dtype == torch.float32
                                   else (gh[q].astype(np.uint32) << 16).view(np.float32))
                          for q in range(W)], axis=0)
            gc.gc_compensated_sum_update(grads, res, lr, w)
            oracle.compensated_sum_update(gh, res_ref, lr, w_ref)
            scale += lr * msg / W
            torch.cuda.synchronize()
        for q in range(W):
            np.testing.assert_array_equal(host_f32(res[q]).view(np.uint32), res_ref[q].view(np.uint32))
        assert_close(host_f32(w), w_ref, scale, what=f"weights step {step}")


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_batched_quantize_matches_oracle(dtype):
    """Buffers of different sizes (ragged tails, an empty one, several tiles)
    quantised by one launch, over three steps."""
    sizes = [100_003, 0, 1, 512, 4097, 1_000_000, 17]
    t = 0.5
    res = [guarded(n, torch.float32) for n in sizes]
    for r, n in zip(res, sizes):
        r[:n].zero_()
    codes = [guarded(gc.code_words(n), torch.int32) for n in sizes]
    r_ref = [np.zeros(n, np.float32) for n in sizes]
    for step in range(3):
        grads = [wl.normal(n, 0.7, seed=500 + 10 * step + b, device=DEV, dtype=dtype)
                 for b, n in enumerate(sizes)]
        gc.gc_2bit_quantize_batched(grads, [r[:n] for r, n in zip(res, sizes)],
                                    [c[:gc.code_words(n)] for c, n in zip(codes, sizes)], t)
        refs = [oracle.twobit_quantize(_grad_host(g), r_ref[b], t) for b, g in enumerate(grads)]
        torch.cuda.synchronize()
        for b, n in enumerate(sizes):
            np.testing.assert_array_equal(host_u32(codes[b][:gc.code_words(n)]), refs[b])
            np.testing.assert_array_equal(host_f32(res[b][:n]).view(np.uint32), r_ref[b].view(np.uint32))
    for b, n in enumerate(sizes):
        check_guard(res[b], n)
        check_guard(codes[b], gc.code_words(n))


def test_batched_config_twobit_dq_sgd_sampled():
    """The 8-worker, 25,557,032-element workload through the batched quantiser
    and the dequant-sum + SGD, 3 steps, checked on sampled chunks (every
    element's chain is independent of the others)."""
    from gpu_helpers import sample_chunks
    cfg = wl.TWOBIT_DQ_SGD
    n, W, t, lr = cfg.n, cfg.workers, cfg.threshold, cfg.lr
    res = [torch.zeros(n, device=DEV) for _ in range(W)]
    codes = [torch.empty(gc.code_words(n), dtype=torch.int32, device=DEV) for _ in range(W)]
    w = wl.twobit_weights(cfg, device=DEV)
    chunks = sample_chunks(n, 48, 4096, align=16, seed=3)
    w0 = host_f32(w)
    w_ref = {c: w0[c[0]:c[1]].astype(np.float64) for c in chunks}
    r_ref = {(c, q): np.zeros(c[1] - c[0], np.float32) for c in chunks for q in range(W)}
    scale = {c: np.abs(w_ref[c]).copy() for c in chunks}
    for step in range(3):
        grads = [wl.twobit_grad(cfg, step, q, device=DEV) for q in range(W)]
        gc.gc_2bit_quantize_batched(grads, res, codes, t)
        gc.gc_2bit_dequant_sum_update(codes, n, t, gc.GC_UPD_SGD, lr=lr, weights=w)
        gh = [host_f32(g) for g in grads]
        torch.cuda.synchronize()
        hc = [host_u32(c) for c in codes]
        for c in chunks:
            lo, hi = c
            cr = [oracle.twobit_quantize(np.ascontiguousarray(gh[q][lo:hi]), r_ref[(c, q)], t)
                  for q in range(W)]
            oracle.twobit_dequant_sum_update(cr, hi - lo, t, oracle.KIND_SGD, lr=lr, weights=w_ref[c])
            scale[c] += lr * t
            for q in range(W):
                np.testing.assert_array_equal(hc[q][lo // 16:(hi + 15) // 16], cr[q])
    hw = host_f32(w)
    hr = [host_f32(r) for r in res]
    for c in chunks:
        lo, hi = c
        for q in range(W):
            np.testing.assert_array_equal(hr[q][lo:hi].view(np.uint32), r_ref[(c, q)].view(np.uint32))
        assert_close(hw[lo:hi], w_ref[c], scale[c], what=f"weights {c}")


def test_quantize_reads_pinned_host_gradients_in_place():
    """A page-locked host gradient is read directly by the kernel (no staging
    copy); results equal the oracle's, single and batched."""
    n = 300_007
    t = 0.5
    g_host = wl.normal(n, 0.7, 31).pin_memory()
    r = torch.zeros(n, device=DEV)
    codes = torch.empty(gc.code_words(n), dtype=torch.int32, device=DEV)
    r_ref = np.zeros(n, np.float32)
    gc.gc_2bit_quantize(g_host, r, codes, t)
    c_ref = oracle.twobit_quantize(g_host.numpy(), r_ref, t)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(host_u32(codes), c_ref)
    np.testing.assert_array_equal(host_f32(r).view(np.uint32), r_ref.view(np.uint32))
    gc.gc_2bit_quantize_batched([g_host, g_host], [r, r.clone()], [codes, codes.clone()], t)
    c_ref = oracle.twobit_quantize(g_host.numpy(), r_ref, t)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(host_u32(codes), c_ref)


@pytest.mark.parametrize("kind", [gc.GC_UPD_NONE, gc.GC_UPD_SGD, gc.GC_UPD_EASGD])
@pytest.mark.parametrize("n,W", [(1, 1), (513, 3), (100_003, 8), (262_144, 2)])
def test_fused_step_is_bitwise_the_two_calls(kind, n, W):
    t, lr, alpha = 2e-3, 0.1, 0.9
    grads = [wl.normal(n, 1e-3, 60 + w, device=DEV) for w in range(W)]
    r0 = [wl.normal(n, 1e-3, 80 + w, device=DEV) for w in range(W)]
    w0 = wl.uniform(n, 0.05, 7, device=DEV)
    c0 = wl.uniform(n, 0.05, 9, device=DEV)
    ra, rb = [x.clone() for x in r0], [x.clone() for x in r0]
    ca = [torch.empty(gc.code_words(n), dtype=torch.int32, device=DEV) for _ in range(W)]
    cb = [torch.empty(gc.code_words(n), dtype=torch.int32, device=DEV) for _ in range(W)]
    wa, wb = w0.clone(), w0.clone()
    oa, ob = torch.empty(n, device=DEV), torch.empty(n, device=DEV)
    kw = dict(lr=lr, alpha=alpha, center=c0 if kind == gc.GC_UPD_EASGD else None,
              weights=None if kind == gc.GC_UPD_NONE else None)
    gc.gc_2bit_quantize_batched(grads, ra, ca, t)
    gc.gc_2bit_dequant_sum_update(ca, n, t, kind, lr=lr, alpha=alpha, center=kw["center"],
                                  weights=wa if kind != gc.GC_UPD_NONE else None,
                                  out=oa if kind == gc.GC_UPD_NONE else None)
    gc.gc_2bit_step(grads, rb, cb, t, kind, lr=lr, alpha=alpha, center=kw["center"],
                    weights=wb if kind != gc.GC_UPD_NONE else None, out=ob if kind == gc.GC_UPD_NONE else None)
    torch.cuda.synchronize()
    for w in range(W):
        assert torch.equal(ra[w].view(torch.int32), rb[w].view(torch.int32))
        assert torch.equal(ca[w], cb[w])
    if kind == gc.GC_UPD_NONE:
        assert torch.equal(oa.view(torch.int32), ob.view(torch.int32))
    else:
        assert torch.equal(wa.view(torch.int32), wb.view(torch.int32))


@pytest.mark.parametrize("local", [False, True], ids=["plain", "local"])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("kind", [gc.GC_UPD_NONE, gc.GC_UPD_SGD, gc.GC_UPD_EASGD])
@pytest.mark.parametrize("n,W", [(1, 1), (513, 3), (100_003, 4), (262_144 + 16, 2)])
def test_fused_step_dtypes_and_local_weights_are_bitwise_the_separate_calls(kind, dtype, local, n, W):
    """gc_2bit_step on fp32 or bf16 gradients, optionally writing the CD-SGD
    eq. 11 local weights (gc_2bit_step_local), equals bit for bit the batched
    quantiser (or gc_2bit_quantize_local) followed by the dequant-sum update:
    codes, residuals, local weights and the updated weights (or output)."""
    t, lr, alpha, llr = 1e-3, 0.01, 0.9, 0.1
    grads = [wl.normal(n, 5e-4, 260 + w, device=DEV, dtype=dtype) for w in range(W)]
    r0 = [wl.normal(n, 5e-4, 280 + w, device=DEV) for w in range(W)]
    w0 = wl.uniform(n, 0.05, 27, device=DEV)
    c0 = wl.uniform(n, 0.05, 29, device=DEV)
    ra, rb = [x.clone() for x in r0], [x.clone() for x in r0]
    ca = [torch.empty(gc.code_words(n), dtype=torch.int32, device=DEV) for _ in range(W)]
    cb = [torch.full((gc.code_words(n),), 7, dtype=torch.int32, device=DEV) for _ in range(W)]
    wa, wb = w0.clone(), w0.clone()
    oa, ob = torch.empty(n, device=DEV), guarded(n, torch.float32)
    la = [torch.empty(n, device=DEV) for _ in range(W)]
    lb = [guarded(n, torch.float32) for _ in range(W)]
    center = c0 if kind == gc.GC_UPD_EASGD else None
    upd = dict(lr=lr, alpha=alpha, center=center, weights=wa if kind != gc.GC_UPD_NONE else None,
               out=oa if kind == gc.GC_UPD_NONE else None)
    if local:
        gc.gc_2bit_quantize_local(grads, ra, ca, wa, la, t, llr)
    else:
        gc.gc_2bit_quantize_batched(grads, ra, ca, t)
    gc.gc_2bit_dequant_sum_update(ca, n, t, kind, **upd)
    gc.gc_2bit_step(grads, rb, cb, t, kind, lr=lr, alpha=alpha, center=center,
                    weights=wb if (kind != gc.GC_UPD_NONE or local) else None,
                    out=ob[:n] if kind == gc.GC_UPD_NONE else None,
                    local_weights=[x[:n] for x in lb] if local else None, local_lr=llr)
    torch.cuda.synchronize()
    for w in range(W):
        assert torch.equal(ra[w].view(torch.int32), rb[w].view(torch.int32)), "residuals"
        assert torch.equal(ca[w], cb[w]), "codes"
        if local:
            assert torch.equal(la[w].view(torch.int32), lb[w][:n].view(torch.int32)), "local weights"
            check_guard(lb[w], n)
    if kind == gc.GC_UPD_NONE:
        assert torch.equal(oa.view(torch.int32), ob[:n].view(torch.int32))
        check_guard(ob, n)
    else:
        assert torch.equal(wa.view(torch.int32), wb.view(torch.int32))


@pytest.mark.parametrize("n,W", [(517, 3), (100_003, 4)])
def test_fused_bf16_step_with_local_weights_against_oracle(n, W):
    """The configured CD-SGD compressed step (bf16 gradients, fp32 residuals,
    SGD on the averaged dequantised sum) with eq. 11 local weights, in one
    pass, element by element against the oracle."""
    t, lr, llr = 1e-3, 0.01, 0.1
    grads = [wl.normal(n, 5e-4, 360 + w, device=DEV, dtype=torch.bfloat16) for w in range(W)]
    res = [wl.normal(n, 5e-4, 380 + w, device=DEV) for w in range(W)]
    r_ref = [host_f32(r).copy() for r in res]
    codes = [torch.empty(gc.code_words(n), dtype=torch.int32, device=DEV) for _ in range(W)]
    w0 = wl.uniform(n, 0.05, 37, device=DEV)
    w_ref = host_f32(w0).astype(np.float64)
    local = [torch.empty(n, device=DEV) for _ in range(W)]
    gc.gc_2bit_step(grads, res, codes, t, gc.GC_UPD_SGD, lr=lr, weights=w0, local_weights=local, local_lr=llr)
    torch.cuda.synchronize()
    gh = [_grad_host(g) for g in grads]
    l_ref = [oracle.cdsgd_local_update(gh[w], w_ref, llr) for w in range(W)]
    c_ref = [oracle.twobit_quantize(gh[w], r_ref[w], t) for w in range(W)]
    scale = np.abs(w_ref) + lr * t
    lscale = [np.abs(w_ref) + llr * np.abs((gh[w].astype(np.uint32) << 16).view(np.float32)) for w in range(W)]
    oracle.twobit_dequant_sum_update(c_ref, n, t, oracle.KIND_SGD, lr=lr, weights=w_ref)
    for w in range(W):
        np.testing.assert_array_equal(host_u32(codes[w]), c_ref[w])
        np.testing.assert_array_equal(host_f32(res[w]).view(np.uint32), r_ref[w].view(np.uint32))
        assert_close(host_f32(local[w]), l_ref[w], lscale[w], what="local weights")
    assert_close(host_f32(w0), w_ref, scale, what="weights")


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("n,B", [(1, 1), (517, 2), (100_003, 4)])
def test_quantize_with_local_update(n, B, dtype):
    t, lr_loc = 1e-3, 0.1
    grads = [wl.normal(n, 5e-4, 90 + b, device=DEV, dtype=dtype) for b in range(B)]
    res = [torch.zeros(n, device=DEV) for _ in range(B)]
    codes = [torch.empty(gc.code_words(n), dtype=torch.int32, device=DEV) for _ in range(B)]
    weights = wl.uniform(n, 0.05, 8, device=DEV)
    local = [guarded(n, torch.float32) for _ in range(B)]
    gc.gc_2bit_quantize_local(grads, res, codes, weights, [x[:n] for x in local], t, lr_loc)
    torch.cuda.synchronize()
    wh = host_f32(weights).astype(np.float64)
    for b in range(B):
        gh = _grad_host(grads[b])
        r_ref = np.zeros(n, np.float32)
        c_ref = oracle.twobit_quantize(gh, r_ref, t)
        np.testing.assert_array_equal(host_u32(codes[b]), c_ref)
        np.testing.assert_array_equal(host_f32(res[b]).view(np.uint32), r_ref.view(np.uint32))
        l_ref = oracle.cdsgd_local_update(gh, wh, lr_loc)
        gf = gh if dtype == torch.float32 else (gh.astype(np.uint32) << 16).view(np.float32)
        assert_close(host_f32(local[b][:n]), l_ref, np.abs(wh) + lr_loc * np.abs(gf), what="local weights")
        check_guard(local[b], n)


@pytest.mark.parametrize("n,W", [(517, 3), (100_003, 8)])
def test_fused_step_against_oracle(n, W):
    """gc_2bit_step (SGD) element by element against the oracle: every worker's
    codes and residual bit-exact, the weights within the float tolerance."""
    t, lr = 2e-3, 0.1
    grads = [wl.normal(n, 1e-3, 160 + w, device=DEV) for w in range(W)]
    res = [wl.normal(n, 1e-3, 180 + w, device=DEV) for w in range(W)]
    r_ref = [host_f32(r).copy() for r in res]
    codes = [torch.empty(gc.code_words(n), dtype=torch.int32, device=DEV) for _ in range(W)]
    w0 = wl.uniform(n, 0.05, 17, device=DEV)
    w_ref = host_f32(w0).astype(np.float64)
    gc.gc_2bit_step(grads, res, codes, t, gc.GC_UPD_SGD, lr=lr, weights=w0)
    torch.cuda.synchronize()
    c_ref = [oracle.twobit_quantize(host_f32(grads[w]), r_ref[w], t) for w in range(W)]
    scale = np.abs(w_ref) + lr * t
    oracle.twobit_dequant_sum_update(c_ref, n, t, oracle.KIND_SGD, lr=lr, weights=w_ref)
    for w in range(W):
        np.testing.assert_array_equal(host_u32(codes[w]), c_ref[w])
        np.testing.assert_array_equal(host_f32(res[w]).view(np.uint32), r_ref[w].view(np.uint32))
    assert_close(host_f32(w0), w_ref, scale, what="weights")


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("n,S", [(1, 1), (517, 3), (1 << 20, 10), (100_003, 7)])
def test_multi_step_quantize_bit_exact_against_oracle(n, S, dtype):
    """gc_2bit_quantize_steps: S successive steps of one worker in one launch
    (the configured ten steps of 2^20 elements at t = 0.5 among them), each
    step's codes and dequantised values and the final residual bit-exact with
    the oracle run step by step."""
    t = 0.5
    grads = [wl.normal(n, 1.0, 400 + st, device=DEV, dtype=dtype) for st in range(S)]
    r = wl.normal(n, 0.2, 420, device=DEV)
    r_ref = host_f32(r).copy()
    codes = [guarded(gc.code_words(n), torch.int32) for _ in range(S)]
    outs = [guarded(n, torch.float32) for _ in range(S)]
    gc.gc_2bit_quantize_steps(grads, r, [c[:gc.code_words(n)] for c in codes], t, out=[o[:n] for o in outs])
    torch.cuda.synchronize()
    for st in range(S):
        c_ref = oracle.twobit_quantize(_grad_host(grads[st]), r_ref, t)
        np.testing.assert_array_equal(host_u32(codes[st][:gc.code_words(n)]), c_ref)
        d_ref = oracle.twobit_dequant_sum_update([c_ref], n, t, oracle.KIND_NONE)
        np.testing.assert_array_equal(host_f32(outs[st][:n]).astype(np.float64), d_ref)
        check_guard(codes[st], gc.code_words(n))
        check_guard(outs[st], n)
    np.testing.assert_array_equal(host_f32(r).view(np.uint32), r_ref.view(np.uint32))


@pytest.mark.parametrize("with_out", [False, True], ids=["codes", "codes+out"])
def test_multi_step_equals_separate_calls(with_out):
    n, S, t = 262_144 + 37, 5, 2e-3
    grads = [wl.normal(n, 1e-3, 440 + st, device=DEV) for st in range(S)]
    r0 = wl.normal(n, 1e-3, 460, device=DEV)
    ra, rb = r0.clone(), r0.clone()
    ca = [torch.empty(gc.code_words(n), dtype=torch.int32, device=DEV) for _ in range(S)]
    cb = [torch.full((gc.code_words(n),), 9, dtype=torch.int32, device=DEV) for _ in range(S)]
    oa = [torch.empty(n, device=DEV) for _ in range(S)]
    ob = [torch.empty(n, device=DEV) for _ in range(S)]
    for st in range(S):
        gc.gc_2bit_quantize(grads[st], ra, ca[st], t)
        if with_out:
            gc.gc_2bit_dequant_sum_update([ca[st]], n, t, gc.GC_UPD_NONE, out=oa[st])
    gc.gc_2bit_quantize_steps(grads, rb, cb, t, out=ob if with_out else None)
    torch.cuda.synchronize()
    assert torch.equal(ra.view(torch.int32), rb.view(torch.int32))
    for st in range(S):
        assert torch.equal(ca[st], cb[st])
        if with_out:
            assert torch.equal(oa[st].view(torch.int32), ob[st].view(torch.int32))
