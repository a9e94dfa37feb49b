"""GPU parity of QSGD quantise and dequantise-sum through the C ABI.

Bar: per-bucket norms within rel 1e-5 (and, as computed, almost always
bit-identical: both sides round the exact l2 norm); codes byte-identical
except for levels whose deciding value x = |v| * (s / norm) + u lies within
1e-6 of an integer (both sides decide in fp32; a one-ulp norm difference can
only move such levels), and those mismatches are counted and reported.  The
dequantised sums are checked on the GPU's own codes and norms against the
oracle's sum of the same codes, on every element, within rel 1e-5 of
sum |terms|.
"""
import numpy as np
import pytest
import torch

import gradient_compression_sgd_gc_gb300 as gc
from gradient_compression_sgd_gc_gb300 import workloads as wl
import oracle
from gpu_helpers import (assert_close, check_guard, compare_codes, guarded, host_f32,
                         qsgd_sum_reference)

pytestmark = pytest.mark.gpu
DEV = "cuda"


CASES = [(n, b, s) for n in (1, 2, 511, 512, 513, 5 * 512 + 297, 100_001) for b in (128, 512, 2048)
         for s in (7, 127)] + [(3, 512, 1), (1000, 256, 3), (4097, 1024, 64)] + [
    # s = 1 (ternary) and s = floor(sqrt(d)), the dense regime, per bucket size
    (100_001, 512, 1), (100_001, 512, 22), (5 * 512 + 297, 128, 11), (70_000, 2048, 45)]


@pytest.mark.parametrize("n,bucket,s", CASES)
def test_quantize_parity(n, bucket, s):
    cfg = wl.scaled(wl.QSGD_S7, n)
    mism = 0
    for worker in (0, 3):
        v = wl.qsgd_grad(cfg, worker, device=DEV)
        nb = gc.qsgd_num_buckets(n, bucket)
        cb = gc.qsgd_code_bytes(n, s)
        norms = guarded(nb, torch.float32)
        codes = guarded(cb, torch.uint8)
        gc.qsgd_quantize(v, bucket, s, 42, worker, norms[:nb], codes[:cb])
        vh = host_f32(v)
        rn, rc = oracle.qsgd_quantize(vh, bucket, s, 42, worker)
        torch.cuda.synchronize()
        gn = host_f32(norms[:nb])
        assert_close(gn, rn, np.abs(rn), what="norms")
        m, _ = compare_codes(codes[:cb].cpu().numpy(), rc, vh, n, bucket, s, 42, worker)
        mism += m
        check_guard(norms, nb)
        check_guard(codes, cb)
    print(f"qsgd n={n} bucket={bucket} s={s}: level mismatches at boundaries: {mism}")


def test_zero_buckets_and_signed_zero():
    n = 2048
    v = torch.zeros(n, device=DEV)
    v[700] = -0.0
    v[1500] = 3.0
    v[1400] = -4.0
    for s in (7, 127):
        norms = torch.empty(4, device=DEV)
        codes = torch.empty(gc.qsgd_code_bytes(n, s), dtype=torch.uint8, device=DEV)
        gc.qsgd_quantize(v, 512, s, 1, 0, norms, codes)
        rn, rc = oracle.qsgd_quantize(host_f32(v), 512, s, 1, 0)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(host_f32(norms), rn)
        np.testing.assert_array_equal(codes.cpu().numpy(), rc)
        assert host_f32(norms)[2] == 5.0


def test_norms_bit_identical_on_heavy_tails():
    """The GPU rounds the exact norm too: on a heavy-tailed vector of 2^20
    elements essentially every norm is bit-identical to the oracle's."""
    cfg = wl.scaled(wl.QSGD_S127, 1 << 20)
    v = wl.qsgd_grad(cfg, 1, device=DEV)
    nb = gc.qsgd_num_buckets(cfg.n, 512)
    norms = torch.empty(nb, device=DEV)
    codes = torch.empty(cfg.n, dtype=torch.uint8, device=DEV)
    gc.qsgd_quantize(v, 512, 127, 42, 1, norms, codes)
    rn, rc = oracle.qsgd_quantize(host_f32(v), 512, 127, 42, 1)
    torch.cuda.synchronize()
    diff = int((host_f32(norms) != rn).sum())
    print(f"norms differing from the correctly rounded value: {diff} of {nb}")
    assert diff <= 2
    m, _ = compare_codes(codes.cpu().numpy(), rc, host_f32(v), cfg.n, 512, 127, 42, 1)
    print(f"level mismatches: {m}")


@pytest.mark.parametrize("s", [7, 127])
@pytest.mark.parametrize("n,W", [(1, 1), (513, 2), (5 * 512 + 297, 4), (100_001, 4), (4096, 9)])
def test_dequant_sum_parity(n, W, s):
    _dequant_sum_case(n, W, s, 512)


@pytest.mark.parametrize("n,W,s,bucket", [
    (3_000_017, 4, 7, 128), (3_000_017, 9, 127, 128), (3_000_017, 8, 7, 512), (3_000_017, 3, 100, 256),
    (12_000_013, 5, 7, 2048), (12_000_013, 9, 127, 2048), (12_000_013, 4, 127, 512),
    (200_003, 64, 7, 128), (200_003, 64, 127, 512)])
def test_dequant_sum_many_buckets_per_warp(n, W, s, bucket):
    """Sizes at which every warp of the persistent grid walks several
    buckets (or, at 64 workers, 16 worker groups of one bucket), so the
    shared-memory stages of the copy pipeline are reused and worker groups of
    1..4 alternate; the ragged last bucket included."""
    _dequant_sum_case(n, W, s, bucket)


def _dequant_sum_case(n, W, s, bucket):
    cfg = wl.scaled(wl.QSGD_S7, n)
    nb = gc.qsgd_num_buckets(n, bucket)
    cb = gc.qsgd_code_bytes(n, s)
    codes, norms = [], []
    mism = 0
    for w in range(W):
        v = wl.qsgd_grad(cfg, w, device=DEV)
        c = torch.empty(cb, dtype=torch.uint8, device=DEV)
        nm = torch.empty(nb, device=DEV)
        gc.qsgd_quantize(v, bucket, s, 42, w, nm, c)
        rn, rc = oracle.qsgd_quantize(host_f32(v), bucket, s, 42, w)
        torch.cuda.synchronize()
        assert_close(host_f32(nm), rn, np.abs(rn), what="norms")
        mism += compare_codes(c.cpu().numpy(), rc, host_f32(v), n, bucket, s, 42, w)[0]
        codes.append(c)
        norms.append(nm)
    scale = 1.0 / W
    out = guarded(n, torch.float32)
    gc.qsgd_dequant_sum(codes, norms, n, bucket, s, scale, out[:n])
    ref, terms = qsgd_sum_reference([c.cpu().numpy() for c in codes], [host_f32(x) for x in norms],
                                    n, bucket, s, scale)
    torch.cuda.synchronize()
    assert_close(host_f32(out[:n]), ref, terms, what="dequant-sum")
    check_guard(out, n)
    print(f"qsgd dequant n={n} W={W} s={s}: level mismatches at boundaries: {mism}")


@pytest.mark.parametrize("scale", [1e-40, 1e-25, 1e25])
def test_tiny_and_huge_buckets_match_oracle(scale):
    """Buckets whose squares underflow or overflow fp32 (subnormal-sized or
    huge gradients): norms within rel 1e-5, codes equal up to boundary cases;
    the subnormal case also exercises the s / norm overflow reading."""
    n = 2048
    rng = np.random.default_rng(5)
    vh = (rng.normal(0, 1, n) * scale).astype(np.float32)
    vh[512:520] = 0.0
    vh[1024:1536] = 0.0
    vh[1100] = np.float32(scale)
    v = torch.from_numpy(vh).to(DEV)
    for s in (7, 127):
        norms = torch.empty(4, device=DEV)
        codes = torch.empty(gc.qsgd_code_bytes(n, s), dtype=torch.uint8, device=DEV)
        gc.qsgd_quantize(v, 512, s, 4, 0, norms, codes)
        rn, rc = oracle.qsgd_quantize(vh, 512, s, 4, 0)
        torch.cuda.synchronize()
        assert_close(host_f32(norms), rn, np.abs(rn), what="norms")
        assert host_f32(norms)[2] == rn[2]          # one nonzero value: |v| exactly
        compare_codes(codes.cpu().numpy(), rc, vh, n, 512, s, 4, 0)
        ref, terms = qsgd_sum_reference([codes.cpu().numpy()], [host_f32(norms)], n, 512, s, 1.0)
        out = torch.empty(n, device=DEV)
        gc.qsgd_dequant_sum([codes], [norms], n, 512, s, 1.0, out)
        torch.cuda.synchronize()
        assert_close(host_f32(out), ref, terms, what="dequant of tiny/huge buckets")


@pytest.mark.parametrize("s", [1, 7, 22, 127])
@pytest.mark.parametrize("n,bucket", [(1, 512), (5 * 512 + 297, 512), (100_001, 128), (70_000, 2048)])
def test_maxnorm_quantize_parity(n, bucket, s):
    """Knowl 8 max-norm scaling (and the s = 1 ternary and s ~ sqrt(d) dense
    level counts): the scale is a max, exact on both sides, so scales and
    codes are bit-exact; the dequant-sum within tolerance."""
    cfg = wl.scaled(wl.QSGD_S7, n)
    v = wl.qsgd_grad(cfg, 2, device=DEV)
    nb, cb = gc.qsgd_num_buckets(n, bucket), gc.qsgd_code_bytes(n, s)
    scales = guarded(nb, torch.float32)
    codes = guarded(cb, torch.uint8)
    gc.qsgd_quantize_maxnorm(v, bucket, s, 42, 2, scales[:nb], codes[:cb])
    out = torch.empty(n, device=DEV)
    gc.qsgd_dequant_sum([codes[:cb]], [scales[:nb]], n, bucket, s, 1.0, out)
    vh = host_f32(v)
    rs, rc = oracle.qsgd_quantize_maxnorm(vh, bucket, s, 42, 2)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(host_f32(scales[:nb]), rs)
    np.testing.assert_array_equal(codes[:cb].cpu().numpy(), rc)
    check_guard(scales, nb)
    check_guard(codes, cb)
    ref = oracle.qsgd_dequant_sum([rc], [rs], n, bucket, s)
    assert_close(host_f32(out), ref, np.abs(ref), what="maxnorm dequant")


@pytest.mark.parametrize("maxnorm", [False, True], ids=["l2", "maxnorm"])
@pytest.mark.parametrize("s", [1, 7, 22, 127])
@pytest.mark.parametrize("n,bucket,W", [(1, 512, 1), (5 * 512 + 297, 512, 4), (100_001, 128, 3),
                                         (70_000, 2048, 2), (4096 * 3 + 1, 256, 9)])
def test_one_pass_step_is_bitwise_the_separate_calls(n, bucket, W, s, maxnorm):
    """qsgd_step == W x qsgd_quantize (or _maxnorm) + qsgd_dequant_sum, bit for
    bit: codes, norms and the sum."""
    cfg = wl.scaled(wl.QSGD_S7, n)
    vs = [wl.qsgd_grad(cfg, w, device=DEV) for w in range(W)]
    nb, cb = gc.qsgd_num_buckets(n, bucket), gc.qsgd_code_bytes(n, s)
    n1 = [torch.empty(nb, device=DEV) for _ in range(W)]
    c1 = [torch.empty(cb, dtype=torch.uint8, device=DEV) for _ in range(W)]
    q = gc.qsgd_quantize_maxnorm if maxnorm else gc.qsgd_quantize
    for w in range(W):
        q(vs[w], bucket, s, 77, w, n1[w], c1[w])
    o1 = torch.empty(n, device=DEV)
    gc.qsgd_dequant_sum(c1, n1, n, bucket, s, 1.0 / W, o1)
    n2 = [torch.full((nb,), 7.0, device=DEV) for _ in range(W)]
    c2 = [torch.full((cb,), 0xEE, dtype=torch.uint8, device=DEV) for _ in range(W)]
    o2 = guarded(n, torch.float32)
    gc.qsgd_step(vs, bucket, s, 77, n2, c2, 1.0 / W, o2[:n], maxnorm=maxnorm)
    torch.cuda.synchronize()
    check_guard(o2, n)
    for w in range(W):
        assert torch.equal(n1[w].view(torch.int32), n2[w].view(torch.int32))
        assert torch.equal(c1[w], c2[w])
    assert torch.equal(o1.view(torch.int32), o2[:n].view(torch.int32))


@pytest.mark.parametrize("s", [7, 127])
@pytest.mark.parametrize("n,W", [(5 * 512 + 297, 4), (100_001, 3)])
def test_one_pass_step_against_oracle(n, W, s):
    """qsgd_step element by element against the oracle: norms within rel 1e-5
    (bit-equal in practice), codes up to boundary cases, and the average of
    the GPU's own codes within the float tolerance on every element."""
    cfg = wl.scaled(wl.QSGD_S7, n)
    d = 512
    vs = [wl.qsgd_grad(cfg, w, device=DEV) for w in range(W)]
    nb, cb = gc.qsgd_num_buckets(n, d), gc.qsgd_code_bytes(n, s)
    norms = [torch.empty(nb, device=DEV) for _ in range(W)]
    codes = [torch.empty(cb, dtype=torch.uint8, device=DEV) for _ in range(W)]
    out = torch.empty(n, device=DEV)
    gc.qsgd_step(vs, d, s, 31, norms, codes, 1.0 / W, out)
    torch.cuda.synchronize()
    for w in range(W):
        vh = host_f32(vs[w])
        rn, rc = oracle.qsgd_quantize(vh, d, s, 31, w)
        assert_close(host_f32(norms[w]), rn, np.abs(rn), what="norms")
        compare_codes(codes[w].cpu().numpy(), rc, vh, n, d, s, 31, w)
    ref, terms = qsgd_sum_reference([c.cpu().numpy() for c in codes], [host_f32(x) for x in norms],
                                    n, d, s, 1.0 / W)
    assert_close(host_f32(out), ref, terms, what="average")


def _mixed_scale_vector(n, seed):
    """Buckets of 512 cycling through normal, subnormal-sized (flagged: the
    sum of squares underflows), huge (flagged: it overflows) and all-zero
    values, with a ragged tail."""
    rng = np.random.default_rng(seed)
    v = rng.normal(0, 1, n)
    for b in range((n + 511) // 512):
        kind = b % 4
        sl = slice(512 * b, min(n, 512 * b + 512))
        if kind == 1:
            v[sl] *= 1e-41
        elif kind == 2:
            v[sl] *= 1e25
        elif kind == 3:
            v[sl] = 0.0
    return v.astype(np.float32)


@pytest.mark.parametrize("s", [7, 127])
@pytest.mark.parametrize("n", [512 * 37 + 111, 512 * 300])
def test_flagged_buckets_are_redone(n, s):
    """Buckets whose sum of squares under- or overflows are finished by the
    fix-up launch: half of all buckets here, spread over many 32-bucket scan
    groups, plus zero buckets and the ragged tail; norms and codes against
    the oracle, and the dequantised sum of the GPU's codes."""
    vh = _mixed_scale_vector(n, 17 + s)
    v = torch.from_numpy(vh).to(DEV)
    nb, cb = gc.qsgd_num_buckets(n, 512), gc.qsgd_code_bytes(n, s)
    norms = guarded(nb, torch.float32)
    codes = guarded(cb, torch.uint8)
    gc.qsgd_quantize(v, 512, s, 11, 2, norms[:nb], codes[:cb])
    rn, rc = oracle.qsgd_quantize(vh, 512, s, 11, 2)
    torch.cuda.synchronize()
    gn = host_f32(norms[:nb])
    assert np.all(gn >= 0), "a flagged norm was left behind"
    assert_close(gn, rn, np.abs(rn), what="norms")
    compare_codes(codes[:cb].cpu().numpy(), rc, vh, n, 512, s, 11, 2)
    check_guard(norms, nb)
    check_guard(codes, cb)
    out = torch.empty(n, device=DEV)
    gc.qsgd_dequant_sum([codes[:cb]], [norms[:nb]], n, 512, s, 1.0, out)
    ref, terms = qsgd_sum_reference([codes[:cb].cpu().numpy()], [gn], n, 512, s, 1.0)
    torch.cuda.synchronize()
    assert_close(host_f32(out), ref, terms, what="dequant")


@pytest.mark.parametrize("s", [7, 127])
def test_one_pass_step_with_flagged_buckets(s):
    """qsgd_step when some workers' buckets are flagged (their whole bucket is
    redone for every worker by the step's fix-up): bit for bit the separate
    calls, and the oracle's codes."""
    n, W = 512 * 41 + 7, 3
    vhs = [_mixed_scale_vector(n, 40 + w + s) for w in range(W)]
    vhs[1][512 * 4:512 * 8] = np.random.default_rng(3).normal(0, 1, 2048).astype(np.float32)
    vs = [torch.from_numpy(x).to(DEV) for x in vhs]
    nb, cb = gc.qsgd_num_buckets(n, 512), gc.qsgd_code_bytes(n, s)
    n1 = [torch.empty(nb, device=DEV) for _ in range(W)]
    c1 = [torch.empty(cb, dtype=torch.uint8, device=DEV) for _ in range(W)]
    for w in range(W):
        gc.qsgd_quantize(vs[w], 512, s, 5, w, n1[w], c1[w])
    o1 = torch.empty(n, device=DEV)
    gc.qsgd_dequant_sum(c1, n1, n, 512, s, 1.0 / W, o1)
    n2 = [torch.full((nb,), 3.0, device=DEV) for _ in range(W)]
    c2 = [torch.full((cb,), 0x5A, dtype=torch.uint8, device=DEV) for _ in range(W)]
    o2 = guarded(n, torch.float32)
    gc.qsgd_step(vs, 512, s, 5, n2, c2, 1.0 / W, o2[:n])
    torch.cuda.synchronize()
    check_guard(o2, n)
    for w in range(W):
        assert torch.equal(n1[w].view(torch.int32), n2[w].view(torch.int32))
        assert torch.equal(c1[w], c2[w])
        rn, rc = oracle.qsgd_quantize(vhs[w], 512, s, 5, w)
        assert_close(host_f32(n2[w]), rn, np.abs(rn), what="norms")
        compare_codes(c2[w].cpu().numpy(), rc, vhs[w], n, 512, s, 5, w)
    assert torch.equal(o1.view(torch.int32), o2[:n].view(torch.int32))
