"""Pins for the oracle's QSGD quantiser and dequantise-sum, and for the
counter-based hash both QSGD and SAPS draw from.

Sources: "QSGD: Communication-Efficient SGD via Gradient Quantization and
Encoding" (summary page): Knowl 1 (operator Q_s, sgn(0) = +1, Q_s(0) = 0,
unbiasedness, variance bound, expected sparsity), Knowl 2 (norm stored as a
single-precision float; tuple (norm, sign, level)), Knowl 3 (average of K
decoded messages), Knowl 8 (bucketing, per-bucket variance bound).
The hash is SplitMix64 (Steele, Lea, Flood, OOPSLA 2014); its known answers
are the first two outputs of the generator seeded with 0.
"""
import math
from fractions import Fraction

import numpy as np
import pytest

import oracle


# ---------------------------------------------------------------- hash

def test_splitmix64_known_answers():
    assert oracle.splitmix64(0) == 0xE220A8397B1DCDAF
    assert oracle.splitmix64(0x9E3779B97F4A7C15) == 0x6E789E6AA1B965F4


def test_uniform_grid_mean_and_flatness():
    keys = range(1 << 16)
    u = np.array([oracle.uniform(k ^ 0x1234_5678_9ABC) for k in keys])
    assert np.all(u >= 0.0) and np.all(u < 1.0)
    assert np.all(u * 2 ** 24 == np.floor(u * 2 ** 24))       # multiples of 2^-24
    assert abs(u.mean() - 0.5) < 5 * math.sqrt(1 / 12 / u.size)
    hist = np.bincount((u * 256).astype(int), minlength=256)
    expected = u.size / 256
    chi2 = float(((hist - expected) ** 2 / expected).sum())
    # 255 degrees of freedom: mean 255, sd ~22.6; 5 sd bound
    assert chi2 < 255 + 5 * math.sqrt(2 * 255)


def test_qsgd_dither_fields_of_published_splitmix64_outputs():
    """The pair (2j, 2j + 1) shares z = splitmix64(seed_w ^ j): bits 40..63
    for the even element, bits 8..31 for the odd one.  SplitMix64 seeded with 0
    gives 0xE220A8397B1DCDAF and then 0x6E789E6AA1B965F4 (Steele, Lea and
    Flood 2014); as counters those are splitmix64(0) and
    splitmix64(0x9E3779B97F4A7C15)."""
    g = 0x9E3779B97F4A7C15
    assert oracle.qsgd_dither(0, 0, 0) == 0xE220A8 / 2 ** 24
    assert oracle.qsgd_dither(0, 0, 1) == 0x7B1DCD / 2 ** 24
    assert oracle.qsgd_dither(g, 0, 0) == 0x6E789E / 2 ** 24
    assert oracle.qsgd_dither(g, 0, 1) == 0xA1B965 / 2 ** 24
    # index 2j and 2j + 1 use the counter seed_w ^ j: j = 1 with seed_w = g ^ 1
    assert oracle.qsgd_dither(g ^ 1, 0, 2) == 0x6E789E / 2 ** 24
    assert oracle.qsgd_dither(g ^ 1, 0, 3) == 0xA1B965 / 2 ** 24
    # the worker is folded in at bit 48, indices above 2^32 keep their high bits
    w, big = 3, (5 << 33) | 6
    assert oracle.qsgd_dither(g ^ (w << 48) ^ (big >> 1), w, big) == 0x6E789E / 2 ** 24
    assert oracle.qsgd_dither(g ^ (big >> 1), 0, big + 1) == 0xA1B965 / 2 ** 24


def test_qsgd_dither_fields_uniform_and_independent():
    """Both fields are uniform on the 2^-24 grid, and the two fields of one
    output, and neighbouring pairs, are uncorrelated."""
    n = 1 << 16
    u = np.array([oracle.qsgd_dither(0x5EED, 2, i) for i in range(2 * n)])
    assert np.all(u >= 0.0) and np.all(u < 1.0)
    assert np.all(u * 2 ** 24 == np.floor(u * 2 ** 24))
    for part in (u[0::2], u[1::2]):
        assert abs(part.mean() - 0.5) < 5 * math.sqrt(1 / 12 / n)
        hist = np.bincount((part * 256).astype(int), minlength=256)
        chi2 = float(((hist - n / 256) ** 2 / (n / 256)).sum())
        assert chi2 < 255 + 5 * math.sqrt(2 * 255)
    for a, b in ((u[0::2], u[1::2]), (u[1:-1:2], u[2::2]), (u[:-2], u[2:])):
        r = np.corrcoef(a, b)[0, 1]
        assert abs(r) < 5 / math.sqrt(a.size)
    # the joint distribution of the pair's fields: 16 x 16 cells
    hist2 = np.bincount((u[0::2] * 16).astype(int) * 16 + (u[1::2] * 16).astype(int), minlength=256)
    chi2 = float(((hist2 - n / 256) ** 2 / (n / 256)).sum())
    assert chi2 < 255 + 5 * math.sqrt(2 * 255)


# ---------------------------------------------------------------- norm

def _exact_rounding_check(v: np.ndarray, r: np.float32) -> None:
    """r must be the fp32 value nearest to sqrt(sum v^2), in exact rationals."""
    X = sum(Fraction(float(x)) ** 2 for x in v)
    r = Fraction(float(r))
    up = Fraction(float(np.nextafter(np.float32(r), np.float32(np.inf))))
    dn = Fraction(float(np.nextafter(np.float32(r), np.float32(0)))) if r > 0 else Fraction(0)
    assert ((r + dn) / 2) ** 2 <= X <= ((r + up) / 2) ** 2


def test_norm_closed_forms():
    assert oracle.l2norm_fp32(np.array([3, 4], np.float32)) == np.float32(5)
    assert oracle.l2norm_fp32(np.array([-2.5], np.float32)) == np.float32(2.5)
    assert oracle.l2norm_fp32(np.zeros(512, np.float32)) == 0
    assert oracle.l2norm_fp32(np.ones(512, np.float32)) == np.float32(math.sqrt(512))
    assert oracle.l2norm_fp32(np.full(4, 0.5, np.float32)) == np.float32(1.0)


def test_norm_is_correctly_rounded_exact_rationals():
    rng = np.random.default_rng(11)
    for trial in range(60):
        n = int(rng.integers(1, 600))
        scale = 10.0 ** rng.uniform(-8, 8)
        v = (rng.normal(0, 1, n) * scale).astype(np.float32)
        if trial % 5 == 0:
            v[rng.random(n) < 0.01] *= 100       # heavy tails as in the workload
        _exact_rounding_check(v, oracle.l2norm_fp32(v))


# ---------------------------------------------------------------- codes

def _parse_codes(codes: np.ndarray, n: int, s: int):
    """Decode sign and level from the byte layout (4-bit: element 2j in the
    high nibble; 8-bit: bit 7 = sign)."""
    sign = np.zeros(n, int)
    level = np.zeros(n, int)
    for i in range(n):
        if s <= 7:
            byte = int(codes[i // 2])
            c = byte >> 4 if i % 2 == 0 else byte & 0xF
            sign[i], level[i] = c >> 3, c & 7
        else:
            c = int(codes[i])
            sign[i], level[i] = c >> 7, c & 0x7F
    return sign, level


def test_code_layout_deterministic_cases():
    # buckets of one element: |v|/||v|| = 1, so the level is s whatever u is
    v = np.array([2.0, -5.0, 0.0], np.float32)
    norms, codes = oracle.qsgd_quantize(v, bucket=1, s=7, seed=3, worker=0)
    np.testing.assert_array_equal(norms, np.array([2, 5, 0], np.float32))
    assert codes.tolist() == [0x7F, 0x00]       # +7 high nibble, -7 low; zero bucket -> 0
    norms, codes = oracle.qsgd_quantize(v, bucket=1, s=127, seed=3, worker=0)
    assert codes.tolist() == [0x7F, 0xFF, 0x00]


def test_zero_bucket_and_negative_zero():
    v = np.zeros(1024, np.float32)
    v[600] = -0.0
    v[700] = 1.0
    norms, codes = oracle.qsgd_quantize(v, bucket=512, s=7, seed=1, worker=2)
    assert norms[0] == 0 and np.all(codes[:256] == 0)
    sign, level = _parse_codes(codes, 1024, 7)
    assert sign[600] == 0            # sgn(-0) = +1
    assert level[700] == 7 and sign[700] == 0


def test_single_nonzero_bucket():
    rng = np.random.default_rng(12)
    for s in (7, 127):
        for trial in range(50):
            v = np.zeros(512, np.float32)
            j = int(rng.integers(0, 512))
            v[j] = np.float32(rng.normal() * 10 ** rng.uniform(-4, 4))
            norms, codes = oracle.qsgd_quantize(v, 512, s, seed=trial, worker=0)
            assert norms[0] == abs(v[j])
            sign, level = _parse_codes(codes, 512, s)
            assert level[j] in (s - 1, s)
            assert sign[j] == int(v[j] < 0)
            assert np.all(level[np.arange(512) != j] == 0)


@pytest.mark.parametrize("s", [7, 127])
def test_level_in_floor_or_floor_plus_one(s):
    """Knowl 1: the level is l or l + 1 where l = floor(|v_i| / ||v|| * s),
    computed here in exact rationals from the stored fp32 norm."""
    rng = np.random.default_rng(13 + s)
    n, d = 2000, 512
    v = rng.normal(0, 1e-2, n).astype(np.float32)
    v[rng.random(n) < 0.01] *= 100
    norms, codes = oracle.qsgd_quantize(v, d, s, seed=99, worker=1)
    sign, level = _parse_codes(codes, n, s)
    for i in range(n):
        a = Fraction(abs(float(v[i]))) / Fraction(float(norms[i // d])) * s
        fl = math.floor(a)
        near_int = abs(a - round(a)) < Fraction(1, 10 ** 5)
        lo, hi = (fl - 1, fl + 2) if near_int else (fl, fl + 1)
        assert max(0, lo) <= level[i] <= min(s, hi)
        assert sign[i] == int(v[i] < 0)


def _dequant_samples(v, d, s, seeds, worker=0):
    out = []
    for seed in seeds:
        norms, codes = oracle.qsgd_quantize(v, d, s, seed=seed, worker=worker)
        out.append(oracle.qsgd_dequant_sum([codes], [norms], v.size, d, s))
    return np.stack(out)


@pytest.mark.parametrize("s", [7, 127])
def test_unbiased_over_1e4_seeds(s):
    """Knowl 1 property 1: E[Q_s(v)] = v.  Over 10^4 seeds the per-coordinate
    mean must sit within 3 sigma, sigma^2 = (norm/s)^2 p (1 - p) / 10^4 with
    p = frac(|v| / norm * s) (Knowl 1 two-point distribution); at least 99%
    of coordinates inside, mean z-score within +-3/sqrt(m)."""
    rng = np.random.default_rng(21)
    d, nb, T = 512, 4, 10_000
    v = rng.normal(0, 1e-2, d * nb).astype(np.float32)
    v[rng.random(v.size) < 0.01] *= 100
    acc = np.zeros(v.size)
    norms = None
    for seed in range(T):
        norms, codes = oracle.qsgd_quantize(v, d, s, seed=seed, worker=0)
        acc += oracle.qsgd_dequant_sum([codes], [norms], v.size, d, s)
    mean = acc / T
    nb_norm = np.repeat(norms.astype(np.float64), d)
    a = np.abs(v.astype(np.float64)) / nb_norm * s
    p = a - np.floor(a)
    sigma = nb_norm / s * np.sqrt(p * (1 - p) / T)
    mask = sigma > 0
    z = (mean[mask] - v.astype(np.float64)[mask]) / sigma[mask]
    assert np.mean(np.abs(z) <= 3) >= 0.99
    assert abs(z.mean()) <= 3 / math.sqrt(z.size) * 1.5
    # coordinates with p == 0 are deterministic: exact
    np.testing.assert_allclose(mean[~mask], v[~mask], rtol=1e-6, atol=0)


@pytest.mark.parametrize("s", [7, 127])
def test_variance_and_sparsity_bounds(s):
    """Knowl 8: E||Q(v_b) - v_b||^2 <= min(d/s^2, sqrt(d)/s) ||v_b||^2 per
    bucket; Knowl 1: E||Q(v)||_0 <= s (s + sqrt(d))."""
    rng = np.random.default_rng(31)
    d, T = 512, 400
    v = rng.normal(0, 1e-2, d).astype(np.float32)
    q = _dequant_samples(v, d, s, range(T))
    err2 = ((q - v.astype(np.float64)) ** 2).sum(axis=1).mean()
    nrm2 = float((v.astype(np.float64) ** 2).sum())
    assert err2 <= min(d / s ** 2, math.sqrt(d) / s) * nrm2 * 1.05
    nnz = (q != 0).sum(axis=1).mean()
    assert nnz <= s * (s + math.sqrt(d))


def test_dequant_sum_is_linear_over_workers_and_scaled():
    rng = np.random.default_rng(41)
    n, d, s, W = 1500, 512, 7, 3
    vs = [rng.normal(0, 1, n).astype(np.float32) for _ in range(W)]
    qs = [oracle.qsgd_quantize(vs[k], d, s, seed=5, worker=k) for k in range(W)]
    singles = [oracle.qsgd_dequant_sum([c], [nm], n, d, s) for nm, c in qs]
    both = oracle.qsgd_dequant_sum([c for _, c in qs], [nm for nm, _ in qs], n, d, s,
                                   scale=0.25)
    np.testing.assert_allclose(both, 0.25 * np.sum(singles, axis=0), rtol=1e-12, atol=0)
    # decode of one worker = norm * sign * level / s, from the byte layout
    nm, c = qs[0]
    sign, level = _parse_codes(c, n, s)
    expect = np.repeat(nm.astype(np.float64), d)[:n] * level / s * np.where(sign == 1, -1, 1)
    np.testing.assert_allclose(singles[0], expect, rtol=1e-15, atol=0)


def test_workers_draw_independent_randomness():
    v = np.full(512, 0.3, np.float32)   # every coordinate has the same fractional part
    _, c0 = oracle.qsgd_quantize(v, 512, 7, seed=5, worker=0)
    _, c1 = oracle.qsgd_quantize(v, 512, 7, seed=5, worker=1)
    _, c0b = oracle.qsgd_quantize(v, 512, 7, seed=5, worker=0)
    assert not np.array_equal(c0, c1)
    np.testing.assert_array_equal(c0, c0b)


def test_ragged_last_bucket_and_odd_n():
    rng = np.random.default_rng(51)
    n, d = 512 * 4 + 297, 512
    v = rng.normal(0, 1, n).astype(np.float32)
    norms, codes = oracle.qsgd_quantize(v, d, 7, seed=1, worker=0)
    assert norms.size == 5 and codes.size == (n + 1) // 2
    _exact_rounding_check(v[4 * d:], norms[4])
    assert codes[-1] & 0x0F == 0        # the unused low nibble of the last byte


def test_tiny_norm_bucket_zero_coordinate_gets_level_zero():
    """When s / norm overflows fp32 (a bucket of subnormal values), a zero
    coordinate still quantises to level 0 (Q_s scales |v_i| = 0) and the
    nonzero ones saturate at s."""
    v = np.zeros(512, np.float32)
    v[:8] = np.float32(1e-40)
    norms, codes = oracle.qsgd_quantize(v, 512, 127, seed=4, worker=0)
    with np.errstate(over="ignore"):
        assert np.isinf(np.float32(127) / norms[0])
    sign, level = _parse_codes(codes, 512, 127)
    assert np.all(level[8:] == 0) and np.all(level[:8] == 127)


@pytest.mark.parametrize("s", [7, 127])
def test_maxnorm_scale_levels_and_unbiasedness(s):
    """Knowl 8 max-norm scaling: the stored scale is max |v| of the bucket,
    the largest coordinate gets level s or s-1, no level exceeds s, and the
    decoded vector is unbiased over 10^4 seeds (3 sigma, as for the l2 form)."""
    rng = np.random.default_rng(77 + s)
    d, nb, T = 512, 2, 10_000
    v = rng.normal(0, 1e-2, d * nb).astype(np.float32)
    v[rng.random(v.size) < 0.01] *= 100
    scales, codes = oracle.qsgd_quantize_maxnorm(v, d, s, seed=1, worker=0)
    for b in range(nb):
        np.testing.assert_array_equal(scales[b], np.max(np.abs(v[b * d:(b + 1) * d])))
    sign, level = _parse_codes(codes, v.size, s)
    assert level.max() <= s
    for b in range(nb):
        j = b * d + int(np.argmax(np.abs(v[b * d:(b + 1) * d])))
        assert level[j] in (s - 1, s)
    acc = np.zeros(v.size)
    for seed in range(T):
        sc, c = oracle.qsgd_quantize_maxnorm(v, d, s, seed=seed, worker=0)
        acc += oracle.qsgd_dequant_sum([c], [sc], v.size, d, s)
    mean = acc / T
    scl = np.repeat(scales.astype(np.float64), d)
    a = np.abs(v.astype(np.float64)) / scl * s
    p = a - np.floor(a)
    sigma = scl / s * np.sqrt(p * (1 - p) / T)
    mask = sigma > 0
    z = (mean[mask] - v.astype(np.float64)[mask]) / sigma[mask]
    assert np.mean(np.abs(z) <= 3) >= 0.99


# ---------------------------------------------------------------- deciding value

def _levels_from_scaled(x: np.ndarray, s: int) -> np.ndarray:
    """Knowl 1's level from the deciding value: min(floor(x), s), and 0 where
    x is NaN (0 * inf: a zero coordinate in a bucket whose s / scale overflows)."""
    lv = np.zeros(x.size, np.int64)
    ok = ~np.isnan(x)
    lv[ok] = np.minimum(np.floor(x[ok].astype(np.float64)), s).astype(np.int64)
    return lv


def _mixed_buckets(rng, d: int) -> np.ndarray:
    """Five buckets and a ragged tail: Gaussian, heavy-tailed, all zero,
    subnormal (s / scale overflows fp32, zeros inside), huge values, and a
    short last bucket of 37 elements."""
    parts = [rng.normal(0, 1, d),
             rng.normal(0, 1e-2, d) * np.where(rng.random(d) < 0.05, 100, 1),
             np.zeros(d),
             np.where(np.arange(d) % 3 == 0, 0.0, 1e-42 * rng.integers(1, 9, d)),
             rng.normal(0, 1e30, d),
             rng.normal(0, 3, 37)]
    return np.concatenate(parts).astype(np.float32)


@pytest.mark.parametrize("maxnorm", [False, True], ids=["l2", "maxnorm"])
@pytest.mark.parametrize("s", [1, 7, 22, 127])
def test_scaled_values_decide_every_written_level(s, maxnorm):
    """The deciding value the GPU tests use to excuse a level that sits on a
    rounding boundary must be the one the quantiser floors: on every element
    of buckets of every kind (zero norm, overflowing s / norm, huge values,
    ragged tail), for a nonzero worker and a bucket-aligned slice at i0 != 0,
    min(floor(x), s) (0 for NaN) equals the level written.  A dropped u, a
    wrong index offset, a worker missing from the seed or the other scale
    would each move levels and fail here."""
    rng = np.random.default_rng(900 + s)
    d = 512
    v = _mixed_buckets(rng, d)
    q = oracle.qsgd_quantize_maxnorm if maxnorm else oracle.qsgd_quantize
    for worker, i0 in ((0, 0), (3, 7 * d), (1, (1 << 33) + 5 * d)):
        x = oracle.qsgd_scaled_values(v, d, s, 42, worker, i0, maxnorm=maxnorm)
        _, codes = q(v, d, s, 42, worker, i0)
        _, level = _parse_codes(codes, v.size, s)
        np.testing.assert_array_equal(_levels_from_scaled(x, s), level.astype(np.int64))
        assert np.all(x[2 * d:3 * d] == 0)                      # the all-zero bucket
        assert np.isnan(x[3 * d]) and level[3 * d] == 0          # 0 * inf in the subnormal bucket
        sub = slice(3 * d + 1, 4 * d)
        assert np.all(np.isinf(x[sub][v[sub] != 0])) and np.all(level[sub][v[sub] != 0] == s)


def test_scaled_values_of_a_slice_equal_the_whole():
    """A bucket-aligned slice decided at its global index i0 gives the same
    deciding values as the same elements of the whole vector."""
    rng = np.random.default_rng(31)
    d = 256
    v = rng.normal(0, 1, 9 * d + 11).astype(np.float32)
    whole = oracle.qsgd_scaled_values(v, d, 7, 5, 2)
    part = oracle.qsgd_scaled_values(v[4 * d:], d, 7, 5, 2, i0=4 * d)
    np.testing.assert_array_equal(part, whole[4 * d:])


def test_scaled_values_single_nonzero_bucket_closed_form():
    """One nonzero coordinate c in a bucket: the l2 norm and the max are |c|
    exactly, so x = fl(|c| * fl(s / |c|)) + u lies within one ulp of s + u,
    and every zero coordinate has x = u, the uniform draw of its own index."""
    d, s = 512, 127
    v = np.zeros(d, np.float32)
    v[100] = np.float32(-0.3)
    for maxnorm in (False, True):
        for worker, i0 in ((0, 0), (3, 7 * d), (1, (1 << 33) + d)):
            x = oracle.qsgd_scaled_values(v, d, s, 9, worker, i0=i0, maxnorm=maxnorm)
            u = np.array([oracle.qsgd_dither(9, worker, i0 + i) for i in range(d)], np.float32)
            zero = np.arange(d) != 100
            np.testing.assert_array_equal(x[zero], u[zero])
            assert abs(float(x[100]) - (s + float(u[100]))) <= 2 * np.spacing(np.float32(s + 1))
