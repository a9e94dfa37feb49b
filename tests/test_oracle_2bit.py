"""Pins for the oracle's 2-bit threshold quantiser, its dequantise-sum-update
and the CD-SGD correction step.

Sources: "2bit gradient compression" (MXNet PR #8662), sections "Two bit
quantization", "Format of compressed gradient", "Local kvstore"; "CD-SGD"
eq. 1, eq. 10, Algorithm 1 and section 3.4.1 (no data loss in quantisation).
None of these checks re-types the oracle's formula: they use the printed word,
the binary string notation the page prints, exact conservation laws on dyadic
inputs and closed-form special cases.
"""
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "mxnet_2bit_format.txt")


def _golden():
    vals = {}
    with open(GOLDEN) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            key, rest = line.split(" ", 1)
            vals[key] = rest.strip()
    return vals


def _bit_groups(word: int) -> list[str]:
    s = format(int(word), "032b")
    return [s[2 * j: 2 * j + 2] for j in range(16)]


def test_printed_example_word():
    g = _golden()
    t = float(g["threshold"])
    # pattern 0, +, 0, -, +, 0, 0, -   (values exactly at +-t included)
    grad = np.array([0.5, 2.0, -1.0, -2.5, 3.0, 1.9, -1.9, -2.0], dtype=np.float32)
    r = np.zeros(8, dtype=np.float32)
    codes = oracle.twobit_quantize(grad, r, t)
    assert codes.shape == (1,)
    printed = g["word_bits"].replace(" ", "")
    assert format(int(codes[0]), "032b") == printed
    assert int(codes[0]) == int(g["word_hex"], 16)
    # the quantisation error stays in the residual
    np.testing.assert_array_equal(r, np.array([0.5, 0.0, -1.0, -0.5, 1.0, 1.9, -1.9, 0.0],
                                              dtype=np.float32))


@pytest.mark.parametrize("fill,expected", [(0.0, 0x00000000), (0.75, 0xFFFFFFFF),
                                           (-0.75, 0xAAAAAAAA)])
def test_uniform_words(fill, expected):
    grad = np.full(16, fill, dtype=np.float32)
    r = np.zeros(16, dtype=np.float32)
    codes = oracle.twobit_quantize(grad, r, 0.5)
    assert int(codes[0]) == expected


def test_first_and_last_element_positions():
    t = 0.5
    g = np.zeros(16, dtype=np.float32)
    g[0] = 1.0
    assert int(oracle.twobit_quantize(g, np.zeros(16, np.float32), t)[0]) == 0xC0000000
    g = np.zeros(16, dtype=np.float32)
    g[15] = -1.0
    assert int(oracle.twobit_quantize(g, np.zeros(16, np.float32), t)[0]) == 0x00000002


def test_ties_and_just_below_threshold():
    t = np.float32(0.5)
    below = np.nextafter(t, np.float32(0))
    g = np.array([t, -t, below, -below], dtype=np.float32)
    r = np.zeros(4, np.float32)
    codes = oracle.twobit_quantize(g, r, float(t))
    assert _bit_groups(codes[0])[:4] == ["11", "10", "00", "00"]
    np.testing.assert_array_equal(r, np.array([0, 0, below, -below], np.float32))


def test_brute_force_classes_against_string_notation():
    """Every element position with every class, plus random mixtures: the word's
    printed binary string (2-bit groups, first element first) must spell the
    classes, and the tail beyond n must read 00."""
    rng = np.random.default_rng(1)
    t = 1.0
    cls_val = {"11": 1.5, "10": -1.5, "00": 0.25}
    for trial in range(400):
        n = int(rng.integers(1, 64))
        labels = rng.choice(["11", "10", "00"], size=n)
        g = np.array([cls_val[c] for c in labels], dtype=np.float32)
        codes = oracle.twobit_quantize(g, np.zeros(n, np.float32), t)
        assert codes.size == (n + 15) // 16
        groups = [grp for w in codes for grp in _bit_groups(w)]
        assert groups[:n] == list(labels)
        assert all(grp == "00" for grp in groups[n:])


def _dyadic(rng, shape, scale_pow=8, bound=8):
    return (rng.integers(-bound * 2 ** scale_pow, bound * 2 ** scale_pow + 1, size=shape)
            / 2.0 ** scale_pow).astype(np.float32)


def _decode_string(codes, n, t):
    """Decode through the binary-string notation: 11 -> +t, 10 -> -t, else 0."""
    groups = [grp for w in codes for grp in _bit_groups(w)][:n]
    m = {"11": t, "10": -t}
    return np.array([m.get(grp, 0.0) for grp in groups], dtype=np.float64)


def test_conservation_exact_on_dyadic_inputs():
    """No data loss: sum of transmitted (dequantised) values plus the final
    residual equals the sum of all gradients, exactly (every intermediate is
    a dyadic rational representable in fp32)."""
    rng = np.random.default_rng(2)
    n, steps, t = 1000, 12, 0.5
    r = np.zeros(n, np.float32)
    sent = np.zeros(n)
    total = np.zeros(n)
    for _ in range(steps):
        g = _dyadic(rng, n)
        total += g
        codes = oracle.twobit_quantize(g, r, t)
        sent += _decode_string(codes, n, t)
    np.testing.assert_array_equal(sent + r.astype(np.float64), total)


def test_residual_bounded_by_threshold():
    """With |g| < t and |r| < t the residual stays inside (-t, t)."""
    rng = np.random.default_rng(3)
    n, t = 4096, 0.5
    r = np.zeros(n, np.float32)
    for _ in range(20):
        g = rng.uniform(-0.49, 0.49, n).astype(np.float32)
        oracle.twobit_quantize(g, r, t)
        assert np.all(np.abs(r) < t)


def test_bf16_matches_fp32_of_same_values():
    rng = np.random.default_rng(4)
    n = 777
    g32 = rng.normal(0, 1, n).astype(np.float32)
    bits = (g32.view(np.uint32) >> 16).astype(np.uint16)        # truncate to bf16
    g_from_bits = (bits.astype(np.uint32) << 16).view(np.float32)
    r1 = np.zeros(n, np.float32)
    r2 = np.zeros(n, np.float32)
    c1 = oracle.twobit_quantize(bits, r1, 0.5)
    c2 = oracle.twobit_quantize(g_from_bits, r2, 0.5)
    np.testing.assert_array_equal(c1, c2)
    np.testing.assert_array_equal(r1, r2)


def test_dequant_single_worker_values():
    rng = np.random.default_rng(5)
    n, t = 333, 0.5
    labels = rng.choice(["11", "10", "00"], size=n)
    g = np.array([{"11": 0.9, "10": -0.9, "00": 0.1}[c] for c in labels], np.float32)
    codes = oracle.twobit_quantize(g, np.zeros(n, np.float32), t)
    out = oracle.twobit_dequant_sum_update([codes], n, t, oracle.KIND_NONE)
    expect = np.array([{"11": t, "10": -t, "00": 0.0}[c] for c in labels])
    np.testing.assert_array_equal(out, expect)


def test_dequant_code_01_reads_zero():
    codes = np.array([0x40000000 | 0x3], dtype=np.uint32)  # element 0 = 01, element 15 = 11
    out = oracle.twobit_dequant_sum_update([codes], 16, 0.25, oracle.KIND_NONE)
    assert out[0] == 0.0 and out[15] == 0.25 and np.all(out[1:15] == 0.0)


def test_dequant_sum_counts_classes():
    """avg * W / t is the integer (#workers sending +) - (#workers sending -)."""
    rng = np.random.default_rng(6)
    n, W, t = 517, 8, 2e-3
    labels = rng.choice([1, -1, 0], size=(W, n))
    codes = []
    for k in range(W):
        g = (labels[k] * 3e-3 + (labels[k] == 0) * 1e-3).astype(np.float32)
        codes.append(oracle.twobit_quantize(g, np.zeros(n, np.float32), t))
    out = oracle.twobit_dequant_sum_update(codes, n, t, oracle.KIND_NONE)
    count = np.rint(out * W / np.float64(np.float32(t)))
    np.testing.assert_array_equal(count, labels.sum(axis=0))
    assert np.all(np.abs(out * W / np.float32(t) - count) < 1e-9)


def test_sgd_update_closed_forms():
    n, W, t = 64, 4, 0.5
    ones = np.full(n, 1.0, np.float32)
    codes = [oracle.twobit_quantize(ones, np.zeros(n, np.float32), t) for _ in range(W)]
    w0 = np.linspace(-1, 1, n)
    # lr = 0: weights unchanged bit for bit
    w = w0.copy()
    oracle.twobit_dequant_sum_update(codes, n, t, oracle.KIND_SGD, lr=0.0, weights=w)
    np.testing.assert_array_equal(w, w0)
    # every worker sends +t: avg = t, eq. 10 gives w - lr * t
    w = w0.copy()
    lr = 0.25
    oracle.twobit_dequant_sum_update(codes, n, t, oracle.KIND_SGD, lr=lr, weights=w)
    np.testing.assert_array_equal(w, w0 - lr * t)
    # half the workers send +t, half -t: avg = 0
    neg = [oracle.twobit_quantize(-ones, np.zeros(n, np.float32), t) for _ in range(W // 2)]
    w = w0.copy()
    oracle.twobit_dequant_sum_update(codes[:W // 2] + neg, n, t, oracle.KIND_SGD, lr=lr,
                                     weights=w)
    np.testing.assert_array_equal(w, w0)


def test_easgd_kind_closed_forms():
    n, t = 32, 0.5
    zeros = np.zeros(n, np.float32)
    codes = [oracle.twobit_quantize(zeros, np.zeros(n, np.float32), t)]
    w0 = np.linspace(-1, 1, n)
    c = np.linspace(2, 3, n)
    w = w0.copy()
    oracle.twobit_dequant_sum_update(codes, n, t, oracle.KIND_EASGD, lr=0.5, alpha=1.0,
                                     center=c, weights=w)
    np.testing.assert_allclose(w, c, rtol=0, atol=1e-15)   # alpha = 1 pulls onto the center
    w = w0.copy()
    oracle.twobit_dequant_sum_update(codes, n, t, oracle.KIND_EASGD, lr=0.5, alpha=0.5,
                                     center=c, weights=w)
    np.testing.assert_allclose(w, (w0 + c) / 2, rtol=0, atol=1e-15)


def test_correction_step_is_plain_ssgd_when_residual_empty():
    """eq. 1: with empty residuals the correction step is W - eta/N sum g."""
    rng = np.random.default_rng(7)
    n, W, lr = 300, 4, 0.125
    grads = [_dyadic(rng, n) for _ in range(W)]
    res = [np.zeros(n, np.float32) for _ in range(W)]
    w = np.linspace(-1, 1, n)
    w_expect = w - lr * np.mean(np.stack(grads).astype(np.float64), axis=0)
    oracle.compensated_sum_update(grads, res, lr, w)
    np.testing.assert_array_equal(w, w_expect)
    for r in res:
        assert np.all(r == 0)


def test_cdsgd_k_step_conservation():
    """Eight steps with k = 4 (steps 4 and 8 full precision): residuals are empty
    after a correction step and the total weight change is exactly
    -lr/W * (sum of all gradients - final residuals)."""
    rng = np.random.default_rng(8)
    n, W, t, lr, k = 500, 4, 0.5, 0.0625, 4
    res = [np.zeros(n, np.float32) for _ in range(W)]
    w0 = _dyadic(rng, n).astype(np.float64)
    w = w0.copy()
    total = np.zeros(n)
    for step in range(1, 8 + 1):
        grads = [_dyadic(rng, n, bound=2) for _ in range(W)]
        total += np.sum(np.stack(grads).astype(np.float64), axis=0)
        if step % k != 0:
            codes = [oracle.twobit_quantize(grads[q], res[q], t) for q in range(W)]
            oracle.twobit_dequant_sum_update(codes, n, t, oracle.KIND_SGD, lr=lr, weights=w)
        else:
            oracle.compensated_sum_update(grads, res, lr, w)
            for r in res:
                assert np.all(r == 0)
    final_res = np.sum(np.stack(res).astype(np.float64), axis=0)
    np.testing.assert_array_equal(w, w0 - lr / W * (total - final_res))


def test_correction_with_bf16_gradients():
    rng = np.random.default_rng(9)
    n, W = 100, 2
    g32 = [rng.normal(0, 1, n).astype(np.float32) for _ in range(W)]
    bits = [(g.view(np.uint32) >> 16).astype(np.uint16) for g in g32]
    asf = [(b.astype(np.uint32) << 16).view(np.float32) for b in bits]
    r0 = [rng.normal(0, 0.1, n).astype(np.float32) for _ in range(W)]
    ra = [r.copy() for r in r0]
    rb = [r.copy() for r in r0]
    wa = np.zeros(n)
    wb = np.zeros(n)
    oracle.compensated_sum_update(bits, ra, 0.01, wa)
    oracle.compensated_sum_update(asf, rb, 0.01, wb)
    np.testing.assert_array_equal(wa, wb)


def test_local_update_pins():
    """CD-SGD eq. 11: lr = 0 or g = 0 leaves the local copy equal to the
    global weights; on dyadic inputs (w - local) / lr is the gradient exactly;
    bf16 bits give the same as their fp32 values."""
    rng = np.random.default_rng(12)
    n = 400
    w = _dyadic(rng, n).astype(np.float64)
    g = _dyadic(rng, n)
    np.testing.assert_array_equal(oracle.cdsgd_local_update(g, w, 0.0), w)
    np.testing.assert_array_equal(oracle.cdsgd_local_update(np.zeros(n, np.float32), w, 0.1), w)
    loc = oracle.cdsgd_local_update(g, w, 0.125)
    np.testing.assert_array_equal((w - loc) / 0.125, g.astype(np.float64))
    bits = (g.view(np.uint32) >> 16).astype(np.uint16)
    asf = (bits.astype(np.uint32) << 16).view(np.float32)
    np.testing.assert_array_equal(oracle.cdsgd_local_update(bits, w, 0.1), oracle.cdsgd_local_update(asf, w, 0.1))
