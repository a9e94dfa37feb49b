"""Pins for the oracle's QSGD Elias coding in the sparse regimes.

Source: "QSGD: Communication-Efficient SGD via Gradient Quantization and
Encoding" (summary page), Knowl 2: items 1 (s >= 2: the distances between
non-zero coordinates are coded with Elias omega, and the expected length of
a bucket is at most (3 + (3/2 + o(1)) log2(2 (s^2 + n) / (s (s + sqrt n))))
s (s + sqrt n) + 32 bits) and 1' (s = 1, levels in {-1, 0, 1}).  The stream
layout is pinned to hand-assembled words (tests/golden/
qsgd_elias_sparse_streams.txt); the codewords themselves are pinned in
test_oracle_elias.py against a table written out from Elias (1975).
"""
import math
import os

import numpy as np
import pytest

import oracle
from test_oracle_elias import GOLDEN, _canonical, _codewords, _pack, _unpack


def _sparse_streams():
    out = []
    with open(os.path.join(GOLDEN, "qsgd_elias_sparse_streams.txt")) as f:
        for line in f:
            if line.startswith("stream"):
                lhs, rhs = line.split("->")
                _, s, norm, *pairs = lhs.split()
                codes = [tuple(int(x) for x in p.split(",")) for p in pairs]
                out.append((int(s), float(norm), codes, [int(w, 16) for w in rhs.split()]))
    return out


@pytest.mark.parametrize("case", range(4))
def test_sparse_stream_matches_hand_assembled(case):
    s, norm, codes, words = _sparse_streams()[case]
    n = len(codes)
    buf = _pack(codes, s)
    w, off = oracle.qsgd_elias_encode_sparse(buf, np.array([norm], np.float32), n, n, s)
    assert w.tolist() == words
    assert off.tolist() == [0, len(words)]
    dc, dn, bad = oracle.qsgd_elias_decode_sparse(w, off, n, n, s)
    assert bad == 0
    assert dn.view(np.uint32)[0] == np.float32(norm).view(np.uint32)
    np.testing.assert_array_equal(dc, _canonical(buf, n, s))


def test_sparse_two_buckets_ragged_offsets():
    """Two buckets of 8 and a ragged third of 3 (the first and the last worked
    streams): the stream is their concatenation, each on its own word."""
    s0, n0, c0, w0 = _sparse_streams()[0]
    _, n3, c3, w3 = _sparse_streams()[3]
    codes = c0 + c0 + c3
    buf = _pack(codes, 7)
    norms = np.array([n0, n0, n3], np.float32)
    w, off = oracle.qsgd_elias_encode_sparse(buf, norms, len(codes), 8, 7)
    assert w.tolist() == w0 + w0 + w3
    assert off.tolist() == [0, 2, 4, 6]
    dc, dn, bad = oracle.qsgd_elias_decode_sparse(w, off, len(codes), 8, 7)
    assert bad == 0
    np.testing.assert_array_equal(dc, _canonical(buf, len(codes), 7))


def test_omega_length_bound_behind_the_capacity():
    """The capacity qsgd_elias_sparse_max_words allows 18 bits per coordinate;
    it rests on |omega(g)| <= g + 2 for every distance g >= 1 (the distances of
    a bucket sum to its length)."""
    for g in range(1, 4097):
        assert len(oracle.elias_omega(g)) <= g + 2, g
    assert len(oracle.elias_omega(128)) == 14                 # the longest level code (s = 127)


@pytest.mark.parametrize("s,d,n", [(1, 128, 1000), (2, 512, 3 * 512 + 41), (7, 512, 4 * 512 + 297),
                                   (22, 512, 3 * 512 + 1), (127, 2048, 2 * 2048 + 33)])
def test_sparse_roundtrip_and_lengths(s, d, n):
    """Round trip of the quantiser's codes (level-0 signs cleared), and every
    bucket's word count from the codeword table: 32 + for each non-zero
    coordinate |omega(distance)| + 1 + (s >= 2) |omega(level)|, plus the
    closing distance."""
    rng = np.random.default_rng(s * 77 + d)
    v = rng.standard_normal(n).astype(np.float32) * 1e-2
    v[rng.random(n) < 0.01] *= 100
    v[:50] = 0.0
    v[60:70] = -0.0
    norms, codes = oracle.qsgd_quantize(v, d, s, seed=5, worker=1)
    w, off = oracle.qsgd_elias_encode_sparse(codes, norms, n, d, s)
    table = _codewords()

    def omega_len(g):
        # from the table where it reaches; above it, omega(N) is the code of
        # bitlength(N) - 1 followed by N's binary digits (Elias 1975)
        bl = int(g).bit_length()
        key = 1 << (bl - 1)
        return len(table[key]) if key in table else bl + omega_len(bl - 1)

    _, lv = _unpack(codes, n, s)
    for b in range((n + d - 1) // d):
        seg = lv[b * d:(b + 1) * d]
        bits, p = 32, -1
        for i in np.nonzero(seg)[0]:
            bits += omega_len(i - p) + 1 + (omega_len(seg[i]) if s >= 2 else 0)
            p = i
        bits += omega_len(len(seg) - p)
        assert int(off[b + 1]) - int(off[b]) == (bits + 31) // 32
    dc, dn, bad = oracle.qsgd_elias_decode_sparse(w, off, n, d, s)
    assert bad == 0
    np.testing.assert_array_equal(dc, _canonical(codes, n, s))
    np.testing.assert_array_equal(dn.view(np.uint32), norms.view(np.uint32))
    assert w.size <= oracle.qsgd_elias_sparse_max_words(n, d)


def test_overshooting_distance_is_reported():
    """A stream whose distance runs past the bucket's end is not one the
    encoder writes: the decoder counts the bucket."""
    s, norm, codes, words = _sparse_streams()[0]
    bad_words = list(words)
    bad_words[1] = 0xFC000000          # omega(15) = 11 1111 0: jumps past the 8 coordinates
    _, _, bad = oracle.qsgd_elias_decode_sparse(np.array(bad_words, np.uint32), np.array([0, 2], np.uint32),
                                                8, 8, s)
    assert bad == 1


@pytest.mark.parametrize("s", [2, 7, 22])
def test_sparse_mean_length_within_the_pages_bound(s):
    """Knowl 2 item 1: the expected length of a bucket of d coordinates is at
    most (3 + (3/2 + o(1)) log2(2(s^2 + d)/(s(s + sqrt d)))) s (s + sqrt d) + 32
    bits; with o(1) = 0 the mean over 40 seeds on Gaussian buckets must stay
    below it (the code used here is well under)."""
    d, nb = 512, 16
    v = np.random.default_rng(s).standard_normal(d * nb).astype(np.float32)
    bound = (3 + 1.5 * math.log2(2 * (s * s + d) / (s * (s + math.sqrt(d))))) * s * (s + math.sqrt(d)) + 32
    total = 0
    for seed in range(40):
        nr, codes = oracle.qsgd_quantize(v, d, s, seed=(seed + 1) * 0x9E3779B97F4A7C15 % 2 ** 64, worker=0)
        w, off = oracle.qsgd_elias_encode_sparse(codes, nr, d * nb, d, s)
        total += 32 * w.size
    assert total / 40 / nb <= bound, (total / 40 / nb, bound)


def test_ternary_sparse_stream_is_shorter_than_dense():
    """With s = 1 most levels are 0 and no level is sent: the sparse stream of
    a Gaussian bucket is a fraction of the dense one (which spends at least a
    bit on every coordinate)."""
    d, nb = 512, 8
    v = np.random.default_rng(3).standard_normal(d * nb).astype(np.float32)
    nr, codes = oracle.qsgd_quantize(v, d, 1, seed=9, worker=0)
    ws, _ = oracle.qsgd_elias_encode_sparse(codes, nr, d * nb, d, 1)
    wd, _ = oracle.qsgd_elias_encode(codes, nr, d * nb, d, 1)
    assert ws.size < 0.5 * wd.size
