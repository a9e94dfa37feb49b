"""The Elias decoders' CTA sizing rule (host logic, no GPU): a decoding thread
walks one bucket's stream ("QSGD ...", Knowl 2, dense and sparse regimes), so
an SM's time is the number of buckets it holds, and the decoders choose the
buckets per CTA so that the grid fills the fewest waves of resident CTAs with
the buckets spread evenly.  Checked here through the library's testing hook,
against brute force on small sizes and on the 61.1 M-coordinate QSGD
workload's sizes."""
import ctypes
import itertools

import pytest

import gradient_compression_sgd_gc_gb300 as gc


def _bpc(nb, W, slots, maxb):
    out = ctypes.c_int64(-7)
    rc = gc.load().gc_testing_decode_buckets_per_cta(nb, W, slots, maxb, ctypes.byref(out))
    return rc, out.value


def _ceil(a, b):
    return -(-a // b)


def test_qsgd_workload_sizes():
    nb = _ceil(61_100_840, 512)                                      # 119,338 buckets
    assert _bpc(nb, 1, 152 * 4, 256) == (gc.GC_OK, 197)             # 4-bit codes: 606 CTAs, one wave
    assert _bpc(nb, 1, 152 * 1, 1024) == (gc.GC_OK, 786)            # 8-bit codes: 152 CTAs, one per SM
    assert _bpc(nb, 4, 152 * 4, 256) == (gc.GC_OK, 197)             # four streams: four waves
    assert _ceil(nb, 197) == 606 and _ceil(nb, 786) == 152


def test_rule_against_brute_force():
    """bpc <= maxb; the grid takes the fewest waves any CTA size up to maxb
    allows; and bpc is the smallest size that fits those waves (one bucket
    fewer per CTA would need more CTAs than the waves hold)."""
    for nb, W, slots, maxb in itertools.product(list(range(1, 40)) + [97, 256, 257, 1000, 4099],
                                                (1, 2, 3, 4, 64), (1, 3, 8, 152, 608), (1, 2, 7, 32, 256)):
        rc, b = _bpc(nb, W, slots, maxb)
        assert rc == gc.GC_OK and 1 <= b <= maxb, (nb, W, slots, maxb, b)
        waves_min = min(_ceil(W * _ceil(nb, c), slots) for c in range(1, maxb + 1))
        assert _ceil(W * _ceil(nb, b), slots) == waves_min, (nb, W, slots, maxb, b)
        if b > 1:
            assert W * _ceil(nb, b - 1) > slots * waves_min, (nb, W, slots, maxb, b)


def test_spread_is_even_within_one_bucket():
    """In the waves used, no CTA holds more than one bucket above the mean
    (nb * W buckets over W * ceil(nb / bpc) CTAs)."""
    for nb, W, slots, maxb in ((119_338, 1, 608, 256), (119_338, 1, 152, 1024), (5000, 3, 152, 256),
                               (131_072, 2, 608, 256), (999, 1, 1000, 1024)):
        _, b = _bpc(nb, W, slots, maxb)
        grid = _ceil(nb, b)
        assert b - nb / grid < 1.0 + 1e-9 or grid == 1


@pytest.mark.parametrize("args", [(0, 1, 152, 256), (-1, 1, 152, 256), (10, 0, 152, 256),
                                  (10, gc.GC_MAX_WORKERS + 1, 152, 256), (10, 1, 0, 256), (10, 1, 152, 0),
                                  (10, 1, 152, 1025), (1 << 41, 1, 152, 256), (10, 1, 1 << 21, 256)])
def test_invalid_arguments(args):
    assert _bpc(*args)[0] == gc.GC_ERR_INVALID
    assert gc.load().gc_testing_decode_buckets_per_cta(10, 1, 152, 256, None) == gc.GC_ERR_INVALID
