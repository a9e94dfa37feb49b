"""Helpers shared by the GPU parity tests: host views of device buffers,
sentinel-guarded allocations and the float tolerance used throughout.

QSGD levels: both sides decide a level in fp32 from the same deciding value
x = |v| * (s / norm) + u; a level may differ from the oracle's only where x
lies within QSGD_BOUNDARY (absolute) of an integer, and those cases are
counted.

Float tolerance: the floating-point outputs (sums, averages, weight updates,
dequantised values, elastic averaging) must agree with the fp64 oracle within
a relative 1e-5 of the magnitude of the terms that form them,
|gpu - oracle| <= 1e-5 * sum|terms| (elementwise), so that a cancelling sum is
judged against the size of its terms.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle

REL = 1e-5
QSGD_BOUNDARY = 1e-6
SENTINEL = 0x5A5A5A5A


def host_u32(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy().view(np.uint32)


def host_f32(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy().astype(np.float32, copy=False)


def host_bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().view(torch.int16).cpu().numpy().view(np.uint16)


def guarded(n: int, dtype, pad: int = 64, fill: int = SENTINEL, device="cuda") -> torch.Tensor:
    """A device buffer of n + pad elements whose tail is a sentinel pattern;
    ``check_guard`` verifies nothing wrote past element n."""
    itemsize = torch.empty(0, dtype=dtype).element_size()
    nbytes = (n + pad) * itemsize
    raw = torch.empty((nbytes + 3) // 4 * 4, dtype=torch.uint8, device=device)
    raw.view(torch.int32).fill_(int(np.uint32(fill).view(np.int32)))
    return raw[:nbytes].view(dtype)


def check_guard(buf: torch.Tensor, n: int, fill: int = SENTINEL) -> None:
    tail = buf[n:].detach().cpu().contiguous().view(torch.uint8).numpy()
    pattern = np.frombuffer(np.uint32(fill).tobytes() * (tail.size // 4 + 2), dtype=np.uint8)
    byte_off = n * buf.element_size()
    # the sentinel repeats every 4 bytes from the start of the buffer
    phase = byte_off % 4
    assert np.array_equal(tail, pattern[phase:phase + tail.size]), "write past the end of a buffer"


def assert_close(gpu: np.ndarray, ref: np.ndarray, scale: np.ndarray, rel: float = REL,
                 what: str = "") -> None:
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    scale = np.broadcast_to(np.asarray(scale, dtype=np.float64), ref.shape)
    err = np.abs(gpu - ref)
    bad = err > rel * scale + 1e-30
    if bad.any():
        i = int(np.argmax(bad))
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} beyond rel {rel}; first at "
                             f"{i}: gpu={gpu[i]!r} ref={ref[i]!r} scale={scale[i]!r}")


def sample_chunks(n: int, count: int, size: int, align: int = 16, seed: int = 0):
    """Deterministic list of [lo, hi) element ranges spread over [0, n): the
    first and last elements are always covered; lo is a multiple of ``align``."""
    rng = np.random.default_rng(seed)
    size = min(size, n)
    out = [(0, size)]
    last_lo = max(0, ((n - size) // align) * align)
    out.append((last_lo, n))
    for lo in sorted(rng.integers(0, max(1, n - size), count - 2)):
        lo = int(lo) // align * align
        out.append((lo, min(n, lo + size)))
    # merge overlaps
    out.sort()
    merged = []
    for lo, hi in out:
        if merged and lo <= merged[-1][1]:
            merged[-1] = (merged[-1][0], max(merged[-1][1], hi))
        else:
            merged.append((lo, hi))
    return merged


def qsgd_levels(codes: np.ndarray, n: int, s: int):
    """(sign, level) arrays of n elements from packed QSGD codes (4-bit codes
    two per byte, element 2j in the high nibble; 8-bit codes, bit 7 = sign)."""
    if s <= 7:
        hi = (codes >> 4) & 0xF
        lo = codes & 0xF
        c = np.empty(2 * codes.size, np.uint8)
        c[0::2], c[1::2] = hi, lo
        c = c[:n]
        return c >> 3, c & 7
    return codes[:n] >> 7, codes[:n] & 0x7F


def compare_codes(gpu_codes, ref_codes, v, n, bucket, s, seed, worker, i0=0, maxnorm=False):
    """Asserts the GPU's QSGD codes equal the oracle's except for levels that
    differ by one where the oracle's deciding value x lies within
    QSGD_BOUNDARY of the integer between them; signs must agree everywhere.
    Returns (mismatch count, boolean mask of the mismatched elements)."""
    if np.array_equal(gpu_codes, ref_codes):
        return 0, np.zeros(n, bool)
    gs, gl = qsgd_levels(gpu_codes, n, s)
    rs, rl = qsgd_levels(ref_codes, n, s)
    assert np.array_equal(gs, rs), "sign bits differ"
    bad = gl != rl
    x = oracle.qsgd_scaled_values(v, bucket, s, seed, worker, i0, maxnorm=maxnorm)[bad]
    k = np.maximum(gl[bad], rl[bad]).astype(np.float64)
    assert np.all(np.abs(gl[bad].astype(int) - rl[bad].astype(int)) == 1), "levels differ by more than one"
    assert np.all(np.abs(x.astype(np.float64) - k) <= QSGD_BOUNDARY), \
        "a level differs where the deciding value is not within 1e-6 of a rounding boundary"
    if s <= 7 and n % 2:
        assert gpu_codes[-1] & 0xF == 0
    return int(bad.sum()), bad


def qsgd_sum_reference(codes_list, norms_list, n: int, bucket: int, s: int, scale: float):
    """The oracle's dequantise-sum of the given (host) codes and norms, and the
    tolerance scale: scale * sum over workers of |each worker's decoded value|.
    The GPU tests pass the GPU's own codes and norms, so every element of the
    GPU sum is compared, boundary-case levels included."""
    ref = oracle.qsgd_dequant_sum(codes_list, norms_list, n, bucket, s, scale)
    terms = np.zeros(n)
    for c, nm in zip(codes_list, norms_list):
        terms += np.abs(oracle.qsgd_dequant_sum([c], [nm], n, bucket, s))
    return ref, abs(float(np.float32(scale))) * terms
