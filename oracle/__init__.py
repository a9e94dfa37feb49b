"""CPU oracle for the gradient-compression hot path (test infrastructure).

This package is TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline legs of ``bench.py`` may import it.  The product library
(``gradient_compression_sgd_gc_gb300``) never imports, links or executes
anything here, and this package never imports the product.

The arithmetic lives in ``oracle.c`` (plain C, compiled ``-O2
-ffp-contract=off``); this module only builds it with gcc and marshals numpy
arrays through ctypes.  Every function cites the page passage it follows in
``oracle.c``.

Pins: every function here is checked by ``tests/test_oracle_*.py`` against
values printed on the pages, closed forms, invariants, exact rational
arithmetic or brute force (none of them re-types the oracle's own formula).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_CFLAGS = ["-O2", "-ffp-contract=off", "-fno-fast-math", "-std=c11", "-fPIC", "-shared"]

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into ``oracle/_build/liboracle.so`` (gcc, this host's arch)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    fresh = os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)
    if fresh and not force:
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", *_CFLAGS, _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = build()
        lib = ctypes.CDLL(path)
        u64, i64, i32, f32, f64, vp = (ctypes.c_uint64, ctypes.c_int64, ctypes.c_int,
                                       ctypes.c_float, ctypes.c_double, ctypes.c_void_p)
        sig = {
            "orc_splitmix64": (u64, [u64]),
            "orc_uniform": (f64, [u64]),
            "orc_qsgd_dither": (f64, [u64, u64]),
            "orc_round_seed": (u64, [u64, u64]),
            "orc_2bit_quantize": (None, [vp, i32, vp, vp, i64, f32]),
            "orc_2bit_dequant_sum_update": (None, [vp, i32, i64, f32, i32, f64, f64, vp, vp, vp]),
            "orc_compensated_sum_update": (None, [vp, i32, vp, i32, i64, f64, vp]),
            "orc_cdsgd_local_update": (None, [vp, i32, vp, vp, i64, f64]),
            "orc_l2norm_fp32": (f32, [vp, i64]),
            "orc_qsgd_quantize": (None, [vp, i64, i64, i32, u64, i32, i64, vp, vp]),
            "orc_qsgd_scaled_values": (None, [vp, i64, i64, i32, u64, i32, i64, vp]),
            "orc_easgd_step_from_sum": (None, [vp, vp, i32, i64, f64, f64, vp]),
            "orc_qsgd_scaled_values_maxnorm": (None, [vp, i64, i64, i32, u64, i32, i64, vp]),
            "orc_qsgd_quantize_maxnorm": (None, [vp, i64, i64, i32, u64, i32, i64, vp, vp]),
            "orc_elias_omega_bits": (i32, [ctypes.c_uint32, ctypes.c_char_p]),
            "orc_qsgd_elias_encode": (i64, [vp, vp, i64, i64, i32, vp, vp]),
            "orc_qsgd_elias_decode": (None, [vp, vp, i64, i64, i32, vp, vp]),
            "orc_qsgd_elias_quarter_marks": (None, [vp, i64, i64, i32, vp]),
            "orc_qsgd_elias_encode_sparse": (i64, [vp, vp, i64, i64, i32, vp, vp]),
            "orc_qsgd_elias_decode_sparse": (i64, [vp, vp, i64, i64, i32, vp, vp]),
            "orc_qsgd_dequant_sum": (None, [vp, vp, i32, i64, i64, i32, f64, vp]),
            "orc_saps_mask_compact": (i64, [i64, f64, u64, vp, i32, i64, vp, vp, i64]),
            "orc_saps_matching": (i32, [u64, i32, vp]),
            "orc_saps_peer_average": (None, [vp, vp, vp, i64, vp, i32]),
            "orc_easgd_step": (None, [vp, i32, i64, f64, f64, vp]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def _check(a: np.ndarray, dtype, name: str, size: int | None = None) -> None:
    if not isinstance(a, np.ndarray) or a.dtype != np.dtype(dtype):
        raise TypeError(f"{name}: expected numpy {np.dtype(dtype)}, got {getattr(a, 'dtype', type(a))}")
    if not a.flags.c_contiguous:
        raise ValueError(f"{name}: must be C-contiguous")
    if size is not None and a.size < size:
        raise ValueError(f"{name}: needs at least {size} elements, has {a.size}")


def _ptr_array(arrays):
    return (ctypes.c_void_p * len(arrays))(*[a.ctypes.data for a in arrays])


# --------------------------------------------------------------------------
# counter-based random numbers
# --------------------------------------------------------------------------

def splitmix64(x: int) -> int:
    return int(_load().orc_splitmix64(x & 0xFFFFFFFFFFFFFFFF))


def uniform(key: int) -> float:
    return float(_load().orc_uniform(key & 0xFFFFFFFFFFFFFFFF))


def qsgd_dither(seed: int, worker: int, i: int) -> float:
    """QSGD's dither u of global element index i for (seed, worker): one
    SplitMix64 output per pair of elements (see orc_qsgd_dither)."""
    seed_w = (seed ^ ((worker & 0xFFFFFFFF) << 48)) & 0xFFFFFFFFFFFFFFFF
    return float(_load().orc_qsgd_dither(seed_w, i & 0xFFFFFFFFFFFFFFFF))


def round_seed(base: int, t: int) -> int:
    return int(_load().orc_round_seed(base & 0xFFFFFFFFFFFFFFFF, t & 0xFFFFFFFFFFFFFFFF))


# --------------------------------------------------------------------------
# 2-bit threshold quantisation
# --------------------------------------------------------------------------

def _grad_kind(g: np.ndarray) -> int:
    """0 for fp32 gradients, 1 for bf16 gradients held as raw uint16 bits."""
    if g.dtype == np.float32:
        return 0
    if g.dtype == np.uint16:
        return 1
    raise TypeError("gradient must be float32 or bf16 bits as uint16")


def twobit_quantize(grad: np.ndarray, residual: np.ndarray, threshold: float) -> np.ndarray:
    """Quantise in place: updates ``residual`` (fp32), returns uint32 codes [ceil(n/16)]."""
    n = grad.size
    kind = _grad_kind(grad)
    _check(grad, grad.dtype, "grad")
    _check(residual, np.float32, "residual", n)
    codes = np.zeros((n + 15) // 16, dtype=np.uint32)
    _load().orc_2bit_quantize(_ptr(grad), kind, _ptr(residual), _ptr(codes), n,
                              ctypes.c_float(np.float32(threshold)))
    return codes


KIND_NONE, KIND_SGD, KIND_EASGD = 0, 1, 2


def twobit_dequant_sum_update(codes_list, n: int, threshold: float, kind: int,
                              lr: float = 0.0, alpha: float = 0.0,
                              center: np.ndarray | None = None,
                              weights: np.ndarray | None = None) -> np.ndarray | None:
    """Dequantise + sum W workers' codes.  kind NONE returns the fp64 average;
    SGD/EASGD update ``weights`` (fp64) in place and return None."""
    W = len(codes_list)
    for c in codes_list:
        _check(c, np.uint32, "codes", (n + 15) // 16)
    out = None
    if kind == KIND_NONE:
        out = np.zeros(n, dtype=np.float64)
    else:
        _check(weights, np.float64, "weights", n)
    if kind == KIND_EASGD:
        _check(center, np.float64, "center", n)
    arr = _ptr_array(codes_list)
    _load().orc_2bit_dequant_sum_update(
        arr, W, n, ctypes.c_float(np.float32(threshold)), kind,
        float(np.float32(lr)), float(np.float32(alpha)),
        _ptr(center) if center is not None else None,
        _ptr(weights) if weights is not None else None,
        _ptr(out) if out is not None else None)
    return out


def compensated_sum_update(grads, residuals, lr: float, weights: np.ndarray) -> None:
    """CD-SGD correction step: m_w = r_w + g_w (fp32), r_w <- 0, w -= lr * mean_w m_w (fp64)."""
    W = len(grads)
    n = grads[0].size
    kind = _grad_kind(grads[0])
    for g in grads:
        _check(g, grads[0].dtype, "grad", n)
    for r in residuals:
        _check(r, np.float32, "residual", n)
    _check(weights, np.float64, "weights", n)
    _load().orc_compensated_sum_update(_ptr_array(grads), kind, _ptr_array(residuals), W, n,
                                       float(np.float32(lr)), _ptr(weights))


def cdsgd_local_update(grad: np.ndarray, weights: np.ndarray, lr: float) -> np.ndarray:
    """CD-SGD eq. 11: local weights = weights - lr * grad (fp64)."""
    n = grad.size
    kind = _grad_kind(grad)
    _check(weights, np.float64, "weights", n)
    out = np.zeros(n, dtype=np.float64)
    _load().orc_cdsgd_local_update(_ptr(grad), kind, _ptr(weights), _ptr(out), n, float(np.float32(lr)))
    return out


# --------------------------------------------------------------------------
# QSGD
# --------------------------------------------------------------------------

def l2norm_fp32(v: np.ndarray) -> np.float32:
    _check(v, np.float32, "v")
    return np.float32(_load().orc_l2norm_fp32(_ptr(v), v.size))


def qsgd_code_bytes(n: int, s: int) -> int:
    return (n + 1) // 2 if s <= 7 else n


def qsgd_quantize(v: np.ndarray, bucket: int, s: int, seed: int, worker: int, i0: int = 0):
    """Returns (norms fp32 [ceil(n/bucket)], codes uint8).  ``v`` may be a
    bucket-aligned slice starting at global element index ``i0``."""
    _check(v, np.float32, "v")
    n = v.size
    norms = np.zeros((n + bucket - 1) // bucket, dtype=np.float32)
    codes = np.zeros(qsgd_code_bytes(n, s), dtype=np.uint8)
    _load().orc_qsgd_quantize(_ptr(v), n, bucket, s, seed & 0xFFFFFFFFFFFFFFFF, worker, i0,
                              _ptr(norms), _ptr(codes))
    return norms, codes


def qsgd_quantize_maxnorm(v: np.ndarray, bucket: int, s: int, seed: int, worker: int, i0: int = 0):
    """QSGD with each bucket scaled by max |v| (Knowl 8).  Returns (scales, codes)."""
    _check(v, np.float32, "v")
    n = v.size
    norms = np.zeros((n + bucket - 1) // bucket, dtype=np.float32)
    codes = np.zeros(qsgd_code_bytes(n, s), dtype=np.uint8)
    _load().orc_qsgd_quantize_maxnorm(_ptr(v), n, bucket, s, seed & 0xFFFFFFFFFFFFFFFF, worker, i0,
                                      _ptr(norms), _ptr(codes))
    return norms, codes


def qsgd_scaled_values(v: np.ndarray, bucket: int, s: int, seed: int, worker: int,
                       i0: int = 0, maxnorm: bool = False) -> np.ndarray:
    """fp32 x = |v| * (s / scale) + u whose floor decides each level (0 where
    the bucket's scale is 0); scale = the l2 norm, or max |v| with ``maxnorm``."""
    _check(v, np.float32, "v")
    x = np.zeros(v.size, dtype=np.float32)
    fn = _load().orc_qsgd_scaled_values_maxnorm if maxnorm else _load().orc_qsgd_scaled_values
    fn(_ptr(v), v.size, bucket, s, seed & 0xFFFFFFFFFFFFFFFF, worker, i0, _ptr(x))
    return x


def qsgd_dequant_sum(codes_list, norms_list, n: int, bucket: int, s: int,
                     scale: float = 1.0) -> np.ndarray:
    W = len(codes_list)
    for c in codes_list:
        _check(c, np.uint8, "codes", qsgd_code_bytes(n, s))
    for nm in norms_list:
        _check(nm, np.float32, "norms", (n + bucket - 1) // bucket)
    out = np.zeros(n, dtype=np.float64)
    _load().orc_qsgd_dequant_sum(_ptr_array(codes_list), _ptr_array(norms_list), W, n, bucket,
                                 s, float(np.float32(scale)), _ptr(out))
    return out


def elias_omega(N: int) -> str:
    """The Elias omega codeword of N >= 1 as a string of '0'/'1'."""
    buf = ctypes.create_string_buffer(64)
    length = _load().orc_elias_omega_bits(int(N), buf)
    return buf.value.decode()[:length]


def qsgd_elias_max_words(n: int, bucket: int) -> int:
    """Upper bound on the encoded words: 32 norm bits + at most 15 bits per
    coordinate (Elias-omega of 128 is 14 bits, plus the sign), per bucket."""
    nb = (n + bucket - 1) // bucket
    return nb * (1 + (15 * bucket + 31) // 32) + 1


def qsgd_elias_encode(codes: np.ndarray, norms: np.ndarray, n: int, bucket: int, s: int):
    """Returns (words uint32 [total], offsets uint32 [nbuckets + 1])."""
    _check(codes, np.uint8, "codes", qsgd_code_bytes(n, s))
    nb = (n + bucket - 1) // bucket
    _check(norms, np.float32, "norms", nb)
    words = np.zeros(qsgd_elias_max_words(n, bucket), dtype=np.uint32)
    offsets = np.zeros(nb + 1, dtype=np.uint32)
    total = int(_load().orc_qsgd_elias_encode(_ptr(codes), _ptr(norms), n, bucket, s, _ptr(words),
                                              _ptr(offsets)))
    return words[:total].copy(), offsets


def qsgd_elias_decode(words: np.ndarray, offsets: np.ndarray, n: int, bucket: int, s: int):
    """Returns (codes uint8, norms fp32)."""
    _check(words, np.uint32, "words")
    _check(offsets, np.uint32, "offsets", (n + bucket - 1) // bucket + 1)
    codes = np.zeros(qsgd_code_bytes(n, s), dtype=np.uint8)
    norms = np.zeros((n + bucket - 1) // bucket, dtype=np.float32)
    _load().orc_qsgd_elias_decode(_ptr(words), _ptr(offsets), n, bucket, s, _ptr(codes), _ptr(norms))
    return codes, norms


# --------------------------------------------------------------------------
# SAPS + EASGD
# --------------------------------------------------------------------------

def saps_mask_compact(n: int, p: float, seed_t: int, models, capacity: int | None = None,
                      i0: int = 0):
    """Returns (count, idx uint32 [min(count, capacity)], vals list of fp64 arrays).
    ``models`` may be a slice of n elements starting at global index ``i0``."""
    W = len(models)
    for m in models:
        _check(m, np.float64, "model", n)
    if capacity is None:
        capacity = n
    idx = np.zeros(max(capacity, 1), dtype=np.uint32)
    vals = [np.zeros(max(capacity, 1), dtype=np.float64) for _ in range(W)]
    K = int(_load().orc_saps_mask_compact(n, float(p), seed_t & 0xFFFFFFFFFFFFFFFF,
                                          _ptr_array(models), W, i0, _ptr(idx), _ptr_array(vals),
                                          capacity))
    kept = min(K, capacity)
    return K, idx[:kept].copy(), [v[:kept].copy() for v in vals]


def saps_matching(seed_t: int, W: int) -> np.ndarray:
    pairs = np.zeros(max(W, 1), dtype=np.int32)
    rc = _load().orc_saps_matching(seed_t & 0xFFFFFFFFFFFFFFFF, W, _ptr(pairs))
    if rc != 0:
        raise ValueError("W must be a positive even number")
    return pairs[:W].copy()


def saps_peer_average(models, vals, idx: np.ndarray, pairs: np.ndarray) -> None:
    W = len(models)
    K = idx.size
    for m in models:
        _check(m, np.float64, "model")
    vals = [np.ascontiguousarray(v, dtype=np.float64) for v in vals]
    idx = np.ascontiguousarray(idx, dtype=np.uint32)
    pairs = np.ascontiguousarray(pairs, dtype=np.int32)
    _load().orc_saps_peer_average(_ptr_array(models), _ptr_array(vals), _ptr(idx), K,
                                  _ptr(pairs), W)


def easgd_step(models, alpha: float, beta: float, center: np.ndarray) -> None:
    W = len(models)
    n = center.size
    for m in models:
        _check(m, np.float64, "model", n)
    _check(center, np.float64, "center", n)
    _load().orc_easgd_step(_ptr_array(models), W, n, float(np.float32(alpha)),
                           float(np.float32(beta)), _ptr(center))


def easgd_step_from_sum(model: np.ndarray, model_sum: np.ndarray, W: int, alpha: float, beta: float,
                        center: np.ndarray) -> None:
    """One worker's EASGD step given the sum of all W workers' models (fp64, in place)."""
    n = center.size
    _check(model, np.float64, "model", n)
    _check(model_sum, np.float64, "model_sum", n)
    _check(center, np.float64, "center", n)
    _load().orc_easgd_step_from_sum(_ptr(model), _ptr(model_sum), int(W), n, float(np.float32(alpha)),
                                    float(np.float32(beta)), _ptr(center))


def qsgd_elias_sparse_max_words(n: int, bucket: int) -> int:
    """Upper bound on the sparse-regime stream: per bucket 32 norm bits plus
    at most 18 bits per coordinate (distances sum to the bucket length and
    |omega(g)| <= g + 2; sign 1 bit; omega(level) <= 14 bits) and 2 bits."""
    nb = (n + bucket - 1) // bucket
    return nb * (1 + (18 * bucket + 2 + 31) // 32) + 1


def qsgd_elias_encode_sparse(codes: np.ndarray, norms: np.ndarray, n: int, bucket: int, s: int):
    """Knowl 2 sparse regime (distances between non-zero coordinates).
    Returns (words uint32 [total], offsets uint32 [nbuckets + 1])."""
    _check(codes, np.uint8, "codes", qsgd_code_bytes(n, s))
    nb = (n + bucket - 1) // bucket
    _check(norms, np.float32, "norms", nb)
    words = np.zeros(qsgd_elias_sparse_max_words(n, bucket), dtype=np.uint32)
    offsets = np.zeros(nb + 1, dtype=np.uint32)
    total = int(_load().orc_qsgd_elias_encode_sparse(_ptr(codes), _ptr(norms), n, bucket, s, _ptr(words),
                                                     _ptr(offsets)))
    return words[:total].copy(), offsets


def qsgd_elias_decode_sparse(words: np.ndarray, offsets: np.ndarray, n: int, bucket: int, s: int):
    """Inverse of qsgd_elias_encode_sparse: (codes, norms, overshooting buckets)."""
    words = np.ascontiguousarray(words, dtype=np.uint32)
    offsets = np.ascontiguousarray(offsets, dtype=np.uint32)
    nb = (n + bucket - 1) // bucket
    codes = np.zeros(qsgd_code_bytes(n, s), dtype=np.uint8)
    norms = np.zeros(nb, dtype=np.float32)
    bad = int(_load().orc_qsgd_elias_decode_sparse(_ptr(words), _ptr(offsets), n, bucket, s, _ptr(codes),
                                                   _ptr(norms)))
    return codes, norms, bad


def qsgd_elias_quarter_marks(codes: np.ndarray, n: int, bucket: int, s: int) -> np.ndarray:
    """uint16 [3 * nbuckets]: bit offset (from the bucket's first word) where the
    codeword of each bucket's coordinate k*bucket/4 starts, k = 1..3."""
    _check(codes, np.uint8, "codes", qsgd_code_bytes(n, s))
    nb = (n + bucket - 1) // bucket
    marks = np.zeros(3 * nb, dtype=np.uint16)
    _load().orc_qsgd_elias_quarter_marks(_ptr(codes), n, bucket, s, _ptr(marks))
    return marks
