"""GB300-native gradient compression with error feedback.

Thin Python binding over ``libgc_gb300.so`` (C ABI in ``include/gc_gb300.h``).
Every function here only checks and marshals arguments -- torch tensors in,
device pointers and the current CUDA stream out -- and calls the entry point of
the same name.  All arithmetic runs in the library's sm_103a kernels; there is
no CPU or PyTorch fallback: if the library cannot be built or loaded, every
call raises.

Entry points (same names as the C ABI):
  gc_2bit_quantize, gc_2bit_quantize_batched, gc_2bit_quantize_steps, gc_2bit_dequant_sum_update,
  gc_2bit_step,
  gc_2bit_quantize_local, gc_2bit_step_local (through gc_2bit_step with local_weights),
  gc_compensated_sum_update,
  qsgd_quantize, qsgd_quantize_maxnorm, qsgd_dequant_sum, qsgd_step,
  qsgd_elias_encode, qsgd_elias_decode, qsgd_elias_decode_batched, qsgd_elias_max_words,
  qsgd_elias_encode_marked, qsgd_elias_decode_quarters,
  qsgd_elias_encode_sparse, qsgd_elias_decode_sparse, qsgd_elias_sparse_max_words,
  qsgd_elias_workspace_bytes,
  saps_round_seed, saps_matching, saps_matching_bandwidth, saps_workspace_bytes, saps_mask_compact,
  saps_mask_compact_noalloc, saps_peer_average, saps_pair_average_remote, easgd_step_from_sum, saps_average_easgd_step, easgd_step,
  saps_round, gc_status_string, gc_version, gc_l2_fetch_granularity
Front ends over them (per-key state, parameter rules): ``compression.py``.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import _build

__all__ = [
    "GcError", "load", "library_path",
    "GC_OK", "GC_ERR_INVALID", "GC_ERR_ALIGN", "GC_ERR_CUDA", "GC_ERR_CAPACITY", "GC_ERR_TIMEOUT",
    "GC_UPD_NONE", "GC_UPD_SGD", "GC_UPD_EASGD", "GC_MAX_WORKERS",
    "gc_status_string", "gc_version", "gc_2bit_quantize", "gc_2bit_quantize_batched",
    "gc_2bit_dequant_sum_update",
    "gc_compensated_sum_update", "qsgd_quantize", "qsgd_dequant_sum", "saps_round_seed", "saps_matching_bandwidth", "qsgd_elias_encode_sparse", "qsgd_elias_decode_sparse",
    "qsgd_elias_sparse_max_words", "saps_pair_average_remote", "easgd_step_from_sum", "gossip_matrix", "NEVER",
    "saps_matching", "saps_workspace_bytes", "saps_mask_compact", "saps_peer_average",
    "easgd_step", "code_words", "qsgd_code_bytes", "qsgd_num_buckets",
    "saps_mask_compact_noalloc", "GC_NOALLOC_MAX_N", "PreparedCall", "saps_average_easgd_step",
    "gc_2bit_step", "gc_2bit_quantize_local", "gc_2bit_quantize_steps", "qsgd_quantize_maxnorm",
    "GC_ERR_CORRUPT", "qsgd_elias_encode", "qsgd_elias_decode", "qsgd_elias_max_words",
    "qsgd_elias_workspace_bytes", "saps_round", "qsgd_step", "qsgd_elias_decode_batched",
    "qsgd_elias_encode_marked", "qsgd_elias_decode_quarters", "qsgd_elias_encode_status",
    "gc_l2_fetch_granularity",
]

GC_OK, GC_ERR_INVALID, GC_ERR_ALIGN, GC_ERR_CUDA, GC_ERR_CAPACITY, GC_ERR_TIMEOUT = 0, -1, -2, -3, -4, -5
GC_ERR_CORRUPT = -6
GC_F32, GC_BF16 = 0, 1
GC_UPD_NONE, GC_UPD_SGD, GC_UPD_EASGD = 0, 1, 2
GC_MAX_WORKERS = 64
GC_NOALLOC_MAX_N = 1 << 26

_lock = threading.Lock()
_lib = None


class GcError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {gc_status_string(status)} ({status})")
        self.status = status


def library_path() -> str:
    return _build.LIB


def load():
    """Load libgc_gb300.so, building it with nvcc first if it is missing or
    stale.  Raises if it cannot be built or loaded."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.build()
        lib = ctypes.CDLL(path)
        vp, i32, i64, u64, f32, f64, sz = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64,
                                           ctypes.c_uint64, ctypes.c_float, ctypes.c_double,
                                           ctypes.c_size_t)
        sig = {
            "gc_status_string": (ctypes.c_char_p, [i32]),
            "gc_version": (i32, []),
            "gc_l2_fetch_granularity": (i32, [sz, vp]),
            "gc_2bit_quantize": (i32, [vp, i32, vp, vp, i64, f32, vp]),
            "gc_2bit_quantize_batched": (i32, [vp, i32, vp, vp, vp, i32, f32, vp]),
            "gc_2bit_step": (i32, [vp, i32, vp, vp, i32, i64, f32, i32, f32, f32, vp, vp, vp, vp]),
            "qsgd_elias_encode_sparse": (i32, [vp, vp, i64, i32, i32, vp, u64, vp, vp, sz, vp]),
            "qsgd_elias_sparse_max_words": (u64, [i64, i32]),
            "qsgd_elias_decode_sparse": (i32, [vp, vp, i64, i32, i32, vp, vp, vp, vp]),
            "saps_pair_average_remote": (i32, [vp, vp, vp, vp, vp, i64, vp]),
            "easgd_step_from_sum": (i32, [vp, vp, i32, i64, f32, f32, vp, vp]),
            "saps_matching_bandwidth": (i32, [i32, vp, f64, vp, i64, i64, u64, vp]),
            "gc_2bit_quantize_steps": (i32, [vp, i32, vp, vp, vp, i32, i64, f32, vp]),
            "gc_2bit_step_local": (i32, [vp, i32, vp, vp, vp, f32, i32, i64, f32, i32, f32, f32, vp, vp, vp,
                                         vp]),
            "gc_2bit_quantize_local": (i32, [vp, i32, vp, vp, vp, vp, i32, i64, f32, f32, vp]),
            "gc_2bit_dequant_sum_update": (i32, [vp, i32, i64, f32, i32, f32, f32, vp, vp, vp, vp]),
            "gc_compensated_sum_update": (i32, [vp, i32, vp, i32, i64, f32, vp, vp]),
            "qsgd_quantize": (i32, [vp, i64, i32, i32, u64, i32, vp, vp, vp]),
            "qsgd_dequant_sum": (i32, [vp, vp, i32, i64, i32, i32, f32, vp, vp]),
            "qsgd_quantize_maxnorm": (i32, [vp, i64, i32, i32, u64, i32, vp, vp, vp]),
            "qsgd_step": (i32, [vp, i32, i64, i32, i32, u64, i32, vp, vp, f32, vp, vp]),
            "qsgd_elias_encode": (i32, [vp, vp, i64, i32, i32, vp, u64, vp, vp, sz, vp]),
            "qsgd_elias_max_words": (u64, [i64, i32, i32]),
            "qsgd_elias_workspace_bytes": (sz, [i64, i32]),
            "qsgd_elias_decode": (i32, [vp, vp, i64, i32, i32, vp, vp, vp, vp]),
            "qsgd_elias_decode_batched": (i32, [vp, vp, i32, i64, i32, i32, vp, vp, vp, vp]),
            "qsgd_elias_encode_marked": (i32, [vp, vp, i64, i32, i32, vp, u64, vp, vp, vp, sz, vp]),
            "qsgd_elias_decode_quarters": (i32, [vp, vp, vp, i64, i32, i32, vp, vp, vp, vp]),
            "saps_round_seed": (u64, [u64, u64]),
            "saps_matching": (i32, [u64, i32, vp]),
            "saps_workspace_bytes": (sz, [i64]),
            "saps_mask_compact": (i32, [i64, f64, u64, vp, i32, vp, vp, i64, vp, vp, sz, vp, vp]),
            "saps_peer_average": (i32, [vp, vp, vp, vp, vp, i32, i64, vp]),
            "easgd_step": (i32, [vp, i32, i64, f32, f32, vp, vp]),
            "saps_average_easgd_step": (i32, [vp, vp, vp, vp, i32, i64, i64, f32, f32, vp, vp, sz, vp]),
            "saps_round": (i32, [i64, f64, u64, vp, i32, vp, f32, f32, vp, vp, vp, i64, vp, vp, sz, vp, vp]),
            "gc_testing_saps_round_one_pass": (i32, [i64, f64, u64, vp, i32, vp, f32, f32, vp, vp, vp, i64, vp,
                                                     vp, sz, vp, vp]),
            "saps_mask_compact_noalloc": (i32, [i64, f64, u64, vp, i32, vp, vp, i64, vp, vp, vp]),
            "gc_testing_qsgd_elias_encode_withhold": (i32, [vp, vp, i64, i32, i32, vp, u64, vp, vp, sz, i64, u64,
                                                              vp]),
            "gc_testing_saps_mask_compact_withhold": (i32, [i64, f64, u64, vp, i32, vp, vp, i64, vp, vp, sz,
                                                            vp, i64, u64, vp]),
            "gc_testing_decode_buckets_per_cta": (i32, [i64, i32, i64, i32, vp]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


# ---------------------------------------------------------------- helpers

def _stream(stream, t: torch.Tensor | None = None):
    if stream is None:
        dev = t.device if t is not None else torch.device("cuda", torch.cuda.current_device())
        return ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _dev(t: torch.Tensor, name: str, dtype=None, numel: int | None = None,
         pinned_ok: bool = False) -> int:
    """Address of a contiguous tensor the GPU can read.  ``pinned_ok`` also
    accepts page-locked host tensors (read in place by the kernel over the
    host link; the address is the same on both sides with unified addressing)."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor")
    if not t.is_cuda and not (pinned_ok and t.is_pinned()):
        raise ValueError(f"{name}: must be a CUDA tensor" + (" or pinned host tensor" if pinned_ok else ""))
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if numel is not None and t.numel() < numel:
        raise ValueError(f"{name}: needs at least {numel} elements, has {t.numel()}")
    return t.data_ptr()


def _ptrs(ts, name, dtype=None, numel=None, pinned_ok=False):
    return (ctypes.c_void_p * len(ts))(*[_dev(t, f"{name}[{i}]", dtype, numel, pinned_ok)
                                         for i, t in enumerate(ts)])


def _pairs(pairs, W: int, where: str):
    """Host int array of the matching (pairs (p[2q], p[2q+1])); the library
    checks that it is a permutation of 0..W-1."""
    if len(pairs) != W:
        raise ValueError(f"{where}: pairs must list all {W} workers, got {len(pairs)} entries")
    return (ctypes.c_int * W)(*[int(q) for q in pairs])


def _check(status: int, where: str) -> None:
    if status != GC_OK:
        raise GcError(status, where)


class PreparedCall:
    """One validated entry-point call with its ctypes arguments already built
    (device pointers, pointer tables, stream).  Calling it launches again on
    the same buffers and stream; the buffers must stay alive meanwhile.  Used
    in hot loops, where re-checking the tensors on every launch would cost more
    host time than the kernel takes."""
    __slots__ = ("fn", "args", "where", "keep")

    def __init__(self, fn, args, where, keep=()):
        self.fn, self.args, self.where, self.keep = fn, args, where, keep

    def __call__(self) -> None:
        st = self.fn(*self.args)
        if st != GC_OK:
            raise GcError(st, self.where)


def _invoke(fn, args, where: str, prepare: bool, keep=()):
    if prepare:
        return PreparedCall(fn, args, where, keep)
    _check(fn(*args), where)
    return None


def _gdtype(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return GC_F32
    if t.dtype == torch.bfloat16:
        return GC_BF16
    raise TypeError(f"gradient dtype must be float32 or bfloat16, got {t.dtype}")


def code_words(n: int) -> int:
    """uint32 words of 2-bit codes for n elements."""
    return (n + 15) // 16


def qsgd_code_bytes(n: int, s_levels: int) -> int:
    return (n + 1) // 2 if s_levels <= 7 else n


def qsgd_num_buckets(n: int, bucket: int) -> int:
    return (n + bucket - 1) // bucket


# ---------------------------------------------------------------- entry points

def gc_status_string(status: int) -> str:
    return load().gc_status_string(int(status)).decode()


def gc_version() -> int:
    return int(load().gc_version())


def gc_2bit_quantize(grad: torch.Tensor, residual: torch.Tensor, codes: torch.Tensor,
                     threshold: float, stream=None, prepare: bool = False):
    n = grad.numel()
    lib = load()
    args = (_dev(grad, "grad", pinned_ok=True), _gdtype(grad), _dev(residual, "residual", torch.float32, n),
            _dev(codes, "codes", torch.int32, code_words(n)), n, float(threshold),
            _stream(stream, residual))
    return _invoke(lib.gc_2bit_quantize, args, "gc_2bit_quantize", prepare, (grad, residual, codes))


def gc_2bit_quantize_batched(grads, residuals, codes, threshold: float, stream=None,
                             prepare: bool = False):
    """gc_2bit_quantize on B buffers (lists of equal length) in one launch."""
    lib = load()
    B = len(grads)
    if not (len(residuals) == len(codes) == B) or B == 0:
        raise ValueError("grads, residuals and codes must be non-empty lists of equal length")
    dt = _gdtype(grads[0])
    ns = [g.numel() for g in grads]
    n_arr = (ctypes.c_int64 * B)(*ns)
    args = (_ptrs(grads, "grads", grads[0].dtype, pinned_ok=True),
            dt, (ctypes.c_void_p * B)(*[_dev(r, f"residuals[{i}]", torch.float32, ns[i]) for i, r in enumerate(residuals)]),
            (ctypes.c_void_p * B)(*[_dev(c, f"codes[{i}]", torch.int32, code_words(ns[i])) for i, c in enumerate(codes)]),
            n_arr, B, float(threshold), _stream(stream, residuals[0]))
    return _invoke(lib.gc_2bit_quantize_batched, args, "gc_2bit_quantize_batched", prepare,
                   (list(grads), list(residuals), list(codes), n_arr))


def gc_2bit_step(grads, residuals, codes, threshold: float, kind: int = GC_UPD_SGD, lr: float = 0.0,
                 alpha: float = 0.0, center=None, weights=None, out=None, stream=None,
                 prepare: bool = False, local_weights=None, local_lr: float = 0.0):
    """Quantise W equal-sized fp32 or bf16 gradients and apply the dequant-sum
    update in one pass (bit-identical to gc_2bit_quantize_batched +
    gc_2bit_dequant_sum_update).  With ``local_weights`` (W fp32 tensors) the
    CD-SGD eq. 11 local weights weights - local_lr * grads[w] are written too
    (gc_2bit_step_local)."""
    lib = load()
    W = len(grads)
    n = grads[0].numel()
    dt = _gdtype(grads[0])
    head = (_ptrs(grads, "grads", grads[0].dtype, n, pinned_ok=True), dt,
            _ptrs(residuals, "residuals", torch.float32, n), _ptrs(codes, "codes", torch.int32, code_words(n)))
    tail = (W, n, float(threshold), int(kind), float(lr), float(alpha),
            _dev(center, "center", torch.float32, n) if center is not None else None,
            _dev(weights, "weights", torch.float32, n) if weights is not None else None,
            _dev(out, "out", torch.float32, n) if out is not None else None,
            _stream(stream, residuals[0]))
    keep = (list(grads), list(residuals), list(codes), center, weights, out)
    if local_weights is None:
        return _invoke(lib.gc_2bit_step, head + tail, "gc_2bit_step", prepare, keep)
    if len(local_weights) != W:
        raise ValueError("gc_2bit_step: one local weight buffer per worker")
    args = head + (_ptrs(local_weights, "local_weights", torch.float32, n), float(local_lr)) + tail
    return _invoke(lib.gc_2bit_step_local, args, "gc_2bit_step_local", prepare, keep + (list(local_weights),))


def gc_2bit_quantize_steps(grads, residual: torch.Tensor, codes, threshold: float, out=None, stream=None,
                           prepare: bool = False):
    """S successive 2-bit steps of one worker in one launch: grads[s] quantised
    into codes[s] with the residual carried; with ``out`` (S fp32 tensors) the
    dequantised values of each step too."""
    lib = load()
    S = len(grads)
    n = residual.numel()
    if len(codes) != S or (out is not None and len(out) != S):
        raise ValueError("gc_2bit_quantize_steps: one code (and out) buffer per step")
    args = (_ptrs(grads, "grads", grads[0].dtype, n, pinned_ok=True), _gdtype(grads[0]),
            _dev(residual, "residual", torch.float32, n),
            _ptrs(codes, "codes", torch.int32, code_words(n)),
            _ptrs(out, "out", torch.float32, n) if out is not None else None,
            S, n, float(threshold), _stream(stream, residual))
    return _invoke(lib.gc_2bit_quantize_steps, args, "gc_2bit_quantize_steps", prepare,
                   (list(grads), residual, list(codes), list(out) if out is not None else None))


def gc_2bit_quantize_local(grads, residuals, codes, weights: torch.Tensor, local_weights,
                           threshold: float, local_lr: float, stream=None, prepare: bool = False):
    """gc_2bit_quantize on B workers plus CD-SGD eq. 11 local weights
    local_weights[b] = weights - local_lr * grads[b], one launch."""
    lib = load()
    B = len(grads)
    n = weights.numel()
    dt = _gdtype(grads[0])
    args = (_ptrs(grads, "grads", grads[0].dtype, n, pinned_ok=True), dt,
            _ptrs(residuals, "residuals", torch.float32, n), _ptrs(codes, "codes", torch.int32, code_words(n)),
            _dev(weights, "weights", torch.float32, n), _ptrs(local_weights, "local_weights", torch.float32, n),
            B, n, float(threshold), float(local_lr), _stream(stream, weights))
    return _invoke(lib.gc_2bit_quantize_local, args, "gc_2bit_quantize_local", prepare,
                   (list(grads), list(residuals), list(codes), weights, list(local_weights)))


def gc_2bit_dequant_sum_update(codes, n: int, threshold: float, kind: int = GC_UPD_NONE,
                               lr: float = 0.0, alpha: float = 0.0, center=None, weights=None,
                               out=None, stream=None, prepare: bool = False):
    """codes: list of W int32 tensors (the packed uint32 words)."""
    lib = load()
    W = len(codes)
    arr = _ptrs(codes, "codes", torch.int32, code_words(n))
    args = (arr, W, n, float(threshold), int(kind), float(lr), float(alpha),
            _dev(center, "center", torch.float32, n) if center is not None else None,
            _dev(weights, "weights", torch.float32, n) if weights is not None else None,
            _dev(out, "out", torch.float32, n) if out is not None else None,
            _stream(stream, codes[0] if W else None))
    return _invoke(lib.gc_2bit_dequant_sum_update, args, "gc_2bit_dequant_sum_update", prepare,
                   (list(codes), center, weights, out))


def gc_compensated_sum_update(grads, residuals, lr: float, weights: torch.Tensor, stream=None,
                              prepare: bool = False):
    lib = load()
    W = len(grads)
    n = weights.numel()
    dt = _gdtype(grads[0])
    args = (_ptrs(grads, "grads", grads[0].dtype, n), dt,
            _ptrs(residuals, "residuals", torch.float32, n), W, n,
            float(lr), _dev(weights, "weights", torch.float32, n), _stream(stream, weights))
    return _invoke(lib.gc_compensated_sum_update, args, "gc_compensated_sum_update", prepare,
                   (list(grads), list(residuals), weights))


def qsgd_quantize(grad: torch.Tensor, bucket: int, s_levels: int, seed: int, worker: int,
                  norms: torch.Tensor, codes: torch.Tensor, stream=None, prepare: bool = False):
    lib = load()
    n = grad.numel()
    args = (_dev(grad, "grad", torch.float32), n, int(bucket), int(s_levels),
            int(seed) & 0xFFFFFFFFFFFFFFFF, int(worker),
            _dev(norms, "norms", torch.float32, qsgd_num_buckets(n, bucket)),
            _dev(codes, "codes", torch.uint8, qsgd_code_bytes(n, s_levels)),
            _stream(stream, grad))
    return _invoke(lib.qsgd_quantize, args, "qsgd_quantize", prepare, (grad, norms, codes))


def qsgd_quantize_maxnorm(grad: torch.Tensor, bucket: int, s_levels: int, seed: int, worker: int,
                          scales: torch.Tensor, codes: torch.Tensor, stream=None, prepare: bool = False):
    """QSGD with each bucket scaled by its max |v| (Knowl 8)."""
    lib = load()
    n = grad.numel()
    args = (_dev(grad, "grad", torch.float32), n, int(bucket), int(s_levels),
            int(seed) & 0xFFFFFFFFFFFFFFFF, int(worker),
            _dev(scales, "scales", torch.float32, qsgd_num_buckets(n, bucket)),
            _dev(codes, "codes", torch.uint8, qsgd_code_bytes(n, s_levels)), _stream(stream, grad))
    return _invoke(lib.qsgd_quantize_maxnorm, args, "qsgd_quantize_maxnorm", prepare, (grad, scales, codes))


def qsgd_dequant_sum(codes, norms, n: int, bucket: int, s_levels: int, scale: float,
                     out: torch.Tensor, stream=None, prepare: bool = False):
    lib = load()
    W = len(codes)
    args = (_ptrs(codes, "codes", torch.uint8, qsgd_code_bytes(n, s_levels)),
            _ptrs(norms, "norms", torch.float32, qsgd_num_buckets(n, bucket)),
            W, n, int(bucket), int(s_levels), float(scale),
            _dev(out, "out", torch.float32, n), _stream(stream, out))
    return _invoke(lib.qsgd_dequant_sum, args, "qsgd_dequant_sum", prepare, (list(codes), list(norms), out))


def qsgd_elias_max_words(n: int, bucket: int, s_levels: int) -> int:
    """Words the Elias stream of n coordinates can take at most."""
    return int(load().qsgd_elias_max_words(int(n), int(bucket), int(s_levels)))


def qsgd_elias_workspace_bytes(n: int, bucket: int) -> int:
    return int(load().qsgd_elias_workspace_bytes(int(n), int(bucket)))


def qsgd_elias_encode(codes: torch.Tensor, norms: torch.Tensor, n: int, bucket: int, s_levels: int,
                      words: torch.Tensor, offsets: torch.Tensor, workspace: torch.Tensor,
                      stream=None, prepare: bool = False):
    """Elias-omega stream of QSGD codes (Knowl 2).  words/offsets are int32
    tensors holding uint32 bit patterns; offsets[nbuckets] is the length."""
    lib = load()
    nb = qsgd_num_buckets(n, bucket)
    args = (_dev(codes, "codes", torch.uint8, qsgd_code_bytes(n, s_levels)),
            _dev(norms, "norms", torch.float32, nb), int(n), int(bucket), int(s_levels),
            _dev(words, "words", torch.int32), words.numel(),
            _dev(offsets, "offsets", torch.int32, nb + 1),
            _dev(workspace, "workspace", torch.uint8), workspace.numel(), _stream(stream, codes))
    return _invoke(lib.qsgd_elias_encode, args, "qsgd_elias_encode", prepare,
                   (codes, norms, words, offsets, workspace))


def qsgd_elias_decode(words: torch.Tensor, offsets: torch.Tensor, n: int, bucket: int, s_levels: int,
                      codes: torch.Tensor, norms: torch.Tensor, status: torch.Tensor | None = None,
                      stream=None, prepare: bool = False):
    """Inverse of qsgd_elias_encode; ``status`` (device int32 [1]) receives
    GC_ERR_CORRUPT for a stream that does not decode."""
    lib = load()
    nb = qsgd_num_buckets(n, bucket)
    args = (_dev(words, "words", torch.int32), _dev(offsets, "offsets", torch.int32, nb + 1),
            int(n), int(bucket), int(s_levels),
            _dev(codes, "codes", torch.uint8, qsgd_code_bytes(n, s_levels)),
            _dev(norms, "norms", torch.float32, nb),
            None if status is None else _dev(status, "status", torch.int32, 1), _stream(stream, words))
    keep = (words, offsets, codes, norms) + (() if status is None else (status,))
    return _invoke(lib.qsgd_elias_decode, args, "qsgd_elias_decode", prepare, keep)


def gc_l2_fetch_granularity(nbytes: int) -> int:
    """Sets the current context's L2 fetch-granularity hint (0..128 bytes);
    returns the value it replaces."""
    prev = ctypes.c_size_t(0)
    rc = load().gc_l2_fetch_granularity(int(nbytes), ctypes.byref(prev))
    if rc != GC_OK:
        raise GcError(rc, "gc_l2_fetch_granularity")
    return int(prev.value)


def qsgd_elias_encode_status(workspace: torch.Tensor) -> int:
    """The device status the last qsgd_elias_encode(_marked) left in its
    workspace (its first 4 bytes): GC_OK or GC_ERR_TIMEOUT.  Synchronises."""
    return int(workspace[:4].view(torch.int32).item())


def qsgd_elias_encode_marked(codes: torch.Tensor, norms: torch.Tensor, n: int, bucket: int, s_levels: int,
                             words: torch.Tensor, offsets: torch.Tensor, marks: torch.Tensor,
                             workspace: torch.Tensor, stream=None, prepare: bool = False):
    """qsgd_elias_encode that also writes the quarter marks: an int16 tensor
    [3 * nbuckets] holding uint16 bit positions (the start of each bucket's
    quarters 1..3 within its stream)."""
    lib = load()
    nb = qsgd_num_buckets(n, bucket)
    args = (_dev(codes, "codes", torch.uint8, qsgd_code_bytes(n, s_levels)),
            _dev(norms, "norms", torch.float32, nb), int(n), int(bucket), int(s_levels),
            _dev(words, "words", torch.int32), words.numel(),
            _dev(offsets, "offsets", torch.int32, nb + 1), _dev(marks, "marks", torch.int16, 3 * nb),
            _dev(workspace, "workspace", torch.uint8), workspace.numel(), _stream(stream, codes))
    return _invoke(lib.qsgd_elias_encode_marked, args, "qsgd_elias_encode_marked", prepare,
                   (codes, norms, words, offsets, marks, workspace))


def qsgd_elias_decode_quarters(words: torch.Tensor, offsets: torch.Tensor, marks: torch.Tensor, n: int,
                               bucket: int, s_levels: int, codes: torch.Tensor, norms: torch.Tensor,
                               status: torch.Tensor | None = None, stream=None, prepare: bool = False):
    """qsgd_elias_decode of a marked stream, one thread per quarter bucket."""
    lib = load()
    nb = qsgd_num_buckets(n, bucket)
    args = (_dev(words, "words", torch.int32), _dev(offsets, "offsets", torch.int32, nb + 1),
            _dev(marks, "marks", torch.int16, 3 * nb), int(n), int(bucket), int(s_levels),
            _dev(codes, "codes", torch.uint8, qsgd_code_bytes(n, s_levels)),
            _dev(norms, "norms", torch.float32, nb),
            None if status is None else _dev(status, "status", torch.int32, 1), _stream(stream, words))
    keep = (words, offsets, marks, codes, norms) + (() if status is None else (status,))
    return _invoke(lib.qsgd_elias_decode_quarters, args, "qsgd_elias_decode_quarters", prepare, keep)


def qsgd_elias_sparse_max_words(n: int, bucket: int) -> int:
    return int(load().qsgd_elias_sparse_max_words(int(n), int(bucket)))


def qsgd_elias_encode_sparse(codes: torch.Tensor, norms: torch.Tensor, n: int, bucket: int, s_levels: int,
                             words: torch.Tensor, offsets: torch.Tensor, workspace: torch.Tensor,
                             stream=None, prepare: bool = False):
    """Sparse-regime Elias stream of QSGD codes (Knowl 2 items 1 and 1'):
    distances between non-zero coordinates, signs, and levels when s >= 2."""
    lib = load()
    nb = qsgd_num_buckets(n, bucket)
    args = (_dev(codes, "codes", torch.uint8, qsgd_code_bytes(n, s_levels)),
            _dev(norms, "norms", torch.float32, nb), int(n), int(bucket), int(s_levels),
            _dev(words, "words", torch.int32), words.numel(),
            _dev(offsets, "offsets", torch.int32, nb + 1),
            _dev(workspace, "workspace", torch.uint8), workspace.numel(), _stream(stream, codes))
    return _invoke(lib.qsgd_elias_encode_sparse, args, "qsgd_elias_encode_sparse", prepare,
                   (codes, norms, words, offsets, workspace))


def qsgd_elias_decode_sparse(words: torch.Tensor, offsets: torch.Tensor, n: int, bucket: int, s_levels: int,
                             codes: torch.Tensor, norms: torch.Tensor, status: torch.Tensor | None = None,
                             stream=None, prepare: bool = False):
    """Inverse of qsgd_elias_encode_sparse; ``status`` receives GC_ERR_CORRUPT."""
    lib = load()
    nb = qsgd_num_buckets(n, bucket)
    args = (_dev(words, "words", torch.int32), _dev(offsets, "offsets", torch.int32, nb + 1),
            int(n), int(bucket), int(s_levels),
            _dev(codes, "codes", torch.uint8, qsgd_code_bytes(n, s_levels)),
            _dev(norms, "norms", torch.float32, nb),
            None if status is None else _dev(status, "status", torch.int32, 1), _stream(stream, words))
    keep = (words, offsets, codes, norms) + (() if status is None else (status,))
    return _invoke(lib.qsgd_elias_decode_sparse, args, "qsgd_elias_decode_sparse", prepare, keep)


def qsgd_elias_decode_batched(words, offsets, n: int, bucket: int, s_levels: int, codes, norms,
                              status: torch.Tensor | None = None, stream=None, prepare: bool = False):
    """qsgd_elias_decode of W streams (lists of equal length) in one launch."""
    lib = load()
    W = len(words)
    if not (len(offsets) == len(codes) == len(norms) == W) or W == 0:
        raise ValueError("words, offsets, codes and norms must be non-empty lists of equal length")
    nb = qsgd_num_buckets(n, bucket)
    args = (_ptrs(words, "words", torch.int32), _ptrs(offsets, "offsets", torch.int32, nb + 1), W,
            int(n), int(bucket), int(s_levels),
            _ptrs(codes, "codes", torch.uint8, qsgd_code_bytes(n, s_levels)),
            _ptrs(norms, "norms", torch.float32, nb),
            None if status is None else _dev(status, "status", torch.int32, 1), _stream(stream, words[0]))
    keep = (list(words), list(offsets), list(codes), list(norms)) + (() if status is None else (status,))
    return _invoke(lib.qsgd_elias_decode_batched, args, "qsgd_elias_decode_batched", prepare, keep)

def qsgd_step(grads, bucket: int, s_levels: int, seed: int, norms, codes, scale: float,
              out: torch.Tensor, maxnorm: bool = False, stream=None, prepare: bool = False):
    """Every worker's qsgd_quantize (worker index = position) and the
    dequant-sum, in one pass; bit-identical to the separate calls."""
    lib = load()
    W = len(grads)
    n = out.numel()
    args = (_ptrs(grads, "grads", torch.float32, n), W, n, int(bucket), int(s_levels),
            int(seed) & 0xFFFFFFFFFFFFFFFF, 1 if maxnorm else 0,
            _ptrs(norms, "norms", torch.float32, qsgd_num_buckets(n, bucket)),
            _ptrs(codes, "codes", torch.uint8, qsgd_code_bytes(n, s_levels)), float(scale),
            _dev(out, "out", torch.float32, n), _stream(stream, out))
    return _invoke(lib.qsgd_step, args, "qsgd_step", prepare, (list(grads), list(norms), list(codes), out))


def saps_round_seed(base_seed: int, t: int) -> int:
    return int(load().saps_round_seed(int(base_seed) & 0xFFFFFFFFFFFFFFFF, int(t) & 0xFFFFFFFFFFFFFFFF))


def saps_matching(seed_t: int, W: int) -> list[int]:
    buf = (ctypes.c_int * max(W, 1))()
    _check(load().saps_matching(int(seed_t) & 0xFFFFFFFFFFFFFFFF, int(W), buf), "saps_matching")
    return list(buf)[:W]


NEVER = -(1 << 63)


def saps_matching_bandwidth(bandwidth, b_thres: float, last_round, t: int, t_thres: int,
                            seed_t: int) -> list[int]:
    """SAPS Algorithm 3 (host): the round's perfect matching from the W x W
    bandwidth matrix.  ``last_round`` is a W x W int64 numpy array updated in
    place (the rounds pairs were last matched; NEVER for never)."""
    import numpy as np
    B = np.ascontiguousarray(bandwidth, dtype=np.float64)
    W = B.shape[0]
    if B.shape != (W, W) or not isinstance(last_round, np.ndarray) or last_round.shape != (W, W) \
            or last_round.dtype != np.int64 or not last_round.flags.c_contiguous:
        raise ValueError("saps_matching_bandwidth: bandwidth and last_round must be W x W "
                         "(last_round a C-contiguous int64 array)")
    buf = (ctypes.c_int * max(W, 1))()
    _check(load().saps_matching_bandwidth(int(W), B.ctypes.data, float(b_thres), last_round.ctypes.data,
                                          int(t), int(t_thres), int(seed_t) & 0xFFFFFFFFFFFFFFFF, buf),
           "saps_matching_bandwidth")
    return list(buf)[:W]


def gossip_matrix(pairs):
    """The doubly stochastic W x W gossip matrix of a perfect matching given as
    pairs (pairs[2q], pairs[2q+1]): 1/2 on i,i / i,j / j,i / j,j per pair."""
    import numpy as np
    W = len(pairs)
    M = np.zeros((W, W))
    for q in range(0, W, 2):
        a, b = pairs[q], pairs[q + 1]
        M[a, a] = M[b, b] = M[a, b] = M[b, a] = 0.5
    return M


def saps_pair_average_remote(model: torch.Tensor, idx: torch.Tensor, d_count: torch.Tensor,
                             mine: torch.Tensor, peer: torch.Tensor, stream=None, prepare: bool = False):
    """Pair average for a worker whose peer is another process: model[idx[k]] =
    (mine[k] + peer[k]) / 2 for k < min(count, capacity)."""
    lib = load()
    cap = idx.numel()
    args = (_dev(model, "model", torch.float32), _dev(idx, "idx", torch.int32, cap),
            _dev(d_count, "d_count", torch.int64, 1), _dev(mine, "mine", torch.float32, cap),
            _dev(peer, "peer", torch.float32, cap), cap, _stream(stream, model))
    return _invoke(lib.saps_pair_average_remote, args, "saps_pair_average_remote", prepare,
                   (model, idx, d_count, mine, peer))


def easgd_step_from_sum(model: torch.Tensor, model_sum: torch.Tensor, W: int, alpha: float, beta: float,
                        center: torch.Tensor, stream=None, prepare: bool = False):
    """Elastic step of one worker from the sum of all W workers' models."""
    lib = load()
    n = model.numel()
    args = (_dev(model, "model", torch.float32, n), _dev(model_sum, "model_sum", torch.float32, n), int(W), n,
            float(alpha), float(beta), _dev(center, "center", torch.float32, n), _stream(stream, model))
    return _invoke(lib.easgd_step_from_sum, args, "easgd_step_from_sum", prepare, (model, model_sum, center))


def saps_workspace_bytes(n: int) -> int:
    return int(load().saps_workspace_bytes(int(n)))


def saps_mask_compact(n: int, p: float, seed_t: int, models, idx: torch.Tensor, vals,
                      d_count: torch.Tensor, workspace: torch.Tensor, d_status: torch.Tensor,
                      stream=None, prepare: bool = False):
    """models: W fp32 tensors [n]; idx: int32 (uint32 bits) [capacity]; vals: W fp32
    [capacity]; d_count: int64 [1]; workspace: uint8 [saps_workspace_bytes(n)];
    d_status: int32 [1] (zeroed by the caller)."""
    lib = load()
    W = len(models)
    capacity = idx.numel()
    args = (int(n), float(p), int(seed_t) & 0xFFFFFFFFFFFFFFFF,
            _ptrs(models, "models", torch.float32, n), W,
            _dev(idx, "idx", torch.int32), _ptrs(vals, "vals", torch.float32, capacity),
            capacity, _dev(d_count, "d_count", torch.int64, 1),
            _dev(workspace, "workspace", torch.uint8), workspace.numel(),
            _dev(d_status, "d_status", torch.int32, 1), _stream(stream, idx))
    return _invoke(lib.saps_mask_compact, args, "saps_mask_compact", prepare,
                   (list(models), idx, list(vals), d_count, workspace, d_status))


def saps_peer_average(models, vals, idx: torch.Tensor, d_count: torch.Tensor, pairs,
                      stream=None, prepare: bool = False):
    lib = load()
    W = len(models)
    pairs_arr = _pairs(pairs, W, "saps_peer_average")
    capacity = idx.numel()
    args = (_ptrs(models, "models", torch.float32), _ptrs(vals, "vals", torch.float32, capacity),
            _dev(idx, "idx", torch.int32), _dev(d_count, "d_count", torch.int64, 1),
            pairs_arr, W, capacity, _stream(stream, idx))
    return _invoke(lib.saps_peer_average, args, "saps_peer_average", prepare,
                   (list(models), list(vals), idx, d_count))


def saps_average_easgd_step(models, vals, d_count: torch.Tensor, pairs, alpha: float, beta: float,
                            center: torch.Tensor, workspace: torch.Tensor, stream=None,
                            prepare: bool = False):
    """saps_peer_average + easgd_step in one pass; ``workspace`` must be the one
    the preceding saps_mask_compact used."""
    lib = load()
    W = len(models)
    n = center.numel()
    capacity = vals[0].numel() if vals else 0
    pairs_arr = _pairs(pairs, W, "saps_average_easgd_step")
    args = (_ptrs(models, "models", torch.float32, n), _ptrs(vals, "vals", torch.float32, capacity),
            _dev(d_count, "d_count", torch.int64, 1), pairs_arr, W, n, capacity, float(alpha),
            float(beta), _dev(center, "center", torch.float32, n),
            _dev(workspace, "workspace", torch.uint8), workspace.numel(), _stream(stream, center))
    return _invoke(lib.saps_average_easgd_step, args, "saps_average_easgd_step", prepare,
                   (list(models), list(vals), d_count, center, workspace, pairs_arr))


def saps_round(n: int, p: float, seed_t: int, models, pairs, alpha: float, beta: float,
               center: torch.Tensor, idx: torch.Tensor, vals, d_count: torch.Tensor,
               workspace: torch.Tensor, d_status: torch.Tensor, stream=None, prepare: bool = False,
               _one_pass: bool = False):
    """One SAPS round in one pass: saps_mask_compact + saps_peer_average +
    easgd_step, bit for bit while the count fits idx.numel().  ``_one_pass``
    (tests only) forces the one-pass kernel whatever p is."""
    lib = load()
    fn = lib.gc_testing_saps_round_one_pass if _one_pass else lib.saps_round
    W = len(models)
    capacity = idx.numel()
    pairs_arr = _pairs(pairs, W, "saps_round")
    args = (int(n), float(p), int(seed_t) & 0xFFFFFFFFFFFFFFFF,
            _ptrs(models, "models", torch.float32, n), W, pairs_arr, float(alpha), float(beta),
            _dev(center, "center", torch.float32, n), _dev(idx, "idx", torch.int32),
            _ptrs(vals, "vals", torch.float32, capacity), capacity,
            _dev(d_count, "d_count", torch.int64, 1), _dev(workspace, "workspace", torch.uint8),
            workspace.numel(), _dev(d_status, "d_status", torch.int32, 1), _stream(stream, center))
    return _invoke(fn, args, "saps_round", prepare,
                   (list(models), center, idx, list(vals), d_count, workspace, d_status, pairs_arr))


def easgd_step(models, alpha: float, beta: float, center: torch.Tensor, stream=None,
               prepare: bool = False):
    lib = load()
    W = len(models)
    n = center.numel()
    args = (_ptrs(models, "models", torch.float32, n), W, n, float(alpha), float(beta),
            _dev(center, "center", torch.float32, n), _stream(stream, center))
    return _invoke(lib.easgd_step, args, "easgd_step", prepare, (list(models), center))


def saps_mask_compact_noalloc(n: int, p: float, seed_t: int, models, idx: torch.Tensor, vals,
                              d_count: torch.Tensor, d_status: torch.Tensor, stream=None) -> None:
    """saps_mask_compact without a workspace, for callers that cannot allocate
    one: the look-back scratch is a fixed array inside the library, so n is
    limited to GC_NOALLOC_MAX_N elements, and calls that overlap on the GPU
    race (order them on one stream).  Arguments as saps_mask_compact."""
    if n > GC_NOALLOC_MAX_N:
        raise ValueError(f"saps_mask_compact_noalloc: n = {n} exceeds the fixed scratch limit of "
                         f"{GC_NOALLOC_MAX_N} elements; use saps_mask_compact with a workspace")
    lib = load()
    W = len(models)
    capacity = idx.numel()
    st = lib.saps_mask_compact_noalloc(int(n), float(p), int(seed_t) & 0xFFFFFFFFFFFFFFFF,
                                       _ptrs(models, "models", torch.float32, n), W,
                                       _dev(idx, "idx", torch.int32),
                                       _ptrs(vals, "vals", torch.float32, capacity), capacity,
                                       _dev(d_count, "d_count", torch.int64, 1),
                                       _dev(d_status, "d_status", torch.int32, 1), _stream(stream, idx))
    _check(st, "saps_mask_compact_noalloc")
