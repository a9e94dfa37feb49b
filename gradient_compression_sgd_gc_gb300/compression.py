"""Key-value style gradient compression on top of the C ABI.

"2bit gradient compression" (MXNet PR #8662), sections "Usage" and "Backend
API": the user sets the compression once as a dict of parameters,
``{'type': '2bit', 'threshold': t}``; the threshold has no default; every
gradient (one per key) carries its own residual; the receiver dequantises
every worker's codes and averages them.  Switching compression off after it
was on is an error; changing the threshold is allowed, and codes produced
with the old threshold are then decoded with the new one (the page warns of
that transient).

This module keeps the per-key residuals and code buffers as device tensors
and calls the library for all arithmetic; it holds no fallback.
"""
from __future__ import annotations

import math

import torch

from . import (GC_MAX_WORKERS, GC_UPD_EASGD, GC_UPD_NONE, GC_UPD_SGD, code_words,
               gc_2bit_dequant_sum_update, gc_2bit_quantize, gc_2bit_quantize_batched,
               gc_2bit_quantize_local, gc_2bit_step, gc_compensated_sum_update)

__all__ = ["GradientCompression", "CDSGD", "QSGD", "SAPSGossip"]

_TYPES = ("none", "2bit")


def _check_params(params) -> dict:
    if not isinstance(params, dict):
        raise TypeError("compression params must be a dict such as {'type': '2bit', 'threshold': 0.5}")
    unknown = set(params) - {"type", "threshold"}
    if unknown:
        raise ValueError(f"unknown compression parameters: {sorted(unknown)}")
    kind = params.get("type")
    if kind not in _TYPES:
        raise ValueError(f"compression type must be one of {_TYPES}, got {kind!r}")
    if kind == "2bit":
        if "threshold" not in params:
            raise ValueError("2bit compression needs a threshold (there is no default)")
        t = float(params["threshold"])
        if not (math.isfinite(t) and t > 0.0):
            raise ValueError(f"threshold must be finite and positive, got {params['threshold']!r}")
        return {"type": "2bit", "threshold": t}
    if "threshold" in params:
        raise ValueError("'none' compression takes no threshold")
    return {"type": "none"}


class GradientCompression:
    """Per-key 2-bit compression state: residuals and codes on the device."""

    def __init__(self, params):
        self._params = _check_params(params)
        self._residual: dict = {}
        self._codes: dict = {}
        self._used = False

    @property
    def params(self) -> dict:
        return dict(self._params)

    @property
    def threshold(self) -> float | None:
        return self._params.get("threshold")

    def set_params(self, params) -> None:
        """Re-configure.  Turning compression off once it has compressed a
        gradient raises; a new threshold applies from the next call."""
        new = _check_params(params)
        if self._used and self._params["type"] == "2bit" and new["type"] == "none":
            raise ValueError("compression cannot be switched off after it has been used")
        self._params = new

    def _state(self, key, grad: torch.Tensor):
        n = grad.numel()
        r = self._residual.get(key)
        if r is None or r.numel() != n or r.device != grad.device:
            r = torch.zeros(n, dtype=torch.float32, device=grad.device)
            self._residual[key] = r
            self._codes[key] = torch.empty(code_words(n), dtype=torch.int32, device=grad.device)
        return r, self._codes[key]

    def residual(self, key) -> torch.Tensor | None:
        return self._residual.get(key)

    def compress(self, key, grad: torch.Tensor) -> torch.Tensor:
        """The packed codes of ``grad`` (fp32 or bf16), the key's residual
        carried over; for 'none' the gradient itself, untouched."""
        if self._params["type"] == "none":
            return grad
        r, c = self._state(key, grad)
        gc_2bit_quantize(grad.reshape(-1), r, c, self._params["threshold"])
        self._used = True
        return c

    def decompress(self, codes, n: int, out: torch.Tensor | None = None) -> torch.Tensor:
        """The average of the workers' dequantised codes (one code buffer per
        worker), as the receiver forms it.  With 'none' there is nothing to
        decode: the caller reduces the uncompressed gradients itself."""
        if self._params["type"] == "none":
            raise ValueError("no compression configured: reduce the uncompressed gradients directly")
        out = out if out is not None else torch.empty(n, dtype=torch.float32, device=codes[0].device)
        gc_2bit_dequant_sum_update(list(codes), n, self._params["threshold"], GC_UPD_NONE, out=out)
        return out

    def apply(self, codes, weights: torch.Tensor, lr: float, alpha: float = 0.0,
              center: torch.Tensor | None = None) -> None:
        """weights -= lr * (average of the dequantised codes), and the EASGD
        elastic term when ``center`` is given (2bit only)."""
        if self._params["type"] != "2bit":
            raise ValueError("apply() needs 2bit compression")
        kind = GC_UPD_EASGD if center is not None else GC_UPD_SGD
        gc_2bit_dequant_sum_update(list(codes), weights.numel(), self._params["threshold"], kind, lr=lr,
                                   alpha=alpha, center=center, weights=weights)

    def step(self, keys, grads, weights: torch.Tensor, lr: float) -> None:
        """Every worker's compression (one key per worker) and the averaged
        SGD update in one pass over the data (fp32 gradients of one size)."""
        if self._params["type"] != "2bit":
            raise ValueError("step() needs 2bit compression")
        res, codes = zip(*[self._state(k, g) for k, g in zip(keys, grads)])
        gc_2bit_step([g.reshape(-1) for g in grads], list(res), list(codes), self._params["threshold"],
                     GC_UPD_SGD, lr=lr, weights=weights)
        self._used = True


class CDSGD:
    """CD-SGD's step schedule for W workers held on this GPU ("CD-SGD:
    Distributed Stochastic Gradient Descent with Compression and Delay
    Compensation", Algorithm 1, eq. 10 and eq. 11).  Steps are counted from 1;
    every k-th step is a correction step: each worker sends its
    residual-compensated full-precision gradient r + g (its residual is then
    zeroed) and the weights take their average; every other step each worker
    2-bit quantises its gradient with its residual and the weights take the
    dequantised average.  With ``local_lr`` set, a compressed step also writes
    each worker's local weights W - local_lr * g (eq. 11) from the weights
    before the update.  Gradients are fp32 or bf16, one size for all."""

    def __init__(self, n: int, workers: int, threshold: float, lr: float, k: int = 4,
                 local_lr: float | None = None, device="cuda"):
        if not (1 <= workers <= GC_MAX_WORKERS):
            raise ValueError(f"need 1 <= workers <= {GC_MAX_WORKERS}")
        if int(k) != k or k < 1:
            raise ValueError("the correction period k must be a positive integer")
        if not (math.isfinite(threshold) and threshold > 0.0):
            raise ValueError("threshold must be finite and positive")
        if not math.isfinite(lr) or (local_lr is not None and not math.isfinite(local_lr)):
            raise ValueError("learning rates must be finite")
        self.n, self.W, self.k = int(n), int(workers), int(k)
        self.threshold, self.lr, self.local_lr = float(threshold), float(lr), local_lr
        self.residuals = [torch.zeros(self.n, dtype=torch.float32, device=device) for _ in range(self.W)]
        self.codes = [torch.empty(code_words(self.n), dtype=torch.int32, device=device) for _ in range(self.W)]
        self.t = 0

    def is_correction(self, t: int) -> bool:
        """Whether step t (1-based) sends full precision."""
        return t % self.k == 0

    def step(self, grads, weights: torch.Tensor, local_weights=None) -> bool:
        """One step; returns True for a correction step."""
        if len(grads) != self.W:
            raise ValueError(f"expected {self.W} gradients")
        if self.local_lr is not None and local_weights is None and not self.is_correction(self.t + 1):
            raise ValueError("local_lr is set: pass one local-weights buffer per worker")
        self.t += 1
        if self.is_correction(self.t):
            gc_compensated_sum_update(list(grads), self.residuals, self.lr, weights)
            return True
        if self.local_lr is not None:
            gc_2bit_quantize_local(list(grads), self.residuals, self.codes, weights, list(local_weights),
                                   self.threshold, self.local_lr)
        else:
            gc_2bit_quantize_batched(list(grads), self.residuals, self.codes, self.threshold)
        gc_2bit_dequant_sum_update(self.codes, self.n, self.threshold, GC_UPD_SGD, lr=self.lr, weights=weights)
        return False


class QSGD:
    """QSGD for W workers held on this GPU ("QSGD: Communication-Efficient SGD
    via Gradient Quantization and Encoding", Knowl 1-3 and 8): bucketed
    stochastic quantisation with s levels (4-bit codes for s <= 7, else
    8-bit), optional max-norm scaling, the average of the decoded messages,
    and the Elias-omega stream of a worker's message (Knowl 2)."""

    def __init__(self, n: int, workers: int, bucket: int = 512, s: int = 7, seed: int = 0,
                 maxnorm: bool = False, device="cuda"):
        from . import qsgd_code_bytes, qsgd_num_buckets
        if not (1 <= s <= 127) or bucket not in (128, 256, 512, 1024, 2048) or workers < 1:
            raise ValueError("need 1 <= s <= 127, bucket in {128, ..., 2048} and at least one worker")
        self.n, self.W, self.bucket, self.s, self.seed, self.maxnorm = n, workers, bucket, s, seed, maxnorm
        nb, cb = qsgd_num_buckets(n, bucket), qsgd_code_bytes(n, s)
        self.norms = [torch.empty(nb, dtype=torch.float32, device=device) for _ in range(workers)]
        self.codes = [torch.empty(cb, dtype=torch.uint8, device=device) for _ in range(workers)]

    def step(self, grads, out: torch.Tensor) -> torch.Tensor:
        """Every worker's message (worker w quantises grads[w] with its own
        draws) and their average into ``out``, in one pass."""
        from . import qsgd_step
        if len(grads) != self.W:
            raise ValueError(f"expected {self.W} gradients")
        qsgd_step(list(grads), self.bucket, self.s, self.seed, self.norms, self.codes, 1.0 / self.W, out,
                  maxnorm=self.maxnorm)
        return out

    def encode(self, worker: int):
        """The Elias-omega stream of a worker's last message: (words, offsets),
        offsets[-1] being its length in 32-bit words."""
        from . import qsgd_elias_encode, qsgd_elias_max_words, qsgd_elias_workspace_bytes, qsgd_num_buckets
        dev = self.codes[worker].device
        words = torch.empty(qsgd_elias_max_words(self.n, self.bucket, self.s), dtype=torch.int32, device=dev)
        offsets = torch.empty(qsgd_num_buckets(self.n, self.bucket) + 1, dtype=torch.int32, device=dev)
        ws = torch.empty(max(16, qsgd_elias_workspace_bytes(self.n, self.bucket)), dtype=torch.uint8, device=dev)
        qsgd_elias_encode(self.codes[worker], self.norms[worker], self.n, self.bucket, self.s, words, offsets, ws)
        return words, offsets

    def decode(self, words: torch.Tensor, offsets: torch.Tensor, worker: int) -> None:
        """Replace a worker's message by the decoded stream."""
        from . import qsgd_elias_decode
        qsgd_elias_decode(words, offsets, self.n, self.bucket, self.s, self.codes[worker], self.norms[worker])

    def decode_all(self, streams) -> None:
        """Replace every worker's message by its decoded stream, streams[w] =
        (words, offsets), in one launch."""
        from . import qsgd_elias_decode_batched
        if len(streams) != self.W:
            raise ValueError(f"expected {self.W} streams")
        qsgd_elias_decode_batched([w for w, _ in streams], [o for _, o in streams], self.n, self.bucket, self.s,
                                  self.codes, self.norms)


class SAPSGossip:
    """SAPS rounds for W workers held on this GPU ("Communication-Efficient
    Decentralized Learning with Sparsification and Adaptive Peer Selection",
    section II, with the EASGD elastic step): round t draws its shared seed
    from the base seed, the seeded perfect matching, the Bernoulli(p) mask,
    the compacted (index, value) messages, the pair averages and the elastic
    step -- one pass over the models."""

    def __init__(self, models, center: torch.Tensor, p: float, alpha: float, beta: float,
                 base_seed: int = 0, capacity: int | None = None):
        from . import saps_workspace_bytes
        self.models, self.center = list(models), center
        self.W, self.n = len(self.models), center.numel()
        if self.W < 2 or self.W % 2:
            raise ValueError("SAPS pairs the workers: W must be even")
        self.p, self.alpha, self.beta, self.base_seed = p, alpha, beta, base_seed
        dev = center.device
        cap = capacity if capacity is not None else self.n
        self.idx = torch.empty(cap, dtype=torch.int32, device=dev)
        self.vals = [torch.empty(cap, dtype=torch.float32, device=dev) for _ in range(self.W)]
        self.count = torch.zeros(1, dtype=torch.int64, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.workspace = torch.empty(saps_workspace_bytes(self.n), dtype=torch.uint8, device=dev)

    def round(self, t: int):
        """Run round t; returns its matching (host list)."""
        from . import saps_matching, saps_round, saps_round_seed
        seed_t = saps_round_seed(self.base_seed, t)
        pairs = saps_matching(seed_t, self.W)
        saps_round(self.n, self.p, seed_t, self.models, pairs, self.alpha, self.beta, self.center, self.idx,
                   self.vals, self.count, self.workspace, self.status)
        return pairs
