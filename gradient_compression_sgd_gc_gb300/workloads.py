"""Seeded synthetic inputs for the gradient-compression workloads.

This module holds shapes, seeds and random draws only -- none of the
method's arithmetic.  Both the product path (tests, benchmark) and the CPU
oracle take their inputs from here; the oracle gets host copies of exactly the
tensors the GPU path sees.

The flat sizes stand in for real models' gradients: 25,557,032 is the
parameter count of ResNet-50 and 61,100,840 that of AlexNet; no model, weight
file or dataset is used.
"""
from __future__ import annotations

import dataclasses

import torch


@dataclasses.dataclass(frozen=True)
class TwoBitConfig:
    """2-bit threshold compression, W workers, optional dequant-sum + update."""
    name: str
    n: int
    workers: int
    threshold: float
    steps: int
    grad_std: float
    lr: float = 0.0
    weight_range: float = 0.0
    grad_dtype: torch.dtype = torch.float32
    correction_every: int = 0          # CD-SGD k; 0 = never

    def grad_seed(self, step: int, worker: int) -> int:
        if self.name == "twobit_w1":
            return step
        if self.name.startswith("cdsgd"):
            return 3000 + 10 * step + worker
        return 1000 * step + worker


@dataclasses.dataclass(frozen=True)
class QsgdConfig:
    name: str
    n: int
    workers: int
    bucket: int
    s: int
    seed: int = 42
    grad_std: float = 1e-2
    heavy_frac: float = 0.01
    heavy_scale: float = 100.0

    def grad_seed(self, worker: int) -> int:
        return 2000 + worker


@dataclasses.dataclass(frozen=True)
class SapsConfig:
    name: str
    n: int
    workers: int
    p: float
    rounds: int
    alpha: float = 0.9
    beta: float = 0.9
    base_seed: int = 5
    model_std: float = 0.05

    def model_seed(self, worker: int) -> int:
        return 4000 + worker


TWOBIT_W1 = TwoBitConfig("twobit_w1", n=1 << 20, workers=1, threshold=0.5, steps=10,
                         grad_std=1.0)
TWOBIT_DQ_SGD = TwoBitConfig("twobit_dq_sgd", n=25_557_032, workers=8, threshold=2e-3,
                             steps=20, grad_std=1e-3, lr=0.1, weight_range=0.05)
QSGD_S7 = QsgdConfig("qsgd_s7", n=61_100_840, workers=4, bucket=512, s=7)
QSGD_S127 = QsgdConfig("qsgd_s127", n=61_100_840, workers=4, bucket=512, s=127)
CDSGD = TwoBitConfig("cdsgd", n=1_300_000_000, workers=4, threshold=1e-3, steps=8,
                     grad_std=5e-4, lr=0.01, weight_range=0.05, grad_dtype=torch.bfloat16,
                     correction_every=4)
SAPS_P01 = SapsConfig("saps_p01", n=25_557_032, workers=16, p=0.01, rounds=50)
SAPS_P001 = SapsConfig("saps_p001", n=25_557_032, workers=16, p=0.001, rounds=50)

ALL = {c.name: c for c in (TWOBIT_W1, TWOBIT_DQ_SGD, QSGD_S7, QSGD_S127, CDSGD,
                           SAPS_P01, SAPS_P001)}


def scaled(cfg, n: int, **kw):
    """The same workload recipe at another size (for parity runs the oracle
    finishes in seconds)."""
    return dataclasses.replace(cfg, n=n, **kw)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def normal(n: int, std: float, seed: int, device="cpu", dtype=torch.float32,
           out: torch.Tensor | None = None) -> torch.Tensor:
    """N(0, std^2) draws (fp32), cast to ``dtype``; written into ``out`` if given."""
    x = torch.randn(n, generator=_gen(seed, device), device=device, dtype=torch.float32)
    x.mul_(std)
    if out is not None:
        out.copy_(x)
        return out
    return x.to(dtype)


def uniform(n: int, half_range: float, seed: int, device="cpu") -> torch.Tensor:
    """U(-half_range, half_range) fp32 draws."""
    x = torch.rand(n, generator=_gen(seed, device), device=device, dtype=torch.float32)
    return x.mul_(2 * half_range).sub_(half_range)


def twobit_grad(cfg: TwoBitConfig, step: int, worker: int, device="cpu",
                out: torch.Tensor | None = None) -> torch.Tensor:
    return normal(cfg.n, cfg.grad_std, cfg.grad_seed(step, worker), device, cfg.grad_dtype,
                  out=out)


def twobit_weights(cfg: TwoBitConfig, device="cpu", seed: int = 7) -> torch.Tensor:
    return uniform(cfg.n, cfg.weight_range, seed, device)


def qsgd_grad(cfg: QsgdConfig, worker: int, device="cpu") -> torch.Tensor:
    """N(0, std^2) with a seeded ``heavy_frac`` of entries scaled by ``heavy_scale``."""
    seed = cfg.grad_seed(worker)
    x = normal(cfg.n, cfg.grad_std, seed, device)
    heavy = torch.rand(cfg.n, generator=_gen(seed + 0x5EED, device), device=device) < cfg.heavy_frac
    x[heavy] *= cfg.heavy_scale
    return x


def saps_models(cfg: SapsConfig, device="cpu") -> list[torch.Tensor]:
    return [normal(cfg.n, cfg.model_std, cfg.model_seed(w), device) for w in range(cfg.workers)]


def saps_initial_center(models: list[torch.Tensor]) -> torch.Tensor:
    """Initial EASGD center: the elementwise mean of the initial models,
    accumulated in fp64 and rounded once to fp32."""
    acc = torch.zeros_like(models[0], dtype=torch.float64)
    for m in models:
        acc += m.to(torch.float64)
    return (acc / len(models)).to(torch.float32)
