"""Data-parallel exchange between processes, one worker (and one GPU) per rank.

On one GPU the library simulates the W workers as W buffers and the
"collective" is a kernel that reads all of them.  Across processes each rank
holds one worker's buffers and the methods' own exchange steps run over
``torch.distributed`` (NCCL between GPUs): plain collectives into local
buffers, then the same kernels as on one GPU.

* 2-bit (MXNet PR #8662 "Dist kvstore"; CD-SGD eq. 10): every rank quantises
  its gradient with its own residual, the packed codes (n/16 words per rank)
  are all-gathered, and every rank applies the same dequant-sum + update to
  its replica of the weights -- the replicas stay bit-identical.
* QSGD (Knowl 3, synchronous parallel QSGD): every rank quantises its
  gradient (worker index = rank), codes and bucket norms are all-gathered,
  and every rank forms the same dequantised average.
* SAPS + EASGD ("Communication-Efficient Decentralized Learning with
  Sparsification and Adaptive Peer Selection", section II; EASGD from the
  IMerge design notes): every rank draws the round's shared mask, compacts
  its masked coordinates, swaps the gathered values with its matched peer
  (send/receive of a fixed-capacity buffer: the indices are the same on both
  sides and need not travel), averages them in, then all-reduces a copy of
  its model to take the elastic step against its replica of the center.

The kernels are reached through an ``ops`` object, by default the library's
CUDA entry points (CUDA tensors only, no fallback).  Nothing here computes a
value itself: this module only allocates the exchange buffers and orders the
collectives.
"""
from __future__ import annotations

import torch
import torch.distributed as dist

from . import (GC_UPD_SGD, code_words, easgd_step_from_sum, gc_2bit_dequant_sum_update, gc_2bit_quantize,
               qsgd_code_bytes, qsgd_dequant_sum, qsgd_num_buckets, qsgd_quantize, saps_mask_compact,
               saps_pair_average_remote, saps_round_seed, saps_workspace_bytes)


class KernelOps:
    """The library's CUDA entry points, as the exchange classes call them."""
    quantize_2bit = staticmethod(gc_2bit_quantize)
    dequant_sum_update_2bit = staticmethod(gc_2bit_dequant_sum_update)
    qsgd_quantize = staticmethod(qsgd_quantize)
    qsgd_dequant_sum = staticmethod(qsgd_dequant_sum)
    saps_mask_compact = staticmethod(saps_mask_compact)
    saps_pair_average_remote = staticmethod(saps_pair_average_remote)
    easgd_step_from_sum = staticmethod(easgd_step_from_sum)


def _group_info(group):
    return dist.get_world_size(group), dist.get_rank(group)


def peer_of(pairs, rank: int) -> int:
    """The partner of ``rank`` in a perfect matching given as pairs
    (pairs[2q], pairs[2q+1])."""
    for q in range(0, len(pairs), 2):
        if pairs[q] == rank:
            return pairs[q + 1]
        if pairs[q + 1] == rank:
            return pairs[q]
    raise ValueError(f"rank {rank} is not in the matching")


class TwoBitExchange:
    """One 2-bit data-parallel step per call: quantise locally, all-gather the
    codes, apply the dequant-sum update on every rank."""

    def __init__(self, n: int, threshold: float, device, group=None, ops=None):
        self.n, self.t, self.group = n, float(threshold), group
        self.world, self.rank = _group_info(group)
        self.ops = ops or KernelOps
        self.codes = torch.empty(code_words(n), dtype=torch.int32, device=device)
        # flat buffers (gloo and NCCL both take a 1-D output), used as [world, ...]
        self._gathered = torch.empty(self.world * code_words(n), dtype=torch.int32, device=device)
        self.gathered = self._gathered.view(self.world, code_words(n))

    def step(self, grad, residual, weights=None, lr: float = 0.0, kind: int = GC_UPD_SGD, alpha: float = 0.0,
             center=None, out=None):
        self.ops.quantize_2bit(grad, residual, self.codes, self.t)
        dist.all_gather_into_tensor(self._gathered, self.codes, group=self.group)
        self.ops.dequant_sum_update_2bit(list(self.gathered.unbind(0)), self.n, self.t, kind, lr=lr, alpha=alpha,
                                         center=center, weights=weights, out=out)
        return self.gathered


class QSGDExchange:
    """Synchronous parallel QSGD: quantise locally (worker = rank), all-gather
    codes and norms, and form the dequantised sum (scale 1/world: the
    average) on every rank."""

    def __init__(self, n: int, bucket: int, s: int, seed: int, device, group=None, ops=None):
        self.n, self.bucket, self.s, self.seed, self.group = n, bucket, s, seed, group
        self.world, self.rank = _group_info(group)
        self.ops = ops or KernelOps
        nb, cb = qsgd_num_buckets(n, bucket), qsgd_code_bytes(n, s)
        self.codes = torch.empty(cb, dtype=torch.uint8, device=device)
        self.norms = torch.empty(nb, dtype=torch.float32, device=device)
        self._g_codes = torch.empty(self.world * cb, dtype=torch.uint8, device=device)
        self._g_norms = torch.empty(self.world * nb, dtype=torch.float32, device=device)
        self.g_codes = self._g_codes.view(self.world, cb)
        self.g_norms = self._g_norms.view(self.world, nb)

    def step(self, grad, out, scale: float | None = None):
        self.ops.qsgd_quantize(grad, self.bucket, self.s, self.seed, self.rank, self.norms, self.codes)
        dist.all_gather_into_tensor(self._g_codes, self.codes, group=self.group)
        dist.all_gather_into_tensor(self._g_norms, self.norms, group=self.group)
        self.ops.qsgd_dequant_sum(list(self.g_codes.unbind(0)), list(self.g_norms.unbind(0)), self.n, self.bucket,
                                  self.s, 1.0 / self.world if scale is None else scale, out)


class SAPSExchange:
    """One SAPS gossip round + EASGD elastic step per call, this rank's
    worker against its matched peer."""

    def __init__(self, n: int, p: float, base_seed: int, alpha: float, beta: float, device, group=None,
                 capacity: int | None = None, ops=None):
        self.n, self.p, self.base_seed, self.alpha, self.beta, self.group = n, p, base_seed, alpha, beta, group
        self.world, self.rank = _group_info(group)
        self.ops = ops or KernelOps
        cap = capacity if capacity is not None else int(n * p * 1.2 + 10_000)
        self.capacity = min(cap, n)
        self.idx = torch.empty(self.capacity, dtype=torch.int32, device=device)
        self.count = torch.zeros(1, dtype=torch.int64, device=device)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        self.ws = torch.empty(saps_workspace_bytes(n), dtype=torch.uint8, device=device)
        self.mine = self.peer = self.sum = None     # the model's dtype, at the first round

    def round(self, t: int, model, center, pairs):
        """Round t with the matching ``pairs`` (the same on every rank, e.g.
        saps_matching or saps_matching_bandwidth of the round).  The device
        status (capacity overflow, look-back timeout) is left in self.status."""
        if self.sum is None:
            self.mine = torch.zeros(self.capacity, dtype=model.dtype, device=model.device)
            self.peer = torch.zeros(self.capacity, dtype=model.dtype, device=model.device)
            self.sum = torch.empty(self.n, dtype=model.dtype, device=model.device)
        seed_t = saps_round_seed(self.base_seed, t)
        self.status.zero_()
        self.ops.saps_mask_compact(self.n, self.p, seed_t, [model], self.idx, [self.mine], self.count, self.ws,
                                   self.status)
        peer = peer_of(pairs, self.rank)
        ops = [dist.P2POp(dist.isend, self.mine, peer, group=self.group),
               dist.P2POp(dist.irecv, self.peer, peer, group=self.group)]
        for req in dist.batch_isend_irecv(ops):
            req.wait()
        self.ops.saps_pair_average_remote(model, self.idx, self.count, self.mine, self.peer)
        self.sum.copy_(model)
        dist.all_reduce(self.sum, group=self.group)
        self.ops.easgd_step_from_sum(model, self.sum, self.world, self.alpha, self.beta, center)
