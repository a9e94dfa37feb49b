"""The allocation-free compaction entry point, saps_mask_compact_noalloc.

It exists for callers that cannot hand the library a workspace: a plug-in
inside a host framework whose device allocator it may not call, a loop whose
device memory is fixed up front, code that must avoid the implicit
synchronisation of cudaMalloc/cudaFree.  Its scratch is a fixed array inside
the library, so two calls in a row must each clear what they use: the second
call here runs with a different seed on the same size, and would read the first
call's look-back states if they were left behind.  Results must equal the
workspace entry point's bit for bit (counts, indices, gathered values), the
tolerance these tests use for integer and copied data.

This file is collected last so that a failure here cannot hide other tests.
"""
import numpy as np
import pytest
import torch

import gradient_compression_sgd_gc_gb300 as gc
from gradient_compression_sgd_gc_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _buffers(n, W, capacity):
    idx = torch.empty(capacity, dtype=torch.int32, device=DEV)
    vals = [torch.empty(capacity, device=DEV) for _ in range(W)]
    cnt = torch.zeros(1, dtype=torch.int64, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    return idx, vals, cnt, st


def _host(idx, vals, cnt, st):
    torch.cuda.synchronize()
    K = int(cnt.item())
    k = min(K, idx.numel())
    return K, idx[:k].cpu().numpy(), [v[:k].cpu().numpy() for v in vals], int(st.item())


def test_noalloc_matches_workspace_entry_on_two_calls():
    n, W, p = 3_000_017, 4, 0.01
    capacity = 40_000
    models = [wl.normal(n, 0.05, 4000 + w, device=DEV) for w in range(W)]
    ws = torch.empty(gc.saps_workspace_bytes(n), dtype=torch.uint8, device=DEV)
    for call, seed_t in enumerate((gc.saps_round_seed(5, 0), gc.saps_round_seed(5, 1))):
        a = _buffers(n, W, capacity)
        gc.saps_mask_compact(n, p, seed_t, models, a[0], a[1], a[2], ws, a[3])
        b = _buffers(n, W, capacity)
        gc.saps_mask_compact_noalloc(n, p, seed_t, models, b[0], b[1], b[2], b[3])
        Ka, ia, va, sa = _host(*a)
        Kb, ib, vb, sb = _host(*b)
        assert sa == 0 and sb == 0, f"call {call}: device status {sa}, {sb}"
        assert Ka == Kb and Ka > 0, f"call {call}: counts {Ka} vs {Kb}"
        np.testing.assert_array_equal(ib, ia)
        for w in range(W):
            np.testing.assert_array_equal(vb[w].view(np.uint32), va[w].view(np.uint32))


def test_noalloc_rejects_sizes_beyond_its_scratch():
    lib = gc.load()
    import ctypes
    fake = ctypes.c_void_p(0x10000)
    ptrs = (ctypes.c_void_p * 1)(0x10000)
    st = lib.saps_mask_compact_noalloc(gc.GC_NOALLOC_MAX_N + 1, 0.01, 1, ptrs, 1, fake, ptrs, 10,
                                       fake, fake, None)
    assert st == gc.GC_ERR_INVALID
    with pytest.raises(ValueError, match="scratch limit"):
        gc.saps_mask_compact_noalloc(gc.GC_NOALLOC_MAX_N + 1, 0.01, 1, [], None, [], None, None)
