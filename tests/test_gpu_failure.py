"""Failure detection without a GPU fault: a compaction tile that never
publishes its look-back state makes its successors' bounded waits run out;
the kernel still finishes, GC_ERR_TIMEOUT reaches the caller's device status,
and the context stays usable for the next, correct call."""
import ctypes

import numpy as np
import pytest
import torch

import gradient_compression_sgd_gc_gb300 as gc
from gradient_compression_sgd_gc_gb300 import workloads as wl
import oracle

pytestmark = pytest.mark.gpu
DEV = "cuda"


def test_withheld_lookback_state_times_out_and_recovers():
    n, W, p = 100_000, 2, 0.01
    models = [wl.normal(n, 0.05, 70 + w, device=DEV) for w in range(W)]
    idx = torch.empty(n, dtype=torch.int32, device=DEV)
    vals = [torch.empty(n, device=DEV) for _ in range(W)]
    cnt = torch.zeros(1, dtype=torch.int64, device=DEV)
    ws = torch.empty(gc.saps_workspace_bytes(n), dtype=torch.uint8, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    lib = gc.load()
    mp = (ctypes.c_void_p * W)(*[m.data_ptr() for m in models])
    vp = (ctypes.c_void_p * W)(*[v.data_ptr() for v in vals])
    stream = torch.cuda.current_stream().cuda_stream
    rc = lib.gc_testing_saps_mask_compact_withhold(n, p, 1234, mp, W, idx.data_ptr(), vp, n, cnt.data_ptr(),
                                                   ws.data_ptr(), ws.numel(), st.data_ptr(), 3, 50_000_000,
                                                   stream)
    assert rc == gc.GC_OK
    torch.cuda.synchronize()
    assert int(st.item()) == gc.GC_ERR_TIMEOUT
    # the context is fine and the next call is correct
    st.zero_()
    gc.saps_mask_compact(n, p, 1234, models, idx, vals, cnt, ws, st)
    torch.cuda.synchronize()
    K, ridx, _ = oracle.saps_mask_compact(n, p, 1234, [m.cpu().numpy().astype(np.float64) for m in models])
    assert int(st.item()) == 0 and int(cnt.item()) == K
    np.testing.assert_array_equal(idx[:K].cpu().numpy().view(np.uint32), ridx)
