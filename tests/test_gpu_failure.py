"""Failure detection without a GPU fault: a compaction tile (or an Elias
bucket) that never publishes its look-back state makes its successors'
bounded waits run out; the kernel still finishes, GC_ERR_TIMEOUT reaches the
caller's device status, and the context stays usable for the next, correct
call."""
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


def test_elias_encoder_withheld_bucket_times_out_and_recovers():
    """The one-pass Elias encoder: bucket 70 (in the second CTA's chunk)
    never publishes; the buckets after it give up after 20 ms, the status word
    in the workspace reads GC_ERR_TIMEOUT, and the next call writes the
    oracle's stream."""
    n, d, s = 512 * 200 + 77, 512, 7
    v = wl.qsgd_grad(wl.scaled(wl.QSGD_S7, n), 0, device="cpu").numpy()
    norms, codes = oracle.qsgd_quantize(v, d, s, 42, 0)
    nb = gc.qsgd_num_buckets(n, d)
    cap = gc.qsgd_elias_max_words(n, d, s)
    c, nm = torch.from_numpy(codes).to(DEV), torch.from_numpy(norms).to(DEV)
    words = torch.empty(cap, dtype=torch.int32, device=DEV)
    offs = torch.empty(nb + 1, dtype=torch.int32, device=DEV)
    ws = torch.empty(gc.qsgd_elias_workspace_bytes(n, d), dtype=torch.uint8, device=DEV)
    lib = gc.load()
    stream = torch.cuda.current_stream().cuda_stream
    rc = lib.gc_testing_qsgd_elias_encode_withhold(c.data_ptr(), nm.data_ptr(), n, d, s, words.data_ptr(), cap,
                                                   offs.data_ptr(), ws.data_ptr(), ws.numel(), 70, 20_000_000,
                                                   stream)
    assert rc == gc.GC_OK
    torch.cuda.synchronize()
    assert gc.qsgd_elias_encode_status(ws) == gc.GC_ERR_TIMEOUT
    gc.qsgd_elias_encode(c, nm, n, d, s, words, offs, ws)
    torch.cuda.synchronize()
    assert gc.qsgd_elias_encode_status(ws) == gc.GC_OK
    ref_w, ref_off = oracle.qsgd_elias_encode(codes, norms, n, d, s)
    np.testing.assert_array_equal(offs.cpu().numpy().view(np.uint32), ref_off)
    np.testing.assert_array_equal(words[:ref_w.size].cpu().numpy().view(np.uint32), ref_w)
