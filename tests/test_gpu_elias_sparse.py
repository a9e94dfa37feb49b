"""GPU parity of QSGD's sparse-regime Elias coding (Knowl 2 items 1 and 1')
through the C ABI: streams and offsets bit-exact with the oracle's encoder on
the same codes, the decoder's codes and norms equal to the oracle's decode,
and corrupt streams reported."""
import numpy as np
import pytest
import torch

import gradient_compression_sgd_gc_gb300 as gc
from gradient_compression_sgd_gc_gb300 import workloads as wl
import oracle
from gpu_helpers import check_guard, guarded, host_f32, host_u32

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _codes_for(n, d, s, seed):
    cfg = wl.scaled(wl.QSGD_S7, n, seed=seed)
    v = wl.qsgd_grad(cfg, 1, device="cpu").numpy().astype(np.float32)
    v[: min(n, 300)] = 0.0                     # a whole zero bucket at the start for d <= 256
    v[300:320] = -0.0
    return oracle.qsgd_quantize(v, d, s, 77, 1)


def _canonical(codes, n, s):
    """Codes with every level-0 coordinate's sign cleared."""
    if s <= 7:
        nib = np.stack([codes >> 4, codes & 15], axis=1).reshape(-1)
        nib = np.where((nib & 7) == 0, 0, nib)
        if n % 2:
            nib[n] = 0
        return ((nib[0::2] << 4) | nib[1::2]).astype(np.uint8)
    return np.where((codes & 127) == 0, 0, codes).astype(np.uint8)


def _encode(codes_h, norms_h, n, d, s):
    nb = gc.qsgd_num_buckets(n, d)
    cap = gc.qsgd_elias_sparse_max_words(n, d)
    words = guarded(cap, torch.int32)
    offs = guarded(nb + 1, torch.int32)
    ws = torch.empty(gc.qsgd_elias_workspace_bytes(n, d), dtype=torch.uint8, device=DEV)
    gc.qsgd_elias_encode_sparse(torch.from_numpy(codes_h).to(DEV), torch.from_numpy(norms_h).to(DEV), n, d, s,
                                words[:cap], offs[:nb + 1], ws)
    return words, offs, cap, nb


@pytest.mark.parametrize("s", [1, 2, 7, 22, 127])
@pytest.mark.parametrize("n,d", [(1, 128), (300, 128), (5 * 512 + 297, 512), (100_003, 128), (70_001, 2048)])
def test_sparse_encode_bit_exact(n, d, s):
    rn, rc = _codes_for(n, d, s, 3)
    ref_w, ref_off = oracle.qsgd_elias_encode_sparse(rc, rn, n, d, s)
    words, offs, cap, nb = _encode(rc, rn, n, d, s)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(host_u32(offs[:nb + 1]), ref_off)
    np.testing.assert_array_equal(host_u32(words[:ref_w.size]), ref_w)
    check_guard(words, cap)
    check_guard(offs, nb + 1)


@pytest.mark.parametrize("s", [1, 7, 127])
@pytest.mark.parametrize("n,d", [(1, 512), (5 * 512 + 297, 512), (100_003, 128), (70_001, 2048)])
def test_sparse_decode_of_the_oracle_stream(n, d, s):
    rn, rc = _codes_for(n, d, s, 4)
    ref_w, ref_off = oracle.qsgd_elias_encode_sparse(rc, rn, n, d, s)
    nb, cb = gc.qsgd_num_buckets(n, d), gc.qsgd_code_bytes(n, s)
    codes = guarded(cb, torch.uint8, fill=0xA5A5A5A5)
    norms = guarded(nb, torch.float32)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    gc.qsgd_elias_decode_sparse(torch.from_numpy(ref_w.view(np.int32)).to(DEV),
                                torch.from_numpy(ref_off.view(np.int32)).to(DEV), n, d, s, codes[:cb], norms[:nb], st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    np.testing.assert_array_equal(codes[:cb].cpu().numpy(), _canonical(rc, n, s))
    np.testing.assert_array_equal(host_f32(norms[:nb]).view(np.uint32), rn.view(np.uint32))
    check_guard(codes, cb, fill=0xA5A5A5A5)
    check_guard(norms, nb)


@pytest.mark.parametrize("s", [1, 7, 127])
def test_sparse_round_trip_on_gpu_codes(s):
    """GPU quantise -> sparse encode -> sparse decode gives back the codes
    (level-0 signs cleared) and the norms, on the configured bucket of 512."""
    n, d = 1_000_003, 512
    cfg = wl.scaled(wl.QSGD_S7, n)
    v = wl.qsgd_grad(cfg, 0, device=DEV)
    nb, cb = gc.qsgd_num_buckets(n, d), gc.qsgd_code_bytes(n, s)
    norms = torch.empty(nb, device=DEV)
    codes = torch.empty(cb, dtype=torch.uint8, device=DEV)
    gc.qsgd_quantize(v, d, s, 42, 0, norms, codes)
    cap = gc.qsgd_elias_sparse_max_words(n, d)
    words = torch.empty(cap, dtype=torch.int32, device=DEV)
    offs = torch.empty(nb + 1, dtype=torch.int32, device=DEV)
    ws = torch.empty(gc.qsgd_elias_workspace_bytes(n, d), dtype=torch.uint8, device=DEV)
    gc.qsgd_elias_encode_sparse(codes, norms, n, d, s, words, offs, ws)
    dc = torch.empty_like(codes)
    dn = torch.empty_like(norms)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    gc.qsgd_elias_decode_sparse(words, offs, n, d, s, dc, dn, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    np.testing.assert_array_equal(dc.cpu().numpy(), _canonical(codes.cpu().numpy(), n, s))
    assert torch.equal(dn.view(torch.int32), norms.view(torch.int32))
    total = int(host_u32(offs[nb:nb + 1])[0])
    ref_w, _ = oracle.qsgd_elias_encode_sparse(codes.cpu().numpy(), host_f32(norms), n, d, s)
    assert total == ref_w.size
    print(f"s={s}: sparse stream {32 * total / n:.3f} bits per coordinate")


def test_sparse_corrupt_streams_are_reported():
    n, d, s = 2048, 512, 7
    rn, rc = _codes_for(n, d, s, 5)
    ref_w, ref_off = oracle.qsgd_elias_encode_sparse(rc, rn, n, d, s)
    nb, cb = gc.qsgd_num_buckets(n, d), gc.qsgd_code_bytes(n, s)

    def decode(words, offs, s_dec=s):
        codes = torch.empty(gc.qsgd_code_bytes(n, s_dec), dtype=torch.uint8, device=DEV)
        norms = torch.empty(nb, device=DEV)
        st = torch.zeros(1, dtype=torch.int32, device=DEV)
        gc.qsgd_elias_decode_sparse(torch.from_numpy(words.view(np.int32)).to(DEV),
                                    torch.from_numpy(offs.view(np.int32)).to(DEV), n, d, s_dec, codes, norms, st)
        torch.cuda.synchronize()
        return int(st.item())

    assert decode(ref_w, ref_off) == 0
    bad = ref_w.copy()
    bad[ref_off[2] + 1] = 0xFFFFFFFF              # a codeword longer than any valid one
    assert decode(bad, ref_off) == gc.GC_ERR_CORRUPT
    short = ref_off.copy()
    short[1] = short[0] + 1                       # bucket 0 keeps only its norm word
    assert decode(ref_w, short) == gc.GC_ERR_CORRUPT
    # levels above the decoder's s: an s = 127 stream read as s = 7
    rn8, rc8 = _codes_for(n, d, 127, 6)
    w8, o8 = oracle.qsgd_elias_encode_sparse(rc8, rn8, n, d, 127)
    assert decode(w8, o8, s_dec=7) == gc.GC_ERR_CORRUPT


def test_sparse_encode_capacity_refused():
    n, d, s = 4096, 512, 7
    nb = gc.qsgd_num_buckets(n, d)
    cap = gc.qsgd_elias_sparse_max_words(n, d)
    codes = torch.zeros(gc.qsgd_code_bytes(n, s), dtype=torch.uint8, device=DEV)
    norms = torch.zeros(nb, device=DEV)
    words = torch.empty(cap - 1, dtype=torch.int32, device=DEV)
    offs = torch.empty(nb + 1, dtype=torch.int32, device=DEV)
    ws = torch.empty(gc.qsgd_elias_workspace_bytes(n, d), dtype=torch.uint8, device=DEV)
    with pytest.raises(RuntimeError, match="GC_ERR_CAPACITY"):
        gc.qsgd_elias_encode_sparse(codes, norms, n, d, s, words, offs, ws)


def test_sparse_empty_input():
    """n = 0: the sparse encoder writes only offsets[0] = 0; the decoder
    touches nothing."""
    offsets = torch.full((4,), 7, dtype=torch.int32, device=DEV)
    words = torch.zeros(4, dtype=torch.int32, device=DEV)
    codes = torch.full((16,), 9, dtype=torch.uint8, device=DEV)
    norms = torch.zeros(4, device=DEV)
    ws = torch.full((64,), 0xA5, dtype=torch.uint8, device=DEV)
    gc.qsgd_elias_encode_sparse(codes, norms, 0, 512, 7, words, offsets, ws)
    gc.qsgd_elias_decode_sparse(words, offsets, 0, 512, 7, codes, norms)
    torch.cuda.synchronize()
    assert host_u32(offsets).tolist() == [0, 7, 7, 7]
    assert codes.cpu().tolist() == [9] * 16
    assert gc.qsgd_elias_encode_status(ws) == gc.GC_OK
