"""GPU parity of the quarter-marked dense Elias stream (QSGD Knowl 2, dense
regime, with side information added here so that a bucket's four quarters
decode in parallel) through the C ABI.

qsgd_elias_encode_marked must write the oracle's stream and offsets word for
word and the oracle's quarter marks value for value (integer work:
bit-exact); qsgd_elias_decode_quarters must give back the oracle decoder's
codes and norms exactly, and report streams whose quarters do not meet at
their marks.
"""
import numpy as np
import pytest
import torch

import gradient_compression_sgd_gc_gb300 as gc
from gradient_compression_sgd_gc_gb300 import workloads as wl
import oracle
from gpu_helpers import check_guard, guarded, host_f32, host_u32

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _oracle_codes(cfg, n, bucket, s, worker=0):
    v = wl.qsgd_grad(wl.scaled(cfg, n), worker, device="cpu").numpy()
    return oracle.qsgd_quantize(v, bucket, s, cfg.seed, worker)


def _host_u16(t):
    return t.cpu().numpy().view(np.uint16)


def _encode_marked(codes_h, norms_h, n, bucket, s):
    nb = gc.qsgd_num_buckets(n, bucket)
    cap = gc.qsgd_elias_max_words(n, bucket, s)
    words = guarded(cap, torch.int32)
    offsets = guarded(nb + 1, torch.int32)
    marks = guarded(3 * nb, torch.int16)
    ws = torch.empty(max(16, gc.qsgd_elias_workspace_bytes(n, bucket)), dtype=torch.uint8, device=DEV)
    ws.fill_(0xA5)
    gc.qsgd_elias_encode_marked(torch.from_numpy(codes_h).to(DEV), torch.from_numpy(norms_h).to(DEV), n, bucket,
                                s, words[:cap], offsets[:nb + 1], marks[:3 * nb], ws)
    torch.cuda.synchronize()
    check_guard(words, cap)
    check_guard(offsets, nb + 1)
    check_guard(marks, 3 * nb)
    return words, offsets, marks[:3 * nb]


def _decode_quarters(words, offsets, marks, n, bucket, s):
    nb, cb = gc.qsgd_num_buckets(n, bucket), gc.qsgd_code_bytes(n, s)
    codes = guarded(cb, torch.uint8)
    codes[:cb].fill_(0xEE)                 # every byte must be written
    norms = guarded(nb, torch.float32)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    gc.qsgd_elias_decode_quarters(words, offsets, marks, n, bucket, s, codes[:cb], norms[:nb], st)
    torch.cuda.synchronize()
    check_guard(codes, cb)
    check_guard(norms, nb)
    return codes[:cb].cpu().numpy(), host_f32(norms[:nb]), int(st.item())


def _dev_u16(a):
    return torch.from_numpy(a.view(np.int16).copy()).to(DEV)


def _dev_u32(a):
    return torch.from_numpy(a.view(np.int32).copy()).to(DEV)


CASES = [
    (wl.QSGD_S7, 512 * 150 + 297, 512, 7),       # 151 buckets: 3 CTAs of 64, ragged odd tail
    (wl.QSGD_S7, 128 * 400 + 77, 128, 7),        # quarters of 32 coordinates; tail ends in quarter 2
    (wl.QSGD_S7, 256 * 70, 256, 1),
    (wl.QSGD_S127, 512 * 130 + 1, 512, 127),     # a last bucket of one coordinate
    (wl.QSGD_S127, 2048 * 70 + 1001, 2048, 127),
    (wl.QSGD_S127, 512 * 129 + 384, 512, 22),    # tail ends exactly on a quarter
    (wl.QSGD_S7, 1024 * 65, 1024, 5),
    (wl.QSGD_S7, 300, 512, 7),                   # one short bucket
    (wl.QSGD_S127, 1, 128, 127),
]


@pytest.mark.parametrize("cfg,n,bucket,s", CASES, ids=lambda x: getattr(x, "name", str(x)))
def test_marked_encode_and_quarter_decode(cfg, n, bucket, s):
    norms, codes = _oracle_codes(cfg, n, bucket, s)
    nb = gc.qsgd_num_buckets(n, bucket)
    ref_w, ref_off = oracle.qsgd_elias_encode(codes, norms, n, bucket, s)
    ref_m = oracle.qsgd_elias_quarter_marks(codes, n, bucket, s)
    words, offsets, marks = _encode_marked(codes, norms, n, bucket, s)
    np.testing.assert_array_equal(host_u32(offsets[:nb + 1]), ref_off)
    np.testing.assert_array_equal(host_u32(words[:ref_w.size]), ref_w)
    np.testing.assert_array_equal(_host_u16(marks), ref_m)
    rc, rn = oracle.qsgd_elias_decode(ref_w, ref_off, n, bucket, s)
    dc, dn, st = _decode_quarters(words, offsets, marks, n, bucket, s)
    assert st == 0
    np.testing.assert_array_equal(dc, rc)
    np.testing.assert_array_equal(dn.view(np.uint32), rn.view(np.uint32))


@pytest.mark.parametrize("s", [7, 127])
def test_quarter_decode_of_the_oracle_stream(s):
    """Stream and marks from the oracle alone: the quarter decoder reads what
    the pages' code and the marks' definition fix, not the GPU encoder."""
    cfg, n, bucket = (wl.QSGD_S7 if s == 7 else wl.QSGD_S127), 512 * 200 + 129, 512
    norms, codes = _oracle_codes(cfg, n, bucket, s, worker=2)
    ref_w, ref_off = oracle.qsgd_elias_encode(codes, norms, n, bucket, s)
    ref_m = oracle.qsgd_elias_quarter_marks(codes, n, bucket, s)
    dc, dn, st = _decode_quarters(_dev_u32(ref_w), _dev_u32(ref_off), _dev_u16(ref_m), n, bucket, s)
    rc, rn = oracle.qsgd_elias_decode(ref_w, ref_off, n, bucket, s)
    assert st == 0
    np.testing.assert_array_equal(dc, rc)
    np.testing.assert_array_equal(dn.view(np.uint32), rn.view(np.uint32))


def _pack(level, sign, n, s):
    """Codes in qsgd_quantize's layout: sign-magnitude, 4 bits (first
    coordinate in the high nibble) for s <= 7, else 8 bits."""
    if s <= 7:
        nib = np.zeros(2 * ((n + 1) // 2), np.int64)
        nib[:n] = (sign << 3) | level
        return ((nib[0::2] << 4) | nib[1::2]).astype(np.uint8)
    return ((sign << 7) | level).astype(np.uint8)


@pytest.mark.parametrize("s", [7, 127])
def test_extreme_buckets(s):
    """All-zero buckets (one bit per coordinate, quarters 1 bit apart per
    coordinate) and buckets at the longest codeword everywhere."""
    n, bucket = 512 * 70 + 201, 512
    level = np.zeros(n, np.int64)
    sign = np.zeros(n, np.int64)
    level[512 * 3:512 * 4] = s                    # every coordinate at level s
    sign[512 * 3:512 * 4:3] = 1
    level[512 * 5:512 * 6:2] = s                  # level s and 0 alternating
    sign[512 * 5:512 * 6] = 1                     # (the level-0 signs are not sent)
    level[512 * 70:] = s                          # the short last bucket too
    norms = np.random.default_rng(5).uniform(0.5, 2.0, gc.qsgd_num_buckets(n, bucket)).astype(np.float32)
    codes = _pack(level, sign, n, s)
    ref_w, ref_off = oracle.qsgd_elias_encode(codes, norms, n, bucket, s)
    ref_m = oracle.qsgd_elias_quarter_marks(codes, n, bucket, s)
    assert int(ref_m[0]) == 32 + 128              # a zero bucket: one bit per coordinate
    words, offsets, marks = _encode_marked(codes, norms, n, bucket, s)
    np.testing.assert_array_equal(host_u32(words[:ref_w.size]), ref_w)
    np.testing.assert_array_equal(_host_u16(marks), ref_m)
    dc, dn, st = _decode_quarters(words, offsets, marks, n, bucket, s)
    rc, _ = oracle.qsgd_elias_decode(ref_w, ref_off, n, bucket, s)
    assert st == 0
    np.testing.assert_array_equal(dc, rc)


def test_corrupt_middle_mark_of_four_bit_streams():
    """4-bit codes decode in halves from the middle mark (marks[3b + 1]): a
    middle mark one bit off, or a short bucket's middle mark not at its end,
    is reported."""
    cfg, n, bucket, s = wl.QSGD_S7, 512 * 8 + 200, 512, 7
    norms, codes = _oracle_codes(cfg, n, bucket, s)
    ref_w, ref_off = oracle.qsgd_elias_encode(codes, norms, n, bucket, s)
    ref_m = oracle.qsgd_elias_quarter_marks(codes, n, bucket, s)
    words, offs = _dev_u32(ref_w), _dev_u32(ref_off)
    assert _decode_quarters(words, offs, _dev_u16(ref_m), n, bucket, s)[2] == 0
    for i in (1, 3 * 5 + 1, 3 * 8 + 1):           # buckets 0 and 5, and the short last bucket (200)
        for delta in (1, -1):
            m = ref_m.copy()
            m[i] = np.uint16(int(m[i]) + delta)
            assert _decode_quarters(words, offs, _dev_u16(m), n, bucket, s)[2] == gc.GC_ERR_CORRUPT


def test_corrupt_marks_and_streams_are_reported():
    cfg, n, bucket, s = wl.QSGD_S127, 512 * 8 + 100, 512, 127
    norms, codes = _oracle_codes(cfg, n, bucket, s)
    ref_w, ref_off = oracle.qsgd_elias_encode(codes, norms, n, bucket, s)
    ref_m = oracle.qsgd_elias_quarter_marks(codes, n, bucket, s)
    words, offs = _dev_u32(ref_w), _dev_u32(ref_off)
    assert _decode_quarters(words, offs, _dev_u16(ref_m), n, bucket, s)[2] == 0
    # a mark one bit off: quarters 1 and 2 of full buckets, and in the short
    # last bucket (100 coordinates, all in quarter 0) the marks past its end
    for i in (0, 4, 3 * 8, 3 * 8 + 2):
        m = ref_m.copy()
        m[i] += 1
        assert _decode_quarters(words, offs, _dev_u16(m), n, bucket, s)[2] == gc.GC_ERR_CORRUPT
    m = ref_m.copy()
    m[5] = 0xFFFF                                 # a mark past the bucket's words
    assert _decode_quarters(words, offs, _dev_u16(m), n, bucket, s)[2] == gc.GC_ERR_CORRUPT
    trunc = ref_off.copy()
    trunc[4] = ref_off[3] + 1                     # bucket 3 cut to its norm word
    assert _decode_quarters(words, _dev_u32(trunc), _dev_u16(ref_m), n, bucket, s)[2] == gc.GC_ERR_CORRUPT
    assert int((codes & 127).max()) > 22          # levels above the decoder's s
    assert _decode_quarters(words, offs, _dev_u16(ref_m), n, bucket, 22)[2] == gc.GC_ERR_CORRUPT


@pytest.mark.parametrize("s", [7, 127])
def test_round_trip_on_gpu_codes(s):
    """GPU quantise -> marked encode -> quarter decode gives back the plain
    decoder's codes and the quantiser's norms (about 1 M coordinates)."""
    n, d = 1_000_003, 512
    v = wl.qsgd_grad(wl.scaled(wl.QSGD_S7, n), 0, device=DEV)
    nb, cb = gc.qsgd_num_buckets(n, d), gc.qsgd_code_bytes(n, s)
    norms = torch.empty(nb, device=DEV)
    codes = torch.empty(cb, dtype=torch.uint8, device=DEV)
    gc.qsgd_quantize(v, d, s, 42, 0, norms, codes)
    cap = gc.qsgd_elias_max_words(n, d, s)
    words = torch.empty(cap, dtype=torch.int32, device=DEV)
    offs = torch.empty(nb + 1, dtype=torch.int32, device=DEV)
    marks = torch.empty(3 * nb, dtype=torch.int16, device=DEV)
    ws = torch.empty(gc.qsgd_elias_workspace_bytes(n, d), dtype=torch.uint8, device=DEV)
    gc.qsgd_elias_encode_marked(codes, norms, n, d, s, words, offs, marks, ws)
    a, an = torch.empty_like(codes), torch.empty_like(norms)
    b, bn = torch.empty_like(codes), torch.empty_like(norms)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    gc.qsgd_elias_decode(words, offs, n, d, s, a, an, st)
    gc.qsgd_elias_decode_quarters(words, offs, marks, n, d, s, b, bn, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(a, b)
    assert torch.equal(bn.view(torch.int32), norms.view(torch.int32))
    ref_m = oracle.qsgd_elias_quarter_marks(codes.cpu().numpy(), n, d, s)
    np.testing.assert_array_equal(_host_u16(marks), ref_m)


@pytest.mark.parametrize("cfg", [wl.QSGD_S7, wl.QSGD_S127], ids=lambda c: c.name)
def test_full_size_marks_and_quarter_decode(cfg):
    """The QSGD workload at full size (61,100,840 coordinates, 119,338 buckets
    of 512, last 296): marks equal the oracle's, and the quarter decoder
    returns the oracle decoder's codes."""
    n, d, s = cfg.n, cfg.bucket, cfg.s
    v = wl.qsgd_grad(cfg, 1, device="cpu").numpy()
    norms, codes = oracle.qsgd_quantize(v, d, s, cfg.seed, 1)
    del v
    ref_w, ref_off = oracle.qsgd_elias_encode(codes, norms, n, d, s)
    ref_m = oracle.qsgd_elias_quarter_marks(codes, n, d, s)
    words, offsets, marks = _encode_marked(codes, norms, n, d, s)
    np.testing.assert_array_equal(host_u32(words[:ref_w.size]), ref_w)
    np.testing.assert_array_equal(_host_u16(marks), ref_m)
    dc, dn, st = _decode_quarters(words, offsets, marks, n, d, s)
    rc, rn = oracle.qsgd_elias_decode(ref_w, ref_off, n, d, s)
    assert st == 0
    np.testing.assert_array_equal(dc, rc)
    np.testing.assert_array_equal(dn.view(np.uint32), rn.view(np.uint32))


@pytest.mark.parametrize("s,nb", [(7, 90_000), (127, 66_000)])
def test_buckets_past_the_staged_words(s, nb):
    """Every coordinate at level s (the longest codeword: 129 words a bucket
    of 512 for 4-bit codes, 241 for 8-bit codes), with enough buckets that a
    decoding CTA's buckets hold about twice the words its shared memory
    stages: its last buckets are read from global memory, by the whole-bucket
    and by the quarter decoder.  Both give back the input codes (all levels
    non-zero, so the input is the canonical form), and the marked encoder
    writes the oracle's stream and marks."""
    n, d = 512 * nb, 512
    if s <= 7:
        codes = np.full(n // 2, ((0x8 | s) << 4) | s, np.uint8)     # signs - and + alternating
    else:
        codes = np.empty(n, np.uint8)
        codes[0::2], codes[1::2] = 0x80 | s, s
    norms = np.random.default_rng(3).uniform(0.5, 2.0, nb).astype(np.float32)
    ref_w, ref_off = oracle.qsgd_elias_encode(codes, norms, n, d, s)
    assert int(ref_off[1]) == (129 if s <= 7 else 241)
    ref_m = oracle.qsgd_elias_quarter_marks(codes, n, d, s)
    words, offsets, marks = _encode_marked(codes, norms, n, d, s)
    np.testing.assert_array_equal(host_u32(words[:ref_w.size]), ref_w)
    np.testing.assert_array_equal(_host_u16(marks), ref_m)
    del ref_w, ref_m
    cb = gc.qsgd_code_bytes(n, s)
    dc = torch.empty(cb, dtype=torch.uint8, device=DEV)
    dn = torch.empty(nb, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    gc.qsgd_elias_decode(words, offsets, n, d, s, dc, dn, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    np.testing.assert_array_equal(dc.cpu().numpy(), codes)
    np.testing.assert_array_equal(host_f32(dn).view(np.uint32), norms.view(np.uint32))
    qc, qn, qst = _decode_quarters(words, offsets, marks, n, d, s)
    assert qst == 0
    np.testing.assert_array_equal(qc, codes)
    np.testing.assert_array_equal(qn.view(np.uint32), norms.view(np.uint32))


def test_empty_input():
    """n = 0: the marked encoder writes only offsets[0] = 0 and a clean
    status word; the quarter decoder touches nothing."""
    offsets = torch.full((4,), 7, dtype=torch.int32, device=DEV)
    words = torch.zeros(4, dtype=torch.int32, device=DEV)
    marks = torch.full((8,), 5, dtype=torch.int16, device=DEV)
    codes = torch.full((16,), 9, dtype=torch.uint8, device=DEV)
    norms = torch.zeros(4, device=DEV)
    ws = torch.full((64,), 0xA5, dtype=torch.uint8, device=DEV)
    gc.qsgd_elias_encode_marked(codes, norms, 0, 512, 7, words, offsets, marks, ws)
    gc.qsgd_elias_decode_quarters(words, offsets, marks, 0, 512, 7, codes, norms)
    torch.cuda.synchronize()
    assert host_u32(offsets).tolist() == [0, 7, 7, 7]
    assert marks.cpu().tolist() == [5] * 8 and codes.cpu().tolist() == [9] * 16
    assert gc.qsgd_elias_encode_status(ws) == gc.GC_OK
