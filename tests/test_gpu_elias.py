"""GPU parity of the QSGD Elias-omega codec (Knowl 2) against the oracle.

The encoder's input codes and norms come from the oracle's quantiser on the
seeded workload recipe, so the GPU stream must equal the oracle's stream word
for word (integer work: bit-exact), offsets included; the decoder must give
back the oracle decoder's codes and norms exactly.  Sizes span several CTAs of
64 buckets and a ragged last bucket; the full-size cases use the QSGD
workload (61,100,840 coordinates, buckets of 512).
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
    norms, codes = oracle.qsgd_quantize(v, bucket, s, cfg.seed, worker)
    return v, norms, codes


def _encode_gpu(codes_h, norms_h, n, bucket, s):
    nb = gc.qsgd_num_buckets(n, bucket)
    cap = gc.qsgd_elias_max_words(n, bucket, s)
    codes = torch.from_numpy(codes_h).to(DEV)
    norms = torch.from_numpy(norms_h).to(DEV)
    words = guarded(cap, torch.int32)
    offsets = guarded(nb + 1, torch.int32)
    ws = torch.empty(max(16, gc.qsgd_elias_workspace_bytes(n, bucket)), dtype=torch.uint8, device=DEV)
    ws.fill_(0xA5)                 # the workspace needs no initialisation
    gc.qsgd_elias_encode(codes, norms, n, bucket, s, words[:cap], offsets[:nb + 1], ws)
    torch.cuda.synchronize()
    check_guard(offsets, nb + 1)
    check_guard(words, cap)
    return words, offsets


def _decode_gpu(words, offsets, n, bucket, s):
    nb = gc.qsgd_num_buckets(n, bucket)
    cb = gc.qsgd_code_bytes(n, s)
    codes = guarded(cb, torch.uint8)
    codes[:cb].fill_(0xEE)       # every byte must be written
    norms = guarded(nb, torch.float32)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    gc.qsgd_elias_decode(words, offsets, n, bucket, s, codes[:cb], norms[:nb], st)
    torch.cuda.synchronize()
    check_guard(codes, cb)
    check_guard(norms, nb)
    return codes[:cb].cpu().numpy(), host_f32(norms[:nb]), int(st.item())


CASES = [
    (wl.QSGD_S7, 512 * 150 + 297, 512, 7),       # 151 buckets: 3 CTAs, ragged odd tail
    (wl.QSGD_S7, 128 * 400 + 77, 128, 7),
    (wl.QSGD_S7, 256 * 70, 256, 1),              # s = 1 (ternary)
    (wl.QSGD_S127, 512 * 130 + 1, 512, 127),
    (wl.QSGD_S127, 2048 * 70 + 1001, 2048, 127),
    (wl.QSGD_S127, 512 * 129 + 400, 512, 22),    # s = floor(sqrt(512)): the dense regime
    (wl.QSGD_S7, 1024 * 65, 1024, 5),
    (wl.QSGD_S7, 300, 512, 7),                   # one short bucket
    (wl.QSGD_S127, 1, 128, 127),
]


@pytest.mark.parametrize("cfg,n,bucket,s", CASES, ids=lambda x: getattr(x, "name", str(x)))
def test_encode_decode_parity(cfg, n, bucket, s):
    _, norms, codes = _oracle_codes(cfg, n, bucket, s)
    ref_w, ref_off = oracle.qsgd_elias_encode(codes, norms, n, bucket, s)
    words, offsets = _encode_gpu(codes, norms, n, bucket, s)
    nb = gc.qsgd_num_buckets(n, bucket)
    np.testing.assert_array_equal(host_u32(offsets[:nb + 1]), ref_off)
    total = int(ref_off[-1])
    np.testing.assert_array_equal(host_u32(words[:total]), ref_w)
    dc, dn, st = _decode_gpu(words, offsets, n, bucket, s)
    rc, rn = oracle.qsgd_elias_decode(ref_w, ref_off, n, bucket, s)
    assert st == 0
    np.testing.assert_array_equal(dc, rc)
    np.testing.assert_array_equal(dn.view(np.uint32), rn.view(np.uint32))


@pytest.mark.parametrize("cfg,n,bucket,s", [CASES[0], CASES[3], CASES[5]], ids=lambda x: getattr(x, "name", str(x)))
def test_batched_decode_equals_the_single_decodes(cfg, n, bucket, s):
    """Three workers' streams decoded in one launch: each equals the oracle's
    decode of that worker's stream; a corrupt third stream flags the shared
    status without changing the other two."""
    nb = gc.qsgd_num_buckets(n, bucket)
    cb = gc.qsgd_code_bytes(n, s)
    streams, refs = [], []
    for w in range(3):
        _, norms, codes = _oracle_codes(cfg, n, bucket, s, worker=w)
        ref_w, ref_off = oracle.qsgd_elias_encode(codes, norms, n, bucket, s)
        words, offsets = _encode_gpu(codes, norms, n, bucket, s)
        streams.append((words, offsets))
        refs.append(oracle.qsgd_elias_decode(ref_w, ref_off, n, bucket, s))
    out_c = [guarded(cb, torch.uint8) for _ in range(3)]
    out_n = [guarded(nb, torch.float32) for _ in range(3)]
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    gc.qsgd_elias_decode_batched([w for w, _ in streams], [o[:nb + 1] for _, o in streams], n, bucket, s,
                                 [c[:cb] for c in out_c], [m[:nb] for m in out_n], st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for w in range(3):
        np.testing.assert_array_equal(out_c[w][:cb].cpu().numpy(), refs[w][0])
        np.testing.assert_array_equal(host_f32(out_n[w][:nb]).view(np.uint32), refs[w][1].view(np.uint32))
        check_guard(out_c[w], cb)
        check_guard(out_n[w], nb)
    # truncate the third stream's first bucket to its norm word: corrupt
    bad_off = streams[2][1][:nb + 1].clone()
    bad_off[1] = bad_off[0] + 1
    bad_off[2:] = torch.maximum(bad_off[2:], bad_off[1])
    gc.qsgd_elias_decode_batched([w for w, _ in streams], [streams[0][1][:nb + 1], streams[1][1][:nb + 1], bad_off],
                                 n, bucket, s, [c[:cb] for c in out_c], [m[:nb] for m in out_n], st)
    torch.cuda.synchronize()
    assert int(st.item()) == gc.GC_ERR_CORRUPT
    for w in range(2):
        np.testing.assert_array_equal(out_c[w][:cb].cpu().numpy(), refs[w][0])


def test_batched_decode_of_sixty_four_streams():
    """The largest batch (GC_MAX_WORKERS streams) of short ragged streams."""
    cfg, n, bucket, s = wl.QSGD_S7, 2 * 128 + 37, 128, 7
    nb = gc.qsgd_num_buckets(n, bucket)
    cb = gc.qsgd_code_bytes(n, s)
    words, offs, refs = [], [], []
    for w in range(gc.GC_MAX_WORKERS):
        _, norms, codes = _oracle_codes(cfg, n, bucket, s, worker=w)
        ref_w, ref_off = oracle.qsgd_elias_encode(codes, norms, n, bucket, s)
        words.append(torch.from_numpy(ref_w.view(np.int32)).to(DEV))
        offs.append(torch.from_numpy(ref_off.view(np.int32)).to(DEV))
        refs.append(oracle.qsgd_elias_decode(ref_w, ref_off, n, bucket, s))
    out_c = [torch.empty(cb, dtype=torch.uint8, device=DEV) for _ in range(gc.GC_MAX_WORKERS)]
    out_n = [torch.empty(nb, device=DEV) for _ in range(gc.GC_MAX_WORKERS)]
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    gc.qsgd_elias_decode_batched(words, offs, n, bucket, s, out_c, out_n, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for w in range(gc.GC_MAX_WORKERS):
        np.testing.assert_array_equal(out_c[w].cpu().numpy(), refs[w][0])
        np.testing.assert_array_equal(host_f32(out_n[w]).view(np.uint32), refs[w][1].view(np.uint32))
    with pytest.raises(gc.GcError):
        gc.qsgd_elias_decode_batched(words + words[:1], offs + offs[:1], n, bucket, s, out_c + out_c[:1],
                                     out_n + out_n[:1], st)


def test_empty():
    offsets = torch.full((4,), 7, dtype=torch.int32, device=DEV)
    words = torch.zeros(4, dtype=torch.int32, device=DEV)
    codes = torch.zeros(16, dtype=torch.uint8, device=DEV)
    norms = torch.zeros(4, device=DEV)
    ws = torch.zeros(64, dtype=torch.uint8, device=DEV)
    gc.qsgd_elias_encode(codes, norms, 0, 512, 7, words, offsets, ws)
    gc.qsgd_elias_decode(words, offsets, 0, 512, 7, codes, norms)
    torch.cuda.synchronize()
    assert host_u32(offsets).tolist() == [0, 7, 7, 7]


@pytest.mark.parametrize("s", [7, 127])
def test_worst_case_fills_the_bound(s):
    """Every coordinate at the top level with sign -: each codeword takes the
    longest form, and the stream is exactly qsgd_elias_max_words long."""
    n, bucket = 512 * 70 + 33, 512
    nb = gc.qsgd_num_buckets(n, bucket)
    cb = gc.qsgd_code_bytes(n, s)
    top = 0x8 | s if s <= 7 else 0x80 | s
    codes = np.full(cb, (top << 4) | top if s <= 7 else top, np.uint8)
    if s <= 7 and n % 2:
        codes[-1] &= 0xF0
    norms = np.linspace(0.5, 2.0, nb).astype(np.float32)
    ref_w, ref_off = oracle.qsgd_elias_encode(codes, norms, n, bucket, s)
    assert ref_w.size == gc.qsgd_elias_max_words(n, bucket, s)
    words, offsets = _encode_gpu(codes, norms, n, bucket, s)
    np.testing.assert_array_equal(host_u32(offsets[:nb + 1]), ref_off)
    np.testing.assert_array_equal(host_u32(words[:ref_w.size]), ref_w)
    dc, dn, st = _decode_gpu(words, offsets, n, bucket, s)
    assert st == 0
    np.testing.assert_array_equal(dc, codes)


def test_all_zero_buckets():
    """Norm 0: level 0 everywhere, one bit per coordinate; negative zeros and
    negative values in a zero-norm bucket send no sign."""
    n, bucket, s = 512 * 66, 512, 7
    v = np.zeros(n, np.float32)
    v[::3] = -0.0
    v[512 * 10:512 * 11] = np.linspace(-1, 1, 512, dtype=np.float32)
    norms, codes = oracle.qsgd_quantize(v, bucket, s, seed=1, worker=0)
    ref_w, ref_off = oracle.qsgd_elias_encode(codes, norms, n, bucket, s)
    words, offsets = _encode_gpu(codes, norms, n, bucket, s)
    np.testing.assert_array_equal(host_u32(offsets[:67]), ref_off)
    np.testing.assert_array_equal(host_u32(words[:ref_w.size]), ref_w)
    assert int(ref_off[1]) == 1 + 512 // 32


def test_roundtrip_through_dequant_sum():
    """quantise -> encode -> decode -> dequant-sum on the GPU equals quantise ->
    dequant-sum: the codec is lossless for everything the decoder reads."""
    cfg, n, bucket = wl.QSGD_S7, 512 * 300 + 5, 512
    for s in (7, 127):
        W = 3
        nb, cb = gc.qsgd_num_buckets(n, bucket), gc.qsgd_code_bytes(n, s)
        cap = gc.qsgd_elias_max_words(n, bucket, s)
        ws = torch.empty(gc.qsgd_elias_workspace_bytes(n, bucket), dtype=torch.uint8, device=DEV)
        codes, norms, dcodes, dnorms = [], [], [], []
        for w in range(W):
            v = wl.qsgd_grad(wl.scaled(cfg, n), w, device=DEV)
            c = torch.empty(cb, dtype=torch.uint8, device=DEV)
            nr = torch.empty(nb, device=DEV)
            gc.qsgd_quantize(v, bucket, s, cfg.seed, w, nr, c)
            words = torch.empty(cap, dtype=torch.int32, device=DEV)
            offs = torch.empty(nb + 1, dtype=torch.int32, device=DEV)
            gc.qsgd_elias_encode(c, nr, n, bucket, s, words, offs, ws)
            dc = torch.empty(cb, dtype=torch.uint8, device=DEV)
            dn = torch.empty(nb, device=DEV)
            gc.qsgd_elias_decode(words, offs, n, bucket, s, dc, dn)
            codes.append(c), norms.append(nr), dcodes.append(dc), dnorms.append(dn)
        a = torch.empty(n, device=DEV)
        b = torch.empty(n, device=DEV)
        gc.qsgd_dequant_sum(codes, norms, n, bucket, s, 1.0 / W, a)
        gc.qsgd_dequant_sum(dcodes, dnorms, n, bucket, s, 1.0 / W, b)
        torch.cuda.synchronize()
        assert bool((a == b).all())
        for w in range(W):
            assert torch.equal(norms[w], dnorms[w])


def test_corrupt_streams_are_reported():
    """Streams that cannot be the encoder's output: the decoder stays inside
    each bucket's words and reports GC_ERR_CORRUPT."""
    cfg, n, bucket, s = wl.QSGD_S127, 512 * 8, 512, 127
    _, norms, codes = _oracle_codes(cfg, n, bucket, s)
    ref_w, ref_off = oracle.qsgd_elias_encode(codes, norms, n, bucket, s)
    words = torch.from_numpy(ref_w.view(np.int32)).to(DEV)
    # (a) bucket 3 cut to its norm word alone
    # (bucket 4 then starts inside bucket 3's codewords; every read stays
    # below offsets[nbuckets])
    trunc_off = ref_off.copy()
    trunc_off[4] = ref_off[3] + 1
    _, _, st = _decode_gpu(words, torch.from_numpy(trunc_off.view(np.int32)).to(DEV),
                           n, bucket, s)
    assert st == gc.GC_ERR_CORRUPT
    # (b) levels above s: an s = 127 stream decoded as s = 22
    offsets = torch.from_numpy(ref_off.view(np.int32)).to(DEV)
    assert int((codes & 127).max()) > 22
    _, _, st = _decode_gpu(words, offsets, n, bucket, 22)
    assert st == gc.GC_ERR_CORRUPT
    # the untouched stream decodes cleanly
    _, _, st = _decode_gpu(words, offsets, n, bucket, s)
    assert st == 0


def _levels_signs(codes, n, s):
    """Per-coordinate (level, sign) of a code array in qsgd_quantize's layout."""
    if s <= 7:
        c = np.empty(n, dtype=np.uint8)
        c[0::2] = codes[:(n + 1) // 2] >> 4
        c[1::2] = codes[:n // 2] & 15
        return c & 7, c >> 3
    return codes[:n] & 127, codes[:n] >> 7


def _pack(level, sign, s):
    level = level.astype(np.uint8)
    sign = sign.astype(np.uint8)
    n = level.size
    if s <= 7:
        c = (sign << 3) | level
        out = (c[0::2] << 4).astype(np.uint8)
        out[:n // 2] |= c[1::2]
        return out
    return (sign << 7) | level


@pytest.mark.parametrize("cfg,n,bucket,s,s_dec", [
    (wl.QSGD_S127, 512 * 40 + 77, 512, 127, 22),
    (wl.QSGD_S127, 512 * 40 + 77, 512, 127, 7),    # 8-bit stream into 4-bit codes
    (wl.QSGD_S127, 256 * 50 + 3, 256, 127, 1),
    (wl.QSGD_S7, 512 * 40 + 77, 512, 7, 3),
    (wl.QSGD_S7, 128 * 90 + 1, 128, 7, 1),
], ids=lambda x: getattr(x, "name", str(x)))
def test_levels_above_s_are_clamped_in_step(cfg, n, bucket, s, s_dec):
    """A stream decoded with a smaller s: every level above it is written as
    s (sign kept), the status says GC_ERR_CORRUPT, and every other code is
    the oracle's -- the decoder stays in step with the codewords.  The
    expected codes are the oracle decoder's, clamped."""
    _, norms, codes = _oracle_codes(cfg, n, bucket, s)
    ref_w, ref_off = oracle.qsgd_elias_encode(codes, norms, n, bucket, s)
    ref_codes, ref_norms = oracle.qsgd_elias_decode(ref_w, ref_off, n, bucket, s)
    level, sign = _levels_signs(ref_codes, n, s)
    assert int(level.max()) > s_dec
    want = _pack(np.minimum(level, s_dec), sign, s_dec)
    words = torch.from_numpy(ref_w.view(np.int32)).to(DEV)
    offsets = torch.from_numpy(ref_off.view(np.int32)).to(DEV)
    dc, dn, st = _decode_gpu(words, offsets, n, bucket, s_dec)
    assert st == gc.GC_ERR_CORRUPT
    np.testing.assert_array_equal(dn.view(np.uint32), ref_norms.view(np.uint32))
    np.testing.assert_array_equal(dc, want)


@pytest.mark.parametrize("cfg,n,bucket,s,most", [
    (wl.QSGD_S7, 512 * 600 + 41, 512, 7, 40),      # 3 CTAs of 256 buckets
    (wl.QSGD_S127, 512 * 600 + 41, 512, 127, 40),
    (wl.QSGD_S127, 128 * 1500 + 9, 128, 127, 300),  # CTAs whose words outgrow the shared copy
], ids=lambda x: getattr(x, "name", str(x)))
def test_words_after_a_bucket_are_ignored(cfg, n, bucket, s, most):
    """Buckets followed by 0..most random words (offsets still mark each
    bucket's first word): the decoder reads only what the codewords need, so
    codes, norms and status are those of the packed stream -- whichever
    buckets of a CTA its shared-memory copy holds."""
    _, norms, codes = _oracle_codes(cfg, n, bucket, s)
    ref_w, ref_off = oracle.qsgd_elias_encode(codes, norms, n, bucket, s)
    ref_codes, ref_norms = oracle.qsgd_elias_decode(ref_w, ref_off, n, bucket, s)
    rng = np.random.default_rng(11)
    nb = ref_off.size - 1
    pad = rng.integers(0, most + 1, size=nb)
    parts, offs, pos = [], [0], 0
    for b in range(nb):
        body = ref_w[ref_off[b]:ref_off[b + 1]]
        junk = rng.integers(0, 2**32, size=int(pad[b]), dtype=np.uint64).astype(np.uint32)
        parts += [body, junk]
        pos += body.size + junk.size
        offs.append(pos)
    words_h = np.concatenate(parts)
    off_h = np.asarray(offs, dtype=np.uint32)
    dc, dn, st = _decode_gpu(torch.from_numpy(words_h.view(np.int32)).to(DEV),
                             torch.from_numpy(off_h.view(np.int32)).to(DEV), n, bucket, s)
    assert st == 0
    np.testing.assert_array_equal(dn.view(np.uint32), ref_norms.view(np.uint32))
    np.testing.assert_array_equal(dc, ref_codes)


@pytest.mark.parametrize("cfg", [wl.QSGD_S7, wl.QSGD_S127], ids=lambda c: c.name)
def test_full_size_stream_bit_exact(cfg):
    """The QSGD workload at full size (61,100,840 coordinates, 119,338
    buckets, last 296): the whole GPU stream equals the oracle's, and the
    GPU decoder returns the oracle decoder's codes."""
    n, d, s = cfg.n, cfg.bucket, cfg.s
    v = wl.qsgd_grad(cfg, 1, device="cpu").numpy()
    norms, codes = oracle.qsgd_quantize(v, d, s, cfg.seed, 1)
    del v
    ref_w, ref_off = oracle.qsgd_elias_encode(codes, norms, n, d, s)
    words, offsets = _encode_gpu(codes, norms, n, d, s)
    nb = gc.qsgd_num_buckets(n, d)
    np.testing.assert_array_equal(host_u32(offsets[:nb + 1]), ref_off)
    np.testing.assert_array_equal(host_u32(words[:ref_w.size]), ref_w)
    dc, dn, st = _decode_gpu(words, offsets, n, d, s)
    rc, rn = oracle.qsgd_elias_decode(ref_w, ref_off, n, d, s)
    assert st == 0
    np.testing.assert_array_equal(dc, rc)
    np.testing.assert_array_equal(dn.view(np.uint32), rn.view(np.uint32))
    print(f"{cfg.name}: {32 * ref_w.size / n:.3f} bits/coordinate, "
          f"{32 * (ref_w.size + nb + 1) / n:.3f} with offsets")
