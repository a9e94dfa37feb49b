"""The C ABI without a GPU: the library builds and loads, exports every entry
point the header declares, and its host-side logic (argument validation,
status strings, round seeds, the random perfect matching) behaves as
documented.  No kernel is launched here: every call below is rejected by host
validation before any CUDA call, or is host-only."""
import ctypes
import os
import re

import pytest

import gradient_compression_sgd_gc_gb300 as gc
import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = sorted(os.path.join(ROOT, "include", h) for h in os.listdir(os.path.join(ROOT, "include"))
                 if h.endswith(".h"))


def _declared_functions():
    names = []
    for header in HEADERS:
        with open(header) as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^GC_API\s+[a-z0-9_ ]+?\**\s*([a-z_][a-z0-9_]*)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_entry_points():
    names = _declared_functions()
    assert len(HEADERS) >= 2 and "gc_testing_saps_mask_compact_withhold" in names
    for required in ("gc_2bit_quantize", "gc_2bit_dequant_sum_update", "qsgd_quantize",
                     "qsgd_dequant_sum", "saps_mask_compact", "saps_peer_average",
                     "gc_compensated_sum_update", "easgd_step", "saps_matching",
                     "saps_round_seed", "saps_workspace_bytes", "gc_status_string"):
        assert required in names


def test_library_exports_every_declared_symbol():
    lib = gc.load()
    for name in _declared_functions():
        assert hasattr(lib, name), name
    assert gc.gc_version() >> 16 == 1


def test_library_is_the_in_tree_build():
    assert os.path.realpath(gc.library_path()).startswith(os.path.realpath(ROOT))
    assert os.path.exists(gc.library_path())


def test_status_strings():
    for code in (0, -1, -2, -3, -4, -5, -6):
        s = gc.gc_status_string(code)
        assert s and (code != 0 or s == "GC_OK")
    assert gc.gc_status_string(12345) == "unknown status"


FAKE = 0x10000          # an aligned non-null address; never dereferenced below
MISALIGNED = 0x10004


def _call(name, *args):
    return getattr(gc.load(), name)(*args)


def test_quantize_validation():
    f = "gc_2bit_quantize"
    assert _call(f, FAKE, 0, FAKE, FAKE, -1, 0.5, None) == gc.GC_ERR_INVALID
    assert _call(f, FAKE, 0, FAKE, FAKE, 10, 0.0, None) == gc.GC_ERR_INVALID
    assert _call(f, FAKE, 0, FAKE, FAKE, 10, -1.0, None) == gc.GC_ERR_INVALID
    assert _call(f, FAKE, 0, FAKE, FAKE, 10, float("inf"), None) == gc.GC_ERR_INVALID
    assert _call(f, FAKE, 0, FAKE, FAKE, 10, float("nan"), None) == gc.GC_ERR_INVALID
    assert _call(f, FAKE, 7, FAKE, FAKE, 10, 0.5, None) == gc.GC_ERR_INVALID
    assert _call(f, None, 0, FAKE, FAKE, 10, 0.5, None) == gc.GC_ERR_INVALID
    assert _call(f, MISALIGNED, 0, FAKE, FAKE, 10, 0.5, None) == gc.GC_ERR_ALIGN
    assert _call(f, FAKE, 0, MISALIGNED, FAKE, 10, 0.5, None) == gc.GC_ERR_ALIGN
    assert _call(f, None, 0, None, None, 0, 0.5, None) == gc.GC_OK     # n == 0: no-op


def _ptrs(*addrs):
    return (ctypes.c_void_p * len(addrs))(*addrs)


def test_dequant_validation():
    f = "gc_2bit_dequant_sum_update"
    codes = _ptrs(FAKE, FAKE)
    assert _call(f, codes, 0, 10, 0.5, 0, 0.0, 0.0, None, None, FAKE, None) == gc.GC_ERR_INVALID
    assert _call(f, codes, 65, 10, 0.5, 0, 0.0, 0.0, None, None, FAKE, None) == gc.GC_ERR_INVALID
    assert _call(f, codes, 2, 10, 0.5, 3, 0.0, 0.0, None, None, FAKE, None) == gc.GC_ERR_INVALID
    assert _call(f, codes, 2, 10, 0.5, 0, 0.0, 0.0, None, None, None, None) == gc.GC_ERR_INVALID
    assert _call(f, codes, 2, 10, 0.5, 1, 0.1, 0.0, None, None, None, None) == gc.GC_ERR_INVALID
    assert _call(f, codes, 2, 10, 0.5, 2, 0.1, 0.9, None, FAKE, None, None) == gc.GC_ERR_INVALID
    assert _call(f, _ptrs(FAKE, MISALIGNED), 2, 10, 0.5, 0, 0.0, 0.0, None, None, FAKE,
                 None) == gc.GC_ERR_ALIGN
    assert _call(f, _ptrs(FAKE, 0), 2, 10, 0.5, 0, 0.0, 0.0, None, None, FAKE,
                 None) == gc.GC_ERR_INVALID


def test_qsgd_validation():
    f = "qsgd_quantize"
    assert _call(f, FAKE, 100, 500, 7, 1, 0, FAKE, FAKE, None) == gc.GC_ERR_INVALID   # bucket
    assert _call(f, FAKE, 100, 512, 0, 1, 0, FAKE, FAKE, None) == gc.GC_ERR_INVALID   # s
    assert _call(f, FAKE, 100, 512, 128, 1, 0, FAKE, FAKE, None) == gc.GC_ERR_INVALID
    assert _call(f, FAKE, 100, 512, 7, 1, -1, FAKE, FAKE, None) == gc.GC_ERR_INVALID  # worker
    assert _call(f, MISALIGNED, 100, 512, 7, 1, 0, FAKE, FAKE, None) == gc.GC_ERR_ALIGN
    g = "qsgd_dequant_sum"
    assert _call(g, _ptrs(FAKE), _ptrs(FAKE), 1, 100, 512, 7, float("nan"), FAKE,
                 None) == gc.GC_ERR_INVALID
    assert _call(g, _ptrs(FAKE), _ptrs(FAKE), 0, 100, 512, 7, 1.0, FAKE, None) == gc.GC_ERR_INVALID


def test_elias_sizes_and_validation():
    assert gc.qsgd_elias_max_words(1024, 512, 7) == 2 * (1 + 512 * 8 // 32)
    assert gc.qsgd_elias_max_words(1024 + 3, 512, 127) == 2 * (1 + 512 * 15 // 32) + 1 + 2
    assert gc.qsgd_elias_max_words(100, 500, 7) == 0
    assert gc.qsgd_elias_workspace_bytes(100, 500) == 0
    ws = gc.qsgd_elias_workspace_bytes(10_000, 512)
    assert ws >= 4 * 20 and ws % 16 == 0
    f = "qsgd_elias_encode"
    cap = gc.qsgd_elias_max_words(10_000, 512, 7)
    assert _call(f, FAKE, FAKE, 10_000, 500, 7, FAKE, cap, FAKE, FAKE, ws, None) == gc.GC_ERR_INVALID
    assert _call(f, FAKE, FAKE, 10_000, 512, 0, FAKE, cap, FAKE, FAKE, ws, None) == gc.GC_ERR_INVALID
    assert _call(f, FAKE, FAKE, 10_000, 512, 7, FAKE, cap - 1, FAKE, FAKE, ws, None) == gc.GC_ERR_CAPACITY
    assert _call(f, FAKE, FAKE, 10_000, 512, 7, FAKE, cap, FAKE, FAKE, ws - 1, None) == gc.GC_ERR_INVALID
    assert _call(f, FAKE, FAKE, 10_000, 512, 7, FAKE, cap, None, FAKE, ws, None) == gc.GC_ERR_INVALID
    assert _call(f, FAKE, FAKE, 10_000, 512, 7, MISALIGNED, cap, FAKE, FAKE, ws, None) == gc.GC_ERR_ALIGN
    # offsets must stay 32-bit: a stream bound above 2^32 - 1 words is refused
    big = 1 << 34
    assert _call(f, FAKE, FAKE, big, 512, 127, FAKE, 1 << 40, FAKE, FAKE, 1 << 40, None) == gc.GC_ERR_INVALID
    g = "qsgd_elias_decode"
    assert _call(g, FAKE, FAKE, 10_000, 512, 128, FAKE, FAKE, None, None) == gc.GC_ERR_INVALID
    assert _call(g, None, FAKE, 10_000, 512, 7, FAKE, FAKE, None, None) == gc.GC_ERR_INVALID
    assert _call(g, FAKE, FAKE, 10_000, 512, 7, FAKE, MISALIGNED, None, None) == gc.GC_ERR_ALIGN
    assert _call(g, FAKE, FAKE, 10_000, 512, 7, FAKE, FAKE, MISALIGNED + 1, None) == gc.GC_ERR_ALIGN
    assert _call(g, None, None, 0, 512, 7, None, None, None, None) == gc.GC_OK
    h = "qsgd_elias_decode_batched"
    two = _ptrs(FAKE, FAKE)
    assert _call(h, two, two, 0, 10_000, 512, 7, two, two, None, None) == gc.GC_ERR_INVALID       # W = 0
    assert _call(h, two, two, 65, 10_000, 512, 7, two, two, None, None) == gc.GC_ERR_INVALID      # W > 64
    assert _call(h, two, _ptrs(FAKE, None), 2, 10_000, 512, 7, two, two, None, None) == gc.GC_ERR_INVALID
    assert _call(h, two, two, 2, 10_000, 512, 7, _ptrs(FAKE, MISALIGNED), two, None, None) == gc.GC_ERR_ALIGN
    assert _call(h, two, two, 2, 10_000, 500, 7, two, two, None, None) == gc.GC_ERR_INVALID
    assert _call(h, None, None, 2, 0, 512, 7, None, None, None, None) == gc.GC_OK
    m = "qsgd_elias_encode_marked"
    assert _call(m, FAKE, FAKE, 10_000, 512, 7, FAKE, cap, FAKE, None, FAKE, ws, None) == gc.GC_ERR_INVALID
    assert _call(m, FAKE, FAKE, 10_000, 512, 7, FAKE, cap, FAKE, MISALIGNED, FAKE, ws, None) == gc.GC_ERR_ALIGN
    assert _call(m, FAKE, FAKE, 10_000, 500, 7, FAKE, cap, FAKE, FAKE, FAKE, ws, None) == gc.GC_ERR_INVALID
    assert _call(m, FAKE, FAKE, 10_000, 512, 7, FAKE, cap - 1, FAKE, FAKE, FAKE, ws, None) == gc.GC_ERR_CAPACITY
    t = "gc_testing_qsgd_elias_encode_withhold"
    assert _call(t, FAKE, FAKE, 10_000, 512, 7, FAKE, cap, FAKE, FAKE, ws, 3, 0, None) == gc.GC_ERR_INVALID
    assert _call(t, FAKE, FAKE, 10_000, 512, 7, FAKE, cap, FAKE, FAKE, ws, 3, 2_000_000_000, None) == gc.GC_ERR_INVALID
    assert _call(t, FAKE, FAKE, 10_000, 512, 7, FAKE, cap, FAKE, FAKE, ws, -1, 1000, None) == gc.GC_ERR_INVALID
    assert _call(t, FAKE, FAKE, 10_000, 512, 7, FAKE, cap - 1, FAKE, FAKE, ws, 3, 1000, None) == gc.GC_ERR_CAPACITY
    q = "qsgd_elias_decode_quarters"
    assert _call(q, FAKE, FAKE, None, 10_000, 512, 7, FAKE, FAKE, None, None) == gc.GC_ERR_INVALID
    assert _call(q, FAKE, FAKE, MISALIGNED, 10_000, 512, 7, FAKE, FAKE, None, None) == gc.GC_ERR_ALIGN
    assert _call(q, FAKE, FAKE, FAKE, 10_000, 512, 0, FAKE, FAKE, None, None) == gc.GC_ERR_INVALID
    assert _call(q, FAKE, FAKE, FAKE, 10_000, 512, 7, FAKE, FAKE, MISALIGNED + 1, None) == gc.GC_ERR_ALIGN
    assert _call(q, None, None, None, 0, 512, 7, None, None, None, None) == gc.GC_OK


def test_l2_fetch_granularity_validation():
    assert _call("gc_l2_fetch_granularity", 129, None) == gc.GC_ERR_INVALID
    assert _call("gc_l2_fetch_granularity", 1 << 40, None) == gc.GC_ERR_INVALID


def test_saps_validation():
    f = "saps_mask_compact"
    ws = gc.saps_workspace_bytes(1000)
    models, vals = _ptrs(FAKE), _ptrs(FAKE)
    ok = (1000, 0.01, 5, models, 1, FAKE, vals, 100, FAKE, FAKE, ws, FAKE, None)

    def with_(i, v):
        a = list(ok)
        a[i] = v
        return _call(f, *a)
    assert with_(1, 0.0) == gc.GC_ERR_INVALID
    assert with_(1, 1.5) == gc.GC_ERR_INVALID
    assert with_(0, 1 << 33) == gc.GC_ERR_INVALID          # indices are uint32
    assert with_(10, ws - 1) == gc.GC_ERR_INVALID           # workspace too small
    assert with_(11, None) == gc.GC_ERR_INVALID             # d_status
    assert with_(9, MISALIGNED) == gc.GC_ERR_ALIGN          # workspace
    g = "saps_peer_average"
    pairs = (ctypes.c_int * 4)(0, 1, 2, 2)                  # not a permutation
    assert _call(g, _ptrs(FAKE, FAKE, FAKE, FAKE), _ptrs(FAKE, FAKE, FAKE, FAKE), FAKE, FAKE,
                 pairs, 4, 10, None) == gc.GC_ERR_INVALID
    assert _call(g, _ptrs(FAKE), _ptrs(FAKE), FAKE, FAKE, (ctypes.c_int * 1)(0), 1, 10,
                 None) == gc.GC_ERR_INVALID
    h = "easgd_step"
    assert _call(h, _ptrs(FAKE), 1, 10, float("inf"), 0.9, FAKE, None) == gc.GC_ERR_INVALID
    assert _call(h, _ptrs(FAKE), 1, 10, 0.9, 0.9, MISALIGNED, None) == gc.GC_ERR_ALIGN


def test_workspace_size_grows_with_n():
    assert gc.saps_workspace_bytes(0) >= 16
    assert gc.saps_workspace_bytes(25_557_032) > gc.saps_workspace_bytes(1000)


@pytest.mark.parametrize("W", [2, 4, 16, 64])
def test_matching_agrees_with_oracle(W):
    for t in range(20):
        seed_t = gc.saps_round_seed(5, t)
        assert seed_t == oracle.round_seed(5, t)
        assert gc.saps_matching(seed_t, W) == oracle.saps_matching(seed_t, W).tolist()


def test_matching_rejects_bad_w():
    for W in (0, 1, 3, 66):
        with pytest.raises(gc.GcError):
            gc.saps_matching(1, W)


def test_batched_quantize_validation():
    f = "gc_2bit_quantize_batched"
    two = (ctypes.c_int64 * 2)(10, 20)
    p2 = _ptrs(FAKE, FAKE)
    assert _call(f, p2, 0, p2, p2, two, 0, 0.5, None) == gc.GC_ERR_INVALID           # B = 0
    assert _call(f, p2, 0, p2, p2, two, 65, 0.5, None) == gc.GC_ERR_INVALID          # B > 64
    assert _call(f, p2, 0, p2, p2, two, 2, 0.0, None) == gc.GC_ERR_INVALID           # threshold
    assert _call(f, p2, 0, p2, p2, (ctypes.c_int64 * 2)(10, -1), 2, 0.5, None) == gc.GC_ERR_INVALID
    assert _call(f, _ptrs(FAKE, MISALIGNED), 0, p2, p2, two, 2, 0.5, None) == gc.GC_ERR_ALIGN
    assert _call(f, _ptrs(FAKE, 0), 0, p2, p2, two, 2, 0.5, None) == gc.GC_ERR_INVALID
    # every buffer empty: a no-op that never touches the (null) pointers
    assert _call(f, _ptrs(0, 0), 0, _ptrs(0, 0), _ptrs(0, 0), (ctypes.c_int64 * 2)(0, 0), 2, 0.5,
                 None) == gc.GC_OK


def test_fused_average_easgd_validation():
    f = "saps_average_easgd_step"
    ws = gc.saps_workspace_bytes(1000)
    p4 = _ptrs(FAKE, FAKE, FAKE, FAKE)
    good = (ctypes.c_int * 4)(2, 0, 3, 1)
    ok = [p4, p4, FAKE, good, 4, 1000, 100, 0.9, 0.9, FAKE, FAKE, ws, None]

    def with_(i, v):
        a = list(ok)
        a[i] = v
        return _call(f, *a)
    assert with_(3, (ctypes.c_int * 4)(0, 0, 1, 2)) == gc.GC_ERR_INVALID    # not a permutation
    assert with_(4, 3) == gc.GC_ERR_INVALID                                 # odd W
    assert with_(11, ws - 1) == gc.GC_ERR_INVALID                           # workspace too small
    assert with_(9, MISALIGNED) == gc.GC_ERR_ALIGN                          # center
    assert with_(7, float("nan")) == gc.GC_ERR_INVALID
    assert with_(5, 0) == gc.GC_OK                                          # n == 0 no-op


def test_testing_hook_validates_its_wait_bound():
    f = "gc_testing_saps_mask_compact_withhold"
    ws = gc.saps_workspace_bytes(1000)
    p1 = _ptrs(FAKE)
    for bad in (0, 2_000_000_000):
        assert _call(f, 1000, 0.01, 5, p1, 1, FAKE, p1, 100, FAKE, FAKE, ws, FAKE, 3, bad,
                     None) == gc.GC_ERR_INVALID


def test_one_pass_entry_validation():
    f = "qsgd_step"
    g3 = _ptrs(FAKE, FAKE, FAKE)
    assert _call(f, g3, 3, 1000, 500, 7, 1, 0, g3, g3, 1.0, FAKE, None) == gc.GC_ERR_INVALID    # bucket
    assert _call(f, g3, 3, 1000, 512, 0, 1, 0, g3, g3, 1.0, FAKE, None) == gc.GC_ERR_INVALID    # s
    assert _call(f, g3, 3, 1000, 512, 7, 1, 2, g3, g3, 1.0, FAKE, None) == gc.GC_ERR_INVALID    # maxnorm flag
    assert _call(f, g3, 0, 1000, 512, 7, 1, 0, g3, g3, 1.0, FAKE, None) == gc.GC_ERR_INVALID    # W
    assert _call(f, g3, 3, 1000, 512, 7, 1, 0, g3, g3, float("inf"), FAKE, None) == gc.GC_ERR_INVALID
    assert _call(f, g3, 3, 1000, 512, 7, 1, 0, g3, g3, 1.0, MISALIGNED, None) == gc.GC_ERR_ALIGN
    assert _call(f, _ptrs(FAKE, MISALIGNED, FAKE), 3, 1000, 512, 7, 1, 0, g3, g3, 1.0, FAKE, None) == gc.GC_ERR_ALIGN
    assert _call(f, g3, 3, 0, 512, 7, 1, 0, g3, g3, 1.0, FAKE, None) == gc.GC_OK               # n == 0
    r = "saps_round"
    ws = gc.saps_workspace_bytes(1000)
    m4, v4 = _ptrs(FAKE, FAKE, FAKE, FAKE), _ptrs(FAKE, FAKE, FAKE, FAKE)
    pairs = (ctypes.c_int * 4)(0, 1, 2, 3)
    bad_pairs = (ctypes.c_int * 4)(0, 0, 2, 3)
    ok_args = dict(n=1000, p=0.01, seed=1, models=m4, W=4, pairs=pairs, alpha=0.9, beta=0.9, center=FAKE,
                   idx=FAKE, vals=v4, cap=1000, cnt=FAKE, ws=FAKE, wsb=ws, st=FAKE)

    def call(**kw):
        a = dict(ok_args, **kw)
        return _call(r, a["n"], a["p"], a["seed"], a["models"], a["W"], a["pairs"], a["alpha"], a["beta"],
                     a["center"], a["idx"], a["vals"], a["cap"], a["cnt"], a["ws"], a["wsb"], a["st"], None)

    assert call(W=3) == gc.GC_ERR_INVALID
    assert call(pairs=bad_pairs) == gc.GC_ERR_INVALID
    assert call(p=0.0) == gc.GC_ERR_INVALID
    assert call(p=1.5) == gc.GC_ERR_INVALID
    assert call(alpha=float("nan")) == gc.GC_ERR_INVALID
    assert call(wsb=ws - 1) == gc.GC_ERR_INVALID
    assert call(st=None) == gc.GC_ERR_INVALID
    assert call(n=1 << 33) == gc.GC_ERR_INVALID
    assert call(center=MISALIGNED) == gc.GC_ERR_ALIGN
    assert call(models=_ptrs(FAKE, MISALIGNED, FAKE, FAKE)) == gc.GC_ERR_ALIGN



def test_step_and_multistep_validation():
    """gc_2bit_step takes fp32 and bf16; gc_2bit_step_local needs its local
    weight pointers and the weights; gc_2bit_quantize_steps checks S, the
    residual and every step's buffers.  Host validation only (no launch)."""
    p2 = _ptrs(FAKE, FAKE)
    f = "gc_2bit_step"
    #      grads dtype res codes W  n     t    kind lr   alpha center weights out  stream
    assert _call(f, p2, 2, p2, p2, 2, 1000, 0.5, 1, 0.1, 0.0, None, FAKE, None, None) == gc.GC_ERR_INVALID   # dtype
    assert _call(f, p2, 1, p2, p2, 2, 1000, 0.5, 1, 0.1, 0.0, None, None, None, None) == gc.GC_ERR_INVALID   # weights
    assert _call(f, p2, 1, p2, p2, 2, 0, 0.5, 1, 0.1, 0.0, None, FAKE, None, None) == gc.GC_OK            # bf16, n == 0
    g = "gc_2bit_step_local"
    assert _call(g, p2, 1, p2, p2, None, 0.1, 2, 1000, 0.5, 1, 0.1, 0.0, None, FAKE, None, None) == gc.GC_ERR_INVALID
    assert _call(g, p2, 1, p2, p2, _ptrs(FAKE, 0), 0.1, 2, 1000, 0.5, 1, 0.1, 0.0, None, FAKE, None,
                 None) == gc.GC_ERR_INVALID
    assert _call(g, p2, 1, p2, p2, _ptrs(FAKE, MISALIGNED), 0.1, 2, 1000, 0.5, 1, 0.1, 0.0, None, FAKE, None,
                 None) == gc.GC_ERR_ALIGN
    assert _call(g, p2, 1, p2, p2, p2, float("nan"), 2, 1000, 0.5, 1, 0.1, 0.0, None, FAKE, None,
                 None) == gc.GC_ERR_INVALID
    # kind NONE with local weights still needs the weights (read for W_loc)
    assert _call(g, p2, 1, p2, p2, p2, 0.1, 2, 1000, 0.5, 0, 0.0, 0.0, None, None, FAKE, None) == gc.GC_ERR_INVALID
    h = "gc_2bit_quantize_steps"
    #      grads dtype residual codes out S  n     t
    assert _call(h, p2, 0, FAKE, p2, None, 0, 1000, 0.5, None) == gc.GC_ERR_INVALID        # S
    assert _call(h, p2, 0, FAKE, p2, None, 65, 1000, 0.5, None) == gc.GC_ERR_INVALID       # S > 64
    assert _call(h, p2, 0, None, p2, None, 2, 1000, 0.5, None) == gc.GC_ERR_INVALID        # residual
    assert _call(h, p2, 0, MISALIGNED, p2, None, 2, 1000, 0.5, None) == gc.GC_ERR_ALIGN
    assert _call(h, p2, 0, FAKE, _ptrs(FAKE, 0), None, 2, 1000, 0.5, None) == gc.GC_ERR_INVALID
    assert _call(h, p2, 0, FAKE, p2, _ptrs(FAKE, MISALIGNED), 2, 1000, 0.5, None) == gc.GC_ERR_ALIGN
    assert _call(h, p2, 0, FAKE, p2, None, 2, 1000, -0.5, None) == gc.GC_ERR_INVALID       # threshold
    assert _call(h, p2, 3, FAKE, p2, None, 2, 1000, 0.5, None) == gc.GC_ERR_INVALID        # dtype
    assert _call(h, p2, 0, FAKE, p2, None, 2, 0, 0.5, None) == gc.GC_OK                    # n == 0


def test_binding_wants_the_whole_matching():
    """A matching shorter than the worker list is refused on the host (a short
    list padded with zeros could still be a permutation)."""
    import torch
    models = [torch.zeros(4) for _ in range(4)]
    for call in (lambda: gc.saps_peer_average(models, models, torch.zeros(4, dtype=torch.int32),
                                              torch.zeros(1, dtype=torch.int64), [1, 2, 3]),
                 lambda: gc.saps_average_easgd_step(models, models, torch.zeros(1, dtype=torch.int64),
                                                    [1, 2, 3], 0.9, 0.9, torch.zeros(4),
                                                    torch.zeros(16, dtype=torch.uint8)),
                 lambda: gc.saps_round(4, 0.5, 1, models, [1, 2, 3], 0.9, 0.9, torch.zeros(4),
                                       torch.zeros(4, dtype=torch.int32), models,
                                       torch.zeros(1, dtype=torch.int64), torch.zeros(16, dtype=torch.uint8),
                                       torch.zeros(1, dtype=torch.int32))):
        with pytest.raises(ValueError, match="pairs must list all 4 workers"):
            call()
