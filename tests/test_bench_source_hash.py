"""The hash that ties a committed ncu capture to its kernel source
(bench.source_sha): comments and layout do not change it, code does, and
comment markers inside string or character literals are code."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402

SRC = '''// header comment
__global__ void k(float* x) {   /* block
   comment */
    const char* s = "a // b /* c */";
    char q = '"';
    x[0] = 1.0f;  // trailing
}
'''


def test_comments_and_layout_do_not_count():
    edited = SRC.replace("// header comment", "// another header\n\n// two lines").replace(
        "/* block\n   comment */", "/* shorter */").replace("    x[0]", "\t\tx[0]")
    assert bench.code_only(edited) == bench.code_only(SRC)


def test_code_changes_count():
    for old, new in (("1.0f", "2.0f"), ("x[0]", "x[1]"), ('"a // b /* c */"', '"a // b"'), ("'\"'", "'x'")):
        assert bench.code_only(SRC.replace(old, new)) != bench.code_only(SRC), (old, new)


def test_literals_keep_their_comment_markers():
    out = bench.code_only(SRC)
    assert '"a // b /* c */"' in out
    assert "trailing" not in out and "header" not in out and "block" not in out


def test_every_kernel_source_hashes():
    for name in ("twobit.cu", "qsgd.cu", "saps.cu", "elias.cu"):
        rel = os.path.join("gradient_compression_sgd_gc_gb300", "csrc", name)
        h = bench.source_sha(rel)
        assert len(h) == 16 and int(h, 16) >= 0
