"""bench.py reads a kernel's DRAM traffic from its committed ncu summary only
while the summary's recorded source digest matches the kernel code: comments
and whitespace do not count, any change to the code does."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402

CODE = """// header comment
#include "x.cuh"
/* block
   comment */
__global__ void k(int *p) {  // trailing comment
    p[0] = 1;
}
"""


def digest_of(tmp_path, text, name="k.cu"):
    (tmp_path / name).write_text(text)
    return bench.source_digest(name, src_dir=str(tmp_path))


def test_comments_and_whitespace_do_not_change_the_digest(tmp_path):
    a = digest_of(tmp_path, CODE)
    b = digest_of(tmp_path, "// another header\n" + CODE.replace("    p[0] = 1;", "  p[0]  =  1;   // set"))
    assert a == b


def test_a_code_change_changes_the_digest(tmp_path):
    a = digest_of(tmp_path, CODE)
    b = digest_of(tmp_path, CODE.replace("p[0] = 1", "p[0] = 2"))
    assert a != b


def test_a_stale_digest_gives_no_traffic():
    assert bench.profiled_traffic("decode_kernel_qwen3_decode.md", "0" * 16) is None
