"""bench.py host logic that needs no GPU: the digest that ties an ncu
traffic capture to the kernel sources it was taken on."""

import os
import shutil

import bench

CSRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                    "paged_split_kv_02_gb300", "csrc")


def test_digest_ignores_comments_and_sees_code(tmp_path):
    d = tmp_path / "csrc"
    shutil.copytree(CSRC, d, ignore=shutil.ignore_patterns("*.o", "*.so"))
    base = bench._kernel_sources_digest(str(d))
    assert base == bench._kernel_sources_digest(CSRC)
    k = d / "pd_kernel.cuh"
    text = k.read_text()
    # comments and blank lines added or reworded: same digest
    k.write_text("// a new comment line\n\n/* and a block\n   comment */\n" +
                 text.replace("// ring and Q tile are dead from here on", "// reworded"))
    assert bench._kernel_sources_digest(str(d)) == base
    # a code change (even inside a line that also holds a comment): another digest
    k.write_text(text.replace("constexpr int kSpec = 256;", "constexpr int kSpec = 128;"))
    assert bench._kernel_sources_digest(str(d)) != base
    # a string literal that contains "//" is code, not a comment
    k.write_text(text + '\nstatic const char *kPdTestLiteral = "a // b";\n')
    other = bench._kernel_sources_digest(str(d))
    k.write_text(text + '\nstatic const char *kPdTestLiteral = "a // c";\n')
    assert bench._kernel_sources_digest(str(d)) != other
