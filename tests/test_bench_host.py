"""Host-side checks of bench.py's bookkeeping, CPU only."""
import os
import sys

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402


def test_source_hash_follows_code_not_comments():
    # the recorded DRAM traffic of the GEMM is tied to a hash of its sources;
    # an edit to a comment keeps the hash, an edit to the code changes it
    a = "int x = 1;  // one\n/* a block\n   comment */\nint y = 2;\n"
    b = "int x = 1;  // uno\n\n/* another */\nint y = 2;   \n"
    c = "int x = 1;\nint y = 3;\n"
    assert bench.strip_comments(a) == bench.strip_comments(b)
    assert bench.strip_comments(a) != bench.strip_comments(c)
    def read(path, edit=None):
        src = open(os.path.join(bench.ROOT, path), encoding="utf-8").read()
        return edit(src) if edit else src
    h0 = bench.gemm_sources_hash(read)
    assert bench.gemm_sources_hash(lambda p: read(p, lambda s: "// a new first line\n" + s)) == h0
    assert bench.gemm_sources_hash(lambda p: read(p, lambda s: s + "\nint extra_symbol;\n")) != h0
