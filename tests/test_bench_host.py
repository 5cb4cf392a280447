"""Host-side checks of bench.py's bookkeeping, CPU only."""
import os
import sys

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402


def test_source_hash_follows_every_edit():
    # the recorded DRAM traffic of the GEMM is tied to a hash of its sources
    # as written: any edit - code, a comment, or text inside a string literal
    # such as an inline-PTX statement - changes the hash and voids the figure
    def read(path, edit=None):
        src = open(os.path.join(bench.ROOT, path), encoding="utf-8").read()
        return edit(src) if edit else src
    h0 = bench.gemm_sources_hash(read)
    assert bench.gemm_sources_hash(read) == h0
    assert bench.gemm_sources_hash(lambda p: read(p, lambda s: "// a new first line\n" + s)) != h0
    assert bench.gemm_sources_hash(lambda p: read(p, lambda s: s + "\nint extra_symbol;\n")) != h0
    asm = 'asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");'
    assert bench.gemm_sources_hash(lambda p: read(p, lambda s: s + asm)) != \
        bench.gemm_sources_hash(lambda p: read(p, lambda s: s + asm.replace("before", "after")))
