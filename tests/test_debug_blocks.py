"""The debug build's check blocks in the CUDA sources (no GPU).

Device-side index checks live only in blocks that open with the line
`#if HQ_DEBUG_BOUNDS` and close with their matching `#endif`; the product build
(libhq.so) compiles none of them.  The benchmark's kernel-source hash, which
decides whether recorded DRAM counters still describe the kernels, is taken over
the sources with those blocks left out.  These tests pin that rule: the stripping
removes exactly such blocks (nested directives included), and every mention of
the macro in the sources is such an opening line, with no #else / #elif branch
that the product build would compile.
"""
import os

import bench

CSRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "quantized_gemm_dequant_gb300",
                    "csrc")


def test_product_source_drops_only_debug_blocks():
    text = ("a\n#if HQ_DEBUG_BOUNDS\nx\n#if FOO\ny\n#endif\nz\n#endif\nb\n"
            "#if FOO\nc\n#endif\n  #if HQ_DEBUG_BOUNDS\n  w\n  #endif\nd")
    assert bench.product_source(text) == "a\nb\n#if FOO\nc\n#endif\nd"
    plain = "int f();\n#if X\n#endif\n"
    assert bench.product_source(plain) == plain


def test_debug_blocks_are_well_formed():
    blocks = 0
    for f in sorted(os.listdir(CSRC)):
        if not f.endswith((".cu", ".cuh", ".h")):
            continue
        depth = 0
        for no, line in enumerate(open(os.path.join(CSRC, f)).read().splitlines(), 1):
            s = line.strip()
            if "HQ_DEBUG_BOUNDS" in s:
                assert s == "#if HQ_DEBUG_BOUNDS" and depth == 0, f"{f}:{no}: {s}"
                depth, blocks = 1, blocks + 1
                continue
            if depth:
                if s.startswith("#if"):
                    depth += 1
                elif s.startswith("#endif"):
                    depth -= 1
                elif depth == 1 and s.startswith(("#else", "#elif")):
                    raise AssertionError(f"{f}:{no}: a debug block may not have a product-build branch")
        assert depth == 0, f"{f}: unclosed debug block"
    assert blocks > 0
