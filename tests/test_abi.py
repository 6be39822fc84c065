"""The C-ABI library loads and exports every entry point that include/hq.h declares (no GPU needed)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
LIB = os.path.join(ROOT, "quantized_gemm_dequant_gb300", "libhq.so")


def declared():
    src = open(os.path.join(ROOT, "include", "hq.h")).read()
    return sorted(set(re.findall(r"HQ_API\s+[\w\s\*]+?\b(hq_\w+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared()
    for must in ("hq_pack_weights", "hq_gemm", "hq_moe_gemm", "hq_unpack_weights", "hq_workspace_bytes"):
        assert must in names


def test_library_exports_every_declared_symbol():
    if not os.path.exists(LIB):
        import __graft_entry__
        __graft_entry__.build()
    lib = ctypes.CDLL(LIB)
    for name in declared():
        assert hasattr(lib, name), name


def test_host_only_queries_work_without_a_gpu():
    import quantized_gemm_dequant_gb300 as hq
    f = hq.make_format("uint4_zp", 14336, 4096)
    # packed bytes: 112 tiles x 32 groups x 8576 bytes
    assert hq.packed_bytes(f) == 112 * 32 * 8576
    assert hq.packed_bytes(hq.make_format("int4_sym", 100, 100)) == 0
    assert hq.status_string(hq.HQ_ERR_BAD_ROUTING).startswith("top-k")
    assert set(hq.EXPORTS) == set(declared())
