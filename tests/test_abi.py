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
    # the launch plan is host logic: register-decode kernel for small M, tcgen05 for large M, formats only the
    # register-decode kernel reads at any M, MXFP4 x MXFP4 on its own tcgen05 variant, bad arguments refused
    assert hq.launch_plan(f, 1)["kernel"] == "regdec"
    big = hq.launch_plan(f, 8192)
    assert big["kernel"] == "umma" and big["variant"] == 0 and big["bt"] == 256
    assert hq.launch_plan(hq.make_format("uint3_zp", 4096, 4096), 4096)["kernel"] == "regdec"
    x = hq.launch_plan(hq.make_format("mxfp4", 4096, 7168, act_type=hq.HQ_A_MXFP4), 1024)
    assert x["kernel"] == "umma" and x["variant"] == 4
    with pytest.raises(hq.HQError):
        hq.launch_plan(f, 0)
    # MXFP4 weights for MXFP4 activations are packed like NVFP4 (256-K blocks of 18432 bytes)
    assert hq.packed_bytes(hq.make_format("mxfp4", 256, 1024, act_type=hq.HQ_A_MXFP4)) == 2 * 4 * 18432


def _lib():
    import quantized_gemm_dequant_gb300 as hq
    return hq


def test_quantize_act_host_checks_without_a_gpu():
    """Argument errors of hq_quantize_act come back before anything touches the device (fake pointers are never
    dereferenced on these paths)."""
    hq = _lib()
    L = hq._lib
    X, D, S, G, WS = 0x10000, 0x20000, 0x30000, 0x40000, 0x50000
    nv, f8 = hq.HQ_A_NVFP4, hq.HQ_A_E4M3_TOKEN
    assert L.hq_quantize_act(99, X, 4, 64, None, D, S, G, WS, 1 << 20, None) == hq.HQ_ERR_UNSUPPORTED
    assert L.hq_quantize_act(nv, X, -1, 64, None, D, S, G, WS, 1 << 20, None) == hq.HQ_ERR_INVALID_ARG
    assert L.hq_quantize_act(nv, X, 4, 8, None, D, S, G, WS, 1 << 20, None) == hq.HQ_ERR_INVALID_ARG
    assert L.hq_quantize_act(nv, X, 4, 24, None, D, S, G, WS, 1 << 20, None) == hq.HQ_ERR_ALIGNMENT
    assert L.hq_quantize_act(nv, X, 4, 64, None, D, S, None, WS, 1 << 20, None) == hq.HQ_ERR_INVALID_ARG
    assert L.hq_quantize_act(f8, None, 4, 64, None, D, S, None, None, 0, None) == hq.HQ_ERR_INVALID_ARG
    assert L.hq_quantize_act(f8, X + 8, 4, 64, None, D, S, None, None, 0, None) == hq.HQ_ERR_ALIGNMENT
    assert L.hq_quantize_act(nv, X, 4, 64, None, D, S, G, None, 0, None) == hq.HQ_ERR_WORKSPACE
    assert L.hq_quantize_act(nv, X, 4, 64, None, D, S, G, WS, 64, None) == hq.HQ_ERR_WORKSPACE
    assert L.hq_quantize_act(f8, X, 0, 64, None, D, S, None, None, 0, None) == hq.HQ_OK  # nothing to do
    assert hq.quantize_act_workspace_bytes("nvfp4", 8192, 7168) == 4 * 4096
    assert hq.quantize_act_workspace_bytes("e4m3_tok", 8192, 7168) == 0
    assert L.hq_quantize_act_workspace_bytes(nv, 8, 24) == 0


def test_swiglu_host_checks_without_a_gpu():
    hq = _lib()
    L = hq._lib
    assert L.hq_swiglu(0x10000, -1, 64, 0x20000, None) == hq.HQ_ERR_INVALID_ARG
    assert L.hq_swiglu(0x10000, 4, 12, 0x20000, None) == hq.HQ_ERR_ALIGNMENT
    assert L.hq_swiglu(None, 4, 64, 0x20000, None) == hq.HQ_ERR_INVALID_ARG
    assert L.hq_swiglu(0x10008, 4, 64, 0x20000, None) == hq.HQ_ERR_ALIGNMENT
    assert L.hq_swiglu(None, 0, 64, None, None) == hq.HQ_OK  # no rows


def test_moe_combine_host_checks_without_a_gpu():
    import ctypes
    hq = _lib()
    L = hq._lib
    f = hq.make_format("int4_sym", 2048, 768, num_experts=128)
    A = hq.Act(0x10000, None, None)
    args = lambda T, k, ids=0x30000, C=0x40000: (ctypes.byref(f), ctypes.byref(A), 0x20000, ids, None, T, k, C,
                                                 0x50000, 1 << 30, None)
    assert L.hq_moe_gemm_combine(*args(-1, 8)) == hq.HQ_ERR_INVALID_ARG
    assert L.hq_moe_gemm_combine(*args(4, 0)) == hq.HQ_ERR_INVALID_ARG
    assert L.hq_moe_gemm_combine(*args(0, 8)) == hq.HQ_OK  # no tokens
    assert L.hq_moe_gemm_combine(*args(4, 8, ids=None)) == hq.HQ_ERR_INVALID_ARG
    assert L.hq_moe_gemm_combine(*args(4, 8, C=None)) == hq.HQ_ERR_INVALID_ARG
    bad = hq.make_format("int4_sym", 2048, 768, num_experts=128, group_size=64)
    assert L.hq_moe_gemm_combine(ctypes.byref(bad), ctypes.byref(A), 0x20000, 0x30000, None, 4, 8, 0x40000, 0x50000,
                                 1 << 30, None) == hq.HQ_ERR_UNSUPPORTED
    # the workspace holds the plan's regions and one fp32 row of N per token; the call adds one rounding kernel
    assert L.hq_moe_combine_workspace_bytes(ctypes.byref(f), 4096, 8) >= 4096 * 2048 * 4 + 256
    assert L.hq_moe_combine_workspace_bytes(ctypes.byref(f), -1, 8) == 0
    assert hq.kernels_per_call(f, 4096, 8, moe="combine") == hq.kernels_per_call(f, 4096, 8, moe=True) + 1
