"""Tensor checks of the Python binding (no GPU).

The C ABI takes bare pointers and sizes, so the binding checks every tensor it
turns into a pointer before calling the library: its dtype where the interface
fixes one (bf16 activations, outputs and bias; int32 routing ids; fp32 top-k
weights and scales), contiguity, that it holds at least the bytes the call reads
or writes, and that it lives in the current CUDA device's memory.  Each test
here builds host tensors that fail exactly one of these checks (or, with every
other property right, only the device one) and expects HQArgError, which is both
an HQError with status HQ_ERR_INVALID_ARG and a ValueError, raised before the
library is reached.
"""
import numpy as np
import pytest
import torch

hq = pytest.importorskip("quantized_gemm_dequant_gb300")

M, N, K = 4, 128, 256


def _fmt(w="uint4_zp", E=1, n=N, k=K):
    return hq.make_format(w, n, k, E)


def _packed(fmt):
    return torch.zeros(hq.packed_bytes(fmt), dtype=torch.uint8)


def _raises(fn, *words):
    with pytest.raises(hq.HQArgError) as e:
        fn()
    assert e.value.code == hq.HQ_ERR_INVALID_ARG
    assert isinstance(e.value, hq.HQError) and isinstance(e.value, ValueError)
    for w in words:
        assert w in str(e.value), str(e.value)
    return e.value


def test_gemm_activation_checks():
    fmt = _fmt()
    p = _packed(fmt)
    _raises(lambda: hq.gemm(fmt, {"data": torch.zeros(M, K, dtype=torch.float16)}, p, M), "act['data']", "dtype")
    _raises(lambda: hq.gemm(fmt, {"data": torch.zeros(K, M, dtype=torch.bfloat16).t()}, p, M), "contiguous")
    _raises(lambda: hq.gemm(fmt, {"data": torch.zeros(M - 1, K, dtype=torch.bfloat16)}, p, M),
            f"holds {2 * (M - 1) * K} bytes", f"{2 * M * K}")
    _raises(lambda: hq.gemm(fmt, {"data": np.zeros((M, K), dtype=np.float32)}, p, M), "torch.Tensor")
    # everything right but the memory it lives in
    _raises(lambda: hq.gemm(fmt, {"data": torch.zeros(M, K, dtype=torch.bfloat16)}, p, M), "device memory")
    _raises(lambda: hq.gemm_static_scratch(fmt, {"data": torch.zeros(M, K, dtype=torch.bfloat16)}, p, M),
            "device memory")


def test_gemm_scaled_activation_checks():
    # FP8 activations with a per-token scale: the scale must be fp32 [M]
    fmt = _fmt("mxfp4")
    p = _packed(fmt)
    data = torch.zeros(M, K, dtype=torch.uint8)
    _raises(lambda: hq.gemm(fmt, {"data": data, "scale": torch.zeros(M, dtype=torch.float16)}, p, M),
            "act['scale']", "dtype")
    _raises(lambda: hq.gemm(fmt, {"data": data, "scale": torch.zeros(M - 1, dtype=torch.float32)}, p, M),
            "act['scale']", "bytes")
    # NVFP4 activations: packed e2m1 rows of K/2 bytes, block scales of K/16 bytes
    fmt = _fmt("nvfp4")
    p = _packed(fmt)
    _raises(lambda: hq.gemm(fmt, {"data": torch.zeros(M, K // 2 - 1, dtype=torch.uint8)}, p, M), "act['data']")
    _raises(lambda: hq.gemm(fmt, {"data": torch.zeros(M, K // 2, dtype=torch.uint8),
                                  "scale": torch.zeros(M, K // 16 - 1, dtype=torch.uint8)}, p, M), "act['scale']")


def test_gemm_weight_bias_output_and_workspace_checks():
    fmt = _fmt()
    a = {"data": torch.zeros(M, K, dtype=torch.bfloat16)}
    p = _packed(fmt)
    _raises(lambda: hq.gemm(fmt, a, p[:-16], M), "packed", "bytes")
    _raises(lambda: hq.gemm(fmt, a, p, M, bias=torch.zeros(N, dtype=torch.float32)), "bias", "dtype")
    _raises(lambda: hq.gemm(fmt, a, p, M, bias=torch.zeros(N - 1, dtype=torch.bfloat16)), "bias", "bytes")
    _raises(lambda: hq.gemm(fmt, a, p, M, out=torch.zeros(M, N, dtype=torch.float32)), "out", "dtype")
    _raises(lambda: hq.gemm(fmt, a, p, M, out=torch.zeros(M, N - 1, dtype=torch.bfloat16)), "out", "bytes")
    _raises(lambda: hq.gemm(fmt, a, p, M, out=torch.zeros(N, M, dtype=torch.bfloat16).t()), "out", "contiguous")
    _raises(lambda: hq.gemm(fmt, a, p, M, workspace=torch.zeros(64, 4, dtype=torch.uint8).t()), "workspace",
            "contiguous")
    _raises(lambda: hq.gemm_static_scratch(fmt, a, p, M, out=torch.zeros(M, N, dtype=torch.float16)), "out")


def test_moe_routing_checks():
    fmt = _fmt("int4_sym", E=8)
    p = _packed(fmt)
    a = {"data": torch.zeros(M, K, dtype=torch.bfloat16)}
    ids64 = torch.zeros(M, 2, dtype=torch.int64)  # what torch.topk returns
    _raises(lambda: hq.moe_gemm(fmt, a, p, ids64), "topk_ids", "torch.int32")
    _raises(lambda: hq.moe_gemm(fmt, a, p, torch.zeros(M * 2, dtype=torch.int32)), "2-D")
    ids = torch.zeros(M, 2, dtype=torch.int32)
    _raises(lambda: hq.moe_gemm(fmt, a, p, ids, torch.zeros(M, 2, dtype=torch.float64)), "topk_weights", "dtype")
    _raises(lambda: hq.moe_gemm(fmt, a, p, ids, torch.zeros(M, 1, dtype=torch.float32)), "topk_weights", "bytes")
    _raises(lambda: hq.moe_gemm(fmt, a, p, torch.zeros(2, M, dtype=torch.int32).t()), "topk_ids", "contiguous")
    _raises(lambda: hq.moe_gemm(fmt, a, p, ids), "topk_ids", "device memory")
    _raises(lambda: hq.moe_gemm_combine(fmt, a, p, ids64), "topk_ids", "torch.int32")
    # the combine reads T * topk routed rows: M tokens of top-2 need 2M activation rows
    _raises(lambda: hq.moe_gemm_combine(fmt, a, p, ids), "act['data']", f"{2 * 2 * M * K}")
    a2 = {"data": torch.zeros(2 * M, K, dtype=torch.bfloat16)}
    _raises(lambda: hq.moe_gemm_combine(fmt, a2, p, ids, out=torch.zeros(M, N - 1, dtype=torch.bfloat16)), "out",
            "bytes")
    _raises(lambda: hq.moe_gemm_combine(fmt, a2, p, ids), "topk_ids", "device memory")
    # moe_gemm writes T * topk output rows
    _raises(lambda: hq.moe_gemm(fmt, a, p, ids, out=torch.zeros(M, N, dtype=torch.bfloat16)), "out", "bytes")


def test_swiglu_and_quantize_checks():
    _raises(lambda: hq.swiglu(torch.zeros(4, 7, dtype=torch.bfloat16)), "2-D")
    _raises(lambda: hq.swiglu(torch.zeros(4, 8, dtype=torch.float32)), "x", "dtype")
    _raises(lambda: hq.swiglu(torch.zeros(8, 4, dtype=torch.bfloat16).t()), "contiguous")
    _raises(lambda: hq.swiglu(torch.zeros(4, 8, dtype=torch.bfloat16)), "device memory")
    _raises(lambda: hq.quantize_act("e4m3_tok", torch.zeros(4, 32, dtype=torch.float32)), "x", "dtype")
    _raises(lambda: hq.quantize_act("e4m3_tok", torch.zeros(128, dtype=torch.bfloat16)), "2-D")
    _raises(lambda: hq.quantize_act("nvfp4", torch.zeros(4, 32, dtype=torch.bfloat16),
                                    global_amax=torch.zeros(1, dtype=torch.float16)), "global_amax", "dtype")


def test_pack_checks():
    fmt = _fmt("uint4_zp", E=2)
    codes = torch.zeros(2, N, K // 2, dtype=torch.uint8)
    scales = torch.zeros(2, N, 2 * (K // 128), dtype=torch.uint8)
    zeros = torch.zeros(2, N, K // 128, dtype=torch.uint8)
    _raises(lambda: hq.pack_weights(fmt, codes[:1], scales, zeros), "codes", "bytes")
    _raises(lambda: hq.pack_weights(fmt, codes, scales[:, :, :1], zeros), "scales")
    _raises(lambda: hq.pack_weights(fmt, codes, scales, zeros[:1]), "zeros", "bytes")
    _raises(lambda: hq.pack_weights(fmt, codes, scales, zeros), "device memory")
    _raises(lambda: hq.pack_weights(fmt, None, scales, zeros), "required")
    nv = _fmt("nvfp4", E=2)
    _raises(lambda: hq.pack_weights(nv, torch.zeros(2, N, K // 2, dtype=torch.uint8),
                                    torch.zeros(2, N, K // 16, dtype=torch.uint8), None,
                                    torch.zeros(2, dtype=torch.float64)), "global_scale", "dtype")
    # UINT3 codes are a 3-bit string per row: K * 3 / 8 bytes
    u3 = _fmt("uint3_zp")
    _raises(lambda: hq.pack_weights(u3, torch.zeros(N, K * 3 // 8 - 1, dtype=torch.uint8),
                                    torch.zeros(N, 2 * (K // 128), dtype=torch.uint8),
                                    torch.zeros(N, K // 128, dtype=torch.uint8)), "codes", "bytes")


def test_status_and_workspace_checks():
    _raises(lambda: hq.last_device_status(torch.zeros(1, dtype=torch.uint8)), "workspace", "bytes")
    _raises(lambda: hq.last_device_status(torch.zeros(256, dtype=torch.uint8)), "device memory")


@pytest.mark.gpu
def test_host_tensors_beside_device_tensors_are_refused(lib):
    """On a GPU: a host tensor among device tensors, or device tensors of the wrong dtype, are refused by name; a
    call with every argument right still runs and leaves the workspace status clean."""
    fmt = lib.make_format("uint4_zp", N, K)
    a = {"data": torch.zeros(M, K, dtype=torch.bfloat16, device="cuda")}
    p = torch.zeros(lib.packed_bytes(fmt), dtype=torch.uint8, device="cuda")
    _raises(lambda: lib.gemm(fmt, a, p, M, bias=torch.zeros(N, dtype=torch.bfloat16)), "bias", "device memory")
    _raises(lambda: lib.gemm(fmt, a, p.cpu(), M), "packed", "device memory")
    ws = lib.make_workspace(fmt, M)
    y = lib.gemm(fmt, a, p, M, workspace=ws)
    torch.cuda.synchronize()
    assert y.shape == (M, N) and lib.last_device_status(ws) == lib.HQ_OK
    moe = lib.make_format("int4_sym", N, K, 4)
    pm = torch.zeros(lib.packed_bytes(moe), dtype=torch.uint8, device="cuda")
    ids = torch.zeros(M, 2, dtype=torch.int64, device="cuda")
    _raises(lambda: lib.moe_gemm(moe, a, pm, ids), "topk_ids", "torch.int32")
