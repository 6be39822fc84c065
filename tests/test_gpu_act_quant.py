"""Activation quantization on the GPU against the CPU oracle (bit-exact codes and scales), and its use as the GEMM's
activation operand.

Codes are integer decisions taken on binary32 results, so the kernel and the oracle must agree bit for bit: codes,
block scales and the fp32 scales (compared as bit patterns).
"""
import numpy as np
import pytest
import torch

import oracle
from tests import ref_helpers as R
from workload import configs as W

pytestmark = pytest.mark.gpu

SHAPES = [(1, 16), (3, 48), (17, 7168), (130, 2048), (64, 4096), (5, 4112)]


def _x(seed, M, K):
    """bf16 [M, K] on the device: N(0, 1) with x20 outliers, rows scaled by powers of two, and the awkward rows (a
    zero row, a single-spike row, a row of values whose scales underflow)."""
    x = W.acts_fp32(seed, M, K, outliers=True, device="cuda")
    x = x * torch.exp2(torch.arange(M, device="cuda", dtype=torch.float32).remainder(13) - 6).unsqueeze(1)
    if M > 3:
        x[1] = 0.0
        x[2] = 0.0
        x[2, K // 3] = -3.0e4
        x[3] = x[3] * 1e-30
    return x.to(torch.bfloat16).contiguous()


def _bits(x):
    return R.np_bits(x)


def _f32bits(t):
    return t.detach().cpu().numpy().astype(np.float32).view(np.uint32)


@pytest.mark.parametrize("M,K", SHAPES)
@pytest.mark.parametrize("seed", [0, 1])
def test_fp8_per_token_bit_exact(lib, M, K, seed):
    x = _x(seed, M, K)
    out = lib.quantize_act("e4m3_tok", x)
    torch.cuda.synchronize()
    q, s = oracle.quantize_act_e4m3_per_token(_bits(x))
    assert np.array_equal(out["data"].cpu().numpy(), q)
    assert np.array_equal(_f32bits(out["scale"]), s.view(np.uint32))


@pytest.mark.parametrize("M,K", SHAPES)
@pytest.mark.parametrize("seed", [0, 1])
@pytest.mark.parametrize("calibrated", [False, True])
def test_nvfp4_bit_exact(lib, M, K, seed, calibrated):
    x = _x(seed, M, K)
    xb = _bits(x)
    amax = None
    if calibrated:  # a calibrated amax below the true one: the outliers saturate
        amax = np.float32(np.abs((xb.astype(np.uint32) << 16).view(np.float32)).max() / 3)
    out = lib.quantize_act("nvfp4", x, global_amax=None if amax is None else torch.tensor([amax], device="cuda"))
    torch.cuda.synchronize()
    q, sb, g = oracle.quantize_act_nvfp4(xb, global_amax=amax)
    assert np.array_equal(out["data"].cpu().numpy(), q)
    assert np.array_equal(out["scale"].cpu().numpy(), sb)
    assert _f32bits(out["gscale"])[0] == np.float32(g).view(np.uint32)


@pytest.mark.parametrize("e", [-80, -88, -92, -96, -104, -118])
@pytest.mark.parametrize("calibrated", [False, True])
def test_nvfp4_tiny_scales_bit_exact(lib, e, calibrated):
    """Tensors whose global scale g = amax / 2688 lies near or below 2^-100: the block-scale and code divisions leave
    the reciprocal shortcut for IEEE division there, and the codes must not change at the switch.  Rows span 2^-30
    of magnitude, so the blocks' quotients cover the e4m3 and e2m1 rounding boundaries down to zero codes."""
    M, K = 48, 1024
    x = W.acts_fp32(7, M, K, outliers=True, device="cuda")
    x = x * torch.exp2(e - torch.arange(M, device="cuda", dtype=torch.float32).remainder(31)).unsqueeze(1)
    x = x.to(torch.bfloat16).contiguous()
    xb = _bits(x)
    amax = None
    if calibrated:
        amax = np.float32(np.abs((xb.astype(np.uint32) << 16).view(np.float32)).max() / 3)
    out = lib.quantize_act("nvfp4", x, global_amax=None if amax is None else torch.tensor([amax], device="cuda"))
    torch.cuda.synchronize()
    q, sb, g = oracle.quantize_act_nvfp4(xb, global_amax=amax)
    assert np.array_equal(out["scale"].cpu().numpy(), sb)
    assert np.array_equal(out["data"].cpu().numpy(), q)
    assert _f32bits(out["gscale"])[0] == np.float32(g).view(np.uint32)


def test_zero_tensor_and_empty_rows(lib):
    x = torch.zeros((7, 64), dtype=torch.bfloat16, device="cuda")
    o8 = lib.quantize_act("e4m3_tok", x)
    o4 = lib.quantize_act("nvfp4", x)
    torch.cuda.synchronize()
    assert not o8["data"].any() and not o8["scale"].any()
    assert not o4["data"].any() and not o4["scale"].any() and float(o4["gscale"][0]) == 0.0
    e = torch.empty((0, 64), dtype=torch.bfloat16, device="cuda")
    o4 = lib.quantize_act("nvfp4", e)
    o8 = lib.quantize_act("e4m3_tok", e)
    torch.cuda.synchronize()
    assert float(o4["gscale"][0]) == 0.0 and o8["data"].numel() == 0


def test_rejects_bad_arguments(lib):
    x = torch.zeros((4, 24), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(lib.HQError) as e:
        lib.quantize_act("nvfp4", x)
    assert e.value.code == lib.HQ_ERR_ALIGNMENT
    x = torch.zeros((4, 32), dtype=torch.bfloat16, device="cuda")
    out = dict(data=torch.empty((4, 16), dtype=torch.uint8, device="cuda"),
               scale=torch.empty((4, 2), dtype=torch.uint8, device="cuda"),
               gscale=torch.empty((1,), dtype=torch.float32, device="cuda"))
    with pytest.raises(lib.HQError) as e:
        lib.quantize_act("nvfp4", x, out=out, workspace=torch.empty(16, dtype=torch.uint8, device="cuda"))
    assert e.value.code == lib.HQ_ERR_WORKSPACE


@pytest.mark.parametrize("wfmt", ["nvfp4", "mxfp4"])
def test_quantized_activations_feed_the_gemm(lib, wfmt):
    """bf16 activations quantized on the device, then the W4A4 / W4A8 GEMM: the result matches the oracle's GEMM
    on the oracle's quantization of the same activations."""
    afmt = "nvfp4" if wfmt == "nvfp4" else "e4m3_tok"
    c = dict(kind="dense", wfmt=wfmt, afmt=afmt, G=16 if wfmt == "nvfp4" else 32)
    M, N, K = 37, 300, 768
    inp = W.make_dense(c, M, seed=3, N=N, K=K)
    x = _x(3, M, K)
    act = lib.quantize_act(afmt, x)
    fmt, packed = lib.pack_inputs(inp, "cuda")
    y = lib.gemm(fmt, act, packed, M)
    torch.cuda.synchronize()
    if afmt == "nvfp4":
        q, sb, g = oracle.quantize_act_nvfp4(_bits(x))
        adeq = oracle.dequant_acts("nvfp4", q, sb, np.array([g], np.float32))
    else:
        q, s = oracle.quantize_act_e4m3_per_token(_bits(x))
        adeq = oracle.dequant_acts("e4m3_tok", q, s)
    ref = oracle.gemm(adeq, R.weights_of(inp))
    R.assert_parity(y, ref, f"{wfmt} on device-quantized activations")


@pytest.mark.parametrize("afmt", ["e4m3_tok", "nvfp4"])
def test_full_size_sampled_rows(lib, afmt):
    """M = 8192, K = 7168 (the NVFP4 and MXFP4 workloads' largest activation): sampled rows bit-exact; NVFP4 takes
    the tensor's amax, which the oracle receives from the whole tensor."""
    M, K = 8192, 7168
    x = _x(4, M, K)
    out = lib.quantize_act(afmt, x)
    torch.cuda.synchronize()
    rows = np.array([0, 1, 2, 3, 4, 777, 4095, 8191])
    xb = _bits(x[torch.as_tensor(rows, device="cuda")])
    if afmt == "e4m3_tok":
        q, s = oracle.quantize_act_e4m3_per_token(xb)
        assert np.array_equal(out["data"][rows].cpu().numpy(), q)
        assert np.array_equal(_f32bits(out["scale"][rows]), s.view(np.uint32))
    else:
        amax = np.float32(x.float().abs().max().item())  # exact: the max of bf16 values
        q, sb, g = oracle.quantize_act_nvfp4(xb, global_amax=amax)
        assert np.array_equal(out["data"][rows].cpu().numpy(), q)
        assert np.array_equal(out["scale"][rows].cpu().numpy(), sb)
        assert _f32bits(out["gscale"])[0] == np.float32(g).view(np.uint32)
