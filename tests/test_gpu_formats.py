"""More weight formats through the same decode component, against the CPU oracle (GPU).

INT8 (the e0m7 value set), UINT1 / UINT2 / UINT3 with zero points, MXINT4 (e8m0
block-32 scales) and FP8 E4M3 weights, each with bf16 activations: the other WnA16
widths and formats of "Results: kernel microbenchmarks" and the zero-exponent
INT8 of "Results: quantization support".  The register-decode kernel reads
them at every token count (32-token tiles beyond 16 tokens).  Checked here:
repack round trips bit for bit, element-wise parity against the oracle for
dense calls (ragged N, several token counts, bias) and MoE calls, and bit-exact
results for integer activations with power-of-two scales.
"""
import numpy as np
import pytest
import torch

from tests import ref_helpers as R
from workload import make_dense, make_moe, quant

pytestmark = pytest.mark.gpu

FORMS = {
    "int8_sym": dict(kind="dense", wfmt="int8_sym", afmt="bf16", G=128),
    "uint2_zp": dict(kind="dense", wfmt="uint2_zp", afmt="bf16", G=128),
    "mxint4": dict(kind="dense", wfmt="mxint4", afmt="bf16", G=32),
    "e4m3": dict(kind="dense", wfmt="e4m3", afmt="bf16", G=128),
    "uint1_zp": dict(kind="dense", wfmt="uint1_zp", afmt="bf16", G=128),
    "uint3_zp": dict(kind="dense", wfmt="uint3_zp", afmt="bf16", G=128),
}
CODE_BITS = {"int8_sym": 8, "e4m3": 8, "uint2_zp": 2, "mxint4": 4, "uint1_zp": 1, "uint3_zp": 3}
ZERO_BITS = {"uint2_zp": 2, "uint1_zp": 1, "uint3_zp": 3}


@pytest.mark.parametrize("wfmt", list(FORMS))
def test_pack_unpack_round_trip_bit_exact(lib, wfmt):
    E, N, K = 2, 300, 512
    g = FORMS[wfmt]["G"]
    gen = torch.Generator().manual_seed(21)
    codes = torch.randint(0, 256, (E, N, K * CODE_BITS[wfmt] // 8), generator=gen, dtype=torch.uint8)
    if wfmt == "mxint4":
        scales = torch.randint(0, 256, (E, N, K // g), generator=gen, dtype=torch.uint8)
    else:
        scales = torch.randint(0, 65536, (E, N, K // g), generator=gen, dtype=torch.int32).to(torch.int16)
        scales = scales.view(torch.uint8).reshape(E, N, 2 * (K // g))
    zeros = (torch.randint(0, 1 << ZERO_BITS[wfmt], (E, N, K // g), generator=gen, dtype=torch.uint8)
             if wfmt in ZERO_BITS else None)
    fmt = lib.make_format(wfmt, N, K, E)
    packed = lib.pack_weights(fmt, codes.cuda(), scales.cuda(), zeros.cuda() if zeros is not None else None)
    c2 = torch.zeros_like(codes).cuda()
    s2 = torch.zeros_like(scales).cuda()
    z2 = torch.zeros_like(zeros).cuda() if zeros is not None else None
    lib.unpack_weights(fmt, packed, c2, s2, z2)
    torch.cuda.synchronize()
    assert torch.equal(c2.cpu(), codes)
    assert torch.equal(s2.cpu(), scales)
    if zeros is not None:
        assert torch.equal(z2.cpu(), zeros)


@pytest.mark.parametrize("wfmt", list(FORMS))
@pytest.mark.parametrize("M", [1, 7, 16, 33, 100])
def test_dense_parity(lib, wfmt, M):
    inp = make_dense(FORMS[wfmt], M, seed=M + 7, N=300, K=640, with_bias=M % 2 == 1)
    fmt, packed = lib.pack_inputs(inp, "cuda")
    act = {k: v.cuda() for k, v in inp["a"].items()}
    bias = inp["bias"].cuda() if inp.get("bias") is not None else None
    y = lib.gemm(fmt, act, packed, M, bias=bias)
    torch.cuda.synchronize()
    R.assert_parity(y, R.dense_ref(inp), f"{wfmt} M={M}")


@pytest.mark.parametrize("wfmt", list(FORMS))
@pytest.mark.parametrize("T", [1, 9, 60])
def test_moe_parity(lib, wfmt, T):
    form = dict(FORMS[wfmt], kind="moe", topk=2)
    inp = make_moe(form, T, seed=T, E=5, N=256, K=512, topk=2)
    fmt, packed = lib.pack_inputs(inp, "cuda")
    act = {k: v.cuda() for k, v in inp["a"].items()}
    y = lib.moe_gemm(fmt, act, packed, inp["ids"].cuda(), inp["topk_w"].cuda())
    torch.cuda.synchronize()
    R.assert_parity(y, R.moe_ref(inp), f"moe {wfmt} T={T}")


@pytest.mark.parametrize("wfmt", list(FORMS))
def test_exact_integer_pow2_bit_exact(lib, wfmt):
    """Integer activations and power-of-two scales (e4m3 weights with exponents near 0): every partial sum is exact
    in fp32, so C equals the bf16 rounding of the exact result bit for bit."""
    gen = torch.Generator().manual_seed(9)
    M, N, K = 20, 256, 512
    G = FORMS[wfmt]["G"]
    j = torch.randint(-3, 1, (N, K // G), generator=gen)
    pow2_bf16 = ((j + 127) << 7).to(torch.int16).view(torch.bfloat16)
    if wfmt == "int8_sym":
        q = torch.randint(-127, 128, (N, K), generator=gen)
        w = dict(codes=(q & 0xFF).to(torch.uint8), scales=pow2_bf16)
    elif wfmt == "uint2_zp":
        q = torch.randint(0, 4, (N, K), generator=gen)
        w = dict(codes=quant.pack_crumbs(q.to(torch.uint8)), scales=pow2_bf16,
                 zeros=torch.randint(0, 4, (N, K // G), generator=gen, dtype=torch.uint8))
    elif wfmt in ("uint1_zp", "uint3_zp"):
        b = CODE_BITS[wfmt]
        q = torch.randint(0, 1 << b, (N, K), generator=gen)
        w = dict(codes=quant.pack_bits(q.to(torch.uint8), b), scales=pow2_bf16,
                 zeros=torch.randint(0, 1 << b, (N, K // G), generator=gen, dtype=torch.uint8))
    elif wfmt == "mxint4":
        q = torch.randint(-7, 8, (N, K), generator=gen)
        w = dict(codes=quant.pack_nibbles((q & 0xF).to(torch.uint8)), scales=(j + 127).to(torch.uint8))
    else:
        sgn = torch.randint(0, 2, (N, K), generator=gen) << 7
        ex = torch.randint(5, 9, (N, K), generator=gen) << 3  # |w| in [0.25, 4): products stay exact
        w = dict(codes=(sgn | ex | torch.randint(0, 8, (N, K), generator=gen)).to(torch.uint8), scales=pow2_bf16)
    inp = dict(M=M, N=N, K=K, wfmt=wfmt, afmt="bf16", G=G, w=w,
               a=dict(data=torch.randint(-3, 4, (M, K), generator=gen).to(torch.bfloat16)))
    fmt, packed = lib.pack_inputs(inp, "cuda")
    y = lib.gemm(fmt, {"data": inp["a"]["data"].cuda()}, packed, M)
    torch.cuda.synchronize()
    ref = R.dense_ref(inp)
    assert np.max(np.abs(ref)) < 2 ** 20
    want = torch.from_numpy(np.asarray(ref, dtype=np.float32)).to(torch.bfloat16)
    assert torch.equal(y.cpu(), want), "not bit-exact"


# ------------------------------------------------------------------ MXFP4 weights x MXFP8 activations (W4A8, MX)
MX8 = dict(kind="dense", wfmt="mxfp4", afmt="mxfp8", G=32)


@pytest.mark.parametrize("M", [1, 16, 100, 300])
def test_mxfp8_act_dense_parity(lib, M):
    """The microscaled W4A8 variant ("W8A8 / W4A8 / W4A4"): e8m0 block scales on both operands of the block-scaled
    tcgen05 MMA."""
    inp = make_dense(MX8, M, seed=M + 3, N=320, K=1024)
    fmt, packed = lib.pack_inputs(inp, "cuda")
    act = {k: v.cuda() for k, v in inp["a"].items()}
    y = lib.gemm(fmt, act, packed, M)
    torch.cuda.synchronize()
    R.assert_parity(y, R.dense_ref(inp), f"mxfp4 x mxfp8 M={M}")


@pytest.mark.parametrize("path", ["indexed", "grouped"])
@pytest.mark.parametrize("T", [5, 60, 300])
def test_mxfp8_act_moe_parity(lib, monkeypatch, path, T):
    monkeypatch.setenv("HQ_MOE_PATH", path)
    inp = make_moe(dict(MX8, kind="moe", topk=3), T, seed=T, E=6, N=256, K=1024, topk=3)
    fmt, packed = lib.pack_inputs(inp, "cuda")
    act = {k: v.cuda() for k, v in inp["a"].items()}
    y = lib.moe_gemm(fmt, act, packed, inp["ids"].cuda(), inp["topk_w"].cuda())
    torch.cuda.synchronize()
    R.assert_parity(y, R.moe_ref(inp), f"moe mxfp4 x mxfp8 {path} T={T}")


def test_mxfp8_act_exact_pow2_bit_exact(lib):
    """e2m1 weights, e4m3 activations with small exponents and power-of-two block scales on both sides: every partial
    sum is exact in fp32, so C equals the bf16 rounding of the exact result."""
    gen = torch.Generator().manual_seed(13)
    M, N, K = 24, 256, 1024
    jw = torch.randint(-1, 2, (N, K // 32), generator=gen)
    ja = torch.randint(-2, 2, (M, K // 32), generator=gen)
    sgn = torch.randint(0, 2, (M, K), generator=gen) << 7
    ex = torch.randint(6, 9, (M, K), generator=gen) << 3
    a8 = (sgn | ex | torch.randint(0, 8, (M, K), generator=gen)).to(torch.uint8)
    inp = dict(M=M, N=N, K=K, wfmt="mxfp4", afmt="mxfp8", G=32,
               w=dict(codes=torch.randint(0, 256, (N, K // 2), generator=gen, dtype=torch.uint8),
                      scales=(jw + 127).to(torch.uint8)),
               a=dict(data=a8, scale=(ja + 127).to(torch.uint8)))
    fmt, packed = lib.pack_inputs(inp, "cuda")
    y = lib.gemm(fmt, {k: v.cuda() for k, v in inp["a"].items()}, packed, M)
    torch.cuda.synchronize()
    ref = R.dense_ref(inp)
    assert np.max(np.abs(ref)) < 2 ** 20
    assert torch.equal(y.cpu(), torch.from_numpy(np.asarray(ref, dtype=np.float32)).to(torch.bfloat16))


def test_mxfp8_act_needs_k_multiple_of_512(lib):
    fmt = lib.make_format("mxfp4", 256, 640, act_type=lib.HQ_A_MXFP8)
    assert lib.packed_bytes(fmt) == 0


# ------------------------------------------------------------------ MXFP4 weights x MXFP4 activations (W4A4, MX)
MX4 = dict(kind="dense", wfmt="mxfp4", afmt="mxfp4", G=32)


def test_mxfp4_act_repack_round_trip_bit_exact(lib):
    """MXFP4 weights meant for MXFP4 activations take their own packed layout (packed e2m1 in the MMA)."""
    E, N, K = 2, 300, 1024
    gen = torch.Generator().manual_seed(23)
    codes = torch.randint(0, 256, (E, N, K // 2), generator=gen, dtype=torch.uint8)
    scales = torch.randint(0, 256, (E, N, K // 32), generator=gen, dtype=torch.uint8)
    fmt = lib.make_format("mxfp4", N, K, E, act_type=lib.HQ_A_MXFP4)
    packed = lib.pack_weights(fmt, codes.cuda(), scales.cuda())
    c2 = torch.zeros_like(codes).cuda()
    s2 = torch.zeros_like(scales).cuda()
    lib.unpack_weights(fmt, packed, c2, s2)
    torch.cuda.synchronize()
    assert torch.equal(c2.cpu(), codes) and torch.equal(s2.cpu(), scales)


@pytest.mark.parametrize("M", [1, 16, 100, 300])
def test_mxfp4_act_dense_parity(lib, M):
    """The microscaled W4A4 variant ("W8A8 / W4A8 / W4A4"): packed e2m1 on both operands, e8m0 block scales on both
    (kind::mxf4nvf4, scale_vec::2X)."""
    inp = make_dense(MX4, M, seed=M + 5, N=320, K=1024)
    fmt, packed = lib.pack_inputs(inp, "cuda")
    act = {k: v.cuda() for k, v in inp["a"].items()}
    y = lib.gemm(fmt, act, packed, M)
    torch.cuda.synchronize()
    R.assert_parity(y, R.dense_ref(inp), f"mxfp4 x mxfp4 M={M}")


@pytest.mark.parametrize("path", ["indexed", "grouped"])
@pytest.mark.parametrize("T", [5, 60, 300])
def test_mxfp4_act_moe_parity(lib, monkeypatch, path, T):
    monkeypatch.setenv("HQ_MOE_PATH", path)
    inp = make_moe(dict(MX4, kind="moe", topk=3), T, seed=T + 1, E=6, N=256, K=1024, topk=3)
    fmt, packed = lib.pack_inputs(inp, "cuda")
    act = {k: v.cuda() for k, v in inp["a"].items()}
    y = lib.moe_gemm(fmt, act, packed, inp["ids"].cuda(), inp["topk_w"].cuda())
    torch.cuda.synchronize()
    R.assert_parity(y, R.moe_ref(inp), f"moe mxfp4 x mxfp4 {path} T={T}")


def test_mxfp4_act_exact_pow2_bit_exact(lib):
    """e2m1 on both sides with power-of-two block scales: every partial sum is exact in fp32, so C equals the bf16
    rounding of the exact result bit for bit."""
    gen = torch.Generator().manual_seed(17)
    M, N, K = 24, 256, 1024
    jw = torch.randint(-1, 2, (N, K // 32), generator=gen)
    ja = torch.randint(-2, 2, (M, K // 32), generator=gen)
    inp = dict(M=M, N=N, K=K, wfmt="mxfp4", afmt="mxfp4", G=32,
               w=dict(codes=torch.randint(0, 256, (N, K // 2), generator=gen, dtype=torch.uint8),
                      scales=(jw + 127).to(torch.uint8)),
               a=dict(data=torch.randint(0, 256, (M, K // 2), generator=gen, dtype=torch.uint8),
                      scale=(ja + 127).to(torch.uint8)))
    fmt, packed = lib.pack_inputs(inp, "cuda")
    y = lib.gemm(fmt, {k: v.cuda() for k, v in inp["a"].items()}, packed, M)
    torch.cuda.synchronize()
    ref = R.dense_ref(inp)
    assert np.max(np.abs(ref)) < 2 ** 20
    assert torch.equal(y.cpu(), torch.from_numpy(np.asarray(ref, dtype=np.float32)).to(torch.bfloat16))


def test_mxfp4_act_needs_k_multiple_of_512(lib):
    fmt = lib.make_format("mxfp4", 256, 640, act_type=lib.HQ_A_MXFP4)
    assert lib.packed_bytes(fmt) == 0
