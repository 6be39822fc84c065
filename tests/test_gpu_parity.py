"""CUDA path against the CPU oracle through the C ABI (GPU).

Small cases span several 128-row weight tiles, several K stages and ragged
token / N tails and are compared element by element; full workload sizes are
compared on sampled output rows.
"""
import numpy as np
import pytest
import torch

from tests import ref_helpers as R
from workload import make_dense, make_moe, quant
from workload import configs as W

pytestmark = pytest.mark.gpu

DENSE_FORMS = {
    "int4_sym": dict(kind="dense", wfmt="int4_sym", afmt="bf16", G=128),
    "uint4_zp": dict(kind="dense", wfmt="uint4_zp", afmt="bf16", G=128),
    "nvfp4": dict(kind="dense", wfmt="nvfp4", afmt="nvfp4", G=16),
    "mxfp4": dict(kind="dense", wfmt="mxfp4", afmt="e4m3_tok", G=32),
}
MOE_FORMS = {
    "int4_sym": dict(kind="moe", wfmt="int4_sym", afmt="bf16", G=128, topk=3),
    "mxfp4": dict(kind="moe", wfmt="mxfp4", afmt="e4m3_tok", G=32, topk=3),
    "nvfp4": dict(kind="moe", wfmt="nvfp4", afmt="nvfp4", G=16, topk=3),
    "uint4_zp": dict(kind="moe", wfmt="uint4_zp", afmt="bf16", G=128, topk=3),
}


def _k_for(wfmt):
    return 768 if wfmt == "nvfp4" else 640


def _run_dense(lib, inp):
    fmt, packed = lib.pack_inputs(inp, "cuda")
    act = {k: v.cuda() for k, v in inp["a"].items()}
    bias = inp["bias"].cuda() if inp.get("bias") is not None else None
    y = lib.gemm(fmt, act, packed, inp["M"], bias=bias)
    torch.cuda.synchronize()
    return y


def _run_moe(lib, inp, ws=None):
    fmt, packed = lib.pack_inputs(inp, "cuda")
    act = {k: v.cuda() for k, v in inp["a"].items()}
    y = lib.moe_gemm(fmt, act, packed, inp["ids"].cuda(), inp["topk_w"].cuda(), workspace=ws)
    torch.cuda.synchronize()
    return y


# ------------------------------------------------------------------ repack
@pytest.mark.parametrize("wfmt", ["int4_sym", "uint4_zp", "nvfp4", "mxfp4"])
def test_pack_unpack_round_trip_bit_exact(lib, wfmt):
    E, N, K = 3, 300, 512
    g = {"int4_sym": 128, "uint4_zp": 128, "nvfp4": 16, "mxfp4": 32}[wfmt]
    gen = torch.Generator().manual_seed(11)
    codes = torch.randint(0, 256, (E, N, K // 2), generator=gen, dtype=torch.uint8)
    if wfmt in ("int4_sym", "uint4_zp"):
        scales = torch.randint(0, 65536, (E, N, K // g), generator=gen, dtype=torch.int32).to(torch.int16).view(torch.uint8)
        scales = scales.reshape(E, N, 2 * (K // g))
    else:
        scales = torch.randint(0, 256, (E, N, K // g), generator=gen, dtype=torch.uint8)
    zeros = torch.randint(0, 16, (E, N, K // g), generator=gen, dtype=torch.uint8) if wfmt == "uint4_zp" else None
    gscale = torch.rand(E, generator=gen) if wfmt == "nvfp4" else None
    fmt = lib.make_format(wfmt, N, K, E)
    dev = lambda t: None if t is None else t.cuda()
    packed = lib.pack_weights(fmt, dev(codes), dev(scales), dev(zeros), dev(gscale))
    c2 = torch.zeros_like(codes).cuda()
    s2 = torch.zeros_like(scales).cuda()
    z2 = torch.zeros_like(zeros).cuda() if zeros is not None else None
    g2 = torch.zeros_like(gscale).cuda() if gscale is not None else None
    lib.unpack_weights(fmt, packed, c2, s2, z2, g2)
    torch.cuda.synchronize()
    assert torch.equal(c2.cpu(), codes)
    assert torch.equal(s2.cpu(), scales)
    if zeros is not None:
        assert torch.equal(z2.cpu(), zeros)
    if gscale is not None:
        assert torch.equal(g2.cpu(), gscale)
    assert packed.numel() == lib.packed_bytes(fmt)


# ------------------------------------------------------------------ dense, element by element
@pytest.mark.parametrize("wfmt", list(DENSE_FORMS))
@pytest.mark.parametrize("M", [1, 13, 16, 40, 64, 100, 200, 300])
def test_dense_parity_small(lib, wfmt, M):
    inp = make_dense(DENSE_FORMS[wfmt], M, seed=M, N=320, K=_k_for(wfmt), with_bias=wfmt in ("int4_sym", "uint4_zp"))
    y = _run_dense(lib, inp)
    R.assert_parity(y, R.dense_ref(inp), f"{wfmt} M={M}")


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_dense_seeds(lib, seed):
    inp = make_dense("w4a16_sym", 8, seed=seed)
    R.assert_parity(_run_dense(lib, inp), R.dense_ref(inp), f"w4a16_sym seed {seed}")


# ------------------------------------------------------------------ MoE, element by element
@pytest.mark.parametrize("wfmt", list(MOE_FORMS))
@pytest.mark.parametrize("T", [1, 5, 40, 200])
def test_moe_parity_small(lib, wfmt, T):
    inp = make_moe(MOE_FORMS[wfmt], T, seed=T, E=8, N=256, K=_k_for(wfmt) - 128 if wfmt != "nvfp4" else 512, topk=3)
    y = _run_moe(lib, inp)
    R.assert_parity(y, R.moe_ref(inp), f"moe {wfmt} T={T}")


def test_moe_one_expert_equals_dense(lib):
    """E = 1, top-1, unit weights: the MoE call reproduces the dense call bit for bit."""
    inp = make_dense("w4a16_sym", 37, seed=3, N=256, K=512)
    fmt, packed = lib.pack_inputs(inp, "cuda")
    act = {k: v.cuda() for k, v in inp["a"].items()}
    yd = lib.gemm(fmt, act, packed, 37)
    ids = torch.zeros(37, 1, dtype=torch.int32, device="cuda")
    ym = lib.moe_gemm(fmt, act, packed, ids, torch.ones(37, 1, device="cuda"))
    torch.cuda.synchronize()
    assert torch.equal(yd, ym)


# ------------------------------------------------------------------ exact arithmetic
def _bf16_rne(x):
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)


@pytest.mark.parametrize("wfmt", list(DENSE_FORMS))
def test_exact_integer_pow2_bit_exact(lib, wfmt):
    """Integer-valued operands, power-of-two scales: every partial sum is exact in fp32, so C = bf16(exact)."""
    gen = torch.Generator().manual_seed(5)
    M, N, K = 24, 256, 512
    f = DENSE_FORMS[wfmt]
    inp = dict(M=M, N=N, K=K, wfmt=wfmt, afmt=f["afmt"], G=f["G"])
    codes = torch.randint(0, 256, (N, K // 2), generator=gen, dtype=torch.uint8)
    G = f["G"]
    if wfmt == "int4_sym":
        q = torch.randint(-7, 8, (N, K), generator=gen)
        codes = quant.pack_nibbles((q & 0xF).to(torch.uint8))
        j = torch.randint(-3, 1, (N, K // G), generator=gen)
        scales = ((j + 127) << 7).to(torch.int16).view(torch.bfloat16)
        w = dict(codes=codes, scales=scales)
    elif wfmt == "uint4_zp":
        j = torch.randint(-3, 1, (N, K // G), generator=gen)
        scales = ((j + 127) << 7).to(torch.int16).view(torch.bfloat16)
        w = dict(codes=codes, scales=scales, zeros=torch.randint(0, 16, (N, K // G), generator=gen, dtype=torch.uint8))
    elif wfmt == "nvfp4":
        j = torch.randint(-2, 3, (N, K // 16), generator=gen)
        w = dict(codes=codes, scales=((j + 7) << 3).to(torch.uint8), gscale=torch.tensor([1.0]))
    else:
        j = torch.randint(-1, 2, (N, K // 32), generator=gen)
        w = dict(codes=codes, scales=(j + 127).to(torch.uint8))
    inp["w"] = w
    if f["afmt"] == "bf16":
        a = torch.randint(-3, 4, (M, K), generator=gen).to(torch.bfloat16)
        inp["a"] = dict(data=a)
    elif f["afmt"] == "nvfp4":
        ja = torch.randint(-2, 2, (M, K // 16), generator=gen)
        inp["a"] = dict(data=torch.randint(0, 256, (M, K // 2), generator=gen, dtype=torch.uint8),
                        scale=((ja + 7) << 3).to(torch.uint8), gscale=torch.tensor([0.5]))
    else:
        # e4m3 with exponent field 6..8 (|a| in [0.5, 4)): every partial sum stays exact in fp32
        sgn = torch.randint(0, 2, (M, K), generator=gen) << 7
        ex = torch.randint(6, 9, (M, K), generator=gen) << 3
        a8 = (sgn | ex | torch.randint(0, 8, (M, K), generator=gen)).to(torch.uint8)
        st = torch.pow(2.0, torch.randint(-2, 2, (M,), generator=gen).float())
        inp["a"] = dict(data=a8, scale=st)
    y = _run_dense(lib, inp)
    ref = R.dense_ref(inp)
    assert np.max(np.abs(ref)) < 2 ** 20
    assert torch.equal(y.cpu(), _bf16_rne(ref)), "not bit-exact"


# ------------------------------------------------------------------ edge cases and errors
def test_zero_rows_is_a_no_op(lib):
    inp = make_dense("w4a16_sym", 1, N=128, K=256)
    fmt, packed = lib.pack_inputs(inp, "cuda")
    out = torch.full((0, 128), 7.0, dtype=torch.bfloat16, device="cuda")
    lib.gemm(fmt, {"data": inp["a"]["data"].cuda()}, packed, 0, out=out)


def test_host_errors(lib):
    inp = make_dense("w4a16_sym", 4, N=128, K=256)
    fmt, packed = lib.pack_inputs(inp, "cuda")
    a = inp["a"]["data"].cuda()
    bad = lib.make_format("int4_sym", 128, 256, group_size=64)
    with pytest.raises(lib.HQError) as e:
        lib.gemm(bad, {"data": a}, packed, 4, workspace=torch.zeros(1 << 20, dtype=torch.uint8, device="cuda"))
    assert e.value.code == lib.HQ_ERR_UNSUPPORTED
    bad = lib.make_format("int4_sym", 128, 200)
    assert lib.packed_bytes(bad) == 0
    with pytest.raises(lib.HQError) as e:
        lib.gemm(fmt, {"data": a}, packed, 4, workspace=torch.zeros(16, dtype=torch.uint8, device="cuda"))
    assert e.value.code == lib.HQ_ERR_WORKSPACE
    buf = torch.zeros(4 * 256 * 2 + 2, dtype=torch.uint8, device="cuda")
    mis = buf[2:].view(torch.bfloat16).view(4, 256)
    with pytest.raises(lib.HQError) as e:
        lib.gemm(fmt, {"data": mis}, packed, 4)
    assert e.value.code == lib.HQ_ERR_ALIGNMENT


def test_bad_routing_is_reported_and_other_rows_correct(lib):
    inp = make_moe(MOE_FORMS["int4_sym"], 6, seed=4, E=8, N=128, K=256, topk=2)
    inp["ids"][2, 1] = 9  # out of range
    fmt, packed = lib.pack_inputs(inp, "cuda")
    ws = lib.make_workspace(fmt, 6, 2)
    act = {k: v.cuda() for k, v in inp["a"].items()}
    y = lib.moe_gemm(fmt, act, packed, inp["ids"].cuda(), inp["topk_w"].cuda(), workspace=ws)
    assert lib.last_device_status(ws) == lib.HQ_ERR_BAD_ROUTING
    assert lib.last_device_status(ws) == lib.HQ_OK  # reading clears it
    ref = R.moe_ref(inp)
    good = [r for r in range(12) if r != 2 * 2 + 1]
    R.assert_parity(y[good], ref[good], "rows with valid ids")


def test_workspace_is_reusable_across_calls(lib):
    inp = make_dense("w4a16_asym", 3, seed=9, N=1024, K=2048)
    fmt, packed = lib.pack_inputs(inp, "cuda")
    act = {"data": inp["a"]["data"].cuda()}
    ws = lib.make_workspace(fmt, 3)
    y1 = lib.gemm(fmt, act, packed, 3, workspace=ws)
    y2 = lib.gemm(fmt, act, packed, 3, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)
    assert lib.last_device_status(ws) == lib.HQ_OK


# ------------------------------------------------------------------ both INT4 kernels on the same inputs
@pytest.mark.parametrize("path", ["small", "umma"])
@pytest.mark.parametrize("wfmt", ["int4_sym", "uint4_zp"])
@pytest.mark.parametrize("M", [1, 8, 16, 24, 32, 40, 64])
def test_int4_kernels_forced(lib, monkeypatch, path, wfmt, M):
    """HQ_FORCE_PATH selects the register-decode mma.sync kernel or the UMMA kernel; both must match the oracle."""
    monkeypatch.setenv("HQ_FORCE_PATH", path)
    inp = make_dense(DENSE_FORMS[wfmt], M, seed=100 + M, N=384, K=1024, with_bias=True)
    R.assert_parity(_run_dense(lib, inp), R.dense_ref(inp), f"{wfmt} M={M} path={path}")


@pytest.mark.parametrize("path", ["small", "umma"])
@pytest.mark.parametrize("T", [1, 9, 70])
def test_int4_moe_kernels_forced(lib, monkeypatch, path, T):
    monkeypatch.setenv("HQ_FORCE_PATH", path)
    inp = make_moe(MOE_FORMS["int4_sym"], T, seed=T, E=16, N=256, K=512, topk=4)
    R.assert_parity(_run_moe(lib, inp), R.moe_ref(inp), f"moe T={T} path={path}")


def test_int4_kernels_agree_exactly_on_integer_inputs(lib, monkeypatch):
    """Integer codes and activations with power-of-two scales: both kernels give identical bits."""
    gen = torch.Generator().manual_seed(21)
    M, N, K = 16, 256, 512
    q = torch.randint(-7, 8, (N, K), generator=gen)
    j = torch.randint(-3, 1, (N, K // 128), generator=gen)
    inp = dict(M=M, N=N, K=K, wfmt="int4_sym", afmt="bf16", G=128,
               w=dict(codes=quant.pack_nibbles((q & 0xF).to(torch.uint8)),
                      scales=((j + 127) << 7).to(torch.int16).view(torch.bfloat16)),
               a=dict(data=torch.randint(-3, 4, (M, K), generator=gen).to(torch.bfloat16)))
    outs = []
    for path in ("small", "umma"):
        monkeypatch.setenv("HQ_FORCE_PATH", path)
        outs.append(_run_dense(lib, inp).cpu())
    assert torch.equal(outs[0], outs[1])
    assert torch.equal(outs[0], _bf16_rne(R.dense_ref(inp)))


# ------------------------------------------------------------------ MoE: indexed (gather4) and grouped (permuted) paths
@pytest.mark.parametrize("moe_path", ["indexed", "grouped"])
@pytest.mark.parametrize("wfmt", list(MOE_FORMS))
@pytest.mark.parametrize("T", [3, 150])
def test_moe_activation_paths(lib, monkeypatch, moe_path, wfmt, T):
    """HQ_MOE_PATH forces the row gather (Indexed) or the expert-contiguous copy (Grouped); both match the oracle."""
    monkeypatch.setenv("HQ_MOE_PATH", moe_path)
    inp = make_moe(MOE_FORMS[wfmt], T, seed=7 + T, E=6, N=256, K=512, topk=3)
    R.assert_parity(_run_moe(lib, inp), R.moe_ref(inp), f"moe {wfmt} T={T} {moe_path}")


def test_moe_grouped_wide_tiles_match_indexed(lib, monkeypatch):
    """Wide token tiles (200 rows per expert) through both activation paths give the same bits."""
    inp = make_moe(MOE_FORMS["int4_sym"], 400, seed=9, E=4, N=256, K=512, topk=2)
    outs = []
    for moe_path in ("indexed", "grouped"):
        monkeypatch.setenv("HQ_MOE_PATH", moe_path)
        outs.append(_run_moe(lib, inp).cpu())
    assert torch.equal(outs[0], outs[1])
    R.assert_parity(outs[1], R.moe_ref(inp), "grouped wide tiles")


@pytest.mark.parametrize("moe_path", ["indexed", "grouped"])
def test_moe_mxfp4_256_token_tiles(lib, monkeypatch, moe_path):
    """More than 128 routed rows per expert take MXFP4's 256-token tiles (wide tiles with per-row tables)."""
    monkeypatch.setenv("HQ_MOE_PATH", moe_path)
    inp = make_moe(MOE_FORMS["mxfp4"], 300, seed=11, E=4, N=256, K=512, topk=2)
    R.assert_parity(_run_moe(lib, inp), R.moe_ref(inp), f"moe mxfp4 256-token tiles {moe_path}")


# ------------------------------------------------------------------ code and scale bit patterns, odd N, degenerate groups
def _random_bits(inp, seed):
    """Replace the weight codes, scales (and zeros) and the quantized activations of a dense input by random valid
    bit patterns covering each format's whole code range and a wide scale range (NaN encodings excluded)."""
    g = torch.Generator().manual_seed(seed)
    w = inp["w"]
    w["codes"] = torch.randint(0, 256, w["codes"].shape, generator=g, dtype=torch.int32).to(torch.uint8)
    if inp["wfmt"] in ("int4_sym", "uint4_zp"):
        mag = torch.randn(w["scales"].shape, generator=g) * torch.exp2(torch.randint(-12, 4, w["scales"].shape, generator=g).float())
        w["scales"] = mag.to(torch.bfloat16)
        if "zeros" in w:
            w["zeros"] = torch.randint(0, 16, w["zeros"].shape, generator=g, dtype=torch.int32).to(torch.uint8)
    elif inp["wfmt"] == "nvfp4":
        w["scales"] = torch.randint(1, 0x7F, w["scales"].shape, generator=g, dtype=torch.int32).to(torch.uint8)
    else:  # mxfp4: e8m0 2^-30 .. 2^30
        w["scales"] = torch.randint(97, 158, w["scales"].shape, generator=g, dtype=torch.int32).to(torch.uint8)
    a = inp["a"]
    if inp["afmt"] == "e4m3_tok":
        b = torch.randint(0, 256, a["data"].shape, generator=g, dtype=torch.int32).to(torch.uint8)
        b[(b & 0x7F) == 0x7F] = 0x3C  # no NaN
        a["data"] = b
        a["scale"] = torch.rand(a["scale"].shape, generator=g) * 4 + 0.01
    elif inp["afmt"] == "nvfp4":
        a["data"] = torch.randint(0, 256, a["data"].shape, generator=g, dtype=torch.int32).to(torch.uint8)
        a["scale"] = torch.randint(1, 0x7F, a["scale"].shape, generator=g, dtype=torch.int32).to(torch.uint8)
    return inp


@pytest.mark.parametrize("wfmt", list(DENSE_FORMS))
@pytest.mark.parametrize("M", [7, 40, 300])
def test_dense_random_bit_patterns(lib, wfmt, M):
    """Every code value and a wide range of scale exponents (ue4m3 subnormals included) decode as the oracle does.

    FP4 operands enter the MMA exactly, so the general parity bound applies.  INT4 weights enter as bf16((q - z) * s),
    one rounding of the exact weight (relative error at most 2^-9), accumulated in fp32 and rounded once to bf16: the
    bound is then 2^-9 * sum_k |a_k w_k| + 2^-8 * |y| (+ fp32 accumulation), taken from the oracle's exact operands.
    Random scales spanning 2^-12 .. 2^4 make the general bound too tight for that rounding; a decode error (a wrong
    code, zero point or scale) is of the size of the weight itself and fails either bound."""
    inp = make_dense(DENSE_FORMS[wfmt], M, seed=M, N=264, K=512)
    inp = _random_bits(inp, seed=1000 + M)
    y = _run_dense(lib, inp)
    ref = np.asarray(R.dense_ref(inp))
    if wfmt in ("int4_sym", "uint4_zp"):
        s_abs = np.abs(np.asarray(R.acts_of(inp))) @ np.abs(np.asarray(R.weights_of(inp))).T
        bound = 2.0**-9 * s_abs * 1.01 + 2.0**-8 * np.abs(ref) + 1e-6 * s_abs
        err = np.abs(y.float().cpu().numpy().astype(np.float64) - ref)
        worst = float(np.max(err / np.maximum(bound, 1e-300)))
        assert worst <= 1.0, f"{wfmt} M={M} random bits: error {worst:.3f} of the bf16-decode bound"
    else:
        R.assert_parity(y, ref, f"{wfmt} M={M} random bits")


@pytest.mark.parametrize("wfmt", list(DENSE_FORMS))
@pytest.mark.parametrize("N", [129, 131])
@pytest.mark.parametrize("M", [5, 300])
def test_dense_odd_n(lib, wfmt, N, M):
    """An odd N leaves a ragged last weight tile and forbids paired 4-byte stores (the per-element path runs)."""
    inp = make_dense(DENSE_FORMS[wfmt], M, seed=N + M, N=N, K=512, with_bias=wfmt in ("int4_sym", "uint4_zp"))
    R.assert_parity(_run_dense(lib, inp), R.dense_ref(inp), f"{wfmt} M={M} N={N}")


@pytest.mark.parametrize("wfmt", ["int4_sym", "uint4_zp"])
def test_degenerate_groups(lib, wfmt):
    """All-zero and constant weight groups quantize to zero scale (and zero point); the rest of the row is unaffected."""
    c = DENSE_FORMS[wfmt]
    w = W.weights_fp32(3, 1, 256, 512)
    w[:, 0:128] = 0.0
    w[:64, 128:256] = 0.75
    inp = make_dense(c, 24, seed=3, N=256, K=512)
    inp["w"] = W.quantize_weights(c["wfmt"], w, c["G"])
    assert float(inp["w"]["scales"].float()[:, 0].abs().max()) == 0.0
    R.assert_parity(_run_dense(lib, inp), R.dense_ref(inp), f"{wfmt} degenerate groups")


@pytest.mark.parametrize("route", ["fused", "kernel"])
@pytest.mark.parametrize("T", [1, 4, 5, 60])
def test_moe_small_routing_in_kernel_and_by_routing_kernel(lib, monkeypatch, route, T):
    """Small MoE calls (at most 512 routed rows) route inside the register-decode kernel: every CTA builds the same
    per-expert row lists in shared memory (one warp up to 32 routed rows: T = 1, 4; a histogram beyond: T = 5, 60).
    Both that and the separate routing kernel match the oracle."""
    if route == "kernel":
        monkeypatch.setenv("HQ_ROUTE_KERNEL", "1")
    inp = make_moe(MOE_FORMS["int4_sym"], T, seed=T + 40, E=64, N=384, K=1024, topk=8)  # <= 16 rows per expert
    fmt, packed = lib.pack_inputs(inp, "cuda")
    assert lib.kernels_per_call(fmt, T, 8, moe=True) == (1 if route == "fused" else 2)
    R.assert_parity(_run_moe(lib, inp), R.moe_ref(inp), f"moe routing {route} T={T}")


def test_int4_tcgen05_rounding_witness(lib):
    """The tcgen05 INT4 path feeds the MMA bf16((q - z) * s): one rounding per weight, shared by every weight of a
    group with the same code.  On this workload-recipe input (MoE INT4, T = 200, E = 8, K = 640, seed 4) that
    rounding takes one element to 1.087 of the general element-wise bound (a CPU emulation of the arithmetic gives
    the same value bit for bit; exact weights give 0.315).  The path is held here to the rigorous bound of its own
    arithmetic, 2^-9 sum_k |a_k w_k| + 2^-8 |y_ref| (+ fp32 accumulation), which any decode error (a wrong code,
    zero point or scale, of the size of the weight itself) would break."""
    from tests import debug_bounds_cases as D

    c = D.moe_case("witness", "int4_sym", 200, 8, 256, 640)
    assert c["plan"]["kernel"] == "umma" and c["bound"] == "bf16-decode", c["plan"]
    assert c["status"] == lib.HQ_OK, lib.status_string(c["status"])
    assert c["ratio"] <= 1.0, f"{c['ratio']:.3f} of the bf16-decode bound"
