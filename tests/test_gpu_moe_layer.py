"""The MoE layer pieces around the grouped GEMMs on the GPU against the CPU oracle: the Down GEMM with the top-k
combine fused into its epilogue, and the gated activation (SwiGLU) between Gate-up and Down."""
import numpy as np
import pytest
import torch

import oracle
from tests import ref_helpers as R
from workload import configs as W

pytestmark = pytest.mark.gpu

FORMS = {
    "int4_sym": dict(kind="moe", wfmt="int4_sym", afmt="bf16", G=128),
    "uint4_zp": dict(kind="moe", wfmt="uint4_zp", afmt="bf16", G=128),
    "nvfp4": dict(kind="moe", wfmt="nvfp4", afmt="nvfp4", G=16),
    "mxfp4": dict(kind="moe", wfmt="mxfp4", afmt="e4m3_tok", G=32),
    "mxfp4_mx": dict(kind="moe", wfmt="mxfp4", afmt="mxfp4", G=32),  # MXFP4 x MXFP4 (K a multiple of 512)
}


def _down_case(wfmt, T, topk=3, E=5, N=264, K=None, seed=0):
    """Expert weights, routing and the T*topk routed activation rows (quantized to the format's activation type)."""
    c = dict(FORMS[wfmt], topk=topk)
    K = K or {"nvfp4": 768, "mxfp4_mx": 1024}.get(wfmt, 640)
    inp = W.make_moe(c, T, seed=seed, E=E, N=N, K=K, topk=topk)
    rows = W.acts_fp32(seed + 7, T * topk, K, outliers=c["afmt"] == "nvfp4")
    inp["a"] = W.quantize_acts(c["afmt"], rows)
    return inp


def _run_combine(lib, inp, tw=True):
    fmt, packed = lib.pack_inputs(inp, "cuda")
    act = {k: v.cuda() for k, v in inp["a"].items()}
    ws = lib.make_combine_workspace(fmt, inp["T"], inp["topk"])
    y = lib.moe_gemm_combine(fmt, act, packed, inp["ids"].cuda(), inp["topk_w"].cuda() if tw else None,
                             workspace=ws)
    torch.cuda.synchronize()
    return y, ws


def _combine_ref(inp, tw=True, tokens=None):
    cache = {}

    def w_of(e):
        if e < 0 or e >= inp["E"]:
            return None
        if e not in cache:
            cache[e] = R.weights_of(inp, e)
        return cache[e]

    return oracle.moe_combine(R.acts_of(inp), w_of, inp["N"], inp["ids"].cpu().numpy(),
                              inp["topk_w"].cpu().numpy() if tw else None, tokens)


@pytest.mark.parametrize("wfmt", list(FORMS))
@pytest.mark.parametrize("T", [1, 37, 300])
def test_combine_parity(lib, wfmt, T):
    inp = _down_case(wfmt, T)
    y, ws = _run_combine(lib, inp)
    assert lib.last_device_status(ws) == 0
    R.assert_parity(y, _combine_ref(inp), f"combine {wfmt} T={T}")


@pytest.mark.parametrize("path", ["indexed", "grouped"])
@pytest.mark.parametrize("wfmt", ["int4_sym", "mxfp4", "nvfp4"])
def test_combine_paths(lib, monkeypatch, path, wfmt):
    monkeypatch.setenv("HQ_MOE_PATH", path)
    inp = _down_case(wfmt, 90, topk=4, E=6, seed=2)
    y, _ = _run_combine(lib, inp)
    R.assert_parity(y, _combine_ref(inp), f"combine {wfmt} {path}")


@pytest.mark.parametrize("path", ["small", "umma"])
def test_combine_int4_kernels(lib, monkeypatch, path):
    monkeypatch.setenv("HQ_FORCE_PATH", path)
    inp = _down_case("uint4_zp", 21, topk=2, E=4, seed=3)
    y, _ = _run_combine(lib, inp)
    R.assert_parity(y, _combine_ref(inp), f"combine uint4 {path}")


def test_combine_without_weights_and_with_a_bad_id(lib):
    inp = _down_case("int4_sym", 16, topk=2, E=4, seed=4)
    y, _ = _run_combine(lib, inp, tw=False)
    R.assert_parity(y, _combine_ref(inp, tw=False), "combine, unit weights")
    inp["ids"][3, 1] = 99  # out of range: that routed row adds nothing, the status records it
    y, ws = _run_combine(lib, inp)
    assert lib.last_device_status(ws) == lib.HQ_ERR_BAD_ROUTING
    R.assert_parity(y, _combine_ref(inp), "combine with a bad id")


def test_combine_rejects_odd_n_and_small_workspace(lib):
    inp = _down_case("int4_sym", 4, topk=2, E=3, N=130, seed=5)
    fmt, packed = lib.pack_inputs(inp, "cuda")
    act = {k: v.cuda() for k, v in inp["a"].items()}
    with pytest.raises(lib.HQError) as e:
        lib.moe_gemm_combine(fmt, act, packed, inp["ids"].cuda(), inp["topk_w"].cuda(),
                             workspace=torch.zeros(1 << 20, dtype=torch.uint8, device="cuda"))
    assert e.value.code == lib.HQ_ERR_ALIGNMENT
    inp = _down_case("int4_sym", 4, topk=2, E=3, seed=5)
    fmt, packed = lib.pack_inputs(inp, "cuda")
    act = {k: v.cuda() for k, v in inp["a"].items()}
    with pytest.raises(lib.HQError) as e:
        lib.moe_gemm_combine(fmt, act, packed, inp["ids"].cuda(), inp["topk_w"].cuda(),
                             workspace=torch.zeros(256, dtype=torch.uint8, device="cuda"))
    assert e.value.code == lib.HQ_ERR_WORKSPACE


@pytest.mark.parametrize("wfmt,E,N,K", [("int4_sym", 128, 2048, 768), ("mxfp4", 256, 7168, 2048)])
def test_combine_full_size_sampled_tokens(lib, wfmt, E, N, K):
    """Down-GEMM shapes of the MoE workloads (hidden N, intermediate K), T = 512 tokens, top-8: sampled tokens
    against the oracle; only the experts those tokens use are generated (the others stay zero and unused)."""
    T, topk = 512, 8
    c = dict(FORMS[wfmt], topk=topk)
    ids, _ = W.zipf_route(0, T, E, topk)
    toks = [0, 1, 255, 511]
    used = sorted({int(e) for t in toks for e in ids[t]})
    inp = W.make_moe(c, T, seed=0, E=E, N=N, K=K, topk=topk, experts_subset=used)
    inp["a"] = W.quantize_acts(c["afmt"], W.acts_fp32(9, T * topk, K))
    y, ws = _run_combine(lib, inp)
    assert lib.last_device_status(ws) == 0
    R.assert_parity(y[toks], _combine_ref(inp, tokens=toks), f"combine {wfmt} full size")


@pytest.mark.parametrize("R_,I", [(1, 8), (37, 264), (300, 768)])
def test_swiglu(lib, R_, I):
    g = torch.Generator().manual_seed(R_ + I)
    x = (torch.randn(R_, 2 * I, generator=g) * 4).to(torch.bfloat16)
    x[0, :4] = torch.tensor([0.0, -100.0, 100.0, -0.0])
    y = lib.swiglu(x.cuda())
    torch.cuda.synchronize()
    ref = oracle.swiglu((R.np_bits(x).astype(np.uint32) << 16).view(np.float32))
    got = y.float().cpu().double().numpy()
    # fp32 arithmetic and one round to nearest-even bf16: within 2^-8 relative (bf16 half-ulp 2^-9, plus fp32)
    assert np.all(np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-30), np.max(np.abs(got - ref) / (np.abs(ref) + 1e-30))


@pytest.mark.parametrize("wfmt", ["int4_sym", "mxfp4"])
def test_moe_layer_chain(lib, wfmt):
    """Gate-up GEMM (unweighted routed rows) -> SwiGLU -> quantization of the activation for the Down GEMM's format
    -> Down GEMM with combine; each stage against the oracle applied to the previous stage's device output, and the
    chain against the float64 oracle chain."""
    T, topk, E, H, Ih = 40, 2, 4, 512, 256  # hidden H, intermediate Ih (gate-up N = 2 Ih)
    c = dict(FORMS[wfmt], topk=topk)
    gu = W.make_moe(c, T, seed=11, E=E, N=2 * Ih, K=H, topk=topk)
    dn = W.make_moe(c, T, seed=12, E=E, N=H, K=Ih, topk=topk)
    dn["ids"], dn["topk_w"] = gu["ids"], gu["topk_w"]
    fmt_gu, p_gu = lib.pack_inputs(gu, "cuda")
    fmt_dn, p_dn = lib.pack_inputs(dn, "cuda")
    ids = gu["ids"].cuda()
    h = lib.moe_gemm(fmt_gu, {k: v.cuda() for k, v in gu["a"].items()}, p_gu, ids, None)
    s = lib.swiglu(h)
    if c["afmt"] == "bf16":
        act = dict(data=s)
    else:
        act = lib.quantize_act(c["afmt"], s)
    y = lib.moe_gemm_combine(fmt_dn, act, p_dn, ids, gu["topk_w"].cuda())
    torch.cuda.synchronize()
    # stage by stage
    w_gu = {e: R.weights_of(gu, e) for e in range(E)}
    w_dn = {e: R.weights_of(dn, e) for e in range(E)}
    h_ref = oracle.moe_gemm(R.acts_of(gu), lambda e: w_gu[e], 2 * Ih, gu["ids"].numpy())
    R.assert_parity(h, h_ref, "gate-up")
    h_dev = R.np_bits(h).astype(np.uint32) << 16
    s_ref = oracle.swiglu(h_dev.view(np.float32))
    got = s.float().cpu().double().numpy()
    assert np.all(np.abs(got - s_ref) <= 2.0 ** -8 * np.abs(s_ref) + 1e-30)
    if c["afmt"] == "bf16":
        a_dn = oracle.decode_bf16(R.np_bits(s))
    else:
        q, sc = oracle.quantize_act_e4m3_per_token(R.np_bits(s))
        assert np.array_equal(act["data"].cpu().numpy(), q)
        a_dn = oracle.dequant_acts("e4m3_tok", q, sc)
    y_ref = oracle.moe_combine(a_dn, lambda e: w_dn[e], H, gu["ids"].numpy(), gu["topk_w"].numpy())
    R.assert_parity(y, y_ref, "down + combine")
    # whole chain in float64 (no intermediate rounding or activation quantization on the oracle side): looser, the
    # device rounds h and s to bf16 and, for W4A8, quantizes s to e4m3
    chain = oracle.moe_combine(oracle.swiglu(h_ref), lambda e: w_dn[e], H, gu["ids"].numpy(), gu["topk_w"].numpy())
    err = np.abs(y.float().cpu().double().numpy() - chain)
    rms = float(np.sqrt(np.mean(chain ** 2)))
    tol = 0.02 if c["afmt"] == "bf16" else 0.15
    assert np.max(err) <= tol * rms * 10 and np.sqrt(np.mean(err ** 2)) <= tol * rms
