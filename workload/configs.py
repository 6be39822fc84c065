"""The five synthetic workloads of the fused-dequant GEMM benchmark, and their input makers.

Sizes and recipes (quantized GEMM microbenchmarks of the Humming announcement,
"Results: kernel microbenchmarks", plus the workload table of this project):

  w4a16_sym   dense, M=8, K=1024, N=1024, INT4 symmetric group 128, bf16 act
  w4a16_asym  dense, K=4096, N=14336, M in {1,16,64,256,1024,4096,8192},
              UINT4 + zero point group 128, bf16 act
  nvfp4       dense, K=7168, N=4096, M in {1,128,1024,8192}, NVFP4 weights and
              activations (1% of activations x20 outliers before quantization)
  moe_w4a16   MoE, E=128, top-8, K=2048, N=1536, T in {1,32,512,4096},
              INT4 symmetric group 128, bf16 act
  moe_mxfp4   MoE, E=256, top-8, K=7168, N=4096, T in {1,64,1024,8192},
              MXFP4 weights, FP8 e4m3 per-token activations
  w8a16, w2a16, w1a16, w3a16, mxint4_a16, fp8w_a16
              dense, K=4096, N=14336, M in {1,16,64,256}: INT8 (e0m7) g128,
              UINT2 / UINT1 / UINT3 + zero point g128, MXINT4 (e8m0 per 32),
              FP8 E4M3 g128 weights, bf16 act
  w4a8_mx     dense, K=7168, N=4096, M in {1,128,1024,8192}: MXFP4 weights,
              MXFP8 activations (e4m3 + e8m0 per 32)
  w4a4_mx     the same with MXFP4 activations (e2m1 + e8m0 per 32)

Weights are fp32 N(0, 0.02) and activations N(0, 1) before quantization.  MoE
routing draws k distinct experts per token from Zipf(1.1) popularities by
Gumbel-top-k and softmaxes k N(0,1) logits into the top-k weights.

Each maker returns a dict of torch tensors in the canonical (unpacked-layout)
format, on the requested device.  Stream ids keep tensors independent.
"""
import math

import torch

from . import philox, quant

SID_W, SID_A, SID_OUTLIER, SID_ROUTE, SID_LOGIT, SID_BIAS = 1, 2, 3, 4, 5, 6

CONFIGS = {
    "w4a16_sym": dict(kind="dense", wfmt="int4_sym", afmt="bf16", N=1024, K=1024, G=128, sizes=[8]),
    "w4a16_asym": dict(kind="dense", wfmt="uint4_zp", afmt="bf16", N=14336, K=4096, G=128,
                       sizes=[1, 16, 64, 256, 1024, 4096, 8192]),
    "nvfp4": dict(kind="dense", wfmt="nvfp4", afmt="nvfp4", N=4096, K=7168, G=16, sizes=[1, 128, 1024, 8192]),
    "moe_w4a16": dict(kind="moe", wfmt="int4_sym", afmt="bf16", E=128, topk=8, N=1536, K=2048, G=128,
                      sizes=[1, 32, 512, 4096]),
    "moe_mxfp4": dict(kind="moe", wfmt="mxfp4", afmt="e4m3_tok", E=256, topk=8, N=4096, K=7168, G=32,
                      sizes=[1, 64, 1024, 8192]),
    # more weight formats through the same decode component (the dense W4A16 shape of the sweep above), and the
    # microscaled W4A8 variant (MXFP4 weights x MXFP8 activations) on the NVFP4 shape
    "w8a16": dict(kind="dense", wfmt="int8_sym", afmt="bf16", N=14336, K=4096, G=128, sizes=[1, 16, 64, 256]),
    "w2a16": dict(kind="dense", wfmt="uint2_zp", afmt="bf16", N=14336, K=4096, G=128, sizes=[1, 16, 64, 256]),
    "mxint4_a16": dict(kind="dense", wfmt="mxint4", afmt="bf16", N=14336, K=4096, G=32, sizes=[1, 16, 64, 256]),
    "w1a16": dict(kind="dense", wfmt="uint1_zp", afmt="bf16", N=14336, K=4096, G=128, sizes=[1, 16, 64, 256]),
    "w3a16": dict(kind="dense", wfmt="uint3_zp", afmt="bf16", N=14336, K=4096, G=128, sizes=[1, 16, 64, 256]),
    "fp8w_a16": dict(kind="dense", wfmt="e4m3", afmt="bf16", N=14336, K=4096, G=128, sizes=[1, 16, 64, 256]),
    "w4a4_mx": dict(kind="dense", wfmt="mxfp4", afmt="mxfp4", N=4096, K=7168, G=32, sizes=[1, 128, 1024, 8192]),
    "w4a8_mx": dict(kind="dense", wfmt="mxfp4", afmt="mxfp8", N=4096, K=7168, G=32, sizes=[1, 128, 1024, 8192]),
}
# Down GEMMs of the two MoE workloads' layers (hidden N, intermediate K = half the Gate-up N), with the top-k combine
# fused into the epilogue: the routed rows T*k of K in, T token rows of N out.
CONFIGS["moe_w4a16_down"] = dict(CONFIGS["moe_w4a16"], N=2048, K=768, down=True)
CONFIGS["moe_mxfp4_down"] = dict(CONFIGS["moe_mxfp4"], N=7168, K=2048, down=True)

W_STD = 0.02


def weights_fp32(seed, E, N, K, expert=0, device="cpu"):
    """fp32 N(0, 0.02) weights of one expert, [N, K]; element (e, n, k) is fixed by its index."""
    n_el = N * K
    return (philox.normal(seed, SID_W, n_el, offset=expert * (n_el // 4), device=device) * W_STD).reshape(N, K)


def acts_fp32(seed, M, K, outliers=False, device="cpu"):
    a = philox.normal(seed, SID_A, M * K, device=device).reshape(M, K)
    if outliers:
        u = philox.uniform(seed, SID_OUTLIER, M * K, device=device).reshape(M, K)
        a = torch.where(u < 0.01, a * 20.0, a)
    return a


def quantize_weights(wfmt, w, G):
    """fp32 [..., N, K] -> dict(codes, scales, zeros?, gscale?) in the canonical layout."""
    if wfmt == "int4_sym":
        c, s = quant.quant_int4_sym(w, G)
        return dict(codes=c, scales=s)
    if wfmt == "uint4_zp":
        c, s, z = quant.quant_uint4_zp(w, G)
        return dict(codes=c, scales=s, zeros=z)
    if wfmt == "nvfp4":
        c, s, g = quant.quant_nvfp4(w)
        return dict(codes=c, scales=s, gscale=g.reshape(1))
    if wfmt == "mxfp4":
        c, s = quant.quant_mxfp4(w)
        return dict(codes=c, scales=s)
    if wfmt == "int8_sym":
        c, s = quant.quant_int8_sym(w, G)
        return dict(codes=c, scales=s)
    if wfmt == "uint2_zp":
        c, s, z = quant.quant_uint2_zp(w, G)
        return dict(codes=c, scales=s, zeros=z)
    if wfmt in ("uint1_zp", "uint3_zp"):
        c, s, z = quant.quant_uint_zp(w, G, 1 if wfmt == "uint1_zp" else 3)
        return dict(codes=c, scales=s, zeros=z)
    if wfmt == "mxint4":
        c, s = quant.quant_mxint4(w)
        return dict(codes=c, scales=s)
    if wfmt == "e4m3":
        c, s = quant.quant_e4m3_grouped(w, G)
        return dict(codes=c, scales=s)
    raise ValueError(wfmt)


def quantize_acts(afmt, a):
    if afmt == "bf16":
        return dict(data=a.to(torch.bfloat16).contiguous())
    if afmt == "e4m3_tok":
        q, s = quant.quant_e4m3_per_token(a)
        return dict(data=q, scale=s)
    if afmt == "nvfp4":
        c, s, g = quant.quant_nvfp4(a)
        return dict(data=c, scale=s, gscale=g.reshape(1))
    if afmt == "mxfp8":
        q, s = quant.quant_mxfp8(a)
        return dict(data=q, scale=s)
    if afmt == "mxfp4":
        c, s = quant.quant_mxfp4(a)
        return dict(data=c, scale=s)
    raise ValueError(afmt)


def make_dense(cfg, M, seed=0, device="cpu", N=None, K=None, with_bias=False):
    """Inputs of one dense call: {'w': {...}, 'a': {...}, 'bias'?, 'M','N','K'}; N, K override the config."""
    c = CONFIGS[cfg] if isinstance(cfg, str) else cfg
    N = N or c["N"]
    K = K or c["K"]
    w = weights_fp32(seed, 1, N, K, device=device)
    out = dict(M=M, N=N, K=K, wfmt=c["wfmt"], afmt=c["afmt"], G=c["G"])
    out["w"] = quantize_weights(c["wfmt"], w, c["G"])
    del w
    a = acts_fp32(seed, M, K, outliers=(c["afmt"] == "nvfp4"), device=device)
    out["a"] = quantize_acts(c["afmt"], a)
    if with_bias:
        out["bias"] = philox.normal(seed, SID_BIAS, N, device=device).to(torch.bfloat16)
    return out


def zipf_route(seed, T, E, k, s=1.1, device="cpu"):
    """(topk_ids int32 [T, k], topk_weights fp32 [T, k]).

    Experts are drawn without replacement with popularity p_e ~ (e+1)**-s through
    Gumbel-top-k (argtopk of log p_e + Gumbel noise); equal keys go to the lower id.
    The k weights are a softmax over k N(0, 1) logits, one per selected slot.
    """
    logp = -s * torch.log(torch.arange(1, E + 1, dtype=torch.float64, device=device))
    logp = logp - torch.logsumexp(logp, 0)
    u = philox.uniform(seed, SID_ROUTE, T * E, device=device).reshape(T, E)
    keys = logp.unsqueeze(0) - torch.log(-torch.log(u))
    order = torch.sort(keys, dim=1, descending=True, stable=True).indices
    ids = order[:, :k].to(torch.int32).contiguous()
    logits = philox.normal(seed, SID_LOGIT, T * k, device=device).reshape(T, k).to(torch.float64)
    w = torch.softmax(logits, dim=1).to(torch.float32).contiguous()
    return ids, w


def make_moe(cfg, T, seed=0, device="cpu", E=None, N=None, K=None, topk=None, experts_subset=None):
    """Inputs of one MoE call: {'w': {...} stacked over E, 'a', 'ids', 'topk_w', ...}.

    `experts_subset` (a list of expert ids) generates only those experts' weights
    and leaves the others zero: for sampled checks at full size.
    """
    c = CONFIGS[cfg] if isinstance(cfg, str) else cfg
    E = E or c["E"]
    N = N or c["N"]
    K = K or c["K"]
    topk = topk or c["topk"]
    out = dict(T=T, E=E, N=N, K=K, topk=topk, wfmt=c["wfmt"], afmt=c["afmt"], G=c["G"])
    parts = []
    for e in range(E):
        if experts_subset is not None and e not in experts_subset:
            parts.append(None)
            continue
        parts.append(quantize_weights(c["wfmt"], weights_fp32(seed, E, N, K, expert=e, device=device), c["G"]))
    ref = next(p for p in parts if p is not None)
    stacked = {}
    for key in ref:
        stacked[key] = torch.stack([p[key] if p is not None else torch.zeros_like(ref[key]) for p in parts])
    if "gscale" in stacked:
        stacked["gscale"] = stacked["gscale"].reshape(E)
    out["w"] = stacked
    a = acts_fp32(seed, T, K, device=device)
    out["a"] = quantize_acts(c["afmt"], a)
    out["ids"], out["topk_w"] = zipf_route(seed, T, E, topk, device=device)
    return out


def dense_flops(M, N, K):
    return 2.0 * M * N * K


def weight_bytes(wfmt, N, K, G, experts=1):
    """Canonical bytes of codes + scales + zeros + global scale for `experts` experts."""
    codes = N * K // 2
    if wfmt in ("int8_sym", "e4m3"):
        return experts * (N * K + N * (K // G) * 2)
    if wfmt == "uint2_zp":
        return experts * (N * K // 4 + N * (K // G) * 2 + N * (K // G) // 4)  # zeros are 2-bit values
    if wfmt in ("uint1_zp", "uint3_zp"):
        b = 1 if wfmt == "uint1_zp" else 3
        return experts * (N * K * b // 8 + N * (K // G) * 2 + N * (K // G) * b // 8)  # zeros are b-bit values
    if wfmt == "mxint4":
        return experts * (codes + N * (K // 32))
    if wfmt == "int4_sym":
        sc = N * (K // G) * 2
    elif wfmt == "uint4_zp":
        sc = N * (K // G) * 2 + N * (K // G) // 2  # zeros are 4-bit values
    elif wfmt == "nvfp4":
        sc = N * (K // 16) + 4
    elif wfmt == "mxfp4":
        sc = N * (K // 32)
    else:
        raise ValueError(wfmt)
    return experts * (codes + sc)


def act_bytes(afmt, M, K):
    if afmt == "bf16":
        return M * K * 2
    if afmt == "e4m3_tok":
        return M * K + M * 4
    if afmt == "nvfp4":
        return M * K // 2 + M * K // 16 + 4
    if afmt == "mxfp8":
        return M * K + M * K // 32
    if afmt == "mxfp4":
        return M * K // 2 + M * K // 32
    raise ValueError(afmt)


def ceil_div(a, b):
    return -(-a // b)


__all__ = ["CONFIGS", "make_dense", "make_moe", "zipf_route", "weights_fp32", "acts_fp32",
           "quantize_weights", "quantize_acts", "dense_flops", "weight_bytes", "act_bytes", "math"]
