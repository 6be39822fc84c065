"""Glue between the workload dicts (torch tensors) and the numpy oracle, plus the parity bound."""
import numpy as np
import torch

import oracle

RTOL = 1e-2  # |y - y_ref| <= RTOL * |y_ref| + ATOL_RMS * rms(y_ref), per element
ATOL_RMS = 1e-2


def np_bits(t):
    """bf16 tensor -> uint16 bit patterns; byte tensors -> uint8."""
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def weights_of(inp, expert=None):
    """Decoded fp64 weights [N, K] of one expert (or the dense layer)."""
    w = inp["w"]
    pick = (lambda t: t[expert]) if expert is not None else (lambda t: t)
    g = w.get("gscale")
    if g is not None:
        g = np_bits(g)
        g = g[expert:expert + 1] if expert is not None else g
    return oracle.dequant_weights(inp["wfmt"], np_bits(pick(w["codes"])), np_bits(pick(w["scales"])),
                                  np_bits(pick(w["zeros"])) if "zeros" in w else None, g, group=inp["G"])


def acts_of(inp, rows=None):
    a = inp["a"]
    data = np_bits(a["data"])
    scale = np_bits(a["scale"]) if a.get("scale") is not None else None
    if rows is not None:
        data = data[rows]
        if scale is not None:
            scale = scale[rows]
    return oracle.dequant_acts(inp["afmt"], data, scale, np_bits(a["gscale"]) if a.get("gscale") is not None else None)


def dense_ref(inp, rows=None):
    bias = np_bits(inp["bias"]) if inp.get("bias") is not None else None
    return oracle.gemm(acts_of(inp, rows), weights_of(inp), bias)


def moe_ref(inp, rows=None):
    cache = {}

    def w_of(e):
        if e < 0 or e >= inp["E"]:
            return None
        if e not in cache:
            cache[e] = weights_of(inp, e)
        return cache[e]

    return oracle.moe_gemm(acts_of(inp), w_of, inp["N"], inp["ids"].cpu().numpy(), inp["topk_w"].cpu().numpy(), rows)


def error_ratio(y_gpu, y_ref):
    """max over elements of |y - y_ref| / (RTOL |y_ref| + ATOL_RMS rms(y_ref)); <= 1 passes."""
    y = y_gpu.detach().float().cpu().double().numpy() if isinstance(y_gpu, torch.Tensor) else np.asarray(y_gpu)
    ref = np.asarray(y_ref, dtype=np.float64)
    rms = float(np.sqrt(np.mean(ref ** 2)))
    bound = RTOL * np.abs(ref) + ATOL_RMS * rms
    if y.size == 0:
        return 0.0
    return float(np.max(np.abs(y - ref) / np.maximum(bound, 1e-300)))


def assert_parity(y_gpu, y_ref, what=""):
    r = error_ratio(y_gpu, y_ref)
    assert np.isfinite(r) and r <= 1.0, f"{what}: error ratio {r:.4f} exceeds the bound"
    return r
