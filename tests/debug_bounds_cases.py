"""Cases for the debug build's device-side index checks, run in a child process with HQ_LIBRARY=debug.

Run by tests/test_gpu_debug_bounds.py, which reads one JSON line per case from
stdout.  Every case calls libhq_debug.so through the binding on small shapes
that reach each kernel family and each store path (register-decode and
tcgen05 kernels, Stream-K partial sums and the split-K reduction, dense and
table epilogues, MoE routed rows, the top-k combine).  Clean cases must leave
the workspace status at HQ_OK and match the oracle.  Trigger cases lower the
output rows a call may write below the rows that exist (HQ_DEBUG_ROW_LIMIT):
the checks must report HQ_ERR_BOUNDS, skip exactly the rows at or past the
limit (a sentinel value stays there), and the rows below it must still match
the oracle.  No access leaves the real buffers, so nothing can fault.

Each case reports its error against the bound that holds for the kernel that
ran: the general parity bound, except on the tcgen05 INT4 path, whose weights
enter the MMA as bf16((q - z) * s) and which is held to the rigorous bound of
that arithmetic (the one the random-bit-pattern parity test uses for INT4).
"""
import json
import os
import sys

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import oracle  # noqa: E402
import quantized_gemm_dequant_gb300 as hq  # noqa: E402
from tests import ref_helpers as R  # noqa: E402
from workload import configs as W  # noqa: E402

SENTINEL = 7.0  # exact in bf16; no output of these cases can take it by chance at every element of a row

DENSE = {
    "uint4_zp": dict(kind="dense", wfmt="uint4_zp", afmt="bf16", G=128),
    "nvfp4": dict(kind="dense", wfmt="nvfp4", afmt="nvfp4", G=16),
    "mxfp4": dict(kind="dense", wfmt="mxfp4", afmt="e4m3_tok", G=32),
}
MOE = {
    "int4_sym": dict(kind="moe", wfmt="int4_sym", afmt="bf16", G=128, topk=3),
    "mxfp4": dict(kind="moe", wfmt="mxfp4", afmt="e4m3_tok", G=32, topk=3),
}


def _limit(rows):
    if rows is None:
        os.environ.pop("HQ_DEBUG_ROW_LIMIT", None)
    else:
        os.environ["HQ_DEBUG_ROW_LIMIT"] = str(rows)


def _split(y, ref, limit, s_abs=None):
    """(error ratio of the rows below `limit`, whether every row from `limit` on still holds the sentinel).  With
    s_abs = sum_k |a_k w_k| per output (tcgen05 INT4), the ratio is taken against the bf16-decode bound
    2^-9 s_abs + 2^-8 |y_ref| (+ fp32 accumulation); otherwise against the general parity bound."""
    y = y.float().cpu()
    lim = y.shape[0] if limit is None else limit
    if lim == 0:
        ratio = 0.0
    elif s_abs is None:
        ratio = R.error_ratio(y[:lim], ref[:lim])
    else:
        bound = 2.0 ** -9 * s_abs[:lim] * 1.01 + 2.0 ** -8 * np.abs(ref[:lim]) + 1e-6 * s_abs[:lim]
        err = np.abs(y[:lim].numpy().astype(np.float64) - ref[:lim])
        ratio = float(np.max(err / np.maximum(bound, 1e-300)))
    untouched = bool(torch.all(y[lim:] == SENTINEL).item()) if lim < y.shape[0] else None
    return ratio, untouched


def _int4_tcgen05(wfmt, plan):
    return wfmt in ("int4_sym", "uint4_zp") and plan["kernel"] == "umma"


def _moe_abs(inp, combine):
    """sum_k |a_k w_k| times |top-k weight| per routed row (MoE) or summed over a token's rows (combine)."""
    A = np.abs(np.asarray(R.acts_of(inp)))
    ids, tw = inp["ids"].cpu().numpy(), np.abs(inp["topk_w"].cpu().numpy())
    T, k = ids.shape
    out = np.zeros((T if combine else T * k, inp["N"]))
    for e in np.unique(ids):
        Wa = np.abs(np.asarray(R.weights_of(inp, int(e))))
        for t, j in zip(*np.nonzero(ids == e)):
            row = A[t * k + j] if combine else A[t]
            out[t if combine else t * k + j] += tw[t, j] * (row @ Wa.T)
    return out


def dense_case(name, wfmt, M, N, K, limit=None):
    inp = W.make_dense(DENSE[wfmt], M, seed=3, N=N, K=K, with_bias=True)
    fmt, packed = hq.pack_inputs(inp, "cuda")
    act = {k: v.cuda() for k, v in inp["a"].items()}
    ws = hq.make_workspace(fmt, M)
    out = torch.full((M, N), SENTINEL, dtype=torch.bfloat16, device="cuda")
    _limit(limit)
    hq.gemm(fmt, act, packed, M, bias=inp["bias"].cuda(), out=out, workspace=ws)
    _limit(None)
    torch.cuda.synchronize()
    plan = hq.launch_plan(fmt, M)
    s_abs = None
    if _int4_tcgen05(wfmt, plan):
        s_abs = np.abs(np.asarray(R.acts_of(inp))) @ np.abs(np.asarray(R.weights_of(inp))).T
    ratio, untouched = _split(out, R.dense_ref(inp), limit, s_abs)
    return dict(case=name, status=hq.last_device_status(ws), ratio=ratio, untouched=untouched, plan=plan,
                bound="bf16-decode" if s_abs is not None else "general")


def moe_case(name, wfmt, T, E, N, K, limit=None):
    inp = W.make_moe(MOE[wfmt], T, seed=4, E=E, N=N, K=K, topk=3)
    fmt, packed = hq.pack_inputs(inp, "cuda")
    act = {k: v.cuda() for k, v in inp["a"].items()}
    ws = hq.make_workspace(fmt, T, 3)
    out = torch.full((T * 3, N), SENTINEL, dtype=torch.bfloat16, device="cuda")
    _limit(limit)
    hq.moe_gemm(fmt, act, packed, inp["ids"].cuda(), inp["topk_w"].cuda(), out=out, workspace=ws)
    _limit(None)
    torch.cuda.synchronize()
    plan = hq.launch_plan(fmt, T, 3, moe=True)
    s_abs = _moe_abs(inp, False) if _int4_tcgen05(wfmt, plan) else None
    ratio, untouched = _split(out, R.moe_ref(inp), limit, s_abs)
    return dict(case=name, status=hq.last_device_status(ws), ratio=ratio, untouched=untouched, plan=plan,
                bound="bf16-decode" if s_abs is not None else "general")


def combine_case(name, T, E=5, N=264, K=640):
    c = dict(MOE["int4_sym"])
    inp = W.make_moe(c, T, seed=5, E=E, N=N, K=K, topk=3)
    inp["a"] = W.quantize_acts(c["afmt"], W.acts_fp32(12, T * 3, K))
    fmt, packed = hq.pack_inputs(inp, "cuda")
    act = {k: v.cuda() for k, v in inp["a"].items()}
    ws = hq.make_combine_workspace(fmt, T, 3)
    y = hq.moe_gemm_combine(fmt, act, packed, inp["ids"].cuda(), inp["topk_w"].cuda(), workspace=ws)
    torch.cuda.synchronize()
    cache = {}

    def w_of(e):
        if e not in cache:
            cache[e] = R.weights_of(inp, e)
        return cache[e]

    ref = oracle.moe_combine(R.acts_of(inp), w_of, N, inp["ids"].cpu().numpy(), inp["topk_w"].cpu().numpy(), None)
    plan = hq.launch_plan(fmt, T, 3, moe="combine")
    s_abs = _moe_abs(inp, True) if _int4_tcgen05("int4_sym", plan) else None
    ratio, _ = _split(y, ref, None, s_abs)
    return dict(case=name, status=hq.last_device_status(ws), ratio=ratio, untouched=None, plan=plan,
                bound="bf16-decode" if s_abs is not None else "general")


CASES = [
    # clean: every check passes, the output matches the oracle
    lambda: dense_case("dense regdec stream-k", "uint4_zp", 8, 1024, 4096),
    lambda: dense_case("dense tcgen05 split-k", "uint4_zp", 64, 512, 4096),
    lambda: dense_case("dense tcgen05 ragged", "uint4_zp", 300, 384, 640),
    lambda: dense_case("dense nvfp4", "nvfp4", 128, 256, 768),
    lambda: dense_case("dense mxfp4 table", "mxfp4", 40, 256, 640),
    lambda: moe_case("moe regdec fused routing", "int4_sym", 4, 8, 256, 640),
    lambda: moe_case("moe tcgen05 grouped", "int4_sym", 200, 8, 256, 640),
    lambda: moe_case("moe mxfp4", "mxfp4", 64, 8, 256, 640),
    lambda: combine_case("combine T=37", 37),
    lambda: combine_case("combine T=300", 300),
    # triggers: rows at or past the limit exist but are declared absent
    lambda: dense_case("trigger dense regdec", "uint4_zp", 8, 1024, 4096, limit=7),
    lambda: dense_case("trigger dense tcgen05 split-k", "uint4_zp", 64, 512, 4096, limit=63),
    lambda: dense_case("trigger dense tcgen05 pairs", "uint4_zp", 300, 384, 640, limit=299),
    lambda: dense_case("trigger dense mxfp4 table", "mxfp4", 40, 256, 640, limit=33),
    lambda: moe_case("trigger moe regdec", "int4_sym", 4, 8, 256, 640, limit=11),
    lambda: moe_case("trigger moe tcgen05", "int4_sym", 200, 8, 256, 640, limit=500),
]


def main():
    assert hq.DEBUG, "run with HQ_LIBRARY=debug"
    for case in CASES:
        print(json.dumps(case()), flush=True)


if __name__ == "__main__":
    main()
