"""Full workload sizes, in the launch configuration the benchmark times, on sampled output rows (GPU).

Inputs are generated on the device by the seeded generator; the oracle receives
copies of exactly those bytes and computes the sampled rows in fp64.  Every
output element is also checked to be finite.
"""
import numpy as np
import pytest
import torch

import oracle
from tests import ref_helpers as R
from workload import CONFIGS, make_dense, make_moe
from workload import configs as W

pytestmark = pytest.mark.gpu


def _sample_rows(n, k=6, seed=0):
    rng = np.random.default_rng(seed)
    rows = {0, n - 1, n // 2}
    rows |= set(rng.integers(0, n, size=k).tolist())
    return sorted(r for r in rows if 0 <= r < n)


@pytest.fixture(scope="module")
def dense_layers(lib):
    cache = {}

    def get(cfg):
        if cfg not in cache:
            base = make_dense(cfg, 1, seed=0, device="cuda")
            fmt, packed = lib.pack_inputs(base, "cuda")
            host = dict(base, w={k: v.cpu() for k, v in base["w"].items()})
            cache[cfg] = (fmt, packed, R.weights_of(host))
        return cache[cfg]

    return get


OTHER_DENSE = ["w8a16", "w2a16", "w1a16", "w3a16", "mxint4_a16", "fp8w_a16", "w4a8_mx", "w4a4_mx"]


@pytest.mark.parametrize("cfg,M", [("w4a16_sym", 8)] + [("w4a16_asym", m) for m in CONFIGS["w4a16_asym"]["sizes"]]
                         + [("nvfp4", m) for m in CONFIGS["nvfp4"]["sizes"]]
                         + [(c, m) for c in OTHER_DENSE for m in (CONFIGS[c]["sizes"][0], CONFIGS[c]["sizes"][-1])])
def test_dense_full_size_sampled(lib, dense_layers, cfg, M):
    c = CONFIGS[cfg]
    fmt, packed, wdeq = dense_layers(cfg)
    a = W.quantize_acts(c["afmt"], W.acts_fp32(0, M, c["K"], outliers=c["afmt"] == "nvfp4", device="cuda"))
    y = lib.gemm(fmt, a, packed, M)
    torch.cuda.synchronize()
    assert bool(torch.isfinite(y.float()).all())
    rows = _sample_rows(M, seed=M)
    host = dict(M=M, afmt=c["afmt"], a={k: v.cpu() for k, v in a.items()})
    ref = oracle.gemm(R.acts_of(host, rows), wdeq)
    R.assert_parity(y[rows], ref, f"{cfg} M={M} rows {rows}")


@pytest.fixture(scope="module")
def moe_layers(lib):
    cache = {}

    def get(cfg):
        if cfg not in cache:
            base = make_moe(cfg, 1, seed=0, device="cuda")
            fmt, packed = lib.pack_inputs(base, "cuda")
            host_w = {k: v.cpu() for k, v in base["w"].items()}
            del base
            torch.cuda.empty_cache()
            cache[cfg] = (fmt, packed, host_w)
        return cache[cfg]

    return get


@pytest.mark.parametrize("cfg,T", [("moe_w4a16", t) for t in CONFIGS["moe_w4a16"]["sizes"]]
                         + [("moe_mxfp4", t) for t in CONFIGS["moe_mxfp4"]["sizes"]])
def test_moe_full_size_sampled(lib, moe_layers, cfg, T):
    c = CONFIGS[cfg]
    fmt, packed, host_w = moe_layers(cfg)
    a = W.quantize_acts(c["afmt"], W.acts_fp32(0, T, c["K"], device="cuda"))
    ids, tw = W.zipf_route(0, T, c["E"], c["topk"], device="cuda")
    y = lib.moe_gemm(fmt, a, packed, ids, tw)
    torch.cuda.synchronize()
    assert bool(torch.isfinite(y.float()).all())
    rows = _sample_rows(T * c["topk"], k=5, seed=T)
    host = dict(T=T, E=c["E"], N=c["N"], K=c["K"], G=c["G"], wfmt=c["wfmt"], afmt=c["afmt"],
                w=host_w, a={k: v.cpu() for k, v in a.items()}, ids=ids.cpu(), topk_w=tw.cpu())
    ref = R.moe_ref(host, rows)
    R.assert_parity(y[rows], ref, f"{cfg} T={T} rows {rows}")
