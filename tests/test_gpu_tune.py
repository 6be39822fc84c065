"""Launch choices set through HQ_TUNE (the way the offline sweep times them) against the CPU oracle (GPU).

Every choice the sweep can put in the table must give correct results: each kernel, token tile, Stream-K on and
off, one or two CTAs per SM and both MoE activation paths, plus choices the planner has to refuse (a token tile
no kernel has)."""
import pytest

from tests import ref_helpers as R
from workload import make_dense, make_moe

pytestmark = pytest.mark.gpu

DENSE = [
    ("int4_sym", 5, "kernel=1,bt=8,sk=0,slots=1"),
    ("int4_sym", 40, "kernel=1,bt=16,sk=1,slots=1"),
    ("int4_sym", 40, "kernel=1,bt=32,sk=0"),
    ("int4_sym", 5, "kernel=1,bt=8,sk=1,cpb=3"),  # fewer, longer Stream-K pieces
    ("uint4_zp", 200, "kernel=0,bt=64,sk=1,cpb=5"),
    ("uint4_zp", 40, "kernel=0,bt=16,sk=0"),
    ("uint4_zp", 200, "kernel=0,bt=64,sk=1"),
    ("uint4_zp", 9, "kernel=0,bt=256,sk=1"),
    ("uint4_zp", 33, "bt=48,sk=1"),  # no kernel has 48-token tiles: the planner keeps its own
    ("nvfp4", 100, "bt=32,sk=1"),
    ("nvfp4", 20, "bt=128,sk=0"),
    ("mxfp4", 70, "bt=16,sk=0"),
    # MXFP4 tiles of 128 and 256 tokens (two expanded-weight slots) with Stream-K pieces of two tiles in one CTA
    ("mxfp4", 2048, "bt=128,sk=1"),
    ("mxfp4", 2048, "bt=256,sk=1"),
    ("int8_sym", 20, "bt=8,sk=0,slots=2"),
    ("e4m3", 3, "bt=32,sk=1"),
]
FORM = {"int4_sym": ("bf16", 128), "uint4_zp": ("bf16", 128), "nvfp4": ("nvfp4", 16), "mxfp4": ("e4m3_tok", 32),
        "int8_sym": ("bf16", 128), "e4m3": ("bf16", 128)}


@pytest.mark.parametrize("wfmt,M,choice", DENSE)
def test_dense_choice(lib, monkeypatch, wfmt, M, choice):
    monkeypatch.setenv("HQ_TUNE", choice)
    afmt, G = FORM[wfmt]
    inp = make_dense(dict(kind="dense", wfmt=wfmt, afmt=afmt, G=G), M, seed=M, N=320, K=1024)
    fmt, packed = lib.pack_inputs(inp, "cuda")
    act = {k: v.cuda() for k, v in inp["a"].items()}
    y = lib.gemm(fmt, act, packed, M)
    R.assert_parity(y, R.dense_ref(inp), f"{wfmt} M={M} {choice}")


MOE = [
    ("int4_sym", 6, "kernel=1,bt=8,sk=1,slots=1,grouped=0"),
    ("int4_sym", 40, "kernel=0,bt=32,sk=0,grouped=0"),
    ("int4_sym", 40, "kernel=1,bt=16,sk=1,cpb=2,grouped=0"),
    ("int4_sym", 40, "kernel=0,bt=64,sk=1,grouped=1"),
    ("uint4_zp", 90, "kernel=1,bt=32,sk=0,grouped=1"),
    ("mxfp4", 40, "bt=64,sk=1,grouped=0"),
    ("mxfp4", 300, "bt=128,sk=1,grouped=1"),
    ("nvfp4", 40, "bt=256,sk=0,grouped=1"),  # 256-token NVFP4 MoE tiles do not exist: the planner keeps its own
]


@pytest.mark.parametrize("wfmt,T,choice", MOE)
def test_moe_choice(lib, monkeypatch, wfmt, T, choice):
    monkeypatch.setenv("HQ_TUNE", choice)
    afmt, G = FORM[wfmt]
    inp = make_moe(dict(kind="moe", wfmt=wfmt, afmt=afmt, G=G, topk=3), T, seed=T, E=6, N=256, K=1024, topk=3)
    fmt, packed = lib.pack_inputs(inp, "cuda")
    act = {k: v.cuda() for k, v in inp["a"].items()}
    y = lib.moe_gemm(fmt, act, packed, inp["ids"].cuda(), inp["topk_w"].cuda())
    R.assert_parity(y, R.moe_ref(inp), f"moe {wfmt} T={T} {choice}")
