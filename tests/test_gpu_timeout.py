"""The bounded-wait error path of the GEMM kernels (GPU), exercised without a GPU fault.

Every pipeline wait inside the GEMM kernels gives up after a time bound; the
kernel then records HQ_ERR_TIMEOUT in the workspace status, lets the copies and
MMAs it already issued land, frees its tensor memory and returns.  These tests
shorten the bound to 1 ns (hq_set_wait_limit_ns), so that the first wait that
is not already satisfied runs out, and check that

  - the call returns and the stream completes (no hang),
  - the workspace status reads HQ_ERR_TIMEOUT,
  - the next call with the default bound on the same workspace matches the
    oracle element by element and leaves the status clean.

Each kernel family is covered: the tcgen05 (UMMA) kernel with 256-token tiles
(INT4 decode into tensor memory), with NVFP4 block-scaled MMAs and with MoE
gathers, and the register-decode mma.sync kernel for small token counts.
"""
import pytest
import torch

from tests import ref_helpers as R
from workload import make_dense, make_moe

pytestmark = pytest.mark.gpu

ATTEMPTS = 5  # a wait satisfied on its first test cannot run out; a few calls make a miss practically impossible


@pytest.fixture
def short_waits(lib):
    yield lib
    lib.set_wait_limit_ns(0)  # back to the default bound whatever happened


def _timeout_then_recover(lib, run, ref):
    """run(ws) enqueues one call on workspace ws and returns its output tensor."""
    ws = run(None, want_ws=True)
    codes = []
    lib.set_wait_limit_ns(1)
    for _ in range(ATTEMPTS):
        run(ws)
        torch.cuda.synchronize()
        st = lib.last_device_status(ws)
        codes.append(st)
        if st == lib.HQ_ERR_TIMEOUT:
            break
    assert lib.HQ_ERR_TIMEOUT in codes, f"no wait ran out with a 1 ns bound: statuses {codes}"
    assert all(c in (lib.HQ_OK, lib.HQ_ERR_TIMEOUT) for c in codes), codes
    lib.set_wait_limit_ns(0)
    y = run(ws)
    torch.cuda.synchronize()
    assert lib.last_device_status(ws) == lib.HQ_OK
    R.assert_parity(y, ref, "call after a timed-out call on the same workspace")


def _dense(lib, cfg, M, N, K, seed=3):
    inp = make_dense(cfg, M, seed=seed, N=N, K=K)
    fmt, packed = lib.pack_inputs(inp, "cuda")
    act = {k: v.cuda() for k, v in inp["a"].items()}
    out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")

    def run(ws, want_ws=False):
        if want_ws:
            return lib.make_workspace(fmt, M)
        return lib.gemm(fmt, act, packed, M, out=out, workspace=ws)

    return run, R.dense_ref(inp)


@pytest.mark.parametrize("case", [("uint4_zp", 256, 512, 2048), ("int4_sym", 16, 384, 1024),
                                  ("nvfp4", 128, 256, 1536)])
def test_dense_wait_timeout_then_recovery(short_waits, case):
    lib = short_waits
    wfmt, M, N, K = case
    cfg = {"uint4_zp": "w4a16_asym", "int4_sym": "w4a16_sym", "nvfp4": "nvfp4"}[wfmt]
    run, ref = _dense(lib, cfg, M, N, K)
    _timeout_then_recover(lib, run, ref)


def test_moe_wait_timeout_then_recovery(short_waits):
    lib = short_waits
    inp = make_moe("moe_mxfp4", 48, seed=4, E=6, N=256, K=512, topk=2)
    fmt, packed = lib.pack_inputs(inp, "cuda")
    act = {k: v.cuda() for k, v in inp["a"].items()}
    ids, tw = inp["ids"].cuda(), inp["topk_w"].cuda()
    out = torch.empty((48 * 2, 256), dtype=torch.bfloat16, device="cuda")

    def run(ws, want_ws=False):
        if want_ws:
            return lib.make_workspace(fmt, 48, 2)
        return lib.moe_gemm(fmt, act, packed, ids, tw, out=out, workspace=ws)

    _timeout_then_recover(lib, run, R.moe_ref(inp))
