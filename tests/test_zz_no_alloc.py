"""hq_gemm_static_scratch: the dense GEMM for callers that cannot allocate device memory (GPU).

Such callers (a host framework that owns all device memory through its own pool,
or a latency-critical loop that must not risk a synchronising cudaMalloc) get
their scratch from a fixed per-GPU array inside the library.  The test calls the
entry point through the C ABI twice in a row, with different shapes that use
the scratch differently (split-K partials in both), and checks each result
bit for bit against the workspace-taking hq_gemm (the same kernels on the same
inputs) and element by element against the oracle within the parity bound.  It
also checks the property the entry point exists for: after a first call (which
may load the library's device code and its static array), the calls leave the
device's free memory unchanged.  It lives in its own file, collected last.
"""
import pytest
import torch

from tests import ref_helpers as R
from workload import make_dense

pytestmark = pytest.mark.gpu


def _case(lib, cfg, M, N, K, seed):
    inp = make_dense(cfg, M, seed=seed, N=N, K=K, with_bias=True)
    fmt, packed = lib.pack_inputs(inp, "cuda")
    act = {k: v.cuda() for k, v in inp["a"].items()}
    bias = inp["bias"].cuda()
    return inp, fmt, packed, act, bias


def test_static_scratch_matches_workspace_call_twice(lib):
    cases = [("w4a16_asym", 16, 1024, 2048, 1), ("w4a16_asym", 64, 2048, 4096, 2)]
    prepared = []
    for cfg, M, N, K, seed in cases:
        inp, fmt, packed, act, bias = _case(lib, cfg, M, N, K, seed)
        assert lib.workspace_bytes(fmt, M) <= 16 << 20
        y_ws = lib.gemm(fmt, act, packed, M, bias=bias)
        out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        prepared.append((cfg, M, inp, fmt, packed, act, bias, y_ws, out))
    # warm-up call: the first call on a device may load the library's module (and with it the static array)
    cfg, M, inp, fmt, packed, act, bias, y_ws, out = prepared[0]
    lib.gemm_static_scratch(fmt, act, packed, M, bias=bias, out=out)
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for cfg, M, inp, fmt, packed, act, bias, y_ws, out in prepared:
        out.zero_()
        torch.cuda.synchronize()
        lib.gemm_static_scratch(fmt, act, packed, M, bias=bias, out=out)
        torch.cuda.synchronize()
        assert torch.equal(out, y_ws), f"{cfg} M={M}: differs from hq_gemm on the same inputs"
        R.assert_parity(out, R.dense_ref(inp), f"{cfg} M={M} against the oracle")
    assert torch.cuda.mem_get_info()[0] == free0, "the calls changed the device's free memory"


def test_static_scratch_rejects_oversized_calls(lib):
    # 512 tokens over 4096 x 4096: 64 tiles of 256 tokens are split along K (Stream-K), whose ~40 MB of partial
    # sums exceed the fixed 16 MiB
    fmt = lib.make_format("uint4_zp", 4096, 4096)
    assert lib.workspace_bytes(fmt, 512) > 16 << 20
    act = {"data": torch.zeros(512, 4096, dtype=torch.bfloat16, device="cuda")}
    packed = torch.zeros(lib.packed_bytes(fmt), dtype=torch.uint8, device="cuda")
    with pytest.raises(lib.HQError) as e:
        lib.gemm_static_scratch(fmt, act, packed, 512)
    assert e.value.code == lib.HQ_ERR_WORKSPACE
