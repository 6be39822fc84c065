"""The debug build's device-side index checks (libhq_debug.so; GPU).

libhq_debug.so is the library compiled with HQ_DEBUG_BOUNDS: before every global
store of an output row, every fp32 reduction into a combine row and every access
to a Stream-K partial-sum slot, a kernel compares the index with the buffer's
extent; an index outside it records HQ_ERR_BOUNDS in the workspace status and the
access is skipped (no trap, the context stays usable).  The binding loads one
library per process, so the cases run in a child process with HQ_LIBRARY=debug
(tests/debug_bounds_cases.py).  Clean calls must report HQ_OK and match the
oracle: the checks catch nothing in correct kernels.  Calls whose writable rows
are lowered below the rows that exist (HQ_DEBUG_ROW_LIMIT) must report
HQ_ERR_BOUNDS, leave the rows past the limit untouched and match the oracle on
the rows below it.  Errors are taken against the bound of the kernel that ran:
the general parity bound, or on the tcgen05 INT4 path the rigorous bound of its
bf16((q - z) * s) weight arithmetic.
"""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def results(lib):
    env = dict(os.environ, HQ_LIBRARY="debug")
    env.pop("HQ_DEBUG_ROW_LIMIT", None)
    r = subprocess.run([sys.executable, os.path.join(ROOT, "tests", "debug_bounds_cases.py")], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, f"debug-build cases failed:\n{r.stdout[-2000:]}\n{r.stderr[-4000:]}"
    out = [json.loads(line) for line in r.stdout.splitlines() if line.startswith("{")]
    assert len(out) == 16, r.stdout
    return {c["case"]: c for c in out}


def test_clean_calls_report_ok_and_match_the_oracle(lib, results):
    clean = {k: v for k, v in results.items() if not k.startswith("trigger")}
    assert len(clean) == 10
    for name, c in clean.items():
        assert c["status"] == lib.HQ_OK, f"{name}: {lib.status_string(c['status'])} ({c['plan']})"
        assert c["ratio"] <= 1.0, f"{name}: error ratio {c['ratio']:.3f} of the {c['bound']} bound ({c['plan']})"
    # the cases reach both kernels, Stream-K on each and the grouped MoE path
    plans = [c["plan"] for c in clean.values()]
    assert any(p["kernel"] == "regdec" and p["sk"] for p in plans)
    assert any(p["kernel"] == "umma" and p["sk"] for p in plans)
    assert any(p["kernel"] == "umma" and p["grouped"] for p in plans)


def test_rows_declared_absent_are_caught_and_skipped(lib, results):
    trig = {k: v for k, v in results.items() if k.startswith("trigger")}
    assert len(trig) == 6
    for name, c in trig.items():
        assert c["status"] == lib.HQ_ERR_BOUNDS, f"{name}: {lib.status_string(c['status'])} ({c['plan']})"
        assert c["untouched"] is True, f"{name}: a row past the limit was written ({c['plan']})"
        assert c["ratio"] <= 1.0, f"{name}: rows below the limit at {c['ratio']:.3f} of the {c['bound']} bound"
