"""The offline sweep's table writer (host logic, no GPU): bucket rows merge, stay in key order and keep the
built-in rule where no choice wins by the margin."""
import re

import pytest

pytest.importorskip("torch")


def _result(cls, moe, lo, hi, choice, ratio):
    return dict(cls=cls, workload="w", moe=moe, key_lo=lo, key_max=hi, sizes=[hi], choice=choice,
                ratio_vs_builtin=ratio, per_size={})


def test_rows_merge_and_keep_order(tmp_path, monkeypatch):
    from quantized_gemm_dequant_gb300 import tune
    monkeypatch.setattr(tune, "TABLE", str(tmp_path / "t.h"))
    a = dict(kernel=1, bt=8, sk=1, slots=2, grouped=-1, cpb=2)
    res = [_result("int4", 0, 0, 1, a, 0.8), _result("int4", 0, 1, 8, a, 0.9),
           _result("int4", 0, 8, 16, dict(tune.AUTO), 1.0), _result("int4", 0, 16, tune.INF, a, 0.95),
           _result("nvfp4", 1, 0, 4, dict(tune.AUTO), 1.0)]
    tune.write_table(res, "test device")
    text = (tmp_path / "t.h").read_text()
    rows = re.findall(r"^\s*\{(-?\d+), (-?\d+), (\w+), \{(-?\d+), (-?\d+), (-?\d+), (-?\d+), (-?\d+), (-?\d+)\}\}",
                      text, re.M)
    assert rows == [("0", "0", "8", "1", "8", "1", "2", "-1", "2"), ("0", "0", "16", "-1", "0", "-1", "0", "-1", "0"),
                    ("0", "0", "INT64_MAX", "1", "8", "1", "2", "-1", "2"),
                    ("2", "1", "4", "-1", "0", "-1", "0", "-1", "0")]
    assert text.rstrip().endswith("}  // namespace hq")
    assert "{-1, -1, 0, {}}," in text


def test_candidates_are_valid():
    from quantized_gemm_dequant_gb300 import tune
    for cls, cfg, moe, buckets in tune.PLANS:
        for _, sizes in buckets:
            for M in sizes:
                c_cfg = tune.W.CONFIGS[cfg]
                key = -(-M * c_cfg["topk"] // c_cfg["E"]) if moe else M
                for c in tune.candidates(cls, moe, key, M):
                    assert c["bt"] in (0, 8, 16, 32, 64, 128, 256)
                    if c["kernel"] == 1:
                        assert c["bt"] <= 32 and (c["slots"] <= 1 or c["bt"] <= 16)
                    if moe and cls in ("nvfp4", "mxfp4a"):
                        assert c["bt"] <= 128
                    if cls == "regdec":
                        assert c["kernel"] in (-1, 1)
