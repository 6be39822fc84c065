"""Offline sweep of the launch choices per (format class, size bucket); writes the table the library plans with.

For every format class and size bucket this times each valid choice of GEMM kernel (INT4 only: UMMA or
register-decode), token tile, Stream-K split on or off, CTAs per SM and (MoE) activation path on the workload
shapes of that class, against the planner's built-in rule ("Tuning and JIT compilation per workload": device
heuristics per range of input sizes; "Future plans": autotune).  A bucket takes the best choice only where it
beats the built-in rule by more than the noise margin on every size measured in it; elsewhere its row keeps the
built-in rule, so no bucket gets slower.  Each candidate's output is checked against the built-in rule's before
it can be chosen.

Run on the target GPU from the repository root, then rebuild so the library carries the new table:
    python -m quantized_gemm_dequant_gb300.tune [--classes int4,nvfp4,...] [--quick]
    python -c "from quantized_gemm_dequant_gb300 import build; build.build()"
Writes csrc/hq_tune_table.h and tune_results.json beside this file.
"""
import argparse
import json
import os
import statistics
import sys
import time

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))

import quantized_gemm_dequant_gb300 as hq  # noqa: E402
from workload import configs as W  # noqa: E402

TABLE = os.path.join(HERE, "csrc", "hq_tune_table.h")
RESULTS = os.path.join(HERE, "tune_results.json")
INF = 1 << 62
AUTO = dict(kernel=-1, bt=0, sk=-1, slots=0, grouped=-1, cpb=0)
MARGIN = 0.97  # a tuned choice must be at least 3 % faster than the built-in rule on every size of its bucket
CLASS_ID = {"int4": 0, "regdec": 1, "nvfp4": 2, "mxfp4": 3, "mxfp4a": 4}

# (class, workload config, kind (0 dense, 1 MoE, 2 MoE Down GEMM with the top-k combine), buckets: [(key upper bound,
# sizes measured)]); MoE keys are routed rows per expert, rounded up (E=128 top-8: key = T/16; E=256 top-8: key = T/32)
PLANS = [
    ("int4", "w4a16_asym", 0, [(1, [1]), (8, [4, 8]), (16, [16]), (32, [24, 32]), (64, [48, 64]), (128, [96, 128]),
                               (256, [256]), (512, [512]), (1024, [1024]), (2048, [2048]), (4096, [4096]),
                               (INF, [8192])]),
    ("int4", "moe_w4a16", 1, [(1, [1, 16]), (2, [32]), (4, [64]), (8, [128]), (16, [256]), (32, [512]),
                              (64, [1024]), (128, [2048]), (256, [4096]), (INF, [8192])]),
    ("regdec", "w8a16", 0, [(1, [1]), (8, [8]), (16, [16]), (32, [32]), (64, [64]), (INF, [256])]),
    ("nvfp4", "nvfp4", 0, [(1, [1]), (16, [16]), (64, [64]), (128, [128]), (256, [256]), (512, [512]),
                           (1024, [1024]), (2048, [2048]), (4096, [4096]), (INF, [8192])]),
    ("int4", "moe_w4a16_down", 2, [(1, [1, 16]), (2, [32]), (4, [64]), (8, [128]), (16, [256]), (32, [512]),
                                   (64, [1024]), (128, [2048]), (256, [4096]), (INF, [8192])]),
    ("mxfp4", "moe_mxfp4", 1, [(1, [1, 32]), (2, [64]), (8, [256]), (32, [1024]), (128, [4096]), (INF, [8192])]),
    ("mxfp4", "moe_mxfp4_down", 2, [(1, [1, 32]), (2, [64]), (8, [256]), (32, [1024]), (128, [4096]),
                                    (INF, [8192])]),
    ("mxfp4a", "w4a8_mx", 0, [(1, [1]), (128, [128]), (256, [256]), (1024, [1024]), (4096, [4096]),
                              (INF, [8192])]),
]


def candidates(cls, moe, key, M=None):
    """Every valid choice for one call (the library also re-checks each); key = M (dense) or routed rows per expert
    (MoE, whose tiles are sized by the busiest experts: every tile width up to twice the token count is tried)."""
    out = [dict(AUTO)]
    span = M if (moe and M is not None) else key
    umma_bts = [b for b in (16, 32, 64, 128, 256) if b < 2 * max(span, 8)]
    if moe and cls in ("nvfp4", "mxfp4a"):
        umma_bts = [b for b in umma_bts if b <= 128]
    if cls == "regdec" or (cls == "int4" and key <= (64 if moe else 256)):
        for bt in (8, 16, 32):
            for sk in (0, 1):
                for slots in ((1, 2) if bt <= 16 else (1,)):
                    for cpb in ((0, 2, 6) if sk else (0,)):
                        out.append(dict(kernel=1, bt=bt, sk=sk, slots=slots, grouped=0 if moe else -1, cpb=cpb))
    if cls != "regdec":
        for bt in umma_bts:
            for sk in (0, 1):
                for grouped in ((0, 1) if moe else (-1,)):
                    out.append(dict(kernel=0 if cls == "int4" else -1, bt=bt, sk=sk, slots=0, grouped=grouped, cpb=0))
    return out


def env_of(c):
    return ",".join(f"{k}={v}" for k, v in c.items())


def make_sized_calls(cfg_name, sizes, dev, seed=0):
    """Per size: a function call(choice) -> (median ms per call, output of the last call); inputs resident, R
    replicas rotated so that the weights come from HBM."""
    c = W.CONFIGS[cfg_name]
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    res = {}
    if c["kind"] == "dense":
        base = W.make_dense(cfg_name, 1, seed=seed, device=dev)
        fmt, packed = hq.pack_inputs(base, dev)
    else:
        base = W.make_moe(cfg_name, 1, seed=seed, device=dev)
        fmt, packed = hq.pack_inputs(base, dev)
    del base
    R = max(2, min(8, (3 * l2) // max(1, packed.numel()) + 1))
    packs = [packed] + [packed.clone() for _ in range(R - 1)]
    for M in sizes:
        if c["kind"] == "dense":
            a = W.quantize_acts(c["afmt"], W.acts_fp32(seed, M, c["K"], outliers=c["afmt"] == "nvfp4", device=dev))
            outs = [torch.empty((M, c["N"]), dtype=torch.bfloat16, device=dev) for _ in range(R)]

            def run(r, ws, a=a, outs=outs, M=M):
                hq.gemm(fmt, a, packs[r], M, out=outs[r], workspace=ws)
                return outs[r]
        elif c.get("down"):  # Down GEMM + combine: the T * topk routed rows in, the T token rows out
            a = W.quantize_acts(c["afmt"], W.acts_fp32(seed, M * c["topk"], c["K"], device=dev))
            ids, tw = W.zipf_route(seed, M, c["E"], c["topk"], device=dev)
            outs = [torch.empty((M, c["N"]), dtype=torch.bfloat16, device=dev) for _ in range(R)]

            def run(r, ws, a=a, ids=ids, tw=tw, outs=outs):
                hq.moe_gemm_combine(fmt, a, packs[r], ids, tw, out=outs[r], workspace=ws)
                return outs[r]
        else:
            a = W.quantize_acts(c["afmt"], W.acts_fp32(seed, M, c["K"], device=dev))
            ids, tw = W.zipf_route(seed, M, c["E"], c["topk"], device=dev)
            outs = [torch.empty((M * c["topk"], c["N"]), dtype=torch.bfloat16, device=dev) for _ in range(R)]

            def run(r, ws, a=a, ids=ids, tw=tw, outs=outs):
                hq.moe_gemm(fmt, a, packs[r], ids, tw, out=outs[r], workspace=ws)
                return outs[r]
        res[M] = (run, c["topk"] if c["kind"] == "moe" else 1, bool(c.get("down")))
    return fmt, res, R


def time_choice(fmt, run, M, topk, R, choice, bursts, per_burst, down=False):
    os.environ["HQ_TUNE"] = env_of(choice)
    try:
        mk = hq.make_combine_workspace if down else hq.make_workspace
        wss = [mk(fmt, M, topk) for _ in range(R)]
        for r in range(R):
            run(r, wss[r])
        torch.cuda.synchronize()
        ts = []
        n = 0
        for _ in range(bursts):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            torch.cuda._sleep(2_000_000)
            e0.record()
            for _ in range(per_burst):
                y = run(n % R, wss[n % R])
                n += 1
            e1.record()
            ts.append((e0, e1))
        torch.cuda.synchronize()
        status = max(hq.last_device_status(w) for w in wss)
        if status != 0:
            return None, None
        return statistics.median(a.elapsed_time(b) / per_burst for a, b in ts), y.float().clone()
    finally:
        del os.environ["HQ_TUNE"]


def close(y, ref):
    d = (y - ref).abs().max().item()
    return d <= 2e-2 * max(1.0, ref.abs().max().item())


def sweep(plans, quick, dev):
    results = []
    bursts, per_burst = (5, 6) if quick else (9, 10)
    for cls, cfg, moe, buckets in plans:
        sizes = sorted({s for _, ss in buckets for s in ss})
        fmt, calls, R = make_sized_calls(cfg, sizes, dev)
        meas = {}
        for M in sizes:
            run, topk, down = calls[M]
            t_auto, y_auto = time_choice(fmt, run, M, topk, R, AUTO, bursts, per_burst, down)
            rows = []
            c_cfg = W.CONFIGS[cfg]
            key = -(-M * c_cfg["topk"] // c_cfg["E"]) if moe else M
            for c in candidates(cls, moe, key, M):
                t, y = (t_auto, y_auto) if c == AUTO else time_choice(fmt, run, M, topk, R, c, bursts, per_burst, down)
                ok = t is not None and close(y, y_auto)
                rows.append(dict(choice=c, ms=t, ok=ok))
            meas[M] = dict(auto_ms=t_auto, rows=rows)
            best = min((r for r in rows if r["ok"]), key=lambda r: r["ms"])
            print(f"{cls:7s} {cfg:12s} M={M:5d}: built-in {1e3 * t_auto:9.2f} us, best {1e3 * best['ms']:9.2f} us "
                  f"{env_of(best['choice'])}", flush=True)
        lo = 0
        for ub, ss in buckets:
            # the choice minimising the worst ratio to the built-in rule over the bucket's sizes
            keys = [env_of(r["choice"]) for r in meas[ss[0]]["rows"]]
            score = {}
            for k in keys:
                worst = 0.0
                for M in ss:
                    r = next((r for r in meas[M]["rows"] if env_of(r["choice"]) == k), None)
                    if r is None or not r["ok"]:
                        worst = float("inf")
                        break
                    worst = max(worst, r["ms"] / meas[M]["auto_ms"])
                score[k] = worst
            k_best = min(score, key=score.get)
            chosen = k_best if score[k_best] < MARGIN else env_of(AUTO)
            choice = next(r["choice"] for r in meas[ss[0]]["rows"] if env_of(r["choice"]) == chosen)
            results.append(dict(cls=cls, workload=cfg, moe=moe, key_lo=lo, key_max=ub, sizes=ss,
                                choice=choice, ratio_vs_builtin=min(score[chosen], 1.0),
                                per_size={str(M): dict(builtin_us=1e3 * meas[M]["auto_ms"],
                                                       chosen_us=1e3 * next(r["ms"] for r in meas[M]["rows"]
                                                                            if env_of(r["choice"]) == chosen),
                                                       candidates=[dict(choice=r["choice"], ok=r["ok"],
                                                                        us=None if r["ms"] is None else 1e3 * r["ms"])
                                                                   for r in meas[M]["rows"]])
                                          for M in ss}))
            lo = ub
        del calls
        torch.cuda.empty_cache()
    return results


def write_table(results, device_name):
    lines = ["// Launch-choice rows per (format class, size bucket), written by tune.py from a timing sweep on",
             f"// {device_name}; regenerate with that script rather than editing by hand.  Rows of one class are in",
             "// ascending key order; a row whose fields are all -1 / 0 keeps the built-in rule.  The sentinel row",
             "// ends the table.",
             "#pragma once", "namespace hq {", "static const TuneRow kTuneRows[] = {"]
    merged = []
    for r in results:
        c = r["choice"]
        if merged and merged[-1]["cls"] == r["cls"] and merged[-1]["moe"] == r["moe"] and merged[-1]["choice"] == c:
            merged[-1]["key_max"] = r["key_max"]
            merged[-1]["ratio"] = max(merged[-1]["ratio"], r["ratio_vs_builtin"])
            continue
        merged.append(dict(cls=r["cls"], moe=r["moe"], key_lo=r["key_lo"], key_max=r["key_max"], choice=c,
                           ratio=r["ratio_vs_builtin"], workload=r["workload"]))
    for m in merged:
        c = m["choice"]
        key = "INT64_MAX" if m["key_max"] >= INF else str(m["key_max"])
        note = "built-in rule" if c == AUTO else f"at most {m['ratio']:.2f}x the built-in time"
        lines.append(f"    {{{CLASS_ID[m['cls']]}, {m['moe']}, {key}, {{{c['kernel']}, {c['bt']}, {c['sk']}, "
                     f"{c['slots']}, {c['grouped']}, {c.get('cpb', 0)}}}}},  // {m['workload']} key ({m['key_lo']}, "
                     f"{key}]: {note}")
    lines += ["    {-1, -1, 0, {}},", "};", "}  // namespace hq", ""]
    with open(TABLE, "w") as f:
        f.write("\n".join(lines))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--classes", default=",".join(CLASS_ID))
    ap.add_argument("--quick", action="store_true")
    args = ap.parse_args()
    if not torch.cuda.is_available():
        raise SystemExit("tune.py needs a GPU")
    want = set(args.classes.split(","))
    plans = [p for p in PLANS if p[0] in want]
    dev = torch.device("cuda:0")
    t0 = time.time()
    results = sweep(plans, args.quick, dev)
    name = torch.cuda.get_device_name(dev)
    with open(RESULTS, "w") as f:
        json.dump(dict(device=name, seconds=round(time.time() - t0, 1), margin=MARGIN, buckets=results), f, indent=1)
    write_table(results, name)
    print(f"wrote {TABLE} and {RESULTS} in {time.time() - t0:.0f} s")


if __name__ == "__main__":
    main()
