"""Benchmark of the fused-dequantization quantized GEMM on GB300.

Default workload: dense W4A16 with UINT4 codes + zero points (group 128),
K=4096, N=14336, swept over M in {1, 16, 64, 256, 1024, 4096, 8192}.  One step
is one call per M (the whole hot path: repacked weights are resident, every
call decodes, multiplies and runs the epilogue).  Calls of one size are timed
as bursts of back-to-back launches with CUDA events on their stream (the way
the GEMMs of a decode step follow one another), with a cold L2 as in the
microbenchmark protocol of the Humming announcement ("Results: kernel
microbenchmarks": cold L2, warmed, independent samples): every call reads its
own replica of weights, activations and output, rotated over enough replicas
that their total is far above the L2 size, so no flush kernel runs (a write
flush would leave the L2 full of dirty lines whose write-back slows the next
kernel's reads).

Prints one JSON line (rank 0).  `--impl reference` times the CPU oracle on a
bounded sample of the same workload instead.  `--config` selects another
workload (nvfp4, moe_w4a16, moe_mxfp4, w4a16_sym) for ad-hoc measurement, or the
activation quantizers that feed the W4A8 / W4A4 paths (aq_e4m3_tok, aq_nvfp4).
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from workload import configs as W  # noqa: E402

FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# dense tensor-core peaks relative to bf16 (nominal 2.25 / 4.5 / 13.5 PFLOP/s)
DTYPE_RATIO = {"bf16": 1.0, "fp8": 2.0, "fp4": 6.0}
PATH_DTYPE = {"int4_sym": "bf16", "uint4_zp": "bf16", "nvfp4": "fp4", "mxfp4": "fp8", "int8_sym": "bf16",
              "uint2_zp": "bf16", "mxint4": "bf16", "e4m3": "bf16", "uint1_zp": "bf16", "uint3_zp": "bf16"}


def path_dtype(c):
    """The MMA's operand type of a workload: FP4 on both sides (NVFP4, MXFP4 x MXFP4) runs at the FP4 rate."""
    return "fp4" if c["afmt"] in ("nvfp4", "mxfp4") else PATH_DTYPE[c["wfmt"]]


SPIN_CYCLES = 2_000_000  # about 1 ms at 2 GHz: longer than the host side of one burst of calls (at most 12 calls,
#                           each with the binding's argument checks and the library's launch)


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK), "fallback"


def max_over_ranks(x, device=None):
    """The largest value of x over the ranks of the initialised process group (x itself on one rank)."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def env_rank():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("LOCAL_RANK", "0"))


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.proc = None
        import tempfile
        self.path = os.path.join(tempfile.gettempdir(), f"hq_clocks_{os.getpid()}.csv")  # raw samples; summary in the line
        self.gpu = gpu_index

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.f,
                                         stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self, t0=None, t1=None):
        """Summary of the samples taken between wall times t0 and t1 (all samples if too few)."""
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        import datetime
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 10:
                try:
                    ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                except ValueError:
                    ts = None
                rows.append((ts, parts[1:]))
        if not rows:
            return None
        inside = [p for ts, p in rows if ts is not None and t0 is not None and t0 <= ts <= t1]
        window = "timed region"
        if len(inside) < 3:
            inside, window = [p for _, p in rows], "whole run"
        sm = [float(r[1]) for r in inside if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in inside if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(inside), "window": window}


# ------------------------------------------------------------------ workload
# (the Down GEMM workloads moe_w4a16_down / moe_mxfp4_down are in workload.configs)
REPLICAS_OVERRIDE = None  # --replicas (profiling runs keep the device footprint small)


def replicas_for(touched_min, packed_bytes, l2):
    """Copies of every input so that a call never finds its data in L2: consecutive reuses of one
    replica are separated by more than three L2 sizes of other replicas' data."""
    if REPLICAS_OVERRIDE:
        return REPLICAS_OVERRIDE
    r = max(2, -(-3 * l2 // max(1, touched_min)))
    r = min(r, 12, max(2, (40 << 30) // max(1, packed_bytes)))
    return int(r)


def make_calls(cfg_name, seed, device):
    """Inputs resident on the device for every size of the sweep, R replicas each.

    Returns (fmt, calls, R) with calls = [(size, call(r, stream), info, acts[r], outs[r], wss[r])]."""
    import quantized_gemm_dequant_gb300 as hq
    c = W.CONFIGS[cfg_name]
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    calls = []
    if c["kind"] == "dense":
        base = W.make_dense(cfg_name, 1, seed=seed, device=device)
        fmt, packed = hq.pack_inputs(base, device)
        del base
        wbytes = W.weight_bytes(c["wfmt"], c["N"], c["K"], c["G"])
        R = replicas_for(wbytes, packed.numel(), l2)
        packs = [packed] + [packed.clone() for _ in range(R - 1)]
        for M in c["sizes"]:
            a0 = W.quantize_acts(c["afmt"], W.acts_fp32(seed, M, c["K"], outliers=c["afmt"] == "nvfp4", device=device))
            acts = [a0] + [{k: v.clone() for k, v in a0.items()} for _ in range(R - 1)]
            wss = [hq.make_workspace(fmt, M, 1, device) for _ in range(R)]
            outs = [torch.empty((M, c["N"]), dtype=torch.bfloat16, device=device) for _ in range(R)]
            info = dict(M=M, flops=W.dense_flops(M, c["N"], c["K"]), weight_bytes=wbytes,
                        total_bytes=wbytes + W.act_bytes(c["afmt"], M, c["K"]) + 2 * M * c["N"],
                        h2d=sum(t.numel() * t.element_size() for t in a0.values()), d2h=2 * M * c["N"])

            def call(r, stream=None, acts=acts, wss=wss, outs=outs, M=M):
                return hq.gemm(fmt, acts[r], packs[r], M, out=outs[r], workspace=wss[r], stream=stream)

            calls.append((M, call, info, acts, outs, wss))
        return fmt, calls, R
    E, k = c["E"], c["topk"]
    base = W.make_moe(cfg_name, 1, seed=seed, device=device)
    fmt, packed = hq.pack_inputs(base, device)
    del base
    per_expert = W.weight_bytes(c["wfmt"], c["N"], c["K"], c["G"])
    routes = {T: W.zipf_route(seed, T, E, k, device=device) for T in c["sizes"]}
    hit_min = min(int(torch.unique(ids).numel()) for ids, _ in routes.values())
    R = replicas_for(per_expert * hit_min, packed.numel(), l2)
    packs = [packed] + [packed.clone() for _ in range(R - 1)]
    down = bool(c.get("down"))
    for T in c["sizes"]:
        a_rows = T * k if down else T  # the Down GEMM reads one activation row per routed row
        a0 = W.quantize_acts(c["afmt"], W.acts_fp32(seed, a_rows, c["K"], device=device))
        ids, tw = routes[T]
        hit = int(torch.unique(ids).numel())
        acts = [dict(a0, ids=ids, tw=tw)] + [dict({kk: v.clone() for kk, v in a0.items()}, ids=ids.clone(), tw=tw.clone())
                                             for _ in range(R - 1)]
        out_rows = T if down else T * k
        wss = [(hq.make_combine_workspace(fmt, T, k, device) if down else hq.make_workspace(fmt, T, k, device))
               for _ in range(R)]
        outs = [torch.empty((out_rows, c["N"]), dtype=torch.bfloat16, device=device) for _ in range(R)]
        info = dict(M=T, flops=2.0 * T * k * c["N"] * c["K"], weight_bytes=per_expert * hit, experts_hit=hit,
                    total_bytes=per_expert * hit + W.act_bytes(c["afmt"], a_rows, c["K"]) + 2 * out_rows * c["N"]
                    + 8 * T * k,
                    h2d=sum(t.numel() * t.element_size() for t in a0.values()) + 8 * T * k, d2h=2 * out_rows * c["N"])
        gemm_fn = hq.moe_gemm_combine if down else hq.moe_gemm

        def call(r, stream=None, acts=acts, wss=wss, outs=outs, gemm_fn=gemm_fn):
            a = acts[r]
            return gemm_fn(fmt, {kk: v for kk, v in a.items() if kk not in ("ids", "tw")}, packs[r], a["ids"],
                           a["tw"], out=outs[r], workspace=wss[r], stream=stream)

        calls.append((T, call, info, acts, outs, wss))
    return fmt, calls, R


def roofline_of(info, t_s, pk, dt):
    tc = pk["bf16_tflops"] * DTYPE_RATIO[dt] * 1e12
    t_hbm = info["total_bytes"] / (pk["hbm_gbs"] * 1e9)
    t_tc = info["flops"] / tc
    bound = "hbm" if t_hbm >= t_tc else "tensor"
    return bound, max(t_hbm, t_tc) / t_s


# ------------------------------------------------------------------ GPU arm
MIN_SAMPLES = 20       # samples per size (bursts, and isolated calls)
MIN_SAMPLES_FAST = 100  # below 10 us per call
OTHER_CONFIGS = ["w4a16_sym", "nvfp4", "moe_w4a16", "moe_mxfp4", "moe_w4a16_down", "moe_mxfp4_down", "w8a16", "w2a16",
                 "w1a16", "w3a16", "mxint4_a16", "fp8w_a16", "w4a8_mx", "w4a4_mx"]


def _burst(call, n, R, stream, counter):
    """One event window holding n back-to-back calls of one size (each on the next input replica), preceded by a
    GPU spin so that the window holds the calls' GPU work and not the host's launch latency."""
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    torch.cuda._sleep(SPIN_CYCLES)
    e0.record(stream)
    for _ in range(n):
        call(counter[0] % R, stream=stream)
        counter[0] += 1
    e1.record(stream)
    return (e0, e1, n)


def sample_sizes(calls, R, burst, stream, counter, dev):
    """Per size: >= 20 bursts of back-to-back calls (>= 100 below 10 us per call) and as many isolated calls (one
    call alone in its event window after a spin: no overlap with a previous GEMM, cold L2 through the replicas).
    Returns [(burst samples in ms per call, burst call counts, isolated samples in ms)] per size."""
    out = []
    for (M, call, info, _, _, _) in calls:
        bs = [_burst(call, burst, R, stream, counter) for _ in range(MIN_SAMPLES)]
        iso = [_burst(call, 1, R, stream, counter) for _ in range(MIN_SAMPLES)]
        torch.cuda.synchronize(dev)
        per = [a.elapsed_time(b) / n for a, b, n in bs]
        if statistics.median(per) < 0.010:
            bs += [_burst(call, burst, R, stream, counter) for _ in range(MIN_SAMPLES_FAST - MIN_SAMPLES)]
            iso += [_burst(call, 1, R, stream, counter) for _ in range(MIN_SAMPLES_FAST - MIN_SAMPLES)]
            torch.cuda.synchronize(dev)
        out.append(([a.elapsed_time(b) / n for a, b, n in bs], [n for _, _, n in bs],
                    [a.elapsed_time(b) for a, b, _ in iso]))
    return out


def _q(xs, f):
    q = sorted(xs)
    return q[min(len(q) - 1, int(f * len(q)))]


def summarize(cfg_name, calls, samples, pk, pk_src, dt):
    """Per-size records (burst median / p10 / p90 and isolated median / p10 / p90, throughput, roofline fraction)
    and the roofline of the dominant kernel over the burst samples."""
    sweep, by_kernel = [], {}
    for (M, _, info, _, _, _), (ms, ns, iso) in zip(calls, samples):
        t = statistics.median(ms) * 1e-3
        ti = statistics.median(iso) * 1e-3
        bound, frac = roofline_of(info, t, pk, dt)
        _, frac_i = roofline_of(info, ti, pk, dt)
        e = dict(M=M, us=round(t * 1e6, 2), p10_us=round(_q(ms, 0.1) * 1e3, 2), p90_us=round(_q(ms, 0.9) * 1e3, 2),
                 samples=len(ms), tflops=round(info["flops"] / t / 1e12, 3),
                 weight_gbs=round(info["weight_bytes"] / t / 1e9, 1), total_gbs=round(info["total_bytes"] / t / 1e9, 1),
                 bound=bound, roofline_frac=round(frac, 4),
                 iso_us=round(ti * 1e6, 2), iso_p10_us=round(_q(iso, 0.1) * 1e3, 2),
                 iso_p90_us=round(_q(iso, 0.9) * 1e3, 2), iso_roofline_frac=round(frac_i, 4))
        if "experts_hit" in info:
            e["experts_hit"] = info["experts_hit"]
        sweep.append(e)
        key = kernel_name(cfg_name, M)
        k = by_kernel.setdefault(key, dict(flops=0.0, bytes=0.0, t=0.0, n=0))
        k["flops"] += info["flops"] * sum(ns)
        k["bytes"] += info["total_bytes"] * sum(ns)
        k["t"] += sum(m * n for m, n in zip(ms, ns)) * 1e-3
        k["n"] += sum(ns)
    dom = max(by_kernel, key=lambda k: by_kernel[k]["t"])
    d = by_kernel[dom]
    tc_peak = pk["bf16_tflops"] * DTYPE_RATIO[dt]
    t_launch = d["t"] / d["n"]
    if d["flops"] / (tc_peak * 1e12) >= d["bytes"] / (pk["hbm_gbs"] * 1e9):
        ach = d["flops"] / d["n"] / t_launch / 1e12
        roof = dict(bound="tensor", achieved=round(ach, 2), peak=tc_peak, unit="TFLOP/s", frac=round(ach / tc_peak, 4))
    else:
        ach = d["bytes"] / d["n"] / t_launch / 1e9
        roof = dict(bound="hbm", achieved=round(ach, 1), peak=pk["hbm_gbs"], unit="GB/s",
                    frac=round(ach / pk["hbm_gbs"], 4))
    roof.update(kernel=dom, peak_source=f"{pk_src} ({dt} {'burst bf16 x nominal ratio' if dt != 'bf16' else 'burst'})",
                traffic=traffic_of(dom, cfg_name),
                note="achieved = algorithmic bytes (or FLOPs) of the kernel's launches / their CUDA-event time in "
                     "the burst samples")
    return sweep, roof


def measure_other_config(cfg_name, args, pk, pk_src, stream, dev):
    """The burst + isolated samples of another workload (no timed steps): per-size records and its dominant
    kernel's roofline, as for the headline workload."""
    c = W.CONFIGS[cfg_name]
    dt = path_dtype(c)
    fmt, calls, R = make_calls(cfg_name, args.seed, dev)
    counter = [0]
    burst = R if args.burst is None else max(1, args.burst)
    for (M, call, *_r) in calls:  # warm-up
        for _ in range(max(3, args.warmup)):
            _burst(call, burst, R, stream, counter)
    torch.cuda.synchronize(dev)
    samples = sample_sizes(calls, R, burst, stream, counter, dev)
    sweep, roof = summarize(cfg_name, calls, samples, pk, pk_src, dt)
    import quantized_gemm_dequant_gb300 as hq
    for (_, _, _, _, _, wss) in calls:
        for ws in wss:
            st = hq.last_device_status(ws)
            if st != 0:
                raise RuntimeError(f"{cfg_name}: device status {hq.status_string(st)} after sampling")
    flops = sum(info["flops"] for (_, _, info, *_r) in calls)
    t = sum(e["us"] for e in sweep) * 1e-6
    out = {"workload": workload_name(cfg_name), "dtype": dt, "replicas": R, "burst": burst,
           "value": round(flops / t / 1e12, 3), "unit": "TFLOP/s",
           "value_note": "one call per size: total FLOPs / sum of the per-size burst medians",
           "roofline": roof, "sweep": sweep}
    if not args.no_context:
        out["context_cublas_bf16"] = cublas_context(cfg_name, args, calls, sweep, stream, dev)
    del calls
    torch.cuda.synchronize(dev)
    torch.cuda.empty_cache()
    return out


# ------------------------------------------------------------------ GPU arm
def run_ours(args):
    rank, world, local = env_rank()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    pk, pk_src = peaks()
    c = W.CONFIGS[args.config]
    dt = path_dtype(c)
    fmt, calls, R = make_calls(args.config, args.seed, dev)
    stream = torch.cuda.current_stream(dev)
    counter = [0]

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize(dev)

    burst = R if args.burst is None else max(1, args.burst)

    def run_steps(n_steps, times):
        # n_steps steps, one call per size each.  Calls of a size run in bursts of back-to-back launches (as
        # the layers of a decode step do), each on the next input replica; a burst's event window holds
        # `count` calls of one size.
        done = 0
        while done < n_steps:
            count = min(burst, n_steps - done)
            for i, (M, call, info, _, _, _) in enumerate(calls):
                times[i].append(_burst(call, count, R, stream, counter))
            done += count

    warm = [[] for _ in calls]
    run_steps(args.warmup, warm)
    barrier()
    times = [[] for _ in calls]
    clk = ClockSampler(local)
    clk.start()
    time.sleep(0.5)  # nvidia-smi needs a moment before its first sample
    barrier()
    t_wall0 = time.perf_counter()
    t_epoch0 = time.time()
    run_steps(args.steps, times)
    barrier()
    t_wall = time.perf_counter() - t_wall0
    step_ms = sum(sum(a.elapsed_time(b) for a, b, _ in ts) for ts in times) / args.steps
    # per-size statistics: their own samples (>= 20 bursts per size, >= 100 below 10 us), whatever --steps is
    samples = sample_sizes(calls, R, burst, stream, counter, dev)
    clocks = clk.stop(t_epoch0, time.time())
    # device status must be clean after the run
    import quantized_gemm_dequant_gb300 as hq
    for (_, _, _, _, _, wss) in calls:
        for ws in wss:
            st = hq.last_device_status(ws)
            if st != 0:
                raise RuntimeError(f"device status {hq.status_string(st)} after the timed run")
    step_ms = max_over_ranks(step_ms, dev)  # the slowest rank's step time
    flops_step = sum(info["flops"] for (_, _, info, _, _, _) in calls)
    value = world * flops_step / (step_ms * 1e-3) / 1e12
    sweep, roof = summarize(args.config, calls, samples, pk, pk_src, dt)
    roof["launches_per_step"] = sum(1 for (M, *_r) in calls if kernel_name(args.config, M) == roof["kernel"])

    e2e = measure_e2e(args, calls, stream, dev) if not args.no_e2e else None
    ctx = cublas_context(args.config, args, calls, sweep, stream, dev) if (rank == 0 and not args.no_context) else None
    n_launch = gpu_launches(args.config, fmt, calls) * args.steps
    del calls
    torch.cuda.synchronize(dev)
    torch.cuda.empty_cache()
    others = None
    if rank == 0 and not args.no_others and not args.sizes:
        others = {}
        for name in OTHER_CONFIGS:
            if name != args.config:
                others[name] = measure_other_config(name, args, pk, pk_src, stream, dev)
        for name in AQ_CONFIGS:
            others[name] = measure_act_quant(name, args, pk, pk_src, stream, dev)
    cpu = cpu_baseline_line(args) if (rank == 0 and not args.no_cpu) else None
    line = {
        "metric": "quantized GEMM TFLOP/s and weight GB/s vs M; % of HBM / tensor-core roofline",
        "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(step_ms, 4), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": dt, "data": "synthetic (seeded Philox draws, quantized by the workload recipe)",
        "config": {"workload": workload_name(args.config), "sizes": c["sizes"],
                   "l2": f"inputs larger than L2: each call reads its own replica of the weights, activations "
                         f"and output ({R} replicas, rotated; no flush kernel)",
                   "timing": f"CUDA events around bursts of {burst} back-to-back calls of one size on their "
                             f"stream (each call on its own replica), divided by the burst length; step = one call "
                             f"per size; per-size records: >= {MIN_SAMPLES} bursts (>= {MIN_SAMPLES_FAST} below "
                             f"10 us) plus as many isolated single calls (iso_*)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "roofline": roof, "sweep": sweep, "gpu_launches": n_launch,
        "clocks": clocks, "wall_s_timed": round(t_wall, 3), "e2e": e2e, "cpu_baseline": cpu,
        "context_cublas_bf16": ctx, "configs": others,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()




def kernel_name(cfg, M):
    """The GEMM kernel instance a call of this workload with M rows (dense) or T tokens (MoE) launches, from the
    library's own launch plan (built-in rule and tuned table)."""
    import quantized_gemm_dequant_gb300 as hq
    c = W.CONFIGS[cfg]
    fmt = hq.make_format(c["wfmt"], c["N"], c["K"], c.get("E", 1))
    fmt.act_type = hq._ACT_FMT[c["afmt"]]
    moe = c["kind"] != "dense"
    p = hq.launch_plan(fmt, M, c.get("topk", 1), ("combine" if c.get("down") else True) if moe else False)
    if p["kernel"] == "regdec":
        return f"hq::hq_gemm_small_kernel<{p['bt']}, {p['variant']}>"
    return f"hq::hq_gemm_kernel<{p['variant']}, {p['bt']}, {1 if c.get('down') else 0}>"


def gpu_launches(cfg, fmt, calls):
    """This library's kernels per step (one call per size): GEMM, split-K reduction, MoE routing and row
    permutation, as the launch plan of each call has them."""
    import quantized_gemm_dequant_gb300 as hq
    c = W.CONFIGS[cfg]
    moe = c["kind"] != "dense"
    if moe and c.get("down"):
        moe = "combine"
    return sum(hq.kernels_per_call(fmt, M, c.get("topk", 1), moe) for (M, *_rest) in calls)


def product_source(text):
    """A CUDA source as the product build compiles it: each block from a line `#if HQ_DEBUG_BOUNDS` to its matching
    `#endif` (the index checks of the debug build, libhq_debug.so) is left out, lines and all."""
    out, depth = [], 0
    for line in text.splitlines(keepends=True):
        s = line.strip()
        if depth:
            depth += 1 if s.startswith("#if") else (-1 if s.startswith("#endif") else 0)
            continue
        if s == "#if HQ_DEBUG_BOUNDS":
            depth = 1
            continue
        out.append(line)
    return "".join(out)


def kernel_source_hash():
    """sha256 over the CUDA sources of the product build: DRAM counters recorded for another version of them are
    stale.  The debug build's check blocks are not part of the kernels those counters describe."""
    import hashlib
    h = hashlib.sha256()
    d = os.path.join(ROOT, "quantized_gemm_dequant_gb300", "csrc")
    for f in sorted(os.listdir(d)):
        if f.endswith((".cu", ".cuh", ".h")):
            h.update(f.encode())
            with open(os.path.join(d, f), "rb") as fh:
                h.update(product_source(fh.read().decode("utf-8")).encode("utf-8"))
    return h.hexdigest()[:16]


def traffic_of(kernel, cfg):
    """DRAM bytes per launch of `kernel` from the committed ncu summary (profiles/traffic.json), or None
    when there is none or it was taken on other kernel sources."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    try:
        with open(p) as f:
            d = json.load(f)
        e = d.get(cfg, {}).get(kernel)
        if not e or e.get("source_hash") != kernel_source_hash():
            return None
        return e.get("dram_bytes_per_launch")
    except Exception:
        return None


def workload_name(cfg):
    c = W.CONFIGS[cfg]
    if c["kind"] == "dense":
        return (f"dense {c['wfmt']} x {c['afmt']} (group {c['G']}), K={c['K']}, N={c['N']}, "
                f"M in {c['sizes']}")
    what = "MoE Down GEMM + top-k combine" if c.get("down") else "MoE"
    return (f"{what} {c['wfmt']} x {c['afmt']}, E={c['E']}, top-{c['topk']}, K={c['K']}, N={c['N']}, "
            f"T in {c['sizes']}, Zipf(1.1) routing")


def cublas_context(cfg_name, args, calls, sweep, stream, dev):
    """Context only (the pages compare W4A16 with cuBLAS at small batch): torch.matmul in bf16 on bf16 weights of the
    same shape, timed with the same protocol (bursts of back-to-back calls over weight replicas that together exceed
    three L2 sizes, so that cuBLAS too reads its weights from HBM)."""
    c = W.CONFIGS[cfg_name]
    if c["kind"] != "dense" or c["afmt"] != "bf16":
        return None
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    R = int(min(256, max(4, -(-3 * l2 // (2 * c["N"] * c["K"])))))
    w0 = W.weights_fp32(args.seed, 1, c["N"], c["K"], device=dev).to(torch.bfloat16)
    wts = [w0] + [w0.clone() for _ in range(R - 1)]
    rows = []
    for (M, call, info, acts, outs, wss), ours in zip(calls, sweep):
        a = acts[0]["data"]
        outs_c = [torch.empty((M, c["N"]), dtype=torch.bfloat16, device=dev) for _ in range(R)]
        samples = []
        nb = min(R, 12)  # calls per window: few enough that the spin covers their host-side launch
        ctr = 0
        for it in range(max(6, 2 * R // nb + 2)):
            torch.cuda._sleep(SPIN_CYCLES)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(nb):
                r = ctr % R
                torch.matmul(a, wts[r].t(), out=outs_c[r])
                ctr += 1
            e1.record(stream)
            samples.append((e0, e1))
        torch.cuda.synchronize(dev)
        t = statistics.median(e0.elapsed_time(e1) / nb for e0, e1 in samples[1:]) * 1e-3
        rows.append(dict(M=M, us=round(t * 1e6, 2), tflops=round(info["flops"] / t / 1e12, 3),
                         ours_speedup=round(t / (ours["us"] * 1e-6), 3)))
    del wts
    return {"what": "torch.matmul bf16 x bf16 weights of the same shape (cuBLAS), same burst protocol; context, "
                    "not the metric", "sweep": rows}


def measure_e2e(args, calls, stream, dev):
    """Same sweep through the C ABI with pinned host buffers: H2D of the inputs, the call, D2H of C."""
    hosts = []
    for (M, call, info, acts, outs, wss) in calls:
        ha = {k: v.detach().cpu().pin_memory() for k, v in acts[0].items()}
        hout = torch.empty(outs[0].shape, dtype=outs[0].dtype).pin_memory()
        hosts.append((ha, hout))

    def one(times):
        for (M, call, info, acts, outs, wss), (ha, hout) in zip(calls, hosts):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for k, v in ha.items():
                acts[0][k].copy_(v, non_blocking=True)
            call(0, stream=stream)
            hout.copy_(outs[0], non_blocking=True)
            e1.record(stream)
            times.append((e0, e1))

    for _ in range(max(1, args.warmup)):
        one([])
    torch.cuda.synchronize(dev)
    ts = []
    steps = min(args.steps, 20)  # every step moves the whole sweep's activations and outputs over PCIe/C2C
    for _ in range(steps):
        one(ts)
    torch.cuda.synchronize(dev)
    ms = sum(a.elapsed_time(b) for a, b in ts) / steps
    flops = sum(info["flops"] for (_, _, info, _, _, _) in calls)
    return {"value": round(flops / (ms * 1e-3) / 1e12, 3), "unit": "TFLOP/s",
            "h2d_bytes_per_step": int(sum(info["h2d"] for (_, _, info, _, _, _) in calls)),
            "d2h_bytes_per_step": int(sum(info["d2h"] for (_, _, info, _, _, _) in calls)),
            "ms_per_step": round(ms, 4), "steps": steps, "note": "weights packed once and resident; per call: H2D of the "
            "activations (pinned), the C-ABI call, D2H of C; no L2 flush"}


# ------------------------------------------------------------------ CPU oracle
def _slice_weights(inp, n_feat):
    """The workload dict with only the first n_feat output features of every expert's weights (a bounded sample)."""
    if not n_feat or n_feat >= inp["N"]:
        return inp
    w = {k: (v if k == "gscale" else v[..., :n_feat, :]) for k, v in inp["w"].items()}
    return dict(inp, w=w, N=n_feat)


def oracle_step(cfg_name, seed, state, n_feat=None):
    """One bounded sample of the workload through the CPU oracle: for each size of the sweep,
    decode the weights (the first n_feat output features when given) and compute min(M, 2) output rows in fp64.
    Returns (flops, seconds)."""
    import numpy as np
    import oracle
    from tests import ref_helpers as R
    c = W.CONFIGS[cfg_name]
    if "inp" not in state:
        if c["kind"] == "dense":
            state["inp"] = W.make_dense(cfg_name, 2, seed=seed)
        else:
            state["inp"] = W.make_moe(cfg_name, 2, seed=seed, experts_subset=None) if c["E"] <= 128 else None
    inp = state["inp"]
    if inp is None and "one" not in state:  # too large for the host: one expert stands for the sample
        state["one"] = W.make_moe(cfg_name, 2, seed=seed, experts_subset=[0])
    src = _slice_weights(inp if inp is not None else state["one"], n_feat)
    n_out = src["N"]
    flops, t0 = 0.0, time.perf_counter()
    for M in c["sizes"]:
        rows = min(M, 2)
        if c["kind"] == "dense":
            y = oracle.gemm(R.acts_of(src, list(range(rows))), R.weights_of(src))
        else:
            y = oracle.gemm(R.acts_of(src, list(range(rows))), R.weights_of(src, 0))
        flops += 2.0 * rows * n_out * c["K"]
        assert np.all(np.isfinite(y))
    return flops, time.perf_counter() - t0


def cpu_cores():
    for v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        if os.environ.get(v):
            return int(os.environ[v])
    return os.cpu_count()


def cpu_baseline_line(args, min_seconds=10.0, max_passes=4):
    """The oracle on passes of the sweep (min(M, 2) output rows per size, full weight decode) until about 10 s of
    CPU work is done (at most 4 passes)."""
    state = {}
    flops = s = 0.0
    passes = 0
    while passes < max_passes and (passes == 0 or s < min_seconds):
        f, t = oracle_step(args.config, args.seed, state)
        flops += f
        s += t
        passes += 1
    return {"value": round(flops / s / 1e12, 9), "unit": "TFLOP/s", "cores": cpu_cores(), "kind": "oracle",
            "sample": f"{passes} pass(es) of the sweep with min(M, 2) output rows per size: full weight decode to "
                      f"fp64 plus the fp64 matmul of those rows (numpy)", "seconds": round(s, 2)}


REF_FEATURES = 64  # output features per size in a reference-arm step: about 0.1 s of numpy per step


def run_reference(args):
    rank, world, _ = env_rank()
    if rank != 0:
        return
    state = {}
    for _ in range(args.warmup):
        oracle_step(args.config, args.seed, state, n_feat=REF_FEATURES)
    flops = secs = 0.0
    for _ in range(args.steps):
        f, s = oracle_step(args.config, args.seed, state, n_feat=REF_FEATURES)
        flops += f
        secs += s
    value = flops / secs / 1e12
    c = W.CONFIGS[args.config]
    line = {
        "metric": "quantized GEMM TFLOP/s and weight GB/s vs M; % of HBM / tensor-core roofline",
        "impl": "reference", "value": round(value, 9), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(secs / args.steps * 1e3, 2), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": workload_name(args.config), "sizes": c["sizes"]},
        "cpu_baseline": {"value": round(value, 9), "unit": "TFLOP/s", "kind": "oracle", "cores": cpu_cores(),
                         "sample": f"per step: each size of the sweep, weight decode of the first {REF_FEATURES} output "
                                   f"features + fp64 matmul of min(M, 2) rows (bounded so that the run takes minutes)"},
        "e2e": {"value": round(value, 9), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ activation quantization
# bf16 activations -> the FP8 per-token / NVFP4 operands (the W4A8 and W4A4 paths), on the K = 7168 activations of
# the MXFP4 MoE and NVFP4 workloads.  Memory-bound: the metric is GB/s of algorithmic bytes.
AQ_CONFIGS = {
    "aq_e4m3_tok": dict(afmt="e4m3_tok", K=7168, sizes=[1, 64, 1024, 8192]),
    "aq_nvfp4": dict(afmt="nvfp4", K=7168, sizes=[1, 128, 1024, 8192]),
}
AQ_METRIC = "activation quantization GB/s of algorithmic bytes; % of the HBM roofline"


def aq_bytes(afmt, M, K, calibrated=False):
    """Algorithmic bytes of one call: bf16 reads of x (twice for NVFP4 with the tensor's own amax: the amax must be
    known before the first block is quantized) plus the quantized data and scales written."""
    x = 2 * M * K
    if afmt == "e4m3_tok":
        return x + M * K + 4 * M
    return (x if calibrated else 2 * x) + M * K // 2 + M * K // 16 + 4


def aq_workload_name(cfg):
    c = AQ_CONFIGS[cfg]
    what = "per-token FP8 e4m3" if c["afmt"] == "e4m3_tok" else "NVFP4 (block-16 e4m3 + fp32 tensor amax)"
    return f"activation quantization bf16 -> {what}, K={c['K']}, M in {c['sizes']}"


def aq_oracle_step(cfg, seed, rows=32):  # 32 rows per size: about 0.06 s (a reference-arm step)
    """The CPU oracle on a bounded sample: `rows` rows of every size of the sweep.  Returns (bytes, seconds)."""
    import numpy as np
    import oracle
    c = AQ_CONFIGS[cfg]
    nbytes, t = 0.0, 0.0
    for M in c["sizes"]:
        r = min(M, rows)
        x = W.acts_fp32(seed, r, c["K"], outliers=c["afmt"] == "nvfp4").to(torch.bfloat16)
        bits = x.view(torch.int16).numpy().view(np.uint16)
        t0 = time.perf_counter()
        if c["afmt"] == "e4m3_tok":
            oracle.quantize_act_e4m3_per_token(bits)
        else:
            oracle.quantize_act_nvfp4(bits)
        t += time.perf_counter() - t0
        nbytes += aq_bytes(c["afmt"], r, c["K"])
    return nbytes, t


def _aq_calls(cfg, args, dev):
    import quantized_gemm_dequant_gb300 as hq
    c = AQ_CONFIGS[cfg]
    afmt, K = c["afmt"], c["K"]
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    calls = []
    sizes = [int(v) for v in args.sizes.split(",")] if getattr(args, "sizes", None) else c["sizes"]
    for M in sizes:
        R = REPLICAS_OVERRIDE or int(min(12, max(2, -(-3 * l2 // (2 * M * K)))))
        x0 = W.acts_fp32(args.seed, M, K, outliers=afmt == "nvfp4", device=dev).to(torch.bfloat16)
        xs = [x0] + [x0.clone() for _ in range(R - 1)]
        outs = [hq.quantize_act(afmt, xs[r]) for r in range(R)]
        nws = max(16, hq.quantize_act_workspace_bytes(afmt, M, K))
        wss = [torch.empty(nws, dtype=torch.uint8, device=dev) for _ in range(R)]
        amax = x0.float().abs().max().reshape(1).contiguous()  # calibrated-amax variant: the quantize kernel alone

        def call(r, stream=None, xs=xs, outs=outs, wss=wss):
            return hq.quantize_act(afmt, xs[r], out=outs[r], workspace=wss[r], stream=stream)

        def call_cal(r, stream=None, xs=xs, outs=outs, amax=amax):
            return hq.quantize_act(afmt, xs[r], global_amax=amax, out=outs[r], stream=stream)

        calls.append(dict(M=M, R=R, call=call, call_cal=call_cal, xs=xs, outs=outs, bytes=aq_bytes(afmt, M, K),
                          bytes_cal=aq_bytes(afmt, M, K, calibrated=True)))
    return calls


def _aq_timed(fn, R, n, stream):
    out = []
    done, i = 0, 0
    while done < n:
        cnt = min(R, n - done)
        torch.cuda._sleep(SPIN_CYCLES)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(cnt):
            fn(i % R, stream=stream)
            i += 1
        e1.record(stream)
        out.append((e0, e1, cnt))
        done += cnt
    return out


def _aq_summary(cfg, calls, rec, rec_cal, pk, pk_src):
    c = AQ_CONFIGS[cfg]
    afmt = c["afmt"]
    sweep = []
    kern_t = kern_b = 0.0
    for i, (cl, ts) in enumerate(zip(calls, rec)):
        per = sorted(a.elapsed_time(b) / n for a, b, n in ts)
        t = statistics.median(per) * 1e-3
        e = dict(M=cl["M"], us=round(t * 1e6, 2), p10_us=round(_q(per, 0.1) * 1e3, 2),
                 p90_us=round(_q(per, 0.9) * 1e3, 2), samples=len(per),
                 gbs=round(cl["bytes"] / t / 1e9, 1), roofline_frac=round(cl["bytes"] / t / 1e9 / pk["hbm_gbs"], 4))
        kts = rec_cal[i] if rec_cal else ts
        kper = sorted(a.elapsed_time(b) / n for a, b, n in kts)
        kt = statistics.median(kper) * 1e-3
        if rec_cal:
            e["quantize_kernel_us"] = round(kt * 1e6, 2)
        sweep.append(e)
        kern_t += kt
        kern_b += cl["bytes_cal"] if rec_cal else cl["bytes"]
    kname = "hq::act_quant_e4m3_kernel" if afmt == "e4m3_tok" else "hq::act_quant_nvfp4_kernel"
    ach = kern_b / kern_t / 1e9
    roof = dict(bound="hbm", achieved=round(ach, 1), peak=pk["hbm_gbs"], unit="GB/s", frac=round(ach / pk["hbm_gbs"], 4),
                kernel=kname, launches_per_step=len(calls), peak_source=f"{pk_src} (copy bandwidth)",
                traffic=traffic_of(kname, cfg),
                note="achieved = algorithmic bytes of the sweep's launches / their median event time, one launch "
                     "per size" + ("; NVFP4: the quantize kernel alone, with a calibrated amax (one read of x)"
                                   if rec_cal else ""))
    return sweep, roof


def measure_act_quant(cfg, args, pk, pk_src, stream, dev):
    """Per-size samples of an activation quantizer (>= 20 bursts per size, 100 below 10 us): its sweep and its
    kernel's roofline, for the per-config block of the default benchmark line."""
    calls = _aq_calls(cfg, args, dev)
    for cl in calls:
        _aq_timed(cl["call"], cl["R"], 3 * cl["R"], stream)
    torch.cuda.synchronize(dev)
    rec, rec_cal = [], []
    for cl in calls:
        n = MIN_SAMPLES_FAST if cl["M"] <= 1024 else MIN_SAMPLES
        rec.append(_aq_timed(cl["call"], cl["R"], n * cl["R"], stream))
        if AQ_CONFIGS[cfg]["afmt"] == "nvfp4":
            rec_cal.append(_aq_timed(cl["call_cal"], cl["R"], n * cl["R"], stream))
    torch.cuda.synchronize(dev)
    sweep, roof = _aq_summary(cfg, calls, rec, rec_cal or None, pk, pk_src)
    total = sum(cl["bytes"] for cl in calls)
    t = sum(e["us"] for e in sweep) * 1e-6
    del calls
    torch.cuda.empty_cache()
    return {"workload": aq_workload_name(cfg), "dtype": "f32", "value": round(total / t / 1e9, 1), "unit": "GB/s",
            "value_note": "one call per size: algorithmic bytes / sum of the per-size burst medians",
            "roofline": roof, "sweep": sweep}


def run_act_quant(args):
    rank, world, local = env_rank()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pk, pk_src = peaks()
    c = AQ_CONFIGS[args.config]
    afmt, K = c["afmt"], c["K"]
    stream = torch.cuda.current_stream(dev)
    calls = _aq_calls(args.config, args, dev)
    for cl in calls:
        _aq_timed(cl["call"], cl["R"], args.warmup * cl["R"], stream)
    torch.cuda.synchronize(dev)
    clk = ClockSampler(local)
    clk.start()
    time.sleep(0.5)
    torch.cuda.synchronize(dev)
    t_epoch0 = time.time()
    t_wall0 = time.perf_counter()
    rec = [_aq_timed(cl["call"], cl["R"], args.steps, stream) for cl in calls]
    torch.cuda.synchronize(dev)
    t_wall = time.perf_counter() - t_wall0
    clocks = clk.stop(t_epoch0, time.time())
    rec_cal = None
    if afmt == "nvfp4":  # the quantize kernel alone (calibrated amax), for its roofline
        rec_cal = [_aq_timed(cl["call_cal"], cl["R"], args.steps, stream) for cl in calls]
        torch.cuda.synchronize(dev)
    step_ms = sum(sum(a.elapsed_time(b) for a, b, _ in ts) for ts in rec) / args.steps
    sweep, roof = _aq_summary(args.config, calls, rec, rec_cal, pk, pk_src)
    total_bytes = sum(cl["bytes"] for cl in calls)
    value = world * total_bytes / (step_ms * 1e-3) / 1e9
    e2e = None
    if not args.no_e2e:
        hosts = [(cl["xs"][0].cpu().pin_memory(), {k: torch.empty(v.shape, dtype=v.dtype).pin_memory()
                                                   for k, v in cl["outs"][0].items()}) for cl in calls]

        def one(tl):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for cl, (hx, ho) in zip(calls, hosts):
                cl["xs"][0].copy_(hx, non_blocking=True)
                cl["call"](0, stream=stream)
                for k, v in ho.items():
                    v.copy_(cl["outs"][0][k], non_blocking=True)
            e1.record(stream)
            tl.append((e0, e1))

        for _ in range(3):
            one([])
        torch.cuda.synchronize(dev)
        tl = []
        nsteps = min(args.steps, 20)
        for _ in range(nsteps):
            one(tl)
        torch.cuda.synchronize(dev)
        ms = sum(a.elapsed_time(b) for a, b in tl) / nsteps
        e2e = {"value": round(total_bytes / (ms * 1e-3) / 1e9, 1), "unit": "GB/s",
               "h2d_bytes_per_step": int(sum(2 * cl["M"] * K for cl in calls)),
               "d2h_bytes_per_step": int(sum(sum(v.numel() * v.element_size() for v in cl["outs"][0].values())
                                             for cl in calls)),
               "ms_per_step": round(ms, 4), "steps": nsteps}
    cpu = None
    if rank == 0 and not args.no_cpu:
        b, sec = aq_oracle_step(args.config, args.seed, rows=4096)
        cpu = {"value": round(b / sec / 1e9, 4), "unit": "GB/s", "cores": cpu_cores(), "kind": "oracle",
               "sample": "4096 rows (or M if smaller) of every size of the sweep, quantized by the numpy oracle",
               "seconds": round(sec, 2)}
    line = {"metric": AQ_METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(step_ms, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic (seeded Philox draws, bf16)",
            "config": {"workload": aq_workload_name(args.config), "sizes": c["sizes"],
                       "l2": "each call reads its own replica of x; replicas exceed three L2 sizes except at small M",
                       "timing": "CUDA events around bursts of back-to-back calls of one size"},
            "roofline": roof, "sweep": sweep,
            "gpu_launches": args.steps * len(calls) * (1 if afmt == "e4m3_tok" else 2),
            "clocks": clocks, "wall_s_timed": round(t_wall, 3), "e2e": e2e, "cpu_baseline": cpu}
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_act_quant_reference(args):
    rank, world, _ = env_rank()
    if rank != 0:
        return
    for _ in range(args.warmup):
        aq_oracle_step(args.config, args.seed)
    b = sec = 0.0
    for _ in range(args.steps):
        bb, ss = aq_oracle_step(args.config, args.seed)
        b += bb
        sec += ss
    value = b / sec / 1e9
    c = AQ_CONFIGS[args.config]
    print(json.dumps({
        "metric": AQ_METRIC, "impl": "reference", "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(sec / args.steps * 1e3, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": aq_workload_name(args.config), "sizes": c["sizes"]},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "kind": "oracle", "cores": cpu_cores(),
                         "sample": "per step: 32 rows (or M) of every size, numpy oracle"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}),
        flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="w4a16_asym", choices=list(W.CONFIGS) + list(AQ_CONFIGS))
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-context", action="store_true", help="skip the cuBLAS bf16 context timing")
    ap.add_argument("--no-others", action="store_true", help="time only the selected workload (no per-config block)")
    ap.add_argument("--sizes", default=None, help="comma list overriding the sweep (profiling)")
    ap.add_argument("--replicas", type=int, default=None, help="input replicas (default: enough to exceed L2)")
    ap.add_argument("--burst", type=int, default=None, help="back-to-back calls per timed window (default: replicas)")
    ap.add_argument("--source-hash", action="store_true", help="print the kernel-source hash and exit")
    args = ap.parse_args()
    if args.source_hash:
        print(kernel_source_hash())
        return
    global REPLICAS_OVERRIDE
    REPLICAS_OVERRIDE = args.replicas
    if args.sizes:
        table = AQ_CONFIGS if args.config in AQ_CONFIGS else W.CONFIGS
        table[args.config] = dict(table[args.config], sizes=[int(x) for x in args.sizes.split(",")])
    args.warmup = max(3, args.warmup) if args.impl == "ours" else args.warmup
    if args.config in AQ_CONFIGS:
        (run_act_quant_reference if args.impl == "reference" else run_act_quant)(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
