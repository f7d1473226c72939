#!/usr/bin/env python3
"""Benchmark of the NVFP4 W4A4 small-M decode projection on GB300.

Metric: small-M NVFP4 GEMV us/call and achieved HBM GB/s (% of peak), M=1..8,
Qwen3 shapes.  One step = for M in 1..8, for each Qwen3-32B projection (qkv,
o, gate_up, down): quantize a fresh BF16 activation [M, K] to NVFP4 on the GPU
and run the small-M GEMV against resident NVFP4 weights -- 32 quantize+GEMV
calls streaming 2.3 GB of weights.  Between two uses of one weight matrix the
step streams >= 245 MB of other weights, more than the 129 MB L2, so every
call reads its weights from HBM (no flush kernel needed).

value = algorithmic HBM bytes of the step (weight codes + scales, activation
in/out, outputs) / device time of the step, in GB/s.  The step is one CUDA
graph in decode-chain order (quantize -> GEMV, 32 times, with programmatic
dependent launches so that each GEMV prefetches its weights while its
quantizer runs).  The roofline times the GEMV kernels alone: one graph of the
same GEMV launches, replayed right after the timed steps; per-M graphs of the
GEMVs give the per-M breakdown.  A cold-L2 breakdown per (projection, M)
follows (512 MB flush before each call).  `e2e` repeats the step through the
public API with the activations copied from pinned host memory and the
outputs copied back inside the timed region: the step's calls captured in a
CUDA graph and replayed (`e2e.eager`: issued one by one from Python).

Launch: python bench.py [--gpus N --steps K --warmup W] [--impl reference]
(for N > 1 under torch.distributed.run: N independent replicas, weak scaling).
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from nvfp4_w4a4_decode_gemv_gb300 import synth  # noqa: E402

METRIC = "small-M NVFP4 GEMV µs/call and achieved HBM GB/s (% peak), M=1–8, Qwen3 shapes"

# DRAM traffic of the tensor-core GEMV from one ncu capture of this bench (the
# launch list in profiles/launch_list_qwen3-32b_sweep_tc.md): read + write
# bytes per launch of the GEMV on quantized activations, averaged over the 32
# (M, projection) calls of the Qwen3-32B sweep, valid only while the kernel
# source is the one that was measured.
TRAFFIC_RECORD = {"source": "nvfp4_w4a4_decode_gemv_gb300/csrc/gemv_tc.cu",
                  "sha256": "16de29400665bd3139280542a6af34870d0d042fdd8ccaa7153464c7b9062020",
                  "workload": "qwen3-32b", "bytes_per_launch": 69002212}


def recorded_traffic(workload):
    import hashlib
    path = os.path.join(ROOT, TRAFFIC_RECORD["source"])
    try:
        digest = hashlib.sha256(open(path, "rb").read()).hexdigest()
    except OSError:
        return None
    if digest != TRAFFIC_RECORD["sha256"] or workload != TRAFFIC_RECORD["workload"]:
        return None
    return TRAFFIC_RECORD["bytes_per_launch"]
WORKLOADS = {"qwen3-32b": (synth.QWEN3_32B, list(range(1, 9))), "qwen3-8b": (synth.QWEN3_8B, [1, 2, 4, 8]),
             "qwen3-14b": (synth.QWEN3_14B, [1, 2, 4, 8]),
             "qwen3-32b-decode": (synth.QWEN3_32B, [1, 4, 8]), "reset-sampler": (None, [8]),
             "qwen3-32b-prefill": (synth.QWEN3_32B, [128])}
SAMPLER_METRIC = "ReSET sampler latency per decode step, FP32 logits [8, 151936] (entropy, state update, T, sample)"
PREFILL_METRIC = "prefill NVFP4 GEMM (M=128 tokens) µs/call and achieved HBM GB/s, Qwen3-32B shapes"
DECODE_METRIC = "Qwen3-32B-shaped decode step latency (64 NVFP4 layers + BF16 lm_head + ReSET sampler, one CUDA graph)"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="qwen3-32b", choices=sorted(WORKLOADS))
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-extras", action="store_true",
                    help="headline line only: skip per_proj, the cold per-call table, sampler and decode_step")
    ap.add_argument("--decode-steps", type=int, default=1500, help="decode_step key: graph replays per M")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--route", default="one-call", choices=["one-call", "two-call"],
                    help="sweep: nvfp4_quantize_gemv_packed per projection (one launch where it pays), or "
                         "nvfp4_quantize_act + nvfp4_gemv_smallm_packed")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="target length of the CPU oracle sample")
    ap.add_argument("--only", default=None, help="time a single call, e.g. gate_up:8 (for profiling)")
    ap.add_argument("--m", type=int, default=None, help="decode workload: the number of tokens M (1, 4 or 8)")
    ap.add_argument("--top-p", type=float, default=1.0,
                    help="sampler workload: nucleus mass (1 = no truncation; the pages' evaluation uses 0.95)")
    ap.add_argument("--threshold", default="reset", choices=["reset", "fixed", "window"],
                    help="sampler workload: the entropy-threshold policy")
    ap.add_argument("--layers", type=int, default=64, help="decode workload: decoder layers")
    ap.add_argument("--weights", default="packed", choices=["packed", "rowmajor"],
                    help="weight layout: packed (nvfp4_pack_weights, offline) or row-major codes/scales")
    return ap.parse_args()


SPEC_HBM_GBS = 8000.0      # GB300 HBM3e nominal (~8 TB/s), the second denominator


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi sampled every 200 ms while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.uuid = None
        try:
            self.uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            if not self.uuid.startswith("GPU-"):
                self.uuid = "GPU-" + self.uuid
        except Exception:
            pass
        self.proc = None
        self.out = None

    def __enter__(self):
        try:
            self.out = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200"]
            if self.uuid:
                cmd.insert(1, f"--id={self.uuid}")
            self.proc = subprocess.Popen(cmd, stdout=self.out, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if self.out is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.out.flush()
        rows = []
        with open(self.out.name) as f:
            for line in f:
                p = [x.strip() for x in line.split(",")]
                if len(p) >= 9 and p[1].isdigit():
                    rows.append(p)
        os.unlink(self.out.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [int(r[1]) for r in rows]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": int(rows[0][2]), "reasons": reasons,
                "samples": len(rows), "power_w_max": max(float(r[3]) for r in rows if r[3].replace('.', '').isdigit())}


def dist_setup(args):
    """One process per GPU (replicas: the path does not shard, so ranks share
    nothing but the barrier and the max of their timings).  NCCL on GPUs; gloo
    where there is no GPU (the host-side logic is tested that way)."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    gpu = torch.cuda.is_available()
    if gpu:
        torch.cuda.set_device(local if world > 1 else 0)
    if world > 1:
        torch.distributed.init_process_group("nccl" if gpu else "gloo")
    return world, rank


def barrier(world):
    if world > 1:
        torch.distributed.barrier()
    if torch.cuda.is_available():
        torch.cuda.synchronize()


def max_over_ranks(world, v):
    if world == 1:
        return v
    dev = "cuda" if torch.distributed.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def aggregate_gbs(world, bytes_per_step, steps, ms_max):
    """Whole-job throughput of `world` replicas that each moved bytes_per_step
    per step, over the slowest rank's time."""
    return world * bytes_per_step * steps / (ms_max * 1e-3) / 1e9


# ---------------------------------------------------------------------------
def gemv_call(api, c, w, ws, y=None):
    y = c["y"] if y is None else y
    if isinstance(w, api.NVFP4PackedWeight):
        return api.nvfp4_gemv_smallm_packed(c["xq"], w, y=y, workspace=ws)
    return api.nvfp4_gemv_smallm(c["xq"], w, y=y, workspace=ws)


def project(api, c, w, ws, route, x=None, y=None):
    """One projection of the sweep from its BF16 activation: the one-call route
    (nvfp4_quantize_gemv_packed) or the quantizer followed by the GEMV."""
    x = c["x"] if x is None else x
    if route == "one-call":
        return api.nvfp4_quantize_gemv_packed(x, w, y=c["y"] if y is None else y, workspace=ws)
    api.nvfp4_quantize_act(x, out=c["xq"])
    return gemv_call(api, c, w, ws, y=y)


def one_launch(M, N, K):
    """Whether nvfp4_quantize_gemv_packed runs this shape as one launch (the
    library's answer); used to count launches."""
    from nvfp4_w4a4_decode_gemv_gb300 import api
    return api.nvfp4_quantize_gemv_launches(M, N, K) == 1

def build_problem(shapes, Ms, rank, only=None, packed=True):
    from nvfp4_w4a4_decode_gemv_gb300 import api
    dev = torch.device("cuda")
    weights = {}
    for i, (name, K, N) in enumerate(shapes):
        g = torch.Generator(device=dev)
        g.manual_seed(1000 + i)
        wb = (torch.randn((N, K), generator=g, device=dev, dtype=torch.float32) * synth.W_STD).to(torch.bfloat16)
        weights[name] = api.nvfp4_quantize_act(wb)
        del wb
        if packed:                   # offline weight preparation, outside any timed region
            weights[name] = api.nvfp4_pack_weights(weights[name])
            torch.cuda.synchronize()
    calls = []
    for M in Ms:
        for i, (name, K, N) in enumerate(shapes):
            if only and f"{name}:{M}" != only:
                continue
            x = synth.activations(M, K, seed=100 * M + i).to(dev)
            calls.append(dict(M=M, name=name, K=K, N=N, x=x, xq=api.NVFP4Tensor.empty(M, K, dev),
                              y=torch.empty((M, N), dtype=torch.float32, device=dev),
                              gemv_bytes=synth.gemv_bytes(M, N, K), q_bytes=synth.quantize_bytes(M, K),
                              qg_bytes=synth.quantize_gemv_bytes(M, N, K)))
    ws_bytes = max(api.nvfp4_quantize_gemv_workspace_bytes(c["M"], c["N"], c["K"]) for c in calls)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=dev)
    torch.cuda.synchronize()
    return weights, calls, ws


def run_ours(args, world, rank):
    from nvfp4_w4a4_decode_gemv_gb300 import api
    shapes, Ms = WORKLOADS[args.workload]
    weights, calls, ws = build_problem(shapes, Ms, rank, args.only, packed=args.weights == "packed")
    route = args.route if args.weights == "packed" else "two-call"
    other = "two-call" if route == "one-call" else "one-call"
    groups = {}
    for c in calls:
        groups.setdefault(c["M"], []).append(c)
    order = sorted(groups)

    def gemv_all(cs):
        for c in cs:
            gemv_call(api, c, weights[c["name"]], ws)

    def step_m(cs, rt=route):        # the decode-chain order: qkv, o, gate_up, down, each from its BF16 activation
        for c in cs:
            project(api, c, weights[c["name"]], ws, rt)

    for M in order:                  # initialises kernel attributes outside capture; the quantized
        step_m(groups[M], "two-call")    # activations the GEMV-only graph reads
        if route == "one-call":
            step_m(groups[M])
    torch.cuda.synchronize()
    # The whole step (every M, decode-chain order, programmatic dependent
    # launches between the kernels) is one CUDA graph; so are the GEMV
    # launches alone (on the quantized activations), whose replays time the
    # GEMV kernel for the roofline.  Per M, a graph of its GEMVs alone gives
    # the per-M breakdown; the other route's step is a graph of its own.
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        g_step, g_gemv, g_other = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph(), None
        with torch.cuda.graph(g_step, stream=stream):
            for M in order:
                step_m(groups[M])
        if args.weights == "packed":       # the other route, timed after the main steps for comparison
            g_other = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g_other, stream=stream):
                for M in order:
                    step_m(groups[M], other)
        with torch.cuda.graph(g_gemv, stream=stream):
            for M in order:
                gemv_all(groups[M])
        ggraphs = {}
        for M in order:
            gg = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gg, stream=stream):
                gemv_all(groups[M])
            ggraphs[M] = gg
    torch.cuda.synchronize()
    ev = lambda: torch.cuda.Event(enable_timing=True)
    ev_gemv = [(ev(), ev()) for _ in range(args.steps)]
    ev_m = [[(ev(), ev()) for _ in order] for _ in range(args.steps)]
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            g_step.replay()
            g_gemv.replay()
    barrier(world)
    t0, t1 = ev(), ev()
    with ClockSampler(torch.cuda.current_device()) as clk:
        with torch.cuda.stream(stream):
            t0.record()
            for k in range(args.steps):          # the timed steps
                g_step.replay()
            t1.record()
            for k in range(args.steps):          # the GEMV kernels alone, same launches, for the roofline
                ev_gemv[k][0].record()
                g_gemv.replay()
                ev_gemv[k][1].record()
            for k in range(args.steps):          # per-M breakdown
                for i, M in enumerate(order):
                    ev_m[k][i][0].record()
                    ggraphs[M].replay()
                    ev_m[k][i][1].record()
            if g_other is not None:
                for _ in range(3):
                    g_other.replay()
                o0, o1 = ev(), ev()
                o0.record()
                for k in range(args.steps):
                    g_other.replay()
                o1.record()
        torch.cuda.synchronize()
    barrier(world)
    ms_total = max_over_ranks(world, t0.elapsed_time(t1))
    clocks = clk.summary()
    gemv_ms_total = float(np.mean([a.elapsed_time(b) for a, b in ev_gemv]))
    gemv_ms = {M: float(np.mean([ev_m[k][i][0].elapsed_time(ev_m[k][i][1]) for k in range(args.steps)]))
               for i, M in enumerate(order)}
    other_ms = o0.elapsed_time(o1) / args.steps if g_other is not None else None
    per_call = None if args.no_extras else cold_per_call(calls, weights, ws)
    proj = None if args.no_extras else per_projection(calls, weights, ws)

    route_bytes = lambda c, rt: c["qg_bytes"] if rt == "one-call" else c["gemv_bytes"] + c["q_bytes"]
    step_bytes = sum(route_bytes(c, route) for c in calls)
    value_gbs = aggregate_gbs(world, step_bytes, args.steps, ms_total)
    gemv_bytes_total = sum(c["gemv_bytes"] for c in calls)
    per_m = {f"M{M}": {"gemv_us_per_call": round(gemv_ms[M] * 1e3 / len(groups[M]), 2),
                       "gemv_gbs": round(sum(c["gemv_bytes"] for c in groups[M]) / (gemv_ms[M] * 1e-3) / 1e9, 1)}
             for M in order}
    peak, peak_kind = measured_peaks()
    cuda_cores = False                # the CUDA-core kernel is a test cross-check, not a bench path
    # the quantizer and the GEMV, or one launch of the GEMV that quantizes its activation
    launches_per_step = sum(1 if route == "one-call" and one_launch(c["M"], c["N"], c["K"]) else 2 for c in calls)
    gemv_name = ("nvfp4_gemv_smallm_packed (tensor-core GEMV kernel)" if args.weights == "packed" else
                 "nvfp4_gemv_smallm (" + ("activation-record + CUDA-core GEMV kernels" if cuda_cores
                                          else "tensor-core GEMV kernel") + ")")
    achieved = gemv_bytes_total / (gemv_ms_total * 1e-3) / 1e9
    result = {
        "metric": METRIC, "value": round(value_gbs, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_total / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "nvfp4 (e2m1 x e4m3/16 x fp32) w4a4, fp32 accumulate",
        "data": "synthetic (seeded N(0,0.02) weights; N(0,1) activations with 1% x20 outlier channels)",
        "config": {"workload": f"{args.workload} decode projections qkv/o/gate_up/down, M={Ms[0]}..{Ms[-1]}, "
                               f"quantize+GEMV per call",
                   "route": route + (" (nvfp4_quantize_gemv_packed: one launch for M <= 3, quantizer + GEMV above)"
                                     if route == "one-call" else " (nvfp4_quantize_act + nvfp4_gemv_smallm)"),
                   "bytes": "per call: weights + BF16 activation + FP32 output (one-call route); two-call "
                            "route: + the quantized activation written and read",
                   "calls_per_step": len(calls), "weights": args.weights, "weights_resident_gb": round(sum(
                       w.packed.numel() if hasattr(w, "packed") else w.codes.numel() + w.scales.numel()
                       for w in weights.values()) / 1e9, 3),
                   "l2": "inputs larger than L2: >=245 MB of other weights between two uses of one matrix",
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4),
                     "frac_spec": round(achieved / SPEC_HBM_GBS, 4), "peak_spec": SPEC_HBM_GBS,
                     "traffic": recorded_traffic(args.workload) if args.weights == "packed" and not cuda_cores else None,
                     "traffic_unit": "bytes per GEMV launch (ncu dram__bytes_read + dram__bytes_write, sweep mean)",
                     "algorithmic_bytes_per_launch": round(gemv_bytes_total / len(calls)),
                     "kernel": f"{gemv_name}: algorithmic bytes of all GEMV calls / their event-timed duration "
                               "(one graph of the step's GEMV launches alone, replayed right after the timed steps)",
                     "peak_source": f"{peak_kind} hbm_gbs"},
        "clocks": clocks,
        "gpu_launches": launches_per_step * args.steps,
        "per_m": per_m,
    }
    if other_ms is not None:
        result["other_route"] = {"route": other, "ms_per_step": round(other_ms, 4),
                                 "gbs": round(sum(route_bytes(c, other) for c in calls) / (other_ms * 1e-3) / 1e9, 1),
                                 "method": "the same step through the other route, one graph replayed after the "
                                           "timed steps"}
    if proj is not None:
        result["per_proj"] = proj
    if per_call is not None:
        result["per_call_cold_l2"] = per_call
    return result, calls, weights, ws


def _l2_bytes():
    return int(getattr(torch.cuda.get_device_properties(torch.cuda.current_device()), "L2_cache_size", 128 << 20))


def _weight_clone(api, w):
    if isinstance(w, api.NVFP4PackedWeight):
        return api.NVFP4PackedWeight(w.packed.clone(), w.global_scale, w.N, w.K)
    return api.NVFP4Tensor(w.codes.clone(), w.scales.clone(), w.global_scale)


def _weight_bytes(w):
    return w.packed.numel() if hasattr(w, "packed") else w.codes.numel() + w.scales.numel()


def per_projection(calls, weights, ws, R=64, trials=5):
    """Each (projection, M) alone: a CUDA graph of R chained GEMV calls of that
    projection (programmatic dependent launches between them, as in a decode
    chain), replayed after an L2 flush.  Call r reads weight copy r mod n, with
    n chosen so that the other copies between two uses of one copy exceed
    2x the L2 size: every call streams its weights from HBM.  A second graph
    chains quantize -> GEMV pairs, a third nvfp4_quantize_gemv_packed calls.
    Median over `trials` replays."""
    from nvfp4_w4a4_decode_gemv_gb300 import api
    peak, _ = measured_peaks()
    l2 = _l2_bytes()
    flush = torch.empty(2 * l2, dtype=torch.uint8, device="cuda")
    copies = {}
    for name, w in weights.items():
        n = 1 + -(-2 * l2 // _weight_bytes(w))
        copies[name] = [w] + [_weight_clone(api, w) for _ in range(n - 1)]
    torch.cuda.synchronize()
    stream = torch.cuda.Stream()
    out = {}
    for c in calls:
        cp = copies[c["name"]]
        graphs = {}
        with torch.cuda.stream(stream):
            for with_q in (False, True, "one"):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    for r in range(R):
                        if with_q == "one":
                            api.nvfp4_quantize_gemv_packed(c["x"], cp[r % len(cp)], y=c["y"], workspace=ws)
                            continue
                        if with_q:
                            api.nvfp4_quantize_act(c["x"], out=c["xq"])
                        gemv_call(api, c, cp[r % len(cp)], ws)
                graphs[with_q] = g
        t = {False: [], True: [], "one": []}
        with torch.cuda.stream(stream):
            for _ in range(trials):
                for with_q in (False, True, "one"):
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    flush.zero_()
                    e0.record()
                    graphs[with_q].replay()
                    e1.record()
                    e1.synchronize()
                    t[with_q].append(e0.elapsed_time(e1) * 1e3 / R)
        g_us, q_us, o_us = float(np.median(t[False])), float(np.median(t[True])), float(np.median(t["one"]))
        gbs = c["gemv_bytes"] / (g_us * 1e-6) / 1e9
        qgbs = (c["gemv_bytes"] + c["q_bytes"]) / (q_us * 1e-6) / 1e9
        out[f"{c['name']}_M{c['M']}"] = {"gemv_us": round(g_us, 3), "gemv_gbs": round(gbs, 1),
                                         "frac": round(gbs / peak, 4), "frac_spec": round(gbs / SPEC_HBM_GBS, 4),
                                         "quant_gemv_us": round(q_us, 3), "quant_gemv_gbs": round(qgbs, 1),
                                         "one_call_us": round(o_us, 3),
                                         "one_call_gbs": round(c["qg_bytes"] / (o_us * 1e-6) / 1e9, 1)}
        del graphs
    del flush, copies
    torch.cuda.synchronize()
    fr = [v["frac"] for v in out.values()]
    out["summary"] = {"min_frac": round(min(fr), 4), "mean_frac": round(float(np.mean(fr)), 4),
                      "min_frac_by_proj": {n: round(min(v["frac"] for k, v in out.items() if k.startswith(n + "_M")), 4)
                                           for n in weights},
                      "method": f"graph of {R} chained calls of one projection, weight copies rotated so that "
                                f">= 2x L2 of other weights lies between two uses of one copy; L2 flushed before "
                                f"each replay; median of {trials} replays; frac against the measured copy peak, "
                                f"frac_spec against {SPEC_HBM_GBS:.0f} GB/s"}
    return out


def prefill_summary(M=128, R=16, trials=5, only=None):
    """The prefill-sized GEMM (nvfp4_gemm_packed) on the Qwen3-32B projections
    at M = 128 tokens: per projection a graph of R chained calls over rotated
    weight copies (>= 2x L2 between two uses of one copy), L2 flushed before
    each replay, median of `trials` replays; the activation is quantized once,
    outside the timed region (the decode sweep times the quantizer)."""
    from nvfp4_w4a4_decode_gemv_gb300 import api
    peak, _ = measured_peaks()
    l2 = _l2_bytes()
    dev = torch.device("cuda")
    flush = torch.empty(2 * l2, dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream()
    out = {}
    for i, (name, K, N) in enumerate(synth.QWEN3_32B):
        if only and name != only:
            continue
        g = torch.Generator(device=dev)
        g.manual_seed(1000 + i)
        wb = (torch.randn((N, K), generator=g, device=dev, dtype=torch.float32) * synth.W_STD).to(torch.bfloat16)
        w = api.nvfp4_pack_weights(api.nvfp4_quantize_act(wb))
        del wb
        n = 1 + -(-2 * l2 // w.packed.numel())
        cps = [w] + [_weight_clone(api, w) for _ in range(n - 1)]
        X = api.nvfp4_quantize_act(synth.activations(M, K, seed=500 + i).to(dev))
        y = torch.empty((M, N), dtype=torch.float32, device=dev)
        ws = torch.zeros(api.nvfp4_gemm_workspace_bytes(M, N, K), dtype=torch.uint8, device=dev)
        with torch.cuda.stream(stream):
            api.nvfp4_gemm_packed(X, cps[0], y=y, workspace=ws)
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gr, stream=stream):
                for r in range(R):
                    api.nvfp4_gemm_packed(X, cps[r % n], y=y, workspace=ws)
            ts = []
            for _ in range(trials):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                flush.zero_()
                e0.record()
                gr.replay()
                e1.record()
                e1.synchronize()
                ts.append(e0.elapsed_time(e1) * 1e3 / R)
        us = float(np.median(ts))
        by = synth.gemv_bytes(M, N, K)
        gbs = by / (us * 1e-6) / 1e9
        out[name] = {"us": round(us, 3), "gbs": round(gbs, 1), "frac": round(gbs / peak, 4),
                     "frac_spec": round(gbs / SPEC_HBM_GBS, 4), "tflops": round(2.0 * M * N * K / (us * 1e-6) / 1e12, 1)}
        del gr, cps, w, ws
        torch.cuda.synchronize()
    del flush
    out["method"] = (f"M={M}: graph of {R} chained nvfp4_gemm_packed calls per projection over rotated weight copies, "
                     f"L2 flushed per replay, median of {trials}; bytes = weights + NVFP4 activation + FP32 y; "
                     f"frac against the measured copy peak (the GEMM is HBM-bound at M=128: ~455 flop/B)")
    return out


def cold_per_call(calls, weights, ws, R=200, trials=7):
    """us per call with L2 flushed before every call (a write of 2x the L2
    size): graphs of R x [flush + quantize + GEMV], R x [flush + quantize],
    R x [flush + GEMV] and R x [flush]; the call's time is the difference over
    R, per replay; p50 and max over `trials` replays (event clock resolution
    divided by R)."""
    from nvfp4_w4a4_decode_gemv_gb300 import api
    flush = torch.empty(2 * _l2_bytes(), dtype=torch.uint8, device="cuda")
    stream = torch.cuda.Stream()

    def capture(body):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(g, stream=stream):
                for _ in range(R):
                    flush.zero_()
                    body()
        return g

    def time_graph(g):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record()
            g.replay()
            e1.record()
        e1.synchronize()
        return e0.elapsed_time(e1) * 1e3

    g_flush = capture(lambda: None)
    out = {}
    for c in calls:
        w = weights[c["name"]]
        q = lambda: api.nvfp4_quantize_act(c["x"], out=c["xq"])
        gv = lambda: gemv_call(api, c, w, ws)
        gs = {"flush": g_flush, "q": capture(q), "qg": capture(lambda: (q(), gv())), "g": capture(gv)}
        tt = {k: [] for k in gs}
        for _ in range(trials):
            for k, g in gs.items():
                tt[k].append(time_graph(g))
        f = np.array(tt["flush"])
        quant = (np.array(tt["q"]) - f) / R
        gemv_chain = (np.array(tt["qg"]) - np.array(tt["q"])) / R
        gemv_alone = (np.array(tt["g"]) - f) / R
        ga = float(np.median(gemv_alone))
        out[f"{c['name']}_M{c['M']}"] = {
            "gemv_us": round(ga, 3), "gemv_us_max": round(float(gemv_alone.max()), 3),
            "gemv_gbs": round(c["gemv_bytes"] / (ga * 1e-6) / 1e9, 1),
            "quant_us": round(float(np.median(quant)), 3), "quant_us_max": round(float(quant.max()), 3),
            "gemv_after_quant_us": round(float(np.median(gemv_chain)), 3)}
        del gs
    del g_flush, flush
    torch.cuda.synchronize()
    out["method"] = (f"graphs of {R} x [L2 flush (2x L2 write) + call] minus {R} x [flush]; median (p50) and max "
                     f"over {trials} replays; gemv_us = a lone GEMV, gemv_after_quant_us = the GEMV behind its "
                     f"quantizer (programmatic dependent launch)")
    return out


def run_e2e(args, calls, weights, ws, world=1):
    """The step end to end through the public API, with the step's activations
    arriving in one copy from pinned host memory and its outputs leaving in one
    copy to pinned host memory, every step's copies inside the timed region.
    The step's API calls (one per projection on the one-call route, two on the
    two-call route) are captured once in a CUDA graph, as a decode loop runs
    them.  `value`: two sets of device buffers and three streams, so that
    step i's copies overlap steps i - 1 and i + 1's compute (copy in, compute
    and copy out of one step stay ordered by events, and a set is reused only
    after its previous step's copy out); `serial`: copy in, replay, copy out
    on one stream; `eager`: the same calls issued one by one from Python each
    step, serially.  (One copy per M group on a second stream, overlapped with
    the other groups' compute, measured slower: 1.21 against 0.74 ms per step.)"""
    from nvfp4_w4a4_decode_gemv_gb300 import api
    dev = calls[0]["x"].device
    # one arena per direction and buffer set; every piece is a multiple of 512
    # bytes, so each view stays 16-byte aligned
    x_sizes = [c["x"].numel() for c in calls]
    y_sizes = [c["y"].numel() for c in calls]
    host_x = torch.cat([c["x"].reshape(-1).cpu() for c in calls]).pin_memory()
    sets = []
    for _ in range(2):
        xa = torch.empty(sum(x_sizes), dtype=torch.bfloat16, device=dev)
        ya = torch.empty(sum(y_sizes), dtype=torch.float32, device=dev)
        hy = torch.empty(sum(y_sizes), dtype=torch.float32).pin_memory()
        xv = [v.view(c["x"].shape) for v, c in zip(torch.split(xa, x_sizes), calls)]
        yv = [v.view(c["y"].shape) for v, c in zip(torch.split(ya, y_sizes), calls)]
        sets.append((xa, ya, hy, xv, yv))

    route = args.route if args.weights == "packed" else "two-call"

    def compute(b):
        _, _, _, xv, yv = sets[b]
        for j, c in enumerate(calls):
            project(api, c, weights[c["name"]], ws, route, x=xv[j], y=yv[j])

    expected = torch.cat([c["y"].reshape(-1) for c in calls]).cpu()

    def check(bufs):
        for b in bufs:
            _, ya, hy, _, _ = sets[b]
            if not torch.equal(ya.cpu(), expected):
                raise RuntimeError("end-to-end step disagrees with the device-resident step")
            if not torch.equal(hy, expected):
                raise RuntimeError("end-to-end outputs did not all reach the host")

    s_in, s_comp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    step_bytes = sum(c["qg_bytes"] if route == "one-call" else c["gemv_bytes"] + c["q_bytes"] for c in calls)
    out = {}
    graphs = []
    with torch.cuda.stream(s_comp):
        for b in range(2):
            sets[b][0].copy_(host_x, non_blocking=True)
            for _ in range(3):
                compute(b)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s_comp):
                compute(b)
            graphs.append(g)
    torch.cuda.synchronize()

    def timed(run_steps, first, last):
        for _ in range(max(3, args.warmup)):
            run_steps(1)
        torch.cuda.synchronize()
        barrier(world)
        for b in range(2):
            sets[b][2].zero_()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(first):
            t0.record()
        run_steps(args.steps)
        with torch.cuda.stream(last):
            t1.record()
        t1.synchronize()
        torch.cuda.synchronize()
        barrier(world)
        ms = max_over_ranks(world, t0.elapsed_time(t1))      # the whole job: every rank's bytes, the slowest time
        return {"value": round(aggregate_gbs(world, step_bytes, args.steps, ms), 1), "unit": "GB/s",
                "ms_per_step": round(ms / args.steps, 4)}

    # serial: one stream, set 0 (eager: the calls from Python; graph: replay)
    for mode in ("eager", "serial"):
        def run_serial(n, mode=mode):
            xa, ya, hy, _, _ = sets[0]
            with torch.cuda.stream(s_comp):
                for _ in range(n):
                    xa.copy_(host_x, non_blocking=True)
                    if mode == "serial":
                        graphs[0].replay()
                    else:
                        compute(0)
                    hy.copy_(ya, non_blocking=True)
        out[mode] = timed(run_serial, s_comp, s_comp)
        check([0])

    # pipelined: step i on set i % 2; its copy in waits for the set's previous
    # compute, its compute for its copy in and the set's previous copy out
    ev_in = [torch.cuda.Event(), torch.cuda.Event()]
    ev_comp = [torch.cuda.Event(), torch.cuda.Event()]
    ev_out = [torch.cuda.Event(), torch.cuda.Event()]
    for b in range(2):
        for ev in (ev_comp[b], ev_out[b]):
            with torch.cuda.stream(s_comp):
                ev.record()
    step_no = [0]

    def run_pipelined(n):
        for _ in range(n):
            b = step_no[0] % 2
            step_no[0] += 1
            xa, ya, hy, _, _ = sets[b]
            with torch.cuda.stream(s_in):
                s_in.wait_event(ev_comp[b])
                xa.copy_(host_x, non_blocking=True)
                ev_in[b].record()
            with torch.cuda.stream(s_comp):
                s_comp.wait_event(ev_in[b])
                s_comp.wait_event(ev_out[b])
                graphs[b].replay()
                ev_comp[b].record()
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_comp[b])
                hy.copy_(ya, non_blocking=True)
                ev_out[b].record()
    out["pipelined"] = timed(run_pipelined, s_in, s_out)
    check([0, 1])
    del graphs
    torch.cuda.synchronize()
    return {"value": out["pipelined"]["value"], "unit": "GB/s", "ms_per_step": out["pipelined"]["ms_per_step"],
            "h2d_bytes_per_step": int(host_x.numel() * host_x.element_size()) * world,     # all ranks
            "d2h_bytes_per_step": int(sets[0][2].numel() * sets[0][2].element_size()) * world,
            "method": f"per step: pinned host->device copy of the activations, the step's {len(calls)} projections "
                      f"({route} route; API calls captured once in a CUDA graph, replayed), device->host copy of "
                      f"all outputs; two buffer sets on three streams so one step's copies overlap its neighbours' "
                      f"compute; every rank's bytes over the slowest rank's time",
            "serial": out["serial"], "eager": out["eager"]}


def decode_stage_times(st, stream, reps=20):
    """Per-launch time of the decode step's non-projection stages, each launched
    `reps` times back to back (with programmatic dependent launch between
    them, as in the step) between two events on the step's stream.  Inputs are
    the step's own buffers, so these are L2-warm figures; the weight-streaming
    projections are measured by the sweep."""
    from nvfp4_w4a4_decode_gemv_gb300 import api
    M = st.M
    calls = {
        "rms_norm_quantize": lambda: api.nvfp4_rms_norm_quantize(st.h, eps=st.eps, out=st.xq, stream=stream),
        "quantize_f32_query_slice": lambda: api.nvfp4_quantize_f32(st.y_qkv, K=st.k_o, out=st.xq_o, stream=stream),
        "silu_mul_quantize": lambda: api.nvfp4_silu_mul_quantize(st.y_gu, out=st.xq_d, stream=stream),
        "rms_norm_bf16": lambda: api.nvfp4_rms_norm_bf16(st.h, eps=st.eps, out=st.r, stream=stream),
        "lm_head_bf16_gemv_tc": lambda: api.nvfp4_bf16_gemv_tc(st.r, st.lm_head, y=st.logits, workspace=st.ws,
                                                                stream=stream),
        "reset_sample": lambda: st.sampler(st.logits, st.step_start, st.u, stream=stream),
    }
    out = {}
    with torch.cuda.stream(stream):
        for name, fn in calls.items():
            for _ in range(3):
                fn()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            for _ in range(reps):
                fn()
            b.record()
            torch.cuda.synchronize()
            out[name] = round(a.elapsed_time(b) * 1e3 / reps, 2)
    out["lm_head_gbs"] = round(st.lm_head.numel() * 2 / (out["lm_head_bf16_gemv_tc"] * 1e-6) / 1e9, 1)
    out["note"] = f"M={M}; each stage {reps}x back to back, L2-warm inputs"
    return out


def run_decode(args, world, rank):
    """The synthetic decode step: `--layers` layers of the four projections,
    the lm_head and the sampler, captured as one CUDA graph and replayed
    `--steps` times (per-step latency)."""
    from nvfp4_w4a4_decode_gemv_gb300.decode_step import DecodeStep
    M = args.m or 1
    st = DecodeStep(M=M, layers=args.layers, seed=rank)
    st.h_in.copy_(synth.activations(M, st.hidden, seed=100 + M).float().cuda())
    us = torch.from_numpy(synth.reset_uniforms(args.steps + args.warmup + 1, M)).cuda()
    st.u.copy_(us[0])
    st.run()                         # sets kernel attributes outside the capture
    torch.cuda.synchronize()
    g = st.capture()
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            st.u.copy_(us[1 + i], non_blocking=True)
            g.replay()
    torch.cuda.synchronize()
    barrier(world)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    with ClockSampler(torch.cuda.current_device()) as clk:
        with torch.cuda.stream(stream):
            for i in range(args.steps):
                st.u.copy_(us[1 + args.warmup + i], non_blocking=True)
                evs[i][0].record()
                g.replay()
                evs[i][1].record()
        torch.cuda.synchronize()
    barrier(world)
    ms = np.array([a.elapsed_time(b) for a, b in evs])
    ms_mean = max_over_ranks(world, float(ms.mean()))
    # End to end: every step copies its inputs (hidden state, uniforms) in from
    # pinned host memory, replays the step and copies the tokens, entropies and
    # temperatures back.
    host_h = st.h_in.cpu().pin_memory()
    host_u = us.cpu().pin_memory()
    host_out = torch.empty(3 * M, dtype=torch.int32).pin_memory()
    outs = (st.sampler.token, st.sampler.H.view(torch.int32), st.sampler.T.view(torch.int32))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record()
        for i in range(args.steps):
            st.h_in.copy_(host_h, non_blocking=True)
            st.u.copy_(host_u[1 + args.warmup + i], non_blocking=True)
            g.replay()
            for k, t in enumerate(outs):
                host_out[k * M:(k + 1) * M].copy_(t, non_blocking=True)
        e1.record()
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(world, e0.elapsed_time(e1) / args.steps)
    stages = decode_stage_times(st, stream)
    weight_bytes = sum(w.packed.numel() for layer in st.weights for w in layer.values())
    step_bytes = weight_bytes + st.lm_head.numel() * 2 + st.logits.numel() * 4 * 2
    peak, peak_kind = measured_peaks()
    return {
        "metric": DECODE_METRIC, "value": round(ms_mean, 4), "unit": "ms/step", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_mean, 4), "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "nvfp4 w4a4 projections, bf16 lm_head, fp32 sampler",
        "data": "synthetic (seeded random weights; fixed N(0,1) input hidden state; seeded uniforms)",
        "config": {"workload": f"qwen3-32b decode step, M={M}, {args.layers} layers, lm_head 5120->151936, "
                               f"ReSET sampler", "parallelism": f"replicas x{world}"},
        "p50_ms": round(float(np.percentile(ms, 50)), 4), "p99_ms": round(float(np.percentile(ms, 99)), 4),
        "tokens_per_s": round(world * M * 1000.0 / ms_mean, 1),
        "roofline": {"bound": "hbm", "achieved": round(step_bytes / (ms_mean * 1e-3) / 1e9, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(step_bytes / (ms_mean * 1e-3) / 1e9 / peak, 4), "traffic": None,
                     "kernel": "whole step: weight, lm_head and logits bytes / step time",
                     "peak_source": f"{peak_kind} hbm_gbs"},
        "e2e": {"value": round(e2e_ms, 4), "unit": "ms/step", "h2d_bytes_per_step": host_h.numel() * 4 + M * 4,
                "d2h_bytes_per_step": 3 * M * 4},
        "stages_us": stages,
        "clocks": clk.summary(),
        "gpu_launches": (args.layers * 8 + 3) * args.steps,   # per layer: 2 norm+quantize, 2 quantizers, 4 GEMVs
    }


def sampler_workload(args) -> str:
    text = f"reset sampler, M=8, V={synth.LM_HEAD_VOCAB}, w=8, tau0=0.6, T=0.3/1.0"
    if args.threshold != "reset":
        text += f", {args.threshold} threshold"
    if args.top_p < 1.0:
        text += f", top-p {args.top_p:g}"
    return text


def run_sampler(args, world, rank):
    """The sampler workload: M = 8 rows over the 151936-token vocabulary, one
    step per iteration.  Each step's logits are generated on the device from
    the seeded generator (sigma per step from {1, 3, 8}), then L2 is flushed,
    then the sampler call alone is timed with events (its first pass reads the
    logits from HBM)."""
    from nvfp4_w4a4_decode_gemv_gb300 import api
    dev = torch.device("cuda")
    M, V = 8, synth.LM_HEAD_VOCAB
    total = args.warmup + args.steps
    sig = synth.reset_sigmas(total)
    starts = torch.from_numpy(synth.reset_boundaries(total, M)).to(dev)
    us = torch.from_numpy(synth.reset_uniforms(total, M)).to(dev)
    sampler = api.ResetSampler(M, V, 0.6, 0.3, 1.0, 8, device=dev, threshold=args.threshold, top_p=args.top_p)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    logits = torch.empty((M, V), dtype=torch.float32, device=dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(total)]
    barrier(world)
    with ClockSampler(torch.cuda.current_device()) as clk:
        for i in range(total):
            logits.copy_(synth.reset_logits(i + 1000 * rank, M, V, float(sig[i]), device=dev))
            flush.zero_()
            ev[i][0].record()
            sampler(logits, starts[i], us[i])
            ev[i][1].record()
        torch.cuda.synchronize()
    barrier(world)
    ms = np.array([a.elapsed_time(b) for a, b in ev[args.warmup:]])
    ms_mean = max_over_ranks(world, float(ms.mean()))
    first_pass = 4 * M * V
    peak, peak_kind = measured_peaks()
    gbs = first_pass / (ms_mean * 1e-3) / 1e9
    return {
        "metric": SAMPLER_METRIC, "value": round(ms_mean * 1e3, 2), "unit": "us/step", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_mean, 4), "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "fp32 (entropy and sample), integer masses (top-p), fp64 (state sums)",
        "data": "synthetic (seeded N(0, sigma) logits per step, sigma in {1,3,8}; geometric step boundaries; "
                "PCG64 uniforms)",
        "config": {"workload": sampler_workload(args),
                   "l2": "flushed before every timed call (256 MB write)", "parallelism": f"replicas x{world}"},
        "p50_us": round(float(np.percentile(ms, 50)) * 1e3, 2), "p99_us": round(float(np.percentile(ms, 99)) * 1e3, 2),
        "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(gbs / peak, 4), "traffic": None,
                     "kernel": "reset_cluster_kernel (one thread-block cluster per row" +
                               (", top-p inside" if args.top_p < 1.0 else "") +
                               "): first-pass logits bytes (4 M V) / call time; latency-bound",
                     "peak_source": f"{peak_kind} hbm_gbs"},
        "e2e": {"value": round(ms_mean * 1e3, 2), "unit": "us/step", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0, "note": "device-resident logits, as the lm_head leaves them"},
        "clocks": clk.summary(),
        "gpu_launches": args.steps,                 # one cluster launch per call (V <= 262144)
    }


def sampler_summary(top_p, n=200, trials=3):
    """The sampler workload (M = 8 rows x 151936 logits, sigma per step from
    {1, 3, 8}, geometric step boundaries, PCG64 uniforms), n calls each on its
    own logits (all resident, 0.97 GB), L2 flushed (2x L2 write) before every
    call.  Mean: a graph of n x [flush + call] minus n x [flush], median of
    `trials` replays.  p50 / p99: n eager calls, each between its own two events
    (resolution of the event clock, ~2 us)."""
    from nvfp4_w4a4_decode_gemv_gb300 import api
    dev = torch.device("cuda")
    M, V = 8, synth.LM_HEAD_VOCAB
    sig = synth.reset_sigmas(n)
    logits = torch.empty((n, M, V), dtype=torch.float32, device=dev)
    for i in range(n):
        logits[i].copy_(synth.reset_logits(i, M, V, float(sig[i]), device=dev))
    starts = torch.from_numpy(synth.reset_boundaries(n, M)).to(dev)
    us = torch.from_numpy(synth.reset_uniforms(n, M)).to(dev)
    sampler = api.ResetSampler(M, V, 0.6, 0.3, 1.0, 8, device=dev, top_p=top_p)
    flush = torch.empty(2 * _l2_bytes(), dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        for i in range(3):
            sampler(logits[i], starts[i], us[i])
        g_s, g_f = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_s, stream=stream):
            for i in range(n):
                flush.zero_()
                sampler(logits[i], starts[i], us[i])
        with torch.cuda.graph(g_f, stream=stream):
            for i in range(n):
                flush.zero_()
    torch.cuda.synchronize()
    ts, tf = [], []
    with torch.cuda.stream(stream):
        for _ in range(trials):
            for g, acc in ((g_s, ts), (g_f, tf)):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                g.replay()
                e1.record()
                e1.synchronize()
                acc.append(e0.elapsed_time(e1) * 1e3)
    mean_us = float(np.median((np.array(ts) - np.array(tf)) / n))
    single = []
    with torch.cuda.stream(stream):
        for i in range(n):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            flush.zero_()
            e0.record()
            sampler(logits[i], starts[i], us[i])
            e1.record()
            e1.synchronize()
            single.append(e0.elapsed_time(e1) * 1e3)
    del logits, flush, g_s, g_f
    torch.cuda.synchronize()
    peak, _ = measured_peaks()
    gbs = 4 * M * V / (mean_us * 1e-6) / 1e9
    return {"workload": f"M={M}, V={V}, w=8, tau0=0.6, T=0.3/1.0" + (f", top-p {top_p:g}" if top_p < 1 else ""),
            "us_mean": round(mean_us, 2), "us_p50": round(float(np.percentile(single, 50)), 2),
            "us_p99": round(float(np.percentile(single, 99)), 2), "calls": n,
            "launches_per_call": 1,
            "first_pass_gbs": round(gbs, 1), "frac": round(gbs / peak, 4),
            "method": f"mean: graph of {n} x [L2 flush + call] minus {n} x [flush], median of {trials}; "
                      f"p50/p99: {n} single calls between events (~2 us event-clock resolution)"}


def decode_summary(args, Ms=(1, 4, 8), warmup=20):
    """The synthetic Qwen3-32B-shaped decode step (64 layers of the four NVFP4
    projections with their quantizers, BF16 lm_head, ReSET sampler) as one CUDA
    graph per M, replayed args.decode_steps times, each replay between two
    events; one model's weights serve every M."""
    from nvfp4_w4a4_decode_gemv_gb300.decode_step import DecodeStep
    peak, _ = measured_peaks()
    base, out = None, {}
    steps = args.decode_steps
    for M in Ms:
        st = DecodeStep(M=M, layers=args.layers, share_weights=base)
        base = base or st
        st.h_in.copy_(synth.activations(M, st.hidden, seed=100 + M).float().cuda())
        us = torch.from_numpy(synth.reset_uniforms(steps + warmup, M)).cuda()
        st.u.copy_(us[0])
        st.run()
        torch.cuda.synchronize()
        g = st.capture()
        stream = torch.cuda.Stream()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        with torch.cuda.stream(stream):
            for i in range(warmup):
                st.u.copy_(us[i], non_blocking=True)
                g.replay()
            for i in range(steps):
                st.u.copy_(us[warmup + i], non_blocking=True)
                evs[i][0].record()
                g.replay()
                evs[i][1].record()
        torch.cuda.synchronize()
        ms = np.array([a.elapsed_time(b) for a, b in evs])
        weight_bytes = sum(w.packed.numel() for layer in st.weights for w in layer.values())
        step_bytes = weight_bytes + st.lm_head.numel() * 2 + st.logits.numel() * 4 * 2
        gbs = step_bytes / (ms.mean() * 1e-3) / 1e9
        out[f"M{M}"] = {"ms_mean": round(float(ms.mean()), 4), "ms_p50": round(float(np.percentile(ms, 50)), 4),
                        "ms_p99": round(float(np.percentile(ms, 99)), 4), "tokens_per_s": round(M * 1e3 / ms.mean(), 1),
                        "gbs": round(gbs, 1), "frac": round(gbs / peak, 4)}
        del g, st.graph
    out["method"] = (f"{args.layers} layers + lm_head 5120->151936 + ReSET sampler as one CUDA graph; {steps} replays "
                     f"per M after {warmup} warm-up replays, each between two events; frac = (NVFP4 weight + BF16 "
                     f"lm_head + 2 x logits bytes) / mean step time / measured copy peak")
    del base
    torch.cuda.synchronize()
    return out


# ---------------------------------------------------------------------------
def cpu_oracle_sample(args, seconds):
    """The oracle as it stands, on the host: per call, quantize the activation
    and multiply against a sample of pre-quantized weight rows (FP64 dequant +
    matmul), cycling through the workload's (M, projection) calls until about
    `seconds` of CPU time.  Returns (GB/s of algorithmic bytes, sample text, threads)."""
    from oracle import nvfp4 as Q
    shapes, Ms = WORKLOADS[args.workload]
    rows = 128
    prepared = {}
    for i, (name, K, N) in enumerate(shapes):
        w = synth.weights(rows, K, seed=1000 + i)
        prepared[name] = Q.quantize_bf16(synth.bf16_bits(w))
    xs = {(M, name): synth.bf16_bits(synth.activations(M, K, seed=100 * M + i))
          for M in Ms for i, (name, K, N) in enumerate(shapes)}
    done_bytes, calls = 0, 0
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < seconds:
        for M in Ms:
            for name, K, N in shapes:
                xq, xsc, xg = Q.quantize_bf16(xs[(M, name)])
                wq, wsc, wg = prepared[name]
                Q.gemv(xq, xsc, xg, wq, wsc, wg)
                done_bytes += synth.gemv_bytes(M, rows, K) + synth.quantize_bytes(M, K)
                calls += 1
    dt = time.perf_counter() - t0
    threads = torch.get_num_threads()
    try:
        import threadpoolctl
        info = threadpoolctl.threadpool_info()
        threads = max([i.get("num_threads", 1) for i in info] + [1])
    except Exception:
        pass
    sample = (f"{calls} calls of the {args.workload} sweep (M={Ms[0]}..{Ms[-1]} x 4 projections), each: oracle "
              f"quantize of the BF16 activation + FP64 GEMV against {rows} pre-quantized weight rows; {dt:.1f} s")
    return done_bytes / dt / 1e9, sample, threads, dt


def cpu_sampler_sample(args, seconds):
    """The oracle sampler as it stands, on the host: per step, for the 8 rows,
    the FP64 entropy, the ReSET update and the FP64 inverse-CDF sample, over
    the same seeded logits as the GPU workload, until about `seconds`."""
    from oracle import reset as R
    M, V = 8, synth.LM_HEAD_VOCAB
    p = R.ResetParams(tau0=0.6, t_low=0.3, t_high=1.0, w=8, threshold=args.threshold,
                      top_p=float(np.float32(args.top_p)))
    total = max(1, args.warmup + args.steps)
    sig = synth.reset_sigmas(total)
    starts = synth.reset_boundaries(total, M)
    us = synth.reset_uniforms(total, M)
    states = [R.RowState(w=8) for _ in range(M)]
    t0 = time.perf_counter()
    done = 0
    while time.perf_counter() - t0 < seconds:
        t = done % total
        ln = synth.reset_logits(t, M, V, float(sig[t])).numpy().astype(np.float64)
        for r in range(M):
            res = R.reset_update(states[r], R.token_entropy(ln[r]), bool(starts[t, r]), p)
            R.sample_inverse_cdf(ln[r], res.T, float(us[t, r]), p.top_p)
        done += 1
    dt = time.perf_counter() - t0
    return dt / done * 1e6, f"{done} steps of the reset-sampler workload (M={M}, V={V}); {dt:.1f} s"


def main():
    args = parse()
    world, rank = dist_setup(args)
    if args.impl == "reference" and args.workload == "reset-sampler":
        if rank != 0:
            return
        us_step, sample = cpu_sampler_sample(args, seconds=max(5.0, min(60.0, args.cpu_seconds)))
        threads = torch.get_num_threads()
        line = {"metric": SAMPLER_METRIC, "value": round(us_step, 1), "unit": "us/step", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(us_step / 1e3, 4),
                "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
                "dtype": "f64 (oracle entropy and inverse-CDF sample)", "data": "synthetic", "impl": "reference",
                "config": {"workload": sampler_workload(args)},
                "cpu_baseline": {"value": round(us_step, 1), "unit": "us/step", "cores": threads, "kind": "oracle",
                                 "sample": sample},
                "e2e": {"value": round(us_step, 1), "unit": "us/step", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return
    if args.impl == "reference":
        if rank != 0:
            return
        gbs, sample, threads, dt = cpu_oracle_sample(args, seconds=max(5.0, min(60.0, args.cpu_seconds)))
        _, Ms = WORKLOADS[args.workload]
        line = {"metric": METRIC, "value": round(gbs, 4), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": None, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f64 (oracle: FP32 quantize recipe, FP64 dequant and dot)",
                "data": "synthetic", "impl": "reference",
                "config": {"workload": f"{args.workload} decode projections qkv/o/gate_up/down, M={Ms[0]}..{Ms[-1]}, "
                                       f"quantize+GEMV per call"},
                "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                                 "sample": sample},
                "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return
    if args.workload == "qwen3-32b-prefill":
        if args.impl == "reference" or world > 1:
            if rank == 0:
                print(json.dumps({"impl": args.impl, "unavailable": "the prefill workload is measured on one GPU, "
                                                                     "for our kernel only"}))
            return
        res = prefill_summary(only=args.only, trials=max(3, args.steps))
        names = [k for k in res if k != "method"]
        by = sum(synth.gemv_bytes(128, N, K) for n, K, N in synth.QWEN3_32B if n in names)
        us = sum(res[n]["us"] for n in names)
        peak, peak_kind = measured_peaks()
        gbs = by / (us * 1e-6) / 1e9
        print(json.dumps({"metric": PREFILL_METRIC, "value": round(gbs, 1), "unit": "GB/s", "n_gpus": 1,
                          "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(us / 1e3, 4),
                          "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                          "dtype": "nvfp4 w4a4, fp32 accumulate", "data": "synthetic",
                          "config": {"workload": "qwen3-32b prefill projections at M=128: " + ",".join(names)},
                          "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s",
                                       "frac": round(gbs / peak, 4), "traffic": None,
                                       "peak_source": f"{peak_kind} hbm_gbs"},
                          "per_proj": res, "gpu_launches": 16 * len(names) * max(3, args.steps)}))
        return
    if args.workload in ("qwen3-32b-decode", "reset-sampler"):
        line = (run_decode if args.workload == "qwen3-32b-decode" else run_sampler)(args, world, rank)
        if rank == 0 and args.workload == "reset-sampler" and not args.no_cpu_baseline:
            us_step, sample = cpu_sampler_sample(args, seconds=args.cpu_seconds)
            line["cpu_baseline"] = {"value": round(us_step, 1), "unit": "us/step", "cores": torch.get_num_threads(),
                                    "kind": "oracle", "sample": sample}
        if rank == 0:
            print(json.dumps(line))
        if world > 1:
            torch.distributed.destroy_process_group()
        return
    result, calls, weights, ws = run_ours(args, world, rank)
    if not args.no_e2e:
        result["e2e"] = run_e2e(args, calls, weights, ws, world)
    if not args.no_extras and args.workload == "qwen3-32b":
        del calls, weights, ws
        torch.cuda.synchronize()
        result["sampler"] = {"plain": sampler_summary(1.0), "top_p_0.95": sampler_summary(0.95)}
        result["decode_step"] = decode_summary(args)
        result["prefill_m128"] = prefill_summary()
    if rank == 0:
        if not args.no_cpu_baseline:
            gbs, sample, threads, _ = cpu_oracle_sample(args, seconds=args.cpu_seconds)
            result["cpu_baseline"] = {"value": round(gbs, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                                      "sample": sample}
        print(json.dumps(result))
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
