#!/usr/bin/env python
"""Throughput of the token-choice MoE layer forward on B300, one JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload mixtral] [--T 16384] [--no-cpu-baseline]

A step is one moe_layer_forward (router, dispatch, stats, gather, expert up
and down projections, shared expert when present, combine) over one batch of
T synthetic tokens of the named workload (default: the Mixtral-8x7B-shaped
layer, d=4096, E=8, k=2, SwiGLU d_ff=14336, bf16, T=16384), inputs resident
in HBM.  The weights (2.8 GB) are larger than L2, so every step streams them
from HBM; no L2 flush is needed.  By default each step is one replay of a
CUDA graph holding one captured moe_layer_forward (--launch eager calls the
C ABI directly instead); the graph removes host launch gaps, not work.

Metric: tokens/s over the whole job (all ranks).  Under torchrun each rank
runs its own batch on its own GPU (weak scaling, no collective on the data
path); the time is the max over ranks.

Extra keys: roofline of the dominant kernel (the grouped up projection,
timed live with CUDA events around it on the launching stream), the layer's
own roofline fraction, per-stage times, e2e (host buffers through the public
LayerPipeline, every step's H2D and D2H copies inside the timed region,
overlapping the layer on the neighbouring steps), clocks sampled during
the timed region, gpu_launches counted by the library, and cpu_baseline (the
fp64 oracle on a bounded sample, on the host cores).

--impl reference times the oracle (the only other implementation of the
layer) on the host cores, each step a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import moe_inputs as mi  # noqa: E402

FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def algorithmic(w, T, n_kept, counts_nonzero):
    """Work the method itself must do (dense work it avoids is not counted).

    FLOPs: router 2*d*E per token + per kept (token, slot) 2*m*d*F (m = 3
    SwiGLU, 2 ReLU) + shared 6*d*Fs per token.  Bytes: weights of experts with
    at least one token, shared weights, W_r, x read once, y written once
    (bf16)."""
    d, E, F, Fs = w.d_model, w.n_experts, w.d_ff, w.d_ff_shared
    m = 3 if w.act == "swiglu" else 2
    eb = 2 if w.dtype == "bf16" else 4
    flops = 2.0 * d * E * T + 2.0 * m * d * F * n_kept + 6.0 * d * Fs * T
    bytes_ = (m * d * F * eb) * counts_nonzero + 3 * d * Fs * eb + 4 * d * E + 2 * T * d * eb
    up_flops = 2.0 * d * F * n_kept * (2 if w.act == "swiglu" else 1)
    # up projection alone: its weights (W1, W3) of the active experts, its
    # input rows and its output h
    up_bytes = ((2 if w.act == "swiglu" else 1) * d * F * eb * counts_nonzero
                + n_kept * d * eb + n_kept * F * eb)
    return flops, bytes_, up_flops, up_bytes


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        sms, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sms.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sms) if sms else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sms)}


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v, world, device="cuda"):
    """The slowest rank's time (the job's time)."""
    if world == 1:
        return v
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world, tokens_per_rank, steps, ms):
    """Tokens/s of the whole job: every rank's tokens over the slowest rank's time."""
    return world * tokens_per_rank * steps / (ms / 1e3)


# --------------------------------------------------------------------------- oracle timing

def oracle_sample_run(w, inp_cpu64, S):
    """The oracle as it stands on a batch of the first S tokens."""
    import oracle.moe_oracle as om
    sub = dict(inp_cpu64)
    sub["x"] = inp_cpu64["x"][:S]
    t0 = time.perf_counter()
    if w.routing == "expert":
        om.moe_forward_expert_choice(sub, w.top_k, w.act, w.capacity_factor, None, w.dtype)
    else:
        om.moe_forward(sub, w.top_k, w.act, w.capacity_factor, "probs", w.quantile_balance,
                       None, w.dtype, reroute_rounds=w.reroute_rounds)
    return time.perf_counter() - t0


def host_inputs_f64(inp):
    """Widen the generated inputs to float64 numpy once (input preparation)."""
    out = {}
    for k, v in inp.items():
        if v is None:
            out[k] = None
        else:
            out[k] = v.detach().float().cpu().numpy().astype(np.float64)
    return out


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 0) for i in threadpool_info() if i.get("user_api") == "blas"]
        return max(n) if n else os.cpu_count()
    except Exception:
        return os.cpu_count()


def calibrated_sample(w, inp64, T, target_s):
    """Tokens S for which one oracle run on the first S tokens takes about
    target_s seconds on this host: a line t = a + b S through timed runs at
    8 and 32 tokens, capped at T."""
    s1, s2 = min(T, 8), min(T, 32)
    oracle_sample_run(w, inp64, s1)
    t1 = oracle_sample_run(w, inp64, s1)
    if s2 == s1:
        return s1
    t2 = oracle_sample_run(w, inp64, s2)
    b = max((t2 - t1) / (s2 - s1), 1e-9)
    a = max(t1 - b * s1, 0.0)
    return int(max(s1, min(T, (target_s - a) / b)))


# --------------------------------------------------------------------------- arms

def run_reference(args, w, T):
    # Under torchrun only rank 0 times the oracle; the other ranks exit at once.
    if int(os.environ.get("RANK", "0")) != 0:
        return
    # each step a bounded sample: about 4 s, so that warm-up and timed steps
    # end within a few minutes
    inp = mi.generate(w, T, "cpu")
    inp64 = host_inputs_f64(inp)
    S = calibrated_sample(w, inp64, T, 4.0)
    for _ in range(args.warmup):
        oracle_sample_run(w, inp64, S)
    times = [oracle_sample_run(w, inp64, S) for _ in range(args.steps)]
    total = sum(times)
    value = S * args.steps / total
    cores = blas_threads()
    line = {
        "impl": "reference", "metric": "MoE-layer fwd tokens/s on 1 B300 (bf16) and % of roofline",
        "value": value, "unit": "tokens/s", "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": f"{w.name}-shaped layer d={w.d_model} E={w.n_experts} "
                               f"k={w.top_k} d_ff={w.d_ff} T={T}", "sample_tokens": S},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"first {S} tokens of the T={T} batch as one batch "
                                   "(routing, dispatch, stats, FFN, combine), per step"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def source_hash(text):
    """First 16 hex digits of the SHA-256 of a C++ source without its //
    comments, trailing blanks and blank lines (code edits change it,
    comment edits do not)."""
    lines = []
    for line in text.splitlines():
        i = line.find("//")
        if i >= 0:
            line = line[:i]
        line = line.rstrip()
        if line:
            lines.append(line)
    return hashlib.sha256("\n".join(lines).encode()).hexdigest()[:16]


def traffic_record(kernel_file):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current source of the kernel."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.md")
    if not os.path.exists(path):
        return None
    with open(os.path.join(ROOT, "sparse_mixture_experts_47_b300", "csrc", kernel_file)) as f:
        h = source_hash(f.read())
    recs = []
    for line in open(path):
        line = line.strip()
        if line.startswith("{") and line.endswith("}"):
            try:
                r = json.loads(line)
            except ValueError:
                continue
            if r.get("source_sha256_16") == h:
                recs.append(r)
    return recs


def stage_pass(moe, cfg, inp, weights, ws, outs, args, use_graph, dev, reps=None):
    """Summed per-stage milliseconds over `reps` layer calls, and the number
    of calls.  Graph mode captures one call with stage events on and reads
    the events after each replay; eager mode times `reps` eager calls."""
    reps = reps or max(3, min(args.steps, 10))
    if use_graph:
        moe.stage_timing(True)
        try:
            g = moe.LayerGraph(cfg, inp["x"], weights, workspace=ws, outputs=outs, warm=False)
            tot = {k: 0.0 for k in moe.STAGES}
            for _ in range(reps):
                g.replay()
                ms, _ = moe.stage_times()
                for k in tot:
                    tot[k] += ms[k]
            del g
            return tot, reps
        except moe.MoEError:
            pass        # event timing inside graphs unavailable: time eager calls
        finally:
            moe.stage_timing(False)
    moe.stage_timing(True)
    for _ in range(reps):
        moe.layer_forward(cfg, inp["x"], weights, workspace=ws, outputs=outs)
    torch.cuda.synchronize(dev)
    res = moe.stage_times()
    moe.stage_timing(False)
    return res


def run_ours(args, w, T):
    import sparse_mixture_experts_47_b300 as moe
    if args.pair_tiles:
        moe.debug_set_pair_tiles(args.pair_tiles)
    if args.var_up:
        moe.debug_set_var_up_tiles(args.var_up)

    world, rank, local = dist_setup(args)
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    inp = mi.generate(w, T, dev)
    if world > 1:      # each rank its own batch of tokens (weak scaling)
        g = torch.Generator(device=dev)
        g.manual_seed(1000 + rank)
        inp["x"] = torch.randn(inp["x"].shape, generator=g, device=dev).to(inp["x"].dtype)
    cfg = moe.config_for(w, T, out_dtype=moe.DTYPE_BF16)
    weights = {k: inp.get(k) for k in moe._WEIGHT_KEYS}
    ws = moe.Workspace(dev)
    outs = moe.layer_forward(cfg, inp["x"], weights, workspace=ws)
    stream = torch.cuda.current_stream(dev)

    for _ in range(args.warmup):
        moe.layer_forward(cfg, inp["x"], weights, workspace=ws, outputs=outs)
    torch.cuda.synchronize(dev)
    assert moe.device_status(dev) == 0
    l0 = moe.kernel_launches()
    moe.layer_forward(cfg, inp["x"], weights, workspace=ws, outputs=outs)
    launches_per_step = moe.kernel_launches() - l0

    graph = None
    if args.launch == "graph":
        graph = moe.LayerGraph(cfg, inp["x"], weights, workspace=ws, outputs=outs, warm=False)

    def step():
        if graph is not None:
            graph.replay()
        else:
            moe.layer_forward(cfg, inp["x"], weights, workspace=ws, outputs=outs)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    assert moe.device_status(dev) == 0

    clocks = ClockSampler(dev.index)
    clocks.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize(dev)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(args.steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    clk = clocks.stop()
    ms = ev0.elapsed_time(ev1)
    ms = max_over_ranks(ms, world)
    assert moe.device_status(dev) == 0
    launches = launches_per_step * args.steps

    # Per-stage times (CUDA events the library records around each stage on
    # the launching stream), in a separate pass so that recording them does
    # not perturb the timed region above.
    stage_ms, calls = stage_pass(moe, cfg, inp, weights, ws, outs, args, graph is not None, dev)

    # End to end with host buffers: every step copies its batch in from pinned
    # host memory and its output back.  Graph mode runs the public
    # LayerPipeline (copies of neighbouring batches overlap the layer); eager
    # mode calls the layer between the two copies.
    x_host = inp["x"].cpu().pin_memory()
    y_hosts = [torch.empty(outs["y"].shape, dtype=outs["y"].dtype).pin_memory()
               for _ in range(2)]
    if graph is not None:
        pipe = moe.LayerPipeline(cfg, weights, dev, workspace=ws)

        def e2e_run(n):
            pipe.run([x_host] * n, [y_hosts[i % 2] for i in range(n)])
    else:
        x_dev = torch.empty_like(inp["x"])

        def e2e_run(n):
            for i in range(n):
                x_dev.copy_(x_host, non_blocking=True)
                moe.layer_forward(cfg, x_dev, weights, workspace=ws, outputs=outs)
                y_hosts[i % 2].copy_(outs["y"], non_blocking=True)

    e2e_run(3)
    torch.cuda.synchronize(dev)
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    e2e_run(args.steps)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world)
    x_host_bytes = x_host.numel() * x_host.element_size()
    y_host_bytes = y_hosts[0].numel() * y_hosts[0].element_size()

    n_dropped = int(outs["n_dropped"][0])
    counts = outs["counts"].cpu().numpy()
    if w.routing == "expert":
        # every expert serves exactly its counts[e] rows; n_dropped counts the
        # tokens no expert took
        n_kept = int(counts.sum())
        nz = int((counts > 0).sum())
    else:
        # counts are assignments before capacity; served rows = T*k - dropped
        n_kept = T * w.top_k - n_dropped
        nz = int((counts > 0).sum())
    flops, bytes_, up_flops, up_bytes = algorithmic(w, T, n_kept, nz)
    peaks, src = load_peaks()
    step_s = ms / 1e3 / args.steps
    tc_peak = peaks["bf16_tflops_sustained"] * 1e12
    tc_burst = peaks["bf16_tflops"] * 1e12
    hbm = peaks["hbm_gbs"] * 1e9
    roof_s = max(flops / tc_burst, bytes_ / hbm)
    roof_sus_s = max(flops / tc_peak, bytes_ / hbm)
    up_ms = stage_ms["up"] / max(calls, 1)
    up_tflops = up_flops / (up_ms / 1e3) / 1e12
    up_gbs = up_bytes / (up_ms / 1e3) / 1e9
    recs = [r for r in traffic_record("gemm_tcgen05.cu") or []
            if r.get("workload") == w.name and not args.n_experts and not args.d_ff]
    exact = [r for r in recs if r.get("T") == T]
    tr = exact[0] if exact else (recs[-1] if recs else None)
    # The dominant kernel is timed per launch inside short graph replays, a
    # burst window: its tensor-bound fraction is quoted against the measured
    # burst bf16 peak; the sustained peak (a seconds-long loop under the
    # power cap) is reported beside it.
    up_tensor_bound = up_flops / tc_burst >= up_bytes / hbm
    if up_tensor_bound:
        roof = {"bound": "tensor", "achieved": up_tflops, "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s", "frac": up_tflops * 1e12 / tc_burst,
                "frac_of_sustained": up_tflops * 1e12 / tc_peak,
                "peak_source": f"{src} bf16_tflops (burst)"}
    else:
        roof = {"bound": "hbm", "achieved": up_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": up_gbs / peaks["hbm_gbs"], "peak_source": f"{src} hbm_gbs"}
    plan = moe.ffn_plan(cfg) if w.dtype == "bf16" else {}
    roof["kernel"] = ("grouped_gemm_pair_kernel (up projection, 256-row tiles on SM pairs)"
                      if plan.get("up_pair") else
                      "grouped_gemm_tc_kernel (up projection, weights on the M side, the MMA N "
                      "set per tile)" if plan.get("rows_per_tile") == 256 else
                      "grouped_gemm_tc_kernel (up projection)")
    roof["algorithmic_per_launch"] = {"flops": up_flops, "bytes": up_bytes}
    roof["ms_per_launch"] = up_ms
    roof["traffic"] = None
    if tr:
        if tr.get("T") == T:
            roof["traffic"] = tr["dram_bytes_per_launch"]
        elif "weight_bytes" in tr:
            # captured at a smaller T: the weights are read once whatever T is,
            # the row traffic (x_sorted in, h out) grows with T
            rows = tr["dram_bytes_per_launch"] - tr["weight_bytes"]
            roof["traffic"] = tr["weight_bytes"] + rows * T / tr["T"]
        roof["traffic_source"] = (
            f"not measured in this run: dram__bytes_read.sum + dram__bytes_write.sum of one "
            f"ncu capture at T={tr.get('T')} of the same kernel source (hash "
            f"{tr.get('source_sha256_16')}), recorded in profiles/ncu_traffic.md"
            + ("" if tr.get("T") == T else f", scaled to T={T} by its row traffic"))
    else:
        roof["traffic_source"] = "no ncu record of the current kernel source"

    if rank != 0:
        return
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        inp64 = host_inputs_f64(inp)
        S = calibrated_sample(w, inp64, T, 15.0)      # about 15 s of CPU work
        t = oracle_sample_run(w, inp64, S)
        cpu = {"value": S / t, "unit": "tokens/s", "cores": blas_threads(), "kind": "oracle",
               "sample": f"first {S} of the {T} tokens as one batch (routing, dispatch, "
                         "stats, FFN, combine), fp64 numpy, one run"}
    value = job_throughput(world, T, args.steps, ms)
    line = {
        "metric": "MoE-layer fwd tokens/s on 1 B300 (bf16) and % of roofline",
        "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{w.name}-shaped layer d={w.d_model} E={w.n_experts} "
                               f"k={w.top_k} d_ff={w.d_ff} T={T}",
                   "tokens_per_rank": T, "parallelism": f"replicas x{world}",
                   "l2": "no flush: weights larger than L2 stream from HBM every step",
                   "out_dtype": "bf16",
                   "launch": ("one CUDA graph replay of moe_layer_forward per step"
                              if args.launch == "graph" else "eager moe_layer_forward calls")},
        "roofline": roof,
        "layer_roofline": {"flops": flops, "bytes": bytes_, "roofline_ms": roof_s * 1e3,
                           "frac": roof_s / step_s,
                           "frac_of_sustained": roof_sus_s / step_s,
                           "bound": "tensor" if flops / tc_burst > bytes_ / hbm else "hbm",
                           "peaks": f"{src}: {peaks['bf16_tflops']} TF/s burst "
                                    f"({peaks['bf16_tflops_sustained']} sustained), "
                                    f"{peaks['hbm_gbs']} GB/s"},
        "stage_ms": {k: v / max(calls, 1) for k, v in stage_ms.items()},
        "e2e": {"value": job_throughput(world, T, args.steps, e2e_ms), "unit": "tokens/s",
                "h2d_bytes_per_step": x_host_bytes, "d2h_bytes_per_step": y_host_bytes,
                "how": ("LayerPipeline: H2D of step i+1 and D2H of step i-1 overlap the layer "
                        "on step i" if graph is not None
                        and x_host_bytes >= moe.LayerPipeline.OVERLAP_MIN_BYTES else
                        "H2D, layer, D2H in sequence on one stream")},
        "clocks": clk,
        "gpu_launches": launches,
        "cpu_baseline": cpu,
        "n_dropped": n_dropped,
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="mixtral", choices=list(mi.WORKLOADS))
    ap.add_argument("--T", type=int, default=None)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--launch", default="graph", choices=["graph", "eager"],
                    help="replay one captured CUDA graph of the layer per step (default) "
                         "or call the layer eagerly")
    ap.add_argument("--n-experts", type=int, default=None,
                    help="override the workload's expert count (a reduced case for profiler "
                         "captures; with --T scaled alike it keeps the rows per expert)")
    ap.add_argument("--d-ff", type=int, default=None,
                    help="override the routed experts' width (a reduced case for profiler "
                         "captures of the router and the row kernels, whose work does not "
                         "depend on it)")
    ap.add_argument("--pair-tiles", type=int, default=0, choices=[-1, 0, 1],
                    help="the library's switch of the 256-row SM-pair GEMM tiles: 0 its own "
                         "rule (default), -1 never, 1 wherever the geometry allows")
    ap.add_argument("--var-up", type=int, default=0, choices=[-1, 0, 1],
                    help="the library's switch of the up projection's per-tile-width "
                         "geometry: 1 wherever the experts average more than 64 rows, "
                         "0 (default) and -1 never")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)     # at least 3 untimed warm-up steps
    w = mi.workload(args.workload)
    if args.n_experts:
        w = w.with_sizes(n_experts=args.n_experts)
    if args.d_ff:
        w = w.with_sizes(d_ff=args.d_ff)
    T = args.T or max(w.tokens)
    if args.impl == "reference":
        run_reference(args, w, T)
    else:
        run_ours(args, w, T)


if __name__ == "__main__":
    main()
