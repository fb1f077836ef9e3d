#!/usr/bin/env python
"""Benchmark of the sparse MoE FFN layer forward on B300.

One step = one pass of the whole layer over one batch: router (logits, top-k,
gate), dispatch, routed expert FFN (tcgen05 grouped GEMM), shared expert (if
the workload has one), combine, and the per-expert load statistics.  Inputs
and all expert weights are resident in HBM before the timed region.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Prints one JSON line (rank 0).  Under torchrun (N > 1) every rank runs an
independent replica of the layer on its own GPU (the layer does not shard:
replicas only); the time is the max over ranks and the value counts the tokens
of all ranks.  ``--impl reference`` times the CPU oracle instead (rank 0 only).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "MoE-layer fwd tokens/s at Mixtral shape; % of BF16 tensor / HBM roofline"
DEFAULT_WORKLOAD = "mixtral_prefill"


# ----------------------------------------------------------------------------- accounting
def layer_flops(wl, kept_rows: int) -> dict:
    """Algorithmic FLOPs: router + kept assignments' experts + shared expert."""
    mats = 3 if wl.act == "swiglu" else 2
    router = 2.0 * wl.T * wl.d * wl.N
    ffn = 2.0 * kept_rows * wl.d * wl.F * mats
    shared = 2.0 * wl.T * wl.d * wl.shared_F * mats if wl.shared_F else 0.0
    return {"router": router, "expert_ffn": ffn, "shared_ffn": shared, "total": router + ffn + shared}


def expert_weight_bytes(wl, fp8: bool) -> float:
    """Bytes of one expert's weights: 2 (bf16) / 4 (float32) per weight, or 1 per E4M3
    code plus a float32 scale per row (W1, W3: F rows; W2: d rows)."""
    mats = 3 if wl.act == "swiglu" else 2
    if fp8:
        return float(mats * wl.d * wl.F + ((mats - 1) * wl.F + wl.d) * 4)
    return float(mats * wl.d * wl.F * (2 if wl.dtype == "bf16" else 4))


def layer_bytes(wl, touched_experts: int, fp8: bool = False) -> float:
    """Algorithmic bytes: weights of experts with kept rows, x once, out once, W_g."""
    es = 2 if wl.dtype == "bf16" else 4
    mats = 3 if wl.act == "swiglu" else 2
    w = touched_experts * expert_weight_bytes(wl, fp8)
    sw = mats * wl.d * wl.shared_F * es if wl.shared_F else 0
    return float(w + sw + 2 * wl.T * wl.d * es + wl.d * wl.N * 4)


# DRAM bytes (read + write) of the expert-FFN launches of one step, from ncu captures
# of the kernel revision named here (profiles/); keyed by (workload, FP8 weights).
# A workload whose kernel has changed since its capture reports None.
NCU_TRAFFIC = {("mixtral_prefill", False): {"bytes": 3.689e9, "kernel_rev": "pair2"},
               ("mixtral_decode", True): {"bytes": 1.4267e9, "kernel_rev": "fp8ffn1"}}
KERNEL_REV = {False: "pair2", True: "fp8ffn1"}


def stage_work(wl, kept_rows: int, touched: int, fp8: bool = False) -> dict:
    """Algorithmic (flops, bytes) per stage of one layer step.

    route: x read once, W_g, logits written, top-k ids + weights written;
    dispatch: ids read, x rows read once, x_perm written, index arrays;
    expert_ffn: kept rows' FLOPs; weights of touched experts, x_perm read, y_perm written;
    shared_ffn: every token; its weights, x read, y written;
    combine: y_perm (+ shared y) read, out written, ids + weights read;
    load_stats: logits and counts read."""
    es = 2 if wl.dtype == "bf16" else 4
    mats = 3 if wl.act == "swiglu" else 2
    T, d, N, k, F, S = wl.T, wl.d, wl.N, wl.k, wl.F, kept_rows
    w = {
        "route": (2.0 * T * d * N, T * d * es + d * N * 4 + T * N * 4 + T * k * 8),
        "dispatch": (0.0, T * k * 4 + T * d * es + S * d * es + T * k * 4 + S * 4 + 3 * N * 4),
        "expert_ffn": (2.0 * S * d * F * mats, touched * expert_weight_bytes(wl, fp8) + 2 * S * d * es),
        "combine": (0.0, S * d * es + T * d * es + T * k * 8 + (T * d * es if wl.shared_F else 0)),
        "load_stats": (0.0, T * N * 4 + 2 * N * 4),
    }
    if wl.shared_F:
        w["shared_ffn"] = (2.0 * T * d * wl.shared_F * mats, mats * d * wl.shared_F * es + 2 * T * d * es)
    return w


# float32 CUDA-core peak: 148 SMs x 128 FP32 lanes x 2 FLOP (one FMA) x 2032 MHz
# (maximum SM clock) = 77.0 TFLOP/s; the float32 workload's GEMMs run there.
F32_ALU_TFLOPS = 148 * 128 * 2 * 2.032e9 / 1e12


def stage_roofline(flops, nbytes, ms, peaks, sustained, alu=False):
    """The bound whose time is longer at peak; achieved rate and fraction of that peak."""
    tf_peak = peaks["bf16_tflops_sustained"] if sustained else peaks["bf16_tflops"]
    if alu:
        tf_peak = F32_ALU_TFLOPS
    t_tensor = flops / (tf_peak * 1e12)
    t_hbm = nbytes / (peaks["hbm_gbs"] * 1e9)
    s = ms / 1e3
    if flops > 0 and t_tensor >= t_hbm:
        return {"ms": ms, "bound": "alu" if alu else "tensor", "achieved": flops / s / 1e12, "peak": tf_peak,
                "unit": "TFLOP/s", "frac": t_tensor / s}
    return {"ms": ms, "bound": "hbm", "achieved": nbytes / s / 1e9, "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": t_hbm / s}


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}, "fallback"


def blas_threads() -> int:
    """Threads the oracle's float64 matmuls run on (BLAS pool), else the host's cores."""
    try:
        import threadpoolctl
        return max((p.get("num_threads", 1) for p in threadpoolctl.threadpool_info()), default=1)
    except ImportError:
        for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
            if os.environ.get(var, "").isdigit():
                return int(os.environ[var])
        return os.cpu_count() or 1


def _traffic(name, fp8: bool = False):
    t = NCU_TRAFFIC.get((name, fp8))
    return t["bytes"] if t and t["kernel_rev"] == KERNEL_REV[fp8] else None


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in getattr(self, "lines", []):
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = max(mx, float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_min_mhz": min(sm), "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------- distributed
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world):
    if world <= 1:
        return None
    import torch.distributed as dist
    os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
    dist.init_process_group("gloo")
    return dist


def max_over_ranks(dist, v: float) -> float:
    if dist is None:
        return v
    import torch
    t = torch.tensor([v], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------- reference arm
def run_reference(args, wl):
    """The CPU oracle, as it stands, on a bounded sample of the same workload per step.

    Without a capacity limit every token is routed and processed on its own, so a
    step is the oracle's layer on `--ref-sample` seeded tokens taken as a layer of
    their own (routing, gate, their experts, combine, statistics); with a capacity
    limit the routing and dispatch of all tokens come first, then the experts on
    the sampled tokens, extrapolated to all tokens."""
    import dataclasses
    import oracle
    inp = synth.make_inputs(wl)
    sample = min(args.ref_sample, wl.T)
    rng = np.random.default_rng(wl.seed)

    def step():
        toks = np.sort(rng.choice(wl.T, size=sample, replace=False))
        if wl.capacity_factor <= 0:
            sub = dataclasses.replace(inp, wl=wl.scaled(T=sample), x=inp.x[toks])
            t0 = time.perf_counter()
            oracle.layer_forward(sub)
            return (time.perf_counter() - t0) * wl.T / sample                # seconds per full layer
        t0 = time.perf_counter()
        oracle.layer_forward(inp, tokens=np.array([], dtype=np.int64))      # routing + dispatch + stats, all T
        t1 = time.perf_counter()
        oracle.layer_forward(inp, tokens=toks)                                # + experts on the sample
        t2 = time.perf_counter()
        ffn_per_token = max(0.0, (t2 - t1) - (t1 - t0)) / len(toks)
        return (t1 - t0) + ffn_per_token * wl.T                               # extrapolated full-layer seconds

    for _ in range(args.warmup):
        step()
    secs = [step() for _ in range(args.steps)]
    per_step = float(np.mean(secs))
    cores = blas_threads()
    value = wl.T / per_step
    if wl.capacity_factor <= 0:
        desc = (f"oracle (numpy float64): each step the whole layer on {sample} seeded token(s) taken as a layer "
                f"of their own (tokens are independent without a capacity limit), including the float64 widening "
                f"of each touched expert's weights, scaled to {wl.T} tokens")
    else:
        desc = (f"oracle (numpy float64): routing, dispatch and statistics on all {wl.T} tokens, expert FFN on "
                f"{sample} sampled tokens per step, extrapolated linearly to {wl.T} tokens")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": per_step * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_of(wl),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": desc},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def cpu_baseline(wl, inp, budget_tokens: int):
    import oracle
    toks = np.sort(np.random.default_rng(wl.seed + 1).choice(wl.T, size=min(budget_tokens, wl.T), replace=False))
    t0 = time.perf_counter()
    oracle.layer_forward(inp, tokens=np.array([], dtype=np.int64))
    t1 = time.perf_counter()
    oracle.layer_forward(inp, tokens=toks)
    t2 = time.perf_counter()
    per_token = max(0.0, (t2 - t1) - (t1 - t0)) / len(toks)
    est = (t1 - t0) + per_token * wl.T
    cores = blas_threads()
    return {"value": wl.T / est, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": (f"numpy float64 oracle: routing, dispatch and statistics on all {wl.T} tokens, expert FFN "
                       f"on {len(toks)} sampled tokens, extrapolated linearly to {wl.T} tokens "
                       f"({t2 - t0:.1f} s of CPU work)")}


L2_BYTES = 126 << 20


def needs_l2_flush(wl, fp8: bool = False) -> bool:
    """All expert weights together within twice the L2: steps would hit in L2."""
    return wl.N * expert_weight_bytes(wl, fp8) < 2 * L2_BYTES


def config_of(wl, fp8: bool = False):
    return {"workload": wl.name, "T": wl.T, "d": wl.d, "N": wl.N, "k": wl.k, "ffn": wl.F, "act": wl.act,
            "gate": wl.gate, "shared_ffn": wl.shared_F, "capacity_factor": wl.capacity_factor,
            "l2": ("flushed before every timed step (256 MB written outside the step's events): the weights "
                   "fit in L2" if needs_l2_flush(wl, fp8) else
                   "no flush: inputs larger than L2 (every step streams all touched expert weights)")}


# ----------------------------------------------------------------------------- our arm
def _to_dev(a, dtype):
    import torch
    if a is None:
        return None
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def build_layer(moe, inp):
    wl = inp.wl
    cap = moe.moe_capacity(wl.capacity_factor, wl.T, wl.k, wl.N) if wl.capacity_factor > 0 else 0
    cfg = moe.make_config(wl.T, wl.d, wl.N, wl.k, wl.F, wl.shared_F,
                          {"softmax": moe.GATE_SOFTMAX_TOPK, "sigmoid": moe.GATE_SIGMOID_BIAS,
                           "softmax_full": moe.GATE_SOFTMAX_FULL}[wl.gate],
                          moe.ACT_SWIGLU if wl.act == "swiglu" else moe.ACT_RELU,
                          moe.DTYPE_BF16 if wl.dtype == "bf16" else moe.DTYPE_F32, cap)
    dt = wl.dtype
    return moe.MoELayer(cfg, _to_dev(inp.Wg, "f32"), _to_dev(inp.w1, dt), _to_dev(inp.w3, dt), _to_dev(inp.w2, dt),
                        _to_dev(inp.sw1, dt), _to_dev(inp.sw3, dt), _to_dev(inp.sw2, dt),
                        _to_dev(inp.logit_bias, "f32"), _to_dev(inp.sel_bias, "f32"))


def run_ours(args, wl, dist, rank, local):
    import torch

    import sparse_mixture_experts_62_b300 as moe

    torch.cuda.set_device(local)
    inp = synth.make_inputs(wl)
    to_dev = _to_dev
    layer = build_layer(moe, inp)
    if args.fp8:  # weights quantised once, outside the timed region (like any weight packing)
        if wl.dtype != "bf16":
            raise SystemExit("--fp8 needs a bf16 workload")
        layer.quantize_fp8()
        torch.cuda.synchronize()
    x = to_dev(inp.x, wl.dtype)
    out = torch.empty((wl.T, wl.d), dtype=x.dtype, device="cuda")
    cfg, ws, v = layer.cfg, layer.ws, layer.views()
    stream = torch.cuda.current_stream()
    stats = torch.zeros(2 * wl.N + 4, dtype=torch.float32, device="cuda")
    has_shared = wl.shared_F > 0
    stages = ["route", "dispatch", "expert_ffn"] + (["shared_ffn"] if has_shared else []) + ["combine", "load_stats"]

    def step(ev=None):
        # the launches of moe_layer_forward, stage by stage, + the statistics, on
        # the current stream (which is the capture stream while a graph records)
        cur = torch.cuda.current_stream()
        s = cur.cuda_stream
        rec = (lambda i: ev[i].record(cur)) if ev is not None else (lambda i: None)
        rec(0)
        moe.moe_route(cfg, x, layer.Wg, layer.logit_bias, layer.sel_bias, v["logits"], v["topk_idx"], v["topk_w"],
                      ws, s)
        rec(1)
        moe.moe_dispatch(cfg, v["topk_idx"], x, v["counts_routed"], v["counts_kept"], v["offsets"], v["dest_row"],
                         v["src_token"], v["x_perm"], ws, s)
        rec(2)
        if layer.fp8 is not None:
            moe.moe_expert_ffn_fp8(cfg, v["x_perm"], v["offsets"], *layer.fp8, v["y_perm"], ws, s)
        else:
            moe.moe_expert_ffn(cfg, v["x_perm"], v["offsets"], layer.w1, layer.w3, layer.w2, v["y_perm"], ws, s)
        i = 3
        if has_shared:
            rec(i)
            moe.moe_shared_ffn(cfg, x, layer.sw1, layer.sw3, layer.sw2, v["y_shared"], ws, s)
            i += 1
        rec(i)
        moe.moe_combine(cfg, v["y_perm"], v["dest_row"], v["topk_w"], v["y_shared"] if has_shared else None, out, s)
        rec(i + 1)
        moe.moe_load_stats(cfg, v["logits"], v["counts_routed"], v["counts_kept"], stats[:wl.N],
                           stats[wl.N:2 * wl.N], stats[2 * wl.N:2 * wl.N + 3], ws, s)
        rec(i + 2)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if layer.device_status() != 0:
        raise RuntimeError("device status not clean after warm-up")
    # per-stage durations: an eager pass with events between the stages
    nev = len(stages) + 1
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(nev)] for _ in range(args.steps)]
    for k in range(args.steps):
        step(evs[k])
    torch.cuda.synchronize()
    stage_ms = {n: float(np.mean([evs[k][j].elapsed_time(evs[k][j + 1]) for k in range(args.steps)]))
                for j, n in enumerate(stages)}
    # the timed region: the step captured once as a CUDA graph and replayed (the
    # same launches, without the host's per-call overhead); eager if capture fails
    graph = None
    if not args.eager:
        try:
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                step()
            for _ in range(args.warmup):
                graph.replay()
            torch.cuda.synchronize()
        except RuntimeError as exc:  # pragma: no cover - reported, then timed eagerly
            sys.stderr.write(f"graph capture failed ({exc}); timing eager launches\n")
            graph = None
    run = graph.replay if graph is not None else step
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    marks = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    flush = needs_l2_flush(wl, args.fp8)
    if flush:  # each step timed on its own, after 256 MB of writes have evicted the layer from L2
        scratch = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=stream.device)
        begins = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    with ClockSampler(local) as clk:
        start.record(stream)
        for k in range(args.steps):
            if flush:
                scratch.zero_()
                begins[k].record(stream)
            run()
            marks[k].record(stream)
        end.record(stream)
        torch.cuda.synchronize()
    if flush:
        step_ms = [begins[k].elapsed_time(marks[k]) for k in range(args.steps)]
    else:
        step_ms = [start.elapsed_time(marks[0])] + [marks[k - 1].elapsed_time(marks[k])
                                                    for k in range(1, args.steps)]
    if dist is not None:
        dist.barrier()
    if layer.device_status() != 0:
        raise RuntimeError("device status not clean after the timed region")
    total_ms = float(sum(step_ms)) if flush else start.elapsed_time(end)
    t_max = max_over_ranks(dist, total_ms)
    ms_per_step = t_max / args.steps
    world = dist.get_world_size() if dist is not None else 1
    value = wl.T * args.steps * world / (t_max / 1e3)

    # optional: the backward step (gradients of a fixed dout), graph-replayed
    bwd = None
    if args.backward:
        bwd = time_backward(args, moe, layer, x, wl, stream)

    # routing facts of this run (for the algorithmic counts)
    counts_kept = v["counts_kept"].cpu().numpy()
    kept_rows = int(counts_kept.sum())
    touched = int(np.count_nonzero(counts_kept))
    fl = layer_flops(wl, kept_rows)
    peaks, peak_src = measured_peaks()
    clocks = clk.summary()
    sustained = "sw_power_cap" in clocks.get("reasons", [])
    work = stage_work(wl, kept_rows, touched, args.fp8)
    f32 = wl.dtype == "f32"
    stages = {n: stage_roofline(work[n][0], work[n][1], stage_ms[n], peaks, sustained,
                                alu=f32 and n in ("route", "expert_ffn", "shared_ffn")) for n in stages}
    ffn = stages["expert_ffn"]
    roof = {"bound": ffn["bound"], "achieved": ffn["achieved"], "peak": ffn["peak"], "unit": ffn["unit"],
            "frac": ffn["frac"], "traffic": _traffic(wl.name, args.fp8),
            "kernel": ((("fp8_ffn_decode_kernel (tcgen05, E4M3 weights converted into tensor memory as the A "
                          "operand), moe_expert_ffn_fp8: gate/up and down in one cooperative launch")
                         if wl.T <= 64 else
                         ("grouped_gemm_fp8 (tcgen05, E4M3 weights converted into a shared-memory B operand), "
                          "moe_expert_ffn_fp8: gate/up + down launches"))
                        if args.fp8 else "grouped_gemm (tcgen05), moe_expert_ffn: gate/up + down launches"),
            "peak_source": ("derived float32 CUDA-core peak (148 SMs x 128 lanes x 2 FLOP x 2032 MHz)"
                            if ffn["bound"] == "alu" else f"{peak_src} " + ("hbm_gbs" if ffn["bound"] == "hbm" else
                            ("bf16_tflops_sustained (power cap seen in the timed region)" if sustained
                             else "bf16_tflops (burst)")))}

    # End to end through the public API: every step copies its x in from pinned host
    # memory and its output and statistics back.  Copies run on their own streams
    # with two device buffers, so step i+1's upload and step i-1's readback overlap
    # step i's compute (the layer's workspace keeps compute on one stream).
    x_host = x.cpu().pin_memory()
    out_host = [torch.empty_like(out, device="cpu").pin_memory() for _ in range(2)]
    stats_host = [torch.empty_like(stats, device="cpu").pin_memory() for _ in range(2)]
    x_dev = [torch.empty_like(x) for _ in range(2)]
    out_dev = [torch.empty_like(out) for _ in range(2)]
    stats_dev = [torch.empty_like(stats) for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()  # noqa: E731
    x_ready, comp_done, x_free, out_free = ([ev(), ev()] for _ in range(4))
    for b in range(2):
        x_free[b].record(stream)
        out_free[b].record(stream)

    def compute(b):
        layer.forward(x_dev[b], out_dev[b])
        layer.load_stats()
        stats_dev[b].copy_(layer._stats)  # this step's statistics, off the shared buffer

    # the compute of each buffer slot as a CUDA graph (the copies stay on their streams)
    slot_graphs = None
    if graph is not None:
        slot_graphs = []
        for b in range(2):
            compute(b)  # warm
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                compute(b)
            slot_graphs.append(g)
        torch.cuda.synchronize()

    def e2e_step(i):
        b = i & 1
        s_in.wait_event(x_free[b])
        with torch.cuda.stream(s_in):
            x_dev[b].copy_(x_host, non_blocking=True)
        x_ready[b].record(s_in)
        stream.wait_event(x_ready[b])
        stream.wait_event(out_free[b])
        if slot_graphs is not None:
            slot_graphs[b].replay()
        else:
            compute(b)
        x_free[b].record(stream)
        comp_done[b].record(stream)
        s_out.wait_event(comp_done[b])
        with torch.cuda.stream(s_out):
            out_host[b].copy_(out_dev[b], non_blocking=True)
            stats_host[b].copy_(stats_dev[b], non_blocking=True)
        out_free[b].record(s_out)

    for i in range(args.warmup):
        e2e_step(i)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    s_in.wait_stream(stream)
    for i in range(args.steps):
        e2e_step(i)
    stream.wait_stream(s_out)
    stream.wait_stream(s_in)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(dist, e0.elapsed_time(e1))
    e2e_val = wl.T * args.steps * world / (e2e_ms / 1e3)
    h2d = x.numel() * x.element_size()
    d2h = out.numel() * out.element_size() + stats.numel() * 4

    # route: split W_g + tensor-core logits + top-k (bf16) or logits + top-k (float32);
    # dispatch: histogram, scan, rank, gather; experts: 2; shared: 2; combine: 1; stats: 2
    ffn_launches = 1 if (args.fp8 and wl.T <= 64) else 2  # FP8 decode: gate/up and down in one launch
    launches_per_step = (3 if wl.dtype == "bf16" else 2) + 4 + ffn_launches + (2 if has_shared else 0) + 1 + 2
    if rank == 0:
        sys.stderr.write("per-stage ms: " + json.dumps({k: round(val, 4) for k, val in stage_ms.items()}) + "\n")
        line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
                "step_ms": {"p10": float(np.percentile(step_ms, 10)), "p50": float(np.percentile(step_ms, 50)),
                            "p90": float(np.percentile(step_ms, 90))},
                "vs_baseline": None, "dtype": wl.dtype, "data": "synthetic",
                "config": {**config_of(wl, args.fp8), "launch": "cuda_graph" if graph is not None else "eager",
                           **({"expert_weights": "fp8 e4m3, one float32 scale per row"} if args.fp8 else {})},
                "roofline": roof,
                "stages": stages,
                "layer": {"flops": fl["total"], "tflops": fl["total"] / (ms_per_step / 1e3) / 1e12,
                          "kept_rows": kept_rows, "touched_experts": touched,
                          "algorithmic_bytes": layer_bytes(wl, touched, args.fp8)},
                "e2e": {"value": e2e_val, "unit": "tokens/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
                "gpu_launches": launches_per_step * args.steps,
                **({"backward": bwd} if bwd is not None else {}),
                "clocks": clocks}
        if args.cpu_baseline_tokens > 0:
            line["cpu_baseline"] = cpu_baseline(wl, inp, args.cpu_baseline_tokens)
        print(json.dumps(line), flush=True)


def time_backward(args, moe, layer, x, wl, stream):
    """Time moe_layer_backward (after a forward) as a CUDA-graph replay; FLOPs of its
    GEMMs in units of 2 R d F (R the kept rows): dh 1, the a/u recompute 2, dx rows
    2, dW2 1, dW1/dW3 2 = 8 for SwiGLU; 5 for ReLU (no u, du or dW3)."""
    import torch
    cfg = layer.cfg
    sw = wl.act == "swiglu"
    dout = torch.randn((wl.T, wl.d), device="cuda").to(x.dtype)
    f32 = lambda *shape: torch.empty(shape, device="cuda")  # noqa: E731
    dx, dWg = f32(wl.T, wl.d), f32(wl.d, wl.N)
    dw1, dw3, dw2 = f32(wl.N, wl.F, wl.d), (f32(wl.N, wl.F, wl.d) if sw else None), f32(wl.N, wl.d, wl.F)
    Fs = wl.shared_F
    dsw1, dsw3, dsw2 = (f32(Fs, wl.d), f32(Fs, wl.d) if sw else None, f32(wl.d, Fs)) if Fs else (None, None, None)
    bws = torch.empty(moe.moe_backward_workspace_size(cfg), dtype=torch.uint8, device="cuda")

    def step():
        moe.moe_layer_backward(cfg, x, layer.Wg, layer.w1, layer.w3, layer.w2, layer.sw1, layer.sw3, layer.sw2,
                               dout, dx, dWg, dw1, dw3, dw2, dsw1, dsw3, dsw2, layer.ws, bws)

    layer.forward(x)
    for _ in range(args.warmup):
        step()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for _ in range(args.warmup):
        g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        g.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    if layer.device_status() != 0:
        raise RuntimeError("device status not clean after the backward")
    ms = e0.elapsed_time(e1) / args.steps
    R = int(layer.views()["counts_kept"].sum().item())
    units = 8 if sw else 5
    gemm_flops = units * 2.0 * R * wl.d * wl.F + (units * 2.0 * wl.T * wl.d * Fs if Fs else 0.0)
    return {"ms_per_step": ms, "tokens_per_s": wl.T / (ms / 1e3), "gemm_flops": gemm_flops,
            "gemm_tflops_over_step": gemm_flops / (ms / 1e3) / 1e12}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(synth.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-baseline-tokens", type=int, default=512,
                    help="tokens the oracle runs the expert FFN on for cpu_baseline (0 = skip)")
    ap.add_argument("--ref-sample", type=int, default=1, help="tokens per reference-arm step")
    ap.add_argument("--override", nargs="*", default=[], help="workload fields to change, e.g. N=32 T=1024")
    ap.add_argument("--eager", action="store_true", help="time eager launches instead of a CUDA-graph replay")
    ap.add_argument("--backward", action="store_true", help="also time the backward step (bf16 token choice)")
    ap.add_argument("--fp8", action="store_true", help="FP8 E4M3 expert weights with per-row scales (bf16 workloads)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world, rank, local = dist_env()
    wl = synth.WORKLOADS[args.workload]
    if args.override:  # smaller variants of a workload, for profiling captures
        kw = {}
        for item in args.override:
            key, val = item.split("=")
            kw[key] = type(getattr(wl, key))(val)
        wl = wl.scaled(name=wl.name + "+" + ",".join(args.override), **kw)
    if args.impl == "reference":
        if rank == 0:
            run_reference(args, wl)
        return
    dist = init_dist(world)
    run_ours(args, wl, dist, rank, local)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
