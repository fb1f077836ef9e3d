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


# DRAM bytes (read + write) per step of the expert-FFN launches come from an ncu
# capture, listed in profiles/traffic.md with a hash of the kernel sources the
# capture ran; a workload whose sources have changed since reports None.
TRAFFIC_TABLE = os.path.join(ROOT, "profiles", "traffic.md")
KERNEL_SOURCES = {False: ("moe_ffn_tc.cu", "moe_common.cuh", "moe_api.cu"),
                  True: ("moe_ffn_fp8_tc.cu", "moe_common.cuh", "moe_api.cu")}


def code_of(text: str) -> str:
    """C/CUDA source without its comments, whitespace runs collapsed to one space
    (the sources hold no comment markers inside string literals)."""
    import re
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_hash(fp8: bool) -> str:
    """First 16 hex digits of the SHA-256 of the code of the expert-FFN kernel
    sources (and the launcher that picks their tile forms), concatenated in a fixed
    order; comments do not count."""
    import hashlib
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[fp8]:
        with open(os.path.join(ROOT, "sparse_mixture_experts_62_b300", "csrc", name)) as f:
            h.update(code_of(f.read()).encode())
    return h.hexdigest()[:16]


def traffic_table(path: str = TRAFFIC_TABLE) -> dict:
    """{(workload, fp8): (bytes per step, source hash)} from the table rows
    `| workload | bf16 or fp8 | source hash | bytes | ... |`."""
    out = {}
    if not os.path.exists(path):
        return out
    with open(path) as f:
        for ln in f:
            cells = [c.strip() for c in ln.strip().strip("|").split("|")]
            if len(cells) < 4 or cells[1] not in ("bf16", "fp8"):
                continue
            try:
                out[(cells[0], cells[1] == "fp8")] = (float(cells[3]), cells[2])
            except ValueError:
                continue
    return out


def _traffic(name, fp8: bool = False, table=None):
    t = (traffic_table() if table is None else table).get((name, fp8))
    return t[0] if t and t[1] == kernel_source_hash(fp8) else None


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


def stage_roofline(flops, nbytes, ms, peaks, clocks=None, alu=False):
    """The bound whose time is longer at peak; achieved rate and fraction of that peak.

    Tensor-bound work is measured against the burst bf16 peak (`frac`), with two
    extra readings: against the sustained (power-capped) peak (`frac_sustained`),
    and against the burst peak scaled by the median SM clock of the timed region
    over the maximum clock (`frac_clock_norm`; the in-band probe's clock when there
    is one, else nvidia-smi's)."""
    tf_peak = F32_ALU_TFLOPS if alu else peaks["bf16_tflops"]
    t_tensor = flops / (tf_peak * 1e12)
    t_hbm = nbytes / (peaks["hbm_gbs"] * 1e9)
    s = ms / 1e3
    if flops > 0 and t_tensor >= t_hbm:
        ach = flops / s / 1e12
        r = {"ms": ms, "bound": "alu" if alu else "tensor", "achieved": ach, "peak": tf_peak, "unit": "TFLOP/s",
             "frac": ach / tf_peak}
        if not alu:
            r["frac_sustained"] = ach / peaks["bf16_tflops_sustained"]
            mhz = (clocks or {}).get("sm_mhz_in_band") or (clocks or {}).get("sm_mhz")
            fmax = (clocks or {}).get("sm_max_mhz") or peaks.get("sm_max_mhz")
            if mhz and fmax:
                r["frac_clock_norm"] = ach / (tf_peak * min(mhz, fmax) / fmax)
        return r
    r = {"ms": ms, "bound": "hbm", "achieved": nbytes / s / 1e9, "peak": peaks["hbm_gbs"], "unit": "GB/s",
         "frac": t_hbm / s}
    if flops > 0 and not alu:
        # a contraction at the ridge: its tensor rate as well, against the burst peak
        # and against the burst peak scaled to the measured SM clock
        ach = flops / s / 1e12
        r["tflops"] = ach
        r["tensor_frac"] = ach / tf_peak
        mhz = (clocks or {}).get("sm_mhz_in_band") or (clocks or {}).get("sm_mhz")
        fmax = (clocks or {}).get("sm_max_mhz") or peaks.get("sm_max_mhz")
        if mhz and fmax:
            r["tensor_frac_clock_norm"] = ach / (tf_peak * min(mhz, fmax) / fmax)
    return r


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
def oracle_step(wl, inp, sample: int, rng):
    """One bounded step of the oracle, as it stands, on the workload.

    Without a capacity limit the tokens do not interact, so the step is the
    whole layer (routing, gate, dispatch, the experts -- whose weights the oracle
    widens to float64 on every call -- combine, statistics) on `sample` seeded
    tokens taken as a batch of their own: tokens/s = sample / seconds.  With a
    capacity limit the drop set couples all tokens: the step routes, dispatches
    and takes the statistics of all T tokens, then runs the experts on `sample`
    seeded tokens; tokens/s extrapolates the expert time linearly to T.
    Returns (seconds spent, tokens/s, description)."""
    import dataclasses
    import oracle
    sample = min(sample, wl.T)
    toks = np.sort(rng.choice(wl.T, size=sample, replace=False))
    if wl.capacity_factor <= 0:
        sub = dataclasses.replace(inp, wl=wl.scaled(T=sample), x=inp.x[toks])
        t0 = time.perf_counter()
        oracle.layer_forward(sub)
        dt = time.perf_counter() - t0
        return dt, sample / dt, (f"numpy float64 oracle: the whole layer on {sample} seeded tokens of the "
                                 f"{wl.T}-token batch per step, as a batch of their own (tokens are independent "
                                 f"without a capacity limit), float64 widening of the touched experts' weights "
                                 f"included")
    t0 = time.perf_counter()
    oracle.layer_forward(inp, tokens=np.array([], dtype=np.int64))      # routing + dispatch + stats, all T
    t1 = time.perf_counter()
    oracle.layer_forward(inp, tokens=toks)                                # + experts on the sample
    t2 = time.perf_counter()
    per_token = max(0.0, (t2 - t1) - (t1 - t0)) / len(toks)
    est = (t1 - t0) + per_token * wl.T
    return t2 - t0, wl.T / est, (f"numpy float64 oracle: routing, dispatch and statistics on all {wl.T} tokens, "
                                 f"expert FFN on {sample} seeded tokens per step, extrapolated linearly to "
                                 f"{wl.T} tokens (capacity couples the tokens)")


def run_reference(args, wl):
    """The reference arm: the CPU oracle timed per step on a bounded sample of the
    same workload (oracle_step), on the host's cores."""
    inp = synth.make_inputs(wl)
    rng = np.random.default_rng(wl.seed)
    for _ in range(args.warmup):
        oracle_step(wl, inp, args.ref_sample, rng)
    runs = [oracle_step(wl, inp, args.ref_sample, rng) for _ in range(args.steps)]
    secs = float(np.mean([r[0] for r in runs]))
    value = float(np.mean([r[1] for r in runs]))
    cores = blas_threads()
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_of(wl),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": runs[0][2]},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def cpu_baseline(wl, inp, sample: int):
    """The oracle on the host's cores: one step of oracle_step (the reference arm's step)."""
    secs, value, desc = oracle_step(wl, inp, sample, np.random.default_rng(wl.seed + 1))
    return {"value": value, "unit": "tokens/s", "cores": blas_threads(), "kind": "oracle",
            "sample": f"{desc} ({secs:.1f} s of CPU work)"}


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


def layer_stages(moe, layer, x, out, stats, wl):
    """The launches of moe_layer_forward, stage by stage, plus the statistics; each
    stage a function of no arguments issuing on torch's current stream (the
    capture stream while a graph records)."""
    cfg, ws, v = layer.cfg, layer.ws, layer.views()
    has_shared = wl.shared_F > 0
    cur = lambda: __import__("torch").cuda.current_stream().cuda_stream  # noqa: E731

    def route():
        moe.moe_route(cfg, x, layer.Wg, layer.logit_bias, layer.sel_bias, v["logits"], v["topk_idx"], v["topk_w"],
                      ws, cur())

    def dispatch():
        moe.moe_dispatch(cfg, v["topk_idx"], x, v["counts_routed"], v["counts_kept"], v["offsets"], v["dest_row"],
                         v["src_token"], v["x_perm"], ws, cur())

    def expert_ffn():
        if layer.fp8 is not None:
            moe.moe_expert_ffn_fp8(cfg, v["x_perm"], v["offsets"], *layer.fp8, v["y_perm"], ws, cur())
        else:
            moe.moe_expert_ffn(cfg, v["x_perm"], v["offsets"], layer.w1, layer.w3, layer.w2, v["y_perm"], ws, cur())

    def shared_ffn():
        moe.moe_shared_ffn(cfg, x, layer.sw1, layer.sw3, layer.sw2, v["y_shared"], ws, cur())

    def combine():
        moe.moe_combine(cfg, v["y_perm"], v["dest_row"], v["topk_w"], v["y_shared"] if has_shared else None, out,
                        cur())

    def load_stats():
        moe.moe_load_stats(cfg, v["logits"], v["counts_routed"], v["counts_kept"], stats[:wl.N],
                           stats[wl.N:2 * wl.N], stats[2 * wl.N:2 * wl.N + 3], ws, cur())

    st = [("route", route), ("dispatch", dispatch), ("expert_ffn", expert_ffn)]
    if has_shared:
        st.append(("shared_ffn", shared_ffn))
    st += [("combine", combine), ("load_stats", load_stats)]
    return st


def time_layer(args, moe, layer, x, wl, stream, dist=None, clk_gpu=None):
    """Warm-up, then the timed region: `args.steps` steps, bracketed by a barrier
    and synchronisation, with CUDA events on the launching stream.  Each step is a
    CUDA graph of the whole step, captured once per timed step so that each holds
    its own two event-record nodes around the expert-FFN stage: the dominant
    kernel's time comes from the timed steps themselves.  (Event nodes between all
    stages cost about 4 us each per step, 6% of a decode step, so the timed steps
    carry only these two.)  Then, still inside the clock sampling, a stage pass:
    `args.steps` more steps of per-stage graphs with events between the stages,
    for the per-stage table.  With --eager the stages are launched directly.
    Returns step_ms (per step), total_ms, ffn_ms (mean over the timed steps),
    stage_ms (mean per stage, stage pass), graph flag, clock summary."""
    import torch
    out = torch.empty((wl.T, wl.d), dtype=x.dtype, device="cuda")
    stats = torch.zeros(2 * wl.N + 4, dtype=torch.float32, device="cuda")
    stages = layer_stages(moe, layer, x, out, stats, wl)
    nst = len(stages)
    jf = [n for n, _ in stages].index("expert_ffn")

    def step(ev=None, all_stages=False):
        for j, (_, fn) in enumerate(stages):
            if ev is not None and (all_stages or j == jf):
                ev[j if all_stages else 0].record()
            fn()
            if ev is not None and not all_stages and j == jf:
                ev[1].record()
        if ev is not None and all_stages:
            ev[nst].record()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if layer.device_status() != 0:
        raise RuntimeError("device status not clean after warm-up")
    ext = lambda: torch.cuda.Event(enable_timing=True, external=True)  # noqa: E731
    fev = [[ext(), ext()] for _ in range(args.steps)]
    sev = [[ext() for _ in range(nst + 1)] for _ in range(args.steps)]
    graphs = stage_graphs = None
    if not args.eager:
        try:
            graphs, stage_graphs, pool = [], [], None
            for k in range(args.steps):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, pool=pool):
                    step(fev[k])
                pool = g.pool()
                graphs.append(g)
                g2 = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g2, pool=pool):
                    step(sev[k], all_stages=True)
                stage_graphs.append(g2)
            for k in range(min(args.warmup, args.steps)):
                graphs[k].replay()
            torch.cuda.synchronize()
        except RuntimeError as exc:  # pragma: no cover - reported, then timed eagerly
            sys.stderr.write(f"graph capture failed ({exc}); timing eager launches\n")
            graphs = stage_graphs = None
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    marks = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    flush = needs_l2_flush(wl, layer.fp8 is not None)
    if flush:  # each step timed on its own, after 256 MB of writes have evicted the layer from L2
        scratch = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=stream.device)
        begins = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    # SM clock sampled in-band during the timed steps: one sleeping thread on a side
    # stream records (ns, cycles) pairs every 200 us for the expected duration
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    (graphs[0].replay() if graphs is not None else step(fev[0]))
    e1.record(stream)
    torch.cuda.synchronize()
    est_ms = e0.elapsed_time(e1) * args.steps * 1.5 + 2.0
    n_probe = int(min(50000, max(8, est_ms * 5)))  # (n - 1) x 200 us stays under the probe's 10 s limit
    probe = torch.zeros(2 * n_probe, dtype=torch.int64, device="cuda")
    s_probe = torch.cuda.Stream()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(clk_gpu if clk_gpu is not None else torch.cuda.current_device()) as clk:
        moe.moe_clock_probe(probe, n_probe, 200_000, s_probe)
        start.record(stream)
        for k in range(args.steps):
            if flush:
                scratch.zero_()
                begins[k].record(stream)
            if graphs is not None:
                graphs[k].replay()
            else:
                step(fev[k])
            marks[k].record(stream)
        end.record(stream)
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
        # stage pass (not part of the step timing)
        for k in range(args.steps):
            if flush:
                scratch.zero_()
            if stage_graphs is not None:
                stage_graphs[k].replay()
            else:
                step(sev[k], all_stages=True)
        torch.cuda.synchronize()
    # kernel pass (not part of the step timing): device time of each kernel inside
    # whole steps, from CUPTI records, without the event nodes' own cost
    def replay(k):
        if flush:
            scratch.zero_()
        if graphs is not None:
            graphs[k].replay()
        else:
            step(fev[k])

    nk = min(args.steps, 5)
    recs = cupti_kernels(replay, nk)
    kern = kernel_stage_us(recs, nk, wl.shared_F > 0) if recs else None
    if kern is not None and not kern[0]:  # no kernel of the library among the records
        kern = None
    if flush:
        step_ms = [begins[k].elapsed_time(marks[k]) for k in range(args.steps)]
    else:
        step_ms = [start.elapsed_time(marks[0])] + [marks[k - 1].elapsed_time(marks[k])
                                                    for k in range(1, args.steps)]
    if layer.device_status() != 0:
        raise RuntimeError("device status not clean after the timed region")
    ffn_ms = float(np.mean([fev[k][0].elapsed_time(fev[k][1]) for k in range(args.steps)]))
    stage_ms = {n: float(np.mean([sev[k][j].elapsed_time(sev[k][j + 1]) for k in range(args.steps)]))
                for j, (n, _) in enumerate(stages)}
    total_ms = float(sum(step_ms)) if flush else start.elapsed_time(end)
    clocks = clk.summary()
    clocks.update(probe_clock(probe.cpu().numpy(), start.elapsed_time(end)))
    return {"step_ms": step_ms, "total_ms": total_ms, "ffn_ms": ffn_ms, "stage_ms": stage_ms,
            "graph": graphs is not None, "clocks": clocks, "out": out, "stats": stats, "launches": nst,
            "kernels": kern}


_STAGE_OF = (("route", ("router_", "split_wg", "ec_scores", "ec_select", "fill_counts")),
             ("dispatch", ("dispatch_", "scatter_rows", "gather_rows")),
             ("combine", ("combine",)),
             ("load_stats", ("stats_",)))
_GEMM_NAMES = ("grouped_gemm", "fp8_ffn", "simt_gemm")


def kernel_stage_us(kernels, steps: int, shared: bool):
    """Per-kernel and per-stage device time (us per step) and the library's kernel
    launches per step, from (name, start_ns, duration_ns) records of `steps` whole
    steps.  A kernel belongs to the stage its name names; the grouped GEMM launches
    of a step are the routed experts' and, with a shared expert, its last two
    launches the shared expert's."""
    mine = sorted((k for k in kernels if "moe::" in k[0] and "clock_probe" not in k[0]), key=lambda k: k[1])
    per_kernel, per_stage = {}, {}
    gemms = [k for k in mine if any(g in k[0] for g in _GEMM_NAMES)]
    period = len(gemms) // steps if steps else 0
    for i, (name, _, dur) in enumerate(mine):
        short = name.replace("(anonymous namespace)::", "").replace("void ", "").split("(")[0]
        per_kernel[short] = per_kernel.get(short, 0.0) + dur / 1e3 / steps
        stage = "other"
        if any(g in name for g in _GEMM_NAMES):
            pos = gemms.index((name, mine[i][1], dur)) % period if period else 0
            stage = "shared_ffn" if shared and pos >= period - 2 else "expert_ffn"
        else:
            for st, keys in _STAGE_OF:
                if any(key in name for key in keys):
                    stage = st
                    break
        per_stage[stage] = per_stage.get(stage, 0.0) + dur / 1e3 / steps
    return per_kernel, per_stage, len(mine) / steps if steps else 0.0


def cupti_kernels(replay, steps: int):
    """(name, start_ns, duration_ns) of every kernel the `steps` calls of replay()
    launch, from CUPTI activity records (torch.profiler); None if unavailable."""
    import torch
    try:
        from torch.profiler import ProfilerActivity, profile
        with profile(activities=[ProfilerActivity.CUDA]) as prof:
            for k in range(steps):
                replay(k)
            torch.cuda.synchronize()
        out = []
        for ev in prof.events():
            if ev.device_type == torch.autograd.DeviceType.CUDA:
                tr = ev.time_range
                out.append((ev.name, int(tr.start * 1000), int((tr.end - tr.start) * 1000)))
        return out
    except Exception as exc:  # pragma: no cover - reported; the event-timed stages remain
        sys.stderr.write(f"CUPTI kernel records unavailable ({exc})\n")
        return None


def probe_clock(samples, region_ms: float) -> dict:
    """Median SM clock (MHz) over the probe's intervals that fall inside the timed
    region (the probe starts with it), from (ns, cycles) sample pairs."""
    s = np.asarray(samples, dtype=np.int64).reshape(-1, 2)
    s = s[s[:, 0] > 0]
    if len(s) < 2:
        return {}
    t, c = s[:, 0].astype(np.float64), s[:, 1].astype(np.float64)
    keep = t <= t[0] + region_ms * 1e6
    dt, dc = np.diff(t[keep]), np.diff(c[keep])
    ok = dt > 0
    if not np.any(ok):
        return {}
    mhz = dc[ok] / dt[ok] * 1e3
    return {"sm_mhz_in_band": float(np.median(mhz)), "sm_mhz_in_band_p10": float(np.percentile(mhz, 10)),
            "sm_mhz_in_band_p90": float(np.percentile(mhz, 90)), "in_band_intervals": int(ok.sum())}


def ffn_kernel_label(wl, fp8: bool) -> str:
    if fp8:
        if wl.T <= 64:
            return ("fp8_ffn_decode_kernel (tcgen05, E4M3 weights converted into tensor memory as the A operand), "
                    "moe_expert_ffn_fp8: gate/up and down in one cooperative launch")
        return ("grouped_gemm_fp8 (tcgen05, E4M3 weights converted into a shared-memory B operand), "
                "moe_expert_ffn_fp8: gate/up + down launches")
    if wl.dtype == "f32":
        return "simt_gemm_kernel (float32 CUDA-core FMA), moe_expert_ffn: gate/up + down launches"
    return "grouped_gemm (tcgen05), moe_expert_ffn: gate/up + down launches"


def launches_per_step(wl, fp8: bool) -> int:
    """Kernels of one step: route = split W_g + tensor-core logits + top-k (bf16, more
    than 64 tokens), one kernel (float32, 4 or 8 experts, more than 64 tokens) or
    CUDA-core logits + top-k; dispatch = histogram, scan, rank, copy (one fused
    kernel + copy for at most 128 tokens); experts 2 (1 for the one-launch FP8
    decode FFN); shared 2; combine 1; statistics 2 (1 for at most 32 tokens)."""
    ffn = 1 if (fp8 and wl.T <= 64) else 2
    if wl.dtype == "bf16":
        route = 3 if wl.T > 64 else 2
    else:
        route = 1 if (wl.T > 64 and wl.N in (4, 8)) else 2
    dispatch = 4 if wl.T > 128 else 2
    stats = 2 if wl.T > 32 else 1
    return route + dispatch + ffn + (2 if wl.shared_F else 0) + 1 + stats


def layer_report(wl, layer, t, peaks, peak_src, fp8: bool, steps: int, world: int = 1):
    """Tokens/s, stage rooflines and the dominant kernel's roofline object of one
    timed run `t` (time_layer's result)."""
    v = layer.views()
    counts_kept = v["counts_kept"].cpu().numpy()
    kept_rows = int(counts_kept.sum())
    touched = int(np.count_nonzero(counts_kept))
    work = stage_work(wl, kept_rows, touched, fp8)
    f32 = wl.dtype == "f32"
    clocks = t["clocks"]
    # per stage: its kernels' device time inside whole steps (CUPTI), else the time
    # between the events around it in the stage pass
    kern = t.get("kernels")
    stage_ms = dict(t["stage_ms"])
    if kern is not None:
        stage_ms.update({n: us / 1e3 for n, us in kern[1].items() if n in stage_ms})
    stages = {n: stage_roofline(work[n][0], work[n][1], ms, peaks, clocks,
                                alu=f32 and n in ("route", "expert_ffn", "shared_ffn"))
              for n, ms in stage_ms.items()}
    for n in stages:
        stages[n]["ms_events"] = t["stage_ms"][n]
        stages[n]["timing"] = "cupti kernel time in whole steps" if kern is not None else "events, stage pass"
    # the dominant kernel against its bound, from the events around it in the timed steps
    ffn = stage_roofline(work["expert_ffn"][0], work["expert_ffn"][1], t["ffn_ms"], peaks, clocks,
                         alu=f32)
    roof = {k: ffn[k] for k in ("bound", "achieved", "peak", "unit", "frac", "frac_clock_norm", "frac_sustained",
                                "tflops", "tensor_frac", "tensor_frac_clock_norm", "ms") if k in ffn}
    roof["traffic"] = _traffic(wl.name, fp8)
    roof["kernel"] = ffn_kernel_label(wl, fp8)
    roof["peak_source"] = ("derived float32 CUDA-core peak (148 SMs x 128 lanes x 2 FLOP x 2032 MHz)"
                           if ffn["bound"] == "alu" else
                           f"{peak_src} " + ("hbm_gbs" if ffn["bound"] == "hbm" else "bf16_tflops (burst)"))
    ms_per_step = t["total_ms"] / steps
    fl = layer_flops(wl, kept_rows)
    lb = layer_bytes(wl, touched, fp8)
    layer = {"flops": fl["total"], "tflops": fl["total"] / (ms_per_step / 1e3) / 1e12, "kept_rows": kept_rows,
             "touched_experts": touched, "algorithmic_bytes": lb, "gbs": lb / (ms_per_step / 1e3) / 1e9,
             "hbm_frac": lb / (ms_per_step / 1e3) / 1e9 / peaks["hbm_gbs"]}
    rep = {"value": wl.T * steps * world / (t["total_ms"] / 1e3), "ms_per_step": ms_per_step,
           "stages": stages, "roofline": roof, "layer": layer}
    if kern is not None:
        rep["kernels_us"] = {k: round(v, 2) for k, v in sorted(kern[0].items(), key=lambda kv: -kv[1])}
    return rep


def time_decode(args, moe, layer, peaks, peak_src, stream, fp8: bool):
    """The Mixtral-shaped decode layer (T = 16, the prefill layer's own weights and
    router) on the same GPU and process: its step, stages, and the layer's
    algorithmic bytes over the step time against the measured HBM bandwidth."""
    import torch
    dwl = synth.WORKLOADS["mixtral_decode"]
    x = _to_dev(synth.normal(dwl.seed, synth.TID_X, (dwl.T, dwl.d), 1.0, "bf16"), "bf16")
    cfg = moe.make_config(dwl.T, dwl.d, dwl.N, dwl.k, dwl.F, 0, moe.GATE_SOFTMAX_TOPK, moe.ACT_SWIGLU,
                          moe.DTYPE_BF16, 0)
    dl = moe.MoELayer(cfg, layer.Wg, layer.w1, layer.w3, layer.w2)
    if fp8:
        dl.fp8 = layer.fp8 if layer.fp8 is not None else dl.quantize_fp8()
        torch.cuda.synchronize()
    t = time_layer(args, moe, dl, x, dwl, stream)
    r = layer_report(dwl, dl, t, peaks, peak_src, fp8, args.steps)
    return {"workload": dwl.name, "T": dwl.T, "expert_weights": "fp8 e4m3, one float32 scale per row" if fp8
            else "bf16", "value": r["value"], "unit": "tokens/s", "ms_per_step": r["ms_per_step"],
            "step_ms_p50": float(np.percentile(t["step_ms"], 50)),
            "layer_bytes": r["layer"]["algorithmic_bytes"], "touched_experts": r["layer"]["touched_experts"],
            "achieved_gbs": r["layer"]["gbs"], "peak_gbs": peaks["hbm_gbs"], "frac": r["layer"]["hbm_frac"],
            "stages": r["stages"], "kernels_us": r.get("kernels_us"), "roofline": r["roofline"],
            "clocks": t["clocks"]}


def run_ours(args, wl, dist, rank, local):
    import torch

    import sparse_mixture_experts_62_b300 as moe

    torch.cuda.set_device(local)
    inp = synth.make_inputs(wl)
    layer = build_layer(moe, inp)
    if args.fp8:  # weights quantised once, outside the timed region (like any weight packing)
        if wl.dtype != "bf16":
            raise SystemExit("--fp8 needs a bf16 workload")
        layer.quantize_fp8()
        torch.cuda.synchronize()
    x = _to_dev(inp.x, wl.dtype)
    stream = torch.cuda.current_stream()
    t = time_layer(args, moe, layer, x, wl, stream, dist, local)
    t_max = max_over_ranks(dist, t["total_ms"])
    world = dist.get_world_size() if dist is not None else 1
    t["total_ms"] = t_max
    peaks, peak_src = measured_peaks()
    rep = layer_report(wl, layer, t, peaks, peak_src, args.fp8, args.steps, world)
    out, stats = t["out"], t["stats"]
    frac = rep["roofline"]["frac"]
    if frac > 1.15:  # above a measured peak by this much, the timed kernel is not doing the work
        raise RuntimeError(f"roofline fraction {frac:.3f} exceeds the measured peak: accounting error")

    # optional: the backward step (gradients of a fixed dout), graph-replayed
    bwd = None
    if args.backward:
        bwd = time_backward(args, moe, layer, x, wl, stream)
    # the decode-shaped layer on the prefill layer's weights, same process and GPU
    decode = decode_fp8 = None
    if wl.name == "mixtral_prefill" and not args.no_decode:
        decode = time_decode(args, moe, layer, peaks, peak_src, stream, args.fp8)
        if not args.fp8:  # the same decode step with the experts' weights in FP8 E4M3
            decode_fp8 = time_decode(args, moe, layer, peaks, peak_src, stream, True)

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
    if t["graph"]:
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

    if rank == 0:
        sys.stderr.write("per-stage ms: " + json.dumps({k: round(val, 4) for k, val in t["stage_ms"].items()}) + "\n")
        step_ms = t["step_ms"]
        # the library's kernels per step: counted from the CUPTI records where there
        # are some, else from the launch plan; plus the clock probe's one launch
        n_launch = launches_per_step(wl, args.fp8)
        if t.get("kernels") is not None:
            n_launch = int(round(t["kernels"][2]))
        line = {"metric": METRIC, "value": rep["value"], "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": rep["ms_per_step"], "higher_is_better": True,
                "scaling": "weak",
                "step_ms": {"p10": float(np.percentile(step_ms, 10)), "p50": float(np.percentile(step_ms, 50)),
                            "p90": float(np.percentile(step_ms, 90))},
                "vs_baseline": None, "dtype": wl.dtype, "data": "synthetic",
                "config": {**config_of(wl, args.fp8),
                           **({"expert_weights": "fp8 e4m3, one float32 scale per row"} if args.fp8 else {})},
                "launch": "cuda_graph" if t["graph"] else "eager",
                "roofline": rep["roofline"],
                "stages": rep["stages"],
                "layer": rep["layer"],
                "e2e": {"value": e2e_val, "unit": "tokens/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
                "kernels_us": rep.get("kernels_us"),
                # timed region: one step's launches per step, and the clock probe
                "gpu_launches": n_launch * args.steps + 1,
                **({"decode": decode} if decode is not None else {}),
                **({"decode_fp8": decode_fp8} if decode_fp8 is not None else {}),
                **({"backward": bwd} if bwd is not None else {}),
                "clocks": t["clocks"]}
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
                    help="tokens of the oracle's cpu_baseline step (as the reference arm's; 0 = skip)")
    ap.add_argument("--ref-sample", type=int, default=512, help="tokens per reference-arm step")
    ap.add_argument("--override", nargs="*", default=[], help="workload fields to change, e.g. N=32 T=1024")
    ap.add_argument("--eager", action="store_true", help="time eager launches instead of a CUDA-graph replay")
    ap.add_argument("--backward", action="store_true", help="also time the backward step (bf16 token choice)")
    ap.add_argument("--fp8", action="store_true", help="FP8 E4M3 expert weights with per-row scales (bf16 workloads)")
    ap.add_argument("--no-decode", action="store_true",
                    help="skip the decode-shaped layer that the Mixtral prefill run also times")
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
