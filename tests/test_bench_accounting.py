"""The bench's algorithmic FLOP and byte counts and its roofline arithmetic (CPU).

The counts are pinned against figures worked out independently from the model
shapes: the active FLOPs and algorithmic bytes of the Mixtral-shaped prefill and
decode layers, the DeepSeek-V3-shaped layer with its shared expert, and one
expert's bytes in bf16 and in FP8 with row scales.
"""
import numpy as np
import pytest

import bench
import synth

W = synth.WORKLOADS


def test_prefill_counts():
    wl = W["mixtral_prefill"]
    kept = wl.T * wl.k                                   # no capacity: every assignment kept
    fl = bench.layer_flops(wl, kept)
    # 8192 rows x (2 x 4096 x 14336 x 3) = 2.886 TFLOP; router 2 x 4096 x 4096 x 8
    assert fl["expert_ffn"] == pytest.approx(2.886e12, rel=1e-3)
    assert fl["router"] == 2 * 4096 * 4096 * 8
    # weights of all 8 experts (2.819 GB) + x and out (2 x 33.5 MB) + W_g
    assert bench.layer_bytes(wl, 8) == pytest.approx(2.886e9, rel=1e-3)
    assert bench.expert_weight_bytes(wl, False) == 3 * 4096 * 14336 * 2


def test_decode_counts():
    wl = W["mixtral_decode"]
    assert bench.expert_weight_bytes(wl, False) == pytest.approx(352.3e6, rel=1e-3)
    # FP8: one byte per weight plus a float32 scale per row of W1, W3 (F rows) and W2 (d rows)
    assert bench.expert_weight_bytes(wl, True) == 3 * 4096 * 14336 + (2 * 14336 + 4096) * 4
    assert bench.layer_flops(wl, 32)["expert_ffn"] == pytest.approx(11.27e9, rel=1e-3)


def test_dsv3_counts():
    wl = W["dsv3_finegrained"]
    fl = bench.layer_flops(wl, wl.T * wl.k)
    # routed 65536 rows x 2 x 7168 x 2048 x 3 + shared 8192 rows of the same = 6.494 TFLOP
    assert fl["expert_ffn"] + fl["shared_ffn"] == pytest.approx(6.494e12, rel=1e-3)
    # 256 experts (22.55 GB) + the shared expert + x and out + W_g = 22.88 GB
    assert bench.layer_bytes(wl, 256) == pytest.approx(22.88e9, rel=1e-3)


def test_stage_work_matches_layer_counts():
    wl = W["mixtral_prefill"]
    kept = wl.T * wl.k
    work = bench.stage_work(wl, kept, 8)
    assert work["expert_ffn"][0] == bench.layer_flops(wl, kept)["expert_ffn"]
    assert work["route"][0] == bench.layer_flops(wl, kept)["router"]
    # expert FFN bytes: touched weights + x_perm read + y_perm written
    assert work["expert_ffn"][1] == 8 * bench.expert_weight_bytes(wl, False) + 2 * kept * wl.d * 2
    # combine: y_perm read, out written, ids + weights
    assert work["combine"][1] == kept * wl.d * 2 + wl.T * wl.d * 2 + wl.T * wl.k * 8


def test_stage_roofline_picks_the_longer_bound():
    peaks = {"hbm_gbs": 6000.0, "bf16_tflops": 2000.0, "bf16_tflops_sustained": 1500.0}
    # 3 TFLOP and 3 GB: 1.5 ms at the burst tensor peak, 0.5 ms at HBM -> tensor, against the burst peak
    r = bench.stage_roofline(3e12, 3e9, 2.0, peaks)
    assert r["bound"] == "tensor" and r["peak"] == 2000.0
    assert r["achieved"] == pytest.approx(1500.0) and r["frac"] == pytest.approx(0.75)
    assert r["frac_sustained"] == pytest.approx(1.0) and "frac_clock_norm" not in r
    # a power cap seen in the clock samples changes no peak; the clock-normalised reading
    # divides by the burst peak scaled to the median sampled SM clock
    clocks = {"sm_mhz": 1016.0, "sm_max_mhz": 2032.0, "reasons": ["sw_power_cap"]}
    r = bench.stage_roofline(3e12, 3e9, 2.0, peaks, clocks)
    assert r["peak"] == 2000.0 and r["frac"] == pytest.approx(0.75)
    assert r["frac_clock_norm"] == pytest.approx(1.5)
    # 10 GFLOP and 3 GB: HBM governs; the tensor rate rides along
    r = bench.stage_roofline(1e10, 3e9, 1.0, peaks)
    assert r["bound"] == "hbm" and r["achieved"] == pytest.approx(3000.0) and r["frac"] == pytest.approx(0.5)
    assert r["tflops"] == pytest.approx(10.0) and r["tensor_frac"] == pytest.approx(0.005)
    r = bench.stage_roofline(1e12, 6e9, 1.0, peaks, clocks)  # 1 PFLOP/s at half the maximum clock
    assert r["bound"] == "hbm" and r["tensor_frac"] == pytest.approx(0.5)
    assert r["tensor_frac_clock_norm"] == pytest.approx(1.0)
    # float32 work against the CUDA-core peak
    r = bench.stage_roofline(1e9, 1e6, 1.0, peaks, alu=True)
    assert r["bound"] == "alu" and r["peak"] == pytest.approx(bench.F32_ALU_TFLOPS)


def test_l2_flush_only_when_the_weights_fit():
    assert bench.needs_l2_flush(W["shazeer_tiny_f32"])
    for name in ("mixtral_prefill", "mixtral_decode", "dsv3_finegrained", "qwen3_skew_drop"):
        assert not bench.needs_l2_flush(W[name]) and not bench.needs_l2_flush(W[name], True)


def test_traffic_only_for_the_captured_kernel_sources(tmp_path):
    """The traffic table row counts only while the kernel sources hash as they did
    when it was captured."""
    h = bench.kernel_source_hash(False)
    assert len(h) == 16 and h != bench.kernel_source_hash(True)
    p = tmp_path / "traffic.md"
    p.write_text("| workload | weights | sources | bytes | command |\n|---|---|---|---|---|\n"
                 f"| mixtral_prefill | bf16 | {h} | 3.5e9 | ncu ... |\n"
                 "| qwen3_skew_drop | bf16 | 0123456789abcdef | 1e9 | ncu ... |\n")
    table = bench.traffic_table(str(p))
    assert bench._traffic("mixtral_prefill", table=table) == 3.5e9
    assert bench._traffic("qwen3_skew_drop", table=table) is None      # captured on other sources
    assert bench._traffic("mixtral_prefill", True, table=table) is None
    assert bench._traffic("dsv3_finegrained", table=table) is None


def test_source_hash_ignores_comments_only():
    a = "int f(int x) {  // one\n  return x + 1; /* two\n lines */ }\n"
    b = "int f(int x) {\n  return x + 1;\n}\n"
    c = "int f(int x) { return x + 2; }"
    assert bench.code_of(a) == bench.code_of(b) != bench.code_of(c)


def test_fp32_kernel_label():
    assert "simt" in bench.ffn_kernel_label(W["shazeer_tiny_f32"], False)
    assert "tcgen05" in bench.ffn_kernel_label(W["mixtral_prefill"], False)
    assert "one cooperative launch" in bench.ffn_kernel_label(W["mixtral_decode"], True)


def test_reference_arm_prints_the_contract_line():
    """`bench.py --impl reference` times the oracle on host cores and prints one JSON
    line with the same metric and config as the GPU arm, a cpu_baseline describing
    the run, and an e2e of its own value with no host-device bytes."""
    import json
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference", "--workload",
                        "shazeer_tiny_f32", "--steps", "2", "--warmup", "3"], capture_output=True, text=True,
                       timeout=600, cwd=root)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "tokens/s"
    assert d["value"] > 0 and d["higher_is_better"] is True and d["steps"] == 2 and d["warmup"] == 3
    assert d["config"]["workload"] == "shazeer_tiny_f32" and d["vs_baseline"] is None
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_probe_clock_median_inside_the_timed_region():
    # samples every 200 us: 1500 MHz for the first 1 ms, then 2000 MHz; region of 1 ms
    t = np.arange(11) * 200_000
    c = np.concatenate([[0], np.cumsum(np.where(np.arange(1, 11) <= 5, 1500 * 200, 2000 * 200))])
    s = np.stack([t + 10**9, c], axis=1).ravel()
    r = bench.probe_clock(s, 1.0)
    assert r["sm_mhz_in_band"] == pytest.approx(1500.0) and r["in_band_intervals"] == 5
    r = bench.probe_clock(s, 2.0)
    assert r["in_band_intervals"] == 10
    assert bench.probe_clock(np.zeros(8, np.int64), 1.0) == {}


def test_clock_norm_prefers_the_in_band_clock():
    peaks = {"hbm_gbs": 6000.0, "bf16_tflops": 2000.0, "bf16_tflops_sustained": 1500.0, "sm_max_mhz": 2000.0}
    clocks = {"sm_mhz": 2000.0, "sm_max_mhz": 2000.0, "sm_mhz_in_band": 1500.0}
    r = bench.stage_roofline(3e12, 3e9, 2.0, peaks, clocks)
    assert r["frac"] == pytest.approx(0.75) and r["frac_clock_norm"] == pytest.approx(1.0)


def test_kernel_records_to_stages():
    """CUPTI-style (name, start, duration) records of two steps: stages by kernel
    name, the last two grouped GEMM launches of each step to the shared expert, the
    clock probe and foreign kernels left out."""
    step = [("void moe::rtc::split_wg_kernel(float)", 2000), ("void moe::rtc::router_gemm_kernel<128>(x)", 10000),
            ("void moe::(anonymous namespace)::router_topk_kernel<4>(x)", 5000),
            ("void moe::(anonymous namespace)::dispatch_hist_kernel(x)", 1000),
            ("void moe::(anonymous namespace)::scatter_rows_kernel(x)", 3000),
            ("void moe::tc::grouped_gemm_kernel<0>(x)", 100000), ("void moe::tc::grouped_gemm_kernel<2>(x)", 50000),
            ("void moe::tc::grouped_gemm_pair_kernel<0>(x)", 20000),
            ("void moe::tc::grouped_gemm_pair_kernel<2>(x)", 10000),
            ("void moe::(anonymous namespace)::combine_warp_kernel<true, 8>(x)", 4000),
            ("void moe::(anonymous namespace)::stats_partial_kernel(x)", 700),
            ("void moe::(anonymous namespace)::stats_final_kernel(x)", 800),
            ("void at::native::elementwise_kernel<...>(x)", 9999)]
    recs, t = [], 0
    for _ in range(2):
        for name, dur in step:
            recs.append((name, t, dur))
            t += dur + 100
    recs.append(("void moe::(anonymous namespace)::clock_probe_kernel(x)", 0, 10**7))
    per_kernel, per_stage, per_step = bench.kernel_stage_us(recs, 2, shared=True)
    assert per_step == 12
    assert per_stage["route"] == pytest.approx(17.0) and per_stage["dispatch"] == pytest.approx(4.0)
    assert per_stage["expert_ffn"] == pytest.approx(150.0) and per_stage["shared_ffn"] == pytest.approx(30.0)
    assert per_stage["combine"] == pytest.approx(4.0) and per_stage["load_stats"] == pytest.approx(1.5)
    assert "other" not in per_stage and per_kernel["moe::tc::grouped_gemm_kernel<0>"] == pytest.approx(100.0)
    # without a shared expert every grouped GEMM launch is the routed experts'
    _, per_stage, _ = bench.kernel_stage_us(recs, 2, shared=False)
    assert per_stage["expert_ffn"] == pytest.approx(180.0) and "shared_ffn" not in per_stage
