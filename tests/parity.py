"""Helpers for the GPU-vs-oracle parity tests (imported by the tests only).

Parity rules (bf16 workloads; the float32 workload uses 1e-4 relative):
  * top-k: the set is compared exactly on every token whose oracle gap between
    the k-th and (k+1)-th selection scores exceeds 1e-4; the order inside the
    set exactly where the gaps between adjacent selected scores also exceed
    1e-4.  The remaining (near-tie) tokens are checked by running the oracle's
    selection on the GPU's own float32 logits, which must reproduce the GPU's
    choice exactly.
  * gate weights: within 1e-6 of the oracle's weights at the GPU's indices.
  * dispatch (counts, offsets, dest_row, src_token, the drop set): exact,
    against the oracle's dispatch of the GPU's top-k.
  * layer output: max|gpu - ref| <= 2e-2 * max|ref| + 1e-3 (bf16), <= 1e-4 * max|ref|
    (float32), with the oracle run on the GPU's top-k.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import sparse_mixture_experts_62_b300 as moe
import synth

GAP = 1e-4


def to_dev(a, dtype: str, device="cuda"):
    """numpy input (bf16 bits as uint16, or float32) -> device tensor."""
    if a is None:
        return None
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(device)


def to_np_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def config_of(wl: synth.Workload):
    cap = oracle.capacity(wl.capacity_factor, wl.T, wl.k, wl.N) if wl.capacity_factor > 0 else 0
    return moe.make_config(wl.T, wl.d, wl.N, wl.k, wl.F, wl.shared_F,
                           {"softmax": moe.GATE_SOFTMAX_TOPK, "sigmoid": moe.GATE_SIGMOID_BIAS,
                           "softmax_full": moe.GATE_SOFTMAX_FULL}[wl.gate],
                           moe.ACT_SWIGLU if wl.act == "swiglu" else moe.ACT_RELU,
                           moe.DTYPE_BF16 if wl.dtype == "bf16" else moe.DTYPE_F32, cap)


def layer_on_device(inp) -> moe.MoELayer:
    wl = inp.wl
    dt = wl.dtype
    f32 = lambda a: None if a is None else to_dev(a, "f32")  # noqa: E731
    return moe.MoELayer(config_of(wl), f32(inp.Wg), to_dev(inp.w1, dt), to_dev(inp.w3, dt), to_dev(inp.w2, dt),
                        to_dev(inp.sw1, dt), to_dev(inp.sw3, dt), to_dev(inp.sw2, dt), f32(inp.logit_bias),
                        f32(inp.sel_bias))


def check_routing(inp, z_gpu: np.ndarray, idx_gpu: np.ndarray, w_gpu: np.ndarray, ref: oracle.LayerResult):
    """Top-k and gate parity; returns the number of near-tie tokens."""
    wl = inp.wl
    k, N = wl.k, wl.N
    # logits agree to float32 accumulation error
    assert np.max(np.abs(z_gpu.astype(np.float64) - ref.z.astype(np.float64))) < 1e-3, "router logits differ"
    sel = ref.sel.astype(np.float64)
    srt = -np.sort(-sel, axis=1)
    kth_gap = (srt[:, k - 1] - srt[:, k]) if k < N else np.full(wl.T, np.inf)
    clear = kth_gap > GAP
    # sets on clear tokens
    a = np.sort(idx_gpu[clear], axis=1)
    b = np.sort(ref.idx[clear], axis=1)
    assert np.array_equal(a, b), f"top-k sets differ on {np.sum(np.any(a != b, axis=1))} clear tokens"
    # order where adjacent selected gaps are also clear
    adj = np.all((srt[:, :k - 1] - srt[:, 1:k]) > GAP, axis=1) if k > 1 else np.ones(wl.T, bool)
    ordered = clear & adj
    assert np.array_equal(idx_gpu[ordered], ref.idx[ordered]), "top-k order differs"
    # near-tie tokens: the oracle's selection on the GPU's own logits
    near = ~clear
    if np.any(near):
        sel_g, _ = oracle.selection_scores(z_gpu[near], wl.gate, inp.sel_bias)
        assert np.array_equal(oracle.topk(sel_g, k), idx_gpu[near]), "near-tie selection differs"
    # gate weights at the GPU's indices
    _, s = oracle.selection_scores(ref.z, wl.gate, inp.sel_bias)
    w_ref = oracle.gate_weights(ref.z, s, idx_gpu, wl.gate)
    assert np.max(np.abs(w_gpu - w_ref)) <= 1e-6, f"gate weights differ by {np.max(np.abs(w_gpu - w_ref))}"
    return int(np.sum(near))


def check_dispatch(wl, idx_gpu, counts_routed, counts_kept, offsets, dest_row, src_token, cap):
    d = oracle.dispatch(idx_gpu, wl.N, cap)
    assert np.array_equal(counts_routed, d.counts_routed)
    assert np.array_equal(counts_kept, d.counts_kept)
    assert np.array_equal(offsets, d.offsets)
    assert np.array_equal(dest_row, d.dest_row)
    S = int(d.offsets[-1])
    assert np.array_equal(src_token[:S], d.src_token)
    return d


def assert_close_out(gpu: np.ndarray, ref: np.ndarray, dtype: str, what="output"):
    scale = float(np.max(np.abs(ref))) if ref.size else 0.0
    err = float(np.max(np.abs(gpu - ref))) if ref.size else 0.0
    tol = 2e-2 * scale + 1e-3 if dtype == "bf16" else 1e-4 * scale
    assert err <= tol, f"{what}: max|gpu-ref| = {err:.3e} > tol {tol:.3e} (max|ref| = {scale:.3e})"
    return err, tol
