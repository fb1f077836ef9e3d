"""Helpers for the GPU-vs-oracle parity tests (imported by the tests only).

The oracle always runs on the seeded inputs alone, with its own routing; nothing
the GPU computed is ever fed to it.  Parity rules (bf16 workloads; the float32
workload uses 1e-4 relative):
  * top-k: every token whose oracle gap between the k-th and (k+1)-th selection
    scores exceeds 1e-4 must have the oracle's set, and its order where the gaps
    between adjacent selected scores also exceed 1e-4.  A token where the GPU's
    choice differs from the oracle's must be a valid choice by the oracle's
    scores (every expert above the k-th score + 1e-4 taken, nothing below the
    k-th score - 1e-4, order descending up to 1e-4); such tokens must be rare
    (at most max(1, T / 1000)) and are left out of the float comparisons below.
  * gate weights: within 1e-6 of the oracle's on tokens whose top-k equals it.
  * dispatch: equal to the oracle's where no differing token touches the expert;
    every expert's rows, counts and offsets satisfy the dispatch definition on the
    GPU's own top-k.
  * layer output: max|gpu - ref| <= 2e-2 * max|ref| + 1e-3 (bf16), <= 1e-4 * max|ref|
    (float32), on tokens whose top-k and kept set equal the oracle's.
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
    """Top-k and gate parity against the oracle's own routing `ref`.  Returns the
    mask of tokens whose top-k equals the oracle's, slot by slot."""
    wl = inp.wl
    k, N, T = wl.k, wl.N, wl.T
    # logits agree to float32 accumulation error
    assert np.max(np.abs(z_gpu.astype(np.float64) - ref.z.astype(np.float64))) < 1e-3, "router logits differ"
    assert np.all((idx_gpu >= 0) & (idx_gpu < N)), "expert index out of range"
    assert np.all(np.sort(idx_gpu, axis=1)[:, 1:] != np.sort(idx_gpu, axis=1)[:, :-1]), "repeated expert"
    sel = ref.sel.astype(np.float64)
    srt = -np.sort(-sel, axis=1)
    kth_gap = (srt[:, k - 1] - srt[:, k]) if k < N else np.full(T, np.inf)
    clear = kth_gap > GAP
    a = np.sort(idx_gpu[clear], axis=1)
    b = np.sort(ref.idx[clear], axis=1)
    assert np.array_equal(a, b), f"top-k sets differ on {np.sum(np.any(a != b, axis=1))} clear tokens"
    adj = np.all((srt[:, :k - 1] - srt[:, 1:k]) > GAP, axis=1) if k > 1 else np.ones(T, bool)
    ordered = clear & adj
    assert np.array_equal(idx_gpu[ordered], ref.idx[ordered]), "top-k order differs"
    same = np.all(idx_gpu == ref.idx, axis=1)
    diff = np.nonzero(~same)[0]
    assert diff.size <= max(1, T // 1000), f"{diff.size} tokens routed differently from the oracle"
    for t in diff:  # a valid choice by the oracle's scores
        kth = srt[t, k - 1]
        chosen = sel[t, idx_gpu[t]]
        assert np.all(chosen >= kth - GAP), f"token {t}: an expert below the k-th score"
        must = np.nonzero(sel[t] > kth + GAP)[0]
        assert set(must.tolist()) <= set(idx_gpu[t].tolist()), f"token {t}: a clear winner left out"
        assert np.all(chosen[:-1] >= chosen[1:] - GAP), f"token {t}: order"
    # gate weights where the routing is the oracle's
    assert np.max(np.abs(w_gpu[same] - ref.w[same]), initial=0.0) <= 1e-6, "gate weights differ"
    return same


def check_dispatch_definition(N, idx, cap, counts_routed, counts_kept, offsets, dest_row, src_token):
    """The dispatch of `idx` by definition: per-expert histogram, the first `cap`
    assignments in token order kept (all when cap = 0), rows grouped by expert in
    token order, dest_row the inverse of src_token, -1 for a dropped assignment."""
    T, k = idx.shape
    assert np.array_equal(counts_routed, np.bincount(idx.ravel(), minlength=N))
    assert np.array_equal(counts_kept, np.minimum(counts_routed, cap) if cap > 0 else counts_routed)
    assert np.array_equal(offsets, np.concatenate([[0], np.cumsum(counts_kept)]))
    expect = np.full((T, k), -1, dtype=np.int64)
    for e in range(N):
        tt, jj = np.nonzero(idx == e)                  # row-major: ascending token order
        n = int(counts_kept[e])
        seg = src_token[offsets[e]:offsets[e] + n]
        assert np.array_equal(seg, tt[:n]), f"expert {e}: rows"
        expect[tt[:n], jj[:n]] = offsets[e] + np.arange(n)
    assert np.array_equal(dest_row, expect)


def check_layer_dispatch(wl, idx_gpu, same, counts_routed, counts_kept, offsets, dest_row, src_token, cap,
                         ref: oracle.LayerResult):
    """The GPU's dispatch against the oracle's own.  Returns the mask of tokens
    whose top-k and kept set both equal the oracle's."""
    check_dispatch_definition(wl.N, idx_gpu, cap, counts_routed, counts_kept, offsets, dest_row, src_token)
    ref_disp = ref.disp
    ref_kept = ref_disp.dest_row >= 0
    if np.all(same):
        assert np.array_equal(counts_routed, ref_disp.counts_routed)
        assert np.array_equal(counts_kept, ref_disp.counts_kept)
        assert np.array_equal(offsets, ref_disp.offsets)
        assert np.array_equal(dest_row, ref_disp.dest_row)
        assert np.array_equal(src_token[:int(offsets[-1])], ref_disp.src_token)
        return np.ones(wl.T, bool)
    # experts that a differing token touches, on either side, may differ
    touched = set()
    diff = np.nonzero(~same)[0]
    touched.update(idx_gpu[diff].ravel().tolist())
    touched.update(ref.idx[diff].ravel().tolist())
    for e in range(wl.N):
        if e in touched:
            continue
        assert counts_routed[e] == ref_disp.counts_routed[e] and counts_kept[e] == ref_disp.counts_kept[e]
        a = src_token[offsets[e]:offsets[e + 1]]
        b = ref_disp.src_token[ref_disp.offsets[e]:ref_disp.offsets[e + 1]]
        assert np.array_equal(a, b), f"expert {e}: rows"
    return same & np.all((dest_row >= 0) == ref_kept, axis=1)


def check_dispatch(wl, idx, counts_routed, counts_kept, offsets, dest_row, src_token, cap):
    """The GPU's dispatch of a host-made top-k `idx` against the oracle's dispatch
    of the same `idx`: exact."""
    d = oracle.dispatch(idx, wl.N, cap)
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
