"""Helpers for the GPU-vs-oracle parity tests (imported by the tests only).

The oracle always runs on the seeded inputs alone, with its own routing; nothing
the GPU computed is ever fed to it.  Parity rules (bf16 workloads; the float32
workload uses 1e-4 relative):
  * top-k against the GPU's own logits: on every token, the GPU's experts and
    their slot order are exactly the (selection score desc, index asc) top-k
    of the selection scores that its own dumped float32 logits define, worked
    out here in double (sigmoid rounded once to float32, then + b in float32);
    its gate weights are within 1e-6 of the gate those logits define.  Exact
    ties go to the lower index, so this also pins the tie-break.
  * top-k against the oracle: every token whose oracle gap between the k-th and
    (k+1)-th selection scores exceeds 1e-4 must have the oracle's set, and its
    order where the gaps between adjacent selected scores also exceed 1e-4.  A
    token where the GPU's choice differs from the oracle's must be a valid
    choice by the oracle's scores (every expert above the k-th score + 1e-4
    taken, nothing below the k-th score - 1e-4, order descending up to 1e-4);
    such tokens must be rare (at most max(1, T / 1000)).
  * gate weights: within 1e-6 of the oracle's on tokens whose top-k equals it.
  * dispatch: equal to the oracle's where no differing token touches the expert;
    every expert's rows, counts and offsets satisfy the dispatch definition on the
    GPU's own top-k.
  * layer output: max|gpu - ref| <= 2e-2 * max|ref| + 1e-3 (bf16), <= 1e-4 * max|ref|
    (float32).  A token whose top-k and kept set equal the oracle's is compared
    with the oracle's output row; any other token with the sum, over the slots
    the GPU kept, of the gate (from the GPU's logits) times the oracle's expert
    output for the expert the GPU chose (plus the oracle's shared expert).
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


def own_logit_routing(z_gpu: np.ndarray, gate: str, sel_bias, k: int):
    """The top-k and gate weights that the GPU's dumped float32 logits define,
    worked out here from the definitions (not by the oracle, which never sees a
    GPU result): selection score z (softmax gates) or fl32(fl32(sigmoid(z)) + b)
    (sigmoid gate, sigmoid in double); experts ordered by (score desc, index asc)
    -- a stable sort keeps equal scores in index order, so exact ties go to the
    lower index; gates: softmax over the selected logits, the full softmax kept
    on the selected, or the raw affinities normalised over the selected.
    Returns (idx [T, k] int32, w [T, k] float64, sel [T, N] float32)."""
    z64 = z_gpu.astype(np.float64)
    s = None
    if gate == "sigmoid":
        s = (1.0 / (1.0 + np.exp(-z64))).astype(np.float32)
        sel = s if sel_bias is None else (s + np.asarray(sel_bias, np.float32)[None, :]).astype(np.float32)
    else:
        sel = z_gpu.astype(np.float32)
    order = np.argsort(-sel, axis=1, kind="stable")
    idx = order[:, :k].astype(np.int32)
    rows = np.arange(z64.shape[0])[:, None]
    if gate == "softmax":
        zs = z64[rows, idx]
        e = np.exp(zs - zs.max(axis=1, keepdims=True))
        w = e / e.sum(axis=1, keepdims=True)
    elif gate == "softmax_full":
        m = z64.max(axis=1, keepdims=True)
        e = np.exp(z64 - m)
        w = e[rows, idx] / e.sum(axis=1, keepdims=True)
    else:
        ss = s.astype(np.float64)[rows, idx]
        w = ss / ss.sum(axis=1, keepdims=True)
    return idx, w, sel


def check_own_logits(z_gpu: np.ndarray, idx_gpu: np.ndarray, w_gpu: np.ndarray, gate: str, sel_bias, k: int):
    """Every token's top-k (set and slot order) bit-exact, and its gate weights
    within 1e-6, against what the GPU's own logits define.  Returns the gate
    weights those logits define (float64)."""
    idx_own, w_own, _ = own_logit_routing(z_gpu, gate, sel_bias, k)
    bad = np.nonzero(np.any(idx_gpu != idx_own, axis=1))[0]
    assert bad.size == 0, (f"{bad.size} tokens' top-k differ from the top-k of the GPU's own logits "
                           f"(first: token {bad[0]}: gpu {idx_gpu[bad[0]].tolist()}, "
                           f"own logits {idx_own[bad[0]].tolist()})" if bad.size else "")
    assert np.max(np.abs(w_gpu - w_own), initial=0.0) <= 1e-6, "gate weights differ from the GPU's own logits' gate"
    return w_own


def check_routing(inp, z_gpu: np.ndarray, idx_gpu: np.ndarray, w_gpu: np.ndarray, ref: oracle.LayerResult):
    """Top-k and gate parity: against the GPU's own logits on every token, and
    against the oracle's own routing `ref`.  Returns the mask of tokens whose
    top-k equals the oracle's, slot by slot."""
    wl = inp.wl
    k, N, T = wl.k, wl.N, wl.T
    check_own_logits(z_gpu, idx_gpu, w_gpu, wl.gate, inp.sel_bias, k)
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


def rows_by_gpu_routing(inp, ref: oracle.LayerResult, tokens, z_gpu, idx_gpu, dest_row) -> np.ndarray:
    """Expected output rows [len(tokens), d] for tokens whose routing or kept set
    differs from the oracle's: the oracle's shared-expert row plus, over the slots
    the GPU kept (dest_row >= 0), the gate that the GPU's logits define times the
    oracle's output of the chosen expert on that token.  The chosen experts have
    been checked to be valid by the oracle's own scores (check_routing) and the
    kept slots to follow the dispatch definition (check_dispatch_definition)."""
    wl = inp.wl
    tokens = np.asarray(tokens, dtype=np.int64)
    out = np.zeros((tokens.size, wl.d))
    if tokens.size == 0:
        return out
    _, w_own, _ = own_logit_routing(z_gpu[tokens], wl.gate, inp.sel_bias, wl.k)
    x64 = oracle.widen(inp.x[tokens], wl.dtype)
    if ref.y_sh is not None:
        out += ref.y_sh[tokens]
    for e in np.unique(idx_gpu[tokens]):
        hit = [(i, j) for i, t in enumerate(tokens) for j in range(wl.k)
               if idx_gpu[t, j] == e and dest_row[t, j] >= 0]
        if not hit:
            continue
        ii = np.array([i for i, _ in hit])
        W3 = oracle.widen(inp.w3[e], wl.dtype) if inp.w3 is not None else None
        y = oracle.expert_ffn(x64[ii], oracle.widen(inp.w1[e], wl.dtype), W3, oracle.widen(inp.w2[e], wl.dtype),
                              wl.act)
        for r, (i, j) in enumerate(hit):
            out[i] += w_own[i, j] * y[r]
    return out


def assert_close_out(gpu: np.ndarray, ref: np.ndarray, dtype: str, what="output"):
    scale = float(np.max(np.abs(ref))) if ref.size else 0.0
    err = float(np.max(np.abs(gpu - ref))) if ref.size else 0.0
    tol = 2e-2 * scale + 1e-3 if dtype == "bf16" else 1e-4 * scale
    assert err <= tol, f"{what}: max|gpu-ref| = {err:.3e} > tol {tol:.3e} (max|ref| = {scale:.3e})"
    return err, tol
