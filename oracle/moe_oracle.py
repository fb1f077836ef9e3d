"""CPU oracle of the sparse token-choice Mixture-of-Experts FFN layer forward.

TEST INFRASTRUCTURE ONLY.  Nothing in the library imports this file; only the
tests, the smoke check and the CPU-baseline leg of the benchmark call it.  It
shares no code with the CUDA path.

Plain numpy, float64 arithmetic, written for a reader checking it against the
pages by eye:

  * "Lecture29" (CS25 lecture 29 notes, Mixtral): section "Top-two routing: from
    logits to weighted expert output" -- router logits z, top-k set S_k(x), gate
    g_i = exp(z_i) / sum_{j in S_k} exp(z_j), output y = sum_i g_i Expert_i(x);
    section "A dense Transformer layer" -- the SwiGLU expert W2(SiLU(W1 x) * W3 x);
    section "Inference load balance" -- capacity C = ceil(alpha T k / E);
    section "Myth 3" -- the imbalance ratio I = max_i n_i / (T k / E).
  * "Chapter 19: MoE" (awesome-ai-roadmap): 19.3.2 -- softmax over the selected
    logits equals the full softmax renormalised over the top-k; 19.3.3 -- the
    Switch balance quantities f_i and P_i; 19.3.4 -- DeepSeek-V3 selection bias
    used only for choosing experts, mixing weights from the raw affinities;
    19.6.1 -- T k / N assignments per expert on average, overflow dropped with
    the residual path kept.
  * "Stanford CS336 lecture 4: Mixture of Experts": section 5 (top-K routing,
    the router is a linear scorer); section 6 (shared experts, always on);
    section 9 (loss N * sum_i f_i P_i; DeepSeek-V3 bias b_i used only for
    routing); section 10 (a dropped token's expert output is zero, the residual
    passes); section 11 (router kept in float32).
  * "Outrageously Large Neural Networks" notes (Shazeer et al. 2017): the gate
    matrix W_g is d x n; each expert is a one-hidden-layer ReLU network
    512 -> 1024 -> 512 with no biases.

Readings where the pages leave a step open (each is listed in the design notes):
  - top-k order: selection score descending, ties to the lower expert index;
  - capacity keeps, per expert, the first C assignments in ascending token
    index regardless of the slot j; no renormalisation after a drop;
  - f_i counts routed assignments before capacity, divided by T*k;
  - P_i: the full N-way softmax of z (softmax gate) or s_i / sum_l s_l
    (sigmoid gate, without the selection bias);
  - the sigmoid affinity s = fl32(1 / (1 + exp(-z))) computed in double, the
    selection score fl32(s + b);
  - the output is the MoE branch only (the residual add belongs to the caller).
"""
from __future__ import annotations

import concurrent.futures
import dataclasses
import os
from fractions import Fraction
from typing import Optional

import numpy as np


# --------------------------------------------------------------------------- inputs
def widen(a: np.ndarray, dtype: str) -> np.ndarray:
    """Exact float64 value of a stored tensor: bf16 bit patterns (uint16) or float32."""
    if dtype == "bf16":
        return (np.asarray(a).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return np.asarray(a, dtype=np.float32).astype(np.float64)


# --------------------------------------------------------------------------- routing
def router_logits(x64: np.ndarray, Wg: np.ndarray, logit_bias: Optional[np.ndarray]) -> np.ndarray:
    """z = x . W_g (+ beta), summed in double and rounded once to float32.

    Lecture29, "Top-two routing" (z = W_r x); CS336 lecture 4, section 5 (the
    router is a linear scorer, not an MLP) and section 11 (router in float32).
    beta is the workload's additive logit skew (zero unless given)."""
    z = x64 @ Wg.astype(np.float64)
    if logit_bias is not None:
        z = z + logit_bias.astype(np.float64)[None, :]
    return z.astype(np.float32)


def sigmoid_affinity(z: np.ndarray) -> np.ndarray:
    """DeepSeek-V3 affinity s = sigmoid(z), computed in double, rounded to float32.

    Chapter 19, 19.3.2 and 19.3.4 (sigmoid affinity, not a softmax)."""
    z64 = z.astype(np.float64)
    return (1.0 / (1.0 + np.exp(-z64))).astype(np.float32)


def selection_scores(z: np.ndarray, gate: str, sel_bias: Optional[np.ndarray]):
    """Returns (sel, s): the scores top-k ranks on, and the sigmoid affinities (or None).

    softmax gates: sel = z (softmax is monotone, so ranking z ranks the
    probabilities).  sigmoid gate: sel = fl32(s + b), where the bias b only
    steers the choice (Chapter 19, 19.3.4; CS336 lecture 4, section 9)."""
    if gate in ("softmax", "softmax_full"):
        return z, None
    s = sigmoid_affinity(z)
    if sel_bias is None:
        return s, s
    sel = (s.astype(np.float64) + sel_bias.astype(np.float64)[None, :]).astype(np.float32)
    return sel, s


def topk(sel: np.ndarray, k: int) -> np.ndarray:
    """Indices of the k largest scores per token, ordered by (score desc, index asc).

    Lecture29, "Top-two routing" (S_k(x) = indices of the k largest logits).
    A stable sort of the negated scores keeps equal scores in index order."""
    order = np.argsort(-sel, axis=1, kind="stable")
    return order[:, :k].astype(np.int32)


def gate_weights(z: np.ndarray, s: Optional[np.ndarray], idx: np.ndarray, gate: str) -> np.ndarray:
    """Gate weight of each selected slot, float64.

    softmax: g_j = exp(z_j) / sum_{l in S} exp(z_l)  (Lecture29 "Top-two routing";
      shifted by the selected maximum, which cancels).
    softmax_full: g_j = exp(z_j) / sum_{l=1..N} exp(z_l), the full softmax kept
      on the top-k and not renormalised (CS336 lecture 4, section 5 pseudocode:
      s = softmax(u . e); g_i = s_i if i in TopK(s) else 0).
    sigmoid: g_j = s_j / sum_{l in S} s_l from the raw affinities, no bias
      (Chapter 19, 19.3.4)."""
    T, k = idx.shape
    w = np.zeros((T, k), dtype=np.float64)
    for t in range(T):
        if gate == "softmax":
            zs = z[t, idx[t]].astype(np.float64)
            e = np.exp(zs - zs.max())
            w[t] = e / e.sum()
        elif gate == "softmax_full":
            zt = z[t].astype(np.float64)
            e = np.exp(zt - zt.max())
            w[t] = e[idx[t]] / e.sum()
        else:
            ss = s[t, idx[t]].astype(np.float64)
            w[t] = ss / ss.sum()
    return w


# --------------------------------------------------------------------------- dispatch
def capacity(alpha: float, T: int, k: int, N: int) -> int:
    """C = ceil(alpha * T * k / N), exactly (alpha taken as its exact binary value).

    Lecture29, "Inference load balance"; Chapter 19, 19.6.1."""
    return int(-((-Fraction(alpha) * T * k) // N))


@dataclasses.dataclass
class Dispatch:
    counts_routed: np.ndarray   # [N] int32
    counts_kept: np.ndarray     # [N] int32
    offsets: np.ndarray         # [N+1] int32, exclusive scan of counts_kept
    dest_row: np.ndarray        # [T, k] int32, -1 = dropped
    src_token: np.ndarray       # [S] int32, token of each permuted row


def dispatch(idx: np.ndarray, N: int, cap: int) -> Dispatch:
    """Group the (token, slot) assignments by expert.

    Lecture29, "Top-k routing semantics" (rearrange tokens by expert, then
    restore the order) and "Inference load balance" (an expert holds at most C
    assignments; overflow is dropped).  Per expert, assignments are ranked by
    token index -- a token picks an expert at most once, so the token alone
    orders them, whatever the slot j -- and rank r is kept iff r < C.
    cap <= 0 means no limit."""
    T, k = idx.shape
    counts_routed = np.zeros(N, dtype=np.int64)
    for t in range(T):
        for j in range(k):
            counts_routed[idx[t, j]] += 1
    limit = cap if cap > 0 else T * k
    counts_kept = np.minimum(counts_routed, limit)
    offsets = np.zeros(N + 1, dtype=np.int64)
    for e in range(N):
        offsets[e + 1] = offsets[e] + counts_kept[e]
    seen = np.zeros(N, dtype=np.int64)
    dest_row = np.full((T, k), -1, dtype=np.int64)
    src_token = np.zeros(offsets[N], dtype=np.int64)
    for t in range(T):
        for j in range(k):
            e = idx[t, j]
            r = seen[e]
            seen[e] += 1
            if r < limit:
                dest_row[t, j] = offsets[e] + r
                src_token[offsets[e] + r] = t
    return Dispatch(counts_routed.astype(np.int32), counts_kept.astype(np.int32),
                    offsets.astype(np.int32), dest_row.astype(np.int32), src_token.astype(np.int32))


# --------------------------------------------------------------------------- experts
def silu(a: np.ndarray) -> np.ndarray:
    return a / (1.0 + np.exp(-a))


def expert_ffn(xr: np.ndarray, W1: np.ndarray, W3: Optional[np.ndarray], W2: np.ndarray, act: str) -> np.ndarray:
    """One expert on rows xr [m, d] (float64); W1, W3: [F, d]; W2: [d, F].

    swiglu: W2 (SiLU(W1 x) * W3 x)   (Lecture29, "A dense Transformer layer")
    relu:   W2 ReLU(W1 x)            (Shazeer et al. notes: one ReLU hidden layer)
    The hidden activation stays in float64 (no rounding)."""
    a = xr @ W1.T
    if act == "swiglu":
        h = silu(a) * (xr @ W3.T)
    else:
        h = np.maximum(a, 0.0)
    return h @ W2.T


def combine(y_rows: np.ndarray, dest_row: np.ndarray, w: np.ndarray, y_shared: Optional[np.ndarray]) -> np.ndarray:
    """out[t] = y_shared[t] + sum over kept slots j of w[t, j] * y_rows[dest_row[t, j]].

    Lecture29, "Top-two routing" (y = sum_i g_i Expert_i(x)) and "Top-k routing
    semantics" (restore the token order); CS336 lecture 4, section 10 (a dropped
    slot, dest_row = -1, adds nothing)."""
    T, k = dest_row.shape
    out = np.zeros((T, y_rows.shape[1])) if y_shared is None else np.array(y_shared, dtype=np.float64)
    for t in range(T):
        for j in range(k):
            r = dest_row[t, j]
            if r >= 0:
                out[t] += w[t, j] * y_rows[r]
    return out


# --------------------------------------------------------------------------- stats
@dataclasses.dataclass
class LoadStats:
    f: np.ndarray        # [N] routed fraction
    P: np.ndarray        # [N] mean router probability
    aux: float           # N * sum f_i P_i
    imbalance: float     # max_i n_i / (T k / N)
    drop_rate: float     # 1 - kept / (T k)


def router_probabilities(z: np.ndarray, gate: str) -> np.ndarray:
    """p_i(t): the full N-way softmax of z, or s_i / sum_l s_l for the sigmoid gate."""
    z64 = z.astype(np.float64)
    if gate in ("softmax", "softmax_full"):
        e = np.exp(z64 - z64.max(axis=1, keepdims=True))
        return e / e.sum(axis=1, keepdims=True)
    s = sigmoid_affinity(z).astype(np.float64)
    return s / s.sum(axis=1, keepdims=True)


def load_stats(z: np.ndarray, gate: str, d: Dispatch, k: int) -> LoadStats:
    """Switch balance quantities.  Chapter 19, 19.3.3 (f_i, P_i); CS336 lecture 4,
    section 9 (loss = N sum_i f_i P_i); Lecture29, "Myth 3" (imbalance I)."""
    T, N = z.shape
    f = d.counts_routed.astype(np.float64) / (T * k)
    P = router_probabilities(z, gate).mean(axis=0)
    aux = N * float(np.sum(f * P))
    imb = float(d.counts_routed.max()) / (T * k / N)
    drop = 1.0 - float(d.offsets[N]) / (T * k)
    return LoadStats(f, P, aux, imb, drop)


# --------------------------------------------------------------------------- expert-choice routing
@dataclasses.dataclass
class ExpertChoice:
    scores: np.ndarray      # [T, N] float64: full softmax over experts per token
    chosen: np.ndarray      # [N, C] int32: expert e's tokens, ascending token index
    dest_row: np.ndarray    # [T, N] int32: row e*C + r of token t in expert e, or -1
    offsets: np.ndarray     # [N+1] int32: e*C


def expert_choice(z: np.ndarray, C: int) -> ExpertChoice:
    """Each expert picks the C tokens with the largest scores.

    "Chapter 19: MoE", 19.6.1 (expert choice: every expert selects a fixed number
    of tokens; a token may be processed by any number of experts, zero included)
    and CS336 lecture 4, section 4 (top-K taken along the token axis of the score
    matrix, so each expert gets exactly the same number of tokens).  Scores are
    the full softmax over experts of each token's logits (CS336 lecture 4,
    section 5); ties go to the lower token index; C is capped at T.  An expert's
    rows are its tokens in ascending token order."""
    z64 = z.astype(np.float64)
    e_ = np.exp(z64 - z64.max(axis=1, keepdims=True))
    return expert_choice_select(e_ / e_.sum(axis=1, keepdims=True), C)


def expert_choice_select(sc: np.ndarray, C: int) -> ExpertChoice:
    """The selection step of expert_choice on given scores [T, N]."""
    T, N = sc.shape
    C = min(C, T)
    chosen = np.zeros((N, C), dtype=np.int32)
    dest = np.full((T, N), -1, dtype=np.int32)
    for e in range(N):
        order = sorted(range(T), key=lambda t: (-sc[t, e], t))[:C]
        toks = sorted(order)
        chosen[e] = toks
        for r, t in enumerate(toks):
            dest[t, e] = e * C + r
    offsets = (np.arange(N + 1) * C).astype(np.int32)
    return ExpertChoice(sc, chosen, dest, offsets)


def expert_choice_forward(inp, C: int) -> tuple:
    """y[t] = shared(x_t) + sum over experts e that chose t of s[t, e] * FFN_e(x_t).
    Returns (out [T, d] float64, the ExpertChoice routing).  Logits as in
    router_logits (with the optional logit bias); the gate is the score itself."""
    wl = inp.wl
    dt = wl.dtype
    x64 = widen(inp.x, dt)
    z = router_logits(x64, inp.Wg, inp.logit_bias)
    ec = expert_choice(z, C)
    out = np.zeros((wl.T, wl.d))
    if wl.shared_F:
        sw3 = widen(inp.sw3, dt) if inp.sw3 is not None else None
        out += expert_ffn(x64, widen(inp.sw1, dt), sw3, widen(inp.sw2, dt), wl.act)
    for e in range(wl.N):
        toks = ec.chosen[e]
        if toks.size == 0:
            continue
        W3 = widen(inp.w3[e], dt) if inp.w3 is not None else None
        y = expert_ffn(x64[toks], widen(inp.w1[e], dt), W3, widen(inp.w2[e], dt), wl.act)
        out[toks] += ec.scores[toks, e][:, None] * y
    return out, ec


# --------------------------------------------------------------------------- router training-side reductions
def router_z_loss(z: np.ndarray) -> float:
    """mean over tokens of (log Z)^2, Z = sum_i exp(z_i): the router z-loss.

    CS336 lecture 4, section 11 (the square of the softmax normaliser's log is
    added as a loss); Chapter 19, 19.6.2 (it penalises the log-sum-exp of the
    logits, not their L2 norm).  log Z is taken as m + log sum exp(z - m)."""
    z64 = z.astype(np.float64)
    m = z64.max(axis=1, keepdims=True)
    lse = m[:, 0] + np.log(np.exp(z64 - m).sum(axis=1))
    return float(np.mean(lse ** 2))


def sequence_balance_loss(z: np.ndarray, idx: np.ndarray, gate: str, seq_len: int) -> float:
    """DeepSeek-V3's sequence-wise balance loss: the Switch loss N sum_i f_i P_i
    computed within each sequence and averaged over the sequences.

    "Chapter 19: MoE", 19.3.4 (V3 keeps a small sequence-wise auxiliary balance
    loss against extreme imbalance inside one sequence); CS336 lecture 4,
    section 9 (it is the removed auxiliary loss with the unit of statistics
    changed from the batch to one sequence).  Tokens form consecutive sequences
    of seq_len (the last may be shorter); f_i counts the routed assignments of the
    sequence (before any capacity) over its L k; P_i is the mean router
    probability (as in load_stats) over the sequence's tokens."""
    T, N = z.shape
    k = idx.shape[1]
    p = router_probabilities(z, gate)
    losses = []
    for s0 in range(0, T, seq_len):
        s1 = min(T, s0 + seq_len)
        L = s1 - s0
        f = np.zeros(N)
        for t in range(s0, s1):
            for j in range(k):
                f[idx[t, j]] += 1.0
        f /= L * k
        P = p[s0:s1].mean(axis=0)
        losses.append(N * float(np.sum(f * P)))
    return float(np.mean(losses))


def bias_update(sel_bias: np.ndarray, counts_routed: np.ndarray, T: int, k: int, gamma: float) -> np.ndarray:
    """DeepSeek-V3 auxiliary-loss-free balancing, one step after a batch:
    b_i + gamma if expert i got fewer than the mean T k / N assignments,
    b_i - gamma if it got more, unchanged if exactly the mean (CS336 lecture 4,
    section 9; Chapter 19, 19.3.4).  Returned in float32."""
    N = len(counts_routed)
    out = sel_bias.astype(np.float64).copy()
    for i in range(N):
        if counts_routed[i] * N < T * k:
            out[i] += gamma
        elif counts_routed[i] * N > T * k:
            out[i] -= gamma
    return out.astype(np.float32)


# --------------------------------------------------------------------------- layer
@dataclasses.dataclass
class LayerResult:
    z: np.ndarray            # [T, N] float32 logits
    sel: np.ndarray          # [T, N] float32 selection scores
    idx: np.ndarray          # [T, k] int32
    w: np.ndarray            # [T, k] float64 gate weights
    disp: Dispatch
    out: np.ndarray          # [T, d] float64 (rows outside `tokens` are NaN)
    y_sh: Optional[np.ndarray]
    stats: LoadStats


def layer_forward(inp, tokens: Optional[np.ndarray] = None, cap: Optional[int] = None) -> LayerResult:
    """The whole layer: route every token, dispatch, run the experts and combine.

    `inp` carries the workload and its tensors (see the input module).
    `tokens`: compute the output only for these token rows (routing, dispatch and
    stats are always computed for all tokens, since capacity couples them).
    `cap`: a capacity in place of the workload's capacity factor."""
    wl = inp.wl
    dt = wl.dtype
    x64 = widen(inp.x, dt)
    z = router_logits(x64, inp.Wg, inp.logit_bias)
    sel, s = selection_scores(z, wl.gate, inp.sel_bias)
    idx = topk(sel, wl.k)
    w = gate_weights(z, s, idx, wl.gate)
    if cap is None:
        cap = capacity(wl.capacity_factor, wl.T, wl.k, wl.N) if wl.capacity_factor > 0 else 0
    disp = dispatch(idx, wl.N, cap)
    stats = load_stats(z, wl.gate, disp, wl.k)

    T = wl.T
    want = np.arange(T) if tokens is None else np.asarray(tokens)
    want_set = np.zeros(T, dtype=bool)
    want_set[want] = True
    out = np.full((T, wl.d), np.nan)
    out[want] = 0.0
    y_sh = None
    if wl.shared_F:
        # CS336 lecture 4, section 6: the shared expert runs for every token.
        sw3 = widen(inp.sw3, dt) if inp.sw3 is not None else None
        y_sh = np.full((T, wl.d), np.nan)
        y_sh[want] = expert_ffn(x64[want], widen(inp.sw1, dt), sw3, widen(inp.sw2, dt), wl.act)
        out[want] += y_sh[want]
    # expert outputs for the kept rows that feed a wanted token
    for e in range(wl.N):
        rows = np.arange(disp.offsets[e], disp.offsets[e + 1])
        rows = rows[want_set[disp.src_token[rows]]]
        if rows.size == 0:
            continue
        W1 = widen(inp.w1[e], dt)
        W3 = widen(inp.w3[e], dt) if inp.w3 is not None else None
        W2 = widen(inp.w2[e], dt)
        y = expert_ffn(x64[disp.src_token[rows]], W1, W3, W2, wl.act)
        # combine: y_out[t] += g_tj * Expert_e(x_t)  (Lecture29, "Top-two routing")
        for r, yr in zip(rows, y):
            t = disp.src_token[r]
            j = int(np.nonzero(idx[t] == e)[0][0])
            out[t] += w[t, j] * yr
    return LayerResult(z, sel, idx, w, disp, out, y_sh, stats)


# --------------------------------------------------------------------------- backward
@dataclasses.dataclass
class Params:
    """float64 parameters of one layer (shared expert optional)."""
    Wg: np.ndarray
    w1: np.ndarray
    w3: Optional[np.ndarray]
    w2: np.ndarray
    sw1: Optional[np.ndarray] = None
    sw3: Optional[np.ndarray] = None
    sw2: Optional[np.ndarray] = None


def params64(inp) -> Params:
    dt = inp.wl.dtype
    w = lambda a: None if a is None else widen(a, dt)  # noqa: E731
    return Params(inp.Wg.astype(np.float64), w(inp.w1), w(inp.w3), w(inp.w2), w(inp.sw1), w(inp.sw3), w(inp.sw2))


def _gates64(z64: np.ndarray, idx: np.ndarray, gate: str) -> np.ndarray:
    """Gate weights from float64 logits at fixed indices (no float32 rounding)."""
    T, k = idx.shape
    w = np.zeros((T, k))
    for t in range(T):
        if gate == "softmax":
            zs = z64[t, idx[t]]
            e = np.exp(zs - zs.max())
            w[t] = e / e.sum()
        elif gate == "softmax_full":
            e = np.exp(z64[t] - z64[t].max())
            w[t] = e[idx[t]] / e.sum()
        else:
            ss = 1.0 / (1.0 + np.exp(-z64[t, idx[t]]))
            w[t] = ss / ss.sum()
    return w


def forward_fixed_routing(x64, beta, P: Params, act: str, gate: str, idx: np.ndarray, disp: Dispatch) -> np.ndarray:
    """The layer in float64 with the top-k indices and the kept set held fixed
    (a smooth function of x and the parameters; used for gradient checks)."""
    z = x64 @ P.Wg + (0.0 if beta is None else beta.astype(np.float64)[None, :])
    w = _gates64(z, idx, gate)
    T, k = idx.shape
    out = np.zeros((T, P.w2.shape[1]))
    if P.sw1 is not None:
        out += expert_ffn(x64, P.sw1, P.sw3, P.sw2, act)
    for t in range(T):
        for j in range(k):
            if disp.dest_row[t, j] >= 0:
                e = idx[t, j]
                out[t] += w[t, j] * expert_ffn(x64[t:t + 1], P.w1[e], None if P.w3 is None else P.w3[e], P.w2[e], act)[0]
    return out


@dataclasses.dataclass
class Grads:
    dx: np.ndarray
    dWg: np.ndarray
    dw1: np.ndarray
    dw3: Optional[np.ndarray]
    dw2: np.ndarray
    dsw1: Optional[np.ndarray] = None
    dsw3: Optional[np.ndarray] = None
    dsw2: Optional[np.ndarray] = None
    dgate: Optional[np.ndarray] = None   # [T, k] dL/dw of the kept slots


def _expert_backward(xr, W1, W3, W2, dy, act):
    """Gradients of y = W2 act(W1 x [, W3 x]) for rows xr, given dy; float64."""
    a = xr @ W1.T
    if act == "swiglu":
        u = xr @ W3.T
        sig = 1.0 / (1.0 + np.exp(-a))
        h = a * sig * u
        dh = dy @ W2
        da = dh * u * (sig * (1.0 + a * (1.0 - sig)))   # d SiLU(a) / da = sig (1 + a (1 - sig))
        du = dh * a * sig
        dW2 = dy.T @ h
        dW1 = da.T @ xr
        dW3 = du.T @ xr
        dx = da @ W1 + du @ W3
        return dx, dW1, dW3, dW2
    h = np.maximum(a, 0.0)
    dh = dy @ W2
    da = dh * (a > 0)
    return da @ W1, da.T @ xr, None, dy.T @ h


def _dz_row(z_t: np.ndarray, idx_t: np.ndarray, w_t: np.ndarray, g: np.ndarray, gate: str) -> np.ndarray:
    """dL/dz of one token from the gradients g of its gate weights (0 on dropped slots)."""
    N = z_t.shape[0]
    dz = np.zeros(N)
    if gate == "softmax":
        dz[idx_t] = w_t * (g - np.sum(w_t * g))
    elif gate == "softmax_full":
        e_ = np.exp(z_t - z_t.max())
        p = e_ / e_.sum()
        gfull = np.zeros(N)
        gfull[idx_t] = g
        dz = p * (gfull - np.sum(p * gfull))
    else:
        s = 1.0 / (1.0 + np.exp(-z_t[idx_t]))
        ds = (g - np.sum(w_t * g)) / s.sum()
        dz[idx_t] = ds * s * (1.0 - s)
    return dz


def layer_backward(x64, beta, P: Params, act: str, gate: str, idx: np.ndarray, disp: Dispatch,
                   dout: np.ndarray) -> Grads:
    """Gradients of L = <dout, out> with the routing held fixed.

    The top-k choice is piecewise constant, so gradients reach the router only
    through the gate weights of the chosen, kept experts, and the experts only
    through the tokens they processed ("Chapter 19: MoE", 19.6.2: the main task's
    gradient flows through the selected gates and experts; unselected experts get
    none from that token).  Gate derivatives: softmax over the selected logits
    dz_j = w_j (dw_j - sum_l w_l dw_l); full softmax dz_i = p_i (g_i - sum_l p_l g_l)
    with g = dw on the selected, 0 elsewhere; sigmoid w_j = s_j / sum s gives
    ds_j = (dw_j - sum_l w_l dw_l) / sum s and dz_j = ds_j s_j (1 - s_j)."""
    T, k = idx.shape
    N = P.Wg.shape[1]
    z = x64 @ P.Wg + (0.0 if beta is None else beta.astype(np.float64)[None, :])
    w = _gates64(z, idx, gate)
    dx = np.zeros_like(x64)
    dw1 = np.zeros_like(P.w1)
    dw3 = None if P.w3 is None else np.zeros_like(P.w3)
    dw2 = np.zeros_like(P.w2)
    dgate = np.zeros((T, k))
    for e in range(N):
        rows = [(t, j) for t in range(T) for j in range(k) if idx[t, j] == e and disp.dest_row[t, j] >= 0]
        if not rows:
            continue
        toks = np.array([t for t, _ in rows])
        slots = np.array([j for _, j in rows])
        xr = x64[toks]
        W3 = None if P.w3 is None else P.w3[e]
        y = expert_ffn(xr, P.w1[e], W3, P.w2[e], act)
        dgate[toks, slots] = np.sum(dout[toks] * y, axis=1)
        dy = w[toks, slots][:, None] * dout[toks]
        gx, g1, g3, g2 = _expert_backward(xr, P.w1[e], W3, P.w2[e], dy, act)
        np.add.at(dx, toks, gx)
        dw1[e] += g1
        dw2[e] += g2
        if g3 is not None:
            dw3[e] += g3
    # through the gates into the logits
    dz = np.zeros((T, N))
    for t in range(T):
        dz[t] = _dz_row(z[t], idx[t], w[t], np.where(disp.dest_row[t] >= 0, dgate[t], 0.0), gate)
    dWg = x64.T @ dz
    dx += dz @ P.Wg.T
    gr = Grads(dx, dWg, dw1, dw3, dw2, dgate=dgate)
    if P.sw1 is not None:
        gx, gr.dsw1, gr.dsw3, gr.dsw2 = _expert_backward(x64, P.sw1, P.sw3, P.sw2, dout, act)
        gr.dx = gr.dx + gx
    return gr


def _logits64(inp, rows: np.ndarray) -> np.ndarray:
    x64 = widen(inp.x[rows], inp.wl.dtype)
    z = x64 @ inp.Wg.astype(np.float64)
    if inp.logit_bias is not None:
        z = z + inp.logit_bias.astype(np.float64)[None, :]
    return z


def backward_dx_tokens(inp, idx: np.ndarray, disp: Dispatch, dout: np.ndarray, tokens: np.ndarray) -> np.ndarray:
    """Rows `tokens` of layer_backward's dx, computed from those tokens alone (a
    token's dx involves only its own experts, gates and logits), with one expert's
    float64 weights in memory at a time: sampled gradient checks of full-size layers.
    dout: float64 [T, d]."""
    wl = inp.wl
    dt = wl.dtype
    tokens = np.asarray(tokens)
    x64 = widen(inp.x[tokens], dt)
    z = _logits64(inp, tokens)
    idx_s = idx[tokens]
    w = _gates64(z, idx_s, wl.gate)
    dx = np.zeros_like(x64)
    dgate = np.zeros(idx_s.shape)
    kept = disp.dest_row[tokens] >= 0
    for e in np.unique(idx_s):
        ii, jj = np.nonzero((idx_s == e) & kept)
        if ii.size == 0:
            continue
        W1, W2 = widen(inp.w1[e], dt), widen(inp.w2[e], dt)
        W3 = widen(inp.w3[e], dt) if inp.w3 is not None else None
        xr = x64[ii]
        y = expert_ffn(xr, W1, W3, W2, wl.act)
        dgate[ii, jj] = np.sum(dout[tokens[ii]] * y, axis=1)
        gx = _expert_backward(xr, W1, W3, W2, w[ii, jj][:, None] * dout[tokens[ii]], wl.act)[0]
        np.add.at(dx, ii, gx)
    Wg64 = inp.Wg.astype(np.float64)
    for i in range(tokens.size):
        dx[i] += _dz_row(z[i], idx_s[i], w[i], np.where(kept[i], dgate[i], 0.0), wl.gate) @ Wg64.T
    if wl.shared_F:
        sw3 = widen(inp.sw3, dt) if inp.sw3 is not None else None
        dx += _expert_backward(x64, widen(inp.sw1, dt), sw3, widen(inp.sw2, dt), dout[tokens], wl.act)[0]
    return dx


def backward_dw_entries(inp, idx: np.ndarray, disp: Dispatch, dout: np.ndarray, which: str,
                        entries) -> np.ndarray:
    """Entries (e, i, j) of layer_backward's dw1 / dw3 ([N, F, d]: i = hidden unit f,
    j = input column) or dw2 ([N, d, F]: i = output column, j = f), each summed over
    the kept rows of expert e from the columns it needs: sampled gradient checks of
    full-size layers.  dout: float64 [T, d]."""
    wl = inp.wl
    dt = wl.dtype
    out = np.zeros(len(entries))
    for n, (e, i, j) in enumerate(entries):
        toks, slots = np.nonzero((idx == e) & (disp.dest_row >= 0))   # row-major: token order
        if toks.size == 0:
            continue
        xr = widen(inp.x[toks], dt)
        w = _gates64(_logits64(inp, toks), idx[toks], wl.gate)[np.arange(toks.size), slots]
        dy = w[:, None] * dout[toks]
        f = i if which in ("w1", "w3") else j
        a = xr @ widen(inp.w1[e][f], dt)
        dh = dy @ widen(inp.w2[e][:, f], dt)
        if wl.act == "swiglu":
            u = xr @ widen(inp.w3[e][f], dt)
            sig = 1.0 / (1.0 + np.exp(-a))
            h = a * sig * u
            da = dh * u * (sig * (1.0 + a * (1.0 - sig)))
            du = dh * a * sig
        else:
            h = np.maximum(a, 0.0)
            da = dh * (a > 0)
            du = None
        if which == "w2":
            out[n] = np.sum(dy[:, i] * h)
        elif which == "w1":
            out[n] = np.sum(da * xr[:, j])
        else:
            out[n] = np.sum(du * xr[:, j])
    return out


# --------------------------------------------------------------------------- FP8 expert weights
# Quantisation of the experts is an open question on the pages ("Stanford CS336
# lecture 4", the section on compressing sparse MoEs: quantisation lowers the
# bits per weight at the cost of scales and a dequantisation step; the Q&A finds a
# heavily quantised Mixtral 8x7B practical on one GPU).  The plainest reading is
# taken: weight-only FP8 E4M3 with one float32 scale per output row (channel),
# activations and accumulation unchanged.

E4M3_MAX = 448.0


def _e4m3_value_def(code: np.ndarray) -> np.ndarray:
    """Value of FP8 E4M3 codes (OCP 8-bit floating point: sign, 4 exponent bits with
    bias 7, 3 mantissa bits; exponent 0 is subnormal, m/8 * 2^-6; no infinities;
    S.1111.111 is NaN, so the largest finite value is 1.75 * 2^8 = 448)."""
    c = np.asarray(code, dtype=np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 15
    m = c & 7
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * 2.0 ** (e - 7.0))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return sign * mag


_E4M3_TABLE = _e4m3_value_def(np.arange(256))


def e4m3_value(code: np.ndarray) -> np.ndarray:
    """Value of FP8 E4M3 codes (the definition above, tabulated for all 256 codes)."""
    return _E4M3_TABLE[np.asarray(code, dtype=np.int64)]


def e4m3_round(v: np.ndarray) -> np.ndarray:
    """float32 values -> E4M3 codes: round to the nearest representable value, ties to
    even (rint), magnitudes above 448 saturated to 448; -0 keeps its sign.  The
    grid: in the binade [2^e, 2^(e+1)) with e >= -6 the values are 2^e (1 + m/8),
    spaced 2^(e-3); below 2^-6 (subnormal) they are spaced 2^-9.  The rounding
    decision is taken on the float32 value."""
    v32 = np.asarray(v, dtype=np.float32)
    a = np.abs(v32.astype(np.float64))
    _, ex = np.frexp(a)                                  # a = f 2^ex with f in [0.5, 1): binade 2^(ex - 1)
    quantum = np.ldexp(1.0, np.maximum(ex - 1, -6) - 3)  # 2^(e - 3), e = max(binade exponent, -6)
    r = np.minimum(np.rint(a / quantum) * quantum, 448.0)  # exact: division by a power of two
    # encode the rounded value (a carry into the next binade is already in r)
    _, er = np.frexp(r)
    eb = np.maximum(er - 1, -6)                          # binade exponent of r (subnormals: -6)
    normal = r >= 2.0 ** -6
    mant = np.where(normal, r / np.ldexp(1.0, eb - 3) - 8.0, r / 2.0 ** -9)
    code = np.where(normal, ((eb + 7) << 3) + mant.astype(np.int64), mant.astype(np.int64))
    return (code | np.where(np.signbit(v32), 0x80, 0)).astype(np.uint8)


def quantize_fp8_rows(w: np.ndarray):
    """One scale per row: s = fl32(max |w| / 448) (1 for an all-zero row), codes =
    E4M3 rounding of fl32(w / s).  w: [..., C] float32 (bf16 values widened).
    Returns (codes uint8 [..., C], scales float32 [...])."""
    w32 = np.asarray(w, dtype=np.float32)
    amax = np.max(np.abs(w32), axis=-1)
    s = np.where(amax > 0, (amax / np.float32(E4M3_MAX)).astype(np.float32), np.float32(1.0)).astype(np.float32)
    # rows are independent: large matrices are rounded in row blocks on all cores
    flat_w, flat_s = w32.reshape(-1, w32.shape[-1]), s.reshape(-1)
    q = np.empty(flat_w.shape, dtype=np.uint8)

    def block(r0):
        r1 = min(r0 + 256, flat_w.shape[0])
        q[r0:r1] = e4m3_round((flat_w[r0:r1] / flat_s[r0:r1, None]).astype(np.float32))
    starts = range(0, flat_w.shape[0], 256)
    if flat_w.size > (1 << 22):
        with concurrent.futures.ThreadPoolExecutor(max_workers=os.cpu_count() or 1) as pool:
            list(pool.map(block, starts))
    else:
        for r0 in starts:
            block(r0)
    return q.reshape(w32.shape), s


def dequantize_fp8_rows(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    """float64 weights q * s (exact: 4 significant bits times a float32)."""
    return e4m3_value(q) * np.asarray(s, dtype=np.float64)[..., None]


def layer_forward_fp8(inp, q1, s1, q3, s3, q2, s2, tokens: Optional[np.ndarray] = None) -> LayerResult:
    """The layer of layer_forward with the expert weights replaced by their FP8
    dequantisation (the router, the shared expert and the activations unchanged);
    outputs for `tokens` (default: all)."""
    wl = inp.wl
    dt = wl.dtype
    ref = layer_forward(inp, tokens=np.array([], dtype=np.int64))
    x64 = widen(inp.x, dt)
    rows = np.arange(wl.T) if tokens is None else np.asarray(tokens)
    out = np.full((wl.T, wl.d), np.nan)
    out[rows] = 0.0
    if wl.shared_F:
        sw3 = widen(inp.sw3, dt) if inp.sw3 is not None else None
        out[rows] += expert_ffn(x64[rows], widen(inp.sw1, dt), sw3, widen(inp.sw2, dt), wl.act)
    want = np.zeros(wl.T, dtype=bool)
    want[rows] = True
    for e in range(wl.N):
        tt, jj = np.nonzero((ref.idx == e) & (ref.disp.dest_row >= 0) & want[:, None])
        if tt.size == 0:
            continue
        W3 = dequantize_fp8_rows(q3[e], s3[e]) if q3 is not None else None
        y = expert_ffn(x64[tt], dequantize_fp8_rows(q1[e], s1[e]), W3, dequantize_fp8_rows(q2[e], s2[e]), wl.act)
        np.add.at(out, tt, ref.w[tt, jj][:, None] * y)
    return dataclasses.replace(ref, out=out)


def dense_mask_forward(inp, cap: Optional[int] = None) -> np.ndarray:
    """Second formulation, with no permutation: y[t] = y_sh[t] + sum_e G[t,e] FFN_e(x_t).

    G[t,e] is the gate weight if expert e was selected for token t and that
    assignment survived the capacity limit (counted in token order), else 0;
    every expert runs on every token.  Lecture29, "Top-two routing"
    (y = sum_{i=1..E} g_i(x) Expert_i(x), with g_i = 0 outside S_k)."""
    wl = inp.wl
    dt = wl.dtype
    x64 = widen(inp.x, dt)
    z = router_logits(x64, inp.Wg, inp.logit_bias)
    sel, s = selection_scores(z, wl.gate, inp.sel_bias)
    idx = topk(sel, wl.k)
    w = gate_weights(z, s, idx, wl.gate)
    if cap is None:
        cap = capacity(wl.capacity_factor, wl.T, wl.k, wl.N) if wl.capacity_factor > 0 else 0
    limit = cap if cap > 0 else wl.T * wl.k
    G = np.zeros((wl.T, wl.N))
    used = np.zeros(wl.N, dtype=np.int64)
    for t in range(wl.T):
        for j in range(wl.k):
            e = idx[t, j]
            if used[e] < limit:
                G[t, e] = w[t, j]
            used[e] += 1
    y = np.zeros((wl.T, wl.d))
    if wl.shared_F:
        sw3 = widen(inp.sw3, dt) if inp.sw3 is not None else None
        y += expert_ffn(x64, widen(inp.sw1, dt), sw3, widen(inp.sw2, dt), wl.act)
    for e in range(wl.N):
        W3 = widen(inp.w3[e], dt) if inp.w3 is not None else None
        y += G[:, e:e + 1] * expert_ffn(x64, widen(inp.w1[e], dt), W3, widen(inp.w2[e], dt), wl.act)
    return y
