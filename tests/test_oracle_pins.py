"""Pins of the CPU oracle against what the pages and the mathematics fix (no GPU).

Each test pins one part of the oracle to something other than the oracle
itself: an identity stated on the pages, a closed form, brute force on tiny
inputs, or an invariant.  They are chosen so that a dropped term, a wrong sign,
a wrong index or a transposed operand in the oracle fails at least one.
"""
import dataclasses
import itertools
import json
import math
import os

import numpy as np
import pytest
import scipy.special

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def tiny(T=24, d=16, N=6, k=2, F=32, act="swiglu", gate="softmax", dtype="bf16", shared_F=0,
         capacity_factor=0.0, sel_bias_range=0.0, zipf_s=0.0, seed=7):
    wl = synth.Workload("tiny", seed, T=T, d=d, N=N, k=k, F=F, act=act, gate=gate, dtype=dtype,
                        shared_F=shared_F, capacity_factor=capacity_factor,
                        sel_bias_range=sel_bias_range, zipf_s=zipf_s)
    return synth.make_inputs(wl)


# --------------------------------------------------------------------------- gate
@pytest.mark.parametrize("N,k", [(8, 2), (64, 6), (256, 8), (5, 5)])
def test_softmax_gate_equals_renormalised_full_softmax(N, k):
    """Chapter 19, 19.3.2: softmax over the selected logits equals the full
    softmax taken over all logits and renormalised over the top-k."""
    rng = np.random.default_rng(N * 100 + k)
    z = (rng.standard_normal((200, N)) * 3).astype(np.float32)
    idx = oracle.topk(z, k)
    w = oracle.gate_weights(z, None, idx, "softmax")
    p = scipy.special.softmax(z.astype(np.float64), axis=1)
    ps = np.take_along_axis(p, idx.astype(np.int64), axis=1)
    ref = ps / ps.sum(axis=1, keepdims=True)
    assert np.max(np.abs(w - ref)) < 1e-12
    # the selected ones are the k largest probabilities
    assert np.all(ps.min(axis=1) >= np.sort(p, axis=1)[:, -k] - 1e-15)


def test_softmax_gate_two_expert_closed_form():
    """Two selected logits a > b: g = (1/(1+e^{b-a}), 1/(1+e^{a-b}))."""
    z = np.array([[0.25, 2.0, -1.0, 1.5]], dtype=np.float32)
    idx = oracle.topk(z, 2)
    assert idx.tolist() == [[1, 3]]
    w = oracle.gate_weights(z, None, idx, "softmax")
    a, b = 2.0, 1.5
    assert abs(w[0, 0] - 1.0 / (1.0 + math.exp(b - a))) < 1e-15
    assert abs(w[0, 1] - 1.0 / (1.0 + math.exp(a - b))) < 1e-15


def _brute_force_topk(sel_row, k):
    """The unique k-subset in which every chosen score beats every unchosen one,
    equal scores going to the lower index; listed by (score desc, index asc)."""
    N = len(sel_row)
    found = []
    for S in itertools.combinations(range(N), k):
        rest = [u for u in range(N) if u not in S]
        if all(sel_row[i] > sel_row[u] or (sel_row[i] == sel_row[u] and i < u) for i in S for u in rest):
            found.append(S)
    assert len(found) == 1
    S = found[0]
    return sorted(S, key=lambda i: (-float(sel_row[i]), i))


@pytest.mark.parametrize("N", [1, 2, 3, 5, 8])
def test_topk_matches_brute_force_with_ties(N):
    rng = np.random.default_rng(N)
    # scores from a 3-value alphabet force many exact ties
    sel = rng.choice(np.array([-1.0, 0.5, 2.0], dtype=np.float32), size=(60, N))
    for k in range(1, N + 1):
        idx = oracle.topk(sel, k)
        for t in range(sel.shape[0]):
            assert idx[t].tolist() == _brute_force_topk(sel[t], k)


def test_topk_distinct_scores_brute_force():
    rng = np.random.default_rng(3)
    sel = rng.standard_normal((100, 7)).astype(np.float32)
    for k in (1, 2, 4, 7):
        idx = oracle.topk(sel, k)
        for t in range(100):
            assert idx[t].tolist() == _brute_force_topk(sel[t], k)


# --------------------------------------------------------------------------- sigmoid gate
def test_sigmoid_gate_properties():
    """Chapter 19, 19.3.4 / CS336 lecture 4, section 9: the bias only steers the
    choice; the mixing weights come from the raw affinities and sum to 1."""
    inp = tiny(gate="sigmoid", N=8, k=3, sel_bias_range=0.05)
    r = oracle.layer_forward(inp)
    assert np.allclose(r.w.sum(axis=1), 1.0, atol=1e-14)
    z64 = r.z.astype(np.float64)
    s_ref = 1.0 / (1.0 + np.exp(-z64))                 # raw affinities
    sel_ref = s_ref.astype(np.float32).astype(np.float64) + inp.sel_bias.astype(np.float64)
    # selected set = top-k of s + b
    for t in range(inp.wl.T):
        chosen = set(r.idx[t].tolist())
        order = sorted(range(8), key=lambda i: (-sel_ref[t, i], i))
        assert chosen == set(order[:3])
        ss = s_ref[t, r.idx[t]]
        assert np.allclose(r.w[t], ss / ss.sum(), rtol=1e-6)


def test_sigmoid_without_bias_selects_topk_of_logits():
    """sigma is monotone, so with b = 0 the selection is the top-k of z."""
    inp = tiny(gate="sigmoid", N=16, k=4)
    r = oracle.layer_forward(inp)
    idx_z = oracle.topk(r.z, 4)
    # compare where the logit gap is clear of float32 sigmoid rounding
    zs = np.sort(r.z, axis=1)[:, ::-1]
    clear = (zs[:, 3] - zs[:, 4]) > 1e-4
    assert np.array_equal(np.sort(r.idx[clear], 1), np.sort(idx_z[clear], 1))


def test_sigmoid_bias_flips_selection_but_not_weights():
    """A large bias on one expert forces it into every token's top-k, yet its
    gate weight is its raw affinity's share, not the biased one."""
    inp = tiny(gate="sigmoid", N=8, k=2)
    inp.sel_bias = np.zeros(8, dtype=np.float32)
    inp.sel_bias[5] = 10.0
    r = oracle.layer_forward(inp)
    assert np.all(r.idx[:, 0] == 5)
    s = 1.0 / (1.0 + np.exp(-r.z.astype(np.float64)))
    for t in range(inp.wl.T):
        ss = s[t, r.idx[t]]
        assert np.allclose(r.w[t], ss / ss.sum(), rtol=1e-6)
        assert r.w[t, 0] < 0.99   # an unbiased share, nowhere near 1


# --------------------------------------------------------------------------- experts
def test_swiglu_and_relu_closed_form():
    """d = F = 1: the expert is a scalar function.  Lecture29 (SwiGLU
    W2(SiLU(W1 x) * W3 x)) and the Shazeer notes (one ReLU hidden layer)."""
    x = np.array([[1.5]])
    W1, W3, W2 = np.array([[0.8]]), np.array([[-2.0]]), np.array([[3.0]])
    a = 0.8 * 1.5
    expect = 3.0 * (a / (1.0 + math.exp(-a))) * (-2.0 * 1.5)
    assert abs(oracle.expert_ffn(x, W1, W3, W2, "swiglu")[0, 0] - expect) < 1e-14
    assert oracle.expert_ffn(x, W1, None, W2, "relu")[0, 0] == pytest.approx(3.0 * 1.2, abs=1e-15)
    assert oracle.expert_ffn(-x, W1, None, W2, "relu")[0, 0] == 0.0
    # SiLU(1) = 1 / (1 + e^-1)
    assert abs(oracle.silu(np.array(1.0)) - 0.7310585786300049) < 1e-15


def _loop_ffn(xr, W1, W3, W2, act):
    """Dense FFN written with scalar loops (independent of the oracle's matmuls)."""
    F, d = W1.shape
    y = np.zeros(W2.shape[0])
    for f in range(F):
        a = sum(W1[f, i] * xr[i] for i in range(d))
        if act == "swiglu":
            u = sum(W3[f, i] * xr[i] for i in range(d))
            h = a / (1.0 + math.exp(-a)) * u
        else:
            h = max(a, 0.0)
        for o in range(W2.shape[0]):
            y[o] += W2[o, f] * h
    return y


@pytest.mark.parametrize("act", ["swiglu", "relu"])
def test_k_equals_N_identical_experts_is_dense_ffn(act):
    """Lecture29, "Top-two routing": y = sum_i g_i Expert_i(x) with the g_i
    summing to 1, so k = N identical experts give the dense FFN."""
    inp = tiny(T=6, d=8, N=4, k=4, F=12, act=act)
    for e in range(1, 4):
        inp.w1[e] = inp.w1[0]
        inp.w2[e] = inp.w2[0]
        if inp.w3 is not None:
            inp.w3[e] = inp.w3[0]
    r = oracle.layer_forward(inp)
    W1 = oracle.widen(inp.w1[0], "bf16")
    W3 = oracle.widen(inp.w3[0], "bf16") if inp.w3 is not None else None
    W2 = oracle.widen(inp.w2[0], "bf16")
    x = oracle.widen(inp.x, "bf16")
    for t in range(6):
        ref = _loop_ffn(x[t], W1, W3, W2, act)
        assert np.allclose(r.out[t], ref, rtol=1e-12, atol=1e-12)


def test_zero_input_gives_zero_output():
    inp = tiny(shared_F=16)
    inp.x[:] = 0
    r = oracle.layer_forward(inp)
    assert np.all(r.out == 0.0)


# --------------------------------------------------------------------------- dispatch / capacity
def test_capacity_formula_values():
    """Lecture29, "Inference load balance": C = ceil(alpha T k / E)."""
    with open(os.path.join(GOLDEN, "page_values.json")) as f:
        g = json.load(f)
    c = g["qwen3_skew_capacity"]
    assert oracle.capacity(c["alpha"], c["T"], c["k"], c["N"]) == c["C"]
    assert oracle.capacity(1.0, 10, 2, 3) == 7           # ceil(20/3)
    assert oracle.capacity(1.0, 9, 2, 3) == 6            # exact, no round-up
    assert oracle.capacity(0.5, 3, 1, 2) == 1            # ceil(0.75)
    for (T, k, N) in [(16, 2, 8), (100, 3, 7), (4096, 2, 8), (16384, 8, 128)]:
        # alpha >= N/k gives C >= T: no expert can overflow
        assert oracle.capacity(N / k, T, k, N) >= T


def _routing(T, N, k, rng, skew=0.0):
    scores = rng.standard_normal((T, N)) + skew * np.linspace(2, -2, N)[None, :]
    return oracle.topk(scores.astype(np.float32), k)


@pytest.mark.parametrize("T,N,k,cap", [(50, 8, 2, 0), (200, 16, 4, 13), (333, 5, 5, 40), (64, 3, 1, 1),
                                       (1, 4, 2, 0), (0, 4, 2, 0), (100, 8, 2, 1000)])
def test_dispatch_invariants(T, N, k, cap):
    """Chapter 19, 19.6.1: T k assignments in all; per expert at most C kept,
    the first C in token order, the rest dropped (their branch contributes 0)."""
    rng = np.random.default_rng(T + N + k)
    idx = _routing(T, N, k, rng, skew=1.5).reshape(T, k)
    d = oracle.dispatch(idx, N, cap)
    assert int(d.counts_routed.sum()) == T * k
    limit = cap if cap > 0 else T * k
    assert np.array_equal(d.counts_kept, np.minimum(d.counts_routed, limit))
    assert d.offsets[0] == 0 and np.array_equal(np.diff(d.offsets), d.counts_kept)
    for e in range(N):
        toks = [t for t in range(T) if e in idx[t].tolist()]        # token order
        assert len(toks) == d.counts_routed[e]
        kept = toks[:limit]
        rows = list(range(d.offsets[e], d.offsets[e + 1]))
        assert d.src_token[rows].tolist() == kept
        for t in toks[limit:]:
            j = idx[t].tolist().index(e)
            assert d.dest_row[t, j] == -1
    # dest_row and src_token are inverse maps on kept assignments
    for t in range(T):
        for j in range(k):
            r = d.dest_row[t, j]
            if r >= 0:
                assert d.src_token[r] == t
                assert d.offsets[idx[t, j]] <= r < d.offsets[idx[t, j] + 1]


def test_no_drops_when_alpha_at_least_N_over_k():
    rng = np.random.default_rng(11)
    T, N, k = 300, 8, 2
    idx = _routing(T, N, k, rng, skew=4.0)
    cap = oracle.capacity(N / k, T, k, N)
    d = oracle.dispatch(idx, N, cap)
    assert np.all(d.dest_row >= 0)


# --------------------------------------------------------------------------- whole layer
CASES = [
    dict(),
    dict(act="relu", dtype="f32", N=8, k=2),
    dict(gate="sigmoid", N=12, k=4, shared_F=24, sel_bias_range=0.05),
    dict(N=8, k=3, capacity_factor=0.6, zipf_s=1.2, T=40),
    dict(N=1, k=1),
    dict(N=5, k=5, T=9),
]


@pytest.mark.parametrize("kw", CASES)
def test_dense_mask_formulation_agrees(kw):
    """The permuted layer (dispatch, expert groups, combine) equals the dense
    per-token sum y = sum_e G[t,e] FFN_e(x_t) with G zero off the kept top-k."""
    inp = tiny(**kw)
    r = oracle.layer_forward(inp)
    y = oracle.dense_mask_forward(inp)
    scale = max(1.0, np.max(np.abs(y)))
    assert np.max(np.abs(r.out - y)) <= 1e-12 * scale


def test_dense_mask_on_the_tiny_fp32_workload():
    inp = synth.make_inputs(synth.WORKLOADS["shazeer_tiny_f32"])
    r = oracle.layer_forward(inp)
    y = oracle.dense_mask_forward(inp)
    assert np.max(np.abs(r.out - y)) <= 1e-12 * np.max(np.abs(y))


def test_capacity_drop_contributes_zero():
    """CS336 lecture 4, section 10: a dropped assignment's expert output is 0.
    With C = 1, a token whose both experts were already taken gets 0."""
    inp = tiny(T=30, N=4, k=2, capacity_factor=0.01)
    r = oracle.layer_forward(inp)
    assert oracle.capacity(0.01, 30, 2, 4) == 1
    for t in range(30):
        if np.all(r.disp.dest_row[t] < 0):
            assert np.all(r.out[t] == 0.0)
    assert r.disp.offsets[-1] == np.count_nonzero(r.disp.counts_routed)


def test_expert_permutation_symmetry():
    """Lecture29, "Myth 1": permuting the experts together with the router's
    output channels leaves the layer's function unchanged."""
    inp = tiny(N=7, k=3, T=30, shared_F=8)
    r = oracle.layer_forward(inp)
    perm = np.array([3, 0, 6, 1, 5, 2, 4])
    inp2 = synth.LayerInputs(inp.wl, inp.x, inp.Wg[:, perm], inp.w1[perm], inp.w3[perm], inp.w2[perm],
                             inp.sw1, inp.sw3, inp.sw2)
    r2 = oracle.layer_forward(inp2)
    assert np.max(np.abs(r.out - r2.out)) <= 1e-12 * np.max(np.abs(r.out))
    # and the routing maps through the permutation
    assert np.array_equal(perm[r2.idx], r.idx)


def test_logit_bias_shift_invariance():
    """Adding a constant to every logit changes neither top-k nor the softmax gate
    (the Zipf skew's normalisation constant is irrelevant)."""
    inp = tiny(N=16, k=4, zipf_s=1.2, T=64)
    r = oracle.layer_forward(inp)
    inp.logit_bias = (inp.logit_bias.astype(np.float64) + 3.0).astype(np.float32)
    r2 = oracle.layer_forward(inp)
    zs = np.sort(r.z, axis=1)[:, ::-1]
    clear = (zs[:, 3] - zs[:, 4]) > 1e-4
    assert np.array_equal(r.idx[clear], r2.idx[clear])
    assert np.max(np.abs(r.w[clear] - r2.w[clear])) < 1e-5


# --------------------------------------------------------------------------- stats
def test_uniform_load_gives_aux_one():
    """CS336 lecture 4, section 9: with uniform routing and uniform router
    probabilities the loss N sum f_i P_i equals 1; imbalance is 1."""
    T, N, k = 64, 8, 1
    z = np.zeros((T, N), dtype=np.float32)
    idx = (np.arange(T) % N).reshape(T, 1).astype(np.int32)
    d = oracle.dispatch(idx, N, 0)
    st = oracle.load_stats(z, "softmax", d, k)
    assert st.aux == pytest.approx(1.0, abs=1e-14)
    assert st.imbalance == pytest.approx(1.0)
    assert st.drop_rate == 0.0
    assert np.allclose(st.f, 1.0 / N) and np.allclose(st.P, 1.0 / N)


def test_stats_sum_to_one_and_imbalance():
    inp = tiny(N=8, k=2, T=200, zipf_s=1.2, capacity_factor=1.0)
    r = oracle.layer_forward(inp)
    st = r.stats
    assert st.f.sum() == pytest.approx(1.0, abs=1e-14)
    assert st.P.sum() == pytest.approx(1.0, abs=1e-12)
    n = r.disp.counts_routed
    assert st.imbalance == pytest.approx(n.max() / (200 * 2 / 8))
    assert st.drop_rate == pytest.approx(1 - r.disp.counts_kept.sum() / 400)
    # all mass on one expert: f = e_0, aux = N * P_0
    z = np.zeros((10, 4), dtype=np.float32)
    z[:, 0] = 50.0
    d = oracle.dispatch(np.zeros((10, 1), dtype=np.int32), 4, 0)
    st = oracle.load_stats(z, "softmax", d, 1)
    assert st.aux == pytest.approx(4.0, rel=1e-12)
    assert st.imbalance == pytest.approx(4.0)


# --------------------------------------------------------------------------- workload shapes
def test_workload_shapes_match_published_model_sizes():
    """The expert shapes reproduce the pages' parameter counts."""
    with open(os.path.join(GOLDEN, "page_values.json")) as f:
        g = json.load(f)
    W = synth.WORKLOADS
    c1 = W["shazeer_tiny_f32"]
    assert c1.d * c1.F + c1.F * c1.d == g["shazeer_expert_weights"]["value"]
    for key, wname in [("mixtral", "mixtral_prefill"), ("dsv3", "dsv3_finegrained"), ("qwen3", "qwen3_skew_drop")]:
        m = g["moe_layers_from_totals"][key]
        wl = W[wname]
        P_e = 3 * wl.d * wl.F
        layers = (m["total"] - m["active"]) / ((wl.N - wl.k) * P_e)
        assert abs(layers - m["layers"]) < 0.1, (key, layers)


def test_logit_bias_closed_form_zipf_probabilities():
    """With W_g = 0 the logits are the skew beta_i = log p_i, so the full softmax
    P_i equals the Zipf popularity p_i exactly and top-k picks the k most
    popular experts (CS336 lecture 4, section 9: P_i is the router's share)."""
    inp = tiny(N=16, k=4, T=20, zipf_s=1.2)
    inp.Wg[:] = 0.0
    r = oracle.layer_forward(inp)
    p = np.array([rk ** -1.2 for rk in range(1, 17)])
    p /= p.sum()
    beta = inp.logit_bias.astype(np.float64)
    assert np.allclose(np.sort(np.exp(beta))[::-1], p, rtol=1e-6)
    assert np.allclose(r.stats.P, np.exp(beta) / np.exp(beta).sum(), rtol=1e-6)
    assert np.allclose(np.sort(r.stats.P)[::-1], p, rtol=1e-6)
    top = sorted(range(16), key=lambda i: -beta[i])[:4]
    assert np.all(r.idx == np.array(top)[None, :])


def test_combine_hand_computed():
    """A 2-token example worked by hand: token 0 keeps both slots, token 1's
    second slot was dropped (-1) and adds nothing."""
    y_rows = np.array([[1.0, 2.0], [10.0, 20.0], [100.0, 200.0]])
    dest = np.array([[2, 0], [1, -1]])
    w = np.array([[0.75, 0.25], [0.5, 0.5]])
    out = oracle.combine(y_rows, dest, w, None)
    assert out.tolist() == [[75.25, 150.5], [5.0, 10.0]]
    out = oracle.combine(y_rows, dest, w, np.array([[1.0, 1.0], [2.0, 2.0]]))
    assert out.tolist() == [[76.25, 151.5], [7.0, 12.0]]


# --------------------------------------------------------------------------- gate variants, router reductions
def test_softmax_full_gate_is_unrenormalised_full_softmax():
    """CS336 lecture 4, section 5: g_i = softmax(z)_i on the top-k, 0 elsewhere;
    renormalising it over the top-k gives the top-k softmax gate (Chapter 19,
    19.3.2), and with k = N it sums to 1."""
    rng = np.random.default_rng(5)
    z = (rng.standard_normal((100, 16)) * 2).astype(np.float32)
    idx = oracle.topk(z, 4)
    w_full = oracle.gate_weights(z, None, idx, "softmax_full")
    p = scipy.special.softmax(z.astype(np.float64), axis=1)
    assert np.max(np.abs(w_full - np.take_along_axis(p, idx.astype(np.int64), axis=1))) < 1e-14
    assert np.all(w_full.sum(axis=1) < 1.0)
    w_top = oracle.gate_weights(z, None, idx, "softmax")
    assert np.max(np.abs(w_full / w_full.sum(axis=1, keepdims=True) - w_top)) < 1e-12
    idx_all = oracle.topk(z, 16)
    assert np.allclose(oracle.gate_weights(z, None, idx_all, "softmax_full").sum(axis=1), 1.0, atol=1e-14)


def test_router_z_loss_closed_forms():
    """All logits equal to c: log Z = c + log N exactly, so the loss is (c + log N)^2;
    one dominant logit L: log Z -> L."""
    for c, N in [(0.0, 8), (1.5, 4), (-2.0, 256)]:
        z = np.full((7, N), c, dtype=np.float32)
        assert oracle.router_z_loss(z) == pytest.approx((c + math.log(N)) ** 2, rel=1e-12)
    z = np.array([[30.0, 0.0, 0.0]], dtype=np.float32)
    assert oracle.router_z_loss(z) == pytest.approx((30.0 + math.log1p(2 * math.exp(-30.0))) ** 2, rel=1e-14)
    # shift invariance fails on purpose: the loss penalises the scale of the logits
    z2 = np.random.default_rng(1).standard_normal((50, 8)).astype(np.float32)
    assert oracle.router_z_loss(z2 + 3) > oracle.router_z_loss(z2)


def test_bias_update_signs():
    """+gamma below the mean load, -gamma above it, unchanged at exactly the mean."""
    counts = np.array([0, 5, 10, 25], dtype=np.int64)   # T k / N = 40 / 4 = 10
    b = np.array([0.5, -0.1, 0.0, 0.2], dtype=np.float32)
    out = oracle.bias_update(b, counts, T=20, k=2, gamma=0.01)
    assert out.tolist() == pytest.approx([0.51, -0.09, 0.0, 0.19], abs=1e-7)


# --------------------------------------------------------------------------- expert choice
@pytest.mark.parametrize("T,N,C", [(9, 3, 4), (6, 4, 6), (5, 2, 9), (12, 5, 1)])
def test_expert_choice_brute_force_and_equal_loads(T, N, C):
    """Every expert gets exactly min(C, T) tokens (CS336 lecture 4, section 4);
    its set is the one where every chosen score beats every unchosen one, ties to
    the lower token index (brute force over all subsets)."""
    rng = np.random.default_rng(T * N)
    z = rng.choice(np.array([-1.0, 0.0, 0.5, 2.0], dtype=np.float32), size=(T, N))   # many ties
    ec = oracle.expert_choice(z, C)
    Ce = min(C, T)
    assert ec.chosen.shape == (N, Ce)
    for e in range(N):
        col = ec.scores[:, e]
        best = _brute_force_topk(col, Ce)
        assert sorted(best) == ec.chosen[e].tolist()
        for r, t in enumerate(ec.chosen[e]):
            assert ec.dest_row[t, e] == e * Ce + r
    assert np.sum(ec.dest_row >= 0) == N * Ce
    assert np.allclose(ec.scores.sum(axis=1), 1.0)


def test_expert_choice_all_tokens_is_dense_softmax_mixture():
    """C = T: every expert processes every token, so y = sum_e softmax(z)_e FFN_e(x);
    with identical experts that is the dense FFN (the softmax weights sum to 1)."""
    inp = tiny(T=5, d=8, N=3, k=1, F=12)
    for e in range(1, 3):
        inp.w1[e], inp.w3[e], inp.w2[e] = inp.w1[0], inp.w3[0], inp.w2[0]
    out, ec = oracle.expert_choice_forward(inp, C=5)
    x = oracle.widen(inp.x, "bf16")
    W1, W3, W2 = (oracle.widen(a[0], "bf16") for a in (inp.w1, inp.w3, inp.w2))
    for t in range(5):
        assert np.allclose(out[t], _loop_ffn(x[t], W1, W3, W2, "swiglu"), rtol=1e-12, atol=1e-12)


def test_expert_choice_unchosen_token_gets_zero():
    inp = tiny(T=20, d=8, N=2, k=1, F=12)
    out, ec = oracle.expert_choice_forward(inp, C=3)
    unchosen = np.all(ec.dest_row < 0, axis=1)
    assert unchosen.sum() >= 14
    assert np.all(out[unchosen] == 0.0)


# --------------------------------------------------------------------------- backward
BWD_CASES = [
    dict(act="swiglu", gate="softmax"),
    dict(act="relu", gate="softmax", dtype="f32"),
    dict(act="swiglu", gate="sigmoid", shared_F=10, sel_bias_range=0.05),
    dict(act="swiglu", gate="softmax_full"),
    dict(act="swiglu", gate="softmax", capacity_factor=0.5, zipf_s=1.2),
    dict(act="swiglu", gate="softmax", N=3, k=3),
]


@pytest.mark.parametrize("kw", BWD_CASES)
def test_backward_matches_central_differences(kw):
    """<grad, v> of L = <dout, out> equals (L(p + eps v) - L(p - eps v)) / (2 eps)
    for random directions v, routing held fixed, for x and every parameter."""
    kw = dict(kw)
    N, k = kw.pop("N", 5), kw.pop("k", 2)
    inp = tiny(T=9, d=6, N=N, k=k, F=7, **kw)
    wl = inp.wl
    ref = oracle.layer_forward(inp)
    P = oracle.params64(inp)
    x64 = oracle.widen(inp.x, wl.dtype)
    rng = np.random.default_rng(17)
    dout = rng.standard_normal((wl.T, wl.d))
    g = oracle.layer_backward(x64, inp.logit_bias, P, wl.act, wl.gate, ref.idx, ref.disp, dout)

    def L(x_, P_):
        return float(np.sum(dout * oracle.forward_fixed_routing(x_, inp.logit_bias, P_, wl.act, wl.gate,
                                                                 ref.idx, ref.disp)))
    # the fixed-routing forward is the oracle's layer (up to the float32 rounding of
    # the logits the layer's gates see)
    assert np.allclose(oracle.forward_fixed_routing(x64, inp.logit_bias, P, wl.act, wl.gate, ref.idx, ref.disp),
                       ref.out, rtol=1e-6, atol=1e-7)
    eps = 1e-6
    names = ["x", "Wg", "w1", "w3", "w2", "sw1", "sw3", "sw2"]
    grads = {"x": g.dx, "Wg": g.dWg, "w1": g.dw1, "w3": g.dw3, "w2": g.dw2, "sw1": g.dsw1, "sw3": g.dsw3,
             "sw2": g.dsw2}
    for name in names:
        base = x64 if name == "x" else getattr(P, name)
        if base is None:
            assert grads[name] is None
            continue
        v = rng.standard_normal(base.shape)

        def shifted(sign):
            if name == "x":
                return L(x64 + sign * eps * v, P)
            P2 = dataclasses.replace(P, **{name: base + sign * eps * v})
            return L(x64, P2)
        fd = (shifted(1) - shifted(-1)) / (2 * eps)
        an = float(np.sum(grads[name] * v))
        assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (name, fd, an)


def test_backward_dropped_slots_get_no_gradient():
    """CS336 lecture 4, section 10: a dropped assignment has no expert output, so
    neither its gate nor its expert receives gradient from it."""
    inp = tiny(T=12, d=6, N=4, k=2, F=7, capacity_factor=0.01)
    wl = inp.wl
    ref = oracle.layer_forward(inp)
    P = oracle.params64(inp)
    dout = np.ones((wl.T, wl.d))
    g = oracle.layer_backward(oracle.widen(inp.x, "bf16"), None, P, wl.act, wl.gate, ref.idx, ref.disp, dout)
    assert np.all(g.dgate[ref.disp.dest_row < 0] == 0.0)
    fully_dropped = np.all(ref.disp.dest_row < 0, axis=1)
    assert fully_dropped.any()
    assert np.all(g.dx[fully_dropped] == 0.0)


def test_sequence_balance_loss_pins():
    """One sequence spanning the batch gives the batch loss; sequences that are
    each uniform give 1; a sequence routed entirely to one expert with all its
    probability there gives N (CS336 lecture 4, section 9: the batch loss with the
    unit changed to a sequence)."""
    rng = np.random.default_rng(8)
    T, N, k = 60, 6, 2
    z = rng.standard_normal((T, N)).astype(np.float32)
    idx = oracle.topk(z, k)
    d = oracle.dispatch(idx, N, 0)
    batch = oracle.load_stats(z, "softmax", d, k).aux
    assert oracle.sequence_balance_loss(z, idx, "softmax", seq_len=T) == pytest.approx(batch, rel=1e-12)
    assert oracle.sequence_balance_loss(z, idx, "softmax", seq_len=1000) == pytest.approx(batch, rel=1e-12)
    # uniform inside every sequence of 6 tokens, k = 1: f = P = 1/N -> 1
    zu = np.zeros((T, N), dtype=np.float32)
    iu = (np.arange(T) % N).reshape(T, 1).astype(np.int32)
    assert oracle.sequence_balance_loss(zu, iu, "softmax", seq_len=6) == pytest.approx(1.0, abs=1e-14)
    # second sequence collapsed onto expert 2 with all probability there: its loss is N
    zc = np.zeros((12, N), dtype=np.float32)
    zc[6:, 2] = 60.0
    ic = np.concatenate([np.arange(6), np.full(6, 2)]).reshape(12, 1).astype(np.int32)
    assert oracle.sequence_balance_loss(zc, ic, "softmax", seq_len=6) == pytest.approx((1.0 + N) / 2, rel=1e-12)
    # averaging: the mean of the per-sequence losses, the short last sequence included
    l1 = oracle.sequence_balance_loss(z[:50], idx[:50], "softmax", seq_len=50)
    l2 = oracle.sequence_balance_loss(z[50:], idx[50:], "softmax", seq_len=50)
    assert oracle.sequence_balance_loss(z, idx, "softmax", seq_len=50) == pytest.approx((l1 + l2) / 2, rel=1e-12)


@pytest.mark.parametrize("kw", BWD_CASES)
def test_sampled_backward_matches_full_backward(kw):
    """The per-token dx and per-entry weight gradients used for sampled checks of
    full-size layers equal the corresponding entries of the full backward (itself
    pinned by central differences above)."""
    kw = dict(kw)
    N, k = kw.pop("N", 5), kw.pop("k", 2)
    inp = tiny(T=40, d=16, N=N, k=k, F=24, **kw)
    wl = inp.wl
    ref = oracle.layer_forward(inp)
    P = oracle.params64(inp)
    rng = np.random.default_rng(23)
    dout = rng.standard_normal((wl.T, wl.d))
    g = oracle.layer_backward(oracle.widen(inp.x, wl.dtype), inp.logit_bias, P, wl.act, wl.gate, ref.idx, ref.disp,
                              dout)
    tokens = np.array([0, 3, 7, 8, 19, 39])
    dx = oracle.backward_dx_tokens(inp, ref.idx, ref.disp, dout, tokens)
    assert np.allclose(dx, g.dx[tokens], rtol=1e-10, atol=1e-12)
    for which, full in (("w1", g.dw1), ("w3", g.dw3), ("w2", g.dw2)):
        if full is None:
            continue
        entries = [(int(rng.integers(N)), int(rng.integers(full.shape[1])), int(rng.integers(full.shape[2])))
                   for _ in range(12)]
        got = oracle.backward_dw_entries(inp, ref.idx, ref.disp, dout, which, entries)
        want = np.array([full[e, i, j] for e, i, j in entries])
        assert np.allclose(got, want, rtol=1e-10, atol=1e-12), which


# --------------------------------------------------------------------------- FP8 expert weights
def test_e4m3_codes_round_trip_and_known_values():
    """OCP FP8 E4M3: every finite code decodes and encodes back to itself; a few
    values worked by hand from the format (bias 7, 3 mantissa bits, max 448)."""
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)])
    assert np.array_equal(oracle.e4m3_round(oracle.e4m3_value(codes).astype(np.float32)), codes.astype(np.uint8))
    cases = {1.0: 0x38, 448.0: 0x7E, 500.0: 0x7E, 1e9: 0x7E, -448.0: 0xFE, 2.0 ** -9: 0x01, 2.0 ** -6: 0x08,
             0.0: 0x00, 1.5: 0x3C, 240.0: 0x77, 0.875 * 2.0 ** -6: 0x07}
    for v, c in cases.items():
        assert oracle.e4m3_round(np.float32(v)) == c, (v, hex(c))
    assert oracle.e4m3_round(np.float32(-0.0)) == 0x80
    assert np.isnan(oracle.e4m3_value(0x7F)) and oracle.e4m3_value(0x7E) == 448.0


def test_e4m3_rounding_is_nearest_with_ties_to_even():
    """Midpoints of adjacent codes go to the even code, anything off the midpoint to
    the nearer value; brute force over all codes and random values."""
    vals = oracle.e4m3_value(np.arange(0, 0x7F))
    for c in range(0, 0x7E):
        mid = (vals[c] + vals[c + 1]) / 2
        if np.float32(mid) != mid:
            continue
        want = c if c % 2 == 0 else c + 1
        assert oracle.e4m3_round(np.float32(mid)) == want
        assert oracle.e4m3_round(np.nextafter(np.float32(mid), np.float32(0))) == c
        assert oracle.e4m3_round(np.nextafter(np.float32(mid), np.float32(1e9))) == c + 1
    rng = np.random.default_rng(3)
    v = (rng.standard_normal(20000) * rng.choice([1e-3, 1e-1, 10.0, 300.0], 20000)).astype(np.float32)
    got = oracle.e4m3_value(oracle.e4m3_round(v))
    allv = oracle.e4m3_value(np.arange(256))
    finite = allv[np.isfinite(allv)]
    best = np.min(np.abs(finite[None, :] - np.clip(v, -448, 448).astype(np.float64)[:, None]), axis=1)
    assert np.allclose(np.abs(got - np.clip(v, -448, 448)), best, rtol=0, atol=1e-12)


def test_fp8_row_quantisation():
    """The largest magnitude of each row maps to +-448; the dequantised weights are
    within half an E4M3 step (2^-4 relative) of the originals for normal values; a
    zero row gets scale 1 and zero codes; weights that are already E4M3 values times
    a scale round-trip exactly, so the FP8 layer then equals the bf16 layer."""
    rng = np.random.default_rng(4)
    w = (rng.standard_normal((6, 40)) * 0.02).astype(np.float32)
    w[2] = 0.0
    q, s = oracle.quantize_fp8_rows(w)
    assert q.dtype == np.uint8 and s.dtype == np.float32
    nz = [0, 1, 3, 4, 5]
    assert np.all(np.max(np.abs(oracle.e4m3_value(q[nz])), axis=1) == 448.0)
    assert s[2] == 1.0 and np.all(q[2] == 0)
    deq = oracle.dequantize_fp8_rows(q, s)
    normal = np.abs(w) >= (2.0 ** -6) * s[:, None]
    assert np.all(np.abs(deq - w)[normal] <= 2.0 ** -4 * np.abs(w)[normal] + 1e-12)
    # layer: bf16 weights that are E4M3 values times per-row scales
    inp = tiny(T=12, d=16, N=4, k=2, F=24)
    wl = inp.wl

    def exact_fp8_bf16(shape, seed):
        r = np.random.default_rng(seed)
        codes = r.integers(0, 0x7E, size=shape)
        codes[..., 0] = 0x7E                                   # every row reaches 448
        codes = codes | np.where(r.random(shape) < 0.5, 0x80, 0)
        scale = 2.0 ** r.integers(-12, -6, size=shape[:-1])    # powers of two: products stay in bf16
        vals = (oracle.e4m3_value(codes) * scale[..., None]).astype(np.float32)
        return (vals.view(np.uint32) >> 16).astype(np.uint16)  # exact: at most 4 significant bits
    import dataclasses as dc
    inp = dc.replace(inp, w1=exact_fp8_bf16(inp.w1.shape, 1), w3=exact_fp8_bf16(inp.w3.shape, 2),
                     w2=exact_fp8_bf16(inp.w2.shape, 3))
    qs = [oracle.quantize_fp8_rows(oracle.widen(w_, "bf16")) for w_ in (inp.w1, inp.w3, inp.w2)]
    for w_, (q_, s_) in zip((inp.w1, inp.w3, inp.w2), qs):
        assert np.array_equal(oracle.dequantize_fp8_rows(q_, s_), oracle.widen(w_, "bf16"))
    ref = oracle.layer_forward(inp)
    f8 = oracle.layer_forward_fp8(inp, qs[0][0], qs[0][1], qs[1][0], qs[1][1], qs[2][0], qs[2][1])
    assert np.allclose(f8.out, ref.out, rtol=0, atol=1e-12)


# --------------------------------------------------------------------------- router helpers, pinned directly
def test_router_logits_orientation_bias_and_single_rounding():
    """z[t, e] = sum_j x[t, j] W[j, e] + beta_e, summed exactly (in double) and rounded
    once: a one-hot x picks a row of W; 1e8 + 1 - 1e8 keeps its 1 (a float32 running
    sum would lose it)."""
    W = np.array([[1.0, 2.0, 3.0], [4.0, 5.0, 6.0]], dtype=np.float32)   # [d=2, N=3]
    x = np.array([[0.0, 1.0], [1.0, 0.0]])
    assert np.array_equal(oracle.router_logits(x, W, None), np.array([[4, 5, 6], [1, 2, 3]], np.float32))
    beta = np.array([0.5, -1.0, 0.25], dtype=np.float32)
    assert np.array_equal(oracle.router_logits(x, W, beta), np.array([[4.5, 4, 6.25], [1.5, 1, 3.25]], np.float32))
    W2 = np.array([[1e8], [1.0], [-1e8]], dtype=np.float32)
    z = oracle.router_logits(np.ones((1, 3)), W2, None)
    assert z.dtype == np.float32 and z[0, 0] == 1.0


def test_sigmoid_affinity_closed_forms():
    z = np.array([0.0, np.log(3.0), -np.log(3.0), 40.0, -40.0], dtype=np.float32)
    s = oracle.sigmoid_affinity(z)
    assert s.dtype == np.float32
    assert s[0] == 0.5 and s[1] == np.float32(0.75) and s[2] == np.float32(0.25)
    assert s[3] == 1.0 and 0 < s[4] < 1e-17
    zz = np.linspace(-8, 8, 101, dtype=np.float32)
    assert np.all(np.abs(oracle.sigmoid_affinity(zz).astype(np.float64) +
                         oracle.sigmoid_affinity(-zz).astype(np.float64) - 1.0) <= 2.0 ** -24)


def test_selection_scores_by_gate():
    z = np.array([[0.0, np.log(3.0)]], dtype=np.float32)
    for gate in ("softmax", "softmax_full"):
        sel, s = oracle.selection_scores(z, gate, None)
        assert sel is z and s is None
    sel, s = oracle.selection_scores(z, "sigmoid", None)
    assert np.array_equal(sel, s) and s[0, 1] == np.float32(0.75)
    b = np.array([0.375, 0.125], dtype=np.float32)
    sel, s = oracle.selection_scores(z, "sigmoid", b)
    assert np.array_equal(sel, np.array([[0.875, 0.875]], np.float32))     # 0.5 + 0.375, 0.75 + 0.125
    assert np.array_equal(s, np.array([[0.5, 0.75]], np.float32))           # the bias does not enter s


def test_router_probabilities_closed_forms():
    z = np.array([[0.0, np.log(3.0)], [5.0, 5.0 + np.log(3.0)]], dtype=np.float32)
    p = oracle.router_probabilities(z, "softmax")
    assert np.allclose(p, [[0.25, 0.75], [0.25, 0.75]], rtol=0, atol=1e-7)  # shift invariance
    assert np.array_equal(oracle.router_probabilities(z, "softmax_full"), p)
    rng = np.random.default_rng(9)
    zr = rng.standard_normal((7, 5)).astype(np.float32)
    pr = oracle.router_probabilities(zr, "softmax")
    assert np.allclose(pr.sum(axis=1), 1.0, atol=1e-14)
    assert np.allclose(pr, np.exp(zr.astype(np.float64)) / np.exp(zr.astype(np.float64)).sum(1, keepdims=True),
                       rtol=1e-13)
    ps = oracle.router_probabilities(np.array([[0.0, np.log(3.0)]], np.float32), "sigmoid")
    assert np.allclose(ps, [[0.5 / 1.25, 0.75 / 1.25]], rtol=1e-7)         # s_i / sum s, no bias


def test_expert_choice_select_worked_example():
    """Each expert takes its C highest-scoring tokens, ties to the lower token index,
    rows in token order; C is clamped to T."""
    sc = np.array([[0.9, 0.1],
                   [0.5, 0.5],
                   [0.5, 0.7],
                   [0.2, 0.7]])
    ec = oracle.expert_choice_select(sc, 2)
    assert ec.chosen.tolist() == [[0, 1], [2, 3]]       # expert 0: 0.9 then the tie 0.5 -> token 1
    assert ec.offsets.tolist() == [0, 2, 4]
    dest = np.full((4, 2), -1)
    dest[0, 0], dest[1, 0], dest[2, 1], dest[3, 1] = 0, 1, 2, 3
    assert np.array_equal(ec.dest_row, dest)
    ec5 = oracle.expert_choice_select(sc, 5)             # C > T: every token, once per expert
    assert ec5.chosen.tolist() == [[0, 1, 2, 3], [0, 1, 2, 3]] and ec5.offsets.tolist() == [0, 4, 8]
