"""Exact ties in the router's top-k go to the lower expert index, on the GPU (B300).

Lecture29, "Top-two routing": S_k(x) is the set of the k largest logits; the
pages leave equal scores open, and the reading taken is the lower expert index
first, slots ordered by (score desc, index asc).  Ties are forced by giving
several experts bit-identical router columns (each column of W_g copied from one
of M < N base columns, the copies spread across lanes and lane slots), with the
selection bias -- where there is one -- copied the same way, and by saturating
the sigmoid (logits above ~17 all give the affinity 1.0 in float32).

Checked on every token: the duplicated columns' logits are bit-identical on the
GPU (so the ties reach the top-k), the GPU's top-k is exactly the (score desc,
index asc) top-k of its own logits, no unselected expert with a score equal to a
selected one has a lower index, and the GPU's top-k equals the oracle's (which
sees the same ties in its own logits) on every token whose k + 1 largest scores
are pairwise either equal or more than 1e-4 apart.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import sparse_mixture_experts_62_b300 as moe
import synth
from parity import GAP, check_own_logits, config_of, own_logit_routing, to_dev

pytestmark = pytest.mark.gpu

TID_BASE_WG, TID_BASE_B = 51, 52


def _tied_inputs(gate, T, d, N, k, M, layout, scale, bias):
    wl = synth.Workload("ties", 777 + N + k, T=T, d=d, N=N, k=k, F=64, act="swiglu", gate=gate, dtype="bf16")
    x = synth.normal(wl.seed, synth.TID_X, (T, d), 1.0, "bf16")
    base = synth.normal(wl.seed, TID_BASE_WG, (d, M), scale / math.sqrt(d), "f32")
    if layout == "mod":
        src = np.arange(N) % M
    else:  # seeded positions
        src = np.random.default_rng(wl.seed).permutation(np.arange(N) % M)
    Wg = np.ascontiguousarray(base[:, src])
    sb = None
    if bias:
        sb = np.ascontiguousarray(synth.uniform(wl.seed, TID_BASE_B, (M,), -0.05, 0.05)[src])
    return synth.LayerInputs(wl, x, Wg, None, None, None, sel_bias=sb), src


def tie_or_clear(sel, k):
    """Tokens whose k + 1 largest scores (with multiplicity) are pairwise either
    exactly equal or more than 1e-4 apart: there the set and order follow from
    the scores' values and the index tie-break alone."""
    srt = -np.sort(-sel.astype(np.float64), axis=1)[:, :k + 1]
    gaps = srt[:, :-1] - srt[:, 1:]
    return np.all((gaps == 0) | (gaps > GAP), axis=1)


CASES = [
    # gate, T, d, N, k, M (distinct columns), layout, W_g scale, selection bias
    ("softmax", 512, 512, 8, 3, 4, "mod", 1.0, False),
    ("softmax", 512, 512, 8, 2, 3, "perm", 1.0, False),
    ("softmax", 512, 2048, 128, 8, 24, "mod", 1.0, False),
    ("softmax", 512, 2048, 128, 8, 40, "perm", 1.0, False),
    ("softmax", 300, 7168, 256, 8, 40, "perm", 1.0, False),
    ("softmax_full", 512, 512, 8, 3, 4, "perm", 1.0, False),
    ("softmax_full", 512, 2048, 256, 8, 40, "mod", 1.0, False),
    ("softmax", 256, 512, 64, 1, 5, "perm", 1.0, False),                 # Switch-style top-1
    ("sigmoid", 512, 512, 8, 3, 4, "mod", 1.0, False),
    ("sigmoid", 512, 2048, 128, 8, 24, "perm", 1.0, True),
    ("sigmoid", 300, 7168, 256, 8, 40, "perm", 1.0, True),
    ("sigmoid", 512, 2048, 256, 8, 40, "mod", 1.0, False),
    ("sigmoid", 512, 512, 8, 2, 8, "mod", 40.0, False),                  # saturated affinities, no copies
    ("sigmoid", 512, 2048, 256, 8, 256, "mod", 40.0, False),             # saturated affinities, N = 256
]


@pytest.mark.parametrize("case", CASES, ids=[f"{c[0]}-N{c[3]}-k{c[4]}-M{c[5]}-{c[6]}"
                                             + ("-sat" if c[7] > 1 else "") + ("-bias" if c[8] else "")
                                             for c in CASES])
def test_exact_ties_go_to_the_lower_index(case):
    gate, T, d, N, k, M, layout, scale, bias = case
    inp, src = _tied_inputs(gate, T, d, N, k, M, layout, scale, bias)
    wl = inp.wl
    cfg = config_of(wl)
    ws = torch.zeros(moe.moe_workspace_size(cfg), dtype=torch.uint8, device="cuda")
    z = torch.empty((T, N), dtype=torch.float32, device="cuda")
    idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), dtype=torch.float32, device="cuda")
    f32 = lambda a: None if a is None else to_dev(a, "f32")  # noqa: E731
    moe.moe_route(cfg, to_dev(inp.x, "bf16"), f32(inp.Wg), None, f32(inp.sel_bias), z, idx, w, ws)
    assert moe.moe_get_device_status(ws) == moe.MOE_OK
    z, idx, w = z.cpu().numpy(), idx.cpu().numpy(), w.cpu().numpy().astype(np.float64)

    # the copies' logits are bit-identical, so the ties reach the top-k
    for m in range(M):
        cols = np.nonzero(src == m)[0]
        assert np.all(z[:, cols] == z[:, cols[:1]]), f"copies of base column {m} differ on the GPU"

    # every token: exactly the (score desc, index asc) top-k of the GPU's own logits
    check_own_logits(z, idx, w, gate, inp.sel_bias, k)
    _, _, sel = own_logit_routing(z, gate, inp.sel_bias, k)
    straddle = 0
    for t in range(T):
        chosen = set(idx[t].tolist())
        for j in range(k):
            e = idx[t, j]
            lower = [f for f in range(e) if f not in chosen and sel[t, f] == sel[t, e]]
            assert not lower, f"token {t}: expert {e} taken over the equal-scored lower index {lower[0]}"
        srt = np.sort(sel[t])[::-1]
        straddle += int(k < N and srt[k - 1] == srt[k])
    # the k-th and (k+1)-th scores are equal on many tokens: the tie-break decides the set
    assert straddle >= T // 10, f"only {straddle} tokens with a tie across the k-th place"

    # the oracle sees the same ties in its own logits and breaks them the same way
    ref = oracle.layer_forward(inp, tokens=np.array([], dtype=np.int64))
    for m in range(M):
        cols = np.nonzero(src == m)[0]
        assert np.all(ref.z[:, cols] == ref.z[:, cols[:1]])
    exact = tie_or_clear(ref.sel, k)
    assert exact.sum() >= T // 2
    assert np.array_equal(idx[exact], ref.idx[exact]), "top-k differs from the oracle's on a tied token"
    assert np.max(np.abs(w[exact] - ref.w[exact])) <= 1e-6
