"""The parity rules of parity.py on the CPU: a GPU that reproduces the oracle
passes, a valid near-tie swap passes with that token left out, and a wrong
choice fails.  The "GPU" results here are made on the host."""
import copy

import numpy as np
import pytest

import oracle
import synth
from parity import GAP, check_dispatch_definition, check_layer_dispatch, check_routing


def _case(cap_factor=0.0):
    wl = synth.Workload("rules", 5, T=400, d=64, N=8, k=2, F=64, act="swiglu", gate="softmax", dtype="bf16",
                        capacity_factor=cap_factor)
    inp = synth.make_inputs(wl)
    return inp, oracle.layer_forward(inp, tokens=np.array([], dtype=np.int64))


def _dispatch_args(d):
    return d.counts_routed, d.counts_kept, d.offsets, d.dest_row, d.src_token


@pytest.mark.parametrize("cap_factor", [0.0, 0.8])
def test_exact_reproduction_passes(cap_factor):
    inp, ref = _case(cap_factor)
    cap = oracle.capacity(cap_factor, 400, 2, 8) if cap_factor else 0
    same = check_routing(inp, ref.z, ref.idx.copy(), ref.w.copy(), ref)
    assert same.all()
    agree = check_layer_dispatch(inp.wl, ref.idx, same, *_dispatch_args(ref.disp), cap, ref)
    assert agree.all()


def _near_tie_ref(ref, t):
    """The oracle's result with token t's 2nd and 3rd selection scores made a near tie."""
    r = copy.deepcopy(ref)
    order = np.argsort(-r.sel[t].astype(np.float64), kind="stable")
    r.sel = r.sel.copy()
    r.sel[t, order[2]] = r.sel[t, order[1]] - np.float32(GAP / 4)
    return r, order


@pytest.mark.parametrize("cap_factor", [0.0, 0.8])
def test_valid_near_tie_swap_is_left_out(cap_factor):
    inp, ref = _case(cap_factor)
    cap = oracle.capacity(cap_factor, 400, 2, 8) if cap_factor else 0
    t = 37
    r, order = _near_tie_ref(ref, t)
    idx = r.idx.copy()
    idx[t, 1] = order[2]                  # the GPU took the other side of the tie
    w = r.w.copy()
    same = check_routing(inp, r.z, idx, w, r)
    assert not same[t] and same.sum() == 399
    d = oracle.dispatch(idx, 8, cap)      # a correct dispatch of that top-k
    agree = check_layer_dispatch(inp.wl, idx, same, *_dispatch_args(d), cap, r)
    assert not agree[t]


def test_clear_swap_fails():
    inp, ref = _case()
    srt = -np.sort(-ref.sel.astype(np.float64), axis=1)
    t = int(np.argmax(srt[:, 1] - srt[:, 2]))   # the clearest token
    idx = ref.idx.copy()
    idx[t, 1] = np.argsort(-ref.sel[t])[2]
    with pytest.raises(AssertionError):
        check_routing(inp, ref.z, idx, ref.w, ref)


def test_wrong_gate_weight_fails():
    inp, ref = _case()
    w = ref.w.copy()
    w[5, 0] += 1e-5
    with pytest.raises(AssertionError):
        check_routing(inp, ref.z, ref.idx, w, ref)


@pytest.mark.parametrize("mutate", ["count", "order", "dest", "cap"])
def test_dispatch_definition_catches_mistakes(mutate):
    inp, ref = _case(0.8)
    cap = oracle.capacity(0.8, 400, 2, 8)
    d = copy.deepcopy(ref.disp)
    check_dispatch_definition(8, ref.idx, cap, *_dispatch_args(d))
    if mutate == "count":
        d.counts_routed[0] += 1
    elif mutate == "order":
        d.src_token[[0, 1]] = d.src_token[[1, 0]]
    elif mutate == "dest":
        d.dest_row[3, 0] = -1
    else:
        d.counts_kept[2] -= 1
    with pytest.raises(AssertionError):
        check_dispatch_definition(8, ref.idx, cap, *_dispatch_args(d))
