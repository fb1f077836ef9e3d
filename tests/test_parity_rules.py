"""The parity rules of parity.py on the CPU: a GPU that reproduces the oracle
passes, a valid near-tie swap passes with that token left out, and a wrong
choice fails.  The "GPU" results here are made on the host."""
import copy

import numpy as np
import pytest

import oracle
import synth
from parity import (GAP, check_dispatch_definition, check_layer_dispatch, check_own_logits, check_routing,
                    own_logit_routing, rows_by_gpu_routing)


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
    r.z = r.sel.copy()  # softmax gate: the selection score is the logit
    return r, order


@pytest.mark.parametrize("cap_factor", [0.0, 0.8])
def test_valid_near_tie_swap_is_left_out(cap_factor):
    inp, ref = _case(cap_factor)
    cap = oracle.capacity(cap_factor, 400, 2, 8) if cap_factor else 0
    t = 37
    r, order = _near_tie_ref(ref, t)
    # the GPU's logits put the third expert just above the second: it takes the
    # other side of the near tie, consistently with its own logits
    z = r.z.copy()
    z[t, order[2]] = z[t, order[1]] + np.float32(GAP / 8)
    idx, w, _ = own_logit_routing(z, "softmax", None, 2)
    assert idx[t, 0] == order[2] or idx[t, 1] == order[2]
    same = check_routing(inp, z, idx, w, r)
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


@pytest.mark.parametrize("gate", ["softmax", "softmax_full", "sigmoid"])
def test_higher_index_tie_choice_fails(gate):
    """Experts 2 and 5 get bit-identical logits: where exactly one of them makes
    the top-k, it must be 2.  Taking 5 instead fails the own-logits rule."""
    inp, ref = _case()
    z = ref.z.copy()
    z[:, 5] = z[:, 2]
    idx, w, _ = own_logit_routing(z, gate, None, 2)
    check_own_logits(z, idx, w, gate, None, 2)
    one = np.nonzero(np.sum((idx == 2) | (idx == 5), axis=1) == 1)[0]
    assert one.size > 0 and np.all(np.any(idx[one] == 2, axis=1))
    bad = idx.copy()
    t = one[0]
    bad[t][bad[t] == 2] = 5
    with pytest.raises(AssertionError):
        check_own_logits(z, bad, w, gate, None, 2)


def test_own_logits_rule_catches_a_slot_swap_and_a_gate_error():
    inp, ref = _case()
    idx, w, _ = own_logit_routing(ref.z, "softmax", None, 2)
    assert np.array_equal(idx, ref.idx) and np.max(np.abs(w - ref.w)) < 1e-12
    bad = idx.copy()
    bad[7] = bad[7][::-1]
    with pytest.raises(AssertionError):
        check_own_logits(ref.z, bad, w, "softmax", None, 2)
    w2 = w.copy()
    w2[9, 1] += 2e-6
    with pytest.raises(AssertionError):
        check_own_logits(ref.z, idx, w2, "softmax", None, 2)


def test_rows_by_gpu_routing_reproduces_the_oracle_on_its_own_routing():
    """With the oracle's own routing in place of the GPU's, the per-token
    composition equals the oracle's output rows (to rounding)."""
    wl = synth.Workload("rules2", 6, T=64, d=64, N=8, k=2, F=64, act="swiglu", gate="sigmoid", dtype="bf16",
                        shared_F=64, sel_bias_range=0.05)
    inp = synth.make_inputs(wl)
    ref = oracle.layer_forward(inp)
    toks = np.array([0, 5, 63])
    got = rows_by_gpu_routing(inp, ref, toks, ref.z, ref.idx, ref.disp.dest_row)
    assert np.max(np.abs(got - ref.out[toks])) <= 1e-5 * np.max(np.abs(ref.out[toks]))
