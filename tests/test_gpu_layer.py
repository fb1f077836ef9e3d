"""Whole-layer parity of moe_layer_forward + moe_load_stats against the oracle (B300).

Small layers are compared on every output; the full-size workloads (the
Mixtral-shaped prefill and decode layers, the DeepSeek-V3-shaped and the
Qwen3-shaped layers) are run in the launch configuration the benchmark times,
with routing, dispatch and statistics compared on all tokens and the layer
output on all tokens -- except the DeepSeek-V3-shaped layer, whose output is
compared on the tokens of the first and last row of every 128-row tile of every
expert group and of the shared expert, plus a seeded sample.  The oracle routes
on its own; the rules for the rare token the two route differently are in
parity.py.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from parity import (assert_close_out, check_layer_dispatch, check_routing, layer_on_device, rows_by_gpu_routing,
                    to_dev, to_np_f64)

pytestmark = pytest.mark.gpu


def tile_edge_tokens(disp, T, extra, seed, tile=128):
    """Tokens whose rows are the first or last row of a 128-row tile of an
    expert group (in the oracle's own dispatch) or of the shared expert's rows
    (token order), plus `extra` seeded tokens."""
    toks = set()
    off = disp.offsets
    for e in range(len(off) - 1):
        for r0 in range(int(off[e]), int(off[e + 1]), tile):
            r1 = min(r0 + tile, int(off[e + 1])) - 1
            toks.add(int(disp.src_token[r0]))
            toks.add(int(disp.src_token[r1]))
    for r0 in range(0, T, tile):
        toks.update((r0, min(r0 + tile, T) - 1))
    toks.update(np.random.default_rng(seed).choice(T, extra, replace=False).tolist())
    return np.array(sorted(toks), dtype=np.int64)


def run_and_check(inp, sample=None):
    """sample: None (every token's output), an int (that many seeded tokens) or
    "tiles" (tile_edge_tokens of the oracle's dispatch plus 256 seeded tokens)."""
    wl = inp.wl
    layer = layer_on_device(inp)
    x = to_dev(inp.x, wl.dtype)
    out = layer.forward(x)
    f, P, summ = layer.load_stats()
    torch.cuda.synchronize()
    assert layer.device_status() == 0
    v = layer.views()
    z = v["logits"].cpu().numpy()
    idx = v["topk_idx"].cpu().numpy()
    w = v["topk_w"].cpu().numpy().astype(np.float64)
    if sample is None:
        tokens = None
    elif sample == "tiles":
        own = oracle.layer_forward(inp, tokens=np.array([], dtype=np.int64))  # the oracle's own dispatch
        tokens = tile_edge_tokens(own.disp, wl.T, 256, wl.seed)
    else:
        tokens = np.sort(np.random.default_rng(wl.seed).choice(wl.T, sample, replace=False))
    ref = oracle.layer_forward(inp, tokens=tokens)  # the oracle's own routing, from the inputs alone
    same = check_routing(inp, z, idx, w, ref)
    cap = layer.cfg.capacity
    agree = check_layer_dispatch(wl, idx, same, v["counts_routed"].cpu().numpy(), v["counts_kept"].cpu().numpy(),
                                 v["offsets"].cpu().numpy(), v["dest_row"].cpu().numpy(),
                                 v["src_token"].cpu().numpy(), cap, ref)
    got = to_np_f64(out)
    rows = np.arange(wl.T) if tokens is None else tokens
    other = rows[~agree[rows]]
    rows = rows[agree[rows]]
    err, tol = assert_close_out(got[rows], ref.out[rows], wl.dtype)
    # tokens routed (or kept) differently: the GPU's own routing with the oracle's experts
    if other.size:
        dest = v["dest_row"].cpu().numpy()
        assert_close_out(got[other], rows_by_gpu_routing(inp, ref, other, z, idx, dest), wl.dtype,
                         what="output of tokens routed differently from the oracle")
    # statistics: exact where no differing token touches an expert
    fg = f.cpu().numpy()
    if np.all(same):
        assert np.array_equal(fg, ref.stats.f.astype(np.float32))
    assert np.max(np.abs(fg - ref.stats.f)) <= 2.0 * np.sum(~same) / (wl.T * wl.k) + 1e-7
    assert np.max(np.abs(P.cpu().numpy() - ref.stats.P)) < 1e-5
    s = summ.cpu().numpy().astype(np.float64)
    exact = bool(np.all(same))
    assert s[0] == pytest.approx(ref.stats.aux, rel=1e-5 if exact else 1e-3)
    assert s[1] == pytest.approx(ref.stats.imbalance, rel=1e-6 if exact else 1e-2)
    assert s[2] == pytest.approx(ref.stats.drop_rate, rel=1e-6 if exact else 1e-2, abs=1e-7 if exact else 1e-3)
    # sequence-wise balance loss over sequences of a quarter of the batch
    L = max(1, wl.T // 4)
    sbl = float(layer.seq_balance_loss(L).item())
    sref = oracle.sequence_balance_loss(ref.z, ref.idx, wl.gate, L)
    assert sbl == pytest.approx(sref, rel=1e-5 if exact else 1e-3)
    return dict(err=err, tol=tol, differing=int(np.sum(~same)), kept=int(v["offsets"][-1]))


SMALL = [
    dict(T=333, d=256, N=8, k=2, F=384),                                   # ragged tails everywhere
    dict(T=200, d=512, N=16, k=4, F=256, gate="sigmoid", shared_F=384, sel_bias_range=0.05),
    dict(T=500, d=256, N=8, k=3, F=128, capacity_factor=0.75, zipf_s=1.2),
    dict(T=64, d=64, N=1, k=1, F=64),
    dict(T=50, d=128, N=4, k=4, F=192),
    dict(T=129, d=320, N=7, k=2, F=136, act="relu"),
    dict(T=1, d=64, N=8, k=2, F=64),
    dict(T=1500, d=256, N=4, k=2, F=384),                                  # CTA-pair tiles (750 rows/expert)
    dict(T=400, d=256, N=16, k=4, F=256, gate="softmax_full"),             # full softmax, no renormalisation
    dict(T=300, d=256, N=32, k=1, F=256, capacity_factor=1.0),             # Switch-style top-1 with capacity
    dict(T=2000, d=256, N=8, k=2, F=256, capacity_factor=1.25, zipf_s=1.2),  # capacity: pair and single tiles
]


@pytest.mark.parametrize("kw", SMALL)
def test_layer_small(kw):
    kw = dict(kw)
    wl = synth.Workload("small", 21, act=kw.pop("act", "swiglu"), gate=kw.pop("gate", "softmax"), dtype="bf16", **kw)
    run_and_check(synth.make_inputs(wl))


def test_layer_shazeer_tiny_f32_full():
    """The float32 workload at full size: T=256, d=512, 8 ReLU experts 512->1024->512."""
    run_and_check(synth.make_inputs(synth.WORKLOADS["shazeer_tiny_f32"]))


def test_layer_mixtral_decode_full():
    run_and_check(synth.make_inputs(synth.WORKLOADS["mixtral_decode"]))


def test_layer_qwen3_skew_drop_full():
    r = run_and_check(synth.make_inputs(synth.WORKLOADS["qwen3_skew_drop"]))
    assert r["kept"] < 16384 * 8  # capacity actually drops assignments


def test_layer_mixtral_prefill_full():
    run_and_check(synth.make_inputs(synth.WORKLOADS["mixtral_prefill"]))


def test_layer_dsv3_finegrained_full():
    run_and_check(synth.make_inputs(synth.WORKLOADS["dsv3_finegrained"]), sample="tiles")


def test_layer_deterministic():
    wl = synth.Workload("det", 5, T=300, d=256, N=8, k=2, F=256, act="swiglu", gate="softmax", dtype="bf16")
    inp = synth.make_inputs(wl)
    layer = layer_on_device(inp)
    x = to_dev(inp.x, "bf16")
    a = layer.forward(x).clone()
    b = layer.forward(x).clone()
    assert torch.equal(a, b)


def test_layer_deterministic_with_pair_tiles():
    """Groups of ~1024 rows run on CTA pairs, which take their tiles in issue order
    from a counter, so which pair computes which tile changes from run to run; each
    tile is computed by one pair in a fixed K order, so the output must not."""
    wl = synth.Workload("detp", 6, T=2048, d=512, N=4, k=2, F=1024, act="swiglu", gate="softmax", dtype="bf16")
    inp = synth.make_inputs(wl)
    layer = layer_on_device(inp)
    x = to_dev(inp.x, "bf16")
    ref = layer.forward(x).clone()
    for _ in range(4):
        assert torch.equal(layer.forward(x), ref)
    assert layer.device_status() == 0  # MOE_OK
