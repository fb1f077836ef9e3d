"""Backward pass on the GPU against the oracle's (B300).

The forward runs through moe_layer_forward; moe_layer_backward then produces
float32 gradients, compared with oracle.layer_backward on the oracle's own
routing (its top-k and kept set, from the inputs alone) under the bf16 rule
max|gpu - ref| <= 2e-2 max|ref| + 1e-3 per tensor: the backward's intermediates
(dy, dh, a, u, dA, dx rows) are bf16.  The router gradient couples every token,
so each case requires the GPU to have routed every token as the oracle did
(checked first; none of these seeded cases has a token near enough to a tie to
flip).
"""
import numpy as np
import pytest
import torch

import oracle
import sparse_mixture_experts_62_b300 as moe
import synth
from parity import assert_close_out, check_layer_dispatch, check_routing, layer_on_device, to_dev

pytestmark = pytest.mark.gpu

CASES = [
    dict(T=200, d=128, N=8, k=2, F=192),
    dict(T=300, d=256, N=16, k=4, F=128, gate="sigmoid", shared_F=192, sel_bias_range=0.05),
    dict(T=256, d=128, N=8, k=3, F=256, gate="softmax_full"),
    dict(T=400, d=128, N=8, k=2, F=128, capacity_factor=0.6, zipf_s=1.2),
    dict(T=150, d=192, N=5, k=2, F=160, act="relu"),
    dict(T=1500, d=256, N=4, k=2, F=256),            # CTA-pair tiles in the GEMMs
    dict(T=512, d=1024, N=8, k=2, F=2048),
    dict(T=2000, d=128, N=8, k=2, F=128, capacity_factor=1.25, zipf_s=1.2),  # pair tiles for the capped groups
]


@pytest.mark.parametrize("kw", CASES)
def test_backward_parity(kw):
    kw = dict(kw)
    wl = synth.Workload("bwd", 41, act=kw.pop("act", "swiglu"), gate=kw.pop("gate", "softmax"), dtype="bf16", **kw)
    inp = synth.make_inputs(wl)
    layer = layer_on_device(inp)
    x = to_dev(inp.x, "bf16")
    layer.forward(x)
    cfg = layer.cfg
    dout_np = synth.normal(wl.seed, 77, (wl.T, wl.d), 1.0, "bf16")
    dout = to_dev(dout_np, "bf16")
    f32 = lambda shape: torch.full(shape, float("nan"), device="cuda")  # noqa: E731  (all must be overwritten)
    sw = wl.act == "swiglu"
    g = dict(dx=f32((wl.T, wl.d)), dWg=f32((wl.d, wl.N)), dw1=f32((wl.N, wl.F, wl.d)),
             dw3=f32((wl.N, wl.F, wl.d)) if sw else None, dw2=f32((wl.N, wl.d, wl.F)))
    Fs = wl.shared_F
    if Fs:
        g.update(dsw1=f32((Fs, wl.d)), dsw3=f32((Fs, wl.d)) if sw else None, dsw2=f32((wl.d, Fs)))
    bws = torch.zeros(moe.moe_backward_workspace_size(cfg), dtype=torch.uint8, device="cuda")
    moe.moe_layer_backward(cfg, x, layer.Wg, layer.w1, layer.w3, layer.w2, layer.sw1, layer.sw3, layer.sw2, dout,
                           g["dx"], g["dWg"], g["dw1"], g.get("dw3"), g["dw2"], g.get("dsw1"), g.get("dsw3"),
                           g.get("dsw2"), layer.ws, bws)
    torch.cuda.synchronize()
    assert layer.device_status() == 0
    v = layer.views()
    own = oracle.layer_forward(inp, tokens=np.array([], dtype=np.int64))  # the oracle's routing
    idx = v["topk_idx"].cpu().numpy()
    same = check_routing(inp, v["logits"].cpu().numpy(), idx, v["topk_w"].cpu().numpy().astype(np.float64), own)
    agree = check_layer_dispatch(wl, idx, same, v["counts_routed"].cpu().numpy(), v["counts_kept"].cpu().numpy(),
                                 v["offsets"].cpu().numpy(), v["dest_row"].cpu().numpy(),
                                 v["src_token"].cpu().numpy(), cfg.capacity, own)
    assert np.all(agree), "the GPU routed a token differently from the oracle"
    disp = own.disp
    ref = oracle.layer_backward(oracle.widen(inp.x, "bf16"), inp.logit_bias, oracle.params64(inp), wl.act, wl.gate,
                                own.idx, disp, oracle.widen(dout_np, "bf16"))
    pairs = [("dx", ref.dx), ("dWg", ref.dWg), ("dw1", ref.dw1), ("dw2", ref.dw2)]
    if sw:
        pairs.append(("dw3", ref.dw3))
    if Fs:
        pairs += [("dsw1", ref.dsw1), ("dsw2", ref.dsw2)] + ([("dsw3", ref.dsw3)] if sw else [])
    for name, r in pairs:
        got = g[name].cpu().numpy().astype(np.float64)
        assert np.all(np.isfinite(got)), name
        assert_close_out(got, r, "bf16", what=name)
    # experts that processed no token get exactly zero gradient
    unused = np.nonzero(disp.counts_kept == 0)[0]
    for e in unused:
        assert np.all(g["dw1"][e].cpu().numpy() == 0.0) and np.all(g["dw2"][e].cpu().numpy() == 0.0)


def test_backward_rejects_unsupported_configs():
    cfg = moe.make_config(64, 64, 8, 2, 128, dtype=moe.DTYPE_F32)
    with pytest.raises(moe.MoeError) as e:
        moe.moe_backward_workspace_size(cfg)
    assert e.value.code == moe.MOE_ERR_UNSUPPORTED


def test_backward_mixtral_prefill_full_sampled():
    """The backward at the Mixtral prefill size in the launch configuration the
    bench times (CTA-pair tiles, pair weight-gradient GEMMs): dx on a seeded sample
    of tokens and 16 seeded entries of each expert weight gradient against the
    oracle's per-token / per-entry gradients, under the bf16 rule per tensor."""
    wl = synth.WORKLOADS["mixtral_prefill"]
    inp = synth.make_inputs(wl)
    layer = layer_on_device(inp)
    x = to_dev(inp.x, "bf16")
    layer.forward(x)
    cfg = layer.cfg
    dout_np = synth.normal(wl.seed, 77, (wl.T, wl.d), 1.0, "bf16")
    dout = to_dev(dout_np, "bf16")
    f32 = lambda shape: torch.full(shape, float("nan"), device="cuda")  # noqa: E731
    dx, dWg = f32((wl.T, wl.d)), f32((wl.d, wl.N))
    dw1, dw3, dw2 = f32((wl.N, wl.F, wl.d)), f32((wl.N, wl.F, wl.d)), f32((wl.N, wl.d, wl.F))
    bws = torch.zeros(moe.moe_backward_workspace_size(cfg), dtype=torch.uint8, device="cuda")
    moe.moe_layer_backward(cfg, x, layer.Wg, layer.w1, layer.w3, layer.w2, None, None, None, dout, dx, dWg, dw1, dw3,
                           dw2, None, None, None, layer.ws, bws)
    torch.cuda.synchronize()
    assert layer.device_status() == 0
    v = layer.views()
    own = oracle.layer_forward(inp, tokens=np.array([], dtype=np.int64))  # the oracle's routing
    idx = v["topk_idx"].cpu().numpy()
    same = check_routing(inp, v["logits"].cpu().numpy(), idx, v["topk_w"].cpu().numpy().astype(np.float64), own)
    agree = check_layer_dispatch(wl, idx, same, v["counts_routed"].cpu().numpy(), v["counts_kept"].cpu().numpy(),
                                 v["offsets"].cpu().numpy(), v["dest_row"].cpu().numpy(),
                                 v["src_token"].cpu().numpy(), cfg.capacity, own)
    assert np.all(agree), "the GPU routed a token differently from the oracle"
    dout64 = oracle.widen(dout_np, "bf16")
    rng = np.random.default_rng(wl.seed)
    tokens = np.sort(rng.choice(wl.T, 24, replace=False))
    ref_dx = oracle.backward_dx_tokens(inp, own.idx, own.disp, dout64, tokens)
    got_dx = dx[torch.from_numpy(tokens).cuda()].cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(got_dx))
    assert_close_out(got_dx, ref_dx, "bf16", what="dx (sampled tokens)")
    for which, t, shape in (("w1", dw1, (wl.N, wl.F, wl.d)), ("w3", dw3, (wl.N, wl.F, wl.d)),
                            ("w2", dw2, (wl.N, wl.d, wl.F))):
        entries = [(int(rng.integers(shape[0])), int(rng.integers(shape[1])), int(rng.integers(shape[2])))
                   for _ in range(16)]
        ref = oracle.backward_dw_entries(inp, own.idx, own.disp, dout64, which, entries)
        got = np.array([float(t[e, i, j].item()) for e, i, j in entries])
        assert_close_out(got, ref, "bf16", what=f"d{which} (sampled entries)")
