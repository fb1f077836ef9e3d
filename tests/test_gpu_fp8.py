"""FP8 E4M3 expert weights on the GPU against the oracle (B300).

The codes and scales of moe_quantize_fp8 equal the oracle's quantisation exactly
(both take the rounding decision on the same float32 quotient); the FP8 expert
FFN and layer are compared with the oracle's layer on its own dequantised weights
(its own quantisation of the same bf16 weights) under the bf16 rule.
"""
import numpy as np
import pytest
import torch

import oracle
import sparse_mixture_experts_62_b300 as moe
import synth
from parity import assert_close_out, check_layer_dispatch, check_routing, layer_on_device, to_dev, to_np_f64

pytestmark = pytest.mark.gpu


def _quantize_on_gpu(w_bits):
    w = to_dev(w_bits, "bf16")
    q = torch.empty(w.shape, dtype=torch.uint8, device="cuda")
    s = torch.empty(w.shape[:-1], dtype=torch.float32, device="cuda")
    moe.moe_quantize_fp8(w, q, s)
    return q, s


@pytest.mark.parametrize("shape,std", [((4, 96, 64), 0.02), ((2, 48, 1024), 1.0), ((3, 16, 32), 1e-4)])
def test_quantize_matches_oracle(shape, std):
    w = synth.normal(7, 11, shape, std, "bf16")
    w[0, 3] = 0                                  # an all-zero row
    q, s = _quantize_on_gpu(w)
    q_ref, s_ref = oracle.quantize_fp8_rows(oracle.widen(w, "bf16"))
    assert np.array_equal(s.cpu().numpy(), s_ref)
    assert np.array_equal(q.cpu().numpy(), q_ref)


def _fp8_ffn_case(N, counts, d, F, act, seed, T=None, k=1):
    """counts must sum to T * k (the routed rows); T bounds a group's rows for the kernel choice."""
    R = int(sum(counts))
    T = R if T is None else T
    assert R == T * k
    cfg = moe.make_config(T, d, N, k, F, 0, moe.GATE_SOFTMAX_TOPK,
                          moe.ACT_SWIGLU if act == "swiglu" else moe.ACT_RELU, moe.DTYPE_BF16, 0)
    xp = synth.normal(seed, 99, (R, d), 1.0, "bf16")
    w1 = synth.normal(seed, 3, (N, F, d), d ** -0.5, "bf16")
    w3 = synth.normal(seed, 4, (N, F, d), d ** -0.5, "bf16") if act == "swiglu" else None
    w2 = synth.normal(seed, 5, (N, d, F), F ** -0.5, "bf16")
    (q1, s1), (q2, s2) = _quantize_on_gpu(w1), _quantize_on_gpu(w2)
    q3, s3 = _quantize_on_gpu(w3) if w3 is not None else (None, None)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    ws = torch.zeros(moe.moe_workspace_size(cfg), dtype=torch.uint8, device="cuda")
    y = torch.empty((R, d), dtype=torch.bfloat16, device="cuda")
    moe.moe_expert_ffn_fp8(cfg, to_dev(xp, "bf16"), torch.from_numpy(offsets).cuda(), q1, s1, q3, s3, q2, s2, y, ws)
    assert moe.moe_get_device_status(ws) == moe.MOE_OK
    y = to_np_f64(y)
    x64 = oracle.widen(xp, "bf16")
    r1, r2 = oracle.quantize_fp8_rows(oracle.widen(w1, "bf16")), oracle.quantize_fp8_rows(oracle.widen(w2, "bf16"))
    r3 = oracle.quantize_fp8_rows(oracle.widen(w3, "bf16")) if w3 is not None else None
    for e in range(N):
        a, b = offsets[e], offsets[e + 1]
        if b == a:
            continue
        ref = oracle.expert_ffn(x64[a:b], oracle.dequantize_fp8_rows(r1[0][e], r1[1][e]),
                                oracle.dequantize_fp8_rows(r3[0][e], r3[1][e]) if r3 is not None else None,
                                oracle.dequantize_fp8_rows(r2[0][e], r2[1][e]), act)
        assert_close_out(y[a:b], ref, "bf16", what=f"expert {e}")


@pytest.mark.parametrize("act", ["swiglu", "relu"])
def test_fp8_expert_ffn_ragged_groups(act):
    """Empty, one-row and multi-tile groups; F and d multiples of 16 but not of the tile."""
    _fp8_ffn_case(5, [0, 1, 130, 257, 64], d=208, F=336, act=act, seed=2)


def test_fp8_expert_ffn_deep_k():
    _fp8_ffn_case(4, [40, 3, 200, 129], d=1024, F=512, act="swiglu", seed=3)


# Decode-sized groups (at most 64 rows per group by the config's T): the weights
# take the M side of the MMA and the tokens come in tiles of 16, 32 or 64 rows.
# Groups larger than T (possible through moe_expert_ffn_fp8's own offsets) take
# several token tiles; widths are not multiples of the 128-row or 128-wide K tiles.
@pytest.mark.parametrize("act", ["swiglu", "relu"])
@pytest.mark.parametrize("T,k,counts", [(16, 4, [0, 1, 40, 23]), (30, 3, [30, 0, 29, 31]),
                                        (64, 2, [64, 0, 50, 14]), (5, 1, [0, 0, 5, 0])])
def test_fp8_expert_ffn_decode_groups(act, T, k, counts):
    _fp8_ffn_case(len(counts), counts, d=208, F=336, act=act, seed=4, T=T, k=k)


def test_fp8_expert_ffn_decode_deep_k():
    _fp8_ffn_case(4, [16, 3, 9, 4], d=1024, F=1536, act="swiglu", seed=5, T=16, k=2)


_NAN_CODES = (0x7F, 0xFF)


def _all_codes(n):
    c = (np.arange(n) % 256).astype(np.uint8)
    c[np.isin(c, _NAN_CODES)] = 0
    return c


@pytest.mark.parametrize("T", [16, 100])
@pytest.mark.parametrize("path", ["down", "up"])
def test_fp8_every_code_exact(T, path):
    """Every finite E4M3 code through the weight converter, compared exactly.

    One expert, d = F = 256, every token x = e_0.  W1[:, 0] = 16.0 makes the gate
    pre-activation 16, whose SiLU rounds to 16 in float32; then
      down: W3[5, 0] = 1 only, so h = 16 e_5, and y[n] = 16 s2[n] v(W2[n, 5]);
      up:   W3[f, 0] = code f, W2 = I, so y[n] = bf16(silu(16) v(code n)) = 16 v(code n).
    Each y is a short binary fraction, exact in bf16.  T = 16 runs the decode
    kernel (weights on the M side), T = 100 the token-tile kernel.  The value of a
    code comes from the oracle's E4M3 table.
    """
    d = F = 256
    rng = np.random.default_rng(8)
    finite = np.setdiff1d(np.arange(256), _NAN_CODES).astype(np.uint8)
    rand = lambda shape: rng.choice(finite, size=shape).astype(np.uint8)
    q1, q3, q2 = rand((1, F, d)), rand((1, F, d)), rand((1, d, F))
    s1, s3, s2 = np.ones((1, F), np.float32), np.ones((1, F), np.float32), np.ones((1, d), np.float32)
    q1[0, :, 0] = 0x58                                   # 16.0
    if path == "down":
        q3[0, :, 0] = 0
        q3[0, 5, 0] = 0x38                               # 1.0
        q2[0, :, 5] = _all_codes(d)
        s2[0] = 2.0 ** (np.arange(d) % 5 - 2)
        expect = 16.0 * s2[0].astype(np.float64) * oracle.e4m3_value(q2[0, :, 5])
    else:
        q3[0, :, 0] = _all_codes(F)
        q2[0] = 0
        q2[0, np.arange(d), np.arange(d)] = 0x38
        expect = 16.0 * oracle.e4m3_value(q3[0, :, 0])
    x = np.zeros((T, d), np.float32)
    x[:, 0] = 1.0
    cfg = moe.make_config(T, d, 1, 1, F)
    ws = torch.zeros(moe.moe_workspace_size(cfg), dtype=torch.uint8, device="cuda")
    y = torch.empty((T, d), dtype=torch.bfloat16, device="cuda")
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    offsets = dev(np.array([0, T], np.int32))
    moe.moe_expert_ffn_fp8(cfg, torch.from_numpy(x).to(torch.bfloat16).cuda(), offsets, dev(q1), dev(s1), dev(q3),
                           dev(s3), dev(q2), dev(s2), y, ws)
    assert moe.moe_get_device_status(ws) == moe.MOE_OK
    got = y.float().cpu().numpy().astype(np.float64)
    assert np.array_equal(got, np.broadcast_to(expect, got.shape))


def _fp8_layer_check(inp, sample=None):
    wl = inp.wl
    layer = layer_on_device(inp)
    layer.quantize_fp8()
    out = layer.forward(to_dev(inp.x, "bf16"))
    torch.cuda.synchronize()
    assert layer.device_status() == 0
    v = layer.views()
    tokens = None if sample is None else np.sort(np.random.default_rng(wl.seed).choice(wl.T, sample, replace=False))
    q = [oracle.quantize_fp8_rows(oracle.widen(w, "bf16")) if w is not None else (None, None)
         for w in (inp.w1, inp.w3, inp.w2)]
    ref = oracle.layer_forward_fp8(inp, q[0][0], q[0][1], q[1][0], q[1][1], q[2][0], q[2][1], tokens=tokens)
    idx = v["topk_idx"].cpu().numpy()
    same = check_routing(inp, v["logits"].cpu().numpy(), idx, v["topk_w"].cpu().numpy().astype(np.float64), ref)
    agree = check_layer_dispatch(wl, idx, same, v["counts_routed"].cpu().numpy(), v["counts_kept"].cpu().numpy(),
                                 v["offsets"].cpu().numpy(), v["dest_row"].cpu().numpy(),
                                 v["src_token"].cpu().numpy(), layer.cfg.capacity, ref)
    rows = np.arange(wl.T) if tokens is None else tokens
    rows = rows[agree[rows]]
    assert_close_out(to_np_f64(out)[rows], ref.out[rows], "bf16")


@pytest.mark.parametrize("kw", [
    dict(T=333, d=256, N=8, k=2, F=384),
    dict(T=200, d=512, N=16, k=4, F=256, gate="sigmoid", shared_F=384, sel_bias_range=0.05),
    dict(T=500, d=256, N=8, k=3, F=128, capacity_factor=0.75, zipf_s=1.2),
    dict(T=129, d=320, N=7, k=2, F=144, act="relu"),
])
def test_fp8_layer_small(kw):
    kw = dict(kw)
    wl = synth.Workload("fp8", 23, act=kw.pop("act", "swiglu"), gate=kw.pop("gate", "softmax"), dtype="bf16", **kw)
    _fp8_layer_check(synth.make_inputs(wl))


@pytest.mark.parametrize("kw", [
    dict(T=16, d=256, N=8, k=2, F=384),
    dict(T=48, d=512, N=16, k=4, F=256, gate="sigmoid", shared_F=384, sel_bias_range=0.05),
    dict(T=30, d=256, N=8, k=3, F=128, capacity_factor=0.75, zipf_s=1.2, act="relu"),
])
def test_fp8_layer_decode_sized(kw):
    kw = dict(kw)
    wl = synth.Workload("fp8d", 29, act=kw.pop("act", "swiglu"), gate=kw.pop("gate", "softmax"), dtype="bf16", **kw)
    _fp8_layer_check(synth.make_inputs(wl))


def test_fp8_layer_mixtral_decode_full():
    """The decode layer the FP8 weights are meant for, at full size, all tokens."""
    _fp8_layer_check(synth.make_inputs(synth.WORKLOADS["mixtral_decode"]))


def test_fp8_rejects_unaligned_widths():
    cfg = moe.make_config(64, 72, 4, 2, 128)      # d = 72: code rows not a multiple of 16 bytes
    ws = torch.zeros(moe.moe_workspace_size(cfg), dtype=torch.uint8, device="cuda")
    t = torch.zeros(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(moe.MoeError) as e:
        moe.moe_expert_ffn_fp8(cfg, t, t, t, t, t, t, t, t, t, ws)
    assert e.value.code == moe.MOE_ERR_UNSUPPORTED


@pytest.mark.parametrize("T,N,C,shared_F", [(64, 8, 16, 0), (200, 8, 40, 256)])
def test_fp8_expert_choice_layer(T, N, C, shared_F):
    """Expert choice with FP8 weights: every group holds exactly C rows (C <= 64: the
    one-launch decode FFN).  Reference: the oracle's routing and expert choice on its
    own scores, its FFN on its own dequantised weights, the gate the score."""
    from test_gpu_expert_choice import check_selection
    wl = synth.Workload("ec8", T + N, T=T, d=256, N=N, k=1, F=384, act="swiglu", gate="softmax", dtype="bf16",
                        shared_F=shared_F)
    inp = synth.make_inputs(wl)
    cfg = moe.make_config(T, wl.d, N, 1, wl.F, shared_F, capacity=C, routing=moe.ROUTING_EXPERT_CHOICE)
    layer = moe.MoELayer(cfg, to_dev(inp.Wg, "f32"), to_dev(inp.w1, "bf16"), to_dev(inp.w3, "bf16"),
                         to_dev(inp.w2, "bf16"), to_dev(inp.sw1, "bf16"), to_dev(inp.sw3, "bf16"),
                         to_dev(inp.sw2, "bf16"))
    layer.quantize_fp8()
    out = layer.forward(to_dev(inp.x, "bf16"))
    torch.cuda.synchronize()
    assert layer.device_status() == 0
    v = layer.views()
    x64 = oracle.widen(inp.x, "bf16")
    ec = oracle.expert_choice(oracle.router_logits(x64, inp.Wg, inp.logit_bias), C)
    chosen = v["src_token"].cpu().numpy().reshape(N, C)
    check_selection(ec.scores, chosen, C)
    q = [oracle.quantize_fp8_rows(oracle.widen(w, "bf16")) for w in (inp.w1, inp.w3, inp.w2)]
    ref = np.zeros((T, wl.d))
    if shared_F:
        ref += oracle.expert_ffn(x64, oracle.widen(inp.sw1, "bf16"), oracle.widen(inp.sw3, "bf16"),
                                 oracle.widen(inp.sw2, "bf16"), "swiglu")
    deq = lambda i, e: oracle.dequantize_fp8_rows(q[i][0][e], q[i][1][e])  # noqa: E731
    for e in range(N):
        toks = ec.chosen[e]
        ref[toks] += ec.scores[toks, e][:, None] * oracle.expert_ffn(x64[toks], deq(0, e), deq(1, e), deq(2, e),
                                                                     "swiglu")
    mine = v["dest_row"].cpu().numpy() >= 0
    theirs = np.zeros((T, N), bool)
    for e in range(N):
        theirs[ec.chosen[e], e] = True
    agree = np.all(mine == theirs, axis=1)
    assert np.sum(~agree) <= max(2, T // 100)
    assert_close_out(to_np_f64(out)[agree], ref[agree], "bf16")
