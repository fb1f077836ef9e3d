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


def _fp8_ffn_case(N, counts, d, F, act, seed):
    T = int(sum(counts))
    cfg = moe.make_config(T, d, N, 1, F, 0, moe.GATE_SOFTMAX_TOPK,
                          moe.ACT_SWIGLU if act == "swiglu" else moe.ACT_RELU, moe.DTYPE_BF16, 0)
    xp = synth.normal(seed, 99, (T, d), 1.0, "bf16")
    w1 = synth.normal(seed, 3, (N, F, d), d ** -0.5, "bf16")
    w3 = synth.normal(seed, 4, (N, F, d), d ** -0.5, "bf16") if act == "swiglu" else None
    w2 = synth.normal(seed, 5, (N, d, F), F ** -0.5, "bf16")
    (q1, s1), (q2, s2) = _quantize_on_gpu(w1), _quantize_on_gpu(w2)
    q3, s3 = _quantize_on_gpu(w3) if w3 is not None else (None, None)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    ws = torch.zeros(moe.moe_workspace_size(cfg), dtype=torch.uint8, device="cuda")
    y = torch.empty((T, d), dtype=torch.bfloat16, device="cuda")
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
