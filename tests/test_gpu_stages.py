"""Per-stage parity of the CUDA path against the oracle (B300).

Each stage gets the same host-made inputs on both sides (never an output of
the GPU), so integer stages compare exactly and float stages compare within the
stated tolerance.
"""
import numpy as np
import pytest
import torch

import oracle
import sparse_mixture_experts_62_b300 as moe
import synth
from parity import assert_close_out, check_dispatch, check_routing, config_of, to_dev, to_np_f64

pytestmark = pytest.mark.gpu

BF16 = "bf16"


def _rand_bf16(shape, seed, std=1.0):
    return synth.normal(seed, 99, shape, std, "bf16")


def _ws(cfg):
    n = moe.moe_workspace_size(cfg)
    return torch.zeros(n, dtype=torch.uint8, device="cuda")


def _expert_ffn_case(N, counts, d, F, act, seed):
    T = int(sum(counts))
    rows = T  # k = 1: one row per token
    cfg = moe.make_config(T, d, N, 1, F, 0, moe.GATE_SOFTMAX_TOPK,
                          moe.ACT_SWIGLU if act == "swiglu" else moe.ACT_RELU, moe.DTYPE_BF16, 0)
    xp = _rand_bf16((rows, d), seed)
    w1 = synth.normal(seed, 3, (N, F, d), d ** -0.5, "bf16")
    w3 = synth.normal(seed, 4, (N, F, d), d ** -0.5, "bf16") if act == "swiglu" else None
    w2 = synth.normal(seed, 5, (N, d, F), F ** -0.5, "bf16")
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    ws = _ws(cfg)
    y = torch.empty((rows, d), dtype=torch.bfloat16, device="cuda")
    moe.moe_expert_ffn(cfg, to_dev(xp, BF16), torch.from_numpy(offsets).cuda(), to_dev(w1, BF16),
                       to_dev(w3, BF16), to_dev(w2, BF16), y, ws)
    assert moe.moe_get_device_status(ws) == moe.MOE_OK
    y = to_np_f64(y)
    x64 = oracle.widen(xp, "bf16")
    for e in range(N):
        r0, r1 = offsets[e], offsets[e + 1]
        if r1 == r0:
            continue
        ref = oracle.expert_ffn(x64[r0:r1], oracle.widen(w1[e], "bf16"),
                                oracle.widen(w3[e], "bf16") if w3 is not None else None,
                                oracle.widen(w2[e], "bf16"), act)
        assert_close_out(y[r0:r1], ref, "bf16", what=f"expert {e}")


def _gather_case(N, counts, T, d, F, act, seed, bad_row=None):
    """moe_expert_ffn_gather against the oracle's expert FFN on the gathered rows
    x[src_token[r]] (src_token drawn with repeats); with bad_row, that entry of
    src_token points past x: MOE_ERR_BOUNDS is recorded and every other row is
    still exact (that row's output is unspecified)."""
    rows = int(sum(counts))
    cfg = moe.make_config(T, d, N, 1, F, 0, moe.GATE_SOFTMAX_TOPK,
                          moe.ACT_SWIGLU if act == "swiglu" else moe.ACT_RELU, moe.DTYPE_BF16, 0)
    # the workspace and the row bound follow T * k routed rows: give T * k >= rows
    assert rows <= T
    x = _rand_bf16((T, d), seed)
    src = np.random.default_rng(seed).integers(0, T, rows).astype(np.int32)
    if bad_row is not None:
        src[bad_row] = T + 5
    w1 = synth.normal(seed, 3, (N, F, d), d ** -0.5, "bf16")
    w3 = synth.normal(seed, 4, (N, F, d), d ** -0.5, "bf16") if act == "swiglu" else None
    w2 = synth.normal(seed, 5, (N, d, F), F ** -0.5, "bf16")
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    ws = _ws(cfg)
    y = torch.full((T, d), 7.0, dtype=torch.bfloat16, device="cuda")
    moe.moe_expert_ffn_gather(cfg, to_dev(x, BF16), torch.from_numpy(src).cuda(), torch.from_numpy(offsets).cuda(),
                              to_dev(w1, BF16), to_dev(w3, BF16), to_dev(w2, BF16), y, ws)
    status = moe.moe_get_device_status(ws)
    assert status == (moe.MOE_OK if bad_row is None else moe.MOE_ERR_BOUNDS)
    y = to_np_f64(y)
    x64 = oracle.widen(x, "bf16")
    good = src < T
    xg = np.where(good[:, None], x64[np.minimum(src, T - 1)], 0.0)
    for e in range(N):
        r0, r1 = offsets[e], offsets[e + 1]
        if r1 == r0:
            continue
        ref = oracle.expert_ffn(xg[r0:r1], oracle.widen(w1[e], "bf16"),
                                oracle.widen(w3[e], "bf16") if w3 is not None else None,
                                oracle.widen(w2[e], "bf16"), act)
        keep = good[r0:r1]
        assert_close_out(y[r0:r1][keep], ref[keep], "bf16", what=f"expert {e}")


@pytest.mark.parametrize("act", ["swiglu", "relu"])
def test_gathered_ffn_single_ctas(act):
    """Rows gathered from x by index: ragged width (d = 192: the last k-block holds
    24 of its 64 columns), empty, one-row, swapped and multi-tile groups."""
    _gather_case(5, [0, 1, 130, 257, 64], T=600, d=192, F=320, act=act, seed=8)


@pytest.mark.parametrize("act", ["swiglu", "relu"])
def test_gathered_ffn_pair_tiles(act):
    """Groups averaging >= 512 rows (CTA pairs): both CTAs of a pair gather their rows."""
    _gather_case(3, [600, 1100, 301], T=2100, d=320, F=520, act=act, seed=9)


def test_gathered_ffn_flags_a_row_index_past_x():
    _gather_case(2, [70, 90], T=200, d=128, F=128, act="swiglu", seed=10, bad_row=75)


def test_tc_gemm_single_tile():
    """One expert, 128 rows, K = 64: a single tile and a single K block."""
    _expert_ffn_case(1, [128], d=64, F=128, act="swiglu", seed=1)


@pytest.mark.parametrize("act", ["swiglu", "relu"])
def test_tc_gemm_ragged_groups(act):
    """Empty, single-row and multi-tile groups; F and d not multiples of the tile width."""
    _expert_ffn_case(5, [0, 1, 130, 257, 64], d=192, F=320, act=act, seed=2)


@pytest.mark.parametrize("act", ["swiglu", "relu"])
def test_tc_gemm_pair_tiles(act):
    """Groups averaging >= 512 rows run on CTA pairs (256-row tiles): a last pair
    tile with rows for one CTA only, F and d not multiples of the tile width."""
    _expert_ffn_case(3, [600, 1100, 301], d=320, F=520, act=act, seed=4)


@pytest.mark.parametrize("act", ["swiglu", "relu"])
def test_tc_gemm_long_k_mixed_groups(act):
    """K >= 1024 with groups of 64 to 513 rows: tiles of one row past a 128-row
    multiple, a group of at most 128 rows (swapped operands), an empty group, widths
    not multiples of the tile."""
    _expert_ffn_case(5, [300, 0, 129, 64, 513], d=1024, F=1088, act=act, seed=6)


def test_tc_gemm_many_experts_deep_k():
    _expert_ffn_case(16, [3, 40, 0, 200, 129, 1, 77, 128, 256, 5, 0, 9, 64, 300, 17, 2], d=1024, F=512,
                     act="swiglu", seed=3)


def test_bad_offsets_are_flagged_not_written():
    cfg = moe.make_config(64, 64, 2, 1, 128)
    ws = _ws(cfg)
    xp = torch.zeros((64, 64), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((2, 128, 64), dtype=torch.bfloat16, device="cuda")
    w2 = torch.zeros((2, 64, 128), dtype=torch.bfloat16, device="cuda")
    y = torch.full((64, 64), 7.0, dtype=torch.bfloat16, device="cuda")
    offsets = torch.tensor([0, 10, 1000], dtype=torch.int32, device="cuda")  # past the 64 rows
    moe.moe_expert_ffn(cfg, xp, offsets, w, w, w2, y, ws)
    assert moe.moe_get_device_status(ws) == moe.MOE_ERR_BOUNDS
    assert torch.all(y[10:] == 7.0)


ROUTER_CASES = [
    dict(T=333, d=256, N=8, k=2, gate="softmax"),
    dict(T=200, d=512, N=256, k=8, gate="sigmoid", sel_bias_range=0.05),
    dict(T=130, d=7168, N=256, k=8, gate="sigmoid", sel_bias_range=0.05),
    dict(T=257, d=2048, N=128, k=8, gate="softmax", zipf_s=1.2),
    dict(T=64, d=64, N=5, k=5, gate="softmax"),
    dict(T=64, d=64, N=1, k=1, gate="softmax"),
    dict(T=100, d=512, N=8, k=2, gate="softmax", dtype="f32", act="relu"),
    dict(T=300, d=256, N=16, k=4, gate="softmax_full"),
    dict(T=64, d=128, N=64, k=1, gate="softmax"),                        # Switch-style top-1
    # few experts, long K, every gate (bf16: the tensor-core route)
    dict(T=200, d=4096, N=8, k=2, gate="softmax_full"),
    dict(T=1000, d=4096, N=8, k=2, gate="sigmoid", sel_bias_range=0.05),
    dict(T=97, d=1000, N=4, k=2, gate="softmax", zipf_s=1.2),
    # one-launch CUDA-core route (float32 x, N = 4 or 8, more than 64 tokens): long
    # K, a K range ending inside a warp's share (d = 1000), a ragged last CTA, gates
    dict(T=65, d=4096, N=8, k=1, gate="softmax", dtype="f32", act="relu"),
    dict(T=97, d=1000, N=4, k=2, gate="sigmoid", sel_bias_range=0.05, dtype="f32", act="relu"),
    dict(T=300, d=512, N=8, k=3, gate="softmax_full", dtype="f32", act="relu"),
]


@pytest.mark.parametrize("kw", ROUTER_CASES)
def test_route_parity(kw):
    kw = dict(kw)
    wl = synth.Workload("r", 11, F=64, act=kw.pop("act", "swiglu"), dtype=kw.pop("dtype", "bf16"), **kw)
    inp = synth.make_inputs(wl, weights=False)
    ref = oracle.layer_forward(synth.LayerInputs(wl, inp.x, inp.Wg, None, None, None,
                                                 logit_bias=inp.logit_bias, sel_bias=inp.sel_bias),
                               tokens=np.array([], dtype=np.int64))
    cfg = config_of(wl)
    ws = _ws(cfg)
    z = torch.empty((wl.T, wl.N), dtype=torch.float32, device="cuda")
    idx = torch.empty((wl.T, wl.k), dtype=torch.int32, device="cuda")
    w = torch.empty((wl.T, wl.k), dtype=torch.float32, device="cuda")
    f32 = lambda a: None if a is None else to_dev(a, "f32")  # noqa: E731
    moe.moe_route(cfg, to_dev(inp.x, wl.dtype), f32(inp.Wg), f32(inp.logit_bias), f32(inp.sel_bias), z, idx, w, ws)
    assert moe.moe_get_device_status(ws) == moe.MOE_OK
    check_routing(inp, z.cpu().numpy(), idx.cpu().numpy(), w.cpu().numpy().astype(np.float64), ref)


def test_route_flags_nonfinite_logits():
    wl = synth.Workload("r", 12, T=40, d=64, N=8, k=2, F=64, act="swiglu", gate="softmax", dtype="bf16")
    inp = synth.make_inputs(wl, weights=False)
    cfg = config_of(wl)
    ws = _ws(cfg)
    x = to_dev(inp.x, "bf16")
    x[3, 5] = float("nan")
    z = torch.empty((40, 8), device="cuda")
    idx = torch.empty((40, 2), dtype=torch.int32, device="cuda")
    w = torch.empty((40, 2), device="cuda")
    moe.moe_route(cfg, x, to_dev(inp.Wg, "f32"), None, None, z, idx, w, ws)
    assert moe.moe_get_device_status(ws) == moe.MOE_ERR_NONFINITE
    assert moe.moe_get_device_status(ws) == moe.MOE_OK  # reading clears it


@pytest.mark.parametrize("T,N,k,cap,dtype", [(333, 8, 2, 0, "bf16"), (1000, 16, 4, 150, "bf16"),
                                             (128, 256, 8, 3, "bf16"), (97, 8, 2, 20, "bf16"),
                                             (4096, 128, 8, 200, "bf16"), (257, 5, 5, 0, "f32"),
                                             (1, 4, 2, 0, "bf16"), (300, 3, 1, 1, "bf16"),
                                             (5000, 256, 8, 0, "bf16")])
def test_dispatch_parity(T, N, k, cap, dtype):
    rng = np.random.default_rng(T * 7 + N)
    scores = rng.standard_normal((T, N)) + 1.5 * np.linspace(2, -2, N)[None, :]
    idx = oracle.topk(scores.astype(np.float32), k)
    d = 64
    x = synth.normal(5, 1, (T, d), 1.0, dtype)
    cfg = moe.make_config(T, d, N, k, 64, 0, 0, 1, moe.DTYPE_BF16 if dtype == "bf16" else moe.DTYPE_F32, cap)
    ws = _ws(cfg)
    dev = lambda shape: torch.full(shape, -7, dtype=torch.int32, device="cuda")  # noqa: E731
    cr, ck, off, dr, st = dev((N,)), dev((N,)), dev((N + 1,)), dev((T, k)), dev((T * k,))
    xt = to_dev(x, dtype)
    xp = torch.zeros((T * k, d), dtype=xt.dtype, device="cuda")
    moe.moe_dispatch(cfg, torch.from_numpy(idx).cuda(), xt, cr, ck, off, dr, st, xp, ws)
    assert moe.moe_get_device_status(ws) == moe.MOE_OK
    ref = check_dispatch(synth.Workload("d", 0, T, d, N, k, 64, "swiglu", "softmax", dtype), idx,
                         cr.cpu().numpy(), ck.cpu().numpy(), off.cpu().numpy(), dr.cpu().numpy(), st.cpu().numpy(),
                         cap)
    S = int(ref.offsets[-1])
    # the permuted rows are exact copies
    assert torch.equal(xp[:S].cpu(), xt.cpu()[torch.from_numpy(ref.src_token.astype(np.int64))])


@pytest.mark.parametrize("T", [300, 100])  # several 128-token chunks; one chunk (a single fused kernel)
def test_dispatch_repeated_expert_is_flagged_and_dropped(T):
    """A top-k input that lists an expert twice for one token: the repeat is not
    counted and gets no row, the device status reports MOE_ERR_INVALID_ARG, and
    the rest is the dispatch of the input without the repeat."""
    N, k, d = 8, 3, 64
    rng = np.random.default_rng(9)
    idx = np.stack([rng.permutation(N)[:k] for _ in range(T)]).astype(np.int32)
    idx[17, 2] = idx[17, 0]
    idx[T - 3, 1] = idx[T - 3, 0]
    cfg = moe.make_config(T, d, N, k, 64)
    ws = _ws(cfg)
    x = to_dev(synth.normal(5, 1, (T, d), 1.0, "bf16"), "bf16")
    dev = lambda shape: torch.full(shape, -7, dtype=torch.int32, device="cuda")  # noqa: E731
    cr, ck, off, dr, st = dev((N,)), dev((N,)), dev((N + 1,)), dev((T, k)), dev((T * k,))
    xp = torch.zeros((T * k, d), dtype=torch.bfloat16, device="cuda")
    moe.moe_dispatch(cfg, torch.from_numpy(idx).cuda(), x, cr, ck, off, dr, st, xp, ws)
    assert moe.moe_get_device_status(ws) == moe.MOE_ERR_INVALID_ARG
    dest = dr.cpu().numpy()
    assert dest[17, 2] == -1 and dest[T - 3, 1] == -1
    # everything else: the oracle's dispatch with the repeats removed by hand
    counts = np.bincount(idx.ravel(), minlength=N)
    counts[idx[17, 0]] -= 1
    counts[idx[T - 3, 0]] -= 1
    assert np.array_equal(cr.cpu().numpy(), counts)
    offn = off.cpu().numpy()
    assert np.array_equal(offn, np.concatenate([[0], np.cumsum(counts)]))
    S = int(counts.sum())
    src = st.cpu().numpy()[:S]
    for e in range(N):
        toks = [t for t in range(T) if e in idx[t].tolist()]
        assert np.array_equal(src[offn[e]:offn[e + 1]], toks)
    assert torch.equal(xp[:S].cpu(), x.cpu()[torch.from_numpy(src.astype(np.int64))])


@pytest.mark.parametrize("dtype,shared", [("bf16", False), ("bf16", True), ("f32", False)])
def test_combine_parity(dtype, shared):
    T, k, d = 300, 4, 256
    rows = 900
    rng = np.random.default_rng(5)
    y = synth.normal(7, 1, (rows, d), 1.0, dtype)
    ysh = synth.normal(7, 2, (T, d), 1.0, dtype) if shared else None
    dest = rng.permutation(T * k)[: T * k].reshape(T, k) % (rows + 200)
    dest = np.where(dest >= rows, -1, dest).astype(np.int32)
    w = rng.random((T, k)).astype(np.float32)
    cfg = moe.make_config(T, d, 8, k, 64, 0, 0, 1, moe.DTYPE_BF16 if dtype == "bf16" else moe.DTYPE_F32, 0)
    out = torch.empty((T, d), dtype=torch.bfloat16 if dtype == "bf16" else torch.float32, device="cuda")
    moe.moe_combine(cfg, to_dev(y, dtype), torch.from_numpy(dest).cuda(), torch.from_numpy(w).cuda(),
                    to_dev(ysh, dtype) if shared else None, out)
    ref = oracle.combine(oracle.widen(y, dtype), dest, w.astype(np.float64),
                         oracle.widen(ysh, dtype) if shared else None)
    assert_close_out(to_np_f64(out), ref, dtype)
    if dtype == "f32":
        assert np.max(np.abs(to_np_f64(out) - ref)) <= 1e-5 * np.max(np.abs(ref))


@pytest.mark.parametrize("gate,T,N,k", [("softmax", 1000, 8, 2), ("sigmoid", 700, 256, 8), ("softmax", 3000, 128, 8)])
def test_load_stats_parity(gate, T, N, k):
    rng = np.random.default_rng(T)
    z = (rng.standard_normal((T, N)) * 2).astype(np.float32)
    idx = oracle.topk(z, k)
    cap = max(1, T * k // N // 2)
    disp = oracle.dispatch(idx, N, cap)
    ref = oracle.load_stats(z, gate, disp, k)
    cfg = moe.make_config(T, 64, N, k, 64, 0, moe.GATE_SIGMOID_BIAS if gate == "sigmoid" else 0, 1, 1, cap)
    ws = _ws(cfg)
    f = torch.empty(N, device="cuda")
    P = torch.empty(N, device="cuda")
    summ = torch.empty(3, device="cuda")
    moe.moe_load_stats(cfg, torch.from_numpy(z).cuda(), torch.from_numpy(disp.counts_routed).cuda(),
                       torch.from_numpy(disp.counts_kept).cuda(), f, P, summ, ws)
    assert np.array_equal(f.cpu().numpy(), ref.f.astype(np.float32))
    assert np.max(np.abs(P.cpu().numpy() - ref.P)) < 1e-6
    s = summ.cpu().numpy().astype(np.float64)
    assert s[0] == pytest.approx(ref.aux, rel=1e-5)
    assert s[1] == pytest.approx(ref.imbalance, rel=1e-6)
    assert s[2] == pytest.approx(ref.drop_rate, rel=1e-6, abs=1e-7)


def test_device_wait_gives_up_and_reports_timeout():
    """A pipeline wait that nothing can end returns after its limit with
    MOE_ERR_TIMEOUT in the status word; the context stays usable."""
    cfg = moe.make_config(8, 64, 2, 1, 64)
    ws = _ws(cfg)
    moe.moe_check_wait_timeout(ws, 20_000_000)  # 20 ms
    assert moe.moe_get_device_status(ws) == moe.MOE_ERR_TIMEOUT
    assert moe.moe_get_device_status(ws) == moe.MOE_OK
    x = torch.ones(4, device="cuda")
    assert float((x * 2).sum().item()) == 8.0  # the GPU still works


@pytest.mark.parametrize("T,N", [(1000, 8), (333, 256), (4096, 128), (1, 4)])
def test_router_zloss_parity(T, N):
    rng = np.random.default_rng(T + N)
    z = (rng.standard_normal((T, N)) * 3 + 1).astype(np.float32)
    cfg = moe.make_config(T, 64, N, 1, 64)
    ws = _ws(cfg)
    out = torch.zeros(1, device="cuda")
    moe.moe_router_zloss(cfg, torch.from_numpy(z).cuda(), out, ws)
    ref = oracle.router_z_loss(z)
    assert abs(float(out.item()) - ref) <= 1e-5 * ref


def test_bias_update_parity():
    T, N, k = 1000, 16, 2
    rng = np.random.default_rng(3)
    counts = rng.multinomial(T * k, np.ones(N) / N).astype(np.int32)
    counts[3] = T * k // N  # exactly the mean: unchanged
    b = rng.uniform(-0.05, 0.05, N).astype(np.float32)
    cfg = moe.make_config(T, 64, N, k, 64, gate=moe.GATE_SIGMOID_BIAS)
    bd = torch.from_numpy(b.copy()).cuda()
    gamma = float(np.float32(0.001))  # the C ABI takes gamma as float32: give the oracle that value
    moe.moe_bias_update(cfg, torch.from_numpy(counts).cuda(), bd, gamma)
    ref = oracle.bias_update(b, counts.astype(np.int64), T, k, gamma)
    assert np.array_equal(bd.cpu().numpy(), ref)


def _skewed_topk(rng, T, N, k):
    """Distinct experts per token, drawn with Zipf-like preferences (host-made input)."""
    keys = np.log(1.0 / np.arange(1, N + 1) ** 1.1)[None, :] + rng.gumbel(size=(T, N))
    return np.argsort(-keys, axis=1, kind="stable")[:, :k].astype(np.int32)


@pytest.mark.parametrize("gate,T,N,k,seq_lens", [
    ("softmax", 1000, 8, 2, [1, 5, 31, 32, 33, 100, 256, 999, 1000, 5000]),
    ("sigmoid", 777, 256, 8, [1, 7, 32, 64, 300, 777]),
    ("softmax_full", 4096, 128, 8, [4096, 1024, 96, 3]),
    ("softmax", 1, 4, 2, [1, 8]),
])
def test_seq_balance_loss_parity(gate, T, N, k, seq_lens):
    rng = np.random.default_rng(T + N + k)
    z = (rng.standard_normal((T, N)) * 1.5).astype(np.float32)
    idx = _skewed_topk(rng, T, N, k)
    g = {"softmax": moe.GATE_SOFTMAX_TOPK, "sigmoid": moe.GATE_SIGMOID_BIAS, "softmax_full": moe.GATE_SOFTMAX_FULL}
    cfg = moe.make_config(T, 64, N, k, 64, 0, g[gate])
    ws = _ws(cfg)
    zd, idd = torch.from_numpy(z).cuda(), torch.from_numpy(idx).cuda()
    out = torch.full((1,), float("nan"), device="cuda")
    for L in seq_lens:
        moe.moe_seq_balance_loss(cfg, zd, idd, L, out, ws)
        ref = oracle.sequence_balance_loss(z, idx, "sigmoid" if gate == "sigmoid" else "softmax", L)
        got = float(out.item())
        assert abs(got - ref) <= 1e-5 * abs(ref) + 1e-7, (L, got, ref)
    assert moe.moe_get_device_status(ws) == moe.MOE_OK
    # deterministic
    moe.moe_seq_balance_loss(cfg, zd, idd, seq_lens[0], out, ws)
    a = out.clone()
    moe.moe_seq_balance_loss(cfg, zd, idd, seq_lens[0], out, ws)
    assert torch.equal(a, out)


def test_seq_balance_loss_flags_bad_indices():
    T, N, k = 100, 8, 2
    z = np.zeros((T, N), np.float32)
    idx = np.tile(np.array([[0, 1]], np.int32), (T, 1))
    idx[40, 1] = 8  # out of range
    cfg = moe.make_config(T, 64, N, k, 64)
    ws = _ws(cfg)
    out = torch.zeros(1, device="cuda")
    for L in (10, 50):
        moe.moe_seq_balance_loss(cfg, torch.from_numpy(z).cuda(), torch.from_numpy(idx).cuda(), L, out, ws)
        assert moe.moe_get_device_status(ws) == moe.MOE_ERR_BOUNDS
