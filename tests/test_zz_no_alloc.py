"""moe_dispatch_noalloc: the dispatch entry point for callers that cannot allocate.

Some callers -- a plug-in inside a host program that has already reserved the
GPU's memory and passes the plug-in only its inputs and outputs -- can neither
call cudaMalloc nor provide a workspace.  moe_dispatch_noalloc keeps its scratch
in a fixed array inside the library instead.  These tests check, through the C
ABI, that it produces exactly what moe_dispatch produces and what the oracle's
dispatch of the same top-k gives, on two calls in a row (the second call must not
see the first call's leftovers), and that sizes past the fixed scratch are
refused.
"""
import numpy as np
import pytest
import torch

import oracle
import sparse_mixture_experts_62_b300 as moe
import synth


def test_noalloc_rejects_sizes_beyond_its_scratch():
    # ceil(T / 128) * N = 520 * 256 > 131072 entries: refused before any launch
    cfg = moe.make_config(520 * 128, 64, 256, 8, 64)
    A = 1 << 20
    with pytest.raises(moe.MoeError) as e:
        moe.moe_dispatch_noalloc(cfg, A, A, A, A, A, A, A, A, None, 0)
    assert e.value.code == moe.MOE_ERR_UNSUPPORTED


def _dispatch_both(T, N, k, cap, seed):
    rng = np.random.default_rng(seed)
    scores = rng.standard_normal((T, N)) + 1.5 * np.linspace(2, -2, N)[None, :]
    idx = torch.from_numpy(oracle.topk(scores.astype(np.float32), k)).cuda()
    d = 128
    x = torch.from_numpy(synth.normal(seed, 1, (T, d), 1.0, "bf16").view(np.int16)).view(torch.bfloat16).cuda()
    cfg = moe.make_config(T, d, N, k, 64, capacity=cap)
    outs = []
    for noalloc in (False, True):
        i32 = lambda shape: torch.full(shape, -5, dtype=torch.int32, device="cuda")  # noqa: E731
        bufs = [i32((N,)), i32((N,)), i32((N + 1,)), i32((T, k)), i32((T * k,))]
        xp = torch.zeros((T * k, d), dtype=torch.bfloat16, device="cuda")
        if noalloc:
            status = torch.zeros(1, dtype=torch.int32, device="cuda")
            moe.moe_dispatch_noalloc(cfg, idx, x, *bufs, xp, status)
            torch.cuda.synchronize()
            assert int(status.item()) == 0
        else:
            ws = torch.zeros(moe.moe_workspace_size(cfg), dtype=torch.uint8, device="cuda")
            moe.moe_dispatch(cfg, idx, x, *bufs, xp, ws)
            torch.cuda.synchronize()
        outs.append([b.cpu() for b in bufs] + [xp.cpu()])
    return outs, idx.cpu().numpy(), x.cpu()


@pytest.mark.gpu
def test_noalloc_matches_moe_dispatch_on_two_calls_in_a_row():
    # a large call first (fills much of the fixed scratch), then a smaller one with
    # other experts: every output of both must equal moe_dispatch's exactly
    for (T, N, k, cap, seed) in [(6000, 128, 8, 300, 1), (333, 8, 2, 0, 2)]:
        (ref, got), idx, x = _dispatch_both(T, N, k, cap, seed)
        S = int(ref[2][-1])
        for a, b in zip(ref[:4], got[:4]):
            assert torch.equal(a, b)
        assert torch.equal(ref[4][:S], got[4][:S])
        assert torch.equal(ref[5][:S], got[5][:S])
        # and the dispatch definition itself, as the oracle computes it
        d = oracle.dispatch(idx, N, cap)
        assert np.array_equal(got[0].numpy(), d.counts_routed)
        assert np.array_equal(got[1].numpy(), d.counts_kept)
        assert np.array_equal(got[2].numpy(), d.offsets)
        assert np.array_equal(got[3].numpy(), d.dest_row)
        assert np.array_equal(got[4][:S].numpy(), d.src_token)
        assert torch.equal(got[5][:S], x[torch.from_numpy(d.src_token.astype(np.int64))])
