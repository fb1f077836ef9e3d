"""The shared input generator: stream definition, distributions, slicing (no GPU)."""
import math

import numpy as np

import synth

MASK = (1 << 64) - 1
GAMMA = 0x9E3779B97F4A7C15


def _mix(z):
    z ^= z >> 30
    z = (z * 0xBF58476D1CE4E5B9) & MASK
    z ^= z >> 27
    z = (z * 0x94D049BB133111EB) & MASK
    return z ^ (z >> 31)


def test_stream_is_splitmix64():
    """word n of (seed, id) is SplitMix64 output n from the state key(seed, id)."""
    seed, tid = 62002, 3
    key = _mix((seed * GAMMA + _mix((tid + GAMMA) & MASK)) & MASK)
    ref = [_mix((key + (n + 1) * GAMMA) & MASK) for n in range(1000, 1010)]
    assert synth.words(seed, tid, 10, start=1000).tolist() == ref


def test_normal_moments_and_bf16_rounding():
    a = synth.normal(5, 1, (1 << 20,), 2.0, "f32").astype(np.float64)
    assert abs(a.mean()) < 0.01 and abs(a.std() - 2.0) < 0.01
    b = synth.normal(5, 1, (1 << 20,), 2.0, "bf16")
    assert np.array_equal(b, synth.f32_to_bf16(a.astype(np.float32)))
    # round-to-nearest-even on exact halfway cases
    halfway = np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8], dtype=np.float32)
    assert synth.bf16_to_f32(synth.f32_to_bf16(halfway)).tolist() == [1.0, 1.0 + 2 * 2.0 ** -7]


def test_slices_and_determinism():
    full = synth.normal(9, 4, (3, 5, 7), 1.0, "bf16")
    part = synth.normal(9, 4, (5, 7), 1.0, "bf16", start=35)
    assert np.array_equal(full[1], part)
    assert np.array_equal(full, synth.normal(9, 4, (3, 5, 7), 1.0, "bf16"))
    wl = synth.WORKLOADS["shazeer_tiny_f32"].scaled(T=8, N=3, d=16, F=24)
    inp = synth.make_inputs(wl)
    assert np.array_equal(synth.expert_rows(wl, synth.TID_W1, 2), inp.w1[2])
    assert np.array_equal(synth.expert_rows(wl, synth.TID_W2, 1), inp.w2[1])


def test_workload_distributions():
    wl = synth.WORKLOADS["dsv3_finegrained"].scaled(T=64, d=256, N=32, F=64, shared_F=64)
    inp = synth.make_inputs(wl)
    assert inp.sel_bias.min() >= -0.05 and inp.sel_bias.max() < 0.05
    w2 = synth.bf16_to_f32(inp.w2).astype(np.float64)
    assert abs(w2.std() - 1 / math.sqrt(64)) < 0.01
    zipf = synth.zipf_logit_bias(62005, 128, 1.2)
    p = np.exp(zipf.astype(np.float64))
    assert abs(p.sum() - 1.0) < 1e-5
    ranks = np.argsort(-p)
    assert sorted(ranks.tolist()) == list(range(128))
    expect = np.array([r ** -1.2 for r in range(1, 129)])
    assert np.allclose(np.sort(p)[::-1], expect / expect.sum(), rtol=1e-5)
