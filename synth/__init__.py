"""Seeded synthetic inputs for the sparse MoE layer, shared by the oracle and the CUDA path.

This module holds the five workload definitions (shapes, value distributions,
seeds) and the generator that turns them into arrays.  It contains none of the
layer's arithmetic (no routing, gating, dispatch or expert math): it only
produces x, the router weight, the expert weights and the per-expert bias
vectors that the workloads prescribe.

bf16 tensors are returned as numpy ``uint16`` arrays holding the raw bf16 bit
patterns; ``bf16_to_f64`` / ``bf16_to_f32`` widen them exactly.

Tensor layouts (row-major):
  x      [T, d]            activations (bf16, or f32 for the fp32 workload)
  Wg     [d, N]  f32       router weight, logits = x @ Wg
  w1, w3 [N, F, d]         expert e's W1 / W3, each F x d ("W1 x" maps d -> F)
  w2     [N, d, F]         expert e's W2, d x F (maps F -> d)
  sw1, sw3 [Fs, d], sw2 [d, Fs]   the shared expert (if any)
  logit_bias [N] f32       additive router-logit skew (Zipf workload) or None
  sel_bias   [N] f32       selection-only bias (sigmoid workload) or None
"""
from __future__ import annotations

import ctypes
import dataclasses
import math
import os
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth_gen.c")
_SO = os.path.join(_HERE, "_synth_gen.so")
_lib = None

# tensor ids of the counter-based streams
TID_X, TID_WG, TID_W1, TID_W3, TID_W2, TID_SW1, TID_SW3, TID_SW2, TID_SELB, TID_PERM = range(1, 11)


def build(force: bool = False) -> str:
    """Compile the generator with gcc into an in-tree shared object."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-pthread", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        u64, i32, dbl, vp = ctypes.c_uint64, ctypes.c_int, ctypes.c_double, ctypes.c_void_p
        for name in ("synth_normal_f32", "synth_normal_bf16"):
            fn = getattr(lib, name)
            fn.argtypes = [u64, u64, u64, u64, dbl, vp, i32]
            fn.restype = i32
        lib.synth_uniform_f32.argtypes = [u64, u64, u64, u64, dbl, dbl, vp, i32]
        lib.synth_uniform_f32.restype = i32
        lib.synth_words.argtypes = [u64, u64, u64, u64, vp]
        lib.synth_words.restype = None
        _lib = lib
    return _lib


def _threads() -> int:
    return max(1, min(64, os.cpu_count() or 1))


def normal(seed: int, tid: int, shape, std: float, dtype: str, start: int = 0) -> np.ndarray:
    """Elements start.. of stream (seed, tid) as N(0, std^2); dtype 'f32' or 'bf16' (uint16 bits)."""
    lib = _load()
    n = int(np.prod(shape))
    if dtype == "f32":
        out = np.empty(n, dtype=np.float32)
        rc = lib.synth_normal_f32(seed, tid, start, n, float(std), out.ctypes.data, _threads())
    elif dtype == "bf16":
        out = np.empty(n, dtype=np.uint16)
        rc = lib.synth_normal_bf16(seed, tid, start, n, float(std), out.ctypes.data, _threads())
    else:
        raise ValueError(dtype)
    if rc != 0:
        raise RuntimeError("synth generator failed")
    return out.reshape(shape)


def uniform(seed: int, tid: int, shape, lo: float, hi: float) -> np.ndarray:
    lib = _load()
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.float32)
    if lib.synth_uniform_f32(seed, tid, 0, n, float(lo), float(hi), out.ctypes.data, _threads()) != 0:
        raise RuntimeError("synth generator failed")
    return out.reshape(shape)


def words(seed: int, tid: int, n: int, start: int = 0) -> np.ndarray:
    lib = _load()
    out = np.empty(n, dtype=np.uint64)
    lib.synth_words(seed, tid, start, n, out.ctypes.data)
    return out


def bf16_to_f32(a: np.ndarray) -> np.ndarray:
    return (a.astype(np.uint32) << 16).view(np.float32)


def bf16_to_f64(a: np.ndarray) -> np.ndarray:
    return bf16_to_f32(a).astype(np.float64)


def f32_to_bf16(a: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 bits, nearest-even (finite inputs)."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = u + 0x7FFF + ((u >> 16) & 1)
    return (u >> 16).astype(np.uint16)


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic layer.  gate: 'softmax' | 'sigmoid'; act: 'relu' | 'swiglu'; dtype: 'f32' | 'bf16'."""
    name: str
    seed: int
    T: int
    d: int
    N: int
    k: int
    F: int
    act: str
    gate: str
    dtype: str
    shared_F: int = 0
    capacity_factor: float = 0.0   # 0: no capacity limit
    sel_bias_range: float = 0.0    # sigmoid workload: b ~ U(-r, r)
    zipf_s: float = 0.0            # skewed workload: logit skew log(p_rank), p_r ~ r^-s

    def with_tokens(self, T: int) -> "Workload":
        return dataclasses.replace(self, T=T)

    def scaled(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five layers: seed = 62*1000 + workload number.
WORKLOADS = {
    "shazeer_tiny_f32": Workload("shazeer_tiny_f32", 62001, T=256, d=512, N=8, k=2, F=1024,
                                 act="relu", gate="softmax", dtype="f32"),
    "mixtral_prefill": Workload("mixtral_prefill", 62002, T=4096, d=4096, N=8, k=2, F=14336,
                                act="swiglu", gate="softmax", dtype="bf16"),
    "mixtral_decode": Workload("mixtral_decode", 62003, T=16, d=4096, N=8, k=2, F=14336,
                               act="swiglu", gate="softmax", dtype="bf16"),
    "dsv3_finegrained": Workload("dsv3_finegrained", 62004, T=8192, d=7168, N=256, k=8, F=2048,
                                 act="swiglu", gate="sigmoid", dtype="bf16", shared_F=2048,
                                 sel_bias_range=0.05),
    "qwen3_skew_drop": Workload("qwen3_skew_drop", 62005, T=16384, d=2048, N=128, k=8, F=768,
                                act="swiglu", gate="softmax", dtype="bf16", capacity_factor=1.25,
                                zipf_s=1.2),
}
# the decode layer uses exactly the prefill layer's weights and router
_WEIGHT_SEED = {"mixtral_decode": 62002}


def zipf_logit_bias(seed: int, N: int, s: float) -> np.ndarray:
    """beta_i = log p_rank(i), p_r = r^-s / sum_r r^-s, rank from a seeded Fisher-Yates shuffle."""
    w = words(seed, TID_PERM, N)
    perm = list(range(N))
    for i in range(N - 1, 0, -1):
        j = int(w[N - 1 - i] % np.uint64(i + 1))
        perm[i], perm[j] = perm[j], perm[i]
    ranks = np.empty(N, dtype=np.int64)
    ranks[np.array(perm)] = np.arange(1, N + 1)   # expert perm[r-1] gets rank r
    p = np.array([r ** (-s) for r in range(1, N + 1)], dtype=np.float64)
    p /= p.sum()
    return np.log(p[ranks - 1]).astype(np.float32)


@dataclasses.dataclass
class LayerInputs:
    wl: Workload
    x: np.ndarray
    Wg: np.ndarray
    w1: np.ndarray
    w3: Optional[np.ndarray]
    w2: np.ndarray
    sw1: Optional[np.ndarray] = None
    sw3: Optional[np.ndarray] = None
    sw2: Optional[np.ndarray] = None
    logit_bias: Optional[np.ndarray] = None
    sel_bias: Optional[np.ndarray] = None


def make_inputs(wl: Workload, weights: bool = True) -> LayerInputs:
    """Generate every input of workload `wl` (weights=False skips the expert weights)."""
    wseed = _WEIGHT_SEED.get(wl.name, wl.seed)
    dt = wl.dtype
    x = normal(wl.seed, TID_X, (wl.T, wl.d), 1.0, dt)
    Wg = normal(wseed, TID_WG, (wl.d, wl.N), 1.0 / math.sqrt(wl.d), "f32")
    w1 = w3 = w2 = sw1 = sw3 = sw2 = None
    if weights:
        w1 = normal(wseed, TID_W1, (wl.N, wl.F, wl.d), 1.0 / math.sqrt(wl.d), dt)
        if wl.act == "swiglu":
            w3 = normal(wseed, TID_W3, (wl.N, wl.F, wl.d), 1.0 / math.sqrt(wl.d), dt)
        w2 = normal(wseed, TID_W2, (wl.N, wl.d, wl.F), 1.0 / math.sqrt(wl.F), dt)
        if wl.shared_F:
            sw1 = normal(wseed, TID_SW1, (wl.shared_F, wl.d), 1.0 / math.sqrt(wl.d), dt)
            if wl.act == "swiglu":
                sw3 = normal(wseed, TID_SW3, (wl.shared_F, wl.d), 1.0 / math.sqrt(wl.d), dt)
            sw2 = normal(wseed, TID_SW2, (wl.d, wl.shared_F), 1.0 / math.sqrt(wl.shared_F), dt)
    lb = zipf_logit_bias(wseed, wl.N, wl.zipf_s) if wl.zipf_s else None
    sb = uniform(wseed, TID_SELB, (wl.N,), -wl.sel_bias_range, wl.sel_bias_range) if wl.sel_bias_range else None
    return LayerInputs(wl, x, Wg, w1, w3, w2, sw1, sw3, sw2, lb, sb)


def expert_rows(wl: Workload, tid: int, e: int) -> np.ndarray:
    """Only expert e's slice of w1 / w3 / w2 (for per-token oracle checks at full size)."""
    wseed = _WEIGHT_SEED.get(wl.name, wl.seed)
    if tid in (TID_W1, TID_W3):
        n = wl.F * wl.d
        return normal(wseed, tid, (wl.F, wl.d), 1.0 / math.sqrt(wl.d), wl.dtype, start=e * n)
    if tid == TID_W2:
        n = wl.d * wl.F
        return normal(wseed, tid, (wl.d, wl.F), 1.0 / math.sqrt(wl.F), wl.dtype, start=e * n)
    raise ValueError(tid)
