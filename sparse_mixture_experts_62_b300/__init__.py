"""Python binding of libmoe_b300: the sparse token-choice MoE FFN layer forward on B300.

Argument marshalling only.  Every step of the layer runs in the CUDA kernels of
libmoe_b300.so (built in-tree by ``python sparse_mixture_experts_62_b300/build.py``);
importing this package without that library raises ImportError -- there is no
other implementation to fall back to.  PyTorch supplies device memory and
streams: tensor arguments are passed to the C ABI as raw device pointers.

Functions carry the C names (see include/moe.h for layouts and semantics):
moe_route, moe_dispatch, moe_expert_ffn, moe_shared_ffn, moe_combine,
moe_layer_forward, moe_load_stats, moe_capacity, moe_workspace_size,
moe_workspace_layout, moe_get_device_status, moe_dispatch_noalloc.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe_b300.so")

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_CUDA, MOE_ERR_NONFINITE, MOE_ERR_TIMEOUT, \
    MOE_ERR_BOUNDS = range(7)
GATE_SOFTMAX_TOPK, GATE_SIGMOID_BIAS, GATE_SOFTMAX_FULL = 0, 1, 2
ACT_RELU, ACT_SWIGLU = 0, 1
DTYPE_F32, DTYPE_BF16 = 0, 1
ROUTING_TOKEN_CHOICE, ROUTING_EXPERT_CHOICE = 0, 1

EXPORTS = ("moe_status_string", "moe_capacity", "moe_workspace_size", "moe_workspace_layout", "moe_route",
           "moe_dispatch", "moe_expert_ffn", "moe_shared_ffn", "moe_combine", "moe_layer_forward",
           "moe_load_stats", "moe_get_device_status", "moe_dispatch_noalloc", "moe_check_wait_timeout",
           "moe_router_zloss", "moe_bias_update", "moe_ec_route", "moe_seq_balance_loss",
           "moe_backward_workspace_size", "moe_layer_backward", "moe_quantize_fp8", "moe_expert_ffn_fp8",
           "moe_layer_forward_fp8", "moe_clock_probe", "moe_expert_ffn_gather")


class MoeConfig(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("T", "d", "N", "k", "ffn", "shared_ffn", "gate", "act", "dtype", "capacity", "routing")]


class MoeWsLayout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in
                ("status", "logits", "topk_idx", "topk_w", "counts_routed", "counts_kept", "offsets", "dest_row",
                 "src_token", "x_perm", "h", "y_perm", "h_shared", "y_shared", "scratch", "total")]


class MoeError(RuntimeError):
    def __init__(self, code: int, where: str):
        super().__init__(f"{where}: {status_string(code)} ({code})")
        self.code = code


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with `python sparse_mixture_experts_62_b300/build.py`")
    lib = ctypes.CDLL(LIB_PATH)
    P = ctypes.c_void_p
    C = ctypes.POINTER(MoeConfig)
    lib.moe_status_string.argtypes = [ctypes.c_int]
    lib.moe_status_string.restype = ctypes.c_char_p
    sig = {
        "moe_capacity": [ctypes.c_double, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.POINTER(ctypes.c_int32)],
        "moe_workspace_size": [C, ctypes.POINTER(ctypes.c_size_t)],
        "moe_workspace_layout": [C, ctypes.POINTER(MoeWsLayout)],
        "moe_route": [C, P, P, P, P, P, P, P, P, P],
        "moe_dispatch": [C, P, P, P, P, P, P, P, P, P, P],
        "moe_dispatch_noalloc": [C, P, P, P, P, P, P, P, P, P, P],
        "moe_expert_ffn": [C, P, P, P, P, P, P, P, P],
        "moe_shared_ffn": [C, P, P, P, P, P, P, P],
        "moe_combine": [C, P, P, P, P, P, P],
        "moe_layer_forward": [C, P, P, P, P, P, P, P, P, P, P, P, P, P],
        "moe_load_stats": [C, P, P, P, P, P, P, P, P],
        "moe_get_device_status": [P, P, ctypes.POINTER(ctypes.c_int)],
        "moe_check_wait_timeout": [P, ctypes.c_int64, P],
        "moe_router_zloss": [C, P, P, P, P],
        "moe_seq_balance_loss": [C, P, P, ctypes.c_int32, P, P, P],
        "moe_ec_route": [C, P, P, P, P, P, P, P, P, P, P],
        "moe_backward_workspace_size": [C, ctypes.POINTER(ctypes.c_size_t)],
        "moe_layer_backward": [C] + [P] * 20,
        "moe_bias_update": [C, P, P, ctypes.c_float, P],
        "moe_quantize_fp8": [P, ctypes.c_int64, ctypes.c_int32, P, P, P],
        "moe_expert_ffn_fp8": [C] + [P] * 11,
        "moe_layer_forward_fp8": [C] + [P] * 16,
        "moe_clock_probe": [P, ctypes.c_int32, ctypes.c_int64, P],
        "moe_expert_ffn_gather": [C, P, P, P, P, P, P, P, P, P],
    }
    for name, args in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = ctypes.c_int
    return lib


_lib = _load()


def status_string(code: int) -> str:
    return _lib.moe_status_string(int(code)).decode()


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(code: int, where: str):
    if code != MOE_OK:
        raise MoeError(code, where)


def make_config(T, d, N, k, ffn, shared_ffn=0, gate=GATE_SOFTMAX_TOPK, act=ACT_SWIGLU, dtype=DTYPE_BF16,
                capacity=0, routing=ROUTING_TOKEN_CHOICE) -> MoeConfig:
    return MoeConfig(T, d, N, k, ffn, shared_ffn, gate, act, dtype, capacity, routing)


def moe_capacity(alpha: float, T: int, k: int, N: int) -> int:
    c = ctypes.c_int32(0)
    _check(_lib.moe_capacity(float(alpha), T, k, N, ctypes.byref(c)), "moe_capacity")
    return c.value


def moe_workspace_size(cfg: MoeConfig) -> int:
    n = ctypes.c_size_t(0)
    _check(_lib.moe_workspace_size(ctypes.byref(cfg), ctypes.byref(n)), "moe_workspace_size")
    return n.value


def moe_workspace_layout(cfg: MoeConfig) -> MoeWsLayout:
    L = MoeWsLayout()
    _check(_lib.moe_workspace_layout(ctypes.byref(cfg), ctypes.byref(L)), "moe_workspace_layout")
    return L


def moe_route(cfg, x, Wg, logit_bias, sel_bias, logits, topk_idx, topk_w, ws, stream=None):
    _check(_lib.moe_route(ctypes.byref(cfg), _ptr(x), _ptr(Wg), _ptr(logit_bias), _ptr(sel_bias), _ptr(logits),
                          _ptr(topk_idx), _ptr(topk_w), _ptr(ws), _stream(stream)), "moe_route")


def moe_dispatch(cfg, topk_idx, x, counts_routed, counts_kept, offsets, dest_row, src_token, x_perm, ws,
                 stream=None):
    _check(_lib.moe_dispatch(ctypes.byref(cfg), _ptr(topk_idx), _ptr(x), _ptr(counts_routed), _ptr(counts_kept),
                             _ptr(offsets), _ptr(dest_row), _ptr(src_token), _ptr(x_perm), _ptr(ws),
                             _stream(stream)), "moe_dispatch")


def moe_dispatch_noalloc(cfg, topk_idx, x, counts_routed, counts_kept, offsets, dest_row, src_token, x_perm,
                         status=None, stream=None):
    """moe_dispatch with its scratch in a fixed array inside the library: no workspace, no allocation.

    For callers that cannot allocate device memory or pass a workspace (see
    include/moe.h).  Calls that overlap on the GPU race on the shared array."""
    _check(_lib.moe_dispatch_noalloc(ctypes.byref(cfg), _ptr(topk_idx), _ptr(x), _ptr(counts_routed),
                                     _ptr(counts_kept), _ptr(offsets), _ptr(dest_row), _ptr(src_token),
                                     _ptr(x_perm), _ptr(status), _stream(stream)), "moe_dispatch_noalloc")


def moe_expert_ffn(cfg, x_perm, offsets, w1, w3, w2, y_perm, ws, stream=None):
    _check(_lib.moe_expert_ffn(ctypes.byref(cfg), _ptr(x_perm), _ptr(offsets), _ptr(w1), _ptr(w3), _ptr(w2),
                               _ptr(y_perm), _ptr(ws), _stream(stream)), "moe_expert_ffn")


def moe_expert_ffn_gather(cfg, x, src_token, offsets, w1, w3, w2, y_perm, ws, stream=None):
    _check(_lib.moe_expert_ffn_gather(ctypes.byref(cfg), _ptr(x), _ptr(src_token), _ptr(offsets), _ptr(w1),
                                      _ptr(w3), _ptr(w2), _ptr(y_perm), _ptr(ws), _stream(stream)),
           "moe_expert_ffn_gather")


def moe_shared_ffn(cfg, x, sw1, sw3, sw2, y_shared, ws, stream=None):
    _check(_lib.moe_shared_ffn(ctypes.byref(cfg), _ptr(x), _ptr(sw1), _ptr(sw3), _ptr(sw2), _ptr(y_shared),
                               _ptr(ws), _stream(stream)), "moe_shared_ffn")


def moe_combine(cfg, y_perm, dest_row, topk_w, y_shared, out, stream=None):
    _check(_lib.moe_combine(ctypes.byref(cfg), _ptr(y_perm), _ptr(dest_row), _ptr(topk_w), _ptr(y_shared),
                            _ptr(out), _stream(stream)), "moe_combine")


def moe_layer_forward(cfg, x, Wg, logit_bias, sel_bias, w1, w3, w2, sw1, sw3, sw2, out, ws, stream=None):
    _check(_lib.moe_layer_forward(ctypes.byref(cfg), _ptr(x), _ptr(Wg), _ptr(logit_bias), _ptr(sel_bias), _ptr(w1),
                                  _ptr(w3), _ptr(w2), _ptr(sw1), _ptr(sw3), _ptr(sw2), _ptr(out), _ptr(ws),
                                  _stream(stream)), "moe_layer_forward")


def moe_load_stats(cfg, logits, counts_routed, counts_kept, f, P, summary, ws, stream=None):
    _check(_lib.moe_load_stats(ctypes.byref(cfg), _ptr(logits), _ptr(counts_routed), _ptr(counts_kept), _ptr(f),
                               _ptr(P), _ptr(summary), _ptr(ws), _stream(stream)), "moe_load_stats")


def moe_ec_route(cfg, x, Wg, logit_bias, logits, scores, offsets, src_token, dest_row, ws, stream=None):
    _check(_lib.moe_ec_route(ctypes.byref(cfg), _ptr(x), _ptr(Wg), _ptr(logit_bias), _ptr(logits), _ptr(scores),
                             _ptr(offsets), _ptr(src_token), _ptr(dest_row), _ptr(ws), _stream(stream)),
           "moe_ec_route")


def moe_backward_workspace_size(cfg: MoeConfig) -> int:
    n = ctypes.c_size_t(0)
    _check(_lib.moe_backward_workspace_size(ctypes.byref(cfg), ctypes.byref(n)), "moe_backward_workspace_size")
    return n.value


def moe_layer_backward(cfg, x, Wg, w1, w3, w2, sw1, sw3, sw2, dout, dx, dWg, dw1, dw3, dw2, dsw1, dsw3, dsw2,
                       fwd_ws, bwd_ws, stream=None):
    _check(_lib.moe_layer_backward(ctypes.byref(cfg), _ptr(x), _ptr(Wg), _ptr(w1), _ptr(w3), _ptr(w2), _ptr(sw1),
                                   _ptr(sw3), _ptr(sw2), _ptr(dout), _ptr(dx), _ptr(dWg), _ptr(dw1), _ptr(dw3),
                                   _ptr(dw2), _ptr(dsw1), _ptr(dsw3), _ptr(dsw2), _ptr(fwd_ws), _ptr(bwd_ws),
                                   _stream(stream)), "moe_layer_backward")


def moe_router_zloss(cfg, logits, z_loss, ws, stream=None):
    _check(_lib.moe_router_zloss(ctypes.byref(cfg), _ptr(logits), _ptr(z_loss), _ptr(ws), _stream(stream)),
           "moe_router_zloss")


def moe_seq_balance_loss(cfg, logits, topk_idx, seq_len: int, loss, ws, stream=None):
    _check(_lib.moe_seq_balance_loss(ctypes.byref(cfg), _ptr(logits), _ptr(topk_idx), int(seq_len), _ptr(loss),
                                     _ptr(ws), _stream(stream)), "moe_seq_balance_loss")


def moe_quantize_fp8(w, q, scales, stream=None):
    """w [..., cols] bf16 (device) -> q [..., cols] uint8 E4M3 codes, scales [...] float32, one per row."""
    cols = int(w.shape[-1])
    rows = int(w.numel() // cols) if cols else 0
    _check(_lib.moe_quantize_fp8(_ptr(w), rows, cols, _ptr(q), _ptr(scales), _stream(stream)), "moe_quantize_fp8")


def moe_expert_ffn_fp8(cfg, x_perm, offsets, w1q, w1s, w3q, w3s, w2q, w2s, y_perm, ws, stream=None):
    _check(_lib.moe_expert_ffn_fp8(ctypes.byref(cfg), _ptr(x_perm), _ptr(offsets), _ptr(w1q), _ptr(w1s), _ptr(w3q),
                                   _ptr(w3s), _ptr(w2q), _ptr(w2s), _ptr(y_perm), _ptr(ws), _stream(stream)),
           "moe_expert_ffn_fp8")


def moe_layer_forward_fp8(cfg, x, Wg, logit_bias, sel_bias, w1q, w1s, w3q, w3s, w2q, w2s, sw1, sw3, sw2, out, ws,
                          stream=None):
    _check(_lib.moe_layer_forward_fp8(ctypes.byref(cfg), _ptr(x), _ptr(Wg), _ptr(logit_bias), _ptr(sel_bias),
                                      _ptr(w1q), _ptr(w1s), _ptr(w3q), _ptr(w3s), _ptr(w2q), _ptr(w2s), _ptr(sw1),
                                      _ptr(sw3), _ptr(sw2), _ptr(out), _ptr(ws), _stream(stream)),
           "moe_layer_forward_fp8")


def moe_bias_update(cfg, counts_routed, sel_bias, gamma: float, stream=None):
    _check(_lib.moe_bias_update(ctypes.byref(cfg), _ptr(counts_routed), _ptr(sel_bias), float(gamma),
                                _stream(stream)), "moe_bias_update")


def moe_check_wait_timeout(ws, limit_ns: int, stream=None):
    _check(_lib.moe_check_wait_timeout(_ptr(ws), int(limit_ns), _stream(stream)), "moe_check_wait_timeout")


def moe_clock_probe(samples, n: int, interval_ns: int, stream=None):
    _check(_lib.moe_clock_probe(_ptr(samples), int(n), int(interval_ns), _stream(stream)), "moe_clock_probe")


def moe_get_device_status(ws, stream=None) -> int:
    st = ctypes.c_int(0)
    _check(_lib.moe_get_device_status(_ptr(ws), _stream(stream), ctypes.byref(st)), "moe_get_device_status")
    return st.value


from .layer import MoELayer  # noqa: E402,F401
