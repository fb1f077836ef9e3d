"""MoELayer: resident weights + workspace around the C ABI (marshalling only).

The layer keeps every expert resident in device memory (all N experts, the
router, the optional shared expert) and one workspace; ``forward`` is one call
to moe_layer_forward on the caller's stream.
"""
from __future__ import annotations

from typing import Optional

import torch

from . import (DTYPE_BF16, MoeConfig, moe_get_device_status, moe_layer_forward, moe_layer_forward_fp8, moe_load_stats,
               moe_quantize_fp8, moe_seq_balance_loss, moe_workspace_layout, moe_workspace_size)


class MoELayer:
    def __init__(self, cfg: MoeConfig, Wg: torch.Tensor, w1: torch.Tensor, w3: Optional[torch.Tensor],
                 w2: torch.Tensor, sw1=None, sw3=None, sw2=None, logit_bias=None, sel_bias=None):
        self.cfg = cfg
        self.Wg, self.w1, self.w3, self.w2 = Wg, w1, w3, w2
        self.sw1, self.sw3, self.sw2 = sw1, sw3, sw2
        self.logit_bias, self.sel_bias = logit_bias, sel_bias
        self.device = Wg.device
        self.act_dtype = torch.bfloat16 if cfg.dtype == DTYPE_BF16 else torch.float32
        nbytes = moe_workspace_size(cfg)
        raw = torch.empty(nbytes + 256, dtype=torch.uint8, device=self.device)
        off = (-raw.data_ptr()) % 256
        self._ws_raw = raw
        self.ws = raw[off:off + nbytes]
        self.ws.zero_()
        self.layout = moe_workspace_layout(cfg)
        self._stats = torch.zeros(2 * cfg.N + 4, dtype=torch.float32, device=self.device)
        self.fp8 = None  # (w1q, w1s, w3q, w3s, w2q, w2s) once quantize_fp8 has run

    def quantize_fp8(self, stream=None):
        """Quantise the routed experts to FP8 E4M3 with one float32 scale per weight row
        (on the device); forward then runs the FP8 layer.  The shared expert stays bf16."""
        def q(w):
            if w is None:
                return None, None
            codes = torch.empty(w.shape, dtype=torch.uint8, device=self.device)
            scales = torch.empty(w.shape[:-1], dtype=torch.float32, device=self.device)
            moe_quantize_fp8(w, codes, scales, stream)
            return codes, scales
        self.fp8 = (*q(self.w1), *q(self.w3), *q(self.w2))
        return self.fp8

    # ------------------------------------------------------------------ forward
    def forward(self, x: torch.Tensor, out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
        c = self.cfg
        if out is None:
            out = torch.empty((c.T, c.d), dtype=self.act_dtype, device=self.device)
        if self.fp8 is not None:
            moe_layer_forward_fp8(c, x, self.Wg, self.logit_bias, self.sel_bias, *self.fp8, self.sw1, self.sw3,
                                  self.sw2, out, self.ws, stream)
        else:
            moe_layer_forward(c, x, self.Wg, self.logit_bias, self.sel_bias, self.w1, self.w3, self.w2,
                              self.sw1, self.sw3, self.sw2, out, self.ws, stream)
        return out

    def load_stats(self, stream=None):
        """(f [N], P [N], summary [aux, imbalance, drop_rate]) of the last forward, on device."""
        c = self.cfg
        v = self.views()
        f = self._stats[:c.N]
        P = self._stats[c.N:2 * c.N]
        summary = self._stats[2 * c.N:2 * c.N + 3]
        moe_load_stats(c, v["logits"], v["counts_routed"], v["counts_kept"], f, P, summary, self.ws, stream)
        return f, P, summary

    def seq_balance_loss(self, seq_len: int, stream=None) -> torch.Tensor:
        """Sequence-wise balance loss of the last forward (token choice), a device scalar."""
        v = self.views()
        out = self._stats[2 * self.cfg.N + 3:2 * self.cfg.N + 4]
        moe_seq_balance_loss(self.cfg, v["logits"], v["topk_idx"], seq_len, out, self.ws, stream)
        return out

    def device_status(self, stream=None) -> int:
        return moe_get_device_status(self.ws, stream)

    # ------------------------------------------------------------------ views
    def views(self):
        """Typed views of the workspace intermediates of the last forward."""
        c, L = self.cfg, self.layout
        T, N, k, d, F, Fs = c.T, c.N, c.k, c.d, c.ffn, c.shared_ffn
        ec = c.routing == 1
        C = min(c.capacity, T) if ec else 0
        rows = N * C if ec else T * k
        sl = N if ec else k
        ws = self.ws

        def view(off, n, dtype, shape):
            nb = n * torch.empty((), dtype=dtype).element_size()
            return ws[off:off + nb].view(dtype).view(shape)

        out = {
            "logits": view(L.logits, T * N, torch.float32, (T, N)),
            "topk_idx": view(L.topk_idx, T * k, torch.int32, (T, k)),
            "topk_w": view(L.topk_w, T * sl, torch.float32, (T, sl)),
            "counts_routed": view(L.counts_routed, N, torch.int32, (N,)),
            "counts_kept": view(L.counts_kept, N, torch.int32, (N,)),
            "offsets": view(L.offsets, N + 1, torch.int32, (N + 1,)),
            "dest_row": view(L.dest_row, T * sl, torch.int32, (T, sl)),
            "src_token": view(L.src_token, rows, torch.int32, (rows,)),
            "x_perm": view(L.x_perm, rows * d, self.act_dtype, (rows, d)),
            "h": view(L.h, rows * F, self.act_dtype, (rows, F)),
            "y_perm": view(L.y_perm, rows * d, self.act_dtype, (rows, d)),
        }
        if Fs:
            out["h_shared"] = view(L.h_shared, T * Fs, self.act_dtype, (T, Fs))
            out["y_shared"] = view(L.y_shared, T * d, self.act_dtype, (T, d))
        return out
