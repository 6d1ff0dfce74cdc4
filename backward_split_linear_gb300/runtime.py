"""Owning wrapper around a libzb stage: device weights, float32 accumulators, workspace.

Marshalling and ownership only; every step runs in libzb's kernels.
"""
from __future__ import annotations

import numpy as np
import torch

from . import binding as zb

# parameter name -> accumulator field of zb_layer_params
GRAD_FIELD = {"w_qkv": "dw_qkv", "w_o": "dw_o", "w_gu": "dw_gu", "w_down": "dw_down",
              "gamma1": "dgamma1", "gamma2": "dgamma2", "w": "dw"}


def bf16_from_bits(bits, device="cuda"):
    """uint16 bf16 bit patterns (numpy) -> torch.bfloat16 tensor on `device`."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    return t.to(device)


def bits_from_bf16(t):
    """torch.bfloat16 tensor -> uint16 numpy bit patterns (host)."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def f64_from_bf16(t):
    return (bits_from_bf16(t).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


class Stage:
    """One pipeline stage on the current CUDA device."""

    def __init__(self, kind, n_layers, hidden, ffn, n_heads=0, n_kv_heads=0, head_dim=0, eps=1e-5,
                 max_tokens=128, max_inflight=1, params=None, device="cuda", attention="standin", seq_len=0):
        self.kind = kind
        self.hidden, self.ffn = hidden, ffn
        self.out_dim = ffn if kind == "linear" else hidden
        self.cfg = zb.make_config(kind, n_layers, hidden, ffn, n_heads, n_kv_heads, head_dim, eps,
                                  max_tokens, max_inflight, attention, seq_len)
        nbytes = zb.zb_stage_workspace_bytes(self.cfg)
        if nbytes == 0:
            raise zb.ZBError(-1, "zb_stage_workspace_bytes (invalid config)")
        self.workspace = torch.empty(nbytes + 256, dtype=torch.uint8, device=device)
        off = (-self.workspace.data_ptr()) % 256
        self.ws_ptr = self.workspace.data_ptr() + off
        self.ws_bytes = nbytes
        self.params = params  # list of dicts name -> device tensor
        self.grads = []
        layers = []
        for prm in params:
            d, g = {}, {}
            for name, t in prm.items():
                d[name] = t
                acc = torch.zeros(t.shape, dtype=torch.float32, device=device)
                g[name] = acc
                d[GRAD_FIELD[name]] = acc
            layers.append(d)
            self.grads.append(g)
        self.handle = zb.zb_stage_create(self.cfg, layers, self.ws_ptr, self.ws_bytes)

    @staticmethod
    def from_synth(kind, n_layers, hidden, ffn, n_heads=0, n_kv_heads=0, head_dim=0, eps=1e-5,
                   max_tokens=128, max_inflight=1, params_bits=None, device="cuda", attention="standin", seq_len=0):
        params = []
        for layer in params_bits:
            params.append({k: (bf16_from_bits(v, device) if v.dtype == np.uint16
                               else torch.from_numpy(v).to(device)) for k, v in layer.items()})
        return Stage(kind, n_layers, hidden, ffn, n_heads, n_kv_heads, head_dim, eps, max_tokens,
                     max_inflight, params, device, attention, seq_len)

    def zero_grads(self):
        for g in self.grads:
            for t in g.values():
                t.zero_()

    def forward(self, mb, x, y, stream=None):
        zb.zb_stage_forward(self.handle, mb, x, x.shape[0], y, stream)

    def backward_input(self, mb, dy, dx, stream=None):
        zb.zb_backward_input(self.handle, mb, dy, dx, stream)

    def backward_weight(self, mb, stream=None):
        zb.zb_backward_weight(self.handle, mb, stream)

    def flush(self, stream=None):
        zb.zb_wgrad_flush(self.handle, stream)

    def sync(self, stream=None):
        zb.zb_stage_sync(self.handle, stream)

    def stats(self):
        return zb.zb_stage_stats(self.handle)

    def stash(self, mb, layer, name):
        """A view (no copy) of one stashed tensor of microbatch `mb`, layer `layer`, inside the
        workspace: bf16 [rows, cols] or float32 [rows, cols].  Valid until the microbatch's W."""
        ptr, rows, cols, eb = zb.zb_stage_stash_view(self.handle, mb, layer, name)
        off = ptr - self.workspace.data_ptr()
        nbytes = rows * cols * eb
        if off < 0 or off + nbytes > self.workspace.numel():
            raise zb.ZBError(-1, "zb_stage_stash_view (address outside the workspace)")
        raw = self.workspace[off:off + nbytes]
        return raw.view(torch.bfloat16 if eb == 2 else torch.float32).view(rows, cols)

    def set_tracing(self, enable):
        zb.zb_stage_set_tracing(self.handle, enable)

    def read_tracing(self, reset=True):
        return zb.zb_stage_read_tracing(self.handle, reset)

    def close(self):
        if self.handle:
            zb.zb_stage_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
