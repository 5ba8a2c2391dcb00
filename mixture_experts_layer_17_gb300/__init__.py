"""GB300-native fused Mixture-of-Experts layer (forward + backward).

The compute lives in libmoe.so (hand-written sm_103a CUDA: tcgen05/TMEM/TMA
grouped GEMMs with fused routing, SwiGLU, combine and router-gradient
epilogues).  This package holds its ctypes binding (``libmoe``), the in-tree
build (``build``) and ``MoeLayer``, which sizes and owns the workspaces with
torch and calls the C ABI.
"""

from __future__ import annotations

from typing import Dict, Optional

import torch

from . import libmoe
from .libmoe import (MoeConfig, MoeError, make_config, moe_backward,  # noqa: F401
                     moe_backward_accumulate, moe_forward, moe_gemm_bf16, moe_get_device_status, moe_launch_count,
                     moe_profile_enable, moe_profile_read, moe_profile_select, moe_route,
                     moe_status_string, moe_workspace_size)


class MoeLayer:
    """One MoE layer shape with its device workspaces.

    ``forward`` writes y and keeps the context the matching ``backward`` needs;
    weights and activations are caller-owned bf16 CUDA tensors.
    """

    def __init__(self, T: int, H: int, F: int, E: int, top_k: int, precision: str = "bf16",
                 flags: int = 0, device="cuda", max_sms: int = 0):
        self.cfg = make_config(T, H, F, E, top_k, precision, flags, max_sms)
        self.T, self.H, self.F, self.E, self.top_k = T, H, F, E, top_k
        self.device = torch.device(device)
        f, c, b = moe_workspace_size(self.cfg)
        self.fwd_ws = torch.empty(max(f, 256), dtype=torch.uint8, device=self.device)
        self.ctx = torch.empty(max(c, 256), dtype=torch.uint8, device=self.device)
        self.bwd_ws = torch.empty(max(b, 256), dtype=torch.uint8, device=self.device)

    def route(self, x, W_r, logit_bias=None, with_logits=True, stream=None) -> Dict[str, torch.Tensor]:
        T, E, k = self.T, self.E, self.top_k
        d = self.device
        out = {
            "logits": torch.empty(T, E, dtype=torch.float32, device=d) if with_logits else None,
            "topk_idx": torch.empty(T, k, dtype=torch.int32, device=d),
            "topk_w": torch.empty(T, k, dtype=torch.float32, device=d),
            "counts": torch.empty(E, dtype=torch.int32, device=d),
            "offsets": torch.empty(E + 1, dtype=torch.int32, device=d),
            "perm_token": torch.empty(T * k, dtype=torch.int32, device=d),
            "slot_row": torch.empty(T, k, dtype=torch.int32, device=d),
        }
        moe_route(self.cfg, x, W_r, logit_bias, out["logits"], out["topk_idx"], out["topk_w"],
                  out["counts"], out["offsets"], out["perm_token"], out["slot_row"],
                  self.fwd_ws, stream)
        return out

    def forward(self, x, W_r, W_gate, W_up, W_down, logit_bias=None,
                y: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
        if y is None:
            y = torch.empty(self.T, self.H, dtype=torch.bfloat16, device=self.device)
        moe_forward(self.cfg, x, W_r, logit_bias, W_gate, W_up, W_down, y, self.ctx,
                    self.fwd_ws, stream)
        return y

    def backward(self, x, W_r, W_gate, W_up, W_down, dY, grads: Optional[Dict] = None,
                 stream=None) -> Dict[str, torch.Tensor]:
        if grads is None:
            grads = {"dx": torch.empty_like(x), "dW_r": torch.empty_like(W_r),
                     "dW_gate": torch.empty_like(W_gate), "dW_up": torch.empty_like(W_up),
                     "dW_down": torch.empty_like(W_down)}
        moe_backward(self.cfg, x, W_r, W_gate, W_up, W_down, self.ctx, dY, grads["dx"],
                     grads["dW_r"], grads["dW_gate"], grads["dW_up"], grads["dW_down"],
                     self.bwd_ws, stream)
        return grads

    def prepare_weights(self, W_gate, W_up, W_down, stream=None) -> torch.Tensor:
        """MXFP8 / FP8_BWD: quantise the expert weights once (every orientation
        the GEMMs read) and let the following forward and backward calls use
        them; call again whenever the weights change.  Returns the buffer."""
        n = libmoe.moe_prepared_weights_size(self.cfg)
        self.wq = torch.empty(max(n, 256), dtype=torch.uint8, device=self.device)
        libmoe.moe_prepare_weights(self.cfg, W_gate, W_up, W_down, self.wq, stream)
        self.cfg.prepared_weights = self.wq.data_ptr()
        return self.wq

    def drop_prepared_weights(self) -> None:
        self.cfg.prepared_weights = None
        self.wq = None

    def backward_accumulate(self, x, W_r, W_gate, W_up, W_down, dY, acc: Dict[str, torch.Tensor],
                            dx: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
        """Adds the weight gradients into the fp32 tensors acc["dW_r"],
        acc["dW_gate"], acc["dW_up"], acc["dW_down"]; returns dx (bf16)."""
        if dx is None:
            dx = torch.empty_like(x)
        moe_backward_accumulate(self.cfg, x, W_r, W_gate, W_up, W_down, self.ctx, dY, dx,
                                acc["dW_r"], acc["dW_gate"], acc["dW_up"], acc["dW_down"],
                                self.bwd_ws, stream)
        return dx

    def device_status(self, which: str = "fwd", stream=None) -> int:
        ws = self.fwd_ws if which == "fwd" else self.bwd_ws
        return moe_get_device_status(ws, stream)
