"""A thin holder that turns torch weight tensors into the C structs of
``include/moe.h`` and calls the library.  Marshalling only: no arithmetic of
the layer happens here.
"""

from __future__ import annotations

from typing import Optional

import torch

from . import binding as B
from .synth import (FMT_BF16, FMT_FP8_B128, FMT_NVFP4, ROUTE_SIGMOID_BIAS, LayerConfig,
                    LayerWeights, QMatT)

_FMT = {FMT_BF16: B.MOE_W_BF16, FMT_FP8_B128: B.MOE_W_FP8_B128, FMT_NVFP4: B.MOE_W_NVFP4}
_PATH = {"auto": B.MOE_PATH_AUTO, "token_major": B.MOE_PATH_TOKEN_MAJOR,
         "grouped": B.MOE_PATH_GROUPED}


def make_config(cfg: LayerConfig, path: str = "auto", experts=None,
                exclude_shared: bool = False, accumulate: bool = False) -> B.moe_config_t:
    """``experts`` = (begin, end): the routed experts this call holds (expert
    parallelism; None = all).  ``exclude_shared``: leave the shared expert out.
    ``accumulate``: add the layer's output into ``out``."""
    c = B.moe_config_t()
    c.hidden, c.num_experts, c.top_k = cfg.hidden, cfg.num_experts, cfg.top_k
    c.inter, c.shared_inter = cfg.inter, cfg.shared_inter
    c.routing = B.MOE_ROUTE_SIGMOID_BIAS if cfg.routing == ROUTE_SIGMOID_BIAS else B.MOE_ROUTE_SOFTMAX
    c.norm_topk_prob = 1 if cfg.norm_topk_prob else 0
    c.routed_scaling_factor = cfg.routed_scaling_factor
    c.expert_fmt = _FMT[cfg.expert_fmt]
    c.path = _PATH[path]
    c.rms_norm_eps = cfg.rms_norm_eps
    if experts is not None:
        c.expert_begin, c.expert_end = int(experts[0]), int(experts[1])
    c.exclude_shared = 1 if exclude_shared else 0
    c.accumulate = 1 if accumulate else 0
    c.router_fmt = _FMT[cfg.router_fmt]
    return c


def _qmat(q: Optional[QMatT]) -> B.moe_qmat_t:
    m = B.moe_qmat_t()
    if q is None:
        return m
    m.w = q.w.data_ptr()
    m.scale = q.scale.data_ptr() if q.scale is not None else None
    m.scale2 = q.scale2.data_ptr() if q.scale2 is not None else None
    return m


def make_weights(lw: LayerWeights) -> B.moe_weights_t:
    w = B.moe_weights_t()
    w.router_w = lw.router_w.data_ptr()
    w.correction_bias = lw.correction_bias.data_ptr() if lw.correction_bias is not None else None
    w.gate, w.up, w.down = _qmat(lw.gate), _qmat(lw.up), _qmat(lw.down)
    w.sh_gate, w.sh_up, w.sh_down = _qmat(lw.sh_gate), _qmat(lw.sh_up), _qmat(lw.sh_down)
    w.shared_gate_w = lw.shared_gate_w.data_ptr() if lw.shared_gate_w is not None else None
    w.pre_expert_norm_w = (lw.pre_expert_norm_w.data_ptr() if lw.pre_expert_norm_w is not None
                           else None)
    w.router_q = _qmat(lw.router_q)
    return w


class MoeLayer:
    """One MoE layer on the current CUDA device.

    ``forward(x)`` runs router, top-k, experts and blend through ``moe_forward``
    on the current torch stream and returns ``(out, idx, w)``.

    Expert parallelism: with ``experts=(begin, end)`` the weight stacks of
    ``weights`` hold only those experts (``synth.expert_slice``) and the output
    is this rank's partial; ``exclude_shared`` leaves the shared expert out;
    ``accumulate`` adds the result into ``out`` (which must then be given).
    """

    def __init__(self, weights: LayerWeights, max_tokens: int, path: str = "auto",
                 experts=None, exclude_shared: bool = False, accumulate: bool = False):
        self.weights = weights
        self.cfg = weights.cfg
        self.accumulate = accumulate
        self.c_cfg = make_config(self.cfg, path, experts, exclude_shared, accumulate)
        self.c_w = make_weights(weights)
        self.ws_bytes = B.moe_workspace_bytes(self.c_cfg, max_tokens)
        if self.ws_bytes == 0:
            raise B.MoeError("invalid layer configuration")
        dev = weights.router_w.device
        # The control block (first 256 bytes) must start at zero; calls keep it zero.
        self.ws = torch.zeros(self.ws_bytes, dtype=torch.uint8, device=dev)
        self.max_tokens = max_tokens

    def forward(self, x: torch.Tensor, out=None, idx=None, w=None, stream=None,
                routing: bool = True):
        """``routing=False``: do not return the routing (idx and w are None), so
        a call that holds no routed expert can skip it."""
        n = x.shape[0]
        k = self.cfg.top_k
        dev = x.device
        if out is None:
            if self.accumulate:
                raise ValueError("accumulate needs out")
            out = torch.empty(n, self.cfg.hidden, dtype=torch.bfloat16, device=dev)
        if routing:
            idx = torch.empty(n, k, dtype=torch.int32, device=dev) if idx is None else idx
            w = torch.empty(n, k, dtype=torch.float32, device=dev) if w is None else w
        B.check(B.moe_forward(self.c_cfg, self.c_w, x, n, out, idx, w, self.ws, self.ws_bytes,
                              stream))
        return out, idx, w

    def device_error(self, stream=None) -> int:
        """Reads and clears the workspace's device error word (syncs the stream)."""
        s, v = B.moe_workspace_check(self.ws, self.ws_bytes, stream)
        B.check(s)
        return v

    def route(self, x: torch.Tensor, logits: bool = True, stream=None):
        n, k, E = x.shape[0], self.cfg.top_k, self.cfg.num_experts
        idx = torch.empty(n, k, dtype=torch.int32, device=x.device)
        w = torch.empty(n, k, dtype=torch.float32, device=x.device)
        lg = torch.empty(n, E, dtype=torch.float32, device=x.device) if logits else None
        B.check(B.moe_route(self.c_cfg, self.c_w, x, n, idx, w, lg, self.ws, self.ws_bytes, stream))
        return idx, w, lg

    def experts(self, x: torch.Tensor, idx: torch.Tensor, w: torch.Tensor, stream=None):
        n = x.shape[0]
        out = torch.empty(n, self.cfg.hidden, dtype=torch.bfloat16, device=x.device)
        B.check(B.moe_experts(self.c_cfg, self.c_w, x, n, idx, w, out, self.ws, self.ws_bytes,
                              stream))
        return out
