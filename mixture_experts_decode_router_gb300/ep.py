"""Expert parallelism over ``torch.distributed``.

The EP branch of MoeLayer::forward and forward_token_major_decode (pages
"metrale_model_layers/layers/moe/forward.rs" and
"spark_model/layers/moe/forward_token_major.rs"): every rank routes each token
over all experts, but evaluates only the routed experts it holds, and its blend
leaves the shared expert out; the BF16 partial outputs are summed over ranks
(an all-reduce of ``N x H`` BF16 values); the shared expert, gated, is then
added once (the pages' residual_add / moe_batched_blend).

Here each step is a library call: the partial is ``moe_forward`` with the
rank's expert range and ``exclude_shared``; the addition of the shared expert
is ``moe_forward`` with no routed expert and ``accumulate``.  This module only
orders those calls around the collective.
"""

from __future__ import annotations

from typing import Callable, Optional, Tuple

import torch
import torch.distributed as dist

from .layer import MoeLayer
from .synth import LayerWeights, expert_slice


def expert_range(rank: int, world_size: int, num_experts: int) -> Tuple[int, int]:
    """Contiguous block [begin, end) of the routed experts rank ``rank`` holds:
    ``num_experts // world_size`` each, the first ``num_experts % world_size``
    ranks one more."""
    if not (0 <= rank < world_size) or num_experts < 0:
        raise ValueError("bad rank, world size or expert count")
    q, r = divmod(num_experts, world_size)
    begin = rank * q + min(rank, r)
    return begin, begin + q + (1 if rank < r else 0)


def ep_forward(x: torch.Tensor,
               partial_fn: Callable[[torch.Tensor], torch.Tensor],
               add_shared_fn: Optional[Callable[[torch.Tensor, torch.Tensor], None]],
               group=None) -> torch.Tensor:
    """One expert-parallel layer step on this rank: the rank's partial
    (``partial_fn(x)``, BF16 [N, H], no shared expert), summed in place over the
    ranks of ``group``, then the shared expert added once
    (``add_shared_fn(x, out)``, in place; None when the layer has none)."""
    out = partial_fn(x)
    if dist.is_initialized() and dist.get_world_size(group) > 1:
        dist.all_reduce(out, op=dist.ReduceOp.SUM, group=group)
    if add_shared_fn is not None:
        add_shared_fn(x, out)
    return out


class ExpertParallelMoe:
    """This rank's part of an expert-parallel MoE layer on its CUDA device.

    ``weights`` is the whole layer; the rank keeps views of its own expert
    block (``synth.expert_slice``), the router and the shared expert.
    """

    def __init__(self, weights: LayerWeights, max_tokens: int, rank: int, world_size: int,
                 group=None, path: str = "auto"):
        cfg = weights.cfg
        self.experts = expert_range(rank, world_size, cfg.num_experts)
        local = expert_slice(weights, *self.experts)
        self.group = group
        self.partial = MoeLayer(local, max_tokens, path, experts=self.experts,
                                exclude_shared=True)
        E = cfg.num_experts
        self.shared = (MoeLayer(local, max_tokens, path, experts=(E, E), accumulate=True)
                       if cfg.shared_inter > 0 else None)

    def forward(self, x: torch.Tensor) -> torch.Tensor:
        def partial(xx):
            out, _, _ = self.partial.forward(xx)
            return out

        def add_shared(xx, out):
            self.shared.forward(xx, out=out, routing=False)

        return ep_forward(x, partial, add_shared if self.shared is not None else None, self.group)
