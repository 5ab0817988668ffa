"""Test helpers: host copies of device weights for the oracle, and the oracle's
near-tie margin as the generator's ``gap_fn``."""

from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

from mixture_experts_decode_router_gb300.synth import LayerWeights, QMatT
from oracle import moe_oracle as O


class LazyExperts:
    """Index [e] -> host numpy array of expert e, fetched from the device on demand
    (so a 256-expert FP8 layer never has to be copied to the host whole)."""

    def __init__(self, t: torch.Tensor, as_uint16: bool = False):
        self.t = t
        self.as_uint16 = as_uint16
        self._cache = {}

    def __getitem__(self, e):
        e = int(e)
        if e not in self._cache:
            a = self.t[e].contiguous()
            if self.as_uint16:
                a = a.view(torch.int16).cpu().numpy().view(np.uint16)
            else:
                a = a.cpu().numpy()
            self._cache[e] = a
        return self._cache[e]


def host_qmat(q: QMatT) -> O.QMat:
    if q.fmt == O.FMT_BF16:
        return O.QMat(q.fmt, LazyExperts(q.w, as_uint16=True))
    if q.fmt == O.FMT_FP8_B128:
        return O.QMat(q.fmt, LazyExperts(q.w), q.scale.cpu().numpy())
    return O.QMat(q.fmt, LazyExperts(q.w), LazyExperts(q.scale), q.scale2.cpu().numpy())


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def oracle_layer(lw: LayerWeights) -> O.OracleLayer:
    c = lw.cfg
    return O.OracleLayer(
        hidden=c.hidden, num_experts=c.num_experts, top_k=c.top_k, inter=c.inter,
        shared_inter=c.shared_inter, routing=c.routing, norm_topk_prob=c.norm_topk_prob,
        routed_scaling_factor=c.routed_scaling_factor, router_w=bf16_bits(lw.router_w),
        gate=host_qmat(lw.gate), up=host_qmat(lw.up), down=host_qmat(lw.down),
        sh_gate=host_qmat(lw.sh_gate) if lw.sh_gate is not None else None,
        sh_up=host_qmat(lw.sh_up) if lw.sh_up is not None else None,
        sh_down=host_qmat(lw.sh_down) if lw.sh_down is not None else None,
        correction_bias=lw.correction_bias.cpu().numpy() if lw.correction_bias is not None else None,
        shared_gate_w=bf16_bits(lw.shared_gate_w) if lw.shared_gate_w is not None else None,
        pre_expert_norm_w=(bf16_bits(lw.pre_expert_norm_w) if lw.pre_expert_norm_w is not None
                           else None),
        rms_norm_eps=c.rms_norm_eps,
        router_q=host_qmat(lw.router_q) if lw.router_q is not None else None)


def gap_fn_for(layer: O.OracleLayer):
    """Per-row margin between the k-th and (k+1)-th selection score (fp64)."""
    def fn(x_bits: np.ndarray) -> np.ndarray:
        x = O.bf16_decode(x_bits)
        lg = O.router_logits(x, O.router_weights(layer))
        return O.topk_gap(O.selection_scores(lg, layer.routing, layer.correction_bias),
                          layer.top_k)
    return fn


def tolerance(fmt: str) -> float:
    """max|err| bound as a fraction of RMS(oracle): 2e-2 for BF16 and FP8
    experts, 5e-2 for NVFP4."""
    return 5e-2 if fmt == O.FMT_NVFP4 else 2e-2


def oracle_forward_threaded(layer: O.OracleLayer, x_bits: np.ndarray, rows=None, threads=None):
    """``O.moe_forward`` of ``rows`` computed as the sum of expert-parallel
    partials over contiguous expert ranges (each holding about the same number
    of the touched experts) plus the shared-expert-only call, the parts run in
    threads (numpy releases the GIL in its array loops).  The oracle itself is
    unchanged: a sum of its own partials, which the oracle pins show equal to
    the whole layer.  Returns (out, idx, w) like ``O.moe_forward``."""
    x = O.bf16_decode(x_bits)
    rows = np.arange(x.shape[0]) if rows is None else np.asarray(rows)
    lg = O.router_logits(x[rows], O.router_weights(layer))
    idx, w = O.route(lg, layer.routing, layer.top_k, layer.norm_topk_prob,
                     layer.routed_scaling_factor, layer.correction_bias)
    touched = np.unique(idx)
    threads = threads or max(1, min(8, os.cpu_count() or 1))
    chunks = [c for c in np.array_split(touched, threads) if len(c)]
    ranges = [(int(c[0]), int(c[-1]) + 1) for c in chunks]

    def part(r):
        return O.moe_forward(layer, x_bits, rows=rows, experts=r, include_shared=False)[0]

    def shared():
        return O.moe_forward(layer, x_bits, rows=rows, experts=(0, 0), include_shared=True)[0]

    with ThreadPoolExecutor(max_workers=len(ranges) + 1) as ex:
        futs = [ex.submit(part, r) for r in ranges] + [ex.submit(shared)]
        out = sum(f.result() for f in futs)
    return out, idx, w
