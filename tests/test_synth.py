"""The seeded input generators (CPU): shapes, determinism, and the views the
expert-parallel tests take."""

import numpy as np
import torch

from mixture_experts_decode_router_gb300 import synth


def _cfg(fmt, **kw):
    return synth.LayerConfig("t", 64, 8, 2, 32, 32, synth.ROUTE_SIGMOID_BIAS, True, 2.5, fmt, 3,
                             **kw)


def test_norm_weight_is_seeded_and_near_one():
    a = synth.make_weights(_cfg(synth.FMT_BF16, pre_expert_norm=True))
    b = synth.make_weights(_cfg(synth.FMT_BF16, pre_expert_norm=True))
    assert a.pre_expert_norm_w.dtype == torch.bfloat16 and a.pre_expert_norm_w.shape == (64,)
    assert torch.equal(a.pre_expert_norm_w, b.pre_expert_norm_w)
    assert float((a.pre_expert_norm_w.float() - 1).abs().max()) < 1.0
    assert synth.make_weights(_cfg(synth.FMT_BF16)).pre_expert_norm_w is None


def test_expert_slice_views_the_stacks():
    for fmt in (synth.FMT_BF16, synth.FMT_FP8_B128, synth.FMT_NVFP4):
        lw = synth.make_weights(_cfg(fmt))
        part = synth.expert_slice(lw, 3, 7)
        for name in ("gate", "up", "down"):
            q, p = getattr(lw, name), getattr(part, name)
            assert p.w.shape[0] == 4 and torch.equal(p.w, q.w[3:7])
            if q.scale is not None:
                assert torch.equal(p.scale, q.scale[3:7])
            if q.scale2 is not None:
                assert torch.equal(p.scale2, q.scale2[3:7])
        assert part.sh_gate is lw.sh_gate and part.router_w is lw.router_w
        assert synth.expert_slice(lw, 8, 8).gate.w.shape[0] == 0


def test_nvfp4_router_is_the_quantised_bf16_router():
    from oracle import moe_oracle as O
    from tests.moe_helpers import bf16_bits, host_qmat
    lw = synth.make_weights(_cfg(synth.FMT_BF16, router_fmt=synth.FMT_NVFP4))
    q = lw.router_q
    assert q.w.shape == (1, 8, 32) and q.scale.shape == (1, 8, 4) and q.scale2.shape == (1,)
    dq = host_qmat(q).expert(0)
    ref = O.bf16_decode(bf16_bits(lw.router_w))
    # E2M1 with an E4M3 block scale: within a quarter of each block's largest magnitude.
    blk = np.abs(ref).reshape(8, 4, 16).max(axis=2).repeat(16, axis=1)
    assert np.all(np.abs(dq - ref) <= 0.25 * blk + 1e-3 * np.abs(ref).max())
    assert synth.make_weights(_cfg(synth.FMT_BF16)).router_q is None
