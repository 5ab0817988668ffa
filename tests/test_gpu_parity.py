"""Parity of the CUDA path (through the C ABI) with the fp64 oracle.

* Indices: bit-exact, in slot order (the generator redraws any input row whose
  k-th and (k+1)-th selection scores are within 1e-3, so the decision does not
  hang on rounding).
* Routing weights: within 1e-5 * routed_scaling_factor of the oracle.
* Router logits: within 1e-4 * RMS(logits).
* Output: max|err| <= 2e-2 * RMS(oracle) for BF16 and FP8 experts,
  <= 5e-2 * RMS(oracle) for NVFP4.
* Batch invariance: a row's output bits do not depend on which rows share the
  call (computed alone, permuted, duplicated).
* Expert parallelism: each rank's partial against the oracle's, and the
  partials summed (plus one shared-expert-only call) against the whole layer.
"""

import dataclasses

import numpy as np
import pytest
import torch

from mixture_experts_decode_router_gb300 import binding as B
from mixture_experts_decode_router_gb300 import synth
from mixture_experts_decode_router_gb300.layer import MoeLayer
from oracle import moe_oracle as O
from tests.moe_helpers import (bf16_bits, gap_fn_for, oracle_forward_threaded, oracle_layer,
                               tolerance)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    B.load()


_SMALL = dict(hidden=256, num_experts=16, top_k=2, inter=128, shared_inter=128,
              routing=synth.ROUTE_SOFTMAX, norm_topk_prob=True, routed_scaling_factor=1.0,
              expert_fmt=synth.FMT_BF16, n_tokens=1)


def small(name, **kw):
    d = dict(_SMALL)
    d.update(kw)
    return synth.LayerConfig(name, **d)


def _check(cfg, n=None, path="auto", rows=None, x=None, lw=None, threaded=False):
    n = cfg.n_tokens if n is None else n
    lw = synth.make_weights(cfg, "cuda") if lw is None else lw
    L = oracle_layer(lw)
    if x is None:
        x = synth.make_input(cfg, n, "cuda", gap_fn=gap_fn_for(L))
    layer = MoeLayer(lw, n, path)
    out, idx, w = layer.forward(x)
    torch.cuda.synchronize()
    xb = bf16_bits(x)
    # Routing for every row (cheap), the layer output for `rows`.
    lg_ref = O.router_logits(O.bf16_decode(xb), O.router_weights(L))
    idx_ref, w_ref = O.route(lg_ref, L.routing, L.top_k, L.norm_topk_prob,
                             L.routed_scaling_factor, L.correction_bias)
    assert np.array_equal(idx.cpu().numpy(), idx_ref), "expert indices differ"
    assert np.max(np.abs(w.cpu().numpy() - w_ref)) <= 1e-5 * max(1.0, cfg.routed_scaling_factor)
    rows = np.arange(n) if rows is None else np.asarray(rows)
    if threaded:    # the full-size layers: the oracle's expert partials in threads
        ref, _, _ = oracle_forward_threaded(L, xb, rows=rows)
    else:
        ref, _, _, _ = O.moe_forward(L, xb, rows=rows)
    got = out.float().cpu().numpy()[rows]
    rms = float(np.sqrt(np.mean(ref ** 2)))
    err = float(np.max(np.abs(got - ref)))
    assert err <= tolerance(cfg.expert_fmt) * rms, f"max|err| {err:.3e} vs RMS {rms:.3e}"
    return lw, x, out, idx, w, layer


# ---------------------------------------------------------------- small, element by element

SMALL_CASES = [
    small("bf16_softmax_k2"),
    small("bf16_sigmoid", routing=synth.ROUTE_SIGMOID_BIAS, routed_scaling_factor=2.5, top_k=4),
    small("fp8_softmax", expert_fmt=synth.FMT_FP8_B128, top_k=3),
    small("fp8_ragged", expert_fmt=synth.FMT_FP8_B128, hidden=288, inter=160, shared_inter=96,
          routing=synth.ROUTE_SIGMOID_BIAS, routed_scaling_factor=1.5),
    small("nvfp4_softmax", expert_fmt=synth.FMT_NVFP4, top_k=2),
    small("nvfp4_ragged", expert_fmt=synth.FMT_NVFP4, hidden=352, inter=96, shared_inter=160,
          num_experts=40, top_k=5),
    small("no_norm", norm_topk_prob=False, routed_scaling_factor=1.0, top_k=3),
    small("no_shared", shared_inter=0, top_k=2),
    small("shared_gate", shared_gate=True, routing=synth.ROUTE_SIGMOID_BIAS),
    small("top1", top_k=1, num_experts=8),
    small("all_experts", top_k=8, num_experts=8),
    small("wide_E", num_experts=1024, top_k=32, hidden=128, inter=64, shared_inter=64),
    small("E33", num_experts=33, top_k=6, routing=synth.ROUTE_SIGMOID_BIAS),
    small("pre_norm", pre_expert_norm=True, shared_gate=True, routing=synth.ROUTE_SIGMOID_BIAS,
          top_k=3, routed_scaling_factor=2.5),
    small("pre_norm_fp8", expert_fmt=synth.FMT_FP8_B128, pre_expert_norm=True, rms_norm_eps=1e-5),
    small("pre_norm_nvfp4", expert_fmt=synth.FMT_NVFP4, pre_expert_norm=True, num_experts=40,
          top_k=5, hidden=352),
    small("router_nvfp4", router_fmt=synth.FMT_NVFP4, routing=synth.ROUTE_SIGMOID_BIAS,
          shared_gate=True, top_k=4, num_experts=32, routed_scaling_factor=2.5),
    small("router_nvfp4_fp8", router_fmt=synth.FMT_NVFP4, expert_fmt=synth.FMT_FP8_B128,
          hidden=288, num_experts=24, top_k=3),
]


@pytest.mark.parametrize("cfg", SMALL_CASES, ids=lambda c: c.name)
@pytest.mark.parametrize("n", [1, 2, 3, 4, 16, 17, 40])
def test_small_layers(cfg, n):
    _check(cfg, n)


@pytest.mark.parametrize("path", ["token_major", "grouped"])
@pytest.mark.parametrize("fmt", [synth.FMT_BF16, synth.FMT_FP8_B128, synth.FMT_NVFP4])
def test_forced_paths(path, fmt):
    cfg = small(f"path_{fmt}", expert_fmt=fmt, num_experts=32, top_k=4,
                routing=synth.ROUTE_SIGMOID_BIAS, routed_scaling_factor=2.5)
    for n in (1, 16, 17, 70):
        _check(cfg, n, path=path)


@pytest.mark.parametrize("fmt", [synth.FMT_BF16, synth.FMT_FP8_B128, synth.FMT_NVFP4])
@pytest.mark.parametrize("n", [33, 150])
def test_all_tokens_on_one_expert(fmt, n):
    """Every route on the same two experts: at 150 tokens each expert's tokens
    span three tensor-core token segments (64 + 64 + 22)."""
    cfg = small("one_expert", num_experts=16, top_k=2, expert_fmt=fmt)
    lw = synth.make_weights(cfg, "cuda")
    x1 = synth.make_input(cfg, 1, "cuda", gap_fn=gap_fn_for(oracle_layer(lw)))
    x = x1.repeat(n, 1)
    rows = sorted({r for r in (0, 31, 63, 64, 127, 128, n - 1) if r < n})
    _, _, _, _, _, layer = _check(cfg, n, x=x, lw=lw, rows=rows)
    assert layer.device_error() == 0


@pytest.mark.parametrize("norm,router", [(False, synth.FMT_BF16), (True, synth.FMT_BF16),
                                         (False, synth.FMT_NVFP4)])
def test_route_and_experts_entry_points(norm, router):
    cfg = small("split", routing=synth.ROUTE_SIGMOID_BIAS, top_k=3, routed_scaling_factor=2.5,
                shared_gate=True, pre_expert_norm=norm, router_fmt=router)
    lw = synth.make_weights(cfg, "cuda")
    L = oracle_layer(lw)
    x = synth.make_input(cfg, 9, "cuda", gap_fn=gap_fn_for(L))
    layer = MoeLayer(lw, 9)
    idx, w, lg = layer.route(x)
    torch.cuda.synchronize()
    lg_ref = O.router_logits(O.bf16_decode(bf16_bits(x)), O.router_weights(L))
    rms = np.sqrt(np.mean(lg_ref ** 2))
    assert np.max(np.abs(lg.cpu().numpy() - lg_ref)) <= 1e-4 * rms
    # moe_experts on the oracle's routing (as int32/fp32), then against the oracle output.
    idx_ref, w_ref = O.route(lg_ref, L.routing, L.top_k, L.norm_topk_prob,
                             L.routed_scaling_factor, L.correction_bias)
    out = layer.experts(x, torch.from_numpy(idx_ref.astype(np.int32)).cuda(),
                        torch.from_numpy(w_ref.astype(np.float32)).cuda())
    fwd, _, _ = layer.forward(x)
    # On the library's own routing, moe_route + moe_experts is moe_forward bit for bit.
    own = layer.experts(x, idx, w)
    torch.cuda.synchronize()
    ref, _, _, _ = O.moe_forward(L, bf16_bits(x))
    rms_o = np.sqrt(np.mean(ref ** 2))
    assert np.max(np.abs(out.float().cpu().numpy() - ref)) <= 2e-2 * rms_o
    assert torch.equal(own, fwd)


# ---------------------------------------------------------------- the grouped path's tensor-core router

def _route_against_oracle(cfg, n, path="auto"):
    lw = synth.make_weights(cfg, "cuda")
    L = oracle_layer(lw)
    x = synth.make_input(cfg, n, "cuda", gap_fn=gap_fn_for(L))
    layer = MoeLayer(lw, n, path)
    idx, w, lg = layer.route(x)
    torch.cuda.synchronize()
    lg_ref = O.router_logits(O.bf16_decode(bf16_bits(x)), O.router_weights(L))
    idx_ref, w_ref = O.route(lg_ref, L.routing, L.top_k, L.norm_topk_prob,
                             L.routed_scaling_factor, L.correction_bias)
    rms = float(np.sqrt(np.mean(lg_ref ** 2)))
    err = float(np.max(np.abs(lg.cpu().numpy() - lg_ref)))
    assert err <= 1e-4 * rms, f"logits max|err| {err:.3e} vs RMS {rms:.3e}"
    assert np.array_equal(idx.cpu().numpy(), idx_ref), "expert indices differ"
    assert np.max(np.abs(w.cpu().numpy() - w_ref)) <= 1e-5 * max(1.0, cfg.routed_scaling_factor)
    return x, layer, idx, w, lg


@pytest.mark.parametrize("n", [4, 16, 129, 300])
def test_tensor_core_router_logits(n):
    """moe_route on the grouped path (the tensor-core router: 16 K splits of 128
    at H = 2048; 129 and 300 tokens span two and three token tiles, the last
    ragged) against the oracle's fp64 logits and routing."""
    cfg = dataclasses.replace(synth.WORKLOADS["decode_n16"], name="tc_router")
    _route_against_oracle(cfg, n)


def test_tensor_core_router_wide_splits():
    """H = 7168: 16 K splits of 448 (seven 64-element boxes each)."""
    cfg = small("tc_router_7168", hidden=7168, num_experts=64, top_k=4, inter=128, shared_inter=128)
    _route_against_oracle(cfg, 20)


def test_tensor_core_and_cuda_core_routers_agree():
    """The same tokens routed by the grouped path's tensor-core router and by the
    token-major path's CUDA-core router: the same experts, logits within the
    accumulation-order difference."""
    cfg = small("tc_vs_cc", num_experts=40, top_k=5, routing=synth.ROUTE_SIGMOID_BIAS,
                routed_scaling_factor=2.5)
    x, _, idx_g, w_g, lg_g = _route_against_oracle(cfg, 24, path="grouped")
    lw = synth.make_weights(cfg, "cuda")
    idx_t, w_t, lg_t = MoeLayer(lw, 24, "token_major").route(x)
    torch.cuda.synchronize()
    assert torch.equal(idx_g, idx_t)
    scale = float(lg_t.abs().max())
    assert float((lg_g - lg_t).abs().max()) <= 1e-5 * scale
    assert float((w_g - w_t).abs().max()) <= 1e-5 * cfg.routed_scaling_factor


def test_router_partials_over_the_cap_take_the_cuda_core_router():
    """E = 1024 at 160 tokens: 16 x 160 x 1024 x 4 bytes of partials exceed the
    8 MiB cap, so the grouped path routes on the CUDA cores; the layer still
    matches the oracle."""
    cfg = small("tc_cap", num_experts=1024, top_k=8, hidden=2048, inter=64, shared_inter=64)
    _route_against_oracle(cfg, 160)
    _check(cfg, 160)


@pytest.mark.parametrize("routing", [synth.ROUTE_SOFTMAX, synth.ROUTE_SIGMOID_BIAS])
@pytest.mark.parametrize("n", [1, 3, 16])
def test_exact_ties_go_to_the_lower_index(routing, n):
    """Two experts with identical, dominant router rows (and equal biases) tie
    exactly on every token: the lower index takes the single slot (k = 1) on
    every path.  An all-zero router ties all experts: slots 0..k-1 in order."""
    cfg = small("ties", num_experts=16, top_k=1, routing=routing,
                routed_scaling_factor=1.0 if routing == synth.ROUTE_SOFTMAX else 2.5)
    lw = synth.make_weights(cfg, "cuda")
    for lo, hi in ((0, 1), (2, 5), (9, 14)):
        router = lw.router_w.clone()
        router[hi] = router[lo] = (lw.router_w[lo].float() * 40).to(torch.bfloat16)
        bias = lw.correction_bias.clone() if lw.correction_bias is not None else None
        if bias is not None:
            bias[hi] = bias[lo]
        tied = dataclasses.replace(lw, router_w=router, correction_bias=bias)
        x = synth.make_input(cfg, n, "cuda")
        # Make the tied experts dominate: x along their (shared) router row.
        x = (x.float() * 0.1 + router[lo].float() / router[lo].float().norm()).to(torch.bfloat16)
        out, idx, w = MoeLayer(tied, n).forward(x)
        torch.cuda.synchronize()
        assert torch.all(idx == lo), (lo, hi, idx.flatten().tolist())
        L = oracle_layer(tied)
        _, idx_ref, _, _ = O.moe_forward(L, bf16_bits(x))
        assert np.all(idx_ref == lo)
    zero = dataclasses.replace(lw, router_w=torch.zeros_like(lw.router_w),
                               correction_bias=(torch.zeros_like(lw.correction_bias)
                                                if lw.correction_bias is not None else None))
    for k in (1, 3):
        zk = dataclasses.replace(zero, cfg=zero.cfg.with_(top_k=k))
        x = synth.make_input(cfg, n, "cuda")
        _, idx, w = MoeLayer(zk, n).forward(x)
        torch.cuda.synchronize()
        assert torch.equal(idx.cpu(), torch.arange(k, dtype=torch.int32).repeat(n, 1))
        expect = (1.0 / k) * (1.0 if routing == synth.ROUTE_SOFTMAX else 2.5)
        assert torch.allclose(w.cpu(), torch.full((n, k), expect), rtol=1e-6)


@pytest.mark.parametrize("fmt", [synth.FMT_BF16, synth.FMT_FP8_B128, synth.FMT_NVFP4])
@pytest.mark.parametrize("n", [1, 3, 16])
def test_host_mapped_input_and_output(fmt, n):
    """x and out in pinned host memory: the kernels read x and write out across
    the host link, with the bits of the device-buffer call."""
    cfg = small("host_mapped", expert_fmt=fmt, shared_gate=True, top_k=3)
    lw = synth.make_weights(cfg, "cuda")
    x = synth.make_input(cfg, n, "cuda", gap_fn=gap_fn_for(oracle_layer(lw)))
    layer = MoeLayer(lw, n)
    ref, idx_ref, w_ref = layer.forward(x)
    x_h = x.cpu().pin_memory()
    out_h = torch.full((n, cfg.hidden), float("nan"), dtype=torch.bfloat16).pin_memory()
    idx = torch.empty_like(idx_ref)
    w = torch.empty_like(w_ref)
    stream = torch.cuda.current_stream().cuda_stream
    B.check(B.moe_forward(layer.c_cfg, layer.c_w, x_h, n, out_h, idx, w, layer.ws, layer.ws_bytes, stream))
    torch.cuda.synchronize()
    assert torch.equal(out_h.view(torch.int16), ref.cpu().view(torch.int16))
    assert torch.equal(idx, idx_ref) and torch.equal(w, w_ref)
    # accumulate: out (host) += the layer output
    acc_layer = MoeLayer(lw, n, accumulate=True)
    base = synth.make_input(cfg, n, "cuda").cpu()
    out2 = base.clone().pin_memory()
    B.check(B.moe_forward(acc_layer.c_cfg, acc_layer.c_w, x_h, n, out2, idx, w, acc_layer.ws,
                          acc_layer.ws_bytes, stream))
    torch.cuda.synchronize()
    out2_ref = base.cuda()
    acc_layer.forward(x, out=out2_ref)
    torch.cuda.synchronize()
    assert torch.equal(out2.view(torch.int16), out2_ref.cpu().view(torch.int16))
    assert layer.device_error() == 0 and acc_layer.device_error() == 0


def test_pageable_host_memory_is_refused_and_host_route_matches():
    cfg = small("host_refuse")
    lw = synth.make_weights(cfg, "cuda")
    x = synth.make_input(cfg, 5, "cuda", gap_fn=gap_fn_for(oracle_layer(lw)))
    layer = MoeLayer(lw, 5)
    stream = torch.cuda.current_stream().cuda_stream
    out = torch.empty(5, cfg.hidden, dtype=torch.bfloat16, device="cuda")
    idx = torch.empty(5, cfg.top_k, dtype=torch.int32, device="cuda")
    w = torch.empty(5, cfg.top_k, dtype=torch.float32, device="cuda")
    x_pageable = x.cpu()   # not pinned
    assert not x_pageable.is_pinned()
    s = B.moe_forward(layer.c_cfg, layer.c_w, x_pageable, 5, out, idx, w, layer.ws, layer.ws_bytes, stream)
    assert s == B.MOE_ERR_HOST_MEMORY
    out_pageable = torch.empty(5, cfg.hidden, dtype=torch.bfloat16)
    s = B.moe_forward(layer.c_cfg, layer.c_w, x, 5, out_pageable, idx, w, layer.ws, layer.ws_bytes, stream)
    assert s == B.MOE_ERR_HOST_MEMORY
    # moe_route with x in pinned host memory: the device-buffer result, bit for bit
    idx_d, w_d, lg_d = layer.route(x)
    x_h = x.cpu().pin_memory()
    lg = torch.empty(5, cfg.num_experts, dtype=torch.float32, device="cuda")
    B.check(B.moe_route(layer.c_cfg, layer.c_w, x_h, 5, idx, w, lg, layer.ws, layer.ws_bytes, stream))
    torch.cuda.synchronize()
    assert torch.equal(idx, idx_d) and torch.equal(w, w_d) and torch.equal(lg, lg_d)
    assert layer.device_error() == 0


def test_zero_tokens_is_a_noop():
    cfg = small("empty")
    lw = synth.make_weights(cfg, "cuda")
    layer = MoeLayer(lw, 4)
    x = torch.empty(0, cfg.hidden, dtype=torch.bfloat16, device="cuda")
    out, idx, w = layer.forward(x)
    torch.cuda.synchronize()
    assert out.shape == (0, cfg.hidden)


@pytest.mark.parametrize("norm", [False, True])
@pytest.mark.parametrize("fmt", [synth.FMT_BF16, synth.FMT_FP8_B128, synth.FMT_NVFP4])
def test_rows_do_not_depend_on_the_batch_token_major(fmt, norm):
    """The token-major kernels (forced), and one token alone: the single-token
    kernel, which keeps the token-major arithmetic (the RMSNorm included)."""
    cfg = small("invariance", expert_fmt=fmt, num_experts=32, top_k=4,
                routing=synth.ROUTE_SIGMOID_BIAS, routed_scaling_factor=2.5,
                pre_expert_norm=norm)
    lw = synth.make_weights(cfg, "cuda")
    L = oracle_layer(lw)
    x = synth.make_input(cfg, 12, "cuda", gap_fn=gap_fn_for(L))
    layer = MoeLayer(lw, 64, path="token_major")
    full, _, _ = layer.forward(x)
    perm = torch.randperm(12, generator=torch.Generator().manual_seed(3)).cuda()
    permuted, _, _ = layer.forward(x[perm])
    alone = torch.cat([layer.forward(x[r:r + 1])[0] for r in range(12)])
    dup, _, _ = layer.forward(torch.cat([x, x[:4]]))
    torch.cuda.synchronize()
    assert torch.equal(permuted, full[perm])
    assert torch.equal(alone, full)
    assert torch.equal(dup[12:], full[:4])


@pytest.mark.parametrize("norm", [False, True])
@pytest.mark.parametrize("fmt", [synth.FMT_BF16, synth.FMT_FP8_B128, synth.FMT_NVFP4])
def test_rows_do_not_depend_on_the_batch_grouped(fmt, norm):
    """N >= 4: the expert-grouped tensor-core path."""
    cfg = small("invariance_g", expert_fmt=fmt, num_experts=32, top_k=4,
                routing=synth.ROUTE_SIGMOID_BIAS, routed_scaling_factor=2.5,
                pre_expert_norm=norm)
    lw = synth.make_weights(cfg, "cuda")
    L = oracle_layer(lw)
    x = synth.make_input(cfg, 40, "cuda", gap_fn=gap_fn_for(L))
    layer = MoeLayer(lw, 300)
    full, _, _ = layer.forward(x)
    perm = torch.randperm(40, generator=torch.Generator().manual_seed(4)).cuda()
    permuted, _, _ = layer.forward(x[perm])
    part, _, _ = layer.forward(x[:17])
    many, _, _ = layer.forward(x.repeat(7, 1))        # 280 rows: experts past 128 tokens
    torch.cuda.synchronize()
    assert torch.equal(permuted, full[perm])
    assert torch.equal(part, full[:17])
    assert torch.equal(many[-40:], full)


def _scale_at_offset(q, off):
    """q with its block scales moved to a buffer `off` bytes past a 256-byte
    aligned allocation (the same bytes at another address)."""
    flat = q.scale.contiguous().view(torch.uint8).flatten()
    buf = torch.zeros(flat.numel() + 256, dtype=torch.uint8, device=flat.device)
    buf[off:off + flat.numel()] = flat
    moved = buf[off:off + flat.numel()].view(q.scale.dtype).view(q.scale.shape)
    assert moved.data_ptr() % 16 == off % 16
    return dataclasses.replace(q, scale=moved)


@pytest.mark.parametrize("n", [17, 150])
def test_nvfp4_scales_at_a_4_byte_offset(n):
    """The API asks only 4-byte alignment of block scales: the same NVFP4
    scales 4 bytes off a 16-byte boundary give bit-identical outputs (and the
    aligned call matches the oracle)."""
    cfg = small("nvfp4_scale_offset", expert_fmt=synth.FMT_NVFP4, hidden=512, top_k=4, num_experts=32)
    lw, x, out, idx, w, layer = _check(cfg, n)
    moved = dataclasses.replace(lw, gate=_scale_at_offset(lw.gate, 4), up=_scale_at_offset(lw.up, 4),
                                sh_gate=_scale_at_offset(lw.sh_gate, 4), sh_up=_scale_at_offset(lw.sh_up, 4))
    assert moved.gate.scale.data_ptr() % 16 == 4
    out2, idx2, _ = MoeLayer(moved, n).forward(x)
    torch.cuda.synchronize()
    assert torch.equal(idx2, idx)
    assert torch.equal(out2, out)


def test_both_groupings_of_the_top_k_kernel_agree():
    """The grouped path's top-k kernel sorts the routes by expert with a token
    bitmap per expert while it fits (E * ceil(n / 32) <= 8192 words and
    n * k <= 8192), else with per-warp counts.  With 1024 experts, 250 tokens
    take the bitmap and 300 the counts: the 300-token call matches the oracle,
    and the rows both calls share are identical, bit for bit.  (FP8 experts:
    their f16 intermediate keeps 300 rows of this small layer well inside the
    tolerance; BF16's bf16 intermediate at K = 64 reaches ~2e-2 RMS at the tail
    of 38k outputs.)"""
    cfg = small("groupings", num_experts=1024, top_k=8, hidden=128, inter=64, shared_inter=64,
                expert_fmt=synth.FMT_FP8_B128)
    lw, x, out, idx, w, layer = _check(cfg, 300)
    part, idx_p, w_p = layer.forward(x[:250])
    torch.cuda.synchronize()
    assert torch.equal(idx_p, idx[:250])
    assert torch.equal(w_p, w[:250])
    assert torch.equal(part, out[:250])


# ---------------------------------------------------------------- expert parallelism

def _ep_check(cfg, n, ranges, path="auto", rows=None):
    """Each rank's partial (its experts only, no shared expert) against the
    oracle's partial; the partials summed plus one shared-expert-only call
    against the whole layer.  Routing is the same on every rank.

    A partial is a sparse, heavy-tailed matrix (rows with no local route are
    exactly zero), so its RMS is small next to its largest entries and the
    BF16 rounding of the output alone (up to 2^-9 of an entry) can exceed
    tol * RMS.  The bound is therefore tol * RMS (over the rows with a local
    route) plus 2^-8 of each oracle entry; for the sum, plus 2^-8 of the sum of
    the partials' magnitudes (each partial and the sum are BF16)."""
    lw = synth.make_weights(cfg, "cuda")
    L = oracle_layer(lw)
    x = synth.make_input(cfg, n, "cuda", gap_fn=gap_fn_for(L))
    xb = bf16_bits(x)
    rows = np.arange(n) if rows is None else np.asarray(rows)
    tol = tolerance(cfg.expert_fmt)
    full_ref, idx_ref, _, _ = O.moe_forward(L, xb, rows=rows)
    total = torch.zeros(n, cfg.hidden, dtype=torch.float32, device="cuda")
    mag = np.zeros_like(full_ref)          # sum over ranks of |oracle partial|
    idx0 = None
    for (b, e) in ranges:
        layer = MoeLayer(synth.expert_slice(lw, b, e), n, path, experts=(b, e),
                         exclude_shared=True)
        out, idx, _ = layer.forward(x)
        torch.cuda.synchronize()
        assert layer.device_error() == 0
        if idx0 is None:
            idx0 = idx.clone()
        assert torch.equal(idx, idx0), "routing differs between ranks"
        ref, _, _, _ = O.moe_forward(L, xb, rows=rows, experts=(b, e), include_shared=False)
        got = out.float().cpu().numpy()[rows]
        live = np.any(ref != 0, axis=1)                    # rows with a route to this rank
        assert not np.any(got[~live]), f"rank [{b}, {e}): non-zeros in rows it does not serve"
        if np.any(live):
            rms = float(np.sqrt(np.mean(ref[live] ** 2)))
            bound = tol * rms + 2.0 ** -8 * np.abs(ref)
            assert np.all(np.abs(got - ref) <= bound), \
                f"rank [{b}, {e}): max excess {float(np.max(np.abs(got - ref) - bound)):.3e}"
        mag += np.abs(ref)
        total += out.float()
    assert np.array_equal(idx0.cpu().numpy()[rows], idx_ref)
    # The all-reduce's result: the partials summed, in BF16.
    reduced = total.to(torch.bfloat16)
    if cfg.shared_inter > 0:
        E = cfg.num_experts
        none = synth.expert_slice(lw, E, E)
        sh = MoeLayer(none, n, path, experts=(E, E))
        out, _, _ = sh.forward(x)                  # the shared expert alone (routing computed)
        torch.cuda.synchronize()
        ref, _, _, _ = O.moe_forward(L, xb, rows=rows, experts=(E, E))
        rms = float(np.sqrt(np.mean(ref ** 2)))
        assert np.max(np.abs(out.float().cpu().numpy()[rows] - ref)) <= tol * rms, "shared only"
        # Added once into the reduced output (routing skipped, then computed:
        # the same bits).
        add = MoeLayer(none, n, path, experts=(E, E), accumulate=True)
        again = reduced.clone()
        add.forward(x, out=reduced, routing=False)
        add.forward(x, out=again)
        torch.cuda.synchronize()
        assert add.device_error() == 0
        assert torch.equal(reduced, again)
    rms = float(np.sqrt(np.mean(full_ref ** 2)))
    diff = np.abs(reduced.float().cpu().numpy()[rows] - full_ref)
    bound = tol * rms + 2.0 ** -8 * (mag + np.abs(full_ref))
    assert np.all(diff <= bound), \
        f"reduced partials + shared: max excess {float(np.max(diff - bound)):.3e} (RMS {rms:.3e})"


_EP_RANGES = [[(0, 8), (8, 16), (16, 24), (24, 32)], [(0, 5), (5, 21), (21, 32)]]


@pytest.mark.parametrize("ranges", _EP_RANGES, ids=["even4", "uneven3"])
@pytest.mark.parametrize("fmt", [synth.FMT_BF16, synth.FMT_FP8_B128, synth.FMT_NVFP4])
@pytest.mark.parametrize("n", [1, 3, 16, 40])
def test_expert_parallel_partials(fmt, n, ranges):
    cfg = small(f"ep_{fmt}", expert_fmt=fmt, num_experts=32, top_k=4,
                routing=synth.ROUTE_SIGMOID_BIAS, routed_scaling_factor=2.5, shared_gate=True,
                pre_expert_norm=(n == 16))
    _ep_check(cfg, n, ranges)


@pytest.mark.parametrize("path", ["token_major", "grouped"])
def test_expert_parallel_forced_paths(path):
    cfg = small("ep_paths", num_experts=32, top_k=4, routing=synth.ROUTE_SIGMOID_BIAS,
                routed_scaling_factor=2.5)
    for n in (1, 17):
        _ep_check(cfg, n, _EP_RANGES[1], path=path)


def test_expert_parallel_no_shared_expert_and_empty_rank():
    """No shared expert: a rank that holds no expert at all writes zeros."""
    cfg = small("ep_noshared", shared_inter=0, num_experts=16, top_k=2)
    lw = synth.make_weights(cfg, "cuda")
    x = synth.make_input(cfg, 20, "cuda", gap_fn=gap_fn_for(oracle_layer(lw)))
    for n in (1, 2, 20):
        layer = MoeLayer(synth.expert_slice(lw, 16, 16), n, experts=(16, 16))
        out, _, _ = layer.forward(x[:n], out=torch.full((n, cfg.hidden), 3.0, dtype=torch.bfloat16,
                                                         device="cuda"))
        torch.cuda.synchronize()
        assert int(out.count_nonzero()) == 0
    _ep_check(cfg, 20, [(0, 3), (3, 16)])


def test_accumulate_adds_into_out():
    """accumulate = 1 on a whole layer: BF16(out + layer) on every path."""
    cfg = small("acc", num_experts=32, top_k=4, routing=synth.ROUTE_SIGMOID_BIAS,
                routed_scaling_factor=2.5, shared_gate=True)
    lw = synth.make_weights(cfg, "cuda")
    L = oracle_layer(lw)
    x = synth.make_input(cfg, 40, "cuda", gap_fn=gap_fn_for(L))
    for n in (1, 3, 40):
        base = synth.make_input(cfg.with_(seed=5), n, "cuda")
        plain, _, _ = MoeLayer(lw, n).forward(x[:n])
        got = base.clone()
        MoeLayer(lw, n, accumulate=True).forward(x[:n], out=got)
        torch.cuda.synchronize()
        ref, _, _, _ = O.moe_forward(L, bf16_bits(x[:n]))
        ref = ref + base.float().cpu().numpy()
        rms = float(np.sqrt(np.mean(ref ** 2)))
        assert np.max(np.abs(got.float().cpu().numpy() - ref)) <= 2e-2 * rms
        # Within one BF16 rounding of the two-step sum.
        atol = float(plain.float().abs().max()) * 2 ** -8 + 1e-6
        assert torch.allclose(got.float(), base.float() + plain.float(), rtol=2 ** -8, atol=atol)


def test_expert_parallel_driver_single_rank():
    """Without a process group ExpertParallelMoe is the whole layer: the partial
    of all experts, then the shared expert added."""
    from mixture_experts_decode_router_gb300.ep import ExpertParallelMoe
    cfg = small("ep_driver", num_experts=32, top_k=4, routing=synth.ROUTE_SIGMOID_BIAS,
                routed_scaling_factor=2.5, shared_gate=True, pre_expert_norm=True)
    lw = synth.make_weights(cfg, "cuda")
    L = oracle_layer(lw)
    x = synth.make_input(cfg, 16, "cuda", gap_fn=gap_fn_for(L))
    for n in (1, 16):
        got = ExpertParallelMoe(lw, n, 0, 1).forward(x[:n])
        torch.cuda.synchronize()
        ref, _, _, _ = O.moe_forward(L, bf16_bits(x[:n]))
        part, _, _, _ = O.moe_forward(L, bf16_bits(x[:n]), include_shared=False)
        rms = float(np.sqrt(np.mean(ref ** 2)))
        # Two BF16 roundings: the partial, then the sum with the shared expert.
        bound = 2e-2 * rms + 2.0 ** -8 * (np.abs(part) + np.abs(ref))
        assert np.all(np.abs(got.float().cpu().numpy() - ref) <= bound)


def test_expert_parallel_full_size():
    """decode_n16 over 8 ranks of 32 experts each, with the pre-expert norm."""
    cfg = synth.WORKLOADS["decode_n16"].with_(pre_expert_norm=True)
    _ep_check(cfg, 16, [(32 * r, 32 * r + 32) for r in range(8)], rows=[0, 5, 11, 15])


# ---------------------------------------------------------------- the five workloads at full size

@pytest.mark.parametrize("name", ["tiny_n1", "decode_n1", "decode_n16", "fp8_n64", "nvfp4_n256"])
def test_workloads_full_size(name):
    """Every output row of every workload, element by element (each touched
    expert decoded once for the whole batch)."""
    _check(synth.WORKLOADS[name], threaded=True)


@pytest.mark.parametrize("name", ["decode_n1", "decode_n16", "nvfp4_n256"])
def test_nvfp4_router_full_size(name):
    """The NVFP4 router on the full-size layers (one token: token-major), every row."""
    _check(synth.WORKLOADS[name].with_(router_fmt=synth.FMT_NVFP4), threaded=True)


@pytest.mark.parametrize("name", ["decode_n1", "decode_n16", "nvfp4_n256"])
def test_pre_norm_and_shared_gate_full_size(name):
    """The pre-expert RMSNorm and the shared-expert sigmoid gate on the
    full-size layers (one token: the single-token kernel, which applies both
    itself), every row."""
    _check(synth.WORKLOADS[name].with_(pre_expert_norm=True, shared_gate=True), threaded=True)


# ---------------------------------------------------------------- device error word

def test_workspace_check_clean_after_calls():
    cfg = synth.WORKLOADS["decode_n1"]
    lw = synth.make_weights(cfg, "cuda")
    layer = MoeLayer(lw, 16)
    for n in (1, 16):
        layer.forward(synth.make_input(cfg, n, "cuda"))
    assert layer.device_error() == 0
    # The single-token kernel's grid-barrier words (bytes 12..19 of the
    # control block) are back to zero after every call.
    assert int(layer.ws[12:20].count_nonzero()) == 0


def test_fp8_grouped_combine_waits_for_a_cleared_error():
    """The FP8 grouped path's down kernel also runs the combine, after a grid
    barrier.  With a device error pending (a failed earlier call may have left
    the barrier's count dirty) it does not combine: out is left unwritten, the
    check reports the error and clears the control block, and the next call
    matches the first bit for bit."""
    cfg = small("fp8_pending", expert_fmt=synth.FMT_FP8_B128, num_experts=32, top_k=4)
    lw = synth.make_weights(cfg, "cuda")
    L = oracle_layer(lw)
    x = synth.make_input(cfg, 40, "cuda", gap_fn=gap_fn_for(L))
    layer = MoeLayer(lw, 40)
    good, _, _ = layer.forward(x)
    torch.cuda.synchronize()
    assert layer.device_error() == 0
    layer.ws[8:12] = torch.tensor([5, 0, 0, 0], dtype=torch.uint8, device="cuda")   # Ctrl::err = 5
    sentinel = torch.full_like(good, 7)
    out, _, _ = layer.forward(x, out=sentinel.clone())
    torch.cuda.synchronize()
    assert torch.equal(out, sentinel)          # not combined: nothing written
    assert layer.device_error() == 5           # reported, and cleared
    again, _, _ = layer.forward(x)
    torch.cuda.synchronize()
    assert layer.device_error() == 0
    assert torch.equal(again, good)


def test_single_token_kernel_refuses_a_dirty_control_block():
    cfg = small("dirty", num_experts=32, top_k=4)
    lw = synth.make_weights(cfg, "cuda")
    L = oracle_layer(lw)
    x = synth.make_input(cfg, 1, "cuda", gap_fn=gap_fn_for(L))
    layer = MoeLayer(lw, 1)
    good, _, _ = layer.forward(x)
    torch.cuda.synchronize()
    # A control block that was never zeroed (here: a grid-barrier word of all ones).
    layer.ws[12:16] = 255
    sentinel = torch.full_like(good, 7)
    out, _, _ = layer.forward(x, out=sentinel.clone())
    assert layer.device_error() == 20
    assert torch.equal(out, sentinel)          # refused: nothing written
    layer.ws[:256] = 0
    again, _, _ = layer.forward(x)
    assert layer.device_error() == 0
    assert torch.equal(again, good)
