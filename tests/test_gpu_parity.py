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
"""

import numpy as np
import pytest
import torch

from mixture_experts_decode_router_gb300 import binding as B
from mixture_experts_decode_router_gb300 import synth
from mixture_experts_decode_router_gb300.layer import MoeLayer
from oracle import moe_oracle as O
from tests.moe_helpers import bf16_bits, gap_fn_for, oracle_layer, tolerance

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


def _check(cfg, n=None, path="auto", rows=None, x=None, lw=None):
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
    lg_ref = O.router_logits(O.bf16_decode(xb), L.router_w)
    idx_ref, w_ref = O.route(lg_ref, L.routing, L.top_k, L.norm_topk_prob,
                             L.routed_scaling_factor, L.correction_bias)
    assert np.array_equal(idx.cpu().numpy(), idx_ref), "expert indices differ"
    assert np.max(np.abs(w.cpu().numpy() - w_ref)) <= 1e-5 * max(1.0, cfg.routed_scaling_factor)
    rows = np.arange(n) if rows is None else np.asarray(rows)
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


def test_all_tokens_on_one_expert():
    cfg = small("one_expert", num_experts=16, top_k=2)
    lw = synth.make_weights(cfg, "cuda")
    x1 = synth.make_input(cfg, 1, "cuda", gap_fn=gap_fn_for(oracle_layer(lw)))
    x = x1.repeat(33, 1)      # 33 copies: every route lands on the same two experts
    _check(cfg, 33, x=x, lw=lw)


def test_route_and_experts_entry_points():
    cfg = small("split", routing=synth.ROUTE_SIGMOID_BIAS, top_k=3, routed_scaling_factor=2.5,
                shared_gate=True)
    lw = synth.make_weights(cfg, "cuda")
    L = oracle_layer(lw)
    x = synth.make_input(cfg, 9, "cuda", gap_fn=gap_fn_for(L))
    layer = MoeLayer(lw, 9)
    idx, w, lg = layer.route(x)
    torch.cuda.synchronize()
    lg_ref = O.router_logits(O.bf16_decode(bf16_bits(x)), L.router_w)
    rms = np.sqrt(np.mean(lg_ref ** 2))
    assert np.max(np.abs(lg.cpu().numpy() - lg_ref)) <= 1e-4 * rms
    # moe_experts on the oracle's routing (as int32/fp32), then against the oracle output.
    idx_ref, w_ref = O.route(lg_ref, L.routing, L.top_k, L.norm_topk_prob,
                             L.routed_scaling_factor, L.correction_bias)
    out = layer.experts(x, torch.from_numpy(idx_ref.astype(np.int32)).cuda(),
                        torch.from_numpy(w_ref.astype(np.float32)).cuda())
    fwd, _, _ = layer.forward(x)
    torch.cuda.synchronize()
    ref, _, _, _ = O.moe_forward(L, bf16_bits(x))
    rms_o = np.sqrt(np.mean(ref ** 2))
    assert np.max(np.abs(out.float().cpu().numpy() - ref)) <= 2e-2 * rms_o
    assert torch.equal(out, fwd)


def test_zero_tokens_is_a_noop():
    cfg = small("empty")
    lw = synth.make_weights(cfg, "cuda")
    layer = MoeLayer(lw, 4)
    x = torch.empty(0, cfg.hidden, dtype=torch.bfloat16, device="cuda")
    out, idx, w = layer.forward(x)
    torch.cuda.synchronize()
    assert out.shape == (0, cfg.hidden)


@pytest.mark.parametrize("fmt", [synth.FMT_BF16, synth.FMT_FP8_B128, synth.FMT_NVFP4])
def test_rows_do_not_depend_on_the_batch_token_major(fmt):
    """The token-major kernels (forced), and one token alone: the single-token
    kernel, which keeps the token-major arithmetic."""
    cfg = small("invariance", expert_fmt=fmt, num_experts=32, top_k=4,
                routing=synth.ROUTE_SIGMOID_BIAS, routed_scaling_factor=2.5)
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


@pytest.mark.parametrize("fmt", [synth.FMT_BF16, synth.FMT_FP8_B128, synth.FMT_NVFP4])
def test_rows_do_not_depend_on_the_batch_grouped(fmt):
    """N >= 4: the expert-grouped tensor-core path."""
    cfg = small("invariance_g", expert_fmt=fmt, num_experts=32, top_k=4,
                routing=synth.ROUTE_SIGMOID_BIAS, routed_scaling_factor=2.5)
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


# ---------------------------------------------------------------- the five workloads at full size

@pytest.mark.parametrize("name,rows", [
    ("tiny_n1", None),
    ("decode_n1", None),
    ("decode_n16", None),
    ("fp8_n64", [0, 9, 31, 32, 50, 63]),
    ("nvfp4_n256", list(range(0, 256, 8)) + [255]),
])
def test_workloads_full_size(name, rows):
    cfg = synth.WORKLOADS[name]
    _check(cfg, rows=rows)


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
