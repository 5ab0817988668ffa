"""Pins of the fp64 oracle to facts outside itself (CPU only).

Each test checks an oracle function against something the format definitions,
the mathematics or a library routine fixes: printed code tables, closed forms,
brute force over all subsets, pure-Python loop evaluations on tiny layers, and
invariants (weights summing to routed_scaling_factor, row-grouping
invariance).  A plausible mistake in the oracle (a swapped nibble, a wrong
exponent bias, a transposed router, a dropped shared expert, a bias that leaks
into the weights) fails at least one of them.
"""

import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import moe_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "fp_formats.json")


def _golden():
    with open(GOLDEN) as f:
        return json.load(f)


def _same(a, b):
    if isinstance(b, str) and b == "nan":
        return math.isnan(a)
    return a == b and math.copysign(1.0, a) == math.copysign(1.0, b)


# ------------------------------------------------------------------ formats

def test_bf16_anchor_values():
    for code, val in _golden()["bf16"]:
        assert _same(float(O.bf16_decode(int(code, 16))), val), code


def test_bf16_all_codes_match_torch():
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = O.bf16_decode(codes)
    ref = torch.from_numpy(codes.view(np.int16)).view(torch.bfloat16).double().numpy()
    finite = np.isfinite(ref)
    assert np.array_equal(ours[finite], ref[finite])
    assert np.array_equal(np.isnan(ours), np.isnan(ref))


def test_e4m3_anchor_values():
    for code, val in _golden()["e4m3"]:
        assert _same(float(O.e4m3_decode(int(code, 16))), val), code


def test_e4m3_all_codes_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    ours = O.e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    # Exactly two NaN codes and no infinity in the "fn" variant.
    assert nan.sum() == 2 and not np.isinf(ours).any()


def test_e2m1_table():
    table = _golden()["e2m1"]
    ours = O.e2m1_decode(np.arange(16, dtype=np.uint8))
    for c in range(16):
        assert _same(float(ours[c]), table[c]), c


def test_dequant_fp8_block_scale_ragged():
    rng = np.random.default_rng(1)
    out_d, in_d = 200, 300          # ragged edge tiles in both directions
    scale = rng.uniform(0.5, 2.0, size=(2, 3)).astype(np.float32)
    q = np.full((out_d, in_d), 0x38, dtype=np.uint8)    # E4M3 1.0 everywhere
    w = O.dequant_fp8_b128(q, scale)
    for o, i in [(0, 0), (127, 127), (128, 127), (127, 128), (199, 299), (150, 260), (5, 256)]:
        assert w[o, i] == float(scale[o // 128, i // 128]), (o, i)
    # Unit scales give the element table back.
    codes = rng.integers(0, 256, size=(out_d, in_d), dtype=np.uint8)
    codes[codes & 0x7F == 0x7F] = 0x38
    w1 = O.dequant_fp8_b128(codes, np.ones((2, 3), np.float32))
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    assert np.array_equal(w1, ref)


def test_dequant_nvfp4_nibble_order_and_scales():
    out_d, in_d = 2, 64
    packed = np.zeros((out_d, in_d // 2), dtype=np.uint8)
    packed[0, 0] = 0x21          # element 0 <- low nibble 1 (0.5), element 1 <- high nibble 2 (1.0)
    packed[0, 8] = 0xF7          # elements 16, 17 <- 7 (6.0), 15 (-6.0)
    packed[1, 31] = 0x9B         # elements 62, 63 <- 11 (-1.5), 9 (-0.5)
    s16 = np.full((out_d, in_d // 16), 0x38, dtype=np.uint8)   # 1.0
    s16[0, 1] = 0x40             # elements 16..31 of row 0 scaled by 2
    s16[1, 3] = 0x30             # elements 48..63 of row 1 scaled by 0.5
    w = O.dequant_nvfp4(packed, s16, 0.25)
    expect = np.zeros((out_d, in_d))
    expect[0, 0], expect[0, 1] = 0.5 * 0.25, 1.0 * 0.25
    expect[0, 16], expect[0, 17] = 6.0 * 2 * 0.25, -6.0 * 2 * 0.25
    expect[1, 62], expect[1, 63] = -1.5 * 0.5 * 0.25, -0.5 * 0.5 * 0.25
    assert np.array_equal(w, expect)


# ------------------------------------------------------------------ router

def _bf16_bits(a):
    return torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16).view(torch.int16) \
        .numpy().view(np.uint16)


def test_router_one_hot_picks_a_column():
    rng = np.random.default_rng(2)
    wr = _bf16_bits(rng.normal(size=(5, 7)))
    x = np.zeros((1, 7)); x[0, 3] = 1.0
    l = O.router_logits(x, wr)
    assert np.array_equal(l[0], O.bf16_decode(wr)[:, 3])


def test_router_matches_python_loops():
    rng = np.random.default_rng(3)
    E, H, N = 4, 6, 3
    wr = _bf16_bits(rng.normal(size=(E, H)))
    x = rng.normal(size=(N, H))
    l = O.router_logits(x, wr)
    wv = [[float(O.bf16_decode(wr[e, h])) for h in range(H)] for e in range(E)]
    for t in range(N):
        for e in range(E):
            s = sum(float(x[t, h]) * wv[e][h] for h in range(H))
            assert abs(l[t, e] - s) <= 1e-12 * (1 + abs(s))


# ------------------------------------------------------------------ top-k

@pytest.mark.parametrize("E,k", [(4, 1), (6, 2), (8, 3), (10, 3), (16, 2)])
def test_topk_brute_force_over_subsets(E, k):
    rng = np.random.default_rng(E * 10 + k)
    for trial in range(30):
        s = rng.integers(-3, 4, size=(1, E)).astype(np.float64)   # many exact ties
        if trial % 3 == 0:
            s = rng.normal(size=(1, E))
        sel = O.topk_select(s, k)[0]
        # The set must be one the brute force accepts: every chosen score >= every other.
        valid = [set(c) for c in itertools.combinations(range(E), k)
                 if min(s[0, list(c)]) >= max(np.delete(s[0], list(c)), default=-np.inf)]
        assert set(sel.tolist()) in valid
        # Among valid sets, ties go to the lower indices: the lexicographically smallest
        # sorted index tuple among sets with the maximal score multiset.
        best = min(valid, key=lambda c: sorted(c))
        assert sorted(sel.tolist()) == sorted(best)
        # Slots in descending score, equal scores by ascending index.
        keys = [(-s[0, e], e) for e in sel]
        assert keys == sorted(keys)


def test_topk_gap():
    s = np.array([[0.1, 0.5, 0.3, 0.45]])
    assert abs(O.topk_gap(s, 1)[0] - 0.05) < 1e-15
    assert abs(O.topk_gap(s, 2)[0] - 0.15) < 1e-15
    assert O.topk_gap(s, 4)[0] == np.inf


# ------------------------------------------------------------------ weights

def test_softmax_two_expert_closed_form():
    l = np.array([[0.0, math.log(3.0)]])
    idx, w = O.route(l, O.ROUTE_SOFTMAX, 2, False, 1.0)
    assert idx[0].tolist() == [1, 0]
    assert abs(w[0, 0] - 0.75) < 1e-15 and abs(w[0, 1] - 0.25) < 1e-15


@pytest.mark.parametrize("routing", [O.ROUTE_SOFTMAX, O.ROUTE_SIGMOID_BIAS])
@pytest.mark.parametrize("scale", [1.0, 2.5])
def test_renormalised_weights_sum_to_scale(routing, scale):
    rng = np.random.default_rng(5)
    l = rng.normal(size=(50, 32))
    bias = rng.uniform(-0.1, 0.1, size=32) if routing == O.ROUTE_SIGMOID_BIAS else None
    _, w = O.route(l, routing, 8, True, scale, bias)
    assert np.all(np.abs(w.sum(axis=1) - scale) <= 1e-12)
    assert np.all(w > 0)


def test_all_experts_softmax_equals_full_softmax():
    rng = np.random.default_rng(6)
    l = rng.normal(size=(3, 9))
    idx, w = O.route(l, O.ROUTE_SOFTMAX, 9, True, 1.7)
    full = torch.softmax(torch.from_numpy(l), dim=1).numpy()
    assert np.allclose(w, np.take_along_axis(full, idx, 1) * 1.7, atol=1e-14, rtol=0)


def test_top1_renormalised_weight_is_scale():
    rng = np.random.default_rng(7)
    l = rng.normal(size=(10, 12))
    _, w = O.route(l, O.ROUTE_SIGMOID_BIAS, 1, True, 2.5, np.zeros(12))
    assert np.all(w == 2.5)


def test_sigmoid_weight_of_zero_logit_and_bias_only_selects():
    l = np.array([[0.0, 0.2, -0.1]])
    # The bias lifts expert 2 over expert 1 for selection ...
    idx, w = O.route(l, O.ROUTE_SIGMOID_BIAS, 2, False, 3.0, np.array([0.0, 0.0, 0.2]))
    assert idx[0].tolist() == [2, 1]
    # ... but the weights stay sigmoid(logit) * scale (sigmoid(-0.1), sigmoid(0.2)).
    assert abs(w[0, 0] - 3.0 / (1 + math.exp(0.1))) < 1e-15
    assert abs(w[0, 1] - 3.0 / (1 + math.exp(-0.2))) < 1e-15
    idx0, w0 = O.route(np.zeros((1, 3)), O.ROUTE_SIGMOID_BIAS, 1, False, 2.0, np.zeros(3))
    assert idx0[0, 0] == 0 and w0[0, 0] == 1.0       # sigmoid(0) = 1/2, tie -> index 0


# ------------------------------------------------------------------ experts and blend

def test_silu_values():
    assert O.silu(0.0) == 0.0
    assert abs(O.silu(1.0) - 0.7310585786300049) < 1e-15
    assert abs(O.silu(-1.0) + 0.2689414213699951) < 1e-15


def test_swiglu_scalar_hand_case():
    # x = 2, Wg = 1, Wu = 3, Wd = 0.5: g = 2, u = 6, d = 0.5 * SiLU(2) * 6.
    d = O.swiglu_mlp(np.array([2.0]), np.array([[1.0]]), np.array([[3.0]]), np.array([[0.5]]))
    assert abs(d[0] - 0.5 * 6.0 * 2.0 / (1.0 + math.exp(-2.0))) < 1e-14


def test_swiglu_one_hot_columns():
    rng = np.random.default_rng(8)
    wg, wu, wd = rng.normal(size=(3, 5)), rng.normal(size=(3, 5)), rng.normal(size=(5, 3))
    x = np.zeros(5); x[2] = 1.0
    g, u = wg[:, 2], wu[:, 2]
    expect = wd @ (g / (1 + np.exp(-g)) * u)
    assert np.allclose(O.swiglu_mlp(x, wg, wu, wd), expect, rtol=0, atol=1e-15)


def _tiny_layer(rng, fmt=O.FMT_BF16, E=5, H=64, I=32, S=32, k=2, routing=O.ROUTE_SOFTMAX,
                norm=True, scale=1.0, shared_gate=False):
    def bits(shape, std=0.3):
        return _bf16_bits(rng.normal(size=shape) * std)

    def qmat(e, out_d, in_d):
        if fmt == O.FMT_BF16:
            return O.QMat(fmt, bits((e, out_d, in_d)))
        if fmt == O.FMT_FP8_B128:
            q = rng.integers(0, 256, size=(e, out_d, in_d), dtype=np.uint8)
            q[(q & 0x7F) == 0x7F] = 0x38
            sc = rng.uniform(0.001, 0.01, size=(e, -(-out_d // 128), -(-in_d // 128)))
            return O.QMat(fmt, q, sc.astype(np.float32))
        p = rng.integers(0, 256, size=(e, out_d, in_d // 2), dtype=np.uint8)
        s16 = rng.integers(0x20, 0x48, size=(e, out_d, in_d // 16), dtype=np.uint8)
        s2 = rng.uniform(0.01, 0.1, size=e).astype(np.float32)
        return O.QMat(fmt, p, s16, s2)

    bias = rng.uniform(-0.1, 0.1, size=E).astype(np.float32) \
        if routing == O.ROUTE_SIGMOID_BIAS else None
    return O.OracleLayer(
        hidden=H, num_experts=E, top_k=k, inter=I, shared_inter=S, routing=routing,
        norm_topk_prob=norm, routed_scaling_factor=scale, router_w=bits((E, H)),
        gate=qmat(E, I, H), up=qmat(E, I, H), down=qmat(E, H, I),
        sh_gate=qmat(1, S, H) if S else None, sh_up=qmat(1, S, H) if S else None,
        sh_down=qmat(1, H, S) if S else None, correction_bias=bias,
        shared_gate_w=bits((H,)) if shared_gate else None)


def _python_loop_forward(L, xb):
    """The layer for one token in plain Python loops over scalars."""
    x = [float(v) for v in O.bf16_decode(xb)]
    H, E, k = L.hidden, L.num_experts, L.top_k
    wr = L.router_q.expert(0) if L.router_q is not None else O.bf16_decode(L.router_w)
    logit = [sum(x[h] * float(wr[e, h]) for h in range(H)) for e in range(E)]
    if L.routing == O.ROUTE_SOFTMAX:
        m = max(logit)
        z = [math.exp(v - m) for v in logit]
        p = [v / sum(z) for v in z]
        score = logit
    else:
        p = [1 / (1 + math.exp(-v)) for v in logit]
        score = [p[e] + float(L.correction_bias[e]) for e in range(E)]
    order = sorted(range(E), key=lambda e: (-score[e], e))[:k]
    wsel = [p[e] for e in order]
    if L.norm_topk_prob:
        tot = sum(wsel)
        wsel = [v / tot for v in wsel]
    wsel = [v * L.routed_scaling_factor for v in wsel]

    xe = x
    if L.pre_expert_norm_w is not None:
        nw = O.bf16_decode(L.pre_expert_norm_w)
        inv = 1.0 / math.sqrt(sum(v * v for v in x) / H + L.rms_norm_eps)
        xe = [x[h] * inv * float(nw[h]) for h in range(H)]

    def mlp(wg, wu, wd):
        inner = wg.shape[0]
        g = [sum(float(wg[i, h]) * xe[h] for h in range(H)) for i in range(inner)]
        u = [sum(float(wu[i, h]) * xe[h] for h in range(H)) for i in range(inner)]
        a = [g[i] / (1 + math.exp(-g[i])) * u[i] for i in range(inner)]
        return [sum(float(wd[o, i]) * a[i] for i in range(inner)) for o in range(H)]

    out = [0.0] * H
    for j, e in enumerate(order):
        d = mlp(L.gate.expert(e), L.up.expert(e), L.down.expert(e))
        out = [out[o] + wsel[j] * d[o] for o in range(H)]
    if L.shared_inter:
        ds = mlp(L.sh_gate.expert(0), L.sh_up.expert(0), L.sh_down.expert(0))
        gs = 1.0
        if L.shared_gate_w is not None:
            gw = O.bf16_decode(L.shared_gate_w)
            gs = 1 / (1 + math.exp(-sum(x[h] * float(gw[h]) for h in range(H))))
        out = [out[o] + gs * ds[o] for o in range(H)]
    return np.array(out), order, wsel


@pytest.mark.parametrize("fmt", [O.FMT_BF16, O.FMT_FP8_B128, O.FMT_NVFP4])
@pytest.mark.parametrize("routing,norm,scale,sg", [
    (O.ROUTE_SOFTMAX, True, 1.0, False), (O.ROUTE_SIGMOID_BIAS, True, 2.5, True),
    (O.ROUTE_SIGMOID_BIAS, False, 1.5, False), (O.ROUTE_SOFTMAX, False, 1.0, True)])
def test_forward_matches_python_loops(fmt, routing, norm, scale, sg):
    rng = np.random.default_rng(11)
    L = _tiny_layer(rng, fmt, E=5, H=32, I=32, S=32, k=2, routing=routing, norm=norm,
                    scale=scale, shared_gate=sg)
    xb = _bf16_bits(rng.normal(size=(3, 32)))
    out, idx, w, _ = O.moe_forward(L, xb)
    for t in range(3):
        ref, order, wsel = _python_loop_forward(L, xb[t])
        assert idx[t].tolist() == order
        assert np.allclose(w[t], wsel, rtol=0, atol=1e-13)
        assert np.allclose(out[t], ref, rtol=1e-11, atol=1e-12)


def test_expert_major_equals_slotwise():
    rng = np.random.default_rng(12)
    L = _tiny_layer(rng, O.FMT_NVFP4, E=6, H=64, I=32, S=32, k=3,
                    routing=O.ROUTE_SIGMOID_BIAS, scale=2.5)
    xb = _bf16_bits(rng.normal(size=(9, 64)))
    a, ia, wa, _ = O.moe_forward(L, xb)
    b, ib, wb = O.moe_forward_slotwise(L, xb)
    assert np.array_equal(ia, ib) and np.array_equal(wa, wb)
    assert np.allclose(a, b, rtol=1e-12, atol=1e-14)


def test_single_expert_layer_is_two_textbook_mlps():
    rng = np.random.default_rng(13)
    L = _tiny_layer(rng, O.FMT_BF16, E=1, H=32, I=32, S=32, k=1)
    xb = _bf16_bits(rng.normal(size=(4, 32)))
    out, idx, w, _ = O.moe_forward(L, xb)
    assert np.all(idx == 0) and np.all(w == 1.0)
    x = torch.from_numpy(O.bf16_decode(xb))

    def mlp_torch(q_g, q_u, q_d):
        g = x @ torch.from_numpy(q_g.expert(0)).T
        u = x @ torch.from_numpy(q_u.expert(0)).T
        return (torch.nn.functional.silu(g) * u) @ torch.from_numpy(q_d.expert(0)).T

    ref = mlp_torch(L.gate, L.up, L.down) + mlp_torch(L.sh_gate, L.sh_up, L.sh_down)
    assert np.allclose(out, ref.numpy(), rtol=1e-12, atol=1e-13)


def test_blend_special_cases():
    rng = np.random.default_rng(14)
    L = _tiny_layer(rng, O.FMT_BF16, E=4, H=32, I=32, S=32, k=2)
    xb = _bf16_bits(rng.normal(size=(3, 32)))
    x = O.bf16_decode(xb)
    shared = O.swiglu_mlp(x, L.sh_gate.expert(0), L.sh_up.expert(0), L.sh_down.expert(0))
    # Routed weights scaled to zero: only the shared expert remains.
    L.routed_scaling_factor = 0.0
    out, _, _, _ = O.moe_forward(L, xb)
    assert np.array_equal(out, shared)
    # No shared expert: only the routed sum remains.
    L.routed_scaling_factor = 1.0
    L2 = O.OracleLayer(**{**L.__dict__, "shared_inter": 0, "sh_gate": None, "sh_up": None,
                          "sh_down": None, "_cache": {}})
    routed, idx, w, _ = O.moe_forward(L2, xb)
    full, _, _, _ = O.moe_forward(L, xb)
    assert np.allclose(full - routed, shared, rtol=0, atol=1e-14)
    # Shared gate: sigmoid(x . gw) scales the shared expert only.
    gw = _bf16_bits(rng.normal(size=32))
    L3 = O.OracleLayer(**{**L.__dict__, "shared_gate_w": gw, "_cache": {}})
    gated, _, _, _ = O.moe_forward(L3, xb)
    gs = 1 / (1 + np.exp(-(x @ O.bf16_decode(gw))))
    assert np.allclose(gated - routed, gs[:, None] * shared, rtol=0, atol=1e-14)


def test_rows_do_not_depend_on_grouping():
    rng = np.random.default_rng(15)
    L = _tiny_layer(rng, O.FMT_FP8_B128, E=8, H=128, I=64, S=64, k=3,
                    routing=O.ROUTE_SIGMOID_BIAS, scale=2.5)
    xb = _bf16_bits(rng.normal(size=(12, 128)))
    full, idx, w, _ = O.moe_forward(L, xb)
    perm = rng.permutation(12)
    p_out, p_idx, p_w, _ = O.moe_forward(L, xb[perm])
    assert np.array_equal(p_out, full[perm]) and np.array_equal(p_idx, idx[perm])
    for r in (0, 5, 11):
        one, i1, w1, _ = O.moe_forward(L, xb, rows=[r])
        assert np.array_equal(one[0], full[r]) and np.array_equal(i1[0], idx[r])
    dup = np.concatenate([xb, xb[:4]])
    d_out, _, _, _ = O.moe_forward(L, dup)
    assert np.array_equal(d_out[12:], full[:4])


# ------------------------------------------------------------------ next rows

def test_rms_norm_closed_form_and_scale_invariance():
    x = np.array([[3.0, 4.0]])
    w = _bf16_bits(np.array([1.0, 2.0]))
    y = O.rms_norm(x, w, 0.0)
    r = math.sqrt(12.5)
    assert abs(y[0, 0] - 3.0 / r) < 1e-15 and abs(y[0, 1] - 8.0 / r) < 1e-15
    rng = np.random.default_rng(21)
    xs = rng.normal(size=(4, 64))
    ws = _bf16_bits(rng.normal(size=64))
    assert np.array_equal(O.rms_norm(2.0 * xs, ws, 0.0), O.rms_norm(xs, ws, 0.0))
    # eps moves the result toward zero by the closed-form factor
    y1 = O.rms_norm(x, w, 3.5)
    assert abs(y1[0, 0] - 3.0 / 4.0) < 1e-15


@pytest.mark.parametrize("fmt", [O.FMT_BF16, O.FMT_NVFP4])
def test_pre_expert_norm_matches_python_loops(fmt):
    rng = np.random.default_rng(22)
    L = _tiny_layer(rng, fmt, E=5, H=32, I=32, S=32, k=2, routing=O.ROUTE_SIGMOID_BIAS,
                    scale=2.5, shared_gate=True)
    L.pre_expert_norm_w = _bf16_bits(rng.uniform(0.5, 1.5, size=32))
    L.rms_norm_eps = 1e-5
    xb = _bf16_bits(rng.normal(size=(3, 32)) * 3.0)
    out, idx, w, _ = O.moe_forward(L, xb)
    for t in range(3):
        ref, order, wsel = _python_loop_forward(L, xb[t])
        assert idx[t].tolist() == order
        assert np.allclose(out[t], ref, rtol=1e-11, atol=1e-12)


def test_nvfp4_router_matches_python_loops():
    rng = np.random.default_rng(23)
    L = _tiny_layer(rng, O.FMT_BF16, E=6, H=64, I=32, S=32, k=2)
    p = rng.integers(0, 256, size=(1, 6, 32), dtype=np.uint8)
    s16 = rng.integers(0x30, 0x40, size=(1, 6, 4), dtype=np.uint8)
    L.router_q = O.QMat(O.FMT_NVFP4, p, s16, np.array([0.05], np.float32))
    xb = _bf16_bits(rng.normal(size=(3, 64)))
    out, idx, w, lg = O.moe_forward(L, xb)
    wr = O.dequant_nvfp4(p[0], s16[0], float(np.float32(0.05)))
    assert np.allclose(lg, O.bf16_decode(xb) @ wr.T, rtol=1e-13, atol=1e-14)
    for t in range(3):
        ref, order, _ = _python_loop_forward(L, xb[t])
        assert idx[t].tolist() == order
        assert np.allclose(out[t], ref, rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("ranks", [2, 3, 5])
def test_expert_parallel_partials_sum_to_the_layer(ranks):
    """Each rank keeps its experts' routes, the shared expert is left out of
    every partial and added once after the sum (the EP branch)."""
    rng = np.random.default_rng(24)
    L = _tiny_layer(rng, O.FMT_FP8_B128, E=10, H=128, I=64, S=64, k=3,
                    routing=O.ROUTE_SIGMOID_BIAS, scale=2.5, shared_gate=True)
    xb = _bf16_bits(rng.normal(size=(7, 128)))
    full, idx, w, _ = O.moe_forward(L, xb)
    bounds = np.linspace(0, 10, ranks + 1).astype(int)
    parts = [O.moe_forward(L, xb, experts=(bounds[r], bounds[r + 1]), include_shared=False)[0]
             for r in range(ranks)]
    shared_only = O.moe_forward(L, xb, experts=(0, 0), include_shared=True)[0]
    assert np.allclose(sum(parts) + shared_only, full, rtol=1e-12, atol=1e-13)
    # A rank whose experts no token chose contributes exactly zero.
    unused = sorted(set(range(10)) - set(idx.ravel().tolist()))
    if unused:
        e = unused[0]
        z = O.moe_forward(L, xb, experts=(e, e + 1), include_shared=False)[0]
        assert not z.any()
