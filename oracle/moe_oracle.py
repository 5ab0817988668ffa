"""fp64 CPU oracle for the Mixture-of-Experts decode-layer forward.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this module:
only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
(and its ``--impl reference`` arm) may call it.  It shares no code with the CUDA
path: every decoding rule and every step of the layer is written out here again,
plainly, in numpy float64.

What it computes, per token ``t`` (the method of the pages
"metrale_model_layers/layers/moe/forward.rs" (``MoeLayer::forward``) and
"spark_model/layers/moe/forward_token_major.rs" (``forward_token_major_decode``)):

1. router logits ``l[t,e] = sum_h x[t,h] * Wr[e,h]``        (the ``gate`` step);
2. the selection score ``c``: the logit itself for softmax routing (softmax is
   monotone), or ``sigmoid(l) + bias`` for sigmoid routing with a correction
   bias; the top-k experts are the k largest ``c``, ties to the lower expert
   index, slots ordered by descending ``c``          (the ``topk`` step);
3. routing weights: softmax ``p = exp(l - max) / sum_all exp(l - max)`` or
   sigmoid ``p = sigmoid(l)`` (the bias never enters a weight); if
   ``norm_topk_prob`` the k selected ``p`` are divided by their sum; every
   weight is then multiplied by ``routed_scaling_factor``;
4. per slot j with expert ``e``: ``g = Wg[e] x``, ``u = Wu[e] x``,
   ``a = SiLU(g) * u`` with ``SiLU(g) = g / (1 + exp(-g))``, ``d = Wd[e] a``
   (the ``exp_gate_up`` / ``exp_silu_down`` steps);
5. the always-on shared expert, the same SwiGLU with its own three matrices;
6. ``out = sum_j w_j d_j + g_s * d_shared`` with ``g_s = sigmoid(x . gw)`` when a
   shared-expert gate weight is given, else 1 (the ``wsum_blend`` step).

Weight formats (decoded exactly, from the format definitions):

* BF16: the upper 16 bits of an IEEE-754 binary32.
* FP8 E4M3 (OCP 8-bit floating point, "fn" variant): sign, 4 exponent bits with
  bias 7, 3 mantissa bits; exponent field 0 is subnormal; ``S.1111.111`` is NaN;
  there is no infinity.  Block-scaled: one fp32 scale per 128x128 tile of the
  ``[out, in]`` matrix (ragged edge tiles allowed); ``w = e4m3(q) * scale``.
* NVFP4: E2M1 elements (sign, 2 exponent bits with bias 1, 1 mantissa bit:
  magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6), two per byte with the even element in
  the low nibble, one E4M3 scale per 16 consecutive elements along ``in``, and
  one fp32 ``scale2`` per (expert, matrix): ``w = e2m1(q) * e4m3(s16) * scale2``.

Expert matrices are decoded one expert at a time, so the largest layer (256
experts of 3 x 7168 x 2048 FP8 weights) never has to exist in float64 at once.

Readings taken where the pages leave a step open are stated beside the step.
Every function here is pinned by ``tests/test_oracle_pins.py`` against values
fixed by the format definitions, closed forms, brute force or a library
routine; none is marked "parity unpinned".
"""

from __future__ import annotations

from dataclasses import dataclass, field
from typing import Dict, Optional

import numpy as np

ROUTE_SOFTMAX = "softmax"
ROUTE_SIGMOID_BIAS = "sigmoid_bias"
FMT_BF16 = "bf16"
FMT_FP8_B128 = "fp8_b128"
FMT_NVFP4 = "nvfp4"

FP8_BLOCK = 128      # FP8 scale tile edge (rows and columns of [out, in])
NVFP4_BLOCK = 16     # NVFP4 elements per E4M3 scale, along `in`


# --------------------------------------------------------------------------
# Element decoders (format definitions)
# --------------------------------------------------------------------------

def bf16_decode(bits) -> np.ndarray:
    """BF16 bit patterns (uint16) -> float64.  BF16 is the high half of a
    binary32, so the value is the binary32 whose low 16 bits are zero."""
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def e4m3_decode(codes) -> np.ndarray:
    """FP8 E4M3 ("fn": no infinities, NaN only at S.1111.111) -> float64."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where((c >> 7) & 1, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    normal = (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0)
    subnormal = (m / 8.0) * np.exp2(-6.0)
    mag = np.where(e == 0, subnormal, normal)
    mag = np.where((e == 0xF) & ((c & 0x7) == 0x7), np.nan, mag)
    return sign * mag


def e2m1_decode(nibbles) -> np.ndarray:
    """FP4 E2M1 codes (0..15) -> float64: bit 3 sign, bits 2..1 exponent
    (bias 1), bit 0 mantissa; exponent 0 is subnormal (0 or 0.5)."""
    n = np.asarray(nibbles, dtype=np.uint8).astype(np.int64) & 0xF
    sign = np.where((n >> 3) & 1, -1.0, 1.0)
    e = (n >> 1) & 0x3
    m = (n & 0x1).astype(np.float64)
    normal = (1.0 + m / 2.0) * np.exp2(e.astype(np.float64) - 1.0)
    subnormal = m * 0.5
    return sign * np.where(e == 0, subnormal, normal)


# --------------------------------------------------------------------------
# Matrix dequantisation (one [out, in] matrix of one expert)
# --------------------------------------------------------------------------

def dequant_bf16(w_bits: np.ndarray) -> np.ndarray:
    return bf16_decode(w_bits)


def dequant_fp8_b128(q: np.ndarray, scale: np.ndarray) -> np.ndarray:
    """w[o, i] = e4m3(q[o, i]) * scale[o // 128, i // 128]."""
    out_dim, in_dim = q.shape
    vals = e4m3_decode(q)
    s = np.asarray(scale, dtype=np.float64)
    rows = np.arange(out_dim) // FP8_BLOCK
    cols = np.arange(in_dim) // FP8_BLOCK
    return vals * s[rows][:, cols]


def dequant_nvfp4(packed: np.ndarray, s16: np.ndarray, scale2: float) -> np.ndarray:
    """w[o, i] = e2m1(nibble(o, i)) * e4m3(s16[o, i // 16]) * scale2, where the
    element with even ``i`` sits in the low nibble of byte ``i // 2``."""
    p = np.asarray(packed, dtype=np.uint8)
    out_dim, half = p.shape
    in_dim = 2 * half
    codes = np.empty((out_dim, in_dim), dtype=np.uint8)
    codes[:, 0::2] = p & 0x0F
    codes[:, 1::2] = p >> 4
    vals = e2m1_decode(codes)
    blk = e4m3_decode(s16)[:, np.arange(in_dim) // NVFP4_BLOCK]
    return vals * blk * float(scale2)


# --------------------------------------------------------------------------
# Layer description (host copies of what the C-ABI receives)
# --------------------------------------------------------------------------

@dataclass
class QMat:
    """One stacked expert matrix in the library's layout (host numpy).

    bf16:     w uint16 [E, out, in]
    fp8_b128: w uint8 [E, out, in], scale float32 [E, ceil(out/128), ceil(in/128)]
    nvfp4:    w uint8 [E, out, in/2], scale uint8 (E4M3) [E, out, in/16],
              scale2 float32 [E]
    """
    fmt: str
    w: np.ndarray
    scale: Optional[np.ndarray] = None
    scale2: Optional[np.ndarray] = None

    def expert(self, e: int) -> np.ndarray:
        """Decoded float64 [out, in] of expert e."""
        if self.fmt == FMT_BF16:
            return dequant_bf16(self.w[e])
        if self.fmt == FMT_FP8_B128:
            return dequant_fp8_b128(self.w[e], self.scale[e])
        if self.fmt == FMT_NVFP4:
            return dequant_nvfp4(self.w[e], self.scale[e], float(self.scale2[e]))
        raise ValueError(f"unknown format {self.fmt}")


@dataclass
class OracleLayer:
    hidden: int
    num_experts: int
    top_k: int
    inter: int
    shared_inter: int
    routing: str
    norm_topk_prob: bool
    routed_scaling_factor: float
    router_w: np.ndarray                       # uint16 BF16 [E, H]
    gate: QMat                                 # [E, I, H]
    up: QMat                                   # [E, I, H]
    down: QMat                                 # [E, H, I]
    sh_gate: Optional[QMat] = None             # [1, S, H]
    sh_up: Optional[QMat] = None               # [1, S, H]
    sh_down: Optional[QMat] = None             # [1, H, S]
    correction_bias: Optional[np.ndarray] = None   # float32 [E]
    shared_gate_w: Optional[np.ndarray] = None     # uint16 BF16 [H]
    pre_expert_norm_w: Optional[np.ndarray] = None  # uint16 BF16 [H] (RMSNorm weight) or None
    rms_norm_eps: float = 1e-6
    router_q: Optional["QMat"] = None              # NVFP4 router [1, E, H]; replaces router_w
    _cache: Dict = field(default_factory=dict, repr=False)


# --------------------------------------------------------------------------
# Routing: router, selection, weights
# --------------------------------------------------------------------------

def router_logits(x: np.ndarray, router_w_bits) -> np.ndarray:
    """Router logits [N, E] = x [N, H] . Wr[E, H]^T, all in float64 (the
    ``gate`` step: ``decode_gate_gemv`` for one row, ``dense_gemm`` for N).
    ``router_w_bits``: BF16 bits [E, H], or an already decoded float matrix."""
    wr = router_w_bits if np.asarray(router_w_bits).dtype == np.float64 else bf16_decode(router_w_bits)
    x = np.atleast_2d(np.asarray(x, dtype=np.float64))
    # One matrix-vector product per row, so a row's logits never depend on
    # which other rows are in the call (a batched BLAS product may block them).
    return np.stack([wr @ x[t] for t in range(x.shape[0])]) if x.shape[0] else \
        np.zeros((0, wr.shape[0]))


def rms_norm(x: np.ndarray, w_bits: np.ndarray, eps: float) -> np.ndarray:
    """RMSNorm of each row of x: x / sqrt(mean(x^2) + eps) * w (the
    ``pre_expert_norm`` step of MoeLayer::forward: the expert input only)."""
    x = np.atleast_2d(np.asarray(x, dtype=np.float64))
    w = bf16_decode(w_bits)
    ms = np.array([float(x[t] @ x[t]) / x.shape[1] for t in range(x.shape[0])])
    return x / np.sqrt(ms + eps)[:, None] * w


def router_weights(layer) -> np.ndarray:
    """The router matrix [E, H] in float64: BF16, or NVFP4 (``gate_nvfp4``)."""
    if layer.router_q is not None:
        return layer.router_q.expert(0)
    return bf16_decode(layer.router_w)


def sigmoid(v):
    return 1.0 / (1.0 + np.exp(-np.asarray(v, dtype=np.float64)))


def selection_scores(logits: np.ndarray, routing: str,
                     bias: Optional[np.ndarray] = None) -> np.ndarray:
    """The score the top-k selection ranks.  Softmax routing ranks the logits
    (softmax is strictly increasing, so the order is the same); sigmoid
    routing ranks ``sigmoid(l) + bias`` (``moe_topk_sigmoid_batched`` is passed
    the correction bias beside the logits; reading: the bias only selects)."""
    if routing == ROUTE_SOFTMAX:
        return np.asarray(logits, dtype=np.float64)
    if routing == ROUTE_SIGMOID_BIAS:
        b = np.zeros(logits.shape[-1]) if bias is None else np.asarray(bias, np.float64)
        return sigmoid(logits) + b
    raise ValueError(routing)


def topk_select(scores: np.ndarray, k: int) -> np.ndarray:
    """Indices [N, k] of the k largest scores per row, in descending score;
    equal scores go to the lower expert index."""
    s = np.asarray(scores, dtype=np.float64)
    n, e = s.shape
    out = np.empty((n, k), dtype=np.int64)
    for t in range(n):
        order = np.lexsort((np.arange(e), -s[t]))   # primary: -score, then index
        out[t] = order[:k]
    return out


def topk_gap(scores: np.ndarray, k: int) -> np.ndarray:
    """Per row, the k-th largest score minus the (k+1)-th (inf when k == E):
    the margin by which the selected set is decided."""
    s = np.sort(np.asarray(scores, dtype=np.float64), axis=1)[:, ::-1]
    if k >= s.shape[1]:
        return np.full(s.shape[0], np.inf)
    return s[:, k - 1] - s[:, k]


def routing_probs(logits: np.ndarray, routing: str) -> np.ndarray:
    """Per-expert routing probabilities before selection: the full softmax over
    all E logits, or the element-wise sigmoid."""
    l = np.asarray(logits, dtype=np.float64)
    if routing == ROUTE_SOFTMAX:
        z = np.exp(l - l.max(axis=1, keepdims=True))
        return z / z.sum(axis=1, keepdims=True)
    if routing == ROUTE_SIGMOID_BIAS:
        return sigmoid(l)
    raise ValueError(routing)


def route(logits: np.ndarray, routing: str, top_k: int, norm_topk_prob: bool,
          routed_scaling_factor: float, bias: Optional[np.ndarray] = None):
    """Top-k routing: (indices [N, k] int64, weights [N, k] float64).

    Reading: ``routed_scaling_factor`` multiplies the weights for both routing
    kinds (the sigmoid top-k and the hash route are passed it; the softmax
    configurations here all use 1.0, so the reading does not move a result).
    No epsilon guards the renormalisation: every probability is positive."""
    idx = topk_select(selection_scores(logits, routing, bias), top_k)
    p = routing_probs(logits, routing)
    w = np.take_along_axis(p, idx, axis=1)
    if norm_topk_prob:
        w = w / w.sum(axis=1, keepdims=True)
    return idx, w * float(routed_scaling_factor)


# --------------------------------------------------------------------------
# Experts and blend
# --------------------------------------------------------------------------

def silu(v):
    v = np.asarray(v, dtype=np.float64)
    return v / (1.0 + np.exp(-v))


def swiglu_mlp(x: np.ndarray, wg: np.ndarray, wu: np.ndarray, wd: np.ndarray) -> np.ndarray:
    """``Wd (SiLU(Wg x) * (Wu x))`` for one token x [H], or row by row for x [R, H]."""
    x = np.asarray(x, dtype=np.float64)
    if x.ndim == 2:
        return np.stack([swiglu_mlp(x[r], wg, wu, wd) for r in range(x.shape[0])]) \
            if x.shape[0] else np.zeros((0, wd.shape[0]))
    g = wg @ x
    u = wu @ x
    return wd @ (silu(g) * u)


def moe_forward(layer: OracleLayer, x_bits: np.ndarray, rows=None, experts=None,
                include_shared: bool = True):
    """The whole layer for the tokens ``rows`` (default: all) of the BF16 input
    ``x_bits`` (uint16 [N, H]).  Returns (out float64 [R, H], indices int64
    [R, k], weights float64 [R, k], logits float64 [R, E]) for those rows.

    Each row is computed on its own, so the result for a row cannot depend on
    which other rows share the call.  Experts are decoded one at a time and
    every routed (token, slot) pair of that expert is evaluated with it.

    Expert parallelism (the EP branch of MoeLayer::forward and
    forward_token_major_decode): ``experts`` = (begin, end) keeps only the
    routes to experts in [begin, end) -- one rank's partial output, routing
    still computed over all experts -- and ``include_shared=False`` leaves the
    shared expert out (it is added once, after the partials are summed).

    With a pre-expert RMSNorm weight, the experts (routed and shared) take
    ``rms_norm(x)``; the router and the shared-expert gate take ``x``."""
    x_all = bf16_decode(x_bits)
    rows = np.arange(x_all.shape[0]) if rows is None else np.asarray(rows)
    x = x_all[rows]
    logits = router_logits(x, router_weights(layer))
    idx, w = route(logits, layer.routing, layer.top_k, layer.norm_topk_prob,
                   layer.routed_scaling_factor, layer.correction_bias)
    xe = x if layer.pre_expert_norm_w is None else rms_norm(x, layer.pre_expert_norm_w,
                                                            layer.rms_norm_eps)
    n, h = x.shape
    out = np.zeros((n, h), dtype=np.float64)
    # Routed experts: one expert decoded at a time.
    for e in np.unique(idx):
        if experts is not None and not (experts[0] <= e < experts[1]):
            continue
        wg, wu, wd = layer.gate.expert(e), layer.up.expert(e), layer.down.expert(e)
        tok, slot = np.nonzero(idx == e)
        d = swiglu_mlp(xe[tok], wg, wu, wd)
        out[tok] += w[tok, slot][:, None] * d
    # Always-on shared expert.
    if include_shared and layer.shared_inter > 0 and layer.sh_gate is not None:
        ds = swiglu_mlp(xe, layer.sh_gate.expert(0), layer.sh_up.expert(0),
                        layer.sh_down.expert(0))
        if layer.shared_gate_w is not None:
            gw = bf16_decode(layer.shared_gate_w)
            gs = sigmoid(np.array([float(x[t] @ gw) for t in range(n)]))
        else:
            gs = np.ones(n)
        out += gs[:, None] * ds
    return out, idx, w, logits


def moe_forward_slotwise(layer: OracleLayer, x_bits: np.ndarray):
    """The same layer evaluated slot by slot in the pages' order (route, then
    for each (token, slot) its own expert MLP, then the blend), without grouping
    tokens by expert.  Small inputs only; used to pin ``moe_forward``'s
    expert-major evaluation order."""
    x = bf16_decode(x_bits)
    logits = router_logits(x, router_weights(layer))
    idx, w = route(logits, layer.routing, layer.top_k, layer.norm_topk_prob,
                   layer.routed_scaling_factor, layer.correction_bias)
    xe = x if layer.pre_expert_norm_w is None else rms_norm(x, layer.pre_expert_norm_w,
                                                            layer.rms_norm_eps)
    n, h = x.shape
    out = np.zeros((n, h))
    for t in range(n):
        acc = np.zeros(h)
        for j in range(layer.top_k):
            e = idx[t, j]
            d = swiglu_mlp(xe[t], layer.gate.expert(e), layer.up.expert(e),
                           layer.down.expert(e))
            acc = acc + w[t, j] * d
        if layer.shared_inter > 0 and layer.sh_gate is not None:
            ds = swiglu_mlp(xe[t], layer.sh_gate.expert(0), layer.sh_up.expert(0),
                            layer.sh_down.expert(0))
            gs = 1.0 if layer.shared_gate_w is None else float(
                sigmoid(x[t] @ bf16_decode(layer.shared_gate_w)))
            acc = acc + gs * ds
        out[t] = acc
    return out, idx, w
