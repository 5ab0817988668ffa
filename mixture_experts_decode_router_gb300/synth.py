"""Seeded synthetic inputs for the MoE decode layer.

This module only draws random tensors and stores them in the library's
layouts; it holds none of the layer's arithmetic, and it serves the CUDA path,
the oracle and the benchmark alike.  Every tensor has its own seeded stream
(``torch.Generator`` seeded from ``(seed, tensor id, sub-index)``), so a
tensor, or one expert's matrix, is the same whatever else was drawn.

Recipe (one layer):
  * router weight  ~ N(0, std) -> BF16 (round to nearest even)        [E, H]
  * expert / shared-expert matrices ~ N(0, std), then stored as
      - BF16: rounded to nearest even                                 [E, out, in]
      - block-scaled FP8 E4M3: per 128x128 tile s = amax / 448 (1 when the
        tile is all zero), q = E4M3(w / s) with round-to-nearest-even
        and saturation at +-448; scales fp32 [E, ceil(out/128), ceil(in/128)]
      - NVFP4: per matrix scale2 = amax / (448 * 6) (1 when zero); per 16
        elements along ``in`` s16 = E4M3(amax16 / (6 * scale2)); codes
        q = E2M1(w / (s16 * scale2)) rounded to the nearest magnitude of
        {0, .5, 1, 1.5, 2, 3, 4, 6} (saturating), 0 where s16 is 0; two codes
        per byte, the even element in the low nibble
  * correction bias ~ U(-r, r) fp32 [E] (sigmoid routing only)
  * input rows ~ N(0, 1) -> BF16.  An optional ``gap_fn`` (supplied by the
    caller) returns, per row, the margin between the k-th and (k+1)-th
    selection score; rows whose margin is <= ``min_gap`` are redrawn from the
    next stream until every row is decided by more than ``min_gap``.
  * ``dup_frac``: that share of the N rows are copies of the distinct rows:
    ``N - round(N * dup_frac)`` distinct rows are drawn (with the gap rule),
    a seeded set of positions receives copies of uniformly drawn distinct rows,
    and the other positions hold the distinct rows in order.

The quantisers are a storage convention of this generator: the layer decodes
whatever codes it is given, so parity does not depend on them.
"""

from __future__ import annotations

from dataclasses import dataclass, replace
from typing import Callable, Dict, Optional

import numpy as np
import torch

ROUTE_SOFTMAX = "softmax"
ROUTE_SIGMOID_BIAS = "sigmoid_bias"
FMT_BF16 = "bf16"
FMT_FP8_B128 = "fp8_b128"
FMT_NVFP4 = "nvfp4"

_TID = {"router": 1, "gate": 2, "up": 3, "down": 4, "sh_gate": 5, "sh_up": 6,
        "sh_down": 7, "bias": 8, "shared_gate_w": 9, "x": 10, "dup": 11, "norm": 12}


@dataclass(frozen=True)
class LayerConfig:
    """One synthetic MoE layer and the token count of its workload."""
    name: str
    hidden: int
    num_experts: int
    top_k: int
    inter: int
    shared_inter: int
    routing: str
    norm_topk_prob: bool
    routed_scaling_factor: float
    expert_fmt: str
    n_tokens: int
    dup_frac: float = 0.0
    bias_range: float = 0.1
    weight_std: float = 0.02
    shared_gate: bool = False
    pre_expert_norm: bool = False      # an RMSNorm weight on the experts' input
    router_fmt: str = FMT_BF16         # BF16 router, or NVFP4 (quantised from the same matrix)
    rms_norm_eps: float = 1e-6
    seed: int = 0

    def with_(self, **kw) -> "LayerConfig":
        return replace(self, **kw)


# The five workloads the library is checked and measured on.
WORKLOADS: Dict[str, LayerConfig] = {
    # Tiny single-token decode.
    "tiny_n1": LayerConfig("tiny_n1", 256, 16, 2, 128, 128, ROUTE_SOFTMAX, True, 1.0,
                           FMT_BF16, 1),
    # Single-token decode, 256 experts (1 MB BF16 router), top-8.
    "decode_n1": LayerConfig("decode_n1", 2048, 256, 8, 512, 512, ROUTE_SOFTMAX, True, 1.0,
                             FMT_BF16, 1),
    # Batched decode, 16 tokens, sigmoid routing with a correction bias.
    "decode_n16": LayerConfig("decode_n16", 2048, 256, 8, 512, 512, ROUTE_SIGMOID_BIAS,
                              True, 2.5, FMT_BF16, 16),
    # 64 tokens, hidden 7168, FP8 E4M3 experts with 128x128 fp32 block scales.
    "fp8_n64": LayerConfig("fp8_n64", 7168, 256, 8, 2048, 2048, ROUTE_SIGMOID_BIAS, True,
                           2.5, FMT_FP8_B128, 64),
    # 256-row speculative verify, NVFP4 experts, 25% duplicated rows.
    "nvfp4_n256": LayerConfig("nvfp4_n256", 2048, 256, 8, 512, 512, ROUTE_SOFTMAX, True,
                              1.0, FMT_NVFP4, 256, dup_frac=0.25),
}


def _gen(device, seed: int, tensor: str, sub: int = 0) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed((seed * 1_000_003 + _TID[tensor] * 10_007 + sub * 7_919 + 17) % (2**63 - 1))
    return g


# ---------------------------------------------------------------- quantisers

def _quant_fp8_b128(w: torch.Tensor):
    """[out, in] fp32 -> (uint8 codes [out, in], fp32 scales [ceil(out/128), ceil(in/128)])."""
    out_d, in_d = w.shape
    ob, ib = -(-out_d // 128), -(-in_d // 128)
    pad = torch.zeros(ob * 128, ib * 128, dtype=torch.float32, device=w.device)
    pad[:out_d, :in_d] = w
    blk = pad.view(ob, 128, ib, 128).abs().amax(dim=(1, 3))
    s = torch.where(blk > 0, blk / 448.0, torch.ones_like(blk))
    sx = s.repeat_interleave(128, 0).repeat_interleave(128, 1)[:out_d, :in_d]
    q = (w / sx).clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)
    return q.contiguous(), s.contiguous()


_E2M1_MAG = torch.tensor([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
_E2M1_MID = torch.tensor([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])


def _e2m1_codes(v: torch.Tensor) -> torch.Tensor:
    mid = _E2M1_MID.to(v.device)
    mag = v.abs().clamp(max=6.0)
    code = torch.bucketize(mag, mid)            # 0..7, nearest magnitude
    sign = (v < 0) & (code > 0)
    return (code + 8 * sign.to(code.dtype)).to(torch.uint8)


def _quant_nvfp4(w: torch.Tensor):
    """[out, in] fp32 -> (packed uint8 [out, in/2], E4M3 uint8 [out, in/16], scale2 float)."""
    out_d, in_d = w.shape
    amax = w.abs().amax()
    scale2 = (amax / (448.0 * 6.0)) if float(amax) > 0 else torch.tensor(1.0, device=w.device)
    scale2 = scale2.to(torch.float32)
    blk = w.view(out_d, in_d // 16, 16).abs().amax(dim=2)
    s16 = (blk / (6.0 * scale2)).clamp(max=448.0).to(torch.float8_e4m3fn)
    s16v = s16.to(torch.float32)
    denom = (s16v * scale2).repeat_interleave(16, dim=1)
    safe = torch.where(denom > 0, denom, torch.ones_like(denom))
    codes = torch.where(denom > 0, _e2m1_codes(w / safe), torch.zeros_like(w, dtype=torch.uint8))
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).to(torch.uint8)
    return packed.contiguous(), s16.view(torch.uint8).contiguous(), float(scale2)


@dataclass
class QMatT:
    """Stacked expert matrix on a device, in the library's layout."""
    fmt: str
    w: torch.Tensor
    scale: Optional[torch.Tensor] = None
    scale2: Optional[torch.Tensor] = None


def matrix_dims(cfg: LayerConfig, tensor: str):
    """(out, in) of one expert matrix of `tensor`."""
    H, I, S = cfg.hidden, cfg.inter, cfg.shared_inter
    return {"gate": (I, H), "up": (I, H), "down": (H, I), "sh_gate": (S, H), "sh_up": (S, H),
            "sh_down": (H, S)}[tensor]


def expert_matrix(cfg: LayerConfig, tensor: str, e: int, device="cpu"):
    """The stored form of expert e's `tensor` matrix alone: (w, scale, scale2)
    -- identical to slice e of the stacked tensor make_weights builds."""
    out_d, in_d = matrix_dims(cfg, tensor)
    m = torch.randn(out_d, in_d, generator=_gen(device, cfg.seed, tensor, e), device=device,
                    dtype=torch.float32) * cfg.weight_std
    if cfg.expert_fmt == FMT_BF16:
        return m.to(torch.bfloat16), None, None
    if cfg.expert_fmt == FMT_FP8_B128:
        q, s = _quant_fp8_b128(m)
        return q, s, None
    q, s, s2 = _quant_nvfp4(m)
    return q, s, s2


def _stacked(cfg: LayerConfig, tensor: str, n_exp: int, out_d: int, in_d: int,
             device) -> QMatT:
    fmt = cfg.expert_fmt
    if fmt == FMT_BF16:
        w = torch.empty(n_exp, out_d, in_d, dtype=torch.bfloat16, device=device)
    elif fmt == FMT_FP8_B128:
        w = torch.empty(n_exp, out_d, in_d, dtype=torch.uint8, device=device)
        sc = torch.empty(n_exp, -(-out_d // 128), -(-in_d // 128), dtype=torch.float32,
                         device=device)
    elif fmt == FMT_NVFP4:
        w = torch.empty(n_exp, out_d, in_d // 2, dtype=torch.uint8, device=device)
        sc = torch.empty(n_exp, out_d, in_d // 16, dtype=torch.uint8, device=device)
        s2 = torch.empty(n_exp, dtype=torch.float32, device=device)
    else:
        raise ValueError(fmt)
    for e in range(n_exp):
        q, s, s2v = expert_matrix(cfg, tensor, e, device)
        w[e] = q
        if fmt != FMT_BF16:
            sc[e] = s
        if fmt == FMT_NVFP4:
            s2[e] = s2v
    if fmt == FMT_BF16:
        return QMatT(fmt, w)
    if fmt == FMT_FP8_B128:
        return QMatT(fmt, w, sc)
    return QMatT(fmt, w, sc, s2)


@dataclass
class LayerWeights:
    cfg: LayerConfig
    router_w: torch.Tensor                   # bf16 [E, H]
    gate: QMatT
    up: QMatT
    down: QMatT
    sh_gate: Optional[QMatT]
    sh_up: Optional[QMatT]
    sh_down: Optional[QMatT]
    correction_bias: Optional[torch.Tensor]  # fp32 [E]
    shared_gate_w: Optional[torch.Tensor]    # bf16 [H]
    pre_expert_norm_w: Optional[torch.Tensor] = None   # bf16 [H]
    router_q: Optional[QMatT] = None                   # NVFP4 router [1, E, H]


def _router_fp32(cfg: LayerConfig, device) -> torch.Tensor:
    return torch.randn(cfg.num_experts, cfg.hidden, generator=_gen(device, cfg.seed, "router"),
                       device=device) * cfg.weight_std


def make_router(cfg: LayerConfig, device="cpu") -> torch.Tensor:
    return _router_fp32(cfg, device).to(torch.bfloat16)


def make_router_q(cfg: LayerConfig, device="cpu") -> Optional[QMatT]:
    """The NVFP4 router (one matrix [E, H], stacked as [1, E, H]) quantised from
    the BF16 router's fp32 draw, or None for a BF16 router."""
    if cfg.router_fmt == FMT_BF16:
        return None
    if cfg.router_fmt != FMT_NVFP4:
        raise ValueError(cfg.router_fmt)
    q, sc, s2 = _quant_nvfp4(_router_fp32(cfg, device))
    return QMatT(FMT_NVFP4, q[None].contiguous(), sc[None].contiguous(),
                 torch.tensor([s2], dtype=torch.float32, device=device))


def make_bias(cfg: LayerConfig, device="cpu") -> Optional[torch.Tensor]:
    if cfg.routing != ROUTE_SIGMOID_BIAS:
        return None
    u = torch.rand(cfg.num_experts, generator=_gen(device, cfg.seed, "bias"), device=device)
    return ((u * 2.0 - 1.0) * cfg.bias_range).to(torch.float32)


def make_shared_gate_w(cfg: LayerConfig, device="cpu") -> Optional[torch.Tensor]:
    if not cfg.shared_gate:
        return None
    return (torch.randn(cfg.hidden, generator=_gen(device, cfg.seed, "shared_gate_w"),
                        device=device) * cfg.weight_std).to(torch.bfloat16)


def make_weights(cfg: LayerConfig, device="cpu") -> LayerWeights:
    E, H, I, S = cfg.num_experts, cfg.hidden, cfg.inter, cfg.shared_inter
    router = make_router(cfg, device)
    gate = _stacked(cfg, "gate", E, I, H, device)
    up = _stacked(cfg, "up", E, I, H, device)
    down = _stacked(cfg, "down", E, H, I, device)
    if S > 0:
        sh_gate = _stacked(cfg, "sh_gate", 1, S, H, device)
        sh_up = _stacked(cfg, "sh_up", 1, S, H, device)
        sh_down = _stacked(cfg, "sh_down", 1, H, S, device)
    else:
        sh_gate = sh_up = sh_down = None
    return LayerWeights(cfg, router, gate, up, down, sh_gate, sh_up, sh_down,
                        make_bias(cfg, device), make_shared_gate_w(cfg, device),
                        make_norm_w(cfg, device), make_router_q(cfg, device))


def make_norm_w(cfg: LayerConfig, device="cpu") -> Optional[torch.Tensor]:
    """RMSNorm weight, BF16 [H]: 1 + 0.1 * N(0, 1), the spread of a trained
    norm's gains around one."""
    if not cfg.pre_expert_norm:
        return None
    z = torch.randn(cfg.hidden, generator=_gen(device, cfg.seed, "norm"), device=device)
    return (1.0 + 0.1 * z).to(torch.bfloat16)


def expert_slice(lw: LayerWeights, begin: int, end: int) -> LayerWeights:
    """The routed experts [begin, end) of a layer, as one expert-parallel rank
    holds them (views of the full stacks; the shared expert and router kept)."""
    def part(q: QMatT) -> QMatT:
        return QMatT(q.fmt, q.w[begin:end],
                     q.scale[begin:end] if q.scale is not None else None,
                     q.scale2[begin:end] if q.scale2 is not None else None)
    return replace(lw, gate=part(lw.gate), up=part(lw.up), down=part(lw.down))


GapFn = Callable[[np.ndarray], np.ndarray]


def _draw_rows(cfg: LayerConfig, n: int, device, gap_fn: Optional[GapFn], min_gap: float,
               stream_base: int, max_attempts: int = 200) -> torch.Tensor:
    H = cfg.hidden
    x = torch.empty(n, H, dtype=torch.bfloat16, device=device)
    pending = torch.arange(n, device=device)
    for attempt in range(max_attempts):
        g = _gen(device, cfg.seed, "x", stream_base + attempt)
        cand = torch.randn(n, H, generator=g, device=device).to(torch.bfloat16)
        x[pending] = cand[pending]
        if gap_fn is None:
            return x
        bits = x[pending].view(torch.int16).cpu().numpy().view(np.uint16)
        gaps = np.asarray(gap_fn(bits))
        keep = torch.from_numpy(gaps <= min_gap).to(device)
        pending = pending[keep]
        if pending.numel() == 0:
            return x
    raise RuntimeError("could not draw rows without near-ties")


def make_input(cfg: LayerConfig, n: Optional[int] = None, device="cpu",
               gap_fn: Optional[GapFn] = None, min_gap: float = 1e-3,
               dup_frac: Optional[float] = None, stream: int = 0) -> torch.Tensor:
    """BF16 input rows [n, H] (see the module recipe)."""
    n = cfg.n_tokens if n is None else n
    dup = cfg.dup_frac if dup_frac is None else dup_frac
    base = stream * 100_000
    if n == 0:
        return torch.empty(0, cfg.hidden, dtype=torch.bfloat16, device=device)
    n_dup = int(round(n * dup))
    n_dist = n - n_dup
    distinct = _draw_rows(cfg, n_dist, device, gap_fn, min_gap, base)
    if n_dup == 0:
        return distinct
    g = _gen("cpu", cfg.seed, "dup", stream)
    pos = torch.randperm(n, generator=g)
    dup_pos = torch.sort(pos[:n_dup]).values
    src = torch.randint(0, n_dist, (n_dup,), generator=g)
    is_dup = torch.zeros(n, dtype=torch.bool)
    is_dup[dup_pos] = True
    x = torch.empty(n, cfg.hidden, dtype=torch.bfloat16, device=device)
    x[(~is_dup).nonzero().flatten().to(device)] = distinct
    x[dup_pos.to(device)] = distinct[src.to(device)]
    return x


def matrix_bytes(fmt: str, out_d: int, in_d: int) -> int:
    """Bytes of one [out, in] matrix, scales included."""
    if fmt == FMT_BF16:
        return out_d * in_d * 2
    if fmt == FMT_FP8_B128:
        return out_d * in_d + 4 * (-(-out_d // 128)) * (-(-in_d // 128))
    if fmt == FMT_NVFP4:
        return out_d * in_d // 2 + out_d * in_d // 16 + 4
    raise ValueError(fmt)


def layer_bytes(cfg: LayerConfig) -> dict:
    """Byte counts of the parts of one layer, for the touched-bytes metric."""
    H, I, S, E = cfg.hidden, cfg.inter, cfg.shared_inter, cfg.num_experts
    per_expert = 2 * matrix_bytes(cfg.expert_fmt, I, H) + matrix_bytes(cfg.expert_fmt, H, I)
    shared = (2 * matrix_bytes(cfg.expert_fmt, S, H) + matrix_bytes(cfg.expert_fmt, H, S)
              if S > 0 else 0)
    extra = ((4 * E if cfg.routing == ROUTE_SIGMOID_BIAS else 0) + (2 * H if cfg.shared_gate else 0)
             + (2 * H if cfg.pre_expert_norm else 0))
    router = E * H * 2 if cfg.router_fmt == FMT_BF16 else matrix_bytes(cfg.router_fmt, E, H)
    return {"router": router, "per_expert": per_expert, "shared": shared, "extra": extra,
            "hidden": H}


def touched_bytes(cfg: LayerConfig, indices: np.ndarray) -> int:
    """Algorithmic bytes of one call: router + each distinct routed expert's
    three matrices + shared expert + bias/gate vectors + BF16 input and output."""
    d = layer_bytes(cfg)
    idx = np.asarray(indices)
    n = idx.shape[0]
    distinct = len(np.unique(idx)) if idx.size else 0
    return int(d["router"] + distinct * d["per_expert"] + d["shared"] + d["extra"]
               + 2 * n * d["hidden"] * 2)
