"""Host-only checks of the C ABI (no GPU): the library loads, exports every
function include/moe.h declares, its structs have the header's layout, and
every validation error is returned by name before anything is launched."""

import ctypes
import os
import re
import subprocess

import pytest

from mixture_experts_decode_router_gb300 import binding as B
from mixture_experts_decode_router_gb300 import synth
from mixture_experts_decode_router_gb300.layer import make_config

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe.h")


@pytest.fixture(scope="module")
def lib():
    return B.load()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*[a-z_][\w\s\*]*?\b(moe_\w+)\s*\(", text, flags=re.M)))


def test_library_exports_every_declared_function(lib):
    names = _declared_functions()
    assert set(names) == set(B.EXPORTED), names
    for n in names:
        assert hasattr(lib, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", B.lib_path()], capture_output=True,
                         text=True).stdout
    for n in names:
        assert re.search(rf"\bT {n}$", out, flags=re.M), n
    assert lib.moe_abi_version() == 2


def test_struct_layout_matches_header(tmp_path):
    src = tmp_path / "layout.c"
    src.write_text(
        '#include <stdio.h>\n#include <stddef.h>\n#include "moe.h"\n'
        'int main(void){printf("%zu %zu %zu %zu %zu %zu %zu %zu\\n", sizeof(moe_config_t),'
        ' sizeof(moe_qmat_t), sizeof(moe_weights_t), offsetof(moe_config_t, routed_scaling_factor),'
        ' offsetof(moe_weights_t, sh_down), offsetof(moe_weights_t, shared_gate_w),'
        ' offsetof(moe_config_t, exclude_shared), offsetof(moe_weights_t, pre_expert_norm_w));return 0;}\n')
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c99", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)],
                   check=True)
    got = [int(v) for v in subprocess.run([str(exe)], capture_output=True, text=True).stdout.split()]
    assert got == [ctypes.sizeof(B.moe_config_t), ctypes.sizeof(B.moe_qmat_t),
                   ctypes.sizeof(B.moe_weights_t), B.moe_config_t.routed_scaling_factor.offset,
                   B.moe_weights_t.sh_down.offset, B.moe_weights_t.shared_gate_w.offset,
                   B.moe_config_t.exclude_shared.offset, B.moe_weights_t.pre_expert_norm_w.offset]


def _cfg(**kw):
    c = make_config(synth.WORKLOADS["decode_n16"])
    for k, v in kw.items():
        setattr(c, k, v)
    return c


FAKE = 0x7f0000000000      # a 16-aligned address that is never dereferenced here


def _weights(sigmoid=True, **kw):
    w = B.moe_weights_t()
    w.router_w = FAKE
    w.correction_bias = FAKE if sigmoid else None
    for m in ("gate", "up", "down", "sh_gate", "sh_up", "sh_down"):
        getattr(w, m).w = FAKE
    for k, v in kw.items():
        setattr(w, k, v)
    return w


@pytest.mark.parametrize("field,value", [
    ("num_experts", 0), ("num_experts", 1025), ("top_k", 0), ("top_k", 33), ("hidden", 100),
    ("hidden", 0), ("inter", 48), ("shared_inter", -32), ("shared_inter", 40), ("routing", 7),
    ("norm_topk_prob", 2), ("expert_fmt", 9), ("path", 5), ("routed_scaling_factor", float("nan")),
    ("expert_begin", -1), ("expert_end", 257), ("exclude_shared", 2), ("rms_norm_eps", -1.0),
    ("accumulate", 2), ("router_fmt", 1), ("router_fmt", 3),
    ("rms_norm_eps", float("nan")),
])
def test_invalid_config(lib, field, value):
    c = _cfg(**{field: value})
    assert B.moe_workspace_bytes(c, 16) == 0
    s = B.moe_forward(c, _weights(), FAKE, 16, FAKE + 0x100000, None, None, FAKE, 1 << 40, 0)
    assert s == B.MOE_ERR_INVALID_CONFIG


def test_top_k_above_num_experts(lib):
    assert B.moe_forward(_cfg(num_experts=4, top_k=5), _weights(), FAKE, 1, FAKE + 0x100000, None,
                         None, FAKE, 1 << 40, 0) == B.MOE_ERR_INVALID_CONFIG


def test_null_and_alignment_and_alias(lib):
    c = _cfg()
    big = 1 << 40
    out = FAKE + 0x100000
    assert B.moe_forward(None, _weights(), FAKE, 1, out, None, None, FAKE, big, 0) == B.MOE_ERR_NULL
    assert B.moe_forward(c, _weights(router_w=None), FAKE, 1, out, None, None, FAKE, big, 0) \
        == B.MOE_ERR_NULL
    assert B.moe_forward(c, _weights(correction_bias=None), FAKE, 1, out, None, None, FAKE, big, 0) \
        == B.MOE_ERR_NULL
    assert B.moe_forward(c, _weights(), None, 1, out, None, None, FAKE, big, 0) == B.MOE_ERR_NULL
    assert B.moe_forward(c, _weights(), FAKE + 8, 1, out, None, None, FAKE, big, 0) \
        == B.MOE_ERR_ALIGNMENT
    assert B.moe_forward(c, _weights(), FAKE, 4, FAKE + 64, None, None, FAKE, big, 0) \
        == B.MOE_ERR_ALIAS
    # A softmax layer given a correction bias is refused rather than ignored.
    cs = _cfg(routing=B.MOE_ROUTE_SOFTMAX)
    assert B.moe_forward(cs, _weights(sigmoid=True), FAKE, 1, out, None, None, FAKE, big, 0) \
        == B.MOE_ERR_INVALID_CONFIG
    # FP8 needs block scales; NVFP4 needs scales and scale2.
    c8 = _cfg(expert_fmt=B.MOE_W_FP8_B128)
    assert B.moe_forward(c8, _weights(), FAKE, 1, out, None, None, FAKE, big, 0) == B.MOE_ERR_NULL
    w4 = _weights()
    for m in ("gate", "up", "down", "sh_gate", "sh_up", "sh_down"):
        getattr(w4, m).scale = FAKE
    c4 = _cfg(expert_fmt=B.MOE_W_NVFP4)
    assert B.moe_forward(c4, w4, FAKE, 1, out, None, None, FAKE, big, 0) == B.MOE_ERR_NULL
    # No shared expert: its matrices may be NULL; then the workspace check comes next.
    w0 = _weights()
    for m in ("sh_gate", "sh_up", "sh_down"):
        getattr(w0, m).w = None
    assert B.moe_forward(_cfg(shared_inter=0), w0, FAKE, 1, out, None, None, FAKE, 16, 0) \
        == B.MOE_ERR_WORKSPACE


def test_expert_parallel_ranges(lib):
    """[expert_begin, expert_end): (0, 0) means all experts; begin > end or end > E
    is refused; a rank holding no expert passes no routed weights."""
    big, out = 1 << 40, FAKE + 0x100000
    assert B.moe_forward(_cfg(expert_begin=10, expert_end=5), _weights(), FAKE, 1, out, None, None,
                         FAKE, big, 0) == B.MOE_ERR_INVALID_CONFIG
    assert B.moe_forward(_cfg(expert_begin=0, expert_end=257), _weights(), FAKE, 1, out, None,
                         None, FAKE, big, 0) == B.MOE_ERR_INVALID_CONFIG
    # A full range and (0, 0) need the same workspace; leaving the shared expert
    # out needs no more.
    full = B.moe_workspace_bytes(_cfg(), 16)
    assert B.moe_workspace_bytes(_cfg(expert_begin=0, expert_end=256), 16) == full
    assert B.moe_workspace_bytes(_cfg(expert_begin=64, expert_end=128), 16) == full
    assert 0 < B.moe_workspace_bytes(_cfg(exclude_shared=1), 16) <= full
    # No local expert: routed matrices may be NULL (the workspace check comes next) ...
    wn = _weights()
    for m in ("gate", "up", "down"):
        getattr(wn, m).w = None
    assert B.moe_forward(_cfg(expert_begin=256, expert_end=256), wn, FAKE, 1, out, None, None,
                         FAKE, 16, 0) == B.MOE_ERR_WORKSPACE
    # ... but are required as soon as the call holds one.
    assert B.moe_forward(_cfg(expert_begin=255, expert_end=256), wn, FAKE, 1, out, None, None,
                         FAKE, 16, 0) == B.MOE_ERR_NULL
    # Without the shared expert its matrices may be NULL.
    ws_ = _weights()
    for m in ("sh_gate", "sh_up", "sh_down"):
        getattr(ws_, m).w = None
    assert B.moe_forward(_cfg(exclude_shared=1), ws_, FAKE, 1, out, None, None, FAKE, 16, 0) \
        == B.MOE_ERR_WORKSPACE


def test_nvfp4_router_weights(lib):
    """An NVFP4 router needs router_q (codes, scales, scale2) and not router_w."""
    big, out = 1 << 40, FAKE + 0x100000
    c = _cfg(router_fmt=B.MOE_W_NVFP4)
    w = _weights(router_w=None)
    assert B.moe_forward(c, w, FAKE, 1, out, None, None, FAKE, big, 0) == B.MOE_ERR_NULL
    w.router_q.w, w.router_q.scale = FAKE, FAKE
    assert B.moe_forward(c, w, FAKE, 1, out, None, None, FAKE, big, 0) == B.MOE_ERR_NULL
    w.router_q.scale2 = FAKE
    assert B.moe_forward(c, w, FAKE, 1, out, None, None, FAKE, 16, 0) == B.MOE_ERR_WORKSPACE
    w.router_q.w = FAKE + 8
    assert B.moe_forward(c, w, FAKE, 1, out, None, None, FAKE, big, 0) == B.MOE_ERR_ALIGNMENT
    # A BF16 router still needs router_w.
    assert B.moe_forward(_cfg(), _weights(router_w=None), FAKE, 1, out, None, None, FAKE, big, 0) \
        == B.MOE_ERR_NULL


def test_scale_and_norm_alignment(lib):
    """Scales need 4-byte alignment (a rank's slice of a stacked scale array);
    the norm weight needs 16."""
    big, out = 1 << 40, FAKE + 0x100000
    w8 = _weights()
    for m in ("gate", "up", "down", "sh_gate", "sh_up", "sh_down"):
        getattr(w8, m).scale = FAKE + 4
    c8 = _cfg(expert_fmt=B.MOE_W_FP8_B128)
    assert B.moe_forward(c8, w8, FAKE, 1, out, None, None, FAKE, 16, 0) == B.MOE_ERR_WORKSPACE
    w8.down.scale = FAKE + 2
    assert B.moe_forward(c8, w8, FAKE, 1, out, None, None, FAKE, big, 0) == B.MOE_ERR_ALIGNMENT
    assert B.moe_forward(_cfg(), _weights(pre_expert_norm_w=FAKE + 4), FAKE, 1, out, None, None,
                         FAKE, big, 0) == B.MOE_ERR_ALIGNMENT


def test_workspace_checks(lib):
    c = _cfg()
    need = B.moe_workspace_bytes(c, 16)
    assert need > 0 and need % 256 == 0
    assert B.moe_workspace_bytes(c, 32) > need
    assert B.moe_workspace_bytes(c, -1) == 0
    out = FAKE + 0x1000000
    assert B.moe_forward(c, _weights(), FAKE, 16, out, None, None, FAKE, need - 1, 0) \
        == B.MOE_ERR_WORKSPACE
    assert B.moe_forward(c, _weights(), FAKE, 16, out, None, None, None, need, 0) \
        == B.MOE_ERR_WORKSPACE
    assert B.moe_route(c, _weights(), FAKE, 16, FAKE, FAKE, None, FAKE, need - 1, 0) \
        == B.MOE_ERR_WORKSPACE
    assert B.moe_experts(c, _weights(), FAKE, 16, FAKE, FAKE, out, FAKE, need - 1, 0) \
        == B.MOE_ERR_WORKSPACE


def test_zero_tokens_and_negative(lib):
    c = _cfg()
    assert B.moe_forward(c, _weights(), None, 0, None, None, None, None, 0, 0) == B.MOE_OK
    assert B.moe_forward(c, _weights(), FAKE, -1, FAKE, None, None, FAKE, 1 << 40, 0) \
        == B.MOE_ERR_INVALID_CONFIG


def test_status_strings(lib):
    for s in range(9):
        assert B.moe_status_string(s).startswith("MOE_")
    assert "unknown" in B.moe_status_string(99)
