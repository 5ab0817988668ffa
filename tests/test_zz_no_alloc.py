"""The static-workspace entry point, moe_forward_static_ws, and its check call.

moe_forward_static_ws exists for callers that cannot allocate device memory (a
plugin whose host owns every allocation, or code recording a CUDA graph, where
cudaMalloc is not allowed): it takes no workspace and uses one device array
inside the library.  These tests call it through the C ABI twice in a row, on
two different inputs, and check each result bit for bit against moe_forward
with a caller workspace (the same kernels on the same inputs), and once
against the oracle.  moe_static_workspace_check reads and clears the array's
device error word: a dirty control block (planted from the host) makes a
one-token call refuse, the check reports it, and the next call is clean.
They must pass alone in a fresh process and after every other test, so they
live in a file pytest collects last.
"""

import numpy as np
import pytest
import torch

from mixture_experts_decode_router_gb300 import binding as B
from mixture_experts_decode_router_gb300 import synth
from mixture_experts_decode_router_gb300.layer import MoeLayer, make_config
from oracle import moe_oracle as O
from tests.moe_helpers import bf16_bits, gap_fn_for, oracle_layer, tolerance

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    B.load()


def _static_call(layer, x, out=None):
    n, k = x.shape[0], layer.cfg.top_k
    if out is None:
        out = torch.empty(n, layer.cfg.hidden, dtype=torch.bfloat16, device=x.device)
    idx = torch.empty(n, k, dtype=torch.int32, device=x.device)
    w = torch.empty(n, k, dtype=torch.float32, device=x.device)
    s = B.moe_forward_static_ws(layer.c_cfg, layer.c_w, x, n, out, idx, w)
    return s, out, idx, w


def _static_error():
    s, err, _ = B.moe_static_workspace_check()
    assert s == B.MOE_OK, B.moe_status_string(s)
    return err


@pytest.mark.parametrize("name,n", [("decode_n1", 1), ("decode_n16", 16)])
def test_static_workspace_matches_moe_forward(name, n):
    cfg = synth.WORKLOADS[name]
    lw = synth.make_weights(cfg, "cuda")
    layer = MoeLayer(lw, n)
    xs = [synth.make_input(cfg, n, "cuda", stream=s) for s in (1, 2)]
    for x in xs:                                   # two calls in a row
        s, out, idx, w = _static_call(layer, x)
        assert s == B.MOE_OK, B.moe_status_string(s)
        ref_out, ref_idx, ref_w = layer.forward(x)
        torch.cuda.synchronize()
        assert torch.equal(idx, ref_idx)
        assert torch.equal(w, ref_w)
        assert torch.equal(out, ref_out)
    assert _static_error() == 0
    assert layer.device_error() == 0


def test_static_workspace_matches_the_oracle():
    cfg = synth.WORKLOADS["decode_n16"]
    lw = synth.make_weights(cfg, "cuda")
    L = oracle_layer(lw)
    x = synth.make_input(cfg, 6, "cuda", gap_fn=gap_fn_for(L))
    layer = MoeLayer(lw, 6)
    s, out, idx, w = _static_call(layer, x)
    assert s == B.MOE_OK, B.moe_status_string(s)
    torch.cuda.synchronize()
    ref, ref_idx, ref_w, _ = O.moe_forward(L, bf16_bits(x))
    assert np.array_equal(idx.cpu().numpy(), ref_idx)
    assert np.max(np.abs(w.cpu().numpy() - ref_w)) <= 1e-5 * max(1.0, cfg.routed_scaling_factor)
    rms = float(np.sqrt(np.mean(ref ** 2)))
    assert float(np.max(np.abs(out.float().cpu().numpy() - ref))) <= tolerance(cfg.expert_fmt) * rms
    assert _static_error() == 0


class _DeviceBytes:
    """A device address and a length, as a CUDA array (so torch can view it)."""

    def __init__(self, addr, nbytes):
        self.__cuda_array_interface__ = {"shape": (nbytes,), "typestr": "|u1",
                                         "data": (addr, False), "version": 2}


def test_static_check_reports_and_clears_a_dirty_control_block():
    cfg = synth.WORKLOADS["tiny_n1"]
    lw = synth.make_weights(cfg, "cuda")
    x = synth.make_input(cfg, 1, "cuda")
    layer = MoeLayer(lw, 1)
    s, good, _, _ = _static_call(layer, x)
    assert s == B.MOE_OK
    s, err, addr = B.moe_static_workspace_check()
    assert s == B.MOE_OK and err == 0 and addr
    ctrl = torch.as_tensor(_DeviceBytes(addr, 256), device="cuda")
    # Plant, from the host, what a call that ended early leaves behind: a
    # single-token grid-barrier word that is not zero.
    ctrl[12:16] = 255
    torch.cuda.synchronize()
    sentinel = torch.full_like(good, 7)
    s, out, _, _ = _static_call(layer, x, out=sentinel.clone())
    assert s == B.MOE_OK                     # the refusal happens on the device
    torch.cuda.synchronize()
    assert torch.equal(out, sentinel)        # refused: nothing written
    assert _static_error() == 20             # reported once, and cleared
    assert int(ctrl[8:16].count_nonzero()) == 0
    s, again, _, _ = _static_call(layer, x)
    assert s == B.MOE_OK
    torch.cuda.synchronize()
    assert torch.equal(again, good)
    assert _static_error() == 0


def test_static_workspace_rejects_sizes_beyond_its_capacity():
    cfg = synth.WORKLOADS["fp8_n64"].with_(num_experts=8)
    cc = make_config(cfg)
    n = 4096
    assert B.moe_workspace_bytes(cc, n) > B.MOE_STATIC_WORKSPACE_BYTES
    # Real device buffers, so no check order could make the call touch a bad address.
    x = torch.zeros(n, cfg.hidden, dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(x)
    lw = synth.make_weights(cfg.with_(n_tokens=1), "cuda")
    layer = MoeLayer(lw, 1)
    s = B.moe_forward_static_ws(cc, layer.c_w, x, n, out, None, None)
    assert s == B.MOE_ERR_WORKSPACE
