"""The static-workspace entry point, moe_forward_static_ws.

It exists for callers that cannot allocate device memory (a plugin whose host
owns every allocation, or code recording a CUDA graph, where cudaMalloc is not
allowed): it takes no workspace and uses one device array inside the library.
This test calls it through the C ABI twice in a row, on two different inputs,
and checks each result against moe_forward with a caller workspace, within the
tolerances of the parity tests.  It must pass alone in a fresh process and
after every other test, so it lives in a file pytest collects last.
"""

import numpy as np
import pytest
import torch

from mixture_experts_decode_router_gb300 import binding as B
from mixture_experts_decode_router_gb300 import synth
from mixture_experts_decode_router_gb300.layer import MoeLayer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    B.load()


def _static_call(layer, x):
    n, k = x.shape[0], layer.cfg.top_k
    out = torch.empty(n, layer.cfg.hidden, dtype=torch.bfloat16, device=x.device)
    idx = torch.empty(n, k, dtype=torch.int32, device=x.device)
    w = torch.empty(n, k, dtype=torch.float32, device=x.device)
    s = B.moe_forward_static_ws(layer.c_cfg, layer.c_w, x, n, out, idx, w)
    return s, out, idx, w


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
        assert float((w - ref_w).abs().max()) <= 1e-5 * max(1.0, cfg.routed_scaling_factor)
        ref = ref_out.float().cpu().numpy()
        rms = float(np.sqrt(np.mean(ref ** 2)))
        err = float(np.max(np.abs(out.float().cpu().numpy() - ref)))
        assert err <= 2e-2 * rms


def test_static_workspace_rejects_sizes_beyond_its_capacity():
    cfg = synth.WORKLOADS["fp8_n64"].with_(num_experts=8)
    c = MoeLayer.__new__(MoeLayer)
    from mixture_experts_decode_router_gb300.layer import make_config
    cc = make_config(cfg)
    n = 4096
    assert B.moe_workspace_bytes(cc, n) > B.MOE_STATIC_WORKSPACE_BYTES
    w = B.moe_weights_t()
    s = B.moe_forward_static_ws(cc, w, 16, n, 32, None, None)
    assert s == B.MOE_ERR_WORKSPACE
    del c
