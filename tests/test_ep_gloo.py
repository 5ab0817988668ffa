"""Host-side logic of expert parallelism on 2, 3, 4 and 8 gloo ranks on the CPU
(4 and 8 ranks over 256 experts, the full expert count of the workloads): the
expert partition, the all-reduce of the BF16 partials, and the shared expert
added once.  The per-rank compute is the fp64 oracle's partial (the
CUDA partials are checked against the same oracle partials on the GPU)."""

import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from mixture_experts_decode_router_gb300.ep import expert_range


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


@pytest.mark.parametrize("world,E", [(1, 8), (2, 8), (3, 8), (8, 256), (5, 33), (4, 3)])
def test_expert_range_partitions_the_experts(world, E):
    spans = [expert_range(r, world, E) for r in range(world)]
    assert spans[0][0] == 0 and spans[-1][1] == E
    for (b0, e0), (b1, _) in zip(spans, spans[1:]):
        assert e0 == b1                                  # contiguous, no overlap
    sizes = [e - b for b, e in spans]
    assert max(sizes) - min(sizes) <= 1 and sum(sizes) == E


def test_expert_range_refuses_bad_ranks():
    with pytest.raises(ValueError):
        expert_range(2, 2, 8)
    with pytest.raises(ValueError):
        expert_range(-1, 2, 8)


def _bf16(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)


def _rank(rank, world, port, shared_gate, E, k, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", init_method="env://", rank=rank, world_size=world)
    from mixture_experts_decode_router_gb300 import synth
    from mixture_experts_decode_router_gb300.ep import ep_forward
    from oracle import moe_oracle as O
    from tests.moe_helpers import bf16_bits, gap_fn_for, oracle_layer

    cfg = synth.LayerConfig("ep", 64, E, k, 32, 32, synth.ROUTE_SIGMOID_BIAS, True, 2.5,
                            synth.FMT_BF16, 5, shared_gate=shared_gate)
    lw = synth.make_weights(cfg)
    L = oracle_layer(lw)
    x = synth.make_input(cfg, gap_fn=gap_fn_for(L))
    xb = bf16_bits(x)
    b, e = expert_range(rank, world, cfg.num_experts)

    def partial(_x):
        ref, _, _, _ = O.moe_forward(L, xb, experts=(b, e), include_shared=False)
        return _bf16(ref)

    def add_shared(_x, o):
        sh, _, _, _ = O.moe_forward(L, xb, experts=(cfg.num_experts, cfg.num_experts))
        o.copy_(_bf16(o.float().numpy() + sh))

    got = ep_forward(x, partial, add_shared)
    full, idx, _, _ = O.moe_forward(L, xb)
    # How many of the call's routes this rank's experts served.
    served = int(((idx >= b) & (idx < e)).sum())
    out[rank] = (got.float().numpy(), full, (b, e), served)
    dist.destroy_process_group()


@pytest.mark.parametrize("world,shared_gate,E,k", [(2, False, 12, 3), (3, True, 12, 3),
                                                   (4, True, 256, 8), (8, False, 256, 8)])
def test_ep_ranks_sum_to_the_layer(world, shared_gate, E, k):
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_rank, args=(world, port, shared_gate, E, k, out), nprocs=world,
                       start_method="spawn")
    got0, full = out[0][:2]
    for r in range(1, world):
        assert np.array_equal(out[r][0], got0)          # every rank holds the same sum
    # The ranks' expert blocks tile [0, E), and together they served every route
    # of the call exactly once (the shared expert is added once, after the sum).
    spans = sorted(out[r][2] for r in range(world))
    assert spans[0][0] == 0 and spans[-1][1] == E
    assert all(a[1] == b[0] for a, b in zip(spans, spans[1:]))
    assert sum(out[r][3] for r in range(world)) == full.shape[0] * k
    rms = float(np.sqrt(np.mean(full ** 2)))
    # BF16 partials, a BF16 sum, one BF16 rounding after the shared expert.
    assert np.max(np.abs(got0 - full)) <= 2e-2 * rms
