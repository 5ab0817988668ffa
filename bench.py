#!/usr/bin/env python
"""Benchmark of the MoE decode-layer forward on one GB300 (or N replicas).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload all|<name>]
    python bench.py --impl reference ...      # the fp64 CPU oracle, timed on host cores

A step is one ``moe_forward`` call (router, top-k, expert grouping, gate+up,
down+blend) over one batch of synthetic input of a workload.  By default every
workload is measured (tiny_n1, decode_n1, decode_n16, fp8_n64, nvfp4_n256:
N = 1 to 256 tokens); the line's headline fields (value, ms_per_step,
roofline, e2e, cpu_baseline) are the single-token decode's (decode_n1: hidden
2048, 256 experts, top-8), and ``workloads`` holds one entry per workload with
the same figures.  The L2 is flushed (a write of 2.5x its size) between steps,
outside the timed events, because the weights one call touches fit in L2.
Prints one JSON line.

Multi-GPU: the measured layer has no exchange step, so N GPUs run N
independent replicas ("scaling": "weak"); value = tokens of all ranks / the
slowest rank's time.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "MoE layer µs/call, tokens/s and HBM GB/s (frac of ~8 TB/s) at N=1–256"
HEADLINE = "decode_n1"
ALL_WORKLOADS = ("tiny_n1", "decode_n1", "decode_n16", "fp8_n64", "nvfp4_n256")
# The steps beside the five workloads' path -- the pre-expert RMSNorm with the
# shared-expert sigmoid gate, and the NVFP4 router -- on a workload's layer:
# measured in the default run without the end-to-end legs and the oracle
# (``next_rows``), or alone with --workload NAME.
VARIANTS = {
    "decode_n16+norm+gate": ("decode_n16", {"pre_expert_norm": True, "shared_gate": True}),
    "nvfp4_n256+nvfp4_router": ("nvfp4_n256", {"router_fmt": "nvfp4"}),
}
# Kernel sequence of each expert path, by the number of stage markers a call records.
STAGES_BY_MARKS = {
    2: ["fused"],
    5: ["router", "topk_group", "gate_up", "down_blend"],
    6: ["router", "topk_group", "gather", "gate_up", "down_combine"],
    7: ["router", "topk_group", "gather", "gate_up", "down", "combine"],
}


def parse_args(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--workload", default="all",
                   help="'all' (every workload; headline decode_n1) or one workload name")
    p.add_argument("--path", default="auto", choices=["auto", "token_major", "grouped"])
    p.add_argument("--tokens", type=int, default=0, help="override the workload's token count")
    p.add_argument("--experts", type=int, default=0,
                   help="override the workload's expert count (a smaller layer of the same kernels, "
                        "for profiler captures)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--oracle-budget", type=float, default=6.0,
                   help="seconds of oracle work per CPU baseline sample (each workload, each core count)")
    p.add_argument("--oracle-child", action="store_true", help=argparse.SUPPRESS)
    p.add_argument("--oracle-tokens", type=int, default=0, help=argparse.SUPPRESS)
    p.add_argument("--oracle-procs", type=int, default=1, help=argparse.SUPPRESS)
    return p.parse_args(argv)


def workload_names(args):
    if args.workload == "all":
        return list(ALL_WORKLOADS)
    return [args.workload]


# ------------------------------------------------------------------ helpers

def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def _src_hash(files) -> str:
    h = hashlib.sha256()
    d = os.path.join(ROOT, "mixture_experts_decode_router_gb300", "csrc")
    for f in files:
        with open(os.path.join(d, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def _ncu_entry(kernel: str, workload: str):
    """The committed ncu figures of `kernel` on `workload`, or None when the
    kernel's source changed since they were captured."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    try:
        with open(path) as f:
            d = json.load(f)
    except Exception:
        return None
    ent = d.get(workload, {}).get(kernel)
    if not ent:
        return None
    try:
        if _src_hash(ent["sources"]) != ent["sha"]:
            return None
    except OSError:
        return None
    return ent


def _traffic(kernel: str, workload: str):
    """dram bytes per launch of `kernel` from the committed ncu summary, or None."""
    ent = _ncu_entry(kernel, workload)
    return float(ent["dram_bytes_per_launch"]) if ent else None


def _tensor_pipe(kernel: str, workload: str):
    """Tensor-pipe active % of `kernel` from the committed ncu summary, or None."""
    ent = _ncu_entry(kernel, workload)
    v = ent.get("tensor_pipe_active_pct") if ent else None
    return float(v) if v is not None else None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled while the timed loop runs."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.06)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sms, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [v.strip() for v in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sms.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sms:
            return None
        sms.sort()
        return {"sm_mhz": sms[len(sms) // 2], "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sms)}


def max_over_ranks(v: float, device="cpu") -> float:
    """The largest value any rank holds (the slowest rank's time), or v alone."""
    import torch
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized() or dist.get_world_size() == 1:
        return v
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tokens_per_s(world: int, n_tokens: int, steps: int, max_ms: float) -> float:
    """Tokens all ranks processed over the slowest rank's device time."""
    return world * n_tokens * steps / (max_ms * 1e-3)


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


# ------------------------------------------------------------------ oracle (CPU) leg

def _oracle_pool_tokens(cfg) -> int:
    """Tokens of the oracle's sample pool: a few, fewer for the largest layer
    (each of its tokens touches 8 experts of 3 x 14.7 M elements)."""
    return 4 if cfg.hidden * cfg.inter >= 4 << 20 else 8


def _oracle_child(args):
    """Runs in a fresh process with no GPU and one BLAS thread per process: the
    oracle as it stands on a bounded sample of the workload's tokens, one token
    per call, in ``--oracle-procs`` worker processes that each take the pool's
    tokens in turn.  Prints one JSON object."""
    import numpy as np
    import torch

    from mixture_experts_decode_router_gb300 import synth
    from oracle import moe_oracle as O

    cfg = workload_config(args, args.workload)
    n_pool = _oracle_pool_tokens(cfg)
    # Input preparation (outside the timed region): the pool's rows, their
    # routing, and only the experts that routing touches, generated with every
    # host thread.
    torch.set_num_threads(max(1, os.cpu_count() or 1))
    x = synth.make_input(cfg, n_pool, "cpu", dup_frac=0.0, stream=7)
    xb = x.view(torch.int16).numpy().view(np.uint16)
    router = synth.make_router(cfg).view(torch.int16).numpy().view(np.uint16)
    bias = synth.make_bias(cfg)
    bias = bias.numpy() if bias is not None else None
    sgw = synth.make_shared_gate_w(cfg)
    sgw = sgw.view(torch.int16).numpy().view(np.uint16) if sgw is not None else None
    lg = O.router_logits(O.bf16_decode(xb), router)
    idx, _ = O.route(lg, cfg.routing, cfg.top_k, cfg.norm_topk_prob, cfg.routed_scaling_factor,
                     bias)
    need = sorted(set(int(e) for e in np.unique(idx)))

    def qm(tensor, experts):
        w, sc, s2 = {}, {}, {}
        for e in experts:
            q, s, s2v = synth.expert_matrix(cfg, tensor, e)
            w[e] = q.view(torch.int16).numpy().view(np.uint16) if q.dtype == torch.bfloat16 \
                else q.numpy()
            if s is not None:
                sc[e] = s.numpy()
            if s2v is not None:
                s2[e] = np.float32(s2v)
        return O.QMat(cfg.expert_fmt, w, sc or None, s2 or None)

    sh = [0] if cfg.shared_inter > 0 else []
    layer = O.OracleLayer(hidden=cfg.hidden, num_experts=cfg.num_experts, top_k=cfg.top_k,
                          inter=cfg.inter, shared_inter=cfg.shared_inter, routing=cfg.routing,
                          norm_topk_prob=cfg.norm_topk_prob,
                          routed_scaling_factor=cfg.routed_scaling_factor, router_w=router,
                          gate=qm("gate", need), up=qm("up", need), down=qm("down", need),
                          sh_gate=qm("sh_gate", sh) if sh else None,
                          sh_up=qm("sh_up", sh) if sh else None,
                          sh_down=qm("sh_down", sh) if sh else None,
                          correction_bias=bias, shared_gate_w=sgw)
    torch.set_num_threads(1)

    budget = args.oracle_budget
    limit = args.oracle_tokens if args.oracle_tokens > 0 else 10**9

    def work(wid: int, q):
        done = 0
        t0 = time.perf_counter()
        while done < limit:
            O.moe_forward(layer, xb, rows=[(wid + done) % n_pool])
            done += 1
            if time.perf_counter() - t0 >= budget:
                break
        q.put((done, time.perf_counter() - t0))

    procs = max(1, args.oracle_procs)
    if procs == 1:
        import queue
        q = queue.Queue()
        work(0, q)
        done, el = q.get()
    else:
        # This process never touches a GPU, so its workers may be forked.
        import multiprocessing as mp
        ctx = mp.get_context("fork")
        q = ctx.Queue()
        t0 = time.perf_counter()
        ps = [ctx.Process(target=work, args=(i, q)) for i in range(procs)]
        for p in ps:
            p.start()
        res = [q.get() for _ in ps]
        for p in ps:
            p.join()
        el = time.perf_counter() - t0
        done = sum(r[0] for r in res)
    print(json.dumps({"tokens": done, "seconds": el, "tokens_per_s": done / el, "procs": procs}))


def workload_config(args, name):
    """The workload's layer, with the --tokens / --experts overrides applied."""
    from mixture_experts_decode_router_gb300 import synth
    if name in VARIANTS:
        base, kw = VARIANTS[name]
        cfg = synth.WORKLOADS[base].with_(name=name, **kw)
    else:
        cfg = synth.WORKLOADS[name]
    if args.tokens > 0:
        cfg = cfg.with_(n_tokens=args.tokens, name=f"{cfg.name}@n{args.tokens}")
    if args.experts > 0:
        cfg = cfg.with_(num_experts=args.experts, top_k=min(cfg.top_k, args.experts),
                        name=f"{cfg.name}@e{args.experts}")
    return cfg


def _oracle_run(args, name, budget, procs, tokens=0):
    env = dict(os.environ)
    for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[v] = "1"
    env["CUDA_VISIBLE_DEVICES"] = ""
    cmd = [sys.executable, os.path.abspath(__file__), "--oracle-child", "--workload", name,
           "--oracle-budget", str(budget), "--oracle-tokens", str(tokens),
           "--oracle-procs", str(procs), "--tokens", str(args.tokens), "--experts", str(args.experts)]
    r = subprocess.run(cmd, capture_output=True, text=True, env=env, timeout=budget * 4 + 900)
    if r.returncode != 0:
        raise RuntimeError(f"oracle child failed:\n{r.stderr[-2000:]}")
    return json.loads(r.stdout.strip().splitlines()[-1])


def cpu_baseline(args, name: str, budget: float):
    """The oracle on one host core, and on every host core (one worker process
    per core, os.cpu_count()), each for about ``budget`` seconds."""
    ncpu = os.cpu_count() or 1
    one = _oracle_run(args, name, budget, 1)
    allc = _oracle_run(args, name, budget, ncpu) if ncpu > 1 else one
    what = (f"of {name}, one token per oracle call, fp64 numpy, 1 BLAS thread per process "
            f"(expert generation excluded)")
    return {"value": one["tokens_per_s"], "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"{one['tokens']} token(s) {what}, {one['seconds']:.1f} s",
            "all_cores": {"value": allc["tokens_per_s"], "unit": "tokens/s", "cores": allc["procs"],
                          "host_cpu_count": ncpu,
                          "sample": f"{allc['tokens']} token(s) {what}, {allc['procs']} worker "
                                    f"processes, {allc['seconds']:.1f} s"}}


# ------------------------------------------------------------------ our arm

def compute_dtype(fmt: str, grouped: bool) -> str:
    """The arithmetic the path computes in: BF16 operands (tensor cores on the
    grouped path, CUDA cores otherwise) with fp32 accumulation; FP8 / NVFP4
    weights dequantised to f16 for the grouped path's f16 MMA, to fp32 in the
    CUDA-core kernels."""
    if fmt == "bf16":
        return "bf16"
    w = "fp8e4m3" if fmt == "fp8_b128" else "nvfp4"
    return f"f16 ({w} weights dequantised, bf16 activations as f16, fp32 accumulate)" if grouped \
        else f"fp32 ({w} weights dequantised, bf16 activations)"


def e2e_line(world, n, H, steps, zero_copy_ms, copies_ms):
    """The end-to-end figure: the faster of the two host-buffer modes, both reported.
    Zero-copy wins at a few tokens (no copy launches); at many tokens the kernels'
    re-reads of x across the host link cost more than one copy in."""
    modes = {
        "zero_copy": ("x and out in pinned host memory, read and written by the kernels", zero_copy_ms),
        "with_copies": ("cudaMemcpyAsync H2D of x, the call on device buffers, D2H of out", copies_ms),
    }
    best = min(modes, key=lambda m: modes[m][1])
    line = {"value": round(whole_job_tokens_per_s(world, n, steps, modes[best][1]), 2), "unit": "tokens/s",
            "h2d_bytes_per_step": n * H * 2, "d2h_bytes_per_step": n * H * 2,
            "us_per_call": round(modes[best][1] / steps * 1e3, 3), "mode": best}
    for m, (what, ms) in modes.items():
        line[m] = {"value": round(whole_job_tokens_per_s(world, n, steps, ms), 2), "unit": "tokens/s",
                   "us_per_call": round(ms / steps * 1e3, 3), "what": what}
    return line


def stage_alg_bytes(cfg, n, distinct, touched, nm, has_bias):
    """Algorithmic bytes per launch of each stage of the path that ran."""
    from mixture_experts_decode_router_gb300 import synth
    H, I, S, E, k = cfg.hidden, cfg.inter, cfg.shared_inter, cfg.num_experts, cfg.top_k
    mb = synth.matrix_bytes
    fmt = cfg.expert_fmt
    nk = n * k
    w_gu = distinct * 2 * mb(fmt, I, H) + (2 * mb(fmt, S, H) if S else 0)
    w_dn = distinct * mb(fmt, H, I) + (mb(fmt, H, S) if S else 0)
    # The pre-expert RMSNorm: on the token-major path its own kernel at the
    # start of the gate/up stage (x in, the weight, the normalised rows out);
    # the grouped path's gather applies it as it copies (the weight only).
    norm = ((2 * n * H * 2 + H * 2) if nm == 5 else H * 2) if cfg.pre_expert_norm else 0
    return {
        "fused": touched,
        # router matrix (BF16 or NVFP4 codes + scales), x, the logits; the
        # shared-gate row and its logit when the layer has one
        "router": (mb(cfg.router_fmt, E, H) if cfg.router_fmt != "bf16" else E * H * 2) + n * H * 2 + n * E * 4
        + ((H * 2 + n * 4) if cfg.shared_gate else 0),
        # top-k (logits in, routes out) + grouping (routes in, counts/offsets/permutation out)
        "topk_group": n * E * 4 + nk * 8 + (4 * E if has_bias else 0)
        + nk * 4 + 4 * (3 * E + 1) + nk * 4,
        # token-major: fp32 activations; grouped: 16-bit activations
        "gate_up": w_gu + n * H * 2 + (4 if nm == 5 else 2) * (nk * I + n * S)
        + (2 * (nk * H + n * H) if nm in (6, 7) else 0) + (norm if nm == 5 else 0),
        "down_blend": w_dn + 4 * (nk * I + n * S) + n * H * 2 + nk * 8,
        "gather": 2 * 2 * (nk * H + n * H) + norm,
        "down": w_dn + 2 * (nk * I + n * S) + 4 * (nk * H + (n * H if S else 0)),
        "combine": 4 * (nk * H + (n * H if S else 0)) + n * H * 2 + nk * 4,
        # the down kernel with the combine folded in: weights and activations in,
        # the BF16 output and the route positions (its fp32 rows stay internal)
        "down_combine": w_dn + 2 * (nk * I + n * S) + n * H * 2 + nk * 4,
    }


def measure_workload(args, name, dev, flush, world, local, light=False):
    """Times one workload: K moe_forward calls (L2 flushed between them), the
    per-stage split, the end-to-end legs with host buffers, and a device copy
    of the same byte count.  Returns the workload's entry of the JSON line
    (device times are this rank's; the caller takes the maximum over ranks)."""
    import numpy as np
    import torch

    from mixture_experts_decode_router_gb300 import binding as B
    from mixture_experts_decode_router_gb300 import synth
    from mixture_experts_decode_router_gb300.layer import MoeLayer

    cfg = workload_config(args, name)
    n = cfg.n_tokens
    lw = synth.make_weights(cfg, dev)
    x = synth.make_input(cfg, device=dev)
    layer = MoeLayer(lw, n, args.path)
    out = torch.empty(n, cfg.hidden, dtype=torch.bfloat16, device=dev)
    idx = torch.empty(n, cfg.top_k, dtype=torch.int32, device=dev)
    wts = torch.empty(n, cfg.top_k, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    sptr = stream.cuda_stream

    def step():
        s = B.moe_forward(layer.c_cfg, layer.c_w, x, n, out, idx, wts, layer.ws, layer.ws_bytes,
                          sptr)
        if s != B.MOE_OK:
            raise B.MoeError(B.moe_status_string(s))

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()

    K = args.steps
    ev_s = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ev_e = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    clocks = ClockSampler(local)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)       # let the sampler start before the timed loop
    t0 = time.perf_counter()
    for i in range(K):
        flush.zero_()
        ev_s[i].record(stream)
        step()
        ev_e[i].record(stream)
    torch.cuda.synchronize()
    t1 = time.perf_counter()
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    per = np.array([a.elapsed_time(b) for a, b in zip(ev_s, ev_e)])   # ms
    dev_ms = max_over_ranks(float(per.sum()), dev)

    # Touched bytes from this input's routing (constant over the steps).
    idx_h = idx.cpu().numpy()
    touched = synth.touched_bytes(cfg, idx_h)
    distinct = len(np.unique(idx_h))

    # Per-stage durations (moe_forward_timed: events between the kernels).
    Kp = min(K, 500)
    nev = 10
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(nev)] for _ in range(Kp)]
    for row in evs:          # torch creates the CUDA event on its first record
        for e in row:
            e.record(stream)
    torch.cuda.synchronize()
    nm = 0
    for i in range(Kp):
        flush.zero_()
        s, nm = B.moe_forward_timed(layer.c_cfg, layer.c_w, x, n, out, idx, wts, layer.ws,
                                    layer.ws_bytes, sptr, [e.cuda_event for e in evs[i]])
        if s != B.MOE_OK or nm not in STAGES_BY_MARKS:
            raise B.MoeError(f"timed forward: status {s}, markers {nm}")
    torch.cuda.synchronize()
    stages_run = STAGES_BY_MARKS[nm]
    stage_ms = np.array([[evs[i][j].elapsed_time(evs[i][j + 1]) for j in range(nm - 1)]
                         for i in range(Kp)]).mean(axis=0)
    dev_err = layer.device_error()
    if dev_err:
        raise B.MoeError(f"device error word {dev_err}")

    alg = stage_alg_bytes(cfg, n, distinct, touched, nm, lw.correction_bias is not None)
    peak, peak_kind = _peaks()
    dom = stages_run[int(np.argmax(stage_ms))]
    dom_ms = float(stage_ms[stages_run.index(dom)])
    achieved = alg[dom] / (dom_ms * 1e-3) / 1e9
    stages = {s: {"us": round(float(stage_ms[j]) * 1e3, 3), "alg_bytes": int(alg[s]),
                  "gbs": round(alg[s] / (stage_ms[j] * 1e-3) / 1e9, 1),
                  "frac_of_measured": round(alg[s] / (stage_ms[j] * 1e-3) / 1e9 / peak, 4)}
              for j, s in enumerate(stages_run)}

    e2e, size_copy, copy_ratio = None, None, None
    if not light:
        # End to end through the public API with host buffers, two ways, each step
        # taking a fresh input from pinned host memory and leaving the result there:
        # (a) zero-copy: x and out are the pinned host buffers themselves; the
        #     kernels read x and write out across the host link (NVLink-C2C);
        # (b) explicit copies: H2D of x, the call on device buffers, D2H of out.
        x_h = x.cpu().pin_memory()
        out_h = torch.empty(n, cfg.hidden, dtype=torch.bfloat16).pin_memory()
        x_d = torch.empty_like(x)
        Ke = min(K, 1000)

        def timed_e2e(zero_copy):
            starts = [torch.cuda.Event(enable_timing=True) for _ in range(Ke)]
            ends = [torch.cuda.Event(enable_timing=True) for _ in range(Ke)]
            for i in range(Ke):
                flush.zero_()
                starts[i].record(stream)
                if zero_copy:
                    s = B.moe_forward(layer.c_cfg, layer.c_w, x_h, n, out_h, idx, wts, layer.ws, layer.ws_bytes, sptr)
                else:
                    x_d.copy_(x_h, non_blocking=True)
                    s = B.moe_forward(layer.c_cfg, layer.c_w, x_d, n, out, idx, wts, layer.ws, layer.ws_bytes, sptr)
                if s != B.MOE_OK:
                    raise B.MoeError(B.moe_status_string(s))
                if not zero_copy:
                    out_h.copy_(out, non_blocking=True)
                ends[i].record(stream)
            torch.cuda.synchronize()
            return max_over_ranks(float(np.sum([a.elapsed_time(b) for a, b in zip(starts, ends)])), dev)

        e2e_ms = timed_e2e(True)
        if not torch.equal(out_h.view(torch.int16), out.cpu().view(torch.int16)):
            raise B.MoeError("zero-copy output differs from the device-buffer output")
        e2e_copy_ms = timed_e2e(False)

        # A device-to-device copy moving the call's touched bytes (half read, half
        # written: the measured peak's own method), timed the same way: what one
        # launch of plain streaming reaches at this size on this GPU.
        half = max(16, touched // 2 // 16 * 16)
        src = torch.ones(half, dtype=torch.uint8, device=dev)
        dst = torch.empty_like(src)
        for _ in range(3):
            flush.zero_()
            dst.copy_(src)
        cs = [torch.cuda.Event(enable_timing=True) for _ in range(Ke)]
        ce = [torch.cuda.Event(enable_timing=True) for _ in range(Ke)]
        for i in range(Ke):
            flush.zero_()
            cs[i].record(stream)
            dst.copy_(src)
            ce[i].record(stream)
        torch.cuda.synchronize()
        copy_ms = float(np.mean([a.elapsed_time(b) for a, b in zip(cs, ce)]))
        del src, dst
        e2e = e2e_line(world, n, cfg.hidden, Ke, e2e_ms, e2e_copy_ms)
        size_copy = {
            "us": round(copy_ms * 1e3, 3), "bytes": 2 * half,
            "gbs": round(2 * half / (copy_ms * 1e-3) / 1e9, 1),
            "frac_of_measured": round(2 * half / (copy_ms * 1e-3) / 1e9 / peak, 4),
            "what": "torch copy_ of touched/2 bytes on the device (read + write = the call's touched "
                    "bytes), L2 flushed, event-timed like the call"}
        copy_ratio = round((dev_ms / K) / copy_ms, 3)

    ms_step = dev_ms / K
    grouped = nm in (6, 7)
    # This library's kernels per call: one a stage, plus the norm (the grouped
    # path's gather applies it), plus the
    # shared-gate row's own router launch beside the CUDA-core NVFP4 router (on
    # the grouped path the top-k kernel forms it), plus the BF16 expansion of
    # an NVFP4 router for the tensor-core router.
    per_call = len(stages_run) + (1 if cfg.pre_expert_norm and not grouped else 0) \
        + (1 if cfg.shared_gate and cfg.router_fmt != "bf16" and not grouped else 0) \
        + (1 if cfg.router_fmt != "bf16" and grouped else 0)
    entry = {
        "us_per_call": round(ms_step * 1e3, 3),
        "us_per_call_p10_p50_p90": [round(float(np.percentile(per, q)) * 1e3, 3) for q in (10, 50, 90)],
        "tokens_per_s": round(whole_job_tokens_per_s(world, n, K, dev_ms), 2),
        "steps": K,
        "touched_bytes": touched,
        "distinct_experts": distinct,
        "hbm_gbs": round(touched / (ms_step * 1e-3) / 1e9, 1),
        "hbm_frac_of_measured": round(touched / (ms_step * 1e-3) / 1e9 / peak, 4),
        "size_matched_copy": size_copy,
        "call_time_over_copy_time": copy_ratio,
        "dtype": compute_dtype(cfg.expert_fmt, grouped),
        "config": {"workload": cfg.name, "n_tokens": n, "hidden": cfg.hidden,
                   "num_experts": cfg.num_experts, "top_k": cfg.top_k, "inter": cfg.inter,
                   "shared_inter": cfg.shared_inter, "routing": cfg.routing,
                   "expert_fmt": cfg.expert_fmt, "dup_frac": cfg.dup_frac, "path": args.path,
                   "router_fmt": cfg.router_fmt, "pre_expert_norm": cfg.pre_expert_norm,
                   "shared_gate": cfg.shared_gate},
        "wall_s_timed_loop": round(t1 - t0, 3),
        "gpu_launches": K * per_call,
        "stages": stages,
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": round(achieved, 1),
                     "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": _traffic(dom, cfg.name),
                     "tensor_pipe_active_pct": _tensor_pipe(dom, cfg.name),
                     "alg_bytes_per_launch": int(alg[dom]),
                     "avg_launch_us": round(dom_ms * 1e3, 3)},
        "e2e": e2e,
        "clocks": clk,
    }
    del layer, lw, x, out
    torch.cuda.empty_cache()
    return entry


def run_ours(args):
    import torch
    import torch.distributed as dist

    from mixture_experts_decode_router_gb300 import binding as B

    world, rank, local = _dist()
    if world > 1:
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    B.load()

    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(int(2.5 * l2) // 4 * 4, dtype=torch.uint8, device=dev)
    names = workload_names(args)
    head = HEADLINE if HEADLINE in names else names[0]
    entries = {nm: measure_workload(args, nm, dev, flush, world, local) for nm in names}
    next_rows = ({nm: measure_workload(args, nm, dev, flush, world, local, light=True) for nm in VARIANTS}
                 if args.workload == "all" else {})

    # The oracle on the host cores (rank 0 at N = 1 only), after every GPU
    # measurement so the two never share the host.
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        for nm in names:
            entries[nm]["cpu_baseline"] = cpu_baseline(args, nm, args.oracle_budget)

    if rank == 0:
        h = entries[head]
        K = args.steps
        line = {
            "metric": METRIC,
            "value": h["tokens_per_s"],
            "unit": "tokens/s",
            "n_gpus": world,
            "steps": K,
            "warmup": args.warmup,
            "ms_per_step": round(h["us_per_call"] / 1e3, 6),
            "us_per_call": h["us_per_call"],
            "us_per_call_p10_p50_p90": h["us_per_call_p10_p50_p90"],
            "hbm_gbs": h["hbm_gbs"],
            "hbm_frac_of_measured": h["hbm_frac_of_measured"],
            "touched_bytes": h["touched_bytes"],
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": h["dtype"],
            "data": "synthetic (seeded; weights N(0,0.02), input N(0,1))",
            "config": dict(h["config"], l2="flushed between steps (2.5x L2 write), flush outside the events",
                           parallelism=f"replicas{world}" if world > 1 else "single"),
            "gpu_launches": h["gpu_launches"],
            "roofline": h["roofline"],
            "e2e": h["e2e"],
            "clocks": h["clocks"],
            "cpu_baseline": h.get("cpu_baseline"),
            "size_matched_copy": h["size_matched_copy"],
            "stages": h["stages"],
            "workloads": entries,
            "next_rows": next_rows,
        }
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


# ------------------------------------------------------------------ reference arm

def run_reference(args):
    """The fp64 oracle on the host cores (one worker process per core), on the
    headline workload: each worker takes one token per oracle call until the
    run has made max(1, steps) tokens per worker or about a minute has passed."""
    world, rank, _ = _dist()
    if rank != 0:
        return
    name = HEADLINE if args.workload == "all" else args.workload
    cfg = workload_config(args, name)
    ncpu = os.cpu_count() or 1
    d = _oracle_run(args, name, 60.0, ncpu, tokens=max(1, args.steps))
    tok_s = d["tokens_per_s"]
    line = {
        "metric": METRIC, "impl": "reference", "value": round(tok_s, 4), "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * cfg.n_tokens / tok_s, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": cfg.name, "n_tokens": cfg.n_tokens},
        "cpu_baseline": {"kind": "oracle", "cores": d["procs"], "host_cpu_count": ncpu,
                         "sample": f"{d['tokens']} token(s) of {name}, one token per oracle call, "
                                   f"fp64 numpy, {d['procs']} worker processes with 1 BLAS thread "
                                   f"each, {d['seconds']:.1f} s",
                         "value": round(tok_s, 4), "unit": "tokens/s"},
        "e2e": {"value": round(tok_s, 4), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def main(argv=None):
    args = parse_args(argv)
    if args.oracle_child:
        _oracle_child(args)
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
