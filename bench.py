#!/usr/bin/env python3
"""Benchmark of the resolvent-operator causal head on GB300.

A step is one call of the hot path on one batch of seeded synthetic inputs already resident
in HBM: resolvent_head_forward (gate preparation + fused head kernel, and the chain scan for
heads at qk = 0, beta = 0) for the head workloads, resolvent_chain_scan for the chain
workload. The default workload is the gated softmax head (B=8 H=16 n=2048 d=dv=64 bf16,
(beta, qk, g) = (1, 1, 0.5)).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

Prints one JSON line (rank 0). `--impl reference` times the fp64 CPU oracle instead, on the
host cores, with a bounded sample of the same workload per step.
Multi-GPU (torchrun): every rank runs its own full batch (independent heads, no collective
on the data path): weak scaling; the time is the max over ranks.
"""
import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

L2_BYTES = 129 * 1024 * 1024
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=50)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--workload", default="gated_softmax", choices=sorted(W.WORKLOADS))
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--cpu-seconds", type=float, default=12.0,
                   help="target CPU time of the oracle sample (cpu_baseline and --impl reference)")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--B", type=int, default=None, help="override the batch (smaller profiling cases)")
    p.add_argument("--H", type=int, default=None, help="override the heads")
    p.add_argument("--n", type=int, default=None, help="override the sequence length")
    return p.parse_args()


def make_inputs(args):
    kw = {k: getattr(args, k) for k in ("B", "H", "n") if getattr(args, k) is not None}
    return W.WORKLOADS[args.workload](**kw)


# ------------------------------------------------------------------ distributed plumbing

def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def dist_init(world, backend):
    if world > 1:
        import torch.distributed as dist
        if not dist.is_initialized():
            dist.init_process_group(backend)


def dist_max(x: float, world: int, device) -> float:
    """Max of a host scalar over ranks (identity at world size 1)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def dist_barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------------ work accounting

def live_entries(u_head, g):
    """Causal entries (i, j) whose path modulus R_ij = prod_{k=j+1..i} m_k is nonzero in fp32,
    the precision the kernel evaluates G in: no exact zero gate on the path and the product
    at least the smallest fp32 subnormal (2^-149). Entries past it are exact zeros of the evaluation and
    count as no work. Per row the live keys are a contiguous run ending at j = i."""
    u = np.asarray(u_head, dtype=np.float64)
    n = u.size
    m = np.clip((1.0 - g) + g * u, 0.0, 1.0)
    m[0] = 1.0  # a_0 is never read
    with np.errstate(divide="ignore"):
        lg = np.where(m > 0.0, np.log2(np.maximum(m, 1e-300)), -1e9)
    L = np.cumsum(lg)  # L[k] = sum_{t<=k} log2 m_t, non-increasing
    # R_ij = 2^(L[i] - L[j]) >= 2^-149  <=>  -L[j] >= -L[i] - 149 (a suffix of j, -L ascending)
    first = np.searchsorted(-L, -L - 149.0, side="left")
    return float(np.sum(np.arange(n) - first + 1))


def head_work(hi: W.HeadInputs):
    """Algorithmic flops of the fused head kernel(s) for one call: per head with qk != 0,
    live entries x (2 d + 2 dv c), c = 2 with complex gates (g != 0), else 1. Heads with
    qk = 0 run as O(n) chains (O_i = y_i Z_i^-beta) and count as chain tokens."""
    beta, qk, g = hi.switches_bh()
    flops, chain_tokens = 0.0, 0
    for h in range(hi.B * hi.H):
        if qk[h] == 0.0:
            chain_tokens += hi.n
            continue
        per_entry = 2 * hi.d + 2 * hi.dv * (2 if g[h] != 0.0 else 1)
        flops += per_entry * (live_entries(hi.u[h], g[h]) if g[h] != 0.0
                              else hi.n * (hi.n + 1) / 2)
    return flops, chain_tokens


def position_work(pi: W.PositionInputs):
    """Algorithmic flops of the position-only head: per head, 2 dv per causal entry whose
    kernel value e^{qk a(d) - M} is not 0 once rounded to bf16 (an offset d contributes
    n - d entries)."""
    beta, qk = pi.switches_bh()
    flops = 0.0
    cnt = np.arange(pi.n, 0, -1, dtype=np.float64)  # entries at offset d: n - d
    for h in range(pi.B * pi.H):
        t = qk[h] * pi.a[h % pi.H].astype(np.float64)
        live = np.exp(t - t.max()) >= 2.0 ** -134
        flops += 2 * pi.dv * float(cnt[live].sum())
    return flops


def chain_bytes_per_token(dv, b_bytes=4):
    return b_bytes * dv + 8 + 8 * dv  # read b and (u, theta); write y_re, y_im


# ------------------------------------------------------------------ clocks

class Clocks:
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100", "-f", self.path],
                stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self, t0, t1):
        """Summary of the samples taken in [t0, t1] (wall clock), widened to the whole
        sampling window when fewer than 3 samples fall inside."""
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 10:
                    continue
                try:
                    ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                    rows.append((ts, float(parts[2]), float(parts[3]), parts[5:]))
                except ValueError:
                    continue
        os.unlink(self.path)
        inside = [r for r in rows if t0 - 1.0 <= r[0] <= t1 + 1.0]
        use = inside if len(inside) >= 3 else rows
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in use for i, v in enumerate(r[3][1:5])
                          if v.lower().startswith("active")})
        return {"sm_mhz": statistics.median(r[1] for r in use), "sm_max_mhz": max(r[2] for r in use),
                "reasons": reasons, "samples": len(use), "samples_in_timed_region": len(inside)}


KERNEL_SOURCES = {"head_fwd_kernel": ["head_fwd.cu", "head_common.cuh", "common.cuh", "gate_products.cuh"],
                  "chain_scan_kernel": ["chain_scan.cu", "common.cuh"],
                  "operator_kernel": ["operator.cu", "head_common.cuh", "common.cuh", "gate_products.cuh"],
                  "position_head_kernel": ["position.cu", "head_common.cuh", "common.cuh", "gate_products.cuh"]}


def measured_traffic(kernel, workload):
    """DRAM bytes per launch from profiles/dram_traffic.txt, if the kernel's sources are
    unchanged since that capture (else None)."""
    import hashlib
    m = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "gated_causal_attention_gb300", "csrc", f), "rb") as fh:
            m.update(fh.read())
    digest = m.hexdigest()[:16]
    try:
        with open(os.path.join(ROOT, "profiles", "dram_traffic.txt")) as fh:
            for line in fh:
                parts = line.split()
                if len(parts) >= 4 and not line.startswith("#") and parts[0] == kernel \
                        and parts[1] == workload and parts[2] == digest:
                    return float(parts[3])
    except OSError:
        pass
    return None


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {k: float(p[k]) for k in FALLBACK_PEAKS}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


# ------------------------------------------------------------------ the oracle on the host

def oracle_sample_head(hi: W.HeadInputs, target_s: float, seed: int = 1):
    """Times the oracle on seeded random rows of every head; returns (rows/s, rows, s)."""
    import oracle
    oracle.build()
    rng = np.random.default_rng(seed)
    beta, qk, g = [np.asarray(x, np.float32).astype(np.float64) for x in hi.switches_bh()]

    def run(count):
        rows = np.sort(rng.choice(hi.n, size=max(1, count), replace=False))
        t = time.perf_counter()
        oracle.head_rows(hi.q, hi.k, hi.u, hi.theta, hi.v, beta, qk, g, rows)
        return rows.size * hi.B * hi.H, time.perf_counter() - t

    tok, dt = run(min(hi.n, 4))
    count = int(min(hi.n, max(1, 4 * target_s / max(dt, 1e-3))))
    tok, dt = run(count)
    return tok / dt, tok, dt


def oracle_sample_chain(ci: W.ChainInputs, target_s: float):
    import oracle
    oracle.build()
    g = np.asarray(ci.switches_bh()[2], np.float32).astype(np.float64)

    def run(heads):
        t = time.perf_counter()
        oracle.chain_heads(ci.u[:heads], ci.theta[:heads], g[:heads], ci.b[:heads])
        return heads * ci.n, time.perf_counter() - t

    tok, dt = run(1)
    heads = int(min(ci.B * ci.H, max(1, target_s / max(dt, 1e-3))))
    tok, dt = run(heads)
    return tok / dt, tok, dt


def oracle_sample_operator(hi: W.HeadInputs, target_s: float):
    """The oracle's dense W of whole heads: entries per second."""
    import oracle
    oracle.build()
    beta, qk, g = [np.asarray(x, np.float32).astype(np.float64) for x in hi.switches_bh()]
    heads, t0 = 0, time.perf_counter()
    while heads < hi.B * hi.H and (heads == 0 or time.perf_counter() - t0 < target_s):
        oracle.operator(hi.q[heads], hi.k[heads], hi.u[heads], hi.theta[heads], beta[heads],
                        qk[heads], g[heads])
        heads += 1
    dt = time.perf_counter() - t0
    return heads * hi.n * hi.n / dt, heads * hi.n * hi.n, dt


def oracle_sample_position(pi: W.PositionInputs, target_s: float):
    """The oracle on whole position-only heads: one head (one core) for a short sample,
    else as many heads as the host has cores, in one parallel pass."""
    import oracle
    oracle.build()
    beta, qk = [np.asarray(x, np.float32).astype(np.float64) for x in pi.switches_bh()]
    heads = 1 if target_s < 8.0 else max(1, min(pi.B * pi.H, oracle.max_threads()))
    t0 = time.perf_counter()
    oracle.position_heads(pi.a, pi.v[:heads], beta[:heads], qk[:heads])
    dt = time.perf_counter() - t0
    return heads * pi.n / dt, heads * pi.n, dt


def cpu_cores():
    import oracle
    oracle.build()
    return oracle.max_threads()


def config_of(args, inp, world):
    if isinstance(inp, W.ChainInputs):
        cfg = {"workload": args.workload, "B": inp.B, "H": inp.H, "n": inp.n, "dv": inp.dv,
               "dtype_b": "fp32", "switches": "(0,0,1)"}
    elif isinstance(inp, W.PositionInputs):
        sw = sorted({(float(b), float(q)) for b, q in zip(inp.beta, inp.qk)})
        cfg = {"workload": args.workload, "B": inp.B, "H": inp.H, "n": inp.n, "dv": inp.dv,
               "dtype_v": inp.dtype, "logits": "a_h(d) = -2^(-8(h+1)/H) d + 0.5 N(0,1)",
               "switches (beta, qk; g = 0)": sw[0] if len(sw) == 1 else f"{len(sw)} per-head settings"}
    else:
        sw = sorted({(float(b), float(q), float(g)) for b, q, g in zip(inp.beta, inp.qk, inp.g)})
        cfg = {"workload": args.workload, "B": inp.B, "H": inp.H, "n": inp.n, "d": inp.d,
               "dv": inp.dv, "dtype_qkv": inp.dtype,
               "switches": sw[0] if len(sw) == 1 else f"{len(sw)} per-head settings"}
    cfg["parallelism"] = f"replicas{world}" if world > 1 else "single"
    return cfg


# ------------------------------------------------------------------ reference arm

def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    inp = make_inputs(args)
    per_step = max(1.0, args.cpu_seconds / max(1, args.steps + args.warmup) * 2)
    is_chain = isinstance(inp, W.ChainInputs)
    is_op = args.workload == "operator"
    is_pos = isinstance(inp, W.PositionInputs)
    if is_chain:
        sample = lambda: oracle_sample_chain(inp, per_step)
    elif is_pos:
        sample = lambda: oracle_sample_position(inp, per_step)
    elif is_op:
        sample = lambda: oracle_sample_operator(inp, per_step)
    else:
        sample = lambda: oracle_sample_head(inp, per_step, seed=7)
    for _ in range(args.warmup):
        sample()
    rates, toks, secs = [], 0, 0.0
    for _ in range(args.steps):
        r, t, s = sample()
        rates.append(r)
        toks += t
        secs += s
    value = toks / secs
    cores = cpu_cores()
    unit = "entries/s" if is_op else "tokens/s"
    metric = ("chain tokens/s (B*H*n/s)" if is_chain else
              "operator entries/s (B*H*n*n/s)" if is_op else
              "position tokens/s (B*H*n/s)" if is_pos else "head tokens/s (B*H*n/s)")
    line = {"impl": "reference", "metric": metric,
            "value": value, "unit": unit, "n_gpus": 0, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * secs / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded, workloads.py)", "config": config_of(args, inp, 1),
            "cpu_baseline": {"value": value, "unit": unit, "cores": cores, "kind": "oracle",
                             "sample": ("whole heads of the chain" if is_chain else
                                        "whole heads' W" if is_op else
                                        "whole position-only heads" if is_pos else
                                        "seeded random rows of every head") +
                             f", {toks} {'entries' if is_op else 'tokens'} in {secs:.1f} s"},
            "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ our arm

def run_ours(args):
    import torch
    rank, world, local = dist_env()
    assert world == args.gpus or world == 1, "--gpus must match the torchrun world size"
    dist_init(world, "nccl")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    import gated_causal_attention_gb300 as R
    import __graft_entry__
    __graft_entry__.build()

    inp = make_inputs(args)
    is_chain = isinstance(inp, W.ChainInputs)
    is_op = args.workload == "operator"
    is_pos = isinstance(inp, W.PositionInputs)
    shp = (inp.B, inp.H, inp.n)
    tdev = lambda x, s, dt=torch.float32: torch.from_numpy(np.ascontiguousarray(x).reshape(s)).to(
        device=device, dtype=dt)
    status = R.new_status(device)
    if is_chain:
        u, th = tdev(inp.u, shp), tdev(inp.theta, shp)
        b = tdev(inp.b, (*shp, inp.dv))
        out = (torch.empty_like(b), torch.empty_like(b))
        ws = torch.empty(max(1, R.chain_workspace_bytes(*shp, inp.dv)), dtype=torch.uint8, device=device)
        step = lambda: R.chain_scan(u, th, inp.g, b, out=out, workspace=ws, status=status, sync=False)
        tokens = inp.B * inp.H * inp.n
        work = tokens * chain_bytes_per_token(inp.dv)
        host_in = [inp.u, inp.theta, inp.b]
    elif is_op:
        q, k = tdev(inp.q, (*shp, inp.d), torch.bfloat16), tdev(inp.k, (*shp, inp.d), torch.bfloat16)
        u, th = tdev(inp.u, shp), tdev(inp.theta, shp)
        out = (torch.empty(*shp, inp.n, device=device), torch.empty(*shp, inp.n, device=device))
        ws = torch.empty(max(1, R.operator_workspace_bytes(*shp, inp.d, torch.bfloat16)),
                         dtype=torch.uint8, device=device)
        step = lambda: R.operator(q, k, u, th, inp.beta, inp.qk, inp.g, out=out, workspace=ws,
                                  status=status, sync=False)
        tokens = inp.B * inp.H * inp.n * inp.n  # entries of W
        # bytes: W written (8 B per entry); q, k read (2 B x d each per token); u, theta
        work = tokens * 8 + inp.B * inp.H * inp.n * (4 * inp.d + 8)
        host_in = [inp.q, inp.k, inp.u, inp.theta]
    elif is_pos:
        a = tdev(inp.a, (inp.H, inp.n))
        v = tdev(inp.v, (*shp, inp.dv), torch.bfloat16)
        out = torch.empty(*shp, inp.dv, device=device)
        ws = torch.empty(max(1, R.position_workspace_bytes(*shp, inp.dv, torch.bfloat16)),
                         dtype=torch.uint8, device=device)
        step = lambda: R.position_head(a, v, inp.beta, inp.qk, out=out, workspace=ws, status=status,
                                       sync=False)
        tokens = inp.B * inp.H * inp.n
        work = position_work(inp)
        host_in = [inp.a, inp.v]
    else:
        dt = torch.bfloat16 if inp.dtype == "bf16" else torch.float32
        q, k = tdev(inp.q, (*shp, inp.d), dt), tdev(inp.k, (*shp, inp.d), dt)
        v = tdev(inp.v, (*shp, inp.dv), dt)
        u, th = tdev(inp.u, shp), tdev(inp.theta, shp)
        out = (torch.empty(*shp, inp.dv, device=device), torch.empty(*shp, inp.dv, device=device))
        ws = torch.empty(max(1, R.head_workspace_bytes(*shp, inp.d, inp.dv, dt)), dtype=torch.uint8,
                         device=device)
        step = lambda: R.head_forward(q, k, u, th, v, inp.beta, inp.qk, inp.g, out=out, workspace=ws,
                                      status=status, sync=False)
        tokens = inp.B * inp.H * inp.n
        work, chain_tokens = head_work(inp)
        host_in = [inp.q, inp.k, inp.v, inp.u, inp.theta]

    # warm-up, and a refusal check of the inputs
    for _ in range(args.warmup):
        step()
    R.status_sync(status)
    launches_per_step = R.last_launch_count()
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=device)

    clocks = Clocks(torch.cuda.current_device() if "CUDA_VISIBLE_DEVICES" not in os.environ
                    else local)
    clocks.start()
    time.sleep(0.3)
    R.profile_enable(True)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    dist_barrier(world)
    torch.cuda.synchronize()
    w0 = time.time()
    for i in range(args.steps):
        flush.zero_()  # L2 flush between timed iterations (outside the step's events)
        ev[i][0].record()
        step()
        ev[i][1].record()
    torch.cuda.synchronize()
    dist_barrier(world)
    w1 = time.time()
    kernel_ms = R.profile_collect()
    R.profile_enable(False)
    R.status_sync(status)
    clk = clocks.stop(w0, w1)
    step_ms = [a.elapsed_time(b) for a, b in ev]
    ms_local = sum(step_ms) / len(step_ms)
    ms = dist_max(ms_local, world, device)
    value = tokens * world / (ms / 1e3)

    pk, pk_kind = peaks()
    kern = statistics.mean(kernel_ms) if kernel_ms else float("nan")
    if is_chain or is_op:
        kname = "chain_scan_kernel" if is_chain else "operator_kernel"
        achieved = work / (kern / 1e3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / pk["hbm_gbs"],
                "traffic": measured_traffic(kname, args.workload), "kernel": kname,
                "kernel_ms": kern, "peak_kind": pk_kind,
                "algorithmic_bytes_per_launch": work}
    else:
        kname = "position_head_kernel" if is_pos else "head_fwd_kernel"
        achieved = work / (kern / 1e3) / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                "frac": achieved / pk["bf16_tflops"],
                "traffic": measured_traffic(kname, args.workload), "kernel": kname,
                "kernel_ms": kern, "peak_kind": pk_kind + " burst",
                "algorithmic_flops_per_launch": work}

    # end to end through the public API, pinned host buffers in and out
    e2e = None
    if not args.no_e2e:
        pinned = [torch.from_numpy(np.ascontiguousarray(x)).pin_memory() for x in host_in]
        if is_op:
            pinned[0] = pinned[0].to(torch.bfloat16).pin_memory()
            pinned[1] = pinned[1].to(torch.bfloat16).pin_memory()
        elif is_pos:
            pinned[1] = pinned[1].to(torch.bfloat16).pin_memory()
        elif not is_chain and inp.dtype == "bf16":
            pinned[0] = pinned[0].to(torch.bfloat16).pin_memory()
            pinned[1] = pinned[1].to(torch.bfloat16).pin_memory()
            pinned[2] = pinned[2].to(torch.bfloat16).pin_memory()
        outs_host = [torch.empty((out if is_pos else out[0]).shape, dtype=torch.float32).pin_memory()
                     for _ in range(1 if is_pos else 2)]
        h2d = sum(p.numel() * p.element_size() for p in pinned)
        d2h = sum(o.numel() * o.element_size() for o in outs_host)

        def e2e_step():
            dv_in = [p.to(device, non_blocking=True) for p in pinned]
            if is_chain:
                uu, tt, bb = dv_in
                o = R.chain_scan(uu.view(shp), tt.view(shp), inp.g, bb.view(*shp, inp.dv), out=out,
                                 workspace=ws, status=status, sync=False)
            elif is_op:
                qq, kk, uu, tt = dv_in
                o = R.operator(qq.view(*shp, inp.d), kk.view(*shp, inp.d), uu.view(shp),
                               tt.view(shp), inp.beta, inp.qk, inp.g, out=out, workspace=ws,
                               status=status, sync=False)
            elif is_pos:
                aa, vv = dv_in
                o = (R.position_head(aa.view(inp.H, inp.n), vv.view(*shp, inp.dv), inp.beta, inp.qk,
                                     out=out, workspace=ws, status=status, sync=False),)
            else:
                qq, kk, vv, uu, tt = dv_in
                o = R.head_forward(qq.view(*shp, inp.d), kk.view(*shp, inp.d), uu.view(shp),
                                   tt.view(shp), vv.view(*shp, inp.dv), inp.beta, inp.qk, inp.g,
                                   out=out, workspace=ws, status=status, sync=False)
            for oh, od in zip(outs_host, o):
                oh.copy_(od, non_blocking=True)

        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize()
        dist_barrier(world)
        a, b2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(args.steps):
            e2e_step()
        b2.record()
        torch.cuda.synchronize()
        e_ms = dist_max(a.elapsed_time(b2) / args.steps, world, device)
        R.status_sync(status)
        e2e = {"value": tokens * world / (e_ms / 1e3), "unit": "entries/s" if is_op else "tokens/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e_ms}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rate, toks, secs = (oracle_sample_chain(inp, args.cpu_seconds) if is_chain
                            else oracle_sample_operator(inp, args.cpu_seconds) if is_op
                            else oracle_sample_position(inp, args.cpu_seconds) if is_pos
                            else oracle_sample_head(inp, args.cpu_seconds))
        cpu = {"value": rate, "unit": "entries/s" if is_op else "tokens/s", "cores": cpu_cores(),
               "kind": "oracle",
               "sample": (f"{toks // inp.n} whole heads" if is_chain or is_pos else
                          f"{toks // (inp.n * inp.n)} whole heads' W" if is_op else
                          f"{toks // (inp.B * inp.H)} seeded random rows of each of the "
                          f"{inp.B * inp.H} heads") + f" ({toks} {'entries' if is_op else 'tokens'}, {secs:.1f} s)"}

    if rank == 0:
        line = {"metric": ("chain tokens/s (B*H*n/s)" if is_chain else
                           "operator entries/s (B*H*n*n/s)" if is_op else
                           "position tokens/s (B*H*n/s)" if is_pos else "head tokens/s (B*H*n/s)"),
                "value": value, "unit": "entries/s" if is_op else "tokens/s", "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None,
                "dtype": "f32" if (is_chain or is_op) else "bf16" if is_pos else ("bf16" if inp.dtype == "bf16" else "f32->bf16"),
                "data": "synthetic (seeded, workloads.py)",
                "config": dict(config_of(args, inp, world), l2="flushed between timed steps"),
                "roofline": roof, "cpu_baseline": cpu, "e2e": e2e, "clocks": clk,
                "gpu_launches": launches_per_step * args.steps,
                "kernel_ms_per_step": kern}
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
