#!/usr/bin/env python3
"""Benchmark of the resolvent-operator causal head on GB300.

A step is one call of the hot path on one batch of seeded synthetic inputs already resident
in HBM: resolvent_head_forward (gate preparation, the fused head kernel for heads with
qk != 0, the O(n) readout for heads with qk = 0) for the head workloads, resolvent_chain_scan
for the chain, resolvent_operator, resolvent_position_head, resolvent_gate_prep. The
default workload is the largest single-GPU configuration, the mixed-switch heads (B=1 H=64
n=32768 d=dv=128 bf16, every dispatch class: gated and g = 0 heads on the fused kernel, qk = 0
heads on the O(n) readout).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

Prints one JSON line (rank 0): the throughput, the roofline of the dominant kernel, per-class
figures (mixed heads), the fp64 oracle on the host cores (cpu_baseline), the same metric end
to end from pinned host memory through the overlapped host pipeline (e2e), and the SM clocks
sampled during the timed region. `--impl reference` times the fp64 CPU oracle instead, on the
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
    p.add_argument("--workload", default="mixed", choices=sorted(W.WORKLOADS))
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
    c = head_classes(hi)
    return c["gated_flops"] + c["real_flops"], c["chain_tokens"]


def head_classes(hi: W.HeadInputs):
    """Per dispatch class of a head workload: the fused kernel's gated heads (g != 0) and real
    heads (g = 0) with their algorithmic flops and entry counts, and the qk = 0 heads that run
    as O(n) readouts."""
    beta, qk, g = hi.switches_bh()
    out = {"gated_heads": 0, "gated_flops": 0.0, "gated_live": 0.0, "gated_causal": 0.0,
           "real_heads": 0, "real_flops": 0.0, "chain_heads": 0, "chain_tokens": 0}
    causal = hi.n * (hi.n + 1) / 2
    for h in range(hi.B * hi.H):
        if qk[h] == 0.0:
            out["chain_heads"] += 1
            out["chain_tokens"] += hi.n
        elif g[h] != 0.0:
            live = live_entries(hi.u[h], g[h])
            out["gated_heads"] += 1
            out["gated_live"] += live
            out["gated_causal"] += causal
            out["gated_flops"] += live * (2 * hi.d + 4 * hi.dv)
        else:
            out["real_heads"] += 1
            out["real_flops"] += causal * (2 * hi.d + 2 * hi.dv)
    return out


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

class NvmlClocks:
    """SM clock, throttle reasons and power sampled every ~2 ms from NVML (read only) in a
    thread, so that the timed region itself is covered."""
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, device):
        import ctypes
        import threading
        import torch
        self.ct = ctypes
        L = ctypes.CDLL("libnvidia-ml.so.1")
        if L.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        h = ctypes.c_void_p()
        ok = False
        try:
            uuid = str(torch.cuda.get_device_properties(device).uuid)
            uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
            ok = L.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(h)) == 0
        except Exception:
            ok = False
        if not ok:
            cnt = ctypes.c_uint(0)
            L.nvmlDeviceGetCount_v2(ctypes.byref(cnt))
            idx = 0 if cnt.value == 1 else torch.device(device).index or 0
            if L.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(idx), ctypes.byref(h)) != 0:
                raise OSError("no NVML handle")
        self.L, self.h = L, h
        self.reasons_fn = getattr(L, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            L.nvmlDeviceGetCurrentClocksThrottleReasons
        mx = ctypes.c_uint(0)
        L.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx))  # NVML_CLOCK_SM
        self.max_mhz = float(mx.value)
        self.samples = []
        self.stop_flag = threading.Event()
        self.thread = threading.Thread(target=self._run, daemon=True)

    def _sample(self):
        ct = self.ct
        clk, rs, pw = ct.c_uint(0), ct.c_ulonglong(0), ct.c_uint(0)
        self.L.nvmlDeviceGetClockInfo(self.h, 1, ct.byref(clk))
        self.reasons_fn(self.h, ct.byref(rs))
        self.L.nvmlDeviceGetPowerUsage(self.h, ct.byref(pw))
        self.samples.append((time.perf_counter(), float(clk.value), int(rs.value), pw.value / 1e3))

    def _run(self):
        while not self.stop_flag.is_set():
            self._sample()
            time.sleep(0.002)

    def start(self):
        self.thread.start()

    def stop(self, t0, t1):
        self.stop_flag.set()
        self.thread.join(timeout=5)
        inside = [x for x in self.samples if t0 <= x[0] <= t1]
        use = inside if inside else self.samples
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": ["no samples"]}
        bits = 0
        for x in use:
            bits |= x[2]
        return {"sm_mhz": statistics.median(x[1] for x in use), "sm_max_mhz": self.max_mhz,
                "reasons": sorted(v for b, v in self.REASONS.items() if bits & b),
                "power_w_max": max(x[3] for x in use), "samples": len(use),
                "samples_in_timed_region": len(inside), "source": "nvml, every ~2 ms"}


class SmiClocks:
    """Fallback: nvidia-smi sampling every 100 ms (too coarse for short timed regions)."""
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
                "reasons": reasons, "samples": len(use), "samples_in_timed_region": len(inside),
                "source": "nvidia-smi, every 100 ms"}


def make_clocks(device, local):
    try:
        return NvmlClocks(device)
    except Exception:
        return SmiClocks(local)


KERNEL_SOURCES = {"head_fwd_kernel": ["head_fwd.cu", "head_common.cuh", "common.cuh", "gate_products.cuh"],
                  "chain_scan_kernel": ["chain_scan.cu", "common.cuh"],
                  "operator_kernel": ["operator.cu", "head_common.cuh", "common.cuh", "gate_products.cuh"],
                  "position_head_kernel": ["position.cu", "head_common.cuh", "common.cuh", "gate_products.cuh"],
                  "gate_prep_kernel": ["gate_prep.cu", "gate_products.cuh", "common.cuh"]}


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


def oracle_sample_gate(gi: W.GateInputs, target_s: float):
    """The oracle's gate preparation (blend, gate, block products) of whole heads."""
    import oracle
    oracle.build()
    g = np.asarray(gi.switches_bh()[2], np.float32).astype(np.float64)
    heads, t0 = 0, time.perf_counter()
    while heads < gi.B * gi.H and (heads == 0 or time.perf_counter() - t0 < target_s):
        oracle.gate_prep(gi.u[heads:heads + 1], gi.theta[heads:heads + 1], g[heads:heads + 1])
        heads += 1
    dt = time.perf_counter() - t0
    return heads * gi.n / dt, heads * gi.n, dt


def cpu_cores():
    import oracle
    oracle.build()
    return oracle.max_threads()


def kind_of(inp, workload):
    if isinstance(inp, W.ChainInputs):
        return "chain"
    if isinstance(inp, W.PositionInputs):
        return "position"
    if isinstance(inp, W.GateInputs):
        return "gate_prep"
    return "operator" if workload == "operator" else "head"


METRICS = {"chain": ("chain tokens/s (B*H*n/s)", "tokens/s"),
           "position": ("position tokens/s (B*H*n/s)", "tokens/s"),
           "gate_prep": ("gate-prep tokens/s (B*H*n/s)", "tokens/s"),
           "operator": ("operator entries/s (B*H*n*n/s)", "entries/s"),
           "head": ("head tokens/s (B*H*n/s)", "tokens/s")}


def config_of(args, inp, world):
    if isinstance(inp, W.ChainInputs):
        cfg = {"workload": args.workload, "B": inp.B, "H": inp.H, "n": inp.n, "dv": inp.dv,
               "dtype_b": "fp32", "switches": "(0,0,1)"}
    elif isinstance(inp, W.PositionInputs):
        sw = sorted({(float(b), float(q)) for b, q in zip(inp.beta, inp.qk)})
        cfg = {"workload": args.workload, "B": inp.B, "H": inp.H, "n": inp.n, "dv": inp.dv,
               "dtype_v": inp.dtype, "logits": "a_h(d) = -2^(-8(h+1)/H) d + 0.5 N(0,1)",
               "switches (beta, qk; g = 0)": sw[0] if len(sw) == 1 else f"{len(sw)} per-head settings"}
    elif isinstance(inp, W.GateInputs):
        cfg = {"workload": args.workload, "B": inp.B, "H": inp.H, "n": inp.n,
               "inputs": "u ~ U(-0.5,1.5), theta ~ U(-pi,pi) fp32", "g": "per head, grid {0, 0.3, 1}",
               "outputs": "m, theta', gate, prefix, suffix, block carries"}
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
    kind = kind_of(inp, args.workload)
    is_op = kind == "operator"
    sample = {"chain": lambda: oracle_sample_chain(inp, per_step),
              "position": lambda: oracle_sample_position(inp, per_step),
              "operator": lambda: oracle_sample_operator(inp, per_step),
              "gate_prep": lambda: oracle_sample_gate(inp, per_step),
              "head": lambda: oracle_sample_head(inp, per_step, seed=7)}[kind]
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
    metric, unit = METRICS[kind]
    line = {"impl": "reference", "metric": metric,
            "value": value, "unit": unit, "n_gpus": 0, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * secs / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded, workloads.py)", "config": config_of(args, inp, 1),
            "cpu_baseline": {"value": value, "unit": unit, "cores": cores, "kind": "oracle",
                             "sample": {"chain": "whole heads of the chain",
                                        "operator": "whole heads' W",
                                        "position": "whole position-only heads",
                                        "gate_prep": "whole heads' gate preparation",
                                        "head": "seeded random rows of every head"}[kind] +
                             f", {toks} {'entries' if is_op else 'tokens'} in {secs:.1f} s"},
            "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ our arm

def setup_workload(args, inp, device, R):
    """The device-resident step, its work accounting and its end-to-end description."""
    import torch
    kind = kind_of(inp, args.workload)
    shp = (inp.B, inp.H, inp.n)
    tdev = lambda x, s, dt=torch.float32: torch.from_numpy(np.ascontiguousarray(x).reshape(s)).to(
        device=device, dtype=dt)
    status = R.new_status(device)
    w = {"kind": kind, "status": status}
    if kind == "chain":
        u, th = tdev(inp.u, shp), tdev(inp.theta, shp)
        b = tdev(inp.b, (*shp, inp.dv))
        ws = torch.empty(max(1, R.chain_workspace_bytes(*shp, inp.dv)), dtype=torch.uint8, device=device)

        def call(di, do, stream=None):
            R.chain_scan(di[0], di[1], inp.g, di[2], out=(do[0], do[1]), workspace=ws, status=status,
                         stream=stream, sync=False)
        dev_in = [u, th, b]
        dev_out = [torch.empty_like(b), torch.empty_like(b)]
        host_in = [(inp.u, shp, torch.float32), (inp.theta, shp, torch.float32),
                   (inp.b, (*shp, inp.dv), torch.float32)]
        w.update(tokens=inp.B * inp.H * inp.n, main=[R.PROF_CHAIN], bound="hbm",
                 kname="chain_scan_kernel", dtype="f32",
                 work=inp.B * inp.H * inp.n * chain_bytes_per_token(inp.dv))
    elif kind == "operator":
        q, k = tdev(inp.q, (*shp, inp.d), torch.bfloat16), tdev(inp.k, (*shp, inp.d), torch.bfloat16)
        u, th = tdev(inp.u, shp), tdev(inp.theta, shp)
        ws = torch.empty(max(1, R.operator_workspace_bytes(*shp, inp.d, torch.bfloat16)),
                         dtype=torch.uint8, device=device)

        def call(di, do, stream=None):
            R.operator(di[0], di[1], di[2], di[3], inp.beta, inp.qk, inp.g, out=(do[0], do[1]),
                       workspace=ws, status=status, stream=stream, sync=False)
        dev_in = [q, k, u, th]
        dev_out = [torch.empty(*shp, inp.n, device=device), torch.empty(*shp, inp.n, device=device)]
        host_in = [(inp.q, (*shp, inp.d), torch.bfloat16), (inp.k, (*shp, inp.d), torch.bfloat16),
                   (inp.u, shp, torch.float32), (inp.theta, shp, torch.float32)]
        entries = inp.B * inp.H * inp.n * inp.n
        # bytes: W written (8 B per entry); q, k read (2 B x d each per token); u, theta
        w.update(tokens=entries, main=[R.PROF_OPERATOR], bound="hbm", kname="operator_kernel",
                 dtype="f32", work=entries * 8 + inp.B * inp.H * inp.n * (4 * inp.d + 8))
    elif kind == "position":
        a = tdev(inp.a, (inp.H, inp.n))
        v = tdev(inp.v, (*shp, inp.dv), torch.bfloat16)
        ws = torch.empty(max(1, R.position_workspace_bytes(*shp, inp.dv, torch.bfloat16)),
                         dtype=torch.uint8, device=device)

        def call(di, do, stream=None):
            R.position_head(di[0], di[1], inp.beta, inp.qk, out=do[0], workspace=ws, status=status,
                            stream=stream, sync=False)
        dev_in = [a, v]
        dev_out = [torch.empty(*shp, inp.dv, device=device)]
        host_in = [(inp.a, (inp.H, inp.n), torch.float32), (inp.v, (*shp, inp.dv), torch.bfloat16)]
        w.update(tokens=inp.B * inp.H * inp.n, main=[R.PROF_POSITION], bound="tensor",
                 kname="position_head_kernel", dtype="bf16", work=position_work(inp))
    elif kind == "gate_prep":
        u, th = tdev(inp.u, shp), tdev(inp.theta, shp)
        outs = R.gate_prep_outputs(*shp, device)
        names = ["m", "theta_p", "gate", "prefix", "suffix", "carry"]

        def call(di, do, stream=None):
            R.gate_prep(di[0], di[1], inp.g, out=dict(zip(names, do)), status=status, stream=stream,
                        sync=False)
        dev_in = [u, th]
        dev_out = [outs[k] for k in names]
        host_in = [(inp.u, shp, torch.float32), (inp.theta, shp, torch.float32)]
        nb = (inp.n + 127) // 128
        tokens = inp.B * inp.H * inp.n
        # u, theta read; m, theta' (4 B each) and gate, prefix, suffix (8 B each) written; carries
        w.update(tokens=tokens, main=[R.PROF_GATE_PREP], bound="hbm", kname="gate_prep_kernel",
                 dtype="f32", work=tokens * (8 + 32) + inp.B * inp.H * nb * 8)
    else:
        dt = torch.bfloat16 if inp.dtype == "bf16" else torch.float32
        q, k = tdev(inp.q, (*shp, inp.d), dt), tdev(inp.k, (*shp, inp.d), dt)
        v = tdev(inp.v, (*shp, inp.dv), dt)
        u, th = tdev(inp.u, shp), tdev(inp.theta, shp)
        ws = torch.empty(max(1, R.head_workspace_bytes(*shp, inp.d, inp.dv, dt)), dtype=torch.uint8,
                         device=device)

        def call(di, do, stream=None):
            R.head_forward(di[0], di[1], di[2], di[3], di[4], inp.beta, inp.qk, inp.g,
                           out=(do[0], do[1]), workspace=ws, status=status, stream=stream, sync=False)
        dev_in = [q, k, u, th, v]
        dev_out = [torch.empty(*shp, inp.dv, device=device), torch.empty(*shp, inp.dv, device=device)]
        host_in = [(inp.q, (*shp, inp.d), dt), (inp.k, (*shp, inp.d), dt), (inp.u, shp, torch.float32),
                   (inp.theta, shp, torch.float32), (inp.v, (*shp, inp.dv), dt)]
        cls = head_classes(inp)
        w.update(tokens=inp.B * inp.H * inp.n, main=[R.PROF_HEAD_GATED, R.PROF_HEAD_REAL],
                 bound="tensor", kname="head_fwd_kernel",
                 dtype="bf16" if inp.dtype == "bf16" else "f32->bf16",
                 work=cls["gated_flops"] + cls["real_flops"], classes=cls)
    w.update(call=call, dev_in=dev_in, dev_out=dev_out, host_in=host_in,
             step=lambda: call(dev_in, dev_out))
    return w


def class_figures(w, inp, per_kind_ms, pk):
    """Per dispatch class of a head workload: time per step, throughput and roofline fraction
    of the gated and real fused-kernel launches and of the O(n) readout of qk = 0 heads."""
    import gated_causal_attention_gb300 as R
    c = w.get("classes")
    if not c:
        return None
    out = {}
    t = per_kind_ms.get(R.PROF_HEAD_GATED, 0.0)
    if c["gated_heads"]:
        tf = c["gated_flops"] / (t / 1e3) / 1e12 if t > 0 else None
        out["k2_gated"] = {"heads": c["gated_heads"], "ms": t, "tflops": tf,
                           "frac": tf / pk["bf16_tflops"] if tf else None,
                           "skip_fraction": 1.0 - c["gated_live"] / c["gated_causal"]}
    t = per_kind_ms.get(R.PROF_HEAD_REAL, 0.0)
    if c["real_heads"]:
        tf = c["real_flops"] / (t / 1e3) / 1e12 if t > 0 else None
        out["k2_real"] = {"heads": c["real_heads"], "ms": t, "tflops": tf,
                          "frac": tf / pk["bf16_tflops"] if tf else None}
    t = per_kind_ms.get(R.PROF_READOUT, 0.0)
    if c["chain_heads"]:
        vb = 2 if inp.dtype == "bf16" else 4
        byt = c["chain_tokens"] * (vb * inp.dv + 8 + 8 * inp.dv)
        gbs = byt / (t / 1e3) / 1e9 if t > 0 else None
        out["qk0_readout"] = {"heads": c["chain_heads"], "ms": t, "gbs": gbs,
                              "frac": gbs / pk["hbm_gbs"] if gbs else None,
                              "bytes_per_token": vb * inp.dv + 8 + 8 * inp.dv}
    return out


def run_e2e(args, w, device, world, R):
    """The same metric end to end: every step uploads its inputs from pinned host memory, runs
    the call and reads its outputs back to pinned host memory, through the overlapped host
    pipeline (uploads, calls and downloads on three streams, double-buffered device memory)."""
    import torch
    from gated_causal_attention_gb300.pipeline import HostPipeline
    pinned = [torch.from_numpy(np.ascontiguousarray(x).reshape(s)).to(dt).pin_memory()
              for x, s, dt in w["host_in"]]
    specs_in = [(tuple(p.shape), p.dtype) for p in pinned]
    specs_out = [(tuple(o.shape), o.dtype) for o in w["dev_out"]]
    pipe = HostPipeline(lambda di, do, st: w["call"](di, do, st), specs_in, specs_out, device=device)
    host_out = [[torch.empty(s, dtype=dt).pin_memory() for s, dt in specs_out] for _ in range(2)]
    h2d = sum(p.numel() * p.element_size() for p in pinned)
    d2h = sum(o.numel() * o.element_size() for o in host_out[0])
    for i in range(3):
        pipe.submit(pinned, host_out[i % 2])
    pipe.synchronize()
    dist_barrier(world)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(pipe.up[0])
    for s in pipe.up[1:] + pipe.down + [pipe.comp]:
        s.wait_event(e0)  # every stream of the timed steps starts after e0
    for i in range(args.steps):
        pipe.submit(pinned, host_out[i % 2])
    for s in pipe.down[1:] + pipe.up + [pipe.comp]:
        pipe.down[0].wait_stream(s)
    e1.record(pipe.down[0])
    pipe.synchronize()
    e_ms = dist_max(e0.elapsed_time(e1) / args.steps, world, device)
    R.status_sync(w["status"])
    unit = METRICS[w["kind"]][1]
    return {"value": w["tokens"] * world / (e_ms / 1e3), "unit": unit, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": e_ms,
            "how": "pinned host buffers; uploads, calls and downloads overlapped on three streams"}


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
    w = setup_workload(args, inp, device, R)
    step = w["step"]

    # warm-up, and a refusal check of the inputs
    for _ in range(args.warmup):
        step()
    R.status_sync(w["status"])
    launches_per_step = R.last_launch_count()
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=device)

    clocks = make_clocks(device, local)
    clocks.start()
    time.sleep(0.05)
    R.profile_enable(True)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    dist_barrier(world)
    torch.cuda.synchronize()
    w0 = time.perf_counter() if isinstance(clocks, NvmlClocks) else time.time()
    for i in range(args.steps):
        flush.zero_()  # L2 flush between timed iterations (outside the step's events)
        ev[i][0].record()
        step()
        ev[i][1].record()
    torch.cuda.synchronize()
    w1 = time.perf_counter() if isinstance(clocks, NvmlClocks) else time.time()
    dist_barrier(world)
    pairs = R.profile_collect(kinds=True)
    R.profile_enable(False)
    R.status_sync(w["status"])
    clk = clocks.stop(w0, w1)
    step_ms = [a.elapsed_time(b) for a, b in ev]
    ms_local = sum(step_ms) / len(step_ms)
    ms = dist_max(ms_local, world, device)
    value = w["tokens"] * world / (ms / 1e3)

    per_kind = {}
    for t, kd in pairs:
        per_kind[kd] = per_kind.get(kd, 0.0) + t / args.steps
    kern = sum(per_kind.get(kd, 0.0) for kd in w["main"]) or float("nan")
    pk, pk_kind = peaks()
    if w["bound"] == "hbm":
        achieved = w["work"] / (kern / 1e3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / pk["hbm_gbs"], "algorithmic_bytes_per_launch": w["work"]}
    else:
        achieved = w["work"] / (kern / 1e3) / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                "frac": achieved / pk["bf16_tflops"], "algorithmic_flops_per_launch": w["work"]}
    roof.update(traffic=measured_traffic(w["kname"], args.workload), kernel=w["kname"],
                kernel_ms=kern, peak_kind=pk_kind + (" burst" if w["bound"] == "tensor" else " copy"))
    classes = class_figures(w, inp, per_kind, pk)

    e2e = None if args.no_e2e else run_e2e(args, w, device, world, R)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        kind = w["kind"]
        rate, toks, secs = {"chain": lambda: oracle_sample_chain(inp, args.cpu_seconds),
                            "operator": lambda: oracle_sample_operator(inp, args.cpu_seconds),
                            "position": lambda: oracle_sample_position(inp, args.cpu_seconds),
                            "gate_prep": lambda: oracle_sample_gate(inp, args.cpu_seconds),
                            "head": lambda: oracle_sample_head(inp, args.cpu_seconds)}[kind]()
        sample = {"chain": f"{toks // inp.n} whole heads", "position": f"{toks // inp.n} whole heads",
                  "gate_prep": f"{toks // inp.n} whole heads",
                  "operator": f"{toks // (inp.n * inp.n)} whole heads' W",
                  "head": f"{toks // (inp.B * inp.H)} seeded random rows of each of the {inp.B * inp.H} heads"}[kind]
        cpu = {"value": rate, "unit": METRICS[kind][1], "cores": cpu_cores(), "kind": "oracle",
               "sample": sample + f" ({toks} {'entries' if kind == 'operator' else 'tokens'}, {secs:.1f} s)"}

    if rank == 0:
        metric, unit = METRICS[w["kind"]]
        line = {"metric": metric, "value": value, "unit": unit, "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": w["dtype"],
                "data": "synthetic (seeded, workloads.py)",
                "config": dict(config_of(args, inp, world), l2="flushed between timed steps"),
                "roofline": roof, "classes": classes, "cpu_baseline": cpu, "e2e": e2e, "clocks": clk,
                "gpu_launches": launches_per_step * args.steps,
                "kernel_ms_per_step": {str(k): v for k, v in sorted(per_kind.items())}}
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
