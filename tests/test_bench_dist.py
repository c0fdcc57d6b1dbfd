"""The multi-rank path of bench.py on CPU: world size 2 over gloo.

Heads are independent, so each rank runs its own full batch with no collective on the data
path; the only exchange is the max over ranks of the measured time. These tests run that
host logic (rendezvous on 127.0.0.1, barrier, max-reduction) without a GPU.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, q):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import bench
    r, w, local = bench.dist_env()
    bench.dist_init(w, "gloo")
    bench.dist_barrier(w)
    t = bench.dist_max(1.0 + rank, w, "cpu")  # each rank's "time"
    q.put((r, w, local, t))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_ranks_take_the_max_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert [g[0] for g in got] == [0, 1]
    assert all(g[1] == 2 for g in got)
    assert all(g[3] == 2.0 for g in got)  # the max over ranks, seen by both


def test_single_rank_is_identity():
    import bench
    assert bench.dist_max(3.5, 1, "cpu") == 3.5


def test_work_accounting_counts_structurally_live_entries():
    import numpy as np
    import bench
    u = np.array([0.0, 0.5, 0.0, 0.7, 0.9], dtype=np.float32)
    # g = 1: m = u; zero at k = 2 (k = 0 is never read): rows 0..4 see 1, 2, 1, 2, 3 entries
    assert bench.live_entries(u, 1.0) == 9.0
    assert bench.live_entries(u, 0.0) == 15.0  # g = 0: every gate is 1


def test_work_accounting_stops_at_fp32_underflow():
    import numpy as np
    import bench
    # m = 1/2 everywhere: R_ij = 2^-(i-j) is nonzero in fp32 down to 2^-149, so row i has
    # min(i, 149) + 1 live keys
    n = 400
    u = np.full(n, 0.5)
    want = sum(min(i, 149) + 1 for i in range(n))
    assert bench.live_entries(u, 1.0) == float(want)
    # brute force with fp32 products on random gates
    r = np.random.default_rng(3)
    u = r.uniform(0.3, 1.0, 300)
    m = np.clip(u, 0.0, 1.0).astype(np.float32)
    cnt = 0
    for i in range(300):
        R = np.float32(1.0)
        for j in range(i, -1, -1):
            if j < i:
                R = np.float32(R * m[j + 1])
            if R == 0:
                break
            cnt += 1
    # fp32 rounding in the subnormal range can keep a product at 2^-149 for a few more keys
    # than the exact product: the count is exact-arithmetic, so never above the fp32 one
    got = bench.live_entries(u, 1.0)
    assert got <= cnt and cnt - got <= 0.01 * cnt


def test_reference_arm_prints_one_contract_line():
    """`bench.py --impl reference` (the oracle timed on the host cores) prints exactly one JSON
    line with the keys the driver reads, for the head, position-only, gate-preparation and
    mixed-switch workloads (small sizes)."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    for wl in ("tiny", "position", "gate_prep", "mixed"):
        args = [sys.executable, os.path.join(root, "bench.py"), "--impl", "reference",
                "--workload", wl, "--steps", "1", "--warmup", "0", "--cpu-seconds", "0.2"]
        if wl in ("position", "gate_prep", "mixed"):
            args += ["--B", "1", "--H", "2", "--n", "512"]
        out = subprocess.run(args, capture_output=True, text=True, timeout=300, cwd=root)
        assert out.returncode == 0, out.stderr[-2000:]
        lines = [l for l in out.stdout.splitlines() if l.strip().startswith("{")]
        assert len(lines) == 1
        d = json.loads(lines[0])
        for k in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                  "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                  "cpu_baseline", "e2e"):
            assert k in d, k
        assert d["impl"] == "reference" and d["value"] > 0 and d["steps"] == 1
        assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
        assert d["e2e"]["value"] == d["value"] and d["e2e"]["h2d_bytes_per_step"] == 0
        assert d["config"]["workload"] == wl


def test_mixed_workload_dispatch_classes():
    """The mixed grid (head h takes point h mod 27 of beta x qk x g): of 64 heads, 22 have
    qk = 0 (O(n) readout), 14 have g = 0 and qk != 0 (the real fused kernel), 28 are gated."""
    import bench
    import workloads as W
    hi = W.mixed(B=1, H=64, n=256)
    c = bench.head_classes(hi)
    assert (c["chain_heads"], c["real_heads"], c["gated_heads"]) == (22, 14, 28)
    assert c["chain_tokens"] == 22 * 256
    causal = 256 * 257 / 2
    assert c["real_flops"] == 14 * causal * (2 * 128 + 2 * 128)
    assert 0 < c["gated_live"] <= c["gated_causal"] == 28 * causal
