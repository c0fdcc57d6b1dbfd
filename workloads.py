"""Seeded synthetic inputs for the resolvent-operator causal head.

This module holds no arithmetic of the method: it only draws numbers. The same buffers
feed the CUDA library and the fp64 oracle, so both sides always see identical values.

Generator (counter-based, so any slice can be drawn independently and in parallel):
  * splitmix64 (Steele, Lea, Flood, "Fast splittable pseudorandom number generators",
    OOPSLA 2014): state_i = base + (i+1) * 0x9E3779B97F4A7C15, output = mix(state_i);
    base = mix(seed * 256 + stream).
  * uniform in [0,1): the top 53 bits of the output times 2^-53.
  * normal: Box-Muller on the uniforms of counters 2i and 2i+1 (cosine branch).
Values are drawn in fp64, rounded to fp32, and then to bf16 (round to nearest even) where
a workload stores bf16. Seeds: 0x5EED0000 + workload index; streams q=1, k=2, v/b=3, u=4,
theta=5, positions=6, forced gate values=7, position-only logits=8.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
SEED_BASE = 0x5EED0000
STREAM = {"q": 1, "k": 2, "v": 3, "b": 3, "u": 4, "theta": 5, "pos": 6, "forced": 7, "a": 8}
_CHUNK = 1 << 22


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _base(seed: int, stream: int) -> np.uint64:
    with np.errstate(over="ignore"):
        return _mix(np.array([(seed * 256 + stream) & 0xFFFFFFFFFFFFFFFF], dtype=np.uint64))[0]


def _uniform_chunk(base, start, count):
    with np.errstate(over="ignore"):
        ctr = np.arange(start + 1, start + 1 + count, dtype=np.uint64)
        z = _mix(base + ctr * GAMMA)
    return (z >> np.uint64(11)).astype(np.float64) * (1.0 / 9007199254740992.0)


def _parallel(fn, total):
    starts = list(range(0, total, _CHUNK))
    if len(starts) <= 1:
        return fn(0, total)
    workers = min(len(starts), os.cpu_count() or 1)
    with ThreadPoolExecutor(workers) as ex:
        parts = list(ex.map(lambda s: fn(s, min(_CHUNK, total - s)), starts))
    return np.concatenate(parts)


def uniform(seed: int, stream: int, count: int, offset: int = 0) -> np.ndarray:
    """count uniforms in [0,1) from counters offset .. offset+count-1 (fp64)."""
    base = _base(seed, stream)
    return _parallel(lambda s, c: _uniform_chunk(base, offset + s, c), count)


def normal(seed: int, stream: int, count: int, offset: int = 0) -> np.ndarray:
    """count standard normals (fp64), Box-Muller on counter pairs (2i, 2i+1)."""
    base = _base(seed, stream)

    def chunk(s, c):
        u = _uniform_chunk(base, 2 * (offset + s), 2 * c)
        u1, u2 = u[0::2], u[1::2]
        return np.sqrt(-2.0 * np.log1p(-u1)) * np.cos(2.0 * math.pi * u2)

    return _parallel(chunk, count)


def to_bf16_values(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest even); returned as fp32 holding bf16 values."""
    f = np.ascontiguousarray(x, dtype=np.float32)
    b = f.view(np.uint32).astype(np.uint64)
    b = (b + np.uint64(0x7FFF) + ((b >> np.uint64(16)) & np.uint64(1))) & np.uint64(0xFFFF0000)
    return b.astype(np.uint32).view(np.float32).reshape(f.shape)


@dataclass
class HeadInputs:
    """One batch of head inputs: q, k [BH,n,d], v [BH,n,dv], u, theta [BH,n] (fp32 arrays
    holding the stored values) and per-head switches beta, qk, g [H]."""
    B: int
    H: int
    n: int
    d: int
    dv: int
    dtype: str
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    u: np.ndarray
    theta: np.ndarray
    beta: np.ndarray
    qk: np.ndarray
    g: np.ndarray
    name: str = ""
    extra: dict = field(default_factory=dict)

    def switches_bh(self):
        """Per-(batch, head) switch arrays [B*H] (head h of every batch shares row h)."""
        return (np.tile(self.beta, self.B), np.tile(self.qk, self.B), np.tile(self.g, self.B))


def _positions(seed, BH, n, frac_zero, frac_forced):
    """Per head: disjoint seeded sets of round(frac*n) positions (a seeded permutation)."""
    nz, nf = int(round(frac_zero * n)), int(round(frac_forced * n))
    zeros, forced = [], []
    for h in range(BH):
        keys = uniform(seed, STREAM["pos"], n, offset=h * n)
        perm = np.argsort(keys, kind="stable")
        zeros.append(perm[:nz])
        forced.append(perm[nz:nz + nf])
    return zeros, forced


def head_inputs(B, H, n, d, dv, *, seed, dtype="bf16", q_scale=1.0, u_range=(0.0, 1.0),
                theta_range=(-math.pi, math.pi), zero_frac=0.0, beta=1.0, qk=1.0, g=0.0,
                name="") -> HeadInputs:
    """Generic seeded head inputs: q = q_scale * N(0,1), k, v ~ N(0,1), u ~ U(u_range),
    theta ~ U(theta_range), round(zero_frac*n) positions of u per head set exactly to 0."""
    BH = B * H
    rnd = (lambda x: to_bf16_values(x)) if dtype == "bf16" else (lambda x: x.astype(np.float32))
    q = rnd((normal(seed, STREAM["q"], BH * n * d) * q_scale).astype(np.float32)).reshape(BH, n, d)
    k = rnd(normal(seed, STREAM["k"], BH * n * d).astype(np.float32)).reshape(BH, n, d)
    v = rnd(normal(seed, STREAM["v"], BH * n * dv).astype(np.float32)).reshape(BH, n, dv)
    lo, hi = u_range
    u = (lo + (hi - lo) * uniform(seed, STREAM["u"], BH * n)).astype(np.float32).reshape(BH, n)
    tlo, thi = theta_range
    theta = (tlo + (thi - tlo) * uniform(seed, STREAM["theta"], BH * n)).astype(
        np.float32).reshape(BH, n)
    if zero_frac > 0:
        zeros, _ = _positions(seed, BH, n, zero_frac, 0.0)
        for h in range(BH):
            u[h, zeros[h]] = 0.0

    def per_head(x):
        x = np.asarray(x, dtype=np.float64).reshape(-1)
        return np.full(H, x[0]) if x.size == 1 else x.copy()

    return HeadInputs(B, H, n, d, dv, dtype, q, k, v, u, theta, per_head(beta), per_head(qk),
                      per_head(g), name)


# ------------------------------------------------------------------ the five workloads

def tiny(switch_index: int = 0) -> HeadInputs:
    """Tiny oracle case: B=1 H=1 n=64 d=dv=16 fp32; q,k,v ~ N(0,1); u ~ U(0,1) with 10%
    (6 positions) exactly 0; theta ~ U(-pi,pi); switches (1,1,0), (0,1,0), (0,0,1),
    (0.5,0.7,0.3) by index."""
    sw = [(1.0, 1.0, 0.0), (0.0, 1.0, 0.0), (0.0, 0.0, 1.0), (0.5, 0.7, 0.3)][switch_index]
    return head_inputs(1, 1, 64, 16, 16, seed=SEED_BASE + 0, dtype="fp32", zero_frac=0.1,
                       beta=sw[0], qk=sw[1], g=sw[2], name=f"tiny n64 d16 {sw}")


def gated_softmax(B=8, H=16, n=2048) -> HeadInputs:
    """Gated softmax head: B=8 H=16 n=2048 d=dv=64 bf16; q = N(0,1)/sqrt(64), k, v ~ N(0,1);
    u ~ U(0.9,1); theta ~ U(-0.1,0.1); (beta,qk,g) = (1,1,0.5)."""
    return head_inputs(B, H, n, 64, 64, seed=SEED_BASE + 1, q_scale=1.0 / 8.0,
                       u_range=(0.9, 1.0), theta_range=(-0.1, 0.1), beta=1.0, qk=1.0, g=0.5,
                       name=f"gated softmax B{B} H{H} n{n} d64")


def long_softmax(B=4, H=32, n=8192) -> HeadInputs:
    """Long softmax corner: B=4 H=32 n=8192 d=dv=128 bf16; q,k,v ~ N(0,1); u ~ U(0,1),
    theta ~ U(-pi,pi) (ignored at g = 0); (beta,qk,g) = (1,1,0)."""
    return head_inputs(B, H, n, 128, 128, seed=SEED_BASE + 2, beta=1.0, qk=1.0, g=0.0,
                       name=f"long softmax B{B} H{H} n{n} d128")


def mixed(B=1, H=64, n=32768) -> HeadInputs:
    """Mixed-switch heads: B=1 H=64 n=32768 d=dv=128 bf16; q,k,v ~ N(0,1); u ~ U(-0.5,1.5);
    theta ~ U(-pi,pi); head h takes grid point h mod 27 = 9*ib + 3*iqk + ig of
    beta in {0,0.5,1}, qk in {0,0.5,1}, g in {0,0.3,1}."""
    grid = [0.0, 0.5, 1.0], [0.0, 0.5, 1.0], [0.0, 0.3, 1.0]
    pts = [(grid[0][(h % 27) // 9], grid[1][(h % 9) // 3], grid[2][h % 3]) for h in range(H)]
    return head_inputs(B, H, n, 128, 128, seed=SEED_BASE + 4, u_range=(-0.5, 1.5),
                       beta=[p[0] for p in pts], qk=[p[1] for p in pts], g=[p[2] for p in pts],
                       name=f"mixed B{B} H{H} n{n} d128")


@dataclass
class ChainInputs:
    """Chain inputs: b [BH,n,dv] fp32, u, theta [BH,n], switches per head [H]."""
    B: int
    H: int
    n: int
    dv: int
    b: np.ndarray
    u: np.ndarray
    theta: np.ndarray
    beta: np.ndarray
    qk: np.ndarray
    g: np.ndarray
    name: str = ""

    def switches_bh(self):
        return (np.tile(self.beta, self.B), np.tile(self.qk, self.B), np.tile(self.g, self.B))


def chain(B=2, H=16, n=65536, dv=64) -> ChainInputs:
    """Path-product corner chain: b ~ N(0,1) fp32 with b_0 = 0; u ~ U(0.95,1) with 1% exact
    zeros and 5% of gates forced to -1/0/+1 ((u,theta) = (1,pi), (0,0), (1,0), uniformly);
    heads h < H/2 take the constant phase 0.01, the rest theta ~ U(-pi,pi);
    (beta,qk,g) = (0,0,1)."""
    seed = SEED_BASE + 3
    BH = B * H
    b = normal(seed, STREAM["b"], BH * n * dv).astype(np.float32).reshape(BH, n, dv)
    b[:, 0, :] = 0.0
    u = (0.95 + 0.05 * uniform(seed, STREAM["u"], BH * n)).astype(np.float32).reshape(BH, n)
    theta = (-math.pi + 2 * math.pi * uniform(seed, STREAM["theta"], BH * n)).astype(
        np.float32).reshape(BH, n)
    for bh in range(BH):
        if (bh % H) < H // 2:
            theta[bh, :] = np.float32(0.01)
    zeros, forced = _positions(seed, BH, n, 0.01, 0.05)
    forced_u = np.array([1.0, 0.0, 1.0], dtype=np.float32)
    forced_t = np.array([math.pi, 0.0, 0.0], dtype=np.float32)
    for bh in range(BH):
        u[bh, zeros[bh]] = 0.0
        pick = np.minimum((uniform(seed, STREAM["forced"], forced[bh].size, offset=bh * n)
                           * 3).astype(np.int64), 2)
        u[bh, forced[bh]] = forced_u[pick]
        theta[bh, forced[bh]] = forced_t[pick]
    return ChainInputs(B, H, n, dv, b, u, theta, np.zeros(H), np.zeros(H), np.ones(H),
                       f"chain B{B} H{H} n{n} dv{dv}")


def operator_heads(B=1, H=8, n=4096) -> HeadInputs:
    """Materialised operator W of gated softmax heads (the gated-softmax inputs at n = 4096):
    B=1 H=8 n=4096 d=64 bf16; q = N(0,1)/8; u ~ U(0.9,1); theta ~ U(-0.1,0.1); (1,1,0.5)."""
    return head_inputs(B, H, n, 64, 8, seed=SEED_BASE + 5, q_scale=1.0 / 8.0,
                       u_range=(0.9, 1.0), theta_range=(-0.1, 0.1), beta=1.0, qk=1.0, g=0.5,
                       name=f"operator B{B} H{H} n{n} d64")


@dataclass
class PositionInputs:
    """Position-only heads: a [H,n] logit per offset d = i - j (row h serves head h of every
    batch), v [BH,n,dv] (fp32 arrays holding the stored values), switches beta, qk [H]."""
    B: int
    H: int
    n: int
    dv: int
    dtype: str
    a: np.ndarray
    v: np.ndarray
    beta: np.ndarray
    qk: np.ndarray
    name: str = ""

    def switches_bh(self):
        return (np.tile(self.beta, self.B), np.tile(self.qk, self.B))


def position_inputs(B, H, n, dv, *, seed, dtype="bf16", noise=0.5, slope_scale=1.0, beta=1.0,
                    qk=1.0, name="") -> PositionInputs:
    """a_h(d) = -s_h d + noise * N(0,1) with geometric slopes s_h = slope_scale * 2^{-8(h+1)/H}
    (one per head, steep to gentle); v ~ N(0,1)."""
    BH = B * H
    rnd = (lambda x: to_bf16_values(x)) if dtype == "bf16" else (lambda x: x.astype(np.float32))
    d = np.arange(n, dtype=np.float64)
    slopes = slope_scale * 2.0 ** (-8.0 * (np.arange(H) + 1) / H)
    a = (-slopes[:, None] * d[None, :] + noise * normal(seed, STREAM["a"], H * n).reshape(H, n))
    v = rnd(normal(seed, STREAM["v"], BH * n * dv).astype(np.float32)).reshape(BH, n, dv)

    def per_head(x):
        x = np.asarray(x, dtype=np.float64).reshape(-1)
        return np.full(H, x[0]) if x.size == 1 else x.copy()

    return PositionInputs(B, H, n, dv, dtype, a.astype(np.float32), v, per_head(beta),
                          per_head(qk), name)


def position(B=4, H=32, n=8192) -> PositionInputs:
    """Position-only heads at the long-softmax shape: B=4 H=32 n=8192 dv=128 bf16 v ~ N(0,1);
    a_h(d) = -2^{-8(h+1)/32} d + 0.5 N(0,1); (beta, qk) = (1, 1)."""
    return position_inputs(B, H, n, 128, seed=SEED_BASE + 6, name=f"position B{B} H{H} n{n} dv128")


@dataclass
class GateInputs:
    """Gate-preparation inputs: u, theta [BH,n] fp32 and per-head g [H]."""
    B: int
    H: int
    n: int
    u: np.ndarray
    theta: np.ndarray
    g: np.ndarray
    name: str = ""

    def switches_bh(self):
        return (np.zeros(self.B * self.H), np.zeros(self.B * self.H), np.tile(self.g, self.B))


def gate_prep(B=1, H=64, n=32768) -> GateInputs:
    """Gate preparation alone at the mixed-switch shape: the mixed workload's u ~ U(-0.5,1.5),
    theta ~ U(-pi,pi) (same seed and streams) and its per-head g from the grid."""
    seed = SEED_BASE + 4
    BH = B * H
    u = (-0.5 + 2.0 * uniform(seed, STREAM["u"], BH * n)).astype(np.float32).reshape(BH, n)
    theta = (-math.pi + 2 * math.pi * uniform(seed, STREAM["theta"], BH * n)).astype(
        np.float32).reshape(BH, n)
    grid_g = [0.0, 0.3, 1.0]
    g = np.array([grid_g[h % 3] for h in range(H)], dtype=np.float64)
    return GateInputs(B, H, n, u, theta, g, f"gate prep B{B} H{H} n{n}")


WORKLOADS = {
    "tiny": tiny,
    "gated_softmax": gated_softmax,
    "long_softmax": long_softmax,
    "chain": chain,
    "mixed": mixed,
    "operator": operator_heads,
    "position": position,
    "gate_prep": gate_prep,
}
