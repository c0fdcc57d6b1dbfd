"""GPU edge cases of the head and the operator, through the C ABI, against the fp64 oracle:
the pages' large-logit and overflow rows, the lazy rescale of the running maximum, the zero
pattern of G as the fused head kernel itself produces it, and the bounded waits of the head
and operator kernels.

Citations: "Resolvent Operator" (teerth.dev/Aether-Lang/integrated/resolvent/), its "Test
evidence" table (`logits_of_ten_thousand_stay_finite_at_beta_one`,
`an_overflowing_logit_never_becomes_nan`, `a_closed_gate_annihilates_every_path_through_it_exactly`),
its section "Evaluation and refusals" (the log-domain normaliser, the overflow row away from
beta = 1) and its Lean table (`pathProd_eq_zero_iff`).
"""
import math

import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu

O_TOL = 1e-2   # bf16 tensor-core contractions: max-abs 1e-2 * max|O|
W_TOL = 1e-3   # the operator: logits from the tensor cores, the rest fp32


@pytest.fixture(scope="module")
def R():
    import __graft_entry__
    __graft_entry__.build()
    import gated_causal_attention_gb300 as R
    assert torch.cuda.is_available(), "the GPU tests need a CUDA device"
    return R


def dev(x, dtype=torch.float32):
    return torch.from_numpy(np.ascontiguousarray(x)).to(dtype).cuda()


def f32(xs):
    return np.asarray(xs, dtype=np.float32).astype(np.float64)


def run_head(R, hi):
    dt = torch.bfloat16 if hi.dtype == "bf16" else torch.float32
    shp = (hi.B, hi.H, hi.n)
    Ore, Oim = R.head_forward(dev(hi.q.reshape(*shp, hi.d), dt), dev(hi.k.reshape(*shp, hi.d), dt),
                              dev(hi.u.reshape(shp)), dev(hi.theta.reshape(shp)),
                              dev(hi.v.reshape(*shp, hi.dv), dt), hi.beta, hi.qk, hi.g)
    torch.cuda.synchronize()
    return (Ore.cpu().double().numpy().reshape(hi.B * hi.H, hi.n, hi.dv),
            Oim.cpu().double().numpy().reshape(hi.B * hi.H, hi.n, hi.dv))


def oracle_head(oracle_mod, hi):
    beta, qk, g = [f32(x) for x in hi.switches_bh()]
    O, st = oracle_mod.head_rows(hi.q, hi.k, hi.u, hi.theta, hi.v, beta, qk, g, np.arange(hi.n))
    assert np.all(st == 0)
    return O


def run_operator(R, hi):
    shp = (hi.B, hi.H, hi.n)
    Wre, Wim = R.operator(dev(hi.q.reshape(*shp, hi.d), torch.bfloat16),
                          dev(hi.k.reshape(*shp, hi.d), torch.bfloat16), dev(hi.u.reshape(shp)),
                          dev(hi.theta.reshape(shp)), hi.beta, hi.qk, hi.g)
    torch.cuda.synchronize()
    return (Wre.cpu().double().numpy().reshape(hi.B * hi.H, hi.n, hi.n),
            Wim.cpu().double().numpy().reshape(hi.B * hi.H, hi.n, hi.n))


def close_per_head(got, ref, tol, what):
    for h in range(ref.shape[0]):
        scale = max(np.max(np.abs(ref[h].real)), np.max(np.abs(ref[h].imag)))
        err = max(np.max(np.abs(got[h].real - ref[h].real)), np.max(np.abs(got[h].imag - ref[h].imag)))
        assert err <= tol * scale, f"{what} head {h}: err {err:.3e} > {tol} * {scale:.3e}"


def set_rows(x, rows, vec):
    """Rows `rows` of every head of x [BH, n, d] become the vector vec (first len(vec) entries,
    zeros after): exact bf16 values, so the logits between such rows are exact."""
    x[:, rows, :] = 0.0
    x[:, rows, :len(vec)] = np.asarray(vec, dtype=np.float32)


# ------------------------------------------------------------------ logits of 1e4 at beta = 1


def big_logit_heads(seed, theta_zero=False):
    """Two heads (g = 0 and g = 0.5), beta = 1, qk = 1, n = 300, d = dv = 64. Query rows I are
    200 (e_0 + e_1) and key rows J+ / J- are +-200 (e_0 + e_1), so s_ij = +-1e4 exactly on
    I x J+- (<q, k> = 80000, sqrt(d) = 8); q_i for i in I against other keys gives logits of
    tens to about a hundred."""
    hi = W.head_inputs(1, 2, 300, 64, 64, seed=seed, q_scale=1 / 8, u_range=(0.9, 1.0),
                       beta=1.0, qk=1.0, g=[0.0, 0.5],
                       theta_range=(0.0, 0.0) if theta_zero else (-math.pi, math.pi))
    I = np.arange(10, 300, 3)
    set_rows(hi.q, I, [200.0, 200.0])
    set_rows(hi.k, [5, 140, 141, 290], [200.0, 200.0])
    set_rows(hi.k, [7, 200, 260], [-200.0, -200.0])
    return hi


def test_logits_of_ten_thousand_stay_finite_at_beta_one(R, oracle_mod):
    """beta = 1 with logits of +-1e4: every output finite and within 1e-2 max|O| of the
    oracle's log-domain evaluation, per head."""
    hi = big_logit_heads(31)
    re, im = run_head(R, hi)
    assert np.all(np.isfinite(re)) and np.all(np.isfinite(im))
    close_per_head(re + 1j * im, oracle_head(oracle_mod, hi), O_TOL, "logits 1e4")
    assert np.all(im[0] == 0)  # g = 0 head: no imaginary part


def test_logits_of_ten_thousand_rows_stay_stochastic(R):
    """The same logits with real gates (theta = 0) and V = 1: O_i = sum_j W_ij = 1 for every
    row (rows of W are stochastic at beta = 1), to the bf16 rounding of P."""
    hi = big_logit_heads(32, theta_zero=True)
    hi.v[:] = 1.0
    re, im = run_head(R, hi)
    assert np.max(np.abs(re - 1.0)) <= O_TOL
    assert np.all(im == 0)


def test_operator_logits_of_ten_thousand_at_beta_one(R, oracle_mod):
    """W itself at logits of +-1e4, beta = 1: finite, |W| <= 1 and within 1e-3 max|W| of the
    oracle, with its exact zeros."""
    hi = big_logit_heads(33)
    Wre, Wim = run_operator(R, hi)
    Wg = Wre + 1j * Wim
    assert np.all(np.isfinite(Wg)) and np.max(np.abs(Wg)) <= 1.0 + 1e-5
    for h in range(2):
        ref = oracle_mod.operator(hi.q[h], hi.k[h], hi.u[h], hi.theta[h], 1.0, 1.0, f32(hi.g)[h])
        assert np.max(np.abs(Wg[h] - ref)) <= W_TOL * np.max(np.abs(ref)), f"head {h}"
        assert np.all(Wg[h][ref == 0] == 0)


# ------------------------------------------------------------------ lazy rescale of the maximum


@pytest.mark.parametrize("g", [0.0, 0.5])
def test_running_maximum_growing_in_small_steps(R, oracle_mod, g):
    """Logits that grow by about 3 nats per key tile towards earlier keys (the kernel walks key
    tiles from the diagonal back), so the running maximum moves again and again by less than
    the 2^8 the kernel lets a stale maximum lag: beta = 1, every row against the oracle."""
    n = 1024
    hi = W.head_inputs(1, 1, n, 64, 64, seed=35, u_range=(0.97, 1.0), beta=1.0, qk=1.0, g=g)
    hi.q[:] = 0.0
    hi.q[:, :, 0] = 8.0
    hi.q[:, :, 1] = 1.0
    hi.k[:, :, 0] = W.to_bf16_values(np.float32(-3.0 / 128.0) * np.arange(n, dtype=np.float32))
    re, im = run_head(R, hi)
    close_per_head(re + 1j * im, oracle_head(oracle_mod, hi), O_TOL, f"g={g}")


@pytest.mark.parametrize("d,col,j,sign", [(64, 60, 5, 1.0), (64, 17, 40, -1.0),
                                           (128, 100, 77, 1.0), (128, 3, 126, -1.0)])
def test_running_maximum_jumps_on_a_later_tile(R, oracle_mod, d, col, j, sign):
    """Gated head (g = 0.5, beta = 1, qk = +-1), n = 384: the query rows of the last block see
    small logits on key tile 1 (their first tile) and, on key tile 0, one key whose single
    element at column `col` makes a logit of 2400 / sqrt(d) nats (300 or 212). The running
    maximum must move on that later tile, or P = 2^{t - M} overflows. The big element sits in
    either 64-column half of K and Q, at key rows of different warps, with qk of either sign.
    Every row against the oracle."""
    n = 384
    hi = W.head_inputs(1, 1, n, d, d, seed=39, q_scale=1 / math.sqrt(d), u_range=(0.97, 1.0),
                       theta_range=(-0.1, 0.1), beta=1.0, qk=sign, g=0.5)
    hi.q[:, 256:, col] = 4.0
    hi.k[:, j, col] = 600.0 * sign
    re, im = run_head(R, hi)
    assert np.all(np.isfinite(re)) and np.all(np.isfinite(im))
    close_per_head(re + 1j * im, oracle_head(oracle_mod, hi), O_TOL, f"d={d} col={col} j={j}")


# ------------------------------------------------------------------ overflow away from beta = 1


def overflow_heads(seed, s_big_vec, v_scale=1.0, beta=0.0):
    """Two heads with real gates (g = 0; g = 0.5 with theta = 0 and a few closed gates, u = -1),
    n = 300, d = dv = 64. Query rows I and key rows J carry the vector s_big_vec, so the
    logit on I x J is |s_big_vec|^2 / 8 exactly; everything else is small."""
    n = 300
    hi = W.head_inputs(1, 2, n, 64, 64, seed=seed, q_scale=1 / 8, u_range=(0.9, 1.0),
                       theta_range=(0.0, 0.0), beta=beta, qk=1.0, g=[0.0, 0.5])
    hi.u[1, [120, 121, 250]] = -1.0  # m = clamp(0.5 + 0.5 u) = 0: closed gates
    I = np.arange(40, n, 2)
    J = [100, 200]
    set_rows(hi.q, I, s_big_vec)
    set_rows(hi.k, J, s_big_vec)
    hi.v *= np.float32(v_scale)
    hi.v[:] = W.to_bf16_values(hi.v)
    return hi, I, J


def row_classes(hi, I, J):
    """Per head: rows with a live big logit (some j in J, j <= i, with G_ij != 0), rows of I
    without one, and the other rows."""
    out = []
    for h in range(hi.B * hi.H):
        g = f32(hi.g)[h % hi.H]
        m = np.clip((1 - g) + g * hi.u[h].astype(np.float64), 0, 1)
        live = np.zeros(hi.n, bool)
        for i in I:
            for j in J:
                if j <= i and np.all(m[j + 1:i + 1] > 0):
                    live[i] = True
        inI = np.zeros(hi.n, bool)
        inI[I] = True
        out.append((live, inI & ~live, ~inI))
    return out


def test_overflowing_logit_reads_inf_never_nan(R, oracle_mod):
    """beta = 0 with a logit of 200 (e^200 overflows fp32, not fp64): O = +-inf exactly where
    the oracle's value overflows fp32, never NaN; the imaginary lane of real gates stays
    exactly 0 (no 0 * inf); every other row within 1e-2 of the oracle (per class of rows)."""
    hi, I, J = overflow_heads(36, [40.0])  # 40 * 40 / 8 = 200
    re, im = run_head(R, hi)
    ref = oracle_head(oracle_mod, hi)
    assert not np.any(np.isnan(re)) and not np.any(np.isnan(im))
    assert np.all(im == 0)
    with np.errstate(over="ignore"):
        ref32 = ref.real.astype(np.float32).astype(np.float64)
    for h, (live, other_I, rest) in enumerate(row_classes(hi, I, J)):
        assert live.any() and other_I.any()
        assert np.all(np.isinf(ref32[h][live]))
        assert np.array_equal(re[h][live], ref32[h][live]), f"head {h}: inf rows"
        for cls in (other_I, rest):
            scale = np.max(np.abs(ref.real[h][cls]))
            assert np.all(np.isfinite(re[h][cls]))
            assert np.max(np.abs(re[h][cls] - ref.real[h][cls])) <= O_TOL * scale, f"head {h}"


def test_output_in_range_survives_a_row_factor_past_it(R, oracle_mod):
    """beta = 0, a logit of 90 (e^90 = 1.2e39 is past fp32) on rows whose values are 1e-3:
    O ~ 1e36 is within fp32, and so must the output be (the row factor is applied in two
    halves); within 1e-2 of the oracle per class of rows."""
    hi, I, J = overflow_heads(37, [24.0, 12.0], v_scale=1e-3)  # (576 + 144) / 8 = 90
    re, im = run_head(R, hi)
    ref = oracle_head(oracle_mod, hi)
    assert np.all(np.isfinite(re)) and np.all(im == 0)
    for h, (live, other_I, rest) in enumerate(row_classes(hi, I, J)):
        assert np.max(np.abs(ref.real[h][live])) > 1e35
        for cls in (live, other_I, rest):
            scale = np.max(np.abs(ref.real[h][cls]))
            assert np.max(np.abs(re[h][cls] - ref.real[h][cls])) <= O_TOL * scale, f"head {h}"


def test_operator_overflowing_logit_reads_inf_never_nan(R, oracle_mod):
    """W at beta = 0 with a logit of 200: W_ij = G_ij e^{s_ij} reads +inf exactly where the
    oracle's value overflows fp32 and G_ij != 0, every other entry keeps its finite value
    (within 1e-3 of its row's largest finite |W|), never NaN; Im W = 0 exactly (real gates);
    exact zeros where G is 0."""
    hi, I, J = overflow_heads(38, [40.0])
    Wre, Wim = run_operator(R, hi)
    assert not np.any(np.isnan(Wre)) and not np.any(np.isnan(Wim))
    assert np.all(Wim == 0)
    for h in range(2):
        ref = oracle_mod.operator(hi.q[h], hi.k[h], hi.u[h], hi.theta[h], 0.0, 1.0, f32(hi.g)[h]).real
        with np.errstate(over="ignore"):
            ref32 = ref.astype(np.float32).astype(np.float64)
        big = np.isinf(ref32)
        assert big.any()
        assert np.array_equal(Wre[h][big], ref32[big])
        assert np.all(Wre[h][ref == 0] == 0)
        fin = ~big
        for i in range(hi.n):
            f = fin[i]
            scale = np.max(np.abs(ref[i][f]))
            assert np.max(np.abs(Wre[h][i][f] - ref[i][f])) <= W_TOL * scale, f"head {h} row {i}"


# ------------------------------------------------------------------ the zero pattern, through K2


@pytest.mark.parametrize("beta", [0.0, 1.0])
def test_head_kernel_zero_pattern_is_exact(R, oracle_mod, beta):
    """q = 0 with qk = 1 (every logit 0, so P = 1 on live entries, yet the call runs the fused
    head kernel, not the qk = 0 chain) and V a one-hot window, V_j = e_{j - j0} for
    j0 <= j < j0 + 128 (dv = 128): then O_i[c] = W_{i, j0 + c}. O must be exactly 0 wherever
    the oracle's W is 0 (a closed gate on the path, or above the diagonal) and nonzero
    elsewhere, with values within 1e-2 of the largest |W|. Windows slide across block edges;
    gates close at 5% of positions (g = 1: u = 0; g = 0.5: u = -1)."""
    n, j0s = 400, [0, 64, 100, 127, 128, 200, 256, 272]
    B, H = len(j0s), 2
    hi = W.head_inputs(B, H, n, 64, 128, seed=40 + int(beta), u_range=(0.9, 1.0),
                       beta=beta, qk=1.0, g=[1.0, 0.5])
    r = np.random.default_rng(41)
    for bh in range(B * H):
        closed = r.choice(np.arange(1, n), size=20, replace=False)
        hi.u[bh, closed] = 0.0 if bh % H == 0 else -1.0
    hi.q[:] = 0.0
    hi.v[:] = 0.0
    for b, j0 in enumerate(j0s):
        for c in range(128):
            if j0 + c < n:
                hi.v[b * H:(b + 1) * H, j0 + c, c] = 1.0
    re, im = run_head(R, hi)
    Og = re + 1j * im
    for bh in range(B * H):
        b, h = divmod(bh, H)
        j0 = j0s[b]
        Wref = oracle_mod.operator(hi.q[bh], hi.k[bh], hi.u[bh], hi.theta[bh], beta, 1.0,
                                   f32(hi.g)[h])
        want = np.zeros((n, 128), complex)
        cols = np.arange(128)
        ok = j0 + cols < n
        want[:, ok] = Wref[:, j0 + cols[ok]]
        zero = want == 0
        assert zero.any() and (~zero).any()
        assert np.all(Og[bh][zero] == 0), f"b={b} h={h}: structural zeros"
        assert np.all(Og[bh][~zero] != 0), f"b={b} h={h}: nonzero entries"
        assert np.max(np.abs(Og[bh] - want)) <= O_TOL * np.max(np.abs(want)), f"b={b} h={h}"


# ------------------------------------------------------------------ bounded waits


@pytest.mark.parametrize("g", [0.5, 0.0])
def test_head_bounded_wait_reports_timeout(R, oracle_mod, g):
    """A block of the fused head kernel whose K and V loads stop after its first key tile: the
    next wait for a tile runs out (2 s), the status word says timeout, every block winds down
    (each waits for the copies and products it started) and the call returns; the next call
    is correct."""
    hi = W.head_inputs(1, 2, 640, 64, 64, seed=44, q_scale=1 / 8, u_range=(0.9, 1.0),
                       beta=1.0, qk=1.0, g=g)
    R.test_set_head_withhold(0)  # block 0 takes the last query tile: five key tiles
    try:
        with pytest.raises(R.DeviceTimeout):
            run_head(R, hi)
    finally:
        R.test_set_head_withhold(-1)
    re, im = run_head(R, hi)
    close_per_head(re + 1j * im, oracle_head(oracle_mod, hi), O_TOL, "after timeout")


@pytest.mark.parametrize("launch,block", [(0, 5), (1, 0)])
def test_operator_bounded_wait_reports_timeout(R, oracle_mod, launch, block):
    """The operator's statistics launch (block 5: query tile 5, four key tiles) or write
    launch (block 0: two lower tiles) with one block that loads nothing for its second tile:
    its wait runs out, the call reports a timeout and returns; the next call is correct."""
    hi = W.head_inputs(1, 2, 2048, 64, 8, seed=45, q_scale=1 / 8, u_range=(0.9, 1.0),
                       beta=1.0, qk=1.0, g=0.5)
    R.test_set_operator_withhold(launch, block)
    try:
        with pytest.raises(R.DeviceTimeout):
            run_operator(R, hi)
    finally:
        R.test_set_operator_withhold(0, -1)
    Wre, Wim = run_operator(R, hi)
    rows = [0, 1, 127, 128, 640, 1500, 2047]
    for h in range(2):
        got = Wre[h][rows] + 1j * Wim[h][rows]
        ref = oracle_mod.operator_rows(hi.q[h], hi.k[h], hi.u[h], hi.theta[h], 1.0, 1.0, 0.5, rows)
        assert np.max(np.abs(got - ref)) <= W_TOL * np.max(np.abs(ref)), f"head {h}"


# ------------------------------------------------------------------ refusal scan of qk = 0 heads


@pytest.mark.parametrize("dtype,n,d", [("bf16", 64, 64), ("fp32", 64, 64), ("bf16", 301, 8), ("fp32", 301, 8)])
def test_qk0_scan_finds_every_position(R, dtype, n, d):
    """Heads with qk = 0 never form a logit, so their q and k are scanned for values that are
    not finite ("Evaluation and refusals", the NonFinite refusal). The scan reads 16-byte units
    (eight bf16 or four fp32 values): a NaN or an infinity at each of the eight positions of a
    unit, in q or in k, in the second head, must refuse; the same inputs with finite values must
    not."""
    base = W.head_inputs(1, 2, n, d, d, seed=31, beta=0.5, qk=0.0, g=0.3)
    base.dtype = dtype
    run_head(R, base)  # every value finite: no refusal
    bad_values = [np.nan, np.inf, -np.inf]
    for pos in range(8):
        hi = W.head_inputs(1, 2, n, d, d, seed=31, beta=0.5, qk=0.0, g=0.3)
        hi.dtype = dtype
        x = hi.q if pos % 2 == 0 else hi.k
        x.reshape(-1)[n * d + 8 * (pos + 3) + pos] = bad_values[pos % 3]  # head 1, lane pos of a unit
        with pytest.raises(R.NonFinite):
            run_head(R, hi)
