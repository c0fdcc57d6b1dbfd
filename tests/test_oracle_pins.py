"""Pins of the fp64 oracle against what the pages and the mathematics fix.

Every test checks the oracle against something other than itself: values the pages print
(fixtures under tests/golden/), closed forms, library routines that reduce to the same
mathematics (numpy matrix powers, scipy's softmax, triangular solve and IIR filter), or
invariants that a dropped term, a wrong sign or index, or a transposed operand would break.

Source for every citation below: "Resolvent Operator" (teerth.dev/Aether-Lang/integrated/
resolvent/) -- its "Object" definition block, its corners table, its Lean table, its
section "Evaluation and refusals" and its "Test evidence" table -- plus "Op Specs"
(docs.theformalera.com/models/op-specs), section "Attention" (`softmax`, `causalGQA`), and
"A position-only causal softmax head is a causal convolution divided by a prefix
normalizer" (proofs.blah.dev), its theorem `pos-head-is-causal-convolution`.
"""
import math

import numpy as np
import pytest
import scipy.linalg
import scipy.signal
import scipy.special

from conftest import golden


def rng(seed):
    return np.random.default_rng(seed)


def rand_head(seed, n, d, dv=None, u_lo=0.0, u_hi=1.0, zero_frac=0.0):
    r = rng(seed)
    q = r.standard_normal((n, d)).astype(np.float32)
    k = r.standard_normal((n, d)).astype(np.float32)
    v = r.standard_normal((n, dv or d)).astype(np.float32)
    u = r.uniform(u_lo, u_hi, n).astype(np.float32)
    th = r.uniform(-math.pi, math.pi, n).astype(np.float32)
    if zero_frac:
        u[r.choice(n, int(round(zero_frac * n)), replace=False)] = 0.0
    return q, k, v, u, th


def gates_of(oracle_mod, u, th, g):
    return np.array([oracle_mod.gate(*oracle_mod.blend(float(a), float(b), g))
                     for a, b in zip(u, th)])


def neumann(a):
    """sum_{k<n} A^k with A[i, i-1] = a_i (the gate shift), by matrix powers."""
    n = len(a)
    A = np.zeros((n, n), dtype=complex)
    for i in range(1, n):
        A[i, i - 1] = a[i]
    G = np.zeros((n, n), dtype=complex)
    P = np.eye(n, dtype=complex)
    for _ in range(n):
        G += P
        P = P @ A
    return G, A


# ------------------------------------------------------------------ gate


def test_blend_endpoints_and_clamp(oracle_mod):
    """g = 0 removes the gate exactly; g = 1 passes (u, theta) exactly; clamp to [0,1]
    ("Object", blended-gate row; "Test evidence", `an_off_switch_deletes_its_term_exactly`)."""
    r = rng(1)
    for u, th in zip(r.uniform(-3, 3, 50), r.uniform(-10, 10, 50)):
        assert oracle_mod.blend(u, th, 0.0) == (1.0, 0.0) or oracle_mod.blend(u, th, 0.0)[0] == 1.0
        assert oracle_mod.blend(u, th, 0.0)[1] == 0.0
    for u, th in zip(r.uniform(0, 1, 50), r.uniform(-10, 10, 50)):
        assert oracle_mod.blend(u, th, 1.0) == (u, th)
    assert oracle_mod.blend(-0.5, 1.0, 1.0)[0] == 0.0
    assert oracle_mod.blend(1.5, 1.0, 1.0)[0] == 1.0
    assert oracle_mod.blend(-0.5, 2.0, 0.3) == pytest.approx((0.7 - 0.15, 0.6), abs=1e-15)
    assert oracle_mod.blend(0.2, 2.0, 0.5) == pytest.approx((0.6, 1.0), abs=1e-15)


def test_bedm_gate_values(oracle_mod):
    """-1, 0, +1 are the gates (m, theta) = (1, pi), (0, 0), (1, 0) (golden fixture)."""
    for m, th, re, im_bound in golden("bedm_gates.txt"):
        a = oracle_mod.gate(float(m), math.pi if th == "pi" else float(th))
        assert a.real == float(re)
        assert abs(a.imag) <= float(im_bound)


# ------------------------------------------------------------------ path product


@pytest.mark.parametrize("n", [1, 2, 5, 12])
def test_path_product_is_neumann_resolvent(oracle_mod, n):
    """G = (I - A)^{-1} = sum_{k<n} A^k and G (I - A) = I to 1e-14 ("The path-product corner
    is a resolvent"; Lean `occupancy_is_exact_inverse`; "Test evidence", chain row)."""
    r = rng(10 + n)
    a = r.uniform(0, 1, n) * np.exp(1j * r.uniform(-math.pi, math.pi, n))
    a[0] = 7.0 + 3.0j  # a_0 is never read: any value must leave G unchanged
    G = oracle_mod.path_product(a)
    Gn, A = neumann(a)
    assert np.max(np.abs(G - Gn)) <= 1e-14
    I = np.eye(n)
    assert np.max(np.abs(G @ (I - A) - I)) <= 1e-14
    assert np.max(np.abs((I - A) @ G - I)) <= 1e-14
    a2 = a.copy(); a2[0] = 0.0
    assert np.array_equal(oracle_mod.path_product(a2), G)


def test_path_product_modulus_and_zero_pattern(oracle_mod):
    """|G_ij| = prod m_k <= 1; |G_ij| = 1 iff every magnitude on the path is 1; G_ij = 0
    exactly iff some m_k = 0 on the path (Lean `pathProd_abs`, `pathProd_eq_zero_iff`;
    "Test evidence", `a_closed_gate_annihilates_every_path_through_it_exactly`)."""
    n = 40
    r = rng(3)
    m = r.uniform(0.2, 0.999, n)
    m[r.choice(n, 10, replace=False)] = 1.0
    m[[7, 19, 33]] = 0.0
    a = m * np.exp(1j * r.uniform(-math.pi, math.pi, n))
    G = oracle_mod.path_product(a)
    for i in range(n):
        for j in range(i + 1):
            path = m[j + 1:i + 1]
            R = np.prod(path)
            assert abs(abs(G[i, j]) - R) <= 1e-14
            assert abs(G[i, j]) <= 1.0 + 1e-15
            if np.any(path == 0.0):
                assert G[i, j].real == 0.0 and G[i, j].imag == 0.0
            else:
                assert G[i, j] != 0.0
            if np.all(path == 1.0):
                assert abs(abs(G[i, j]) - 1.0) <= 1e-14
            else:
                assert abs(G[i, j]) < 1.0 - 1e-4
        assert np.all(G[i, i + 1:] == 0)


def test_constant_phase_is_rope(oracle_mod):
    """A unit gate of constant phase omega gives G_ij = e^{i omega (i-j)} (Toeplitz) to
    1e-13 (Lean `constant_phase_gate_is_rope`; "Test evidence" RoPE row)."""
    n, w = 64, 0.37
    G = oracle_mod.path_product(np.exp(1j * w * np.ones(n)))
    for i in range(n):
        for j in range(i + 1):
            assert abs(G[i, j] - np.exp(1j * w * (i - j))) <= 1e-13


def test_cumulative_phase_separates(oracle_mod):
    """Any phase schedule on unit gates gives e^{i (Theta_i - Theta_j)}, Theta the prefix
    sum of the phases (Lean `cumulative_phase_is_separable`)."""
    n = 50
    th = rng(4).uniform(-math.pi, math.pi, n)
    G = oracle_mod.path_product(np.exp(1j * th))
    Theta = np.cumsum(th)
    for i in range(n):
        for j in range(i + 1):
            assert abs(G[i, j] - np.exp(1j * (Theta[i] - Theta[j]))) <= 1e-12


def test_scalar_gates_commute_in_window(oracle_mod):
    """Permuting the gates inside a window leaves every path product covering it unchanged
    to 1e-15; entries whose window misses it are bitwise unchanged (Lean
    `PhaseH.scalar_gate_commutes`; "Test evidence" `scalar_gates_commute_within_a_window`)."""
    n, p, q = 30, 10, 16
    r = rng(5)
    a = r.uniform(0.5, 1, n) * np.exp(1j * r.uniform(-1, 1, n))
    b = a.copy()
    b[p:q + 1] = a[p:q + 1][r.permutation(q + 1 - p)]
    Ga, Gb = oracle_mod.path_product(a), oracle_mod.path_product(b)
    for i in range(n):
        for j in range(i + 1):
            if j < p and i >= q:      # the window (j, i] holds the whole permuted range
                assert abs(Ga[i, j] - Gb[i, j]) <= 1e-15
            elif i < p or j >= q:     # the window misses the permuted range
                assert Ga[i, j] == Gb[i, j]


# ------------------------------------------------------------------ corners


def causal_softmax(s):
    """Causal softmax per "Op Specs", `softmax` with visible = (l <= pos), via scipy."""
    n = s.shape[0]
    masked = np.where(np.tril(np.ones((n, n), bool)), s, -np.inf)
    return scipy.special.softmax(masked, axis=1)


def test_softmax_corner_is_causal_softmax(oracle_mod):
    """(1,1,0) is causal softmax attention to 1e-14 with Im exactly 0 (corners table; "Test
    evidence" `the_softmax_corner_is_causal_softmax...`); its readout is `causalGQA`
    ("Op Specs", Attention) with scale 1/sqrt(d)."""
    n, d = 48, 16
    q, k, v, u, th = rand_head(6, n, d)
    W = oracle_mod.operator(q, k, u, th, 1.0, 1.0, 0.0)
    s = (q.astype(np.float64) @ k.astype(np.float64).T) / math.sqrt(d)
    P = causal_softmax(s)
    assert np.max(np.abs(W.real - P)) <= 1e-14
    assert np.all(W.imag == 0.0)
    O = oracle_mod.readout(W, v)
    assert np.max(np.abs(O.real - P @ v.astype(np.float64))) <= 1e-13
    assert np.all(O.imag == 0.0)


def test_kernel_corner_is_bare_exponential(oracle_mod):
    """(0,1,0) is W_ij = e^{s_ij} on the causal triangle and 0 above (corners table)."""
    n, d = 32, 8
    q, k, v, u, th = rand_head(7, n, d)
    W = oracle_mod.operator(q, k, u, th, 0.0, 1.0, 0.0)
    s = (q.astype(np.float64) @ k.astype(np.float64).T) / math.sqrt(d)
    E = np.where(np.tril(np.ones((n, n), bool)), np.exp(s), 0.0)
    assert np.max(np.abs(W.real - E) / np.maximum(E, 1e-300)) <= 1e-13
    assert np.all(W.imag == 0.0)
    assert np.all(W[np.triu_indices(n, 1)] == 0)


def test_path_corner_is_the_resolvent(oracle_mod):
    """(0,0,1) is W = G = sum_k A^k with a_k = clamp(u_k) e^{i theta_k} (corners table)."""
    n, d = 12, 4
    q, k, v, u, th = rand_head(8, n, d, zero_frac=0.2)
    W = oracle_mod.operator(q, k, u, th, 0.0, 0.0, 1.0)
    a = np.clip(u.astype(np.float64), 0, 1) * np.exp(1j * th.astype(np.float64))
    Gn, _ = neumann(a)
    assert np.max(np.abs(W - Gn)) <= 1e-14
    assert np.array_equal(W, oracle_mod.path_product(gates_of(oracle_mod, u, th, 1.0)))


def test_corners_distinct_worked_example(oracle_mod):
    """Entry (1,0) reads 1/2 at beta = 1 and 1 at beta = 0 (golden fixture)."""
    for n, beta, qk, g, i, j, re, im in golden("corners_distinct.txt"):
        n = int(n)
        q = np.ones((n, 1), np.float32); k = np.ones((n, 1), np.float32)
        u = np.full(n, 0.3, np.float32); th = np.full(n, 1.1, np.float32)
        W = oracle_mod.operator(q, k, u, th, float(beta), float(qk), float(g))
        assert W[int(i), int(j)] == complex(float(re), float(im))


def test_random_inputs_separate_the_corners(oracle_mod):
    """Random inputs separate every pair of corners by more than 0.5 ("Test evidence"
    `the_three_corners_are_distinct_operators`)."""
    q, k, v, u, th = rand_head(9, 16, 8)
    Ws = [oracle_mod.operator(q, k, u, th, *c) for c in
          [(1.0, 1.0, 0.0), (0.0, 1.0, 0.0), (0.0, 0.0, 1.0)]]
    for x in range(3):
        for y in range(x + 1, 3):
            assert np.max(np.abs(Ws[x] - Ws[y])) > 0.5


# ------------------------------------------------------------------ normaliser


def test_beta_one_rows_are_stochastic(oracle_mod):
    """At beta = 1 rows sum to 1 within 1e-14 with gates on or off (real gates); with
    phases the moduli sum to 1 (Lean `softmax_row_sum_one`, `beta_one_row_is_one`)."""
    n, d = 40, 8
    q, k, v, u, th = rand_head(11, n, d, zero_frac=0.1)
    zero_th = np.zeros_like(th)
    for g in (0.0, 0.4, 1.0):
        W = oracle_mod.operator(q, k, u, zero_th, 1.0, 1.0, g)
        assert np.max(np.abs(W.sum(axis=1) - 1.0)) <= 1e-14
        Wp = oracle_mod.operator(q, k, u, th, 1.0, 1.0, g)
        assert np.max(np.abs(np.abs(Wp).sum(axis=1) - 1.0)) <= 1e-14


def test_bare_kernel_rows_sum_to_i_plus_one(oracle_mod):
    """g = 0, qk = 0, beta = 0: row i sums to exactly i + 1 (golden fixture)."""
    rows = golden("bare_row_sums.txt")
    n = len(rows)
    q, k, v, u, th = rand_head(12, n, 4)
    W = oracle_mod.operator(q, k, u, th, 0.0, 0.0, 0.0)
    for i, s in rows:
        assert W[int(i)].sum() == complex(float(s), 0.0)


def test_beta_interior_self_consistent(oracle_mod):
    """beta in (0,1) -- the pages make no statement there ("parity unpinned"); the oracle
    only has to satisfy W(beta)_ij Z_i^beta = W(0)_ij with Z_i = sum_j |W(0)_ij|."""
    n, d = 24, 8
    q, k, v, u, th = rand_head(13, n, d, zero_frac=0.1)
    W0 = oracle_mod.operator(q, k, u, th, 0.0, 0.8, 0.6)
    Z = np.abs(W0).sum(axis=1)
    for beta in (0.25, 0.5, 0.7):
        Wb = oracle_mod.operator(q, k, u, th, beta, 0.8, 0.6)
        lhs = Wb * (Z ** beta)[:, None]
        assert np.max(np.abs(lhs - W0) / np.maximum(np.abs(W0), 1e-300)) <= 1e-12


# ------------------------------------------------------------------ chain


def test_chain_is_forward_substitution(oracle_mod):
    """The chain solves (I - A) y = b (scipy triangular solve) and equals the path-product
    readout to 1e-12; beta = 1 breaks it (planted negative) ("The path-product corner is a
    resolvent"; Lean `chain_path_product`, `chain_eq_sum`)."""
    n, d, dv = 30, 4, 5
    q, k, v, u, th = rand_head(14, n, d, dv=dv, u_lo=0.5, zero_frac=0.1)
    a = gates_of(oracle_mod, u, th, 1.0)
    y = oracle_mod.chain(a, v)
    _, A = neumann(a)
    ys = scipy.linalg.solve_triangular(np.eye(n) - A, v.astype(np.float64), lower=True)
    assert np.max(np.abs(y - ys)) <= 1e-12 * max(1.0, np.max(np.abs(ys)))
    W = oracle_mod.operator(q, k, u, th, 0.0, 0.0, 1.0)
    assert np.max(np.abs(oracle_mod.readout(W, v) - y)) <= 1e-12
    W1 = oracle_mod.operator(q, k, u, th, 1.0, 0.0, 1.0)
    assert np.max(np.abs(oracle_mod.readout(W1, v) - y)) > 0.1
    # the page's form: b_0 = 0 gives y_0 = 0
    v0 = v.copy(); v0[0] = 0
    assert np.all(oracle_mod.chain(a, v0)[0] == 0)


def test_chain_constant_gate_is_iir_filter(oracle_mod):
    """With a constant gate a the chain is the one-pole filter y = b / (1 - a z^-1)."""
    n = 200
    a0 = 0.97 * np.exp(0.01j)
    b = rng(15).standard_normal((n, 3)).astype(np.float32)
    y = oracle_mod.chain(np.full(n, a0), b)
    for c in range(3):
        ref = scipy.signal.lfilter([1.0], [1.0, -a0], b[:, c].astype(np.float64))
        assert np.max(np.abs(y[:, c] - ref)) <= 1e-12


# ------------------------------------------------------------------ float64 properties


def test_future_never_moves_the_past(oracle_mod):
    """Rows up to t are bitwise unchanged when later inputs change; entries above the
    diagonal are exactly 0 ("Test evidence" `perturbing_the_future_never_moves_the_past`)."""
    n, d, t0 = 20, 4, 9
    q, k, v, u, th = rand_head(16, n, d)
    q2, k2, v2, u2, th2 = rand_head(17, n, d)
    for arr, arr2 in ((q, q2), (k, k2), (v, v2), (u, u2), (th, th2)):
        arr2[:t0 + 1] = arr[:t0 + 1]
    for sw in [(1.0, 1.0, 0.5), (0.0, 1.0, 1.0), (0.5, 0.7, 0.3)]:
        W = oracle_mod.operator(q, k, u, th, *sw)
        W2 = oracle_mod.operator(q2, k2, u2, th2, *sw)
        assert np.array_equal(W[:t0 + 1], W2[:t0 + 1])
        assert np.array_equal(oracle_mod.readout(W, v)[:t0 + 1],
                              oracle_mod.readout(W2, v2)[:t0 + 1])
        assert np.all(W[np.triu_indices(n, 1)] == 0)


def test_off_switches_delete_their_terms(oracle_mod):
    """g = 0 removes the gates exactly; qk = 0 removes q and k exactly ("Test evidence"
    `an_off_switch_deletes_its_term_exactly`)."""
    n, d = 16, 4
    q, k, v, u, th = rand_head(18, n, d)
    q2, k2, v2, u2, th2 = rand_head(19, n, d)
    assert np.array_equal(oracle_mod.operator(q, k, u, th, 0.6, 0.9, 0.0),
                          oracle_mod.operator(q, k, u2, th2, 0.6, 0.9, 0.0))
    assert np.array_equal(oracle_mod.operator(q, k, u, th, 0.6, 0.0, 0.4),
                          oracle_mod.operator(q2, k2, u, th, 0.6, 0.0, 0.4))


def test_large_logits_stay_finite_at_beta_one(oracle_mod):
    """Logits of +-1e4 at beta = 1 stay finite, rows stochastic to 1e-9, and match softmax
    to 1e-9 (golden fixture; "Evaluation and refusals")."""
    n = 12
    r = rng(20)
    sgn = np.where(r.uniform(size=n) < 0.5, -1.0, 1.0)
    q = (100.0 * sgn).astype(np.float32).reshape(n, 1)
    k = (100.0 * np.where(r.uniform(size=n) < 0.5, -1.0, 1.0)).astype(np.float32).reshape(n, 1)
    u = r.uniform(0.2, 1, n).astype(np.float32); th = np.zeros(n, np.float32)
    s = q.astype(np.float64) @ k.astype(np.float64).T
    assert np.max(np.abs(np.tril(s))) == 1e4
    for g in (0.0, 0.5):
        W = oracle_mod.operator(q, k, u, th, 1.0, 1.0, g)
        assert np.all(np.isfinite(W))
        assert np.max(np.abs(W.sum(axis=1) - 1)) <= 1e-9
        assert np.max(np.abs(W)) <= 1.0
    W = oracle_mod.operator(q, k, u, th, 1.0, 1.0, 0.0)
    assert np.max(np.abs(W.real - causal_softmax(s))) <= 1e-9


def test_overflowing_logit_reads_inf_never_nan(oracle_mod):
    """At beta = 0 a logit of 2e4 reads +inf, never NaN; an exactly-zero lane of G stays 0
    (golden fixture; "Evaluation and refusals", overflow row)."""
    rows = [r for r in golden("overflow_values.txt") if r[0] == "overflow_at_beta_zero"]
    logit = float(rows[0][1])
    n = 3
    x = np.float32(math.sqrt(logit))
    q = np.full((n, 1), x, np.float32); k = np.full((n, 1), x, np.float32)
    s = float(q[0, 0]) * float(k[0, 0])
    u = np.ones(n, np.float32); th = np.zeros(n, np.float32)
    W = oracle_mod.operator(q, k, u, th, 0.0, 1.0, 1.0)
    assert s > 709.8
    tri = W[np.tril_indices(n)]
    assert np.all(tri.real == np.inf)
    assert np.all(tri.imag == 0.0)          # the zero lane stays 0, not 0 * inf
    assert not np.any(np.isnan(W.real)) and not np.any(np.isnan(W.imag))


def test_non_finite_inputs_are_refused(oracle_mod):
    """Each non-finite input class is refused; with qk = 0 a dot product that would
    overflow is accepted ("Evaluation and refusals", non-finite row)."""
    n, d = 6, 3
    q, k, v, u, th = rand_head(21, n, d)
    base = dict(q=q, k=k, u=u, theta=th, beta=1.0, qk=1.0, g=0.5)

    def run(**kw):
        a = dict(base); a.update(kw)
        return oracle_mod.operator(a["q"], a["k"], a["u"], a["theta"], a["beta"], a["qk"], a["g"])

    run()
    for name in ("q", "k", "u", "theta"):
        for bad in (np.nan, np.inf, -np.inf):
            x = base[name].copy()
            x.flat[3] = bad
            with pytest.raises(oracle_mod.NonFinite):
                run(**{name: x})
    for name in ("beta", "qk", "g"):
        with pytest.raises(oracle_mod.NonFinite):
            run(**{name: float("nan")})
        with pytest.raises(oracle_mod.NonFinite):
            run(**{name: float("inf")})
    with pytest.raises(oracle_mod.NonFinite):     # g * theta overflows
        run(g=1e300, theta=np.full(n, 1e30, np.float32))
    big = np.full((n, d), 3.0e38, np.float32)
    with pytest.raises(oracle_mod.NonFinite):     # qk * s overflows
        run(q=big, k=big, qk=1e300)
    W = run(q=big, k=big, qk=0.0)                 # qk = 0: the dot product is not taken
    assert np.all(np.isfinite(W))


def test_empty_sequence_and_closed_gates(oracle_mod):
    """Empty in, empty out; closing every gate leaves the identity ("Evaluation and
    refusals", all-masked and empty rows; "Test evidence", last row)."""
    e = np.zeros((0, 4), np.float32)
    assert oracle_mod.operator(e, e, np.zeros(0, np.float32), np.zeros(0, np.float32),
                               1.0, 1.0, 0.5).shape == (0, 0)
    with pytest.raises(oracle_mod.ShapeError):
        oracle_mod.operator(np.zeros((3, 0), np.float32), np.zeros((3, 0), np.float32),
                            np.zeros(3, np.float32), np.zeros(3, np.float32), 1.0, 1.0, 0.5)
    n, d = 10, 4
    q, k, v, u, th = rand_head(22, n, d)
    closed = np.zeros(n, np.float32)
    W1 = oracle_mod.operator(q, k, closed, th, 1.0, 1.0, 1.0)
    assert np.array_equal(W1, np.eye(n))
    W0 = oracle_mod.operator(q, k, closed, th, 0.0, 1.0, 1.0)
    s = np.einsum("ij,ij->i", q.astype(np.float64), k.astype(np.float64)) / 2.0
    assert np.max(np.abs(np.diag(W0) - np.exp(s)) / np.exp(s)) <= 1e-14
    assert np.all(W0 - np.diag(np.diag(W0)) == 0)


def test_position_only_head_is_a_causal_convolution(oracle_mod):
    """Logits that depend only on i - j: the softmax-corner readout is the causal
    convolution of v with e^{a} divided by the prefix sum of e^{a} ("A position-only causal
    softmax head ...", theorem `pos-head-is-causal-convolution`)."""
    n, c0, c1, c2 = 40, 0.5, 0.25, -0.0625
    i = np.arange(n, dtype=np.float64)
    # q_i . k_j = c0 + c1 (i-j) + c2 (i-j)^2, every term exact in fp32 and fp64
    q = np.stack([np.ones(n), i, i * i], axis=1).astype(np.float32)
    k = np.stack([c0 - c1 * i + c2 * i * i, c1 - 2 * c2 * i, np.full(n, c2)], axis=1).astype(
        np.float32)
    v = rng(23).standard_normal((n, 2)).astype(np.float32)
    u = np.ones(n, np.float32); th = np.zeros(n, np.float32)
    O = oracle_mod.readout(oracle_mod.operator(q, k, u, th, 1.0, 1.0, 0.0), v)
    dd = np.arange(n, dtype=np.float64)
    ea = np.exp((c0 + c1 * dd + c2 * dd * dd) / math.sqrt(3.0))
    for ch in range(2):
        num = np.convolve(ea, v[:, ch].astype(np.float64))[:n]
        ref = num / np.cumsum(ea)
        assert np.max(np.abs(O[:, ch].real - ref)) <= 1e-13
    assert np.all(O.imag == 0)


def _offset_qk(n, c0, c1, c2):
    """q, k [n,4] with <q_i, k_j> / sqrt(4) = (c0 + c1 (i-j) + c2 (i-j)^2) / 2 exactly (fp32
    and fp64 alike for small dyadic c and n), and the same logits per offset d."""
    i = np.arange(n, dtype=np.float64)
    q = np.stack([np.ones(n), i, i * i, np.zeros(n)], axis=1).astype(np.float32)
    k = np.stack([c0 - c1 * i + c2 * i * i, c1 - 2 * c2 * i, np.full(n, c2), np.zeros(n)],
                 axis=1).astype(np.float32)
    d = np.arange(n, dtype=np.float64)
    return q, k, ((c0 + c1 * d + c2 * d * d) / 2.0).astype(np.float32)


@pytest.mark.parametrize("beta,qk", [(1.0, 1.0), (0.0, 1.0), (1.0, -0.75), (0.0, 0.5)])
def test_position_head_is_the_operator_with_offset_logits(oracle_mod, beta, qk):
    """The position-only head equals the general operator (pinned above) followed by the
    readout, at g = 0, when <q_i, k_j>/sqrt(d) depends only on i - j."""
    n = 48
    q, k, a = _offset_qk(n, 0.5, 0.125, -0.015625)
    v = rng(31).standard_normal((n, 3)).astype(np.float32)
    u = np.ones(n, np.float32); th = np.zeros(n, np.float32)
    ref = oracle_mod.readout(oracle_mod.operator(q, k, u, th, beta, qk, 0.0), v)
    O = oracle_mod.position_head(a, v, beta, qk)
    assert np.max(np.abs(O - ref.real)) <= 1e-12 * max(1.0, np.max(np.abs(ref)))
    assert np.all(ref.imag == 0)


def test_position_head_is_a_causal_convolution_over_a_prefix_sum(oracle_mod):
    """The theorem's right-hand side: (sum_d e^{a(d)} v_{i-d}) / (sum_{d<=i} e^{a(d)}),
    by numpy's convolution and cumulative sum."""
    n = 64
    a = rng(32).standard_normal(n).astype(np.float32)
    v = rng(33).standard_normal((n, 4)).astype(np.float32)
    O = oracle_mod.position_head(a, v, 1.0, 1.0)
    ea = np.exp(a.astype(np.float64))
    for ch in range(4):
        ref = np.convolve(ea, v[:, ch].astype(np.float64))[:n] / np.cumsum(ea)
        assert np.max(np.abs(O[:, ch] - ref)) <= 1e-13


def test_position_head_closed_forms(oracle_mod):
    """Constant logits: a prefix mean at beta = 1, e^{qk c} times a prefix sum at beta = 0;
    qk = 0 ignores a entirely."""
    n = 30
    v = rng(34).standard_normal((n, 2)).astype(np.float32).astype(np.float64)
    cnt = np.arange(1, n + 1)[:, None]
    c = np.full(n, 0.75, np.float32)
    assert np.max(np.abs(oracle_mod.position_head(c, v, 1.0, 2.0) - np.cumsum(v, 0) / cnt)) <= 1e-13
    assert np.max(np.abs(oracle_mod.position_head(c, v, 0.0, 2.0) - math.exp(1.5) * np.cumsum(v, 0))) <= 1e-12
    a = rng(35).standard_normal(n).astype(np.float32)
    assert np.max(np.abs(oracle_mod.position_head(a, v, 1.0, 0.0) - np.cumsum(v, 0) / cnt)) <= 1e-13
    # causality: row i reads v_0 .. v_i only
    O = oracle_mod.position_head(a, v, 1.0, 1.0)
    v2 = v.copy(); v2[17:] += 5.0
    O2 = oracle_mod.position_head(a, v2, 1.0, 1.0)
    assert np.array_equal(O[:17], O2[:17]) and not np.array_equal(O[17:], O2[17:])


@pytest.mark.parametrize("beta", [0.25, 0.5, 0.75])
def test_intermediate_beta_closed_forms(oracle_mod, beta):
    """beta strictly inside (0, 1), where W = G e^{qk s} / Z^beta has closed forms when every
    logit is the same: with q = 0 and open gates (g = 0), Z_i = i + 1 and
    W_ij = (i + 1)^-beta; a position-only head with constant logits c gives
    O_i = e^{qk c (1 - beta)} (i + 1)^-beta sum_{j<=i} v_j. A wrong exponent (Z^{1-beta},
    Z^-beta left out, or beta applied to the shift) fails them."""
    n, d = 24, 8
    q = np.zeros((n, d), np.float32)
    k = rng(44).standard_normal((n, d)).astype(np.float32)
    u = rng(45).uniform(0.0, 1.0, n).astype(np.float32)
    th = rng(46).uniform(-3.0, 3.0, n).astype(np.float32)
    Wm = oracle_mod.operator(q, k, u, th, beta, 0.7, 0.0)
    i = np.arange(n)[:, None].astype(np.float64)
    expect = np.tril(np.ones((n, n))) * (i + 1.0) ** -beta
    assert np.max(np.abs(Wm - expect)) <= 1e-14
    v = rng(47).standard_normal((n, 3)).astype(np.float32).astype(np.float64)
    c = np.full(n, -1.25, np.float32)
    qk = 0.8
    O = oracle_mod.position_head(c, v, beta, qk)
    ref = math.exp(qk * -1.25 * (1.0 - beta)) * (i + 1.0) ** -beta * np.cumsum(v, 0)
    assert np.max(np.abs(O - ref)) <= 1e-12 * (1.0 + np.max(np.abs(ref)))


def test_operator_rows_are_rows_of_the_operator(oracle_mod):
    """The row-sampled operator (for large n) gives exactly the rows of the dense one, with
    closed gates, complex phases and every switch corner, and refuses the same inputs."""
    n, d = 45, 8
    q = rng(40).standard_normal((n, d)).astype(np.float32)
    k = rng(41).standard_normal((n, d)).astype(np.float32)
    u = rng(42).uniform(-0.3, 1.2, n).astype(np.float32); u[[7, 30]] = 0.0
    th = rng(43).uniform(-3.0, 3.0, n).astype(np.float32)
    rows = [0, 1, 7, 8, 29, 31, 44, 8]
    for beta, qk, g in [(1.0, 1.0, 0.5), (0.0, 1.0, 0.0), (0.0, 0.0, 1.0), (0.5, 0.7, 0.3)]:
        full = oracle_mod.operator(q, k, u, th, beta, qk, g)
        part = oracle_mod.operator_rows(q, k, u, th, beta, qk, g, rows)
        assert np.array_equal(part, full[rows])
    bad = q.copy(); bad[3, 2] = np.inf
    with pytest.raises(oracle_mod.NonFinite):
        oracle_mod.operator_rows(bad, k, u, th, 1.0, 1.0, 0.5, [5])
    with pytest.raises(oracle_mod.ShapeError):
        oracle_mod.operator_rows(q, k, u, th, 1.0, 1.0, 0.5, [-1])


def test_position_rows_are_rows_of_the_head(oracle_mod):
    """The row-sampled evaluation (for long sequences) gives exactly the rows of the whole
    head, at every switch setting, and refuses the same inputs."""
    n = 57
    a = rng(38).standard_normal(n).astype(np.float32)
    v = rng(39).standard_normal((n, 3)).astype(np.float32)
    rows = [0, 1, 17, 56, 33, 0]
    for beta, qk in [(1.0, 1.0), (0.0, 0.5), (0.5, -0.75), (1.0, 0.0)]:
        full = oracle_mod.position_head(a, v, beta, qk)
        part = oracle_mod.position_rows(a, v, beta, qk, rows)
        assert np.array_equal(part, full[rows])
    bad = a.copy(); bad[40] = np.nan
    with pytest.raises(oracle_mod.NonFinite):
        oracle_mod.position_rows(bad, v, 1.0, 1.0, [3])
    with pytest.raises(oracle_mod.ShapeError):
        oracle_mod.position_rows(a, v, 1.0, 1.0, [n])


def test_position_head_refusals_and_batching(oracle_mod):
    n = 12
    v = rng(36).standard_normal((n, 2)).astype(np.float32)
    a = rng(37).standard_normal(n).astype(np.float32)
    bad = a.copy(); bad[5] = np.inf
    with pytest.raises(oracle_mod.NonFinite):
        oracle_mod.position_head(bad, v, 1.0, 0.0)       # refused even at qk = 0
    big = np.full(n, 1e10, np.float32)
    with pytest.raises(oracle_mod.NonFinite):
        oracle_mod.position_head(big, v, 1.0, 1e300)     # qk * a overflows
    assert oracle_mod.position_head(np.zeros(0, np.float32), np.zeros((0, 2), np.float32),
                                    1.0, 1.0).shape == (0, 2)
    # batched: head h of every batch reads table h; per-head switches
    H, B = 2, 3
    tab = rng(38).standard_normal((H, n)).astype(np.float32)
    vv = rng(39).standard_normal((B * H, n, 2)).astype(np.float32)
    beta = np.array([1.0, 0.0] * B); qk = np.array([1.0, 0.5] * B)
    O, st = oracle_mod.position_heads(tab, vv, beta, qk)
    assert np.all(st == 0)
    for h in range(B * H):
        assert np.array_equal(O[h], oracle_mod.position_head(tab[h % H], vv[h], beta[h], qk[h]))


# ------------------------------------------------------------------ batched routines


def test_head_rows_equals_operator_then_readout(oracle_mod):
    """The row-sampled batched readout is bitwise the dense operator followed by readout."""
    BH, n, d, dv = 3, 37, 8, 6
    r = rng(24)
    q = r.standard_normal((BH, n, d)).astype(np.float32)
    k = r.standard_normal((BH, n, d)).astype(np.float32)
    v = r.standard_normal((BH, n, dv)).astype(np.float32)
    u = r.uniform(-0.5, 1.5, (BH, n)).astype(np.float32)
    th = r.uniform(-3, 3, (BH, n)).astype(np.float32)
    beta, qk, g = [1.0, 0.5, 0.0], [1.0, 0.0, 0.7], [0.3, 1.0, 0.0]
    rows = [0, 5, 17, 36]
    O, st = oracle_mod.head_rows(q, k, u, th, v, beta, qk, g, rows)
    assert np.all(st == 0)
    for h in range(BH):
        W = oracle_mod.operator(q[h], k[h], u[h], th[h], beta[h], qk[h], g[h])
        Od = oracle_mod.readout(W, v[h])
        assert np.array_equal(O[h], Od[rows])


def test_gate_prep_block_products_are_path_products(oracle_mod):
    """prefix_i = G[i, s-1], suffix_j = G[e, j], carry_b = G[e, s-1] for every block [s, e]
    (first block from index 1): bitwise against the path product, and to 1e-14 against the
    Neumann resolvent."""
    BH, n, blk = 2, 45, 8
    r = rng(25)
    u = r.uniform(-0.3, 1.3, (BH, n)).astype(np.float32)
    th = r.uniform(-3, 3, (BH, n)).astype(np.float32)
    gp = oracle_mod.gate_prep(u, th, [0.7, 1.0], block=blk)
    assert np.all(gp["status"] == 0)
    for h, g in enumerate([0.7, 1.0]):
        a = gates_of(oracle_mod, u[h], th[h], g)
        assert np.array_equal(gp["gate"][h], a)
        G = oracle_mod.path_product(a)
        Gn, _ = neumann(a)
        for b in range((n + blk - 1) // blk):
            s, e = b * blk, min(b * blk + blk - 1, n - 1)
            c = max(s - 1, 0)
            for i in range(s, e + 1):
                assert gp["prefix"][h, i] == G[i, c]
                assert gp["suffix"][h, i] == G[e, i]
                assert abs(gp["prefix"][h, i] - Gn[i, c]) <= 1e-14
                assert abs(gp["suffix"][h, i] - Gn[e, i]) <= 1e-14
            assert gp["carry"][h, b] == G[e, c]


def test_chain_heads_matches_single_chain(oracle_mod):
    BH, n, dv = 3, 50, 4
    r = rng(26)
    u = r.uniform(0.8, 1.0, (BH, n)).astype(np.float32)
    th = r.uniform(-3, 3, (BH, n)).astype(np.float32)
    b = r.standard_normal((BH, n, dv)).astype(np.float32)
    y, env, st = oracle_mod.chain_heads(u, th, [1.0, 0.5, 0.0], b)
    assert np.all(st == 0)
    for h, g in enumerate([1.0, 0.5, 0.0]):
        yh, eh = oracle_mod.chain(gates_of(oracle_mod, u[h], th[h], g), b[h], with_envelope=True)
        assert np.array_equal(y[h], yh) and np.array_equal(env[h], eh)
        assert np.all(np.abs(yh) <= eh * (1 + 1e-12) + 1e-300)


def test_chain_envelope_is_the_chain_of_moduli(oracle_mod):
    """The forward-error envelope that scales every GPU chain tolerance,
    env_i = |a_i| env_{i-1} + |b_i|, is the same chain over the reals with |a| and |b|
    ("Resolvent Operator", Lean table, `CEQ.V15Fork.chain_eq_sum`: the chain is
    sum_{s<=i} (prod_{k=s+1..i} a_k) b_s): env_i = sum_{s<=i} R_is |b_s| with R_is the modulus of
    the path product (pinned to the Neumann resolvent above), to 1e-12. For one constant gate
    it is the first-order IIR filter of |b| with pole |a| (scipy's lfilter)."""
    n, dv = 60, 3
    r = rng(27)
    for g, lo in ((1.0, 0.7), (0.5, -0.3), (0.0, 0.0)):
        u = r.uniform(lo, 1.0, n).astype(np.float32)
        u[r.choice(n, 3, replace=False)] = 0.0
        th = r.uniform(-3, 3, n).astype(np.float32)
        b = r.standard_normal((n, dv)).astype(np.float32)
        a = gates_of(oracle_mod, u, th, g)
        _, env = oracle_mod.chain(a, b, with_envelope=True)
        R = np.abs(oracle_mod.path_product(a))
        want = np.tril(R) @ np.abs(b.astype(np.float64))
        assert np.max(np.abs(env - want) / np.maximum(want, 1e-300)) <= 1e-12, g
        # the batched routine returns the same envelope
        _, env_b, st = oracle_mod.chain_heads(u[None], th[None], [g], b[None])
        assert st[0] == 0 and np.array_equal(env_b[0], env)
    # one constant gate of modulus 0.9 and any phase
    a0 = 0.9 * np.exp(1j * 0.7)
    b = r.standard_normal((200, dv)).astype(np.float32)
    a = np.full(200, a0)
    _, env = oracle_mod.chain(a, b, with_envelope=True)
    for c in range(dv):
        ref = scipy.signal.lfilter([1.0], [1.0, -abs(a0)], np.abs(b[:, c].astype(np.float64)))
        assert np.max(np.abs(env[:, c] - ref) / ref) <= 1e-12
