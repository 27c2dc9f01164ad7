"""Pins for the float64 oracle: each test checks it against something other
than its own formulas (library routines, inverse functions, finite
differences, closed forms, brute force, invariants)."""
import math

import numpy as np
import pytest
from scipy.special import expit, logit

import oracle
import synthetic as syn

RNG = np.random.default_rng(1234)


def _prm(a_z=0.0, a_r=0.0, a_c=0.0, b_z=0.0, b_r=0.0, b_c=0.0):
    return [a_z, a_r, a_c, b_z, b_r, b_c]


def _params(d_h, rng, scale=1.0, bias=0.0):
    return {k: (rng.uniform(-scale, scale, d_h) if k.startswith("a") else
                rng.uniform(-bias, bias, d_h)) for k in oracle.GATE_ORDER}


# ---------------------------------------------------------------- the cell f
def test_cell_at_zero_state_is_z_times_c():
    """At h = 0 the cell reduces to sigma(P_z + b_z) * tanh(P_c + b_c) (r drops out)."""
    for _ in range(50):
        pz, pr, pc = RNG.normal(0, 2, 3)
        b = RNG.normal(0, 0.5, 3)
        a = RNG.uniform(-1, 1, 3)
        f, _ = oracle.cell(0.0, pz, pr, pc, [*a, *b])
        assert f == pytest.approx(expit(pz + b[0]) * np.tanh(pc + b[2]), abs=1e-15)


def test_cell_update_gate_recovered_by_logit():
    """With a_c = 0, c_t = tanh(P_c) is known; 1 - z_t = (h_t - c_t)/(h_{t-1} - c_t)
    and logit(z_t) - P_z = a_z h_{t-1} must recover a_z."""
    T, a_z = 40, 0.73
    P = RNG.normal(0, 1, (1, T, 3))
    H = oracle.sequential(P, [[a_z], [0.4], [0.0], [0.0], [0.0], [0.0]])[0, :, 0]
    c = np.tanh(P[0, :, 2])
    hp = np.concatenate([[0.0], H[:-1]])
    z = 1.0 - (H - c) / (hp - c)
    est = (logit(z) - P[0, :, 0])[1:] / hp[1:]
    ok = np.abs(hp[1:]) > 0.05
    np.testing.assert_allclose(est[ok], a_z, atol=1e-7)


def test_cell_candidate_and_reset_recovered_by_inverses():
    """With z = 1 (P_z large), h_t = c_t = tanh(P_c + a_c r_t h_{t-1}).  With r = 1
    (P_r large) arctanh recovers a_c; with P_r random it recovers r_t and logit(r_t)
    recovers a_r."""
    T = 40
    P = RNG.normal(0, 0.6, (1, T, 3))
    P[0, :, 0] = 60.0
    P1 = P.copy()
    P1[0, :, 1] = 60.0
    a_c = -0.81
    H = oracle.sequential(P1, [[0.3], [0.2], [a_c], [0.0], [0.0], [0.0]])[0, :, 0]
    hp = np.concatenate([[0.0], H[:-1]])
    est = (np.arctanh(H) - P1[0, :, 2])[1:] / hp[1:]
    ok = np.abs(hp[1:]) > 0.05
    np.testing.assert_allclose(est[ok], a_c, atol=1e-9)

    a_r = 0.57
    H = oracle.sequential(P, [[0.3], [a_r], [a_c], [0.0], [0.0], [0.0]])[0, :, 0]
    hp = np.concatenate([[0.0], H[:-1]])
    r = (np.arctanh(H) - P[0, :, 2])[1:] / (a_c * hp[1:])
    ok = np.abs(hp[1:]) > 0.1
    est = (logit(r[ok]) - P[0, 1:, 1][ok]) / hp[1:][ok]
    np.testing.assert_allclose(est, a_r, atol=1e-6)


def test_cell_biases_enter_their_own_gate():
    """Moving s from P_g into b_g leaves f unchanged, gate by gate."""
    for _ in range(30):
        h = RNG.uniform(-0.9, 0.9)
        p = RNG.normal(0, 1, 3)
        a = RNG.uniform(-1, 1, 3)
        f0, J0 = oracle.cell(h, *p, [*a, 0, 0, 0])
        for g in range(3):
            s = RNG.normal()
            q = p.copy()
            q[g] -= s
            bias = [0.0, 0.0, 0.0]
            bias[g] = s
            f1, J1 = oracle.cell(h, *q, [*a, *bias])
            assert f1 == pytest.approx(f0, abs=1e-14)
            assert J1 == pytest.approx(J0, abs=1e-13)


def test_cell_limits():
    """z -> 0 keeps h; z -> 1 with a_c = 0 gives tanh(P_c)."""
    f, J = oracle.cell(0.37, -60.0, 0.3, 1.2, _prm(0.5, 0.5, 0.5))
    assert f == pytest.approx(0.37, abs=1e-15) and J == pytest.approx(1.0, abs=1e-15)
    f, J = oracle.cell(0.37, 60.0, 0.3, 1.2, _prm(0.5, 0.5, 0.0))
    assert f == pytest.approx(math.tanh(1.2), abs=1e-15) and J == pytest.approx(0.0, abs=1e-15)


# ------------------------------------------------------------ the Jacobian J
def test_jacobian_matches_central_difference():
    eps = 1e-5
    for _ in range(200):
        h = RNG.uniform(-0.99, 0.99)
        p = RNG.normal(0, 1.5, 3)
        prm = [*RNG.uniform(-1.5, 1.5, 3), *RNG.normal(0, 0.3, 3)]
        _, J = oracle.cell(h, *p, prm)
        fp, _ = oracle.cell(h + eps, *p, prm)
        fm, _ = oracle.cell(h - eps, *p, prm)
        assert J == pytest.approx((fp - fm) / (2 * eps), abs=2e-9)


# ------------------------------------------------------- the sequential unroll
def test_sequential_matches_a_plain_python_unroll():
    """A second float64 path written from the cell's definition with the math
    module: z = sig(P_z + a_z h + b_z), r = sig(P_r + a_r h + b_r),
    c = tanh(P_c + a_c (r h) + b_c), h <- (1 - z) h + z c, from h = 0; and the
    Jacobian J = (1 - z) + z (1 - z) a_z (c - h) + z (1 - c^2) a_c (r + h r (1 - r) a_r)
    the chain rule gives, evaluated by hand at every step."""
    rng = np.random.default_rng(77)
    B, T, d_h = 2, 5, 3
    P = rng.normal(0, 1.5, size=(B, T, 3 * d_h))
    prm = _params(d_h, rng, scale=1.5, bias=0.7)
    H = oracle.sequential(P, prm)
    sig = lambda v: 1.0 / (1.0 + math.exp(-v))   # noqa: E731
    for b in range(B):
        for j in range(d_h):
            a_z, a_r, a_c = prm["a_z"][j], prm["a_r"][j], prm["a_c"][j]
            b_z, b_r, b_c = prm["b_z"][j], prm["b_r"][j], prm["b_c"][j]
            h = 0.0
            for t in range(T):
                pz, pr, pc = P[b, t, j], P[b, t, d_h + j], P[b, t, 2 * d_h + j]
                z = sig(pz + a_z * h + b_z)
                r = sig(pr + a_r * h + b_r)
                c = math.tanh(pc + a_c * (r * h) + b_c)
                J = (1 - z) + z * (1 - z) * a_z * (c - h) + z * (1 - c * c) * a_c * (r + h * r * (1 - r) * a_r)
                f, J_or = oracle.cell(h, pz, pr, pc, [a_z, a_r, a_c, b_z, b_r, b_c])
                h = (1 - z) * h + z * c
                assert abs(f - h) <= 1e-14
                assert abs(J_or - J) <= 1e-13
                assert abs(H[b, t, j] - h) <= 1e-14


def test_sequential_state_stays_in_unit_interval():
    w = syn.small_workload(B=3, T=500, d_h=12)
    P = syn.direct_preact(w) * 4.0
    H = oracle.sequential(P, syn.make_params(w))
    assert np.all(np.abs(H) < 1.0)


def test_sequential_pack_equals_independent_rows():
    lens = [5, 0, 17, 1, 30]
    cu = syn.cu_from_lengths(lens)
    N = int(cu[-1])
    P = RNG.normal(0, 1, (1, N, 9))
    prm = _params(3, RNG)
    H = oracle.sequential(P, prm, cu_seqlens=cu)
    for i in range(len(lens)):
        s0, s1 = cu[i], cu[i + 1]
        if s1 > s0:
            Hi = oracle.sequential(P[:, s0:s1], prm)
            np.testing.assert_array_equal(H[:, s0:s1], Hi)


# --------------------------------------------------------- the Newton solver
def test_newton_with_K_equal_T_is_the_unroll():
    """Iteration k makes step k exact, so K = T reproduces the unroll."""
    T, d_h = 24, 5
    P = RNG.normal(0, 1, (2, T, 3 * d_h))
    prm = _params(d_h, RNG, scale=1.5, bias=0.3)
    Hs = oracle.sequential(P, prm)
    Hn, rho = oracle.newton(P, prm, K=T)
    np.testing.assert_allclose(Hn, Hs, atol=1e-13)
    assert rho < 1e-13


@pytest.mark.parametrize("k", [1, 2, 3, 5])
def test_newton_first_k_steps_exact(k):
    T, d_h = 40, 4
    P = RNG.normal(0, 1, (1, T, 3 * d_h))
    prm = _params(d_h, RNG, scale=1.0)
    Hs = oracle.sequential(P, prm)
    Hn, _ = oracle.newton(P, prm, K=k)
    np.testing.assert_allclose(Hn[:, :k], Hs[:, :k], atol=1e-15)
    if k < 5:
        assert np.max(np.abs(Hn[:, k:] - Hs[:, k:])) > 1e-12   # not exact yet


def test_newton_exact_in_one_step_when_gates_ignore_state():
    """a_z = a_r = a_c = 0 makes f affine in h: one Newton step is exact and
    equals h_t = sum_s z_s c_s prod_{u=s+1..t} (1 - z_u)."""
    T, d_h = 50, 3
    P = RNG.normal(0, 1, (1, T, 3 * d_h))
    prm = {k: np.zeros(d_h) for k in oracle.GATE_ORDER}
    prm["b_z"] = np.array([0.1, -0.2, 0.3])
    Hn, rho = oracle.newton(P, prm, K=1)
    z = expit(P[0, :, :d_h] + prm["b_z"])
    c = np.tanh(P[0, :, 2 * d_h:])
    ref = np.zeros((T, d_h))
    for t in range(T):
        for s in range(t + 1):
            ref[t] += z[s] * c[s] * np.prod(1.0 - z[s + 1:t + 1], axis=0)
    np.testing.assert_allclose(Hn[0], ref, atol=1e-14)
    assert rho < 1e-14


def test_residual_of_unroll_is_zero_and_at_zero_state_is_closed_form():
    w = syn.small_workload(B=2, T=64, d_h=6)
    P = syn.direct_preact(w).astype(np.float64)
    prm = syn.make_params(w)
    Hs = oracle.sequential(P, prm)
    assert oracle.residual(P, prm, Hs) < 1e-15
    _, rho0 = oracle.newton(P, prm, K=0)
    d = w.d_h
    assert rho0 == pytest.approx(np.max(np.abs(expit(P[..., :d]) * np.tanh(P[..., 2 * d:]))),
                                 abs=1e-15)


def test_residual_counts_nan_as_infinite():
    P = RNG.normal(0, 1, (1, 8, 3))
    G = np.zeros((1, 8, 1))
    G[0, 3, 0] = np.nan
    assert oracle.residual(P, _params(1, RNG), G) == math.inf


def test_newton_pack_heads_match_per_segment_unroll():
    """J = 0 and zero shifted state at heads: with K = longest segment the
    packed Newton equals each segment's own unroll; with small K it equals
    Newton run on each segment alone."""
    lens = [7, 1, 0, 12, 3, 9]
    cu = syn.cu_from_lengths(lens)
    N, d_h = int(cu[-1]), 3
    P = RNG.normal(0, 1, (1, N, 3 * d_h))
    prm = _params(d_h, RNG)
    Hn, _ = oracle.newton(P, prm, K=max(lens), cu_seqlens=cu)
    Hs = oracle.sequential(P, prm, cu_seqlens=cu)
    np.testing.assert_allclose(Hn, Hs, atol=1e-14)
    H2, _ = oracle.newton(P, prm, K=2, cu_seqlens=cu)
    for i in range(len(lens)):
        s0, s1 = cu[i], cu[i + 1]
        if s1 > s0:
            Hi, _ = oracle.newton(P[:, s0:s1], prm, K=2)
            np.testing.assert_allclose(H2[:, s0:s1], Hi, atol=1e-15)


def test_threads_split_gives_identical_result():
    w = syn.small_workload(B=2, T=100, d_h=13)
    P = syn.direct_preact(w)
    prm = syn.make_params(w)
    a, ra = oracle.newton(P, prm, 3, threads=1)
    b, rb = oracle.newton(P, prm, 3, threads=4)
    np.testing.assert_array_equal(a, b)
    assert ra == rb


def test_columns_restriction_is_exact():
    w = syn.small_workload(B=2, T=80, d_h=10)
    P = syn.direct_preact(w)
    prm = syn.make_params(w)
    H, _ = oracle.newton(P, prm, 3)
    units = [0, 3, 9]
    Pc, prmc = oracle.columns(P, prm, units)
    Hc, _ = oracle.newton(Pc, prmc, 3)
    np.testing.assert_array_equal(H[..., units], Hc)


def test_input_projection_is_matmul():
    x = RNG.normal(size=(2, 5, 4))
    W = RNG.normal(size=(6, 4))
    P = oracle.input_projection(x, W)
    assert P.shape == (2, 5, 6)
    assert P[1, 3, 4] == pytest.approx(sum(x[1, 3, i] * W[4, i] for i in range(4)), abs=1e-14)


# ------------------------------------------------- Picard and warm-started Newton
@pytest.mark.parametrize("n", [1, 2, 5])
def test_picard_first_n_steps_exact_and_T_sweeps_is_unroll(n):
    """Sweep n makes step n exact (the shifted state of step n is exact after
    n - 1 sweeps); T sweeps reproduce the unroll."""
    T, d_h = 30, 4
    P = RNG.normal(0, 1, (2, T, 3 * d_h))
    prm = _params(d_h, RNG)
    Hs = oracle.sequential(P, prm)
    G = oracle.picard(P, prm, n)
    np.testing.assert_allclose(G[:, :n], Hs[:, :n], atol=1e-15)
    assert np.max(np.abs(G[:, n:] - Hs[:, n:])) > 1e-12
    np.testing.assert_allclose(oracle.picard(P, prm, T), Hs, atol=1e-15)


def test_picard_fixed_point_is_the_unroll():
    w = syn.small_workload(B=2, T=200, d_h=8, seed=8)
    P = syn.direct_preact(w).astype(np.float64)
    prm = syn.make_params(w)
    Hs = oracle.sequential(P, prm)
    # one more sweep applied to the unroll changes nothing: f(h_{t-1}) = h_t
    G = oracle.picard(P, prm, 1)  # from zero: first step only
    assert np.allclose(G[:, 0], Hs[:, 0], atol=1e-15)
    Hn, rho = oracle.newton_init(P, prm, 3, Hs)   # Newton at the fixed point stays there
    np.testing.assert_allclose(Hn, Hs, atol=1e-15)
    assert rho < 1e-15


def test_newton_init_from_zero_equals_newton_and_warm_start_exactness():
    T, d_h = 40, 3
    P = RNG.normal(0, 1, (1, T, 3 * d_h))
    prm = _params(d_h, RNG)
    a, ra = oracle.newton(P, prm, 3)
    b, rb = oracle.newton_init(P, prm, 3, np.zeros((1, T, d_h)))
    np.testing.assert_array_equal(a, b)
    assert ra == rb
    Hs = oracle.sequential(P, prm)
    G = oracle.picard(P, prm, 2)            # steps 1..2 exact
    H, _ = oracle.newton_init(P, prm, 3, G)  # each Newton iteration adds one exact step
    np.testing.assert_allclose(H[:, :5], Hs[:, :5], atol=1e-15)
    cu = syn.cu_from_lengths([9, 0, 20, 11])
    Gp = oracle.picard(P, prm, 40, cu_seqlens=cu)
    np.testing.assert_allclose(Gp, oracle.sequential(P, prm, cu_seqlens=cu), atol=1e-15)


def test_decode_steps_repeated_are_the_unroll():
    """T decode steps with the state carried reproduce the unroll of the same
    preactivations (each slot a row)."""
    w = syn.small_workload(B=3, T=20, d_h=5, seed=60)
    P = syn.direct_preact(w).astype(np.float64)
    prm = syn.make_params(w)
    Hs = oracle.sequential(P, prm)
    h = None
    for t in range(w.T):
        h = oracle.decode_step(P[:, t], prm, h)
        np.testing.assert_allclose(h, Hs[:, t], atol=1e-15)


# --------------------------------------------------------------- the adjoint
def _loss(P, prm, wts, cu=None):
    return float(np.sum(wts * oracle.sequential(P, prm, cu_seqlens=cu)))


@pytest.mark.parametrize("ragged", [False, True])
def test_backward_matches_finite_differences(ragged):
    """dL/dP and dL/d(params) of L = sum(w * H_unroll) against central
    differences of the unroll (a path that never calls the adjoint)."""
    rng = np.random.default_rng(70)
    if ragged:
        cu = syn.cu_from_lengths([6, 0, 9, 1, 4])
        B, T = 1, int(cu[-1])
    else:
        cu, B, T = None, 2, 14
    d_h = 3
    P = rng.normal(0, 1, (B, T, 3 * d_h))
    prm = oracle.pack_params(_params(d_h, rng, scale=1.2, bias=0.4))
    wts = rng.normal(size=(B, T, d_h))
    H = oracle.sequential(P, prm, cu_seqlens=cu)
    gP, gprm = oracle.backward(P, prm, H, wts, cu_seqlens=cu)
    eps = 1e-6
    for idx in [(0, 0, 0), (0, T - 1, 3 * d_h - 1), (B - 1, T // 2, d_h + 1), (0, 3, 2 * d_h),
                (B - 1, 1, 4)]:
        Pp, Pm = P.copy(), P.copy()
        Pp[idx] += eps
        Pm[idx] -= eps
        fd = (_loss(Pp, prm, wts, cu) - _loss(Pm, prm, wts, cu)) / (2 * eps)
        assert gP[idx] == pytest.approx(fd, abs=1e-7)
    for g in range(6):
        for j in range(d_h):
            pp, pm = prm.copy(), prm.copy()
            pp[g, j] += eps
            pm[g, j] -= eps
            fd = (_loss(P, pp, wts, cu) - _loss(P, pm, wts, cu)) / (2 * eps)
            assert gprm[g, j] == pytest.approx(fd, abs=1e-7)
