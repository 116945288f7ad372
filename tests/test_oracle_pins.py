"""Pins of the fp64 oracle against what the pages and the mathematics fix.

Each test names the passage it follows.  None of them re-types the oracle's
own loop: they use printed values (tests/golden), closed forms, the dense
exact Kalman filter on cases where the diagonal projection is exact,
special-case reductions (Delta rule / KDA) and brute-force products of the
pages' Moebius matrices.
"""
import numpy as np
import pytest

import oracle
from oracle import dense


def _scalar_inputs(T, k=1.0, q=1.0, v=1.0, r=1.0, log_alpha=0.0, omega=0.0):
    full = lambda x, shp: np.full(shp, x, dtype=np.float64)
    return dict(
        q=full(q, (1, T, 1, 1)), k=full(k, (1, T, 1, 1)), v=full(v, (1, T, 1, 1)),
        log_alpha=full(log_alpha, (1, T, 1, 1)), r=full(r, (1, T, 1)),
    )


# ---------------------------------------------------------------- printed values
@pytest.mark.parametrize("variant", ["diag", "iso"])
def test_gain_scalar_example(golden, variant):
    """KDN paper Sec. 3.2 teaching example: k = r = 1, prior 9 -> 0.9, 0.1 -> 0.0909."""
    g = golden("gain_scalar_example")
    for p0, key in ((9.0, "kappa_pred_var_9"), (0.1, "kappa_pred_var_0p1")):
        x = _scalar_inputs(1)
        om = np.zeros((1, 1, 1, 1)) if variant == "diag" else np.zeros((1, 1, 1))
        pshape = (1, 1, 1) if variant == "diag" else (1, 1)
        out = oracle.forward(variant, **x, omega=om, p0=np.full(pshape, p0), mu=1.0,
                             want_kappa=True)
        val, tol = g[key]
        assert abs(out["kappa"][0, 0, 0, 0] - val) <= tol
        # S_0 = 0, v = 1: the write is kappa itself and the post-write read sees it
        assert out["o"][0, 0, 0, 0] == pytest.approx(out["kappa"][0, 0, 0, 0], abs=1e-15)


@pytest.mark.parametrize("variant", ["diag", "iso"])
def test_repeated_observation_variance(variant):
    """KDN paper Sec. 3.2 example: D = 1, Omega = 0, p_0 = 1, mu = 1 -> p_n = 1/(n+1)."""
    for n in (1, 2, 5, 17, 50):
        x = _scalar_inputs(n)
        om = np.zeros((1, n, 1, 1)) if variant == "diag" else np.zeros((1, n, 1))
        out = oracle.forward(variant, **x, omega=om, mu=1.0)
        assert out["p_T"].ravel()[0] == pytest.approx(1.0 / (n + 1), rel=1e-14)


def test_steady_state_gain(golden):
    """Bayesian Layer App. E.1 Eq. 42: r = omega = 0.05 -> gain 0.618034 and
    predictive variance x_inf = (w + sqrt(w^2 + 4 r w)) / 2."""
    T = 400
    x = _scalar_inputs(T, r=0.05)
    out = oracle.forward("diag", **x, omega=np.full((1, T, 1, 1), 0.05), mu=1.0,
                         want_kappa=True, want_phat=True)
    val, tol = golden("steady_state_gain")["g_inf_r0p05_l0p05"]
    assert abs(out["kappa"][0, -1, 0, 0] - val) <= tol
    w = r = 0.05
    x_inf = (w + np.sqrt(w * w + 4 * r * w)) / 2
    assert out["phat"][0, -1, 0, 0] == pytest.approx(x_inf, rel=1e-12)
    assert out["kappa"][0, -1, 0, 0] == pytest.approx(x_inf / (r + x_inf), rel=1e-12)


@pytest.mark.parametrize("variant", ["diag", "iso"])
def test_information_scaling_uniform_energy(golden, variant):
    """KDN paper App. B Eq. 60-65: m = 128 uniform-energy key, p = r = 1:
    projected directional variance 0.9922 at mu = 1, 0.5 at mu = 128; exact 0.5."""
    g = golden("uniform_energy_scaling")
    m = 128
    rng = np.random.default_rng(5)
    k = rng.choice([-1.0, 1.0], size=m) / np.sqrt(m)
    x = dict(q=k.reshape(1, 1, 1, m), k=k.reshape(1, 1, 1, m), v=np.ones((1, 1, 1, 1)),
             log_alpha=np.zeros((1, 1, 1, m)), r=np.ones((1, 1, 1)))
    om = np.zeros((1, 1, 1, m)) if variant == "diag" else np.zeros((1, 1, 1))
    for mu, key in ((1.0, "v_proj_m128_mu1"), (128.0, "v_proj_m128_mu128")):
        out = oracle.forward(variant, **x, omega=om, mu=mu)
        pT = out["p_T"].ravel()
        pvec = pT if variant == "diag" else np.full(m, pT[0])
        v_proj = float(np.sum(k * k * pvec))
        val, tol = g[key]
        assert abs(v_proj - val) <= tol
        assert v_proj == pytest.approx(m / (m + mu), rel=1e-12)
    ex = dense.dense_kalman(k[None], np.ones((1, 1)), k[None], np.ones(1), np.zeros((m, 1)), np.eye(m))
    val, tol = g["v_exact_m128"]
    assert abs(float(k @ ex["P_T"] @ k) - val) <= tol


def test_collision_trajectory(golden):
    """Bayesian Layer App. E.3-E.4 deterministic collision: pins dense_kalman."""
    g = golden("collision_trajectory")
    D, m, rho = 16, 6, 0.92
    keys = np.zeros((6, D))
    keys[0, 0] = 1.0
    keys[1, 0], keys[1, 1] = rho, np.sqrt(1 - rho ** 2)
    for i in range(2, 6):
        keys[i, i] = 1.0
    sched = list(range(6)) * 2 + [1] * 40 + [0] * 60
    K, V = keys[sched], np.eye(6)[sched]
    T = len(sched)
    r = np.full(T, 0.05)
    Q = np.tile(keys[1], (T, 1))
    out = dense.dense_kalman(K, V, Q, r, np.zeros((D, m)), 3 * np.eye(D),
                             Omega=np.full((T, D), 0.05))
    y = out["o"]
    pAB = np.exp(y[:, 1]) / (np.exp(y[:, 0]) + np.exp(y[:, 1]))
    gain = out["z"] / (r + out["z"])
    for key, got in (("bl_pAB_step52", pAB[51]), ("bl_pAB_step112", pAB[111]),
                     ("bl_gain_step53", gain[52]), ("bl_gain_step112", gain[111])):
        val, tol = g[key]
        assert abs(got - val) <= tol, (key, got, val)
    # reset / Delta control: the covariance is reset to l^2 I before every write.
    # Its gains come from the filter with a zero covariance transition (only the
    # gains of that run are used; its mean is wiped by D = 0):
    ex = dense.dense_kalman(K, V, Q, r, np.zeros((D, m)), np.zeros((D, D)),
                            D=np.zeros((T, D)), Omega=np.full((T, D), 0.05))
    # the mean of the reset control is the fixed-gain Delta rule:
    S = np.zeros((D, m))
    for t in range(T):
        S = S + 0.5 * np.outer(K[t], V[t] - S.T @ K[t])
    yB = S.T @ keys[1]
    val, tol = g["delta_pAB_step112"]
    assert abs(np.exp(yB[1]) / (np.exp(yB[0]) + np.exp(yB[1])) - val) <= tol
    # and the reset filter's own gain is exactly 0.5 each step
    assert np.allclose(ex["z"] / (r + ex["z"]), 0.5, atol=1e-15)


def test_direction_example(golden):
    """Bayesian Layer Sec. 2.4: P_bar = diag(0.05, 2), k = (0.8, 0.6) -> u = P_bar k = (0.04, 1.2)."""
    g = golden("direction_example")
    k = np.array([[0.8, 0.6]])
    out = dense.dense_kalman(k, np.zeros((1, 1)), k, np.ones(1), np.zeros((2, 1)),
                             np.diag([0.05, 2.0]))
    u = out["kappa"][0] * (1.0 + out["z"][0])
    for i in range(2):
        val, tol = g[f"u_{i}"]
        assert abs(u[i] - val) <= tol


# ---------------------------------------------------------------- closed forms
def test_no_decay_filter_is_weighted_ridge():
    """Preconditioned DeltaNet Eq. 1-5 / Gated KalmaNet ridge view: with D = I and
    Omega = 0 the exact filter's mean is the weighted ridge solution."""
    rng = np.random.default_rng(1)
    T, dk, dv, p0 = 23, 5, 3, 0.7
    K = rng.standard_normal((T, dk))
    V = rng.standard_normal((T, dv))
    r = 0.1 + rng.random(T)
    out = dense.dense_kalman(K, V, K, r, np.zeros((dk, dv)), p0 * np.eye(dk))
    ref = dense.ridge_closed_form(K, V, r, p0 * np.eye(dk))
    np.testing.assert_allclose(out["S_T"], ref, rtol=1e-10, atol=1e-12)
    # brute force: minimise sum_t (1/r_t)||S^T k_t - v_t||^2 + (1/p0)||S||^2 by normal equations
    A = np.vstack([K / np.sqrt(r)[:, None], np.eye(dk) / np.sqrt(p0)])
    Bm = np.vstack([V / np.sqrt(r)[:, None], np.zeros((dk, dv))])
    lsq = np.linalg.lstsq(A, Bm, rcond=None)[0]
    np.testing.assert_allclose(ref, lsq, rtol=1e-9, atol=1e-12)


def test_diag_one_hot_no_decay_is_diagonal_ridge():
    """Diagonal KDN with one-hot keys, mu = 1, no decay or process noise equals
    the ridge solution, which for axis-aligned keys is a per-row weighted mean."""
    rng = np.random.default_rng(2)
    B, T, H, dk, dv, p0 = 2, 31, 3, 6, 4, 1.3
    j = rng.integers(0, dk, size=(B, T, H))
    c = rng.uniform(0.5, 1.5, size=(B, T, H)) * rng.choice([-1, 1], size=(B, T, H))
    k = np.zeros((B, T, H, dk))
    np.put_along_axis(k, j[..., None], c[..., None], axis=-1)
    v = rng.standard_normal((B, T, H, dv))
    r = 0.05 + rng.random((B, T, H))
    out = oracle.forward("diag", rng.standard_normal((B, T, H, dk)), k, v,
                         np.zeros((B, T, H, dk)), np.zeros((B, T, H, dk)), r,
                         p0=np.full((B, H, dk), p0), mu=1.0)
    for b in range(B):
        for h in range(H):
            num = np.zeros((dk, dv))
            den = np.full(dk, 1.0 / p0)
            for t in range(T):
                num[j[b, t, h]] += c[b, t, h] * v[b, t, h] / r[b, t, h]
                den[j[b, t, h]] += c[b, t, h] ** 2 / r[b, t, h]
            np.testing.assert_allclose(out["S_T"][b, h], num / den[:, None], rtol=1e-11, atol=1e-13)
            np.testing.assert_allclose(out["p_T"][b, h], 1.0 / den, rtol=1e-12)


# ------------------------------------------------------- exact-filter brute force
def _random_case(rng, B, T, H, dk, dv):
    return dict(
        q=rng.standard_normal((B, T, H, dk)),
        v=rng.standard_normal((B, T, H, dv)),
        log_alpha=-rng.uniform(0.01, 0.5, size=(B, T, H, dk)),
        omega=rng.uniform(0.01, 0.3, size=(B, T, H, dk)),
        r=0.05 + rng.random((B, T, H)),
    )


def test_single_step_reverse_kl_projection():
    """KDN paper Sec. 4.1 Eq. 28-30 (App. A.2): one step from a diagonal prior,
    mu = 1: the mean equals the dense exact posterior mean and
    p_i = 1 / (P*^{-1})_ii (not the diagonal of P*)."""
    rng = np.random.default_rng(3)
    B, H, dk, dv = 2, 3, 7, 5
    x = _random_case(rng, B, 1, H, dk, dv)
    k = rng.standard_normal((B, 1, H, dk))
    S0 = rng.standard_normal((B, H, dk, dv))
    p0 = rng.uniform(0.2, 2.0, size=(B, H, dk))
    out = oracle.forward("diag", x["q"], k, x["v"], x["log_alpha"], x["omega"], x["r"],
                         S0=S0, p0=p0, mu=1.0)
    for b in range(B):
        for h in range(H):
            a = np.exp(x["log_alpha"][b, 0, h])
            ex = dense.dense_kalman(k[b, :, h], x["v"][b, :, h], x["q"][b, :, h], x["r"][b, :, h],
                                    S0[b, h], np.diag(p0[b, h]), D=a[None],
                                    Omega=x["omega"][b, :, h])
            np.testing.assert_allclose(out["S_T"][b, h], ex["S_T"], rtol=1e-12, atol=1e-13)
            np.testing.assert_allclose(out["o"][b, 0, h], ex["o"][0], rtol=1e-12, atol=1e-13)
            prec = np.linalg.inv(ex["P_T"])
            np.testing.assert_allclose(out["p_T"][b, h], 1.0 / np.diag(prec), rtol=1e-11)
            assert not np.allclose(out["p_T"][b, h], np.diag(ex["P_T"]), rtol=1e-6)


def test_one_hot_trajectory_matches_dense_kalman():
    """Axis-aligned keys keep the exact posterior diagonal, so Diagonal KDN with
    mu = 1 equals the dense exact filter at every token (KDN paper Sec. 4.1,
    App. A.2, applied along a whole trajectory)."""
    rng = np.random.default_rng(4)
    B, T, H, dk, dv = 2, 40, 3, 6, 4
    x = _random_case(rng, B, T, H, dk, dv)
    j = rng.integers(0, dk, size=(B, T, H))
    k = np.zeros((B, T, H, dk))
    np.put_along_axis(k, j[..., None], rng.uniform(0.3, 1.5, size=(B, T, H, 1)), axis=-1)
    S0 = rng.standard_normal((B, H, dk, dv))
    p0 = rng.uniform(0.2, 2.0, size=(B, H, dk))
    out = oracle.forward("diag", x["q"], k, x["v"], x["log_alpha"], x["omega"], x["r"],
                         S0=S0, p0=p0, mu=1.0, want_kappa=True)
    for b in range(B):
        for h in range(H):
            ex = dense.dense_kalman(k[b, :, h], x["v"][b, :, h], x["q"][b, :, h], x["r"][b, :, h],
                                    S0[b, h], np.diag(p0[b, h]),
                                    D=np.exp(x["log_alpha"][b, :, h]), Omega=x["omega"][b, :, h])
            np.testing.assert_allclose(out["o"][b, :, h], ex["o"], rtol=1e-10, atol=1e-12)
            np.testing.assert_allclose(out["kappa"][b, :, h], ex["kappa"], rtol=1e-10, atol=1e-14)
            np.testing.assert_allclose(out["S_T"][b, h], ex["S_T"], rtol=1e-10, atol=1e-12)
            np.testing.assert_allclose(out["p_T"][b, h], np.diag(ex["P_T"]), rtol=1e-10)
            off = ex["P_T"] - np.diag(np.diag(ex["P_T"]))
            assert np.max(np.abs(off)) == 0.0


# ------------------------------------------------------------- reductions
def _kda_loop(q, k, v, log_alpha, beta, S0):
    """Independent KDA recurrence S = D S + beta k (v - (D S)^T k)^T, o = S^T q
    (KDN paper Sec. 2 / Sec. 3.3 Eq. 18-20, Bayesian Layer Prop. 2)."""
    T = k.shape[0]
    S = S0.copy()
    o = np.zeros((T, v.shape[1]))
    for t in range(T):
        DS = np.exp(log_alpha[t])[:, None] * S
        S = DS + beta[t] * np.outer(k[t], v[t] - DS.T @ k[t])
        o[t] = S.T @ q[t]
    return o, S


@pytest.mark.parametrize("variant", ["diag", "iso"])
def test_delta_rule_reduction(variant):
    """With the information update switched off (mu = 0) and omega chosen so that
    the predictive variance equals a token-wise lambda_t (an isotropic surrogate,
    no tracking), the KDN write is the KDA / gated delta rule with
    beta_t = lambda_t / (r_t + lambda_t ||k_t||^2) (KDN paper Sec. 3.3 Eq. 18-20)."""
    rng = np.random.default_rng(6)
    B, T, H, dk, dv = 2, 30, 2, 5, 3
    x = _random_case(rng, B, T, H, dk, dv)
    k = rng.standard_normal((B, T, H, dk))
    lam = rng.uniform(0.2, 3.0, size=(B, T, H))
    a2 = np.exp(2 * x["log_alpha"])
    lam_prev = np.concatenate([np.ones((B, 1, H)), lam[:, :-1]], axis=1)   # p_0 = 1
    if variant == "diag":
        om = lam[..., None] - a2 * lam_prev[..., None]
    else:
        om = lam - a2.mean(-1) * lam_prev
    S0 = rng.standard_normal((B, H, dk, dv))
    out = oracle.forward(variant, x["q"], k, x["v"], x["log_alpha"], om, x["r"], S0=S0, mu=0.0)
    for b in range(B):
        for h in range(H):
            kk = k[b, :, h]
            beta = lam[b, :, h] / (x["r"][b, :, h] + lam[b, :, h] * np.sum(kk * kk, -1))
            o, S = _kda_loop(x["q"][b, :, h], kk, x["v"][b, :, h], x["log_alpha"][b, :, h], beta, S0[b, h])
            np.testing.assert_allclose(out["o"][b, :, h], o, rtol=1e-10, atol=1e-12)
            np.testing.assert_allclose(out["S_T"][b, h], S, rtol=1e-10, atol=1e-12)


def test_diag_equals_iso_on_uniform_cases():
    """Diagonal and Isotropic KDN coincide (KDN paper Sec. 4.1 vs 4.2 / App. C):
    (i) uniform decay, noise and prior with uniform-energy keys k_i = +-1/sqrt(d_k), any mu;
    (ii) uniform decay, noise and prior with mu = 0, any keys."""
    rng = np.random.default_rng(7)
    B, T, H, dk, dv = 2, 25, 2, 8, 3
    la_tok = -rng.uniform(0.01, 0.3, size=(B, T, H, 1))
    la = np.repeat(la_tok, dk, axis=-1)
    om_tok = rng.uniform(0.01, 0.2, size=(B, T, H))
    om_diag = np.repeat(om_tok[..., None], dk, axis=-1)
    q = rng.standard_normal((B, T, H, dk))
    v = rng.standard_normal((B, T, H, dv))
    r = 0.05 + rng.random((B, T, H))
    p0 = rng.uniform(0.5, 2.0, size=(B, H))
    p0d = np.repeat(p0[..., None], dk, axis=-1)
    k_uniform = rng.choice([-1.0, 1.0], size=(B, T, H, dk)) / np.sqrt(dk)
    k_any = rng.standard_normal((B, T, H, dk))
    for k, mu in ((k_uniform, 3.0), (k_uniform, float(dk)), (k_any, 0.0)):
        d = oracle.forward("diag", q, k, v, la, om_diag, r, p0=p0d, mu=mu)
        i = oracle.forward("iso", q, k, v, la, om_tok, r, p0=p0, mu=mu)
        np.testing.assert_allclose(d["o"], i["o"], rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(d["S_T"], i["S_T"], rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(d["p_T"], np.repeat(i["p_T"][..., None], dk, -1), rtol=1e-12)


# ------------------------------------------------------------- Moebius scan
def test_mobius_bracketing_is_associative():
    """KDN paper Eq. 32-37: the ordered product of the 2x2 matrices does not
    depend on the bracketing (chunking) and equals sequential iteration."""
    rng = np.random.default_rng(8)
    T, d = 57, 4
    M = dense.mobius_matrices(-rng.uniform(0.01, 0.3, (T, d)), rng.uniform(0.01, 0.2, (T, d)),
                              rng.standard_normal((T, d)), 0.1 + rng.random(T), mu=3.0)
    seq = np.broadcast_to(np.eye(2), (d, 2, 2)).copy()
    for t in range(T):
        seq = np.einsum("dij,djk->dik", M[t], seq)
    for trial in range(6):
        split = (lambda lo, hi: int(rng.integers(lo + 1, hi)))
        P = dense.mobius_product(M, 0, T, split=split)
        np.testing.assert_allclose(P, seq, rtol=1e-12)
    # chunked: summaries of 8-token chunks, then the carry
    carry = np.broadcast_to(np.eye(2), (d, 2, 2)).copy()
    for lo in range(0, T, 8):
        carry = np.einsum("dij,djk->dik", dense.mobius_product(M, lo, min(T, lo + 8)), carry)
    np.testing.assert_allclose(carry, seq, rtol=1e-12)


@pytest.mark.parametrize("variant", ["diag", "iso"])
def test_mobius_scan_matches_oracle_uncertainty(variant):
    """The oracle's uncertainty states equal the pages' Moebius form applied to
    [p_0; 1]: p_{t-1} from the product of M_1..M_{t-1}, then
    p_hat_t = a^2 p_{t-1} + omega_t (KDN paper Eq. 32-37; App. C for the scalar case)."""
    rng = np.random.default_rng(9)
    B, T, H, dk, dv = 1, 33, 2, 6, 2
    x = _random_case(rng, B, T, H, dk, dv)
    k = rng.standard_normal((B, T, H, dk))
    mu = 2.5
    om = x["omega"] if variant == "diag" else x["omega"][..., 0]
    p0 = rng.uniform(0.3, 2.0, size=(B, H, dk) if variant == "diag" else (B, H))
    out = oracle.forward(variant, x["q"], k, x["v"], x["log_alpha"], om, x["r"], p0=p0, mu=mu,
                         want_phat=True)
    for h in range(H):
        if variant == "diag":
            M = dense.mobius_matrices(x["log_alpha"][0, :, h], om[0, :, h], k[0, :, h], x["r"][0, :, h], mu)
            pinit = p0[0, h]
            a2 = np.exp(2 * x["log_alpha"][0, :, h])
            omt = om[0, :, h]
        else:
            # scalar: a_bar = mean a^2 (trace projection), u = mu ||k||^2 / (d_k r)
            a_bar = np.exp(2 * x["log_alpha"][0, :, h]).mean(-1)
            kn = np.sqrt(np.sum(k[0, :, h] ** 2, -1) / dk)
            M = dense.mobius_matrices(0.5 * np.log(a_bar)[:, None], om[0, :, h][:, None], kn[:, None],
                                      x["r"][0, :, h], mu)
            pinit = np.array([p0[0, h]])
            a2 = a_bar[:, None]
            omt = om[0, :, h][:, None]
        for t in range(T):
            p_prev = dense.mobius_apply(dense.mobius_product(M, 0, t), pinit)
            phat = a2[t] * p_prev + omt[t]
            got = out["phat"][0, t, h] if variant == "diag" else np.array([out["phat"][0, t, h]])
            np.testing.assert_allclose(got, phat, rtol=1e-12)
        pT = dense.mobius_apply(dense.mobius_product(M, 0, T), pinit)
        np.testing.assert_allclose(np.ravel(out["p_T"][0, h]), pT, rtol=1e-12)


# ------------------------------------------------------------- invariants
@pytest.mark.parametrize("variant", ["diag", "iso"])
def test_state_continuation_step_and_invariants(variant):
    """The recurrent state is the checkpoint (KDN paper Sec. 5.1: the scan and
    token-by-token inference are the same recurrence): split runs, step loops and
    the full run agree; 0 <= beta_eff = k^T kappa < 1 (App. B Eq. 58-61);
    0 < p <= p_hat."""
    rng = np.random.default_rng(10)
    B, T, H, dk, dv = 2, 24, 2, 5, 4
    x = _random_case(rng, B, T, H, dk, dv)
    k = rng.standard_normal((B, T, H, dk))
    om = x["omega"] if variant == "diag" else x["omega"][..., 0]
    full = oracle.forward(variant, x["q"], k, x["v"], x["log_alpha"], om, x["r"],
                          want_kappa=True, want_phat=True)
    T1 = 9
    sl = lambda a, s: a[:, s]
    a = oracle.forward(variant, sl(x["q"], slice(0, T1)), sl(k, slice(0, T1)), sl(x["v"], slice(0, T1)),
                       sl(x["log_alpha"], slice(0, T1)), sl(om, slice(0, T1)), sl(x["r"], slice(0, T1)))
    b = oracle.forward(variant, sl(x["q"], slice(T1, T)), sl(k, slice(T1, T)), sl(x["v"], slice(T1, T)),
                       sl(x["log_alpha"], slice(T1, T)), sl(om, slice(T1, T)), sl(x["r"], slice(T1, T)),
                       S0=a["S_T"], p0=a["p_T"])
    np.testing.assert_allclose(np.concatenate([a["o"], b["o"]], 1), full["o"], rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(b["S_T"], full["S_T"], rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(b["p_T"], full["p_T"], rtol=1e-13)
    S = np.zeros((B, H, dk, dv))
    p = np.ones((B, H, dk) if variant == "diag" else (B, H))
    for t in range(T):
        o, S, p = oracle.step(variant, x["q"][:, t], k[:, t], x["v"][:, t], x["log_alpha"][:, t],
                              om[:, t], x["r"][:, t], S, p)
        np.testing.assert_allclose(o, full["o"][:, t], rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(S, full["S_T"], rtol=1e-13, atol=1e-14)
    beta_eff = np.sum(k * full["kappa"], -1)
    assert np.all(beta_eff >= 0.0) and np.all(beta_eff < 1.0)
    assert np.all(full["p_T"] > 0.0)
    assert np.all(full["phat"] > 0.0)


def test_information_scale_leaves_current_write_unchanged():
    """KDN paper App. B: changing mu at token t (same predictive prior) leaves that
    token's write and output unchanged; only later gains move."""
    rng = np.random.default_rng(11)
    B, T, H, dk, dv = 1, 6, 1, 4, 3
    x = _random_case(rng, B, T, H, dk, dv)
    k = rng.standard_normal((B, T, H, dk))
    o1 = oracle.forward("diag", x["q"], k, x["v"], x["log_alpha"], x["omega"], x["r"], mu=1.0,
                        want_kappa=True)
    o2 = oracle.forward("diag", x["q"], k, x["v"], x["log_alpha"], x["omega"], x["r"], mu=9.0,
                        want_kappa=True)
    np.testing.assert_allclose(o1["kappa"][:, 0], o2["kappa"][:, 0], rtol=1e-15)
    np.testing.assert_allclose(o1["o"][:, 0], o2["o"][:, 0], rtol=1e-15)
    assert not np.allclose(o1["kappa"][:, 1], o2["kappa"][:, 1], rtol=1e-6)
    # later writes are weaker with larger mu (more protection)
    be1 = np.sum(k * o1["kappa"], -1)[:, 1:]
    be2 = np.sum(k * o2["kappa"], -1)[:, 1:]
    assert np.all(be2 < be1)
