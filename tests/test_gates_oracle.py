"""Pins of the gate activations and the effective write strength (oracle/gates.py).

Gates: KDN reading notes Sec. 5.1 -- alpha = sigma(a), omega = softplus(w),
r = r_min + softplus(rho), r_min = 0.01.  The pins use closed forms at zero,
the symmetries sigma(a) + sigma(-a) = 1 and softplus(x) - softplus(-x) = x,
scipy's logistic routines (an implementation independent of the oracle's
logaddexp), and the asymptotes.  Every check is a function of the gate
implementation, and planted mistakes (a flipped sign, r_min dropped or moved,
another activation) are shown to fail at least one of them.

Effective write strength: reading notes Sec. 3.2 (App. B, Eq. 58-61),
beta_eff = k^T kappa = z / (r + z), z = k^T P_hat k.  Pinned by the worked
one-dimensional example of Sec. 3.2 (golden file), the repeated-observation
closed form, and the identity with z formed from the recurrence's predictive
variances.
"""
import math

import numpy as np
import pytest

from oracle import gates, recurrence

special = pytest.importorskip("scipy.special")

LN2 = math.log(2.0)


def _gate_pin_failures(gv):
    """Names of the pins that the gate implementation ``gv`` violates."""
    bad = []
    g0 = gv(np.zeros(3), np.zeros(3), np.zeros(3), 0.01)
    if not np.allclose(g0["log_alpha"], -LN2, rtol=0, atol=1e-15):
        bad.append("log_alpha(0) = -ln 2")
    if not np.allclose(g0["omega"], LN2, rtol=0, atol=1e-15):
        bad.append("omega(0) = ln 2")
    if not np.allclose(g0["r"], 0.01 + LN2, rtol=0, atol=1e-15):
        bad.append("r(0) = r_min + ln 2")
    x = np.linspace(-30.0, 30.0, 241)
    g = gv(x, x, x, 0.01)
    if not np.allclose(g["log_alpha"], special.log_expit(x), rtol=1e-13, atol=1e-300):
        bad.append("log_alpha = log_expit")
    if not np.allclose(np.exp(g["log_alpha"]), special.expit(x), rtol=1e-13, atol=0):
        bad.append("alpha = expit")
    sp = -special.log_expit(-x)   # softplus(x) = -log sigma(-x)
    if not np.allclose(g["omega"], sp, rtol=1e-13, atol=1e-300):
        bad.append("omega = softplus")
    if not np.allclose(g["r"], 0.01 + sp, rtol=1e-13, atol=0):
        bad.append("r = r_min + softplus")
    gm = gv(-x, -x, -x, 0.01)
    if not np.allclose(np.exp(g["log_alpha"]) + np.exp(gm["log_alpha"]), 1.0, rtol=0, atol=1e-15):
        bad.append("sigma(a) + sigma(-a) = 1")
    if not np.allclose(g["omega"] - gm["omega"], x, rtol=0, atol=1e-13):
        bad.append("softplus(x) - softplus(-x) = x")
    # asymptotes: softplus(50) = 50 + e^-50, log sigma(-50) = -50 - e^-50, r -> r_min
    big = gv(np.array([50.0, -50.0]), np.array([50.0, -50.0]), np.array([-60.0, -20.0]), 0.25)
    if abs(big["omega"][0] - 50.0) > 1e-13 or abs(big["omega"][1] - math.exp(-50.0)) > 1e-30:
        bad.append("softplus asymptotes")
    if abs(big["log_alpha"][1] + 50.0) > 1e-13 or abs(big["log_alpha"][0] + math.exp(-50.0)) > 1e-30:
        bad.append("log sigma asymptotes")
    if abs(big["r"][0] - 0.25) > 1e-20 or abs((big["r"][1] - 0.25) / math.exp(-20.0) - 1.0) > 1e-6:
        bad.append("r -> r_min + e^rho")
    return bad


def test_gate_values_pins():
    """KDN reading notes Sec. 5.1: the three gate branches."""
    assert _gate_pin_failures(gates.gate_values) == []


def _sp(x):
    return np.logaddexp(0.0, np.asarray(x, dtype=np.float64))


MUTANTS = {
    "log sigma(-a)": lambda a, w, p, rm: {"log_alpha": -_sp(a), "omega": _sp(w), "r": rm + _sp(p)},
    "log alpha^2": lambda a, w, p, rm: {"log_alpha": -2.0 * _sp(-a), "omega": _sp(w), "r": rm + _sp(p)},
    "omega + r_min": lambda a, w, p, rm: {"log_alpha": -_sp(-a), "omega": rm + _sp(w), "r": rm + _sp(p)},
    "r without r_min": lambda a, w, p, rm: {"log_alpha": -_sp(-a), "omega": _sp(w), "r": _sp(p)},
    "omega = exp(w)": lambda a, w, p, rm: {"log_alpha": -_sp(-a), "omega": np.exp(w), "r": rm + _sp(p)},
    "alpha = tanh": lambda a, w, p, rm: {"log_alpha": np.log(np.abs(np.tanh(a)) + 1e-300), "omega": _sp(w),
                                         "r": rm + _sp(p)},
    "r = r_min * softplus": lambda a, w, p, rm: {"log_alpha": -_sp(-a), "omega": _sp(w), "r": rm * _sp(p)},
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_gate_pins_reject_planted_mistakes(name):
    assert _gate_pin_failures(MUTANTS[name]), name


def _scalar(T, p0, variant, r=1.0):
    """One-dimensional sequence: k = q = v = 1, alpha = 1 (logit +inf), omega = 0
    (logit -inf), r_t = r (logit chosen so that r_min + softplus(rho) = r)."""
    full = lambda x, shp: np.full(shp, x, dtype=np.float64)
    rho = math.log(math.expm1(r - gates.R_MIN))
    om = full(-np.inf, (1, T, 1, 1) if variant == "diag" else (1, T, 1))
    pshape = (1, 1, 1) if variant == "diag" else (1, 1)
    return dict(q=full(1.0, (1, T, 1, 1)), k=full(1.0, (1, T, 1, 1)), v=full(1.0, (1, T, 1, 1)),
                alpha_logit=full(np.inf, (1, T, 1, 1)), omega_logit=om, r_logit=full(rho, (1, T, 1)),
                p0=np.full(pshape, p0))


@pytest.mark.parametrize("variant", ["diag", "iso"])
def test_beta_eff_worked_example(golden, variant):
    """Reading notes Sec. 3.2 example: k = r = 1, predictive variance 9 -> 0.9,
    0.1 -> 0.0909; with k = 1 the effective write strength is the gain itself."""
    g = golden("gain_scalar_example")
    for p0, key in ((9.0, "kappa_pred_var_9"), (0.1, "kappa_pred_var_0p1")):
        out = gates.gated_forward(variant, mu=1.0, **_scalar(1, p0, variant))
        val, tol = g[key]
        assert abs(out["beta_eff"][0, 0, 0] - val) <= tol
        assert out["log_alpha"][0, 0, 0, 0] == 0.0 and out["r"][0, 0, 0] == pytest.approx(1.0, abs=1e-15)


@pytest.mark.parametrize("variant", ["diag", "iso"])
def test_beta_eff_repeated_observations(variant):
    """Sec. 3.2: D = 1, Omega = 0, p_0 = 1, equal-noise observations give posterior
    1/(n+1), so token n (1-based) sees predictive variance 1/n and
    beta_eff_n = (1/n) / (1 + 1/n) = 1/(n+1)."""
    T = 40
    out = gates.gated_forward(variant, mu=1.0, **_scalar(T, 1.0, variant))
    n = np.arange(1, T + 1)
    np.testing.assert_allclose(out["beta_eff"][0, :, 0], 1.0 / (n + 1), rtol=1e-13)


@pytest.mark.parametrize("variant", ["diag", "iso"])
def test_beta_eff_equals_z_over_r_plus_z(variant):
    """App. B Eq. 58-61: k^T kappa = z / (r + z) with z = k^T P_hat k, z formed
    here from the recurrence's predictive variances (not from its gains)."""
    rng = np.random.default_rng(11)
    B, T, H, d = 2, 30, 3, 8
    k = rng.standard_normal((B, T, H, d))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    q = rng.standard_normal((B, T, H, d))
    v = rng.standard_normal((B, T, H, d))
    a = rng.uniform(1.0, 5.0, (B, T, H, d))
    w = rng.normal(-3.0, 1.0, (B, T, H, d) if variant == "diag" else (B, T, H))
    rho = rng.standard_normal((B, T, H))
    out = gates.gated_forward(variant, q, k, v, a, w, rho, want_phat=True)
    ph = out["phat"]
    z = np.einsum("bthi,bthi->bth", ph, k * k) if variant == "diag" else ph * np.sum(k * k, axis=-1)
    np.testing.assert_allclose(out["beta_eff"], z / (out["r"] + z), rtol=1e-12)
    assert np.all(out["beta_eff"] >= 0.0) and np.all(out["beta_eff"] < 1.0)


@pytest.mark.parametrize("variant", ["diag", "iso"])
def test_gated_forward_is_the_recurrence_on_the_gates(variant):
    """gated_forward composes Sec. 5.1's gates with the pinned recurrence: the
    same outputs as the recurrence driven by scipy's logistic routines."""
    rng = np.random.default_rng(12)
    B, T, H, d = 1, 20, 2, 8
    k = rng.standard_normal((B, T, H, d))
    q = rng.standard_normal((B, T, H, d))
    v = rng.standard_normal((B, T, H, d))
    a = rng.uniform(-2.0, 6.0, (B, T, H, d))
    w = rng.normal(-4.0, 2.0, (B, T, H, d) if variant == "diag" else (B, T, H))
    rho = rng.standard_normal((B, T, H))
    out = gates.gated_forward(variant, q, k, v, a, w, rho, r_min=0.05)
    ref = recurrence.forward(variant, q, k, v, special.log_expit(a), -special.log_expit(-w),
                             0.05 - special.log_expit(-rho))
    for n in ("o", "S_T", "p_T"):
        np.testing.assert_allclose(out[n], ref[n], rtol=1e-11, atol=1e-13)
