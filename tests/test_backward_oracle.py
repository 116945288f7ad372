"""Pins of the fp64 backward oracle (oracle/backward.py) on the CPU.

The pages print no gradients, so the adjoint is pinned against the forward
itself: its own forward must agree with the C oracle's token recurrence, and
every gradient entry must agree with a central finite difference of the C
oracle's forward (an implementation that shares no code with the adjoint) for
the loss sum(dO*o) + sum(dS_T*S_T) + sum(dp_T*p_T) with random upstream
weights.  Diagonal and Isotropic variants, default and unit information scale,
with and without an initial state.
"""
import numpy as np
import pytest

import oracle
from oracle.backward import forward_backward
from uncertainty_aware_delta_gb300.inputs import make_inputs

NAMES = ("q", "k", "v", "log_alpha", "omega", "r")


def _loss(variant, x, S0, p0, mu, w):
    out = oracle.forward(variant, *(x[n] for n in NAMES), S0=S0, p0=p0, mu=mu)
    return float(np.sum(w["o"] * out["o"]) + np.sum(w["S"] * out["S_T"]) + np.sum(w["p"] * out["p_T"]))


@pytest.mark.parametrize("variant,mu,with_state", [("diag", None, False), ("diag", 1.0, True),
                                                   ("iso", None, True), ("iso", 1.0, False)])
def test_backward_matches_finite_differences(variant, mu, with_state):
    B, T, H, d = 1, 6, 2, 4
    x = {n: np.asarray(a, np.float64) for n, a in make_inputs(variant, B, T, H, d, d, io="f32", seed=71).items()
         if n != "io"}
    rng = np.random.default_rng(72)
    pshape = (B, H, d) if variant == "diag" else (B, H)
    S0 = rng.standard_normal((B, H, d, d)) if with_state else None
    p0 = rng.uniform(0.3, 2.0, size=pshape) if with_state else None
    w = {"o": rng.standard_normal((B, T, H, d)), "S": rng.standard_normal((B, H, d, d)),
         "p": rng.standard_normal(pshape)}
    out, g = forward_backward(variant, *(x[n] for n in NAMES), S0=S0, p0=p0, mu=mu, dO=w["o"], dS_T=w["S"],
                              dp_T=w["p"])
    ref = oracle.forward(variant, *(x[n] for n in NAMES), S0=S0, p0=p0, mu=mu)
    for n in ("o", "S_T", "p_T"):
        assert np.allclose(out[n], ref[n], rtol=1e-12, atol=1e-14), n

    inputs = dict(x)
    inputs["S0"] = np.zeros((B, H, d, d)) if S0 is None else S0.copy()
    inputs["p0"] = np.ones(pshape) if p0 is None else p0.copy()
    for name, arr in inputs.items():
        flat = arr.reshape(-1)
        for idx in range(flat.size):
            h = 1e-6 * max(1.0, abs(flat[idx]))
            old = flat[idx]
            flat[idx] = old + h
            lp = _loss(variant, {n: inputs[n] for n in NAMES}, inputs["S0"], inputs["p0"], mu, w)
            flat[idx] = old - h
            lm = _loss(variant, {n: inputs[n] for n in NAMES}, inputs["S0"], inputs["p0"], mu, w)
            flat[idx] = old
            fd = (lp - lm) / (2.0 * h)
            adj = g[name].reshape(-1)[idx]
            assert abs(fd - adj) <= 1e-6 * max(1.0, abs(adj)), (variant, name, idx, fd, adj)


def test_backward_of_an_empty_sequence_passes_the_state_gradients_through():
    B, T, H, d = 1, 0, 2, 4
    x = {n: np.asarray(a, np.float64) for n, a in make_inputs("diag", B, T, H, d, d, io="f32", seed=3).items()
         if n != "io"}
    rng = np.random.default_rng(4)
    dS, dp = rng.standard_normal((B, H, d, d)), rng.standard_normal((B, H, d))
    _, g = forward_backward("diag", *(x[n] for n in NAMES), dS_T=dS, dp_T=dp)
    assert np.array_equal(g["S0"], dS) and np.array_equal(g["p0"], dp)


def test_backward_single_token_closed_form():
    """One token from S0 = 0: o = S'^T q = (q . kappa) v, so do/dv = (q . kappa) I
    and the gradient of sum(dO*o) with respect to v is (q . kappa) dO."""
    B, T, H, d = 1, 1, 1, 5
    x = {n: np.asarray(a, np.float64) for n, a in make_inputs("diag", B, T, H, d, d, io="f32", seed=8).items()
         if n != "io"}
    dO = np.random.default_rng(9).standard_normal((B, T, H, d))
    _, g = forward_backward("diag", *(x[n] for n in NAMES), dO=dO)
    a = np.exp(x["log_alpha"][0, 0, 0])
    ph = a * a * 1.0 + x["omega"][0, 0, 0]
    kt = x["k"][0, 0, 0]
    kap = ph * kt / (x["r"][0, 0, 0] + np.sum(ph * kt * kt))
    assert np.allclose(g["v"][0, 0, 0], float(x["q"][0, 0, 0] @ kap) * dO[0, 0, 0], rtol=1e-13, atol=1e-15)


def test_a_planted_mistake_in_the_adjoint_is_caught():
    """The finite-difference pin fails for an adjoint that drops one term (the
    dependence of the gain denominator on the predicted variance)."""
    import oracle.backward as bw

    src = open(bw.__file__).read()
    assert src.count("dph += dden * kt * kt") == 1
    ns = {}
    exec(compile(src.replace("dph += dden * kt * kt", "dph += 0.0 * kt"), "planted_mistake", "exec"), ns)
    B, T, H, d = 1, 4, 1, 4
    x = {n: np.asarray(a, np.float64) for n, a in make_inputs("diag", B, T, H, d, d, io="f32", seed=5).items()
         if n != "io"}
    rng = np.random.default_rng(6)
    w = {"o": rng.standard_normal((B, T, H, d)), "S": np.zeros((B, H, d, d)), "p": np.zeros((B, H, d))}
    _, g = ns["forward_backward"]("diag", *(x[n] for n in NAMES), dO=w["o"])
    worst = 0.0
    flat = x["omega"].reshape(-1)
    for idx in range(flat.size):
        h, old = 1e-6, flat[idx]
        flat[idx] = old + h
        lp = _loss("diag", x, None, None, None, w)
        flat[idx] = old - h
        lm = _loss("diag", x, None, None, None, w)
        flat[idx] = old
        adj = g["omega"].reshape(-1)[idx]
        worst = max(worst, abs((lp - lm) / (2 * h) - adj) / max(1.0, abs(adj)))
    assert worst > 1e-4
