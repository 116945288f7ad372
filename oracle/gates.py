"""Gate activations of the KDN layer and the effective write strength (fp64).

TEST INFRASTRUCTURE ONLY (see the package docstring).

gate_values    -- the parameter branches of the end-to-end network, KDN reading
                  notes Sec. 5.1 (the paragraph on the parameters the network
                  actually learns): alpha_t = sigma(a_t), omega_t = softplus(w_t)
                  (one scalar per token-head for Isotropic KDN), and
                  r_t = r_min + softplus(rho_t) with r_min = 0.01, where a, w, rho
                  are the projections W x + b of the layer input (the "logits";
                  computing them is the caller's GEMM).  The mixer consumes
                  log alpha, so the first branch is written as
                  log alpha = log sigma(a) = -softplus(-a).
beta_eff       -- effective write strength beta_eff_t = k_t^T kappa_t, KDN reading
                  notes Sec. 3.2 (after Eq. 12-17; the paper's App. B, Eq. 58-61):
                  with z_t = k_t^T P_hat_t k_t it equals z_t / (r_t + z_t), the
                  fraction of the innovation along k_t that the write removes.
gated_forward  -- gate_values, then the fp64 recurrence (recurrence.forward) on the
                  resulting log alpha, omega, r, then beta_eff from its gains.

Pinned by tests/test_gates_oracle.py: closed forms at zero logits, the symmetry
identities of the logistic function and softplus, scipy's independent logistic
routines, the asymptotes, and for beta_eff the worked one-dimensional example of
Sec. 3.2 (tests/golden/gain_scalar_example.txt), the repeated-observation closed
form 1 / (n + 1) and the identity k^T kappa = z / (r + z) with z from the
recurrence's predictive variances.
"""
from __future__ import annotations

import numpy as np

from . import recurrence

R_MIN = 0.01   # the notes' r_min (Sec. 5.1)


def _f64(x):
    return None if x is None else np.asarray(x, dtype=np.float64)


def softplus(x):
    """log(1 + e^x), evaluated without overflow as logaddexp(0, x)."""
    return np.logaddexp(0.0, _f64(x))


def gate_values(alpha_logit, omega_logit, r_logit, r_min=R_MIN):
    """The three gate branches of Sec. 5.1 on pre-activations (any shapes).

    Returns a dict: log_alpha = log sigma(alpha_logit) (< 0), omega =
    softplus(omega_logit) (> 0), r = r_min + softplus(r_logit) (> r_min).
    """
    return {
        "log_alpha": -softplus(-_f64(alpha_logit)),
        "omega": softplus(omega_logit),
        "r": float(r_min) + softplus(r_logit),
    }


def beta_eff(k, kappa):
    """beta_eff_t = k_t^T kappa_t per token-head; k, kappa [B,T,H,dk] -> [B,T,H]."""
    return np.einsum("bthi,bthi->bth", _f64(k), _f64(kappa))


def gated_forward(variant, q, k, v, alpha_logit, omega_logit, r_logit, S0=None, p0=None,
                  mu=None, r_min=R_MIN, want_phat=False):
    """The KDN forward driven by gate logits: ``recurrence.forward`` on
    :func:`gate_values`, plus ``beta_eff`` [B,T,H] and the gate values themselves.

    alpha_logit [B,T,H,dk]; omega_logit [B,T,H,dk] (diag) or [B,T,H] (iso);
    r_logit [B,T,H]; the rest as in ``recurrence.forward``.
    """
    g = gate_values(alpha_logit, omega_logit, r_logit, r_min)
    out = recurrence.forward(variant, q, k, v, g["log_alpha"], g["omega"], g["r"], S0=S0, p0=p0,
                             mu=mu, want_kappa=True, want_phat=want_phat)
    out["beta_eff"] = beta_eff(k, out["kappa"])
    out.update(g)
    return out
