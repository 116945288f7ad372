"""numpy fp64 companions of the oracle, for tiny inputs only.

TEST INFRASTRUCTURE ONLY (see the package docstring).

dense_kalman       -- the exact Kalman associative memory with a dense key-space
                      covariance: KDN paper Sec. 3.2, Eq. 12-17 (predict
                      S_hat = D S, P_hat = D P D^T + Omega; gain
                      kappa = P_hat k / (r + k^T P_hat k); write
                      S = S_hat + kappa (v - S_hat^T k)^T; P = (I - kappa k^T) P_hat;
                      read o = S^T q after the write).  The Bayesian Layer
                      paper's Prop. 1 (its Eq. 9-13) is the same recursion.
mobius_matrices    -- the per-channel 2x2 matrices of the information-scaled
                      uncertainty recurrence, KDN paper Eq. 32-37:
                      M_t = [[a^2, omega], [u a^2, 1 + u omega]],
                      u = mu k^2 / r, [n; d]_t = M_t [n; d]_{t-1}, p = n / d.
mobius_product     -- ordered product M_hi ... M_lo (newest on the left) under
                      any bracketing; associativity is what the scan relies on.
ridge_closed_form  -- weighted ridge regression mean
                      (P0^{-1} + sum_t k_t k_t^T / r_t)^{-1} sum_t k_t v_t^T / r_t
                      (Preconditioned DeltaNet Eq. 1-5; Gated KalmaNet's
                      test-time ridge regression), the no-decay exact filter.
"""
from __future__ import annotations

import numpy as np


def dense_kalman(k, v, q, r, S0, P0, D=None, Omega=None):
    """Exact Kalman associative memory for one sequence, dense covariance.

    k, q: [T, dk]; v: [T, dv]; r: [T] (observation-noise variance);
    S0: [dk, dv]; P0: [dk, dk];
    D: None (identity), [T, dk] (diagonal transition) or [T, dk, dk];
    Omega: None (zero), [T, dk] (diagonal process noise) or [T, dk, dk].
    Returns dict(o [T,dv], S [T,dk,dv] post-write means, P [T,dk,dk],
    P_hat [T,dk,dk], kappa [T,dk], z [T], S_T, P_T).
    """
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    q = np.asarray(q, np.float64)
    r = np.asarray(r, np.float64)
    T, dk = k.shape
    dv = v.shape[1]
    S = np.array(S0, np.float64, copy=True)
    P = np.array(P0, np.float64, copy=True)
    I = np.eye(dk)
    out = {
        "o": np.zeros((T, dv)), "S": np.zeros((T, dk, dv)), "P": np.zeros((T, dk, dk)),
        "P_hat": np.zeros((T, dk, dk)), "kappa": np.zeros((T, dk)), "z": np.zeros(T),
    }
    for t in range(T):
        if D is None:
            Dt = I
        else:
            Dt = np.asarray(D[t], np.float64)
            if Dt.ndim == 1:
                Dt = np.diag(Dt)
        if Omega is None:
            Om = np.zeros((dk, dk))
        else:
            Om = np.asarray(Omega[t], np.float64)
            if Om.ndim == 1:
                Om = np.diag(Om)
        S_hat = Dt @ S
        P_hat = Dt @ P @ Dt.T + Om
        kt = k[t]
        Pk = P_hat @ kt
        z = float(kt @ Pk)
        kappa = Pk / (r[t] + z)
        delta = v[t] - S_hat.T @ kt
        S = S_hat + np.outer(kappa, delta)
        P = (I - np.outer(kappa, kt)) @ P_hat
        out["o"][t] = S.T @ q[t]
        out["S"][t] = S
        out["P"][t] = P
        out["P_hat"][t] = P_hat
        out["kappa"][t] = kappa
        out["z"][t] = z
    out["S_T"] = S
    out["P_T"] = P
    return out


def mobius_matrices(log_alpha, omega, k, r, mu):
    """Per-token, per-channel Moebius matrices M_t (shape [T, d, 2, 2]).

    log_alpha, omega, k: [T, d]; r: [T]; mu: scalar.
    For the isotropic variant pass a_bar (as log of its square root) per
    token with d = 1 and u folded in through k and r; callers build those.
    """
    la = np.asarray(log_alpha, np.float64)
    om = np.asarray(omega, np.float64)
    kk = np.asarray(k, np.float64)
    rr = np.asarray(r, np.float64)[:, None]
    a2 = np.exp(2.0 * la)
    u = mu * kk * kk / rr
    M = np.empty(la.shape + (2, 2))
    M[..., 0, 0] = a2
    M[..., 0, 1] = om
    M[..., 1, 0] = u * a2
    M[..., 1, 1] = 1.0 + u * om
    return M


def mobius_product(M, lo, hi, split=None):
    """Ordered product M[hi-1] @ ... @ M[lo] over the token axis (axis 0).

    ``split(lo, hi)`` picks the bracketing point (default: the midpoint);
    any choice must give the same product since matrix products associate.
    Returns an array of shape M.shape[1:] (per channel 2x2).
    """
    if hi - lo == 1:
        return M[lo].copy()
    if hi <= lo:
        eye = np.zeros(M.shape[1:])
        eye[..., 0, 0] = 1.0
        eye[..., 1, 1] = 1.0
        return eye
    m = (lo + hi) // 2 if split is None else split(lo, hi)
    left = mobius_product(M, m, hi, split)    # newer tokens
    right = mobius_product(M, lo, m, split)   # older tokens
    return np.einsum("...ij,...jk->...ik", left, right)


def mobius_apply(Mprod, p0):
    """p = n / d with [n; d] = Mprod [p0; 1]."""
    p0 = np.asarray(p0, np.float64)
    n = Mprod[..., 0, 0] * p0 + Mprod[..., 0, 1]
    d = Mprod[..., 1, 0] * p0 + Mprod[..., 1, 1]
    return n / d


def ridge_closed_form(k, v, r, P0):
    """Weighted ridge mean (P0^{-1} + sum k k^T / r)^{-1} sum k v^T / r."""
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    r = np.asarray(r, np.float64)
    w = 1.0 / r
    G = np.linalg.inv(np.asarray(P0, np.float64)) + (k * w[:, None]).T @ k
    C = (k * w[:, None]).T @ v
    return np.linalg.solve(G, C)
