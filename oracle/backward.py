"""Reverse-mode gradients of the KDN forward, fp64, token by token.

TEST INFRASTRUCTURE ONLY (see the package docstring).

The pages define the forward recurrence and no backward pass; the gradients
here are the adjoint of that recurrence, written out step by step in the
reverse order of the forward (KDN paper Sec. 4.1, Eq. 23-27 and 60-65 for the
Diagonal variant; Sec. 4.2, Eq. 40 and App. C for the Isotropic one).  For one
token, with a = exp(log_alpha):

  Diagonal:  p_hat = a^2 p + omega            Isotropic:  b_hat = mean(a^2) b + omega
             kappa = p_hat k / (r + sum p_hat k^2)         kappa = k b_hat / (r + b_hat ||k||^2)
             p'    = p_hat / (1 + (mu / r) k^2 p_hat)      b' = b_hat / (1 + mu ||k||^2 / (d_k r) b_hat)
  both:      S_hat = diag(a) S,  delta = v - S_hat^T k,  S' = S_hat + kappa delta^T,  o = S'^T q.

``forward_backward`` runs that forward in numpy (keeping each token's
intermediates) and then the adjoint sweep for upstream gradients dO, dS_T,
dp_T of the outputs o, S_T, p_T.  It is pinned by central finite differences
of the forward and by agreement of its forward with the C oracle
(tests/test_backward_oracle.py).  Tiny inputs only: Python loops over
(b, h, t).
"""
from __future__ import annotations

import numpy as np


def _f64(x):
    return None if x is None else np.asarray(x, dtype=np.float64)


def forward_backward(variant, q, k, v, log_alpha, omega, r, S0=None, p0=None, mu=None,
                     dO=None, dS_T=None, dp_T=None):
    """Forward outputs and the gradients of sum(dO*o) + sum(dS_T*S_T) + sum(dp_T*p_T).

    Shapes as ``oracle.forward``: q, k, log_alpha [B,T,H,dk]; v [B,T,H,dv];
    omega [B,T,H,dk] (diag) or [B,T,H] (iso); r [B,T,H]; S0 [B,H,dk,dv] or None
    (zeros); p0 [B,H,dk] / [B,H] or None (ones); mu None means d_k.  Upstream
    gradients default to zero.  Returns (out, grads): out has o, S_T, p_T;
    grads has q, k, v, log_alpha, omega, r, S0, p0.
    """
    if variant not in ("diag", "iso"):
        raise ValueError(variant)
    iso = variant == "iso"
    q, k, v, la, om, r = (_f64(x) for x in (q, k, v, log_alpha, omega, r))
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    mu = float(dk) if mu is None else float(mu)
    pshape = (B, H) if iso else (B, H, dk)
    S0 = np.zeros((B, H, dk, dv)) if S0 is None else _f64(S0)
    p0 = np.ones(pshape) if p0 is None else _f64(p0)
    dO = np.zeros((B, T, H, dv)) if dO is None else _f64(dO)
    dS_T = np.zeros((B, H, dk, dv)) if dS_T is None else _f64(dS_T)
    dp_T = np.zeros(pshape) if dp_T is None else _f64(dp_T)

    out = {"o": np.zeros((B, T, H, dv)), "S_T": np.zeros((B, H, dk, dv)), "p_T": np.zeros(pshape)}
    g = {"q": np.zeros_like(q), "k": np.zeros_like(k), "v": np.zeros_like(v), "log_alpha": np.zeros_like(la),
         "omega": np.zeros_like(om), "r": np.zeros_like(r), "S0": np.zeros((B, H, dk, dv)),
         "p0": np.zeros(pshape)}

    for b in range(B):
        for h in range(H):
            S = S0[b, h].copy()
            p = np.array(p0[b, h], dtype=np.float64, copy=True)
            tape = []
            # ---- forward, keeping what the adjoint needs
            for t in range(T):
                a = np.exp(la[b, t, h])
                kt, qt, vt, rt = k[b, t, h], q[b, t, h], v[b, t, h], r[b, t, h]
                if iso:
                    abar = np.mean(a * a)
                    ph = abar * p + om[b, t, h]
                    K2 = float(kt @ kt)
                    den = rt + ph * K2
                    beta = ph / den
                    kap = beta * kt
                    u = mu * K2 / (dk * rt)
                else:
                    ph = a * a * p + om[b, t, h]
                    den = rt + float(np.sum(ph * kt * kt))
                    kap = ph * kt / den
                    u = mu * kt * kt / rt
                Sh = a[:, None] * S
                delta = vt - Sh.T @ kt
                Sn = Sh + np.outer(kap, delta)
                out["o"][b, t, h] = Sn.T @ qt
                gq = 1.0 + u * ph
                tape.append((a, p, ph, den, kap, u, gq, S, Sh, delta, Sn) + ((abar, K2, beta) if iso else ()))
                S = Sn
                p = ph / gq
            out["S_T"][b, h] = S
            out["p_T"][b, h] = p
            # ---- adjoint sweep, newest token first
            dS = dS_T[b, h].copy()
            dp = np.array(dp_T[b, h], dtype=np.float64, copy=True)
            for t in range(T - 1, -1, -1):
                a, pprev, ph, den, kap, u, gq, Sprev, Sh, delta, Sn = tape[t][:11]
                kt, qt, rt = k[b, t, h], q[b, t, h], r[b, t, h]
                do = dO[b, t, h]
                # read: o = S'^T q
                dSn = dS + np.outer(qt, do)
                g["q"][b, t, h] += Sn @ do
                # write: S' = S_hat + kappa delta^T
                dSh = dSn.copy()
                dkap = dSn @ delta
                ddelta = dSn.T @ kap
                # innovation: delta = v - S_hat^T k
                g["v"][b, t, h] += ddelta
                dSh -= np.outer(kt, ddelta)
                gk = -(Sh @ ddelta)
                # prediction of the mean: S_hat = diag(a) S
                dS = a[:, None] * dSh
                da = np.sum(dSh * Sprev, axis=1)
                # information update: p' = p_hat / gq, gq = 1 + u p_hat
                dph = dp / (gq * gq)
                du = -dp * ph * ph / (gq * gq)
                if iso:
                    abar, K2, beta = tape[t][11:]
                    # kappa = beta k, beta = p_hat / den, den = r + p_hat ||k||^2
                    dbeta = float(dkap @ kt)
                    gk += beta * dkap
                    dph += dbeta / den
                    dden = -dbeta * ph / (den * den)
                    g["r"][b, t, h] += dden
                    dph += dden * K2
                    dK2 = dden * ph
                    # u = mu ||k||^2 / (d_k r)
                    dK2 += du * mu / (dk * rt)
                    g["r"][b, t, h] += -du * mu * K2 / (dk * rt * rt)
                    gk += 2.0 * dK2 * kt
                    # p_hat = mean(a^2) b + omega
                    dp = abar * dph
                    dabar = pprev * dph
                    g["omega"][b, t, h] += dph
                    da += dabar * 2.0 * a / dk
                else:
                    # kappa = p_hat k / den, den = r + sum p_hat k^2
                    dph += dkap * kt / den
                    gk += dkap * ph / den
                    dden = -float(np.sum(dkap * ph * kt)) / (den * den)
                    g["r"][b, t, h] += dden
                    dph += dden * kt * kt
                    gk += 2.0 * dden * ph * kt
                    # u = mu k^2 / r
                    gk += du * 2.0 * mu * kt / rt
                    g["r"][b, t, h] += float(np.sum(-du * mu * kt * kt / (rt * rt)))
                    # p_hat = a^2 p + omega
                    dp = a * a * dph
                    da += 2.0 * a * pprev * dph
                    g["omega"][b, t, h] += dph
                g["k"][b, t, h] += gk
                g["log_alpha"][b, t, h] += da * a
            g["S0"][b, h] = dS
            g["p0"][b, h] = dp
    return out, g
