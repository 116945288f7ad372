"""Planted mistakes in the oracle must fail a pin.

Each mutant is the oracle's C file with one plausible slip (a dropped term, a
wrong operand, a wrong sign or normalisation), compiled on the CPU into a
temporary library.  The pin checks below (the same facts the pin tests use:
the dense exact filter on axis-aligned keys, the pages' Moebius matrices, the
Delta-rule reduction, the printed scalar examples) must all pass for the real
oracle and at least one must fail for every mutant.
"""
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle
from oracle import dense, recurrence

SRC = os.path.join(os.path.dirname(recurrence.__file__), "kdn_oracle.c")

MUTANTS = {
    "alpha_not_squared": ("phat[i] = a[i] * a[i] * p[i] + omt[i];", "phat[i] = a[i] * p[i] + omt[i];"),
    "mean_not_decayed": ("for (int j = 0; j < dv; ++j) S[(size_t)i * dv + j] *= a[i];",
                         "for (int j = 0; j < dv; ++j) S[(size_t)i * dv + j] *= 1.0;"),
    "gain_uses_posterior": ("kappa[i] = phat[i] * kt[i] / (rt + z);", "kappa[i] = p[i] * kt[i] / (rt + z);"),
    "innovation_wrong_key": ("pred += S[(size_t)i * dv + j] * kt[i];", "pred += S[(size_t)i * dv + j] * qt[i];"),
    "innovation_sign": ("delta[j] = vt[j] - pred;", "delta[j] = pred - vt[j];"),
    "info_scale_times_r": ("const double u = (J->mu / rt) * kt[i] * kt[i];",
                           "const double u = (J->mu * rt) * kt[i] * kt[i];"),
    "iso_no_trace_mean": ("abar /= (double)dk;", "abar /= 1.0;"),
    "iso_info_no_dk": ("const double u = J->mu * knorm2 / ((double)dk * rt);",
                       "const double u = J->mu * knorm2 / rt;"),
    "iso_beta_no_norm": ("const double beta = phat[0] / (rt + phat[0] * knorm2);",
                         "const double beta = phat[0] / (rt + phat[0]);"),
    "z_missing_square": ("z += phat[i] * kt[i] * kt[i];", "z += phat[i] * kt[i];"),
}


def _close(a, b, rtol=1e-9, atol=1e-11):
    return np.allclose(a, b, rtol=rtol, atol=atol)


def pin_suite(lib):
    """Return the list of pin names that FAIL for the oracle build ``lib``."""
    fails = []
    rng = np.random.default_rng(123)
    fw = lambda *a, **kw: oracle.forward(*a, lib=lib, **kw)
    # 1. axis-aligned keys, mu = 1: diagonal KDN == dense exact filter
    B, T, H, dk, dv = 1, 25, 2, 5, 3
    q = rng.standard_normal((B, T, H, dk))
    v = rng.standard_normal((B, T, H, dv))
    la = -rng.uniform(0.05, 0.5, (B, T, H, dk))
    om = rng.uniform(0.01, 0.3, (B, T, H, dk))
    r = 0.05 + rng.random((B, T, H))
    j = rng.integers(0, dk, (B, T, H))
    k1 = np.zeros((B, T, H, dk))
    np.put_along_axis(k1, j[..., None], rng.uniform(0.3, 1.5, (B, T, H, 1)), -1)
    S0 = rng.standard_normal((B, H, dk, dv))
    p0 = rng.uniform(0.2, 2.0, (B, H, dk))
    out = fw("diag", q, k1, v, la, om, r, S0=S0, p0=p0, mu=1.0)
    for h in range(H):
        ex = dense.dense_kalman(k1[0, :, h], v[0, :, h], q[0, :, h], r[0, :, h], S0[0, h],
                                np.diag(p0[0, h]), D=np.exp(la[0, :, h]), Omega=om[0, :, h])
        if not (_close(out["o"][0, :, h], ex["o"]) and _close(out["p_T"][0, h], np.diag(ex["P_T"]))):
            fails.append("one_hot_dense")
            break
    # 2. Moebius form of the uncertainty (diag and iso), dense keys, mu != 1
    k = rng.standard_normal((B, T, H, dk))
    mu = 2.5
    for variant in ("diag", "iso"):
        omv = om if variant == "diag" else om[..., 0]
        o2 = fw(variant, q, k, v, la, omv, r, mu=mu)
        h = 1
        if variant == "diag":
            M = dense.mobius_matrices(la[0, :, h], om[0, :, h], k[0, :, h], r[0, :, h], mu)
            pT = dense.mobius_apply(dense.mobius_product(M, 0, T), np.ones(dk))
        else:
            a_bar = np.exp(2 * la[0, :, h]).mean(-1)
            kn = np.sqrt(np.sum(k[0, :, h] ** 2, -1) / dk)
            M = dense.mobius_matrices(0.5 * np.log(a_bar)[:, None], om[0, :, h, :1], kn[:, None],
                                      r[0, :, h], mu)
            pT = dense.mobius_apply(dense.mobius_product(M, 0, T), np.ones(1))
        if not _close(np.ravel(o2["p_T"][0, h]), pT):
            fails.append(f"mobius_{variant}")
    # 3. Delta-rule / KDA reduction (mu = 0, predictive variance forced to lambda_t)
    lam = rng.uniform(0.2, 3.0, (B, T, H))
    a2 = np.exp(2 * la)
    lam_prev = np.concatenate([np.ones((B, 1, H)), lam[:, :-1]], 1)
    for variant in ("diag", "iso"):
        omv = lam[..., None] - a2 * lam_prev[..., None] if variant == "diag" else lam - a2.mean(-1) * lam_prev
        o3 = fw(variant, q, k, v, la, omv, r, S0=S0, mu=0.0)
        h = 0
        S = S0[0, h].copy()
        ok = True
        for t in range(T):
            kk = k[0, t, h]
            beta = lam[0, t, h] / (r[0, t, h] + lam[0, t, h] * kk @ kk)
            DS = np.exp(la[0, t, h])[:, None] * S
            S = DS + beta * np.outer(kk, v[0, t, h] - DS.T @ kk)
            ok = ok and _close(o3["o"][0, t, h], S.T @ q[0, t, h])
        if not ok:
            fails.append(f"kda_{variant}")
    # 4. scalar example: prior 9, k = r = 1 -> gain 0.9 (S_0 = 0, v = q = 1 -> o = gain)
    one = np.ones((1, 1, 1, 1))
    for variant in ("diag", "iso"):
        omv = np.zeros((1, 1, 1, 1)) if variant == "diag" else np.zeros((1, 1, 1))
        p0v = np.full((1, 1, 1) if variant == "diag" else (1, 1), 9.0)
        o4 = fw(variant, one, one, one, np.zeros((1, 1, 1, 1)), omv, np.ones((1, 1, 1)), p0=p0v, mu=1.0)
        if abs(o4["o"].ravel()[0] - 0.9) > 1e-12:
            fails.append(f"scalar_{variant}")
    return fails


def test_real_oracle_passes_pin_suite():
    assert pin_suite(None) == []


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, name):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor not found once: {old}"
    mpath = tmp_path / f"kdn_oracle_{name}.c"
    mpath.write_text(src.replace(old, new))
    so = tmp_path / f"libkdn_oracle_{name}.so"
    others = [f for f in recurrence.sources() if os.path.basename(f) != "kdn_oracle.c"]
    subprocess.check_call(["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-o", str(so), str(mpath)]
                          + others + ["-lm", "-lpthread"])
    lib = recurrence.open_library(str(so))
    assert pin_suite(lib), f"mutant {name} passed every pin"
