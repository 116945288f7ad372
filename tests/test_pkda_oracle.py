"""Pins of the fp64 PKDA oracle (preconditioned delta rule with per-channel
decay) against what the Preconditioned DeltaNet pages and the mathematics fix,
and planted mistakes in its C file that must fail one of them.

None of the checks re-types the oracle's loop: they use printed values
(tests/golden/pdn_examples.txt), the exact apply-to-key theorem against ridge
regression, the printed chunk formula of the key statistic, the one-step
eigenvalues of the transition, and a reduction to the independently written
KDN oracle (its Delta-rule special case).
"""
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle
from oracle import dense, recurrence


def _pk(lib=None, **kw):
    return recurrence.pkda_forward(lib=lib, **kw)


# ---------------------------------------------------------------- the pin checks
def check_teaching_example(lib=None):
    """Sec. 2.4 (Eq. 9): A_1 = (16, 1) built from A_0 = (15, 0) and this token's
    k = (1, 1) (the statistic includes the current key), mu = log 4, x = 1.5
    -> write scale (0.790, 1.266); with S_0 = 0, v = beta = 1 the write is
    S_1 = B * k, so S_T reads the scale."""
    g = oracle_golden("pdn_examples")
    one = lambda *s: np.ones(s)
    out = _pk(lib, q=one(1, 1, 1, 2), k=one(1, 1, 1, 2), v=one(1, 1, 1, 1),
              log_alpha=np.zeros((1, 1, 1, 2)), beta=one(1, 1, 1), alpha_p=one(1, 1, 1),
              beta_p=one(1, 1, 1), center=np.array([np.log(4.0)]),
              A0=np.array([[[15.0, 0.0]]]), x=1.5)
    ok = np.allclose(out["A_T"].ravel(), [16.0, 1.0], rtol=0, atol=1e-12)
    for i in range(2):
        val, tol = g[f"squash_B_{i}"]
        ok = ok and abs(out["S_T"][0, 0, i, 0] - val) <= tol
    return ok


def check_diag_atk_counterexample(lib=None):
    """App. C.2: lambda = 1, k_1 = v_1 = (1, 1), diagonal apply-to-key -> S_1 = (1/3) 1 1^T."""
    g = oracle_golden("pdn_examples")
    one = lambda *s: np.ones(s)
    out = _pk(lib, q=one(1, 1, 1, 2), k=one(1, 1, 1, 2), v=one(1, 1, 1, 2),
              log_alpha=np.zeros((1, 1, 1, 2)), beta=one(1, 1, 1), mode="diag_atk", lam=1.0)
    val, tol = g["diag_atk_S1_entry"]
    return bool(np.all(np.abs(out["S_T"][0, 0] - val) <= tol))


def check_exact_atk_is_ridge(lib=None):
    """Sec. 2.2 Theorem 3.1: with the exact write key P_{t-1} k / (1 + k^T P_{t-1} k),
    beta = 1 and no decay, every prefix state equals the ridge solution
    (lambda I + sum k k^T)^{-1} sum k v^T, so o_t = S_t^T q_t with that S_t; and
    the write key equals P_t k_t."""
    rng = np.random.default_rng(11)
    T, dk, dv, lam = 14, 5, 3, 0.7
    k = rng.standard_normal((1, T, 1, dk))
    v = rng.standard_normal((1, T, 1, dv))
    q = rng.standard_normal((1, T, 1, dk))
    out = _pk(lib, q=q, k=k, v=v, log_alpha=np.zeros((1, T, 1, dk)), beta=np.ones((1, T, 1)),
              mode="exact_atk", lam=lam, want_kappa=True)
    ok = True
    for t in range(T):
        S = dense.ridge_closed_form(k[0, :t + 1, 0], v[0, :t + 1, 0], np.ones(t + 1), np.eye(dk) / lam)
        ok = ok and np.allclose(out["o"][0, t, 0], S.T @ q[0, t, 0], rtol=1e-9, atol=1e-11)
        G = lam * np.eye(dk) + k[0, :t + 1, 0].T @ k[0, :t + 1, 0]
        ok = ok and np.allclose(out["kappa"][0, t, 0], np.linalg.solve(G, k[0, t, 0]), rtol=1e-9,
                                atol=1e-11)
    S = dense.ridge_closed_form(k[0, :, 0], v[0, :, 0], np.ones(T), np.eye(dk) / lam)
    return ok and np.allclose(out["S_T"][0, 0], S, rtol=1e-9, atol=1e-11)


def check_statistic_chunk_formula(lib=None):
    """Sec. 2.6: A_out = (prod alpha_p) A_in + sum_j (prod_{l>j} alpha_p_l) beta_p_j k_j^2."""
    rng = np.random.default_rng(12)
    T, dk = 37, 6
    k = rng.standard_normal((1, T, 1, dk))
    ap = np.exp(-rng.uniform(0.0, 0.3, (1, T, 1)))
    bp = rng.uniform(0.0, 2.0, (1, T, 1))
    A0 = rng.uniform(0.0, 3.0, (1, 1, dk))
    out = _pk(lib, q=k, k=k, v=np.zeros((1, T, 1, 1)), log_alpha=np.zeros((1, T, 1, dk)),
              beta=np.zeros((1, T, 1)), alpha_p=ap, beta_p=bp, center=np.ones(1), A0=A0)
    a = ap[0, :, 0]
    after = np.array([np.prod(a[j + 1:]) for j in range(T)])   # prod_{l > j} alpha_p_l
    want = np.prod(a) * A0[0, 0] + np.sum((after * bp[0, :, 0])[:, None] * k[0, :, 0] ** 2, axis=0)
    return np.allclose(out["A_T"][0, 0], want, rtol=1e-12, atol=1e-14)


def check_kda_reduction(lib=None):
    """x = 1 makes every write scale 1 (Sec. 2.7: x = 1 degenerates to the
    ungated-preconditioner model), so PKDA is the gated Delta rule with write
    strength beta_t.  KDN with mu = 0 and its predictive variance forced to
    lambda_t is the same Delta rule with beta_t = lambda_t / (r_t + lambda_t ||k_t||^2)
    (KDN paper Sec. 2: Delta/KDA as the fixed-variance special case): the two
    independently written oracles must agree."""
    rng = np.random.default_rng(13)
    B, T, H, dk, dv = 1, 23, 2, 4, 3
    q = rng.standard_normal((B, T, H, dk))
    k = rng.standard_normal((B, T, H, dk))
    v = rng.standard_normal((B, T, H, dv))
    la = -rng.uniform(0.02, 0.4, (B, T, H, dk))
    r = 0.1 + rng.random((B, T, H))
    lam = rng.uniform(0.2, 3.0, (B, T, H))
    S0 = rng.standard_normal((B, H, dk, dv))
    a2 = np.exp(2 * la)
    lam_prev = np.concatenate([np.ones((B, 1, H)), lam[:, :-1]], 1)
    om = lam[..., None] - a2 * lam_prev[..., None]          # p_hat_t = lambda_t on every channel
    ref = oracle.forward("diag", q, k, v, la, om, r, S0=S0, mu=0.0)
    beta = lam / (r + lam * np.sum(k * k, -1))
    out = _pk(lib, q=q, k=k, v=v, log_alpha=la, beta=beta, alpha_p=rng.random((B, T, H)),
              beta_p=rng.random((B, T, H)), center=np.ones(H), S0=S0, x=1.0)
    return (np.allclose(out["o"], ref["o"], rtol=1e-10, atol=1e-12)
            and np.allclose(out["S_T"], ref["S_T"], rtol=1e-10, atol=1e-12))


def check_one_step_eigenvalues(lib=None):
    """Sec. 2.7 (App. E.3): one PGDN step acts on the state through
    alpha (I - beta k k_til^T) (transposed here), whose eigenvalues are alpha
    (d_k - 1 times) and alpha (1 - beta k^T k_til); for a unit key k^T k_til
    lies in [1/x, x]."""
    rng = np.random.default_rng(14)
    dk, x = 6, 1.5
    k = rng.standard_normal(dk)
    k /= np.linalg.norm(k)
    alpha, beta = 0.9, 0.8
    out = _pk(lib, q=np.zeros((1, 1, 1, dk)), k=k.reshape(1, 1, 1, dk), v=np.zeros((1, 1, 1, dk)),
              log_alpha=np.full((1, 1, 1, dk), np.log(alpha)), beta=np.full((1, 1, 1), beta),
              alpha_p=np.ones((1, 1, 1)), beta_p=np.ones((1, 1, 1)), center=np.array([0.3]),
              S0=np.eye(dk).reshape(1, 1, dk, dk), x=x, want_kappa=True)
    kt = out["kappa"][0, 0, 0] / beta
    ev = np.sort(np.linalg.eigvals(out["S_T"][0, 0]).real)
    want = np.sort(np.r_[np.full(dk - 1, alpha), alpha * (1 - beta * k @ kt)])
    return (np.allclose(ev, want, rtol=1e-10, atol=1e-12) and 1 / x - 1e-12 <= k @ kt <= x + 1e-12)


def check_pure_decay(lib=None):
    """No writes (beta = 0): S_t = diag(prod a) S_0 and o_t = S_t^T q_t (Sec. 2.5, D_t = Diag(alpha_t))."""
    rng = np.random.default_rng(15)
    T, dk, dv = 9, 4, 3
    la = -rng.uniform(0.0, 0.5, (1, T, 1, dk))
    S0 = rng.standard_normal((1, 1, dk, dv))
    q = rng.standard_normal((1, T, 1, dk))
    out = _pk(lib, q=q, k=rng.standard_normal((1, T, 1, dk)), v=rng.standard_normal((1, T, 1, dv)),
              log_alpha=la, beta=np.zeros((1, T, 1)), alpha_p=np.ones((1, T, 1)),
              beta_p=np.ones((1, T, 1)), center=np.ones(1), S0=S0)
    G = np.cumsum(la[0, :, 0], axis=0)
    ok = np.allclose(out["S_T"][0, 0], np.exp(G[-1])[:, None] * S0[0, 0], rtol=1e-13)
    for t in range(T):
        ok = ok and np.allclose(out["o"][0, t, 0], (np.exp(G[t])[:, None] * S0[0, 0]).T @ q[0, t, 0],
                                rtol=1e-12, atol=1e-14)
    return ok


PIN_CHECKS = {
    "teaching_example": check_teaching_example,
    "diag_atk_counterexample": check_diag_atk_counterexample,
    "exact_atk_is_ridge": check_exact_atk_is_ridge,
    "statistic_chunk_formula": check_statistic_chunk_formula,
    "kda_reduction": check_kda_reduction,
    "one_step_eigenvalues": check_one_step_eigenvalues,
    "pure_decay": check_pure_decay,
}


def oracle_golden(name):
    from conftest import load_golden
    return load_golden(name)


@pytest.mark.parametrize("name", sorted(PIN_CHECKS))
def test_pkda_pin(name):
    assert PIN_CHECKS[name](), name


def test_pkda_continuation():
    """Splitting a sequence and resuming from (S_T, A_T) is the same recurrence."""
    rng = np.random.default_rng(16)
    B, T, H, dk, dv = 2, 31, 2, 8, 5
    x = dict(q=rng.standard_normal((B, T, H, dk)), k=rng.standard_normal((B, T, H, dk)),
             v=rng.standard_normal((B, T, H, dv)), log_alpha=-rng.uniform(0, 0.2, (B, T, H, dk)),
             beta=rng.random((B, T, H)), alpha_p=rng.random((B, T, H)), beta_p=rng.random((B, T, H)))
    ce = rng.uniform(0.1, 2.0, H)
    full = recurrence.pkda_forward(**x, center=ce)
    cut = 13
    first = recurrence.pkda_forward(**{n: a[:, :cut] for n, a in x.items()}, center=ce)
    second = recurrence.pkda_forward(**{n: a[:, cut:] for n, a in x.items()}, center=ce,
                                     S0=first["S_T"], A0=first["A_T"])
    assert np.allclose(np.concatenate([first["o"], second["o"]], 1), full["o"], rtol=1e-12, atol=1e-13)
    assert np.allclose(second["S_T"], full["S_T"], rtol=1e-12, atol=1e-13)
    assert np.allclose(second["A_T"], full["A_T"], rtol=1e-12, atol=1e-14)


def test_pkda_step_is_one_token():
    rng = np.random.default_rng(17)
    B, H, dk, dv = 3, 2, 4, 3
    S = rng.standard_normal((B, H, dk, dv))
    A = rng.random((B, H, dk))
    args = [rng.standard_normal((B, H, dk)), rng.standard_normal((B, H, dk)),
            rng.standard_normal((B, H, dv)), -rng.random((B, H, dk)), rng.random((B, H)),
            rng.random((B, H)), rng.random((B, H)), rng.uniform(0.1, 2.0, H)]
    o, S1, A1 = recurrence.pkda_step(*args, S, A)
    full = recurrence.pkda_forward(*[a[:, None] if i < 7 else a for i, a in enumerate(args)], S0=S, A0=A)
    assert np.array_equal(o, full["o"][:, 0]) and np.array_equal(S1, full["S_T"])
    assert np.array_equal(A1, full["A_T"])


# ---------------------------------------------------------------- planted mistakes
PKDA_MUTANTS = {
    "statistic_after_scale": (
        "                A[i] = ap * A[i] + bp * kv[i] * kv[i];\n"
        "                const double rho = log(A[i] > kStatFloor ? A[i] : kStatFloor) - mu;\n",
        "                const double rho = log(A[i] > kStatFloor ? A[i] : kStatFloor) - mu;\n"
        "                A[i] = ap * A[i] + bp * kv[i] * kv[i];\n"),
    "statistic_not_squared": ("A[i] = ap * A[i] + bp * kv[i] * kv[i];", "A[i] = ap * A[i] + bp * kv[i];"),
    "no_softsign": ("const double s = rho / (1.0 + fabs(rho));", "const double s = rho;"),
    "scale_sign": ("kt[i] = exp(-logx * s) * kv[i];", "kt[i] = exp(logx * s) * kv[i];"),
    "residual_with_write_key": ("pred += S[(size_t)i * dv + j] * kv[i];", "pred += S[(size_t)i * dv + j] * kt[i];"),
    "no_decay": ("for (int j = 0; j < dv; ++j) S[(size_t)i * dv + j] *= a;",
                 "for (int j = 0; j < dv; ++j) S[(size_t)i * dv + j] *= 1.0;"),
    "no_beta": ("S[(size_t)i * dv + j] += bt * kt[i] * delta[j];", "S[(size_t)i * dv + j] += kt[i] * delta[j];"),
    "atk_no_normaliser": ("for (int i = 0; i < dk; ++i) kt[i] = Pk[i] / (1.0 + kpk);",
                          "for (int i = 0; i < dk; ++i) kt[i] = Pk[i];"),
    "read_before_write": (
        "        for (int i = 0; i < dk; ++i)\n"
        "            for (int j = 0; j < dv; ++j) S[(size_t)i * dv + j] += bt * kt[i] * delta[j];\n\n"
        "        for (int j = 0; j < dv; ++j) {\n"
        "            double acc = 0.0;\n"
        "            for (int i = 0; i < dk; ++i) acc += S[(size_t)i * dv + j] * qt[i];\n"
        "            ot[j] = acc;\n"
        "        }\n",
        "        for (int j = 0; j < dv; ++j) {\n"
        "            double acc = 0.0;\n"
        "            for (int i = 0; i < dk; ++i) acc += S[(size_t)i * dv + j] * qt[i];\n"
        "            ot[j] = acc;\n"
        "        }\n"
        "        for (int i = 0; i < dk; ++i)\n"
        "            for (int j = 0; j < dv; ++j) S[(size_t)i * dv + j] += bt * kt[i] * delta[j];\n\n"),
}


def test_real_pkda_oracle_passes_every_pin():
    assert [n for n, f in PIN_CHECKS.items() if not f()] == []


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
@pytest.mark.parametrize("name", sorted(PKDA_MUTANTS))
def test_pkda_mutant_is_caught(tmp_path, name):
    old, new = PKDA_MUTANTS[name]
    srcs = recurrence.sources()
    src_path = [f for f in srcs if os.path.basename(f) == "pkda_oracle.c"][0]
    src = open(src_path).read()
    assert src.count(old) == 1, f"mutation anchor not found once: {old}"
    mpath = tmp_path / f"pkda_oracle_{name}.c"
    mpath.write_text(src.replace(old, new))
    so = tmp_path / f"libpkda_{name}.so"
    others = [f for f in srcs if f != src_path]
    subprocess.check_call(["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-o", str(so), str(mpath)]
                          + others + ["-lm", "-lpthread"])
    lib = recurrence.open_library(str(so))
    failed = [n for n, f in PIN_CHECKS.items() if not f(lib)]
    assert failed, f"mutant {name} passed every pin"
