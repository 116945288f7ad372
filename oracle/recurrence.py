"""ctypes wrappers over the fp64 token-by-token recurrences: KDN
(``kdn_oracle.c``) and the preconditioned delta rule PKDA / PGDN / PDN
(``pkda_oracle.c``).

TEST INFRASTRUCTURE ONLY (see the package docstring).

The C files are compiled with the host ``gcc`` into ``oracle/libkdn_oracle.so``
by :func:`build_oracle` (called from ``__graft_entry__.build()``); it is
rebuilt whenever a source is newer than the library.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRCS = [os.path.join(_HERE, "kdn_oracle.c"), os.path.join(_HERE, "pkda_oracle.c")]
_LIB = os.path.join(_HERE, "libkdn_oracle.so")
_lock = threading.Lock()
_lib = None

DIAG, ISO = 0, 1


def library_path() -> str:
    return _LIB


def sources() -> list:
    """The C files the oracle library is built from."""
    return list(_SRCS)


def build_oracle(force: bool = False) -> str:
    """Compile the oracle C files into a shared library (plain gcc, -O2, no fast-math)."""
    newest = max(os.path.getmtime(src) for src in _SRCS)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < newest:
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-o", tmp] + _SRCS + ["-lm", "-lpthread"]
        )
        os.replace(tmp, _LIB)
    return _LIB


def open_library(path: str):
    """Load an oracle shared library from ``path`` and declare its signatures."""
    lib = ctypes.CDLL(path)
    dp = ctypes.POINTER(ctypes.c_double)
    lib.kdn_oracle_forward.restype = ctypes.c_int
    lib.kdn_oracle_forward.argtypes = (
        [ctypes.c_int] * 6 + [ctypes.c_double] + [dp] * 6 + [dp] * 2 + [dp] * 3 + [dp] * 2
        + [ctypes.c_int]
    )
    lib.pkda_oracle_forward.restype = ctypes.c_int
    lib.pkda_oracle_forward.argtypes = (
        [ctypes.c_int] * 6 + [ctypes.c_double] * 2 + [dp] * 8 + [dp] * 2 + [dp] * 4 + [ctypes.c_int]
    )
    lib.kdn_oracle_default_threads.restype = ctypes.c_int
    lib.kdn_oracle_default_threads.argtypes = []
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build_oracle()
            _lib = open_library(_LIB)
    return _lib


def default_threads() -> int:
    return int(_load().kdn_oracle_default_threads())


def _f64(x):
    return None if x is None else np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def forward(variant, q, k, v, log_alpha, omega, r, S0=None, p0=None, mu=None,
            want_kappa=False, want_phat=False, nthreads=0, lib=None):
    """Run the KDN recurrence token by token in fp64.

    variant: "diag" / "iso" (or 0 / 1).
    q, k, log_alpha: [B,T,H,dk]; v: [B,T,H,dv]; omega: [B,T,H,dk] (diag) or
    [B,T,H] (iso); r: [B,T,H] observation-noise variance; S0: [B,H,dk,dv] or
    None (zeros); p0: [B,H,dk] (diag) / [B,H] (iso) or None (ones);
    mu: information scale, None means d_k (the paper's default).
    Returns a dict with o [B,T,H,dv], S_T, p_T and optionally kappa
    [B,T,H,dk] and phat (the predictive variance used by each token's gain).
    ``lib`` selects another build of the oracle (used by the mutation test).
    """
    var = {"diag": DIAG, "iso": ISO}.get(variant, variant)
    q, k, v, la, om, r = (_f64(x) for x in (q, k, v, log_alpha, omega, r))
    S0, p0 = _f64(S0), _f64(p0)
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    assert k.shape == (B, T, H, dk) and la.shape == (B, T, H, dk)
    assert v.shape == (B, T, H, dv) and r.shape == (B, T, H)
    nu_shape = (B, T, H, dk) if var == DIAG else (B, T, H)
    assert om.shape == nu_shape, (om.shape, nu_shape)
    if S0 is not None:
        assert S0.shape == (B, H, dk, dv)
    pshape = (B, H, dk) if var == DIAG else (B, H)
    if p0 is not None:
        assert p0.shape == pshape
    mu = float(dk if mu is None else mu)
    o = np.zeros((B, T, H, dv))
    S_T = np.zeros((B, H, dk, dv))
    p_T = np.zeros(pshape)
    kap = np.zeros((B, T, H, dk)) if want_kappa else None
    ph = np.zeros(nu_shape) if want_phat else None
    rc = (lib or _load()).kdn_oracle_forward(
        var, B, T, H, dk, dv, mu,
        _ptr(q), _ptr(k), _ptr(v), _ptr(la), _ptr(om), _ptr(r),
        _ptr(S0), _ptr(p0), _ptr(o), _ptr(S_T), _ptr(p_T), _ptr(kap), _ptr(ph), int(nthreads),
    )
    if rc != 0:
        raise RuntimeError(f"kdn_oracle_forward failed with code {rc}")
    out = {"o": o, "S_T": S_T, "p_T": p_T}
    if want_kappa:
        out["kappa"] = kap
    if want_phat:
        out["phat"] = ph
    return out


def step(variant, q, k, v, log_alpha, omega, r, S, p, mu=None):
    """One token of the recurrence for B independent sequences (decode).

    Per-token inputs are [B,H,d] (omega [B,H] for iso, r [B,H]); S [B,H,dk,dv]
    and p are the state before the token.  Returns (o [B,H,dv], S_new, p_new).
    """
    add_t = lambda x: None if x is None else np.asarray(x, dtype=np.float64)[:, None]
    out = forward(variant, add_t(q), add_t(k), add_t(v), add_t(log_alpha), add_t(omega),
                  add_t(r), S, p, mu)
    return out["o"][:, 0], out["S_T"], out["p_T"]


PKDA_MODES = {"squash": 0, "diag_atk": 1, "exact_atk": 2}
PKDA_X = 1.5   # the pages' bound: every channel's write scale lies in [1/x, x]


def pkda_forward(q, k, v, log_alpha, beta, alpha_p=None, beta_p=None, center=None, S0=None,
                 A0=None, x=PKDA_X, mode="squash", lam=1.0, want_kappa=False, nthreads=0, lib=None):
    """Run the preconditioned delta rule token by token in fp64 (``pkda_oracle.c``).

    q, k, log_alpha: [B,T,H,dk]; v: [B,T,H,dv]; beta, alpha_p, beta_p: [B,T,H];
    center: [H] (the per-head log-space centre mu_h); S0 [B,H,dk,dv] or None
    (zeros); A0 [B,H,dk] or None (zeros; lambda for "diag_atk").
    mode: "squash" (the trained write key, Preconditioned DeltaNet Eq. 9),
    "diag_atk" (diagonal statistic with the Sherman-Morrison normaliser,
    App. C.2) or "exact_atk" (dense apply-to-key, Theorem 3.1, P_0 = I / lam).
    Returns a dict with o [B,T,H,dv], S_T, A_T [B,H,dk] and optionally kappa
    = beta * k_til [B,T,H,dk].  ``lib`` selects another build of the oracle
    (used by the mutation test).
    """
    md = PKDA_MODES[mode]
    q, k, v, la, be = (_f64(t) for t in (q, k, v, log_alpha, beta))
    ap, bp, ce, S0, A0 = (_f64(t) for t in (alpha_p, beta_p, center, S0, A0))
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    assert k.shape == (B, T, H, dk) and la.shape == (B, T, H, dk)
    assert v.shape == (B, T, H, dv) and be.shape == (B, T, H)
    if md == 0:
        assert ap.shape == (B, T, H) and bp.shape == (B, T, H) and ce.shape == (H,)
    if S0 is not None:
        assert S0.shape == (B, H, dk, dv)
    if A0 is not None:
        assert A0.shape == (B, H, dk)
    o = np.zeros((B, T, H, dv))
    S_T = np.zeros((B, H, dk, dv))
    A_T = np.zeros((B, H, dk))
    kap = np.zeros((B, T, H, dk)) if want_kappa else None
    rc = (lib or _load()).pkda_oracle_forward(
        md, B, T, H, dk, dv, float(x), float(lam),
        _ptr(q), _ptr(k), _ptr(v), _ptr(la), _ptr(be), _ptr(ap), _ptr(bp), _ptr(ce),
        _ptr(S0), _ptr(A0), _ptr(o), _ptr(S_T), _ptr(A_T), _ptr(kap), int(nthreads),
    )
    if rc != 0:
        raise RuntimeError(f"pkda_oracle_forward failed with code {rc}")
    out = {"o": o, "S_T": S_T, "A_T": A_T}
    if want_kappa:
        out["kappa"] = kap
    return out


def pkda_step(q, k, v, log_alpha, beta, alpha_p, beta_p, center, S, A, x=PKDA_X):
    """One token of the PKDA recurrence for B sequences: inputs [B,H,d] / [B,H];
    S [B,H,dk,dv], A [B,H,dk] before the token.  Returns (o [B,H,dv], S_new, A_new)."""
    add_t = lambda t: None if t is None else np.asarray(t, dtype=np.float64)[:, None]
    out = pkda_forward(add_t(q), add_t(k), add_t(v), add_t(log_alpha), add_t(beta), add_t(alpha_p),
                       add_t(beta_p), center, S, A, x=x)
    return out["o"][:, 0], out["S_T"], out["A_T"]
