"""ctypes wrapper over the fp64 token-by-token KDN recurrence (``kdn_oracle.c``).

TEST INFRASTRUCTURE ONLY (see the package docstring).

The C file is compiled with the host ``gcc`` into ``oracle/libkdn_oracle.so``
by :func:`build_oracle` (called from ``__graft_entry__.build()``); it is
rebuilt whenever the source is newer than the library.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kdn_oracle.c")
_LIB = os.path.join(_HERE, "libkdn_oracle.so")
_lock = threading.Lock()
_lib = None

DIAG, ISO = 0, 1


def library_path() -> str:
    return _LIB


def build_oracle(force: bool = False) -> str:
    """Compile the oracle C file into a shared library (plain gcc, -O2, no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm", "-lpthread"]
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
