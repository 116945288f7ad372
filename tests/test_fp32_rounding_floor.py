"""Evidence for the fp32 error metric's floor (the reading of "max relative
error <= 1e-4" that the fp32 parity tests use).

A plain fp32 restatement of the token recurrence (KDN paper Sec. 4.1 Eq. 23-27
and 60-65 for the Diagonal variant, Sec. 4.2 Eq. 40 and App. C for the
Isotropic one; written here with numpy float32, vectorised over the
sequences, one token at a time) is compared with the fp64 oracle on d = 128
inputs.  No blocking, no reordering beyond fp32 rounding: any fp32
implementation of the method carries at least this error.

Measured with three floors of the per-element relative error
|x - y| / max(|y|, floor):
  * floor = rms(y)         (the metric the fp32 tests assert, bound 1e-4),
  * floor = 1e-2 * rms(y)  (a stricter reading of the bound),
  * no floor               (pure element-wise).
The plain fp32 run stays far inside 1e-4 under the rms floor (about 3e-6),
while under the 1%-of-rms floor it already exceeds the bound (about 1.4e-4
Diagonal, 1.7e-4 Isotropic), set by outputs near zero: that floor would
measure fp32 rounding of near-zero outputs, not the kernels.
"""
import numpy as np
import pytest

import oracle
from uncertainty_aware_delta_gb300.inputs import make_inputs


def fp32_recurrence(variant, x, mu):
    """The token recurrence in float32 (no chunking): returns o, S_T, p_T."""
    f = np.float32
    q, k, v = (x[n].astype(f) for n in ("q", "k", "v"))
    la, om, r = x["log_alpha"].astype(f), x["omega"].astype(f), x["r"].astype(f)
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    S = np.zeros((B, H, dk, dv), f)
    p = np.ones((B, H, dk) if variant == "diag" else (B, H), f)
    o = np.zeros((B, T, H, dv), f)
    mu = f(mu)
    for t in range(T):
        a = np.exp(la[:, t])                                  # [B,H,dk]
        kt, vt, qt, rt = k[:, t], v[:, t], q[:, t], r[:, t]
        if variant == "diag":
            ph = a * a * p + om[:, t]                          # predicted variances
            z = rt + np.sum(ph * kt * kt, axis=-1)
            kap = ph * kt / z[..., None]
        else:
            ph = np.mean(a * a, axis=-1) * p + om[:, t]        # predicted scalar variance
            beta = ph / (rt + ph * np.sum(kt * kt, axis=-1))
            kap = beta[..., None] * kt
        Sh = a[..., None] * S                                  # diag(a) S
        delta = vt - np.einsum("bhij,bhi->bhj", Sh, kt)
        S = Sh + kap[..., None] * delta[..., None, :]
        o[:, t] = np.einsum("bhij,bhi->bhj", S, qt)
        if variant == "diag":
            u = (mu / rt)[..., None] * kt * kt
        else:
            u = mu * np.sum(kt * kt, axis=-1) / (f(dk) * rt)
        p = ph / (f(1) + u * ph)
    return o, S, p


def rel_err(x, y, floor_frac):
    x = np.asarray(x, np.float64)
    y = np.asarray(y, np.float64)
    floor = floor_frac * np.sqrt(np.mean(y * y)) if floor_frac > 0 else 1e-300
    return float(np.max(np.abs(x - y) / np.maximum(np.abs(y), floor)))


@pytest.mark.parametrize("variant", ["diag", "iso"])
def test_plain_fp32_recurrence_error_by_floor(variant):
    x = make_inputs(variant, 1, 512, 4, 128, 128, io="f32", seed=4242)
    ref = oracle.forward(variant, x["q"], x["k"], x["v"], x["log_alpha"], x["omega"], x["r"])
    got = fp32_recurrence(variant, x, 128.0)
    rows = {}
    for name, g, y in zip(("o", "S_T", "p_T"), got, (ref["o"], ref["S_T"], ref["p_T"])):
        rows[name] = (rel_err(g, y, 1.0), rel_err(g, y, 1e-2), rel_err(g, y, 0.0))
    print(variant, {n: tuple(f"{e:.2e}" for e in r) for n, r in rows.items()})
    # rms floor: fp32 rounding alone stays an order of magnitude inside the 1e-4 bound
    assert max(r[0] for r in rows.values()) <= 2e-5, rows
    # 1%-of-rms floor: the same fp32 run already exceeds the 1e-4 bound on o
    # (1.4e-4 Diagonal, 1.7e-4 Isotropic with this seed)
    assert rows["o"][1] > 1e-4, rows
    # element-wise without a floor: larger still (near-zero outputs dominate)
    assert rows["o"][2] >= rows["o"][1], rows
