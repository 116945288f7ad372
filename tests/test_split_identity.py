"""The algebra behind the sequence split, checked on the fp64 oracle alone.

For fixed gains the KDN state update (KDN paper Sec. 3.2, Eq. 12-17) is affine
in the state, and the gains depend only on the uncertainty recurrence.  So a
segment that starts from S_in with the variances p_in maps S_in to
S_out = Phi S_in + S_loc, and its outputs are o_t = o_loc,t + S_in^T (Phi_t^T q_t),
where (o_loc, S_loc) come from running the segment from S = 0 and
(Phi_t^T q_t, Phi) from running it from S = I with zero values, both from p_in.
The GPU split kernels rely on exactly these identities; here they are checked
against the unsplit oracle run, for the Diagonal and Isotropic variants, to
fp64 rounding.
"""
import numpy as np
import pytest

import oracle
from uncertainty_aware_delta_gb300.inputs import make_inputs


@pytest.mark.parametrize("variant", ["diag", "iso"])
def test_segment_outputs_and_state_are_affine_in_the_initial_state(variant):
    B, T, H, d, cut = 1, 40, 2, 8, 23
    x = make_inputs(variant, B, T, H, d, d, io="f32", seed=606)
    rng = np.random.default_rng(606)
    S0 = rng.standard_normal((B, H, d, d))
    p0 = rng.uniform(0.5, 2.0, size=(B, H, d) if variant == "diag" else (B, H))
    names = ("q", "k", "v", "log_alpha", "omega", "r")
    whole = oracle.forward(variant, *(x[n] for n in names), S0=S0, p0=p0)

    first = oracle.forward(variant, *(x[n][:, :cut] for n in names), S0=S0, p0=p0)
    seg = {n: x[n][:, cut:] for n in names}
    S_in, p_in = first["S_T"], first["p_T"]
    loc = oracle.forward(variant, *(seg[n] for n in names), S0=np.zeros_like(S0), p0=p_in)
    ident = np.broadcast_to(np.eye(d), (B, H, d, d))
    seg0 = dict(seg, v=np.zeros_like(seg["v"]))
    phi = oracle.forward(variant, *(seg0[n] for n in names), S0=ident, p0=p_in)

    # o_t = o_loc,t + S_in^T q~_t with q~_t = Phi_t^T q_t (the outputs of the S = I run)
    o2 = loc["o"] + np.einsum("bhij,bthi->bthj", S_in, phi["o"])
    S_T = np.einsum("bhik,bhkj->bhij", phi["S_T"], S_in) + loc["S_T"]
    scale = np.max(np.abs(whole["o"]))
    assert np.max(np.abs(o2 - whole["o"][:, cut:])) <= 1e-12 * scale
    assert np.max(np.abs(S_T - whole["S_T"])) <= 1e-12 * np.max(np.abs(whole["S_T"]))
    # the variances never see S: both segment runs end where the whole run does
    assert np.allclose(loc["p_T"], whole["p_T"], rtol=1e-13, atol=0)
    assert np.allclose(phi["p_T"], whole["p_T"], rtol=1e-13, atol=0)
    # and the map is not trivial: the correction term carries a real part of o
    assert np.max(np.abs(o2 - loc["o"])) > 1e-3 * scale
