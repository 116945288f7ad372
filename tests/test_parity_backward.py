"""GPU backward (kdn_backward) parity against the fp64 adjoint oracle.

The oracle (oracle/backward.py) is the step-by-step adjoint of the token
recurrence, pinned by central finite differences of the C oracle's forward.
The CUDA path is called through the C ABI; both sides see the same rounded
inputs and the same upstream gradients dO, dS_T, dp_T.  Every gradient (q, k,
v, log_alpha, omega, r, S0, p0) is compared element by element.

Tolerances: those of the forward.  fp32 inputs: the rms-floor relative error,
bound 1e-4 (measured: at most 4e-6 on these cases); bf16 inputs: the normalised
max-abs error, bound 2e-2 (the backward computes in fp32 on the rounded bf16
inputs, so it lands far inside: about 6e-7).
"""
import numpy as np
import pytest

from kdn_testutil import max_rel, norm_max_abs, to_host
from oracle.backward import forward_backward
from uncertainty_aware_delta_gb300.inputs import make_inputs

pytestmark = pytest.mark.gpu

GRADS = ("q", "k", "v", "log_alpha", "omega", "r", "S0", "p0")
FP32_BW_TOL = 1e-4
BF16_BW_TOL = 2e-2


def _kdn():
    import uncertainty_aware_delta_gb300 as kdn
    from uncertainty_aware_delta_gb300.build import build_library

    build_library()
    return kdn


def _case(variant, B, T, H, dk, dv, io, seed, with_state=True, upstream=("o", "S", "p")):
    x = make_inputs(variant, B, T, H, dk, dv, io=io, seed=seed)
    rng = np.random.default_rng(seed + 1)
    pshape = (B, H, dk) if variant == "diag" else (B, H)
    S0 = (0.3 * rng.standard_normal((B, H, dk, dv))).astype(np.float32) if with_state else None
    p0 = rng.uniform(0.3, 2.0, size=pshape).astype(np.float32) if with_state else None
    dO = rng.standard_normal((B, T, H, dv)).astype(np.float32) if "o" in upstream else None
    if dO is not None and io == "bf16":
        from uncertainty_aware_delta_gb300.inputs import round_bf16
        dO = round_bf16(dO)
    dS = rng.standard_normal((B, H, dk, dv)).astype(np.float32) if "S" in upstream else None
    dp = rng.standard_normal(pshape).astype(np.float32) if "p" in upstream else None
    return x, S0, p0, dO, dS, dp


def _run_gpu(kdn, variant, x, S0, p0, dO, dS, dp, mu):
    import torch

    dev = "cuda"
    iot = torch.bfloat16 if x["io"] == "bf16" else torch.float32
    t = {n: torch.from_numpy(np.ascontiguousarray(x[n])).to(dev) for n in ("q", "k", "v", "log_alpha", "omega", "r")}
    for n in ("q", "k", "v"):
        t[n] = t[n].to(iot)
    opt = lambda a, dt=torch.float32: None if a is None else torch.from_numpy(a).to(dev).to(dt)
    g = kdn.kdn_backward(variant, t["q"], t["k"], t["v"], t["log_alpha"], t["omega"], t["r"], opt(S0), opt(p0),
                         opt(dO, iot), opt(dS), opt(dp), mu=mu)
    return {n: to_host(g[n]) for n in GRADS}


def _compare(got, ref, io, what):
    errs = {}
    for n in GRADS:
        e = max_rel(got[n], ref[n]) if io == "f32" else norm_max_abs(got[n], ref[n])
        errs[n] = e
    print(f"[parity] backward {what}: " + ", ".join(f"{n} {e:.2e}" for n, e in errs.items()))
    bound = FP32_BW_TOL if io == "f32" else BF16_BW_TOL
    assert all(np.isfinite(got[n]).all() for n in GRADS), what
    assert max(errs.values()) <= bound, (what, errs)
    return errs


CASES = [
    # variant, B, T, H, dk, dv, io, mu, with_state
    ("diag", 1, 16, 1, 16, 16, "f32", None, True),
    ("iso", 1, 16, 1, 16, 16, "f32", None, True),
    ("diag", 2, 37, 2, 16, 32, "f32", None, True),     # ragged tail, dk != dv
    ("iso", 2, 37, 2, 32, 16, "f32", 1.0, True),
    ("diag", 1, 100, 2, 32, 32, "f32", 1.0, False),
    ("iso", 1, 100, 1, 64, 64, "f32", None, False),
    ("diag", 1, 1, 3, 16, 16, "f32", None, True),        # a single token
    ("diag", 1, 70, 2, 128, 128, "f32", None, True),
    ("iso", 1, 70, 1, 128, 128, "f32", None, True),
    ("diag", 1, 80, 2, 128, 128, "bf16", None, True),
    ("iso", 2, 50, 1, 64, 64, "bf16", None, True),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(map(str, c)))
def test_backward_matches_oracle(case):
    variant, B, T, H, dk, dv, io, mu, with_state = case
    kdn = _kdn()
    x, S0, p0, dO, dS, dp = _case(variant, B, T, H, dk, dv, io, seed=2000 + T + dk, with_state=with_state)
    got = _run_gpu(kdn, variant, x, S0, p0, dO, dS, dp, mu)
    _, ref = forward_backward(variant, x["q"], x["k"], x["v"], x["log_alpha"], x["omega"], x["r"], S0=S0, p0=p0,
                              mu=mu, dO=dO, dS_T=dS, dp_T=dp)
    _compare(got, ref, io, "-".join(map(str, case)))


@pytest.mark.parametrize("variant", ["diag", "iso"])
def test_backward_single_upstream_gradients(variant):
    """Each upstream gradient alone (dO only, dS_T only, dp_T only): the three paths
    of the adjoint separately."""
    kdn = _kdn()
    for up in (("o",), ("S",), ("p",)):
        x, S0, p0, dO, dS, dp = _case(variant, 1, 40, 2, 32, 32, "f32", seed=77, upstream=up)
        got = _run_gpu(kdn, variant, x, S0, p0, dO, dS, dp, None)
        _, ref = forward_backward(variant, x["q"], x["k"], x["v"], x["log_alpha"], x["omega"], x["r"], S0=S0,
                                  p0=p0, dO=dO, dS_T=dS, dp_T=dp)
        _compare(got, ref, "f32", f"{variant} upstream {up}")


def test_backward_empty_sequence_passes_the_state_gradients():
    import torch

    kdn = _kdn()
    B, H, d = 2, 2, 16
    x = make_inputs("diag", B, 0, H, d, d, io="f32", seed=1)
    t = {n: torch.from_numpy(x[n]).cuda() for n in ("q", "k", "v", "log_alpha", "omega", "r")}
    dS = torch.randn(B, H, d, d, device="cuda")
    dp = torch.randn(B, H, d, device="cuda")
    g = kdn.kdn_backward("diag", t["q"], t["k"], t["v"], t["log_alpha"], t["omega"], t["r"], dS_T=dS, dp_T=dp)
    assert torch.equal(g["S0"], dS) and torch.equal(g["p0"], dp)


def test_backward_strong_decay():
    """Chunks with strong decay on one head (log alpha = -1.5 per token): the
    backward's chunk factors use the mid-chunk reference; gradients still match."""
    kdn = _kdn()
    x, S0, p0, dO, dS, dp = _case("diag", 1, 48, 2, 32, 32, "f32", seed=91)
    x["log_alpha"][:, :, 0] = -1.5
    got = _run_gpu(kdn, "diag", x, S0, p0, dO, dS, dp, None)
    _, ref = forward_backward("diag", x["q"], x["k"], x["v"], x["log_alpha"], x["omega"], x["r"], S0=S0, p0=p0,
                              dO=dO, dS_T=dS, dp_T=dp)
    _compare(got, ref, "f32", "strong decay")


def test_backward_directional_derivative_at_headline_shape():
    """At the full headline shape (B8 H16 T4096 d128, bf16 io) the backward runs in
    the benchmark's configuration; a property that holds at any size checks it: for a
    random direction d_v of the values, the directional derivative <grad_v, d_v> of
    L = sum(dO o) equals (L(v + e d_v) - L(v - e d_v)) / 2e through the (linear in v)
    forward -- exact up to rounding because o is affine in v for fixed gains.  The
    CUDA-core fp32 forward evaluates L.  Every head's gradients are also checked
    finite; two heads are compared element by element with the oracle on a
    1024-token prefix-free run below."""
    import torch

    kdn = _kdn()
    from uncertainty_aware_delta_gb300.inputs import WORKLOADS, workload_inputs

    w = WORKLOADS["diag-bf16-b8h16t4096d128"]
    x = workload_inputs(w)
    dev = "cuda"
    t = {n: torch.from_numpy(np.ascontiguousarray(x[n])).to(dev) for n in ("q", "k", "v", "log_alpha", "omega", "r")}
    for n in ("q", "k", "v"):
        t[n] = t[n].to(torch.bfloat16)
    g = torch.Generator(device=dev)
    g.manual_seed(5)
    dO = torch.randn(w.B, w.T, w.H, w.d, device=dev, generator=g).to(torch.bfloat16)
    grads = kdn.kdn_backward("diag", t["q"], t["k"], t["v"], t["log_alpha"], t["omega"], t["r"], dO=dO)
    for n in GRADS:
        assert torch.isfinite(grads[n]).all(), n
    # o is affine in v for fixed gains: L(v) = <dO, o(v)> is linear plus a constant
    dvdir = torch.randn(w.B, w.T, w.H, w.d, device=dev, generator=g)
    qf, kf = t["q"].float(), t["k"].float()

    def L(vv):
        o, _, _ = kdn.kdn_diag_forward(qf, kf, vv, t["log_alpha"], t["omega"], t["r"], chunk=64)
        return float((o.double() * dO.double()).sum())

    vf = t["v"].float()
    eps = 1.0
    fd = (L(vf + eps * dvdir) - L(vf - eps * dvdir)) / (2 * eps)
    an = float((grads["v"].double() * dvdir.double()).sum())
    assert abs(fd - an) <= 2e-3 * max(abs(an), 1.0), (fd, an)
    print(f"[parity] backward headline shape: <grad_v, d> {an:.6e} vs central difference {fd:.6e}")


@pytest.mark.parametrize("variant", ["diag", "iso"])
def test_backward_long_sequence_two_heads(variant):
    """1024 tokens of two d = 128 heads (bf16 io): every gradient element against
    the oracle over a sequence 16 times longer than the memory-adjoint chunk and 16
    checkpoint blocks of the gain adjoint."""
    kdn = _kdn()
    x, S0, p0, dO, dS, dp = _case(variant, 1, 1024, 2, 128, 128, "bf16", seed=4242)
    got = _run_gpu(kdn, variant, x, S0, p0, dO, dS, dp, None)
    _, ref = forward_backward(variant, x["q"], x["k"], x["v"], x["log_alpha"], x["omega"], x["r"], S0=S0, p0=p0,
                              dO=dO, dS_T=dS, dp_T=dp)
    _compare(got, ref, "bf16", f"{variant} T=1024 d=128")
