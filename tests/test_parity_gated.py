"""GPU parity of the gated forward (kdn_gated_forward) against the fp64 oracle.

The oracle (oracle/gates.py) applies the gate branches of the KDN reading notes
Sec. 5.1 (alpha = sigma(a), omega = softplus(w), r = r_min + softplus(rho)) to
the same logits the GPU sees (bf16-rounded for bf16 io), runs the pinned fp64
recurrence on them, and forms beta_eff = k^T kappa from its gains (Sec. 3.2;
App. B, Eq. 58-61).  The CUDA path is called through the C ABI.

Paths covered: the gate prologue followed by the fused tensor-core kernel (bf16,
d = 128, chunk 64, whole sequences) over several chunks with a ragged tail, given
initial states, and strongly decaying chunks (mid-chunk decay reference); the
CUDA-core path (fp32 io, small d; beta_eff from the gain scan's gains); the
sequence split (beta_eff off: the split path; beta_eff on: whole sequences); T = 0;
and the full gated headline workload in the benchmark's launch configuration,
every sequence.

Tolerances: those of the ungated forward (kdn_testutil): fp32 max_rel 1e-4, bf16
norm_max_abs 2e-2, for o, S_T, p_T and beta_eff alike.
"""
import numpy as np
import pytest

from kdn_testutil import err, report, to_host, tol
from oracle import gates
from uncertainty_aware_delta_gb300.inputs import WORKLOADS, make_gated_inputs, workload_inputs

pytestmark = pytest.mark.gpu

LOGITS = ("alpha_logit", "omega_logit", "r_logit")


def _kdn():
    import uncertainty_aware_delta_gb300 as kdn
    from uncertainty_aware_delta_gb300.build import build_library

    build_library()
    return kdn


def _dev(x, dev="cuda"):
    import torch

    iot = torch.bfloat16 if x["io"] == "bf16" else torch.float32
    # exact: the stored values are representable in the io dtype
    return {n: torch.from_numpy(np.ascontiguousarray(x[n])).to(dev).to(iot) for n in ("q", "k", "v") + LOGITS}


def _run(kdn, variant, t, **kw):
    return kdn.kdn_gated_forward(variant, t["q"], t["k"], t["v"], t["alpha_logit"], t["omega_logit"],
                                 t["r_logit"], **kw)


def _oracle(variant, x, **kw):
    return gates.gated_forward(variant, x["q"], x["k"], x["v"], x["alpha_logit"], x["omega_logit"],
                               x["r_logit"], **kw)


def _check(what, got, ref, io, with_beta=True):
    o, S_T, p_T, be = got
    res = {"o": to_host(o), "S_T": to_host(S_T), "p_T": to_host(p_T)}
    if with_beta:
        res["beta_eff"] = to_host(be)
    for n, a in res.items():
        assert np.all(np.isfinite(a)), (what, n)
    e = {n: err(a, ref[n], io) for n, a in res.items()}
    report(f"gated {what}", res, {n: ref[n] for n in res}, io)
    assert all(v <= tol(io) for v in e.values()), (what, e)
    return e


TC_CASES = [
    # variant, B, T, H   (bf16 io, d_k = d_v = 128, chunk 64: the fused gated kernel)
    ("diag", 2, 333, 3), ("iso", 2, 333, 3), ("diag", 1, 50, 2), ("iso", 1, 64, 2), ("diag", 1, 1, 2),
    ("diag", 3, 128, 1),
]


@pytest.mark.parametrize("case", TC_CASES, ids=lambda c: "-".join(map(str, c)))
def test_gated_tensor_core_path_matches_oracle(case):
    import torch

    variant, B, T, H = case
    kdn = _kdn()
    x = make_gated_inputs(variant, B, T, H, 128, 128, io="bf16", seed=700 + T)
    rng = np.random.default_rng(T + 1)
    S0 = (0.2 * rng.standard_normal((B, H, 128, 128))).astype(np.float32)
    p0 = rng.uniform(0.3, 2.0, size=(B, H, 128) if variant == "diag" else (B, H)).astype(np.float32)
    t = _dev(x)
    ref = _oracle(variant, x, S0=S0, p0=p0)
    got = _run(kdn, variant, t, S0=torch.from_numpy(S0).cuda(), p0=torch.from_numpy(p0).cuda(), chunk=64,
               beta_eff=True)
    _check(f"{variant} tensor-core B{B} T{T} H{H}", got, ref, "bf16")
    # without beta_eff the outputs do not change
    o2, S2, p2, be2 = _run(kdn, variant, t, S0=torch.from_numpy(S0).cuda(), p0=torch.from_numpy(p0).cuda(),
                           chunk=64)
    assert be2 is None
    assert torch.equal(o2, got[0]) and torch.equal(S2, got[1]) and torch.equal(p2, got[2])


@pytest.mark.parametrize("variant", ["diag", "iso"])
def test_gated_tensor_core_path_strong_decay(variant):
    """Head 0 decays by about 1.5 per token (alpha logit -1.26: log sigma = -1.5),
    so every chunk of 64 tokens exceeds the start-reference bound (80) and takes
    the mid-chunk reference; small r and large omega keep the carried state
    relevant."""
    kdn = _kdn()
    B, T, H = 2, 200, 2
    x = make_gated_inputs(variant, B, T, H, 128, 128, io="bf16", seed=78)
    from uncertainty_aware_delta_gb300.inputs import round_bf16

    x["alpha_logit"][:, :, 0] = round_bf16(np.full(x["alpha_logit"][:, :, 0].shape, -1.26, np.float32))
    x["r_logit"][:, :, 0] = round_bf16(np.full(x["r_logit"][:, :, 0].shape, -6.0, np.float32))
    x["omega_logit"][:, :, 0] = round_bf16(np.full(x["omega_logit"][:, :, 0].shape, 0.5, np.float32))
    t = _dev(x)
    ref = _oracle(variant, x)
    assert np.all(ref["log_alpha"][:, :, 0] < -1.45)
    got = _run(kdn, variant, t, chunk=64, beta_eff=True)
    _check(f"{variant} strong decay", got, ref, "bf16")


@pytest.mark.parametrize("variant", ["diag", "iso"])
@pytest.mark.parametrize("r_min", [None, 0.2])
def test_cuda_core_gated_path_matches_oracle(variant, r_min):
    """fp32 io (and d != 128): the CUDA-core path on the expanded gates, beta_eff
    from its gains."""
    kdn = _kdn()
    B, T, H, dk, dv = 2, 150, 3, 64, 32
    x = make_gated_inputs(variant, B, T, H, dk, dv, io="f32", seed=91)
    t = _dev(x)
    ref = _oracle(variant, x, r_min=gates.R_MIN if r_min is None else r_min)
    got = _run(kdn, variant, t, chunk=32, r_min=r_min, beta_eff=True)
    _check(f"{variant} cuda-core r_min={r_min}", got, ref, "f32")


@pytest.mark.parametrize("variant", ["diag", "iso"])
def test_portable_flag_on_tensor_core_shape(variant):
    """KDN_FLAG_PORTABLE on the tensor-core shape: the CUDA-core path with bf16 io."""
    kdn = _kdn()
    x = make_gated_inputs(variant, 1, 130, 2, 128, 128, io="bf16", seed=93)
    t = _dev(x)
    ref = _oracle(variant, x)
    got = _run(kdn, variant, t, chunk=64, flags=kdn.KDN_FLAG_PORTABLE, beta_eff=True)
    _check(f"{variant} portable bf16", got, ref, "bf16")


@pytest.mark.parametrize("variant", ["diag", "iso"])
def test_sequence_split_with_and_without_beta_eff(variant):
    """Two sequences of 2048 tokens split into segments on the tensor-core path:
    without beta_eff the gates go through the split; with it the fused kernel runs
    whole sequences.  Both match the oracle."""
    kdn = _kdn()
    vcode = kdn.KDN_DIAG if variant == "diag" else kdn.KDN_ISO
    assert kdn.forward_kernel_count(vcode, 1, 2048, 2, 128, 128, 64, kdn.KDN_BF16, 0) == 6
    x = make_gated_inputs(variant, 1, 2048, 2, 128, 128, io="bf16", seed=95)
    t = _dev(x)
    ref = _oracle(variant, x)
    split = _run(kdn, variant, t, chunk=64)
    _check(f"{variant} split", split, ref, "bf16", with_beta=False)
    whole = _run(kdn, variant, t, chunk=64, beta_eff=True)
    _check(f"{variant} split shape, beta_eff", whole, ref, "bf16")


def test_empty_sequence_copies_state():
    import torch

    kdn = _kdn()
    x = make_gated_inputs("diag", 2, 0, 2, 128, 128, io="bf16", seed=1)
    t = _dev(x)
    S0 = torch.randn(2, 2, 128, 128, device="cuda")
    p0 = torch.rand(2, 2, 128, device="cuda") + 0.5
    o, S_T, p_T, be = _run(kdn, "diag", t, S0=S0, p0=p0, beta_eff=True)
    assert o.shape == (2, 0, 2, 128) and be.shape == (2, 0, 2)
    assert torch.equal(S_T, S0) and torch.equal(p_T, p0)


def test_gated_headline_workload_every_sequence():
    """The gated headline workload (B8 H16 T4096 d128, bf16, beta_eff off as the
    benchmark times it, then on) against the oracle on every (b, h) sequence."""
    kdn = _kdn()
    w = WORKLOADS["gated-diag-bf16-b8h16t4096d128"]
    x = workload_inputs(w)
    t = _dev(x)
    got = _run(kdn, "diag", t, chunk=w.chunk, beta_eff=True)
    plain = _run(kdn, "diag", t, chunk=w.chunk)
    import torch

    assert torch.equal(plain[0], got[0]) and torch.equal(plain[1], got[1])
    res = [to_host(a) for a in got]
    del t, got, plain
    ref = _oracle("diag", x)
    e = _check(w.name, res, ref, w.io)
    worst = 0.0
    for b in range(w.B):
        for h in range(w.H):
            eo = err(res[0][b, :, h], ref["o"][b, :, h], w.io)
            es = err(res[1][b, h], ref["S_T"][b, h], w.io)
            eb = err(res[3][b, :, h], ref["beta_eff"][b, :, h], w.io)
            worst = max(worst, eo, es, eb)
            assert max(eo, es, eb) <= tol(w.io), (b, h, eo, es, eb)
    print(f"[parity] {w.name}: worst per-sequence error {worst:.2e} (tensor-wide {e})")
