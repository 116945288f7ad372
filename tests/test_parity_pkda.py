"""GPU parity of the preconditioned delta rule with per-channel decay (PKDA,
Preconditioned DeltaNet Sec. 2.4 Eq. 9 and Sec. 2.5) against its fp64 oracle.

The CUDA path is called through the C ABI (the ctypes binding): the fused
tensor-core kernel for bf16 io with d_k = d_v = 128 and chunk 64, the
CUDA-core path (statistic scan + chunk pass) otherwise.  Cases span several
chunks and a ragged tail, given initial states, in-place resume, T = 0, the
write-scale bound x = 1, a statistic pushed above the log-space centre, key
channels that stay zero (the statistic's logarithm floor), strong decay, the
full-size workload (sampled) and single-token decode.
"""
import numpy as np
import pytest

from kdn_testutil import err, max_rel, to_host, tol
from oracle import recurrence
from uncertainty_aware_delta_gb300.inputs import WORKLOADS, make_pkda_inputs, workload_inputs

pytestmark = pytest.mark.gpu

NAMES = ("q", "k", "v", "log_alpha", "beta", "alpha_p", "beta_p", "center")


def _kdn():
    import uncertainty_aware_delta_gb300 as kdn
    from uncertainty_aware_delta_gb300.build import build_library

    build_library()
    return kdn


def _dev(x, dev="cuda:0"):
    import torch

    out = {}
    for n in NAMES:
        t = torch.from_numpy(np.ascontiguousarray(x[n]))
        if n in ("q", "k", "v") and x["io"] == "bf16":
            t = t.to(torch.bfloat16)
        out[n] = t.to(dev)
    return out


def _ref(inp, **kw):
    return recurrence.pkda_forward(*(inp[n] for n in NAMES[:5]), alpha_p=inp["alpha_p"], beta_p=inp["beta_p"],
                                   center=inp["center"], **kw)


def _run(kdn, t, **kw):
    return kdn.kdn_pkda_forward(*(t[n] for n in NAMES), **kw)


def _check(got, ref, io, what=""):
    o, S_T, A_T = (to_host(a) for a in got)
    e = {"o": err(o, ref["o"], io), "S_T": err(S_T, ref["S_T"], io), "A_T": max_rel(A_T, ref["A_T"])}
    assert e["o"] <= tol(io) and e["S_T"] <= tol(io) and e["A_T"] <= 1e-4, (what, e)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(S_T))
    return e


CASES = [
    # B, T, H, dk, dv, chunk, io
    (1, 64, 2, 16, 16, 16, "f32"),
    (2, 100, 3, 32, 64, 32, "f32"),         # ragged tail
    (1, 200, 2, 128, 128, 64, "f32"),
    (2, 77, 2, 64, 128, 64, "f32"),
    (2, 300, 2, 128, 128, 64, "bf16"),      # tensor-core path
    (1, 17, 1, 16, 128, 16, "bf16"),
    (1, 1, 3, 128, 128, 64, "f32"),         # a single token
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(map(str, c)))
def test_pkda_forward_matches_oracle(case):
    B, T, H, dk, dv, chunk, io = case
    kdn = _kdn()
    x = make_pkda_inputs(B, T, H, dk, dv, io=io, seed=2000 + T + dk)
    got = _run(kdn, _dev(x), chunk=chunk)
    _check(got, _ref(x), io)


TC_CASES = [(2, 333, 3), (1, 50, 2), (1, 1, 2), (3, 128, 1)]


@pytest.mark.parametrize("case", TC_CASES, ids=lambda c: "-".join(map(str, c)))
def test_pkda_tensor_core_path_with_state(case):
    """The fused kernel from a given (S_0, A_0), against the oracle and the CUDA-core path."""
    import torch

    B, T, H = case
    kdn = _kdn()
    assert kdn.forward_kernel_count(kdn.KDN_PKDA, B, T, H, 128, 128, 64, kdn.KDN_BF16, 0) == 1
    x = make_pkda_inputs(B, T, H, 128, 128, io="bf16", seed=700 + T)
    rng = np.random.default_rng(T)
    S0 = (0.2 * rng.standard_normal((B, H, 128, 128))).astype(np.float32)
    A0 = rng.uniform(0.0, 0.5, size=(B, H, 128)).astype(np.float32)
    t = _dev(x)
    S0d, A0d = torch.from_numpy(S0).cuda(), torch.from_numpy(A0).cuda()
    ref = _ref(x, S0=S0, A0=A0)
    tc = _run(kdn, t, S0=S0d, A0=A0d, chunk=64)
    e = _check(tc, ref, "bf16", "tensor-core")
    simt = _run(kdn, t, S0=S0d, A0=A0d, chunk=64, flags=kdn.KDN_FLAG_PORTABLE)
    _check(simt, ref, "bf16", "portable")
    for a, b_ in zip(tc, simt):
        assert np.max(np.abs(to_host(a) - to_host(b_))) <= 2e-2 * max(1e-3, np.max(np.abs(to_host(b_)))), e


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_pkda_statistic_above_centre(io):
    """beta_p scaled up so log A crosses the centre: both branches of the softsign."""
    kdn = _kdn()
    x = make_pkda_inputs(2, 150, 2, 128, 128, io=io, seed=31, log_alpha_range=(1e-3, 0.05), beta_p_scale=200.0)
    ref = _ref(x, want_kappa=True)
    scale = np.abs(ref["kappa"]) / np.maximum(np.abs(x["k"]) * x["beta"][..., None], 1e-30)
    valid = np.abs(x["k"]) > 1e-3
    assert np.any(scale[valid] < 0.99) and np.any(scale[valid] > 1.01)
    _check(_run(kdn, _dev(x), chunk=64), ref, io)


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_pkda_bound_one_is_the_gated_delta_rule(io):
    """x = 1: every write scale is 1 (Sec. 2.7), the statistic does not matter."""
    kdn = _kdn()
    x = make_pkda_inputs(1, 130, 2, 128, 128, io=io, seed=41)
    ref = _ref(x, x=1.0)
    _check(_run(kdn, _dev(x), x=1.0, chunk=64), ref, io)
    x2 = dict(x)
    x2["beta_p"] = x["beta_p"] * 50.0
    ref2 = _ref(x2, x=1.0)
    assert np.allclose(ref2["o"], ref["o"], rtol=0, atol=1e-12)


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_pkda_zero_key_channels_stay_finite(io):
    """Key channels that are zero at every token keep a zero statistic; its
    logarithm is floored, and nothing turns into NaN."""
    kdn = _kdn()
    x = make_pkda_inputs(1, 100, 2, 128, 128, io=io, seed=51)
    x["k"][..., 3] = 0.0
    x["k"][..., 77] = 0.0
    ref = _ref(x)
    got = _run(kdn, _dev(x), chunk=64)
    _check(got, ref, io)
    assert np.all(to_host(got[2])[..., 3] == 0.0)


def test_pkda_strong_decay_tensor_core():
    """Head 0 decays by 64 x 1.5 = 96 per chunk: the fused kernel's mid-chunk reference."""
    import torch

    kdn = _kdn()
    B, T, H = 2, 200, 2
    x = make_pkda_inputs(B, T, H, 128, 128, io="bf16", seed=61)
    x["log_alpha"][:, :, 0] = -1.5
    ws = torch.empty(kdn.workspace_size(kdn.KDN_PKDA, B, T, H, 128, 128, 64, kdn.KDN_BF16, 0), dtype=torch.uint8,
                     device="cuda")
    got = _run(kdn, _dev(x), chunk=64, workspace=ws)
    assert kdn.kdn_read_device_status(ws) == 0
    _check(got, _ref(x), "bf16", "strong decay")


def test_pkda_in_place_resume_and_continuation():
    import torch

    kdn = _kdn()
    x = make_pkda_inputs(2, 150, 2, 32, 32, io="f32", seed=71)
    t = _dev(x)
    T1 = 70
    first = {n: (v[:, :T1].contiguous() if n != "center" else v) for n, v in t.items()}
    second = {n: (v[:, T1:].contiguous() if n != "center" else v) for n, v in t.items()}
    o1, S1, A1 = _run(kdn, first, chunk=32)
    o2 = torch.empty_like(t["v"][:, T1:])
    _run(kdn, second, S0=S1, A0=A1, chunk=32, out=(o2, S1, A1))   # S_T, A_T alias S0, A0
    _check((torch.cat([o1, o2], 1), S1, A1), _ref(x), "f32", "continuation in place")


def test_pkda_empty_sequence_copies_state():
    import torch

    kdn = _kdn()
    B, H, d = 2, 3, 32
    x = make_pkda_inputs(B, 0, H, d, d, io="f32", seed=1)
    t = _dev(x)
    S0 = torch.randn(B, H, d, d, device="cuda")
    A0 = torch.rand(B, H, d, device="cuda")
    o, S_T, A_T = _run(kdn, t, S0=S0, A0=A0)
    assert o.shape == (B, 0, H, d) and torch.equal(S_T, S0) and torch.equal(A_T, A0)
    o, S_T, A_T = _run(kdn, t)
    assert torch.count_nonzero(S_T) == 0 and torch.count_nonzero(A_T) == 0


def test_pkda_full_size_sampled():
    """The benchmark workload (B = 8, H = 16, T = 4096, d = 128, bf16) in the
    benchmark's launch configuration; sampled sequences against the oracle."""
    kdn = _kdn()
    w = WORKLOADS["pkda-bf16-b8h16t4096d128"]
    x = workload_inputs(w)
    got = _run(kdn, _dev(x), chunk=w.chunk)
    o, S_T, A_T = (to_host(a) for a in got)
    assert np.all(np.isfinite(o))
    for b, h in [(0, 0), (7, 15), (3, 9)]:
        sl = {n: (x[n][b:b + 1, :, h:h + 1] if n != "center" else x[n][h:h + 1]) for n in NAMES}
        sl["io"] = x["io"]
        ref = _ref(sl)
        e = (err(o[b:b + 1, :, h:h + 1], ref["o"], w.io), err(S_T[b:b + 1, h:h + 1], ref["S_T"], w.io),
             max_rel(A_T[b:b + 1, h:h + 1], ref["A_T"]))
        assert e[0] <= tol(w.io) and e[1] <= tol(w.io) and e[2] <= 1e-4, (b, h, e)


@pytest.mark.parametrize("case", [(3, 2, 128, 128, "f32"), (2, 3, 16, 64, "f32"), (2, 2, 128, 128, "bf16"),
                                  # more (sequence, head) pairs than SMs: each persistent CTA of the
                                  # 128 x 128 decode walks several heads through its buffer ring
                                  (100, 4, 128, 128, "f32"), (80, 5, 128, 128, "bf16")],
                         ids=lambda c: "-".join(map(str, c)))
def test_pkda_steps_after_prefill(case):
    import torch

    B, H, dk, dv, io = case
    kdn = _kdn()
    prefill, steps = (40, 12) if B * H < 100 else (8, 3)
    x = make_pkda_inputs(B, prefill + steps, H, dk, dv, io=io, seed=88 + dk)
    t = _dev(x)
    pre = {n: (v[:, :prefill].contiguous() if n != "center" else v) for n, v in t.items()}
    _, S, A = _run(kdn, pre, chunk=16)
    ws = torch.empty(kdn.workspace_size(kdn.KDN_PKDA, B, 1, H, dk, dv), dtype=torch.uint8, device="cuda")
    outs = []
    for s in range(steps):
        tt = prefill + s
        step_in = [t[n][:, tt].contiguous() for n in NAMES[:7]]
        outs.append(kdn.kdn_pkda_step(*step_in, t["center"], S, A, workspace=ws).clone())
    torch.cuda.synchronize()
    ref = _ref(x)
    assert err(to_host(torch.stack(outs, 1)), ref["o"][:, prefill:], io) <= tol(io)
    assert err(to_host(S), ref["S_T"], io) <= tol(io)
    assert max_rel(to_host(A), ref["A_T"]) <= 1e-4


def test_pkda_sequence_split():
    """Few long sequences: the PKDA forward runs as chained segments (statistic
    carries from the scan, affine state maps) and matches the oracle and the
    unsplit kernel."""
    kdn = _kdn()
    B, T, H = 1, 3000, 2
    assert kdn.forward_kernel_count(kdn.KDN_PKDA, B, T, H, 128, 128, 64, kdn.KDN_BF16, 0) == 6
    x = make_pkda_inputs(B, T, H, 128, 128, io="bf16", seed=62)
    t = _dev(x)
    got = _run(kdn, t, chunk=64)
    _check(got, _ref(x), "bf16", "split")
    whole = _run(kdn, t, chunk=64, flags=kdn.KDN_FLAG_NO_SPLIT)
    for a, b_ in zip(got, whole):
        a, b_ = to_host(a), to_host(b_)
        assert np.max(np.abs(a - b_)) <= 2e-2 * max(1e-3, np.max(np.abs(b_)))
