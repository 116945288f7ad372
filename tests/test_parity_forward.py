"""GPU forward parity against the fp64 oracle (Diagonal and Isotropic KDN).

The CUDA path is called through the C ABI (the ctypes binding); the oracle
runs the token-by-token recurrence on the same rounded inputs.  Shapes span
several chunks and a ragged tail; edge cases cover T = 0, given initial
states, in-place resume, the chunk-length invariance and split-sequence
continuation.
"""
import numpy as np
import pytest

import oracle
from kdn_testutil import err, report, to_device, to_host, tol
from uncertainty_aware_delta_gb300.inputs import WORKLOADS, make_inputs, workload_inputs

pytestmark = pytest.mark.gpu


def _kdn():
    import uncertainty_aware_delta_gb300 as kdn
    from uncertainty_aware_delta_gb300.build import build_library

    build_library()
    return kdn


def _run(kdn, variant, t, **kw):
    fn = kdn.kdn_diag_forward if variant == "diag" else kdn.kdn_iso_forward
    return fn(t["q"], t["k"], t["v"], t["log_alpha"], t["omega"], t["r"], **kw)


def _check(variant, x, got, ref, io, what=""):
    o, S_T, p_T = (to_host(a) for a in got)
    e = {"o": err(o, ref["o"], io), "S_T": err(S_T, ref["S_T"], io), "p_T": err(p_T, ref["p_T"], io)}
    report(f"{variant} {what}", {"o": o, "S_T": S_T, "p_T": p_T}, ref, io)
    bound = tol(io)
    assert all(v <= bound for v in e.values()), (variant, what, e)
    return e


CASES = [
    # variant, B, T, H, dk, dv, chunk, io, mu
    ("diag", 1, 64, 2, 16, 16, 16, "f32", None),
    ("iso", 1, 64, 2, 16, 16, 16, "f32", None),
    ("diag", 2, 100, 3, 32, 64, 32, "f32", None),       # ragged tail
    ("iso", 2, 100, 3, 64, 32, 16, "f32", 1.0),
    ("diag", 1, 200, 2, 128, 128, 64, "f32", 1.0),
    ("diag", 2, 77, 2, 64, 64, 64, "f32", 0.0),
    ("iso", 1, 150, 2, 128, 128, 64, "f32", None),
    ("diag", 2, 300, 2, 128, 128, 64, "bf16", None),
    ("iso", 2, 300, 2, 128, 128, 64, "bf16", None),
    ("diag", 1, 1, 3, 128, 128, 64, "f32", None),       # a single token
    ("diag", 1, 17, 1, 16, 128, 16, "bf16", None),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(map(str, c)))
def test_forward_matches_oracle(case):
    variant, B, T, H, dk, dv, chunk, io, mu = case
    kdn = _kdn()
    x = make_inputs(variant, B, T, H, dk, dv, io=io, seed=1000 + T + dk)
    t = to_device(x)
    got = _run(kdn, variant, t, chunk=chunk, mu=mu)
    ref = oracle.forward(variant, x["q"], x["k"], x["v"], x["log_alpha"], x["omega"], x["r"], mu=mu)
    _check(variant, x, got, ref, io)


@pytest.mark.parametrize("variant", ["diag", "iso"])
def test_initial_state_and_in_place_resume(variant):
    import torch

    kdn = _kdn()
    B, T, H, dk, dv = 2, 90, 2, 64, 64
    x = make_inputs(variant, B, T, H, dk, dv, io="f32", seed=5)
    rng = np.random.default_rng(6)
    S0 = (0.3 * rng.standard_normal((B, H, dk, dv))).astype(np.float32)
    p0 = rng.uniform(0.2, 2.0, size=(B, H, dk) if variant == "diag" else (B, H)).astype(np.float32)
    t = to_device(x)
    S0d, p0d = torch.from_numpy(S0).cuda(), torch.from_numpy(p0).cuda()
    ref = oracle.forward(variant, x["q"], x["k"], x["v"], x["log_alpha"], x["omega"], x["r"], S0=S0, p0=p0)
    got = _run(kdn, variant, t, S0=S0d, p0=p0d, chunk=32)
    _check(variant, x, got, ref, "f32", "given state")
    # resume in place: S_T and p_T alias S0 and p0
    o = torch.empty_like(got[0])
    got2 = _run(kdn, variant, t, S0=S0d, p0=p0d, chunk=32, out=(o, S0d, p0d))
    _check(variant, x, got2, ref, "f32", "in place")


@pytest.mark.parametrize("variant", ["diag", "iso"])
def test_chunk_length_does_not_change_the_result(variant):
    kdn = _kdn()
    x = make_inputs(variant, 1, 130, 2, 64, 64, io="f32", seed=9)
    t = to_device(x)
    ref = oracle.forward(variant, x["q"], x["k"], x["v"], x["log_alpha"], x["omega"], x["r"])
    outs = [_run(kdn, variant, t, chunk=c) for c in (16, 32, 64)]
    for got in outs:
        _check(variant, x, got, ref, "f32")
    for a, b in zip(outs[0], outs[2]):
        assert np.max(np.abs(to_host(a) - to_host(b))) <= 1e-4 * max(1.0, np.max(np.abs(to_host(b))))


@pytest.mark.parametrize("variant", ["diag", "iso"])
def test_split_sequence_continuation(variant):
    import torch

    kdn = _kdn()
    x = make_inputs(variant, 2, 150, 2, 32, 32, io="f32", seed=11)
    t = to_device(x)
    T1 = 70
    first = {n: v[:, :T1].contiguous() for n, v in t.items()}
    second = {n: v[:, T1:].contiguous() for n, v in t.items()}
    o1, S1, p1 = _run(kdn, variant, first, chunk=32)
    o2, S2, p2 = _run(kdn, variant, second, S0=S1, p0=p1, chunk=32)
    ref = oracle.forward(variant, x["q"], x["k"], x["v"], x["log_alpha"], x["omega"], x["r"])
    _check(variant, x, (torch.cat([o1, o2], 1), S2, p2), ref, "f32", "continuation")


@pytest.mark.parametrize("variant", ["diag", "iso"])
def test_empty_sequence_copies_state(variant):
    import torch

    kdn = _kdn()
    B, H, d = 2, 3, 32
    x = make_inputs(variant, B, 0, H, d, d, io="f32", seed=1)
    t = to_device(x)
    S0 = torch.randn(B, H, d, d, device="cuda")
    pshape = (B, H, d) if variant == "diag" else (B, H)
    p0 = torch.rand(pshape, device="cuda") + 0.5
    o, S_T, p_T = _run(kdn, variant, t, S0=S0, p0=p0)
    assert o.shape == (B, 0, H, d)
    assert torch.equal(S_T, S0) and torch.equal(p_T, p0)
    o, S_T, p_T = _run(kdn, variant, t)
    assert torch.count_nonzero(S_T) == 0 and torch.all(p_T == 1.0)


def test_empty_batch_is_a_no_op():
    kdn = _kdn()
    x = make_inputs("diag", 0, 10, 2, 16, 16, io="f32", seed=1)
    o, S_T, p_T = _run(kdn, "diag", to_device(x))
    assert o.numel() == 0 and S_T.numel() == 0 and p_T.numel() == 0


def test_device_status_is_ok_after_a_normal_call():
    import torch

    kdn = _kdn()
    x = make_inputs("diag", 1, 64, 1, 16, 16, io="f32", seed=2)
    t = to_device(x)
    ws = torch.empty(kdn.workspace_size(0, 1, 64, 1, 16, 16, 16, 0, 0), dtype=torch.uint8, device="cuda")
    _run(kdn, "diag", t, chunk=16, workspace=ws)
    assert kdn.kdn_read_device_status(ws) == 0


def test_extreme_decay_is_reported_not_faulted():
    """A chunk whose cumulative log-decay exceeds the supported range sets the
    device status word (KDN_ERR_RANGE); the call itself completes."""
    import torch

    kdn = _kdn()
    x = make_inputs("diag", 1, 64, 1, 16, 16, io="f32", seed=3)
    x["log_alpha"][:] = -5.0     # 64 tokens x 5 = 320 > 160
    t = to_device(x)
    ws = torch.empty(kdn.workspace_size(0, 1, 64, 1, 16, 16, 64, 0, 0), dtype=torch.uint8, device="cuda")
    _run(kdn, "diag", t, chunk=64, workspace=ws)
    assert kdn.kdn_read_device_status(ws) == 9


# ------------------------------------------------------------ full-size workloads
def _full_parity(name, variant):
    """Run a full-size workload on the GPU in the benchmark's launch
    configuration and compare EVERY (b, h) sequence, element by element,
    with the oracle on the same inputs (the oracle runs all sequences on the
    host cores)."""
    kdn = _kdn()
    w = WORKLOADS[name]
    x = workload_inputs(w, variant)
    t = to_device(x)
    got = _run(kdn, variant, t, chunk=w.chunk)
    o, S_T, p_T = (to_host(a) for a in got)
    del t, got
    ref = oracle.forward(variant, x["q"], x["k"], x["v"], x["log_alpha"], x["omega"], x["r"])
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(S_T)) and np.all(np.isfinite(p_T))
    e = _check(variant, x, (o, S_T, p_T), ref, w.io, f"{name} all sequences")
    # per sequence as well: a mistake confined to a few (b, h) pairs would be
    # diluted by the tensor-wide normalisation above
    worst = 0.0
    for b in range(w.B):
        for h in range(w.H):
            eo = err(o[b, :, h], ref["o"][b, :, h], w.io)
            es = err(S_T[b, h], ref["S_T"][b, h], w.io)
            worst = max(worst, eo, es)
            assert max(eo, es) <= tol(w.io), (name, variant, b, h, eo, es)
    print(f"[parity] {name} {variant}: worst per-sequence error {worst:.2e}")
    return e


@pytest.mark.parametrize("variant", ["diag", "iso"])
def test_full_size_b8h16t4096(variant):
    _full_parity("diag-bf16-b8h16t4096d128" if variant == "diag" else "iso-bf16-b8h16t4096d128", variant)


@pytest.mark.parametrize("variant", ["diag", "iso"])
def test_full_size_long_context(variant):
    _full_parity("diag-bf16-b1h16t65536d128", variant)


def test_small_workload_every_output():
    w = WORKLOADS["diag-f32-b1h2t64d16"]
    _full_parity(w.name, "diag")
    _full_parity(w.name, "iso")


# ------------------------------------------------------------ tensor-core path
TC_CASES = [
    # variant, B, T, H  (bf16 io, d_k = d_v = 128, chunk 64 -> fused tensor-core kernel)
    ("diag", 2, 333, 3), ("iso", 2, 333, 3), ("diag", 1, 50, 2), ("iso", 1, 50, 2),
    ("diag", 1, 1, 2), ("diag", 3, 128, 1),
]


@pytest.mark.parametrize("case", TC_CASES, ids=lambda c: "-".join(map(str, c)))
def test_tensor_core_path_matches_oracle_and_portable_path(case):
    import torch

    variant, B, T, H = case
    kdn = _kdn()
    vcode = kdn.KDN_DIAG if variant == "diag" else kdn.KDN_ISO
    assert kdn.forward_kernel_count(vcode, B, T, H, 128, 128, 64, kdn.KDN_BF16, 0) == 1
    x = make_inputs(variant, B, T, H, 128, 128, io="bf16", seed=500 + T)
    rng = np.random.default_rng(T)
    S0 = (0.2 * rng.standard_normal((B, H, 128, 128))).astype(np.float32)
    p0 = rng.uniform(0.3, 2.0, size=(B, H, 128) if variant == "diag" else (B, H)).astype(np.float32)
    t = to_device(x)
    S0d, p0d = torch.from_numpy(S0).cuda(), torch.from_numpy(p0).cuda()
    ref = oracle.forward(variant, x["q"], x["k"], x["v"], x["log_alpha"], x["omega"], x["r"], S0=S0, p0=p0)
    tc = _run(kdn, variant, t, S0=S0d, p0=p0d, chunk=64)
    e = _check(variant, x, tc, ref, "bf16", "tensor-core")
    simt = _run(kdn, variant, t, S0=S0d, p0=p0d, chunk=64, flags=kdn.KDN_FLAG_PORTABLE)
    for a, b_ in zip(tc, simt):
        assert np.max(np.abs(to_host(a) - to_host(b_))) <= 2e-2 * max(1e-3, np.max(np.abs(to_host(b_)))), e


@pytest.mark.parametrize("variant", ["diag", "iso"])
def test_tensor_core_path_strong_decay(variant):
    """Chunks whose log-decay exceeds 80 in magnitude (here 64 x 1.5 = 96 on head 0)
    switch the fused kernel to the mid-chunk decay reference; the result must
    still match the oracle, and no range error is reported (|G_C| <= 160)."""
    import torch

    kdn = _kdn()
    B, T, H = 2, 200, 2
    x = make_inputs(variant, B, T, H, 128, 128, io="bf16", seed=77)
    x["log_alpha"][:, :, 0] = -1.5
    # large gains on that head (small observation noise, large process noise), so the
    # state carried from one strongly decaying chunk into the next is not negligible
    x["r"][:, :, 0] = 1e-3
    x["omega"][:, :, 0] = 1.0
    t = to_device(x)
    ws = torch.empty(kdn.workspace_size(kdn.KDN_DIAG if variant == "diag" else kdn.KDN_ISO, B, T, H, 128, 128,
                                        64, kdn.KDN_BF16, 0), dtype=torch.uint8, device="cuda")
    got = _run(kdn, variant, t, chunk=64, workspace=ws)
    assert kdn.kdn_read_device_status(ws) == 0
    ref = oracle.forward(variant, x["q"], x["k"], x["v"], x["log_alpha"], x["omega"], x["r"])
    _check(variant, x, got, ref, "bf16", "strong decay")


@pytest.mark.parametrize("variant", ["diag", "iso"])
def test_tensor_core_path_zero_prior_variance(variant):
    """p_0 = 0 with no process noise on head 0: every gain of that head is zero
    (the isotropic kernel takes its prior variance b_hat into the triangular
    system as r / b_hat, here with b_hat = 0), so its state only decays and its
    final variance stays 0; head 1 runs with an ordinary prior beside it."""
    import torch

    kdn = _kdn()
    B, T, H = 1, 150, 2
    x = make_inputs(variant, B, T, H, 128, 128, io="bf16", seed=31)
    x["omega"][:, :, 0] = 0.0
    rng = np.random.default_rng(31)
    S0 = (0.5 * rng.standard_normal((B, H, 128, 128))).astype(np.float32)
    p0 = np.ones((B, H, 128) if variant == "diag" else (B, H), dtype=np.float32)
    p0[:, 0] = 0.0
    t = to_device(x)
    ref = oracle.forward(variant, x["q"], x["k"], x["v"], x["log_alpha"], x["omega"], x["r"], S0=S0, p0=p0)
    got = _run(kdn, variant, t, S0=torch.from_numpy(S0).cuda(), p0=torch.from_numpy(p0).cuda(), chunk=64)
    _check(variant, x, got, ref, "bf16", "zero prior variance")
    assert np.all(to_host(got[2])[:, 0] == 0.0)
    assert np.all(np.isfinite(to_host(got[0]))) and np.all(np.isfinite(to_host(got[1])))


# ------------------------------------------------------------ sequence split
SPLIT_CASES = [
    # variant, B, T, H, with an initial state: few long sequences -> segments on separate SMs
    ("diag", 1, 4096, 2, False),    # 4 segments of 1024 tokens
    ("iso", 1, 4096, 2, False),
    ("diag", 1, 4000, 2, True),     # 3 segments, the last with a ragged tail; resume from a state
    ("iso", 2, 2600, 1, True),
]


@pytest.mark.parametrize("case", SPLIT_CASES, ids=lambda c: "-".join(map(str, c)))
def test_sequence_split_matches_oracle_and_unsplit_run(case):
    """The tensor-core forward of few long sequences runs each sequence as
    segments chained through their affine state maps; it must match the
    oracle, and the unsplit kernel on the same inputs."""
    import torch

    variant, B, T, H, with_state = case
    kdn = _kdn()
    vcode = kdn.KDN_DIAG if variant == "diag" else kdn.KDN_ISO
    assert kdn.forward_kernel_count(vcode, B, T, H, 128, 128, 64, kdn.KDN_BF16, 0) == 6
    assert kdn.forward_kernel_count(vcode, B, T, H, 128, 128, 64, kdn.KDN_BF16, kdn.KDN_FLAG_NO_SPLIT) == 1
    x = make_inputs(variant, B, T, H, 128, 128, io="bf16", seed=900 + T)
    t = to_device(x)
    kw, ref_kw = {}, {}
    if with_state:
        rng = np.random.default_rng(T)
        S0 = (0.2 * rng.standard_normal((B, H, 128, 128))).astype(np.float32)
        p0 = rng.uniform(0.3, 2.0, size=(B, H, 128) if variant == "diag" else (B, H)).astype(np.float32)
        kw = {"S0": torch.from_numpy(S0).cuda(), "p0": torch.from_numpy(p0).cuda()}
        ref_kw = {"S0": S0, "p0": p0}
    ref = oracle.forward(variant, x["q"], x["k"], x["v"], x["log_alpha"], x["omega"], x["r"], **ref_kw)
    got = _run(kdn, variant, t, chunk=64, **kw)
    _check(variant, x, got, ref, "bf16", "split")
    whole = _run(kdn, variant, t, chunk=64, flags=kdn.KDN_FLAG_NO_SPLIT, **kw)
    for a, b_ in zip(got, whole):
        a, b_ = to_host(a), to_host(b_)
        assert np.max(np.abs(a - b_)) <= 2e-2 * max(1e-3, np.max(np.abs(b_)))


def test_sequence_split_strong_decay():
    """Segments whose chunks decay strongly (mid-chunk reference, split frame
    factor) chain correctly: the transition map of such a segment is tiny."""
    import torch

    kdn = _kdn()
    B, T, H = 1, 2048, 2
    x = make_inputs("diag", B, T, H, 128, 128, io="bf16", seed=78)
    x["log_alpha"][:, :, 0] = -1.5
    x["r"][:, :, 0] = 1e-3
    x["omega"][:, :, 0] = 1.0
    t = to_device(x)
    ws = torch.empty(kdn.workspace_size(kdn.KDN_DIAG, B, T, H, 128, 128, 64, kdn.KDN_BF16, 0),
                     dtype=torch.uint8, device="cuda")
    got = _run(kdn, "diag", t, chunk=64, workspace=ws)
    assert kdn.kdn_read_device_status(ws) == 0
    ref = oracle.forward("diag", x["q"], x["k"], x["v"], x["log_alpha"], x["omega"], x["r"])
    _check("diag", x, got, ref, "bf16", "split, strong decay")
