"""GPU parity of the dense-covariance (exact) Kalman memory forward against the
fp64 oracle's dense filter (KDN paper Sec. 3.2, Eq. 12-17).

The CUDA kernel is called through the C ABI (ctypes binding); the oracle runs
the same filter token by token in fp64 on the same rounded inputs, per
(batch, head).  Cases cover d = 32, 64, 128, fp32 and bf16 io, a given initial
state and covariance (and in-place resume), T = 0, continuation, and the
exact-filter case where the Diagonal KDN coincides with it (one-hot keys,
mu = 1).
"""
import numpy as np
import pytest

import oracle
from kdn_testutil import err, to_device, to_host, tol
from uncertainty_aware_delta_gb300.inputs import make_inputs

pytestmark = pytest.mark.gpu


def _kdn():
    import uncertainty_aware_delta_gb300 as kdn
    from uncertainty_aware_delta_gb300.build import build_library

    build_library()
    return kdn


def _reference(x, S0=None, P0=None):
    B, T, H, d = x["q"].shape
    o = np.zeros((B, T, H, d))
    S_T = np.zeros((B, H, d, d))
    P_T = np.zeros((B, H, d, d))
    for b in range(B):
        for h in range(H):
            s0 = np.zeros((d, d)) if S0 is None else S0[b, h]
            p0 = np.eye(d) if P0 is None else P0[b, h]
            if T == 0:
                S_T[b, h], P_T[b, h] = s0, p0
                continue
            ref = oracle.dense_kalman(x["k"][b, :, h], x["v"][b, :, h], x["q"][b, :, h], x["r"][b, :, h],
                                      s0, p0, D=np.exp(x["log_alpha"][b, :, h].astype(np.float64)),
                                      Omega=x["omega"][b, :, h])
            o[b, :, h] = ref["o"]
            S_T[b, h], P_T[b, h] = ref["S_T"], ref["P_T"]
    return o, S_T, P_T


def _spd(rng, B, H, d):
    A = rng.standard_normal((B, H, d, d))
    return (np.einsum("bhij,bhkj->bhik", A, A) / d + 0.1 * np.eye(d)).astype(np.float32)


def _check(got, ref, io, what):
    e = {n: err(to_host(g), r, io) for n, g, r in zip(("o", "S_T", "P_T"), got, ref)}
    assert all(v <= tol(io) for v in e.values()), (what, e)
    return e


CASES = [
    # B, T, H, d, io
    (1, 50, 2, 32, "f32"),
    (2, 40, 1, 64, "f32"),
    (1, 30, 2, 128, "f32"),
    (1, 60, 2, 128, "bf16"),
    (2, 17, 3, 64, "bf16"),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(map(str, c)))
def test_dense_forward_matches_oracle(case):
    B, T, H, d, io = case
    kdn = _kdn()
    x = make_inputs("diag", B, T, H, d, d, io=io, seed=3000 + T + d)
    t = to_device(x)
    got = kdn.kdn_dense_forward(t["q"], t["k"], t["v"], t["log_alpha"], t["omega"], t["r"])
    _check(got, _reference(x), io, case)


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_dense_forward_long_sequence_stays_symmetric(io):
    """A 4096-token sequence (the length of the dense filter's bench workload):
    the fp32 covariance update P_hat - kappa u^T is not symmetrised, so check
    that P_T stays symmetric and finite over the whole run, and that o, S_T
    and P_T still match the fp64 filter."""
    kdn = _kdn()
    x = make_inputs("diag", 1, 4096, 1, 128, 128, io=io, seed=3999)
    t = to_device(x)
    got = kdn.kdn_dense_forward(t["q"], t["k"], t["v"], t["log_alpha"], t["omega"], t["r"])
    o, S_T, P_T = (to_host(a) for a in got)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(S_T)) and np.all(np.isfinite(P_T))
    P = P_T[0, 0].astype(np.float64)
    asym = np.max(np.abs(P - P.T)) / np.max(np.abs(P))
    assert asym <= 1e-5, asym
    assert np.min(np.linalg.eigvalsh(0.5 * (P + P.T))) > 0.0
    e = _check(got, _reference(x), io, f"long {io}")
    print(f"[parity] dense T=4096 {io}: {e}, P_T asymmetry {asym:.2e}")


def test_dense_initial_state_in_place_resume_and_empty_sequence():
    import torch

    kdn = _kdn()
    B, T, H, d = 1, 40, 2, 64
    rng = np.random.default_rng(5)
    x = make_inputs("diag", B, T, H, d, d, io="f32", seed=41)
    S0 = (0.3 * rng.standard_normal((B, H, d, d))).astype(np.float32)
    P0 = _spd(rng, B, H, d)
    ref = _reference(x, S0, P0)
    t = to_device(x)
    S, P = torch.from_numpy(S0).cuda(), torch.from_numpy(P0).cuda()
    o = torch.empty((B, T, H, d), dtype=torch.float32, device="cuda")
    got = kdn.kdn_dense_forward(t["q"], t["k"], t["v"], t["log_alpha"], t["omega"], t["r"], S, P,
                                out=(o, S, P))   # S_T == S0, P_T == P0
    _check(got, ref, "f32", "in-place resume")
    # T = 0: the state is copied (identity covariance when P0 is absent)
    x0 = make_inputs("diag", B, 0, H, d, d, io="f32", seed=1)
    t0 = to_device(x0)
    S1 = torch.from_numpy(S0).cuda()
    _, S_T, P_T = kdn.kdn_dense_forward(t0["q"], t0["k"], t0["v"], t0["log_alpha"], t0["omega"], t0["r"], S1)
    assert np.array_equal(to_host(S_T), S0)
    assert np.array_equal(to_host(P_T), np.broadcast_to(np.eye(d, dtype=np.float32), (B, H, d, d)))


def test_dense_continuation():
    kdn = _kdn()
    B, T, H, d = 1, 64, 2, 128
    x = make_inputs("diag", B, T, H, d, d, io="f32", seed=77)
    t = to_device(x)
    whole = kdn.kdn_dense_forward(t["q"], t["k"], t["v"], t["log_alpha"], t["omega"], t["r"])
    n = 23
    # (clone: fresh 16-byte aligned buffers; a token slice of a B = 1 tensor is already contiguous)
    names = ("q", "k", "v", "log_alpha", "omega", "r")
    first = kdn.kdn_dense_forward(*(t[k][:, :n].clone() for k in names))
    second = kdn.kdn_dense_forward(*(t[k][:, n:].clone() for k in names), first[1], first[2])
    o = np.concatenate([to_host(first[0]), to_host(second[0])], axis=1)
    assert err(o, to_host(whole[0]), "f32") <= 1e-5
    assert err(to_host(second[1]), to_host(whole[1]), "f32") <= 1e-5
    assert err(to_host(second[2]), to_host(whole[2]), "f32") <= 1e-5


def test_dense_equals_diagonal_kdn_on_one_hot_keys():
    """Axis-aligned one-hot keys keep the covariance diagonal, so with mu = 1
    (exact information update) the Diagonal KDN and the dense filter agree
    token for token (the oracle pins the same identity in fp64)."""
    import torch

    kdn = _kdn()
    B, T, H, d = 1, 80, 2, 32
    x = make_inputs("diag", B, T, H, d, d, io="f32", seed=9)
    rng = np.random.default_rng(9)
    idx = rng.integers(0, d, size=(B, T, H))
    onehot = np.zeros((B, T, H, d), np.float32)
    np.put_along_axis(onehot, idx[..., None], 1.0, axis=-1)
    x["k"] = onehot
    t = to_device(x)
    dense = kdn.kdn_dense_forward(t["q"], t["k"], t["v"], t["log_alpha"], t["omega"], t["r"])
    diag = kdn.kdn_diag_forward(t["q"], t["k"], t["v"], t["log_alpha"], t["omega"], t["r"], mu=1.0, chunk=16)
    assert err(to_host(dense[0]), to_host(diag[0]), "f32") <= 1e-4
    assert err(to_host(dense[1]), to_host(diag[1]), "f32") <= 1e-4
    P_T = to_host(dense[2])
    assert err(np.diagonal(P_T, axis1=-2, axis2=-1), to_host(diag[2]), "f32") <= 1e-4
    assert np.max(np.abs(P_T - np.einsum("bhi,ij->bhij", np.diagonal(P_T, axis1=-2, axis2=-1), np.eye(d)))) == 0.0
    del torch


@pytest.mark.parametrize("io, d", [("f32", 64), ("bf16", 128)])
def test_dense_strong_decay_renormalises(io, d):
    """Channels that decay by e^-2 and e^-2.4 per token: the covariance pass holds the
    decay outside P and folds it back in whenever a channel's running decay would
    fall below 2^-20, here every six to seven tokens; the mean pass's 64-token chunks
    then decay by 128 and 154 (within its range of 160, and beyond the 80 at which the
    fused kernel takes the mid-chunk reference).  The result must still be the fp64
    filter's; bf16 d = 128 takes the tensor-core mean pass, fp32 the CUDA-core one."""
    import torch

    kdn = _kdn()
    B, T, H = 1, 150, 2
    x = make_inputs("diag", B, T, H, d, d, io=io, seed=3131)
    x["log_alpha"][:, :, 0, : d // 8] = -2.0
    x["log_alpha"][:, :, 1, : d // 16] = -2.4
    t = to_device(x)
    ws = torch.empty(kdn.dense_workspace_size(B, T, H, d, kdn.KDN_BF16 if io == "bf16" else kdn.KDN_F32),
                     dtype=torch.uint8, device="cuda")
    got = kdn.kdn_dense_forward(t["q"], t["k"], t["v"], t["log_alpha"], t["omega"], t["r"], workspace=ws)
    assert kdn.kdn_read_device_status(ws) == 0
    o, S_T, P_T = (to_host(a) for a in got)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(S_T)) and np.all(np.isfinite(P_T))
    e = _check(got, _reference(x), io, f"strong decay {io} d={d}")
    print(f"[parity] dense strong decay {io} d={d}: {e}")


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_dense_blocks_end_early_on_concentrated_decay(io):
    """For d = 128 the covariance pass runs blocks of up to 16 tokens, and a block
    ends where some channel's log decay from the block start would exceed 40.
    Eight tokens of log decay -6 on a few channels end blocks early, and one token of
    log decay -45 on one channel is a block of its own, taken about its own decay.
    The result must still be the fp64 filter's, through both mean paths."""
    import torch

    kdn = _kdn()
    B, T, H, d = 1, 100, 2, 128
    x = make_inputs("diag", B, T, H, d, d, io=io, seed=4242)
    x["log_alpha"][:, 20:28, 0, :4] = -6.0
    x["log_alpha"][:, 60, 1, 5] = -45.0
    t = to_device(x)
    ws = torch.empty(kdn.dense_workspace_size(B, T, H, d, kdn.KDN_BF16 if io == "bf16" else kdn.KDN_F32),
                     dtype=torch.uint8, device="cuda")
    got = kdn.kdn_dense_forward(t["q"], t["k"], t["v"], t["log_alpha"], t["omega"], t["r"], workspace=ws)
    assert kdn.kdn_read_device_status(ws) == 0
    o, S_T, P_T = (to_host(a) for a in got)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(S_T)) and np.all(np.isfinite(P_T))
    e = _check(got, _reference(x), io, f"blocks end early {io}")
    print(f"[parity] dense blocks ending early {io}: {e}")
