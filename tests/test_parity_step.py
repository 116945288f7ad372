"""GPU decode (kdn_step) parity against the fp64 oracle.

A prefill runs through the forward path, then single-token steps update the
state in place; the oracle runs the whole token sequence in one recurrence.
"""
import numpy as np
import pytest

import oracle
from kdn_testutil import err, max_rel, to_device, to_host, tol
from uncertainty_aware_delta_gb300.inputs import WORKLOADS, decode_step_inputs, make_inputs, workload_inputs

pytestmark = pytest.mark.gpu


def _kdn():
    import uncertainty_aware_delta_gb300 as kdn
    from uncertainty_aware_delta_gb300.build import build_library

    build_library()
    return kdn


def _prefill_then_steps(kdn, variant, x, prefill, steps, chunk=64, check_every=1, seqs=None):
    import torch

    t = to_device(x)
    fwd = kdn.kdn_diag_forward if variant == "diag" else kdn.kdn_iso_forward
    pre = {n: v[:, :prefill].contiguous() for n, v in t.items()}
    _, S, p = fwd(pre["q"], pre["k"], pre["v"], pre["log_alpha"], pre["omega"], pre["r"], chunk=chunk)
    ws = torch.empty(kdn.workspace_size(0, S.shape[0], 1, S.shape[1], S.shape[2], S.shape[3]),
                     dtype=torch.uint8, device="cuda")
    outs = []
    for s in range(steps):
        tt = prefill + s
        o = kdn.kdn_step(variant, *(t[n][:, tt].contiguous() for n in ("q", "k", "v", "log_alpha", "omega", "r")),
                         S, p, workspace=ws)
        outs.append(o.clone())
    torch.cuda.synchronize()
    return torch.stack(outs, 1), S, p


CASES = [("diag", 3, 2, 128, 128, "f32"), ("iso", 3, 2, 128, 128, "f32"), ("diag", 2, 3, 16, 64, "f32"),
         ("iso", 2, 2, 64, 32, "f32"), ("diag", 2, 2, 128, 128, "bf16"), ("iso", 2, 2, 32, 128, "bf16"),
         # more (sequence, head) pairs than SMs: each persistent CTA of the 128 x 128
         # decode walks several heads through its buffer ring
         ("diag", 100, 4, 128, 128, "f32"), ("iso", 100, 4, 128, 128, "f32"),
         ("diag", 80, 5, 128, 128, "bf16"), ("iso", 80, 5, 128, 128, "bf16")]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(map(str, c)))
def test_steps_after_prefill(case):
    variant, B, H, dk, dv, io = case
    kdn = _kdn()
    prefill, steps = (40, 12) if B * H < 100 else (8, 3)
    x = make_inputs(variant, B, prefill + steps, H, dk, dv, io=io, seed=77 + dk)
    o, S, p = _prefill_then_steps(kdn, variant, x, prefill, steps, chunk=16)
    ref = oracle.forward(variant, x["q"], x["k"], x["v"], x["log_alpha"], x["omega"], x["r"])
    assert err(to_host(o), ref["o"][:, prefill:], io) <= tol(io)
    assert err(to_host(S), ref["S_T"], io) <= tol(io)
    assert err(to_host(p), ref["p_T"], io) <= tol(io)


def test_step_from_zero_state_is_one_token_forward():
    import torch

    kdn = _kdn()
    x = make_inputs("diag", 4, 1, 3, 64, 64, io="f32", seed=3)
    t = to_device(x)
    S = torch.zeros(4, 3, 64, 64, device="cuda")
    p = torch.ones(4, 3, 64, device="cuda")
    o = kdn.kdn_step("diag", *(t[n][:, 0].contiguous() for n in ("q", "k", "v", "log_alpha", "omega", "r")), S, p)
    ref = oracle.forward("diag", x["q"], x["k"], x["v"], x["log_alpha"], x["omega"], x["r"])
    assert max_rel(to_host(o), ref["o"][:, 0]) <= 1e-4
    assert max_rel(to_host(S), ref["S_T"]) <= 1e-4
    assert max_rel(to_host(p), ref["p_T"]) <= 1e-4


def _oracle_steps_in_place(x, S, p, o, mu=None):
    """One oracle token for every sequence, the fp64 state (S, p) updated in place
    (the C oracle copies each sequence's initial state before it writes that
    sequence's final state, so the same buffers may serve as both)."""
    import ctypes

    lib = oracle.recurrence._load()
    f64 = lambda a: np.ascontiguousarray(np.asarray(a, np.float64)[:, None])
    q, k, v, la, om, r = (f64(x[n][:, 0]) for n in ("q", "k", "v", "log_alpha", "omega", "r"))
    B, _, H, dk = q.shape
    dv = v.shape[-1]
    P = lambda a: a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))
    rc = lib.kdn_oracle_forward(0, B, 1, H, dk, dv, float(dk if mu is None else mu), P(q), P(k), P(v), P(la), P(om),
                                P(r), P(S), P(p), P(o), P(S), P(p), None, None, 0)
    assert rc == 0


def test_decode_workload_every_sequence():
    """The decode workload at full size (256 sequences x 16 heads, d = 128,
    512-token prefill, 1024 steps): every sequence against the oracle, the
    outputs of every step and the final state of every (sequence, head)."""
    import torch

    kdn = _kdn()
    w = WORKLOADS["diag-decode-f32-s256h16d128"]
    x = workload_inputs(w)
    t = to_device(x)
    _, S, p = kdn.kdn_diag_forward(t["q"], t["k"], t["v"], t["log_alpha"], t["omega"], t["r"],
                                   chunk=w.chunk)
    del t
    ref = oracle.forward("diag", x["q"], x["k"], x["v"], x["log_alpha"], x["omega"], x["r"])
    S_ref, p_ref = ref["S_T"], ref["p_T"]
    del x, ref
    assert max_rel(to_host(S), S_ref) <= 1e-4 and max_rel(to_host(p), p_ref) <= 1e-4
    ws = torch.empty(kdn.workspace_size(0, w.B, 1, w.H, w.d, w.d), dtype=torch.uint8, device="cuda")
    names = ("q", "k", "v", "log_alpha", "omega", "r")
    o_ref = np.zeros((w.B, 1, w.H, w.d))
    worst_o = 0.0
    for s in range(w.steps):
        y = decode_step_inputs(w, s)
        ty = to_device(y)
        o = kdn.kdn_step("diag", *(ty[n][:, 0] for n in names), S, p, workspace=ws)
        _oracle_steps_in_place(y, S_ref, p_ref, o_ref)
        e = max_rel(to_host(o), o_ref[:, 0])
        worst_o = max(worst_o, e)
        assert e <= 1e-4, (s, e)
        assert np.all(np.isfinite(to_host(o)))
    assert kdn.kdn_read_device_status(ws) == 0
    S, p = to_host(S), to_host(p)
    eS, ep = max_rel(S, S_ref), max_rel(p, p_ref)
    print(f"[parity] decode all sequences: worst step o {worst_o:.2e}, final S {eS:.2e}, final p {ep:.2e}")
    assert eS <= 1e-4 and ep <= 1e-4
    for b in range(w.B):
        for h in range(w.H):
            assert max_rel(S[b, h], S_ref[b, h]) <= 1e-4, (b, h)
