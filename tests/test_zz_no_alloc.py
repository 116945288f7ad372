"""kdn_forward_noalloc: the forward for callers that cannot allocate device memory.

Some callers may not call cudaMalloc where they run the mixer (a host
framework that owns all device memory, or a loop that must not pay for an
allocation that can synchronise the device).  For them the library keeps a
static device scratch array and this entry point takes no workspace.  These
tests call it through the C ABI and check that it gives the same outputs as
the regular workspace-taking entry point, on two calls in a row (the second
call must not see stale contents of the shared array), and that a problem
larger than the array is refused before anything runs.

This file is named to be collected last, so a run that stops at the first
failure has already run every other test; it passes alone as well.
"""
import numpy as np
import pytest

import oracle
from kdn_testutil import FP32_TOL, max_rel, to_device, to_host
from uncertainty_aware_delta_gb300.inputs import make_inputs

pytestmark = pytest.mark.gpu


def _kdn():
    import uncertainty_aware_delta_gb300 as kdn
    from uncertainty_aware_delta_gb300.build import build_library

    build_library()
    return kdn


@pytest.mark.parametrize("variant", ["diag", "iso"])
def test_noalloc_matches_workspace_forward_on_two_calls(variant):
    import torch

    kdn = _kdn()
    B, T, H, d = 2, 300, 3, 64
    fwd = kdn.kdn_diag_forward if variant == "diag" else kdn.kdn_iso_forward
    for call, seed in enumerate((101, 202)):
        x = make_inputs(variant, B, T, H, d, d, io="f32", seed=seed)
        t = to_device(x)
        args = (t["q"], t["k"], t["v"], t["log_alpha"], t["omega"], t["r"])
        ref_o, ref_S, ref_p = fwd(*args, chunk=32, flags=kdn.KDN_FLAG_PORTABLE)
        o = torch.full_like(ref_o, float("nan"))
        S_T = torch.full_like(ref_S, float("nan"))
        p_T = torch.full_like(ref_p, float("nan"))
        status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        kdn.kdn_forward_noalloc(variant, *args, chunk=32, flags=kdn.KDN_FLAG_PORTABLE,
                                out=(o, S_T, p_T), status_out=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0, f"call {call}: device status {int(status.item())}"
        for got, ref in ((o, ref_o), (S_T, ref_S), (p_T, ref_p)):
            assert max_rel(to_host(got), to_host(ref)) <= FP32_TOL, f"call {call}"
        if call == 0:
            orc = oracle.forward(variant, x["q"], x["k"], x["v"], x["log_alpha"], x["omega"], x["r"])
            assert max_rel(to_host(o), orc["o"]) <= FP32_TOL


@pytest.mark.parametrize("variant", ["diag", "iso"])
def test_noalloc_tensor_core_split_path_on_two_calls(variant):
    """The tensor-core path with the sequence split (bf16, d = 128, chunk 64, few
    long sequences): its scan summaries, carries, segment states and
    transformed queries are carved from the built-in scratch; two calls in a
    row must match the workspace-taking entry point."""
    import torch

    kdn = _kdn()
    B, T, H, d = 1, 2048, 2, 128
    vcode = kdn.KDN_DIAG if variant == "diag" else kdn.KDN_ISO
    assert kdn.forward_kernel_count(vcode, B, T, H, d, d, 64, kdn.KDN_BF16, 0) == 6   # split into segments
    assert kdn.workspace_size(vcode, B, T, H, d, d, 64, kdn.KDN_BF16, 0) <= 32 * 2 ** 20
    fwd = kdn.kdn_diag_forward if variant == "diag" else kdn.kdn_iso_forward
    for call, seed in enumerate((303, 404)):
        x = make_inputs(variant, B, T, H, d, d, io="bf16", seed=seed)
        t = to_device(x)
        args = (t["q"], t["k"], t["v"], t["log_alpha"], t["omega"], t["r"])
        ref = fwd(*args, chunk=64)
        outs = tuple(torch.full_like(a, float("nan")) for a in ref)
        status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        kdn.kdn_forward_noalloc(variant, *args, chunk=64, out=outs, status_out=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0, f"call {call}: device status {int(status.item())}"
        for got, want in zip(outs, ref):
            g, w = to_host(got), to_host(want)
            assert np.all(np.isfinite(g))
            assert np.max(np.abs(g - w)) <= 1e-3 * max(1e-3, np.max(np.abs(w))), f"call {call}"


def test_noalloc_refuses_problems_larger_than_its_scratch():
    import torch

    kdn = _kdn()
    # gains alone need 4 * B*T*H*d_k bytes = 64 MiB > the 32 MiB built-in scratch
    B, T, H, d = 1, 8192, 16, 128
    need = kdn.workspace_size(kdn.KDN_DIAG, B, T, H, d, d, 64, kdn.KDN_F32, kdn.KDN_FLAG_PORTABLE)
    assert need > 32 * 2 ** 20
    q = torch.zeros(B, T, H, d, device="cuda")
    r = torch.ones(B, T, H, device="cuda")
    o = torch.empty_like(q)
    S_T = torch.empty(B, H, d, d, device="cuda")
    p_T = torch.empty(B, H, d, device="cuda")
    with pytest.raises(kdn.KDNError) as e:
        kdn.kdn_forward_noalloc("diag", q, q, q, q, q, r, chunk=64, flags=kdn.KDN_FLAG_PORTABLE,
                                out=(o, S_T, p_T))
    assert e.value.status == 5   # KDN_ERR_WORKSPACE
