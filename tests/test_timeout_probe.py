"""The bounded-wait path on the GPU, driven without a fault.

Every wait of the kernels that consume asynchronous copies (the fused
tensor-core forward and the d = 128 decode kernel) is bounded; when a bound
runs out the kernel records KDN_ERR_TIMEOUT in the status word, stops issuing
work, lets the copies it has already issued land and exits.  The test flag
KDN_FLAG_TIMEOUT_PROBE makes that happen on purpose: the kernel's first wait
is on a barrier that nothing completes, with a bound of a few milliseconds,
while its first copies are in flight.  The tests check that the call returns,
that the status word reads KDN_ERR_TIMEOUT, and that a normal call right after
it, on the same stream and workspace, matches the oracle (the context and the
device stayed usable).
"""
import numpy as np
import pytest

import oracle
from kdn_testutil import err, max_rel, to_device, to_host, tol
from uncertainty_aware_delta_gb300.inputs import make_inputs

pytestmark = pytest.mark.gpu

KDN_ERR_TIMEOUT = 8


def _kdn():
    import uncertainty_aware_delta_gb300 as kdn
    from uncertainty_aware_delta_gb300.build import build_library

    build_library()
    return kdn


@pytest.mark.parametrize("variant", ["diag", "iso"])
def test_fused_forward_timeout_is_reported_and_recovered(variant):
    import torch

    kdn = _kdn()
    B, T, H = 2, 200, 3
    vcode = kdn.KDN_DIAG if variant == "diag" else kdn.KDN_ISO
    assert kdn.forward_kernel_count(vcode, B, T, H, 128, 128, 64, kdn.KDN_BF16, 0) == 1   # fused kernel
    x = make_inputs(variant, B, T, H, 128, 128, io="bf16", seed=4040)
    t = to_device(x)
    fn = kdn.kdn_diag_forward if variant == "diag" else kdn.kdn_iso_forward
    ws = torch.empty(kdn.workspace_size(vcode, B, T, H, 128, 128, 64, kdn.KDN_BF16, 0), dtype=torch.uint8,
                     device="cuda")
    args = (t["q"], t["k"], t["v"], t["log_alpha"], t["omega"], t["r"])
    fn(*args, chunk=64, workspace=ws, flags=kdn.KDN_FLAG_TIMEOUT_PROBE)
    assert kdn.kdn_read_device_status(ws) == KDN_ERR_TIMEOUT
    got = fn(*args, chunk=64, workspace=ws)
    assert kdn.kdn_read_device_status(ws) == 0
    ref = oracle.forward(variant, x["q"], x["k"], x["v"], x["log_alpha"], x["omega"], x["r"])
    e = [err(to_host(a), ref[n], "bf16") for a, n in zip(got, ("o", "S_T", "p_T"))]
    assert max(e) <= tol("bf16"), e


def test_decode_stream_timeout_is_reported_and_recovered():
    import torch

    kdn = _kdn()
    B, H, d = 40, 4, 128     # 160 (sequence, head) pairs: more than one head per persistent CTA
    x = make_inputs("diag", B, 2, H, d, d, io="f32", seed=4041)
    t = to_device(x)
    names = ("q", "k", "v", "log_alpha", "omega", "r")
    rng = np.random.default_rng(4041)
    S0 = (0.3 * rng.standard_normal((B, H, d, d))).astype(np.float32)
    p0 = rng.uniform(0.3, 2.0, size=(B, H, d)).astype(np.float32)
    S = torch.from_numpy(S0).cuda()
    p = torch.from_numpy(p0).cuda()
    ws = torch.empty(kdn.workspace_size(0, B, 1, H, d, d), dtype=torch.uint8, device="cuda")
    step0 = [t[n][:, 0].contiguous() for n in names]
    # the probe call: its results are undefined, so it runs on copies of the state
    Sx, px = S.clone(), p.clone()
    kdn.kdn_step("diag", *step0, Sx, px, workspace=ws, flags=kdn.KDN_FLAG_TIMEOUT_PROBE)
    assert kdn.kdn_read_device_status(ws) == KDN_ERR_TIMEOUT
    # normal steps afterwards on the same stream and workspace
    o1 = kdn.kdn_step("diag", *step0, S, p, workspace=ws)
    assert kdn.kdn_read_device_status(ws) == 0
    step1 = [t[n][:, 1].contiguous() for n in names]
    o2 = kdn.kdn_step("diag", *step1, S, p, workspace=ws)
    ref = oracle.forward("diag", x["q"], x["k"], x["v"], x["log_alpha"], x["omega"], x["r"], S0=S0, p0=p0)
    assert max_rel(to_host(o1), ref["o"][:, 0]) <= 1e-4
    assert max_rel(to_host(o2), ref["o"][:, 1]) <= 1e-4
    assert max_rel(to_host(S), ref["S_T"]) <= 1e-4
    assert max_rel(to_host(p), ref["p_T"]) <= 1e-4
