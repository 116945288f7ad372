"""The C-ABI library loads and exports every entry point include/kdn.h declares.

These tests run without a GPU: they only load the library, read constants
and exercise host-side validation on arguments that are rejected before
anything is enqueued (so no CUDA call is ever reached).
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "kdn.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b(kdn_[a-z_]+)\s*\(", text)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    from uncertainty_aware_delta_gb300.build import build_library
    import uncertainty_aware_delta_gb300 as kdn

    build_library()
    return kdn.library()


def test_header_declares_the_boundary():
    names = _declared_functions()
    for n in ("kdn_diag_forward", "kdn_iso_forward", "kdn_step", "kdn_workspace_size",
              "kdn_read_device_status", "kdn_status_string", "kdn_abi_version",
              "kdn_forward_kernel_count", "kdn_forward_noalloc", "kdn_pkda_forward", "kdn_pkda_step",
              "kdn_dense_forward", "kdn_step_ex", "kdn_backward", "kdn_backward_workspace_size",
              "kdn_gated_forward", "kdn_gated_workspace_size", "kdn_dense_workspace_size"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    raw = ctypes.CDLL(lib._name)
    for n in _declared_functions():
        assert hasattr(raw, n), f"{n} declared in kdn.h but not exported"


def test_status_strings_and_version(lib):
    import uncertainty_aware_delta_gb300 as kdn

    assert lib.kdn_abi_version() == 106
    for code in range(0, 11):
        s = kdn.status_string(code)
        assert s and s != "unknown status"
    assert kdn.status_string(99) == "unknown status"


def test_workspace_size_rules(lib):
    import uncertainty_aware_delta_gb300 as kdn

    ws = kdn.workspace_size
    # unsupported sizes are rejected with 0
    assert ws(0, 1, 64, 2, 24, 16, 16, 0, 0) == 0
    assert ws(0, 1, 64, 2, 16, 16, 48, 0, 0) == 0
    assert ws(0, -1, 64, 2, 16, 16, 16, 0, 0) == 0
    assert ws(3, 1, 64, 2, 16, 16, 16, 0, 0) == 0
    # PKDA keeps a per-channel statistic: the same scratch as the diagonal variant
    assert ws(2, 2, 100, 3, 32, 16, 16, 0, 1) == ws(0, 2, 100, 3, 32, 16, 16, 0, 1)
    assert ws(0, 1, 64, 2, 16, 16, 16, 5, 0) == 0
    # the portable path stores gains [B,T,H,dk] fp32 plus the scan summaries
    n = ws(0, 2, 100, 3, 32, 16, 16, 0, 1)
    assert n >= 256 + 4 * 2 * 100 * 3 * 32
    assert n % 256 == 0
    # decode needs only the status word
    assert ws(0, 256, 1, 16, 128, 128, 0, 0, 1) >= 256


def test_forward_kernel_count(lib):
    import uncertainty_aware_delta_gb300 as kdn

    assert kdn.forward_kernel_count(0, 1, 64, 2, 16, 16, 16, 0, 0) == 4   # scan (3) + chunk pass
    assert kdn.forward_kernel_count(1, 1, 64, 2, 16, 16, 16, 0, 1) == 4
    assert kdn.forward_kernel_count(0, 1, 0, 2, 16, 16, 0, 0, 0) == 1     # state copy
    assert kdn.forward_kernel_count(0, 0, 64, 2, 16, 16, 0, 0, 0) == 0
    assert kdn.forward_kernel_count(0, 1, 64, 2, 24, 16, 0, 0, 0) == 0
    assert kdn.forward_kernel_count(2, 1, 64, 2, 16, 16, 16, 0, 0) == 4   # PKDA: statistic scan + chunk pass
    assert kdn.forward_kernel_count(2, 1, 64, 2, 128, 128, 64, 1, 0) == 1  # fused tensor-core kernel


def test_sequence_split_plan(lib):
    """Few long sequences on the tensor-core path run as segments (scan carries,
    segment maps, chaining, output correction: 6 launches) with their state maps
    and transformed queries in the workspace; many sequences, short ones or the
    opt-out flag keep one launch."""
    import uncertainty_aware_delta_gb300 as kdn

    kc, ws = kdn.forward_kernel_count, kdn.workspace_size
    NO = kdn.KDN_FLAG_NO_SPLIT
    for v in (0, 1, 2):
        # 16 sequences x 65536 tokens: 152 // 16 = 9 segments of 29 x 256 tokens
        assert kc(v, 1, 65536, 16, 128, 128, 64, 1, 0) == 6
        assert kc(v, 1, 65536, 16, 128, 128, 64, 1, NO) == 1
        assert kc(v, 8, 4096, 16, 128, 128, 64, 1, 0) == 1      # 128 sequences fill the GPU
        assert kc(v, 1, 1500, 2, 128, 128, 64, 1, 0) == 1       # under 2 x 1024 tokens
        assert kc(v, 1, 2048, 2, 128, 128, 64, 1, 0) == 6
        nu = 1 if v == 1 else 128
        n_split, n_whole = ws(v, 1, 65536, 16, 128, 128, 64, 1, 0), ws(v, 1, 65536, 16, 128, 128, 64, 1, NO)
        # three [16 x 9][128][128] fp32 state arrays, the scan summaries and carries (256 gain
        # chunks) and the transformed queries (bf16, one per token-head)
        assert n_split - n_whole >= 4 * (3 * 16 * 9 * 128 * 128 + 5 * 16 * 256 * nu) + 2 * 65536 * 16 * 128
        assert ws(v, 8, 4096, 16, 128, 128, 64, 1, 0) == ws(v, 8, 4096, 16, 128, 128, 64, 1, NO)


def _fwd_args(**over):
    a = dict(B=1, T=64, H=2, dk=16, dv=16, chunk=16, mu=-1.0, io=0, flags=0,
             q=64, k=64, v=64, la=64, om=64, r=64, S0=None, p0=None, o=1 << 20, S_T=2 << 20,
             p_T=3 << 20, ws=4 << 20, wsb=1 << 20)
    a.update(over)
    return a


def _call(lib, a, variant=0):
    fn = lib.kdn_diag_forward if variant == 0 else lib.kdn_iso_forward
    vp = lambda x: None if x is None else ctypes.c_void_p(x)
    return fn(a["B"], a["T"], a["H"], a["dk"], a["dv"], a["chunk"], a["mu"], a["io"], a["flags"],
              vp(a["q"]), vp(a["k"]), vp(a["v"]), vp(a["la"]), vp(a["om"]), vp(a["r"]), vp(a["S0"]),
              vp(a["p0"]), vp(a["o"]), vp(a["S_T"]), vp(a["p_T"]), vp(a["ws"]), a["wsb"], None)


@pytest.mark.parametrize("variant", [0, 1])
def test_validation_rejects_before_launch(lib, variant):
    # each case fails a host check, so nothing reaches the device
    assert _call(lib, _fwd_args(dk=24), variant) == 6          # KDN_ERR_UNSUPPORTED
    assert _call(lib, _fwd_args(chunk=8), variant) == 6
    assert _call(lib, _fwd_args(io=3), variant) == 3           # KDN_ERR_DTYPE
    assert _call(lib, _fwd_args(T=-1), variant) == 2           # KDN_ERR_SHAPE
    assert _call(lib, _fwd_args(q=None), variant) == 1         # KDN_ERR_NULL
    assert _call(lib, _fwd_args(S_T=None), variant) == 1
    assert _call(lib, _fwd_args(ws=None), variant) == 5        # KDN_ERR_WORKSPACE
    assert _call(lib, _fwd_args(wsb=16), variant) == 5
    assert _call(lib, _fwd_args(k=72), variant) == 4           # KDN_ERR_ALIGN (72 % 16 != 0)
    assert _call(lib, _fwd_args(o=64 + 16), variant) == 10     # KDN_ERR_ALIAS (o overlaps q)
    assert _call(lib, _fwd_args(ws=1 << 20), variant) == 10    # workspace overlaps o


def test_gated_workspace_rules(lib):
    import uncertainty_aware_delta_gb300 as kdn

    gws, ws = kdn.gated_workspace_size, kdn.workspace_size
    assert gws(2, 1, 64, 2, 16, 16, 16, 0, 0) == 0            # PKDA has no gates
    assert gws(0, 1, 64, 2, 24, 16, 16, 0, 0) == 0
    # every path: the ungated scratch plus fp32 log alpha, omega and r
    for (B, T, H, d, io) in ((2, 100, 3, 32, 0), (8, 4096, 16, 128, 1), (1, 65536, 16, 128, 1)):
        for v, nu in ((0, d), (1, 1)):
            n = B * T * H
            assert gws(v, B, T, H, d, d, 0, io, 0) >= ws(v, B, T, H, d, d, 0, io, 0) + 4 * n * (d + nu + 1)
            assert gws(v, B, T, H, d, d, 0, io, 0) % 256 == 0
    # T = 0: nothing beyond the status word
    assert gws(0, 2, 0, 2, 128, 128, 0, 1, 0) == ws(0, 2, 0, 2, 128, 128, 0, 1, 0)


def test_gated_validation_rejects_before_launch(lib):
    vp = lambda x: None if x is None else ctypes.c_void_p(x)

    def call(variant=0, dk=16, io=0, T=64, r_min=-1.0, wsb=1 << 20, **ptr):
        p = dict(q=64, k=64, v=64, al=64, wl=64, rl=64, S0=None, p0=None, o=1 << 20, S_T=2 << 20, p_T=3 << 20,
                 be=None, ws=4 << 20)
        p.update(ptr)
        return lib.kdn_gated_forward(variant, 1, T, 2, dk, 16, 16, -1.0, r_min, io, 0, vp(p["q"]), vp(p["k"]),
                                     vp(p["v"]), vp(p["al"]), vp(p["wl"]), vp(p["rl"]), vp(p["S0"]), vp(p["p0"]),
                                     vp(p["o"]), vp(p["S_T"]), vp(p["p_T"]), vp(p["be"]), vp(p["ws"]), wsb, None)

    assert call(variant=2) == 2                      # KDN_ERR_SHAPE: no gates for PKDA
    assert call(dk=24) == 6                          # KDN_ERR_UNSUPPORTED
    assert call(io=3) == 3                           # KDN_ERR_DTYPE
    assert call(T=-1) == 2
    assert call(r_min=float("nan")) == 2
    assert call(r_min=float("inf")) == 2
    assert call(q=None) == 1                         # KDN_ERR_NULL
    assert call(wl=None) == 1
    assert call(S_T=None) == 1
    assert call(ws=None) == 5                        # KDN_ERR_WORKSPACE
    assert call(wsb=256) == 5
    assert call(rl=72) == 4                          # KDN_ERR_ALIGN
    assert call(be=(5 << 20) + 8) == 4
    assert call(o=64 + 16) == 10                     # KDN_ERR_ALIAS: o overlaps the inputs
    assert call(be=(1 << 20) + 64) == 10             # beta_eff overlaps o
    assert call(be=64) == 10                         # beta_eff overlaps the inputs
    assert call(ws=(3 << 20)) == 10                  # workspace overlaps p_T


def test_dense_validation_rejects_before_launch(lib):
    # B=1 T=64 H=2 d=32: inputs of 64*2*32 elements; each case fails a host check
    vp = ctypes.c_void_p

    def call(d=32, io=0, T=64, wsb=1 << 20, **ptr):
        p = dict(q=1 << 16, k=2 << 16, v=3 << 16, la=4 << 16, om=5 << 16, r=6 << 16, S0=None, P0=None,
                 o=1 << 20, S_T=2 << 20, P_T=3 << 20, ws=4 << 20)
        p.update(ptr)
        args = [vp(p[n]) if p[n] is not None else None
                for n in ("q", "k", "v", "la", "om", "r", "S0", "P0", "o", "S_T", "P_T", "ws")]
        return lib.kdn_dense_forward(1, T, 2, d, io, *args, wsb, None)

    # the workspace holds the status word and the gains kappa [B,T,H,d] fp32
    assert lib.kdn_dense_workspace_size(1, 64, 2, 32, 0) >= 256 + 4 * 64 * 2 * 32
    assert lib.kdn_dense_workspace_size(1, 64, 2, 16, 0) == 0
    assert lib.kdn_dense_workspace_size(1, 64, 2, 32, 2) == 0

    assert call(d=16) == 6                     # KDN_ERR_UNSUPPORTED
    assert call(io=2) == 3                     # KDN_ERR_DTYPE
    assert call(T=-1) == 2                     # KDN_ERR_SHAPE
    assert call(q=None) == 1                   # KDN_ERR_NULL
    assert call(P_T=None) == 1
    assert call(k=(2 << 16) + 8) == 4          # KDN_ERR_ALIGN
    assert call(o=(1 << 16) + 64) == 10        # KDN_ERR_ALIAS: o overlaps q
    assert call(P_T=(2 << 20) + 256) == 10     # P_T overlaps S_T
    assert call(P0=(2 << 20)) == 10            # P0 overlaps S_T
    assert call(ws=None) == 5                  # KDN_ERR_WORKSPACE
    assert call(wsb=1024) == 5
    assert call(ws=(3 << 20) + 4096) == 10     # workspace overlaps P_T


def test_step_validation_rejects_before_launch(lib):
    vp = ctypes.c_void_p
    base = [0, 4, 2, 16, 16, -1.0, 0]
    ptrs = [vp(1 << 12), vp(2 << 12), vp(3 << 12), vp(4 << 12), vp(5 << 12), vp(6 << 12),
            vp(1 << 20), vp(2 << 20), vp(3 << 20)]
    ws = [vp(4 << 20), 256, None]
    assert lib.kdn_step(*base, *ptrs, None, 256, None) == 5
    assert lib.kdn_step(*base, *ptrs, vp(4 << 20), 8, None) == 5
    bad = list(base)
    bad[3] = 48
    assert lib.kdn_step(*bad, *ptrs, *ws) == 6
    p2 = list(ptrs)
    p2[6] = vp((1 << 20) + 8)
    assert lib.kdn_step(*base, *p2, *ws) == 4
    p3 = list(ptrs)
    p3[8] = vp((1 << 20) + 64)                               # o overlaps S
    assert lib.kdn_step(*base, *p3, *ws) == 10
    # kdn_step_ex: the same validation; flags other than the timeout probe are refused
    assert lib.kdn_step_ex(*base, 0, *p3, *ws) == 10
    assert lib.kdn_step_ex(*base, 0x1, *ptrs, *ws) == 6
    assert lib.kdn_step_ex(*bad, 0x100, *ptrs, *ws) == 6


def _pkda_call(lib, **over):
    a = dict(B=1, T=64, H=2, dk=16, dv=16, chunk=16, x=1.5, io=0, flags=0,
             q=64, k=64, v=64, la=64, beta=64, ap=64, bp=64, ce=64, S0=None, A0=None,
             o=1 << 20, S_T=2 << 20, A_T=3 << 20, ws=4 << 20, wsb=1 << 20)
    a.update(over)
    vp = lambda x: None if x is None else ctypes.c_void_p(x)
    return lib.kdn_pkda_forward(a["B"], a["T"], a["H"], a["dk"], a["dv"], a["chunk"], a["x"], a["io"],
                                a["flags"], vp(a["q"]), vp(a["k"]), vp(a["v"]), vp(a["la"]), vp(a["beta"]),
                                vp(a["ap"]), vp(a["bp"]), vp(a["ce"]), vp(a["S0"]), vp(a["A0"]), vp(a["o"]),
                                vp(a["S_T"]), vp(a["A_T"]), vp(a["ws"]), a["wsb"], None)


def test_pkda_validation_rejects_before_launch(lib):
    assert _pkda_call(lib, dk=24) == 6
    assert _pkda_call(lib, io=3) == 3
    assert _pkda_call(lib, beta=None) == 1
    assert _pkda_call(lib, ce=None) == 1
    assert _pkda_call(lib, A_T=None) == 1
    assert _pkda_call(lib, bp=72) == 4
    assert _pkda_call(lib, o=64 + 16) == 10
    assert _pkda_call(lib, ws=None) == 5


def test_pkda_step_validation_rejects_before_launch(lib):
    vp = ctypes.c_void_p
    base = [4, 2, 16, 16, 1.5, 0]
    ptrs = [vp(1 << 12), vp(2 << 12), vp(3 << 12), vp(4 << 12), vp(5 << 12), vp(6 << 12), vp(7 << 12),
            vp(8 << 12), vp(1 << 20), vp(2 << 20), vp(3 << 20)]
    ws = [vp(4 << 20), 256, None]
    assert lib.kdn_pkda_step(*base, *ptrs, None, 256, None) == 5
    p1 = list(ptrs)
    p1[4] = None                                               # beta
    assert lib.kdn_pkda_step(*base, *p1, *ws) == 1
    p2 = list(ptrs)
    p2[10] = vp((1 << 20) + 64)                                # o overlaps S
    assert lib.kdn_pkda_step(*base, *p2, *ws) == 10
    # the KDN step entry point does not take the PKDA variant
    assert lib.kdn_step(2, 4, 2, 16, 16, -1.0, 0, *ptrs[:6], vp(1 << 20), vp(2 << 20), vp(3 << 20), *ws) == 2
