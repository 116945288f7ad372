"""Thin ctypes binding over ``libkdn.so`` (include/kdn.h).

Argument marshalling only: every step of the mixer runs in the library's
CUDA kernels.  Tensors are PyTorch CUDA tensors (PyTorch supplies device
memory and the current stream); there is no CPU fallback, and a missing
library raises immediately.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libkdn.so")
_lock = threading.Lock()
_lib = None

KDN_F32, KDN_BF16 = 0, 1
KDN_DIAG, KDN_ISO, KDN_PKDA = 0, 1, 2
KDN_FLAG_PORTABLE = 0x1
KDN_FLAG_NO_SPLIT = 0x2
KDN_FLAG_TIMEOUT_PROBE = 0x100   # test facility of the bounded-wait path (include/kdn.h)

EXPORTED = (
    "kdn_workspace_size", "kdn_diag_forward", "kdn_iso_forward", "kdn_step",
    "kdn_read_device_status", "kdn_status_string", "kdn_abi_version", "kdn_forward_kernel_count",
    "kdn_forward_noalloc", "kdn_pkda_forward", "kdn_pkda_step", "kdn_dense_forward", "kdn_step_ex",
    "kdn_backward", "kdn_backward_workspace_size", "kdn_gated_forward", "kdn_gated_workspace_size",
    "kdn_dense_workspace_size",
)


class KDNError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: status {status} ({status_string(status)})")
        self.status = status


def library_path() -> str:
    return _PATH


def library():
    """Load libkdn.so (once); raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_PATH):
                raise RuntimeError(
                    f"{_PATH} is missing: build it with uncertainty_aware_delta_gb300.build.build_library() "
                    "(there is no fallback implementation)")
            lib = ctypes.CDLL(_PATH)
            vp, fp, i32, u32, f32, sz = (ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                                         ctypes.c_uint32, ctypes.c_float, ctypes.c_size_t)
            lib.kdn_workspace_size.restype = sz
            lib.kdn_workspace_size.argtypes = [i32] * 8 + [u32]
            fwd = [i32] * 6 + [f32, i32, u32] + [vp] * 3 + [fp] * 5 + [vp, fp, fp] + [vp, sz, vp]
            for name in ("kdn_diag_forward", "kdn_iso_forward"):
                getattr(lib, name).restype = i32
                getattr(lib, name).argtypes = fwd
            lib.kdn_step.restype = i32
            lib.kdn_step.argtypes = [i32] * 5 + [f32, i32] + [vp] * 3 + [fp] * 3 + [fp, fp, vp] + [vp, sz, vp]
            lib.kdn_step_ex.restype = i32
            lib.kdn_step_ex.argtypes = [i32] * 5 + [f32, i32, u32] + [vp] * 3 + [fp] * 3 + [fp, fp, vp] + \
                [vp, sz, vp]
            lib.kdn_pkda_forward.restype = i32
            lib.kdn_pkda_forward.argtypes = [i32] * 6 + [f32, i32, u32] + [vp] * 3 + [fp] * 5 + \
                [fp, fp] + [vp, fp, fp] + [vp, sz, vp]
            lib.kdn_pkda_step.restype = i32
            lib.kdn_pkda_step.argtypes = [i32] * 4 + [f32, i32] + [vp] * 3 + [fp] * 5 + [fp, fp, vp] + \
                [vp, sz, vp]
            lib.kdn_read_device_status.restype = i32
            lib.kdn_read_device_status.argtypes = [vp, vp]
            lib.kdn_status_string.restype = ctypes.c_char_p
            lib.kdn_status_string.argtypes = [i32]
            lib.kdn_forward_kernel_count.restype = i32
            lib.kdn_forward_kernel_count.argtypes = [i32] * 8 + [u32]
            lib.kdn_forward_noalloc.restype = i32
            lib.kdn_forward_noalloc.argtypes = [i32] * 7 + [f32, i32, u32] + [vp] * 3 + [fp] * 5 + \
                [vp, fp, fp, vp, vp]
            lib.kdn_dense_forward.restype = i32
            lib.kdn_dense_forward.argtypes = [i32] * 5 + [vp] * 3 + [fp] * 5 + [vp, fp, fp] + [vp, sz, vp]
            lib.kdn_dense_workspace_size.restype = sz
            lib.kdn_dense_workspace_size.argtypes = [i32] * 5
            lib.kdn_backward_workspace_size.restype = sz
            lib.kdn_backward_workspace_size.argtypes = [i32] * 7
            lib.kdn_backward.restype = i32
            lib.kdn_backward.argtypes = [i32] * 6 + [f32, i32] + [vp] * 3 + [fp] * 5 + [vp, fp, fp] + [fp] * 8 + \
                [vp, sz, vp]
            lib.kdn_gated_workspace_size.restype = sz
            lib.kdn_gated_workspace_size.argtypes = [i32] * 8 + [u32]
            lib.kdn_gated_forward.restype = i32
            lib.kdn_gated_forward.argtypes = [i32] * 7 + [f32, f32, i32, u32] + [vp] * 6 + [fp, fp] + \
                [vp, fp, fp, fp] + [vp, sz, vp]
            lib.kdn_abi_version.restype = i32
            lib.kdn_abi_version.argtypes = []
            _lib = lib
    return _lib


def status_string(status: int) -> str:
    return library().kdn_status_string(int(status)).decode()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream, device):
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def _check(t, name, dtype, shape, device):
    if t is None:
        return
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if t.dtype != dtype:
        raise TypeError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def workspace_size(variant, B, T, H, dk, dv, chunk=0, io=KDN_BF16, flags=0) -> int:
    return int(library().kdn_workspace_size(variant, B, T, H, dk, dv, chunk, io, flags))


def forward_kernel_count(variant, B, T, H, dk, dv, chunk=0, io=KDN_BF16, flags=0) -> int:
    """Kernels one forward call with these arguments enqueues."""
    return int(library().kdn_forward_kernel_count(variant, B, T, H, dk, dv, chunk, io, flags))


def _forward(variant, q, k, v, log_alpha, omega, r, S0, p0, mu, chunk, flags, out, workspace,
             stream):
    lib = library()
    device = q.device
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    io = KDN_BF16 if q.dtype == torch.bfloat16 else KDN_F32
    iot = torch.bfloat16 if io == KDN_BF16 else torch.float32
    nu = (dk,) if variant == KDN_DIAG else ()
    _check(q, "q", iot, (B, T, H, dk), device)
    _check(k, "k", iot, (B, T, H, dk), device)
    _check(v, "v", iot, (B, T, H, dv), device)
    _check(log_alpha, "log_alpha", torch.float32, (B, T, H, dk), device)
    _check(omega, "omega", torch.float32, (B, T, H) + nu, device)
    _check(r, "r", torch.float32, (B, T, H), device)
    _check(S0, "S0", torch.float32, (B, H, dk, dv), device)
    _check(p0, "p0", torch.float32, (B, H) + nu, device)
    if out is None:
        o = torch.empty((B, T, H, dv), dtype=iot, device=device)
        S_T = torch.empty((B, H, dk, dv), dtype=torch.float32, device=device)
        p_T = torch.empty((B, H) + nu, dtype=torch.float32, device=device)
    else:
        o, S_T, p_T = out
        _check(o, "o", iot, (B, T, H, dv), device)
        _check(S_T, "S_T", torch.float32, (B, H, dk, dv), device)
        _check(p_T, "p_T", torch.float32, (B, H) + nu, device)
    need = lib.kdn_workspace_size(variant, B, T, H, dk, dv, chunk, io, flags)
    if need == 0:
        raise KDNError(6, "kdn_workspace_size rejected the arguments")
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=device)
    elif workspace.numel() * workspace.element_size() < need:
        raise ValueError(f"workspace holds {workspace.numel()} bytes, {need} needed")
    fn = lib.kdn_diag_forward if variant == KDN_DIAG else lib.kdn_iso_forward
    mu = -1.0 if mu is None else float(mu)
    with torch.cuda.device(device):
        st = fn(B, T, H, dk, dv, int(chunk), mu, io, int(flags), _ptr(q), _ptr(k), _ptr(v),
                _ptr(log_alpha), _ptr(omega), _ptr(r), _ptr(S0), _ptr(p0), _ptr(o), _ptr(S_T),
                _ptr(p_T), _ptr(workspace), workspace.numel() * workspace.element_size(),
                _stream(stream, device))
    if st != 0:
        raise KDNError(st, fn.__name__)
    return o, S_T, p_T


def kdn_diag_forward(q, k, v, log_alpha, omega, r, S0=None, p0=None, *, mu=None, chunk=0, flags=0,
                     out=None, workspace=None, stream=None):
    """Diagonal KDN forward (KDN paper Sec. 4.1).  Returns (o, S_T, p_T).

    q, k [B,T,H,dk] and v [B,T,H,dv] in fp32 or bf16; log_alpha, omega
    [B,T,H,dk], r [B,T,H] fp32; optional S0 [B,H,dk,dv], p0 [B,H,dk] fp32.
    mu=None selects d_k.  ``out=(o, S_T, p_T)`` writes into given tensors.
    """
    return _forward(KDN_DIAG, q, k, v, log_alpha, omega, r, S0, p0, mu, chunk, flags, out,
                    workspace, stream)


def kdn_iso_forward(q, k, v, log_alpha, omega, r, S0=None, p0=None, *, mu=None, chunk=0, flags=0,
                    out=None, workspace=None, stream=None):
    """Isotropic KDN forward (KDN paper Sec. 4.2): omega [B,T,H], p0/p_T [B,H]."""
    return _forward(KDN_ISO, q, k, v, log_alpha, omega, r, S0, p0, mu, chunk, flags, out,
                    workspace, stream)


def gated_workspace_size(variant, B, T, H, dk, dv, chunk=0, io=KDN_BF16, flags=0) -> int:
    return int(library().kdn_gated_workspace_size(variant, B, T, H, dk, dv, chunk, io, flags))


def kdn_gated_forward(variant, q, k, v, alpha_logit, omega_logit, r_logit, S0=None, p0=None, *, mu=None,
                      r_min=None, chunk=0, flags=0, beta_eff=False, out=None, workspace=None, stream=None):
    """KDN forward driven by gate pre-activations (KDN notes Sec. 5.1):
    alpha = sigmoid(alpha_logit), omega = softplus(omega_logit), r = r_min +
    softplus(r_logit).  Returns (o, S_T, p_T, beta_eff or None).

    variant: "diag" / "iso" (or KDN_DIAG / KDN_ISO).  The logits have the io dtype
    of q: alpha_logit [B,T,H,dk], omega_logit [B,T,H,dk] (diag) or [B,T,H] (iso),
    r_logit [B,T,H].  r_min=None selects 0.01.  ``beta_eff=True`` also returns the
    effective write strength k^T kappa [B,T,H] fp32 (or pass a tensor to fill).
    ``out=(o, S_T, p_T)`` writes into given tensors.
    """
    variant = {"diag": KDN_DIAG, "iso": KDN_ISO}.get(variant, variant)
    lib = library()
    device = q.device
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    io = KDN_BF16 if q.dtype == torch.bfloat16 else KDN_F32
    iot = torch.bfloat16 if io == KDN_BF16 else torch.float32
    nu = (dk,) if variant == KDN_DIAG else ()
    _check(q, "q", iot, (B, T, H, dk), device)
    _check(k, "k", iot, (B, T, H, dk), device)
    _check(v, "v", iot, (B, T, H, dv), device)
    _check(alpha_logit, "alpha_logit", iot, (B, T, H, dk), device)
    _check(omega_logit, "omega_logit", iot, (B, T, H) + nu, device)
    _check(r_logit, "r_logit", iot, (B, T, H), device)
    _check(S0, "S0", torch.float32, (B, H, dk, dv), device)
    _check(p0, "p0", torch.float32, (B, H) + nu, device)
    if out is None:
        o = torch.empty((B, T, H, dv), dtype=iot, device=device)
        S_T = torch.empty((B, H, dk, dv), dtype=torch.float32, device=device)
        p_T = torch.empty((B, H) + nu, dtype=torch.float32, device=device)
    else:
        o, S_T, p_T = out
        _check(o, "o", iot, (B, T, H, dv), device)
        _check(S_T, "S_T", torch.float32, (B, H, dk, dv), device)
        _check(p_T, "p_T", torch.float32, (B, H) + nu, device)
    if beta_eff is True:
        be = torch.empty((B, T, H), dtype=torch.float32, device=device)
    elif beta_eff is False or beta_eff is None:
        be = None
    else:
        be = beta_eff
        _check(be, "beta_eff", torch.float32, (B, T, H), device)
    need = lib.kdn_gated_workspace_size(variant, B, T, H, dk, dv, chunk, io, flags)
    if need == 0:
        raise KDNError(6, "kdn_gated_workspace_size rejected the arguments")
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=device)
    elif workspace.numel() * workspace.element_size() < need:
        raise ValueError(f"workspace holds {workspace.numel()} bytes, {need} needed")
    mu = -1.0 if mu is None else float(mu)
    r_min = -1.0 if r_min is None else float(r_min)
    with torch.cuda.device(device):
        st = lib.kdn_gated_forward(variant, B, T, H, dk, dv, int(chunk), mu, r_min, io, int(flags), _ptr(q),
                                   _ptr(k), _ptr(v), _ptr(alpha_logit), _ptr(omega_logit), _ptr(r_logit),
                                   _ptr(S0), _ptr(p0), _ptr(o), _ptr(S_T), _ptr(p_T), _ptr(be), _ptr(workspace),
                                   workspace.numel() * workspace.element_size(), _stream(stream, device))
    if st != 0:
        raise KDNError(st, "kdn_gated_forward")
    return o, S_T, p_T, be


def kdn_step(variant, q, k, v, log_alpha, omega, r, S, p, *, mu=None, o=None, workspace=None,
             stream=None, flags=0):
    """One decode token per sequence; S and p are updated in place.  Returns o [B,H,dv].
    flags (kdn_step_ex): 0, or KDN_FLAG_TIMEOUT_PROBE in tests of the bounded-wait path."""
    lib = library()
    variant = {"diag": KDN_DIAG, "iso": KDN_ISO}.get(variant, variant)
    device = q.device
    B, H, dk = q.shape
    dv = v.shape[-1]
    io = KDN_BF16 if q.dtype == torch.bfloat16 else KDN_F32
    iot = torch.bfloat16 if io == KDN_BF16 else torch.float32
    nu = (dk,) if variant == KDN_DIAG else ()
    _check(q, "q", iot, (B, H, dk), device)
    _check(k, "k", iot, (B, H, dk), device)
    _check(v, "v", iot, (B, H, dv), device)
    _check(log_alpha, "log_alpha", torch.float32, (B, H, dk), device)
    _check(omega, "omega", torch.float32, (B, H) + nu, device)
    _check(r, "r", torch.float32, (B, H), device)
    _check(S, "S", torch.float32, (B, H, dk, dv), device)
    _check(p, "p", torch.float32, (B, H) + nu, device)
    if o is None:
        o = torch.empty((B, H, dv), dtype=iot, device=device)
    _check(o, "o", iot, (B, H, dv), device)
    need = lib.kdn_workspace_size(variant, B, 1, H, dk, dv, 0, io, 0)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=device)
    mu = -1.0 if mu is None else float(mu)
    with torch.cuda.device(device):
        args = (_ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(omega), _ptr(r), _ptr(S), _ptr(p), _ptr(o),
                _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream, device))
        if flags:
            st = lib.kdn_step_ex(variant, B, H, dk, dv, mu, io, int(flags), *args)
        else:
            st = lib.kdn_step(variant, B, H, dk, dv, mu, io, *args)
    if st != 0:
        raise KDNError(st, "kdn_step")
    return o


def kdn_pkda_forward(q, k, v, log_alpha, beta, alpha_p, beta_p, center, S0=None, A0=None, *, x=1.5,
                     chunk=0, flags=0, out=None, workspace=None, stream=None):
    """Preconditioned delta rule with per-channel decay (Preconditioned DeltaNet
    Sec. 2.4 Eq. 9, Sec. 2.5).  Returns (o, S_T, A_T).

    q, k [B,T,H,dk] and v [B,T,H,dv] in fp32 or bf16; log_alpha [B,T,H,dk];
    beta, alpha_p, beta_p [B,T,H]; center [H]; optional S0 [B,H,dk,dv] and
    A0 [B,H,dk] (the key statistic; zero when omitted).  ``x`` bounds the
    write scale to [1/x, x].  ``out=(o, S_T, A_T)`` writes into given tensors.
    """
    lib = library()
    device = q.device
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    io = KDN_BF16 if q.dtype == torch.bfloat16 else KDN_F32
    iot = torch.bfloat16 if io == KDN_BF16 else torch.float32
    f32 = torch.float32
    for t, name, dt, shp in ((q, "q", iot, (B, T, H, dk)), (k, "k", iot, (B, T, H, dk)),
                             (v, "v", iot, (B, T, H, dv)), (log_alpha, "log_alpha", f32, (B, T, H, dk)),
                             (beta, "beta", f32, (B, T, H)), (alpha_p, "alpha_p", f32, (B, T, H)),
                             (beta_p, "beta_p", f32, (B, T, H)), (center, "center", f32, (H,)),
                             (S0, "S0", f32, (B, H, dk, dv)), (A0, "A0", f32, (B, H, dk))):
        _check(t, name, dt, shp, device)
    if out is None:
        o = torch.empty((B, T, H, dv), dtype=iot, device=device)
        S_T = torch.empty((B, H, dk, dv), dtype=f32, device=device)
        A_T = torch.empty((B, H, dk), dtype=f32, device=device)
    else:
        o, S_T, A_T = out
        _check(o, "o", iot, (B, T, H, dv), device)
        _check(S_T, "S_T", f32, (B, H, dk, dv), device)
        _check(A_T, "A_T", f32, (B, H, dk), device)
    need = lib.kdn_workspace_size(KDN_PKDA, B, T, H, dk, dv, chunk, io, flags)
    if need == 0:
        raise KDNError(6, "kdn_workspace_size rejected the arguments")
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=device)
    elif workspace.numel() * workspace.element_size() < need:
        raise ValueError(f"workspace holds {workspace.numel()} bytes, {need} needed")
    with torch.cuda.device(device):
        st = lib.kdn_pkda_forward(B, T, H, dk, dv, int(chunk), float(x), io, int(flags), _ptr(q), _ptr(k),
                                  _ptr(v), _ptr(log_alpha), _ptr(beta), _ptr(alpha_p), _ptr(beta_p),
                                  _ptr(center), _ptr(S0), _ptr(A0), _ptr(o), _ptr(S_T), _ptr(A_T),
                                  _ptr(workspace), workspace.numel() * workspace.element_size(),
                                  _stream(stream, device))
    if st != 0:
        raise KDNError(st, "kdn_pkda_forward")
    return o, S_T, A_T


def kdn_pkda_step(q, k, v, log_alpha, beta, alpha_p, beta_p, center, S, A, *, x=1.5, o=None,
                  workspace=None, stream=None):
    """One PKDA decode token per sequence; S and A are updated in place.  Returns o [B,H,dv]."""
    lib = library()
    device = q.device
    B, H, dk = q.shape
    dv = v.shape[-1]
    io = KDN_BF16 if q.dtype == torch.bfloat16 else KDN_F32
    iot = torch.bfloat16 if io == KDN_BF16 else torch.float32
    f32 = torch.float32
    if o is None:
        o = torch.empty((B, H, dv), dtype=iot, device=device)
    for t, name, dt, shp in ((q, "q", iot, (B, H, dk)), (k, "k", iot, (B, H, dk)), (v, "v", iot, (B, H, dv)),
                             (log_alpha, "log_alpha", f32, (B, H, dk)), (beta, "beta", f32, (B, H)),
                             (alpha_p, "alpha_p", f32, (B, H)), (beta_p, "beta_p", f32, (B, H)),
                             (center, "center", f32, (H,)), (S, "S", f32, (B, H, dk, dv)),
                             (A, "A", f32, (B, H, dk)), (o, "o", iot, (B, H, dv))):
        _check(t, name, dt, shp, device)
    need = lib.kdn_workspace_size(KDN_PKDA, B, 1, H, dk, dv, 0, io, 0)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=device)
    with torch.cuda.device(device):
        st = lib.kdn_pkda_step(B, H, dk, dv, float(x), io, _ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha),
                               _ptr(beta), _ptr(alpha_p), _ptr(beta_p), _ptr(center), _ptr(S), _ptr(A),
                               _ptr(o), _ptr(workspace), workspace.numel() * workspace.element_size(),
                               _stream(stream, device))
    if st != 0:
        raise KDNError(st, "kdn_pkda_step")
    return o


def kdn_forward_noalloc(variant, q, k, v, log_alpha, omega, r, S0=None, p0=None, *, mu=None,
                        chunk=0, flags=0, out, status_out=None, stream=None):
    """Forward that allocates nothing: for callers that may not allocate device
    memory where they run the mixer.  Its scratch is the library's built-in
    static device array (include/kdn.h, KDN_STATIC_SCRATCH_BYTES), shared by
    every call in the process, so calls must not overlap on the GPU.  The
    outputs ``out=(o, S_T, p_T)`` are required (this wrapper creates no
    tensors); ``status_out`` is an optional int32 CUDA tensor of one element
    that receives the device status word.
    """
    lib = library()
    variant = {"diag": KDN_DIAG, "iso": KDN_ISO}.get(variant, variant)
    device = q.device
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    io = KDN_BF16 if q.dtype == torch.bfloat16 else KDN_F32
    iot = torch.bfloat16 if io == KDN_BF16 else torch.float32
    nu = (dk,) if variant == KDN_DIAG else ()
    o, S_T, p_T = out
    for t, name, dt, shp in ((q, "q", iot, (B, T, H, dk)), (k, "k", iot, (B, T, H, dk)),
                             (v, "v", iot, (B, T, H, dv)), (log_alpha, "log_alpha", torch.float32, (B, T, H, dk)),
                             (omega, "omega", torch.float32, (B, T, H) + nu), (r, "r", torch.float32, (B, T, H)),
                             (S0, "S0", torch.float32, (B, H, dk, dv)), (p0, "p0", torch.float32, (B, H) + nu),
                             (o, "o", iot, (B, T, H, dv)), (S_T, "S_T", torch.float32, (B, H, dk, dv)),
                             (p_T, "p_T", torch.float32, (B, H) + nu)):
        _check(t, name, dt, shp, device)
    if status_out is not None:
        _check(status_out, "status_out", torch.int32, (1,), device)
    mu = -1.0 if mu is None else float(mu)
    with torch.cuda.device(device):
        st = lib.kdn_forward_noalloc(variant, B, T, H, dk, dv, int(chunk), mu, io, int(flags), _ptr(q),
                                     _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(omega), _ptr(r), _ptr(S0),
                                     _ptr(p0), _ptr(o), _ptr(S_T), _ptr(p_T), _ptr(status_out),
                                     _stream(stream, device))
    if st != 0:
        raise KDNError(st, "kdn_forward_noalloc")
    return o, S_T, p_T


def dense_workspace_size(B, T, H, d, io=KDN_BF16) -> int:
    return int(library().kdn_dense_workspace_size(B, T, H, d, io))


def kdn_dense_forward(q, k, v, log_alpha, omega, r, S0=None, P0=None, *, out=None, workspace=None, stream=None):
    """Dense-covariance (exact) Kalman memory forward (KDN paper Sec. 3.2).  Returns (o, S_T, P_T).

    q, k, v [B,T,H,d] in fp32 or bf16 (d in 32, 64, 128); log_alpha, omega [B,T,H,d],
    r [B,T,H] fp32; optional S0 [B,H,d,d] (zero) and P0 [B,H,d,d] (identity) fp32.
    ``out=(o, S_T, P_T)`` writes into given tensors; ``workspace`` (uint8 device
    tensor of dense_workspace_size() bytes) is allocated when not given.
    """
    lib = library()
    device = q.device
    B, T, H, d = q.shape
    io = KDN_BF16 if q.dtype == torch.bfloat16 else KDN_F32
    iot = torch.bfloat16 if io == KDN_BF16 else torch.float32
    for t, name, dt, shape in ((q, "q", iot, (B, T, H, d)), (k, "k", iot, (B, T, H, d)),
                               (v, "v", iot, (B, T, H, d)), (log_alpha, "log_alpha", torch.float32, (B, T, H, d)),
                               (omega, "omega", torch.float32, (B, T, H, d)), (r, "r", torch.float32, (B, T, H)),
                               (S0, "S0", torch.float32, (B, H, d, d)), (P0, "P0", torch.float32, (B, H, d, d))):
        _check(t, name, dt, shape, device)
    if out is None:
        o = torch.empty((B, T, H, d), dtype=iot, device=device)
        S_T = torch.empty((B, H, d, d), dtype=torch.float32, device=device)
        P_T = torch.empty((B, H, d, d), dtype=torch.float32, device=device)
    else:
        o, S_T, P_T = out
        _check(o, "o", iot, (B, T, H, d), device)
        _check(S_T, "S_T", torch.float32, (B, H, d, d), device)
        _check(P_T, "P_T", torch.float32, (B, H, d, d), device)
    need = lib.kdn_dense_workspace_size(B, T, H, d, io)
    if need == 0:
        raise KDNError(6, "kdn_dense_workspace_size rejected the arguments")
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=device)
    elif workspace.numel() * workspace.element_size() < need:
        raise ValueError(f"workspace holds {workspace.numel()} bytes, {need} needed")
    with torch.cuda.device(device):
        st = lib.kdn_dense_forward(B, T, H, d, io, _ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(omega),
                                   _ptr(r), _ptr(S0), _ptr(P0), _ptr(o), _ptr(S_T), _ptr(P_T), _ptr(workspace),
                                   workspace.numel() * workspace.element_size(), _stream(stream, device))
    if st != 0:
        raise KDNError(st, "kdn_dense_forward")
    return o, S_T, P_T


def kdn_backward(variant, q, k, v, log_alpha, omega, r, S0=None, p0=None, dO=None, dS_T=None, dp_T=None, *,
                 mu=None, workspace=None, stream=None):
    """Gradients of sum(dO o) + sum(dS_T S_T) + sum(dp_T p_T) of the KDN forward with these
    inputs.  Returns a dict of fp32 tensors: q, k, v, log_alpha, omega, r, S0, p0."""
    lib = library()
    variant = {"diag": KDN_DIAG, "iso": KDN_ISO}.get(variant, variant)
    device = q.device
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    io = KDN_BF16 if q.dtype == torch.bfloat16 else KDN_F32
    iot = torch.bfloat16 if io == KDN_BF16 else torch.float32
    nu = (dk,) if variant == KDN_DIAG else ()
    for t, name, dt, shape in ((q, "q", iot, (B, T, H, dk)), (k, "k", iot, (B, T, H, dk)),
                               (v, "v", iot, (B, T, H, dv)), (log_alpha, "log_alpha", torch.float32, (B, T, H, dk)),
                               (omega, "omega", torch.float32, (B, T, H) + nu), (r, "r", torch.float32, (B, T, H)),
                               (S0, "S0", torch.float32, (B, H, dk, dv)), (p0, "p0", torch.float32, (B, H) + nu),
                               (dO, "dO", iot, (B, T, H, dv)), (dS_T, "dS_T", torch.float32, (B, H, dk, dv)),
                               (dp_T, "dp_T", torch.float32, (B, H) + nu)):
        _check(t, name, dt, shape, device)
    f = dict(dtype=torch.float32, device=device)
    g = {"q": torch.empty((B, T, H, dk), **f), "k": torch.empty((B, T, H, dk), **f),
         "v": torch.empty((B, T, H, dv), **f), "log_alpha": torch.empty((B, T, H, dk), **f),
         "omega": torch.empty((B, T, H) + nu, **f), "r": torch.empty((B, T, H), **f),
         "S0": torch.empty((B, H, dk, dv), **f), "p0": torch.empty((B, H) + nu, **f)}
    need = lib.kdn_backward_workspace_size(variant, B, T, H, dk, dv, io)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=device)
    mu = -1.0 if mu is None else float(mu)
    with torch.cuda.device(device):
        st = lib.kdn_backward(variant, B, T, H, dk, dv, mu, io, _ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha),
                              _ptr(omega), _ptr(r), _ptr(S0), _ptr(p0), _ptr(dO), _ptr(dS_T), _ptr(dp_T),
                              *(_ptr(g[n]) for n in ("q", "k", "v", "log_alpha", "omega", "r", "S0", "p0")),
                              _ptr(workspace), workspace.numel() * workspace.element_size(),
                              _stream(stream, device))
    if st != 0:
        raise KDNError(st, "kdn_backward")
    return g


def kdn_read_device_status(workspace, stream=None) -> int:
    """Synchronise the stream and return the device status word of ``workspace``."""
    lib = library()
    with torch.cuda.device(workspace.device):
        return int(lib.kdn_read_device_status(_ptr(workspace), _stream(stream, workspace.device)))
