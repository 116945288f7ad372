"""GB300-native Kalman Delta Network (KDN) mixer.

The compute lives in ``libkdn.so`` (CUDA kernels for sm_103a behind the C ABI
of ``include/kdn.h``); :mod:`.binding` is a thin ctypes layer over it that
takes PyTorch CUDA tensors.  :mod:`.inputs` draws the seeded synthetic
workloads.  The library is loaded on first use and its absence is an error:
there is no CPU fallback.
"""
from .binding import (  # noqa: F401
    KDN_BF16,
    KDN_DIAG,
    KDN_F32,
    KDN_FLAG_NO_SPLIT,
    KDN_FLAG_PORTABLE,
    KDN_FLAG_TIMEOUT_PROBE,
    KDN_ISO,
    KDN_PKDA,
    KDNError,
    kdn_backward,
    kdn_diag_forward,
    kdn_forward_noalloc,
    kdn_gated_forward,
    kdn_iso_forward,
    kdn_dense_forward,
    kdn_pkda_forward,
    kdn_pkda_step,
    kdn_read_device_status,
    kdn_step,
    dense_workspace_size,
    forward_kernel_count,
    gated_workspace_size,
    library,
    library_path,
    status_string,
    workspace_size,
)
