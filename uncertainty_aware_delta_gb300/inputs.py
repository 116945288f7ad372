"""Seeded synthetic inputs for the KDN mixer workloads.

This module only draws random numbers and rounds them to the storage types:
it holds none of the method's arithmetic, and it is the one piece both the
CUDA path's tests and the fp64 oracle consume.

Recipe (all draws i.i.d., numpy PCG64 in fp64, in this fixed order):
  q, k       ~ N(0, 1), then L2-normalised over d_k per (b, t, h), in fp64,
               with no epsilon, before rounding;
  v          ~ N(0, 1);
  log_alpha  = -U(lo, hi) per (b, t, h, channel)   (decay per key channel);
  r          = softplus(N(0, 1)) + 1e-3 per (b, t, h)   (observation-noise variance);
  omega      ~ U(1e-4, 1e-2): per (b, t, h, channel) for the diagonal variant,
               per (b, t, h) for the isotropic variant (process-noise variance).
Rounding: fp64 -> fp32 (round to nearest even); q, k, v of bf16 workloads are
then rounded fp32 -> bf16 (round to nearest even).  Every consumer, the oracle
included, sees the rounded values.  The initial state is S_0 = 0, p_0 = 1
unless a test passes one.

PKDA (preconditioned delta rule, Preconditioned DeltaNet Sec. 2.4-2.5) draws
q, k, v and log_alpha as above, then per (b, t, h)
  beta       = sigmoid(N(0, 1))            write strength in (0, 1);
  alpha_p    = exp(-U(lo, hi))             statistic decay (same range as log_alpha);
  beta_p     = sigmoid(N(0, 1)) * scale    statistic weight (scale 1 unless a test
                                           widens it to push log A above the centre);
and per head center = exp(N(0, 0.5)) (the pages' positive log-space centre).

Gated workloads (the layer's gate pre-activations, KDN notes Sec. 5.1) draw q,
k, v as above, then the logits, stored like q, k, v (bf16 for bf16 workloads):
  alpha_logit ~ U(2.3, 6.9) per (b, t, h, channel): sigma of it lies in about
               [0.90, 0.999], the decay range of the log_alpha recipe;
  omega_logit ~ N(-6, 1): per (b, t, h, channel) (diagonal) or per (b, t, h)
               (isotropic); its softplus is about e^-6, as the omega recipe;
  r_logit     ~ N(0, 1) per (b, t, h).
The pages' models L2-normalise q and k (their architecture table), as here.

The shapes follow the KDN paper's 750M/1.3B mixer layers (16 heads of width
128, 4K training length; Sec. 5.1 and the Fig. 4 throughput setup); the pages
measure mixer speed on such layers, not on a dataset, so no dataset is
imitated here.
"""
from __future__ import annotations

import dataclasses

import numpy as np


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    variant: str          # "diag", "iso", "pkda", "dense", "backward" or "gated"
    B: int
    H: int
    T: int
    d: int                # d_k = d_v
    chunk: int
    io: str               # "f32" or "bf16" storage of q, k, v, o
    log_alpha_range: tuple
    seed: int
    prefill: int = 0      # decode workloads: tokens run by the forward path first
    steps: int = 0        # decode workloads: single-token calls after the prefill


WORKLOADS = {
    w.name: w
    for w in [
        Workload("diag-f32-b1h2t64d16", "diag", 1, 2, 64, 16, 16, "f32", (1e-3, 0.1), 20260907),
        Workload("iso-bf16-b8h16t4096d128", "iso", 8, 16, 4096, 128, 64, "bf16", (1e-3, 0.1), 20260908),
        Workload("diag-bf16-b8h16t4096d128", "diag", 8, 16, 4096, 128, 64, "bf16", (1e-3, 0.1), 20260909),
        Workload("diag-bf16-b1h16t65536d128", "diag", 1, 16, 65536, 128, 64, "bf16", (1e-4, 1e-2), 20260910),
        Workload("diag-decode-f32-s256h16d128", "diag", 256, 16, 512 + 1024, 128, 64, "f32", (1e-3, 0.1),
                 20260911, prefill=512, steps=1024),
        Workload("pkda-bf16-b8h16t4096d128", "pkda", 8, 16, 4096, 128, 64, "bf16", (1e-3, 0.1), 20260912),
        # the dense-covariance (exact) filter on the headline shape; inputs as the diagonal recipe
        Workload("dense-bf16-b8h16t4096d128", "dense", 8, 16, 4096, 128, 0, "bf16", (1e-3, 0.1), 20260913),
        # the backward pass of the diagonal forward on the headline shape; inputs as the diagonal recipe
        Workload("backward-diag-bf16-b8h16t4096d128", "backward", 8, 16, 4096, 128, 16, "bf16", (1e-3, 0.1),
                 20260914),
        # the diagonal forward driven by bf16 gate logits (fused gate prologue)
        Workload("gated-diag-bf16-b8h16t4096d128", "gated", 8, 16, 4096, 128, 64, "bf16", (1e-3, 0.1), 20260915),
    ]
}


def round_bf16(x32: np.ndarray) -> np.ndarray:
    """Round fp32 values to the nearest bf16 (ties to even); returns fp32 storage."""
    x32 = np.ascontiguousarray(x32, dtype=np.float32)
    bits = x32.view(np.uint32).astype(np.uint64)
    bias = 0x7FFF + ((bits >> 16) & 1)
    out = ((bits + bias) & 0xFFFF0000).astype(np.uint32)
    return out.view(np.float32)


def _softplus(x):
    return np.logaddexp(0.0, x)


def make_inputs(variant: str, B: int, T: int, H: int, dk: int, dv: int, io: str = "f32",
                seed: int = 0, log_alpha_range=(1e-3, 0.1), omega_range=(1e-4, 1e-2)):
    """Draw one batch; returns a dict of fp32 numpy arrays (bf16-valued where io == "bf16").

    Keys: q, k [B,T,H,dk]; v [B,T,H,dv]; log_alpha [B,T,H,dk]; r [B,T,H];
    omega [B,T,H,dk] (diag) or [B,T,H] (iso); plus "io".
    """
    if variant not in ("diag", "iso"):
        raise ValueError(variant)
    rng = np.random.Generator(np.random.PCG64(seed))
    out = {"io": io}

    def store(x64):
        x32 = x64.astype(np.float32)
        return round_bf16(x32) if io == "bf16" else x32

    for name in ("q", "k"):
        x = rng.standard_normal((B, T, H, dk))
        if dk > 0 and x.size:
            x /= np.sqrt(np.sum(x * x, axis=-1, keepdims=True))
        out[name] = store(x)
        del x
    out["v"] = store(rng.standard_normal((B, T, H, dv)))
    lo, hi = log_alpha_range
    out["log_alpha"] = (-rng.uniform(lo, hi, size=(B, T, H, dk))).astype(np.float32)
    out["r"] = (_softplus(rng.standard_normal((B, T, H))) + 1e-3).astype(np.float32)
    olo, ohi = omega_range
    oshape = (B, T, H, dk) if variant == "diag" else (B, T, H)
    out["omega"] = rng.uniform(olo, ohi, size=oshape).astype(np.float32)
    return out


def make_gated_inputs(variant: str, B: int, T: int, H: int, dk: int, dv: int, io: str = "f32",
                      seed: int = 0, alpha_logit_range=(2.3, 6.9), omega_logit_mean: float = -6.0):
    """Draw one batch of the gated recipe; returns a dict of fp32 numpy arrays
    (bf16-valued where io == "bf16").

    Keys: q, k [B,T,H,dk]; v [B,T,H,dv]; alpha_logit [B,T,H,dk]; omega_logit
    [B,T,H,dk] (diag) or [B,T,H] (iso); r_logit [B,T,H]; plus "io".
    """
    if variant not in ("diag", "iso"):
        raise ValueError(variant)
    rng = np.random.Generator(np.random.PCG64(seed))
    out = {"io": io}

    def store(x64):
        x32 = x64.astype(np.float32)
        return round_bf16(x32) if io == "bf16" else x32

    for name in ("q", "k"):
        x = rng.standard_normal((B, T, H, dk))
        if dk > 0 and x.size:
            x /= np.sqrt(np.sum(x * x, axis=-1, keepdims=True))
        out[name] = store(x)
        del x
    out["v"] = store(rng.standard_normal((B, T, H, dv)))
    lo, hi = alpha_logit_range
    out["alpha_logit"] = store(rng.uniform(lo, hi, size=(B, T, H, dk)))
    oshape = (B, T, H, dk) if variant == "diag" else (B, T, H)
    out["omega_logit"] = store(omega_logit_mean + rng.standard_normal(oshape))
    out["r_logit"] = store(rng.standard_normal((B, T, H)))
    return out


def _sigmoid(x):
    return 1.0 / (1.0 + np.exp(-x))


def make_pkda_inputs(B: int, T: int, H: int, dk: int, dv: int, io: str = "f32", seed: int = 0,
                     log_alpha_range=(1e-3, 0.1), beta_p_scale: float = 1.0):
    """Draw one PKDA batch (recipe above); returns a dict of fp32 numpy arrays.

    Keys: q, k [B,T,H,dk]; v [B,T,H,dv]; log_alpha [B,T,H,dk]; beta, alpha_p,
    beta_p [B,T,H]; center [H]; plus "io".
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    out = {"io": io}

    def store(x64):
        x32 = x64.astype(np.float32)
        return round_bf16(x32) if io == "bf16" else x32

    for name in ("q", "k"):
        x = rng.standard_normal((B, T, H, dk))
        if dk > 0 and x.size:
            x /= np.sqrt(np.sum(x * x, axis=-1, keepdims=True))
        out[name] = store(x)
        del x
    out["v"] = store(rng.standard_normal((B, T, H, dv)))
    lo, hi = log_alpha_range
    out["log_alpha"] = (-rng.uniform(lo, hi, size=(B, T, H, dk))).astype(np.float32)
    out["beta"] = _sigmoid(rng.standard_normal((B, T, H))).astype(np.float32)
    out["alpha_p"] = np.exp(-rng.uniform(lo, hi, size=(B, T, H))).astype(np.float32)
    out["beta_p"] = (_sigmoid(rng.standard_normal((B, T, H))) * beta_p_scale).astype(np.float32)
    out["center"] = np.exp(0.5 * rng.standard_normal(H)).astype(np.float32)
    return out


def workload_inputs(w: Workload, variant: str | None = None):
    """Inputs of a named workload.  ``variant`` overrides the workload's own
    (the isotropic variant is also run on the diagonal workloads' shapes, with
    its own per-(b,t,h) omega drawn from the same seed).  For a decode
    workload this returns the prefill tokens only; see :func:`decode_step_inputs`."""
    T = w.prefill if w.steps else w.T
    variant = variant or w.variant
    if variant in ("dense", "backward"):   # these take the diagonal recipe's inputs
        variant = "diag"
    if variant == "pkda":
        return make_pkda_inputs(w.B, T, w.H, w.d, w.d, w.io, w.seed, w.log_alpha_range)
    if variant == "gated":
        return make_gated_inputs("diag", w.B, T, w.H, w.d, w.d, w.io, w.seed)
    return make_inputs(variant, w.B, T, w.H, w.d, w.d, w.io, w.seed, w.log_alpha_range)


def decode_step_inputs(w: Workload, step: int, variant: str | None = None):
    """Inputs of decode step ``step`` (0-based) of a decode workload: one token
    per (sequence, head), drawn with the recipe above from seed
    ``w.seed * 4096 + 1 + step`` so any step can be regenerated on its own."""
    if (variant or w.variant) == "pkda":
        return make_pkda_inputs(w.B, 1, w.H, w.d, w.d, w.io, w.seed * 4096 + 1 + step, w.log_alpha_range)
    return make_inputs(variant or w.variant, w.B, 1, w.H, w.d, w.d, w.io, w.seed * 4096 + 1 + step,
                       w.log_alpha_range)
