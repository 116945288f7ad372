"""Helpers shared by the GPU parity tests: error metrics and host/device moves.

Error metrics (the tolerances the tests assert):
  max_rel        max_i |x_i - y_i| / max(|y_i|, rms(y)): relative error for
                 entries at least as large as the tensor's rms, error relative
                 to the rms below it (a plain fp32 token-by-token recurrence
                 scores ~2e-6 on these workloads; with a floor of 1% of the
                 rms it already scores ~1.3e-4, i.e. that floor measures fp32
                 rounding of near-zero outputs).  fp32 path bound: 1e-4.
  norm_max_abs   max_i |x_i - y_i| / max_i |y_i|.  bf16-io path bound: 2e-2.
"""
import numpy as np
import torch

FP32_TOL = 1e-4
BF16_TOL = 2e-2
NAMES = ("q", "k", "v", "log_alpha", "omega", "r")


def max_rel(x, y):
    x = np.asarray(x, np.float64)
    y = np.asarray(y, np.float64)
    if y.size == 0:
        return 0.0
    floor = np.sqrt(np.mean(y * y)) + 1e-300
    return float(np.max(np.abs(x - y) / np.maximum(np.abs(y), floor)))


def norm_max_abs(x, y):
    x = np.asarray(x, np.float64)
    y = np.asarray(y, np.float64)
    if y.size == 0:
        return 0.0
    return float(np.max(np.abs(x - y)) / max(np.max(np.abs(y)), 1e-300))


def err(x, y, io):
    return max_rel(x, y) if io == "f32" else norm_max_abs(x, y)


def rel_floors(x, y):
    """(rms floor, 1%-of-rms floor, no floor) per-element relative errors: the
    asserted fp32 metric, the stricter floor a plain fp32 recurrence already
    fails (see test_fp32_rounding_floor.py), and the pure element-wise value."""
    x = np.asarray(x, np.float64)
    y = np.asarray(y, np.float64)
    if y.size == 0:
        return (0.0, 0.0, 0.0)
    rms = np.sqrt(np.mean(y * y))
    d = np.abs(x - y)
    ay = np.abs(y)
    return (float(np.max(d / np.maximum(ay, rms + 1e-300))), float(np.max(d / np.maximum(ay, 1e-2 * rms + 1e-300))),
            float(np.max(d / np.maximum(ay, 1e-300))))


def report(what, got, ref, io):
    """Print the asserted error and, for fp32, the other two floors beside it
    (shown with pytest -s, and on failure)."""
    line = {}
    for name in got:
        e = err(got[name], ref[name], io)
        if io == "f32":
            a, b, c = rel_floors(got[name], ref[name])
            line[name] = f"{e:.2e} (1%-rms {b:.2e}, elementwise {c:.2e})"
        else:
            line[name] = f"{e:.2e}"
    print(f"[parity] {what} [{io}]: {line}")
    return line


def tol(io):
    return FP32_TOL if io == "f32" else BF16_TOL


def to_device(x, dev="cuda:0"):
    """numpy inputs (fp32 storage, bf16-valued for io == 'bf16') -> torch CUDA tensors."""
    io = x["io"]
    out = {}
    for n in NAMES:
        t = torch.from_numpy(np.ascontiguousarray(x[n]))
        if n in ("q", "k", "v") and io == "bf16":
            t = t.to(torch.bfloat16)   # exact: the values are bf16-representable
        out[n] = t.to(dev)
    return out


def to_host(t):
    if isinstance(t, np.ndarray):
        return t
    return t.detach().float().cpu().numpy()
