"""fp64 CPU oracle for the Kalman Delta Network (KDN) mixer.

TEST INFRASTRUCTURE ONLY.  The tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may use this package; the product path (the
CUDA library and its Python binding) never imports or calls it, and this
package imports nothing from the product.

Contents
  recurrence  -- ctypes wrapper over ``kdn_oracle.c``: the token-by-token fp64
                 recurrence of Diagonal and Isotropic KDN (KDN paper Sec. 4.1,
                 Eq. 23-27 and 60-65; Sec. 4.2, Eq. 40 and App. C).
  dense       -- numpy fp64 companions used only on tiny inputs: the dense
                 exact Kalman filter (KDN paper Sec. 3.2, Eq. 12-17; Bayesian
                 Layer Prop. 1), the Moebius 2x2 matrices of the uncertainty
                 recurrence (KDN paper Eq. 32-37) and the weighted ridge
                 regression closed form (Preconditioned DeltaNet Eq. 1-5;
                 Gated KalmaNet test-time ridge regression).
  gates       -- the gate branches of the end-to-end layer (KDN reading notes
                 Sec. 5.1: alpha = sigma(.), omega = softplus(.), r = r_min +
                 softplus(.), r_min = 0.01), the effective write strength
                 beta_eff = k^T kappa (Sec. 3.2, App. B Eq. 58-61), and the
                 forward driven by gate logits.
  backward    -- numpy fp64 adjoint of the token recurrence (the gradients of
                 a weighted sum of o, S_T and p_T with respect to every input),
                 for tiny inputs; the pages give no backward pass.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
against printed values, closed forms, special-case reductions and brute force;
the backward by ``tests/test_backward_oracle.py`` against central finite
differences of the forward; the gates by ``tests/test_gates_oracle.py``.
"""
from .recurrence import build_oracle, forward, step, library_path  # noqa: F401
from .dense import (  # noqa: F401
    dense_kalman,
    mobius_matrices,
    mobius_apply,
    mobius_product,
    ridge_closed_form,
)
from . import gates  # noqa: F401,E402
