"""The block form of the dense covariance recurrence, checked on the CPU against
the oracle's token-by-token filter (KDN paper Sec. 3.2, Eq. 12-17).

The d = 128 covariance pass of the CUDA path runs blocks of up to 16 tokens.
Inside a block every token's y is a combination of u_j = (Ptil + diag(dacc_j)) w_j
taken with the covariance of the block start, through the elimination
H(j, .) = Gamma(j, .) - sum_{i<j} s_i H(i, j) H(i, .) on Gamma(l, j) = u_l . w_j.
The decay is held outside the covariance about a per-channel reference in the
middle of the block's log decay, and a block ends where some channel's log decay
would exceed 40.  This test restates that algebra in fp64 numpy (independent of
the kernel's code) and pins it to the exact filter: the gains and the final
covariance agree to rounding, also with strongly decaying channels, a single
token of log decay -150 (a block of its own) and lengths that are not multiples
of the block.  It documents why the kernel's restructuring is exact; GPU parity
of the kernel itself is in test_parity_dense.py.
"""
import numpy as np
import pytest

from oracle.dense import dense_kalman


def _block_form(k, la, om, r, P0, M=16, limit=40.0):
    T, d = k.shape
    kap = np.zeros((T, d))
    Pt = P0.copy()
    prev_end = np.zeros(d)
    t0 = 0
    while t0 < T:
        n = min(M, T - t0)
        K = np.zeros((M, d)); L = np.zeros((M, d)); W = np.zeros((M, d)); R = np.ones(M)
        K[:n] = k[t0:t0 + n]; L[:n] = la[t0:t0 + n]; W[:n] = om[t0:t0 + n]; R[:n] = r[t0:t0 + n]
        Lc = np.cumsum(L, axis=0)
        m = n   # block length: up to the first token (after the first) beyond the bound
        for j in range(1, n):
            if np.any(np.abs(Lc[j]) > limit):
                m = j
                break
        Lend = Lc[m - 1]
        ref = np.where(np.abs(Lend) > limit, Lend, 0.5 * Lend)
        f = np.exp(ref + prev_end)              # change of frame into this block
        prev_end = Lend - ref
        Pt = f[:, None] * Pt * f[None, :]
        G = np.ones((M, d)); Wm = np.zeros((M, d)); dacc = np.zeros((M, d)); acc = np.zeros(d)
        for j in range(m):
            G[j] = np.exp(Lc[j] - ref)
            Wm[j] = G[j] * K[j]
            acc = acc + W[j] / G[j] ** 2
            dacc[j] = acc
        dacc[m:] = acc
        R[m:] = 1.0
        U = dacc * Wm + Wm @ Pt
        Gam = U @ Wm.T
        H = Gam.copy(); s = np.zeros(M); N = np.zeros((M, M))
        for j in range(M):
            s[j] = 1.0 / (R[j] + H[j, j])
            for jp in range(j + 1, M):
                N[jp, j] = s[j] * H[j, jp]
                H[jp, :] -= N[jp, j] * H[j, :]
        Y = np.zeros((M, d))
        for j in range(M):
            Y[j] = U[j] - N[j, :j] @ Y[:j]
        for j in range(m):
            kap[t0 + j] = s[j] * G[j] * Y[j]
        Pt = Pt + np.diag(dacc[-1]) - (Y.T * s) @ Y
        t0 += m
    E = np.exp(prev_end)
    return kap, E[:, None] * Pt * E[None, :]


@pytest.mark.parametrize("d, T, mode", [(16, 37, "plain"), (16, 50, "strong"), (16, 40, "single"), (8, 5, "plain"),
                                        (12, 33, "strong")])
def test_block_form_equals_token_by_token_filter(d, T, mode):
    rng = np.random.default_rng(100 + T + d)
    k = rng.standard_normal((T, d)) / np.sqrt(d)
    la = -rng.uniform(0.001, 0.1, (T, d))
    if mode == "strong":
        la[:, :3] = -2.4
    if mode == "single":
        la[5, 2] = -150.0
        la[20:24, 1] = -30.0
    om = rng.uniform(0.0, 0.05, (T, d))
    r = rng.uniform(0.01, 0.1, T)
    A = rng.standard_normal((d, d))
    P0 = A @ A.T / d + 0.1 * np.eye(d)
    ref = dense_kalman(k, np.zeros((T, 1)), np.zeros((T, d)), r, np.zeros((d, 1)), P0, D=np.exp(la), Omega=om)
    kap, P_T = _block_form(k, la, om, r, P0)
    assert np.max(np.abs(kap - ref["kappa"])) <= 1e-12 * np.max(np.abs(ref["kappa"]))
    assert np.max(np.abs(P_T - ref["P_T"])) <= 1e-12 * np.max(np.abs(ref["P_T"]))
