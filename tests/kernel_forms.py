"""Kernel-structured forms used only by the tests.

These restate, in fp64 numpy, how a tensor-core kernel would organise a
computation (its blocking, its choice of reference tokens), so that a test can
check that organisation against the plain definition.  They are not part of
the oracle, which holds only the definitions and their independent
restatements.
"""
import numpy as np


def kda_intra_blocks(q, k, Gam, beta, sub=16, split=8):
    """A (strictly lower) and P (lower, with the diagonal) of one KDA chunk,
    written the way a tensor-core kernel forms them (fp64 here): the pairwise
    factor e^{Gam_i - Gam_j} (one per key channel) is never formed for j in an
    earlier sub-chunk; instead both operands are rescaled to a reference token
    r between them, k_i e^{Gam_i - Gam_r} and k_j e^{Gam_r - Gam_j} (both
    factors at most 1), and only pairs inside one ``split``-token block take
    the pairwise factor.  Sub-chunks of ``sub`` tokens use r = the token
    before the sub-chunk; inside a sub-chunk, the halves of ``split`` tokens
    use r = the last token of the first half.  q, k: [n][dk]; Gam: [n][dk]
    cumulative log decays; beta: [n].  Returns (A, P)."""
    n = q.shape[0]
    A = np.zeros((n, n))
    P = np.zeros((n, n))

    def cross(i_rows, j_rows, r):
        ql = q[i_rows] * np.exp(Gam[i_rows] - Gam[r])
        kl = k[i_rows] * np.exp(Gam[i_rows] - Gam[r])
        kr = k[j_rows] * np.exp(Gam[r] - Gam[j_rows])
        P[np.ix_(i_rows, j_rows)] = ql @ kr.T
        A[np.ix_(i_rows, j_rows)] = beta[i_rows][:, None] * (kl @ kr.T)

    for I0 in range(0, n, sub):
        I1 = min(I0 + sub, n)
        if I0 > 0:
            cross(np.arange(I0, I1), np.arange(0, I0), I0 - 1)
        for h0 in range(I0, I1, split):
            h1 = min(h0 + split, I1)
            if h0 > I0:
                cross(np.arange(h0, h1), np.arange(I0, h0), h0 - 1)
            for i in range(h0, h1):
                for j in range(h0, i + 1):
                    f = np.exp(Gam[i] - Gam[j])
                    P[i, j] = np.sum(q[i] * k[j] * f)
                    if j < i:
                        A[i, j] = beta[i] * np.sum(k[i] * k[j] * f)
    return A, P
