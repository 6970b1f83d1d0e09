"""Cyclic Jacobi eigensolver for real symmetric matrices, float64, LAPACK-free.

Test infrastructure: part of the oracle (see oracle/__init__.py).

Method: the classical two-sided Jacobi method (Jacobi 1846; Golub & Van Loan,
"Matrix Computations", 4th ed., section 8.5: the symmetric Schur 2x2 rotation
and the cyclic Jacobi sweep), with the sweep visited in round-robin
("tournament") order (Brent & Luk 1985; Golub & Van Loan 8.5.5).  Each round
pairs every index with exactly one other, so the n/2 rotations of a round act
on disjoint index pairs, commute, and are applied together; a sweep of n-1
rounds rotates every off-diagonal pair once.  Sweeps repeat until the
off-diagonal Frobenius norm falls to `tol` times the matrix norm.

The pages fix the eigensolver only as "sequential SVD" over the unfoldings
(Joint Tucker-rank and residual-bit KV allocator, Implementation notes) and
ST-HOSVD (Technical Summary: A JOLT for the KV Cache, Methodology 1); a
Jacobi solve is one exact way to take it.
"""
from __future__ import annotations

from typing import List, Tuple

import numpy as np


def round_robin_rounds(n: int) -> List[Tuple[np.ndarray, np.ndarray]]:
    """Index pairs of the n-1 rounds of a round-robin tournament (circle
    method).  For odd n a dummy player n is added and its pairs dropped."""
    m = n + (n % 2)
    players = list(range(m))
    rounds = []
    for _ in range(m - 1):
        p = np.array(players[: m // 2], dtype=np.int64)
        q = np.array([players[m - 1 - i] for i in range(m // 2)], dtype=np.int64)
        keep = (p < n) & (q < n)
        rounds.append((p[keep], q[keep]))
        players = [players[0], players[-1]] + players[1:-1]
    return rounds


def schur2(app: np.ndarray, apq: np.ndarray, aqq: np.ndarray):
    """Cosine/sine of the symmetric Schur rotation that zeroes a_pq
    (Golub & Van Loan, Algorithm 8.5.1), elementwise over arrays."""
    c = np.ones_like(apq)
    s = np.zeros_like(apq)
    nz = apq != 0.0
    tau = (aqq[nz] - app[nz]) / (2.0 * apq[nz])
    # t = sign(tau) / (|tau| + sqrt(1 + tau^2)), the smaller root; for
    # |tau| beyond 1e150 it is 1/(2 tau) to working precision.
    big = np.abs(tau) > 1e150
    ta = np.where(big, 1.0, np.abs(tau))
    t = np.where(big, 0.5 / np.where(big, tau, 1.0),
                 np.sign(tau + (tau == 0.0)) / (ta + np.sqrt(1.0 + ta * ta)))
    cc = 1.0 / np.sqrt(1.0 + t * t)
    c[nz] = cc
    s[nz] = t * cc
    return c, s


def jacobi_eigh(S: np.ndarray, tol: float = 1e-14, max_sweeps: int = 60):
    """Eigen-decomposition of the symmetric matrix S.

    Returns (w, V, sweeps): eigenvalues in descending order (ties broken by
    the lower original index), the matching orthonormal eigenvectors as the
    columns of V, and the number of sweeps taken.  Raises RuntimeError if the
    off-diagonal norm has not reached tol * ||S||_F after max_sweeps.
    """
    A = np.array(S, dtype=np.float64, copy=True)
    n = A.shape[0]
    if A.shape != (n, n):
        raise ValueError("square matrix expected")
    A = 0.5 * (A + A.T)
    V = np.eye(n)
    norm = np.sqrt(np.sum(A * A))
    rounds = round_robin_rounds(n)
    sweeps = 0

    def off_norm(M):
        O = M.copy()
        np.fill_diagonal(O, 0.0)
        return np.sqrt(np.sum(O * O))

    while norm > 0.0 and off_norm(A) > tol * norm:
        if sweeps >= max_sweeps:
            raise RuntimeError("Jacobi did not converge in %d sweeps" % max_sweeps)
        for p, q in rounds:
            if p.size == 0:
                continue
            c, s = schur2(A[p, p], A[p, q], A[q, q])
            # A <- A J (columns p, q), then J^T A (rows p, q); V <- V J
            ap, aq = A[:, p].copy(), A[:, q].copy()
            A[:, p] = ap * c - aq * s
            A[:, q] = ap * s + aq * c
            ap, aq = A[p, :].copy(), A[q, :].copy()
            A[p, :] = c[:, None] * ap - s[:, None] * aq
            A[q, :] = s[:, None] * ap + c[:, None] * aq
            A[p, q] = 0.0
            A[q, p] = 0.0
            vp, vq = V[:, p].copy(), V[:, q].copy()
            V[:, p] = vp * c - vq * s
            V[:, q] = vp * s + vq * c
        sweeps += 1
    w = np.diag(A).copy()
    order = np.lexsort((np.arange(n), -w))  # descending value, then index
    return w[order], V[:, order], sweeps
