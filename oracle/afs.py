"""Adaptive frequency sampling (AFS) reduced-order model, CPU oracle --
TEST INFRASTRUCTURE ONLY (same rule as the rest of `oracle/`: only tests,
the smoke check and the CPU legs of the benchmark import it).

Follows malusrfworks.com, "Solving Dense Matrices Fast in the Browser",
section "Fewer frequency points: adaptive frequency sampling", whose four
steps are taken in the page's order:

1. a handful of candidates get full solves; the real and imaginary parts of
   those solutions, made orthonormal, are the columns of a real basis V;
2. projecting the three frequency-independent matrices onto V gives a q x q
   system Z_r = j*omega*V^T L V - j*V^T Psi V/omega + Zs*V^T G V;
3. every candidate gets the residual ||Z(omega) V y - b|| of its small-system
   answer, and the worst one is the next full solve;
4. the loop ends once no candidate's residual reaches 1e-4.

Readings of points the page leaves open (each restated where it is used):
- "a few frequencies" to start: the two ends of the candidate list (only the
  first if the list has one entry or one exact solve is allowed);
- the residual is relative, ||Z V y - b||_2 / ||b||_2, per right-hand side,
  and a candidate's residual is the largest over its right-hand sides;
- y solves the Galerkin system Z_r y = V^T b (the page solves the small
  system at each frequency; with V real, V^T is the projection);
- the residual estimate uses only small quantities, as the page says: with
  W = [L V | Psi V | G V] (n x 3q) and c = [j*omega*y; -j*y/omega; Zs*y],
  Z V y = W c, so ||Z V y - b||^2 = c^H (W^T W) c - 2 Re(c^H W^T b) + ||b||^2;
- orthonormalisation is classical Gram-Schmidt applied twice; a vector whose
  norm after both passes is at most `drop` times its norm before is dropped
  as already in the span;
- the next exact solve is at the largest residual among the candidates not
  yet solved exactly, the lowest index on ties;
- the loop also stops when the solve or basis limits are reached (reported
  as not converged);
- the output at every candidate, the exactly solved ones included, is the
  reduced-order solution V y (the page: it matches the exact solution there).

Exact solves use this package's complex128 LU with partial pivoting; the
q x q reduced systems use LAPACK through numpy (a library step).
"""
from __future__ import annotations

import dataclasses

import numpy as np

from . import assemble, solve


@dataclasses.dataclass
class AfsResult:
    X: np.ndarray            # (m, nrhs, n) complex128: V y at every candidate
    sampled: list            # candidate indices solved exactly, in order
    resid: np.ndarray        # (m,) final estimated relative residual (max over RHS)
    history: list            # per evaluation: the (m,) residual estimates
    V: np.ndarray            # (n, q) orthonormal real basis
    Y: np.ndarray            # (m, nrhs, q) complex reduced solutions
    converged: bool
    exact: dict              # candidate index -> (nrhs, n) exact solution used


def orth_append(V: np.ndarray, v: np.ndarray, drop: float):
    """Classical Gram-Schmidt, two passes; returns (V with v appended, kept)."""
    v = np.array(v, dtype=np.float64)
    n0 = np.linalg.norm(v)
    if not np.isfinite(n0) or n0 == 0.0:
        return V, False
    for _ in range(2):
        h = V.T @ v
        v = v - V @ h
    n1 = np.linalg.norm(v)
    if not n1 > drop * n0:
        return V, False
    return np.column_stack([V, v / n1]), True


def reduced_terms(L, Psi, G, V, B):
    """Everything step 2 and the residual estimate need, from one basis."""
    LV, PV, GV = L @ V, Psi @ V, G @ V
    Lr, Pr, Gr = V.T @ LV, V.T @ PV, V.T @ GV
    W = np.hstack([LV, PV, GV])
    M = W.T @ W
    Bt = np.atleast_2d(B).T                       # (n, nrhs)
    wb = W.T @ Bt                                  # (3q, nrhs) complex
    br = V.T @ Bt                                  # (q, nrhs) complex
    bb = np.sum(np.abs(np.atleast_2d(B)) ** 2, axis=1)
    return Lr, Pr, Gr, M, wb, br, bb


def reduced_matrix(Lr, Pr, Gr, omega: float, zs: complex) -> np.ndarray:
    """Z_r = j*omega*Lr - j*Pr/omega + Zs*Gr, parts in the order the formula is written."""
    zs = complex(zs)
    return (zs.real * Gr) + 1j * ((omega * Lr - Pr / omega) + zs.imag * Gr)


def residual_estimate(y: np.ndarray, omega: float, zs: complex, M, wb_r, bb_r) -> float:
    """||Z V y - b|| / ||b|| from the small Gram quantities (see the header);
    0 for a zero right-hand side (whose solution, zero, is exact)."""
    if bb_r == 0.0:
        return 0.0
    c = np.concatenate([1j * omega * y, -1j * y / omega, complex(zs) * y])
    s = np.real(np.conj(c) @ (M @ c)) - 2.0 * np.real(np.conj(c) @ wb_r) + bb_r
    return float(np.sqrt(max(s, 0.0) / bb_r))


def evaluate(Lr, Pr, Gr, M, wb, br, bb, omega, zs):
    """Steps 2-3 at every candidate: reduced solutions and residual estimates."""
    m, nrhs, q = len(omega), br.shape[1], br.shape[0]
    Y = np.zeros((m, nrhs, q), dtype=np.complex128)
    res = np.zeros((m, nrhs))
    for i in range(m):
        Zr = reduced_matrix(Lr, Pr, Gr, omega[i], zs[i])
        try:
            Yi = np.linalg.solve(Zr, br)           # (q, nrhs)
        except np.linalg.LinAlgError:              # exactly singular: y = 0, estimate +inf
            res[i] = np.inf
            continue
        for r in range(nrhs):
            Y[i, r] = Yi[:, r]
            res[i, r] = residual_estimate(Yi[:, r], omega[i], zs[i], M, wb[:, r], bb[r])
    return Y, res.max(axis=1)


def afs_sweep(L, Psi, G, omega, zs, B, tol: float = 1e-4, max_solves: int = 32,
              max_basis: int = 96, drop: float = 1e-8) -> AfsResult:
    """The adaptive frequency sampling loop over the candidate list omega.
    The exact solves are the oracle's own assembly and direct solve."""
    L, Psi, G = (np.asarray(a, dtype=np.float64) for a in (L, Psi, G))
    B = np.atleast_2d(np.asarray(B, dtype=np.complex128))
    omega = np.asarray(omega, dtype=np.float64)
    zs = np.asarray(zs, dtype=np.complex128)
    n, nrhs, m = L.shape[0], B.shape[0], len(omega)
    V = np.zeros((n, 0))
    sampled, history, exact = [], [], {}
    pending = [0] if (m == 1 or max_solves == 1) else [0, m - 1]
    converged, full = False, False
    Y = np.zeros((m, nrhs, 0), dtype=np.complex128)
    resid = np.full(m, np.inf)
    while m > 0:
        # step 1: exact solves, real and imaginary parts into the basis
        for k in pending:
            Xk = solve(assemble(L, Psi, G, omega[k], zs[k]), B)
            exact[k] = Xk
            sampled.append(k)
            for r in range(nrhs):
                for part in (Xk[r].real, Xk[r].imag):
                    if V.shape[1] >= max_basis:
                        full = True
                        break
                    V, _ = orth_append(V, part, drop)
        # steps 2-3 at every candidate
        terms = reduced_terms(L, Psi, G, V, B)
        Y, resid = evaluate(*terms, omega, zs)
        history.append(resid.copy())
        # step 4
        worst = np.where(np.isnan(resid), np.inf, resid).max()
        if worst < tol:
            converged = True
            break
        if len(sampled) >= min(max_solves, m) or full:
            break
        rest = np.array([i for i in range(m) if i not in set(sampled)])
        pending = [int(rest[np.argmax(resid[rest])])]
    X = np.einsum("nq,mrq->mrn", V, Y) if m else np.zeros((0, nrhs, n), dtype=np.complex128)
    return AfsResult(X, sampled, resid, history, V, Y, converged, exact)
