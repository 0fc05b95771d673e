"""Pins of the adaptive-frequency-sampling oracle (oracle/afs.py) against
what the page and the mathematics fix, not against the oracle itself
(malusrfworks.com, "Solving Dense Matrices Fast in the Browser", section
"Fewer frequency points: adaptive frequency sampling"):

- the residual estimate built from q-sized quantities equals the residual
  of the full system, ||Z(omega) x - b|| / ||b|| with Z assembled in
  complex128 and x = V y (catches a wrong sign or factor in c, a missing
  term of the Gram expansion);
- Z_r equals V^T Z(omega) V of the assembled Z and is symmetric, since V is
  real (the page: reciprocity is kept);
- at an exactly solved frequency the model reproduces the exact solution
  (the page states the model reproduces the full solution there);
- once the basis spans R^n the model is exact at every candidate;
- every greedy pick is the candidate with the largest true residual;
- after convergence the error obeys ||x - V y|| / ||x|| <= cond(Z) * residual;
- a zero right-hand side, a single candidate and a full basis behave as the
  readings in the oracle's header say.
"""
from __future__ import annotations

import numpy as np
import pytest

import workload as wlm
from oracle import afs, assemble, backward_error, solve


def _direct_residual(wl, i, x):
    Z = assemble(wl.L, wl.Psi, wl.G, wl.omega[i], wl.zs[i])
    return backward_error(Z, x, wl.B)


@pytest.fixture(scope="module")
def res_case():
    wl = wlm.make_resonant_small(120, 11, 17, nrhs=2, psi_scale=0.1)
    r = afs.afs_sweep(wl.L, wl.Psi, wl.G, wl.omega, wl.zs, wl.B)
    return wl, r


def test_orth_append_orthonormal_and_drops_span():
    rng = np.random.default_rng(0)
    n = 50
    V = np.zeros((n, 0))
    vs = [rng.normal(size=n) for _ in range(6)]
    for v in vs:
        V, kept = afs.orth_append(V, v, 1e-8)
        assert kept
    assert np.abs(V.T @ V - np.eye(6)).max() < 1e-14
    for v in vs:  # every input lies in the span
        assert np.linalg.norm(v - V @ (V.T @ v)) < 1e-13 * np.linalg.norm(v)
    comb = 0.3 * vs[0] - 2.0 * vs[4]
    V2, kept = afs.orth_append(V, comb, 1e-8)
    assert not kept and V2.shape == V.shape
    V3, kept = afs.orth_append(V, np.zeros(n), 1e-8)
    assert not kept


def test_residual_estimate_equals_full_residual(res_case):
    wl, _ = res_case
    # a basis from two exact solves, then every candidate
    V = np.zeros((wl.n, 0))
    for k in (0, len(wl.omega) - 1):
        X = solve(assemble(wl.L, wl.Psi, wl.G, wl.omega[k], wl.zs[k]), wl.B)
        for r in range(X.shape[0]):
            for part in (X[r].real, X[r].imag):
                V, _ = afs.orth_append(V, part, 1e-8)
    terms = afs.reduced_terms(wl.L, wl.Psi, wl.G, V, wl.B)
    Lr, Pr, Gr, M, wb, br, bb = terms
    checked = 0
    for i in range(len(wl.omega)):
        y = np.linalg.solve(afs.reduced_matrix(Lr, Pr, Gr, wl.omega[i], wl.zs[i]), br)
        x = (V @ y).T
        direct = _direct_residual(wl, i, x)
        for r in range(wl.B.shape[0]):
            est = afs.residual_estimate(y[:, r], wl.omega[i], wl.zs[i], M, wb[:, r], bb[r])
            if direct[r] > 1e-5:
                assert est == pytest.approx(direct[r], rel=1e-6)
                checked += 1
            else:  # floor of the Gram form: ~sqrt(3q * eps) of the relative residual
                assert abs(est - direct[r]) < 1e-6
    assert checked > 10


def test_reduced_matrix_is_projection_and_symmetric(res_case):
    wl, r = res_case
    V = r.V
    Lr, Pr, Gr, *_ = afs.reduced_terms(wl.L, wl.Psi, wl.G, V, wl.B)
    for i in (0, 5, 16):
        Zr = afs.reduced_matrix(Lr, Pr, Gr, wl.omega[i], wl.zs[i])
        Z = assemble(wl.L, wl.Psi, wl.G, wl.omega[i], wl.zs[i])
        P = V.T @ Z @ V
        assert np.abs(Zr - P).max() < 1e-12 * np.abs(P).max()
        assert np.abs(Zr - Zr.T).max() < 1e-12 * np.abs(Zr).max()


def test_exact_at_sampled_frequencies(res_case):
    wl, r = res_case
    assert r.converged and len(r.sampled) >= 3
    for k in r.sampled:
        x = solve(assemble(wl.L, wl.Psi, wl.G, wl.omega[k], wl.zs[k]), wl.B)
        err = np.linalg.norm(r.X[k] - x) / np.linalg.norm(x)
        assert err < 1e-10, (k, err)


def test_spanning_basis_is_exact_everywhere():
    wl = wlm.make_resonant_small(6, 5, 5, nrhs=1, psi_scale=0.1)
    r = afs.afs_sweep(wl.L, wl.Psi, wl.G, wl.omega, wl.zs, wl.B, tol=1e-300, max_solves=3)
    assert r.V.shape[1] == 6 and not r.converged
    for i in range(5):
        Z = assemble(wl.L, wl.Psi, wl.G, wl.omega[i], wl.zs[i])
        x = np.linalg.solve(Z, wl.B.T).T  # LAPACK, independent of the oracle's LU
        assert np.linalg.norm(r.X[i] - x) / np.linalg.norm(x) < 1e-11


def test_greedy_pick_is_largest_true_residual(res_case):
    wl, r = res_case
    m = len(wl.omega)
    for j in range(2, len(r.sampled)):
        part = afs.afs_sweep(wl.L, wl.Psi, wl.G, wl.omega, wl.zs, wl.B, max_solves=j)
        assert part.sampled == r.sampled[:j]
        rest = [i for i in range(m) if i not in part.sampled]
        true = [max(_direct_residual(wl, i, part.X[i])) for i in rest]
        assert rest[int(np.argmax(true))] == r.sampled[j]


def test_converged_error_within_condition_bound(res_case):
    wl, r = res_case
    for i in range(len(wl.omega)):
        Z = assemble(wl.L, wl.Psi, wl.G, wl.omega[i], wl.zs[i])
        x = solve(Z, wl.B)
        err = np.linalg.norm(r.X[i] - x, axis=1) / np.linalg.norm(x, axis=1)
        bound = np.linalg.cond(Z) * max(r.resid[i], 1e-8)
        assert np.all(err <= 1.01 * bound + 1e-12), (i, err, bound)
        assert r.resid[i] < 1e-4


def test_zero_rhs_and_single_candidate():
    wl = wlm.make_resonant_small(40, 2, 7, nrhs=1)
    z = afs.afs_sweep(wl.L, wl.Psi, wl.G, wl.omega, wl.zs, np.zeros_like(wl.B))
    assert z.converged and z.V.shape[1] == 0 and not np.any(z.X) and not np.any(z.resid)
    one = afs.afs_sweep(wl.L, wl.Psi, wl.G, wl.omega[3:4], wl.zs[3:4], wl.B)
    assert one.sampled == [0] and one.converged
    x = solve(assemble(wl.L, wl.Psi, wl.G, wl.omega[3], wl.zs[3]), wl.B)
    assert np.linalg.norm(one.X[0] - x) / np.linalg.norm(x) < 1e-11


def test_full_basis_stops_unconverged():
    wl = wlm.make_resonant_small(80, 4, 21, nrhs=1, psi_scale=0.03)
    r = afs.afs_sweep(wl.L, wl.Psi, wl.G, wl.omega, wl.zs, wl.B, max_basis=6)
    assert not r.converged and r.V.shape[1] == 6
    # two ends and one pick fill the six columns; the next pick's vectors find
    # no room, which ends the loop
    assert len(r.sampled) == 4
