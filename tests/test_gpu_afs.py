"""Parity of the adaptive-frequency-sampling path (zsolve_afs_* through the
C-ABI) with the CPU oracle (oracle/afs.py), on seeded inputs from `workload`
(malusrfworks.com, "Solving Dense Matrices Fast in the Browser", section
"Fewer frequency points: adaptive frequency sampling").

What must agree:
- the candidates solved exactly, in order (an integer decision both sides
  take in float64 on the largest residual estimate), the basis size, the
  convergence flag;
- the reduced-order solutions V y at every candidate: within 1e-8 relative
  l2 per (candidate, right-hand side).  Derivation: the two sides' exact
  solves differ by up to ~1e-11 (the refinement stops below a relative
  correction of 1e-11; the oracle solves directly), and on these workloads a
  1e-12 perturbation of the exact solves moves the model by <= 8e-11 (an
  amplification under 100 through the orthogonalisation and the q x q
  solves), so ~1e-9 is expected and 1e-8 leaves a factor of ten;
- the residual estimates: within 1e-6 + 1e-5 relative.  The Gram form
  c^H (W^T W) c - 2 Re(c^H W^T b) + ||b||^2 loses about 3q * eps * ||b||^2 of
  the SQUARED residual to cancellation, so near convergence the relative
  residual itself is resolved only to sqrt(3q * eps) ~ 1e-7 (q <= 96); both
  sides then return noise of that size (or 0 where the noise is negative),
  two orders below the stopping tolerance 1e-4.
"""
import numpy as np
import pytest

import workload
from oracle import afs as oafs
from oracle import assemble, solve

pytestmark = pytest.mark.gpu

AFS_PARITY = 1e-8


@pytest.fixture(scope="module")
def zs():
    import mixed_precision_refinement_gb300 as m
    return m


@pytest.fixture(scope="module")
def torch():
    import torch as t
    return t


def dev(torch, a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def run_gpu(zs, torch, wl, omega, zsv, B, nrhs_max=None, want_x=True, **opts):
    s = zs.Solver(wl.n, nrhs_max or B.shape[0])
    try:
        with zs.Afs(s, **opts) as a:
            L, P, G = dev(torch, wl.L), dev(torch, wl.Psi), dev(torch, wl.G)
            b = dev(torch, B)
            m = len(omega)
            x = torch.empty((m, B.shape[0], wl.n), dtype=torch.complex128, device="cuda") if want_x else None
            sampled, resid, info = a.sweep(L, P, G, omega, zsv, b, x)
            torch.cuda.synchronize()
            launches = zs.zsolve_afs_launches(a.afs)
            return sampled, resid, info, (x.cpu().numpy() if want_x else None), launches
    finally:
        s.close()


def compare(ref, sampled, resid, info, X, cand=None):
    assert sampled == ref.sampled
    assert info.n_exact == len(ref.sampled)
    assert info.q == ref.V.shape[1]
    assert bool(info.converged) == ref.converged
    m = len(ref.resid)
    idx = range(m) if cand is None else cand
    worst = 0.0
    for i in idx:
        num = np.linalg.norm(X[i] - ref.X[i], axis=1)
        den = np.linalg.norm(ref.X[i], axis=1)
        e = np.where(den > 0, num / np.where(den > 0, den, 1), num)
        worst = max(worst, float(e.max()))
    assert worst <= AFS_PARITY, worst
    r_ref = np.where(np.isfinite(ref.resid), ref.resid, 1e300)
    r_got = np.where(np.isfinite(resid), resid, 1e300)
    assert np.all(np.abs(r_got - r_ref) <= 1e-6 + 1e-5 * np.abs(r_ref))
    return worst


def test_afs_resonant_two_rhs(zs, torch):
    wl = workload.make_resonant_small(300, 7, 41, nrhs=2, psi_scale=0.1)
    ref = oafs.afs_sweep(wl.L, wl.Psi, wl.G, wl.omega, wl.zs, wl.B)
    assert len(ref.sampled) > 6  # the greedy loop runs many steps
    sampled, resid, info, X, launches = run_gpu(zs, torch, wl, wl.omega, wl.zs, wl.B)
    compare(ref, sampled, resid, info, X)
    assert info.evals == len(ref.history) and launches > 0


def test_afs_copper_physics_config0(zs, torch):
    # configuration 0's matrices over 41 candidates of its band: j*omega*L
    # dominates, two exact solves make the model exact to ~1e-11
    wl = workload.make(0)
    omega = 2 * np.pi * np.linspace(1e9, 5e9, 41)
    zsv = workload.surface_impedance(omega)
    ref = oafs.afs_sweep(wl.L, wl.Psi, wl.G, omega, zsv, wl.B)
    sampled, resid, info, X, _ = run_gpu(zs, torch, wl, omega, zsv, wl.B)
    compare(ref, sampled, resid, info, X)
    for i in (3, 20, 37):
        x = solve(assemble(wl.L, wl.Psi, wl.G, omega[i], zsv[i]), wl.B)
        assert np.linalg.norm(X[i] - x) / np.linalg.norm(x) < 1e-8


def test_afs_ragged_three_rhs(zs, torch):
    wl = workload.make_resonant_small(131, 3, 13, nrhs=3)
    ref = oafs.afs_sweep(wl.L, wl.Psi, wl.G, wl.omega, wl.zs, wl.B)
    sampled, resid, info, X, _ = run_gpu(zs, torch, wl, wl.omega, wl.zs, wl.B, nrhs_max=4)
    compare(ref, sampled, resid, info, X)


def test_afs_basis_full(zs, torch):
    wl = workload.make_resonant_small(80, 4, 21, nrhs=1, psi_scale=0.03)
    ref = oafs.afs_sweep(wl.L, wl.Psi, wl.G, wl.omega, wl.zs, wl.B, max_basis=6)
    sampled, resid, info, X, _ = run_gpu(zs, torch, wl, wl.omega, wl.zs, wl.B, max_basis=6)
    compare(ref, sampled, resid, info, X)
    assert info.basis_full == 1 and info.converged == 0


def test_afs_solve_limit(zs, torch):
    wl = workload.make_resonant_small(90, 8, 15, nrhs=1, psi_scale=0.05)
    ref = oafs.afs_sweep(wl.L, wl.Psi, wl.G, wl.omega, wl.zs, wl.B, max_solves=3)
    sampled, resid, info, X, _ = run_gpu(zs, torch, wl, wl.omega, wl.zs, wl.B, max_solves=3)
    compare(ref, sampled, resid, info, X)
    assert len(sampled) == 3


def test_afs_edge_cases(zs, torch):
    wl = workload.make_resonant_small(70, 9, 6, nrhs=1)
    # no candidates
    sampled, resid, info, X, _ = run_gpu(zs, torch, wl, wl.omega[:0], wl.zs[:0], wl.B)
    assert sampled == [] and info.converged == 1 and info.n_exact == 0
    # one candidate: exact there
    ref = oafs.afs_sweep(wl.L, wl.Psi, wl.G, wl.omega[2:3], wl.zs[2:3], wl.B)
    sampled, resid, info, X, _ = run_gpu(zs, torch, wl, wl.omega[2:3], wl.zs[2:3], wl.B)
    compare(ref, sampled, resid, info, X)
    # one exact solve allowed: only the first end
    ref = oafs.afs_sweep(wl.L, wl.Psi, wl.G, wl.omega, wl.zs, wl.B, max_solves=1)
    sampled, resid, info, X, _ = run_gpu(zs, torch, wl, wl.omega, wl.zs, wl.B, max_solves=1)
    compare(ref, sampled, resid, info, X)
    assert sampled == [0]
    # zero right-hand side: zero solutions, converged, empty basis
    Z0 = np.zeros_like(wl.B)
    sampled, resid, info, X, _ = run_gpu(zs, torch, wl, wl.omega, wl.zs, Z0)
    assert info.converged == 1 and info.q == 0 and not np.any(X) and not np.any(resid)
    # without x
    sampled2, resid2, info2, _, _ = run_gpu(zs, torch, wl, wl.omega, wl.zs, wl.B, want_x=False)
    ref = oafs.afs_sweep(wl.L, wl.Psi, wl.G, wl.omega, wl.zs, wl.B)
    assert sampled2 == ref.sampled


def test_afs_invalid_arguments(zs, torch):
    wl = workload.make_resonant_small(40, 1, 5, nrhs=2)
    s = zs.Solver(wl.n, 1)
    try:
        with pytest.raises(zs.ZsolveError):
            zs.zsolve_afs_create(s.ctx, zs.make_afs_opts(max_basis=zs.ZSOLVE_AFS_MAX_BASIS + 1))
        with pytest.raises(zs.ZsolveError):
            zs.zsolve_afs_create(s.ctx, zs.make_afs_opts(max_solves=0))
        with zs.Afs(s) as a:
            L, P, G = dev(torch, wl.L), dev(torch, wl.Psi), dev(torch, wl.G)
            with pytest.raises(zs.ZsolveError):  # two right-hand sides, room for one
                a.sweep(L, P, G, wl.omega, wl.zs, dev(torch, wl.B))
            om = wl.omega.copy()
            om[2] = -1.0
            with pytest.raises(zs.ZsolveError):
                a.sweep(L, P, G, om, wl.zs, dev(torch, wl.B[:1]))
            # the handle stays usable after a rejected call
            sampled, _, info = a.sweep(L, P, G, wl.omega, wl.zs, dev(torch, wl.B[:1]))
            assert info.n_exact == len(sampled) >= 2
    finally:
        s.close()


@pytest.mark.parametrize("kind", ["resonant", "copper"])
def test_afs_full_size_1001_candidates(zs, torch, kind):
    # the benchmark's workloads: configuration 1 (N=2157, 1 RHS) over 1001
    # candidates, with the resonant stand-in and with the copper physics
    if kind == "resonant":
        wl = workload.make_resonant(1, 1001)
        omega, zsv = wl.omega, wl.zs
    else:
        wl = workload.make(1)
        omega = 2 * np.pi * np.linspace(1e9, 10e9, 1001)
        zsv = workload.surface_impedance(omega)
    ref = oafs.afs_sweep(wl.L, wl.Psi, wl.G, omega, zsv, wl.B)
    sampled, resid, info, X, _ = run_gpu(zs, torch, wl, omega, zsv, wl.B)
    rng = np.random.default_rng(5)
    cand = sorted(set(rng.choice(1001, 24, replace=False).tolist()) | set(ref.sampled))
    compare(ref, sampled, resid, info, X, cand=cand)
    assert info.converged == 1
