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
- the residual estimates, which decide the stop and the next solve (both
  decisions are checked exactly above): within each candidate's rounding
  floor plus 1e-6 relative.  The estimate is sqrt(s) with
  s = c^H M c - 2 Re(c^H W^T b) + ||b||^2, M = W^T W.  Each entry of M and
  W^T b is a length-n dot product (error <= n eps ||W_a|| ||W_b||), and the
  quadratic form adds 3q + 1 more roundings per term; with
  |M_ab| <= ||W_a|| ||W_b|| the error in s is at most
  (n + 3q + 1) eps (sum_a |c_a| ||W_a|| + ||b||)^2 on each side, so two
  sides differ in sqrt(s) / ||b|| by at most
  sqrt(2 (n + 3q + 1) eps) (sum_a |c_a| ||W_a|| / ||b|| + 1).  Near a
  resonance j*omega*L V y and -j*Psi V y/omega nearly cancel, sum_a |c_a| ||W_a||
  is many times ||b|| and the floor reaches ~1e-5, still below the stopping
  tolerance 1e-4.
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
    s = zs.Solver(wl.n, nrhs_max or B.shape[0], batch=2)  # AFS solves at most two frequencies at once
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


def estimate_floor(wl, ref, omega, zsv, B):
    """Per candidate: the bound on |estimate_gpu - estimate_oracle| from
    rounding (see the module docstring), from the oracle's basis."""
    V = ref.V
    n, q = V.shape
    m = len(ref.resid)
    if q == 0:
        return np.zeros(m)
    *_, M, _, _, bb = oafs.reduced_terms(wl.L, wl.Psi, wl.G, V, B)
    wn = np.sqrt(np.maximum(np.diag(M), 0.0))
    k = np.sqrt(2.0 * (n + 3 * q + 1) * np.finfo(np.float64).eps)
    out = np.zeros(m)
    for i in range(m):
        for r in range(B.shape[0]):
            if bb[r] == 0:
                continue
            y = ref.Y[i, r]
            c = np.concatenate([1j * omega[i] * y, -1j * y / omega[i], zsv[i] * y])
            out[i] = max(out[i], k * (np.sum(np.abs(c) * wn) / np.sqrt(bb[r]) + 1.0))
    return out



def compare(ref, got, wl, omega, zsv, B, cand=None):
    sampled, resid, info, X = got[:4]
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
    floor = estimate_floor(wl, ref, omega, zsv, B)
    diff = np.abs(r_got - r_ref)
    bad = diff > floor + 1e-6 * np.abs(r_ref) + 1e-12
    assert not np.any(bad), (np.flatnonzero(bad)[:8], diff[bad][:8], floor[bad][:8])
    return worst


def test_afs_resonant_two_rhs(zs, torch):
    wl = workload.make_resonant_small(300, 7, 41, nrhs=2, psi_scale=0.1)
    ref = oafs.afs_sweep(wl.L, wl.Psi, wl.G, wl.omega, wl.zs, wl.B)
    assert len(ref.sampled) > 6  # the greedy loop runs many steps
    got = run_gpu(zs, torch, wl, wl.omega, wl.zs, wl.B)
    sampled, resid, info, X, launches = got
    compare(ref, got, wl, wl.omega, wl.zs, wl.B)
    assert info.evals == len(ref.history) and launches > 0


def test_afs_copper_physics_config0(zs, torch):
    # configuration 0's matrices over 41 candidates of its band: j*omega*L
    # dominates, two exact solves make the model exact to ~1e-11
    wl = workload.make(0)
    omega = 2 * np.pi * np.linspace(1e9, 5e9, 41)
    zsv = workload.surface_impedance(omega)
    ref = oafs.afs_sweep(wl.L, wl.Psi, wl.G, omega, zsv, wl.B)
    got = run_gpu(zs, torch, wl, omega, zsv, wl.B)
    sampled, resid, info, X, _ = got
    compare(ref, got, wl, omega, zsv, wl.B)
    for i in (3, 20, 37):
        x = solve(assemble(wl.L, wl.Psi, wl.G, omega[i], zsv[i]), wl.B)
        assert np.linalg.norm(X[i] - x) / np.linalg.norm(x) < 1e-8


def test_afs_ragged_three_rhs(zs, torch):
    wl = workload.make_resonant_small(131, 3, 13, nrhs=3)
    ref = oafs.afs_sweep(wl.L, wl.Psi, wl.G, wl.omega, wl.zs, wl.B)
    got = run_gpu(zs, torch, wl, wl.omega, wl.zs, wl.B, nrhs_max=4)
    sampled, resid, info, X, _ = got
    compare(ref, got, wl, wl.omega, wl.zs, wl.B)


def test_afs_basis_full(zs, torch):
    wl = workload.make_resonant_small(80, 4, 21, nrhs=1, psi_scale=0.03)
    ref = oafs.afs_sweep(wl.L, wl.Psi, wl.G, wl.omega, wl.zs, wl.B, max_basis=6)
    got = run_gpu(zs, torch, wl, wl.omega, wl.zs, wl.B, max_basis=6)
    sampled, resid, info, X, _ = got
    compare(ref, got, wl, wl.omega, wl.zs, wl.B)
    assert info.basis_full == 1 and info.converged == 0


def test_afs_solve_limit(zs, torch):
    wl = workload.make_resonant_small(90, 8, 15, nrhs=1, psi_scale=0.05)
    ref = oafs.afs_sweep(wl.L, wl.Psi, wl.G, wl.omega, wl.zs, wl.B, max_solves=3)
    got = run_gpu(zs, torch, wl, wl.omega, wl.zs, wl.B, max_solves=3)
    sampled, resid, info, X, _ = got
    compare(ref, got, wl, wl.omega, wl.zs, wl.B)
    assert len(sampled) == 3


def test_afs_edge_cases(zs, torch):
    wl = workload.make_resonant_small(70, 9, 6, nrhs=1)
    # no candidates
    got = run_gpu(zs, torch, wl, wl.omega[:0], wl.zs[:0], wl.B)
    sampled, resid, info, X, _ = got
    assert sampled == [] and info.converged == 1 and info.n_exact == 0
    # one candidate: exact there
    ref = oafs.afs_sweep(wl.L, wl.Psi, wl.G, wl.omega[2:3], wl.zs[2:3], wl.B)
    got = run_gpu(zs, torch, wl, wl.omega[2:3], wl.zs[2:3], wl.B)
    compare(ref, got, wl, wl.omega[2:3], wl.zs[2:3], wl.B)
    # one exact solve allowed: only the first end
    ref = oafs.afs_sweep(wl.L, wl.Psi, wl.G, wl.omega, wl.zs, wl.B, max_solves=1)
    got = run_gpu(zs, torch, wl, wl.omega, wl.zs, wl.B, max_solves=1)
    sampled, resid, info, X, _ = got
    compare(ref, got, wl, wl.omega, wl.zs, wl.B)
    assert sampled == [0]
    # zero right-hand side: zero solutions, converged, empty basis
    Z0 = np.zeros_like(wl.B)
    got = run_gpu(zs, torch, wl, wl.omega, wl.zs, Z0)
    sampled, resid, info, X, _ = got
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


@pytest.mark.parametrize("kind", ["resonant", "resonant_psi0.1", "copper"])
def test_afs_full_size_1001_candidates(zs, torch, kind):
    # the benchmark's workloads: configuration 1 (N=2157, 1 RHS) over 1001
    # candidates, with the resonant stand-in (Psi x 0.3: 5 exact solves, q = 10;
    # Psi x 0.1: 32 exact solves, q = 64) and with the copper physics
    if kind.startswith("resonant"):
        wl = workload.make_resonant(1, 1001, psi_scale=0.1 if kind.endswith("0.1") else workload.AFS_PSI_SCALE)
        omega, zsv = wl.omega, wl.zs
    else:
        wl = workload.make(1)
        omega = 2 * np.pi * np.linspace(1e9, 10e9, 1001)
        zsv = workload.surface_impedance(omega)
    ref = oafs.afs_sweep(wl.L, wl.Psi, wl.G, omega, zsv, wl.B)
    got = run_gpu(zs, torch, wl, omega, zsv, wl.B)
    rng = np.random.default_rng(5)
    cand = sorted(set(rng.choice(1001, 24, replace=False).tolist()) | set(ref.sampled))
    compare(ref, got, wl, omega, zsv, wl.B, cand=cand)
    assert got[2].converged == 1


def test_afs_two_handles_on_one_context(zs, torch):
    # a handle with a small basis created after one with a large basis must
    # not shrink the shared memory the large one's evaluations need
    wl = workload.make_resonant_small(300, 7, 41, nrhs=2, psi_scale=0.1)  # q = 56
    ref = oafs.afs_sweep(wl.L, wl.Psi, wl.G, wl.omega, wl.zs, wl.B)
    s = zs.Solver(wl.n, 2, batch=2)
    try:
        with zs.Afs(s) as big, zs.Afs(s, max_basis=8) as small:
            L, P, G = dev(torch, wl.L), dev(torch, wl.Psi), dev(torch, wl.G)
            b = dev(torch, wl.B)
            _, _, info_small = small.sweep(L, P, G, wl.omega, wl.zs, b)
            assert info_small.q <= 8
            x = torch.empty((len(wl.omega), 2, wl.n), dtype=torch.complex128, device="cuda")
            sampled, resid, info = big.sweep(L, P, G, wl.omega, wl.zs, b, x)
            torch.cuda.synchronize()
            got = (sampled, resid, info, x.cpu().numpy())
            compare(ref, got, wl, wl.omega, wl.zs, wl.B)
    finally:
        s.close()
