"""The two factorisation modes through the C-ABI: symmetric (opts.symmetric
= 1, the default) and the full trailing update (0).

Z(omega) is complex symmetric (malusrfworks.com, "Solving Dense Matrices Fast
in the Browser", section "Measure first": exploiting the symmetry halves the
factorisation's work against LU).  For an unpivoted LU of a complex
symmetric matrix U = D L^T holds in exact arithmetic, with D = diag(U); in
this mode the trailing update forms only the lower tiles and each U12 solve
takes A12^T from A21.  Checked here:
- the float32 factors reconstruct the float32 matrix as well as the full
  mode's do, their upper part is D L^T up to float32-class rounding, and they
  are the unpivoted LU of the oracle up to the same rounding;
- sweeps agree with the oracle's complex128 direct solve to 1e-10 (ragged
  sizes, several right-hand sides, batched and two-lane, the N=2157 sweep);
- an input that is not symmetric is still solved to the same bar (the
  double-precision residual uses all of Z).
"""
import numpy as np
import pytest

import oracle
import workload

pytestmark = pytest.mark.gpu

PARITY = 1e-10
FACTOR_TOL = {"TF32X3": 2e-5, "TF32": 3e-3}
LDLT_TOL = {"TF32X3": 1e-3, "TF32": 0.3}


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


def rel_err(x, ref):
    x, ref = np.atleast_2d(x), np.atleast_2d(ref)
    return np.linalg.norm(x - ref, axis=-1) / np.linalg.norm(ref, axis=-1)


@pytest.mark.parametrize("sym", [1, 0])
@pytest.mark.parametrize("gemm", ["TF32X3", "TF32"])
@pytest.mark.parametrize("n", [129, 300, 513, 1000])
def test_symmetric_factor_is_ldlt(zs, torch, n, gemm, sym):
    wl = workload.make_small(n, seed=20 + n, nf=1)
    s = zs.Solver(n, 1, gemm=getattr(zs, "ZSOLVE_GEMM_" + gemm), symmetric=sym)
    try:
        zs.zsolve_assemble(s.ctx, dev(torch, wl.L), dev(torch, wl.Psi), dev(torch, wl.G), wl.omega[0],
                           wl.zs[0].real, wl.zs[0].imag)
        re = torch.empty((n, n), dtype=torch.float32, device="cuda")
        im = torch.empty_like(re)
        zs.zsolve_get_z32(s.ctx, re, im)
        Z32 = (re.cpu().numpy() + 1j * im.cpu().numpy()).astype(np.complex128)
        assert np.array_equal(Z32, Z32.T)
        zs.zsolve_factor(s.ctx)
        assert zs.zsolve_pivot_flag(s.ctx) == 0
        zs.zsolve_get_z32(s.ctx, re, im)
        LU = re.cpu().numpy().astype(np.float64) + 1j * im.cpu().numpy()
        Lf = np.tril(LU, -1) + np.eye(n)
        Uf = np.triu(LU)
        err = np.linalg.norm(Lf @ Uf - Z32) / np.linalg.norm(Z32)
        assert err < FACTOR_TOL[gemm], err
        D = np.diag(Uf)
        ldlt = np.linalg.norm(np.triu(Uf, 1) - np.triu(D[:, None] * Lf.T, 1)) / np.linalg.norm(Uf)
        assert ldlt < LDLT_TOL[gemm], ldlt  # holds for both modes: U = D L^T for a symmetric Z
        LUo, st = oracle.lu_nopiv(Z32)
        assert st == 0
        assert np.linalg.norm(LU - LUo) / np.linalg.norm(LUo) < LDLT_TOL[gemm]
    finally:
        s.close()


@pytest.mark.parametrize("sym", [1, 0])
@pytest.mark.parametrize("gemm", ["TF32X3", "TF32"])
@pytest.mark.parametrize("n,nrhs,nf,batch", [(1, 1, 2, 0), (130, 3, 4, 3), (301, 4, 3, 0), (257, 8, 2, 1),
                                              (700, 1, 3, 3)])
def test_symmetric_sweep_parity(zs, torch, n, nrhs, nf, batch, gemm, sym):
    wl = workload.make_small(n, seed=40 + n, nf=nf, nrhs=nrhs, f_lo=0.5e9, f_hi=20e9)
    ref = oracle.solve_sweep(wl)
    s = zs.Solver(n, nrhs, gemm=getattr(zs, "ZSOLVE_GEMM_" + gemm), batch=batch, symmetric=sym)
    try:
        x = torch.empty((nf, nrhs, n), dtype=torch.complex128, device="cuda")
        infos = zs.zsolve_sweep(s.ctx, dev(torch, wl.L), dev(torch, wl.Psi), dev(torch, wl.G), wl.omega, wl.zs,
                                dev(torch, wl.B), x)
        X = x.cpu().numpy()
        for f in range(nf):
            assert infos[f].status == 0
            assert np.all(rel_err(X[f], ref[f]) <= PARITY), (f, rel_err(X[f], ref[f]), infos[f].as_dict())
    finally:
        s.close()


@pytest.mark.parametrize("sym", [1, 0])
def test_symmetric_config1_full_sweep(zs, torch, config1_oracle, sym):
    """N=2157, all 21 frequencies in one batched sweep, two lanes: the
    oracle's direct solve at every frequency to the parity bound, and the
    oracle's backward error of every returned x."""
    wl, ref_all = config1_oracle
    nf = len(wl.omega)
    s = zs.Solver(wl.n, 1, batch=nf, symmetric=sym)
    try:
        x = torch.empty((nf, 1, wl.n), dtype=torch.complex128, device="cuda")
        infos = zs.zsolve_sweep(s.ctx, dev(torch, wl.L), dev(torch, wl.Psi), dev(torch, wl.G), wl.omega, wl.zs,
                                dev(torch, wl.B), x)
        X = x.cpu().numpy()
        for f in range(nf):
            assert infos[f].status == 0 and infos[f].fallback == 0, infos[f].as_dict()
            Z = oracle.assemble(wl.L, wl.Psi, wl.G, wl.omega[f], wl.zs[f])
            R = oracle.residual(Z, X[f], wl.B)
            eta = np.linalg.norm(R, axis=1) / (np.linalg.norm(Z) * np.linalg.norm(X[f], axis=1)
                                               + np.linalg.norm(wl.B, axis=1))
            assert np.all(eta < 1e-15), (f, eta)
        errs = np.array([rel_err(X[f], ref_all[f]).max() for f in range(nf)])
        assert np.all(errs <= PARITY), errs
    finally:
        s.close()


@pytest.mark.parametrize("sym", [1, 0])
@pytest.mark.parametrize("gemm", ["TF32X3", "TF32"])
def test_tcgen05_many_tiles_per_cta(zs, torch, monkeypatch, gemm, sym):
    """The tcgen05 launches capped at 2, 3 or 8 CTAs (ZSOLVE_TC_GRID, a
    testing aid), so that every CTA takes many tiles and the epilogue, the
    MMA issuer and the loads drift apart by the most their barriers allow:
    the sweep is bit-identical to the uncapped one (a tile's result does not
    depend on the CTA that forms it) and matches the oracle."""
    n, nrhs, nf = 1000, 2, 3
    wl = workload.make_small(n, seed=77, nf=nf, nrhs=nrhs, f_lo=0.5e9, f_hi=20e9)
    ref = oracle.solve_sweep(wl)
    out = {}
    for cap in ("", "2", "3", "8"):
        if cap:
            monkeypatch.setenv("ZSOLVE_TC_GRID", cap)
        else:
            monkeypatch.delenv("ZSOLVE_TC_GRID", raising=False)
        s = zs.Solver(n, nrhs, gemm=getattr(zs, "ZSOLVE_GEMM_" + gemm), batch=nf, symmetric=sym)
        try:
            x = torch.empty((nf, nrhs, n), dtype=torch.complex128, device="cuda")
            infos = zs.zsolve_sweep(s.ctx, dev(torch, wl.L), dev(torch, wl.Psi), dev(torch, wl.G), wl.omega,
                                    wl.zs, dev(torch, wl.B), x)
            out[cap] = x.cpu().numpy()
        finally:
            s.close()
        assert all(i.status == 0 for i in infos)
        for f in range(nf):
            assert np.all(rel_err(out[cap][f], ref[f]) <= PARITY), (cap, f)
    for cap in ("2", "3", "8"):
        assert np.array_equal(out[cap], out[""]), cap


@pytest.mark.parametrize("gemm", ["TF32X3", "TF32"])
@pytest.mark.parametrize("n,nrhs,nf,batch", [(1000, 2, 1, 1), (700, 1, 3, 3), (129, 1, 2, 2), (2157, 1, 2, 2),
                                              (300, 4, 9, 9)])
def test_lookahead_matches_plain_order(zs, torch, monkeypatch, gemm, n, nrhs, nf, batch):
    """The next diagonal block ahead of the trailing update (ZSOLVE_LOOKAHEAD
    = 1; by default for up to 4 frequencies per lane) against the plain
    order (0): bit-identical sweeps, since every tile, block and pack is
    formed by the same arithmetic; and the oracle's solutions."""
    wl = workload.make_small(n, seed=300 + n, nf=nf, nrhs=nrhs, f_lo=0.5e9, f_hi=20e9)
    ref = oracle.solve_sweep(wl)
    out = {}
    for ahead in ("0", "1"):
        monkeypatch.setenv("ZSOLVE_LOOKAHEAD", ahead)
        s = zs.Solver(n, nrhs, gemm=getattr(zs, "ZSOLVE_GEMM_" + gemm), batch=batch)
        try:
            x = torch.empty((nf, nrhs, n), dtype=torch.complex128, device="cuda")
            infos = zs.zsolve_sweep(s.ctx, dev(torch, wl.L), dev(torch, wl.Psi), dev(torch, wl.G), wl.omega,
                                    wl.zs, dev(torch, wl.B), x)
            out[ahead] = x.cpu().numpy()
        finally:
            s.close()
        assert all(i.status == 0 and i.fallback == 0 for i in infos)
        for f in range(nf):
            assert np.all(rel_err(out[ahead][f], ref[f]) <= PARITY), (ahead, f)
    assert np.array_equal(out["0"], out["1"])


def test_symmetric_mode_with_a_nonsymmetric_input(zs, torch):
    # G made non-symmetric: the factors are those of the matrix the lower
    # triangle defines, but the float64 residual uses all of Z, so the
    # answer still meets the bar (by refinement or the fallback)
    wl = workload.make_small(260, seed=77, nf=3, nrhs=2, f_lo=0.5e9, f_hi=20e9)
    G = wl.G.copy()
    G[3, 200] += 0.3
    G[100, 7] -= 0.2
    wl2 = workload.Workload(wl.points, wl.L, wl.Psi, G, wl.freqs, wl.omega, wl.zs, wl.B, None)
    ref = oracle.solve_sweep(wl2)
    s = zs.Solver(wl.n, 2, batch=3, symmetric=1)
    try:
        x = torch.empty((3, 2, wl.n), dtype=torch.complex128, device="cuda")
        infos = zs.zsolve_sweep(s.ctx, dev(torch, wl.L), dev(torch, wl.Psi), dev(torch, G), wl.omega, wl.zs,
                                dev(torch, wl.B), x)
        X = x.cpu().numpy()
        for f in range(3):
            assert infos[f].status == 0
            assert np.all(rel_err(X[f], ref[f]) <= PARITY), (f, rel_err(X[f], ref[f]), infos[f].as_dict())
    finally:
        s.close()
