"""Failure detection and routing, made on the host or by inputs, never by a
GPU fault: through the C-ABI.

- A bounded device-side wait that cannot be satisfied gives up: the
  triangular solve is run with its first task withheld (every other task
  waits, directly or through the chain, for that block) and a short wait
  limit; the call returns ZSOLVE_ETIMEOUT and the same context then solves
  normally.
- A natural stall: a well-conditioned Z (2-norm condition about 3) whose unpivoted
  float32 factorisation loses the trailing block in rounding (a tiny leading
  pivot, eps = 3e-9 relative, far above the tiny-pivot test).  The refinement
  neither converges nor flags a pivot; its relative corrections stay near 1,
  so it stalls by growth or after max_iter corrections and the frequency is
  solved by the float64 pivoted LU (the page's section "Double-precision
  answers from a GPU without double precision", the paragraph after the
  steps: a refinement that does not converge switches to a direct solve).
  The answer must then agree with the oracle's direct solve to the parity
  bound, as any other frequency's.
"""
import numpy as np
import pytest

import oracle
import workload

pytestmark = pytest.mark.gpu

PARITY = 1e-10


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
    x = np.atleast_2d(x)
    ref = np.atleast_2d(ref)
    return np.linalg.norm(x - ref, axis=-1) / np.linalg.norm(ref, axis=-1)


@pytest.mark.parametrize("n,nrhs", [(100, 1), (300, 2), (700, 4)])
def test_bounded_wait_gives_up_and_context_stays_usable(zs, torch, n, nrhs):
    wl = workload.make_small(n, seed=500 + n, nf=1, nrhs=nrhs)
    s = zs.Solver(n, nrhs, wait_limit=2048)
    try:
        zs.zsolve_assemble(s.ctx, dev(torch, wl.L), dev(torch, wl.Psi), dev(torch, wl.G), wl.omega[0],
                           wl.zs[0].real, wl.zs[0].imag)
        zs.zsolve_factor(s.ctx)
        assert zs.zsolve_selftest_wait(s.ctx, nrhs) == zs.ZSOLVE_ETIMEOUT
        assert "gave up" in zs.zsolve_last_error(s.ctx)
        # the same context afterwards: a low-precision solve against the
        # oracle's substitution with the same float32 factors, then a
        # refinement against the oracle's direct solve
        re = torch.empty((n, n), dtype=torch.float32, device="cuda")
        im = torch.empty_like(re)
        zs.zsolve_get_z32(s.ctx, re, im)
        LU = re.cpu().numpy().astype(np.float64) + 1j * im.cpu().numpy()
        b = dev(torch, wl.B)
        d = torch.empty_like(b)
        zs.zsolve_lowprec_solve(s.ctx, b, d)
        ref = oracle.lu_solve(LU, None, oracle.cast_c64(wl.B).astype(np.complex128))
        assert np.all(rel_err(d.cpu().numpy(), ref) < 1e-4)
        x = torch.empty_like(b)
        info = zs.zsolve_refine(s.ctx, b, x)
        Z = oracle.assemble(wl.L, wl.Psi, wl.G, wl.omega[0], wl.zs[0])
        assert info.fallback == 0
        assert np.all(rel_err(x.cpu().numpy(), oracle.solve(Z, wl.B)) <= PARITY)
    finally:
        s.close()


@pytest.mark.parametrize("resid", ["F64", "OZ", "LPG"])
@pytest.mark.parametrize("gemm", ["FFMA", "TF32X3", "TF32"])
@pytest.mark.parametrize("n,nrhs,nf", [(130, 1, 1), (300, 2, 3)])
def test_natural_stall_reaches_fallback(zs, torch, gemm, n, nrhs, nf, resid):
    # OZ and LPG: a lane whose residual reads L, Psi, G assembles the float32
    # planes alone (OZ: four or more pairs; with 3 frequencies x 2 right-hand
    # sides the lanes hold 4 and 2), so the fallback forms the float64 matrix
    wl = workload.make_growth(n, seed=n, nf=nf, nrhs=nrhs)
    ref = oracle.solve_sweep(wl)
    s = zs.Solver(n, nrhs, gemm=getattr(zs, "ZSOLVE_GEMM_" + gemm), batch=nf,
                  resid=getattr(zs, "ZSOLVE_RESID_" + resid))
    try:
        x = torch.empty((nf, nrhs, n), dtype=torch.complex128, device="cuda")
        infos = zs.zsolve_sweep(s.ctx, dev(torch, wl.L), dev(torch, wl.Psi), dev(torch, wl.G), wl.omega, wl.zs,
                                dev(torch, wl.B), x)
        X = x.cpu().numpy()
        for f in range(nf):
            i = infos[f]
            assert i.status == 0 and i.fallback == 1, i.as_dict()
            if gemm == "TF32" and i.pivot_flag:
                # with 10-bit products the trailing matrix I - v v^T / eps loses
                # its identity part entirely and can cancel to an exactly zero
                # pivot, which the pivot test catches before any correction
                assert i.iters == 0, i.as_dict()
            else:
                # no pivot was flagged: the refinement itself gave up
                assert i.pivot_flag == 0 and 1 <= i.iters <= 10, i.as_dict()
            assert np.all(rel_err(X[f], ref[f]) <= PARITY), (f, rel_err(X[f], ref[f]))
        if gemm != "TF32":
            assert all(i.pivot_flag == 0 for i in infos)
    finally:
        s.close()
