"""ZSOLVE_GEMM_AUTO through the C-ABI: the arithmetic of the factorisation
(TF32, 3xTF32 or FFMA) picked by measured convergence and speed on the first
frequency of the first sweep, then used for the whole sweep.

- On an ordinary system every arithmetic converges; the choice must be the
  one with the smallest measured probe time, and every frequency must use it.
- On a well-conditioned system whose unpivoted factorisation grows entries by
  about 1/eps (eps = 3e-6), the float32-class arithmetics still converge but
  plain TF32 (a 10-bit significand in the products) does not: the probe must
  record the TF32 stall and the choice must be 3xTF32 or FFMA, after which
  the sweep converges without the fallback.
Every solution is held to the oracle's direct solve at the parity bound.
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
    return np.linalg.norm(np.atleast_2d(x) - np.atleast_2d(ref), axis=-1) / np.linalg.norm(np.atleast_2d(ref), axis=-1)


def run_auto(zs, torch, wl, **opts):
    nf, nrhs, n = len(wl.omega), wl.B.shape[0], wl.n
    s = zs.Solver(n, nrhs, gemm=zs.ZSOLVE_GEMM_AUTO, batch=nf, **opts)
    try:
        before = zs.zsolve_get_gemm_choice(s.ctx)
        assert before.done == 0 and before.chosen == zs.ZSOLVE_GEMM_TF32X3
        x = torch.empty((nf, nrhs, n), dtype=torch.complex128, device="cuda")
        infos = zs.zsolve_sweep(s.ctx, dev(torch, wl.L), dev(torch, wl.Psi), dev(torch, wl.G), wl.omega, wl.zs,
                                dev(torch, wl.B), x)
        probe = zs.zsolve_get_gemm_choice(s.ctx)
        # a second sweep keeps the choice (the probe runs once per context)
        infos2 = zs.zsolve_sweep(s.ctx, dev(torch, wl.L), dev(torch, wl.Psi), dev(torch, wl.G), wl.omega, wl.zs,
                                 dev(torch, wl.B), x)
        assert zs.zsolve_get_gemm_choice(s.ctx).chosen == probe.chosen
        return x.cpu().numpy(), infos, infos2, probe
    finally:
        s.close()


@pytest.mark.parametrize("n,nrhs,nf", [(300, 1, 3), (700, 2, 2)])
def test_auto_picks_the_fastest_converged_arithmetic(zs, torch, n, nrhs, nf):
    wl = workload.make_small(n, seed=900 + n, nf=nf, nrhs=nrhs)
    X, infos, infos2, probe = run_auto(zs, torch, wl)
    assert probe.done == 1
    conv = [k for k in range(3) if not probe.fallback[k]]
    assert conv, probe.as_dict()
    best = min(conv, key=lambda k: probe.ms[k])
    assert probe.chosen == best + 1, probe.as_dict()
    assert all(i.gemm == probe.chosen for i in list(infos) + list(infos2))
    ref = oracle.solve_sweep(wl)
    for f in range(nf):
        assert infos[f].fallback == 0
        assert np.all(rel_err(X[f], ref[f]) <= PARITY)


def test_auto_avoids_tf32_where_its_refinement_stalls(zs, torch):
    wl = workload.make_growth(300, seed=2, eps=3e-6, nf=2, nrhs=1)
    X, infos, _, probe = run_auto(zs, torch, wl)
    d = probe.as_dict()
    assert probe.done == 1 and probe.fallback[zs.ZSOLVE_GEMM_TF32 - 1] == 1, d
    assert probe.fallback[zs.ZSOLVE_GEMM_TF32X3 - 1] == 0 or probe.fallback[zs.ZSOLVE_GEMM_FFMA - 1] == 0, d
    assert probe.chosen in (zs.ZSOLVE_GEMM_TF32X3, zs.ZSOLVE_GEMM_FFMA), d
    ref = oracle.solve_sweep(wl)
    for f in range(2):
        assert infos[f].fallback == 0 and infos[f].gemm == probe.chosen, infos[f].as_dict()
        assert np.all(rel_err(X[f], ref[f]) <= PARITY)


def test_fixed_arithmetic_reports_itself(zs, torch):
    s = zs.Solver(64, 1, gemm=zs.ZSOLVE_GEMM_FFMA)
    try:
        p = zs.zsolve_get_gemm_choice(s.ctx)
        assert p.done == 0 and p.chosen == zs.ZSOLVE_GEMM_FFMA
    finally:
        s.close()
