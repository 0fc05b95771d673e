"""The allocation-free solve (zsolve_lowprec_solve_noalloc), through the
C-ABI, against the oracle's complex128 substitution with the same float32
factors and against the context-based solve (zsolve_lowprec_solve).

It is for callers that cannot allocate device memory where they solve (a
pool-managed application, a real-time loop, a plug-in whose host framework
owns device memory): its scratch is a static device array inside the
library.  This file is collected last so that a failure here cannot hide the
result of any other test; it passes alone in a fresh process too, because
the entry point sets its scratch up on its first call.
"""
import ctypes

import numpy as np
import pytest

import oracle
import workload

pytestmark = pytest.mark.gpu

# the context path applies the diagonal blocks through explicit inverses and
# the allocation-free one by substitution: both are float32 solves with the
# same factors, held to the tolerance the low-precision solve tests use (the
# oracle solves with those factors in complex128)
TOL = 1e-4


def _oracle_solve(fac_re, fac_im, B):
    """The oracle's unit-lower / upper substitution with the float32 factors."""
    LU = fac_re.astype(np.float64) + 1j * fac_im.astype(np.float64)
    return oracle.lu_solve(LU, None, oracle.cast_c64(B).astype(np.complex128))


def _factored(zs, torch, wl, f):
    s = zs.Solver(wl.n, wl.B.shape[0])
    zs.zsolve_assemble(s.ctx, torch.from_numpy(wl.L).cuda(), torch.from_numpy(wl.Psi).cuda(),
                       torch.from_numpy(wl.G).cuda(), wl.omega[f], wl.zs[f].real, wl.zs[f].imag)
    zs.zsolve_factor(s.ctx)
    return s


def _rel(a, b):
    return np.linalg.norm(a - b, axis=-1) / np.linalg.norm(b, axis=-1)


def test_noalloc_solve_matches_context_solve_on_two_calls():
    import torch

    import mixed_precision_refinement_gb300 as zs

    n, nrhs = 300, 3  # 3 right-hand sides: two launches (2 + 1) inside each call
    wl = workload.make_small(n, seed=77, nf=1, nrhs=nrhs)
    s = _factored(zs, torch, wl, 0)
    try:
        fac = torch.empty(2 * n * n, dtype=torch.float32, device="cuda")
        zs.zsolve_get_z32(s.ctx, fac[: n * n], fac[n * n:])
        b = torch.from_numpy(wl.B).cuda()
        ref = torch.empty_like(b)
        zs.zsolve_lowprec_solve(s.ctx, b, ref)
        ref = ref.cpu().numpy()
        F = fac.cpu().numpy()
        exact = _oracle_solve(F[: n * n].reshape(n, n), F[n * n:].reshape(n, n), wl.B)
        assert np.all(_rel(ref, exact) <= TOL)
        lib = zs.raw_lib()
        for _ in range(2):  # the second call finds the previous call's scratch contents
            v = b.to(torch.complex64).contiguous()
            st = lib.zsolve_lowprec_solve_noalloc(fac.data_ptr(), n, n * n, 2 * n * n, n, 1, v.data_ptr(),
                                                  nrhs * n, nrhs,
                                                  ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
            assert st == zs.ZSOLVE_OK, zs.zsolve_strerror(st)
            got = v.cpu().numpy().astype(np.complex128)
            assert np.all(_rel(got, exact) <= TOL)
            assert np.all(_rel(got, ref) <= TOL)
    finally:
        s.close()


def test_noalloc_solve_two_systems_and_limits():
    import torch

    import mixed_precision_refinement_gb300 as zs

    n, nrhs = 150, 1
    wl = workload.make_small(n, seed=78, nf=2, nrhs=nrhs)
    fac = torch.empty(2, 2 * n * n, dtype=torch.float32, device="cuda")
    refs = []
    b = torch.from_numpy(wl.B).cuda()
    for f in range(2):
        s = _factored(zs, torch, wl, f)
        try:
            zs.zsolve_get_z32(s.ctx, fac[f, : n * n], fac[f, n * n:])
            r = torch.empty_like(b)
            zs.zsolve_lowprec_solve(s.ctx, b, r)
            refs.append(r.cpu().numpy())
        finally:
            s.close()
    F = fac.cpu().numpy()
    exact = [_oracle_solve(F[f, : n * n].reshape(n, n), F[f, n * n:].reshape(n, n), wl.B) for f in range(2)]
    for _ in range(2):
        v = torch.stack([b, b]).to(torch.complex64).contiguous()
        zs.zsolve_lowprec_solve_noalloc(fac, n, n * n, 2 * n * n, n, 2, v, nrhs * n, nrhs)
        got = v.cpu().numpy().astype(np.complex128)
        for f in range(2):
            assert np.all(_rel(got[f], exact[f]) <= TOL)
            assert np.all(_rel(got[f], refs[f]) <= TOL)
    lib = zs.raw_lib()
    v = torch.zeros(65 * n, dtype=torch.complex64, device="cuda")
    assert lib.zsolve_lowprec_solve_noalloc(fac.data_ptr(), n, n * n, 2 * n * n, n, 65, v.data_ptr(), n, 1,
                                            None) == zs.ZSOLVE_EINVAL
