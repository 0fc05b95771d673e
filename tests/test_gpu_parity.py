"""Parity of the CUDA path (through the C-ABI) with the CPU oracle.

Every input comes from the seeded generator in `workload`; every expected
value comes from `oracle`.  Bars: the float64 assembly is bit-identical to
the oracle's (both round each operation of the formula separately and in the
same order) and its float32 copy is the round-to-nearest cast of it; the
solutions agree with the oracle's complex128 direct solve to <= 1e-10
relative l2 per (frequency, right-hand side).
"""
import math

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


def dev(torch, a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda()


def rel_err(x, ref):
    x = np.atleast_2d(x)
    ref = np.atleast_2d(ref)
    return np.linalg.norm(x - ref, axis=-1) / np.linalg.norm(ref, axis=-1)


def solve_single(zs, torch, wl, f, gemm, nrhs=None, **opts):
    B = wl.B if nrhs is None else wl.B[:nrhs]
    s = zs.Solver(wl.n, B.shape[0], gemm=gemm, **opts)
    try:
        L, P, G = dev(torch, wl.L), dev(torch, wl.Psi), dev(torch, wl.G)
        zs.zsolve_assemble(s.ctx, L, P, G, wl.omega[f], wl.zs[f].real, wl.zs[f].imag)
        zs.zsolve_factor(s.ctx)
        b = dev(torch, B)
        x = torch.empty_like(b)
        info = zs.zsolve_refine(s.ctx, b, x)
        torch.cuda.synchronize()
        return x.cpu().numpy(), info
    finally:
        s.close()


# ---------------------------------------------------------------- assembly (bit-exact)


@pytest.mark.parametrize("n", [1, 2, 33, 130, 256, 301])
def test_assemble_bit_exact(zs, torch, n):
    wl = workload.make_small(n, seed=n, nf=2)
    s = zs.Solver(n, 1)
    try:
        L, P, G = dev(torch, wl.L), dev(torch, wl.Psi), dev(torch, wl.G)
        for f in range(2):
            zs.zsolve_assemble(s.ctx, L, P, G, wl.omega[f], wl.zs[f].real, wl.zs[f].imag)
            z = torch.empty((n, n), dtype=torch.complex128, device="cuda")
            zs.zsolve_get_z64(s.ctx, z)
            ref = oracle.assemble(wl.L, wl.Psi, wl.G, wl.omega[f], wl.zs[f])
            got = z.cpu().numpy()
            assert np.array_equal(got.view(np.float64), ref.view(np.float64))
            re = torch.empty((n, n), dtype=torch.float32, device="cuda")
            im = torch.empty((n, n), dtype=torch.float32, device="cuda")
            zs.zsolve_get_z32(s.ctx, re, im)
            c64 = oracle.cast_c64(ref)
            assert np.array_equal(re.cpu().numpy(), c64.real) and np.array_equal(im.cpu().numpy(), c64.imag)
    finally:
        s.close()


def test_assemble_bit_exact_full_size_and_signed_zeros(zs, torch):
    # every entry of the N=2157 workload at three frequencies, then a matrix
    # built to hit every signed-zero case of the formula (L = -0, Psi = +-0,
    # G = +-0) with negative and positive Zs parts
    wl = workload.make(1)
    s = zs.Solver(wl.n, 1)
    try:
        L, P, G = dev(torch, wl.L), dev(torch, wl.Psi), dev(torch, wl.G)
        z = torch.empty((wl.n, wl.n), dtype=torch.complex128, device="cuda")
        for f in (0, 10, 20):
            zs.zsolve_assemble(s.ctx, L, P, G, wl.omega[f], wl.zs[f].real, wl.zs[f].imag)
            zs.zsolve_get_z64(s.ctx, z)
            ref = oracle.assemble(wl.L, wl.Psi, wl.G, wl.omega[f], wl.zs[f])
            assert np.array_equal(z.cpu().numpy().view(np.float64), ref.view(np.float64))
    finally:
        s.close()
    n = 64
    rng = np.random.default_rng(3)
    vals = np.array([0.0, -0.0, 0.25, 1.0, -0.5, 3.0])
    L = rng.choice(vals, size=(n, n))
    P = rng.choice(vals, size=(n, n))
    G = rng.choice(vals, size=(n, n))
    s = zs.Solver(n, 1)
    try:
        for zsv in (complex(-0.01, -0.02), complex(0.01, -0.02), complex(-0.01, 0.02), complex(0.0, 0.0)):
            w = 2 * math.pi * 1.3e9
            zs.zsolve_assemble(s.ctx, dev(torch, L), dev(torch, P), dev(torch, G), w, zsv.real, zsv.imag)
            z = torch.empty((n, n), dtype=torch.complex128, device="cuda")
            zs.zsolve_get_z64(s.ctx, z)
            ref = oracle.assemble(L, P, G, w, zsv)
            got = z.cpu().numpy()
            assert np.array_equal(got.view(np.int64), ref.view(np.int64))  # signs of zero included
            re = torch.empty((n, n), dtype=torch.float32, device="cuda")
            im = torch.empty_like(re)
            zs.zsolve_get_z32(s.ctx, re, im)
            c64 = oracle.cast_c64(ref)
            assert np.array_equal(re.cpu().numpy().view(np.int32), c64.real.copy().view(np.int32))
            assert np.array_equal(im.cpu().numpy().view(np.int32), c64.imag.copy().view(np.int32))
    finally:
        s.close()


def _ulp_distance32(a, b):
    """|a - b| in float32 ulps (ordered integer images of the bit patterns)."""
    def ordered(x):
        i = np.ascontiguousarray(x, dtype=np.float32).view(np.int32).astype(np.int64)
        return np.where(i < 0, -(i & 0x7FFFFFFF), i)
    return np.abs(ordered(a) - ordered(b))


@pytest.mark.parametrize("case", ["small", "full_size", "signed_zeros"])
def test_assemble32_within_one_ulp(zs, torch, monkeypatch, case):
    """The float32-only assembly (used by sweeps whose residual reads L, Psi,
    G) against RN32 of the oracle's float64 matrix: every entry within one
    float32 ulp, nearly all equal, zeros with the same sign.  ZSOLVE_ASM32=1
    (a testing aid) makes zsolve_assemble rewrite the float32 planes with it."""
    monkeypatch.setenv("ZSOLVE_ASM32", "1")
    if case == "signed_zeros":
        n = 64
        rng = np.random.default_rng(3)
        vals = np.array([0.0, -0.0, 0.25, 1.0, -0.5, 3.0])
        L, P, G = (rng.choice(vals, size=(n, n)) for _ in range(3))
        cases = [(L, P, G, 2 * math.pi * 1.3e9, zsv) for zsv in
                 (complex(-0.01, -0.02), complex(0.01, -0.02), complex(-0.01, 0.02), complex(0.0, 0.0))]
    else:
        wl = workload.make(1) if case == "full_size" else workload.make_small(301, seed=5, nf=3)
        n = wl.n
        cases = [(wl.L, wl.Psi, wl.G, wl.omega[f], wl.zs[f]) for f in (0, len(wl.omega) // 2, len(wl.omega) - 1)]
    s = zs.Solver(n, 1)
    try:
        re = torch.empty((n, n), dtype=torch.float32, device="cuda")
        im = torch.empty_like(re)
        for L, P, G, w, zsv in cases:
            zs.zsolve_assemble(s.ctx, dev(torch, L), dev(torch, P), dev(torch, G), w, zsv.real, zsv.imag)
            zs.zsolve_get_z32(s.ctx, re, im)
            c64 = oracle.cast_c64(oracle.assemble(L, P, G, w, zsv))
            for got, want in ((re.cpu().numpy(), c64.real), (im.cpu().numpy(), c64.imag)):
                d = _ulp_distance32(got, want)
                assert d.max() <= 1, d.max()
                assert np.count_nonzero(d) <= 1e-4 * d.size, np.count_nonzero(d)
                zero = want == 0
                assert np.array_equal(np.signbit(got[zero]), np.signbit(want[zero]))
    finally:
        s.close()


def test_assemble_term_isolation(zs, torch):
    # L = 0, G = 0, and a balanced scaling: each term of Z must appear exactly
    n = 70
    wl = workload.make_small(n, seed=5, nf=1)
    O = np.zeros((n, n))
    cases = [(O, wl.Psi, wl.G), (wl.L, wl.Psi, O), (wl.L * 1e-9, wl.Psi * 1e9, wl.G * 1e3), (O, O, wl.G)]
    s = zs.Solver(n, 1)
    try:
        for L, P, G in cases:
            zs.zsolve_assemble(s.ctx, dev(torch, L), dev(torch, P), dev(torch, G), wl.omega[0], wl.zs[0].real,
                               wl.zs[0].imag)
            z = torch.empty((n, n), dtype=torch.complex128, device="cuda")
            zs.zsolve_get_z64(s.ctx, z)
            ref = oracle.assemble(L, P, G, wl.omega[0], wl.zs[0])
            assert np.array_equal(z.cpu().numpy().view(np.float64), ref.view(np.float64))
    finally:
        s.close()


# ---------------------------------------------------------------- stages


@pytest.mark.parametrize("resid", ["F64", "FX"])
@pytest.mark.parametrize("n,nrhs", [(1, 1), (64, 2), (237, 1), (257, 3), (300, 8), (2157, 1), (1000, 7)])
def test_residual_against_oracle(zs, torch, n, nrhs, resid):
    wl = workload.make_small(n, seed=10 + n, nf=1, nrhs=nrhs)
    X = workload.random_rhs(n, nrhs, seed=3)
    s = zs.Solver(n, nrhs, resid=getattr(zs, "ZSOLVE_RESID_" + resid))
    try:
        zs.zsolve_assemble(s.ctx, dev(torch, wl.L), dev(torch, wl.Psi), dev(torch, wl.G), wl.omega[0],
                           wl.zs[0].real, wl.zs[0].imag)
        b, x = dev(torch, wl.B), dev(torch, X)
        r = torch.empty_like(b)
        zs.zsolve_residual(s.ctx, b, x, r)
        Z = oracle.assemble(wl.L, wl.Psi, wl.G, wl.omega[0], wl.zs[0])
        ref = oracle.residual(Z, X, wl.B)
        # different summation order: bounded by a few ulps of sum |z||x| per row
        scale = np.abs(X) @ np.abs(Z).T + np.abs(wl.B)
        assert np.all(np.abs(r.cpu().numpy() - ref) <= 4 * n * 2.3e-16 * scale + 1e-300)
    finally:
        s.close()


def _fx_case(kind, n, nrhs):
    """Inputs that stress the fixed-point residual: its per-lane scale, its
    real-part path, zeros, and x spread over many binades."""
    wl = workload.make_small(n, seed=600 + n, nf=1, nrhs=nrhs)
    L, Psi, G = wl.L, wl.Psi, wl.G
    X = workload.random_rhs(n, nrhs, seed=5)
    rng = np.random.default_rng(n)
    if kind == "dense_g":      # Re Z dense: every step takes the real-part products
        G = workload.random_symmetric_real(n, seed=n, scale=0.5)
    elif kind == "x_spread":   # x entries from 1e-30 to 1e30 (and exact zeros)
        X = X * 10.0 ** rng.uniform(-30, 30, size=X.shape)
        X[:, ::7] = 0.0
    elif kind == "z_spread":   # Z entries over 60 binades, some exactly zero
        f = 2.0 ** rng.integers(-30, 30, size=n)
        L = L * np.outer(f, f)
        Psi = np.zeros_like(Psi)
        L[3, :] = 0.0
        L[:, 3] = 0.0
        L[3, 3] = 1.0
    elif kind == "x_zero":     # one right-hand side exactly zero: r = b
        X[0] = 0.0
    return workload.Workload(wl.points, L, Psi, G, wl.freqs, wl.omega, wl.zs, wl.B, None), X


@pytest.mark.parametrize("kind", ["dense_g", "x_spread", "z_spread", "x_zero"])
@pytest.mark.parametrize("n,nrhs", [(33, 1), (300, 2), (1000, 4)])
def test_residual_fx_edge_cases(zs, torch, kind, n, nrhs):
    wl, X = _fx_case(kind, n, nrhs)
    s = zs.Solver(n, nrhs, resid=zs.ZSOLVE_RESID_FX)
    try:
        zs.zsolve_assemble(s.ctx, dev(torch, wl.L), dev(torch, wl.Psi), dev(torch, wl.G), wl.omega[0],
                           wl.zs[0].real, wl.zs[0].imag)
        b, x = dev(torch, wl.B), dev(torch, X)
        r = torch.empty_like(b)
        zs.zsolve_residual(s.ctx, b, x, r)
        Z = oracle.assemble(wl.L, wl.Psi, wl.G, wl.omega[0], wl.zs[0])
        ref = oracle.residual(Z, X, wl.B)
        R = r.cpu().numpy()
        # the float64 GEMV's own bound, row by row
        scale = np.abs(X) @ np.abs(Z).T + np.abs(wl.B)
        assert np.all(np.abs(R - ref) <= 4 * n * 2.3e-16 * scale + 1e-300)
        if kind == "x_zero":
            assert np.array_equal(R[0], wl.B[0])
    finally:
        s.close()


@pytest.mark.parametrize("n,nrhs", [(1, 1), (64, 2), (237, 1), (300, 3), (2157, 1)])
def test_residual_lpg_against_oracle(zs, torch, n, nrhs):
    # r = b - (j w L x - j Psi x / w + Zs G x) from L, Psi, G: each of the
    # three float64 sums is bounded by its own terms, so the bound is the
    # float64 GEMV's with |Z| replaced by w|L| + |Psi|/w + |Zs||G|
    wl = workload.make_small(n, seed=110 + n, nf=1, nrhs=nrhs)
    X = workload.random_rhs(n, nrhs, seed=6)
    s = zs.Solver(n, nrhs)
    try:
        L, P, G = dev(torch, wl.L), dev(torch, wl.Psi), dev(torch, wl.G)
        zs.zsolve_assemble(s.ctx, L, P, G, wl.omega[0], wl.zs[0].real, wl.zs[0].imag)
        b, x = dev(torch, wl.B), dev(torch, X)
        r = torch.empty_like(b)
        zs.zsolve_residual_lpg(s.ctx, L, P, G, b, x, r)
        Z = oracle.assemble(wl.L, wl.Psi, wl.G, wl.omega[0], wl.zs[0])
        ref = oracle.residual(Z, X, wl.B)
        w = wl.omega[0]
        terms = w * np.abs(wl.L) + np.abs(wl.Psi) / w + abs(wl.zs[0]) * np.abs(wl.G)
        scale = np.abs(X) @ terms.T + np.abs(wl.B)
        assert np.all(np.abs(r.cpu().numpy() - ref) <= 4 * (n + 4) * 2.3e-16 * scale + 1e-300)
    finally:
        s.close()


U64 = 2.0 ** -53


def _lpg_scale(wl, X):
    w = wl.omega[0]
    terms = w * np.abs(wl.L) + np.abs(wl.Psi) / w + abs(wl.zs[0]) * np.abs(wl.G)
    return np.abs(X) @ terms.T + np.abs(wl.B)


def _oz_bound(wl, X):
    """Error bound of the tensor-core residual (mode OZ), per entry of r:
    the float64 combination's, as for the L, Psi, G residual, plus the
    splitting's.  For one product sum Y_i = sum_j a_ij x_j (a row of L, Psi
    or G; the real or imaginary part of x) the 8 digits of 7 bits keep every
    entry to 2^-55 of its row's (column's) largest |entry|, and the digit
    products left out (levels k_a + k_x >= 8, at most 15 - l pairs of digits
    |d| <= 64 at weight 2^(7 (14 - l))) add at most 2^-51.2 max|a| max|x| per
    term: below 2^-49 n max_j|a_ij| max|x| in all.  A residual component
    combines w Y_L, Y_Psi / w and both parts of Zs Y_G."""
    n = wl.n
    w, z = wl.omega[0], abs(wl.zs[0])
    amax = w * np.abs(wl.L).max(axis=1) + np.abs(wl.Psi).max(axis=1) / w + 2 * z * np.abs(wl.G).max(axis=1)
    xmax = np.maximum(np.abs(X.real).max(axis=1), np.abs(X.imag).max(axis=1))
    return 4 * (n + 4) * 2.3e-16 * _lpg_scale(wl, X) + 2.0 ** -49 * n * np.outer(xmax, amax) + 1e-300


def _oz_residual(zs, torch, wl, X):
    n, nrhs = wl.n, X.shape[0]
    s = zs.Solver(n, nrhs)
    try:
        L, P, G = dev(torch, wl.L), dev(torch, wl.Psi), dev(torch, wl.G)
        zs.zsolve_assemble(s.ctx, L, P, G, wl.omega[0], wl.zs[0].real, wl.zs[0].imag)
        b, x = dev(torch, wl.B), dev(torch, X)
        r = torch.empty_like(b)
        zs.zsolve_residual_oz(s.ctx, L, P, G, b, x, r)
        return r.cpu().numpy()
    finally:
        s.close()


@pytest.mark.parametrize("n,nrhs", [(1, 1), (7, 1), (64, 2), (129, 1), (237, 3), (300, 16), (2157, 1), (1000, 5)])
def test_residual_oz_against_oracle(zs, torch, n, nrhs):
    wl = workload.make_small(n, seed=130 + n, nf=1, nrhs=nrhs)
    X = workload.random_rhs(n, nrhs, seed=8)
    R = _oz_residual(zs, torch, wl, X)
    Z = oracle.assemble(wl.L, wl.Psi, wl.G, wl.omega[0], wl.zs[0])
    ref = oracle.residual(Z, X, wl.B)
    err = np.abs(R - ref)
    assert np.all(err <= _oz_bound(wl, X)), (err / _oz_bound(wl, X)).max()
    # and in practice at the float64 level of the terms (a dropped digit
    # level or a wrong scale would show far above this)
    assert err.max() <= 64 * U64 * _lpg_scale(wl, X).max()


@pytest.mark.parametrize("kind", ["dense_g", "x_spread", "z_spread", "x_zero"])
@pytest.mark.parametrize("n,nrhs", [(33, 1), (300, 2), (1000, 4)])
def test_residual_oz_edge_cases(zs, torch, kind, n, nrhs):
    wl, X = _fx_case(kind, n, nrhs)
    R = _oz_residual(zs, torch, wl, X)
    Z = oracle.assemble(wl.L, wl.Psi, wl.G, wl.omega[0], wl.zs[0])
    ref = oracle.residual(Z, X, wl.B)
    assert np.all(np.abs(R - ref) <= _oz_bound(wl, X))
    if kind == "x_zero":
        assert np.array_equal(R[0], wl.B[0])


def test_residual_oz_non_finite(zs, torch):
    # a NaN in x (or an infinity in a row of L) gives NaN residuals there, so
    # that the refinement sees a non-finite correction and stops
    n, nrhs = 200, 2
    wl = workload.make_small(n, seed=7, nf=1, nrhs=nrhs)
    X = workload.random_rhs(n, nrhs, seed=9)
    X[0, 17] = complex(np.nan, 0.0)
    R = _oz_residual(zs, torch, wl, X)
    assert np.all(np.isnan(R[0]))
    assert np.all(np.isfinite(R[1]))
    L = wl.L.copy()
    L[5, 9] = np.inf
    wl2 = workload.Workload(wl.points, L, wl.Psi, wl.G, wl.freqs, wl.omega, wl.zs, wl.B, None)
    X[0, 17] = 1.0
    R = _oz_residual(zs, torch, wl2, X)
    assert np.all(np.isnan(R[:, 5])) and np.all(np.isfinite(np.delete(R, 5, axis=1)))


@pytest.mark.parametrize("resid", ["FX", "LPG", "OZ"])
@pytest.mark.parametrize("n,nrhs,nf", [(130, 2, 3), (700, 1, 3), (301, 4, 2), (1, 1, 2), (257, 1, 9)])
def test_sweep_parity_fixed_point_and_lpg_residual(zs, torch, n, nrhs, nf, resid):
    wl = workload.make_small(n, seed=85 + n, nf=nf, nrhs=nrhs, f_lo=0.5e9, f_hi=20e9)
    ref = oracle.solve_sweep(wl)
    s = zs.Solver(n, nrhs, resid=getattr(zs, "ZSOLVE_RESID_" + resid))
    try:
        x = torch.empty((nf, nrhs, n), dtype=torch.complex128, device="cuda")
        infos = zs.zsolve_sweep(s.ctx, dev(torch, wl.L), dev(torch, wl.Psi), dev(torch, wl.G), wl.omega, wl.zs,
                                dev(torch, wl.B), x)
        X = x.cpu().numpy()
        for f in range(nf):
            assert infos[f].status == 0 and infos[f].fallback == 0, infos[f].as_dict()
            assert np.all(rel_err(X[f], ref[f]) <= PARITY), (f, rel_err(X[f], ref[f]))
    finally:
        s.close()


@pytest.mark.parametrize("n,nrhs,nf,batch,lanes", [(300, 1, 20, 20, 1), (257, 4, 6, 6, 2), (130, 3, 12, 12, 3)])
def test_sweep_parity_oz_many_columns(zs, torch, n, nrhs, nf, batch, lanes):
    # more than 32 columns of x in one evaluation (several column groups),
    # several right-hand sides per slot, and three lanes
    wl = workload.make_small(n, seed=140 + n, nf=nf, nrhs=nrhs, f_lo=0.5e9, f_hi=20e9)
    ref = oracle.solve_sweep(wl)
    s = zs.Solver(n, nrhs, batch=batch, lanes=lanes, resid=zs.ZSOLVE_RESID_OZ)
    try:
        x = torch.empty((nf, nrhs, n), dtype=torch.complex128, device="cuda")
        infos = zs.zsolve_sweep(s.ctx, dev(torch, wl.L), dev(torch, wl.Psi), dev(torch, wl.G), wl.omega, wl.zs,
                                dev(torch, wl.B), x)
        X = x.cpu().numpy()
        for f in range(nf):
            assert infos[f].status == 0 and infos[f].fallback == 0, infos[f].as_dict()
            assert np.all(rel_err(X[f], ref[f]) <= PARITY), (f, rel_err(X[f], ref[f]))
    finally:
        s.close()


# backward error of the float32 factors, per trailing-update arithmetic
FACTOR_TOL = {"FFMA": 2e-6, "TF32X3": 2e-5, "TF32": 3e-3}


@pytest.mark.parametrize("n,nrhs", [(1, 1), (237, 1), (300, 3), (2157, 1), (513, 8)])
def test_residual_double_float_against_oracle(zs, torch, n, nrhs):
    wl = workload.make_small(n, seed=70 + n, nf=1, nrhs=nrhs)
    X = workload.random_rhs(n, nrhs, seed=4)
    s = zs.Solver(n, nrhs, resid=zs.ZSOLVE_RESID_DF)
    try:
        assert zs.zsolve_get_resid_mode(s.ctx) == zs.ZSOLVE_RESID_DF  # start-up self-test passed
        zs.zsolve_assemble(s.ctx, dev(torch, wl.L), dev(torch, wl.Psi), dev(torch, wl.G), wl.omega[0],
                           wl.zs[0].real, wl.zs[0].imag)
        b, x = dev(torch, wl.B), dev(torch, X)
        r = torch.empty_like(b)
        zs.zsolve_residual(s.ctx, b, x, r)
        Z = oracle.assemble(wl.L, wl.Psi, wl.G, wl.omega[0], wl.zs[0])
        ref = oracle.residual(Z, X, wl.B)
        # double-float: about 2^-46 per product, accumulated per lane
        scale = np.abs(X) @ np.abs(Z).T + np.abs(wl.B)
        assert np.all(np.abs(r.cpu().numpy() - ref) <= 1e-12 * scale + 1e-300)
    finally:
        s.close()


@pytest.mark.parametrize("n,nrhs,nf", [(130, 2, 3), (700, 1, 3), (301, 4, 2)])
def test_sweep_parity_double_float_residual(zs, torch, n, nrhs, nf):
    wl = workload.make_small(n, seed=80 + n, nf=nf, nrhs=nrhs, f_lo=0.5e9, f_hi=20e9)
    ref = oracle.solve_sweep(wl)
    s = zs.Solver(n, nrhs, resid=zs.ZSOLVE_RESID_DF)
    try:
        x = torch.empty((nf, nrhs, n), dtype=torch.complex128, device="cuda")
        infos = zs.zsolve_sweep(s.ctx, dev(torch, wl.L), dev(torch, wl.Psi), dev(torch, wl.G), wl.omega, wl.zs,
                                dev(torch, wl.B), x)
        X = x.cpu().numpy()
        for f in range(nf):
            assert infos[f].status == 0 and infos[f].fallback == 0, infos[f].as_dict()
            assert np.all(rel_err(X[f], ref[f]) <= PARITY), (f, rel_err(X[f], ref[f]))
    finally:
        s.close()


@pytest.mark.parametrize("gemm", ["FFMA", "TF32X3", "TF32"])
@pytest.mark.parametrize("n", [1, 31, 128, 129, 300, 513, 1000])
def test_factor_reconstructs_z32(zs, torch, n, gemm):
    wl = workload.make_small(n, seed=20 + n, nf=1)
    s = zs.Solver(n, 1, gemm=getattr(zs, "ZSOLVE_GEMM_" + gemm))
    try:
        zs.zsolve_assemble(s.ctx, dev(torch, wl.L), dev(torch, wl.Psi), dev(torch, wl.G), wl.omega[0],
                           wl.zs[0].real, wl.zs[0].imag)
        re = torch.empty((n, n), dtype=torch.float32, device="cuda")
        im = torch.empty_like(re)
        zs.zsolve_get_z32(s.ctx, re, im)
        Z32 = (re.cpu().numpy() + 1j * im.cpu().numpy()).astype(np.complex128)
        zs.zsolve_factor(s.ctx)
        assert zs.zsolve_pivot_flag(s.ctx) == 0
        zs.zsolve_get_z32(s.ctx, re, im)
        LU = re.cpu().numpy().astype(np.float64) + 1j * im.cpu().numpy()
        Lf = np.tril(LU, -1) + np.eye(n)
        Uf = np.triu(LU)
        err = np.linalg.norm(Lf @ Uf - Z32) / np.linalg.norm(Z32)
        assert err < FACTOR_TOL[gemm], err
        # and the factors are those of the unpivoted LU up to the arithmetic's rounding
        LUo, st = oracle.lu_nopiv(Z32)
        assert st == 0
        assert np.linalg.norm(LU - LUo) / np.linalg.norm(LUo) < (1e-3 if gemm != "TF32" else 0.3)
    finally:
        s.close()


@pytest.mark.parametrize("n,nrhs", [(1, 1), (65, 1), (200, 2), (300, 4), (129, 8), (150, 3)])
def test_lowprec_solve(zs, torch, n, nrhs):
    wl = workload.make_small(n, seed=30 + n, nf=1, nrhs=nrhs)
    s = zs.Solver(n, nrhs, gemm=zs.ZSOLVE_GEMM_FFMA)
    try:
        zs.zsolve_assemble(s.ctx, dev(torch, wl.L), dev(torch, wl.Psi), dev(torch, wl.G), wl.omega[0],
                           wl.zs[0].real, wl.zs[0].imag)
        zs.zsolve_factor(s.ctx)
        re = torch.empty((n, n), dtype=torch.float32, device="cuda")
        im = torch.empty_like(re)
        zs.zsolve_get_z32(s.ctx, re, im)
        LU = re.cpu().numpy().astype(np.float64) + 1j * im.cpu().numpy()
        v = dev(torch, wl.B)
        d = torch.empty_like(v)
        zs.zsolve_lowprec_solve(s.ctx, v, d)
        D = d.cpu().numpy()
        # the solve with the float32 factors: compare with the same factors in complex128
        ref = oracle.lu_solve(LU, None, oracle.cast_c64(wl.B).astype(np.complex128))
        assert np.all(rel_err(D, ref) < 1e-4)
    finally:
        s.close()


@pytest.mark.parametrize("n,nrhs,nf", [(300, 8, 1), (257, 4, 3), (400, 6, 2)])
def test_solve_chains_per_rhs_group(zs, torch, monkeypatch, n, nrhs, nf):
    """Right-hand sides solved as 1, 2 or 4 per chain (ZSOLVE_TRSV_R; unset:
    chosen per solve) give bit-identical sweeps: a right-hand side's sums are
    formed in the same order whatever its chain holds.  The sweep matches the
    oracle's direct solves."""
    wl = workload.make_small(n, seed=90 + n, nf=nf, nrhs=nrhs)
    ref = oracle.solve_sweep(wl)
    out = {}
    for r in ("", "1", "2", "4"):
        if r:
            monkeypatch.setenv("ZSOLVE_TRSV_R", r)
        else:
            monkeypatch.delenv("ZSOLVE_TRSV_R", raising=False)
        s = zs.Solver(n, nrhs, batch=nf)
        try:
            x = torch.empty((nf, nrhs, n), dtype=torch.complex128, device="cuda")
            infos = zs.zsolve_sweep(s.ctx, dev(torch, wl.L), dev(torch, wl.Psi), dev(torch, wl.G), wl.omega, wl.zs,
                                    dev(torch, wl.B), x)
            X = x.cpu().numpy()
        finally:
            s.close()
        assert all(i.status == 0 for i in infos)
        assert np.all(rel_err(X, ref) <= 1e-10), (r, rel_err(X, ref).max())
        out[r] = X
    for r in ("1", "2", "4"):
        assert np.array_equal(out[r], out[""]), r


# ---------------------------------------------------------------- end to end


@pytest.mark.parametrize("gemm", ["FFMA", "TF32X3"])
def test_refine_config0_every_frequency(zs, torch, gemm):
    wl = workload.make(0)
    ref = oracle.solve_sweep(wl)
    for f in range(len(wl.omega)):
        x, info = solve_single(zs, torch, wl, f, getattr(zs, "ZSOLVE_GEMM_" + gemm))
        assert info.fallback == 0 and 1 <= info.iters <= 10
        assert np.all(rel_err(x, ref[f]) <= PARITY), (f, rel_err(x, ref[f]), info.as_dict())


@pytest.mark.parametrize("gemm", ["FFMA", "TF32X3", "TF32"])
@pytest.mark.parametrize("n,nrhs,nf,batch", [(1, 1, 2, 0), (33, 2, 3, 2), (130, 3, 4, 3), (301, 4, 3, 0),
                                              (257, 8, 2, 1), (700, 1, 3, 3)])
def test_sweep_ragged_parity(zs, torch, n, nrhs, nf, batch, gemm):
    wl = workload.make_small(n, seed=40 + n, nf=nf, nrhs=nrhs, f_lo=0.5e9, f_hi=20e9)
    ref = oracle.solve_sweep(wl)
    s = zs.Solver(n, nrhs, gemm=getattr(zs, "ZSOLVE_GEMM_" + gemm), batch=batch)
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


@pytest.mark.parametrize("gemm", ["FFMA", "TF32X3"])
@pytest.mark.parametrize("n,nrhs,nf,batch", [(300, 2, 5, 5), (257, 1, 7, 4), (129, 3, 2, 0)])
def test_sweep_two_lanes_match_one_lane(zs, torch, n, nrhs, nf, batch, gemm):
    """A batch split over two or three concurrent lanes (streams and host
    threads) runs the same kernels on the same per-frequency data as one lane:
    the solutions agree bit for bit, and all match the oracle."""
    wl = workload.make_small(n, seed=70 + n, nf=nf, nrhs=nrhs, f_lo=0.5e9, f_hi=20e9)
    ref = oracle.solve_sweep(wl)
    out = {}
    for lanes in (1, 2, 3):
        s = zs.Solver(n, nrhs, gemm=getattr(zs, "ZSOLVE_GEMM_" + gemm), batch=batch, lanes=lanes)
        try:
            x = torch.empty((nf, nrhs, n), dtype=torch.complex128, device="cuda")
            infos = zs.zsolve_sweep(s.ctx, dev(torch, wl.L), dev(torch, wl.Psi), dev(torch, wl.G), wl.omega, wl.zs,
                                    dev(torch, wl.B), x)
            out[lanes] = (x.cpu().numpy(), [i.iters for i in infos])
            for f in range(nf):
                assert infos[f].status == 0 and infos[f].fallback == 0
                assert np.all(rel_err(out[lanes][0][f], ref[f]) <= PARITY)
        finally:
            s.close()
    assert out[1][1] == out[2][1] == out[3][1]
    assert np.array_equal(out[1][0], out[2][0]) and np.array_equal(out[1][0], out[3][0])


def test_sweep_term_isolation_parity(zs, torch):
    # the Psi/omega and Zs*G terms are tiny next to j*omega*L in the benchmark
    # configurations; solve systems where they dominate or vanish
    n = 150
    wl = workload.make_small(n, seed=7, nf=2)
    O = np.zeros((n, n))
    cases = [(wl.L * 1e-9, wl.Psi * 1e9, wl.G * 1e3), (wl.L, O, wl.G), (O, wl.Psi + 0 * wl.L, wl.G * 1e2)]
    s = zs.Solver(n, 1, gemm=zs.ZSOLVE_GEMM_FFMA)
    try:
        for L, P, G in cases:
            x = torch.empty((2, 1, n), dtype=torch.complex128, device="cuda")
            infos = zs.zsolve_sweep(s.ctx, dev(torch, L), dev(torch, P), dev(torch, G), wl.omega, wl.zs,
                                    dev(torch, wl.B), x)
            X = x.cpu().numpy()
            for f in range(2):
                Z = oracle.assemble(L, P, G, wl.omega[f], wl.zs[f])
                ref = oracle.solve(Z, wl.B)
                assert np.all(rel_err(X[f], ref) <= PARITY), (f, infos[f].as_dict())
    finally:
        s.close()


@pytest.mark.parametrize("resid", ["F64", "OZ"])
def test_sweep_host_matches_device(zs, torch, resid):
    # the host-pointer sweep copies L, Psi, G in row bands that the first
    # assembly (and the OZ residual's digits of L, Psi, G) follow band by band
    wl = workload.make_small(200, seed=50, nf=3, nrhs=2)
    s = zs.Solver(200, 2, gemm=zs.ZSOLVE_GEMM_FFMA, resid=getattr(zs, "ZSOLVE_RESID_" + resid))
    try:
        x = torch.empty((3, 2, 200), dtype=torch.complex128, device="cuda")
        zs.zsolve_sweep(s.ctx, dev(torch, wl.L), dev(torch, wl.Psi), dev(torch, wl.G), wl.omega, wl.zs,
                        dev(torch, wl.B), x)
        xh = np.zeros((3, 2, 200), dtype=np.complex128)
        zs.zsolve_sweep_host(s.ctx, wl.L, wl.Psi, wl.G, wl.omega, wl.zs, wl.B, xh)
        assert np.array_equal(xh, x.cpu().numpy())
    finally:
        s.close()


# ---------------------------------------------------------------- fallback


def test_fallback_solve_direct(zs, torch):
    wl = workload.make_small(160, seed=60, nf=1, nrhs=3)
    s = zs.Solver(160, 3)
    try:
        zs.zsolve_assemble(s.ctx, dev(torch, wl.L), dev(torch, wl.Psi), dev(torch, wl.G), wl.omega[0],
                           wl.zs[0].real, wl.zs[0].imag)
        b = dev(torch, wl.B)
        x = torch.empty_like(b)
        zs.zsolve_fallback_solve(s.ctx, b, x)
        ref = oracle.solve(oracle.assemble(wl.L, wl.Psi, wl.G, wl.omega[0], wl.zs[0]), wl.B)
        assert np.all(rel_err(x.cpu().numpy(), ref) <= 1e-12)
    finally:
        s.close()


@pytest.mark.parametrize("resid", ["F64", "OZ", "LPG"])
def test_forced_fallback_sweep(zs, torch, resid):
    # with OZ (four or more pairs per lane) and LPG the sweep assembles the
    # float32 planes alone: the fallback forms the float64 matrix itself
    wl = workload.make_small(97, seed=61, nf=2, nrhs=2)
    s = zs.Solver(97, 2, gemm=zs.ZSOLVE_GEMM_FFMA, force_fallback=1, resid=getattr(zs, "ZSOLVE_RESID_" + resid),
                  lanes=1)
    try:
        x = torch.empty((2, 2, 97), dtype=torch.complex128, device="cuda")
        infos = zs.zsolve_sweep(s.ctx, dev(torch, wl.L), dev(torch, wl.Psi), dev(torch, wl.G), wl.omega, wl.zs,
                                dev(torch, wl.B), x)
        ref = oracle.solve_sweep(wl)
        for f in range(2):
            assert infos[f].fallback == 1 and infos[f].status == 0
            assert np.all(rel_err(x.cpu().numpy()[f], ref[f]) <= 1e-12)
    finally:
        s.close()


def test_zero_pivot_triggers_fallback(zs, torch):
    # L = [[0,1],[1,0]] (+) I with Psi = G = 0: Z = j*omega*L has a zero leading
    # pivot, so the unpivoted factorisation flags it and the pivoted LU solves
    n = 40
    L = np.eye(n)
    L[:2, :2] = [[0.0, 1.0], [1.0, 0.0]]
    O = np.zeros((n, n))
    w = 2 * math.pi * 1e9
    B = workload.random_rhs(n, 1, seed=62)
    s = zs.Solver(n, 1, gemm=zs.ZSOLVE_GEMM_FFMA)
    try:
        zs.zsolve_assemble(s.ctx, dev(torch, L), dev(torch, O), dev(torch, O), w, 0.0, 0.0)
        zs.zsolve_factor(s.ctx)
        assert zs.zsolve_pivot_flag(s.ctx) == 1
        b = dev(torch, B)
        x = torch.empty_like(b)
        info = zs.zsolve_refine(s.ctx, b, x)
        assert info.fallback == 1 and info.pivot_flag == 1
        ref = oracle.solve(oracle.assemble(L, O, O, w, 0j), B)
        assert np.all(rel_err(x.cpu().numpy(), ref) <= 1e-13)
    finally:
        s.close()


def test_singular_reported(zs, torch):
    n = 8
    O = np.zeros((n, n))
    s = zs.Solver(n, 1, gemm=zs.ZSOLVE_GEMM_FFMA)
    try:
        zs.zsolve_assemble(s.ctx, dev(torch, O), dev(torch, O), dev(torch, O), 1e9, 0.0, 0.0)
        zs.zsolve_factor(s.ctx)
        b = dev(torch, workload.random_rhs(n, 1, seed=1))
        x = torch.empty_like(b)
        with pytest.raises(zs.ZsolveError) as e:
            zs.zsolve_refine(s.ctx, b, x)
        assert e.value.status == zs.ZSOLVE_ESINGULAR
    finally:
        s.close()


# ---------------------------------------------------------------- argument errors


def test_argument_errors(zs, torch):
    s = zs.Solver(16, 2)
    try:
        lib = zs.raw_lib()
        assert lib.zsolve_factor(s.ctx) == zs.ZSOLVE_ESTATE
        L = dev(torch, np.eye(16))
        assert lib.zsolve_assemble(s.ctx, L.data_ptr(), L.data_ptr(), L.data_ptr(), -1.0, 0.0, 0.0) == zs.ZSOLVE_EINVAL
        assert lib.zsolve_assemble(s.ctx, L.data_ptr(), L.data_ptr(), L.data_ptr(), 1e9, 0.0, 0.0) == 0
        b = torch.zeros((3, 16), dtype=torch.complex128, device="cuda")
        assert lib.zsolve_refine(s.ctx, b.data_ptr(), b.data_ptr(), 3, None) == zs.ZSOLVE_EINVAL
        assert lib.zsolve_refine(s.ctx, b.data_ptr(), b.data_ptr(), 1, None) == zs.ZSOLVE_ESTATE
        assert "before" in zs.zsolve_last_error(s.ctx)
    finally:
        s.close()


# ---------------------------------------------------------------- full size (the benchmark launch)


@pytest.mark.parametrize("gemm,resid", [("FFMA", "F64"), ("TF32X3", "F64"), ("TF32X3", "DF"), ("TF32X3", "FX"),
                                        ("TF32X3", "LPG"), ("TF32X3", "OZ")])
def test_config1_full_sweep_every_frequency(zs, torch, config1_oracle, gemm, resid):
    """N=2157, all 21 frequencies in one batched sweep (as the benchmark runs
    it): the oracle's direct solve at every frequency, element by element to
    the parity bound, and the oracle's double-precision backward error of
    every returned x."""
    wl, ref_all = config1_oracle
    nf = len(wl.omega)
    s = zs.Solver(wl.n, 1, batch=nf, gemm=getattr(zs, "ZSOLVE_GEMM_" + gemm), resid=getattr(zs, "ZSOLVE_RESID_" + resid))
    try:
        x = torch.empty((nf, 1, wl.n), dtype=torch.complex128, device="cuda")
        infos = zs.zsolve_sweep(s.ctx, dev(torch, wl.L), dev(torch, wl.Psi), dev(torch, wl.G), wl.omega, wl.zs,
                                dev(torch, wl.B), x)
        X = x.cpu().numpy()
        for f in range(nf):
            assert infos[f].status == 0 and infos[f].fallback == 0, infos[f].as_dict()
            Z = oracle.assemble(wl.L, wl.Psi, wl.G, wl.omega[f], wl.zs[f])
            # normwise backward error ||b - Z x|| / (||Z||_F ||x|| + ||b||) of a
            # double-precision-accurate solution
            R = oracle.residual(Z, X[f], wl.B)
            eta = np.linalg.norm(R, axis=1) / (np.linalg.norm(Z) * np.linalg.norm(X[f], axis=1)
                                               + np.linalg.norm(wl.B, axis=1))
            assert np.all(eta < 1e-15), (f, eta)
        errs = np.array([rel_err(X[f], ref_all[f]).max() for f in range(nf)])
        assert np.all(errs <= PARITY), errs
    finally:
        s.close()
