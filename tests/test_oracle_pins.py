"""Pins for the CPU oracle: each check ties it to something other than itself.

Brute force (Cramer's rule by permutation expansion, exact integer sums),
hand-worked fixtures under tests/golden/, closed forms (diagonal systems, the
surface impedance), structural invariants (Z^T = Z, unit-lower/upper
factors, backward error) and LAPACK through numpy.  A dropped term, a wrong
sign, a transposed operand or a swapped real/imaginary part in the oracle
fails at least one of them.
"""
import itertools
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
import workload

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


def _perm_sign(p):
    inv = sum(1 for i in range(len(p)) for j in range(i + 1, len(p)) if p[i] > p[j])
    return -1 if inv % 2 else 1


def _det_brute(M):
    n = len(M)
    total = 0
    for p in itertools.permutations(range(n)):
        term = _perm_sign(p)
        for i in range(n):
            term = term * M[i][p[i]]
        total += term
    return total


def _cramer(Z, b):
    n = len(b)
    d = _det_brute(Z)
    x = []
    for k in range(n):
        Mk = [[(b[i] if j == k else Z[i][j]) for j in range(n)] for i in range(n)]
        x.append(_det_brute(Mk) / d)
    return x


def _random_complex_symmetric(n, seed):
    rng = np.random.default_rng(seed)
    a = rng.normal(size=(n, n)) + 1j * rng.normal(size=(n, n))
    return np.triu(a) + np.triu(a, 1).T + n * np.eye(n) * (0.2 + 0.1j)


# ---------------------------------------------------------------- assembly


def test_assembly_golden_2x2():
    rows = {r[0]: r[1:] for r in _read_golden("assembly_2x2.txt") if r[0] != "Z"}
    zrows = [r for r in _read_golden("assembly_2x2.txt") if r[0] == "Z"]
    omega = float(rows["omega"][0])
    zs = complex(float(rows["zs"][0]), float(rows["zs"][1]))
    L = np.array([float(v) for v in rows["L"]]).reshape(2, 2)
    Psi = np.array([float(v) for v in rows["Psi"]]).reshape(2, 2)
    G = np.array([float(v) for v in rows["G"]]).reshape(2, 2)
    Z = oracle.assemble(L, Psi, G, omega, zs)
    for _, i, j, re, im in zrows:
        assert Z[int(i), int(j)] == complex(float(re), float(im))


def test_assembly_special_cases_exact():
    n = 7
    I = np.eye(n)
    O = np.zeros((n, n))
    w = 2 * math.pi * 3.3e9
    zs = 0.0123 + 0.0456j
    assert np.array_equal(oracle.assemble(I, O, O, w, zs), 1j * w * I)
    assert np.array_equal(oracle.assemble(O, O, I, w, zs), zs * I)
    Zp = oracle.assemble(O, I, O, w, zs)
    assert np.array_equal(Zp.real, O) and np.array_equal(Zp.imag, -I / w)


def test_assembly_acts_as_the_three_term_operator():
    # Z x computed from the assembled matrix must equal j w (L x) - j (Psi x)/w + Zs (G x)
    # computed by matrix products of the separate terms: a different route.
    wl = workload.make_small(40, seed=3, nf=2)
    rng = np.random.default_rng(9)
    x = rng.normal(size=40) + 1j * rng.normal(size=40)
    for w, zs in zip(wl.omega, wl.zs):
        Z = oracle.assemble(wl.L, wl.Psi, wl.G, w, zs)
        lhs = Z @ x
        rhs = 1j * w * (wl.L @ x) - 1j * (wl.Psi @ x) / w + zs * (wl.G @ x)
        scale = np.abs(Z) @ np.abs(x)
        assert np.max(np.abs(lhs - rhs) / scale) < 1e-14


def test_assembly_balanced_terms():
    # scale L down and Psi up so the three terms are comparable at GHz; the
    # per-term operator identity must still hold (guards against a term that
    # is too small to matter in the benchmark configurations)
    wl = workload.make_small(30, seed=4, nf=1)
    L = wl.L * 1e-9
    Psi = wl.Psi * 1e9
    G = wl.G * 1e3
    w, zs = wl.omega[0], wl.zs[0]
    Z = oracle.assemble(L, Psi, G, w, zs)
    t1, t2, t3 = np.abs(w * L).max(), np.abs(Psi / w).max(), np.abs(zs * G).max()
    assert max(t1, t2, t3) / min(t1, t2, t3) < 1e3
    x = np.ones(30) + 0.5j
    lhs = Z @ x
    rhs = 1j * w * (L @ x) - 1j * (Psi @ x) / w + zs * (G @ x)
    assert np.max(np.abs(lhs - rhs)) < 1e-13 * np.max(np.abs(Z) @ np.abs(x))


def test_assembly_symmetric_bitwise():
    wl = workload.make(0)
    for w, zs in zip(wl.omega, wl.zs):
        Z = oracle.assemble(wl.L, wl.Psi, wl.G, w, zs)
        assert np.array_equal(Z, Z.T)


# ---------------------------------------------------------------- solve


def test_solve_golden_2x2():
    g = {r[0]: complex(float(r[1]), float(r[2])) for r in _read_golden("cramer_2x2.txt")}
    Z = np.array([[g["Z00"], g["Z01"]], [g["Z01"], g["Z11"]]])
    b = np.array([[g["b0"], g["b1"]]])
    x = oracle.solve(Z, b)[0]
    expect = np.array([g["x0_num61"], g["x1_num61"]]) / 61.0
    assert np.max(np.abs(x - expect)) < 1e-15


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 6])
def test_solve_matches_cramer_bruteforce(n):
    Z = _random_complex_symmetric(n, seed=100 + n)
    rng = np.random.default_rng(n)
    b = rng.normal(size=n) + 1j * rng.normal(size=n)
    x_ref = np.array(_cramer(Z.tolist(), b.tolist()))
    x = oracle.solve(Z, b[None, :])[0]
    assert np.linalg.norm(x - x_ref) / np.linalg.norm(x_ref) < 1e-12


def test_solve_exact_rational_3x3():
    # integer complex-symmetric system; Cramer's rule in exact rationals
    Zi = [[(4, 1), (1, -2), (0, 3)], [(1, -2), (5, 0), (2, 1)], [(0, 3), (2, 1), (-3, 2)]]
    bi = [(1, 0), (0, 1), (2, -1)]

    def cplx(p):
        return (Fraction(p[0]), Fraction(p[1]))

    def cmul(a, b):
        return (a[0] * b[0] - a[1] * b[1], a[0] * b[1] + a[1] * b[0])

    def cadd(a, b):
        return (a[0] + b[0], a[1] + b[1])

    def det3(M):
        tot = (Fraction(0), Fraction(0))
        for p in itertools.permutations(range(3)):
            t = (Fraction(_perm_sign(p)), Fraction(0))
            for i in range(3):
                t = cmul(t, M[i][p[i]])
            tot = cadd(tot, t)
        return tot

    Z = [[cplx(v) for v in row] for row in Zi]
    b = [cplx(v) for v in bi]
    d = det3(Z)
    dd = d[0] * d[0] + d[1] * d[1]
    xs = []
    for k in range(3):
        Mk = [[(b[i] if j == k else Z[i][j]) for j in range(3)] for i in range(3)]
        nk = det3(Mk)
        q = cmul(nk, (d[0], -d[1]))
        xs.append(complex(q[0] / dd, q[1] / dd))
    Zn = np.array([[complex(*v) for v in row] for row in Zi])
    x = oracle.solve(Zn, np.array([[complex(*v) for v in bi]]))[0]
    assert np.max(np.abs(x - np.array(xs))) < 1e-15 * max(1.0, np.max(np.abs(xs)))


def test_solve_closed_form_diagonal():
    n = 64
    rng = np.random.default_rng(5)
    L = np.diag(rng.uniform(0.5, 2.0, n))
    Psi = np.diag(rng.uniform(50, 300, n))
    G = np.diag(rng.uniform(0.5, 1.5, n))
    b = rng.normal(size=n) + 1j * rng.normal(size=n)
    w = 2 * math.pi * 2.5e9
    zs = complex(workload.surface_impedance(w))
    Z = oracle.assemble(L, Psi, G, w, zs)
    x = oracle.solve(Z, b[None, :])[0]
    d = np.array([1j * w * L[i, i] - 1j * Psi[i, i] / w + zs * G[i, i] for i in range(n)])
    assert np.max(np.abs(x - b / d) / np.abs(b / d)) < 1e-15


def test_solve_needs_pivoting_zero_leading_pivot():
    n = 6
    Z = np.eye(n, dtype=np.complex128)
    Z[:2, :2] = [[0, 1], [1, 0]]
    b = np.arange(1, n + 1) + 0.5j
    x = oracle.solve(Z, b[None, :])[0]
    expect = b.copy()
    expect[0], expect[1] = b[1], b[0]
    assert np.array_equal(x, expect)
    _, st = oracle.lu_nopiv(Z)
    assert st == 1  # the unpivoted factorisation meets the zero pivot at step 0


def test_solve_pivot_choice_and_exact_singular():
    Z = np.array([[1, 2], [3, 4]], dtype=np.complex128)
    _, piv, st = oracle.lu_pp(Z)
    assert st == 0 and list(piv) == [1, 1]
    S = np.array([[1, 2], [2, 4]], dtype=np.complex128)
    _, _, st = oracle.lu_pp(S)
    assert st == 2
    with pytest.raises(oracle.SingularError):
        oracle.solve(S, np.ones((1, 2)))


def test_solve_matches_lapack_and_backward_error_config0():
    wl = workload.make(0)
    for w, zs in zip(wl.omega, wl.zs):
        Z = oracle.assemble(wl.L, wl.Psi, wl.G, w, zs)
        X = oracle.solve(Z, wl.B)
        X_np = np.linalg.solve(Z, wl.B.T).T
        cond = np.linalg.cond(Z)
        rel = np.linalg.norm(X - X_np) / np.linalg.norm(X_np)
        assert rel < cond * 1e-15
        assert np.all(oracle.backward_error(Z, X, wl.B) < 1e-13)


def test_solve_backward_error_ragged_multi_rhs():
    wl = workload.make_small(301, seed=11, nf=2, nrhs=3)
    for w, zs in zip(wl.omega, wl.zs):
        Z = oracle.assemble(wl.L, wl.Psi, wl.G, w, zs)
        X = oracle.solve(Z, wl.B)
        assert X.shape == (3, 301)
        assert np.all(oracle.backward_error(Z, X, wl.B) < 1e-13)


# ---------------------------------------------------------------- factors


def test_lu_nopiv_reconstructs_and_matches_pivoted_when_no_swaps():
    n = 48
    Z = _random_complex_symmetric(n, seed=7) + 40 * np.eye(n)  # strongly diagonally dominant
    LUn, st = oracle.lu_nopiv(Z)
    assert st == 0
    Lf = np.tril(LUn, -1) + np.eye(n)
    Uf = np.triu(LUn)
    assert np.linalg.norm(Lf @ Uf - Z) / np.linalg.norm(Z) < 1e-14
    LUp, piv, st = oracle.lu_pp(Z)
    assert st == 0 and np.array_equal(piv, np.arange(n))
    assert np.array_equal(LUp, LUn)


def test_lu_pp_reconstructs_with_permutation():
    n = 50
    rng = np.random.default_rng(8)
    Z = rng.normal(size=(n, n)) + 1j * rng.normal(size=(n, n))
    LU, piv, st = oracle.lu_pp(Z)
    assert st == 0
    P = np.eye(n)
    for k, p in enumerate(piv):
        P[[k, p]] = P[[p, k]]
    Lf = np.tril(LU, -1) + np.eye(n)
    Uf = np.triu(LU)
    assert np.linalg.norm(Lf @ Uf - P @ Z) / np.linalg.norm(Z) < 1e-14
    # the pivot maximises |Re|+|Im| in its column, so every multiplier has
    # modulus at most sqrt(2), and the pivot row's own multiplier is 1
    assert np.all(np.abs(np.tril(LU, -1)) <= math.sqrt(2) * (1 + 1e-15))


# ---------------------------------------------------------------- residual / norms


def test_residual_exact_on_integers():
    rng = np.random.default_rng(12)
    n, nrhs = 23, 2
    Zi = rng.integers(-9, 10, size=(n, n)) + 1j * rng.integers(-9, 10, size=(n, n))
    Xi = rng.integers(-9, 10, size=(nrhs, n)) + 1j * rng.integers(-9, 10, size=(nrhs, n))
    Bi = rng.integers(-99, 100, size=(nrhs, n)) + 1j * rng.integers(-99, 100, size=(nrhs, n))
    R = oracle.residual(Zi, Xi, Bi)
    for r in range(nrhs):
        for i in range(n):
            s = sum(complex(Zi[i, j]) * complex(Xi[r, j]) for j in range(n))
            exact = complex(Bi[r, i]) - s
            assert R[r, i] == exact


def test_residual_vs_matmul_rounding():
    wl = workload.make_small(120, seed=13, nf=1, nrhs=2)
    Z = oracle.assemble(wl.L, wl.Psi, wl.G, wl.omega[0], wl.zs[0])
    X = workload.random_rhs(120, 2, seed=14)
    R = oracle.residual(Z, X, wl.B)
    R_np = wl.B - X @ Z.T
    scale = (np.abs(X) @ np.abs(Z).T).max()
    assert np.max(np.abs(R - R_np)) < 1e-14 * scale


def test_condest_against_exact_one_norm_condition():
    for seed in range(3):
        wl = workload.make_small(60, seed=20 + seed, nf=1)
        Z = oracle.assemble(wl.L, wl.Psi, wl.G, wl.omega[0], wl.zs[0])
        exact = np.linalg.cond(Z, 1)
        est = oracle.condest1(Z)
        assert exact / 3 <= est <= exact * (1 + 1e-8)
    assert oracle.norm1(np.array([[1 + 1j, 2], [3j, -4]])) == pytest.approx(max(math.sqrt(2) + 3, 6))


# ---------------------------------------------------------------- generator


def test_surface_impedance_closed_form():
    for f, val in _read_golden("surface_impedance.txt"):
        zs = complex(workload.surface_impedance(2 * math.pi * float(f)))
        assert zs.real == zs.imag
        assert abs(zs.real - float(val)) < 5e-7 * float(val)


def test_generator_shapes_and_structure():
    wl = workload.make(0)
    assert wl.L.shape == (256, 256) and wl.B.shape == (1, 256)
    assert np.allclose(wl.freqs, [1e9, 2e9, 3e9, 4e9, 5e9], rtol=0, atol=0)
    assert np.array_equal(wl.L, wl.L.T) and np.array_equal(wl.Psi, wl.Psi.T)
    assert np.all(np.diag(wl.L) == 1.0) and np.all(np.diag(wl.Psi) == 250.0)
    assert np.count_nonzero(wl.G) == 256 + 2 * 255
    assert np.min(np.linalg.eigvalsh(wl.L)) > 0  # SPD
    wl1 = workload.make(1, nf=2)
    assert wl1.L.shape == (2157, 2157) and wl1.freqs[1] == pytest.approx(1.45e9)


def test_generator_port_excitation():
    points, ports, B = workload.draw_points_and_rhs(2)
    assert points.shape == (6614, 2) and B.shape == (2, 6614) and len(ports) == 2
    for r, p in enumerate(ports):
        assert abs(B[r, p] - 1.0) < 1e-2
        rest = np.delete(B[r], p)
        assert 0.5e-3 < np.std(rest.real) < 2e-3 and 0.5e-3 < np.std(rest.imag) < 2e-3
    _, _, B0 = workload.draw_points_and_rhs(0)
    assert np.array_equal(B0, workload.make(0).B)


def test_unpivoted_lu_of_complex_symmetric_is_ldlt():
    # the symmetric factorisation mode rests on two facts: for Z = Z^T the
    # unpivoted LU has U = D L^T with D = diag(U), and the Schur complement
    # left after eliminating a leading block is symmetric again, so its lower
    # part determines it
    wl = workload.make_small(70, seed=5, nf=1)
    Z = oracle.assemble(wl.L, wl.Psi, wl.G, wl.omega[0], wl.zs[0])
    LU, st = oracle.lu_nopiv(Z)
    assert st == 0
    L = np.tril(LU, -1) + np.eye(70)
    U = np.triu(LU)
    D = np.diag(U)
    assert np.abs(U - D[:, None] * L.T).max() <= 1e-12 * np.abs(U).max()
    k = 32
    S = Z[k:, k:] - Z[k:, :k] @ np.linalg.solve(Z[:k, :k], Z[:k, k:])
    assert np.abs(S - S.T).max() <= 1e-12 * np.abs(S).max()
