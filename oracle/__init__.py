"""CPU oracle for the frequency-sweep solver -- TEST INFRASTRUCTURE ONLY.

Only `tests/`, `__graft_entry__.smoke()` and the CPU-baseline leg of
`bench.py` may import this package.  The CUDA library and its Python binding
never import it, link it or call it; the two share no code.  The only data
both sides see comes from the seeded generator in `workload`.

The oracle computes the plain definition of the method's answer: for each
frequency, Z(omega) = j*omega*L - j*Psi/omega + Zs(omega)*G assembled in
complex128 and x = Z^-1 b by an unblocked LU with partial pivoting plus
substitution (oracle.c states the steps and the passages they follow:
malusrfworks.com, "Solving Dense Matrices Fast in the Browser", section
"Fewer frequency points" for the form of Z, section "Double-precision answers
from a GPU without double precision" for the double-precision CPU direct solve
the refined answer must agree with, section "Measure first" for partial
pivoting as the robust CPU solve).

Every function here is pinned by `tests/test_oracle_pins.py` against
something other than itself (brute-force Cramer's rule, closed forms,
invariants, LAPACK through numpy).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "_oracle.so")
_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile oracle.c with gcc (OpenMP, no FMA contraction)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
               "-shared", "-std=c11", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            i64, dbl, ptr = ctypes.c_int64, ctypes.c_double, ctypes.c_void_p
            lib.orc_assemble.argtypes = [i64, ptr, ptr, ptr, dbl, dbl, dbl, ptr]
            lib.orc_assemble.restype = None
            lib.orc_lu_pp.argtypes = [i64, ptr, ptr]
            lib.orc_lu_pp.restype = ctypes.c_int
            lib.orc_lu_nopiv.argtypes = [i64, ptr]
            lib.orc_lu_nopiv.restype = ctypes.c_int
            lib.orc_lu_solve.argtypes = [i64, ptr, ptr, i64, ptr]
            lib.orc_lu_solve.restype = None
            lib.orc_inv_norm1_est.argtypes = [i64, ptr, ptr]
            lib.orc_inv_norm1_est.restype = dbl
            lib.orc_norm1.argtypes = [i64, ptr]
            lib.orc_norm1.restype = dbl
            lib.orc_residual.argtypes = [i64, ptr, i64, ptr, ptr, ptr]
            lib.orc_residual.restype = None
            lib.orc_num_threads.argtypes = []
            lib.orc_num_threads.restype = ctypes.c_int
            lib.orc_set_threads.argtypes = [ctypes.c_int]
            lib.orc_set_threads.restype = None
            _lib = lib
    return _lib


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64)


def _c128(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.complex128)


def num_threads() -> int:
    """OpenMP threads the oracle uses."""
    return _load().orc_num_threads()


def set_threads(t: int) -> None:
    _load().orc_set_threads(int(t))


def assemble(L, Psi, G, omega: float, zs: complex) -> np.ndarray:
    """Z(omega) in complex128, entry by entry as the formula is written."""
    L, Psi, G = _f64(L), _f64(Psi), _f64(G)
    n = L.shape[0]
    assert L.shape == Psi.shape == G.shape == (n, n)
    Z = np.empty((n, n), dtype=np.complex128)
    zs = complex(zs)
    _load().orc_assemble(n, _p(L), _p(Psi), _p(G), float(omega), zs.real, zs.imag, _p(Z))
    return Z


def lu_pp(Z):
    """LU with partial pivoting: returns (LU, piv, status); status 0 or k+1."""
    A = _c128(Z).copy()
    n = A.shape[0]
    piv = np.zeros(n, dtype=np.int64)
    st = _load().orc_lu_pp(n, _p(A), _p(piv))
    return A, piv, int(st)


def lu_nopiv(Z):
    """LU without row interchanges, complex128: returns (LU, status)."""
    A = _c128(Z).copy()
    st = _load().orc_lu_nopiv(A.shape[0], _p(A))
    return A, int(st)


def lu_solve(LU, piv, B) -> np.ndarray:
    """X with A X^T = B^T for B given as (nrhs, n) rows; piv may be None."""
    LU = _c128(LU)
    X = _c128(np.atleast_2d(B)).copy()
    n = LU.shape[0]
    pv = None if piv is None else np.ascontiguousarray(piv, dtype=np.int64)
    _load().orc_lu_solve(n, _p(LU), None if pv is None else _p(pv), X.shape[0], _p(X))
    return X


class SingularError(ValueError):
    pass


def solve(Z, B) -> np.ndarray:
    """x = Z^-1 b for each row b of B (nrhs, n)."""
    LU, piv, st = lu_pp(Z)
    if st:
        raise SingularError(f"exactly singular at column {st - 1}")
    return lu_solve(LU, piv, B)


def residual(Z, X, B) -> np.ndarray:
    """R = B - Z X row by row (nrhs, n), in double precision."""
    Z = _c128(Z)
    X = _c128(np.atleast_2d(X))
    B = _c128(np.atleast_2d(B))
    R = np.empty_like(B)
    _load().orc_residual(Z.shape[0], _p(Z), X.shape[0], _p(X), _p(B), _p(R))
    return R


def backward_error(Z, X, B) -> np.ndarray:
    """||b - Z x||_2 / ||b||_2 per right-hand side."""
    R = residual(Z, X, B)
    return np.linalg.norm(R, axis=1) / np.linalg.norm(np.atleast_2d(B), axis=1)


def norm1(Z) -> float:
    Z = _c128(Z)
    return float(_load().orc_norm1(Z.shape[0], _p(Z)))


def condest1(Z) -> float:
    """Estimate of the 1-norm condition number ||Z||_1 ||Z^-1||_1."""
    LU, piv, st = lu_pp(Z)
    if st:
        return float("inf")
    return norm1(Z) * float(_load().orc_inv_norm1_est(LU.shape[0], _p(LU), _p(piv)))


def cast_c64(Z) -> np.ndarray:
    """Round-to-nearest cast of complex128 to complex64 (the low-precision copy)."""
    return np.asarray(Z, dtype=np.complex128).astype(np.complex64)


def solve_sweep(wl, freq_idx=None) -> np.ndarray:
    """Direct solves of a generated workload: X[f, r, :] for each frequency."""
    idx = range(len(wl.omega)) if freq_idx is None else freq_idx
    out = []
    for f in idx:
        Z = assemble(wl.L, wl.Psi, wl.G, wl.omega[f], wl.zs[f])
        out.append(solve(Z, wl.B))
    return np.stack(out)
