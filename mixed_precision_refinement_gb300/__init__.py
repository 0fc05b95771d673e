"""Python binding of the zsolve C-ABI (include/zsolve.h): argument marshalling only.

Every function below has the name of the C entry point it calls and does
nothing but turn tensors into pointers and status codes into exceptions; all
of the arithmetic runs in the CUDA kernels of libzsolve.so.  Device arrays
are torch CUDA tensors (float64 for L, Psi, G; complex128 for right-hand
sides and solutions), C-contiguous.  PyTorch supplies device memory and
streams only.

There is no CPU fallback: if the native library cannot be loaded, importing
this package raises.
"""
from __future__ import annotations

import ctypes
import os
import re

import numpy as np

from . import build as _build

ZSOLVE_OK = 0
ZSOLVE_EINVAL = -1
ZSOLVE_ENOMEM = -2
ZSOLVE_ECUDA = -3
ZSOLVE_ESTATE = -4
ZSOLVE_ENONFINITE = -5
ZSOLVE_ESINGULAR = -6
ZSOLVE_ETIMEOUT = -7

ZSOLVE_GEMM_AUTO = 0
ZSOLVE_GEMM_TF32 = 1
ZSOLVE_GEMM_TF32X3 = 2
ZSOLVE_GEMM_FFMA = 3

ZSOLVE_RESID_F64 = 0
ZSOLVE_RESID_DF = 1
ZSOLVE_RESID_FX = 2
ZSOLVE_RESID_LPG = 3
ZSOLVE_RESID_OZ = 4

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "zsolve.h")


class zsolve_opts(ctypes.Structure):
    _fields_ = [("tol", ctypes.c_double), ("max_iter", ctypes.c_int), ("gemm", ctypes.c_int),
                ("outer_block", ctypes.c_int), ("batch", ctypes.c_int), ("force_fallback", ctypes.c_int),
                ("profile", ctypes.c_int), ("resid", ctypes.c_int), ("lanes", ctypes.c_int),
                ("symmetric", ctypes.c_int), ("wait_limit", ctypes.c_int)]


STAGES = ("assemble", "diag", "trsm", "schur", "trsv", "residual", "update", "fallback", "pack")


class zsolve_profile(ctypes.Structure):
    _fields_ = [("launches", ctypes.c_int64 * len(STAGES)), ("ms", ctypes.c_double * len(STAGES))]

    def as_dict(self):
        return {st: {"launches": int(self.launches[i]), "ms": float(self.ms[i])} for i, st in enumerate(STAGES)}


class zsolve_info(ctypes.Structure):
    _fields_ = [("iters", ctypes.c_int), ("fallback", ctypes.c_int), ("status", ctypes.c_int),
                ("pivot_flag", ctypes.c_int), ("relcorr", ctypes.c_double), ("ms_assemble", ctypes.c_float),
                ("ms_factor", ctypes.c_float), ("ms_refine", ctypes.c_float), ("gemm", ctypes.c_int)]

    def as_dict(self):
        return {f: getattr(self, f) for f, _ in self._fields_}


class zsolve_gemm_probe(ctypes.Structure):
    _fields_ = [("done", ctypes.c_int), ("chosen", ctypes.c_int), ("ms", ctypes.c_float * 3),
                ("iters", ctypes.c_int * 3), ("fallback", ctypes.c_int * 3)]

    def as_dict(self):
        names = ("TF32", "TF32X3", "FFMA")
        return {"done": self.done, "chosen": {1: "TF32", 2: "TF32X3", 3: "FFMA"}.get(self.chosen, self.chosen),
                "probe": {nm: {"ms": float(self.ms[k]), "iters": int(self.iters[k]),
                               "fallback": int(self.fallback[k])} for k, nm in enumerate(names)}}


class zsolve_afs_opts(ctypes.Structure):
    _fields_ = [("tol", ctypes.c_double), ("max_solves", ctypes.c_int), ("max_basis", ctypes.c_int),
                ("drop", ctypes.c_double)]


class zsolve_afs_info(ctypes.Structure):
    _fields_ = [("n_exact", ctypes.c_int), ("q", ctypes.c_int), ("converged", ctypes.c_int),
                ("basis_full", ctypes.c_int), ("evals", ctypes.c_int), ("fallbacks", ctypes.c_int),
                ("max_resid", ctypes.c_double), ("eval_gflop", ctypes.c_double),
                ("ms_exact", ctypes.c_float), ("ms_basis", ctypes.c_float),
                ("ms_eval", ctypes.c_float), ("ms_expand", ctypes.c_float)]

    def as_dict(self):
        return {f: getattr(self, f) for f, _ in self._fields_}


ZSOLVE_AFS_MAX_BASIS = 96


class ZsolveError(RuntimeError):
    def __init__(self, status, message):
        super().__init__(f"zsolve status {status}: {message}")
        self.status = status


def _load():
    path = _build.build()
    lib = ctypes.CDLL(path)
    P, I, I64, D = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double
    sig = {
        "zsolve_default_opts": (I, [ctypes.POINTER(zsolve_opts)]),
        "zsolve_create": (I, [ctypes.POINTER(P), I64, I, ctypes.POINTER(zsolve_opts)]),
        "zsolve_set_stream": (I, [P, P]),
        "zsolve_assemble": (I, [P, P, P, P, D, D, D]),
        "zsolve_factor": (I, [P]),
        "zsolve_refine": (I, [P, P, P, I, ctypes.POINTER(zsolve_info)]),
        "zsolve_sweep": (I, [P, P, P, P, P, P, I, P, P, I, ctypes.POINTER(zsolve_info)]),
        "zsolve_sweep_host": (I, [P, P, P, P, P, P, I, P, P, I, ctypes.POINTER(zsolve_info)]),
        "zsolve_residual": (I, [P, P, P, P, I]),
        "zsolve_residual_lpg": (I, [P, P, P, P, P, P, P, I]),
        "zsolve_residual_oz": (I, [P, P, P, P, P, P, P, I]),
        "zsolve_lowprec_solve": (I, [P, P, P, I]),
        "zsolve_fallback_solve": (I, [P, P, P, I]),
        "zsolve_selftest_wait": (I, [P, I]),
        "zsolve_get_z64": (I, [P, P]),
        "zsolve_get_z32": (I, [P, P, P]),
        "zsolve_pivot_flag": (I, [P, ctypes.POINTER(I)]),
        "zsolve_lowprec_solve_noalloc": (I, [P, I64, I64, I64, I64, I, P, I64, I, P]),
        "zsolve_get_profile": (I, [P, ctypes.POINTER(zsolve_profile)]),
        "zsolve_get_resid_mode": (I, [P, ctypes.POINTER(I)]),
        "zsolve_get_gemm_choice": (I, [P, ctypes.POINTER(zsolve_gemm_probe)]),
        "zsolve_reset_profile": (I, [P]),
        "zsolve_strerror": (ctypes.c_char_p, [I]),
        "zsolve_last_error": (ctypes.c_char_p, [P]),
        "zsolve_destroy": (None, [P]),
        "zsolve_afs_default_opts": (I, [ctypes.POINTER(zsolve_afs_opts)]),
        "zsolve_afs_create": (I, [ctypes.POINTER(P), P, ctypes.POINTER(zsolve_afs_opts)]),
        "zsolve_afs_sweep": (I, [P, P, P, P, P, P, I, P, P, I, P, P, ctypes.POINTER(zsolve_afs_info)]),
        "zsolve_afs_launches": (I64, [P]),
        "zsolve_afs_last_error": (ctypes.c_char_p, [P]),
        "zsolve_afs_destroy": (None, [P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


try:
    _lib = _load()
except Exception as exc:  # no silent fallback: the package is unusable without the library
    raise ImportError(f"libzsolve.so could not be built or loaded: {exc}") from exc

LIB_PATH = _build.LIB


def declared_symbols() -> list[str]:
    """Names of the functions include/zsolve.h declares."""
    with open(HEADER) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(zsolve_[a-z0-9_]+)\s*\(", text)))


def _check(ctx, status):
    if status != ZSOLVE_OK:
        msg = _lib.zsolve_last_error(ctx).decode() if ctx else ""
        raise ZsolveError(status, f"{_lib.zsolve_strerror(status).decode()}: {msg}")


def _ptr(t) -> int:
    if t is None:
        return 0
    if hasattr(t, "data_ptr"):
        if not t.is_contiguous():
            raise ValueError("tensor must be contiguous")
        return t.data_ptr()
    if isinstance(t, np.ndarray):
        if not t.flags.c_contiguous:
            raise ValueError("array must be C-contiguous")
        return t.ctypes.data
    raise TypeError(f"expected a tensor or array, got {type(t)}")


def _require(t, dtype_name: str, cuda: bool):
    import torch
    want = {"f64": torch.float64, "c128": torch.complex128}[dtype_name]
    if t.dtype != want:
        raise TypeError(f"expected {want}, got {t.dtype}")
    if t.is_cuda != cuda:
        raise ValueError("expected a CUDA tensor" if cuda else "expected a CPU tensor")


# ---------------------------------------------------------------- C entry points


def zsolve_default_opts() -> zsolve_opts:
    o = zsolve_opts()
    _check(None, _lib.zsolve_default_opts(ctypes.byref(o)))
    return o


def zsolve_create(n: int, nrhs_max: int, opts: zsolve_opts | None = None) -> ctypes.c_void_p:
    ctx = ctypes.c_void_p()
    st = _lib.zsolve_create(ctypes.byref(ctx), int(n), int(nrhs_max), ctypes.byref(opts) if opts else None)
    _check(None, st)
    return ctx


def zsolve_set_stream(ctx, stream=None) -> None:
    """stream: a torch.cuda.Stream, a raw handle, or None for torch's current stream."""
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    _check(ctx, _lib.zsolve_set_stream(ctx, ctypes.c_void_p(handle)))


def zsolve_assemble(ctx, L, Psi, G, omega: float, zs_re: float, zs_im: float) -> None:
    for t in (L, Psi, G):
        _require(t, "f64", True)
    _check(ctx, _lib.zsolve_assemble(ctx, _ptr(L), _ptr(Psi), _ptr(G), float(omega), float(zs_re), float(zs_im)))


def zsolve_factor(ctx) -> None:
    _check(ctx, _lib.zsolve_factor(ctx))


def zsolve_refine(ctx, b, x) -> zsolve_info:
    _require(b, "c128", True)
    _require(x, "c128", True)
    nrhs = b.shape[0] if b.dim() == 2 else 1
    info = zsolve_info()
    _check(ctx, _lib.zsolve_refine(ctx, _ptr(b), _ptr(x), nrhs, ctypes.byref(info)))
    return info


def _sweep_args(omega, zs):
    om = np.ascontiguousarray(np.asarray(omega, dtype=np.float64).reshape(-1))
    z = np.asarray(zs, dtype=np.complex128).reshape(-1)
    if z.shape != om.shape:
        raise ValueError("omega and zs must have the same length")
    zz = np.ascontiguousarray(np.stack([z.real, z.imag], axis=1).reshape(-1))
    return om, zz


def zsolve_sweep(ctx, L, Psi, G, omega, zs, b, x) -> list:
    """x: complex128 CUDA tensor (nf, nrhs, n).  Returns the per-frequency infos."""
    for t in (L, Psi, G):
        _require(t, "f64", True)
    _require(b, "c128", True)
    _require(x, "c128", True)
    om, zz = _sweep_args(omega, zs)
    nf = om.shape[0]
    nrhs = b.shape[0] if b.dim() == 2 else 1
    infos = (zsolve_info * max(nf, 1))()
    _check(ctx, _lib.zsolve_sweep(ctx, _ptr(L), _ptr(Psi), _ptr(G), om.ctypes.data, zz.ctypes.data, nf, _ptr(b),
                                  _ptr(x), nrhs, infos))
    return list(infos)[:nf]


def zsolve_sweep_host(ctx, L, Psi, G, omega, zs, b, x) -> list:
    """Host-pointer sweep: L, Psi, G (float64), b, x (complex128) are CPU
    tensors or numpy arrays (pinned tensors give the fastest copies)."""
    om, zz = _sweep_args(omega, zs)
    nf = om.shape[0]
    nrhs = b.shape[0] if b.ndim == 2 else 1
    infos = (zsolve_info * max(nf, 1))()
    _check(ctx, _lib.zsolve_sweep_host(ctx, _ptr(L), _ptr(Psi), _ptr(G), om.ctypes.data, zz.ctypes.data, nf,
                                       _ptr(b), _ptr(x), nrhs, infos))
    return list(infos)[:nf]


def zsolve_residual(ctx, b, x, r) -> None:
    for t in (b, x, r):
        _require(t, "c128", True)
    nrhs = b.shape[0] if b.dim() == 2 else 1
    _check(ctx, _lib.zsolve_residual(ctx, _ptr(b), _ptr(x), _ptr(r), nrhs))


def zsolve_residual_lpg(ctx, L, Psi, G, b, x, r) -> None:
    for t in (L, Psi, G):
        _require(t, "f64", True)
    for t in (b, x, r):
        _require(t, "c128", True)
    nrhs = b.shape[0] if b.dim() == 2 else 1
    _check(ctx, _lib.zsolve_residual_lpg(ctx, _ptr(L), _ptr(Psi), _ptr(G), _ptr(b), _ptr(x), _ptr(r), nrhs))


def zsolve_residual_oz(ctx, L, Psi, G, b, x, r) -> None:
    for t in (L, Psi, G):
        _require(t, "f64", True)
    for t in (b, x, r):
        _require(t, "c128", True)
    nrhs = b.shape[0] if b.dim() == 2 else 1
    _check(ctx, _lib.zsolve_residual_oz(ctx, _ptr(L), _ptr(Psi), _ptr(G), _ptr(b), _ptr(x), _ptr(r), nrhs))


def zsolve_lowprec_solve(ctx, v, d) -> None:
    _require(v, "c128", True)
    _require(d, "c128", True)
    nrhs = v.shape[0] if v.dim() == 2 else 1
    _check(ctx, _lib.zsolve_lowprec_solve(ctx, _ptr(v), _ptr(d), nrhs))


def zsolve_fallback_solve(ctx, b, x) -> None:
    _require(b, "c128", True)
    _require(x, "c128", True)
    nrhs = b.shape[0] if b.dim() == 2 else 1
    _check(ctx, _lib.zsolve_fallback_solve(ctx, _ptr(b), _ptr(x), nrhs))


def zsolve_selftest_wait(ctx, nrhs: int = 1) -> int:
    """Status of the bounded-wait check (ZSOLVE_ETIMEOUT when the waits give up as they should)."""
    return int(_lib.zsolve_selftest_wait(ctx, int(nrhs)))


def zsolve_get_z64(ctx, dst) -> None:
    _require(dst, "c128", True)
    _check(ctx, _lib.zsolve_get_z64(ctx, _ptr(dst)))


def zsolve_get_z32(ctx, re, im) -> None:
    _check(ctx, _lib.zsolve_get_z32(ctx, _ptr(re), _ptr(im)))


def zsolve_pivot_flag(ctx) -> int:
    f = ctypes.c_int()
    _check(ctx, _lib.zsolve_pivot_flag(ctx, ctypes.byref(f)))
    return f.value


def zsolve_lowprec_solve_noalloc(z32, ld: int, plane: int, sys_stride: int, n: int, nsys: int, v,
                                 v_stride: int, nrhs: int, stream=None) -> None:
    """v (complex64 CUDA tensor) <- (L U)^-1 v with caller-held float32 factors, allocating nothing."""
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    if v.dtype != torch.complex64 or not v.is_cuda:
        raise TypeError("v must be a complex64 CUDA tensor")
    _check(None, _lib.zsolve_lowprec_solve_noalloc(_ptr(z32), ld, plane, sys_stride, n, nsys, _ptr(v), v_stride,
                                                   nrhs, ctypes.c_void_p(handle)))


def zsolve_get_profile(ctx) -> zsolve_profile:
    p = zsolve_profile()
    _check(ctx, _lib.zsolve_get_profile(ctx, ctypes.byref(p)))
    return p


def zsolve_get_gemm_choice(ctx) -> zsolve_gemm_probe:
    p = zsolve_gemm_probe()
    _check(ctx, _lib.zsolve_get_gemm_choice(ctx, ctypes.byref(p)))
    return p


def zsolve_get_resid_mode(ctx) -> int:
    m = ctypes.c_int()
    _check(ctx, _lib.zsolve_get_resid_mode(ctx, ctypes.byref(m)))
    return m.value


def zsolve_reset_profile(ctx) -> None:
    _check(ctx, _lib.zsolve_reset_profile(ctx))


def zsolve_strerror(status: int) -> str:
    return _lib.zsolve_strerror(int(status)).decode()


def zsolve_last_error(ctx) -> str:
    return _lib.zsolve_last_error(ctx).decode()


def zsolve_destroy(ctx) -> None:
    _lib.zsolve_destroy(ctx)


def zsolve_afs_default_opts() -> zsolve_afs_opts:
    o = zsolve_afs_opts()
    _check(None, _lib.zsolve_afs_default_opts(ctypes.byref(o)))
    return o


def _check_afs(afs, status):
    if status != ZSOLVE_OK:
        msg = _lib.zsolve_afs_last_error(afs).decode() if afs else ""
        raise ZsolveError(status, f"{_lib.zsolve_strerror(status).decode()}: {msg}")


def zsolve_afs_create(ctx, opts: zsolve_afs_opts | None = None) -> ctypes.c_void_p:
    afs = ctypes.c_void_p()
    st = _lib.zsolve_afs_create(ctypes.byref(afs), ctx, ctypes.byref(opts) if opts else None)
    _check(None, st)
    return afs


def zsolve_afs_sweep(afs, L, Psi, G, omega, zs, b, x=None):
    """x: complex128 CUDA tensor (m, nrhs, n) or None.  Returns (sampled
    candidate indices in solve order, final residual estimates (m,), info)."""
    for t in (L, Psi, G):
        _require(t, "f64", True)
    _require(b, "c128", True)
    if x is not None:
        _require(x, "c128", True)
    om, zz = _sweep_args(omega, zs)
    m = om.shape[0]
    nrhs = b.shape[0] if b.dim() == 2 else 1
    sampled = np.full(max(m, 1), -1, dtype=np.int32)
    resid = np.zeros(max(m, 1), dtype=np.float64)
    info = zsolve_afs_info()
    _check_afs(afs, _lib.zsolve_afs_sweep(afs, _ptr(L), _ptr(Psi), _ptr(G), om.ctypes.data, zz.ctypes.data, m,
                                          _ptr(b), _ptr(x), nrhs, sampled.ctypes.data, resid.ctypes.data,
                                          ctypes.byref(info)))
    return [int(k) for k in sampled[:info.n_exact]], resid[:m].copy(), info


def zsolve_afs_launches(afs) -> int:
    return int(_lib.zsolve_afs_launches(afs))


def zsolve_afs_last_error(afs) -> str:
    return _lib.zsolve_afs_last_error(afs).decode()


def zsolve_afs_destroy(afs) -> None:
    _lib.zsolve_afs_destroy(afs)


def make_afs_opts(**kw) -> zsolve_afs_opts:
    o = zsolve_afs_default_opts()
    for k, v in kw.items():
        if not hasattr(o, k):
            raise KeyError(k)
        setattr(o, k, v)
    return o


def raw_lib():
    """The ctypes handle of libzsolve.so (for calls with explicit status checks)."""
    return _lib


def make_opts(**kw) -> zsolve_opts:
    o = zsolve_default_opts()
    for k, v in kw.items():
        if not hasattr(o, k):
            raise KeyError(k)
        setattr(o, k, v)
    return o


class Solver:
    """Owns one context; methods forward to the entry points above."""

    def __init__(self, n: int, nrhs_max: int = 1, **opts):
        self.n = n
        self.ctx = zsolve_create(n, nrhs_max, make_opts(**opts))
        zsolve_set_stream(self.ctx)

    def close(self):
        if self.ctx:
            zsolve_destroy(self.ctx)
            self.ctx = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class Afs:
    """Owns one adaptive-frequency-sampling handle on a Solver's context.

    Example (device tensors L, Psi, G float64 n x n; b complex128 nrhs x n)::

        with Solver(n, nrhs, batch=2) as s, Afs(s, tol=1e-4) as a:
            x = torch.empty((m, nrhs, n), dtype=torch.complex128, device="cuda")
            sampled, resid, info = a.sweep(L, Psi, G, omega, zs, b, x)
            # x[i] is the reduced-order solution at omega[i]; `sampled` lists
            # the candidates solved in full, in order; info.converged is 1 if
            # every residual estimate is below tol
    """

    def __init__(self, solver: Solver, **opts):
        self.solver = solver
        self.afs = zsolve_afs_create(solver.ctx, make_afs_opts(**opts))

    def sweep(self, L, Psi, G, omega, zs, b, x=None):
        return zsolve_afs_sweep(self.afs, L, Psi, G, omega, zs, b, x)

    def close(self):
        if self.afs:
            zsolve_afs_destroy(self.afs)
            self.afs = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
