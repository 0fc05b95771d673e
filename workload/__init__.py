"""Seeded synthetic inputs for the frequency-sweep solver.

This module only *draws* inputs: the frequency-independent matrices L, Psi, G,
the frequency list, the surface impedance Zs(omega) a caller would supply, and
the right-hand sides.  It holds none of the solver's arithmetic (no assembly of
Z, no factorisation, no residual), so both the CPU oracle and the CUDA library
can be fed bit-identical data from it without sharing any method code.

Workloads follow the five synthetic configurations of the frequency-sweep
benchmark (malusrfworks.com, "Solving Dense Matrices Fast in the Browser",
section "Fewer frequency points", which states the form
Z(omega) = j*omega*L - j*Psi/omega + Zs(omega)*G with L, Psi, G independent of
frequency):

    id  N      kernel lengths (L / Psi)  frequencies (inclusive)  RHS
    0   256    0.1  / 0.05               5 over 1-5 GHz            1 x CN(0,1)
    1   2157   0.1  / 0.05               21 over 1-10 GHz          1 x CN(0,1)
    2   6614   0.1  / 0.05               41 over 0.5-20 GHz        2 x (e_p + CN(0,1e-3))
    3   8000   0.1  / 0.05               1 at 5 GHz                8 x CN(0,1)
    4   16384  0.05 / 0.025              11 over 1-20 GHz          4 x CN(0,1)

Recipe (all configurations): points x_i uniform in [0,1]^2; distances are
Euclidean; L_ij = exp(-|x_i-x_j|/len_L); Psi_ij = 200*exp(-|x_i-x_j|/len_Psi)
+ 50*delta_ij; G tridiagonal with 1.0 on the diagonal and 0.25 beside it;
omega = 2*pi*f; Zs(omega) = (1+j)*sqrt(omega*mu0/(2*sigma)) with
mu0 = 4*pi*1e-7 and sigma = 5.8e7 (copper skin-effect surface impedance).
The generator of configuration c is numpy.random.default_rng(c); it draws, in
this order, the points (N x 2), the port indices (configuration 2 only), the
real parts of B (nrhs x N), then the imaginary parts of B.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

MU0 = 4.0 * math.pi * 1e-7
SIGMA_CU = 5.8e7


@dataclasses.dataclass(frozen=True)
class Config:
    n: int
    len_l: float
    len_psi: float
    f_lo: float
    f_hi: float
    nf: int
    nrhs: int
    rhs: str  # "normal" or "port"
    name: str


CONFIGS = (
    Config(256, 0.1, 0.05, 1e9, 5e9, 5, 1, "normal", "N=256, 5 freq 1-5 GHz, 1 RHS"),
    Config(2157, 0.1, 0.05, 1e9, 10e9, 21, 1, "normal", "N=2157, 21 freq 1-10 GHz, 1 RHS"),
    Config(6614, 0.1, 0.05, 0.5e9, 20e9, 41, 2, "port", "N=6614, 41 freq 0.5-20 GHz, 2 port RHS"),
    Config(8000, 0.1, 0.05, 5e9, 5e9, 1, 8, "normal", "N=8000, 1 freq 5 GHz, 8 RHS"),
    Config(16384, 0.05, 0.025, 1e9, 20e9, 11, 4, "normal", "N=16384, 11 freq 1-20 GHz, 4 RHS"),
)


@dataclasses.dataclass
class Workload:
    """One generated problem: everything a caller hands to the solver."""

    points: np.ndarray  # (N, 2) float64
    L: np.ndarray  # (N, N) float64, symmetric
    Psi: np.ndarray  # (N, N) float64, symmetric
    G: np.ndarray  # (N, N) float64, symmetric
    freqs: np.ndarray  # (nf,) Hz
    omega: np.ndarray  # (nf,) rad/s
    zs: np.ndarray  # (nf,) complex128, surface impedance per frequency
    B: np.ndarray  # (nrhs, N) complex128, same for every frequency
    ports: np.ndarray | None  # (nrhs,) port indices for port excitations

    @property
    def n(self) -> int:
        return self.L.shape[0]


def surface_impedance(omega) -> np.ndarray:
    """Zs(omega) = (1+j) sqrt(omega mu0 / (2 sigma)) for copper."""
    omega = np.asarray(omega, dtype=np.float64)
    s = np.sqrt(omega * MU0 / (2.0 * SIGMA_CU))
    return s + 1j * s


def frequencies(cfg: Config) -> np.ndarray:
    """Evenly spaced frequencies with both endpoints included (Hz)."""
    if cfg.nf == 1:
        return np.array([cfg.f_lo], dtype=np.float64)
    return np.linspace(cfg.f_lo, cfg.f_hi, cfg.nf)


def distances(points: np.ndarray) -> np.ndarray:
    """Euclidean distance matrix; exactly symmetric with a zero diagonal."""
    dx = points[:, 0][:, None] - points[:, 0][None, :]
    dx *= dx
    dy = points[:, 1][:, None] - points[:, 1][None, :]
    dy *= dy
    dx += dy
    del dy
    return np.sqrt(dx, out=dx)


def kernel_matrices(points: np.ndarray, len_l: float, len_psi: float):
    """L, Psi and the tridiagonal G drawn from the point cloud."""
    n = points.shape[0]
    D = distances(points)
    L = np.exp(-D / len_l)
    Psi = 200.0 * np.exp(-D / len_psi)
    Psi[np.diag_indices(n)] += 50.0
    G = np.zeros((n, n))
    G[np.diag_indices(n)] = 1.0
    if n > 1:
        i = np.arange(n - 1)
        G[i, i + 1] = 0.25
        G[i + 1, i] = 0.25
    return L, Psi, G


def draw_points_and_rhs(cfg_id: int):
    """The random draws of configuration `cfg_id`: (points, ports, B)."""
    cfg = CONFIGS[cfg_id]
    rng = np.random.default_rng(cfg_id)
    points = rng.random((cfg.n, 2))
    ports = None
    if cfg.rhs == "port":
        ports = np.array([rng.integers(cfg.n) for _ in range(cfg.nrhs)], dtype=np.int64)
        scale = 1e-3
    else:
        scale = 1.0
    b_re = rng.normal(0.0, scale, (cfg.nrhs, cfg.n))
    b_im = rng.normal(0.0, scale, (cfg.nrhs, cfg.n))
    B = b_re + 1j * b_im
    if ports is not None:
        B[np.arange(cfg.nrhs), ports] += 1.0
    return points, ports, np.ascontiguousarray(B)


def make(cfg_id: int, nf: int | None = None) -> Workload:
    """Generate configuration `cfg_id` (seed = cfg_id).

    `nf` optionally keeps only the first nf frequencies (same matrices and
    right-hand sides), for bounded samples of a sweep.
    """
    cfg = CONFIGS[cfg_id]
    points, ports, B = draw_points_and_rhs(cfg_id)
    L, Psi, G = kernel_matrices(points, cfg.len_l, cfg.len_psi)
    freqs = frequencies(cfg)
    if nf is not None:
        freqs = freqs[:nf]
    omega = 2.0 * math.pi * freqs
    return Workload(points, L, Psi, G, freqs, omega, surface_impedance(omega), B, ports)


def make_small(n: int, seed: int, nf: int = 3, nrhs: int = 1, len_l: float = 0.1,
               len_psi: float = 0.05, f_lo: float = 1e9, f_hi: float = 5e9) -> Workload:
    """Same recipe at an arbitrary size, for tests that need ragged sizes."""
    rng = np.random.default_rng(seed)
    points = rng.random((n, 2))
    B = rng.normal(0.0, 1.0, (nrhs, n)) + 1j * rng.normal(0.0, 1.0, (nrhs, n))
    L, Psi, G = kernel_matrices(points, len_l, len_psi)
    freqs = np.linspace(f_lo, f_hi, nf) if nf > 1 else np.array([f_lo])
    omega = 2.0 * math.pi * freqs
    return Workload(points, L, Psi, G, freqs, omega, surface_impedance(omega),
                    np.ascontiguousarray(B), None)


def random_symmetric_real(n: int, seed: int, scale: float = 1.0) -> np.ndarray:
    """A dense real symmetric matrix with N(0, scale^2) entries."""
    rng = np.random.default_rng(seed)
    a = rng.normal(0.0, scale, (n, n))
    return np.triu(a) + np.triu(a, 1).T


def random_rhs(n: int, nrhs: int, seed: int) -> np.ndarray:
    """nrhs x n complex N(0,1) right-hand sides."""
    rng = np.random.default_rng(seed)
    return np.ascontiguousarray(rng.normal(size=(nrhs, n)) + 1j * rng.normal(size=(nrhs, n)))


# Resonant stand-in for the adaptive-frequency-sampling workloads.  The
# page's presets are circuit structures whose response changes character
# across the band (resonances); with the copper recipe above, j*omega*L
# dominates Z at every frequency and the solution is nearly one vector times
# 1/omega.  This variant keeps the point-cloud matrices and right-hand sides
# of a configuration, scales Psi so that the spectrum of L^-1 Psi overlaps
# omega^2 over the band, and uses a normalised angular frequency with a
# skin-effect-like loss Zs = zs_scale * (1+j) * sqrt(omega).
AFS_PSI_SCALE = 0.3
AFS_W_LO, AFS_W_HI = 1.0, 4.0
AFS_ZS_SCALE = 0.02


def afs_candidates(m: int, w_lo: float = AFS_W_LO, w_hi: float = AFS_W_HI, zs_scale: float = AFS_ZS_SCALE):
    """m evenly spaced normalised angular frequencies and their Zs."""
    omega = np.linspace(w_lo, w_hi, m) if m > 1 else np.array([w_lo], dtype=np.float64)[:m]
    s = zs_scale * np.sqrt(omega)
    return omega, s + 1j * s


def make_resonant(cfg_id: int, m: int, psi_scale: float = AFS_PSI_SCALE) -> Workload:
    """Configuration cfg_id's L, G, B with Psi * psi_scale over m candidates."""
    cfg = CONFIGS[cfg_id]
    points, ports, B = draw_points_and_rhs(cfg_id)
    L, Psi, G = kernel_matrices(points, cfg.len_l, cfg.len_psi)
    Psi *= psi_scale
    omega, zs = afs_candidates(m)
    return Workload(points, L, Psi, G, omega / (2.0 * math.pi), omega, zs, B, ports)


def make_resonant_small(n: int, seed: int, m: int, nrhs: int = 1, psi_scale: float = AFS_PSI_SCALE) -> Workload:
    """The resonant stand-in at an arbitrary size (recipe of make_small)."""
    wl = make_small(n, seed, nf=1, nrhs=nrhs)
    omega, zs = afs_candidates(m)
    return Workload(wl.points, wl.L, wl.Psi * psi_scale, wl.G, omega / (2.0 * math.pi), omega, zs, wl.B, None)


def make_growth(n: int, seed: int, eps: float = 3e-9, nf: int = 1, nrhs: int = 1,
                f_lo: float = 1e9, f_hi: float = 5e9) -> Workload:
    """A well-conditioned system on which the unpivoted low-precision LU fails.

    L is the identity with a tiny leading entry eps and a dense first row and
    column v (N(0, 1/n) entries); Psi and G are zero, so Z = j*omega*L.  The
    leading pivot is small (eps relative) but far above any tiny-pivot test;
    eliminating it adds entries of size |v|^2/eps to the trailing block, in
    whose float32 rounding the identity is lost.  Z itself stays well
    conditioned (2-norm condition about 3), so its double-precision solution is well
    defined, while the refinement on float32 factors stalls (relative
    corrections near 1).
    """
    rng = np.random.default_rng(seed)
    v = rng.normal(0.0, 1.0 / math.sqrt(n), n - 1)
    L = np.eye(n)
    L[0, 0] = eps
    L[0, 1:] = v
    L[1:, 0] = v
    B = rng.normal(0.0, 1.0, (nrhs, n)) + 1j * rng.normal(0.0, 1.0, (nrhs, n))
    freqs = np.linspace(f_lo, f_hi, nf) if nf > 1 else np.array([f_lo])
    omega = 2.0 * math.pi * freqs
    Z0 = np.zeros((n, n))
    return Workload(np.zeros((n, 2)), L, Z0, Z0.copy(), freqs, omega, surface_impedance(omega),
                    np.ascontiguousarray(B), None)
