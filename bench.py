"""Benchmark: solved frequency points per second of the mixed-precision sweep.

One step = one zsolve_sweep over the whole frequency list of the workload
(assembly, low-precision factorisation, refinement, any fallback) with the
inputs already resident in HBM.  The default workload is the N=2157,
21-frequency (1-10 GHz), 1-RHS sweep; --config picks another of the five
synthetic workloads in `workload`.  Inputs are synthetic (seeded generator).

Prints ONE JSON line on rank 0.  Under torchrun each rank solves the same
sweep on its own GPU (weak scaling, no collective on the data path); the
barrier-bracketed time is the max over ranks.

--impl reference times the CPU oracle (complex128 pivoted LU) on bounded
samples of the same workload instead.
"""
from __future__ import annotations

import argparse
import atexit
import dataclasses
import datetime
import json
import re
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workload  # noqa: E402

METRIC = "solved freq points/s at N=2157; LU TFLOP/s; FP64 residual GEMV HBM GB/s"
RESID_NAMES = {0: "F64", 1: "DF", 2: "FX", 3: "LPG", 4: "OZ"}
RESID_ARITH = {
    "F64": "float64 DFMA GEMV over the assembled Z",
    "DF": "double-float (2 x float32, ~46 bits)",
    "FX": "exact 72-bit fixed-point products and sums on the integer pipes, float64-accurate",
    "LPG": "float64 DFMA from L, Psi, G, four frequencies per pass (no assembled Z read)",
    "OZ": "L x, Psi x, G x of a lane's frequencies as one bf16 tensor-core product with error-free splitting "
          "(8 digits of 7 bits per value, exact digit products and sums), rounded once to float64",
}
UNIT = "freq points/s"
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
SMS, FP32_LANES, SM_MAX_MHZ = 152, 128, 2070.0
TF32_OVER_BF16 = 1.1 / 2.25  # nominal dense tf32 / bf16 tensor rates
FP64_NOMINAL_TFLOPS = 1.25   # nominal FP64 rate of the part


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(PEAKS_FALLBACK), "fallback"


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def workload_name(cfg):
    c = workload.CONFIGS[cfg]
    return (f"dense complex-symmetric sweep N={c.n}, {c.nf} frequencies {c.f_lo / 1e9:g}-{c.f_hi / 1e9:g} GHz, "
            f"{c.nrhs} RHS, Z = jwL - jPsi/w + Zs G")


def profile_traffic(kernel):
    """DRAM bytes per launch of `kernel` recorded by an ncu capture in
    profiles/traffic.json, or None when there is no record or the kernel's
    source file has changed since (each record holds the SHA-256 of the
    source it was measured with)."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f).get("kernels", {}).get(kernel)
    if not rec:
        return None
    src = os.path.join(ROOT, rec["source"])
    if not os.path.exists(src):
        return None
    with open(src, "rb") as f:
        if hashlib.sha256(f.read()).hexdigest() != rec.get("source_sha256"):
            return None
    return float(rec["dram_bytes_per_launch"])


# Kernels of the path and the profile stages their launches are counted in
# (k_cgemm_tc runs both the block solves and the trailing updates in the
# tensor-core modes; the FP32 mode has its own kernels for both).
STAGE_KERNELS = {
    "diag": "k_diag_block", "assemble": "k_assemble", "trsv": "k_trsv_inv", "residual": "k_residual",
    "pack": "k_pack_trsm", "update": "k_update + k_relcorr", "fallback": "k_lu64",
}


def kernel_times(stage_ms, gemm):
    """Device time per kernel (ms) from the per-stage sums of a profiled pass."""
    out = {STAGE_KERNELS[k]: v for k, v in stage_ms.items() if k in STAGE_KERNELS}
    if gemm == "FFMA":
        out["k_trsm_l + k_trsm_u"] = stage_ms.get("trsm", 0.0)
        out["k_schur_simt"] = stage_ms.get("schur", 0.0)
    else:
        out["k_cgemm_tc"] = stage_ms.get("trsm", 0.0) + stage_ms.get("schur", 0.0)
    return out


def oz_lane_evaluations(iters, lanes):
    """Residual evaluations per sweep in the mode OZ: each lane evaluates its
    frequencies together, once per correction of its slowest frequency (the
    lanes split the batch as the library does: lane k takes nf / K, the first
    nf % K one more)."""
    nf = len(iters)
    out, at = 0, 0
    for k in range(lanes):
        c = nf // lanes + (1 if k < nf % lanes else 0)
        if c:
            out += max(iters[at:at + c])
        at += c
    return out


def dominant_kernel(times, candidates):
    """The candidate with the largest device time in this run's profiled pass."""
    return max(candidates, key=lambda k: times.get(k, 0.0))


def diag_flops(nb=128):
    """Algorithmic real flops of one frequency's diagonal-block step: the LU of
    the nb x nb complex block (8/3 nb^3) and the inverses of its two
    triangles (4/3 nb^3 each)."""
    return 16.0 / 3.0 * nb ** 3


def trsm_flops(n, nb=128):
    """Useful real flops of all tensor-core block solves of one factorisation
    (L21 = A21 U11^-1 and U12 = L11^-1 A12: 2 x m2 x nb x nb complex MACs)."""
    tot = 0
    J = 0
    while J + nb < n:
        m2 = n - J - nb
        tot += 2 * 8 * m2 * nb * nb
        J += nb
    return tot


def schur_flops(n, nb=128, lower=False):
    """Useful real flops of all trailing updates of one factorisation (lower:
    the symmetric mode, whose update needs only the m2 (m2 + 1) / 2 entries on
    and below the diagonal)."""
    tot = 0
    J = 0
    while J + nb < n:
        m2 = n - J - nb
        tot += 8 * nb * (m2 * (m2 + 1) // 2 if lower else m2 * m2)
        J += nb
    return tot


class ClockSampler:
    """nvidia-smi every 50 ms from before the warm-up steps; only the samples
    whose own timestamps fall inside the timed span [mark, stop] are kept (the
    tool's output may be block-buffered, so the rows are read at the end)."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.proc = None
        self.t0 = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=self.file, stderr=subprocess.DEVNULL)
            atexit.register(self._end)
        except (OSError, ValueError):
            self.proc = None

    def _end(self):
        if self.proc is not None and self.proc.poll() is None:
            self.proc.kill()

    def mark(self):
        self.t0 = datetime.datetime.now()

    def stop(self):
        if self.proc is None:
            return None
        t1 = datetime.datetime.now()
        time.sleep(0.1)  # the sample taken at the end of the span
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        rows = [r.split(",") for r in self.file.read().strip().splitlines() if r.strip()]
        os.unlink(self.file.name)
        timed = []
        for r in rows:
            r = [x.strip() for x in r]
            try:
                ts = datetime.datetime.strptime(r[0], "%Y/%m/%d %H:%M:%S.%f")
                timed.append((ts, float(r[2]), float(r[3]), r[6:10]))
            except (ValueError, IndexError):
                continue
        t0 = self.t0 or t1
        lo, hi = t0 - datetime.timedelta(milliseconds=25), t1 + datetime.timedelta(milliseconds=60)
        inside = [t for t in timed if lo <= t[0] <= hi]
        if not inside:  # a span shorter than the period: the first sample after its start
            inside = [t for t in timed if t[0] >= lo][:1]
        if not inside:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = {nm for t in inside for nm, v in zip(names, t[3]) if v.lower().startswith("active")}
        return {"sm_mhz": statistics.median(t[1] for t in inside), "sm_max_mhz": max(t[2] for t in inside),
                "reasons": sorted(reasons), "samples": len(inside)}


def cpu_baseline(cfg, budget_s=10.0, max_freqs=None):
    """The oracle, as it stands, on a bounded sample of the workload's frequencies."""
    import oracle

    wl = workload.make(cfg)
    nf = len(wl.omega) if max_freqs is None else min(max_freqs, len(wl.omega))
    t0 = time.perf_counter()
    done = 0
    for f in range(nf):
        Z = oracle.assemble(wl.L, wl.Psi, wl.G, wl.omega[f], wl.zs[f])
        oracle.solve(Z, wl.B)
        done += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    return {"value": done / dt, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{done} of {len(wl.omega)} frequencies of N={wl.n} (assemble + complex128 pivoted LU + "
                      f"substitution, {wl.B.shape[0]} RHS), {dt:.1f} s"}


def profiled_pass(zs, torch, wl, args, L, P, G, b, x, flush):
    """The timed steps again, on a context with per-launch CUDA events
    (opts.profile) on the streams the kernels run on: per-stage device times
    and the tensor-core kernels' mean launch duration.  Returns the profile
    and the pass's ms per step."""
    n, nf, nrhs = wl.n, len(wl.omega), wl.B.shape[0]
    s = zs.Solver(n, nrhs, gemm=getattr(zs, "ZSOLVE_GEMM_" + args.gemm_eff), batch=args.batch or nf, profile=1,
                  resid=getattr(zs, "ZSOLVE_RESID_" + args.resid), symmetric=args.symmetric)
    try:
        for _ in range(args.warmup):
            zs.zsolve_sweep(s.ctx, L, P, G, wl.omega, wl.zs, b, x)
        torch.cuda.synchronize()
        zs.zsolve_reset_profile(s.ctx)
        st = torch.cuda.current_stream()
        ms = 0.0
        for _ in range(args.steps):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(st)
            zs.zsolve_sweep(s.ctx, L, P, G, wl.omega, wl.zs, b, x)
            e1.record(st)
            torch.cuda.synchronize()
            ms += e0.elapsed_time(e1)
        return zs.zsolve_get_profile(s.ctx).as_dict(), ms / args.steps
    finally:
        s.close()


def sweep_variant(zs, torch, wl, args, resid, symmetric=None):
    """The same timed sweep with another residual arithmetic (or factor mode):
    points/s and the residual stage's HBM rate (16 n^2 + 32 n nrhs bytes per
    evaluation over its CUDA-event time)."""
    n, nf, nrhs = wl.n, len(wl.omega), wl.B.shape[0]
    sym = args.symmetric if symmetric is None else symmetric
    s = zs.Solver(n, nrhs, gemm=getattr(zs, "ZSOLVE_GEMM_" + args.gemm_eff), batch=args.batch or nf, profile=1,
                  resid=getattr(zs, "ZSOLVE_RESID_" + resid), symmetric=sym)
    try:
        mode = RESID_NAMES[zs.zsolve_get_resid_mode(s.ctx)]
        L = torch.from_numpy(wl.L).cuda()
        P = torch.from_numpy(wl.Psi).cuda()
        G = torch.from_numpy(wl.G).cuda()
        b = torch.from_numpy(wl.B).cuda()
        x = torch.empty((nf, nrhs, n), dtype=torch.complex128, device="cuda")
        for _ in range(args.warmup):
            zs.zsolve_sweep(s.ctx, L, P, G, wl.omega, wl.zs, b, x)
        torch.cuda.synchronize()
        zs.zsolve_reset_profile(s.ctx)
        st = torch.cuda.current_stream()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(st)
        iters = 0
        for _ in range(args.steps):
            infos = zs.zsolve_sweep(s.ctx, L, P, G, wl.omega, wl.zs, b, x)
            iters += sum(i.iters for i in infos)
        e1.record(st)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / args.steps
        prof = zs.zsolve_get_profile(s.ctx).as_dict()
        res_ms = prof["residual"]["ms"] / args.steps
        res_bytes = iters / args.steps * (16.0 * n * n + 32.0 * n * nrhs)
        peaks, _ = load_peaks()
        gbs = res_bytes / (res_ms / 1e3) / 1e9 if res_ms > 0 else None
        out = {"mode_in_use": mode, "points_per_s": nf / (ms / 1e3), "resid_ms_per_step": res_ms,
               "resid_gbs": gbs, "resid_hbm_frac": (gbs / peaks["hbm_gbs"]) if gbs else None,
               "arith": RESID_ARITH[mode]}
        if mode in ("LPG", "OZ"):  # read L, Psi, G (or their digits), not Z (16 n^2 per frequency)
            out["note"] = "resid_gbs counts the float64 Z bytes the GEMV would read, for comparison"
        return out
    finally:
        s.close()


def afs_variant(zs, torch, args, flush):
    """Adaptive frequency sampling over 1001 candidates (the page's point limit)
    on the configuration's matrices: the resonant stand-in (Psi scaled so the
    band holds resonances, normalised omega in [1, 4]; Psi x 0.3 takes a few
    exact solves, Psi x 0.1 about thirty with a basis of ~64, the page's
    "q around 20-60") and the copper physics of the configuration's own band.  Candidate points/s = 1001 / the CUDA-event
    time of one whole zsolve_afs_sweep (exact solves, basis, evaluations and
    x = V y at every candidate), L2 flushed before each timed call."""
    m = 1001
    out = {"metric": "candidate points/s, reduced-order solution x = V y formed at every candidate",
           "m": m, "tol": 1e-4}
    cfg = workload.CONFIGS[args.config]
    cases = {"resonant": workload.make_resonant(args.config, m),
             "resonant_psi0.1": workload.make_resonant(args.config, m, psi_scale=0.1)}
    cu = workload.make(args.config)
    om = 2 * np.pi * np.linspace(cfg.f_lo, cfg.f_hi, m)
    cases["copper"] = dataclasses.replace(cu, omega=om, freqs=om / (2 * np.pi), zs=workload.surface_impedance(om))
    for name, wl in cases.items():
        n, nrhs = wl.n, wl.B.shape[0]
        s = zs.Solver(n, nrhs, batch=2)  # the exact solves take at most two frequencies at once
        try:
            with zs.Afs(s) as a:
                L = torch.from_numpy(wl.L).cuda()
                P = torch.from_numpy(wl.Psi).cuda()
                G = torch.from_numpy(wl.G).cuda()
                b = torch.from_numpy(wl.B).cuda()
                x = torch.empty((m, nrhs, n), dtype=torch.complex128, device="cuda")
                for _ in range(max(1, args.warmup - 1)):
                    a.sweep(L, P, G, wl.omega, wl.zs, b, x)
                st = torch.cuda.current_stream()
                times, info, l0 = [], None, zs.zsolve_afs_launches(a.afs)
                for _ in range(args.steps):
                    flush.fill_(1)
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    torch.cuda.synchronize()
                    e0.record(st)
                    sampled, resid, info = a.sweep(L, P, G, wl.omega, wl.zs, b, x)
                    e1.record(st)
                    torch.cuda.synchronize()
                    times.append(e0.elapsed_time(e1))
                launches = (zs.zsolve_afs_launches(a.afs) - l0) / args.steps
                ms = float(np.median(times))
                out[name] = {
                    "workload": (f"N={n}, {nrhs} RHS, " + (
                        f"Psi x {0.1 if name.endswith('0.1') else workload.AFS_PSI_SCALE}, normalised omega "
                        f"{workload.AFS_W_LO}-{workload.AFS_W_HI}, Zs = {workload.AFS_ZS_SCALE}(1+j)sqrt(omega)"
                        if name.startswith("resonant") else f"copper Zs, {cfg.f_lo / 1e9:g}-{cfg.f_hi / 1e9:g} GHz")),
                    "points_per_s": m / (ms / 1e3), "ms": ms, "n_exact": info.n_exact, "q": info.q,
                    "evals": info.evals, "converged": bool(info.converged), "max_resid": info.max_resid,
                    "sampled": sampled,
                    "phase_ms": {"exact": info.ms_exact, "basis": info.ms_basis, "eval": info.ms_eval,
                                 "expand": info.ms_expand},
                    "afs_launches": launches,
                    # k_afs_eval is float64-bound: its algorithmic flops over the
                    # evaluation phase's time (which also holds one small copy
                    # back per pass) against the part's nominal float64 rate
                    "eval_roofline": {
                        "kernel": "k_afs_eval", "bound": "fp64", "unit": "TFLOP/s",
                        "achieved": info.eval_gflop / info.ms_eval if info.ms_eval > 0 else None,
                        "peak": FP64_NOMINAL_TFLOPS, "peak_source": "nominal float64 rate of the part",
                        "frac": (info.eval_gflop / info.ms_eval / FP64_NOMINAL_TFLOPS) if info.ms_eval > 0 else None}}
                if args.cpu_baseline and name == "resonant":
                    import oracle
                    from oracle import afs as oafs
                    t0 = time.perf_counter()
                    oafs.afs_sweep(wl.L, wl.Psi, wl.G, wl.omega, wl.zs, wl.B)
                    t_cpu = time.perf_counter() - t0
                    out[name]["cpu_oracle"] = {"s": t_cpu, "cores": oracle.num_threads(), "points_per_s": m / t_cpu,
                                               "kind": "oracle (complex128 pivoted LU exact solves, numpy model)"}
        finally:
            s.close()
    return out


def large_configs(zs, torch, args):
    """The metric's large-system figures (one bounded pass each, headline
    settings, no variants): configuration 3 (N=8000, one frequency, 8 RHS)
    and configuration 4 (N=16384, 11 frequencies, 4 RHS).  Per configuration:
    points/s of whole sweeps (CUDA events on the launching stream, inputs
    resident, L2 flushed before each), the factorisation rate (8 N^3 / 3 real
    flops per frequency over the lanes' factorisation spans), and the
    residual's rate (16 N^2 + 32 N nrhs bytes per evaluation and frequency
    over the residual stage's device time, per-launch CUDA events)."""
    out = {}
    flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
    for cfg, warm, steps, batch in ((3, 2, 2, 1), (4, 1, 1, 6)):
        wl = workload.make(cfg)
        n, nf, nrhs = wl.n, len(wl.omega), wl.B.shape[0]
        s = zs.Solver(n, nrhs, gemm=getattr(zs, "ZSOLVE_GEMM_" + args.gemm_eff), batch=batch, profile=1,
                      resid=getattr(zs, "ZSOLVE_RESID_" + args.resid), symmetric=args.symmetric)
        try:
            L = torch.from_numpy(wl.L).cuda()
            P = torch.from_numpy(wl.Psi).cuda()
            G = torch.from_numpy(wl.G).cuda()
            b = torch.from_numpy(wl.B).cuda()
            x = torch.empty((nf, nrhs, n), dtype=torch.complex128, device="cuda")
            for _ in range(warm):
                zs.zsolve_sweep(s.ctx, L, P, G, wl.omega, wl.zs, b, x)
            torch.cuda.synchronize()
            zs.zsolve_reset_profile(s.ctx)
            st = torch.cuda.current_stream()
            ms, infos = 0.0, None
            for _ in range(steps):
                flush.zero_()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(st)
                infos = zs.zsolve_sweep(s.ctx, L, P, G, wl.omega, wl.zs, b, x)
                e1.record(st)
                torch.cuda.synchronize()
                ms += e0.elapsed_time(e1)
            ms /= steps
            prof = zs.zsolve_get_profile(s.ctx).as_dict()
            fac_ms = sum(i.ms_factor for i in infos)
            iters = [i.iters for i in infos]
            res_ms = prof["residual"]["ms"] / steps
            res_bytes = sum(iters) * (16.0 * n * n + 32.0 * n * nrhs)
            out[f"config{cfg}"] = {
                "workload": workload_name(cfg), "n": n, "nf": nf, "nrhs": nrhs, "batch": batch,
                "warmup": warm, "steps": steps, "ms_per_sweep": ms, "points_per_s": nf / (ms / 1e3),
                "lu_tflops": (8.0 * n ** 3 / 3.0 * nf) / (fac_ms / 1e3) / 1e12 if fac_ms > 0 else None,
                "resid_gbs": res_bytes / (res_ms / 1e3) / 1e9 if res_ms > 0 else None,
                "iters": iters, "fallbacks": sum(i.fallback for i in infos),
                "stage_ms_per_sweep": {k: v["ms"] / steps for k, v in prof.items()}}
            del L, P, G, b, x
        finally:
            s.close()
            torch.cuda.empty_cache()
    return out


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle

    wl = workload.make(args.config)
    per_step = 1  # frequencies per step: one direct solve each
    times = []
    for i in range(args.warmup + args.steps):
        f = i % len(wl.omega)
        t0 = time.perf_counter()
        for _ in range(per_step):
            Z = oracle.assemble(wl.L, wl.Psi, wl.G, wl.omega[f], wl.zs[f])
            oracle.solve(Z, wl.B)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            times.append(dt)
    tot = sum(times)
    value = per_step * len(times) / tot
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot / len(times),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": workload_name(args.config), "step": "one frequency"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
                             "sample": f"{per_step} frequency per step of N={wl.n}"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args):
    import torch

    import mixed_precision_refinement_gb300 as zs

    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    dist = None
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    cfg = workload.CONFIGS[args.config]
    wl = workload.make(args.config)
    n, nf, nrhs = wl.n, len(wl.omega), wl.B.shape[0]
    gemm = getattr(zs, "ZSOLVE_GEMM_" + args.gemm)
    # the headline pass runs without per-launch events (they add about 2 % to a
    # step); the profiled pass after it times every stage and launch
    solver = zs.Solver(n, nrhs, gemm=gemm, batch=args.batch or nf, profile=0,
                       resid=getattr(zs, "ZSOLVE_RESID_" + args.resid), symmetric=args.symmetric)
    ctx = solver.ctx
    resid_mode = RESID_NAMES[zs.zsolve_get_resid_mode(ctx)]
    L = torch.from_numpy(wl.L).cuda()
    P = torch.from_numpy(wl.Psi).cuda()
    G = torch.from_numpy(wl.G).cuda()
    b = torch.from_numpy(wl.B).cuda()
    x = torch.empty((nf, nrhs, n), dtype=torch.complex128, device="cuda")
    flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")  # > L2 (129 MB)
    stream = torch.cuda.current_stream()

    def step():
        return zs.zsolve_sweep(ctx, L, P, G, wl.omega, wl.zs, b, x)

    sampler = ClockSampler(torch.cuda.current_device()) if rank == 0 else None

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    # the arithmetic in use (AUTO: picked by its probe in the first warm-up
    # sweep); the profiled pass and the variants keep it fixed
    choice = zs.zsolve_get_gemm_choice(ctx)
    args.gemm_eff = {zs.ZSOLVE_GEMM_TF32: "TF32", zs.ZSOLVE_GEMM_TF32X3: "TF32X3", zs.ZSOLVE_GEMM_FFMA: "FFMA"}[choice.chosen]
    zs.zsolve_reset_profile(ctx)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    if sampler:
        sampler.mark()
    wall0 = time.perf_counter()
    infos = None
    for i in range(args.steps):
        flush.zero_()  # evict L2 between timed steps (outside the measured span)
        ev[i][0].record(stream)
        infos = step()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    wall = time.perf_counter() - wall0
    clocks = sampler.stop() if sampler else None
    ms = sum(a.elapsed_time(bb) for a, bb in ev)
    launch_counts = zs.zsolve_get_profile(ctx).as_dict()  # counted on every pass
    from mixed_precision_refinement_gb300 import sharding
    ms = sharding.max_over_ranks(ms, device="cuda")
    ms_step = ms / args.steps
    value = ws * nf / (ms_step / 1e3)

    # e2e: the public host-pointer API, host<->device copies inside the timed span
    Lh = torch.from_numpy(wl.L).pin_memory()
    Ph = torch.from_numpy(wl.Psi).pin_memory()
    Gh = torch.from_numpy(wl.G).pin_memory()
    bh = torch.from_numpy(wl.B).pin_memory()
    xh = torch.empty((nf, nrhs, n), dtype=torch.complex128).pin_memory()
    zs.zsolve_sweep_host(ctx, Lh, Ph, Gh, wl.omega, wl.zs, bh, xh)  # warm the host path once
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        zs.zsolve_sweep_host(ctx, Lh, Ph, Gh, wl.omega, wl.zs, bh, xh)
    e2e_s = (time.perf_counter() - t0) / args.steps
    e2e_s = sharding.max_over_ranks(e2e_s, device="cuda")
    prof, prof_ms_step = profiled_pass(zs, torch, wl, args, L, P, G, b, x, flush)
    if dist:
        dist.destroy_process_group()
    if rank != 0:
        return 0

    # --------------------------------------------------------------- derived numbers
    peaks, peak_src = load_peaks()
    iters = [i.iters for i in infos]
    n_res_calls = sum(iters)  # residual evaluations per step (one per correction)
    st = {k: v for k, v in prof.items()}
    steps = args.steps
    schur_f = schur_flops(n, lower=bool(args.symmetric)) * nf
    # factorisation time per step: the lanes' factorisation spans summed (each
    # frequency's info.ms_factor is its lane's span / the lane's frequencies),
    # so the overlap of the two lanes is not credited
    fac_ms = sum(i.ms_factor for i in infos)
    lu_tflops = (8.0 * n ** 3 / 3.0 * nf) / (fac_ms / 1e3) / 1e12 if fac_ms > 0 else None
    res_bytes = n_res_calls * (16.0 * n * n + 32.0 * n * nrhs)
    res_ms = st["residual"]["ms"] / steps
    res_gbs = res_bytes / (res_ms / 1e3) / 1e9 if res_ms > 0 else None
    stage_ms = {k: v["ms"] / steps for k, v in st.items()}
    fp32_peak = SMS * FP32_LANES * 2 * SM_MAX_MHZ * 1e6 / 1e12
    tf32_peak = peaks["bf16_tflops"] * TF32_OVER_BF16
    hbm = peaks["hbm_gbs"]
    # Roofline objects of the path's kernels: achieved = algorithmic work per
    # launch (flops or bytes, per unit as stated in "work") / the mean launch
    # duration from the profiled pass (CUDA events around every launch, on
    # the stream it runs on; with two lanes the launches run beside the other
    # lane's kernels).
    def obj(kernel, bound, stage_ms_tot, launches, work_tot, peak, unit, peak_source, work, **extra):
        launches = max(1, launches)
        lms = stage_ms_tot / launches
        ach = (work_tot / launches) / (lms / 1e3) / (1e12 if unit == "TFLOP/s" else 1e9) if lms > 0 else None
        o = {"kernel": kernel, "bound": bound, "achieved": ach, "peak": peak, "unit": unit,
             "frac": (ach / peak) if ach else None, "peak_source": peak_source, "work": work,
             "launch_ms": lms, "launches_per_step": launches / steps}
        o.update(extra)
        return o

    rl = {}
    tc = args.gemm_eff != "FFMA"
    tc_launches = st["schur"]["launches"] + (st["trsm"]["launches"] if tc else 0)
    tc_ms_tot = st["schur"]["ms"] + (st["trsm"]["ms"] if tc else 0.0)
    tc_flops_tot = (schur_f + (trsm_flops(n) * nf if tc else 0)) * steps
    if tc:
        rl["k_cgemm_tc"] = obj(
            "k_cgemm_tc", "tensor", tc_ms_tot, tc_launches, tc_flops_tot, tf32_peak, "TFLOP/s",
            f"tf32 = {peak_src} bf16 {peaks['bf16_tflops']} x 1.1/2.25",
            "useful complex-product flops (8 per complex MAC) of the trailing updates and block solves; "
            "the 3xTF32 split runs 3x that on the pipe",
            traffic=profile_traffic("k_cgemm_tc") if (args.config == 1 and args.gemm_eff == "TF32X3") else None)
    else:
        rl["k_schur_simt"] = obj(
            "k_schur_simt", "alu", st["schur"]["ms"], st["schur"]["launches"], schur_f * steps, fp32_peak,
            "TFLOP/s", "FP32 FFMA: 152 SMs x 128 lanes x 2 flop x 2070 MHz", "useful trailing-update flops")
    # k_diag_block: one CTA per frequency; the frequencies one launch covers x diag_flops
    d_launches = max(1, st["diag"]["launches"])
    d_units = nf * steps * ((n + 127) // 128) / d_launches
    dobj = obj("k_diag_block", "alu", st["diag"]["ms"], d_launches, diag_flops() * d_units * d_launches,
               fp32_peak, "TFLOP/s", "FP32 FFMA: 152 SMs x 128 lanes x 2 flop x 2070 MHz",
               f"16/3 x 128^3 real flop per frequency, {d_units:.1f} frequencies (one CTA each) per launch",
               traffic=profile_traffic("k_diag_block") if args.config == 1 else None)
    if dobj["achieved"]:
        dobj["frac_of_busy_sms"] = dobj["achieved"] / (fp32_peak * d_units / SMS)
    rl["k_diag_block"] = dobj
    # triangular solves: the float32 factors (8 n^2 bytes) once per solve and frequency
    n_solves = sum(i.iters + 1 for i in infos if not i.fallback)
    rl["k_trsv_inv"] = obj("k_trsv_inv", "hbm", st["trsv"]["ms"], st["trsv"]["launches"],
                           n_solves * 8.0 * n * n * math.ceil(nrhs / 4) * steps, hbm, "GB/s", f"{peak_src} copy",
                           "8 n^2 bytes of float32 factors per solve and frequency")
    if resid_mode == "OZ":
        # per sweep: the digits of L, Psi, G formed once (24 n^2 read, 48 n^2
        # written); per evaluation of a lane's frequencies: the 48 n^2 bytes of
        # digits read by the tensor-core product (x's digits and the partial
        # products are O(n) per column)
        lanes_eval = oz_lane_evaluations(iters, 2 if nf >= 2 else 1)
        oz_bytes = 72.0 * n * n + lanes_eval * 48.0 * n * n
        rl["k_residual"] = obj("k_oz_gemm", "hbm", st["residual"]["ms"], st["residual"]["launches"],
                               oz_bytes * steps, hbm, "GB/s", f"{peak_src} copy",
                               "48 n^2 bytes of digits per evaluation of a lane's frequencies, plus 72 n^2 per "
                               "sweep to form them; over the residual stage's device time (digit formation, "
                               "product, combination)", evaluations_per_step=lanes_eval,
                               traffic_k_oz_gemm=profile_traffic("k_oz_gemm") if args.config == 1 else None)
    else:
        rl["k_residual"] = obj({"F64": "k_residual", "DF": "k_residual_df", "FX": "k_residual_fx",
                                "LPG": "k_residual_lpg"}[resid_mode], "hbm", st["residual"]["ms"],
                               st["residual"]["launches"], res_bytes * steps, hbm, "GB/s", f"{peak_src} copy",
                               "16 n^2 + 32 n nrhs bytes per evaluation and frequency")
    lanes = 2 if nf >= 2 else 1
    # a lane whose residual reads L, Psi, G (LPG; OZ with four or more pairs)
    # assembles the float32 planes alone (k_assemble32: 8 n^2 written per
    # frequency), the others the float64 matrix too (k_assemble: 24 n^2)
    asm_bytes, only32 = 0.0, []
    for k in range(lanes):
        c = nf // lanes + (1 if k < nf % lanes else 0)
        o32 = resid_mode == "LPG" or (resid_mode == "OZ" and c * nrhs >= 4)
        only32.append(o32)
        asm_bytes += 24.0 * n * n + (8.0 if o32 else 24.0) * n * n * c
    asm_kernel = "k_assemble32" if all(only32) else "k_assemble" if not any(only32) else "k_assemble32 + k_assemble"
    rl["k_assemble"] = obj(asm_kernel, "hbm", st["assemble"]["ms"], st["assemble"]["launches"],
                           asm_bytes * steps, hbm, "GB/s", f"{peak_src} copy",
                           "24 n^2 bytes of L, Psi, G read once per lane + 8 n^2 (float32 planes alone) or 24 n^2 "
                           "(with the float64 matrix) written per frequency",
                           traffic=profile_traffic("k_assemble32")
                           if (args.config == 1 and asm_kernel == "k_assemble32") else None)
    ktimes = kernel_times(stage_ms, args.gemm_eff)
    dom = dominant_kernel(ktimes, list(rl))
    tot_k = sum(ktimes.values())
    launches = sum(v["launches"] for v in launch_counts.values())
    h2d = 3 * 8 * n * n + 16 * n * nrhs
    d2h = 16 * nf * nrhs * n
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32 factor + " + {"F64": "f64", "DF": "double-float f32x2", "FX": "f64-accurate int fixed-point",
                                    "LPG": "f64", "OZ": "f64-accurate bf16 tensor-core split"}[resid_mode]
                 + " residual",
        "data": "synthetic",
        "config": {"workload": workload_name(args.config), "n": n, "nf": nf, "nrhs": nrhs,
                   "gemm": args.gemm if args.gemm == args.gemm_eff else f"{args.gemm} -> {args.gemm_eff}",
                   "resid": resid_mode, "factor": "symmetric (lower tiles)" if args.symmetric else "full LU update",
                   "batch": args.batch or nf, "l2": "flushed between steps (512 MB write)",
                   "parallelism": f"{ws} independent replicas" if ws > 1 else "single GPU"},
        "lu_tflops": lu_tflops, "resid_gbs": res_gbs,
        "resid_gbs_basis": "16 n^2 + 32 n nrhs bytes per frequency and evaluation (what the float64 GEMV over Z "
                           "reads) over the residual stage's device time"
                           + ("; the OZ mode reads 48 n^2 bytes of digits per evaluation of a lane's frequencies "
                              "instead: its own rate is rooflines_other.k_residual" if resid_mode == "OZ" else ""),
        # the kernel with the largest device time in this run's profiled pass
        "roofline": rl[dom],
        "rooflines_other": {k: v for k, v in rl.items() if k != dom},
        "kernel_time_share_pct": {k: round(100.0 * v / tot_k, 2) for k, v in ktimes.items()} if tot_k else None,
        "stage_ms_per_step": stage_ms,
        "stage_note": "from a second pass of the same steps with CUDA events around every launch "
                      f"({prof_ms_step:.3f} ms per step with the events); per-stage sums of per-launch device "
                      "times; the two lanes run side by side, so the stages add up to more than a step",
        "iters": iters, "fallbacks": sum(i.fallback for i in infos),
        "gemm_choice": choice.as_dict(),
        "gpu_launches": int(launches),
        "e2e": {"value": ws * nf / e2e_s, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "clocks": clocks, "wall_s": wall,
    }
    solver.close()
    line["resid_variants"] = {
        args.resid: {"mode_in_use": resid_mode, "points_per_s": value / ws, "resid_gbs": res_gbs,
                     "resid_hbm_frac": (res_gbs / peaks["hbm_gbs"]) if res_gbs else None,
                     "arith": RESID_ARITH[resid_mode]}}
    for other in ("F64", "FX", "DF", "LPG", "OZ"):
        if other != args.resid:
            line["resid_variants"][other] = sweep_variant(zs, torch, wl, args, other)
    # the other factorisation mode: full trailing update, or the symmetric one
    # (lower tiles only, U12 from A21; same float64 residual and stopping rule)
    osym = 1 - args.symmetric
    line["factor_variants"] = {
        ("symmetric" if args.symmetric else "full"): {"points_per_s": value / ws},
        ("symmetric" if osym else "full"): sweep_variant(zs, torch, wl, args, args.resid, symmetric=osym)}
    if args.afs:
        line["afs"] = afs_variant(zs, torch, args, flush)
    if args.large and args.config == 1:
        line["large"] = large_configs(zs, torch, args)
    if args.cpu_baseline and args.gpus <= 1 and ws == 1:
        line["cpu_baseline"] = cpu_baseline(args.config, budget_s=args.cpu_budget)
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)  # ~0.6 s timed: about 12 clock samples
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", type=int, default=1)
    ap.add_argument("--gemm", default="AUTO", choices=["AUTO", "TF32", "TF32X3", "FFMA"])
    ap.add_argument("--batch", type=int, default=0)
    ap.add_argument("--resid", default="OZ", choices=["F64", "DF", "FX", "LPG", "OZ"])
    ap.add_argument("--cpu-budget", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", dest="cpu_baseline", action="store_false")
    ap.add_argument("--no-afs", dest="afs", action="store_false")
    ap.add_argument("--no-large", dest="large", action="store_false",
                    help="skip the N=8000 and N=16384 passes of the default line")
    ap.add_argument("--symmetric", type=int, default=1, choices=[0, 1],
                    help="1 (default): trailing update on the lower tiles only (Z is complex symmetric); 0: full")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
