"""Host check of the premise of the natural-stall test (tests/test_gpu_failure.py):
the growth workload is well conditioned in double precision, while its
unpivoted elimination grows the entries by about 1/eps."""
import numpy as np

import oracle
import workload


def test_growth_workload_is_well_conditioned():
    wl = workload.make_growth(300, seed=3)
    Z = oracle.assemble(wl.L, wl.Psi, wl.G, wl.omega[0], wl.zs[0])
    # 1-norm condition a few hundred at n = 300 (2-norm condition about 3)
    assert oracle.condest1(Z) < 1e3
    LU, st = oracle.lu_nopiv(oracle.cast_c64(Z))
    assert st == 0
    # unpivoted elimination grows the entries by about 1/eps
    assert np.abs(LU).max() > 1e6 * np.abs(Z).max()
