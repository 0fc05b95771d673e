"""Host-side arithmetic of bench.py, without a GPU: the flop counts behind
the roofline objects, the choice of the roofline kernel from a run's own
per-stage times, and the source-hash check that keeps a recorded DRAM
traffic figure from outliving the kernel it was measured on."""
import hashlib
import json
import os

import pytest

import bench


@pytest.mark.parametrize("blocks", [1, 2, 3, 5])
def test_blocked_flops_add_up_to_the_lu(blocks):
    # n a multiple of the outer block: the diagonal blocks' LU (8/3 nb^3
    # each), the block solves (counted as dense products with the explicit
    # inverses, twice the triangular work) and the trailing updates make up
    # the 8 n^3 / 3 real flops of a complex LU exactly
    nb = 128
    n = blocks * nb
    diag_lu = blocks * 8.0 * nb ** 3 / 3.0
    total = diag_lu + bench.trsm_flops(n, nb) / 2.0 + bench.schur_flops(n, nb)
    assert total == pytest.approx(8.0 * n ** 3 / 3.0, rel=1e-12)


def test_diag_flops():
    # LU of the block and the inverses of its two triangles: 8/3 + 2 x 4/3
    assert bench.diag_flops(128) == pytest.approx(16.0 / 3.0 * 128 ** 3)


def test_schur_and_trsm_flops_small_cases():
    assert bench.schur_flops(128) == 0 and bench.trsm_flops(128) == 0  # one block: no update
    # two blocks: one update of a 128 x 128 block with K = 128, two 128 x 128 solves
    assert bench.schur_flops(256) == 8 * 128 ** 3
    assert bench.schur_flops(256, lower=True) == 8 * 128 * (128 * 129 // 2)
    assert bench.trsm_flops(256) == 2 * 8 * 128 ** 3


def test_dominant_kernel_from_stage_times():
    stage = {"assemble": 1.0, "diag": 3.9, "trsm": 1.9, "schur": 2.2, "trsv": 1.4, "residual": 1.7,
             "update": 0.1, "fallback": 0.0, "pack": 1.2}
    t = bench.kernel_times(stage, "TF32X3")
    assert t["k_cgemm_tc"] == pytest.approx(4.1) and t["k_diag_block"] == 3.9
    assert bench.dominant_kernel(t, ["k_diag_block", "k_cgemm_tc", "k_residual"]) == "k_cgemm_tc"
    stage["diag"] = 4.5
    assert bench.dominant_kernel(bench.kernel_times(stage, "TF32X3"), ["k_diag_block", "k_cgemm_tc"]) == "k_diag_block"
    f = bench.kernel_times(stage, "FFMA")
    assert "k_cgemm_tc" not in f and f["k_schur_simt"] == 2.2


def test_profile_traffic_follows_the_source_hash(tmp_path, monkeypatch):
    src_dir = tmp_path / "mixed_precision_refinement_gb300" / "csrc"
    src_dir.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    src = src_dir / "k.cu"
    src.write_bytes(b"// kernel source\n")
    digest = hashlib.sha256(src.read_bytes()).hexdigest()
    rec = {"kernels": {"k": {"dram_bytes_per_launch": 12345, "source_sha256": digest,
                             "source": "mixed_precision_refinement_gb300/csrc/k.cu"}}}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.profile_traffic("k") == 12345.0
    src.write_bytes(b"// kernel source, changed\n")
    assert bench.profile_traffic("k") is None
    assert bench.profile_traffic("missing") is None
    assert os.path.exists(src)


def test_committed_traffic_records_are_well_formed():
    with open(os.path.join(bench.ROOT, "profiles", "traffic.json")) as f:
        rec = json.load(f)["kernels"]
    for k, r in rec.items():
        assert k.startswith("k_") and r["dram_bytes_per_launch"] > 0
        assert os.path.exists(os.path.join(bench.ROOT, r["source"])) and len(r["source_sha256"]) == 64
