"""Host-side arithmetic of bench.py, without a GPU: the flop counts behind
the roofline objects, the parser of the committed ncu launch list, and the
source-hash check that keeps a recorded DRAM traffic figure from outliving
the kernel it was measured on."""
import hashlib
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


def test_launch_list_shares_parse_the_committed_profile():
    shares = bench.launch_list_shares()
    assert "k_cgemm_tc" in shares and "k_diag_block" in shares
    assert sum(shares.values()) == pytest.approx(100.0, abs=1.5)
    assert max(shares, key=shares.get) in ("k_cgemm_tc", "k_diag_block")


def test_profile_traffic_follows_the_source_hash(tmp_path, monkeypatch):
    src_dir = tmp_path / "mixed_precision_refinement_gb300" / "csrc"
    src_dir.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    src = src_dir / "k.cu"
    src.write_bytes(b"// kernel source\n")
    digest = hashlib.sha256(src.read_bytes()).hexdigest()
    (tmp_path / "profiles" / "k_n.md").write_text(
        f"# k\n\n- dram_bytes_per_launch: `12345`\n- source_sha256: `{digest}`\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.profile_traffic("k_n", "k.cu") == 12345.0
    src.write_bytes(b"// kernel source, changed\n")
    assert bench.profile_traffic("k_n", "k.cu") is None
    assert bench.profile_traffic("missing", "k.cu") is None
    assert os.path.exists(src)
