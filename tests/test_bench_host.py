"""Host-side pieces of bench.py that need no GPU: the roofline denominators and
the recorded DRAM traffic, which must go null when its kernel source changes."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_peaks_have_every_denominator():
    pk = bench.peaks()
    assert pk["source"] in ("measured", "fallback")
    for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained"):
        assert pk[k] > 0
    assert pk["bf16_tflops_sustained"] <= pk["bf16_tflops"]


def test_recorded_traffic_follows_the_kernel_source(tmp_path, monkeypatch):
    # a private copy of the tree with the table and the two kernel sources
    csrc = tmp_path / "newton_schulz_04_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    src = b"// kernel v1\n"
    (csrc / "tc_gemm.cu").write_bytes(src)
    (csrc / "elementwise.cu").write_bytes(b"// other\n")
    import hashlib
    sha = hashlib.sha256(src).hexdigest()[:16]
    (tmp_path / "profiles" / "dram_traffic.md").write_text(
        "| workload | kernel | sha | launches | read | write | traffic | us |\n|---|---|---|---|---|---|---|---|\n"
        f"| c2 | tc_sym | {sha} | 8 | 36.77 | 0.30 | 37.07 | 33.3 |\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.recorded_traffic("c2", "tc_sym") == 37.07e6
    assert bench.recorded_traffic("c3", "tc_sym") is None       # no row for the workload
    assert bench.recorded_traffic("c2", "pack") is None         # no row for the kernel
    (csrc / "tc_gemm.cu").write_bytes(b"// kernel v2\n")
    assert bench.recorded_traffic("c2", "tc_sym") is None       # source changed since capture


def test_committed_traffic_rows_parse():
    rows = 0
    for line in open(os.path.join(ROOT, "profiles", "dram_traffic.md")):
        cells = [c.strip() for c in line.strip().strip("|").split("|")]
        if len(cells) == 8 and cells[0].startswith("c") and cells[3].isdigit():
            rows += 1
            assert abs(float(cells[6]) - (float(cells[4]) + float(cells[5]))) <= 0.011
    assert rows >= 1
