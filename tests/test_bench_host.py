"""Host-side pieces of bench.py that need no GPU: the roofline denominators and
the recorded DRAM traffic, which must go null when its kernel source changes."""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402

NCU_HEADER = ('"ID","Process ID","Process Name","Host Name","Kernel Name","Context","Stream","Block Size",'
              '"Grid Size","Device","CC","Section Name","Metric Name","Metric Unit","Metric Value"\n')


def _row(i, kernel, metric, unit, value):
    return (f'"{i}","1","python3","h","{kernel}","1","7","(320, 1, 1)","(152, 1, 1)","0","10.3",'
            f'"Command line profiler metrics","{metric}","{unit}","{value}"\n')


def test_peaks_have_every_denominator():
    pk = bench.peaks()
    assert pk["source"] in ("measured", "fallback")
    for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained"):
        assert pk[k] > 0
    assert pk["bf16_tflops_sustained"] <= pk["bf16_tflops"]


def test_kernel_families():
    for label in ("tc_rect", "tc_syrk_x3", "tc_program", "void muon::tc_gemm_kernel<16>(muon::TcProgram<16>)",
                  "void tc_gemm_kernel<16>(TcProgram<T1>)"):
        assert bench.family_of(label) == "tc_gemm"
    assert bench.family_of("simt_sym") == "simt_gemm"
    assert bench.family_of("void muon::pack_vec_kernel<false>(muon::PackArgs)") == "pack"
    assert bench.family_of("norm_finalize") == "norm_finalize"


def test_recorded_traffic_follows_the_kernel_source(tmp_path, monkeypatch):
    # a private copy of the tree with the kernel sources and an ncu metrics log
    csrc = tmp_path / "newton_schulz_04_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    (csrc / "tc_gemm.cu").write_bytes(b"// kernel v1\n")
    (csrc / "elementwise.cu").write_bytes(b"// other\n")
    log = tmp_path / "traffic.csv"
    k_tc = "void muon::tc_gemm_kernel<1>(muon::TcProgram<1>)"
    k_pk = "void muon::pack_vec_kernel<false>(muon::PackArgs)"
    log.write_text("==PROF== Connected to process 1\n" + NCU_HEADER +
                   _row(0, k_pk, "dram__bytes_read.sum", "Mbyte", "100.5") +
                   _row(0, k_pk, "dram__bytes_write.sum", "Mbyte", "75.5") +
                   _row(0, k_pk, "gpu__time_duration.sum", "usecond", "35.9") +
                   _row(1, k_tc, "dram__bytes_read.sum", "Gbyte", "1.5") +
                   _row(1, k_tc, "dram__bytes_write.sum", "Mbyte", "500") +
                   _row(1, k_tc, "gpu__time_duration.sum", "msecond", "2") +
                   _row(2, k_tc, "dram__bytes_read.sum", "Gbyte", "0.5") +
                   _row(2, k_tc, "dram__bytes_write.sum", "Mbyte", "1,500") +
                   _row(2, k_tc, "gpu__time_duration.sum", "ns", "4000000"))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    parsed = bench.parse_ncu_csv(str(log))
    assert parsed[1]["dram__bytes_read.sum"] == 1.5e9 and parsed[2]["dram__bytes_write.sum"] == 1.5e9
    bench.record_traffic(str(log), "c3", "ncu ...", scale=4.0, note="scaled")
    doc = json.load(open(tmp_path / "profiles" / "dram_traffic.json"))
    tc = [r for r in doc["rows"] if r["family"] == "tc_gemm"][0]
    assert tc["launches"] == 2 and tc["bytes_per_launch"] == 4.0 * (2.0e9 + 2.0e9) / 2
    assert abs(tc["ncu_us_per_launch"] - 3000.0) < 1e-6
    assert bench.recorded_traffic("c3", "tc_gemm") == 8.0e9
    assert bench.recorded_traffic("c3", "pack") == 4.0 * 176e6
    assert bench.recorded_traffic("c2", "tc_gemm") is None       # no row for the workload
    assert bench.recorded_traffic("c3", "simt_gemm") is None     # no row for the family
    (csrc / "tc_gemm.cu").write_bytes(b"// kernel v2\n")
    assert bench.recorded_traffic("c3", "tc_gemm") is None       # source changed since capture
    assert bench.recorded_traffic("c3", "pack") == 4.0 * 176e6   # its own source is unchanged


def test_committed_traffic_rows_are_consistent():
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(path):
        return
    doc = json.load(open(path))
    for r in doc["rows"]:
        assert abs(r["bytes_per_launch"] - r["read_bytes_per_launch"] - r["write_bytes_per_launch"]) <= \
            1e-9 * r["bytes_per_launch"] + 1
        assert r["family"] in bench.FAMILY_SOURCES and r["command"]


def test_c5_config_names():
    assert bench.c5_params("c5f32_n4096_t10") == (4096, 10)
    assert bench.c5_params("c5_n16384") == (16384, 5)
    assert "layers" in bench.workload_desc("c3_l2")


def test_clock_records_that_are_rejected():
    """hw/thermal slowdowns, or a clock stuck far below its maximum without a
    power-cap reason, reject a timed region; the power cap alone does not."""
    import bench
    ok = {"sm_mhz": 1600.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"]}
    assert not bench.clocks_rejected(ok)
    assert not bench.clocks_rejected({"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": []})
    assert bench.clocks_rejected(dict(ok, reasons=["sw_power_cap", "hw_slowdown"]))
    assert bench.clocks_rejected(dict(ok, reasons=["sw_thermal_slowdown"]))
    assert bench.clocks_rejected({"sm_mhz": 900.0, "sm_max_mhz": 2070.0, "reasons": []})
    assert not bench.clocks_rejected({"sm_mhz": 900.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"]})
    assert not bench.clocks_rejected({"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]})
