"""Host logic of the benchmark's GEMM roofline object (no GPU): the bound is
whichever roofline time is larger, FLOP at the dense tensor peak or
algorithmic bytes at the measured HBM bandwidth, and frac is the achieved
fraction of that peak, equal to t_roofline / t; the measured DRAM traffic is
reported only while the GEMM sources hash to the digest it was taken on; the
clock record's throttle reasons are read from nvidia-smi lines or NVML bits."""
import os
import sys

import pytest

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402

PEAKS = {"bf16_tflops": 1892.9, "hbm_gbs": 6776.3}


def test_mixtral_fprop_is_tensor_bound():
    # 2 M N K FLOP; A + W of the live experts (+ scales) + bf16 C
    M, N, K, G = 16384, 14336, 4096, 8
    flops = 2.0 * M * N * K
    nbytes = M * K * (1 + 1 / 32) + G * N * K * (1 + 1 / 32) + M * N * 2
    r = bench.gemm_roofline("g", flops, nbytes, 0.6, PEAKS, "measured", False, None)
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert r["peak"] == pytest.approx(2 * 1892.9, rel=1e-4)
    assert r["achieved"] == pytest.approx(flops / 0.6e-3 / 1e12, rel=1e-3)
    assert r["frac"] == pytest.approx(r["t_roofline_over_t"], rel=1e-3)


def test_rowscaled_nvfp4_layer_is_hbm_bound():
    # 32 experts, K 7168, N 2048, M 16384 (all experts live), bf16 C: the
    # algorithmic bytes take longer at HBM bandwidth than the FLOP at the NVFP4 peak
    M, N, K, G = 16384, 2048, 7168, 32
    flops = 2.0 * M * N * K
    nbytes = M * K * (0.5 + 1 / 16) + G * N * K * (0.5 + 1 / 16) + M * N * 2 + 4 * (M + G * N)
    t = 0.1105
    r = bench.gemm_roofline("g", flops, nbytes, t, PEAKS, "measured", True, 123)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["peak"] == PEAKS["hbm_gbs"]
    assert r["t_hbm_roofline_ms"] > r["t_tensor_roofline_ms"]
    assert r["frac"] == pytest.approx(nbytes / (PEAKS["hbm_gbs"] * 1e9) / (t * 1e-3), rel=1e-3)
    assert r["frac"] == pytest.approx(r["t_roofline_over_t"], rel=1e-3)
    assert r["tflops_frac"] == pytest.approx(flops / (t * 1e-3) / 1e12 / (6 * 1892.9), rel=1e-3)
    assert r["traffic"] == 123


def test_finegrained_sits_just_on_the_tensor_side():
    # G 64, K 2048, N 1408, M 32768: near the ridge, the FLOP time is the larger
    M, N, K = 32768, 1408, 2048
    flops = 2.0 * M * N * K
    live = 43
    nbytes = M * K * (1 + 1 / 32) + live * N * K * (1 + 1 / 32) + M * N * 2
    r = bench.gemm_roofline("g", flops, nbytes, 0.0924, PEAKS, "measured", False, None)
    assert r["bound"] == "tensor"
    assert r["t_tensor_roofline_ms"] > r["t_hbm_roofline_ms"]


ROW = "| mixtral_fprop_mxfp8 | `k` | 568991744 | 446700800 | 1015692544 | 620.7 | alg |\n"


def test_traffic_is_reported_only_for_the_measured_sources(tmp_path, monkeypatch):
    head = "| workload | kernel | read bytes | write bytes | traffic bytes | us | alg |\n|---|---|---|---|---|---|---|\n"
    fresh = tmp_path / "fresh.md"
    fresh.write_text("sources sha256: `%s`\n\n" % bench.gemm_source_digest() + head + ROW)
    monkeypatch.setattr(bench, "TRAFFIC_SUMMARY", str(fresh))
    assert bench.measured_traffic("mixtral_fprop_mxfp8") == 1015692544
    assert bench.measured_traffic("no_such_workload") is None
    # the same table measured on other sources (the kernel changed since): none
    stale = tmp_path / "stale.md"
    stale.write_text("sources sha256: `%s`\n\n" % ("0" * 64) + head + ROW)
    monkeypatch.setattr(bench, "TRAFFIC_SUMMARY", str(stale))
    assert bench.measured_traffic("mixtral_fprop_mxfp8") is None
    # no summary at all: none
    monkeypatch.setattr(bench, "TRAFFIC_SUMMARY", str(tmp_path / "absent.md"))
    assert bench.measured_traffic("mixtral_fprop_mxfp8") is None


def test_traffic_table_row_is_read_by_workload(tmp_path, monkeypatch):
    digest = bench.gemm_source_digest()
    table = ("sources sha256: `%s`\n\n| workload | kernel | read bytes | write bytes | traffic bytes |\n"
             "|---|---|---|---|---|\n| wl_a | `k` | 1 | 2 | 3 |\n| wl_b | `k` | 10 | 20 | 30 |\n" % digest)
    f = tmp_path / "traffic.md"
    f.write_text(table)
    monkeypatch.setattr(bench, "TRAFFIC_SUMMARY", str(f))
    assert bench.measured_traffic("wl_a") == 3
    assert bench.measured_traffic("wl_b") == 30


def test_digest_ignores_comments_but_not_code():
    src = "int f(int a) {  // returns a + 1\n  /* block\n comment */ return a + 1;\n}\n"
    same = "int f(int a) {\n  return a + 1;   // reworded comment\n}\n"
    other = "int f(int a) {\n  return a + 2;\n}\n"
    assert bench.code_only(src) == bench.code_only(same)
    assert bench.code_only(src) != bench.code_only(other)


class _Done:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0

    def kill(self):
        pass


class _Joined:
    def join(self, timeout=None):
        pass


def test_clock_reasons_from_nvidia_smi_lines():
    c = bench.ClockSampler(0)
    c.proc, c.t = _Done(), _Joined()
    c.lines = ["2070, 2070, 900.5, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
               "1980, 2070, 1390.1, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
               "2070, 2070, 1200.0, 0x0000000000000008, Active, Not Active, Not Active, Not Active",
               "garbage line"]
    r = c.stop()
    assert r["sm_mhz"] == 2070 and r["sm_max_mhz"] == 2070 and r["samples"] == 3
    assert r["reasons"] == ["hw_slowdown", "sw_power_cap"]


def test_clock_reasons_from_nvml_samples():
    c = bench.ClockSampler(0)
    c.nvml, c.t, c.running = object(), _Joined(), True
    c.samples = [(2070, 2070, 0x0), (2070, 2070, 0x4), (1500, 2070, 0x40), (2070, 2070, 0x1)]
    r = c.stop()
    assert r["sm_mhz"] == 2070 and r["sm_max_mhz"] == 2070 and r["samples"] == 4
    # 0x1 (idle) is not a throttle reason; 0x4 power cap, 0x40 hardware thermal
    assert r["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"]
