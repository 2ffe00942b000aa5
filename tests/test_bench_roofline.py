"""Host logic of the benchmark's GEMM roofline object (no GPU): the bound is
whichever roofline time is larger, FLOP at the dense tensor peak or
algorithmic bytes at the measured HBM bandwidth, and frac is the achieved
fraction of that peak, equal to t_roofline / t; the measured DRAM traffic is
reported only while the GEMM sources and compile flags hash to the digest it
was taken on; the oracle timing sample is the same in both arms; the
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


def test_traffic_is_reported_only_for_the_measured_sources():
    fresh = {"digest": bench.gemm_source_digest(),
             "bytes": {"mixtral_fprop_mxfp8": 1015692544, "wgrad_mxfp8": 30}}
    assert bench.measured_traffic("mixtral_fprop_mxfp8", fresh) == 1015692544
    assert bench.measured_traffic("wgrad_mxfp8", fresh) == 30
    assert bench.measured_traffic("no_such_workload", fresh) is None
    # the same table measured on other sources or flags (the kernel changed since): none
    stale = dict(fresh, digest="0" * 64)
    assert bench.measured_traffic("mixtral_fprop_mxfp8", stale) is None
    # no table at all: none
    assert bench.measured_traffic("mixtral_fprop_mxfp8", {"digest": None, "bytes": {}}) is None


def test_digest_covers_the_compile_flags(monkeypatch):
    from moe_grouped_block_gb300 import build as mxg_build
    d0 = bench.gemm_source_digest()
    monkeypatch.setattr(mxg_build, "NVCC_FLAGS", mxg_build.NVCC_FLAGS + ["-maxrregcount=128"])
    assert bench.gemm_source_digest() != d0


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


def test_oracle_sample_covers_every_expert_and_an_eighth_of_the_columns():
    """The oracle's timing sample: every live row of each expert and the first
    eighth of the output columns (rounded up to 128); FLOP = 2 m c K."""
    from moe_grouped_block_gb300 import workloads
    wl = workloads.WORKLOADS["tiny_fprop_mxfp8"].scaled(N=1024)
    inp = workloads.make_inputs(wl)
    smp = bench.oracle_sample(wl, inp)
    assert list(smp["sizes"]) == [128, 0, 256, 128] and smp["cols"] == 128
    assert tuple(smp["x"].shape) == (512, wl.K) and tuple(smp["w"].shape) == (wl.G, 128, wl.K)
    quarter = bench.oracle_sample(wl, inp, 0.25)
    assert list(quarter["sizes"]) == [128, 0, 128, 128]
    t, f = bench.oracle_pass(wl, smp)
    assert f == 2.0 * 512 * 128 * wl.K and t > 0
    for name in ("wgrad_mxfp8", "dgrad_mxfp8", "rowscaled_fprop_nvfp4", "wgrad_nvfp4"):
        w2 = workloads.WORKLOADS[name].scaled(M=512, K=256, N=256, G=2, sizes="fixed",
                                              fixed_sizes=(384, 128))
        s2 = bench.oracle_sample(w2, workloads.make_inputs(w2))
        t2, f2 = bench.oracle_pass(w2, s2)
        assert f2 == 2.0 * 512 * 128 * 256, name


def test_single_core_child_runs_the_same_pass():
    from moe_grouped_block_gb300 import workloads
    wl = workloads.WORKLOADS["tiny_fprop_mxfp8"]
    smp = bench.oracle_sample(wl, workloads.make_inputs(wl))
    r = bench.single_core_pass(wl, smp)
    assert r is not None and r[1] == bench.oracle_pass(wl, smp)[1]


def test_digest_does_not_depend_on_the_checkout_path(monkeypatch):
    """The recorded digest must match on another machine, where the repository
    sits elsewhere and the include flag names that path."""
    from moe_grouped_block_gb300 import build as mxg_build
    d0 = bench.gemm_source_digest()
    moved = [("-I/elsewhere/checkout/include" if f.startswith("-I") else f)
             for f in mxg_build.NVCC_FLAGS]
    monkeypatch.setattr(bench, "ROOT", "/elsewhere/checkout")
    monkeypatch.setattr(mxg_build, "NVCC_FLAGS", moved)
    src_root = os.path.join(os.path.dirname(os.path.abspath(bench.__file__)))
    real_open = open

    def open_from_repo(path, *a, **k):
        if str(path).startswith("/elsewhere/checkout"):
            path = src_root + str(path)[len("/elsewhere/checkout"):]
        return real_open(path, *a, **k)
    monkeypatch.setattr("builtins.open", open_from_repo)
    assert bench.gemm_source_digest() == d0
