"""The seeded input recipe (no GPU): group sizes per workload (sums, 128-row
multiples, empty groups where the recipe asks for one), determinism by seed,
shapes per mode, and the value distributions the workloads stand for."""
import numpy as np
import pytest
import torch

from moe_grouped_block_gb300 import workloads

ALL = sorted(workloads.WORKLOADS)


@pytest.mark.parametrize("name", ALL)
def test_group_sizes_partition_the_rows(name):
    wl = workloads.WORKLOADS[name]
    s = workloads.group_sizes(wl)
    assert s.dtype == np.int32 and s.shape == (wl.G,)
    assert int(s.sum()) == wl.M and (s >= 0).all()
    if wl.sizes != "dirichlet_rows":
        assert (s % 128 == 0).all()
    # the same seed gives the same routing
    assert np.array_equal(s, workloads.group_sizes(wl))


def test_tiny_workload_sizes_are_the_fixed_ones():
    assert workloads.group_sizes(workloads.WORKLOADS["tiny_fprop_mxfp8"]).tolist() == [128, 0, 256, 128]


def test_finegrained_routing_has_empty_groups_and_a_heavy_head():
    wl = workloads.WORKLOADS["finegrained_fprop_mxfp8"]
    s = workloads.group_sizes(wl)
    assert (s == 0).any()
    # Zipf(1.2) over 64 experts: the largest expert takes far more than 1/64 of the rows
    assert s.max() > 8 * wl.M / wl.G


def test_unaligned_routing_has_sizes_off_the_128_grid():
    s = workloads.group_sizes(workloads.WORKLOADS["mixtral_fprop_mxfp8_unaligned"])
    assert (s % 128 != 0).any()


@pytest.mark.parametrize("name", ALL)
def test_inputs_are_deterministic_and_shaped_by_mode(name):
    wl = workloads.WORKLOADS[name].scaled(M=512, K=256, N=256)
    if wl.sizes == "fixed":
        wl = wl.scaled(fixed_sizes=(128, 0, 256, 128))
    elif wl.sizes != "dirichlet_rows":
        wl = wl.scaled(G=min(wl.G, 4))
    a, b = workloads.make_inputs(wl), workloads.make_inputs(wl)
    R, G, N, K = wl.rows_capacity, wl.G, wl.N, wl.K
    expect = {"fprop": {"x": (R, K), "w": (G, N, K)}, "wgrad": {"x": (R, K), "dy": (R, N)},
              "dgrad": {"dy": (R, N), "w": (G, N, K)}}[wl.mode]
    for key, shape in expect.items():
        assert tuple(a[key].shape) == shape and a[key].dtype == torch.bfloat16, key
        assert torch.equal(a[key], b[key]), key
    assert torch.equal(a["sizes"], b["sizes"])


def _stats(t):
    v = t.float().numpy().reshape(-1).astype(np.float64)
    return v.mean(), v.std(), v


def test_value_distributions():
    # activations N(0, 1), weights N(0, 0.02), gradients N(0, 1e-3) (std, our reading)
    wl = workloads.WORKLOADS["wgrad_mxfp8"].scaled(M=4096, K=512, N=512, G=4)
    inp = workloads.make_inputs(wl)
    m, s, _ = _stats(inp["x"])
    assert abs(m) < 0.01 and abs(s - 1.0) < 0.01
    m, s, _ = _stats(inp["dy"])
    assert abs(s - 1e-3) < 2e-5
    wf = workloads.WORKLOADS["mixtral_fprop_mxfp8"].scaled(M=512, K=512, N=512, G=4)
    m, s, _ = _stats(workloads.make_inputs(wf)["w"])
    assert abs(s - 0.02) < 5e-4


def test_finegrained_outliers_and_student_t_tails():
    # 0.1 % of the activations scaled by 100
    wl = workloads.WORKLOADS["finegrained_fprop_mxfp8"].scaled(M=4096, K=512, N=256, G=4)
    _, _, v = _stats(workloads.make_inputs(wl)["x"])
    frac = np.mean(np.abs(v) > 20.0)
    assert 0.0005 < frac < 0.0015
    # Student-t(3): heavy tails (kurtosis far above the normal's 3)
    wn = workloads.WORKLOADS["rowscaled_fprop_nvfp4"].scaled(M=4096, K=512, N=256, G=4)
    _, _, v = _stats(workloads.make_inputs(wn)["x"])
    kurt = np.mean((v - v.mean()) ** 4) / np.var(v) ** 2
    assert kurt > 10.0
