"""The oracle still reproduces the stored tiny-workload fixture
(tests/golden/tiny_fprop_mxfp8.json, written by tests/golden/make_golden.py)."""
import hashlib
import json
import os

import numpy as np

import oracle
from moe_grouped_block_gb300 import workloads

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "tiny_fprop_mxfp8.json")


def test_oracle_reproduces_golden():
    gold = json.load(open(GOLDEN))
    wl = workloads.WORKLOADS["tiny_fprop_mxfp8"]
    inp = workloads.make_inputs(wl)
    G, N, K, M = wl.G, wl.N, wl.K, wl.M
    ws, st = oracle.group_offsets(inp["sizes"].numpy(), 1, K, M)
    assert [int(v) for v in ws] == gold["offsets_workspace"] and st == gold["status"]
    qx = oracle.mxfp8_quantize(inp["x"], M, M, rowwise=True, colwise=True)
    qw = oracle.mxfp8_quantize(inp["w"].reshape(G * N, K), G * N, G * N, rowwise=True)
    got = {"x_q_row": qx["q_row"], "x_sf_row": qx["sf_row"], "x_q_col": qx["q_col"],
           "x_sf_col": qx["sf_col"], "w_q_row": qw["q_row"], "w_sf_row": qw["sf_row"]}
    for k, v in got.items():
        assert hashlib.sha256(np.ascontiguousarray(v).tobytes()).hexdigest() == gold["sha256"][k], k
    rows = sorted({r for r, _, _ in gold["gemm_samples"]})
    _, _, C = oracle.grouped_gemm_fprop("mxfp8", {"q": qx["q_row"], "sf": qx["sf_row"]},
                                        {"q": qw["q_row"], "sf": qw["sf_row"]},
                                        oracle.live_rows(ws, G), N, K, sample_rows=rows)
    for r, c, v in gold["gemm_samples"]:
        assert C[rows.index(r), c] == v
