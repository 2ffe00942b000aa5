"""Writes tests/golden/tiny_fprop_mxfp8.json from the oracle alone.

Workload: 4 experts, K = N = 256, group rows [128, 0, 256, 128], seed 0 (the
tiny MXFP8 grouped fprop case).  Stored: the int64 offsets workspace, SHA-256
digests of the quantized bytes and swizzled scales (rowwise and colwise of X,
rowwise of W), and a handful of fp64 GEMM outputs.  The pages print no worked
example, so these values pin the oracle against unintended change only; its
correctness pins are the tests/test_oracle_*.py suites.

Run from the repository root:  python tests/golden/make_golden.py
"""
import hashlib
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from moe_grouped_block_gb300 import workloads  # noqa: E402

SAMPLES = [(0, 0), (5, 17), (127, 255), (128, 3), (300, 128), (383, 200), (384, 1), (511, 255)]


def sha(a: np.ndarray) -> str:
    return hashlib.sha256(np.ascontiguousarray(a).tobytes()).hexdigest()


def main():
    wl = workloads.WORKLOADS["tiny_fprop_mxfp8"]
    inp = workloads.make_inputs(wl)
    G, N, K, M = wl.G, wl.N, wl.K, wl.M
    ws, st = oracle.group_offsets(inp["sizes"].numpy(), 1, K, M)
    qx = oracle.mxfp8_quantize(inp["x"], M, M, rowwise=True, colwise=True)
    qw = oracle.mxfp8_quantize(inp["w"].reshape(G * N, K), G * N, G * N, rowwise=True)
    offs = oracle.live_rows(ws, G)
    a = {"q": qx["q_row"], "sf": qx["sf_row"]}
    b = {"q": qw["q_row"], "sf": qw["sf_row"]}
    rows = sorted({r for r, _ in SAMPLES})
    r_, c_, C = oracle.grouped_gemm_fprop("mxfp8", a, b, offs, N, K, sample_rows=rows)
    out = {
        "workload": "tiny_fprop_mxfp8",
        "source": "written by tests/golden/make_golden.py from oracle/ only",
        "offsets_workspace": [int(v) for v in ws],
        "status": st,
        "sha256": {k: sha(v) for k, v in {"x_q_row": qx["q_row"], "x_sf_row": qx["sf_row"],
                                          "x_q_col": qx["q_col"], "x_sf_col": qx["sf_col"],
                                          "w_q_row": qw["q_row"], "w_sf_row": qw["sf_row"]}.items()},
        "gemm_samples": [[r, c, float(C[rows.index(r), c])] for r, c in SAMPLES],
    }
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_fprop_mxfp8.json")
    with open(path, "w") as f:
        json.dump(out, f, indent=1)
    print("wrote", path)


if __name__ == "__main__":
    main()
