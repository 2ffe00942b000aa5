"""Seeded synthetic inputs for the grouped quantize + grouped GEMM path.

This module draws random numbers and nothing else: it holds none of the
method's arithmetic, so the CUDA path and the test oracle can both take their
inputs from it.  Every tensor is drawn in fp32 with
``numpy.random.Generator(PCG64(seed))`` and rounded to bf16 (round to nearest
even) by torch.

Workloads (shapes of the MoE layers the pages build for: Mixtral-style 8-expert
FFN, fine-grained 64-expert FFN, the wgrad of the first, and a row-scaled NVFP4
32-expert layer):

==========================  ===  ====  =====  =====  ===========================
name                         G    K     N      M      group sizes / data
==========================  ===  ====  =====  =====  ===========================
tiny_fprop_mxfp8             4   256   256    512    [128, 0, 256, 128]; seed 0
mixtral_fprop_mxfp8          8   4096  14336  16384  Dirichlet(1) multinomial
finegrained_fprop_mxfp8      64  2048  1408   32768  Zipf(1.2), >= 1 empty group,
                                                     0.1% of X scaled x100
wgrad_mxfp8                  8   4096  14336  16384  Dirichlet(1); dY ~ N(0, 1e-3)
rowscaled_fprop_nvfp4        32  7168  2048   16384  Dirichlet(1); X Student-t(3)
wgrad_nvfp4                  8   4096  14336  16384  Dirichlet(1); row-scaled NVFP4
dgrad_mxfp8                  8   4096  14336  16384  Dirichlet(1); dX = dY W_g
mixtral_fprop_mxfp8_unal.    8   4096  14336  16384  Dirichlet(1) over rows: sizes
                                                     of any value (not x128)
==========================  ===  ====  =====  =====  ===========================

Group sizes are ``128 * Multinomial(M / 128, p)``: they sum to M exactly and
are multiples of 128, as the 128-row alignment of the grouped quantize and
grouped GEMM requires -- except ``dirichlet_rows``, ``Multinomial(M, p)``, for
the entry points that take groups of any size.  X ~ N(0, 1), W ~ N(0, 0.02)
and dY ~ N(0, 1e-3) unless stated.
"""
from __future__ import annotations

import dataclasses
from dataclasses import dataclass

import numpy as np


@dataclass(frozen=True)
class Workload:
    name: str
    mode: str          # "fprop", "dgrad" (ragged rows) or "wgrad" (ragged contraction)
    fmt: str           # "mxfp8" or "nvfp4"
    G: int
    K: int
    N: int
    M: int             # live rows (sum of group sizes)
    seed: int
    sizes: str         # "fixed" | "dirichlet" | "zipf" | "dirichlet_rows"
    fixed_sizes: tuple = ()
    x_dist: str = "normal"       # "normal" | "normal_outliers" | "student_t3"
    dy_std: float = 1e-3
    w_std: float = 0.02
    M_cap: int = 0     # buffer rows (>= M); 0 means M

    @property
    def rows_capacity(self) -> int:
        return self.M_cap if self.M_cap else self.M

    def flops(self) -> float:
        return 2.0 * self.M * self.N * self.K

    def scaled(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    "tiny_fprop_mxfp8": Workload("tiny_fprop_mxfp8", "fprop", "mxfp8", 4, 256, 256, 512, 0,
                                 "fixed", (128, 0, 256, 128)),
    "mixtral_fprop_mxfp8": Workload("mixtral_fprop_mxfp8", "fprop", "mxfp8", 8, 4096, 14336,
                                    16384, 1, "dirichlet"),
    "finegrained_fprop_mxfp8": Workload("finegrained_fprop_mxfp8", "fprop", "mxfp8", 64, 2048,
                                        1408, 32768, 2, "zipf", x_dist="normal_outliers"),
    "wgrad_mxfp8": Workload("wgrad_mxfp8", "wgrad", "mxfp8", 8, 4096, 14336, 16384, 3,
                            "dirichlet"),
    "rowscaled_fprop_nvfp4": Workload("rowscaled_fprop_nvfp4", "fprop", "nvfp4", 32, 7168, 2048,
                                      16384, 4, "dirichlet", x_dist="student_t3"),
    "wgrad_nvfp4": Workload("wgrad_nvfp4", "wgrad", "nvfp4", 8, 4096, 14336, 16384, 5,
                            "dirichlet"),
    "dgrad_mxfp8": Workload("dgrad_mxfp8", "dgrad", "mxfp8", 8, 4096, 14336, 16384, 6,
                            "dirichlet"),
    "mixtral_fprop_mxfp8_unaligned": Workload("mixtral_fprop_mxfp8_unaligned", "fprop", "mxfp8",
                                              8, 4096, 14336, 16384, 7, "dirichlet_rows"),
}


def _rng(seed: int, stream: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64([seed, stream]))


def group_sizes(w: Workload) -> np.ndarray:
    """int32 [G] row counts summing to w.M: multiples of 128, or of any value
    for ``dirichlet_rows``."""
    if w.sizes == "fixed":
        s = np.asarray(w.fixed_sizes, np.int64)
        assert s.size == w.G and s.sum() == w.M
        return s.astype(np.int32)
    rng = _rng(w.seed, 0)
    if w.sizes == "dirichlet_rows":
        return rng.multinomial(w.M, rng.dirichlet(np.ones(w.G))).astype(np.int32)
    units = w.M // 128
    if w.sizes == "dirichlet":
        p = rng.dirichlet(np.ones(w.G))
    elif w.sizes == "zipf":
        ranks = np.arange(1, w.G + 1, dtype=np.float64)
        p_sorted = ranks ** -1.2
        p_sorted /= p_sorted.sum()
        p = p_sorted[rng.permutation(w.G)]
    else:
        raise ValueError(w.sizes)
    counts = rng.multinomial(units, p)
    return (counts * 128).astype(np.int32)


def _bf16(a32: np.ndarray):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a32, dtype=np.float32)).to(torch.bfloat16)


def _activations(w: Workload, rng: np.random.Generator, rows: int, cols: int) -> np.ndarray:
    if w.x_dist == "normal":
        return rng.standard_normal((rows, cols), dtype=np.float32)
    if w.x_dist == "normal_outliers":
        x = rng.standard_normal((rows, cols), dtype=np.float32)
        n_out = max(1, int(round(0.001 * rows * cols)))
        idx = rng.choice(rows * cols, size=n_out, replace=False)
        x.reshape(-1)[idx] *= 100.0
        return x
    if w.x_dist == "student_t3":
        return rng.standard_t(3, size=(rows, cols)).astype(np.float32)
    raise ValueError(w.x_dist)


def make_inputs(w: Workload) -> dict:
    """CPU torch tensors for one batch of ``w``.

    fprop: ``x`` bf16 [M_cap, K], ``w`` bf16 [G, N, K], ``sizes`` int32 [G].
    wgrad: ``x`` bf16 [M_cap, K], ``dy`` bf16 [M_cap, N], ``sizes`` int32 [G].
    dgrad: ``dy`` bf16 [M_cap, N], ``w`` bf16 [G, N, K], ``sizes`` int32 [G].
    Rows >= M of ``x`` / ``dy`` are filled with draws as well (they are never
    read by the path; tests use them to check that).
    """
    import torch
    sizes = group_sizes(w)
    R = w.rows_capacity
    out = {"sizes": torch.from_numpy(sizes.copy())}
    if w.mode != "dgrad":
        out["x"] = _bf16(_activations(w, _rng(w.seed, 1), R, w.K))
    if w.mode in ("fprop", "dgrad"):
        wr = _rng(w.seed, 2)
        out["w"] = _bf16(wr.standard_normal((w.G, w.N, w.K), dtype=np.float32) * w.w_std)
    if w.mode in ("wgrad", "dgrad"):
        dr = _rng(w.seed, 3)
        out["dy"] = _bf16(dr.standard_normal((R, w.N), dtype=np.float32) * w.dy_std)
    return out


def random_bf16(shape, seed: int, scale: float = 1.0, dist: str = "normal"):
    """Generic seeded bf16 tensor (for edge-case tests)."""
    rng = _rng(seed, 7)
    if dist == "normal":
        a = rng.standard_normal(shape, dtype=np.float32) * scale
    elif dist == "uniform":
        a = (rng.random(shape, dtype=np.float32) * 2 - 1) * scale
    elif dist == "student_t3":
        a = rng.standard_t(3, size=shape).astype(np.float32) * scale
    else:
        raise ValueError(dist)
    return _bf16(a)
