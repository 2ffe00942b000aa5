"""Benchmark of the grouped quantize + grouped GEMM hot path.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl mxg|reference]
                    [--config mixtral_fprop_mxfp8|finegrained_fprop_mxfp8|wgrad_mxfp8|
                              rowscaled_fprop_nvfp4|tiny_fprop_mxfp8] [--out bf16|f32]

One step is one pass of the whole path over one batch of synthetic input:
  fprop:  group offsets -> quantize X (MXFP8 rowwise + transposed colwise, or
          row-scaled NVFP4) -> quantize W (rowwise) -> grouped GEMM fprop
  wgrad:  group offsets -> quantize X and dY (MXFP8 colwise, transposed) ->
          grouped GEMM wgrad
The metric is grouped quant+GEMM TFLOP/s: 2*M*N*K algorithmic FLOP of the
GEMM over the time of the whole step, with the inputs resident in HBM.  Each
step is timed with CUDA events on the launching stream; L2 is flushed (a
512 MB write) before every timed step, outside its events.  "e2e" repeats the
measurement through the same C-ABI calls with the inputs copied from pinned
host memory and the output copied back inside the timed region.

For N > 1 (torchrun) every rank runs an independent replica on its own GPU
and its own seeded batch (the path has no exchange step); the job value is the
FLOP of all ranks over the slowest rank's time.  ``--impl reference`` times
the CPU oracle (the only other implementation there is) on a bounded sample
of the same workload, on rank 0 only.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "grouped quant+GEMM TFLOP/s (frac of dense MXFP8 peak); quantize HBM GB/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ----------------------------------------------------------------------------- helpers
def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


GEMM_SOURCES = ("gemm.cu", "mxg_device.cuh", "mxg_host.h", "tmap.cu")
TRAFFIC_SUMMARY = os.path.join(ROOT, "profiles", "grouped_gemm_pair_kernel_dram_traffic.md")


def code_only(text: str) -> str:
    """C/C++ source without its comments and with runs of whitespace folded, so
    that an edit of comments alone leaves the digest below unchanged."""
    import re
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def gemm_source_digest() -> str:
    """sha256 over the GEMM kernel's sources (code only, in a fixed order): a
    DRAM traffic figure is reported only while the kernel it was measured on is
    unchanged."""
    import hashlib
    h = hashlib.sha256()
    for f in GEMM_SOURCES:
        with open(os.path.join(ROOT, "moe_grouped_block_gb300", "csrc", f)) as fh:
            h.update(code_only(fh.read()).encode())
    return h.hexdigest()


def measured_traffic(workload: str):
    """DRAM bytes (read + write) of one GEMM launch of this workload, from the
    committed ncu summary, or None if there is none or the sources changed
    since it was taken.  The summary's table rows read
    `| workload | kernel | read bytes | write bytes | traffic bytes | ... |` and
    it carries a line `sources sha256: <hex>`."""
    if not os.path.exists(TRAFFIC_SUMMARY):
        return None
    text = open(TRAFFIC_SUMMARY).read()
    digest = None
    for line in text.splitlines():
        if line.startswith("sources sha256:"):
            digest = line.split(":", 1)[1].strip().strip("`")
    if digest != gemm_source_digest():
        return None
    for line in text.splitlines():
        cells = [c.strip().strip("`") for c in line.strip().strip("|").split("|")]
        if len(cells) >= 5 and cells[0] == workload:
            try:
                return int(cells[4])
            except ValueError:
                return None
    return None


def max_over_ranks(value: float, dist=None, device=None) -> float:
    """MAX of a per-rank scalar over all ranks (identity without a group)."""
    if dist is None or not dist.is_initialized():
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_workload(wl, rank: int):
    """Each rank runs an independent replica on its own seeded batch."""
    return wl if rank == 0 else wl.scaled(seed=wl.seed + 1000 * rank)


def job_tflops(flop_per_rank: float, world: int, ms_max: float) -> float:
    """Whole-job throughput: the FLOP of all ranks over the slowest rank's time."""
    return world * flop_per_rank / (ms_max * 1e-3) / 1e12


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


class ClockSampler:
    """SM clock and clock-event reasons during the timed region.  Reads NVML
    (the driver's libnvidia-ml, through ctypes) every millisecond on a thread
    between start() and stop(); the device is found by the CUDA device's UUID.
    Without NVML it falls back to nvidia-smi every 200 ms.  Read-only: no
    setting of the GPU is changed."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    # nvmlClocksEventReason* bits
    REASON_BITS = {"sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20,
                   "hw_thermal_slowdown": 0x40, "hw_power_brake_slowdown": 0x80}

    def __init__(self, gpu_index: int, uuid=None):
        self.idx = gpu_index
        self.uuid = uuid
        self.proc = None
        self.lines = []
        self.nvml = None
        self.samples = []
        self.running = False

    def _nvml_handle(self):
        import ctypes
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
        except OSError:
            return None
        if lib.nvmlInit_v2() != 0:
            return None
        h = ctypes.c_void_p()
        ok = False
        if self.uuid:
            ok = lib.nvmlDeviceGetHandleByUUID(("GPU-%s" % self.uuid).encode(), ctypes.byref(h)) == 0
        if not ok:
            ok = lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(self.idx), ctypes.byref(h)) == 0
        if not ok:
            return None
        reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons")
        return lib, h, reasons_fn

    def _poll(self):
        import ctypes
        lib, h, reasons_fn = self.nvml
        clk, mx, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        while self.running:
            if (lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0 and   # NVML_CLOCK_SM
                    lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0 and
                    reasons_fn(h, ctypes.byref(rs)) == 0):
                self.samples.append((clk.value, mx.value, rs.value))
            time.sleep(0.001)

    def start(self):
        try:
            self.nvml = self._nvml_handle()
        except (OSError, AttributeError):
            self.nvml = None
        if self.nvml is not None:
            self.running = True
            self.t = threading.Thread(target=self._poll, daemon=True)
            self.t.start()
            return
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            time.sleep(0.3)
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.nvml is not None:
            self.running = False
            self.t.join(timeout=2)
            sm = [c for c, _, _ in self.samples]
            reasons = {n for _, _, r in self.samples for n, b in self.REASON_BITS.items() if r & b}
            return {"sm_mhz": statistics.median(sm) if sm else None,
                    "sm_max_mhz": max(m for _, m, _ in self.samples) if self.samples else None,
                    "reasons": sorted(reasons), "samples": len(sm), "source": "nvml, 1 ms"}
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.t.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm), "source": "nvidia-smi, 200 ms"}


# ----------------------------------------------------------------------------- the path
class Path:
    """Device buffers and the C-ABI calls of one step."""

    def __init__(self, wl, out_bf16: bool, dev, rank: int = 0, epilogue: str = "none",
                 inputs=None):
        import torch
        from moe_grouped_block_gb300 import mxg, workloads
        self.mxg, self.torch = mxg, torch
        self.wl = wl
        self.dev = dev
        inp = inputs if inputs is not None else workloads.make_inputs(replica_workload(wl, rank))
        self.host = inp
        G, N, K, R = wl.G, wl.N, wl.K, wl.rows_capacity
        self.G, self.N, self.K, self.R = G, N, K, R
        self.unaligned = wl.sizes == "dirichlet_rows"
        self.sizes = inp["sizes"].to(dev)
        self.ws = mxg.alloc_offsets(G, dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.out_type = mxg.MXG_OUT_BF16 if out_bf16 else mxg.MXG_OUT_F32
        cdt = torch.bfloat16 if out_bf16 else torch.float32
        # per-group bias and alpha in the GEMM epilogue (fprop only)
        self.bias = self.alpha = None
        if epilogue == "bias_alpha":
            g = torch.Generator().manual_seed(wl.seed)
            self.bias = torch.randn((G, N), generator=g).float().to(dev)
            self.alpha = (0.5 + torch.rand(G, generator=g)).float().to(dev)
        if wl.mode == "fprop":
            self.x = inp["x"].to(dev)
            self.w = inp["w"].to(dev).reshape(G * N, K)
            if self.unaligned:
                self.qx = mxg.alloc_mxfp8_unaligned(R, K, G, rowwise=True, colwise=True, device=dev)
                self.qw = mxg.alloc_mxfp8(G * N, K, device=dev)
            elif wl.fmt == "mxfp8":
                self.qx = mxg.alloc_mxfp8(R, K, rowwise=True, colwise=True, device=dev)
                self.qw = mxg.alloc_mxfp8(G * N, K, device=dev)
            else:
                self.qx = mxg.alloc_nvfp4(R, K, device=dev)
                self.qw = mxg.alloc_nvfp4(G * N, K, device=dev)
            self.C = torch.empty((R, N), dtype=cdt, device=dev)
        elif wl.mode == "dgrad":
            self.dy = inp["dy"].to(dev)
            self.w = inp["w"].to(dev).reshape(G * N, K)
            self.qd = mxg.alloc_mxfp8(R, N, device=dev)
            self.qwt = mxg.alloc_mxfp8(G * N, K, rowwise=False, colwise=True, device=dev)
            self.C = torch.empty((R, K), dtype=cdt, device=dev)
        else:
            self.x = inp["x"].to(dev)
            self.dy = inp["dy"].to(dev)
            if wl.fmt == "mxfp8":
                self.qx = mxg.alloc_mxfp8(R, K, rowwise=False, colwise=True, device=dev)
                self.qd = mxg.alloc_mxfp8(R, N, rowwise=False, colwise=True, device=dev)
            else:
                self.qx = mxg.alloc_nvfp4(R, K, device=dev, rowwise=False, colwise=True, G=G)
                self.qd = mxg.alloc_nvfp4(R, N, device=dev, rowwise=False, colwise=True, G=G)
            self.C = torch.empty((G, N, K), dtype=cdt, device=dev)

    # each stage returns nothing; all work is enqueued on the current stream
    def stages(self):
        m, wl = self.mxg, self.wl
        G, N, K, R = self.G, self.N, self.K, self.R
        out = []
        if self.unaligned:
            out.append(("group_offsets", lambda: m.mxg_group_offsets_unaligned(
                self.sizes, 1, K, R, self.ws, self.status)))
        else:
            out.append(("group_offsets", lambda: m.mxg_group_offsets(
                self.sizes, 1, N if wl.mode == "dgrad" else K, R, self.ws, self.status)))
        if self.unaligned:
            q = self.qx
            out.append(("quantize_x_mxfp8_both", lambda: m.mxg_group_quantize_unaligned(
                m.MXG_BOTH, self.x, R, K, self.ws, G, q["q_row"], q["sf_row"], q["q_col"],
                q["sf_col"], self.status)))
            out.append(("quantize_w_mxfp8_row", lambda: m.mxg_group_quantize(
                m.MXG_MXFP8_E4M3, m.MXG_ROWWISE, self.w, G * N, K, None, G, self.qw["q_row"],
                self.qw["sf_row"], None, None, None, self.status)))
            out.append(("grouped_gemm_fprop_mxfp8", lambda: m.mxg_grouped_gemm_unaligned(
                m.MXG_FPROP_TN, (q["q_row"], q["sf_row"]), (self.qw["q_row"], self.qw["sf_row"]),
                self.ws, G, R, N, K, alpha=self.alpha, C=self.C, out_type=self.out_type,
                dev_status=self.status, bias=self.bias)))
        elif wl.mode == "dgrad":
            out.append(("quantize_dy_mxfp8_row", lambda: m.mxg_group_quantize(
                m.MXG_MXFP8_E4M3, m.MXG_ROWWISE, self.dy, R, N, self.ws, G, self.qd["q_row"],
                self.qd["sf_row"], None, None, None, self.status)))
            out.append(("quantize_w_mxfp8_col", lambda: m.mxg_group_quantize(
                m.MXG_MXFP8_E4M3, m.MXG_COLWISE, self.w, G * N, K, None, G, None, None,
                self.qwt["q_col"], self.qwt["sf_col"], None, self.status)))
            out.append(("grouped_gemm_dgrad_mxfp8", lambda: m.mxg_grouped_gemm(
                m.MXG_MXFP8_E4M3, m.MXG_DGRAD_NN, (self.qd["q_row"], self.qd["sf_row"], None),
                (self.qwt["q_col"], self.qwt["sf_col"], None), self.ws, G, R, N, K, C=self.C,
                out_type=self.out_type, dev_status=self.status)))
        elif wl.mode == "wgrad" and wl.fmt == "nvfp4":
            qx, qd = self.qx, self.qd
            out.append(("quantize_x_nvfp4_col", lambda: m.mxg_group_quantize(
                m.MXG_NVFP4_ROWSCALED, m.MXG_COLWISE, self.x, R, K, self.ws, G, None, None,
                qx["q_col"], qx["sf_col"], None, self.status, outer_col=qx["outer_col"])))
            out.append(("quantize_dy_nvfp4_col", lambda: m.mxg_group_quantize(
                m.MXG_NVFP4_ROWSCALED, m.MXG_COLWISE, self.dy, R, N, self.ws, G, None, None,
                qd["q_col"], qd["sf_col"], None, self.status, outer_col=qd["outer_col"])))
            out.append(("grouped_gemm_wgrad_nvfp4", lambda: m.mxg_grouped_gemm(
                m.MXG_NVFP4_ROWSCALED, m.MXG_WGRAD_NT, (qd["q_col"], qd["sf_col"], qd["outer_col"]),
                (qx["q_col"], qx["sf_col"], qx["outer_col"]), self.ws, G, R, N, K, C=self.C,
                out_type=self.out_type, dev_status=self.status)))
        elif wl.mode == "fprop" and wl.fmt == "mxfp8":
            q = self.qx
            out.append(("quantize_x_mxfp8_both", lambda: m.mxg_group_quantize(
                m.MXG_MXFP8_E4M3, m.MXG_BOTH, self.x, R, K, self.ws, G, q["q_row"], q["sf_row"],
                q["q_col"], q["sf_col"], None, self.status)))
            out.append(("quantize_w_mxfp8_row", lambda: m.mxg_group_quantize(
                m.MXG_MXFP8_E4M3, m.MXG_ROWWISE, self.w, G * N, K, None, G, self.qw["q_row"],
                self.qw["sf_row"], None, None, None, self.status)))
            out.append(("grouped_gemm_fprop_mxfp8", lambda: m.mxg_grouped_gemm(
                m.MXG_MXFP8_E4M3, m.MXG_FPROP_TN, (q["q_row"], q["sf_row"], None),
                (self.qw["q_row"], self.qw["sf_row"], None), self.ws, G, R, N, K,
                alpha=self.alpha, C=self.C, out_type=self.out_type, dev_status=self.status,
                bias=self.bias)))
        elif wl.mode == "fprop":
            q, qw = self.qx, self.qw
            out.append(("quantize_x_nvfp4", lambda: m.mxg_group_quantize(
                m.MXG_NVFP4_ROWSCALED, m.MXG_ROWWISE, self.x, R, K, self.ws, G, q["q_row"],
                q["sf_row"], None, None, q["outer_row"], self.status)))
            out.append(("quantize_w_nvfp4", lambda: m.mxg_group_quantize(
                m.MXG_NVFP4_ROWSCALED, m.MXG_ROWWISE, self.w, G * N, K, None, G, qw["q_row"],
                qw["sf_row"], None, None, qw["outer_row"], self.status)))
            out.append(("grouped_gemm_fprop_nvfp4", lambda: m.mxg_grouped_gemm(
                m.MXG_NVFP4_ROWSCALED, m.MXG_FPROP_TN, (q["q_row"], q["sf_row"], q["outer_row"]),
                (qw["q_row"], qw["sf_row"], qw["outer_row"]), self.ws, G, R, N, K, C=self.C,
                out_type=self.out_type, dev_status=self.status)))
        else:
            out.append(("quantize_x_mxfp8_col", lambda: m.mxg_group_quantize(
                m.MXG_MXFP8_E4M3, m.MXG_COLWISE, self.x, R, K, self.ws, G, None, None,
                self.qx["q_col"], self.qx["sf_col"], None, self.status)))
            out.append(("quantize_dy_mxfp8_col", lambda: m.mxg_group_quantize(
                m.MXG_MXFP8_E4M3, m.MXG_COLWISE, self.dy, R, N, self.ws, G, None, None,
                self.qd["q_col"], self.qd["sf_col"], None, self.status)))
            out.append(("grouped_gemm_wgrad_mxfp8", lambda: m.mxg_grouped_gemm(
                m.MXG_MXFP8_E4M3, m.MXG_WGRAD_NT, (self.qd["q_col"], self.qd["sf_col"], None),
                (self.qx["q_col"], self.qx["sf_col"], None), self.ws, G, R, N, K, C=self.C,
                out_type=self.out_type, dev_status=self.status)))
        return out

    def kernel_bytes(self, name: str) -> float:
        """Algorithmic HBM bytes of one launch (inputs read once, outputs
        written once; the GEMM's are reported too though it is tensor-bound)."""
        wl, G, N, K, R = self.wl, self.G, self.N, self.K, self.R
        M = wl.M
        obytes = self.C.element_size()
        if name == "group_offsets":
            return 4 * G + 8 * (2 * G + 1)
        if name == "quantize_x_mxfp8_both":
            return M * K * (2 + 2 + 2 / 32)
        if name == "quantize_w_mxfp8_row":
            return G * N * K * (2 + 1 + 1 / 32)
        if name == "quantize_x_nvfp4":
            return M * K * (2 + 0.5 + 1 / 16) + 4 * M
        if name == "quantize_w_nvfp4":
            return G * N * K * (2 + 0.5 + 1 / 16) + 4 * G * N
        if name == "quantize_x_mxfp8_col":
            return M * K * (2 + 1 + 1 / 32)
        if name == "quantize_dy_mxfp8_col":
            return M * N * (2 + 1 + 1 / 32)
        if name == "quantize_dy_mxfp8_row":
            return M * N * (2 + 1 + 1 / 32)
        if name == "quantize_w_mxfp8_col":
            return G * N * K * (2 + 1 + 1 / 32)
        if name == "quantize_x_nvfp4_col":  # + the [G, K] outer scales
            return M * K * (2 + 0.5 + 1 / 16) + 4 * G * K
        if name == "quantize_dy_nvfp4_col":
            return M * N * (2 + 0.5 + 1 / 16) + 4 * G * N
        sizes = self.host["sizes"].numpy()
        live_experts = int((sizes > 0).sum())
        extra = 0 if self.bias is None else 4 * G * (N + 1)
        if name == "grouped_gemm_fprop_mxfp8":
            return (M * K * (1 + 1 / 32) + live_experts * N * K * (1 + 1 / 32) + M * N * obytes
                    + extra)
        if name == "grouped_gemm_dgrad_mxfp8":
            return M * N * (1 + 1 / 32) + live_experts * N * K * (1 + 1 / 32) + M * K * obytes
        if name == "grouped_gemm_wgrad_nvfp4":
            return (N + K) * M * (0.5 + 1 / 16) + 4 * G * (N + K) + G * N * K * obytes
        if name == "grouped_gemm_fprop_nvfp4":
            return (M * K * (0.5 + 1 / 16) + live_experts * N * K * (0.5 + 1 / 16) + M * N * obytes
                    + 4 * (M + live_experts * N))
        if name == "grouped_gemm_wgrad_mxfp8":
            return (N + K) * M * (1 + 1 / 32) + G * N * K * obytes
        return 0.0

    def input_tensors(self):
        if self.wl.mode == "fprop":
            return [("sizes", self.sizes), ("x", self.x), ("w", self.w)]
        if self.wl.mode == "dgrad":
            return [("sizes", self.sizes), ("dy", self.dy), ("w", self.w)]
        return [("sizes", self.sizes), ("x", self.x), ("dy", self.dy)]


def measure_e2e(path, step, args, dist, dev, flush, stream):
    """The step through the same C-ABI calls with host buffers: every step
    copies its inputs from pinned host memory to the device and its output
    back, inside the timed region.  Returns (ms per step, H2D bytes, D2H bytes)."""
    import torch
    host_in = [(n, t.cpu().pin_memory()) for n, t in path.input_tensors()]
    host_out = torch.empty(path.C.shape, dtype=path.C.dtype).pin_memory()
    dev_in = dict(path.input_tensors())
    h2d = sum(t.numel() * t.element_size() for _, t in host_in)
    d2h = host_out.numel() * host_out.element_size()

    def e2e_step():
        for n, t in host_in:
            dev_in[n].copy_(t, non_blocking=True)
        step()
        host_out.copy_(path.C, non_blocking=True)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    if dist:
        dist.barrier()
    for e0, e1 in ev:
        flush.fill_(1.0)
        e0.record(stream)
        e2e_step()
        e1.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(float(np.mean([a.elapsed_time(b) for a, b in ev])), dist, dev)
    return ms, h2d, d2h


def measure_e2e_pipelined(paths, args, dist, dev):
    """End to end with host buffers, two buffer sets in flight: every step
    copies its inputs from pinned host memory (copy stream), runs the C-ABI
    calls (compute stream) and copies its output back (a third stream); step
    i + 1's input copies overlap step i's compute and output copy, which run
    on the other direction of the link.  Returns ms per step in steady state
    (K steps between a start event before the first copy and an end event
    after the last output copy)."""
    import torch
    host_in = [(n, t.cpu().pin_memory()) for n, t in paths[0].input_tensors()]
    host_out = [torch.empty(p.C.shape, dtype=p.C.dtype).pin_memory() for p in paths]
    dev_in = [dict(p.input_tensors()) for p in paths]
    stages = [p.stages() for p in paths]
    sh, sc, sd = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in paths]
    ev_comp = [torch.cuda.Event() for _ in paths]
    ev_out = [torch.cuda.Event() for _ in paths]

    def issue(i):
        b = i % 2
        if i >= 2:
            sh.wait_event(ev_comp[b])  # set b's inputs are no longer read
        with torch.cuda.stream(sh):
            for n, t in host_in:
                dev_in[b][n].copy_(t, non_blocking=True)
            ev_in[b].record(sh)
        sc.wait_event(ev_in[b])
        if i >= 2:
            sc.wait_event(ev_out[b])  # set b's output has been copied out
        with torch.cuda.stream(sc):
            for _, fn in stages[b]:
                fn()
            ev_comp[b].record(sc)
        sd.wait_event(ev_comp[b])
        with torch.cuda.stream(sd):
            host_out[b].copy_(paths[b].C, non_blocking=True)
            ev_out[b].record(sd)

    for i in range(2):
        issue(i)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(sh)
    for i in range(args.steps):
        issue(i)
    t1.record(sd)
    torch.cuda.synchronize()
    ms = max_over_ranks(t0.elapsed_time(t1) / args.steps, dist, dev)
    # both buffer sets computed the same step: their outputs agree bit for bit
    if not torch.equal(host_out[0], host_out[1]):
        raise RuntimeError("the two e2e buffer sets disagree")
    for p in paths:
        if int(p.status.item()) != 0:
            raise RuntimeError("device status %d in the e2e run" % int(p.status.item()))
    return ms


def gemm_roofline(gemm_name, flops, gemm_bytes, gemm_ms, peaks, peak_src, nvfp4, traffic):
    """The roofline object of the GEMM launch.  Its roofline time is the larger
    of its algorithmic FLOP at the dense tensor peak (measured bf16 x 2 for
    MXFP8, x 6 for NVFP4: the nominal ratios) and its algorithmic bytes at the
    measured HBM bandwidth; that one names the bound (HBM for the row-scaled
    NVFP4 layer, tensor for the others) and sets achieved / peak / frac."""
    peak_tc = peaks["bf16_tflops"] * (6.0 if nvfp4 else 2.0)
    tflops = flops / (gemm_ms * 1e-3) / 1e12
    t_tensor_ms = flops / (peak_tc * 1e12) * 1e3
    t_hbm_ms = gemm_bytes / (peaks["hbm_gbs"] * 1e9) * 1e3
    common = {"kernel": gemm_name,
              "peak_source": "%s bf16_tflops (burst) x %d; %s hbm_gbs" % (
                  peak_src, 6 if nvfp4 else 2, peak_src),
              "traffic": traffic,
              "traffic_source": "ncu dram__bytes_read.sum + dram__bytes_write.sum of one full-size "
                                "launch (profiles/grouped_gemm_pair_kernel_dram_traffic.md); "
                                "null when the kernel changed since",
              "algorithmic_bytes": gemm_bytes, "algorithmic_flop": flops,
              "t_tensor_roofline_ms": round(t_tensor_ms, 5), "t_hbm_roofline_ms": round(t_hbm_ms, 5),
              "t_roofline_over_t": round(max(t_tensor_ms, t_hbm_ms) / gemm_ms, 4)}
    if t_hbm_ms > t_tensor_ms:
        gbs = gemm_bytes / (gemm_ms * 1e-3) / 1e9
        return {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": round(gbs / peaks["hbm_gbs"], 4),
                "tflops": round(tflops, 1), "tflops_frac": round(tflops / peak_tc, 4), **common}
    return {"bound": "tensor", "achieved": round(tflops, 1), "peak": round(peak_tc, 1),
            "unit": "TFLOP/s", "frac": round(tflops / peak_tc, 4), **common}


def run_mxg(args, wl, ws_world, rank, local):
    import torch
    from moe_grouped_block_gb300 import mxg
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    dist = None
    if ws_world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    path = Path(wl, args.out == "bf16", dev, rank=rank, epilogue=args.epilogue)
    stages = path.stages()
    stream = torch.cuda.current_stream()
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)

    def step():
        for _, fn in stages:
            fn()

    for _ in range(args.warmup):
        flush.fill_(1.0)
        step()
    torch.cuda.synchronize()
    if int(path.status.item()) != 0:
        raise RuntimeError("device status %d after warm-up" % int(path.status.item()))

    # one CUDA graph per stage, captured after the warm-up: the timed steps
    # replay them with CUDA events around each replay on this stream
    graphs, graph_note, graph_launches = None, None, 0
    if not args.no_graph:
        try:
            n0 = mxg.mxg_launch_count()
            graphs = []
            for _, fn in stages:
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g):
                    fn()
                graphs.append(g)
            graph_launches = mxg.mxg_launch_count() - n0  # kernels one replay of all stages runs
            for g in graphs:
                g.replay()
            torch.cuda.synchronize()
            if int(path.status.item()) != 0:
                raise RuntimeError("device status %d after graph replay" % int(path.status.item()))
        except Exception as e:  # capture unavailable: time eager launches instead
            graphs, graph_note = None, "graph capture failed (%s); eager launches timed" % e
            torch.cuda.synchronize()

    # ---- timed region: K steps, per-step and per-kernel CUDA events
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in stages] for _ in range(args.steps)]
    uuid = getattr(torch.cuda.get_device_properties(dev), "uuid", None)
    clocks = ClockSampler(local, str(uuid) if uuid is not None else None)
    clocks.start()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    launches0 = mxg.mxg_launch_count()
    t_wall = time.perf_counter()
    for s in range(args.steps):
        flush.fill_(1.0)
        for i, ((name, fn), (e0, e1)) in enumerate(zip(stages, ev[s])):
            e0.record(stream)
            if graphs is not None:
                graphs[i].replay()
            else:
                fn()
            e1.record(stream)
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall
    if dist:
        dist.barrier()
    # graph replays do not pass through the C ABI: count what one capture launched
    launches = (graph_launches * args.steps if graphs is not None
                else mxg.mxg_launch_count() - launches0)
    clk = clocks.stop()
    per_kernel = {name: [ev[s][i][0].elapsed_time(ev[s][i][1]) for s in range(args.steps)]
                  for i, (name, _) in enumerate(stages)}
    step_ms = [ev[s][0][0].elapsed_time(ev[s][-1][1]) for s in range(args.steps)]
    ms = max_over_ranks(float(np.mean(step_ms)), dist, dev)
    ms_median = max_over_ranks(float(np.median(step_ms)), dist, dev)
    if int(path.status.item()) != 0:
        raise RuntimeError("device status %d" % int(path.status.item()))

    # ---- e2e: host buffers, copies inside the timed region
    e2e_ms, h2d, d2h = (None, 0, 0) if args.no_e2e else measure_e2e(path, step, args, dist, dev,
                                                                      flush, stream)
    e2e_pipe_ms = None
    if not args.no_e2e:
        path2 = Path(wl, args.out == "bf16", dev, rank=rank, epilogue=args.epilogue,
                     inputs=path.host)
        if path.bias is not None:  # the same epilogue operands in both sets
            path2.bias.copy_(path.bias)
            path2.alpha.copy_(path.alpha)
        e2e_pipe_ms = measure_e2e_pipelined([path, path2], args, dist, dev)
        del path2

    peaks, peak_src = load_peaks()
    flops = wl.flops()
    kernels = {}
    for name, times in per_kernel.items():
        t = float(np.mean(times))
        d = {"ms": round(t, 5)}
        b = path.kernel_bytes(name)
        if b:
            d["GB/s"] = round(b / (t * 1e-3) / 1e9, 1)
            d["hbm_frac"] = round(b / (t * 1e-3) / 1e9 / peaks["hbm_gbs"], 4)
        if name.startswith("grouped_gemm"):
            d["TFLOP/s"] = round(flops / (t * 1e-3) / 1e12, 1)
        kernels[name] = d
    gemm_name = [n for n in per_kernel if n.startswith("grouped_gemm")][0]
    gemm_ms = float(np.mean(per_kernel[gemm_name]))
    nvfp4 = wl.fmt == "nvfp4"
    roofline = gemm_roofline(gemm_name, flops, path.kernel_bytes(gemm_name), gemm_ms, peaks,
                             peak_src, nvfp4, measured_traffic(wl.name))
    value = job_tflops(flops, ws_world, ms)
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": ws_world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 5),
        "ms_per_step_median": round(ms_median, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "nvfp4(e2m1/ue4m3)->f32" if nvfp4 else "mxfp8(e4m3/e8m0)->f32",
        "data": "synthetic (seeded; shapes and distributions of the workload)",
        "config": {"workload": wl.name, "G": wl.G, "K": wl.K, "N": wl.N, "M": wl.M,
                   "mode": wl.mode, "out": args.out, "epilogue": args.epilogue,
                   "step": " -> ".join(n for n, _ in stages),
                   "l2": "flushed before every timed step (512 MB write); inputs also exceed L2",
                   "timing": graph_note or ("CUDA events around CUDA-graph replays (one graph per "
                                            "kernel)" if graphs is not None else
                                            "CUDA events around eager launches"),
                   "parallelism": "replicas" if ws_world > 1 else "single GPU"},
        "roofline": roofline,
        "kernels": kernels,
        "e2e": None if e2e_ms is None else {
            "value": round(job_tflops(flops, ws_world, e2e_pipe_ms), 2), "unit": "TFLOP/s",
            "ms_per_step": round(e2e_pipe_ms, 4), "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h,
            "note": "same C-ABI calls; every step copies its inputs from pinned host memory and its "
                    "output back inside the timed region, with two buffer sets so that step i+1's "
                    "input copies overlap step i's compute and output copy (steady state over K "
                    "steps)",
            "serial": {"value": round(job_tflops(flops, ws_world, e2e_ms), 2),
                       "ms_per_step": round(e2e_ms, 4),
                       "note": "copy in, compute, copy out, one step at a time"}},
        "gpu_launches": int(launches),
        "clocks": clk,
        "wall_s_timed_region": round(t_wall, 4),
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, budget_s=args.cpu_budget)
    if dist:
        dist.destroy_process_group()
    return line


# ----------------------------------------------------------------------------- oracle timing
def _oracle_sample(wl, rows_per_group: int, cols_per_group: int):
    """One bounded sample of the workload through the oracle: quantize the
    sampled activation rows and weight rows, then the fp64 GEMM on them.
    Returns (seconds, algorithmic GEMM FLOP of the sample)."""
    import torch
    import oracle
    from moe_grouped_block_gb300 import workloads
    inp = workloads.make_inputs(wl) if not hasattr(wl, "_cached") else wl._cached
    sizes = inp["sizes"].numpy()
    G, N, K = wl.G, wl.N, wl.K
    flop = 0.0
    t0 = time.perf_counter()
    ws, _ = (oracle.group_offsets_unaligned if wl.sizes == "dirichlet_rows" else
             oracle.group_offsets)(sizes, 1, K, wl.rows_capacity)
    offs = oracle.live_rows(ws, G)
    for g in range(G):
        lo, hi = int(offs[g]), int(offs[g + 1])
        if hi == lo:
            continue
        r = min(rows_per_group, hi - lo)
        r128 = max(128, (r + 127) // 128 * 128)
        lo2 = min(lo, hi - r128) if hi - lo >= r128 else lo
        c128 = max(128, min(N, (cols_per_group + 127) // 128 * 128))
        if wl.mode == "fprop":
            xs = inp["x"][lo2:lo2 + r128]
            wsub = inp["w"][g, :c128]
            if wl.fmt == "mxfp8":
                qa = oracle.mxfp8_quantize(xs, r128, r128, rowwise=True, colwise=True)
                qb = oracle.mxfp8_quantize(wsub, c128, c128)
                a = {"q": qa["q_row"], "sf": qa["sf_row"]}
                b = {"q": qb["q_row"], "sf": qb["sf_row"]}
            else:
                qa = oracle.nvfp4_quantize(xs, r128, r128)
                qb = oracle.nvfp4_quantize(wsub, c128, c128)
                a = {"q": qa["q_row"], "sf": qa["sf_row"], "outer": qa["outer_row"]}
                b = {"q": qb["q_row"], "sf": qb["sf_row"], "outer": qb["outer_row"]}
            oracle.grouped_gemm_fprop(wl.fmt, a, b, [0, r128], c128, K)
            flop += 2.0 * r128 * c128 * K
        elif wl.mode == "dgrad":
            ds = inp["dy"][lo2:lo2 + r128]
            wsub = inp["w"][g, :, :c128].contiguous()  # [N, c128]: the sample's K columns
            qd = oracle.mxfp8_quantize(ds, r128, r128, rowwise=True)
            qwt = oracle.mxfp8_quantize(wsub, N, N, rowwise=False, colwise=True)
            oracle.grouped_gemm_dgrad({"q": qd["q_row"], "sf": qd["sf_row"]},
                                      {"q": qwt["q_col"], "sf": qwt["sf_col"]}, [0, r128], 1,
                                      N, c128)
            flop += 2.0 * r128 * N * c128
        else:
            xs = inp["x"][lo2:lo2 + r128]
            ds = inp["dy"][lo2:lo2 + r128, :c128].contiguous()
            kk = min(K, c128)
            if wl.fmt == "mxfp8":
                qx = oracle.mxfp8_quantize(xs, r128, r128, rowwise=False, colwise=True)
                qd = oracle.mxfp8_quantize(ds, r128, r128, rowwise=False, colwise=True)
                a = {"q": qd["q_col"], "sf": qd["sf_col"]}
                b = {"q": qx["q_col"], "sf": qx["sf_col"]}
            else:
                qx = oracle.nvfp4_quantize_colwise(xs, [0, r128], r128)
                qd = oracle.nvfp4_quantize_colwise(ds, [0, r128], r128)
                a = {"q": qd["q_col"], "sf": qd["sf_col"], "outer": qd["outer_col"]}
                b = {"q": qx["q_col"], "sf": qx["sf_col"], "outer": qx["outer_col"]}
            oracle.grouped_gemm_wgrad(a, b, [0, r128], r128, c128, K, sample_k=np.arange(kk),
                                      fmt=wl.fmt)
            flop += 2.0 * r128 * c128 * kk
    return time.perf_counter() - t0, flop


def _size_sample(wl, budget_s: float):
    """Grow the per-expert sample (rows = weight rows = side) by doubling
    until one sample takes at least a quarter of the budget."""
    side = 128
    t, f = _oracle_sample(wl, side, side)
    while t < budget_s / 4 and side < max(wl.N, wl.K):
        side *= 2
        t, f = _oracle_sample(wl, side, side)
    return side, t, f


def cpu_baseline(wl, budget_s: float = 15.0):
    import oracle
    oracle.build()
    side, t, f = _size_sample(wl, budget_s)
    return {"value": round(f / t / 1e12, 6), "unit": "TFLOP/s", "cores": os.cpu_count(),
            "kind": "oracle", "seconds": round(t, 2),
            "sample": "per expert: up to %d activation rows x %d weight rows (full K=%d): "
                      "MXFP8/NVFP4 quantize of both operands + fp64 GEMM; throughput = "
                      "2*rows*cols*K of the sample / its time" % (side, min(side, wl.N), wl.K)}


def run_reference(args, wl, ws_world, rank):
    if rank != 0:
        return None
    import oracle
    oracle.build()
    # each step is a bounded sample; the whole run stays within a few minutes
    per_step_budget = max(1.0, min(20.0, 150.0 / max(1, args.steps + args.warmup)))
    side, _, _ = _size_sample(wl, per_step_budget)
    for _ in range(args.warmup):
        _oracle_sample(wl, side, side)
    times, flops = [], []
    for _ in range(args.steps):
        t, f = _oracle_sample(wl, side, side)
        times.append(t)
        flops.append(f)
    value = sum(flops) / sum(times) / 1e12
    sample = "per expert: %d activation rows x %d weight rows, full K=%d" % (side, side, wl.K)
    return {"metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": ws_world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * float(np.mean(times)), 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference",
            "config": {"workload": wl.name, "G": wl.G, "K": wl.K, "N": wl.N, "M": wl.M,
                       "mode": wl.mode},
            "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": os.cpu_count(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="mxg", choices=["mxg", "reference"])
    ap.add_argument("--config", default="mixtral_fprop_mxfp8")
    ap.add_argument("--out", default="bf16", choices=["bf16", "f32"])
    ap.add_argument("--epilogue", default="none", choices=["none", "bias_alpha"],
                    help="fprop: per-group bias and alpha in the GEMM epilogue")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer measurement")
    ap.add_argument("--no-graph", action="store_true",
                    help="time eager launches instead of CUDA-graph replays")
    ap.add_argument("--M", type=int, default=0, help="override live rows (profiling runs)")
    ap.add_argument("--N", type=int, default=0, help="override N (profiling runs)")
    ap.add_argument("--K", type=int, default=0, help="override K (profiling runs)")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "mxg":
        args.warmup = 3
    from moe_grouped_block_gb300 import workloads
    wl = workloads.WORKLOADS[args.config]
    over = {k: v for k, v in (("M", args.M), ("N", args.N), ("K", args.K)) if v}
    if over:
        wl = wl.scaled(name=wl.name + "_reduced", **over)
    ws_world, rank, local = dist_env()
    if args.impl == "reference":
        line = run_reference(args, wl, ws_world, rank)
    else:
        line = run_mxg(args, wl, ws_world, rank, local)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
