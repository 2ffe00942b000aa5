"""Benchmark of the grouped quantize + grouped GEMM hot path.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl mxg|reference]
                    [--config mixtral_fprop_mxfp8|finegrained_fprop_mxfp8|wgrad_mxfp8|
                              rowscaled_fprop_nvfp4|wgrad_nvfp4|dgrad_mxfp8|...]
                    [--configs a,b,c] [--out bf16|f32]

One step is one pass of the whole path over one batch of synthetic input:
  fprop:  group offsets -> quantize X (MXFP8 rowwise + transposed colwise, or
          row-scaled NVFP4) -> quantize W (rowwise) -> grouped GEMM fprop
  wgrad:  group offsets -> quantize X and dY (colwise, transposed) ->
          grouped GEMM wgrad
The metric is grouped quant+GEMM TFLOP/s: 2*M*N*K algorithmic FLOP of the
GEMM over the time of the whole step, with the inputs resident in HBM.  Each
step is timed with CUDA events on the launching stream; L2 is flushed (a
512 MB write, then a read of it that evicts the dirty lines) before every
timed step, outside its events.  "e2e" repeats the
measurement through the same C-ABI calls with the inputs copied from pinned
host memory and the output copied back inside the timed region.

The headline line is the Mixtral-shaped fprop workload; on one GPU the other
workloads of the metric (--configs: fine-grained fprop, wgrad, row-scaled
NVFP4 fprop by default) are timed after it the same way and reported under
"configs", each with its per-kernel times, GEMM roofline and the oracle's
timing.

For N > 1 (torchrun) every rank runs an independent replica on its own GPU
and its own seeded batch (the path has no exchange step); the job value is the
FLOP of all ranks over the slowest rank's time.  ``--impl reference`` times
the CPU oracle (the only other implementation there is) on rank 0 only, each
step a fixed sample of the workload -- the sample this arm's cpu_baseline
times too.
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
# measured after the headline workload and reported under "configs"
EXTRA_CONFIGS = ("finegrained_fprop_mxfp8", "wgrad_mxfp8", "rowscaled_fprop_nvfp4")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ----------------------------------------------------------------------------- helpers
def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


GEMM_SOURCES = ("gemm.cu", "mxg_device.cuh", "mxg_host.h", "tmap.cu")

# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum, bytes) of one
# full-size GEMM launch per workload, from single-pass ncu captures of
#   ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum,gpu__time_duration.sum
#       --clock-control none -k regex:grouped_gemm -s 3 -c 1
#       python bench.py --config <workload> --steps 1 --warmup 3 --no-cpu-baseline --no-e2e
#       --configs ''
# taken on the GEMM sources and compile flags whose digest is "digest"; after
# any change to either, "traffic" is reported as null until the counters are
# taken again.
GEMM_DRAM_TRAFFIC = {
    "digest": "1457bd49de8be5761559e8f027fd391cf64eebe741d6c9be4bf97ebb11fb867e",
    "bytes": {
        "mixtral_fprop_mxfp8": 1010531072,
        "finegrained_fprop_mxfp8": 263889408,
        "wgrad_mxfp8": 1227288064,
        "rowscaled_fprop_nvfp4": 339469056,
        "wgrad_nvfp4": 1063350272,
        "dgrad_mxfp8": 1373057536,
        "mixtral_fprop_mxfp8_unaligned": 999637760,
    },
}


def code_only(text: str) -> str:
    """C/C++ source without its comments and with runs of whitespace folded, so
    that an edit of comments alone leaves the digest below unchanged."""
    import re
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def gemm_source_digest() -> str:
    """sha256 over the GEMM kernel's sources (code only, in a fixed order) and
    the nvcc flags the library is built with: a DRAM traffic figure is
    reported only while the kernel it was measured on is unchanged."""
    import hashlib
    from moe_grouped_block_gb300 import build as mxg_build
    h = hashlib.sha256()
    for f in GEMM_SOURCES:
        with open(os.path.join(ROOT, "moe_grouped_block_gb300", "csrc", f)) as fh:
            h.update(code_only(fh.read()).encode())
    # include paths relative to the repository, so that a checkout elsewhere
    # (another machine) gives the same digest
    flags = [("-I" + os.path.relpath(f[2:], ROOT)) if f.startswith("-I") else f
             for f in mxg_build.ARCH + mxg_build.NVCC_FLAGS]
    h.update(" ".join(flags).encode())
    return h.hexdigest()


def measured_traffic(workload: str, table=None):
    """DRAM bytes (read + write) of one GEMM launch of this workload, or None
    if none was measured or the kernel changed since."""
    table = GEMM_DRAM_TRAFFIC if table is None else table
    if table.get("digest") != gemm_source_digest():
        return None
    return table.get("bytes", {}).get(workload)


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


class L2Flush:
    """Empties L2 between timed steps: a 512 MB write (four times L2) evicts
    everything a step could reuse, then a read of the same buffer evicts the
    write's dirty lines (written back here, outside the timed region), so the
    next step starts with no reusable and no dirty lines and each kernel pays
    for its own traffic only."""

    def __init__(self, dev, nbytes: int = 512 * 1024 * 1024):
        import torch
        self.buf = torch.empty(nbytes // 4, dtype=torch.float32, device=dev)
        self.sink = torch.empty(1, dtype=torch.float32, device=dev)

    def __call__(self):
        import torch
        self.buf.fill_(1.0)
        torch.amax(self.buf, dim=0, keepdim=True, out=self.sink)


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
        flush()
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
                                "launch (GEMM_DRAM_TRAFFIC in bench.py); null when the kernel "
                                "changed since",
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


def time_path(path, args, steps, dist, dev, flush, stream):
    """Warm-up, one CUDA graph per stage, then `steps` timed steps with CUDA
    events around every stage's replay on `stream` (L2 flushed before each
    step, outside the events).  Returns per-stage times, step times, the
    number of library kernels launched in the timed region, the timing note
    and the clock record of the timed region."""
    import torch
    from moe_grouped_block_gb300 import mxg
    stages = path.stages()
    for _ in range(args.warmup):
        flush()
        for _, fn in stages:
            fn()
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

    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in stages] for _ in range(steps)]
    uuid = getattr(torch.cuda.get_device_properties(dev), "uuid", None)
    clocks = ClockSampler(dev.index or 0, str(uuid) if uuid is not None else None)
    clocks.start()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    launches0 = mxg.mxg_launch_count()
    t_wall = time.perf_counter()
    for s in range(steps):
        flush()
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
    launches = (graph_launches * steps if graphs is not None
                else mxg.mxg_launch_count() - launches0)
    clk = clocks.stop()
    if int(path.status.item()) != 0:
        raise RuntimeError("device status %d" % int(path.status.item()))
    per_kernel = {name: [ev[s][i][0].elapsed_time(ev[s][i][1]) for s in range(steps)]
                  for i, (name, _) in enumerate(stages)}
    step_ms = [ev[s][0][0].elapsed_time(ev[s][-1][1]) for s in range(steps)]
    timing = graph_note or ("CUDA events around CUDA-graph replays (one graph per kernel)"
                            if graphs is not None else "CUDA events around eager launches")
    return {"stages": stages, "per_kernel": per_kernel, "step_ms": step_ms,
            "launches": int(launches), "timing": timing, "clocks": clk, "wall_s": t_wall}


def kernel_table(path, wl, per_kernel, peaks):
    """Per-stage mean ms, algorithmic GB/s and HBM fraction (and TFLOP/s for
    the GEMM), and the GEMM's roofline object."""
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
    return kernels, gemm_name, gemm_ms


def run_mxg(args, wl, ws_world, rank, local):
    import torch
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    dist = None
    if ws_world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    path = Path(wl, args.out == "bf16", dev, rank=rank, epilogue=args.epilogue)
    stream = torch.cuda.current_stream()
    flush = L2Flush(dev)
    peaks, peak_src = load_peaks()

    # ---- timed region: K steps, per-step and per-kernel CUDA events
    r = time_path(path, args, args.steps, dist, dev, flush, stream)
    stages = r["stages"]
    ms = max_over_ranks(float(np.mean(r["step_ms"])), dist, dev)
    ms_median = max_over_ranks(float(np.median(r["step_ms"])), dist, dev)

    def step():
        for _, fn in stages:
            fn()

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

    flops = wl.flops()
    kernels, gemm_name, gemm_ms = kernel_table(path, wl, r["per_kernel"], peaks)
    roofline = gemm_roofline(gemm_name, flops, path.kernel_bytes(gemm_name), gemm_ms, peaks,
                             peak_src, wl.fmt == "nvfp4", measured_traffic(wl.name))
    value = job_tflops(flops, ws_world, ms)
    nvfp4 = wl.fmt == "nvfp4"
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
                   "l2": "flushed before every timed step (512 MB write, then a read of it that "
                         "evicts the dirty lines); inputs also exceed L2",
                   "timing": r["timing"],
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
        "gpu_launches": r["launches"],
        "clocks": r["clocks"],
        "wall_s_timed_region": round(r["wall_s"], 4),
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, path.host)
    del path

    # ---- the other workloads of the same metric, one GPU only
    extra = [c for c in args.configs.split(",") if c and c != wl.name]
    if ws_world == 1 and extra:
        from moe_grouped_block_gb300 import workloads
        out = {}
        for name in extra:
            ewl = workloads.WORKLOADS[name]
            epath = Path(ewl, args.out == "bf16", dev)
            er = time_path(epath, args, min(args.steps, 20), None, dev, flush, stream)
            ek, egn, egms = kernel_table(epath, ewl, er["per_kernel"], peaks)
            eroof = gemm_roofline(egn, ewl.flops(), epath.kernel_bytes(egn), egms, peaks,
                                  peak_src, ewl.fmt == "nvfp4", measured_traffic(ewl.name))
            ems = float(np.mean(er["step_ms"]))
            d = {"value": round(ewl.flops() / (ems * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
                 "ms_per_step": round(ems, 5), "steps": len(er["step_ms"]),
                 "config": {"G": ewl.G, "K": ewl.K, "N": ewl.N, "M": ewl.M, "mode": ewl.mode,
                            "fmt": ewl.fmt, "step": " -> ".join(n for n, _ in er["stages"])},
                 "roofline": eroof, "kernels": ek, "gpu_launches": er["launches"],
                 "clocks": er["clocks"]}
            if not args.no_cpu_baseline:
                d["cpu_baseline"] = cpu_baseline(ewl, epath.host, full=True, single_core=False)
            out[name] = d
            del epath
            torch.cuda.empty_cache()
        line["configs"] = out
    if dist:
        dist.destroy_process_group()
    return line


# ----------------------------------------------------------------------------- oracle timing
# The oracle is timed on a fixed sample of the workload, the same in the
# reference arm and in this arm's cpu_baseline: every expert's live rows and
# the first eighth of its output columns (rounded up to 128), with the full
# contraction.  A pass quantizes the sample's operands as the GPU step does
# (offsets, activations / dY, weights) and runs the fp64 grouped GEMM.
ORACLE_COL_FRAC = 1.0 / 8.0
SINGLE_CORE_ROW_FRAC = 1.0 / 4.0  # the single-core figure takes a quarter of those rows


def _ceil128(v: float) -> int:
    return max(128, int(-(-int(np.ceil(v)) // 128)) * 128)


def oracle_sample(wl, inp, row_frac: float = 1.0, col_frac: float = ORACLE_COL_FRAC):
    """The sample's inputs: per expert the first ceil128(row_frac * M_g) of
    its rows (at most M_g, rounded down to 128 for groups of any size) and the
    first ceil128(col_frac * out) output columns.  Returns a dict of CPU
    tensors with the sample's group sizes."""
    import torch
    G, N, K = wl.G, wl.N, wl.K
    sizes = inp["sizes"].numpy().astype(np.int64)
    if wl.sizes == "dirichlet_rows":  # timing only: whole 128-row blocks of each group
        sizes = sizes // 128 * 128
    offs = np.concatenate([[0], np.cumsum(sizes)])
    rows = []
    new_sizes = []
    for g in range(G):
        r = min(int(sizes[g]), _ceil128(row_frac * sizes[g])) if sizes[g] else 0
        r = r // 128 * 128
        rows.append(np.arange(offs[g], offs[g] + r))
        new_sizes.append(r)
    rows = np.concatenate(rows).astype(np.int64) if rows else np.zeros(0, np.int64)
    rsel = torch.from_numpy(rows)
    out = {"sizes": np.asarray(new_sizes, np.int64)}
    out_cols = K if wl.mode == "dgrad" else N
    c = min(out_cols, _ceil128(col_frac * out_cols))
    out["cols"] = c
    if wl.mode == "fprop":
        out["x"] = inp["x"][rsel].contiguous()
        out["w"] = inp["w"][:, :c].contiguous()             # [G, c, K]
    elif wl.mode == "wgrad":
        out["x"] = inp["x"][rsel].contiguous()               # [m, K]
        out["dy"] = inp["dy"][rsel][:, :c].contiguous()      # [m, c]
    else:
        out["dy"] = inp["dy"][rsel].contiguous()             # [m, N]
        out["w"] = inp["w"][:, :, :c].contiguous()           # [G, N, c]
    return out


def oracle_pass(wl, smp):
    """One pass of the path through the oracle on a sample from
    oracle_sample.  Returns (seconds, algorithmic GEMM FLOP of the sample)."""
    import oracle
    G, N, K = wl.G, wl.N, wl.K
    sizes, c = smp["sizes"], smp["cols"]
    m = int(sizes.sum())
    t0 = time.perf_counter()
    ws, _ = oracle.group_offsets(sizes, 1, K if wl.mode != "dgrad" else N, max(m, 128))
    offs = oracle.live_rows(ws, G)
    if m == 0:
        return time.perf_counter() - t0, 0.0
    if wl.mode == "fprop":
        wq = smp["w"].reshape(G * c, K)
        if wl.fmt == "mxfp8":
            qa = oracle.mxfp8_quantize(smp["x"], m, m, rowwise=True, colwise=True)
            qb = oracle.mxfp8_quantize(wq, G * c, G * c)
            a = {"q": qa["q_row"], "sf": qa["sf_row"]}
            b = {"q": qb["q_row"], "sf": qb["sf_row"]}
        else:
            qa = oracle.nvfp4_quantize(smp["x"], m, m)
            qb = oracle.nvfp4_quantize(wq, G * c, G * c)
            a = {"q": qa["q_row"], "sf": qa["sf_row"], "outer": qa["outer_row"]}
            b = {"q": qb["q_row"], "sf": qb["sf_row"], "outer": qb["outer_row"]}
        oracle.grouped_gemm_fprop(wl.fmt, a, b, offs, c, K)
        flop = 2.0 * m * c * K
    elif wl.mode == "wgrad":
        if wl.fmt == "mxfp8":
            qx = oracle.mxfp8_quantize(smp["x"], m, m, rowwise=False, colwise=True)
            qd = oracle.mxfp8_quantize(smp["dy"], m, m, rowwise=False, colwise=True)
            a = {"q": qd["q_col"], "sf": qd["sf_col"]}
            b = {"q": qx["q_col"], "sf": qx["sf_col"]}
        else:
            qx = oracle.nvfp4_quantize_colwise(smp["x"], offs, m)
            qd = oracle.nvfp4_quantize_colwise(smp["dy"], offs, m)
            a = {"q": qd["q_col"], "sf": qd["sf_col"], "outer": qd["outer_col"]}
            b = {"q": qx["q_col"], "sf": qx["sf_col"], "outer": qx["outer_col"]}
        oracle.grouped_gemm_wgrad(a, b, offs, m, c, K, fmt=wl.fmt)
        flop = 2.0 * m * c * K
    else:
        qd = oracle.mxfp8_quantize(smp["dy"], m, m, rowwise=True)
        wq = smp["w"].reshape(G * N, c)
        qwt = oracle.mxfp8_quantize(wq, G * N, G * N, rowwise=False, colwise=True)
        oracle.grouped_gemm_dgrad({"q": qd["q_row"], "sf": qd["sf_row"]},
                                  {"q": qwt["q_col"], "sf": qwt["sf_col"]}, offs, G, N, c)
        flop = 2.0 * m * N * c
    return time.perf_counter() - t0, flop


def _sample_text(wl, smp, row_frac):
    out_cols = wl.K if wl.mode == "dgrad" else wl.N
    rows = ("every live row of each expert" if row_frac >= 1 else
            "the first %g of each expert's live rows" % row_frac)
    return ("%s x the first %d of %d output columns, full contraction: offsets, "
            "quantize of both operands and the fp64 grouped GEMM (%d sample rows)"
            % (rows, smp["cols"], out_cols, int(smp["sizes"].sum())))


def _single_core_main(path: str) -> None:
    """Child process of the single-core timing: the sample is read from
    `path` (saved by single_core_pass) and run with one thread."""
    import torch
    from moe_grouped_block_gb300 import workloads
    d = torch.load(path, weights_only=False)
    wl = workloads.WORKLOADS[d["workload"]]
    t, f = oracle_pass(wl, d["sample"])
    print(json.dumps({"seconds": t, "flop": f}))


def single_core_pass(wl, smp):
    """The oracle pass on `smp` in a child process limited to one thread
    (OpenMP and BLAS).  Returns (seconds, FLOP) or None if it failed."""
    import tempfile
    import torch
    with tempfile.TemporaryDirectory() as d:
        f = os.path.join(d, "sample.pt")
        torch.save({"workload": wl.name, "sample": smp}, f)
        env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1",
                   MKL_NUM_THREADS="1", OMP_DYNAMIC="false")
        r = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-single-core", f],
                           env=env, capture_output=True, text=True, timeout=600)
    if r.returncode != 0:
        return None
    out = json.loads(r.stdout.strip().splitlines()[-1])
    return out["seconds"], out["flop"]


def cpu_baseline(wl, inp, full: bool = True, single_core: bool = True):
    """The oracle on the host cores: the shared sample (the line's value), the
    whole workload once (full), and a quarter of the sample's rows on one
    thread (single_core)."""
    import oracle
    oracle.build()
    smp = oracle_sample(wl, inp)
    oracle_pass(wl, smp)  # first touch of the libraries
    t, f = oracle_pass(wl, smp)
    out = {"value": round(f / t / 1e12, 6), "unit": "TFLOP/s", "cores": os.cpu_count(),
           "kind": "oracle", "seconds": round(t, 3), "sample": _sample_text(wl, smp, 1.0),
           "same_sample_as": "bench.py --impl reference (one step)"}
    if full:
        fs = oracle_sample(wl, inp, 1.0, 1.0)
        tf, ff = oracle_pass(wl, fs)
        out["full"] = {"value": round(ff / tf / 1e12, 6), "seconds": round(tf, 3),
                       "sample": "the whole workload: " + _sample_text(wl, fs, 1.0)}
    if single_core:
        s1 = oracle_sample(wl, inp, SINGLE_CORE_ROW_FRAC)
        r = single_core_pass(wl, s1)
        if r is not None:
            out["single_core"] = {"value": round(r[1] / r[0] / 1e12, 6), "cores": 1,
                                  "seconds": round(r[0], 3),
                                  "sample": _sample_text(wl, s1, SINGLE_CORE_ROW_FRAC)}
    return out


def run_reference(args, wl, ws_world, rank):
    if rank != 0:
        return None
    import oracle
    from moe_grouped_block_gb300 import workloads
    oracle.build()
    inp = workloads.make_inputs(wl)
    smp = oracle_sample(wl, inp)  # the sample the other arm's cpu_baseline times
    for _ in range(args.warmup):
        oracle_pass(wl, smp)
    times, flops = [], []
    for _ in range(args.steps):
        t, f = oracle_pass(wl, smp)
        times.append(t)
        flops.append(f)
    value = sum(flops) / sum(times) / 1e12
    sample = _sample_text(wl, smp, 1.0)
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
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer measurement")
    ap.add_argument("--no-graph", action="store_true",
                    help="time eager launches instead of CUDA-graph replays")
    ap.add_argument("--M", type=int, default=0, help="override live rows (profiling runs)")
    ap.add_argument("--N", type=int, default=0, help="override N (profiling runs)")
    ap.add_argument("--K", type=int, default=0, help="override K (profiling runs)")
    ap.add_argument("--configs", default=",".join(EXTRA_CONFIGS),
                    help="other workloads measured after the headline one (1 GPU; '' for none)")
    ap.add_argument("--oracle-single-core", default=None, help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.oracle_single_core:
        _single_core_main(args.oracle_single_core)
        return
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
