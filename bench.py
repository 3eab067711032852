#!/usr/bin/env python3
"""Benchmark of the fused MoE permute + grouped-matmul backward (d_x).

One step = one pass of the whole path on one batch: the routing preprocess
(groupList scan, row-block list, inverse index, ranks) and the persistent
grouped GEMM with the fused ordered scatter-add into FP32 d_x. Inputs are
seeded synthetic tensors already resident in HBM; L2 is flushed between
steps, outside the per-step CUDA events: a 256 MiB write, then a 256 MiB read
of another buffer, so that the write's dirty lines are written back before
the step starts rather than during it.

The default workload is large-bf16 (batch 13500, topK 8, G 60, K 7168,
N 2048: the scale of "MoeInitRoutingGroupedMatmulGrad design", section 1.2).
Before the warm-up, the same step runs untimed for --burn-in seconds so that
the GPU is at its steady clock; SM clocks and clock-event reasons are sampled
(NVML, read-only) during the burn-in and the timed region.

Metric: fused d_x TFLOP/s = 2*M*N*K / step time, with the roofline fraction
of the grouped-GEMM kernel (against the measured burst bf16 peak) and the
workspace bytes. Also reported: the median step, the same steps with L2
left warm, and the torch allocator's peak over the library calls (0: the
library allocates nothing).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--op dx|dw|fwd|unperm]
  python bench.py --impl reference ...   # the fp64 oracle on the host cores

--op dw times the companion weight-gradient kernel (x^T d_y per expert with
the x rows gathered by the routing) on the same workload instead; --op fwd
the forward y = expanded_x W per expert it differentiates; --op unperm the
probs-weighted unpermute backward.

Under torchrun (N > 1) every rank runs an independent replica of the same
workload on its own GPU (the path needs no exchange); value sums the work of
all ranks over the slowest rank's time.
"""

from __future__ import annotations

import argparse
import hashlib
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

DEFAULT_WORKLOAD = "large-bf16"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
METRIC = "fused d_x TFLOP/s (2*M*N*K/s) & % of roofline, 1xGB300; peak workspace bytes"
_COMMON = ["permute_grouped_gemm_gb300/csrc/pgg_ptx.cuh"]
# grouped-GEMM kernel -> the sources its ncu counters depend on
_GATHER = "permute_grouped_gemm_gb300/csrc/pgg_gather.cuh"
_EPILOGUE = "permute_grouped_gemm_gb300/csrc/pgg_epilogue.cuh"
KERNEL_SOURCES = {
    "gmm_dx_kernel": ["permute_grouped_gemm_gb300/csrc/gmm_dx.cu", _GATHER, *_COMMON],
    "gmm_dx_simt_kernel": ["permute_grouped_gemm_gb300/csrc/gmm_dx_simt.cu", *_COMMON],
    "gmm_dx_owner_kernel": ["permute_grouped_gemm_gb300/csrc/gmm_dx_owner.cu", *_COMMON],
    "unpermute_grad_kernel": ["permute_grouped_gemm_gb300/csrc/unpermute_grad.cu", *_COMMON],
    "gmm_dw_kernel": ["permute_grouped_gemm_gb300/csrc/gmm_dw.cu", _GATHER, _EPILOGUE,
                       *_COMMON],
    "gmm_dw_simt_kernel": ["permute_grouped_gemm_gb300/csrc/gmm_dw_simt.cu", *_COMMON],
    "gmm_fwd_kernel": ["permute_grouped_gemm_gb300/csrc/gmm_fwd.cu", _GATHER, _EPILOGUE,
                       *_COMMON],
    "gmm_fwd_simt_kernel": ["permute_grouped_gemm_gb300/csrc/gmm_fwd_simt.cu", *_COMMON],
}
SIMT_VARIANT = 3
OWNER_VARIANT = 4
FP32_LANES_PER_SM = 128    # FP32 fused multiply-add lanes per SM
NOMINAL_SM_MHZ = 2070.0    # maximum SM clock of the part


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--op", default="dx", choices=["dx", "dw", "fwd", "unperm"],
                    help="dx: the fused input gradient (default); dw: the weight gradient; "
                         "fwd: the forward; unperm: the probs-weighted unpermute backward")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="target CPU time of the oracle baseline sample")
    ap.add_argument("--burn-in", type=float, default=3.0,
                    help="seconds of untimed steps before the warm-up (0: none)")
    return ap.parse_args()


def dist_info():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(values, dist, device):
    """Element-wise maximum of ``values`` (floats) over all ranks of ``dist``
    (the slowest replica's times); the values themselves without one."""
    if dist is None:
        return [float(v) for v in values]
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def kernel_hash(kernel: str = "gmm_dx_kernel") -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per grouped-GEMM launch from the committed ncu summary, if it
    was taken on the current kernel source (matching hash), else None."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    vals = {}
    for line in text.splitlines():
        line = line.strip().strip("|").strip()
        for key in ("kernel_source_hash", "dram_bytes_per_launch"):
            if line.startswith(key + ":"):
                vals[key] = line.split(":", 1)[1].strip().split()[0]
    if vals.get("kernel_source_hash") != kernel_hash(kernel):
        return None
    try:
        return int(float(vals["dram_bytes_per_launch"]))
    except (KeyError, ValueError):
        return None


# Clock-event reason bits of NVML (nvmlClocksEventReason*) that a run reports.
_REASON_BITS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
                0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}


class _Nvml:
    """Read-only NVML queries through ctypes (SM clock, its maximum, the active
    clock-event reasons, board power) for the GPU behind a CUDA device index.
    Changes no setting of the GPU."""
    CLOCK_SM = 1

    def __init__(self, cuda_index: int):
        import ctypes
        self.ct = ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.lib = lib
        self.h = ctypes.c_void_p()
        try:
            import torch
            u = str(torch.cuda.get_device_properties(cuda_index).uuid)
            uuid = u if u.startswith("GPU-") else "GPU-" + u
        except Exception:  # noqa: BLE001 - fall back to the index
            uuid = None
        rc = 1
        if uuid:
            rc = lib.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(self.h))
        if rc != 0:
            rc = lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(cuda_index),
                                                   ctypes.byref(self.h))
        if rc != 0:
            raise OSError("no NVML handle for the device")
        self.reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None)
        if self.reasons_fn is None:
            self.reasons_fn = lib.nvmlDeviceGetCurrentClocksThrottleReasons
        v = ctypes.c_uint()
        self.max_mhz = (float(v.value) if lib.nvmlDeviceGetMaxClockInfo(
            self.h, self.CLOCK_SM, ctypes.byref(v)) == 0 else None)

    def sample(self):
        ct = self.ct
        mhz, mw, rs = ct.c_uint(), ct.c_uint(), ct.c_ulonglong()
        if self.lib.nvmlDeviceGetClockInfo(self.h, self.CLOCK_SM, ct.byref(mhz)) != 0:
            return None
        if self.reasons_fn(self.h, ct.byref(rs)) != 0:
            rs.value = 0
        watts = mw.value / 1000.0 if self.lib.nvmlDeviceGetPowerUsage(
            self.h, ct.byref(mw)) == 0 else None
        return float(mhz.value), self.max_mhz, int(rs.value), watts


class ClockSampler:
    """SM clock and clock-event reasons sampled from a thread, each sample
    stamped with the host clock, so that the samples inside any window (the
    timed region, the burn-in) can be summarised. NVML through ctypes every
    millisecond; nvidia-smi every 50 ms where NVML cannot be loaded."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int, period_s: float = 0.001):
        self.index = index
        self.period = period_s
        self.samples = []  # (host time, sm MHz, max MHz, reason names, power W)
        self.proc = None
        self.nvml = None
        self.source = "none"
        self._stop = threading.Event()
        self.t = None

    def __enter__(self):
        try:
            self.nvml = _Nvml(self.index)
            self.source = "nvml"
            self.t = threading.Thread(target=self._poll, daemon=True)
            self.t.start()
            return self
        except (OSError, AttributeError):
            self.nvml = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.source = "nvidia-smi"
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None
        return self

    def _poll(self):
        while not self._stop.is_set():
            s = self.nvml.sample()
            if s is not None:
                mhz, mx, bits, w = s
                names = tuple(n for b, n in _REASON_BITS.items() if bits & b)
                self.samples.append((time.perf_counter(), mhz, mx, names, w))
            self._stop.wait(self.period)

    def _read(self):
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.strip().split(",")]
            if len(parts) < 9:
                continue
            try:
                mhz, mx = float(parts[1]), float(parts[2])
            except ValueError:
                continue
            try:
                w = float(parts[3])
            except ValueError:
                w = None
            active = tuple(n for n, v in zip(names, parts[5:9]) if v.lower() == "active")
            self.samples.append((time.perf_counter(), mhz, mx, active, w))

    def __exit__(self, *exc):
        self._stop.set()
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.t is not None:
            self.t.join(timeout=2)

    def summary(self, t0=None, t1=None):
        """Median SM clock, maximum clock, the reasons seen and the sample count
        for the samples taken between host times t0 and t1 (all if None)."""
        sel = [s for s in self.samples
               if (t0 is None or s[0] >= t0) and (t1 is None or s[0] <= t1)]
        if not sel:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0,
                    "source": self.source}
        reasons = sorted({n for s in sel for n in s[3]})
        watts = [s[4] for s in sel if s[4] is not None]
        maxes = [s[2] for s in sel if s[2] is not None]
        return {"sm_mhz": statistics.median(s[1] for s in sel),
                "sm_max_mhz": max(maxes) if maxes else None,
                "reasons": reasons, "samples": len(sel),
                "power_w_max": max(watts) if watts else None, "source": self.source}


class DxOp:
    """d_x: the fused permute + grouped-matmul backward (the default)."""
    name = "dx"
    metric = METRIC

    def __init__(self, inp, pgg, dev):
        import torch
        self.inp, self.pgg = inp, pgg
        w = inp.workload
        self.dt = pgg.dtype_code(inp.grad_y.dtype)
        self.sizes = (w.M, w.N, w.K, w.G, w.M, w.batch, w.top_k)
        self.plan = pgg.pgg_dx_plan(*self.sizes, w.row_idx_type, self.dt)
        self.ws_bytes = pgg.pgg_dx_workspace_size(*self.sizes, w.row_idx_type, self.dt)
        self.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device=dev)
        self.out = torch.empty(w.batch, w.K, dtype=torch.float32, device=dev)
        v = self.plan["variant"]
        self.kernel = {SIMT_VARIANT: "gmm_dx_simt_kernel",
                       OWNER_VARIANT: "gmm_dx_owner_kernel"}.get(v, "gmm_dx_kernel")
        # routing step: scan, inverse, ranks (the owner kernel's slab bounds
        # in the same launch for topK <= 32, in a fourth above); grouped GEMM:
        # one kernel (+ the ticketed kernel after the owner kernel, which works
        # only when the rows are not sorted)
        if v == OWNER_VARIANT:
            self.launches = 5 if w.top_k <= 32 else 6
        else:
            self.launches = 4

    def values(self):
        return self.inp.grad_y, self.inp.weight

    def stage1(self, idx, gl, sp):
        w = self.inp.workload
        return self.pgg.pgg_dx_route_prep(idx.data_ptr(), gl.data_ptr(), *self.sizes,
                                          w.row_idx_type, self.dt, self.ws.data_ptr(),
                                          self.ws_bytes, sp)

    def stage2(self, a, b, idx, gl, out, sp):
        w = self.inp.workload
        return self.pgg.pgg_dx_grouped_gemm(a.data_ptr(), b.data_ptr(), idx.data_ptr(),
                                            gl.data_ptr(), *self.sizes, w.row_idx_type, self.dt,
                                            self.ws.data_ptr(), self.ws_bytes, out.data_ptr(), sp)

    def execute(self, a, b, idx, gl, out, sp):
        w = self.inp.workload
        return self.pgg.pgg_dx_execute(a.data_ptr(), b.data_ptr(), idx.data_ptr(), gl.data_ptr(),
                                       *self.sizes, w.row_idx_type, self.dt, self.ws.data_ptr(),
                                       self.ws_bytes, out.data_ptr(), sp)

    def algorithmic(self):
        """(flops, bytes) of one step: 2*M*N*K, and d_y once + weight of non-empty
        experts once + d_x written once + the two index arrays."""
        inp = self.inp
        w = inp.workload
        es = {"fp32": 4, "fp16": 2, "bf16": 2}[w.dtype]
        nonempty = int((inp.group_list > 0).sum())
        flops = 2 * w.M * w.N * w.K
        nbytes = (w.M * w.N * es + nonempty * w.K * w.N * es + w.batch * w.K * 4
                  + w.M * 8 + w.G * 8)
        return flops, nbytes

    def oracle_sample(self, host, rng, n):
        """Runs the oracle on n sampled units; returns the flops of the sample."""
        import oracle
        w = host.workload
        n = max(1, min(w.batch, n))
        toks = np.sort(rng.choice(w.batch, n, replace=False))
        oracle.dx(host.grad_y, host.weight, host.expanded_row_idx, host.group_list, w.batch,
                  w.top_k, w.row_idx_type, tokens=toks)
        return 2 * w.top_k * w.N * w.K * n, f"{n} of {w.batch} tokens (all topK rows each)"

    def units(self):
        return self.inp.workload.batch


class DwOp(DxOp):
    """d_weight: the companion weight-gradient grouped matmul."""
    name = "dw"
    metric = ("d_weight TFLOP/s (2*M*N*K/s) & % of roofline, 1xGB300: x^T d_y per expert, "
              "x rows gathered by routing")

    def __init__(self, inp, pgg, dev):
        import torch
        from workloads.moe import forward_input
        self.inp, self.pgg = inp, pgg
        w = inp.workload
        self.dt = pgg.dtype_code(inp.grad_y.dtype)
        self.sizes = (w.M, w.N, w.K, w.G, w.M, w.batch, w.top_k)
        self.plan = pgg.pgg_dw_plan(*self.sizes, w.row_idx_type, self.dt)
        self.ws_bytes = pgg.pgg_dw_workspace_size(*self.sizes, w.row_idx_type, self.dt)
        self.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device=dev)
        self.x = forward_input(inp, dev)
        self.out = torch.empty(w.G, w.K, w.N, dtype=inp.grad_y.dtype, device=dev)
        self.kernel = "gmm_dw_simt_kernel" if self.plan["variant"] == SIMT_VARIANT else "gmm_dw_kernel"

    def values(self):
        return self.x, self.inp.grad_y

    def stage2(self, a, b, idx, gl, out, sp):
        w = self.inp.workload
        return self.pgg.pgg_dw_grouped_gemm(a.data_ptr(), b.data_ptr(), idx.data_ptr(),
                                            gl.data_ptr(), *self.sizes, w.row_idx_type, self.dt,
                                            self.dt, self.ws.data_ptr(), self.ws_bytes,
                                            out.data_ptr(), sp)

    def execute(self, a, b, idx, gl, out, sp):
        w = self.inp.workload
        return self.pgg.pgg_dw_execute(a.data_ptr(), b.data_ptr(), idx.data_ptr(), gl.data_ptr(),
                                       *self.sizes, w.row_idx_type, self.dt, self.dt,
                                       self.ws.data_ptr(), self.ws_bytes, out.data_ptr(), sp)

    def algorithmic(self):
        """(flops, bytes): 2*M*N*K, and x once + d_y once + d_weight written once
        (input dtype) + the two index arrays."""
        w = self.inp.workload
        es = {"fp32": 4, "fp16": 2, "bf16": 2}[w.dtype]
        flops = 2 * w.M * w.N * w.K
        nbytes = (w.batch * w.K * es + w.M * w.N * es + w.G * w.K * w.N * es
                  + w.M * 8 + w.G * 8)
        return flops, nbytes

    def oracle_sample(self, host, rng, n):
        import oracle
        from workloads.moe import forward_input
        w = host.workload
        if not hasattr(self, "_host_x"):
            self._host_x = self.x.cpu()
        n = max(1, min(w.G * w.K, n))
        g = rng.integers(0, w.G, n)
        k = rng.integers(0, w.K, n)
        oracle.dw(self._host_x, host.grad_y, host.expanded_row_idx, host.group_list, w.batch,
                  w.top_k, w.row_idx_type, sel=(g, k))
        rows = host.group_list.numpy()[g]
        return int(2 * w.N * rows.sum()), f"{n} of {w.G * w.K} rows (g, k) of d_weight"

    def units(self):
        return self.inp.workload.G * self.inp.workload.K


class FwdOp(DxOp):
    """The forward y = GroupedMatmul(Permute(x), weight) these are the gradients of."""
    name = "fwd"
    metric = ("forward TFLOP/s (2*M*N*K/s) & % of roofline, 1xGB300: y = expanded_x W per expert, "
              "x rows gathered by routing")

    def __init__(self, inp, pgg, dev):
        import torch
        from workloads.moe import forward_input
        self.inp, self.pgg = inp, pgg
        w = inp.workload
        self.dt = pgg.dtype_code(inp.grad_y.dtype)
        self.sizes = (w.M, w.N, w.K, w.G, w.M, w.batch, w.top_k)
        self.plan = pgg.pgg_fwd_plan(*self.sizes, w.row_idx_type, self.dt)
        self.ws_bytes = pgg.pgg_fwd_workspace_size(*self.sizes, w.row_idx_type, self.dt)
        self.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device=dev)
        self.x = forward_input(inp, dev)
        self.out = torch.empty(w.M, w.N, dtype=inp.grad_y.dtype, device=dev)
        self.kernel = ("gmm_fwd_simt_kernel" if self.plan["variant"] == SIMT_VARIANT
                       else "gmm_fwd_kernel")

    def values(self):
        return self.x, self.inp.weight

    def stage1(self, idx, gl, sp):
        w = self.inp.workload
        return self.pgg.pgg_fwd_route_prep(idx.data_ptr(), gl.data_ptr(), *self.sizes,
                                           w.row_idx_type, self.dt, self.ws.data_ptr(),
                                           self.ws_bytes, sp)

    def stage2(self, a, b, idx, gl, out, sp):
        w = self.inp.workload
        return self.pgg.pgg_fwd_grouped_gemm(a.data_ptr(), b.data_ptr(), idx.data_ptr(),
                                             gl.data_ptr(), *self.sizes, w.row_idx_type, self.dt,
                                             self.dt, self.ws.data_ptr(), self.ws_bytes,
                                             out.data_ptr(), sp)

    def execute(self, a, b, idx, gl, out, sp):
        w = self.inp.workload
        return self.pgg.pgg_fwd_execute(a.data_ptr(), b.data_ptr(), idx.data_ptr(),
                                        gl.data_ptr(), *self.sizes, w.row_idx_type, self.dt,
                                        self.dt, self.ws.data_ptr(), self.ws_bytes,
                                        out.data_ptr(), sp)

    def algorithmic(self):
        """(flops, bytes): 2*M*N*K, and x once + weight of non-empty experts once +
        y written once (input dtype) + the two index arrays."""
        inp = self.inp
        w = inp.workload
        es = {"fp32": 4, "fp16": 2, "bf16": 2}[w.dtype]
        nonempty = int((inp.group_list > 0).sum())
        flops = 2 * w.M * w.N * w.K
        nbytes = (w.batch * w.K * es + nonempty * w.K * w.N * es + w.M * w.N * es
                  + w.M * 8 + w.G * 8)
        return flops, nbytes

    def oracle_sample(self, host, rng, n):
        import oracle
        w = host.workload
        if not hasattr(self, "_host_x"):
            self._host_x = self.x.cpu()
        n = max(1, min(w.M, n))
        rows = np.sort(rng.choice(w.M, n, replace=False))
        oracle.fwd(self._host_x, host.weight, host.expanded_row_idx, host.group_list, w.batch,
                   w.top_k, w.row_idx_type, rows=rows)
        return 2 * w.N * w.K * n, f"{n} of {w.M} rows of y"

    def units(self):
        return self.inp.workload.M


class UnpermOp(DxOp):
    """The probs-weighted unpermute backward (perm_grad and probs_grad)."""
    name = "unperm"
    metric = ("probs-weighted unpermute backward GB/s (algorithmic bytes / s) & % of HBM roofline, "
              "1xGB300")
    unit = "GB/s"

    def __init__(self, inp, pgg, dev):
        import torch
        from workloads.moe import unpermute_inputs
        self.inp, self.pgg = inp, pgg
        w = inp.workload
        self.dt = pgg.dtype_code(inp.grad_y.dtype)
        self.sizes = (w.M, w.N, w.batch, w.top_k)
        self.plan = {"variant": 0, "threads": 256, "ctas_per_token": 1}
        self.ws_bytes = pgg.pgg_unpermute_grad_workspace_size(w.M, w.batch, w.top_k)
        self.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device=dev)
        self.d_out, self.probs = unpermute_inputs(inp, dev)
        self.out = torch.empty(w.M, w.N, dtype=inp.grad_y.dtype, device=dev)
        self.qg = torch.empty(w.batch, w.top_k, dtype=inp.grad_y.dtype, device=dev)
        self.kernel = "unpermute_grad_kernel"

    def values(self):
        return self.inp.grad_y, self.d_out

    def stage1(self, idx, gl, sp):
        # index validation and inverse map (timed as route_prep)
        w = self.inp.workload
        return self.pgg.pgg_unpermute_grad_prep(idx.data_ptr(), w.M, w.batch, w.top_k,
                                                w.row_idx_type, self.ws.data_ptr(), self.ws_bytes,
                                                sp)

    def stage2(self, a, b, idx, gl, out, sp):
        # the unpermute kernel alone (timed as grouped_gemm: the roofline's kernel)
        w = self.inp.workload
        return self.pgg.pgg_unpermute_grad_apply(a.data_ptr(), b.data_ptr(),
                                                 self.probs.data_ptr(), idx.data_ptr(), w.M, w.N,
                                                 w.batch, w.top_k, w.row_idx_type, self.dt,
                                                 self.dt, self.ws.data_ptr(), self.ws_bytes,
                                                 out.data_ptr(), self.qg.data_ptr(), sp)

    def execute(self, a, b, idx, gl, out, sp):
        # the one call a user makes (prep + apply)
        w = self.inp.workload
        return self.pgg.pgg_unpermute_grad(a.data_ptr(), b.data_ptr(), self.probs.data_ptr(),
                                           idx.data_ptr(), w.M, w.N, w.batch, w.top_k,
                                           w.row_idx_type, self.dt, self.dt, self.ws.data_ptr(),
                                           self.ws_bytes, out.data_ptr(), self.qg.data_ptr(), sp)

    def algorithmic(self):
        """(flops, bytes): 3*M*N (scale + dot); bytes: d_out once, permuted once,
        perm_grad written once, probs and probs_grad, the index."""
        w = self.inp.workload
        es = {"fp32": 4, "fp16": 2, "bf16": 2}[w.dtype]
        flops = 3 * w.M * w.N
        nbytes = (w.batch * w.N * es + 2 * w.M * w.N * es + 2 * w.M * es + w.M * 8)
        return flops, nbytes

    def oracle_sample(self, host, rng, n):
        import oracle
        w = host.workload
        if not hasattr(self, "_host"):
            self._host = (self.d_out.cpu(), self.probs.cpu())
        oracle.unpermute_grad(host.grad_y, self._host[0], self._host[1], host.expanded_row_idx,
                              w.batch, w.top_k, w.row_idx_type)
        _, nbytes = self.algorithmic()
        return nbytes, f"all {w.batch} tokens (whole problem: the oracle has no token sample)"

    def units(self):
        return 1


OPS = {"dx": DxOp, "dw": DwOp, "fwd": FwdOp, "unperm": UnpermOp}


def cpu_baseline(op, target_s: float):
    """The oracle (as it stands) on a bounded sample of the workload."""
    import oracle
    oracle.build()
    host = op.inp.to("cpu")
    rng = np.random.default_rng(0)
    cores = oracle.host_cores()
    n = cores
    t0 = time.perf_counter()
    flops, desc = op.oracle_sample(host, rng, n)
    dt = time.perf_counter() - t0
    if dt < target_s / 4 and n < op.units():
        n = int(min(op.units(), max(n, n * target_s / max(dt, 1e-3))))
        t0 = time.perf_counter()
        flops, desc = op.oracle_sample(host, rng, n)
        dt = time.perf_counter() - t0
    if getattr(op, "unit", "TFLOP/s") == "GB/s":
        value, unit = flops / dt / 1e9, "GB/s"  # oracle_sample returns bytes for this op
    else:
        value, unit = flops / dt / 1e12, "TFLOP/s"
    return {"value": value, "unit": unit, "cores": min(cores, n),
            "kind": "oracle", "sample": f"{desc}, fp64 C++ loops, {dt:.1f} s"}


def run_reference(args):
    """The oracle timed on the host cores: each step a bounded sample."""
    rank, world, _ = dist_info()
    if rank != 0:
        return
    import oracle
    from workloads import WORKLOADS, make_inputs
    oracle.build()
    w = WORKLOADS[args.workload]
    inp = make_inputs(w, device="cpu")
    op = OPS[args.op].__new__(OPS[args.op])
    op.inp = inp
    if args.op in ("dw", "fwd"):
        from workloads.moe import forward_input
        op.x = forward_input(inp, "cpu")
    if args.op == "unperm":
        from workloads.moe import unpermute_inputs
        op.d_out, op.probs = unpermute_inputs(inp, "cpu")
    cores = oracle.host_cores()
    # size each step to ~ (a few minutes) / (steps + warmup)
    budget = 150.0 / max(1, args.steps + args.warmup)
    rng = np.random.default_rng(0)
    n = cores
    t0 = time.perf_counter()
    op.oracle_sample(inp, rng, n)
    probe = time.perf_counter() - t0
    n = int(max(1, min(op.units(), n * budget / max(probe, 1e-3))))
    times, flops, desc = [], 0, ""
    for s in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        flops_s, desc = op.oracle_sample(inp, rng, n)
        if s >= args.warmup:
            times.append(time.perf_counter() - t0)
            flops += flops_s
    dt = sum(times)
    if getattr(op, "unit", "TFLOP/s") == "GB/s":
        value, unit = flops / dt / 1e9, "GB/s"  # oracle_sample returns bytes for this op
    else:
        value, unit = flops / dt / 1e12, "TFLOP/s"
    sample = f"{desc} per step, fp64 C++ loops"
    line = {
        "impl": "reference", "metric": op.metric, "value": value, "unit": unit,
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt / max(1, len(times)) * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {**w.describe(), "op": args.op, "sample_units": n},
        "cpu_baseline": {"value": value, "unit": unit, "cores": min(cores, n),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_ours(args):
    import torch
    import permute_grouped_gemm_gb300 as pgg
    from permute_grouped_gemm_gb300 import build as pbuild
    from workloads import WORKLOADS, make_inputs

    rank, world, local = dist_info()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        dist = None
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())
    pbuild.build()
    pgg.load()

    w = WORKLOADS[args.workload]
    inp = make_inputs(w, device=dev)
    op = OPS[args.op](inp, pgg, dev)
    plan, ws, ws_bytes, out = op.plan, op.ws, op.ws_bytes, op.out
    flush_w = torch.empty(256 * 2**20, dtype=torch.uint8, device=dev)
    flush_r = torch.ones(65536, 1024, dtype=torch.float32, device=dev)  # 256 MiB
    flush_acc = torch.empty(1024, dtype=torch.float32, device=dev)

    def flush_l2():
        flush_w.zero_()
        torch.sum(flush_r, dim=0, out=flush_acc)
    stream = torch.cuda.current_stream(dev)
    sp = stream.cuda_stream
    va, vb = op.values()
    idx, gl = inp.expanded_row_idx, inp.group_list

    def route_prep():
        rc = op.stage1(idx, gl, sp)
        if rc:
            raise pgg.PggError(rc, "route_prep")

    def gemm():
        rc = op.stage2(va, vb, idx, gl, out, sp)
        if rc:
            raise pgg.PggError(rc, "grouped_gemm")

    def check_status():
        if pgg.status(ws) != 0:
            raise RuntimeError(f"device status {pgg.STATUS[pgg.status(ws)]}")

    with ClockSampler(torch.cuda.current_device()) as clk:
        # Untimed burn-in of the same step, so that the GPU (and any outside
        # clock sampler) is under load and at its steady clock before timing.
        t0 = time.perf_counter()
        burn_steps = 0
        while time.perf_counter() - t0 < args.burn_in:
            for _ in range(16):
                flush_l2()
                route_prep()
                gemm()
            burn_steps += 16
            torch.cuda.synchronize()
        burn_window = (t0, time.perf_counter())
        for _ in range(args.warmup):
            flush_l2()
            route_prep()
            gemm()
        torch.cuda.synchronize()
        check_status()

        # The torch allocator's peak over the library calls alone (the flush's
        # reduction allocates scratch of its own, outside them).
        base_alloc = torch.cuda.memory_allocated(dev)
        torch.cuda.reset_peak_memory_stats(dev)
        route_prep()
        gemm()
        torch.cuda.synchronize()
        alloc_delta = torch.cuda.max_memory_allocated(dev) - base_alloc

        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
        if dist:
            dist.barrier()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for s in range(args.steps):
            flush_l2()
            ev[s][0].record(stream)
            route_prep()
            ev[s][1].record(stream)
            gemm()
            ev[s][2].record(stream)
        torch.cuda.synchronize()
        timed_window = (t0, time.perf_counter())
        if dist:
            dist.barrier()
        step_ms = [ev[s][0].elapsed_time(ev[s][2]) for s in range(args.steps)]
        gemm_ms = [ev[s][1].elapsed_time(ev[s][2]) for s in range(args.steps)]
        prep_ms = [ev[s][0].elapsed_time(ev[s][1]) for s in range(args.steps)]
        check_status()

        # The same steps with L2 left warm (no flush between them).
        wev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
        torch.cuda.synchronize()
        wev[0].record(stream)
        for s in range(args.steps):
            route_prep()
            gemm()
            wev[s + 1].record(stream)
        torch.cuda.synchronize()
        warm_ms = [wev[s].elapsed_time(wev[s + 1]) for s in range(args.steps)]
        check_status()
    mean_step = statistics.mean(step_ms)
    mean_gemm = statistics.mean(gemm_ms)
    med_step = statistics.median(step_ms)
    med_warm = statistics.median(warm_ms)
    mean_step, mean_gemm, med_step, med_warm = max_over_ranks(
        [mean_step, mean_gemm, med_step, med_warm], dist, dev)

    flops, nbytes = op.algorithmic()
    value_unit = getattr(op, "unit", "TFLOP/s")
    work = nbytes / 1e9 if value_unit == "GB/s" else flops / 1e12  # per step and GPU
    value = world * work / (mean_step * 1e-3)

    peaks, peak_src = load_peaks()
    clocks = clk.summary(*timed_window)
    burn_clocks = clk.summary(*burn_window)
    # The fraction is taken against the burst (short-run) tensor peak: the
    # timed kernel runs for milliseconds at a time. A power cap seen by the
    # clock samples is reported beside it, not folded into the peak.
    tc_key = "bf16_tflops"
    t_tc = flops / (peaks[tc_key] * 1e12)
    t_hbm = nbytes / (peaks["hbm_gbs"] * 1e9)
    simt = plan["variant"] == SIMT_VARIANT
    kernel = op.kernel
    if simt:
        # FP32 pipes: SMs x FP32 lanes x 2 flops x the maximum SM clock
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        mhz = clocks.get("sm_max_mhz") or NOMINAL_SM_MHZ
        bound, achieved = "alu", flops / (mean_gemm * 1e-3) / 1e12
        peak, unit = sms * FP32_LANES_PER_SM * 2 * mhz * 1e6 / 1e12, "TFLOP/s"
        peak_src = f"derived: {sms} SMs x {FP32_LANES_PER_SM} FP32 lanes x 2 x {mhz:.0f} MHz"
    elif t_tc >= t_hbm:
        bound, achieved = "tensor", flops / (mean_gemm * 1e-3) / 1e12
        peak, unit = peaks[tc_key], "TFLOP/s"
        peak_src = f"{peak_src} {tc_key}"
        if w.dtype == "fp32":
            # 3 tf32 products per fp32 product; tf32 dense rate is half of bf16
            peak = peaks[tc_key] / 2 / 3
    else:
        bound, achieved = "hbm", nbytes / (mean_gemm * 1e-3) / 1e9
        peak, unit = peaks["hbm_gbs"], "GB/s"
        peak_src = f"{peak_src} hbm_gbs"
    src_note = ("MEASURED_PEAKS.json" if peak_src.startswith("measured")
                else "profiling recipe fallback")
    roofline = {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
                "frac": achieved / peak, "traffic": recorded_traffic(kernel, w.name),
                "peak_source": peak_src if simt else f"{peak_src} ({src_note})",
                "kernel": kernel, "algorithmic_flops": flops, "algorithmic_bytes": nbytes}
    if clocks.get("sm_mhz"):
        # clock-independent size of the kernel: thousands of SM cycles per launch
        roofline["kcycles_per_launch_at_median_clock"] = mean_gemm * clocks["sm_mhz"]

    e2e = None
    if not args.no_e2e:
        e2e = measure_e2e(op, pgg, w, dev, stream, flops, nbytes, world, dist)

    line = {
        "metric": op.metric, "value": value, "unit": value_unit, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": mean_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": w.dtype, "data": "synthetic (seeded; routing and value recipe in workloads/moe.py)",
        "config": {**w.describe(), "l2": "flushed between steps (256 MiB write, then 256 MiB read)",
                   "parallelism": f"replicas{world}" if world > 1 else "single GPU",
                   "plan": plan, **({"op": op.name} if op.name != "dx" else {})},
        "workspace_bytes": ws_bytes,
        "torch_alloc_delta_bytes": int(alloc_delta),
        "phases_ms": {"route_prep": statistics.mean(prep_ms), "grouped_gemm": mean_gemm},
        "median_ms_per_step": med_step,
        "median_value": world * work / (med_step * 1e-3),
        "warm_l2": {"ms_per_step_median": med_warm,
                    "value": world * work / (med_warm * 1e-3),
                    "l2": "not flushed: the same steps back to back"},
        "roofline": roofline,
        "clocks": clocks,
        "burn_in": {"seconds": burn_window[1] - burn_window[0], "steps": burn_steps,
                    "clocks": burn_clocks},
        "gpu_launches": getattr(op, "launches", 4) * args.steps,
        "wall_s_timed_region": timed_window[1] - timed_window[0],
    }
    if e2e:
        line["e2e"] = e2e
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(op, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def measure_e2e(op, pgg, w, dev, stream, flops, nbytes, world, dist):
    """Same metric through the public call with host buffers: every step copies
    the inputs from pinned host memory, runs the execute call and copies the
    result back."""
    import torch
    va, vb = op.values()
    inp = op.inp
    hosts = [t.cpu().pin_memory() for t in (va, vb, inp.expanded_row_idx, inp.group_list)]
    devs = [torch.empty_like(t) for t in (va, vb, inp.expanded_row_idx, inp.group_list)]
    d_out = torch.empty_like(op.out)
    h_out = torch.empty(d_out.shape, dtype=d_out.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in hosts)
    d2h = h_out.numel() * h_out.element_size()
    steps = 5

    def step():
        for d, h in zip(devs, hosts):
            d.copy_(h, non_blocking=True)
        rc = op.execute(*devs, d_out, stream.cuda_stream)
        if rc:
            raise pgg.PggError(rc, "execute")
        h_out.copy_(d_out, non_blocking=True)

    for _ in range(2):
        step()
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    if dist:
        dist.barrier()
    a.record(stream)
    for _ in range(steps):
        step()
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / steps
    ms = max_over_ranks([ms], dist, dev)[0]
    if not torch.equal(h_out, d_out.cpu()):
        raise RuntimeError("e2e readback mismatch")
    if getattr(op, "unit", "TFLOP/s") == "GB/s":
        value, unit = world * nbytes / (ms * 1e-3) / 1e9, "GB/s"
    else:
        value, unit = world * flops / (ms * 1e-3) / 1e12, "TFLOP/s"
    return {"value": value, "unit": unit,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": ms}


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
