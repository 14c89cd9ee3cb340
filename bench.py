#!/usr/bin/env python3
"""Bench: BF16 GEMM TFLOP/s on one GB300 (replicas on N GPUs), and every configured workload.

One step is one call of the C-ABI GEMM (tensor-map encode, persistent tcgen05
kernel: tile scheduling, TMA producer, MMA, epilogue) on the 4096^3 workload:
A[4096, 4096] and B[4096, 4096] row-major with N(0, 1) entries rounded to
bf16, FP32 accumulate, bf16 C, alpha = 1, beta = 0 (the square BF16 GEMM that
"cp.async / ldmatrix ablation plan" section 0.3 times at 4096^3). `value` is
that workload's throughput.

Beside it, the "configs" field times every configured workload the same way:
the 256^3 uniform GEMM into FP32 C, the 4096^3 GEMM, the K-sweep of section 2.3
(K in {256, 512, 1024, 4096, 8192} x M = N in {512, 4096}), the backward pair of
"fused A2A/GEMM Perfetto profile protocol" (dX = dY W, and dW += dY^T X with
beta = 1 into bf16), lower SYRK 8192 x 4096 with beta = 1 into FP32, and, beyond
those, lower SYR2K of the same size, the FP8 E4M3 and MXFP8 GEMMs at 4096^3
and the BF16 -> MXFP8 quantization of a 4096 x 4096 matrix.

Timing: the headline is W warm-up steps, then exactly K steps between two CUDA
events on the launching stream, bracketed by a barrier and a device
synchronisation on both sides; the max over ranks is taken. Each configured
workload is also timed as 10 warm-up + 50 iterations with one event pair per
iteration (the protocol page's official timing rule), reported as p50, p95
and min, and as the average of 100 back-to-back calls between one event pair
(where each kernel's set-up overlaps the previous one's tail) and of 100 calls
replayed from one CUDA graph. The 4096^3 call is finally timed over a long
back-to-back loop, where the power cap sets the clock ("sustained"). Inputs
are resident in HBM; every step uses the next of several input sets whose
total is larger than twice the L2, so no step finds its operands in L2. Clocks, power and throttle reasons are sampled through NVML during every
timed window (one sample forced at each window's end as well as a 5 ms poll).
`e2e` repeats the headline measurement through the same C-ABI call with the
inputs in pinned host memory: each step copies A and B to the device and C back
inside the timed region, pipelined over two device buffer sets and three
streams (uploads, GEMMs, downloads).

`--impl reference` times the CPU oracle (plain double-precision triple loop)
on a bounded sample of the same workload; it is the comparison arm, not a
target.

Prints ONE JSON line on rank 0.
"""

from __future__ import annotations

import argparse
import ctypes
import hashlib
import re
import json
import os
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "BF16 GEMM TFLOP/s (4096³ + K-sweep) and % of GB300 dense BF16 tensor peak"
UNIT = "TFLOP/s"
# Best 4096^3 BF16 figure printed by the pages (TMA multistage kernel, 4.006 ms,
# on an sm_120-class card): context, not the target.
PAGES_4096_TFLOPS = 34.31
L2_BYTES = 129 * 1024 * 1024
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
PER_ITER_WARMUP = 10
PER_ITER_TIMED = 50
BACK_TO_BACK_CALLS = 100
GRAPH_CALLS = 100

MAIN = dict(name="gemm_bf16_4096x4096x4096_nn_bf16c", m=4096, n=4096, k=4096, ta=0, tb=0, std=1.0,
            beta=0.0, cbf=True)
SWEEP = [dict(name=f"sweep_{mn}x{mn}x{k}", m=mn, n=mn, k=k, ta=0, tb=0, std=1.0, beta=0.0, cbf=True)
         for mn in (512, 4096) for k in (256, 512, 1024, 4096, 8192)]
SMALL = dict(name="gemm_256x256x256_uniform_f32c", m=256, n=256, k=256, ta=0, tb=0, std=None, beta=0.0, cbf=False)
BWD = [
    dict(name="bwd_dX_2048x5120x5120", m=2048, n=5120, k=5120, ta=0, tb=0, std=0.02, beta=0.0, cbf=True),
    dict(name="bwd_dW_5120x5120x2048_transA_beta1", m=5120, n=5120, k=2048, ta=1, tb=0, std=0.02,
         beta=1.0, cbf=True),
]
FP8 = [
    dict(name="gemm_e4m3_4096x4096x4096_tn_bf16c", m=4096, n=4096, k=4096, ta=0, tb=1, std=1.0, beta=0.0,
         cbf=True, e4m3=True),
    dict(name="gemm_mxfp8_4096x4096x4096_tn_bf16c", m=4096, n=4096, k=4096, ta=0, tb=1, std=1.0, beta=0.0,
         cbf=True, mxfp8=True),
]
SYRK_CFG = dict(name="syrk_lower_8192x4096_f32c_beta1", n=8192, k=4096, beta=1.0)
SYR2K_CFG = dict(name="syr2k_lower_8192x4096_f32c_beta1", n=8192, k=4096, beta=1.0, two=True)
QUANT_CFG = dict(name="quantize_mxfp8_4096x4096_bf16", rows=4096, k=4096, quant=True)
# (label, workload) in report order: the configured workloads C1..C5, then the extras
CONFIG_ORDER = ([("C1", SMALL), ("C2", MAIN)] + [("C3", c) for c in SWEEP] + [("C4a", BWD[0]), ("C4b", BWD[1]),
                ("C5", SYRK_CFG), ("extra", SYR2K_CFG)] + [("extra", c) for c in FP8] + [("extra", QUANT_CFG)])
EXTRA = [SMALL] + BWD + FP8  # GEMM workloads beyond the sweep (for --workload)


# ----------------------------------------------------------------------------- work accounting
def gemm_flops(m, n, k):
    """2*M*N*K, the convention of the pages' 4096^3 tables (e.g. 2*4096^3 / 4.259 ms = 32.27 TFLOP/s)."""
    return 2 * m * n * k


def syrk_flops(n, k):
    """Products of the referenced triangle incl. the diagonal: n(n+1)/2 outputs x 2k."""
    return n * (n + 1) * k


def gemm_bytes(m, n, k, c_bytes, beta):
    """Each operand read once, C written once (and read once when beta != 0)."""
    return 2 * (m * k + k * n) + c_bytes * m * n * (2 if beta != 0 else 1)


def syrk_bytes(n, k, c_bytes, beta):
    tri = n * (n + 1) // 2
    return 2 * n * k + c_bytes * tri * (2 if beta != 0 else 1)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS, source="fallback")


def _code_only(text):
    """C++ source without comments and with whitespace runs collapsed, so that
    comment edits do not mark a profile of unchanged code as stale."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_hash(csrc=None):
    h = hashlib.sha256()
    csrc = csrc or os.path.join(ROOT, "blas3_tensor_core_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name.endswith((".cu", ".cuh", ".h")):
            with open(os.path.join(csrc, name), encoding="utf-8") as f:
                h.update(name.encode())
                h.update(_code_only(f.read()).encode())
    return h.hexdigest()


def profiled_traffic(workload):
    """DRAM bytes per launch from the committed ncu summary, if it matches the current kernel source."""
    path = os.path.join(ROOT, "profiles", f"{workload}.ncu.txt")
    try:
        text = open(path).read()
    except OSError:
        return None, None
    fields = {}
    for line in text.splitlines():
        if ":" in line and not line.startswith(" "):
            key, _, val = line.partition(":")
            fields[key.strip()] = val.strip()
    if fields.get("kernel_source_sha256") != kernel_source_hash():
        return None, "stale"
    try:
        return float(fields["dram_bytes_per_launch"]), os.path.relpath(path, ROOT)
    except (KeyError, ValueError):
        return None, None


def percentile(values, q):
    """q-th percentile (0..100) with linear interpolation between order statistics."""
    v = sorted(values)
    if not v:
        return None
    pos = (len(v) - 1) * q / 100.0
    lo = int(pos)
    hi = min(lo + 1, len(v) - 1)
    return v[lo] + (v[hi] - v[lo]) * (pos - lo)


# ----------------------------------------------------------------------------- clocks (NVML via ctypes)
class ClockSampler:
    """Samples SM clock, power and clock-event reasons every few ms on a host thread;
    `sample_now()` adds one on demand (each timed window forces one while it runs)."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, torch_device, period_s=0.005):
        self.period = period_s
        self.samples = []
        self.windows = []
        self.max_mhz = None
        self.ok = False
        self._stop = threading.Event()
        self._thread = None
        try:
            self.nvml = ctypes.CDLL("libnvidia-ml.so.1")
            if self.nvml.nvmlInit_v2() != 0:
                return
            self.handle = ctypes.c_void_p()
            got = False
            try:
                import torch
                props = torch.cuda.get_device_properties(torch_device)
                bus = f"{props.pci_domain_id:08X}:{props.pci_bus_id:02X}:{props.pci_device_id:02X}.0"
                got = self.nvml.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(self.handle)) == 0
            except Exception:
                got = False
            if not got and self.nvml.nvmlDeviceGetHandleByIndex_v2(0, ctypes.byref(self.handle)) != 0:
                return
            mx = ctypes.c_uint()
            if self.nvml.nvmlDeviceGetMaxClockInfo(self.handle, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = mx.value
            self._reasons_fn = getattr(self.nvml, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                getattr(self.nvml, "nvmlDeviceGetCurrentClocksThrottleReasons")
            self.ok = True
        except (OSError, AttributeError):
            self.ok = False

    def _sample(self):
        clk, pw, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        self.nvml.nvmlDeviceGetClockInfo(self.handle, 1, ctypes.byref(clk))
        self.nvml.nvmlDeviceGetPowerUsage(self.handle, ctypes.byref(pw))
        self._reasons_fn(self.handle, ctypes.byref(rs))
        return (time.perf_counter(), clk.value, pw.value / 1000.0, rs.value)

    def sample_now(self):
        if self.ok:
            try:
                self.samples.append(self._sample())
            except Exception:
                pass

    def _run(self):
        while not self._stop.is_set():
            self.sample_now()
            time.sleep(self.period)

    def start(self):
        if self.ok:
            self._thread = threading.Thread(target=self._run, daemon=True)
            self._thread.start()

    def mark(self, t0, t1):
        self.windows.append((t0, t1))

    def stop(self):
        if self._thread is not None:
            self._stop.set()
            self._thread.join()

    def summary(self):
        if not self.ok:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "source": "unavailable"}
        wins = self.windows or [(float("-inf"), float("inf"))]
        inside = [s for s in self.samples if any(t0 <= s[0] <= t1 for t0, t1 in wins)]
        reasons = set()
        for s in inside:
            for bit, name in self.REASONS.items():
                if s[3] & bit:
                    reasons.add(name)
        return {"sm_mhz": statistics.median([s[1] for s in inside]) if inside else None,
                "sm_mhz_min": min((s[1] for s in inside), default=None),
                "sm_max_mhz": self.max_mhz,
                "power_w_max": max((s[2] for s in inside), default=None),
                "reasons": sorted(reasons), "samples": len(inside), "windows": len(self.windows),
                "source": "nvml"}


class NoSampler:
    def sample_now(self):
        pass

    def mark(self, t0, t1):
        pass


# ----------------------------------------------------------------------------- distributed plumbing
class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = False
        if self.world > 1:
            import torch.distributed as dist
            os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
            dist.init_process_group("gloo", rank=self.rank, world_size=self.world)
            self.pg = True

    def barrier(self):
        if self.pg:
            import torch.distributed as dist
            dist.barrier()

    def max(self, value: float) -> float:
        if not self.pg:
            return value
        import torch
        import torch.distributed as dist
        t = torch.tensor([value], dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg:
            import torch.distributed as dist
            dist.destroy_process_group()


# ----------------------------------------------------------------------------- GPU workloads
def host_inputs(cfg):
    import numpy as np
    import bm_inputs as gen
    m, n, k, ta, tb = cfg["m"], cfg["n"], cfg["k"], cfg["ta"], cfg["tb"]
    if cfg.get("e4m3") or cfg.get("mxfp8"):  # A [m, k], B [n, k] E4M3 codes, C = A B^T
        A, B = gen.matrix_e4m3(m, k, "normal", seed=1), gen.matrix_e4m3(n, k, "normal", seed=2)
        if cfg.get("mxfp8"):  # one UE8M0 scale per 32 elements of K: 2^-3 .. 2^3
            g = (k + 31) // 32
            SA = gen.integers(3, m * g, 124, 130).reshape(m, g).astype(np.uint8)
            SB = gen.integers(4, n * g, 124, 130).reshape(n, g).astype(np.uint8)
            return A, B, None, (SA, SB)
        return A, B, None, None
    ra, ca = (k, m) if ta else (m, k)
    rb, cb = (n, k) if tb else (k, n)
    if cfg["std"] is None:
        A = gen.matrix_bf16(ra, ca, "uniform", seed=1)
        B = gen.matrix_bf16(rb, cb, "uniform", seed=2)
    else:
        A = gen.matrix_bf16(ra, ca, "normal", seed=1, std=cfg["std"])
        B = gen.matrix_bf16(rb, cb, "normal", seed=2, std=cfg["std"])
    C0 = None
    if cfg["beta"] != 0:
        C0 = gen.matrix_bf16(m, n, "normal", seed=3, std=cfg["std"] or 1.0)
    return A, B, C0, None


def tiled_scales(S, rows, k):
    """UE8M0 codes [rows, groups] in the tiled atom layout the library reads (padding code 0)."""
    import numpy as np
    import blas3_tensor_core_gb300 as bm
    groups = (k + 31) // 32
    out = np.zeros(bm.mxfp8_scale_bytes(rows, k), np.uint8)
    r = np.repeat(np.arange(rows, dtype=np.int64), groups)
    g = np.tile(np.arange(groups, dtype=np.int64), rows)
    out[bm.mxfp8_scale_offset(r, g, k)] = S[:rows, :groups].reshape(-1)
    return out


class GemmWorkload:
    """Device-resident input sets for one GEMM shape, rotated so that no step hits L2."""

    def __init__(self, cfg, torch_mod, min_total=2 * L2_BYTES, max_sets=1024):
        import numpy as np
        t = torch_mod
        self.cfg = cfg
        self.name = cfg["name"]
        self.t = t
        A, B, C0, scales = host_inputs(cfg)
        self.A_host, self.B_host, self.C0_host = A, B, C0
        self.e4m3 = bool(cfg.get("e4m3"))
        self.mxfp8 = bool(cfg.get("mxfp8"))
        m, n, k = cfg["m"], cfg["n"], cfg["k"]
        if self.e4m3 or self.mxfp8:
            dA = t.from_numpy(A).cuda()
            dB = t.from_numpy(B).cuda()
        else:
            dA = t.from_numpy(A.view(np.int16)).view(t.bfloat16).cuda()
            dB = t.from_numpy(B.view(np.int16)).view(t.bfloat16).cuda()
        self.dSA = self.dSB = None
        if self.mxfp8:
            self.dSA = t.from_numpy(tiled_scales(scales[0], m, k)).cuda()
            self.dSB = t.from_numpy(tiled_scales(scales[1], n, k)).cuda()
        cdt = t.bfloat16 if cfg["cbf"] else t.float32
        dC = t.empty((m, n), dtype=cdt, device="cuda")
        if C0 is not None:
            dC.copy_(t.from_numpy(C0.view(np.int16)).view(t.bfloat16).to(cdt))
        per_set = dA.numel() * dA.element_size() + dB.numel() * dB.element_size() + dC.numel() * dC.element_size()
        nsets = max(2, min(max_sets, -(-min_total // per_set)))
        self.sets = [(dA, dB, dC)] + [(dA.clone(), dB.clone(), dC.clone()) for _ in range(nsets - 1)]
        self.set_bytes = per_set
        import blas3_tensor_core_gb300 as bm
        self.bm = bm
        if self.mxfp8:
            need = bm.bm_gemm_mxfp8_workspace_size(m, n, k)
            st, self.plan = bm.bm_gemm_mxfp8_plan(m, n, k, need)
        elif self.e4m3:
            need = bm.bm_gemm_e4m3_workspace_size(m, n, k)
            # reported as the plan of a bf16 GEMM with half the K (same bytes per k-block); an E4M3
            # call keeps the larger tail-split threshold, so its tail may run as N halves instead
            st, self.plan = bm.bm_gemm_bf16_plan(m, n, k // 2, need)
        else:
            need = bm.bm_gemm_bf16_workspace_size(m, n, k)
            st, self.plan = bm.bm_gemm_bf16_plan(m, n, k, need)
        assert st == 0
        self.ws = t.empty(max(need // 4, 1), dtype=t.float32, device="cuda") if need else None
        self.ws_bytes = need
        self.lda = A.shape[1]
        self.ldb = B.shape[1]

    def call(self, i, stream_handle):
        dA, dB, dC = self.sets[i % len(self.sets)]
        self.call_set(dA, dB, dC, stream_handle)

    def call_set(self, dA, dB, dC, stream_handle):
        c = self.cfg
        ws = None if self.ws is None else self.ws.data_ptr()
        ct = self.bm.BM_C_BF16 if c["cbf"] else self.bm.BM_C_F32
        if self.mxfp8:
            st = self.bm.bm_gemm_mxfp8(c["m"], c["n"], c["k"], 1.0, dA.data_ptr(), self.lda, self.dSA.data_ptr(),
                                       dB.data_ptr(), self.ldb, self.dSB.data_ptr(), c["beta"], dC.data_ptr(),
                                       c["n"], ct, ws, self.ws_bytes, stream_handle)
        elif self.e4m3:
            st = self.bm.bm_gemm_e4m3(c["m"], c["n"], c["k"], 1.0, dA.data_ptr(), self.lda, dB.data_ptr(), self.ldb,
                                      c["beta"], dC.data_ptr(), c["n"], ct, ws, self.ws_bytes, stream_handle)
        else:
            st = self.bm.bm_gemm_bf16(c["m"], c["n"], c["k"], c["ta"], c["tb"], 1.0, dA.data_ptr(), self.lda,
                                      dB.data_ptr(), self.ldb, c["beta"], dC.data_ptr(), c["n"], ct, ws,
                                      self.ws_bytes, stream_handle)
        if st != 0:
            raise RuntimeError(f"{self.name}: {self.bm.bm_status_string(st)}")

    def flops(self):
        c = self.cfg
        return gemm_flops(c["m"], c["n"], c["k"])

    def bytes(self):
        c = self.cfg
        m, n, k = c["m"], c["n"], c["k"]
        b = gemm_bytes(m, n, k, 2 if c["cbf"] else 4, c["beta"])
        if self.e4m3 or self.mxfp8:
            b -= m * k + k * n  # 1-byte operands
        if self.mxfp8:
            b += self.dSA.numel() + self.dSB.numel()
        return b

    def tensor_peak(self, peaks):
        # FP8 tensor peak: the measured bf16 peak times the nominal FP8 / BF16 ratio (4.5 / 2.25 PF)
        return peaks["bf16_tflops"] * (2.0 if (self.e4m3 or self.mxfp8) else 1.0)

    def kind(self):
        return "mxfp8 gemm" if self.mxfp8 else ("e4m3 gemm" if self.e4m3 else "bf16 gemm")

    def flop_convention(self):
        return "2mnk"


class SyrkWorkload:
    """Lower SYRK (or SYR2K) 8192 x 4096 with beta = 1 into a symmetric FP32 C, two C buffers
    of 256 MiB each (larger than L2) alternating."""

    def __init__(self, cfg, torch_mod):
        import numpy as np
        import bm_inputs as gen
        import blas3_tensor_core_gb300 as bm
        t = torch_mod
        self.t, self.bm, self.cfg, self.name = t, bm, cfg, cfg["name"]
        self.two = bool(cfg.get("two"))
        n, k = cfg["n"], cfg["k"]
        self.A_host = gen.matrix_bf16(n, k, "normal", seed=1)
        self.dA = t.from_numpy(self.A_host.view(np.int16)).view(t.bfloat16).cuda()
        self.dB = (t.from_numpy(gen.matrix_bf16(n, k, "normal", seed=2).view(np.int16)).view(t.bfloat16).cuda()
                   if self.two else self.dA)
        C0 = gen.symmetric_f32(n, seed=3)
        self.dCs = [t.from_numpy(C0).cuda() for _ in range(2)]
        size_fn = bm.bm_syr2k_bf16_workspace_size if self.two else bm.bm_syrk_bf16_workspace_size
        need = size_fn(bm.BM_LOWER, n, k)
        self.ws = t.empty(max(need // 4, 1), dtype=t.float32, device="cuda") if need else None
        self.ws_bytes = need
        st, self.plan = bm.bm_syrk_bf16_plan(bm.BM_LOWER, n, k, need)
        assert st == 0

    def call(self, i, hh):
        c, bm = self.cfg, self.bm
        n, k = c["n"], c["k"]
        ws = None if self.ws is None else self.ws.data_ptr()
        C = self.dCs[i % 2].data_ptr()
        if self.two:
            st = bm.bm_syr2k_bf16(bm.BM_LOWER, bm.BM_OP_N, n, k, 1.0, self.dA.data_ptr(), k, self.dB.data_ptr(), k,
                                  c["beta"], C, n, bm.BM_C_F32, ws, self.ws_bytes, hh)
        else:
            st = bm.bm_syrk_bf16(bm.BM_LOWER, bm.BM_OP_N, n, k, 1.0, self.dA.data_ptr(), k, c["beta"], C, n,
                                 bm.BM_C_F32, ws, self.ws_bytes, hh)
        if st != 0:
            raise RuntimeError(f"{self.name}: {bm.bm_status_string(st)}")

    def flops(self):
        return (2 if self.two else 1) * syrk_flops(self.cfg["n"], self.cfg["k"])

    def bytes(self):
        n, k = self.cfg["n"], self.cfg["k"]
        return syrk_bytes(n, k, 4, self.cfg["beta"]) + (2 * n * k if self.two else 0)

    def tensor_peak(self, peaks):
        return peaks["bf16_tflops"]

    def kind(self):
        return "bf16 syr2k" if self.two else "bf16 syrk"

    def flop_convention(self):
        return f"{2 if self.two else 1} n(n+1)k (lower triangle incl. diagonal)"


class QuantWorkload:
    """BF16 [4096, 4096] N(0, 1) -> MXFP8 codes and tiled scales, input sets rotated past L2."""

    def __init__(self, cfg, torch_mod, min_total=2 * L2_BYTES):
        import numpy as np
        import bm_inputs as gen
        import blas3_tensor_core_gb300 as bm
        t = torch_mod
        self.t, self.bm, self.cfg, self.name = t, bm, cfg, cfg["name"]
        rows, k = cfg["rows"], cfg["k"]
        X = gen.matrix_bf16(rows, k, "normal", seed=1)
        dX = t.from_numpy(X.view(np.int16)).view(t.bfloat16).cuda()
        dQ = t.empty((rows, k), dtype=t.uint8, device="cuda")
        dS = t.empty(bm.mxfp8_scale_bytes(rows, k), dtype=t.uint8, device="cuda")
        per_set = dX.numel() * 2 + dQ.numel() + dS.numel()
        nsets = max(2, -(-min_total // per_set))
        self.sets = [(dX, dQ, dS)] + [(dX.clone(), dQ.clone(), dS.clone()) for _ in range(nsets - 1)]
        self.plan = None

    def call(self, i, hh):
        dX, dQ, dS = self.sets[i % len(self.sets)]
        rows, k = self.cfg["rows"], self.cfg["k"]
        st = self.bm.bm_quantize_mxfp8(rows, k, dX.data_ptr(), k, dQ.data_ptr(), k, dS.data_ptr(), hh)
        if st != 0:
            raise RuntimeError(f"{self.name}: {self.bm.bm_status_string(st)}")

    def flops(self):
        return 0

    def bytes(self):
        rows, k = self.cfg["rows"], self.cfg["k"]
        return rows * k * 3 + self.bm.mxfp8_scale_bytes(rows, k)

    def tensor_peak(self, peaks):
        return peaks["bf16_tflops"]

    def kind(self):
        return "bf16 -> mxfp8 quantization"

    def flop_convention(self):
        return "none (memory-bound: 2 bytes read, 1 + 1/32 written per element)"


def make_workload(cfg, torch_mod):
    if cfg.get("quant"):
        return QuantWorkload(cfg, torch_mod)
    return SyrkWorkload(cfg, torch_mod) if "m" not in cfg else GemmWorkload(cfg, torch_mod)


def _check_device(wl, h):
    st = wl.bm.bm_get_last_device_error(h)
    if st != 0:
        raise RuntimeError(f"device error: {wl.bm.bm_status_string(st)}")


def timed_steps(wl, steps, warmup, dist, sampler=None):
    """Device time (ms) of exactly `steps` calls between one pair of events, max over ranks."""
    t = wl.t
    sampler = sampler or NoSampler()
    stream = t.cuda.current_stream()
    h = stream.cuda_stream
    for i in range(warmup):
        wl.call(i, h)
    t.cuda.synchronize()
    dist.barrier()
    t.cuda.synchronize()
    ev0, ev1 = t.cuda.Event(enable_timing=True), t.cuda.Event(enable_timing=True)
    host0 = time.perf_counter()
    ev0.record(stream)
    for i in range(steps):
        wl.call(warmup + i, h)
    ev1.record(stream)
    sampler.sample_now()  # the launches are queued: the GPU is busy with them now
    t.cuda.synchronize()
    host1 = time.perf_counter()
    sampler.mark(host0, host1)
    dist.barrier()
    t.cuda.synchronize()
    _check_device(wl, h)
    return dist.max(ev0.elapsed_time(ev1))


def per_iteration(wl, dist, sampler=None, iters=PER_ITER_TIMED, warmup=PER_ITER_WARMUP):
    """Per-call device times (ms): `warmup` untimed calls, then `iters` calls with one event pair
    each. Returns {p50, p95, min, mean} in ms, each the max over ranks."""
    t = wl.t
    sampler = sampler or NoSampler()
    stream = t.cuda.current_stream()
    h = stream.cuda_stream
    for i in range(warmup):
        wl.call(i, h)
    t.cuda.synchronize()
    dist.barrier()
    t.cuda.synchronize()
    evs = [(t.cuda.Event(enable_timing=True), t.cuda.Event(enable_timing=True)) for _ in range(iters)]
    host0 = time.perf_counter()
    for i, (e0, e1) in enumerate(evs):
        e0.record(stream)
        wl.call(warmup + i, h)
        e1.record(stream)
    sampler.sample_now()
    t.cuda.synchronize()
    host1 = time.perf_counter()
    sampler.mark(host0, host1)
    dist.barrier()
    _check_device(wl, h)
    ms = [e0.elapsed_time(e1) for e0, e1 in evs]
    return {"p50": dist.max(percentile(ms, 50)), "p95": dist.max(percentile(ms, 95)),
            "min": dist.max(min(ms)), "mean": dist.max(sum(ms) / len(ms)), "n": len(ms)}


def graph_steps(wl, steps):
    """Device time (ms) per call when `steps` calls are captured in one CUDA graph and replayed."""
    t = wl.t
    side = t.cuda.Stream()
    side.wait_stream(t.cuda.current_stream())
    with t.cuda.stream(side):  # first-call set-up (device state, attributes) happens outside capture
        wl.call(0, side.cuda_stream)
    t.cuda.current_stream().wait_stream(side)
    t.cuda.synchronize()
    g = t.cuda.CUDAGraph()
    with t.cuda.graph(g):
        h = t.cuda.current_stream().cuda_stream
        for i in range(steps):
            wl.call(i, h)
    g.replay()
    t.cuda.synchronize()
    ev0, ev1 = t.cuda.Event(enable_timing=True), t.cuda.Event(enable_timing=True)
    stream = t.cuda.current_stream()
    ev0.record(stream)
    g.replay()
    ev1.record(stream)
    t.cuda.synchronize()
    _check_device(wl, stream.cuda_stream)
    ms = ev0.elapsed_time(ev1) / steps
    del g
    return ms


def e2e_steps(wl, steps, warmup, dist):
    """Same call with pinned host inputs: H2D of A and B and D2H of C inside the timed region.

    The steps are pipelined the way a stream of GEMMs would be fed: two device
    buffer sets and three streams, so the upload of step i + 1 and the download
    of step i - 1 overlap the GEMM of step i. Events order each buffer set's
    reuse (upload after the GEMM two steps back has read it, GEMM after the
    download two steps back has read its C). Every step still moves its whole
    A and B to the device and its whole C back.
    """
    import numpy as np
    t = wl.t
    main = t.cuda.current_stream()
    h = main.cuda_stream
    s_in, s_out = t.cuda.Stream(), t.cuda.Stream()
    hA = t.from_numpy(wl.A_host.view(np.int16)).view(t.bfloat16).pin_memory()
    hB = t.from_numpy(wl.B_host.view(np.int16)).view(t.bfloat16).pin_memory()
    slots = wl.sets[:2]
    hC = t.empty(slots[0][2].shape, dtype=slots[0][2].dtype).pin_memory()
    hC0 = None
    if wl.C0_host is not None:  # beta != 0: the step's input C travels too
        hC0 = t.from_numpy(wl.C0_host.view(np.int16)).view(t.bfloat16).to(slots[0][2].dtype).pin_memory()
    read_done = [t.cuda.Event(), t.cuda.Event()]   # GEMM of the slot's last step has read A, B (and C)
    out_done = [t.cuda.Event(), t.cuda.Event()]    # download of the slot's last step has read C
    in_done = [t.cuda.Event(), t.cuda.Event()]

    def step(i):
        s = i % 2
        dA, dB, dC = slots[s]
        if i >= 2:
            s_in.wait_event(read_done[s])
            if hC0 is not None:
                s_in.wait_event(out_done[s])
        with t.cuda.stream(s_in):
            dA.copy_(hA, non_blocking=True)
            dB.copy_(hB, non_blocking=True)
            if hC0 is not None:
                dC.copy_(hC0, non_blocking=True)
        in_done[s].record(s_in)
        main.wait_event(in_done[s])
        if i >= 2:
            main.wait_event(out_done[s])
        wl.call_set(dA, dB, dC, h)
        read_done[s].record(main)
        s_out.wait_event(read_done[s])
        with t.cuda.stream(s_out):
            hC.copy_(dC, non_blocking=True)
        out_done[s].record(s_out)

    def run(n):
        s_in.wait_stream(main)
        s_out.wait_stream(main)
        for i in range(n):
            step(i)
        main.wait_stream(s_in)
        main.wait_stream(s_out)

    run(warmup)
    t.cuda.synchronize()
    dist.barrier()
    t.cuda.synchronize()
    ev0, ev1 = t.cuda.Event(enable_timing=True), t.cuda.Event(enable_timing=True)
    ev0.record(main)
    run(steps)
    ev1.record(main)
    t.cuda.synchronize()
    dist.barrier()
    ms = dist.max(ev0.elapsed_time(ev1))
    h2d = hA.numel() * 2 + hB.numel() * 2 + (0 if hC0 is None else hC0.numel() * hC0.element_size())
    d2h = hC.numel() * hC.element_size()
    return ms, h2d, d2h, hC


# ----------------------------------------------------------------------------- CPU oracle legs
def oracle_rows_rate(A, B, cfg, budget_s):
    """Oracle TFLOP/s on the first R rows of the workload, R sized to about budget_s of CPU work."""
    import oracle
    o = oracle.default()
    m, n, k = cfg["m"], cfg["n"], cfg["k"]
    # calibrate on a probe that gives every oracle thread rows and runs long enough (>= 2 %
    # of the budget) that the call's fixed cost (thread start-up) does not shrink the sample
    rows = min(m, 4 * max(1, o.num_threads()))
    while True:
        t0 = time.perf_counter()
        o.gemm(rows, n, k, 0, 0, 1.0, A[:rows], B)
        dt = max(time.perf_counter() - t0, 1e-6)
        if dt >= 0.02 * budget_s or rows >= m:
            break
        rows = min(m, rows * 4)
    R = int(max(4, min(m, rows * budget_s / dt)))
    t0 = time.perf_counter()
    ref, bound = o.gemm(R, n, k, 0, 0, 1.0, A[:R], B)
    dt = time.perf_counter() - t0
    return {"rows": R, "seconds": dt, "tflops": gemm_flops(R, n, k) / dt / 1e12, "cores": o.num_threads(),
            "ref": ref, "bound": bound}


def cpu_baseline_leg(wl, budget_s):
    """The oracle timed on a bounded sample (the first rows of C); also checks those rows of the GPU C."""
    import numpy as np
    import oracle
    cfg = wl.cfg
    res = oracle_rows_rate(wl.A_host, wl.B_host, cfg, budget_s)
    dC = wl.sets[0][2]
    got = dC[:res["rows"]].float().cpu().numpy().astype(np.float64)
    ok, worst, _ = oracle.compare(got, res["ref"], res["bound"], 1.0, 0.0, None, cfg["cbf"])
    return {"value": round(res["tflops"], 6), "unit": UNIT, "cores": res["cores"], "kind": "oracle",
            "sample": f"first {res['rows']} of {cfg['m']} rows of C for {cfg['name']} "
                      f"({res['seconds']:.1f} s of CPU work; TFLOP/s scaled by 2*rows*n*k)",
            "parity_rows_checked": res["rows"], "parity_ok": bool(ok), "worst_err_over_tol": round(worst, 6)}


def reference_arm(args, dist):
    """--impl reference: the CPU oracle, each step a bounded sample of the 4096^3 workload."""
    if dist.rank != 0:
        return None
    import numpy as np
    import oracle
    cfg = MAIN
    A, B, _, _ = host_inputs(cfg)
    o = oracle.default()
    if dist.world > 1:
        # torchrun caps every rank at one OpenMP thread; the other ranks do no work
        # here, so rank 0 takes all of the host's cores.
        o.set_num_threads(os.cpu_count() or 1)
    n, k = cfg["n"], cfg["k"]
    budget = float(args.reference_budget_s)
    total_steps = args.steps + args.warmup
    per_step_s = max(budget / max(total_steps, 1), 0.002)
    rng = np.random.default_rng(0)
    # calibrate entries per step
    probe = 64
    rows, cols = rng.integers(0, cfg["m"], probe), rng.integers(0, n, probe)
    t0 = time.perf_counter()
    o.gemm_entries(k, 0, 0, 1.0, A, B, rows, cols)
    dt = max(time.perf_counter() - t0, 1e-6)
    entries = int(max(1, min(cfg["m"] * n, probe * per_step_s / dt)))
    samples = [(rng.integers(0, cfg["m"], entries), rng.integers(0, n, entries)) for _ in range(4)]
    for i in range(args.warmup):
        o.gemm_entries(k, 0, 0, 1.0, A, B, *samples[i % 4])
    t0 = time.perf_counter()
    for i in range(args.steps):
        o.gemm_entries(k, 0, 0, 1.0, A, B, *samples[i % 4])
    dt = time.perf_counter() - t0
    flops = 2.0 * entries * k * args.steps
    value = flops / dt / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt / max(args.steps, 1) * 1e3, 6), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": main_config(),
        "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": o.num_threads(), "kind": "oracle",
                         "sample": f"{entries} random entries of C per step for {cfg['name']} "
                                   f"(2*k flops each)"},
        "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    return line


def main_config():
    """The headline workload, identical in both arms."""
    cfg = MAIN
    return {"workload": cfg["name"], "m": cfg["m"], "n": cfg["n"], "k": cfg["k"], "transA": "N", "transB": "N",
            "A": "row-major [4096,4096] N(0,1) rounded to bf16 (seed 1)",
            "B": "row-major [4096,4096] N(0,1) rounded to bf16 (seed 2)",
            "C": "bf16 [4096,4096], alpha=1, beta=0", "accumulate": "fp32",
            "parallelism": "replicas (one independent GEMM per GPU, no collective)"}


def config_record(label, wl, stats, peaks, b2b_ms, graph_ms):
    """One configured workload: per-call times (p50, p95, min: one event pair per call, so each
    call's launch and set-up are exposed), the average over back-to-back calls (one event pair
    around them, the kernels' set-up overlapping the previous call) and over calls replayed from a
    CUDA graph; the roofline fraction at p50 and at the back-to-back average."""
    p50 = stats["p50"] * 1e-3
    tf = wl.flops() / p50 / 1e12
    plan = {}
    if wl.plan is not None:
        plan = {k: getattr(wl.plan, k) for k in ("tile_m", "tile_n", "cta_pair", "tiles", "k_splits",
                                                  "n_splits", "split_tiles", "kernels", "ctas")}
        if getattr(wl, "e4m3", False):
            plan["note"] = ("bf16 plan of K/2; the E4M3 call keeps a 6 us tail-split threshold, so its "
                            "tail tiles may run as N halves instead of a K split")
    gbs = wl.bytes() / p50 / 1e9
    tpeak = wl.tensor_peak(peaks)
    frac_t, frac_h = tf / tpeak, gbs / peaks["hbm_gbs"]
    bound = "tensor" if wl.flops() / (tpeak * 1e12) >= wl.bytes() / (peaks["hbm_gbs"] * 1e9) else "hbm"
    rec = {"config": label, "workload": wl.name, "kind": wl.kind(),
           "us_p50": round(stats["p50"] * 1e3, 3), "us_p95": round(stats["p95"] * 1e3, 3),
           "us_min": round(stats["min"] * 1e3, 3), "us_mean": round(stats["mean"] * 1e3, 3),
           "iterations": stats["n"],
           "tflops_p50": round(tf, 2), "tflops_best": round(wl.flops() / (stats["min"] * 1e-3) / 1e12, 2),
           "gbs_best": round(wl.bytes() / (stats["min"] * 1e-3) / 1e9, 1),
           "gbs_p50": round(gbs, 1), "frac_tensor_p50": round(frac_t, 4), "frac_hbm_p50": round(frac_h, 4),
           "bound": bound, "roofline_frac_p50": round(frac_t if bound == "tensor" else frac_h, 4),
           "flops": wl.flops(), "algorithmic_bytes": wl.bytes(), "flops_convention": wl.flop_convention(),
           "plan": plan}
    b2b = b2b_ms * 1e-3
    rec["us_back_to_back"] = round(b2b_ms * 1e3, 3)
    rec["tflops_back_to_back"] = round(wl.flops() / b2b / 1e12, 2)
    rec["roofline_frac_back_to_back"] = round(
        wl.flops() / b2b / 1e12 / tpeak if bound == "tensor" else wl.bytes() / b2b / 1e9 / peaks["hbm_gbs"], 4)
    rec["us_per_call_graph"] = round(graph_ms * 1e3, 3)
    return rec


# ----------------------------------------------------------------------------- main
def run_gpu_arm(args, dist):
    import torch
    torch.cuda.set_device(dist.local)
    import blas3_tensor_core_gb300 as bm
    if not os.path.exists(bm.library_path):
        from blas3_tensor_core_gb300 import build
        build.build()
    peaks = load_peaks()
    wl = GemmWorkload(MAIN, torch)
    sampler = ClockSampler(torch.cuda.current_device())
    sampler.start()
    ms = timed_steps(wl, args.steps, args.warmup, dist, sampler)
    per_step = ms / args.steps
    value = dist.world * wl.flops() * args.steps / (ms * 1e-3) / 1e12
    achieved = wl.flops() / (per_step * 1e-3) / 1e12
    main_stats = per_iteration(wl, dist, sampler)
    traffic, traffic_src = profiled_traffic(MAIN["name"])
    roofline = {"bound": "tensor", "achieved": round(achieved, 3), "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s", "frac": round(achieved / peaks["bf16_tflops"], 4),
                "traffic": traffic,
                "peak_kind": f"burst bf16 dense ({peaks['source']}, MEASURED_PEAKS.json bf16_tflops)",
                "frac_of_sustained": round(achieved / peaks["bf16_tflops_sustained"], 4),
                "algorithmic_flops_per_launch": wl.flops(),
                "algorithmic_bytes_per_launch": wl.bytes(),
                # template <BN, STAGES, PAIR, ELEM, k-blocks per stage, EPI>: a bf16 GEMM whose C
                # takes a tensor map runs the TMA-store copy (EPI 1) at beta = 0, the combine copy
                # (EPI 2) otherwise
                "kernel": (f"bm_gemm_tcgen05_kernel<{wl.plan.tile_n},{wl.plan.stages},{wl.plan.cta_pair},0,"
                           f"{wl.plan.stage_kblocks},{1 if MAIN['beta'] == 0 else 2}>"
                           + (" + bm_splitk_reduce_kernel" if wl.plan.kernels > 1 else "")),
                "traffic_source": traffic_src}
    graph_ms = graph_steps(wl, GRAPH_CALLS)
    e2e_ms, h2d, d2h, _ = e2e_steps(wl, args.e2e_steps, max(3, args.warmup // 10), dist)
    e2e = {"value": round(dist.world * wl.flops() * args.e2e_steps / (e2e_ms * 1e-3) / 1e12, 3), "unit": UNIT,
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": args.e2e_steps,
           "ms_per_step": round(e2e_ms / args.e2e_steps, 4),
           "pipeline": "two device buffer sets; uploads, GEMMs and downloads on three streams, "
                       "so step i+1's H2D and step i-1's D2H overlap step i's GEMM"}
    launches = args.steps * wl.plan.kernels
    configs = []
    if not args.no_configs:
        for label, cfg in CONFIG_ORDER:
            if cfg is MAIN:
                cw, stats = wl, main_stats
            else:
                cw = make_workload(cfg, torch)
                stats = per_iteration(cw, dist, sampler)
            b2b_ms = timed_steps(cw, BACK_TO_BACK_CALLS, 3, dist, sampler) / BACK_TO_BACK_CALLS
            g_ms = graph_steps(cw, GRAPH_CALLS)
            configs.append(config_record(label, cw, stats, peaks, b2b_ms, g_ms))
            if cw is not wl:
                del cw
                torch.cuda.empty_cache()
    # last: the same call over a long loop (about 0.2 s), where the power cap sets the clock
    long_steps = max(args.sustained_steps, 1)
    sus_ms = timed_steps(wl, long_steps, 3, dist, sampler) / long_steps
    sampler.stop()
    clocks = sampler.summary()
    cpu = None
    if dist.rank == 0 and dist.world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline_leg(wl, args.cpu_budget_s)
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": dist.world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(per_step, 6), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": round(value / PAGES_4096_TFLOPS, 2),
        "vs_baseline_ref": f"{PAGES_4096_TFLOPS} TFLOP/s on one GPU: the pages' best 4096^3 BF16 figure "
                           "(TMA multistage, sm_120-class card, other hardware)",
        "dtype": "bf16", "data": "synthetic", "config": main_config(),
        "l2": (f"inputs larger than L2: {len(wl.sets)} rotating input sets of {wl.set_bytes / 2**20:.0f} MiB "
               f"(> 2 x 129 MB L2)"),
        "plan": wl.plan.as_dict(),
        "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": launches, "clocks": clocks,
        "frac_of_peak": round(achieved / peaks["bf16_tflops"], 4),
        "per_call": {"us_p50": round(main_stats["p50"] * 1e3, 3), "us_p95": round(main_stats["p95"] * 1e3, 3),
                     "us_min": round(main_stats["min"] * 1e3, 3),
                     "tflops_p50": round(wl.flops() / (main_stats["p50"] * 1e-3) / 1e12, 2),
                     "note": f"{PER_ITER_WARMUP} warm-up + {PER_ITER_TIMED} calls, one event pair each"},
        "sustained": {"steps": long_steps, "us_per_step": round(sus_ms * 1e3, 3),
                      "tflops": round(wl.flops() / (sus_ms * 1e-3) / 1e12, 2),
                      "frac_of_sustained_peak": round(wl.flops() / (sus_ms * 1e-3) / 1e12
                                                      / peaks["bf16_tflops_sustained"], 4),
                      "note": "the same call back to back over a long loop (the power cap sets the clock)"},
        "graph": {"us_per_step": round(graph_ms * 1e3, 3),
                  "value": round(dist.world * wl.flops() / (graph_ms * 1e-3) / 1e12, 3), "unit": UNIT,
                  "note": f"{GRAPH_CALLS} calls captured in one CUDA graph, one replay timed"},
        "configs": configs,
    }
    return line


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--sustained-steps", type=int, default=2000)
    ap.add_argument("--no-configs", action="store_true", help="time only the headline workload")
    ap.add_argument("--workload", default=None,
                    help="time only this named workload (for profiling); prints one JSON line for it")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget-s", type=float, default=15.0)
    ap.add_argument("--reference-budget-s", type=float, default=120.0)
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.steps < 1:
        ap.error("--steps must be >= 1")
    return args


def workload_only(args, dist):
    """--workload NAME: W warm-up and K timed steps of one named workload (used for ncu captures)."""
    import torch
    torch.cuda.set_device(dist.local)
    import blas3_tensor_core_gb300 as bm
    if not os.path.exists(bm.library_path):
        from blas3_tensor_core_gb300 import build
        build.build()
    cfg = next((c for _, c in CONFIG_ORDER if c["name"] == args.workload), None)
    if cfg is None:
        raise SystemExit(f"unknown workload {args.workload!r}")
    wl = make_workload(cfg, torch)
    ms = timed_steps(wl, args.steps, args.warmup, dist)
    t = ms / args.steps * 1e-3
    return {"workload": cfg["name"], "us_per_step": round(t * 1e6, 3), "tflops": round(wl.flops() / t / 1e12, 2),
            "steps": args.steps, "warmup": args.warmup, "plan": wl.plan.as_dict() if wl.plan is not None else None}


def main(argv=None):
    args = parse_args(argv)
    dist = Dist()
    try:
        if args.impl == "reference":
            line = reference_arm(args, dist)
        elif args.workload:
            line = workload_only(args, dist)
        else:
            line = run_gpu_arm(args, dist)
        if dist.rank == 0 and line is not None:
            print(json.dumps(line), flush=True)
    finally:
        dist.close()
    return 0


if __name__ == "__main__":
    sys.exit(main())
