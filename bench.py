#!/usr/bin/env python
"""Benchmark of the GB300 BitDelta hot path.

One JSON line on rank 0.  The headline workload is the decode sweep on a
4096x4096 layer (alpha per row, x rows M in {1,2,4,8,16}); one *step* is one
pass of the hot path over a stack of 32 such layers:

    compress (signs + alpha) -> reconstruct to memory -> fused linear at
    M = 1, 2, 4, 8, 16

run phase by phase (all 32 layers through one kernel before the next), so no
kernel reads data the previous kernel touched: the 32 layers (2.2 GB) are far
larger than L2, and the reuse distance of every input is >= 31 launches.
``value`` is algorithmic bytes per step / time per step (GB/s).  The same JSON
line carries the prefill (M = 2048 on the four Llama-70B projections) and
multi-tenant grouped workloads under ``workloads``, each with its own
roofline.

Timing: inputs resident in HBM, W warm-up steps, then K steps captured as a
CUDA graph and replayed, bracketed by barrier + synchronize + CUDA events.
Per-kernel durations come from event-record nodes at phase boundaries inside
the graph.  nvidia-smi samples SM clocks during the timed region.

--impl reference times the CPU oracle (single-threaded C++, fp64) on a sample
of the same workload; it is a deliberately slow baseline, not a target.
"""
from __future__ import annotations

import argparse
import ctypes
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "bitdelta_linear TFLOP/s (prefill) & GB/s (decode) as % of GB300 roofline"
# DRAM bytes (read + write) of one decode launch (4096 x 4096, M = 8) from an ncu
# capture of `python bench.py --profile decode` (dram__bytes_read.sum +
# dram__bytes_write.sum of gemv_single_async_kernel).  Valid for the kernel
# build that capture was taken on; None whenever that kernel has changed since.
DECODE_TRAFFIC_BYTES = 35_749_632

# --------------------------------------------------------------------------- peaks


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured (MEASURED_PEAKS.json)"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback (earlier GB300 measurement)"}


# --------------------------------------------------------------------------- cudart events


class _Cudart:
    """Raw CUDA events through the runtime, so that event-record nodes can be
    placed inside a captured graph (cudaEventRecordExternal)."""

    def __init__(self):
        lib = None
        for name in ("libcudart.so.13", "/usr/local/cuda/lib64/libcudart.so.13",
                     "/usr/local/cuda/lib64/libcudart.so"):
            try:
                lib = ctypes.CDLL(name)
                break
            except OSError:
                continue
        if lib is None:
            raise RuntimeError("libcudart not found")
        self.lib = lib
        lib.cudaEventCreate.argtypes = [ctypes.POINTER(ctypes.c_void_p)]
        lib.cudaEventRecordWithFlags.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_uint]
        lib.cudaEventElapsedTime.argtypes = [ctypes.POINTER(ctypes.c_float), ctypes.c_void_p,
                                             ctypes.c_void_p]
        lib.cudaEventDestroy.argtypes = [ctypes.c_void_p]

    def create(self):
        ev = ctypes.c_void_p()
        rc = self.lib.cudaEventCreate(ctypes.byref(ev))
        if rc != 0:
            raise RuntimeError(f"cudaEventCreate failed ({rc})")
        return ev

    def record_external(self, ev):
        stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        rc = self.lib.cudaEventRecordWithFlags(ev, stream, 1)  # cudaEventRecordExternal
        if rc != 0:
            raise RuntimeError(f"cudaEventRecordWithFlags failed ({rc})")

    def elapsed_ms(self, a, b) -> float:
        ms = ctypes.c_float()
        rc = self.lib.cudaEventElapsedTime(ctypes.byref(ms), a, b)
        if rc != 0:
            raise RuntimeError(f"cudaEventElapsedTime failed ({rc})")
        return float(ms.value)


# --------------------------------------------------------------------------- clocks


class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.device_index = device_index
        self.proc = None
        self.lines = []
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.device_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._reader = threading.Thread(target=self._read, daemon=True)
            self._reader.start()
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, which):
        if which == "start":
            self.t0 = time.time()
        else:
            self.t1 = time.time()

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for ts, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            rows.append((ts, parts))
        inside = [r for r in rows if self.t0 is not None and self.t0 <= r[0] <= (self.t1 or 1e30)]
        use = inside if inside else rows
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(p[0]) for _, p in use if p[0].replace(".", "").isdigit()]
        smax = [float(p[1]) for _, p in use if p[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for _, p in use:
            for name, val in zip(names, p[4:8]):
                if val.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(use),
                "samples_in_timed_region": len(inside)}


# --------------------------------------------------------------------------- workloads


def bf16_bits_host(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def graph_ms(fn, reps: int = 5) -> float:
    """Median device time (ms) of one replay of `fn` captured as a CUDA graph."""
    fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(g, stream=stream):
        fn()
    g.replay()
    torch.cuda.synchronize()
    times = []
    for _ in range(reps):
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        g.replay()
        e.record()
        torch.cuda.synchronize()
        times.append(s.elapsed_time(e))
    del g
    return statistics.median(times)


def eager_us(fn, reps: int = 200) -> float:
    """Mean wall time of one eager call (launch latency included), in us."""
    for _ in range(10):
        fn()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(reps):
        fn()
    torch.cuda.synchronize()
    return (time.perf_counter() - t0) / reps * 1e6


def hbm_roofline(gbs: float, peaks: dict, traffic=None) -> dict:
    return {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": gbs / peaks["hbm_gbs"], "traffic": traffic, "peak_source": peaks["source"]}


def tensor_roofline(tflops: float, peaks: dict, key: str = "bf16_tflops") -> dict:
    return {"bound": "tensor", "achieved": tflops, "peak": peaks[key], "unit": "TFLOP/s",
            "frac": tflops / peaks[key], "traffic": None, "peak_source": peaks["source"]}


def host_cores() -> int:
    return os.cpu_count() or 1


class Tiny:
    """The tiny single layer (seed 0): W_base bf16 [256, 512] ~ N(0, 0.02),
    Δ ~ Laplace(0, 1e-3), compress with α per matrix and per row, then the
    fused linear on x [4, 512]; and the 8x16 case with |Δ| = 2^-10 whose
    reconstruction is exact.  Launch-bound: reported as latency per call."""

    name = "tiny_256x512_M4_alpha_per_matrix_and_per_row_plus_8x16_exact"

    def __init__(self, bd):
        import synth
        self.bd = bd
        self.wb_h, self.wf_h = synth.layer(0, 256, 512)
        self.x_h = synth.activations(0, 4, 512)
        self.cb_h, self.cf_h, _ = synth.constant_magnitude_case(0)
        dev = lambda b: torch.from_numpy(b.view(np.int16)).cuda().view(torch.bfloat16)
        self.wb, self.wf, self.x = dev(self.wb_h), dev(self.wf_h), dev(self.x_h)
        self.cb, self.cf = dev(self.cb_h), dev(self.cf_h)

    def report(self):
        bd = self.bd
        out = {"workload": self.name}
        for per_row in (False, True):
            tag = "alpha_per_row" if per_row else "alpha_per_matrix"
            packed, alpha = bd.bitdelta_compress(self.wb, self.wf, per_row=per_row)
            ws = torch.empty(max(bd.bitdelta_compress_workspace_bytes(256, 512, per_row), 1),
                             dtype=torch.uint8, device="cuda")
            y = torch.empty((4, 256), dtype=torch.bfloat16, device="cuda")
            out[f"compress_{tag}_us"] = eager_us(lambda: bd.bitdelta_compress(
                self.wb, self.wf, per_row=per_row, packed_out=packed, alpha_out=alpha,
                workspace=ws))
            out[f"linear_{tag}_us"] = eager_us(lambda: bd.bitdelta_linear(
                self.x, self.wb, packed, alpha, per_row=per_row, out=y))
        cp, ca = bd.bitdelta_compress(self.cb, self.cf, per_row=True)
        w8 = torch.empty_like(self.cb)
        out["exact_8x16_compress_plus_reconstruct_us"] = eager_us(
            lambda: (bd.bitdelta_compress(self.cb, self.cf, per_row=True, packed_out=cp,
                                          alpha_out=ca),
                     bd.bitdelta_reconstruct(self.cb, cp, ca, per_row=True, out=w8)))
        out["note"] = ("eager calls from Python through the C ABI, launch latency included "
                       "(wall time per call, synchronised once per 200 calls)")
        return out

    def oracle_sample(self):
        import oracle
        t = {}
        for per_row in (False, True):
            tag = "alpha_per_row" if per_row else "alpha_per_matrix"
            t0 = time.perf_counter()
            for _ in range(20):
                p_, a_, _ = oracle.compress(self.wb_h, self.wf_h, per_row)
            t[f"compress_{tag}_us"] = (time.perf_counter() - t0) / 20 * 1e6
            t0 = time.perf_counter()
            for _ in range(20):
                oracle.linear(self.x_h, self.wb_h, p_, a_, per_row)
            t[f"linear_{tag}_us"] = (time.perf_counter() - t0) / 20 * 1e6
        return {"value": t["linear_alpha_per_row_us"], "unit": "us per linear call",
                "cores": 1, "kind": "oracle", "per_call_us": t,
                "sample": "the whole tiny workload, 20 calls of each, 1 host core of "
                          f"{host_cores()}"}


class DecodeStack:
    """Decode sweep on 4096x4096 layers (alpha per row), 32 distinct layers."""

    name = "decode_sweep_4096x4096_alpha_per_row_M1-16_stack32"
    d_out = d_in = 4096
    Ms = (1, 2, 4, 8, 16)
    L = 32

    def __init__(self, bd, seed: int = 1):
        import synth.device as sd
        self.bd = bd
        self.layers = []
        for l in range(self.L):
            wb, wf = sd.layer(seed, self.d_out, self.d_in, stream=l)
            packed = torch.empty((self.d_out, self.d_in // 8), dtype=torch.uint8, device="cuda")
            alpha = torch.empty((self.d_out,), dtype=torch.float32, device="cuda")
            bd.bitdelta_compress(wb, wf, per_row=True, packed_out=packed, alpha_out=alpha)
            self.layers.append((wb, wf, packed, alpha))
        self.x = sd.normal_bf16((max(self.Ms), self.d_in), seed, 9999)
        self.w_eff = torch.empty((self.d_out, self.d_in), dtype=torch.bfloat16, device="cuda")
        self.y = {M: torch.empty((M, self.d_out), dtype=torch.bfloat16, device="cuda")
                  for M in self.Ms}
        torch.cuda.synchronize()
        n = self.d_out * self.d_in
        self.bytes = {
            "compress": n * (4 + 1 / 8) + 4 * self.d_out,
            "reconstruct": n * (4 + 1 / 8) + 4 * self.d_out,
        }
        for M in self.Ms:
            self.bytes[f"linear_M{M}"] = n * (2 + 1 / 8) + 4 * self.d_out + 2 * M * (
                self.d_in + self.d_out)
        self.phases = ["compress", "reconstruct"] + [f"linear_M{M}" for M in self.Ms]

    def launches_per_step(self):
        return len(self.phases) * self.L

    def bytes_per_step(self):
        return sum(self.bytes[p] for p in self.phases) * self.L

    def run_phase(self, phase):
        bd = self.bd
        for (wb, wf, packed, alpha) in self.layers:
            if phase == "compress":
                bd.bitdelta_compress(wb, wf, per_row=True, packed_out=packed, alpha_out=alpha)
            elif phase == "reconstruct":
                bd.bitdelta_reconstruct(wb, packed, alpha, per_row=True, out=self.w_eff)
            else:
                M = int(phase.split("M")[1])
                bd.bitdelta_linear(self.x[:M], wb, packed, alpha, per_row=True, out=self.y[M])

    def dominant(self):
        return [p for p in self.phases if p.startswith("linear")]

    def unfused_timing(self):
        """The unfused reference on the same 32-layer stack: bitdelta_reconstruct
        of W_eff to memory, then cuBLAS bf16 x·W_effᵀ, per layer and M.  Rates
        are the fused op's algorithmic bytes over the unfused time."""
        bd = self.bd
        out = {}
        for M in self.Ms:
            def f():
                for (wb, wf, packed, alpha) in self.layers:
                    bd.bitdelta_reconstruct(wb, packed, alpha, per_row=True, out=self.w_eff)
                    torch.matmul(self.x[:M], self.w_eff.T, out=self.y[M])
            ms = graph_ms(f)
            us = ms * 1e3 / self.L
            out[f"M{M}"] = {"us_per_layer": us,
                            "GB/s_of_fused_bytes": self.bytes[f"linear_M{M}"] / (us * 1e-6) / 1e9}
        return out

    # ---------------------------------------------------------------- oracle

    def oracle_sample(self, budget_s: float):
        """Time the oracle on one layer's worth of the step (host arrays)."""
        import oracle
        wb, wf, packed, alpha = self.layers[0]
        wb_h, wf_h = bf16_bits_host(wb), bf16_bits_host(wf)
        x_h = bf16_bits_host(self.x)
        reps, t_total = 0, 0.0
        while True:
            t0 = time.perf_counter()
            p_h, a_h, _ = oracle.compress(wb_h, wf_h, True)
            oracle.reconstruct(wb_h, p_h, a_h, True)
            for M in self.Ms:
                oracle.linear(x_h[:M], wb_h, p_h, a_h, True)
            t_total += time.perf_counter() - t0
            reps += 1
            if t_total >= budget_s or reps >= 50:
                break
        per_layer_bytes = sum(self.bytes[p] for p in self.phases)
        return {"value": per_layer_bytes * reps / t_total / 1e9, "unit": "GB/s", "cores": 1,
                "kind": "oracle",
                "sample": f"{reps} x one 4096x4096 layer of the step (compress, reconstruct, "
                          f"linear M=1,2,4,8,16) on 1 host core, {t_total:.1f} s"}


class Prefill:
    """Prefill GEMMs, M = 2048 tokens, Llama-70B projections, alpha per row."""

    name = "prefill_M2048_llama70b_qkv_o_gateup_down_alpha_per_row"
    M = 2048
    shapes = [("qkv", 10240, 8192), ("o", 8192, 8192), ("gate_up", 57344, 8192),
              ("down", 8192, 28672)]

    def __init__(self, bd, seed: int = 3):
        import synth.device as sd
        self.bd = bd
        self.mats = {}
        for i, (nm, d_out, d_in) in enumerate(self.shapes):
            wb, wf = sd.layer(seed, d_out, d_in, stream=i)
            packed, alpha = bd.bitdelta_compress(wb, wf, per_row=True)
            del wf
            self.mats[nm] = (wb, packed, alpha)
        self.x = {d_in: sd.normal_bf16((self.M, d_in), seed, 5000 + d_in)
                  for d_in in sorted({s[2] for s in self.shapes})}
        self.y = {nm: torch.empty((self.M, d_out), dtype=torch.bfloat16, device="cuda")
                  for nm, d_out, _ in self.shapes}
        torch.cuda.synchronize()
        self.flops = {nm: 2.0 * self.M * d_out * d_in for nm, d_out, d_in in self.shapes}
        self.phases = [nm for nm, _, _ in self.shapes]
        # split-schedule workspace (bitdelta_linear_ws): one for every shape
        need = max(bd.bitdelta_linear_workspace_bytes(self.M, d_out, d_in)
                   for _, d_out, d_in in self.shapes)
        self.ws = torch.empty(max(need, 1), dtype=torch.uint8, device="cuda") if need else None
        self.split = True

    def linear(self, x, wb, packed, alpha, y):
        if self.split:
            self.bd.bitdelta_linear_ws(x, wb, packed, alpha, self.ws, per_row=True, out=y)
        else:
            self.bd.bitdelta_linear(x, wb, packed, alpha, per_row=True, out=y)

    def launches_per_step(self):
        return len(self.phases)

    def flops_per_step(self):
        return sum(self.flops.values())

    def run_phase(self, phase):
        d_in = dict((nm, di) for nm, _, di in self.shapes)[phase]
        wb, packed, alpha = self.mats[phase]
        self.linear(self.x[d_in], wb, packed, alpha, self.y[phase])

    def oracle_sample(self):
        """The oracle on 16 of the 2048 tokens through the O projection
        (8192 -> 8192): compression untimed, the linear timed; the FLOP rate
        extrapolates to the whole step (labelled so)."""
        import oracle
        import synth.device as sd
        nm, d_out, d_in = self.shapes[1]
        wb, wf = sd.layer(3, d_out, d_in, stream=1)
        wb_h, wf_h = bf16_bits_host(wb), bf16_bits_host(wf)
        del wb, wf
        x_h = bf16_bits_host(self.x[d_in][:16])
        packed, alpha, _ = oracle.compress(wb_h, wf_h, True)
        t0 = time.perf_counter()
        oracle.linear(x_h, wb_h, packed, alpha, True)
        dt = time.perf_counter() - t0
        tflops = 2.0 * 16 * d_out * d_in / dt / 1e12
        return {"value": tflops, "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
                "extrapolated_ms_per_step": self.flops_per_step() / (tflops * 1e12) * 1e3,
                "sample": f"16 of {self.M} tokens through the O projection ({d_in}->{d_out}), "
                          f"{dt:.1f} s on 1 host core of {host_cores()}; the step time is "
                          "extrapolated from that FLOP rate"}

    def cublas_reference(self, reps=5):
        """cuBLAS bf16 GEMM x·W_baseᵀ, and reconstruct-to-HBM + cuBLAS (unfused)."""
        out = {}
        w_eff = {nm: torch.empty_like(self.mats[nm][0]) for nm in self.phases}
        for mode in ("cublas_plain", "unfused"):
            times = []
            for _ in range(reps + 2):
                s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                s.record()
                for nm, d_out, d_in in self.shapes:
                    wb, packed, alpha = self.mats[nm]
                    if mode == "unfused":
                        self.bd.bitdelta_reconstruct(wb, packed, alpha, per_row=True,
                                                     out=w_eff[nm])
                        torch.matmul(self.x[d_in], w_eff[nm].T, out=self.y[nm])
                    else:
                        torch.matmul(self.x[d_in], wb.T, out=self.y[nm])
                e.record()
                torch.cuda.synchronize()
                times.append(s.elapsed_time(e))
            t = statistics.median(times[2:])
            out[mode] = {"ms_per_step": t, "tflops": self.flops_per_step() / (t * 1e-3) / 1e12}
        # fused against unfused at fewer tokens (same four shapes, eager launches
        # for both): the unfused path pays its reconstruct once per weight, the
        # fused kernel its transform once per token tile (256 or 512 tokens)
        out["fused_vs_unfused_by_tokens"] = {}
        for m in (512, 1024):
            res = {}
            for mode in ("fused", "unfused"):
                times = []
                for _ in range(reps + 2):
                    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    s.record()
                    for nm, d_out, d_in in self.shapes:
                        wb, packed, alpha = self.mats[nm]
                        x = self.x[d_in][:m]
                        y = self.y[nm][:m]
                        if mode == "unfused":
                            self.bd.bitdelta_reconstruct(wb, packed, alpha, per_row=True,
                                                         out=w_eff[nm])
                            torch.matmul(x, w_eff[nm].T, out=y)
                        else:
                            self.linear(x, wb, packed, alpha, y)
                    e.record()
                    torch.cuda.synchronize()
                    times.append(s.elapsed_time(e))
                t = statistics.median(times[2:])
                fl = self.flops_per_step() * m / self.M
                res[mode] = {"ms_per_step": t, "tflops": fl / (t * 1e-3) / 1e12}
            out["fused_vs_unfused_by_tokens"][f"M{m}"] = res
        del w_eff
        return out


class Grouped:
    """Multi-tenant: shared W_base 4096->14336, 14 variants, 64 decode rows +
    4 prefill segments of 512, ids uniform over {base, 1..14}."""

    name = "grouped_W4096x14336_14variants_64decode_4x512prefill"
    d_out, d_in, n_var = 14336, 4096, 14
    sets = 3   # rotating copies of W_base + deltas (3 x 220 MB > L2)

    def __init__(self, bd, seed: int = 4):
        import synth
        import synth.device as sd
        self.bd = bd
        scales = synth.variant_scales(seed, self.n_var)
        lengths = [1] * 64 + [512] * 4
        off, var = synth.segments(seed, lengths, self.n_var)
        self.off = torch.from_numpy(off).cuda()
        self.var = torch.from_numpy(var).cuda()
        self.var_host = var
        self.M = int(off[-1])
        self.copies = []
        for c in range(self.sets):
            wb = sd.normal_bf16((self.d_out, self.d_in), seed, 100 + c, 0.02)
            packs, alphas = [], []
            for v in range(self.n_var):
                wf = sd.finetuned_bf16(wb, seed, 1000 + 100 * c + v, float(scales[v]))
                p, a = bd.bitdelta_compress(wb, wf, per_row=True)
                del wf
                packs.append(p)
                alphas.append(a)
            pt, at = bd.variant_tables(packs, alphas, "cuda")
            self.copies.append((wb, packs, alphas, pt, at))
        self.x = sd.normal_bf16((self.M, self.d_in), seed, 77)
        self.y = torch.empty((self.M, self.d_out), dtype=torch.bfloat16, device="cuda")
        torch.cuda.synchronize()
        self.flops = 2.0 * self.M * self.d_in * self.d_out
        distinct = len(set(int(v) for v in var if v > 0))
        n = self.d_out * self.d_in
        self.bytes = (2 * n + distinct * (n / 8 + 4 * self.d_out) + 2 * self.M * self.d_in
                      + 2 * self.M * self.d_out)
        self.phases = [f"set{c}" for c in range(self.sets)]

    def launches_per_step(self):
        return 2 * self.sets   # tensor-core kernel + decode kernel per call

    def unfused_timing(self):
        """The unfused reference for one call on copy 0: for each variant in
        the batch, bitdelta_reconstruct of its W_eff to memory, then cuBLAS
        bf16 products of that variant's rows (gathered, multiplied,
        scattered); base rows multiply W_base directly."""
        bd = self.bd
        wb, packs, alphas, _, _ = self.copies[0]
        off = self.off.cpu().numpy()
        rows_of = {}
        for s_, v in enumerate(self.var_host):
            rows_of.setdefault(int(v), []).extend(range(int(off[s_]), int(off[s_ + 1])))
        idx = {v: torch.tensor(r, dtype=torch.int64, device="cuda") for v, r in rows_of.items()}
        w_eff = torch.empty_like(wb)
        y = torch.empty_like(self.y)

        def f():
            for v, ix in idx.items():
                w = wb
                if v > 0:
                    bd.bitdelta_reconstruct(wb, packs[v - 1], alphas[v - 1], per_row=True,
                                            out=w_eff)
                    w = w_eff
                y.index_copy_(0, ix, torch.matmul(self.x.index_select(0, ix), w.T))
        ms = graph_ms(f)
        return {"ms_per_call": ms, "TFLOP/s": self.flops / (ms * 1e-3) / 1e12,
                "variants_reconstructed": len([v for v in idx if v > 0])}

    def oracle_sample(self):
        """The oracle on 16 rows of one call (8 of the one-row decode segments
        and 2 rows of each 512-row segment, each as a one-row segment of its
        variant); compression of the variants involved untimed.  Rows/s
        extrapolate to the whole call (labelled so)."""
        import oracle
        import synth
        import synth.device as sd
        wb = self.copies[0][0]
        wb_h = bf16_bits_host(wb)
        off = self.off.cpu().numpy()
        rows, n_decode = [], 0
        for s_ in range(len(self.var_host)):
            a, b = int(off[s_]), int(off[s_ + 1])
            if b - a == 1 and n_decode < 8:
                rows.append(a)
                n_decode += 1
            elif b - a > 1:
                rows.extend([a, b - 1])
        rows = np.array(sorted(rows))
        seg_of = np.searchsorted(off, rows, side="right") - 1
        var = self.var_host[seg_of].astype(np.int32)
        scales = synth.variant_scales(4, self.n_var)
        packs, alphas = [], []
        for v in range(1, self.n_var + 1):
            if v in set(int(u) for u in var):
                wf = sd.finetuned_bf16(wb, 4, 1000 + v - 1, float(scales[v - 1]))
                p_, a_, _ = oracle.compress(wb_h, bf16_bits_host(wf), True)
                del wf
            else:   # not referenced by the sample: any table entry of the right shape
                p_ = np.zeros((self.d_out, self.d_in // 8), np.uint8)
                a_ = np.zeros(self.d_out, np.float32)
            packs.append(p_)
            alphas.append(a_)
        x_h = bf16_bits_host(self.x[torch.from_numpy(rows).cuda()])
        sub_off = np.arange(len(rows) + 1, dtype=np.int32)
        t0 = time.perf_counter()
        oracle.linear_grouped(x_h, sub_off, var, wb_h, packs, alphas, True)
        dt = time.perf_counter() - t0
        rps = len(rows) / dt
        return {"value": rps, "unit": "rows/s", "cores": 1, "kind": "oracle",
                "extrapolated_ms_per_call": self.M / rps * 1e3,
                "sample": f"{len(rows)} of the call's {self.M} rows, {dt:.1f} s on 1 host core "
                          f"of {host_cores()}; the call time is extrapolated from that row rate"}

    def run_phase(self, phase):
        c = int(phase[3:])
        wb, packs, alphas, pt, at = self.copies[c]
        self.bd.bitdelta_linear_grouped(self.x, self.off, self.var, wb, pt, at, n_var=self.n_var,
                                        max_seg_len=512, per_row=True, out=self.y)


class Slice40:
    """A 40-layer slice of a Llama-70B-sized model: per layer QKV 8192->10240,
    O 8192->8192, gate+up 8192->57344, down 28672->8192 (855.6M weights per
    layer, 68.45 GB of bf16 base weights), two compressed variants resident
    (per-row α), and per layer the compression of a third variant whose
    fine-tuned weights are drawn on the device one layer at a time.

    Phases: "prefill" (512 tokens of variant 1 through all 160 projections),
    "decode" (batch of 8 rows alternating variants 1, 2, 1, 2, ... as eight
    one-row segments of the grouped linear, all 160 projections) and
    "compress" (variant 3, all 160 projections; its W_ft is drawn outside
    the timed kernels).  Each projection takes a fresh N(0,1) input of its
    width: the projections are not chained through attention."""

    name = "slice40_llama70b_prefill512_decode8x2variants_compress3rd"
    L = 40
    shapes = Prefill.shapes
    prefill_M = 512   # synth.device.SLICE_PREFILL_TOKENS
    decode_M = 8      # synth.device.SLICE_DECODE_ROWS

    def __init__(self, bd, seed: int = 5):
        import synth.device as sd
        self.bd = bd
        self.layers = []
        for l in range(self.L):
            mats = {}
            for i, (nm, d_out, d_in) in enumerate(self.shapes):
                wb = sd.slice_base(l, i, seed)
                var = []
                for v in (1, 2):
                    wf = sd.slice_finetuned(wb, l, i, v, seed)
                    var.append(bd.bitdelta_compress(wb, wf, per_row=True))
                    del wf
                pt, at = bd.variant_tables([var[0][0], var[1][0]], [var[0][1], var[1][1]], "cuda")
                mats[nm] = (wb, var, pt, at)
            self.layers.append(mats)
        self.seed = seed
        widths = sorted({d_in for _, _, d_in in self.shapes})
        self.xp = {d: sd.slice_inputs(d, self.prefill_M, False, seed) for d in widths}
        self.xd = {d: sd.slice_inputs(d, self.decode_M, True, seed) for d in widths}
        self.yp = {nm: torch.empty((self.prefill_M, d_out), dtype=torch.bfloat16, device="cuda")
                   for nm, d_out, _ in self.shapes}
        self.yd = {nm: torch.empty((self.decode_M, d_out), dtype=torch.bfloat16, device="cuda")
                   for nm, d_out, _ in self.shapes}
        off = np.arange(self.decode_M + 1, dtype=np.int32)
        var = np.array([1 + (r % 2) for r in range(self.decode_M)], np.int32)
        self.seg_off = torch.from_numpy(off).cuda()
        self.seg_var = torch.from_numpy(var).cuda()
        # one layer's worth of variant-3 buffers, reused layer after layer
        self.wf3 = {nm: torch.empty((d_out, d_in), dtype=torch.bfloat16, device="cuda")
                    for nm, d_out, d_in in self.shapes}
        self.p3 = {nm: torch.empty((d_out, d_in // 8), dtype=torch.uint8, device="cuda")
                   for nm, d_out, d_in in self.shapes}
        self.a3 = {nm: torch.empty((d_out,), dtype=torch.float32, device="cuda")
                   for nm, d_out, _ in self.shapes}
        torch.cuda.synchronize()
        n = sum(d_out * d_in for _, d_out, d_in in self.shapes)
        self.weights_per_layer = n
        self.prefill_flops = 2.0 * self.prefill_M * n * self.L
        # decode: W_base once + both variants' signs and α + x + y, per layer
        rows = sum(d_out for _, d_out, _ in self.shapes)
        self.decode_bytes = self.L * (2 * n + 2 * (n / 8 + 4 * rows)
                                      + 2 * self.decode_M * sum(d_in + d_out
                                                                for _, d_out, d_in in self.shapes))
        # compress: W_base + W_ft read, signs + α written, per layer
        self.compress_bytes = self.L * (4 * n + n / 8 + 4 * rows)

    def run_prefill(self):
        for mats in self.layers:
            for nm, d_out, d_in in self.shapes:
                wb, var, _, _ = mats[nm]
                self.bd.bitdelta_linear(self.xp[d_in], wb, var[0][0], var[0][1], per_row=True,
                                        out=self.yp[nm])

    def run_decode(self):
        for mats in self.layers:
            for nm, d_out, d_in in self.shapes:
                wb, _, pt, at = mats[nm]
                self.bd.bitdelta_linear_grouped(self.xd[d_in], self.seg_off, self.seg_var, wb, pt,
                                                at, n_var=2, max_seg_len=1, per_row=True,
                                                out=self.yd[nm])

    def timed(self, fn, reps=3):
        fn()
        torch.cuda.synchronize()
        times = []
        for _ in range(reps):
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record()
            fn()
            e.record()
            torch.cuda.synchronize()
            times.append(s.elapsed_time(e))
        return statistics.median(times)

    def compress_ms(self):
        """Per layer: draw variant 3's W_ft (untimed), then time its four
        compress calls with CUDA events; returns the sum over the 40 layers."""
        import synth.device as sd
        total = 0.0
        for l, mats in enumerate(self.layers):
            for i, (nm, d_out, d_in) in enumerate(self.shapes):
                sd.slice_finetuned(mats[nm][0], l, i, 3, self.seed, out=self.wf3[nm])
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record()
            for nm, d_out, d_in in self.shapes:
                self.bd.bitdelta_compress(mats[nm][0], self.wf3[nm], per_row=True,
                                          packed_out=self.p3[nm], alpha_out=self.a3[nm])
            e.record()
            torch.cuda.synchronize()
            total += s.elapsed_time(e)
        return total

    def run_decode_unfused(self, w_eff):
        """The unfused reference of the decode step: per projection, each
        variant's W_eff reconstructed to memory, then cuBLAS bf16 products of
        that variant's rows."""
        rows = {v: torch.tensor([r for r in range(self.decode_M) if 1 + r % 2 == v],
                                dtype=torch.int64, device="cuda") for v in (1, 2)}
        for mats in self.layers:
            for nm, d_out, d_in in self.shapes:
                wb, var, _, _ = mats[nm]
                w = w_eff[:d_out * d_in].view(d_out, d_in)
                for v in (1, 2):
                    self.bd.bitdelta_reconstruct(wb, var[v - 1][0], var[v - 1][1], per_row=True,
                                                 out=w)
                    self.yd[nm].index_copy_(0, rows[v], torch.matmul(
                        self.xd[d_in].index_select(0, rows[v]), w.T))

    def oracle_sample(self):
        """The oracle on the O projection (8192 -> 8192) of layer 0: the third
        variant's compression, the decode batch (8 rows alternating variants
        1 and 2, their compression untimed) and 4 of the 512 prefill tokens of
        variant 1, each timed on 1 host core; per-leg rates over the same
        algorithmic bytes or FLOPs as the GPU legs."""
        import oracle
        import synth.device as sd
        proj = 1
        nm, d_out, d_in = self.shapes[proj]
        wb = self.layers[0][nm][0]
        wb_h = bf16_bits_host(wb)
        fts = {v: bf16_bits_host(sd.slice_finetuned(wb, 0, proj, v, self.seed)) for v in (1, 2, 3)}
        n = d_out * d_in
        t0 = time.perf_counter()
        oracle.compress(wb_h, fts[3], True)
        t_comp = time.perf_counter() - t0
        comp = {v: oracle.compress(wb_h, fts[v], True) for v in (1, 2)}
        xd = bf16_bits_host(self.xd[d_in])
        off = np.arange(self.decode_M + 1, dtype=np.int32)
        var = np.array([1 + r % 2 for r in range(self.decode_M)], np.int32)
        t0 = time.perf_counter()
        oracle.linear_grouped(xd, off, var, wb_h, [comp[1][0], comp[2][0]],
                              [comp[1][1], comp[2][1]], True)
        t_dec = time.perf_counter() - t0
        xp = bf16_bits_host(self.xp[d_in][:4])
        t0 = time.perf_counter()
        oracle.linear(xp, wb_h, comp[1][0], comp[1][1], True)
        t_pre = time.perf_counter() - t0
        dec_bytes = 2 * n + 2 * (n / 8 + 4 * d_out) + 2 * self.decode_M * (d_in + d_out)
        return {"value": dec_bytes / t_dec / 1e9, "unit": "GB/s (decode leg)", "cores": 1,
                "kind": "oracle",
                "compress_GB/s": (4 * n + n / 8 + 4 * d_out) / t_comp / 1e9,
                "prefill_TFLOP/s": 2.0 * 4 * n / t_pre / 1e12,
                "sample": f"the O projection ({d_in}->{d_out}) of layer 0: compression of the "
                          f"third variant ({t_comp:.1f} s), the 8-row decode batch "
                          f"({t_dec:.1f} s), 4 of 512 prefill tokens ({t_pre:.1f} s), on 1 "
                          f"host core of {host_cores()}"}

    def report(self, peaks, cpu: bool = True):
        pre = self.timed(self.run_prefill)
        dec = self.timed(self.run_decode)
        comp = self.compress_ms()
        pre_tf = self.prefill_flops / (pre * 1e-3) / 1e12
        dec_gbs = self.decode_bytes / (dec * 1e-3) / 1e9
        comp_gbs = self.compress_bytes / (comp * 1e-3) / 1e9
        w_eff = torch.empty(max(d_out * d_in for _, d_out, d_in in self.shapes),
                            dtype=torch.bfloat16, device="cuda")
        dec_unfused = self.timed(lambda: self.run_decode_unfused(w_eff), reps=2)
        del w_eff
        return {
            "workload": self.name,
            "prefill": {"ms": pre, "TFLOP/s": pre_tf, "tokens": self.prefill_M,
                        "launches": 4 * self.L,
                        "roofline": tensor_roofline(pre_tf, peaks, "bf16_tflops_sustained")},
            "decode": {"ms_per_step": dec, "GB/s": dec_gbs,
                       "batch": self.decode_M, "variants": "rows alternate 1,2,1,2,...",
                       "launches": 4 * self.L, "roofline": hbm_roofline(dec_gbs, peaks),
                       "unfused_reconstruct_plus_cublas_ms_per_step": dec_unfused},
            "compress": {"ms": comp, "GB/s": comp_gbs, "ms_per_layer": comp / self.L,
                         "roofline": hbm_roofline(comp_gbs, peaks)},
            "resident_weights_gb": (2 * self.weights_per_layer * self.L
                                    + 2 * self.L * (self.weights_per_layer / 8)) / 1e9,
            "cpu_baseline": self.oracle_sample() if cpu else None,
        }


class DeltaCacheLoads:
    """The delta cache's cold loads: variants of 1 GiB each (packed signs and
    α of about 17 GB of bf16 weights) in pinned host memory, a device arena of
    two slots, requests cycling over four variants so every request after the
    first two evicts and loads.  Reports the copy bandwidth and the time a
    full 70B-model delta (8.75 GB, the page's figure) would take at it."""

    name = "delta_cache_cold_loads_4x1GiB_variants_2_slots"
    blob = 1 << 30

    def __init__(self, bd):
        self.bd = bd
        self.blobs = []
        for v in range(4):
            b = torch.empty(self.blob, dtype=torch.uint8).pin_memory()
            b.fill_(v + 1)
            self.blobs.append(b)
        arena = torch.empty(2 * self.blob, dtype=torch.uint8, device="cuda")
        self.cache = bd.DeltaCache(arena, self.blob, pin_top_k=0)
        for v, b in enumerate(self.blobs):
            self.cache.register(v, b)

    def report(self, requests: int = 12):
        cache = self.cache
        stream = torch.cuda.current_stream()
        cache.acquire(0)
        cache.release(0)
        stream.synchronize()
        base = cache.stats()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0 = time.perf_counter()
        s.record()
        host_us = []
        for i in range(requests):
            v = 1 + i % 3          # 1, 2, 3, 1, ...: with two slots, every request misses
            h0 = time.perf_counter()
            cache.acquire(v)
            host_us.append((time.perf_counter() - h0) * 1e6)
            cache.release(v)
        e.record()
        stream.synchronize()
        wall = time.perf_counter() - t0
        ms = s.elapsed_time(e)
        st = cache.stats()
        loaded = st["bytes_loaded"] - base["bytes_loaded"]
        gbs = loaded / (ms * 1e-3) / 1e9
        last = 1 + (requests - 1) % 3   # the variant requested last is resident
        h0 = time.perf_counter()
        for _ in range(100):       # hits: acquire and release of a resident variant
            cache.acquire(last)
            cache.release(last)
        hit_us = (time.perf_counter() - h0) / 100 * 1e6
        return {
            "workload": self.name, "loads": st["loads"] - base["loads"],
            "bytes_loaded": loaded, "ms": ms, "wall_s": wall, "GB/s": gbs,
            "ms_for_8.75GB_delta": 8.75e9 / (gbs * 1e9) * 1e3,
            "page_ms_for_8.75GB_delta": 200.0,
            "acquire_host_us_median_on_miss": statistics.median(host_us),
            "acquire_release_host_us_on_hit": hit_us,
            "evictions": st["evictions"] - base["evictions"],
        }

    def close(self):
        self.cache.close()


class DecodeLarge:
    """bitdelta_linear decode on the 40-layer slice's largest projection
    (gate+up, W_base 8192 -> 57344, 940 MB per layer), per-row α, at M = 1, 8
    and 16, two distinct layers alternating (1.9 GB, far beyond L2): the
    kernel's steady-state streaming rate, without the per-launch ramp that
    bounds the 4096 x 4096 layers of the headline sweep."""

    name = "decode_large_57344x8192_alpha_per_row_M1_8_16_2layers"
    d_out, d_in, n_layers = 57344, 8192, 2

    def __init__(self, bd, seed: int = 6):
        import synth.device as sd
        self.bd = bd
        self.layers = []
        for l in range(self.n_layers):
            wb = sd.normal_bf16((self.d_out, self.d_in), seed, 2 * l + 1, 0.02)
            wf = sd.finetuned_bf16(wb, seed, 2 * l + 2, 1e-3)
            p, a = bd.bitdelta_compress(wb, wf, per_row=True)
            del wf
            self.layers.append((wb, p, a))
        self.x = sd.normal_bf16((16, self.d_in), seed, 99)

    def report(self, peaks, reps: int = 4):
        out = {"workload": self.name}
        for M in (1, 8, 16):
            y = torch.empty((M, self.d_out), dtype=torch.bfloat16, device="cuda")
            x = self.x[:M]

            def f():
                for _ in range(reps):
                    for wb, p, a in self.layers:
                        self.bd.bitdelta_linear(x, wb, p, a, per_row=True, out=y)

            ms = graph_ms(f) / (reps * self.n_layers)
            byts = (self.d_out * self.d_in * (2 + 1 / 8) + 4 * self.d_out
                    + 2 * M * (self.d_in + self.d_out))
            gbs = byts / (ms * 1e-3) / 1e9
            out[f"M{M}"] = {"us_per_launch": ms * 1e3, "GB/s": gbs,
                            "roofline": hbm_roofline(gbs, peaks),
                            "kernel": "gemv_single_async_kernel" if M <= 8
                            else "gemv_single_kernel (grid of 3584 CTAs: several waves)"}
        return out


class KMergeSimilarity:
    """K-Merge's first step on the grouped workload's layer (W_base
    4096->14336, 14 variants): the cosine similarity of variant 1's 1-bit task
    vector with the other 13 and the most similar of them.  Reads 14 packed
    sign matrices of 7.34 MB (plus α)."""

    name = "kmerge_similarity_14336x4096_1_vs_13"
    d_out, d_in, n_var = 14336, 4096, 14

    def __init__(self, bd, seed: int = 4):
        import synth
        import synth.device as sd
        self.bd = bd
        scales = synth.variant_scales(seed, self.n_var)
        wb = sd.normal_bf16((self.d_out, self.d_in), seed, 100, 0.02)
        self.packs, self.alphas = [], []
        for v in range(self.n_var):
            wf = sd.finetuned_bf16(wb, seed, 1000 + v, float(scales[v]))
            p, a = bd.bitdelta_compress(wb, wf, per_row=True)
            self.packs.append(p)
            self.alphas.append(a)
            del wf
        self.pt, self.at = bd.variant_tables(self.packs[1:], self.alphas[1:], "cuda")
        self.bytes = self.n_var * (self.d_out * self.d_in / 8 + 4 * self.d_out)

    def report(self, reps=50):
        n_b = self.n_var - 1
        cos = torch.empty(n_b, dtype=torch.float64, device="cuda")
        best = torch.empty(1, dtype=torch.int32, device="cuda")
        ws = torch.empty(self.bd.bitdelta_sign_similarity_workspace_bytes(self.d_out, n_b) + 256,
                         dtype=torch.uint8, device="cuda")
        f = lambda: self.bd.bitdelta_sign_similarity(self.packs[0], self.alphas[0], self.pt,
                                                     self.at, n_b, True, out=cos, best=best,
                                                     workspace=ws)
        f()
        torch.cuda.synchronize()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        for _ in range(reps):
            f()
        e.record()
        torch.cuda.synchronize()
        ms = s.elapsed_time(e) / reps
        return {"workload": self.name, "us_per_call": ms * 1e3,
                "GB/s": self.bytes / (ms * 1e-3) / 1e9, "most_similar_variant": int(best.item()) + 2,
                "cos_max": float(cos.max()), "cos_min": float(cos.min()),
                "note": "per call: a 4-byte memset of the workspace counter + the kernel"}


class MonoSoupMerge:
    """MonoSoup merge of k = 4 fine-tuned checkpoints of one 4096 x 4096 layer
    at rank 32 (two power iterations).  Each checkpoint's Δ_i is a rank-32
    signal plus Laplace(0, 1e-4) noise (synth.monosoup_checkpoints)."""

    name = "monosoup_4096x4096_k4_rank32_q2"
    d_out = d_in = 4096
    k, rank, q = 4, 32, 2

    def __init__(self, bd, seed: int = 6):
        import synth
        self.bd = bd
        wb = synth.base_weight(seed, self.d_out, self.d_in)
        ws = synth.monosoup_checkpoints(seed, wb, self.k, self.rank)
        dev = lambda b: torch.from_numpy(b.view(np.int16)).cuda().view(torch.bfloat16)
        self.wb = dev(wb)
        self.ws = [dev(w) for w in ws]
        self.out = torch.empty_like(self.wb)
        self.ws_buf = torch.empty(
            bd.bitdelta_monosoup_workspace_bytes(self.d_out, self.d_in, self.k, self.rank) + 256,
            dtype=torch.uint8, device="cuda")
        n = self.d_out * self.d_in
        passes = 2 * self.q + 2          # products with Δ_i per checkpoint
        # HBM bytes of the algorithm as run: each pass reads W_base once for all
        # k checkpoints and each W_i once (bf16); the merge reads W_base and
        # writes W_merged.  (The factors, a few MB, are left out.)
        self.bytes = passes * (self.k + 1) * 2 * n + 4 * n
        # fp32-equivalent work: Δ_i·V products and the rank-k·r merge
        self.flops = self.k * passes * 2 * n * self.rank + 2 * n * self.k * self.rank

    def report(self, reps=10):
        f = lambda: self.bd.bitdelta_monosoup(self.wb, self.ws, self.rank, power_iters=self.q,
                                              seed=1, out=self.out, workspace=self.ws_buf)
        for _ in range(2):
            f()
        torch.cuda.synchronize()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        for _ in range(reps):
            f()
        e.record()
        torch.cuda.synchronize()
        ms = s.elapsed_time(e) / reps
        peaks = load_peaks()
        gbs = self.bytes / (ms * 1e-3) / 1e9
        tflops = self.flops / (ms * 1e-3) / 1e12
        # 18 FLOP per byte, far below the bf16 tensor balance (~280): HBM-bound
        return {"workload": self.name, "ms_per_merge": ms, "GB/s": gbs,
                "TFLOP/s_fp32_equivalent": tflops,
                "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"],
                             "unit": "GB/s", "frac": gbs / peaks["hbm_gbs"], "traffic": None,
                             "peak_source": peaks["source"]},
                "algorithmic": {"bytes": self.bytes, "flops": self.flops,
                                "note": "Delta products and merge on the tensor cores "
                                        "(bf16 terms, fp32 accumulation)"}}


# --------------------------------------------------------------------------- timing


def capture_steps(cudart, wl, steps):
    """Capture `steps` steps of workload `wl` into one CUDA graph with an
    event-record node at every phase boundary.  Returns (graph, events)."""
    n_ev = steps * len(wl.phases) + 1
    events = [cudart.create() for _ in range(n_ev)]
    g = torch.cuda.CUDAGraph()
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(g, stream=stream):
        k = 0
        cudart.record_external(events[k])
        for _ in range(steps):
            for ph in wl.phases:
                wl.run_phase(ph)
                k += 1
                cudart.record_external(events[k])
    torch.cuda.synchronize()
    return g, events


def phase_times(cudart, wl, events, steps):
    """Mean duration (ms) of each phase over the captured steps."""
    acc = {ph: 0.0 for ph in wl.phases}
    k = 0
    for _ in range(steps):
        for ph in wl.phases:
            acc[ph] += cudart.elapsed_ms(events[k], events[k + 1])
            k += 1
    return {ph: acc[ph] / steps for ph in wl.phases}


def timed_run(cudart, wl, steps, warmup, dist, clock=None, graph_steps=None):
    """Warm-up, then `steps` steps as replays of a captured graph.  Returns
    (ms_per_step (max over ranks), phase means from the last replay)."""
    for _ in range(max(warmup, 1)):
        for ph in wl.phases:
            wl.run_phase(ph)
    torch.cuda.synchronize()
    per_graph = graph_steps or steps
    per_graph = max(1, min(per_graph, steps))
    g, events = capture_steps(cudart, wl, per_graph)
    g.replay()   # untimed replay of the captured graph (part of the warm-up)
    torch.cuda.synchronize()
    replays, rem = divmod(steps, per_graph)
    g_rem = None
    if rem:
        g_rem, _ = capture_steps(cudart, wl, rem)
        g_rem.replay()
        torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if clock:
        clock.mark("start")
    start.record()
    for _ in range(replays):
        g.replay()
    if g_rem is not None:
        g_rem.replay()
    end.record()
    torch.cuda.synchronize()
    if clock:
        clock.mark("end")
    if dist is not None:
        dist.barrier()
    ms = max_over_ranks(dist, start.elapsed_time(end) / steps)
    phases = phase_times(cudart, wl, events, per_graph) if replays > 0 else {}
    del g, g_rem
    return ms, phases


# --------------------------------------------------------------------------- e2e


def e2e_decode(bd, steps: int):
    """End to end through the public API: per step, pinned host -> device copy
    of one layer's inputs (W_base, W_ft, x), compress, reconstruct, fused
    linear at M = 1..16, device -> host copy of the results.  Steps are
    pipelined the way a server streams layers: two buffer sets, copies in on
    one stream, compute on a second, copies out on a third, ordered by events
    (step i's upload overlaps step i-1's compute and step i-2's download).
    Every step's own copies lie inside the timed region."""
    import synth
    d = 4096
    Ms = (1, 2, 4, 8, 16)
    wb_h, wf_h = synth.layer(21, d, d)
    x_h = synth.activations(21, max(Ms), d)

    def pinned(a):
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).pin_memory()
    hb, hf, hx = pinned(wb_h), pinned(wf_h), pinned(x_h)
    sets = []
    for _ in range(2):
        st = {
            "db": torch.empty_like(hb, device="cuda"), "df": torch.empty_like(hf, device="cuda"),
            "dx": torch.empty_like(hx, device="cuda"),
            "packed": torch.empty((d, d // 8), dtype=torch.uint8, device="cuda"),
            "alpha": torch.empty((d,), dtype=torch.float32, device="cuda"),
            "w_eff": torch.empty((d, d), dtype=torch.bfloat16, device="cuda"),
            "ys": {M: torch.empty((M, d), dtype=torch.bfloat16, device="cuda") for M in Ms},
            "o_packed": torch.empty((d, d // 8), dtype=torch.uint8).pin_memory(),
            "o_alpha": torch.empty((d,), dtype=torch.float32).pin_memory(),
            "o_weff": torch.empty((d, d), dtype=torch.bfloat16).pin_memory(),
            "o_ys": {M: torch.empty((M, d), dtype=torch.bfloat16).pin_memory() for M in Ms},
            "ev_in": torch.cuda.Event(), "ev_comp": torch.cuda.Event(),
            "ev_out": torch.cuda.Event(),
        }
        sets.append(st)
    s_in, s_comp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()

    def step(i):
        st = sets[i % 2]
        with torch.cuda.stream(s_in):
            s_in.wait_event(st["ev_comp"])          # step i-2 has finished reading this set
            st["db"].copy_(hb, non_blocking=True)
            st["df"].copy_(hf, non_blocking=True)
            st["dx"].copy_(hx, non_blocking=True)
            st["ev_in"].record(s_in)
        with torch.cuda.stream(s_comp):
            s_comp.wait_event(st["ev_in"])
            s_comp.wait_event(st["ev_out"])         # step i-2's results have left
            bd.bitdelta_compress(st["db"], st["df"], per_row=True, packed_out=st["packed"],
                                 alpha_out=st["alpha"], stream=s_comp)
            bd.bitdelta_reconstruct(st["db"], st["packed"], st["alpha"], per_row=True,
                                    out=st["w_eff"], stream=s_comp)
            for M in Ms:
                bd.bitdelta_linear(st["dx"][:M], st["db"], st["packed"], st["alpha"],
                                   per_row=True, out=st["ys"][M], stream=s_comp)
            st["ev_comp"].record(s_comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(st["ev_comp"])
            st["o_packed"].copy_(st["packed"], non_blocking=True)
            st["o_alpha"].copy_(st["alpha"], non_blocking=True)
            st["o_weff"].copy_(st["w_eff"], non_blocking=True)
            for M in Ms:
                st["o_ys"][M].copy_(st["ys"][M], non_blocking=True)
            st["ev_out"].record(s_out)

    for i in range(4):
        step(i)
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(s_in)
    s_comp.wait_event(start)
    s_out.wait_event(start)
    for i in range(steps):
        step(i)
    s_in.wait_stream(s_comp)
    s_in.wait_stream(s_out)
    end.record(s_in)
    torch.cuda.synchronize()
    ms = start.elapsed_time(end) / steps
    h2d = hb.numel() * 2 + hf.numel() * 2 + hx.numel() * 2
    d2h = d * (d // 8) + d * 4 + d * d * 2 + sum(M * d * 2 for M in Ms)
    n = d * d
    alg = 2 * (n * (4 + 1 / 8) + 4 * d) + sum(n * (2 + 1 / 8) + 4 * d + 2 * M * 2 * d for M in Ms)
    return {"value": alg / (ms * 1e-3) / 1e9, "unit": "GB/s", "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "ms_per_step": ms,
            "note": "one 4096x4096 layer per step, inputs copied from pinned host memory; "
                    "steps pipelined on copy-in / compute / copy-out streams with two "
                    "buffer sets"}


# --------------------------------------------------------------------------- main


def init_dist(args=None):
    """One process per GPU (torchrun env).  NCCL when CUDA is present, gloo
    otherwise (the host-side logic runs on CPU-only test hosts too)."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as tdist
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
            tdist.init_process_group("nccl")
        else:
            tdist.init_process_group("gloo")
        dist = tdist
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return dist, rank, world, local


def max_over_ranks(dist, value: float) -> float:
    """The slowest rank's time: an all-reduce (MAX) over the process group, or
    the value itself for one process."""
    if dist is None:
        return value
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_value(world: int, units_per_rank: float, seconds: float) -> float:
    """Whole-job throughput: every rank processes the same units per step
    (independent replicas), over the slowest rank's time."""
    return world * units_per_rank / seconds


def run_reference(args, rank, world):
    """CPU oracle on the same workload and metric (bounded sample per step)."""
    if rank != 0:
        return 0
    import oracle
    import synth
    oracle.build()
    d = 4096
    rows = 256   # bounded sample: the first 256 output rows of one 4096x4096 layer
    Ms = (1, 2, 4, 8, 16)
    wb, wf = synth.layer(1, d, d)
    wb, wf = wb[:rows].copy(), wf[:rows].copy()
    x = synth.activations(1, max(Ms), d)
    n = rows * d
    per_layer = 2 * (n * (4 + 1 / 8) + 4 * rows) + sum(
        n * (2 + 1 / 8) + 4 * rows + 2 * M * (d + rows) for M in Ms)

    def step():
        p, a, _ = oracle.compress(wb, wf, True)
        oracle.reconstruct(wb, p, a, True)
        for M in Ms:
            oracle.linear(x[:M], wb, p, a, True)
    for _ in range(max(0, min(args.warmup, 1))):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / args.steps
    value = per_layer / dt / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,0.02) base, Laplace(0,1e-3) delta, N(0,1) x)",
        "config": {"workload": DecodeStack.name,
                   "sample": "256 of the 4096 output rows of one 4096x4096 layer per step",
                   "l2": "not applicable (host oracle)"},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": "per step: rows 0-255 of one 4096x4096 layer through "
                                   "compress, reconstruct, linear M=1,2,4,8,16 "
                                   "(single-threaded C++ fp64)"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_profile(kind: str, prefill_tile: str = "auto"):
    """A few eager launches of one kernel on a small case, for ncu captures."""
    import bit_weight_delta_gb300 as bd
    import synth.device as sd
    bd.load()
    torch.cuda.set_device(0)
    bd.bitdelta_set_prefill_tile(prefill_tile if prefill_tile == "auto" else int(prefill_tile))
    if kind in ("decode", "decode16", "compress", "reconstruct"):
        layers = []
        for l in range(4):
            wb, wf = sd.layer(1, 4096, 4096, stream=l)
            p, a = bd.bitdelta_compress(wb, wf, per_row=True)
            layers.append((wb, wf, p, a))
        x = sd.normal_bf16((16, 4096), 1, 9999)
        y = torch.empty((16, 4096), dtype=torch.bfloat16, device="cuda")
        w = torch.empty((4096, 4096), dtype=torch.bfloat16, device="cuda")
        for i in range(6):
            wb, wf, p, a = layers[i % 4]
            if kind == "decode":
                bd.bitdelta_linear(x[:8], wb, p, a, per_row=True, out=y[:8])
            elif kind == "decode16":
                bd.bitdelta_linear(x, wb, p, a, per_row=True, out=y)
            elif kind == "compress":
                bd.bitdelta_compress(wb, wf, per_row=True, packed_out=p, alpha_out=a)
            else:
                bd.bitdelta_reconstruct(wb, p, a, per_row=True, out=w)
    elif kind == "prefill":
        wb, wf = sd.layer(3, 8192, 8192, stream=1)
        p, a = bd.bitdelta_compress(wb, wf, per_row=True)
        del wf
        x = sd.normal_bf16((2048, 8192), 3, 5000)
        y = torch.empty((2048, 8192), dtype=torch.bfloat16, device="cuda")
        for _ in range(4):
            bd.bitdelta_linear(x, wb, p, a, per_row=True, out=y)
    elif kind == "prefill_split":
        # the QKV projection (8192 -> 10240), whose last round of 512-token
        # tiles is small: through bitdelta_linear_ws, split over the pairs
        wb, wf = sd.layer(3, 10240, 8192, stream=0)
        p, a = bd.bitdelta_compress(wb, wf, per_row=True)
        del wf
        x = sd.normal_bf16((2048, 8192), 3, 5000)
        y = torch.empty((2048, 10240), dtype=torch.bfloat16, device="cuda")
        ws = torch.empty(bd.bitdelta_linear_workspace_bytes(2048, 10240, 8192),
                         dtype=torch.uint8, device="cuda")
        for _ in range(4):
            bd.bitdelta_linear_ws(x, wb, p, a, ws, per_row=True, out=y)
    elif kind == "grouped":
        grp = Grouped(bd)
        for i in range(4):
            grp.run_phase(f"set{i % grp.sets}")
    elif kind == "slice_decode":
        # the 40-layer slice's decode instance on its largest projection
        # (gate+up, 8192 -> 57344): 8 rows alternating two variants through
        # the grouped linear, and the single-variant decode of the same rows
        wb = sd.slice_base(0, 2)
        var = []
        for v in (1, 2):
            wf = sd.slice_finetuned(wb, 0, 2, v)
            var.append(bd.bitdelta_compress(wb, wf, per_row=True))
            del wf
        pt, at = bd.variant_tables([var[0][0], var[1][0]], [var[0][1], var[1][1]], "cuda")
        x = sd.slice_inputs(wb.shape[1], 8, True)
        off = torch.arange(9, dtype=torch.int32, device="cuda")
        seg_var = torch.tensor([1 + r % 2 for r in range(8)], dtype=torch.int32, device="cuda")
        y = torch.empty((8, wb.shape[0]), dtype=torch.bfloat16, device="cuda")
        for _ in range(3):
            bd.bitdelta_linear_grouped(x, off, seg_var, wb, pt, at, n_var=2, max_seg_len=1,
                                       per_row=True, out=y)
            bd.bitdelta_linear(x, wb, var[0][0], var[0][1], per_row=True, out=y)
    elif kind == "kmerge":
        km = KMergeSimilarity(bd)
        n_b = km.n_var - 1
        ws = torch.empty(bd.bitdelta_sign_similarity_workspace_bytes(km.d_out, n_b) + 256,
                         dtype=torch.uint8, device="cuda")
        for _ in range(4):
            bd.bitdelta_sign_similarity(km.packs[0], km.alphas[0], km.pt, km.at, n_b, True,
                                        workspace=ws)
    elif kind == "monosoup":
        ms_wl = MonoSoupMerge(bd)
        for _ in range(2):
            bd.bitdelta_monosoup(ms_wl.wb, ms_wl.ws, ms_wl.rank, power_iters=ms_wl.q, seed=1,
                                 out=ms_wl.out, workspace=ms_wl.ws_buf)
    else:
        raise SystemExit(f"unknown profile kind {kind}")
    torch.cuda.synchronize()
    assert bd.bitdelta_check_error() == 0
    print(f"profile {kind}: ok")
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workloads", default="all", help="comma list of tiny,prefill,grouped,slice40,decode_large,"
                         "cache,kmerge,monosoup; or all|none")
    ap.add_argument("--cpu-budget", type=float, default=12.0,
                    help="seconds of oracle time for cpu_baseline")
    ap.add_argument("--no-cpu", action="store_true",
                    help="skip the per-workload oracle samples (cpu_baseline of each workload)")
    ap.add_argument("--profile", default=None,
                    help="decode|decode16|compress|reconstruct|prefill|prefill_split|grouped|"
                         "slice_decode|kmerge|monosoup: a few eager launches for ncu")
    ap.add_argument("--prefill-tile", default="auto", choices=["auto", "256", "512"],
                    help="token width of the tensor-core kernel's pair tiles (profile runs)")
    args = ap.parse_args()
    if args.profile:
        return run_profile(args.profile, args.prefill_tile)

    dist, rank, world, local = init_dist(args)
    if args.impl == "reference":
        rc = run_reference(args, rank, world)
        if dist is not None:
            dist.destroy_process_group()
        return rc

    import bit_weight_delta_gb300 as bd
    bd.load()
    peaks = load_peaks()
    cudart = _Cudart()

    dec = DecodeStack(bd)
    clock = ClockSampler(local) if rank == 0 else None
    if clock:
        clock.start()
    ms, phases = timed_run(cudart, dec, args.steps, args.warmup, dist, clock,
                           graph_steps=min(args.steps, 20))
    clocks = clock.stop() if clock else None
    bytes_step = dec.bytes_per_step()
    value = weak_scaling_value(world, bytes_step, ms * 1e-3) / 1e9

    dom = dec.dominant()
    dom_bytes = sum(dec.bytes[p] * dec.L for p in dom)
    dom_ms = sum(phases[p] for p in dom)
    achieved = dom_bytes / (dom_ms * 1e-3) / 1e9
    per_kernel = {p: {"us_per_launch": phases[p] * 1e3 / dec.L,
                      "GB/s": dec.bytes[p] * dec.L / (phases[p] * 1e-3) / 1e9,
                      "frac_of_hbm_peak": dec.bytes[p] * dec.L / (phases[p] * 1e-3) / 1e9
                      / peaks["hbm_gbs"]}
                  for p in dec.phases}

    decode_unfused = dec.unfused_timing()

    workloads = {}
    wanted = set(args.workloads.split(",")) if args.workloads not in ("all", "none") else (
        {"tiny", "prefill", "grouped", "slice40", "decode_large", "cache", "kmerge", "monosoup"}
        if args.workloads == "all"
        else set())
    cpu_on = rank == 0 and not args.no_cpu
    if "tiny" in wanted:
        tw = Tiny(bd)
        workloads["tiny"] = tw.report()
        if cpu_on:
            workloads["tiny"]["cpu_baseline"] = tw.oracle_sample()
        del tw
    if "prefill" in wanted:
        pre = Prefill(bd)
        pms, pph = timed_run(cudart, pre, 10, 3, dist, None, graph_steps=10)
        ref = pre.cublas_reference()
        # the same step through bitdelta_linear (no split workspace), timed
        # after the cuBLAS reference so that the reference sees the GPU in the
        # same state as the fused step before it
        pre.split = False
        nms, nph = timed_run(cudart, pre, 10, 3, dist, None, graph_steps=10)
        pre.split = True
        tfl = pre.flops_per_step() / (pms * 1e-3) / 1e12
        workloads["prefill"] = {
            "workload": pre.name, "ms_per_step": pms, "TFLOP/s": tfl,
            "roofline": {"bound": "tensor", "achieved": tfl,
                         "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                         "frac": tfl / peaks["bf16_tflops"], "traffic": None},
            "per_projection": {p: {"ms": pph[p], "TFLOP/s": pre.flops[p] / (pph[p] * 1e-3) / 1e12}
                               for p in pre.phases},
            "cublas_bf16_gemm_same_shapes": ref["cublas_plain"],
            "unfused_reconstruct_plus_cublas": ref["unfused"],
            "fused_vs_unfused_by_tokens": ref["fused_vs_unfused_by_tokens"],
            "frac_of_cublas": ref["cublas_plain"]["ms_per_step"] / pms,
            "call": "bitdelta_linear_ws (split schedule, workspace "
                    f"{0 if pre.ws is None else pre.ws.numel() >> 20} MiB)",
            "without_workspace": {
                "call": "bitdelta_linear", "ms_per_step": nms,
                "TFLOP/s": pre.flops_per_step() / (nms * 1e-3) / 1e12,
                "per_projection": {p: {"ms": nph[p],
                                       "TFLOP/s": pre.flops[p] / (nph[p] * 1e-3) / 1e12}
                                   for p in pre.phases}},
        }
        if cpu_on:
            workloads["prefill"]["cpu_baseline"] = pre.oracle_sample()
        del pre
        torch.cuda.empty_cache()
    if "grouped" in wanted:
        grp = Grouped(bd)
        gms, gph = timed_run(cudart, grp, 30, 3, dist, None, graph_steps=30)
        per_call = gms / grp.sets
        tfl = grp.flops / (per_call * 1e-3) / 1e12
        t_roof = max(grp.flops / (peaks["bf16_tflops"] * 1e12), grp.bytes / (peaks["hbm_gbs"] * 1e9))
        workloads["grouped"] = {
            "workload": grp.name, "ms_per_call": per_call, "TFLOP/s": tfl,
            "rows/s": grp.M / (per_call * 1e-3),
            "roofline": {"bound": "tensor", "achieved": tfl, "peak": peaks["bf16_tflops"],
                         "unit": "TFLOP/s", "frac": tfl / peaks["bf16_tflops"],
                         "roofline_time_ms": t_roof * 1e3,
                         "frac_of_roofline_time": t_roof * 1e3 / per_call, "traffic": None},
            "unfused_reconstruct_plus_cublas": grp.unfused_timing(),
        }
        if cpu_on:
            workloads["grouped"]["cpu_baseline"] = grp.oracle_sample()
        del grp
        torch.cuda.empty_cache()
    if "slice40" in wanted:
        sl = Slice40(bd)
        workloads["slice40"] = sl.report(peaks, cpu=cpu_on)
        del sl
        torch.cuda.empty_cache()
    if "decode_large" in wanted:
        dl = DecodeLarge(bd)
        workloads["decode_large"] = dl.report(peaks)
        del dl
        torch.cuda.empty_cache()
    if "kmerge" in wanted:
        km = KMergeSimilarity(bd)
        workloads["kmerge"] = km.report()
        del km
        torch.cuda.empty_cache()
    if "monosoup" in wanted:
        ms_wl = MonoSoupMerge(bd)
        workloads["monosoup"] = ms_wl.report()
        del ms_wl
        torch.cuda.empty_cache()
    if "cache" in wanted:
        dc = DeltaCacheLoads(bd)
        workloads["delta_cache"] = dc.report()
        dc.close()
        del dc
        torch.cuda.empty_cache()

    e2e = e2e_decode(bd, 20)
    e2e["value"] *= world

    cpu = None
    if rank == 0:
        cpu = dec.oracle_sample(args.cpu_budget)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0,0.02) base, Laplace(0,1e-3) delta, N(0,1) x)",
            "config": {"workload": dec.name, "layers_per_step": dec.L,
                       "l2": "inputs larger than L2: 32 distinct layers (2.2 GB) per step, "
                             "each input reused only after >= 31 other launches",
                       "alpha": "per row", "parallelism": f"replicas x{world}"},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"],
                         "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                         "traffic": DECODE_TRAFFIC_BYTES,
                         "traffic_source": "ncu dram__bytes_read.sum + dram__bytes_write.sum of "
                                           "one gemv_single_async_kernel launch, 4096x4096, M=8",
                         "kernel": "bitdelta_linear decode: gemv_single_async_kernel (M=1..16; "
                                   "the 4096x4096 grid is one wave at two CTAs per SM)",
                         "peak_source": peaks["source"]},
            "per_kernel": per_kernel,
            "decode_unfused_reconstruct_plus_cublas": decode_unfused,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": dec.launches_per_step() * args.steps,
            "clocks": clocks,
            "workloads": workloads,
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
