"""Benchmark of the quantized-weight GEMM hot path on B300.

Default workload (one JSON line on rank 0): the W4A16 asymmetric sweep --
UINT4 weights with bf16 group-128 scales and uint4 zero points, bf16
activations, (N, K) in {(4096, 4096), (11008, 4096), (4096, 11008)} x
M in {1, 4, 16, 64, 256, 1024}.  One step runs all 18 GEMMs once through the
library's C ABI; every GEMM has its own weight and activation buffers, so a
step touches ~438 MB and each GEMM reads its operands cold from HBM (the
126 MB L2 is flushed by the rest of the step).  The step is captured in a
CUDA graph and replayed.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload sweep|w4a16_m16|large|w4a8|moe16|moe256|moe4096|
                              f16s|w8a16|nvfp4|w4a4|w4a4_large|
                              shape:M,N,K[,sym|asym][,bf16|fp16][,w4a4]]

Other workloads (--workload) are for kernel studies and print the same line
format for their own configuration.  --impl reference times the CPU oracle
(test infrastructure) on a bounded sample of the same workload.
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

L2_BYTES = 126 * 1024 * 1024
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}


def load_peaks():
    try:
        with open(PEAKS_FILE) as f:
            d = json.load(f)
        return d, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


# ------------------------------------------------------------------ workloads

def sweep_points():
    pts = []
    for m in synth.W4A16_ASYM_MS:
        for (n, k) in synth.W4A16_ASYM_SHAPES:
            pts.append(dict(m=m, n=n, k=k, g=128, asym=True, adt="bf16"))
    return pts


def workload_points(name):
    if name.startswith("shape:"):
        # one W4A16 GEMM of the given shape (kernel studies, profiling)
        f = name[len("shape:"):].split(",")
        m, n, k = (int(v) for v in f[:3])
        asym = "asym" in f[3:]
        adt = "fp16" if "fp16" in f[3:] else "bf16"
        sdt = "fp16" if "f16s" in f[3:] else adt     # f16s: fp16 scales (bf16 activations)
        if "w4a4" in f[3:]:   # NVFP4 weights and activations
            return [dict(kind="w4a4", m=m, n=n, k=k, g=16, asym=False, adt="bf16")], dict(
                workload=f"w4a4_nvfp4_{m}x{n}x{k}", m=m, n=n, k=k, weights="nvfp4",
                act="bf16 -> nvfp4 per token")
        return [dict(m=m, n=n, k=k, g=128, asym=asym, adt=adt, sdt=sdt)], dict(
            workload=f"w4a16_{'asym' if asym else 'sym'}_{m}x{n}x{k}"
                     + ("_f16scales" if sdt != adt else ""), m=m, n=n, k=k, group=128,
            weights="uint4+zp" if asym else "int4", scales=sdt, act=adt)
    if name == "sweep":
        return sweep_points(), dict(workload="w4a16_asym_sweep", shapes=synth.W4A16_ASYM_SHAPES,
                                    ms=synth.W4A16_ASYM_MS, group=128, weights="uint4+zp",
                                    act="bf16")
    if name == "w8a16":
        # the sweep's shapes with 8-bit weights (UINT8 + zero points)
        return ([dict(p, kind="w8a16") for p in sweep_points()],
                dict(workload="w8a16_asym_sweep", shapes=synth.W4A16_ASYM_SHAPES,
                     ms=synth.W4A16_ASYM_MS, group=128, weights="uint8+zp", act="bf16"))
    if name == "f16s":
        # the sweep with fp16 scales against bf16 activations
        return ([dict(p, sdt="fp16") for p in sweep_points()],
                dict(workload="w4a16_asym_f16scales_sweep", shapes=synth.W4A16_ASYM_SHAPES,
                     ms=synth.W4A16_ASYM_MS, group=128, weights="uint4+zp", scales="fp16",
                     act="bf16"))
    if name == "nvfp4":
        # the sweep's shapes with NVFP4 weights (e2m1 + e4m3 per 16 k + fp32 tensor scale)
        return ([dict(p, kind="nvfp4", g=16, asym=False) for p in sweep_points()],
                dict(workload="w4a16_nvfp4_sweep", shapes=synth.W4A16_ASYM_SHAPES,
                     ms=synth.W4A16_ASYM_MS, group=16, weights="nvfp4 (e2m1 + e4m3/16 + fp32)",
                     act="bf16"))
    if name == "w4a4":
        # the sweep's shapes with NVFP4 weights and NVFP4 activations
        return ([dict(p, kind="w4a4", g=16, asym=False) for p in sweep_points()],
                dict(workload="w4a4_nvfp4_sweep", shapes=synth.W4A16_ASYM_SHAPES,
                     ms=synth.W4A16_ASYM_MS, group=16,
                     weights="nvfp4 (e2m1 + e4m3/16 + fp32)",
                     act="bf16 -> nvfp4 per token (e2m1 + e4m3/16, fp32 tensor scale)"))
    if name == "w4a4_large":
        s = synth.LARGE_SHAPE
        return ([dict(kind="w4a4", m=s["m"], n=s["n"], k=s["k"], g=16, asym=False, adt="bf16")],
                dict(workload="w4a4_nvfp4_8192x8192x8192", m=s["m"], n=s["n"], k=s["k"],
                     weights="nvfp4", act="bf16 -> nvfp4 per token"))
    if name == "w4a16_m16":
        s = synth.W4A16_SYM_SHAPE
        return [dict(m=s["m"], n=s["n"], k=s["k"], g=128, asym=False, adt="fp16")], dict(
            workload="w4a16_sym_m16_4096x4096", m=16, n=4096, k=4096, group=128, weights="int4",
            act="fp16")
    if name == "large":
        s = synth.LARGE_SHAPE
        return [dict(m=s["m"], n=s["n"], k=s["k"], g=128, asym=False, adt="bf16")], dict(
            workload="w4a16_sym_8192x8192x8192", m=8192, n=8192, k=8192, group=128,
            weights="int4", act="bf16")
    if name == "w4a8" or name.startswith("w4a8:"):
        # w4a8:M: one M of the set (kernel studies, profiling)
        s = synth.W4A8_SHAPE
        ms = [int(name[5:])] if name.startswith("w4a8:") else synth.W4A8_MS
        return ([dict(kind="w4a8", m=m, n=s["n"], k=s["k"], g=32, asym=False, adt="bf16")
                 for m in ms],
                dict(workload="w4a8_mxfp4_7168x2048", n=s["n"], k=s["k"], ms=synth.W4A8_MS,
                     weights="mxfp4 (e2m1 + e8m0/32)", act="bf16 -> e4m3 per token"))
    if name.startswith("moe"):
        t = int(name[3:])
        s = synth.MOE_SHAPE
        return ([dict(kind="moe", m=t, n=s["hidden"], k=s["hidden"], g=128, asym=False,
                      adt="bf16")],
                dict(workload=f"grouped_moe_w4a16_T{t}", tokens=t, experts=s["experts"],
                     topk=s["topk"], hidden=s["hidden"], inter=s["inter"], group=128,
                     weights="int4 per expert"))
    raise ValueError(name)


def point_bytes(p):
    m, n, k, g = p["m"], p["n"], p["k"], p["g"]
    kind = p.get("kind", "w4a16")
    if kind == "w4a8":
        # GEMM: bf16 activations read once, codes, e8m0 scales, bf16 out; above
        # 8 rows the per-token quantization is its own kernel (bf16 in, e4m3
        # and scales out, read back by the GEMM), at most 8 rows it runs
        # inside the small-M kernel
        gemm = 2 * m * k + n * k // 2 + n * k // 32 + 2 * m * n
        return gemm + (m * k + 4 * m) * 2 if m > 8 else gemm
    if kind == "w8a16":
        # 8-bit codes, scales, 8-bit zero points, activations, output
        return n * k + (k // g) * n * 2 + (k // g) * n + m * k * 2 + m * n * 2
    if kind == "nvfp4":
        # codes, block scales as the kernel reads them (16-bit per 16 k), activations, output
        return n * k // 2 + (k // 16) * n * 2 + m * k * 2 + m * n * 2
    if kind == "w4a4":
        # bf16 activations read by the quantizer, its codes and block scales
        # written and read back by the GEMM, weight codes and block scales, output
        return 2 * m * k + 2 * (m * k // 2 + m * k // 16) + n * k // 2 + n * k // 16 + 2 * m * n
    if kind == "moe":
        s = synth.MOE_SHAPE
        e, h, i, topk = s["experts"], s["hidden"], s["inter"], s["topk"]
        r = m * topk
        active = min(e, r)   # upper bound on the experts that receive a row
        w_e = (h * 2 * i + i * h) // 2 + (h // 128) * 2 * i * 2 + (i // 128) * h * 2
        act = (2 * m * h + 2 * r * h * 2            # permute: read tokens, write a_perm (+read)
               + 2 * r * i                          # gated GEMM1 out
               + 2 * r * i + 2 * r * h * 2 + 2 * m * h)   # GEMM2 in/out, combine
        return active * w_e + act
    b = n * k // 2 + (k // g) * n * 2 + m * k * 2 + m * n * 2
    if p["asym"]:
        b += (k // g) * n // 2
    return b


def point_flops(p):
    if p.get("kind") == "moe":
        s = synth.MOE_SHAPE
        return 2 * p["m"] * s["topk"] * (s["hidden"] * 2 * s["inter"] + s["inter"] * s["hidden"])
    return 2 * p["m"] * p["n"] * p["k"]


# ------------------------------------------------------------------ clocks

def _nvml_sampler(index):
    """(max SM MHz, sample) where sample() returns (SM MHz, clock-event reason
    bits) through NVML's C library (read-only queries, ctypes; the Python
    binding is not needed)."""
    import ctypes
    nv = ctypes.CDLL("libnvidia-ml.so.1")
    if nv.nvmlInit_v2() != 0:
        raise RuntimeError("nvmlInit failed")
    h = ctypes.c_void_p()
    if nv.nvmlDeviceGetHandleByIndex_v2(index, ctypes.byref(h)) != 0:
        raise RuntimeError("no NVML handle for device %d" % index)
    clk, mx, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
    nvml_clock_sm = 1
    nv.nvmlDeviceGetMaxClockInfo(h, nvml_clock_sm, ctypes.byref(mx))

    def sample():
        if nv.nvmlDeviceGetClockInfo(h, nvml_clock_sm, ctypes.byref(clk)) != 0:
            raise RuntimeError("nvmlDeviceGetClockInfo failed")
        if nv.nvmlDeviceGetCurrentClocksEventReasons(h, ctypes.byref(rs)) != 0:
            raise RuntimeError("nvmlDeviceGetCurrentClocksEventReasons failed")
        return clk.value, rs.value
    return mx.value, sample


def _clock_sampler_proc(index, period, stop, conn):
    """Child process of ClockSampler: NVML SM clock and clock-event reasons
    (read-only queries) every `period` seconds until `stop` is set.  A process
    of its own, so that the sampling does not wait on the interpreter lock of
    the process that launches the work."""
    import time
    try:
        mx, sample = _nvml_sampler(index)
        conn.send(("ready", mx))
    except Exception as e:   # no NVML here: the parent samples by itself
        conn.send(("error", str(e)))
        return
    out = []
    while not stop.is_set():
        t = time.monotonic()
        try:
            out.append((t, *sample()))
        except Exception:
            pass
        time.sleep(period)
    conn.send(("done", out))


class ClockSampler:
    """SM clock and clock-event reasons sampled through NVML every `period`
    seconds while the timed region runs: in a spawned child process (no CUDA in
    it), else on a background thread, else by polling nvidia-smi.  mark_start /
    mark_end bound the window whose samples stop() summarises."""

    REASONS = {"hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20, "hw_thermal_slowdown": 0x40,
               "sw_power_cap": 0x4, "hw_power_brake_slowdown": 0x80}

    def __init__(self, index, period=0.005):
        self.index = index
        self.period = period
        self.samples = []          # (time.monotonic(), sm_mhz, reasons)
        self.max_mhz = None
        self._stop = None
        self._thread = None
        self._proc = None
        self._conn = None
        self.window = None
        self.error = None
        self.how = None

    def mark_start(self):
        self.window = [time.monotonic(), None]

    def mark_end(self):
        if self.window:
            self.window[1] = time.monotonic()

    def _start_process(self):
        import multiprocessing as mp
        ctx = mp.get_context("spawn")
        self._stop = ctx.Event()
        self._conn, child = ctx.Pipe(duplex=False)
        self._proc = ctx.Process(target=_clock_sampler_proc,
                                 args=(self.index, self.period, self._stop, child), daemon=True)
        self._proc.start()
        child.close()
        t_end = time.monotonic() + 60
        while not self._conn.poll(0.1):
            if not self._proc.is_alive() or time.monotonic() > t_end:
                raise RuntimeError("clock sampler process did not start")
        tag, val = self._conn.recv()
        if tag != "ready":
            self._proc.join(10)
            raise RuntimeError(f"clock sampler process: {val}")
        self.max_mhz = val
        self.how = "nvml, own process"

    def start(self):
        try:
            self._start_process()
            return
        except Exception as e:            # no spawn or no NVML binding: sample in this process
            self.error = str(e)
            if self._proc is not None and self._proc.is_alive():
                self._proc.kill()
            self._proc = None
        import threading
        self._stop = threading.Event()
        try:
            self.max_mhz, sample = _nvml_sampler(self.index)
            self.how = "nvml, thread"
        except Exception:            # no NVML library: poll nvidia-smi instead
            import subprocess
            q = ["nvidia-smi", "-i", str(self.index), "--format=csv,noheader,nounits",
                 "--query-gpu=clocks.sm,clocks.max.sm,clocks_event_reasons.active"]
            self.how = "nvidia-smi, thread"

            def sample():
                out = subprocess.run(q, capture_output=True, text=True, timeout=5).stdout
                sm, smax, active = [x.strip() for x in out.strip().split(",")[:3]]
                self.max_mhz = float(smax)
                return float(sm), int(active, 16)

        def run():
            while not self._stop.is_set():
                try:
                    t = time.monotonic()
                    self.samples.append((t, *sample()))
                except Exception as e:
                    self.error = str(e)
                self._stop.wait(self.period)

        self._thread = threading.Thread(target=run, daemon=True)
        self._thread.start()

    def stop(self):
        if self._proc is not None:
            self._stop.set()
            if self._conn.poll(60):
                tag, out = self._conn.recv()
                self.samples = out
            else:
                self.error = "clock sampler process sent no samples"
            self._proc.join(10)
            if self._proc.is_alive():
                self._proc.kill()
        elif self._thread is not None:
            self._stop.set()
            self._thread.join()
        return self.summary()

    def summary(self):
        s = self.samples
        if self.window and self.window[1] is not None:
            t0, t1 = self.window
            inside = [x for x in s if t0 <= x[0] <= t1]
            # a window shorter than the sampling period: the samples next to it
            s = inside or [x for x in s if t0 - 0.05 <= x[0] <= t1 + 0.05]
        if not s:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "samples": 0,
                    "reasons": [self.error or "no samples"], "how": self.how}
        reasons = sorted({nm for _, _, rs in s for nm, bit in self.REASONS.items() if rs & bit})
        return {"sm_mhz": statistics.median(m for _, m, _ in s), "sm_max_mhz": self.max_mhz,
                "samples": len(s), "reasons": reasons, "how": self.how}


class GemmPoint:
    """Buffers of one GEMM of the workload (own weights, activations, output).

    ``clone()`` duplicates every device buffer, so that a rotation of clones
    reads its operands cold from HBM.  A W4A8 point's launch is one library
    call on its bf16 activations: the per-token FP8 quantization runs inside
    the small-M kernel at M <= 8, else as its own kernel ahead of the GEMM."""

    def __init__(self, p, seed, device, host=False, src=None):
        import torch
        from quantized_weight_gemm_run_b300 import qgemm as Q
        from quantized_weight_gemm_run_b300.api import (NVFP4Linear, W4A16Linear, W4A8Linear,
                                                         W8A16Linear)
        self.p, self.Q = p, Q
        self.mx = p.get("kind") == "w4a8"
        m, n, k, gs = p["m"], p["n"], p["k"], p["g"]
        dt = torch.float16 if p["adt"] == "fp16" else torch.bfloat16
        if src is None:
            g = synth.rng(seed)
            if self.mx:
                codes = torch.from_numpy(synth.random_bytes(g, (n, k // 2))).to(device)
                b = torch.from_numpy(synth.random_bytes(g, (n, k // 32), 116, 124)).to(device)
                self.lin = W4A8Linear(codes, b, n, k)
                del codes, b
            elif p.get("kind") == "w8a16":
                qweight = torch.from_numpy(synth.random_words(g, (k // 4, n))).to(device)
                scales = torch.from_numpy(
                    synth.random_scales_fp32(g, (k // gs, n))).to(dt).to(device)
                qzeros = torch.from_numpy(synth.random_words(g, (k // gs, n // 4))).to(device)
                self.lin = W8A16Linear(qweight, scales, qzeros, n, k, gs, dt)
                del qweight, scales, qzeros
            elif p.get("kind") == "w4a4":
                from quantized_weight_gemm_run_b300.api import W4A4Linear
                codes = torch.from_numpy(synth.random_bytes(g, (n, k // 2))).to(device)
                sb = torch.from_numpy(synth.random_bytes(g, (n, k // 16), 0x30, 0x48)).to(device)
                ts = torch.full((1,), 2.0 ** -9, dtype=torch.float32, device=device)
                # activations ~ N(0, 1): a tensor scale that maps |x| = 6 to 448 * 6
                a_ts = torch.full((1,), 6.0 / (6 * 448), dtype=torch.float32, device=device)
                self.lin = W4A4Linear(codes, sb, ts, a_ts, n, k)
                del codes, sb
            elif p.get("kind") == "nvfp4":
                codes = torch.from_numpy(synth.random_bytes(g, (n, k // 2))).to(device)
                sb = torch.from_numpy(synth.random_bytes(g, (n, k // 16), 0x30, 0x48)).to(device)
                ts = torch.full((1,), 2.0 ** -9, dtype=torch.float32, device=device)
                self.lin = NVFP4Linear(codes, sb, ts, n, k, dt)
                del codes, sb
            else:
                qweight = torch.from_numpy(synth.random_words(g, (k // 8, n))).to(device)
                sdt = torch.float16 if p.get("sdt", p["adt"]) == "fp16" else torch.bfloat16
                scales = torch.from_numpy(
                    synth.random_scales_fp32(g, (k // gs, n))).to(sdt).to(device)
                qzeros = (torch.from_numpy(synth.random_words(g, (k // gs, n // 8))).to(device)
                          if p["asym"] else None)
                self.lin = W4A16Linear(qweight, scales, qzeros, n, k, gs, dt, scale_dtype=sdt)
                del qweight, scales, qzeros
            self.a = torch.from_numpy(synth.activations_fp32(g, m, k)).to(dt).to(device)
        else:
            import copy
            self.lin = copy.copy(src.lin)
            self.lin.packed = src.lin.packed.clone()
            self.a = src.a.clone()
        self.layer = self.lin.layer_bf16 if self.mx else self.lin.layer
        self.a_scale = self.lin.act_scale if p.get("kind") == "w4a4" else None
        self.c = torch.empty(m, n, dtype=dt, device=device)
        st, nbytes = Q.qgemm_workspace_size(self.layer, self.lin.dense, None, m)
        Q.check(st)
        self.ws = torch.zeros(nbytes, dtype=torch.uint8, device=device)
        if host:
            self.a_host = self.a.cpu().pin_memory()
            self.c_host = torch.empty(m, n, dtype=dt).pin_memory()
        self.launches = 2 if (self.mx and m > 8) or p.get("kind") == "w4a4" else 1

    def clone(self):
        return GemmPoint(self.p, 0, self.c.device, src=self)

    def launch(self):
        Q = self.Q
        m = self.p["m"]
        Q.check(Q.qgemm_run(self.layer, self.lin.dense, None, m, self.a, self.a_scale,
                            self.lin.packed, None, self.c, self.ws, self.ws.numel()))

    def copy_in(self):
        self.a.copy_(self.a_host, non_blocking=True)

    def copy_out(self):
        self.c_host.copy_(self.c, non_blocking=True)

    def status(self):
        """The library status of this point's launches so far (and clears it)."""
        return self.Q.qgemm_check_status(self.ws)


class MoEPoint:
    """One grouped-MoE W4A16 layer (E=64, top-8, hidden 2048, intermediate
    1408) over T tokens: permute, gate|up GEMM with the SiLU gate in its
    epilogue, down GEMM, combine.
    Router logits are drawn seeded and routed once at set-up (softmax top-k on
    the device, outside the timed region)."""

    def __init__(self, p, seed, device, host=False):
        import torch
        from quantized_weight_gemm_run_b300 import qgemm as Q
        from quantized_weight_gemm_run_b300.api import MoELayer, W4A16Linear
        self.p, self.Q = p, Q
        s = synth.MOE_SHAPE
        e, h, i, topk, t = s["experts"], s["hidden"], s["inter"], s["topk"], p["m"]
        g = synth.rng(seed)
        bf = torch.bfloat16

        def expert_stack(k, n, gated=False):
            qw = torch.from_numpy(synth.random_words(g, (e * k // 8, n))).to(device)
            sc = torch.from_numpy(synth.random_scales_fp32(g, (e * k // 128, n))).to(bf).to(device)
            return W4A16Linear(qw, sc, None, n, k, 128, bf, num_experts=e, gated=gated)

        self.l1 = expert_stack(h, 2 * i, gated=True)
        self.l2 = expert_stack(i, h)
        self.layer = MoELayer(self.l1, self.l2, e, topk)
        self.x = torch.from_numpy(synth.activations_fp32(g, t, h)).to(bf).to(device)
        logits = torch.from_numpy(synth.router_logits_fp32(g, t, e)).to(device)
        probs = torch.softmax(logits.double(), dim=-1)
        w, ids = torch.topk(probs, topk, dim=-1)
        self.ids = ids.to(torch.int32).contiguous()
        self.wts = w.to(torch.float32).contiguous()
        self.y = torch.empty(t, h, dtype=bf, device=device)
        self.layer(self.x, self.ids, self.wts, out=self.y)   # sizes the workspaces once
        torch.cuda.synchronize()
        if host:
            self.x_host = self.x.cpu().pin_memory()
            self.y_host = torch.empty(t, h, dtype=bf).pin_memory()
        # sort (one kernel up to 2048 slots, else count + place), gather,
        # gated GEMM1, GEMM2, combine
        self.launches = (1 if t * topk <= 2048 else 2) + 4

    def clone(self):
        return self   # 285 MB of expert weights already exceed twice the L2

    def launch(self):
        self.layer(self.x, self.ids, self.wts, out=self.y)

    def copy_in(self):
        self.x.copy_(self.x_host, non_blocking=True)

    def copy_out(self):
        self.y_host.copy_(self.y, non_blocking=True)

    def status(self):
        st1, st2 = self.l1.status(), self.l2.status()
        return st1 if st1 != self.Q.QGEMM_OK else st2

    @property
    def a(self):
        return self.x

    @property
    def c(self):
        return self.y


def make_point(p, seed, device, host=False):
    if p.get("kind") == "moe":
        return MoEPoint(p, seed, device, host)
    return GemmPoint(p, seed, device, host)


def source_without_comments(text: str) -> str:
    """C/C++ source with its comments and blank lines removed (string
    literals holding comment markers are not expected in the kernels)."""
    import re
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(line.rstrip() for line in text.splitlines() if line.strip())


# the sources that decide what the tcgen05 GEMM kernel does: the kernel, its
# PTX wrappers and shared declarations, and the planner that configures it
TRAFFIC_SOURCES = ("internal.h", "ptx.cuh", "qgemm_api.cu", "w4a16_gemm.cu")


def kernel_source_digest(read=None):
    """Digest of the tcgen05 GEMM kernel's sources (TRAFFIC_SOURCES: the
    kernel and the planner that configures it), comments ignored; a committed
    ncu traffic figure of that kernel is used only while it matches.
    ``read(name)`` returns a file's text (default: the tree)."""
    import hashlib
    d = os.path.join(ROOT, "quantized_weight_gemm_run_b300", "csrc")
    if read is None:
        def read(name):
            with open(os.path.join(d, name)) as fh:
                return fh.read()
    h = hashlib.sha256()
    for f in TRAFFIC_SOURCES:
        h.update(source_without_comments(read(f)).encode())
    return h.hexdigest()[:16]


def committed_traffic():
    """DRAM bytes per launch from the committed ncu summaries under profiles/:
    lines 'traffic shape=MxNxK(,asym|,sym)(,bf16|,fp16) dram_bytes=B source=D'."""
    out = {}
    pdir = os.path.join(ROOT, "profiles")
    if not os.path.isdir(pdir):
        return out
    for fn in sorted(os.listdir(pdir)):
        if not fn.endswith((".md", ".txt")):
            continue
        with open(os.path.join(pdir, fn)) as fh:
            for line in fh:
                line = line.strip().strip("`")
                if not line.startswith("traffic "):
                    continue
                kv = dict(t.split("=", 1) for t in line.split()[1:] if "=" in t)
                if {"shape", "dram_bytes", "source"} <= kv.keys():
                    out[kv["shape"]] = (int(kv["dram_bytes"]), kv["source"])
    return out


def f16_scales(p):
    return p.get("sdt", p["adt"]) != p["adt"]


def shape_key(p):
    return (f"{p['m']}x{p['n']}x{p['k']},{'asym' if p.get('asym') else 'sym'},{p['adt']}"
            + (",f16s" if f16_scales(p) else "")
            if p.get("kind", "w4a16") == "w4a16" else None)


def cold_copies(p):
    """Distinct buffer sets needed so that a rotation exceeds twice the L2."""
    return int(np.ceil(2 * L2_BYTES / point_bytes(p))) + 1


def kernel_name(p):
    kind = p.get("kind", "w4a16")
    if kind == "moe":
        return "moe_layer (sort, gather, SiLU-gated grouped GEMM, grouped GEMM, combine)"
    m = p["m"]
    if kind == "w4a4":
        bt = 16 if m <= 16 else 32 if m <= 32 else 64 if m <= 64 else 128
        if m > 16:   # the planner's smaller tile while the tiles fit one wave on 148 SMs
            bt = next((b for b in (32, 64) if b < bt and -(-m // b) * (p["n"] // 128) <= 148), bt)
        return f"act_quant_nvfp4_kernel + w4a4_kernel<{bt}>"
    nv_small = kind == "nvfp4" and (p["n"] * p["k"] <= 1 << 24 or (m <= 8 and p["k"] <= 4096))
    # the planner's long-K rule: 9-16 rows with K >= 2 N go to the tcgen05 kernel
    long_k = kind == "w4a16" and not f16_scales(p) and m > 8 and p["k"] >= 2 * p["n"]
    mx_rows = kind == "w4a8" and m > 8   # W4A8 above 8 rows: the tcgen05 kernel
    if (kind in ("w4a16", "w4a8") or nv_small) and m <= 16 and not long_k and not mx_rows:
        # the planner's default for dense INT4/UINT4 and W4A8 GEMMs of at most
        # 16 rows, and for NVFP4 ones up to 2^24 weights or 8 rows with K <= 4096
        dt = ("w4a8_fused_act_quant" if kind == "w4a8" else "nvfp4_" + p["adt"] if nv_small
              else "bf16_f16scales" if f16_scales(p) else "fp16" if p["adt"] == "fp16" else "bf16")
        return f"w4a16_mma_kernel<{dt},{1 if m <= 8 else 2}>"
    bt = 16 if m <= 16 else 32 if m <= 32 else 64 if m <= 64 else 128
    if kind == "w4a8" and bt == 128 and -(-m // 64) * (p["n"] // 128) <= 148:
        bt = 64   # the planner's one-wave 64-token tiles for W4A8
    fmt = ("w4a8_mxf8f6f4" if kind == "w4a8" else "nvfp4_bf16" if kind == "nvfp4"
           else f"int8_{p['adt']}" if kind == "w8a16"
           else "bf16_f16scales" if f16_scales(p) else "fp16" if p["adt"] == "fp16" else "bf16")
    name = f"w4a16_kernel<{bt},{fmt},dense>"
    return "act_quant_fp8_kernel + " + name if kind == "w4a8" else name


EXTRA_WORKLOADS = ["w4a16_m16", "w4a8", "moe16", "moe256", "moe4096", "large", "w4a4_large"]
REPLAYS = 7


def graph_time_us(launch, n_launch, stream, replays=REPLAYS):
    """Median over `replays` replays of a graph holding n_launch back-to-back
    launches (`launch(j)` issues the j-th), per launch, by CUDA events on the
    launching stream after three warm-up replays."""
    import torch
    with torch.cuda.stream(stream):   # library handles and workspaces are made outside capture
        launch(0)
    torch.cuda.synchronize()
    g2 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g2, stream=stream):
        for j in range(n_launch):
            launch(j)
    torch.cuda.synchronize()
    ts = []
    with torch.cuda.stream(stream):
        for _ in range(3):
            g2.replay()
        for _ in range(replays):
            a0 = torch.cuda.Event(enable_timing=True)
            a1 = torch.cuda.Event(enable_timing=True)
            a0.record(stream)
            g2.replay()
            a1.record(stream)
            ts.append((a0, a1))
    torch.cuda.synchronize()
    us = sorted(a0.elapsed_time(a1) * 1e3 / n_launch for a0, a1 in ts)
    del g2
    return us[len(us) // 2], us[0], us[-1]


def cublas_context_us(p, stream):
    """torch.matmul (cuBLAS) of the same shape in the activation dtype on
    dense 16-bit weights, over a rotation of cold copies: the library
    comparison point of the pages' small-batch claim.  Context only."""
    import torch
    if p.get("kind") == "moe":
        return None
    m, n, k = p["m"], p["n"], p["k"]
    dt = torch.float16 if p["adt"] == "fp16" else torch.bfloat16
    per = 2 * (m * k + k * n + m * n)
    copies = int(np.ceil(2 * L2_BYTES / per)) + 1
    bufs = [(torch.randn(m, k, device="cuda").to(dt), torch.randn(k, n, device="cuda").to(dt),
             torch.empty(m, n, device="cuda", dtype=dt)) for _ in range(copies)]
    r = max(20, copies)

    def launch(j):
        a, b, c = bufs[j % copies]
        torch.matmul(a, b, out=c)
    med, _, _ = graph_time_us(launch, r, stream)
    del bufs
    torch.cuda.empty_cache()
    return med


def measure_point(bp, p, peaks, stream):
    """One point of the table: the launch timed back to back over a rotation
    of cold clones in a graph (median of REPLAYS replays), with its rates and
    fractions of the measured peaks, and the cuBLAS context time."""
    import torch
    is_moe = p.get("kind") == "moe"
    copies = [bp] + ([] if is_moe else [bp.clone() for _ in range(cold_copies(p) - 1)])
    r = max(20, len(copies))
    med, lo, hi = graph_time_us(lambda j: copies[j % len(copies)].launch(), r, stream)
    bad = sum(1 for c in {id(c): c for c in copies}.values() if c.status() != 0)
    del copies
    torch.cuda.empty_cache()
    fl, by = point_flops(p), point_bytes(p)
    d = dict(m=p["m"], n=p["n"], k=p["k"], us=round(med, 3), us_min=round(lo, 3),
             us_max=round(hi, 3), tflops=round(fl / med / 1e6, 2),
             gbs=round(by / med / 1e3, 1), hbm_frac=round(by / med / 1e3 / peaks["hbm_gbs"], 3),
             kernel=kernel_name(p))
    if bad:   # a kernel gave up a bounded wait: the time is not a valid measurement
        d["kernel_timeouts"] = bad
        print(f"warning: {bad} workspace(s) of point {p} report a timeout", file=sys.stderr)
    if p.get("kind") == "w4a8":
        fp8 = peaks.get("fp8_tflops")
        d["fp8_tensor_frac"] = round(fl / med / 1e6 / fp8, 3) if fp8 else None
    elif p.get("kind") == "w4a4":
        # dense FP4 peak: the measured bf16 peak times the nominal FP4 / bf16
        # ratio (13.5 / 2.25 PFLOP/s)
        d["fp4_tensor_frac"] = round(fl / med / 1e6 / (peaks["bf16_tflops"] * 6.0), 3)
    else:
        d["tensor_frac"] = round(fl / med / 1e6 / peaks["bf16_tflops"], 3)
    if is_moe:
        d["tokens_per_s"] = round(p["m"] / (med * 1e-6), 1)
        d.pop("n"), d.pop("k")
        d["tokens"] = d.pop("m")
    else:
        cb = cublas_context_us(p, stream)
        d["cublas_bf16_us"] = round(cb, 3)
        d["speedup_vs_cublas"] = round(cb / med, 2)
    return d


def launch_floor_us(stream):
    """The harness floor: a one-element fill kernel launched back to back in
    the same graph harness (no data, no dependency beyond stream order)."""
    import torch
    x = torch.empty(1, device="cuda")
    med, _, _ = graph_time_us(lambda j: x.fill_(float(j)), 40, stream)
    return round(med, 3)


def marginal_rates(per_point, pts):
    """Marginal HBM rate per M between the 4096 x 4096 GEMM and the two
    larger ones: extra algorithmic bytes / extra time (GB/s).  Separates the
    fixed cost of a launch from its streaming rate."""
    out = []
    by = {(p["m"], p["n"], p["k"]): (pp["us"], point_bytes(p)) for pp, p in zip(per_point, pts)}
    for m in sorted({p["m"] for p in pts}):
        base = by.get((m, 4096, 4096))
        if not base:
            continue
        for nk in [(11008, 4096), (4096, 11008)]:
            other = by.get((m,) + nk)
            if other and other[0] > base[0]:
                out.append(dict(m=m, vs=f"{nk[0]}x{nk[1]}",
                                gbs=round((other[1] - base[1]) / (other[0] - base[0]) / 1e3, 1)))
    return out


def measured_peaks_here(stream, peaks):
    """The dense FP8 e4m3 tensor peak, measured once per run (torch._scaled_mm,
    8192^3, best of 10 replays of 10 launches; read-only), so that W4A8 gets a
    tensor fraction; stored into `peaks` as fp8_tflops."""
    import torch
    try:
        n = 8192
        a = torch.randn(n, n, device="cuda").to(torch.float8_e4m3fn)
        b = torch.randn(n, n, device="cuda").to(torch.float8_e4m3fn).t()
        one = torch.ones((), device="cuda")

        def launch(_):
            torch._scaled_mm(a, b, scale_a=one, scale_b=one, out_dtype=torch.bfloat16)
        launch(0)
        torch.cuda.synchronize()
        _, best, _ = graph_time_us(launch, 10, stream, replays=10)
        tf = 2 * n ** 3 / best / 1e6
        peaks["fp8_tflops"] = round(tf, 1)
        return {"fp8_tflops": round(tf, 1), "how": "torch._scaled_mm e4m3 8192^3, best of 10"}
    except Exception as e:   # no FP8 GEMM in this torch build
        return {"fp8_tflops": None, "error": str(e)[:120]}


def nvtx(name):
    """An NVTX range around a phase of the run (for timeline tools; no cost
    inside the timed loops, which it only brackets)."""
    import torch
    return torch.cuda.nvtx.range(name)


def run_ours(args, rank, world, device):
    import torch
    pts, cfg = workload_points(args.workload)
    peaks, peak_src = load_peaks()
    torch.cuda.set_device(device)
    # one buffer set per GEMM of the step
    base = [make_point(p, 1000 + i, device, host=True) for i, p in enumerate(pts)]
    gemms = list(base)
    step_bytes = sum(point_bytes(p) for p in pts)
    if step_bytes < 2 * L2_BYTES:     # single-GEMM workloads: rotate clones to stay cold
        reps = int(np.ceil(2 * L2_BYTES / step_bytes)) + 1
        gemms = [gm if r == 0 else gm.clone() for r in range(reps) for gm in base]
    torch.cuda.synchronize()

    stream = torch.cuda.Stream(device)

    def step_body():
        for gm in gemms:
            gm.launch()

    # warm up eagerly (builds plans, sets kernel attributes), then capture
    with torch.cuda.stream(stream):
        step_body()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step_body()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):   # replays and events on one stream
        for _ in range(args.warmup):
            graph.replay()
    torch.cuda.synchronize()

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    # the timed region can be a few ms: sample every half millisecond, from a
    # process of its own, and keep the samples taken inside the region
    clocks = ClockSampler(torch.cuda.current_device(), period=0.0005)
    clocks.start()
    barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    clocks.mark_start()
    with torch.cuda.stream(stream), nvtx("timed steps"):
        e0.record(stream)
        for _ in range(args.steps):
            graph.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    clocks.mark_end()
    barrier()
    clk = clocks.stop()
    # a kernel that gave up a bounded wait makes the step time invalid
    step_timeouts = sum(1 for gm in {id(g): g for g in gemms}.values() if gm.status() != 0)
    if step_timeouts:
        print(f"warning: {step_timeouts} workspace(s) of the timed step report a timeout",
              file=sys.stderr)
    ms_total = e0.elapsed_time(e1)
    ms_total = reduce_max(ms_total, world)
    flops_step = sum(point_flops(gm.p) for gm in gemms)
    bytes_step = sum(point_bytes(gm.p) for gm in gemms)
    ms_step = ms_total / args.steps
    is_moe = pts[0].get("kind") == "moe"
    if is_moe:
        tokens_step = sum(gm.p["m"] for gm in gemms)
        value = whole_job_rate(tokens_step, args.steps, ms_total, world)
        unit = "tokens/s"
    else:
        value = whole_job_rate(flops_step, args.steps, ms_total, world) / 1e12
        unit = "TFLOP/s"

    # per-GEMM device times (dominant kernel and the per-M table)
    clocks_pts = ClockSampler(torch.cuda.current_device())
    clocks_pts.start()
    with nvtx("points"):
        per_point = [measure_point(bp, p, peaks, stream) for bp, p in zip(base, pts)]
    # the other configurations of the workload set, each timed the same way
    extra_points = []
    if not args.no_extra and args.workload == "sweep":
        for wl in EXTRA_WORKLOADS:
            xpts, xcfg = workload_points(wl)
            for i, p in enumerate(xpts):
                bp = make_point(p, 2000 + i, device)
                torch.cuda.synchronize()
                d = measure_point(bp, p, peaks, stream)
                d["workload"] = xcfg["workload"]
                extra_points.append(d)
                del bp
                torch.cuda.empty_cache()
    clk_pts = clocks_pts.stop()
    # the FP8 peak last: a seconds-long FP8 GEMM loop heats the part and
    # would slow the points measured right after it
    peaks_here = measured_peaks_here(stream, peaks)
    for d in extra_points:
        if "fp8_tensor_frac" in d and peaks.get("fp8_tflops"):
            d["fp8_tensor_frac"] = round(d["tflops"] / peaks["fp8_tflops"], 3)
    # dominant kernel: the instantiation with the largest share of step time
    share = {}
    for pp, p in zip(per_point, pts):
        share.setdefault(pp["kernel"], [0.0, 0, 0, []])
        share[pp["kernel"]][0] += pp["us"]
        share[pp["kernel"]][1] += point_flops(p)
        share[pp["kernel"]][2] += point_bytes(p)
        share[pp["kernel"]][3].append(p["m"])
    dom = max(share.items(), key=lambda kv: kv[1][0])   # over the workload's own GEMMs
    dom_us, dom_flops, dom_bytes, dom_ms = dom[1]
    dom_launches = len(dom_ms)
    # W4A4 runs on the FP4 tensor cores: its peak is the measured bf16 peak
    # times the nominal dense FP4 / bf16 ratio (13.5 / 2.25 PFLOP/s)
    fp4 = pts[0].get("kind") == "w4a4"
    t_peak = peaks["bf16_tflops"] * (6.0 if fp4 else 1.0)
    tensor_bound = (dom_flops / dom_bytes) > t_peak * 1e12 / (peaks["hbm_gbs"] * 1e9)
    if tensor_bound:
        achieved = dom_flops / dom_us / 1e6
        roof = dict(bound="tensor", achieved=round(achieved, 2), peak=round(t_peak, 1),
                    unit="TFLOP/s", frac=round(achieved / t_peak, 4), traffic=None)
    else:
        achieved = dom_bytes / dom_us / 1e3
        roof = dict(bound="hbm", achieved=round(achieved, 1), peak=peaks["hbm_gbs"],
                    unit="GB/s", frac=round(achieved / peaks["hbm_gbs"], 4), traffic=None)
    # DRAM traffic per launch of the dominant kernel from the committed ncu
    # captures of its shapes, while they match the current kernel source
    traffic = committed_traffic()
    digest = kernel_source_digest()
    dom_pts = [p for pp, p in zip(per_point, pts) if pp["kernel"] == dom[0]]
    keys = [shape_key(p) for p in dom_pts]
    if keys and all(k in traffic and traffic[k][1] == digest for k in keys):
        roof["traffic"] = int(sum(traffic[k][0] for k in keys) / len(keys))
    roof.update(kernel=dom[0], launches_per_step=dom_launches,
                per_launch="algorithmic bytes/flops of its GEMMs / mean CUDA-event time per launch",
                peak_source=f"{peak_src} ({'copy bandwidth' if not tensor_bound else 'bf16 burst x 6, the nominal FP4 / bf16 ratio' if fp4 else 'bf16 burst'})")

    # end to end through the C ABI with host buffers (pinned), copies inside the
    # timed region: every step copies each GEMM's activations in and its output
    # back, pipelined over three streams (the copy-in of GEMM i + 1 and the
    # copy-out of GEMM i - 1 overlap GEMM i; opposite directions overlap each
    # other); a buffer is reused only after the previous step's use of it ends
    host_gemms = base
    h2d = sum(gm.a.numel() * gm.a.element_size() for gm in host_gemms)
    d2h = sum(gm.c.numel() * gm.c.element_size() for gm in host_gemms)
    s_in, s_cmp, s_out = (torch.cuda.Stream(device) for _ in range(3))
    done_cmp = [None] * len(host_gemms)    # GEMM i of the previous step (its input is free)
    done_out = [None] * len(host_gemms)    # copy-out i of the previous step (its output is free)

    def e2e_step():
        for i, gm in enumerate(host_gemms):
            ev_in = torch.cuda.Event()
            with torch.cuda.stream(s_in):
                if done_cmp[i] is not None:
                    s_in.wait_event(done_cmp[i])
                gm.copy_in()
                ev_in.record(s_in)
            ev_c = torch.cuda.Event()
            with torch.cuda.stream(s_cmp):
                s_cmp.wait_event(ev_in)
                if done_out[i] is not None:
                    s_cmp.wait_event(done_out[i])
                gm.launch()
                ev_c.record(s_cmp)
            ev_o = torch.cuda.Event()
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_c)
                gm.copy_out()
                ev_o.record(s_out)
            done_cmp[i], done_out[i] = ev_c, ev_o

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    barrier()
    b0 = torch.cuda.Event(enable_timing=True)
    b1 = torch.cuda.Event(enable_timing=True)
    cur = torch.cuda.current_stream(device)
    b0.record(cur)
    for st_ in (s_in, s_cmp, s_out):
        st_.wait_event(b0)
    e2e_steps = max(3, min(args.steps, 20))
    for _ in range(e2e_steps):
        e2e_step()
    for st_ in (s_in, s_cmp, s_out):
        ev = torch.cuda.Event()
        ev.record(st_)
        cur.wait_event(ev)
    b1.record(cur)
    torch.cuda.synchronize()
    e2e_ms = reduce_max(b0.elapsed_time(b1), world)
    flops_pts = sum(point_flops(p) for p in pts)
    if is_moe:
        e2e_val = whole_job_rate(sum(p["m"] for p in pts), e2e_steps, e2e_ms, world)
    else:
        e2e_val = whole_job_rate(flops_pts, e2e_steps, e2e_ms, world) / 1e12

    line = {
        "metric": "W4A16 GEMM TFLOP/s and HBM GB/s vs M (frac of B300 roofline); MoE tokens/s",
        "value": round(value, 3),
        "unit": unit,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": ("bf16 x e4m3 (fp32 acc)" if pts[0].get("kind") == "w4a8"
                  else "bf16" if pts[0]["adt"] == "bf16" else "fp16"),
        "data": "synthetic (seeded random codes, scales, zero points, N(0,1) activations)",
        "config": dict(cfg, gemms_per_step=len(gemms), bytes_per_step=bytes_step,
                       l2="operands of every GEMM are distinct buffers; a step touches "
                          f"{bytes_step / 1e6:.0f} MB > 2x L2, so every GEMM reads cold",
                       parallelism=f"replicas x{world}"),
        "hbm_gbs": round(world * bytes_step * args.steps / (ms_total * 1e-3) / 1e9, 1),
        "roofline": roof,
        "points": per_point + extra_points,
        "floor_us": launch_floor_us(stream),
        "marginal": marginal_rates(per_point, pts),
        "peaks_here": peaks_here,
        "clocks_points": clk_pts,
        "e2e": {"value": round(e2e_val, 3), "unit": unit, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": sum(gm.launches for gm in gemms) * args.steps,
        "clocks": clk,
        "kernel_timeouts": step_timeouts,
    }
    if rank == 0:
        line["cpu_baseline"] = cpu_baseline(pts) if not args.no_cpu else None
    return line


def reduce_max(x, world):
    """The maximum of x over the ranks (NCCL: a device tensor; gloo: host)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank_step, steps, ms_max, world):
    """Whole-job throughput: every rank processes units_per_rank_step per step
    (weak scaling), and the job takes the slowest rank's time."""
    return world * units_per_rank_step * steps / (ms_max * 1e-3)


# ------------------------------------------------------------------ CPU oracle

def _oracle_point(p, seed):
    """The oracle on one unit of the workload: a GEMM (dequant + float64
    matmul; W4A8 with its per-token FP8 quantization), or for MoE the whole
    layer for two tokens.  Returns the units done (flops, or tokens)."""
    from oracle import codecs, gemm, moe, quant
    g = synth.rng(seed)
    m, n, k, gs = p["m"], p["n"], p["k"], p["g"]
    kind = p.get("kind", "w4a16")
    if kind == "w4a8":
        codes = synth.random_bytes(g, (n, k // 2))
        b = synth.random_bytes(g, (n, k // 32), 116, 124)
        ckn, bkn = quant.unpack_mxfp4(codes, b)
        x = codecs.bf16(synth.activations_fp32(g, m, k))
        a8, sc = gemm.act_quant_fp8(x)
        gemm.w4a8_output(a8, sc, ckn, bkn)
        return point_flops(p)
    if kind == "w8a16":
        q = quant.unpack_int_kn(synth.random_words(g, (k // 4, n)), 8, signed=False)
        s = codecs.round_dtype(p["adt"])(
            synth.random_scales_fp32(g, (k // gs, n)).astype(np.float64))
        z = quant.unpack_zeros_bits(synth.random_words(g, (k // gs, n // 4)), 8)
        a = codecs.round_dtype(p["adt"])(synth.activations_fp32(g, m, k))
        gemm.w4a16_output(a, quant.dequant_int(q, s, z, gs, p["adt"]), p["adt"])
        return point_flops(p)
    if kind == "nvfp4":
        codes = synth.random_bytes(g, (n, k // 2))
        sb = synth.random_bytes(g, (n, k // 16), 0x30, 0x48)
        ckn, skn = quant.unpack_nvfp4(codes, sb)
        a = codecs.bf16(synth.activations_fp32(g, m, k))
        gemm.w4a16_output(a, quant.dequant_nvfp4(ckn, skn, 2.0 ** -9), "bf16")
        return point_flops(p)
    if kind == "w4a4":
        codes = synth.random_bytes(g, (n, k // 2))
        sb = synth.random_bytes(g, (n, k // 16), 0x30, 0x48)
        ckn, skn = quant.unpack_nvfp4(codes, sb)
        x = codecs.bf16(synth.activations_fp32(g, m, k))
        a_ts = 6.0 / (6 * 448)
        ac, asb = gemm.act_quant_nvfp4(x, a_ts)
        gemm.w4a4_output(ac, asb, a_ts, ckn, skn, 2.0 ** -9)
        return point_flops(p)
    if kind == "moe":
        s = synth.MOE_SHAPE
        e, h, i, topk, t = s["experts"], s["hidden"], s["inter"], s["topk"], 2
        x = codecs.bf16(synth.activations_fp32(g, t, h))
        ids, wts = moe.route(synth.router_logits_fp32(g, t, e), topk)

        def w_hat(k_, n_):
            def f(_):
                q = quant.unpack_int4_kn(synth.random_words(g, (k_ // 8, n_)), True)
                sc = codecs.bf16(synth.random_scales_fp32(g, (k_ // 128, n_)).astype(np.float64))
                return quant.dequant_int(q, sc, None, 128, "bf16")
            return f
        moe.moe_layer(x, ids, wts, w_hat(h, 2 * i), w_hat(i, h), e, i)
        return t
    qw = synth.random_words(g, (k // 8, n))
    s = codecs.round_dtype(p.get("sdt", p["adt"]))(
        synth.random_scales_fp32(g, (k // gs, n)).astype(np.float64))
    q = quant.unpack_int4_kn(qw, signed=not p["asym"])
    z = quant.unpack_zeros(synth.random_words(g, (k // gs, n // 8))) if p["asym"] else None
    a = codecs.bf16(synth.activations_fp32(g, m, k))
    w_hat = quant.dequant_int(q, s, z, gs, p["adt"])
    gemm.w4a16_output(a, w_hat, p["adt"])
    return point_flops(p)


def _unit_of(pts):
    return "tokens/s" if pts[0].get("kind") == "moe" else "TFLOP/s"


def _scale(units, seconds, pts):
    return units / seconds if pts[0].get("kind") == "moe" else units / seconds / 1e12


def _label(p):
    return f"T={p['m']}" if p.get("kind") == "moe" else f"{p['m']}x{p['n']}x{p['k']}"


def cpu_baseline(pts, budget_s=15.0):
    """Time the oracle on a bounded sample of the workload (its smallest
    units first, until about budget_s of CPU work)."""
    cores = len(os.sched_getaffinity(0))
    done, units, t_used = [], 0, 0.0
    order = sorted(range(len(pts)), key=lambda i: (pts[i]["n"] * pts[i]["k"], pts[i]["m"]))
    t0 = time.perf_counter()
    for i in order:
        if t_used > budget_s:
            break
        units += _oracle_point(pts[i], 77 + i)
        t_used = time.perf_counter() - t0
        done.append(_label(pts[i]))
    what = ("2 tokens through the whole layer" if pts[0].get("kind") == "moe"
            else "numpy float64 dequant + matmul")
    return {"value": round(_scale(units, t_used, pts), 6), "unit": _unit_of(pts), "cores": cores,
            "kind": "oracle",
            "sample": f"{len(done)} of {len(pts)} units ({', '.join(done)}), {what}, "
                      f"{t_used:.1f} s"}


def run_reference(args):
    pts, cfg = workload_points(args.workload)
    cores = len(os.sched_getaffinity(0))
    order = sorted(range(len(pts)), key=lambda i: (pts[i]["n"] * pts[i]["k"], pts[i]["m"]))
    for w in range(args.warmup):
        _oracle_point(pts[order[w % len(order)]], 300 + w)
    units, names = 0, []
    t0 = time.perf_counter()
    for st in range(args.steps):
        p = pts[order[st % len(order)]]
        units += _oracle_point(p, 400 + st)
        names.append(_label(p))
    dt = time.perf_counter() - t0
    v = _scale(units, dt, pts)
    unit = _unit_of(pts)
    sample = (f"one unit of the workload per step, cycling smallest first "
              f"({', '.join(sorted(set(names)))}); the CPU oracle in numpy float64")
    return {"impl": "reference", "metric": "W4A16 GEMM TFLOP/s and HBM GB/s vs M (frac of B300 "
            "roofline); MoE tokens/s", "value": round(v, 6), "unit": unit, "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(dt * 1e3 / max(args.steps, 1), 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": cfg,
            "cpu_baseline": {"value": round(v, 6), "unit": unit, "cores": cores,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(v, 6), "unit": unit, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


# ------------------------------------------------------------------ main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="sweep",
                    help="sweep | f16s | w8a16 | nvfp4 | w4a4 | w4a4_large | w4a16_m16 | large | "
                         "w4a8 | moe16 | moe256 | moe4096 | "
                         "shape:M,N,K[,sym|asym][,bf16|fp16][,f16s][,w4a4]")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--no-extra", action="store_true",
                    help="sweep only: skip timing the other configurations")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    try:
        workload_points(args.workload)
    except (ValueError, IndexError):
        ap.error(f"unknown workload {args.workload!r}")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return
    import torch
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    line = run_ours(args, rank, world, f"cuda:{local}")
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
