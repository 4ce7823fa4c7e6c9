"""Benchmark of the quantized-weight GEMM hot path on B300.

Default workload (one JSON line on rank 0): the W4A16 asymmetric sweep --
UINT4 weights with bf16 group-128 scales and uint4 zero points, bf16
activations, (N, K) in {(4096, 4096), (11008, 4096), (4096, 11008)} x
M in {1, 4, 16, 64, 256, 1024}.  One step runs all 18 GEMMs once through the
library's C ABI; every GEMM has its own weight and activation buffers, so a
step touches ~330 MB and each GEMM reads its operands cold from HBM (the
126 MB L2 is flushed by the rest of the step).  The step is captured in a
CUDA graph and replayed.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload sweep|w4a16_m16|large|moe]

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
    if name == "sweep":
        return sweep_points(), dict(workload="w4a16_asym_sweep", shapes=synth.W4A16_ASYM_SHAPES,
                                    ms=synth.W4A16_ASYM_MS, group=128, weights="uint4+zp",
                                    act="bf16")
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
    raise ValueError(name)


def point_bytes(p):
    m, n, k, g = p["m"], p["n"], p["k"], p["g"]
    b = n * k // 2 + (k // g) * n * 2 + m * k * 2 + m * n * 2
    if p["asym"]:
        b += (k // g) * n // 2
    return b


def point_flops(p):
    return 2 * p["m"] * p["n"] * p["k"]


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """SM clock and clock-event reasons sampled through NVML (read-only queries)
    every 50 ms on a background thread while the timed region runs."""

    REASONS = {"hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20, "hw_thermal_slowdown": 0x40,
               "sw_power_cap": 0x4, "hw_power_brake_slowdown": 0x80}

    def __init__(self, index):
        self.index = index
        self.samples = []
        self.max_mhz = None
        self._stop = None
        self._thread = None
        self.error = None

    def start(self):
        import threading
        try:
            import pynvml
            pynvml.nvmlInit()
            h = pynvml.nvmlDeviceGetHandleByIndex(self.index)
            self.max_mhz = pynvml.nvmlDeviceGetMaxClockInfo(h, pynvml.NVML_CLOCK_SM)
        except Exception as e:       # no NVML: report it instead of clocks
            self.error = f"nvml unavailable: {e}"
            return
        self._stop = threading.Event()

        def run():
            while not self._stop.is_set():
                try:
                    mhz = pynvml.nvmlDeviceGetClockInfo(h, pynvml.NVML_CLOCK_SM)
                    rs = pynvml.nvmlDeviceGetCurrentClocksEventReasons(h)
                    self.samples.append((mhz, rs))
                except Exception as e:
                    self.error = str(e)
                self._stop.wait(0.05)

        self._thread = threading.Thread(target=run, daemon=True)
        self._thread.start()

    def stop(self):
        if self._thread is not None:
            self._stop.set()
            self._thread.join()
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "samples": 0,
                    "reasons": [self.error or "no samples"]}
        reasons = sorted({nm for _, rs in self.samples for nm, bit in self.REASONS.items()
                          if rs & bit})
        return {"sm_mhz": statistics.median(m for m, _ in self.samples),
                "sm_max_mhz": self.max_mhz, "samples": len(self.samples), "reasons": reasons}


# ------------------------------------------------------------------ our arm

class GemmPoint:
    """Buffers of one GEMM of the workload (own weights, activations, output).

    ``clone()`` duplicates every device buffer, so that a rotation of clones
    reads its operands cold from HBM."""

    def __init__(self, p, seed, device, host=False, src=None):
        import torch
        from quantized_weight_gemm_run_b300 import qgemm as Q
        from quantized_weight_gemm_run_b300.api import W4A16Linear
        self.p, self.Q = p, Q
        m, n, k, gs = p["m"], p["n"], p["k"], p["g"]
        dt = torch.bfloat16 if p["adt"] == "bf16" else torch.float16
        if src is None:
            g = synth.rng(seed)
            qweight = torch.from_numpy(synth.random_words(g, (k // 8, n))).to(device)
            scales = torch.from_numpy(synth.random_scales_fp32(g, (k // gs, n))).to(dt).to(device)
            qzeros = (torch.from_numpy(synth.random_words(g, (k // gs, n // 8))).to(device)
                      if p["asym"] else None)
            self.lin = W4A16Linear(qweight, scales, qzeros, n, k, gs, dt)
            del qweight, scales, qzeros
            self.a = torch.from_numpy(synth.activations_fp32(g, m, k)).to(dt).to(device)
        else:
            import copy
            self.lin = copy.copy(src.lin)
            self.lin.w = src.lin.w.clone()
            self.lin.s = src.lin.s.clone()
            self.lin.z = None if src.lin.z is None else src.lin.z.clone()
            self.a = src.a.clone()
        self.c = torch.empty(m, n, dtype=dt, device=device)
        st, nbytes = Q.qgemm_workspace_size(self.lin.layer, self.lin.dense, None, m)
        Q.check(st)
        self.ws = torch.zeros(nbytes, dtype=torch.uint8, device=device)
        if host:
            self.a_host = self.a.cpu().pin_memory()
            self.c_host = torch.empty(m, n, dtype=dt).pin_memory()

    def clone(self):
        return GemmPoint(self.p, 0, self.c.device, src=self)

    def launch(self):
        Q = self.Q
        Q.check(Q.qgemm_run(self.lin.layer, self.lin.dense, None, self.p["m"], self.a, None,
                            self.lin.w, self.lin.s, self.lin.z, None, self.c, self.ws,
                            self.ws.numel()))

    def launch_e2e(self):
        self.a.copy_(self.a_host, non_blocking=True)
        self.launch()
        self.c_host.copy_(self.c, non_blocking=True)


def cold_copies(p):
    """Distinct buffer sets needed so that a rotation exceeds twice the L2."""
    return int(np.ceil(2 * L2_BYTES / point_bytes(p))) + 1


def kernel_name(p):
    bt = 16 if p["m"] <= 16 else 32 if p["m"] <= 32 else 64 if p["m"] <= 64 else 128
    return f"w4a16_kernel<{bt},{'fp16' if p['adt'] == 'fp16' else 'bf16'},dense>"


def run_ours(args, rank, world, device):
    import torch
    pts, cfg = workload_points(args.workload)
    peaks, peak_src = load_peaks()
    torch.cuda.set_device(device)
    # one buffer set per GEMM of the step
    base = [GemmPoint(p, 1000 + i, device, host=True) for i, p in enumerate(pts)]
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

    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(args.steps):
            graph.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    clk = clocks.stop()
    ms_total = e0.elapsed_time(e1)
    ms_total = reduce_max(ms_total, world)
    flops_step = sum(point_flops(gm.p) for gm in gemms)
    bytes_step = sum(point_bytes(gm.p) for gm in gemms)
    ms_step = ms_total / args.steps
    value = world * flops_step * args.steps / (ms_total * 1e-3) / 1e12

    # per-GEMM device times (dominant kernel and the per-M table): each GEMM
    # launched back to back over a rotation of cold clones, inside a graph
    per_point = []
    for i, p in enumerate(pts):
        copies = [base[i]] + [base[i].clone() for _ in range(cold_copies(p) - 1)]
        r = max(20, len(copies))
        g2 = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g2, stream=stream):
            for j in range(r):
                copies[j % len(copies)].launch()
        torch.cuda.synchronize()
        a0 = torch.cuda.Event(enable_timing=True)
        a1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            for _ in range(3):
                g2.replay()
            a0.record(stream)
            g2.replay()
            a1.record(stream)
        torch.cuda.synchronize()
        us = a0.elapsed_time(a1) * 1e3 / r
        per_point.append(dict(m=p["m"], n=p["n"], k=p["k"], us=round(us, 3),
                              tflops=round(point_flops(p) / us / 1e6, 2),
                              gbs=round(point_bytes(p) / us / 1e3, 1),
                              hbm_frac=round(point_bytes(p) / us / 1e3 / peaks["hbm_gbs"], 3),
                              tensor_frac=round(point_flops(p) / us / 1e6 / peaks["bf16_tflops"], 3),
                              kernel=kernel_name(p)))
        del g2, copies
        torch.cuda.empty_cache()
    # dominant kernel: the instantiation with the largest share of step time
    share = {}
    for pp, p in zip(per_point, pts):
        share.setdefault(pp["kernel"], [0.0, 0, 0, []])
        share[pp["kernel"]][0] += pp["us"]
        share[pp["kernel"]][1] += point_flops(p)
        share[pp["kernel"]][2] += point_bytes(p)
        share[pp["kernel"]][3].append(p["m"])
    dom = max(share.items(), key=lambda kv: kv[1][0])
    dom_us, dom_flops, dom_bytes, dom_ms = dom[1]
    dom_launches = len(dom_ms)
    tensor_bound = (dom_flops / dom_bytes) > peaks["bf16_tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
    if tensor_bound:
        achieved = dom_flops / dom_us / 1e6
        roof = dict(bound="tensor", achieved=round(achieved, 2), peak=peaks["bf16_tflops"],
                    unit="TFLOP/s", frac=round(achieved / peaks["bf16_tflops"], 4),
                    traffic=None)
    else:
        achieved = dom_bytes / dom_us / 1e3
        roof = dict(bound="hbm", achieved=round(achieved, 1), peak=peaks["hbm_gbs"],
                    unit="GB/s", frac=round(achieved / peaks["hbm_gbs"], 4), traffic=None)
    roof.update(kernel=dom[0], launches_per_step=dom_launches,
                per_launch="algorithmic bytes/flops of its GEMMs / mean CUDA-event time per launch",
                peak_source=f"{peak_src} ({'bf16 burst' if tensor_bound else 'copy bandwidth'})")

    # end to end through the C ABI with host buffers (pinned), copies inside the timed region
    host_gemms = base
    h2d = sum(gm.a.numel() * gm.a.element_size() for gm in host_gemms)
    d2h = sum(gm.c.numel() * gm.c.element_size() for gm in host_gemms)
    for _ in range(2):
        for gm in host_gemms:
            gm.launch_e2e()
    torch.cuda.synchronize()
    barrier()
    t0 = time.perf_counter()
    b0 = torch.cuda.Event(enable_timing=True)
    b1 = torch.cuda.Event(enable_timing=True)
    b0.record()
    e2e_steps = max(3, min(args.steps, 20))
    for _ in range(e2e_steps):
        for gm in host_gemms:
            gm.launch_e2e()
    b1.record()
    torch.cuda.synchronize()
    e2e_ms = reduce_max(b0.elapsed_time(b1), world)
    flops_pts = sum(point_flops(p) for p in pts)
    e2e_val = world * flops_pts * e2e_steps / (e2e_ms * 1e-3) / 1e12

    line = {
        "metric": "W4A16 GEMM TFLOP/s and HBM GB/s vs M (frac of B300 roofline); MoE tokens/s",
        "value": round(value, 3),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if pts[0]["adt"] == "bf16" else "fp16",
        "data": "synthetic (seeded random 4-bit codes, scales, zero points, N(0,1) activations)",
        "config": dict(cfg, gemms_per_step=len(gemms), bytes_per_step=bytes_step,
                       l2="operands of every GEMM are distinct buffers; a step touches "
                          f"{bytes_step / 1e6:.0f} MB > 2x L2, so every GEMM reads cold",
                       parallelism=f"replicas x{world}"),
        "hbm_gbs": round(world * bytes_step * args.steps / (ms_total * 1e-3) / 1e9, 1),
        "roofline": roof,
        "points": per_point,
        "e2e": {"value": round(e2e_val, 3), "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": len(gemms) * args.steps,
        "clocks": clk,
    }
    if rank == 0:
        line["cpu_baseline"] = cpu_baseline(pts) if not args.no_cpu else None
    return line


def reduce_max(x, world):
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ CPU oracle

def _oracle_point(p, seed):
    """The oracle on one GEMM of the workload (dequant + float64 matmul)."""
    from oracle import codecs, quant, gemm
    g = synth.rng(seed)
    m, n, k, gs = p["m"], p["n"], p["k"], p["g"]
    qw = synth.random_words(g, (k // 8, n))
    s = codecs.bf16(synth.random_scales_fp32(g, (k // gs, n)).astype(np.float64))
    q = quant.unpack_int4_kn(qw, signed=not p["asym"])
    z = quant.unpack_zeros(synth.random_words(g, (k // gs, n // 8))) if p["asym"] else None
    a = codecs.bf16(synth.activations_fp32(g, m, k))
    w_hat = quant.dequant_int(q, s, z, gs, p["adt"])
    return gemm.w4a16_output(a, w_hat, p["adt"])


def cpu_baseline(pts, budget_s=15.0):
    """Time the oracle on a bounded sample of the workload's GEMMs."""
    cores = len(os.sched_getaffinity(0))
    done, flops, t_used = [], 0, 0.0
    order = sorted(range(len(pts)), key=lambda i: (pts[i]["n"] * pts[i]["k"], pts[i]["m"]))
    t0 = time.perf_counter()
    for i in order:
        if t_used > budget_s:
            break
        p = pts[i]
        t1 = time.perf_counter()
        _oracle_point(p, 77 + i)
        t_used = time.perf_counter() - t0
        flops += point_flops(p)
        done.append(f"{p['m']}x{p['n']}x{p['k']}")
    return {"value": round(flops / t_used / 1e12, 6), "unit": "TFLOP/s", "cores": cores,
            "kind": "oracle",
            "sample": f"{len(done)} of {len(pts)} GEMMs ({', '.join(done)}), numpy float64 "
                      f"dequant + matmul, {t_used:.1f} s"}


def run_reference(args):
    pts, cfg = workload_points(args.workload)
    cores = len(os.sched_getaffinity(0))
    order = sorted(range(len(pts)), key=lambda i: (pts[i]["n"] * pts[i]["k"], pts[i]["m"]))
    for w in range(args.warmup):
        _oracle_point(pts[order[w % len(order)]], 300 + w)
    flops, names = 0, []
    t0 = time.perf_counter()
    for s in range(args.steps):
        p = pts[order[s % len(order)]]
        _oracle_point(p, 400 + s)
        flops += point_flops(p)
        names.append(f"{p['m']}x{p['n']}x{p['k']}")
    dt = time.perf_counter() - t0
    v = flops / dt / 1e12
    sample = (f"one GEMM of the workload per step, cycling smallest first "
              f"({', '.join(sorted(set(names)))}); numpy float64 dequant + matmul")
    return {"impl": "reference", "metric": "W4A16 GEMM TFLOP/s and HBM GB/s vs M (frac of B300 "
            "roofline); MoE tokens/s", "value": round(v, 6), "unit": "TFLOP/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(dt * 1e3 / max(args.steps, 1), 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": cfg,
            "cpu_baseline": {"value": round(v, 6), "unit": "TFLOP/s", "cores": cores,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(v, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


# ------------------------------------------------------------------ main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="sweep", choices=["sweep", "w4a16_m16", "large"])
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
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
