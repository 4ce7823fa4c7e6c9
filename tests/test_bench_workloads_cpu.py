"""The benchmark's host-side bookkeeping on CPU: the algorithmic bytes and
flops it divides by, the kernel each point is charged to (which must match
the planner's routing), and the keys under which committed DRAM-traffic
figures are looked up."""

import sys

import pytest

from conftest import ROOT

sys.path.insert(0, ROOT)

import bench  # noqa: E402
import synth  # noqa: E402


def _pt(name, i=0):
    return bench.workload_points(name)[0][i]


def test_algorithmic_bytes_by_format():
    m, n, k, g = 16, 4096, 4096, 128
    acts, out = m * k * 2, m * n * 2
    scales, zeros4, zeros8 = (k // g) * n * 2, (k // g) * n // 2, (k // g) * n
    base = dict(m=m, n=n, k=k, g=g, adt="bf16")
    assert bench.point_bytes(dict(base, asym=False)) == n * k // 2 + scales + acts + out
    assert bench.point_bytes(dict(base, asym=True)) == n * k // 2 + scales + zeros4 + acts + out
    assert bench.point_bytes(dict(base, asym=True, kind="w8a16")) == \
        n * k + scales + zeros8 + acts + out
    nv = dict(base, kind="nvfp4", g=16, asym=False)
    assert bench.point_bytes(nv) == n * k // 2 + (k // 16) * n * 2 + acts + out
    assert bench.point_flops(dict(base, asym=False)) == 2 * m * n * k


@pytest.mark.parametrize("name", ["sweep", "f16s", "w8a16", "nvfp4"])
def test_sweep_workloads_cover_the_same_shapes(name):
    pts, cfg = bench.workload_points(name)
    got = sorted((p["m"], p["n"], p["k"]) for p in pts)
    want = sorted((m, n, k) for m in synth.W4A16_ASYM_MS for (n, k) in synth.W4A16_ASYM_SHAPES)
    assert got == want and cfg["workload"].endswith("sweep")


def test_kernel_names_follow_the_planner():
    # dense INT4/UINT4 with scales in the activation dtype: small-M kernel up to 16 rows
    assert bench.kernel_name(dict(_pt("sweep"), m=16)).startswith("w4a16_mma_kernel")
    assert bench.kernel_name(dict(_pt("sweep"), m=17)) == "w4a16_kernel<32,bf16,dense>"
    # ... except 9-16 rows on a long K (K >= 2 N): the tcgen05 kernel
    long_k = dict(_pt("sweep"), n=4096, k=11008)
    assert bench.kernel_name(dict(long_k, m=16)) == "w4a16_kernel<16,bf16,dense>"
    assert bench.kernel_name(dict(long_k, m=8)) == "w4a16_mma_kernel<bf16,1>"
    # fp16 scales with bf16 activations: small-M kernel up to 16 rows, as for the sweep
    assert bench.kernel_name(dict(_pt("f16s"), m=1)) == "w4a16_mma_kernel<bf16_f16scales,1>"
    assert bench.kernel_name(dict(_pt("f16s"), m=64)) == "w4a16_kernel<64,bf16_f16scales,dense>"
    # 8-bit codes: the tcgen05 kernel at every m
    assert bench.kernel_name(dict(_pt("w8a16"), m=1)) == "w4a16_kernel<16,int8_bf16,dense>"
    assert bench.kernel_name(dict(_pt("w8a16"), m=1024)) == "w4a16_kernel<128,int8_bf16,dense>"
    # NVFP4 weights: the small-M kernel up to 2^24 weights, or at m <= 8 with k <= 4096
    nv = _pt("nvfp4")
    assert bench.kernel_name(dict(nv, m=16, n=4096, k=4096)) == "w4a16_mma_kernel<nvfp4_bf16,2>"
    assert bench.kernel_name(dict(nv, m=8, n=11008, k=4096)) == "w4a16_mma_kernel<nvfp4_bf16,1>"
    assert bench.kernel_name(dict(nv, m=9, n=11008, k=4096)) == "w4a16_kernel<16,nvfp4_bf16,dense>"
    assert bench.kernel_name(dict(nv, m=1, n=4096, k=11008)) == "w4a16_kernel<16,nvfp4_bf16,dense>"
    assert bench.kernel_name(dict(nv, m=256)) == "w4a16_kernel<128,nvfp4_bf16,dense>"
    # W4A4: 16-token tiles up to 16 rows, then the smallest tile whose tiles fit one wave
    w4 = _pt("w4a4")
    for m, n, bt in ((16, 4096, 16), (64, 4096, 32), (64, 11008, 64), (256, 4096, 64),
                     (256, 11008, 128), (1024, 4096, 128)):
        assert bench.kernel_name(dict(w4, m=m, n=n)) == f"act_quant_nvfp4_kernel + w4a4_kernel<{bt}>"


def test_traffic_keys_separate_formats():
    p = dict(_pt("sweep"), m=256)
    assert bench.shape_key(p) == f"256x{p['n']}x{p['k']},asym,bf16"
    assert bench.shape_key(dict(_pt("f16s"), m=256)) == f"256x{p['n']}x{p['k']},asym,bf16,f16s"
    assert bench.shape_key(_pt("w8a16")) is None       # no committed figures for 8-bit codes
    key16 = bench.shape_key(bench.workload_points("shape:16,4096,4096,sym,fp16")[0][0])
    assert key16 == "16x4096x4096,sym,fp16"


def test_committed_traffic_lines_parse():
    """Every committed traffic line has a shape key the bench can produce, a
    byte count and a 16-hex-digit source digest (the bench reports a figure
    only while that digest matches the sources; comments do not count)."""
    import re
    lines = bench.committed_traffic()
    assert lines
    for key, (nbytes, src) in lines.items():
        assert re.fullmatch(r"\d+x\d+x\d+,(sym|asym),(bf16|fp16)(,f16s)?", key), key
        assert nbytes > 0 and re.fullmatch(r"[0-9a-f]{16}", src)
    assert bench.source_without_comments("int a; // x\n/* y */ int b;\n") == "int a;\n int b;"


def test_clock_sampler_keeps_the_timed_window():
    """The summary keeps the samples taken inside [mark_start, mark_end]: the
    median SM clock and the union of the named clock-event reasons there."""
    c = bench.ClockSampler(0)
    c.window = [10.0, 10.01]
    c.samples = [(9.0, 1200, 0x4), (10.002, 2032, 0x0), (10.006, 2000, 0x4), (11.0, 900, 0x40)]
    s = c.summary()
    assert s["samples"] == 2 and s["sm_mhz"] == 2016.0 and s["reasons"] == ["sw_power_cap"]
    # a window with no sample inside takes the samples within 50 ms of it
    c.window = [10.003, 10.004]
    s = c.summary()
    assert s["samples"] == 2 and s["sm_mhz"] == 2016.0
    c.samples = []
    assert c.summary()["samples"] == 0
