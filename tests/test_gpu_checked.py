"""The checked build (libqgemm_checked.so: the library compiled with
QGEMM_CHECKED, every kernel testing the global-memory indexes it computes
before each access) on the GPU, in a child process that loads it
(QGEMM_LIBRARY=checked):

- its self-test records an index-check failure in the workspace status word
  and qgemm_check_status reports QGEMM_ERR_DEVICE (nothing is accessed);
- a caller mistake the host cannot see, an out-of-range inverse permutation
  given to qgemm_moe_combine, is caught by the combine kernel's test (the
  bad reads are skipped) and reported by qgemm_checked_status;
- on valid inputs no test fires and every result is bitwise that of the
  unchecked build: the persistent kernel's split tiles (atomic and fixed
  order), whole tiles, the cluster split, the small-M kernel, W4A8 with the
  fused quantization, the gated epilogue and a grouped MoE layer.

The out-of-range call runs in the checked child only."""

import os
import subprocess
import sys

import numpy as np
import pytest
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
if HERE not in sys.path:
    sys.path.insert(0, HERE)
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def _cases():
    """Seeded layers and activations -> {name: output uint16 bits}."""
    import synth
    from gpu_helpers import DEV, TD, Case, linear
    from oracle import quant
    from quantized_weight_gemm_run_b300 import qgemm as Q
    from quantized_weight_gemm_run_b300.api import MoELayer, W4A16Linear, W4A8Linear
    Q.qgemm_set_wait_limit_ns(1_000_000_000)
    out = {}

    def bits(t):
        torch.cuda.synchronize()
        return t.cpu().view(torch.int16).numpy().copy()

    runs = [
        ("stream_k", Case(300, 640, 2048, 128, "bf16", False, seed=1),
         dict(tuning=Q.tuning_config(block_tok=64, max_ctas=7))),
        ("fixed_order", Case(70, 384, 1536, 64, "fp16", True, seed=2, bias=True),
         dict(tuning=Q.tuning_config(block_tok=32, max_ctas=5), deterministic=True)),
        ("whole", Case(200, 512, 1024, 128, "bf16", True, seed=3),
         dict(tuning=Q.tuning_config(split_k=1))),
        ("cluster", Case(45, 384, 11 * 128, 128, "bf16", False, seed=4),
         dict(tuning=Q.tuning_config(block_tok=64, split_k=4, kernel=3))),
        ("small_m", Case(5, 512, 2048, 128, "fp16", True, seed=5), dict()),
    ]
    for name, c, kw in runs:
        lin = linear(c, **kw)
        out[name] = bits(lin(c.dev_act()))
        assert lin.status() == Q.QGEMM_OK, (name, Q.last_error())
    c = Case(37, 384, 512, 128, "bf16", False, seed=6, bias=True)
    qw, sc, qz = c.dev_weights()
    lin = W4A16Linear(qw, sc, qz, c.n, c.k, c.g, TD[c.adt], bias=c.dev_bias(), gated=True)
    out["gated"] = bits(lin(c.dev_act()))
    assert lin.status() == Q.QGEMM_OK
    g = synth.rng(7)
    for m in (3, 70):
        w = synth.weights_fp32(g, 2048, 640)
        ckn, bkn = quant.quantize_mxfp4(w)
        cnk, bnk = quant.pack_mxfp4(ckn, bkn)
        lin = W4A8Linear(torch.from_numpy(cnk).to(DEV), torch.from_numpy(bnk).to(DEV), 640, 2048)
        x = torch.from_numpy(synth.activations_fp32(g, m, 2048)).to(torch.bfloat16).to(DEV)
        out[f"w4a8_{m}"] = bits(lin(x))
        assert lin.status() == Q.QGEMM_OK
    e, topk, hid, inter, t = 4, 2, 256, 128, 9

    def stack(k, n, gated=False):
        qw = torch.from_numpy(synth.random_words(g, (e * k // 8, n))).to(DEV)
        sc = torch.from_numpy(synth.random_scales_fp32(g, (e * k // 128, n))).to(
            torch.bfloat16).to(DEV)
        return W4A16Linear(qw, sc, None, n, k, 128, torch.bfloat16, num_experts=e, gated=gated)
    l1, l2 = stack(hid, 2 * inter, gated=True), stack(inter, hid)
    layer = MoELayer(l1, l2, e, topk)
    x = torch.from_numpy(synth.activations_fp32(g, t, hid)).to(torch.bfloat16).to(DEV)
    ids = torch.from_numpy(synth.rng(8).integers(0, e, size=(t, topk)).astype(np.int32)).to(DEV)
    wts = torch.full((t, topk), 0.5, dtype=torch.float32, device=DEV)
    out["moe"] = bits(layer(x, ids, wts))
    assert l1.status() == Q.QGEMM_OK and l2.status() == Q.QGEMM_OK
    assert Q.qgemm_checked_status() == Q.QGEMM_OK, Q.last_error()
    return out


def _child(path):
    from quantized_weight_gemm_run_b300 import qgemm as Q
    assert Q.qgemm_checked_build() == 1, Q._LIB_PATH
    dev = "cuda:0"
    # 1. the self-test: one failing index test, reported as a device error
    ws = torch.zeros(256, dtype=torch.uint8, device=dev)
    assert Q.qgemm_checked_selftest(ws) == Q.QGEMM_OK
    assert Q.qgemm_check_status(ws) == Q.QGEMM_ERR_DEVICE
    assert "index check" in Q.last_error()
    assert Q.qgemm_check_status(ws) == Q.QGEMM_OK          # read and cleared
    # 2. a caller's out-of-range inverse permutation: the reads are skipped
    t, topk, hidden = 4, 2, 256
    y2 = torch.ones(t * topk, hidden, dtype=torch.bfloat16, device=dev)
    inv = torch.tensor([0, 1, 2, 3, 4, 5, 6, 1 << 20], dtype=torch.int32, device=dev)
    wts = torch.full((t, topk), 0.5, dtype=torch.float32, device=dev)
    y = torch.empty(t, hidden, dtype=torch.bfloat16, device=dev)
    assert Q.qgemm_moe_combine(y2, inv, wts, t, topk, hidden, y) == Q.QGEMM_OK
    assert Q.qgemm_checked_status() == Q.QGEMM_ERR_DEVICE
    assert Q.qgemm_checked_status() == Q.QGEMM_OK
    assert torch.all(y[:3].float() == 1.0) and torch.all(y[3].float() == 0.5)
    # 3. valid inputs: no test fires
    np.savez(path, **_cases())


@pytest.mark.gpu
def test_checked_build_on_gpu(tmp_path):
    path = str(tmp_path / "checked.npz")
    env = dict(os.environ, QGEMM_LIBRARY="checked")
    res = subprocess.run([sys.executable, os.path.abspath(__file__), path], env=env,
                         capture_output=True, text=True, timeout=900)
    assert res.returncode == 0, res.stdout[-3000:] + res.stderr[-3000:]
    got = np.load(path)
    from quantized_weight_gemm_run_b300 import qgemm as Q
    assert Q.qgemm_checked_build() == 0
    want = _cases()
    assert sorted(got.files) == sorted(want)
    for name, bits in want.items():
        assert np.array_equal(got[name], bits), f"{name}: checked build differs"


if __name__ == "__main__":
    _child(sys.argv[1])
