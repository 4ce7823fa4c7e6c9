"""CPU-side checks of the library boundary: the shared library loads, exports
every entry point the header declares, and its host-side validation rejects
bad configurations without needing a GPU."""

import os
import re

import pytest

from conftest import ROOT


def _header_functions():
    src = open(os.path.join(ROOT, "include", "qgemm.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(qgemm_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def Q():
    from quantized_weight_gemm_run_b300 import qgemm
    return qgemm


def test_header_declares_the_boundary():
    names = _header_functions()
    for required in ("qgemm_pack_weights", "qgemm_run", "qgemm_grouped_run"):
        assert required in names


def test_library_exports_every_declared_symbol(Q):
    missing = [n for n in _header_functions() if not hasattr(Q.lib, n)]
    assert not missing, missing


def test_binding_has_every_entry_point(Q):
    missing = [n for n in _header_functions() if not callable(getattr(Q, n, None))]
    assert not missing, missing


def _layer(Q, **kw):
    d = dict(n=4096, k=4096, group_size=128, weight_format=Q.QGEMM_W_INT4_SYM,
             scale_format=Q.QGEMM_S_FP16, zero_format=Q.QGEMM_Z_NONE, act_dtype=Q.QGEMM_FP16,
             out_dtype=Q.QGEMM_FP16, has_bias=0, num_experts=1)
    d.update(kw)
    return Q.layer_config(**d)


def test_packed_size_host_only(Q):
    blocks = (4096 // 128) ** 2
    st, b = Q.qgemm_packed_size(_layer(Q))
    assert st == Q.QGEMM_OK
    assert b == blocks * (8192 + 256)                    # codes + one scale per row
    st, b = Q.qgemm_packed_size(_layer(Q, weight_format=Q.QGEMM_W_UINT4_ZP,
                                       zero_format=Q.QGEMM_Z_UINT4, group_size=32,
                                       num_experts=3))
    assert st == Q.QGEMM_OK and b == 3 * blocks * (8192 + 4 * 256 + 4 * 128)
    st, b = Q.qgemm_packed_size(_layer(Q, weight_format=Q.QGEMM_W_MXFP4,
                                       scale_format=Q.QGEMM_S_E8M0, group_size=32,
                                       act_dtype=Q.QGEMM_FP8E4M3, out_dtype=Q.QGEMM_BF16))
    assert st == Q.QGEMM_OK and b == blocks * (8192 + 512)
    # NVFP4: codes + 8 x 128 16-bit block scales per block, then the fp32 tensor
    # scales of the experts padded to 16 bytes
    st, b = Q.qgemm_packed_size(_layer(Q, weight_format=Q.QGEMM_W_NVFP4,
                                       scale_format=Q.QGEMM_S_E4M3, group_size=16,
                                       act_dtype=Q.QGEMM_BF16, out_dtype=Q.QGEMM_BF16,
                                       num_experts=5))
    assert st == Q.QGEMM_OK and b == 5 * blocks * (8192 + 2048) + 32
    # the gate/up interleave of a gated layer moves columns, it adds no bytes
    st, b = Q.qgemm_packed_size(_layer(Q, act_dtype=Q.QGEMM_BF16, out_dtype=Q.QGEMM_BF16,
                                       scale_format=Q.QGEMM_S_BF16, gated_act=1))
    assert st == Q.QGEMM_OK and b == blocks * (8192 + 256)
    # W8A16: 16384 code bytes per block, the scales and zero points as INT4
    st, b = Q.qgemm_packed_size(_layer(Q, weight_format=Q.QGEMM_W_INT8_SYM))
    assert st == Q.QGEMM_OK and b == blocks * (16384 + 256)
    st, b = Q.qgemm_packed_size(_layer(Q, weight_format=Q.QGEMM_W_UINT8_ZP,
                                       zero_format=Q.QGEMM_Z_UINT8, group_size=64,
                                       num_experts=2))
    assert st == Q.QGEMM_OK and b == 2 * blocks * (16384 + 2 * 256 + 2 * 128)
    # fp16 scales against bf16 activations: the scales keep their 16 bits
    st, b = Q.qgemm_packed_size(_layer(Q, act_dtype=Q.QGEMM_BF16, out_dtype=Q.QGEMM_BF16,
                                       scale_format=Q.QGEMM_S_FP16))
    assert st == Q.QGEMM_OK and b == blocks * (8192 + 256)


@pytest.mark.parametrize("bad,code", [
    (dict(n=100), "UNSUPPORTED"),
    (dict(k=1000), "UNSUPPORTED"),
    (dict(group_size=48), "UNSUPPORTED"),
    (dict(group_size=384), "UNSUPPORTED"),          # does not divide K = 4096
    (dict(zero_format=1), "UNSUPPORTED"),           # zeros with symmetric INT4
    (dict(out_dtype=1), "UNSUPPORTED"),             # W4A16 output dtype differs
    (dict(scale_format=1), "UNSUPPORTED"),          # bf16 scales with fp16 activations
    (dict(weight_format=2, scale_format=2, group_size=32, act_dtype=2, out_dtype=1,
          zero_format=1), "UNSUPPORTED"),          # zero points with MXFP4
    (dict(weight_format=9), "UNSUPPORTED"),
    (dict(n=0), "INVALID_ARG"),
    (dict(num_experts=0), "INVALID_ARG"),
    (dict(has_bias=2), "INVALID_ARG"),
    (dict(gated_act=2), "INVALID_ARG"),
    (dict(weight_format=3, scale_format=3, group_size=32), "UNSUPPORTED"),   # NVFP4 is per 16
    (dict(weight_format=3, scale_format=0, group_size=16), "UNSUPPORTED"),   # needs e4m3 scales
    (dict(weight_format=3, scale_format=3, group_size=16, zero_format=1), "UNSUPPORTED"),
    (dict(gated_act=1), "UNSUPPORTED"),             # a gated output must be bf16
    (dict(weight_format=4, zero_format=2), "UNSUPPORTED"),   # zeros with symmetric INT8
    (dict(weight_format=5, zero_format=1), "UNSUPPORTED"),   # UINT8 needs 8-bit zeros
    (dict(weight_format=4, act_dtype=1, out_dtype=1), "UNSUPPORTED"),   # fp16 scales, bf16 act
    (dict(weight_format=4, group_size=48), "UNSUPPORTED"),
])
def test_rejections_are_clear(Q, bad, code):
    st, _ = Q.qgemm_packed_size(_layer(Q, **bad))
    assert Q.status_string(st) == f"QGEMM_ERR_{code}"
    assert Q.last_error()


def test_status_strings(Q):
    assert Q.status_string(Q.QGEMM_OK) == "QGEMM_OK"
    assert Q.status_string(Q.QGEMM_ERR_TIMEOUT) == "QGEMM_ERR_TIMEOUT"
    assert Q.status_string(99) == "QGEMM_UNKNOWN_STATUS"


def test_pack_rejects_missing_pointers_before_launch(Q):
    assert Q.qgemm_pack_weights(_layer(Q), None, None, None, None, 0) == \
        Q.QGEMM_ERR_INVALID_ARG
    asym = _layer(Q, weight_format=Q.QGEMM_W_UINT4_ZP, zero_format=Q.QGEMM_Z_UINT4,
                  act_dtype=Q.QGEMM_BF16, out_dtype=Q.QGEMM_BF16, scale_format=Q.QGEMM_S_BF16)
    # zero-point tensors are required for UINT4
    assert Q.qgemm_pack_weights(asym, 16, 16, None, 16, 0) == Q.QGEMM_ERR_INVALID_ARG


@pytest.mark.parametrize("name", ["qgemm_layer_config", "qgemm_compute_config",
                                  "qgemm_tuning_config"])
def test_binding_structs_match_header(Q, name):
    """The ctypes mirrors list the header's fields in the same order and widths."""
    src = open(os.path.join(ROOT, "include", "qgemm.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    body = re.search(r"typedef struct\s*\{([^}]*)\}\s*" + name + r"\s*;", src).group(1)
    fields = re.findall(r"(int32_t|int64_t)\s+(\w+)\s*;", body)
    cls = getattr(Q, name)
    got = [(f, ctypes_t) for f, ctypes_t in cls._fields_]
    assert [f for f, _ in got] == [f for _, f in fields]
    import ctypes
    width = {"int32_t": ctypes.c_int32, "int64_t": ctypes.c_int64}
    assert [t for _, t in got] == [width[t] for t, _ in fields]


def test_compute_config_rejections_before_any_device_work(Q):
    layer = _layer(Q)
    for bad in (Q.compute_config(batch_invariant=2), Q.compute_config(deterministic=3),
                Q.compute_config(gemm_type=7)):
        st, _ = Q.qgemm_workspace_size(layer, bad, None, 16)
        assert st == Q.QGEMM_ERR_INVALID_ARG, Q.last_error()


def test_checked_build_exports_the_same_symbols_and_says_so(Q):
    """The checked build (index tests in every kernel) is the same boundary:
    every declared entry point, and qgemm_checked_build tells the two apart
    (host calls only)."""
    import ctypes
    path = os.path.join(ROOT, "quantized_weight_gemm_run_b300", "libqgemm_checked.so")
    assert os.path.exists(path), "build() also builds the checked library"
    lib = ctypes.CDLL(path)
    missing = [n for n in _header_functions() if not hasattr(lib, n)]
    assert not missing, missing
    lib.qgemm_checked_build.restype = ctypes.c_int
    assert lib.qgemm_checked_build() == 1
    assert Q.qgemm_checked_build() == 0


def test_selftest_is_refused_by_the_unchecked_build(Q):
    assert Q.qgemm_checked_selftest(16, 0) == Q.QGEMM_ERR_UNSUPPORTED
