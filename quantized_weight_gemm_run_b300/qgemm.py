"""Python binding of the C ABI in ``include/qgemm.h`` (ctypes).

Argument marshalling only: every function here has the name of its C entry
point, converts torch tensors (or raw integer addresses) to pointers and the
current torch CUDA stream to a ``cudaStream_t``, and returns the C status code.
All computation happens in the CUDA library; if ``libqgemm.so`` is missing the
import fails loudly (build it with ``python -m quantized_weight_gemm_run_b300.build``).
"""

from __future__ import annotations

import ctypes
import os

# QGEMM_LIBRARY=checked selects the checked build (index tests in every
# kernel; see include/qgemm.h)
_LIB_NAME = "libqgemm_checked.so" if os.environ.get("QGEMM_LIBRARY") == "checked" else "libqgemm.so"
_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), _LIB_NAME)

# status codes
QGEMM_OK = 0
QGEMM_ERR_INVALID_ARG = 1
QGEMM_ERR_UNSUPPORTED = 2
QGEMM_ERR_WORKSPACE = 3
QGEMM_ERR_CUDA = 4
QGEMM_ERR_TIMEOUT = 5
QGEMM_ERR_DEVICE = 6
# weight / scale / zero formats, dtypes, GEMM types
QGEMM_W_INT4_SYM, QGEMM_W_UINT4_ZP, QGEMM_W_MXFP4, QGEMM_W_NVFP4 = 0, 1, 2, 3
QGEMM_W_INT8_SYM, QGEMM_W_UINT8_ZP = 4, 5
QGEMM_W_INT3_SYM, QGEMM_W_UINT3_ZP = 6, 7
QGEMM_S_FP16, QGEMM_S_BF16, QGEMM_S_E8M0, QGEMM_S_E4M3 = 0, 1, 2, 3
QGEMM_Z_NONE, QGEMM_Z_UINT4, QGEMM_Z_UINT8, QGEMM_Z_UINT3 = 0, 1, 2, 3
QGEMM_FP16, QGEMM_BF16, QGEMM_FP8E4M3, QGEMM_NVFP4 = 0, 1, 2, 3
QGEMM_GEMM_DENSE, QGEMM_GEMM_GROUPED = 0, 1
QGEMM_ACT_NONE, QGEMM_ACT_SILU_GLU = 0, 1


class qgemm_layer_config(ctypes.Structure):
    _fields_ = [("n", ctypes.c_int64), ("k", ctypes.c_int64), ("group_size", ctypes.c_int32),
                ("weight_format", ctypes.c_int32), ("scale_format", ctypes.c_int32),
                ("zero_format", ctypes.c_int32), ("act_dtype", ctypes.c_int32),
                ("out_dtype", ctypes.c_int32), ("has_bias", ctypes.c_int32),
                ("num_experts", ctypes.c_int32), ("gated_act", ctypes.c_int32)]


class qgemm_compute_config(ctypes.Structure):
    _fields_ = [("gemm_type", ctypes.c_int32), ("batch_invariant", ctypes.c_int32),
                ("deterministic", ctypes.c_int32)]


class qgemm_tuning_config(ctypes.Structure):
    _fields_ = [("block_tok", ctypes.c_int32), ("stages", ctypes.c_int32),
                ("max_ctas", ctypes.c_int32), ("split_k", ctypes.c_int32),
                ("cta_pair", ctypes.c_int32), ("kernel", ctypes.c_int32)]


class QGemmError(RuntimeError):
    def __init__(self, status, message=""):
        super().__init__(f"{status_string(status)}: {message}")
        self.status = status


def _load():
    if not os.path.exists(_LIB_PATH):
        raise ImportError(f"{_LIB_PATH} is missing: build it with "
                          "`python -m quantized_weight_gemm_run_b300.build`"
                          + (" --checked" if _LIB_NAME != "libqgemm.so" else ""))
    return ctypes.CDLL(_LIB_PATH)


lib = _load()

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I32 = ctypes.c_int32
_SZ = ctypes.c_size_t
_L = ctypes.POINTER(qgemm_layer_config)
_C = ctypes.POINTER(qgemm_compute_config)
_T = ctypes.POINTER(qgemm_tuning_config)

_SIGS = {
    "qgemm_packed_size": [_L, ctypes.POINTER(_SZ)],
    "qgemm_pack_weights": [_L, _P, _P, _P, _P, _P],
    "qgemm_workspace_size": [_L, _C, _T, _I64, ctypes.POINTER(_SZ)],
    "qgemm_workspace_init": [_P, _SZ, _P],
    "qgemm_run": [_L, _C, _T, _I64, _P, _P, _P, _P, _P, _P, _SZ, _P],
    "qgemm_run_noalloc": [_L, _C, _T, _I64, _P, _P, _P, _P, _P, _P],
    "qgemm_grouped_run": [_L, _C, _T, _P, _I64, _P, _P, _P, _P, _P, _P, _SZ, _P],
    "qgemm_quantize_act_fp8": [_P, _I64, _I64, _P, _P, _P],
    "qgemm_quantize_act_nvfp4": [_P, _I64, _I64, _P, _P, _P, _P],
    "qgemm_moe_permute": [_P, _I64, _I32, _I32, _P, _P, _P, _P, _P, _I64, _P],
    "qgemm_moe_silu_mul": [_P, _I64, _I64, _P, _P],
    "qgemm_moe_combine": [_P, _P, _P, _I64, _I32, _I64, _P, _P],
    "qgemm_debug_dequant": [_L, _P, _P, _P],
    "qgemm_check_status": [_P, _P],
    "qgemm_noalloc_check_status": [_P],
    "qgemm_checked_status": [_P],
    "qgemm_checked_selftest": [_P, _P],
    "qgemm_describe_plan": [_L, _C, _I64, ctypes.c_char_p, _SZ],
}
for _name, _args in _SIGS.items():
    _f = getattr(lib, _name)
    _f.argtypes = _args
    _f.restype = ctypes.c_int
lib.qgemm_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
lib.qgemm_set_wait_limit_ns.restype = None
lib.qgemm_status_string.argtypes = [ctypes.c_int]
lib.qgemm_status_string.restype = ctypes.c_char_p
lib.qgemm_last_error.argtypes = []
lib.qgemm_last_error.restype = ctypes.c_char_p
lib.qgemm_checked_build.argtypes = []
lib.qgemm_checked_build.restype = ctypes.c_int


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _ref(x):
    return None if x is None else ctypes.byref(x)


def status_string(status: int) -> str:
    return lib.qgemm_status_string(status).decode()


def last_error() -> str:
    return lib.qgemm_last_error().decode()


def check(status: int) -> None:
    """Raise QGemmError unless status is QGEMM_OK."""
    if status != QGEMM_OK:
        raise QGemmError(status, last_error())


def layer_config(n, k, group_size, weight_format, scale_format, zero_format, act_dtype,
                 out_dtype, has_bias=0, num_experts=1, gated_act=0) -> qgemm_layer_config:
    return qgemm_layer_config(n, k, group_size, weight_format, scale_format, zero_format,
                              act_dtype, out_dtype, has_bias, num_experts, gated_act)


def compute_config(gemm_type=QGEMM_GEMM_DENSE, batch_invariant=0,
                   deterministic=0) -> qgemm_compute_config:
    return qgemm_compute_config(gemm_type, batch_invariant, deterministic)


def tuning_config(block_tok=0, stages=0, max_ctas=0, split_k=0, cta_pair=0, kernel=0):
    return qgemm_tuning_config(block_tok, stages, max_ctas, split_k, cta_pair, kernel)


# ------------------------------------------------------------- entry points

def qgemm_packed_size(layer):
    b = _SZ()
    st = lib.qgemm_packed_size(ctypes.byref(layer), ctypes.byref(b))
    return st, b.value


def qgemm_pack_weights(layer, qweight, scales, qzeros, packed, stream=None):
    return lib.qgemm_pack_weights(ctypes.byref(layer), _ptr(qweight), _ptr(scales), _ptr(qzeros),
                                  _ptr(packed), _stream(stream))


def qgemm_workspace_size(layer, compute, tuning, m):
    b = _SZ()
    st = lib.qgemm_workspace_size(ctypes.byref(layer), ctypes.byref(compute), _ref(tuning), m,
                                  ctypes.byref(b))
    return st, b.value


def qgemm_workspace_init(workspace, nbytes, stream=None):
    return lib.qgemm_workspace_init(_ptr(workspace), nbytes, _stream(stream))


def qgemm_run(layer, compute, tuning, m, a, a_scale, packed, bias, c, workspace,
              workspace_bytes, stream=None):
    return lib.qgemm_run(ctypes.byref(layer), ctypes.byref(compute), _ref(tuning), m, _ptr(a),
                         _ptr(a_scale), _ptr(packed), _ptr(bias), _ptr(c), _ptr(workspace),
                         workspace_bytes, _stream(stream))


def qgemm_run_noalloc(layer, compute, tuning, m, a, a_scale, packed, bias, c, stream=None):
    return lib.qgemm_run_noalloc(ctypes.byref(layer), ctypes.byref(compute), _ref(tuning), m,
                                 _ptr(a), _ptr(a_scale), _ptr(packed), _ptr(bias), _ptr(c),
                                 _stream(stream))


def qgemm_grouped_run(layer, compute, tuning, expert_offsets, total_rows, a, a_scale, packed,
                      bias, c, workspace, workspace_bytes, stream=None):
    return lib.qgemm_grouped_run(ctypes.byref(layer), ctypes.byref(compute), _ref(tuning),
                                 _ptr(expert_offsets), total_rows, _ptr(a), _ptr(a_scale),
                                 _ptr(packed), _ptr(bias), _ptr(c), _ptr(workspace),
                                 workspace_bytes, _stream(stream))


def qgemm_quantize_act_fp8(x, m, k, a8, a_scale, stream=None):
    return lib.qgemm_quantize_act_fp8(_ptr(x), m, k, _ptr(a8), _ptr(a_scale), _stream(stream))


def qgemm_quantize_act_nvfp4(x, m, k, a_ts, codes, block_scales, stream=None):
    return lib.qgemm_quantize_act_nvfp4(_ptr(x), m, k, _ptr(a_ts), _ptr(codes),
                                        _ptr(block_scales), _stream(stream))


def qgemm_moe_permute(topk_ids, t, topk, e, offsets, perm, inv_perm, a, a_perm, hidden,
                      stream=None):
    return lib.qgemm_moe_permute(_ptr(topk_ids), t, topk, e, _ptr(offsets), _ptr(perm),
                                 _ptr(inv_perm), _ptr(a), _ptr(a_perm), hidden, _stream(stream))


def qgemm_moe_silu_mul(gu, rows, inter, h, stream=None):
    return lib.qgemm_moe_silu_mul(_ptr(gu), rows, inter, _ptr(h), _stream(stream))


def qgemm_moe_combine(y2, inv_perm, topk_weights, t, topk, hidden, y, stream=None):
    return lib.qgemm_moe_combine(_ptr(y2), _ptr(inv_perm), _ptr(topk_weights), t, topk, hidden,
                                 _ptr(y), _stream(stream))


def qgemm_debug_dequant(layer, packed, out_kn, stream=None):
    return lib.qgemm_debug_dequant(ctypes.byref(layer), _ptr(packed), _ptr(out_kn),
                                   _stream(stream))


def qgemm_check_status(workspace, stream=None):
    return lib.qgemm_check_status(_ptr(workspace), _stream(stream))


def qgemm_noalloc_check_status(stream=None):
    return lib.qgemm_noalloc_check_status(_stream(stream))


def qgemm_checked_build() -> int:
    return lib.qgemm_checked_build()


def qgemm_checked_status(stream=None):
    return lib.qgemm_checked_status(_stream(stream))


def qgemm_checked_selftest(workspace, stream=None):
    return lib.qgemm_checked_selftest(_ptr(workspace), _stream(stream))


def qgemm_set_wait_limit_ns(ns: int) -> None:
    lib.qgemm_set_wait_limit_ns(ns)


def qgemm_describe_plan(layer, compute, m):
    buf = ctypes.create_string_buffer(1024)
    st = lib.qgemm_describe_plan(ctypes.byref(layer), ctypes.byref(compute), m, buf, 1024)
    return st, buf.value.decode()


def qgemm_status_string(status: int) -> str:
    return status_string(status)


def qgemm_last_error() -> str:
    return last_error()
