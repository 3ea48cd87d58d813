"""ctypes binding of libfp8fg.so: the C ABI of include/fp8fg.h under the same names.

Argument marshalling only. Every raw function takes device pointers as integers and
sizes exactly as the C function does; the tensor helpers in ``ops`` build those from
torch tensors. A nonzero return raises ``Fp8fgError`` with the library's message.
There is no fallback: if the library is missing, every call raises.
"""
from __future__ import annotations

import ctypes
import os

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libfp8fg.so")

FP8FG_OK = 0
FP8FG_ERR_ARG = -1
FP8FG_ERR_CUDA = -2
FP8FG_ERR_TIMEOUT = -3
FP8FG_ERR_DEVICE_ARG = -4
FP8FG_ERR_UNSUPPORTED = -5

FP8FG_OUT_F32 = 0
FP8FG_OUT_BF16 = 1
FP8FG_SB_BLOCK_128x128 = 0
FP8FG_SB_ROW_1x128 = 1

_ERR_NAMES = {
    FP8FG_ERR_ARG: "FP8FG_ERR_ARG",
    FP8FG_ERR_CUDA: "FP8FG_ERR_CUDA",
    FP8FG_ERR_TIMEOUT: "FP8FG_ERR_TIMEOUT",
    FP8FG_ERR_DEVICE_ARG: "FP8FG_ERR_DEVICE_ARG",
    FP8FG_ERR_UNSUPPORTED: "FP8FG_ERR_UNSUPPORTED",
}

# name -> (restype, argtypes), mirroring include/fp8fg.h
_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I = ctypes.c_int
SIGNATURES = {
    "fp8_quant_act_1x128": (_I, [_P, _I64, _I64, _I64, _I, _P, _P, _P]),
    "fp8_quant_act_1x128_transposed_pair": (_I, [_P, _I64, _I64, _P, _P, _P, _I64, _I64, _P, _P, _I64, _P]),
    "fp8_quant_act_delayed": (_I, [_P, _I64, _I64, _I64, _P, _I, _P, _P, _P]),
    "fp8_quant_w_128x128": (_I, [_P, _I64, _I64, _I64, _P, _P, _P]),
    "fp8_quant_act_1x128_dual": (_I, [_P, _I64, _I64, _I64, _P, _P, _P, _P, _P]),
    "fp8_quant_w_128x128_dual": (_I, [_P, _I64, _I64, _I64, _P, _P, _P, _P, _P]),
    "fp8_blockscaled_gemm": (_I, [_P, _P, _P, _P, _I, _P, _I, _I64, _I64, _I64, _P]),
    "fp8_blockscaled_gemm_ws": (_I, [_P, _P, _P, _P, _I, _P, _I, _I64, _I64, _I64, _P, _I64, _P]),
    "fp8_blockscaled_gemm_workspace_bytes": (_I64, []),
    "fp8_blockscaled_gemm_sk_static": (_I, [_P, _P, _P, _P, _I, _P, _I, _I64, _I64, _I64, _P]),
    "fp8_blockscaled_gemm_e4m3": (_I, [_P, _P, _P, _P, _I, _P, _P, _I64, _I64, _I64, _P]),
    "fp8_grouped_gemm": (_I, [_P, _P, _P, _P, _P, _I, _I64, _P, _I, _I64, _I64, _P]),
    "fp8fg_last_error": (ctypes.c_char_p, []),
    "fp8fg_sync_status": (_I, [_P]),
    "fp8fg_version": (_I, []),
    "fp8fg_selftest_wait_timeout": (_I, [_P]),
}


class Fp8fgError(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__(f"{_ERR_NAMES.get(code, code)}: {message}")
        self.code = code


_lib = None


def lib() -> ctypes.CDLL:
    """Load libfp8fg.so once; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with `python -m fp8_fine_grained_cast_b300.build`")
        handle = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


def _check(rc: int) -> int:
    if rc != FP8FG_OK:
        raise Fp8fgError(rc, fp8fg_last_error())
    return rc


def fp8fg_last_error() -> str:
    return lib().fp8fg_last_error().decode()


def fp8fg_version() -> int:
    return lib().fp8fg_version()


def fp8_quant_act_1x128(x, M, K, ldx, transposed, q, s, stream):
    return _check(lib().fp8_quant_act_1x128(x, M, K, ldx, transposed, q, s, stream))


def fp8_quant_act_1x128_transposed_pair(x0, K0, ldx0, q0, s0, x1, K1, ldx1, q1, s1, M, stream):
    return _check(lib().fp8_quant_act_1x128_transposed_pair(x0, K0, ldx0, q0, s0, x1, K1, ldx1, q1, s1, M, stream))


def fp8_quant_act_delayed(x, M, K, ldx, amax_history, H, q, s, stream):
    return _check(lib().fp8_quant_act_delayed(x, M, K, ldx, amax_history, H, q, s, stream))


def fp8_quant_w_128x128(w, N, K, ldw, q, s, stream):
    return _check(lib().fp8_quant_w_128x128(w, N, K, ldw, q, s, stream))


def fp8_quant_act_1x128_dual(x, M, K, ldx, q, s, qt, st, stream):
    return _check(lib().fp8_quant_act_1x128_dual(x, M, K, ldx, q, s, qt, st, stream))


def fp8_quant_w_128x128_dual(w, N, K, ldw, q, s, qt, st, stream):
    return _check(lib().fp8_quant_w_128x128_dual(w, N, K, ldw, q, s, qt, st, stream))


def fp8_blockscaled_gemm(qa, sa, qb, sb, sb_kind, c, c_dtype, M, N, K, stream):
    return _check(lib().fp8_blockscaled_gemm(qa, sa, qb, sb, sb_kind, c, c_dtype, M, N, K, stream))


def fp8_blockscaled_gemm_ws(qa, sa, qb, sb, sb_kind, c, c_dtype, M, N, K, workspace, workspace_bytes, stream):
    return _check(lib().fp8_blockscaled_gemm_ws(qa, sa, qb, sb, sb_kind, c, c_dtype, M, N, K, workspace,
                                                workspace_bytes, stream))


def fp8_blockscaled_gemm_sk_static(qa, sa, qb, sb, sb_kind, c, c_dtype, M, N, K, stream):
    return _check(lib().fp8_blockscaled_gemm_sk_static(qa, sa, qb, sb, sb_kind, c, c_dtype, M, N, K, stream))


def fp8_blockscaled_gemm_workspace_bytes():
    n = lib().fp8_blockscaled_gemm_workspace_bytes()
    if n < 0:
        raise Fp8fgError(int(n), fp8fg_last_error())
    return n


def fp8_blockscaled_gemm_e4m3(qa, sa, qb, sb, sb_kind, c_q, c_s, M, N, K, stream):
    return _check(lib().fp8_blockscaled_gemm_e4m3(qa, sa, qb, sb, sb_kind, c_q, c_s, M, N, K, stream))


def fp8_grouped_gemm(qa, sa, qb, sb, group_offsets, E, Mtot, c, c_dtype, N, K, stream):
    return _check(lib().fp8_grouped_gemm(qa, sa, qb, sb, group_offsets, E, Mtot, c, c_dtype, N, K, stream))


def fp8fg_selftest_wait_timeout(stream):
    return _check(lib().fp8fg_selftest_wait_timeout(stream))


def fp8fg_sync_status(stream):
    return _check(lib().fp8fg_sync_status(stream))
