"""ctypes declarations of libq4mm's C ABI (include/q4mm.h).  Loads the in-tree library and
fails loudly if it is missing: there is no other implementation to fall back to."""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libq4mm.so")

_P = ctypes.c_void_p
_I = ctypes.c_int64
_S = ctypes.c_int

SIGNATURES = {
    "q4mm_status_string": ([_S], ctypes.c_char_p),
    "q4mm_version": ([], _S),
    "q4mm_device_errors": ([_P, _S], _S),
    "q4mm_selftest_wait_timeout": ([_P, ctypes.c_uint32, _P], _S),
    "q4_dequant": ([_P, _P, _P, _I, _I, _P, _S, _P], _S),
    "q4_gemv": ([_P, _P, _P, _P, _P, _I, _I, _I, _P], _S),
    "q4_gemv_ex": ([_P, _P, _P, _P, _P, _I, _I, _I, ctypes.c_uint32, _P], _S),
    "q4_gemm": ([_P, _P, _P, _P, _P, _I, _I, _I, _P], _S),
    "lut4_matmul": ([_P, _P, _P, _P, _P, _I, _I, _I, _I, _S, _P], _S),
    "lut4_matmul_ex": ([_P, _P, _P, _P, _P, _I, _I, _I, _I, _S, ctypes.c_uint32, _P], _S),
    "lut4_dequant": ([_P, _P, _P, _I, _I, _I, _P, _S, _P], _S),
    "q4_0_route": ([_P, _I, _I, _P, _P, _P, _P], _S),
    "q4_0_matmul_id_workspace_size": ([_I, _I, _I, _I, _I], ctypes.c_size_t),
    "q4_0_matmul_id": ([_P, _P, _P, _P, _I, _I, _I, _I, _I, ctypes.c_uint64, _S, _P,
                        ctypes.c_size_t, _P], _S),
    "q4_0_matmul_id_swiglu": ([_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, ctypes.c_uint64, _P], _S),
    "q8_0_matmul_id_workspace_size": ([_I, _I, _I, _I, _I], ctypes.c_size_t),
    "q8_0_matmul_id": ([_P, _P, _P, _P, _I, _I, _I, _I, _I, ctypes.c_uint64, _S, _P, ctypes.c_size_t, _P], _S),
    "q4_gemv_record": ([_I, _I, _I, ctypes.c_uint32, ctypes.POINTER(_P)], _S),
    "q4_gemv_record_launch": ([_P, _P, _P, _P, _P, _P, _P], _S),
    "q4_gemv_record_launch_n": ([ctypes.POINTER(_P)] * 6 + [_I, _P], _S),
    "q4_0_matmul_id_mv_record": ([_I, _I, _I, _I, _I, ctypes.c_uint64, _S, ctypes.POINTER(_P)], _S),
    "q4_0_matmul_id_mv_record_launch": ([_P, _P, _P, _P, _P, _P, _P], _S),
    "q4mm_record_free": ([_P], None),
    "q4_0_matmul_id_noalloc": ([_P, _P, _P, _P, _I, _I, _I, _I, _I, ctypes.c_uint64, _P], _S),
}

_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"libq4mm.so not found at {LIB_PATH}; build it with "
                "`python -m weight_only_bit_int4_gb300.build` (or __graft_entry__.build())")
        L = ctypes.CDLL(LIB_PATH)
        for name, (args, res) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = res
        _lib = L
    return _lib
