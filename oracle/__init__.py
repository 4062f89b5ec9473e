"""CPU oracle for the weight-only 4-bit matmul library -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py``
may import this package.  The product path (``weight_only_bit_int4_gb300``) never
imports, links or calls it, and this package never imports the product.

The arithmetic lives in ``q4_oracle.c`` (plain C, fp64 accumulation, compiled with
``-ffp-contract=off``); this module is a numpy/ctypes shim around it.  Each wrapper
names the page and section whose definition the C function writes out.

Parity status of every function is listed in the module-level ``PINS`` table; the
pins themselves are the ``-m "not gpu"`` tests in ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "q4_oracle.c")
_LIB = os.path.join(_HERE, "liboracle_q4.so")

# Compiler flags shared with __graft_entry__.build(): no contraction, no fast-math.
CFLAGS = ["-O2", "-std=c99", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]

PINS = {
    "f32_to_bf16 / f32_to_f16 / f16_to_f32": "pinned: numpy float16 casts, nearest-neighbour brute force, special values",
    "q4_dequant": "pinned: hand-built words, single-nibble case, quantizer round trip, fp64 exactness",
    "q4_matmul": "pinned: hand-built 2x64x8 closed form, all-zero-nibble closed form, single-nibble case",
    "lut4_dequant / lut4_matmul": "pinned: the lut4.rs CPU test's worked example (both transposes, exact)",
    "lut4_matmul_rounded": "pinned: identity when every decoded value is already representable, f16 "
                           "underflow to exact zero and overflow to infinity, one-hot x equals the numpy "
                           "cast of the decoded matrix",
    "q4_0_matmul_id": "pinned: hand-built block, q=8 zero case, one-hot x, top_k=1 dense reduction, id permutation",
    "q4_0_route": "pinned: hand-written lists and brute-force invariants",
    "q4_0_matmul_id_swiglu": "pinned: sigmoid(+-ln 3) closed form, zero gate/up, odd part = plain routed "
                             "matmul, even part = z tanh(z/2) via numpy, per-row independence",
}


def build(force: bool = False) -> str:
    """Compile ``q4_oracle.c`` into ``liboracle_q4.so`` beside it (idempotent)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def lib() -> ctypes.CDLL:
    """The compiled oracle.  Q4MM_ORACLE_LIB names another build of q4_oracle.c to load
    instead (the mutation tests load copies with a planted mistake this way)."""
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(os.environ.get("Q4MM_ORACLE_LIB") or build())
        _declare(_lib)
    return _lib


_P = ctypes.c_void_p
_I = ctypes.c_int64


def _declare(L: ctypes.CDLL) -> None:
    sig = {
        "oracle_bf16_to_f32": ([ctypes.c_uint16], ctypes.c_float),
        "oracle_f32_to_bf16": ([ctypes.c_float], ctypes.c_uint16),
        "oracle_f16_to_f32": ([ctypes.c_uint16], ctypes.c_float),
        "oracle_f32_to_f16": ([ctypes.c_float], ctypes.c_uint16),
        "oracle_f32_to_bf16_n": ([_P, _P, _I], None),
        "oracle_f32_to_f16_n": ([_P, _P, _I], None),
        "oracle_f16_to_f32_n": ([_P, _P, _I], None),
        "oracle_q4_dequant": ([_P, _P, _P, _I, _I, _P], None),
        "oracle_q4_dequant_inexact": ([_P, _P, _P, _I, _I], _I),
        "oracle_q4_matmul": ([_P, _P, _P, _P, _I, _I, _I, _P], None),
        "oracle_q4_matmul_at": ([_P, _P, _P, _P, _I, _P, _P, _I, _P], None),
        "oracle_q4_quantize": ([_P, _I, _I, _P, _P, _P, _P], None),
        "oracle_lut4_dequant": ([_P, _P, _P, _I, _I, _I, _P], None),
        "oracle_lut4_matmul": ([_P, _P, _P, _P, _I, _I, _I, _I, ctypes.c_int, _P], None),
        "oracle_lut4_matmul_at": ([_P, _P, _P, _P, _I, _I, _I, ctypes.c_int, _P, _P, _I, _P], None),
        "oracle_lut4_matmul_rounded": ([_P, _P, _P, _P, _I, _I, _I, _I, ctypes.c_int, ctypes.c_int, _P], None),
        "oracle_lut4_matmul_rounded_at": ([_P, _P, _P, _P, _I, _I, _I, ctypes.c_int, ctypes.c_int, _P, _P, _I,
                                           _P], None),
        "oracle_q4_0_dequant_row": ([_P, _I, _P], None),
        "oracle_q4_0_matmul_id": ([_P, _P, _P, _I, _I, _I, _I, _I, ctypes.c_uint64, _P], None),
        "oracle_q4_0_matmul_id_rows": ([_P, _P, _P, _I, _I, _I, _I, ctypes.c_uint64, _P, _I, _P], None),
        "oracle_q8_0_dequant_row": ([_P, _I, _P], None),
        "oracle_q8_0_matmul_id": ([_P, _P, _P, _I, _I, _I, _I, _I, ctypes.c_uint64, _P], None),
        "oracle_q8_0_matmul_id_rows": ([_P, _P, _P, _I, _I, _I, _I, ctypes.c_uint64, _P, _I, _P], None),
        "oracle_q4_0_route": ([_P, _I, _I, _P, _P, _P], None),
        "oracle_q4_0_matmul_id_swiglu": ([_P, _P, _P, _P, _I, _I, _I, _I, ctypes.c_uint64, _P], None),
        "oracle_q4_0_matmul_id_swiglu_rows": ([_P, _P, _P, _P, _I, _I, _I, ctypes.c_uint64, _P, _I, _P],
                                              None),
    }
    for name, (args, res) in sig.items():
        f = getattr(L, name)
        f.argtypes = args
        f.restype = res


def _c(a: np.ndarray, dtype) -> np.ndarray:
    a = np.ascontiguousarray(a, dtype=dtype)
    return a


def _p(a: np.ndarray) -> int:
    return a.ctypes.data


# --- storage conversions -----------------------------------------------------------------

def f32_to_bf16(a) -> np.ndarray:
    """Nearest bfloat16 (ties to even) of each fp32 value, as uint16 bits."""
    a = _c(a, np.float32)
    out = np.empty(a.shape, np.uint16)
    lib().oracle_f32_to_bf16_n(_p(a), _p(out), a.size)
    return out


def f32_to_f16(a) -> np.ndarray:
    """Nearest IEEE binary16 (ties to even) of each fp32 value, as uint16 bits."""
    a = _c(a, np.float32)
    out = np.empty(a.shape, np.uint16)
    lib().oracle_f32_to_f16_n(_p(a), _p(out), a.size)
    return out


def f16_to_f32(a) -> np.ndarray:
    a = _c(a, np.uint16)
    out = np.empty(a.shape, np.float32)
    lib().oracle_f16_to_f32_n(_p(a), _p(out), a.size)
    return out


def bf16_to_f32(a) -> np.ndarray:
    """bfloat16 bits -> fp32 (the bf16 value is the top half of the binary32)."""
    a = _c(a, np.uint16)
    return (a.astype(np.uint32) << 16).view(np.float32)


# --- INT4 group-32 affine (quant_fastkernel.rs) -----------------------------------------

def q4_dequant(w, scales, biases, N: int, K: int) -> np.ndarray:
    """fp32 [N, K]: fmaf(nibble, scale, bias), low nibble first (quant_fastkernel.rs,
    kernel W-tile dequant and the test module's host ground truth)."""
    w, s, b = _c(w, np.uint32), _c(scales, np.uint16), _c(biases, np.uint16)
    out = np.empty((N, K), np.float32)
    lib().oracle_q4_dequant(_p(w), _p(s), _p(b), N, K, _p(out))
    return out


def q4_dequant_inexact(w, scales, biases, N: int, K: int) -> int:
    w, s, b = _c(w, np.uint32), _c(scales, np.uint16), _c(biases, np.uint16)
    return int(lib().oracle_q4_dequant_inexact(_p(w), _p(s), _p(b), N, K))


def q4_matmul(x, w, scales, biases, M: int, N: int, K: int) -> np.ndarray:
    """fp64 [M, N]: sum_k x[m][k] * dequant(W)[n][k], k ascending."""
    x, w, s, b = _c(x, np.uint16), _c(w, np.uint32), _c(scales, np.uint16), _c(biases, np.uint16)
    y = np.empty((M, N), np.float64)
    lib().oracle_q4_matmul(_p(x), _p(w), _p(s), _p(b), M, N, K, _p(y))
    return y


def q4_matmul_at(x, w, scales, biases, K: int, mi, ni) -> np.ndarray:
    x, w, s, b = _c(x, np.uint16), _c(w, np.uint32), _c(scales, np.uint16), _c(biases, np.uint16)
    mi, ni = _c(mi, np.int64), _c(ni, np.int64)
    out = np.empty(mi.shape, np.float64)
    lib().oracle_q4_matmul_at(_p(x), _p(w), _p(s), _p(b), K, _p(mi), _p(ni), mi.size, _p(out))
    return out


def q4_quantize(wf, N: int, K: int):
    """Reference affine quantizer (pins only): returns (words, scales, biases, zp)."""
    wf = _c(wf, np.float32)
    words = np.zeros((N, K // 8), np.uint32)
    s = np.zeros((N, K // 32), np.uint16)
    b = np.zeros((N, K // 32), np.uint16)
    zp = np.zeros((N, K // 32), np.uint8)
    lib().oracle_q4_quantize(_p(wf), N, K, _p(words), _p(s), _p(b), _p(zp))
    return words, s, b, zp


# --- LUT4 (lut4.rs) ------------------------------------------------------------------------

def lut4_dequant(packed, scales, book, rows: int, cols: int, block: int) -> np.ndarray:
    """fp32 [rows, cols]: fl32(book[code] * scales[f / block]), high nibble for even f
    (lut4.rs, the CPU branch of `execute`)."""
    p, s, bk = _c(packed, np.uint8), _c(scales, np.float32), _c(book, np.float32)
    out = np.empty((rows, cols), np.float32)
    lib().oracle_lut4_dequant(_p(p), _p(s), _p(bk), rows, cols, block, _p(out))
    return out


def lut4_matmul(x, packed, scales, book, M: int, N: int, K: int, block: int, transpose: int) -> np.ndarray:
    x, p, s, bk = _c(x, np.uint16), _c(packed, np.uint8), _c(scales, np.float32), _c(book, np.float32)
    y = np.empty((M, N), np.float64)
    lib().oracle_lut4_matmul(_p(x), _p(p), _p(s), _p(bk), M, N, K, block, int(transpose), _p(y))
    return y


def lut4_matmul_at(x, packed, scales, book, N: int, K: int, block: int, transpose: int, mi, ni) -> np.ndarray:
    x, p, s, bk = _c(x, np.uint16), _c(packed, np.uint8), _c(scales, np.float32), _c(book, np.float32)
    mi, ni = _c(mi, np.int64), _c(ni, np.int64)
    out = np.empty(mi.shape, np.float64)
    lib().oracle_lut4_matmul_at(_p(x), _p(p), _p(s), _p(bk), N, K, block, int(transpose),
                                _p(mi), _p(ni), mi.size, _p(out))
    return out


_ROUNDING = {None: 0, "f16": 1, "bf16": 2}


def lut4_matmul_rounded(x, packed, scales, book, M: int, N: int, K: int, block: int, transpose: int,
                        rounding) -> np.ndarray:
    """lut4_matmul with the decoded weight rounded to ``rounding`` ("f16" or "bf16", nearest
    even) and widened back before the product (lut4.rs, `rounded_weight`)."""
    x, p, s, bk = _c(x, np.uint16), _c(packed, np.uint8), _c(scales, np.float32), _c(book, np.float32)
    y = np.empty((M, N), np.float64)
    lib().oracle_lut4_matmul_rounded(_p(x), _p(p), _p(s), _p(bk), M, N, K, block, int(transpose),
                                     _ROUNDING[rounding], _p(y))
    return y


def lut4_matmul_rounded_at(x, packed, scales, book, N: int, K: int, block: int, transpose: int, rounding,
                           mi, ni) -> np.ndarray:
    x, p, s, bk = _c(x, np.uint16), _c(packed, np.uint8), _c(scales, np.float32), _c(book, np.float32)
    mi, ni = _c(mi, np.int64), _c(ni, np.int64)
    out = np.empty(mi.shape, np.float64)
    lib().oracle_lut4_matmul_rounded_at(_p(x), _p(p), _p(s), _p(bk), N, K, block, int(transpose),
                                        _ROUNDING[rounding], _p(mi), _p(ni), mi.size, _p(out))
    return out


# --- GGML Q4_0 expert-routed (quantized_matmul_id_ggml.rs) ---------------------------------

def q4_0_dequant_row(row_bytes, K: int) -> np.ndarray:
    r = _c(row_bytes, np.uint8)
    out = np.empty(K, np.float32)
    lib().oracle_q4_0_dequant_row(_p(r), K, _p(out))
    return out


def q4_0_matmul_id(x, w, ids, n_tokens: int, top_k: int, N: int, K: int, n_experts: int,
                   expert_stride: int) -> np.ndarray:
    """fp64 [n_tokens*top_k, N]: out[r] = x[r / top_k] . dequant(W[ids[r]])^T."""
    x, w, ids = _c(x, np.float32), _c(w, np.uint8), _c(ids, np.uint32)
    out = np.empty((n_tokens * top_k, N), np.float64)
    lib().oracle_q4_0_matmul_id(_p(x), _p(w), _p(ids), n_tokens, top_k, N, K, n_experts,
                                expert_stride, _p(out))
    return out


def q4_0_matmul_id_rows(x, w, ids, top_k: int, N: int, K: int, n_experts: int,
                        expert_stride: int, rows) -> np.ndarray:
    x, w, ids = _c(x, np.float32), _c(w, np.uint8), _c(ids, np.uint32)
    rows = _c(rows, np.int64)
    out = np.empty((rows.size, N), np.float64)
    lib().oracle_q4_0_matmul_id_rows(_p(x), _p(w), _p(ids), top_k, N, K, n_experts,
                                     expert_stride, _p(rows), rows.size, _p(out))
    return out


def q8_0_dequant_row(row_bytes, K: int) -> np.ndarray:
    r = _c(row_bytes, np.uint8)
    out = np.empty(K, np.float32)
    lib().oracle_q8_0_dequant_row(_p(r), K, _p(out))
    return out


def q8_0_matmul_id(x, w, ids, n_tokens: int, top_k: int, N: int, K: int, n_experts: int,
                   expert_stride: int) -> np.ndarray:
    """fp64 [n_tokens*top_k, N]: out[r] = x[r / top_k] . dequant(W[ids[r]])^T, Q8_0 blocks."""
    x, w, ids = _c(x, np.float32), _c(w, np.uint8), _c(ids, np.uint32)
    out = np.empty((n_tokens * top_k, N), np.float64)
    lib().oracle_q8_0_matmul_id(_p(x), _p(w), _p(ids), n_tokens, top_k, N, K, n_experts,
                                expert_stride, _p(out))
    return out


def q8_0_matmul_id_rows(x, w, ids, top_k: int, N: int, K: int, n_experts: int,
                        expert_stride: int, rows) -> np.ndarray:
    x, w, ids = _c(x, np.float32), _c(w, np.uint8), _c(ids, np.uint32)
    rows = _c(rows, np.int64)
    out = np.empty((rows.size, N), np.float64)
    lib().oracle_q8_0_matmul_id_rows(_p(x), _p(w), _p(ids), top_k, N, K, n_experts,
                                     expert_stride, _p(rows), rows.size, _p(out))
    return out


def q4_0_matmul_id_swiglu(gate, up, w, ids, N: int, K: int, n_experts: int,
                          expert_stride: int) -> np.ndarray:
    """fp64 [n_rows, N]: out[r] = (silu(gate[r]) * up[r]) . dequant(W[ids[r]])^T; gate and up
    are [n_rows, K] f32, one row per routed row."""
    gate, up, w, ids = _c(gate, np.float32), _c(up, np.float32), _c(w, np.uint8), _c(ids, np.uint32)
    n_rows = ids.size
    assert gate.size == n_rows * K and up.size == n_rows * K
    out = np.empty((n_rows, N), np.float64)
    lib().oracle_q4_0_matmul_id_swiglu(_p(gate), _p(up), _p(w), _p(ids), n_rows, N, K, n_experts,
                                       expert_stride, _p(out))
    return out


def q4_0_matmul_id_swiglu_rows(gate, up, w, ids, N: int, K: int, n_experts: int,
                               expert_stride: int, rows) -> np.ndarray:
    gate, up, w, ids = _c(gate, np.float32), _c(up, np.float32), _c(w, np.uint8), _c(ids, np.uint32)
    rows = _c(rows, np.int64)
    out = np.empty((rows.size, N), np.float64)
    lib().oracle_q4_0_matmul_id_swiglu_rows(_p(gate), _p(up), _p(w), _p(ids), N, K, n_experts,
                                            expert_stride, _p(rows), rows.size, _p(out))
    return out


def q4_0_route(ids, n_experts: int):
    """(htpe [n_experts] u32, hids [n_valid] i32, n_invalid): per-expert ascending lists."""
    ids = _c(ids, np.uint32)
    htpe = np.zeros(n_experts, np.uint32)
    hids = np.full(ids.size, -1, np.int32)
    bad = np.zeros(1, np.uint32)
    lib().oracle_q4_0_route(_p(ids), ids.size, n_experts, _p(htpe), _p(hids), _p(bad))
    nvalid = int(htpe.sum())
    return htpe, hids[:nvalid].copy(), int(bad[0])


# --- tolerance --------------------------------------------------------------------------

def matmul_tolerance(y_ref: np.ndarray) -> np.ndarray:
    """Per-element bound for a float matmul output: 2^-8 |y_ref| + 1e-2 rms(y_ref)."""
    y_ref = np.asarray(y_ref, np.float64)
    rms = float(np.sqrt(np.mean(y_ref * y_ref))) if y_ref.size else 0.0
    return np.abs(y_ref) * 2.0 ** -8 + 1e-2 * rms
