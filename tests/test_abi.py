"""CPU-side checks of the C ABI: the library loads, exports every function include/q4mm.h
declares, and rejects bad arguments on the host before touching the GPU."""
import ctypes
import os
import re

import pytest

from weight_only_bit_int4_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "q4mm.h")


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b([a-z_0-9]+)\s*\([^;{]*\)\s*;", text)))


@pytest.fixture(scope="module")
def L():
    return _lib.lib()


def test_header_declares_the_hot_path():
    names = _declared_functions()
    for n in ["q4_dequant", "q4_gemv", "q4_gemm", "lut4_matmul", "lut4_dequant", "q4_0_route",
              "q4_0_matmul_id", "q4_0_matmul_id_workspace_size", "q4_0_matmul_id_swiglu",
              "q4mm_status_string"]:
        assert n in names


def test_every_declared_symbol_is_exported(L):
    for name in _declared_functions():
        assert hasattr(L, name), name
    assert set(_declared_functions()) <= set(_lib.SIGNATURES)


def test_status_strings(L):
    assert L.q4mm_status_string(0) == b"ok"
    assert L.q4mm_status_string(3).startswith(b"workspace")
    assert L.q4mm_version() >= 100


FAKE = 1 << 20   # an aligned non-null address; never dereferenced: the checks fail first


def test_int4_argument_checks(L):
    # null pointers, K not a multiple of 32, M out of range -> INVALID_ARG, nothing launched
    assert L.q4_gemv(None, FAKE, FAKE, FAKE, FAKE, 1, 64, 64, None) == 1
    assert L.q4_gemv(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 64, 48, None) == 1
    assert L.q4_gemv(FAKE, FAKE, FAKE, FAKE, FAKE, 17, 64, 64, None) == 1
    assert L.q4_gemm(FAKE, FAKE, FAKE, FAKE, FAKE, -1, 64, 64, None) == 1
    assert L.q4_dequant(FAKE, FAKE, FAKE, 4, 64, FAKE, 7, None) == 1
    # misaligned operand -> UNSUPPORTED
    assert L.q4_gemv(FAKE + 2, FAKE, FAKE, FAKE, FAKE, 1, 64, 64, None) == 2
    # zero tokens -> OK with nothing enqueued
    assert L.q4_gemv(None, None, None, None, None, 0, 64, 64, None) == 0
    # unknown launch flag bits -> INVALID_ARG (checked first); the known flag passes the check
    assert L.q4_gemv_ex(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 64, 64, 0x2, None) == 1
    assert L.q4_gemv_ex(None, None, None, None, None, 0, 64, 64, 0x1, None) == 0
    assert L.q4_gemm(None, None, None, None, None, 0, 64, 64, None) == 0


def test_lut4_argument_checks(L):
    book = (ctypes.c_float * 16)()
    assert L.lut4_matmul(FAKE, FAKE, FAKE, book, FAKE, 1, 4, 4, 3, 1, None) == 1      # odd block
    assert L.lut4_matmul(FAKE, FAKE, FAKE, None, FAKE, 1, 4, 4, 4, 1, None) == 1      # no book
    assert L.lut4_matmul(FAKE, FAKE, FAKE, book, FAKE, 1, 4, 4, 4, 2, None) == 1      # bad transpose flag
    assert L.lut4_matmul_ex(FAKE, FAKE, FAKE, book, FAKE, 1, 4, 4, 4, 1, 0x8, None) == 1  # unknown flag bit
    assert L.lut4_matmul_ex(FAKE, FAKE, FAKE, book, FAKE, 1, 4, 4, 4, 1, 0x6, None) == 1  # both roundings
    assert L.lut4_matmul_ex(None, None, None, None, None, 0, 4, 4, 4, 1, 0x6, None) == 1  # even at M = 0
    assert L.lut4_matmul_ex(None, None, None, None, None, 0, 4, 4, 4, 1, 0x3, None) == 0  # M = 0, valid flags
    assert L.lut4_matmul_ex(FAKE, FAKE, FAKE, book, FAKE, 1, 4, 4, 3, 1, 0x2, None) == 1  # odd block
    assert L.lut4_matmul_ex(None, None, None, None, None, 0, 4, 4, 4, 1, 0x1, None) == 0  # M = 0


def test_moe_argument_checks(L):
    # expert_stride smaller than one expert -> INVALID_ARG
    assert L.q4_0_matmul_id(FAKE, FAKE, FAKE, FAKE, 2, 8, 64, 64, 16, 64 * 2 * 18 - 1, 1, None, 0, None) == 1
    # K not a multiple of 32
    assert L.q4_0_matmul_id(FAKE, FAKE, FAKE, FAKE, 2, 8, 64, 48, 16, 1 << 20, 1, None, 0, None) == 1
    # mat-mat mode without workspace -> WORKSPACE
    assert L.q4_0_matmul_id(FAKE, FAKE, FAKE, FAKE, 64, 8, 64, 64, 16, 64 * 2 * 18, 2, None, 0, None) == 3
    need = L.q4_0_matmul_id_workspace_size(64, 8, 64, 64, 16)
    assert need > 0
    assert L.q4_0_matmul_id(FAKE, FAKE, FAKE, FAKE, 64, 8, 64, 64, 16, 64 * 2 * 18, 2, FAKE, need - 1, None) == 3
    # fused SwiGLU: null up, K not a multiple of 32, misaligned gate
    assert L.q4_0_matmul_id_swiglu(FAKE, None, FAKE, FAKE, FAKE, 1, 8, 64, 64, 16, 1 << 20, None) == 1
    assert L.q4_0_matmul_id_swiglu(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 8, 64, 48, 16, 1 << 20, None) == 1
    assert L.q4_0_matmul_id_swiglu(FAKE + 4, FAKE, FAKE, FAKE, FAKE, 1, 8, 64, 64, 16, 1 << 20, None) == 2
    assert L.q4_0_matmul_id_swiglu(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 8, 64, 64, 16, 64 * 2 * 18 - 1, None) == 1
    assert L.q4_0_matmul_id_swiglu(None, None, None, None, None, 0, 8, 64, 64, 16, 0, None) == 0
    # routing: too many experts
    assert L.q4_0_route(FAKE, 8, 2000, FAKE, FAKE, None, None) == 1
    # a top_k so large that n_tokens * top_k would overflow int64 is refused, not wrapped
    assert L.q4_0_matmul_id(FAKE, FAKE, FAKE, FAKE, 1 << 40, 1 << 40, 64, 64, 16, 1 << 20, 1, None, 0, None) == 1
    assert L.q4_0_matmul_id_workspace_size(1 << 40, 1 << 40, 64, 64, 16) == 0


def test_q8_0_argument_checks(L):
    stride = 64 * 2 * 34
    # expert_stride smaller than one expert (34-byte blocks) -> INVALID_ARG
    assert L.q8_0_matmul_id(FAKE, FAKE, FAKE, FAKE, 2, 8, 64, 64, 16, stride - 1, 1, None, 0, None) == 1
    # K not a multiple of 32, bad mode
    assert L.q8_0_matmul_id(FAKE, FAKE, FAKE, FAKE, 2, 8, 64, 48, 16, 1 << 20, 1, None, 0, None) == 1
    assert L.q8_0_matmul_id(FAKE, FAKE, FAKE, FAKE, 2, 8, 64, 64, 16, stride, 3, None, 0, None) == 1
    # mat-mat without (enough) workspace -> WORKSPACE; misaligned x -> UNSUPPORTED
    assert L.q8_0_matmul_id(FAKE, FAKE, FAKE, FAKE, 64, 8, 64, 64, 16, stride, 2, None, 0, None) == 3
    need = L.q8_0_matmul_id_workspace_size(64, 8, 64, 64, 16)
    assert need == L.q4_0_matmul_id_workspace_size(64, 8, 64, 64, 16)   # the same routing and gathered rows
    assert L.q8_0_matmul_id(FAKE, FAKE, FAKE, FAKE, 64, 8, 64, 64, 16, stride, 2, FAKE, need - 1, None) == 3
    assert L.q8_0_matmul_id(FAKE + 4, FAKE, FAKE, FAKE, 2, 8, 64, 64, 16, stride, 1, None, 0, None) == 2
    # n_tokens == 0 is a no-op
    assert L.q8_0_matmul_id(None, None, None, None, 0, 8, 64, 64, 16, 0, 0, None, 0, None) == 0


def test_record_argument_checks(L):
    out = ctypes.c_void_p(123)
    # bad shapes and flags are refused before any device work, and *out is cleared
    assert L.q4_gemv_record(0, 64, 64, 0, ctypes.byref(out)) == 1 and out.value is None
    assert L.q4_gemv_record(17, 64, 64, 0, ctypes.byref(out)) == 1
    assert L.q4_gemv_record(1, 64, 48, 0, ctypes.byref(out)) == 1
    assert L.q4_gemv_record(1, 64, 64, 0x2, ctypes.byref(out)) == 1
    assert L.q4_gemv_record(1, 64, 64, 0, None) == 1
    assert L.q4_0_matmul_id_mv_record(1, 8, 64, 64, 16, 64 * 2 * 18 - 1, 0, ctypes.byref(out)) == 1
    assert L.q4_0_matmul_id_mv_record(1, 8, 64, 64, 16, 1 << 20, 2, ctypes.byref(out)) == 1
    # launching without a record, and freeing NULL
    assert L.q4_gemv_record_launch(None, FAKE, FAKE, FAKE, FAKE, FAKE, None) == 1
    # the batched replay: n = 0 is a no-op, missing arrays, records or pointers are refused
    arr = (ctypes.c_void_p * 1)
    assert L.q4_gemv_record_launch_n(None, None, None, None, None, None, 0, None) == 0
    assert L.q4_gemv_record_launch_n(None, None, None, None, None, None, 1, None) == 1
    assert L.q4_gemv_record_launch_n(arr(None), arr(FAKE), arr(FAKE), arr(FAKE), arr(FAKE), arr(FAKE), 1, None) == 1
    assert L.q4_gemv_record_launch_n(arr(None), arr(FAKE), arr(FAKE), arr(FAKE), arr(FAKE), arr(FAKE), -1, None) == 1
    assert L.q4_0_matmul_id_mv_record_launch(None, FAKE, None, FAKE, FAKE, FAKE, None) == 1
    L.q4mm_record_free(None)


def test_record_batch_checks_its_lists():
    # the Python side refuses lists of different lengths before any library call
    import weight_only_bit_int4_gb300 as q
    with pytest.raises(ValueError):
        q.RecordBatch([], [1], [], [], [], [])
