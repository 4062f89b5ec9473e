"""libq4mm: weight-only 4-bit quantized matmuls, y = x . dequant(W)^T, for one GB300.

Every function here has the name of a C-ABI entry point in include/q4mm.h and does
argument marshalling only (tensor -> device pointer, shape -> sizes, current CUDA stream);
every step of the computation runs in the library's own CUDA kernels.  A non-OK status
raises Q4MMError.  There is no CPU path.
"""
from __future__ import annotations

import ctypes

import torch

from ._lib import lib

Q4MM_OK = 0
Q4MM_F32, Q4MM_BF16, Q4MM_F16 = 0, 1, 2
MM_ID_THRESHOLD = 32
_DTYPES = {torch.float32: Q4MM_F32, torch.bfloat16: Q4MM_BF16, torch.float16: Q4MM_F16}


class Q4MMError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn}: {lib().q4mm_status_string(status).decode()} (status {status})")


def _check(fn: str, status: int) -> None:
    if status != Q4MM_OK:
        raise Q4MMError(fn, status)


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _stream(stream) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def version() -> int:
    return lib().q4mm_version()


def device_errors(clear: bool = True) -> int:
    v = ctypes.c_uint32(0)
    _check("q4mm_device_errors", lib().q4mm_device_errors(ctypes.byref(v), int(clear)))
    return v.value


def q4_dequant(w, scales, biases, out, stream=None) -> None:
    """out[N, K] (float32/bfloat16/float16) = fmaf(code, scale, bias), codes low nibble first."""
    N, K = w.shape[0], w.shape[1] * 8
    _check("q4_dequant", lib().q4_dequant(_ptr(w), _ptr(scales), _ptr(biases), N, K, _ptr(out),
                                          _DTYPES[out.dtype], _stream(stream)))


GEMV_STATIC_WEIGHTS = 0x1
LUT4_ROUND_F16, LUT4_ROUND_BF16 = 0x2, 0x4


def q4_gemv(x, w, scales, biases, y, stream=None, static_weights: bool = False) -> None:
    """y[M, N] = x[M, K] . W^T for 1 <= M <= 16 (bf16 in/out).

    static_weights=True promises that the kernel before this call in the stream does not
    write w/scales/biases; the call then streams W while that kernel finishes (q4_gemv_ex
    with Q4MM_GEMV_STATIC_WEIGHTS).  Results are identical either way."""
    M, K = x.shape
    N = w.shape[0]
    if static_weights:
        _check("q4_gemv_ex", lib().q4_gemv_ex(_ptr(x), _ptr(w), _ptr(scales), _ptr(biases), _ptr(y), M, N, K,
                                              GEMV_STATIC_WEIGHTS, _stream(stream)))
        return
    _check("q4_gemv", lib().q4_gemv(_ptr(x), _ptr(w), _ptr(scales), _ptr(biases), _ptr(y), M, N, K,
                                    _stream(stream)))


def q4_gemm(x, w, scales, biases, y, stream=None) -> None:
    """y[M, N] = x[M, K] . W^T on the tensor cores (bf16 in/out)."""
    M, K = x.shape
    N = w.shape[0]
    _check("q4_gemm", lib().q4_gemm(_ptr(x), _ptr(w), _ptr(scales), _ptr(biases), _ptr(y), M, N, K,
                                    _stream(stream)))


def _book_ptr(book):
    arr = (ctypes.c_float * 16)(*[float(v) for v in book])
    return arr, ctypes.cast(arr, ctypes.c_void_p)


_LUT4_ROUND = {None: 0, "f16": LUT4_ROUND_F16, "bf16": LUT4_ROUND_BF16}


def lut4_matmul(x, packed, scales, book, y, N: int, K: int, block: int, transpose: int,
                stream=None, static_weights: bool = False, rounding=None) -> None:
    """y[M, N] = x[M, K] . W^T with W[n][k] = fl32(book[code] * scale) (see q4mm.h).
    static_weights=True: lut4_matmul_ex with Q4MM_GEMV_STATIC_WEIGHTS (see q4_gemv).
    rounding="f16" | "bf16": lut4_matmul_ex with Q4MM_LUT4_ROUND_F16 | _BF16 (the decoded
    weight is rounded to that type before the product)."""
    M = x.shape[0]
    keep, bp = _book_ptr(book)
    flags = (GEMV_STATIC_WEIGHTS if static_weights else 0) | _LUT4_ROUND[rounding]
    if flags:
        _check("lut4_matmul_ex", lib().lut4_matmul_ex(_ptr(x), _ptr(packed), _ptr(scales), bp, _ptr(y), M, N,
                                                      K, block, int(transpose), flags, _stream(stream)))
    else:
        _check("lut4_matmul", lib().lut4_matmul(_ptr(x), _ptr(packed), _ptr(scales), bp, _ptr(y), M, N,
                                                K, block, int(transpose), _stream(stream)))
    del keep


def lut4_dequant(packed, scales, book, rows: int, cols: int, block: int, out, stream=None) -> None:
    keep, bp = _book_ptr(book)
    _check("lut4_dequant", lib().lut4_dequant(_ptr(packed), _ptr(scales), bp, rows, cols, block,
                                              _ptr(out), _DTYPES[out.dtype], _stream(stream)))
    del keep


def q4_0_route(ids, n_experts: int, htpe, hids, n_invalid=None, stream=None) -> None:
    _check("q4_0_route", lib().q4_0_route(_ptr(ids), ids.numel(), n_experts, _ptr(htpe), _ptr(hids),
                                          _ptr(n_invalid), _stream(stream)))


def q4_0_matmul_id_workspace_size(n_tokens: int, top_k: int, N: int, K: int, n_experts: int) -> int:
    return int(lib().q4_0_matmul_id_workspace_size(n_tokens, top_k, N, K, n_experts))


def q4_0_matmul_id(x, w, ids, out, top_k: int, N: int, K: int, n_experts: int,
                   expert_stride: int, mode: int = 0, workspace=None, stream=None) -> None:
    """out[n_tokens*top_k, N] f32: row r = x[r // top_k] . dequant_q4_0(W[ids[r]])^T."""
    n_tokens = x.shape[0]
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("q4_0_matmul_id", lib().q4_0_matmul_id(
        _ptr(x), _ptr(w), _ptr(ids), _ptr(out), n_tokens, top_k, N, K, n_experts, expert_stride,
        mode, _ptr(workspace), ws_bytes, _stream(stream)))


def q8_0_matmul_id_workspace_size(n_tokens: int, top_k: int, N: int, K: int, n_experts: int) -> int:
    return int(lib().q8_0_matmul_id_workspace_size(n_tokens, top_k, N, K, n_experts))


def q8_0_matmul_id(x, w, ids, out, top_k: int, N: int, K: int, n_experts: int,
                   expert_stride: int, mode: int = 0, workspace=None, stream=None) -> None:
    """out[n_tokens*top_k, N] f32: row r = x[r // top_k] . dequant_q8_0(W[ids[r]])^T."""
    n_tokens = x.shape[0]
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("q8_0_matmul_id", lib().q8_0_matmul_id(
        _ptr(x), _ptr(w), _ptr(ids), _ptr(out), n_tokens, top_k, N, K, n_experts, expert_stride,
        mode, _ptr(workspace), ws_bytes, _stream(stream)))


def q4_0_matmul_id_swiglu(gate, up, w, ids, out, top_k: int, N: int, K: int, n_experts: int,
                          expert_stride: int, stream=None) -> None:
    """out[r, N] f32 = (silu(gate[r]) * up[r]) . dequant_q4_0(W[ids[r]])^T for every routed row
    r; gate and up are [n_tokens*top_k, K] f32 (one row per routed row)."""
    n_rows, K_ = gate.shape
    assert K_ == K and n_rows % top_k == 0
    _check("q4_0_matmul_id_swiglu", lib().q4_0_matmul_id_swiglu(
        _ptr(gate), _ptr(up), _ptr(w), _ptr(ids), _ptr(out), n_rows // top_k, top_k, N, K, n_experts,
        expert_stride, _stream(stream)))


def q4_0_matmul_id_noalloc(x, w, ids, out, top_k: int, N: int, K: int, n_experts: int,
                           expert_stride: int, stream=None) -> None:
    """Mat-mat form of q4_0_matmul_id for callers that cannot provide (or allocate) a
    workspace: the library's own fixed scratch array is used instead (see q4mm.h)."""
    n_tokens = x.shape[0]
    _check("q4_0_matmul_id_noalloc", lib().q4_0_matmul_id_noalloc(
        _ptr(x), _ptr(w), _ptr(ids), _ptr(out), n_tokens, top_k, N, K, n_experts, expert_stride,
        _stream(stream)))


class Record:
    """A dispatch record (q4mm.h): one decode call planned once, replayed with new tensors.
    Owns the library's host-side record and frees it when garbage-collected or closed."""

    def __init__(self, kind: str, handle: int):
        self.kind = kind
        self._h = handle

    def close(self) -> None:
        if self._h:
            lib().q4mm_record_free(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def gemv(self, x, w, scales, biases, y, stream=None) -> None:
        _check("q4_gemv_record_launch", lib().q4_gemv_record_launch(
            self._h, _ptr(x), _ptr(w), _ptr(scales), _ptr(biases), _ptr(y), _stream(stream)))

    def matmul_id_mv(self, x, w, ids, out, up=None, stream=None) -> None:
        _check("q4_0_matmul_id_mv_record_launch", lib().q4_0_matmul_id_mv_record_launch(
            self._h, _ptr(x), _ptr(up), _ptr(w), _ptr(ids), _ptr(out), _stream(stream)))


def q4_gemv_record(M: int, N: int, K: int, static_weights: bool = False) -> Record:
    h = ctypes.c_void_p()
    _check("q4_gemv_record", lib().q4_gemv_record(M, N, K, GEMV_STATIC_WEIGHTS if static_weights else 0,
                                                  ctypes.byref(h)))
    return Record("gemv", h.value)


class RecordBatch:
    """A prepared q4_gemv_record_launch_n call: records[i] on xs[i], ws[i], scales[i],
    biases[i], ys[i].  The host pointer arrays are built once (the tensors are kept alive);
    launch() replays all the records in order in one library call."""

    def __init__(self, records, xs, ws, scales, biases, ys):
        n = len(records)
        if not all(len(v) == n for v in (xs, ws, scales, biases, ys)):
            raise ValueError("RecordBatch: every list needs one entry per record")
        arr = ctypes.c_void_p * n
        self._keep = (list(records), list(xs), list(ws), list(scales), list(biases), list(ys))
        self._arrays = (arr(*[r._h for r in records]), arr(*[_ptr(t) for t in xs]), arr(*[_ptr(t) for t in ws]),
                        arr(*[_ptr(t) for t in scales]), arr(*[_ptr(t) for t in biases]),
                        arr(*[_ptr(t) for t in ys]))
        self._n = n

    def launch(self, stream=None) -> None:
        _check("q4_gemv_record_launch_n", lib().q4_gemv_record_launch_n(*self._arrays, self._n, _stream(stream)))


def q4_gemv_record_launch_n(records, xs, ws, scales, biases, ys, stream=None) -> None:
    """Replay gemv records in order in one library call: records[i] on xs[i], ws[i],
    scales[i], biases[i], ys[i] (q4_gemv_record_launch_n)."""
    RecordBatch(records, xs, ws, scales, biases, ys).launch(stream)


def q4_0_matmul_id_mv_record(n_tokens: int, top_k: int, N: int, K: int, n_experts: int,
                             expert_stride: int, swiglu: bool = False) -> Record:
    h = ctypes.c_void_p()
    _check("q4_0_matmul_id_mv_record", lib().q4_0_matmul_id_mv_record(
        n_tokens, top_k, N, K, n_experts, expert_stride, int(swiglu), ctypes.byref(h)))
    return Record("swiglu" if swiglu else "mv", h.value)
