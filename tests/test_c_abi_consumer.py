"""The C ABI from plain C: tests/c_abi_consumer.c includes only include/q4mm.h and the CUDA
runtime header, links libq4mm.so, and runs the decode GEMV, the prefill GEMM, the LUT4 matmul
and the routed Q4_0 mat-vec on its own stream.  No Python or PyTorch is on that path; this
test only writes the seeded inputs and compares the program's outputs with the oracle."""
import os
import subprocess

import numpy as np
import pytest

import oracle
from weight_only_bit_int4_gb300 import synth

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
SRC = os.path.join(HERE, "c_abi_consumer.c")
PKG = os.path.join(ROOT, "weight_only_bit_int4_gb300")
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")
CFLAGS = ["-std=c99", "-Wall", "-Wextra", "-Werror", "-O1", "-I", os.path.join(ROOT, "include"),
          "-I", os.path.join(CUDA, "include")]


def test_consumer_compiles_as_c99(tmp_path):
    """The public header is valid C99 (compile only: no library or GPU needed)."""
    subprocess.check_call(["gcc", *CFLAGS, "-c", SRC, "-o", str(tmp_path / "c.o")])


def _build(tmp_path):
    exe = str(tmp_path / "c_abi_consumer")
    lib64 = os.path.join(CUDA, "lib64")
    subprocess.check_call(["gcc", *CFLAGS, SRC, "-o", exe, "-L", PKG, "-lq4mm", "-L", lib64, "-lcudart",
                           f"-Wl,-rpath,{PKG}", f"-Wl,-rpath,{lib64}"])
    return exe


def _write(d, name, a):
    np.ascontiguousarray(a).tofile(os.path.join(d, name))


@pytest.mark.gpu
def test_consumer_runs_and_matches_oracle(tmp_path):
    d = str(tmp_path)
    exe = _build(tmp_path)
    M, N, K = 5, 300, 1024                 # decode GEMV (M <= 16) and GEMM on the same operands
    ML, NL, KL = 2, 256, 1024              # LUT4, K-split decode kernel
    T, TOPK, NQ, KQ, E = 3, 4, 96, 512, 6  # routed Q4_0 mat-vec
    w, s, b = synth.int4_weights(800, N, K)
    x = synth.activations_bf16(801, M, K)
    packed, lsc, book = synth.lut4_weights(802, NL, KL, 64)
    xl = synth.activations_bf16(803, ML, KL)
    wq, stride = synth.q4_0_experts(804, E, NQ, KQ)
    ids = synth.routing_ids(805, T, TOPK, E)
    xq = synth.activations_f32(806, T, KQ)
    for name, a in [("int4_x.bin", x), ("int4_w.bin", w), ("int4_s.bin", s), ("int4_b.bin", b),
                    ("lut4_x.bin", xl), ("lut4_p.bin", packed), ("lut4_s.bin", lsc),
                    ("lut4_book.bin", np.asarray(book, np.float32)), ("moe_x.bin", xq), ("moe_w.bin", wq),
                    ("moe_ids.bin", ids)]:
        _write(d, name, a)
    with open(os.path.join(d, "dims.txt"), "w") as f:
        f.write(f"{M} {N} {K} {ML} {NL} {KL} {T} {TOPK} {NQ} {KQ} {E} {stride}\n")
    r = subprocess.run([exe, d], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr

    def bf16_file(name, shape):
        return synth.bf16_bits_to_f32(np.fromfile(os.path.join(d, name), np.uint16).reshape(shape)).astype(np.float64)

    def check(got, ref, what):
        tol = oracle.matmul_tolerance(ref)
        assert np.all(np.abs(got - ref) <= tol), what

    ref = oracle.q4_matmul(x, w, s, b, M, N, K)
    check(bf16_file("gemv_y.bin", (M, N)), ref, "q4_gemv from C")
    check(bf16_file("gemm_y.bin", (M, N)), ref, "q4_gemm from C")
    check(bf16_file("lut4_y.bin", (ML, NL)), oracle.lut4_matmul(xl, packed, lsc, book, ML, NL, KL, 64, 1),
          "lut4_matmul from C")
    got = np.fromfile(os.path.join(d, "moe_out.bin"), np.float32).reshape(T * TOPK, NQ).astype(np.float64)
    check(got, oracle.q4_0_matmul_id(xq, wq, ids, T, TOPK, NQ, KQ, E, stride), "q4_0_matmul_id from C")
