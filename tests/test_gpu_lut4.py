"""LUT4 (frozen codebook, blocked scales): CUDA path against the CPU oracle."""
import os

import numpy as np
import pytest
import torch

import oracle
import weight_only_bit_int4_gb300 as q
from weight_only_bit_int4_gb300 import synth

from gpu_util import DEV, assert_within_tolerance, bf16_out, dev, poisoned_bf16

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _case(seed, M, N, K, block=64, transpose=1):
    rows, cols = (N, K) if transpose else (K, N)
    packed, scales, book = synth.lut4_weights(seed, rows, cols, block)
    x = synth.activations_bf16(seed + 1, M, K)
    return x, packed, scales, book


# M <= 4 with K % 512 == 0 and block 32/64/128 runs the K-split decode kernel with the
# codebook pair table (ragged N, each block size, small and large K); the rest the others.
# M > 16 with K % 256 == 0 and block 128 runs the TMA GEMM with four scales per scale-tile row.
@pytest.mark.parametrize("M,N,K,block", [(1, 256, 512, 64), (16, 200, 96, 32), (5, 130, 1024, 128),
                                         (512, 256, 512, 64), (40, 300, 640, 64), (129, 128, 256, 64),
                                         (3, 130, 1024, 128), (2, 200, 2048, 32), (4, 1000, 512, 64),
                                         (1, 72, 4096, 128), (2, 4104, 1024, 64), (300, 512, 2048, 64),
                                         (33, 72, 4096, 128), (300, 520, 1024, 128)])
def test_lut4_fast_paths(M, N, K, block):
    x, packed, scales, book = _case(60 + M, M, N, K, block)
    ref = oracle.lut4_matmul(x, packed, scales, book, M, N, K, block, 1)
    y = poisoned_bf16(M, N)
    q.lut4_matmul(dev(x), dev(packed), dev(scales), book, y, N, K, block, 1)
    assert_within_tolerance(bf16_out(y), ref, f"lut4 M={M} N={N} K={K} block={block}")


@pytest.mark.parametrize("M,N,K,block,transpose", [(3, 5, 7, 4, 0), (20, 33, 70, 6, 1), (2, 64, 96, 10, 0),
                                                   (17, 40, 50, 2, 1)])
def test_lut4_general_layouts(M, N, K, block, transpose):
    x, packed, scales, book = _case(70 + M, M, N, K, block, transpose)
    ref = oracle.lut4_matmul(x, packed, scales, book, M, N, K, block, transpose)
    y = poisoned_bf16(M, N)
    q.lut4_matmul(dev(x), dev(packed), dev(scales), book, y, N, K, block, transpose)
    assert_within_tolerance(bf16_out(y), ref, f"lut4 general transpose={transpose}")


def test_lut4_worked_example_on_gpu():
    book = np.array([i * i / 32.0 for i in range(16)], np.float32)
    with open(os.path.join(GOLDEN, "lut4_worked_example.txt")) as f:
        lines = [l.split() for l in f if l.strip() and not l.startswith("#")]
    for parts in lines:
        byte, scale, transpose = int(parts[0], 16), float(parts[1]), int(parts[2])
        expected = [float(v) for v in parts[3:]]
        K, N = (5, 3) if transpose else (3, 5)
        x = synth.to_bf16_bits(np.full((2, K), 0.25, np.float32))
        y = poisoned_bf16(2, N)
        q.lut4_matmul(dev(x), dev(np.full(32, byte, np.uint8)), dev(np.array([scale], np.float32)),
                      book, y, N, K, 64, transpose)
        got = bf16_out(y)
        # the exact results are dyadic with few bits: bf16 holds them exactly
        np.testing.assert_array_equal(got, np.array([expected, expected]))


# (64, 128, 64), (129, 512, 32) and (4096, 4096, 64) take the vectorised kernel; (33, 70, 64)
# too, with a tail of 6 elements past the last whole 32; (3, 5, 4) and (33, 70, 6) the
# element kernel.
@pytest.mark.parametrize("rows,cols,block", [(64, 128, 64), (3, 5, 4), (33, 70, 6), (33, 70, 64),
                                             (129, 512, 32), (4096, 4096, 64)])
def test_lut4_dequant_bit_exact(rows, cols, block):
    packed, scales, book = synth.lut4_weights(80, rows, cols, block)
    ref = oracle.lut4_dequant(packed, scales, book, rows, cols, block)
    for dt, conv in ((torch.float32, None), (torch.bfloat16, oracle.f32_to_bf16), (torch.float16, oracle.f32_to_f16)):
        out = torch.empty((rows, cols), dtype=dt, device=DEV)
        q.lut4_dequant(dev(packed), dev(scales), book, rows, cols, block, out)
        if conv is None:
            np.testing.assert_array_equal(out.cpu().numpy().view(np.uint32), ref.view(np.uint32))
        else:
            np.testing.assert_array_equal(out.view(torch.int16).cpu().numpy().view(np.uint16), conv(ref))


@pytest.mark.parametrize("M,static_weights", [(1, False), (1, True), (512, False)])
def test_lut4_full_size_sampled(M, static_weights):
    N = K = 4096
    x, packed, scales, book = _case(3000 + M, M, N, K)
    y = poisoned_bf16(M, N)
    q.lut4_matmul(dev(x), dev(packed), dev(scales), book, y, N, K, 64, 1, static_weights=static_weights)
    got = bf16_out(y)
    assert np.all(np.isfinite(got))
    rng = np.random.default_rng(M)
    mi = rng.integers(0, M, 600)
    ni = rng.integers(0, N, 600)
    ref = oracle.lut4_matmul_at(x, packed, scales, book, N, K, 64, 1, mi, ni)
    assert_within_tolerance(got[mi, ni], ref, f"lut4 full M={M}")


def _lut4_chain(M, D, layers, static_weights, graph=False):
    """`layers` dependent D x D LUT4 decode matmuls on one stream, each reading the previous
    call's output; two weight sets alternate.  Returns every activation as host uint16."""
    sets = []
    for i in range(2):
        packed, scales, book = synth.lut4_weights(720 + i, D, D, 64)
        sets.append((dev(packed), dev(scales), book))
    x0 = dev(synth.activations_bf16(730, M, D))
    bufs = [poisoned_bf16(M, D) for _ in range(layers + 1)]
    bufs[0].copy_(x0)

    def calls():
        for i in range(layers):
            P, S, book = sets[i % 2]
            q.lut4_matmul(bufs[i], P, S, book, bufs[i + 1], D, D, 64, 1, static_weights=static_weights)

    if graph:
        st = torch.cuda.Stream()
        st.wait_stream(torch.cuda.current_stream())
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=st):
            calls()
        torch.cuda.synchronize()
        g.replay()
    else:
        calls()
    torch.cuda.synchronize()
    return [b.cpu().numpy().view(np.uint16).copy() for b in bufs]


@pytest.mark.parametrize("M,D", [(1, 4096), (3, 1024), (8, 512)])
def test_lut4_static_weights_chain_is_bit_identical(M, D):
    """Overlapped launches (Q4MM_GEMV_STATIC_WEIGHTS) read x only after the producing call has
    finished: a read-after-write chain gives exactly the plain launches' bits, also in a graph."""
    plain = _lut4_chain(M, D, 5, False)
    for graph in (False, True):
        over = _lut4_chain(M, D, 5, True, graph=graph)
        for a, b_ in zip(plain, over):
            np.testing.assert_array_equal(a, b_)


@pytest.mark.parametrize("M,N,K,block", [(1, 1, 512, 64), (1, 1, 32, 32), (17, 1, 64, 64), (3, 2, 512, 128),
                                         (1, 1, 2, 2), (20, 1, 128, 64)])
def test_lut4_tiny_shapes(M, N, K, block):
    x, packed, scales, book = _case(80 + M + K, M, N, K, block)
    ref = oracle.lut4_matmul(x, packed, scales, book, M, N, K, block, 1)
    y = poisoned_bf16(M, N)
    q.lut4_matmul(dev(x), dev(packed), dev(scales), book, y, N, K, block, 1)
    assert_within_tolerance(bf16_out(y), ref, f"lut4 tiny M={M} N={N} K={K} block={block}")


# Scales only 4-byte aligned (the header's minimum) and scale rows whose pitch is not a
# multiple of 16 bytes (block 128 with K % 512 != 0): the decode calls take the general
# kernel and the GEMM its non-TMA form, and the results are those of the aligned call.
# Block 128 keeps every cp.async copy of the scales 4 bytes wide.
@pytest.mark.parametrize("M,N,K,block,offset", [(1, 256, 1024, 128, 4), (5, 130, 1024, 128, 4),
                                                (40, 200, 1024, 128, 4), (40, 200, 768, 128, 0),
                                                (300, 130, 1280, 128, 0)])
def test_lut4_scale_alignment_and_pitch(M, N, K, block, offset):
    x, packed, scales, book = _case(950 + M + K, M, N, K, block)
    ref = oracle.lut4_matmul(x, packed, scales, book, M, N, K, block, 1)
    pad = np.zeros(offset // 4, np.float32)
    S = dev(np.concatenate([pad, scales]))[offset // 4:]
    assert S.data_ptr() % 16 == offset
    y = poisoned_bf16(M, N)
    q.lut4_matmul(dev(x), dev(packed), S, book, y, N, K, block, 1)
    assert_within_tolerance(bf16_out(y), ref, f"lut4 scales offset {offset} M={M} K={K}")


def _bf16_round(a):
    return synth.bf16_bits_to_f32(synth.to_bf16_bits(np.asarray(a, np.float32))).astype(np.float64)


# (3000, 1792, 512) runs 384-token tiles; (600, 640, 1024) 256-token ones.
@pytest.mark.parametrize("M,N,K", [(3000, 1792, 512), (600, 640, 1024)])
def test_lut4_gemm_matches_bf16_operand_model(M, N, K):
    """The tensor-core path multiplies bf16(W) (W = fl32(book * scale), the oracle's exact
    decode) by bf16 x with fp32 accumulation and rounds y to bf16 once.  With many tokens per
    weight row, a row whose weights round unluckily shows errors against the fp64 value of
    about 1 % of rms(y) in a few elements (every token of the row shares those roundings);
    against the bf16-operand model the only differences left are fp32 summation and the
    output rounding."""
    x, packed, scales, book = _case(500 + M, M, N, K, 64)
    y = poisoned_bf16(M, N)
    q.lut4_matmul(dev(x), dev(packed), dev(scales), book, y, N, K, 64, 1)
    w = oracle.lut4_dequant(packed, scales, book, N, K, 64)
    model = synth.bf16_bits_to_f32(x).astype(np.float64) @ _bf16_round(w).T
    got = bf16_out(y)
    rms = float(np.sqrt(np.mean(model * model)))
    assert np.all(np.abs(got - model) <= np.abs(model) * 2.0 ** -8 + 1e-4 * rms)


# ---------------------------------------------------------------------------------------
# The rounded-weight variant (Q4MM_LUT4_ROUND_F16 / _BF16): every route against the oracle's
# rounded matmul with a tight bound.  The rounded weight enters exactly (f16: fp32 FMA on
# CUDA cores; bf16: the tensor cores' bf16 operand, or fp32 FMA), so what is left is fp32
# summation and the bf16 output rounding.
# ---------------------------------------------------------------------------------------

def _assert_tight(got, ref, what):
    rms = float(np.sqrt(np.mean(ref * ref))) if ref.size else 0.0
    bad = np.abs(got - ref) > np.abs(ref) * 2.0 ** -8 + 1e-4 * rms
    assert not np.any(bad), f"{what}: {int(bad.sum())} of {ref.size} outside the bound"


# route per rounding: f16 -> row kernel (fast layout) or general kernel; bf16 -> row kernel
# (M <= 4, K % 512 == 0), decode kernels (M <= 16), tensor-core GEMM (M > 16, K and block
# % 64 == 0), row kernel (other fast shapes), general kernel (other layouts)
@pytest.mark.parametrize("rounding", ["f16", "bf16"])
@pytest.mark.parametrize("M,N,K,block,transpose", [
    (1, 256, 512, 64, 1), (2, 200, 2048, 32, 1), (5, 130, 1024, 128, 1), (16, 200, 96, 32, 1),
    (40, 300, 640, 64, 1), (129, 128, 256, 64, 1), (40, 300, 96, 32, 1), (33, 72, 4096, 128, 1),
    (3, 5, 7, 4, 0), (17, 40, 50, 2, 1), (1, 1, 32, 32, 1), (20, 1, 128, 64, 1)])
def test_lut4_rounded_every_route(rounding, M, N, K, block, transpose):
    x, packed, scales, book = _case(900 + M + N, M, N, K, block, transpose)
    ref = oracle.lut4_matmul_rounded(x, packed, scales, book, M, N, K, block, transpose, rounding)
    y = poisoned_bf16(M, N)
    q.lut4_matmul(dev(x), dev(packed), dev(scales), book, y, N, K, block, transpose, rounding=rounding)
    got = bf16_out(y)
    _assert_tight(got, ref, f"lut4 {rounding} M={M} N={N} K={K} block={block} t={transpose}")
    assert_within_tolerance(got, ref, "lut4 rounded")


@pytest.mark.parametrize("M,N,K,block,transpose", [(1, 64, 512, 64, 1), (40, 64, 128, 64, 1),
                                                   (3, 5, 7, 4, 0), (2, 300, 2048, 32, 1)])
def test_lut4_rounded_f16_underflow_and_overflow(M, N, K, block, transpose):
    """|W| <= 2^-30 rounds to binary16 zero: y is exactly 0, while bfloat16 (fp32's exponent
    range) and the unrounded call keep it.  |W| >= 2^17 rounds to binary16 infinity: with
    positive x and codebook, y is +inf."""
    rows, cols = (N, K) if transpose else (K, N)
    rng = np.random.default_rng(M * 7 + K)
    packed = rng.integers(0, 256, (rows * cols + 1) // 2, dtype=np.uint8)
    book = np.linspace(0.0625, 1.0, 16).astype(np.float32)
    x = synth.to_bf16_bits(rng.uniform(0.5, 1.0, (M, K)).astype(np.float32))
    n_scales = -(-rows * cols // block)
    for scale, rounding, check in ((2.0 ** -30, "f16", lambda g: np.all(g == 0.0)),
                                   (2.0 ** -30, "bf16", lambda g: np.all(g > 0.0)),
                                   (2.0 ** -30, None, lambda g: np.all(g > 0.0)),
                                   (2.0 ** 21, "f16", lambda g: np.all(np.isposinf(g))),
                                   (2.0 ** 21, "bf16", lambda g: np.all(np.isfinite(g)))):
        scales = np.full(n_scales, scale, np.float32)
        y = poisoned_bf16(M, N)
        q.lut4_matmul(dev(x), dev(packed), dev(scales), book, y, N, K, block, transpose, rounding=rounding)
        assert check(bf16_out(y)), (scale, rounding)


@pytest.mark.parametrize("M,rounding", [(1, "f16"), (1, "bf16"), (512, "f16"), (512, "bf16")])
def test_lut4_rounded_full_size_sampled(M, rounding):
    N = K = 4096
    x, packed, scales, book = _case(3100 + M, M, N, K)
    y = poisoned_bf16(M, N)
    q.lut4_matmul(dev(x), dev(packed), dev(scales), book, y, N, K, 64, 1, rounding=rounding,
                  static_weights=True)
    got = bf16_out(y)
    assert np.all(np.isfinite(got))
    rng = np.random.default_rng(M + 11)
    mi = rng.integers(0, M, 500)
    ni = rng.integers(0, N, 500)
    ref = oracle.lut4_matmul_rounded_at(x, packed, scales, book, N, K, 64, 1, rounding, mi, ni)
    _assert_tight(got[mi, ni], ref, f"lut4 {rounding} full M={M}")
