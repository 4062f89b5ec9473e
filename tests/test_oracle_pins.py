"""Pins for the CPU oracle: each test checks it against something other than itself --
values fixed by the pages, closed forms, invariants, library routines, brute force.

None of these tests needs a GPU.
"""
import os

import numpy as np
import pytest

import oracle
from weight_only_bit_int4_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf16(v):
    return synth.to_bf16_bits(np.asarray(v, np.float32))


# ---------------------------------------------------------------------------------------
# storage conversions
# ---------------------------------------------------------------------------------------

def _probe_floats():
    rng = np.random.default_rng(7)
    mags = np.ldexp(rng.uniform(1.0, 2.0, 20000), rng.integers(-160, 130, 20000))
    with np.errstate(over="ignore"):
        v = (mags * rng.choice([-1.0, 1.0], 20000)).astype(np.float32)
    special = np.array([0.0, -0.0, 1.0, -1.0, 65504.0, 65519.99, 65520.0, 65536.0, 1e-8,
                        2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -26, 2.0 ** -14, 6.1e-5,
                        np.finfo(np.float32).max, np.finfo(np.float32).tiny, 1e-45,
                        np.inf, -np.inf], np.float32)
    # exact ties for bf16 and f16 rounding
    ties = np.array([1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, 1 + 2.0 ** -11, 1 + 3 * 2.0 ** -11,
                     -(2 + 2.0 ** -7)], np.float32)
    return np.concatenate([v, special, ties])


def test_f16_conversion_matches_numpy():
    v = _probe_floats()
    got = oracle.f32_to_f16(v)
    with np.errstate(over="ignore"):
        want = v.astype(np.float16).view(np.uint16)
    np.testing.assert_array_equal(got, want)


def test_f16_decode_all_patterns_matches_numpy():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.f16_to_f32(bits)
    want = bits.view(np.float16).astype(np.float32)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    np.testing.assert_array_equal(got[~nan], want[~nan])


def test_bf16_conversion_is_nearest_ties_even():
    v = _probe_floats()
    v = v[np.isfinite(v)]
    got = oracle.f32_to_bf16(v).astype(np.uint32)
    u = v.view(np.uint32)
    lo = (u >> 16).astype(np.uint32)            # truncation toward zero in magnitude
    hi = lo + 1
    def dec(b):
        # decode, reading the infinity pattern as the virtual next value 2^128 so that
        # "nearest" includes rounding past the largest finite bf16 (IEEE overflow rule)
        f = (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        return np.where(np.isinf(f), np.copysign(2.0 ** 128, f), f)
    dlo = np.abs(dec(lo) - v.astype(np.float64))
    dhi = np.abs(dec(hi) - v.astype(np.float64))
    pick = np.where(dlo < dhi, lo, np.where(dhi < dlo, hi, np.where(lo % 2 == 0, lo, hi)))
    np.testing.assert_array_equal(got, pick)
    # hand-checked values
    assert oracle.f32_to_bf16(np.float32(1.0)) == 0x3F80
    assert oracle.f32_to_bf16(np.float32(1 + 2.0 ** -8)) == 0x3F80   # tie -> even
    assert oracle.f32_to_bf16(np.float32(1 + 3 * 2.0 ** -8)) == 0x3F82
    assert oracle.f32_to_bf16(np.finfo(np.float32).max) == 0x7F80     # rounds to inf


# ---------------------------------------------------------------------------------------
# INT4 group-32 affine (quant_fastkernel.rs)
# ---------------------------------------------------------------------------------------

def test_q4_dequant_hand_built_low_nibble_first():
    # Row 0: four words whose nibbles, low nibble first, read 0..7, 8..15, 7..0, 15..8.
    w = np.array([[0x76543210, 0xFEDCBA98, 0x01234567, 0x89ABCDEF],
                  [0x11111111, 0x11111111, 0x11111111, 0x11111111]], np.uint32)
    s = bf16([[0.5], [0.25]])
    b = bf16([[-2.0], [0.0]])
    nib0 = [0, 1, 2, 3, 4, 5, 6, 7, 8, 9, 10, 11, 12, 13, 14, 15,
            7, 6, 5, 4, 3, 2, 1, 0, 15, 14, 13, 12, 11, 10, 9, 8]
    want = np.array([[q * 0.5 - 2.0 for q in nib0], [0.25] * 32], np.float32)
    got = oracle.q4_dequant(w, s, b, 2, 32)
    np.testing.assert_array_equal(got, want)


def test_q4_matmul_hand_built_2x64x8():
    # Row n of W: every nibble equals n.  Group 0 scale 1, bias -0.5; group 1 scale 2, bias 0.25.
    K, N = 64, 8
    w = np.array([[n * 0x11111111] * (K // 8) for n in range(N)], np.uint32)
    s = bf16([[1.0, 2.0]] * N)
    b = bf16([[-0.5, 0.25]] * N)
    x = bf16([[1.0] * 64, [1.0] * 32 + [-1.0] * 32])
    # y0[n] = 32(n - 0.5) + 32(2n + 0.25) = 96n - 8 ; y1[n] = 32(n - 0.5) - 32(2n + 0.25) = -32n - 24
    want = np.array([[-8, 88, 184, 280, 376, 472, 568, 664],
                     [-24, -56, -88, -120, -152, -184, -216, -248]], np.float64)
    np.testing.assert_array_equal(oracle.q4_matmul(x, w, s, b, 2, N, K), want)


def test_q4_matmul_all_zero_nibbles_closed_form():
    M, N, K = 3, 5, 96
    _, s, b = synth.int4_weights(11, N, K)
    x = synth.activations_bf16(12, M, K)
    w = np.zeros((N, K // 8), np.uint32)
    xf = synth.bf16_bits_to_f32(x).astype(np.float64)
    bf = synth.bf16_bits_to_f32(b).astype(np.float64)
    xg = xf.reshape(M, K // 32, 32).sum(axis=2)          # sum of x over each group
    want = xg @ bf.T                                     # y = sum_g b[n][g] * sum_{k in g} x[m][k]
    got = oracle.q4_matmul(x, w, s, b, M, N, K)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("n0,k0,nib", [(0, 0, 1), (2, 13, 15), (4, 63, 7), (1, 40, 9)])
def test_q4_matmul_single_nibble(n0, k0, nib):
    M, N, K = 2, 5, 64
    w = np.zeros((N, K // 8), np.uint32)
    w[n0, k0 // 8] = np.uint32(nib << (4 * (k0 % 8)))
    _, s, _ = synth.int4_weights(21, N, K)
    b = np.zeros((N, K // 32), np.uint16)
    x = synth.activations_bf16(22, M, K)
    got = oracle.q4_matmul(x, w, s, b, M, N, K)
    want = np.zeros((M, N))
    xf = synth.bf16_bits_to_f32(x).astype(np.float64)
    sf = synth.bf16_bits_to_f32(s).astype(np.float64)
    want[:, n0] = xf[:, k0] * nib * sf[n0, k0 // 32]
    np.testing.assert_array_equal(got, want)


def test_q4_quantizer_round_trip():
    N, K = 6, 128
    wf = (synth.normal(31, 0, N * K) * 0.02).astype(np.float32).reshape(N, K)
    words, s, b, zp = oracle.q4_quantize(wf, N, K)
    q = ((words[..., None] >> (4 * np.arange(8, dtype=np.uint32))) & 15).reshape(N, K)
    deq = oracle.q4_dequant(words, s, b, N, K).astype(np.float64)
    sf = np.repeat(synth.bf16_bits_to_f32(s).astype(np.float64), 32, axis=1)
    zf = np.repeat(zp.astype(np.float64), 32, axis=1)
    # re-quantising the dequantised values with the same (scale, zero point) returns q exactly
    q2 = np.clip(np.rint(deq / sf) + zf, 0, 15)
    np.testing.assert_array_equal(q2, q)
    # and the dequantised value is within half a step (plus bf16 rounding of s, b) of w
    bound = sf / 2 + 16 * sf * 2.0 ** -8 + 1e-7
    assert np.all(np.abs(deq - wf) <= bound)


def test_q4_dequant_exact_on_affine_construction():
    w, s, b = synth.int4_weights(1000, 256, 512)
    assert oracle.q4_dequant_inexact(w, s, b, 256, 512) == 0


def test_q4_matmul_at_matches_full():
    M, N, K = 4, 7, 64
    w, s, b = synth.int4_weights(41, N, K)
    x = synth.activations_bf16(42, M, K)
    full = oracle.q4_matmul(x, w, s, b, M, N, K)
    mi = np.array([0, 3, 2, 1]); ni = np.array([6, 0, 3, 5])
    np.testing.assert_array_equal(oracle.q4_matmul_at(x, w, s, b, K, mi, ni), full[mi, ni])


# ---------------------------------------------------------------------------------------
# LUT4 (lut4.rs)
# ---------------------------------------------------------------------------------------

def _load_lut4_golden():
    rows = []
    with open(os.path.join(GOLDEN, "lut4_worked_example.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            parts = line.split()
            rows.append((int(parts[0], 16), float(parts[1]), int(parts[2]),
                         [float(v) for v in parts[3:]]))
    return rows


@pytest.mark.parametrize("case", _load_lut4_golden())
def test_lut4_worked_example(case):
    byte, scale, transpose, expected = case
    book = np.array([i * i / 32.0 for i in range(16)], np.float32)
    packed = np.full(32, byte, np.uint8)
    scales = np.array([scale], np.float32)
    rows, cols = 3, 5
    K, N = (cols, rows) if transpose else (rows, cols)
    x = bf16(np.full((2, K), 0.25))
    y = oracle.lut4_matmul(x, packed, scales, book, 2, N, K, 64, transpose)
    for r in range(2):
        assert list(y[r]) == expected


def test_lut4_dequant_nibble_order_and_blocks():
    # byte 0xAB: even flat index -> 0xA, odd -> 0xB; block 4 -> scale changes every 4 elements
    book = np.arange(16, dtype=np.float32)
    packed = np.array([0xAB, 0x01, 0x23, 0x45], np.uint8)
    scales = np.array([1.0, 0.5], np.float32)
    got = oracle.lut4_dequant(packed, scales, book, 2, 4, 4)
    want = np.array([[10, 11, 0, 1], [2 * 0.5, 3 * 0.5, 4 * 0.5, 5 * 0.5]], np.float32)
    np.testing.assert_array_equal(got, want)


def test_lut4_transposes_agree_on_transposed_storage():
    # The same logical W stored [N, K] (transpose=1) and [K, N] (transpose=0) with block 1
    # (one scale per element, so storage order does not change the scales) gives one y.
    M, N, K = 3, 4, 6
    rng = np.random.default_rng(5)
    codes = rng.integers(0, 16, (N, K))
    sc = rng.uniform(0.5, 1.5, (N, K)).astype(np.float32)
    book = synth.lut4_book(3)
    def pack(c):
        f = c.reshape(-1)
        return ((f[0::2] << 4) | f[1::2]).astype(np.uint8)
    x = synth.activations_bf16(6, M, K)
    y1 = oracle.lut4_matmul(x, pack(codes), sc.reshape(-1), book, M, N, K, 1, 1)
    y0 = oracle.lut4_matmul(x, pack(codes.T.copy()), sc.T.reshape(-1), book, M, N, K, 1, 0)
    np.testing.assert_array_equal(y0, y1)



@pytest.mark.parametrize("transpose", [0, 1])
def test_lut4_matmul_at_matches_full(transpose):
    # The sampled form used by the full-size checks equals the pinned full matmul at every
    # chosen (m, n), for both storage orders, with a block (32) that does not divide K (48),
    # so scale blocks straddle rows of the stored matrix.  M < N and the pairs include
    # m != n, so an (m, n) mix-up in the sampled index shows.
    M, N, K, block = 4, 5, 48, 32
    rng = np.random.default_rng(77)
    packed = rng.integers(0, 256, N * K // 2, dtype=np.uint8)
    scales = rng.uniform(0.5, 1.5, -(-N * K // block)).astype(np.float32)
    book = synth.lut4_book(78)
    x = synth.activations_bf16(79, M, K)
    full = oracle.lut4_matmul(x, packed, scales, book, M, N, K, block, transpose)
    mi = np.array([0, 3, 2, 1, 3, 0]); ni = np.array([4, 0, 3, 2, 1, 0])
    np.testing.assert_array_equal(
        oracle.lut4_matmul_at(x, packed, scales, book, N, K, block, transpose, mi, ni), full[mi, ni])

# The rounded-weight variant (lut4.rs, `rounded_weight`): Cast(decode, half|bf16) and back.

def _pack_codes(c):
    f = c.reshape(-1)
    return ((f[0::2] << 4) | f[1::2]).astype(np.uint8)


def _bf16_round_bits_trick(v):
    # nearest-even bf16 by the integer carry method (a different route from the oracle's
    # scale-and-rint); finite inputs only
    u = np.asarray(v, np.float32).view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint32) << 16
    return r.astype(np.uint32).view(np.float32)


@pytest.mark.parametrize("transpose", [0, 1])
def test_lut4_rounded_one_hot_x_is_the_cast_decoded_matrix(transpose):
    # x = identity (M = K): y[k][n] is exactly round(W[n][k]); f16 by numpy's cast, bf16 by
    # the carry method.  A swapped rounding type, a transposed W or a dropped cast fails.
    N, K, block = 6, 8, 4
    rng = np.random.default_rng(31)
    book = synth.lut4_book(9)
    rows, cols = (N, K) if transpose else (K, N)
    codes = rng.integers(0, 16, (rows, cols))
    scales = rng.uniform(0.3, 3.0, rows * cols // block).astype(np.float32)
    packed = _pack_codes(codes)
    Wst = oracle.lut4_dequant(packed, scales, book, rows, cols, block)
    W = Wst if transpose else Wst.T              # [N, K]
    x = bf16(np.eye(K))
    y16 = oracle.lut4_matmul_rounded(x, packed, scales, book, K, N, K, block, transpose, "f16")
    ybf = oracle.lut4_matmul_rounded(x, packed, scales, book, K, N, K, block, transpose, "bf16")
    np.testing.assert_array_equal(y16, W.T.astype(np.float16).astype(np.float64))
    np.testing.assert_array_equal(ybf, _bf16_round_bits_trick(W.T).astype(np.float64))
    assert not np.array_equal(y16, ybf)
    y0 = oracle.lut4_matmul_rounded(x, packed, scales, book, K, N, K, block, transpose, None)
    np.testing.assert_array_equal(y0, W.T.astype(np.float64))


def test_lut4_rounded_is_identity_on_representable_weights():
    # book entries j/8 and power-of-two scales: every decoded value has <= 4 significant bits
    # and lies well inside both ranges, so both casts are exact and y equals the plain matmul.
    M, N, K, block = 3, 5, 64, 16
    rng = np.random.default_rng(32)
    book = (np.arange(16) - 8).astype(np.float32) / 8
    packed = _pack_codes(rng.integers(0, 16, (N, K)))
    scales = np.ldexp(1.0, rng.integers(-6, 6, N * K // block)).astype(np.float32)
    x = synth.activations_bf16(33, M, K)
    plain = oracle.lut4_matmul(x, packed, scales, book, M, N, K, block, 1)
    for r in ("f16", "bf16"):
        np.testing.assert_array_equal(
            oracle.lut4_matmul_rounded(x, packed, scales, book, M, N, K, block, 1, r), plain)


def test_lut4_rounded_f16_underflow_and_overflow():
    M, N, K, block = 2, 4, 32, 32
    rng = np.random.default_rng(34)
    book = np.linspace(0.0625, 1.0, 16).astype(np.float32)
    packed = _pack_codes(rng.integers(1, 16, (N, K)))
    x = bf16(rng.uniform(0.5, 1.0, (M, K)))      # positive: no inf - inf
    # |W| <= 2^-30 < 2^-25 (half the smallest f16 subnormal): the f16 cast gives +0 exactly,
    # while bf16 keeps fp32's exponent range and the value survives.
    tiny = np.full(N * K // block, 2.0 ** -30, np.float32)
    y16 = oracle.lut4_matmul_rounded(x, packed, tiny, book, M, N, K, block, 1, "f16")
    assert np.all(y16 == 0.0)
    ybf = oracle.lut4_matmul_rounded(x, packed, tiny, book, M, N, K, block, 1, "bf16")
    assert np.all(ybf > 0.0)
    # |W| >= 0.0625 * 2^21 = 131072 > 65520: every f16 weight is +inf.
    big = np.full(N * K // block, 2.0 ** 21, np.float32)
    assert np.all(np.isposinf(oracle.lut4_matmul_rounded(x, packed, big, book, M, N, K, block, 1, "f16")))
    assert np.all(np.isfinite(oracle.lut4_matmul_rounded(x, packed, big, book, M, N, K, block, 1, "bf16")))


def test_lut4_rounded_sampled_matches_full():
    M, N, K, block = 4, 7, 96, 32
    packed, scales, book = synth.lut4_weights(35, N, K, block)
    x = synth.activations_bf16(36, M, K)
    mi = np.array([0, 3, 2, 1, 3]); ni = np.array([6, 0, 3, 5, 2])
    for r in (None, "f16", "bf16"):
        full = oracle.lut4_matmul_rounded(x, packed, scales, book, M, N, K, block, 1, r)
        np.testing.assert_array_equal(
            oracle.lut4_matmul_rounded_at(x, packed, scales, book, N, K, block, 1, r, mi, ni), full[mi, ni])


# ---------------------------------------------------------------------------------------
# GGML Q4_0 expert-routed (quantized_matmul_id_ggml.rs)
# ---------------------------------------------------------------------------------------

def _hand_block():
    # d = 0.5 (fp16 0x3800, little endian), qs[j] = j | (15 - j) << 4
    return np.array([0x00, 0x38] + [j | ((15 - j) << 4) for j in range(16)], np.uint8)


def test_q4_0_block_hand_built():
    got = oracle.q4_0_dequant_row(_hand_block(), 32)
    want = [(j - 8) * 0.5 for j in range(16)] + [(7 - j) * 0.5 for j in range(16)]
    np.testing.assert_array_equal(got, np.array(want, np.float32))


def test_q4_0_all_eights_give_zero():
    n_exp, N, K = 3, 5, 64
    w, stride = synth.q4_0_experts(51, n_exp, N, K)
    blocks = w.reshape(-1, 18)
    blocks[:, 2:] = 0x88
    x = synth.activations_f32(52, 2, K)
    ids = np.array([0, 2, 1, 0], np.uint32)
    out = oracle.q4_0_matmul_id(x, w, ids, 2, 2, N, K, n_exp, stride)
    assert np.all(out == 0.0)


def test_q4_0_one_hot_x_reads_a_column():
    n_exp, N, K = 2, 3, 64
    w = np.zeros(n_exp * N * (K // 32) * 18, np.uint8)
    blocks = w.reshape(n_exp, N, K // 32, 18)
    blocks[1, 2, 1] = _hand_block()            # expert 1, row 2, second block (k = 32..63)
    blocks[..., 1] = np.where(blocks[..., 1] == 0, 0x3C, blocks[..., 1])   # other d = 1.0
    k0 = 32 + 17                               # element 17 of that block: (7 - 1) * 0.5 = 3.0
    x = np.zeros((1, K), np.float32); x[0, k0] = 1.0
    out = oracle.q4_0_matmul_id(x, w, np.array([1], np.uint32), 1, 1, N, K, n_exp,
                                N * (K // 32) * 18)
    # rows 0 and 1 of expert 1 hold nibble 0 -> (0 - 8) * 1.0
    np.testing.assert_array_equal(out[0], [-8.0, -8.0, 3.0])


def test_q4_0_top1_ids_zero_is_dense_matmul():
    n_exp, N, K, T = 2, 6, 96, 5
    w, stride = synth.q4_0_experts(61, n_exp, N, K, expert_stride=N * (K // 32) * 18 + 64)
    x = synth.activations_f32(62, T, K)
    out = oracle.q4_0_matmul_id(x, w, np.zeros(T, np.uint32), T, 1, N, K, n_exp, stride)
    Wd = np.stack([oracle.q4_0_dequant_row(w[n * (K // 32) * 18:(n + 1) * (K // 32) * 18], K)
                   for n in range(N)]).astype(np.float64)
    np.testing.assert_allclose(out, x.astype(np.float64) @ Wd.T, rtol=1e-12, atol=1e-12)


def test_q4_0_routing_rows_follow_ids():
    n_exp, N, K, T, top_k = 5, 4, 64, 3, 2
    w, stride = synth.q4_0_experts(71, n_exp, N, K)
    x = synth.activations_f32(72, T, K)
    ids = np.array([4, 1, 0, 4, 2, 3], np.uint32)
    out = oracle.q4_0_matmul_id(x, w, ids, T, top_k, N, K, n_exp, stride)
    # row r reads token r // top_k against expert ids[r]: compare with top_k = 1 calls
    for r in range(T * top_k):
        one = oracle.q4_0_matmul_id(x[r // top_k:r // top_k + 1], w, ids[r:r + 1], 1, 1, N, K,
                                    n_exp, stride)
        np.testing.assert_array_equal(out[r], one[0])
    # permuting the slots of a token permutes its output rows
    ids2 = ids.reshape(T, top_k)[:, ::-1].reshape(-1).copy()
    out2 = oracle.q4_0_matmul_id(x, w, ids2, T, top_k, N, K, n_exp, stride)
    np.testing.assert_array_equal(out2.reshape(T, top_k, N)[:, ::-1], out.reshape(T, top_k, N))
    # an out-of-range id (far out, or exactly n_experts) gives a zero row
    for bad_id in (99, n_exp):
        ids3 = ids.copy(); ids3[3] = bad_id
        out3 = oracle.q4_0_matmul_id(x, w, ids3, T, top_k, N, K, n_exp, stride)
        assert np.all(out3[3] == 0.0)
        np.testing.assert_array_equal(np.delete(out3, 3, 0), np.delete(out, 3, 0))



def test_q4_0_matmul_id_rows_matches_full():
    # The routed-row form used by the full-size checks equals the matching rows of the
    # pinned full routed matmul.  top_k = 3 and rows that are not multiples of top_k check
    # the token row r / top_k.  x holds n_tokens * top_k rows, of which the full call reads
    # only the first n_tokens: a row read at the wrong token stays inside the buffer and
    # gives a different value.
    n_exp, N, K, T, top_k = 6, 5, 96, 4, 3
    w, stride = synth.q4_0_experts(91, n_exp, N, K)
    x = synth.activations_f32(92, T * top_k, K)
    ids = synth.routing_ids(93, T, top_k, n_exp)
    full = oracle.q4_0_matmul_id(x, w, ids, T, top_k, N, K, n_exp, stride)
    rows = np.array([0, 5, 7, 11, 3, 10, 1])
    np.testing.assert_array_equal(
        oracle.q4_0_matmul_id_rows(x, w, ids, top_k, N, K, n_exp, stride, rows), full[rows])

# ---------------------------------------------------------------------------------------
# GGML Q8_0 expert-routed (the same routing; 34-byte blocks: fp16 d, 32 signed bytes)
# ---------------------------------------------------------------------------------------

def _q8_hand_block():
    # d = 0.5 (fp16 0x3800, little endian); qs[j] = 8j - 128 (two's complement bytes),
    # except qs[31] = 127: the signed range's ends are both present
    qs = [(8 * j - 128) & 0xFF for j in range(31)] + [127]
    return np.array([0x00, 0x38] + qs, np.uint8)


def test_q8_0_block_hand_built():
    got = oracle.q8_0_dequant_row(_q8_hand_block(), 32)
    want = [(8 * j - 128) * 0.5 for j in range(31)] + [127 * 0.5]
    np.testing.assert_array_equal(got, np.array(want, np.float32))


def test_q8_0_zero_bytes_give_zero_and_one_hot_reads_a_column():
    n_exp, N, K = 2, 3, 64
    w = np.zeros(n_exp * N * (K // 32) * 34, np.uint8)
    blocks = w.reshape(n_exp, N, K // 32, 34)
    blocks[..., 1] = 0x3C                      # d = 1.0, qs = 0 everywhere
    x = synth.activations_f32(95, 2, K)
    ids = np.array([1, 0, 0, 1], np.uint32)
    assert np.all(oracle.q8_0_matmul_id(x, w, ids, 2, 2, N, K, n_exp, N * (K // 32) * 34) == 0.0)
    blocks[1, 2, 1] = _q8_hand_block()         # expert 1, row 2, second block (k = 32..63)
    k0 = 32 + 5                                # element 5: (40 - 128) * 0.5 = -44
    x1 = np.zeros((1, K), np.float32); x1[0, k0] = 1.0
    out = oracle.q8_0_matmul_id(x1, w, np.array([1], np.uint32), 1, 1, N, K, n_exp, N * (K // 32) * 34)
    np.testing.assert_array_equal(out[0], [0.0, 0.0, -44.0])


def test_q8_0_top1_ids_zero_is_dense_matmul_and_rows_follow_ids():
    n_exp, N, K, T, top_k = 3, 6, 96, 5, 2
    w, stride = synth.q8_0_experts(97, n_exp, N, K, expert_stride=N * (K // 32) * 34 + 32)
    x = synth.activations_f32(98, T, K)
    out = oracle.q8_0_matmul_id(x, w, np.zeros(T, np.uint32), T, 1, N, K, n_exp, stride)
    Wd = np.stack([oracle.q8_0_dequant_row(w[n * (K // 32) * 34:(n + 1) * (K // 32) * 34], K)
                   for n in range(N)]).astype(np.float64)
    np.testing.assert_allclose(out, x.astype(np.float64) @ Wd.T, rtol=1e-12, atol=1e-12)
    ids = np.array([2, 1, 0, 2, 1, 1, 0, 0, 2, 99], np.uint32)      # the last id is out of range
    full = oracle.q8_0_matmul_id(x, w, ids, T, top_k, N, K, n_exp, stride)
    for r in range(T * top_k - 1):
        one = oracle.q8_0_matmul_id(x[r // top_k:r // top_k + 1], w, ids[r:r + 1], 1, 1, N, K, n_exp, stride)
        np.testing.assert_array_equal(full[r], one[0])
    assert np.all(full[-1] == 0.0)
    xr = synth.activations_f32(99, T * top_k, K)   # extra rows: a wrong token row reads real data
    rows = np.array([0, 3, 5, 8, 9, 1])
    np.testing.assert_array_equal(oracle.q8_0_matmul_id_rows(xr, w, ids, top_k, N, K, n_exp, stride, rows),
                                  oracle.q8_0_matmul_id(xr, w, ids, T, top_k, N, K, n_exp, stride)[rows])


# ---------------------------------------------------------------------------------------
# Fused SwiGLU + routed Q4_0 mat-vec (quantized_matmul_id_ggml.rs,
# quantized_matmul_id_swiglu_q4_0): out[r] = (silu(gate[r]) * up[r]) . dequant(W[ids[r]])^T
# ---------------------------------------------------------------------------------------

def _dense_rows(w, stride, e, N, K):
    """Expert e's dequantised rows [N, K] from the (pinned) Q4_0 block decode."""
    rb = (K // 32) * 18
    base = e * stride
    return np.stack([oracle.q4_0_dequant_row(w[base + n * rb:base + (n + 1) * rb], K)
                     for n in range(N)]).astype(np.float64)


def test_swiglu_closed_form_at_plus_minus_ln3():
    # sigmoid(ln 3) = 3/4 and sigmoid(-ln 3) = 1/4, so silu(ln 3) = 0.75 ln 3 and
    # silu(-ln 3) = -0.25 ln 3; every other gate entry is 0 and silu(0) = 0.
    n_exp, N, K = 3, 4, 64
    w, stride = synth.q4_0_experts(81, n_exp, N, K)
    ln3 = float(np.log(3.0))
    gate = np.zeros((2, K), np.float32)
    up = synth.activations_f32(82, 2, K)
    k0, k1 = 5, 40
    gate[:, k0], gate[:, k1] = np.float32(ln3), np.float32(-ln3)
    up[:, k0], up[:, k1] = 2.0, 4.0
    ids = np.array([2, 0], np.uint32)
    out = oracle.q4_0_matmul_id_swiglu(gate, up, w, ids, N, K, n_exp, stride)
    g = float(np.float32(ln3))   # the stored gate value
    for r in range(2):
        Wd = _dense_rows(w, stride, int(ids[r]), N, K)
        s_pos = g / (1.0 + 1.0 / 3.0 * np.exp(ln3 - g))   # = 0.75 g up to the f32 rounding of ln 3
        s_neg = -g / (1.0 + 3.0 * np.exp(g - ln3))
        want = Wd[:, k0] * s_pos * 2.0 + Wd[:, k1] * s_neg * 4.0
        np.testing.assert_allclose(out[r], want, rtol=1e-12, atol=1e-15)
        np.testing.assert_allclose(out[r], Wd[:, k0] * 1.5 * ln3 - Wd[:, k1] * ln3, rtol=1e-6)


def test_swiglu_zero_gate_or_zero_up_gives_zero():
    n_exp, N, K = 2, 5, 96
    w, stride = synth.q4_0_experts(83, n_exp, N, K)
    ids = np.array([1, 0, 1], np.uint32)
    x = synth.activations_f32(84, 3, K)
    zero = np.zeros_like(x)
    assert np.all(oracle.q4_0_matmul_id_swiglu(zero, x, w, ids, N, K, n_exp, stride) == 0.0)
    assert np.all(oracle.q4_0_matmul_id_swiglu(x, zero, w, ids, N, K, n_exp, stride) == 0.0)


def _exact_gate_up(seed, T, K):
    # gate on a 1/16 grid in [-4, 4) and up in {+-1/2, +-1, +-2}: every product gate * up is
    # exact in f32, so it can be fed to the plain routed matmul as its x.
    r = synth.u64(seed, 0, 2 * T * K)
    gate = ((r[:T * K] % np.uint64(128)).astype(np.float32) - 64.0) / 16.0
    up = np.array([-2.0, -1.0, -0.5, 0.5, 1.0, 2.0], np.float32)[(r[T * K:] % np.uint64(6)).astype(np.int64)]
    return gate.reshape(T, K), up.reshape(T, K)


def test_swiglu_odd_part_is_the_plain_routed_matmul():
    # silu(z) - silu(-z) = z, so out(gate) - out(-gate) = the routed matmul of x = gate * up.
    n_exp, N, K, T = 4, 6, 128, 5
    w, stride = synth.q4_0_experts(85, n_exp, N, K)
    gate, up = _exact_gate_up(86, T, K)
    ids = np.array([3, 0, 2, 2, 1], np.uint32)
    diff = (oracle.q4_0_matmul_id_swiglu(gate, up, w, ids, N, K, n_exp, stride) -
            oracle.q4_0_matmul_id_swiglu(-gate, up, w, ids, N, K, n_exp, stride))
    plain = oracle.q4_0_matmul_id(gate * up, w, ids, T, 1, N, K, n_exp, stride)
    np.testing.assert_allclose(diff, plain, rtol=1e-11, atol=1e-11)


def test_swiglu_even_part_is_z_tanh_half_z():
    # silu(z) + silu(-z) = z tanh(z / 2); with the odd part this fixes silu(z) = z sigmoid(z).
    n_exp, N, K, T = 3, 4, 64, 3
    w, stride = synth.q4_0_experts(87, n_exp, N, K)
    gate, up = _exact_gate_up(88, T, K)
    ids = np.array([2, 1, 2], np.uint32)
    summ = (oracle.q4_0_matmul_id_swiglu(gate, up, w, ids, N, K, n_exp, stride) +
            oracle.q4_0_matmul_id_swiglu(-gate, up, w, ids, N, K, n_exp, stride))
    g = gate.astype(np.float64)
    h = g * np.tanh(g / 2.0) * up.astype(np.float64)
    for r in range(T):
        want = _dense_rows(w, stride, int(ids[r]), N, K) @ h[r]
        np.testing.assert_allclose(summ[r], want, rtol=1e-11, atol=1e-11)


def test_swiglu_rows_follow_ids_and_inputs():
    n_exp, N, K, T = 5, 3, 64, 6
    w, stride = synth.q4_0_experts(89, n_exp, N, K)
    gate = synth.activations_f32(90, T, K)
    up = synth.activations_f32(91, T, K)
    ids = np.array([4, 1, 0, 4, 2, 3], np.uint32)
    out = oracle.q4_0_matmul_id_swiglu(gate, up, w, ids, N, K, n_exp, stride)
    # a routed row depends only on its own gate/up row and its own expert
    perm = np.array([5, 3, 0, 1, 4, 2])
    outp = oracle.q4_0_matmul_id_swiglu(gate[perm], up[perm], w, ids[perm], N, K, n_exp, stride)
    np.testing.assert_array_equal(outp, out[perm])
    rows = np.array([4, 0, 4])
    np.testing.assert_array_equal(
        oracle.q4_0_matmul_id_swiglu_rows(gate, up, w, ids, N, K, n_exp, stride, rows), out[rows])
    ids2 = ids.copy(); ids2[2] = 77   # out of range: zero row, the others unchanged
    out2 = oracle.q4_0_matmul_id_swiglu(gate, up, w, ids2, N, K, n_exp, stride)
    assert np.all(out2[2] == 0.0)
    np.testing.assert_array_equal(np.delete(out2, 2, 0), np.delete(out, 2, 0))


def test_q4_0_route_hand_written():
    htpe, hids, bad = oracle.q4_0_route(np.array([3, 0, 3, 1, 0, 3, 7], np.uint32), 4)
    assert list(htpe) == [2, 1, 0, 3]
    assert list(hids) == [1, 4, 3, 0, 2, 5]
    assert bad == 1


def test_q4_0_route_id_range_boundary():
    # n_experts - 1 is the last valid id; n_experts itself and 2^32 - 1 are invalid
    htpe, hids, bad = oracle.q4_0_route(np.array([4, 3, 0xFFFFFFFF, 3, 4], np.uint32), 4)
    assert list(htpe) == [0, 0, 0, 2]
    assert list(hids) == [1, 3]
    assert bad == 3


def test_q4_0_route_invariants_brute_force():
    ids = synth.routing_ids(81, 37, 8, 64)
    htpe, hids, bad = oracle.q4_0_route(ids, 64)
    assert bad == 0 and htpe.sum() == ids.size
    assert sorted(hids.tolist()) == list(range(ids.size))
    off = 0
    for e in range(64):
        seg = hids[off:off + htpe[e]]
        assert list(seg) == [r for r in range(ids.size) if ids[r] == e]
        off += htpe[e]
    # each token's top_k experts are distinct
    assert all(len(set(ids[t * 8:(t + 1) * 8])) == 8 for t in range(37))


def test_tolerance_formula():
    y = np.array([[3.0, -4.0]])
    tol = oracle.matmul_tolerance(y)
    rms = np.sqrt(12.5)
    np.testing.assert_allclose(tol, [[3 / 256 + 0.01 * rms, 4 / 256 + 0.01 * rms]])
