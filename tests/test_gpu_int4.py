"""INT4 group-32 affine: CUDA path (through the C ABI) against the CPU oracle."""
import numpy as np
import pytest
import torch

import oracle
import weight_only_bit_int4_gb300 as q
from weight_only_bit_int4_gb300 import synth

from gpu_util import DEV, assert_within_tolerance, bf16_out, dev, host_u16, poisoned_bf16

pytestmark = pytest.mark.gpu


def _case(seed, M, N, K, outliers=0.0):
    w, s, b = synth.int4_weights(seed, N, K)
    x = synth.activations_bf16(seed + 1, M, K, outlier_frac=outliers)
    return x, w, s, b


# ---------------------------------------------------------------- dequant: bit-exact
@pytest.mark.parametrize("N,K", [(256, 512), (3, 96), (37, 4096)])
def test_q4_dequant_bit_exact(N, K):
    _, w, s, b = _case(10, 1, N, K)
    ref = oracle.q4_dequant(w, s, b, N, K)
    wd, sd, bd = dev(w), dev(s), dev(b)
    out = torch.full((N, K), float("nan"), dtype=torch.float32, device=DEV)
    q.q4_dequant(wd, sd, bd, out)
    np.testing.assert_array_equal(out.cpu().numpy().view(np.uint32), ref.view(np.uint32))
    for dt, conv in ((torch.bfloat16, oracle.f32_to_bf16), (torch.float16, oracle.f32_to_f16)):
        o = torch.empty((N, K), dtype=dt, device=DEV)
        q.q4_dequant(wd, sd, bd, o)
        np.testing.assert_array_equal(o.view(torch.int16).cpu().numpy().view(np.uint16), conv(ref))


# ---------------------------------------------------------------- decode GEMV
@pytest.mark.parametrize("M,N,K", [(16, 256, 512), (1, 256, 512), (4, 256, 512), (7, 200, 96),
                                   (9, 130, 1024), (16, 64, 4096), (3, 1000, 2080)])
def test_q4_gemv_parity(M, N, K):
    x, w, s, b = _case(20 + M, M, N, K)
    ref = oracle.q4_matmul(x, w, s, b, M, N, K)
    y = poisoned_bf16(M, N)
    q.q4_gemv(dev(x), dev(w), dev(s), dev(b), y)
    assert_within_tolerance(bf16_out(y), ref, f"q4_gemv M={M} N={N} K={K}")


def test_q4_gemv_deterministic_and_no_stray_writes():
    M, N, K = 5, 304, 1024
    x, w, s, b = _case(31, M, N, K)
    args = (dev(x), dev(w), dev(s), dev(b))
    big = poisoned_bf16(M + 2, N, 0x7FC3)      # one guard row above and below
    y = big[1:M + 1]
    q.q4_gemv(*args, y)
    first = host_u16(y).copy()
    y2 = poisoned_bf16(M, N, 0x7FC5)
    q.q4_gemv(*args, y2)
    np.testing.assert_array_equal(first, host_u16(y2))
    g = host_u16(big)
    assert np.all(g[0] == 0x7FC3) and np.all(g[-1] == 0x7FC3)


@pytest.mark.parametrize("M", [1, 4, 16])
@pytest.mark.parametrize("K,N", [(4096, 14336), (14336, 4096), (4096, 4096)])
def test_q4_gemv_full_size_sampled(M, K, N):
    x, w, s, b = _case(1000 + M, M, N, K)
    y = poisoned_bf16(M, N)
    q.q4_gemv(dev(x), dev(w), dev(s), dev(b), y)
    got_all = bf16_out(y)
    assert np.all(np.isfinite(got_all))
    rng = np.random.default_rng(M * 7 + K)
    mi = rng.integers(0, M, 600)
    ni = np.concatenate([rng.integers(0, N, 590), np.arange(N - 10, N)])
    ref = oracle.q4_matmul_at(x, w, s, b, K, mi, ni)
    assert_within_tolerance(got_all[mi, ni], ref, f"q4_gemv full M={M} K={K} N={N}")


# ---------------------------------------------------------------- prefill GEMM (tensor cores)
@pytest.mark.parametrize("M,N,K", [(16, 256, 512), (256, 128, 64), (300, 200, 96), (17, 130, 1024),
                                   (600, 384, 2048), (513, 256, 160)])
def test_q4_gemm_parity(M, N, K):
    # config-0 data (no outlier columns) at tile-spanning sizes with ragged M, N and K tails;
    # the outlier-column activations of the prefill configuration are checked at its own
    # sizes in test_q4_gemm_full_size_sampled.
    x, w, s, b = _case(40 + M, M, N, K)
    ref = oracle.q4_matmul(x, w, s, b, M, N, K)
    y = poisoned_bf16(M, N)
    q.q4_gemm(dev(x), dev(w), dev(s), dev(b), y)
    assert_within_tolerance(bf16_out(y), ref, f"q4_gemm M={M} N={N} K={K}")
    assert q.device_errors() == 0


@pytest.mark.parametrize("M,K,N", [(512, 4096, 14336), (2048, 14336, 4096), (8192, 4096, 6144)])
def test_q4_gemm_full_size_sampled(M, K, N):
    x, w, s, b = _case(2000 + M, M, N, K, outliers=0.01)
    y = poisoned_bf16(M, N)
    q.q4_gemm(dev(x), dev(w), dev(s), dev(b), y)
    got_all = bf16_out(y)
    assert np.all(np.isfinite(got_all))
    rng = np.random.default_rng(M + K)
    mi = np.concatenate([rng.integers(0, M, 500), np.full(20, M - 1)])
    ni = np.concatenate([rng.integers(0, N, 500), np.arange(N - 20, N)])
    ref = oracle.q4_matmul_at(x, w, s, b, K, mi, ni)
    assert_within_tolerance(got_all[mi, ni], ref, f"q4_gemm full M={M} K={K} N={N}")
    assert q.device_errors() == 0


def test_gemv_and_gemm_agree_on_small_case():
    M, N, K = 16, 256, 512
    x, w, s, b = _case(1000, M, N, K)
    a = [dev(v) for v in (x, w, s, b)]
    y1, y2 = poisoned_bf16(M, N), poisoned_bf16(M, N)
    q.q4_gemv(*a, y1)
    q.q4_gemm(*a, y2)
    ref = oracle.q4_matmul(x, w, s, b, M, N, K)
    assert_within_tolerance(bf16_out(y1), ref, "gemv")
    assert_within_tolerance(bf16_out(y2), ref, "gemm")


def test_zero_tokens_is_a_no_op():
    x, w, s, b = _case(50, 1, 64, 64)
    y = poisoned_bf16(1, 64)
    xd = dev(x)[:0]
    q.q4_gemv(xd, dev(w), dev(s), dev(b), y)
    q.q4_gemm(xd, dev(w), dev(s), dev(b), y)
    assert np.all(host_u16(y) == 0x7FC1)


def _bf16_round(a):
    return synth.bf16_bits_to_f32(synth.to_bf16_bits(np.asarray(a, np.float32))).astype(np.float64)


@pytest.mark.parametrize("M,N,K", [(513, 256, 160), (300, 200, 96), (40, 64, 4096)])
def test_q4_gemm_matches_bf16_operand_model(M, N, K):
    """The tensor-core path multiplies bf16(W) (W the exact fp32 dequant) by bf16 x with fp32
    accumulation and rounds y to bf16 once.  Checked to within one bf16 ulp of that model on
    outlier-column activations, where the bf16 rounding of single large terms is what
    separates y from the exact fp64 value."""
    x, w, s, b = _case(40 + M, M, N, K, outliers=0.01)
    y = poisoned_bf16(M, N)
    q.q4_gemm(dev(x), dev(w), dev(s), dev(b), y)
    model = _bf16_round(synth.bf16_bits_to_f32(x).astype(np.float64)
                        @ _bf16_round(oracle.q4_dequant(w, s, b, N, K)).T)
    got = bf16_out(y)
    ulp = np.ldexp(1.0, np.floor(np.log2(np.maximum(np.abs(model), 1e-30))).astype(int) - 7)
    assert np.all(np.abs(got - model) <= ulp + 1e-30)
