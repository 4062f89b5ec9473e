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
                                   (9, 130, 1024), (16, 64, 4096), (3, 1000, 2080), (2, 304, 1024),
                                   (3, 200, 384), (1, 72, 14336), (4, 1000, 128), (3, 1000, 512),
                                   (1, 9, 256), (2, 4104, 2048), (8, 300, 2048), (12, 1000, 4096),
                                   (6, 72, 14336), (13, 4104, 384), (5, 130, 256), (11, 4104, 768),
                                   (16, 200, 768), (7, 64, 512), (10, 2000, 14336),
                                   (1, 1000, 2304), (9, 1500, 2304), (16, 40, 7424), (1, 2100, 2304)])
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


@pytest.mark.parametrize("static_weights", [False, True])
@pytest.mark.parametrize("M", [1, 4, 16])
@pytest.mark.parametrize("K,N", [(4096, 14336), (14336, 4096), (4096, 4096)])
def test_q4_gemv_full_size_sampled(M, K, N, static_weights):
    x, w, s, b = _case(1000 + M, M, N, K)
    y = poisoned_bf16(M, N)
    q.q4_gemv(dev(x), dev(w), dev(s), dev(b), y, static_weights=static_weights)
    got_all = bf16_out(y)
    assert np.all(np.isfinite(got_all))
    rng = np.random.default_rng(M * 7 + K)
    mi = rng.integers(0, M, 600)
    ni = np.concatenate([rng.integers(0, N, 590), np.arange(N - 10, N)])
    ref = oracle.q4_matmul_at(x, w, s, b, K, mi, ni)
    assert_within_tolerance(got_all[mi, ni], ref, f"q4_gemv full M={M} K={K} N={N}")


# ------------------------------------------------ overlapped launches (Q4MM_GEMV_STATIC_WEIGHTS)
def _chain(M, D, layers, static_weights, ping_pong, graph=False):
    """Run `layers` dependent D x D decode matmuls back to back on one stream, each reading
    the previous call's output (and, with ping_pong, writing over the previous call's input);
    two weight sets alternate.  Returns every stored activation as host uint16."""
    sets = [tuple(dev(a) for a in synth.int4_weights(700 + i, D, D)) for i in range(2)]
    x0 = dev(synth.activations_bf16(710, M, D))
    n_buf = 2 if ping_pong else layers + 1
    bufs = [poisoned_bf16(M, D) for _ in range(n_buf)]
    bufs[0].copy_(x0)

    def calls():
        for i in range(layers):
            src, dst = bufs[i % n_buf], bufs[(i + 1) % n_buf]
            q.q4_gemv(src, *sets[i % 2], dst, static_weights=static_weights)

    if graph:
        st = torch.cuda.Stream()
        st.wait_stream(torch.cuda.current_stream())
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=st):
            calls()
        bufs[0].copy_(x0)
        torch.cuda.synchronize()
        g.replay()
    else:
        calls()
    torch.cuda.synchronize()
    return [host_u16(b_).copy() for b_ in bufs], sets


@pytest.mark.parametrize("M,D", [(1, 4096), (16, 1024), (4, 1056)])
@pytest.mark.parametrize("ping_pong", [False, True])
def test_q4_gemv_static_weights_chain_is_bit_identical(M, D, ping_pong):
    """Chained calls launched to overlap give exactly the outputs of plain launches: x is
    read only after the producing call has finished (a read-after-write chain), and y is
    written only after the previous call has finished reading it (ping-pong buffers)."""
    layers = 6
    plain, _ = _chain(M, D, layers, False, ping_pong)
    over, _ = _chain(M, D, layers, True, ping_pong)
    for a, b_ in zip(plain, over):
        np.testing.assert_array_equal(a, b_)
    graphed, _ = _chain(M, D, layers, True, ping_pong, graph=True)
    for a, b_ in zip(plain, graphed):
        np.testing.assert_array_equal(a, b_)


def test_q4_gemv_static_weights_first_link_matches_oracle():
    M, D = 4, 1024
    bufs, _ = _chain(M, D, 2, True, False)
    w, s, b = synth.int4_weights(700, D, D)
    x = synth.activations_bf16(710, M, D)
    ref = oracle.q4_matmul(x, w, s, b, M, D, D)
    got = synth.bf16_bits_to_f32(bufs[1]).astype(np.float64)
    assert_within_tolerance(got, ref, "first link")


# ---------------------------------------------------------------- prefill GEMM (tensor cores)
# (512, 4096, 256) and (300, 4096, 256) have few 256-token tiles and run 128-token tiles;
# (512, 1024, 2048) and (300, 512, 4096) split K over a cluster (S = 4 with 128-token tiles,
# S = 8 with a ragged token tile) and sum the partial tiles in distributed shared memory.
# (3072, 1792, 512) and (3000, 1700, 256) run 384-token tiles (a ragged last token tile and
# ragged weight rows in the second).
@pytest.mark.parametrize("M,N,K", [(16, 256, 512), (256, 128, 64), (300, 200, 96), (17, 130, 1024),
                                   (600, 384, 2048), (513, 256, 160), (512, 4096, 256), (300, 4096, 256),
                                   (512, 1024, 2048), (300, 512, 4096), (3072, 1792, 512), (3000, 1700, 256)])
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


@pytest.mark.parametrize("M,K,N", [(512, 4096, 14336), (2048, 14336, 4096), (8192, 4096, 6144),
                                   (512, 14336, 4096)])
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


# ---------------------------------------------------------------- smallest legal shapes
@pytest.mark.parametrize("M,N,K", [(1, 1, 32), (16, 1, 32), (1, 3, 32), (5, 17, 64), (16, 1, 256), (2, 1, 4096)])
def test_q4_gemv_tiny_shapes(M, N, K):
    x, w, s, b = _case(90 + M + N, M, N, K)
    ref = oracle.q4_matmul(x, w, s, b, M, N, K)
    y = poisoned_bf16(M, N)
    q.q4_gemv(dev(x), dev(w), dev(s), dev(b), y)
    assert_within_tolerance(bf16_out(y), ref, f"q4_gemv tiny M={M} N={N} K={K}")


@pytest.mark.parametrize("M,N,K", [(17, 1, 32), (1, 1, 32), (17, 3, 256), (129, 5, 64), (33, 130, 256)])
def test_q4_gemm_tiny_shapes(M, N, K):
    x, w, s, b = _case(95 + M + N, M, N, K)
    ref = oracle.q4_matmul(x, w, s, b, M, N, K)
    y = poisoned_bf16(M, N)
    q.q4_gemm(dev(x), dev(w), dev(s), dev(b), y)
    assert_within_tolerance(bf16_out(y), ref, f"q4_gemm tiny M={M} N={N} K={K}")


@pytest.mark.parametrize("N,K", [(1, 32), (3, 64), (1, 256)])
def test_q4_dequant_tiny_shapes(N, K):
    w, s, b = synth.int4_weights(97 + N, N, K)
    out = torch.empty(N, K, dtype=torch.float32, device=DEV)
    q.q4_dequant(dev(w), dev(s), dev(b), out)
    np.testing.assert_array_equal(out.cpu().numpy().view(np.uint32), oracle.q4_dequant(w, s, b, N, K).view(np.uint32))
