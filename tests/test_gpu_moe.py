"""GGML Q4_0 expert-routed matmul: routing lists (exact) and mat-vec / mat-mat outputs
against the CPU oracle."""
import numpy as np
import pytest
import torch

import oracle
import weight_only_bit_int4_gb300 as q
from weight_only_bit_int4_gb300 import synth

from gpu_util import DEV, assert_within_tolerance, dev

pytestmark = pytest.mark.gpu


def _route_gpu(ids, E):
    idsd = dev(ids)
    htpe = torch.zeros(E, dtype=torch.int32, device=DEV)
    hids = torch.full((ids.size,), -7, dtype=torch.int32, device=DEV)
    bad = torch.zeros(1, dtype=torch.int32, device=DEV)
    q.q4_0_route(idsd, E, htpe, hids, bad)
    return htpe.cpu().numpy().view(np.uint32), hids.cpu().numpy(), int(bad.cpu().numpy()[0])


# (2000, 8, 64) and (20000, 1, 3) hold more ids than the per-expert form stages in shared
# memory and take the single-CTA form.
@pytest.mark.parametrize("n_tokens,top_k,E", [(1, 8, 64), (512, 8, 64), (37, 3, 5), (1000, 1, 7),
                                              (3, 8, 1024), (700, 8, 64), (2000, 8, 64), (20000, 1, 3)])
def test_route_exact(n_tokens, top_k, E):
    ids = synth.routing_ids(90 + n_tokens, n_tokens, top_k, E) if top_k <= E else None
    htpe, hids, bad = _route_gpu(ids, E)
    r_htpe, r_hids, r_bad = oracle.q4_0_route(ids, E)
    np.testing.assert_array_equal(htpe, r_htpe)
    np.testing.assert_array_equal(hids[:r_hids.size], r_hids)
    assert bad == r_bad == 0


def test_route_duplicates_and_invalid_ids():
    ids = np.array([3, 0, 3, 1, 0, 3, 7, 3, 3, 0] * 50, np.uint32)
    htpe, hids, bad = _route_gpu(ids, 4)
    r_htpe, r_hids, r_bad = oracle.q4_0_route(ids, 4)
    np.testing.assert_array_equal(htpe, r_htpe)
    np.testing.assert_array_equal(hids[:r_hids.size], r_hids)
    assert bad == r_bad == 50
    assert q.device_errors() & 0x2


def _moe_case(seed, n_tokens, top_k, E, N, K, pad=0):
    per = N * (K // 32) * 18
    w, stride = synth.q4_0_experts(seed, E, N, K, expert_stride=per + pad)
    ids = synth.routing_ids(seed + 1, n_tokens, top_k, E)
    x = synth.activations_f32(seed + 2, n_tokens, K)
    return x, w, stride, ids


def _run(x, w, ids, top_k, N, K, E, stride, mode):
    n_rows = x.shape[0] * top_k
    out = torch.full((n_rows, N), float("nan"), dtype=torch.float32, device=DEV)
    ws = None
    if mode != 1:
        nbytes = q.q4_0_matmul_id_workspace_size(x.shape[0], top_k, N, K, E)
        ws = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
    q.q4_0_matmul_id(dev(x), dev(w), dev(ids), out, top_k, N, K, E, stride, mode=mode, workspace=ws)
    return out.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("mode", [1, 2])
@pytest.mark.parametrize("n_tokens,top_k,E,N,K,pad", [(1, 8, 64, 96, 256, 0), (5, 2, 6, 64, 2048, 48),
                                                      (40, 8, 16, 130, 512, 16), (33, 1, 3, 256, 96, 0),
                                                      (3, 4, 9, 70, 4096, 0), (2, 4, 7, 48, 1408, 8),
                                                      (3, 2, 5, 40, 384, 0), (2, 2, 3, 20, 128, 0)])
def test_moe_parity(mode, n_tokens, top_k, E, N, K, pad):
    x, w, stride, ids = _moe_case(100 + n_tokens, n_tokens, top_k, E, N, K, pad)
    ref = oracle.q4_0_matmul_id(x, w, ids, n_tokens, top_k, N, K, E, stride)
    got = _run(x, w, ids, top_k, N, K, E, stride, mode)
    assert_within_tolerance(got, ref, f"q4_0_matmul_id mode={mode}")


# Invalid ids in one 32-row chunk, in chunks zeroed by different CTAs, and in an id count
# large enough for the single-CTA routing form.
# K = 128 runs the CUDA-core kernels, K = 256 the tensor-core mat-mat kernel.
@pytest.mark.parametrize("K", [128, 256])
@pytest.mark.parametrize("mode", [1, 2])
@pytest.mark.parametrize("n_tokens,top_k,E,bad_rows", [(6, 2, 4, [5]), (300, 4, 8, [5, 100, 101, 700, 1199]),
                                                       (1600, 8, 8, [0, 4000, 12799])])
def test_moe_invalid_id_gives_zero_row(mode, n_tokens, top_k, E, bad_rows, K):
    N = 64
    x, w, stride, ids = _moe_case(7, n_tokens, top_k, E, N, K)
    ids = ids.copy()
    ids[bad_rows] = 99
    ref = oracle.q4_0_matmul_id(x, w, ids, n_tokens, top_k, N, K, E, stride)
    got = _run(x, w, ids, top_k, N, K, E, stride, mode)
    assert np.all(got[bad_rows] == 0.0)
    assert_within_tolerance(got, ref, "invalid id")
    assert q.device_errors() & 0x2



# Rows of x far outside the fp16 range and far below its normal range: the mat-mat form scales
# each gathered row by a power of two, so every finite f32 row is served.  Each routed row is
# held to the tolerance with rms over that row alone, so a small row is not excused by the
# large ones.  K = 512 runs the tensor-core kernel (fp16 operands); K = 288 the CUDA-core one.
@pytest.mark.parametrize("K", [512, 288])
@pytest.mark.parametrize("mode", [0, 2])
def test_moe_mm_any_f32_row_range(mode, K):
    n_tokens, top_k, E, N = 48, 4, 8, 192
    x, w, stride, ids = _moe_case(4200 + K, n_tokens, top_k, E, N, K)
    x = x.copy()
    gains = np.array([1e6, 1e-6, 1.0, 3e4, 2e-5, 7e7, 1e-30, 5e30], np.float32)
    x *= gains[np.arange(n_tokens) % gains.size][:, None]
    x[5, 17] = 1e9                      # one element far above the rest of its row
    x[9, :] *= np.float32(1e-8)         # a row that sits in f32's low range
    assert np.all(np.isfinite(x))
    q.device_errors()
    got = _run(x, w, ids, top_k, N, K, E, stride, mode)
    ref = oracle.q4_0_matmul_id(x, w, ids, n_tokens, top_k, N, K, E, stride)
    assert np.all(np.isfinite(got))
    for r in range(n_tokens * top_k):
        assert_within_tolerance(got[r], ref[r], f"routed row {r} (token {r // top_k}), mode={mode}, K={K}")
    assert q.device_errors() == 0

@pytest.mark.parametrize("n_tokens", [1, 512])
@pytest.mark.parametrize("mode", [0, 1, 2])
def test_moe_full_size_sampled(n_tokens, mode):
    E, top_k, N, K = 64, 8, 1408, 2048
    x, w, stride, ids = _moe_case(4000 + n_tokens, n_tokens, top_k, E, N, K)
    got = _run(x, w, ids, top_k, N, K, E, stride, mode)
    assert np.all(np.isfinite(got))
    rows = np.unique(np.concatenate([np.arange(min(8, n_tokens * top_k)),
                                     np.random.default_rng(n_tokens).integers(0, n_tokens * top_k, 24)]))
    ref = oracle.q4_0_matmul_id_rows(x, w, ids, top_k, N, K, E, stride, rows)
    assert_within_tolerance(got[rows], ref, f"moe full n_tokens={n_tokens} mode={mode}")


def test_moe_workspace_checks():
    x, w, stride, ids = _moe_case(9, 40, 8, 16, 64, 64)
    out = torch.empty((320, 64), dtype=torch.float32, device=DEV)
    with pytest.raises(q.Q4MMError) as ei:
        q.q4_0_matmul_id(dev(x), dev(w), dev(ids), out, 8, 64, 64, 16, stride, mode=2, workspace=None)
    assert ei.value.status == 3


# ---------------------------------------------------------------------------------------
# Fused SwiGLU + routed Q4_0 mat-vec (quantized_matmul_id_swiglu_q4_0)
# ---------------------------------------------------------------------------------------

def _swiglu_case(seed, n_tokens, top_k, E, N, K, pad=0):
    per = N * (K // 32) * 18
    w, stride = synth.q4_0_experts(seed, E, N, K, expert_stride=per + pad)
    ids = synth.routing_ids(seed + 1, n_tokens, top_k, E)
    gate = synth.activations_f32(seed + 2, n_tokens * top_k, K)
    up = synth.activations_f32(seed + 3, n_tokens * top_k, K)
    return gate, up, w, stride, ids


def _run_swiglu(gate, up, w, ids, top_k, N, K, E, stride):
    out = torch.full((gate.shape[0], N), float("nan"), dtype=torch.float32, device=DEV)
    q.q4_0_matmul_id_swiglu(dev(gate), dev(up), dev(w), dev(ids), out, top_k, N, K, E, stride)
    return out.cpu().numpy().astype(np.float64)


# K % 256 == 0 (16-byte copies), K % 128 == 0 with a 4-block tail chunk and 8-byte copies
# (1408 is the down projection of the 64-expert configuration), K = 128 (one tail chunk),
# and the fp32 FMA kernel (K % 128 != 0, or an expert stride that is not 8-byte aligned).
@pytest.mark.parametrize("n_tokens,top_k,E,N,K,pad", [(1, 8, 64, 96, 256, 0), (1, 8, 64, 2048, 1408, 0),
                                                      (5, 2, 6, 64, 640, 8), (3, 4, 9, 70, 384, 0),
                                                      (2, 3, 4, 24, 128, 0), (4, 2, 5, 33, 96, 0),
                                                      (2, 3, 4, 40, 256, 4), (40, 8, 16, 130, 512, 16)])
def test_swiglu_parity(n_tokens, top_k, E, N, K, pad):
    gate, up, w, stride, ids = _swiglu_case(300 + n_tokens + K, n_tokens, top_k, E, N, K, pad)
    ref = oracle.q4_0_matmul_id_swiglu(gate, up, w, ids, N, K, E, stride)
    got = _run_swiglu(gate, up, w, ids, top_k, N, K, E, stride)
    assert_within_tolerance(got, ref, f"q4_0_matmul_id_swiglu K={K}")


def test_swiglu_saturated_gates():
    # gates far into both tails: silu(-90) ~ 0 (exp overflows to inf in fp32), silu(90) = 90
    n_tokens, top_k, E, N, K = 2, 2, 3, 32, 256
    gate, up, w, stride, ids = _swiglu_case(77, n_tokens, top_k, E, N, K)
    gate[:, ::3] = -90.0
    gate[:, 1::7] = 90.0
    ref = oracle.q4_0_matmul_id_swiglu(gate, up, w, ids, N, K, E, stride)
    got = _run_swiglu(gate, up, w, ids, top_k, N, K, E, stride)
    assert_within_tolerance(got, ref, "swiglu saturated gates")


@pytest.mark.parametrize("K", [1408, 96])
def test_swiglu_invalid_id_gives_zero_row(K):
    n_tokens, top_k, E, N = 3, 4, 6, 48
    gate, up, w, stride, ids = _swiglu_case(81, n_tokens, top_k, E, N, K)
    ids = ids.copy()
    ids[[1, 10]] = 1000
    ref = oracle.q4_0_matmul_id_swiglu(gate, up, w, ids, N, K, E, stride)
    got = _run_swiglu(gate, up, w, ids, top_k, N, K, E, stride)
    assert np.all(got[[1, 10]] == 0.0)
    assert_within_tolerance(got, ref, "swiglu invalid id")
    assert q.device_errors() & 0x2


@pytest.mark.parametrize("n_tokens", [1, 64])
def test_swiglu_full_size_sampled(n_tokens):
    # the down projection of the 64-expert, top-8 configuration: K = 1408 -> N = 2048
    E, top_k, N, K = 64, 8, 2048, 1408
    gate, up, w, stride, ids = _swiglu_case(5000 + n_tokens, n_tokens, top_k, E, N, K)
    got = _run_swiglu(gate, up, w, ids, top_k, N, K, E, stride)
    assert np.all(np.isfinite(got))
    rows = np.unique(np.concatenate([np.arange(min(8, n_tokens * top_k)),
                                     np.random.default_rng(n_tokens).integers(0, n_tokens * top_k, 16)]))
    ref = oracle.q4_0_matmul_id_swiglu_rows(gate, up, w, ids, N, K, E, stride, rows)
    assert_within_tolerance(got[rows], ref, f"swiglu full n_tokens={n_tokens}")


def test_swiglu_zero_tokens_is_a_no_op():
    out = torch.full((4, 8), 5.0, dtype=torch.float32, device=DEV)
    z = torch.empty((0, 64), dtype=torch.float32, device=DEV)
    q.q4_0_matmul_id_swiglu(z, z, out, out, out, 1, 8, 64, 1, 8 * 2 * 18)
    assert torch.all(out == 5.0)


@pytest.mark.parametrize("mode", [1, 2])
@pytest.mark.parametrize("n_tokens,top_k,E,N,K", [(1, 1, 1, 1, 32), (2, 1, 2, 1, 256), (1, 2, 3, 5, 32), (33, 2, 2, 3, 256)])
def test_moe_tiny_shapes(mode, n_tokens, top_k, E, N, K):
    x, w, stride, ids = _moe_case(60 + n_tokens + K, n_tokens, top_k, E, N, K)
    ref = oracle.q4_0_matmul_id(x, w, ids, n_tokens, top_k, N, K, E, stride)
    got = _run(x, w, ids, top_k, N, K, E, stride, mode)
    assert_within_tolerance(got, ref, f"tiny moe mode={mode}")


@pytest.mark.parametrize("n_tokens,top_k,E,N,K", [(1, 1, 1, 1, 32), (1, 2, 3, 1, 128), (2, 1, 2, 3, 256)])
def test_swiglu_tiny_shapes(n_tokens, top_k, E, N, K):
    gate, up, w, stride, ids = _swiglu_case(70 + K, n_tokens, top_k, E, N, K)
    ref = oracle.q4_0_matmul_id_swiglu(gate, up, w, ids, N, K, E, stride)
    got = _run_swiglu(gate, up, w, ids, top_k, N, K, E, stride)
    assert_within_tolerance(got, ref, "tiny swiglu")


# ---------------------------------------------------------------------------------------
# GGML Q8_0 routed matmul: both forms against the oracle
# ---------------------------------------------------------------------------------------

def _q8_case(seed, n_tokens, top_k, E, N, K, pad=0):
    per = N * (K // 32) * 34
    w, stride = synth.q8_0_experts(seed, E, N, K, expert_stride=per + pad)
    ids = synth.routing_ids(seed + 1, n_tokens, top_k, E)
    x = synth.activations_f32(seed + 2, n_tokens, K)
    return x, w, stride, ids


def _run_q8(x, w, ids, top_k, N, K, E, stride, mode):
    n_rows = x.shape[0] * top_k
    out = torch.full((n_rows, N), float("nan"), dtype=torch.float32, device=DEV)
    ws = None
    if mode != 1:
        ws = torch.empty(q.q8_0_matmul_id_workspace_size(x.shape[0], top_k, N, K, E), dtype=torch.uint8, device=DEV)
    q.q8_0_matmul_id(dev(x), dev(w), dev(ids), out, top_k, N, K, E, stride, mode=mode, workspace=ws)
    return out.cpu().numpy().astype(np.float64)


# Mode 2 with K % 256 == 0 and 16-byte aligned expert slabs runs the tensor-core mat-mat
# kernel (fp16 operands); mode 1 with K % 128 == 0 and 8-byte aligned slabs the tensor-core
# mat-vec (16-byte copies when K % 256 == 0 and the slabs allow, else 8-byte copies and, for
# K % 256 != 0, a 4-block tail piece).  The padded stride of 2 bytes and K = 96 or 32 keep the
# CUDA-core kernel.  (300, 4, 4, ...) gives every expert about 300 routed rows.
@pytest.mark.parametrize("mode", [0, 1, 2])
@pytest.mark.parametrize("n_tokens,top_k,E,N,K,pad", [(1, 8, 64, 96, 256, 0), (5, 2, 6, 64, 2048, 2),
                                                      (40, 8, 16, 130, 512, 16), (33, 1, 3, 256, 96, 0),
                                                      (3, 4, 9, 70, 4096, 0), (2, 2, 3, 20, 32, 0),
                                                      (300, 4, 4, 160, 768, 0), (3, 2, 5, 40, 384, 0),
                                                      (2, 4, 7, 48, 1408, 8), (1, 3, 4, 33, 128, 8)])
def test_q8_0_parity(mode, n_tokens, top_k, E, N, K, pad):
    x, w, stride, ids = _q8_case(200 + n_tokens, n_tokens, top_k, E, N, K, pad)
    ref = oracle.q8_0_matmul_id(x, w, ids, n_tokens, top_k, N, K, E, stride)
    got = _run_q8(x, w, ids, top_k, N, K, E, stride, mode)
    assert_within_tolerance(got, ref, f"q8_0_matmul_id mode={mode}")


@pytest.mark.parametrize("K", [128, 256])
@pytest.mark.parametrize("mode", [1, 2])
def test_q8_0_invalid_id_gives_zero_row(mode, K):
    n_tokens, top_k, E, N = 300, 4, 8, 64
    x, w, stride, ids = _q8_case(17, n_tokens, top_k, E, N, K)
    ids = ids.copy()
    bad_rows = [5, 100, 101, 700, 1199]
    ids[bad_rows] = 99
    q.device_errors()
    got = _run_q8(x, w, ids, top_k, N, K, E, stride, mode)
    assert np.all(got[bad_rows] == 0.0)
    assert_within_tolerance(got, oracle.q8_0_matmul_id(x, w, ids, n_tokens, top_k, N, K, E, stride), "q8_0 invalid id")
    assert q.device_errors() & 0x2


@pytest.mark.parametrize("n_tokens,mode", [(1, 1), (512, 2)])
def test_q8_0_full_size_sampled(n_tokens, mode):
    E, top_k, N, K = 64, 8, 1408, 2048
    x, w, stride, ids = _q8_case(4600 + n_tokens, n_tokens, top_k, E, N, K)
    got = _run_q8(x, w, ids, top_k, N, K, E, stride, mode)
    assert np.all(np.isfinite(got))
    rows = np.unique(np.concatenate([np.arange(min(8, n_tokens * top_k)),
                                     np.random.default_rng(n_tokens + 7).integers(0, n_tokens * top_k, 24)]))
    ref = oracle.q8_0_matmul_id_rows(x, w, ids, top_k, N, K, E, stride, rows)
    assert_within_tolerance(got[rows], ref, f"q8_0 full n_tokens={n_tokens} mode={mode}")


# The tensor-core mat-mat form of Q8_0 scales each gathered x row by a power of two, as the
# Q4_0 form does: rows far outside fp16's range are served, each held to its own rms.
def test_q8_0_mm_any_f32_row_range():
    n_tokens, top_k, E, N, K = 48, 4, 8, 192, 512
    x, w, stride, ids = _q8_case(4300, n_tokens, top_k, E, N, K)
    x = x.copy()
    gains = np.array([1e6, 1e-6, 1.0, 3e4, 2e-5, 7e7, 1e-30, 5e30], np.float32)
    x *= gains[np.arange(n_tokens) % gains.size][:, None]
    x[5, 17] = 1e9
    assert np.all(np.isfinite(x))
    q.device_errors()
    got = _run_q8(x, w, ids, top_k, N, K, E, stride, 2)
    ref = oracle.q8_0_matmul_id(x, w, ids, n_tokens, top_k, N, K, E, stride)
    assert np.all(np.isfinite(got))
    for r in range(n_tokens * top_k):
        assert_within_tolerance(got[r], ref[r], f"q8_0 routed row {r} (token {r // top_k})")
    assert q.device_errors() == 0


# ---------------------------------------------------------------------------------------
# Weights near the end of fp16's range in the tensor-core mat-mat forms, which form each
# dequantised weight as one fp16 product.  Q4MM_DEVERR_F16_RANGE is raised for every block
# whose d could give a product beyond fp16 (|d| >= 8192 for Q4_0, >= 512 for Q8_0):
#   "edge":     the largest d below that bound with the extreme code: finite, no flag;
#   "flagged":  a d above the bound whose codes all stay finite: flagged, outputs correct;
#   "overflow": a d above the bound with a code beyond fp16: flagged, and only the outputs
#               that block feeds are not finite.
# ---------------------------------------------------------------------------------------

def _set_block(w, stride, K, bbytes, e, n, b, d, qs):
    off = e * stride + (n * (K // 32) + b) * bbytes
    w[off:off + 2] = np.array([d], np.float16).view(np.uint8)
    w[off + 2:off + bbytes] = qs


@pytest.mark.parametrize("bt", ["q4_0", "q8_0"])
@pytest.mark.parametrize("case", ["edge", "flagged", "overflow"])
def test_mm_weight_range(bt, case):
    n_tokens, top_k, E, N, K = 64, 2, 4, 128, 512
    rng = np.random.default_rng(91)
    if bt == "q4_0":
        x, w, stride, ids = _moe_case(4400, n_tokens, top_k, E, N, K)
        # 8 * 8188 = 65504 is fp16's largest finite value; 7 * 9000 = 63000 is finite, 8 * 9000 is not
        d = 8188.0 if case == "edge" else 9000.0
        nib = rng.integers(1, 16, 32).astype(np.uint8)    # q - 8 in [-7, 7]
        if case != "flagged":
            nib[0] = 0                                    # q - 8 = -8
        qs = (nib[:16] | (nib[16:] << 4)).astype(np.uint8)
        bbytes, run, ref_fn = 18, _run, oracle.q4_0_matmul_id
    else:
        x, w, stride, ids = _q8_case(4500, n_tokens, top_k, E, N, K)
        # 128 * 511.75 = 65504; 100 * 600 = 60000 is finite, 127 * 600 is not
        d = 511.75 if case == "edge" else 600.0
        qv = rng.integers(-100, 101, 32)
        if case == "edge":
            qv[7] = -128
        elif case == "overflow":
            qv[7] = 127
        qs = qv.astype(np.int8).view(np.uint8)
        bbytes, run, ref_fn = 34, _run_q8, oracle.q8_0_matmul_id
    w = w.copy()
    e_big, n_big, b_big = 2, 9, 3
    _set_block(w, stride, K, bbytes, e_big, n_big, b_big, d, qs)
    q.device_errors()
    got = run(x, w, ids, top_k, N, K, E, stride, 2)
    err = q.device_errors()
    ref = ref_fn(x, w, ids, n_tokens, top_k, N, K, E, stride)
    fed = np.zeros(got.shape, bool)
    fed[np.nonzero(ids == e_big)[0], n_big] = True
    assert fed.any()
    assert bool(err & 0x4) == (case != "edge")
    if case == "overflow":
        assert not np.any(np.isfinite(got[fed]))
    else:
        assert_within_tolerance(got[fed], ref[fed], f"{bt} outputs of the large weights ({case})")
    assert_within_tolerance(got[~fed], ref[~fed], f"{bt} other outputs ({case})")
