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
                                                      (3, 4, 9, 70, 4096, 0)])
def test_moe_parity(mode, n_tokens, top_k, E, N, K, pad):
    x, w, stride, ids = _moe_case(100 + n_tokens, n_tokens, top_k, E, N, K, pad)
    ref = oracle.q4_0_matmul_id(x, w, ids, n_tokens, top_k, N, K, E, stride)
    got = _run(x, w, ids, top_k, N, K, E, stride, mode)
    assert_within_tolerance(got, ref, f"q4_0_matmul_id mode={mode}")


# Invalid ids in one 32-row chunk, in chunks zeroed by different CTAs, and in an id count
# large enough for the single-CTA routing form.
@pytest.mark.parametrize("mode", [1, 2])
@pytest.mark.parametrize("n_tokens,top_k,E,bad_rows", [(6, 2, 4, [5]), (300, 4, 8, [5, 100, 101, 700, 1199]),
                                                       (1600, 8, 8, [0, 4000, 12799])])
def test_moe_invalid_id_gives_zero_row(mode, n_tokens, top_k, E, bad_rows):
    N, K = 64, 128
    x, w, stride, ids = _moe_case(7, n_tokens, top_k, E, N, K)
    ids = ids.copy()
    ids[bad_rows] = 99
    ref = oracle.q4_0_matmul_id(x, w, ids, n_tokens, top_k, N, K, E, stride)
    got = _run(x, w, ids, top_k, N, K, E, stride, mode)
    assert np.all(got[bad_rows] == 0.0)
    assert_within_tolerance(got, ref, "invalid id")
    assert q.device_errors() & 0x2


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
