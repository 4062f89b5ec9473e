"""The allocation-free Q4_0 mat-mat entry point (q4_0_matmul_id_noalloc), called through the
C ABI, against the workspace entry point (q4_0_matmul_id, mode 2) on the same inputs.

It exists for callers that cannot allocate device memory when they call the library
(allocator-free serving loops, hosts that own all device buffers); it uses the library's
fixed scratch array instead of a caller workspace.  Two calls
in a row with different sizes check that nothing depends on what the previous call left in
the shared array."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import weight_only_bit_int4_gb300 as q
from weight_only_bit_int4_gb300 import _lib, synth

from gpu_util import DEV, assert_within_tolerance, dev

pytestmark = pytest.mark.gpu


def _call_noalloc(x, w, ids, out, top_k, N, K, E, stride):
    L = _lib.lib()
    return L.q4_0_matmul_id_noalloc(x.data_ptr(), w.data_ptr(), ids.data_ptr(), out.data_ptr(), x.shape[0],
                                    top_k, N, K, E, stride, torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("K", [512, 288])
def test_noalloc_matches_workspace_entry_point_on_two_calls(K):
    # K = 512 runs the tensor-core mat-mat kernel; K = 288 (K % 256 != 0) the CUDA-core kernel
    # over the routed order.  Both read their routing lists from the fixed array.
    E, top_k, N = 16, 8, 256
    for n_tokens, seed in ((64, 501), (40, 502)):
        w, stride = synth.q4_0_experts(seed, E, N, K)
        ids = synth.routing_ids(seed + 1, n_tokens, top_k, E)
        x = synth.activations_f32(seed + 2, n_tokens, K)
        xd, wd, idd = dev(x), dev(w), dev(ids)
        ws = torch.empty(q.q4_0_matmul_id_workspace_size(n_tokens, top_k, N, K, E), dtype=torch.uint8, device=DEV)
        ref = torch.full((n_tokens * top_k, N), float("nan"), dtype=torch.float32, device=DEV)
        q.q4_0_matmul_id(xd, wd, idd, ref, top_k, N, K, E, stride, mode=2, workspace=ws)
        out = torch.full((n_tokens * top_k, N), float("nan"), dtype=torch.float32, device=DEV)
        assert _call_noalloc(xd, wd, idd, out, top_k, N, K, E, stride) == 0
        torch.cuda.synchronize()
        ref_h = ref.cpu().numpy().astype(np.float64)
        got = out.cpu().numpy().astype(np.float64)
        assert np.all(np.isfinite(got))
        # the same kernels on the same inputs: bit for bit, so stale scratch would show
        np.testing.assert_array_equal(got, ref_h, err_msg=f"noalloc vs workspace entry, n_tokens={n_tokens}")
        assert_within_tolerance(got, ref_h, f"noalloc vs workspace entry, n_tokens={n_tokens}")
        # and both against the oracle on a few rows
        rows = np.arange(0, n_tokens * top_k, 37)
        o = oracle.q4_0_matmul_id_rows(x, w, ids, top_k, N, K, E, stride, rows)
        assert_within_tolerance(got[rows], o, "noalloc vs oracle")


def test_noalloc_rejects_requests_beyond_its_array():
    limit = (32 * 1024 * 1024)
    n_tokens, top_k, N, K, E = 4096, 8, 1408, 2048, 64      # needs ~134 MB of scratch
    assert q.q4_0_matmul_id_workspace_size(n_tokens, top_k, N, K, E) > limit
    L = _lib.lib()
    fake = 1 << 20
    st = L.q4_0_matmul_id_noalloc(fake, fake, fake, fake, n_tokens, top_k, N, K, E, N * (K // 32) * 18, None)
    assert st == 3   # Q4MM_ERR_WORKSPACE, nothing launched
