"""Calls on different streams, issued from different host threads, share no hidden state:
every output is bit-identical to the same call made alone.  (The allocation-free entry
point's scratch array is the one documented exception and is not used here.)"""
import threading

import numpy as np
import pytest
import torch

import weight_only_bit_int4_gb300 as q
from weight_only_bit_int4_gb300 import synth

from gpu_util import DEV, dev, host_u16

pytestmark = pytest.mark.gpu


def _int4(seed, M, N, K):
    w, s, b = synth.int4_weights(seed, N, K)
    return dev(synth.activations_bf16(seed + 1, M, K)), (dev(w), dev(s), dev(b))


def _moe(seed, n_tokens, top_k, E, N, K):
    w, stride = synth.q4_0_experts(seed, E, N, K)
    ids = synth.routing_ids(seed + 1, n_tokens, top_k, E)
    x = synth.activations_f32(seed + 2, n_tokens, K)
    ws = torch.empty(q.q4_0_matmul_id_workspace_size(n_tokens, top_k, N, K, E), dtype=torch.uint8, device=DEV)
    return dev(x), dev(w), dev(ids), stride, ws


def test_two_streams_two_threads_match_solo_calls():
    # decode GEMV (K split in the CTA), LUT4 and INT4 prefill GEMMs, routed mat-mat calls with
    # their own workspaces.  Each worker thread's first call is the first CUDA work of that
    # thread (the GEMMs encode tensor maps, which needs the context current).
    x1, W1 = _int4(1100, 4, 4096, 4096)
    x2, W2 = _int4(1200, 300, 2048, 1024)
    mx, mw, mids, stride, ws = _moe(1300, 64, 8, 16, 256, 512)
    mx2, mw2, mids2, stride2, ws2 = _moe(1400, 48, 4, 8, 128, 1024)

    def gemv(y):
        for _ in range(20):
            q.q4_gemv(x1, *W1, y)

    def gemm(y):
        for _ in range(5):
            q.q4_gemm(x2, *W2, y)

    def mm(out):
        for _ in range(5):
            q.q4_0_matmul_id(mx, mw, mids, out, 8, 256, 512, 16, stride, mode=2, workspace=ws)

    def mm2(out):
        for _ in range(5):
            q.q4_0_matmul_id(mx2, mw2, mids2, out, 4, 128, 1024, 8, stride2, mode=2, workspace=ws2)

    packed, lsc, book = synth.lut4_weights(1500, 1024, 2048, 64)
    lx, lp, ls = dev(synth.activations_bf16(1501, 96, 2048)), dev(packed), dev(lsc)

    def lut4(y):
        for _ in range(5):
            q.lut4_matmul(lx, lp, ls, book, y, 1024, 2048, 64, 1)

    # worker 0 takes jobs 0, 2, 4 and worker 1 jobs 1, 3: both start with a tensor-map GEMM
    jobs = [(gemm, lambda: torch.empty((300, 2048), dtype=torch.int16, device=DEV)),
            (lut4, lambda: torch.empty((96, 1024), dtype=torch.int16, device=DEV)),
            (gemv, lambda: torch.empty((4, 4096), dtype=torch.int16, device=DEV)),
            (mm, lambda: torch.empty((512, 256), dtype=torch.float32, device=DEV)),
            (mm2, lambda: torch.empty((192, 128), dtype=torch.float32, device=DEV))]

    solo = []
    for fn, alloc in jobs:
        out = alloc()
        fn(out)
        torch.cuda.synchronize()
        solo.append(out.clone())

    outs = [alloc() for _, alloc in jobs]
    streams = [torch.cuda.Stream() for _ in range(2)]
    errors = []

    def worker(idx):
        try:
            with torch.cuda.stream(streams[idx]):
                for j in range(idx, len(jobs), 2):
                    jobs[j][0](outs[j])
            streams[idx].synchronize()
        except Exception as e:   # surfaced below
            errors.append(e)

    torch.cuda.synchronize()
    threads = [threading.Thread(target=worker, args=(i,)) for i in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    torch.cuda.synchronize()
    for a, b in zip(solo, outs):
        if a.dtype == torch.int16:
            np.testing.assert_array_equal(host_u16(a), host_u16(b))
        else:
            np.testing.assert_array_equal(a.cpu().numpy(), b.cpu().numpy())
