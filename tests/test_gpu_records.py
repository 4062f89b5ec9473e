"""Dispatch records (q4_gemv_record, q4_0_matmul_id_mv_record): a replayed record launches
the kernel the direct call launches, so outputs are bit-identical, also inside CUDA graphs."""
import numpy as np
import pytest
import torch

import oracle
import weight_only_bit_int4_gb300 as q
from weight_only_bit_int4_gb300 import synth

from gpu_util import DEV, assert_within_tolerance, bf16_out, dev, host_u16, poisoned_bf16

pytestmark = pytest.mark.gpu


# ks (M <= 4, K % 256 == 0), gc (K % 128 == 0 only), async (M > 4) and the register-prefetch
# kernel (K % 128 != 0), with and without the static-weights flag.
@pytest.mark.parametrize("static_weights", [False, True])
@pytest.mark.parametrize("M,N,K", [(1, 4096, 4096), (4, 1000, 384), (16, 256, 512), (3, 1000, 2080),
                                   (2, 304, 1024), (9, 130, 1024)])
def test_gemv_record_matches_direct_call(M, N, K, static_weights):
    w, s, b = synth.int4_weights(40 + M, N, K)
    x = synth.activations_bf16(41 + M, M, K)
    W = (dev(w), dev(s), dev(b))
    y0, y1 = poisoned_bf16(M, N), poisoned_bf16(M, N)
    q.q4_gemv(dev(x), *W, y0, static_weights=static_weights)
    rec = q.q4_gemv_record(M, N, K, static_weights=static_weights)
    rec.gemv(dev(x), *W, y1)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(host_u16(y0), host_u16(y1))
    assert_within_tolerance(bf16_out(y1), oracle.q4_matmul(x, w, s, b, M, N, K), "record")
    rec.close()


def test_gemv_record_launch_n_matches_single_replays():
    """The batched replay launches each record's kernel in order on one stream: outputs
    bit-identical to one replay per record, including a chain where a later call reads an
    earlier call's y as its x."""
    shapes = [(1, 4096, 4096), (4, 1000, 384), (16, 256, 512), (3, 1000, 2080), (16, 512, 1000 // 32 * 32)]
    recs, args_b, args_1, outs_b, outs_1 = [], [], [], [], []
    for i, (M, N, K) in enumerate(shapes):
        w, s, b = synth.int4_weights(90 + i, N, K)
        x = dev(synth.activations_bf16(91 + i, M, K))
        W = (dev(w), dev(s), dev(b))
        recs.append(q.q4_gemv_record(M, N, K, static_weights=(i % 2 == 0)))
        yb, y1 = poisoned_bf16(M, N), poisoned_bf16(M, N)
        args_b.append((x, *W, yb))
        args_1.append((x, *W, y1))
        outs_b.append(yb)
        outs_1.append(y1)
    # chain: the last shape's x is the previous shape's y (M = 16, K = 512 -> N = 256 ... ) where
    # the shapes allow it: shape 2 has M = 16, N = 256; feed its y to a record of K = 256
    w, s, b = synth.int4_weights(99, 128, 256)
    W = (dev(w), dev(s), dev(b))
    recs.append(q.q4_gemv_record(16, 128, 256, static_weights=True))
    yb, y1 = poisoned_bf16(16, 128), poisoned_bf16(16, 128)
    args_b.append((outs_b[2], *W, yb))
    args_1.append((outs_1[2], *W, y1))
    outs_b.append(yb)
    outs_1.append(y1)
    q.q4_gemv_record_launch_n(recs, *[list(a) for a in zip(*args_b)])
    for r, a in zip(recs, args_1):
        r.gemv(*a)
    torch.cuda.synchronize()
    for yb, y1 in zip(outs_b, outs_1):
        np.testing.assert_array_equal(host_u16(yb), host_u16(y1))
    for r in recs:
        r.close()


def test_gemv_record_survives_smaller_plans_of_the_same_kernel():
    """Several shapes share one decode kernel with different shared-memory sizes.  A record
    planned for the largest must still launch after smaller shapes of the same kernel were
    recorded and called (the kernel's shared-memory limit is only ever raised)."""
    shapes = [(4, 14336, 4096), (4, 4096, 4096), (1, 4096, 4096)]   # (M, N, K), largest first
    data = {}
    for M, N, K in shapes:
        w, s, b = synth.int4_weights(770 + M + N // 1024, N, K)
        x = synth.activations_bf16(771 + M, M, K)
        data[(M, N, K)] = (x, (dev(w), dev(s), dev(b)))
    recs = [q.q4_gemv_record(M, N, K, static_weights=True) for M, N, K in shapes]
    for M, N, K in shapes[1:]:
        x, W = data[(M, N, K)]
        q.q4_gemv(dev(x), *W, poisoned_bf16(M, N))
    for rec, (M, N, K) in zip(recs, shapes):
        x, W = data[(M, N, K)]
        y0, y1 = poisoned_bf16(M, N), poisoned_bf16(M, N)
        rec.gemv(dev(x), *W, y1)
        q.q4_gemv(dev(x), *W, y0, static_weights=True)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(host_u16(y0), host_u16(y1))
        rec.close()


def test_gemv_records_chain_in_a_graph():
    """A decode chain of recorded calls (x -> y -> next x), captured into a CUDA graph on its
    first replay, gives the bits of the same chain of direct calls."""
    M, D, layers = 4, 1024, 5
    sets = [tuple(dev(a) for a in synth.int4_weights(750 + i, D, D)) for i in range(2)]
    x0 = dev(synth.activations_bf16(760, M, D))

    def run(use_rec, graph):
        bufs = [poisoned_bf16(M, D) for _ in range(layers + 1)]
        bufs[0].copy_(x0)
        rec = q.q4_gemv_record(M, D, D, static_weights=True)

        def calls():
            for i in range(layers):
                if use_rec:
                    rec.gemv(bufs[i], *sets[i % 2], bufs[i + 1])
                else:
                    q.q4_gemv(bufs[i], *sets[i % 2], bufs[i + 1], static_weights=True)

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
        return [host_u16(b_).copy() for b_ in bufs]

    direct = run(False, False)
    for out in (run(True, False), run(True, True)):
        for a, b_ in zip(direct, out):
            np.testing.assert_array_equal(a, b_)


def _moe(seed, n_tokens, top_k, E, N, K, pad=0):
    w, stride = synth.q4_0_experts(seed, E, N, K, expert_stride=N * (K // 32) * 18 + pad)
    ids = synth.routing_ids(seed + 1, n_tokens, top_k, E)
    return w, stride, ids


# 16-byte and 8-byte weight copies on the tensor cores, and the fp32 kernel (K = 96).
@pytest.mark.parametrize("n_tokens,top_k,E,N,K", [(1, 8, 64, 1408, 2048), (2, 4, 9, 200, 1408), (3, 2, 5, 40, 96)])
def test_mv_record_matches_direct_call(n_tokens, top_k, E, N, K):
    w, stride, ids = _moe(90 + K, n_tokens, top_k, E, N, K)
    x = synth.activations_f32(91, n_tokens, K)
    wd, idd, xd = dev(w), dev(ids), dev(x)
    out0 = torch.full((n_tokens * top_k, N), float("nan"), dtype=torch.float32, device=DEV)
    out1 = torch.full_like(out0, float("nan"))
    q.q4_0_matmul_id(xd, wd, idd, out0, top_k, N, K, E, stride, mode=1)
    rec = q.q4_0_matmul_id_mv_record(n_tokens, top_k, N, K, E, stride)
    rec.matmul_id_mv(xd, wd, idd, out1)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(out0.cpu().numpy(), out1.cpu().numpy())


@pytest.mark.parametrize("n_tokens,top_k,E,N,K", [(1, 8, 64, 2048, 1408), (2, 3, 7, 96, 256)])
def test_swiglu_record_matches_direct_call(n_tokens, top_k, E, N, K):
    w, stride, ids = _moe(95 + K, n_tokens, top_k, E, N, K)
    gate = dev(synth.activations_f32(96, n_tokens * top_k, K))
    up = dev(synth.activations_f32(97, n_tokens * top_k, K))
    wd, idd = dev(w), dev(ids)
    out0 = torch.full((n_tokens * top_k, N), float("nan"), dtype=torch.float32, device=DEV)
    out1 = torch.full_like(out0, float("nan"))
    q.q4_0_matmul_id_swiglu(gate, up, wd, idd, out0, top_k, N, K, E, stride)
    rec = q.q4_0_matmul_id_mv_record(n_tokens, top_k, N, K, E, stride, swiglu=True)
    st = torch.cuda.Stream()
    st.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=st):   # first replay inside a capture
        rec.matmul_id_mv(gate, wd, idd, out1, up=up)
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    np.testing.assert_array_equal(out0.cpu().numpy(), out1.cpu().numpy())


def test_record_rejects_misuse():
    N, K, E, top_k = 64, 256, 4, 2
    w, stride, ids = _moe(99, 1, top_k, E, N, K)
    rec = q.q4_0_matmul_id_mv_record(1, top_k, N, K, E, stride)
    wd = dev(np.concatenate([np.zeros(8, np.uint8), w]))
    x = dev(synth.activations_f32(98, 1, K))
    out = torch.empty((top_k, N), dtype=torch.float32, device=DEV)
    with pytest.raises(q.Q4MMError) as ei:   # planned for 16-byte aligned weights
        rec.matmul_id_mv(x, wd[8:], dev(ids), out)
    assert ei.value.status == 2
    with pytest.raises(q.Q4MMError) as ei:   # a plain mat-vec record takes no up operand
        rec.matmul_id_mv(x, wd[:w.size], dev(ids), out, up=x)
    assert ei.value.status == 1
    grec = q.q4_gemv_record(1, N, K)
    # a decode record is not a mat-vec record
    idd = dev(ids)
    assert q.lib().q4_0_matmul_id_mv_record_launch(grec._h, x.data_ptr(), None, wd.data_ptr(), idd.data_ptr(),
                                                   out.data_ptr(), None) == 1
    rec.close()
    grec.close()
