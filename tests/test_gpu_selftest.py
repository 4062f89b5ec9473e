"""The bounded pipeline waits give up cleanly: a self-test kernel waits on a barrier that
nothing completes, with a short limit.  It must record Q4MM_DEVERR_WAIT_TIMEOUT, leave
without a fault (its in-flight copy lands first), and the calls after it must be correct."""
import numpy as np
import pytest
import torch

import oracle
import weight_only_bit_int4_gb300 as q
from weight_only_bit_int4_gb300 import _lib, synth

from gpu_util import DEV, assert_within_tolerance, bf16_out, dev, poisoned_bf16

pytestmark = pytest.mark.gpu


def test_bounded_wait_gives_up_and_later_calls_are_correct():
    L = _lib.lib()
    q.device_errors()                                   # start from a clear error word
    src = torch.arange(4, dtype=torch.int32, device=DEV)
    stream = torch.cuda.current_stream().cuda_stream
    assert L.q4mm_selftest_wait_timeout(src.data_ptr(), 1_000_000, stream) == 0   # 1 ms limit
    assert q.device_errors() & 0x1                      # Q4MM_DEVERR_WAIT_TIMEOUT, then cleared
    # argument checks: no pointer, a zero or too long limit, a misaligned source
    assert L.q4mm_selftest_wait_timeout(None, 1000, stream) == 1
    assert L.q4mm_selftest_wait_timeout(src.data_ptr(), 0, stream) == 1
    assert L.q4mm_selftest_wait_timeout(src.data_ptr(), 2_000_000_000, stream) == 1
    assert L.q4mm_selftest_wait_timeout(src.data_ptr() + 4, 1000, stream) == 2
    # the context is intact: the pipelined kernels (decode, tensor-core GEMM) run correctly
    M, N, K = 16, 256, 512
    w, s, b = synth.int4_weights(1000, N, K)
    x = synth.activations_bf16(1001, M, K)
    ref = oracle.q4_matmul(x, w, s, b, M, N, K)
    for fn in (q.q4_gemv, q.q4_gemm):
        y = poisoned_bf16(M, N)
        fn(dev(x), dev(w), dev(s), dev(b), y)
        assert_within_tolerance(bf16_out(y), ref, f"{fn.__name__} after the self-test")
    assert q.device_errors() == 0
