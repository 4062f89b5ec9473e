"""Helpers shared by the GPU parity tests: host arrays <-> device tensors, bf16 readback,
tolerance checks against the oracle."""
import numpy as np
import torch

import oracle
from weight_only_bit_int4_gb300 import synth

DEV = torch.device("cuda:0")

_VIEW = {np.dtype(np.uint16): np.int16, np.dtype(np.uint32): np.int32, np.dtype(np.uint8): np.uint8,
         np.dtype(np.float32): np.float32, np.dtype(np.int32): np.int32}


def dev(a: np.ndarray) -> torch.Tensor:
    a = np.ascontiguousarray(a)
    return torch.from_numpy(a.view(_VIEW[a.dtype])).to(DEV)


def host_u16(t: torch.Tensor) -> np.ndarray:
    return t.cpu().numpy().view(np.uint16)


def bf16_out(t: torch.Tensor) -> np.ndarray:
    return synth.bf16_bits_to_f32(host_u16(t)).astype(np.float64)


def poisoned_bf16(rows: int, cols: int, pattern: int = 0x7FC1) -> torch.Tensor:
    """bf16 output buffer filled with a NaN pattern, so unwritten elements are caught."""
    return torch.full((rows, cols), pattern, dtype=torch.int16, device=DEV)


def assert_within_tolerance(got: np.ndarray, ref: np.ndarray, what: str) -> None:
    tol = oracle.matmul_tolerance(ref)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output (unwritten element?)"
    err = np.abs(got - ref)
    bad = err > tol
    assert not np.any(bad), (f"{what}: {int(bad.sum())} of {bad.size} elements out of tolerance; "
                             f"worst excess {float(np.max(err - tol)):.3g}")
