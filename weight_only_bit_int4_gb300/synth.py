"""Seeded synthetic inputs for the weight-only 4-bit matmuls.

This module holds the input generators that both the CUDA path's tests/bench and the CPU
oracle consume.  It contains none of the method's arithmetic: it draws random numbers,
rounds them to the storage types and lays out raw bytes, nothing else.  Uniform random
nibbles need no packing step: a uniform random 32-bit word *is* eight independent uniform
nibbles, and a uniform random byte is two.

Random numbers come from SplitMix64 in counter form (state_i = seed + (i+1)*0x9E3779B97F4A7C15,
then the SplitMix64 output mix), so every array is a pure function of (seed, stream, size)
and identical on every host.  Normal samples use the Box-Muller transform.

Workload shapes and value distributions follow the pages' workloads:
  * INT4 group-32 affine (quant_fastkernel.rs test `make_case`, scaled to the decode /
    prefill layer shapes): nibbles U{0..15}, scales bf16 U[0.005, 0.02], zero points
    U{0..15}, biases bf16(-zp*scale), x bf16 N(0,1) (prefill: 1% of columns x20).
  * LUT4 (lut4.rs): codebook = 16 sorted N(0,1) samples scaled to max |v| = 1, f32 block
    scales U[0.01, 0.05] per 64 elements, codes U{0..15} two per byte.
  * GGML Q4_0 routed experts (quantized_matmul_id_ggml.rs): d fp16 U[0.005, 0.02], nibble
    bytes U{0..255}, ids = top_k distinct experts per token (partial Fisher-Yates), x f32 N(0,1).
"""
from __future__ import annotations

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def u64(seed: int, stream: int, n: int) -> np.ndarray:
    """n SplitMix64 outputs for (seed, stream); streams give independent sequences."""
    base = np.uint64((seed * 0x100000001B3 + stream * 0x9E3779B1) & 0xFFFFFFFFFFFFFFFF)
    out = np.empty(n, np.uint64)
    with np.errstate(over="ignore"):
        for s in range(0, n, _CHUNK):
            e = min(n, s + _CHUNK)
            i = np.arange(s + 1, e + 1, dtype=np.uint64)
            out[s:e] = _mix(base + i * _GOLDEN)
    return out


def uniform(seed: int, stream: int, n: int) -> np.ndarray:
    """U[0, 1) doubles from the top 53 bits."""
    return (u64(seed, stream, n) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def normal(seed: int, stream: int, n: int) -> np.ndarray:
    """N(0, 1) doubles by Box-Muller over pairs of uniforms."""
    half = (n + 1) // 2
    u = uniform(seed, stream, 2 * half)
    r = np.sqrt(-2.0 * np.log1p(-u[:half]))
    t = 2.0 * np.pi * u[half:]
    z = np.empty(2 * half, np.float64)
    z[0::2] = r * np.cos(t)
    z[1::2] = r * np.sin(t)
    return z[:n]


def to_bf16_bits(a) -> np.ndarray:
    """Round to bfloat16 (nearest, ties to even) and return the uint16 bit patterns."""
    f = np.ascontiguousarray(a, np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    u = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return u.astype(np.uint16).reshape(f.shape)


def bf16_bits_to_f32(b) -> np.ndarray:
    return (np.ascontiguousarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32)


# --------------------------------------------------------------------------------------
# INT4 group-32 affine MatMulNBits
# --------------------------------------------------------------------------------------

def int4_weights(seed: int, N: int, K: int):
    """(w uint32 [N, K/8], scales bf16-bits [N, K/32], biases bf16-bits [N, K/32])."""
    assert K % 32 == 0
    w = (u64(seed, 1, N * (K // 8)) >> np.uint64(32)).astype(np.uint32).reshape(N, K // 8)
    G = N * (K // 32)
    s = to_bf16_bits(0.005 + 0.015 * uniform(seed, 2, G)).reshape(N, K // 32)
    zp = (u64(seed, 3, G) >> np.uint64(60)).astype(np.float32).reshape(N, K // 32)
    b = to_bf16_bits(-zp * bf16_bits_to_f32(s))
    return w, s, b


def activations_bf16(seed: int, M: int, K: int, outlier_frac: float = 0.0,
                     outlier_scale: float = 20.0) -> np.ndarray:
    """x bf16-bits [M, K] ~ N(0,1); a fixed random `outlier_frac` of columns scaled up."""
    x = normal(seed, 4, M * K).reshape(M, K)
    if outlier_frac > 0.0:
        n_out = max(1, int(round(outlier_frac * K)))
        order = np.argsort(u64(seed, 5, K), kind="stable")
        x[:, order[:n_out]] *= outlier_scale
    return to_bf16_bits(x)


# --------------------------------------------------------------------------------------
# LUT4 frozen-codebook blocked 4-bit
# --------------------------------------------------------------------------------------

def lut4_book(seed: int) -> np.ndarray:
    v = np.sort(normal(seed, 6, 16))
    return (v / np.max(np.abs(v))).astype(np.float32)


def lut4_weights(seed: int, rows: int, cols: int, block: int = 64):
    """(packed uint8 [ceil(rows*cols/2)], scales f32 [ceil(rows*cols/block)], book f32[16])."""
    total = rows * cols
    packed = (u64(seed, 7, (total + 1) // 2) >> np.uint64(56)).astype(np.uint8)
    nblk = -(-total // block)
    scales = (0.01 + 0.04 * uniform(seed, 8, nblk)).astype(np.float32)
    return packed, scales, lut4_book(seed)


# --------------------------------------------------------------------------------------
# GGML Q4_0 expert-routed MoE
# --------------------------------------------------------------------------------------

Q4_0_BLOCK_BYTES = 18


def q4_0_experts(seed: int, n_experts: int, N: int, K: int, expert_stride: int | None = None):
    """(w uint8 [n_experts * expert_stride], expert_stride): each 18-byte block holds an
    fp16 d ~ U[0.005, 0.02] (little endian) followed by 16 uniform random bytes."""
    assert K % 32 == 0
    per_expert = N * (K // 32) * Q4_0_BLOCK_BYTES
    stride = per_expert if expert_stride is None else expert_stride
    assert stride >= per_expert
    nblk = n_experts * N * (K // 32)
    blocks = np.empty((nblk, Q4_0_BLOCK_BYTES), np.uint8)
    d = (0.005 + 0.015 * uniform(seed, 9, nblk)).astype(np.float16).view(np.uint8).reshape(nblk, 2)
    blocks[:, 0:2] = d
    blocks[:, 2:] = (u64(seed, 10, nblk * 16) >> np.uint64(56)).astype(np.uint8).reshape(nblk, 16)
    w = np.zeros(n_experts * stride, np.uint8)
    per = blocks.reshape(n_experts, per_expert)
    for e in range(n_experts):
        w[e * stride:e * stride + per_expert] = per[e]
    return w, stride


Q8_0_BLOCK_BYTES = 34


def q8_0_experts(seed: int, n_experts: int, N: int, K: int, expert_stride: int | None = None):
    """(w uint8 [n_experts * expert_stride], expert_stride): each 34-byte block holds an
    fp16 d ~ U[0.005, 0.02] (little endian) followed by 32 uniform random bytes (signed
    integers -128..127)."""
    assert K % 32 == 0
    per_expert = N * (K // 32) * Q8_0_BLOCK_BYTES
    stride = per_expert if expert_stride is None else expert_stride
    assert stride >= per_expert
    nblk = n_experts * N * (K // 32)
    blocks = np.empty((nblk, Q8_0_BLOCK_BYTES), np.uint8)
    d = (0.005 + 0.015 * uniform(seed, 13, nblk)).astype(np.float16).view(np.uint8).reshape(nblk, 2)
    blocks[:, 0:2] = d
    blocks[:, 2:] = (u64(seed, 14, nblk * 32) >> np.uint64(56)).astype(np.uint8).reshape(nblk, 32)
    w = np.zeros(n_experts * stride, np.uint8)
    per = blocks.reshape(n_experts, per_expert)
    for e in range(n_experts):
        w[e * stride:e * stride + per_expert] = per[e]
    return w, stride


def routing_ids(seed: int, n_tokens: int, top_k: int, n_experts: int) -> np.ndarray:
    """ids uint32 [n_tokens * top_k]: top_k distinct experts per token, uniform."""
    assert top_k <= n_experts
    r = u64(seed, 11, n_tokens * top_k)
    ids = np.empty(n_tokens * top_k, np.uint32)
    for t in range(n_tokens):
        perm = list(range(n_experts))
        for s in range(top_k):
            j = s + int(r[t * top_k + s] % np.uint64(n_experts - s))
            perm[s], perm[j] = perm[j], perm[s]
            ids[t * top_k + s] = perm[s]
    return ids


def activations_f32(seed: int, n: int, K: int) -> np.ndarray:
    return normal(seed, 12, n * K).astype(np.float32).reshape(n, K)
