"""Planted mistakes in the oracle must each fail a pin.

Each case copies oracle/q4_oracle.c into a temporary directory, plants one plausible
mistake (a swapped nibble order, a wrong sign, an off-by-one index, a dropped term, the
wrong rounding rule), compiles the copy and runs tests/test_oracle_pins.py against it
(Q4MM_ORACLE_LIB).  pytest must report failed tests (exit status 1): the pins check the
oracle's arithmetic against outside references, not the oracle against itself.  The
unmodified source, built the same way, must pass.  No GPU is involved.
"""
import os
import subprocess
import sys

import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
PINS = os.path.join(HERE, "test_oracle_pins.py")

# name -> (text in q4_oracle.c, replacement); each text occurs exactly once.
MUTATIONS = {
    "int4 nibble order reversed": (
        "return (word >> (4 * (k % 8))) & 0xFu;",
        "return (word >> (4 * (7 - k % 8))) & 0xFu;"),
    "int4 bias subtracted": (
        "oracle_bf16_to_f32(b[g]));\n}",
        "-oracle_bf16_to_f32(b[g]));\n}"),
    "int4 group index over 64 columns": (
        "int64_t g = n * (K / 32) + k / 32;\n    return fmaf",
        "int64_t g = n * (K / 32) + k / 64;\n    return fmaf"),
    "int4 matmul drops the last k": (
        "for (int64_t k = 0; k < K; ++k)\n                acc += (double)oracle_bf16_to_f32(x[m * K + k]) *\n"
        "                       (double)q4_value",
        "for (int64_t k = 0; k < K - 1; ++k)\n                acc += (double)oracle_bf16_to_f32(x[m * K + k]) *\n"
        "                       (double)q4_value"),
    "bf16 rounding ties away from zero": (
        "double r = rint(v / ulp) * ulp;\n    if (fabs(r) >= ldexp(1.0, 128))",
        "double r = round(v / ulp) * ulp;\n    if (fabs(r) >= ldexp(1.0, 128))"),
    "f16 subnormal ulp halved": (
        "e = -14;                      /* subnormal range: fixed ulp 2^-24 */",
        "e = -15;                      /* subnormal range: fixed ulp 2^-24 */"),
    "lut4 nibble order swapped": (
        "(f % 2 == 0) ? (uint32_t)(byte >> 4) : (uint32_t)(byte & 15);",
        "(f % 2 == 0) ? (uint32_t)(byte & 15) : (uint32_t)(byte >> 4);"),
    "lut4 scale index off by one": (
        "book[code] * scales[f / block];",
        "book[code] * scales[(f + 1) / block];"),
    "lut4 transposes swapped": (
        "return transpose ? n * K + k : k * N + n;",
        "return transpose ? k * N + n : n * K + k;"),
    "lut4 rounding types swapped": (
        "if (rounding == 1)\n        v = oracle_f16_to_f32",
        "if (rounding == 2)\n        v = oracle_f16_to_f32"),
    "lut4 f16 rounding dropped": (
        "v = oracle_f16_to_f32(oracle_f32_to_f16(v));",
        "v = v;"),
    "q4_0 d read big endian": (
        "oracle_f16_to_f32((uint16_t)(blk[0] | (blk[1] << 8)));\n    int64_t j = k % 32;",
        "oracle_f16_to_f32((uint16_t)(blk[1] | (blk[0] << 8)));\n    int64_t j = k % 32;"),
    "q8_0 d read big endian": (
        "oracle_f16_to_f32((uint16_t)(blk[0] | (blk[1] << 8)));\n    int q = (int)blk[2 + k % 32];",
        "oracle_f16_to_f32((uint16_t)(blk[1] | (blk[0] << 8)));\n    int q = (int)blk[2 + k % 32];"),
    "silu is the bare sigmoid": (
        "return z / (1.0 + exp(-z));",
        "return 1.0 / (1.0 + exp(-z));"),
    "q4_0 nibble halves swapped": (
        "(j < 16) ? (blk[2 + j] & 15) : (blk[2 + j - 16] >> 4);",
        "(j < 16) ? (blk[2 + j] >> 4) : (blk[2 + j - 16] & 15);"),
    "q4_0 offset 7 instead of 8": (
        "return (float)(q - 8) * d;",
        "return (float)(q - 7) * d;"),
    "q4_0 token row slot-major": (
        "q4_0_one_row(x, w, ids[r], r / top_k, N, K, n_experts, expert_stride, out + r * N);",
        "q4_0_one_row(x, w, ids[r], r % n_tokens, N, K, n_experts, expert_stride, out + r * N);"),
    "silu sign flipped": (
        "return z / (1.0 + exp(-z));",
        "return z / (1.0 + exp(z));"),
    "swiglu gate and up swapped": (
        "double h = silu((double)gate[r * K + k]) * (double)up[r * K + k];",
        "double h = silu((double)up[r * K + k]) * (double)gate[r * K + k];"),
    "lut4 sampled form swaps m and n": (
        "x[mi[i] * K + k]) *\n                   (double)lut4_value_at(packed, scales, book,\n"
        "                                         lut4_flat(ni[i], k, N, K, transpose), block);",
        "x[ni[i] * K + k]) *\n                   (double)lut4_value_at(packed, scales, book,\n"
        "                                         lut4_flat(mi[i], k, N, K, transpose), block);"),
    "q4_0 routed-row form reads the routed row as the token": (
        "q4_0_one_row(x, w, ids[rows[i]], rows[i] / top_k, N, K, n_experts, expert_stride,",
        "q4_0_one_row(x, w, ids[rows[i]], rows[i], N, K, n_experts, expert_stride,"),
    "q8_0 bytes read as unsigned": (
        "    if (q >= 128)\n        q -= 256;                    /* the byte is a signed integer */\n",
        ""),
    "q8_0 block stride 32 bytes": (
        "const uint8_t *blk = row + (k / 32) * 34;",
        "const uint8_t *blk = row + (k / 32) * 32;"),
    "q8_0 routed-row form reads the routed row as the token": (
        "q8_0_one_row(x, w, ids[rows[i]], rows[i] / top_k, N, K, n_experts, expert_stride,",
        "q8_0_one_row(x, w, ids[rows[i]], rows[i], N, K, n_experts, expert_stride,"),
    "route lists descending": (
        "for (int64_t r = 0; r < n_rows; ++r)\n            if ((int64_t)ids[r] == e) {",
        "for (int64_t r = n_rows - 1; r >= 0; --r)\n            if ((int64_t)ids[r] == e) {"),
    "route invalid count misses id == n_experts": (
        "if ((int64_t)ids[r] >= n_experts)\n            ++bad;",
        "if ((int64_t)ids[r] > n_experts)\n            ++bad;"),
}


def _run_pins(src_text, tmp_path):
    src = tmp_path / "q4_oracle.c"
    src.write_text(src_text)
    so = tmp_path / "liboracle_q4.so"
    subprocess.check_call(["gcc", *oracle.CFLAGS, "-o", str(so), str(src), "-lm"])
    env = dict(os.environ, Q4MM_ORACLE_LIB=str(so))
    return subprocess.run([sys.executable, "-m", "pytest", PINS, "-x", "-q", "-p", "no:cacheprovider"],
                          cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)


def _source():
    with open(os.path.join(ROOT, "oracle", "q4_oracle.c")) as f:
        return f.read()


def test_unmodified_copy_passes_the_pins(tmp_path):
    r = _run_pins(_source(), tmp_path)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_fails_a_pin(name, tmp_path):
    old, new = MUTATIONS[name]
    src = _source()
    assert src.count(old) == 1, f"mutation site for {name!r} not unique or missing"
    r = _run_pins(src.replace(old, new), tmp_path)
    # 1 = some tests failed (not a crash, a collection error or an interrupted run)
    assert r.returncode == 1, f"{name}: pins exit status {r.returncode}\n" + r.stdout[-3000:]
