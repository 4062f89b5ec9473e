// dequant.cu -- standalone INT4 group-32 affine dequant (q4_dequant).
//
// quant_fastkernel.rs (onnxruntime-ep-mlx 0.27.4), kernel W-tile dequant: value =
// nibble * scale + bias with the nibble of element k at bits 4*(k%8) of word k/8.  Here the
// value is formed in fp32 with one fused multiply-add, so an F32 output is bit-identical to
// fmaf(q, s, b); BF16/F16 outputs round that value to nearest even.  lut4.rs uses the same
// decode-then-GEMM pattern (its lookup4 decode kernel) for large M.
//
// Roofline: HBM-bound.  Per 32-element group: 16 B codes + 4 B scale/bias read, 32 * out
// bytes written.
#include "q4mm_internal.cuh"

namespace q4mm {
namespace {

// A thread decodes one 32-bit word (8 elements of one group) per step, so consecutive lanes
// read consecutive 4-byte words and write consecutive 16-byte (bf16 / f16) or 32-byte (f32)
// pieces: every load and store of a warp is one contiguous run.  The code becomes a float
// exactly through the exponent trick (0x4B000000 | q is 2^23 + q), and one fmaf per element
// forms q * s + b.
template <int OUT>   // 0 = f32, 1 = bf16, 2 = f16
__global__ void __launch_bounds__(256) q4_dequant_kernel(const uint32_t *__restrict__ w,
                                                         const uint16_t *__restrict__ scales,
                                                         const uint16_t *__restrict__ biases,
                                                         int64_t words, void *__restrict__ out) {
  constexpr int kU = 4;   // words per thread per step, a warp-width apart
  const int64_t stride = (int64_t)gridDim.x * blockDim.x * kU;
  const int64_t lane0 = (int64_t)blockIdx.x * blockDim.x * kU + (threadIdx.x / 32) * 32 * kU + threadIdx.x % 32;
  for (int64_t base = lane0; base < words; base += stride) {
    uint32_t q[kU];
    float s[kU], b[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int64_t i = base + 32 * u;
      if (i < words) {
        q[u] = __ldg(w + i);
        s[u] = bf16_bits_to_float(ldg_u16(scales + i / 4));
        b[u] = bf16_bits_to_float(ldg_u16(biases + i / 4));
      }
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int64_t i = base + 32 * u;
      if (i >= words) break;
      float v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float qf = __uint_as_float(0x4B000000u | ((q[u] >> (4 * j)) & 0xFu)) - 8388608.0f;   // exact
        v[j] = __fmaf_rn(qf, s[u], b[u]);
      }
      if constexpr (OUT == 0) {
        float4 *o = reinterpret_cast<float4 *>(out) + i * 2;
        o[0] = make_float4(v[0], v[1], v[2], v[3]);
        o[1] = make_float4(v[4], v[5], v[6], v[7]);
      } else {
        uint32_t pk[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          if constexpr (OUT == 1) {
            pk[j] = pack_bf16x2(v[2 * j], v[2 * j + 1]);
          } else {
            __half2 h = __floats2half2_rn(v[2 * j], v[2 * j + 1]);
            pk[j] = *reinterpret_cast<uint32_t *>(&h);
          }
        }
        reinterpret_cast<uint4 *>(out)[i] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
      }
    }
  }
}

}  // namespace

cudaError_t launch_q4_dequant(const uint32_t *w, const uint16_t *scales, const uint16_t *biases,
                              int64_t N, int64_t K, void *out, int out_dtype, cudaStream_t s) {
  const int64_t words = N * (K / 8);
  const int threads = 256;
  int64_t blocks = (words + threads * 4 - 1) / (threads * 4);
  if (blocks > 152 * 16) blocks = 152 * 16;
  switch (out_dtype) {
    case Q4MM_F32: q4_dequant_kernel<0><<<(unsigned)blocks, threads, 0, s>>>(w, scales, biases, words, out); break;
    case Q4MM_BF16: q4_dequant_kernel<1><<<(unsigned)blocks, threads, 0, s>>>(w, scales, biases, words, out); break;
    default: q4_dequant_kernel<2><<<(unsigned)blocks, threads, 0, s>>>(w, scales, biases, words, out); break;
  }
  return cudaGetLastError();
}

}  // namespace q4mm
