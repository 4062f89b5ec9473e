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

template <int OUT>   // 0 = f32, 1 = bf16, 2 = f16
__global__ void __launch_bounds__(256) q4_dequant_kernel(const uint4 *__restrict__ w,
                                                         const uint16_t *__restrict__ scales,
                                                         const uint16_t *__restrict__ biases,
                                                         int64_t groups, void *__restrict__ out) {
  for (int64_t g = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; g < groups;
       g += (int64_t)gridDim.x * blockDim.x) {
    const uint4 q = ldg_stream_v4(w + g);
    const float s = bf16_bits_to_float(ldg_u16(scales + g));
    const float b = bf16_bits_to_float(ldg_u16(biases + g));
    const uint32_t words[4] = {q.x, q.y, q.z, q.w};
    float v[32];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 8; ++j)
        v[i * 8 + j] = __fmaf_rn(static_cast<float>((words[i] >> (4 * j)) & 0xFu), s, b);
    if constexpr (OUT == 0) {
      float4 *o = reinterpret_cast<float4 *>(out) + g * 8;
#pragma unroll
      for (int i = 0; i < 8; ++i) o[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
    } else {
      uint4 *o = reinterpret_cast<uint4 *>(out) + g * 4;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        uint32_t p[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float lo = v[8 * i + 2 * j], hi = v[8 * i + 2 * j + 1];
          if constexpr (OUT == 1) {
            p[j] = pack_bf16x2(lo, hi);
          } else {
            __half2 h = __floats2half2_rn(lo, hi);
            p[j] = *reinterpret_cast<uint32_t *>(&h);
          }
        }
        o[i] = make_uint4(p[0], p[1], p[2], p[3]);
      }
    }
  }
}

}  // namespace

cudaError_t launch_q4_dequant(const uint32_t *w, const uint16_t *scales, const uint16_t *biases,
                              int64_t N, int64_t K, void *out, int out_dtype, cudaStream_t s) {
  const int64_t groups = N * (K / 32);
  const int threads = 256;
  int64_t blocks = (groups + threads - 1) / threads;
  if (blocks > 152 * 16) blocks = 152 * 16;
  const uint4 *w4 = reinterpret_cast<const uint4 *>(w);
  switch (out_dtype) {
    case Q4MM_F32: q4_dequant_kernel<0><<<(unsigned)blocks, threads, 0, s>>>(w4, scales, biases, groups, out); break;
    case Q4MM_BF16: q4_dequant_kernel<1><<<(unsigned)blocks, threads, 0, s>>>(w4, scales, biases, groups, out); break;
    default: q4_dequant_kernel<2><<<(unsigned)blocks, threads, 0, s>>>(w4, scales, biases, groups, out); break;
  }
  return cudaGetLastError();
}

}  // namespace q4mm
