// lut4.cu -- LUT4 (frozen 16-entry codebook, blocked scales) general-layout kernels.
//
// lut4.rs (onnxruntime-ep-mlx 0.31.1): the stored [rows, cols] code matrix is read by flat
// index f, byte f/2, high nibble for even f and low nibble for odd f; the value is
// book[code] * scales[f / block] in fp32 (the lookup4 kernel source, the CPU branch of
// `execute`, and the lookup4 decode kernel).
//
// These kernels serve every layout the pages allow (either transpose, any even block,
// blocks straddling rows).  The fused fast paths for the [N, K/2] layout live in gemv.cu
// (M <= 16) and gemm_tc.cu (M > 16).
//
// Rounded-weight variant (lut4.rs, `rounded_weight` and the Cast matcher of the lookup
// matmul pattern): when the graph casts the decoded weight to half or bfloat16 and back,
// the matmul multiplies by that rounded value.  ROUND = 1 rounds fl32(book * scale) to IEEE
// binary16 and widens it again, ROUND = 2 does the same through bfloat16 (both nearest
// even); the product with x and the sum stay fp32, so the rounded weight enters exactly.
#include "q4mm_internal.cuh"

namespace q4mm {
namespace {

struct Book16 {
  float v[16];
};

__device__ __forceinline__ float lut4_value(const uint8_t *__restrict__ packed,
                                            const float *__restrict__ scales, const float *book,
                                            int64_t f, int64_t block) {
  const uint32_t byte = __ldg(packed + f / 2);
  const uint32_t code = (f & 1) ? (byte & 15u) : (byte >> 4);
  return book[code] * __ldg(scales + f / block);
}

template <int ROUND>   // 0 = as decoded, 1 = through binary16, 2 = through bfloat16
__device__ __forceinline__ float round_weight(float v) {
  if constexpr (ROUND == 1) {
    return __half2float(__float2half_rn(v));
  } else if constexpr (ROUND == 2) {
    return __bfloat162float(__float2bfloat16_rn(v));
  } else {
    return v;
  }
}

__device__ __forceinline__ void store_bf16(uint16_t *dst, float v) {
  __nv_bfloat16 b = __float2bfloat16_rn(v);
  *dst = *reinterpret_cast<uint16_t *>(&b);
}

// One output element per thread; fp32 accumulation, k ascending.
template <int ROUND>
__global__ void __launch_bounds__(128) lut4_general_kernel(
    const uint16_t *__restrict__ x, const uint8_t *__restrict__ packed,
    const float *__restrict__ scales, const __grid_constant__ Book16 bk, uint16_t *__restrict__ y,
    int64_t M, int64_t N, int64_t K, int64_t block, int transpose) {
  __shared__ float book[16];
  if (threadIdx.x < 16) book[threadIdx.x] = bk.v[threadIdx.x];
  __syncthreads();
  const int64_t n = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  if (n >= N) return;
  for (int64_t m = blockIdx.y; m < M; m += gridDim.y) {
    const uint16_t *xr = x + m * K;
    float acc = 0.f;
    for (int64_t k = 0; k < K; ++k) {
      const int64_t f = transpose ? n * K + k : k * N + n;
      acc = __fmaf_rn(bf16_bits_to_float(__ldg(xr + k)),
                      round_weight<ROUND>(lut4_value(packed, scales, book, f, block)), acc);
    }
    store_bf16(y + m * N + n, acc);
  }
}

// The [N, K/2] layout (K % 32 == 0, block % 32 == 0, 16-byte aligned x and packed) on CUDA
// cores: one warp per weight row n, each lane taking 32-code chunks (16 bytes of codes under
// one scale) with the next chunk's load issued before the current one is used; the x rows
// m0 .. m0+15 of blockIdx.y's group are read from L1/L2; fp32 FMA, then a warp sum.
template <int ROUND>
__global__ void __launch_bounds__(256) lut4_rowdot_kernel(
    const uint16_t *__restrict__ x, const uint8_t *__restrict__ packed,
    const float *__restrict__ scales, const __grid_constant__ Book16 bk, uint16_t *__restrict__ y,
    int M, int N, int K, int block) {
  __shared__ float book[16];
  if (threadIdx.x < 16) book[threadIdx.x] = bk.v[threadIdx.x];
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int chunks = K / 32;
  for (int m0 = blockIdx.y * 16; m0 < M; m0 += gridDim.y * 16) {
    const int mc = M - m0 < 16 ? M - m0 : 16;
    for (int n = blockIdx.x * 8 + (threadIdx.x >> 5); n < N; n += gridDim.x * 8) {
      const uint4 *row = reinterpret_cast<const uint4 *>(packed + (size_t)n * (K / 2));
      float acc[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) acc[i] = 0.f;
      uint4 q = make_uint4(0u, 0u, 0u, 0u);
      float s = 0.f;
      if (lane < chunks) {
        q = __ldg(row + lane);
        s = __ldg(scales + ((size_t)n * K + (size_t)lane * 32) / block);
      }
      for (int c = lane; c < chunks; c += 32) {
        const uint4 qc = q;
        const float sc = s;
        if (c + 32 < chunks) {
          q = __ldg(row + c + 32);
          s = __ldg(scales + ((size_t)n * K + (size_t)(c + 32) * 32) / block);
        }
        float w[32];
        const uint32_t words[4] = {qc.x, qc.y, qc.z, qc.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
#pragma unroll
          for (int b = 0; b < 4; ++b) {
            const uint32_t byte = (words[j] >> (8 * b)) & 255u;
            w[8 * j + 2 * b] = round_weight<ROUND>(book[byte >> 4] * sc);
            w[8 * j + 2 * b + 1] = round_weight<ROUND>(book[byte & 15u] * sc);
          }
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          if (i < mc) {
            const uint4 *xr = reinterpret_cast<const uint4 *>(x + (size_t)(m0 + i) * K + (size_t)c * 32);
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              const uint4 xv = __ldg(xr + v);
              const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                acc[i] = __fmaf_rn(__uint_as_float(xw[e] << 16), w[8 * v + 2 * e], acc[i]);
                acc[i] = __fmaf_rn(__uint_as_float(xw[e] & 0xFFFF0000u), w[8 * v + 2 * e + 1], acc[i]);
              }
            }
          }
        }
      }
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        if (i < mc) {
          float v = acc[i];
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
          if (lane == 0) store_bf16(y + (size_t)(m0 + i) * N + n, v);
        }
      }
    }
  }
}

template <int OUT>   // 0 = f32, 1 = bf16, 2 = f16
__global__ void __launch_bounds__(256) lut4_dequant_kernel(const uint8_t *__restrict__ packed,
                                                           const float *__restrict__ scales,
                                                           const __grid_constant__ Book16 bk,
                                                           int64_t total, int64_t block,
                                                           void *__restrict__ out) {
  __shared__ float book[16];
  if (threadIdx.x < 16) book[threadIdx.x] = bk.v[threadIdx.x];
  __syncthreads();
  for (int64_t f = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; f < total;
       f += (int64_t)gridDim.x * blockDim.x) {
    const float v = lut4_value(packed, scales, book, f, block);
    if constexpr (OUT == 0) {
      static_cast<float *>(out)[f] = v;
    } else if constexpr (OUT == 1) {
      __nv_bfloat16 b = __float2bfloat16_rn(v);
      static_cast<uint16_t *>(out)[f] = *reinterpret_cast<uint16_t *>(&b);
    } else {
      __half h = __float2half_rn(v);
      static_cast<uint16_t *>(out)[f] = *reinterpret_cast<uint16_t *>(&h);
    }
  }
}

// Vectorised decode for block % 32 == 0 and 16-byte aligned codes and output: a thread takes
// 8 consecutive elements (4 code bytes, one 4-byte load; they share one scale) per step, so
// consecutive lanes read consecutive words and write consecutive 16-byte (bf16 / f16) or
// 32-byte (f32) pieces.  Each byte's two codebook values come as one pair from a 256-entry
// table in shared memory; fl32(book * scale) is formed in fp32.  Elements past the last whole
// 32 run through the element kernel.
template <int OUT>   // 0 = f32, 1 = bf16, 2 = f16
__global__ void __launch_bounds__(256) lut4_dequant_vec_kernel(const uint8_t *__restrict__ packed,
                                                               const float *__restrict__ scales,
                                                               const __grid_constant__ Book16 bk,
                                                               int64_t n32, int64_t block,
                                                               void *__restrict__ out) {
  __shared__ float2 pairs[256];   // byte b -> (book[b >> 4], book[b & 15]): (even, odd) element
  pairs[threadIdx.x] = make_float2(bk.v[threadIdx.x >> 4], bk.v[threadIdx.x & 15]);
  __syncthreads();
  constexpr int kU = 4;   // words per thread per step, a warp-width apart
  const int64_t words = n32 * 4;
  const int64_t per_scale = block / 8;   // words per scale
  const uint32_t *w32 = reinterpret_cast<const uint32_t *>(packed);
  const int64_t stride = (int64_t)gridDim.x * blockDim.x * kU;
  const int64_t lane0 = (int64_t)blockIdx.x * blockDim.x * kU + (threadIdx.x / 32) * 32 * kU + threadIdx.x % 32;
  for (int64_t base = lane0; base < words; base += stride) {
    uint32_t c[kU];
    float sc[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int64_t i = base + 32 * u;
      if (i < words) {
        c[u] = __ldg(w32 + i);
        sc[u] = __ldg(scales + i / per_scale);
      }
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int64_t i = base + 32 * u;
      if (i >= words) break;
      float v[8];
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const float2 pr = pairs[(c[u] >> (8 * b)) & 0xFFu];
        v[2 * b] = pr.x * sc[u];
        v[2 * b + 1] = pr.y * sc[u];
      }
      if constexpr (OUT == 0) {
        float4 *o = static_cast<float4 *>(out) + i * 2;
        o[0] = make_float4(v[0], v[1], v[2], v[3]);
        o[1] = make_float4(v[4], v[5], v[6], v[7]);
      } else {
        uint32_t h[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          if constexpr (OUT == 1) {
            h[j] = pack_bf16x2(v[2 * j], v[2 * j + 1]);
          } else {
            __half2 hh = __floats2half2_rn(v[2 * j], v[2 * j + 1]);
            h[j] = *reinterpret_cast<uint32_t *>(&hh);
          }
        }
        static_cast<uint4 *>(out)[i] = make_uint4(h[0], h[1], h[2], h[3]);
      }
    }
  }
}

template <int OUT>
__global__ void __launch_bounds__(256) lut4_dequant_tail_kernel(const uint8_t *__restrict__ packed,
                                                                const float *__restrict__ scales,
                                                                const __grid_constant__ Book16 bk,
                                                                int64_t f0, int64_t total, int64_t block,
                                                                void *__restrict__ out) {
  __shared__ float book[16];
  if (threadIdx.x < 16) book[threadIdx.x] = bk.v[threadIdx.x];
  __syncthreads();
  const int64_t f = f0 + threadIdx.x;
  if (f >= total) return;
  const float v = lut4_value(packed, scales, book, f, block);
  if constexpr (OUT == 0) {
    static_cast<float *>(out)[f] = v;
  } else if constexpr (OUT == 1) {
    __nv_bfloat16 b = __float2bfloat16_rn(v);
    static_cast<uint16_t *>(out)[f] = *reinterpret_cast<uint16_t *>(&b);
  } else {
    __half h = __float2half_rn(v);
    static_cast<uint16_t *>(out)[f] = *reinterpret_cast<uint16_t *>(&h);
  }
}

}  // namespace

cudaError_t launch_lut4_general(const uint16_t *x, const uint8_t *packed, const float *scales,
                                const float *book, uint16_t *y, int64_t M, int64_t N,
                                int64_t K, int64_t block, int transpose, int rounding,
                                cudaStream_t s) {
  Book16 bk;
  for (int i = 0; i < 16; ++i) bk.v[i] = book[i];
  dim3 grid((unsigned)((N + 127) / 128), (unsigned)(M < 65535 ? M : 65535), 1);
  if (rounding == 1)
    lut4_general_kernel<1><<<grid, 128, 0, s>>>(x, packed, scales, bk, y, M, N, K, block, transpose);
  else if (rounding == 2)
    lut4_general_kernel<2><<<grid, 128, 0, s>>>(x, packed, scales, bk, y, M, N, K, block, transpose);
  else
    lut4_general_kernel<0><<<grid, 128, 0, s>>>(x, packed, scales, bk, y, M, N, K, block, transpose);
  return cudaGetLastError();
}

cudaError_t launch_lut4_rowdot(const uint16_t *x, const uint8_t *packed, const float *scales,
                               const float *book, uint16_t *y, int M, int N, int K, int block,
                               int rounding, cudaStream_t s) {
  Book16 bk;
  for (int i = 0; i < 16; ++i) bk.v[i] = book[i];
  const int row_blocks = (N + 7) / 8;
  const int m_groups = (M + 15) / 16;
  dim3 grid((unsigned)(row_blocks < 152 * 64 ? row_blocks : 152 * 64),
            (unsigned)(m_groups < 65535 ? m_groups : 65535), 1);
  if (rounding == 1)
    lut4_rowdot_kernel<1><<<grid, 256, 0, s>>>(x, packed, scales, bk, y, M, N, K, block);
  else if (rounding == 2)
    lut4_rowdot_kernel<2><<<grid, 256, 0, s>>>(x, packed, scales, bk, y, M, N, K, block);
  else
    lut4_rowdot_kernel<0><<<grid, 256, 0, s>>>(x, packed, scales, bk, y, M, N, K, block);
  return cudaGetLastError();
}

cudaError_t launch_lut4_dequant(const uint8_t *packed, const float *scales, const float *book,
                                int64_t rows, int64_t cols, int64_t block, void *out,
                                int out_dtype, cudaStream_t s) {
  Book16 bk;
  for (int i = 0; i < 16; ++i) bk.v[i] = book[i];
  const int64_t total = rows * cols;
  const bool vec = block % 32 == 0 && (reinterpret_cast<uintptr_t>(packed) & 15) == 0 &&
                   (reinterpret_cast<uintptr_t>(out) & 15) == 0 && total >= 32;
  if (vec) {
    const int64_t n32 = total / 32, rest = total - n32 * 32;
    int64_t blocks = (n32 * 4 + 1023) / 1024;
    if (blocks > 152 * 16) blocks = 152 * 16;
    switch (out_dtype) {
      case Q4MM_F32:
        lut4_dequant_vec_kernel<0><<<(unsigned)blocks, 256, 0, s>>>(packed, scales, bk, n32, block, out);
        if (rest) lut4_dequant_tail_kernel<0><<<1, 256, 0, s>>>(packed, scales, bk, n32 * 32, total, block, out);
        break;
      case Q4MM_BF16:
        lut4_dequant_vec_kernel<1><<<(unsigned)blocks, 256, 0, s>>>(packed, scales, bk, n32, block, out);
        if (rest) lut4_dequant_tail_kernel<1><<<1, 256, 0, s>>>(packed, scales, bk, n32 * 32, total, block, out);
        break;
      default:
        lut4_dequant_vec_kernel<2><<<(unsigned)blocks, 256, 0, s>>>(packed, scales, bk, n32, block, out);
        if (rest) lut4_dequant_tail_kernel<2><<<1, 256, 0, s>>>(packed, scales, bk, n32 * 32, total, block, out);
        break;
    }
    return cudaGetLastError();
  }
  int64_t blocks = (total + 255) / 256;
  if (blocks > 152 * 16) blocks = 152 * 16;
  switch (out_dtype) {
    case Q4MM_F32: lut4_dequant_kernel<0><<<(unsigned)blocks, 256, 0, s>>>(packed, scales, bk, total, block, out); break;
    case Q4MM_BF16: lut4_dequant_kernel<1><<<(unsigned)blocks, 256, 0, s>>>(packed, scales, bk, total, block, out); break;
    default: lut4_dequant_kernel<2><<<(unsigned)blocks, 256, 0, s>>>(packed, scales, bk, total, block, out); break;
  }
  return cudaGetLastError();
}

}  // namespace q4mm
