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

// One output element per thread; fp32 accumulation, k ascending.
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
      acc = __fmaf_rn(bf16_bits_to_float(__ldg(xr + k)), lut4_value(packed, scales, book, f, block), acc);
    }
    __nv_bfloat16 b = __float2bfloat16_rn(acc);
    y[m * N + n] = *reinterpret_cast<uint16_t *>(&b);
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

}  // namespace

cudaError_t launch_lut4_general(const uint16_t *x, const uint8_t *packed, const float *scales,
                                const float *book, uint16_t *y, int64_t M, int64_t N,
                                int64_t K, int64_t block, int transpose, cudaStream_t s) {
  Book16 bk;
  for (int i = 0; i < 16; ++i) bk.v[i] = book[i];
  dim3 grid((unsigned)((N + 127) / 128), (unsigned)(M < 65535 ? M : 65535), 1);
  lut4_general_kernel<<<grid, 128, 0, s>>>(x, packed, scales, bk, y, M, N, K, block, transpose);
  return cudaGetLastError();
}

cudaError_t launch_lut4_dequant(const uint8_t *packed, const float *scales, const float *book,
                                int64_t rows, int64_t cols, int64_t block, void *out,
                                int out_dtype, cudaStream_t s) {
  Book16 bk;
  for (int i = 0; i < 16; ++i) bk.v[i] = book[i];
  const int64_t total = rows * cols;
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
