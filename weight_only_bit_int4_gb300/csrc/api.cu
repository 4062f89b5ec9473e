// api.cu -- the C ABI of libq4mm (declared in include/q4mm.h): host-side argument checks,
// then launches on the caller's stream.  Nothing here allocates device memory or
// synchronises (except q4mm_device_errors, a diagnostics call); dispatch records are small
// host objects.
//
// The checks mirror the pages' own gates: quant_fastkernel.rs `eligible` (group size 32,
// K a multiple of 32, bf16 activations/scales/biases, uint32 weights) and
// quantized_matmul_id_ggml.rs `quantized_matmul_id_ggml` (non-zero sizes, K divisible by
// the block size, expert_stride at least one expert's bytes, buffer sizes).  Unlike
// `try_apply` on the first page, a failed check never falls back to another path.
#include "q4mm_internal.cuh"

#include <stdint.h>

#include <map>
#include <mutex>
#include <new>
#include <utility>

using namespace q4mm;

namespace q4mm {

cudaError_t ensure_dynamic_smem(const void *fn, int bytes) {
  static std::mutex mu;
  static std::map<std::pair<int, const void *>, int> limit;   // (device, kernel) -> limit set
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  int &cur = limit[{dev, fn}];
  if (bytes <= cur) return cudaSuccess;
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) cur = bytes;
  return e;
}

}  // namespace q4mm

namespace {

constexpr int64_t kMaxDim = int64_t(1) << 30;

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// Compute capability 10.3 (GB300) is the only target.  Cached per device ordinal.
q4mm_status check_device() {
  static int cached[64] = {0};   // 0 unknown, 1 ok, 2 wrong device
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return Q4MM_ERR_CUDA;
  if (dev >= 0 && dev < 64 && cached[dev]) return cached[dev] == 1 ? Q4MM_OK : Q4MM_ERR_DEVICE;
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return Q4MM_ERR_CUDA;
  const bool ok = major == 10 && minor == 3;
  if (dev >= 0 && dev < 64) cached[dev] = ok ? 1 : 2;
  return ok ? Q4MM_OK : Q4MM_ERR_DEVICE;
}

q4mm_status from_cuda(cudaError_t e) { return e == cudaSuccess ? Q4MM_OK : Q4MM_ERR_CUDA; }

bool valid_dtype(int d) { return d == Q4MM_F32 || d == Q4MM_BF16 || d == Q4MM_F16; }

}  // namespace

extern "C" {

const char *q4mm_status_string(int status) {
  switch (status) {
    case Q4MM_OK: return "ok";
    case Q4MM_ERR_INVALID_ARG: return "invalid argument";
    case Q4MM_ERR_UNSUPPORTED: return "unsupported request (alignment or layout)";
    case Q4MM_ERR_WORKSPACE: return "workspace missing or too small";
    case Q4MM_ERR_CUDA: return "CUDA runtime error";
    case Q4MM_ERR_DEVICE: return "current device is not compute capability 10.3";
    default: return "unknown status";
  }
}

int q4mm_version(void) { return 100; }

q4mm_status q4mm_device_errors(uint32_t *out_flags, int clear) {
  if (!out_flags) return Q4MM_ERR_INVALID_ARG;
  if (cudaDeviceSynchronize() != cudaSuccess) return Q4MM_ERR_CUDA;
  unsigned int v = 0;
  if (read_errors_moe(&v, clear) != cudaSuccess) return Q4MM_ERR_CUDA;
  if (read_errors_gemm(&v, clear) != cudaSuccess) return Q4MM_ERR_CUDA;
  if (read_errors_moe_tc(&v, clear) != cudaSuccess) return Q4MM_ERR_CUDA;
  if (read_errors_gemv(&v, clear) != cudaSuccess) return Q4MM_ERR_CUDA;
  if (read_errors_selftest(&v, clear) != cudaSuccess) return Q4MM_ERR_CUDA;
  *out_flags = v;
  return Q4MM_OK;
}

q4mm_status q4mm_selftest_wait_timeout(const void *src16, uint32_t limit_ns, q4mm_stream_t stream) {
  if (!src16 || limit_ns == 0 || limit_ns > 1000000000u) return Q4MM_ERR_INVALID_ARG;
  if (!aligned(src16, 16)) return Q4MM_ERR_UNSUPPORTED;
  q4mm_status st = check_device();
  if (st != Q4MM_OK) return st;
  return from_cuda(launch_wait_timeout_selftest(src16, limit_ns, (cudaStream_t)stream));
}

// ------------------------------------------------------------------------------------------
// INT4 group-32 affine
// ------------------------------------------------------------------------------------------
static q4mm_status check_int4(const void *w, const void *s, const void *b, int64_t N, int64_t K) {
  if (!w || !s || !b) return Q4MM_ERR_INVALID_ARG;
  if (N < 1 || N > kMaxDim || K < 32 || K > kMaxDim || K % 32 != 0) return Q4MM_ERR_INVALID_ARG;
  if (!aligned(w, 16) || !aligned(s, 16) || !aligned(b, 16)) return Q4MM_ERR_UNSUPPORTED;
  return Q4MM_OK;
}

q4mm_status q4_dequant(const uint32_t *w, const uint16_t *scales, const uint16_t *biases,
                       int64_t N, int64_t K, void *out, int out_dtype, q4mm_stream_t stream) {
  if (N == 0) return Q4MM_OK;
  q4mm_status st = check_int4(w, scales, biases, N, K);
  if (st != Q4MM_OK) return st;
  if (!out || !valid_dtype(out_dtype)) return Q4MM_ERR_INVALID_ARG;
  if (!aligned(out, 16)) return Q4MM_ERR_UNSUPPORTED;
  if ((st = check_device()) != Q4MM_OK) return st;
  return from_cuda(launch_q4_dequant(w, scales, biases, N, K, out, out_dtype, (cudaStream_t)stream));
}

q4mm_status q4_gemv(const uint16_t *x, const uint32_t *w, const uint16_t *scales,
                    const uint16_t *biases, uint16_t *y, int64_t M, int64_t N, int64_t K,
                    q4mm_stream_t stream) {
  return q4_gemv_ex(x, w, scales, biases, y, M, N, K, 0u, stream);
}

q4mm_status q4_gemv_ex(const uint16_t *x, const uint32_t *w, const uint16_t *scales,
                       const uint16_t *biases, uint16_t *y, int64_t M, int64_t N, int64_t K,
                       uint32_t flags, q4mm_stream_t stream) {
  if ((flags & ~Q4MM_GEMV_STATIC_WEIGHTS) != 0u) return Q4MM_ERR_INVALID_ARG;
  if (M == 0) return Q4MM_OK;
  if (M < 0 || M > 16) return Q4MM_ERR_INVALID_ARG;
  q4mm_status st = check_int4(w, scales, biases, N, K);
  if (st != Q4MM_OK) return st;
  if (!x || !y) return Q4MM_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(y, 16)) return Q4MM_ERR_UNSUPPORTED;
  if ((st = check_device()) != Q4MM_OK) return st;
  return from_cuda(launch_q4_gemv(x, w, scales, biases, y, (int)M, (int)N, (int)K, (cudaStream_t)stream,
                                  (flags & Q4MM_GEMV_STATIC_WEIGHTS) != 0u));
}

q4mm_status q4_gemm(const uint16_t *x, const uint32_t *w, const uint16_t *scales,
                    const uint16_t *biases, uint16_t *y, int64_t M, int64_t N, int64_t K,
                    q4mm_stream_t stream) {
  if (M == 0) return Q4MM_OK;
  if (M < 0 || M > kMaxDim) return Q4MM_ERR_INVALID_ARG;
  q4mm_status st = check_int4(w, scales, biases, N, K);
  if (st != Q4MM_OK) return st;
  if (!x || !y) return Q4MM_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(y, 16)) return Q4MM_ERR_UNSUPPORTED;
  if ((st = check_device()) != Q4MM_OK) return st;
  return from_cuda(launch_q4_gemm(x, w, scales, biases, y, (int)M, (int)N, (int)K, (cudaStream_t)stream));
}

// ------------------------------------------------------------------------------------------
// LUT4
// ------------------------------------------------------------------------------------------
static q4mm_status check_lut4(const uint8_t *packed, const float *scales, const float *book,
                              int64_t rows, int64_t cols, int64_t block) {
  if (!packed || !scales || !book) return Q4MM_ERR_INVALID_ARG;
  if (rows < 1 || cols < 1 || rows > kMaxDim || cols > kMaxDim) return Q4MM_ERR_INVALID_ARG;
  if (rows * cols > (int64_t(1) << 40)) return Q4MM_ERR_INVALID_ARG;
  if (block <= 0 || block % 2 != 0) return Q4MM_ERR_INVALID_ARG;
  if (!aligned(scales, 4)) return Q4MM_ERR_UNSUPPORTED;
  return Q4MM_OK;
}

q4mm_status lut4_matmul(const uint16_t *x, const uint8_t *packed, const float *scales,
                        const float *book, uint16_t *y, int64_t M, int64_t N, int64_t K,
                        int64_t block, int transpose, q4mm_stream_t stream) {
  return lut4_matmul_ex(x, packed, scales, book, y, M, N, K, block, transpose, 0u, stream);
}

q4mm_status lut4_matmul_ex(const uint16_t *x, const uint8_t *packed, const float *scales,
                           const float *book, uint16_t *y, int64_t M, int64_t N, int64_t K,
                           int64_t block, int transpose, uint32_t flags, q4mm_stream_t stream) {
  const uint32_t known = Q4MM_GEMV_STATIC_WEIGHTS | Q4MM_LUT4_ROUND_F16 | Q4MM_LUT4_ROUND_BF16;
  if ((flags & ~known) != 0u) return Q4MM_ERR_INVALID_ARG;
  if ((flags & Q4MM_LUT4_ROUND_F16) && (flags & Q4MM_LUT4_ROUND_BF16)) return Q4MM_ERR_INVALID_ARG;
  if (M == 0) return Q4MM_OK;
  if (M < 0 || M > kMaxDim || (transpose != 0 && transpose != 1)) return Q4MM_ERR_INVALID_ARG;
  const int64_t rows = transpose ? N : K, cols = transpose ? K : N;
  q4mm_status st = check_lut4(packed, scales, book, rows, cols, block);
  if (st != Q4MM_OK) return st;
  if (!x || !y) return Q4MM_ERR_INVALID_ARG;
  if (!aligned(x, 2) || !aligned(y, 2)) return Q4MM_ERR_UNSUPPORTED;
  if ((st = check_device()) != Q4MM_OK) return st;
  cudaStream_t s = (cudaStream_t)stream;
  const bool fast = transpose == 1 && K % 32 == 0 && block % 32 == 0 && K % block == 0 &&
                    aligned(x, 16) && aligned(packed, 16) && aligned(y, 16);
  const bool overlap = (flags & Q4MM_GEMV_STATIC_WEIGHTS) != 0u;
  // rounding code shared with the CUDA-core kernels: 1 = binary16, 2 = bfloat16
  const int rounding = (flags & Q4MM_LUT4_ROUND_F16) ? 1 : (flags & Q4MM_LUT4_ROUND_BF16) ? 2 : 0;
  if (rounding == 1) {
    // A binary16 weight is not a bfloat16 value, so the tensor-core paths (bf16 operands)
    // cannot take it exactly: fp32 FMA on CUDA cores.
    if (fast)
      return from_cuda(launch_lut4_rowdot(x, packed, scales, book, y, (int)M, (int)N, (int)K, (int)block, 1, s));
    return from_cuda(launch_lut4_general(x, packed, scales, book, y, M, N, K, block, transpose, 1, s));
  }
  if (fast && M <= 16) {
    // The decode kernels stage scales with 8- and 16-byte cp.async copies, which need the
    // scale array 16-byte aligned; the header promises only 4.
    if (!aligned(scales, 16))
      return from_cuda(launch_lut4_general(x, packed, scales, book, y, M, N, K, block, transpose, rounding, s));
    // The decode kernels' bf16 operand is bf16(fl32(book * scale)): the bfloat16 rounding
    // itself, except in the K-split kernel (taken only for M <= 4 and K % 512 == 0), which
    // multiplies by bf16(book) and applies the scale after the MMA.
    if (rounding == 2 && M <= 4 && K % 512 == 0)
      return from_cuda(launch_lut4_rowdot(x, packed, scales, book, y, (int)M, (int)N, (int)K, (int)block, 2, s));
    return from_cuda(launch_lut4_gemv(x, packed, scales, book, y, (int)M, (int)N, (int)K, (int)block, s,
                                      overlap));
  }
  if (fast && K % 64 == 0 && block % 64 == 0) {
    // the GEMM's operand is bf16(fl32(book * scale)) in every plan
    cudaError_t e = launch_lut4_gemm(x, packed, scales, book, y, (int)M, (int)N, (int)K, (int)block, s);
    if (e != cudaErrorNotSupported) return from_cuda(e);
  }
  if (rounding == 2 && fast)
    return from_cuda(launch_lut4_rowdot(x, packed, scales, book, y, (int)M, (int)N, (int)K, (int)block, 2, s));
  return from_cuda(launch_lut4_general(x, packed, scales, book, y, M, N, K, block, transpose, rounding, s));
}

q4mm_status lut4_dequant(const uint8_t *packed, const float *scales, const float *book,
                         int64_t rows, int64_t cols, int64_t block, void *out, int out_dtype,
                         q4mm_stream_t stream) {
  q4mm_status st = check_lut4(packed, scales, book, rows, cols, block);
  if (st != Q4MM_OK) return st;
  if (!out || !valid_dtype(out_dtype)) return Q4MM_ERR_INVALID_ARG;
  if (!aligned(out, 4)) return Q4MM_ERR_UNSUPPORTED;
  if ((st = check_device()) != Q4MM_OK) return st;
  return from_cuda(launch_lut4_dequant(packed, scales, book, rows, cols, block, out, out_dtype,
                                       (cudaStream_t)stream));
}

// ------------------------------------------------------------------------------------------
// GGML Q4_0 expert-routed
// ------------------------------------------------------------------------------------------
q4mm_status q4_0_route(const uint32_t *ids, int64_t n_rows, int64_t n_experts, uint32_t *htpe,
                       int32_t *hids, uint32_t *n_invalid, q4mm_stream_t stream) {
  if (!ids || !htpe || !hids) return Q4MM_ERR_INVALID_ARG;
  if (n_rows < 1 || n_rows > (int64_t(1) << 24) || n_experts < 1 || n_experts > 1024)
    return Q4MM_ERR_INVALID_ARG;
  if (!aligned(ids, 4) || !aligned(htpe, 4) || !aligned(hids, 4) || (n_invalid && !aligned(n_invalid, 4)))
    return Q4MM_ERR_UNSUPPORTED;
  q4mm_status st = check_device();
  if (st != Q4MM_OK) return st;
  return from_cuda(launch_q4_0_route(ids, (int)n_rows, (int)n_experts, htpe, hids, n_invalid,
                                     (cudaStream_t)stream));
}

size_t q4_0_matmul_id_workspace_size(int64_t n_tokens, int64_t top_k, int64_t N, int64_t K,
                                     int64_t n_experts) {
  if (n_tokens < 1 || !routed_rows_ok(n_tokens, top_k) || N < 1 || K < 32 || N > kMaxDim || K > kMaxDim ||
      n_experts < 1 || n_experts > 1024)
    return 0;
  return q4_0_mm_workspace_bytes(n_tokens, top_k, N, K, n_experts);
}

q4mm_status q4_0_matmul_id(const float *x, const void *w, const uint32_t *ids, float *out,
                           int64_t n_tokens, int64_t top_k, int64_t N, int64_t K,
                           int64_t n_experts, uint64_t expert_stride, int mode,
                           void *workspace, size_t workspace_bytes, q4mm_stream_t stream) {
  if (n_tokens == 0) return Q4MM_OK;
  if (!x || !w || !ids || !out) return Q4MM_ERR_INVALID_ARG;
  if (n_tokens < 0 || top_k < 1 || N < 1 || K < 32 || K % 32 != 0 || n_experts < 1 ||
      n_experts > 1024 || N > kMaxDim || K > kMaxDim)
    return Q4MM_ERR_INVALID_ARG;
  if (!routed_rows_ok(n_tokens, top_k)) return Q4MM_ERR_INVALID_ARG;
  const uint64_t per_expert = (uint64_t)N * (uint64_t)(K / 32) * 18u;
  if (expert_stride < per_expert) return Q4MM_ERR_INVALID_ARG;
  if (mode < 0 || mode > 2) return Q4MM_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(out, 16) || !aligned(ids, 4)) return Q4MM_ERR_UNSUPPORTED;
  const bool mm = mode == 2 || (mode == 0 && n_tokens > Q4MM_MM_ID_THRESHOLD);
  if (mm) {
    const size_t need = q4_0_mm_workspace_bytes(n_tokens, top_k, N, K, n_experts);
    if (!workspace || workspace_bytes < need) return Q4MM_ERR_WORKSPACE;
    if (!aligned(workspace, 256)) return Q4MM_ERR_UNSUPPORTED;
  }
  q4mm_status st = check_device();
  if (st != Q4MM_OK) return st;
  cudaStream_t s = (cudaStream_t)stream;
  const uint8_t *wb = static_cast<const uint8_t *>(w);
  if (mm)
    return from_cuda(launch_q4_0_mm(x, wb, ids, out, (int)n_tokens, (int)top_k, (int)N, (int)K,
                                    (int)n_experts, expert_stride, workspace, s));
  return from_cuda(launch_q4_0_mv(x, wb, ids, out, (int)n_tokens, (int)top_k, (int)N, (int)K,
                                  (int)n_experts, expert_stride, s));
}

size_t q8_0_matmul_id_workspace_size(int64_t n_tokens, int64_t top_k, int64_t N, int64_t K,
                                     int64_t n_experts) {
  if (n_tokens < 1 || !routed_rows_ok(n_tokens, top_k) || N < 1 || K < 32 || N > kMaxDim || K > kMaxDim ||
      n_experts < 1 || n_experts > 1024)
    return 0;
  return q8_0_mm_workspace_bytes(n_tokens, top_k, K, n_experts);
}

q4mm_status q8_0_matmul_id(const float *x, const void *w, const uint32_t *ids, float *out,
                           int64_t n_tokens, int64_t top_k, int64_t N, int64_t K,
                           int64_t n_experts, uint64_t expert_stride, int mode,
                           void *workspace, size_t workspace_bytes, q4mm_stream_t stream) {
  if (n_tokens == 0) return Q4MM_OK;
  if (!x || !w || !ids || !out) return Q4MM_ERR_INVALID_ARG;
  if (n_tokens < 0 || top_k < 1 || N < 1 || K < 32 || K % 32 != 0 || n_experts < 1 ||
      n_experts > 1024 || N > kMaxDim || K > kMaxDim)
    return Q4MM_ERR_INVALID_ARG;
  if (!routed_rows_ok(n_tokens, top_k)) return Q4MM_ERR_INVALID_ARG;
  const uint64_t per_expert = (uint64_t)N * (uint64_t)(K / 32) * 34u;
  if (expert_stride < per_expert) return Q4MM_ERR_INVALID_ARG;
  if (mode < 0 || mode > 2) return Q4MM_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(out, 16) || !aligned(ids, 4)) return Q4MM_ERR_UNSUPPORTED;
  const bool mm = mode == 2 || (mode == 0 && n_tokens > Q4MM_MM_ID_THRESHOLD);
  if (mm) {
    const size_t need = q8_0_mm_workspace_bytes(n_tokens, top_k, K, n_experts);
    if (!workspace || workspace_bytes < need) return Q4MM_ERR_WORKSPACE;
    if (!aligned(workspace, 256)) return Q4MM_ERR_UNSUPPORTED;
  }
  q4mm_status st = check_device();
  if (st != Q4MM_OK) return st;
  return from_cuda(launch_q8_0_matmul_id(x, static_cast<const uint8_t *>(w), ids, out, (int)n_tokens, (int)top_k,
                                         (int)N, (int)K, (int)n_experts, expert_stride, mm, workspace,
                                         (cudaStream_t)stream));
}

q4mm_status q4_0_matmul_id_swiglu(const float *gate, const float *up, const void *w,
                                  const uint32_t *ids, float *out, int64_t n_tokens, int64_t top_k,
                                  int64_t N, int64_t K, int64_t n_experts, uint64_t expert_stride,
                                  q4mm_stream_t stream) {
  if (n_tokens == 0) return Q4MM_OK;
  if (!gate || !up || !w || !ids || !out) return Q4MM_ERR_INVALID_ARG;
  if (n_tokens < 0 || top_k < 1 || N < 1 || K < 32 || K % 32 != 0 || n_experts < 1 ||
      n_experts > 1024 || N > kMaxDim || K > kMaxDim)
    return Q4MM_ERR_INVALID_ARG;
  if (!routed_rows_ok(n_tokens, top_k)) return Q4MM_ERR_INVALID_ARG;
  const uint64_t per_expert = (uint64_t)N * (uint64_t)(K / 32) * 18u;
  if (expert_stride < per_expert) return Q4MM_ERR_INVALID_ARG;
  if (!aligned(gate, 16) || !aligned(up, 16) || !aligned(out, 16) || !aligned(ids, 4))
    return Q4MM_ERR_UNSUPPORTED;
  q4mm_status st = check_device();
  if (st != Q4MM_OK) return st;
  return from_cuda(launch_q4_0_swiglu_mv(gate, up, static_cast<const uint8_t *>(w), ids, out,
                                         (int)(n_tokens * top_k), (int)N, (int)K, (int)n_experts,
                                         expert_stride, (cudaStream_t)stream));
}

// ------------------------------------------------------------------------------------------
// Dispatch records
// ------------------------------------------------------------------------------------------
struct q4mm_record {
  int kind;      // kRecGemv, kRecMv or kRecSwiglu
  int device;    // the device current at creation; launches need it current again
  int w_align;   // alignment the weight pointer of every launch must keep
  void *impl;
};

namespace {
constexpr int kRecGemv = 1, kRecMv = 2, kRecSwiglu = 3;

q4mm_status check_record(const q4mm_record *rec, int kind) {
  if (!rec || rec->kind != kind) return Q4MM_ERR_INVALID_ARG;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return Q4MM_ERR_CUDA;
  return dev == rec->device ? Q4MM_OK : Q4MM_ERR_DEVICE;
}
}  // namespace

q4mm_status q4_gemv_record(int64_t M, int64_t N, int64_t K, uint32_t flags, q4mm_record **out) {
  if (!out) return Q4MM_ERR_INVALID_ARG;
  *out = nullptr;
  if ((flags & ~Q4MM_GEMV_STATIC_WEIGHTS) != 0u) return Q4MM_ERR_INVALID_ARG;
  if (M < 1 || M > 16 || N < 1 || N > kMaxDim || K < 32 || K > kMaxDim || K % 32 != 0) return Q4MM_ERR_INVALID_ARG;
  q4mm_status st = check_device();
  if (st != Q4MM_OK) return st;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return Q4MM_ERR_CUDA;
  void *impl = nullptr;
  if (record_q4_gemv((int)M, (int)N, (int)K, (flags & Q4MM_GEMV_STATIC_WEIGHTS) != 0u, &impl) != cudaSuccess)
    return Q4MM_ERR_CUDA;
  q4mm_record *rec = new (std::nothrow) q4mm_record{kRecGemv, dev, 16, impl};
  if (!rec) {
    free_q4_gemv_record(impl);
    return Q4MM_ERR_CUDA;
  }
  *out = rec;
  return Q4MM_OK;
}

q4mm_status q4_gemv_record_launch(const q4mm_record *rec, const uint16_t *x, const uint32_t *w,
                                  const uint16_t *scales, const uint16_t *biases, uint16_t *y,
                                  q4mm_stream_t stream) {
  q4mm_status st = check_record(rec, kRecGemv);
  if (st != Q4MM_OK) return st;
  if (!x || !w || !scales || !biases || !y) return Q4MM_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(w, 16) || !aligned(scales, 16) || !aligned(biases, 16) || !aligned(y, 16))
    return Q4MM_ERR_UNSUPPORTED;
  return from_cuda(replay_q4_gemv(rec->impl, x, w, scales, biases, y, (cudaStream_t)stream));
}

q4mm_status q4_gemv_record_launch_n(const q4mm_record *const *recs, const uint16_t *const *x,
                                    const uint32_t *const *w, const uint16_t *const *scales,
                                    const uint16_t *const *biases, uint16_t *const *y, int64_t n,
                                    q4mm_stream_t stream) {
  if (n == 0) return Q4MM_OK;
  if (n < 0 || n > 65536 || !recs || !x || !w || !scales || !biases || !y) return Q4MM_ERR_INVALID_ARG;
  for (int64_t i = 0; i < n; ++i) {
    if (!recs[i] || recs[i]->kind != kRecGemv) return Q4MM_ERR_INVALID_ARG;
    if (!x[i] || !w[i] || !scales[i] || !biases[i] || !y[i]) return Q4MM_ERR_INVALID_ARG;
  }
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return Q4MM_ERR_CUDA;
  for (int64_t i = 0; i < n; ++i) {
    if (recs[i]->device != dev) return Q4MM_ERR_DEVICE;
    if (!aligned(x[i], 16) || !aligned(w[i], 16) || !aligned(scales[i], 16) || !aligned(biases[i], 16) ||
        !aligned(y[i], 16))
      return Q4MM_ERR_UNSUPPORTED;
  }
  for (int64_t i = 0; i < n; ++i) {
    const cudaError_t e = replay_q4_gemv(recs[i]->impl, x[i], w[i], scales[i], biases[i], y[i], (cudaStream_t)stream);
    if (e != cudaSuccess) return from_cuda(e);
  }
  return Q4MM_OK;
}

q4mm_status q4_0_matmul_id_mv_record(int64_t n_tokens, int64_t top_k, int64_t N, int64_t K,
                                     int64_t n_experts, uint64_t expert_stride, int swiglu,
                                     q4mm_record **out) {
  if (!out) return Q4MM_ERR_INVALID_ARG;
  *out = nullptr;
  if (swiglu != 0 && swiglu != 1) return Q4MM_ERR_INVALID_ARG;
  if (n_tokens < 1 || top_k < 1 || N < 1 || K < 32 || K % 32 != 0 || n_experts < 1 || n_experts > 1024 ||
      N > kMaxDim || K > kMaxDim || !routed_rows_ok(n_tokens, top_k))
    return Q4MM_ERR_INVALID_ARG;
  if (expert_stride < (uint64_t)N * (uint64_t)(K / 32) * 18u) return Q4MM_ERR_INVALID_ARG;
  q4mm_status st = check_device();
  if (st != Q4MM_OK) return st;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return Q4MM_ERR_CUDA;
  void *impl = nullptr;
  int w_align = 1;
  if (record_q4_0_mv((int)(n_tokens * top_k), swiglu ? 1 : (int)top_k, (int)N, (int)K, (int)n_experts,
                     expert_stride, swiglu != 0, &w_align, &impl) != cudaSuccess)
    return Q4MM_ERR_CUDA;
  q4mm_record *rec = new (std::nothrow) q4mm_record{swiglu ? kRecSwiglu : kRecMv, dev, w_align, impl};
  if (!rec) {
    free_q4_0_mv_record(impl);
    return Q4MM_ERR_CUDA;
  }
  *out = rec;
  return Q4MM_OK;
}

q4mm_status q4_0_matmul_id_mv_record_launch(const q4mm_record *rec, const float *x, const float *up,
                                            const void *w, const uint32_t *ids, float *out,
                                            q4mm_stream_t stream) {
  if (!rec || (rec->kind != kRecMv && rec->kind != kRecSwiglu)) return Q4MM_ERR_INVALID_ARG;
  q4mm_status st = check_record(rec, rec->kind);
  if (st != Q4MM_OK) return st;
  const bool swiglu = rec->kind == kRecSwiglu;
  if (!x || !w || !ids || !out || (swiglu && !up) || (!swiglu && up)) return Q4MM_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(out, 16) || !aligned(ids, 4) || (swiglu && !aligned(up, 16)) ||
      !aligned(w, (uintptr_t)rec->w_align))
    return Q4MM_ERR_UNSUPPORTED;
  return from_cuda(replay_q4_0_mv(rec->impl, x, up, static_cast<const uint8_t *>(w), ids, out,
                                  (cudaStream_t)stream));
}

void q4mm_record_free(q4mm_record *rec) {
  if (!rec) return;
  if (rec->kind == kRecGemv)
    free_q4_gemv_record(rec->impl);
  else
    free_q4_0_mv_record(rec->impl);
  delete rec;
}

}  // extern "C"
