// noalloc.cu -- q4_0_matmul_id_noalloc: the mat-mat form of the Q4_0 routed matmul for
// callers that cannot allocate device memory when they call it.
//
// q4_0_matmul_id needs a caller-provided workspace for its routing lists and gathered rows.
// Some callers have no way to get one at the moment of the call: serving loops that must
// never block on the device allocator or fail under memory pressure, and hosts (plugins,
// runtimes) that own every device buffer and hand out none.  This entry point needs no workspace from them: its scratch is one fixed
// array compiled into the library, below.
//
// The array is a file-scope __device__ variable, so every GPU that loads this library holds
// Q4MM_NOALLOC_SCRATCH_BYTES of it until the process exits.  Host code cannot use the
// array's name as a device address; on the first call on a device (with that device
// current) the address is fetched with cudaGetSymbolAddress and kept per device.  Every
// later call fetches it again unless its stream reports that it is capturing (then the kept
// one is used), so a device reset (which reloads the library's module in a new context)
// leaves no stale address behind.
//
// All calls on a device share the one array, which keeps whatever the previous call left.
// Nothing in it has to start at zero: each call's routing pass rewrites every routing field
// and every gathered row it later reads.  Calls whose executions overlap on the GPU (on
// different streams, or from different host threads without ordering) race on the array and
// give wrong results; order them on one stream.
#include "q4mm_internal.cuh"

#include <mutex>

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[Q4MM_NOALLOC_SCRATCH_BYTES];

std::mutex g_scratch_mutex;
void *g_scratch_ptr[64] = {};   // last fetched device address of g_noalloc_scratch, per device ordinal

bool is_aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

}  // namespace

extern "C" q4mm_status q4_0_matmul_id_noalloc(const float *x, const void *w, const uint32_t *ids, float *out,
                                              int64_t n_tokens, int64_t top_k, int64_t N, int64_t K,
                                              int64_t n_experts, uint64_t expert_stride,
                                              q4mm_stream_t stream) {
  if (n_tokens == 0) return Q4MM_OK;
  if (!x || !w || !ids || !out) return Q4MM_ERR_INVALID_ARG;
  const int64_t kMax = int64_t(1) << 30;
  if (n_tokens < 0 || top_k < 1 || N < 1 || K < 32 || K % 32 != 0 || n_experts < 1 || n_experts > 1024 ||
      N > kMax || K > kMax || !q4mm::routed_rows_ok(n_tokens, top_k))
    return Q4MM_ERR_INVALID_ARG;
  if (expert_stride < (uint64_t)N * (uint64_t)(K / 32) * 18u) return Q4MM_ERR_INVALID_ARG;
  if (!is_aligned(x, 16) || !is_aligned(out, 16) || !is_aligned(ids, 4)) return Q4MM_ERR_UNSUPPORTED;
  // The request must fit the fixed array; nothing is allocated to make room.
  if (q4mm::q4_0_mm_workspace_bytes(n_tokens, top_k, N, K, n_experts) > (size_t)Q4MM_NOALLOC_SCRATCH_BYTES)
    return Q4MM_ERR_WORKSPACE;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return Q4MM_ERR_CUDA;
  if (dev < 0 || dev >= 64) return Q4MM_ERR_UNSUPPORTED;
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return Q4MM_ERR_CUDA;
  if (major != 10 || minor != 3) return Q4MM_ERR_DEVICE;

  cudaStreamCaptureStatus capture = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing((cudaStream_t)stream, &capture) != cudaSuccess) return Q4MM_ERR_CUDA;
  void *scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (g_scratch_ptr[dev] == nullptr || capture == cudaStreamCaptureStatusNone) {
      void *p = nullptr;
      if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return Q4MM_ERR_CUDA;
      g_scratch_ptr[dev] = p;
    }
    scratch = g_scratch_ptr[dev];
  }
  const cudaError_t e = q4mm::launch_q4_0_mm(x, static_cast<const uint8_t *>(w), ids, out, (int)n_tokens,
                                             (int)top_k, (int)N, (int)K, (int)n_experts, expert_stride, scratch,
                                             (cudaStream_t)stream);
  return e == cudaSuccess ? Q4MM_OK : Q4MM_ERR_CUDA;
}
