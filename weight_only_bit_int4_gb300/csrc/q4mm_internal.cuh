// q4mm_internal.cuh -- shared device helpers and launcher declarations for libq4mm.
// Everything here is sm_103a-only CUDA C++ with inline PTX; nothing is shared with the
// CPU oracle.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "../../include/q4mm.h"

namespace q4mm {

// --------------------------------------------------------------------------------------
// Device error word (bits Q4MM_DEVERR_*).  Each translation unit keeps its own copy (no
// relocatable device code is needed) and exports a reader; q4mm_device_errors ORs them.
// --------------------------------------------------------------------------------------
static __device__ unsigned int g_device_error = 0;

#define Q4MM_DEFINE_ERROR_READER(fn)                                                  \
  cudaError_t fn(unsigned int *out, int clear) {                                      \
    unsigned int v = 0;                                                               \
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_device_error, sizeof v);              \
    if (e != cudaSuccess) return e;                                                   \
    *out |= v;                                                                        \
    if (clear) {                                                                      \
      const unsigned int z = 0;                                                       \
      e = cudaMemcpyToSymbol(g_device_error, &z, sizeof z);                          \
    }                                                                                 \
    return e;                                                                         \
  }

cudaError_t read_errors_moe(unsigned int *out, int clear);
cudaError_t read_errors_gemm(unsigned int *out, int clear);
cudaError_t read_errors_moe_tc(unsigned int *out, int clear);
cudaError_t read_errors_gemv(unsigned int *out, int clear);
cudaError_t read_errors_selftest(unsigned int *out, int clear);
cudaError_t launch_wait_timeout_selftest(const void *src16, unsigned long long limit_ns, cudaStream_t s);

__device__ __forceinline__ void raise_device_error(unsigned int bit) {
  atomicOr(&g_device_error, bit);
}

// Wall-clock limit of every bounded wait in the library (nanoseconds).
constexpr unsigned long long kWaitLimitNs = 2000000000ull;   // 2 s

// Programmatic dependent launch.  launch_dependents lets the next kernel in the stream (if
// it was launched with programmatic stream serialization) begin launching; wait blocks until
// every grid this one depends on has completed and its writes are visible.  Both are no-ops
// for a kernel launched without the attribute.
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// cp.async group bookkeeping: close the current group; wait until at most N groups are pending.
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// --------------------------------------------------------------------------------------
// Small conversions
// --------------------------------------------------------------------------------------
__device__ __forceinline__ float bf16_bits_to_float(uint16_t h) {
  return __uint_as_float(static_cast<uint32_t>(h) << 16);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  // cvt.rn.bf16x2.f32 d, a, b puts a in the upper half and b in the lower half.
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}

// d = (a & b) | c in one LOP3.
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t r;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
  return r;
}

__device__ __forceinline__ uint32_t bf16x2_sub(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

__device__ __forceinline__ uint32_t bf16x2_fma(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t r;
  asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
  return r;
}

// Streaming 16-byte global load that does not allocate in L1.
__device__ __forceinline__ uint4 ldg_stream_v4(const void *p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ uint16_t ldg_u16(const uint16_t *p) {
  uint16_t v;
  asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}

// --------------------------------------------------------------------------------------
// INT4 affine dequant of one 32-bit word (8 codes, low nibble first) into bf16 pairs.
// Magic-number conversion: (code | 0x4300) is the bf16 value 128 + code (exponent 2^7,
// 7 mantissa bits, so integers 128..255 are exact); subtracting 128 is exact, and the
// following bf16x2 FMA rounds code*s + b once, to nearest even.  One LOP3 pulls codes
// i and i+4 (bits 4i and 16+4i) into the two halves, so the pairs come out as
// (code i, code i+4) for i = 0..3.
// --------------------------------------------------------------------------------------
struct Int4Pairs {
  uint32_t p[4];   // p[i] = (bf16(w_i) low half, bf16(w_{i+4}) high half)
};

__device__ __forceinline__ Int4Pairs int4_word_to_bf16_pairs(uint32_t word, uint32_t s2,
                                                             uint32_t b2) {
  constexpr uint32_t kMask = 0x000F000Fu;
  constexpr uint32_t kMagic = 0x43004300u;   // bf16x2 (128, 128)
  Int4Pairs r;
  r.p[0] = and_or(word, kMask, kMagic);
  r.p[1] = and_or(word >> 4, kMask, kMagic);
  r.p[2] = and_or(word >> 8, kMask, kMagic);
  r.p[3] = and_or(word >> 12, kMask, kMagic);
#pragma unroll
  for (int i = 0; i < 4; ++i) r.p[i] = bf16x2_fma(bf16x2_sub(r.p[i], kMagic), s2, b2);
  return r;
}

// --------------------------------------------------------------------------------------
// Warp-level tensor-core MMA (m16n8k16, bf16 inputs, fp32 accumulate) for the small-M
// decode kernels, where the weight fragment is built in registers straight from HBM.
// --------------------------------------------------------------------------------------
// Not volatile: the MMA has no effect beyond its outputs, so the compiler may interleave
// independent accumulation chains (e.g. two chunks processed together).
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4],
                                               uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// --------------------------------------------------------------------------------------
// Thread-block cluster helpers (distributed shared memory reduction).
// --------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Address of the same shared-memory offset in cluster CTA `rank`.
__device__ __forceinline__ uint32_t map_shared_rank(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

__device__ __forceinline__ float4 ld_shared_cluster_v4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0,%1,%2,%3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr));
  return v;
}

// --------------------------------------------------------------------------------------
// Launchers (host side).  Each returns cudaSuccess or the launch error; arguments are
// validated by the C-ABI layer before these are called.
// --------------------------------------------------------------------------------------
cudaError_t launch_q4_dequant(const uint32_t *w, const uint16_t *scales, const uint16_t *biases,
                              int64_t N, int64_t K, void *out, int out_dtype, cudaStream_t s);

// overlap: launch with programmatic stream serialization, so that the kernel streams its
// weights while the previous kernel in the stream finishes (the weights must not be written
// by that kernel); x is read and y written only after the previous kernel has completed.
cudaError_t launch_q4_gemv(const uint16_t *x, const uint32_t *w, const uint16_t *scales,
                           const uint16_t *biases, uint16_t *y, int M, int N, int K,
                           cudaStream_t s, bool overlap = false);

// Dispatch records (plan once, replay with new pointers).  The record is a host object
// owned by the caller of record_*; replay_* launches exactly what the planned call would.
cudaError_t record_q4_gemv(int M, int N, int K, bool overlap, void **out);
cudaError_t replay_q4_gemv(const void *record, const uint16_t *x, const uint32_t *w, const uint16_t *scales,
                           const uint16_t *biases, uint16_t *y, cudaStream_t s);
void free_q4_gemv_record(void *record);
cudaError_t record_q4_0_mv(int n_rows, int top_k, int N, int K, int n_experts, uint64_t expert_stride,
                           bool swiglu, int *w_align, void **out);
cudaError_t replay_q4_0_mv(const void *record, const float *x, const float *up, const uint8_t *w,
                           const uint32_t *ids, float *out, cudaStream_t s);
void free_q4_0_mv_record(void *record);

cudaError_t launch_lut4_gemv(const uint16_t *x, const uint8_t *packed, const float *scales,
                             const float *book, uint16_t *y, int M, int N, int K, int block,
                             cudaStream_t s, bool overlap = false);

// rounding: 0 = the decoded fp32 weight, 1 = rounded through binary16, 2 = through bfloat16.
cudaError_t launch_lut4_general(const uint16_t *x, const uint8_t *packed, const float *scales,
                                const float *book, uint16_t *y, int64_t M, int64_t N,
                                int64_t K, int64_t block, int transpose, int rounding,
                                cudaStream_t s);

// The [N, K/2] layout on CUDA cores (K % 32 == 0, block % 32 == 0, 16-byte aligned x and
// packed); any M >= 1; same rounding codes.
cudaError_t launch_lut4_rowdot(const uint16_t *x, const uint8_t *packed, const float *scales,
                               const float *book, uint16_t *y, int M, int N, int K, int block,
                               int rounding, cudaStream_t s);

cudaError_t launch_lut4_dequant(const uint8_t *packed, const float *scales, const float *book,
                                int64_t rows, int64_t cols, int64_t block, void *out,
                                int out_dtype, cudaStream_t s);

cudaError_t launch_q4_gemm(const uint16_t *x, const uint32_t *w, const uint16_t *scales,
                           const uint16_t *biases, uint16_t *y, int M, int N, int K,
                           cudaStream_t s);

cudaError_t launch_lut4_gemm(const uint16_t *x, const uint8_t *packed, const float *scales,
                             const float *book, uint16_t *y, int M, int N, int K, int block,
                             cudaStream_t s);

cudaError_t launch_q4_0_route(const uint32_t *ids, int n_rows, int n_experts, uint32_t *htpe,
                              int32_t *hids, uint32_t *n_invalid, cudaStream_t s);

cudaError_t launch_q4_0_mv(const float *x, const uint8_t *w, const uint32_t *ids, float *out,
                           int n_tokens, int top_k, int N, int K, int n_experts,
                           uint64_t expert_stride, cudaStream_t s);

cudaError_t launch_q4_0_swiglu_mv(const float *gate, const float *up, const uint8_t *w, const uint32_t *ids,
                                  float *out, int n_rows, int N, int K, int n_experts, uint64_t expert_stride,
                                  cudaStream_t s);

cudaError_t launch_q4_0_mm(const float *x, const uint8_t *w, const uint32_t *ids, float *out,
                           int n_tokens, int top_k, int N, int K, int n_experts,
                           uint64_t expert_stride, void *workspace, cudaStream_t s);

// Raise kernel `fn`'s dynamic shared-memory limit on the current device to at least `bytes`,
// never lowering it.  The same kernel serves shapes of different sizes, and a dispatch record
// planned for a large shape must still launch after a smaller shape was planned or called.
cudaError_t ensure_dynamic_smem(const void *fn, int bytes);

cudaError_t launch_q8_0_matmul_id(const float *x, const uint8_t *w, const uint32_t *ids, float *out,
                                  int n_tokens, int top_k, int N, int K, int n_experts, uint64_t expert_stride,
                                  bool mm, void *workspace, cudaStream_t s);
size_t q8_0_mm_workspace_bytes(int64_t n_tokens, int64_t top_k, int64_t K, int64_t n_experts);

// Block types of the routed kernels: GGML Q4_0 (18 bytes: fp16 d, 16 bytes of nibbles) and
// Q8_0 (34 bytes: fp16 d, 32 signed bytes).
constexpr int kQ4_0 = 0, kQ8_0 = 1;

// Routed-row count check: n_tokens and top_k are each bounded before their product is
// formed, so a huge top_k cannot overflow int64 and wrap past the 2^24 limit.
inline bool routed_rows_ok(int64_t n_tokens, int64_t top_k) {
  const int64_t kMaxRows = int64_t(1) << 24;
  return n_tokens >= 0 && top_k >= 1 && n_tokens <= kMaxRows && top_k <= kMaxRows &&
         n_tokens * top_k <= kMaxRows;
}
size_t q4_0_mm_workspace_bytes(int64_t n_tokens, int64_t top_k, int64_t N, int64_t K,
                               int64_t n_experts);

// Workspace of the Q4_0 mat-mat path (every part 256-byte aligned):
//   htpe    u32 [E]        per-expert routed counts
//   offs    u32 [E + 1]    exclusive prefix of htpe (offs[E] = number of valid rows)
//   hids    i32 [R]        routed rows grouped by expert, ascending within an expert
//   invalid u32 [1]        rows whose id is >= E
//   blk     int4 [B]       token blocks (expert, first position in hids, count <= kMoeTokBlock, 0)
//   n_blk   u32 [1]        number of token blocks
//   xs      fp16 [R, K]    x rows gathered in hids order, each scaled by a power of two
//                          (the mm operand)
//   xun     f32 [R]        per gathered row, the power of two that undoes its scaling
//   tsc     f32 [R]        per token (first n_tokens entries), the power of two that scales it
constexpr int kMoeTokBlock = 112;
struct MoeWorkspace {
  size_t htpe, offs, hids, invalid, blk, n_blk, xs, xun, tsc, total;
};
inline size_t align256(size_t v) { return (v + 255) & ~size_t(255); }
inline MoeWorkspace moe_workspace_layout(int64_t n_rows, int64_t K, int64_t E) {
  MoeWorkspace w{};
  size_t o = 0;
  w.htpe = o; o = align256(o + 4 * (size_t)E);
  w.offs = o; o = align256(o + 4 * (size_t)(E + 1));
  w.hids = o; o = align256(o + 4 * (size_t)n_rows);
  w.invalid = o; o = align256(o + 4);
  const size_t max_blk = (size_t)(n_rows + kMoeTokBlock - 1) / kMoeTokBlock + (size_t)E;
  w.blk = o; o = align256(o + 16 * max_blk);
  w.n_blk = o; o = align256(o + 4);
  w.xs = o; o = align256(o + 2 * (size_t)n_rows * (size_t)K);
  w.xun = o; o = align256(o + 4 * (size_t)n_rows);
  w.tsc = o; o = align256(o + 4 * (size_t)n_rows);
  w.total = o;
  return w;
}

cudaError_t launch_q4_0_route_blocks(const uint32_t *ids, int n_rows, int n_experts, void *workspace,
                                     cudaStream_t s);
// The tensor-core mat-mat form (after routing) takes whole 256-element TMA boxes of blocks
// (K % 256 == 0) from 16-byte aligned expert slabs.
inline bool routed_mm_tc_ok(int K, uint64_t expert_stride, const void *w) {
  return K % 256 == 0 && expert_stride % 16 == 0 && (reinterpret_cast<uintptr_t>(w) & 15) == 0;
}
// bt: kQ4_0 or kQ8_0.  The workspace must already hold the routing (launch_route_internal).
cudaError_t launch_routed_mm_tc(int bt, const float *x, const uint8_t *w, float *out, int n_tokens, int top_k,
                                int N, int K, int n_experts, uint64_t expert_stride, void *workspace,
                                cudaStream_t s);

}  // namespace q4mm
