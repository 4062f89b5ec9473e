// moe.cu -- GGML Q4_0 expert-routed matmul: routing lists, mat-vec form, and the
// workspace layout of the mat-mat form.
//
// quantized_matmul_id_ggml.rs (mlx-native 0.9.0), module doc: for routed row
// r = token*top_k + slot, expert e = ids[r], out[r][n] = sum_k dequant(W[e][n][k]) * x[token][k].
// Q4_0 block (32 values, 18 bytes): fp16 d, then 16 bytes; element j < 16 is the low nibble
// of byte j, element 16+j its high nibble; value = (q - 8) * d.
//
//  * q4_0_route: the map0 stage of `dispatch_id_mm_for_test` -- per-expert routed counts and
//    ascending routed-row lists -- as a deterministic stable counting sort in one CTA.
//  * mat-vec (`dispatch_id_mv`, `kernel_mul_mv_id_q4_0_f32`): one CTA per (routed row,
//    32 weight rows); fp32 FMA on CUDA cores; the token's x row is held in registers and
//    reused across the 32 weight rows.
#include "q4mm_internal.cuh"

namespace q4mm {

size_t q4_0_mm_workspace_bytes(int64_t n_tokens, int64_t top_k, int64_t N, int64_t K,
                               int64_t n_experts) {
  (void)N;
  return moe_workspace_layout(n_tokens * top_k, K, n_experts).total;
}

namespace {

// ---------------------------------------------------------------------------------------
// Routing: stable counting sort of row indices by expert id.
// Each warp owns a contiguous segment of rows.  Pass 1 counts ids per (warp, expert);
// a scan over (expert, warp) gives every warp its write position per expert; pass 2
// walks the segment again 32 rows at a time, ranking equal ids inside the step with
// __match_any_sync, so the output order equals the input order within each expert.
// ---------------------------------------------------------------------------------------
constexpr int kRouteThreads = 1024;

__global__ void __launch_bounds__(kRouteThreads) route_kernel(const uint32_t *__restrict__ ids,
                                                              int n_rows, int E, int n_warps,
                                                              uint32_t *__restrict__ htpe,
                                                              uint32_t *__restrict__ offs,
                                                              int32_t *__restrict__ hids,
                                                              uint32_t *__restrict__ n_invalid,
                                                              int4 *__restrict__ blk = nullptr,
                                                              uint32_t *__restrict__ n_blk = nullptr) {
  extern __shared__ uint32_t sm[];
  uint32_t *cnt = sm;                       // [n_warps][E]
  uint32_t *pos = sm + n_warps * E;         // [n_warps][E]
  uint32_t *scan = pos + n_warps * E;       // [E + 1]
  __shared__ uint32_t bad_count;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int active_warps = min(n_warps, (int)(blockDim.x / 32));
  for (int i = threadIdx.x; i < n_warps * E; i += blockDim.x) cnt[i] = 0;
  if (threadIdx.x == 0) bad_count = 0;
  __syncthreads();

  const int seg = (n_rows + active_warps - 1) / active_warps;
  const int r_begin = warp * seg;
  const int r_end = min(n_rows, r_begin + seg);
  const unsigned lt = (1u << lane) - 1u;
  if (warp < active_warps) {
    uint32_t bad = 0;
    for (int base = r_begin; base < r_end; base += 32) {
      const int r = base + lane;
      const bool in = r < r_end;
      const uint32_t e = in ? __ldg(ids + r) : 0xFFFFFFFFu;
      const bool valid = in && e < (uint32_t)E;
      bad += (in && !valid) ? 1u : 0u;
      const unsigned peers = __match_any_sync(0xFFFFFFFFu, valid ? e : 0xFFFFFFFFu);
      if (valid && (peers & lt) == 0) cnt[warp * E + e] += __popc(peers);
      __syncwarp();
    }
    if (bad) atomicAdd(&bad_count, bad);
  }
  __syncthreads();

  // htpe[e] = sum over warps; positions: exclusive scan over (e, warp) in e-major order.
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    uint32_t s = 0;
    for (int w = 0; w < n_warps; ++w) s += cnt[w * E + e];
    scan[e] = s;
    htpe[e] = s;
  }
  __syncthreads();
  if (threadIdx.x == 0) {   // E <= 1024: a serial scan is a few microseconds at most
    uint32_t run = 0;
    for (int e = 0; e < E; ++e) {
      const uint32_t c = scan[e];
      scan[e] = run;
      if (offs) offs[e] = run;
      run += c;
    }
    scan[E] = run;
    if (offs) offs[E] = run;
    if (n_invalid) *n_invalid = bad_count;
    if (bad_count) raise_device_error(Q4MM_DEVERR_BAD_EXPERT);
    if (blk) {   // token blocks of at most kMoeTokBlock rows, expert by expert
      uint32_t nb = 0;
      for (int e = 0; e < E; ++e) {
        const uint32_t c = (e + 1 < E ? scan[e + 1] : run) - scan[e];
        for (uint32_t b0 = 0; b0 < c; b0 += kMoeTokBlock)
          blk[nb++] = make_int4(e, (int)(scan[e] + b0), (int)min((uint32_t)kMoeTokBlock, c - b0), 0);
      }
      *n_blk = nb;
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    uint32_t run = scan[e];
    for (int w = 0; w < n_warps; ++w) {
      pos[w * E + e] = run;
      run += cnt[w * E + e];
    }
  }
  __syncthreads();

  if (warp < active_warps) {
    for (int base = r_begin; base < r_end; base += 32) {
      const int r = base + lane;
      const bool in = r < r_end;
      const uint32_t e = in ? __ldg(ids + r) : 0xFFFFFFFFu;
      const bool valid = in && e < (uint32_t)E;
      const unsigned peers = __match_any_sync(0xFFFFFFFFu, valid ? e : 0xFFFFFFFFu);
      if (valid) {
        const uint32_t p = pos[warp * E + e] + __popc(peers & lt);
        hids[p] = r;
      }
      __syncwarp();
      if (valid && (peers & lt) == 0) pos[warp * E + e] += __popc(peers);
      __syncwarp();
    }
  }
}

// ---------------------------------------------------------------------------------------
// Mat-vec: CTA = (routed row, 32 weight rows).  4 warps x 8 weight rows.  Lane l takes
// blocks l, l+32, ... of a K segment; its x values for those blocks stay in registers
// across the warp's 8 weight rows.  Weight rows are first copied to shared memory with
// coalesced loads (18-byte blocks are not 4-byte aligned in global memory).
// ---------------------------------------------------------------------------------------
constexpr int kMvWarps = 4;
constexpr int kMvRowsPerWarp = 8;
constexpr int kMvSegBlocks = 64;   // K segment: 64 blocks = 2048 values = 1152 bytes

struct MvParams {
  const float *x;
  const uint8_t *w;
  const uint32_t *ids;
  const int32_t *order;     // routed rows to visit (nullptr: row i is routed row i)
  const uint32_t *n_order;  // device count of `order` entries (nullptr: all rows)
  float *out;
  int n_rows, top_k, N, K, E;
  uint64_t expert_stride;
};

__device__ __forceinline__ float f16_bits_to_float(uint16_t h) {
  return __half2float(*reinterpret_cast<const __half *>(&h));
}

__global__ void __launch_bounds__(kMvWarps * 32) q4_0_mv_kernel(const __grid_constant__ MvParams p) {
  __shared__ __align__(16) uint8_t wrow[kMvWarps][kMvSegBlocks * 18];
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int n_visit = p.n_order ? (int)*p.n_order : p.n_rows;
  for (int i = blockIdx.y; i < n_visit; i += gridDim.y) {
  const int r = p.order ? p.order[i] : i;
  const uint32_t e = __ldg(p.ids + r);
  const int tok = r / p.top_k;
  const int n_base = blockIdx.x * (kMvWarps * kMvRowsPerWarp) + warp * kMvRowsPerWarp;
  const int nblk = p.K / 32;
  if (e >= (uint32_t)p.E) {   // out-of-range id: zero row, and record it
    if (lane < kMvRowsPerWarp && n_base + lane < p.N) p.out[(size_t)r * p.N + n_base + lane] = 0.f;
    if (threadIdx.x == 0 && blockIdx.x == 0) raise_device_error(Q4MM_DEVERR_BAD_EXPERT);
    continue;
  }
  const uint8_t *wexp = p.w + (size_t)e * p.expert_stride;
  const float *xr = p.x + (size_t)tok * p.K;
  const size_t row_bytes = (size_t)nblk * 18;
  float acc[kMvRowsPerWarp];
#pragma unroll
  for (int j = 0; j < kMvRowsPerWarp; ++j) acc[j] = 0.f;

  for (int sb = 0; sb < nblk; sb += kMvSegBlocks) {
    const int seg_blocks = min(kMvSegBlocks, nblk - sb);
    // this lane's x values for blocks sb + lane and sb + lane + 32
    float xv[2][32];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int b = sb + lane + 32 * h;
      if (lane + 32 * h < seg_blocks) {
        const float4 *src = reinterpret_cast<const float4 *>(xr + (size_t)b * 32);
#pragma unroll
        for (int v = 0; v < 8; ++v) {
          const float4 f = __ldg(src + v);
          xv[h][4 * v] = f.x; xv[h][4 * v + 1] = f.y; xv[h][4 * v + 2] = f.z; xv[h][4 * v + 3] = f.w;
        }
      } else {
#pragma unroll
        for (int v = 0; v < 32; ++v) xv[h][v] = 0.f;
      }
    }
    const int seg_bytes = seg_blocks * 18;
    for (int j = 0; j < kMvRowsPerWarp; ++j) {
      const int n = n_base + j;
      if (n >= p.N) break;
      const uint8_t *src = wexp + (size_t)n * row_bytes + (size_t)sb * 18;
      __syncwarp();
      if ((reinterpret_cast<uintptr_t>(src) & 15) == 0 && (seg_bytes & 15) == 0) {
        for (int o = lane * 16; o < seg_bytes; o += 32 * 16)
          *reinterpret_cast<uint4 *>(&wrow[warp][o]) = ldg_stream_v4(src + o);
      } else {
        for (int o = lane; o < seg_bytes; o += 32) wrow[warp][o] = __ldg(src + o);
      }
      __syncwarp();
      float part = 0.f;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int bl = lane + 32 * h;
        if (bl < seg_blocks) {
          const uint16_t *blk = reinterpret_cast<const uint16_t *>(&wrow[warp][bl * 18]);
          const float d = f16_bits_to_float(blk[0]);
          float s = 0.f;
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const uint32_t two = blk[1 + q];   // qs bytes 2q, 2q+1
#pragma unroll
            for (int bb = 0; bb < 2; ++bb) {
              const uint32_t byte = (two >> (8 * bb)) & 0xFFu;
              const int jj = 2 * q + bb;
              s = __fmaf_rn(xv[h][jj], static_cast<float>((int)(byte & 15u) - 8), s);
              s = __fmaf_rn(xv[h][16 + jj], static_cast<float>((int)(byte >> 4) - 8), s);
            }
          }
          part = __fmaf_rn(d, s, part);
        }
      }
      acc[j] += part;
    }
  }
#pragma unroll
  for (int j = 0; j < kMvRowsPerWarp; ++j) {
    float v = acc[j];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    acc[j] = v;
  }
  if (lane < kMvRowsPerWarp) {
    float v = 0.f;
#pragma unroll
    for (int j = 0; j < kMvRowsPerWarp; ++j)
      if (j == lane) v = acc[j];
    if (n_base + lane < p.N) p.out[(size_t)r * p.N + n_base + lane] = v;
  }
  __syncwarp();
  }
}

// Zero the output rows whose id is out of range (the mat-mat path only visits valid rows).
__global__ void zero_invalid_rows_kernel(const uint32_t *__restrict__ ids, int n_rows, int E,
                                         int N, float *__restrict__ out) {
  const int r = blockIdx.x;
  if (r >= n_rows || __ldg(ids + r) < (uint32_t)E) return;
  for (int n = threadIdx.x; n < N; n += blockDim.x) out[(size_t)r * N + n] = 0.f;
}

int route_warps(int E) {
  int w = 8192 / E;
  if (w > kRouteThreads / 32) w = kRouteThreads / 32;
  if (w < 1) w = 1;
  return w;
}

size_t route_smem(int E, int n_warps) { return (size_t)(2 * n_warps * E + E + 1) * 4; }

cudaError_t launch_route_internal(const uint32_t *ids, int n_rows, int E, uint32_t *htpe,
                                  uint32_t *offs, int32_t *hids, uint32_t *n_invalid,
                                  cudaStream_t s, int4 *blk = nullptr, uint32_t *n_blk = nullptr) {
  const int nw = route_warps(E);
  const size_t sm = route_smem(E, nw);
  cudaError_t e = cudaFuncSetAttribute(route_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  if (e != cudaSuccess) return e;
  route_kernel<<<1, nw * 32, sm, s>>>(ids, n_rows, E, nw, htpe, offs, hids, n_invalid, blk, n_blk);
  return cudaGetLastError();
}

}  // namespace

Q4MM_DEFINE_ERROR_READER(read_errors_moe)

cudaError_t launch_q4_0_route(const uint32_t *ids, int n_rows, int n_experts, uint32_t *htpe,
                              int32_t *hids, uint32_t *n_invalid, cudaStream_t s) {
  return launch_route_internal(ids, n_rows, n_experts, htpe, nullptr, hids, n_invalid, s);
}

cudaError_t launch_q4_0_mv(const float *x, const uint8_t *w, const uint32_t *ids, float *out,
                           int n_tokens, int top_k, int N, int K, int n_experts,
                           uint64_t expert_stride, cudaStream_t s) {
  MvParams p{};
  p.x = x; p.w = w; p.ids = ids; p.order = nullptr; p.n_order = nullptr; p.out = out;
  p.n_rows = n_tokens * top_k; p.top_k = top_k; p.N = N; p.K = K; p.E = n_experts;
  p.expert_stride = expert_stride;
  const int rows_cta = kMvWarps * kMvRowsPerWarp;
  dim3 grid((unsigned)((N + rows_cta - 1) / rows_cta), (unsigned)(p.n_rows < 65535 ? p.n_rows : 65535), 1);
  q4_0_mv_kernel<<<grid, kMvWarps * 32, 0, s>>>(p);
  return cudaGetLastError();
}

// Mat-mat form, first version: route, then visit routed rows expert by expert so that
// the CTAs running at any moment share one expert's weights through L2.
cudaError_t launch_q4_0_mm(const float *x, const uint8_t *w, const uint32_t *ids, float *out,
                           int n_tokens, int top_k, int N, int K, int n_experts,
                           uint64_t expert_stride, void *workspace, cudaStream_t s) {
  const int n_rows = n_tokens * top_k;
  const MoeWorkspace L = moe_workspace_layout(n_rows, K, n_experts);
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  uint32_t *htpe = reinterpret_cast<uint32_t *>(ws + L.htpe);
  uint32_t *offs = reinterpret_cast<uint32_t *>(ws + L.offs);
  int32_t *hids = reinterpret_cast<int32_t *>(ws + L.hids);
  uint32_t *invalid = reinterpret_cast<uint32_t *>(ws + L.invalid);
  int4 *blk = reinterpret_cast<int4 *>(ws + L.blk);
  uint32_t *n_blk = reinterpret_cast<uint32_t *>(ws + L.n_blk);
  cudaError_t e = launch_route_internal(ids, n_rows, n_experts, htpe, offs, hids, invalid, s, blk, n_blk);
  if (e != cudaSuccess) return e;
  zero_invalid_rows_kernel<<<(unsigned)n_rows, 128, 0, s>>>(ids, n_rows, n_experts, N, out);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  // Tensor-core form: K a multiple of 256 (whole 144-byte TMA boxes of Q4_0 blocks) and
  // 16-byte aligned expert slabs.
  const bool tc_ok = K % 256 == 0 && expert_stride % 16 == 0 && (reinterpret_cast<uintptr_t>(w) & 15) == 0;
  if (tc_ok)
    return launch_q4_0_mm_tc(x, w, out, n_tokens, top_k, N, K, n_experts, expert_stride, workspace, s);
  MvParams p{};
  p.x = x; p.w = w; p.ids = ids; p.order = hids; p.n_order = offs + n_experts; p.out = out;
  p.n_rows = n_rows; p.top_k = top_k; p.N = N; p.K = K; p.E = n_experts;
  p.expert_stride = expert_stride;
  const int rows_cta = kMvWarps * kMvRowsPerWarp;
  dim3 grid((unsigned)((N + rows_cta - 1) / rows_cta), (unsigned)(n_rows < 65535 ? n_rows : 65535), 1);
  q4_0_mv_kernel<<<grid, kMvWarps * 32, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace q4mm
