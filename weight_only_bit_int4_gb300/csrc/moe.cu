// moe.cu -- GGML Q4_0 expert-routed matmul: routing lists, mat-vec form, and the
// workspace layout of the mat-mat form.
//
// quantized_matmul_id_ggml.rs (mlx-native 0.9.0), module doc: for routed row
// r = token*top_k + slot, expert e = ids[r], out[r][n] = sum_k dequant(W[e][n][k]) * x[token][k].
// Q4_0 block (32 values, 18 bytes): fp16 d, then 16 bytes; element j < 16 is the low nibble
// of byte j, element 16+j its high nibble; value = (q - 8) * d.
//
//  * q4_0_route: the map0 stage of `dispatch_id_mm_for_test` -- per-expert routed counts and
//    ascending routed-row lists, deterministic: one CTA per expert when the ids fit in shared
//    memory, else a stable counting sort in one CTA.
//  * mat-vec (`dispatch_id_mv`, `kernel_mul_mv_id_q4_0_f32`), and its fused SwiGLU form
//    (`quantized_matmul_id_swiglu_q4_0`): on the tensor cores when K % 128 == 0 (one CTA per
//    (routed row, 16 weight rows), K split over its warps), else fp32 FMA on CUDA cores (one
//    CTA per (routed row, 32 weight rows)).
//  * dispatch records of the mat-vec (plan once, replay with new pointers).
#include "q4mm_internal.cuh"

#include <new>

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
// walks the segment again 32 rows at a time, ranking equal ids inside the step by their
// lane order, so the output order equals the input order within each expert.
// ---------------------------------------------------------------------------------------
constexpr int kRouteThreads = 512;

// Mask of the lanes whose key equals this lane's key (32 shuffles; measured much faster
// here than the match instruction).
__device__ __forceinline__ unsigned lanes_with_same_key(uint32_t key) {
  unsigned m = 0;
#pragma unroll
  for (int l = 0; l < 32; ++l) m |= (__shfl_sync(0xFFFFFFFFu, key, l) == key ? 1u : 0u) << l;
  return m;
}

__global__ void __launch_bounds__(kRouteThreads) route_kernel(const uint32_t *__restrict__ ids,
                                                              int n_rows, int E, int n_warps,
                                                              uint32_t *__restrict__ htpe,
                                                              uint32_t *__restrict__ offs,
                                                              int32_t *__restrict__ hids,
                                                              uint32_t *__restrict__ n_invalid,
                                                              int4 *__restrict__ blk = nullptr,
                                                              uint32_t *__restrict__ n_blk = nullptr,
                                                              float *__restrict__ zero_out = nullptr,
                                                              int zero_cols = 0) {
  extern __shared__ uint32_t sm[];
  uint32_t *cnt = sm;                       // [n_warps][E]
  uint32_t *pos = sm + n_warps * E;         // [n_warps][E]
  uint32_t *scan = pos + n_warps * E;       // [E + 1]
  __shared__ uint32_t bad_count;
  griddep_launch_dependents();   // a mat-mat call's next kernel may start its independent work
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int active_warps = min(n_warps, (int)(blockDim.x / 32));
  for (int i = threadIdx.x; i < n_warps * E; i += blockDim.x) cnt[i] = 0;
  if (threadIdx.x == 0) bad_count = 0;
  __syncthreads();

  const int seg = (n_rows + active_warps - 1) / active_warps;
  const int r_begin = warp * seg;
  const int r_end = min(n_rows, r_begin + seg);
  const unsigned lt = (1u << lane) - 1u;
  // Ids are read 8 x 32 at a time with all loads issued before any is used.
  constexpr int kBatch = 8;
  if (warp < active_warps) {
    uint32_t bad = 0;
    for (int base0 = r_begin; base0 < r_end; base0 += 32 * kBatch) {
    uint32_t ev[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int r = base0 + 32 * u + lane;
      ev[u] = r < r_end ? __ldg(ids + r) : 0xFFFFFFFFu;
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int base = base0 + 32 * u;
      if (base >= r_end) break;
      const int r = base + lane;
      const bool in = r < r_end;
      const uint32_t e = ev[u];
      const bool valid = in && e < (uint32_t)E;
      bad += (in && !valid) ? 1u : 0u;
      if (zero_out) {   // rows routed to no expert get zeros (the matmul visits valid rows only)
        unsigned inv = __ballot_sync(0xFFFFFFFFu, in && !valid);
        while (inv) {
          const int l = __ffs(inv) - 1;
          inv &= inv - 1;
          float *row = zero_out + (size_t)(base + l) * zero_cols;
          for (int n = lane; n < zero_cols; n += 32) row[n] = 0.f;
        }
      }
      const unsigned peers = lanes_with_same_key(valid ? e : 0xFFFFFFFFu);
      if (valid && (peers & lt) == 0) cnt[warp * E + e] += __popc(peers);
      __syncwarp();
    }
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
    for (int base0 = r_begin; base0 < r_end; base0 += 32 * kBatch) {
      uint32_t ev[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int r = base0 + 32 * u + lane;
        ev[u] = r < r_end ? __ldg(ids + r) : 0xFFFFFFFFu;
      }
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int base = base0 + 32 * u;
        if (base >= r_end) break;
        const int r = base + lane;
        const bool in = r < r_end;
        const uint32_t e = ev[u];
        const bool valid = in && e < (uint32_t)E;
        const unsigned peers = lanes_with_same_key(valid ? e : 0xFFFFFFFFu);
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
}

// ---------------------------------------------------------------------------------------
// Mat-vec: CTA = (routed row, 32 weight rows).  4 warps x 8 weight rows.  Lane l takes
// blocks l, l+32, ... of a K segment; its x values for those blocks stay in registers
// across the warp's 8 weight rows.  Weight rows are first copied to shared memory with
// coalesced loads (18- and 34-byte blocks are not 4-byte aligned in global memory).
// BT selects the block type: Q4_0 (18 bytes: fp16 d, 16 bytes of nibbles, value (q - 8) d)
// or Q8_0 (34 bytes: fp16 d, 32 signed bytes, value q d).
// ---------------------------------------------------------------------------------------
constexpr int kMvWarps = 4;
constexpr int kMvRowsPerWarp = 8;
constexpr int kMvSegBlocks = 64;   // K segment: 64 blocks = 2048 values
__host__ __device__ constexpr int block_bytes(int bt) { return bt == kQ8_0 ? 34 : 18; }

struct MvParams {
  const float *x;           // x [n_tokens, K]; the SwiGLU form: gate [n_rows, K]
  const float *up;          // the SwiGLU form: up [n_rows, K] (nullptr otherwise)
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

// The vector a routed row multiplies: x itself, or silu(gate) * up in fp32 (SwiGLU form).
__device__ __forceinline__ float silu_f32(float z) { return z / (1.0f + expf(-z)); }

template <bool SWIGLU>
__device__ __forceinline__ float4 mv_input4(const float *xr, const float *ur, int off) {
  const float4 g = __ldg(reinterpret_cast<const float4 *>(xr + off));
  if constexpr (!SWIGLU) {
    return g;
  } else {
    const float4 u = __ldg(reinterpret_cast<const float4 *>(ur + off));
    return make_float4(silu_f32(g.x) * u.x, silu_f32(g.y) * u.y, silu_f32(g.z) * u.z, silu_f32(g.w) * u.w);
  }
}

template <bool SWIGLU, int BT>
__global__ void __launch_bounds__(kMvWarps * 32) routed_mv_kernel(const __grid_constant__ MvParams p) {
  constexpr int kBB = block_bytes(BT);
  __shared__ __align__(16) uint8_t wrow[kMvWarps][kMvSegBlocks * kBB];
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
  const float *xr = p.x + (SWIGLU ? (size_t)r : (size_t)tok) * p.K;
  const float *ur = SWIGLU ? p.up + (size_t)r * p.K : nullptr;
  const size_t row_bytes = (size_t)nblk * kBB;
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
#pragma unroll
        for (int v = 0; v < 8; ++v) {
          const float4 f = mv_input4<SWIGLU>(xr, ur, b * 32 + 4 * v);
          xv[h][4 * v] = f.x; xv[h][4 * v + 1] = f.y; xv[h][4 * v + 2] = f.z; xv[h][4 * v + 3] = f.w;
        }
      } else {
#pragma unroll
        for (int v = 0; v < 32; ++v) xv[h][v] = 0.f;
      }
    }
    const int seg_bytes = seg_blocks * kBB;
    for (int j = 0; j < kMvRowsPerWarp; ++j) {
      const int n = n_base + j;
      if (n >= p.N) break;
      const uint8_t *src = wexp + (size_t)n * row_bytes + (size_t)sb * kBB;
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
          const uint16_t *blk = reinterpret_cast<const uint16_t *>(&wrow[warp][bl * kBB]);
          const float d = f16_bits_to_float(blk[0]);
          float s = 0.f;
          if constexpr (BT == kQ8_0) {
#pragma unroll
            for (int q = 0; q < 16; ++q) {
              const uint32_t two = blk[1 + q];   // qs bytes 2q, 2q+1: elements 2q, 2q+1
              s = __fmaf_rn(xv[h][2 * q], static_cast<float>(static_cast<int8_t>(two & 0xFFu)), s);
              s = __fmaf_rn(xv[h][2 * q + 1], static_cast<float>(static_cast<int8_t>(two >> 8)), s);
            }
          } else {
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

// ---------------------------------------------------------------------------------------
// Routing, parallel form (used when n_experts * n_rows is moderate): CTA e owns expert e.
// Every CTA histograms all ids in shared memory, which gives it the start of its list
// (the number of valid ids below e) and its token-block base, with no cross-CTA traffic;
// it then places the rows of expert e in ascending order: each warp scans a contiguous
// segment with ballots, and a scan over the warps' counts orders the segments.
// ---------------------------------------------------------------------------------------
constexpr int kRouteParThreads = 256;
constexpr size_t kRouteParSmemMax = 48 * 1024;   // E counts + all ids, without an opt-in

__global__ void __launch_bounds__(kRouteParThreads) route_par_kernel(
    const uint32_t *__restrict__ ids, int n_rows, int E, uint32_t *__restrict__ htpe,
    uint32_t *__restrict__ offs, int32_t *__restrict__ hids, uint32_t *__restrict__ n_invalid,
    int4 *__restrict__ blk, uint32_t *__restrict__ n_blk, float *__restrict__ zero_out, int zero_cols) {
  extern __shared__ uint32_t hist[];                 // [E] counts, then the ids [n_rows]
  __shared__ uint32_t warp_cnt[kRouteParThreads / 32];
  __shared__ uint32_t s_less, s_blkbase, s_total, s_total_blk;
  griddep_launch_dependents();   // a mat-mat call's next kernel may start its independent work
  const int e = blockIdx.x;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const unsigned lt = (1u << lane) - 1u;
  uint32_t *s_ids = hist + E;
  for (int i = threadIdx.x; i < E; i += blockDim.x) hist[i] = 0;
  {   // stage the ids: four independent loads in flight per thread
    int r = threadIdx.x;
    for (; r + 3 * kRouteParThreads < n_rows; r += 4 * kRouteParThreads) {
      const uint32_t a = __ldg(ids + r), b = __ldg(ids + r + kRouteParThreads),
                     c = __ldg(ids + r + 2 * kRouteParThreads), d = __ldg(ids + r + 3 * kRouteParThreads);
      s_ids[r] = a;
      s_ids[r + kRouteParThreads] = b;
      s_ids[r + 2 * kRouteParThreads] = c;
      s_ids[r + 3 * kRouteParThreads] = d;
    }
    for (; r < n_rows; r += kRouteParThreads) s_ids[r] = __ldg(ids + r);
  }
  __syncthreads();
  // Histogram.  Warp w reads 32-row chunks w, w+8, ...; a chunk's ids routed to no expert
  // are zeroed in the output by CTA (chunk mod E), so that work is spread over the grid.
  for (int base = warp * 32; base < n_rows; base += blockDim.x) {
    const int r = base + lane;
    const uint32_t id = r < n_rows ? s_ids[r] : 0u;
    const bool bad = r < n_rows && id >= (uint32_t)E;
    if (r < n_rows && !bad) atomicAdd(&hist[id], 1u);
    if (zero_out != nullptr && (base / 32) % E == e) {
      unsigned m = __ballot_sync(0xFFFFFFFFu, bad);
      while (m) {
        const int rr = base + __ffs(m) - 1;
        m &= m - 1;
        for (int n = lane; n < zero_cols; n += 32) zero_out[(size_t)rr * zero_cols + n] = 0.f;
      }
    }
  }
  __syncthreads();
  if (warp == 0) {   // prefix of counts and of block counts below e (and totals)
    uint32_t less = 0, bbase = 0, tot = 0, tblk = 0;
    for (int i = lane; i < E; i += 32) {
      const uint32_t c = hist[i], b = (c + kMoeTokBlock - 1) / kMoeTokBlock;
      tot += c;
      tblk += b;
      if (i < e) { less += c; bbase += b; }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      less += __shfl_xor_sync(0xFFFFFFFFu, less, o);
      bbase += __shfl_xor_sync(0xFFFFFFFFu, bbase, o);
      tot += __shfl_xor_sync(0xFFFFFFFFu, tot, o);
      tblk += __shfl_xor_sync(0xFFFFFFFFu, tblk, o);
    }
    if (lane == 0) { s_less = less; s_blkbase = bbase; s_total = tot; s_total_blk = tblk; }
  }
  // rows of expert e: warp w scans rows [w*seg, (w+1)*seg)
  const int nw = blockDim.x / 32;
  const int seg = ((n_rows + nw - 1) / nw + 31) / 32 * 32;
  const int r0 = warp * seg, r1 = min(n_rows, r0 + seg);
  uint32_t mine = 0;
  for (int b = r0; b < r1; b += 32) {
    const int r = b + lane;
    const bool hit = r < r1 && s_ids[r] == (uint32_t)e;
    mine += __popc(__ballot_sync(0xFFFFFFFFu, hit));
  }
  if (lane == 0) warp_cnt[warp] = mine;
  __syncthreads();
  uint32_t pos = s_less;
  for (int w = 0; w < warp; ++w) pos += warp_cnt[w];
  for (int b = r0; b < r1; b += 32) {
    const int r = b + lane;
    const bool hit = r < r1 && s_ids[r] == (uint32_t)e;
    const unsigned m = __ballot_sync(0xFFFFFFFFu, hit);
    if (hit) hids[pos + __popc(m & lt)] = r;
    pos += __popc(m);
  }
  if (threadIdx.x == 0) {
    const uint32_t c = hist[e];
    htpe[e] = c;
    if (offs) offs[e] = s_less;
    if (blk) {
      for (uint32_t b0 = 0, k = 0; b0 < c; b0 += kMoeTokBlock, ++k)
        blk[s_blkbase + k] = make_int4(e, (int)(s_less + b0), (int)min((uint32_t)kMoeTokBlock, c - b0), 0);
    }
    if (e == E - 1) {
      if (offs) offs[E] = s_total;
      if (n_blk) *n_blk = s_total_blk;
      if (n_invalid) *n_invalid = (uint32_t)n_rows - s_total;
      if ((uint32_t)n_rows != s_total) raise_device_error(Q4MM_DEVERR_BAD_EXPERT);
    }
  }
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
                                  cudaStream_t s, int4 *blk = nullptr, uint32_t *n_blk = nullptr,
                                  float *zero_out = nullptr, int zero_cols = 0) {
  if ((size_t)(E + n_rows) * 4 <= kRouteParSmemMax) {
    route_par_kernel<<<(unsigned)E, kRouteParThreads, (size_t)(E + n_rows) * 4, s>>>(ids, n_rows, E, htpe, offs, hids,
                                                                          n_invalid, blk, n_blk, zero_out, zero_cols);
    return cudaGetLastError();
  }
  const int nw = route_warps(E);
  const size_t sm = route_smem(E, nw);
  cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void *>(route_kernel), (int)sm);
  if (e != cudaSuccess) return e;
  route_kernel<<<1, nw * 32, sm, s>>>(ids, n_rows, E, nw, htpe, offs, hids, n_invalid, blk, n_blk, zero_out,
                                      zero_cols);
  return cudaGetLastError();
}

}  // namespace

Q4MM_DEFINE_ERROR_READER(read_errors_moe)

cudaError_t launch_q4_0_route(const uint32_t *ids, int n_rows, int n_experts, uint32_t *htpe,
                              int32_t *hids, uint32_t *n_invalid, cudaStream_t s) {
  return launch_route_internal(ids, n_rows, n_experts, htpe, nullptr, hids, n_invalid, s);
}

// ---------------------------------------------------------------------------------------
// Mat-vec form on the tensor cores (K % 128 == 0, 8-byte aligned rows).
//
// A CTA owns routed row r = token * top_k + slot and 16 weight rows of expert ids[r]; its
// KS warps take consecutive K slices.  Each warp streams its slice as chunks of up to 8
// Q4_0 blocks per row (144 bytes; the last chunk of a row holds 4 blocks when K % 256 != 0)
// through a private cp.async ring -- 16-byte copies when every row is 16-byte aligned
// (K % 256 == 0), else 8-byte copies -- and stages its slice of x rounded to bf16 together
// with the per-block sums of those bf16 values.
//
// The product follows the M <= 4 INT4 decode kernel: with one token, B column j of an
// m16n8k16 step carries x on the k-slots of Q4_0 block j (j < 4) and zeros elsewhere, so
// the tensor core forms D = sum (128 + q) * x per (row, block) exactly; the codes enter as
// bf16 128 + q with one LOP3.  Then, in fp32,
//     sum_k (q - 8) d x_k = d * D - 136 * d * X,   X = sum of the block's bf16 x,
// which is the block's contribution with its terms regrouped.  Word m of a block's qs
// holds elements 4m..4m+3 (low nibbles) and 4m+16..4m+19 (high nibbles); the decode pairs
// are (4m, 4m+2), (4m+16, 4m+18), (4m+1, 4m+3), (4m+17, 4m+19) and x is staged in that order.
//
// SWIGLU (quantized_matmul_id_swiglu_q4_0): the vector of routed row r is
// silu(gate[r][k]) * up[r][k], formed in fp32 while x is staged; gate and up have one row
// per routed row.  Everything after the staging is the same.
// ---------------------------------------------------------------------------------------
constexpr int kMvcDepth = 4;                   // chunk stages per warp (at most)
constexpr int kMvcRow = 144;                   // bytes per weight row per chunk (8 blocks)
constexpr int kMvcChunk = 16 * kMvcRow;        // 2304 bytes per chunk stage

__host__ __device__ inline int mvc_depth(int maxc) { return maxc < kMvcDepth ? maxc : kMvcDepth; }
__host__ __device__ inline size_t mvc_warp_bytes(int maxc) {
  return (size_t)mvc_depth(maxc) * kMvcChunk + (size_t)maxc * 8 * 64 + (size_t)maxc * 8 * 4;
}

template <int PIECE>
__device__ __forceinline__ void cp_async_piece(uint32_t dst, const void *src, uint32_t src_bytes) {
  if constexpr (PIECE == 16)
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
  else
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}

// One chunk of 16 weight rows into a ring stage of ROW bytes per row: PIECES copies of PIECE
// bytes per row (compile-time counts, so the row/piece split of an item index is a multiply,
// not a divide).
template <int PIECES, int PIECE, int ROW = kMvcRow>
__device__ __forceinline__ void mv_copy_rows(uint32_t slot, const uint8_t *src, size_t row_bytes, int row0,
                                             int N, int lane) {
#pragma unroll 1
  for (int i = lane; i < 16 * PIECES; i += 32) {
    const int rr = i / PIECES, pc = i - rr * PIECES;
    const bool ok = row0 + rr < N;
    cp_async_piece<PIECE>(slot + (uint32_t)(rr * ROW + pc * PIECE),
                          ok ? src + (size_t)(row0 + rr) * row_bytes + pc * PIECE : src, ok ? (uint32_t)PIECE : 0u);
  }
}

// A warp's x slice of nblk_w 32-element blocks in the decode's k order: item (block, m) is 16
// bytes of bf16 pairs (x[4m], x[4m+2]), (x[4m+16], x[4m+18]), (x[4m+1], x[4m+3]),
// (x[4m+17], x[4m+19]); xsum[block] = the sum of the block's bf16 values in fp32.  The
// SwiGLU form stages silu(gate) * up.
template <bool SWIGLU>
__device__ __forceinline__ void mv_stage_x(uint8_t *xs, float *xsum, const float *xr, const float *ur, int nblk_w,
                                           int lane) {
  for (int it = lane; it < ((nblk_w * 4 + 31) & ~31); it += 32) {   // 4 consecutive lanes share a block
    const int blk = it >> 2, m = it & 3;
    const bool in = blk < nblk_w;
    float4 lo = make_float4(0.f, 0.f, 0.f, 0.f), hi = lo;
    if (in) {
      lo = mv_input4<SWIGLU>(xr, ur, blk * 32 + 4 * m);
      hi = mv_input4<SWIGLU>(xr, ur, blk * 32 + 16 + 4 * m);
    }
    const uint32_t p0 = pack_bf16x2(lo.x, lo.z), p1 = pack_bf16x2(hi.x, hi.z);
    const uint32_t p2 = pack_bf16x2(lo.y, lo.w), p3 = pack_bf16x2(hi.y, hi.w);
    if (in) *reinterpret_cast<uint4 *>(xs + (size_t)blk * 64 + m * 16) = make_uint4(p0, p1, p2, p3);
    float sum = 0.f;
    const uint32_t pv[4] = {p0, p2, p1, p3};
#pragma unroll
    for (int i = 0; i < 4; ++i) sum += __uint_as_float(pv[i] << 16) + __uint_as_float(pv[i] & 0xFFFF0000u);
    sum += __shfl_xor_sync(0xFFFFFFFFu, sum, 1);
    sum += __shfl_xor_sync(0xFFFFFFFFu, sum, 2);
    if (in && m == 0) xsum[blk] = sum;
  }
  __syncwarp();
}

template <int KS, bool SWIGLU, int PIECE>
__global__ void __launch_bounds__(KS * 32) q4_0_mv_mma_kernel(const __grid_constant__ MvParams p, int maxc) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr int kPiecesFull = kMvcRow / PIECE;   // copies per row of an 8-block chunk
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int g = lane / 4, t = lane % 4;
  const int depth = mvc_depth(maxc);
  const size_t wb = mvc_warp_bytes(maxc);
  uint8_t *ring = smem + (size_t)warp * wb;
  uint8_t *xs = ring + (size_t)depth * kMvcChunk;                      // [maxc * 8 blocks][4][16 B]
  float *xsum = reinterpret_cast<float *>(xs + (size_t)maxc * 8 * 64);  // [maxc * 8]
  float *red = reinterpret_cast<float *>(smem + (size_t)KS * wb);       // [KS][16]
  const uint32_t ring_s = smem_u32(ring);
  const int S4 = p.K / 128;                       // 4-block sub-chunks per row
  const int C = (S4 + 1) / 2;                     // chunks of (up to) 8 blocks
  const int c_begin = (int)(((long long)warp * C) / KS);
  const int c_end = (int)(((long long)(warp + 1) * C) / KS);
  const int nch = c_end - c_begin;
  const int nblk_w = min(8 * nch, p.K / 32 - 8 * c_begin);   // blocks in this warp's slice
  const int row0 = blockIdx.x * 16;
  const size_t row_bytes = (size_t)(p.K / 32) * 18;

  for (int r = blockIdx.y; r < p.n_rows; r += gridDim.y) {
    const uint32_t e = __ldg(p.ids + r);
    if (e >= (uint32_t)p.E) {   // routed to no expert: zero row, and record it
      if (threadIdx.x < 16 && row0 + (int)threadIdx.x < p.N) p.out[(size_t)r * p.N + row0 + threadIdx.x] = 0.f;
      if (threadIdx.x == 0 && blockIdx.x == 0) raise_device_error(Q4MM_DEVERR_BAD_EXPERT);
      continue;
    }
    const uint8_t *wexp = p.w + (size_t)e * p.expert_stride;
    auto issue = [&](int c) {
      const uint32_t slot = ring_s + (uint32_t)((c % kMvcDepth) * kMvcChunk);
      const int a = c_begin + c;
      const uint8_t *src = wexp + (size_t)a * kMvcRow;
      if (2 * a + 1 < S4)
        mv_copy_rows<kPiecesFull, PIECE>(slot, src, row_bytes, row0, p.N, lane);
      else   // 4-block tail chunk
        mv_copy_rows<kPiecesFull / 2, PIECE>(slot, src, row_bytes, row0, p.N, lane);
    };
#pragma unroll
    for (int i = 0; i < kMvcDepth - 1; ++i) {
      if (i < nch) issue(i);
      cp_async_commit();
    }

    // x slice: item (block, m) -> 16 bytes of bf16 pairs in decode order; block sums.
    const size_t xrow = SWIGLU ? (size_t)r : (size_t)(r / p.top_k);
    const float *xr = p.x + xrow * p.K + (size_t)c_begin * 256;
    const float *ur = SWIGLU ? p.up + xrow * p.K + (size_t)c_begin * 256 : nullptr;
    mv_stage_x<SWIGLU>(xs, xsum, xr, ur, nblk_w, lane);

    const bool bl = g == t;   // B column g = block g of the sub-chunk (one token: g < 4)
    float acc[2] = {0.f, 0.f};
    for (int c = 0; c < nch; ++c) {
      if (c + kMvcDepth - 1 < nch) issue(c + kMvcDepth - 1);
      cp_async_commit();
      cp_async_wait<kMvcDepth - 1>();
      __syncwarp();
      const uint8_t *slot = ring + (c % kMvcDepth) * kMvcChunk;
      const int nsub = 2 * (c_begin + c) + 1 < S4 ? 2 : 1;
      for (int sc = 0; sc < nsub; ++sc) {   // sub-chunks of 4 blocks; quad lane t decodes block 4 sc + t
        const int bk = 4 * sc + t;
        const int off = 18 * bk + 2;                    // qs of block bk within a row
        const uint32_t sel = (off & 2) ? 0x5432u : 0x3210u;
        uint32_t qs[2][4];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint32_t *u = reinterpret_cast<const uint32_t *>(slot + (g + 8 * h) * kMvcRow + (off & ~3));
          uint32_t v[5];
#pragma unroll
          for (int i = 0; i < 5; ++i) v[i] = u[i];
#pragma unroll
          for (int i = 0; i < 4; ++i) qs[h][i] = prmt(v[i], v[i + 1], sel);
        }
        uint4 xb[4];
        const uint8_t *xl = xs + (size_t)(c * 8 + bk) * 64;
#pragma unroll
        for (int m = 0; m < 4; ++m)
          xb[m] = bl ? *reinterpret_cast<const uint4 *>(xl + m * 16) : make_uint4(0, 0, 0, 0);
        float D[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          const uint32_t w0 = qs[0][m], w1 = qs[1][m];
          constexpr uint32_t kMask = 0x000F000Fu, kMagic = 0x43004300u;   // bf16 128 + q
          const uint32_t a0[4] = {and_or(w0, kMask, kMagic), and_or(w1, kMask, kMagic),
                                  and_or(w0 >> 4, kMask, kMagic), and_or(w1 >> 4, kMask, kMagic)};
          const uint32_t a1[4] = {and_or(w0 >> 8, kMask, kMagic), and_or(w1 >> 8, kMask, kMagic),
                                  and_or(w0 >> 12, kMask, kMagic), and_or(w1 >> 12, kMask, kMagic)};
          mma_bf16_16816(D, a0, xb[m].x, xb[m].y);
          mma_bf16_16816(D, a1, xb[m].z, xb[m].w);
        }
        // columns 2t, 2t+1 = blocks 4 sc + 2t, +1 for t < 2; zero columns for t >= 2
        const int ba = 4 * sc + 2 * (t & 1);
        const float2 X = *reinterpret_cast<const float2 *>(xsum + c * 8 + ba);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint8_t *rowp = slot + (g + 8 * h) * kMvcRow;
          const float da = f16_bits_to_float(*reinterpret_cast<const uint16_t *>(rowp + 18 * ba));
          const float db = f16_bits_to_float(*reinterpret_cast<const uint16_t *>(rowp + 18 * (ba + 1)));
          float a = acc[h];
          a = __fmaf_rn(da, D[2 * h], a);
          a = __fmaf_rn(-136.f * da, X.x, a);
          a = __fmaf_rn(db, D[2 * h + 1], a);
          a = __fmaf_rn(-136.f * db, X.y, a);
          acc[h] = t < 2 ? a : 0.f;
        }
      }
      __syncwarp();
    }
    cp_async_wait<0>();
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const float v = acc[h] + __shfl_xor_sync(0xFFFFFFFFu, acc[h], 1);
      if (t == 0) red[warp * 16 + g + 8 * h] = v;
    }
    __syncthreads();
    if (threadIdx.x < 16) {
      float v = red[threadIdx.x];
#pragma unroll
      for (int w = 1; w < KS; ++w) v += red[w * 16 + threadIdx.x];
      if (row0 + (int)threadIdx.x < p.N) p.out[(size_t)r * p.N + row0 + threadIdx.x] = v;
    }
    __syncthreads();   // ring, x and red are reused by the next routed row
  }
}

// ---------------------------------------------------------------------------------------
// Q8_0 mat-vec on the tensor cores (K % 128 == 0, 8-byte aligned rows): the layout of
// q4_0_mv_mma_kernel with 272-byte row pieces (8 Q8_0 blocks; 136 bytes for a 4-block tail).
//
// A signed byte q is split into two nibble planes that enter the MMA exactly as bf16:
// lo = q & 15 as 128 + lo, and hi = q >> 4 (arithmetic, -8..7) as 136 + hi (the high nibble
// with its top bit flipped).  q = 16 hi + lo, so per (row, block)
//     sum_k q x = 16 D_hi + D_lo - 2304 X,   D_lo = sum (128 + lo) x,  D_hi = sum (136 + hi) x,
// with X the sum of the block's bf16 x; both D are fp32 sums of exact products.
// Qs word m of a block holds elements 4m..4m+3, word m + 4 elements 4m+16..4m+19, so each
// plane's MMA k-slots take the pairs (4m, 4m+2), (4m+16, 4m+18), (4m+1, 4m+3),
// (4m+17, 4m+19): the x order the Q4_0 kernel stages.
// ---------------------------------------------------------------------------------------
constexpr int kMv8Row = 272;                   // bytes per weight row per chunk (8 Q8_0 blocks)
constexpr int kMv8Chunk = 16 * kMv8Row;        // 4352 bytes per chunk stage

__host__ __device__ inline size_t mv8_warp_bytes(int maxc) {
  return (size_t)mvc_depth(maxc) * kMv8Chunk + (size_t)maxc * 8 * 64 + (size_t)maxc * 8 * 4;
}

template <int KS, int PIECE>
__global__ void __launch_bounds__(KS * 32) q8_0_mv_mma_kernel(const __grid_constant__ MvParams p, int maxc) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr int kPiecesFull = kMv8Row / PIECE;   // copies per row of an 8-block chunk
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int g = lane / 4, t = lane % 4;
  const int depth = mvc_depth(maxc);
  const size_t wb = mv8_warp_bytes(maxc);
  uint8_t *ring = smem + (size_t)warp * wb;
  uint8_t *xs = ring + (size_t)depth * kMv8Chunk;                      // [maxc * 8 blocks][4][16 B]
  float *xsum = reinterpret_cast<float *>(xs + (size_t)maxc * 8 * 64);  // [maxc * 8]
  float *red = reinterpret_cast<float *>(smem + (size_t)KS * wb);       // [KS][16]
  const uint32_t ring_s = smem_u32(ring);
  const int S4 = p.K / 128;                       // 4-block sub-chunks per row
  const int C = (S4 + 1) / 2;                     // chunks of (up to) 8 blocks
  const int c_begin = (int)(((long long)warp * C) / KS);
  const int c_end = (int)(((long long)(warp + 1) * C) / KS);
  const int nch = c_end - c_begin;
  const int nblk_w = min(8 * nch, p.K / 32 - 8 * c_begin);   // blocks in this warp's slice
  const int row0 = blockIdx.x * 16;
  const size_t row_bytes = (size_t)(p.K / 32) * 34;

  for (int r = blockIdx.y; r < p.n_rows; r += gridDim.y) {
    const uint32_t e = __ldg(p.ids + r);
    if (e >= (uint32_t)p.E) {   // routed to no expert: zero row, and record it
      if (threadIdx.x < 16 && row0 + (int)threadIdx.x < p.N) p.out[(size_t)r * p.N + row0 + threadIdx.x] = 0.f;
      if (threadIdx.x == 0 && blockIdx.x == 0) raise_device_error(Q4MM_DEVERR_BAD_EXPERT);
      continue;
    }
    const uint8_t *wexp = p.w + (size_t)e * p.expert_stride;
    auto issue = [&](int c) {
      const uint32_t slot = ring_s + (uint32_t)((c % kMvcDepth) * kMv8Chunk);
      const int a = c_begin + c;
      const uint8_t *src = wexp + (size_t)a * kMv8Row;
      if (2 * a + 1 < S4)
        mv_copy_rows<kPiecesFull, PIECE, kMv8Row>(slot, src, row_bytes, row0, p.N, lane);
      else   // 4-block tail chunk
        mv_copy_rows<kPiecesFull / 2, PIECE, kMv8Row>(slot, src, row_bytes, row0, p.N, lane);
    };
#pragma unroll
    for (int i = 0; i < kMvcDepth - 1; ++i) {
      if (i < nch) issue(i);
      cp_async_commit();
    }

    const float *xr = p.x + (size_t)(r / p.top_k) * p.K + (size_t)c_begin * 256;
    mv_stage_x<false>(xs, xsum, xr, nullptr, nblk_w, lane);

    const bool bl = g == t;   // B column g = block g of the sub-chunk (one token: g < 4)
    float acc[2] = {0.f, 0.f};
    for (int c = 0; c < nch; ++c) {
      if (c + kMvcDepth - 1 < nch) issue(c + kMvcDepth - 1);
      cp_async_commit();
      cp_async_wait<kMvcDepth - 1>();
      __syncwarp();
      const uint8_t *slot = ring + (c % kMvcDepth) * kMv8Chunk;
      const int nsub = 2 * (c_begin + c) + 1 < S4 ? 2 : 1;
      for (int sc = 0; sc < nsub; ++sc) {   // sub-chunks of 4 blocks; quad lane t decodes block 4 sc + t
        const int bk = 4 * sc + t;
        const int off = 34 * bk + 2;                    // qs of block bk within a row
        const uint32_t sel = (off & 2) ? 0x5432u : 0x3210u;
        uint32_t qs[2][8];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint32_t *u = reinterpret_cast<const uint32_t *>(slot + (g + 8 * h) * kMv8Row + (off & ~3));
          uint32_t v[9];
#pragma unroll
          for (int i = 0; i < 9; ++i) v[i] = u[i];
#pragma unroll
          for (int i = 0; i < 8; ++i) qs[h][i] = prmt(v[i], v[i + 1], sel);
        }
        uint4 xb[4];
        const uint8_t *xl = xs + (size_t)(c * 8 + bk) * 64;
#pragma unroll
        for (int m = 0; m < 4; ++m)
          xb[m] = bl ? *reinterpret_cast<const uint4 *>(xl + m * 16) : make_uint4(0, 0, 0, 0);
        float Dl[4] = {0.f, 0.f, 0.f, 0.f}, Dh[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          const uint32_t w0 = qs[0][m], w1 = qs[1][m], v0 = qs[0][m + 4], v1 = qs[1][m + 4];
          constexpr uint32_t kMask = 0x000F000Fu, kMagic = 0x43004300u;   // bf16 128 + lo
          constexpr uint32_t kFlip = 0x43084308u;                         // bf16 136 + hi
          const uint32_t l0[4] = {and_or(w0, kMask, kMagic), and_or(w1, kMask, kMagic),
                                  and_or(v0, kMask, kMagic), and_or(v1, kMask, kMagic)};
          const uint32_t l1[4] = {and_or(w0 >> 8, kMask, kMagic), and_or(w1 >> 8, kMask, kMagic),
                                  and_or(v0 >> 8, kMask, kMagic), and_or(v1 >> 8, kMask, kMagic)};
          const uint32_t h0[4] = {((w0 >> 4) & kMask) ^ kFlip, ((w1 >> 4) & kMask) ^ kFlip,
                                  ((v0 >> 4) & kMask) ^ kFlip, ((v1 >> 4) & kMask) ^ kFlip};
          const uint32_t h1[4] = {((w0 >> 12) & kMask) ^ kFlip, ((w1 >> 12) & kMask) ^ kFlip,
                                  ((v0 >> 12) & kMask) ^ kFlip, ((v1 >> 12) & kMask) ^ kFlip};
          mma_bf16_16816(Dl, l0, xb[m].x, xb[m].y);
          mma_bf16_16816(Dl, l1, xb[m].z, xb[m].w);
          mma_bf16_16816(Dh, h0, xb[m].x, xb[m].y);
          mma_bf16_16816(Dh, h1, xb[m].z, xb[m].w);
        }
        // columns 2t, 2t+1 = blocks 4 sc + 2t, +1 for t < 2; zero columns for t >= 2
        const int ba = 4 * sc + 2 * (t & 1);
        const float2 X = *reinterpret_cast<const float2 *>(xsum + c * 8 + ba);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint8_t *rowp = slot + (g + 8 * h) * kMv8Row;
          const float da = f16_bits_to_float(*reinterpret_cast<const uint16_t *>(rowp + 34 * ba));
          const float db = f16_bits_to_float(*reinterpret_cast<const uint16_t *>(rowp + 34 * (ba + 1)));
          float a = acc[h];
          a = __fmaf_rn(da, __fmaf_rn(16.f, Dh[2 * h], Dl[2 * h]), a);
          a = __fmaf_rn(-2304.f * da, X.x, a);
          a = __fmaf_rn(db, __fmaf_rn(16.f, Dh[2 * h + 1], Dl[2 * h + 1]), a);
          a = __fmaf_rn(-2304.f * db, X.y, a);
          acc[h] = t < 2 ? a : 0.f;
        }
      }
      __syncwarp();
    }
    cp_async_wait<0>();
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const float v = acc[h] + __shfl_xor_sync(0xFFFFFFFFu, acc[h], 1);
      if (t == 0) red[warp * 16 + g + 8 * h] = v;
    }
    __syncthreads();
    if (threadIdx.x < 16) {
      float v = red[threadIdx.x];
#pragma unroll
      for (int w = 1; w < KS; ++w) v += red[w * 16 + threadIdx.x];
      if (row0 + (int)threadIdx.x < p.N) p.out[(size_t)r * p.N + row0 + threadIdx.x] = v;
    }
    __syncthreads();   // ring, x and red are reused by the next routed row
  }
}

// A planned mat-vec launch: kernel, grid, shared memory and the shape part of the
// parameters (also kept as a dispatch record and replayed with new pointers).
struct MvSpec {
  const void *fn = nullptr;
  dim3 grid, block;
  size_t smem = 0;
  int maxc = 0;          // tensor-core kernel: chunks per warp (its second argument)
  bool mma = false;
  int w_align = 4;       // alignment the weight pointer must keep for this kernel
  MvParams params{};
};

cudaError_t run_mv_spec(const MvSpec &sp, const MvParams &p, cudaStream_t s) {
  MvParams pp = p;
  int maxc = sp.maxc;
  void *args[] = {&pp, &maxc};
  return cudaLaunchKernel(sp.fn, sp.grid, sp.block, args, sp.smem, s);
}

template <bool SWIGLU, int PIECE>
cudaError_t plan_mv_mma_typed(const MvParams &p, int ks, int maxc, size_t smem, MvSpec *sp) {
  auto kern = ks == 4 ? q4_0_mv_mma_kernel<4, SWIGLU, PIECE>
            : ks == 2 ? q4_0_mv_mma_kernel<2, SWIGLU, PIECE> : q4_0_mv_mma_kernel<1, SWIGLU, PIECE>;
  cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void *>(kern), (int)smem);
  if (e != cudaSuccess) return e;
  sp->fn = reinterpret_cast<const void *>(kern);
  sp->grid = dim3((unsigned)((p.N + 15) / 16), (unsigned)(p.n_rows < 65535 ? p.n_rows : 65535), 1);
  sp->block = dim3(ks * 32);
  sp->smem = smem;
  sp->maxc = maxc;
  sp->mma = true;
  sp->w_align = PIECE;
  sp->params = p;
  return cudaSuccess;
}

// Tensor-core mat-vec when the rows allow it (K % 128 == 0; 16-byte copies need K % 256 == 0
// and 16-byte aligned slabs, 8-byte copies 8-byte aligned ones), else the fp32 FMA kernel.
template <bool SWIGLU>
cudaError_t plan_mv_any(const MvParams &p, MvSpec *sp) {
  const uintptr_t wa = reinterpret_cast<uintptr_t>(p.w);
  const bool a16 = p.K % 256 == 0 && p.expert_stride % 16 == 0 && (wa & 15) == 0;
  const bool a8 = p.K % 128 == 0 && p.expert_stride % 8 == 0 && (wa & 7) == 0;
  if (a16 || a8) {
    const int C = (p.K / 128 + 1) / 2;
    const int ks = C >= 4 ? 4 : (C >= 2 ? 2 : 1);
    const int maxc = (C + ks - 1) / ks;
    const size_t smem = (size_t)ks * mvc_warp_bytes(maxc) + (size_t)ks * 16 * 4;
    if (smem <= 227 * 1024)
      return a16 ? plan_mv_mma_typed<SWIGLU, 16>(p, ks, maxc, smem, sp)
                 : plan_mv_mma_typed<SWIGLU, 8>(p, ks, maxc, smem, sp);
  }
  const int rows_cta = kMvWarps * kMvRowsPerWarp;
  sp->fn = reinterpret_cast<const void *>(routed_mv_kernel<SWIGLU, kQ4_0>);
  sp->grid = dim3((unsigned)((p.N + rows_cta - 1) / rows_cta), (unsigned)(p.n_rows < 65535 ? p.n_rows : 65535), 1);
  sp->block = dim3(kMvWarps * 32);
  sp->smem = 0;
  sp->maxc = 0;
  sp->mma = false;
  sp->w_align = 1;
  sp->params = p;
  return cudaSuccess;
}

template <bool SWIGLU>
cudaError_t launch_mv_any(const MvParams &p, cudaStream_t s) {
  MvSpec sp;
  const cudaError_t e = plan_mv_any<SWIGLU>(p, &sp);
  if (e != cudaSuccess) return e;
  const cudaError_t e2 = run_mv_spec(sp, p, s);
  return e2 != cudaSuccess ? e2 : cudaGetLastError();
}

cudaError_t launch_q4_0_mv(const float *x, const uint8_t *w, const uint32_t *ids, float *out,
                           int n_tokens, int top_k, int N, int K, int n_experts,
                           uint64_t expert_stride, cudaStream_t s) {
  MvParams p{};
  p.x = x; p.up = nullptr; p.w = w; p.ids = ids; p.order = nullptr; p.n_order = nullptr; p.out = out;
  p.n_rows = n_tokens * top_k; p.top_k = top_k; p.N = N; p.K = K; p.E = n_experts;
  p.expert_stride = expert_stride;
  return launch_mv_any<false>(p, s);
}

cudaError_t launch_q4_0_swiglu_mv(const float *gate, const float *up, const uint8_t *w, const uint32_t *ids,
                                  float *out, int n_rows, int N, int K, int n_experts, uint64_t expert_stride,
                                  cudaStream_t s) {
  MvParams p{};
  p.x = gate; p.up = up; p.w = w; p.ids = ids; p.order = nullptr; p.n_order = nullptr; p.out = out;
  p.n_rows = n_rows; p.top_k = 1; p.N = N; p.K = K; p.E = n_experts;
  p.expert_stride = expert_stride;
  return launch_mv_any<true>(p, s);
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
  cudaError_t e =
      launch_route_internal(ids, n_rows, n_experts, htpe, offs, hids, invalid, s, blk, n_blk, out, N);
  if (e != cudaSuccess) return e;
  // Tensor-core form: K a multiple of 256 (whole 144-byte TMA boxes of Q4_0 blocks) and
  // 16-byte aligned expert slabs.
  if (routed_mm_tc_ok(K, expert_stride, w))
    return launch_routed_mm_tc(kQ4_0, x, w, out, n_tokens, top_k, N, K, n_experts, expert_stride, workspace, s);
  MvParams p{};
  p.x = x; p.up = nullptr; p.w = w; p.ids = ids; p.order = hids; p.n_order = offs + n_experts; p.out = out;
  p.n_rows = n_rows; p.top_k = top_k; p.N = N; p.K = K; p.E = n_experts;
  p.expert_stride = expert_stride;
  const int rows_cta = kMvWarps * kMvRowsPerWarp;
  dim3 grid((unsigned)((N + rows_cta - 1) / rows_cta), (unsigned)(n_rows < 65535 ? n_rows : 65535), 1);
  routed_mv_kernel<false, kQ4_0><<<grid, kMvWarps * 32, 0, s>>>(p);
  return cudaGetLastError();
}

// Q8_0 mat-vec on the tensor cores: kernel instance for (warps, copy size).
cudaError_t launch_q8_0_mv_mma(const MvParams &p, int ks, int maxc, size_t smem, bool a16, cudaStream_t s) {
  const void *fn;
  if (a16)
    fn = ks == 4 ? reinterpret_cast<const void *>(q8_0_mv_mma_kernel<4, 16>)
       : ks == 2 ? reinterpret_cast<const void *>(q8_0_mv_mma_kernel<2, 16>)
                 : reinterpret_cast<const void *>(q8_0_mv_mma_kernel<1, 16>);
  else
    fn = ks == 4 ? reinterpret_cast<const void *>(q8_0_mv_mma_kernel<4, 8>)
       : ks == 2 ? reinterpret_cast<const void *>(q8_0_mv_mma_kernel<2, 8>)
                 : reinterpret_cast<const void *>(q8_0_mv_mma_kernel<1, 8>);
  cudaError_t e = ensure_dynamic_smem(fn, (int)smem);
  if (e != cudaSuccess) return e;
  MvParams pp = p;
  int mc = maxc;
  void *args[] = {&pp, &mc};
  const dim3 grid((unsigned)((p.N + 15) / 16), (unsigned)(p.n_rows < 65535 ? p.n_rows : 65535), 1);
  e = cudaLaunchKernel(fn, grid, dim3(ks * 32), args, smem, s);
  return e != cudaSuccess ? e : cudaGetLastError();
}

// GGML Q8_0 routed matmul (the type is among the routed kernels of quantized_matmul_id_ggml.rs):
// mat-vec visits routed rows in order, on the tensor cores when the rows allow it (K % 128
// == 0; 16-byte copies need K % 256 == 0 and 16-byte aligned slabs, 8-byte copies 8-byte
// aligned ones), else on the fp32 FMA kernel.  Mat-mat routes first
// (per-expert lists and token blocks in the workspace); with K % 256 == 0 and 16-byte aligned
// expert slabs it runs the tensor-core kernel of the Q4_0 form with the Q8_0 decode, else it
// visits the rows expert by expert on the FMA kernel, so that the CTAs running at one time
// share an expert's weights through L2.
cudaError_t launch_q8_0_matmul_id(const float *x, const uint8_t *w, const uint32_t *ids, float *out,
                                  int n_tokens, int top_k, int N, int K, int n_experts, uint64_t expert_stride,
                                  bool mm, void *workspace, cudaStream_t s) {
  const int n_rows = n_tokens * top_k;
  MvParams p{};
  p.x = x; p.up = nullptr; p.w = w; p.ids = ids; p.order = nullptr; p.n_order = nullptr; p.out = out;
  p.n_rows = n_rows; p.top_k = top_k; p.N = N; p.K = K; p.E = n_experts;
  p.expert_stride = expert_stride;
  if (!mm) {
    const uintptr_t wa = reinterpret_cast<uintptr_t>(w);
    const bool a16 = K % 256 == 0 && expert_stride % 16 == 0 && (wa & 15) == 0;
    const bool a8 = K % 128 == 0 && expert_stride % 8 == 0 && (wa & 7) == 0;
    if (a16 || a8) {
      const int C = (K / 128 + 1) / 2;
      const int ks = C >= 4 ? 4 : (C >= 2 ? 2 : 1);
      const int maxc = (C + ks - 1) / ks;
      const size_t smem = (size_t)ks * mv8_warp_bytes(maxc) + (size_t)ks * 16 * 4;
      if (smem <= 227 * 1024) return launch_q8_0_mv_mma(p, ks, maxc, smem, a16, s);
    }
  }
  if (mm) {
    const MoeWorkspace L = moe_workspace_layout(n_rows, K, n_experts);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    uint32_t *offs = reinterpret_cast<uint32_t *>(ws + L.offs);
    int32_t *hids = reinterpret_cast<int32_t *>(ws + L.hids);
    cudaError_t e = launch_route_internal(ids, n_rows, n_experts, reinterpret_cast<uint32_t *>(ws + L.htpe), offs,
                                          hids, reinterpret_cast<uint32_t *>(ws + L.invalid), s,
                                          reinterpret_cast<int4 *>(ws + L.blk),
                                          reinterpret_cast<uint32_t *>(ws + L.n_blk), out, N);
    if (e != cudaSuccess) return e;
    if (routed_mm_tc_ok(K, expert_stride, w))
      return launch_routed_mm_tc(kQ8_0, x, w, out, n_tokens, top_k, N, K, n_experts, expert_stride, workspace, s);
    p.order = hids;
    p.n_order = offs + n_experts;
  }
  const int rows_cta = kMvWarps * kMvRowsPerWarp;
  dim3 grid((unsigned)((N + rows_cta - 1) / rows_cta), (unsigned)(n_rows < 65535 ? n_rows : 65535), 1);
  routed_mv_kernel<false, kQ8_0><<<grid, kMvWarps * 32, 0, s>>>(p);
  return cudaGetLastError();
}

size_t q8_0_mm_workspace_bytes(int64_t n_tokens, int64_t top_k, int64_t K, int64_t n_experts) {
  return moe_workspace_layout(n_tokens * top_k, K, n_experts).total;
}

// Dispatch records for the routed mat-vec (quantized_matmul_id_ggml.rs pre-bakes its decode
// mat-vec dispatches the same way): planned for a shape, an expert stride and a weight
// alignment, replayed with new pointers.  *w_align reports the alignment every replayed
// weight pointer must keep (the kernel choice depends on it).
cudaError_t record_q4_0_mv(int n_rows, int top_k, int N, int K, int n_experts, uint64_t expert_stride,
                           bool swiglu, int *w_align, void **out) {
  MvParams p{};
  p.w = nullptr;   // planned as if 16-byte aligned; replay checks the pointer against w_align
  p.n_rows = n_rows; p.top_k = top_k; p.N = N; p.K = K; p.E = n_experts;
  p.expert_stride = expert_stride;
  MvSpec *sp = new (std::nothrow) MvSpec();
  if (sp == nullptr) return cudaErrorMemoryAllocation;
  const cudaError_t e = swiglu ? plan_mv_any<true>(p, sp) : plan_mv_any<false>(p, sp);
  if (e != cudaSuccess) {
    delete sp;
    return e;
  }
  *w_align = sp->w_align;
  *out = sp;
  return cudaSuccess;
}

cudaError_t replay_q4_0_mv(const void *record, const float *x, const float *up, const uint8_t *w,
                           const uint32_t *ids, float *out, cudaStream_t s) {
  const MvSpec *sp = static_cast<const MvSpec *>(record);
  MvParams p = sp->params;
  p.x = x; p.up = up; p.w = w; p.ids = ids; p.out = out; p.order = nullptr; p.n_order = nullptr;
  return run_mv_spec(*sp, p, s);
}

void free_q4_0_mv_record(void *record) { delete static_cast<MvSpec *>(record); }

}  // namespace q4mm
