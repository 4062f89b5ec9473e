// gemv.cu -- decode matmul for 1 <= M <= 16 tokens: INT4 group-32 affine (q4_gemv) and
// LUT4 blocked codebook (lut4_matmul, small M).
//
// What it computes: y[m][n] = sum_k x[m][k] * W[n][k] with W the dequantised weight of
// quant_fastkernel.rs (nibble*scale + bias, low nibble first) or of lut4.rs
// (book[code] * scale, high nibble for even flat index).  The pages leave the decode
// (M <= 16) case to a library GEMV; this kernel is designed for GB300 from scratch.
//
// Design (HBM-bound: every weight byte is read exactly once):
//   * A warp owns 16*RT weight rows.  Lane (g = lane/4, t = lane%4) loads, per 128-wide
//     K chunk and per row pair (g, g+8), one 16-byte vector = one 32-element group of that
//     row (quad lanes t = 0..3 read 64 contiguous bytes per row).  The codes are turned
//     into bf16 pairs in registers and fed to mma.sync m16n8k16 as the A operand (weights
//     are the M side, tokens the N side), so a 16-token step costs the tensor pipe, not
//     the FMA pipe.
//   * A dot product does not care in which order k is summed, as long as x and W agree;
//     the register decode yields pairs (code i, code i+4), so x is staged in shared memory
//     pre-permuted to the same order (LUT4 decodes natural pairs and uses natural order).
//   * Split-K across the CTAs of a thread-block cluster; the partial sums are combined
//     through distributed shared memory in rank order (deterministic, no workspace,
//     no atomics).
#include "q4mm_internal.cuh"

#include <algorithm>

namespace q4mm {
namespace {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kMaxCluster = 8;

struct GemvParams {
  const uint16_t *x;       // bf16 [M, K]
  const uint8_t *w;        // INT4: uint32 [N, K/8]; LUT4: uint8 [N, K/2]  (16 B per group)
  const void *scales;      // INT4: bf16 [N, K/32]; LUT4: f32 [N*K/block]
  const uint16_t *biases;  // INT4 only
  uint16_t *y;             // bf16 [M, N]
  int M, N, K;
  int chunks;              // chunks per row = ceil(K/32 / 4)
  int max_chunks_per_cta;  // smem sizing
  int lut_blocks_per_row;  // LUT4: K / block
  int lut_block_shift_div; // LUT4: block / 32 (groups per block)
  float book[16];
};

// Per (row, group) raw operand: 16 bytes of codes and the group's scale (and bias).
struct Raw {
  uint4 q;
  uint32_t s;   // INT4: bf16x2 (s, s); LUT4: f32 bits
  uint32_t b;   // INT4: bf16x2 (b, b)
};

template <bool LUT>
__device__ __forceinline__ void load_raw(Raw &r, const GemvParams &p, int row, int grp) {
  const int G = p.K / 32;
  if (row < p.N && grp < G) {
    r.q = ldg_stream_v4(p.w + (size_t)row * (size_t)(p.K / 2) + (size_t)grp * 16);
    if constexpr (LUT) {
      const float *sc = static_cast<const float *>(p.scales);
      r.s = __float_as_uint(__ldg(sc + (size_t)row * p.lut_blocks_per_row + grp / p.lut_block_shift_div));
      r.b = 0;
    } else {
      const size_t gi = (size_t)row * G + grp;
      const uint32_t s = ldg_u16(static_cast<const uint16_t *>(p.scales) + gi);
      const uint32_t b = ldg_u16(p.biases + gi);
      r.s = s | (s << 16);
      r.b = b | (b << 16);
    }
  } else {
    r.q = make_uint4(0, 0, 0, 0);
    r.s = 0;
    r.b = 0;
  }
}

// Decode word `word` of a group into 4 bf16 pairs in MMA step order:
// pairs 0,1 feed step 2q (A regs 0/2), pairs 2,3 feed step 2q+1.
template <bool LUT>
__device__ __forceinline__ void decode_word(uint32_t word, const Raw &r, const float *book,
                                            uint32_t (&out)[4]) {
  if constexpr (LUT) {
    // byte j: high nibble = even k (8q+2j), low nibble = odd k (8q+2j+1)
    const float s = __uint_as_float(r.s);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t hi = (word >> (8 * j + 4)) & 0xFu;
      const uint32_t lo = (word >> (8 * j)) & 0xFu;
      out[j] = pack_bf16x2(book[hi] * s, book[lo] * s);
    }
  } else {
    const Int4Pairs pr = int4_word_to_bf16_pairs(word, r.s, r.b);
#pragma unroll
    for (int j = 0; j < 4; ++j) out[j] = pr.p[j];
  }
}

// Shared-memory x layout: token row stride TS bytes; within a row, chunk c occupies 256 B
// as [piece j = 0..3][quad lane t = 0..3][16 B]; piece j of lane t's group holds the
// B-fragment words for MMA steps 2j and 2j+1.  TS = 256 * max_chunks + 64 keeps the two
// token rows a quarter-warp touches on disjoint banks.
__device__ __forceinline__ int x_row_stride(int max_chunks) { return max_chunks * 256 + 64; }

template <bool LUT>
__device__ void stage_x(const GemvParams &p, uint8_t *xs, int tokens, int c_begin, int nch) {
  const int TS = x_row_stride(p.max_chunks_per_cta);
  const int G = p.K / 32;
  const int items = tokens * nch * 4;
  for (int it = threadIdx.x; it < items; it += kThreads) {
    const int tok = it / (nch * 4);
    const int gl = it % (nch * 4);          // group within this CTA's slice
    const int c = gl / 4, t = gl % 4;
    const int grp = (c_begin + c) * 4 + t;  // group within the row
    uint32_t X[16];
    if (tok < p.M && grp < G) {
      const uint4 *src = reinterpret_cast<const uint4 *>(p.x + (size_t)tok * p.K + (size_t)grp * 32);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint4 v = __ldg(src + i);
        X[4 * i] = v.x; X[4 * i + 1] = v.y; X[4 * i + 2] = v.z; X[4 * i + 3] = v.w;
      }
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) X[i] = 0;
    }
    // X[i] = (x[2i], x[2i+1]).  Entry for step s = 2q + r is (b0, b1).
    uint32_t e[16];
#pragma unroll
    for (int q = 0; q < 4; ++q)
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int s = 2 * q + r;
        if constexpr (LUT) {
          // natural order: b0 = (x[4s], x[4s+1]), b1 = (x[4s+2], x[4s+3])
          e[2 * s] = X[2 * s];
          e[2 * s + 1] = X[2 * s + 1];
        } else {
          // (i, i+4) pairs: b0 = (x[8q+2r], x[8q+2r+4]), b1 = (x[8q+2r+1], x[8q+2r+5])
          const uint32_t a = X[4 * q + r], b = X[4 * q + r + 2];
          e[2 * s] = prmt(a, b, 0x5410);
          e[2 * s + 1] = prmt(a, b, 0x7632);
        }
      }
    uint8_t *dst = xs + (size_t)tok * TS + c * 256 + t * 16;
#pragma unroll
    for (int j = 0; j < 4; ++j)
      *reinterpret_cast<uint4 *>(dst + j * 64) = make_uint4(e[4 * j], e[4 * j + 1], e[4 * j + 2], e[4 * j + 3]);
  }
}

template <int MT, int RT, bool LUT>
__global__ void __launch_bounds__(kThreads) gemv_kernel(const __grid_constant__ GemvParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr int kRowsCta = kWarps * 16 * RT;
  constexpr int kTok = 8 * MT;
  const int TS = x_row_stride(p.max_chunks_per_cta);
  uint8_t *xs = smem;
  float *red = reinterpret_cast<float *>(smem + (size_t)kTok * TS);   // [kTok][kRowsCta]
  float *book = red + kTok * kRowsCta;                                  // [16]

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int g = lane / 4, t = lane % 4;
  const int S = gridDim.y;
  const int split = blockIdx.y;
  const int c_begin = (int)(((long long)split * p.chunks) / S);
  const int c_end = (int)(((long long)(split + 1) * p.chunks) / S);
  const int nch = c_end - c_begin;

  if constexpr (LUT) {
    if (threadIdx.x < 16) book[threadIdx.x] = p.book[threadIdx.x];
  }
  stage_x<LUT>(p, xs, kTok, c_begin, nch);
  __syncthreads();

  const int row0 = blockIdx.x * kRowsCta + warp * 16 * RT;
  float acc[RT][MT][4];
#pragma unroll
  for (int rt = 0; rt < RT; ++rt)
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[rt][mt][i] = 0.f;

  Raw cur[RT][2], nxt[RT][2];
  if (nch > 0) {
#pragma unroll
    for (int rt = 0; rt < RT; ++rt)
#pragma unroll
      for (int h = 0; h < 2; ++h)
        load_raw<LUT>(cur[rt][h], p, row0 + rt * 16 + g + 8 * h, c_begin * 4 + t);
  }
  const uint8_t *xlane = xs + (size_t)g * TS + t * 16;

  for (int c = 0; c < nch; ++c) {
    if (c + 1 < nch) {
#pragma unroll
      for (int rt = 0; rt < RT; ++rt)
#pragma unroll
        for (int h = 0; h < 2; ++h)
          load_raw<LUT>(nxt[rt][h], p, row0 + rt * 16 + g + 8 * h, (c_begin + c + 1) * 4 + t);
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint4 xb[MT];
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
        xb[mt] = *reinterpret_cast<const uint4 *>(xlane + (size_t)(8 * mt) * TS + c * 256 + q * 64);
#pragma unroll
      for (int rt = 0; rt < RT; ++rt) {
        const uint32_t w0 = q == 0 ? cur[rt][0].q.x : q == 1 ? cur[rt][0].q.y : q == 2 ? cur[rt][0].q.z : cur[rt][0].q.w;
        const uint32_t w1 = q == 0 ? cur[rt][1].q.x : q == 1 ? cur[rt][1].q.y : q == 2 ? cur[rt][1].q.z : cur[rt][1].q.w;
        uint32_t pg[4], pg8[4];
        decode_word<LUT>(w0, cur[rt][0], book, pg);
        decode_word<LUT>(w1, cur[rt][1], book, pg8);
        const uint32_t a0[4] = {pg[0], pg8[0], pg[1], pg8[1]};
        const uint32_t a1[4] = {pg[2], pg8[2], pg[3], pg8[3]};
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          mma_bf16_16816(acc[rt][mt], a0, xb[mt].x, xb[mt].y);
          mma_bf16_16816(acc[rt][mt], a1, xb[mt].z, xb[mt].w);
        }
      }
    }
#pragma unroll
    for (int rt = 0; rt < RT; ++rt)
#pragma unroll
      for (int h = 0; h < 2; ++h) cur[rt][h] = nxt[rt][h];
  }

  // Partial tile -> shared memory, token-major: red[tok][row].
#pragma unroll
  for (int rt = 0; rt < RT; ++rt)
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      const int rl = warp * 16 * RT + rt * 16 + g;
      const int tk = mt * 8 + 2 * t;
      red[(tk + 0) * kRowsCta + rl] = acc[rt][mt][0];
      red[(tk + 1) * kRowsCta + rl] = acc[rt][mt][1];
      red[(tk + 0) * kRowsCta + rl + 8] = acc[rt][mt][2];
      red[(tk + 1) * kRowsCta + rl + 8] = acc[rt][mt][3];
    }
  cluster_sync_all();

  // Each cluster rank finishes a strided share of the tile, summing ranks 0..S-1 in order.
  const uint32_t rank = cluster_ctarank();
  const int quads = kRowsCta / 4;
  const int items = p.M * quads;
  const uint32_t red_addr = smem_u32(red);
  for (int i = (int)rank * kThreads + threadIdx.x; i < items; i += S * kThreads) {
    const int tok = i / quads, qd = i % quads;
    const uint32_t off = (uint32_t)((tok * kRowsCta + qd * 4) * sizeof(float));
    float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int r = 0; r < S; ++r) {
      const float4 v = ld_shared_cluster_v4(map_shared_rank(red_addr + off, (uint32_t)r));
      sum.x += v.x; sum.y += v.y; sum.z += v.z; sum.w += v.w;
    }
    const int n0 = blockIdx.x * kRowsCta + qd * 4;
    uint16_t *dst = p.y + (size_t)tok * p.N + n0;
    const float vals[4] = {sum.x, sum.y, sum.z, sum.w};
    if (n0 + 3 < p.N && (p.N & 3) == 0) {
      const uint32_t lo = pack_bf16x2(vals[0], vals[1]), hi = pack_bf16x2(vals[2], vals[3]);
      *reinterpret_cast<uint2 *>(dst) = make_uint2(lo, hi);
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (n0 + j < p.N) {
          __nv_bfloat16 b = __float2bfloat16_rn(vals[j]);
          dst[j] = *reinterpret_cast<uint16_t *>(&b);
        }
    }
  }
  cluster_sync_all();   // keep every CTA's shared memory alive until all ranks have read it
}

struct Plan {
  int MT, RT, S, max_chunks;
  size_t smem;
};

size_t smem_bytes(int MT, int RT, int max_chunks) {
  const int tok = 8 * MT;
  return (size_t)tok * (max_chunks * 256 + 64) + (size_t)tok * kWarps * 16 * RT * 4 + 16 * 4;
}

Plan make_plan(int M, int N, int K) {
  Plan pl{};
  pl.MT = M <= 8 ? 1 : 2;
  const int chunks = (K / 32 + 3) / 4;
  int sms = 152;
  int dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && v > 0) sms = v;
  }
  const size_t smem_cap = 227 * 1024;
  // Prefer 32 rows per warp (x staged once per 128 rows); drop to 16 rows per warp when
  // that leaves too few CTAs to keep every SM streaming.
  Plan best{};
  double best_score = -1.0;
  for (int RT = 2; RT >= 1; --RT) {
    const int rows_cta = kWarps * 16 * RT;
    const int rb = (N + rows_cta - 1) / rows_cta;
    for (int S = 1; S <= std::min(kMaxCluster, chunks); ++S) {
      const int maxc = (chunks + S - 1) / S;
      const size_t sm = smem_bytes(pl.MT, RT, maxc);
      if (sm > smem_cap) continue;
      int per_sm = (int)(smem_cap / (sm + 1024));
      per_sm = std::max(1, std::min(per_sm, 16));
      const long long ctas = (long long)rb * S;
      const long long slots = (long long)sms * per_sm;
      const long long waves = (ctas + slots - 1) / slots;
      // fraction of SM-time doing useful streaming, with a mild preference for fewer
      // splits (each split re-stages x) and for 32-row warps
      const double fill = (double)ctas / (double)(waves * slots);
      const double busy = std::min(1.0, (double)ctas / (2.0 * sms));
      const double score = busy * (0.5 + 0.5 * fill) - 0.01 * S + (RT == 2 ? 0.02 : 0.0);
      if (score > best_score) {
        best_score = score;
        best = Plan{pl.MT, RT, S, maxc, sm};
      }
    }
  }
  return best;
}

template <int MT, int RT, bool LUT>
cudaError_t launch_typed(const GemvParams &p, const Plan &pl, cudaStream_t s) {
  auto kern = gemv_kernel<MT, RT, LUT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pl.smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  const int rows_cta = kWarps * 16 * RT;
  cfg.gridDim = dim3((unsigned)((p.N + rows_cta - 1) / rows_cta), (unsigned)pl.S, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = pl.smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = (unsigned)pl.S;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

template <bool LUT>
cudaError_t launch_any(GemvParams &p, cudaStream_t s) {
  const Plan pl = make_plan(p.M, p.N, p.K);
  p.chunks = (p.K / 32 + 3) / 4;
  p.max_chunks_per_cta = pl.max_chunks;
  if (pl.MT == 1) {
    return pl.RT == 2 ? launch_typed<1, 2, LUT>(p, pl, s) : launch_typed<1, 1, LUT>(p, pl, s);
  }
  return pl.RT == 2 ? launch_typed<2, 2, LUT>(p, pl, s) : launch_typed<2, 1, LUT>(p, pl, s);
}

}  // namespace

cudaError_t launch_q4_gemv(const uint16_t *x, const uint32_t *w, const uint16_t *scales,
                           const uint16_t *biases, uint16_t *y, int M, int N, int K,
                           cudaStream_t s) {
  GemvParams p{};
  p.x = x;
  p.w = reinterpret_cast<const uint8_t *>(w);
  p.scales = scales;
  p.biases = biases;
  p.y = y;
  p.M = M; p.N = N; p.K = K;
  return launch_any<false>(p, s);
}

cudaError_t launch_lut4_gemv(const uint16_t *x, const uint8_t *packed, const float *scales,
                             const float *book, uint16_t *y, int M, int N, int K, int block,
                             cudaStream_t s) {
  GemvParams p{};
  p.x = x;
  p.w = packed;
  p.scales = scales;
  p.biases = nullptr;
  p.y = y;
  p.M = M; p.N = N; p.K = K;
  p.lut_blocks_per_row = K / block;
  p.lut_block_shift_div = block / 32;
  for (int i = 0; i < 16; ++i) p.book[i] = book[i];
  return launch_any<true>(p, s);
}

}  // namespace q4mm
