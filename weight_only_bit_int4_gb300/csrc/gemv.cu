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
#include "tc_common.cuh"

#include <cudaTypedefs.h>

#include <new>

#include <algorithm>

namespace q4mm {

Q4MM_DEFINE_ERROR_READER(read_errors_gemv)

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

// Per-lane streaming cursor of one weight row: the lane reads group 4*chunk + t.
struct RowCursor {
  const uint8_t *w;       // codes of group t of chunk 0 of this row (nullptr: row >= N)
  const uint16_t *s, *b;  // INT4 scale / bias of group t (LUT4: s unused)
  const float *ls;        // LUT4 scale row
};

template <bool LUT>
__device__ __forceinline__ RowCursor make_cursor(const GemvParams &p, int row, int t) {
  RowCursor c{};
  if (row < p.N) {
    c.w = p.w + (size_t)row * (size_t)(p.K / 2) + (size_t)t * 16;
    if constexpr (LUT) {
      c.ls = static_cast<const float *>(p.scales) + (size_t)row * p.lut_blocks_per_row;
    } else {
      const size_t gi = (size_t)row * (p.K / 32) + t;
      c.s = static_cast<const uint16_t *>(p.scales) + gi;
      c.b = p.biases + gi;
    }
  }
  return c;
}

template <bool LUT>
__device__ __forceinline__ void load_raw(Raw &r, const GemvParams &p, const RowCursor &cur, int chunk, int t) {
  const int grp = chunk * 4 + t;
  if (cur.w != nullptr && grp < p.K / 32) {
    r.q = ldg_stream_v4(cur.w + (size_t)chunk * 64);
    if constexpr (LUT) {
      r.s = __float_as_uint(__ldg(cur.ls + grp / p.lut_block_shift_div));
      r.b = 0;
    } else {
      const uint32_t s = ldg_u16(cur.s + chunk * 4);
      const uint32_t b = ldg_u16(cur.b + chunk * 4);
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
__device__ void stage_x(const GemvParams &p, uint8_t *xs, int c_begin, int nch,
                        uint16_t *xsum = nullptr, float *xsum32 = nullptr) {
  const int TS = x_row_stride(p.max_chunks_per_cta);
  const int G = p.K / 32;
  const int items = p.M * nch * 4;   // tokens >= M are never read (their B fragments are zero)
  for (int it = threadIdx.x; it < items; it += kThreads) {
    const int tok = it / (nch * 4);
    const int gl = it % (nch * 4);          // group within this CTA's slice
    const int c = gl / 4, t = gl % 4;
    const int grp = (c_begin + c) * 4 + t;  // group within the row
    uint32_t X[16];
    if (grp < G) {
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
    if (xsum != nullptr || xsum32 != nullptr) {   // sum of the group's 32 x values (fp32, fixed order)
      float sum = 0.f;
#pragma unroll
      for (int i = 0; i < 16; ++i)
        sum += __uint_as_float(X[i] << 16) + __uint_as_float(X[i] & 0xFFFF0000u);
      if (xsum32 != nullptr) {
        xsum32[tok * (p.max_chunks_per_cta * 4) + gl] = sum;
      } else {
        __nv_bfloat16 hb = __float2bfloat16_rn(sum);
        xsum[tok * (p.max_chunks_per_cta * 4) + gl] = *reinterpret_cast<uint16_t *>(&hb);
      }
    }
  }
}

template <int kRowsCta>
__device__ __forceinline__ void cluster_sum_store(const GemvParams &p, float *red);

// Partial tile -> shared memory (token-major red[tok][row]) -> sum over the cluster's
// K splits in rank order through distributed shared memory -> bf16 y.
template <int MT, int RT>
__device__ __forceinline__ void cluster_reduce_store(const GemvParams &p, float *red,
                                                     const float (&acc)[RT][MT][4], int warp,
                                                     int g, int t) {
  constexpr int kRowsCta = kWarps * 16 * RT;
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
  cluster_sum_store<kRowsCta>(p, red);
}

// red[tok][row] of every CTA in the cluster (one per K split) -> sum in rank order -> bf16 y.
// Every thread of every CTA in the cluster calls this.
template <int kRowsCta>
__device__ __forceinline__ void cluster_sum_store(const GemvParams &p, float *red) {
  const int S = gridDim.y;
  cluster_sync_all();

  // Each cluster rank finishes a strided share of the tile, summing ranks 0..S-1 in order.
  const uint32_t rank = cluster_ctarank();
  const int quads = kRowsCta / 4;
  const int items = p.M * quads;
  const uint32_t red_addr = smem_u32(red);
  const int nthr = (int)blockDim.x;
  for (int i = (int)rank * nthr + (int)threadIdx.x; i < items; i += S * nthr) {
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
  const int row0 = blockIdx.x * kRowsCta + warp * 16 * RT;

  // Start streaming weights first: three chunks in flight per row pair before x is staged.
  RowCursor cur[RT][2];
#pragma unroll
  for (int rt = 0; rt < RT; ++rt)
#pragma unroll
    for (int h = 0; h < 2; ++h) cur[rt][h] = make_cursor<LUT>(p, row0 + rt * 16 + g + 8 * h, t);
  Raw b0[RT][2], b1[RT][2], b2[RT][2];
  auto load = [&](Raw (&b)[RT][2], int c) {
#pragma unroll
    for (int rt = 0; rt < RT; ++rt)
#pragma unroll
      for (int h = 0; h < 2; ++h) load_raw<LUT>(b[rt][h], p, cur[rt][h], c_begin + c, t);
  };
  if (nch > 0) load(b0, 0);
  if (nch > 1) load(b1, 1);
  if (nch > 2) load(b2, 2);
  // Weights are in flight; x may be the previous kernel's output, and y may still be read by it.
  griddep_launch_dependents();
  griddep_wait();

  if constexpr (LUT) {
    if (threadIdx.x < 16) book[threadIdx.x] = p.book[threadIdx.x];
  }
  stage_x<LUT>(p, xs, c_begin, nch);
  __syncthreads();

  float acc[RT][MT][4];
#pragma unroll
  for (int rt = 0; rt < RT; ++rt)
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[rt][mt][i] = 0.f;

  const uint8_t *xlane = xs + (size_t)g * TS + t * 16;
  bool tok_live[MT];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) tok_live[mt] = g + 8 * mt < p.M;

  auto compute = [&](const Raw (&b)[RT][2], int c) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint4 xb[MT];
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
        xb[mt] = tok_live[mt] ? *reinterpret_cast<const uint4 *>(xlane + (size_t)(8 * mt) * TS + c * 256 + q * 64)
                              : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int rt = 0; rt < RT; ++rt) {
        const uint32_t w0 = q == 0 ? b[rt][0].q.x : q == 1 ? b[rt][0].q.y : q == 2 ? b[rt][0].q.z : b[rt][0].q.w;
        const uint32_t w1 = q == 0 ? b[rt][1].q.x : q == 1 ? b[rt][1].q.y : q == 2 ? b[rt][1].q.z : b[rt][1].q.w;
        uint32_t pg[4], pg8[4];
        decode_word<LUT>(w0, b[rt][0], book, pg);
        decode_word<LUT>(w1, b[rt][1], book, pg8);
        const uint32_t a0[4] = {pg[0], pg8[0], pg[1], pg8[1]};
        const uint32_t a1[4] = {pg[2], pg8[2], pg[3], pg8[3]};
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          mma_bf16_16816(acc[rt][mt], a0, xb[mt].x, xb[mt].y);
          mma_bf16_16816(acc[rt][mt], a1, xb[mt].z, xb[mt].w);
        }
      }
    }
  };

  // Three statically rotated buffers: consume one, refill it three chunks ahead.
  for (int c = 0; c < nch; c += 3) {
    compute(b0, c);
    if (c + 3 < nch) load(b0, c + 3);
    if (c + 1 < nch) {
      compute(b1, c + 1);
      if (c + 4 < nch) load(b1, c + 4);
    }
    if (c + 2 < nch) {
      compute(b2, c + 2);
      if (c + 5 < nch) load(b2, c + 5);
    }
  }

  cluster_reduce_store<MT, RT>(p, red, acc, warp, g, t);
}

// ---------------------------------------------------------------------------------------
// Streaming variant for K % 128 == 0: each warp owns a private shared-memory ring of
// kDepth chunk stages filled with cp.async (16-byte code vectors and 8-byte scale/bias
// runs), so about kDepth chunks per warp are in flight without holding registers.
// Stage layout (per warp): [row half h][lane][16 B codes] then [h][quad g][scales 8 B |
// biases 8 B] (LUT4: [h][quad g][up to four f32 block scales]).
// ---------------------------------------------------------------------------------------
constexpr int kDepth = 8;
constexpr int kStageBytes = 2 * 512 + 2 * 128;
// Chunk stages per warp of gemv_async_kernel: 16 tokens (MT = 2) stage four times the x of
// one MMA column tile, and a shallower ring leaves room for more CTAs per SM.
__host__ __device__ constexpr int async_depth(int MT) { return MT == 2 ? 4 : kDepth; }
// Scale-block ring: chunk a reads block a/4 while chunk a + depth - 1 is being fetched, at
// most (depth + 2) / 4 blocks later.
constexpr int kSbSlots = (kDepth + 2) / 4 + 1;
constexpr int kSbRow = 80, kSbSlot = 16 * kSbRow;

__device__ __forceinline__ void cp_async(uint32_t dst, const void *src, int bytes, uint32_t src_bytes) {
  if (bytes == 16)
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
  else if (bytes == 8)
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
  else
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}

// INT4 weights enter the MMA as fma(128 + q, s, c_hi) in bf16, where c = b - 128 s (exact
// in fp32) splits as c_hi + c_lo, c_hi = bf16(c): the rounded value is that of q*s + b - c_lo,
// a number of the weight's own size, so one rounding per weight as in the plain dequant.
// The remainder sum_g c_lo[n][g] * sum_{k in g} x[m][k] is added by one extra MMA per chunk
// whose k-slot 2t carries (c_lo of lane t's group, that group's x sum).
// SB (INT4, K % 256 == 0): scales and biases arrive as 4-chunk blocks into a ring of
// [16 rows][s 32 B | b 32 B | pad], as in gemv_gc_kernel; the code stages then hold codes only.
template <int MT, int RT, bool LUT, bool SB>
__global__ void __launch_bounds__(kThreads) gemv_async_kernel(const __grid_constant__ GemvParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr int kRowsCta = kWarps * 16 * RT;
  constexpr int kTok = 8 * MT;
  static_assert(!(LUT && SB), "scale blocks are INT4 only");
  constexpr int kD = async_depth(MT);                  // chunk stages per warp
  constexpr int kSl = (kD + 2) / 4 + 1;                // scale-block slots (SB)
  constexpr int kStageC = SB ? 1024 : kStageBytes;   // per row tile
  constexpr int kStage = RT * kStageC;
  const int TS = x_row_stride(p.max_chunks_per_cta);
  uint8_t *ring = smem;
  uint8_t *sbr = smem + kWarps * kD * kStage;                       // SB: [warp][slot][RT]
  uint8_t *xs = sbr + (SB ? kWarps * kSl * kSbSlot * RT : 0);
  float *red = reinterpret_cast<float *>(xs + (size_t)p.M * TS);      // [kTok][kRowsCta]
  float *book = red + kTok * kRowsCta;                                 // [16]
  uint16_t *xsum = reinterpret_cast<uint16_t *>(book + 16);            // [M][4 * max_chunks]

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int g = lane / 4, t = lane % 4;
  const int S = gridDim.y;
  const int split = blockIdx.y;
  const int c_begin = (int)(((long long)split * p.chunks) / S);
  const int c_end = (int)(((long long)(split + 1) * p.chunks) / S);
  const int nch = c_end - c_begin;
  const int row0 = blockIdx.x * kRowsCta + warp * 16 * RT;
  const int G = p.K / 32;

  // Per-lane sources.  Rows past N copy nothing (src-size 0 zero-fills the slot).
  const uint8_t *wsrc[RT][2];
  bool live[RT][2];
#pragma unroll
  for (int rt = 0; rt < RT; ++rt)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int row = row0 + rt * 16 + g + 8 * h;
      live[rt][h] = row < p.N;
      wsrc[rt][h] = p.w + (live[rt][h] ? (size_t)row * (size_t)(p.K / 2) : 0) + (size_t)c_begin * 64 + t * 16;
    }
  // Scale run copied by this lane: INT4 lanes t = 0..3 copy (s, h0) (b, h0) (s, h1) (b, h1),
  // 4 consecutive bf16 each; LUT4 lanes t = 0, 1 copy the f32 block scales of h = t.
  const int sh = LUT ? t : (t >> 1);
  const int sk = LUT ? 0 : (t & 1);
  const bool scopy = LUT ? (t < 2) : true;
  const uint8_t *ssrc[RT];
  bool slive[RT];
  int sbytes = 8;
#pragma unroll
  for (int rt = 0; rt < RT; ++rt) {
    const int srow = row0 + rt * 16 + g + 8 * (sh & 1);
    slive[rt] = scopy && srow < p.N;
    if constexpr (LUT) {
      const int per_chunk = p.lut_block_shift_div <= 4 ? 4 / p.lut_block_shift_div : 1;
      sbytes = 4 * per_chunk;
      ssrc[rt] = reinterpret_cast<const uint8_t *>(static_cast<const float *>(p.scales) +
                                                   (slive[rt] ? (size_t)srow * p.lut_blocks_per_row : 0));
    } else {
      const uint16_t *base = sk ? p.biases : static_cast<const uint16_t *>(p.scales);
      ssrc[rt] = reinterpret_cast<const uint8_t *>(base + (slive[rt] ? (size_t)srow * G : 0) + (size_t)c_begin * 4);
    }
  }
  const uint32_t ring_warp = smem_u32(ring) + (uint32_t)(warp * kD * kStage);
  const uint32_t sdst_off = 1024u + (uint32_t)(sh * 128 + g * 16 + sk * 8);

  const uint32_t sb_warp = smem_u32(sbr) + (uint32_t)(warp * kSl * kSbSlot * RT);
  const int blk0 = c_begin / 4;
  auto issue = [&](int c) {
    const uint32_t slot = ring_warp + (uint32_t)((c % kD) * kStage);
    const int a = c_begin + c;
#pragma unroll
    for (int rt = 0; rt < RT; ++rt) {
      const uint32_t sl = slot + rt * kStageC;
#pragma unroll
      for (int h = 0; h < 2; ++h)
        cp_async(sl + h * 512 + lane * 16, wsrc[rt][h] + (size_t)c * 64, 16, live[rt][h] ? 16u : 0u);
      if constexpr (SB) {
        if (c == 0 || (a & 3) == 0) {   // block a/4: groups 16(a/4) .. +15, 16 rows, s and b
          const int b = a >> 2;
          const uint32_t sslot = sb_warp + (uint32_t)((((b - blk0) % kSl) * RT + rt) * kSbSlot);
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            const int idx = lane + 32 * i;
            const int r = idx >> 2, ten = (idx >> 1) & 1, half = idx & 1;
            const int row = row0 + rt * 16 + r;
            const int g0 = 16 * b + 8 * half;
            const bool ok = row < p.N && g0 < G;
            const uint16_t *base = ten ? p.biases : static_cast<const uint16_t *>(p.scales);
            cp_async(sslot + (uint32_t)(r * kSbRow + ten * 32 + half * 16), base + (ok ? (size_t)row * G + g0 : 0),
                     16, ok ? 16u : 0u);
          }
        }
      } else if (scopy) {
        const uint8_t *src;
        if constexpr (LUT) {
          src = ssrc[rt] + (size_t)(((c_begin + c) * 4) / p.lut_block_shift_div) * 4;
        } else {
          src = ssrc[rt] + (size_t)c * 8;
        }
        cp_async(sl + sdst_off, src, sbytes, slive[rt] ? (uint32_t)sbytes : 0u);
      }
    }
  };

  // Chunks go through the loop in pairs; kD - 2 chunks are in flight ahead of a pair.
#pragma unroll
  for (int i = 0; i < kD - 2; ++i) {
    if (i < nch) issue(i);
    cp_async_commit();
  }
  // Weights are in flight; x may be the previous kernel's output, and y may still be read by it.
  griddep_launch_dependents();
  griddep_wait();
  if constexpr (LUT) {
    if (threadIdx.x < 16) book[threadIdx.x] = p.book[threadIdx.x];
  }
  stage_x<LUT>(p, xs, c_begin, nch, LUT ? nullptr : xsum);
  __syncthreads();

  float acc[RT][MT][4];
#pragma unroll
  for (int rt = 0; rt < RT; ++rt)
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[rt][mt][i] = 0.f;
  const uint8_t *xlane = xs + (size_t)g * TS + t * 16;
  bool tok_live[MT];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) tok_live[mt] = g + 8 * mt < p.M;
  const uint8_t *ring_ptr = ring + warp * kD * kStage;
  const int xsum_stride = p.max_chunks_per_cta * 4;

  auto process = [&](int c) {
    const uint8_t *slot = ring_ptr + (c % kD) * kStage;
    uint4 xb[4][MT];
#pragma unroll
    for (int q = 0; q < 4; ++q)
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
        xb[q][mt] = tok_live[mt] ? *reinterpret_cast<const uint4 *>(xlane + (size_t)(8 * mt) * TS + c * 256 + q * 64)
                                 : make_uint4(0, 0, 0, 0);
    uint32_t xs_b[MT];
    if constexpr (!LUT) {
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
        xs_b[mt] = tok_live[mt] ? (uint32_t)xsum[(g + 8 * mt) * xsum_stride + c * 4 + t] : 0u;
    }
#pragma unroll
    for (int rt = 0; rt < RT; ++rt) {
      const uint8_t *sl = slot + rt * kStageC;
      uint4 qv[2];
      uint32_t s2[2], c2[2];
      float clo[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        qv[h] = *reinterpret_cast<const uint4 *>(sl + h * 512 + lane * 16);
        const uint8_t *sc = sl + 1024 + h * 128 + g * 16;
        if constexpr (LUT) {
          const int idx = p.lut_block_shift_div <= 4 ? t / p.lut_block_shift_div : 0;
          s2[h] = *reinterpret_cast<const uint32_t *>(sc + 4 * idx);
          c2[h] = 0;
          clo[h] = 0.f;
        } else {
          uint32_t sv, bv;
          if constexpr (SB) {
            const int a = c_begin + c;
            const uint8_t *sb = sbr + (size_t)((warp * kSl + ((a >> 2) - blk0) % kSl) * RT + rt) * kSbSlot +
                                (g + 8 * h) * kSbRow + (a & 3) * 8 + 2 * t;
            sv = *reinterpret_cast<const uint16_t *>(sb);
            bv = *reinterpret_cast<const uint16_t *>(sb + 32);
          } else {
            sv = *reinterpret_cast<const uint16_t *>(sc + 2 * t);
            bv = *reinterpret_cast<const uint16_t *>(sc + 8 + 2 * t);
          }
          const float cf = __fmaf_rn(-128.f, __uint_as_float(sv << 16), __uint_as_float(bv << 16));
          const uint32_t chi = pack_bf16x2(cf, cf);
          clo[h] = cf - __uint_as_float(chi << 16);
          s2[h] = sv | (sv << 16);
          c2[h] = chi;
        }
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint32_t w0 = q == 0 ? qv[0].x : q == 1 ? qv[0].y : q == 2 ? qv[0].z : qv[0].w;
        const uint32_t w1 = q == 0 ? qv[1].x : q == 1 ? qv[1].y : q == 2 ? qv[1].z : qv[1].w;
        uint32_t pg[4], pg8[4];
        if constexpr (LUT) {
          Raw r0{qv[0], s2[0], 0}, r1{qv[1], s2[1], 0};
          decode_word<true>(w0, r0, book, pg);
          decode_word<true>(w1, r1, book, pg8);
        } else {
          constexpr uint32_t kMask = 0x000F000Fu, kMagic = 0x43004300u;
          const uint32_t ws0[4] = {w0, w0 >> 4, w0 >> 8, w0 >> 12};
          const uint32_t ws1[4] = {w1, w1 >> 4, w1 >> 8, w1 >> 12};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            pg[j] = bf16x2_fma(and_or(ws0[j], kMask, kMagic), s2[0], c2[0]);
            pg8[j] = bf16x2_fma(and_or(ws1[j], kMask, kMagic), s2[1], c2[1]);
          }
        }
        const uint32_t a0[4] = {pg[0], pg8[0], pg[1], pg8[1]};
        const uint32_t a1[4] = {pg[2], pg8[2], pg[3], pg8[3]};
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          mma_bf16_16816(acc[rt][mt], a0, xb[q][mt].x, xb[q][mt].y);
          mma_bf16_16816(acc[rt][mt], a1, xb[q][mt].z, xb[q][mt].w);
        }
      }
      if constexpr (!LUT) {
        // k-slot 2t: row g -> c_lo(g), row g+8 -> c_lo(g+8); token column -> x sum of the group
        const uint32_t ac[4] = {pack_bf16x2(clo[0], 0.f), pack_bf16x2(clo[1], 0.f), 0u, 0u};
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) mma_bf16_16816(acc[rt][mt], ac, xs_b[mt], 0u);
      }
    }
  };
  int c = 0;
  for (; c + 1 < nch; c += 2) {
    if (c + kD - 2 < nch) issue(c + kD - 2);
    cp_async_commit();
    if (c + kD - 1 < nch) issue(c + kD - 1);
    cp_async_commit();
    cp_async_wait<kD - 2>();
    __syncwarp();
    process(c);
    process(c + 1);
    __syncwarp();
  }
  if (c < nch) {   // odd chunk count: the last chunk alone
    cp_async_wait<0>();
    __syncwarp();
    process(c);
  }
  cp_async_wait<0>();
  cluster_reduce_store<MT, RT>(p, red, acc, warp, g, t);
}

// ---------------------------------------------------------------------------------------
// INT4, 1 <= M <= 4: the scale and bias are applied after the tensor core, per group.
//
// With at most 4 tokens most B columns of an m16n8k16 step would be zero, so the columns
// are spent on quantisation groups instead: in every step the quad lane t supplies the
// k-slots of group t (its own 16-byte code vector) for every row, and B column n = 8u + j
// carries token 2u + j/4 on the k-slots of group j%4 and zeros elsewhere.  Column n of the
// product is then sum_{k in group} (128 + q) x for one (group, token) pair, with the codes
// entering as exact bf16 integers 128 + q (one LOP3 each, no dequantising multiply).
// After the chunk's 8 steps the lane holds columns 2t, 2t+1 of each tile, i.e. groups
// 2(t&1) and 2(t&1)+1 of token 2u + t/2 for rows g and g+8, and adds, in fp32,
//   s * D + (b - 128 s) * X,   X = sum of the group's x,
// which is sum_k (q s + b) x_k for the group: the same dot product, reassociated.
// ---------------------------------------------------------------------------------------
// SB (K % 256 == 0, 16-byte aligned scales and biases): the scales and biases of 4 chunks
// arrive together, two 16-byte copies per lane into a kSbSlots ring of [16 rows][s 32 B |
// b 32 B | 16 B pad]; otherwise each chunk carries its own 8-byte runs as in the stage
// layout above.
template <int MT2, int RT, bool SB>
__global__ void __launch_bounds__(kThreads) gemv_gc_kernel(const __grid_constant__ GemvParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr int kRowsCta = kWarps * 16 * RT;
  constexpr int kStageC = SB ? 1024 : kStageBytes;   // per row tile
  constexpr int kStage = RT * kStageC;

  const int TS = x_row_stride(p.max_chunks_per_cta);
  const int xsum_stride = p.max_chunks_per_cta * 4;
  uint8_t *ring = smem;
  uint8_t *xs = smem + kWarps * kDepth * kStage;
  uint8_t *sbr = ring + kWarps * kDepth * kStage;                     // SB: [warp][slot][RT]
  if constexpr (SB) xs = sbr + kWarps * kSbSlots * kSbSlot * RT;
  float *red = reinterpret_cast<float *>(xs + (size_t)p.M * TS);      // [M][kRowsCta]
  float *xsum = red + p.M * kRowsCta;                                  // [M][4 * max_chunks]

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int g = lane / 4, t = lane % 4;
  const int S = gridDim.y;
  const int split = blockIdx.y;
  const int c_begin = (int)(((long long)split * p.chunks) / S);
  const int c_end = (int)(((long long)(split + 1) * p.chunks) / S);
  const int nch = c_end - c_begin;
  const int row0 = blockIdx.x * kRowsCta + warp * 16 * RT;
  const int G = p.K / 32;

  const uint8_t *wsrc[RT][2];
  bool live[RT][2];
#pragma unroll
  for (int rt = 0; rt < RT; ++rt)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int row = row0 + rt * 16 + g + 8 * h;
      live[rt][h] = row < p.N;
      wsrc[rt][h] = p.w + (live[rt][h] ? (size_t)row * (size_t)(p.K / 2) : 0) + (size_t)c_begin * 64 + t * 16;
    }
  // Lane (g, t) copies 4 consecutive bf16 (scales if t is even, biases if odd) of row
  // g + 8 * (t >> 1) per chunk.
  const int sh = t >> 1, sk = t & 1;
  const uint8_t *ssrc[RT];
  bool slive[RT];
#pragma unroll
  for (int rt = 0; rt < RT; ++rt) {
    const int srow = row0 + rt * 16 + g + 8 * sh;
    slive[rt] = srow < p.N;
    const uint16_t *base = sk ? p.biases : static_cast<const uint16_t *>(p.scales);
    ssrc[rt] = reinterpret_cast<const uint8_t *>(base + (slive[rt] ? (size_t)srow * G : 0) + (size_t)c_begin * 4);
  }
  const uint32_t ring_warp = smem_u32(ring) + (uint32_t)(warp * kDepth * kStage);
  const uint32_t sdst_off = 1024u + (uint32_t)(sh * 128 + g * 16 + sk * 8);

  const uint32_t sb_warp = smem_u32(sbr) + (uint32_t)(warp * kSbSlots * kSbSlot * RT);
  const int blk0 = c_begin / 4;
  auto issue = [&](int c) {
    const uint32_t slot = ring_warp + (uint32_t)((c % kDepth) * kStage);
    const int a = c_begin + c;
#pragma unroll
    for (int rt = 0; rt < RT; ++rt) {
      const uint32_t sl = slot + rt * kStageC;
#pragma unroll
      for (int h = 0; h < 2; ++h)
        cp_async(sl + h * 512 + lane * 16, wsrc[rt][h] + (size_t)c * 64, 16, live[rt][h] ? 16u : 0u);
      if constexpr (!SB) {
        cp_async(sl + sdst_off, ssrc[rt] + (size_t)c * 8, 8, slive[rt] ? 8u : 0u);
      } else if (c == 0 || (a & 3) == 0) {
        // block a/4: groups 16(a/4) .. +15 of 16 rows, scales and biases, in two halves
        const int b = a >> 2;
        const uint32_t sslot = sb_warp + (uint32_t)((((b - blk0) % kSbSlots) * RT + rt) * kSbSlot);
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int idx = lane + 32 * i;
          const int r = idx >> 2, ten = (idx >> 1) & 1, half = idx & 1;
          const int row = row0 + rt * 16 + r;
          const int g0 = 16 * b + 8 * half;
          const bool ok = row < p.N && g0 < G;
          const uint16_t *base = ten ? p.biases : static_cast<const uint16_t *>(p.scales);
          const uint16_t *src = base + (ok ? (size_t)row * G + g0 : 0);
          cp_async(sslot + (uint32_t)(r * kSbRow + ten * 32 + half * 16), src, 16, ok ? 16u : 0u);
        }
      }
    }
  };

  // Chunks go through the loop in pairs; kDepth - 2 chunks are in flight ahead of a pair.
#pragma unroll
  for (int i = 0; i < kDepth - 2; ++i) {
    if (i < nch) issue(i);
    cp_async_commit();
  }
  // Weights are in flight; x may be the previous kernel's output, and y may still be read by it.
  griddep_launch_dependents();
  griddep_wait();
  stage_x<false>(p, xs, c_begin, nch, nullptr, xsum);
  __syncthreads();

  // B operand: tile u, column g -> token 2u + g/4 on group g%4, which is nonzero only in
  // the k-slots of quad lane t == g%4.
  bool bl[MT2];
  const uint8_t *xl[MT2];
#pragma unroll
  for (int u = 0; u < MT2; ++u) {
    const int tok = 2 * u + g / 4;
    bl[u] = (g & 3) == t && tok < p.M;
    xl[u] = xs + (size_t)(bl[u] ? tok : 0) * TS + t * 16;
  }
  // Accumulated columns: tile u -> token 2u + t/2, groups 2(t&1), 2(t&1)+1.
  bool al[MT2];
  const float *xsl[MT2];
#pragma unroll
  for (int u = 0; u < MT2; ++u) {
    const int tok = 2 * u + t / 2;
    al[u] = tok < p.M;
    xsl[u] = xsum + (al[u] ? tok : 0) * xsum_stride + 2 * (t & 1);
  }
  float acc[RT][MT2][2];
#pragma unroll
  for (int rt = 0; rt < RT; ++rt)
#pragma unroll
    for (int u = 0; u < MT2; ++u) acc[rt][u][0] = acc[rt][u][1] = 0.f;
  const uint8_t *ring_ptr = ring + warp * kDepth * kStage;

  auto process = [&](int c) {
    const uint8_t *slot = ring_ptr + (c % kDepth) * kStage;
    uint4 xb[4][MT2];
    float2 X[MT2];
#pragma unroll
    for (int u = 0; u < MT2; ++u) {
#pragma unroll
      for (int q = 0; q < 4; ++q)
        xb[q][u] = bl[u] ? *reinterpret_cast<const uint4 *>(xl[u] + c * 256 + q * 64) : make_uint4(0, 0, 0, 0);
      X[u] = al[u] ? *reinterpret_cast<const float2 *>(xsl[u] + c * 4) : make_float2(0.f, 0.f);
    }
#pragma unroll
    for (int rt = 0; rt < RT; ++rt) {
      const uint8_t *sl = slot + rt * kStageC;
      const uint4 q0 = *reinterpret_cast<const uint4 *>(sl + lane * 16);
      const uint4 q1 = *reinterpret_cast<const uint4 *>(sl + 512 + lane * 16);
      uint32_t su[2], bu[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        if constexpr (SB) {
          const int a = c_begin + c;
          const uint8_t *sc = sbr + (size_t)((warp * kSbSlots + ((a >> 2) - blk0) % kSbSlots) * RT + rt) * kSbSlot +
                              (g + 8 * h) * kSbRow + (a & 3) * 8 + 4 * (t & 1);
          su[h] = *reinterpret_cast<const uint32_t *>(sc);
          bu[h] = *reinterpret_cast<const uint32_t *>(sc + 32);
        } else {
          const uint8_t *sc = sl + 1024 + h * 128 + g * 16 + 4 * (t & 1);
          su[h] = *reinterpret_cast<const uint32_t *>(sc);
          bu[h] = *reinterpret_cast<const uint32_t *>(sc + 8);
        }
      }
      float D[MT2][4];
#pragma unroll
      for (int u = 0; u < MT2; ++u) D[u][0] = D[u][1] = D[u][2] = D[u][3] = 0.f;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint32_t w0 = q == 0 ? q0.x : q == 1 ? q0.y : q == 2 ? q0.z : q0.w;
        const uint32_t w1 = q == 0 ? q1.x : q == 1 ? q1.y : q == 2 ? q1.z : q1.w;
        constexpr uint32_t kMask = 0x000F000Fu, kMagic = 0x43004300u;   // bf16 128 + q
        const uint32_t a0[4] = {and_or(w0, kMask, kMagic), and_or(w1, kMask, kMagic),
                                and_or(w0 >> 4, kMask, kMagic), and_or(w1 >> 4, kMask, kMagic)};
        const uint32_t a1[4] = {and_or(w0 >> 8, kMask, kMagic), and_or(w1 >> 8, kMask, kMagic),
                                and_or(w0 >> 12, kMask, kMagic), and_or(w1 >> 12, kMask, kMagic)};
#pragma unroll
        for (int u = 0; u < MT2; ++u) {
          mma_bf16_16816(D[u], a0, xb[q][u].x, xb[q][u].y);
          mma_bf16_16816(D[u], a1, xb[q][u].z, xb[q][u].w);
        }
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const float s0 = __uint_as_float(su[h] << 16), s1 = __uint_as_float(su[h] & 0xFFFF0000u);
        const float b0 = __uint_as_float(bu[h] << 16), b1 = __uint_as_float(bu[h] & 0xFFFF0000u);
        const float c0 = __fmaf_rn(-128.f, s0, b0), c1 = __fmaf_rn(-128.f, s1, b1);
#pragma unroll
        for (int u = 0; u < MT2; ++u) {
          float a = acc[rt][u][h];
          a = __fmaf_rn(s0, D[u][2 * h], a);
          a = __fmaf_rn(s1, D[u][2 * h + 1], a);
          a = __fmaf_rn(c0, X[u].x, a);
          a = __fmaf_rn(c1, X[u].y, a);
          acc[rt][u][h] = a;
        }
      }
    }
  };
  int c = 0;
  for (; c + 1 < nch; c += 2) {
    if (c + kDepth - 2 < nch) issue(c + kDepth - 2);
    cp_async_commit();
    if (c + kDepth - 1 < nch) issue(c + kDepth - 1);
    cp_async_commit();
    cp_async_wait<kDepth - 2>();
    __syncwarp();
    process(c);
    process(c + 1);
    __syncwarp();
  }
  if (c < nch) {   // odd chunk count: the last chunk alone
    cp_async_wait<0>();
    __syncwarp();
    process(c);
  }
  cp_async_wait<0>();

  // Lanes t and t^1 hold the two group pairs of the same token: add them, store red[tok][row].
#pragma unroll
  for (int rt = 0; rt < RT; ++rt)
#pragma unroll
    for (int u = 0; u < MT2; ++u)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const float v = acc[rt][u][h] + __shfl_xor_sync(0xFFFFFFFFu, acc[rt][u][h], 1);
        if ((t & 1) == 0 && al[u])
          red[(2 * u + t / 2) * kRowsCta + warp * 16 * RT + rt * 16 + g + 8 * h] = v;
      }
  cluster_sum_store<kRowsCta>(p, red);
}

// ---------------------------------------------------------------------------------------
// INT4, 1 <= M <= 4, K % 256 == 0: the group-column product of gemv_gc_kernel with the K
// split inside the CTA.  A CTA owns one 16-row group and its KS warps take consecutive K
// slices; each warp streams its slice through a private cp.async ring (DEPTH code stages
// and a ring of 4-chunk scale blocks) and stages only the x it needs, so nothing couples
// the warps until their partial tiles meet in shared memory, where they are summed in warp
// order.  A further split across the CTAs of a cluster (S > 1) is combined through
// distributed shared memory as above.
// ---------------------------------------------------------------------------------------
__host__ __device__ constexpr int ks_sb_slots(int depth) { return (depth + 2) / 4 + 1; }
__host__ __device__ inline int ks_x_stride(int maxc) { return maxc * 256 + 64; }
// Per-warp shared memory: code ring, scale-block ring, x [M][ks_x_stride], x sums [M][4 maxc].
__host__ __device__ inline size_t ks_warp_bytes(int depth, int M, int maxc) {
  return (size_t)depth * 1024 + (size_t)ks_sb_slots(depth) * kSbSlot + (size_t)M * ks_x_stride(maxc) +
         (size_t)M * maxc * 16;
}

template <int MT2, int KS, int DEPTH>
__global__ void __launch_bounds__(KS * 32) gemv_ks_kernel(const __grid_constant__ GemvParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr int kSlots = ks_sb_slots(DEPTH);
  const int maxc = p.max_chunks_per_cta;
  const int XS = ks_x_stride(maxc);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int g = lane / 4, t = lane % 4;
  uint8_t *wbase = smem + (size_t)warp * ks_warp_bytes(DEPTH, p.M, maxc);
  uint8_t *ring = wbase;
  uint8_t *sbr = wbase + DEPTH * 1024;
  uint8_t *xs = sbr + kSlots * kSbSlot;
  float *xsum = reinterpret_cast<float *>(xs + (size_t)p.M * XS);                  // [M][4 maxc]
  float *red = reinterpret_cast<float *>(smem + (size_t)KS * ks_warp_bytes(DEPTH, p.M, maxc));  // [KS][M][16]

  const int splits = (int)gridDim.y * KS;
  const int sp = (int)blockIdx.y * KS + warp;
  const int c_begin = (int)(((long long)sp * p.chunks) / splits);
  const int c_end = (int)(((long long)(sp + 1) * p.chunks) / splits);
  const int nch = c_end - c_begin;
  const int row0 = blockIdx.x * 16;
  const int G = p.K / 32;

  const uint8_t *wsrc[2];
  bool live[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int row = row0 + g + 8 * h;
    live[h] = row < p.N;
    wsrc[h] = p.w + (live[h] ? (size_t)row * (size_t)(p.K / 2) : 0) + (size_t)c_begin * 64 + t * 16;
  }
  const uint32_t ring_s = smem_u32(ring), sb_s = smem_u32(sbr);
  const int blk0 = c_begin / 4;
  auto issue = [&](int c) {
    const uint32_t slot = ring_s + (uint32_t)((c % DEPTH) * 1024);
#pragma unroll
    for (int h = 0; h < 2; ++h)
      cp_async(slot + h * 512 + lane * 16, wsrc[h] + (size_t)c * 64, 16, live[h] ? 16u : 0u);
    const int a = c_begin + c;
    if (c == 0 || (a & 3) == 0) {   // scales and biases of chunks 4(a/4) .. +3, 16 rows
      const int b = a >> 2;
      const uint32_t sslot = sb_s + (uint32_t)(((b - blk0) % kSlots) * kSbSlot);
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int idx = lane + 32 * i;
        const int r = idx >> 2, ten = (idx >> 1) & 1, half = idx & 1;
        const int row = row0 + r;
        const int g0 = 16 * b + 8 * half;
        const bool ok = row < p.N && g0 < G;
        const uint16_t *base = ten ? p.biases : static_cast<const uint16_t *>(p.scales);
        cp_async(sslot + (uint32_t)(r * kSbRow + ten * 32 + half * 16), base + (ok ? (size_t)row * G + g0 : 0), 16,
                 ok ? 16u : 0u);
      }
    }
  };

  // Chunks go through the loop in pairs; DEPTH - 2 chunks are in flight ahead of a pair.
#pragma unroll
  for (int i = 0; i < DEPTH - 2; ++i) {
    if (i < nch) issue(i);
    cp_async_commit();
  }
  // Weights are in flight; x may be the previous kernel's output, and y may still be read by it.
  griddep_launch_dependents();
  griddep_wait();

  // This warp's x slice, permuted to the decode's (i, i+4) pair order, and its group sums.
  for (int it = lane; it < p.M * nch * 4; it += 32) {
    const int tok = it / (nch * 4);
    const int gl = it % (nch * 4);
    const int c = gl / 4, tq = gl % 4;
    const uint4 *src = reinterpret_cast<const uint4 *>(p.x + (size_t)tok * p.K + (size_t)((c_begin + c) * 4 + tq) * 32);
    uint32_t X[16];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 v = __ldg(src + i);
      X[4 * i] = v.x; X[4 * i + 1] = v.y; X[4 * i + 2] = v.z; X[4 * i + 3] = v.w;
    }
    uint8_t *dst = xs + (size_t)tok * XS + c * 256 + tq * 16;
    float sum = 0.f;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint32_t a0 = X[4 * q], b0 = X[4 * q + 2], a1 = X[4 * q + 1], b1 = X[4 * q + 3];
      *reinterpret_cast<uint4 *>(dst + q * 64) =
          make_uint4(prmt(a0, b0, 0x5410), prmt(a0, b0, 0x7632), prmt(a1, b1, 0x5410), prmt(a1, b1, 0x7632));
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) sum += __uint_as_float(X[i] << 16) + __uint_as_float(X[i] & 0xFFFF0000u);
    xsum[tok * maxc * 4 + gl] = sum;
  }
  __syncwarp();

  bool bl[MT2], al[MT2];
  const uint8_t *xl[MT2];
  const float *xsl[MT2];
#pragma unroll
  for (int u = 0; u < MT2; ++u) {
    const int tb = 2 * u + g / 4;
    bl[u] = (g & 3) == t && tb < p.M;
    xl[u] = xs + (size_t)(bl[u] ? tb : 0) * XS + t * 16;
    const int ta = 2 * u + t / 2;
    al[u] = ta < p.M;
    xsl[u] = xsum + (al[u] ? ta : 0) * maxc * 4 + 2 * (t & 1);
  }
  float acc[MT2][2];
#pragma unroll
  for (int u = 0; u < MT2; ++u) acc[u][0] = acc[u][1] = 0.f;

  // Scale-block read cursor: slot of chunk c's block and c's position in it, advanced per
  // processed chunk (chunks are processed in order).
  int rd_slot = 0, rd_pos = c_begin & 3;
  // B fragments and group sums of the two chunks of a pair.  With one token tile, lanes
  // that carry no x keep them at zero for the whole loop and only the carrying lanes load
  // (no per-chunk selects); with two tiles that would cost too many registers, so the
  // fragments are rebuilt per chunk.
  uint4 xbuf[2][4][MT2];
  float2 Xbuf[2][MT2];
#pragma unroll
  for (int pi = 0; pi < 2; ++pi)
#pragma unroll
    for (int u = 0; u < MT2; ++u) {
#pragma unroll
      for (int q = 0; q < 4; ++q) xbuf[pi][q][u] = make_uint4(0, 0, 0, 0);
      Xbuf[pi][u] = make_float2(0.f, 0.f);
    }
  auto process = [&](int c, int pi) {
    const uint8_t *sl = ring + (c % DEPTH) * 1024;
    uint4 (&xb)[4][MT2] = xbuf[pi];
    float2 (&X)[MT2] = Xbuf[pi];
#pragma unroll
    for (int u = 0; u < MT2; ++u) {
      if constexpr (MT2 == 1) {
        if (bl[u]) {
#pragma unroll
          for (int q = 0; q < 4; ++q) xb[q][u] = *reinterpret_cast<const uint4 *>(xl[u] + c * 256 + q * 64);
        }
        if (al[u]) X[u] = *reinterpret_cast<const float2 *>(xsl[u] + c * 4);
      } else {
#pragma unroll
        for (int q = 0; q < 4; ++q)
          xb[q][u] = bl[u] ? *reinterpret_cast<const uint4 *>(xl[u] + c * 256 + q * 64) : make_uint4(0, 0, 0, 0);
        X[u] = al[u] ? *reinterpret_cast<const float2 *>(xsl[u] + c * 4) : make_float2(0.f, 0.f);
      }
    }
    const uint4 q0 = *reinterpret_cast<const uint4 *>(sl + lane * 16);
    const uint4 q1 = *reinterpret_cast<const uint4 *>(sl + 512 + lane * 16);
    const uint8_t *sc = sbr + rd_slot * kSbSlot + g * kSbRow + rd_pos * 8 + 4 * (t & 1);
    if (++rd_pos == 4) {
      rd_pos = 0;
      rd_slot = rd_slot + 1 == kSlots ? 0 : rd_slot + 1;
    }
    uint32_t su[2], bu[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      su[h] = *reinterpret_cast<const uint32_t *>(sc + h * 8 * kSbRow);
      bu[h] = *reinterpret_cast<const uint32_t *>(sc + h * 8 * kSbRow + 32);
    }
    float D[MT2][4];
#pragma unroll
    for (int u = 0; u < MT2; ++u) D[u][0] = D[u][1] = D[u][2] = D[u][3] = 0.f;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint32_t w0 = q == 0 ? q0.x : q == 1 ? q0.y : q == 2 ? q0.z : q0.w;
      const uint32_t w1 = q == 0 ? q1.x : q == 1 ? q1.y : q == 2 ? q1.z : q1.w;
      constexpr uint32_t kMask = 0x000F000Fu, kMagic = 0x43004300u;   // bf16 128 + q
      const uint32_t a0[4] = {and_or(w0, kMask, kMagic), and_or(w1, kMask, kMagic),
                              and_or(w0 >> 4, kMask, kMagic), and_or(w1 >> 4, kMask, kMagic)};
      const uint32_t a1[4] = {and_or(w0 >> 8, kMask, kMagic), and_or(w1 >> 8, kMask, kMagic),
                              and_or(w0 >> 12, kMask, kMagic), and_or(w1 >> 12, kMask, kMagic)};
#pragma unroll
      for (int u = 0; u < MT2; ++u) {
        mma_bf16_16816(D[u], a0, xb[q][u].x, xb[q][u].y);
        mma_bf16_16816(D[u], a1, xb[q][u].z, xb[q][u].w);
      }
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const float s0 = __uint_as_float(su[h] << 16), s1 = __uint_as_float(su[h] & 0xFFFF0000u);
      const float b0 = __uint_as_float(bu[h] << 16), b1 = __uint_as_float(bu[h] & 0xFFFF0000u);
      const float c0 = __fmaf_rn(-128.f, s0, b0), c1 = __fmaf_rn(-128.f, s1, b1);
#pragma unroll
      for (int u = 0; u < MT2; ++u) {
        float v = acc[u][h];
        v = __fmaf_rn(s0, D[u][2 * h], v);
        v = __fmaf_rn(s1, D[u][2 * h + 1], v);
        v = __fmaf_rn(c0, X[u].x, v);
        v = __fmaf_rn(c1, X[u].y, v);
        acc[u][h] = v;
      }
    }
  };
  int c = 0;
  for (; c + 1 < nch; c += 2) {
    if (c + DEPTH - 2 < nch) issue(c + DEPTH - 2);
    cp_async_commit();
    if (c + DEPTH - 1 < nch) issue(c + DEPTH - 1);
    cp_async_commit();
    cp_async_wait<DEPTH - 2>();
    __syncwarp();
    process(c, 0);
    process(c + 1, 1);
    __syncwarp();
  }
  if (c < nch) {   // odd chunk count: the last chunk alone
    cp_async_wait<0>();
    __syncwarp();
    process(c, 0);
  }
  cp_async_wait<0>();

#pragma unroll
  for (int u = 0; u < MT2; ++u)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const float v = acc[u][h] + __shfl_xor_sync(0xFFFFFFFFu, acc[u][h], 1);
      if ((t & 1) == 0 && al[u]) red[(warp * p.M + 2 * u + t / 2) * 16 + g + 8 * h] = v;
    }
  __syncthreads();
  // Sum the KS slices in warp order into red[tok][row] (slice 0's place), then to y.
  for (int i = threadIdx.x; i < p.M * 16; i += KS * 32) {
    float v = red[i];
#pragma unroll
    for (int w = 1; w < KS; ++w) v += red[w * p.M * 16 + i];
    red[i] = v;
    if (gridDim.y == 1) {
      const int row = row0 + (i & 15);
      if (row < p.N) {
        __nv_bfloat16 hb = __float2bfloat16_rn(v);
        p.y[(size_t)(i >> 4) * p.N + row] = *reinterpret_cast<uint16_t *>(&hb);
      }
    }
  }
  if (gridDim.y > 1) cluster_sum_store<16>(p, red);
}

// ---------------------------------------------------------------------------------------
// LUT4, 1 <= M <= 4, K % 512 == 0, block in {32, 64, 128}: the K-split kernel with a
// codebook decode.  Byte j of a row holds elements 2j (high nibble) and 2j+1 (low nibble),
// so one byte is one bf16 pair in natural k order: the CTA builds a table of the 256 pairs
// (bf16(book[hi]), bf16(book[lo])), replicated 16 times so that the 32 lanes of a lookup
// fall on distinct banks except for lanes l and l+16, and each code byte costs one byte
// extract, one address multiply-add and one shared load.  x is staged in natural order.
// The block scales (f32, one per `block` consecutive k) arrive in 4-chunk blocks like the
// INT4 scales, and the group-column product applies them after the tensor core:
// sum_k book[q_k] s x_k = s * sum_k bf16(book[q_k]) x_k per group (LUT4 has no bias).
// ---------------------------------------------------------------------------------------
constexpr int kLutCopies = 16;
constexpr int kLutTableBytes = 256 * kLutCopies * 4;   // 16 KB

__host__ __device__ constexpr int lks_sb_slots(int depth) { return (depth + 2) / 4 + 1; }
__host__ __device__ inline int lks_row_pitch(int block) { return 2048 / block + 16; }   // scale bytes + pad
__host__ __device__ inline size_t lks_warp_bytes(int depth, int M, int maxc, int block) {
  return (size_t)depth * 1024 + (size_t)lks_sb_slots(depth) * 16 * lks_row_pitch(block) +
         (size_t)M * (maxc * 256 + 64);
}

template <int MT2, int KS, int DEPTH>
__global__ void __launch_bounds__(KS * 32) gemv_lks_kernel(const __grid_constant__ GemvParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr int kSlots = lks_sb_slots(DEPTH);
  const int block = p.lut_block_shift_div * 32;
  const int P = lks_row_pitch(block);
  const int maxc = p.max_chunks_per_cta;
  const int XS = maxc * 256 + 64;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int g = lane / 4, t = lane % 4;
  uint32_t *ltab = reinterpret_cast<uint32_t *>(smem);
  const size_t wbytes = lks_warp_bytes(DEPTH, p.M, maxc, block);
  uint8_t *wbase = smem + kLutTableBytes + (size_t)warp * wbytes;
  uint8_t *ring = wbase;
  uint8_t *sbr = wbase + DEPTH * 1024;
  uint8_t *xs = sbr + kSlots * 16 * P;
  float *red = reinterpret_cast<float *>(smem + kLutTableBytes + (size_t)KS * wbytes);   // [KS][M][16]

  const int splits = (int)gridDim.y * KS;
  const int sp = (int)blockIdx.y * KS + warp;
  const int c_begin = (int)(((long long)sp * p.chunks) / splits);
  const int c_end = (int)(((long long)(sp + 1) * p.chunks) / splits);
  const int nch = c_end - c_begin;
  const int row0 = blockIdx.x * 16;
  const int spr = p.lut_blocks_per_row;            // scales per row
  const int sblk = 512 / block;                    // scales per 4-chunk block
  const int cpr = 128 / block;                     // 16-byte copies per row per 4-chunk block

  const uint8_t *wsrc[2];
  bool live[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int row = row0 + g + 8 * h;
    live[h] = row < p.N;
    wsrc[h] = p.w + (live[h] ? (size_t)row * (size_t)(p.K / 2) : 0) + (size_t)c_begin * 64 + t * 16;
  }
  const uint32_t ring_s = smem_u32(ring), sb_s = smem_u32(sbr);
  const int blk0 = c_begin / 4;
  const float *scales = static_cast<const float *>(p.scales);
  auto issue = [&](int c) {
    const uint32_t slot = ring_s + (uint32_t)((c % DEPTH) * 1024);
#pragma unroll
    for (int h = 0; h < 2; ++h)
      cp_async(slot + h * 512 + lane * 16, wsrc[h] + (size_t)c * 64, 16, live[h] ? 16u : 0u);
    const int a = c_begin + c;
    if (c == 0 || (a & 3) == 0) {   // scales of chunks 4(a/4) .. +3, 16 rows
      const int b = a >> 2;
      const uint32_t sslot = sb_s + (uint32_t)(((b - blk0) % kSlots) * 16 * P);
      for (int i = lane; i < 16 * cpr; i += 32) {
        const int r = i / cpr, pc = i - r * cpr;
        const int row = row0 + r;
        const bool ok = row < p.N;
        cp_async(sslot + (uint32_t)(r * P + pc * 16), scales + (ok ? (size_t)row * spr + (size_t)b * sblk + pc * 4 : 0),
                 16, ok ? 16u : 0u);
      }
    }
  };

  // Chunks go through the loop in pairs; DEPTH - 2 chunks are in flight ahead of a pair.
  // They are issued first, so the weight stream is under way while the table is built.
#pragma unroll
  for (int i = 0; i < DEPTH - 2; ++i) {
    if (i < nch) issue(i);
    cp_async_commit();
  }
  // Pair table: entry (byte, copy) at ltab[byte * 16 + copy].
  for (int i = threadIdx.x; i < 256 * kLutCopies; i += KS * 32) {
    const int byte = i / kLutCopies;
    ltab[i] = pack_bf16x2(p.book[byte >> 4], p.book[byte & 15]);
  }
  // Weights are in flight; x may be the previous kernel's output, and y may still be read by it.
  griddep_launch_dependents();
  griddep_wait();
  for (int it = lane; it < p.M * nch * 16; it += 32) {   // this warp's x slice, 16 bytes a piece
    const int tok = it / (nch * 16), rem = it - tok * (nch * 16);
    *reinterpret_cast<uint4 *>(xs + (size_t)tok * XS + rem * 16) =
        __ldg(reinterpret_cast<const uint4 *>(p.x + (size_t)tok * p.K + (size_t)c_begin * 128) + rem);
  }
  __syncthreads();   // the table is shared by the CTA; x and rings are per warp

  bool bl[MT2], al[MT2];
  const uint8_t *xl[MT2];
#pragma unroll
  for (int u = 0; u < MT2; ++u) {
    const int tb = 2 * u + g / 4;
    bl[u] = (g & 3) == t && tb < p.M;
    xl[u] = xs + (size_t)(bl[u] ? tb : 0) * XS + t * 64;
    al[u] = 2 * u + t / 2 < p.M;
  }
  const uint32_t tab_lane = smem_u32(ltab) + (uint32_t)(lane & (kLutCopies - 1)) * 4u;
  float acc[MT2][2];
#pragma unroll
  for (int u = 0; u < MT2; ++u) acc[u][0] = acc[u][1] = 0.f;

  auto process = [&](int c) {
    const uint8_t *sl = ring + (c % DEPTH) * 1024;
    uint4 xb[4][MT2];
#pragma unroll
    for (int u = 0; u < MT2; ++u)
#pragma unroll
      for (int q = 0; q < 4; ++q)
        xb[q][u] = bl[u] ? *reinterpret_cast<const uint4 *>(xl[u] + c * 256 + q * 16) : make_uint4(0, 0, 0, 0);
    const uint4 q0 = *reinterpret_cast<const uint4 *>(sl + lane * 16);
    const uint4 q1 = *reinterpret_cast<const uint4 *>(sl + 512 + lane * 16);
    const int a = c_begin + c;
    const uint8_t *sc = sbr + ((a >> 2) - blk0) % kSlots * 16 * P;
    // groups 2(t&1), 2(t&1)+1 of this chunk -> scale indices within the 4-chunk block
    const int ga = (a & 3) * 4 + 2 * (t & 1);
    const int ia = (ga * 32) / block, ib = ((ga + 1) * 32) / block;
    float sa[2], sbv[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const float *srow = reinterpret_cast<const float *>(sc + (g + 8 * h) * P);
      sa[h] = srow[ia];
      sbv[h] = srow[ib];
    }
    float D[MT2][4];
#pragma unroll
    for (int u = 0; u < MT2; ++u) D[u][0] = D[u][1] = D[u][2] = D[u][3] = 0.f;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint32_t w0 = q == 0 ? q0.x : q == 1 ? q0.y : q == 2 ? q0.z : q0.w;
      const uint32_t w1 = q == 0 ? q1.x : q == 1 ? q1.y : q == 2 ? q1.z : q1.w;
      uint32_t v[8];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t sel = 0x4440u | (uint32_t)j;   // byte j, zero-extended
        const uint32_t b0 = prmt(w0, 0u, sel), b1 = prmt(w1, 0u, sel);
        asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v[2 * j]) : "r"(tab_lane + b0 * (kLutCopies * 4u)));
        asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v[2 * j + 1]) : "r"(tab_lane + b1 * (kLutCopies * 4u)));
      }
      // step 2q: k-slots (2t, 2t+1) <- byte 4q, (2t+8, 2t+9) <- byte 4q+1; step 2q+1: bytes 4q+2, 4q+3
      const uint32_t a0[4] = {v[0], v[1], v[2], v[3]};
      const uint32_t a1[4] = {v[4], v[5], v[6], v[7]};
#pragma unroll
      for (int u = 0; u < MT2; ++u) {
        mma_bf16_16816(D[u], a0, xb[q][u].x, xb[q][u].y);
        mma_bf16_16816(D[u], a1, xb[q][u].z, xb[q][u].w);
      }
    }
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int u = 0; u < MT2; ++u) {
        float v = acc[u][h];
        v = __fmaf_rn(sa[h], D[u][2 * h], v);
        v = __fmaf_rn(sbv[h], D[u][2 * h + 1], v);
        acc[u][h] = v;
      }
  };
  int c = 0;
  for (; c + 1 < nch; c += 2) {
    if (c + DEPTH - 2 < nch) issue(c + DEPTH - 2);
    cp_async_commit();
    if (c + DEPTH - 1 < nch) issue(c + DEPTH - 1);
    cp_async_commit();
    cp_async_wait<DEPTH - 2>();
    __syncwarp();
    process(c);
    process(c + 1);
    __syncwarp();
  }
  if (c < nch) {
    cp_async_wait<0>();
    __syncwarp();
    process(c);
  }
  cp_async_wait<0>();

#pragma unroll
  for (int u = 0; u < MT2; ++u)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const float v = acc[u][h] + __shfl_xor_sync(0xFFFFFFFFu, acc[u][h], 1);
      if ((t & 1) == 0 && al[u]) red[(warp * p.M + 2 * u + t / 2) * 16 + g + 8 * h] = v;
    }
  __syncthreads();
  for (int i = threadIdx.x; i < p.M * 16; i += KS * 32) {
    float v = red[i];
#pragma unroll
    for (int w = 1; w < KS; ++w) v += red[w * p.M * 16 + i];
    red[i] = v;
    if (gridDim.y == 1) {
      const int row = row0 + (i & 15);
      if (row < p.N) {
        __nv_bfloat16 hb = __float2bfloat16_rn(v);
        p.y[(size_t)(i >> 4) * p.N + row] = *reinterpret_cast<uint16_t *>(&hb);
      }
    }
  }
  if (gridDim.y > 1) cluster_sum_store<16>(p, red);
}

// A planned decode launch kept for replay (a dispatch record): the kernel, its launch
// configuration and attributes, and the shape part of its parameters.  Recording runs the
// same planning and per-kernel attribute set-up as a call, then stops short of the launch.
struct LaunchSpec {
  const void *fn = nullptr;
  cudaLaunchConfig_t cfg{};
  cudaLaunchAttribute attr[2]{};
  GemvParams params{};
  int tma_rows = 0;     // > 0: a TMA-fed kernel whose tensor maps are encoded per launch
  int tma_stages = 0;
};

template <typename Kern>
cudaError_t launch_or_record(const cudaLaunchConfig_t &cfg, Kern kern, const GemvParams &p, LaunchSpec *rec) {
  if (rec == nullptr) return cudaLaunchKernelEx(&cfg, kern, p);
  rec->fn = reinterpret_cast<const void *>(kern);
  rec->cfg = cfg;
  rec->cfg.numAttrs = cfg.numAttrs < 2 ? cfg.numAttrs : 2;
  for (unsigned i = 0; i < rec->cfg.numAttrs; ++i) rec->attr[i] = cfg.attrs[i];
  rec->cfg.attrs = nullptr;   // re-pointed at rec->attr by each replay
  rec->params = p;
  return cudaSuccess;
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
  // Pick (rows per warp, K splits) so that one wave of CTAs fills the SMs as evenly as
  // possible, with the fewest splits (each split re-stages x and adds a cluster
  // reduction) and at least ~12 chunk-rows in flight per SM.
  Plan best{};
  double best_score = -1e30;
  for (int RT = 2; RT >= 1; --RT) {
    const int rows_cta = kWarps * 16 * RT;
    const int rb = (N + rows_cta - 1) / rows_cta;
    for (int S = 1; S <= std::min(kMaxCluster, chunks); ++S) {
      const int maxc = (chunks + S - 1) / S;
      const size_t sm = smem_bytes(pl.MT, RT, maxc);
      if (sm > smem_cap) continue;
      int per_sm = std::min((int)(smem_cap / (sm + 1024)), 8);
      per_sm = std::max(per_sm, 1);
      const long long ctas = (long long)rb * S;
      const long long per_sm_needed = (ctas + sms - 1) / sms;          // CTAs on the busiest SM
      const double balance = (double)ctas / (double)(per_sm_needed * sms);
      const double waves = (double)per_sm_needed / per_sm;               // > 1: CTAs queue
      const double warps_per_sm = (double)std::min<long long>(per_sm_needed, per_sm) * kWarps;
      const double mlp = std::min(1.0, warps_per_sm * RT / 12.0);        // loads in flight
      double score = balance * mlp - 0.015 * S - (waves > 1.0 ? 0.05 * (waves - 1.0) : 0.0);
      if (maxc < 4) score -= 0.05 * (4 - maxc);                          // very short CTAs
      if (score > best_score) {
        best_score = score;
        best = Plan{pl.MT, RT, S, maxc, sm};
      }
    }
  }
  return best;
}

template <int MT, int RT, bool LUT>
cudaError_t launch_typed(const GemvParams &p, const Plan &pl, cudaStream_t s, bool overlap, LaunchSpec *rec) {
  auto kern = gemv_kernel<MT, RT, LUT>;
  cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void *>(kern), (int)pl.smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  const int rows_cta = kWarps * 16 * RT;
  cfg.gridDim = dim3((unsigned)((p.N + rows_cta - 1) / rows_cta), (unsigned)pl.S, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = pl.smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = (unsigned)pl.S;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = overlap ? 2 : 1;
  return launch_or_record(cfg, kern, p, rec);
}

size_t async_smem_bytes(int M, int MT, int RT, int max_chunks, bool sb) {
  const int d = async_depth(MT), slots = (d + 2) / 4 + 1;
  const size_t ring = sb ? (size_t)kWarps * (d * 1024 + slots * kSbSlot) * RT
                         : (size_t)kWarps * d * kStageBytes * RT;
  return ring + (size_t)M * (max_chunks * 256 + 64) +
         (size_t)8 * MT * kWarps * 16 * RT * 4 + 16 * 4 + (size_t)M * max_chunks * 4 * 2 + 16;
}

// All CTAs resident in one wave; among those plans, the best-balanced one with the most
// rows per warp and the fewest K splits.
size_t gc_smem_bytes(int M, int RT, int max_chunks);

// gc: plan for gemv_gc_kernel (INT4, M <= 4), whose shared-memory footprint differs.
Plan make_async_plan(int M, int N, int K, bool gc, bool sb) {
  Plan pl{};
  pl.MT = M <= 8 ? 1 : 2;
  const int chunks = K / 128;
  int sms = 152, dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && v > 0) sms = v;
  }
  double best = -1e30;
  for (int RT = 2; RT >= 1; --RT) {
    const int rb = (N + kWarps * 16 * RT - 1) / (kWarps * 16 * RT);
    for (int S = 1; S <= std::min(kMaxCluster, chunks); S *= 2) {   // clusters of 3, 5, 6, 7 pack poorly
      const int maxc = (chunks + S - 1) / S;
      const size_t sm = gc ? gc_smem_bytes(M, RT, maxc) : async_smem_bytes(M, pl.MT, RT, maxc, sb);
      if (sm > 227 * 1024) continue;
      const int per_sm = std::max(1, std::min((int)((228 * 1024) / (sm + 1024)), 8));
      if (pl.MT == 2 && !gc) {
        // 16 tokens: staging x caps CTAs per SM, so several waves can beat one.  Cost in
        // chunk-steps: waves x (chunks per warp x row tiles + per-CTA set-up and cluster
        // reduction), slowed when fewer than 16 row-tile streams share an SM (fitted to
        // timings on GB300 over K, N in {4096, 14336}).
        const long long ctas = (long long)rb * S;
        const long long waves = (ctas + (long long)sms * per_sm - 1) / ((long long)sms * per_sm);
        const long long busiest = (ctas + sms - 1) / sms;
        const double warps = (double)std::min<long long>(per_sm, busiest) * kWarps * RT;
        const double cost = (double)waves * (maxc * RT + 12.0 + 2.0 * S) / std::min(1.0, warps / 16.0);
        if (-cost > best) {
          best = -cost;
          pl.RT = RT;
          pl.S = S;
          pl.max_chunks = maxc;
          pl.smem = sm;
        }
        continue;
      }
      const long long ctas = (long long)rb * S;
      const long long need = (ctas + sms - 1) / sms;
      if (need > per_sm) continue;                                       // one wave only
      const double balance = (double)ctas / (double)(need * sms);
      const double warps = (double)need * kWarps * RT;                    // row-tile streams per SM
      double score = balance * std::min(1.0, warps / 12.0) - 0.02 * S + 0.01 * RT;
      if (maxc < 4) score -= 0.05 * (4 - maxc);
      if (score > best) {
        best = score;
        pl.RT = RT;
        pl.S = S;
        pl.max_chunks = maxc;
        pl.smem = sm;
      }
    }
  }
  return pl;
}

template <int MT, int RT, bool LUT>
cudaError_t launch_async_typed(const GemvParams &p, const Plan &pl, cudaStream_t s, bool overlap, LaunchSpec *rec) {
  auto kern = gemv_async_kernel<MT, RT, LUT, false>;
  if constexpr (!LUT) {
    if (p.K % 256 == 0) kern = gemv_async_kernel<MT, RT, false, true>;
  }
  cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void *>(kern), (int)pl.smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((p.N + kWarps * 16 * RT - 1) / (kWarps * 16 * RT)), (unsigned)pl.S, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = pl.smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = (unsigned)pl.S;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = overlap ? 2 : 1;
  return launch_or_record(cfg, kern, p, rec);
}

size_t gc_smem_bytes(int M, int RT, int max_chunks) {   // the larger of the two layouts (SB)
  return (size_t)kWarps * (kDepth * 1024 + kSbSlots * kSbSlot) * RT + (size_t)M * (max_chunks * 256 + 64) +
         (size_t)M * kWarps * 16 * RT * 4 + (size_t)M * max_chunks * 4 * 4;
}

template <int MT2, int RT>
cudaError_t launch_gc_typed(const GemvParams &p, const Plan &pl, cudaStream_t s, bool overlap, LaunchSpec *rec) {
  const bool sb = p.K % 256 == 0 && (reinterpret_cast<uintptr_t>(p.scales) & 15u) == 0 &&
                  (reinterpret_cast<uintptr_t>(p.biases) & 15u) == 0;
  auto kern = sb ? gemv_gc_kernel<MT2, RT, true> : gemv_gc_kernel<MT2, RT, false>;
  const size_t smem = gc_smem_bytes(p.M, RT, pl.max_chunks);
  cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void *>(kern), (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((p.N + kWarps * 16 * RT - 1) / (kWarps * 16 * RT)), (unsigned)pl.S, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = (unsigned)pl.S;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = overlap ? 2 : 1;
  return launch_or_record(cfg, kern, p, rec);
}

struct KsPlan {
  int KS = 0, S = 0, depth = 0, maxc = 0;
  size_t smem = 0;
};

// Shapes for gemv_ks_kernel: all CTAs in one wave, as evenly spread over the SMs as possible,
// with enough warps per SM to hide latency and enough chunk stages in flight per SM to keep
// HBM busy; K splits across CTAs (clusters) only when the K split inside a CTA is not enough.
KsPlan make_ks_plan(int M, int N, int K) {
  KsPlan best;
  int sms = 152, dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && v > 0) sms = v;
  }
  const int R = (N + 15) / 16, C = K / 128;
  const int regs = M <= 2 ? 80 : 104;   // per thread, at least what ptxas -v reports
  double best_score = -1e30;
  for (int depth : {4, 8})
    for (int KS : {2, 4, 8})
      for (int S : {1, 2, 4, 8}) {
        if (KS * S > C) continue;
        const int maxc = (C + KS * S - 1) / (KS * S);
        const size_t smem = (size_t)KS * ks_warp_bytes(depth, M, maxc) + (size_t)KS * M * 16 * 4;
        if (smem > 227 * 1024) continue;
        int per_sm = (int)((228 * 1024) / (smem + 1024));
        per_sm = std::min(per_sm, 2048 / (KS * 32));
        per_sm = std::min(per_sm, 65536 / (KS * 32 * regs));
        per_sm = std::min(per_sm, 32);
        if (per_sm < 1) continue;
        const long long ctas = (long long)R * S;
        const long long need = (ctas + sms - 1) / sms;
        if (need > per_sm) continue;
        const double balance = (double)ctas / (double)(need * sms);
        const double warps = (double)need * KS;                       // on the busiest SM
        const double stages_kb = warps * (depth - 1);                  // code stages in flight
        double score = balance * std::min(1.0, warps / 12.0) * std::min(1.0, stages_kb / 48.0);
        score -= (S > 1 ? 0.15 : 0.0) + 0.01 * S;   // cluster reductions measured 10-20% slower
        score += depth == 8 ? 0.01 : 0.0;            // deeper rings measured faster at equal occupancy
        if (maxc < 4) score -= 0.04 * (4 - maxc);
        if (score > best_score) {
          best_score = score;
          best.KS = KS; best.S = S; best.depth = depth; best.maxc = maxc; best.smem = smem;
        }
      }
  return best;
}

template <int MT2, int KS, int DEPTH>
cudaError_t launch_ks_typed(const GemvParams &p, const KsPlan &pl, cudaStream_t s, bool overlap, LaunchSpec *rec) {
  auto kern = gemv_ks_kernel<MT2, KS, DEPTH>;
  cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void *>(kern), (int)pl.smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((p.N + 15) / 16), (unsigned)pl.S, 1);
  cfg.blockDim = dim3(KS * 32, 1, 1);
  cfg.dynamicSmemBytes = pl.smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  int n = 0;
  if (pl.S > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = 1;
    attr[n].val.clusterDim.y = (unsigned)pl.S;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  if (overlap) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = (unsigned)n;
  return launch_or_record(cfg, kern, p, rec);
}

template <int MT2>
cudaError_t launch_ks(const GemvParams &p, const KsPlan &pl, cudaStream_t s, bool overlap, LaunchSpec *rec) {
  if (pl.depth == 4) {
    if (pl.KS == 2) return launch_ks_typed<MT2, 2, 4>(p, pl, s, overlap, rec);
    if (pl.KS == 4) return launch_ks_typed<MT2, 4, 4>(p, pl, s, overlap, rec);
    return launch_ks_typed<MT2, 8, 4>(p, pl, s, overlap, rec);
  }
  if (pl.KS == 2) return launch_ks_typed<MT2, 2, 8>(p, pl, s, overlap, rec);
  if (pl.KS == 4) return launch_ks_typed<MT2, 4, 8>(p, pl, s, overlap, rec);
  return launch_ks_typed<MT2, 8, 8>(p, pl, s, overlap, rec);
}

// Plans for gemv_lks_kernel: the K-split plan search with the codebook table in each CTA.
KsPlan make_lks_plan(int M, int N, int K, int block) {
  KsPlan best;
  int sms = 152, dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && v > 0) sms = v;
  }
  const int R = (N + 15) / 16, C = K / 128;
  const int regs = M <= 2 ? 80 : 104;   // at least what ptxas -v reports
  double best_score = -1e30;
  for (int depth : {4, 8})
    for (int KS : {2, 4, 8})
      for (int S : {1, 2, 4, 8}) {
        if (KS * S > C) continue;
        const int maxc = (C + KS * S - 1) / (KS * S);
        const size_t smem = (size_t)kLutTableBytes + (size_t)KS * lks_warp_bytes(depth, M, maxc, block) +
                            (size_t)KS * M * 16 * 4;
        if (smem > 227 * 1024) continue;
        int per_sm = (int)((228 * 1024) / (smem + 1024));
        per_sm = std::min(per_sm, 2048 / (KS * 32));
        per_sm = std::min(per_sm, 65536 / (KS * 32 * regs));
        per_sm = std::min(per_sm, 32);
        if (per_sm < 1) continue;
        const long long ctas = (long long)R * S;
        const long long need = (ctas + sms - 1) / sms;
        if (need > per_sm) continue;
        const double balance = (double)ctas / (double)(need * sms);
        const double warps = (double)need * KS;
        const double stages_kb = warps * (depth - 1);
        double score = balance * std::min(1.0, warps / 12.0) * std::min(1.0, stages_kb / 48.0);
        score -= (S > 1 ? 0.15 : 0.0) + 0.01 * S;
        score += depth == 8 ? 0.01 : 0.0;
        if (maxc < 4) score -= 0.04 * (4 - maxc);
        if (score > best_score) {
          best_score = score;
          best.KS = KS; best.S = S; best.depth = depth; best.maxc = maxc; best.smem = smem;
        }
      }
  return best;
}

template <int MT2, int KS, int DEPTH>
cudaError_t launch_lks_typed(const GemvParams &p, const KsPlan &pl, cudaStream_t s, bool overlap, LaunchSpec *rec) {
  auto kern = gemv_lks_kernel<MT2, KS, DEPTH>;
  cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void *>(kern), (int)pl.smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((p.N + 15) / 16), (unsigned)pl.S, 1);
  cfg.blockDim = dim3(KS * 32, 1, 1);
  cfg.dynamicSmemBytes = pl.smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  int n = 0;
  if (pl.S > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = 1;
    attr[n].val.clusterDim.y = (unsigned)pl.S;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  if (overlap) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = (unsigned)n;
  return launch_or_record(cfg, kern, p, rec);
}

template <int MT2>
cudaError_t launch_lks(const GemvParams &p, const KsPlan &pl, cudaStream_t s, bool overlap, LaunchSpec *rec) {
  if (pl.depth == 4) {
    if (pl.KS == 2) return launch_lks_typed<MT2, 2, 4>(p, pl, s, overlap, rec);
    if (pl.KS == 4) return launch_lks_typed<MT2, 4, 4>(p, pl, s, overlap, rec);
    return launch_lks_typed<MT2, 8, 4>(p, pl, s, overlap, rec);
  }
  if (pl.KS == 2) return launch_lks_typed<MT2, 2, 8>(p, pl, s, overlap, rec);
  if (pl.KS == 4) return launch_lks_typed<MT2, 4, 8>(p, pl, s, overlap, rec);
  return launch_lks_typed<MT2, 8, 8>(p, pl, s, overlap, rec);
}

#include "gemv_tma.cuh"

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

// Tensor maps of one decode call: codes uint8 [N][K/2] in 128-byte boxes with the 128-byte
// swizzle, scales and biases bf16 [N][K/32] in 8-group boxes; R rows per box, zero fill past N.
cudaError_t make_tq_maps(GemvTmaArgs &a, int R) {
  auto enc = tensor_map_encoder();
  if (!enc) return cudaErrorNotSupported;
  const GemvParams &p = a.p;
  const cuuint32_t estr[2] = {1, 1};
  {
    const cuuint64_t dims[2] = {(cuuint64_t)(p.K / 2), (cuuint64_t)p.N};
    const cuuint64_t strides[1] = {(cuuint64_t)(p.K / 2)};
    const cuuint32_t box[2] = {128u, (cuuint32_t)R};
    if (enc(&a.wmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(p.w), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  const cuuint64_t dims[2] = {(cuuint64_t)(p.K / 32), (cuuint64_t)p.N};
  const cuuint64_t strides[1] = {(cuuint64_t)(p.K / 32) * 2};
  const cuuint32_t box[2] = {8u, (cuuint32_t)R};
  if (enc(&a.smap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(p.scales), dims, strides, box, estr,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS ||
      enc(&a.bmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t *>(p.biases), dims, strides, box, estr,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  return cudaSuccess;
}

struct TqPlan {
  int WC = 0, KS = 1, S = 0, maxnh = 0, stages = 0;
  size_t smem = 0;
};

// Plans for gemv_tma_kernel, from sweeps of (consumer warps, consumer groups, K splits,
// stages) over the decode shapes on GB300.  What they showed: every CTA resident at once and
// at most two CTAs per SM (the next call's CTAs then find room to start streaming while this
// call finishes); the decode arithmetic, not the stream, bounds the kernel, so more consumer
// warps per SM help: 12 consumer warps in two groups over 96-row tiles (6 x 2) win wherever
// their one-CTA-per-SM grid covers nearly every SM (N = 14336: 150 CTAs); otherwise 8
// consumer warps in one group with the K split that spreads the CTAs best.  Each CTA takes
// as many ring stages as its share of shared memory holds.
TqPlan tq_plan_for(int M, int N, int K, int WC, int KS, int S, int sms, int max_need) {
  TqPlan pl;
  const int NH = K / 256, NB = (NH + 1) / 2;
  if (S > NB) return pl;
  const int R = 16 * WC, threads = (WC * KS + 1) * 32, regs = 112;   // regs: >= what ptxas -v reports
  int maxnh = 0;
  for (int sp = 0; sp < S; ++sp) {
    const int b0 = (sp * NB) / S, b1 = ((sp + 1) * NB) / S;
    maxnh = std::max(maxnh, std::min(2 * b1, NH) - 2 * b0);
  }
  const long long ctas = (long long)((N + R - 1) / R) * S;
  const int need = (int)((ctas + sms - 1) / sms);   // CTAs on the busiest SM
  if (need > max_need || need * threads * regs > 65536) return pl;
  // Ring stages.  One consumer group: as many as the CTA's share of shared memory holds
  // (up to 8; measured best).  Two groups (512-k stages): only what fits in half of the SM,
  // at least 2; measured best, since the rest lets the next call's CTAs start early.
  const size_t budget = (size_t)(227 * 1024) / need;
  const size_t fixed = tq_smem_bytes(M, maxnh, R, KS, 0);
  if (fixed >= budget) return pl;
  const size_t per = tq_stage_bytes(R, KS) + 16;
  int stages = (int)std::min<size_t>(8, (budget - fixed) / per);
  if (KS > 1) {
    const size_t half_sm = (size_t)(113 * 1024) / need;
    const int s_half = fixed < half_sm ? (int)((half_sm - fixed) / per) : 0;
    stages = std::min(stages, std::max(s_half, 2));
  }
  if (stages < 2 || stages * KS < 3) return pl;
  pl.WC = WC; pl.KS = KS; pl.S = S; pl.maxnh = maxnh; pl.stages = stages;
  pl.smem = tq_smem_bytes(M, maxnh, R, KS, stages);
  return pl;
}

TqPlan make_tq_plan(int M, int N, int K) {
  int sms = 152, dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && v > 0) sms = v;
  }
  // 12 consumer warps (6 rows groups x 2 consumer groups), one CTA per SM, no K split.
  const TqPlan wide = tq_plan_for(M, N, K, 6, 2, 1, sms, 1);
  if (wide.WC > 0 && (double)((N + 95) / 96) / sms >= 0.95) return wide;
  TqPlan best;
  double best_score = -1e30;
  for (int WC : {8, 4})
    for (int S : {1, 2, 4, 8}) {
      const TqPlan pl = tq_plan_for(M, N, K, WC, 1, S, sms, 2);
      if (pl.WC == 0) continue;
      const long long ctas = (long long)((N + 16 * WC - 1) / (16 * WC)) * S;
      const int need = (int)((ctas + sms - 1) / sms);
      const double balance = (double)ctas / (double)((long long)need * sms);
      const double score = balance * std::min(1.0, need * WC / 8.0) - 1e-3 * S;
      if (score > best_score + 1e-9) {
        best_score = score;
        best = pl;
      }
    }
  return best;
}

template <int NT, int WC, int KS>
cudaError_t launch_tq_typed(GemvParams &p, const TqPlan &pl, cudaStream_t s, bool overlap, LaunchSpec *rec) {
  auto kern = gemv_tma_kernel<NT, WC, KS>;
  cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void *>(kern), (int)pl.smem);
  if (e != cudaSuccess) return e;
  p.max_chunks_per_cta = pl.maxnh;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((p.N + 16 * WC - 1) / (16 * WC)), (unsigned)pl.S, 1);
  cfg.blockDim = dim3((WC * KS + 1) * 32, 1, 1);
  cfg.dynamicSmemBytes = pl.smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  int n = 0;
  if (pl.S > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = 1;
    attr[n].val.clusterDim.y = (unsigned)pl.S;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  if (overlap) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = (unsigned)n;
  if (rec != nullptr) {
    rec->fn = reinterpret_cast<const void *>(kern);
    rec->cfg = cfg;
    for (int i = 0; i < n; ++i) rec->attr[i] = attr[i];
    rec->cfg.attrs = nullptr;   // re-pointed at rec->attr by each replay
    rec->params = p;
    rec->tma_rows = 16 * WC;
    rec->tma_stages = pl.stages;
    return cudaSuccess;
  }
  GemvTmaArgs args{};
  args.p = p;
  args.stages = pl.stages;
  e = make_tq_maps(args, 16 * WC);
  if (e != cudaSuccess) return e;
  return cudaLaunchKernelEx(&cfg, kern, args);
}

template <int NT>
cudaError_t launch_tq_w(GemvParams &p, const TqPlan &pl, cudaStream_t s, bool overlap, LaunchSpec *rec) {
  if (pl.KS == 2) {
    if (pl.WC == 4) return launch_tq_typed<NT, 4, 2>(p, pl, s, overlap, rec);
    if (pl.WC == 6) return launch_tq_typed<NT, 6, 2>(p, pl, s, overlap, rec);
    return launch_tq_typed<NT, 8, 2>(p, pl, s, overlap, rec);
  }
  if (pl.WC == 4) return launch_tq_typed<NT, 4, 1>(p, pl, s, overlap, rec);
  return launch_tq_typed<NT, 8, 1>(p, pl, s, overlap, rec);
}

#ifdef Q4MM_TUNING
// Tuning builds only: environment overrides of the decode plan, for plan sweeps.
int tuning_env(const char *name, int dflt) {
  const char *v = getenv(name);
  return v ? atoi(v) : dflt;
}
#endif

template <bool LUT>
cudaError_t launch_any(GemvParams &p, cudaStream_t s, bool overlap, LaunchSpec *rec = nullptr) {
  p.chunks = (p.K / 32 + 3) / 4;
  // INT4 with K % 256 == 0: the TMA-fed kernel for 3 <= M <= 16; at M <= 2 the K-split
  // group-column kernel below measured faster on the decode shapes.
  bool use_tq = !LUT && p.M >= 3 && p.M <= 16 && p.K % 256 == 0;
#ifdef Q4MM_TUNING
  if (!LUT && p.M <= 16 && p.K % 256 == 0 && getenv("Q4MM_TQ_W")) use_tq = true;
  use_tq = use_tq && tuning_env("Q4MM_TQ", 1) != 0;
#endif
  if (use_tq) {
    TqPlan tp = make_tq_plan(p.M, p.N, p.K);
#ifdef Q4MM_TUNING
    if (getenv("Q4MM_TQ_W") || getenv("Q4MM_TQ_S") || getenv("Q4MM_TQ_ST")) {
      tp.WC = tuning_env("Q4MM_TQ_W", tp.WC);
      tp.KS = tuning_env("Q4MM_TQ_KS", tp.KS);
      tp.S = tuning_env("Q4MM_TQ_S", tp.S);
      const int NH = p.K / 256, NB = (NH + 1) / 2;
      tp.maxnh = 0;
      for (int sp = 0; sp < tp.S; ++sp) {
        const int b0 = (sp * NB) / tp.S, b1 = ((sp + 1) * NB) / tp.S;
        tp.maxnh = std::max(tp.maxnh, std::min(2 * b1, NH) - 2 * b0);
      }
      tp.stages = tuning_env("Q4MM_TQ_ST", tp.stages);
      tp.smem = tq_smem_bytes(p.M, tp.maxnh, 16 * tp.WC, tp.KS, tp.stages);
    }
#endif
    if (tp.WC > 0) return p.M <= 8 ? launch_tq_w<1>(p, tp, s, overlap, rec) : launch_tq_w<2>(p, tp, s, overlap, rec);
  }
  if (LUT && p.M <= 4 && p.K % 512 == 0 &&
      (p.lut_block_shift_div == 1 || p.lut_block_shift_div == 2 || p.lut_block_shift_div == 4) &&
      (reinterpret_cast<uintptr_t>(p.scales) & 15u) == 0) {
    const KsPlan kp = make_lks_plan(p.M, p.N, p.K, p.lut_block_shift_div * 32);
    if (kp.KS > 0) {
      p.max_chunks_per_cta = kp.maxc;
      return p.M <= 2 ? launch_lks<1>(p, kp, s, overlap, rec) : launch_lks<2>(p, kp, s, overlap, rec);
    }
  }
  if (!LUT && p.M <= 4 && p.K % 256 == 0) {
    const KsPlan kp = make_ks_plan(p.M, p.N, p.K);
    if (kp.KS > 0) {
      p.max_chunks_per_cta = kp.maxc;
      return p.M <= 2 ? launch_ks<1>(p, kp, s, overlap, rec) : launch_ks<2>(p, kp, s, overlap, rec);
    }
  }
  const bool lut_ok = !LUT || (p.lut_block_shift_div == 1 || p.lut_block_shift_div == 2 ||
                               p.lut_block_shift_div % 4 == 0);
  if (p.K % 128 == 0 && lut_ok) {
    const bool sb = !LUT && p.K % 256 == 0;
    const Plan pa = make_async_plan(p.M, p.N, p.K, !LUT && p.M <= 4, sb);
    if (pa.S > 0) {
      p.max_chunks_per_cta = pa.max_chunks;
      if (!LUT && p.M <= 4) {
        if (p.M <= 2)
          return pa.RT == 2 ? launch_gc_typed<1, 2>(p, pa, s, overlap, rec) : launch_gc_typed<1, 1>(p, pa, s, overlap, rec);
        return pa.RT == 2 ? launch_gc_typed<2, 2>(p, pa, s, overlap, rec) : launch_gc_typed<2, 1>(p, pa, s, overlap, rec);
      }
      if (pa.MT == 1)
        return pa.RT == 2 ? launch_async_typed<1, 2, LUT>(p, pa, s, overlap, rec) : launch_async_typed<1, 1, LUT>(p, pa, s, overlap, rec);
      return pa.RT == 2 ? launch_async_typed<2, 2, LUT>(p, pa, s, overlap, rec) : launch_async_typed<2, 1, LUT>(p, pa, s, overlap, rec);
    }
  }
  const Plan pl = make_plan(p.M, p.N, p.K);
  p.max_chunks_per_cta = pl.max_chunks;
  if (pl.MT == 1) {
    return pl.RT == 2 ? launch_typed<1, 2, LUT>(p, pl, s, overlap, rec) : launch_typed<1, 1, LUT>(p, pl, s, overlap, rec);
  }
  return pl.RT == 2 ? launch_typed<2, 2, LUT>(p, pl, s, overlap, rec) : launch_typed<2, 1, LUT>(p, pl, s, overlap, rec);
}

}  // namespace

cudaError_t launch_q4_gemv(const uint16_t *x, const uint32_t *w, const uint16_t *scales,
                           const uint16_t *biases, uint16_t *y, int M, int N, int K,
                           cudaStream_t s, bool overlap) {
  GemvParams p{};
  p.x = x;
  p.w = reinterpret_cast<const uint8_t *>(w);
  p.scales = scales;
  p.biases = biases;
  p.y = y;
  p.M = M; p.N = N; p.K = K;
  return launch_any<false>(p, s, overlap);
}

// Dispatch records for q4_gemv: plan once (kernel choice, grid, cluster, shared memory,
// the kernel's attribute set-up), then replay with new pointers.
cudaError_t record_q4_gemv(int M, int N, int K, bool overlap, void **out) {
  GemvParams p{};
  p.M = M; p.N = N; p.K = K;
  LaunchSpec *rec = new (std::nothrow) LaunchSpec();
  if (rec == nullptr) return cudaErrorMemoryAllocation;
  const cudaError_t e = launch_any<false>(p, nullptr, overlap, rec);
  if (e != cudaSuccess || rec->fn == nullptr) {
    delete rec;
    return e != cudaSuccess ? e : cudaErrorInvalidValue;
  }
  *out = rec;
  return cudaSuccess;
}

cudaError_t replay_q4_gemv(const void *record, const uint16_t *x, const uint32_t *w, const uint16_t *scales,
                           const uint16_t *biases, uint16_t *y, cudaStream_t s) {
  const LaunchSpec *rec = static_cast<const LaunchSpec *>(record);
  GemvParams p = rec->params;
  p.x = x;
  p.w = reinterpret_cast<const uint8_t *>(w);
  p.scales = scales;
  p.biases = biases;
  p.y = y;
  cudaLaunchConfig_t cfg = rec->cfg;
  cfg.attrs = const_cast<cudaLaunchAttribute *>(rec->attr);
  cfg.stream = s;
  if (rec->tma_rows > 0) {   // the tensor maps hold the pointers: encode them for this launch
    GemvTmaArgs ta{};
    ta.p = p;
    ta.stages = rec->tma_stages;
    const cudaError_t e = make_tq_maps(ta, rec->tma_rows);
    if (e != cudaSuccess) return e;
    void *args[] = {&ta};
    return cudaLaunchKernelExC(&cfg, rec->fn, args);
  }
  void *args[] = {&p};
  return cudaLaunchKernelExC(&cfg, rec->fn, args);
}

void free_q4_gemv_record(void *record) { delete static_cast<LaunchSpec *>(record); }

cudaError_t launch_lut4_gemv(const uint16_t *x, const uint8_t *packed, const float *scales,
                             const float *book, uint16_t *y, int M, int N, int K, int block,
                             cudaStream_t s, bool overlap) {
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
  return launch_any<true>(p, s, overlap);
}

}  // namespace q4mm
