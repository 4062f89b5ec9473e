// gemm_tc.cu -- prefill matmul (M > 16) on the fifth-generation tensor cores:
// q4_gemm (INT4 group-32 affine) and the fused LUT4 path of lut4_matmul.
//
// What it computes: y[m][n] = sum_k x[m][k] * W[n][k], W dequantised as in
// quant_fastkernel.rs (nibble*scale + bias, low nibble first; module doc "Algorithm":
// per K chunk, dequantise the W tile into shared memory, then tensor-core MMA with fp32
// accumulation, then store bf16) or as in lut4.rs (fl32(book[code] * scale), high nibble
// for even flat index).  The Metal design on those pages (BM=64/BN=32 threadgroup tiles,
// simdgroup 8x8 MMA, a half-precision transposed W tile) is prior art only; this is the
// GB300 design:
//
// Two kernels:
//
//  qgemm_tma_kernel<LUT, TT, SPLIT> (K % 256 == 0; every prefill shape of the workload):
//  * Weights are the MMA's M side: a tile is 128 weight rows x TT tokens, TT in {384, 256,
//    128}, its fp32 accumulator in tensor memory.  TT = 256 / 128 keep two accumulators
//    (2 TT columns), so the epilogue of one tile overlaps the main loop of the next;
//    TT = 384 takes one 384-column accumulator (two MMAs per k step, N = 256 + 128), so a
//    dequantised weight tile serves 1.5 times as many tokens.
//  * SPLIT = false: persistent CTAs, one per SM, walk the tiles with the weight tile
//    varying fastest, so the CTAs running at one time share a few x tiles in L2.
//    SPLIT = true (small M): one (tile, K slice) per CTA, the K slices of a tile form a
//    cluster and sum their fp32 partials in rank order through distributed shared memory.
//  * Warp 0, one lane: TMA loads of the x tiles (bf16, 128-byte swizzle), of the code tiles
//    [128 rows x 32 B] per 64-wide K block and of the scale / bias tiles per 8 K blocks.
//  * Warps 2-9 (256 threads, two per weight row, 32 k each): dequantise from shared memory
//    (INT4: magic-number bf16 conversion + one bf16x2 FMA per pair, so each value is
//    code*s+b rounded once; LUT4: codebook lookup, one fp32 product, rounded to bf16) into
//    the 128-byte-swizzled K-major bf16 tile the MMA reads.
//  * Warp 1, one lane: issues tcgen05.mma (M = 128, K = 16) x4 per K block (x8 for
//    TT = 384) and commits each stage back to the producers and each finished accumulator
//    to the epilogue.
//  * Warps 10-13: tcgen05.ld 32 columns at a time, round to bf16, store y, release the
//    accumulator.
//
//  qgemm_tc_kernel (any K % 32 == 0): the same roles with 256-token tiles, 4 producer warps
//  that load the codes with plain 16-byte loads instead of TMA, and one CTA per SM.
//
//  Every mbarrier wait is bounded (a timeout sets the device error word and unwinds the
//  CTA; tensor memory is always released).
#include "tc_common.cuh"

#include <cstdlib>

#include <cudaTypedefs.h>

namespace q4mm {

Q4MM_DEFINE_ERROR_READER(read_errors_gemm)

namespace {

constexpr int kTileW = 128;     // weight rows per CTA (MMA M)
constexpr int kTileT = 256;     // tokens per CTA (MMA N)
constexpr int kBK = 64;         // K per pipeline stage (one 128-byte swizzle row)
constexpr int kStages = 4;
constexpr int kThreads = 320;   // warp 0 TMA, warp 1 MMA, warps 2-5 producers, warps 6-9 epilogue
constexpr uint32_t kTmemCols = 512;   // two 256-column fp32 accumulators
constexpr uint32_t kABytes = kTileW * kBK * 2;   // 16 KB
constexpr uint32_t kBBytes = kTileT * kBK * 2;   // 32 KB

struct TcGemmParams {
  const uint8_t *w;        // row n at w + n*(K/2)
  const void *scales;      // INT4: bf16 [N, K/32]; LUT4: f32 [N * K/block]
  const uint16_t *biases;  // INT4 only
  uint16_t *y;             // bf16 [M, N]
  int M, N, K;
  int lut_blocks_per_row;  // LUT4: K / block
  int lut_kb_per_block;    // LUT4: block / 64
  int lut_sc_box;          // LUT4 TMA path: f32 scales per 8 K blocks (8 for block 64, 4 for 128)
  int ksplit;              // TMA path: 1 = persistent tiles; S > 1 = each tile's K split over a
                           // cluster of S CTAs (K / 64 a multiple of 8 S), partials summed in DSMEM
  float book[16];
};

struct SmemLayout {
  static constexpr uint32_t a = 0;
  static constexpr uint32_t b = a + kStages * kABytes;
  static constexpr uint32_t bars = b + kStages * kBBytes;  // full_a, full_b, empty, acc_full[2], acc_empty[2]
  static constexpr uint32_t misc = bars + (3 * kStages + 4) * 8;
  static constexpr uint32_t book = misc + 16;
  static constexpr uint32_t total = book + 16 * 4;
};
constexpr size_t kSmemBytes = SmemLayout::total + 1024;   // + alignment slack

// Raw operand of one weight row for one 64-wide K block.
struct RawKb {
  uint4 q0, q1;      // 64 codes
  uint32_t s, b;     // INT4: bf16 scale/bias of groups (2kb, 2kb+1) in low/high half; LUT4: f32 scale
};

template <bool LUT>
__device__ __forceinline__ void load_kb(RawKb &r, const TcGemmParams &p, int row, int kb) {
  r.q0 = make_uint4(0, 0, 0, 0);
  r.q1 = make_uint4(0, 0, 0, 0);
  r.s = 0;
  r.b = 0;
  if (row >= p.N) return;
  const int k0 = kb * kBK;
  const uint8_t *src = p.w + (size_t)row * (size_t)(p.K / 2) + (size_t)k0 / 2;
  const bool second = k0 + 32 < p.K;
  r.q0 = ldg_stream_v4(src);
  if (second) r.q1 = ldg_stream_v4(src + 16);
  if constexpr (LUT) {
    const float *sc = static_cast<const float *>(p.scales);
    r.s = __float_as_uint(__ldg(sc + (size_t)row * p.lut_blocks_per_row + kb / p.lut_kb_per_block));
  } else {
    const int G = p.K / 32;
    const size_t gi = (size_t)row * G + 2 * kb;
    const uint16_t *sc = static_cast<const uint16_t *>(p.scales);
    uint32_t s0 = ldg_u16(sc + gi), b0 = ldg_u16(p.biases + gi), s1 = 0, b1 = 0;
    if (second) {
      s1 = ldg_u16(sc + gi + 1);
      b1 = ldg_u16(p.biases + gi + 1);
    }
    r.s = s0 | (s1 << 16);
    r.b = b0 | (b1 << 16);
  }
}

// Eight consecutive k values (word c of the block) as four natural-order bf16 pairs.
template <bool LUT>
__device__ __forceinline__ uint4 decode_chunk(uint32_t word, int c, const RawKb &r, const float *book) {
  if constexpr (LUT) {
    const float s = __uint_as_float(r.s);
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t hi = (word >> (8 * j + 4)) & 0xFu;   // even k
      const uint32_t lo = (word >> (8 * j)) & 0xFu;       // odd k
      o[j] = pack_bf16x2(book[hi] * s, book[lo] * s);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
  } else {
    const uint32_t sh = c < 4 ? 0u : 16u;                 // words 0-3: group 2kb, 4-7: 2kb+1
    const uint32_t sv = (r.s >> sh) & 0xFFFFu, bv = (r.b >> sh) & 0xFFFFu;
    const Int4Pairs P = int4_word_to_bf16_pairs(word, sv | (sv << 16), bv | (bv << 16));
    // P[i] = (k=i, k=i+4)  ->  (0,1) (2,3) (4,5) (6,7)
    return make_uint4(prmt(P.p[0], P.p[1], 0x5410), prmt(P.p[2], P.p[3], 0x5410),
                      prmt(P.p[0], P.p[1], 0x7632), prmt(P.p[2], P.p[3], 0x7632));
  }
}

// Persistent: one CTA per SM walks tiles blockIdx.x, blockIdx.x + gridDim.x, ...; tile t is
// (token tile t / n_tiles, weight-row tile t % n_tiles), so the CTAs running at one time
// share a few x tiles in L2 while the weight tiles (all of which fit) stay there too.  Every
// role counts pipeline steps j = (tile index within the CTA) * KB + kb.
template <bool LUT>
__global__ void __launch_bounds__(kThreads, 1)
    qgemm_tc_kernel(const __grid_constant__ CUtensorMap tmap_x, const __grid_constant__ TcGemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = smem_u32(smem_raw);
  const uint32_t base = (raw_base + 1023u) & ~1023u;
  uint8_t *smem = smem_raw + (base - raw_base);

  const uint32_t sA = base + SmemLayout::a;
  const uint32_t sB = base + SmemLayout::b;
  const uint32_t bar_full_a = base + SmemLayout::bars;
  const uint32_t bar_full_b = bar_full_a + kStages * 8;
  const uint32_t bar_empty = bar_full_b + kStages * 8;
  const uint32_t bar_acc_full = bar_empty + kStages * 8;    // [2]
  const uint32_t bar_acc_empty = bar_acc_full + 2 * 8;      // [2]
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + SmemLayout::misc);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + SmemLayout::misc + 4);
  float *book = reinterpret_cast<float *>(smem + SmemLayout::book);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int KB = (p.K + kBK - 1) / kBK;
  const int m_tiles = (p.M + kTileT - 1) / kTileT;
  const int n_tiles = (p.N + kTileW - 1) / kTileW;
  const int T = m_tiles * n_tiles;
  const int my_tiles = (int)blockIdx.x < T ? (T - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
  const int steps = my_tiles * KB;
  auto tile_of = [&](int i) { return (int)blockIdx.x + i * (int)gridDim.x; };

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      tc::mbar_init(bar_full_a + 8 * s, 128);
      tc::mbar_init(bar_full_b + 8 * s, 1);
      tc::mbar_init(bar_empty + 8 * s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(bar_acc_full + 8 * b, 1);
      tc::mbar_init(bar_acc_empty + 8 * b, 4);
    }
    *abort_flag = 0;
    tc::fence_mbar_init();
    tc::tma_prefetch_desc(&tmap_x);
  }
  if (LUT && threadIdx.x < 16) book[threadIdx.x] = p.book[threadIdx.x];
  if (warp == 1) {
    tc::tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ---------------- TMA producer: x tiles ----------------
    if (lane == 0) {
      int issued = 0;
      for (int j = 0; j < steps; ++j) {
        const int i = j / KB, kb = j - i * KB;
        const int m0 = (tile_of(i) / n_tiles) * kTileT;
        const int s = j % kStages;
        const uint32_t ph = (j / kStages) & 1;
        if (!tc::mbar_wait(bar_empty + 8 * s, ph ^ 1, abort_flag)) break;
        tc::mbar_arrive_expect_tx(bar_full_b + 8 * s, kBBytes);
        tc::tma_load_2d(sB + s * kBBytes, &tmap_x, kb * kBK, m0, bar_full_b + 8 * s);
        ++issued;
      }
      if (*abort_flag) {
        // drain our own copies still in flight before the CTA can exit
        for (int j = (issued > kStages ? issued - kStages : 0); j < issued; ++j) {
          volatile int dummy = 0;
          tc::mbar_wait(bar_full_b + 8 * (j % kStages), (j / kStages) & 1, &dummy);
        }
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      constexpr uint32_t idesc = tc::idesc_bf16_f32(kTileW, kTileT);
      bool ok = true;
      for (int i = 0; i < my_tiles && ok; ++i) {
        const int ab = i & 1;
        ok = tc::mbar_wait(bar_acc_empty + 8 * ab, ((i >> 1) & 1) ^ 1, abort_flag);
        if (!ok) break;
        tc::tc_fence_after();
        const uint32_t dtm = tmem + (uint32_t)(ab * kTileT);
        for (int kb = 0; kb < KB; ++kb) {
          const int j = i * KB + kb;
          const int s = j % kStages;
          const uint32_t ph = (j / kStages) & 1;
          ok = tc::mbar_wait(bar_full_a + 8 * s, ph, abort_flag) && tc::mbar_wait(bar_full_b + 8 * s, ph, abort_flag);
          if (!ok) break;
          tc::tc_fence_after();
          const uint64_t ad = tc::smem_desc_sw128(sA + s * kABytes);
          const uint64_t bd = tc::smem_desc_sw128(sB + s * kBBytes);
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k)
            tc::mma_bf16(dtm, ad + 2 * k, bd + 2 * k, idesc, (kb | k) != 0);
          tc::mma_commit(bar_empty + 8 * s);
        }
        if (ok) tc::mma_commit(bar_acc_full + 8 * ab);
      }
    }
  } else if (warp < 6) {
    // ---------------- dequant producers (one weight row per thread) ----------------
    const int tp = threadIdx.x - 64;          // 0..127
    auto row_of = [&](int j) { return (tile_of(j / KB) % n_tiles) * kTileW + tp; };
    // Four statically rotated buffers: a block's loads are issued three steps before it is
    // decoded, and no register copy ever waits on a load still in flight.
    RawKb b0, b1, b2, b3;
    auto load = [&](RawKb &r, int j) { load_kb<LUT>(r, p, row_of(j), j % KB); };
    auto step = [&](const RawKb &r, int j) -> bool {
      const int s = j % kStages;
      const uint32_t ph = (j / kStages) & 1;
      if (!tc::mbar_wait(bar_empty + 8 * s, ph ^ 1, abort_flag, 200)) return false;
      uint8_t *a_tile = smem + SmemLayout::a + s * kABytes;
      const uint32_t words[8] = {r.q0.x, r.q0.y, r.q0.z, r.q0.w, r.q1.x, r.q1.y, r.q1.z, r.q1.w};
#pragma unroll
      for (int c = 0; c < 8; ++c)
        *reinterpret_cast<uint4 *>(a_tile + tc::sw128_offset((uint32_t)tp, (uint32_t)c)) =
            decode_chunk<LUT>(words[c], c, r, book);
      tc::fence_proxy_async_smem();
      tc::mbar_arrive(bar_full_a + 8 * s);
      return true;
    };
    if (steps > 0) load(b0, 0);
    if (steps > 1) load(b1, 1);
    if (steps > 2) load(b2, 2);
    for (int j = 0; j < steps; j += 4) {
      if (j + 3 < steps) load(b3, j + 3);
      if (!step(b0, j)) break;
      if (j + 1 >= steps) break;
      if (j + 4 < steps) load(b0, j + 4);
      if (!step(b1, j + 1)) break;
      if (j + 2 >= steps) break;
      if (j + 5 < steps) load(b1, j + 5);
      if (!step(b2, j + 2)) break;
      if (j + 3 >= steps) break;
      if (j + 6 < steps) load(b2, j + 6);
      if (!step(b3, j + 3)) break;
    }
  } else {
    // ---------------- epilogue: TMEM -> bf16 y ----------------
    const int quarter = warp & 3;
    for (int i = 0; i < my_tiles; ++i) {
      const int ab = i & 1;
      if (!tc::mbar_wait(bar_acc_full + 8 * ab, (i >> 1) & 1, abort_flag)) break;
      tc::tc_fence_after();
      const int t = tile_of(i);
      const int m0 = (t / n_tiles) * kTileT;
      const int n = (t % n_tiles) * kTileW + quarter * 32 + lane;
      for (int c0 = 0; c0 < kTileT; c0 += 32) {
        if (m0 + c0 >= p.M) break;
        uint32_t v[32];
        tc::tmem_ld_32x32b_x32(tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(ab * kTileT + c0), v);
        tc::tmem_ld_wait();
        if (n < p.N) {
#pragma unroll
          for (int jj = 0; jj < 32; ++jj) {
            const int m = m0 + c0 + jj;
            if (m < p.M) {
              __nv_bfloat16 h = __float2bfloat16_rn(__uint_as_float(v[jj]));
              p.y[(size_t)m * p.N + n] = *reinterpret_cast<uint16_t *>(&h);
            }
          }
        }
      }
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(bar_acc_empty + 8 * ab);
    }
  }

  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------------------------------
// TMA-fed variant (K % 256 == 0; LUT4 block 64 or 128): the producers issue no global loads.
// Per K block the TMA warp brings the x tile (32 KB, swizzled) and the raw code tile
// [128 rows x 32 B] (4 KB); every 8 K blocks it brings the scale (and bias) tile
// [128 rows x 32 B] into a two-slot ring.  Producers read codes and scales from shared
// memory, so the L1 data pipe only sees their 16-byte swizzled stores.
// ---------------------------------------------------------------------------------------
constexpr uint32_t kRawBytes = kTileW * 32;          // 4 KB of codes per K block
constexpr uint32_t kScBytes = kTileW * 32;           // 4 KB of scales (or biases) per 8 K blocks
constexpr int kScKb = 8;                             // K blocks per scale tile

// TT: tokens per tile, 384, 256 or 128.  128-token tiles double the tile count for small M,
// at the price of dequantising each weight tile for half as many tokens.  384-token tiles
// dequantise each weight tile for 1.5 times as many tokens as 256-token ones, which moves
// the bound from the dequantising producers to the tensor core for large M: two MMAs per
// k step (N = 256 at accumulator column 0, N = 128 at column 256), one 384-column
// accumulator (TMEM holds 512 columns, so no second buffer: the epilogue of a tile is not
// overlapped with the next tile's MMAs), three stages (the x stage is 48 KB), x loaded as
// three 128-row boxes per stage.
template <int TT>
struct TileCfg {
  static constexpr int kStages = TT == 384 ? 3 : 4;
  static constexpr int kAccBufs = TT == 384 ? 1 : 2;             // TMEM accumulator buffers
  static constexpr uint32_t kTmemCols = TT == 384 ? 512u : 2u * TT;
  static constexpr int kXBox = TT == 384 ? 128 : TT;            // rows per x TMA box
};

template <int TT>
struct SmemLayoutT {
  static constexpr int kS = TileCfg<TT>::kStages;
  static constexpr uint32_t kB = TT * kBK * 2;                   // x stage bytes
  static constexpr uint32_t a = 0;
  static constexpr uint32_t b = a + kS * kABytes;
  static constexpr uint32_t raw = b + kS * kB;
  static constexpr uint32_t sc = raw + kS * kRawBytes;           // [2] scales
  static constexpr uint32_t bi = sc + 2 * kScBytes;              // [2] biases
  // full_a, full_b, full_w, empty, acc_full[2], acc_empty[2], sc_full[2], sc_empty[2]
  static constexpr uint32_t bars = bi + 2 * kScBytes;
  static constexpr uint32_t misc = bars + (4 * kS + 8) * 8;
  static constexpr uint32_t book = misc + 16;
  static constexpr uint32_t total = book + 16 * 4;
};
template <int TT>
constexpr size_t smem_bytes_t() { return SmemLayoutT<TT>::total + 1024; }
// warp 0 TMA, warp 1 MMA, warps 2-9 producers (two threads per weight row), warps 10-13
// epilogue (warp w reads TMEM lanes 32 (w % 4) .. + 31)
constexpr int kProducersT = 2 * kTileW;
constexpr int kThreadsT = 64 + kProducersT + 128;

struct TmaMaps {
  CUtensorMap x, w, s, b;
};

template <bool LUT, int TT, bool SPLIT>
__global__ void __launch_bounds__(kThreadsT, 1)
    qgemm_tma_kernel(const __grid_constant__ TmaMaps maps, const __grid_constant__ TcGemmParams p) {
  using L = SmemLayoutT<TT>;
  using C = TileCfg<TT>;
  constexpr int kStages = C::kStages;
  constexpr int kAB = C::kAccBufs;
  constexpr uint32_t kBBytesT = L::kB;
  constexpr uint32_t kTmemColsT = C::kTmemCols;
  static_assert(!(SPLIT && TT == 384), "384-token tiles run unsplit");
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = smem_u32(smem_raw);
  const uint32_t base = (raw_base + 1023u) & ~1023u;
  uint8_t *smem = smem_raw + (base - raw_base);

  const uint32_t sA = base + L::a;
  const uint32_t sB = base + L::b;
  const uint32_t sR = base + L::raw;
  const uint32_t sS = base + L::sc;
  const uint32_t sBi = base + L::bi;
  const uint32_t bar_full_a = base + L::bars;
  const uint32_t bar_full_b = bar_full_a + kStages * 8;
  const uint32_t bar_full_w = bar_full_b + kStages * 8;
  const uint32_t bar_empty = bar_full_w + kStages * 8;
  const uint32_t bar_acc_full = bar_empty + kStages * 8;   // [2]
  const uint32_t bar_acc_empty = bar_acc_full + 2 * 8;     // [2]
  const uint32_t bar_sc_full = bar_acc_empty + 2 * 8;      // [2]
  const uint32_t bar_sc_empty = bar_sc_full + 2 * 8;       // [2]
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::misc);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::misc + 4);
  float *book = reinterpret_cast<float *>(smem + L::book);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  // Split mode (ksplit = S > 1): CTA b of the grid owns tile b / S and K blocks
  // [kb_base, kb_base + KB) of it, kb_base = rank * KB; K-block coordinates add kb_base.
  const int S = SPLIT ? p.ksplit : 1;
  const int KB = p.K / kBK / S;
  const int kb_base = SPLIT ? (int)cluster_ctarank() * KB : 0;
  const int SCB = (KB + kScKb - 1) / kScKb;      // scale tiles per weight tile (or split)
  // Tile t is (token tile t / n_tiles, weight-row tile t % n_tiles): the CTAs running at one
  // time share a few x tiles and walk the weight tiles, which all stay in L2, so x (which
  // can be larger than L2 at large M and K) is read from DRAM about once.
  const int m_tiles = (p.M + TT - 1) / TT;
  const int n_tiles = (p.N + kTileW - 1) / kTileW;
  const int T = m_tiles * n_tiles;
  const int my_tiles = SPLIT ? 1 : ((int)blockIdx.x < T ? (T - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0);
  const int steps = my_tiles * KB;
  auto tile_of = [&](int i) { return SPLIT ? (int)blockIdx.x / S : (int)blockIdx.x + i * (int)gridDim.x; };
  const uint32_t sc_tx = LUT ? (uint32_t)(kTileW * p.lut_sc_box * 4) : 2u * kScBytes;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      tc::mbar_init(bar_full_a + 8 * s, kProducersT);
      tc::mbar_init(bar_full_b + 8 * s, 1);
      tc::mbar_init(bar_full_w + 8 * s, 1);
      tc::mbar_init(bar_empty + 8 * s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(bar_acc_full + 8 * b, 1);
      tc::mbar_init(bar_acc_empty + 8 * b, 4);
      tc::mbar_init(bar_sc_full + 8 * b, 1);
      tc::mbar_init(bar_sc_empty + 8 * b, kProducersT);
    }
    *abort_flag = 0;
    tc::fence_mbar_init();
    tc::tma_prefetch_desc(&maps.x);
    tc::tma_prefetch_desc(&maps.w);
    tc::tma_prefetch_desc(&maps.s);
    if (!LUT) tc::tma_prefetch_desc(&maps.b);
  }
  if (LUT && threadIdx.x < 16) book[threadIdx.x] = p.book[threadIdx.x];
  if (warp == 1) {
    tc::tmem_alloc(smem_u32(tmem_slot), kTmemColsT);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ---------------- TMA: x tiles, code tiles, scale tiles ----------------
    if (lane == 0) {
      int issued = 0, sc_issued = 0;
      bool ok = true;
      for (int j = 0; j < steps && ok; ++j) {
        const int i = j / KB, kb = j - i * KB;
        const int t = tile_of(i);
        const int m0 = (t / n_tiles) * TT;
        const int n0 = (t % n_tiles) * kTileW;
        if (kb % kScKb == 0) {
          const int q = i * SCB + kb / kScKb;              // scale tile counter
          const int slot = q & 1;
          if (!tc::mbar_wait(bar_sc_empty + 8 * slot, ((q >> 1) & 1) ^ 1, abort_flag)) { ok = false; break; }
          tc::mbar_arrive_expect_tx(bar_sc_full + 8 * slot, sc_tx);
          if (LUT) {
            tc::tma_load_2d(sS + slot * kScBytes, &maps.s, ((kb_base + kb) / kScKb) * p.lut_sc_box, n0,
                            bar_sc_full + 8 * slot);
          } else {
            tc::tma_load_2d(sS + slot * kScBytes, &maps.s, ((kb_base + kb) / kScKb) * 16, n0, bar_sc_full + 8 * slot);
            tc::tma_load_2d(sBi + slot * kScBytes, &maps.b, ((kb_base + kb) / kScKb) * 16, n0, bar_sc_full + 8 * slot);
          }
          ++sc_issued;
        }
        const int s = j % kStages;
        const uint32_t ph = (j / kStages) & 1;
        if (!tc::mbar_wait(bar_empty + 8 * s, ph ^ 1, abort_flag)) break;
        tc::mbar_arrive_expect_tx(bar_full_w + 8 * s, kRawBytes);
        tc::tma_load_2d(sR + s * kRawBytes, &maps.w, (kb_base + kb) * 32, n0, bar_full_w + 8 * s);
        tc::mbar_arrive_expect_tx(bar_full_b + 8 * s, kBBytesT);
#pragma unroll
        for (int xb = 0; xb < TT / C::kXBox; ++xb)
          tc::tma_load_2d(sB + s * kBBytesT + xb * C::kXBox * 128, &maps.x, (kb_base + kb) * kBK, m0 + xb * C::kXBox,
                          bar_full_b + 8 * s);
        ++issued;
      }
      if (*abort_flag) {
        // drain our own copies still in flight before the CTA can exit
        for (int j = (issued > kStages ? issued - kStages : 0); j < issued; ++j) {
          volatile int dummy = 0;
          tc::mbar_wait(bar_full_b + 8 * (j % kStages), (j / kStages) & 1, &dummy);
          tc::mbar_wait(bar_full_w + 8 * (j % kStages), (j / kStages) & 1, &dummy);
        }
        for (int q = (sc_issued > 2 ? sc_issued - 2 : 0); q < sc_issued; ++q) {
          volatile int dummy = 0;
          tc::mbar_wait(bar_sc_full + 8 * (q & 1), (q >> 1) & 1, &dummy);
        }
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      constexpr int kN0 = TT > 256 ? 256 : TT;                 // first MMA's N; a second covers the rest
      constexpr uint32_t idesc = tc::idesc_bf16_f32(kTileW, kN0);
      constexpr uint32_t idesc2 = tc::idesc_bf16_f32(kTileW, TT > 256 ? TT - 256 : 16);
      bool ok = true;
      for (int i = 0; i < my_tiles && ok; ++i) {
        const int ab = i % kAB;
        ok = tc::mbar_wait(bar_acc_empty + 8 * ab, ((i / kAB) & 1) ^ 1, abort_flag);
        if (!ok) break;
        tc::tc_fence_after();
        const uint32_t dtm = tmem + (uint32_t)(ab * TT);
        for (int kb = 0; kb < KB; ++kb) {
          const int j = i * KB + kb;
          const int s = j % kStages;
          const uint32_t ph = (j / kStages) & 1;
          ok = tc::mbar_wait(bar_full_a + 8 * s, ph, abort_flag, 100) &&
               tc::mbar_wait(bar_full_b + 8 * s, ph, abort_flag, 100);
          if (!ok) break;
          tc::tc_fence_after();
          const uint64_t ad = tc::smem_desc_sw128(sA + s * kABytes);
          const uint64_t bd = tc::smem_desc_sw128(sB + s * kBBytesT);
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k) {
            tc::mma_bf16(dtm, ad + 2 * k, bd + 2 * k, idesc, (kb | k) != 0);
            if constexpr (TT > 256) {   // tokens 256..TT-1: B rows 256.. (32 KB on), accumulator column 256
              const uint64_t bd2 = tc::smem_desc_sw128(sB + s * kBBytesT + 256 * 128);
              tc::mma_bf16(dtm + 256u, ad + 2 * k, bd2 + 2 * k, idesc2, (kb | k) != 0);
            }
          }
          tc::mma_commit(bar_empty + 8 * s);
        }
        if (ok) tc::mma_commit(bar_acc_full + 8 * ab);
      }
    }
  } else if (warp < 2 + kProducersT / 32) {
    // ---------------- dequant producers: half a weight row (32 k) per thread ----------------
    const int tp = threadIdx.x - 64;
    const int row = tp & (kTileW - 1), half = tp / kTileW;
    const uint8_t *raw_row = smem + L::raw + row * 32 + half * 16;
    // The scale tile lands as a dense [rows][box] array: 32 bytes a row for INT4 and LUT4
    // block 64 (eight scales per eight K blocks), 16 for LUT4 block 128 (four).
    const uint8_t *sc_row = smem + L::sc + row * (LUT ? 4 * p.lut_sc_box : 32);
    const uint8_t *bi_row = smem + L::bi + row * 32;
    // Step j = i * KB + kb walks (tile i, K block kb); scale tile q = i * SCB + kb / kScKb.
    // Counters advance incrementally (no divisions per stage).
    int kb = 0, kk = 0, q = 0, s = 0;
    uint32_t ph = 0;
    for (int j = 0; j < steps; ++j) {
      const int slot = q & 1;
      if (kk == 0 && !tc::mbar_wait(bar_sc_full + 8 * slot, (q >> 1) & 1, abort_flag, 100)) break;
      if (!tc::mbar_wait(bar_full_w + 8 * s, ph, abort_flag, 100)) break;
      RawKb r;
      r.q0 = *reinterpret_cast<const uint4 *>(raw_row + s * kRawBytes);
      r.q1 = r.q0;
      if constexpr (LUT) {
        r.s = *reinterpret_cast<const uint32_t *>(sc_row + slot * kScBytes + 4 * (kk >> (p.lut_kb_per_block - 1)));
        r.b = 0;
      } else {
        r.s = *reinterpret_cast<const uint32_t *>(sc_row + slot * kScBytes + 4 * kk);
        r.b = *reinterpret_cast<const uint32_t *>(bi_row + slot * kScBytes + 4 * kk);
      }
      uint8_t *a_tile = smem + L::a + s * kABytes;
      const uint32_t words[4] = {r.q0.x, r.q0.y, r.q0.z, r.q0.w};
      if (half == 0) {
#pragma unroll
        for (int c = 0; c < 4; ++c)
          *reinterpret_cast<uint4 *>(a_tile + tc::sw128_offset((uint32_t)row, (uint32_t)c)) =
              decode_chunk<LUT>(words[c], c, r, book);
      } else {
#pragma unroll
        for (int c = 4; c < 8; ++c)
          *reinterpret_cast<uint4 *>(a_tile + tc::sw128_offset((uint32_t)row, (uint32_t)c)) =
              decode_chunk<LUT>(words[c - 4], c, r, book);
      }
      tc::fence_proxy_async_smem();
      tc::mbar_arrive(bar_full_a + 8 * s);
      if (kk == kScKb - 1 || kb == KB - 1) tc::mbar_arrive(bar_sc_empty + 8 * slot);
      if (++s == kStages) { s = 0; ph ^= 1u; }
      if (++kb == KB) {          // next tile: its scale tiles start a new group
        kb = 0; kk = 0; ++q;
      } else if (++kk == kScKb) {
        kk = 0; ++q;
      }
    }
  } else {
    // ---------------- epilogue: TMEM -> bf16 y (split mode: fp32 partial tile) ----------------
    const int quarter = warp & 3;
    float *part = reinterpret_cast<float *>(smem + L::a);   // split mode: [TT tokens][128 rows]
    for (int i = 0; i < my_tiles; ++i) {
      const int ab = i % kAB;
      if (!tc::mbar_wait(bar_acc_full + 8 * ab, (i / kAB) & 1, abort_flag)) break;
      tc::tc_fence_after();
      const int t = tile_of(i);
      const int m0 = (t / n_tiles) * TT;
      const int n = (t % n_tiles) * kTileW + quarter * 32 + lane;
      for (int c0 = 0; c0 < TT; c0 += 32) {
        if (m0 + c0 >= p.M) break;
        uint32_t v[32];
        tc::tmem_ld_32x32b_x32(tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(ab * TT + c0), v);
        tc::tmem_ld_wait();
        if constexpr (SPLIT) {   // all MMAs of the (single) tile are done: the stage buffers are free
#pragma unroll
          for (int jj = 0; jj < 32; ++jj) part[(c0 + jj) * kTileW + quarter * 32 + lane] = __uint_as_float(v[jj]);
        } else if (n < p.N) {
#pragma unroll
          for (int jj = 0; jj < 32; ++jj) {
            const int m = m0 + c0 + jj;
            if (m < p.M) {
              __nv_bfloat16 h = __float2bfloat16_rn(__uint_as_float(v[jj]));
              p.y[(size_t)m * p.N + n] = *reinterpret_cast<uint16_t *>(&h);
            }
          }
        }
      }
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(bar_acc_empty + 8 * ab);
    }
  }

  if constexpr (SPLIT) {
    // Sum the S partial tiles of the cluster in rank order; rank r finishes tokens
    // [r TT / S, (r + 1) TT / S) of the tile.  Every thread of every CTA passes both
    // cluster barriers, also after an aborted main loop.
    __syncwarp();
    cluster_sync_all();
    const uint32_t rank = cluster_ctarank();
    const int t = tile_of(0);
    const int m0 = (t / n_tiles) * TT, n0 = (t % n_tiles) * kTileW;
    const int tok_per = TT / S;
    const uint32_t part_s = smem_u32(smem + L::a);
    for (int it = threadIdx.x; it < tok_per * (kTileW / 4); it += kThreadsT) {
      const int tl = (int)rank * tok_per + it / (kTileW / 4);
      const int r4 = (it % (kTileW / 4)) * 4;
      const uint32_t off = (uint32_t)((tl * kTileW + r4) * 4);
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int r = 0; r < S; ++r) {
        const float4 v = ld_shared_cluster_v4(map_shared_rank(part_s + off, (uint32_t)r));
        acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
      }
      const int m = m0 + tl, n = n0 + r4;
      if (m < p.M) {
        uint16_t *dst = p.y + (size_t)m * p.N + n;
        const float vals[4] = {acc.x, acc.y, acc.z, acc.w};
        if (n + 3 < p.N && (p.N & 3) == 0) {
          *reinterpret_cast<uint2 *>(dst) = make_uint2(pack_bf16x2(vals[0], vals[1]), pack_bf16x2(vals[2], vals[3]));
        } else {
#pragma unroll
          for (int j = 0; j < 4; ++j)
            if (n + j < p.N) {
              __nv_bfloat16 h = __float2bfloat16_rn(vals[j]);
              dst[j] = *reinterpret_cast<uint16_t *>(&h);
            }
        }
      }
    }
    cluster_sync_all();   // every rank has read every partial before any CTA exits
  }

  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, kTmemColsT);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
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

// x [rows, K] bf16 row-major, box [box_rows x 64], 128-byte swizzle, zero fill out of bounds.
cudaError_t make_x_map(CUtensorMap *map, const void *x, int rows, int K, int box_rows) {
  auto enc = get_encode_fn();
  if (!enc) return cudaErrorNotSupported;
  cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)K * 2};
  cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(x), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Generic 2D tensor map, no swizzle, zero fill out of bounds.
cudaError_t make_plain_map(CUtensorMap *map, const void *base, CUtensorMapDataType dt, int esize,
                           long long inner, long long rows, int box_inner, int box_rows) {
  auto enc = get_encode_fn();
  if (!enc) return cudaErrorNotSupported;
  cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)inner * (cuuint64_t)esize};
  cuuint32_t box[2] = {(cuuint32_t)box_inner, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, dt, 2, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

int sm_count() {
  int sms = 148, dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return sms;
}

unsigned persistent_grid(const TcGemmParams &p, int tt = kTileT) {
  const int sms = sm_count();
  const long long tiles = (long long)((p.N + kTileW - 1) / kTileW) * ((p.M + tt - 1) / tt);
  return (unsigned)(tiles < sms ? tiles : sms);
}

// Tile plan: tokens per tile (TT: 384, 256 or 128) and K split (S).  A tile's time is set by its K blocks,
// the dequantising producers being the bound: a 128-token tile costs about 7/8 of a
// 256-token one per K block (measured on GB300).  S = 1 runs persistent CTAs over all
// tiles; S > 1 runs one (tile, K slice) per CTA, S CTAs per cluster, plus the reduction of
// the partial tiles (about 10 K blocks' time).  Cost = rounds of CTAs x time per CTA; a
// split is taken only when it is clearly (10 %) cheaper than the best unsplit plan.
struct TilePlan {
  int tt, S;
};
constexpr double kCost384 = 1.33;
TilePlan pick_tile_plan(const TcGemmParams &p) {
  const int sms = sm_count();
  const int KB = p.K / kBK;
  TilePlan best{256, 1};
  double best1 = 1e30, bestS = 1e30;
  TilePlan planS{256, 1};
  for (int tt : {384, 256, 128}) {
    // Time per tile relative to a 256-token tile, measured on GB300: 128-token tiles 7/8;
    // 384-token tiles 1.28-1.36 (1.5x the tokens: the tensor core, not the dequantising
    // producers, now bounds a K block, and the single accumulator exposes the epilogue).
    const double f = tt == 256 ? 1.0 : tt == 128 ? 0.875 : kCost384;
    const long long T = (long long)((p.N + kTileW - 1) / kTileW) * ((p.M + tt - 1) / tt);
    for (int S : {1, 2, 4, 8}) {
      if (S > 1 && (tt == 384 || KB % (8 * S) != 0)) continue;
      const long long ctas = T * S;
      const long long rounds = (ctas + sms - 1) / sms;
      const double cost = (double)rounds * ((double)KB / S * f + (S > 1 ? 10.0 : 0.0));
      if (S == 1 && cost < best1) { best1 = cost; best = TilePlan{tt, 1}; }
      if (S > 1 && cost < bestS) { bestS = cost; planS = TilePlan{tt, S}; }
    }
  }
  TilePlan chosen = bestS < 0.9 * best1 ? planS : best;
#ifdef Q4MM_TUNING
  // Tuning builds only: environment overrides of the tile plan, for plan sweeps.
  if (const char *v = getenv("Q4MM_GEMM_TT")) chosen.tt = atoi(v);
  if (const char *v = getenv("Q4MM_GEMM_S")) chosen.S = atoi(v);
#endif
  return chosen;
}

template <bool LUT, int TT>
cudaError_t set_tma_smem(int S) {
  if constexpr (TT == 384) {   // 384-token tiles run unsplit
    (void)S;
    return cudaFuncSetAttribute(qgemm_tma_kernel<LUT, TT, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)smem_bytes_t<TT>());
  } else {
    if (S <= 1)
      return cudaFuncSetAttribute(qgemm_tma_kernel<LUT, TT, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)smem_bytes_t<TT>());
    return cudaFuncSetAttribute(qgemm_tma_kernel<LUT, TT, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)smem_bytes_t<TT>());
  }
}

template <bool LUT, int TT>
cudaError_t launch_tma_typed(const TmaMaps &maps, const TcGemmParams &q, int S, cudaStream_t s) {
  if (TT == 384 || S <= 1) {
    auto kern = qgemm_tma_kernel<LUT, TT, false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_bytes_t<TT>());
    if (e != cudaSuccess) return e;
    TcGemmParams q1 = q;
    q1.ksplit = 1;
    kern<<<persistent_grid(q1, TT), kThreadsT, smem_bytes_t<TT>(), s>>>(maps, q1);
    return cudaGetLastError();
  }
  if constexpr (TT == 384) {
    return cudaErrorInvalidValue;   // not reached: 384-token tiles run unsplit
  } else {
  auto kern = qgemm_tma_kernel<LUT, TT, true>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_bytes_t<TT>());
  if (e != cudaSuccess) return e;
  TcGemmParams qs = q;
  qs.ksplit = S;
  const long long tiles = (long long)((q.N + kTileW - 1) / kTileW) * ((q.M + TT - 1) / TT);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(tiles * S), 1, 1);
  cfg.blockDim = dim3(kThreadsT, 1, 1);
  cfg.dynamicSmemBytes = smem_bytes_t<TT>();
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)S;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, maps, qs);
  }
}

template <bool LUT>
cudaError_t launch_tc(const TcGemmParams &p, const void *x, cudaStream_t s) {
  // LUT4 scales go through a tensor map too: its base must be 16-byte aligned and its row
  // pitch (K / block scales of 4 bytes) a multiple of 16 bytes; otherwise the producers load
  // them directly (the non-TMA kernel).
  const bool lut_tma = p.lut_blocks_per_row % 4 == 0 && (reinterpret_cast<uintptr_t>(p.scales) & 15u) == 0 &&
                       (p.lut_kb_per_block == 1 || p.lut_kb_per_block == 2);
  const bool tma_path = p.K % 256 == 0 && (!LUT || lut_tma);
  // The kernel's attribute set-up comes first: it makes the device's primary context
  // current on this host thread, which the tensor-map encoding (a driver call) needs when
  // this is the thread's first CUDA work.
  if (tma_path) {
    const TilePlan tp = pick_tile_plan(p);
    const int tt = tp.tt;
    cudaError_t ea = tt == 128 ? set_tma_smem<LUT, 128>(tp.S)
                   : tt == 384 ? set_tma_smem<LUT, 384>(tp.S) : set_tma_smem<LUT, 256>(tp.S);
    if (ea != cudaSuccess) return ea;
    TmaMaps maps;
    cudaError_t e = make_x_map(&maps.x, x, p.M, p.K, tt == 384 ? 128 : tt);
    if (e == cudaSuccess)
      e = make_plain_map(&maps.w, p.w, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, p.K / 2, p.N, 32, kTileW);
    if (LUT) {
      TcGemmParams q = p;
      q.lut_sc_box = 8 / q.lut_kb_per_block;
      if (e == cudaSuccess)
        e = make_plain_map(&maps.s, p.scales, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, p.lut_blocks_per_row, p.N,
                           q.lut_sc_box, kTileW);
      maps.b = maps.s;
      if (e != cudaSuccess) return e;
      return tt == 128 ? launch_tma_typed<true, 128>(maps, q, tp.S, s)
           : tt == 384 ? launch_tma_typed<true, 384>(maps, q, tp.S, s) : launch_tma_typed<true, 256>(maps, q, tp.S, s);
    }
    if (e == cudaSuccess)
      e = make_plain_map(&maps.s, p.scales, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.K / 32, p.N, 16, kTileW);
    if (e == cudaSuccess)
      e = make_plain_map(&maps.b, p.biases, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.K / 32, p.N, 16, kTileW);
    if (e != cudaSuccess) return e;
    return tt == 128 ? launch_tma_typed<false, 128>(maps, p, tp.S, s)
         : tt == 384 ? launch_tma_typed<false, 384>(maps, p, tp.S, s) : launch_tma_typed<false, 256>(maps, p, tp.S, s);
  }
  auto kern = qgemm_tc_kernel<LUT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
  if (e != cudaSuccess) return e;
  CUtensorMap map;
  e = make_x_map(&map, x, p.M, p.K, kTileT);
  if (e != cudaSuccess) return e;
  kern<<<persistent_grid(p), kThreads, kSmemBytes, s>>>(map, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_q4_gemm(const uint16_t *x, const uint32_t *w, const uint16_t *scales,
                           const uint16_t *biases, uint16_t *y, int M, int N, int K,
                           cudaStream_t s) {
  TcGemmParams p{};
  p.w = reinterpret_cast<const uint8_t *>(w);
  p.scales = scales;
  p.biases = biases;
  p.y = y;
  p.M = M; p.N = N; p.K = K;
  return launch_tc<false>(p, x, s);
}

cudaError_t launch_lut4_gemm(const uint16_t *x, const uint8_t *packed, const float *scales,
                             const float *book, uint16_t *y, int M, int N, int K, int block,
                             cudaStream_t s) {
  if (K % kBK != 0 || block % kBK != 0 || K % block != 0) return cudaErrorNotSupported;
  TcGemmParams p{};
  p.w = packed;
  p.scales = scales;
  p.biases = nullptr;
  p.y = y;
  p.M = M; p.N = N; p.K = K;
  p.lut_blocks_per_row = K / block;
  p.lut_kb_per_block = block / kBK;
  for (int i = 0; i < 16; ++i) p.book[i] = book[i];
  return launch_tc<true>(p, x, s);
}

}  // namespace q4mm
