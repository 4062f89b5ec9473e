// moe_tc.cu -- GGML Q4_0 and Q8_0 expert-routed matmul, mat-mat form, on the tensor cores.
//
// quantized_matmul_id_ggml.rs (mlx-native 0.9.0): `dispatch_id_mm_for_test` regroups the
// routed rows per expert (map0) so that a matmul tile reads a single expert's weights and
// reuses them across that expert's routed rows instead of re-reading them per row.  Here:
//
//  1. routing (moe.cu): per-expert counts, ascending row lists, and a list of token blocks
//     of <= kMoeTokBlock (112) rows, each inside one expert;
//  2. gather: xs[p] = fp16(2^e_t * x[t]), t = hids[p] / top_k -- the rows of x in routed
//     order, each token scaled by a power of two that brings its largest magnitude into
//     [2^14, 2^15) (found once per token by token_scale_kernel);
//  3. routed_mm_tc_kernel<BT>, persistent over work items (token block, 128-row weight tile):
//       A = the expert's weight rows, decoded to fp16 by eight producer warps from TMA boxes of
//           8 blocks per row (256 k): 144 bytes for Q4_0 (18-byte blocks), 272 for Q8_0
//           (34-byte blocks);
//       B = the block's gathered x rows (TMA, 64-row boxes, 128-byte swizzle);
//       D = 128 weight rows x (rows rounded up to 16) fp32 in tensor memory;
//     epilogue warps scatter 2^-e_t * D column j to out[hids[p0 + j]][n0 .. n0+127] (fp32).
//     Each expert's weights stream once from HBM per token block.
//
// Operands are fp16 (fp32 accumulation): the blocks' d is already fp16, so (q - 8) * d (Q4_0)
// or q * d (Q8_0) is formed with one fp16 multiply (a single rounding of the exact product),
// and x is rounded from fp32 to fp16 once in the gather.  The power-of-two row scaling is
// exact in both directions, so any finite f32 row is served: its largest element lands near
// 2^14 (no fp16 overflow, and no fp16 subnormals unless an element is 2^-28 below the row's
// largest), and the rounding to fp16 is relative to the row's own range.  A block whose d
// could take a weight beyond fp16's range (|value| >= 65520: |d| >= 8192 in Q4_0, >= 512 in
// Q8_0) is reported as Q4MM_DEVERR_F16_RANGE.  The mat-vec form rounds x to bf16 instead.
//
// Pipeline: stages of two 64-k tiles each (A and B), three for Q4_0 and two for Q8_0.  The
// producers publish a stage on
// full_a once their A tiles are written and the stage's B tiles (TMA) have landed, so the
// single MMA thread waits on one barrier and commits once per 128 k.  That thread sets the
// pace: each tcgen05.mma costs it 50-100 cycles to issue, more than the tensor core needs
// for a 128 x 64 x 16 product.
#include "tc_common.cuh"

#include <cudaTypedefs.h>

#include <utility>

namespace q4mm {

Q4MM_DEFINE_ERROR_READER(read_errors_moe_tc)

namespace {

constexpr int kTW = 128;            // weight rows per tile (MMA M)
constexpr int kBK = 64;             // K per tile (one 128-byte swizzle atom of fp16)
constexpr int kKps = 2;             // K tiles per pipeline stage (one barrier phase)
constexpr int kThreads = 480;       // warp 0 x TMA, 1 MMA, 2-9 producers, 10-13 epilogue, 14 weight TMA
constexpr int kProducers = 256;     // two threads per weight row, one Q4_0 block each per K block
constexpr uint32_t kTmemCols = 256; // two accumulators of kAccCols columns
constexpr uint32_t kABytes = kTW * kBK * 2;               // 16 KB
constexpr uint32_t kBBytes = kMoeTokBlock * kBK * 2;      // 14 KB (112 token rows)
constexpr uint32_t kBoxTok = kMoeTokBlock / 2;            // x rows per TMA box (56: whole 8-row swizzle atoms)
constexpr uint32_t kAccCols = 128;                        // TMEM columns per accumulator (>= kMoeTokBlock)
static_assert(kBBytes % 1024 == 0 && kBoxTok % 8 == 0 && kMoeTokBlock <= (int)kAccCols, "B tile layout");

// Weight boxes: one row of a box is 8 blocks (256 k = 4 K blocks) of one weight row.
//   Q4_0: 8 x 18 = 144 bytes, copied as 144 uint8 elements; 2 boxes in flight (18 KB each);
//   Q8_0: 8 x 34 = 272 bytes, copied as 136 uint16 elements (a box row holds at most 256
//         elements); 2 boxes in flight (34 KB each).
// Pipeline stages (kKps A and B tiles each): 3 for Q4_0, 2 for Q8_0 (its boxes take the room).
template <int BT>
struct RawCfg {
  static constexpr uint32_t kRow = BT == kQ8_0 ? 272 : 144;
  static constexpr uint32_t kBoxX = BT == kQ8_0 ? 136 : 144;   // box row in TMA elements
  static constexpr int kSlots = 2;
  static constexpr uint32_t kBytes = kTW * kRow;
  static constexpr int kStages = BT == kQ8_0 ? 2 : 3;
};

template <int BT>
struct SmemL {
  static constexpr uint32_t a = 0;
  static constexpr int kTiles = kKps * RawCfg<BT>::kStages;
  static constexpr uint32_t b = a + kTiles * kABytes;
  static constexpr uint32_t raw = b + kTiles * kBBytes;    // [kSlots]
  // full_a, full_b, empty, acc_full[2], acc_empty[2], raw_full[kSlots], raw_empty[kSlots]
  static constexpr uint32_t bars = raw + RawCfg<BT>::kSlots * RawCfg<BT>::kBytes;
  static constexpr uint32_t misc = bars + (3 * RawCfg<BT>::kStages + 4 + 2 * RawCfg<BT>::kSlots) * 8;
  static constexpr uint32_t total = misc + 16;
};
template <int BT>
constexpr size_t mm_smem_bytes() { return SmemL<BT>::total + 1024; }
static_assert(mm_smem_bytes<kQ4_0>() <= 227 * 1024 && mm_smem_bytes<kQ8_0>() <= 227 * 1024, "shared memory");

struct MmParams {
  float *out;
  const int32_t *hids;
  const float *xun;   // per gathered row: the power of two that undoes the gather's scaling
  const int4 *blk;
  const uint32_t *n_blk;
  int N, K;
};

struct MmMaps {
  CUtensorMap w;   // 3D: [E][N][row bytes] uint8
  CUtensorMap xs;  // 2D: [R][K] fp16, 128-byte swizzle
};

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, int c0, int c1, int c2,
                                            uint32_t mbar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(mbar)
      : "memory");
}

// K order inside every 32-element Q4_0 block, shared by the decoded weight tile and the
// gathered x rows: 16-byte chunk m (m = 0..3) holds elements
//   4m, 4m+2, 4m+1, 4m+3, 4m+16, 4m+18, 4m+17, 4m+19,
// which are the pairs that qs word m (bytes 4m..4m+3; low nibbles 4m.., high nibbles
// 4m+16..) yields with one mask each.  A dot product is indifferent to the order of k as
// long as both operands use the same one.
//
// qs word m as one 16-byte chunk of (q - 8) * d in fp16.  (code | 0x6400) is the fp16 value
// 1024 + q; subtracting 1032 gives q - 8 exactly, and the product with d is rounded once.
__device__ __forceinline__ uint4 q4_0_chunk(uint32_t word, uint32_t d2) {
  constexpr uint32_t kMask = 0x000F000Fu, kMagic = 0x64006400u, kOff = 0x64086408u;   // 1024, 1032
  const uint32_t c[4] = {and_or(word, kMask, kMagic), and_or(word >> 8, kMask, kMagic),
                         and_or(word >> 4, kMask, kMagic), and_or(word >> 12, kMask, kMagic)};
  uint32_t r[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t q;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(q) : "r"(c[i]), "r"(kOff));
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r[i]) : "r"(q), "r"(d2));
  }
  return make_uint4(r[0], r[1], r[2], r[3]);
}

// Q8_0 qs words m (elements 4m..4m+3) and m + 4 (elements 4m+16..) as one 16-byte chunk of
// q * d in fp16, in the chunk order above.  (byte ^ 0x80) | 0x6400 is the fp16 value
// 1024 + (q + 128) for the signed byte q; subtracting 1152 gives q exactly, and the product
// with d is rounded once.  The mask keeps bytes 0 and 2 (or 1 and 3 after the shift), the
// pairs (4m, 4m+2) and (4m+1, 4m+3).
__device__ __forceinline__ uint4 q8_0_chunk(uint32_t lo, uint32_t hi, uint32_t d2) {
  constexpr uint32_t kMask = 0x00FF00FFu, kFlip = 0x64806480u;   // 0x80 on each byte, exponent bits of 1024
  const uint32_t c[4] = {(lo & kMask) ^ kFlip, ((lo >> 8) & kMask) ^ kFlip, (hi & kMask) ^ kFlip,
                         ((hi >> 8) & kMask) ^ kFlip};
  uint32_t r[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t q;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(q) : "r"(c[i]), "r"(kFlip));   // 0x6480 is 1152
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r[i]) : "r"(q), "r"(d2));
  }
  return make_uint4(r[0], r[1], r[2], r[3]);
}

// The nine 32-bit words of Q8_0 block 2 kk + H of every K block kk from a 272-byte box row:
// block 2kk + H starts at byte 68 kk + 34 H, so H = 0 takes words 17kk .. 17kk + 8 (d in the
// low half of the first) and H = 1 words 17kk + 8 .. 17kk + 16 (d in the high half of the
// first).  Only the 16-byte pieces that hold them are read.
template <int H>
__device__ __forceinline__ void q8_0_box_words(const uint4 *row, uint32_t (&u)[4][9]) {
#pragma unroll
  for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
    for (int i = 0; i < 9; ++i) {
      const int w = 17 * kk + 8 * H + i;
      const uint4 c = row[w >> 2];
      const int j = w & 3;
      u[kk][i] = j == 0 ? c.x : j == 1 ? c.y : j == 2 ? c.z : c.w;
    }
  }
}

template <int BT>
__global__ void __launch_bounds__(kThreads, 1)
    routed_mm_tc_kernel(const __grid_constant__ MmMaps maps, const __grid_constant__ MmParams p) {
  using L = SmemL<BT>;
  constexpr int kStages = RawCfg<BT>::kStages;
  constexpr int kRawSlots = RawCfg<BT>::kSlots;
  constexpr uint32_t kRawBytes = RawCfg<BT>::kBytes;
  constexpr uint32_t kRawRow = RawCfg<BT>::kRow;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = smem_u32(smem_raw);
  const uint32_t base = (raw_base + 1023u) & ~1023u;
  uint8_t *smem = smem_raw + (base - raw_base);
  const uint32_t sA = base + L::a, sB = base + L::b, sR = base + L::raw;
  const uint32_t bar_full_a = base + L::bars;
  const uint32_t bar_full_b = bar_full_a + kStages * 8;
  const uint32_t bar_empty = bar_full_b + kStages * 8;
  const uint32_t bar_acc_full = bar_empty + kStages * 8;
  const uint32_t bar_acc_empty = bar_acc_full + 16;
  const uint32_t bar_raw_full = bar_acc_empty + 16;
  const uint32_t bar_raw_empty = bar_raw_full + 8 * kRawSlots;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::misc);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::misc + 4);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int KB = p.K / kBK;                 // multiple of 4
  const int KJ = KB / kKps;                 // stages per item
  const int n_tiles = (p.N + kTW - 1) / kTW;
  auto item_of = [&](int i) { return (int)blockIdx.x + i * (int)gridDim.x; };

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      tc::mbar_init(bar_full_a + 8 * s, kProducers);
      tc::mbar_init(bar_full_b + 8 * s, 1);
      tc::mbar_init(bar_empty + 8 * s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(bar_acc_full + 8 * b, 1);
      tc::mbar_init(bar_acc_empty + 8 * b, 4);
    }
    for (int b = 0; b < kRawSlots; ++b) {
      tc::mbar_init(bar_raw_full + 8 * b, 1);
      tc::mbar_init(bar_raw_empty + 8 * b, kProducers);
    }
    *abort_flag = 0;
    tc::fence_mbar_init();
    tc::tma_prefetch_desc(&maps.w);
    tc::tma_prefetch_desc(&maps.xs);
  }
  if (warp == 1) {
    tc::tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // Launched as a programmatic dependent of the gather: everything above overlapped its
  // tail; the routing lists and gathered rows are read only after it has completed.
  griddep_wait();
  const int items = (int)*p.n_blk * n_tiles;
  const int my_items = (int)blockIdx.x < items ? (items - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
  const int steps = my_items * KJ;          // stages of this CTA

  if (warp == 14) {
    // ---------------- weight TMA: one 128-row box per 4 K blocks ----------------
    // Runs ahead of the MMA by up to kRawSlots boxes, independently of the x stages.
    if (lane == 0) {
      int raw_issued = 0;
      const int boxes_per_item = KB / 4;
      // The item's expert and row tile are read once per item, and the next item's block
      // entry is loaded one item ahead, so no global load sits between two box issues.
      int i = 0, bq = 0;
      int4 cur = my_items > 0 ? p.blk[item_of(0) / n_tiles] : make_int4(0, 0, 0, 0);
      int4 nxt = my_items > 1 ? p.blk[item_of(1) / n_tiles] : cur;
      for (int q = 0; q < my_items * boxes_per_item; ++q) {
        if (bq == boxes_per_item) {
          bq = 0;
          ++i;
          cur = nxt;
          if (i + 1 < my_items) nxt = p.blk[item_of(i + 1) / n_tiles];
        }
        const int w = item_of(i);
        const int e = cur.x;
        const int n0 = (w % n_tiles) * kTW;
        const int slot = q % kRawSlots;
        if (!tc::mbar_wait(bar_raw_empty + 8 * slot, ((q / kRawSlots) & 1) ^ 1, abort_flag)) break;
        tc::mbar_arrive_expect_tx(bar_raw_full + 8 * slot, kRawBytes);
        tma_load_3d(sR + slot * kRawBytes, &maps.w, bq * (int)RawCfg<BT>::kBoxX, n0, e,
                    bar_raw_full + 8 * slot);
        ++raw_issued;
        ++bq;
      }
      if (*abort_flag) {
        for (int q = (raw_issued > kRawSlots ? raw_issued - kRawSlots : 0); q < raw_issued; ++q) {
          volatile int dummy = 0;
          tc::mbar_wait(bar_raw_full + 8 * (q % kRawSlots), (q / kRawSlots) & 1, &dummy);
        }
      }
    }
  } else if (warp == 0) {
    // ---------------- x TMA: the block's gathered rows, every K block ----------------
    if (lane == 0) {
      int issued = 0;
      int i = 0, jb = 0;
      int4 bi = my_items > 0 ? p.blk[item_of(0) / n_tiles] : make_int4(0, 0, 0, 0);
      int4 bnext = my_items > 1 ? p.blk[item_of(1) / n_tiles] : bi;   // one item ahead
      for (int j = 0; j < steps; ++j, ++jb) {
        if (jb == KJ) {
          jb = 0;
          ++i;
          bi = bnext;
          if (i + 1 < my_items) bnext = p.blk[item_of(i + 1) / n_tiles];
        }
        const int s = j % kStages;
        const uint32_t ph = (j / kStages) & 1;
        if (!tc::mbar_wait(bar_empty + 8 * s, ph ^ 1, abort_flag)) break;
        const int boxes = (bi.z + (int)kBoxTok - 1) / (int)kBoxTok;
        tc::mbar_arrive_expect_tx(bar_full_b + 8 * s, (uint32_t)(kKps * boxes) * kBoxTok * kBK * 2);
        for (int h = 0; h < kKps; ++h)
          for (int bx = 0; bx < boxes; ++bx)
            tc::tma_load_2d(sB + (s * kKps + h) * kBBytes + bx * kBoxTok * kBK * 2, &maps.xs, (jb * kKps + h) * kBK,
                            bi.y + bx * (int)kBoxTok, bar_full_b + 8 * s);
        ++issued;
      }
      if (*abort_flag) {
        for (int j = (issued > kStages ? issued - kStages : 0); j < issued; ++j) {
          volatile int dummy = 0;
          tc::mbar_wait(bar_full_b + 8 * (j % kStages), (j / kStages) & 1, &dummy);
        }
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      bool ok = true;
      int cnt_next = my_items > 0 ? p.blk[item_of(0) / n_tiles].z : 0;   // one item ahead
      for (int i = 0; i < my_items && ok; ++i) {
        const int ab = i & 1;
        const int cnt = cnt_next;
        if (i + 1 < my_items) cnt_next = p.blk[item_of(i + 1) / n_tiles].z;
        const uint32_t idesc = tc::idesc_f16_f32(kTW, ((cnt + 15) / 16) * 16);
        ok = tc::mbar_wait(bar_acc_empty + 8 * ab, ((i >> 1) & 1) ^ 1, abort_flag);
        if (!ok) break;
        tc::tc_fence_after();
        const uint32_t dtm = tmem + (uint32_t)ab * kAccCols;
        for (int jb = 0; jb < KJ; ++jb) {
          const int j = i * KJ + jb, s = j % kStages;
          const uint32_t ph = (j / kStages) & 1;
          ok = tc::mbar_wait(bar_full_a + 8 * s, ph, abort_flag, 100);
          if (!ok) break;
          tc::tc_fence_after();
#pragma unroll
          for (int h = 0; h < kKps; ++h) {
            const uint64_t ad = tc::smem_desc_sw128(sA + (s * kKps + h) * kABytes);
            const uint64_t bd = tc::smem_desc_sw128(sB + (s * kKps + h) * kBBytes);
#pragma unroll
            for (int k = 0; k < kBK / 16; ++k)
              tc::mma_bf16(dtm, ad + 2 * k, bd + 2 * k, idesc, (jb | h | k) != 0);
          }
          tc::mma_commit(bar_empty + 8 * s);
        }
        if (ok) tc::mma_commit(bar_acc_full + 8 * ab);
      }
    }
  } else if (warp < 10) {
    // ---------------- decode producers: thread (row, half) ----------------
    // A row of a weight box (4 K blocks = 8 blocks) is read once into registers (Q4_0: nine
    // 16-byte loads; the 144- and 272-byte row strides put 8 consecutive rows on distinct bank
    // quads); thread half h then decodes block 2*kk + h of K block kk into chunks 4h .. 4h+3 of
    // the fp16 row.  half is uniform within a warp (warps 2-5: 0, warps 6-9: 1).
    // The largest |d| a thread decodes is tracked (fp16 bit patterns of non-negative values
    // order like the values); one at or above 8192 (Q4_0) or 512 (Q8_0), where a code can give
    // a product beyond fp16's range, is reported once at the end.
    constexpr uint32_t kBigD = BT == kQ8_0 ? 0x6000u : 0x7000u;   // fp16 bits of 512 / 8192
    const int pt = threadIdx.x - 64;          // 0..255
    const int tp = pt & (kTW - 1), half = pt >> 7;
    const int boxes_per_item = KB / 4;
    bool ok = true;
    uint32_t dmax = 0;
    for (int q = 0; q < my_items * boxes_per_item && ok; ++q) {
      const int slot = q % kRawSlots;
      if (!tc::mbar_wait(bar_raw_full + 8 * slot, (q / kRawSlots) & 1, abort_flag, 100)) break;
      const uint4 *row = reinterpret_cast<const uint4 *>(smem + L::raw + slot * kRawBytes + tp * kRawRow);
      // v: Q4_0, the whole 144-byte row; Q8_0, the nine words of this thread's block per K block
      uint32_t v[36];
      if constexpr (BT == kQ4_0) {
#pragma unroll
        for (int m = 0; m < 9; ++m) {
          const uint4 r4 = row[m];
          v[4 * m] = r4.x; v[4 * m + 1] = r4.y; v[4 * m + 2] = r4.z; v[4 * m + 3] = r4.w;
        }
      } else {
        uint32_t u[4][9];
        if (half == 0) q8_0_box_words<0>(row, u);
        else q8_0_box_words<1>(row, u);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
#pragma unroll
          for (int i = 0; i < 9; ++i) v[9 * kk + i] = u[kk][i];
      }
      tc::mbar_arrive(bar_raw_empty + 8 * slot);   // registers hold the box now
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const int kbt = q * 4 + kk;               // K tile of this CTA's sequence
        const int j = kbt / kKps, h = kbt % kKps;  // pipeline stage, tile within it
        const int s = j % kStages;
        const uint32_t ph = (j / kStages) & 1;
        constexpr int kQsWords = BT == kQ8_0 ? 8 : 4;
        uint32_t qs[kQsWords], d2;
        if constexpr (BT == kQ4_0) {
          // block 2kk+half: 18 bytes at byte 36kk + 18 half
          if (half == 0) {
            const uint32_t *u = v + 9 * kk;
#pragma unroll
            for (int m = 0; m < 4; ++m) qs[m] = prmt(u[m], u[m + 1], 0x5432u);
            d2 = (u[0] & 0xFFFFu) | (u[0] << 16);
          } else {
            const uint32_t *u = v + 9 * kk + 4;
#pragma unroll
            for (int m = 0; m < 4; ++m) qs[m] = u[1 + m];
            d2 = (u[0] >> 16) | (u[0] & 0xFFFF0000u);
          }
        } else {
          // block 2kk+half: 34 bytes at byte 68kk + 34 half; v + 9kk holds its words
          const uint32_t *u = v + 9 * kk;
          if (half == 0) {
#pragma unroll
            for (int m = 0; m < 8; ++m) qs[m] = prmt(u[m], u[m + 1], 0x5432u);
            d2 = (u[0] & 0xFFFFu) | (u[0] << 16);
          } else {
#pragma unroll
            for (int m = 0; m < 8; ++m) qs[m] = u[1 + m];
            d2 = (u[0] >> 16) | (u[0] & 0xFFFF0000u);
          }
        }
        dmax = max(dmax, d2 & 0x7FFFu);
        if (h == 0 && !tc::mbar_wait(bar_empty + 8 * s, ph ^ 1, abort_flag, 100)) { ok = false; break; }
        uint8_t *a_tile = smem + L::a + (s * kKps + h) * kABytes;
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          uint4 c;
          if constexpr (BT == kQ4_0) c = q4_0_chunk(qs[m], d2);
          else c = q8_0_chunk(qs[m], qs[m + 4], d2);
          *reinterpret_cast<uint4 *>(a_tile + tc::sw128_offset((uint32_t)tp, (uint32_t)(4 * half + m))) = c;
        }
        if (h == kKps - 1) {
          // The stage's B tiles have landed too once full_a completes: every producer waits
          // for them before its arrival, so the MMA issuer waits on one barrier per stage.
          tc::fence_proxy_async_smem();
          if (!tc::mbar_wait(bar_full_b + 8 * s, ph, abort_flag, 100)) { ok = false; break; }
          tc::mbar_arrive(bar_full_a + 8 * s);
        }
      }
    }
    if (dmax >= kBigD) raise_device_error(Q4MM_DEVERR_F16_RANGE);
  } else {
    // ---------------- epilogue: TMEM -> out rows (fp32) ----------------
    const int quarter = warp & 3;
    for (int i = 0; i < my_items; ++i) {
      const int ab = i & 1;
      if (!tc::mbar_wait(bar_acc_full + 8 * ab, (i >> 1) & 1, abort_flag)) break;
      tc::tc_fence_after();
      const int w = item_of(i);
      const int4 bi = p.blk[w / n_tiles];
      const int n = (w % n_tiles) * kTW + quarter * 32 + lane;
      for (int c0 = 0; c0 < bi.z; c0 += 32) {
        uint32_t v[32];
        tc::tmem_ld_32x32b_x32(tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)ab * kAccCols + (uint32_t)c0, v);
        tc::tmem_ld_wait();
        const int r_lane = c0 + lane < bi.z ? p.hids[bi.y + c0 + lane] : 0;
        const float un_lane = c0 + lane < bi.z ? p.xun[bi.y + c0 + lane] : 1.f;
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) {
          const int r = __shfl_sync(0xFFFFFFFFu, r_lane, jj);
          const float un = __shfl_sync(0xFFFFFFFFu, un_lane, jj);
          if (c0 + jj < bi.z && n < p.N) p.out[(size_t)r * p.N + n] = __uint_as_float(v[jj]) * un;
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

// Per token t: the power of two 2^e_t that brings the row's largest magnitude m into
// [2^14, 2^15) (e_t = 15 - frexp exponent of m, clamped to [-126, 127] so that both 2^e_t and
// 2^-e_t are f32 values; m == 0 or a non-finite m keeps e_t = 0).  One CTA per token.
__global__ void __launch_bounds__(256) token_scale_kernel(const float *__restrict__ x, int K,
                                                          float *__restrict__ tsc) {
  __shared__ float red[8];
  griddep_launch_dependents();
  const float4 *row = reinterpret_cast<const float4 *>(x + (size_t)blockIdx.x * K);
  float m = 0.f;
  for (int i = threadIdx.x; i < K / 4; i += blockDim.x) {
    const float4 v = __ldg(row + i);
    m = fmaxf(m, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  if (threadIdx.x % 32 == 0) red[threadIdx.x / 32] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < (int)(blockDim.x / 32); ++w) m = fmaxf(m, red[w]);
    int e = 0;
    if (m > 0.f && m <= 3.402823466e38f) {
      int ex = 0;
      frexpf(m, &ex);          // m in [2^(ex-1), 2^ex)
      e = min(max(15 - ex, -126), 127);
    }
    tsc[blockIdx.x] = ldexpf(1.f, e);
  }
  // Launched as a programmatic dependent of the routing, which it does not read: it runs
  // alongside and completes only after the routing has, so the chain stays ordered.
  griddep_wait();
}

// xs[p] = fp16(2^e_t * x[t]) with t = hids[p] / top_k for p < number of valid routed rows,
// each 32-element block laid out in the chunk order of q4_0_chunk, and xun[p] = 2^-e_t.
// Multiplying by a power of two is exact, so the only rounding is the one to fp16, relative
// to the token row's own range.  Item = (row, block, chunk m): two float4 loads (elements
// 4m.. and 16+4m..) and one 16-byte store; a CTA takes four rows at a time, so each thread
// has four items' loads in flight.
__global__ void __launch_bounds__(256) gather_rows_kernel(const float *__restrict__ x, const int32_t *__restrict__ hids,
                                                          const uint32_t *__restrict__ n_valid, int top_k, int K,
                                                          const float *__restrict__ tsc, uint16_t *__restrict__ xs,
                                                          float *__restrict__ xun, int n_rows) {
  griddep_launch_dependents();
  griddep_wait();   // the routing lists and token scales come from the two kernels before
  const int nv = min((int)*n_valid, n_rows);
  const int per_row = K / 8;   // items per row: K / 32 blocks x 4 chunks
  for (int pos0 = blockIdx.x * 4; pos0 < nv; pos0 += gridDim.x * 4) {
    const float *src[4];
    float f[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int tok = pos0 + u < nv ? hids[pos0 + u] / top_k : 0;
      src[u] = pos0 + u < nv ? x + (size_t)tok * K : nullptr;
      f[u] = pos0 + u < nv ? __ldg(tsc + tok) : 1.f;
      if (threadIdx.x == 0 && pos0 + u < nv) xun[pos0 + u] = 1.0f / f[u];   // exact: a power of two
    }
    for (int i = threadIdx.x; i < per_row; i += blockDim.x) {
      const int off = (i >> 2) * 32 + 4 * (i & 3);
      float4 lo[4], hi[4];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (src[u] != nullptr) {
          lo[u] = __ldg(reinterpret_cast<const float4 *>(src[u] + off));
          hi[u] = __ldg(reinterpret_cast<const float4 *>(src[u] + off + 16));
        }
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (src[u] != nullptr) {
          const float s = f[u];
          const float4 a = lo[u], b = hi[u];
          __half2 h0 = __floats2half2_rn(a.x * s, a.z * s), h1 = __floats2half2_rn(a.y * s, a.w * s);
          __half2 h2 = __floats2half2_rn(b.x * s, b.z * s), h3 = __floats2half2_rn(b.y * s, b.w * s);
          *reinterpret_cast<uint4 *>(xs + (size_t)(pos0 + u) * K + (size_t)i * 8) =
              make_uint4(*reinterpret_cast<uint32_t *>(&h0), *reinterpret_cast<uint32_t *>(&h1),
                         *reinterpret_cast<uint32_t *>(&h2), *reinterpret_cast<uint32_t *>(&h3));
        }
    }
  }
}

// Launch with programmatic stream serialization: the kernel may start while the previous
// kernel in the stream finishes, and must call griddep_wait() before it reads that kernel's
// output.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                             Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

}  // namespace

cudaError_t launch_routed_mm_tc(int bt, const float *x, const uint8_t *w, float *out, int n_tokens, int top_k,
                                int N, int K, int n_experts, uint64_t expert_stride, void *workspace, cudaStream_t s) {
  if (bt != kQ4_0 && bt != kQ8_0) return cudaErrorInvalidValue;
  auto enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  const int n_rows = n_tokens * top_k;
  const MoeWorkspace L = moe_workspace_layout(n_rows, K, n_experts);
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  const int32_t *hids = reinterpret_cast<const int32_t *>(ws + L.hids);
  const uint32_t *offs = reinterpret_cast<const uint32_t *>(ws + L.offs);
  uint16_t *xs = reinterpret_cast<uint16_t *>(ws + L.xs);
  float *xun = reinterpret_cast<float *>(ws + L.xun);
  float *tsc = reinterpret_cast<float *>(ws + L.tsc);
  int sms = 148, dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);

  // token scale, gather and mat-mat are programmatic dependents of the kernel before each
  // (every one waits for its predecessor before it reads what that wrote)
  cudaError_t e = launch_dependent(token_scale_kernel, dim3((unsigned)n_tokens), dim3(256), 0, s, x, K, tsc);
  if (e != cudaSuccess) return e;
  e = launch_dependent(gather_rows_kernel, dim3((unsigned)(4 * sms)), dim3(256), 0, s, x,
                       static_cast<const int32_t *>(hids), offs + n_experts, top_k, K,
                       static_cast<const float *>(tsc), xs, xun, n_rows);
  if (e != cudaSuccess) return e;

  MmMaps maps;
  const bool q8 = bt == kQ8_0;
  const uint64_t row_bytes = (uint64_t)(K / 32) * (q8 ? 34 : 18);
  {
    // Q4_0 rows as uint8 elements (144-element box rows), Q8_0 rows as uint16 elements
    // (136-element box rows: 272 uint8 elements would exceed the 256-element limit of a box
    // dimension)
    const uint64_t esz = q8 ? 2 : 1;
    cuuint64_t dims[3] = {(cuuint64_t)(row_bytes / esz), (cuuint64_t)N, (cuuint64_t)n_experts};
    cuuint64_t strides[2] = {(cuuint64_t)row_bytes, (cuuint64_t)expert_stride};
    cuuint32_t box[3] = {q8 ? RawCfg<kQ8_0>::kBoxX : RawCfg<kQ4_0>::kBoxX, (cuuint32_t)kTW, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    if (enc(&maps.w, q8 ? CU_TENSOR_MAP_DATA_TYPE_UINT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 3,
            const_cast<uint8_t *>(w), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)n_rows};
    cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    cuuint32_t box[2] = {(cuuint32_t)kBK, kBoxTok};
    cuuint32_t estr[2] = {1, 1};
    if (enc(&maps.xs, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, xs, dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  MmParams p{};
  p.out = out;
  p.hids = hids;
  p.xun = xun;
  p.blk = reinterpret_cast<const int4 *>(ws + L.blk);
  p.n_blk = reinterpret_cast<const uint32_t *>(ws + L.n_blk);
  p.N = N;
  p.K = K;
  if (q8) {
    e = ensure_dynamic_smem(reinterpret_cast<const void *>(routed_mm_tc_kernel<kQ8_0>), (int)mm_smem_bytes<kQ8_0>());
    if (e != cudaSuccess) return e;
    e = launch_dependent(routed_mm_tc_kernel<kQ8_0>, dim3((unsigned)sms), dim3(kThreads), mm_smem_bytes<kQ8_0>(), s,
                         maps, p);
  } else {
    e = ensure_dynamic_smem(reinterpret_cast<const void *>(routed_mm_tc_kernel<kQ4_0>), (int)mm_smem_bytes<kQ4_0>());
    if (e != cudaSuccess) return e;
    e = launch_dependent(routed_mm_tc_kernel<kQ4_0>, dim3((unsigned)sms), dim3(kThreads), mm_smem_bytes<kQ4_0>(), s,
                         maps, p);
  }
  return e;
}

}  // namespace q4mm
