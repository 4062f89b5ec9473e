// gemv_tma.cuh -- INT4 decode matmul (1 <= M <= 16, K % 256 == 0), TMA-fed and
// warp-specialised.  Included by gemv.cu, whose GemvParams, LaunchSpec and cluster_sum_store
// it uses.
//
// What it computes: y[m][n] = sum_k x[m][k] * (q[n][k] * s[n][g] + b[n][g]), g = k / 32, the
// INT4 group-32 affine MatMulNBits product of quant_fastkernel.rs (codes low nibble first).
// The sum is regrouped as
//     sum_k x[m][k] * (q s)[n][k]   +   sum_g b[n][g] * X[m][g],   X[m][g] = sum_{k in g} x[m][k],
// both parts on the tensor cores (mma.sync m16n8k16, bf16 operands, fp32 accumulation):
//   * q s: the code enters as the bf16 value 128 + q (one LOP3), and one bf16x2 FMA
//     fma(128 + q, s, -128 s) gives q s rounded once (-128 s is exact in bf16, so the FMA
//     sees q s exactly before its single rounding);
//   * b X: two extra MMA k-steps per 16 groups, with the biases as they are stored (bf16
//     pairs are already A-fragment registers) against X split into bf16 hi + lo parts, so
//     X enters with about 16 significant bits.
//
// Work layout.  A CTA owns R = 16 * WC weight rows over one K slice.  Warp WC is the
// producer: one thread streams the tile's codes, scales and biases from HBM into a ring of
// shared-memory stages with 2D TMA loads (one stage = R rows x 256 k: a 128-byte code box
// with the 128-byte swizzle, and 16-byte scale and bias boxes), completion counted on a
// "full" mbarrier per stage.  Warps 0 .. WC-1 are consumers: warp w decodes rows
// 16w .. 16w+15 of every stage (lane (g, t) holds rows g and g + 8) and releases the stage
// on its "empty" mbarrier.  Several stages are in flight per CTA without holding
// registers, and the consumer warps issue no load instructions for the weights but their
// 16-byte shared reads.  The producer issues its first stages before the kernel waits on
// the previous kernel (weights are static), so the weight stream overlaps that kernel's
// tail.  K slices of one row range form a thread-block cluster whose partial tiles are
// summed in rank order through distributed shared memory (deterministic, no workspace).
//
// k order.  A dot product does not depend on the order of its terms as long as x and W use
// the same one.  Inside a 512-k block (16 groups) lane t handles groups 2t, 2t + 1, 2t + 8,
// 2t + 9 as the four 128-k sub-chunks of the block, and within a group the LOP3 decode
// yields code pairs (i, i + 4); x is staged once per CTA in shared memory in exactly that
// order, so each MMA reads its x fragment with one 16-byte shared load.

struct GemvTmaArgs {
  GemvParams p;
  CUtensorMap wmap;   // codes: uint8 [N][K / 2], box [128 B][R rows], 128-byte swizzle
  CUtensorMap smap;   // scales: bf16 [N][K / 32], box [8 groups][R rows]
  CUtensorMap bmap;   // biases: same
  int stages;         // ring stages in shared memory
};

__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// Named barrier over the consumer warps only (the producer warp does not take part).
__device__ __forceinline__ void consumer_sync(int nthreads) {
  asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");
}

// Shared memory of one CTA (K slice of at most maxnh half-blocks, nbmax = ceil(maxnh / 2)):
//   stage ring   [stages][codes R x 128 B (swizzled) | scales R x 16 B | biases R x 16 B]
//   xs    [M][TS]: token row; sub-chunk c (= 2 * local half + j) at c * 256:
//         [piece p = 0..3][lane t = 0..3][16 B] = B fragments of k-steps 2p, 2p + 1
//   xsum  [M][nbmax][t][16 B]: (hi(2t, 2t+1), hi(2t+8, 2t+9), lo(2t, 2t+1), lo(2t+8, 2t+9))
//         bf16 pairs of the group sums of each 16-group block
//   red   [KS][M][R] fp32 partial tiles of the consumer groups, summed in group order
//   full[stages], empty[stages] mbarriers, abort flag
// A stage holds KS half-blocks (KS consumer groups split it); each half-block sub-stage is
// [codes R x 128 B | scales R x 16 B | biases R x 16 B], a multiple of 1024 bytes.
__host__ __device__ inline uint32_t tq_stage_bytes(int R, int KS) { return (uint32_t)R * 160u * (uint32_t)KS; }
__host__ __device__ inline int tq_ts(int nh) { return nh * 512 + 64; }
__host__ __device__ inline size_t tq_smem_bytes(int M, int nh, int R, int KS, int stages) {
  const int nb = (nh + 1) / 2;
  return 1024 + (size_t)stages * tq_stage_bytes(R, KS) + (size_t)M * tq_ts(nh) + (size_t)M * nb * 64 +
         (size_t)KS * M * R * 4 + (size_t)stages * 16 + 16;
}

template <int NT, int WC, int KS>
__global__ void __launch_bounds__((WC * KS + 1) * 32) gemv_tma_kernel(const __grid_constant__ GemvTmaArgs a) {
  constexpr int R = 16 * WC;
  constexpr int NC = WC * KS;                       // consumer warps; warp NC is the producer
  constexpr uint32_t kSub = R * 160u, kCodes = R * 128u, kStage = kSub * KS;
  const GemvParams &p = a.p;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_s = smem_u32(smem_raw);
  uint8_t *smem = smem_raw + (((raw_s + 1023u) & ~1023u) - raw_s);   // 1024-aligned (swizzle atoms)
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int g = lane / 4, t = lane % 4;
  const int NH = p.K / 256;                  // half-blocks per row
  const int NB = (NH + 1) / 2;               // blocks per row
  const int S = (int)gridDim.y, split = (int)blockIdx.y;
  const int b0 = (split * NB) / S, b1 = ((split + 1) * NB) / S;
  const int h0 = 2 * b0, h1 = min(2 * b1, NH);
  const int nh = h1 - h0;                    // this CTA's half-blocks
  const int nb = b1 - b0;
  const int maxnh = p.max_chunks_per_cta;    // largest nh over the splits (smem sizing)
  const int TS = tq_ts(maxnh);
  const int nbmax = (maxnh + 1) / 2;
  const int ST = a.stages;
  uint8_t *ring = smem;
  uint8_t *xs = ring + (size_t)ST * kStage;
  uint8_t *xsum = xs + (size_t)p.M * TS;
  float *red = reinterpret_cast<float *>(xsum + (size_t)p.M * nbmax * 64);
  const uint32_t full0 = smem_u32(red + KS * p.M * R);
  const uint32_t empty0 = full0 + 8u * (uint32_t)ST;
  volatile int *abort_flag = reinterpret_cast<volatile int *>(red + KS * p.M * R + 4 * ST);
  const int row0 = (int)blockIdx.x * R;
  const int nst = (nh + KS - 1) / KS;        // stages of this slice (the last may hold one half-block)

  if (threadIdx.x == 0) {
    for (int s = 0; s < ST; ++s) {
      tc::mbar_init(full0 + 8 * s, 1);
      tc::mbar_init(empty0 + 8 * s, NC);
    }
    *abort_flag = 0;
    tc::fence_mbar_init();
  }
  __syncthreads();
  griddep_launch_dependents();   // the next kernel may start streaming its (static) weights

  if (warp == NC) {
    // ---------------- producer: TMA of codes, scales and biases, KS half-blocks per stage ----------------
    if (lane == 0) {
      tc::tma_prefetch_desc(&a.wmap);
      tc::tma_prefetch_desc(&a.smap);
      tc::tma_prefetch_desc(&a.bmap);
      int issued = 0;
      for (int i = 0, s = 0, ph = 0; i < nst; ++i) {
        if (i >= ST && !tc::mbar_wait(empty0 + 8 * s, (uint32_t)(ph ^ 1), abort_flag)) break;
        const uint32_t dst = smem_u32(ring) + (uint32_t)s * kStage;
        const uint32_t bar = full0 + 8 * s;
        const int nsub = min(KS, nh - i * KS);
        tc::mbar_arrive_expect_tx(bar, kSub * (uint32_t)nsub);
        for (int j = 0; j < nsub; ++j) {
          const int hb = h0 + i * KS + j;
          const uint32_t d = dst + (uint32_t)j * kSub;
          tc::tma_load_2d(d, &a.wmap, hb * 128, row0, bar);
          tc::tma_load_2d(d + kCodes, &a.smap, hb * 8, row0, bar);
          tc::tma_load_2d(d + kCodes + R * 16, &a.bmap, hb * 8, row0, bar);
        }
        ++issued;
        if (++s == ST) {
          s = 0;
          ph ^= 1;
        }
      }
      if (*abort_flag) {   // let the loads in flight land before the CTA exits
        for (int i = (issued > ST ? issued - ST : 0); i < issued; ++i) {
          volatile int dummy = 0;
          tc::mbar_wait(full0 + 8 * (i % ST), (uint32_t)((i / ST) & 1), &dummy);
        }
      }
    }
  } else {
    // ---------------- consumers ----------------
    // x may be the previous kernel's output, and y may still be read by it.
    griddep_wait();
    // Stage x of the slice in the decode's k order, and the hi/lo group sums.  Each thread
    // takes items (token, group) four at a time and issues all of their loads before using
    // any, so the staging costs about one L2 round trip per four items.
    {
      const int ngrp = 16 * nb;   // groups of the slice's blocks (a last half-block may be missing)
      const int items = p.M * ngrp;
      constexpr int kU = 4;
      for (int it0 = threadIdx.x; it0 < items; it0 += kU * NC * 32) {
        uint4 v[kU][4];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
          const int it = it0 + u * NC * 32;
          const int tok = it / ngrp, gi = 16 * b0 + it % ngrp;
          if (it < items && gi < 8 * h1) {
            const uint4 *src = reinterpret_cast<const uint4 *>(p.x + (size_t)tok * p.K + (size_t)gi * 32);
#pragma unroll
            for (int i = 0; i < 4; ++i) v[u][i] = __ldg(src + i);
          } else {
#pragma unroll
            for (int i = 0; i < 4; ++i) v[u][i] = make_uint4(0u, 0u, 0u, 0u);
          }
        }
#pragma unroll
        for (int u = 0; u < kU; ++u) {
          const int it = it0 + u * NC * 32;
          if (it >= items) break;
          const int tok = it / ngrp, gl = it % ngrp;
          const int gi = 16 * b0 + gl;             // group index in the row
          const int blk = gl >> 4, j16 = gl & 15;
          const int half = j16 >> 3, tt = (j16 & 7) >> 1, jj = j16 & 1;
          uint32_t X[16];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            X[4 * i] = v[u][i].x; X[4 * i + 1] = v[u][i].y; X[4 * i + 2] = v[u][i].z; X[4 * i + 3] = v[u][i].w;
          }
          if (gi < 8 * h1) {
            uint8_t *dst = xs + (size_t)tok * TS + ((blk * 2 + half) * 2 + jj) * 256 + tt * 16;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              // k-step 2q + r takes (x[8q+2r], x[8q+2r+4]) and (x[8q+2r+1], x[8q+2r+5])
              const uint32_t a0 = X[4 * q], b0v = X[4 * q + 2], a1 = X[4 * q + 1], b1v = X[4 * q + 3];
              *reinterpret_cast<uint4 *>(dst + q * 64) = make_uint4(prmt(a0, b0v, 0x5410), prmt(a0, b0v, 0x7632),
                                                                    prmt(a1, b1v, 0x5410), prmt(a1, b1v, 0x7632));
            }
          }
          float sum = 0.f;   // 0 for groups past the slice (their loads were skipped)
#pragma unroll
          for (int i = 0; i < 16; ++i) sum += __uint_as_float(X[i] << 16) + __uint_as_float(X[i] & 0xFFFF0000u);
          // group sum as bf16 hi + lo
          __nv_bfloat16 hb = __float2bfloat16_rn(sum);
          const float hi = __bfloat162float(hb);
          __nv_bfloat16 lb = __float2bfloat16_rn(sum - hi);
          uint8_t *xd = xsum + ((size_t)tok * nbmax + blk) * 64 + tt * 16 + half * 4 + jj * 2;
          *reinterpret_cast<__nv_bfloat16 *>(xd) = hb;
          *reinterpret_cast<__nv_bfloat16 *>(xd + 8) = lb;
        }
      }
    }
    consumer_sync(NC * 32);

    // B-fragment rows: token 8 nt + g (tokens past M read token M - 1; their columns are
    // never stored, and a product column depends only on its own B column).
    const uint8_t *xrow[NT], *srow[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int tok = min(8 * nt + g, p.M - 1);
      xrow[nt] = xs + tok * TS + t * 16;
      srow[nt] = xsum + tok * nbmax * 64 + t * 16;
    }
    float acc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;

    constexpr uint32_t kMask = 0x000F000Fu, kMagic = 0x43004300u, kNeg128 = 0xC300C300u;
    // This warp's rows inside a stage: codes of row r, 16-byte chunk c at r * 128 + ((c ^ (r & 7)) * 16)
    // (the TMA's 128-byte swizzle); lane (g, t) reads chunks 2t, 2t + 1 of rows g and g + 8.
    const int kh = warp / WC;                 // this warp's half-block of every stage
    const int rA = (warp % WC) * 16 + g;
    uint32_t coff[2][2];
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int r = rA + 8 * h;
        coff[h][j] = (uint32_t)(r * 128 + (((2 * t + j) ^ (r & 7)) << 4));
      }
    const uint32_t soff0 = kCodes + (uint32_t)(rA * 16 + t * 4);

    // Main product of local half-block lh from the stage's values (codes qv, scale pairs sv).
    auto half_product = [&](int lh, const uint4 (&qv)[2][2], const uint32_t (&sv)[2]) {
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        uint32_t s2[2], m2[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          s2[h] = prmt(sv[h], 0, j ? 0x3232u : 0x1010u);   // (s, s) of group 2t + j
          m2[h] = bf16x2_mul(s2[h], kNeg128);               // (-128 s, -128 s), exact
        }
        const int xoff = (2 * lh + j) * 256;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint32_t w0 = q == 0 ? qv[0][j].x : q == 1 ? qv[0][j].y : q == 2 ? qv[0][j].z : qv[0][j].w;
          const uint32_t w1 = q == 0 ? qv[1][j].x : q == 1 ? qv[1][j].y : q == 2 ? qv[1][j].z : qv[1][j].w;
          const uint32_t ws0[4] = {w0, w0 >> 4, w0 >> 8, w0 >> 12};
          const uint32_t ws1[4] = {w1, w1 >> 4, w1 >> 8, w1 >> 12};
          uint32_t pg[4], pg8[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            pg[i] = bf16x2_fma(and_or(ws0[i], kMask, kMagic), s2[0], m2[0]);
            pg8[i] = bf16x2_fma(and_or(ws1[i], kMask, kMagic), s2[1], m2[1]);
          }
          const uint32_t a0[4] = {pg[0], pg8[0], pg[1], pg8[1]};
          const uint32_t a1[4] = {pg[2], pg8[2], pg[3], pg8[3]};
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            const uint4 xb = *reinterpret_cast<const uint4 *>(xrow[nt] + xoff + q * 64);
            mma_bf16_16816(acc[nt], a0, xb.x, xb.y);
            mma_bf16_16816(acc[nt], a1, xb.z, xb.w);
          }
        }
      }
    };
    // Bias product of local block lb: A = bias pairs of groups (2t, 2t+1) and (2t+8, 2t+9)
    // for rows g and g + 8, B = the block's group sums (hi, then lo).
    auto bias_product = [&](uint32_t bg0, uint32_t bg8_0, uint32_t bg1, uint32_t bg8_1, int lb) {
      const uint32_t ab[4] = {bg0, bg8_0, bg1, bg8_1};
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const uint4 xf = *reinterpret_cast<const uint4 *>(srow[nt] + lb * 64);
        mma_bf16_16816(acc[nt], ab, xf.x, xf.y);
        mma_bf16_16816(acc[nt], ab, xf.z, xf.w);
      }
    };

    int s = 0, ph = 0;
    bool ok = true;
    // Reads this warp's codes, scale pairs and bias pairs of a half-block sub-stage and
    // releases the stage (its values are then in registers).
    auto take = [&](const uint8_t *st, uint4 (&qv)[2][2], uint32_t (&sv)[2], uint32_t (&bq)[2]) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
#pragma unroll
        for (int jj = 0; jj < 2; ++jj) qv[h][jj] = *reinterpret_cast<const uint4 *>(st + coff[h][jj]);
        sv[h] = *reinterpret_cast<const uint32_t *>(st + soff0 + h * 128);
        bq[h] = *reinterpret_cast<const uint32_t *>(st + soff0 + R * 16 + h * 128);
      }
    };
    auto release = [&]() {
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(empty0 + 8 * s);
      if (++s == ST) {
        s = 0;
        ph ^= 1;
      }
    };
    if constexpr (KS == 1) {
      // Two half-blocks (one 512-k block) per iteration, one stage each.
      for (int lh = 0; lh < nh && ok; lh += 2) {
        uint32_t bA[2], bB[2] = {0u, 0u};
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int l = lh + j;
          if (l < nh) {
            if (!tc::mbar_wait(full0 + 8 * s, (uint32_t)ph, abort_flag, 200)) {
              ok = false;
              break;
            }
            uint4 qv[2][2];
            uint32_t sv[2];
            take(ring + (size_t)s * kStage, qv, sv, j == 0 ? bA : bB);
            release();
            half_product(l, qv, sv);
          }
        }
        if (!ok) break;
        if (lh + 1 < nh) bias_product(bA[0], bA[1], bB[0], bB[1], lh >> 1);
        else bias_product(bA[0], bA[1], bA[0], bA[1], lh >> 1);   // the slice ends after a first half:
                                                                   // that block's other X are zero
      }
    } else {
      // One 512-k block per stage; consumer group kh takes its half-block kh, and its bias
      // product carries zeros in place of the other half's biases.
      for (int i = 0; i < nst; ++i) {
        if (!tc::mbar_wait(full0 + 8 * s, (uint32_t)ph, abort_flag, 200)) {
          ok = false;
          break;
        }
        const int l = 2 * i + kh;
        if (l < nh) {
          uint4 qv[2][2];
          uint32_t sv[2], bq[2];
          take(ring + (size_t)s * kStage + (size_t)kh * kSub, qv, sv, bq);
          release();
          half_product(l, qv, sv);
          if (kh == 0) bias_product(bq[0], bq[1], 0u, 0u, i);
          else bias_product(0u, 0u, bq[0], bq[1], i);
        } else {
          release();
        }
      }
    }

    // Partial tile of this consumer group -> red[kh][tok][row].
    float *rk = red + kh * p.M * R;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int tk = 8 * nt + 2 * t;
      if (tk < p.M) {
        rk[tk * R + rA] = acc[nt][0];
        rk[tk * R + rA + 8] = acc[nt][2];
      }
      if (tk + 1 < p.M) {
        rk[(tk + 1) * R + rA] = acc[nt][1];
        rk[(tk + 1) * R + rA + 8] = acc[nt][3];
      }
    }
  }

  if constexpr (KS > 1) {   // the consumer groups' partials, summed in group order
    __syncthreads();
    for (int i = threadIdx.x; i < p.M * R; i += (NC + 1) * 32) {
      float v = red[i];
#pragma unroll
      for (int k = 1; k < KS; ++k) v += red[k * p.M * R + i];
      red[i] = v;
    }
  }
  // red -> y (one split) or the cluster's rank-order sum; every thread of the CTA takes part.
  if (S > 1) {
    cluster_sum_store<R>(p, red);
    return;
  }
  __syncthreads();
  const int quads = R / 4;
  for (int i = threadIdx.x; i < p.M * quads; i += (NC + 1) * 32) {
    const int tok = i / quads, qd = i % quads;
    const float4 v = *reinterpret_cast<const float4 *>(red + tok * R + qd * 4);
    const int n0 = row0 + qd * 4;
    uint16_t *dst = p.y + (size_t)tok * p.N + n0;
    if (n0 + 3 < p.N && (p.N & 3) == 0) {
      *reinterpret_cast<uint2 *>(dst) = make_uint2(pack_bf16x2(v.x, v.y), pack_bf16x2(v.z, v.w));
    } else {
      const float vals[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (n0 + j < p.N) {
          __nv_bfloat16 b = __float2bfloat16_rn(vals[j]);
          dst[j] = *reinterpret_cast<uint16_t *>(&b);
        }
    }
  }
}
