// Persistent warp-specialised bf16 GEMM on the 5th-generation tensor cores
// (tcgen05 + TMEM), fed by TMA, with these epilogues:
//   * PackEpi: z = acc + b, h = bf16(z) where z > 0, compaction of each
//     (row, T-column tile) into TwELL cells (values, tile-local indices,
//     count) and a per-row overflow flag -- the layer's up-projection with its
//     dense-to-TwELL pack fused in (repo-explainer, "TwELL: The Packing Format
//     That Fits the Machine": dense-to-TwELL and fused MLP execution).  A tile
//     that overflows C also spills its dense bf16 values so that the hybrid's
//     dense fallback row can be assembled without recomputation (ifai.io news,
//     "Reshaping math for the GPU": a dense matrix catches the rare dense
//     tokens).
//   * DenseEpi: bf16 rows with optional bias and ReLU (dense comparator).
//   * PartialEpi: fp32 stores, per K split when the K range is split (the
//     fallback rows' down-projection, dX and weight-gradient shares).
//   * GatedPackEpi: the gated (Llama-style) up-projection with the pack; for
//     training it also keeps (g, u) fp32 beside every stored value.
//   * SampleEpi: dH = dY . W_down^T kept only at the TwELL pattern, plus the
//     L1 term's gradient (bayesiansapien note, TL;DR) -- the backward SDDMM;
//     for the gated layer it forms (dG, dU) = (dh' u, dh' g) at the pattern.
//   * GUEpi: g = X.W_g + b and u = X.W_u of the gated layer's fallback rows,
//     for their share of its backward.
//   * MaskEpi, PartialTEpi: the dense comparator's masked dZ, and the
//     small-batch up-projection with swapped operands (fp32 K-split partials).
//
// C[M, N] = A[M, K] . B^T; A row-major [M][K] (K-major).  B is either
// row-major [N][K] (K-major) or row-major [K][N] (N-major, e.g. W_down read as
// the B operand of H . W_down).  CTA tile 128 x BN, K step 64, one CTA per SM,
// work units (m, n, k-split) strided over CTAs.  Warp roles: 0 = TMA
// producer, 1 = MMA issuer, 2 = TMEM owner, 4..11 = epilogue: warps 4+i and
// 8+i read TMEM lanes 32i..32i+31 (tile rows 32i..), the first taking the
// tile's left half of the columns and the second the right half.
// Accumulators are double-buffered in TMEM so one tile's epilogue runs under
// the next tile's MMAs.  Every pipeline wait is bounded and reports
// TWELL_ERR_WAIT_TIMEOUT.
#include <cuda_runtime.h>

#include <algorithm>

#include "sm103.cuh"
#include "twell_internal.h"

namespace twell {
namespace {

constexpr int kBM = 128;
constexpr int kBK = 64;
constexpr int kUmmaK = 16;
constexpr int kThreads = 384;  // 4 role warps + 8 epilogue warps
constexpr int kEpiThreads = 256;

template <int BN>
struct GemmCfg {
  static constexpr uint32_t kABytes = kBM * kBK * 2;
  static constexpr uint32_t kBBytes = BN * kBK * 2;
  // narrow (swapped-operand) tiles stream A: as many stages as ~192 KB holds
  static constexpr int kStages = BN == 256 ? 4 : BN == 128 ? 6 : static_cast<int>(196608u / (kABytes + kBBytes));
  static constexpr uint32_t kTmemCols = 2 * BN;  // two accumulators
  static constexpr uint32_t kPipeBytes = kStages * (kABytes + kBBytes);
  static constexpr uint32_t kBarBytes = 512;  // barriers, TMEM address, abort flag, per-stage parity
};

struct GemmArgs {
  int M;
  const int32_t* M_dev;  // optional device-side row count (clamped to M)
  int N;
  int K;
  int ksplit;            // K ranges per output tile (partial sums when > 1)
  const int32_t* K_dev;  // optional device-side K (times k_mul, clamped to K); operand rows/cols up to
                         // the next multiple of 64 past it must be zero
  int k_mul;
  int32_t* status;
  uint64_t wait_limit_ns;
  // words that CTA 0 sets to zero for the kernels that follow on the stream
  // (saves separate memset launches on short latency-bound paths)
  int32_t* zero0;
  int n_zero0;
  int32_t* zero1;
  int n_zero1;
  int b_k_wrap;  // N-major B: K row coordinate taken modulo this (0 = no wrap), a multiple of 64
};

// Row i of a 32-column TMEM chunk, picked with a select tree (no local memory).
__device__ __forceinline__ uint32_t pick32(const uint32_t (&r)[32], int k) {
  uint32_t a[16], b[8], c[4], d[2];
#pragma unroll
  for (int i = 0; i < 16; ++i) a[i] = (k & 16) ? r[i + 16] : r[i];
#pragma unroll
  for (int i = 0; i < 8; ++i) b[i] = (k & 8) ? a[i + 8] : a[i];
#pragma unroll
  for (int i = 0; i < 4; ++i) c[i] = (k & 4) ? b[i + 4] : b[i];
#pragma unroll
  for (int i = 0; i < 2; ++i) d[i] = (k & 2) ? c[i + 2] : c[i];
  return (k & 1) ? d[1] : d[0];
}

__device__ __forceinline__ float bias_at(const uint4 (&bq)[4], int i) {
  const uint32_t bw = (&bq[i / 8].x)[(i % 8) / 2];
  return (i & 1) ? bf16_hi(bw) : bf16_lo(bw);
}

// ------------------------------------------------------------ epilogues
struct PackEpi {
  static constexpr bool kDualB = false;
  using Params = PackEpiParams;
  static constexpr int kMaxCap = 32;
  static constexpr uint32_t kSmemBytes = kEpiThreads * kMaxCap * 3;  // per thread: C values (u16) + C indices (u8)

  // A positive z rounds (to nearest, ties to even) to a non-zero bf16 exactly
  // when z > 2^-134: half of the smallest bf16 subnormal, itself a tie that
  // rounds to the even neighbour 0.  So one compare decides "non-zero".
  static __device__ __forceinline__ float nonzero_threshold() { return __uint_as_float(0x00008000u); }

  // h of 32 columns [col, col + 32) of this thread's row, from TMEM.
  static __device__ __forceinline__ void load_h32(const Params& p, uint32_t taddr, int col, uint32_t (&r)[32],
                                                  uint4 (&bq)[4]) {
    tmem_ld32(taddr, r);
    const uint4* bp = reinterpret_cast<const uint4*>(p.bias + col);
#pragma unroll
    for (int q = 0; q < 4; ++q) bq[q] = __ldg(bp + q);
    tmem_ld_wait();
  }

  // One thread = one accumulator row; this warp handles whole T-column tiles:
  // the left or right half of the CTA tile, or all of it (second warp idle)
  // when one T-tile is wider than half.
  template <int BN>
  static __device__ __forceinline__ void apply(const Params& p, uint32_t taddr, int row, int M, int col0, int half,
                                               int, uint8_t* smem, int et) {
    const int T = p.tile, C = p.cap;
    int cb = half * (BN / 2), ce = cb + BN / 2;
    if (T > BN / 2) {
      if (half) return;
      cb = 0;
      ce = BN;
    }
    uint16_t* sv = reinterpret_cast<uint16_t*>(smem) + et * kMaxCap;
    uint8_t* si = smem + kEpiThreads * kMaxCap * 2 + et * kMaxCap;
    const bool valid = row < M;
    const float thr = nonzero_threshold();
    int cnt = 0;
#pragma unroll 1
    for (int c = cb; c < ce; c += 32) {
      uint32_t r[32];
      uint4 bq[4];
      load_h32(p, taddr + c, col0 + c, r, bq);
      const int j0 = c % T;
      if (j0 == 0) {
        cnt = 0;
        const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int q = 0; q < kMaxCap * 2 / 16; ++q) reinterpret_cast<uint4*>(sv)[q] = z;
#pragma unroll
        for (int q = 0; q < kMaxCap / 16; ++q) reinterpret_cast<uint4*>(si)[q] = z;
      }
      uint32_t mask = 0;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const float z = __uint_as_float(r[i]) + bias_at(bq, i);
        r[i] = __float_as_uint(z);
        mask |= (z > thr ? 1u : 0u) << i;
      }
      const int k = __popc(mask);
      if (cnt + k <= C) {
        while (mask) {
          const int i = __ffs(mask) - 1;
          mask &= mask - 1;
          sv[cnt] = float_to_bf16_bits(__uint_as_float(pick32(r, i)));
          si[cnt] = static_cast<uint8_t>(j0 + i);
          ++cnt;
        }
      } else {
        cnt += k;  // the tile overflows: its entries are spilled below instead
      }
      if ((c + 32) % T != 0) continue;
      // ---- the T-column tile [tile_c0, tile_c0 + T) is complete
      const int tile_c0 = c + 32 - T;
      const int t = (col0 + tile_c0) / T;
      const int64_t cell = static_cast<int64_t>(row) * p.n_tiles + t;
      const bool ovf = valid && cnt > C;
      if (valid && !ovf) {
        p.counts[cell] = static_cast<uint8_t>(cnt);
        if ((C & 7) == 0) {
          uint4* gv = reinterpret_cast<uint4*>(p.values + cell * C);
          uint2* gi = reinterpret_cast<uint2*>(p.idx + cell * C);
          for (int q = 0; q < C / 8; ++q) {
            gv[q] = reinterpret_cast<const uint4*>(sv)[q];
            gi[q] = reinterpret_cast<const uint2*>(si)[q];
          }
        } else {
          for (int q = 0; q < C; ++q) {
            p.values[cell * C + q] = sv[q];
            p.idx[cell * C + q] = si[q];
          }
        }
      }
      if (__any_sync(0xffffffffu, ovf)) {
        // The row becomes a fallback row: keep this tile's dense h so the
        // dense row can be assembled later.  TMEM still holds the tile.
        int slot = -1;
        if (ovf) {
          p.row_flag[row] = 1;
          slot = atomicAdd(p.spill_count, 1);
          if (slot >= p.spill_cap) {
            report_error(p.status, TWELL_ERR_FALLBACK_OVERFLOW);
            slot = -1;
          }
          p.counts[cell] = kSpilledCell;
          const uint32_t s24 = slot < 0 ? 0xFFFFFFu : static_cast<uint32_t>(slot);
          p.values[cell * C] = static_cast<uint16_t>(s24 & 0xFFFFu);
          p.idx[cell * C] = static_cast<uint8_t>(s24 >> 16);
        }
        for (int cc = tile_c0; cc < tile_c0 + T; cc += 32) {
          uint32_t rr[32];
          uint4 bb[4];
          load_h32(p, taddr + cc, col0 + cc, rr, bb);
          if (slot >= 0) {
            uint32_t packed[16];
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
              const float z0 = __uint_as_float(rr[i]) + bias_at(bb, i);
              const float z1 = __uint_as_float(rr[i + 1]) + bias_at(bb, i + 1);
              const uint32_t h0 = z0 > 0.0f ? float_to_bf16_bits(z0) : 0u;
              const uint32_t h1 = z1 > 0.0f ? float_to_bf16_bits(z1) : 0u;
              packed[i / 2] = h0 | (h1 << 16);
            }
            uint4* dst = reinterpret_cast<uint4*>(p.spill + static_cast<int64_t>(slot) * T + (cc - tile_c0));
#pragma unroll
            for (int q = 0; q < 4; ++q)
              dst[q] = make_uint4(packed[4 * q], packed[4 * q + 1], packed[4 * q + 2], packed[4 * q + 3]);
          }
        }
      }
    }
  }
};

// Gated (Llama-style) variant of PackEpi: the CTA's B stage holds 128 gate
// rows and 128 up rows of the same hidden units, so TMEM columns [0, BN/2)
// hold z_g = X.W_g and [BN/2, BN) hold z_u = X.W_u for units col0 .. col0+BN/2.
// h = bf16(z_g' * z_u) where z_g' = z_g + b > 0, else +0; a product of fp32
// rounds to a non-zero bf16 exactly when its magnitude exceeds 2^-134.
struct GatedPackEpi {
  static constexpr bool kDualB = true;
  using Params = PackEpiParams;
  static constexpr int kMaxCap = 32;
  static constexpr uint32_t kSmemBytes = kEpiThreads * kMaxCap * 3;

  // fp32 h of 32 units [c, c + 32) of this thread's row (bias applied to the gate)
  template <int BN>
  static __device__ __forceinline__ void load_h32(const Params& p, uint32_t taddr, int col0, int c,
                                                  uint32_t (&g)[32]) {
    uint32_t u[32];
    tmem_ld32(taddr + c, g);
    tmem_ld32(taddr + BN / 2 + c, u);
    const uint4* bp = reinterpret_cast<const uint4*>(p.bias + col0 + c);
    uint4 bq[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) bq[q] = __ldg(bp + q);
    tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const float zg = __uint_as_float(g[i]) + bias_at(bq, i);
      g[i] = __float_as_uint(zg > 0.0f ? zg * __uint_as_float(u[i]) : 0.0f);
    }
  }

  // the gate (bias applied) and up values of 32 units [c, c + 32) of this thread's row
  template <int BN>
  static __device__ __forceinline__ void load_gu32(const Params& p, uint32_t taddr, int col0, int c,
                                                   uint32_t (&g)[32], uint32_t (&u)[32]) {
    tmem_ld32(taddr + c, g);
    tmem_ld32(taddr + BN / 2 + c, u);
    const uint4* bp = reinterpret_cast<const uint4*>(p.bias + col0 + c);
    uint4 bq[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) bq[q] = __ldg(bp + q);
    tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < 32; ++i) g[i] = __float_as_uint(__uint_as_float(g[i]) + bias_at(bq, i));
  }

  template <int BN>
  static __device__ __forceinline__ void apply(const Params& p, uint32_t taddr, int row, int M, int col0, int half,
                                               int, uint8_t* smem, int et) {
    constexpr int U = BN / 2;  // hidden units per CTA tile
    const int T = p.tile, C = p.cap;
    int cb = half * (U / 2), ce = cb + U / 2;
    if (T > U / 2) {
      if (half) return;
      cb = 0;
      ce = U;
    }
    uint16_t* sv = reinterpret_cast<uint16_t*>(smem) + et * kMaxCap;
    uint8_t* si = smem + kEpiThreads * kMaxCap * 2 + et * kMaxCap;
    const bool valid = row < M;
    const float thr = __uint_as_float(0x00008000u);
    int cnt = 0;
#pragma unroll 1
    for (int c = cb; c < ce; c += 32) {
      uint32_t zg[32], zu[32];  // h = zg * zu where zg > 0, else +0
      load_gu32<BN>(p, taddr, col0, c, zg, zu);
      const int j0 = c % T;
      if (j0 == 0) {
        cnt = 0;
        const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int q = 0; q < kMaxCap * 2 / 16; ++q) reinterpret_cast<uint4*>(sv)[q] = z;
#pragma unroll
        for (int q = 0; q < kMaxCap / 16; ++q) reinterpret_cast<uint4*>(si)[q] = z;
      }
      uint32_t mask = 0;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const float g = __uint_as_float(zg[i]);
        const float h = g > 0.0f ? g * __uint_as_float(zu[i]) : 0.0f;
        mask |= (fabsf(h) > thr ? 1u : 0u) << i;
      }
      const int k = __popc(mask);
      if (cnt + k <= C) {
        // (g, u) of each stored slot, for the backward
        float* gu = (p.gu && valid)
                        ? p.gu + (static_cast<int64_t>(row) * p.n_tiles + (col0 + c - j0) / T) * C * 2
                        : nullptr;
        while (mask) {
          const int i = __ffs(mask) - 1;
          mask &= mask - 1;
          const float g = __uint_as_float(pick32(zg, i)), u = __uint_as_float(pick32(zu, i));
          sv[cnt] = float_to_bf16_bits(g * u);
          si[cnt] = static_cast<uint8_t>(j0 + i);
          if (gu) *reinterpret_cast<float2*>(gu + 2 * cnt) = make_float2(g, u);
          ++cnt;
        }
      } else {
        cnt += k;
      }
      if ((c + 32) % T != 0) continue;
      const int tile_c0 = c + 32 - T;
      const int t = (col0 + tile_c0) / T;
      const int64_t cell = static_cast<int64_t>(row) * p.n_tiles + t;
      const bool ovf = valid && cnt > C;
      if (valid && !ovf) {
        p.counts[cell] = static_cast<uint8_t>(cnt);
        if ((C & 7) == 0) {
          uint4* gv = reinterpret_cast<uint4*>(p.values + cell * C);
          uint2* gi = reinterpret_cast<uint2*>(p.idx + cell * C);
          for (int q = 0; q < C / 8; ++q) {
            gv[q] = reinterpret_cast<const uint4*>(sv)[q];
            gi[q] = reinterpret_cast<const uint2*>(si)[q];
          }
        } else {
          for (int q = 0; q < C; ++q) {
            p.values[cell * C + q] = sv[q];
            p.idx[cell * C + q] = si[q];
          }
        }
      }
      if (__any_sync(0xffffffffu, ovf)) {
        int slot = -1;
        if (ovf) {
          p.row_flag[row] = 1;
          slot = atomicAdd(p.spill_count, 1);
          if (slot >= p.spill_cap) {
            report_error(p.status, TWELL_ERR_FALLBACK_OVERFLOW);
            slot = -1;
          }
          p.counts[cell] = kSpilledCell;
          const uint32_t s24 = slot < 0 ? 0xFFFFFFu : static_cast<uint32_t>(slot);
          p.values[cell * C] = static_cast<uint16_t>(s24 & 0xFFFFu);
          p.idx[cell * C] = static_cast<uint8_t>(s24 >> 16);
        }
        for (int cc = tile_c0; cc < tile_c0 + T; cc += 32) {
          uint32_t hh[32];
          load_h32<BN>(p, taddr, col0, cc, hh);
          if (slot >= 0) {
            uint32_t packed[16];
#pragma unroll
            for (int i = 0; i < 32; i += 2)
              packed[i / 2] = static_cast<uint32_t>(float_to_bf16_bits(__uint_as_float(hh[i]))) |
                              (static_cast<uint32_t>(float_to_bf16_bits(__uint_as_float(hh[i + 1]))) << 16);
            uint4* dst = reinterpret_cast<uint4*>(p.spill + static_cast<int64_t>(slot) * T + (cc - tile_c0));
#pragma unroll
            for (int q = 0; q < 4; ++q)
              dst[q] = make_uint4(packed[4 * q], packed[4 * q + 1], packed[4 * q + 2], packed[4 * q + 3]);
          }
        }
      }
    }
  }
};

struct DenseEpi {
  static constexpr bool kDualB = false;
  using Params = DenseEpiParams;
  static constexpr uint32_t kSmemBytes = 0;

  template <int BN>
  static __device__ __forceinline__ void apply(const Params& p, uint32_t taddr, int row, int M, int col0, int half,
                                               int ks, uint8_t*, int) {
    (void)ks;
    const bool valid = row < M;
#pragma unroll 1
    for (int c = half * (BN / 64); c < (half + 1) * (BN / 64); ++c) {
      uint32_t r[32];
      tmem_ld32(taddr + c * 32, r);
      uint4 bq[4] = {};
      if (p.bias) {
        const uint4* bp = reinterpret_cast<const uint4*>(p.bias + col0 + c * 32);
#pragma unroll
        for (int q = 0; q < 4; ++q) bq[q] = __ldg(bp + q);
      }
      tmem_ld_wait();
      uint32_t packed[16];
#pragma unroll
      for (int i = 0; i < 32; i += 2) {
        float z0 = __uint_as_float(r[i]), z1 = __uint_as_float(r[i + 1]);
        if (p.bias) {
          z0 += bias_at(bq, i);
          z1 += bias_at(bq, i + 1);
        }
        if (p.relu) {
          z0 = z0 > 0.0f ? z0 : 0.0f;
          z1 = z1 > 0.0f ? z1 : 0.0f;
        }
        packed[i / 2] = static_cast<uint32_t>(float_to_bf16_bits(z0)) |
                        (static_cast<uint32_t>(float_to_bf16_bits(z1)) << 16);
      }
      if (valid) {
        uint4* dst = reinterpret_cast<uint4*>(p.out + static_cast<int64_t>(row) * p.ldo + col0 + c * 32);
#pragma unroll
        for (int q = 0; q < 4; ++q)
          dst[q] = make_uint4(packed[4 * q], packed[4 * q + 1], packed[4 * q + 2], packed[4 * q + 3]);
      }
    }
  }
};

// Dense comparator's backward through the ReLU and the L1 term: dZ = acc +
// lambda where the dense forward's h > 0, else 0, stored as bf16 rows.
struct MaskEpi {
  static constexpr bool kDualB = false;
  using Params = MaskEpiParams;
  static constexpr uint32_t kSmemBytes = 0;

  template <int BN>
  static __device__ __forceinline__ void apply(const Params& p, uint32_t taddr, int row, int M, int col0, int half,
                                               int, uint8_t*, int) {
    const bool valid = row < M;
#pragma unroll 1
    for (int c = half * (BN / 64); c < (half + 1) * (BN / 64); ++c) {
      uint32_t r[32];
      tmem_ld32(taddr + c * 32, r);
      uint4 hq[4] = {};
      if (valid) {
        const uint4* hp = reinterpret_cast<const uint4*>(p.H + static_cast<int64_t>(row) * p.ld + col0 + c * 32);
#pragma unroll
        for (int q = 0; q < 4; ++q) hq[q] = hp[q];
      }
      tmem_ld_wait();
      if (!valid) continue;
      uint32_t packed[16];
#pragma unroll
      for (int i = 0; i < 32; i += 2) {
        const float z0 = bias_at(hq, i) > 0.0f ? __uint_as_float(r[i]) + p.lambda : 0.0f;
        const float z1 = bias_at(hq, i + 1) > 0.0f ? __uint_as_float(r[i + 1]) + p.lambda : 0.0f;
        packed[i / 2] = static_cast<uint32_t>(float_to_bf16_bits(z0)) |
                        (static_cast<uint32_t>(float_to_bf16_bits(z1)) << 16);
      }
      uint4* dst = reinterpret_cast<uint4*>(p.out + static_cast<int64_t>(row) * p.ld + col0 + c * 32);
#pragma unroll
      for (int q = 0; q < 4; ++q)
        dst[q] = make_uint4(packed[4 * q], packed[4 * q + 1], packed[4 * q + 2], packed[4 * q + 3]);
    }
  }
};

// fp32 tile store.  Each warp turns its 32 rows x 32 columns around in shared
// memory so that its stores write whole 128-byte row segments, four rows per
// 16-byte-per-lane instruction.  The 16-byte chunks of a staged row are
// XOR-swizzled by the row (chunk k of row r sits at k ^ (r & 7)), so both the
// row-wise writes and the column-wise reads are free of bank conflicts.
struct PartialEpi {
  static constexpr bool kDualB = false;
  using Params = PartialEpiParams;
  static constexpr uint32_t kSmemBytes = (kEpiThreads / 32) * 32 * 32 * 4;

  template <int BN>
  static __device__ __forceinline__ void apply(const Params& p, uint32_t taddr, int row, int M, int col0, int half,
                                               int ks, uint8_t* smem, int et) {
    const int lane = threadIdx.x & 31;
    const int row0 = row - lane;  // first row of this warp's 32
    float* st = reinterpret_cast<float*>(smem) + (et >> 5) * 32 * 32;
    float* base = p.part + static_cast<int64_t>(ks) * p.split_stride + col0;
    const int k_rd = lane & 7;         // 16-byte chunk this lane reads / stores
    const int r_rd = lane >> 3;        // row within each group of four
#pragma unroll 1
    for (int c = half * (BN / 64); c < (half + 1) * (BN / 64); ++c) {
      uint32_t r[32];
      tmem_ld32(taddr + c * 32, r);
      tmem_ld_wait();
#pragma unroll
      for (int k = 0; k < 8; ++k)
        *reinterpret_cast<uint4*>(st + lane * 32 + 4 * (k ^ (lane & 7))) =
            make_uint4(r[4 * k], r[4 * k + 1], r[4 * k + 2], r[4 * k + 3]);
      __syncwarp();
#pragma unroll
      for (int g = 0; g < 8; ++g) {
        const int rr = 4 * g + r_rd;
        const uint4 v = *reinterpret_cast<const uint4*>(st + rr * 32 + 4 * (k_rd ^ (rr & 7)));
        if (row0 + rr < M)
          *reinterpret_cast<uint4*>(base + static_cast<int64_t>(row0 + rr) * p.ld + c * 32 + 4 * k_rd) = v;
      }
      __syncwarp();
    }
  }
};

// Swapped operands (small batches): accumulator rows are hidden units, the BN
// columns are tokens; each epilogue half stores BN/2 token columns of fp32
// partial sums, token-major so a warp's 32 units form one 128-byte run.
struct PartialTEpi {
  static constexpr bool kDualB = false;
  using Params = PartialTEpiParams;
  static constexpr uint32_t kSmemBytes = 0;

  template <int BN>
  static __device__ __forceinline__ void apply(const Params& p, uint32_t taddr, int row, int M, int col0, int half,
                                               int ks, uint8_t*, int) {
    static_assert(BN % 16 == 0 && BN <= 64, "narrow tiles only");
    float* base = p.part + static_cast<int64_t>(ks) * p.split_stride + row;
#pragma unroll
    for (int c = 0; c < BN / 2; c += 8) {
      uint32_t r[8];
      tmem_ld8(taddr + half * (BN / 2) + c, r);
      tmem_ld_wait();
      if (row < M) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int tok = col0 + half * (BN / 2) + c + i;
          if (tok < p.n_tok) base[static_cast<int64_t>(tok) * p.ld] = __uint_as_float(r[i]);
        }
      }
    }
  }
};

struct SampleEpi {
  static constexpr bool kDualB = false;
  using Params = SampleEpiParams;
  static constexpr uint32_t kSmemBytes = 0;

  template <int BN>
  static __device__ __forceinline__ void apply(const Params& p, uint32_t taddr, int row, int M, int col0, int half,
                                               int ks, uint8_t*, int) {
    (void)ks;
    const bool valid = row < M;
    const int fb = valid ? p.row_fb[row] : -1;
    const int T = p.tile, C = p.cap;
#pragma unroll 1
    for (int c = half * (BN / 64); c < (half + 1) * (BN / 64); ++c) {
      uint32_t r[32];
      tmem_ld32(taddr + c * 32, r);
      tmem_ld_wait();
      const int col = col0 + c * 32;
      if (!valid) continue;
      if (fb < 0) {
        // TwELL row: the stored entries of this chunk's tile that fall in it
        const int t = col / T;
        const int64_t cell = static_cast<int64_t>(row) * p.n_tiles + t;
        const int cnt = p.counts[cell];
        const int lo = col - t * T;
        for (int s = 0; s < cnt; ++s) {
          const int j = static_cast<int>(p.idx[cell * C + s]) - lo;
          if (j >= 0 && j < 32) {
            const float h = bf16_bits_to_float(p.values[cell * C + s]);
            const float dh = __uint_as_float(pick32(r, j));
            if (p.gu) {
              // gated: stored slots hold h != 0; (dG, dU) = (dh' u, dh' g)
              const float dhl = dh + (h > 0.0f ? p.lambda : -p.lambda);
              const float2 gv = *reinterpret_cast<const float2*>(p.gu + (cell * C + s) * 2);
              reinterpret_cast<float2*>(p.dz_cells)[cell * C + s] =
                  h != 0.0f ? make_float2(dhl * gv.y, dhl * gv.x) : make_float2(0.0f, 0.0f);
            } else {
              p.dz_cells[cell * C + s] = h > 0.0f ? dh + p.lambda : 0.0f;
            }
          }
        }
      } else if (fb < p.fb_cap && p.gu) {
        // gated fallback row: dense dh' (0 where h == 0); dG and dU are formed
        // once the fallback rows' g and u are in (a second stream computes them)
        const uint4* hp = reinterpret_cast<const uint4*>(p.fb_dense + static_cast<int64_t>(fb) * p.d_ff + col);
        uint4 hq[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) hq[q] = hp[q];
        float4* o = reinterpret_cast<float4*>(p.dh_fb + static_cast<int64_t>(fb) * p.d_ff + col);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          float v[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float h = bias_at(hq, 4 * q + e);
            v[e] = h != 0.0f ? __uint_as_float(r[4 * q + e]) + (h > 0.0f ? p.lambda : -p.lambda) : 0.0f;
          }
          o[q] = make_float4(v[0], v[1], v[2], v[3]);
        }
      } else if (fb < p.fb_cap) {
        // fallback row: dense dZ over all 32 columns
        const uint4* hp = reinterpret_cast<const uint4*>(p.fb_dense + static_cast<int64_t>(fb) * p.d_ff + col);
        uint4 hq[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) hq[q] = hp[q];
        uint32_t hi[16], lo[16];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          float o[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int i = 4 * q + e;
            const float h = bias_at(hq, i);
            o[e] = h > 0.0f ? __uint_as_float(r[i]) + p.lambda : 0.0f;
            // dz = hi + lo with both halves in bf16 (the fallback rows' dX runs
            // on the tensor cores as two bf16 products)
            const uint16_t hb = float_to_bf16_bits(o[e]);
            const uint16_t lb = float_to_bf16_bits(o[e] - bf16_bits_to_float(hb));
            if (i & 1) {
              hi[i / 2] |= static_cast<uint32_t>(hb) << 16;
              lo[i / 2] |= static_cast<uint32_t>(lb) << 16;
            } else {
              hi[i / 2] = hb;
              lo[i / 2] = lb;
            }
          }
        }
        uint4* dh = reinterpret_cast<uint4*>(p.dz_hl + static_cast<int64_t>(2 * fb) * p.d_ff + col);
        uint4* dl = reinterpret_cast<uint4*>(p.dz_hl + static_cast<int64_t>(2 * fb + 1) * p.d_ff + col);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          dh[q] = make_uint4(hi[4 * q], hi[4 * q + 1], hi[4 * q + 2], hi[4 * q + 3]);
          dl[q] = make_uint4(lo[4 * q], lo[4 * q + 1], lo[4 * q + 2], lo[4 * q + 3]);
        }
      }
    }
  }
};

// (g, u) of the gated layer's fallback rows (dual-B GEMM: the stage's two B
// halves are W_g and W_u rows of the same BN / 2 units): each epilogue thread
// writes its row's units of its half of the tile as (g + b, u) fp32 pairs.
struct GUEpi {
  static constexpr bool kDualB = true;
  using Params = GUEpiParams;
  static constexpr uint32_t kSmemBytes = 0;

  template <int BN>
  static __device__ __forceinline__ void apply(const Params& p, uint32_t taddr, int row, int M, int col0, int half,
                                               int, uint8_t*, int) {
    constexpr int U = BN / 2;
    const bool valid = row < M;
#pragma unroll 1
    for (int c = half * (U / 2); c < (half + 1) * (U / 2); c += 32) {
      uint32_t g[32], u[32];
      tmem_ld32(taddr + c, g);
      tmem_ld32(taddr + U + c, u);
      const uint4* bp = reinterpret_cast<const uint4*>(p.bias + col0 + c);
      uint4 bq[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) bq[q] = __ldg(bp + q);
      tmem_ld_wait();
      if (!valid) continue;
      float4* out = reinterpret_cast<float4*>(p.gu + (static_cast<int64_t>(row) * p.d_ff + col0 + c) * 2);
#pragma unroll
      for (int i = 0; i < 32; i += 2)
        out[i / 2] = make_float4(__uint_as_float(g[i]) + bias_at(bq, i), __uint_as_float(u[i]),
                                 __uint_as_float(g[i + 1]) + bias_at(bq, i + 1), __uint_as_float(u[i + 1]));
    }
  }
};

// ------------------------------------------------------------ kernel
template <int BN, class Epi, bool kANMajor, bool kBNMajor>
__global__ void __launch_bounds__(kThreads, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmB2, const GemmArgs args, const typename Epi::Params ep) {
  using Cfg = GemmCfg<BN>;
  constexpr int S = Cfg::kStages;
  static_assert(2 * S * 8 + 4 * 8 + 8 + 8 + S * 4 <= static_cast<int>(Cfg::kBarBytes), "barrier region");
  grid_dependency_wait();  // before the first read of device memory (M_dev, K_dev, operands)
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + S * Cfg::kABytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + Cfg::kPipeBytes);
  uint64_t* empty = full + S;
  uint64_t* tfull = empty + S;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_holder + 1);
  int* issued_parity = const_cast<int*>(abort) + 1;  // [S] parity of the last fill of each stage, -1 = none
  uint8_t* epi_smem = smem + Cfg::kPipeBytes + Cfg::kBarBytes;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  int M = args.M;
  if (args.M_dev) M = min(M, max(0, *args.M_dev));
  const int num_m = (M + kBM - 1) / kBM;
  // dual-B tiles cover BN/2 output units (gate and up halves of the B stage)
  constexpr int kUnitsPerTile = Epi::kDualB ? BN / 2 : BN;
  const int num_n = args.N / kUnitsPerTile;
  const int K = args.K_dev ? min(args.K, max(0, *args.K_dev) * args.k_mul) : args.K;
  const int num_k = (K + kBK - 1) / kBK;
  const int num_units = num_k > 0 ? num_m * num_n * args.ksplit : 0;
  // K split ks covers k-blocks [ks * num_k / ksplit, (ks + 1) * num_k / ksplit):
  // balanced, every split non-empty when ksplit <= num_k

  if (blockIdx.x == 0) {
    for (int i = threadIdx.x; i < args.n_zero0; i += blockDim.x) args.zero0[i] = 0;
    for (int i = threadIdx.x; i < args.n_zero1; i += blockDim.x) args.zero1[i] = 0;
  }
  // nothing to compute (e.g. no fallback rows this call): leave before setting
  // up barriers and TMEM (uniform over the CTA and the grid)
  if (num_units == 0) return;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
      issued_parity[s] = -1;
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], kEpiThreads);
    }
    mbar_init(drain, 1);
    *abort = 0;
    mbar_fence_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    if (Epi::kDualB) tma_prefetch_desc(&tmB2);
  }
  if (warp == 2) tmem_alloc(tmem_holder, Cfg::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  const uint64_t limit = args.wait_limit_ns;

  if (warp == 0) {
    if (lane == 0 && num_units > 0) {
      // ---------------- TMA producer
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < num_units; u += gridDim.x) {
        const int m_blk = u % num_m, rest = u / num_m;
        const int n_blk = rest % num_n, ks = rest / num_n;
        const int kb0 = ks * num_k / args.ksplit, kb1 = (ks + 1) * num_k / args.ksplit;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, limit, abort)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[stage], Cfg::kABytes + Cfg::kBBytes);
          if (kANMajor) {
            // A is [K][M]: two boxes of 64 M-columns x 64 K-rows, 8 KB apart
            tma_load_2d(sA + stage * Cfg::kABytes, &tmA, &full[stage], m_blk * kBM, kb * kBK);
            tma_load_2d(sA + stage * Cfg::kABytes + 8192, &tmA, &full[stage], m_blk * kBM + 64, kb * kBK);
          } else {
            tma_load_2d(sA + stage * Cfg::kABytes, &tmA, &full[stage], kb * kBK, m_blk * kBM);
          }
          if (Epi::kDualB) {
            // rows of the two B matrices for the same units stacked in one stage
            tma_load_2d(sB + stage * Cfg::kBBytes, &tmB, &full[stage], kb * kBK, n_blk * (BN / 2));
            tma_load_2d(sB + stage * Cfg::kBBytes + Cfg::kBBytes / 2, &tmB2, &full[stage], kb * kBK,
                        n_blk * (BN / 2));
          } else if (kBNMajor) {
            // B is [K][N]: BN/64 boxes of 64 N-columns x 64 K-rows, 8 KB apart
#pragma unroll
            for (int q = 0; q < BN / 64; ++q)
              tma_load_2d(sB + stage * Cfg::kBBytes + q * 8192, &tmB, &full[stage], n_blk * BN + q * 64,
                          args.b_k_wrap ? (kb * kBK) % args.b_k_wrap : kb * kBK);
          } else {
            tma_load_2d(sB + stage * Cfg::kBBytes, &tmB, &full[stage], kb * kBK, n_blk * BN);
          }
          issued_parity[stage] = static_cast<int>(phase);
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        report_error(args.status, TWELL_ERR_WAIT_TIMEOUT);
        // let the copies already in flight land before the CTA leaves
        for (int s = 0; s < S; ++s) {
          if (issued_parity[s] >= 0) {
            volatile int never = 0;
            mbar_wait(&full[s], static_cast<uint32_t>(issued_parity[s]), 10000000ull, &never);
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && num_units > 0) {
      // ---------------- MMA issuer
      constexpr uint32_t idesc =
          idesc_bf16_f32(kBM, BN) | (kANMajor ? (1u << 15) : 0u) | (kBNMajor ? (1u << 16) : 0u);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < num_units; u += gridDim.x) {
        const int ks = (u / num_m) / num_n;
        const int kb0 = ks * num_k / args.ksplit, kb1 = (ks + 1) * num_k / args.ksplit;
        if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, limit, abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(&full[stage], phase, limit, abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t adesc = kANMajor ? smem_desc_sw128_nmajor(smem_u32(sA + stage * Cfg::kABytes), 8192)
                                          : smem_desc_sw128(smem_u32(sA + stage * Cfg::kABytes));
          const uint64_t bdesc = kBNMajor ? smem_desc_sw128_nmajor(smem_u32(sB + stage * Cfg::kBBytes), 8192)
                                          : smem_desc_sw128(smem_u32(sB + stage * Cfg::kBBytes));
#pragma unroll
          for (int k = 0; k < kBK / kUmmaK; ++k) {
            // K step of 16: +32 B along a K-major row, or +16 rows (2 KB) of an N-major tile
            const uint64_t a_step = kANMajor ? 128u * k : 2u * k;
            const uint64_t b_step = kBNMajor ? 128u * k : 2u * k;
            mma_bf16(d_tmem, adesc + a_step, bdesc + b_step, idesc, (kb > kb0 || k > 0) ? 1u : 0u);
          }
          mma_commit(&empty[stage]);
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit(&tfull[acc]);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      if (!ok) {
        report_error(args.status, TWELL_ERR_WAIT_TIMEOUT);
        // wait for the MMAs already issued before TMEM is released
        mma_commit(drain);
        volatile int never = 0;
        mbar_wait(drain, 0, 10000000ull, &never);
      }
    }
  } else if (warp >= 4) {
    // ---------------- epilogue
    const int lg = warp & 3;              // TMEM lane quarter
    const int half = (warp - 4) >> 2;     // column half of the tile
    const int et = threadIdx.x - 128;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int u = blockIdx.x; u < num_units; u += gridDim.x) {
      const int m_blk = u % num_m, rest = u / num_m;
      const int n_blk = rest % num_n, ks = rest / num_n;
      if (!mbar_wait(&tfull[acc], acc_phase, limit, abort)) {
        report_error(args.status, TWELL_ERR_WAIT_TIMEOUT);
        break;
      }
      tc_fence_after();
      const int row = m_blk * kBM + lg * 32 + lane;
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(lg * 32) << 16) + static_cast<uint32_t>(acc * BN);
      Epi::template apply<BN>(ep, taddr, row, M, n_blk * kUnitsPerTile, half, ks, epi_smem, et);
      tc_fence_before();
      mbar_arrive(&tempty[acc]);
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem_base, Cfg::kTmemCols);
  }
}

template <int BN, class Epi, bool kANMajor, bool kBNMajor>
int launch_gemm(const uint16_t* A, const uint16_t* B, int M, const int32_t* M_dev, int N, int K, int ksplit,
                const typename Epi::Params& p, int32_t* status, int kernel_id, cudaStream_t s,
                const int32_t* K_dev = nullptr, int k_mul = 1, int64_t lda = 0, const uint16_t* B2 = nullptr,
                int b_rows = 0, int32_t* zero0 = nullptr, int n_zero0 = 0, int32_t* zero1 = nullptr,
                int n_zero1 = 0, int b_k_wrap = 0) {
  using Cfg = GemmCfg<BN>;
  if (M <= 0 || N <= 0 || K <= 0) return TWELL_OK;
  const int num_k = (K + kBK - 1) / kBK;
  if (ksplit < 1 || ksplit > num_k) return TWELL_ERR_UNSUPPORTED;
  if (K_dev && ksplit > 1) return TWELL_ERR_UNSUPPORTED;  // a device-side K could leave a split empty
  CUtensorMap ta, tb, tb2;
  int rc;
  if (kANMajor)
    rc = encode_tmap_2d(&ta, A, static_cast<uint64_t>(M), static_cast<uint64_t>(K),
                        static_cast<uint64_t>(lda ? lda : M) * 2, 64, kBK);
  else
    rc = encode_tmap_2d(&ta, A, static_cast<uint64_t>(K), static_cast<uint64_t>(M),
                        static_cast<uint64_t>(lda ? lda : K) * 2, kBK, kBM);
  if (rc) return rc;
  if (Epi::kDualB) {
    if (!B2) return TWELL_ERR_INVALID_ARG;
    rc = encode_tmap_2d(&tb, B, static_cast<uint64_t>(K), static_cast<uint64_t>(N), static_cast<uint64_t>(K) * 2, kBK,
                        BN / 2);
    if (rc) return rc;
    rc = encode_tmap_2d(&tb2, B2, static_cast<uint64_t>(K), static_cast<uint64_t>(N), static_cast<uint64_t>(K) * 2,
                        kBK, BN / 2);
  } else if (kBNMajor) {
    if (b_k_wrap % kBK != 0 || b_k_wrap < 0) return TWELL_ERR_UNSUPPORTED;
    rc = encode_tmap_2d(&tb, B, static_cast<uint64_t>(N), static_cast<uint64_t>(b_k_wrap ? b_k_wrap : K),
                        static_cast<uint64_t>(N) * 2, 64, kBK);
  } else {
    // b_rows < N: the rows past b_rows are read as zeros (TMA fill)
    rc = encode_tmap_2d(&tb, B, static_cast<uint64_t>(K), static_cast<uint64_t>(b_rows > 0 ? b_rows : N),
                        static_cast<uint64_t>(K) * 2, kBK, BN);
  }
  if (rc) return rc;
  if (!Epi::kDualB) tb2 = tb;
  const uint32_t smem = 1024 + Cfg::kPipeBytes + Cfg::kBarBytes + Epi::kSmemBytes;
  auto kern = tc_gemm_kernel<BN, Epi, kANMajor, kBNMajor>;
  rc = set_max_dynamic_smem(reinterpret_cast<const void*>(kern), static_cast<int>(smem));
  if (rc) return rc;
  const int units = ((M + kBM - 1) / kBM) * (N / (Epi::kDualB ? BN / 2 : BN)) * ksplit;
  const int grid = std::max(1, std::min(units, sm_count()));
  GemmArgs args{M,      M_dev,        N,     K,       ksplit, K_dev, k_mul, status, kWaitLimitNs,
                zero0,  zero0 ? n_zero0 : 0, zero1, zero1 ? n_zero1 : 0, b_k_wrap};
  {
    LaunchScope ls(kernel_id, s);
    if (launch_pdl(kern, dim3(grid), dim3(kThreads), smem, s, ta, tb, tb2, args, p) != cudaSuccess) {
      cudaGetLastError();
      return TWELL_ERR_CUDA;
    }
  }
  return cudaGetLastError() == cudaSuccess ? TWELL_OK : TWELL_ERR_CUDA;
}

}  // namespace

int launch_gemm_pack(const uint16_t* A, const uint16_t* B, int M, int N, int K, const PackEpiParams& p,
                     int32_t* status, cudaStream_t s) {
  if (p.cap > PackEpi::kMaxCap) return TWELL_ERR_UNSUPPORTED;
  if (N % 256 == 0)
    return launch_gemm<256, PackEpi, false, false>(A, B, M, nullptr, N, K, 1, p, status, TWELL_KERNEL_UP_PACK, s);
  if (N % 128 == 0 && p.tile <= 128)
    return launch_gemm<128, PackEpi, false, false>(A, B, M, nullptr, N, K, 1, p, status, TWELL_KERNEL_UP_PACK, s);
  return TWELL_ERR_UNSUPPORTED;
}

int launch_gemm_dense(const uint16_t* A, const uint16_t* B, bool b_n_major, int M, const int32_t* M_dev, int N,
                      int K, const DenseEpiParams& p, int32_t* status, int kernel_id, cudaStream_t s) {
  if (b_n_major) {
    if (N % 256 == 0) return launch_gemm<256, DenseEpi, false, true>(A, B, M, M_dev, N, K, 1, p, status, kernel_id, s);
    if (N % 128 == 0) return launch_gemm<128, DenseEpi, false, true>(A, B, M, M_dev, N, K, 1, p, status, kernel_id, s);
    return TWELL_ERR_UNSUPPORTED;
  }
  if (N % 256 == 0) return launch_gemm<256, DenseEpi, false, false>(A, B, M, M_dev, N, K, 1, p, status, kernel_id, s);
  if (N % 128 == 0) return launch_gemm<128, DenseEpi, false, false>(A, B, M, M_dev, N, K, 1, p, status, kernel_id, s);
  return TWELL_ERR_UNSUPPORTED;
}

int choose_fb_ksplit(int K, int max_split) {
  const int num_k = (K + kBK - 1) / kBK;
  return std::max(1, std::min(max_split, num_k));
}

int swap_ksplit(int K) { return choose_fb_ksplit(K, 8); }

int launch_gemm_swap_partial(const uint16_t* W, const uint16_t* X, int M, int n_tok, int K, int ksplit,
                             const PartialTEpiParams& p, int32_t* status, int kernel_id, cudaStream_t s,
                             int32_t* zero0, int n_zero0, int32_t* zero1, int n_zero1) {
  if (n_tok <= 0) return TWELL_OK;
  if (n_tok > kSwapMaxTokens || M % kBM != 0 || K <= 0) return TWELL_ERR_UNSUPPORTED;
  if (n_tok <= 16)
    return launch_gemm<16, PartialTEpi, false, false>(W, X, M, nullptr, 16, K, ksplit, p, status, kernel_id, s,
                                                      nullptr, 1, 0, nullptr, n_tok, zero0, n_zero0, zero1, n_zero1);
  return launch_gemm<32, PartialTEpi, false, false>(W, X, M, nullptr, 32, K, ksplit, p, status, kernel_id, s, nullptr,
                                                    1, 0, nullptr, n_tok, zero0, n_zero0, zero1, n_zero1);
}

int launch_gemm_partial_nmajor(const uint16_t* A, const uint16_t* B, int M, const int32_t* M_dev, int N, int K,
                               int ksplit, const PartialEpiParams& p, int32_t* status, int kernel_id,
                               cudaStream_t s, int64_t lda, int b_k_wrap) {
  if (N % 128 != 0) return TWELL_ERR_UNSUPPORTED;
  return launch_gemm<128, PartialEpi, false, true>(A, B, M, M_dev, N, K, ksplit, p, status, kernel_id, s, nullptr, 1,
                                                   lda, nullptr, 0, nullptr, 0, nullptr, 0, b_k_wrap);
}

int launch_gemm_gated_pack(const uint16_t* A, const uint16_t* Bg, const uint16_t* Bu, int M, int N, int K,
                           const PackEpiParams& p, int32_t* status, cudaStream_t s) {
  if (p.cap > GatedPackEpi::kMaxCap || N % 128 != 0 || 128 % p.tile != 0) return TWELL_ERR_UNSUPPORTED;
  return launch_gemm<256, GatedPackEpi, false, false>(A, Bg, M, nullptr, N, K, 1, p, status, TWELL_KERNEL_UP_PACK, s,
                                                      nullptr, 1, 0, Bu);
}

int launch_gemm_gu(const uint16_t* A, int64_t lda, const uint16_t* Bg, const uint16_t* Bu, int M, const int32_t* M_dev,
                   int N, int K, const GUEpiParams& p, int32_t* status, int kernel_id, cudaStream_t s) {
  if (N % 128 != 0) return TWELL_ERR_UNSUPPORTED;
  return launch_gemm<256, GUEpi, false, false>(A, Bg, M, M_dev, N, K, 1, p, status, kernel_id, s, nullptr, 1, lda,
                                               Bu);
}

int launch_gemm_mask(const uint16_t* A, const uint16_t* B, int M, int N, int K, const MaskEpiParams& p,
                     int32_t* status, int kernel_id, cudaStream_t s) {
  if (N % 256 == 0) return launch_gemm<256, MaskEpi, false, false>(A, B, M, nullptr, N, K, 1, p, status, kernel_id, s);
  if (N % 128 == 0) return launch_gemm<128, MaskEpi, false, false>(A, B, M, nullptr, N, K, 1, p, status, kernel_id, s);
  return TWELL_ERR_UNSUPPORTED;
}

int launch_gemm_store_mn(const uint16_t* A, const uint16_t* B, int M, int N, int K, const int32_t* K_dev, int k_mul,
                         float* out, int64_t ld, int32_t* status, int kernel_id, cudaStream_t s) {
  if (M % 128 != 0 || N % 128 != 0) return TWELL_ERR_UNSUPPORTED;
  PartialEpiParams p{out, ld, 0};
  if (N % 256 == 0)
    return launch_gemm<256, PartialEpi, true, true>(A, B, M, nullptr, N, K, 1, p, status, kernel_id, s, K_dev, k_mul);
  return launch_gemm<128, PartialEpi, true, true>(A, B, M, nullptr, N, K, 1, p, status, kernel_id, s, K_dev, k_mul);
}

int launch_gemm_sample(const uint16_t* A, const uint16_t* B, int M, int N, int K, const SampleEpiParams& p,
                       int32_t* status, cudaStream_t s, int32_t* zero, int n_zero) {
  const int nz = zero ? n_zero : 0;
  if (N % 256 == 0)
    return launch_gemm<256, SampleEpi, false, false>(A, B, M, nullptr, N, K, 1, p, status, TWELL_KERNEL_SDDMM, s,
                                                     nullptr, 1, 0, nullptr, 0, zero, nz);
  if (N % 128 == 0)
    return launch_gemm<128, SampleEpi, false, false>(A, B, M, nullptr, N, K, 1, p, status, TWELL_KERNEL_SDDMM, s,
                                                     nullptr, 1, 0, nullptr, 0, zero, nz);
  return TWELL_ERR_UNSUPPORTED;
}

}  // namespace twell
