// Persistent warp-specialised bf16 GEMM on the 5th-generation tensor cores
// (tcgen05 + TMEM), fed by TMA, with two epilogues:
//   * PackEpi: z = acc + b, h = bf16(z) where z > 0, compaction of each
//     (row, T-column tile) into TwELL cells (values, tile-local indices,
//     count) and a per-row overflow flag -- the up-projection of the sparse
//     layer with its pack fused in (the pages' "fused MLP execution" and
//     "dense-to-TwELL" paths, repo-explainer "TwELL: The Packing Format...").
//   * DenseEpi: bf16 rows with optional bias and ReLU (dense fallback rows,
//     dense comparator).
//
// C[M, N] = A[M, K] . B[N, K]^T, A and B row-major bf16 (both K-major).
// CTA tile 128 x BN, K step 64, one CTA per SM, tiles strided over CTAs.
// Warp roles: 0 = TMA producer, 1 = MMA issuer, 2 = TMEM owner, 4..7 =
// epilogue (warp 4+i reads TMEM lanes 32i..32i+31, i.e. tile rows 32i..).
// Accumulators are double-buffered in TMEM so the epilogue of one tile runs
// under the MMAs of the next.
#include <cuda_runtime.h>

#include <algorithm>

#include "sm103.cuh"
#include "twell_internal.h"

namespace twell {
namespace {

constexpr int kBM = 128;
constexpr int kBK = 64;
constexpr int kUmmaK = 16;
constexpr int kThreads = 256;

template <int BN>
struct GemmCfg {
  static constexpr int kStages = BN == 256 ? 4 : 6;
  static constexpr uint32_t kABytes = kBM * kBK * 2;
  static constexpr uint32_t kBBytes = BN * kBK * 2;
  static constexpr uint32_t kTmemCols = 2 * BN;  // two accumulators
  static constexpr uint32_t kPipeBytes = kStages * (kABytes + kBBytes);
  static constexpr uint32_t kBarBytes = 256;
};

struct GemmArgs {
  int M;
  const int32_t* M_dev;  // optional device-side row count (clamped to M)
  int N;
  int K;
  int32_t* status;
  uint64_t wait_limit_ns;
};

// ------------------------------------------------------------ epilogues
struct PackEpi {
  using Params = PackEpiParams;
  static constexpr int kMaxCap = 32;
  static constexpr uint32_t kSmemBytes = 128 * kMaxCap * 3;  // per thread: C values (u16) + C indices (u8)

  // One thread = one accumulator row; processes columns [col0, col0 + BN).
  template <int BN>
  static __device__ __forceinline__ void apply(const Params& p, uint32_t taddr, int row, int M, int col0,
                                               uint8_t* smem, int et) {
    uint16_t* sv = reinterpret_cast<uint16_t*>(smem) + et * kMaxCap;
    uint8_t* si = smem + 128 * kMaxCap * 2 + et * kMaxCap;
    const int T = p.tile, C = p.cap;
    const bool valid = row < M;
    int cnt = 0;
#pragma unroll 1
    for (int c = 0; c < BN / 32; ++c) {
      uint32_t r[32];
      tmem_ld32(taddr + c * 32, r);
      const uint4* bp = reinterpret_cast<const uint4*>(p.bias + col0 + c * 32);
      uint4 bq[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) bq[q] = __ldg(bp + q);
      tmem_ld_wait();
      const int j0 = (c * 32) % T;
      if (j0 == 0) {
        cnt = 0;
        uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int q = 0; q < kMaxCap * 2 / 16; ++q) reinterpret_cast<uint4*>(sv)[q] = z;
#pragma unroll
        for (int q = 0; q < kMaxCap / 16; ++q) reinterpret_cast<uint4*>(si)[q] = z;
      }
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const uint32_t bw = (&bq[i / 8].x)[(i % 8) / 2];
        const float bias = (i & 1) ? bf16_hi(bw) : bf16_lo(bw);
        const float z = __uint_as_float(r[i]) + bias;
        if (z > 0.0f) {
          const uint16_t h = float_to_bf16_bits(z);
          if (h != 0) {
            if (cnt < C) {
              sv[cnt] = h;
              si[cnt] = static_cast<uint8_t>(j0 + i);
            }
            ++cnt;
          }
        }
      }
      if (((c + 1) * 32) % T == 0 && valid) {
        const int t = (col0 + c * 32) / T;
        const int64_t cell = static_cast<int64_t>(row) * p.n_tiles + t;
        p.counts[cell] = static_cast<uint8_t>(cnt < C ? cnt : C);
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
        if (cnt > C) p.row_flag[row] = 1;
      }
    }
  }
};

struct DenseEpi {
  using Params = DenseEpiParams;
  static constexpr uint32_t kSmemBytes = 0;

  template <int BN>
  static __device__ __forceinline__ void apply(const Params& p, uint32_t taddr, int row, int M, int col0,
                                               uint8_t*, int) {
    const bool valid = row < M;
#pragma unroll 1
    for (int c = 0; c < BN / 32; ++c) {
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
          const uint32_t bw = (&bq[i / 8].x)[(i % 8) / 2];
          z0 += bf16_lo(bw);
          z1 += bf16_hi(bw);
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

// ------------------------------------------------------------ kernel
template <int BN, class Epi>
__global__ void __launch_bounds__(kThreads, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const GemmArgs args, const typename Epi::Params ep) {
  using Cfg = GemmCfg<BN>;
  constexpr int S = Cfg::kStages;
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
  const int num_n = args.N / BN;
  const int num_tiles = num_m * num_n;
  const int num_k = (args.K + kBK - 1) / kBK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
      issued_parity[s] = -1;
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 128);
    }
    mbar_init(drain, 1);
    *abort = 0;
    mbar_fence_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 2) tmem_alloc(tmem_holder, Cfg::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  const uint64_t limit = args.wait_limit_ns;

  if (warp == 0) {
    if (lane == 0 && num_tiles > 0) {
      // ---------------- TMA producer
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
        const int m_blk = tile % num_m, n_blk = tile / num_m;
        for (int kb = 0; kb < num_k; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, limit, abort)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[stage], Cfg::kABytes + Cfg::kBBytes);
          tma_load_2d(sA + stage * Cfg::kABytes, &tmA, &full[stage], kb * kBK, m_blk * kBM);
          tma_load_2d(sB + stage * Cfg::kBBytes, &tmB, &full[stage], kb * kBK, n_blk * BN);
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
    if (lane == 0 && num_tiles > 0) {
      // ---------------- MMA issuer
      constexpr uint32_t idesc = idesc_bf16_f32(kBM, BN);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
        if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, limit, abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        for (int kb = 0; kb < num_k; ++kb) {
          if (!mbar_wait(&full[stage], phase, limit, abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t adesc = smem_desc_sw128(smem_u32(sA + stage * Cfg::kABytes));
          const uint64_t bdesc = smem_desc_sw128(smem_u32(sB + stage * Cfg::kBBytes));
#pragma unroll
          for (int k = 0; k < kBK / kUmmaK; ++k) {
            // +32 B per K step of 16 bf16, in 16-byte descriptor units
            mma_bf16(d_tmem, adesc + 2u * k, bdesc + 2u * k, idesc, (kb | k) != 0 ? 1u : 0u);
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
    const int lg = warp & 3;
    const int et = threadIdx.x - 128;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
      const int m_blk = tile % num_m, n_blk = tile / num_m;
      if (!mbar_wait(&tfull[acc], acc_phase, limit, abort)) {
        report_error(args.status, TWELL_ERR_WAIT_TIMEOUT);
        break;
      }
      tc_fence_after();
      const int row = m_blk * kBM + lg * 32 + lane;
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(lg * 32) << 16) + static_cast<uint32_t>(acc * BN);
      Epi::template apply<BN>(ep, taddr, row, M, n_blk * BN, epi_smem, et);
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

template <int BN, class Epi>
int launch_gemm(const uint16_t* A, const uint16_t* B, int M, const int32_t* M_dev, int N, int K,
                const typename Epi::Params& p, int32_t* status, int kernel_id, cudaStream_t s) {
  using Cfg = GemmCfg<BN>;
  if (M <= 0 || N <= 0 || K <= 0) return TWELL_OK;
  CUtensorMap ta, tb;
  int rc = encode_tmap_2d(&ta, A, static_cast<uint64_t>(K), static_cast<uint64_t>(M), static_cast<uint64_t>(K) * 2,
                          kBK, kBM);
  if (rc) return rc;
  rc = encode_tmap_2d(&tb, B, static_cast<uint64_t>(K), static_cast<uint64_t>(N), static_cast<uint64_t>(K) * 2, kBK,
                      BN);
  if (rc) return rc;
  const uint32_t smem = 1024 + Cfg::kPipeBytes + Cfg::kBarBytes + Epi::kSmemBytes;
  auto kern = tc_gemm_kernel<BN, Epi>;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
      return TWELL_ERR_CUDA;
    attr_set[dev] = true;
  }
  const int tiles = ((M + kBM - 1) / kBM) * (N / BN);
  const int grid = std::max(1, std::min(tiles, sm_count()));
  GemmArgs args{M, M_dev, N, K, status, kWaitLimitNs};
  {
    LaunchScope ls(kernel_id, s);
    kern<<<grid, kThreads, smem, s>>>(ta, tb, args, p);
  }
  return cudaGetLastError() == cudaSuccess ? TWELL_OK : TWELL_ERR_CUDA;
}

}  // namespace

int launch_gemm_pack(const uint16_t* A, const uint16_t* B, int M, const int32_t* M_dev, int N, int K,
                     const PackEpiParams& p, int32_t* status, cudaStream_t s) {
  if (p.cap > PackEpi::kMaxCap) return TWELL_ERR_UNSUPPORTED;
  if (N % 256 == 0) return launch_gemm<256, PackEpi>(A, B, M, M_dev, N, K, p, status, TWELL_KERNEL_UP_PACK, s);
  if (N % 128 == 0 && p.tile <= 128)
    return launch_gemm<128, PackEpi>(A, B, M, M_dev, N, K, p, status, TWELL_KERNEL_UP_PACK, s);
  return TWELL_ERR_UNSUPPORTED;
}

int launch_gemm_dense(const uint16_t* A, const uint16_t* B, int M, const int32_t* M_dev, int N, int K,
                      const DenseEpiParams& p, int32_t* status, int kernel_id, cudaStream_t s) {
  if (N % 256 == 0) return launch_gemm<256, DenseEpi>(A, B, M, M_dev, N, K, p, status, kernel_id, s);
  if (N % 128 == 0) return launch_gemm<128, DenseEpi>(A, B, M, M_dev, N, K, p, status, kernel_id, s);
  return TWELL_ERR_UNSUPPORTED;
}

}  // namespace twell
