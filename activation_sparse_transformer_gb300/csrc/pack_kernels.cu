// Standalone dense <-> TwELL conversions (the pages' "dense-to-TwELL and
// TwELL-to-dense paths", repo-explainer "TwELL: The Packing Format That Fits
// the Machine"; format per the bayesiansapien note's Figure 1 description).
//
// pack_cells_kernel: a warp reads 4 x 256 consecutive bf16 of one row with
//   16-byte loads (8 columns per lane, all loads issued first); per 256
//   columns the T/8 lanes of each tile compact their non-zeros with a
//   segmented popcount prefix into a shared-memory copy of the cells
//   (ascending column order), which one lane per cell writes out with the
//   padding, in whole vectors; it stores the count and flags the row
//   (row_fb = 1) when a tile overflows C.
// fb_copy_kernel: dense rows of fallback rows -> fb_dense, their cells cleared.
// unpack_run_kernel: a warp builds a 2048-column run of a row in shared
//   memory (zeros, then the cells' entries or dense tiles) and writes it out
//   with coalesced 16-byte stores (a fallback row is copied whole).
// check_cells_kernel / check_order_kernel: the format rules of a layout
//   (cell contents, then the numbering of fallback rows or dense tiles),
//   reported as a mask of broken rules.
#include <cuda_runtime.h>

#include <algorithm>

#include "sm103.cuh"
#include "twell_internal.h"

namespace twell {
namespace {

struct Layout {
  int32_t N, f, T, C, fb_cap, nt, hybrid;
  uint16_t* values;
  uint8_t* idx;
  uint8_t* counts;
  int32_t* row_fb;
  int32_t* fb_rows;
  uint16_t* fb_dense;
  int32_t* n_fb;
  int32_t* status;
};

Layout flat(const twell_t& L) {
  return Layout{L.n_rows, L.d_ff, L.tile, L.cap, L.fb_cap, L.d_ff / L.tile, L.hybrid, L.values, L.idx,
                L.counts, L.row_fb, L.fb_rows, L.fb_dense, L.n_fb, L.status};
}

constexpr int kWarps = 8;

__device__ __forceinline__ uint16_t half_word(const uint32_t (&w)[4], int k) {
  return static_cast<uint16_t>((k & 1) ? (w[k / 2] >> 16) : (w[k / 2] & 0xFFFFu));
}

// Compaction of 8 consecutive columns [col, col + 8) of one row per lane (a
// warp covers 256 columns); w holds the 8 bf16 values.  Called by all lanes.
__device__ __forceinline__ void pack_lane8(const Layout& L, int row, int col, bool in, const uint32_t (&w)[4]) {
  const int lane = threadIdx.x & 31;
  uint32_t nzmask = 0;
#pragma unroll
  for (int k = 0; k < 8; ++k)
    if ((half_word(w, k) & 0x7FFFu) != 0) nzmask |= 1u << k;  // +0 and -0 are zeros
  const int G = L.T / 8;  // lanes per tile: 4, 8, 16 or 32
  const int gl = lane % G;
  const int local = __popc(nzmask);
  int incl = local;
  for (int o = 1; o < G; o <<= 1) {
    const int x = __shfl_up_sync(0xffffffffu, incl, o);
    if (gl >= o) incl += x;
  }
  const int total = __shfl_sync(0xffffffffu, incl, (lane / G) * G + G - 1);
  if (!in) return;
  const int C = L.C;
  const int64_t cell = static_cast<int64_t>(row) * L.nt + col / L.T;
  // tile-granular hybrid: an over-full tile becomes a dense tile (its pool
  // slot is written into the cell once all rows are counted)
  const bool dense = L.hybrid == TWELL_HYBRID_TILES && total > C;
  int slot = incl - local;
  if (!dense) {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      if ((nzmask >> k) & 1u) {
        if (slot < C) {
          L.values[cell * C + slot] = half_word(w, k);
          L.idx[cell * C + slot] = static_cast<uint8_t>(gl * 8 + k);
        }
        ++slot;
      }
    }
  }
  const int stored = dense ? 0 : (total < C ? total : C);
  for (int s = stored + gl; s < C; s += G) {
    L.values[cell * C + s] = 0;
    L.idx[cell * C + s] = 0;
  }
  if (gl == 0) {
    L.counts[cell] = dense ? static_cast<uint8_t>(TWELL_DENSE_TILE) : static_cast<uint8_t>(stored);
    if (total > C) L.row_fb[row] = 1;
  }
}

// Dense -> cells.  A warp takes kPackSeg consecutive 256-column segments of
// one row and requests all of them (16 bytes per lane and segment) before it
// uses any, so each warp has 2 KB of H in flight.  Per segment, each lane
// finds the non-zeros of its 8 columns with branch-free bit arithmetic, the
// T/8 lanes of each tile take a segmented popcount prefix, and the lanes that
// hold non-zeros write them (in ascending column order) into the warp's
// staging copy of its cells in shared memory, one area per segment, so a
// single warp barrier follows all segments.  One lane per cell then writes
// the cell out: its first count slots from the staging copy and padding in
// the rest, as 16- and 8-byte vectors when C is a multiple of 8.
constexpr int kPackSeg = 4;
constexpr int kPackCells = kPackSeg * (256 / 32);   // the most cells a warp's chunk holds (T = 32)
constexpr int kPackStage = kPackCells * 32;         // x the largest C

// Non-zero pattern of the 8 bf16 values of one lane: bit 15 / bit 31 of word q
// is set when value 2q / 2q + 1 is not +-0.
__device__ __forceinline__ void nonzero_halves(const uint4& v, uint32_t (&t)[4]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) t[q] = ((w[q] & 0x7FFF7FFFu) + 0x7FFF7FFFu) & 0x80008000u;
}

template <int T>
__global__ void __launch_bounds__(kWarps * 32, 6)
    pack_cells_kernel(Layout L, const uint16_t* __restrict__ H, int64_t ldh) {
  __shared__ __align__(16) uint16_t st_vals[kWarps][kPackStage];
  __shared__ __align__(16) uint8_t st_idx[kWarps][kPackStage];
  __shared__ int st_cnt[kWarps][kPackCells];  // entries found per cell (may exceed C)
  constexpr int G = T / 8;                    // lanes per tile: 4, 8, 16 or 32
  constexpr int cps = 256 / T;                // cells per segment
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int chunk_cols = kPackSeg * 256;
  const int chunks = (L.f + chunk_cols - 1) / chunk_cols;
  const int64_t gw = static_cast<int64_t>(blockIdx.x) * kWarps + warp;
  if (gw >= static_cast<int64_t>(L.N) * chunks) return;  // whole warp leaves together
  const int row = static_cast<int>(gw / chunks);
  const int c0 = static_cast<int>(gw % chunks) * chunk_cols;
  const uint16_t* hrow = H + static_cast<int64_t>(row) * ldh;
  uint4 v[kPackSeg];
#pragma unroll
  for (int sg = 0; sg < kPackSeg; ++sg) {
    const int col = c0 + sg * 256 + lane * 8;
    v[sg] = col < L.f ? __ldg(reinterpret_cast<const uint4*>(hrow + col)) : make_uint4(0, 0, 0, 0);
  }
  const int C = L.C;
  const int gl = lane % G;
  uint16_t* sv = st_vals[warp];
  uint8_t* si = st_idx[warp];
  int* sc = st_cnt[warp];
  const int ncell = min(chunk_cols, L.f - c0) / T;  // cells of this chunk (f % T == 0)
#pragma unroll
  for (int sg = 0; sg < kPackSeg; ++sg) {
    uint32_t t[4];
    nonzero_halves(v[sg], t);
    const int local = __popc(t[0]) + __popc(t[1]) + __popc(t[2]) + __popc(t[3]);
    int incl = local;
#pragma unroll
    for (int o = 1; o < G; o <<= 1) {
      const int x = __shfl_up_sync(0xffffffffu, incl, o);
      if (gl >= o) incl += x;
    }
    const int cell = sg * cps + lane / G;  // the lane's cell within the chunk
    if (gl == G - 1 && cell < ncell) sc[cell] = incl;
    // this lane's non-zeros in ascending column (half h of word q is column
    // 2q + h), each to the next slot while slots remain.  At the layer's
    // sparsity most lanes hold none, so only words with a non-zero half are
    // visited.
    if (local) {
      const uint32_t w[4] = {v[sg].x, v[sg].y, v[sg].z, v[sg].w};
      uint16_t* cv = sv + cell * C;
      uint8_t* ci = si + cell * C;
      int slot = incl - local;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        if (t[q] == 0u) continue;
        if (t[q] & 0x8000u) {
          if (slot < C) {
            cv[slot] = static_cast<uint16_t>(w[q] & 0xFFFFu);
            ci[slot] = static_cast<uint8_t>(gl * 8 + 2 * q);
          }
          ++slot;
        }
        if (t[q] & 0x80000000u) {
          if (slot < C) {
            cv[slot] = static_cast<uint16_t>(w[q] >> 16);
            ci[slot] = static_cast<uint8_t>(gl * 8 + 2 * q + 1);
          }
          ++slot;
        }
      }
    }
  }
  __syncwarp();
  // one lane per cell writes it out; rows with an over-full tile are flagged
  const int64_t gcell0 = static_cast<int64_t>(row) * L.nt + c0 / T;
  bool over = false;
  for (int c = lane; c < ncell; c += 32) {
    const int found = sc[c];
    over |= found > C;
    const bool dense = L.hybrid == TWELL_HYBRID_TILES && found > C;
    const int cnt = dense ? 0 : min(found, C);
    const int64_t g = gcell0 + c;
    if ((C & 7) == 0) {
      for (int q = 0; q < C / 8; ++q) {
        // keep the first cnt - 8q slots of this 8-slot chunk, pad the rest
        const int keep = min(max(cnt - 8 * q, 0), 8);
        const uint4 sv4 = reinterpret_cast<const uint4*>(sv + c * C)[q];
        const uint2 si2 = reinterpret_cast<const uint2*>(si + c * C)[q];
        const uint32_t vw[4] = {sv4.x, sv4.y, sv4.z, sv4.w};
        uint32_t vo[4];
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          const int k0 = 2 * h;
          vo[h] = (keep > k0 + 1) ? vw[h] : (keep > k0 ? (vw[h] & 0xFFFFu) : 0u);
        }
        const uint64_t imask = keep >= 8 ? ~0ull : ((1ull << (8 * keep)) - 1ull);
        const uint64_t iv = (static_cast<uint64_t>(si2.y) << 32 | si2.x) & imask;
        reinterpret_cast<uint4*>(L.values + g * C)[q] = make_uint4(vo[0], vo[1], vo[2], vo[3]);
        reinterpret_cast<uint2*>(L.idx + g * C)[q] = make_uint2(static_cast<uint32_t>(iv), static_cast<uint32_t>(iv >> 32));
      }
    } else {
      for (int q = 0; q < C; ++q) {
        L.values[g * C + q] = q < cnt ? sv[c * C + q] : static_cast<uint16_t>(0);
        L.idx[g * C + q] = q < cnt ? si[c * C + q] : static_cast<uint8_t>(0);
      }
    }
    L.counts[g] = dense ? static_cast<uint8_t>(TWELL_DENSE_TILE) : static_cast<uint8_t>(cnt);
  }
  if (__any_sync(0xffffffffu, over) && lane == 0) L.row_fb[row] = 1;
}

// Routing of a small batch (at most 32 rows) by one CTA: the result of
// route_kernel (fallback rows numbered in ascending row order, rows past
// fb_cap left with empty cells, n_fb, the overflow status).
__device__ void route_small(const Layout& L) {
  __shared__ int slot_s[32];
  if (threadIdx.x < 32) {
    const int r = threadIdx.x;
    const bool fl = r < L.N && __ldcg(&L.row_fb[r]) != 0;
    const unsigned m = __ballot_sync(0xffffffffu, fl);
    const int slot = __popc(m & ((1u << r) - 1u));
    if (r < L.N) {
      L.row_fb[r] = fl ? slot : -1;
      if (fl && slot < L.fb_cap) L.fb_rows[slot] = r;
    }
    slot_s[r] = fl ? slot : -1;
    if (r == 0) {
      *L.n_fb = __popc(m);
      if (__popc(m) > L.fb_cap) report_error(L.status, TWELL_ERR_FALLBACK_OVERFLOW);
    }
  }
  __syncthreads();
  for (int r = 0; r < L.N && r < 32; ++r) {
    if (slot_s[r] < L.fb_cap) continue;  // TwELL row (-1) or stored fallback row
    const int64_t cell0 = static_cast<int64_t>(r) * L.nt;
    for (int c = threadIdx.x; c < L.nt; c += blockDim.x) L.counts[cell0 + c] = 0;
    for (int c = threadIdx.x; c < L.nt * L.C; c += blockDim.x) {
      L.values[cell0 * L.C + c] = 0;
      L.idx[cell0 * L.C + c] = 0;
    }
  }
}

// Small-batch variant: z = sum of the K-split partial sums (split order) +
// b, h = bf16(z) where z > 2^-134 (the smallest z whose bf16 rounding is not
// zero), else +0; h is also stored densely in H for the fallback copy.  With
// an arrival counter (zeroed, at most 32 rows) the CTA that finishes last
// also routes the rows, so no separate routing launch is needed.
__global__ void __launch_bounds__(kWarps * 32)
    pack_partials_kernel(Layout L, const float* __restrict__ part, int ksplit, const uint16_t* __restrict__ b,
                         uint16_t* __restrict__ H, int32_t* arrivals) {
  __shared__ int last_s;
  grid_dependency_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int segs = (L.f + 255) / 256;
  const int64_t gw = static_cast<int64_t>(blockIdx.x) * kWarps + warp;
  if (gw < static_cast<int64_t>(L.N) * segs) {  // whole warps
    const int row = static_cast<int>(gw / segs);
    const int col = static_cast<int>(gw % segs) * 256 + lane * 8;
    const bool in = col < L.f;
    uint32_t w[4] = {0u, 0u, 0u, 0u};
    if (in) {
      float z[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      const int64_t split = static_cast<int64_t>(L.N) * L.f;
      const float* p = part + static_cast<int64_t>(row) * L.f + col;
#pragma unroll 8
      for (int ks = 0; ks < ksplit; ++ks) {
        const float4 a = *reinterpret_cast<const float4*>(p + ks * split);
        const float4 c = *reinterpret_cast<const float4*>(p + ks * split + 4);
        z[0] += a.x; z[1] += a.y; z[2] += a.z; z[3] += a.w;
        z[4] += c.x; z[5] += c.y; z[6] += c.z; z[7] += c.w;
      }
      const uint4 bq = __ldg(reinterpret_cast<const uint4*>(b + col));
      const uint32_t bw[4] = {bq.x, bq.y, bq.z, bq.w};
      const float thr = __uint_as_float(0x00008000u);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float zb = z[k] + ((k & 1) ? bf16_hi(bw[k / 2]) : bf16_lo(bw[k / 2]));
        const uint32_t h = zb > thr ? float_to_bf16_bits(zb) : 0u;
        w[k / 2] |= (k & 1) ? (h << 16) : h;
      }
      *reinterpret_cast<uint4*>(H + static_cast<int64_t>(row) * L.f + col) = make_uint4(w[0], w[1], w[2], w[3]);
    }
    pack_lane8(L, row, col, in, w);
  }
  if (!arrivals) return;
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    last_s = atomicAdd(arrivals, 1) == static_cast<int>(gridDim.x) - 1;
  }
  __syncthreads();
  if (!last_s) return;
  __threadfence();
  route_small(L);
}

// Fallback rows: copy the dense row, clear the row's cells.
__global__ void fb_copy_kernel(Layout L, const uint16_t* __restrict__ H, int64_t ldh) {
  const int nfb = min(*L.n_fb, L.fb_cap);
  for (int slot = blockIdx.x; slot < nfb; slot += gridDim.x) {
    const int row = L.fb_rows[slot];
    const uint4* src = reinterpret_cast<const uint4*>(H + static_cast<int64_t>(row) * ldh);
    uint4* dst = reinterpret_cast<uint4*>(L.fb_dense + static_cast<int64_t>(slot) * L.f);
    for (int i = threadIdx.x; i < L.f / 8; i += blockDim.x) dst[i] = src[i];
    const int64_t cell0 = static_cast<int64_t>(row) * L.nt;
    for (int i = threadIdx.x; i < L.nt; i += blockDim.x) L.counts[cell0 + i] = 0;
    for (int i = threadIdx.x; i < L.nt * L.C; i += blockDim.x) {
      L.values[cell0 * L.C + i] = 0;
      L.idx[cell0 * L.C + i] = 0;
    }
  }
}

// Cells -> dense.  A warp takes runs of kUnpackCols columns of one row
// (grid-stride over (row, run)) and builds each run in its own shared-memory
// buffer: zeros, then every cell's stored entries (or a dense tile of the
// tile-granular variant, copied from its pool slot), then the run goes out
// as coalesced 16-byte stores, so every byte of H is written exactly once
// and no scattered partial-sector writes reach L2.  The row's routing word,
// each lane's first cell's count and (C a multiple of 8) its first 8 slots
// are requested together before any of them is used.  A fallback row's run
// is copied from fb_dense (zeros past fb_cap: such a row is stored nowhere).
constexpr int kUnpackCols = 2048;  // 4 KB of bf16 per warp

__device__ __forceinline__ uint16_t slot_value8(const uint4& v, int sl) {
  const uint32_t w = sl < 2 ? v.x : (sl < 4 ? v.y : (sl < 6 ? v.z : v.w));
  return static_cast<uint16_t>((sl & 1) ? (w >> 16) : (w & 0xFFFFu));
}

__device__ __forceinline__ int slot_index8(const uint2& v, int sl) {
  return static_cast<int>(((sl < 4 ? v.x : v.y) >> (8 * (sl & 3))) & 0xFFu);
}

__global__ void __launch_bounds__(kWarps * 32, 5)
    unpack_run_kernel(Layout L, uint16_t* __restrict__ H, int64_t ldh) {
  extern __shared__ uint4 urun4[];  // [kWarps][kUnpackCols / 8]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint4* run4 = urun4 + warp * (kUnpackCols / 8);
  uint16_t* run = reinterpret_cast<uint16_t*>(run4);
  const int T = L.T, C = L.C;
  const bool c8 = (C & 7) == 0;
  const bool tiles = L.hybrid == TWELL_HYBRID_TILES;
  const int runs = (L.f + kUnpackCols - 1) / kUnpackCols;
  const int64_t total = static_cast<int64_t>(L.N) * runs;
  const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
  for (int64_t gw = static_cast<int64_t>(blockIdx.x) * kWarps + warp; gw < total;
       gw += static_cast<int64_t>(gridDim.x) * kWarps) {
    const int row = static_cast<int>(gw / runs);
    const int c0 = static_cast<int>(gw % runs) * kUnpackCols;
    const int ncol = min(kUnpackCols, L.f - c0);  // a multiple of T (f % T == 0)
    const int vecs = ncol / 8;
    const int ncell = ncol / T;
    const int64_t cell0 = static_cast<int64_t>(row) * L.nt + c0 / T;
    uint4* hrun = reinterpret_cast<uint4*>(H + static_cast<int64_t>(row) * ldh + c0);
    const int fb = L.row_fb[row];
    int cnt0 = 0;
    uint4 val0 = zero;
    uint2 idx0 = make_uint2(0u, 0u);
    if (lane < ncell) {
      cnt0 = L.counts[cell0 + lane];
      if (c8) {
        val0 = *reinterpret_cast<const uint4*>(L.values + (cell0 + lane) * C);
        idx0 = *reinterpret_cast<const uint2*>(L.idx + (cell0 + lane) * C);
      }
    }
    if (fb >= 0) {  // uniform over the warp: the whole row is dense
      if (fb < L.fb_cap) {
        const uint4* src = reinterpret_cast<const uint4*>(L.fb_dense + static_cast<int64_t>(fb) * L.f + c0);
        for (int i = lane; i < vecs; i += 32) hrun[i] = src[i];
      } else {
        for (int i = lane; i < vecs; i += 32) hrun[i] = zero;
      }
      continue;
    }
    for (int i = lane; i < vecs; i += 32) run4[i] = zero;
    __syncwarp();
    for (int c = lane; c < ncell; c += 32) {
      const int64_t cell = cell0 + c;
      int cnt = cnt0;
      uint4 vv = val0;
      uint2 ii = idx0;
      if (c != lane) {
        cnt = L.counts[cell];
        if (c8 && cnt > 0) {
          vv = *reinterpret_cast<const uint4*>(L.values + cell * C);
          ii = *reinterpret_cast<const uint2*>(L.idx + cell * C);
        }
      }
      if (cnt == 0) continue;
      uint16_t* cr = run + c * T;
      if (tiles && cnt == TWELL_DENSE_TILE) {
        const int64_t slot = c8 ? (static_cast<int64_t>(vv.x & 0xFFFFu) | (static_cast<int64_t>(ii.x & 0xFFu) << 16))
                                : (static_cast<int64_t>(L.values[cell * C]) | (static_cast<int64_t>(L.idx[cell * C]) << 16));
        if (slot < static_cast<int64_t>(L.fb_cap) * L.nt) {
          const uint4* src = reinterpret_cast<const uint4*>(L.fb_dense + slot * T);
          for (int k = 0; k < T / 8; ++k) reinterpret_cast<uint4*>(cr)[k] = src[k];
        }
        continue;
      }
      // (indices bounded by T so that a malformed layout cannot write past the cell)
      const int n = min(cnt, C);
      int sl = 0;
      if (c8) {
        for (; sl < min(n, 8); ++sl) {
          const int j = slot_index8(ii, sl);
          if (j < T) cr[j] = slot_value8(vv, sl);
        }
      }
      for (; sl < n; ++sl) {
        const int j = L.idx[cell * C + sl];
        if (j < T) cr[j] = L.values[cell * C + sl];
      }
    }
    __syncwarp();
    for (int i = lane; i < vecs; i += 32) hrun[i] = run4[i];
    __syncwarp();  // every lane has read the run before the buffer is zeroed again
  }
}

// ---------------------------------------------------------------- format check
// Rule numbers of the violation mask (bit k = rule k), as twell.h lists them.
constexpr int kRuleCount = 1, kRuleFbCell = 2, kRuleIdxRange = 3, kRuleIdxOrder = 4, kRuleZero = 5,
              kRulePad = 6, kRuleRowMap = 7, kRuleFbOrder = 8, kRuleFbCount = 9, kRuleTileOrder = 10,
              kRuleTileCount = 11, kRuleTileSparse = 12;

__device__ __forceinline__ bool bf16_is_zero(uint16_t v) { return (v & 0x7FFFu) == 0; }

// OR of every lane's bits, one atomic per warp; all lanes must arrive.
__device__ __forceinline__ void flag_rules(int32_t* mask, int32_t* status, int bits) {
  bits = static_cast<int>(__reduce_or_sync(0xffffffffu, static_cast<unsigned>(bits)));
  if ((threadIdx.x & 31) == 0 && bits) {
    atomicOr(mask, bits);
    report_error(status, TWELL_ERR_BAD_FORMAT);
  }
}

// One thread per cell (grid-stride): the count, the stored entries, the
// padding, and for a dense tile the pool tile it names.
__global__ void __launch_bounds__(256) check_cells_kernel(Layout L, int32_t* mask) {
  const bool tiles = L.hybrid == TWELL_HYBRID_TILES;
  const int64_t cells = static_cast<int64_t>(L.N) * L.nt;
  const int64_t pool = static_cast<int64_t>(L.fb_cap) * L.nt;
  int bits = 0;
  for (int64_t cell = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; cell < cells;
       cell += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int cnt = L.counts[cell];
    const uint16_t* v = L.values + cell * L.C;
    const uint8_t* ix = L.idx + cell * L.C;
    int s_begin = 0, entries = cnt;  // slots [s_begin, entries) hold entries, the rest padding
    if (tiles && cnt == TWELL_DENSE_TILE) {
      const int64_t slot = static_cast<int64_t>(v[0]) | (static_cast<int64_t>(ix[0]) << 16);
      if (slot < pool) {  // a slot past the pool breaks the numbering rule instead
        const uint16_t* p = L.fb_dense + slot * L.T;
        int nz = 0;
        for (int i = 0; i < L.T; ++i) nz += bf16_is_zero(p[i]) ? 0 : 1;
        if (nz <= L.C) bits |= 1 << kRuleTileSparse;
      }
      s_begin = 1;  // slot 0 holds the pool slot
      entries = 0;
    } else {
      if (!tiles && cnt != 0 && L.row_fb[cell / L.nt] >= 0) bits |= 1 << kRuleFbCell;
      if (cnt > L.C) {
        bits |= 1 << kRuleCount;
        continue;  // the slots' meaning is unknown
      }
    }
    for (int s = s_begin; s < L.C; ++s) {
      const uint16_t vs = v[s];
      const int is = ix[s];
      if (s < entries) {
        if (is >= L.T) bits |= 1 << kRuleIdxRange;
        if (s > 0 && is <= ix[s - 1]) bits |= 1 << kRuleIdxOrder;
        if (bf16_is_zero(vs)) bits |= 1 << kRuleZero;
      } else if (vs != 0 || is != 0) {
        bits |= 1 << kRulePad;
      }
    }
  }
  flag_rules(mask, L.status, bits);
}

// One CTA numbers the fallback rows (rows variant) or the dense tiles (tiles
// variant) in order with a block-wide exclusive scan, 1024 items per pass,
// and checks each against the slot it holds; then the totals and fb_rows.
constexpr int kCheckThreads = 1024;

__global__ void __launch_bounds__(kCheckThreads) check_order_kernel(Layout L, int32_t* mask) {
  __shared__ int warp_tot[kCheckThreads / 32];
  __shared__ int64_t base_s;
  const bool tiles = L.hybrid == TWELL_HYBRID_TILES;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t items = tiles ? static_cast<int64_t>(L.N) * L.nt : L.N;
  const int64_t pool = static_cast<int64_t>(L.fb_cap) * L.nt;
  int bits = 0;
  if (tid == 0) base_s = 0;
  __syncthreads();
  for (int64_t i0 = 0; i0 < items; i0 += kCheckThreads) {
    const int64_t i = i0 + tid;
    bool marked = false;
    int64_t slot = -1;
    if (i < items) {
      if (tiles) {
        marked = L.counts[i] == TWELL_DENSE_TILE;
        if (marked) slot = static_cast<int64_t>(L.values[i * L.C]) | (static_cast<int64_t>(L.idx[i * L.C]) << 16);
      } else {
        slot = L.row_fb[i];
        marked = slot >= 0;
        if (slot < -1) bits |= 1 << kRuleRowMap;
      }
    }
    const unsigned ball = __ballot_sync(0xffffffffu, marked);
    if (lane == 0) warp_tot[warp] = __popc(ball);
    __syncthreads();
    if (warp == 0) {
      const int w = warp_tot[lane];
      int incl = w;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += u;
      }
      warp_tot[lane] = incl - w;  // exclusive prefix of the warps' counts
    }
    __syncthreads();
    const int64_t base = base_s;
    const int64_t rank = base + warp_tot[warp] + __popc(ball & ((1u << lane) - 1u));
    if (marked) {
      if (tiles) {
        if (slot != rank || slot >= pool) bits |= 1 << kRuleTileOrder;
      } else {
        if (slot != rank) bits |= 1 << kRuleFbOrder;
        if (slot < L.fb_cap && L.fb_rows[slot] != i) bits |= 1 << kRuleRowMap;
      }
    }
    __syncthreads();
    if (tid == kCheckThreads - 1) base_s = rank + (marked ? 1 : 0);
    __syncthreads();
  }
  const int64_t marked_total = base_s;
  const int64_t n_fb = *L.n_fb;
  if (tiles) {
    for (int r = tid; r < L.N; r += kCheckThreads)
      if (L.row_fb[r] != -1) bits |= 1 << kRuleRowMap;
    if (tid == 0 && marked_total != min(n_fb, pool)) bits |= 1 << kRuleTileCount;
  } else {
    const int64_t stored = min(n_fb, static_cast<int64_t>(L.fb_cap));
    for (int64_t s = 1 + tid; s < stored; s += kCheckThreads)
      if (L.fb_rows[s] <= L.fb_rows[s - 1]) bits |= 1 << kRuleFbOrder;
    if (tid == 0 && marked_total != n_fb) bits |= 1 << kRuleFbCount;
  }
  flag_rules(mask, L.status, bits);
}

int64_t warps_needed(const twell_t& L) {
  return static_cast<int64_t>(L.n_rows) * ((L.d_ff + 255) / 256);
}

}  // namespace

int launch_pack_cells(const uint16_t* H, int64_t ldh, const twell_t& L, cudaStream_t s) {
  const int64_t warps = static_cast<int64_t>(L.n_rows) * ((L.d_ff + kPackSeg * 256 - 1) / (kPackSeg * 256));
  const int64_t blocks = (warps + kWarps - 1) / kWarps;
  if (blocks <= 0) return TWELL_OK;
  if (blocks > 0x7FFFFFFF) return TWELL_ERR_UNSUPPORTED;
  const unsigned g = static_cast<unsigned>(blocks);
  LaunchScope ls(TWELL_KERNEL_PACK, s);
  switch (L.tile) {
    case 32: pack_cells_kernel<32><<<g, kWarps * 32, 0, s>>>(flat(L), H, ldh); break;
    case 64: pack_cells_kernel<64><<<g, kWarps * 32, 0, s>>>(flat(L), H, ldh); break;
    case 128: pack_cells_kernel<128><<<g, kWarps * 32, 0, s>>>(flat(L), H, ldh); break;
    default: pack_cells_kernel<256><<<g, kWarps * 32, 0, s>>>(flat(L), H, ldh); break;
  }
  return cudaGetLastError() == cudaSuccess ? TWELL_OK : TWELL_ERR_CUDA;
}

int launch_pack_partials(const float* part, int ksplit, const uint16_t* b, uint16_t* H, const twell_t& L,
                         int32_t* arrivals, cudaStream_t s) {
  const int64_t blocks = (warps_needed(L) + kWarps - 1) / kWarps;
  if (blocks <= 0) return TWELL_OK;
  if (blocks > 0x7FFFFFFF || L.d_ff % 8 != 0) return TWELL_ERR_UNSUPPORTED;
  if (arrivals && L.n_rows > 32) return TWELL_ERR_UNSUPPORTED;
  LaunchScope ls(TWELL_KERNEL_PACK, s);
  if (launch_pdl(pack_partials_kernel, dim3(static_cast<unsigned>(blocks)), dim3(kWarps * 32), 0, s, flat(L), part,
                 ksplit, b, H, arrivals) != cudaSuccess)
    return TWELL_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? TWELL_OK : TWELL_ERR_CUDA;
}

int launch_fb_copy(const uint16_t* H, int64_t ldh, const twell_t& L, cudaStream_t s) {
  if (L.fb_cap <= 0) return TWELL_OK;
  const int grid = std::max(1, std::min(L.fb_cap, 2 * sm_count()));
  LaunchScope ls(TWELL_KERNEL_PACK, s);
  fb_copy_kernel<<<grid, 256, 0, s>>>(flat(L), H, ldh);
  return cudaGetLastError() == cudaSuccess ? TWELL_OK : TWELL_ERR_CUDA;
}

int launch_unpack(const twell_t& L, uint16_t* H, int64_t ldh, cudaStream_t s) {
  if (L.n_rows <= 0) return TWELL_OK;
  const int64_t warps = static_cast<int64_t>(L.n_rows) * ((L.d_ff + kUnpackCols - 1) / kUnpackCols);
  const size_t smem = sizeof(uint16_t) * kWarps * kUnpackCols;
  const int per_sm = std::max(1, resident_ctas_per_sm(reinterpret_cast<const void*>(unpack_run_kernel),
                                                      kWarps * 32, smem));
  const int64_t blocks = std::min<int64_t>((warps + kWarps - 1) / kWarps, static_cast<int64_t>(per_sm) * sm_count());
  LaunchScope ls(TWELL_KERNEL_UNPACK, s);
  unpack_run_kernel<<<static_cast<unsigned>(blocks), kWarps * 32, smem, s>>>(flat(L), H, ldh);
  return cudaGetLastError() == cudaSuccess ? TWELL_OK : TWELL_ERR_CUDA;
}

int launch_check_format(const twell_t& L, int32_t* violations, cudaStream_t s) {
  if (cudaMemsetAsync(violations, 0, sizeof(int32_t), s) != cudaSuccess) return TWELL_ERR_CUDA;
  const int64_t cells = static_cast<int64_t>(L.n_rows) * (L.d_ff / L.tile);
  if (cells > 0) {
    const int64_t blocks = std::min<int64_t>((cells + 255) / 256, 8 * static_cast<int64_t>(sm_count()));
    LaunchScope ls(TWELL_KERNEL_CHECK_FORMAT, s);
    check_cells_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(flat(L), violations);
    if (cudaGetLastError() != cudaSuccess) return TWELL_ERR_CUDA;
  }
  LaunchScope ls(TWELL_KERNEL_CHECK_FORMAT, s);
  check_order_kernel<<<1, kCheckThreads, 0, s>>>(flat(L), violations);
  return cudaGetLastError() == cudaSuccess ? TWELL_OK : TWELL_ERR_CUDA;
}

}  // namespace twell
