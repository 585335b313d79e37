// Backward of the TwELL layer for  L = sum(Y * dY) + lambda * sum|H|
// (L1 on the activations: bayesiansapien note, TL;DR; training kernels are
// part of the release, "What it claims").
//
//   SDDMM     dZ[n][j] = dY[n] . W_down[j] + lambda, kept only at the stored
//             non-zeros of H (the ReLU mask is the pattern): a tcgen05 GEMM
//             dY . W_down^T whose epilogue samples the accumulator at the TwELL
//             pattern (gemm_tcgen05.cu)
//   dX        dX[n] = sum_j dZ[n][j] W_in^T[j]: the gather-SpMM (spmm.cu) with
//             fp32 values for TwELL rows; for fallback rows a split-K tcgen05
//             GEMM of dZ (as bf16 high + low parts) with W_in^T read N-major
//   unit lists  the TwELL entries regrouped by hidden unit, rows ascending,
//             built deterministically in one launch (a CTA per tile of units:
//             counts, scans and row masks in shared memory)
//   dw_unitcta_kernel  dW_down[j] = sum_n h[n][j] dY[n], dW_in^T[j] = sum_n dZ[n][j] X[n],
//             db[j] = sum_n dZ[n][j] over the TwELL entries
//   fallback  the dense fallback rows' share of dW_down and dW_in^T stored
//             first by tcgen05 GEMMs with both operands M/N-major (H_fb^T .
//             dY_fb and dZ_fb^T . X_fb, dZ as high + low bf16 parts) on the
//             second stream; dw_unitcta_kernel adds the TwELL share on top; a column
//             sum adds the fallback share of db
// The gated layer (h = bf16(g u), g = X.W_g + b > 0, u = X.W_u) runs the same
// steps with pairs: its SDDMM forms (dG, dU) = (dh' u, dh' g) at the pattern
// (dh' = dY.W_down^T + lambda sign(h)) from the (g, u) its forward kept; dX
// gathers two weight rows per entry; the unit lists carry dU beside dG and the
// walk adds dW_u^T[j] = sum_n dU[n][j] X[n] from the same X loads.  Its
// fallback rows get g and u recomputed on the tensor cores (GUEpi) beside the
// SDDMM, then dG, dU as high + low parts, three store GEMMs and two dX GEMMs.
// No atomics on outputs, so every result is deterministic.
#include <cuda_runtime.h>

#include <algorithm>

#include "sm103.cuh"
#include "twell_internal.h"

namespace twell {
namespace {

struct Layout {
  int32_t N, f, T, C, fb_cap, nt;
  const uint16_t* values;
  const uint8_t* idx;
  const uint8_t* counts;
  const int32_t* row_fb;
  const int32_t* fb_rows;
  const uint16_t* fb_dense;
  const int32_t* n_fb;
};

Layout flat(const twell_t& L) {
  return Layout{L.n_rows, L.d_ff, L.tile, L.cap, L.fb_cap, L.d_ff / L.tile, L.values, L.idx,
                L.counts, L.row_fb, L.fb_rows, L.fb_dense, L.n_fb};
}

constexpr int kWarps = 8;
constexpr int kU = 4;  // entries in flight per lane in dw_unitcta_kernel (2 rows each)

// Unit-major regrouping of the TwELL entries, one launch: a CTA per tile t
// builds the lists of the tile's T hidden units (every unit of a tile lives in
// the same column of cells, so the tile's bookkeeping stays in shared memory)
// into the tile's own region of the entry arrays, [t * N * C, (t + 1) * N * C).
// Warp w owns a contiguous range of 32-row blocks.  Pass 1 counts each unit's
// entries per warp; scans over the warps and then over the units give every
// (warp, unit) its start.  Pass 2 walks each warp's blocks in order: a 32-bit
// mask per unit (bit = row of the block) places row r's entry at the unit's
// start + the warp's running cursor + popc(mask below r).  Rows ascend within
// every unit, nothing is atomic on the output, and the result is a pure
// function of the pattern.
constexpr int kListWarps = 32;
constexpr int kListChunk = 4;  // row blocks whose cells a warp loads before using them

// The 8 slot indices (C == 8) or values of one cell, loaded as whole vectors so
// that a chunk of blocks costs one memory latency, not one per block.
__device__ __forceinline__ int cell_idx8(uint2 w, int sl) {
  const uint64_t v = (static_cast<uint64_t>(w.y) << 32) | w.x;
  return static_cast<int>((v >> (8 * sl)) & 0xFFu);
}

// skip_fb (a row view of a tile-granular layout, else null): rows with
// skip_fb[r] >= 0 are the view's fallback rows, whose cells (which may name
// dense tiles) take no part in the lists.
// kGated: dz_cells holds (dG, dU) pairs per slot; dG goes to col_dz and dU to col_du.
template <bool kC8, bool kGated>
__global__ void __launch_bounds__(kListWarps * 32)
    unit_lists_kernel(Layout L, const float* __restrict__ dz_cells, int32_t* __restrict__ col_beg,
                      int32_t* __restrict__ col_end, int32_t* __restrict__ col_rows, uint16_t* __restrict__ col_h,
                      float* __restrict__ col_dz, const int32_t* __restrict__ skip_fb, float* __restrict__ col_du) {
  extern __shared__ int32_t lsm[];
  grid_dependency_wait();
  const int T = L.T, t = blockIdx.x;
  int32_t* wcur = lsm;                                            // [kListWarps][T]: counts, then cursors
  uint32_t* wmask = reinterpret_cast<uint32_t*>(lsm + kListWarps * T);  // [kListWarps][T]
  int32_t* ustart = lsm + 2 * kListWarps * T;                     // [T]
  __shared__ int scan_tot[kListWarps];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nblk = (L.N + 31) / 32;
  const int per = (nblk + kListWarps - 1) / kListWarps;
  const int b0 = min(nblk, warp * per), b1 = min(nblk, b0 + per);
  for (int i = tid; i < kListWarps * T; i += blockDim.x) wcur[i] = 0;
  __syncthreads();
  // ---- pass 1: entries per (warp, unit), kListChunk blocks' cells loaded at once
  for (int c0 = b0; c0 < b1; c0 += kListChunk) {
    int cnt[kListChunk];
    uint2 iw[kListChunk];
#pragma unroll
    for (int j = 0; j < kListChunk; ++j) {
      const int r = (c0 + j) * 32 + lane;
      const bool ok = c0 + j < b1 && r < L.N && (!skip_fb || skip_fb[r] < 0);
      const int64_t cell = static_cast<int64_t>(r) * L.nt + t;
      cnt[j] = ok ? L.counts[cell] : 0;
      if (kC8) iw[j] = ok ? *reinterpret_cast<const uint2*>(L.idx + cell * 8) : make_uint2(0u, 0u);
    }
#pragma unroll
    for (int j = 0; j < kListChunk; ++j) {
      const int64_t cell = static_cast<int64_t>((c0 + j) * 32 + lane) * L.nt + t;
      for (int sl = 0; sl < cnt[j]; ++sl)
        atomicAdd(&wcur[warp * T + (kC8 ? cell_idx8(iw[j], sl) : L.idx[cell * L.C + sl])], 1);
    }
  }
  __syncthreads();
  // ---- scans: over the warps per unit (counts -> exclusive starts), then over the units
  int total = 0;
  if (tid < T) {
    for (int w = 0; w < kListWarps; ++w) {
      const int c = wcur[w * T + tid];
      wcur[w * T + tid] = total;
      total += c;
    }
  }
  int incl = total;  // threads past T hold 0
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int x = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += x;
  }
  if (lane == 31) scan_tot[warp] = incl;
  __syncthreads();
  int before = 0;
  for (int w = 0; w < warp; ++w) before += scan_tot[w];
  const int64_t base = static_cast<int64_t>(t) * L.N * L.C;
  if (tid < T) {
    const int start = before + incl - total;
    ustart[tid] = start;
    col_beg[t * T + tid] = static_cast<int32_t>(base + start);
    col_end[t * T + tid] = static_cast<int32_t>(base + start + total);
  }
  __syncthreads();
  // ---- pass 2: place every entry, blocks of each warp in ascending order
  uint32_t* m = wmask + warp * T;
  int32_t* cur = wcur + warp * T;
  for (int c0 = b0; c0 < b1; c0 += kListChunk) {
    int cnt[kListChunk];
    uint2 iw[kListChunk];
#pragma unroll
    for (int j = 0; j < kListChunk; ++j) {
      const int r = (c0 + j) * 32 + lane;
      const bool ok = c0 + j < b1 && r < L.N && (!skip_fb || skip_fb[r] < 0);
      const int64_t cell = static_cast<int64_t>(r) * L.nt + t;
      cnt[j] = ok ? L.counts[cell] : 0;
      if (kC8) iw[j] = ok ? *reinterpret_cast<const uint2*>(L.idx + cell * 8) : make_uint2(0u, 0u);
    }
#pragma unroll
    for (int j = 0; j < kListChunk; ++j) {
      if (c0 + j >= b1) break;  // uniform over the warp
      const int r = (c0 + j) * 32 + lane;
      const int64_t cell = static_cast<int64_t>(r) * L.nt + t;
      // the block's values and dZ, requested before the masks are built
      uint4 hv = make_uint4(0u, 0u, 0u, 0u);
      float4 dz0 = make_float4(0.f, 0.f, 0.f, 0.f), dz1 = dz0, dz2 = dz0, dz3 = dz0;
      if (kC8 && cnt[j] > 0) {
        hv = *reinterpret_cast<const uint4*>(L.values + cell * 8);
        if (kGated) {
          const float4* q = reinterpret_cast<const float4*>(dz_cells + cell * 16);
          dz0 = q[0];
          dz1 = q[1];
          dz2 = q[2];
          dz3 = q[3];
        } else {
          dz0 = *reinterpret_cast<const float4*>(dz_cells + cell * 8);
          dz1 = *reinterpret_cast<const float4*>(dz_cells + cell * 8 + 4);
        }
      }
      for (int u = lane; u < T; u += 32) m[u] = 0;
      __syncwarp();
      for (int sl = 0; sl < cnt[j]; ++sl)
        atomicOr(&m[kC8 ? cell_idx8(iw[j], sl) : L.idx[cell * L.C + sl]], 1u << lane);
      __syncwarp();
      const uint32_t hw[4] = {hv.x, hv.y, hv.z, hv.w};
      // slot sl's dZ (kGated: its (dG, dU) pair is dzs[2 sl], dzs[2 sl + 1])
      float dzs[kGated ? 16 : 8];
      const float4 dzq[4] = {dz0, dz1, dz2, dz3};
#pragma unroll
      for (int q = 0; q < (kGated ? 4 : 2); ++q) {
        dzs[4 * q] = dzq[q].x;
        dzs[4 * q + 1] = dzq[q].y;
        dzs[4 * q + 2] = dzq[q].z;
        dzs[4 * q + 3] = dzq[q].w;
      }
      for (int sl = 0; sl < cnt[j]; ++sl) {
        const int u = kC8 ? cell_idx8(iw[j], sl) : L.idx[cell * L.C + sl];
        const int64_t pos = base + ustart[u] + cur[u] + __popc(m[u] & ((1u << lane) - 1u));
        col_rows[pos] = r;
        if (kC8) {
          col_h[pos] = static_cast<uint16_t>(hw[sl >> 1] >> (16 * (sl & 1)));
          if (kGated) {
            col_dz[pos] = dzs[2 * sl];
            col_du[pos] = dzs[2 * sl + 1];
          } else {
            col_dz[pos] = dzs[sl];
          }
        } else {
          col_h[pos] = L.values[cell * L.C + sl];
          if (kGated) {
            col_dz[pos] = dz_cells[(cell * L.C + sl) * 2];
            col_du[pos] = dz_cells[(cell * L.C + sl) * 2 + 1];
          } else {
            col_dz[pos] = dz_cells[cell * L.C + sl];
          }
        }
      }
      __syncwarp();
      for (int u = lane; u < T; u += 32) cur[u] += __popc(m[u]);
      __syncwarp();
    }
  }
}

size_t unit_lists_smem(int T) { return sizeof(int32_t) * (2 * static_cast<size_t>(kListWarps) * T + T); }

// One staged entry of a hidden unit's list (row, h, dZ); rows ascend.  h is
// exactly a bf16 value, so the dW_down update uses the mixed bf16 x bf16 +
// fp32 fma; the dW_in^T update multiplies the fp32 dZ by X two lanes at a time.
// The gated layer's entries carry (dG, dU) in (dz, du).
struct UnitEntry {
  int32_t row;
  uint32_t h_bits;  // bf16 bits of h in the low half
  float dz;
  float du;
};

// A CTA per hidden unit at a time (persistent, stride gridDim.x): the unit's
// entries are staged once per 256 into shared memory by the whole CTA, and
// warp w accumulates column blocks w, w + 8, ... from them (the same entries
// serve every column block, so they are read from global memory once).
constexpr int kDwChunk = kWarps * 32;

// kGated: also dW_u^T[j] = sum_n dU[n][j] X[n] from the same X loads (dW_inT
// is then dW_g^T, summing dG).
template <bool kGated>
__global__ void __launch_bounds__(kWarps * 32, kGated ? 2 : 3)
    dw_unitcta_kernel(int f, const int32_t* __restrict__ col_beg, const int32_t* __restrict__ col_end,
                      const int32_t* __restrict__ col_rows,
                      const uint16_t* __restrict__ col_h, const float* __restrict__ col_dz,
                      const uint16_t* __restrict__ X, const uint16_t* __restrict__ dY, int d,
                      float* __restrict__ dW_inT, float* __restrict__ dW_down, float* __restrict__ db,
                      const int32_t* __restrict__ n_fb, int fb_cap, const float* __restrict__ col_du,
                      float* __restrict__ dW_uT) {
  __shared__ UnitEntry stage[kDwChunk];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool have_fb = min(*n_fb, fb_cap) > 0;
  const int cbs = (d + 255) / 256;
  // Rounds of kWarps 256-column blocks outermost (two rounds at d_model 4096):
  // the CTAs, which move through their units at about the same pace, then
  // touch one round's columns of X and dY at a time, a working set that stays
  // in L2 where all the columns (67 MB at N 4096, d_model 4096) did not.  Each
  // round writes its own columns of the outputs, so nothing is re-read.
  for (int cb0 = 0; cb0 < cbs; cb0 += kWarps) {
    for (int j = blockIdx.x; j < f; j += gridDim.x) {
      const int e0 = col_beg[j], e1 = col_end[j];
      const int c0 = (cb0 + warp) * 256 + lane * 8;
      const bool active = cb0 + warp < cbs && c0 < d;
      float a_down[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      float a_in[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      float a_u[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      float gb = 0.f;
      for (int b = e0; b < e1; b += kDwChunk) {
        const int m = min(kDwChunk, e1 - b);
        __syncthreads();  // the previous chunk has been consumed
        if (static_cast<int>(threadIdx.x) < m) {
          const int q = b + threadIdx.x;
          stage[threadIdx.x] = UnitEntry{col_rows[q], static_cast<uint32_t>(col_h[q]),
                                         col_dz[q], kGated ? col_du[q] : 0.f};
        }
        __syncthreads();
        int e = 0;
        // the gated walk's larger rows (d_model 4096) want more loads in
        // flight: 8 entries per lane at 2 CTAs per SM (2.98 -> 2.92 ms per
        // gated training step); the plain walk keeps 4 at 3 CTAs per SM
        constexpr int kUw = kGated ? 8 : kU;
        for (; e + kUw <= m; e += kUw) {
          uint4 g[kUw], x[kUw];
          UnitEntry en[kUw];
#pragma unroll
          for (int u = 0; u < kUw; ++u) {
            en[u] = stage[e + u];
            if (active) {
              g[u] = __ldg(reinterpret_cast<const uint4*>(dY + static_cast<int64_t>(en[u].row) * d + c0));
              x[u] = __ldg(reinterpret_cast<const uint4*>(X + static_cast<int64_t>(en[u].row) * d + c0));
            }
          }
#pragma unroll
          for (int u = 0; u < kUw; ++u) {
            gb += en[u].dz;
            if (active) {
              fma8_bf16(a_down, static_cast<uint16_t>(en[u].h_bits), g[u]);
              fma8_f32x2(a_in, en[u].dz, x[u]);
              if (kGated) fma8_f32x2(a_u, en[u].du, x[u]);
            }
          }
        }
        for (; e < m; ++e) {
          const UnitEntry en = stage[e];
          gb += en.dz;
          if (active) {
            fma8_bf16(a_down, static_cast<uint16_t>(en.h_bits),
                      __ldg(reinterpret_cast<const uint4*>(dY + static_cast<int64_t>(en.row) * d + c0)));
            const uint4 xr = __ldg(reinterpret_cast<const uint4*>(X + static_cast<int64_t>(en.row) * d + c0));
            fma8_f32x2(a_in, en.dz, xr);
            if (kGated) fma8_f32x2(a_u, en.du, xr);
          }
        }
      }
      if (active) {
        float4* od = reinterpret_cast<float4*>(dW_down + static_cast<int64_t>(j) * d + c0);
        float4* oi = reinterpret_cast<float4*>(dW_inT + static_cast<int64_t>(j) * d + c0);
        if (have_fb) {
          // the fallback rows' share was stored first by the tensor cores
          const float4 d0 = od[0], d1 = od[1], i0 = oi[0], i1 = oi[1];
          a_down[0] += d0.x; a_down[1] += d0.y; a_down[2] += d0.z; a_down[3] += d0.w;
          a_down[4] += d1.x; a_down[5] += d1.y; a_down[6] += d1.z; a_down[7] += d1.w;
          a_in[0] += i0.x; a_in[1] += i0.y; a_in[2] += i0.z; a_in[3] += i0.w;
          a_in[4] += i1.x; a_in[5] += i1.y; a_in[6] += i1.z; a_in[7] += i1.w;
        }
        od[0] = make_float4(a_down[0], a_down[1], a_down[2], a_down[3]);
        od[1] = make_float4(a_down[4], a_down[5], a_down[6], a_down[7]);
        oi[0] = make_float4(a_in[0], a_in[1], a_in[2], a_in[3]);
        oi[1] = make_float4(a_in[4], a_in[5], a_in[6], a_in[7]);
        if (kGated) {
          float4* ou = reinterpret_cast<float4*>(dW_uT + static_cast<int64_t>(j) * d + c0);
          if (have_fb) {
            const float4 u0 = ou[0], u1 = ou[1];
            a_u[0] += u0.x; a_u[1] += u0.y; a_u[2] += u0.z; a_u[3] += u0.w;
            a_u[4] += u1.x; a_u[5] += u1.y; a_u[6] += u1.z; a_u[7] += u1.w;
          }
          ou[0] = make_float4(a_u[0], a_u[1], a_u[2], a_u[3]);
          ou[1] = make_float4(a_u[4], a_u[5], a_u[6], a_u[7]);
        }
      }
      if (cb0 == 0 && threadIdx.x == 0) db[j] = gb;
    }
  }
}

// Operands of the fallback rows' weight-gradient GEMMs, K = fallback slot:
// hfb[s] = fb_dense[s], dyg[s] = dY[fb_rows[s]] for s < n_fb, and
// xg2[2s] = xg2[2s+1] = X[fb_rows[s]] (paired with the high and low parts of
// dZ, interleaved the same way).  Rows from n_fb (2 n_fb for the paired
// buffers) up to the next multiple of 64 are zero, as the GEMM's device-side K
// requires (du_hl, the gated layer's dU parts, is padded like dz_hl).
__global__ void fb_operands_kernel(Layout L, const uint16_t* __restrict__ X, const uint16_t* __restrict__ dY, int d,
                                   uint16_t* __restrict__ hfb, uint16_t* __restrict__ dyg, uint16_t* __restrict__ xg2,
                                   uint16_t* __restrict__ dz_hl, int fb_pad, uint16_t* __restrict__ du_hl) {
  const int nfb = min(*L.n_fb, L.fb_cap);
  const int k1 = min(fb_pad, (nfb + 63) & ~63);
  const int k2 = min(2 * fb_pad, (2 * nfb + 63) & ~63);
  const uint4 z = make_uint4(0, 0, 0, 0);
  // single rows: hfb, dyg
  for (int slot = blockIdx.x; slot < k1; slot += gridDim.x) {
    const bool real = slot < nfb;
    const int row = real ? L.fb_rows[slot] : 0;
    uint4* h = reinterpret_cast<uint4*>(hfb + static_cast<int64_t>(slot) * L.f);
    const uint4* hs = reinterpret_cast<const uint4*>(L.fb_dense + static_cast<int64_t>(real ? slot : 0) * L.f);
    for (int i = threadIdx.x; i < L.f / 8; i += blockDim.x) h[i] = real ? hs[i] : z;
    uint4* g = reinterpret_cast<uint4*>(dyg + static_cast<int64_t>(slot) * d);
    const uint4* gs = reinterpret_cast<const uint4*>(dY + static_cast<int64_t>(row) * d);
    for (int i = threadIdx.x; i < d / 8; i += blockDim.x) g[i] = real ? gs[i] : z;
  }
  // paired rows: xg2 (X twice), dz_hl padding
  for (int k = blockIdx.x; k < k2; k += gridDim.x) {
    const bool real = k < 2 * nfb;
    const int row = real ? L.fb_rows[k >> 1] : 0;
    uint4* x = reinterpret_cast<uint4*>(xg2 + static_cast<int64_t>(k) * d);
    const uint4* xs = reinterpret_cast<const uint4*>(X + static_cast<int64_t>(row) * d);
    for (int i = threadIdx.x; i < d / 8; i += blockDim.x) x[i] = real ? xs[i] : z;
    if (!real) {
      uint4* a = reinterpret_cast<uint4*>(dz_hl + static_cast<int64_t>(k) * L.f);
      for (int i = threadIdx.x; i < L.f / 8; i += blockDim.x) a[i] = z;
      if (du_hl) {
        uint4* u = reinterpret_cast<uint4*>(du_hl + static_cast<int64_t>(k) * L.f);
        for (int i = threadIdx.x; i < L.f / 8; i += blockDim.x) u[i] = z;
      }
    }
  }
}

// The gated layer's fallback rows: dG = dh' u and dU = dh' g from the SDDMM's
// dense dh' and the recomputed (g, u), as high + low bf16 parts (rows 2 s and
// 2 s + 1 of dz_hl and du_hl); eight units per thread.
__global__ void __launch_bounds__(256)
    gated_fb_parts_kernel(Layout L, const float* __restrict__ dh_fb, const float* __restrict__ gu_fb,
                          uint16_t* __restrict__ dz_hl, uint16_t* __restrict__ du_hl) {
  const int nfb = min(*L.n_fb, L.fb_cap);
  for (int slot = blockIdx.x; slot < nfb; slot += gridDim.x) {
    for (int j = threadIdx.x * 8; j < L.f; j += blockDim.x * 8) {
      const int64_t o = static_cast<int64_t>(slot) * L.f + j;
      const float4* dp = reinterpret_cast<const float4*>(dh_fb + o);
      const float4* gp = reinterpret_cast<const float4*>(gu_fb + 2 * o);
      const float4 d0 = dp[0], d1 = dp[1];
      const float dh[8] = {d0.x, d0.y, d0.z, d0.w, d1.x, d1.y, d1.z, d1.w};
      uint32_t w[4][4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float4 p2 = gp[q];  // (g, u) of units j + 2q and j + 2q + 1
        const float g[2] = {p2.x, p2.z}, u[2] = {p2.y, p2.w};
        w[0][q] = w[1][q] = w[2][q] = w[3][q] = 0u;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const float dg = dh[2 * q + e] * u[e], du = dh[2 * q + e] * g[e];
          const uint16_t gh = float_to_bf16_bits(dg), uh = float_to_bf16_bits(du);
          const uint16_t gl = float_to_bf16_bits(dg - bf16_bits_to_float(gh));
          const uint16_t ul = float_to_bf16_bits(du - bf16_bits_to_float(uh));
          w[0][q] |= static_cast<uint32_t>(gh) << (16 * e);
          w[1][q] |= static_cast<uint32_t>(gl) << (16 * e);
          w[2][q] |= static_cast<uint32_t>(uh) << (16 * e);
          w[3][q] |= static_cast<uint32_t>(ul) << (16 * e);
        }
      }
      const int64_t hi = static_cast<int64_t>(2 * slot) * L.f + j, lo = hi + L.f;
      *reinterpret_cast<uint4*>(dz_hl + hi) = make_uint4(w[0][0], w[0][1], w[0][2], w[0][3]);
      *reinterpret_cast<uint4*>(dz_hl + lo) = make_uint4(w[1][0], w[1][1], w[1][2], w[1][3]);
      *reinterpret_cast<uint4*>(du_hl + hi) = make_uint4(w[2][0], w[2][1], w[2][2], w[2][3]);
      *reinterpret_cast<uint4*>(du_hl + lo) = make_uint4(w[3][0], w[3][1], w[3][2], w[3][3]);
    }
  }
}

// db[j] += sum over the fallback slots of dZ[slot][j] (= high + low part): a
// CTA covers 32 units, warp w sums slots w, w + 8, ... and the eight partial
// sums are added in warp order (a fixed order, so the result is deterministic).
__global__ void __launch_bounds__(256) fb_db_kernel(Layout L, const uint16_t* __restrict__ dz_hl,
                                                    float* __restrict__ db) {
  __shared__ float part[8][32];
  grid_dependency_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int j = blockIdx.x * 32 + lane;
  const int nfb = min(*L.n_fb, L.fb_cap);
  float s = 0.f;
  if (j < L.f)
#pragma unroll 4
    for (int slot = warp; slot < nfb; slot += 8)
      s += bf16_bits_to_float(dz_hl[static_cast<int64_t>(2 * slot) * L.f + j]) +
           bf16_bits_to_float(dz_hl[static_cast<int64_t>(2 * slot + 1) * L.f + j]);
  part[warp][lane] = s;
  __syncthreads();
  if (warp == 0 && j < L.f) {
    float t = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) t += part[w][lane];
    db[j] += t;
  }
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

size_t bwd_workspace_layout(int N, int d_model, int d_ff, int T, int C, int fb_cap, BwdWorkspace* ws,
                            void* base, bool gated) {
  const int nt = d_ff / T;
  const int64_t cells = static_cast<int64_t>(N) * nt * C;
  const int ksplit = fb_cap > 0 ? choose_fb_ksplit(d_ff) : 1;
  const int fb_pad = (fb_cap + 63) & ~63;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off += align256(bytes);
    return o;
  };
  const size_t padf = static_cast<size_t>(fb_pad) * d_ff;
  const size_t padd = static_cast<size_t>(fb_pad) * d_model;
  const int pairs = gated ? 2 : 1;
  const size_t o_dzc = take(sizeof(float) * cells * pairs);
  const size_t o_hl = take(sizeof(uint16_t) * 2 * padf);
  // The fallback rows' gathered operands (and, gated, their recomputed (g, u)
  // and dh') are dead once the store GEMMs have run; the split-K partials of
  // their dX are written after those GEMMs on the same stream, so both share
  // one region.
  const size_t s_hfb = align256(sizeof(uint16_t) * padf), s_dyg = align256(sizeof(uint16_t) * padd);
  const size_t s_xg = align256(sizeof(uint16_t) * 2 * padd);
  const size_t s_gufb = gated ? align256(sizeof(float) * 2 * padf) : 0;
  const size_t s_dhfb = gated ? align256(sizeof(float) * padf) : 0;
  const size_t s_part = sizeof(float) * pairs * ksplit * static_cast<size_t>(fb_cap) * d_model;
  const size_t o_opnd = take(std::max(s_hfb + s_dyg + s_xg + s_gufb + s_dhfb, s_part));
  const size_t o_hfb = o_opnd, o_dyg = o_hfb + s_hfb, o_xg = o_dyg + s_dyg;
  const size_t o_gufb = o_xg + s_xg, o_dhfb = o_gufb + s_gufb;
  const size_t o_part = o_opnd;
  const size_t o_beg = take(sizeof(int32_t) * static_cast<size_t>(d_ff));
  const size_t o_end = take(sizeof(int32_t) * static_cast<size_t>(d_ff));
  const size_t o_rows = take(sizeof(int32_t) * cells);
  const size_t o_h = take(sizeof(uint16_t) * cells);
  const size_t o_dz = take(sizeof(float) * cells);
  const size_t o_cnt = take(sizeof(int32_t) * 8);  // row counters, one per dX gather pass
  const size_t o_duhl = gated ? take(sizeof(uint16_t) * 2 * padf) : 0;
  const size_t o_du = gated ? take(sizeof(float) * cells) : 0;
  const int dx_passes = gated ? spmm_pair_passes(d_model, d_ff, T) : 1;
  const size_t o_dxacc = dx_passes > 1 ? take(sizeof(float) * static_cast<size_t>(N) * d_model) : 0;
  if (ws && base) {
    uint8_t* b = static_cast<uint8_t*>(base);
    ws->dz_cells = reinterpret_cast<float*>(b + o_dzc);
    ws->dz_hl = reinterpret_cast<uint16_t*>(b + o_hl);
    ws->hfb = reinterpret_cast<uint16_t*>(b + o_hfb);
    ws->dyg = reinterpret_cast<uint16_t*>(b + o_dyg);
    ws->xg2 = reinterpret_cast<uint16_t*>(b + o_xg);
    ws->fb_pad = fb_pad;
    ws->part = reinterpret_cast<float*>(b + o_part);
    ws->ksplit = ksplit;
    ws->col_beg = reinterpret_cast<int32_t*>(b + o_beg);
    ws->col_end = reinterpret_cast<int32_t*>(b + o_end);
    ws->col_rows = reinterpret_cast<int32_t*>(b + o_rows);
    ws->col_h = reinterpret_cast<uint16_t*>(b + o_h);
    ws->col_dz = reinterpret_cast<float*>(b + o_dz);
    ws->row_counter = reinterpret_cast<int32_t*>(b + o_cnt);
    ws->du_hl = gated ? reinterpret_cast<uint16_t*>(b + o_duhl) : nullptr;
    ws->gu_fb = gated ? reinterpret_cast<float*>(b + o_gufb) : nullptr;
    ws->dh_fb = gated ? reinterpret_cast<float*>(b + o_dhfb) : nullptr;
    ws->col_du = gated ? reinterpret_cast<float*>(b + o_du) : nullptr;
    ws->dx_acc = dx_passes > 1 ? reinterpret_cast<float*>(b + o_dxacc) : nullptr;
    ws->dx_passes = dx_passes;
  }
  return off;
}

#define TW_CHECK_LAUNCH()                                         \
  do {                                                            \
    if (cudaGetLastError() != cudaSuccess) return TWELL_ERR_CUDA; \
  } while (0)
#define TW_TRY_RC(expr)              \
  do {                               \
    const int rc_ = (expr);          \
    if (rc_ != TWELL_OK) return rc_; \
  } while (0)

int launch_bwd(const uint16_t* X, const uint16_t* W_inT, const uint16_t* W_down, const twell_t& Lh,
               const uint16_t* dY, float lambda, uint16_t* dX, float* dW_inT, float* dW_down, float* db,
               int d, const BwdWorkspace& ws, cudaStream_t s, bool row_view, const GatedBwd* gt) {
  const Layout L = flat(Lh);
  const int f = Lh.d_ff;
  const int N = Lh.n_rows;
  const bool fb = Lh.fb_cap > 0 && N > 0;
  const int fb_grid = std::max(1, std::min(2 * ws.fb_pad, 2 * sm_count()));
  // Second stream: the fallback rows' weight-gradient share (stored into dW
  // first), then dX (the TwELL rows' gather-SpMM, then the fallback rows' GEMM).  This
  // stream: the SDDMM, the unit-major lists (independent of the fallback share), then
  // dw_unitcta_kernel adds the TwELL share once the fallback share is in place.
  AuxFork fork(s);
  TW_TRY_RC(fork.status());
  cudaStream_t a = fork.aux();
  if (gt && fb) {
    // gated, beside the SDDMM: the fallback rows' operands, then their g and
    // u, recomputed on the tensor cores from the gathered X rows (row s of xg2
    // read with stride 2 d_model)
    {
      LaunchScope ls(TWELL_KERNEL_DW_FALLBACK, a);
      fb_operands_kernel<<<fb_grid, 256, 0, a>>>(L, X, dY, d, ws.hfb, ws.dyg, ws.xg2, ws.dz_hl, ws.fb_pad, ws.du_hl);
    }
    TW_CHECK_LAUNCH();
    GUEpiParams gp{gt->b, ws.gu_fb, f};
    TW_TRY_RC(launch_gemm_gu(ws.xg2, 2 * static_cast<int64_t>(d), W_inT, gt->W_uT, Lh.fb_cap, Lh.n_fb, f, d, gp,
                             Lh.status, TWELL_KERNEL_DW_FALLBACK, a));
  }
  if (N > 0) {
    // dZ at the pattern (and dense for fallback rows: its bf16 parts, or the
    // gated layer's dh')
    SampleEpiParams sp{Lh.values, Lh.idx,   Lh.counts, Lh.row_fb, Lh.fb_dense, Lh.fb_cap,
                       f / Lh.tile, Lh.tile, Lh.cap,   f,         lambda,      ws.dz_cells,
                       ws.dz_hl,    gt ? gt->gu : nullptr, gt ? ws.dh_fb : nullptr};
    // its CTA 0 also zeroes the dX gather's row counters
    TW_TRY_RC(launch_gemm_sample(dY, W_down, N, f, d, sp, Lh.status, s, ws.row_counter, ws.dx_passes));
  }
  TW_TRY_RC(fork.aux_wait_main());  // the SDDMM's outputs are in
  if (fb) {
    if (gt) {
      LaunchScope ls(TWELL_KERNEL_DW_FALLBACK, a);
      gated_fb_parts_kernel<<<std::max(1, std::min(Lh.fb_cap, 2 * sm_count())), 256, 0, a>>>(L, ws.dh_fb, ws.gu_fb,
                                                                                          ws.dz_hl, ws.du_hl);
    } else {
      LaunchScope ls(TWELL_KERNEL_DW_FALLBACK, a);
      fb_operands_kernel<<<fb_grid, 256, 0, a>>>(L, X, dY, d, ws.hfb, ws.dyg, ws.xg2, ws.dz_hl, ws.fb_pad, nullptr);
    }
    TW_CHECK_LAUNCH();
    TW_TRY_RC(launch_gemm_store_mn(ws.hfb, ws.dyg, f, d, ws.fb_pad, Lh.n_fb, 1, dW_down, d, Lh.status,
                                   TWELL_KERNEL_DW_FALLBACK, a));
    // K = (slot, part): the high and low parts of dZ against X twice
    TW_TRY_RC(launch_gemm_store_mn(ws.dz_hl, ws.xg2, f, d, 2 * ws.fb_pad, Lh.n_fb, 2, dW_inT, d, Lh.status,
                                   TWELL_KERNEL_DW_FALLBACK, a));
    if (gt)
      TW_TRY_RC(launch_gemm_store_mn(ws.du_hl, ws.xg2, f, d, 2 * ws.fb_pad, Lh.n_fb, 2, gt->dW_uT, d, Lh.status,
                                     TWELL_KERNEL_DW_FALLBACK, a));
  }
  TW_TRY_RC(fork.mark_aux());  // dW holds the fallback share from here on
  if (N > 0) {
    // the TwELL rows' dX gather first: it needs only the SDDMM's output and,
    // queued after the fallback rows' dX, it waited for SMs held by the dW walk
    if (gt)
      TW_TRY_RC(launch_spmm_f32x2(Lh, ws.dz_cells, W_inT, gt->W_uT, d, dX, ws.row_counter, ws.dx_acc, ws.dx_passes,
                                  TWELL_KERNEL_DX, a));
    else
      TW_TRY_RC(launch_spmm_f32(Lh, ws.dz_cells, W_inT, d, dX, ws.row_counter, TWELL_KERNEL_DX, a));
    if (fb) {
      // one GEMM over K = 2 d_ff: row s of dz_hl viewed with stride 2 d_ff is
      // [high_s | low_s], and both halves meet the same W_in^T rows (K wraps);
      // gated: a second GEMM of dU's parts with W_u^T into the next ksplit splits
      const int64_t split = static_cast<int64_t>(Lh.fb_cap) * d;
      PartialEpiParams pp{ws.part, d, split};
      TW_TRY_RC(launch_gemm_partial_nmajor(ws.dz_hl, W_inT, Lh.fb_cap, Lh.n_fb, d, 2 * f, ws.ksplit, pp, Lh.status,
                                           TWELL_KERNEL_DX_FALLBACK, a, 2 * static_cast<int64_t>(f), f));
      if (gt) {
        PartialEpiParams pu{ws.part + ws.ksplit * split, d, split};
        TW_TRY_RC(launch_gemm_partial_nmajor(ws.du_hl, gt->W_uT, Lh.fb_cap, Lh.n_fb, d, 2 * f, ws.ksplit, pu,
                                             Lh.status, TWELL_KERNEL_DX_FALLBACK, a, 2 * static_cast<int64_t>(f), f));
      }
      TW_TRY_RC(launch_fb_reduce(Lh, ws.part, gt ? 2 * ws.ksplit : ws.ksplit, d, dX, TWELL_KERNEL_DX_FALLBACK, a));
    }
  }
  // ---- weight gradients: TwELL entries regrouped by hidden unit (a CTA per tile)
  const size_t lsm = unit_lists_smem(Lh.tile);
  auto lk = Lh.cap == 8 ? (gt ? unit_lists_kernel<true, true> : unit_lists_kernel<true, false>)
                        : (gt ? unit_lists_kernel<false, true> : unit_lists_kernel<false, false>);
  if (set_max_dynamic_smem(reinterpret_cast<const void*>(lk), static_cast<int>(unit_lists_smem(256))) != TWELL_OK)
    return TWELL_ERR_CUDA;
  {
    LaunchScope ls(TWELL_KERNEL_AUX, s);
    if (launch_pdl(lk, dim3(f / Lh.tile), dim3(kListWarps * 32), lsm, s, L, ws.dz_cells, ws.col_beg, ws.col_end,
                   ws.col_rows, ws.col_h, ws.col_dz, row_view ? Lh.row_fb : nullptr,
                   gt ? ws.col_du : nullptr) != cudaSuccess)
      return TWELL_ERR_CUDA;
  }
  TW_CHECK_LAUNCH();
  TW_TRY_RC(fork.main_wait_mark());  // the fallback share is in dW before the TwELL share is added
  {
    LaunchScope ls(TWELL_KERNEL_DW, s);
    const int grid = std::max(1, std::min(f, (gt ? 2 : 3) * sm_count()));
    auto wk = gt ? dw_unitcta_kernel<true> : dw_unitcta_kernel<false>;
    wk<<<grid, kWarps * 32, 0, s>>>(f, ws.col_beg, ws.col_end, ws.col_rows, ws.col_h, ws.col_dz, X, dY, d, dW_inT,
                                   dW_down, db, Lh.n_fb, fb ? Lh.fb_cap : 0, gt ? ws.col_du : nullptr,
                                   gt ? gt->dW_uT : nullptr);
  }
  TW_CHECK_LAUNCH();
  if (fb) {
    LaunchScope ls(TWELL_KERNEL_DW_FALLBACK, s);
    if (launch_pdl(fb_db_kernel, dim3((f + 31) / 32), dim3(256), 0, s, L, ws.dz_hl, db) != cudaSuccess)
      return TWELL_ERR_CUDA;
  }
  TW_CHECK_LAUNCH();
  TW_TRY_RC(fork.join());
  return TWELL_OK;
}

}  // namespace twell
