// Forward-pass kernels around the tensor-core up-projection:
//   route_kernel     hybrid routing: rows whose tiles overflowed C become
//                    fallback rows, numbered in ascending row order
//                    (ifai.io news, "Reshaping math for the GPU": a dense
//                    matrix catches the rare dense tokens; bayesiansapien note,
//                    Figure 1 "hybrid" splits rows between formats)
//   fb_assemble_kernel builds each fallback row of fb_dense from its cells:
//                    tiles that overflowed were spilled densely by the
//                    up-projection's epilogue, the others hold <= C entries;
//                    the row's cells are then cleared
//   fb_reduce_kernel Y rows of the fallback rows: the K-split partial sums of
//                    fb_dense . W_down (tensor cores) added in split order
#include <cuda_runtime.h>

#include <algorithm>

#include "sm103.cuh"
#include "twell_internal.h"

namespace twell {
namespace {

// Flat copy of the layout for kernel parameters.
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

constexpr int kRouteThreads = 1024;
constexpr int kRouteRows = 8;  // rows per thread per pass

// Rows variant: row_fb holds overflow flags on entry (1 for a flagged row,
// `empty` for the others: 0 after twell_pack, -1 in the forward) and -1 /
// fallback slot on exit.  With empty = -1 a reader that only asks "is this a
// fallback row" (row_fb >= 0) gets the same answer before, during and after
// routing, so the forward's gather-SpMM need not wait for it.  Tiles variant: row_fb holds each row's number of dense tiles
// on entry and, on exit, the pool slot of the row's first dense tile (-1 for
// rows without one); n_fb counts the dense tiles.  One CTA: an exclusive
// block scan gives the slots in ascending row order, so the result is
// deterministic.
__global__ void __launch_bounds__(kRouteThreads) route_kernel(Layout L, int32_t empty, int clear_past) {
  __shared__ int warp_tot[kRouteThreads / 32];
  __shared__ int base_s;
  grid_dependency_wait();
  const bool tiles = L.hybrid == TWELL_HYBRID_TILES;
  const int64_t cap = tiles ? static_cast<int64_t>(L.fb_cap) * L.nt : L.fb_cap;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) base_s = 0;
  __syncthreads();
  for (int start = 0; start < L.N; start += kRouteThreads * kRouteRows) {
    const int r0 = start + tid * kRouteRows;
    int cnt[kRouteRows];
    int local = 0;
#pragma unroll
    for (int i = 0; i < kRouteRows; ++i) {
      const int r = r0 + i;
      const int v = r < L.N ? L.row_fb[r] : (tiles ? 0 : empty);
      cnt[i] = tiles ? v : (v != empty ? 1 : 0);
      local += cnt[i];
    }
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      int w = warp_tot[lane];
      int wi = w;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, wi, o);
        if (lane >= o) wi += v;
      }
      warp_tot[lane] = wi - w;  // exclusive prefix of warp totals
    }
    __syncthreads();
    int slot = base_s + warp_tot[warp] + incl - local;
#pragma unroll
    for (int i = 0; i < kRouteRows; ++i) {
      const int r = r0 + i;
      if (r >= L.N) break;
      if (tiles) {
        L.row_fb[r] = cnt[i] > 0 ? slot : -1;
      } else if (cnt[i]) {
        L.row_fb[r] = slot;
        if (slot < L.fb_cap) {
          L.fb_rows[slot] = r;
        } else if (clear_past) {
          // past the capacity (an error the status word reports): the row is
          // not stored anywhere, but its cells still become empty
          const int64_t cell0 = static_cast<int64_t>(r) * L.nt;
          for (int c = 0; c < L.nt; ++c) L.counts[cell0 + c] = 0;
          for (int c = 0; c < L.nt * L.C; ++c) {
            L.values[cell0 * L.C + c] = 0;
            L.idx[cell0 * L.C + c] = 0;
          }
        }
      } else {
        L.row_fb[r] = -1;
      }
      slot += cnt[i];
    }
    __syncthreads();
    if (tid == kRouteThreads - 1) base_s = slot;
    __syncthreads();
  }
  if (tid == 0) {
    *L.n_fb = base_s;
    if (base_s > cap) report_error(L.status, TWELL_ERR_FALLBACK_OVERFLOW);
  }
}

// Tiles variant, before routing: a row flagged by the pack (row_fb != 0) gets
// its number of dense tiles (cells marked 255).  A warp per row, grid-stride.
__global__ void __launch_bounds__(256) tile_count_kernel(Layout L) {
  const int lane = threadIdx.x & 31;
  const int64_t gw0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t gws = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  for (int64_t r = gw0; r < L.N; r += gws) {
    if (L.row_fb[r] == 0) continue;
    int n = 0;
    for (int t0 = 0; t0 < L.nt; t0 += 32) {
      const int t = t0 + lane;
      const bool dense = t < L.nt && L.counts[r * L.nt + t] == TWELL_DENSE_TILE;
      n += __popc(__ballot_sync(0xffffffffu, dense));
    }
    if (lane == 0) L.row_fb[r] = n;
  }
}

// Tiles variant, after routing: each dense tile of a row takes the next pool
// slot (row_fb = the row's first slot) in tile order; its T values are copied
// into the pool from the dense H (standalone pack) or from the spill buffer
// the up-projection wrote (fused forward, spill index in the cell's first
// entry), and the cell's first entry becomes the pool slot.  A dense tile past
// the pool's capacity leaves an empty cell.  row_fb ends at -1 for every row.
__global__ void __launch_bounds__(256)
    tile_assign_kernel(Layout L, const uint16_t* __restrict__ H, int64_t ldh, const uint16_t* __restrict__ spill,
                       int32_t spill_cap) {
  const int lane = threadIdx.x & 31;
  const int64_t cap = static_cast<int64_t>(L.fb_cap) * L.nt;
  const int vec = L.T / 8;  // 16-byte vectors per tile
  const int64_t gw0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t gws = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  for (int64_t r = gw0; r < L.N; r += gws) {
    const int base = L.row_fb[r];
    if (base < 0) continue;
    int64_t slot = base;
    for (int t0 = 0; t0 < L.nt; t0 += 32) {
      const int tl = t0 + lane;
      unsigned m = __ballot_sync(0xffffffffu, tl < L.nt && L.counts[r * L.nt + tl] == TWELL_DENSE_TILE);
      while (m) {
        const int t = t0 + __ffs(m) - 1;
        m &= m - 1;
        const int64_t cell = r * L.nt + t;
        if (slot < cap) {
          uint4* dst = reinterpret_cast<uint4*>(L.fb_dense + slot * L.T);
          if (spill) {
            const uint32_t s24 = static_cast<uint32_t>(L.values[cell * L.C]) |
                                 (static_cast<uint32_t>(L.idx[cell * L.C]) << 16);
            const bool have = s24 < static_cast<uint32_t>(spill_cap);
            const uint4* src = reinterpret_cast<const uint4*>(spill + static_cast<int64_t>(s24) * L.T);
            for (int q = lane; q < vec; q += 32) dst[q] = have ? src[q] : make_uint4(0, 0, 0, 0);
          } else {
            const uint4* src = reinterpret_cast<const uint4*>(H + r * ldh + static_cast<int64_t>(t) * L.T);
            for (int q = lane; q < vec; q += 32) dst[q] = src[q];
          }
        }
        __syncwarp();  // the spill index is read before the cell is rewritten
        const bool keep = slot < cap;
        for (int q = lane; q < L.C; q += 32) {
          L.values[cell * L.C + q] = (keep && q == 0) ? static_cast<uint16_t>(slot & 0xFFFF) : 0;
          L.idx[cell * L.C + q] = (keep && q == 0) ? static_cast<uint8_t>((slot >> 16) & 0xFF) : 0;
        }
        if (lane == 0 && !keep) L.counts[cell] = 0;
        __syncwarp();
        ++slot;
      }
    }
    if (lane == 0) L.row_fb[r] = -1;
  }
}

// A warp per (fallback slot, tile), grid-stride over all of them: the dense
// tile comes from the spill buffer when the cell overflowed, else it is
// rebuilt from the cell's entries; then the cell becomes empty (count 0,
// padding).  Every (slot, tile) is independent, so the few fallback rows still
// spread over the whole GPU.
__global__ void __launch_bounds__(256)
    fb_assemble_kernel(Layout L, const uint16_t* __restrict__ spill, int32_t spill_cap) {
  grid_dependency_wait();
  const int nfb = min(*L.n_fb, L.fb_cap);
  const int lane = threadIdx.x & 31;
  const int vec = L.T / 8;  // 16-byte vectors per tile
  const int64_t items = static_cast<int64_t>(nfb) * L.nt;
  const int64_t gw0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t gws = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  for (int64_t it = gw0; it < items; it += gws) {
    const int slot = static_cast<int>(it / L.nt), t = static_cast<int>(it % L.nt);
    const int row = L.fb_rows[slot];
    uint16_t* out_row = L.fb_dense + static_cast<int64_t>(slot) * L.f;
    const int64_t cell = static_cast<int64_t>(row) * L.nt + t;
    const int cnt = L.counts[cell];
    uint4* dst = reinterpret_cast<uint4*>(out_row + static_cast<int64_t>(t) * L.T);
    if (cnt == kSpilledCell) {
      const uint32_t s24 = static_cast<uint32_t>(L.values[cell * L.C]) |
                           (static_cast<uint32_t>(L.idx[cell * L.C]) << 16);
      const bool have = s24 < static_cast<uint32_t>(spill_cap);
      const uint4* src = reinterpret_cast<const uint4*>(spill + static_cast<int64_t>(s24) * L.T);
      for (int q = lane; q < vec; q += 32) dst[q] = have ? src[q] : make_uint4(0, 0, 0, 0);
    } else {
      for (int q = lane; q < vec; q += 32) dst[q] = make_uint4(0, 0, 0, 0);
      __syncwarp();
      if (lane < cnt) out_row[static_cast<int64_t>(t) * L.T + L.idx[cell * L.C + lane]] = L.values[cell * L.C + lane];
    }
    __syncwarp();
    if (lane == 0) L.counts[cell] = 0;
    for (int q = lane; q < L.C; q += 32) {
      L.values[cell * L.C + q] = 0;
      L.idx[cell * L.C + q] = 0;
    }
    __syncwarp();
  }
}

__device__ __forceinline__ uint4 pack8_bf16(const float (&a)[8]) {
  uint32_t p[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    p[i] = static_cast<uint32_t>(float_to_bf16_bits(a[2 * i])) |
           (static_cast<uint32_t>(float_to_bf16_bits(a[2 * i + 1])) << 16);
  return make_uint4(p[0], p[1], p[2], p[3]);
}

// Y[fb_rows[r]] = bf16(sum over splits of part[ks][r]), splits in order.
__global__ void fb_reduce_kernel(Layout L, const float* __restrict__ part, int ksplit, int d,
                                 uint16_t* __restrict__ Y) {
  grid_dependency_wait();
  const int nfb = min(*L.n_fb, L.fb_cap);
  const int64_t stride = static_cast<int64_t>(L.fb_cap) * d;
  for (int slot = blockIdx.x; slot < nfb; slot += gridDim.x) {
    const int row = L.fb_rows[slot];
    for (int c = threadIdx.x * 8; c < d; c += blockDim.x * 8) {
      float a[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      for (int ks = 0; ks < ksplit; ++ks) {
        const float4* src = reinterpret_cast<const float4*>(part + ks * stride + static_cast<int64_t>(slot) * d + c);
        const float4 x = src[0], y = src[1];
        a[0] += x.x; a[1] += x.y; a[2] += x.z; a[3] += x.w;
        a[4] += y.x; a[5] += y.y; a[6] += y.z; a[7] += y.w;
      }
      *reinterpret_cast<uint4*>(Y + static_cast<int64_t>(row) * d + c) = pack8_bf16(a);
    }
  }
}

// Column sums of a bf16 matrix, deterministic: block (column block of 256,
// row chunk) sums its rows per column in fp32 (warp w takes rows w, w + 8, ...;
// the 8 warps' sums are added in warp order), then one thread per column adds
// the chunks' partial sums in chunk order.
__global__ void __launch_bounds__(256)
    colsum_part_kernel(const uint16_t* __restrict__ Z, int M, int N, int rows_per_chunk, float* __restrict__ part) {
  __shared__ float red[8][256];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c0 = blockIdx.x * 256 + lane * 8;
  const int r0 = blockIdx.y * rows_per_chunk, r1 = min(M, r0 + rows_per_chunk);
  float a[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  if (c0 < N) {
#pragma unroll 4
    for (int r = r0 + warp; r < r1; r += 8) {
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(Z + static_cast<int64_t>(r) * N + c0));
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int k = 0; k < 8; ++k) a[k] += (k & 1) ? bf16_hi(w[k / 2]) : bf16_lo(w[k / 2]);
    }
  }
#pragma unroll
  for (int k = 0; k < 8; ++k) red[warp][lane * 8 + k] = a[k];
  __syncthreads();
  const int c = blockIdx.x * 256 + threadIdx.x;
  if (c < N) {
    float sum = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) sum += red[w][threadIdx.x];
    part[static_cast<int64_t>(blockIdx.y) * N + c] = sum;
  }
}

__global__ void colsum_final_kernel(const float* __restrict__ part, int chunks, int N, float* __restrict__ out) {
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= N) return;
  float sum = 0.f;
  for (int k = 0; k < chunks; ++k) sum += part[static_cast<int64_t>(k) * N + c];
  out[c] = sum;
}

}  // namespace

int launch_tile_count(const twell_t& L, cudaStream_t s) {
  if (L.n_rows <= 0) return TWELL_OK;
  const int grid = std::max(1, std::min((L.n_rows + 7) / 8, 4 * sm_count()));
  LaunchScope ls(TWELL_KERNEL_ROUTE, s);
  tile_count_kernel<<<grid, 256, 0, s>>>(flat(L));
  return cudaGetLastError() == cudaSuccess ? TWELL_OK : TWELL_ERR_CUDA;
}

int launch_tile_assign(const twell_t& L, const uint16_t* H, int64_t ldh, const uint16_t* spill, int32_t spill_cap,
                       cudaStream_t s) {
  if (L.n_rows <= 0) return TWELL_OK;
  const int grid = std::max(1, std::min((L.n_rows + 7) / 8, 4 * sm_count()));
  LaunchScope ls(TWELL_KERNEL_FB_ASSEMBLE, s);
  tile_assign_kernel<<<grid, 256, 0, s>>>(flat(L), H, ldh, spill, spill_cap);
  return cudaGetLastError() == cudaSuccess ? TWELL_OK : TWELL_ERR_CUDA;
}

int launch_route(const twell_t& L, cudaStream_t s, int32_t empty, bool clear_past) {
  LaunchScope ls(TWELL_KERNEL_ROUTE, s);
  if (launch_pdl(route_kernel, dim3(1), dim3(kRouteThreads), 0, s, flat(L), empty, clear_past ? 1 : 0) !=
      cudaSuccess)
    return TWELL_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? TWELL_OK : TWELL_ERR_CUDA;
}

// ---- row view of a tile-granular layout (the backward's input): a row that
// holds a dense tile becomes a fallback row of the view, with its dense h
// assembled from its cells and its pool tiles; its cells are not touched.

// flags[r] = 1 when row r holds a dense tile, else 0.  A warp per row.
__global__ void __launch_bounds__(256) tile_row_flags_kernel(Layout L, int32_t* __restrict__ flags) {
  grid_dependency_wait();
  const int lane = threadIdx.x & 31;
  const int64_t gw0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t gws = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  for (int64_t r = gw0; r < L.N; r += gws) {
    bool dense = false;
    for (int t = lane; t < L.nt; t += 32) dense |= L.counts[r * L.nt + t] == TWELL_DENSE_TILE;
    dense = __any_sync(0xffffffffu, dense);
    if (lane == 0) flags[r] = dense ? 1 : 0;
  }
}

// The dense h of each routed row of the view (slots below min(n_fb, cap)): a
// CTA per slot zeroes the row, then writes each cell's stored entries or
// copies its pool tile (indices bounded by T, slots by the pool).
__global__ void __launch_bounds__(256) tile_rows_assemble_kernel(Layout L, const int32_t* __restrict__ v_rows,
                                                                 const int32_t* __restrict__ v_n, int v_cap,
                                                                 uint16_t* __restrict__ dense) {
  grid_dependency_wait();
  const int n = min(*v_n, v_cap);
  const int64_t pool = static_cast<int64_t>(L.fb_cap) * L.nt;
  for (int slot = blockIdx.x; slot < n; slot += gridDim.x) {
    const int r = v_rows[slot];
    uint16_t* out = dense + static_cast<int64_t>(slot) * L.f;
    for (int i = threadIdx.x; i < L.f / 8; i += blockDim.x)
      reinterpret_cast<uint4*>(out)[i] = make_uint4(0u, 0u, 0u, 0u);
    __syncthreads();
    for (int t = threadIdx.x; t < L.nt; t += blockDim.x) {
      const int64_t cell = static_cast<int64_t>(r) * L.nt + t;
      const int cnt = L.counts[cell];
      uint16_t* o = out + static_cast<int64_t>(t) * L.T;
      if (cnt == TWELL_DENSE_TILE) {
        const int64_t ps = static_cast<int64_t>(L.values[cell * L.C]) | (static_cast<int64_t>(L.idx[cell * L.C]) << 16);
        if (ps < pool)
          for (int k = 0; k < L.T; ++k) o[k] = L.fb_dense[ps * L.T + k];
      } else {
        for (int sl = 0; sl < min(cnt, L.C); ++sl) {
          const int j = L.idx[cell * L.C + sl];
          if (j < L.T) o[j] = L.values[cell * L.C + sl];
        }
      }
    }
    __syncthreads();  // the next slot's zeroing comes after these writes
  }
}

int launch_tile_row_view(const twell_t& H, const twell_t& V, cudaStream_t s) {
  if (H.n_rows <= 0) return TWELL_OK;
  {
    const int grid = std::max(1, std::min((H.n_rows + 7) / 8, 4 * sm_count()));
    LaunchScope ls(TWELL_KERNEL_AUX, s);
    if (launch_pdl(tile_row_flags_kernel, dim3(grid), dim3(256), 0, s, flat(H), V.row_fb) != cudaSuccess)
      return TWELL_ERR_CUDA;
  }
  if (cudaGetLastError() != cudaSuccess) return TWELL_ERR_CUDA;
  // slots in ascending row order; a row past the view's capacity is reported
  // (overflow status) and its cells are left as they are
  const int rc = launch_route(V, s, 0, false);
  if (rc != TWELL_OK) return rc;
  if (V.fb_cap <= 0) return TWELL_OK;
  const int grid = std::max(1, std::min(V.fb_cap, 2 * sm_count()));
  LaunchScope ls(TWELL_KERNEL_AUX, s);
  if (launch_pdl(tile_rows_assemble_kernel, dim3(grid), dim3(256), 0, s, flat(H), V.fb_rows, V.n_fb, V.fb_cap,
                 V.fb_dense) != cudaSuccess)
    return TWELL_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? TWELL_OK : TWELL_ERR_CUDA;
}

int launch_fb_assemble(const twell_t& L, const uint16_t* spill, const int32_t* /*spill_count*/,
                       int32_t spill_cap, cudaStream_t s) {
  if (L.fb_cap <= 0) return TWELL_OK;
  const int64_t warps = static_cast<int64_t>(L.fb_cap) * (L.d_ff / L.tile);
  const int grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>((warps + 7) / 8, 4 * sm_count())));
  LaunchScope ls(TWELL_KERNEL_FB_ASSEMBLE, s);
  if (launch_pdl(fb_assemble_kernel, dim3(grid), dim3(256), 0, s, flat(L), spill, spill_cap) != cudaSuccess)
    return TWELL_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? TWELL_OK : TWELL_ERR_CUDA;
}

int launch_fb_down(const twell_t& L, const uint16_t* W_down, int d_model, uint16_t* Y, float* part, int ksplit,
                   cudaStream_t s) {
  if (L.fb_cap <= 0) return TWELL_OK;
  PartialEpiParams pp{part, d_model, static_cast<int64_t>(L.fb_cap) * d_model};
  int rc = launch_gemm_partial_nmajor(L.fb_dense, W_down, L.fb_cap, L.n_fb, d_model, L.d_ff, ksplit, pp, L.status,
                                      TWELL_KERNEL_FB_DOWN, s);
  if (rc != TWELL_OK) return rc;
  return launch_fb_reduce(L, part, ksplit, d_model, Y, TWELL_KERNEL_FB_DOWN, s);
}

int launch_fb_reduce(const twell_t& L, const float* part, int nsplit, int d_model, uint16_t* out, int kernel_id,
                     cudaStream_t s) {
  if (L.fb_cap <= 0) return TWELL_OK;
  const int grid = std::max(1, std::min(L.fb_cap, 2 * sm_count()));
  LaunchScope ls(kernel_id, s);
  if (launch_pdl(fb_reduce_kernel, dim3(grid), dim3(256), 0, s, flat(L), part, nsplit, d_model, out) != cudaSuccess)
    return TWELL_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? TWELL_OK : TWELL_ERR_CUDA;
}

}  // namespace twell

namespace twell {

int launch_colsum_bf16(const uint16_t* Z, int M, int N, float* part, float* out, int kernel_id, cudaStream_t s) {
  if (N <= 0) return TWELL_OK;
  if (N % 8 != 0) return TWELL_ERR_UNSUPPORTED;
  const int rows_per_chunk = std::max(1, (M + kColsumChunks - 1) / kColsumChunks);
  {
    LaunchScope ls(kernel_id, s);
    colsum_part_kernel<<<dim3((N + 255) / 256, kColsumChunks), 256, 0, s>>>(Z, M, N, rows_per_chunk, part);
  }
  if (cudaGetLastError() != cudaSuccess) return TWELL_ERR_CUDA;
  LaunchScope ls(kernel_id, s);
  colsum_final_kernel<<<(N + 255) / 256, 256, 0, s>>>(part, kColsumChunks, N, out);
  return cudaGetLastError() == cudaSuccess ? TWELL_OK : TWELL_ERR_CUDA;
}

}  // namespace twell
