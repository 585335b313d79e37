// Hybrid routing shared by its own launch (route_kernel) and the fused
// up-projection's last CTA: rows whose tiles overflowed C become fallback rows,
// numbered in ascending row order (ifai.io news, "Reshaping math for the GPU":
// a dense matrix catches the rare dense tokens; bayesiansapien note, Figure 1
// "hybrid" splits rows between formats).
#pragma once

#include <cstdint>

#include "sm103.cuh"
#include "twell_internal.h"

namespace twell {

struct RouteRows {
  int32_t N, nt, C, fb_cap;
  bool tiles;
  uint16_t* values;
  uint8_t* idx;
  uint8_t* counts;
  int32_t* row_fb;
  int32_t* fb_rows;
  int32_t* n_fb;
  int32_t* status;
};

constexpr int kRouteRows = 8;  // rows per thread per pass

// Rows variant: row_fb holds 0/1 overflow flags on entry and -1 / fallback
// slot on exit.  Tiles variant: row_fb holds each row's number of dense tiles
// on entry and, on exit, the pool slot of the row's first dense tile (-1 for
// rows without one); n_fb counts the dense tiles.  Run by all kThreads threads
// of one CTA: an exclusive block scan gives the slots in ascending row order,
// so the result is deterministic.
template <int kThreads>
__device__ __forceinline__ void route_block(const RouteRows& L) {
  static_assert(kThreads % 32 == 0 && kThreads <= 1024, "whole warps");
  constexpr int kW = kThreads / 32;
  __shared__ int warp_tot[32];
  __shared__ int base_s;
  const bool tiles = L.tiles;
  const int64_t cap = tiles ? static_cast<int64_t>(L.fb_cap) * L.nt : L.fb_cap;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) base_s = 0;
  __syncthreads();
  for (int start = 0; start < L.N; start += kThreads * kRouteRows) {
    const int r0 = start + tid * kRouteRows;
    int cnt[kRouteRows];
    int local = 0;
#pragma unroll
    for (int i = 0; i < kRouteRows; ++i) {
      const int r = r0 + i;
      const int v = r < L.N ? L.row_fb[r] : 0;
      cnt[i] = tiles ? v : (v != 0 ? 1 : 0);
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
      const int w = lane < kW ? warp_tot[lane] : 0;
      int wi = w;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, wi, o);
        if (lane >= o) wi += v;
      }
      if (lane < kW) warp_tot[lane] = wi - w;  // exclusive prefix of warp totals
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
        } else {
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
    if (tid == kThreads - 1) base_s = slot;
    __syncthreads();
  }
  if (tid == 0) {
    *L.n_fb = base_s;
    if (base_s > cap) report_error(L.status, TWELL_ERR_FALLBACK_OVERFLOW);
  }
}

}  // namespace twell
