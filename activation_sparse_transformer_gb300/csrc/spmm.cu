// TwELL gather-SpMM:  out[n, :] = sum_t sum_{s < count[n,t]} v[n,t,s] * W[t*T + idx[n,t,s], :]
//
// The down-projection Y = H . W_down of the sparse layer reads only the W_down
// rows named by the stored tile-local indices (repo-explainer, "TwELL: The
// Packing Format That Fits the Machine": fused MLP execution from the packed
// form); the backward's dX = dZ . W_in^T has the same shape with fp32 values.
//
// At ~1% density a W row is used by ~1% of the tokens, so staging W slabs for
// a token block buys almost no reuse unless the block holds thousands of
// tokens (far more accumulators than an SM has registers).  The kernels are
// therefore built for memory-level parallelism instead.  The main one
// (spmm_rowcta_kernel) gives a CTA one token row at a time (a persistent grid,
// four CTAs per SM, rows handed out from a counter): the CTA flattens the row's stored entries (tile-major,
// slots ascending, so hidden units ascend) into one shared-memory list, and
// its eight warps stream the named W rows for 256-column blocks w, w + 8, ...
// with coalesced 16-byte loads, kU independent loads in flight per lane,
// accumulating in fp32 registers.  Each output sums its terms in ascending
// hidden-unit order.  Fallback rows are skipped: their rows of the output
// belong to the dense fallback path, which may run at the same time on
// another stream.
//
// spmm_row_kernel, a warp per (row, 256-column block), serves the two other
// cases.  The tile-granular hybrid: after a row's TwELL entries it gathers the
// non-zeros of the row's dense tiles from the tile pool.  Small batches: too
// few rows to fill the GPU, so the row's tiles are cut into gridDim.z
// consecutive ranges (each warp flattens and streams only its range); each
// range's fp32 sums go to a partial buffer, and the last CTA to finish among
// the ranges of a (row block, column block) adds them in range order (an
// arrival counter, no waiting).  A small batch's fallback rows are gathered
// here too, from the dense h its pack pass keeps, so no tensor-core fallback
// GEMM and reduction follow on the second stream.
//
// Two more uses of the row kernel.  Pair entries (float2 values) meet two
// weight matrices at once: the gated layer's dX = dG . W_g + dU . W_u.  And
// when the rows a gather may name are larger than L2 holds across one pass
// (two 117 MB matrices for the gated dX, or a 117 MB W_down), the gather runs
// in consecutive launches over tile ranges -- each range's weight rows stay in
// L2 for its launch -- with the fp32 sums carried between launches in range
// order (the last one writes bf16).
#include <cuda_runtime.h>

#include <algorithm>
#include <type_traits>

#include "sm103.cuh"
#include "twell_internal.h"

namespace twell {
namespace {

constexpr int kWarps = 8;  // rows per CTA
constexpr int kU = 8;      // W row loads in flight per lane
constexpr int kMaxDynSmem = 224 * 1024;  // entry lists; the rest of the 227 KB holds the static words

struct SpmmArgs {
  const void* values;     // [N][nt][C] VT
  const uint8_t* idx;     // [N][nt][C]
  const uint8_t* counts;  // [N][nt]
  const int32_t* row_fb;  // [N]: rows >= 0 are fallback rows, left to the fallback path
  uint16_t* out;          // [N][d] bf16
  float* part;            // [gridDim.z][N][d] fp32 when the tiles are split into ranges, else null
  int32_t* arrivals;      // [gridDim.x][gridDim.y] zeroed counters when the tiles are split
  const uint16_t* pool;   // tile-granular hybrid: the pool of dense tiles, else null
  int32_t* row_counter;   // zeroed word: rows handed out past the first gridDim.x, else null (fixed stride)
  int N, d, nt, T, C;
  int32_t* status;
  // small batches: every row's h as dense bf16 [N][nt * T]; the fallback rows
  // (row_fb >= 0) are then gathered from it here instead of by the fallback path
  const uint16_t* dense_h;
  // pair entries (float2 values): the second value multiplies this matrix's rows
  const uint16_t* W2;
  // the CTA-per-row kernel: tiles [t_lo, t_hi) only (t_hi == 0: all), and with
  // acc non-null the sums go through an fp32 [N][d] buffer: acc_mode 0 stores
  // them, 1 adds them to it, 2 adds them and writes the bf16 result to out
  int t_lo, t_hi;
  float* acc;
  int acc_mode;
};

// Entry of the per-warp list.  bf16 values: one word, hidden unit j in the low
// 16 bits and the value's bits in the high 16.  fp32 values: (j, value).
template <typename VT>
struct RowEntry;
template <>
struct RowEntry<uint16_t> {
  uint32_t w;
  static __device__ __forceinline__ RowEntry make(int j, uint16_t v) {
    return RowEntry{static_cast<uint32_t>(j) | (static_cast<uint32_t>(v) << 16)};
  }
  __device__ __forceinline__ int j() const { return static_cast<int>(w & 0xFFFFu); }
  __device__ __forceinline__ void fma(float (&acc)[8], const uint4& wr) const {
    fma8_bf16(acc, static_cast<uint16_t>(w >> 16), wr);
  }
};
template <>
struct RowEntry<float> {
  int32_t jj;
  float v;
  static __device__ __forceinline__ RowEntry make(int j, float val) { return RowEntry{j, val}; }
  __device__ __forceinline__ int j() const { return jj; }
  __device__ __forceinline__ void fma(float (&acc)[8], const uint4& wr) const { fma8_f32x2(acc, v, wr); }
};

// Pair entries (the gated layer's dX): (dG, dU) at hidden unit j meet the rows
// j of W_g^T and of W_u^T.
template <>
struct RowEntry<float2> {
  int32_t jj;
  float a, b;
  int32_t pad;
  static __device__ __forceinline__ RowEntry make(int j, float2 v) { return RowEntry{j, v.x, v.y, 0}; }
  __device__ __forceinline__ int j() const { return jj; }
};

__device__ __forceinline__ uint4 pack8_bf16(const float (&acc)[8]) {
  uint32_t p[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    p[i] = static_cast<uint32_t>(float_to_bf16_bits(acc[2 * i])) |
           (static_cast<uint32_t>(float_to_bf16_bits(acc[2 * i + 1])) << 16);
  return make_uint4(p[0], p[1], p[2], p[3]);
}

template <typename VT>
__device__ __forceinline__ VT from_bf16(uint16_t v);
template <>
__device__ __forceinline__ uint16_t from_bf16<uint16_t>(uint16_t v) { return v; }
template <>
__device__ __forceinline__ float from_bf16<float>(uint16_t v) { return bf16_bits_to_float(v); }

// acc += sum over list[0, total) of value x (W row j)[c0, c0 + 8), kU rows in flight.
template <typename VT>
__device__ __forceinline__ void stream_list(const SpmmArgs& a, const uint16_t* __restrict__ W, int c0,
                                            const RowEntry<VT>* list, int total, float (&acc)[8]) {
  const uint16_t* __restrict__ wcol = W + c0;
  if constexpr (std::is_same<VT, float2>::value) {
    // pairs: two W rows per entry, so half as many entries in flight
    constexpr int kU2 = kU / 2;
    const uint16_t* __restrict__ wcol2 = a.W2 + c0;
    int e = 0;
    for (; e + kU2 <= total; e += kU2) {
      uint4 w[kU2], w2[kU2];
      RowEntry<VT> en[kU2];
#pragma unroll
      for (int u = 0; u < kU2; ++u) {
        en[u] = list[e + u];
        w[u] = __ldg(reinterpret_cast<const uint4*>(wcol + static_cast<int64_t>(en[u].j()) * a.d));
        w2[u] = __ldg(reinterpret_cast<const uint4*>(wcol2 + static_cast<int64_t>(en[u].j()) * a.d));
      }
#pragma unroll
      for (int u = 0; u < kU2; ++u) {
        fma8_f32x2(acc, en[u].a, w[u]);
        fma8_f32x2(acc, en[u].b, w2[u]);
      }
    }
    for (; e < total; ++e) {
      const RowEntry<VT> en = list[e];
      fma8_f32x2(acc, en.a, __ldg(reinterpret_cast<const uint4*>(wcol + static_cast<int64_t>(en.j()) * a.d)));
      fma8_f32x2(acc, en.b, __ldg(reinterpret_cast<const uint4*>(wcol2 + static_cast<int64_t>(en.j()) * a.d)));
    }
  } else {
    int e = 0;
    for (; e + kU <= total; e += kU) {
      uint4 w[kU];
      RowEntry<VT> en[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        en[u] = list[e + u];
        w[u] = __ldg(reinterpret_cast<const uint4*>(wcol + static_cast<int64_t>(en[u].j()) * a.d));
      }
#pragma unroll
      for (int u = 0; u < kU; ++u) en[u].fma(acc, w[u]);
    }
    for (; e < total; ++e) {
      const RowEntry<VT> en = list[e];
      en.fma(acc, __ldg(reinterpret_cast<const uint4*>(wcol + static_cast<int64_t>(en.j()) * a.d)));
    }
  }
}

// Sum of one row's stored entries in tiles [t_beg, t_end) times the W rows
// they name, for this lane's 8 columns starting at c0 (the whole warp calls it
// for one row; inactive lanes only help flatten).  With dense = true the row
// is a fallback row of a small batch: its non-zeros come from the dense h
// (a.dense_h) instead of the cells, in ascending column order, streamed every
// time the list (max_entries) fills.
template <typename VT>
__device__ __forceinline__ void row_block_sum(const SpmmArgs& a, const uint16_t* __restrict__ W, RowEntry<VT>* list,
                                              int lane, int row, int c0, bool active, int t_beg, int t_end,
                                              float (&acc)[8], bool dense = false, int max_entries = 0) {
  const VT* vals = static_cast<const VT*>(a.values);
  const int64_t cell0 = static_cast<int64_t>(row) * a.nt;

  if (dense) {
    const uint16_t* hrow = a.dense_h + static_cast<int64_t>(row) * a.nt * a.T;
    int n = 0;
    for (int c = t_beg * a.T; c < t_end * a.T; c += 32) {  // T is a multiple of 32
      if (n + 32 > max_entries) {
        __syncwarp();
        if (active) stream_list<VT>(a, W, c0, list, n, acc);
        __syncwarp();  // the list is free again
        n = 0;
      }
      const uint16_t v = hrow[c + lane];
      const bool nz = (v & 0x7FFFu) != 0;
      const unsigned b = __ballot_sync(0xffffffffu, nz);
      if (nz) list[n + __popc(b & ((1u << lane) - 1u))] = RowEntry<VT>::make(c + lane, from_bf16<VT>(v));
      n += __popc(b);
    }
    __syncwarp();
    if (active) stream_list<VT>(a, W, c0, list, n, acc);
    __syncwarp();  // the list is rewritten by the warp's next item
    return;
  }

  // ---- flatten: tiles in order, 32 per round (dense tiles come after)
  int total = 0;
  for (int t0 = t_beg; t0 < t_end; t0 += 32) {
    const int t = t0 + lane;
    const int cnt_raw = t < t_end ? a.counts[cell0 + t] : 0;
    const int cnt = (a.pool && cnt_raw == TWELL_DENSE_TILE) ? 0 : cnt_raw;
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int x = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += x;
    }
    const int base = total + incl - cnt;
    const int64_t cell = cell0 + t;
    for (int s = 0; s < cnt; ++s)
      list[base + s] = RowEntry<VT>::make(t * a.T + a.idx[cell * a.C + s], vals[cell * a.C + s]);
    total += __shfl_sync(0xffffffffu, incl, 31);
  }
  __syncwarp();

  // ---- stream the named W rows, kU loads in flight
  if (active) stream_list<VT>(a, W, c0, list, total, acc);

  // ---- tile-granular hybrid: each dense tile's non-zeros, gathered the same way
  if (a.pool) {
    for (int t0 = t_beg; t0 < t_end; t0 += 32) {
      const int tl = t0 + lane;
      unsigned m = __ballot_sync(0xffffffffu, tl < t_end && a.counts[cell0 + tl] == TWELL_DENSE_TILE);
      while (m) {
        const int t = t0 + __ffs(m) - 1;
        m &= m - 1;
        const int64_t cell = cell0 + t;
        const int64_t slot = static_cast<int64_t>(static_cast<const uint16_t*>(a.values)[cell * a.C]) |
                             (static_cast<int64_t>(a.idx[cell * a.C]) << 16);
        const uint16_t* tile = a.pool + slot * a.T;
        __syncwarp();  // the list is free again
        int n = 0;
        for (int i0 = 0; i0 < a.T; i0 += 32) {
          const uint16_t v = tile[i0 + lane];
          const bool nz = (v & 0x7FFFu) != 0;
          const unsigned b = __ballot_sync(0xffffffffu, nz);
          if (nz) list[n + __popc(b & ((1u << lane) - 1u))] = RowEntry<VT>::make(t * a.T + i0 + lane, from_bf16<VT>(v));
          n += __popc(b);
        }
        __syncwarp();
        if (active) stream_list<VT>(a, W, c0, list, n, acc);
      }
    }
  }
  __syncwarp();  // the list is rewritten by the warp's next item
}

// max_entries = n_tiles * C bounds the entries a row can store.
//
// Whole rows (gridDim.z == 1): a persistent grid whose warps walk the (row,
// 256-column block) items with a fixed stride, so a warp that drew short rows
// takes the next item instead of idling until its CTA's longest row ends; the
// 8 warps of a CTA start on the 8 column blocks of one row.
template <typename VT>
__global__ void __launch_bounds__(kWarps * 32, 3)
    spmm_row_kernel(const SpmmArgs a, const uint16_t* __restrict__ W, int max_entries) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ int last_s;
  grid_dependency_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  RowEntry<VT>* list = reinterpret_cast<RowEntry<VT>*>(smem_raw) + warp * max_entries;

  if (gridDim.z == 1) {
    const int cbs = (a.d + 255) / 256;
    const int64_t items = static_cast<int64_t>(a.N) * cbs;
    for (int64_t it = static_cast<int64_t>(blockIdx.x) * kWarps + warp; it < items;
         it += static_cast<int64_t>(gridDim.x) * kWarps) {
      const int row = static_cast<int>(it / cbs);
      const bool fb_row = a.row_fb[row] >= 0;
      // written by the fallback path, which may run concurrently (unless gathered from dense h here)
      if (fb_row && !a.dense_h) continue;
      const int c0 = static_cast<int>(it % cbs) * 256 + lane * 8;
      const bool active = c0 < a.d;
      float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      row_block_sum<VT>(a, W, list, lane, row, c0, active, 0, a.nt, acc, fb_row, max_entries);
      if (active) *reinterpret_cast<uint4*>(a.out + static_cast<int64_t>(row) * a.d + c0) = pack8_bf16(acc);
    }
    return;
  }

  const int row = blockIdx.x * kWarps + warp;
  const bool fb_row = row < a.N && a.row_fb[row] >= 0;
  const bool work = row < a.N && (!fb_row || a.dense_h);
  const int c0 = blockIdx.y * 256 + lane * 8;
  const bool active = work && c0 < a.d;
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  if (work) {
    // this warp's range of tiles, one of gridDim.z consecutive ranges
    const int per = (a.nt + gridDim.z - 1) / gridDim.z;
    const int t_beg = min(a.nt, static_cast<int>(blockIdx.z) * per);
    const int t_end = min(a.nt, t_beg + per);
    row_block_sum<VT>(a, W, list, lane, row, c0, active, t_beg, t_end, acc, fb_row, max_entries);
  }

  // ---- tile ranges: store this range's sums; the CTA that finishes last among
  // the gridDim.z ranges of this (row block, column block) adds them in range
  // order and writes Y (no waiting: the others have already left)
  if (active) {
    float4* dst = reinterpret_cast<float4*>(a.part + (static_cast<int64_t>(blockIdx.z) * a.N + row) * a.d + c0);
    dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const int done = atomicAdd(a.arrivals + blockIdx.x * gridDim.y + blockIdx.y, 1);
    last_s = done == static_cast<int>(gridDim.z) - 1;
  }
  __syncthreads();
  if (!last_s || !active) return;
  __threadfence();
  float sum[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll 8
  for (int z = 0; z < static_cast<int>(gridDim.z); ++z) {
    const float4* src = reinterpret_cast<const float4*>(a.part + (static_cast<int64_t>(z) * a.N + row) * a.d + c0);
    const float4 x = __ldcg(src), y = __ldcg(src + 1);
    sum[0] += x.x; sum[1] += x.y; sum[2] += x.z; sum[3] += x.w;
    sum[4] += y.x; sum[5] += y.y; sum[6] += y.z; sum[7] += y.w;
  }
  *reinterpret_cast<uint4*>(a.out + static_cast<int64_t>(row) * a.d + c0) = pack8_bf16(sum);
}

// Whole rows, row-granular hybrid: a CTA per row at a time (persistent).
// Every 256-column block of a row gathers the same W rows, so the CTA
// flattens the row's entries once -- warp w expands tiles [w * tpw, (w + 1) *
// tpw), a CTA prefix over the warps' totals places them in ascending
// hidden-unit order -- and its 8 warps then stream column blocks w, w + 8, ...
// from that one shared list.  Rows are handed out dynamically (a CTA starts on
// row blockIdx.x and takes the next unclaimed row from a counter), so a CTA
// that drew long rows does not hold up the launch; the claim for the next row
// is issued when a row starts, so its latency hides under the row's loads.
template <typename VT>
__global__ void __launch_bounds__(kWarps * 32, 4)
    spmm_rowcta_kernel(const SpmmArgs a, const uint16_t* __restrict__ W) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ int warp_tot[kWarps + 1];
  __shared__ int next_row_s[2];  // by iteration parity: a skipped row has no barrier before the next write
  grid_dependency_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  RowEntry<VT>* list = reinterpret_cast<RowEntry<VT>*>(smem_raw);
  const VT* vals = static_cast<const VT*>(a.values);
  const int cbs = (a.d + 255) / 256;
  const int t_lo = a.t_lo, t_hi = a.t_hi > 0 ? a.t_hi : a.nt;
  const int tpw = (t_hi - t_lo + kWarps - 1) / kWarps;
  for (int row = blockIdx.x, it = 0; row < a.N; it ^= 1) {
    int claim = 0;
    if (threadIdx.x == 0)
      claim = a.row_counter ? static_cast<int>(gridDim.x) + atomicAdd(a.row_counter, 1) : row + gridDim.x;
    // fallback rows are written by the fallback path, which may run concurrently
    if (a.row_fb[row] < 0) {  // uniform over the CTA
      const int64_t cell0 = static_cast<int64_t>(row) * a.nt;
      const int t_beg = min(t_hi, t_lo + warp * tpw), t_end = min(t_hi, t_beg + tpw);
      // this warp's tiles: counts, warp prefix (rounds of 32 tiles)
      int wtotal = 0;
      for (int t0 = t_beg; t0 < t_end; t0 += 32) {
        const int t = t0 + lane;
        const int cnt = t < t_end ? a.counts[cell0 + t] : 0;
        wtotal += __reduce_add_sync(0xffffffffu, cnt);
      }
      if (lane == 0) warp_tot[warp] = wtotal;
      __syncthreads();
      int base = 0, total = 0;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const int v = warp_tot[w];
        base += w < warp ? v : 0;
        total += v;
      }
      for (int t0 = t_beg; t0 < t_end; t0 += 32) {
        const int t = t0 + lane;
        const int cnt = t < t_end ? a.counts[cell0 + t] : 0;
        int incl = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int x = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += x;
        }
        const int64_t cell = cell0 + t;
        const int pos = base + incl - cnt;
        for (int s2 = 0; s2 < cnt; ++s2)
          list[pos + s2] = RowEntry<VT>::make(t * a.T + a.idx[cell * a.C + s2], vals[cell * a.C + s2]);
        base += __shfl_sync(0xffffffffu, incl, 31);
      }
      __syncthreads();
      // the claim has had the flatten's loads to arrive; publishing it here
      // keeps it out of the streaming loop's registers
      if (threadIdx.x == 0) next_row_s[it] = claim;
      for (int cb = warp; cb < cbs; cb += kWarps) {
        const int c0 = cb * 256 + lane * 8;
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        if (c0 < a.d) {
          stream_list<VT>(a, W, c0, list, total, acc);
          const int64_t o = static_cast<int64_t>(row) * a.d + c0;
          if (a.acc) {
            float4* pa = reinterpret_cast<float4*>(a.acc + o);
            if (a.acc_mode > 0) {
              const float4 x = pa[0], y = pa[1];
              acc[0] += x.x; acc[1] += x.y; acc[2] += x.z; acc[3] += x.w;
              acc[4] += y.x; acc[5] += y.y; acc[6] += y.z; acc[7] += y.w;
            }
            if (a.acc_mode < 2) {
              pa[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
              pa[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
              continue;
            }
          }
          *reinterpret_cast<uint4*>(a.out + o) = pack8_bf16(acc);
        }
      }
    } else if (threadIdx.x == 0) {
      next_row_s[it] = claim;
    }
    __syncthreads();  // the list and warp totals are rewritten for the next row
    row = next_row_s[it];
  }
}

// The CTA-per-row kernel over whole rows (row-granular hybrid, no split).
template <typename VT>
int launch_spmm_rowcta(const SpmmArgs& a, const uint16_t* W, int kernel_id, cudaStream_t s) {
  auto rk = spmm_rowcta_kernel<VT>;
  const size_t rsmem = static_cast<size_t>(a.nt) * a.C * sizeof(RowEntry<VT>);
  if (rsmem > kMaxDynSmem) return TWELL_ERR_UNSUPPORTED;
  if (set_max_dynamic_smem(reinterpret_cast<const void*>(rk), kMaxDynSmem) != TWELL_OK) return TWELL_ERR_CUDA;
  const int rgrid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(a.N, 4 * static_cast<int64_t>(sm_count()))));
  {
    LaunchScope ls(kernel_id, s);
    if (launch_pdl(rk, dim3(rgrid), dim3(kWarps * 32), rsmem, s, a, W) != cudaSuccess) return TWELL_ERR_CUDA;
  }
  return cudaGetLastError() == cudaSuccess ? TWELL_OK : TWELL_ERR_CUDA;
}

template <typename VT>
int launch_spmm_rows(const SpmmArgs& a, const uint16_t* W, int nsplit, int kernel_id, cudaStream_t s) {
  if (a.N <= 0) return TWELL_OK;
  if (a.C > 32 || a.d % 128 != 0) return TWELL_ERR_UNSUPPORTED;
  if (a.nt * a.T > 65536) return TWELL_ERR_UNSUPPORTED;  // hidden unit fits the entry's 16 bits
  // a dense tile's (or a small batch's dense row's) non-zeros pass through the same list
  const int max_entries = (a.pool || a.dense_h) ? std::max(a.nt * a.C, a.T) : a.nt * a.C;
  const size_t smem = static_cast<size_t>(kWarps) * max_entries * sizeof(RowEntry<VT>);
  if (smem > kMaxDynSmem) return TWELL_ERR_UNSUPPORTED;
  auto kern = spmm_row_kernel<VT>;
  if (set_max_dynamic_smem(reinterpret_cast<const void*>(kern), kMaxDynSmem) != TWELL_OK) return TWELL_ERR_CUDA;
  if (nsplit < 1 || nsplit > 64 || (nsplit > 1 && (!a.part || !a.arrivals))) return TWELL_ERR_INVALID_ARG;
  if (nsplit > 1) {
    // no more tile ranges than fit in one wave of resident CTAs: a second wave
    // would repeat the whole latency chain of this short launch
    const int per_sm = resident_ctas_per_sm(reinterpret_cast<const void*>(kern), kWarps * 32, smem);
    if (per_sm <= 0) return TWELL_ERR_CUDA;
    const int64_t per_split = static_cast<int64_t>((a.N + kWarps - 1) / kWarps) * ((a.d + 255) / 256);
    const int fit = static_cast<int>(std::max<int64_t>(1, static_cast<int64_t>(per_sm) * sm_count() / per_split));
    nsplit = std::min(nsplit, fit);
  }
  dim3 grid((a.N + kWarps - 1) / kWarps, (a.d + 255) / 256, nsplit);
  if (nsplit > 1 && static_cast<int64_t>(grid.x) * grid.y > kSpmmMaxArrivals) return TWELL_ERR_UNSUPPORTED;
  // a CTA per row: one shared flatten for all column blocks; persistent, four
  // CTAs per SM (the register limit)
  if (nsplit == 1 && !a.pool && !a.dense_h) return launch_spmm_rowcta<VT>(a, W, kernel_id, s);
  if (nsplit == 1) {
    // persistent: three CTAs per SM (the register limit), warps stride over the items
    const int64_t items = static_cast<int64_t>(a.N) * ((a.d + 255) / 256);
    grid = dim3(static_cast<unsigned>(std::max<int64_t>(
                    1, std::min<int64_t>((items + kWarps - 1) / kWarps, 3 * static_cast<int64_t>(sm_count())))),
                1, 1);
  }
  {
    LaunchScope ls(kernel_id, s);
    if (launch_pdl(kern, grid, dim3(kWarps * 32), smem, s, a, W, max_entries) != cudaSuccess) return TWELL_ERR_CUDA;
  }
  return cudaGetLastError() == cudaSuccess ? TWELL_OK : TWELL_ERR_CUDA;
}

}  // namespace

// Tile ranges per row so that a small batch (at most kSwapMaxTokens rows)
// still launches ~4096 warps (at most 16 ranges); larger batches are not split.
int spmm_nsplit(int n_rows, int d_model) {
  const int64_t warps = static_cast<int64_t>(n_rows) * ((d_model + 255) / 256);
  if (warps <= 0 || n_rows > kSwapMaxTokens) return 1;
  return static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(16, (4096 + warps - 1) / warps)));
}

int spmm_single_passes(int d_model, int d_ff, int tile) {
  const double bytes = 2.0 * d_ff * static_cast<double>(d_model);
  return std::max(1, std::min({d_ff / tile, 8, static_cast<int>(bytes / (64.0 * 1024 * 1024) + 0.999)}));
}

int launch_spmm(const twell_t& L, const uint16_t* W_down, int d_model, uint16_t* Y, float* part, int nsplit,
                int32_t* arrivals, int32_t* row_counter, cudaStream_t s, const uint16_t* dense_h, int passes,
                float* acc) {
  if (dense_h && (L.hybrid == TWELL_HYBRID_TILES || L.tile % 32 != 0)) return TWELL_ERR_UNSUPPORTED;
  SpmmArgs a{L.values,
             L.idx,
             L.counts,
             L.row_fb,
             Y,
             part,
             arrivals,
             L.hybrid == TWELL_HYBRID_TILES ? L.fb_dense : nullptr,
             row_counter,
             L.n_rows,
             d_model,
             L.d_ff / L.tile,
             L.tile,
             L.cap,
             L.status,
             dense_h};
  if (passes > 1) {
    // whole TwELL rows in tile-range passes (the CTA-per-row kernel)
    if (nsplit != 1 || a.pool || dense_h || !acc || passes > a.nt) return TWELL_ERR_INVALID_ARG;
    if (a.N <= 0) return TWELL_OK;
    if (a.C > 32 || a.d % 128 != 0 || a.nt * a.T > 65536) return TWELL_ERR_UNSUPPORTED;
    for (int p = 0; p < passes; ++p) {
      a.t_lo = p * a.nt / passes;
      a.t_hi = (p + 1) * a.nt / passes;
      a.row_counter = row_counter ? row_counter + p : nullptr;
      a.acc = acc;
      a.acc_mode = p == 0 ? 0 : (p + 1 < passes ? 1 : 2);
      const int rc = launch_spmm_rowcta<uint16_t>(a, W_down, TWELL_KERNEL_SPMM, s);
      if (rc != TWELL_OK) return rc;
    }
    return TWELL_OK;
  }
  return launch_spmm_rows<uint16_t>(a, W_down, nsplit, TWELL_KERNEL_SPMM, s);
}

int launch_spmm_f32(const twell_t& L, const float* vals, const uint16_t* W, int d_model, uint16_t* out,
                    int32_t* row_counter, int kernel_id, cudaStream_t s) {
  SpmmArgs a{vals,     L.idx,   L.counts, L.row_fb,         out,    nullptr, nullptr, nullptr, row_counter,
             L.n_rows, d_model, L.d_ff / L.tile, L.tile, L.cap, L.status, nullptr};
  return launch_spmm_rows<float>(a, W, 1, kernel_id, s);
}

// Passes over tile ranges for the pair gather: each range's rows of both
// weight matrices should stay in L2 (at most 64 MB of them per pass; 48, 64
// and 96 MB per pass timed within 1% of each other at d_model 4096, d_ff 14336,
// 24 and 32 MB 3% slower).
int spmm_pair_passes(int d_model, int d_ff, int tile) {
  const double bytes = 2.0 * 2.0 * d_ff * static_cast<double>(d_model);
  const int nt = d_ff / tile;
  return std::max(1, std::min({nt, 8, static_cast<int>(bytes / (64.0 * 1024 * 1024) + 0.999)}));
}

int launch_spmm_f32x2(const twell_t& L, const float* pairs, const uint16_t* W_a, const uint16_t* W_b, int d_model,
                      uint16_t* out, int32_t* row_counters, float* acc, int passes, int kernel_id, cudaStream_t s) {
  if (L.hybrid != TWELL_HYBRID_ROWS) return TWELL_ERR_UNSUPPORTED;
  SpmmArgs a{pairs,    L.idx,   L.counts,        L.row_fb, out,   nullptr,  nullptr, nullptr, row_counters,
             L.n_rows, d_model, L.d_ff / L.tile, L.tile,   L.cap, L.status, nullptr, W_b};
  // whole TwELL rows, a CTA per row
  if (a.N <= 0) return TWELL_OK;
  if (a.C > 32 || a.d % 128 != 0) return TWELL_ERR_UNSUPPORTED;
  if (passes < 1 || passes > a.nt || (passes > 1 && !acc)) return TWELL_ERR_INVALID_ARG;
  // with several passes, pass p takes tiles [p nt / passes, (p + 1) nt / passes),
  // its own zeroed row counter, and the fp32 sums of the passes before it
  for (int p = 0; p < passes; ++p) {
    a.t_lo = p * a.nt / passes;
    a.t_hi = (p + 1) * a.nt / passes;
    a.row_counter = row_counters ? row_counters + p : nullptr;
    a.acc = passes > 1 ? acc : nullptr;
    a.acc_mode = p == 0 ? 0 : (p + 1 < passes ? 1 : 2);
    const int rc = launch_spmm_rowcta<float2>(a, W_a, kernel_id, s);
    if (rc != TWELL_OK) return rc;
  }
  return TWELL_OK;
}

}  // namespace twell
