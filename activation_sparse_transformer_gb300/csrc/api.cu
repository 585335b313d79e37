// Host side of the C ABI declared in include/twell.h: argument checks,
// TMA descriptor encoding, the launch sequence of each call, the device
// status word, launch counting and optional per-kernel event timing (totals
// per kernel id and a launch timeline).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <map>
#include <mutex>
#include <set>
#include <tuple>
#include <vector>

#include "twell_internal.h"

namespace twell {

// ---------------------------------------------------------------- launches
namespace {
struct Pending {
  int kernel;
  cudaEvent_t start, stop;
  cudaStream_t stream;
};
std::mutex g_mu;
int64_t g_launches = 0;
bool g_profiling = false;
std::vector<Pending> g_pending;
std::vector<cudaEvent_t> g_event_pool;
int64_t g_prof_launches[TWELL_KERNEL_COUNT] = {};
double g_prof_ms[TWELL_KERNEL_COUNT] = {};

cudaEvent_t take_event() {
  if (!g_event_pool.empty()) {
    cudaEvent_t e = g_event_pool.back();
    g_event_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}
}  // namespace

LaunchScope::LaunchScope(int kernel_id, cudaStream_t stream) : kernel_(kernel_id), stream_(stream) {
  std::lock_guard<std::mutex> lk(g_mu);
  ++g_launches;
  if (g_profiling) {
    start_ = take_event();
    cudaEventRecord(start_, stream_);
  }
}

LaunchScope::~LaunchScope() {
  if (!start_) return;
  std::lock_guard<std::mutex> lk(g_mu);
  cudaEvent_t stop = take_event();
  cudaEventRecord(stop, stream_);
  g_pending.push_back(Pending{kernel_, start_, stop, stream_});
}

// ---------------------------------------------------------------- aux stream
namespace {
std::mutex g_aux_mu;
// the second stream of each (device, caller stream), created on first use
std::map<std::pair<int, cudaStream_t>, cudaStream_t> g_aux_streams;

cudaStream_t aux_stream_for(int dev, cudaStream_t s) {
  std::lock_guard<std::mutex> lk(g_aux_mu);
  auto it = g_aux_streams.find({dev, s});
  if (it != g_aux_streams.end()) return it->second;
  // the second stream carries the small fallback-row work next to a large
  // kernel on the caller's stream: the highest priority lets its CTAs take
  // SMs as they free up instead of queueing behind the large grid
  int least = 0, greatest = 0;
  cudaStream_t a = nullptr;
  if (cudaDeviceGetStreamPriorityRange(&least, &greatest) != cudaSuccess ||
      cudaStreamCreateWithPriority(&a, cudaStreamNonBlocking, greatest) != cudaSuccess)
    return nullptr;
  g_aux_streams[{dev, s}] = a;
  return a;
}
}  // namespace

AuxFork::AuxFork(cudaStream_t s) : s_(s) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    rc_ = TWELL_ERR_CUDA;
    return;
  }
  aux_ = aux_stream_for(dev, s);
  if (!aux_ || cudaEventCreateWithFlags(&fork_, cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&join_, cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&mid_, cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&refork_, cudaEventDisableTiming) != cudaSuccess) {
    rc_ = TWELL_ERR_CUDA;
    return;
  }
  if (cudaEventRecord(fork_, s_) != cudaSuccess || cudaStreamWaitEvent(aux_, fork_, 0) != cudaSuccess)
    rc_ = TWELL_ERR_CUDA;
}

int AuxFork::join() {
  if (joined_ || rc_ != 0) return rc_;
  joined_ = true;
  if (cudaEventRecord(join_, aux_) != cudaSuccess || cudaStreamWaitEvent(s_, join_, 0) != cudaSuccess)
    rc_ = TWELL_ERR_CUDA;
  return rc_;
}

int AuxFork::mark_aux() {
  if (joined_ || rc_ != 0) return rc_;
  if (cudaEventRecord(mid_, aux_) != cudaSuccess) rc_ = TWELL_ERR_CUDA;
  return rc_;
}

int AuxFork::main_wait_mark() {
  if (joined_ || rc_ != 0) return rc_;
  if (cudaStreamWaitEvent(s_, mid_, 0) != cudaSuccess) rc_ = TWELL_ERR_CUDA;
  return rc_;
}

int AuxFork::aux_wait_main() {
  if (joined_ || rc_ != 0) return rc_;
  if (cudaEventRecord(refork_, s_) != cudaSuccess || cudaStreamWaitEvent(aux_, refork_, 0) != cudaSuccess)
    rc_ = TWELL_ERR_CUDA;
  return rc_;
}

AuxFork::~AuxFork() {
  join();
  // released by the runtime once the recorded work has completed
  for (cudaEvent_t e : {fork_, join_, mid_, refork_})
    if (e) cudaEventDestroy(e);
}

// ---------------------------------------------------------------- kernel attributes
namespace {
std::mutex g_attr_mu;
std::set<std::pair<int, const void*>> g_smem_set;
std::map<std::tuple<int, const void*, int, size_t>, int> g_resident;
}  // namespace

int set_max_dynamic_smem(const void* func, int bytes) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return TWELL_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_attr_mu);
  if (g_smem_set.count({dev, func})) return TWELL_OK;
  if (cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess)
    return TWELL_ERR_CUDA;
  g_smem_set.insert({dev, func});
  return TWELL_OK;
}

int resident_ctas_per_sm(const void* func, int block, size_t smem) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  std::lock_guard<std::mutex> lk(g_attr_mu);
  const auto key = std::make_tuple(dev, func, block, smem);
  auto it = g_resident.find(key);
  if (it != g_resident.end()) return it->second;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, func, block, smem) != cudaSuccess) return 0;
  g_resident[key] = n;
  return n;
}

// ---------------------------------------------------------------- device facts
// Device facts are fixed for the process: cached per device, the caches read
// and written atomically (two threads that race compute the same value).
int sm_count() {
  static std::atomic<int> cached[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64) {
    const int c = cached[dev].load(std::memory_order_relaxed);
    if (c) return c;
  }
  int n = 0;
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  if (n <= 0) n = 1;
  if (dev >= 0 && dev < 64) cached[dev].store(n, std::memory_order_relaxed);
  return n;
}

bool device_is_sm103() {
  static std::atomic<int> cached[64] = {};  // 0 unknown, 1 yes, 2 no
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  if (dev >= 0 && dev < 64) {
    const int c = cached[dev].load(std::memory_order_relaxed);
    if (c) return c == 1;
  }
  int major = 0, minor = 0;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  const bool ok = major == 10 && minor == 3;
  if (dev >= 0 && dev < 64) cached[dev].store(ok ? 1 : 2, std::memory_order_relaxed);
  return ok;
}

namespace {
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}
}  // namespace

namespace {
int encode_bf16_2d(CUtensorMap* map, const void* base, uint64_t inner_elems, uint64_t rows, uint64_t row_stride_bytes,
                   uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle swz) {
  auto fn = encode_fn();
  if (!fn) return TWELL_ERR_CUDA;
  cuuint64_t dims[2] = {inner_elems, rows};
  cuuint64_t strides[1] = {row_stride_bytes};
  cuuint32_t box[2] = {box_inner, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? TWELL_OK : TWELL_ERR_CUDA;
}
}  // namespace

int encode_tmap_2d(CUtensorMap* map, const void* base, uint64_t inner_elems, uint64_t rows,
                   uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_rows) {
  return encode_bf16_2d(map, base, inner_elems, rows, row_stride_bytes, box_inner, box_rows,
                        CU_TENSOR_MAP_SWIZZLE_128B);
}

int encode_tmap_2d_plain(CUtensorMap* map, const void* base, uint64_t inner_elems, uint64_t rows,
                         uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_rows) {
  return encode_bf16_2d(map, base, inner_elems, rows, row_stride_bytes, box_inner, box_rows,
                        CU_TENSOR_MAP_SWIZZLE_NONE);
}

}  // namespace twell

using namespace twell;

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The layout's fields (no device query).
int check_layout_fields(const twell_t* L) {
  if (!L) return TWELL_ERR_INVALID_ARG;
  if (L->n_rows < 0 || L->d_ff <= 0 || L->fb_cap < 0) return TWELL_ERR_INVALID_ARG;
  if (L->hybrid != TWELL_HYBRID_ROWS && L->hybrid != TWELL_HYBRID_TILES) return TWELL_ERR_INVALID_ARG;
  const int T = L->tile;
  if (T != 32 && T != 64 && T != 128 && T != 256) return TWELL_ERR_INVALID_ARG;
  if (L->cap < 1 || L->cap > T || L->cap > 32) return TWELL_ERR_INVALID_ARG;
  if (L->d_ff % T != 0) return TWELL_ERR_INVALID_ARG;
  if (L->d_ff % 128 != 0) return TWELL_ERR_UNSUPPORTED;
  // tile pool slots are 24-bit
  if (L->hybrid == TWELL_HYBRID_TILES && static_cast<int64_t>(L->fb_cap) * (L->d_ff / T) > 0xFFFFFF)
    return TWELL_ERR_UNSUPPORTED;
  if (!L->n_fb || !L->status) return TWELL_ERR_INVALID_ARG;
  if (L->n_rows > 0 && (!L->values || !L->idx || !L->counts || !L->row_fb)) return TWELL_ERR_INVALID_ARG;
  if (L->fb_cap > 0 && (!L->fb_rows || !L->fb_dense)) return TWELL_ERR_INVALID_ARG;
  if (!aligned16(L->values) || !aligned16(L->idx) || !aligned16(L->counts) || !aligned16(L->row_fb))
    return TWELL_ERR_MISALIGNED;
  if (L->fb_cap > 0 && (!aligned16(L->fb_rows) || !aligned16(L->fb_dense))) return TWELL_ERR_MISALIGNED;
  return TWELL_OK;
}

// The layout's fields, then the device (an sm_103a GPU current).
int check_layout(const twell_t* L) {
  const int rc = check_layout_fields(L);
  if (rc != TWELL_OK) return rc;
  return device_is_sm103() ? TWELL_OK : TWELL_ERR_NO_DEVICE;
}

int check_dense(const void* p) {
  if (!p) return TWELL_ERR_INVALID_ARG;
  if (!aligned16(p)) return TWELL_ERR_MISALIGNED;
  return TWELL_OK;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

#define TW_TRY(expr)             \
  do {                           \
    const int rc_ = (expr);      \
    if (rc_ != TWELL_OK) return rc_; \
  } while (0)

#define TW_CUDA(expr)                                  \
  do {                                                 \
    if ((expr) != cudaSuccess) return TWELL_ERR_CUDA;  \
  } while (0)

// status = 0 and every row_fb word = `row_fill` repeated in its four bytes
// (0x00: 0, 0xFF: -1)
int reset_words(const twell_t* L, cudaStream_t s, int row_fill = 0) {
  TW_CUDA(cudaMemsetAsync(L->status, 0, sizeof(int32_t), s));
  if (L->n_rows > 0)
    TW_CUDA(cudaMemsetAsync(L->row_fb, row_fill, sizeof(int32_t) * static_cast<size_t>(L->n_rows), s));
  return TWELL_OK;
}

}  // namespace

extern "C" {

int twell_pack(const uint16_t* H, int64_t ldh, const twell_t* out, twell_stream_t stream) {
  TW_TRY(check_layout(out));
  TW_TRY(check_dense(H));
  if (ldh < out->d_ff || ldh % 8 != 0) return TWELL_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  TW_TRY(reset_words(out, s));
  TW_TRY(launch_pack_cells(H, ldh, *out, s));
  if (out->hybrid == TWELL_HYBRID_TILES) {
    TW_TRY(launch_tile_count(*out, s));
    TW_TRY(launch_route(*out, s));
    return launch_tile_assign(*out, H, ldh, nullptr, 0, s);
  }
  TW_TRY(launch_route(*out, s));
  TW_TRY(launch_fb_copy(H, ldh, *out, s));
  return TWELL_OK;
}

int twell_unpack(const twell_t* in, uint16_t* H, int64_t ldh, twell_stream_t stream) {
  TW_TRY(check_layout(in));
  TW_TRY(check_dense(H));
  if (ldh < in->d_ff || ldh % 8 != 0) return TWELL_ERR_INVALID_ARG;
  return launch_unpack(*in, H, ldh, reinterpret_cast<cudaStream_t>(stream));
}

int twell_check_format(const twell_t* layout, int32_t* violations, twell_stream_t stream) {
  if (!layout || !violations) return TWELL_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(violations) % alignof(int32_t) != 0) return TWELL_ERR_MISALIGNED;
  TW_TRY(check_layout(layout));
  return launch_check_format(*layout, violations, reinterpret_cast<cudaStream_t>(stream));
}

namespace {
// Forward workspace: [spill tiles][spill counter and the gather's row
// counters][fallback down-projection partials] then, for small batches,
// [up-projection K-split partials][dense H] and [SpMM tile-range partials], or,
// when W_down is too large for L2, [fp32 sums carried between the gather's
// tile-range passes].
struct FwdWorkspace {
  size_t spill_off, count_off, part_off, total;
  int32_t spill_cap;
  int ksplit;                // fallback down-projection K splits
  bool swap;                 // small batch: swapped-operand up-projection
  int up_ksplit;
  size_t up_part_off, h_off, arrivals_off;
  int spmm_nsplit;
  size_t spmm_part_off;
  int spmm_passes;           // whole-row gather in tile-range passes (row-granular layouts)
  size_t spmm_acc_off;       // their fp32 sums [N][d_model]
};

FwdWorkspace fwd_workspace_layout(int32_t n_rows, int32_t d_model, int32_t d_ff, int32_t tile, int32_t fb_cap,
                                  bool tiles = false) {
  FwdWorkspace w{};
  const int64_t nt = d_ff / tile;
  w.spill_cap = static_cast<int32_t>(std::min<int64_t>(static_cast<int64_t>(fb_cap) * nt, 0xFFFFFF));
  // K splits of the fallback rows' down-projection: enough (128 x 128) output
  // tiles x splits (~256) that few fallback rows still stream W_down on every SM
  const int fb_tiles = ((fb_cap + 127) / 128) * ((d_model + 127) / 128);
  const int fb_want = fb_tiles > 0 ? std::max(4, std::min(16, (256 + fb_tiles - 1) / fb_tiles)) : 4;
  w.ksplit = fb_cap > 0 ? choose_fb_ksplit(d_ff, fb_want) : 1;
  w.spill_off = 0;
  w.count_off = align256(sizeof(uint16_t) * static_cast<size_t>(w.spill_cap) * static_cast<size_t>(tile));
  w.part_off = w.count_off + 256;
  size_t off = w.part_off +
               align256(sizeof(float) * static_cast<size_t>(w.ksplit) * static_cast<size_t>(fb_cap) * d_model);
  w.swap = n_rows > 0 && n_rows <= kSwapMaxTokens && d_ff % 128 == 0;
  w.up_ksplit = 1;
  if (w.swap) {
    w.up_ksplit = swap_ksplit(d_model);
    w.up_part_off = off;
    off += align256(sizeof(float) * static_cast<size_t>(w.up_ksplit) * n_rows * d_ff);
    w.h_off = off;
    off += align256(sizeof(uint16_t) * static_cast<size_t>(n_rows) * d_ff);
  }
  w.spmm_nsplit = n_rows > 0 ? spmm_nsplit(n_rows, d_model) : 1;
  if (w.swap || w.spmm_nsplit > 1) {
    // arrival counters: [0] the pack pass, [64, 64 + kSpmmMaxArrivals) the SpMM ranges
    w.arrivals_off = off;
    off += align256(sizeof(int32_t) * (64 + kSpmmMaxArrivals));
  }
  if (w.spmm_nsplit > 1) {
    w.spmm_part_off = off;
    off += align256(sizeof(float) * static_cast<size_t>(w.spmm_nsplit) * n_rows * d_model);
  }
  // the count word's 256 bytes hold the spill count and one row counter per pass
  w.spmm_passes = (!w.swap && w.spmm_nsplit == 1 && !tiles) ? spmm_single_passes(d_model, d_ff, tile) : 1;
  if (w.spmm_passes > 1) {
    w.spmm_acc_off = off;
    off += align256(sizeof(float) * static_cast<size_t>(n_rows) * d_model);
  }
  w.total = off;
  return w;
}
}  // namespace

size_t twell_fwd_workspace_bytes(int32_t n_rows, int32_t d_model, int32_t d_ff, int32_t tile, int32_t cap,
                                 int32_t fb_cap) {
  (void)cap;
  if (n_rows < 0 || d_model <= 0 || d_ff <= 0 || tile <= 0 || fb_cap < 0) return 0;
  return fwd_workspace_layout(n_rows, d_model, d_ff, tile, fb_cap).total;
}

}  // extern "C"

namespace {
// The forward of both layer kinds: the fused up-projection (plain ReLU, or
// gated when W_uT is given), routing, then the TwELL rows' gather-SpMM on the
// caller's stream and the dense-fallback rows on a second stream.
int ffn_fwd(const uint16_t* X, const uint16_t* W_inT, const uint16_t* W_uT, const uint16_t* b,
            const uint16_t* W_down, int32_t n_rows, int32_t d_model, int32_t d_ff, const twell_t* H, uint16_t* Y,
            void* workspace, size_t workspace_bytes, twell_stream_t stream, float* gu = nullptr) {
  TW_TRY(check_layout_fields(H));
  if (n_rows < 0 || d_model <= 0 || d_ff <= 0) return TWELL_ERR_INVALID_ARG;
  if (H->n_rows != n_rows || H->d_ff != d_ff) return TWELL_ERR_INVALID_ARG;
  if (d_model % 128 != 0) return TWELL_ERR_UNSUPPORTED;
  TW_TRY(check_dense(X));
  TW_TRY(check_dense(W_inT));
  if (W_uT) TW_TRY(check_dense(W_uT));
  TW_TRY(check_dense(b));
  TW_TRY(check_dense(W_down));
  TW_TRY(check_dense(Y));
  if (W_uT && 128 % H->tile != 0) return TWELL_ERR_UNSUPPORTED;
  const bool tiles = H->hybrid == TWELL_HYBRID_TILES;
  // the swapped small-batch path has no tile-granular form (the gated layer never takes it)
  if (tiles && !W_uT && n_rows > 0 && n_rows <= kSwapMaxTokens) return TWELL_ERR_UNSUPPORTED;
  const FwdWorkspace w = fwd_workspace_layout(n_rows, d_model, d_ff, H->tile, H->fb_cap, tiles);
  if (!workspace || workspace_bytes < w.total) return TWELL_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return TWELL_ERR_MISALIGNED;
  if (!device_is_sm103()) return TWELL_ERR_NO_DEVICE;
  if (n_rows == 0) return TWELL_OK;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  uint16_t* spill = reinterpret_cast<uint16_t*>(ws + w.spill_off);
  int32_t* spill_count = reinterpret_cast<int32_t*>(ws + w.count_off);
  float* part = reinterpret_cast<float*>(ws + w.part_off);
  float* spmm_part = w.spmm_nsplit > 1 ? reinterpret_cast<float*>(ws + w.spmm_part_off) : nullptr;
  uint16_t* Hd = w.swap ? reinterpret_cast<uint16_t*>(ws + w.h_off) : nullptr;
  const bool swap = w.swap && !W_uT;
  int32_t* row_counter = swap ? nullptr : spill_count + 1;  // the gather's row counter, zeroed with the count
  int32_t* arrivals = (w.swap || w.spmm_nsplit > 1) ? reinterpret_cast<int32_t*>(ws + w.arrivals_off) : nullptr;
  if (swap) {
    // the up-projection's CTA 0 zeroes row_fb and the arrival counters
    TW_CUDA(cudaMemsetAsync(H->status, 0, sizeof(int32_t), s));
  } else {
    // rows not flagged by the up-projection read -1 (the tile-granular
    // variant counts dense tiles from 0)
    TW_TRY(reset_words(H, s, tiles ? 0 : 0xFF));
    if (arrivals) TW_CUDA(cudaMemsetAsync(arrivals, 0, sizeof(int32_t) * (64 + kSpmmMaxArrivals), s));
  }
  if (swap) {
    // small batch: Z^T = W_in^T . X^T with the hidden units on the 128-row
    // MMA side and K split so the weight stream covers every SM; the partial
    // sums are added, biased and packed by a CUDA-core pass that also keeps
    // the dense h for the fallback copy
    float* up_part = reinterpret_cast<float*>(ws + w.up_part_off);
    PartialTEpiParams tp{up_part, d_ff, static_cast<int64_t>(n_rows) * d_ff, n_rows};
    TW_TRY(launch_gemm_swap_partial(W_inT, X, d_ff, n_rows, d_model, w.up_ksplit, tp, H->status,
                                    TWELL_KERNEL_UP_PACK, s, H->row_fb, n_rows, arrivals, 64 + kSpmmMaxArrivals));
    // the last CTA of the pack pass also routes the rows
    TW_TRY(launch_pack_partials(up_part, w.up_ksplit, b, Hd, *H, arrivals, s));
  } else {
    // the spill count and the gather's row counter(s), one per pass
    TW_CUDA(cudaMemsetAsync(spill_count, 0, (1 + w.spmm_passes) * sizeof(int32_t), s));
    PackEpiParams pp{b, H->values, H->idx, H->counts, H->row_fb, spill, spill_count, w.spill_cap, H->status,
                     d_ff / H->tile, H->tile, H->cap, gu};
    if (W_uT)
      TW_TRY(launch_gemm_gated_pack(X, W_inT, W_uT, n_rows, d_ff, d_model, pp, H->status, s));
    else
      TW_TRY(launch_gemm_pack(X, W_inT, n_rows, d_ff, d_model, pp, H->status, s));
    if (tiles) {
      // tile-granular hybrid: the spilled over-full tiles become the pool's
      // dense tiles in (row, tile) order, and the SpMM reads them there
      TW_TRY(launch_tile_count(*H, s));
      TW_TRY(launch_route(*H, s));
      TW_TRY(launch_tile_assign(*H, nullptr, 0, spill, w.spill_cap, s));
      return launch_spmm(*H, W_down, d_model, Y, spmm_part, w.spmm_nsplit, arrivals ? arrivals + 64 : nullptr,
                         row_counter, s);
    }
  }
  {
    // the dense-fallback rows (routing, assembly or copy, tensor-core
    // down-projection) run on a second stream while the gather-SpMM handles
    // the TwELL rows: it skips every row with row_fb >= 0, which holds for a
    // flagged row before routing (1) and after it (its slot), so it does not
    // wait for the routing scan
    AuxFork fork(s);
    TW_TRY(fork.status());
    if (swap) {
      // small batch: the fallback rows' dense h goes to fb_dense (an output of
      // the layout), and their rows of Y are gathered by the SpMM from the
      // dense h the pack pass kept, beside the TwELL rows: no fallback GEMM
      TW_TRY(launch_fb_copy(Hd, d_ff, *H, fork.aux()));
    } else {
      TW_TRY(launch_route(*H, fork.aux(), -1));
      TW_TRY(launch_fb_assemble(*H, spill, spill_count, w.spill_cap, fork.aux()));
      TW_TRY(launch_fb_down(*H, W_down, d_model, Y, part, w.ksplit, fork.aux()));
    }
    TW_TRY(launch_spmm(*H, W_down, d_model, Y, spmm_part, w.spmm_nsplit, arrivals ? arrivals + 64 : nullptr,
                       row_counter, s, swap ? Hd : nullptr, w.spmm_passes,
                       w.spmm_passes > 1 ? reinterpret_cast<float*>(ws + w.spmm_acc_off) : nullptr));
    TW_TRY(fork.join());
  }
  return TWELL_OK;
}
}  // namespace

namespace {
// The row view of a tile-granular layout that the backward builds in its
// workspace after the base bytes: routing words [n_rows], slots [fb_cap], the
// count word, and the dense rows [fb_cap][d_ff] bf16.
size_t row_view_bytes(int32_t n_rows, int32_t d_ff, int32_t fb_cap) {
  return align256(sizeof(int32_t) * static_cast<size_t>(std::max(n_rows, 1))) +
         align256(sizeof(int32_t) * static_cast<size_t>(std::max(fb_cap, 1))) + 256 +
         align256(sizeof(uint16_t) * static_cast<size_t>(std::max(fb_cap, 0)) * static_cast<size_t>(d_ff));
}

twell_t row_view_in(const twell_t& H, uint8_t* v) {
  twell_t V = H;
  V.hybrid = TWELL_HYBRID_ROWS;
  V.row_fb = reinterpret_cast<int32_t*>(v);
  v += align256(sizeof(int32_t) * static_cast<size_t>(std::max(H.n_rows, 1)));
  V.fb_rows = reinterpret_cast<int32_t*>(v);
  v += align256(sizeof(int32_t) * static_cast<size_t>(std::max(H.fb_cap, 1)));
  V.n_fb = reinterpret_cast<int32_t*>(v);
  v += 256;
  V.fb_dense = reinterpret_cast<uint16_t*>(v);
  return V;
}
}  // namespace

extern "C" {

int twell_ffn_fwd(const uint16_t* X, const uint16_t* W_inT, const uint16_t* b, const uint16_t* W_down,
                  int32_t n_rows, int32_t d_model, int32_t d_ff, const twell_t* H, uint16_t* Y, void* workspace,
                  size_t workspace_bytes, twell_stream_t stream) {
  return ffn_fwd(X, W_inT, nullptr, b, W_down, n_rows, d_model, d_ff, H, Y, workspace, workspace_bytes, stream);
}

int twell_gated_ffn_fwd(const uint16_t* X, const uint16_t* W_gT, const uint16_t* W_uT, const uint16_t* b,
                        const uint16_t* W_down, int32_t n_rows, int32_t d_model, int32_t d_ff, const twell_t* H,
                        uint16_t* Y, void* workspace, size_t workspace_bytes, twell_stream_t stream) {
  if (!W_uT) return TWELL_ERR_INVALID_ARG;
  return ffn_fwd(X, W_gT, W_uT, b, W_down, n_rows, d_model, d_ff, H, Y, workspace, workspace_bytes, stream);
}

int twell_gated_ffn_fwd_train(const uint16_t* X, const uint16_t* W_gT, const uint16_t* W_uT, const uint16_t* b,
                              const uint16_t* W_down, int32_t n_rows, int32_t d_model, int32_t d_ff,
                              const twell_t* H, uint16_t* Y, float* gu, void* workspace, size_t workspace_bytes,
                              twell_stream_t stream) {
  if (!W_uT || !gu) return TWELL_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(gu) % 16 != 0) return TWELL_ERR_MISALIGNED;
  return ffn_fwd(X, W_gT, W_uT, b, W_down, n_rows, d_model, d_ff, H, Y, workspace, workspace_bytes, stream, gu);
}

size_t twell_bwd_workspace_bytes(int32_t n_rows, int32_t d_model, int32_t d_ff, int32_t tile, int32_t cap,
                                 int32_t fb_cap) {
  if (n_rows < 0 || d_ff <= 0 || tile <= 0 || cap <= 0 || fb_cap < 0) return 0;
  return bwd_workspace_layout(n_rows, d_model, d_ff, tile, cap, fb_cap, nullptr, nullptr);
}

int twell_ffn_bwd(const uint16_t* X, const uint16_t* W_inT, const uint16_t* W_down, const twell_t* H,
                  int32_t d_model, const uint16_t* dY, float l1_lambda, uint16_t* dX, float* dW_inT,
                  float* dW_down, float* db, void* workspace, size_t workspace_bytes, twell_stream_t stream) {
  TW_TRY(check_layout(H));
  if (d_model <= 0) return TWELL_ERR_INVALID_ARG;
  if (d_model % 128 != 0) return TWELL_ERR_UNSUPPORTED;
  const bool tiles = H->hybrid == TWELL_HYBRID_TILES;
  // the unit-major lists address the stored entries with 32-bit positions
  if (static_cast<int64_t>(H->n_rows) * (H->d_ff / H->tile) * H->cap > INT32_MAX) return TWELL_ERR_UNSUPPORTED;
  TW_TRY(check_dense(X));
  TW_TRY(check_dense(W_inT));
  TW_TRY(check_dense(W_down));
  TW_TRY(check_dense(dY));
  TW_TRY(check_dense(dX));
  TW_TRY(check_dense(dW_inT));
  TW_TRY(check_dense(dW_down));
  TW_TRY(check_dense(db));
  const size_t base = twell_bwd_workspace_bytes(H->n_rows, d_model, H->d_ff, H->tile, H->cap, H->fb_cap);
  const size_t need =
      tiles ? twell_bwd_tiles_workspace_bytes(H->n_rows, d_model, H->d_ff, H->tile, H->cap, H->fb_cap) : base;
  if (!workspace || workspace_bytes < need) return TWELL_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return TWELL_ERR_MISALIGNED;
  BwdWorkspace ws{};
  bwd_workspace_layout(H->n_rows, d_model, H->d_ff, H->tile, H->cap, H->fb_cap, &ws, workspace);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (!tiles)
    return launch_bwd(X, W_inT, W_down, *H, dY, l1_lambda, dX, dW_inT, dW_down, db, d_model, ws, s);
  // tile-granular layout: the backward of its row view, in which every row
  // holding a dense tile is a fallback row with its dense h (the layer's
  // gradients do not depend on how h is stored)
  twell_t V = row_view_in(*H, static_cast<uint8_t*>(workspace) + base);
  TW_TRY(launch_tile_row_view(*H, V, s));
  return launch_bwd(X, W_inT, W_down, V, dY, l1_lambda, dX, dW_inT, dW_down, db, d_model, ws, s, true);
}

size_t twell_bwd_tiles_workspace_bytes(int32_t n_rows, int32_t d_model, int32_t d_ff, int32_t tile, int32_t cap,
                                       int32_t fb_cap) {
  const size_t base = twell_bwd_workspace_bytes(n_rows, d_model, d_ff, tile, cap, fb_cap);
  return base ? base + row_view_bytes(n_rows, d_ff, fb_cap) : 0;
}

size_t twell_gated_bwd_workspace_bytes(int32_t n_rows, int32_t d_model, int32_t d_ff, int32_t tile, int32_t cap,
                                       int32_t fb_cap) {
  if (n_rows < 0 || d_ff <= 0 || tile <= 0 || cap <= 0 || fb_cap < 0) return 0;
  return bwd_workspace_layout(n_rows, d_model, d_ff, tile, cap, fb_cap, nullptr, nullptr, true);
}

size_t twell_gated_bwd_tiles_workspace_bytes(int32_t n_rows, int32_t d_model, int32_t d_ff, int32_t tile,
                                             int32_t cap, int32_t fb_cap) {
  const size_t base = twell_gated_bwd_workspace_bytes(n_rows, d_model, d_ff, tile, cap, fb_cap);
  return base ? base + row_view_bytes(n_rows, d_ff, fb_cap) : 0;
}

int twell_gated_ffn_bwd(const uint16_t* X, const uint16_t* W_gT, const uint16_t* W_uT, const uint16_t* b,
                        const uint16_t* W_down, const twell_t* H, const float* gu, int32_t d_model,
                        const uint16_t* dY, float l1_lambda, uint16_t* dX, float* dW_gT, float* dW_uT,
                        float* dW_down, float* db, void* workspace, size_t workspace_bytes,
                        twell_stream_t stream) {
  TW_TRY(check_layout_fields(H));
  if (d_model <= 0) return TWELL_ERR_INVALID_ARG;
  if (d_model % 128 != 0 || H->d_ff % 128 != 0) return TWELL_ERR_UNSUPPORTED;
  const bool tiles = H->hybrid == TWELL_HYBRID_TILES;
  if (static_cast<int64_t>(H->n_rows) * (H->d_ff / H->tile) * H->cap > INT32_MAX) return TWELL_ERR_UNSUPPORTED;
  for (const void* p : {static_cast<const void*>(X), static_cast<const void*>(W_gT), static_cast<const void*>(W_uT),
                        static_cast<const void*>(b), static_cast<const void*>(W_down), static_cast<const void*>(dY),
                        static_cast<const void*>(dX), static_cast<const void*>(dW_gT),
                        static_cast<const void*>(dW_uT), static_cast<const void*>(dW_down),
                        static_cast<const void*>(db)})
    TW_TRY(check_dense(p));
  if (!gu) return TWELL_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(gu) % 16 != 0) return TWELL_ERR_MISALIGNED;
  const size_t base = twell_gated_bwd_workspace_bytes(H->n_rows, d_model, H->d_ff, H->tile, H->cap, H->fb_cap);
  const size_t need = tiles ? base + row_view_bytes(H->n_rows, H->d_ff, H->fb_cap) : base;
  if (!workspace || workspace_bytes < need) return TWELL_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return TWELL_ERR_MISALIGNED;
  if (!device_is_sm103()) return TWELL_ERR_NO_DEVICE;
  BwdWorkspace ws{};
  bwd_workspace_layout(H->n_rows, d_model, H->d_ff, H->tile, H->cap, H->fb_cap, &ws, workspace, true);
  GatedBwd g{W_uT, b, gu, dW_uT};
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (!tiles) return launch_bwd(X, W_gT, W_down, *H, dY, l1_lambda, dX, dW_gT, dW_down, db, d_model, ws, s, false, &g);
  // tile-granular layout: the row view, as for twell_ffn_bwd; its fallback rows
  // (every row holding a dense tile) get g and u recomputed, its other rows'
  // slots all have theirs from the forward
  twell_t V = row_view_in(*H, static_cast<uint8_t*>(workspace) + base);
  TW_TRY(launch_tile_row_view(*H, V, s));
  return launch_bwd(X, W_gT, W_down, V, dY, l1_lambda, dX, dW_gT, dW_down, db, d_model, ws, s, true, &g);
}

int twell_dense_ffn_fwd(const uint16_t* X, const uint16_t* W_inT, const uint16_t* b, const uint16_t* W_down,
                        int32_t n_rows, int32_t d_model, int32_t d_ff, uint16_t* Hbuf, uint16_t* Y,
                        twell_stream_t stream) {
  if (n_rows < 0 || d_model <= 0 || d_ff <= 0) return TWELL_ERR_INVALID_ARG;
  if (d_model % 128 != 0 || d_ff % 128 != 0) return TWELL_ERR_UNSUPPORTED;
  TW_TRY(check_dense(X));
  TW_TRY(check_dense(W_inT));
  TW_TRY(check_dense(b));
  TW_TRY(check_dense(W_down));
  TW_TRY(check_dense(Hbuf));
  TW_TRY(check_dense(Y));
  if (!device_is_sm103()) return TWELL_ERR_NO_DEVICE;
  if (n_rows == 0) return TWELL_OK;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  DenseEpiParams up{b, Hbuf, d_ff, 1};
  TW_TRY(launch_gemm_dense(X, W_inT, false, n_rows, nullptr, d_ff, d_model, up, nullptr, TWELL_KERNEL_DENSE_GEMM, s));
  DenseEpiParams down{nullptr, Y, d_model, 0};
  TW_TRY(launch_gemm_dense(Hbuf, W_down, true, n_rows, nullptr, d_model, d_ff, down, nullptr, TWELL_KERNEL_DENSE_GEMM,
                           s));
  return TWELL_OK;
}

size_t twell_dense_bwd_workspace_bytes(int32_t n_rows, int32_t d_model, int32_t d_ff) {
  (void)d_model;
  if (n_rows < 0 || d_ff <= 0) return 0;
  return align256(sizeof(uint16_t) * static_cast<size_t>(n_rows) * d_ff) +
         align256(sizeof(float) * static_cast<size_t>(kColsumChunks) * d_ff);
}

int twell_dense_ffn_bwd(const uint16_t* X, const uint16_t* W_inT, const uint16_t* W_down, const uint16_t* H,
                        int32_t n_rows, int32_t d_model, int32_t d_ff, const uint16_t* dY, float l1_lambda,
                        uint16_t* dX, float* dW_inT, float* dW_down, float* db, void* workspace,
                        size_t workspace_bytes, twell_stream_t stream) {
  if (n_rows < 0 || d_model <= 0 || d_ff <= 0) return TWELL_ERR_INVALID_ARG;
  if (d_model % 128 != 0 || d_ff % 128 != 0) return TWELL_ERR_UNSUPPORTED;
  for (const void* p : {static_cast<const void*>(X), static_cast<const void*>(W_inT),
                        static_cast<const void*>(W_down), static_cast<const void*>(H), static_cast<const void*>(dY),
                        static_cast<const void*>(dX), static_cast<const void*>(dW_inT),
                        static_cast<const void*>(dW_down), static_cast<const void*>(db)})
    TW_TRY(check_dense(p));
  const size_t need = twell_dense_bwd_workspace_bytes(n_rows, d_model, d_ff);
  if (!workspace || workspace_bytes < need) return TWELL_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return TWELL_ERR_MISALIGNED;
  if (!device_is_sm103()) return TWELL_ERR_NO_DEVICE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (n_rows == 0) {
    // no rows: the weight gradients are zero
    TW_CUDA(cudaMemsetAsync(dW_inT, 0, sizeof(float) * static_cast<size_t>(d_ff) * d_model, s));
    TW_CUDA(cudaMemsetAsync(dW_down, 0, sizeof(float) * static_cast<size_t>(d_ff) * d_model, s));
    TW_CUDA(cudaMemsetAsync(db, 0, sizeof(float) * static_cast<size_t>(d_ff), s));
    return TWELL_OK;
  }
  uint16_t* dZ = static_cast<uint16_t*>(workspace);
  float* part = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) +
                                         align256(sizeof(uint16_t) * static_cast<size_t>(n_rows) * d_ff));
  // dZ = (dY . W_down^T + lambda) where h > 0: a dense GEMM with a masking epilogue
  MaskEpiParams mp{H, dZ, d_ff, l1_lambda};
  TW_TRY(launch_gemm_mask(dY, W_down, n_rows, d_ff, d_model, mp, nullptr, TWELL_KERNEL_DENSE_GEMM, s));
  // dX = dZ . W_in (W_in^T read as the N-major B operand)
  DenseEpiParams xp{nullptr, dX, d_model, 0};
  TW_TRY(launch_gemm_dense(dZ, W_inT, true, n_rows, nullptr, d_model, d_ff, xp, nullptr, TWELL_KERNEL_DENSE_GEMM,
                           s));
  // dW_in^T = dZ^T . X and dW_down = H^T . dY, K = the rows
  TW_TRY(launch_gemm_store_mn(dZ, X, d_ff, d_model, n_rows, nullptr, 1, dW_inT, d_model, nullptr,
                              TWELL_KERNEL_DENSE_GEMM, s));
  TW_TRY(launch_gemm_store_mn(H, dY, d_ff, d_model, n_rows, nullptr, 1, dW_down, d_model, nullptr,
                              TWELL_KERNEL_DENSE_GEMM, s));
  return launch_colsum_bf16(dZ, n_rows, d_ff, part, db, TWELL_KERNEL_DENSE_GEMM, s);
}

int twell_read_status(const twell_t* layout, twell_stream_t stream) {
  if (!layout || !layout->status || !layout->n_fb) return TWELL_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return TWELL_ERR_CUDA;
  int32_t st = 0, nfb = 0;
  if (cudaMemcpy(&st, layout->status, sizeof st, cudaMemcpyDeviceToHost) != cudaSuccess) return TWELL_ERR_CUDA;
  if (cudaMemcpy(&nfb, layout->n_fb, sizeof nfb, cudaMemcpyDeviceToHost) != cudaSuccess) return TWELL_ERR_CUDA;
  if (st != 0) return st;
  const int64_t cap = layout->hybrid == TWELL_HYBRID_TILES && layout->tile > 0
                          ? static_cast<int64_t>(layout->fb_cap) * (layout->d_ff / layout->tile)
                          : layout->fb_cap;
  if (nfb > cap) return TWELL_ERR_FALLBACK_OVERFLOW;
  return TWELL_OK;
}

const char* twell_status_string(int code) {
  switch (code) {
    case TWELL_OK: return "ok";
    case TWELL_ERR_INVALID_ARG: return "invalid argument";
    case TWELL_ERR_MISALIGNED: return "pointer not aligned as required";
    case TWELL_ERR_UNSUPPORTED: return "shape not supported by the kernels' tiling";
    case TWELL_ERR_CUDA: return "CUDA runtime or driver call failed";
    case TWELL_ERR_WORKSPACE: return "workspace missing or too small";
    case TWELL_ERR_FALLBACK_OVERFLOW: return "more dense-fallback rows than fb_cap";
    case TWELL_ERR_WAIT_TIMEOUT: return "a bounded pipeline wait on the GPU expired";
    case TWELL_ERR_NO_DEVICE: return "no sm_103a device is current";
    case TWELL_ERR_BAD_FORMAT: return "packed layout breaks a format rule";
    default: return "unknown status";
  }
}

int64_t twell_launch_count(void) {
  std::lock_guard<std::mutex> lk(g_mu);
  return g_launches;
}

int twell_profile_enable(int on) {
  std::lock_guard<std::mutex> lk(g_mu);
  g_profiling = on != 0;
  return TWELL_OK;
}

int twell_profile_reset(void) {
  if (cudaDeviceSynchronize() != cudaSuccess) return TWELL_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  for (auto& p : g_pending) {
    g_event_pool.push_back(p.start);
    g_event_pool.push_back(p.stop);
  }
  g_pending.clear();
  for (int k = 0; k < TWELL_KERNEL_COUNT; ++k) {
    g_prof_launches[k] = 0;
    g_prof_ms[k] = 0.0;
  }
  return TWELL_OK;
}

int twell_profile_timeline(int max, int32_t* kernel, uint64_t* stream, double* start_ms, double* end_ms) {
  if (max < 0 || (max > 0 && (!kernel || !stream || !start_ms || !end_ms))) return TWELL_ERR_INVALID_ARG;
  if (cudaDeviceSynchronize() != cudaSuccess) return TWELL_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  const int n = static_cast<int>(std::min<size_t>(static_cast<size_t>(max), g_pending.size()));
  for (int i = 0; i < n; ++i) {
    const Pending& p = g_pending[i];
    float a = 0.f, b = 0.f;
    if (cudaEventElapsedTime(&a, g_pending[0].start, p.start) != cudaSuccess ||
        cudaEventElapsedTime(&b, g_pending[0].start, p.stop) != cudaSuccess)
      return TWELL_ERR_CUDA;
    kernel[i] = p.kernel;
    stream[i] = static_cast<uint64_t>(reinterpret_cast<uintptr_t>(p.stream));
    start_ms[i] = a;
    end_ms[i] = b;
  }
  return n;
}

int twell_profile_read(int kernel, int64_t* launches, double* total_ms) {
  if (kernel < 0 || kernel >= TWELL_KERNEL_COUNT) return TWELL_ERR_INVALID_ARG;
  if (cudaDeviceSynchronize() != cudaSuccess) return TWELL_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  for (auto& p : g_pending) {
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, p.start, p.stop) == cudaSuccess) {
      g_prof_launches[p.kernel] += 1;
      g_prof_ms[p.kernel] += ms;
    }
    g_event_pool.push_back(p.start);
    g_event_pool.push_back(p.stop);
  }
  g_pending.clear();
  if (launches) *launches = g_prof_launches[kernel];
  if (total_ms) *total_ms = g_prof_ms[kernel];
  return TWELL_OK;
}

}  // extern "C"
