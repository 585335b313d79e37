// Declarations shared by the library's translation units (not part of the ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

#include "../../include/twell.h"

namespace twell {

// Pipeline waits inside kernels give up after this much global time and
// report TWELL_ERR_WAIT_TIMEOUT instead of hanging.
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

// ---------------------------------------------------------------- launches
// Counts every kernel launch and, while profiling is on, brackets it with a
// pair of CUDA events on its stream.
class LaunchScope {
 public:
  LaunchScope(int kernel_id, cudaStream_t stream);
  ~LaunchScope();

 private:
  int kernel_;
  cudaStream_t stream_;
  cudaEvent_t start_ = nullptr;
};

int sm_count();                      // SMs of the current device (cached per device)

// Launches a kernel with programmatic stream serialization: the kernel's
// launch and start overlap the end of the previous kernel on the stream, and
// the kernel executes grid_dependency_wait() before touching memory.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute a[1];
  a[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  a[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = a;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// Sets a kernel's dynamic shared-memory limit on the current device once
// (thread-safe); returns TWELL_OK or TWELL_ERR_CUDA.
int set_max_dynamic_smem(const void* func, int bytes);
// Resident CTAs per SM of a kernel at a block size and dynamic shared memory
// on the current device, cached (thread-safe); 0 when the query fails.
int resident_ctas_per_sm(const void* func, int block, size_t smem);

// A second stream for work that can overlap the caller's stream s (the
// dense-fallback path).  Each (device, caller stream) pair has its own second
// stream, created on first use, so callers on different streams never share
// one; the fork / join events belong to the call.  fork(): aux waits for
// everything queued on s so far; join(): s waits for everything queued on
// aux.  Both are asynchronous.
class AuxFork {
 public:
  explicit AuxFork(cudaStream_t s);
  ~AuxFork();
  int status() const { return rc_; }
  cudaStream_t aux() const { return aux_; }
  int join();
  // mark_aux records the point reached by the work queued on aux so far;
  // main_wait_mark makes s wait for that point (aux continues independently),
  // so s can queue independent work in between
  int mark_aux();
  int main_wait_mark();
  // aux waits for everything queued on s so far (a second fork point)
  int aux_wait_main();

 private:
  cudaStream_t s_;
  cudaStream_t aux_ = nullptr;
  cudaEvent_t fork_ = nullptr, join_ = nullptr, mid_ = nullptr, refork_ = nullptr;
  int rc_ = 0;
  bool joined_ = false;
};
bool device_is_sm103();              // current device is compute capability 10.3
// bf16 2-D tensor maps: 128-byte swizzled (tensor-core operands) or plain
// row-major boxes (shared-memory slabs read by CUDA cores).
int encode_tmap_2d(CUtensorMap* map, const void* base, uint64_t inner_elems, uint64_t rows,
                   uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_rows);
int encode_tmap_2d_plain(CUtensorMap* map, const void* base, uint64_t inner_elems, uint64_t rows,
                         uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_rows);

// ---------------------------------------------------------------- kernels
// A cell whose tile held more than C non-zeros during the fused
// up-projection: its count byte holds this marker and its first slot holds a
// 24-bit index into the spill buffer (value bits 0..15, index byte 16..23),
// where the tile's dense bf16 values were written.  Only fallback rows carry
// such cells, and the fallback assembly clears them.
constexpr uint8_t kSpilledCell = 255;

struct PackEpiParams {
  const uint16_t* bias;   // [d_ff]
  uint16_t* values;       // [M][n_tiles][C]
  uint8_t* idx;
  uint8_t* counts;        // [M][n_tiles]
  int32_t* row_flag;      // [M], set to 1 where a tile overflows C (pre-zeroed)
  uint16_t* spill;        // [spill_cap][T] dense tiles of overflowing cells
  int32_t* spill_count;   // device counter, pre-zeroed
  int32_t spill_cap;
  int32_t* status;
  int32_t n_tiles;
  int32_t tile;           // T
  int32_t cap;            // C
  float* gu;              // gated layer, for its backward: (g, u) fp32 at every stored slot
                          // [M][n_tiles][C][2] (g with the bias), or null
};

struct DenseEpiParams {
  const uint16_t* bias;   // [N] or null
  uint16_t* out;          // [M][ldo]
  int64_t ldo;
  int32_t relu;           // 1: out = bf16(z) where z > 0 else +0
};

// fp32 partial sums of one K split: part[ks * split_stride + row * ld + col]
struct PartialEpiParams {
  float* part;
  int64_t ld;
  int64_t split_stride;
};

// fp32 partial sums of one K split with the operands swapped (accumulator rows
// are hidden units, columns are tokens): part[ks * split_stride + token * ld + unit],
// tokens from n_tok on are not stored.
struct PartialTEpiParams {
  float* part;
  int64_t ld;
  int64_t split_stride;
  int32_t n_tok;
};

// dH = dY . W_down^T sampled at the TwELL pattern (the ReLU mask), plus the
// L1 gradient: dZ = dH + lambda where h > 0.
struct SampleEpiParams {
  const uint16_t* values;   // the packed forward activations
  const uint8_t* idx;
  const uint8_t* counts;
  const int32_t* row_fb;
  const uint16_t* fb_dense;
  int32_t fb_cap;
  int32_t n_tiles, tile, cap, d_ff;
  float lambda;
  float* dz_cells;          // [M][n_tiles][C] fp32, stored slots only
  uint16_t* dz_hl;          // [2 * fb_pad][d_ff] bf16 for the fallback rows' dense dZ (0 where h == 0):
                            // row 2s = bf16(dz) (high part), row 2s+1 = bf16(dz - high) (low
                            // part); high + low carry dz to ~2^-17 relative
  // gated layer (gu non-null): the pattern is h != 0 and dh' = dH + lambda sign(h);
  // dz_cells then holds (dG, dU) = (dh' u, dh' g) pairs per slot ([M][n_tiles][C][2])
  // and the fallback rows' dense dh' goes to dh_fb (dz_hl is not written)
  const float* gu;          // (g, u) at the stored slots [M][n_tiles][C][2]
  float* dh_fb;             // [fb_pad][d_ff] fp32 dh' of the fallback rows (0 where h == 0)
};

// g = X.W_g + b and u = X.W_u of the gated layer's fallback rows, kept as
// (g, u) fp32 pairs [M][d_ff][2] (the dual-B GEMM's two halves).
struct GUEpiParams {
  const uint16_t* bias;
  float* gu;
  int32_t d_ff;
};

// dZ = dH + lambda where h > 0 (else 0) for the dense comparator: dH the
// accumulator, h from the dense H [M][ld] bf16; out [M][ld] bf16.
struct MaskEpiParams {
  const uint16_t* H;
  uint16_t* out;
  int64_t ld;
  float lambda;
};

// C[M, N] = A[M, K] . B^T with A row-major [M][K] (K-major).  B is row-major
// [N][K] (K-major) for the pack / dense / sample GEMMs and row-major [K][N]
// (N-major) for the partial GEMM.  Rows beyond min(M, *M_dev) are not stored.
int launch_gemm_pack(const uint16_t* A, const uint16_t* B, int M, int N, int K, const PackEpiParams& p,
                     int32_t* status, cudaStream_t s);
// Gated up-projection: h = bf16((X.W_g + b) * (X.W_u)) where X.W_g + b > 0,
// packed like launch_gemm_pack; Bg and Bu are [N][K] (K-major).
int launch_gemm_gated_pack(const uint16_t* A, const uint16_t* Bg, const uint16_t* Bu, int M, int N, int K,
                           const PackEpiParams& p, int32_t* status, cudaStream_t s);
int launch_gemm_dense(const uint16_t* A, const uint16_t* B, bool b_n_major, int M, const int32_t* M_dev, int N,
                      int K, const DenseEpiParams& p, int32_t* status, int kernel_id, cudaStream_t s);
// b_k_wrap > 0: B holds b_k_wrap rows of K and row k of the product's K is
// B's row k mod b_k_wrap (the same B against the high and low parts of A).
int launch_gemm_partial_nmajor(const uint16_t* A, const uint16_t* B, int M, const int32_t* M_dev, int N, int K,
                               int ksplit, const PartialEpiParams& p, int32_t* status, int kernel_id,
                               cudaStream_t s, int64_t lda = 0, int b_k_wrap = 0);
// (g, u) of the gated layer's fallback rows: A = their X rows (lda), B = W_gT and W_uT
int launch_gemm_gu(const uint16_t* A, int64_t lda, const uint16_t* Bg, const uint16_t* Bu, int M, const int32_t* M_dev,
                   int N, int K, const GUEpiParams& p, int32_t* status, int kernel_id, cudaStream_t s);
int launch_gemm_mask(const uint16_t* A, const uint16_t* B, int M, int N, int K, const MaskEpiParams& p,
                     int32_t* status, int kernel_id, cudaStream_t s);
// db[j] = sum over rows of Z[r][j] (bf16 [M][N], fp32 sums): row-chunk
// partials [kColsumChunks][N] fp32 in `part`, then their sum in chunk order.
constexpr int kColsumChunks = 16;
int launch_colsum_bf16(const uint16_t* Z, int M, int N, float* part, float* out, int kernel_id, cudaStream_t s);
// zero[0, n_zero) (int32), when given, is zeroed by the GEMM's CTA 0.
int launch_gemm_sample(const uint16_t* A, const uint16_t* B, int M, int N, int K, const SampleEpiParams& p,
                       int32_t* status, cudaStream_t s, int32_t* zero = nullptr, int n_zero = 0);
// out[M][N] = A^T . B (fp32 store) with A row-major [K][M] and B row-major
// [K][N] (both M/N-major); only the first k_mul * (*K_dev) rows of K count,
// rows up to the next multiple of 64 past them must be zero in both operands,
// and nothing is written when k_mul * (*K_dev) is 0.
int launch_gemm_store_mn(const uint16_t* A, const uint16_t* B, int M, int N, int K, const int32_t* K_dev, int k_mul,
                         float* out, int64_t ld, int32_t* status, int kernel_id, cudaStream_t s);
int choose_fb_ksplit(int K, int max_split = 4);   // K splits used for the fallback rows' down-projection
// Small-batch up-projection with the operands swapped: Z^T = W . X^T as
// part[ks][token][unit] fp32 partial sums over ksplit K ranges.  W is [M][K]
// row-major (M hidden units), X is [n_tok][K] row-major with n_tok <= kSwapMaxTokens.
constexpr int kSwapMaxTokens = 32;
int swap_ksplit(int K);
// CTA 0 also sets n_zero0 words at zero0 and n_zero1 at zero1 to zero (state
// of the kernels that follow on the stream).
int launch_gemm_swap_partial(const uint16_t* W, const uint16_t* X, int M, int n_tok, int K, int ksplit,
                             const PartialTEpiParams& p, int32_t* status, int kernel_id, cudaStream_t s,
                             int32_t* zero0 = nullptr, int n_zero0 = 0, int32_t* zero1 = nullptr, int n_zero1 = 0);

// forward helpers (fwd_kernels.cu)
// rows variant: row_fb holds 1 for a flagged row and `empty` for the others;
// clear_past: a row past fb_cap gets empty cells (else its cells are left)
int launch_route(const twell_t& L, cudaStream_t s, int32_t empty = 0, bool clear_past = true);
// the row view V of a tile-granular layout H (V.row_fb, fb_rows, n_fb and
// fb_dense in the backward's workspace; V.fb_cap rows)
int launch_tile_row_view(const twell_t& H, const twell_t& V, cudaStream_t s);
// tile-granular hybrid: dense tiles per flagged row (before launch_route), then
// pool slots, pool copies (from H, or from the spill buffer when H is null)
// and the cells' slot numbers (after it)
int launch_tile_count(const twell_t& L, cudaStream_t s);
int launch_tile_assign(const twell_t& L, const uint16_t* H, int64_t ldh, const uint16_t* spill, int32_t spill_cap,
                       cudaStream_t s);
int launch_fb_assemble(const twell_t& L, const uint16_t* spill, const int32_t* spill_count, int32_t spill_cap,
                       cudaStream_t s);
// Y = H . W_down for the TwELL rows.  With nsplit > 1 each row's tiles are
// cut into nsplit consecutive ranges whose fp32 partial sums go to part
// ([nsplit][N][d_model]) and are added in range order (small batches); the
// arrival counters (kSpmmMaxArrivals int32) must be zero on entry.  Whole
// rows are handed out through row_counter (one int32, zero on entry) when it
// is given, else by a fixed stride.
constexpr int kSpmmMaxArrivals = 1024;
int spmm_nsplit(int n_rows, int d_model);
// passes > 1 (whole rows of the row-granular hybrid only): the gather runs in
// that many launches over consecutive tile ranges, summed in range order
// through acc ([N][d_model] fp32), each with its own zeroed row_counter word
int launch_spmm(const twell_t& L, const uint16_t* W_down, int d_model, uint16_t* Y, float* part, int nsplit,
                int32_t* arrivals, int32_t* row_counter, cudaStream_t s,
                const uint16_t* dense_h = nullptr, int passes = 1, float* acc = nullptr);
// Passes of the forward gather over tile ranges: W_down's rows above ~64 MB
// do not stay in L2 across one pass over all tiles.
int spmm_single_passes(int d_model, int d_ff, int tile);
int launch_spmm_f32(const twell_t& L, const float* vals, const uint16_t* W, int d_model, uint16_t* out,
                    int32_t* row_counter, int kernel_id, cudaStream_t s);
// out[n] = bf16(sum over row n's TwELL entries e of a_e W_a[j_e] + b_e W_b[j_e]),
// (a_e, b_e) fp32 pairs per slot ([N][n_tiles][C][2]); fallback rows skipped.
// passes > 1: in that many launches over consecutive tile ranges, summed in
// range order through acc ([N][d_model] fp32); row_counters: one zeroed word
// per pass (or null)
int spmm_pair_passes(int d_model, int d_ff, int tile);
int launch_spmm_f32x2(const twell_t& L, const float* pairs, const uint16_t* W_a, const uint16_t* W_b, int d_model,
                      uint16_t* out, int32_t* row_counters, float* acc, int passes, int kernel_id, cudaStream_t s);
// out[fb_rows[r]] = bf16(sum over nsplit of part[k][r]) for the fallback rows
int launch_fb_reduce(const twell_t& L, const float* part, int nsplit, int d_model, uint16_t* out, int kernel_id,
                     cudaStream_t s);
int launch_fb_down(const twell_t& L, const uint16_t* W_down, int d_model, uint16_t* Y, float* part, int ksplit,
                   cudaStream_t s);

// standalone pack / unpack (pack_kernels.cu)
int launch_pack_cells(const uint16_t* H, int64_t ldh, const twell_t& L, cudaStream_t s);
int launch_fb_copy(const uint16_t* H, int64_t ldh, const twell_t& L, cudaStream_t s);
// h = bf16(relu(sum over ksplit of part[ks][token][unit] + b[unit])) for every
// token, packed like launch_pack_cells (overflowing rows flagged) and also
// written densely to H [n_rows][d_ff] for the fallback copy.  With an arrival
// counter (one int32 of workspace, zero on entry; n_rows <= 32) the rows are
// also routed, as launch_route would.
int launch_pack_partials(const float* part, int ksplit, const uint16_t* b, uint16_t* H, const twell_t& L,
                         int32_t* arrivals, cudaStream_t s);
int launch_unpack(const twell_t& L, uint16_t* H, int64_t ldh, cudaStream_t s);
// Format rules of a layout -> *violations (mask, zeroed first); two launches.
int launch_check_format(const twell_t& L, int32_t* violations, cudaStream_t s);

// backward (bwd_kernels.cu)
struct BwdWorkspace {
  float* dz_cells;        // [N][n_tiles][C] fp32: dZ at the stored TwELL entries
  uint16_t* dz_hl;        // [2 * fb_pad][d_ff] bf16 high / low parts of the fallback rows' dZ
                          // (0 off the pattern), interleaved by row
  uint16_t* hfb;          // [fb_pad][d_ff] fallback rows of H (zero past n_fb)
  uint16_t* dyg;          // [fb_pad][d_model] dY of the fallback rows (zero past n_fb)
  uint16_t* xg2;          // [2 * fb_pad][d_model] X of the fallback rows, each row twice
  int32_t fb_pad;         // fb_cap rounded up to 64
  float* part;            // [ksplit][fb_cap][d_model] fp32 partial sums of the fallback rows' dX
                          // (shares its region with hfb, dyg, xg2 and, gated, gu_fb, dh_fb,
                          // which are dead before it is written)
  int32_t ksplit;
  int32_t* col_beg;       // [d_ff] start of each hidden unit's entry list (tile t's lists in [t N C, (t + 1) N C))
  int32_t* col_end;       // [d_ff] end of each hidden unit's entry list
  int32_t* col_rows;      // [capacity] row of each entry, grouped by unit, rows ascending
  uint16_t* col_h;        // [capacity] h of each entry (bf16 bits)
  float* col_dz;          // [capacity] dZ of each entry
  int32_t* row_counter;   // [dx_passes] the dX gather's row counters (zeroed by the SDDMM GEMM)
  // gated layer only (null otherwise); dz_cells is then [N][n_tiles][C][2]
  // (dG, dU) pairs and part holds 2 ksplit splits (the gate's, then the up's)
  uint16_t* du_hl;        // [2 * fb_pad][d_ff] bf16 high / low parts of the fallback rows' dU
  float* gu_fb;           // [fb_pad][d_ff][2] (g, u) of the fallback rows, recomputed
  float* dh_fb;           // [fb_pad][d_ff] fp32 dh' of the fallback rows
  float* col_du;          // [capacity] dU of each entry
  float* dx_acc;          // [N][d_model] fp32 sums between the dX gather's passes (null: one pass)
  int32_t dx_passes;
};
size_t bwd_workspace_layout(int N, int d_model, int d_ff, int T, int C, int fb_cap, BwdWorkspace* ws,
                            void* base, bool gated = false);

// The gated layer's extra operands of the backward (H = bf16(g u), g = X.W_g + b > 0,
// u = X.W_u): W_inT is then W_g^T and dW_inT receives dW_g^T.
struct GatedBwd {
  const uint16_t* W_uT;   // [d_ff][d_model] bf16
  const uint16_t* b;      // [d_ff] bf16 gate bias
  const float* gu;        // [N][n_tiles][C][2] (g, u) at the stored slots (the training forward's)
  float* dW_uT;           // [d_ff][d_model] fp32
};
int launch_bwd(const uint16_t* X, const uint16_t* W_inT, const uint16_t* W_down, const twell_t& L,
               const uint16_t* dY, float lambda, uint16_t* dX, float* dW_inT, float* dW_down, float* db,
               int d_model, const BwdWorkspace& ws, cudaStream_t s, bool row_view = false,
               const GatedBwd* gated = nullptr);

}  // namespace twell
