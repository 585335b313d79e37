/*
 * twell.h -- C ABI of the TwELL activation-sparse feed-forward layer for one
 * NVIDIA GB300 (sm_103a).
 *
 * The layer (from "Sparser, Faster, Lighter Transformer Language Models",
 * Sakana AI + NVIDIA, as the pages describe it):
 *     H = ReLU(X . W_in + b)          (the nonlinearity zeroes most units:
 *                                      ifai.io news, opening; iaexpertos blog,
 *                                      "The Challenge of Sparsity Ignored by GPUs")
 *     H is stored in the Tile-wise ELLPACK (TwELL) hybrid format
 *                                     (ifai.io news, "Reshaping math for the GPU";
 *                                      repo-explainer, "TwELL: The Packing Format
 *                                      That Fits the Machine"; bayesiansapien note,
 *                                      flowchart and the description of Figure 1)
 *     Y = H . W_down                  computed from the packed form
 *     plus the backward pass, with the gradient of an L1 penalty on H
 *                                     (bayesiansapien note, TL;DR).
 * The repo-explainer page ("TwELL: The Packing Format...") names the kernel
 * layer's jobs: dense-to-TwELL, TwELL-to-dense, and fused MLP execution.
 *
 * Conventions for every call
 *   - bf16 tensors are passed as uint16_t bit patterns; all tensors are
 *     row-major and dense (the leading dimension equals the row length unless
 *     an ld argument says otherwise).
 *   - Pointers named in a call are DEVICE pointers owned by the caller unless
 *     the comment says host.  The library allocates no device memory inside
 *     these calls; scratch comes from the caller's workspace.
 *   - Calls are asynchronous on `stream` (NULL = the legacy default stream)
 *     and never synchronise, except twell_read_status.
 *   - Return value: TWELL_OK or a negative TWELL_ERR_* code found on the host
 *     before any launch (nothing is launched then).  Errors found on the GPU
 *     are written to the layout's device status word (see twell_t.status) and
 *     read with twell_read_status; kernels never trap.
 *   - Shapes: n_rows >= 0 (0 is a no-op), d_model % 128 == 0, d_ff % 128 == 0,
 *     tile T in {32, 64, 128, 256} with T | d_ff, 1 <= cap C <= min(T, 32).
 *     Device pointers must be 16-byte aligned.
 *
 * Hybrid layout (this build's reading of the pages; capacity C, the overflow
 * rule and byte layouts are not given there):
 *   - d_ff is cut into n_tiles = d_ff / T tiles of T consecutive hidden units.
 *   - Per (row n, tile t) a cell holds up to C non-zero values, their
 *     tile-local indices (strictly increasing, in [0, T)) and a count.
 *   - A row with any tile holding more than C non-zeros is a fallback row: its
 *     dense H row lives in fb_dense, its cells have count 0.  Fallback rows
 *     take slots 0, 1, ... in ascending row order.
 *   - Unused slots are padding: value +0.0 (0x0000), index 0.
 *   - "Non-zero" means the bf16 value compares unequal to zero.
 *
 * Tile-granular variant (twell_t.hybrid = TWELL_HYBRID_TILES; the pages'
 * Figure 1, as the bayesiansapien note describes it, shows hybrids that split
 * between formats; this one splits per (row, tile) instead of per row):
 *   - A tile with more than C non-zeros is a dense tile: its T values live in
 *     the next slot of a tile pool, fb_dense viewed as [fb_cap * n_tiles][T],
 *     slots numbered 0, 1, ... in ascending (row, tile) order.  Its cell has
 *     count 255 (TWELL_DENSE_TILE), the slot number in its first entry (value =
 *     low 16 bits, index = bits 16..23) and padding in the others.
 *   - No row is routed whole: row_fb is -1 for every row, fb_rows is unused,
 *     *n_fb counts dense tiles (may exceed fb_cap * n_tiles; tiles past the
 *     pool are not stored, their cells are left empty, and the status word
 *     reports TWELL_ERR_FALLBACK_OVERFLOW).
 *   - Supported by twell_pack, twell_unpack, twell_ffn_fwd (n_rows > 32), the
 *     gated forward (any n_rows) and both backward calls (through a row view,
 *     see twell_ffn_bwd); the small-batch forward of the plain layer returns
 *     TWELL_ERR_UNSUPPORTED for it.
 */
#ifndef TWELL_H
#define TWELL_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define TWELL_API __attribute__((visibility("default")))
#else
#define TWELL_API
#endif

typedef struct CUstream_st* twell_stream_t; /* same type as cudaStream_t */

enum {
  TWELL_OK = 0,
  TWELL_ERR_INVALID_ARG = -1,        /* null pointer, negative size, bad T/C */
  TWELL_ERR_MISALIGNED = -2,         /* pointer not 16-byte aligned */
  TWELL_ERR_UNSUPPORTED = -3,        /* shape outside the kernels' tiling */
  TWELL_ERR_CUDA = -4,               /* a CUDA runtime/driver call failed */
  TWELL_ERR_WORKSPACE = -5,          /* workspace missing or too small */
  TWELL_ERR_FALLBACK_OVERFLOW = -6,  /* device: more fallback rows than fb_cap */
  TWELL_ERR_WAIT_TIMEOUT = -7,       /* device: a bounded pipeline wait expired */
  TWELL_ERR_NO_DEVICE = -8,          /* no sm_103a device current */
  TWELL_ERR_BAD_FORMAT = -9          /* device: twell_check_format found a broken rule */
};

enum {
  TWELL_HYBRID_ROWS = 0,   /* a row with an over-full tile goes whole to fb_dense */
  TWELL_HYBRID_TILES = 1,  /* only the over-full tiles go, to a pool of dense tiles */
  TWELL_DENSE_TILE = 255   /* cell count of a dense tile (tile-granular variant) */
};

/* A packed activation matrix H [n_rows][d_ff].  The struct itself lives in
 * host memory and is read during the call; every pointer in it is a device
 * pointer to caller-owned memory of the stated size. */
typedef struct twell_t {
  int32_t n_rows;     /* N */
  int32_t d_ff;       /* f */
  int32_t tile;       /* T */
  int32_t cap;        /* C */
  int32_t fb_cap;     /* rows the dense fallback can hold (>= 0) */
  int32_t hybrid;     /* TWELL_HYBRID_ROWS (0) or TWELL_HYBRID_TILES */
  uint16_t* values;   /* [N][f/T][C] bf16 */
  uint8_t* idx;       /* [N][f/T][C] tile-local index */
  uint8_t* counts;    /* [N][f/T] non-zeros stored in the cell (0 for fallback rows;
                         TWELL_DENSE_TILE for a dense tile of the tile-granular variant) */
  int32_t* row_fb;    /* [N] -1 = TwELL row, else slot in fb_dense */
  int32_t* fb_rows;   /* [fb_cap] row of each fallback slot, ascending (rows variant) */
  uint16_t* fb_dense; /* [fb_cap][f] bf16 dense rows, or the pool of fb_cap * f / T dense tiles */
  int32_t* n_fb;      /* device scalar: fallback rows (or dense tiles) found; may exceed the capacity */
  int32_t* status;    /* device scalar: 0 or a TWELL_ERR_* code set by a kernel */
} twell_t;

/* Dense -> TwELL (the pages' "dense-to-TwELL" kernel path; repo-explainer,
 * "TwELL: The Packing Format That Fits the Machine").
 * H: device, [out->n_rows][ldh] bf16, ldh >= d_ff and ldh % 8 == 0.
 * Writes every array of *out, *out->n_fb and resets *out->status to 0 (then
 * TWELL_ERR_FALLBACK_OVERFLOW if n_fb > fb_cap; rows past fb_cap are not
 * stored).  Bit-exact: the output is a pure function of H's bits. */
TWELL_API int twell_pack(const uint16_t* H, int64_t ldh, const twell_t* out, twell_stream_t stream);

/* TwELL -> dense (the pages' "TwELL-to-dense" path).
 * H: device, [in->n_rows][ldh] bf16 output, ldh >= d_ff, ldh % 8 == 0.
 * Every element of the first d_ff columns is written (zeros included).  A
 * fallback row past fb_cap (an overflowed layout: stored nowhere) comes out
 * as zeros. */
TWELL_API int twell_unpack(const twell_t* in, uint16_t* H, int64_t ldh, twell_stream_t stream);

/* Forward of the layer ("fused MLP execution", repo-explainer page; the
 * dense matrix for rare dense tokens, ifai.io news "Reshaping math for the GPU").
 *   X      [n_rows][d_model] bf16      W_inT  [d_ff][d_model] bf16 (W_in transposed,
 *   b      [d_ff] bf16                                             nn.Linear layout)
 *   W_down [d_ff][d_model] bf16 (row j = hidden unit j)
 *   H      packed output; H->n_rows == n_rows, H->d_ff == d_ff
 *   Y      [n_rows][d_model] bf16 output
 * h = bf16(z) where z = X.W_in + b > 0 (fp32 accumulation), else +0; Y is the
 * fp32 sum over h's non-zeros rounded once to bf16.  A tile that overflows C
 * has its dense h kept by the up-projection, so the fallback rows of fb_dense
 * hold exactly the h the GEMM produced.  Batches of at most 32 rows (decode)
 * take a path built for them: the up-projection with the hidden units on the
 * 128-row MMA side and K split over the SMs (its fp32 partial sums added in
 * split order), and the down-projection with each row's tiles cut into ranges
 * added in order; results agree with the large-batch path up to fp32
 * summation order (bit for bit on inputs whose partial sums are exact).  When
 * W_down is larger than ~64 MB (row-granular layouts, more than 32 rows) the
 * down-projection gathers in passes over consecutive tile ranges, whose fp32
 * sums are added in range order, so each pass's W_down rows stay in L2.
 * More fallback rows than fb_cap: the status word reports
 * TWELL_ERR_FALLBACK_OVERFLOW and the rows past fb_cap are stored nowhere
 * (their cells are emptied); their rows of Y are left unwritten, except in
 * the small-batch path, whose gather takes every row's h from its dense copy.
 * workspace: device, >= twell_fwd_workspace_bytes(...) bytes (always > 0),
 * 256-byte aligned; its contents need no initialisation and nothing in it is
 * needed once the call's work on the stream has finished, so one buffer can
 * serve this call and a later twell_ffn_bwd on the same stream. */
TWELL_API int twell_ffn_fwd(const uint16_t* X, const uint16_t* W_inT, const uint16_t* b,
                  const uint16_t* W_down, int32_t n_rows, int32_t d_model, int32_t d_ff,
                  const twell_t* H, uint16_t* Y, void* workspace, size_t workspace_bytes,
                  twell_stream_t stream);

TWELL_API size_t twell_fwd_workspace_bytes(int32_t n_rows, int32_t d_model, int32_t d_ff, int32_t tile,
                                 int32_t cap, int32_t fb_cap);

/* Forward of the gated (Llama-style) ReLU layer: H = ReLU(X.W_g + b) (.) (X.W_u)
 * elementwise, then Y = H.W_down, with H packed in TwELL as for twell_ffn_fwd
 * (the pages name a sparse "sparse_llama" model configuration, repo-explainer
 * "The Repo's Two Jobs").  W_gT and W_uT are [d_ff][d_model] bf16; b applies to
 * the gate.  h = bf16(zg * zu) where zg = X.W_g + b > 0 (fp32), else +0, so h
 * may be negative; "non-zero" is h != 0.  The tile must divide 128.  Both
 * hybrid variants, at any n_rows (there is no separate small-batch path).  Same
 * workspace as twell_ffn_fwd. */
TWELL_API int twell_gated_ffn_fwd(const uint16_t* X, const uint16_t* W_gT, const uint16_t* W_uT,
                                  const uint16_t* b, const uint16_t* W_down, int32_t n_rows,
                                  int32_t d_model, int32_t d_ff, const twell_t* H, uint16_t* Y,
                                  void* workspace, size_t workspace_bytes, twell_stream_t stream);

/* twell_gated_ffn_fwd for training: also keeps, for every stored slot of a
 * TwELL cell, the gate g = X.W_g + b and the up value u = X.W_u (fp32) that
 * twell_gated_ffn_bwd needs (dG = dh u, dU = dh g).
 *   gu  device, [n_rows][d_ff / tile][cap][2] fp32, 16-byte aligned: (g, u) at
 *       the slots below the cell's count; other slots (padding, fallback
 *       rows, overflowed cells) are left as they are. */
TWELL_API int twell_gated_ffn_fwd_train(const uint16_t* X, const uint16_t* W_gT, const uint16_t* W_uT,
                                        const uint16_t* b, const uint16_t* W_down, int32_t n_rows,
                                        int32_t d_model, int32_t d_ff, const twell_t* H, uint16_t* Y, float* gu,
                                        void* workspace, size_t workspace_bytes, twell_stream_t stream);

/* The forward pass for callers that cannot allocate device memory.  (The
 * paper and its pages have no counterpart: this is a deployment convenience
 * of this library.)  Some callers have no allocator of their own to hand --
 * code running inside another framework's memory pool, plugins whose host
 * application owns every cudaMalloc, real-time paths where a cudaMalloc (which
 * may synchronise the device) is not allowed -- so they cannot supply the
 * workspace twell_ffn_fwd needs.  This call takes the same arguments minus the
 * workspace and uses a fixed scratch array compiled into the library instead
 * (twell_ffn_fwd_noalloc_max_scratch() bytes, 4 MiB; every GPU that loads the
 * library holds it until the process exits).  It allocates nothing.
 *   - Sizes: twell_fwd_workspace_bytes(...) must not exceed that maximum
 *     (it grows with fb_cap * d_ff and fb_cap * d_model, and for batches of
 *     at most 32 rows with n_rows * d_ff and n_rows * d_model); otherwise
 *     TWELL_ERR_WORKSPACE is returned and nothing is launched.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.  The address is kept for the process: after
 *     cudaDeviceReset (or anything else that destroys the device's primary
 *     context) the entry point must not be called again on that device.
 *   - All calls share the one array and it keeps the last call's contents
 *     (nothing in it needs to start at zero): calls that overlap on the GPU,
 *     e.g. on two streams, race on it and must be ordered by the caller.
 * Results are identical to twell_ffn_fwd with a caller-provided workspace. */
TWELL_API int twell_ffn_fwd_noalloc(const uint16_t* X, const uint16_t* W_inT, const uint16_t* b,
                                    const uint16_t* W_down, int32_t n_rows, int32_t d_model,
                                    int32_t d_ff, const twell_t* H, uint16_t* Y,
                                    twell_stream_t stream);

TWELL_API size_t twell_ffn_fwd_noalloc_max_scratch(void);

/* Backward of  L = sum(Y * dY) + l1_lambda * sum|H|  (the L1 penalty of the
 * bayesiansapien note's TL;DR, its gradient taken as l1_lambda wherever h > 0).
 *   H    the packed forward activations (pattern = ReLU mask); n_rows = H->n_rows
 *   X [n_rows][d_model], W_inT and W_down [d_ff][d_model]: the forward's inputs
 *   dY   [n_rows][d_model] bf16
 * Outputs (all overwritten):
 *   dX      [n_rows][d_model] bf16      dZ = (dY.W_down^T + l1_lambda) at the pattern
 *   dW_inT  [d_ff][d_model] fp32        dW_inT[j] = sum_n dZ[n][j] X[n]
 *   dW_down [d_ff][d_model] fp32        dW_down[j] = sum_n h[n][j] dY[n]
 *   db      [d_ff] fp32                 db[j] = sum_n dZ[n][j]
 * dH is only formed at H's non-zeros (SDDMM).  Deterministic: every output
 * element is summed by one thread in a fixed order (no atomics on outputs;
 * rows are handed to CTAs through an atomic counter, which changes only who
 * computes a row, not how).
 * workspace: device, >= twell_bwd_workspace_bytes(...) bytes, 256-byte aligned
 * (it may be the forward call's workspace, see twell_ffn_fwd); for the
 * tile-granular variant >= twell_bwd_tiles_workspace_bytes(...).
 * Tile-granular layouts: the gradients are those of the same h, computed on a
 * row view built in the workspace, in which each row holding a dense tile is a
 * fallback row (its dense h assembled from its cells and pool tiles; at most
 * fb_cap such rows, else the status word reports TWELL_ERR_FALLBACK_OVERFLOW
 * and the rows past fb_cap are left out); the layout itself is not modified.
 * TWELL_ERR_UNSUPPORTED when n_rows * (d_ff / tile) * cap exceeds 2^31 - 1
 * (32-bit entry positions). */
TWELL_API int twell_ffn_bwd(const uint16_t* X, const uint16_t* W_inT, const uint16_t* W_down,
                  const twell_t* H, int32_t d_model, const uint16_t* dY, float l1_lambda, uint16_t* dX,
                  float* dW_inT, float* dW_down, float* db, void* workspace,
                  size_t workspace_bytes, twell_stream_t stream);

TWELL_API size_t twell_bwd_workspace_bytes(int32_t n_rows, int32_t d_model, int32_t d_ff, int32_t tile,
                                 int32_t cap, int32_t fb_cap);

/* Workspace of twell_ffn_bwd for a tile-granular layout: twell_bwd_workspace_bytes
 * plus the row view (routing words, fb_cap slots, fb_cap dense rows). */
TWELL_API size_t twell_bwd_tiles_workspace_bytes(int32_t n_rows, int32_t d_model, int32_t d_ff, int32_t tile,
                                                 int32_t cap, int32_t fb_cap);

/* Backward of the gated layer (the Llama-style "sparse_llama" layer of the
 * repo-explainer page, "The Repo's Two Jobs") for
 *   L = sum(Y * dY) + l1_lambda * sum|H|,  Y = H.W_down,
 *   H = bf16(g u) where g = X.W_g + b > 0 (else 0), u = X.W_u,
 * with h's bf16 rounding passed straight through and the pattern h != 0 (the
 * stored entries: h may be negative).  At the pattern
 *   dh = dY.W_down^T + l1_lambda sign(h),  dG = dh u,  dU = dh g
 * and 0 elsewhere.  Inputs as for twell_gated_ffn_fwd (row-granular layout
 * only), plus
 *   gu   device, what twell_gated_ffn_fwd_train kept for the same call: (g, u)
 *        fp32 at every stored slot ([n_rows][d_ff / tile][cap][2]); the
 *        fallback rows' g and u are recomputed here on the tensor cores.
 * Outputs (all overwritten):
 *   dX      [n_rows][d_model] bf16   dX[n] = sum_j dG[n][j] W_g^T[j] + dU[n][j] W_u^T[j]
 *   dW_gT   [d_ff][d_model] fp32     dW_gT[j] = sum_n dG[n][j] X[n]
 *   dW_uT   [d_ff][d_model] fp32     dW_uT[j] = sum_n dU[n][j] X[n]
 *   dW_down [d_ff][d_model] fp32     dW_down[j] = sum_n h[n][j] dY[n]
 *   db      [d_ff] fp32              db[j] = sum_n dG[n][j]  (the bias sits on the gate)
 * Deterministic as twell_ffn_bwd.  workspace: device, >=
 * twell_gated_bwd_workspace_bytes(...) bytes, 256-byte aligned; for the
 * tile-granular variant >= twell_gated_bwd_tiles_workspace_bytes(...).
 * Tile-granular layouts go through the row view that twell_ffn_bwd describes:
 * rows holding a dense tile are fallback rows, whose g and u are recomputed.
 * TWELL_ERR_UNSUPPORTED when d_ff is not a multiple of 128, or n_rows *
 * (d_ff / tile) * cap is above 2^31 - 1; TWELL_ERR_MISALIGNED when gu is not
 * 16-byte aligned. */
TWELL_API int twell_gated_ffn_bwd(const uint16_t* X, const uint16_t* W_gT, const uint16_t* W_uT,
                                  const uint16_t* b, const uint16_t* W_down, const twell_t* H, const float* gu,
                                  int32_t d_model, const uint16_t* dY, float l1_lambda, uint16_t* dX,
                                  float* dW_gT, float* dW_uT, float* dW_down, float* db, void* workspace,
                                  size_t workspace_bytes, twell_stream_t stream);

TWELL_API size_t twell_gated_bwd_workspace_bytes(int32_t n_rows, int32_t d_model, int32_t d_ff, int32_t tile,
                                                 int32_t cap, int32_t fb_cap);

/* Workspace of twell_gated_ffn_bwd for a tile-granular layout:
 * twell_gated_bwd_workspace_bytes plus the row view. */
TWELL_API size_t twell_gated_bwd_tiles_workspace_bytes(int32_t n_rows, int32_t d_model, int32_t d_ff,
                                                       int32_t tile, int32_t cap, int32_t fb_cap);

/* Dense comparator (not part of the method): Y = ReLU(X.W_in + b).W_down with
 * the same tensor-core GEMM and no sparsity.  W_down is [d_ff][d_model] bf16 as
 * for twell_ffn_fwd; Hbuf is caller scratch [n_rows][d_ff] bf16 that receives
 * the dense H. */
TWELL_API int twell_dense_ffn_fwd(const uint16_t* X, const uint16_t* W_inT, const uint16_t* b,
                        const uint16_t* W_down, int32_t n_rows, int32_t d_model, int32_t d_ff,
                        uint16_t* Hbuf, uint16_t* Y, twell_stream_t stream);

/* Backward of the dense comparator (not part of the method): the gradients
 * twell_ffn_bwd computes, for the layer run densely by twell_dense_ffn_fwd,
 * with no sparsity used -- the dense training step the TwELL step is measured
 * against (run time and peak device memory).
 *   H       [n_rows][d_ff] bf16, the dense forward's Hbuf (h = ReLU(z), bf16)
 *   X, W_inT, W_down, dY, and the outputs dX (bf16), dW_inT, dW_down, db
 *   (fp32) as for twell_ffn_bwd.
 * dZ = (dY . W_down^T + l1_lambda) where h > 0, else 0, is formed densely on
 * the tensor cores and kept in bf16 (the dense bf16 layer's own precision);
 * dX = dZ . W_in, dW_inT = dZ^T . X, dW_down = H^T . dY, db = column sums of dZ
 * (fixed order: deterministic).
 * workspace: device, >= twell_dense_bwd_workspace_bytes(...) bytes, 256-byte
 * aligned (holds dZ, n_rows * d_ff bf16, and the column-sum partials). */
TWELL_API int twell_dense_ffn_bwd(const uint16_t* X, const uint16_t* W_inT, const uint16_t* W_down,
                                  const uint16_t* H, int32_t n_rows, int32_t d_model, int32_t d_ff,
                                  const uint16_t* dY, float l1_lambda, uint16_t* dX, float* dW_inT,
                                  float* dW_down, float* db, void* workspace, size_t workspace_bytes,
                                  twell_stream_t stream);

TWELL_API size_t twell_dense_bwd_workspace_bytes(int32_t n_rows, int32_t d_model, int32_t d_ff);

/* Synchronises `stream`, then returns *layout->status if non-zero, else
 * TWELL_ERR_FALLBACK_OVERFLOW when *layout->n_fb exceeds the capacity (fb_cap
 * rows, or fb_cap * d_ff / tile dense tiles for the tile-granular variant),
 * else TWELL_OK. */
TWELL_API int twell_read_status(const twell_t* layout, twell_stream_t stream);

/* Self-test of the failure detection (no counterpart on the pages): launches
 * one small kernel that runs the pipelines' bounded mbarrier wait on a barrier
 * nothing arrives on; after limit_ns of GPU time the wait gives up and
 * *status (device int32) is set to TWELL_ERR_WAIT_TIMEOUT, exactly as a
 * stalled GEMM or SpMM pipeline would report, and the kernel returns.
 * 0 < limit_ns <= 10 s.  Asynchronous on `stream`. */
TWELL_API int twell_selftest_wait_timeout(int32_t* status, uint64_t limit_ns, twell_stream_t stream);

/* Device check of a packed layout against the format rules at the top of this
 * file: a debugging aid for layouts built outside twell_pack / twell_ffn_fwd
 * (the gathers trust stored indices and slot numbers, and read out of bounds
 * when they are wrong).  Zeroes *violations (device int32, 4-byte aligned),
 * then sets bit k of it when rule k is broken anywhere in the layout:
 *    1  a cell count above C (tile variant: and not TWELL_DENSE_TILE)
 *    2  a fallback row with a non-empty cell (rows variant)
 *    3  a stored index >= T
 *    4  stored indices not strictly increasing within a cell
 *    5  a stored value that compares equal to zero
 *    6  a padding slot not (+0.0, 0)
 *    7  rows variant: row_fb below -1, or a fallback row n with slot s < fb_cap
 *       and fb_rows[s] != n; tile variant: row_fb not -1
 *    8  fallback slots not 0, 1, ... in ascending row order (rows past fb_cap
 *       keep their numbers), or fb_rows[0 .. min(n_fb, fb_cap)) not ascending
 *    9  fallback rows marked in row_fb != *n_fb
 *   10  dense-tile slots not 0, 1, ... in (row, tile) order, or past the pool
 *   11  dense tiles marked != min(*n_fb, fb_cap * n_tiles)
 *   12  a dense tile whose pool tile holds at most C non-zeros
 * When the mask is non-zero, *status becomes TWELL_ERR_BAD_FORMAT unless it
 * already holds an error.  Reads the layout's arrays; writes nothing else.
 * Two launches: one thread per cell, then one CTA that numbers the fallback
 * rows (or dense tiles) in order -- O(n_rows * n_tiles) work, not a hot path.
 * A layout straight from twell_pack or twell_ffn_fwd passes, including one
 * whose fallback overflowed fb_cap. */
TWELL_API int twell_check_format(const twell_t* layout, int32_t* violations, twell_stream_t stream);

/* Static string for a TWELL_* code. */
TWELL_API const char* twell_status_string(int code);

/* Number of kernels this library has launched in this process (all calls). */
TWELL_API int64_t twell_launch_count(void);

/* Per-kernel device timing.  While enabled (on != 0) every launch is bracketed
 * by CUDA events on its stream.  twell_profile_read synchronises the device,
 * accumulates the pending event pairs and returns, for the kernel named by
 * `kernel` (a TWELL_KERNEL_* id), the launches and total milliseconds since
 * the last reset.  twell_profile_reset clears the totals. */
enum {
  TWELL_KERNEL_UP_PACK = 0,      /* tcgen05 up-projection + bias/ReLU/TwELL-pack epilogue */
  TWELL_KERNEL_ROUTE = 1,        /* fallback routing scan */
  TWELL_KERNEL_FB_ASSEMBLE = 2,  /* dense fallback rows from spilled tiles + cells */
  TWELL_KERNEL_CHECK_FORMAT = 3, /* twell_check_format */
  TWELL_KERNEL_SPMM = 4,         /* TwELL gather-SpMM down-projection */
  TWELL_KERNEL_FB_DOWN = 5,      /* fallback rows' down-projection */
  TWELL_KERNEL_PACK = 6,         /* standalone dense -> TwELL */
  TWELL_KERNEL_UNPACK = 7,       /* TwELL -> dense */
  TWELL_KERNEL_SDDMM = 8,        /* backward: dZ at the pattern */
  TWELL_KERNEL_DX = 9,           /* backward: dX gather of the TwELL rows */
  TWELL_KERNEL_DW = 10,          /* backward: unit-major walk adding the TwELL rows' dW_down, dW_inT, db */
  TWELL_KERNEL_DENSE_GEMM = 11,  /* dense comparator GEMMs */
  TWELL_KERNEL_AUX = 12,         /* small helpers (clears, transposed indexes) */
  TWELL_KERNEL_DW_FALLBACK = 13, /* backward: the fallback rows' dW_down, dW_inT, db share */
  TWELL_KERNEL_DX_FALLBACK = 14, /* backward: the fallback rows' dX */
  TWELL_KERNEL_COUNT = 15
};
TWELL_API int twell_profile_enable(int on);
TWELL_API int twell_profile_reset(void);
TWELL_API int twell_profile_read(int kernel, int64_t* launches, double* total_ms);

/* Timeline of the launches recorded while profiling was enabled and not yet
 * consumed by twell_profile_read or cleared by twell_profile_reset, in launch
 * order: for entry i, kernel[i] (a TWELL_KERNEL_* id), stream[i] (the
 * cudaStream_t it ran on, as an integer: the caller's stream or the library's
 * second stream), and start_ms[i] / end_ms[i], the device times of the event
 * recorded on that stream just before the launch and just after it, relative
 * to the first entry's start.  Start marks when the stream reached the launch
 * (the kernel may still wait for SMs), end when it finished.  Writes at most
 * `max` entries to the caller's host arrays and returns how many it wrote, or
 * a negative TWELL_* code.  Synchronises the device; the entries stay
 * recorded. */
TWELL_API int twell_profile_timeline(int max, int32_t* kernel, uint64_t* stream, double* start_ms,
                                     double* end_ms);

#ifdef __cplusplus
}
#endif

#endif /* TWELL_H */
