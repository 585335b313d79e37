// twell_ffn_fwd_noalloc: the forward pass for callers that cannot allocate
// device memory themselves.
//
// Some callers have no allocator to hand: code that runs inside another
// framework's memory pool without access to it, plugins loaded into a host
// application that owns every cudaMalloc, or real-time paths where a
// cudaMalloc (which may synchronise the device) is not allowed.  They still
// pass their own inputs and outputs, but cannot supply the forward pass's
// scratch buffer.  This entry point keeps that scratch in a fixed array in
// device memory that is part of the library image.
//
// The array holds what the caller's workspace holds for twell_ffn_fwd, whose
// size twell_fwd_workspace_bytes(...) gives: the dense tiles spilled by
// overflowing cells, the call's counters and overflow flags, the K-split
// partial sums of the fallback rows' down-projection and, for batches of at
// most 32 rows, the up-projection's K-split partial sums, a dense copy of h
// and the gather's tile-range partials.  At most kNoAllocScratchBytes; every
// GPU that loads the library keeps the array until the process exits.
#include <cuda_runtime.h>

#include <mutex>

#include "twell_internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = 4u << 20;  // 4 MiB

static __device__ __align__(256) unsigned char g_fwd_scratch[kNoAllocScratchBytes];

// Device address of g_fwd_scratch, looked up once per device.  In host code
// the symbol names a host-side stand-in, never device memory, so kernels must
// get this address instead.
std::mutex g_scratch_mu;
void* g_scratch_ptr[64] = {};

int scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return TWELL_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_fwd_scratch) != cudaSuccess || !p) return TWELL_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return TWELL_OK;
}

}  // namespace

extern "C" TWELL_API size_t twell_ffn_fwd_noalloc_max_scratch(void) { return kNoAllocScratchBytes; }

extern "C" TWELL_API int twell_ffn_fwd_noalloc(const uint16_t* X, const uint16_t* W_inT, const uint16_t* b,
                                               const uint16_t* W_down, int32_t n_rows, int32_t d_model,
                                               int32_t d_ff, const twell_t* H, uint16_t* Y,
                                               twell_stream_t stream) {
  if (!H) return TWELL_ERR_INVALID_ARG;
  const size_t need = twell_fwd_workspace_bytes(n_rows, d_model, d_ff, H->tile, H->cap, H->fb_cap);
  if (need > kNoAllocScratchBytes) return TWELL_ERR_WORKSPACE;
  if (!twell::device_is_sm103()) return TWELL_ERR_NO_DEVICE;
  void* scratch = nullptr;
  const int rc = scratch_for_current_device(&scratch);
  if (rc != TWELL_OK) return rc;
  return twell_ffn_fwd(X, W_inT, b, W_down, n_rows, d_model, d_ff, H, Y, scratch, kNoAllocScratchBytes, stream);
}
