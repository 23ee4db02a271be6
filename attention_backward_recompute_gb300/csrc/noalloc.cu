// attn_bwd_dense_noalloc: the dense backward without a caller-provided
// workspace, for callers that cannot allocate device memory themselves.
//
// The row statistics the dense backward needs (three fp32 values per
// (batch, head, query row)) live in a file-scope device array of fixed size
// that the library owns: it is part of this module's device image, so every
// GPU that loads the library holds it until the process exits, and no call
// allocates anything.  The call forwards to attn_bwd_dense with that array as
// its workspace; inputs and outputs are still the caller's.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/attn_bwd.h"
#include "api_internal.h"

namespace {

// Bytes of the scratch array: room for ATTN_NOALLOC_MAX_ROWS rows of row
// statistics (three fp32 arrays, each rounded up to 256 bytes).
constexpr size_t kRows = ATTN_NOALLOC_MAX_ROWS;
constexpr size_t kScratchBytes = 3 * ((kRows * 4 + 255) & ~size_t(255));

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

// Device address of the scratch array for the current device.  In host code
// the array's name is only a host-side stand-in, so the address comes from
// cudaGetSymbolAddress, once per device, with that device current.  The
// cached address belongs to the device's primary context: after
// cudaDeviceReset (which tears that context down) it is stale, and this entry
// point must not be used again in the process.
void* scratch_address() {
  static void* addr[64] = {nullptr};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lk(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
    addr[dev] = p;
  }
  return addr[dev];
}

}  // namespace

extern "C" ATTN_API attn_status_t attn_bwd_dense_noalloc(const attn_dense_desc* d, const void* q, const void* k,
                                                         const void* v, const void* dy, const float* key_mask,
                                                         const void* bias, const void* o, const float* lse,
                                                         void* dq, void* dk, void* dv, unsigned wrt_mask,
                                                         void* stream) {
  if (!d) return attn::api_fail(ATTN_ERR_INVALID_ARG, "descriptor is NULL");
  if (d->batch < 0 || d->heads < 0 || d->seq_q < 0) return attn::api_fail(ATTN_ERR_INVALID_ARG, "negative size");
  if (d->dtype != ATTN_DTYPE_BF16)
    return attn::api_fail(ATTN_ERR_UNSUPPORTED,
                          "the library-owned scratch holds row statistics only; fp32 storage also needs split "
                          "copies of the inputs: use attn_bwd_dense with a workspace");
  if (d->mask_flags & ATTN_MASK_ELEM)
    return attn::api_fail(ATTN_ERR_UNSUPPORTED,
                          "the per-element mask's packed bits do not fit the library-owned scratch: use "
                          "attn_bwd_dense_strided with a workspace");
  if (d->options & ATTN_OPT_STORE_DS)
    return attn::api_fail(ATTN_ERR_UNSUPPORTED,
                          "stored dS does not fit the library-owned scratch: use attn_bwd_dense with a workspace");
  const double rows = double(d->batch) * double(d->heads) * double(d->seq_q);
  if (rows > double(kRows))
    return attn::api_fail(ATTN_ERR_UNSUPPORTED,
                          "batch*heads*seq_q = %.0f exceeds the %zu rows of the library-owned scratch; use "
                          "attn_bwd_dense with a workspace",
                          rows, kRows);
  void* ws = scratch_address();
  if (!ws) return attn::api_fail(ATTN_ERR_CUDA, "no CUDA device or the scratch address is unavailable");
  // Every row statistic the kernels read is written earlier in the same call,
  // so the scratch needs no clearing between calls.
  return attn_bwd_dense(d, q, k, v, dy, key_mask, bias, o, lse, dq, dk, dv, wrt_mask, ws, kScratchBytes, stream);
}
