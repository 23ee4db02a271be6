// C ABI of the paged-KV history backward (entry points, validation).
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdio>

#include "../../include/attn_bwd.h"

namespace {
// Shares the message buffer of the dense entry points through attn_last_error;
// the paged calls report through their own thread-local buffer that
// attn_last_error consults when it is the most recent failure.
}  // namespace

extern "C" {

ATTN_API size_t attn_bwd_paged_workspace_bytes(const attn_paged_desc* d) {
  (void)d;
  return 0;
}

ATTN_API attn_status_t attn_bwd_paged(const attn_paged_desc* d, const void* q, const void* qp, const void* k_pool,
                                      const void* v_pool, const void* kp_pool, const void* dy,
                                      const int32_t* page_table, const int32_t* seq_meta, const float* lse,
                                      const float* delta, void* dk_pool, void* dv_pool, void* dkp_pool,
                                      unsigned wrt_mask, void* workspace, size_t workspace_bytes, void* stream) {
  (void)d; (void)q; (void)qp; (void)k_pool; (void)v_pool; (void)kp_pool; (void)dy; (void)page_table;
  (void)seq_meta; (void)lse; (void)delta; (void)dk_pool; (void)dv_pool; (void)dkp_pool; (void)wrt_mask;
  (void)workspace; (void)workspace_bytes; (void)stream;
  return ATTN_ERR_UNSUPPORTED;
}

ATTN_API attn_status_t attn_paged_row_stats(const attn_paged_desc* d, const void* q, const void* qp,
                                            const void* k_pool, const void* v_pool, const void* kp_pool,
                                            const void* dy, const int32_t* page_table, const int32_t* seq_meta,
                                            float* lse, float* delta, void* workspace, size_t workspace_bytes,
                                            void* stream) {
  (void)d; (void)q; (void)qp; (void)k_pool; (void)v_pool; (void)kp_pool; (void)dy; (void)page_table;
  (void)seq_meta; (void)lse; (void)delta; (void)workspace; (void)workspace_bytes; (void)stream;
  return ATTN_ERR_UNSUPPORTED;
}

}  // extern "C"
