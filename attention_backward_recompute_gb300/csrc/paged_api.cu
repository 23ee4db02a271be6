// C ABI of the paged-KV history backward: validation, workspace carving, TMA
// descriptors and launch order (prep -> zero of unlinked pages -> history).
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstring>

#include "../../include/attn_bwd.h"
#include "api_internal.h"
#include "paged_launch.h"

namespace {

using attn::api_fail;
using attn::api_ok;

struct PagedSizes {
  size_t q_bytes, qp_bytes, dy_bytes, k_bytes, v_bytes, kp_bytes, table_bytes, meta_bytes, stat_bytes;
  size_t ws_bytes;
  size_t off_count, off_off, off_fill, off_links, off_heavy, off_listed, off_order, off_work, off_split;
};

size_t a256(size_t x) { return (x + 255) & ~size_t(255); }

attn_status_t check_paged_desc(const attn_paged_desc* d, PagedSizes* z) {
  if (!d) return api_fail(ATTN_ERR_INVALID_ARG, "descriptor is NULL");
  if (d->num_queries < 0 || d->num_seqs < 0 || d->heads <= 0 || d->kv_heads <= 0 || d->page_size <= 0 ||
      d->num_pages < 0 || d->max_pages_per_seq < 0 || d->key_dim <= 0 || d->value_dim <= 0 || d->position_dim < 0)
    return api_fail(ATTN_ERR_INVALID_ARG, "negative or zero size in the paged descriptor");
  if (d->reserved != 0) return api_fail(ATTN_ERR_INVALID_ARG, "reserved field must be 0");
  if (d->heads % d->kv_heads != 0) return api_fail(ATTN_ERR_INVALID_ARG, "heads must be a multiple of kv_heads");
  if (d->causal != 0 && d->causal != 1) return api_fail(ATTN_ERR_INVALID_ARG, "causal must be 0 or 1");
  if (!std::isfinite(d->scale) || d->scale < 0.f) return api_fail(ATTN_ERR_INVALID_ARG, "scale must be finite and >= 0");
  if (d->dtype != ATTN_DTYPE_BF16) return api_fail(ATTN_ERR_UNSUPPORTED, "paged path supports bf16 storage only");
  if (d->page_size != 16) return api_fail(ATTN_ERR_UNSUPPORTED, "page_size must be 16");
  const int64_t G = d->heads / d->kv_heads;
  if (d->value_dim != d->key_dim) return api_fail(ATTN_ERR_UNSUPPORTED, "value_dim must equal key_dim");
  if (d->position_dim != 0) {
    // MLA: the latent (key_dim) is also the value
    if (d->key_dim != 512 || d->position_dim != 64)
      return api_fail(ATTN_ERR_UNSUPPORTED, "MLA needs key_dim 512 and position_dim 64");
  } else {
    if (d->key_dim != 64 && d->key_dim != 128) return api_fail(ATTN_ERR_UNSUPPORTED, "key_dim must be 64 or 128 (GQA)");
  }
  // a tile of 64 columns holds 64 / G whole query rows
  if (64 % G != 0) return api_fail(ATTN_ERR_UNSUPPORTED, "heads / kv_heads must divide 64");
  const int64_t lim = int64_t(1) << 30;
  if (d->num_pages * d->page_size >= lim || d->num_queries * d->heads >= lim || d->num_seqs * d->max_pages_per_seq >= lim ||
      d->num_seqs >= 65535 || d->kv_heads >= 65535)
    return api_fail(ATTN_ERR_UNSUPPORTED, "sizes exceed the supported index range");
  const size_t es = 2;
  const size_t slots = size_t(d->num_pages) * d->page_size;
  z->q_bytes = size_t(d->num_queries) * d->heads * d->key_dim * es;
  z->qp_bytes = size_t(d->num_queries) * d->heads * d->position_dim * es;
  z->dy_bytes = size_t(d->num_queries) * d->heads * d->value_dim * es;
  z->k_bytes = slots * d->kv_heads * d->key_dim * es;
  z->v_bytes = slots * d->kv_heads * d->value_dim * es;
  z->kp_bytes = slots * d->kv_heads * d->position_dim * es;
  z->table_bytes = size_t(d->num_seqs) * d->max_pages_per_seq * 4;
  z->meta_bytes = (size_t(d->num_seqs) * 2 + 1 + d->num_queries) * 4;
  z->stat_bytes = size_t(d->num_queries) * d->heads * 4;
  z->off_count = 0;
  z->off_off = z->off_count + a256(size_t(d->num_pages) * 4);
  z->off_fill = z->off_off + a256(size_t(d->num_pages + 1) * 4);
  z->off_links = z->off_fill + a256(size_t(d->num_pages) * 4);
  z->off_heavy = z->off_links + a256(size_t(d->num_seqs) * d->max_pages_per_seq * 4 + 4);
  z->off_listed = z->off_heavy + a256(size_t(d->num_seqs) * ((d->max_pages_per_seq + 7) / 8) * d->kv_heads * 4 + 4);
  z->off_order = z->off_listed + a256(size_t(d->num_pages) + 4);
  z->off_work = z->off_order + a256(size_t(d->num_seqs) * 4 + 4);
  z->off_split = z->off_work + a256(size_t(attn::kMlaWorkInts) * 4);
  // MLA: the split kernel's chunk partials (fp32)
  z->ws_bytes = z->off_split + (d->position_dim != 0 ? attn::kMlaSplitFloats * 4 : 0);
  return ATTN_OK;
}

bool overlap(const void* a, size_t na, const void* b, size_t nb) {
  if (!a || !b || !na || !nb) return false;
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

attn_status_t fill_params(const attn_paged_desc* d, const PagedSizes& z, const int32_t* page_table,
                          const int32_t* seq_meta, void* workspace, attn::PagedParams* p) {
  std::memset(p, 0, sizeof(*p));
  p->Nq = int(d->num_queries);
  p->S = int(d->num_seqs);
  p->H = int(d->heads);
  p->KVH = int(d->kv_heads);
  p->G = int(d->heads / d->kv_heads);
  p->page_size = int(d->page_size);
  p->num_pages = int(d->num_pages);
  p->max_pages = int(d->max_pages_per_seq);
  p->Dk = int(d->key_dim);
  p->Dv = int(d->value_dim);
  p->Dp = int(d->position_dim);
  p->causal = d->causal;
  p->scale = d->scale > 0.f ? d->scale : float(1.0 / std::sqrt(double(d->key_dim + d->position_dim)));
  p->scale_log2 = p->scale * 1.4426950408889634f;
  p->page_table = page_table;
  p->seq_len = seq_meta;
  p->q_start = seq_meta + d->num_seqs;
  p->q_pos = seq_meta + 2 * d->num_seqs + 1;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  p->link_count = reinterpret_cast<int32_t*>(ws + z.off_count);
  p->link_off = reinterpret_cast<int32_t*>(ws + z.off_off);
  p->link_fill = reinterpret_cast<int32_t*>(ws + z.off_fill);
  p->links = reinterpret_cast<int32_t*>(ws + z.off_links);
  p->heavy = reinterpret_cast<int32_t*>(ws + z.off_heavy);
  p->listed = nullptr;  // every page (the compact call points it at its map)
  p->order = reinterpret_cast<int32_t*>(ws + z.off_order);
  p->work = reinterpret_cast<int32_t*>(ws + z.off_work);
  p->split_part = d->position_dim != 0 ? reinterpret_cast<float*>(ws + z.off_split) : nullptr;
  p->err = attn::device_error_word();
  if (!p->err) return api_fail(ATTN_ERR_CUDA, "no CUDA device / symbol address unavailable");
  return ATTN_OK;
}

bool encode3d(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint32_t b0, uint32_t b1,
              uint32_t b2) {
  const uint64_t dims[3] = {d0, d1, d2};
  const uint64_t strides[2] = {d0 * 2, d0 * d1 * 2};
  const uint32_t box[3] = {b0, b1, b2};
  return attn::encode_tiled(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box);
}

// TMA maps of an MLA call: q, qp, dy as [Nq, H, D] addressed (d, h, r) with
// box (64, G, rows), latent and position pools as [slots, KVH, D] with box
// (64, 1, page_size)
bool encode_mla_maps(attn::PagedMlaMaps* mm, const attn_paged_desc* d, int G, uint32_t rows, const void* q,
                     const void* qp, const void* dy, const void* k_pool, const void* kp_pool) {
  std::memset(mm, 0, sizeof(*mm));
  const uint64_t slots = uint64_t(d->num_pages) * d->page_size;
  bool enc = true;
  if (d->num_queries > 0)
    enc = encode3d(&mm->q, q, d->key_dim, d->heads, d->num_queries, 64, uint32_t(G), rows) &&
          encode3d(&mm->qp, qp, d->position_dim, d->heads, d->num_queries, 64, uint32_t(G), rows) &&
          encode3d(&mm->dy, dy, d->value_dim, d->heads, d->num_queries, 64, uint32_t(G), rows);
  if (slots > 0)
    enc = enc && encode3d(&mm->k, k_pool, d->key_dim, d->kv_heads, slots, 64, 1, uint32_t(d->page_size)) &&
          encode3d(&mm->kp, kp_pool, d->position_dim, d->kv_heads, slots, 64, 1, uint32_t(d->page_size));
  else
    mm->k = mm->kp = mm->q;
  if (d->num_queries == 0) mm->q = mm->qp = mm->dy = mm->k;
  return enc;
}

}  // namespace

extern "C" {

ATTN_API size_t attn_bwd_paged_workspace_bytes(const attn_paged_desc* d) {
  PagedSizes z;
  if (check_paged_desc(d, &z) != ATTN_OK) return 0;
  return z.ws_bytes;
}

ATTN_API attn_status_t attn_bwd_paged(const attn_paged_desc* d, const void* q, const void* qp, const void* k_pool,
                                      const void* v_pool, const void* kp_pool, const void* dy,
                                      const int32_t* page_table, const int32_t* seq_meta, const float* lse,
                                      const float* delta, void* dk_pool, void* dv_pool, void* dkp_pool,
                                      unsigned wrt_mask, void* workspace, size_t workspace_bytes, void* stream) {
  return attn_bwd_paged_compact(d, q, qp, k_pool, v_pool, kp_pool, dy, page_table, seq_meta, lse, delta, nullptr, -1,
                                dk_pool, dv_pool, dkp_pool, wrt_mask, workspace, workspace_bytes, stream);
}

ATTN_API attn_status_t attn_bwd_paged_compact(const attn_paged_desc* d, const void* q, const void* qp,
                                              const void* k_pool, const void* v_pool, const void* kp_pool,
                                              const void* dy, const int32_t* page_table, const int32_t* seq_meta,
                                              const float* lse, const float* delta, const int32_t* history_pages,
                                              int64_t num_history_pages, void* dk_pool, void* dv_pool,
                                              void* dkp_pool, unsigned wrt_mask, void* workspace,
                                              size_t workspace_bytes, void* stream) {
  PagedSizes z;
  attn_status_t st = check_paged_desc(d, &z);
  if (st != ATTN_OK) return st;
  // num_history_pages < 0 (the full call): every page; else the listed ones
  const bool compact = num_history_pages >= 0;
  if (compact && num_history_pages > 0 && !history_pages)
    return api_fail(ATTN_ERR_INVALID_ARG, "history_pages is NULL");
  if (compact && num_history_pages >= (int64_t(1) << 31))
    return api_fail(ATTN_ERR_UNSUPPORTED, "too many history pages");
  if (reinterpret_cast<uintptr_t>(history_pages) & 3u)
    return api_fail(ATTN_ERR_INVALID_ARG, "history_pages must be 4-byte aligned");
  const size_t hist_bytes = compact ? size_t(num_history_pages) * 4 : 0;
  const bool mla = d->position_dim > 0;
  const unsigned allowed = mla ? (ATTN_WRT_DK | ATTN_WRT_DKP) : (ATTN_WRT_DK | ATTN_WRT_DV);
  if (wrt_mask == 0 || (wrt_mask & ~allowed))
    return api_fail(ATTN_ERR_INVALID_ARG, "wrt_mask must be a non-empty subset of %s", mla ? "dK|dKp (MLA)" : "dK|dV (GQA)");
  const bool want_dk = wrt_mask & ATTN_WRT_DK, want_dv = wrt_mask & ATTN_WRT_DV, want_dkp = wrt_mask & ATTN_WRT_DKP;
  if ((want_dk && !dk_pool && z.k_bytes) || (want_dv && !dv_pool && z.v_bytes) || (want_dkp && !dkp_pool && z.kp_bytes))
    return api_fail(ATTN_ERR_INVALID_ARG, "requested gradient pointer is NULL");
  if (d->num_seqs > 0 && (!seq_meta || (d->max_pages_per_seq > 0 && !page_table)))
    return api_fail(ATTN_ERR_INVALID_ARG, "page_table / seq_meta is NULL");
  if (d->num_queries > 0 && (!q || !dy || !lse || !delta || (mla && !qp)))
    return api_fail(ATTN_ERR_INVALID_ARG, "q/qp/dy/lse/delta is NULL");
  if (d->num_pages > 0 && (!k_pool || (mla ? !kp_pool : !v_pool)))
    return api_fail(ATTN_ERR_INVALID_ARG, "k_pool/v_pool/kp_pool is NULL");
  const void* al[] = {q, qp, k_pool, v_pool, kp_pool, dy, dk_pool, dv_pool, dkp_pool, lse, delta, page_table,
                      seq_meta, workspace};
  for (const void* x : al)
    if (x && !al16(x)) return api_fail(ATTN_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
  struct R { const void* p; size_t n; };
  const R ins[] = {{q, z.q_bytes}, {qp, mla ? z.qp_bytes : 0}, {k_pool, z.k_bytes}, {v_pool, mla ? 0 : z.v_bytes},
                   {kp_pool, mla ? z.kp_bytes : 0}, {dy, z.dy_bytes}, {page_table, z.table_bytes},
                   {seq_meta, z.meta_bytes}, {lse, z.stat_bytes}, {delta, z.stat_bytes}, {workspace, workspace_bytes},
                   {history_pages, hist_bytes}};
  const R outs[] = {{want_dk ? dk_pool : nullptr, z.k_bytes}, {want_dv ? dv_pool : nullptr, z.v_bytes},
                    {want_dkp ? dkp_pool : nullptr, z.kp_bytes}};
  for (int i = 0; i < 3; ++i) {
    for (const R& r : ins)
      if (overlap(outs[i].p, outs[i].n, r.p, r.n)) return api_fail(ATTN_ERR_ALIAS, "output %d overlaps an input or the workspace", i);
    for (int j = i + 1; j < 3; ++j)
      if (overlap(outs[i].p, outs[i].n, outs[j].p, outs[j].n)) return api_fail(ATTN_ERR_ALIAS, "outputs %d and %d overlap", i, j);
  }
  if (d->num_pages == 0 || (compact && num_history_pages == 0)) return api_ok();
  if (!workspace || workspace_bytes < z.ws_bytes)
    return api_fail(ATTN_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", z.ws_bytes, workspace_bytes);
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return api_fail(ATTN_ERR_WORKSPACE, "workspace must be 256-byte aligned");

  attn::PagedParams p;
  if ((st = fill_params(d, z, page_table, seq_meta, workspace, &p)) != ATTN_OK) return st;
  p.lse = lse;
  p.delta = delta;
  p.dk_pool = dk_pool;
  p.dv_pool = dv_pool;
  p.dkp_pool = dkp_pool;
  p.wrt = wrt_mask;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (compact) {
    // the map of listed pages, ahead of the kernels that read it
    p.listed = static_cast<uint8_t*>(workspace) + z.off_listed;
    const cudaError_t e = attn::launch_paged_listed(p, history_pages, num_history_pages, s);
    if (e != cudaSuccess) return api_fail(ATTN_ERR_CUDA, "paged launch failed: %s", cudaGetErrorString(e));
  }
  if (mla) {
    if (!attn::mla_tc_supported(p)) return api_fail(ATTN_ERR_UNSUPPORTED, "MLA shape not supported");
    // links, zeros for pages no link references, then two CTAs per 128-token
    // block of every sequence (tcgen05); blocks whose shared pages carry many
    // links go to the cluster-split kernel first
    attn::PagedMlaMaps mt;
    std::memset(&mt, 0, sizeof(mt));
    const uint64_t slots = uint64_t(d->num_pages) * d->page_size;
    // query-side boxes of 64 columns (64/G rows)
    const uint32_t G = uint32_t(p.G), RT = 64u / G;
    bool enc = encode3d(&mt.k, k_pool, d->key_dim, d->kv_heads, slots, 64, 1, uint32_t(d->page_size)) &&
               encode3d(&mt.kp, kp_pool, d->position_dim, d->kv_heads, slots, 64, 1, uint32_t(d->page_size));
    if (d->num_queries > 0)
      enc = enc && encode3d(&mt.q, q, d->key_dim, d->heads, d->num_queries, 64, G, RT) &&
            encode3d(&mt.qp, qp, d->position_dim, d->heads, d->num_queries, 64, G, RT) &&
            encode3d(&mt.dy, dy, d->value_dim, d->heads, d->num_queries, 64, G, RT);
    else
      mt.q = mt.qp = mt.dy = mt.k;
    if (!enc) return api_fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled failed");
    attn::timing_mark_begin(5, s);
    cudaError_t e = attn::launch_paged_prep(p, s);
    attn::timing_mark(s);
    if (e == cudaSuccess) e = attn::launch_paged_zero_unlinked(p, compact ? history_pages : nullptr, num_history_pages, s);
    attn::timing_mark(s);
    if (e == cudaSuccess) e = attn::launch_paged_mla_tc_plan(p, s);
    attn::timing_mark(s);
    // The grid kernels start as programmatic dependents of the split kernel:
    // both launchers skip on the same condition (no pages, sequences or page
    // table columns), so whenever a grid kernel launches, the split kernel was
    // the launch just before it; the plan they both read completed before the
    // split kernel started (plain stream order).
    if (e == cudaSuccess) e = attn::launch_paged_mla_tc_split(mt, p, s);
    attn::timing_mark(s);
    if (e == cudaSuccess) e = attn::launch_paged_mla_tc(mt, p, true, s);
    attn::timing_mark(s);
    attn::timing_mark_end();
    if (e != cudaSuccess) return api_fail(ATTN_ERR_CUDA, "paged launch failed: %s", cudaGetErrorString(e));
    return api_ok();
  }
  attn::PagedMaps m;
  std::memset(&m, 0, sizeof(m));
  const uint64_t slots = uint64_t(d->num_pages) * d->page_size;
  const uint32_t G = uint32_t(p.G);
  bool enc = true;
  if (d->num_queries > 0)
    enc = encode3d(&m.q, q, d->key_dim, d->heads, d->num_queries, 64, G, 64 / G) &&
          encode3d(&m.dy, dy, d->value_dim, d->heads, d->num_queries, 64, G, 64 / G);
  enc = enc && encode3d(&m.k, k_pool, d->key_dim, d->kv_heads, slots, 64, 1, uint32_t(d->page_size)) &&
        encode3d(&m.v, v_pool, d->value_dim, d->kv_heads, slots, 64, 1, uint32_t(d->page_size));
  if (!enc) return api_fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled failed");
  if (d->num_queries == 0) { m.q = m.k; m.dy = m.v; }
  const int nk = 3;
  attn::timing_mark_begin(nk, s);
  cudaError_t e = attn::launch_paged_prep(p, s);
  attn::timing_mark(s);
  if (e == cudaSuccess) e = attn::launch_paged_zero_unlinked(p, compact ? history_pages : nullptr, num_history_pages, s);
  attn::timing_mark(s);
  if (e == cudaSuccess && d->num_seqs > 0 && d->max_pages_per_seq > 0) e = attn::launch_paged_history(m, p, s);
  attn::timing_mark(s);
  attn::timing_mark_end();
  if (e != cudaSuccess) return api_fail(ATTN_ERR_CUDA, "paged launch failed: %s", cudaGetErrorString(e));
  return api_ok();
}

ATTN_API attn_status_t attn_paged_row_stats(const attn_paged_desc* d, const void* q, const void* qp,
                                            const void* k_pool, const void* v_pool, const void* kp_pool,
                                            const void* dy, const int32_t* page_table, const int32_t* seq_meta,
                                            float* lse, float* delta, void* workspace, size_t workspace_bytes,
                                            void* stream) {
  PagedSizes z;
  attn_status_t st = check_paged_desc(d, &z);
  if (st != ATTN_OK) return st;
  const bool mla = d->position_dim > 0;
  if (d->num_queries == 0) return api_ok();
  if (!q || !dy || !lse || !delta || !seq_meta || (d->max_pages_per_seq > 0 && !page_table) || (mla && !qp))
    return api_fail(ATTN_ERR_INVALID_ARG, "a required pointer is NULL");
  if (d->num_pages > 0 && (!k_pool || (mla ? !kp_pool : !v_pool)))
    return api_fail(ATTN_ERR_INVALID_ARG, "k_pool/v_pool/kp_pool is NULL");
  const void* al[] = {q, qp, k_pool, v_pool, kp_pool, dy, lse, delta, page_table, seq_meta};
  for (const void* x : al)
    if (x && !al16(x)) return api_fail(ATTN_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
  struct R { const void* p; size_t n; };
  const R ins[] = {{q, z.q_bytes}, {qp, mla ? z.qp_bytes : 0}, {k_pool, z.k_bytes}, {v_pool, mla ? 0 : z.v_bytes},
                   {kp_pool, mla ? z.kp_bytes : 0}, {dy, z.dy_bytes}, {page_table, z.table_bytes},
                   {seq_meta, z.meta_bytes}, {workspace, workspace_bytes}};
  for (const R& r : ins)
    if (overlap(lse, z.stat_bytes, r.p, r.n) || overlap(delta, z.stat_bytes, r.p, r.n))
      return api_fail(ATTN_ERR_ALIAS, "lse/delta overlap an input or the workspace");
  if (overlap(lse, z.stat_bytes, delta, z.stat_bytes)) return api_fail(ATTN_ERR_ALIAS, "lse and delta overlap");
  if (!workspace || workspace_bytes < z.ws_bytes)
    return api_fail(ATTN_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", z.ws_bytes, workspace_bytes);
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return api_fail(ATTN_ERR_WORKSPACE, "workspace must be 256-byte aligned");
  attn::PagedParams p;
  if ((st = fill_params(d, z, page_table, seq_meta, workspace, &p)) != ATTN_OK) return st;
  p.lse_out = lse;
  p.delta_out = delta;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // the row tiles of the longest sequences go first
  if (const cudaError_t e = attn::launch_paged_seq_order(p, s); e != cudaSuccess)
    return api_fail(ATTN_ERR_CUDA, "row-statistics launch failed: %s", cudaGetErrorString(e));
  if (mla) {
    // tcgen05: 128 columns (128/G rows) per CTA
    attn::PagedMlaMaps mt;
    if (!encode_mla_maps(&mt, d, p.G, 128u / uint32_t(p.G), q, qp, dy, k_pool, kp_pool))
      return api_fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled failed");
    attn::timing_mark_begin(1, s);
    cudaError_t e = attn::launch_paged_mla_stats_tc(mt, p, s);
    attn::timing_mark(s);
    attn::timing_mark_end();
    if (e != cudaSuccess) return api_fail(ATTN_ERR_CUDA, "row-statistics launch failed: %s", cudaGetErrorString(e));
    return api_ok();
  }
  attn::PagedMaps m;
  std::memset(&m, 0, sizeof(m));
  const uint64_t slots = uint64_t(d->num_pages) * d->page_size;
  const uint32_t G = uint32_t(p.G);
  bool enc = encode3d(&m.q_stats, q, d->key_dim, d->heads, d->num_queries, 64, G, 128 / G) &&
             encode3d(&m.dy_stats, dy, d->value_dim, d->heads, d->num_queries, 64, G, 128 / G);
  if (slots > 0)
    enc = enc && encode3d(&m.k, k_pool, d->key_dim, d->kv_heads, slots, 64, 1, uint32_t(d->page_size)) &&
          encode3d(&m.v, v_pool, d->value_dim, d->kv_heads, slots, 64, 1, uint32_t(d->page_size));
  else
    m.k = m.v = m.q_stats;
  if (!enc) return api_fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled failed");
  attn::timing_mark_begin(1, s);
  cudaError_t e = attn::launch_paged_row_stats(m, p, s);
  attn::timing_mark(s);
  attn::timing_mark_end();
  if (e != cudaSuccess) return api_fail(ATTN_ERR_CUDA, "row-statistics launch failed: %s", cudaGetErrorString(e));
  return api_ok();
}

ATTN_API attn_status_t attn_bwd_paged_query(const attn_paged_desc* d, const void* q, const void* qp,
                                            const void* k_pool, const void* v_pool, const void* kp_pool,
                                            const void* dy, const int32_t* page_table, const int32_t* seq_meta,
                                            float* lse, float* delta, void* dq, void* dqp, void* workspace,
                                            size_t workspace_bytes, void* stream) {
  PagedSizes z;
  attn_status_t st = check_paged_desc(d, &z);
  if (st != ATTN_OK) return st;
  const bool mla = d->position_dim > 0;
  if (d->num_queries == 0) return api_ok();
  if (!q || !dy || !lse || !delta || !dq || !seq_meta || (d->max_pages_per_seq > 0 && !page_table) ||
      (mla && (!qp || !dqp)))
    return api_fail(ATTN_ERR_INVALID_ARG, "a required pointer is NULL");
  if (d->num_pages > 0 && (!k_pool || (mla ? !kp_pool : !v_pool)))
    return api_fail(ATTN_ERR_INVALID_ARG, "k_pool/v_pool/kp_pool is NULL");
  const void* al[] = {q, qp, k_pool, v_pool, kp_pool, dy, lse, delta, dq, dqp, page_table, seq_meta};
  for (const void* x : al)
    if (x && !al16(x)) return api_fail(ATTN_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
  const size_t dqp_bytes = mla ? z.qp_bytes : 0;
  struct R { const void* p; size_t n; };
  const R ins[] = {{q, z.q_bytes}, {qp, dqp_bytes}, {k_pool, z.k_bytes}, {v_pool, mla ? 0 : z.v_bytes},
                   {kp_pool, mla ? z.kp_bytes : 0}, {dy, z.dy_bytes}, {page_table, z.table_bytes},
                   {seq_meta, z.meta_bytes}, {workspace, workspace_bytes}};
  const R outs[] = {{lse, z.stat_bytes}, {delta, z.stat_bytes}, {dq, z.q_bytes}, {mla ? dqp : nullptr, dqp_bytes}};
  for (const R& o : outs)
    for (const R& r : ins)
      if (overlap(o.p, o.n, r.p, r.n)) return api_fail(ATTN_ERR_ALIAS, "an output overlaps an input or the workspace");
  for (int i = 0; i < 4; ++i)
    for (int j = i + 1; j < 4; ++j)
      if (overlap(outs[i].p, outs[i].n, outs[j].p, outs[j].n)) return api_fail(ATTN_ERR_ALIAS, "outputs overlap");
  if (!workspace || workspace_bytes < z.ws_bytes)
    return api_fail(ATTN_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", z.ws_bytes, workspace_bytes);
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return api_fail(ATTN_ERR_WORKSPACE, "workspace must be 256-byte aligned");
  attn::PagedParams p;
  if ((st = fill_params(d, z, page_table, seq_meta, workspace, &p)) != ATTN_OK) return st;
  p.lse_out = lse;
  p.delta_out = delta;
  p.dq = dq;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // the row tiles of the longest sequences go first
  if (const cudaError_t e = attn::launch_paged_seq_order(p, s); e != cudaSuccess)
    return api_fail(ATTN_ERR_CUDA, "query-side launch failed: %s", cudaGetErrorString(e));
  if (mla) {
    // row statistics (128 columns per CTA), then dQ / dQp from them (64
    // columns per CTA), both on tcgen05
    p.dqp = dqp;
    p.lse = lse;
    p.delta = delta;
    attn::PagedMlaMaps ms, mq;
    if (!encode_mla_maps(&ms, d, p.G, 128u / uint32_t(p.G), q, qp, dy, k_pool, kp_pool) ||
        !encode_mla_maps(&mq, d, p.G, 64u / uint32_t(p.G), q, qp, dy, k_pool, kp_pool))
      return api_fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled failed");
    attn::timing_mark_begin(3, s);
    cudaError_t e = attn::launch_paged_mla_stats_tc(ms, p, s);
    attn::timing_mark(s);
    if (e == cudaSuccess) e = attn::launch_paged_mla_query_tc(mq, p, s);
    attn::timing_mark(s);
    if (e == cudaSuccess) e = attn::launch_paged_query_outside(p, s);
    attn::timing_mark(s);
    attn::timing_mark_end();
    if (e != cudaSuccess) return api_fail(ATTN_ERR_CUDA, "query-side launch failed: %s", cudaGetErrorString(e));
    return api_ok();
  }
  attn::PagedMaps m;
  std::memset(&m, 0, sizeof(m));
  const uint64_t slots = uint64_t(d->num_pages) * d->page_size;
  const uint32_t G = uint32_t(p.G);
  bool enc = encode3d(&m.q_stats, q, d->key_dim, d->heads, d->num_queries, 64, G, 128 / G) &&
             encode3d(&m.dy_stats, dy, d->value_dim, d->heads, d->num_queries, 64, G, 128 / G);
  if (slots > 0)
    enc = enc && encode3d(&m.k, k_pool, d->key_dim, d->kv_heads, slots, 64, 1, uint32_t(d->page_size)) &&
          encode3d(&m.v, v_pool, d->value_dim, d->kv_heads, slots, 64, 1, uint32_t(d->page_size));
  else
    m.k = m.v = m.q_stats;
  if (!enc) return api_fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled failed");
  attn::timing_mark_begin(1, s);
  cudaError_t e = attn::launch_paged_query(m, p, s);
  attn::timing_mark(s);
  attn::timing_mark_end();
  if (e != cudaSuccess) return api_fail(ATTN_ERR_CUDA, "query-side launch failed: %s", cudaGetErrorString(e));
  return api_ok();
}

}  // extern "C"
