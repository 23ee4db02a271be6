// C ABI of libattnbwd: argument validation, workspace carving, TMA descriptor
// construction and kernel orchestration.  See include/attn_bwd.h for the
// contract of every entry point.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <limits>
#include <mutex>

#include "../../include/attn_bwd.h"
#include "api_internal.h"
#include "dense_launch.h"

namespace {

thread_local char g_msg[512] = "";
thread_local void* const* g_events = nullptr;
thread_local int g_event_count = 0;
thread_local int g_event_next = 0;

// device error word (one per device), set by kernels whose bounded waits expire
__device__ uint32_t g_device_error;

}  // namespace

namespace attn {

attn_status_t api_fail(attn_status_t st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
  return st;
}

attn_status_t api_ok() {
  g_msg[0] = '\0';
  return ATTN_OK;
}

uint32_t* device_error_word() {
  static uint32_t* ptrs[64] = {nullptr};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lk(mu);
  if (!ptrs[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
    ptrs[dev] = static_cast<uint32_t*>(p);
  }
  return ptrs[dev];
}

void timing_mark_begin(int kernels, cudaStream_t s) {
  if (g_events && g_event_count < kernels + 1) g_events = nullptr;
  g_event_next = 0;
  timing_mark(s);
}

void timing_mark(cudaStream_t s) {
  if (g_events && g_event_next < g_event_count)
    cudaEventRecord(static_cast<cudaEvent_t>(g_events[g_event_next]), s);
  ++g_event_next;
}

void timing_mark_end() {
  g_events = nullptr;
  g_event_count = 0;
  g_event_next = 0;
}

}  // namespace attn

namespace {

using attn::api_fail;
using attn::api_ok;
using attn::device_error_word;

// ---------------------------------------------------------------------------
// TMA descriptor encoding through the driver entry point
// ---------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

}  // namespace

bool attn::encode_tiled(CUtensorMap* m, CUtensorMapDataType dt, int rank, const void* base, const uint64_t* dims,
                        const uint64_t* strides, const uint32_t* box) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || rank < 1 || rank > 5) return false;
  cuuint64_t gd[5], gs[4];
  cuuint32_t bx[5], es[5];
  for (int i = 0; i < rank; ++i) {
    gd[i] = dims[i];
    bx[i] = box[i];
    es[i] = 1;
    if (i + 1 < rank) gs[i] = strides[i];
  }
  return fn(m, dt, cuuint32_t(rank), const_cast<void*>(base), gd, gs, bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {

// 4-D map over a [B, S, H, D]-like tensor addressed as (d, s, h, b).
bool encode4d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, const uint64_t dims[4],
              const uint64_t strides_bytes[3], uint32_t box0, uint32_t box1) {
  const uint32_t box[4] = {box0, box1, 1, 1};
  return attn::encode_tiled(m, dt, 4, base, dims, strides_bytes, box);
}

bool ranges_overlap(const void* a, size_t na, const void* b, size_t nb) {
  if (!a || !b || na == 0 || nb == 0) return false;
  const uintptr_t x0 = reinterpret_cast<uintptr_t>(a), x1 = x0 + na;
  const uintptr_t y0 = reinterpret_cast<uintptr_t>(b), y1 = y0 + nb;
  return x0 < y1 && y0 < x1;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct DenseSizes {
  size_t es, q_bytes, k_bytes, bias_bytes, mask_bytes, stat_bytes, ws_bytes;
  size_t split_off;  // fp32 storage: offset of the hi/lo bf16 copies of q, k, v, dy
  size_t elem_off;   // per-element mask: offset of its row and column bits
  size_t ds_off;     // ATTN_OPT_STORE_DS: offset of the stored dS tiles
  int ew_q, ew_k;    // 32-bit words per query row / key column of those bits (even)
};

attn_status_t check_dense_desc(const attn_dense_desc* d, DenseSizes* z) {
  if (!d) return api_fail(ATTN_ERR_INVALID_ARG, "descriptor is NULL");
  if (d->batch < 0 || d->heads < 0 || d->seq_q < 0 || d->seq_k < 0 || d->head_dim <= 0)
    return api_fail(ATTN_ERR_INVALID_ARG, "negative size or head_dim <= 0");
  if (d->dtype != ATTN_DTYPE_F32 && d->dtype != ATTN_DTYPE_BF16)
    return api_fail(ATTN_ERR_INVALID_ARG, "unknown dtype %d", d->dtype);
  if (d->layout != ATTN_LAYOUT_BSHD && d->layout != ATTN_LAYOUT_BHSD)
    return api_fail(ATTN_ERR_INVALID_ARG, "unknown layout %d", d->layout);
  if (d->mask_flags & ~63u) return api_fail(ATTN_ERR_INVALID_ARG, "unknown mask flag bits 0x%x", d->mask_flags);
  if ((d->mask_flags & ATTN_MASK_WINDOW) && d->window < 0) return api_fail(ATTN_ERR_INVALID_ARG, "window < 0");
  if (d->options & ~ATTN_OPT_STORE_DS) return api_fail(ATTN_ERR_INVALID_ARG, "unknown option bits 0x%x", d->options);
  if (!std::isfinite(d->mask_neg) || !(d->mask_neg < 0.f)) return api_fail(ATTN_ERR_INVALID_ARG, "mask_neg must be finite and < 0");
  if (!std::isfinite(d->mask_thr)) return api_fail(ATTN_ERR_INVALID_ARG, "mask_thr must be finite");
  if (!std::isfinite(d->scale) || d->scale < 0.f) return api_fail(ATTN_ERR_INVALID_ARG, "scale must be finite and >= 0");
  const int64_t D = d->head_dim;
  if (D != 8 && D != 16 && D != 32 && D != 64 && D != 128)
    return api_fail(ATTN_ERR_UNSUPPORTED, "head_dim %lld not supported (8, 16, 32, 64, 128)", (long long)D);
  const int64_t lim = int64_t(1) << 31;
  if (d->batch * d->heads >= lim || d->seq_q >= lim || d->seq_k >= lim || d->batch * d->heads * d->seq_q >= lim)
    return api_fail(ATTN_ERR_UNSUPPORTED, "sizes exceed 32-bit indexing");
  if (d->seq_k > 65535LL * 128 || d->seq_q > 65535LL * 128) return api_fail(ATTN_ERR_UNSUPPORTED, "sequence too long");
  z->es = d->dtype == ATTN_DTYPE_BF16 ? 2 : 4;
  z->q_bytes = size_t(d->batch) * d->heads * d->seq_q * D * z->es;
  z->k_bytes = size_t(d->batch) * d->heads * d->seq_k * D * z->es;
  z->bias_bytes = size_t(d->batch) * d->heads * d->seq_q * d->seq_k * z->es;
  z->mask_bytes = size_t(d->batch) * d->seq_k * 4;
  z->stat_bytes = size_t(d->batch) * d->heads * d->seq_q * 4;
  z->split_off = 3 * align256(z->stat_bytes);
  z->ws_bytes = z->split_off;
  if (d->dtype == ATTN_DTYPE_F32) {
    // fp32 storage runs on bf16 tensor cores with every operand split into
    // hi + lo bf16 copies (three products per GEMM); head_dim <= 64 fits the
    // doubled tiles in shared memory.
    if (D > 64) return api_fail(ATTN_ERR_UNSUPPORTED, "fp32 storage supports head_dim <= 64");
    if (d->mask_flags & ATTN_MASK_BIAS) return api_fail(ATTN_ERR_UNSUPPORTED, "fp32 storage does not take a bias");
    if (d->mask_flags & ATTN_MASK_ELEM) return api_fail(ATTN_ERR_UNSUPPORTED, "fp32 storage does not take a per-element mask");
    if (d->options & ATTN_OPT_STORE_DS) return api_fail(ATTN_ERR_UNSUPPORTED, "fp32 storage does not store dS");
    z->ws_bytes += 4 * align256(z->q_bytes / 2) + 4 * align256(z->k_bytes / 2);
  }
  z->elem_off = z->ws_bytes;
  z->ew_q = z->ew_k = 0;
  if (d->mask_flags & ATTN_MASK_ELEM) {
    // bits of the mask, rows [BH, Sq, ew_q] and columns [BH, Sk, ew_k]; even
    // widths so the kernels read 64-bit words
    z->ew_q = int(((d->seq_k + 31) / 32 + 1) & ~int64_t(1));
    z->ew_k = int(((d->seq_q + 31) / 32 + 1) & ~int64_t(1));
    const size_t bh = size_t(d->batch) * d->heads;
    z->ws_bytes += align256(bh * d->seq_q * z->ew_q * 4) + align256(bh * d->seq_k * z->ew_k * 4);
  }
  z->ds_off = z->ws_bytes;
  if (d->options & ATTN_OPT_STORE_DS) {  // dS^T tiles of 128 keys x 64 queries, bf16
    const int64_t tiles = d->batch * d->heads * ((d->seq_k + 127) / 128) * ((d->seq_q + 63) / 64);
    if (tiles >= lim) return api_fail(ATTN_ERR_UNSUPPORTED, "too many dS tiles to store (%lld)", (long long)tiles);
    z->ws_bytes += align256(size_t(tiles) * 16384);
  }
  if (z->ws_bytes == 0) z->ws_bytes = 256;
  return ATTN_OK;
}

// Strides of the descriptor's layout ([B,S,H,D] or [B,H,S,D], contiguous).
void layout_strides(const attn_dense_desc* d, attn_dense_strides* st) {
  const int64_t H = d->heads, Sq = d->seq_q, Sk = d->seq_k, D = d->head_dim;
  attn_strides3 q, k;
  if (d->layout == ATTN_LAYOUT_BSHD) {
    q = attn_strides3{Sq * H * D, H * D, D};
    k = attn_strides3{Sk * H * D, H * D, D};
  } else {
    q = attn_strides3{H * Sq * D, D, Sq * D};
    k = attn_strides3{H * Sk * D, D, Sk * D};
  }
  st->q = st->dy = st->o = st->dq = q;
  st->k = st->v = st->dk = st->dv = k;
}

bool same3(const attn_strides3& a, const attn_strides3& b) {
  return a.batch == b.batch && a.seq == b.seq && a.head == b.head;
}

// Bytes from a tensor's base to one past its last element.
size_t extent_bytes(const attn_strides3& x, int64_t B, int64_t S, int64_t H, int64_t D, size_t es) {
  if (B == 0 || S == 0 || H == 0 || D == 0) return 0;
  return size_t((B - 1) * x.batch + (S - 1) * x.seq + (H - 1) * x.head + D) * es;
}

// Non-negative strides in multiples of 16 bytes (TMA and vector stores need
// that); for an output also no two (batch, seq, head) rows may share bytes.
attn_status_t check_strides3(const attn_strides3& x, int64_t B, int64_t S, int64_t H, int64_t D, size_t es,
                             bool output, const char* name) {
  const int64_t st[3] = {x.batch, x.seq, x.head}, ex[3] = {B, S, H};
  for (int i = 0; i < 3; ++i) {
    if (st[i] < 0) return api_fail(ATTN_ERR_INVALID_ARG, "%s: negative stride", name);
    if (ex[i] > 1 && (size_t(st[i]) * es) % 16 != 0)
      return api_fail(ATTN_ERR_UNSUPPORTED, "%s: strides must be multiples of 16 bytes", name);
  }
  if (!output) return ATTN_OK;
  // sorted by stride, each dimension must step past the whole span of the smaller ones
  int o[3] = {0, 1, 2};
  for (int i = 0; i < 3; ++i)
    for (int j = i + 1; j < 3; ++j)
      if (st[o[j]] < st[o[i]]) std::swap(o[i], o[j]);
  int64_t span = D;
  for (int i = 0; i < 3; ++i) {
    if (ex[o[i]] <= 1) continue;
    if (st[o[i]] < span) return api_fail(ATTN_ERR_INVALID_ARG, "%s: strides make rows overlap", name);
    span = st[o[i]] * ex[o[i]];
  }
  return ATTN_OK;
}

// Whether two strided [B, S, H, D] tensors share a byte.  Disjoint byte
// ranges never do; two views with the same strides (e.g. q, k, v slices of
// one fused tensor) are tested exactly: they overlap when the distance of
// their bases is within D elements of some difference of row offsets
// sum_i k_i * stride_i, |k_i| < extent_i, which for strides that each step
// past the smaller dimensions' span is found by trying the two nearest k at
// every dimension from the largest stride down.  Other pairs count as
// overlapping when their byte ranges do.
bool strided_overlap(const void* a, const attn_strides3& sa, size_t xa, const void* b, const attn_strides3& sb,
                     size_t xb, int64_t B, int64_t S, int64_t H, int64_t D, size_t es) {
  if (!ranges_overlap(a, xa, b, xb)) return false;
  if (!same3(sa, sb)) return true;
  const int64_t diff = int64_t(reinterpret_cast<uintptr_t>(b)) - int64_t(reinterpret_cast<uintptr_t>(a));
  if (diff % int64_t(es) != 0) return true;
  int64_t st[3] = {sa.batch, sa.seq, sa.head}, n[3] = {B, S, H};
  for (int i = 0; i < 3; ++i)
    for (int j = i + 1; j < 3; ++j)
      if (st[j] > st[i]) std::swap(st[i], st[j]), std::swap(n[i], n[j]);
  struct F {
    const int64_t *st, *n;
    int64_t D;
    bool go(int i, int64_t rem) const {
      if (i == 3) return rem > -D && rem < D;
      if (n[i] <= 1 || st[i] == 0) return go(i + 1, rem);
      int64_t k = rem >= 0 ? rem / st[i] : -((-rem + st[i] - 1) / st[i]);
      for (int64_t kk = k; kk <= k + 1; ++kk) {
        const int64_t kc = std::max(-(n[i] - 1), std::min(n[i] - 1, kk));
        if (go(i + 1, rem - kc * st[i])) return true;
      }
      return false;
    }
  } f{st, n, D};
  return f.go(0, diff / int64_t(es));
}

// Kernel parameters, the hi/lo copy buffers of fp32 storage and the TMA
// descriptors shared by the backward and the forward export.  dy may be NULL
// (forward): its maps and copies then alias those of q.  split_hi / split_lo
// receive the copy buffers of q, dy, k, v (fp32 storage; else the inputs).
attn_status_t prepare_dense(const attn_dense_desc* d, const attn_dense_strides& st, const DenseSizes& z,
                            const void* q, const void* k, const void* v, const void* dy, const float* key_mask,
                            const void* bias, const void* o, const float* lse, void* dq, void* dk, void* dv,
                            void* workspace, attn::DenseParams* pp, attn::DenseMaps* mp, void* split_hi[4],
                            void* split_lo[4]) {
  const int64_t B = d->batch, H = d->heads, Sq = d->seq_q, Sk = d->seq_k, D = d->head_dim;
  const bool has_km = (d->mask_flags & ATTN_MASK_KEY) != 0;
  const bool has_bias = (d->mask_flags & ATTN_MASK_BIAS) != 0;
  const bool split = d->dtype == ATTN_DTYPE_F32;
  attn::DenseParams& p = *pp;
  p = attn::DenseParams{};
  p.B = int(B); p.H = int(H); p.Sq = int(Sq); p.Sk = int(Sk); p.D = int(D);
  p.q_off = (Sk > Sq && !(d->mask_flags & ATTN_MASK_TOP_LEFT)) ? int(Sk - Sq) : 0;
  p.causal = (d->mask_flags & (ATTN_MASK_CAUSAL | ATTN_MASK_WINDOW)) ? 1 : 0;
  p.window = (d->mask_flags & ATTN_MASK_WINDOW) ? d->window : -1;
  p.has_key_mask = has_km ? 1 : 0;
  p.has_custom = (has_km || (d->mask_flags & ATTN_MASK_ELEM)) ? 1 : 0;
  p.scale = d->scale > 0.f ? d->scale : float(1.0 / std::sqrt(double(D)));
  p.scale_log2 = p.scale * attn::kLog2e;
  p.masked_x2 = d->mask_neg * attn::kLog2e;
  p.mask_thr = d->mask_thr;
  p.mask_neg = d->mask_neg;
  p.key_mask = key_mask;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  p.L2 = reinterpret_cast<float*>(ws);
  p.delta = reinterpret_cast<float*>(ws + align256(z.stat_bytes));
  p.pm = reinterpret_cast<float*>(ws + 2 * align256(z.stat_bytes));
  p.o = o; p.lse = lse; p.dy = dy;
  p.dq = dq; p.dk = dk; p.dv = dv;
  p.q_ss = st.q.seq; p.q_sh = st.q.head; p.q_sb = st.q.batch;
  p.k_ss = st.k.seq; p.k_sh = st.k.head; p.k_sb = st.k.batch;
  auto put = [](int64_t (&dst)[3], const attn_strides3& x) {
    dst[0] = x.seq;
    dst[1] = x.head;
    dst[2] = x.batch;
  };
  put(p.s_dy, st.dy);
  put(p.s_o, st.o);
  put(p.s_dq, st.dq);
  put(p.s_dk, st.dk);
  put(p.s_dv, st.dv);
  if (d->options & ATTN_OPT_STORE_DS) p.ds_store = ws + z.ds_off;
  if (z.ew_q) {
    p.elem_rows = reinterpret_cast<const uint32_t*>(ws + z.elem_off);
    p.elem_cols = reinterpret_cast<const uint32_t*>(ws + z.elem_off + align256(size_t(B * H * Sq) * z.ew_q * 4));
    p.ew_q = z.ew_q;
    p.ew_k = z.ew_k;
  }
  p.err = device_error_word();
  if (!p.err) return api_fail(ATTN_ERR_CUDA, "no CUDA device / symbol address unavailable");

  // fp32 storage: the tensor-core operands are hi/lo bf16 copies of q, k, v, dy
  // (same layout, bf16 elements) made by a split kernel into the workspace.
  const void *qa = q, *ka = k, *va = v, *dya = dy ? dy : q;
  const void *ql = q, *kl = k, *vl = v, *dyl = dy ? dy : q;
  if (split) {
    uint8_t* c = ws + z.split_off;
    const size_t qc = align256(z.q_bytes / 2), kc = align256(z.k_bytes / 2);
    void* parts[8] = {c, c + qc, c + 2 * qc, c + 3 * qc, c + 4 * qc, c + 4 * qc + kc, c + 4 * qc + 2 * kc,
                      c + 4 * qc + 3 * kc};
    qa = parts[0]; ql = parts[1]; dya = parts[2]; dyl = parts[3];
    ka = parts[4]; kl = parts[5]; va = parts[6]; vl = parts[7];
    if (!dy) dya = qa, dyl = ql;
  }
  split_hi[0] = const_cast<void*>(qa); split_lo[0] = const_cast<void*>(ql);
  split_hi[1] = const_cast<void*>(dya); split_lo[1] = const_cast<void*>(dyl);
  split_hi[2] = const_cast<void*>(ka); split_lo[2] = const_cast<void*>(kl);
  split_hi[3] = const_cast<void*>(va); split_lo[3] = const_cast<void*>(vl);
  // TMA descriptors: (d, s, h, b) with byte strides of s, h, b
  const CUtensorMapDataType dt = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const uint64_t es = 2;  // the tensor-core operands are always bf16
  const uint64_t qdims[4] = {uint64_t(D), uint64_t(Sq), uint64_t(H), uint64_t(B)};
  const uint64_t kdims[4] = {uint64_t(D), uint64_t(Sk), uint64_t(H), uint64_t(B)};
  // (the hi/lo copies of fp32 storage keep the inputs' strides: those are
  // the layout's own there)
  const uint64_t qstr[3] = {uint64_t(st.q.seq) * es, uint64_t(st.q.head) * es, uint64_t(st.q.batch) * es};
  const uint64_t kstr[3] = {uint64_t(st.k.seq) * es, uint64_t(st.k.head) * es, uint64_t(st.k.batch) * es};
  const uint64_t vstr[3] = {uint64_t(st.v.seq) * es, uint64_t(st.v.head) * es, uint64_t(st.v.batch) * es};
  const attn_strides3& dys = dy ? st.dy : st.q;
  const uint64_t dystr[3] = {uint64_t(dys.seq) * es, uint64_t(dys.head) * es, uint64_t(dys.batch) * es};
  attn::DenseMaps& m = *mp;
  std::memset(&m, 0, sizeof(m));
  m.split = split;
  bool enc = encode4d(&m.q64, dt, qa, qdims, qstr, 64, 64) && encode4d(&m.q128, dt, qa, qdims, qstr, 64, 128) &&
             encode4d(&m.dy64, dt, dya, qdims, dystr, 64, 64) && encode4d(&m.dy128, dt, dya, qdims, dystr, 64, 128) &&
             encode4d(&m.k64, dt, ka, kdims, kstr, 64, 64) && encode4d(&m.k128, dt, ka, kdims, kstr, 64, 128) &&
             encode4d(&m.v64, dt, va, kdims, vstr, 64, 64) && encode4d(&m.v128, dt, va, kdims, vstr, 64, 128);
  if (enc && split) {
    enc = encode4d(&m.q64_lo, dt, ql, qdims, qstr, 64, 64) && encode4d(&m.q128_lo, dt, ql, qdims, qstr, 64, 128) &&
          encode4d(&m.dy64_lo, dt, dyl, qdims, dystr, 64, 64) &&
          encode4d(&m.dy128_lo, dt, dyl, qdims, dystr, 64, 128) && encode4d(&m.k64_lo, dt, kl, kdims, kstr, 64, 64) &&
          encode4d(&m.k128_lo, dt, kl, kdims, kstr, 64, 128) && encode4d(&m.v64_lo, dt, vl, kdims, vstr, 64, 64) &&
          encode4d(&m.v128_lo, dt, vl, kdims, vstr, 64, 128);
  } else if (enc) {
    m.q64_lo = m.q64; m.q128_lo = m.q128; m.dy64_lo = m.dy64; m.dy128_lo = m.dy128;
    m.k64_lo = m.k64; m.k128_lo = m.k128; m.v64_lo = m.v64; m.v128_lo = m.v128;
  }
  if (enc && has_bias) {
    const uint64_t bdims[4] = {uint64_t(Sk), uint64_t(Sq), uint64_t(H), uint64_t(B)};
    const uint64_t bstr[3] = {uint64_t(Sk) * es, uint64_t(Sq * Sk) * es, uint64_t(H * Sq * Sk) * es};
    enc = encode4d(&m.bias64, dt, bias, bdims, bstr, 64, 64) && encode4d(&m.bias128, dt, bias, bdims, bstr, 64, 128);
  } else if (enc) {
    m.bias64 = m.q64;  // unused by the kernels without bias
    m.bias128 = m.q128;
  }
  if (!enc) return api_fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled failed (driver entry point or arguments)");
  return ATTN_OK;
}

}  // namespace

extern "C" {

ATTN_API void attn_dense_desc_init(attn_dense_desc* d) {
  if (!d) return;
  std::memset(d, 0, sizeof(*d));
  d->dtype = ATTN_DTYPE_BF16;
  d->layout = ATTN_LAYOUT_BSHD;
  d->mask_thr = 0.5f;
  d->mask_neg = -1e9f;
}

ATTN_API size_t attn_bwd_dense_workspace_bytes(const attn_dense_desc* d) {
  DenseSizes z;
  if (check_dense_desc(d, &z) != ATTN_OK) return 0;
  return z.ws_bytes;
}

ATTN_API void attn_dense_strides_from_layout(const attn_dense_desc* d, attn_dense_strides* st) {
  if (d && st) layout_strides(d, st);
}

ATTN_API attn_status_t attn_bwd_dense(const attn_dense_desc* d, const void* q, const void* k, const void* v,
                                      const void* dy, const float* key_mask, const void* bias, const void* o,
                                      const float* lse, void* dq, void* dk, void* dv, unsigned wrt_mask,
                                      void* workspace, size_t workspace_bytes, void* stream) {
  if (!d) return api_fail(ATTN_ERR_INVALID_ARG, "descriptor is NULL");
  attn_dense_strides sts;
  layout_strides(d, &sts);
  return attn_bwd_dense_strided(d, &sts, q, k, v, dy, key_mask, nullptr, bias, o, lse, dq, dk, dv, wrt_mask,
                                workspace, workspace_bytes, stream);
}

ATTN_API attn_status_t attn_bwd_dense_strided(const attn_dense_desc* d, const attn_dense_strides* sts, const void* q,
                                              const void* k, const void* v, const void* dy, const float* key_mask,
                                              const float* elem_mask, const void* bias, const void* o,
                                              const float* lse, void* dq, void* dk, void* dv, unsigned wrt_mask,
                                              void* workspace, size_t workspace_bytes, void* stream) {
  DenseSizes z;
  attn_status_t st = check_dense_desc(d, &z);
  if (st != ATTN_OK) return st;
  attn_dense_strides lay_st;
  if (!sts) layout_strides(d, &lay_st);
  const attn_dense_strides& S3 = sts ? *sts : lay_st;
  if (wrt_mask == 0 || (wrt_mask & ~7u)) return api_fail(ATTN_ERR_INVALID_ARG, "wrt_mask must be a non-empty subset of dQ|dK|dV");
  const bool has_km = (d->mask_flags & ATTN_MASK_KEY) != 0;
  const bool has_bias = (d->mask_flags & ATTN_MASK_BIAS) != 0;
  if (has_km != (key_mask != nullptr)) return api_fail(ATTN_ERR_INVALID_ARG, "key_mask must be given iff ATTN_MASK_KEY is set");
  if (has_bias != (bias != nullptr)) return api_fail(ATTN_ERR_INVALID_ARG, "bias must be given iff ATTN_MASK_BIAS is set");
  const bool has_elem = (d->mask_flags & ATTN_MASK_ELEM) != 0;
  if (has_elem != (elem_mask != nullptr))
    return api_fail(ATTN_ERR_INVALID_ARG, "elem_mask must be given iff ATTN_MASK_ELEM is set");
  if ((o == nullptr) != (lse == nullptr)) return api_fail(ATTN_ERR_INVALID_ARG, "o and lse must be given together");
  const bool want_dq = wrt_mask & ATTN_WRT_DQ, want_dk = wrt_mask & ATTN_WRT_DK, want_dv = wrt_mask & ATTN_WRT_DV;
  if ((want_dq && !dq && z.q_bytes) || (want_dk && !dk && z.k_bytes) || (want_dv && !dv && z.k_bytes))
    return api_fail(ATTN_ERR_INVALID_ARG, "requested gradient pointer is NULL");
  const int64_t B = d->batch, H = d->heads, Sq = d->seq_q, Sk = d->seq_k, D = d->head_dim;
  const bool empty_q = B * H * Sq == 0, empty_k = B * H * Sk == 0;
  {
    const struct { const attn_strides3* x; int64_t S; bool out; const char* n; } chk[] = {
        {&S3.q, Sq, false, "q"}, {&S3.k, Sk, false, "k"}, {&S3.v, Sk, false, "v"}, {&S3.dy, Sq, false, "dy"},
        {&S3.o, Sq, false, "o"}, {&S3.dq, Sq, true, "dq"}, {&S3.dk, Sk, true, "dk"}, {&S3.dv, Sk, true, "dv"}};
    for (const auto& c : chk)
      if ((st = check_strides3(*c.x, B, c.S, H, D, z.es, c.out, c.n)) != ATTN_OK) return st;
    attn_dense_strides lay;
    layout_strides(d, &lay);
    if (d->dtype == ATTN_DTYPE_F32 &&
        !(same3(S3.q, lay.q) && same3(S3.k, lay.k) && same3(S3.v, lay.v) && same3(S3.dy, lay.dy)))
      return api_fail(ATTN_ERR_UNSUPPORTED, "fp32 storage needs q, k, v, dy in the descriptor's layout");
  }
  const size_t xq = extent_bytes(S3.q, B, Sq, H, D, z.es), xk = extent_bytes(S3.k, B, Sk, H, D, z.es),
               xv = extent_bytes(S3.v, B, Sk, H, D, z.es), xdy = extent_bytes(S3.dy, B, Sq, H, D, z.es),
               xo = extent_bytes(S3.o, B, Sq, H, D, z.es), xdq = extent_bytes(S3.dq, B, Sq, H, D, z.es),
               xdk = extent_bytes(S3.dk, B, Sk, H, D, z.es), xdv = extent_bytes(S3.dv, B, Sk, H, D, z.es);
  // required inputs (only when they have elements)
  if (!empty_q && (!q || !dy)) return api_fail(ATTN_ERR_INVALID_ARG, "q/dy is NULL");
  if (!empty_k && (!k || !v)) return api_fail(ATTN_ERR_INVALID_ARG, "k/v is NULL");
  const void* ptrs[] = {q, k, v, dy, key_mask, elem_mask, bias, o, lse, dq, dk, dv, workspace};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return api_fail(ATTN_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
  if (has_bias && (Sk * z.es) % 16 != 0) return api_fail(ATTN_ERR_UNSUPPORTED, "bias needs Sk * element size to be a multiple of 16");
  // aliasing: no output may overlap an input, the workspace or another output
  struct R { const void* p; size_t n; };
  // plain inputs (contiguous) by byte range; strided tensors against each other exactly
  const R ins[] = {{key_mask, has_km ? z.mask_bytes : 0}, {bias, has_bias ? z.bias_bytes : 0},
                   {elem_mask, has_elem ? z.bias_bytes / z.es * 4 : 0}, {lse, lse ? z.stat_bytes : 0},
                   {workspace, workspace_bytes}};
  struct T { const void* p; const attn_strides3* s; size_t n; int64_t S; };
  const T tin[] = {{q, &S3.q, xq, Sq}, {k, &S3.k, xk, Sk}, {v, &S3.v, xv, Sk}, {dy, &S3.dy, xdy, Sq},
                   {o, &S3.o, o ? xo : 0, Sq}};
  const T tout[] = {{want_dq ? dq : nullptr, &S3.dq, xdq, Sq}, {want_dk ? dk : nullptr, &S3.dk, xdk, Sk},
                    {want_dv ? dv : nullptr, &S3.dv, xdv, Sk}};
  for (int i = 0; i < 3; ++i) {
    const T& w = tout[i];
    for (const R& r : ins)
      if (ranges_overlap(w.p, w.n, r.p, r.n)) return api_fail(ATTN_ERR_ALIAS, "output %d overlaps an input or the workspace", i);
    for (const T& r : tin)  // (S differs between the q- and k-shaped tensors: the byte test then decides)
      if (r.S == w.S ? strided_overlap(w.p, *w.s, w.n, r.p, *r.s, r.n, B, w.S, H, D, z.es)
                     : ranges_overlap(w.p, w.n, r.p, r.n))
        return api_fail(ATTN_ERR_ALIAS, "output %d overlaps an input", i);
    for (int j = i + 1; j < 3; ++j) {
      const T& u = tout[j];
      if (u.S == w.S ? strided_overlap(w.p, *w.s, w.n, u.p, *u.s, u.n, B, w.S, H, D, z.es)
                     : ranges_overlap(w.p, w.n, u.p, u.n))
        return api_fail(ATTN_ERR_ALIAS, "outputs %d and %d overlap", i, j);
    }
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // zero-size problems: zero the selected gradients that have elements
  if (empty_q || empty_k) {
    cudaError_t e = cudaSuccess;
    if (want_dq && e == cudaSuccess) e = attn::launch_zero_rows(dq, S3.dq.batch, S3.dq.seq, S3.dq.head, B, Sq, H, D, z.es, s);
    if (want_dk && e == cudaSuccess) e = attn::launch_zero_rows(dk, S3.dk.batch, S3.dk.seq, S3.dk.head, B, Sk, H, D, z.es, s);
    if (want_dv && e == cudaSuccess) e = attn::launch_zero_rows(dv, S3.dv.batch, S3.dv.seq, S3.dv.head, B, Sk, H, D, z.es, s);
    if (e != cudaSuccess) return api_fail(ATTN_ERR_CUDA, "zero fill failed: %s", cudaGetErrorString(e));
    return api_ok();
  }
  if (!workspace || workspace_bytes < z.ws_bytes)
    return api_fail(ATTN_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", z.ws_bytes, workspace_bytes);
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return api_fail(ATTN_ERR_WORKSPACE, "workspace must be 256-byte aligned");
  const bool split = d->dtype == ATTN_DTYPE_F32;

  attn::DenseParams p;
  attn::DenseMaps m;
  void* his[4];
  void* los[4];
  if ((st = prepare_dense(d, S3, z, q, k, v, dy, key_mask, bias, o, lse, dq, dk, dv, workspace, &p, &m, his, los)) !=
      ATTN_OK)
    return st;
  p.wrt = wrt_mask;
  const bool store_ds = p.ds_store && want_dq;  // dQ from the dS tiles the dK/dV kernel stores
  if (!want_dq) p.ds_store = nullptr;
  const bool run_dkdv = want_dk || want_dv || store_ds;

  const int nk = (split ? 1 : 0) + (has_elem ? 1 : 0) + 1 + (run_dkdv ? 1 : 0) + (want_dq ? 1 : 0);
  attn::timing_mark_begin(nk, s);
  cudaError_t e = cudaSuccess;
  if (has_elem) {
    e = attn::launch_pack_elem_mask(elem_mask, d->mask_thr, B * H, int(Sq), int(Sk), const_cast<uint32_t*>(p.elem_rows),
                                    const_cast<uint32_t*>(p.elem_cols), z.ew_q, z.ew_k, s);
    attn::timing_mark(s);
  }
  if (split) {
    const int64_t nq = int64_t(z.q_bytes / 4), nkv = int64_t(z.k_bytes / 4);
    const float* srcs[4] = {static_cast<const float*>(q), static_cast<const float*>(dy), static_cast<const float*>(k),
                            static_cast<const float*>(v)};
    const int64_t ns[4] = {nq, nq, nkv, nkv};
    e = attn::launch_split_f32(srcs, his, los, ns, s);
    attn::timing_mark(s);
  }
  if (e == cudaSuccess) {
    e = o ? attn::launch_delta_only(p, split ? 0 : 1, s)
          : (split ? attn::launch_fwd_stats(m, p, has_bias, s) : attn::launch_stats2(m, p, has_bias, s));
    attn::timing_mark(s);
  }
  if (e == cudaSuccess && run_dkdv) {
    e = split ? attn::launch_dkdv(m, p, has_bias, s) : attn::launch_dkdv2(m, p, has_bias, s);
    attn::timing_mark(s);
  }
  if (e == cudaSuccess && want_dq) {
    e = split      ? attn::launch_dq(m, p, has_bias, s)
        : store_ds ? attn::launch_dq3(m, p, s)
                   : attn::launch_dq2(m, p, has_bias, s);
    attn::timing_mark(s);
  }
  attn::timing_mark_end();
  if (e != cudaSuccess) return api_fail(ATTN_ERR_CUDA, "kernel launch failed: %s", cudaGetErrorString(e));
  return api_ok();
}

ATTN_API attn_status_t attn_fwd_dense(const attn_dense_desc* d, const void* q, const void* k, const void* v,
                                      const float* key_mask, const void* bias, void* o, float* lse, void* workspace,
                                      size_t workspace_bytes, void* stream) {
  if (!d) return api_fail(ATTN_ERR_INVALID_ARG, "descriptor is NULL");
  attn_dense_strides sts;
  layout_strides(d, &sts);
  return attn_fwd_dense_strided(d, &sts, q, k, v, key_mask, bias, o, lse, workspace, workspace_bytes, stream);
}

ATTN_API attn_status_t attn_fwd_dense_strided(const attn_dense_desc* d, const attn_dense_strides* sts, const void* q,
                                              const void* k, const void* v, const float* key_mask, const void* bias,
                                              void* o, float* lse, void* workspace, size_t workspace_bytes,
                                              void* stream) {
  DenseSizes z;
  attn_status_t st = check_dense_desc(d, &z);
  if (st != ATTN_OK) return st;
  if (d->mask_flags & ATTN_MASK_ELEM)
    return api_fail(ATTN_ERR_UNSUPPORTED, "the forward export does not take a per-element mask");
  attn_dense_strides lay_st;
  if (!sts) layout_strides(d, &lay_st);
  const attn_dense_strides& S3 = sts ? *sts : lay_st;
  const bool has_km = (d->mask_flags & ATTN_MASK_KEY) != 0;
  const bool has_bias = (d->mask_flags & ATTN_MASK_BIAS) != 0;
  if (has_km != (key_mask != nullptr)) return api_fail(ATTN_ERR_INVALID_ARG, "key_mask must be given iff ATTN_MASK_KEY is set");
  if (has_bias != (bias != nullptr)) return api_fail(ATTN_ERR_INVALID_ARG, "bias must be given iff ATTN_MASK_BIAS is set");
  const int64_t B = d->batch, H = d->heads, Sq = d->seq_q, Sk = d->seq_k, D = d->head_dim;
  const bool empty_q = B * H * Sq == 0, empty_k = B * H * Sk == 0;
  {
    const struct { const attn_strides3* x; int64_t S; bool out; const char* n; } chk[] = {
        {&S3.q, Sq, false, "q"}, {&S3.k, Sk, false, "k"}, {&S3.v, Sk, false, "v"}, {&S3.o, Sq, true, "o"}};
    for (const auto& c : chk)
      if ((st = check_strides3(*c.x, B, c.S, H, D, z.es, c.out, c.n)) != ATTN_OK) return st;
    attn_dense_strides lay;
    layout_strides(d, &lay);
    if (d->dtype == ATTN_DTYPE_F32 && !(same3(S3.q, lay.q) && same3(S3.k, lay.k) && same3(S3.v, lay.v)))
      return api_fail(ATTN_ERR_UNSUPPORTED, "fp32 storage needs q, k, v in the descriptor's layout");
  }
  const size_t xq = extent_bytes(S3.q, B, Sq, H, D, z.es), xk = extent_bytes(S3.k, B, Sk, H, D, z.es),
               xv = extent_bytes(S3.v, B, Sk, H, D, z.es), xo = extent_bytes(S3.o, B, Sq, H, D, z.es);
  if (!empty_q && (!q || !o || !lse)) return api_fail(ATTN_ERR_INVALID_ARG, "q/o/lse is NULL");
  if (!empty_k && (!k || !v)) return api_fail(ATTN_ERR_INVALID_ARG, "k/v is NULL");
  const void* ptrs[] = {q, k, v, key_mask, bias, o, lse, workspace};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return api_fail(ATTN_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
  if (has_bias && (Sk * z.es) % 16 != 0) return api_fail(ATTN_ERR_UNSUPPORTED, "bias needs Sk * element size to be a multiple of 16");
  struct R { const void* p; size_t n; };
  const R ins[] = {{q, xq}, {k, xk}, {v, xv}, {key_mask, has_km ? z.mask_bytes : 0},
                   {bias, has_bias ? z.bias_bytes : 0}, {workspace, workspace_bytes}};
  const R outs[] = {{o, xo}, {lse, z.stat_bytes}};
  for (const R& w : outs)
    for (const R& r : ins)
      if (ranges_overlap(w.p, w.n, r.p, r.n)) return api_fail(ATTN_ERR_ALIAS, "an output overlaps an input or the workspace");
  if (ranges_overlap(o, xo, lse, z.stat_bytes)) return api_fail(ATTN_ERR_ALIAS, "o and lse overlap");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (empty_q) return api_ok();
  if (empty_k) {  // no key: O = 0, lse = -inf
    cudaError_t e = attn::launch_zero_rows(o, S3.o.batch, S3.o.seq, S3.o.head, B, Sq, H, D, z.es, s);
    if (e == cudaSuccess)
      e = attn::launch_fill_f32(lse, -std::numeric_limits<float>::infinity(), int64_t(z.stat_bytes / 4), s);
    if (e != cudaSuccess) return api_fail(ATTN_ERR_CUDA, "fill failed: %s", cudaGetErrorString(e));
    return api_ok();
  }
  if (!workspace || workspace_bytes < z.ws_bytes)
    return api_fail(ATTN_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", z.ws_bytes, workspace_bytes);
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return api_fail(ATTN_ERR_WORKSPACE, "workspace must be 256-byte aligned");
  const bool split = d->dtype == ATTN_DTYPE_F32;
  attn::DenseParams p;
  attn::DenseMaps m;
  void* his[4];
  void* los[4];
  if ((st = prepare_dense(d, S3, z, q, k, v, nullptr, key_mask, bias, nullptr, nullptr, nullptr, nullptr, nullptr,
                          workspace, &p, &m, his, los)) != ATTN_OK)
    return st;
  p.fwd_only = 1;
  p.o_out = o;
  p.lse_out = lse;
  attn::timing_mark_begin(split ? 2 : 1, s);
  cudaError_t e = cudaSuccess;
  if (split) {
    const int64_t nq = int64_t(z.q_bytes / 4), nkv = int64_t(z.k_bytes / 4);
    const float* srcs[4] = {static_cast<const float*>(q), nullptr, static_cast<const float*>(k),
                            static_cast<const float*>(v)};
    const int64_t ns[4] = {nq, 0, nkv, nkv};  // no dY in a forward pass
    e = attn::launch_split_f32(srcs, his, los, ns, s);
    attn::timing_mark(s);
  }
  if (e == cudaSuccess) {
    e = attn::launch_fwd_stats(m, p, has_bias, s);
    attn::timing_mark(s);
  }
  attn::timing_mark_end();
  if (e != cudaSuccess) return api_fail(ATTN_ERR_CUDA, "kernel launch failed: %s", cudaGetErrorString(e));
  return api_ok();
}

ATTN_API const char* attn_last_error(void) { return g_msg; }

ATTN_API const char* attn_status_string(attn_status_t s) {
  switch (s) {
    case ATTN_OK: return "ATTN_OK";
    case ATTN_ERR_INVALID_ARG: return "ATTN_ERR_INVALID_ARG";
    case ATTN_ERR_UNSUPPORTED: return "ATTN_ERR_UNSUPPORTED";
    case ATTN_ERR_ALIAS: return "ATTN_ERR_ALIAS";
    case ATTN_ERR_WORKSPACE: return "ATTN_ERR_WORKSPACE";
    case ATTN_ERR_CUDA: return "ATTN_ERR_CUDA";
    case ATTN_ERR_TIMEOUT: return "ATTN_ERR_TIMEOUT";
    default: return "ATTN_ERR_UNKNOWN";
  }
}

ATTN_API attn_status_t attn_check_device_error(void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return api_fail(ATTN_ERR_CUDA, "stream failed: %s", cudaGetErrorString(e));
  uint32_t* w = device_error_word();
  if (!w) return api_fail(ATTN_ERR_CUDA, "no CUDA device");
  uint32_t h = 0;
  if (cudaMemcpy(&h, w, 4, cudaMemcpyDeviceToHost) != cudaSuccess || cudaMemset(w, 0, 4) != cudaSuccess)
    return api_fail(ATTN_ERR_CUDA, "reading the device error word failed");
  if (h & 1u) return api_fail(ATTN_ERR_TIMEOUT, "a device-side wait timed out (error word 0x%x)", h);
  if (h) return api_fail(ATTN_ERR_CUDA, "device error word 0x%x", h);
  return api_ok();
}

ATTN_API void attn_set_timing_events(void* const* events, int count) {
  g_events = events;
  g_event_count = events ? count : 0;
  g_event_next = 0;
}

ATTN_API int attn_version(void) { return 100; }

}  // extern "C"
