// Shared definitions of the dense backward kernels: launch parameters, the
// structural-mask tile arithmetic and the row-statistics layout.
#pragma once

#include <cstdint>
#include <cuda.h>

namespace attn {

// log2(e): scores are carried in base-2 units so that exp() is one ex2.
constexpr float kLog2e = 1.4426950408889634f;

struct DenseParams {
  int B, H, Sq, Sk, D;   // problem sizes (D = real head dim)
  int q_off;             // max(Sk - Sq, 0): bottom-right alignment of the masks
  int causal;            // 1 when keys k > abs_q are hidden (causal or window)
  int window;            // window w, or -1 when there is no lower bound
  int has_key_mask;      // custom per-key mask present
  int has_custom;        // a custom mask (per-key or per-element) present: pm is live
  float scale;           // softmax scale
  float scale_log2;      // scale * log2(e)
  float masked_x2;       // mask_neg * log2(e): a custom-masked score in base-2 units
  float mask_thr;        // key masked when key_mask[b, k] < mask_thr
  float mask_neg;        // masked score (natural units)
  const float* key_mask; // [B, Sk] or null
  // Row statistics (workspace), [B, H, Sq] each:
  float* L2;             // lse * log2(e); +inf for rows with no visible key
  float* delta;          // rowsum(P * dP) = dY . O
  float* pm;             // probability of a custom-masked visible key in the row
  // Optional forward outputs (delta-only prologue).
  const void* o;
  const float* lse;
  const void* dy;        // dY (plain loads in the delta-only prologue)
  // Outputs and their element strides (sequence, head, batch).
  void* dq;
  void* dk;
  void* dv;
  int64_t q_ss, q_sh, q_sb;   // element strides (sequence, head, batch) of q
  int64_t k_ss, k_sh, k_sb;   // ... of k
  // ... of the other tensors the kernels address directly, {s, h, b} each
  int64_t s_dy[3], s_o[3], s_dq[3], s_dk[3], s_dv[3];
  unsigned wrt;               // ATTN_WRT_* bits
  // Forward export (the row-statistics sweep run as a forward pass): when
  // fwd_only is set there is no dY and no delta; o_out (q's layout and dtype)
  // and lse_out ([B, H, Sq], natural log) receive O and the LSE.
  int fwd_only;
  void* o_out;
  float* lse_out;
  // Per-element custom mask as bits (workspace): elem_rows[(bh*Sq + q)*ew_q + k/32]
  // bit k%32 and elem_cols[(bh*Sk + k)*ew_k + q/32] bit q%32 are set for a
  // masked pair; null without the mask.  ew_q, ew_k are even.
  const uint32_t* elem_rows;
  const uint32_t* elem_cols;
  int ew_q, ew_k;
  // Stored dS (ATTN_OPT_STORE_DS, workspace): the dK/dV kernel writes tile
  // (bh, key tile kt of 128, query tile qt of 64) of dS^T, unscaled bf16, at
  // ds_store + ((bh * ceil(Sk/128) + kt) * ceil(Sq/64) + qt) * 16384: chunk c
  // (queries 8c..8c+7, 16 bytes) of key k at byte c * 2048 + k * 16, so that
  // one warp store instruction writes 512 contiguous bytes.  Read as is, this
  // is the unswizzled MN-major operand layout (8-key x 16-byte core matrices,
  // 128 bytes apart along the keys, 2048 along the queries) the dQ kernel
  // gives the tensor core.  Null: dQ by recomputation.
  uint8_t* ds_store;
  uint32_t* err;              // device error word
};

__host__ __device__ inline int cdiv(int a, int b) { return (a + b - 1) / b; }
__host__ __device__ inline int imax(int a, int b) { return a > b ? a : b; }
__host__ __device__ inline int imin(int a, int b) { return a < b ? a : b; }
// floor(a / b) for b > 0 and any sign of a
__host__ __device__ inline int floordiv(int a, int b) { return a >= 0 ? a / b : -((-a + b - 1) / b); }

// Range [lo, hi) of query tiles (rows tq*i .. tq*i+tq-1) that can see at least
// one key of [k0, k1] (inclusive, k1 < Sk).  Query q sees key k when
// k <= q + q_off (causal) and k >= q + q_off - w (window).
__host__ __device__ inline void query_tile_range(const DenseParams& p, int k0, int k1, int tq, int* lo, int* hi) {
  const int nq = cdiv(p.Sq, tq);
  int l = 0, h = nq;
  if (p.causal) l = imax(0, floordiv(k0 - p.q_off, tq));
  if (p.window >= 0) {
    const int qmax = k1 + p.window - p.q_off;  // largest query that sees key k1
    h = qmax < 0 ? 0 : imin(nq, qmax / tq + 1);
  }
  *lo = l;
  *hi = imax(l, h);
}

// Range [lo, hi) of key tiles (keys tk*j .. tk*j+tk-1) visible to at least one
// query of [q0, q1] (inclusive, q1 < Sq).
__host__ __device__ inline void key_tile_range(const DenseParams& p, int q0, int q1, int tk, int* lo, int* hi) {
  const int nk = cdiv(p.Sk, tk);
  int l = 0, h = nk;
  if (p.causal) {
    const int kmax = q1 + p.q_off;  // largest key that query q1 sees
    h = imin(nk, kmax / tk + 1);
  }
  if (p.window >= 0) {
    const int kmin = q0 + p.q_off - p.window;  // smallest key that query q0 sees
    l = kmin <= 0 ? 0 : kmin / tk;
  }
  *lo = l;
  *hi = imax(l, h);
}

// True when every (query, key) pair of the tile is structurally visible and
// in range, so the per-element mask test can be skipped.
__host__ __device__ inline bool tile_fully_visible(const DenseParams& p, int q0, int q1, int k0, int k1) {
  if (q1 >= p.Sq || k1 >= p.Sk) return false;
  if (p.causal && k1 > q0 + p.q_off) return false;
  if (p.window >= 0 && k0 < q1 + p.q_off - p.window) return false;
  return true;
}

__device__ __forceinline__ bool pair_visible(const DenseParams& p, int q, int k) {
  if (k >= p.Sk || q >= p.Sq) return false;
  const int aq = q + p.q_off;
  if (p.causal && k > aq) return false;
  if (p.window >= 0 && k < aq - p.window) return false;
  return true;
}

// Number of structurally visible keys of query row q.
__host__ __device__ inline int visible_keys(const DenseParams& p, int q) {
  const int aq = q + p.q_off;
  int hi = p.Sk - 1, lo = 0;
  if (p.causal) hi = imin(hi, aq);
  if (p.window >= 0) lo = imax(0, aq - p.window);
  return imax(0, hi - lo + 1);
}

}  // namespace attn

#ifdef __CUDACC__
#include <cuda_bf16.h>

#include "sm103.cuh"

namespace attn {

// Write 32 values (columns c0..c0+31 of `row`) into a 128-byte-swizzled
// K-major bf16 tile at shared address `tile`.  With SPLIT the value is stored
// as two bf16 copies, hi = bf16(x) at `tile` and lo = bf16(x - hi) at
// `tile + copy_bytes`, so that hi + lo carries about 16 significant bits.
template <bool SPLIT>
__device__ __forceinline__ void store_row32(uint32_t tile, uint32_t copy_bytes, int row, int c0, const float* x) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    uint32_t hi[4], lo[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float a = x[8 * j + 2 * e], b = x[8 * j + 2 * e + 1];
      const __nv_bfloat162 h2 = __floats2bfloat162_rn(a, b);
      hi[e] = *reinterpret_cast<const uint32_t*>(&h2);
      if (SPLIT) {
        const __nv_bfloat162 l2 = __floats2bfloat162_rn(a - __low2float(h2), b - __high2float(h2));
        lo[e] = *reinterpret_cast<const uint32_t*>(&l2);
      }
    }
    const uint32_t off = sm103::sw128_offset(row, (c0 >> 3) + j);
    sm103::st_shared_v4(tile + off, hi[0], hi[1], hi[2], hi[3]);
    if (SPLIT) sm103::st_shared_v4(tile + copy_bytes + off, lo[0], lo[1], lo[2], lo[3]);
  }
}

// Store 32 fp32 accumulator values (times f) of one output row, columns
// col0..col0+31 limited to D: bf16 (round to nearest even) or, with SPLIT
// (fp32 storage), fp32.  `row_off` is the row's element offset.  A whole
// chunk at a 32-byte aligned address goes out as 32-byte stores.
template <bool SPLIT>
__device__ __forceinline__ void store_out32(void* out, int64_t row_off, int col0, int D, const uint32_t (&r)[32],
                                            float f) {
  if (SPLIT) {
    float* o = reinterpret_cast<float*>(out) + row_off + col0;
    if (col0 + 32 <= D && (reinterpret_cast<uintptr_t>(o) & 31u) == 0) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        uint32_t v[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) v[e] = __float_as_uint(__uint_as_float(r[8 * j + e]) * f);
        sm103::st_global_v8(o + 8 * j, v);
      }
      return;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (col0 + 4 * j < D)
        *reinterpret_cast<float4*>(o + 4 * j) =
            make_float4(__uint_as_float(r[4 * j]) * f, __uint_as_float(r[4 * j + 1]) * f,
                        __uint_as_float(r[4 * j + 2]) * f, __uint_as_float(r[4 * j + 3]) * f);
  } else {
    sm103::store_row32_bf16(reinterpret_cast<__nv_bfloat16*>(out) + row_off + col0, r, f, D - col0);
  }
}

}  // namespace attn
#endif
