// Row-statistics prologue of the dense backward, bf16 storage, self-contained
// mode (no O or LSE from the caller).
//
// One CTA per (batch*head, 128-query tile) sweeps the visible 64-key tiles.
// The tensor core computes, per key tile j,
//   S  = Q_i K_j^T      (A = Q_i held in tensor memory, B = K_j from a TMA ring)
//   dP = dY_i V_j^T     (A = dY_i held in tensor memory, B = V_j)
// and every query row accumulates, with an online maximum m (base-2 units),
//   l    = sum_j 2^(x_j - m)
//   dsum = sum_j 2^(x_j - m) * dP_j
// where x_j = S_j*scale*log2(e) + bias_j*log2(e) for a visible key, the
// custom-mask value mask_neg*log2(e) for a custom-masked visible key, and no
// term for a key the structural mask hides.  Then
//   L2    = m + log2(l)                  (the log-sum-exp in base-2 units)
//   delta = dsum / l = sum_j P_j dP_j    (= dY_i . O_i, the dS row offset)
//   pm    = probability of one custom-masked visible key of the row
// The softmax and the dS offset follow rlx-cpu src/attention_bwd.rs
// (fn backward_dense_head_all: max-subtracted exponentials, dS = P (dP -
// rowsum(P dP))); the masks follow fn apply_synthetic_mask there.  Both sums
// are rescaled by 2^(m_old - m_new) when the maximum grows, which for two
// scalars costs nothing: no output tile is accumulated or rescaled.
//
// Tiles are 128 queries x 128 keys (N = 128 MMAs).  Roles: warp 0 TMA
// producer, warp 1 MMA issuer (whole warp, elect.sync), warps 2..17 four
// column groups of four warps, group g owning key columns [32g, 32g+32) of
// every tile; the groups keep their own (m, l, dsum) per row and merge at the
// end.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "dense_common.cuh"
#include "dense_launch.h"
#include "sm103.cuh"

namespace attn {
using namespace sm103;

namespace {

constexpr int kStages = 2;

template <int DP>
struct Stats2Layout {
  static constexpr int NCH = DP / 64;
  static constexpr int BQ = 128, BK = 128;
  static constexpr int QT = NCH * BQ * 128;  // Q or dY tile (128 rows)
  static constexpr int KT = NCH * BK * 128;  // K or V tile (128 rows)
  static constexpr int BIAS = 2 * BQ * 128;  // two 64-key halves x 128 query rows
  static constexpr int K_OFF = 0;                        // kStages
  static constexpr int V_OFF = K_OFF + kStages * KT;     // kStages
  static constexpr int BIAS_OFF = V_OFF + kStages * KT;  // kStages
  // Q and dY are needed in shared memory only until they are staged into
  // tensor memory: they occupy the K and V slots of stage 1, which the
  // producer fills only after that staging
  static constexpr int Q_OFF = K_OFF + KT;
  static constexpr int DY_OFF = V_OFF + KT;
  static_assert(QT == KT, "Q / dY alias one ring slot");
  // per key column of a tile: sk = scale*log2(e), kb = log2(e), off = 0 for a
  // key the custom mask keeps; sk = kb = 0, off = mask_neg*log2(e) for a
  // custom-masked key (so x = S*sk + bias*kb + off); then the 128-bit set of
  // custom-masked columns
  static constexpr int COL = 3 * BK * 4 + 16;
  static constexpr int COL_OFF = BIAS_OFF + kStages * BIAS;  // kStages
  static constexpr int BYTES = COL_OFF + kStages * COL;
  // TMEM: S[2] [0, 256), dP [256, 384), Q and dY rows as bf16 pairs after
  static constexpr int T_S = 0, T_DP = 256, T_QA = 384, T_DYA = 384 + DP / 2;
  static constexpr int TMEM_COLS = 512;
  static_assert(T_DYA + DP / 2 <= TMEM_COLS, "tensor memory budget");
};

// Lazy rescaling threshold (base-2 units): the running maximum is raised only
// when a score exceeds it by more than this, so every term stays <= 2^8.
constexpr float kRescaleThreshold = 8.0f;

__device__ __forceinline__ bool drain_wait(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_test(bar, parity)) {
    if (global_timer_ns() - t0 > ATTN_WAIT_TIMEOUT_NS) return false;
  }
  return true;
}

// Column groups (warps 2..17, four warps each) and the barrier among them
// (named barrier 1, 512 threads).
constexpr int kGroups = 4;
__device__ __forceinline__ void group_sync() { asm volatile("bar.sync 1, 512;" ::: "memory"); }

template <int DP, bool HAS_BIAS>
__global__ void __launch_bounds__(576, 1)
    stats2_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_dy,
                  const __grid_constant__ CUtensorMap tm_bias, const DenseParams p) {
  using L = Stats2Layout<DP>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t bar_qdy, bar_a_ready, bar_full[kStages], bar_empty[kStages], bar_dp_full, bar_used[2];
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag;
  __shared__ float mg_m[kGroups - 1][128], mg_l[kGroups - 1][128], mg_d[kGroups - 1][128];
  __shared__ int mg_any[kGroups - 1][128];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bh = blockIdx.x;
  const int b = bh / p.H, h = bh - b * p.H;
  const int nqt = cdiv(p.Sq, L::BQ);
  const int it = nqt - 1 - static_cast<int>(blockIdx.y);  // longest rows first under causal masks
  const int q0 = it * L::BQ;
  const int q1 = imin(q0 + L::BQ - 1, p.Sq - 1);
  int j_lo, j_hi;
  key_tile_range(p, q0, q1, L::BK, &j_lo, &j_hi);
  const int n = j_hi - j_lo;
  const Abort ab{&abort_flag, p.err};

  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bar_qdy, 1);
    mbar_init(&bar_a_ready, 8);  // warps 2..9: Q and dY rows staged in tensor memory
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bar_full[s], 2);                 // TMA bytes + key-column constants written
      mbar_init(&bar_empty[s], 1 + 4 * kGroups);  // MMAs of the tile done + stage read by warps 2..17
    }
    mbar_init(&bar_dp_full, 1);  // S(t) and dP(t) done
    for (int s = 0; s < 2; ++s) mbar_init(&bar_used[s], 4 * kGroups);  // S(t), dP(t) read, t = s mod 2
    mbar_fence_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base_sh, L::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;

  if (n > 0 && warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_map(&tm_q);
      tma_prefetch_map(&tm_k);
      tma_prefetch_map(&tm_v);
      tma_prefetch_map(&tm_dy);
      if (HAS_BIAS) tma_prefetch_map(&tm_bias);
      mbar_arrive_expect_tx(&bar_qdy, 2 * L::QT);
      for (int c = 0; c < L::NCH; ++c) {
        tma_load_4d(sm + L::Q_OFF + c * (L::BQ * 128), &tm_q, &bar_qdy, c * 64, q0, h, b);
        tma_load_4d(sm + L::DY_OFF + c * (L::BQ * 128), &tm_dy, &bar_qdy, c * 64, q0, h, b);
      }
    }
    // custom-mask values of keys lane + 32 i of a tile, one tile ahead
    const float* km = p.has_key_mask ? p.key_mask + static_cast<size_t>(b) * p.Sk : nullptr;
    float kmv[4] = {0.f, 0.f, 0.f, 0.f};
    auto km_load = [&](int t) {
      const int kk0 = (j_lo + t) * L::BK;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int key = kk0 + lane + 32 * i;
        kmv[i] = key < p.Sk ? km[key] : 1.f;
      }
    };
    if (p.has_key_mask) km_load(0);
    int last_use[kStages];
    for (int i = 0; i < kStages; ++i) last_use[i] = -1;
    bool ok = true;
    for (int t = 0; t < n && ok; ++t) {
      const int s = t % kStages;
      if (t >= kStages) ok = mbar_wait_warp(&bar_empty[s], ((t / kStages) - 1) & 1, ab);
      if (t == 1 && ok) ok = mbar_wait_warp(&bar_a_ready, 0, ab);  // Q, dY slots free
      if (!ok) break;
      const int kk0 = (j_lo + t) * L::BK;
      if (lane == 0) {
        mbar_arrive_expect_tx(&bar_full[s], 2 * L::KT + (HAS_BIAS ? L::BIAS : 0));
        for (int c = 0; c < L::NCH; ++c) {
          tma_load_4d(sm + L::K_OFF + s * L::KT + c * (L::BK * 128), &tm_k, &bar_full[s], c * 64, kk0, h, b);
          tma_load_4d(sm + L::V_OFF + s * L::KT + c * (L::BK * 128), &tm_v, &bar_full[s], c * 64, kk0, h, b);
        }
        if (HAS_BIAS) {
          uint8_t* bs = sm + L::BIAS_OFF + s * L::BIAS;
          tma_load_4d(bs, &tm_bias, &bar_full[s], kk0, q0, h, b);
          tma_load_4d(bs + L::BQ * 128, &tm_bias, &bar_full[s], kk0 + 64, q0, h, b);
        }
      }
      if (p.has_key_mask) {
        float* col = reinterpret_cast<float*>(sm + L::COL_OFF + s * L::COL);
        uint32_t* bits = reinterpret_cast<uint32_t*>(col + 3 * L::BK);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const bool masked = kmv[i] < p.mask_thr;
          col[lane + 32 * i] = masked ? 0.f : p.scale_log2;
          col[L::BK + lane + 32 * i] = masked ? 0.f : kLog2e;
          col[2 * L::BK + lane + 32 * i] = masked ? p.masked_x2 : 0.f;
          const uint32_t w = __ballot_sync(0xffffffffu, masked);
          if (lane == 0) bits[i] = w;
        }
        if (t + 1 < n) km_load(t + 1);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_full[s]);
      last_use[s] = t;
    }
    if (lane == 0) {
      for (int s = 0; s < kStages; ++s)
        if (last_use[s] >= 0) drain_wait(&bar_full[s], (last_use[s] / kStages) & 1);
      drain_wait(&bar_qdy, 0);
    }
    __syncwarp();
  } else if (n > 0 && warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // the whole warp runs this role (warp-uniform); elected lanes issue
    {
      constexpr uint32_t id_s = idesc_bf16(128, 128, false, false);
      // descriptors built once; k-slices and stages are constant offsets
      const uint64_t dK0 = sdesc_sw128(smem_addr(sm + L::K_OFF), 16, 1024);
      const uint64_t dV0 = sdesc_sw128(smem_addr(sm + L::V_OFF), 16, 1024);
      // D[128 x 128] = A[128 x DP] (tensor memory, bf16 pairs) * B[128 x DP]^T (shared memory, K-major)
      auto issue_xt = [&](uint32_t d, uint32_t a_tmem, uint64_t bk) {
        mma_ts_w<false>(d, a_tmem, bk, id_s);
#pragma unroll
        for (int kk = 1; kk < DP / 16; ++kk) {
          const int c = kk >> 2, o = (kk & 3) * 32;
          mma_ts_w<true>(d, a_tmem + kk * 8, sdesc_add(bk, c * (L::BK * 128) + o), id_s);
        }
      };
      bool ok = mbar_wait_warp(&bar_a_ready, 0, ab);
      tc_fence_after();
      // S(t) may go as soon as its buffer's previous tile (t - 2) was read;
      // dP(t) (single buffer) once tile t - 1 was read.  Each of the two
      // barriers is awaited at most one phase behind its current one.
      for (int t = 0; t < n && ok; ++t) {
        const int s = t % kStages, bb = t & 1;
        if (!(ok = mbar_wait_warp(&bar_full[s], (t / kStages) & 1, ab))) break;
        if (t >= 2 && !(ok = mbar_wait_warp(&bar_used[bb], ((t - 2) >> 1) & 1, ab))) break;
        tc_fence_after();
        issue_xt(tmem + L::T_S + bb * 128, tmem + L::T_QA, sdesc_add(dK0, s * L::KT));
        if (t >= 1 && !(ok = mbar_wait_warp(&bar_used[bb ^ 1], ((t - 1) >> 1) & 1, ab))) break;
        tc_fence_after();
        issue_xt(tmem + L::T_DP, tmem + L::T_DYA, sdesc_add(dV0, s * L::KT));
        mma_commit_w(&bar_dp_full);
        mma_commit_w(&bar_empty[s]);
      }
      // the last commits of each stage arrive before the CTA leaves
      for (int t = imax(0, n - kStages); t < n; ++t) drain_wait(&bar_empty[t % kStages], (t / kStages) & 1);
    }
    __syncwarp();
  } else if (warp >= 2) {
    const int g = (warp - 2) >> 2;  // column group: key columns [32g, 32g + 32) of every tile
    const int lg = warp & 3;
    const int row = lg * 32 + lane;  // query row inside the tile == TMEM lane
    const int q = q0 + row;
    const uint32_t lane_addr = static_cast<uint32_t>(lg * 32) << 16;
    const float kInf = __int_as_float(0x7f800000);
    bool ok = n > 0;
    if (n > 0 && g < 2) {
      // stage this row of Q (group 0) or dY (group 1) in tensor memory as bf16
      // pairs: the A operand of S = Q K^T and dP = dY V^T
      ok = mbar_wait_warp(&bar_qdy, 0, ab);
      if (ok) {
        const uint8_t* src = sm + (g == 0 ? L::Q_OFF : L::DY_OFF);
        const uint32_t dst = tmem + (g == 0 ? L::T_QA : L::T_DYA) + lane_addr;
#pragma unroll
        for (int c = 0; c < L::NCH; ++c) {
          uint32_t w[32];
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const uint4 v = *reinterpret_cast<const uint4*>(src + c * (L::BQ * 128) + sw128_offset(row, j));
            w[4 * j] = v.x;
            w[4 * j + 1] = v.y;
            w[4 * j + 2] = v.z;
            w[4 * j + 3] = v.w;
          }
          tmem_st32(dst + c * 32, w);
        }
        tmem_st_wait();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_a_ready);
    }
    // keys this query sees: [ka, kb] (window: key >= q + q_off - window;
    // causal: key <= q + q_off; key < Sk; none when q >= Sq)
    int ka = -(1 << 30), kb = p.Sk - 1;
    if (p.window >= 0) ka = q + p.q_off - p.window;
    if (p.causal) kb = imin(kb, q + p.q_off);
    if (q >= p.Sq) ka = 1 << 30, kb = -(1 << 30);
    float m2 = -kInf, l = 0.f, dsum = 0.f;
    bool any_unmasked = false;
    for (int t = 0; t < n && ok; ++t) {
      const int s = t % kStages, bb = t & 1;
      const int kk0 = (j_lo + t) * L::BK;
      if (!(ok = mbar_wait_warp(&bar_full[s], (t / kStages) & 1, ab))) break;
      // bias and custom-mask terms of the group's 32 columns while the tensor
      // core works: x = bias*kb + off (S*sk added once S is in)
      const float* col = reinterpret_cast<const float*>(sm + L::COL_OFF + s * L::COL) + 32 * g;
      const uint32_t kbits = p.has_key_mask ? reinterpret_cast<const uint32_t*>(col - 32 * g + 3 * L::BK)[g] : 0u;
      // bias half (64 keys) g >> 1, 16-byte chunks 4 (g & 1) .. + 3 of this row
      const uint8_t* brow = sm + L::BIAS_OFF + s * L::BIAS + (g >> 1) * (L::BQ * 128) + row * 128;
      float x[32];
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {  // 8 keys per 16-byte bias chunk
        float bv[8];
        if (HAS_BIAS) {
          const uint4 w4 = *reinterpret_cast<const uint4*>(brow + (((4 * (g & 1) + jj) ^ (row & 7)) << 4));
          const uint32_t w[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            bv[2 * e] = __uint_as_float(w[e] << 16);
            bv[2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u);
          }
        }
        if (p.has_key_mask) {
#pragma unroll
          for (int h4 = 0; h4 < 2; ++h4) {
            const int c = 8 * jj + 4 * h4;
            const float4 kb4 = *reinterpret_cast<const float4*>(col + L::BK + c);
            const float4 of4 = *reinterpret_cast<const float4*>(col + 2 * L::BK + c);
            const float kbv[4] = {kb4.x, kb4.y, kb4.z, kb4.w}, ofv[4] = {of4.x, of4.y, of4.z, of4.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) x[c + e] = HAS_BIAS ? fmaf(bv[4 * h4 + e], kbv[e], ofv[e]) : ofv[e];
          }
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) x[8 * jj + e] = HAS_BIAS ? bv[e] * kLog2e : 0.f;
        }
      }
      // the dP commit follows the S MMAs of the tile, so it covers both
      if (!(ok = mbar_wait_warp(&bar_dp_full, t & 1, ab))) break;
      tc_fence_after();
      {
        uint32_t sr[32];
        tmem_ld32(tmem + L::T_S + bb * 128 + 32 * g + lane_addr, sr);
        tmem_ld_wait();
        if (p.has_key_mask) {
#pragma unroll
          for (int c4 = 0; c4 < 8; ++c4) {
            const float4 sk4 = *reinterpret_cast<const float4*>(col + 4 * c4);
            const float skv[4] = {sk4.x, sk4.y, sk4.z, sk4.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) x[4 * c4 + e] = fmaf(__uint_as_float(sr[4 * c4 + e]), skv[e], x[4 * c4 + e]);
          }
        } else {
#pragma unroll
          for (int c = 0; c < 32; ++c) x[c] = fmaf(__uint_as_float(sr[c]), p.scale_log2, x[c]);
        }
      }
      uint32_t dr[32];
      tmem_ld32(tmem + L::T_DP + 32 * g + lane_addr, dr);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&bar_used[bb]);
        mbar_arrive(&bar_empty[s]);  // bias and column constants read
      }
      const bool full = tile_fully_visible(p, q0, q0 + L::BQ - 1, kk0, kk0 + L::BK - 1);
      // visible columns of this row among the group's 32: [lo, hi]
      uint32_t vb = 0xffffffffu;
      if (!full) {
        const int lo = ka - kk0 - 32 * g, hi = kb - kk0 - 32 * g;
        vb = 0u;
        if (lo <= 31 && hi >= 0 && lo <= hi) {
          const uint32_t up = hi >= 31 ? 0xffffffffu : ((1u << (hi + 1)) - 1u);
          const uint32_t dn = lo <= 0 ? 0xffffffffu : ~((1u << lo) - 1u);
          vb = up & dn;
        }
#pragma unroll
        for (int c = 0; c < 32; ++c) x[c] = ((vb >> c) & 1u) ? x[c] : -kInf;
      }
      any_unmasked |= (vb & ~kbits) != 0u;
      float mt = -kInf;
#pragma unroll
      for (int c = 0; c < 32; ++c) mt = fmaxf(mt, x[c]);
      if (mt > m2 + kRescaleThreshold || (m2 == -kInf && mt > -kInf)) {
        if (m2 > -kInf) {
          const float alpha = ex2_approx(m2 - mt);
          l *= alpha;
          dsum *= alpha;
        }
        m2 = mt;
      }
      if (m2 > -kInf) {
        float ls = 0.f, ds = 0.f;
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const float e = ex2_approx(x[c] - m2);
          ls += e;
          ds = fmaf(e, __uint_as_float(dr[c]), ds);
        }
        l += ls;
        dsum += ds;
      }
    }
    // merge the four column groups: (m, l, dsum) -> (max m, rescaled sums)
    if (g > 0) {
      mg_m[g - 1][row] = m2;
      mg_l[g - 1][row] = l;
      mg_d[g - 1][row] = dsum;
      mg_any[g - 1][row] = any_unmasked ? 1 : 0;
    }
    group_sync();
    if (g == 0 && (ok || n == 0) && q < p.Sq) {
      float mm = m2;
#pragma unroll
      for (int i = 0; i < kGroups - 1; ++i) {
        mm = fmaxf(mm, mg_m[i][row]);
        any_unmasked = any_unmasked || mg_any[i][row] != 0;
      }
      float lt = 0.f, dt = 0.f;
      if (mm > -kInf) {
        const float a0 = m2 > -kInf ? ex2_approx(m2 - mm) : 0.f;
        lt = l * a0;
        dt = dsum * a0;
#pragma unroll
        for (int i = 0; i < kGroups - 1; ++i) {
          const float mi = mg_m[i][row];
          const float ai = mi > -kInf ? ex2_approx(mi - mm) : 0.f;
          lt = fmaf(mg_l[i][row], ai, lt);
          dt = fmaf(mg_d[i][row], ai, dt);
        }
      }
      float L2 = kInf, dl = 0.f, pm = 0.f;
      if (lt > 0.f) {
        L2 = mm + __log2f(lt);
        dl = dt / lt;
        if (p.has_key_mask) pm = any_unmasked ? ex2_approx(p.masked_x2 - L2) : 1.f / lt;
      }
      const size_t idx = static_cast<size_t>(bh) * p.Sq + q;
      p.L2[idx] = L2;
      p.delta[idx] = dl;
      if (p.has_key_mask) p.pm[idx] = pm;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, L::TMEM_COLS);
  }
}

template <int DP, bool HAS_BIAS>
cudaError_t launch_t(const DenseMaps& m, const DenseParams& p, cudaStream_t s) {
  using L = Stats2Layout<DP>;
  auto kern = stats2_kernel<DP, HAS_BIAS>;
  const int smem = L::BYTES + 1024;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  dim3 grid(p.B * p.H, cdiv(p.Sq, L::BQ));
  kern<<<grid, 576, smem, s>>>(m.q128, m.k128, m.v128, m.dy128, m.bias128, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_stats2(const DenseMaps& m, const DenseParams& p, bool bias, cudaStream_t s) {
  const int DP = padded_head_dim(p.D);
  if (DP == 64) return bias ? launch_t<64, true>(m, p, s) : launch_t<64, false>(m, p, s);
  return bias ? launch_t<128, true>(m, p, s) : launch_t<128, false>(m, p, s);
}

}  // namespace attn
