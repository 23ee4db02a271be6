// Row-statistics prologue of the dense backward, bf16 storage, self-contained
// mode (no O or LSE from the caller).
//
// One CTA per (batch*head, 128-query tile) sweeps the visible 128-key tiles.
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
// A custom-masked key enters through a per-tile bit set, not through its
// score: its term 2^(mask_neg*log2(e) - m) underflows to exactly zero as soon
// as the row has a visible unmasked key (whose x exceeds the masked value by
// far more than 150), so such keys are left out of the sums; a row whose
// visible keys are all custom-masked has equal x = mask_neg*log2(e) on every
// one of them, so its statistics are the count of those keys and the plain
// sum of their dP, kept on the side until an unmasked key shows up.
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
  // the 128-bit set of the tile's custom-masked key columns
  static constexpr int COL = 16;
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

template <int DP, bool HAS_BIAS, bool ELEM>
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
  __shared__ float mg_c[kGroups - 1][128], mg_md[kGroups - 1][128];

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
        uint32_t* bits = reinterpret_cast<uint32_t*>(sm + L::COL_OFF + s * L::COL);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint32_t w = __ballot_sync(0xffffffffu, kmv[i] < p.mask_thr);
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
    float mcnt = 0.f, mdsum = 0.f;  // visible custom-masked keys while no unmasked one is seen
    bool any_unmasked = false;
    for (int t = 0; t < n && ok; ++t) {
      const int s = t % kStages, bb = t & 1;
      const int kk0 = (j_lo + t) * L::BK;
      // per-element mask bits of this row's 32 columns (loaded before the wait)
      uint32_t ebits = 0u;
      if (ELEM && q < p.Sq && kk0 + 32 * g < p.Sk) ebits = p.elem_rows[(static_cast<size_t>(bh) * p.Sq + q) * p.ew_q + (kk0 >> 5) + g];
      if (!(ok = mbar_wait_warp(&bar_full[s], (t / kStages) & 1, ab))) break;
      // bias term of the group's 32 columns while the tensor core works:
      // x = bias*log2(e), as 16 packed pairs of adjacent columns
      const uint32_t kbits =
          (p.has_key_mask ? reinterpret_cast<const uint32_t*>(sm + L::COL_OFF + s * L::COL)[g] : 0u) | ebits;
      // bias half (64 keys) g >> 1, 16-byte chunks 4 (g & 1) .. + 3 of this row
      const uint8_t* brow = sm + L::BIAS_OFF + s * L::BIAS + (g >> 1) * (L::BQ * 128) + row * 128;
      uint64_t x[16];
      if (HAS_BIAS) {
        const uint64_t l2e = f2_pack(kLog2e, kLog2e);
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {  // 8 keys per 16-byte bias chunk
          const uint4 w4 = *reinterpret_cast<const uint4*>(brow + (((4 * (g & 1) + jj) ^ (row & 7)) << 4));
          x[4 * jj] = f2_mul(f2_from_bf16x2(w4.x), l2e);
          x[4 * jj + 1] = f2_mul(f2_from_bf16x2(w4.y), l2e);
          x[4 * jj + 2] = f2_mul(f2_from_bf16x2(w4.z), l2e);
          x[4 * jj + 3] = f2_mul(f2_from_bf16x2(w4.w), l2e);
        }
      }
      // the dP commit follows the S MMAs of the tile, so it covers both
      if (!(ok = mbar_wait_warp(&bar_dp_full, t & 1, ab))) break;
      tc_fence_after();
      {
        uint32_t sr[32];
        tmem_ld32(tmem + L::T_S + bb * 128 + 32 * g + lane_addr, sr);
        tmem_ld_wait();
        const uint64_t sl2 = f2_pack(p.scale_log2, p.scale_log2);
#pragma unroll
        for (int i = 0; i < 16; ++i)
          x[i] = HAS_BIAS ? f2_fma(f2_pack_u(sr[2 * i], sr[2 * i + 1]), sl2, x[i])
                          : f2_mul(f2_pack_u(sr[2 * i], sr[2 * i + 1]), sl2);
      }
      // dP of the same columns; then both buffers go back to the tensor core
      uint32_t dr[32];
      tmem_ld32(tmem + L::T_DP + 32 * g + lane_addr, dr);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&bar_used[bb]);
        mbar_arrive(&bar_empty[s]);  // bias and mask bits read
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
      }
      // visible and not custom-masked
      const uint32_t vis = vb & ~kbits;
      if (vis != 0xffffffffu) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          float a0, a1;
          f2_split(x[i], a0, a1);
          a0 = ((vis >> (2 * i)) & 1u) ? a0 : -kInf;
          a1 = ((vis >> (2 * i + 1)) & 1u) ? a1 : -kInf;
          x[i] = f2_pack(a0, a1);
        }
      }
      any_unmasked |= vis != 0u;
      float mt = -kInf;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        float a0, a1;
        f2_split(x[i], a0, a1);
        mt = fmax3(mt, a0, a1);
      }
      if (mt > m2 + kRescaleThreshold || (m2 == -kInf && mt > -kInf)) {
        if (m2 > -kInf) {
          const float alpha = ex2_approx(m2 - mt);
          l *= alpha;
          dsum *= alpha;
        }
        m2 = mt;
      }
      if (m2 > -kInf) {
        const uint64_t negm = f2_pack(-m2, -m2);
        uint64_t ls = 0ull, ds = 0ull;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          float d0, d1;
          f2_split(f2_add(x[i], negm), d0, d1);
          const uint64_t e = f2_pack(ex2_approx(d0), ex2_approx(d1));
          ls = f2_add(ls, e);
          ds = f2_fma(e, f2_pack_u(dr[2 * i], dr[2 * i + 1]), ds);
        }
        float l0, l1, d0, d1;
        f2_split(ls, l0, l1);
        f2_split(ds, d0, d1);
        l += l0 + l1;
        dsum += d0 + d1;
      } else {
        // no visible unmasked key so far: the row's terms are those of its
        // visible custom-masked keys, each with weight 2^0
        const uint32_t mv = vb & kbits;
        if (mv != 0u) {
          mcnt += static_cast<float>(__popc(mv));
#pragma unroll
          for (int c = 0; c < 32; ++c) mdsum += ((mv >> c) & 1u) ? __uint_as_float(dr[c]) : 0.f;
        }
      }
    }
    // merge the four column groups: (m, l, dsum) -> (max m, rescaled sums)
    if (g > 0) {
      mg_m[g - 1][row] = m2;
      mg_l[g - 1][row] = l;
      mg_d[g - 1][row] = dsum;
      mg_any[g - 1][row] = any_unmasked ? 1 : 0;
      mg_c[g - 1][row] = mcnt;
      mg_md[g - 1][row] = mdsum;
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
      } else if (p.has_custom) {
        // every visible key of the row is custom-masked: all carry the same x
        lt = mcnt;
        dt = mdsum;
#pragma unroll
        for (int i = 0; i < kGroups - 1; ++i) {
          lt += mg_c[i][row];
          dt += mg_md[i][row];
        }
        mm = p.masked_x2;
      }
      float L2 = kInf, dl = 0.f, pm = 0.f;
      if (lt > 0.f) {
        L2 = mm + __log2f(lt);
        dl = dt / lt;
        if (p.has_custom) pm = any_unmasked ? ex2_approx(p.masked_x2 - L2) : 1.f / lt;
      }
      const size_t idx = static_cast<size_t>(bh) * p.Sq + q;
      p.L2[idx] = L2;
      p.delta[idx] = dl;
      if (p.has_custom) p.pm[idx] = pm;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, L::TMEM_COLS);
  }
}

template <int DP, bool HAS_BIAS, bool ELEM>
cudaError_t launch_t(const DenseMaps& m, const DenseParams& p, cudaStream_t s) {
  using L = Stats2Layout<DP>;
  auto kern = stats2_kernel<DP, HAS_BIAS, ELEM>;
  const int smem = max(L::BYTES + 1024, kSmemOneCtaPerSm);  // all 512 TMEM columns: one CTA per SM
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  dim3 grid(p.B * p.H, cdiv(p.Sq, L::BQ));
  kern<<<grid, 576, smem, s>>>(m.q128, m.k128, m.v128, m.dy128, m.bias128, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_stats2(const DenseMaps& m, const DenseParams& p, bool bias, cudaStream_t s) {
  const int DP = padded_head_dim(p.D);
  if (p.elem_rows) {  // per-element custom mask
    if (DP == 64) return bias ? launch_t<64, true, true>(m, p, s) : launch_t<64, false, true>(m, p, s);
    return bias ? launch_t<128, true, true>(m, p, s) : launch_t<128, false, true>(m, p, s);
  }
  if (DP == 64) return bias ? launch_t<64, true, false>(m, p, s) : launch_t<64, false, false>(m, p, s);
  return bias ? launch_t<128, true, false>(m, p, s) : launch_t<128, false, false>(m, p, s);
}

}  // namespace attn
