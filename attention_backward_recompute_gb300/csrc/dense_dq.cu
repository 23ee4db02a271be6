// dQ kernel: one CTA per (batch*head, 128-query tile), looping over the
// visible 64-key tiles (rlx-cpu src/attention_bwd.rs, fn backward_dense_head_all,
// the dQ = dS K product, with scores and softmax recomputed per tile):
//   S  = Q_i K_j^T          (tcgen05, M=128 queries, N=64 keys)
//   dP = dY_i V_j^T         (tcgen05)
//   dS = P * (dP - delta),  P = exp(S*scale + bias - lse), masks in-tile
//   dQ_i += dS K_j          (tcgen05, accumulate in TMEM; scale applied at the end)
// Warp 0: TMA producer; warp 1: MMA issuer; warps 4..11: two warpgroups, each
// owning 32 of the 64 key columns of every tile for all 128 query rows.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "dense_common.cuh"
#include "dense_launch.h"
#include "sm103.cuh"

namespace attn {
using namespace sm103;

namespace {

template <int DP, bool SPLIT>
struct DqLayout {
  static constexpr int NCH = DP / 64;
  static constexpr int NSP = SPLIT ? 2 : 1;    // copies of every operand tile (hi, lo)
  static constexpr int BQ = 128, BK = 64;
  static constexpr int QT = NCH * BQ * 128;    // one copy of the Q or dY tile (128 rows)
  static constexpr int KT = NCH * BK * 128;    // one copy of a K or V tile (64 rows)
  static constexpr int BIAS = SPLIT ? 0 : BQ * 128;  // 128 query rows x 64 keys
  static constexpr int DS = BQ * 128;          // one copy of dS: 128 queries x 64 keys bf16
  static constexpr int Q_OFF = 0;
  static constexpr int DY_OFF = Q_OFF + NSP * QT;
  static constexpr int K_OFF = DY_OFF + NSP * QT;          // 2 stages x NSP copies
  static constexpr int V_OFF = K_OFF + 2 * NSP * KT;       // 2 stages x NSP copies
  static constexpr int BIAS_OFF = V_OFF + 2 * NSP * KT;    // 2 stages
  static constexpr int DS_OFF = BIAS_OFF + 2 * BIAS;       // NSP copies
  static constexpr int BYTES = DS_OFF + NSP * DS;
  static constexpr int TMEM_COLS = 256;  // dQ [0, DP), S [DP, DP+64), dP [DP+64, DP+128)
};

__device__ __forceinline__ bool drain_wait(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_test(bar, parity)) {
    if (global_timer_ns() - t0 > ATTN_WAIT_TIMEOUT_NS) return false;
  }
  return true;
}

template <int DP, bool HAS_BIAS, bool SPLIT>
__global__ void __launch_bounds__(384, 1)
    dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
              const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_dy,
              const __grid_constant__ CUtensorMap tm_bias, const __grid_constant__ CUtensorMap tm_q_lo,
              const __grid_constant__ CUtensorMap tm_k_lo, const __grid_constant__ CUtensorMap tm_v_lo,
              const __grid_constant__ CUtensorMap tm_dy_lo, const DenseParams p) {
  using L = DqLayout<DP, SPLIT>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t bar_qdy, bar_full[2], bar_empty[2], bar_s_full, bar_s_free, bar_dp_full, bar_ds_full,
      bar_ds_free, bar_acc;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag;

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
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bar_full[s], 1);
      mbar_init(&bar_empty[s], 1);
    }
    mbar_init(&bar_s_full, 1);
    mbar_init(&bar_s_free, 8);
    mbar_init(&bar_dp_full, 1);
    mbar_init(&bar_ds_full, 8);
    mbar_init(&bar_ds_free, 1);
    mbar_init(&bar_acc, 1);
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
  const uint32_t t_dq = tmem, t_s = tmem + DP, t_dp = tmem + DP + 64;

  if (n > 0 && warp == 0) {
    // ------------------------------------------------------------ producer
    int last_use[2] = {-1, -1};
    if (lane == 0) {
      tma_prefetch_map(&tm_q);
      tma_prefetch_map(&tm_k);
      tma_prefetch_map(&tm_v);
      tma_prefetch_map(&tm_dy);
      if (HAS_BIAS) tma_prefetch_map(&tm_bias);
      mbar_arrive_expect_tx(&bar_qdy, 2 * L::NSP * L::QT);
      for (int hl = 0; hl < L::NSP; ++hl)
        for (int c = 0; c < L::NCH; ++c) {
          tma_load_4d(sm + L::Q_OFF + hl * L::QT + c * (L::BQ * 128), hl ? &tm_q_lo : &tm_q, &bar_qdy, c * 64, q0,
                      h, b);
          tma_load_4d(sm + L::DY_OFF + hl * L::QT + c * (L::BQ * 128), hl ? &tm_dy_lo : &tm_dy, &bar_qdy, c * 64,
                      q0, h, b);
        }
      bool ok = true;
      for (int t = 0; t < n && ok; ++t) {
        const int s = t & 1;
        if (t >= 2) ok = mbar_wait(&bar_empty[s], ((t >> 1) - 1) & 1, ab);
        if (!ok) break;
        const int kk0 = (j_lo + t) * L::BK;
        mbar_arrive_expect_tx(&bar_full[s], 2 * L::NSP * L::KT + (HAS_BIAS ? L::BIAS : 0));
        for (int hl = 0; hl < L::NSP; ++hl)
          for (int c = 0; c < L::NCH; ++c) {
            const int o = (s * L::NSP + hl) * L::KT + c * (L::BK * 128);
            tma_load_4d(sm + L::K_OFF + o, hl ? &tm_k_lo : &tm_k, &bar_full[s], c * 64, kk0, h, b);
            tma_load_4d(sm + L::V_OFF + o, hl ? &tm_v_lo : &tm_v, &bar_full[s], c * 64, kk0, h, b);
          }
        if (HAS_BIAS) tma_load_4d(sm + L::BIAS_OFF + s * L::BIAS, &tm_bias, &bar_full[s], kk0, q0, h, b);
        last_use[s] = t;
      }
      for (int s = 0; s < 2; ++s)
        if (last_use[s] >= 0) drain_wait(&bar_full[s], (last_use[s] >> 1) & 1);
      drain_wait(&bar_qdy, 0);
    }
    __syncwarp();
  } else if (n > 0 && warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t id_s = idesc_bf16(128, 64, false, false);
      constexpr uint32_t id_acc = idesc_bf16(128, DP, false, true);
      const uint32_t sQ = smem_addr(sm + L::Q_OFF), sDY = smem_addr(sm + L::DY_OFF);
      const uint32_t sDS = smem_addr(sm + L::DS_OFF);
      auto k_at = [&](int s) { return smem_addr(sm + L::K_OFF + s * L::NSP * L::KT); };
      auto v_at = [&](int s) { return smem_addr(sm + L::V_OFF + s * L::NSP * L::KT); };
      // split operands: hi*hi + hi*lo + lo*hi
      constexpr int NPROD = SPLIT ? 3 : 1;
      auto issue_xt = [&](uint32_t d, uint32_t a_base, uint32_t b_base) {
#pragma unroll
        for (int pr = 0; pr < NPROD; ++pr) {
          const uint32_t a0 = a_base + (pr == 2 ? L::QT : 0), b0 = b_base + (pr == 1 ? L::KT : 0);
#pragma unroll
          for (int kk = 0; kk < DP / 16; ++kk) {
            const int c = kk >> 2, o = (kk & 3) * 32;
            const uint64_t ad = sdesc_sw128(a0 + c * (L::BQ * 128) + o, 16, 1024);
            const uint64_t bd = sdesc_sw128(b0 + c * (L::BK * 128) + o, 16, 1024);
            mma_bf16_ss(d, ad, bd, id_s, (pr > 0 || kk > 0) ? 1u : 0u);
          }
        }
      };
      auto issue_dq = [&](int s, bool first) {
#pragma unroll
        for (int pr = 0; pr < NPROD; ++pr) {
          const uint32_t a0 = sDS + (pr == 2 ? L::DS : 0), b0 = k_at(s) + (pr == 1 ? L::KT : 0);
#pragma unroll
          for (int kk = 0; kk < L::BK / 16; ++kk) {
            const uint64_t ad = sdesc_sw128(a0 + kk * 32, 16, 1024);
            const uint64_t bd = sdesc_sw128(b0 + kk * 16 * 128, L::BK * 128, 1024);
            mma_bf16_ss(t_dq, ad, bd, id_acc, (first && pr == 0 && kk == 0) ? 0u : 1u);
          }
        }
      };
      bool ok = mbar_wait(&bar_qdy, 0, ab);
      if (ok) ok = mbar_wait(&bar_full[0], 0, ab);
      if (ok) {
        tc_fence_after();
        issue_xt(t_s, sQ, k_at(0));
        mma_commit(&bar_s_full);
        issue_xt(t_dp, sDY, v_at(0));
        mma_commit(&bar_dp_full);
      }
      for (int t = 0; t < n && ok; ++t) {
        const int s = t & 1;
        if (t + 1 < n) {
          if (!(ok = mbar_wait(&bar_s_free, t & 1, ab))) break;
          if (!(ok = mbar_wait(&bar_full[s ^ 1], ((t + 1) >> 1) & 1, ab))) break;
          tc_fence_after();
          issue_xt(t_s, sQ, k_at(s ^ 1));
          mma_commit(&bar_s_full);
        }
        if (!(ok = mbar_wait(&bar_ds_full, t & 1, ab))) break;
        tc_fence_after();
        issue_dq(s, t == 0);
        mma_commit(&bar_ds_free);
        mma_commit(&bar_empty[s]);
        if (t + 1 < n) {
          issue_xt(t_dp, sDY, v_at(s ^ 1));
          mma_commit(&bar_dp_full);
        }
      }
      mma_commit(&bar_acc);
      drain_wait(&bar_acc, 0);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax / dS warpgroups
    const int wg = (warp - 4) >> 2;
    const int lg = warp & 3;
    const int row = lg * 32 + lane;  // query row inside the tile == TMEM lane
    const int q = q0 + row;
    const int c0 = wg * 32;          // first key column of this warp
    const uint32_t lane_addr = static_cast<uint32_t>(lg * 32) << 16;
    bool ok = n > 0;
    if (n > 0) {
      float L2q = __int_as_float(0x7f800000), dlt = 0.f, pmq = 0.f;
      if (q < p.Sq) {
        const size_t idx = static_cast<size_t>(bh) * p.Sq + q;
        L2q = p.L2[idx];
        dlt = p.delta[idx];
        if (p.has_key_mask) pmq = p.pm[idx];
      }
      const uint32_t sDS = smem_addr(sm + L::DS_OFF);
      for (int t = 0; t < n && ok; ++t) {
        const int s = t & 1;
        const int kk0 = (j_lo + t) * L::BK;
        uint32_t kbits = 0;
        if (p.has_key_mask) {
          const int key = kk0 + c0 + lane;
          const bool m = key < p.Sk && p.key_mask[static_cast<size_t>(b) * p.Sk + key] < p.mask_thr;
          kbits = __ballot_sync(0xffffffffu, m);
        }
        if (!(ok = mbar_wait_warp(&bar_full[s], (t >> 1) & 1, ab))) break;
        if (!(ok = mbar_wait_warp(&bar_s_full, t & 1, ab))) break;
        tc_fence_after();
        uint32_t sr[32];
        tmem_ld32(t_s + lane_addr + c0, sr);
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar_s_free);
        const bool full = tile_fully_visible(p, q0, q0 + L::BQ - 1, kk0, kk0 + L::BK - 1);
        float bias2[32];
        if (HAS_BIAS) {
          const uint32_t bs = smem_addr(sm + L::BIAS_OFF + s * L::BIAS);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            uint32_t w0, w1, w2, w3;
            asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(w0), "=r"(w1), "=r"(w2), "=r"(w3)
                         : "r"(bs + sw128_offset(row, (c0 >> 3) + j)));
            const uint32_t w[4] = {w0, w1, w2, w3};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              bias2[8 * j + 2 * e] = __uint_as_float(w[e] << 16) * kLog2e;
              bias2[8 * j + 2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u) * kLog2e;
            }
          }
        }
        float pr[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          float x = fmaf(__uint_as_float(sr[c]), p.scale_log2, -L2q);
          if (HAS_BIAS) x += bias2[c];
          const bool vis = full || pair_visible(p, q, kk0 + c0 + c);
          float pv = ex2_approx(x);
          if ((kbits >> c) & 1u) pv = pmq;
          pr[c] = vis ? pv : 0.f;
        }
        if (!(ok = mbar_wait_warp(&bar_dp_full, t & 1, ab))) break;
        tc_fence_after();
        uint32_t dr[32];
        tmem_ld32(t_dp + lane_addr + c0, dr);
        tmem_ld_wait();
        float ds[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) ds[c] = pr[c] * (__uint_as_float(dr[c]) - dlt);
        if (t > 0 && !(ok = mbar_wait_warp(&bar_ds_free, (t - 1) & 1, ab))) break;
        store_row32<SPLIT>(sDS, L::DS, row, c0, ds);
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar_ds_full);
      }
      if (ok) ok = mbar_wait_warp(&bar_acc, 0, ab);
      tc_fence_after();
    }
    // ------------------------------------------------------------ epilogue
    // each warpgroup writes half of the dQ row (times the softmax scale)
    if ((p.wrt & 1u) && (ok || n == 0)) {
      const int64_t roff = static_cast<int64_t>(b) * p.s_dq[2] + static_cast<int64_t>(h) * p.s_dq[1] +
                           static_cast<int64_t>(q) * p.s_dq[0];
      const int half = DP / 2;
#pragma unroll 1
      for (int cc = wg * half / 32; cc < (wg + 1) * half / 32 && cc * 32 < p.D; ++cc) {
        uint32_t r[32];
        if (n > 0) {
          tmem_ld32(t_dq + lane_addr + cc * 32, r);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) r[j] = 0u;
        }
        if (q < p.Sq) store_out32<SPLIT>(p.dq, roff, cc * 32, p.D, r, p.scale);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, L::TMEM_COLS);
  }
}

template <int DP, bool HAS_BIAS, bool SPLIT>
cudaError_t launch_dq_t(const DenseMaps& m, const DenseParams& p, cudaStream_t s) {
  using L = DqLayout<DP, SPLIT>;
  auto kern = dq_kernel<DP, HAS_BIAS, SPLIT>;
  const int smem = L::BYTES + 1024;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  dim3 grid(p.B * p.H, cdiv(p.Sq, L::BQ));
  kern<<<grid, 384, smem, s>>>(m.q128, m.k64, m.v64, m.dy128, m.bias128, m.q128_lo, m.k64_lo, m.v64_lo,
                               m.dy128_lo, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_dq(const DenseMaps& m, const DenseParams& p, bool bias, cudaStream_t s) {
  const int DP = padded_head_dim(p.D);
  if (m.split) return launch_dq_t<64, false, true>(m, p, s);
  if (DP == 64) return bias ? launch_dq_t<64, true, false>(m, p, s) : launch_dq_t<64, false, false>(m, p, s);
  return bias ? launch_dq_t<128, true, false>(m, p, s) : launch_dq_t<128, false, false>(m, p, s);
}

}  // namespace attn
