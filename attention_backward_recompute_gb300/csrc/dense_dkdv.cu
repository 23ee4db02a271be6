// dK / dV kernel: one CTA per (batch*head, 128-key tile), looping over the
// visible 64-query tiles.  Follows the five-product backward of rlx-cpu
// src/attention_bwd.rs (fn backward_dense_head_all) with the products kept
// per tile:
//   S^T  = K_j Q_i^T                  (tcgen05, M=128 keys, N=64 queries)
//   P^T  = exp(S^T*scale + bias - lse)  in registers, masks in-tile
//   dV_j += P^T dY_i                  (tcgen05, accumulate in TMEM)
//   dP^T = V_j dY_i^T                 (tcgen05)
//   dS^T = P^T * (dP^T - delta)       in registers (scale folded into dK)
//   dK_j += dS^T Q_i                  (tcgen05, accumulate in TMEM)
// Warp roles: warp 0 loads tiles with TMA, warp 1 issues MMAs (one thread),
// warps 4..11 form two warpgroups that each own 32 of the 64 query columns of
// every tile for all 128 keys (thread = key row = TMEM lane).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "dense_common.cuh"
#include "dense_launch.h"
#include "sm103.cuh"

namespace attn {
using namespace sm103;

namespace {

template <int DP, bool SPLIT>
struct DkdvLayout {
  static constexpr int NCH = DP / 64;          // 128-byte column chunks of a row
  static constexpr int NSP = SPLIT ? 2 : 1;    // copies of every operand tile (hi, lo)
  static constexpr int BK = 128, BQ = 64;
  static constexpr int KV = NCH * BK * 128;     // bytes of one copy of the K (or V) tile
  static constexpr int QT = NCH * BQ * 128;     // bytes of one copy of a Q (or dY) tile
  static constexpr int BIAS = SPLIT ? 0 : 2 * BQ * 128;  // two 64-key halves of 64 query rows
  static constexpr int PT = BK * 128;           // P^T / dS^T: 128 keys x 64 queries bf16
  static constexpr int K_OFF = 0;
  static constexpr int V_OFF = K_OFF + NSP * KV;
  static constexpr int Q_OFF = V_OFF + NSP * KV;          // 2 stages x NSP copies
  static constexpr int DY_OFF = Q_OFF + 2 * NSP * QT;      // 2 stages x NSP copies
  static constexpr int BIAS_OFF = DY_OFF + 2 * NSP * QT;   // 2 stages
  static constexpr int P_OFF = BIAS_OFF + 2 * BIAS;        // NSP copies
  static constexpr int DS_OFF = P_OFF + NSP * PT;          // NSP copies
  static constexpr int ST_OFF = DS_OFF + NSP * PT;         // 2 stages x {L2, delta, pm} x 64 floats
  static constexpr int BYTES = ST_OFF + 2 * 3 * BQ * 4;
  static constexpr int TMEM_COLS = (2 * DP + 128) <= 256 ? 256 : 512;
  // TMEM columns: dV [0, DP), dK [DP, 2DP), S^T [2DP, 2DP+64), dP^T [2DP+64, 2DP+128)
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
    dkdv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_dy,
                const __grid_constant__ CUtensorMap tm_bias, const __grid_constant__ CUtensorMap tm_q_lo,
                const __grid_constant__ CUtensorMap tm_k_lo, const __grid_constant__ CUtensorMap tm_v_lo,
                const __grid_constant__ CUtensorMap tm_dy_lo, const DenseParams p) {
  using L = DkdvLayout<DP, SPLIT>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t bar_kv, bar_full[2], bar_empty[2], bar_s_full, bar_dp_full, bar_p_full, bar_ds_full,
      bar_p_free, bar_ds_free, bar_acc;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bh = blockIdx.x;
  const int b = bh / p.H, h = bh - b * p.H;
  const int k0 = blockIdx.y * L::BK;
  const int k1 = imin(k0 + L::BK - 1, p.Sk - 1);
  int i_lo, i_hi;
  query_tile_range(p, k0, k1, L::BQ, &i_lo, &i_hi);
  const int n = i_hi - i_lo;
  const Abort ab{&abort_flag, p.err};

  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bar_kv, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bar_full[s], 2);   // TMA bytes + statistics written
      mbar_init(&bar_empty[s], 1);  // MMA commit
    }
    mbar_init(&bar_s_full, 1);
    mbar_init(&bar_dp_full, 1);
    mbar_init(&bar_p_full, 8);   // one arrive per compute warp
    mbar_init(&bar_ds_full, 8);
    mbar_init(&bar_p_free, 1);
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
  const uint32_t t_dv = tmem, t_dk = tmem + DP, t_s = tmem + 2 * DP, t_dp = tmem + 2 * DP + 64;

  if (n > 0 && warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_map(&tm_q);
      tma_prefetch_map(&tm_k);
      tma_prefetch_map(&tm_v);
      tma_prefetch_map(&tm_dy);
      if (HAS_BIAS) tma_prefetch_map(&tm_bias);
      mbar_arrive_expect_tx(&bar_kv, 2 * L::NSP * L::KV);
      for (int hl = 0; hl < L::NSP; ++hl)
        for (int c = 0; c < L::NCH; ++c) {
          tma_load_4d(sm + L::K_OFF + hl * L::KV + c * (L::BK * 128), hl ? &tm_k_lo : &tm_k, &bar_kv, c * 64, k0, h, b);
          tma_load_4d(sm + L::V_OFF + hl * L::KV + c * (L::BK * 128), hl ? &tm_v_lo : &tm_v, &bar_kv, c * 64, k0, h, b);
        }
    }
    int last_use[2] = {-1, -1};
    bool ok = true;
    for (int t = 0; t < n && ok; ++t) {
      const int s = t & 1;
      if (t >= 2) ok = mbar_wait(&bar_empty[s], ((t >> 1) - 1) & 1, ab);
      if (!ok) break;
      const int q0 = (i_lo + t) * L::BQ;
      if (lane == 0) {
        const uint32_t bytes = 2 * L::NSP * L::QT + (HAS_BIAS ? L::BIAS : 0);
        mbar_arrive_expect_tx(&bar_full[s], bytes);
        for (int hl = 0; hl < L::NSP; ++hl)
          for (int c = 0; c < L::NCH; ++c) {
            const int o = (s * L::NSP + hl) * L::QT + c * (L::BQ * 128);
            tma_load_4d(sm + L::Q_OFF + o, hl ? &tm_q_lo : &tm_q, &bar_full[s], c * 64, q0, h, b);
            tma_load_4d(sm + L::DY_OFF + o, hl ? &tm_dy_lo : &tm_dy, &bar_full[s], c * 64, q0, h, b);
          }
        if (HAS_BIAS) {
          uint8_t* bs = sm + L::BIAS_OFF + s * L::BIAS;
          tma_load_4d(bs, &tm_bias, &bar_full[s], k0, q0, h, b);
          tma_load_4d(bs + L::BQ * 128, &tm_bias, &bar_full[s], k0 + 64, q0, h, b);
        }
      }
      float* st = reinterpret_cast<float*>(sm + L::ST_OFF) + s * 3 * L::BQ;
      for (int r = lane; r < L::BQ; r += 32) {
        const int q = q0 + r;
        const bool in = q < p.Sq;
        const size_t idx = static_cast<size_t>(bh) * p.Sq + q;
        st[r] = in ? p.L2[idx] : __int_as_float(0x7f800000);
        st[L::BQ + r] = in ? p.delta[idx] : 0.f;
        st[2 * L::BQ + r] = (in && p.has_key_mask) ? p.pm[idx] : 0.f;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_full[s]);
      last_use[s] = t;
    }
    // Let every copy this CTA started land before shared memory is released.
    if (lane == 0) {
      for (int s = 0; s < 2; ++s)
        if (last_use[s] >= 0) drain_wait(&bar_full[s], (last_use[s] >> 1) & 1);
      drain_wait(&bar_kv, 0);
    }
  } else if (n > 0 && warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t id_s = idesc_bf16(128, 64, false, false);
      constexpr uint32_t id_acc = idesc_bf16(128, DP, false, true);
      const uint32_t sK = smem_addr(sm + L::K_OFF), sV = smem_addr(sm + L::V_OFF);
      const uint32_t sP = smem_addr(sm + L::P_OFF), sDS = smem_addr(sm + L::DS_OFF);
      auto q_at = [&](int s) { return smem_addr(sm + L::Q_OFF + s * L::NSP * L::QT); };
      auto dy_at = [&](int s) { return smem_addr(sm + L::DY_OFF + s * L::NSP * L::QT); };
      // Split operands: x = hi + lo (two bf16 copies); a product is
      // hi*hi + hi*lo + lo*hi, all accumulated in fp32.
      constexpr int NPROD = SPLIT ? 3 : 1;
      // X^T-product: D[128 x 64] = A_tile[128 x DP] * B_tile[64 x DP]^T, both K-major.
      auto issue_xt = [&](uint32_t d, uint32_t a_base, uint32_t b_base) {
#pragma unroll
        for (int pr = 0; pr < NPROD; ++pr) {
          const uint32_t a0 = a_base + (pr == 2 ? L::KV : 0), b0 = b_base + (pr == 1 ? L::QT : 0);
#pragma unroll
          for (int kk = 0; kk < DP / 16; ++kk) {
            const int c = kk >> 2, o = (kk & 3) * 32;
            const uint64_t ad = sdesc_sw128(a0 + c * (L::BK * 128) + o, 16, 1024);
            const uint64_t bd = sdesc_sw128(b0 + c * (L::BQ * 128) + o, 16, 1024);
            mma_bf16_ss(d, ad, bd, id_s, (pr > 0 || kk > 0) ? 1u : 0u);
          }
        }
      };
      // accumulate: D[128 x DP] += A[128 x 64] (K-major) * B[64 x DP] (MN-major)
      auto issue_acc = [&](uint32_t d, uint32_t a_base, uint32_t b_base, bool first) {
#pragma unroll
        for (int pr = 0; pr < NPROD; ++pr) {
          const uint32_t a0 = a_base + (pr == 2 ? L::PT : 0), b0 = b_base + (pr == 1 ? L::QT : 0);
#pragma unroll
          for (int kk = 0; kk < L::BQ / 16; ++kk) {
            const uint64_t ad = sdesc_sw128(a0 + kk * 32, 16, 1024);
            const uint64_t bd = sdesc_sw128(b0 + kk * 16 * 128, L::BQ * 128, 1024);
            mma_bf16_ss(d, ad, bd, id_acc, (first && pr == 0 && kk == 0) ? 0u : 1u);
          }
        }
      };
      bool ok = mbar_wait(&bar_kv, 0, ab);
      if (ok) ok = mbar_wait(&bar_full[0], 0, ab);
      if (ok) {
        tc_fence_after();
        issue_xt(t_s, sK, q_at(0));
        mma_commit(&bar_s_full);
        issue_xt(t_dp, sV, dy_at(0));
        mma_commit(&bar_dp_full);
      }
      for (int t = 0; t < n && ok; ++t) {
        const int s = t & 1;
        if (!(ok = mbar_wait(&bar_p_full, t & 1, ab))) break;
        tc_fence_after();
        issue_acc(t_dv, sP, dy_at(s), t == 0);
        mma_commit(&bar_p_free);
        if (t + 1 < n) {
          if (!(ok = mbar_wait(&bar_full[s ^ 1], ((t + 1) >> 1) & 1, ab))) break;
          tc_fence_after();
          issue_xt(t_s, sK, q_at(s ^ 1));
          mma_commit(&bar_s_full);
        }
        if (!(ok = mbar_wait(&bar_ds_full, t & 1, ab))) break;
        tc_fence_after();
        issue_acc(t_dk, sDS, q_at(s), t == 0);
        mma_commit(&bar_ds_free);
        mma_commit(&bar_empty[s]);
        if (t + 1 < n) {
          issue_xt(t_dp, sV, dy_at(s ^ 1));
          mma_commit(&bar_dp_full);
        }
      }
      mma_commit(&bar_acc);
      drain_wait(&bar_acc, 0);  // every issued MMA has finished
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax / dS warpgroups
    const int wg = (warp - 4) >> 2;
    const int lg = warp & 3;
    const int row = lg * 32 + lane;  // key row inside the tile == TMEM lane
    const int key = k0 + row;
    const int c0 = wg * 32;          // first query column of this warp
    const uint32_t lane_addr = static_cast<uint32_t>(lg * 32) << 16;
    bool ok = n > 0;
    if (n > 0) {
      bool kmasked = false;
      if (p.has_key_mask && key < p.Sk) kmasked = p.key_mask[static_cast<size_t>(b) * p.Sk + key] < p.mask_thr;
      const uint32_t sP = smem_addr(sm + L::P_OFF), sDS = smem_addr(sm + L::DS_OFF);
      // bias element (query ql, this key) inside the 64-key half of a stage
      const int half = row >> 6, kc = (row & 63) >> 3, kb = (row & 7) * 2;
      for (int t = 0; t < n && ok; ++t) {
        const int s = t & 1;
        const int q0 = (i_lo + t) * L::BQ;
        if (!(ok = mbar_wait_warp(&bar_full[s], (t >> 1) & 1, ab))) break;
        if (!(ok = mbar_wait_warp(&bar_s_full, t & 1, ab))) break;
        tc_fence_after();
        uint32_t sr[32];
        tmem_ld32(t_s + lane_addr + c0, sr);
        tmem_ld_wait();
        const float* st = reinterpret_cast<const float*>(sm + L::ST_OFF) + s * 3 * L::BQ;
        const bool full = tile_fully_visible(p, q0, q0 + L::BQ - 1, k0, k0 + L::BK - 1);
        const uint8_t* bias_s = sm + L::BIAS_OFF + s * L::BIAS + half * (L::BQ * 128);
        float pr[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const int ql = c0 + c;
          float x = fmaf(__uint_as_float(sr[c]), p.scale_log2, -st[ql]);
          if (HAS_BIAS) {
            const uint32_t off = ql * 128 + ((((kc ^ ql) & 7)) << 4) + kb;
            const uint16_t bb = *reinterpret_cast<const uint16_t*>(bias_s + off);
            x = fmaf(__uint_as_float(static_cast<uint32_t>(bb) << 16), kLog2e, x);
          }
          const bool vis = full || pair_visible(p, q0 + ql, key);
          float pv = ex2_approx(x);
          if (kmasked) pv = st[2 * L::BQ + ql];
          pr[c] = vis ? pv : 0.f;
        }
        if (t > 0 && !(ok = mbar_wait_warp(&bar_p_free, (t - 1) & 1, ab))) break;
        store_row32<SPLIT>(sP, L::PT, row, c0, pr);
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar_p_full);
        if (!(ok = mbar_wait_warp(&bar_dp_full, t & 1, ab))) break;
        tc_fence_after();
        uint32_t dr[32];
        tmem_ld32(t_dp + lane_addr + c0, dr);
        tmem_ld_wait();
        float ds[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) ds[c] = pr[c] * (__uint_as_float(dr[c]) - st[L::BQ + c0 + c]);
        if (t > 0 && !(ok = mbar_wait_warp(&bar_ds_free, (t - 1) & 1, ab))) break;
        store_row32<SPLIT>(sDS, L::PT, row, c0, ds);
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar_ds_full);
      }
      if (ok) ok = mbar_wait_warp(&bar_acc, 0, ab);
      tc_fence_after();
    }
    // ------------------------------------------------------------ epilogue
    // warpgroup 0 writes dV, warpgroup 1 writes dK (times the softmax scale);
    // a tile no query sees gets zeros.
    const bool want = wg == 0 ? (p.wrt & 4u) != 0 : (p.wrt & 2u) != 0;
    if (want && (ok || n == 0)) {
      const int64_t* so = wg == 0 ? p.s_dv : p.s_dk;
      const int64_t roff = static_cast<int64_t>(b) * so[2] + static_cast<int64_t>(h) * so[1] +
                           static_cast<int64_t>(key) * so[0];
      void* out = wg == 0 ? p.dv : p.dk;
      const float f = wg == 0 ? 1.f : p.scale;
      const uint32_t tacc = (wg == 0 ? t_dv : t_dk) + lane_addr;
#pragma unroll 1
      for (int cc = 0; cc < DP / 32 && cc * 32 < p.D; ++cc) {
        uint32_t r[32];
        if (n > 0) {
          tmem_ld32(tacc + cc * 32, r);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) r[j] = 0u;
        }
        if (key < p.Sk) store_out32<SPLIT>(out, roff, cc * 32, p.D, r, f);
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
cudaError_t launch_dkdv_t(const DenseMaps& m, const DenseParams& p, cudaStream_t s) {
  using L = DkdvLayout<DP, SPLIT>;
  auto kern = dkdv_kernel<DP, HAS_BIAS, SPLIT>;
  const int smem = L::BYTES + 1024;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  dim3 grid(p.B * p.H, cdiv(p.Sk, L::BK));
  kern<<<grid, 384, smem, s>>>(m.q64, m.k128, m.v128, m.dy64, m.bias64, m.q64_lo, m.k128_lo, m.v128_lo, m.dy64_lo, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_dkdv(const DenseMaps& m, const DenseParams& p, bool bias, cudaStream_t s) {
  const int DP = padded_head_dim(p.D);
  if (m.split) return launch_dkdv_t<64, false, true>(m, p, s);
  if (DP == 64) return bias ? launch_dkdv_t<64, true, false>(m, p, s) : launch_dkdv_t<64, false, false>(m, p, s);
  return bias ? launch_dkdv_t<128, true, false>(m, p, s) : launch_dkdv_t<128, false, false>(m, p, s);
}

}  // namespace attn
