// Row-statistics prologue of the dense backward.
//
// fwd_stats_kernel (self-contained mode): one CTA per (batch*head, 128-query
// tile) sweeps the visible 64-key tiles like a forward pass with an online
// softmax (scores S = Q K^T on tcgen05, P in registers, O += P V on tcgen05
// into TMEM) and writes per query row
//   L2    = (max + log(sum)) * log2(e)          (+inf for a row with no visible key)
//   delta = rowsum(P * dP) = dY . O              (O normalised)
//   pm    = probability of each custom-masked visible key of the row
// The softmax follows rlx-wgpu src/kernels/attention_bwd.wgsl (fn softmax_row:
// max-subtracted exponentials) and the masks rlx-cpu src/attention_bwd.rs
// (fn apply_synthetic_mask) / attention_bwd.wgsl (fn mask_score).
//
// delta_only_kernel (O and LSE supplied): delta = dY . O per row, L2 from the
// given LSE, pm from LSE and the row's visible-key count.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "dense_common.cuh"
#include "dense_launch.h"
#include "sm103.cuh"

namespace attn {
using namespace sm103;

namespace {

template <int DP, bool SPLIT>
struct FwdLayout {
  static constexpr int NCH = DP / 64;
  static constexpr int NSP = SPLIT ? 2 : 1;        // copies of every operand tile (hi, lo)
  static constexpr int BQ = 128, BK = 64;
  static constexpr int QT = NCH * BQ * 128;
  static constexpr int KT = NCH * BK * 128;
  static constexpr int BIAS = SPLIT ? 0 : BQ * 128;
  static constexpr int PT = BQ * 128;              // P: 128 queries x 64 keys bf16 (one copy)
  static constexpr int Q_OFF = 0;
  static constexpr int DY_OFF = Q_OFF + NSP * QT;
  static constexpr int K_OFF = DY_OFF + NSP * QT;        // 2 stages x NSP copies
  static constexpr int V_OFF = K_OFF + 2 * NSP * KT;     // 2 stages x NSP copies
  static constexpr int BIAS_OFF = V_OFF + 2 * NSP * KT;  // 2 stages
  static constexpr int P_OFF = BIAS_OFF + 2 * BIAS;      // 2 buffers x NSP copies
  static constexpr int BYTES = P_OFF + 2 * NSP * PT;
  static constexpr int TMEM_COLS = 256;  // O [0, DP), S0 [DP, DP+64), S1 [DP+64, DP+128)
};

// Lazy rescaling threshold (base-2 units): the running maximum used for the
// exponentials is only raised when a score exceeds it by more than this, so
// P stays <= 2^8 and the O accumulator is rarely rescaled.
constexpr float kRescaleThreshold = 8.0f;

__device__ __forceinline__ bool drain_wait(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_test(bar, parity)) {
    if (global_timer_ns() - t0 > ATTN_WAIT_TIMEOUT_NS) return false;
  }
  return true;
}

template <int DP, bool HAS_BIAS, bool SPLIT>
__global__ void __launch_bounds__(256, 1)
    fwd_stats_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_dy,
                     const __grid_constant__ CUtensorMap tm_bias, const __grid_constant__ CUtensorMap tm_q_lo,
                     const __grid_constant__ CUtensorMap tm_k_lo, const __grid_constant__ CUtensorMap tm_v_lo,
                     const __grid_constant__ CUtensorMap tm_dy_lo, const DenseParams p) {
  using L = FwdLayout<DP, SPLIT>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t bar_q, bar_dy, bar_full[2], bar_empty[2], bar_s_full[2], bar_p_full[2], bar_p_free[2];
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bh = blockIdx.x;
  const int b = bh / p.H, h = bh - b * p.H;
  const int nqt = cdiv(p.Sq, L::BQ);
  const int it = nqt - 1 - static_cast<int>(blockIdx.y);
  const int q0 = it * L::BQ;
  const int q1 = imin(q0 + L::BQ - 1, p.Sq - 1);
  int j_lo, j_hi;
  key_tile_range(p, q0, q1, L::BK, &j_lo, &j_hi);
  const int n = j_hi - j_lo;
  const Abort ab{&abort_flag, p.err};

  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bar_q, 1);
    mbar_init(&bar_dy, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bar_full[s], 1);
      mbar_init(&bar_empty[s], 1);
      mbar_init(&bar_s_full[s], 1);
      mbar_init(&bar_p_full[s], 4);
      mbar_init(&bar_p_free[s], 1);
    }
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
  const uint32_t t_o = tmem, t_s0 = tmem + DP;

  if (n > 0 && warp == 0) {
    if (lane == 0) {
      tma_prefetch_map(&tm_q);
      tma_prefetch_map(&tm_k);
      tma_prefetch_map(&tm_v);
      tma_prefetch_map(&tm_dy);
      if (HAS_BIAS) tma_prefetch_map(&tm_bias);
      mbar_arrive_expect_tx(&bar_q, L::NSP * L::QT);
      for (int hl = 0; hl < L::NSP; ++hl)
        for (int c = 0; c < L::NCH; ++c)
          tma_load_4d(sm + L::Q_OFF + hl * L::QT + c * (L::BQ * 128), hl ? &tm_q_lo : &tm_q, &bar_q, c * 64, q0, h,
                      b);
      int last_use[2] = {-1, -1};
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
        if (t == 0 && !p.fwd_only) {  // dY is only needed at the end; load it behind the first tile
          mbar_arrive_expect_tx(&bar_dy, L::NSP * L::QT);
          for (int hl = 0; hl < L::NSP; ++hl)
            for (int c = 0; c < L::NCH; ++c)
              tma_load_4d(sm + L::DY_OFF + hl * L::QT + c * (L::BQ * 128), hl ? &tm_dy_lo : &tm_dy, &bar_dy, c * 64,
                          q0, h, b);
        }
      }
      for (int s = 0; s < 2; ++s)
        if (last_use[s] >= 0) drain_wait(&bar_full[s], (last_use[s] >> 1) & 1);
      drain_wait(&bar_q, 0);
      if (last_use[0] >= 0 && !p.fwd_only) drain_wait(&bar_dy, 0);
    }
    __syncwarp();
  } else if (n > 0 && warp == 1) {
    if (lane == 0) {
      constexpr uint32_t id_s = idesc_bf16(128, 64, false, false);
      constexpr uint32_t id_o = idesc_bf16(128, DP, false, true);
      const uint32_t sQ = smem_addr(sm + L::Q_OFF);
      auto k_at = [&](int s) { return smem_addr(sm + L::K_OFF + s * L::NSP * L::KT); };
      auto v_at = [&](int s) { return smem_addr(sm + L::V_OFF + s * L::NSP * L::KT); };
      auto p_at = [&](int s) { return smem_addr(sm + L::P_OFF + s * L::NSP * L::PT); };
      constexpr int NPROD = SPLIT ? 3 : 1;  // hi*hi + hi*lo + lo*hi
      auto issue_s = [&](int t) {
        const int s = t & 1;
#pragma unroll
        for (int pr = 0; pr < NPROD; ++pr) {
          const uint32_t a0 = sQ + (pr == 2 ? L::QT : 0), b0 = k_at(s) + (pr == 1 ? L::KT : 0);
#pragma unroll
          for (int kk = 0; kk < DP / 16; ++kk) {
            const int c = kk >> 2, o = (kk & 3) * 32;
            const uint64_t ad = sdesc_sw128(a0 + c * (L::BQ * 128) + o, 16, 1024);
            const uint64_t bd = sdesc_sw128(b0 + c * (L::BK * 128) + o, 16, 1024);
            mma_bf16_ss(t_s0 + s * 64, ad, bd, id_s, (pr > 0 || kk > 0) ? 1u : 0u);
          }
        }
        mma_commit(&bar_s_full[s]);
      };
      bool ok = mbar_wait(&bar_q, 0, ab);
      if (ok) ok = mbar_wait(&bar_full[0], 0, ab);
      if (ok) {
        tc_fence_after();
        issue_s(0);
      }
      if (ok && n > 1) {
        ok = mbar_wait(&bar_full[1], 0, ab);
        if (ok) {
          tc_fence_after();
          issue_s(1);
        }
      }
      for (int t = 0; t < n && ok; ++t) {
        const int s = t & 1;
        if (!(ok = mbar_wait(&bar_p_full[s], (t >> 1) & 1, ab))) break;
        tc_fence_after();
#pragma unroll
        for (int pr = 0; pr < NPROD; ++pr) {
          const uint32_t a0 = p_at(s) + (pr == 2 ? L::PT : 0), b0 = v_at(s) + (pr == 1 ? L::KT : 0);
#pragma unroll
          for (int kk = 0; kk < L::BK / 16; ++kk) {
            const uint64_t ad = sdesc_sw128(a0 + kk * 32, 16, 1024);
            const uint64_t bd = sdesc_sw128(b0 + kk * 16 * 128, L::BK * 128, 1024);
            mma_bf16_ss(t_o, ad, bd, id_o, (t == 0 && pr == 0 && kk == 0) ? 0u : 1u);
          }
        }
        mma_commit(&bar_p_free[s]);
        mma_commit(&bar_empty[s]);
        if (t + 2 < n) {
          if (!(ok = mbar_wait(&bar_full[s], ((t + 2) >> 1) & 1, ab))) break;
          tc_fence_after();
          issue_s(t + 2);
        }
      }
      // the commit after the last O update already tracks every MMA; wait for it
      if (n > 0) drain_wait(&bar_p_free[(n - 1) & 1], ((n - 1) >> 1) & 1);
    }
    __syncwarp();
  } else if (warp >= 4) {
    const int lg = warp & 3;
    const int row = lg * 32 + lane;
    const int q = q0 + row;
    const uint32_t lane_addr = static_cast<uint32_t>(lg * 32) << 16;
    const float kInf = __int_as_float(0x7f800000);
    float m2 = -kInf, l = 0.f;
    bool any_unmasked = false;
    bool ok = n > 0;
    for (int t = 0; t < n && ok; ++t) {
      const int s = t & 1;
      const int kk0 = (j_lo + t) * L::BK;
      uint32_t kb0 = 0, kb1 = 0;
      if (p.has_key_mask) {
        const float* km = p.key_mask + static_cast<size_t>(b) * p.Sk;
        const int ka = kk0 + lane, kb = kk0 + 32 + lane;
        kb0 = __ballot_sync(0xffffffffu, ka < p.Sk && km[ka] < p.mask_thr);
        kb1 = __ballot_sync(0xffffffffu, kb < p.Sk && km[kb] < p.mask_thr);
      }
      if (!(ok = mbar_wait_warp(&bar_full[s], (t >> 1) & 1, ab))) break;
      if (!(ok = mbar_wait_warp(&bar_s_full[s], (t >> 1) & 1, ab))) break;
      tc_fence_after();
      float x[64];
      {
        uint32_t r0[32], r1[32];
        tmem_ld32(t_s0 + s * 64 + lane_addr, r0);
        tmem_ld32(t_s0 + s * 64 + lane_addr + 32, r1);
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          x[c] = __uint_as_float(r0[c]) * p.scale_log2;
          x[32 + c] = __uint_as_float(r1[c]) * p.scale_log2;
        }
      }
      if (HAS_BIAS) {
        const uint32_t bs = smem_addr(sm + L::BIAS_OFF + s * L::BIAS);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          uint32_t w0, w1, w2, w3;
          asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                       : "=r"(w0), "=r"(w1), "=r"(w2), "=r"(w3)
                       : "r"(bs + sw128_offset(row, j)));
          const uint32_t w[4] = {w0, w1, w2, w3};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            x[8 * j + 2 * e] = fmaf(__uint_as_float(w[e] << 16), kLog2e, x[8 * j + 2 * e]);
            x[8 * j + 2 * e + 1] = fmaf(__uint_as_float(w[e] & 0xffff0000u), kLog2e, x[8 * j + 2 * e + 1]);
          }
        }
      }
      const bool full = tile_fully_visible(p, q0, q0 + L::BQ - 1, kk0, kk0 + L::BK - 1);
      float mt = -kInf;
#pragma unroll
      for (int c = 0; c < 64; ++c) {
        const bool vis = full || pair_visible(p, q, kk0 + c);
        const bool masked = ((c < 32 ? kb0 >> c : kb1 >> (c - 32)) & 1u) != 0;
        if (masked) x[c] = p.masked_x2;
        if (!vis) x[c] = -kInf;
        any_unmasked |= vis && !masked;
        mt = fmaxf(mt, x[c]);
      }
      float alpha = 1.f;
      bool rescale = false;
      if (mt > m2 + kRescaleThreshold || (m2 == -kInf && mt > -kInf)) {
        if (m2 > -kInf) {
          alpha = ex2_approx(m2 - mt);
          rescale = true;
        }
        l *= alpha;
        m2 = mt;
      }
      float sum = 0.f;
      float pr[64];
#pragma unroll
      for (int c = 0; c < 64; ++c) {
        pr[c] = m2 > -kInf ? ex2_approx(x[c] - m2) : 0.f;
        sum += pr[c];
      }
      l += sum;
      // O rows scaled by alpha once every earlier O update has landed
      if (__any_sync(0xffffffffu, rescale) && t > 0) {
        const int ps = (t - 1) & 1;
        if (!(ok = mbar_wait_warp(&bar_p_free[ps], ((t - 1) >> 1) & 1, ab))) break;
        tc_fence_after();
        const float a = rescale ? alpha : 1.f;
#pragma unroll 1
        for (int cc = 0; cc < DP / 32; ++cc) {
          uint32_t r[32];
          tmem_ld32(t_o + lane_addr + cc * 32, r);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) * a);
          tmem_st32(t_o + lane_addr + cc * 32, r);
        }
        tmem_st_wait();
      }
      if (t >= 2 && !(ok = mbar_wait_warp(&bar_p_free[s], ((t - 2) >> 1) & 1, ab))) break;
      const uint32_t sp = smem_addr(sm + L::P_OFF + s * L::NSP * L::PT);
      store_row32<SPLIT>(sp, L::PT, row, 0, pr);
      store_row32<SPLIT>(sp, L::PT, row, 32, pr + 32);
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_p_full[s]);
    }
    float L2 = kInf, dl = 0.f, pm = 0.f;
    // forward export: O / l in the storage dtype (rows of the tile that exist)
    const int64_t o_row = static_cast<int64_t>(b) * p.s_o[2] + static_cast<int64_t>(h) * p.s_o[1] +
                          static_cast<int64_t>(q) * p.s_o[0];
    if (ok && n > 0) {
      ok = mbar_wait_warp(&bar_p_free[(n - 1) & 1], ((n - 1) >> 1) & 1, ab);
      if (ok && !p.fwd_only) ok = mbar_wait_warp(&bar_dy, 0, ab);
      tc_fence_after();
      if (ok) {
        // delta = dY . O / l, O read back from TMEM, dY from the swizzled tile
        float acc = 0.f;
        const uint8_t* dys = sm + L::DY_OFF;
        const float inv_l = l > 0.f ? 1.f / l : 0.f;
#pragma unroll 1
        for (int cc = 0; cc < DP / 32; ++cc) {
          uint32_t r[32];
          tmem_ld32(t_o + lane_addr + cc * 32, r);
          tmem_ld_wait();
          if (p.o_out && q < p.Sq) store_out32<SPLIT>(p.o_out, o_row, cc * 32, p.D, r, inv_l);
          if (p.fwd_only) continue;
#pragma unroll
          for (int hl = 0; hl < L::NSP; ++hl)  // dY = hi (+ lo for split fp32 inputs)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const int col = cc * 32 + j * 8;  // 8 bf16 per 16-byte chunk
              const uint4 w = *reinterpret_cast<const uint4*>(dys + hl * L::QT + (col >> 6) * (L::BQ * 128) +
                                                              sw128_offset(row, (col & 63) >> 3));
              const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                acc = fmaf(__uint_as_float(ws[e] << 16), __uint_as_float(r[8 * j + 2 * e]), acc);
                acc = fmaf(__uint_as_float(ws[e] & 0xffff0000u), __uint_as_float(r[8 * j + 2 * e + 1]), acc);
              }
            }
        }
        if (l > 0.f) {
          L2 = m2 + __log2f(l);
          dl = acc / l;
          if (p.has_key_mask) pm = any_unmasked ? ex2_approx(p.masked_x2 - L2) : 1.f / l;
        }
      }
    }
    if ((ok || n == 0) && q < p.Sq) {
      const size_t idx = static_cast<size_t>(bh) * p.Sq + q;
      p.L2[idx] = L2;
      p.delta[idx] = dl;
      if (p.has_key_mask) p.pm[idx] = pm;
      if (p.lse_out) p.lse_out[idx] = L2 < __int_as_float(0x7f800000) ? L2 * 0.6931471805599453f : -L2;
      if (p.o_out && n == 0) {
        uint32_t z[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) z[j] = 0u;
        for (int cc = 0; cc * 32 < p.D; ++cc) store_out32<SPLIT>(p.o_out, o_row, cc * 32, p.D, z, 0.f);
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
cudaError_t launch_fwd_t(const DenseMaps& m, const DenseParams& p, cudaStream_t s) {
  using L = FwdLayout<DP, SPLIT>;
  auto kern = fwd_stats_kernel<DP, HAS_BIAS, SPLIT>;
  const int smem = L::BYTES + 1024;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  dim3 grid(p.B * p.H, cdiv(p.Sq, L::BQ));
  kern<<<grid, 256, smem, s>>>(m.q128, m.k64, m.v64, m.dy128, m.bias128, m.q128_lo, m.k64_lo, m.v64_lo,
                               m.dy128_lo, p);
  return cudaGetLastError();
}

// x -> (hi, lo): hi = bf16(x), lo = bf16(x - hi), four elements per thread,
// for up to four tensors in one launch (jobs laid end to end in the index
// space of the grid-stride loop).
struct SplitJobs {
  const float* x[4];
  __nv_bfloat16* hi[4];
  __nv_bfloat16* lo[4];
  int64_t end4[4];  // cumulative element counts / 4
  int count;
};

__global__ void split_f32_kernel(const SplitJobs jobs) {
  const int64_t total = jobs.end4[jobs.count - 1];
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    int j = 0;
    while (i >= jobs.end4[j]) ++j;
    const int64_t k = i - (j > 0 ? jobs.end4[j - 1] : 0);
    const float4 v = reinterpret_cast<const float4*>(jobs.x[j])[k];
    const __nv_bfloat162 h0 = __floats2bfloat162_rn(v.x, v.y), h1 = __floats2bfloat162_rn(v.z, v.w);
    const __nv_bfloat162 l0 = __floats2bfloat162_rn(v.x - __low2float(h0), v.y - __high2float(h0));
    const __nv_bfloat162 l1 = __floats2bfloat162_rn(v.z - __low2float(h1), v.w - __high2float(h1));
    reinterpret_cast<__nv_bfloat162*>(jobs.hi[j])[2 * k] = h0;
    reinterpret_cast<__nv_bfloat162*>(jobs.hi[j])[2 * k + 1] = h1;
    reinterpret_cast<__nv_bfloat162*>(jobs.lo[j])[2 * k] = l0;
    reinterpret_cast<__nv_bfloat162*>(jobs.lo[j])[2 * k + 1] = l1;
  }
}

// One warp per query row: delta = dY . O, L2 from the supplied LSE.
template <typename T>
__global__ void __launch_bounds__(256) delta_only_kernel(const DenseParams p) {
  const int64_t rows = static_cast<int64_t>(p.B) * p.H * p.Sq;
  const int lane = threadIdx.x & 31;
  const int64_t w0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nw = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const float kInf = __int_as_float(0x7f800000);
  for (int64_t r = w0; r < rows; r += nw) {
    const int q = static_cast<int>(r % p.Sq);
    const int64_t bh = r / p.Sq;
    const int h = static_cast<int>(bh % p.H), b = static_cast<int>(bh / p.H);
    const T* dy = reinterpret_cast<const T*>(p.dy) + b * p.s_dy[2] + h * p.s_dy[1] + static_cast<int64_t>(q) * p.s_dy[0];
    const T* o = reinterpret_cast<const T*>(p.o) + b * p.s_o[2] + h * p.s_o[1] + static_cast<int64_t>(q) * p.s_o[0];
    float acc = 0.f;
    for (int d = lane; d < p.D; d += 32) acc = fmaf(static_cast<float>(dy[d]), static_cast<float>(o[d]), acc);
#pragma unroll
    for (int sft = 16; sft > 0; sft >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, sft);
    if (lane == 0) {
      const float lse = p.lse[r];
      const int nvis = visible_keys(p, q);
      const bool empty = nvis == 0 || lse == -kInf;
      p.L2[r] = empty ? kInf : lse * kLog2e;
      p.delta[r] = empty ? 0.f : acc;
      if (p.has_custom) {
        // a row whose visible keys are all custom-masked has LSE = mask_neg +
        // log(n), which rounds to mask_neg when |mask_neg| is large
        float pm = 0.f;
        if (!empty) pm = (lse == p.mask_neg) ? 1.f / static_cast<float>(nvis) : ex2_approx((p.mask_neg - lse) * kLog2e);
        p.pm[r] = pm;
      }
    }
  }
}

// The same per row with 16-byte loads: LPR lanes (a power of two, at most 32)
// share a row, lane l of the row reading elements [V l, V l + V), [V (l +
// LPR), ...) of dY and O (V = 16 bytes of T), so a warp covers 32 / LPR rows
// at a time.  Used when the rows start 16-byte aligned and D is a multiple of
// V (the launcher checks); the sums then run in another order than the scalar
// kernel's, which does not change what the library guarantees (one writer per
// row, the same order from run to run).
template <typename T, int LPR>
__global__ void __launch_bounds__(256) delta_only_vec_kernel(const DenseParams p) {
  constexpr int V = 16 / static_cast<int>(sizeof(T));
  constexpr int RPW = 32 / LPR;  // rows per warp at a time
  const int64_t rows = static_cast<int64_t>(p.B) * p.H * p.Sq;
  const int lane = threadIdx.x & 31, sub = lane % LPR;
  const int64_t w0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nw = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const float kInf = __int_as_float(0x7f800000);
  const int nv = p.D / V;  // 16-byte vectors per row
  for (int64_t r0 = w0 * RPW; r0 < rows; r0 += nw * RPW) {
    const int64_t r = r0 + lane / LPR;
    const bool valid = r < rows;
    float acc = 0.f;
    // 32-bit row arithmetic (the launcher takes this kernel only for fewer
    // than 2^31 rows): a 64-bit division per row made the kernel issue-bound
    const uint32_t ru = static_cast<uint32_t>(r), sq = static_cast<uint32_t>(p.Sq);
    const int q = static_cast<int>(ru % sq);
    // the row's LSE is loaded beside dY and O, not after the reduction
    const float lse = (valid && sub == 0) ? p.lse[r] : 0.f;
    if (valid) {
      const uint32_t bh = ru / sq;
      const int h = static_cast<int>(bh % static_cast<uint32_t>(p.H)), b = static_cast<int>(bh / static_cast<uint32_t>(p.H));
      const T* dy = reinterpret_cast<const T*>(p.dy) + b * p.s_dy[2] + h * p.s_dy[1] + static_cast<int64_t>(q) * p.s_dy[0];
      const T* o = reinterpret_cast<const T*>(p.o) + b * p.s_o[2] + h * p.s_o[1] + static_cast<int64_t>(q) * p.s_o[0];
      for (int c = sub; c < nv; c += LPR) {
        const uint4 a = *reinterpret_cast<const uint4*>(dy + c * V);
        const uint4 e = *reinterpret_cast<const uint4*>(o + c * V);
        const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, ew[4] = {e.x, e.y, e.z, e.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          if (sizeof(T) == 2) {
            acc = fmaf(__uint_as_float(aw[i] << 16), __uint_as_float(ew[i] << 16), acc);
            acc = fmaf(__uint_as_float(aw[i] & 0xffff0000u), __uint_as_float(ew[i] & 0xffff0000u), acc);
          } else {
            acc = fmaf(__uint_as_float(aw[i]), __uint_as_float(ew[i]), acc);
          }
        }
      }
    }
#pragma unroll
    for (int sft = LPR / 2; sft > 0; sft >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, sft);
    if (valid && sub == 0) {
      const int nvis = visible_keys(p, q);
      const bool empty = nvis == 0 || lse == -kInf;
      p.L2[r] = empty ? kInf : lse * kLog2e;
      p.delta[r] = empty ? 0.f : acc;
      if (p.has_custom) {
        float pm = 0.f;
        if (!empty) pm = (lse == p.mask_neg) ? 1.f / static_cast<float>(nvis) : ex2_approx((p.mask_neg - lse) * kLog2e);
        p.pm[r] = pm;
      }
    }
  }
}

}  // namespace

cudaError_t launch_fwd_stats(const DenseMaps& m, const DenseParams& p, bool bias, cudaStream_t s) {
  const int DP = padded_head_dim(p.D);
  if (m.split) return launch_fwd_t<64, false, true>(m, p, s);
  if (DP == 64) return bias ? launch_fwd_t<64, true, false>(m, p, s) : launch_fwd_t<64, false, false>(m, p, s);
  return bias ? launch_fwd_t<128, true, false>(m, p, s) : launch_fwd_t<128, false, false>(m, p, s);
}

cudaError_t launch_split_f32(const float* const x[4], void* const hi[4], void* const lo[4], const int64_t n[4],
                             cudaStream_t s) {
  SplitJobs jobs{};
  int64_t acc = 0;
  for (int i = 0; i < 4; ++i) {
    if (n[i] <= 0) continue;
    jobs.x[jobs.count] = x[i];
    jobs.hi[jobs.count] = static_cast<__nv_bfloat16*>(hi[i]);
    jobs.lo[jobs.count] = static_cast<__nv_bfloat16*>(lo[i]);
    acc += n[i] / 4;
    jobs.end4[jobs.count] = acc;
    ++jobs.count;
  }
  if (jobs.count == 0 || acc == 0) return cudaSuccess;
  const int64_t blocks = (acc + 255) / 256;
  split_f32_kernel<<<static_cast<int>(blocks < 152 * 16 ? blocks : 152 * 16), 256, 0, s>>>(jobs);
  return cudaGetLastError();
}

namespace {
__global__ void fill_f32_kernel(float* x, float value, int64_t n) {
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    x[i] = value;
}
}  // namespace

namespace {
// zero D elements of es bytes at every (b, s, h) row of a strided tensor
__global__ void zero_rows_kernel(uint8_t* x, int64_t sb, int64_t ss, int64_t sh, int64_t B, int64_t S, int64_t H,
                                 int64_t D, int64_t es) {
  const int64_t rows = B * S * H, row_bytes = D * es;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < rows * row_bytes;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = i / row_bytes, byte = i - r * row_bytes;
    const int64_t h = r % H, sq = (r / H) % S, b = r / (H * S);
    x[(b * sb + sq * ss + h * sh) * es + byte] = 0;
  }
}
}  // namespace

cudaError_t launch_zero_rows(void* x, int64_t sb, int64_t ss, int64_t sh, int64_t B, int64_t S, int64_t H, int64_t D,
                             size_t es, cudaStream_t s) {
  if (!x || B * S * H * D == 0) return cudaSuccess;
  zero_rows_kernel<<<152 * 4, 256, 0, s>>>(static_cast<uint8_t*>(x), sb, ss, sh, B, S, H, D, int64_t(es));
  return cudaGetLastError();
}

namespace {
// The per-element mask as bits, in both orientations: one warp per 32 x 32
// block of (query, key) pairs, lane = key; the ballot over a query row gives
// its row word, and each lane gathers its key's column word over the rows.
__global__ void pack_elem_mask_kernel(const float* __restrict__ m, float thr, int64_t BH, int Sq, int Sk,
                                      uint32_t* rows, uint32_t* cols, int ew_q, int ew_k) {
  const int lane = threadIdx.x & 31;
  const int nqt = (Sq + 31) / 32, nkt = (Sk + 31) / 32;
  const int64_t blocks = BH * nqt * nkt;
  for (int64_t w = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; w < blocks;
       w += (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5) {
    const int kt = static_cast<int>(w % nkt), qt = static_cast<int>((w / nkt) % nqt);
    const int64_t bh = w / (static_cast<int64_t>(nkt) * nqt);
    const int k = kt * 32 + lane;
    uint32_t colword = 0u;
    for (int i = 0; i < 32; ++i) {
      const int q = qt * 32 + i;
      const bool in = q < Sq && k < Sk;
      const bool masked = in && m[(bh * Sq + q) * Sk + k] < thr;
      const uint32_t rowword = __ballot_sync(0xffffffffu, masked);
      if (lane == 0 && q < Sq) {
        rows[(bh * Sq + q) * ew_q + kt] = rowword;
        if (kt == nkt - 1 && nkt < ew_q) rows[(bh * Sq + q) * ew_q + kt + 1] = 0u;  // even-width padding
      }
      colword |= (masked ? 1u : 0u) << i;
    }
    if (k < Sk) {
      cols[(bh * Sk + k) * ew_k + qt] = colword;
      if (qt == nqt - 1 && nqt < ew_k) cols[(bh * Sk + k) * ew_k + qt + 1] = 0u;
    }
  }
}
}  // namespace

cudaError_t launch_pack_elem_mask(const float* m, float thr, int64_t BH, int Sq, int Sk, uint32_t* rows,
                                  uint32_t* cols, int ew_q, int ew_k, cudaStream_t s) {
  if (BH == 0 || Sq == 0 || Sk == 0) return cudaSuccess;
  pack_elem_mask_kernel<<<152 * 8, 256, 0, s>>>(m, thr, BH, Sq, Sk, rows, cols, ew_q, ew_k);
  return cudaGetLastError();
}

cudaError_t launch_fill_f32(float* x, float value, int64_t n, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  const int64_t blocks = (n + 255) / 256;
  fill_f32_kernel<<<static_cast<int>(blocks < 152 * 8 ? blocks : 152 * 8), 256, 0, s>>>(x, value, n);
  return cudaGetLastError();
}

cudaError_t launch_delta_only(const DenseParams& p, int dtype_bf16, cudaStream_t s) {
  const int64_t rows = static_cast<int64_t>(p.B) * p.H * p.Sq;
  if (rows == 0) return cudaSuccess;
  // 16-byte loads when every row of dY and O starts 16-byte aligned and D is
  // a multiple of 16 bytes of elements
  const int es = dtype_bf16 ? 2 : 4, V = 16 / es;
  auto a16 = [](const void* x, const int64_t* st, int es_) {
    return (reinterpret_cast<uintptr_t>(x) & 15u) == 0 && (st[0] * es_) % 16 == 0 && (st[1] * es_) % 16 == 0 &&
           (st[2] * es_) % 16 == 0;
  };
  if (p.D % V == 0 && rows < (int64_t(1) << 31) && a16(p.dy, p.s_dy, es) && a16(p.o, p.s_o, es)) {
    const int nv = p.D / V;
    const int lpr = nv >= 32 ? 32 : nv >= 16 ? 16 : nv >= 8 ? 8 : nv >= 4 ? 4 : nv >= 2 ? 2 : 1;
    const int64_t warps = (rows * lpr + 31) / 32;
    const int64_t b64 = (warps * 32 + 255) / 256;
    const int blocks = static_cast<int>(b64 < 152 * 16 ? b64 : 152 * 16);
#define ATTN_DELTA_VEC(T_, L_) delta_only_vec_kernel<T_, L_><<<blocks, 256, 0, s>>>(p)
    if (dtype_bf16) {
      switch (lpr) {
        case 32: ATTN_DELTA_VEC(__nv_bfloat16, 32); break;
        case 16: ATTN_DELTA_VEC(__nv_bfloat16, 16); break;
        case 8: ATTN_DELTA_VEC(__nv_bfloat16, 8); break;
        case 4: ATTN_DELTA_VEC(__nv_bfloat16, 4); break;
        case 2: ATTN_DELTA_VEC(__nv_bfloat16, 2); break;
        default: ATTN_DELTA_VEC(__nv_bfloat16, 1); break;
      }
    } else {
      switch (lpr) {
        case 32: ATTN_DELTA_VEC(float, 32); break;
        case 16: ATTN_DELTA_VEC(float, 16); break;
        case 8: ATTN_DELTA_VEC(float, 8); break;
        case 4: ATTN_DELTA_VEC(float, 4); break;
        case 2: ATTN_DELTA_VEC(float, 2); break;
        default: ATTN_DELTA_VEC(float, 1); break;
      }
    }
#undef ATTN_DELTA_VEC
    return cudaGetLastError();
  }
  const int64_t blocks64 = (rows * 32 + 255) / 256;
  const int blocks = static_cast<int>(blocks64 < 152 * 64 ? blocks64 : 152 * 64);
  if (dtype_bf16)
    delta_only_kernel<__nv_bfloat16><<<blocks, 256, 0, s>>>(p);
  else
    delta_only_kernel<float><<<blocks, 256, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace attn
