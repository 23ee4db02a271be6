// Paged row statistics: lse[r, h] and delta[r, h] = dY . O for every packed
// query row and head, by a forward sweep over the row's sequence pages.
//
// ruDNN src/paged_attention/ordered_kernel.rs reads per (row, head) the
// statistics "computed once by the query kernel" (max, denominator, delta);
// this kernel produces them in LSE form.  One CTA per (tile of 128 columns =
// 128/G query rows x the G heads of a KV group, sequence, KV head): S = Q K^T
// on tcgen05 (M = 128 columns, N = 64 tokens = four pages gathered by TMA),
// online softmax in registers (thread = column), O += P V on tcgen05, then
// delta = dY . O / l and lse = (max + log2 l) / log2(e).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "paged_common.cuh"
#include "paged_launch.h"
#include "sm103.cuh"

namespace attn {
using namespace sm103;

namespace {

template <int DP>
struct StatLayout {
  static constexpr int NCH = DP / 64;
  static constexpr int BQ = 128, BK = 64;
  static constexpr int QT = NCH * BQ * 128;
  static constexpr int KT = NCH * BK * 128;
  static constexpr int PT = BQ * 128;
  static constexpr int Q_OFF = 0;
  static constexpr int DY_OFF = Q_OFF + QT;
  // K/V stages: 4 at D = 128 (one CTA per SM either way); 2 at D = 64,
  // where the smaller layout lets two CTAs share an SM
  static constexpr int KS = DP == 64 ? 2 : 4;
  static constexpr int K_OFF = DY_OFF + QT;        // KS stages
  static constexpr int V_OFF = K_OFF + KS * KT;    // KS stages
  static constexpr int P_OFF = V_OFF + KS * KT;    // 2 buffers
  static constexpr int BYTES = P_OFF + 2 * PT;
  static constexpr int TMEM_COLS = 256;
  // dynamic shared memory starts 1024-aligned after the static variables
  // (one 1 KiB granule): no alignment pad, checked at run time
  static_assert(BYTES + 1024 <= 232448, "the layout fits one CTA's shared memory");
};

constexpr float kRescaleThreshold = 8.0f;

__device__ __forceinline__ bool drain_wait(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_test(bar, parity)) {
    if (global_timer_ns() - t0 > ATTN_WAIT_TIMEOUT_NS) return false;
  }
  return true;
}

template <int DP>
__global__ void __launch_bounds__(256, 1)
    paged_stats_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_dy,
                       const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                       const PagedParams p) {
  using L = StatLayout<DP>;
  constexpr int KS = L::KS;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = smem_raw;
  __shared__ uint64_t bar_q, bar_dy, bar_full[KS], bar_empty[KS], bar_s_full[2], bar_p_full[2], bar_p_free[2];
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag;
  __shared__ int max_pos_sh;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __shared__ int tile_sq_sh, tile_r0_sh;
  // block x = tile * KVH + g: row tile `tile` of the sequences in dispatch
  // order (longest first), KV head g
  const int g = static_cast<int>(blockIdx.x % p.KVH);
  const int RT = L::BQ / p.G;  // query rows per tile
  if (threadIdx.x < 32) {  // warp 0
    int sq_, r0_;
    row_tile_at_warp(p, static_cast<int>(blockIdx.x / p.KVH), RT, &sq_, &r0_);
    if (threadIdx.x == 0) {
      tile_sq_sh = sq_;
      tile_r0_sh = r0_;
    }
  }
  __syncthreads();
  const int sq = tile_sq_sh, r0 = tile_r0_sh;
  if (sq < 0) return;  // uniform exit: past the last row tile
  if (smem_addr(smem_raw) & 1023u) {  // uniform: the swizzled tiles need 1024-byte alignment
    if (threadIdx.x == 0 && p.err) atomicOr(p.err, DEV_ERR_LAYOUT);
    return;
  }
  const int r_end = row_end_of(p, sq);
  const int len = seq_len_of(p, sq);
  const int npg = pages_of(len, p.page_size);
  const Abort ab{&abort_flag, p.err};

  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bar_q, 1);
    mbar_init(&bar_dy, 1);
    for (int s = 0; s < KS; ++s) {
      mbar_init(&bar_full[s], 1);
      mbar_init(&bar_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bar_s_full[s], 1);
      mbar_init(&bar_p_full[s], 4);
      mbar_init(&bar_p_free[s], 1);
    }
    mbar_fence_init();
    int mp = -1;
    for (int r = r0; r < r_end && r < r0 + RT; ++r) mp = max(mp, p.causal ? p.q_pos[r] : len - 1);
    max_pos_sh = mp;
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
  // token tiles that can be visible: tokens <= max position, < len
  const int last_tok = min(len - 1, max_pos_sh);
  const int n = last_tok < 0 ? 0 : last_tok / L::BK + 1;
  const int oob_slot = p.num_pages * p.page_size;

  if (n > 0 && warp == 0) {
    if (lane == 0) {
      tma_prefetch_map(&tm_q);
      tma_prefetch_map(&tm_dy);
      tma_prefetch_map(&tm_k);
      tma_prefetch_map(&tm_v);
      mbar_arrive_expect_tx(&bar_q, L::QT);
      for (int c = 0; c < L::NCH; ++c)
        tma_load_3d(sm + L::Q_OFF + c * (L::BQ * 128), &tm_q, &bar_q, c * 64, g * p.G, r0);
      int last_use[KS];
      for (int i = 0; i < KS; ++i) last_use[i] = -1;
      bool ok = true;
      for (int t = 0; t < n && ok; ++t) {
        const int s = t % KS;
        if (t >= KS) ok = mbar_wait(&bar_empty[s], ((t / KS) - 1) & 1, ab);
        if (!ok) break;
        mbar_arrive_expect_tx(&bar_full[s], 2 * L::KT);
        for (int i = 0; i < L::BK / 16; ++i) {
          const int lp = t * (L::BK / 16) + i;
          int slot = oob_slot;
          if (lp < npg) {
            const int ph = p.page_table[static_cast<int64_t>(sq) * p.max_pages + lp];
            if (ph >= 0 && ph < p.num_pages) slot = ph * p.page_size;
          }
          for (int c = 0; c < L::NCH; ++c) {
            tma_load_3d(sm + L::K_OFF + s * L::KT + c * (L::BK * 128) + i * 16 * 128, &tm_k, &bar_full[s], c * 64,
                        g, slot);
            tma_load_3d(sm + L::V_OFF + s * L::KT + c * (L::BK * 128) + i * 16 * 128, &tm_v, &bar_full[s], c * 64,
                        g, slot);
          }
        }
        last_use[s] = t;
        if (t == 0) {
          mbar_arrive_expect_tx(&bar_dy, L::QT);
          for (int c = 0; c < L::NCH; ++c)
            tma_load_3d(sm + L::DY_OFF + c * (L::BQ * 128), &tm_dy, &bar_dy, c * 64, g * p.G, r0);
        }
      }
      for (int s = 0; s < KS; ++s)
        if (last_use[s] >= 0) drain_wait(&bar_full[s], (last_use[s] / KS) & 1);
      drain_wait(&bar_q, 0);
      if (last_use[0] >= 0) drain_wait(&bar_dy, 0);
    }
    __syncwarp();
  } else if (n > 0 && warp == 1) {
    if (lane == 0) {
      constexpr uint32_t id_s = idesc_bf16(128, 64, false, false);
      constexpr uint32_t id_o = idesc_bf16(128, DP, false, true);
      const uint32_t sQ = smem_addr(sm + L::Q_OFF);
      auto k_at = [&](int s) { return smem_addr(sm + L::K_OFF + s * L::KT); };
      auto v_at = [&](int s) { return smem_addr(sm + L::V_OFF + s * L::KT); };
      auto p_at = [&](int s) { return smem_addr(sm + L::P_OFF + s * L::PT); };
      // S(t) into S buffer t & 1 from K stage t mod KS
      auto issue_s = [&](int t) {
        const int s = t & 1, ks = t % KS;
#pragma unroll
        for (int kk = 0; kk < DP / 16; ++kk) {
          const int c = kk >> 2, o = (kk & 3) * 32;
          const uint64_t ad = sdesc_sw128(sQ + c * (L::BQ * 128) + o, 16, 1024);
          const uint64_t bd = sdesc_sw128(k_at(ks) + c * (L::BK * 128) + o, 16, 1024);
          mma_bf16_ss(t_s0 + s * 64, ad, bd, id_s, kk > 0 ? 1u : 0u);
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
        const int s = t & 1, ks = t % KS;
        if (!(ok = mbar_wait(&bar_p_full[s], (t >> 1) & 1, ab))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < L::BK / 16; ++kk) {
          const uint64_t ad = sdesc_sw128(p_at(s) + kk * 32, 16, 1024);
          const uint64_t bd = sdesc_sw128(v_at(ks) + kk * 16 * 128, L::BK * 128, 1024);
          mma_bf16_ss(t_o, ad, bd, id_o, (t == 0 && kk == 0) ? 0u : 1u);
        }
        mma_commit(&bar_p_free[s]);
        mma_commit(&bar_empty[ks]);
        if (t + 2 < n) {
          const int k2 = (t + 2) % KS;
          if (!(ok = mbar_wait(&bar_full[k2], ((t + 2) / KS) & 1, ab))) break;
          tc_fence_after();
          issue_s(t + 2);
        }
      }
      if (n > 0) drain_wait(&bar_p_free[(n - 1) & 1], ((n - 1) >> 1) & 1);
    }
    __syncwarp();
  } else if (warp >= 4) {
    const int lg = warp & 3;
    const int col = lg * 32 + lane;          // column = (row, head) pair == TMEM lane
    const int r = r0 + col / p.G;
    const int hh = g * p.G + col % p.G;
    const bool col_ok = r < r_end;
    const int pos = col_ok ? (p.causal ? p.q_pos[r] : len - 1) : -1;
    const uint32_t lane_addr = static_cast<uint32_t>(lg * 32) << 16;
    const float kInf = __int_as_float(0x7f800000);
    float m2 = -kInf, l = 0.f;
    bool ok = n > 0;
    for (int t = 0; t < n && ok; ++t) {
      const int s = t & 1;
      const int tk0 = t * L::BK;
      if (!(ok = mbar_wait_warp(&bar_s_full[s], (t >> 1) & 1, ab))) break;
      tc_fence_after();
      float x[64];
      {
        uint32_t a0[32], a1[32];
        tmem_ld32(t_s0 + s * 64 + lane_addr, a0);
        tmem_ld32(t_s0 + s * 64 + lane_addr + 32, a1);
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          x[c] = __uint_as_float(a0[c]) * p.scale_log2;
          x[32 + c] = __uint_as_float(a1[c]) * p.scale_log2;
        }
      }
      float mt = -kInf;
#pragma unroll
      for (int c = 0; c < 64; ++c) {
        const int tok = tk0 + c;
        if (!(tok < len && tok <= pos)) x[c] = -kInf;
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
      float pr[64];
      float sum = 0.f;
#pragma unroll
      for (int c = 0; c < 64; ++c) {
        pr[c] = m2 > -kInf ? ex2_approx(x[c] - m2) : 0.f;
        sum += pr[c];
      }
      l += sum;
      if (__any_sync(0xffffffffu, rescale) && t > 0) {
        const int ps = (t - 1) & 1;
        if (!(ok = mbar_wait_warp(&bar_p_free[ps], ((t - 1) >> 1) & 1, ab))) break;
        tc_fence_after();
        const float a = rescale ? alpha : 1.f;
#pragma unroll 1
        for (int cc = 0; cc < DP / 32; ++cc) {
          uint32_t rr[32];
          tmem_ld32(t_o + lane_addr + cc * 32, rr);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 32; ++j) rr[j] = __float_as_uint(__uint_as_float(rr[j]) * a);
          tmem_st32(t_o + lane_addr + cc * 32, rr);
        }
        tmem_st_wait();
      }
      // Slots past the sequence's length inside its last page may hold any bit
      // pattern (NaN included); the tensor core would turn 0 * NaN into NaN in
      // O += P V, so their V rows are zeroed before the product reads them.
      if (tk0 + L::BK > len) {
        // the stage's copies have landed (observed here, not only by the MMA thread)
        if (!(ok = mbar_wait_warp(&bar_full[t % KS], (t / KS) & 1, ab))) break;
        const int row_lo = max(0, len - tk0);
        const int nvec = (L::BK - row_lo) * L::NCH * 8;
        uint8_t* vt = sm + L::V_OFF + (t % KS) * L::KT;
        for (int i = threadIdx.x - 128; i < nvec; i += 128) {
          const int rw = row_lo + i / (L::NCH * 8), rem = i % (L::NCH * 8);
          const int ch = rem >> 3, seg = rem & 7;
          st_shared_v4(smem_addr(vt + ch * (L::BK * 128) + rw * 128 + seg * 16), 0u, 0u, 0u, 0u);
        }
      }
      if (t >= 2 && !(ok = mbar_wait_warp(&bar_p_free[s], ((t - 2) >> 1) & 1, ab))) break;
      const uint32_t sp = smem_addr(sm + L::P_OFF + s * L::PT);
#pragma unroll
      for (int j = 0; j < 8; ++j)
        st_shared_v4(sp + sw128_offset(col, j), pack_bf16x2(pr[8 * j], pr[8 * j + 1]),
                     pack_bf16x2(pr[8 * j + 2], pr[8 * j + 3]), pack_bf16x2(pr[8 * j + 4], pr[8 * j + 5]),
                     pack_bf16x2(pr[8 * j + 6], pr[8 * j + 7]));
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_p_full[s]);
    }
    float lse = -kInf, dl = 0.f;
    if (ok && n > 0) {
      ok = mbar_wait_warp(&bar_p_free[(n - 1) & 1], ((n - 1) >> 1) & 1, ab);
      if (ok) ok = mbar_wait_warp(&bar_dy, 0, ab);
      tc_fence_after();
      if (ok) {
        float acc = 0.f;
        const uint8_t* dys = sm + L::DY_OFF;
#pragma unroll 1
        for (int cc = 0; cc < DP / 32; ++cc) {
          uint32_t rr[32];
          tmem_ld32(t_o + lane_addr + cc * 32, rr);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int cl = cc * 32 + j * 8;
            const uint4 w = *reinterpret_cast<const uint4*>(dys + (cl >> 6) * (L::BQ * 128) +
                                                            sw128_offset(col, (cl & 63) >> 3));
            const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              acc = fmaf(__uint_as_float(ws[e] << 16), __uint_as_float(rr[8 * j + 2 * e]), acc);
              acc = fmaf(__uint_as_float(ws[e] & 0xffff0000u), __uint_as_float(rr[8 * j + 2 * e + 1]), acc);
            }
          }
        }
        if (l > 0.f) {
          lse = (m2 + __log2f(l)) * 0.6931471805599453f;
          dl = acc / l;
        }
      }
    }
    if ((ok || n == 0) && col_ok) {
      const int64_t idx = static_cast<int64_t>(r) * p.H + hh;
      p.lse_out[idx] = lse;
      p.delta_out[idx] = dl;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, L::TMEM_COLS);
  }
}

template <int DP>
cudaError_t launch_stats_t(const PagedMaps& m, const PagedParams& p, cudaStream_t s) {
  using L = StatLayout<DP>;
  auto kern = paged_stats_kernel<DP>;
  const int smem = L::BYTES;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int rt = L::BQ / p.G;
  // row tiles: at most Nq / rt + S (one partial tile per sequence)
  dim3 grid(static_cast<unsigned>((static_cast<int64_t>(p.Nq) / rt + p.S + 1) * p.KVH));
  kern<<<grid, 256, smem, s>>>(m.q_stats, m.dy_stats, m.k, m.v, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_paged_row_stats(const PagedMaps& m, const PagedParams& p, cudaStream_t s) {
  if (p.S == 0 || p.Nq == 0) return cudaSuccess;
  if (p.Dk <= 64) return launch_stats_t<64>(m, p, s);
  return launch_stats_t<128>(m, p, s);
}

}  // namespace attn
