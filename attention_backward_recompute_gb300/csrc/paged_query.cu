// Query side of the paged backward (GQA): the row statistics and dQ of every
// packed query row and head.
//
// ruDNN src/paged_attention/ordered_kernel.rs reads per (row, head) the
// statistics "computed once by the query kernel" and leaves the query
// gradient to that kernel.  This kernel is it: one CTA per (tile of 128
// columns = 128/G query rows x the G heads of a KV group, sequence, KV head)
// sweeps the row's sequence twice over the same 64-token tiles (four 16-token
// pages gathered by TMA), in increasing token order:
//   sweep 1 (forward):   S = Q K^T, online softmax (thread = column),
//                        O += P V; then lse = max + log l and delta = dY.O / l
//   sweep 2 (gradient):  S = Q K^T and dP = dY V^T again,
//                        P = exp(S*scale - lse), dS = P (dP - delta),
//                        dQ += dS K
// and stores dQ = scale * dQ once per (row, head): atomic-free and bit-stable.
// A column with no visible token gets lse = -inf, delta = 0 and dQ = 0.
//
// Warp 0: TMA producer (Q, dY once; K and V tiles through a 2-stage ring for
// both sweeps), warp 1: MMA issuer (one thread), warps 4..7: one thread per
// column.  P (sweep 1) and dS (sweep 2) go to shared memory as bf16 and are
// the A operand of O += P V and dQ += dS K.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "paged_common.cuh"
#include "paged_launch.h"
#include "sm103.cuh"

namespace attn {
using namespace sm103;

namespace {

template <int DP>
struct QueryLayout {
  static constexpr int NCH = DP / 64;
  static constexpr int BQ = 128, BK = 64;
  static constexpr int QT = NCH * BQ * 128;
  static constexpr int KT = NCH * BK * 128;
  static constexpr int PT = BQ * 128;
  static constexpr int Q_OFF = 0;
  static constexpr int DY_OFF = Q_OFF + QT;
  static constexpr int KS = DP == 64 ? 2 : 4;   // K/V stages
  static constexpr int K_OFF = DY_OFF + QT;     // KS stages
  static constexpr int V_OFF = K_OFF + KS * KT; // KS stages
  static constexpr int P_OFF = V_OFF + KS * KT; // 2 buffers: P (sweep 1), dS (sweep 2)
  static constexpr int BYTES = P_OFF + 2 * PT;
  // dynamic shared memory starts 1024-aligned after the static variables
  // (one 1 KiB granule): no alignment pad, checked at run time
  static_assert(BYTES + 1024 <= 232448, "the layout fits one CTA's shared memory");
  // TMEM: O [0, 128), dQ [128, 256), S[2] [256, 384), dP[2] [384, 512)
  static constexpr int T_O = 0, T_DQ = 128, T_S = 256, T_DP = 384, TMEM_COLS = 512;
};

constexpr float kRescaleThreshold = 8.0f;

__device__ __forceinline__ bool drain_wait(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_test(bar, parity)) {
    if (global_timer_ns() - t0 > ATTN_WAIT_TIMEOUT_NS) return false;
  }
  return true;
}

// Zeroes, in a K or V stage, the rows of tokens at or past the sequence's
// length: slots past the length inside the last page may hold any bit pattern
// (NaN included), and the tensor core would turn 0 * NaN into NaN in a
// product that reads them.  Threads 128..255 share the work.
template <int DP>
__device__ __forceinline__ void zero_tail_rows(uint8_t* tile, int row_lo) {
  using L = QueryLayout<DP>;
  const int nvec = (L::BK - row_lo) * L::NCH * 8;
  for (int i = static_cast<int>(threadIdx.x) - 128; i < nvec; i += 128) {
    const int rw = row_lo + i / (L::NCH * 8), rem = i % (L::NCH * 8);
    const int ch = rem >> 3, seg = rem & 7;
    st_shared_v4(smem_addr(tile + ch * (L::BK * 128) + rw * 128 + seg * 16), 0u, 0u, 0u, 0u);
  }
}

template <int DP>
__global__ void __launch_bounds__(256, 1)
    paged_query_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_dy,
                       const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                       const PagedParams p) {
  using L = QueryLayout<DP>;
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
  // token tiles that can be visible: tokens <= max position, < len
  const int last_tok = min(len - 1, max_pos_sh);
  const int n = last_tok < 0 ? 0 : last_tok / L::BK + 1;
  const int NT = 2 * n;  // tiles of both sweeps; tile t covers token tile t mod n
  const int oob_slot = p.num_pages * p.page_size;

  if (n > 0 && warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_map(&tm_q);
      tma_prefetch_map(&tm_dy);
      tma_prefetch_map(&tm_k);
      tma_prefetch_map(&tm_v);
      mbar_arrive_expect_tx(&bar_q, L::QT);
      for (int c = 0; c < L::NCH; ++c)
        tma_load_3d(sm + L::Q_OFF + c * (L::BQ * 128), &tm_q, &bar_q, c * 64, g * p.G, r0);
      bool ok = true;
      for (int t = 0; t < NT && ok; ++t) {
        const int s = t % KS;
        const int u = t < n ? t : t - n;
        if (t >= KS) ok = mbar_wait(&bar_empty[s], ((t / KS) - 1) & 1, ab);
        if (!ok) break;
        mbar_arrive_expect_tx(&bar_full[s], 2 * L::KT);
        for (int i = 0; i < L::BK / 16; ++i) {
          const int lp = u * (L::BK / 16) + i;
          int slot = oob_slot;  // out of the pool: TMA fills zeros
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
        if (t == 0) {
          mbar_arrive_expect_tx(&bar_dy, L::QT);
          for (int c = 0; c < L::NCH; ++c)
            tma_load_3d(sm + L::DY_OFF + c * (L::BQ * 128), &tm_dy, &bar_dy, c * 64, g * p.G, r0);
        }
      }
      // every copy issued has landed before the CTA can leave
      for (int t = max(0, NT - KS); t < NT; ++t) drain_wait(&bar_full[t % KS], (t / KS) & 1);
      drain_wait(&bar_q, 0);
      drain_wait(&bar_dy, 0);
    }
    __syncwarp();
  } else if (n > 0 && warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t id_s = idesc_bf16(128, 64, false, false);
      constexpr uint32_t id_o = idesc_bf16(128, DP, false, true);
      const uint32_t sQ = smem_addr(sm + L::Q_OFF), sDY = smem_addr(sm + L::DY_OFF);
      auto k_at = [&](int s) { return smem_addr(sm + L::K_OFF + s * L::KT); };
      auto v_at = [&](int s) { return smem_addr(sm + L::V_OFF + s * L::KT); };
      auto p_at = [&](int s) { return smem_addr(sm + L::P_OFF + s * L::PT); };
      // D[128 x 64] = A[128 x DP] * B[64 x DP]^T, both K-major in shared memory
      auto issue_xt = [&](uint32_t d, uint32_t a, uint32_t b) {
#pragma unroll
        for (int kk = 0; kk < DP / 16; ++kk) {
          const int c = kk >> 2, o = (kk & 3) * 32;
          const uint64_t ad = sdesc_sw128(a + c * (L::BQ * 128) + o, 16, 1024);
          const uint64_t bd = sdesc_sw128(b + c * (L::BK * 128) + o, 16, 1024);
          mma_bf16_ss(d, ad, bd, id_s, kk > 0 ? 1u : 0u);
        }
      };
      // tile t: S (both sweeps) and dP (sweep 2) into buffer t % 2, from
      // K/V stage t mod KS
      auto issue_tile = [&](int t) {
        const int s = t & 1, ks = t % KS;
        issue_xt(tmem + L::T_S + s * 64, sQ, k_at(ks));
        if (t >= n) issue_xt(tmem + L::T_DP + s * 64, sDY, v_at(ks));
        mma_commit(&bar_s_full[s]);
      };
      bool ok = mbar_wait(&bar_q, 0, ab);
      bool dy_ready = false;
      for (int t = 0; t < 2 && t < NT && ok; ++t) {
        if (!(ok = mbar_wait(&bar_full[t], 0, ab))) break;
        if (t >= n && !dy_ready && !(ok = dy_ready = mbar_wait(&bar_dy, 0, ab))) break;
        tc_fence_after();
        issue_tile(t);
      }
      for (int t = 0; t < NT && ok; ++t) {
        const int s = t & 1, ks = t % KS;
        if (!(ok = mbar_wait(&bar_p_full[s], (t >> 1) & 1, ab))) break;
        tc_fence_after();
        // sweep 1: O += P V; sweep 2: dQ += dS K (B = the V or K tile, MN-major)
        const bool fwd = t < n;
        const uint32_t d = tmem + (fwd ? L::T_O : L::T_DQ);
        const uint32_t b = fwd ? v_at(ks) : k_at(ks);
#pragma unroll
        for (int kk = 0; kk < L::BK / 16; ++kk) {
          const uint64_t ad = sdesc_sw128(p_at(s) + kk * 32, 16, 1024);
          const uint64_t bd = sdesc_sw128(b + kk * 16 * 128, L::BK * 128, 1024);
          mma_bf16_ss(d, ad, bd, id_o, ((t == 0 || t == n) && kk == 0) ? 0u : 1u);
        }
        mma_commit(&bar_p_free[s]);
        mma_commit(&bar_empty[ks]);
        if (t + 2 < NT) {
          if (!(ok = mbar_wait(&bar_full[(t + 2) % KS], ((t + 2) / KS) & 1, ab))) break;
          if (t + 2 >= n && !dy_ready && !(ok = dy_ready = mbar_wait(&bar_dy, 0, ab))) break;
          tc_fence_after();
          issue_tile(t + 2);
        }
      }
      drain_wait(&bar_p_free[(NT - 1) & 1], ((NT - 1) >> 1) & 1);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------------------------------------ one thread per column
    const int lg = warp & 3;
    const int col = lg * 32 + lane;  // column = (row, head) pair == TMEM lane
    const int r = r0 + col / p.G;
    const int hh = g * p.G + col % p.G;
    const bool col_ok = r < r_end;
    const int pos = col_ok ? (p.causal ? p.q_pos[r] : len - 1) : -1;
    const uint32_t lane_addr = static_cast<uint32_t>(lg * 32) << 16;
    const float kInf = __int_as_float(0x7f800000);
    const uint32_t t_o = tmem + L::T_O, t_dq = tmem + L::T_DQ;
    float m2 = -kInf, l = 0.f;
    float lse2 = kInf, dl = 0.f;  // sweep 2: base-2 LSE and delta of the column
    bool ok = n > 0;
    for (int t = 0; t < NT && ok; ++t) {
      const int s = t & 1;
      const int u = t < n ? t : t - n;
      const int tk0 = u * L::BK;
      if (!(ok = mbar_wait_warp(&bar_s_full[s], (t >> 1) & 1, ab))) break;
      tc_fence_after();
      if (t == n) {
        // ---------------------------------------------- statistics from sweep 1
        if (!(ok = mbar_wait_warp(&bar_p_free[(n - 1) & 1], ((n - 1) >> 1) & 1, ab))) break;
        if (!(ok = mbar_wait_warp(&bar_dy, 0, ab))) break;
        tc_fence_after();
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
        float lse = -kInf;
        if (l > 0.f) {
          lse2 = m2 + __log2f(l);
          lse = lse2 * 0.6931471805599453f;
          dl = acc / l;
        }
        if (col_ok) {
          const int64_t idx = static_cast<int64_t>(r) * p.H + hh;
          p.lse_out[idx] = lse;
          p.delta_out[idx] = dl;
        }
      }
      if (t < n) {
        // ---------------------------------------------- sweep 1: S -> P, O += P V
        float x[64];
        {
          uint32_t a0[32], a1[32];
          tmem_ld32(tmem + L::T_S + s * 64 + lane_addr, a0);
          tmem_ld32(tmem + L::T_S + s * 64 + lane_addr + 32, a1);
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
        if (tk0 + L::BK > len) {
          // the stage's copies have landed (observed here, not only by the MMA thread)
          if (!(ok = mbar_wait_warp(&bar_full[t % KS], (t / KS) & 1, ab))) break;
          zero_tail_rows<DP>(sm + L::V_OFF + (t % KS) * L::KT, max(0, len - tk0));
        }
        if (t >= 2 && !(ok = mbar_wait_warp(&bar_p_free[s], ((t - 2) >> 1) & 1, ab))) break;
        const uint32_t sp = smem_addr(sm + L::P_OFF + s * L::PT);
#pragma unroll
        for (int j = 0; j < 8; ++j)
          st_shared_v4(sp + sw128_offset(col, j), pack_bf16x2(pr[8 * j], pr[8 * j + 1]),
                       pack_bf16x2(pr[8 * j + 2], pr[8 * j + 3]), pack_bf16x2(pr[8 * j + 4], pr[8 * j + 5]),
                       pack_bf16x2(pr[8 * j + 6], pr[8 * j + 7]));
      } else {
        // ---------------------------------------------- sweep 2: S, dP -> dS, dQ += dS K
        if (tk0 + L::BK > len) {
          if (!(ok = mbar_wait_warp(&bar_full[t % KS], (t / KS) & 1, ab))) break;
          zero_tail_rows<DP>(sm + L::K_OFF + (t % KS) * L::KT, max(0, len - tk0));
        }
        if (t >= 2 && !(ok = mbar_wait_warp(&bar_p_free[s], ((t - 2) >> 1) & 1, ab))) break;
        const uint32_t sp = smem_addr(sm + L::P_OFF + s * L::PT);
#pragma unroll 1
        for (int hf = 0; hf < 2; ++hf) {  // 32 tokens at a time
          uint32_t sr[32], dr[32];
          tmem_ld32(tmem + L::T_S + s * 64 + 32 * hf + lane_addr, sr);
          tmem_ld32(tmem + L::T_DP + s * 64 + 32 * hf + lane_addr, dr);
          tmem_ld_wait();
          uint32_t w[16];
#pragma unroll
          for (int c2 = 0; c2 < 16; ++c2) {
            float d2[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int c = 2 * c2 + e;
              const int tok = tk0 + 32 * hf + c;
              const bool vis = tok < len && tok <= pos;
              const float pv = ex2_approx(fmaf(__uint_as_float(sr[c]), p.scale_log2, -lse2));
              // a select, not a product: S and dP of tail slots may be NaN
              d2[e] = vis ? pv * (__uint_as_float(dr[c]) - dl) : 0.f;
            }
            w[c2] = pack_bf16x2(d2[0], d2[1]);
          }
#pragma unroll
          for (int j = 0; j < 4; ++j)
            st_shared_v4(sp + sw128_offset(col, 4 * hf + j), w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_p_full[s]);
    }
    // ------------------------------------------------------------ dQ store
    if (ok && n > 0) {
      ok = mbar_wait_warp(&bar_p_free[(NT - 1) & 1], ((NT - 1) >> 1) & 1, ab);
      tc_fence_after();
    }
    // the tensor-memory loads are warp-collective: the condition around them
    // is warp-uniform, and only the stores depend on the column
    if (ok || n == 0) {
      const int64_t roff = (static_cast<int64_t>(r) * p.H + hh) * p.Dk;
      __nv_bfloat16* dq = reinterpret_cast<__nv_bfloat16*>(p.dq);
      if (n == 0 && col_ok) {
        const int64_t idx = static_cast<int64_t>(r) * p.H + hh;
        p.lse_out[idx] = -kInf;
        p.delta_out[idx] = 0.f;
      }
#pragma unroll 1
      for (int cc = 0; cc < DP / 32 && cc * 32 < p.Dk; ++cc) {
        uint32_t rr[32];
        if (n > 0) {
          tmem_ld32(t_dq + lane_addr + cc * 32, rr);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) rr[j] = 0u;
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          uint4 v;
          v.x = pack_bf16x2(__uint_as_float(rr[8 * j]) * p.scale, __uint_as_float(rr[8 * j + 1]) * p.scale);
          v.y = pack_bf16x2(__uint_as_float(rr[8 * j + 2]) * p.scale, __uint_as_float(rr[8 * j + 3]) * p.scale);
          v.z = pack_bf16x2(__uint_as_float(rr[8 * j + 4]) * p.scale, __uint_as_float(rr[8 * j + 5]) * p.scale);
          v.w = pack_bf16x2(__uint_as_float(rr[8 * j + 6]) * p.scale, __uint_as_float(rr[8 * j + 7]) * p.scale);
          if (col_ok) *reinterpret_cast<uint4*>(dq + roff + cc * 32 + 8 * j) = v;
        }
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

// Rows before the first sequence's first row or past the last one belong to
// no sequence: their dQ is zero and their statistics those of a row with no
// visible token.
__global__ void paged_query_outside_kernel(const PagedParams p) {
  const int lo = min(max(p.q_start[0], 0), p.Nq), hi = min(max(p.q_start[p.S], lo), p.Nq);
  __nv_bfloat16* dq = reinterpret_cast<__nv_bfloat16*>(p.dq);
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < static_cast<int64_t>(p.Nq) * p.H;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int r = static_cast<int>(i / p.H);
    if (r >= lo && r < hi) continue;
    p.lse_out[i] = -__int_as_float(0x7f800000);
    p.delta_out[i] = 0.f;
    for (int d = 0; d < p.Dk; ++d) dq[i * p.Dk + d] = __float2bfloat16(0.f);
    if (p.dqp)
      for (int d = 0; d < p.Dp; ++d) static_cast<__nv_bfloat16*>(p.dqp)[i * p.Dp + d] = __float2bfloat16(0.f);
  }
}

template <int DP>
cudaError_t launch_query_t(const PagedMaps& m, const PagedParams& p, cudaStream_t s) {
  using L = QueryLayout<DP>;
  auto kern = paged_query_kernel<DP>;
  const int smem = max(L::BYTES, kSmemOneCtaPerSm);  // all 512 TMEM columns: one CTA per SM
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int rt = L::BQ / p.G;
  // row tiles: at most Nq / rt + S (one partial tile per sequence)
  dim3 grid(static_cast<unsigned>((static_cast<int64_t>(p.Nq) / rt + p.S + 1) * p.KVH));
  kern<<<grid, 256, smem, s>>>(m.q_stats, m.dy_stats, m.k, m.v, p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  paged_query_outside_kernel<<<64, 256, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_paged_query_outside(const PagedParams& p, cudaStream_t s) {
  if (p.Nq == 0) return cudaSuccess;
  paged_query_outside_kernel<<<64, 256, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_paged_query(const PagedMaps& m, const PagedParams& p, cudaStream_t s) {
  if (p.Nq == 0) return cudaSuccess;
  if (p.S == 0) {
    paged_query_outside_kernel<<<64, 256, 0, s>>>(p);
    return cudaGetLastError();
  }
  if (p.Dk <= 64) return launch_query_t<64>(m, p, s);
  return launch_query_t<128>(m, p, s);
}

}  // namespace attn
