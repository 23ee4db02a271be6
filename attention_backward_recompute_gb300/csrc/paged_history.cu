// Paged history backward (GQA): dK and dV of every pool row, atomic-free.
//
// ruDNN src/paged_attention/ordered_kernel.rs (history_backward): for every
// physical token and KV head, sum over the links of its page, over the query
// rows of the linked sequence that see the token (t <= pos(r) when causal) and
// over the query heads of the KV group:
//   p  = exp(q.k * scale - lse),  ds = p * (dY.v - delta) * scale
//   dK += ds * q,   dV += p * dY
// Here one CTA owns 128 tokens (eight 16-token pages) of one sequence and one
// KV head and does the same sums as tile products on tcgen05:
//   S^T  = K_T Q_c^T,  dP^T = V_T dY_c^T            (M=128 tokens, N=64 columns)
//   P^T  = exp2(S^T scale log2e - lse log2e)        softmax warpgroups
//   dS^T = P^T (dP^T - delta)                        dS warpgroup
//   dV_T += P^T dY_c,  dK_T += dS^T Q_c              (A operand from tensor memory)
// where a column c is one (query row, head of the group) pair.  The K/V tile is
// gathered page by page with TMA (3-D map over [slots, KVH, D]); pages past the
// sequence are fetched at an out-of-range coordinate, i.e. read as zeros
// without touching memory.  Passes: the CTA's own sequence first, then the
// other links of the pages it stores, by link index; consecutive pages linked
// from consecutive logical pages of one sequence share a pass (a shared prefix
// costs one pass per (sequence, block), not one per page).
//
// Roles (512 threads): warp 0 TMA producer (K/V pages once, then Q/dY column
// tiles through a 4-stage ring with the columns' statistics), warp 1 MMA
// issuer (whole warp, elect.sync), warps 4..7 / 12..15 softmax of even / odd
// tiles (one per double-buffered S^T), warps 8..11 dS.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "paged_common.cuh"
#include "paged_launch.h"
#include "paged_pass.cuh"
#include "sm103.cuh"

namespace attn {
using namespace sm103;

namespace {

constexpr int kStages = 4;

template <int DP>
struct HistLayout {
  static constexpr int NCH = DP / 64;
  static constexpr int BT = 128, BC = 64;        // tokens x columns per step
  static constexpr int KV = NCH * BT * 128;
  static constexpr int QT = NCH * BC * 128;
  static constexpr int K_OFF = 0;
  static constexpr int V_OFF = K_OFF + KV;
  static constexpr int Q_OFF = V_OFF + KV;             // kStages
  static constexpr int DY_OFF = Q_OFF + kStages * QT;  // kStages
  static constexpr int ST_OFF = DY_OFF + kStages * QT; // kStages x {L2, delta, pos} x 64 + pass info
  static constexpr int ST_STAGE = 3 * BC * 4 + 16;
  static constexpr int BYTES = ST_OFF + kStages * ST_STAGE;
  // TMEM: dV [0, DP), dK [DP, 2DP), S^T[2] and dP^T[2] 64 columns each
  static constexpr int T_S = 2 * DP, T_DP = 2 * DP + 128;
  static constexpr int TMEM_COLS = 512;
};

__device__ __forceinline__ bool drain_wait(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_test(bar, parity)) {
    if (global_timer_ns() - t0 > ATTN_WAIT_TIMEOUT_NS) return false;
  }
  return true;
}

// Registers written by tcgen05.ld are valid only after tcgen05.wait::ld; this
// empty asm ties every later use of r to a point after the wait.
__device__ __forceinline__ void reg_fence16(uint32_t (&r)[16]) {
#pragma unroll
  for (int i = 0; i < 16; ++i) asm volatile("" : "+r"(r[i]));
}

// P^T row of one token over the 64 columns of a tile, S^T read from tensor
// memory in four 16-column chunks (the next chunk's load in flight); chunk i's
// 8 bf16 pairs go to columns [8i, 8i+8) of the same buffer.  A column is
// visible when the token is live and tok <= pos[c] (pos = -1 for a column
// without visible history).
__device__ __forceinline__ void p_row_paged(uint32_t tS, const float* l2s, const int* poss, bool tok_ok, int tok,
                                            float scale_log2) {
  uint32_t s0[16], s1[16], pw[8];
  tmem_ld16(tS, s0);
  tmem_ld_wait();
  reg_fence16(s0);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t(&cur)[16] = (i & 1) ? s1 : s0;
    uint32_t(&nxt)[16] = (i & 1) ? s0 : s1;
    if (i < 3) tmem_ld16(tS + 16 * (i + 1), nxt);
#pragma unroll
    for (int c4 = 0; c4 < 4; ++c4) {
      const int c0 = 16 * i + 4 * c4;
      const float4 l2 = *reinterpret_cast<const float4*>(l2s + c0);
      const int4 ps = *reinterpret_cast<const int4*>(poss + c0);
      const float l2v[4] = {l2.x, l2.y, l2.z, l2.w};
      const int pv4[4] = {ps.x, ps.y, ps.z, ps.w};
      float pv[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float x = fmaf(__uint_as_float(cur[4 * c4 + e]), scale_log2, -l2v[e]);
        const float pe = ex2_approx(x);
        pv[e] = (tok_ok && tok <= pv4[e]) ? pe : 0.f;
      }
      pw[2 * c4] = pack_bf16x2(pv[0], pv[1]);
      pw[2 * c4 + 1] = pack_bf16x2(pv[2], pv[3]);
    }
    tmem_st8(tS + 8 * i, pw);
    if (i < 3) {
      tmem_ld_wait();
      reg_fence16(nxt);
    }
  }
}

template <int DP>
__global__ void __launch_bounds__(512, 1)
    paged_history_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_dy,
                         const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                         const PagedParams p) {
  using L = HistLayout<DP>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t bar_kv, bar_full[kStages], bar_empty[kStages], bar_s_full[2], bar_dp_full[2], bar_p_full[2],
      bar_p_read[2], bar_ds_full[2], bar_acc;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag;
  __shared__ PageInfo pinfo;
  __shared__ int n_steps_sh, any_store_sh;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the KV heads of one token block are neighbours in the grid: together they
  // read (and write) whole slot rows of the same pages
  const int g = blockIdx.x, tb = blockIdx.y, s0 = blockIdx.z;
  const int len0 = seq_len_of(p, s0);
  const int npg = pages_of(len0, p.page_size);
  if (tb * 8 >= npg) return;  // no token of this sequence in the block (uniform exit)
  const int RT = L::BC / p.G;  // query rows per step
  const Abort ab{&abort_flag, p.err};

  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bar_kv, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bar_full[s], 2);  // TMA bytes + column statistics written
      mbar_init(&bar_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bar_s_full[s], 1);
      mbar_init(&bar_dp_full[s], 1);
      mbar_init(&bar_p_full[s], 4);
      mbar_init(&bar_p_read[s], 4);
      mbar_init(&bar_ds_full[s], 4);
    }
    mbar_init(&bar_acc, 1);
    mbar_fence_init();
    any_store_sh = fill_page_info(p, s0, tb, npg, &pinfo);
    // number of steps over all passes
    PassIter it{&p, &pinfo, s0, tb};
    int n = 0;
    if (it.begin(RT)) {
      do ++n;
      while (it.advance(RT));
    }
    n_steps_sh = n;
  }
  __syncthreads();
  // a block whose pages are all stored by other CTAs (their owners) has
  // nothing to write: leave before taking tensor memory (uniform exit)
  if (!any_store_sh) return;
  if (warp == 1) {
    tmem_alloc(&tmem_base_sh, L::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  const uint32_t t_dv = tmem, t_dk = tmem + DP;
  const int n = n_steps_sh;
  const int oob_slot = p.num_pages * p.page_size;  // out-of-range coordinate: TMA fills zeros

  if (n > 0 && warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_map(&tm_q);
      tma_prefetch_map(&tm_dy);
      tma_prefetch_map(&tm_k);
      tma_prefetch_map(&tm_v);
      mbar_arrive_expect_tx(&bar_kv, 2 * L::KV);
      for (int j = 0; j < 8; ++j) {
        const int slot = pinfo.phys[j] >= 0 ? pinfo.phys[j] * p.page_size : oob_slot;
        for (int c = 0; c < L::NCH; ++c) {
          tma_load_3d(sm + L::K_OFF + c * (L::BT * 128) + j * 16 * 128, &tm_k, &bar_kv, c * 64, g, slot);
          tma_load_3d(sm + L::V_OFF + c * (L::BT * 128) + j * 16 * 128, &tm_v, &bar_kv, c * 64, g, slot);
        }
      }
    }
    PassIter it{&p, &pinfo, s0, tb};
    it.begin(RT);
    int last_use[kStages];
    for (int i = 0; i < kStages; ++i) last_use[i] = -1;
    bool ok = true;
    for (int t = 0; t < n && ok; ++t) {
      const int s = t % kStages;
      if (t >= kStages) ok = mbar_wait_warp(&bar_empty[s], ((t / kStages) - 1) & 1, ab);
      if (!ok) break;
      const int row0 = it.r_begin + it.tile * RT;
      if (lane == 0) {
        mbar_arrive_expect_tx(&bar_full[s], 2 * L::QT);
        for (int c = 0; c < L::NCH; ++c) {
          tma_load_3d(sm + L::Q_OFF + s * L::QT + c * (L::BC * 128), &tm_q, &bar_full[s], c * 64, g * p.G, row0);
          tma_load_3d(sm + L::DY_OFF + s * L::QT + c * (L::BC * 128), &tm_dy, &bar_full[s], c * 64, g * p.G, row0);
        }
      }
      uint8_t* st = sm + L::ST_OFF + s * L::ST_STAGE;
      float* sl2 = reinterpret_cast<float*>(st);
      float* sdl = sl2 + L::BC;
      int* spos = reinterpret_cast<int*>(sdl + L::BC);
      int* sinfo = spos + L::BC;
      for (int c = lane; c < L::BC; c += 32) {
        const int r = row0 + c / p.G;
        const int hh = g * p.G + c % p.G;
        const bool in = r < it.r_end;
        float l2 = __int_as_float(0x7f800000), dl = 0.f;
        int pos = -1;
        if (in) {
          const float lse = p.lse[static_cast<int64_t>(r) * p.H + hh];
          if (lse != -__int_as_float(0x7f800000)) {
            l2 = lse * 1.4426950408889634f;
            dl = p.delta[static_cast<int64_t>(r) * p.H + hh];
            pos = p.causal ? p.q_pos[r] : 0x7fffffff;
          }
        }
        sl2[c] = l2;
        sdl[c] = dl;
        spos[c] = pos;
      }
      if (lane == 0) {
        sinfo[0] = it.tbase;
        sinfo[1] = it.ra;
        sinfo[2] = it.rb;
        sinfo[3] = seq_len_of(p, it.seq);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_full[s]);
      last_use[s] = t;
      it.advance(RT);
    }
    if (lane == 0) {
      for (int s = 0; s < kStages; ++s)
        if (last_use[s] >= 0) drain_wait(&bar_full[s], (last_use[s] / kStages) & 1);
      drain_wait(&bar_kv, 0);
    }
  } else if (n > 0 && warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // the whole warp runs this role (warp-uniform); elected lanes issue
    {
      constexpr uint32_t id_s = idesc_bf16(128, 64, false, false);
      constexpr uint32_t id_acc = idesc_bf16(128, DP, false, true);
      const uint64_t dK = sdesc_sw128(smem_addr(sm + L::K_OFF), 16, 1024);
      const uint64_t dV = sdesc_sw128(smem_addr(sm + L::V_OFF), 16, 1024);
      const uint64_t dQ0 = sdesc_sw128(smem_addr(sm + L::Q_OFF), 16, 1024);
      const uint64_t dDY0 = sdesc_sw128(smem_addr(sm + L::DY_OFF), 16, 1024);
      const uint64_t dQm0 = sdesc_sw128(smem_addr(sm + L::Q_OFF), L::BC * 128, 1024);    // MN-major
      const uint64_t dDYm0 = sdesc_sw128(smem_addr(sm + L::DY_OFF), L::BC * 128, 1024);  // MN-major
      // D[128 x 64] = A[128 x DP] * B[64 x DP]^T, both from shared memory, K-major
      auto issue_xt = [&](uint32_t d, uint64_t a, uint64_t bq) {
        mma_ss_w<false>(d, a, bq, id_s);
#pragma unroll
        for (int kk = 1; kk < DP / 16; ++kk) {
          const int c = kk >> 2, o = (kk & 3) * 32;
          mma_ss_w<true>(d, sdesc_add(a, c * (L::BT * 128) + o), sdesc_add(bq, c * (L::BC * 128) + o), id_s);
        }
      };
      // D[128 x DP] (+)= A[128 x 64] (tensor memory, bf16 pairs) * B[64 x DP] (MN-major)
      auto issue_acc = [&](uint32_t d, uint32_t a_tmem, uint64_t bm, bool first) {
        if (first)
          mma_ts_w<false>(d, a_tmem, bm, id_acc);
        else
          mma_ts_w<true>(d, a_tmem, bm, id_acc);
#pragma unroll
        for (int kk = 1; kk < L::BC / 16; ++kk) mma_ts_w<true>(d, a_tmem + kk * 8, sdesc_add(bm, kk * 16 * 128), id_acc);
      };
      auto issue_s = [&](int t) {
        issue_xt(tmem + L::T_S + (t & 1) * 64, dK, sdesc_add(dQ0, (t % kStages) * L::QT));
        mma_commit_w(&bar_s_full[t & 1]);
      };
      auto issue_dp = [&](int t) {
        issue_xt(tmem + L::T_DP + (t & 1) * 64, dV, sdesc_add(dDY0, (t % kStages) * L::QT));
        mma_commit_w(&bar_dp_full[t & 1]);
      };
      bool ok = mbar_wait_warp(&bar_kv, 0, ab);
      for (int t = 0; t < 2 && t < n && ok; ++t) {
        if (!(ok = mbar_wait_warp(&bar_full[t], 0, ab))) break;
        tc_fence_after();
        issue_s(t);
        issue_dp(t);
      }
      // Issue order per tile t: dV(t), S(t+2), dK(t), dP(t+2) (as in the dense
      // dK/dV kernel): S(t+2) overwrites P^T(t) once dV(t) (earlier in the
      // pipe) and the dS warpgroup (p_read) have consumed it; dP(t+2)
      // overwrites dS^T(t), read by dK(t) just before it.
      for (int t = 0; t < n && ok; ++t) {
        const int s = t % kStages, bb = t & 1;
        if (!(ok = mbar_wait_warp(&bar_p_full[bb], (t >> 1) & 1, ab))) break;
        tc_fence_after();
        issue_acc(t_dv, tmem + L::T_S + bb * 64, sdesc_add(dDYm0, s * L::QT), t == 0);
        if (t + 2 < n) {
          if (!(ok = mbar_wait_warp(&bar_full[(t + 2) % kStages], ((t + 2) / kStages) & 1, ab))) break;
          if (!(ok = mbar_wait_warp(&bar_p_read[bb], (t >> 1) & 1, ab))) break;
          tc_fence_after();
          issue_s(t + 2);
        }
        if (!(ok = mbar_wait_warp(&bar_ds_full[bb], (t >> 1) & 1, ab))) break;
        tc_fence_after();
        issue_acc(t_dk, tmem + L::T_DP + bb * 64, sdesc_add(dQm0, s * L::QT), t == 0);
        mma_commit_w(&bar_empty[s]);
        if (t + 2 < n) issue_dp(t + 2);
      }
      mma_commit_w(&bar_acc);
      drain_wait(&bar_acc, 0);
    }
    __syncwarp();
  } else if (warp >= 4) {
    const bool softmax_wg = warp < 8 || warp >= 12;  // warps 4..7, 12..15: P; warps 8..11: dS
    const int sg = warp >= 12 ? 1 : 0;               // softmax group: tiles (and S buffer) of parity sg
    const int lg = warp & 3;
    const int row = lg * 32 + lane;  // token row inside the block == TMEM lane
    const uint32_t lane_addr = static_cast<uint32_t>(lg * 32) << 16;
    bool ok = n > 0;
    if (n > 0 && softmax_wg) {
      // ---------------------------------------------------------- softmax: S^T -> P^T
      // Each group waits every phase of its own S buffer.  Of the stage
      // barrier it skips the phases of the other group's tiles; when it waits
      // for tile t, the phase of tile t - kStages (same stage) has completed,
      // since the tensor core issued S(t - 2) after it.
      for (int t = sg; t < n && ok; t += 2) {
        const int s = t % kStages, bb = t & 1;
        if (!(ok = mbar_wait_warp(&bar_full[s], (t / kStages) & 1, ab))) break;
        const uint8_t* st = sm + L::ST_OFF + s * L::ST_STAGE;
        const float* sl2 = reinterpret_cast<const float*>(st);
        const int* spos = reinterpret_cast<const int*>(sl2 + 2 * L::BC);
        const int* sinfo = spos + L::BC;
        const int tok = sinfo[0] + row;
        const bool tok_ok = row >= sinfo[1] && row < sinfo[2] && tok >= 0 && tok < sinfo[3];
        if (!(ok = mbar_wait_warp(&bar_s_full[bb], (t >> 1) & 1, ab))) break;
        tc_fence_after();
        p_row_paged(tmem + L::T_S + bb * 64 + lane_addr, sl2, spos, tok_ok, tok, p.scale_log2);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar_p_full[bb]);
      }
    } else if (n > 0) {
      // ---------------------------------------------------------- dS: dP^T, P^T -> dS^T
      for (int t = 0; t < n && ok; ++t) {
        const int s = t % kStages, bb = t & 1;
        if (!(ok = mbar_wait_warp(&bar_full[s], (t / kStages) & 1, ab))) break;
        if (!(ok = mbar_wait_warp(&bar_dp_full[bb], (t >> 1) & 1, ab))) break;
        if (!(ok = mbar_wait_warp(&bar_p_full[bb], (t >> 1) & 1, ab))) break;
        tc_fence_after();
        const uint32_t tDP = tmem + L::T_DP + bb * 64 + lane_addr;
        const uint32_t tS = tmem + L::T_S + bb * 64 + lane_addr;
        uint32_t pw[32];
        tmem_ld32(tS, pw);
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar_p_read[bb]);
        const float* dl = reinterpret_cast<const float*>(sm + L::ST_OFF + s * L::ST_STAGE) + L::BC;
        // two halves of 32 columns: half hf reads dP columns [32hf, 32hf+32)
        // and writes dS^T (bf16 pairs) to columns [16hf, 16hf+16).  A masked
        // entry has P = 0 and takes dS = 0 by select: dP of a tail or unowned
        // slot may be NaN.
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          uint32_t dr[32], dsw[16];
          tmem_ld32(tDP + 32 * hf, dr);
          tmem_ld_wait();
#pragma unroll
          for (int c4 = 0; c4 < 8; ++c4) {
            const float4 d4 = *reinterpret_cast<const float4*>(dl + 32 * hf + 4 * c4);
            const float dv4[4] = {d4.x, d4.y, d4.z, d4.w};
            const uint32_t w[2] = {pw[16 * hf + 2 * c4], pw[16 * hf + 2 * c4 + 1]};
            float ds[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float pe = __uint_as_float((e & 1) ? (w[e >> 1] & 0xffff0000u) : (w[e >> 1] << 16));
              ds[e] = pe != 0.f ? pe * (__uint_as_float(dr[4 * c4 + e]) - dv4[e]) : 0.f;
            }
            dsw[2 * c4] = pack_bf16x2(ds[0], ds[1]);
            dsw[2 * c4 + 1] = pack_bf16x2(ds[2], ds[3]);
          }
          tmem_st16(tDP + 16 * hf, dsw);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar_ds_full[bb]);
      }
    }
    if (n > 0) {
      if (ok) ok = mbar_wait_warp(&bar_acc, 0, ab);
      tc_fence_after();
    }
    // ------------------------------------------------------------ epilogue
    // the softmax warpgroups store dV (half of the columns each), the dS
    // warpgroup dK (times the softmax scale), each row of a page this CTA
    // stores; rows of tokens no pass saw are zero
    const int wg = softmax_wg ? 0 : 1;
    const int j = row >> 4;
    const bool want = wg == 0 ? (p.wrt & 4u) != 0 : (p.wrt & 2u) != 0;
    if (want && (ok || n == 0)) {  // warp-uniform: the tensor-memory loads are warp-collective
      const bool mine = pinfo.store[j] != 0;
      const int dim = wg == 0 ? p.Dv : p.Dk;
      const int64_t prow = (static_cast<int64_t>(pinfo.phys[j]) * p.page_size + (row & 15)) * p.KVH + g;
      __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(wg == 0 ? p.dv_pool : p.dk_pool) + prow * dim;
      const float f = wg == 0 ? 1.f : p.scale;
      const uint32_t tacc = (wg == 0 ? t_dv : t_dk) + lane_addr;
      const int c_lo = wg == 0 ? sg * (DP / 64) : 0, c_hi = wg == 0 ? (sg + 1) * (DP / 64) : DP / 32;
#pragma unroll 1
      for (int cc = c_lo; cc < c_hi && cc * 32 < dim; ++cc) {
        uint32_t r[32];
        if (n > 0) {
          tmem_ld32(tacc + cc * 32, r);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int q = 0; q < 32; ++q) r[q] = 0u;
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          if (mine && cc * 32 + q * 8 < dim) {
            uint4 v;
            v.x = pack_bf16x2(__uint_as_float(r[8 * q]) * f, __uint_as_float(r[8 * q + 1]) * f);
            v.y = pack_bf16x2(__uint_as_float(r[8 * q + 2]) * f, __uint_as_float(r[8 * q + 3]) * f);
            v.z = pack_bf16x2(__uint_as_float(r[8 * q + 4]) * f, __uint_as_float(r[8 * q + 5]) * f);
            v.w = pack_bf16x2(__uint_as_float(r[8 * q + 6]) * f, __uint_as_float(r[8 * q + 7]) * f);
            *reinterpret_cast<uint4*>(out + cc * 32 + q * 8) = v;
          }
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

template <int DP>
cudaError_t launch_hist_t(const PagedMaps& m, const PagedParams& p, cudaStream_t s) {
  using L = HistLayout<DP>;
  auto kern = paged_history_kernel<DP>;
  const int smem = max(L::BYTES + 1024, kSmemOneCtaPerSm);  // all 512 TMEM columns: one CTA per SM
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int nblk = (p.max_pages * p.page_size + 127) / 128;
  dim3 grid(p.KVH, nblk, p.S);
  kern<<<grid, 512, smem, s>>>(m.q, m.dy, m.k, m.v, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_paged_history(const PagedMaps& m, const PagedParams& p, cudaStream_t s) {
  if (p.Dk <= 64) return launch_hist_t<64>(m, p, s);
  return launch_hist_t<128>(m, p, s);
}

}  // namespace attn
