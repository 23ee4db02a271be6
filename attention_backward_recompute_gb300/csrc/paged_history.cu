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
//   P^T, dS^T in registers (masks, statistics)
//   dV_T += P^T dY_c,  dK_T += dS^T Q_c              (TMEM accumulators)
// where a column c is one (query row, head of the group) pair.  The K/V tile is
// gathered page by page with TMA (3-D map over [slots, KVH, D]); pages past the
// sequence are fetched at an out-of-range coordinate, i.e. read as zeros
// without touching memory.  Passes: the CTA's own sequence first, then, for
// every page it stores that other links share, those links in increasing link
// order (only that page's 16 rows are live in such a pass).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "paged_common.cuh"
#include "paged_launch.h"
#include "sm103.cuh"

namespace attn {
using namespace sm103;

namespace {

template <int DP>
struct HistLayout {
  static constexpr int NCH = DP / 64;
  static constexpr int BT = 128, BC = 64;        // tokens x columns per step
  static constexpr int KV = NCH * BT * 128;
  static constexpr int QT = NCH * BC * 128;
  static constexpr int PT = BT * 128;
  static constexpr int K_OFF = 0;
  static constexpr int V_OFF = K_OFF + KV;
  static constexpr int Q_OFF = V_OFF + KV;         // 2 stages
  static constexpr int DY_OFF = Q_OFF + 2 * QT;    // 2 stages
  static constexpr int P_OFF = DY_OFF + 2 * QT;
  static constexpr int DS_OFF = P_OFF + PT;
  static constexpr int ST_OFF = DS_OFF + PT;       // 2 stages x {L2, delta, pos, step info}
  static constexpr int ST_STAGE = 3 * BC * 4 + 16;
  static constexpr int BYTES = ST_OFF + 2 * ST_STAGE;
  static constexpr int TMEM_COLS = (2 * DP + 128) <= 256 ? 256 : 512;
};

struct PageInfo {
  int phys[8];    // physical page (or -1)
  int off[8];     // first index of the page's link segment
  int cnt[8];     // links of the page
  int store[8];   // this CTA stores the page
};

// One pass = one (sequence, token mapping, live row range); the passes of a CTA
// are enumerated identically by every role.
struct PassIter {
  const PagedParams* p;
  const PageInfo* pi;
  int s0, tb;
  int j, li;                         // j = -1: own pass; else page j, link index li
  int seq, tbase, ra, rb, r_begin, r_end, tile, ntiles;

  __device__ void load(int sq, int tbs, int a, int b, int rt) {
    seq = sq;
    tbase = tbs;
    ra = a;
    rb = b;
    r_begin = row_begin_of(*p, sq);
    r_end = row_end_of(*p, sq);
    tile = 0;
    ntiles = (r_end - r_begin + rt - 1) / rt;
  }
  // advance to the next pass that has at least one tile; false when done
  __device__ bool next_pass(int rt) {
    while (true) {
      if (j < 0) {
        j = 0;
        li = 1;
      } else {
        ++li;
      }
      while (j < 8 && !(pi->store[j] && li < pi->cnt[j])) {
        ++j;
        li = 1;
      }
      if (j >= 8) return false;
      const int link = p->links[pi->off[j] + li];
      const int s2 = link / p->max_pages, lp2 = link - s2 * p->max_pages;
      load(s2, lp2 * p->page_size - 16 * j, 16 * j, 16 * j + 16, rt);
      if (ntiles > 0) return true;
    }
  }
  __device__ bool begin(int rt) {
    j = -1;
    li = 0;
    load(s0, tb * 128, 0, 128, rt);
    if (ntiles > 0) return true;
    return next_pass(rt);
  }
  __device__ bool advance(int rt) {
    if (++tile < ntiles) return true;
    return next_pass(rt);
  }
};

__device__ __forceinline__ bool drain_wait(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_test(bar, parity)) {
    if (global_timer_ns() - t0 > ATTN_WAIT_TIMEOUT_NS) return false;
  }
  return true;
}

template <int DP>
__global__ void __launch_bounds__(384, 1)
    paged_history_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_dy,
                         const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                         const PagedParams p) {
  using L = HistLayout<DP>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t bar_kv, bar_full[2], bar_empty[2], bar_s_full, bar_dp_full, bar_p_full, bar_ds_full,
      bar_p_free, bar_ds_free, bar_acc;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag;
  __shared__ PageInfo pinfo;
  __shared__ int n_steps_sh;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tb = blockIdx.x, s0 = blockIdx.y, g = blockIdx.z;
  const int len0 = seq_len_of(p, s0);
  const int npg = pages_of(len0, p.page_size);
  if (tb * 8 >= npg) return;  // no token of this sequence in the block (uniform exit)
  const int RT = L::BC / p.G;  // query rows per step
  const Abort ab{&abort_flag, p.err};

  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bar_kv, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bar_full[s], 2);
      mbar_init(&bar_empty[s], 1);
    }
    mbar_init(&bar_s_full, 1);
    mbar_init(&bar_dp_full, 1);
    mbar_init(&bar_p_full, 8);
    mbar_init(&bar_ds_full, 8);
    mbar_init(&bar_p_free, 1);
    mbar_init(&bar_ds_free, 1);
    mbar_init(&bar_acc, 1);
    mbar_fence_init();
    for (int j = 0; j < 8; ++j) {
      const int lp = tb * 8 + j;
      int ph = -1, off = 0, cnt = 0, st = 0;
      if (lp < npg) {
        ph = p.page_table[static_cast<int64_t>(s0) * p.max_pages + lp];
        if (ph >= 0 && ph < p.num_pages) {
          off = p.link_off[ph];
          cnt = p.link_off[ph + 1] - off;
          st = cnt > 0 && p.links[off] == s0 * p.max_pages + lp;
        } else {
          ph = -1;
        }
      }
      pinfo.phys[j] = ph;
      pinfo.off[j] = off;
      pinfo.cnt[j] = cnt;
      pinfo.store[j] = st;
    }
    // number of steps over all passes
    PassIter it{&p, &pinfo, s0, tb};
    int n = 0;
    if (it.begin(RT)) {
      do ++n;
      while (it.advance(RT));
    }
    n_steps_sh = n;
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
    int last_use[2] = {-1, -1};
    bool ok = true;
    for (int t = 0; t < n && ok; ++t) {
      const int s = t & 1;
      if (t >= 2) ok = mbar_wait(&bar_empty[s], ((t >> 1) - 1) & 1, ab);
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
      auto q_at = [&](int s) { return smem_addr(sm + L::Q_OFF + s * L::QT); };
      auto dy_at = [&](int s) { return smem_addr(sm + L::DY_OFF + s * L::QT); };
      auto issue_xt = [&](uint32_t d, uint32_t a_base, uint32_t b_base) {
#pragma unroll
        for (int kk = 0; kk < DP / 16; ++kk) {
          const int c = kk >> 2, o = (kk & 3) * 32;
          const uint64_t ad = sdesc_sw128(a_base + c * (L::BT * 128) + o, 16, 1024);
          const uint64_t bd = sdesc_sw128(b_base + c * (L::BC * 128) + o, 16, 1024);
          mma_bf16_ss(d, ad, bd, id_s, kk > 0 ? 1u : 0u);
        }
      };
      auto issue_acc = [&](uint32_t d, uint32_t a_base, uint32_t b_base, bool first) {
#pragma unroll
        for (int kk = 0; kk < L::BC / 16; ++kk) {
          const uint64_t ad = sdesc_sw128(a_base + kk * 32, 16, 1024);
          const uint64_t bd = sdesc_sw128(b_base + kk * 16 * 128, L::BC * 128, 1024);
          mma_bf16_ss(d, ad, bd, id_acc, (first && kk == 0) ? 0u : 1u);
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
      drain_wait(&bar_acc, 0);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax / dS warpgroups
    const int wg = (warp - 4) >> 2;
    const int lg = warp & 3;
    const int row = lg * 32 + lane;  // token row inside the block == TMEM lane
    const int c0 = wg * 32;
    const uint32_t lane_addr = static_cast<uint32_t>(lg * 32) << 16;
    const uint32_t sP = smem_addr(sm + L::P_OFF), sDS = smem_addr(sm + L::DS_OFF);
    bool ok = n > 0;
    for (int t = 0; t < n && ok; ++t) {
      const int s = t & 1;
      if (!(ok = mbar_wait_warp(&bar_full[s], (t >> 1) & 1, ab))) break;
      const uint8_t* st = sm + L::ST_OFF + s * L::ST_STAGE;
      const float* sl2 = reinterpret_cast<const float*>(st);
      const float* sdl = sl2 + L::BC;
      const int* spos = reinterpret_cast<const int*>(sdl + L::BC);
      const int* sinfo = spos + L::BC;
      const int tok = sinfo[0] + row;
      const bool tok_ok = row >= sinfo[1] && row < sinfo[2] && tok >= 0 && tok < sinfo[3];
      if (!(ok = mbar_wait_warp(&bar_s_full, t & 1, ab))) break;
      tc_fence_after();
      uint32_t sr[32];
      tmem_ld32(t_s + lane_addr + c0, sr);
      tmem_ld_wait();
      float pr[32];
      bool vis[32];
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        vis[c] = tok_ok && tok <= spos[c0 + c];
        const float x = fmaf(__uint_as_float(sr[c]), p.scale_log2, -sl2[c0 + c]);
        pr[c] = vis[c] ? ex2_approx(x) : 0.f;
      }
      if (t > 0 && !(ok = mbar_wait_warp(&bar_p_free, (t - 1) & 1, ab))) break;
#pragma unroll
      for (int jj = 0; jj < 4; ++jj)
        st_shared_v4(sP + sw128_offset(row, (c0 >> 3) + jj), pack_bf16x2(pr[8 * jj], pr[8 * jj + 1]),
                     pack_bf16x2(pr[8 * jj + 2], pr[8 * jj + 3]), pack_bf16x2(pr[8 * jj + 4], pr[8 * jj + 5]),
                     pack_bf16x2(pr[8 * jj + 6], pr[8 * jj + 7]));
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
      for (int c = 0; c < 32; ++c) ds[c] = vis[c] ? pr[c] * (__uint_as_float(dr[c]) - sdl[c0 + c]) : 0.f;
      if (t > 0 && !(ok = mbar_wait_warp(&bar_ds_free, (t - 1) & 1, ab))) break;
#pragma unroll
      for (int jj = 0; jj < 4; ++jj)
        st_shared_v4(sDS + sw128_offset(row, (c0 >> 3) + jj), pack_bf16x2(ds[8 * jj], ds[8 * jj + 1]),
                     pack_bf16x2(ds[8 * jj + 2], ds[8 * jj + 3]), pack_bf16x2(ds[8 * jj + 4], ds[8 * jj + 5]),
                     pack_bf16x2(ds[8 * jj + 6], ds[8 * jj + 7]));
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_ds_full);
    }
    if (n > 0) {
      if (ok) ok = mbar_wait_warp(&bar_acc, 0, ab);
      tc_fence_after();
    }
    // ------------------------------------------------------------ epilogue
    // warpgroup 0 stores dV, warpgroup 1 dK (times the softmax scale), each
    // row of a page this CTA stores; rows of tokens no pass saw are zero.
    const int j = row >> 4;
    const bool want = wg == 0 ? (p.wrt & 4u) != 0 : (p.wrt & 2u) != 0;
    if (want && (ok || n == 0)) {
      const int dim = wg == 0 ? p.Dv : p.Dk;
      const bool mine = pinfo.store[j] != 0;
      const int64_t prow = (static_cast<int64_t>(pinfo.phys[j]) * p.page_size + (row & 15)) * p.KVH + g;
      __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(wg == 0 ? p.dv_pool : p.dk_pool) + prow * dim;
      const float f = wg == 0 ? 1.f : p.scale;
      const uint32_t tacc = (wg == 0 ? t_dv : t_dk) + lane_addr;
#pragma unroll 1
      for (int cc = 0; cc < DP / 32 && cc * 32 < dim; ++cc) {
        uint32_t r[32];
        if (n > 0) {
          tmem_ld32(tacc + cc * 32, r);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int q = 0; q < 32; ++q) r[q] = 0u;
        }
        if (mine) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            if (cc * 32 + q * 8 < dim) {
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
  const int smem = L::BYTES + 1024;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int nblk = (p.max_pages * p.page_size + 127) / 128;
  dim3 grid(nblk, p.S, p.KVH);
  kern<<<grid, 384, smem, s>>>(m.q, m.dy, m.k, m.v, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_paged_history(const PagedMaps& m, const PagedParams& p, cudaStream_t s) {
  if (p.Dk <= 64) return launch_hist_t<64>(m, p, s);
  return launch_hist_t<128>(m, p, s);
}

}  // namespace attn
