// Paged history backward (GQA): dK and dV of every pool row, atomic-free.
//
// ruDNN src/paged_attention/ordered_kernel.rs (history_backward): for every
// physical token and KV head, sum over the links of its page, over the query
// rows of the linked sequence that see the token (t <= pos(r) when causal) and
// over the query heads of the KV group:
//   p  = exp(q.k * scale - lse),  ds = p * (dY.v - delta) * scale
//   dK += ds * q,   dV += p * dY
// A work item is 128 tokens (eight 16-token pages) of one sequence and one KV
// head; the same sums are tile products on tcgen05:
//   S^T  = K_T Q_c^T,  dP^T = V_T dY_c^T            (M=128 tokens, N=64 columns)
//   P^T  = exp2(S^T scale log2e - lse log2e)        written over S^T as bf16
//   dS^T = P^T (dP^T - delta)                        written over dP^T as bf16
//   dV_T += P^T dY_c,  dK_T += dS^T Q_c              (A operand from tensor memory)
// where a column c is one (query row, head of the group) pair.  The K/V tile is
// gathered page by page with TMA (3-D map over [slots, KVH, D]); pages past the
// sequence are fetched at an out-of-range coordinate, i.e. read as zeros
// without touching memory.  Passes: the item's own sequence first, then the
// other links of the pages it stores, by link index; consecutive pages linked
// from consecutive logical pages of one sequence share a pass (a shared prefix
// costs one pass per (sequence, block), not one per page).
//
// The kernel is persistent (one CTA per SM over the items, in a snake order):
// a scheduler warp works out each item's pages (eight lanes, one page each),
// links and tile count ahead of time into a four-slot item ring, and the K/V
// tiles are double-buffered, so that the next item's gather runs while the
// current item computes.
// Roles (384 threads): warp 0 TMA producer (K/V pages per item, Q/dY column
// tiles through a 3-stage ring (4 for D = 64), the columns' statistics through
// a 2-slot ring, fetched one tile ahead), warp 1 MMA issuer (whole warp,
// elect.sync), warp 2 item scheduler,
// warps 4..7 / 8..11 compute groups for even / odd tiles (each forms P and
// then dS of its tiles; group 0 stores dV, group 1 dK).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "paged_common.cuh"
#include "paged_launch.h"
#include "paged_pass.cuh"
#include "sm103.cuh"

namespace attn {
using namespace sm103;

namespace {

constexpr int kStatSlots = 2;
constexpr int kItemSlots = 4;  // items the scheduler prepares ahead

// Two K/V buffers (the next item's pages are gathered while this item runs),
// a ring of Q/dY column tiles, and the column statistics in their own
// two-slot ring.
template <int DP>
struct HistLayout {
  static constexpr int NCH = DP / 64;
  static constexpr int BT = 128, BC = 64;        // tokens x columns per step
  static constexpr int STAGES = DP == 64 ? 4 : 3;
  static constexpr int KV = NCH * BT * 128;
  static constexpr int QT = NCH * BC * 128;
  static constexpr int K_OFF = 0;
  static constexpr int V_OFF = K_OFF + KV;
  static constexpr int KVB = 2 * KV;                   // K/V buffer b at b * KVB
  static constexpr int Q_OFF = 2 * KVB;                // STAGES
  static constexpr int DY_OFF = Q_OFF + STAGES * QT;   // STAGES
  static constexpr int ST_OFF = DY_OFF + STAGES * QT;  // kStatSlots x {-L2, delta, pos} x 64 + pass info
  static constexpr int ST_STAGE = 3 * BC * 4 + 16;
  static constexpr int BYTES = ST_OFF + kStatSlots * ST_STAGE;
  // dynamic shared memory starts 1024-aligned after the static variables
  // (one 1 KiB granule): no alignment pad, checked at run time
  static_assert(BYTES + 1024 <= 232448, "the layout fits one CTA's shared memory");
  // TMEM: dV [0, DP), dK [DP, 2DP), S^T[2] and dP^T[2] 64 columns each
  static constexpr int T_S = 2 * DP, T_DP = 2 * DP + 128;
  static constexpr int TMEM_COLS = 512;
};

// One slot of the item ring: the item's pages and links, its tile count over
// all passes (n = -1: no more items).
struct ItemSlot {
  PageInfo pi;
  int s0, tb, g, n;
};

__device__ __forceinline__ bool drain_wait(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_test(bar, parity)) {
    if (global_timer_ns() - t0 > ATTN_WAIT_TIMEOUT_NS) return false;
  }
  return true;
}

__device__ __forceinline__ float4 lds_f4(const float* p) { return *reinterpret_cast<const float4*>(p); }

template <int DP>
__global__ void __launch_bounds__(384, 1)
    paged_history_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_dy,
                         const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                         const PagedParams p) {
  using L = HistLayout<DP>;
  constexpr int kStages = L::STAGES;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = smem_raw;
  // bar_acc / bar_acc_free: phases count items with tiles (as in the dense
  // persistent kernel); bar_kv[b] / bar_kv_free[b]: the items with tiles
  // that use K/V buffer b (item lv uses buffer lv & 1); bar_item_*: every item
  __shared__ uint64_t bar_item_full[kItemSlots], bar_item_empty[kItemSlots], bar_kv[2], bar_kv_free[2],
      bar_full[kStages], bar_empty[kStages], bar_st_full[kStatSlots], bar_st_empty[kStatSlots], bar_s_full[2],
      bar_dp_full[2], bar_p_full[2], bar_ds_full[2], bar_acc, bar_acc_free;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag;
  __shared__ ItemSlot items[kItemSlots];
  if (smem_addr(smem_raw) & 1023u) {  // uniform: the swizzled tiles need 1024-byte alignment
    if (threadIdx.x == 0 && p.err) atomicOr(p.err, DEV_ERR_LAYOUT);
    return;
  }

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int RT = L::BC / p.G;  // query rows per step
  const Abort ab{&abort_flag, p.err};
  const int nblk = (p.max_pages * p.page_size + 127) / 128;
  const int total = p.KVH * nblk * p.S;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int s = 0; s < kItemSlots; ++s) {
      mbar_init(&bar_item_full[s], 1);
      mbar_init(&bar_item_empty[s], 10);  // producer, MMA warp, 8 compute warps
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bar_s_full[s], 1);
      mbar_init(&bar_dp_full[s], 1);
      mbar_init(&bar_p_full[s], 4);
      mbar_init(&bar_ds_full[s], 4);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bar_kv[b], 1);
      mbar_init(&bar_kv_free[b], 1);
    }
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bar_full[s], 1);
      mbar_init(&bar_empty[s], 1);
    }
    for (int s = 0; s < kStatSlots; ++s) {
      mbar_init(&bar_st_full[s], 1);
      mbar_init(&bar_st_empty[s], 4);  // the four warps of the tile's compute group
    }
    mbar_init(&bar_acc, 1);
    mbar_init(&bar_acc_free, 8);
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
  const uint32_t t_dv = tmem, t_dk = tmem + DP;
  const int oob_slot = p.num_pages * p.page_size;  // out-of-range coordinate: TMA fills zeros

  // every role but the scheduler walks the item ring in order
  auto item_wait = [&](int ii) -> bool {
    return mbar_wait_warp(&bar_item_full[ii % kItemSlots], (ii / kItemSlots) & 1, ab);
  };
  auto item_done = [&](int ii) {
    __syncwarp();
    if (lane == 0) mbar_arrive(&bar_item_empty[ii % kItemSlots]);
  };

  if (warp == 2) {
    // ------------------------------------------------------------ item scheduler
    // the CTA's items: index r*G + c (r*G + G-1-c in odd rounds), KV head
    // fastest, so that the heads of one block of pages run side by side
    int ii = 0;
    bool ok = true;
    for (int r = 0; ok; ++r) {
      const int base = r * static_cast<int>(gridDim.x);
      int idx = base + ((r & 1) ? static_cast<int>(gridDim.x) - 1 - static_cast<int>(blockIdx.x)
                                : static_cast<int>(blockIdx.x));
      const bool last_round = base + static_cast<int>(gridDim.x) >= total;
      if (base >= total) break;
      if (idx < total) {
        const int g = idx % p.KVH, tb = (idx / p.KVH) % nblk, s0 = idx / (p.KVH * nblk);
        const int npg = pages_of(seq_len_of(p, s0), p.page_size);
        if (tb * 8 < npg) {
          if (ii >= kItemSlots &&
              !(ok = mbar_wait_warp(&bar_item_empty[ii % kItemSlots], ((ii / kItemSlots) - 1) & 1, ab)))
            break;
          ItemSlot& it = items[ii % kItemSlots];
          // lanes 0..7 fetch the eight pages' entries side by side
          const int st = lane < 8 ? fill_page_entry(p, s0, tb, npg, lane, &it.pi) : 0;
          const int any = __any_sync(0xffffffffu, st != 0);
          __syncwarp();
          // a block whose pages are all stored by other items (their owners)
          // has nothing to write
          if (any) {
            if (lane == 0) {
              PassIter pit{&p, &it.pi, s0, tb};
              int n = 0;
              if (pit.begin(RT)) {
                do n += pit.ntiles;
                while (pit.next_pass(RT));
              }
              it.s0 = s0;
              it.tb = tb;
              it.g = g;
              it.n = n;
              mbar_arrive(&bar_item_full[ii % kItemSlots]);
            }
            __syncwarp();
            ++ii;
          }
        }
      }
      if (last_round) break;
    }
    // end marker
    if (ok && (ii < kItemSlots ||
               mbar_wait_warp(&bar_item_empty[ii % kItemSlots], ((ii / kItemSlots) - 1) & 1, ab))) {
      if (lane == 0) {
        items[ii % kItemSlots].n = -1;
        mbar_arrive(&bar_item_full[ii % kItemSlots]);
      }
    }
  } else if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_map(&tm_q);
      tma_prefetch_map(&tm_dy);
      tma_prefetch_map(&tm_k);
      tma_prefetch_map(&tm_v);
    }
    int last_use[kStages];
    for (int i = 0; i < kStages; ++i) last_use[i] = -1;
    bool ok = true;
    int gt = 0, lv = 0;  // global tile counter, items with tiles
    // column statistics of a tile (two columns per lane) and its pass's token
    // mapping, fetched one tile ahead
    float f_lse[2], f_dl[2];
    int f_pos[2], f_info[4];
    auto fetch = [&](const PassIter& x, int g) {
      const int row0 = x.r_begin + x.tile * RT;
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int c = lane + 32 * i;
        const int r = row0 + c / p.G;
        const bool in = r < x.r_end;
        const int64_t idx = static_cast<int64_t>(in ? r : 0) * p.H + g * p.G + c % p.G;
        f_lse[i] = in ? p.lse[idx] : -__int_as_float(0x7f800000);
        f_dl[i] = in ? p.delta[idx] : 0.f;
        f_pos[i] = in ? (p.causal ? p.q_pos[r] : 0x7fffffff) : -1;
      }
      f_info[0] = x.tbase;
      f_info[1] = x.ra;
      f_info[2] = x.rb;
      f_info[3] = seq_len_of(p, x.seq);
    };
    for (int ii = 0; ok; ++ii) {
      if (!(ok = item_wait(ii))) break;
      const ItemSlot& it = items[ii % kItemSlots];
      const int n = it.n;
      if (n < 0) break;
      if (n > 0) {
        const int g = it.g;
        // buffer lv & 1: free once item lv - 2's products are done
        const int kb = lv & 1;
        if (lv >= 2 && !(ok = mbar_wait(&bar_kv_free[kb], ((lv >> 1) - 1) & 1, ab))) break;
        if (lane == 0) {
          uint8_t* kvb = sm + kb * L::KVB;
          mbar_arrive_expect_tx(&bar_kv[kb], 2 * L::KV);
          for (int j = 0; j < 8; ++j) {
            const int slot = it.pi.phys[j] >= 0 ? it.pi.phys[j] * p.page_size : oob_slot;
            for (int c = 0; c < L::NCH; ++c) {
              tma_load_3d(kvb + L::K_OFF + c * (L::BT * 128) + j * 16 * 128, &tm_k, &bar_kv[kb], c * 64, g, slot);
              tma_load_3d(kvb + L::V_OFF + c * (L::BT * 128) + j * 16 * 128, &tm_v, &bar_kv[kb], c * 64, g, slot);
            }
          }
        }
        PassIter pit{&p, &it.pi, it.s0, it.tb};
        pit.begin(RT);
        fetch(pit, g);
        for (int t = 0; t < n && ok; ++t) {
          const int gg = gt + t, s = gg % kStages;
          if (gg >= kStages && !(ok = mbar_wait(&bar_empty[s], ((gg / kStages) - 1) & 1, ab))) break;
          const int row0 = pit.r_begin + pit.tile * RT;
          if (lane == 0) {
            mbar_arrive_expect_tx(&bar_full[s], 2 * L::QT);
            for (int c = 0; c < L::NCH; ++c) {
              tma_load_3d(sm + L::Q_OFF + s * L::QT + c * (L::BC * 128), &tm_q, &bar_full[s], c * 64, g * p.G, row0);
              tma_load_3d(sm + L::DY_OFF + s * L::QT + c * (L::BC * 128), &tm_dy, &bar_full[s], c * 64, g * p.G,
                          row0);
            }
          }
          // the tile's column statistics, after its copies are issued: slot
          // gg mod 2 is free once its group has formed dS of tile gg - 2
          const int ss = gg % kStatSlots;
          if (gg >= kStatSlots && !(ok = mbar_wait(&bar_st_empty[ss], ((gg / kStatSlots) - 1) & 1, ab))) break;
          uint8_t* st = sm + L::ST_OFF + ss * L::ST_STAGE;
          float* snl = reinterpret_cast<float*>(st);
          float* sdl = snl + L::BC;
          int* spos = reinterpret_cast<int*>(sdl + L::BC);
          int* sinfo = spos + L::BC;
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            const int c = lane + 32 * i;
            const bool live = f_lse[i] != -__int_as_float(0x7f800000);
            snl[c] = live ? -f_lse[i] * 1.4426950408889634f : -__int_as_float(0x7f800000);
            sdl[c] = live ? f_dl[i] : 0.f;
            spos[c] = live ? f_pos[i] : -1;
          }
          if (lane == 0) {
            sinfo[0] = f_info[0];
            sinfo[1] = f_info[1];
            sinfo[2] = f_info[2];
            sinfo[3] = f_info[3];
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&bar_st_full[ss]);
          last_use[s] = gg;
          if (t + 1 < n) {
            pit.advance(RT);
            fetch(pit, g);
          }
        }
        gt += n;
        ++lv;
      }
      item_done(ii);
    }
    if (lane == 0) {
      for (int s = 0; s < kStages; ++s)
        if (last_use[s] >= 0) drain_wait(&bar_full[s], (last_use[s] / kStages) & 1);
      for (int u = max(lv - 2, 0); u < lv; ++u) drain_wait(&bar_kv[u & 1], (u >> 1) & 1);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // the whole warp runs this role (warp-uniform); elected lanes issue
    constexpr uint32_t id_s = idesc_bf16(128, 64, false, false);
    constexpr uint32_t id_acc = idesc_bf16(128, DP, false, true);
    const uint64_t dK0 = sdesc_sw128(smem_addr(sm + L::K_OFF), 16, 1024);
    const uint64_t dV0 = sdesc_sw128(smem_addr(sm + L::V_OFF), 16, 1024);
    uint64_t dK = dK0, dV = dV0;  // the current item's K/V buffer
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
    auto issue_s = [&](int gg) {
      issue_xt(tmem + L::T_S + (gg & 1) * 64, dK, sdesc_add(dQ0, (gg % kStages) * L::QT));
      mma_commit_w(&bar_s_full[gg & 1]);
    };
    auto issue_dp = [&](int gg) {
      issue_xt(tmem + L::T_DP + (gg & 1) * 64, dV, sdesc_add(dDY0, (gg % kStages) * L::QT));
      mma_commit_w(&bar_dp_full[gg & 1]);
    };
    bool ok = true;
    int g0 = 0, lv = 0;
    for (int ii = 0; ok; ++ii) {
      if (!(ok = item_wait(ii))) break;
      const int n = items[ii % kItemSlots].n;
      if (n < 0) break;
      if (n > 0) {
        const int kb = lv & 1;
        if (!(ok = mbar_wait_warp(&bar_kv[kb], (lv >> 1) & 1, ab))) break;
        dK = sdesc_add(dK0, kb * L::KVB);
        dV = sdesc_add(dV0, kb * L::KVB);
        // the first score and dP tiles of this item go while the epilogue of
        // the previous item still reads dV and dK
        for (int t = 0; t < 2 && t < n && ok; ++t) {
          if (!(ok = mbar_wait_warp(&bar_full[(g0 + t) % kStages], ((g0 + t) / kStages) & 1, ab))) break;
          tc_fence_after();
          issue_s(g0 + t);
          issue_dp(g0 + t);
        }
        if (!ok) break;
        if (n <= 2) mma_commit_w(&bar_kv_free[kb]);
        if (lv > 0 && !(ok = mbar_wait_warp(&bar_acc_free, (lv - 1) & 1, ab))) break;
        tc_fence_after();
        // Per tile g: dV(g) once P(g) is in; then S(g+2) and dK(g) in
        // whichever order their inputs arrive; then dP(g+2).  S(g+2)
        // overwrites P(g), which dV(g) (earlier in the same pipe) consumes,
        // and S(g), which the group finished reading before it handed P(g)
        // over; dP(g+2) overwrites dS(g) and dP(g), read by dK(g) and by the
        // group before dS(g) was handed over.
        for (int t = 0; t < n && ok; ++t) {
          const int g = g0 + t, s = g % kStages, bb = g & 1;
          if (!(ok = mbar_wait_warp(&bar_p_full[bb], (g >> 1) & 1, ab))) break;
          tc_fence_after();
          issue_acc(t_dv, tmem + L::T_S + bb * 64, sdesc_add(dDYm0, s * L::QT), t == 0);
          bool s_next = t + 2 < n, k_now = true;
          PollBudget pb;
          while (s_next || k_now) {
            if (s_next && mbar_test_warp(&bar_full[(g + 2) % kStages], ((g + 2) / kStages) & 1)) {
              tc_fence_after();
              issue_s(g + 2);
              s_next = false;
            }
            if (k_now && mbar_test_warp(&bar_ds_full[bb], (g >> 1) & 1)) {
              tc_fence_after();
              issue_acc(t_dk, tmem + L::T_DP + bb * 64, sdesc_add(dQm0, s * L::QT), t == 0);
              mma_commit_w(&bar_empty[s]);
              k_now = false;
            }
            if ((s_next || k_now) && !(ok = pb.check(ab))) break;
          }
          if (!ok) break;
          if (t + 2 < n) {
            issue_dp(g + 2);
            if (t + 3 == n) mma_commit_w(&bar_kv_free[kb]);  // the item's last S and dP are issued
          }
        }
        if (!ok) break;
        mma_commit_w(&bar_acc);
        g0 += n;
        ++lv;
      }
      item_done(ii);
    }
    if (lv > 0) drain_wait(&bar_acc, (lv - 1) & 1);
    __syncwarp();
  } else if (warp >= 4) {
    const int sg = (warp - 4) >> 2;  // compute group: tiles (and S/dP buffers) of parity sg
    const int lg = warp & 3;
    const int row = lg * 32 + lane;  // token row inside the block == TMEM lane
    const uint32_t lane_addr = static_cast<uint32_t>(lg * 32) << 16;
    bool ok = true;
    int g0 = 0, lv = 0;
    for (int ii = 0; ok; ++ii) {
      if (!(ok = item_wait(ii))) break;
      const ItemSlot& it = items[ii % kItemSlots];
      const int n = it.n;
      if (n < 0) break;
      for (int t = ((g0 & 1) == sg) ? 0 : 1; t < n && ok; t += 2) {
        const int g = g0 + t, bb = g & 1, ss = g % kStatSlots;
        if (!(ok = mbar_wait_warp(&bar_st_full[ss], (g / kStatSlots) & 1, ab))) break;
        const uint8_t* st = sm + L::ST_OFF + ss * L::ST_STAGE;
        const float* snl = reinterpret_cast<const float*>(st);
        const float* sdl = snl + L::BC;
        const int* spos = reinterpret_cast<const int*>(sdl + L::BC);
        const int* sinfo = spos + L::BC;
        const int tok = sinfo[0] + row;
        const bool tok_ok = row >= sinfo[1] && row < sinfo[2] && tok >= 0 && tok < sinfo[3];
        if (!(ok = mbar_wait_warp(&bar_s_full[bb], (g >> 1) & 1, ab))) break;
        tc_fence_after();
        // ---------------------------------------------------- S^T -> P^T
        // two halves of 32 columns: half hf reads S^T columns [32hf, 32hf+32)
        // and writes P^T (bf16 pairs) to columns [16hf, 16hf+16), which half
        // 0 has already read
        const uint32_t tS = tmem + L::T_S + bb * 64 + lane_addr;
        const uint64_t sl2 = f2_pack(p.scale_log2, p.scale_log2);
        uint32_t pw[32];
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          uint32_t sr[32];
          tmem_ld32(tS + 32 * hf, sr);
          tmem_ld_wait();
#pragma unroll
          for (int c4 = 0; c4 < 8; ++c4) {
            const int c0 = 32 * hf + 4 * c4;
            const float4 nl = lds_f4(snl + c0);
            const int4 ps = *reinterpret_cast<const int4*>(spos + c0);
            float x0, x1, x2, x3;
            f2_split(f2_fma(f2_pack_u(sr[4 * c4], sr[4 * c4 + 1]), sl2, f2_pack(nl.x, nl.y)), x0, x1);
            f2_split(f2_fma(f2_pack_u(sr[4 * c4 + 2], sr[4 * c4 + 3]), sl2, f2_pack(nl.z, nl.w)), x2, x3);
            const float p0 = (tok_ok && tok <= ps.x) ? ex2_approx(x0) : 0.f;
            const float p1 = (tok_ok && tok <= ps.y) ? ex2_approx(x1) : 0.f;
            const float p2 = (tok_ok && tok <= ps.z) ? ex2_approx(x2) : 0.f;
            const float p3 = (tok_ok && tok <= ps.w) ? ex2_approx(x3) : 0.f;
            pw[16 * hf + 2 * c4] = pack_bf16x2(p0, p1);
            pw[16 * hf + 2 * c4 + 1] = pack_bf16x2(p2, p3);
          }
          tmem_st16(tS + 16 * hf, *reinterpret_cast<const uint32_t(*)[16]>(pw + 16 * hf));
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar_p_full[bb]);
        // ---------------------------------------------------- dP^T, P^T -> dS^T
        if (!(ok = mbar_wait_warp(&bar_dp_full[bb], (g >> 1) & 1, ab))) break;
        tc_fence_after();
        const uint32_t tDP = tmem + L::T_DP + bb * 64 + lane_addr;
        // a masked entry has P = 0 and takes dS = 0 by select: dP of a tail or
        // unowned slot may be NaN
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          uint32_t dr[32], dsw[16];
          tmem_ld32(tDP + 32 * hf, dr);
          tmem_ld_wait();
#pragma unroll
          for (int c4 = 0; c4 < 8; ++c4) {
            const float4 d4 = lds_f4(sdl + 32 * hf + 4 * c4);
            const float dv4[4] = {d4.x, d4.y, d4.z, d4.w};
            float ds[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const uint32_t w = pw[16 * hf + 2 * c4 + (e >> 1)];
              const float pe = __uint_as_float((e & 1) ? (w & 0xffff0000u) : (w << 16));
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
        if (lane == 0) {
          mbar_arrive(&bar_ds_full[bb]);
          mbar_arrive(&bar_st_empty[ss]);
        }
      }
      if (!ok) break;
      if (n > 0) {
        if (!(ok = mbar_wait_warp(&bar_acc, lv & 1, ab))) break;
        tc_fence_after();
      }
      // ---------------------------------------------------------- epilogue
      // group 0 stores dV, group 1 dK (times the softmax scale), each row of
      // a page this item stores; rows of tokens no pass saw are zero.  Tensor
      // memory goes back (acc_free) once the last chunk is in registers.
      const int j = row >> 4;
      const bool mine = it.pi.store[j] != 0;
      const bool want = sg == 0 ? (p.wrt & 4u) != 0 : (p.wrt & 2u) != 0;
      const int dim = sg == 0 ? p.Dv : p.Dk;
      const int64_t prow = (static_cast<int64_t>(it.pi.phys[j]) * p.page_size + (row & 15)) * p.KVH + it.g;
      __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(sg == 0 ? p.dv_pool : p.dk_pool) + prow * dim;
      const float f = sg == 0 ? 1.f : p.scale;
      const uint32_t tacc = (sg == 0 ? t_dv : t_dk) + lane_addr;
#pragma unroll 1
      for (int cc = 0; want && cc < DP / 32 && cc * 32 < dim; ++cc) {  // warp-uniform (tensor-memory loads)
        uint32_t r[32];
        if (n > 0) {
          tmem_ld32(tacc + cc * 32, r);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int q = 0; q < 32; ++q) r[q] = 0u;
        }
        if (mine) store_row32_bf16(out + cc * 32, r, f, dim - cc * 32);
      }
      if (n > 0) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar_acc_free);
        g0 += n;
        ++lv;
      }
      item_done(ii);
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
  const int smem = max(L::BYTES, kSmemOneCtaPerSm);  // all 512 TMEM columns: one CTA per SM
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  const int nblk = (p.max_pages * p.page_size + 127) / 128;
  const int64_t items = static_cast<int64_t>(p.KVH) * nblk * p.S;
  const int grid = static_cast<int>(items < sms ? items : sms);  // persistent: one CTA per SM
  if (grid <= 0) return cudaSuccess;
  kern<<<grid, 384, smem, s>>>(m.q, m.dy, m.k, m.v, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_paged_history(const PagedMaps& m, const PagedParams& p, cudaStream_t s) {
  if (p.Dk <= 64) return launch_hist_t<64>(m, p, s);
  return launch_hist_t<128>(m, p, s);
}

}  // namespace attn
