// Paged MLA row statistics on tcgen05: lse[r, h] and delta[r, h] for every
// packed query row and head, by a forward sweep over the row's sequence pages.
//
// ruDNN src/paged_attention/ordered_kernel.rs reads per (row, head) the
// statistics "computed once by the query kernel" (max, denominator, delta);
// this kernel produces them in LSE form, with
//   s_t = scale (q . k_lat[t] + qp . k_pos[t]),   dP_t = dY . k_lat[t]
//   lse = log sum_t exp(s_t),   delta = sum_t P_t dP_t  (P_t = exp(s_t - lse))
// over the visible tokens t (t < len, and t <= pos(r) when causal); delta =
// sum_t P_t dP_t equals dY . O for O = sum_t P_t k_lat[t] (the latent is the
// value).  A row with no visible token gets lse = -inf and delta = 0.
//
// One CTA per (KV head, tile of 128 columns = 128/G query rows x the G heads
// of the group); the sweep runs over 64-token tiles (four pages gathered by
// TMA) with, per tile,
//   S  = Q K^T   [128 x 64]: A = Q staged in tensor memory (576 dims as bf16
//                pairs, 288 columns), B = K chunks from shared memory
//   dP = dY K_lat^T          : A = dY resident in shared memory (128 KiB)
// and the compute warps (thread = column) keep an online maximum, the
// denominator and the dP-weighted sum.  K arrives in chunks of [64 tokens x 64
// dims] through a 6-stage ring of two chunks per stage.  Tensor memory: Q
// [0, 288), S[2] [288, 416), dP [416, 480) (single buffer: the group reads
// the whole dP tile into registers before it works on S).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "paged_common.cuh"
#include "paged_launch.h"
#include "sm103.cuh"

namespace attn {
using namespace sm103;

namespace {

constexpr int kLat = 512, kPos = 64;
constexpr int BC = 128;                 // columns per CTA
constexpr int BT = 64;                  // tokens per tile (4 pages of 16)
constexpr int kStages = 6;
constexpr int QCH = BC * 128;           // Q / dY chunk [128 columns][64 dims], 16 KiB
constexpr int KCH = BT * 128;           // K chunk [64 tokens][64 dims], 8 KiB
constexpr int STAGE = 2 * KCH;
constexpr int DY_OFF = 0;               // 8 chunks (Q latent chunks while staging)
constexpr int RING_OFF = DY_OFF + 8 * QCH;  // 4 stages (the Qp chunk while staging)
constexpr int BYTES = RING_OFF + kStages * STAGE;
static_assert(kStages * STAGE >= QCH, "the Qp chunk is staged through the ring");
// dynamic shared memory starts 1024-aligned after the static variables (at
// most 2 KiB here): no alignment pad, checked at run time
static_assert(BYTES + 2048 <= 232448, "the layout fits one CTA's shared memory");
constexpr int T_Q = 0, T_S = 288, T_DP = 416, TMEM_COLS = 512;
constexpr float kRescaleThreshold = 8.0f;

__device__ __forceinline__ bool drain_wait(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_test(bar, parity)) {
    if (global_timer_ns() - t0 > ATTN_WAIT_TIMEOUT_NS) return false;
  }
  return true;
}

// Registers written by tcgen05.ld are valid only after tcgen05.wait::ld.
__device__ __forceinline__ void reg_fence32(uint32_t (&r)[32]) {
#pragma unroll
  for (int i = 0; i < 32; ++i) asm volatile("" : "+r"(r[i]));
}

__global__ void __launch_bounds__(384, 1)
    mla_stats_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_qp,
                        const __grid_constant__ CUtensorMap tm_dy, const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_kp, const PagedParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = smem_raw;
  __shared__ uint64_t bar_q, bar_q_staged, bar_dy, bar_full[kStages], bar_empty[kStages], bar_s_full[2],
      bar_s_read[2], bar_dp_full, bar_dp_read;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag, ntok_sh, seq_sh, r0_sh;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // block x = tile * KVH + g: row tile `tile` of the sequences in dispatch
  // order (longest first), KV head g
  const int g = static_cast<int>(blockIdx.x % p.KVH);
  const int G = p.G, RT = BC / G;
  if (threadIdx.x < 32) {  // warp 0
    int sq, r0;
    row_tile_at_warp(p, static_cast<int>(blockIdx.x / p.KVH), RT, &sq, &r0);
    if (threadIdx.x == 0) {
      seq_sh = sq;
      r0_sh = r0;
    }
  }
  __syncthreads();
  const int s0 = seq_sh, r0 = r0_sh;
  if (s0 < 0) return;  // past the last row tile (uniform exit)
  if (smem_addr(smem_raw) & 1023u) {  // uniform: the swizzled tiles need 1024-byte alignment
    if (threadIdx.x == 0 && p.err) atomicOr(p.err, DEV_ERR_LAYOUT);
    return;
  }
  const int re = row_end_of(p, s0);
  const int len = seq_len_of(p, s0);
  const int npg = pages_of(len, p.page_size);
  const Abort ab{&abort_flag, p.err};
  const int oob_slot = p.num_pages * p.page_size;  // out-of-range coordinate: TMA fills zeros
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bar_q, 1);
    mbar_init(&bar_q_staged, 8);
    mbar_init(&bar_dy, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bar_full[s], 1);
      mbar_init(&bar_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bar_s_full[s], 1);
      mbar_init(&bar_s_read[s], 4);
    }
    mbar_init(&bar_dp_full, 1);
    mbar_init(&bar_dp_read, 4);
    mbar_fence_init();
    int ntok = len;
    if (p.causal) {  // tokens past the largest position of the CTA's rows are never visible
      int mp = -1;
      for (int r = r0; r < r0 + RT && r < re; ++r) mp = max(mp, p.q_pos[r]);
      ntok = min(len, mp + 1);
    }
    ntok_sh = max(ntok, 0);
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base_sh, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  const int n = (ntok_sh + BT - 1) / BT;  // token tiles

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    bool ok = true;
    int last_use[kStages];
    for (int i = 0; i < kStages; ++i) last_use[i] = -1;
    if (n > 0) {
      if (lane == 0) {
        tma_prefetch_map(&tm_q);
        tma_prefetch_map(&tm_qp);
        tma_prefetch_map(&tm_dy);
        tma_prefetch_map(&tm_k);
        tma_prefetch_map(&tm_kp);
        // Q (latent chunks into the dY slots, Qp into the ring) for staging
        mbar_arrive_expect_tx(&bar_q, 9 * QCH);
        for (int c = 0; c < 8; ++c) tma_load_3d(sm + DY_OFF + c * QCH, &tm_q, &bar_q, c * 64, g * G, r0);
        tma_load_3d(sm + RING_OFF, &tm_qp, &bar_q, 0, g * G, r0);
      }
      // the staging warps are done with those slots: dY, then the K ring
      ok = mbar_wait(&bar_q_staged, 0, ab);
      if (ok && lane == 0) {
        mbar_arrive_expect_tx(&bar_dy, 8 * QCH);
        for (int c = 0; c < 8; ++c) tma_load_3d(sm + DY_OFF + c * QCH, &tm_dy, &bar_dy, c * 64, g * G, r0);
      }
    }
    // K chunks of token tile t: (0, 1), (2, 3), (4, 5), (6, 7), (position)
    int q = 0;
    for (int t = 0; t < n && ok; ++t) {
      int slot[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int lp = 4 * t + j;
        slot[j] = oob_slot;
        if (lp < npg) {
          const int ph = p.page_table[static_cast<int64_t>(s0) * p.max_pages + lp];
          if (ph >= 0 && ph < p.num_pages) slot[j] = ph * p.page_size;
        }
      }
      for (int c0 = 0; c0 < 9 && ok; c0 += 2, ++q) {
        const int s = q % kStages;
        if (q >= kStages && !(ok = mbar_wait(&bar_empty[s], ((q / kStages) - 1) & 1, ab))) break;
        const int nch = c0 < 8 ? 2 : 1;
        if (lane == 0) {
          mbar_arrive_expect_tx(&bar_full[s], nch * KCH);
          for (int k = 0; k < nch; ++k) {
            const int c = c0 + k;
            for (int j = 0; j < 4; ++j) {
              uint8_t* dst = sm + RING_OFF + s * STAGE + k * KCH + j * 16 * 128;
              if (c < 8)
                tma_load_3d(dst, &tm_k, &bar_full[s], c * 64, g, slot[j]);
              else
                tma_load_3d(dst, &tm_kp, &bar_full[s], 0, g, slot[j]);
            }
          }
        }
        last_use[s] = q;
      }
    }
    if (lane == 0) {
      for (int s = 0; s < kStages; ++s)
        if (last_use[s] >= 0) drain_wait(&bar_full[s], (last_use[s] / kStages) & 1);
      if (n > 0) {
        drain_wait(&bar_q, 0);
        drain_wait(&bar_dy, 0);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (n > 0) {
      constexpr uint32_t id = idesc_bf16(128, BT, false, false);  // K-major A and B
      const uint64_t dDY0 = sdesc_sw128(smem_addr(sm + DY_OFF), 16, 1024);
      const uint64_t dR0 = sdesc_sw128(smem_addr(sm + RING_OFF), 16, 1024);
      bool ok = mbar_wait_warp(&bar_q_staged, 0, ab) && mbar_wait_warp(&bar_dy, 0, ab);
      tc_fence_after();
      int q = 0;
      for (int t = 0; t < n && ok; ++t) {
        const int bb = t & 1;
        // S(t) overwrites S(t - 2): wait until its group has read it
        if (t >= 2 && !(ok = mbar_wait_warp(&bar_s_read[bb], ((t - 2) >> 1) & 1, ab))) break;
        bool dp_free = t == 0;
        for (int c0 = 0; c0 < 9 && ok; c0 += 2, ++q) {
          const int s = q % kStages;
          if (!mbar_test_warp(&bar_full[s], (q / kStages) & 1) &&
              !(ok = mbar_wait_warp(&bar_full[s], (q / kStages) & 1, ab)))
            break;
          tc_fence_after();
          for (int k = 0; k < 2 && c0 + k < 9; ++k) {
            const int c = c0 + k;
            const uint64_t bk = sdesc_add(dR0, s * STAGE + k * KCH);
            // S += Q_c K_c^T (A from tensor memory: chunk c = columns 32c..)
            const uint32_t ds = tmem + T_S + bb * BT;
            if (c == 0)
              mma_ts_w<false>(ds, tmem + T_Q + 32 * c, bk, id);
            else
              mma_ts_w<true>(ds, tmem + T_Q + 32 * c, bk, id);
#pragma unroll
            for (int kk = 1; kk < 4; ++kk) mma_ts_w<true>(ds, tmem + T_Q + 32 * c + 8 * kk, sdesc_add(bk, kk * 32), id);
            if (c < 8) {
              // dP += dY_c K_c^T; dP(t) overwrites dP(t - 1), read by now
              if (!dp_free) {
                if (!(ok = mbar_wait_warp(&bar_dp_read, (t - 1) & 1, ab))) break;
                tc_fence_after();
                dp_free = true;
              }
              const uint64_t a = sdesc_add(dDY0, c * QCH);
              if (c == 0)
                mma_ss_w<false>(tmem + T_DP, a, bk, id);
              else
                mma_ss_w<true>(tmem + T_DP, a, bk, id);
#pragma unroll
              for (int kk = 1; kk < 4; ++kk)
                mma_ss_w<true>(tmem + T_DP, sdesc_add(a, kk * 32), sdesc_add(bk, kk * 32), id);
            }
          }
          if (!ok) break;
          mma_commit_w(&bar_empty[s]);
        }
        if (!ok) break;
        mma_commit_w(&bar_s_full[bb]);
        mma_commit_w(&bar_dp_full);
      }
      // the last commits arrive before the CTA leaves
      const int nq = n * 5;
      for (int qq = max(0, nq - kStages); qq < nq; ++qq) drain_wait(&bar_empty[qq % kStages], (qq / kStages) & 1);
    }
    __syncwarp();
  } else if (warp >= 4) {
    const int sg = (warp - 4) >> 2;  // compute group: token tiles of parity sg
    const int lg = warp & 3;
    const int col = lg * 32 + lane;  // column of the tile == TMEM lane
    const uint32_t lane_addr = static_cast<uint32_t>(lg * 32) << 16;
    const int r = r0 + col / G;
    const bool col_ok = r < re;
    const int pos = col_ok ? (p.causal ? p.q_pos[r] : 0x7fffffff) : -1;
    const float kInf = __int_as_float(0x7f800000);
    bool ok = n > 0;
    if (n > 0) {
      // stage Q in tensor memory as bf16 pairs: this group's chunks
      ok = mbar_wait_warp(&bar_q, 0, ab);
      if (ok) {
        for (int c = sg; c < 9; c += 2) {
          const uint8_t* src = sm + (c < 8 ? DY_OFF + c * QCH : RING_OFF);
          uint32_t w[32];
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const uint4 v = *reinterpret_cast<const uint4*>(src + sw128_offset(col, j));
            w[4 * j] = v.x;
            w[4 * j + 1] = v.y;
            w[4 * j + 2] = v.z;
            w[4 * j + 3] = v.w;
          }
          tmem_st32(tmem + T_Q + 32 * c + lane_addr, w);
        }
        tmem_st_wait();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_q_staged);
    }
    float m2 = -kInf, l = 0.f, dsum = 0.f;
    for (int t = sg; t < n && ok; t += 2) {
      const int bb = t & 1;
      if (!(ok = mbar_wait_warp(&bar_s_full[bb], (t >> 1) & 1, ab))) break;
      // the dP commit follows the S commit of the same tile, so this covers both
      if (!(ok = mbar_wait_warp(&bar_dp_full, t & 1, ab))) break;
      tc_fence_after();
      // all of dP(t) into registers, then hand the buffer back
      uint32_t dr[64];
      tmem_ld32(tmem + T_DP + lane_addr, *reinterpret_cast<uint32_t(*)[32]>(dr));
      tmem_ld32(tmem + T_DP + 32 + lane_addr, *reinterpret_cast<uint32_t(*)[32]>(dr + 32));
      tmem_ld_wait();
#pragma unroll
      for (int i = 0; i < 64; ++i) asm volatile("" : "+r"(dr[i]));
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_dp_read);
      // visible tokens of this column in the tile: [0, hi) tile-local
      const int tok0 = t * BT;
      const int lim = pos >= len ? len : pos + 1;  // pos may be INT_MAX (no causal mask)
      const int hi = col_ok ? min(lim - tok0, BT) : 0;
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        uint32_t sr[32];
        tmem_ld32(tmem + T_S + bb * BT + 32 * hf + lane_addr, sr);
        tmem_ld_wait();
        reg_fence32(sr);
        if (hf == 1) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bar_s_read[bb]);
        }
        float x[32];
        float mt = -kInf;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          x[i] = (32 * hf + i < hi) ? __uint_as_float(sr[i]) * p.scale_log2 : -kInf;
          mt = fmaxf(mt, x[i]);
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
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const float pe = ex2_approx(x[i] - m2);  // 0 for a hidden token (x = -inf)
            l += pe;
            // a hidden token's dP may be NaN (tail or unowned slot): select, not multiply
            dsum = (32 * hf + i < hi) ? fmaf(pe, __uint_as_float(dr[32 * hf + i]), dsum) : dsum;
          }
        }
      }
    }
    // merge the two groups' statistics of each column
    __shared__ float mg[3][BC];
    if (sg == 1) {
      mg[0][col] = m2;
      mg[1][col] = l;
      mg[2][col] = dsum;
    }
    asm volatile("bar.sync 1, 256;" ::: "memory");  // warps 4..11
    if (sg == 0 && ok && col_ok) {
      const float mb = mg[0][col], lb = mg[1][col], db = mg[2][col];
      const float mm = fmaxf(m2, mb);
      float lt = 0.f, dt = 0.f;
      if (mm > -kInf) {
        const float a0 = m2 > -kInf ? ex2_approx(m2 - mm) : 0.f;
        const float a1 = mb > -kInf ? ex2_approx(mb - mm) : 0.f;
        lt = l * a0 + lb * a1;
        dt = dsum * a0 + db * a1;
      }
      const size_t idx = static_cast<size_t>(r) * p.H + g * G + col % G;
      p.lse_out[idx] = lt > 0.f ? (mm + __log2f(lt)) * 0.6931471805599453f : -kInf;
      p.delta_out[idx] = lt > 0.f ? dt / lt : 0.f;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

}  // namespace

bool mla_stats_tc_supported(const PagedParams& p) {
  return p.Dk == kLat && p.Dp == kPos && p.page_size == 16 && p.G >= 1 && p.G <= BC && BC % p.G == 0;
}

cudaError_t launch_paged_mla_stats_tc(const PagedMlaMaps& m, const PagedParams& p, cudaStream_t s) {
  if (p.Nq == 0 || p.S == 0) return cudaSuccess;
  const int smem = BYTES;
  static_assert(BYTES >= kSmemOneCtaPerSm, "all 512 TMEM columns: one CTA per SM");
  cudaError_t e = cudaFuncSetAttribute(mla_stats_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  // an upper bound on the row tiles of all sequences; each CTA finds its own
  const int RT = BC / p.G;
  dim3 grid(static_cast<unsigned>((static_cast<int64_t>(p.Nq) / RT + p.S + 1) * p.KVH));
  mla_stats_tc_kernel<<<grid, 384, smem, s>>>(m.q, m.qp, m.dy, m.k, m.kp, p);
  return cudaGetLastError();
}

}  // namespace attn
