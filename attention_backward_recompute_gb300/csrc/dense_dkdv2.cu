// dK / dV kernel, bf16 storage: the tensor core forms the score and dP tiles
// of one tile while two groups of compute warps turn earlier tiles into P and
// dS, kept in tensor memory.
//
// Same products as rlx-cpu src/attention_bwd.rs (fn backward_dense_head_all),
// per 128-key tile j and 64-query tile i of one (batch, head):
//   S^T  = K_j Q_i^T                    tcgen05 (smem x smem), TMEM buffer S[b]
//   dP^T = V_j dY_i^T                   tcgen05 (smem x smem), TMEM buffer dP[b]
//   P^T  = exp(S^T*scale + bias - lse)  written as bf16 over the first half of S[b]
//   dS^T = P^T * (dP^T - delta)         written as bf16 over the first half of dP[b]
//   dV_j += P^T dY_i                    tcgen05, A = P^T from tensor memory
//   dK_j += dS^T Q_i                    tcgen05, A = dS^T from tensor memory
// S and dP are double-buffered (b = i % 2).  Compute group b (four warps, one
// TMEM lane quarter each) owns the tiles of parity b: it forms P^T(i), hands
// it to the tensor core, then forms dS^T(i) from the P^T values it still holds
// in registers and dP^T(i).  Once P^T(i) is handed over, nothing reads S[b]
// any more, so the score tile of i + 2 can be formed while the group works on
// dS^T(i).  Q, dY, bias and the row statistics come through a 3-stage TMA
// ring.  Warp 0: TMA producer, warp 1: MMA issuer (whole warp, elect.sync),
// warp 2: row statistics of each stage (global loads, one tile ahead),
// warps 4..7: group 0, warps 8..11: group 1.  The statistics have a warp of
// their own because their global loads, issued beside the compute warps'
// shared-memory traffic, took ~2,000 cycles per tile in the producer's loop,
// which then released each stage's copies that much later.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "dense_common.cuh"
#include "dense_launch.h"
#include "sm103.cuh"

namespace attn {
using namespace sm103;

namespace {


template <int DP, bool HAS_BIAS>
struct Dkdv2Layout {
  static constexpr int NCH = DP / 64;
  static constexpr int BK = 128, BQ = 64;
  // stages of the Q / dY (and bias) ring: 3 with a bias tile in each stage,
  // 4 without
  static constexpr int STAGES = HAS_BIAS ? 3 : 4;
  static constexpr int KV = NCH * BK * 128;       // K (or V) tile
  static constexpr int QT = NCH * BQ * 128;       // Q (or dY) tile
  static constexpr int BIAS = HAS_BIAS ? 2 * BQ * 128 : 0;  // two 64-key halves x 64 query rows
  static constexpr int K_OFF = 0;
  static constexpr int V_OFF = K_OFF + KV;
  static constexpr int Q_OFF = V_OFF + KV;                 // STAGES
  static constexpr int DY_OFF = Q_OFF + STAGES * QT;       // STAGES
  static constexpr int BIAS_OFF = DY_OFF + STAGES * QT;    // STAGES (with a bias)
  static constexpr int ST_OFF = BIAS_OFF + STAGES * BIAS;  // STAGES x {-L2, delta, pm} x 64 floats
  static constexpr int BYTES = ST_OFF + STAGES * 3 * BQ * 4;
  // TMEM: dV [0, DP), dK [DP, 2DP), S[2] and dP[2] 64 columns each after that
  static constexpr int T_S = 2 * DP, T_DP = 2 * DP + 128;
  static constexpr int TMEM_COLS = 2 * DP + 256 <= 256 ? 256 : 512;
};

__device__ __forceinline__ bool drain_wait(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_test(bar, parity)) {
    if (global_timer_ns() - t0 > ATTN_WAIT_TIMEOUT_NS) return false;
  }
  return true;
}

// shared-memory loads through 32-bit shared addresses (ld.shared, not a
// generic load that must first resolve its address space)
__device__ __forceinline__ float4 lds_f4(const float* p) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(smem_addr(p)));
  return v;
}
__device__ __forceinline__ uint32_t lds_u16(uint32_t addr) {
  uint16_t v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
  return v;
}

// Registers written by tcgen05.ld are valid only after tcgen05.wait::ld; this
// empty asm ties every later use of r to a point after the wait.
__device__ __forceinline__ void reg_fence16(uint32_t (&r)[16]) {
#pragma unroll
  for (int i = 0; i < 16; ++i) asm volatile("" : "+r"(r[i]));
}

// 16 queries [c0, c0+16) of the P^T row of one key: exp2(S*scale*log2e +
// bias*log2e - L2) as 8 bf16 pairs, the arithmetic on fp32 pairs.  st holds
// -L2 per query.  bq[m] is the shared address of this key's bias of query m (m < 8) of the
// chunk; query m + 8 is 8 rows further on.  CHECK: zero the queries outside
// [lo, hi] (tile-local range of queries that see this key).  kmasked: the key
// is custom-masked; its visible entries take the row's masked-key
// probability pm instead.
template <bool HAS_BIAS, bool CHECK, bool ELEM>
__device__ __forceinline__ void p_chunk(const uint32_t (&sr)[16], int c0, const float* st, const uint32_t* bq,
                                        float scale_log2, int lo, int hi, bool kmasked, uint32_t ebits,
                                        uint32_t* pw) {
  const uint64_t sl2 = f2_pack(scale_log2, scale_log2);
  const uint64_t l2e = f2_pack(kLog2e, kLog2e);
#pragma unroll
  for (int c4 = 0; c4 < 4; ++c4) {
    const float4 nl = lds_f4(st + c0 + 4 * c4);
    uint64_t x[2];
    x[0] = f2_fma(f2_pack_u(sr[4 * c4], sr[4 * c4 + 1]), sl2, f2_pack(nl.x, nl.y));
    x[1] = f2_fma(f2_pack_u(sr[4 * c4 + 2], sr[4 * c4 + 3]), sl2, f2_pack(nl.z, nl.w));
    if (HAS_BIAS) {
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        const int m0 = 4 * c4 + 2 * h2;  // query of the chunk, 0..15
        const uint32_t b0 = lds_u16(bq[m0 & 7] + (m0 >> 3) * 1024);
        const uint32_t b1 = lds_u16(bq[(m0 + 1) & 7] + ((m0 + 1) >> 3) * 1024);
        x[h2] = f2_fma(f2_pack_u(b0 << 16, b1 << 16), l2e, x[h2]);
      }
    }
    float pv[4];
    f2_split(x[0], pv[0], pv[1]);
    f2_split(x[1], pv[2], pv[3]);
#pragma unroll
    for (int e = 0; e < 4; ++e) pv[e] = ex2_approx(pv[e]);
    // per-element mask bits of these 4 queries
    const uint32_t e4 = ELEM ? (ebits >> (4 * c4)) & 0xfu : 0u;
    if (kmasked || e4) {
      const float4 pm = lds_f4(st + 128 + c0 + 4 * c4);
      const float pmv[4] = {pm.x, pm.y, pm.z, pm.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) pv[e] = (kmasked || ((e4 >> e) & 1u)) ? pmv[e] : pv[e];
    }
    if (CHECK || kmasked || e4) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int ql = c0 + 4 * c4 + e;
        pv[e] = (ql >= lo && ql <= hi) ? pv[e] : 0.f;
      }
    }
    pw[2 * c4] = pack_bf16x2(pv[0], pv[1]);
    pw[2 * c4 + 1] = pack_bf16x2(pv[2], pv[3]);
  }
}

// The P^T row over the 64 queries of a tile into pw (32 bf16 pairs, kept for
// dS), S read from tensor memory in four 16-column chunks with the next
// chunk's load in flight; chunk i's 8 pairs also go to columns [8i, 8i+8) of
// the same buffer, which chunks 0..i have already read.  bias_row points at
// this key's bias column in the tile (query 0).  The caller waits for the
// stores.
template <bool HAS_BIAS, bool CHECK, bool ELEM>
__device__ __forceinline__ void p_row(uint32_t tS, const float* st, const uint8_t* bias_row, int kc,
                                      float scale_log2, int lo, int hi, bool kmasked, uint2 eb, uint32_t (&pw)[32]) {
  // the 128-byte swizzle moves query m's 16-byte chunk to chunk kc ^ (m % 8)
  uint32_t bq[8];
#pragma unroll
  for (int m = 0; m < 8; ++m) bq[m] = smem_addr(bias_row) + m * 128 + (((kc ^ m) & 7) << 4);
  uint32_t s0[16], s1[16];
  tmem_ld16(tS, s0);
  tmem_ld_wait();
  reg_fence16(s0);
#pragma unroll
  for (int i = 0; i < 4; i += 2) {
    tmem_ld16(tS + 16 * (i + 1), s1);
    p_chunk<HAS_BIAS, CHECK, ELEM>(s0, 16 * i, st, bq, scale_log2, lo, hi, kmasked, i < 2 ? eb.x : eb.y,
                                   pw + 8 * i);
    tmem_st8(tS + 8 * i, pw + 8 * i);
#pragma unroll
    for (int m = 0; m < 8; ++m) bq[m] += 16 * 128;
    tmem_ld_wait();
    reg_fence16(s1);
    if (i + 2 < 4) tmem_ld16(tS + 16 * (i + 2), s0);
    p_chunk<HAS_BIAS, CHECK, ELEM>(s1, 16 * (i + 1), st, bq, scale_log2, lo, hi, kmasked,
                                   (i < 2 ? eb.x : eb.y) >> 16, pw + 8 * (i + 1));
    tmem_st8(tS + 8 * (i + 1), pw + 8 * (i + 1));
#pragma unroll
    for (int m = 0; m < 8; ++m) bq[m] += 16 * 128;
    if (i + 2 < 4) {
      tmem_ld_wait();
      reg_fence16(s0);
    }
  }
}

// One work item = one (batch*head, 128-key tile): the visible 64-query tiles
// [i_lo, i_lo + n) of that key tile.
struct Item {
  int bh, kt, i_lo, n;
};

__device__ __forceinline__ Item item_at(const DenseParams& p, int idx) {
  const int BH = p.B * p.H;
  Item it;
  it.kt = idx / BH;
  it.bh = idx - it.kt * BH;
  const int k0 = it.kt * 128;
  int lo, hi;
  query_tile_range(p, k0, imin(k0 + 127, p.Sk - 1), 64, &lo, &hi);
  it.i_lo = lo;
  it.n = hi - lo;
  return it;
}

// Items of this CTA: item indices run key tile major (longest first under a
// causal mask); round r gives CTA c the index r*G + c, or r*G + G-1-c in odd
// rounds (a snake order that evens out the per-CTA totals).
struct ItemIter {
  int r, c, G, total;
  __device__ __forceinline__ bool next(int* idx) {
    while (true) {
      const int base = r * G;
      if (base >= total) return false;
      const int i = base + ((r & 1) ? G - 1 - c : c);
      ++r;
      if (i < total) {
        *idx = i;
        return true;
      }
    }
  }
};

template <int DP, bool HAS_BIAS, bool ELEM, bool DS>
__global__ void __launch_bounds__(384, 1)
    dkdv2_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                 const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_dy,
                 const __grid_constant__ CUtensorMap tm_bias, const DenseParams p) {
  using L = Dkdv2Layout<DP, HAS_BIAS>;
  constexpr int kStages = L::STAGES;
  // dynamic shared memory starts 1024-aligned after the static variables'
  // granule on this GPU; the kernel checks it (the swizzled tiles need it)
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = smem_raw;
  // bar_kv: K/V of a live item loaded; bar_kv_free: every S/dP product of
  // the item done (K/V slots free); bar_acc: every product of the item done;
  // bar_acc_free: the epilogue has read dV and dK out of tensor memory.
  // Their phases count live items (items with at least one query tile).
  __shared__ uint64_t bar_kv, bar_kv_free, bar_full[kStages], bar_empty[kStages], bar_s_full[2], bar_dp_full[2],
      bar_p_full[2], bar_ds_full[2], bar_acc, bar_acc_free;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag;
  if (smem_addr(smem_raw) & 1023u) {  // uniform
    if (threadIdx.x == 0 && p.err) atomicOr(p.err, DEV_ERR_LAYOUT);
    return;
  }

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nkt = cdiv(p.Sk, L::BK);
  const int total = p.B * p.H * nkt;
  const Abort ab{&abort_flag, p.err};

  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bar_kv, 1);
    mbar_init(&bar_kv_free, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bar_full[s], 2);  // TMA bytes + statistics written
      mbar_init(&bar_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bar_s_full[s], 1);
      mbar_init(&bar_dp_full[s], 1);
      mbar_init(&bar_p_full[s], 4);
      mbar_init(&bar_ds_full[s], 4);
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
  ItemIter iter{0, static_cast<int>(blockIdx.x), static_cast<int>(gridDim.x), total};

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_map(&tm_q);
      tma_prefetch_map(&tm_k);
      tma_prefetch_map(&tm_v);
      tma_prefetch_map(&tm_dy);
      if (HAS_BIAS) tma_prefetch_map(&tm_bias);
    }
    int last_use[kStages];
    for (int i = 0; i < kStages; ++i) last_use[i] = -1;
    bool ok = true;
    int g0 = 0, lv = 0, idx;
    while (ok && iter.next(&idx)) {
      const Item it = item_at(p, idx);
      if (it.n == 0) continue;
      const int b = it.bh / p.H, h = it.bh - b * p.H, k0 = it.kt * L::BK;
      if (lv > 0 && !(ok = mbar_wait(&bar_kv_free, (lv - 1) & 1, ab))) break;
      if (lane == 0) {
        mbar_arrive_expect_tx(&bar_kv, 2 * L::KV);
        for (int c = 0; c < L::NCH; ++c) {
          tma_load_4d(sm + L::K_OFF + c * (L::BK * 128), &tm_k, &bar_kv, c * 64, k0, h, b);
          tma_load_4d(sm + L::V_OFF + c * (L::BK * 128), &tm_v, &bar_kv, c * 64, k0, h, b);
        }
      }
      for (int t = 0; t < it.n && ok; ++t) {
        const int g = g0 + t, s = g % kStages;
        if (g >= kStages && !(ok = mbar_wait(&bar_empty[s], ((g / kStages) - 1) & 1, ab))) break;
        const int q0 = (it.i_lo + t) * L::BQ;
        if (lane == 0) {
          mbar_arrive_expect_tx(&bar_full[s], 2 * L::QT + (HAS_BIAS ? L::BIAS : 0));
          for (int c = 0; c < L::NCH; ++c) {
            tma_load_4d(sm + L::Q_OFF + s * L::QT + c * (L::BQ * 128), &tm_q, &bar_full[s], c * 64, q0, h, b);
            tma_load_4d(sm + L::DY_OFF + s * L::QT + c * (L::BQ * 128), &tm_dy, &bar_full[s], c * 64, q0, h, b);
          }
          if (HAS_BIAS) {
            uint8_t* bs = sm + L::BIAS_OFF + s * L::BIAS;
            tma_load_4d(bs, &tm_bias, &bar_full[s], k0, q0, h, b);
            tma_load_4d(bs + L::BQ * 128, &tm_bias, &bar_full[s], k0 + 64, q0, h, b);
          }
          if (t + kStages < it.n) {  // the tile that will reuse this stage, into L2
            const int qn = (it.i_lo + t + kStages) * L::BQ;
            for (int c = 0; c < L::NCH; ++c) {
              tma_prefetch_l2_4d(&tm_q, c * 64, qn, h, b);
              tma_prefetch_l2_4d(&tm_dy, c * 64, qn, h, b);
            }
            if (HAS_BIAS) {
              tma_prefetch_l2_4d(&tm_bias, k0, qn, h, b);
              tma_prefetch_l2_4d(&tm_bias, k0 + 64, qn, h, b);
            }
          }
        }
        last_use[s] = g;
      }
      g0 += it.n;
      ++lv;
    }
    if (lane == 0) {
      for (int s = 0; s < kStages; ++s)
        if (last_use[s] >= 0) drain_wait(&bar_full[s], (last_use[s] / kStages) & 1);
      if (lv > 0) drain_wait(&bar_kv, (lv - 1) & 1);
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------ statistics
    // (-L2, delta, pm) of rows lane and lane + 32 of each tile into its
    // stage (the second arrival on the stage's full barrier), loaded one tile
    // ahead so their latency overlaps the wait for the stage
    float pre[6];
    auto load_stats = [&](int bh, int qb0) {
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int q = qb0 + lane + 32 * i;
        const bool in = q < p.Sq;
        const size_t idx = static_cast<size_t>(bh) * p.Sq + (in ? q : 0);
        pre[3 * i] = in ? -p.L2[idx] : -__int_as_float(0x7f800000);
        pre[3 * i + 1] = in ? p.delta[idx] : 0.f;
        pre[3 * i + 2] = (in && p.has_custom) ? p.pm[idx] : 0.f;
      }
    };
    bool ok = true;
    int g0 = 0, idx;
    while (ok && iter.next(&idx)) {
      const Item it = item_at(p, idx);
      if (it.n == 0) continue;
      load_stats(it.bh, it.i_lo * L::BQ);
      for (int t = 0; t < it.n && ok; ++t) {
        const int g = g0 + t, s = g % kStages;
        if (g >= kStages && !(ok = mbar_wait(&bar_empty[s], ((g / kStages) - 1) & 1, ab))) break;
        float* st = reinterpret_cast<float*>(sm + L::ST_OFF) + s * 3 * L::BQ;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          st[lane + 32 * i] = pre[3 * i];
          st[L::BQ + lane + 32 * i] = pre[3 * i + 1];
          st[2 * L::BQ + lane + 32 * i] = pre[3 * i + 2];
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar_full[s]);
        if (t + 1 < it.n) load_stats(it.bh, (it.i_lo + t + 1) * L::BQ);
      }
      g0 += it.n;
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // the whole warp runs this role (warp-uniform); elected lanes issue
    constexpr uint32_t id_s = idesc_bf16(128, 64, false, false);
    constexpr uint32_t id_acc = idesc_bf16(128, DP, false, true);
    // descriptors built once; k-slices and stages are constant offsets
    const uint64_t dK = sdesc_sw128(smem_addr(sm + L::K_OFF), 16, 1024);
    const uint64_t dV = sdesc_sw128(smem_addr(sm + L::V_OFF), 16, 1024);
    const uint64_t dQ0 = sdesc_sw128(smem_addr(sm + L::Q_OFF), 16, 1024);
    const uint64_t dDY0 = sdesc_sw128(smem_addr(sm + L::DY_OFF), 16, 1024);
    const uint64_t dQm0 = sdesc_sw128(smem_addr(sm + L::Q_OFF), L::BQ * 128, 1024);    // MN-major
    const uint64_t dDYm0 = sdesc_sw128(smem_addr(sm + L::DY_OFF), L::BQ * 128, 1024);  // MN-major
    // D[128 x 64] = A[128 x DP] * B[64 x DP]^T, both from shared memory, K-major
    auto issue_xt = [&](uint32_t d, uint64_t a, uint64_t bq) {
      mma_ss_w<false>(d, a, bq, id_s);
#pragma unroll
      for (int kk = 1; kk < DP / 16; ++kk) {
        const int c = kk >> 2, o = (kk & 3) * 32;
        mma_ss_w<true>(d, sdesc_add(a, c * (L::BK * 128) + o), sdesc_add(bq, c * (L::BQ * 128) + o), id_s);
      }
    };
    // D[128 x DP] (+)= A[128 x 64] (tensor memory, bf16 pairs) * B[64 x DP] (MN-major)
    auto issue_acc = [&](uint32_t d, uint32_t a_tmem, uint64_t bm, bool first) {
      if (first)
        mma_ts_w<false>(d, a_tmem, bm, id_acc);
      else
        mma_ts_w<true>(d, a_tmem, bm, id_acc);
#pragma unroll
      for (int kk = 1; kk < L::BQ / 16; ++kk) mma_ts_w<true>(d, a_tmem + kk * 8, sdesc_add(bm, kk * 16 * 128), id_acc);
    };
    auto issue_s = [&](int g) {  // S(g) into buffer g % 2
      issue_xt(tmem + L::T_S + (g & 1) * 64, dK, sdesc_add(dQ0, (g % kStages) * L::QT));
      mma_commit_w(&bar_s_full[g & 1]);
    };
    auto issue_dp = [&](int g) {  // dP(g) into buffer g % 2
      issue_xt(tmem + L::T_DP + (g & 1) * 64, dV, sdesc_add(dDY0, (g % kStages) * L::QT));
      mma_commit_w(&bar_dp_full[g & 1]);
    };
    bool ok = true;
    int g0 = 0, lv = 0, idx;
    while (ok && iter.next(&idx)) {
      const Item it = item_at(p, idx);
      const int n = it.n;
      if (n == 0) continue;
      if (!(ok = mbar_wait_warp(&bar_kv, lv & 1, ab))) break;
      // the first score and dP tiles of this item go while the epilogue of
      // the previous item still reads dV and dK
      for (int t = 0; t < 2 && t < n && ok; ++t) {
        if (!(ok = mbar_wait_warp(&bar_full[(g0 + t) % kStages], ((g0 + t) / kStages) & 1, ab))) break;
        tc_fence_after();
        issue_s(g0 + t);
        issue_dp(g0 + t);
      }
      if (!ok) break;
      if (n <= 2) mma_commit_w(&bar_kv_free);
      if (lv > 0 && !(ok = mbar_wait_warp(&bar_acc_free, (lv - 1) & 1, ab))) break;
      tc_fence_after();
      // Per tile g: dV(g) once P(g) is in; then S(g+2) and dK(g) in whichever
      // order their inputs arrive; then dP(g+2).  S(g+2) overwrites P(g),
      // which dV(g) (earlier in the same pipe) consumes, and S(g), which the
      // group finished reading before it handed P(g) over; dP(g+2)
      // overwrites dS(g) and dP(g), read by dK(g) and by the group before
      // dS(g) was handed over.  Issuing dK(g) as soon as dS(g) is ready
      // releases tile g's stage early: the copies of tile g+3 wait on it.
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
          if (t + 3 == n) mma_commit_w(&bar_kv_free);  // the item's last S and dP are issued
        }
      }
      if (!ok) break;
      mma_commit_w(&bar_acc);
      g0 += n;
      ++lv;
    }
    // the last commits arrive before the CTA leaves
    if (lv > 0) drain_wait(&bar_acc, (lv - 1) & 1);
    __syncwarp();
  } else if (warp >= 4) {
    const int sg = (warp - 4) >> 2;  // compute group: tiles (and S/dP buffers) of parity sg
    const int lg = warp & 3;
    const int row = lg * 32 + lane;  // key row inside the tile == TMEM lane
    const uint32_t lane_addr = static_cast<uint32_t>(lg * 32) << 16;
    const int half = row >> 6, kc = (row & 63) >> 3, kb = (row & 7) * 2;
    bool ok = true;
    int g0 = 0, lv = 0, idx;
    while (ok && iter.next(&idx)) {
      const Item it = item_at(p, idx);
      const int b = it.bh / p.H, h = it.bh - b * p.H, k0 = it.kt * L::BK;
      const int key = k0 + row;
      const int n = it.n;
      if (n > 0) {
        bool kmasked = false;
        if (p.has_key_mask && key < p.Sk) kmasked = p.key_mask[static_cast<size_t>(b) * p.Sk + key] < p.mask_thr;
        // queries that see this key: [qa, qb] (causal: q + q_off >= key;
        // window: q + q_off - window <= key; q < Sq; none when key >= Sk)
        int qa = -(1 << 30), qb = p.Sq - 1;
        if (p.causal) qa = key - p.q_off;
        if (p.window >= 0) qb = imin(qb, key + p.window - p.q_off);
        if (key >= p.Sk) qa = 1 << 30, qb = -(1 << 30);
        // Each group waits every phase of its own S and dP buffers.  Of the
        // stage barrier it skips the phases of the other group's tiles; when
        // it waits for tile g, the phase of tile g - 3 (same stage, other
        // parity) has completed, since the tensor core issued S(g - 2) after
        // it.
        for (int t = ((g0 & 1) == sg) ? 0 : 1; t < n && ok; t += 2) {
          const int g = g0 + t, s = g % kStages, bb = g & 1;
          const int q0 = (it.i_lo + t) * L::BQ;
          uint2 eb = make_uint2(0u, 0u);  // per-element mask: this key's bits of the tile's 64 queries
          if (ELEM && key < p.Sk)
            eb = *reinterpret_cast<const uint2*>(p.elem_cols + (static_cast<size_t>(it.bh) * p.Sk + key) * p.ew_k +
                                                 (q0 >> 5));
          if (!(ok = mbar_wait_warp(&bar_full[s], (g / kStages) & 1, ab))) break;
          if (!(ok = mbar_wait_warp(&bar_s_full[bb], (g >> 1) & 1, ab))) break;
          tc_fence_after();
          // ---------------------------------------------------- S^T -> P^T
          const uint32_t tS = tmem + L::T_S + bb * 64 + lane_addr;
          const float* st = reinterpret_cast<const float*>(sm + L::ST_OFF) + s * 3 * L::BQ;
          const uint8_t* bias_row = sm + L::BIAS_OFF + s * L::BIAS + half * (L::BQ * 128) + kb;
          const bool full = tile_fully_visible(p, q0, q0 + L::BQ - 1, k0, k0 + L::BK - 1);
          const int lo = qa - q0, hi = qb - q0;
          uint32_t pw[32];
          if (full)
            p_row<HAS_BIAS, false, ELEM>(tS, st, bias_row, kc, p.scale_log2, lo, hi, kmasked, eb, pw);
          else
            p_row<HAS_BIAS, true, ELEM>(tS, st, bias_row, kc, p.scale_log2, lo, hi, kmasked, eb, pw);
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bar_p_full[bb]);
          // ---------------------------------------------------- dP^T, P^T -> dS^T
          if (!(ok = mbar_wait_warp(&bar_dp_full[bb], (g >> 1) & 1, ab))) break;
          tc_fence_after();
          const uint32_t tDP = tmem + L::T_DP + bb * 64 + lane_addr;
          const float* dl = st + L::BQ;
          // stored dS of tile (key tile, query tile i_lo + t): chunk c of this
          // key at c * 2048 + row * 16
          uint4* ds_row = nullptr;
          if (DS) {
            const size_t blob = (static_cast<size_t>(it.bh) * nkt + it.kt) * cdiv(p.Sq, L::BQ) + it.i_lo + t;
            ds_row = reinterpret_cast<uint4*>(p.ds_store + blob * (L::BK * 128)) + row;
          }
          // two halves of 32 queries: half hf reads dP columns [32hf, 32hf+32)
          // and writes dS^T (bf16 pairs) to columns [16hf, 16hf+16), which
          // half 0 has already read
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            uint32_t dr[32], dsw[16];
            tmem_ld32(tDP + 32 * hf, dr);
            tmem_ld_wait();
#pragma unroll
            for (int c4 = 0; c4 < 8; ++c4) {
              const float4 d4 = lds_f4(dl + 32 * hf + 4 * c4);
              const uint32_t w0 = pw[16 * hf + 2 * c4], w1 = pw[16 * hf + 2 * c4 + 1];
              const uint64_t dp01 = f2_add(f2_pack_u(dr[4 * c4], dr[4 * c4 + 1]), f2_pack(-d4.x, -d4.y));
              const uint64_t dp23 = f2_add(f2_pack_u(dr[4 * c4 + 2], dr[4 * c4 + 3]), f2_pack(-d4.z, -d4.w));
              float a0, a1, a2, a3;
              f2_split(f2_mul(f2_from_bf16x2(w0), dp01), a0, a1);
              f2_split(f2_mul(f2_from_bf16x2(w1), dp23), a2, a3);
              dsw[2 * c4] = pack_bf16x2(a0, a1);
              dsw[2 * c4 + 1] = pack_bf16x2(a2, a3);
            }
            tmem_st16(tDP + 16 * hf, dsw);
            if (DS) {
#pragma unroll
              for (int j = 0; j < 4; ++j)
                ds_row[(4 * hf + j) * L::BK] = make_uint4(dsw[4 * j], dsw[4 * j + 1], dsw[4 * j + 2], dsw[4 * j + 3]);
            }
          }
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bar_ds_full[bb]);
        }
        if (!ok) break;
        if (!(ok = mbar_wait_warp(&bar_acc, lv & 1, ab))) break;
        tc_fence_after();
      }
      // -------------------------------------------------------- epilogue
      // group 0 stores dV, group 1 dK (times the softmax scale); a key tile
      // no query sees gets zeros.  Tensor memory is handed back (acc_free)
      // as soon as the last chunk is in registers; the next item's products
      // into dV and dK wait for that.
      const bool want = sg == 0 ? (p.wrt & 4u) != 0 : (p.wrt & 2u) != 0;
      const int64_t* so = sg == 0 ? p.s_dv : p.s_dk;
      const int64_t roff = static_cast<int64_t>(b) * so[2] + static_cast<int64_t>(h) * so[1] +
                           static_cast<int64_t>(key) * so[0];
      void* out = sg == 0 ? p.dv : p.dk;
      const float f = sg == 0 ? 1.f : p.scale;
      const uint32_t tacc = (sg == 0 ? t_dv : t_dk) + lane_addr;
#pragma unroll 1
      for (int cc = 0; want && cc < DP / 32 && cc * 32 < p.D; ++cc) {
        uint32_t r[32];
        if (n > 0) {
          tmem_ld32(tacc + cc * 32, r);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) r[j] = 0u;
        }
        if (key < p.Sk) store_out32<false>(out, roff, cc * 32, p.D, r, f);
      }
      if (n > 0) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar_acc_free);
        g0 += n;
        ++lv;
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

template <int DP, bool HAS_BIAS, bool ELEM, bool DS>
cudaError_t launch_t(const DenseMaps& m, const DenseParams& p, cudaStream_t s) {
  using L = Dkdv2Layout<DP, HAS_BIAS>;
  auto kern = dkdv2_kernel<DP, HAS_BIAS, ELEM, DS>;
  // the static variables take one 1 KiB granule before the dynamic part
  static_assert(L::BYTES + 1024 <= 232448, "the layout fits one CTA's shared memory");
  const int smem = max(L::BYTES, kSmemOneCtaPerSm);  // all 512 TMEM columns: one CTA per SM
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  const int items = p.B * p.H * cdiv(p.Sk, L::BK);
  const int grid = imin(items, imax(sms, 1));  // persistent: one CTA per SM
  kern<<<grid, 384, smem, s>>>(m.q64, m.k128, m.v128, m.dy64, m.bias64, p);
  return cudaGetLastError();
}

template <bool ELEM, bool DS>
cudaError_t launch_dp(const DenseMaps& m, const DenseParams& p, bool bias, cudaStream_t s) {
  if (padded_head_dim(p.D) == 64)
    return bias ? launch_t<64, true, ELEM, DS>(m, p, s) : launch_t<64, false, ELEM, DS>(m, p, s);
  return bias ? launch_t<128, true, ELEM, DS>(m, p, s) : launch_t<128, false, ELEM, DS>(m, p, s);
}

}  // namespace

cudaError_t launch_dkdv2(const DenseMaps& m, const DenseParams& p, bool bias, cudaStream_t s) {
  // per-element custom mask (ELEM) and stored dS (DS) are separate instances
  if (p.elem_rows) return p.ds_store ? launch_dp<true, true>(m, p, bias, s) : launch_dp<true, false>(m, p, bias, s);
  return p.ds_store ? launch_dp<false, true>(m, p, bias, s) : launch_dp<false, false>(m, p, bias, s);
}

}  // namespace attn
