// dQ kernel with the softmax and the dS work on separate warpgroups and P, dS
// kept in tensor memory (bf16 storage path).
//
// rlx-cpu src/attention_bwd.rs (fn backward_dense_head_all, the dQ = dS K
// product), per 128-query tile i and 64-key tile j of one (batch, head):
//   S  = Q_i K_j^T                     tcgen05, A = Q_i from tensor memory, S[b]
//   dP = dY_i V_j^T                    tcgen05, A = dY_i from tensor memory, dP[b]
//   P  = exp(S*scale + bias - lse)     softmax warpgroup, bf16 over S[b]
//   dS = P * (dP - delta)              dS warpgroup, bf16 over dP[b]
//   dQ_i += dS K_j                     tcgen05, A = dS from tensor memory
// with the softmax scale applied to dQ at the end.  Q_i and dY_i are copied
// once into tensor memory (bf16 pairs), so the tensor core reads only the K
// and V tiles from shared memory; K, V and bias tiles come through a 4-stage
// TMA ring.  S and dP are double-buffered (b = j % 2) and each S buffer has
// its own softmax warpgroup.  Warp 0: TMA producer, warp 1: MMA issuer,
// warps 4..7: softmax of even tiles, warps 12..15: softmax of odd tiles,
// warps 8..11: dS.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "dense_common.cuh"
#include "dense_launch.h"
#include "sm103.cuh"

namespace attn {
using namespace sm103;

namespace {

constexpr int kStages = 4;

template <int DP>
struct Dq2Layout {
  static constexpr int NCH = DP / 64;
  static constexpr int BQ = 128, BK = 64;
  static constexpr int QT = NCH * BQ * 128;      // Q or dY tile (128 rows)
  static constexpr int KT = NCH * BK * 128;      // K or V tile (64 rows)
  static constexpr int BIAS = BQ * 128;          // 128 query rows x 64 keys
  static constexpr int K_OFF = 0;                           // kStages
  static constexpr int V_OFF = K_OFF + kStages * KT;        // kStages
  static constexpr int BIAS_OFF = V_OFF + kStages * KT;     // kStages
  static constexpr int BYTES = BIAS_OFF + kStages * BIAS;
  // Q and dY are needed in shared memory only until they are staged into
  // tensor memory: they occupy the K and V slots of stages 2 and 3, which the
  // producer fills only after that staging
  static constexpr int Q_OFF = K_OFF + 2 * KT;
  static constexpr int DY_OFF = V_OFF + 2 * KT;
  static_assert(QT == 2 * KT && kStages >= 4, "Q / dY alias two ring slots");
  // TMEM: dQ [0, DP), S[2] and dP[2] 64 columns each after that, then the
  // Q and dY rows as bf16 pairs (DP/2 columns each)
  static constexpr int T_S = DP, T_DP = DP + 128;
  static constexpr int T_QA = DP + 256, T_DYA = T_QA + DP / 2;
  static constexpr int TMEM_COLS = 512;
  static_assert(T_DYA + DP / 2 <= TMEM_COLS, "tensor memory budget");
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

// Keys [c0, c0+16) of the P row of one query: exp2(S*scale*log2e +
// bias*log2e - L2) as 8 bf16 pairs.  CHECK: keys outside [lo, hi] (tile-local
// range of keys this query sees) give zero and custom-masked keys (bit c - c0
// of kbits) give the row's masked-key probability pmq.
template <bool HAS_BIAS, bool CHECK>
__device__ __forceinline__ void p_chunk(const uint32_t (&sr)[16], int c0, const uint8_t* bias_row, int row,
                                        float scale_log2, float L2q, float pmq, uint32_t kbits, int lo, int hi,
                                        uint32_t* pw) {
#pragma unroll
  for (int jj = 0; jj < 2; ++jj) {  // 8 keys per 16-byte bias chunk
    const int j = c0 / 8 + jj;
    float bias8[8];
    if (HAS_BIAS) {
      const uint4 w4 = *reinterpret_cast<const uint4*>(bias_row + ((j ^ (row & 7)) << 4));
      const uint32_t w[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        bias8[2 * e] = __uint_as_float(w[e] << 16);
        bias8[2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u);
      }
    }
    float pv[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int c = c0 + 8 * jj + e;
      float x = fmaf(__uint_as_float(sr[8 * jj + e]), scale_log2, -L2q);
      if (HAS_BIAS) x = fmaf(bias8[e], kLog2e, x);
      pv[e] = ex2_approx(x);
      if (CHECK) {
        const bool masked = ((kbits >> (8 * jj + e)) & 1u) != 0u;
        pv[e] = (c >= lo && c <= hi) ? (masked ? pmq : pv[e]) : 0.f;
      }
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) pw[4 * jj + e] = pack_bf16x2(pv[2 * e], pv[2 * e + 1]);
  }
}

// The P row over the 64 keys of a tile, S read from tensor memory in four
// 16-column chunks with the next chunk's load in flight; chunk i's 8 bf16
// pairs go to columns [8i, 8i+8) of the same buffer, which chunks 0..i have
// already read.  The caller waits for the stores.
template <bool HAS_BIAS, bool CHECK>
__device__ __forceinline__ void p_row(uint32_t tS, const uint8_t* bias_row, int row, float scale_log2, float L2q,
                                      float pmq, uint32_t kb0, uint32_t kb1, int lo, int hi) {
  uint32_t s0[16], s1[16], pw[8];
  tmem_ld16(tS, s0);
  tmem_ld_wait();
  reg_fence16(s0);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t(&cur)[16] = (i & 1) ? s1 : s0;
    uint32_t(&nxt)[16] = (i & 1) ? s0 : s1;
    if (i < 3) tmem_ld16(tS + 16 * (i + 1), nxt);
    const uint32_t kbits = ((i < 2 ? kb0 : kb1) >> (16 * (i & 1))) & 0xffffu;
    p_chunk<HAS_BIAS, CHECK>(cur, 16 * i, bias_row, row, scale_log2, L2q, pmq, kbits, lo, hi, pw);
    tmem_st8(tS + 8 * i, pw);
    if (i < 3) {
      tmem_ld_wait();
      reg_fence16(nxt);
    }
  }
}

template <int DP, bool HAS_BIAS, bool ELEM>
__global__ void __launch_bounds__(512, 1)
    dq2_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_dy,
               const __grid_constant__ CUtensorMap tm_bias, const DenseParams p) {
  using L = Dq2Layout<DP>;
  // dynamic shared memory starts 1024-aligned after the static variables'
  // granule on this GPU; the kernel checks it (the swizzled tiles need it)
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = smem_raw;
  if (smem_addr(smem_raw) & 1023u) {  // uniform
    if (threadIdx.x == 0 && p.err) atomicOr(p.err, DEV_ERR_LAYOUT);
    return;
  }
  __shared__ uint64_t bar_qdy, bar_a_ready, bar_full[kStages], bar_empty[kStages], bar_s_full[2], bar_dp_full[2],
      bar_p_full[2], bar_p_read[2], bar_ds_full[2], bar_acc;
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
    mbar_init(&bar_a_ready, 8);  // warps 4..11: Q and dY rows staged in tensor memory
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bar_full[s], 1);
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
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base_sh, L::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  const uint32_t t_dq = tmem;

  if (n > 0 && warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_map(&tm_q);
      tma_prefetch_map(&tm_k);
      tma_prefetch_map(&tm_v);
      tma_prefetch_map(&tm_dy);
      if (HAS_BIAS) tma_prefetch_map(&tm_bias);
      mbar_arrive_expect_tx(&bar_qdy, 2 * L::QT);
      for (int c = 0; c < L::NCH; ++c) {
        tma_load_4d(sm + L::Q_OFF + c * (L::BQ * 128), &tm_q, &bar_qdy, c * 64, q0, h, b);
        tma_load_4d(sm + L::DY_OFF + c * (L::BQ * 128), &tm_dy, &bar_qdy, c * 64, q0, h, b);
      }
      int last_use[kStages];
      for (int i = 0; i < kStages; ++i) last_use[i] = -1;
      bool ok = true;
      for (int t = 0; t < n && ok; ++t) {
        const int s = t % kStages;
        if (t >= kStages) ok = mbar_wait(&bar_empty[s], ((t / kStages) - 1) & 1, ab);
        if (t == 2 && ok) ok = mbar_wait(&bar_a_ready, 0, ab);  // Q, dY slots free
        if (!ok) break;
        const int kk0 = (j_lo + t) * L::BK;
        mbar_arrive_expect_tx(&bar_full[s], 2 * L::KT + (HAS_BIAS ? L::BIAS : 0));
        for (int c = 0; c < L::NCH; ++c) {
          tma_load_4d(sm + L::K_OFF + s * L::KT + c * (L::BK * 128), &tm_k, &bar_full[s], c * 64, kk0, h, b);
          tma_load_4d(sm + L::V_OFF + s * L::KT + c * (L::BK * 128), &tm_v, &bar_full[s], c * 64, kk0, h, b);
        }
        if (HAS_BIAS) tma_load_4d(sm + L::BIAS_OFF + s * L::BIAS, &tm_bias, &bar_full[s], kk0, q0, h, b);
        last_use[s] = t;
      }
      for (int s = 0; s < kStages; ++s)
        if (last_use[s] >= 0) drain_wait(&bar_full[s], (last_use[s] / kStages) & 1);
      drain_wait(&bar_qdy, 0);
    }
    __syncwarp();
  } else if (n > 0 && warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // the whole warp runs this role (warp-uniform); elected lanes issue
    {
      constexpr uint32_t id_s = idesc_bf16(128, 64, false, false);
      constexpr uint32_t id_acc = idesc_bf16(128, DP, false, true);
      // descriptors built once; k-slices and stages are constant offsets
      const uint64_t dK0 = sdesc_sw128(smem_addr(sm + L::K_OFF), 16, 1024);
      const uint64_t dV0 = sdesc_sw128(smem_addr(sm + L::V_OFF), 16, 1024);
      const uint64_t dKm0 = sdesc_sw128(smem_addr(sm + L::K_OFF), L::BK * 128, 1024);  // MN-major
      // D[128 x 64] = A[128 x DP] (tensor memory, bf16 pairs) * B[64 x DP]^T (shared memory, K-major)
      auto issue_xt = [&](uint32_t d, uint32_t a_tmem, uint64_t bk) {
        mma_ts_w<false>(d, a_tmem, bk, id_s);
#pragma unroll
        for (int kk = 1; kk < DP / 16; ++kk) {
          const int c = kk >> 2, o = (kk & 3) * 32;
          mma_ts_w<true>(d, a_tmem + kk * 8, sdesc_add(bk, c * (L::BK * 128) + o), id_s);
        }
      };
      auto issue_s = [&](int t) {  // S(t) = Q K^T into buffer t % 2
        issue_xt(tmem + L::T_S + (t & 1) * 64, tmem + L::T_QA, sdesc_add(dK0, (t % kStages) * L::KT));
        mma_commit_w(&bar_s_full[t & 1]);
      };
      auto issue_dp = [&](int t) {  // dP(t) = dY V^T into buffer t % 2
        issue_xt(tmem + L::T_DP + (t & 1) * 64, tmem + L::T_DYA, sdesc_add(dV0, (t % kStages) * L::KT));
        mma_commit_w(&bar_dp_full[t & 1]);
      };
      bool ok = mbar_wait_warp(&bar_a_ready, 0, ab);
      tc_fence_after();
      for (int t = 0; t < 2 && t < n && ok; ++t) {
        if (!(ok = mbar_wait_warp(&bar_full[t], 0, ab))) break;
        tc_fence_after();
        issue_s(t);
        issue_dp(t);
      }
      // Issue order per tile t: S(t+2), dQ(t), dP(t+2).  S(t+2) overwrites
      // P(t) once the dS warpgroup has read it (p_read), without waiting for
      // dS(t); dP(t+2) overwrites dS(t), read by dQ(t) just before it.
      for (int t = 0; t < n && ok; ++t) {
        const int s = t % kStages, bb = t & 1;
        if (t + 2 < n) {
          if (!(ok = mbar_wait_warp(&bar_full[(t + 2) % kStages], ((t + 2) / kStages) & 1, ab))) break;
          if (!(ok = mbar_wait_warp(&bar_p_read[bb], (t >> 1) & 1, ab))) break;
          tc_fence_after();
          issue_s(t + 2);
        }
        if (!(ok = mbar_wait_warp(&bar_ds_full[bb], (t >> 1) & 1, ab))) break;
        tc_fence_after();
        {
          const uint64_t bm = sdesc_add(dKm0, s * L::KT);
          const uint32_t a = tmem + L::T_DP + bb * 64;
          if (t == 0)
            mma_ts_w<false>(t_dq, a, bm, id_acc);
          else
            mma_ts_w<true>(t_dq, a, bm, id_acc);
#pragma unroll
          for (int kk = 1; kk < L::BK / 16; ++kk) mma_ts_w<true>(t_dq, a + kk * 8, sdesc_add(bm, kk * 16 * 128), id_acc);
        }
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
    const int row = lg * 32 + lane;  // query row inside the tile == TMEM lane
    const int q = q0 + row;
    const uint32_t lane_addr = static_cast<uint32_t>(lg * 32) << 16;
    bool ok = n > 0;
    float L2q = __int_as_float(0x7f800000), dlt = 0.f, pmq = 0.f;
    if (q < p.Sq) {
      const size_t idx = static_cast<size_t>(bh) * p.Sq + q;
      L2q = p.L2[idx];
      dlt = p.delta[idx];
      if (p.has_custom) pmq = p.pm[idx];
    }
    if (n > 0 && warp < 12) {
      // stage this row of Q (warps 4..7) or dY (warps 8..11) in tensor memory
      // as bf16 pairs: the A operand of S = Q K^T and dP = dY V^T
      const bool isq = warp < 8;
      ok = mbar_wait_warp(&bar_qdy, 0, ab);
      if (ok) {
        const uint8_t* src = sm + (isq ? L::Q_OFF : L::DY_OFF);
        const uint32_t dst = tmem + (isq ? L::T_QA : L::T_DYA) + lane_addr;
#pragma unroll
        for (int c = 0; c < L::NCH; ++c) {
          uint32_t w[32];
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const uint4 v = *reinterpret_cast<const uint4*>(src + c * (L::BQ * 128) + sw128_offset(row, j));
            w[4 * j] = v.x;
            w[4 * j + 1] = v.y;
            w[4 * j + 2] = v.z;
            w[4 * j + 3] = v.w;
          }
          tmem_st32(dst + c * 32, w);
        }
        tmem_st_wait();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_a_ready);
    }
    if (n > 0 && softmax_wg && ok) {
      // ---------------------------------------------------------- softmax: S -> P
      // keys this query sees: [ka, kb] (window: key >= q + q_off - window;
      // causal: key <= q + q_off; key < Sk; none when q >= Sq)
      int ka = -(1 << 30), kb = p.Sk - 1;
      if (p.window >= 0) ka = q + p.q_off - p.window;
      if (p.causal) kb = imin(kb, q + p.q_off);
      if (q >= p.Sq) ka = 1 << 30, kb = -(1 << 30);
      // custom-mask values of this group's next tile, loaded one tile ahead
      const float* km = p.has_key_mask ? p.key_mask + static_cast<size_t>(b) * p.Sk : nullptr;
      const float inf = __int_as_float(0x7f800000);
      auto km_load = [&](int kk, float* v) {
        v[0] = kk + lane < p.Sk ? km[kk + lane] : inf;
        v[1] = kk + 32 + lane < p.Sk ? km[kk + 32 + lane] : inf;
      };
      float kmv[2] = {0.f, 0.f};
      if (p.has_key_mask && sg < n) km_load((j_lo + sg) * L::BK, kmv);
      // Each group waits every phase of its own S buffer.  Of the stage
      // barrier it skips the phases of the other group's tiles; when it waits
      // for tile t, the phase of tile t - kStages (same stage) has completed,
      // since the tensor core issued S(t - 2) after it.
      for (int t = sg; t < n && ok; t += 2) {
        const int s = t % kStages, bb = t & 1;
        const int kk0 = (j_lo + t) * L::BK;
        uint32_t kb0 = 0, kb1 = 0;
        if (p.has_key_mask) {
          kb0 = __ballot_sync(0xffffffffu, kmv[0] < p.mask_thr);
          kb1 = __ballot_sync(0xffffffffu, kmv[1] < p.mask_thr);
          if (t + 2 < n) km_load(kk0 + 2 * L::BK, kmv);
        }
        if (ELEM && q < p.Sq) {  // per-element mask: this row's bits of the tile's 64 keys
          const uint2 w = *reinterpret_cast<const uint2*>(p.elem_rows + (static_cast<size_t>(bh) * p.Sq + q) * p.ew_q +
                                                           (kk0 >> 5));
          kb0 |= w.x;
          kb1 |= w.y;
        }
        if (!(ok = mbar_wait_warp(&bar_full[s], (t / kStages) & 1, ab))) break;
        if (!(ok = mbar_wait_warp(&bar_s_full[bb], (t >> 1) & 1, ab))) break;
        tc_fence_after();
        const uint32_t tS = tmem + L::T_S + bb * 64 + lane_addr;
        const bool full = tile_fully_visible(p, q0, q0 + L::BQ - 1, kk0, kk0 + L::BK - 1);
        const uint8_t* bias_row = sm + L::BIAS_OFF + s * L::BIAS + row * 128;
        const int lo = ka - kk0, hi = kb - kk0;
        if (full && !p.has_key_mask && !ELEM)
          p_row<HAS_BIAS, false>(tS, bias_row, row, p.scale_log2, L2q, pmq, kb0, kb1, lo, hi);
        else
          p_row<HAS_BIAS, true>(tS, bias_row, row, p.scale_log2, L2q, pmq, kb0, kb1, lo, hi);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar_p_full[bb]);
      }
    } else if (n > 0 && ok) {
      // ---------------------------------------------------------- dS: dP, P -> dS
      for (int t = 0; t < n && ok; ++t) {
        const int bb = t & 1;
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
        // two halves of 32 keys: half hf reads dP columns [32hf, 32hf+32) and
        // writes dS (bf16 pairs) to columns [16hf, 16hf+16), which half 0 has
        // already read
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          uint32_t dr[32], dsw[16];
          tmem_ld32(tDP + 32 * hf, dr);
          tmem_ld_wait();
#pragma unroll
          for (int c2 = 0; c2 < 16; ++c2) {
            const uint32_t w = pw[16 * hf + c2];
            const float p0 = __uint_as_float(w << 16), p1 = __uint_as_float(w & 0xffff0000u);
            dsw[c2] = pack_bf16x2(p0 * (__uint_as_float(dr[2 * c2]) - dlt), p1 * (__uint_as_float(dr[2 * c2 + 1]) - dlt));
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
    // each softmax group stores half of the dQ row (times the softmax scale)
    if (softmax_wg && (p.wrt & 1u) && (ok || n == 0)) {
      const int64_t roff = static_cast<int64_t>(b) * p.s_dq[2] + static_cast<int64_t>(h) * p.s_dq[1] +
                           static_cast<int64_t>(q) * p.s_dq[0];
#pragma unroll 1
      for (int cc = sg * (DP / 64); cc < (sg + 1) * (DP / 64) && cc * 32 < p.D; ++cc) {
        uint32_t r[32];
        if (n > 0) {
          tmem_ld32(t_dq + lane_addr + cc * 32, r);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) r[j] = 0u;
        }
        if (q < p.Sq) store_out32<false>(p.dq, roff, cc * 32, p.D, r, p.scale);
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

template <int DP, bool HAS_BIAS, bool ELEM>
cudaError_t launch_t(const DenseMaps& m, const DenseParams& p, cudaStream_t s) {
  using L = Dq2Layout<DP>;
  auto kern = dq2_kernel<DP, HAS_BIAS, ELEM>;
  // the static variables take one 1 KiB granule before the dynamic part
  static_assert(L::BYTES + 1024 <= 232448, "the layout fits one CTA's shared memory");
  const int smem = max(L::BYTES, kSmemOneCtaPerSm);  // all 512 TMEM columns: one CTA per SM
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  dim3 grid(p.B * p.H, cdiv(p.Sq, L::BQ));
  kern<<<grid, 512, smem, s>>>(m.q128, m.k64, m.v64, m.dy128, m.bias128, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_dq2(const DenseMaps& m, const DenseParams& p, bool bias, cudaStream_t s) {
  const int DP = padded_head_dim(p.D);
  if (p.elem_rows) {  // per-element custom mask
    if (DP == 64) return bias ? launch_t<64, true, true>(m, p, s) : launch_t<64, false, true>(m, p, s);
    return bias ? launch_t<128, true, true>(m, p, s) : launch_t<128, false, true>(m, p, s);
  }
  if (DP == 64) return bias ? launch_t<64, true, false>(m, p, s) : launch_t<64, false, false>(m, p, s);
  return bias ? launch_t<128, true, false>(m, p, s) : launch_t<128, false, false>(m, p, s);
}

}  // namespace attn
