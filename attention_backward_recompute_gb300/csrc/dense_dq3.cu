// dQ from stored dS tiles (bf16 storage path, ATTN_OPT_STORE_DS).
//
// rlx-cpu src/attention_bwd.rs (fn backward_dense_head_all) forms, per query
// row, dQ = scale * sum_k dS[q, k] K[k] with dS = P * (dP - delta).  The dK/dV
// kernel already computes every dS tile; with this option it also writes each
// 128-key x 64-query tile dS^T once to the workspace (bf16, 16-byte chunks of
// 8 queries stored key after key, so that each warp stores 512 contiguous
// bytes; that order is the unswizzled MN-major operand layout), and this
// kernel forms
//   dQ_i = scale * sum_j dS_ij K_j      (M = 128 queries, N = head dim, K = 128 keys per tile)
// on tcgen05 with both operands MN-major in shared memory: A = the two 64-query
// dS^T tiles of query tile i, B = the key tile [128 keys][head dim].  No S or
// dP is recomputed, and every dQ element still has one writer (no atomics).
//
// Roles (256 threads, one persistent CTA per SM over the 128-query tiles):
// warp 0 copies (dS tiles by bulk copy, K by TMA, zeros for a 64-query half
// the dK/dV kernel never visited), warp 1 issues the MMAs, warps 4..7 store
// dQ (tensor-memory lane = query row of the tile).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "dense_common.cuh"
#include "dense_launch.h"
#include "sm103.cuh"

namespace attn {
using namespace sm103;

namespace {

constexpr int kStages = 3;
constexpr int kDsTile = 128 * 128;  // bytes of one stored dS^T tile: 128 keys x 64 queries bf16

template <int DP>
struct Dq3Layout {
  static constexpr int NCH = DP / 64;
  static constexpr int BQ = 128, BK = 128;
  static constexpr int DS = 2 * kDsTile;           // the two 64-query halves, LBO apart
  static constexpr int KT = NCH * BK * 128;        // key tile as NCH chunks [128 keys][64 dims]
  static constexpr int STAGE = DS + KT;
  static constexpr int BYTES = kStages * STAGE;
  static constexpr int TMEM_COLS = 2 * DP;         // two dQ accumulators (alternating items)
};

// 1-D bulk copy global -> shared, completion counted on `bar` (bytes % 16 == 0,
// both addresses 16-byte aligned)
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_addr(dst)),
               "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_addr(bar))
               : "memory");
}

__device__ __forceinline__ bool drain_wait(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_test(bar, parity)) {
    if (global_timer_ns() - t0 > ATTN_WAIT_TIMEOUT_NS) return false;
  }
  return true;
}

// Query tile of work item w: longest rows first under causal masks (query
// tile nqt - 1 - w / BH of head w % BH).
__device__ __forceinline__ void dq3_item(const DenseParams& p, int w, int nqt128, int* bh, int* it) {
  const int BH = p.B * p.H;
  *bh = w % BH;
  *it = nqt128 - 1 - w / BH;
}

// Work item of CTA c in round r: r*G + c, or r*G + G-1-c in odd rounds (a
// snake over the longest-first order, which evens out the CTAs' totals of
// key tiles; it grows with r, so the first index past the end ends the walk).
__device__ __forceinline__ int dq3_round_item(int r, int c, int G) { return r * G + ((r & 1) ? G - 1 - c : c); }

// Persistent: CTA c takes its work items round by round; the copy ring and
// its phases run on across items, and the two dQ accumulators alternate, so
// one item's epilogue overlaps the next item's copies and products.
template <int DP>
__global__ void __launch_bounds__(256, 1)
    dq3_kernel(const __grid_constant__ CUtensorMap tm_k, const DenseParams p) {
  using L = Dq3Layout<DP>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t bar_full[kStages], bar_empty[kStages], bar_acc_full[2], bar_acc_empty[2], bar_fin;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nqt128 = cdiv(p.Sq, L::BQ);
  const int items = p.B * p.H * nqt128;
  const int nkt = cdiv(p.Sk, L::BK), nqt = cdiv(p.Sq, 64);
  const Abort ab{&abort_flag, p.err};
  // key tiles [j_lo, j_hi) of an item
  auto tiles_of = [&](int it, int* j_lo, int* j_hi) {
    const int q0 = it * L::BQ;
    key_tile_range(p, q0, imin(q0 + L::BQ - 1, p.Sq - 1), L::BK, j_lo, j_hi);
  };

  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bar_full[s], 1);
      mbar_init(&bar_empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&bar_acc_full[a], 1);
      mbar_init(&bar_acc_empty[a], 4);  // one arrival per epilogue warp
    }
    mbar_init(&bar_fin, 1);
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

  if (warp == 0) {
    // ------------------------------------------------------------ copies
    if (lane == 0) tma_prefetch_map(&tm_k);
    int last_use[kStages];
    for (int i = 0; i < kStages; ++i) last_use[i] = -1;
    bool ok = true;
    int g = 0;  // running tile number of this CTA
    for (int r = 0, w = dq3_round_item(0, blockIdx.x, gridDim.x); w < items && ok;
         ++r, w = dq3_round_item(r, blockIdx.x, gridDim.x)) {
      int bh, it, j_lo, j_hi;
      dq3_item(p, w, nqt128, &bh, &it);
      tiles_of(it, &j_lo, &j_hi);
      const int b = bh / p.H, h = bh - b * p.H;
      for (int kt = j_lo; kt < j_hi && ok; ++kt, ++g) {
        const int s = g % kStages;
        if (g >= kStages) ok = mbar_wait_warp(&bar_empty[s], ((g / kStages) - 1) & 1, ab);
        if (!ok) break;
        uint8_t* st = sm + s * L::STAGE;
        // the dK/dV kernel visited query tiles [i_lo, i_hi) of key tile kt; a
        // half outside that range holds no stored tile and reads as zeros
        int i_lo, i_hi;
        query_tile_range(p, kt * L::BK, imin(kt * L::BK + L::BK - 1, p.Sk - 1), 64, &i_lo, &i_hi);
        bool have[2];
        uint32_t bytes = L::KT;
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          const int qt = 2 * it + hf;
          have[hf] = qt >= i_lo && qt < i_hi && qt < nqt;
          if (have[hf]) {
            bytes += kDsTile;
          } else {
            uint4* z = reinterpret_cast<uint4*>(st + hf * kDsTile);
            for (int i = lane; i < kDsTile / 16; i += 32) z[i] = make_uint4(0u, 0u, 0u, 0u);
          }
        }
        if (!have[0] || !have[1]) fence_proxy_async_smem();  // zeros visible to the tensor core
        __syncwarp();
        if (lane == 0) {
          mbar_arrive_expect_tx(&bar_full[s], bytes);
#pragma unroll
          for (int hf = 0; hf < 2; ++hf)
            if (have[hf]) {
              const size_t blob = (static_cast<size_t>(bh) * nkt + kt) * nqt + 2 * it + hf;
              bulk_g2s(st + hf * kDsTile, p.ds_store + blob * kDsTile, kDsTile, &bar_full[s]);
            }
          for (int c = 0; c < L::NCH; ++c)
            tma_load_4d(st + L::DS + c * (L::BK * 128), &tm_k, &bar_full[s], c * 64, kt * L::BK, h, b);
        }
        last_use[s] = g;
      }
    }
    if (lane == 0) {
      for (int s = 0; s < kStages; ++s)
        if (last_use[s] >= 0) drain_wait(&bar_full[s], (last_use[s] / kStages) & 1);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (whole warp, elected lane)
    constexpr uint32_t id = idesc_bf16(128, DP, true, true);
    // A: the stored dS as is, unswizzled MN-major (core matrices 2048 bytes
    // apart along the 128 queries of the two halves, 128 along the keys)
    const uint64_t dA = sdesc_none(smem_addr(sm), 128, 2048);
    const uint64_t dB = sdesc_sw128(smem_addr(sm + L::DS), L::BK * 128, 1024);  // MN-major: 64-dim chunks
    bool ok = true;
    int g = 0, li = 0;
    for (int r = 0, w = dq3_round_item(0, blockIdx.x, gridDim.x); w < items && ok;
         ++r, ++li, w = dq3_round_item(r, blockIdx.x, gridDim.x)) {
      int bh, it, j_lo, j_hi;
      dq3_item(p, w, nqt128, &bh, &it);
      tiles_of(it, &j_lo, &j_hi);
      const int a = li & 1;
      // the epilogue has read this accumulator's previous item
      if (li >= 2 && !(ok = mbar_wait_warp(&bar_acc_empty[a], ((li >> 1) - 1) & 1, ab))) break;
      tc_fence_after();
      const uint32_t acc = tmem + a * DP;
      for (int kt = j_lo; kt < j_hi && ok; ++kt, ++g) {
        const int s = g % kStages;
        if (!(ok = mbar_wait_warp(&bar_full[s], (g / kStages) & 1, ab))) break;
        tc_fence_after();
        const uint64_t ad = sdesc_add(dA, s * L::STAGE), bdesc = sdesc_add(dB, s * L::STAGE);
        if (kt == j_lo)
          mma_ss_w<false>(acc, ad, bdesc, id);
        else
          mma_ss_w<true>(acc, ad, bdesc, id);
#pragma unroll
        for (int kk = 1; kk < L::BK / 16; ++kk)  // 16 keys: two core matrices of A, 16 swizzled rows of B
          mma_ss_w<true>(acc, sdesc_add(ad, kk * 256), sdesc_add(bdesc, kk * 16 * 128), id);
        mma_commit_w(&bar_empty[s]);
      }
      if (ok) mma_commit_w(&bar_acc_full[a]);  // also for an item without key tiles (stores zeros)
    }
    mma_commit_w(&bar_fin);
    drain_wait(&bar_fin, 0);
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------------------------------------ epilogue
    const int row = (warp & 3) * 32 + lane;  // query row of the tile == tensor-memory lane
    const uint32_t lane_addr = static_cast<uint32_t>((warp & 3) * 32) << 16;
    bool ok = true;
    int li = 0;
    for (int r = 0, w = dq3_round_item(0, blockIdx.x, gridDim.x); w < items && ok;
         ++r, ++li, w = dq3_round_item(r, blockIdx.x, gridDim.x)) {
      int bh, it, j_lo, j_hi;
      dq3_item(p, w, nqt128, &bh, &it);
      tiles_of(it, &j_lo, &j_hi);
      const int b = bh / p.H, h = bh - b * p.H;
      const int a = li & 1;
      if (!(ok = mbar_wait_warp(&bar_acc_full[a], (li >> 1) & 1, ab))) break;
      tc_fence_after();
      const int q = it * L::BQ + row;
      const int64_t roff = static_cast<int64_t>(b) * p.s_dq[2] + static_cast<int64_t>(h) * p.s_dq[1] +
                           static_cast<int64_t>(q) * p.s_dq[0];
#pragma unroll 1
      for (int cc = 0; cc < DP / 32 && cc * 32 < p.D; ++cc) {  // warp-uniform: tensor-memory loads are collective
        uint32_t r[32];
        if (j_hi > j_lo) {
          tmem_ld32(tmem + a * DP + lane_addr + cc * 32, r);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) r[j] = 0u;
        }
        if (q < p.Sq) store_out32<false>(p.dq, roff, cc * 32, p.D, r, p.scale);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_acc_empty[a]);
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
cudaError_t launch_t(const DenseMaps& m, const DenseParams& p, cudaStream_t s) {
  using L = Dq3Layout<DP>;
  auto kern = dq3_kernel<DP>;
  const int smem = L::BYTES + 1024;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  const int items = p.B * p.H * cdiv(p.Sq, L::BQ);
  const int grid = imin(items, imax(sms, 1));  // one CTA per SM (shared memory)
  kern<<<grid, 256, smem, s>>>(m.k128, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_dq3(const DenseMaps& m, const DenseParams& p, cudaStream_t s) {
  if (padded_head_dim(p.D) == 64) return launch_t<64>(m, p, s);
  return launch_t<128>(m, p, s);
}

}  // namespace attn
