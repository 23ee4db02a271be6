// Query side of the paged MLA backward on tcgen05: dQ (latent, 512) and dQp
// (position, 64) for every packed query row and head, from the row
// statistics lse and delta of the same rows.
//
// ruDNN src/paged_attention/ordered_kernel.rs (the query kernel that pairs
// with history_backward): for query row r, head h and visible token t,
//   p = exp(scale (q . k_lat[t] + qp . k_pos[t]) - lse),
//   ds = p (dY . k_lat[t] - delta) scale,
//   dQ += ds k_lat[t],   dQp += ds k_pos[t]
// with one owner per (row, head) and one final store.
//
// One CTA per (KV head, tile of 64 columns = 64/G rows x the G heads of the
// group); Q, Qp and dY of the tile stay resident in shared memory.  The sweep
// runs over 128-token blocks of the row's sequence (eight pages gathered by
// TMA), with the tokens on the tensor-memory lanes:
//   [S^T | dP^T] = K_lat [Q | dY]^T   [128 tokens x 128], one N = 128
//                                     product per latent chunk (Q and dY
//                                     chunks of the same dims resident back
//                                     to back), S^T += K_pos Qp^T
//   dS^T = P^T (dP^T - delta) scale   compute warps, bf16 into shared memory
//   dQ^T += K^T dS^T                  [576 dims x 64 columns], 4.5 blocks of
//                                     128 dims, A = K chunk pairs (MN-major)
// K arrives as [128 tokens x 64 dims] chunks through a 4-stage ring, twice per
// block: once for the products with Q and dY, once (in pairs of chunks, one
// 128-dim block) for dQ^T; the second pass of block b - 1 follows the first
// pass of block b, so the tensor core forms block b's scores while the
// compute warps turn block b - 1 into dS (the rows of tokens past the
// sequence end are cleared in shared memory before the dQ^T products read
// them).  Each pass is ten ring slots (nine
// chunks and one slot with no copy, which keeps the chunk pairs of the dQ
// pass on even slots; the position block reads rows 64..127 of its A operand
// from that slot and stores only rows 0..63).
// Tensor memory: dQ^T [0, 320) (latent blocks 64 columns each, position block
// at 256), [S^T | dP^T] [320, 448), single-buffered: the compute warps load
// it and release it at once, so the next block's products overlap their dS.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "paged_common.cuh"
#include "paged_launch.h"
#include "sm103.cuh"

namespace attn {
using namespace sm103;

namespace {

constexpr int kLat = 512, kPos = 64, kDims = kLat + kPos;
constexpr int BC = 64;                  // columns per CTA
constexpr int BT = 128;                 // tokens per block (8 pages of 16)
constexpr int kStages = 4;
constexpr int kSlots = 10;              // ring slots per pass
constexpr int QCH = BC * 128;           // Q / dY chunk [64 columns][64 dims], 8 KiB
constexpr int KCH = BT * 128;           // K chunk [128 tokens][64 dims], 16 KiB
constexpr int QD_OFF = 0;               // (Q, dY) latent chunk pairs, 16 KiB each
constexpr int QP_OFF = QD_OFF + 16 * QCH; // the position chunk of Q
constexpr int RING_OFF = QP_OFF + QCH;
constexpr int DS_OFF = RING_OFF + kStages * KCH;  // dS^T [128 tokens][64 columns] bf16
constexpr int ST_OFF = DS_OFF + BT * 128;         // -L2, delta, pos per column
constexpr int BYTES = ST_OFF + 3 * BC * 4;
static_assert(17 * QCH >= BC * kDims * 2, "the output tile is staged in the Q / dY slots");
static_assert(RING_OFF % 1024 == 0 && DS_OFF % 1024 == 0, "swizzled tiles need 1024-byte alignment");
constexpr int T_DQ = 0, T_SDP = 320, TMEM_COLS = 512;

__device__ __forceinline__ bool drain_wait(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_test(bar, parity)) {
    if (global_timer_ns() - t0 > ATTN_WAIT_TIMEOUT_NS) return false;
  }
  return true;
}

__global__ void __launch_bounds__(256, 1)
    mla_query_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_qp,
                        const __grid_constant__ CUtensorMap tm_dy, const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_kp, const PagedParams p) {
  // dynamic shared memory starts 1024-aligned after the static variables'
  // granule on this GPU; the kernel checks it (the swizzled tiles need it)
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = smem_raw;
  if (smem_addr(smem_raw) & 1023u) {  // uniform
    if (threadIdx.x == 0 && p.err) atomicOr(p.err, DEV_ERR_LAYOUT);
    return;
  }
  __shared__ uint64_t bar_qdy, bar_full[kStages], bar_empty[kStages], bar_sdp_full, bar_sdp_read, bar_ds_ready,
      bar_ds_free, bar_acc;
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
  const int re = row_end_of(p, s0);
  const int len = seq_len_of(p, s0);
  const int npg = pages_of(len, p.page_size);
  const Abort ab{&abort_flag, p.err};
  const int oob_slot = p.num_pages * p.page_size;  // out-of-range coordinate: TMA fills zeros
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bar_qdy, 2);  // Q / dY bytes + column statistics written
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bar_full[s], 1);
      mbar_init(&bar_empty[s], 1);
    }
    mbar_init(&bar_sdp_full, 1);
    mbar_init(&bar_sdp_read, 4);
    mbar_init(&bar_ds_ready, 4);
    mbar_init(&bar_ds_free, 1);
    mbar_init(&bar_acc, 1);
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
  const int nb = (ntok_sh + BT - 1) / BT;  // token blocks
  float* snl = reinterpret_cast<float*>(sm + ST_OFF);
  float* sdl = snl + BC;
  int* spos = reinterpret_cast<int*>(sdl + BC);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    bool ok = true;
    int last_use[kStages];
    for (int i = 0; i < kStages; ++i) last_use[i] = -1;
    if (nb > 0) {
      if (lane == 0) {
        tma_prefetch_map(&tm_q);
        tma_prefetch_map(&tm_qp);
        tma_prefetch_map(&tm_dy);
        tma_prefetch_map(&tm_k);
        tma_prefetch_map(&tm_kp);
        mbar_arrive_expect_tx(&bar_qdy, 17 * QCH);
        for (int c = 0; c < 8; ++c) {
          tma_load_3d(sm + QD_OFF + 2 * c * QCH, &tm_q, &bar_qdy, c * 64, g * G, r0);
          tma_load_3d(sm + QD_OFF + (2 * c + 1) * QCH, &tm_dy, &bar_qdy, c * 64, g * G, r0);
        }
        tma_load_3d(sm + QP_OFF, &tm_qp, &bar_qdy, 0, g * G, r0);
      }
      for (int c = lane; c < BC; c += 32) {  // column statistics, two per lane
        const int r = r0 + c / G;
        float nl2 = -__int_as_float(0x7f800000), dl = 0.f;
        int pos = -1;
        if (r < re) {
          const int64_t idx = static_cast<int64_t>(r) * p.H + g * G + c % G;
          const float lse = p.lse[idx];
          if (lse != -__int_as_float(0x7f800000)) {
            nl2 = -lse * 1.4426950408889634f;
            dl = p.delta[idx];
            pos = p.causal ? p.q_pos[r] : 0x7fffffff;
          }
        }
        snl[c] = nl2;
        sdl[c] = dl;
        spos[c] = pos;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_qdy);
    }
    int q = 0;
    int slot[8];
    // one pass over the chunks of block b: nine chunk copies and one slot
    // with no copy
    auto pass = [&](int b) -> bool {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int lp = 8 * b + j;
        slot[j] = oob_slot;
        if (lp < npg) {
          const int ph = p.page_table[static_cast<int64_t>(s0) * p.max_pages + lp];
          if (ph >= 0 && ph < p.num_pages) slot[j] = ph * p.page_size;
        }
      }
      for (int c = 0; c < kSlots; ++c, ++q) {
        const int s = q % kStages;
        if (q >= kStages && !mbar_wait(&bar_empty[s], ((q / kStages) - 1) & 1, ab)) return false;
        if (lane == 0) {
          if (c < 9) {
            mbar_arrive_expect_tx(&bar_full[s], KCH);
            for (int j = 0; j < 8; ++j) {
              uint8_t* dst = sm + RING_OFF + s * KCH + j * 16 * 128;
              if (c < 8)
                tma_load_3d(dst, &tm_k, &bar_full[s], c * 64, g, slot[j]);
              else
                tma_load_3d(dst, &tm_kp, &bar_full[s], 0, g, slot[j]);
            }
          } else {
            mbar_arrive(&bar_full[s]);
          }
        }
        last_use[s] = q;
      }
      return true;
    };
    for (int b = 0; b <= nb && ok; ++b) {
      if (b < nb) ok = pass(b);          // products with Q and dY of block b
      if (ok && b >= 1) ok = pass(b - 1);  // dQ^T of block b - 1
    }
    if (lane == 0) {
      for (int s = 0; s < kStages; ++s)
        if (last_use[s] >= 0) drain_wait(&bar_full[s], (last_use[s] / kStages) & 1);
      if (nb > 0) drain_wait(&bar_qdy, 0);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (nb > 0) {
      constexpr uint32_t id_sdp = idesc_bf16(128, 2 * BC, false, false);  // [S^T | dP^T]: K-major A and B
      constexpr uint32_t id_s = idesc_bf16(128, BC, false, false);         // S^T += K_pos Qp^T
      constexpr uint32_t id_q = idesc_bf16(128, BC, true, true);           // dQ^T: MN-major A and B
      const uint64_t dQD0 = sdesc_sw128(smem_addr(sm + QD_OFF), 16, 1024);  // 128 rows: Q_c then dY_c
      const uint64_t dQP = sdesc_sw128(smem_addr(sm + QP_OFF), 16, 1024);
      const uint64_t dR0 = sdesc_sw128(smem_addr(sm + RING_OFF), 16, 1024);
      const uint64_t dRm0 = sdesc_sw128(smem_addr(sm + RING_OFF), KCH, 1024);  // MN-major, chunk pairs
      const uint64_t dDS = sdesc_sw128(smem_addr(sm + DS_OFF), 16 * 1024, 1024);  // MN-major
      bool ok = mbar_wait_warp(&bar_qdy, 0, ab);
      tc_fence_after();
      int q = 0;
      auto stage_in = [&](int qq) -> bool {
        const int s = qq % kStages;
        if (mbar_test_warp(&bar_full[s], (qq / kStages) & 1)) return true;
        return mbar_wait_warp(&bar_full[s], (qq / kStages) & 1, ab);
      };
      const uint32_t tSDP = tmem + T_SDP;
      for (int b = 0; b <= nb && ok; ++b) {
        if (b < nb) {
          // ------------------------------------------- [S^T | dP^T](b)
          // once the compute warps have loaded block b - 1's
          if (b >= 1 && !(ok = mbar_wait_warp(&bar_sdp_read, (b - 1) & 1, ab))) break;
          tc_fence_after();
          for (int c = 0; c < kSlots && ok; ++c, ++q) {
            if (!(ok = stage_in(q))) break;
            tc_fence_after();
            const uint64_t a = sdesc_add(dR0, (q % kStages) * KCH);
            if (c < 9) {
              const uint64_t bq = c < 8 ? sdesc_add(dQD0, 2 * c * QCH) : dQP;
              const uint32_t id = c < 8 ? id_sdp : id_s;
              if (c == 0)
                mma_ss_w<false>(tSDP, a, bq, id);
              else
                mma_ss_w<true>(tSDP, a, bq, id);
#pragma unroll
              for (int kk = 1; kk < 4; ++kk) mma_ss_w<true>(tSDP, sdesc_add(a, kk * 32), sdesc_add(bq, kk * 32), id);
            }
            mma_commit_w(&bar_empty[q % kStages]);
          }
          if (!ok) break;
          mma_commit_w(&bar_sdp_full);
        }
        if (b >= 1) {
          // ------------------------------------------- dQ^T += K^T dS^T(b - 1)
          const int u = b - 1;
          if (!(ok = mbar_wait_warp(&bar_ds_ready, u & 1, ab))) break;
          tc_fence_after();
          for (int j = 0; j < 5 && ok; ++j, q += 2) {
            if (!(ok = stage_in(q)) || !(ok = stage_in(q + 1))) break;
            tc_fence_after();
            // K rows of tokens past the sequence end (the tail of its last
            // page) hold whatever the pool holds there; they meet dS = 0 in
            // this product, and 0 times a non-finite value is not 0: clear
            // them first (only the block holding the sequence end has any)
            const int r_lo = len - BT * u;
            if (r_lo < BT) {
              for (int k = 0; k < (j < 4 ? 2 : 1); ++k) {
                const uint32_t base = smem_addr(sm + RING_OFF + ((q + k) % kStages) * KCH);
                for (int i = max(r_lo, 0) * 8 + lane; i < BT * 8; i += 32) st_shared_v4(base + 16 * i, 0u, 0u, 0u, 0u);
              }
              fence_proxy_async_smem();
              __syncwarp();
            }
            const uint64_t a = sdesc_add(dRm0, (q % kStages) * KCH);  // q is even: the pair is contiguous
            const uint32_t d = tmem + T_DQ + 64 * j;
            if (u == 0)
              mma_ss_w<false>(d, a, dDS, id_q);
            else
              mma_ss_w<true>(d, a, dDS, id_q);
#pragma unroll
            for (int kk = 1; kk < BT / 16; ++kk)
              mma_ss_w<true>(d, sdesc_add(a, kk * 16 * 128), sdesc_add(dDS, kk * 16 * 128), id_q);
            mma_commit_w(&bar_empty[q % kStages]);
            mma_commit_w(&bar_empty[(q + 1) % kStages]);
          }
          if (!ok) break;
          mma_commit_w(&bar_ds_free);
        }
      }
      mma_commit_w(&bar_acc);
      drain_wait(&bar_acc, 0);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------------------------------------ dS^T, epilogue
    const int lg = warp & 3;
    const int row = lg * 32 + lane;  // token row of the block == TMEM lane
    const uint32_t lane_addr = static_cast<uint32_t>(lg * 32) << 16;
    bool ok = nb > 0;
    if (nb > 0) ok = mbar_wait_warp(&bar_qdy, 0, ab);
    const uint64_t sl2 = f2_pack(p.scale_log2, p.scale_log2);
    for (int b = 0; b < nb && ok; ++b) {
      if (!(ok = mbar_wait_warp(&bar_sdp_full, b & 1, ab))) break;
      tc_fence_after();
      uint32_t sr[64], dr[64];
      tmem_ld32(tmem + T_SDP + lane_addr, *reinterpret_cast<uint32_t(*)[32]>(sr));
      tmem_ld32(tmem + T_SDP + 32 + lane_addr, *reinterpret_cast<uint32_t(*)[32]>(sr + 32));
      tmem_ld32(tmem + T_SDP + BC + lane_addr, *reinterpret_cast<uint32_t(*)[32]>(dr));
      tmem_ld32(tmem + T_SDP + BC + 32 + lane_addr, *reinterpret_cast<uint32_t(*)[32]>(dr + 32));
      tmem_ld_wait();
#pragma unroll
      for (int i = 0; i < 64; ++i) asm volatile("" : "+r"(sr[i]), "+r"(dr[i]));
      // [S^T | dP^T] may now take the next block's products
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_sdp_read);
      const int tok = b * BT + row;
      const bool tok_ok = tok < len;
      uint32_t dsw[32];
#pragma unroll
      for (int c4 = 0; c4 < 16; ++c4) {
        const int c0 = 4 * c4;
        const float4 nl = *reinterpret_cast<const float4*>(snl + c0);
        const float4 dl = *reinterpret_cast<const float4*>(sdl + c0);
        const int4 ps = *reinterpret_cast<const int4*>(spos + c0);
        float x[4];
        f2_split(f2_fma(f2_pack_u(sr[c0], sr[c0 + 1]), sl2, f2_pack(nl.x, nl.y)), x[0], x[1]);
        f2_split(f2_fma(f2_pack_u(sr[c0 + 2], sr[c0 + 3]), sl2, f2_pack(nl.z, nl.w)), x[2], x[3]);
        const int pv[4] = {ps.x, ps.y, ps.z, ps.w};
        const float dv[4] = {dl.x, dl.y, dl.z, dl.w};
        float ds[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const bool vis = tok_ok && tok <= pv[e];
          const float pe = ex2_approx(x[e]);
          // a hidden token's scores may be NaN (tail or unowned slot): select
          ds[e] = vis ? pe * (__uint_as_float(dr[c0 + e]) - dv[e]) * p.scale : 0.f;
        }
        dsw[2 * c4] = pack_bf16x2(ds[0], ds[1]);
        dsw[2 * c4 + 1] = pack_bf16x2(ds[2], ds[3]);
      }
      // dS^T(b) into shared memory once the products of dS^T(b - 1) are done
      if (b >= 1 && !(ok = mbar_wait_warp(&bar_ds_free, (b - 1) & 1, ab))) break;
      const uint32_t drow = smem_addr(sm + DS_OFF);
#pragma unroll
      for (int j = 0; j < 8; ++j)
        st_shared_v4(drow + sw128_offset(row, j), dsw[4 * j], dsw[4 * j + 1], dsw[4 * j + 2], dsw[4 * j + 3]);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_ds_ready);
    }
    if (nb > 0 && ok) {
      ok = mbar_wait_warp(&bar_acc, 0, ab);
      tc_fence_after();
    }
    // -------------------------------------------------------- epilogue
    // dQ^T (lane = dim) -> shared memory [column][576 dims] bf16 in the Q
    // slots, then row-contiguous stores of dQ and dQp; a tile with no
    // visible token stores zeros
    __nv_bfloat16* stg = reinterpret_cast<__nv_bfloat16*>(sm + QD_OFF);
    if (ok || nb == 0) {
      for (int j = 0; j < 5; ++j) {
        const int dim = (j < 4 ? 128 * j : kLat) + row;
        if (j == 4 && lg >= 2) continue;  // position block: dims 0..63 only (warp-uniform)
#pragma unroll 1
        for (int h = 0; h < 2; ++h) {
          uint32_t r32[32];
          if (nb > 0) {
            tmem_ld32(tmem + T_DQ + 64 * j + 32 * h + lane_addr, r32);
            tmem_ld_wait();
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) r32[i] = 0u;
          }
#pragma unroll
          for (int i = 0; i < 32; ++i) stg[(32 * h + i) * kDims + dim] = __float2bfloat16_rn(__uint_as_float(r32[i]));
        }
      }
    }
    asm volatile("bar.sync 1, 128;" ::: "memory");  // warps 4..7
    if (ok || nb == 0) {
      // 64 columns x 72 16-byte pieces (64 of dQ, 8 of dQp)
      for (int i = row; i < BC * 72; i += 128) {
        const int c = i / 72, k = i - c * 72;
        const int r = r0 + c / G;
        if (r >= re) continue;
        const int64_t idx = static_cast<int64_t>(r) * p.H + g * G + c % G;
        const uint4 v = *reinterpret_cast<const uint4*>(stg + c * kDims + 8 * k);
        if (k < 64)
          *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.dq) + idx * kLat + 8 * k) = v;
        else
          *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.dqp) + idx * kPos + 8 * (k - 64)) = v;
      }
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

bool mla_query_tc_supported(const PagedParams& p) {
  return p.Dk == kLat && p.Dp == kPos && p.page_size == 16 && p.G >= 1 && p.G <= BC && BC % p.G == 0;
}

cudaError_t launch_paged_mla_query_tc(const PagedMlaMaps& m, const PagedParams& p, cudaStream_t s) {
  if (p.Nq == 0 || p.S == 0) return cudaSuccess;
  // the static variables take one 1 KiB granule before the dynamic part
  static_assert(BYTES + 1024 <= 232448, "the layout fits one CTA's shared memory");
  static_assert(BYTES >= kSmemOneCtaPerSm, "all 512 TMEM columns: one CTA per SM");
  const int smem = BYTES;
  cudaError_t e = cudaFuncSetAttribute(mla_query_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  // an upper bound on the row tiles of all sequences; each CTA finds its own
  const int RT = BC / p.G;
  dim3 grid(static_cast<unsigned>((static_cast<int64_t>(p.Nq) / RT + p.S + 1) * p.KVH));
  mla_query_tc_kernel<<<grid, 256, smem, s>>>(m.q, m.qp, m.dy, m.k, m.kp, p);
  return cudaGetLastError();
}

}  // namespace attn
