// Paged MLA history backward on tcgen05 (dK of the latent and of the position
// keys), atomic-free.
//
// ruDNN src/paged_attention/ordered_kernel.rs (history_backward with `mla`):
// for query row r, head h and history token t,
//   s = scale * (q[r,h] . k_lat[t] + qp[r,h] . k_pos[t]),  p = exp(s - lse[r,h])
//   ds = p * (dY[r,h] . k_lat[t] - delta[r,h]) * scale
//   dK_lat[t] += ds * q[r,h] + p * dY[r,h]      (the latent is key and value)
//   dKp[t]    += ds * qp[r,h]
// summed over the links of the token's page (link order), the visible rows of
// each linked sequence (t <= pos(r) when causal) and the heads of the group.
//
// As tile products: a CTA owns 128 tokens (eight pages) of one sequence and
// one KV head; a column is one (query row, head of the group) pair and a tile
// is 64 columns (64/G rows).  Per tile:
//   [S^T | dP^T] = K_lat [Q | dY]^T   [128 x 128], 8 chunks of 64 dims
//   S^T += K_pos Qp^T                 [128 x 64], 1 chunk
//   P^T  = exp2(S^T scale log2e - lse log2e),  dS^T = P^T (dP^T - delta) scale
//   acc  += P^T dY[:, part] + dS^T Q[:, part]   (A operands from tensor
//                                                memory, chunk pairs: N = 128)
// The accumulator of 128 tokens x 576 dims does not fit the 512 tensor-memory
// columns next to the score tiles, so the dims are split over two CTAs
// (PART 0: latent dims [0, 256); PART 1: latent dims [256, 512) and the 64
// position dims); each forms the full S^T and dP^T of its tiles.
//
// A block whose shared pages carry many link tiles (a long prefix shared by
// many sequences) would serialise the other sequences' work on its one owner:
// a plan kernel flags such blocks, the grid kernel leaves them, and a
// persistent kernel of 8-CTA clusters takes them (when few are flagged, cut
// into chunks of contiguous tiles).  CTA r of the cluster that takes a chunk
// runs the r-th eighth of its tiles through the same pipeline into its own
// tensor-memory accumulator; the eight partial sums meet in shared memory and
// each CTA adds 16 tokens' partials over the cluster in rank order
// (distributed shared memory), then stores them, or, for a cut block, leaves
// them in a workspace slot that the block's last chunk adds in chunk order:
// every sum in a fixed order, no floating-point atomics.
//
// Shared memory: the K tile stays resident (latent + position, 9 chunks of
// [128 tokens x 64 dims], 144 KiB); Q, Qp and dY arrive as a stream of 8 KiB
// chunks ([64 columns x 64 dims]) through a 5-stage TMA ring of two chunk
// slots each, in the order
//   (Q, dY) pairs of latent chunk c = 0..7 and Qp of tile t (the pair is the
//   B operand [Q | dY]^T of one N = 128 product), then the part's
//   accumulation chunk pairs of tile t - 1
// Tensor memory: the accumulator, one [S^T | dP^T] tile, and P^T, dS^T as
// bf16 pairs.  The compute warps load [S^T | dP^T](t) and release it at
// once, so the tensor core forms [S|dP](t + 1) while they turn tile t into
// P^T and dS^T, which the accumulation of tile t then reads.  Roles (384
// threads): warp 0 TMA producer (also writes each tile's column statistics),
// warp 1 MMA issuer (whole warp, elect.sync), warps 4..11 compute (every
// tile: warps 4..7 its columns [0, 32), warps 8..11 [32, 64); one TMEM lane
// per token).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>

#include "paged_common.cuh"
#include "paged_launch.h"
#include "paged_pass.cuh"
#include "sm103.cuh"

namespace attn {
using namespace sm103;

namespace {

constexpr int kLat = 512, kPos = 64;
constexpr int BT = 128;                  // tokens per CTA (8 pages of 16)
constexpr int BC = 64;                   // columns per tile
constexpr int kStages = 5;               // ring of stages of two chunk slots
constexpr int kStatSlots = 2;
constexpr int KCH = BT * 128;            // K chunk [128 tokens][64 dims], 16 KiB
constexpr int QCH = BC * 128;            // Q / dY chunk [64 columns][64 dims], 8 KiB
constexpr int K_OFF = 0;                 // 8 latent chunks + 1 position chunk
constexpr int RING_OFF = K_OFF + 9 * KCH;
constexpr int STAGE = 2 * QCH;
constexpr int ST_OFF = RING_OFF + kStages * STAGE;
constexpr int ST_SLOT = 3 * BC * 4 + 16;  // -L2, delta, pos per column + pass info
constexpr int BYTES = ST_OFF + kStatSlots * ST_SLOT;
static_assert(RING_OFF % 1024 == 0 && QCH % 1024 == 0, "swizzled tiles need 1024-byte alignment");
// dynamic shared memory starts 1024-aligned after the static variables (one
// 1 KiB granule): no alignment pad, checked at run time
constexpr int kStaticSmem = 1024;
static_assert(BYTES + kStaticSmem <= 232448, "the layout fits one CTA's shared memory");
// TMEM: accumulator [0, 320) (PART 0 uses [0, 256)); [S^T | dP^T] of the
// current tile [320, 448) (one N = 128 product per key chunk); P^T and dS^T
// as bf16 pairs [448, 480) and [480, 512), the A operands of the
// accumulation
constexpr int T_ACC = 0, T_SDP = 320, T_P = 448, T_DS = 480, TMEM_COLS = 512;

template <int PART>
struct PartShape {
  static constexpr int NACC = PART == 0 ? 8 : 9;    // accumulation chunks per tile
  static constexpr int ACC_COLS = PART == 0 ? 256 : 320;
};

__device__ __forceinline__ bool drain_wait(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_test(bar, parity)) {
    if (global_timer_ns() - t0 > ATTN_WAIT_TIMEOUT_NS) return false;
  }
  return true;
}

// The chunk of job a of the accumulation of a tile: a < 4: dY latent chunk
// (4 PART + a), product P^T dY; a >= 4: Q chunk (4 PART + a - 4), or Qp (a ==
// 8, PART 1 only), product dS^T Q.  Its accumulator chunk (64 columns).
template <int PART>
__device__ __forceinline__ int acc_src_chunk(int a) {
  return a < 4 ? 4 * PART + a : 4 * PART + a - 4;  // 8 = the position chunk
}

// The barriers of the block pipeline: one set per CTA, reused block after
// block by a persistent CTA.
struct TcBars {
  uint64_t k, full[kStages], empty[kStages], st_full[kStatSlots], st_empty[kStatSlots], sdp_full, sdp_free,
      pds_full, pds_free, acc;
};

__device__ __forceinline__ void tc_bars_init(TcBars& b) {
  mbar_init(&b.k, 1);
  for (int s = 0; s < kStages; ++s) {
    mbar_init(&b.full[s], 1);
    mbar_init(&b.empty[s], 1);
  }
  for (int s = 0; s < kStatSlots; ++s) {
    mbar_init(&b.st_full[s], 1);
    mbar_init(&b.st_empty[s], 8);  // the eight compute warps
  }
  mbar_init(&b.sdp_full, 1);  // tensor-core commit
  mbar_init(&b.sdp_free, 8);  // every compute warp has read [S^T | dP^T]
  mbar_init(&b.pds_full, 8);  // every compute warp has written P^T, dS^T
  mbar_init(&b.pds_free, 1);  // tensor-core commit: the accumulation read them
  mbar_init(&b.acc, 1);
  mbar_fence_init();
}

// What the CTA ran before the current block: tiles (score buffers, statistics
// slots), ring jobs and blocks with at least one tile (key tile, accumulator
// commit).  Every barrier phase of a block follows from these.
struct TcEpoch {
  int T, Q, B;
};

// ring jobs per tile: S^T chunks in 5 jobs, dP^T in 4, the accumulation in
// ceil(NACC / 2)
template <int PART>
__host__ __device__ constexpr int jobs_per_tile() {
  return 9 + (PartShape<PART>::NACC + 1) / 2;
}

// Start `it` at tile t of the block's tile sequence (one pass at a time).
__device__ __forceinline__ bool pass_seek(PassIter& it, int rt, int t) {
  if (!it.begin(rt)) return false;
  while (t >= it.ntiles - it.tile) {
    t -= it.ntiles - it.tile;
    if (!it.next_pass(rt)) return false;
  }
  it.tile += t;
  return true;
}

// Tiles [t_begin, t_begin + n) (n > 0) of block tb of sequence s0, KV head
// g, accumulated into tensor memory [T_ACC, T_ACC + ACC_COLS) (the first
// contribution overwrites).  Every role of the CTA calls it; when the
// compute warps return, the accumulator is complete.  Returns false (warp-
// uniformly) when a wait ran out or the CTA is aborting.
//
// Per tile the tensor core forms [S^T | dP^T] = K_c [Q_c | dY_c]^T over the
// eight latent key chunks c (one N = 128 product each: the ring stage holds
// the Q chunk and the dY chunk of the same dims back to back) plus
// K_pos Qp^T into the S^T half, then, once the compute warps have written
// P^T and dS^T, the accumulation in N = 128 products over chunk pairs.  The
// compute warps release [S^T | dP^T] as soon as they have loaded it, so the
// products of tile t + 1 run while they turn tile t into P^T and dS^T: the
// tensor core sees [S|dP](t + 1), acc(t), [S|dP](t + 2), acc(t + 1), ...
template <int PART>
__device__ __forceinline__ bool run_block(const CUtensorMap* tm_q, const CUtensorMap* tm_qp, const CUtensorMap* tm_dy,
                                          const CUtensorMap* tm_k, const CUtensorMap* tm_kp, const PagedParams& p,
                                          TcBars& b, uint8_t* sm, uint32_t tmem, const PageInfo& pinfo, int s0, int tb,
                                          int g, int t_begin, int n, const TcEpoch& ep, const Abort& ab) {
  using PS = PartShape<PART>;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int RT = BC / p.G;                         // query rows per tile
  const int oob_slot = p.num_pages * p.page_size;  // out-of-range coordinate: TMA fills zeros
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      mbar_arrive_expect_tx(&b.k, 9 * KCH);
      for (int j = 0; j < 8; ++j) {
        const int slot = pinfo.phys[j] >= 0 ? pinfo.phys[j] * p.page_size : oob_slot;
        for (int c = 0; c < 8; ++c)
          tma_load_3d(sm + K_OFF + c * KCH + j * 16 * 128, tm_k, &b.k, c * 64, g, slot);
        tma_load_3d(sm + K_OFF + 8 * KCH + j * 16 * 128, tm_kp, &b.k, 0, g, slot);
      }
    }
    PassIter it{&p, &pinfo, s0, tb};
    pass_seek(it, RT, t_begin);
    bool ok = true;
    int q = ep.Q;       // job counter of the ring (a job: one or two chunks)
    int prev_row0 = 0;  // first query row of the previous tile
    int last_use[kStages];
    for (int i = 0; i < kStages; ++i) last_use[i] = -1;
    // column statistics of a tile (two columns per lane) and its pass's token
    // mapping, fetched one tile ahead so that their load latency overlaps the
    // chunk copies of the tile before
    float f_lse[2], f_dl[2];
    int f_pos[2], f_info[4];
    auto fetch = [&](const PassIter& x) {
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
    fetch(it);
    // one job into the ring: chunk (m0, dims x0) into the stage's first slot
    // and, when m1 is not null, chunk (m1, dims x1) into its second
    auto load_job = [&](const CUtensorMap* m0, int x0, const CUtensorMap* m1, int x1, int row0) -> bool {
      const int s = q % kStages;
      if (q >= kStages && !mbar_wait(&b.empty[s], ((q / kStages) - 1) & 1, ab)) return false;
      if (lane == 0) {
        mbar_arrive_expect_tx(&b.full[s], (m1 ? 2 : 1) * QCH);
        tma_load_3d(sm + RING_OFF + s * STAGE, m0, &b.full[s], x0, g * p.G, row0);
        if (m1) tma_load_3d(sm + RING_OFF + s * STAGE + QCH, m1, &b.full[s], x1, g * p.G, row0);
      }
      last_use[s] = q;
      ++q;
      return true;
    };
    // the accumulation jobs of a tile: dY chunks of the part in pairs, then
    // its Q chunks in pairs (and Qp alone, PART 1)
    auto load_acc = [&](int row0) -> bool {
      for (int a = 0; a < PS::NACC; a += 2) {
        const int c = acc_src_chunk<PART>(a);
        const CUtensorMap* m = a < 4 ? tm_dy : c == 8 ? tm_qp : tm_q;
        const bool pair = PS::NACC - a >= 2;
        if (!load_job(m, c == 8 ? 0 : c * 64, pair ? m : nullptr, (c + 1) * 64, row0)) return false;
      }
      return true;
    };
    for (int t = 0; t <= n && ok; ++t) {
      if (t < n) {
        const int row0 = it.r_begin + it.tile * RT;
        // [S | dP] chunks of tile t: (Q, dY) latent chunk pairs, then Qp
        for (int c = 0; c < 8 && ok; ++c) ok = load_job(tm_q, c * 64, tm_dy, c * 64, row0);
        if (ok) ok = load_job(tm_qp, 0, nullptr, 0, row0);
        if (!ok) break;
        // column statistics of tile t: -L2, delta, pos per column (a row
        // with lse = -inf sees no token), plus the pass's token mapping;
        // after its chunk copies, so that waiting for the slot (tile t - 2
        // done) never holds them back
        const int gt = ep.T + t, ss = gt % kStatSlots;
        if (gt >= kStatSlots && !(ok = mbar_wait(&b.st_empty[ss], ((gt / kStatSlots) - 1) & 1, ab))) break;
        uint8_t* st = sm + ST_OFF + ss * ST_SLOT;
        float* snl = reinterpret_cast<float*>(st);
        float* sdl = snl + BC;
        int* spos = reinterpret_cast<int*>(sdl + BC);
        int* sinfo = spos + BC;
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
        if (lane == 0) mbar_arrive(&b.st_full[ss]);
        PassIter nx = it;
        if (t + 1 < n) {
          nx.advance(RT);
          fetch(nx);
        }
        // the accumulation chunks of tile t - 1
        if (t >= 1) ok = load_acc(prev_row0);
        if (!ok) break;
        prev_row0 = row0;
        it = nx;
      } else {
        ok = load_acc(prev_row0);
      }
    }
    if (lane == 0) {
      for (int s = 0; s < kStages; ++s)
        if (last_use[s] >= 0) drain_wait(&b.full[s], (last_use[s] / kStages) & 1);
      drain_wait(&b.k, ep.B & 1);
    }
    return ok;
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // the whole warp runs this role (warp-uniform); elected lanes issue
    constexpr uint32_t id_sdp = idesc_bf16(128, 2 * BC, false, false);  // [S^T | dP^T]: K-major A and B
    constexpr uint32_t id_s = idesc_bf16(128, BC, false, false);        // S^T += K_pos Qp^T
    constexpr uint32_t id_acc2 = idesc_bf16(128, 128, false, true);     // acc, a chunk pair: A from TMEM, B MN-major
    constexpr uint32_t id_acc1 = idesc_bf16(128, 64, false, true);      // acc, one chunk (Qp)
    const uint64_t dK0 = sdesc_sw128(smem_addr(sm + K_OFF), 16, 1024);
    const uint64_t dR0 = sdesc_sw128(smem_addr(sm + RING_OFF), 16, 1024);         // K-major, 128 rows per stage
    const uint64_t dRm0 = sdesc_sw128(smem_addr(sm + RING_OFF), QCH, 1024);       // MN-major, chunks QCH apart
    bool ok = mbar_wait_warp(&b.k, ep.B & 1, ab);
    int q = ep.Q;
    // a stage's copies are usually in by the time this warp reaches it: a
    // non-blocking test first, the bounded wait only when it is not
    auto wait_stage = [&](int qq) -> bool {
      const int s = qq % kStages;
      if (mbar_test_warp(&b.full[s], (qq / kStages) & 1)) return true;
      return mbar_wait_warp(&b.full[s], (qq / kStages) & 1, ab);
    };
    // after the job of ring index qq: its stage goes back to the producer
    // once its products are done
    auto release = [&](int qq) { mma_commit_w(&b.empty[qq % kStages]); };
    for (int t = 0; t <= n && ok; ++t) {
      if (t < n) {
        // [S^T | dP^T](t) once the compute warps have loaded tile t - 1's
        const int gt = ep.T + t;
        if (gt >= 1 && !(ok = mbar_wait_warp(&b.sdp_free, (gt - 1) & 1, ab))) break;
        tc_fence_after();
        const uint32_t d = tmem + T_SDP;
        for (int c = 0; c < 9 && ok; ++c, ++q) {
          if (!(ok = wait_stage(q))) break;
          tc_fence_after();
          const uint64_t a = sdesc_add(dK0, c * KCH), bq = sdesc_add(dR0, (q % kStages) * STAGE);
          const uint32_t id = c < 8 ? id_sdp : id_s;
          if (c == 0)
            mma_ss_w<false>(d, a, bq, id);
          else
            mma_ss_w<true>(d, a, bq, id);
#pragma unroll
          for (int kk = 1; kk < 4; ++kk) mma_ss_w<true>(d, sdesc_add(a, kk * 32), sdesc_add(bq, kk * 32), id);
          release(q);
        }
        if (!ok) break;
        mma_commit_w(&b.sdp_full);
      }
      if (t >= 1) {
        // accumulation of tile u = t - 1 once its P^T and dS^T are in: P^T dY
        // chunk pairs, then dS^T Q chunk pairs (and dS^T Qp, PART 1)
        const int u = t - 1, gu = ep.T + u;
        if (!(ok = mbar_wait_warp(&b.pds_full, gu & 1, ab))) break;
        tc_fence_after();
        for (int a0 = 0; a0 < PS::NACC && ok; a0 += 2, ++q) {
          if (!(ok = wait_stage(q))) break;
          tc_fence_after();
          const int c = acc_src_chunk<PART>(a0);
          const uint32_t d = tmem + T_ACC + (c - 4 * PART) * 64;  // chunk 8 (position) -> 256
          const uint32_t at = tmem + (a0 < 4 ? T_P : T_DS);
          const uint64_t bm = sdesc_add(dRm0, (q % kStages) * STAGE);
          const uint32_t id = PS::NACC - a0 >= 2 ? id_acc2 : id_acc1;
          // the first contribution to an accumulator chunk overwrites it:
          // P^T dY for latent chunks, dS^T Qp for the position chunk
          if (u == 0 && (a0 < 4 || c == 8))
            mma_ts_w<false>(d, at, bm, id);
          else
            mma_ts_w<true>(d, at, bm, id);
#pragma unroll
          for (int kk = 1; kk < BC / 16; ++kk) mma_ts_w<true>(d, at + kk * 8, sdesc_add(bm, kk * 16 * 128), id);
          release(q);
        }
        if (!ok) break;
        mma_commit_w(&b.pds_free);
      }
    }
    mma_commit_w(&b.acc);
    drain_wait(&b.acc, ep.B & 1);
    __syncwarp();
    return ok;
  } else if (warp >= 4) {
    // ------------------------------------------------------------ compute
    // every tile: warps 4..7 take its columns [0, 32), warps 8..11 [32, 64),
    // one TMEM lane (token) per thread
    const int sg = (warp - 4) >> 2;
    const int lg = warp & 3;
    const int row = lg * 32 + lane;  // token row inside the block == TMEM lane
    const uint32_t lane_addr = static_cast<uint32_t>(lg * 32) << 16;
    const int cb = 32 * sg;  // first column of this group
    bool ok = true;
    for (int t = 0; t < n && ok; ++t) {
      const int gt = ep.T + t, ss = gt % kStatSlots;
      if (!(ok = mbar_wait_warp(&b.st_full[ss], (gt / kStatSlots) & 1, ab))) break;
      const uint8_t* st = sm + ST_OFF + ss * ST_SLOT;
      const float* snl = reinterpret_cast<const float*>(st);
      const float* sdl = snl + BC;
      const int* spos = reinterpret_cast<const int*>(sdl + BC);
      const int* sinfo = spos + BC;
      const int tok = sinfo[0] + row;
      const bool tok_ok = row >= sinfo[1] && row < sinfo[2] && tok >= 0 && tok < sinfo[3];
      if (!(ok = mbar_wait_warp(&b.sdp_full, gt & 1, ab))) break;
      tc_fence_after();
      uint32_t sr[32], dr[32];
      tmem_ld32(tmem + T_SDP + cb + lane_addr, sr);
      tmem_ld32(tmem + T_SDP + BC + cb + lane_addr, dr);
      tmem_ld_wait();
      // [S^T | dP^T] may now take the next tile's products
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&b.sdp_free);
      // ---------------------------------------------------- S^T -> P^T
      const uint64_t sl2 = f2_pack(p.scale_log2, p.scale_log2);
      uint32_t pw[16], dsw[16];
#pragma unroll
      for (int c4 = 0; c4 < 8; ++c4) {
        const int c0 = cb + 4 * c4;
        const float4 nl = *reinterpret_cast<const float4*>(snl + c0);
        const int4 ps = *reinterpret_cast<const int4*>(spos + c0);
        float x0, x1, x2, x3;
        f2_split(f2_fma(f2_pack_u(sr[4 * c4], sr[4 * c4 + 1]), sl2, f2_pack(nl.x, nl.y)), x0, x1);
        f2_split(f2_fma(f2_pack_u(sr[4 * c4 + 2], sr[4 * c4 + 3]), sl2, f2_pack(nl.z, nl.w)), x2, x3);
        const float p0 = (tok_ok && tok <= ps.x) ? ex2_approx(x0) : 0.f;
        const float p1 = (tok_ok && tok <= ps.y) ? ex2_approx(x1) : 0.f;
        const float p2 = (tok_ok && tok <= ps.z) ? ex2_approx(x2) : 0.f;
        const float p3 = (tok_ok && tok <= ps.w) ? ex2_approx(x3) : 0.f;
        pw[2 * c4] = pack_bf16x2(p0, p1);
        pw[2 * c4 + 1] = pack_bf16x2(p2, p3);
      }
      // ---------------------------------------------------- dP^T, P^T -> dS^T
      // a masked entry has P = 0 and takes dS = 0 by select: dP of a tail or
      // unowned slot may be NaN
#pragma unroll
      for (int c4 = 0; c4 < 8; ++c4) {
        const float4 d4 = *reinterpret_cast<const float4*>(sdl + cb + 4 * c4);
        const float dv[4] = {d4.x, d4.y, d4.z, d4.w};
        float ds[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const uint32_t w = pw[2 * c4 + (e >> 1)];
          const float pe = __uint_as_float((e & 1) ? (w & 0xffff0000u) : (w << 16));
          ds[e] = pe != 0.f ? pe * (__uint_as_float(dr[4 * c4 + e]) - dv[e]) * p.scale : 0.f;
        }
        dsw[2 * c4] = pack_bf16x2(ds[0], ds[1]);
        dsw[2 * c4 + 1] = pack_bf16x2(ds[2], ds[3]);
      }
      // P^T and dS^T of tile gt - 1 have been read by its accumulation
      if (gt >= 1 && !(ok = mbar_wait_warp(&b.pds_free, (gt - 1) & 1, ab))) break;
      tc_fence_after();
      tmem_st16(tmem + T_P + cb / 2 + lane_addr, pw);
      tmem_st16(tmem + T_DS + cb / 2 + lane_addr, dsw);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&b.pds_full);
        mbar_arrive(&b.st_empty[ss]);
      }
    }
    if (ok) ok = mbar_wait_warp(&b.acc, ep.B & 1, ab);
    tc_fence_after();
    return ok;
  }
  return true;
}

// A 128-token block whose link passes (shared pages) exceed this many tiles
// goes to the split kernel (its own pass has 64 rows x G heads / 64 columns).
constexpr int kHeavyLinkTiles = 64;
constexpr int kSplitCL = 8;                       // CTAs of a split cluster; CTA r sums tokens [16r, 16r + 16)
constexpr int kMinPieceTiles = 4;                 // a block is not cut into pieces smaller than this
constexpr int kItemTiles = 8;                     // fixed cost of a split item, in tiles
constexpr int RED_STRIDE = 324;                   // floats per token row of a staged partial (320 + 4: bank spread)
static_assert(BT * RED_STRIDE * 4 <= BYTES, "a partial fits the pipeline's shared memory");
static_assert(BT % kSplitCL == 0, "tokens split evenly over the cluster");

// The rows of the pages this block stores: 32-column chunks of the part's
// accumulator, alternating between the compute groups (latent dims [256 PART
// + 32 cc, ...) for cc < 8, position dims after that, PART 1); rows of tokens
// no pass saw are zero (n = 0).  Called by the compute warps.
template <int PART>
__device__ __forceinline__ void store_block(const PagedParams& p, uint32_t tmem, const PageInfo& pinfo, int g, int n,
                                            bool ok) {
  using PS = PartShape<PART>;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int sg = (warp - 4) >> 2;
  const int lg = warp & 3;
  const int row = lg * 32 + lane;  // token row inside the block == TMEM lane
  const uint32_t lane_addr = static_cast<uint32_t>(lg * 32) << 16;
  if (ok || n == 0) {  // warp-uniform: the tensor-memory loads are warp-collective
    const int j = row >> 4;
    const bool mine = pinfo.store[j] != 0;
    const int64_t prow = (static_cast<int64_t>(pinfo.phys[j]) * p.page_size + (row & 15)) * p.KVH + g;
#pragma unroll 1
    for (int cc = sg; cc < PS::ACC_COLS / 32; cc += 2) {
      const bool pos_chunk = cc >= 8;
      if (!(p.wrt & (pos_chunk ? 8u : 2u))) continue;
      uint32_t r[32];
      if (n > 0) {
        tmem_ld32(tmem + T_ACC + cc * 32 + lane_addr, r);
        tmem_ld_wait();
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) r[i] = 0u;
      }
      if (mine) {
        __nv_bfloat16* out = pos_chunk
                                 ? static_cast<__nv_bfloat16*>(p.dkp_pool) + prow * kPos + (cc - 8) * 32
                                 : static_cast<__nv_bfloat16*>(p.dk_pool) + prow * kLat + 256 * PART + cc * 32;
        store_row32_bf16(out, r, 1.f, 32);
      }
    }
  }
}

// The grid part of the MLA history, one launch per part: persistent CTAs (one
// per SM) take units (sequence, 128-token block, KV head) from the part's
// counter; a unit runs the block's tiles through the pipeline and stores the
// rows of the pages it owns.  Blocks the plan flagged
// belong to the split kernel, blocks past a sequence's end do not exist here.
// Each unit is computed whole by one CTA, so the results do not depend on
// which CTA takes it.
template <int PART>
__global__ void __launch_bounds__(384, 1)
    mla_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_qp,
                  const __grid_constant__ CUtensorMap tm_dy, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_kp, const PagedParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = smem_raw;
  __shared__ TcBars bars;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag;
  __shared__ PageInfo pinfo;
  __shared__ int unit_sh[3], n_tiles_sh, any_store_sh;
  if (smem_addr(smem_raw) & 1023u) {  // uniform: the swizzled tiles need 1024-byte alignment
    if (threadIdx.x == 0 && p.err) atomicOr(p.err, DEV_ERR_LAYOUT);
    return;
  }

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int RT = BC / p.G;  // query rows per tile
  const int nb128 = (p.max_pages + 7) / 8;
  constexpr int part = PART;
  const Abort ab{&abort_flag, p.err};
  // Launched as the programmatic dependent of the kernel before it (the
  // split kernel, or part 0 for part 1), whose results it does not read (the
  // plan it reads completed before the split kernel started): its own
  // dependent may start at once, on the SMs it leaves free, and its last CTA
  // waits for the kernel before after its own units, so that this grid
  // completes after it and later work in the stream sees both.  Without a
  // programmatic launch both are no-ops.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (threadIdx.x == 0) {
    abort_flag = 0;
    tc_bars_init(bars);
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base_sh, TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_map(&tm_q);
    tma_prefetch_map(&tm_qp);
    tma_prefetch_map(&tm_dy);
    tma_prefetch_map(&tm_k);
    tma_prefetch_map(&tm_kp);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  TcEpoch ep{0, 0, 0};
  while (true) {
    __syncthreads();  // the previous unit's readers of pinfo and unit_sh are done
    if (warp == 0) {
      // unit k of the part: sequences in order, each with blocks x KV heads;
      // the warp finds the sequence 32 at a time (a prefix sum of their
      // units) and its lanes 0..7 resolve the block's eight pages
      int k = 0;
      if (lane == 0) k = atomicAdd(p.work + part, 1);
      k = __shfl_sync(0xffffffffu, k, 0);
      int s0 = -1, base = 0;
      for (int c0 = 0; c0 < p.S && s0 < 0; c0 += 32) {  // warp-uniform
        const int s = c0 + lane;
        const int u = s < p.S ? ((seq_len_of(p, s) + BT - 1) / BT) * p.KVH : 0;
        int x = u;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, x, o);
          if (lane >= o) x += y;
        }
        const int excl = base + x - u;
        const unsigned hit = __ballot_sync(0xffffffffu, k >= excl && k < excl + u);
        if (hit) {
          const int l = __ffs(hit) - 1;
          s0 = c0 + l;
          k -= __shfl_sync(0xffffffffu, excl, l);
        }
        base += __shfl_sync(0xffffffffu, x, 31);
      }
      int any = 0, n = 0, g = 0, tb = 0;
      if (s0 >= 0) {
        g = k % p.KVH;
        tb = k / p.KVH;
        const int st = lane < 8 ? fill_page_entry(p, s0, tb, pages_of(seq_len_of(p, s0), p.page_size), lane, &pinfo) : 0;
        any = __any_sync(0xffffffffu, st != 0);
        __syncwarp();
        // a block the plan flagged belongs to the cluster-split kernel
        if (any && p.heavy[(static_cast<int64_t>(s0) * nb128 + tb) * p.KVH + g]) any = 0;
        if (lane == 0 && any) {
          PassIter it{&p, &pinfo, s0, tb};
          if (it.begin(RT)) {
            do n += it.ntiles;
            while (it.next_pass(RT));
          }
        }
      }
      if (lane == 0) {
        unit_sh[0] = s0;
        unit_sh[1] = tb;
        unit_sh[2] = g;
        any_store_sh = any;
        n_tiles_sh = n;
      }
    }
    __syncthreads();
    if (unit_sh[0] < 0) break;  // no units left (uniform)
    // a block whose pages are all stored by other CTAs (their owners) has
    // nothing to write (uniform)
    if (!any_store_sh) continue;
    const int s0 = unit_sh[0], tb = unit_sh[1], g = unit_sh[2];
    const int n = n_tiles_sh;
    bool ok = true;
    if (n > 0) ok = run_block<PART>(&tm_q, &tm_qp, &tm_dy, &tm_k, &tm_kp, p, bars, sm, tmem, pinfo, s0, tb, g, 0, n, ep, ab);
    if (warp >= 4) {
      store_block<PART>(p, tmem, pinfo, g, n, ok);
      tc_fence_before();
    }
    if (n > 0) {
      ep.T += n;
      ep.Q += n * jobs_per_tile<PART>();
      ++ep.B;
    }
  }
  if (blockIdx.x == gridDim.x - 1) asm volatile("griddepcontrol.wait;" ::: "memory");
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// Cluster primitives of the split kernel.
__device__ __forceinline__ int cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return static_cast<int>(r);
}
__device__ __forceinline__ int cluster_count() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return static_cast<int>(r);
}
// All threads of all CTAs of the cluster: shared-memory writes before it are
// visible to the other CTAs' reads after it.  Every CTA of a cluster passes
// the same number of these (its waits give up after a time limit, so none is
// held back for ever).
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}
// the same shared-memory offset in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t map_rank(uint32_t addr, int rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
__device__ __forceinline__ int ld_cluster_s32(uint32_t addr) {
  int v;
  asm volatile("ld.shared::cluster.s32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ float4 ld_cluster_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

// Tiles of the passes at link index li >= 1 of a block (the stored pages
// pi): the passes PassIter::next_pass enumerates at that index, each run of
// consecutive stored pages whose li-th links are consecutive logical pages
// of one sequence counting that sequence's row tiles once.
__device__ int link_tiles_at(const PagedParams& p, const PageInfo& pi, int li, int rt) {
  int n = 0;
  for (int j = 0; j < 8;) {
    if (!(pi.store[j] && li < pi.cnt[j])) {
      ++j;
      continue;
    }
    const int link = p.links[pi.off[j] + li];
    const int s2 = link / p.max_pages, lp2 = link - s2 * p.max_pages;
    int jn = j + 1;
    while (jn < 8 && pi.store[jn] && li < pi.cnt[jn] && lp2 + (jn - j) < p.max_pages &&
           p.links[pi.off[jn] + li] == link + (jn - j))
      ++jn;
    const int rb = row_begin_of(p, s2);
    n += (row_end_of(p, s2) - rb + rt - 1) / rt;
    j = jn;
  }
  return n;
}

// Plan of the MLA history: heavy[(s0 * nblk + tb) * KVH + g] = the block's
// tile count when the pages 128-token block tb of sequence s0 stores carry
// more than kHeavyLinkTiles tiles of other links, else 0; one warp per block,
// its lanes taking the link indices.
__global__ void mla_tc_plan_kernel(const PagedParams p) {
  const int nblk = (p.max_pages + 7) / 8;
  const int n = p.S * nblk;
  const int RT = BC / p.G;
  const int lane = threadIdx.x & 31, wpb = static_cast<int>(blockDim.x >> 5);
  if (blockIdx.x == 0)  // the grid and split kernels' counters
    for (int i = threadIdx.x; i < kMlaWorkInts; i += blockDim.x) p.work[i] = 0;
  for (int i = blockIdx.x * wpb + static_cast<int>(threadIdx.x >> 5); i < n; i += gridDim.x * wpb) {  // warp-uniform
    const int s0 = i / nblk, tb = i - s0 * nblk;
    const int npg = pages_of(seq_len_of(p, s0), p.page_size);
    int heavy = 0;
    if (tb * 8 < npg) {
      PageInfo pi;
      if (fill_page_info(p, s0, tb, npg, &pi)) {
        int lmax = 0;
        for (int k = 0; k < 8; ++k)
          if (pi.store[k] && pi.cnt[k] > lmax) lmax = pi.cnt[k];
        int n_link = 0;
        for (int li = 1 + lane; li < lmax; li += 32) n_link += link_tiles_at(p, pi, li, RT);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) n_link += __shfl_xor_sync(0xffffffffu, n_link, o);
        const int rb = row_begin_of(p, s0);
        const int n_own = (row_end_of(p, s0) - rb + RT - 1) / RT;  // the block's own pass
        heavy = n_link > kHeavyLinkTiles ? n_own + n_link : 0;
      }
    }
    for (int g = lane; g < p.KVH; g += 32) p.heavy[static_cast<int64_t>(i) * p.KVH + g] = heavy;
  }
}

// Persistent clusters of kSplitCL CTAs, one launch per part (a kernel holding
// both parts' pipelines needs more registers and ran slower).  The work of a
// part is nflag x C items: item k is chunk c = k / nflag of the (k mod
// nflag)-th flagged block in flag order, and the clusters take items from the
// part's counter.  C minimises the rounds of the clusters times the item
// cost (its tiles plus a fixed cost): 1 when the blocks already fill whole
// rounds, more when a few heavy blocks would leave clusters idle.
//
// The block's n tiles form 8C contiguous pieces; CTA r of the cluster that
// takes chunk c runs piece 8c + r into its tensor-memory accumulator, stages
// the partial in shared memory, and after a cluster barrier adds tokens
// [16 r, 16 r + 16) over the cluster's partials in rank order.  With C = 1
// that sum is stored; otherwise it goes to the chunk's fp32 slot, and the CTA
// of rank r that completes a block's last chunk (a per-rank counter) adds the
// block's C slots in chunk order and stores the sum.  Every sum has a fixed
// order, so the result does not depend on which cluster takes which item.
template <int PART>
__global__ void __launch_bounds__(384, 1)
    mla_tc_split_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_qp,
                        const __grid_constant__ CUtensorMap tm_dy, const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_kp, const PagedParams p) {
  static_assert(kSplitCL == kMlaSplitRanks, "the counters hold one entry per cluster rank");
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = smem_raw;
  __shared__ TcBars bars;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag, abort_any_sh;
  __shared__ PageInfo pinfo;
  __shared__ int item_sh, k_sh, found_sh, last_sh, min_tiles_sh;
  constexpr int kListed = kMlaSplitSlots / 2;  // more flagged blocks than this: C = 1
  __shared__ int listed_sh[kListed];
  __shared__ int warp_cnt[12];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nwarps = static_cast<int>(blockDim.x >> 5);
  const int rank = cluster_rank(), ncl = cluster_count();
  const int nblk = (p.max_pages + 7) / 8;
  const int nitems = p.S * nblk * p.KVH;
  constexpr int acc_cols = PartShape<PART>::ACC_COLS;
  const Abort ab{&abort_flag, p.err};
  if (smem_addr(smem_raw) & 1023u) {  // every CTA alike: the swizzled tiles need 1024-byte alignment
    if (threadIdx.x == 0 && p.err) atomicOr(p.err, DEV_ERR_LAYOUT);
    return;
  }
  // the kernels launched next (part 1, then the grid kernels) as programmatic
  // dependents may start on the SMs these clusters leave free; part 1's last
  // CTA waits for part 0 at the end, so that the chain completes in order
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (threadIdx.x == 0) {
    abort_flag = 0;
    tc_bars_init(bars);
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base_sh, TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_map(&tm_q);
    tma_prefetch_map(&tm_qp);
    tma_prefetch_map(&tm_dy);
    tma_prefetch_map(&tm_k);
    tma_prefetch_map(&tm_kp);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  float* red = reinterpret_cast<float*>(sm);  // staged partial: [BT][RED_STRIDE] fp32
  float* slots = p.split_part + (PART == 1 ? static_cast<size_t>(kMlaSplitSlots) * BT * 256 : 0);
  int32_t* done = p.work + 4 + PART * kMlaSplitSlots * kMlaSplitRanks;
  TcEpoch ep{0, 0, 0};

  // One window of blockDim.x block indices from c0: the flagged ones are
  // ranked in index order from `base`; returns the window's flagged count and
  // records in found_sh the index ranked `want` if it lies in the window.
  auto window = [&](int c0, int base, int want) {
    const int i = c0 + threadIdx.x;
    const int h = i < nitems ? p.heavy[i] : 0;
    const bool f = h != 0;
    if (want < 0 && f) atomicMin(&min_tiles_sh, h);  // the counting pass
    const uint32_t bal = __ballot_sync(0xffffffffu, f);
    if (lane == 0) warp_cnt[warp] = __popc(bal);
    __syncthreads();
    int before = 0, total = 0;
    for (int w = 0; w < nwarps; ++w) {
      const int c = warp_cnt[w];
      before += w < warp ? c : 0;
      total += c;
    }
    const int at = base + before + __popc(bal & ((1u << lane) - 1u));
    if (f && at == want) found_sh = i;
    if (want < 0 && f && at < kListed) listed_sh[at] = i;  // the counting pass
    __syncthreads();  // warp_cnt is rewritten by the next window
    return total;
  };
  if (threadIdx.x == 0) min_tiles_sh = 0x7fffffff;
  __syncthreads();
  int nflag = 0;
  for (int c0 = 0; c0 < nitems; c0 += blockDim.x) nflag += window(c0, nflag, -1);
  // C: the fewest rounds of the clusters, each item costing its tiles plus a
  // fixed kItemTiles (key tile, pipeline fill and drain, the partials'
  // exchange), no piece of the smallest flagged block below kMinPieceTiles
  // tiles and at most kMlaSplitSlots open chunk partials
  int C = 1;
  if (nflag > 0) {
    const int cmax = max(1, min(kMlaSplitSlots / nflag, min_tiles_sh / (kSplitCL * kMinPieceTiles)));
    int64_t best = -1;
    for (int c = 1; c <= cmax; ++c) {
      const int64_t rounds = (static_cast<int64_t>(nflag) * c + ncl - 1) / ncl;
      const int64_t cost = rounds * ((min_tiles_sh + kSplitCL * c - 1) / (kSplitCL * c) + kItemTiles);
      if (best < 0 || cost < best) {
        best = cost;
        C = c;
      }
    }
  }
  const int n_work = nflag * C;
  // the u-th flagged block: listed when u < kListed (always when C > 1),
  // else searched from where the last search ended (with C = 1 a cluster's
  // items, and so its u, increase)
  int scan_c0 = 0, scan_base = 0;

  auto run_item = [&](int u, int c) {
    int item = u < kListed ? listed_sh[u] : -1;
    while (item < 0 && scan_c0 < nitems) {  // uniform: every thread sees the same windows
      const int total = window(scan_c0, scan_base, u);
      if (u < scan_base + total) {
        item = found_sh;
      } else {
        scan_base += total;
        scan_c0 += blockDim.x;
      }
    }
    if (item < 0) return;  // not reached: u < nflag
    const int g = item % p.KVH, rest = item / p.KVH, tb = rest % nblk, s0 = rest / nblk;
    __syncthreads();  // found_sh is read; the previous item's readers of pinfo are done
    if (warp == 0 && lane < 8)  // the block's eight pages side by side
      fill_page_entry(p, s0, tb, pages_of(seq_len_of(p, s0), p.page_size), lane, &pinfo);
    __syncthreads();
    const int64_t n_all = p.heavy[item], pieces = static_cast<int64_t>(kSplitCL) * C, q = static_cast<int64_t>(c) * kSplitCL + rank;
    const int t0 = static_cast<int>(q * n_all / pieces), n = static_cast<int>((q + 1) * n_all / pieces) - t0;
    // (a wait that gives up sets the abort flag, which the cluster reads below)
    if (n > 0) run_block<PART>(&tm_q, &tm_qp, &tm_dy, &tm_k, &tm_kp, p, bars, sm, tmem, pinfo, s0, tb, g, t0, n, ep, ab);
    // every role is done with the pipeline's shared memory and the
    // accumulator is complete: stage the partial (zeros without tiles)
    __syncthreads();
    if (warp >= 4) {
      const int sg = (warp - 4) >> 2, lg = warp & 3;
      const int row = lg * 32 + lane;
      const uint32_t lane_addr = static_cast<uint32_t>(lg * 32) << 16;
#pragma unroll 1
      for (int cc = sg; cc < acc_cols / 32; cc += 2) {  // warp-uniform
        uint32_t r[32];
        if (n > 0) {
          tmem_ld32(tmem + T_ACC + cc * 32 + lane_addr, r);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) r[i] = 0u;
        }
        float* dst = red + row * RED_STRIDE + cc * 32;
#pragma unroll
        for (int i = 0; i < 8; ++i)
          *reinterpret_cast<uint4*>(dst + 4 * i) = make_uint4(r[4 * i], r[4 * i + 1], r[4 * i + 2], r[4 * i + 3]);
      }
      tc_fence_before();
    }
    // every CTA's abort flag is ORed over the cluster: a partial left
    // incomplete by a timed-out wait must not reach the pool as a finite value
    if (threadIdx.x == 0) abort_any_sh = abort_flag;
    cluster_sync();
    if (threadIdx.x == 0) {
      int any_abort = 0;
      for (int r = 0; r < kSplitCL; ++r) any_abort |= ld_cluster_s32(map_rank(smem_addr(&abort_any_sh), r));
      if (any_abort) abort_flag = 1;
    }
    __syncthreads();
    const bool good = !abort_flag;
    // tokens [16 rank, 16 rank + 16), one page: the partials of CTAs
    // 0..kSplitCL-1 added in that order
    constexpr int kRows = BT / kSplitCL;
    constexpr int quads = acc_cols / 4;
    const int j = (kRows * rank) >> 4;
    auto store4 = [&](int i, int d, float4 sum) {
      const int64_t prow = (static_cast<int64_t>(pinfo.phys[j]) * p.page_size + (i & 15)) * p.KVH + g;
      const uint2 w = make_uint2(pack_bf16x2(sum.x, sum.y), pack_bf16x2(sum.z, sum.w));
      if (d < 256) {
        if (p.wrt & 2u)
          *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(p.dk_pool) + prow * kLat + 256 * PART + d) = w;
      } else if (p.wrt & 8u) {
        *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(p.dkp_pool) + prow * kPos + (d - 256)) = w;
      }
    };
    const bool mine = good && pinfo.store[j] != 0;
    float* slot = C > 1 ? slots + (static_cast<size_t>(u) * C + c) * BT * acc_cols : nullptr;
    if (mine) {
      for (int idx = threadIdx.x; idx < kRows * quads; idx += blockDim.x) {
        const int i = kRows * rank + idx / quads, d = 4 * (idx % quads);
        const uint32_t a = smem_addr(red + i * RED_STRIDE + d);
        float4 sum = ld_cluster_f4(map_rank(a, 0));
#pragma unroll
        for (int r = 1; r < kSplitCL; ++r) {
          const float4 v = ld_cluster_f4(map_rank(a, r));
          sum.x += v.x;
          sum.y += v.y;
          sum.z += v.z;
          sum.w += v.w;
        }
        if (C == 1)
          store4(i, d, sum);
        else
          *reinterpret_cast<float4*>(slot + i * acc_cols + d) = sum;
      }
      if (C > 1) __threadfence();  // the slot rows, before this CTA's count below
    }
    cluster_sync();  // the other CTAs have read this CTA's partial
    if (n > 0) {
      ep.T += n;
      ep.Q += n * jobs_per_tile<PART>();
      ++ep.B;
    }
    if (C > 1 && mine) {
      // the last of the block's C chunks to reach this rank adds the slots
      if (threadIdx.x == 0) {
        last_sh = atomicAdd(done + u * kMlaSplitRanks + rank, 1) == C - 1;
        __threadfence();
      }
      __syncthreads();
      if (last_sh) {
        const float* first = slots + static_cast<size_t>(u) * C * BT * acc_cols;
        for (int idx = threadIdx.x; idx < kRows * quads; idx += blockDim.x) {
          const int i = kRows * rank + idx / quads, d = 4 * (idx % quads);
          const float* src = first + i * acc_cols + d;
          float4 sum = __ldcg(reinterpret_cast<const float4*>(src));
#pragma unroll 4
          for (int c2 = 1; c2 < C; ++c2) {
            const float4 v = __ldcg(reinterpret_cast<const float4*>(src + static_cast<size_t>(c2) * BT * acc_cols));
            sum.x += v.x;
            sum.y += v.y;
            sum.z += v.z;
            sum.w += v.w;
          }
          store4(i, d, sum);
        }
      }
    }
  };

  while (true) {
    // rank 0 takes the cluster's next item; the others read it from rank 0
    // (its next write comes after the item's cluster barriers)
    if (rank == 0 && threadIdx.x == 0) item_sh = atomicAdd(p.work + 2 + PART, 1);
    cluster_sync();
    if (threadIdx.x == 0) k_sh = ld_cluster_s32(map_rank(smem_addr(&item_sh), 0));
    __syncthreads();
    const int k = k_sh;
    if (k >= n_work) break;  // cluster-uniform
    // chunk-major: the clusters running at one time work on the same chunk
    // of different blocks, whose passes read the same query rows (L2 reuse)
    run_item(k % nflag, k / nflag);
  }
  cluster_sync();  // rank 0's shared memory outlives the others' last read of it
  if (PART == 1 && blockIdx.x == gridDim.x - 1) asm volatile("griddepcontrol.wait;" ::: "memory");
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

template <int PART>
cudaError_t launch_split(const PagedMlaMaps& m, const PagedParams& p, int ncl, bool dependent, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(mla_tc_split_kernel<PART>, cudaFuncAttributeMaxDynamicSharedMemorySize, BYTES);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = kSplitCL;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[1].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ncl * kSplitCL, 1, 1);
  cfg.blockDim = dim3(384, 1, 1);
  cfg.dynamicSmemBytes = BYTES;
  cfg.stream = s;
  cfg.attrs = at;
  cfg.numAttrs = dependent ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, mla_tc_split_kernel<PART>, m.q, m.qp, m.dy, m.k, m.kp, p);
}

// How many kSplitCL-CTA clusters of the split kernel fit the GPU at once (one
// CTA per SM), cached per device (host threads may race to fill an entry:
// they store the same value).
cudaError_t split_clusters(int* ncl) {
  static std::atomic<int> cached[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  *ncl = dev < 64 ? cached[dev].load(std::memory_order_relaxed) : 0;
  if (*ncl > 0) return cudaSuccess;
  const int smem = BYTES;
  if ((e = cudaFuncSetAttribute(mla_tc_split_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) != cudaSuccess ||
      (e = cudaFuncSetAttribute(mla_tc_split_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) != cudaSuccess)
    return e;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = kSplitCL;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kSplitCL, 1, 1);
  cfg.blockDim = dim3(384, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  if ((e = cudaOccupancyMaxActiveClusters(ncl, mla_tc_split_kernel<1>, &cfg)) != cudaSuccess) return e;
  if (*ncl < 1) return cudaErrorInvalidConfiguration;
  if (dev < 64) cached[dev].store(*ncl, std::memory_order_relaxed);
  return cudaSuccess;
}

template <int PART>
cudaError_t launch_grid(const PagedMlaMaps& m, const PagedParams& p, bool dependent, cudaStream_t s) {
  auto kern = mla_tc_kernel<PART>;
  const int smem = BYTES;
  static_assert(BYTES >= kSmemOneCtaPerSm, "all 512 TMEM columns: one CTA per SM");
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(sms > 0 ? sms : 1, 1, 1);
  cfg.blockDim = dim3(384, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = dependent ? at : nullptr;
  cfg.numAttrs = dependent ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, m.q, m.qp, m.dy, m.k, m.kp, p);
}

}  // namespace

bool mla_tc_supported(const PagedParams& p) {
  return p.Dk == kLat && p.Dp == kPos && p.page_size == 16 && p.G >= 1 && p.G <= BC && BC % p.G == 0;
}

cudaError_t launch_paged_mla_tc_plan(const PagedParams& p, cudaStream_t s) {
  const int64_t n = static_cast<int64_t>(p.S) * ((p.max_pages + 7) / 8);
  if (n == 0 || p.num_pages == 0) return cudaSuccess;
  const int blocks = static_cast<int>((n + 3) / 4 < 2048 ? (n + 3) / 4 : 2048);  // a warp per block
  mla_tc_plan_kernel<<<blocks, 128, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_paged_mla_tc_split(const PagedMlaMaps& m, const PagedParams& p, cudaStream_t s) {
  if (p.num_pages == 0 || p.S == 0 || p.max_pages == 0) return cudaSuccess;
  // the clusters that fit are shared between the parts (part 1, the larger
  // accumulator, gets the odd one), and part 1 is the programmatic dependent
  // of part 0, so that both run at once and the grid kernels after them
  // start on the SMs the clusters leave free
  int ncl = 0;
  cudaError_t e = split_clusters(&ncl);
  if (e != cudaSuccess) return e;
  const int ncl0 = ncl > 1 ? ncl / 2 : 1, ncl1 = ncl > 1 ? ncl - ncl0 : 1;
  e = launch_split<0>(m, p, ncl0, false, s);
  if (e == cudaSuccess) e = launch_split<1>(m, p, ncl1, true, s);
  return e;
}

cudaError_t launch_paged_mla_tc(const PagedMlaMaps& m, const PagedParams& p, bool after_split, cudaStream_t s) {
  if (p.num_pages == 0 || p.S == 0 || p.max_pages == 0) return cudaSuccess;
  // part 0 overlaps the cluster-split kernel's tail (when that kernel runs
  // just before it), part 1 overlaps part 0's tail
  cudaError_t e = launch_grid<0>(m, p, after_split, s);
  if (e == cudaSuccess) e = launch_grid<1>(m, p, true, s);
  return e;
}

}  // namespace attn
