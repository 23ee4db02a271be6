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
//   S^T  = K_lat Q^T + K_pos Qp^T     [128 x 64], 9 chunks of 64 dims
//   dP^T = K_lat dY^T                 [128 x 64], 8 chunks
//   P^T  = exp2(S^T scale log2e - lse log2e),  dS^T = P^T (dP^T - delta) scale
//   acc  += P^T dY[:, part] + dS^T Q[:, part]   (A operands from tensor memory)
// The accumulator of 128 tokens x 576 dims does not fit the 512 tensor-memory
// columns next to the score tiles, so the dims are split over two CTAs
// (PART 0: latent dims [0, 256); PART 1: latent dims [256, 512) and the 64
// position dims); each forms the full S^T and dP^T of its tiles.
//
// Shared memory: the K tile stays resident (latent + position, 9 chunks of
// [128 tokens x 64 dims], 144 KiB); Q, Qp and dY arrive as a stream of 8 KiB
// chunks ([64 columns x 64 dims]) through a 4-stage TMA ring of two chunk
// slots each (one wait and one release per pair of chunks), in the order
//   S chunks of tile t, the part's accumulation chunks of tile t - 1, dP
//   chunks of tile t
// so the tensor core forms the scores of tile t while the compute warps turn
// tile t - 1 into P and dS.  The score tile is double-buffered in tensor
// memory, the dP tile single-buffered: dP(t) overwrites dS(t - 1) after the
// accumulation of tile t - 1 has read it.  Roles (384 threads): warp 0 TMA producer (also
// writes each tile's column statistics), warp 1 MMA issuer (whole warp,
// elect.sync), warps 4..7 / 8..11 compute groups for even / odd tiles (one
// TMEM lane per token).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

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
constexpr int kStages = 4;               // ring of stages of two chunk slots
constexpr int kStatSlots = 4;
constexpr int KCH = BT * 128;            // K chunk [128 tokens][64 dims], 16 KiB
constexpr int QCH = BC * 128;            // Q / dY chunk [64 columns][64 dims], 8 KiB
constexpr int K_OFF = 0;                 // 8 latent chunks + 1 position chunk
constexpr int RING_OFF = K_OFF + 9 * KCH;
constexpr int STAGE = 2 * QCH;
constexpr int ST_OFF = RING_OFF + kStages * STAGE;
constexpr int ST_SLOT = 3 * BC * 4 + 16;  // -L2, delta, pos per column + pass info
constexpr int BYTES = ST_OFF + kStatSlots * ST_SLOT;
static_assert(RING_OFF % 1024 == 0 && QCH % 1024 == 0, "swizzled tiles need 1024-byte alignment");
// TMEM: accumulator [0, 320) (PART 0 uses [0, 256)), S^T[2] and dP^T 64 columns each
constexpr int T_ACC = 0, T_S = 320, T_DP = 448, TMEM_COLS = 512;

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

template <int PART>
__global__ void __launch_bounds__(384, 1)
    mla_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_qp,
                  const __grid_constant__ CUtensorMap tm_dy, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_kp, const PagedParams p) {
  using PS = PartShape<PART>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t bar_k, bar_full[kStages], bar_empty[kStages], bar_st_full[kStatSlots],
      bar_st_empty[kStatSlots], bar_s_full[2], bar_p_full[2], bar_dp_full, bar_ds_full, bar_acc;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag;
  __shared__ PageInfo pinfo;
  __shared__ int n_tiles_sh, any_store_sh;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = blockIdx.x, tb = blockIdx.y, s0 = blockIdx.z;
  // Launched as the programmatic dependent of the kernel before it (the
  // cluster-split kernel, or PART 0 for PART 1), whose results it does not
  // read: its own dependent may start at once, and the last CTA waits for the
  // kernel before, so that this grid completes after it and later work in
  // the stream sees both.  Without a programmatic launch both are no-ops.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (blockIdx.x == gridDim.x - 1 && blockIdx.y == gridDim.y - 1 && blockIdx.z == gridDim.z - 1)
    asm volatile("griddepcontrol.wait;" ::: "memory");
  const int len0 = seq_len_of(p, s0);
  const int npg = pages_of(len0, p.page_size);
  if (tb * 8 >= npg) return;  // no token of this sequence in the block (uniform exit)
  const int RT = BC / p.G;    // query rows per tile
  const Abort ab{&abort_flag, p.err};

  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bar_k, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bar_full[s], 1);
      mbar_init(&bar_empty[s], 1);
    }
    for (int s = 0; s < kStatSlots; ++s) {
      mbar_init(&bar_st_full[s], 1);
      mbar_init(&bar_st_empty[s], 4);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bar_s_full[s], 1);
      mbar_init(&bar_p_full[s], 4);
    }
    mbar_init(&bar_dp_full, 1);
    mbar_init(&bar_ds_full, 4);
    mbar_init(&bar_acc, 1);
    mbar_fence_init();
    int any = fill_page_info(p, s0, tb, npg, &pinfo);
    // a block with a heavy 64-token half belongs to the cluster-split kernel
    if (any && p.heavy) {
      const int nb64 = (p.max_pages + 3) / 4;
      const int64_t h0 = (static_cast<int64_t>(s0) * nb64 + 2 * tb) * p.KVH + g;
      if (p.heavy[h0] || (2 * tb + 1 < nb64 && p.heavy[h0 + p.KVH])) any = 0;
    }
    any_store_sh = any;
    PassIter it{&p, &pinfo, s0, tb};
    int n = 0;
    if (any && it.begin(RT)) {
      do ++n;
      while (it.advance(RT));
    }
    n_tiles_sh = n;
  }
  __syncthreads();
  // a block whose pages are all stored by other CTAs (their owners) has
  // nothing to write: leave before taking tensor memory (uniform exit)
  if (!any_store_sh) return;
  if (warp == 1) {
    tmem_alloc(&tmem_base_sh, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  const int n = n_tiles_sh;
  const int oob_slot = p.num_pages * p.page_size;  // out-of-range coordinate: TMA fills zeros

  if (n > 0 && warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_map(&tm_q);
      tma_prefetch_map(&tm_qp);
      tma_prefetch_map(&tm_dy);
      tma_prefetch_map(&tm_k);
      tma_prefetch_map(&tm_kp);
      mbar_arrive_expect_tx(&bar_k, 9 * KCH);
      for (int j = 0; j < 8; ++j) {
        const int slot = pinfo.phys[j] >= 0 ? pinfo.phys[j] * p.page_size : oob_slot;
        for (int c = 0; c < 8; ++c)
          tma_load_3d(sm + K_OFF + c * KCH + j * 16 * 128, &tm_k, &bar_k, c * 64, g, slot);
        tma_load_3d(sm + K_OFF + 8 * KCH + j * 16 * 128, &tm_kp, &bar_k, 0, g, slot);
      }
    }
    PassIter it{&p, &pinfo, s0, tb};
    it.begin(RT);
    bool ok = true;
    int q = 0;          // job counter of the ring (a job: one or two chunks)
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
    // one job into the ring: chunks c and c + 1 (nch = 2) or c alone of Q
    // (src 0; chunk 8 is Qp) or dY (src 2)
    auto load_job = [&](int src, int c, int nch, int row0) -> bool {
      const int s = q % kStages;
      if (q >= kStages && !mbar_wait(&bar_empty[s], ((q / kStages) - 1) & 1, ab)) return false;
      if (lane == 0) {
        mbar_arrive_expect_tx(&bar_full[s], nch * QCH);
        for (int k = 0; k < nch; ++k) {
          const int cc = c + k;
          const CUtensorMap* m = src == 2 ? &tm_dy : cc == 8 ? &tm_qp : &tm_q;
          tma_load_3d(sm + RING_OFF + s * STAGE + k * QCH, m, &bar_full[s], cc == 8 ? 0 : cc * 64, g * p.G, row0);
        }
      }
      last_use[s] = q;
      ++q;
      return true;
    };
    // the accumulation jobs of a tile: dY chunks of the part in pairs, then
    // its Q chunks in pairs (and Qp alone, PART 1)
    auto load_acc = [&](int row0) -> bool {
      for (int a = 0; a < PS::NACC; a += 2)
        if (!load_job(a < 4 ? 2 : 0, acc_src_chunk<PART>(a), PS::NACC - a >= 2 ? 2 : 1, row0)) return false;
      return true;
    };
    for (int t = 0; t <= n && ok; ++t) {
      if (t < n) {
        const int row0 = it.r_begin + it.tile * RT;
        // column statistics of tile t: -L2, delta, pos per column (a row
        // with lse = -inf sees no token), plus the pass's token mapping
        const int ss = t % kStatSlots;
        if (t >= kStatSlots && !(ok = mbar_wait(&bar_st_empty[ss], ((t / kStatSlots) - 1) & 1, ab))) break;
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
        if (lane == 0) mbar_arrive(&bar_st_full[ss]);
        PassIter nx = it;
        if (t + 1 < n) {
          nx.advance(RT);
          fetch(nx);
        }
        // S chunks of tile t (Q latent 0..7, Qp), the accumulation chunks of
        // tile t - 1, then the dP chunks of tile t (dY 0..7)
        for (int c = 0; c < 9 && ok; c += 2) ok = load_job(0, c, c < 8 ? 2 : 1, row0);
        if (t >= 1 && ok) ok = load_acc(prev_row0);
        for (int c = 0; c < 8 && ok; c += 2) ok = load_job(2, c, 2, row0);
        if (!ok) break;
        prev_row0 = row0;
        it = nx;
      } else {
        ok = load_acc(prev_row0);
      }
    }
    if (lane == 0) {
      for (int s = 0; s < kStages; ++s)
        if (last_use[s] >= 0) drain_wait(&bar_full[s], (last_use[s] / kStages) & 1);
      drain_wait(&bar_k, 0);
    }
  } else if (n > 0 && warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // the whole warp runs this role (warp-uniform); elected lanes issue
    constexpr uint32_t id_s = idesc_bf16(128, BC, false, false);   // S^T, dP^T: K-major A and B
    constexpr uint32_t id_acc = idesc_bf16(128, 64, false, true);  // acc: A from TMEM, B MN-major
    const uint64_t dK0 = sdesc_sw128(smem_addr(sm + K_OFF), 16, 1024);
    const uint64_t dR0 = sdesc_sw128(smem_addr(sm + RING_OFF), 16, 1024);            // K-major
    const uint64_t dRm0 = sdesc_sw128(smem_addr(sm + RING_OFF), BC * 128, 1024);     // MN-major
    bool ok = mbar_wait_warp(&bar_k, 0, ab);
    int q = 0;
    // a stage's copies are usually in by the time this warp reaches it: a
    // non-blocking test first, the bounded wait only when it is not
    auto wait_stage = [&](int qq) -> bool {
      const int s = qq % kStages;
      if (mbar_test_warp(&bar_full[s], (qq / kStages) & 1)) return true;
      return mbar_wait_warp(&bar_full[s], (qq / kStages) & 1, ab);
    };
    // after the job of ring index qq: its stage goes back to the producer
    // once its products are done
    auto release = [&](int qq) { mma_commit_w(&bar_empty[qq % kStages]); };
    // S^T(t) (kind 0, 9 chunks) or dP^T(t) (kind 1, 8 chunks) into tensor
    // memory, two chunks per job
    auto xt_jobs = [&](int t, int kind) -> bool {
      const int nc = kind == 0 ? 9 : 8;
      const uint32_t d = tmem + (kind == 0 ? T_S + (t & 1) * BC : T_DP);
      for (int c0 = 0; c0 < nc; c0 += 2, ++q) {
        if (!wait_stage(q)) return false;
        tc_fence_after();
        for (int k = 0; k < 2 && c0 + k < nc; ++k) {
          const int c = c0 + k;
          const uint64_t a = sdesc_add(dK0, c * KCH), bq = sdesc_add(dR0, (q % kStages) * STAGE + k * QCH);
          if (c == 0)
            mma_ss_w<false>(d, a, bq, id_s);
          else
            mma_ss_w<true>(d, a, bq, id_s);
#pragma unroll
          for (int kk = 1; kk < 4; ++kk) mma_ss_w<true>(d, sdesc_add(a, kk * 32), sdesc_add(bq, kk * 32), id_s);
        }
        release(q);
      }
      mma_commit_w(kind == 0 ? &bar_s_full[t & 1] : &bar_dp_full);
      return true;
    };
    for (int t = 0; t <= n && ok; ++t) {
      // S^T(t): its buffer's previous tile (t - 2) was accumulated earlier in
      // this stream
      if (t < n && !(ok = xt_jobs(t, 0))) break;
      if (t >= 1) {
        // accumulation of tile u = t - 1: P^T dY chunks once P^T(u) is in,
        // then dS^T Q chunks once dS^T(u) is in
        const int u = t - 1;
        if (!(ok = mbar_wait_warp(&bar_p_full[u & 1], (u >> 1) & 1, ab))) break;
        tc_fence_after();
        for (int a0 = 0; a0 < PS::NACC && ok; a0 += 2, ++q) {
          if (a0 == 4) {
            if (!(ok = mbar_wait_warp(&bar_ds_full, u & 1, ab))) break;
            tc_fence_after();
          }
          if (!(ok = wait_stage(q))) break;
          tc_fence_after();
          for (int k = 0; k < 2 && a0 + k < PS::NACC; ++k) {
            const int a = a0 + k;
            const int c = acc_src_chunk<PART>(a);
            const uint32_t d = tmem + T_ACC + (c - 4 * PART) * 64;  // chunk 8 (position) -> 256
            const uint32_t at = tmem + (a < 4 ? T_S + (u & 1) * BC : T_DP);
            const uint64_t bm = sdesc_add(dRm0, (q % kStages) * STAGE + k * QCH);
            // the first contribution to an accumulator chunk overwrites it:
            // P^T dY for latent chunks, dS^T Qp for the position chunk
            if (u == 0 && (a < 4 || c == 8))
              mma_ts_w<false>(d, at, bm, id_acc);
            else
              mma_ts_w<true>(d, at, bm, id_acc);
#pragma unroll
            for (int kk = 1; kk < BC / 16; ++kk)
              mma_ts_w<true>(d, at + kk * 8, sdesc_add(bm, kk * 16 * 128), id_acc);
          }
          release(q);
        }
        if (!ok) break;
      }
      // dP^T(t) overwrites dS^T(t - 1), whose products were just issued
      if (t < n && !(ok = xt_jobs(t, 1))) break;
    }
    mma_commit_w(&bar_acc);
    drain_wait(&bar_acc, 0);
    __syncwarp();
  } else if (warp >= 4) {
    const int sg = (warp - 4) >> 2;  // compute group: tiles of parity sg
    const int lg = warp & 3;
    const int row = lg * 32 + lane;  // token row inside the block == TMEM lane
    const uint32_t lane_addr = static_cast<uint32_t>(lg * 32) << 16;
    bool ok = n > 0;
    for (int t = sg; t < n && ok; t += 2) {
      const int bb = t & 1, ss = t % kStatSlots;
      if (!(ok = mbar_wait_warp(&bar_st_full[ss], (t / kStatSlots) & 1, ab))) break;
      const uint8_t* st = sm + ST_OFF + ss * ST_SLOT;
      const float* snl = reinterpret_cast<const float*>(st);
      const float* sdl = snl + BC;
      const int* spos = reinterpret_cast<const int*>(sdl + BC);
      const int* sinfo = spos + BC;
      const int tok = sinfo[0] + row;
      const bool tok_ok = row >= sinfo[1] && row < sinfo[2] && tok >= 0 && tok < sinfo[3];
      if (!(ok = mbar_wait_warp(&bar_s_full[bb], (t >> 1) & 1, ab))) break;
      tc_fence_after();
      // ---------------------------------------------------- S^T -> P^T
      // two halves of 32 columns: half hf reads S^T columns [32hf, 32hf+32)
      // and writes P^T (bf16 pairs) to columns [16hf, 16hf+16), which half 0
      // has already read
      const uint32_t tS = tmem + T_S + bb * BC + lane_addr;
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
          const float4 nl = *reinterpret_cast<const float4*>(snl + c0);
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
      // (one dP buffer: its phase t has completed once this group sees it,
      // since dP(t - 1) went into the tensor core before S(t) did)
      if (!(ok = mbar_wait_warp(&bar_dp_full, t & 1, ab))) break;
      tc_fence_after();
      const uint32_t tDP = tmem + T_DP + lane_addr;
      // a masked entry has P = 0 and takes dS = 0 by select: dP of a tail or
      // unowned slot may be NaN
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        uint32_t dr[32], dsw[16];
        tmem_ld32(tDP + 32 * hf, dr);
        tmem_ld_wait();
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4) {
          const float4 d4 = *reinterpret_cast<const float4*>(sdl + 32 * hf + 4 * c4);
          const float dv[4] = {d4.x, d4.y, d4.z, d4.w};
          float ds[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const uint32_t w = pw[16 * hf + 2 * c4 + (e >> 1)];
            const float pe = __uint_as_float((e & 1) ? (w & 0xffff0000u) : (w << 16));
            ds[e] = pe != 0.f ? pe * (__uint_as_float(dr[4 * c4 + e]) - dv[e]) * p.scale : 0.f;
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
        mbar_arrive(&bar_ds_full);
        mbar_arrive(&bar_st_empty[ss]);
      }
    }
    if (n > 0) {
      if (ok) ok = mbar_wait_warp(&bar_acc, 0, ab);
      tc_fence_after();
    }
    // ------------------------------------------------------------ epilogue
    // 32-column chunks of the accumulator, alternating between the groups:
    // latent dims [256 PART + 32 cc, ...) for cc < 8, position dims after
    // that (PART 1); rows of tokens no pass saw are zero
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
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

template <int PART>
cudaError_t launch_part(const PagedMlaMaps& m, const PagedParams& p, bool dependent, cudaStream_t s) {
  auto kern = mla_tc_kernel<PART>;
  const int smem = BYTES + 1024;
  static_assert(BYTES + 1024 >= kSmemOneCtaPerSm, "all 512 TMEM columns: one CTA per SM");
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int nblk = (p.max_pages * p.page_size + BT - 1) / BT;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.KVH, nblk, p.S);
  cfg.blockDim = dim3(384, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = dependent ? at : nullptr;
  cfg.numAttrs = dependent ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, m.q, m.qp, m.dy, m.k, m.kp, p);
}

// heavy[] is planned per 64-token block; a 128-token block of this kernel
// goes to the split kernel when either half is heavy, so both halves are
// flagged for it
__global__ void mla_tc_pair_heavy_kernel(const PagedParams p) {
  const int nb64 = (p.max_pages + 3) / 4;
  const int nb128 = (nb64 + 1) / 2;
  const int n = p.S * nb128 * p.KVH;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
    const int g = i % p.KVH, sb = i / p.KVH, s0 = sb / nb128, b = sb - s0 * nb128;
    const int64_t h0 = (static_cast<int64_t>(s0) * nb64 + 2 * b) * p.KVH + g;
    const bool second = 2 * b + 1 < nb64;
    const int h = p.heavy[h0] | (second ? p.heavy[h0 + p.KVH] : 0);
    p.heavy[h0] = h;
    if (second) p.heavy[h0 + p.KVH] = h;
  }
}

}  // namespace

bool mla_tc_supported(const PagedParams& p) {
  return p.Dk == kLat && p.Dp == kPos && p.page_size == 16 && p.G >= 1 && p.G <= BC && BC % p.G == 0;
}

cudaError_t launch_paged_mla_tc_pair_heavy(const PagedParams& p, cudaStream_t s) {
  if (p.S == 0 || p.max_pages == 0 || p.KVH == 0) return cudaSuccess;
  mla_tc_pair_heavy_kernel<<<64, 256, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_paged_mla_tc(const PagedMlaMaps& m, const PagedParams& p, bool after_split, cudaStream_t s) {
  if (p.num_pages == 0 || p.S == 0 || p.max_pages == 0) return cudaSuccess;
  // PART 0 overlaps the cluster-split kernel's tail (when that kernel runs
  // just before it), PART 1 overlaps PART 0's tail
  cudaError_t e = launch_part<0>(m, p, after_split, s);
  if (e == cudaSuccess) e = launch_part<1>(m, p, true, s);
  return e;
}

}  // namespace attn
