// Paged MLA history backward for the blocks whose shared pages carry many
// links (a long prefix shared by many sequences): the link passes of one such
// block are split over a cluster of 16 CTAs, on the warp-level tensor path
// (mma.sync bf16).  Every other block runs on the tcgen05 history kernel
// (paged_mla_tc.cu), which leaves the flagged blocks to this one.
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
// A plan kernel flags the 64-token blocks whose link passes exceed 128 tiles.
// A cluster CTA runs a contiguous share of such a block's tiles with the
// block's 64 x 576 fp32 accumulator in the registers of its 16 warps (the
// partial of one CTA does not need tensor memory, which keeps the 16 partials
// of a cluster side by side in shared memory for the rank-ordered sum).
// A column is one (query row, head of the group) pair; a tile is 32 columns
// (32 / G rows).  Per tile:
//   phase A  warp (token tile tt, column octet n8): S^T and dP^T (16 x 8) with
//            one k-loop over the 512 latent dims (K fragments shared by both)
//            plus the 64 position dims for S^T; P^T and dS^T in registers,
//            stored to shared memory as bf16
//   phase B  warp (token tile tt, dim quarter dr): dK_lat[., 128 dr ..+128)
//            += dS^T Q + P^T dY and dKp[., 16 dr ..+16) += dS^T Qp
// The K tile (latent + position, 9 chunks of 64 dims) stays in shared memory;
// Q, Qp and dY tiles arrive by TMA in 128-byte-swizzled 64-dim chunks,
// double-buffered.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>

#include "paged_common.cuh"
#include "paged_launch.h"
#include "sm103.cuh"

namespace attn {
using namespace sm103;

namespace {

constexpr int kLat = 512, kPos = 64;
constexpr float kLog2e = 1.4426950408889634f;
constexpr int BT = 64;                      // tokens per CTA (4 pages of 16)
constexpr int BC = 32;                      // columns per tile
constexpr int kThreads = 512;
constexpr int CH = BT * 128;                // K chunk: [64 tokens][64 dims]
constexpr int K_OFF = 0;                    // 8 latent chunks + 1 position chunk
constexpr int CQ = BC * 128;                // column chunk: [32 columns][64 dims]
constexpr int STAGE = 17 * CQ;              // Q (8 chunks), Qp (1), dY (8)
constexpr int ST_OFF = K_OFF + 9 * CH;      // 2 stages
constexpr int PS_STRIDE = BC * 2 + 16;      // P^T / dS^T rows: 32 bf16 + 16 bytes of padding
constexpr int PS = BT * PS_STRIDE;
constexpr int P_OFF = ST_OFF + 2 * STAGE;   // P^T then dS^T
constexpr int BYTES = P_OFF + 2 * PS;
static_assert(ST_OFF % 1024 == 0 && STAGE % 1024 == 0, "swizzled tiles need 1024-byte alignment");

struct MPageInfo {
  int phys[4];    // physical page (or -1)
  int off[4];     // first index of the page's link segment
  int cnt[4];     // links of the page
  int store[4];   // this CTA stores the page
};

// The passes of a CTA: its own sequence over all 64 tokens, then for link
// index li = 1, 2, ... the li-th links of the pages it stores; consecutive
// pages whose li-th links are consecutive logical pages of one sequence share
// one pass (their rows all live), so every page still sees its links in order.
struct MPass {
  const PagedParams* p;
  const MPageInfo* pi;
  int s0, tb;
  int j, jn, li, lmax;
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
  __device__ bool next_pass(int rt) {
    while (true) {
      if (j < 0) {
        j = 0;
        li = 1;
      } else {
        j = jn;
      }
      while (true) {
        while (j < 4 && !(pi->store[j] && li < pi->cnt[j])) ++j;
        if (j < 4) break;
        if (++li >= lmax) return false;
        j = 0;
      }
      const int link = p->links[pi->off[j] + li];
      const int s2 = link / p->max_pages, lp2 = link - s2 * p->max_pages;
      jn = j + 1;
      while (jn < 4 && pi->store[jn] && li < pi->cnt[jn] && lp2 + (jn - j) < p->max_pages &&
             p->links[pi->off[jn] + li] == link + (jn - j))
        ++jn;
      load(s2, lp2 * p->page_size - 16 * j, 16 * j, 16 * jn, rt);
      if (ntiles > 0) return true;
    }
  }
  __device__ bool begin(int rt) {
    j = -1;
    jn = 0;
    li = 0;
    lmax = 0;
    for (int k = 0; k < 4; ++k)
      if (pi->store[k] && pi->cnt[k] > lmax) lmax = pi->cnt[k];
    load(s0, tb * BT, 0, BT, rt);
    if (ntiles > 0) return true;
    return next_pass(rt);
  }
  __device__ bool advance(int rt) {
    if (++tile < ntiles) return true;
    return next_pass(rt);
  }
  // k tiles further on, a pass at a time
  __device__ bool skip(int k, int rt) {
    while (k > 0) {
      const int left = ntiles - 1 - tile;  // tiles after the current one in this pass
      if (k <= left) {
        tile += k;
        return true;
      }
      k -= left + 1;
      if (!next_pass(rt)) return false;  // tile 0 of the next pass that has tiles
    }
    return true;
  }
};

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}
__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t& r0, uint32_t& r1) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(addr) : "memory");
}
// D (16x8 fp32) += A (16x16 bf16, row) * B (16x8 bf16, col)
__device__ __forceinline__ void mma_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// address of the 16-byte piece `piece` (0..7) of row `row` in a 128-byte-swizzled chunk
__device__ __forceinline__ uint32_t swz(uint32_t base, int row, int piece) {
  return base + row * 128 + (((piece ^ row) & 7) << 4);
}

// Pages of block tb (4 pages) of sequence s0: physical page, link segment,
// and whether this block stores the page (it is the page's first link and,
// in compact history, the page is listed).
__device__ __forceinline__ void block_info(const PagedParams& p, int s0, int tb, MPageInfo* pi) {
  const int npg = pages_of(seq_len_of(p, s0), p.page_size);
  for (int j = 0; j < 4; ++j) {
    const int lp = tb * 4 + j;
    int ph = -1, off = 0, cnt = 0, st = 0;
    if (lp < npg) {
      ph = p.page_table[static_cast<int64_t>(s0) * p.max_pages + lp];
      if (ph >= 0 && ph < p.num_pages) {
        off = p.link_off[ph];
        cnt = p.link_off[ph + 1] - off;
        st = cnt > 0 && p.links[off] == s0 * p.max_pages + lp && (!p.listed || p.listed[ph]);
      } else {
        ph = -1;
      }
    }
    pi->phys[j] = ph;
    pi->off[j] = off;
    pi->cnt[j] = cnt;
    pi->store[j] = st;
  }
}

// Cluster primitives of the split kernel.
__device__ __forceinline__ int cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return static_cast<int>(r);
}
__device__ __forceinline__ int cluster_index() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return static_cast<int>(r);
}
__device__ __forceinline__ int cluster_count() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return static_cast<int>(r);
}
// All threads of all CTAs of the cluster: shared-memory writes before it are
// visible to the other CTAs' reads after it.
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
// bounded wait for copies still in flight (after an abort)
__device__ __forceinline__ void drain(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_test(bar, parity))
    if (global_timer_ns() - t0 > ATTN_WAIT_TIMEOUT_NS) return;
}

// A block whose link passes (shared pages) exceed this many tiles is left to
// the split kernel: its owner alone would serialise the other sequences' work.
constexpr int kHeavyLinkTiles = 128;
constexpr int kCL = 16;                      // CTAs of a split cluster; CTA r sums tokens [4r, 4r + 4)
constexpr int RED_STRIDE = kLat + kPos + 8;  // floats per token row of a partial (+8: bank spread)
static_assert(BT * RED_STRIDE * 4 <= BYTES, "a partial fits the tiles' shared memory");
static_assert(BT % kCL == 0, "tokens split evenly over the cluster");

// Plan of the MLA history: heavy[(s0 * nblk + tb) * KVH + g] = 1 when the
// pages block tb of sequence s0 stores carry more than kHeavyLinkTiles tiles of
// other links (counting stops there), else 0; one thread per block.
__global__ void mla_plan_kernel(const PagedParams p) {
  const int nblk = (p.max_pages + 3) / 4;
  const int n = p.S * nblk;
  const int RT = BC / p.G;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
    const int s0 = i / nblk, tb = i - s0 * nblk;
    int heavy = 0;
    if (tb * 4 < pages_of(seq_len_of(p, s0), p.page_size)) {
      MPageInfo pi;
      block_info(p, s0, tb, &pi);
      if (pi.store[0] | pi.store[1] | pi.store[2] | pi.store[3]) {
        MPass it{&p, &pi, s0, tb};
        int n_link = 0;
        if (it.begin(RT)) {
          do n_link += it.j >= 0 ? 1 : 0;
          while (n_link <= kHeavyLinkTiles && it.advance(RT));
        }
        heavy = n_link > kHeavyLinkTiles;
      }
    }
    for (int g = 0; g < p.KVH; ++g) p.heavy[static_cast<int64_t>(i) * p.KVH + g] = heavy;
  }
}

// Persistent clusters of kCL CTAs take the blocks the plan flagged (heavy
// block k to cluster k mod clusters); CTA r of a cluster runs the block's
// tiles [r n / kCL, (r + 1) n / kCL) of its n, the partial sums meet in
// shared memory and each CTA adds its BT / kCL tokens' partials over the
// cluster in rank order (a fixed order: the result does not depend on the
// number of clusters or on timing).  Every other block is done by the
// tcgen05 history kernel, which skips the flagged ones.
__global__ void __launch_bounds__(kThreads, 1)
    mla_split_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_qp,
                   const __grid_constant__ CUtensorMap tm_dy, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_kp, const PagedParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t bar_k, bar_full[2];
  __shared__ int abort_flag;
  __shared__ MPageInfo pinfo;
  __shared__ int n_tiles_sh, tile0_sh, any_store_sh, abort_any_sh;
  // (the copy iterator lives in shared memory: only thread 0 uses it, and in
  // registers it would be held by every thread)
  __shared__ MPass pf;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.G, RT = BC / G;
  const int nblk = (p.max_pages + 3) / 4;
  const int rank = cluster_rank();
  const int ncta = kCL;  // CTAs sharing one block's tiles
  const Abort ab{&abort_flag, p.err};
  const uint32_t sbase = smem_addr(sm);
  const int oob_slot = p.num_pages * p.page_size;  // out-of-range coordinate: TMA fills zeros
  const int tt = warp & 3;        // token tile (16 tokens, = page tt of the block)
  const int n8 = warp >> 2;       // phase A: column octet
  const int dr = warp >> 2;       // phase B: dim quarter
  const int g8 = lane >> 2, t4 = lane & 3;
  const float kInf = __int_as_float(0x7f800000);
  const uint32_t p_base = sbase + P_OFF, ds_base = sbase + P_OFF + PS;

  // the history kernel, launched next as this grid's programmatic dependent,
  // may start on the SMs these clusters leave free
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bar_k, 1);
    mbar_init(&bar_full[0], 1);
    mbar_init(&bar_full[1], 1);
    mbar_fence_init();
  }
  // thread 0's copy bookkeeping (running over the blocks of a persistent CTA)
  int issued[2] = {0, 0}, k_issued = 0;
  int tc = 0;       // tiles this CTA consumed: tile u uses stage u & 1, phase u >> 1
  int k_phase = 0;  // blocks this CTA loaded keys for

  auto run_block = [&](int tb, int s0, int gkv, int item) {
    __syncthreads();  // the previous block's readers of pinfo are done
    if (threadIdx.x == 0) {
      block_info(p, s0, tb, &pinfo);
      const int any = pinfo.store[0] | pinfo.store[1] | pinfo.store[2] | pinfo.store[3];
      MPass it{&p, &pinfo, s0, tb};
      int n_all = 0;
      if (any && it.begin(RT)) {
        do ++n_all;
        while (it.advance(RT));
      }
      any_store_sh = any;
      // this CTA's share of the block's tiles: [t0, t1), contiguous
      const int t0 = rank * n_all / ncta, t1 = (rank + 1) * n_all / ncta;
      tile0_sh = t0;
      n_tiles_sh = t1 - t0;
    }
    __syncthreads();
    // pages all stored by their owners elsewhere: nothing to do here (uniform
    // over the CTA, and over the cluster: same block)
    if (!any_store_sh) return;
    const int n = n_tiles_sh;
    const int tc0 = tc;

    bool pf_live = false;
    auto issue_tile = [&](int u) {
      const int stage = u & 1;
      const int r0 = pf.r_begin + pf.tile * RT;
      uint64_t* bar = &bar_full[stage];
      mbar_arrive_expect_tx(bar, STAGE);
      uint8_t* st = sm + ST_OFF + stage * STAGE;
      for (int c = 0; c < 8; ++c) {
        tma_load_3d(st + c * CQ, &tm_q, bar, c * 64, gkv * G, r0);
        tma_load_3d(st + (9 + c) * CQ, &tm_dy, bar, c * 64, gkv * G, r0);
      }
      tma_load_3d(st + 8 * CQ, &tm_qp, bar, 0, gkv * G, r0);
      ++issued[stage];
    };
    auto pf_next = [&]() -> bool { return pf.advance(RT); };
    if (threadIdx.x == 0 && n > 0 && !abort_flag) {
      tma_prefetch_map(&tm_q);
      tma_prefetch_map(&tm_qp);
      tma_prefetch_map(&tm_dy);
      tma_prefetch_map(&tm_k);
      tma_prefetch_map(&tm_kp);
      mbar_arrive_expect_tx(&bar_k, 9 * CH);
      ++k_issued;
      for (int j = 0; j < 4; ++j) {
        const int slot = pinfo.phys[j] >= 0 ? pinfo.phys[j] * p.page_size : oob_slot;
        for (int c = 0; c < 8; ++c) tma_load_3d(sm + K_OFF + c * CH + j * 16 * 128, &tm_k, &bar_k, c * 64, gkv, slot);
        tma_load_3d(sm + K_OFF + 8 * CH + j * 16 * 128, &tm_kp, &bar_k, 0, gkv, slot);
      }
      pf.p = &p;
      pf.pi = &pinfo;
      pf.s0 = s0;
      pf.tb = tb;
      pf_live = pf.begin(RT);
      if (pf_live) pf_live = pf.skip(tile0_sh, RT);
      for (int t = 0; t < 2 && t < n && pf_live; ++t) {
        issue_tile(tc0 + t);
        pf_live = pf_next();
      }
    }

    float acc[16][4], accp[2][4];
#pragma unroll
    for (int i = 0; i < 16; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
#pragma unroll
    for (int i = 0; i < 2; ++i) accp[i][0] = accp[i][1] = accp[i][2] = accp[i][3] = 0.f;

    MPass it{&p, &pinfo, s0, tb};
    bool live = n > 0 && it.begin(RT);
    if (live) live = it.skip(tile0_sh, RT);
    bool ok = true;
    if (n > 0) {
      ok = mbar_wait_warp(&bar_k, k_phase & 1, ab);
      ++k_phase;
    }
    for (int t = 0; t < n; ++t) {
      const int u = tc0 + t, stage = u & 1;  // running tile number of this CTA
      const uint32_t stb = sbase + ST_OFF + stage * STAGE;
      // column data of this thread's two phase-A columns
      const int r0 = it.r_begin + it.tile * RT;
      float lse_c[2], dl_c[2];
      int pos_c[2];
      bool col_ok[2];
  #pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int c = n8 * 8 + 2 * t4 + e;
        const int r = r0 + c / G, hh = gkv * G + c % G;
        col_ok[e] = r < it.r_end;
        const size_t si = static_cast<size_t>(col_ok[e] ? r : 0) * p.H + hh;
        lse_c[e] = col_ok[e] ? p.lse[si] * kLog2e : kInf;
        dl_c[e] = col_ok[e] ? p.delta[si] : 0.f;
        pos_c[e] = col_ok[e] ? (p.causal ? p.q_pos[r] : 0x7fffffff) : -1;
      }
      if (ok) ok = mbar_wait_warp(&bar_full[stage], (u >> 1) & 1, ab);
      if (ok) {
        // ---------------------------------------------------------------- phase A
        float sacc[4] = {0.f, 0.f, 0.f, 0.f}, dpacc[4] = {0.f, 0.f, 0.f, 0.f};
        const int arow = tt * 16 + (lane & 7) + 8 * ((lane >> 3) & 1);
        const int ahalf = lane >> 4;
        const int brow = n8 * 8 + (lane & 7);
        const int bm = lane >> 3;  // matrix of the x4 B load: 0,1 Q (k halves), 2,3 dY
  #pragma unroll 2
        for (int kc = 0; kc < 8; ++kc) {
  #pragma unroll
          for (int kp = 0; kp < 4; ++kp) {
            uint32_t a[4], bq[4];
            ldsm_x4(swz(sbase + K_OFF + kc * CH, arow, 2 * kp + ahalf), a);
            const uint32_t bchunk = stb + ((bm >> 1) ? (9 + kc) : kc) * CQ;
            ldsm_x4(swz(bchunk, brow, 2 * kp + (bm & 1)), bq);
            mma_16816(sacc, a, bq[0], bq[1]);
            mma_16816(dpacc, a, bq[2], bq[3]);
          }
        }
  #pragma unroll
        for (int kp = 0; kp < 4; ++kp) {
          uint32_t a[4], b0, b1;
          ldsm_x4(swz(sbase + K_OFF + 8 * CH, arow, 2 * kp + ahalf), a);
          ldsm_x2(swz(stb + 8 * CQ, brow, 2 * kp + (bm & 1)), b0, b1);
          mma_16816(sacc, a, b0, b1);
        }
        // P^T and dS^T of this warp's 16 tokens x 8 columns
  #pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
          const int i = tt * 16 + g8 + 8 * hr;  // block-local token
          const int tok = it.tbase + i;
          const bool tok_ok = i >= it.ra && i < it.rb && tok < seq_len_of(p, it.seq);
          float pv[2], dsv[2];
  #pragma unroll
          for (int e = 0; e < 2; ++e) {
            const bool vis = tok_ok && col_ok[e] && tok <= pos_c[e] && lse_c[e] > -kInf;
            const float pe = ex2_approx(fmaf(sacc[2 * hr + e], p.scale_log2, -lse_c[e]));
            // select, not multiply: dP of a tail or unowned slot may be NaN
            pv[e] = vis ? pe : 0.f;
            dsv[e] = vis ? pe * (dpacc[2 * hr + e] - dl_c[e]) * p.scale : 0.f;
          }
          const int c = n8 * 8 + 2 * t4;
          *reinterpret_cast<uint32_t*>(sm + P_OFF + i * PS_STRIDE + c * 2) = pack_bf16x2(pv[0], pv[1]);
          *reinterpret_cast<uint32_t*>(sm + P_OFF + PS + i * PS_STRIDE + c * 2) = pack_bf16x2(dsv[0], dsv[1]);
        }
      }
      __syncthreads();
      if (ok && !abort_flag) {
        // ---------------------------------------------------------------- phase B
        const int arow = tt * 16 + (lane & 7) + 8 * ((lane >> 3) & 1);
        const int bm = lane >> 3;
  #pragma unroll
        for (int ks = 0; ks < 2; ++ks) {
          uint32_t ads[4], ap[4];
          const uint32_t aoff = arow * PS_STRIDE + (ks * 16 + 8 * (lane >> 4)) * 2;
          ldsm_x4(ds_base + aoff, ads);
          ldsm_x4(p_base + aoff, ap);
          const int krow = ks * 16 + (lane & 7) + 8 * (bm & 1);  // column index = B row
  #pragma unroll
          for (int np = 0; np < 8; ++np) {  // pairs of 8-dim tiles: dims 128 dr + 16 np
            const int chunk = 2 * dr + (np >> 2);
            const int piece = 2 * (np & 3) + (bm >> 1);
            uint32_t bq[4], bd[4];
            ldsm_x4_t(swz(stb + chunk * CQ, krow, piece), bq);
            ldsm_x4_t(swz(stb + (9 + chunk) * CQ, krow, piece), bd);
            mma_16816(acc[2 * np], ads, bq[0], bq[1]);
            mma_16816(acc[2 * np + 1], ads, bq[2], bq[3]);
            mma_16816(acc[2 * np], ap, bd[0], bd[1]);
            mma_16816(acc[2 * np + 1], ap, bd[2], bd[3]);
          }
          uint32_t bqp[4];
          ldsm_x4_t(swz(stb + 8 * CQ, krow, 2 * dr + (bm >> 1)), bqp);
          mma_16816(accp[0], ads, bqp[0], bqp[1]);
          mma_16816(accp[1], ads, bqp[2], bqp[3]);
        }
      }
      __syncthreads();  // stage and P^T/dS^T buffers free
      // (the copy iterator runs on past this CTA's share of the tiles: stop at n)
      if (threadIdx.x == 0 && pf_live && t + 2 < n && !abort_flag) {
        issue_tile(u + 2);  // owned tile t + 2, into the stage just freed
        pf_live = pf_next();
      }
      if (live) live = it.advance(RT);
    }
    (void)live;
    tc = tc0 + n;
    // this CTA's partial sums to shared memory as [64 tokens][576 dims]
    // (the tiles' buffers are free: the loop ended on a barrier after the last
    // copy was consumed)
    float* red = reinterpret_cast<float*>(sm);
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      float* row = red + (tt * 16 + g8 + 8 * hr) * RED_STRIDE;
#pragma unroll
      for (int nt = 0; nt < 16; ++nt)
        *reinterpret_cast<float2*>(row + 128 * dr + 8 * nt + 2 * t4) = make_float2(acc[nt][2 * hr], acc[nt][2 * hr + 1]);
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
        *reinterpret_cast<float2*>(row + kLat + 16 * dr + 8 * nt + 2 * t4) =
            make_float2(accp[nt][2 * hr], accp[nt][2 * hr + 1]);
    }
    // every CTA's abort flag is ORed over the cluster: a partial left
    // incomplete by a timed-out wait must not reach the pool as a finite value
    if (threadIdx.x == 0) abort_any_sh = abort_flag;
    cluster_sync();
    if (threadIdx.x == 0) {
      int any_abort = 0;
      for (int r = 0; r < kCL; ++r) any_abort |= ld_cluster_s32(map_rank(smem_addr(&abort_any_sh), r));
      if (any_abort) *ab.flag = 1;
    }
    __syncthreads();
    // tokens [4 rank, 4 rank + 4): the partials of CTAs 0..kCL-1 added in that order
    constexpr int kQuads = (kLat + kPos) / 4;
    const bool good = !abort_flag;
    for (int idx = threadIdx.x; idx < (BT / kCL) * kQuads; idx += kThreads) {
      const int i = (BT / kCL) * rank + idx / kQuads, d = 4 * (idx % kQuads);
      const uint32_t a = smem_addr(red + i * RED_STRIDE + d);
      float4 sum = ld_cluster_f4(map_rank(a, 0));
#pragma unroll
      for (int r = 1; r < kCL; ++r) {
        const float4 v = ld_cluster_f4(map_rank(a, r));
        sum.x += v.x;
        sum.y += v.y;
        sum.z += v.z;
        sum.w += v.w;
      }
      const int j = i >> 4;
      if (good && pinfo.store[j]) {
        const int64_t prow = (static_cast<int64_t>(pinfo.phys[j]) * p.page_size + (i & 15)) * p.KVH + gkv;
        const uint2 w = make_uint2(pack_bf16x2(sum.x, sum.y), pack_bf16x2(sum.z, sum.w));
        if (d < kLat) {
          if (p.wrt & 2u) *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(p.dk_pool) + prow * kLat + d) = w;
        } else if (p.wrt & 8u) {
          *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(p.dkp_pool) + prow * kPos + (d - kLat)) = w;
        }
      }
    }
    cluster_sync();  // the other CTAs have read this CTA's partial
  };

  // the flagged blocks in flag order, heavy block k to cluster k mod clusters
  __shared__ int items_sh[kThreads];
  __shared__ int warp_cnt[kThreads / 32];
  const int cid = cluster_index(), ncl = cluster_count();
  const int nitems = p.S * nblk * p.KVH;
  int base = 0;
  for (int c0 = 0; c0 < nitems; c0 += kThreads) {
    const int i = c0 + threadIdx.x;
    const bool f = i < nitems && p.heavy[i] != 0;
    const uint32_t bal = __ballot_sync(0xffffffffu, f);
    if (lane == 0) warp_cnt[warp] = __popc(bal);
    __syncthreads();
    int before = 0, total = 0;
    for (int w = 0; w < kThreads / 32; ++w) {
      const int c = warp_cnt[w];
      before += w < warp ? c : 0;
      total += c;
    }
    const int k = base + before + __popc(bal & ((1u << lane) - 1u));
    // this cluster's heavy indices in [base, base + total): cid + ncl * m, m in [m0, m1)
    const int m0 = base > cid ? (base - cid + ncl - 1) / ncl : 0;
    const int m1 = base + total > cid ? (base + total - cid + ncl - 1) / ncl : 0;
    if (f && k % ncl == cid) items_sh[k / ncl - m0] = i;
    __syncthreads();
    for (int m = 0; m < m1 - m0; ++m) {
      const int item = items_sh[m];
      const int gkv = item % p.KVH, rest = item / p.KVH;
      run_block(rest % nblk, rest / nblk, gkv, item);
    }
    base += total;
    __syncthreads();  // items_sh and warp_cnt are rewritten next
  }
  // copies still in flight after an abort land before the CTA exits
  if (threadIdx.x == 0) {
    for (int st = 0; st < 2; ++st)
      if (issued[st] > 0) drain(&bar_full[st], static_cast<uint32_t>((issued[st] - 1) & 1));
    if (k_issued > 0) drain(&bar_k, static_cast<uint32_t>((k_issued - 1) & 1));
  }
}

}  // namespace

bool mla_split_supported(const PagedParams& p) {
  return p.Dk == kLat && p.Dp == kPos && p.page_size == 16 && (p.G == 4 || p.G == 8 || p.G == 16 || p.G == 32);
}

cudaError_t launch_paged_mla_plan(const PagedParams& p, cudaStream_t s) {
  const int64_t n = static_cast<int64_t>(p.S) * ((p.max_pages + 3) / 4);
  if (n == 0 || p.num_pages == 0) return cudaSuccess;
  const int blocks = static_cast<int>((n + 127) / 128 < 1024 ? (n + 127) / 128 : 1024);
  mla_plan_kernel<<<blocks, 128, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_paged_mla_split(const PagedMlaMaps& m, const PagedParams& p, cudaStream_t s) {
  if (p.num_pages == 0 || p.S == 0 || p.max_pages == 0) return cudaSuccess;
  const int smem = BYTES + 1024;
  auto kern = mla_split_kernel;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  // 16 CTAs per cluster is above the portable 8
  if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1)) != cudaSuccess) return e;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = kCL;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  // as many clusters as fit the GPU at once (one CTA per SM), cached per
  // device (host threads may race to fill an entry: they store the same value)
  static std::atomic<int> clusters[64];
  int dev = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  int ncl = dev < 64 ? clusters[dev].load(std::memory_order_relaxed) : 0;
  if (ncl == 0) {
    cfg.gridDim = dim3(kCL, 1, 1);
    if ((e = cudaOccupancyMaxActiveClusters(&ncl, kern, &cfg)) != cudaSuccess) return e;
    if (ncl < 1) return cudaErrorInvalidConfiguration;
    if (dev < 64) clusters[dev].store(ncl, std::memory_order_relaxed);
  }
  cfg.gridDim = dim3(ncl * kCL, 1, 1);
  return cudaLaunchKernelEx(&cfg, kern, m.q, m.qp, m.dy, m.k, m.kp, p);
}

}  // namespace attn
