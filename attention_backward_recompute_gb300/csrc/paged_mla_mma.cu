// Paged MLA history backward on the warp-level tensor path (mma.sync bf16).
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
// Why mma.sync and not tcgen05: the accumulator of one 64-token block is
// 64 x 576 fp32 (144 KiB); with the score and dP tiles it does not fit the
// 512 tensor-memory columns, while 16 warps hold it in registers (72 per
// thread).  The warp-level tensor path runs at about a quarter of tcgen05's
// rate on this GPU, which is still far above CUDA-core FMA.
//
// One CTA owns 64 tokens (four 16-token pages) of one sequence and one KV head
// and walks the same passes as the GQA kernel: its own sequence, then the
// other links of the pages it stores, in link order, consecutive pages of a
// shared prefix in one pass.
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

// SPLIT = false: one CTA per (64-token block, sequence, KV head); a block it
// stores is finished here unless the plan flagged its link passes as heavy.
// SPLIT = true: persistent clusters of kCL CTAs take the flagged blocks (heavy
// block k to cluster k mod clusters); CTA r of a cluster runs the block's
// tiles [r n / kCL, (r + 1) n / kCL) of its n, the partial sums meet in
// shared memory and each CTA adds its BT / kCL tokens' partials over the
// cluster in rank order (a fixed order: the result does not depend on the
// number of clusters or on timing).
template <bool SPLIT>
__global__ void __launch_bounds__(kThreads, 1)
    mla_mma_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_qp,
                   const __grid_constant__ CUtensorMap tm_dy, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_kp, const PagedParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t bar_k, bar_full[2];
  __shared__ int abort_flag;
  __shared__ MPageInfo pinfo;
  __shared__ int n_tiles_sh, tile0_sh, any_store_sh, heavy_sh;
  // (the copy iterator lives in shared memory: only thread 0 uses it, and in
  // registers it would be held by every thread)
  __shared__ MPass pf;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.G, RT = BC / G;
  const int nblk = (p.max_pages + 3) / 4;
  const int rank = SPLIT ? cluster_rank() : 0;
  const int ncta = SPLIT ? kCL : 1;  // CTAs sharing one block's tiles
  const Abort ab{&abort_flag, p.err};
  const uint32_t sbase = smem_addr(sm);
  const int oob_slot = p.num_pages * p.page_size;  // out-of-range coordinate: TMA fills zeros
  const int tt = warp & 3;        // token tile (16 tokens, = page tt of the block)
  const int n8 = warp >> 2;       // phase A: column octet
  const int dr = warp >> 2;       // phase B: dim quarter
  const int g8 = lane >> 2, t4 = lane & 3;
  const float kInf = __int_as_float(0x7f800000);
  const uint32_t p_base = sbase + P_OFF, ds_base = sbase + P_OFF + PS;

  if (SPLIT) {
    // the main kernel may start on the SMs these clusters leave free
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  } else {
    // launched as the split kernel's programmatic dependent: the last CTA
    // waits for the split grid, so this grid completes after it and later
    // work in the stream sees both
    if (blockIdx.x == gridDim.x - 1 && blockIdx.y == gridDim.y - 1 && blockIdx.z == gridDim.z - 1)
      asm volatile("griddepcontrol.wait;" ::: "memory");
    const int tb = blockIdx.x, s0 = blockIdx.y;
    if (tb * 4 >= pages_of(seq_len_of(p, s0), p.page_size)) return;  // no token of the sequence here (uniform)
  }
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bar_k, 1);
    mbar_init(&bar_full[0], 1);
    mbar_init(&bar_full[1], 1);
    mbar_fence_init();
  }
  // thread 0's copy bookkeeping (split: running over the blocks of a persistent CTA)
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
      // heavy blocks (flagged by the plan kernel) belong to the split kernel
      const int heavy = !SPLIT && any && p.heavy[item] != 0;
      any_store_sh = any;
      heavy_sh = heavy;
      // this CTA's share of the block's tiles: [t0, t1), contiguous
      const int t0 = rank * n_all / ncta, t1 = (rank + 1) * n_all / ncta;
      tile0_sh = t0;
      n_tiles_sh = t1 - t0;
    }
    __syncthreads();
    // pages all stored by their owners elsewhere, or a heavy block: nothing to
    // do here (uniform over the CTA, and over the cluster: same block)
    if (!any_store_sh || heavy_sh) return;
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
      if (SPLIT) ++issued[stage];
    };
    auto pf_next = [&]() -> bool { return pf.advance(RT); };
    if (threadIdx.x == 0 && n > 0 && !abort_flag) {
      tma_prefetch_map(&tm_q);
      tma_prefetch_map(&tm_qp);
      tma_prefetch_map(&tm_dy);
      tma_prefetch_map(&tm_k);
      tma_prefetch_map(&tm_kp);
      mbar_arrive_expect_tx(&bar_k, 9 * CH);
      if (SPLIT) ++k_issued;
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
    if (!SPLIT) {
      // every issued copy was consumed (each tile waited for its stage); store
      // the pages this CTA owns, one row per token, zeros where nothing was added
      if (n > 0 && (!ok || abort_flag)) return;
      if (!pinfo.store[tt]) return;
      const int slot_base = pinfo.phys[tt] * p.page_size;
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        const int64_t prow = static_cast<int64_t>(slot_base + g8 + 8 * hr) * p.KVH + gkv;
        if (p.wrt & 2u) {
          __nv_bfloat16* o = static_cast<__nv_bfloat16*>(p.dk_pool) + prow * kLat + 128 * dr + 2 * t4;
#pragma unroll
          for (int nt = 0; nt < 16; ++nt)
            *reinterpret_cast<uint32_t*>(o + nt * 8) = pack_bf16x2(acc[nt][2 * hr], acc[nt][2 * hr + 1]);
        }
        if (p.wrt & 8u) {
          __nv_bfloat16* o = static_cast<__nv_bfloat16*>(p.dkp_pool) + prow * kPos + 16 * dr + 2 * t4;
#pragma unroll
          for (int nt = 0; nt < 2; ++nt)
            *reinterpret_cast<uint32_t*>(o + nt * 8) = pack_bf16x2(accp[nt][2 * hr], accp[nt][2 * hr + 1]);
        }
      }
      return;
    }
    // split: this CTA's partial sums to shared memory as [64 tokens][576 dims]
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
    cluster_sync();
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

  if (!SPLIT) {
    run_block(blockIdx.x, blockIdx.y, blockIdx.z, (blockIdx.y * nblk + blockIdx.x) * p.KVH + blockIdx.z);
    return;
  }
  // split: the flagged blocks in flag order, heavy block k to cluster k mod clusters
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

// ---------------------------------------------------------------------------
// Row statistics (lse, delta) of the MLA history on the same tensor path.
// One CTA owns 64 columns (64 / G query rows of one sequence, the G heads of
// one KV head) with their q, qp and dY resident in shared memory, and streams
// the sequence's keys in 32-token tiles (latent + position, double-buffered).
// Warp (token tile tt of 16, column octet n8) computes S^T and dP^T for
// 16 tokens x 8 columns per tile; each thread keeps, for its two columns, the
// online maximum m, l = sum 2^(x - m) and dsum = sum 2^(x - m) dP over its
// tokens (x = S * scale * log2 e); the partial triples are merged across lanes
// and warps at the end:  lse = (m + log2 l) * ln 2,  delta = dsum / l
// (= rowsum(P dP) = dY . O, the dS row offset of the page's backward).
// ---------------------------------------------------------------------------
constexpr int SBT = 32;                   // tokens per step (2 pages)
constexpr int SBC = 64;                   // columns per CTA
constexpr int SKC = SBT * 128;            // key chunk: [32 tokens][64 dims]
constexpr int SK_STAGE = 9 * SKC;         // 8 latent chunks + 1 position chunk
constexpr int SQC = SBC * 128;            // column chunk: [64 columns][64 dims]
constexpr int SQ_OFF = 0;                 // q (8 chunks), qp (1), dY (8)
constexpr int SK_OFF = SQ_OFF + 17 * SQC; // 2 stages
constexpr int S_BYTES = SK_OFF + 2 * SK_STAGE;
static_assert(SK_OFF % 1024 == 0 && SK_STAGE % 1024 == 0, "swizzled tiles need 1024-byte alignment");

// merge two online-softmax partials (base-2 maxima)
__device__ __forceinline__ void merge_stat(float& m, float& l, float& d, float m2, float l2, float d2) {
  const float kNegInf = -__int_as_float(0x7f800000);
  const float mm = fmaxf(m, m2);
  if (mm == kNegInf) return;
  const float a = m > kNegInf ? ex2_approx(m - mm) : 0.f, b = m2 > kNegInf ? ex2_approx(m2 - mm) : 0.f;
  l = l * a + l2 * b;
  d = d * a + d2 * b;
  m = mm;
}

__global__ void __launch_bounds__(kThreads, 1)
    mla_stats_mma_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_qp,
                         const __grid_constant__ CUtensorMap tm_dy, const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_kp, const PagedParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t bar_q, bar_k[2];
  __shared__ int abort_flag, ntok_sh, seq_sh, r0_sh;
  __shared__ float mg[3][SBC];  // the second token tile's partials: (m, l, dsum) per column

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gkv = blockIdx.x;
  const int G = p.G, RT2 = SBC / G;
  // this CTA's (sequence, row tile): the row tiles of every sequence, in order
  if (threadIdx.x == 0) {
    int idx = blockIdx.y, sq = -1, r0 = 0;
    for (int q = 0; q < p.S; ++q) {
      const int tiles = (row_end_of(p, q) - row_begin_of(p, q) + RT2 - 1) / RT2;
      if (idx < tiles) {
        sq = q;
        r0 = row_begin_of(p, q) + idx * RT2;
        break;
      }
      idx -= tiles;
    }
    seq_sh = sq;
    r0_sh = r0;
  }
  __syncthreads();
  const int s = seq_sh, r0 = r0_sh;
  if (s < 0) return;  // past the last row tile (uniform exit)
  const int re = row_end_of(p, s);
  const int len = seq_len_of(p, s);
  const int npg = pages_of(len, p.page_size);
  const Abort ab{&abort_flag, p.err};
  const int oob_slot = p.num_pages * p.page_size;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bar_q, 1);
    mbar_init(&bar_k[0], 1);
    mbar_init(&bar_k[1], 1);
    mbar_fence_init();
    int ntok = len;
    if (p.causal) {  // tokens past the largest position of the CTA's rows are never visible
      int mp = -1;
      for (int r = r0; r < r0 + RT2 && r < re; ++r) mp = max(mp, p.q_pos[r]);
      ntok = min(len, mp + 1);
    }
    ntok_sh = max(ntok, 0);
  }
  __syncthreads();
  const int nt = (ntok_sh + SBT - 1) / SBT;
  auto issue_keys = [&](int t, int stage) {
    uint64_t* bar = &bar_k[stage];
    mbar_arrive_expect_tx(bar, SK_STAGE);
    uint8_t* dst = sm + SK_OFF + stage * SK_STAGE;
    for (int j = 0; j < 2; ++j) {
      const int lp = 2 * t + j;
      int slot = oob_slot;
      if (lp < npg) {
        const int ph = p.page_table[static_cast<int64_t>(s) * p.max_pages + lp];
        if (ph >= 0 && ph < p.num_pages) slot = ph * p.page_size;
      }
      for (int c = 0; c < 8; ++c) tma_load_3d(dst + c * SKC + j * 16 * 128, &tm_k, bar, c * 64, gkv, slot);
      tma_load_3d(dst + 8 * SKC + j * 16 * 128, &tm_kp, bar, 0, gkv, slot);
    }
  };
  if (threadIdx.x == 0) {
    mbar_arrive_expect_tx(&bar_q, 17 * SQC);
    for (int c = 0; c < 8; ++c) {
      tma_load_3d(sm + SQ_OFF + c * SQC, &tm_q, &bar_q, c * 64, gkv * G, r0);
      tma_load_3d(sm + SQ_OFF + (9 + c) * SQC, &tm_dy, &bar_q, c * 64, gkv * G, r0);
    }
    tma_load_3d(sm + SQ_OFF + 8 * SQC, &tm_qp, &bar_q, 0, gkv * G, r0);
    for (int t = 0; t < 2 && t < nt; ++t) issue_keys(t, t);
  }

  const int tt = warp & 1, n8 = warp >> 1;  // 2 token tiles x 8 column octets
  const int g8 = lane >> 2, t4 = lane & 3;
  const float kNegInf = -__int_as_float(0x7f800000);
  int pos_c[2], r_c[2];
  bool col_ok[2];
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    const int c = n8 * 8 + 2 * t4 + e;
    r_c[e] = r0 + c / G;
    col_ok[e] = r_c[e] < re;
    pos_c[e] = col_ok[e] ? (p.causal ? p.q_pos[r_c[e]] : 0x7fffffff) : -1;
  }
  float m[2] = {kNegInf, kNegInf}, l[2] = {0.f, 0.f}, ds[2] = {0.f, 0.f};
  const uint32_t sbase = smem_addr(sm);
  bool ok = nt > 0 ? mbar_wait_warp(&bar_q, 0, ab) : true;
  for (int t = 0; t < nt; ++t) {
    const int stage = t & 1;
    const uint32_t kb = sbase + SK_OFF + stage * SK_STAGE;
    if (ok) ok = mbar_wait_warp(&bar_k[stage], (t >> 1) & 1, ab);
    if (ok) {
      float sacc[4] = {0.f, 0.f, 0.f, 0.f}, dpacc[4] = {0.f, 0.f, 0.f, 0.f};
      const int arow = tt * 16 + (lane & 7) + 8 * ((lane >> 3) & 1);
      const int ahalf = lane >> 4;
      const int brow = n8 * 8 + (lane & 7);
      const int bm = lane >> 3;
#pragma unroll 2
      for (int kc = 0; kc < 8; ++kc) {
#pragma unroll
        for (int kp = 0; kp < 4; ++kp) {
          uint32_t a[4], bq[4];
          ldsm_x4(swz(kb + kc * SKC, arow, 2 * kp + ahalf), a);
          ldsm_x4(swz(sbase + SQ_OFF + ((bm >> 1) ? (9 + kc) : kc) * SQC, brow, 2 * kp + (bm & 1)), bq);
          mma_16816(sacc, a, bq[0], bq[1]);
          mma_16816(dpacc, a, bq[2], bq[3]);
        }
      }
#pragma unroll
      for (int kp = 0; kp < 4; ++kp) {
        uint32_t a[4], b0, b1;
        ldsm_x4(swz(kb + 8 * SKC, arow, 2 * kp + ahalf), a);
        ldsm_x2(swz(sbase + SQ_OFF + 8 * SQC, brow, 2 * kp + (bm & 1)), b0, b1);
        mma_16816(sacc, a, b0, b1);
      }
      // online update of this thread's two columns over its two tokens
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        float x[2];
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
          const int tok = t * SBT + tt * 16 + g8 + 8 * hr;
          const bool vis = col_ok[e] && tok < len && tok <= pos_c[e];
          x[hr] = vis ? sacc[2 * hr + e] * p.scale_log2 : kNegInf;
        }
        const float mt = fmaxf(x[0], x[1]);
        if (mt > m[e]) {
          const float a = m[e] > kNegInf ? ex2_approx(m[e] - mt) : 0.f;
          l[e] *= a;
          ds[e] *= a;
          m[e] = mt;
        }
        if (m[e] > kNegInf) {
#pragma unroll
          for (int hr = 0; hr < 2; ++hr) {
            const float pe = x[hr] > kNegInf ? ex2_approx(x[hr] - m[e]) : 0.f;
            l[e] += pe;
            ds[e] = x[hr] > kNegInf ? fmaf(pe, dpacc[2 * hr + e], ds[e]) : ds[e];
          }
        }
      }
    }
    __syncthreads();  // stage free
    if (threadIdx.x == 0 && t + 2 < nt && ok && !abort_flag) issue_keys(t + 2, stage);
  }
  // merge over the 8 lanes that share a column pair (different tokens) ...
#pragma unroll
  for (int e = 0; e < 2; ++e) {
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, m[e], o);
      const float l2 = __shfl_xor_sync(0xffffffffu, l[e], o);
      const float d2 = __shfl_xor_sync(0xffffffffu, ds[e], o);
      merge_stat(m[e], l[e], ds[e], m2, l2, d2);
    }
  }
  // ... and over the two token tiles
  if (tt == 1 && g8 == 0) {
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int c = n8 * 8 + 2 * t4 + e;
      mg[0][c] = m[e];
      mg[1][c] = l[e];
      mg[2][c] = ds[e];
    }
  }
  __syncthreads();
  if (nt > 0 && (!ok || abort_flag)) return;
  if (tt == 0 && g8 == 0) {
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int c = n8 * 8 + 2 * t4 + e;
      merge_stat(m[e], l[e], ds[e], mg[0][c], mg[1][c], mg[2][c]);
      if (col_ok[e]) {
        const size_t idx = static_cast<size_t>(r_c[e]) * p.H + gkv * G + c % G;
        p.lse_out[idx] = l[e] > 0.f ? (m[e] + __log2f(l[e])) * 0.6931471805599453f : kNegInf;
        p.delta_out[idx] = l[e] > 0.f ? ds[e] / l[e] : 0.f;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Query side of the MLA backward: dQ (latent, 512) and dQp (position, 64) per
// (query row, head), from the row statistics lse and delta of the same rows.
// Same CTA decomposition as the row statistics (64 columns resident, keys in
// 32-token tiles, double-buffered) and the same phase A; then per tile
//   dS^T of the warp's 16 tokens x 8 columns -> shared memory as dS[col][token]
//   phase B  warp (column tile mt of 16, dim quarter dq): dQ[., 128 dq ..+128)
//            += dS K_lat and dQp[., 16 dq ..+16) += dS K_pos  (K as B operand,
//            token-major, read with transposing ldmatrix)
// with the fp32 accumulators (16 x 144 per warp) in registers, stored once.
// ---------------------------------------------------------------------------
constexpr int QDS_STRIDE = SBT * 2 + 16;       // dS rows: 32 bf16 + 16 bytes of padding
constexpr int QDS_OFF = S_BYTES;
constexpr int Q_BYTES = QDS_OFF + SBC * QDS_STRIDE;

__global__ void __launch_bounds__(kThreads, 1)
    mla_query_mma_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_qp,
                         const __grid_constant__ CUtensorMap tm_dy, const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_kp, const PagedParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t bar_q, bar_k[2];
  __shared__ int abort_flag, ntok_sh, seq_sh, r0_sh;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gkv = blockIdx.x;
  const int G = p.G, RT2 = SBC / G;
  if (threadIdx.x == 0) {
    int idx = blockIdx.y, sq = -1, r0 = 0;
    for (int q = 0; q < p.S; ++q) {
      const int tiles = (row_end_of(p, q) - row_begin_of(p, q) + RT2 - 1) / RT2;
      if (idx < tiles) {
        sq = q;
        r0 = row_begin_of(p, q) + idx * RT2;
        break;
      }
      idx -= tiles;
    }
    seq_sh = sq;
    r0_sh = r0;
  }
  __syncthreads();
  const int s = seq_sh, r0 = r0_sh;
  if (s < 0) return;  // past the last row tile (uniform exit)
  const int re = row_end_of(p, s);
  const int len = seq_len_of(p, s);
  const int npg = pages_of(len, p.page_size);
  const Abort ab{&abort_flag, p.err};
  const int oob_slot = p.num_pages * p.page_size;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bar_q, 1);
    mbar_init(&bar_k[0], 1);
    mbar_init(&bar_k[1], 1);
    mbar_fence_init();
    int ntok = len;
    if (p.causal) {
      int mp = -1;
      for (int r = r0; r < r0 + RT2 && r < re; ++r) mp = max(mp, p.q_pos[r]);
      ntok = min(len, mp + 1);
    }
    ntok_sh = max(ntok, 0);
  }
  __syncthreads();
  const int nt = (ntok_sh + SBT - 1) / SBT;
  auto issue_keys = [&](int t, int stage) {
    uint64_t* bar = &bar_k[stage];
    mbar_arrive_expect_tx(bar, SK_STAGE);
    uint8_t* dst = sm + SK_OFF + stage * SK_STAGE;
    for (int j = 0; j < 2; ++j) {
      const int lp = 2 * t + j;
      int slot = oob_slot;
      if (lp < npg) {
        const int ph = p.page_table[static_cast<int64_t>(s) * p.max_pages + lp];
        if (ph >= 0 && ph < p.num_pages) slot = ph * p.page_size;
      }
      for (int c = 0; c < 8; ++c) tma_load_3d(dst + c * SKC + j * 16 * 128, &tm_k, bar, c * 64, gkv, slot);
      tma_load_3d(dst + 8 * SKC + j * 16 * 128, &tm_kp, bar, 0, gkv, slot);
    }
  };
  if (threadIdx.x == 0) {
    mbar_arrive_expect_tx(&bar_q, 17 * SQC);
    for (int c = 0; c < 8; ++c) {
      tma_load_3d(sm + SQ_OFF + c * SQC, &tm_q, &bar_q, c * 64, gkv * G, r0);
      tma_load_3d(sm + SQ_OFF + (9 + c) * SQC, &tm_dy, &bar_q, c * 64, gkv * G, r0);
    }
    tma_load_3d(sm + SQ_OFF + 8 * SQC, &tm_qp, &bar_q, 0, gkv * G, r0);
    for (int t = 0; t < 2 && t < nt; ++t) issue_keys(t, t);
  }

  const int tt = warp & 1, n8 = warp >> 1;  // phase A: 2 token tiles x 8 column octets
  const int mt = warp & 3, dq = warp >> 2;  // phase B: 4 column tiles x 4 dim quarters
  const int g8 = lane >> 2, t4 = lane & 3;
  const float kInf = __int_as_float(0x7f800000);
  // phase-A columns of this thread: statistics, position
  float lse_c[2], dl_c[2];
  int pos_c[2];
  bool col_ok[2];
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    const int c = n8 * 8 + 2 * t4 + e;
    const int r = r0 + c / G, hh = gkv * G + c % G;
    col_ok[e] = r < re;
    const size_t si = static_cast<size_t>(col_ok[e] ? r : 0) * p.H + hh;
    lse_c[e] = col_ok[e] ? p.lse[si] * kLog2e : kInf;
    dl_c[e] = col_ok[e] ? p.delta[si] : 0.f;
    pos_c[e] = col_ok[e] ? (p.causal ? p.q_pos[r] : 0x7fffffff) : -1;
  }
  float acc[16][4], accp[2][4];
#pragma unroll
  for (int i = 0; i < 16; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
#pragma unroll
  for (int i = 0; i < 2; ++i) accp[i][0] = accp[i][1] = accp[i][2] = accp[i][3] = 0.f;
  const uint32_t sbase = smem_addr(sm);
  const uint32_t ds_base = sbase + QDS_OFF;
  bool ok = nt > 0 ? mbar_wait_warp(&bar_q, 0, ab) : true;
  for (int t = 0; t < nt; ++t) {
    const int stage = t & 1;
    const uint32_t kb = sbase + SK_OFF + stage * SK_STAGE;
    if (ok) ok = mbar_wait_warp(&bar_k[stage], (t >> 1) & 1, ab);
    if (ok) {
      // ---------------------------------------------------------------- phase A
      float sacc[4] = {0.f, 0.f, 0.f, 0.f}, dpacc[4] = {0.f, 0.f, 0.f, 0.f};
      const int arow = tt * 16 + (lane & 7) + 8 * ((lane >> 3) & 1);
      const int ahalf = lane >> 4;
      const int brow = n8 * 8 + (lane & 7);
      const int bm = lane >> 3;
#pragma unroll 2
      for (int kc = 0; kc < 8; ++kc) {
#pragma unroll
        for (int kp = 0; kp < 4; ++kp) {
          uint32_t a[4], bq[4];
          ldsm_x4(swz(kb + kc * SKC, arow, 2 * kp + ahalf), a);
          ldsm_x4(swz(sbase + SQ_OFF + ((bm >> 1) ? (9 + kc) : kc) * SQC, brow, 2 * kp + (bm & 1)), bq);
          mma_16816(sacc, a, bq[0], bq[1]);
          mma_16816(dpacc, a, bq[2], bq[3]);
        }
      }
#pragma unroll
      for (int kp = 0; kp < 4; ++kp) {
        uint32_t a[4], b0, b1;
        ldsm_x4(swz(kb + 8 * SKC, arow, 2 * kp + ahalf), a);
        ldsm_x2(swz(sbase + SQ_OFF + 8 * SQC, brow, 2 * kp + (bm & 1)), b0, b1);
        mma_16816(sacc, a, b0, b1);
      }
      // dS of this warp's 16 tokens x 8 columns, stored column-major for phase B
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        const int i = tt * 16 + g8 + 8 * hr;  // tile-local token
        const int tok = t * SBT + i;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const bool vis = col_ok[e] && tok < len && tok <= pos_c[e] && lse_c[e] < kInf;
          const float pe = ex2_approx(fmaf(sacc[2 * hr + e], p.scale_log2, -lse_c[e]));
          // select, not multiply: S and dP of a tail slot may be NaN
          const float dsv = vis ? pe * (dpacc[2 * hr + e] - dl_c[e]) * p.scale : 0.f;
          const int c = n8 * 8 + 2 * t4 + e;
          *reinterpret_cast<__nv_bfloat16*>(sm + QDS_OFF + c * QDS_STRIDE + i * 2) = __float2bfloat16_rn(dsv);
        }
      }
    }
    __syncthreads();
    if (t * SBT + SBT > len) {  // uniform: the barrier below is reached by every thread
      // key rows of tokens past the length inside the last page may hold any
      // bit pattern; phase B multiplies them by dS = 0, so they are zeroed
      if (ok) {
        const int row_lo = max(0, len - t * SBT);
        const int nvec = (SBT - row_lo) * 9 * 8;
        for (int i = threadIdx.x; i < nvec; i += kThreads) {
          const int rw = row_lo + i / 72, rem = i % 72;
          st_shared_v4(kb + (rem >> 3) * SKC + rw * 128 + (rem & 7) * 16, 0u, 0u, 0u, 0u);
        }
      }
      __syncthreads();
    }
    if (ok && !abort_flag) {
      // ---------------------------------------------------------------- phase B
      const int arow = mt * 16 + (lane & 7) + 8 * ((lane >> 3) & 1);
      const int bm = lane >> 3;
#pragma unroll
      for (int ks = 0; ks < 2; ++ks) {
        uint32_t ads[4];
        ldsm_x4(ds_base + arow * QDS_STRIDE + (ks * 16 + 8 * (lane >> 4)) * 2, ads);
        const int krow = ks * 16 + (lane & 7) + 8 * (bm & 1);  // token index = B row
#pragma unroll
        for (int np = 0; np < 8; ++np) {  // pairs of 8-dim tiles: dims 128 dq + 16 np
          const int chunk = 2 * dq + (np >> 2);
          const int piece = 2 * (np & 3) + (bm >> 1);
          uint32_t bk[4];
          ldsm_x4_t(swz(kb + chunk * SKC, krow, piece), bk);
          mma_16816(acc[2 * np], ads, bk[0], bk[1]);
          mma_16816(acc[2 * np + 1], ads, bk[2], bk[3]);
        }
        uint32_t bkp[4];
        ldsm_x4_t(swz(kb + 8 * SKC, krow, 2 * dq + (bm >> 1)), bkp);
        mma_16816(accp[0], ads, bkp[0], bkp[1]);
        mma_16816(accp[1], ads, bkp[2], bkp[3]);
      }
    }
    __syncthreads();  // stage and dS buffer free
    if (threadIdx.x == 0 && t + 2 < nt && ok && !abort_flag) issue_keys(t + 2, stage);
  }
  if (nt > 0 && (!ok || abort_flag)) return;
  // one store per (row, head): zeros for a column that saw no token
#pragma unroll
  for (int hr = 0; hr < 2; ++hr) {
    const int c = mt * 16 + g8 + 8 * hr;
    const int r = r0 + c / G, hh = gkv * G + c % G;
    if (r >= re) continue;
    const int64_t row = static_cast<int64_t>(r) * p.H + hh;
    __nv_bfloat16* o = static_cast<__nv_bfloat16*>(p.dq) + row * kLat + 128 * dq + 2 * t4;
#pragma unroll
    for (int n = 0; n < 16; ++n)
      *reinterpret_cast<uint32_t*>(o + n * 8) = pack_bf16x2(acc[n][2 * hr], acc[n][2 * hr + 1]);
    __nv_bfloat16* op = static_cast<__nv_bfloat16*>(p.dqp) + row * kPos + 16 * dq + 2 * t4;
#pragma unroll
    for (int n = 0; n < 2; ++n)
      *reinterpret_cast<uint32_t*>(op + n * 8) = pack_bf16x2(accp[n][2 * hr], accp[n][2 * hr + 1]);
  }
}

}  // namespace

bool mla_mma_supported(const PagedParams& p) {
  return p.Dk == kLat && p.Dp == kPos && p.page_size == 16 && (p.G == 4 || p.G == 8 || p.G == 16 || p.G == 32);
}

cudaError_t launch_paged_mla_stats_mma(const PagedMlaMaps& m, const PagedParams& p, cudaStream_t s) {
  if (p.Nq == 0 || p.S == 0) return cudaSuccess;
  const int smem = S_BYTES + 1024;
  cudaError_t e = cudaFuncSetAttribute(mla_stats_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  // an upper bound on the row tiles of all sequences; each CTA finds its own
  const int RT2 = SBC / p.G;
  dim3 grid(p.KVH, p.Nq / RT2 + p.S + 1, 1);
  mla_stats_mma_kernel<<<grid, kThreads, smem, s>>>(m.q, m.qp, m.dy, m.k, m.kp, p);
  return cudaGetLastError();
}

cudaError_t launch_paged_mla_mma(const PagedMlaMaps& m, const PagedParams& p, cudaStream_t s) {
  if (p.num_pages == 0 || p.S == 0 || p.max_pages == 0) return cudaSuccess;
  const int smem = BYTES + 1024;
  auto kern = mla_mma_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  // programmatic dependent of the split kernel launched just before it: it
  // may start while the split clusters run (it reads none of their results)
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((p.max_pages + 3) / 4, p.S, p.KVH);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, m.q, m.qp, m.dy, m.k, m.kp, p);
}

cudaError_t launch_paged_mla_plan(const PagedParams& p, cudaStream_t s) {
  const int64_t n = static_cast<int64_t>(p.S) * ((p.max_pages + 3) / 4);
  if (n == 0 || p.num_pages == 0) return cudaSuccess;
  const int blocks = static_cast<int>((n + 127) / 128 < 1024 ? (n + 127) / 128 : 1024);
  mla_plan_kernel<<<blocks, 128, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_paged_mla_mma_split(const PagedMlaMaps& m, const PagedParams& p, cudaStream_t s) {
  if (p.num_pages == 0 || p.S == 0 || p.max_pages == 0) return cudaSuccess;
  const int smem = BYTES + 1024;
  auto kern = mla_mma_kernel<true>;
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

namespace attn {

cudaError_t launch_paged_mla_query_mma(const PagedMlaMaps& m, const PagedParams& p, cudaStream_t s) {
  if (p.Nq == 0 || p.S == 0) return cudaSuccess;
  const int smem = Q_BYTES + 1024;
  cudaError_t e = cudaFuncSetAttribute(mla_query_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int RT2 = SBC / p.G;
  dim3 grid(p.KVH, p.Nq / RT2 + p.S + 1, 1);
  mla_query_mma_kernel<<<grid, kThreads, smem, s>>>(m.q, m.qp, m.dy, m.k, m.kp, p);
  return cudaGetLastError();
}

}  // namespace attn
