// Paged MLA history backward and MLA row statistics (CUDA cores).
//
// ruDNN src/paged_attention/ordered_kernel.rs (history_backward with `mla`):
// the score of query row r, head h and history token t is
//   s = scale * (q[r,h] . k_lat[t] + qp[r,h] . k_pos[t]),
// the latent is both key and value, and for every physical token and KV head
//   p   = exp(s - lse[r,h])
//   ds  = p * (dY[r,h] . k_lat[t] - delta[r,h]) * scale
//   dK_lat[t] += ds * q[r,h] + p * dY[r,h]       ("retain both derivatives")
//   dKp[t]    += ds * qp[r,h]
// summed over the links of the token's page (in link order), the visible rows
// of each linked sequence (t <= pos(r) when causal) and the heads of the group.
//
// mla_history_kernel: one CTA per (physical page, KV head); warp w owns slot w
// of the page (the page's owner stores all 16 slots once, zeros for slots no
// link makes valid).  Query rows are staged in shared memory with bulk copies
// (all G heads of one row at a time: q, qp, dY), so the 16 slot-warps share
// every load.  Lane l handles latent dims 16l..16l+15 and position dims
// 2l, 2l+1 (key_dim 512, position_dim 64).
//
// mla_stats_kernel: one CTA per (query row, KV head), one warp per head of the
// group; the row's visible history is staged one 16-token page at a time and
// every warp runs an online softmax with O += p * k_lat, then
// delta = dY . O / l and lse = m + log l.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "paged_common.cuh"
#include "paged_launch.h"
#include "sm103.cuh"

namespace attn {
using namespace sm103;

namespace {

constexpr int kLat = 512, kPos = 64;

__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_addr(dst)),
               "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_addr(bar))
               : "memory");
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// 16 consecutive bf16 at p (32-byte aligned) -> fp32
__device__ __forceinline__ void load16(const __nv_bfloat16* p, float (&v)[16]) {
  const uint4 a = reinterpret_cast<const uint4*>(p)[0];
  const uint4 b = reinterpret_cast<const uint4*>(p)[1];
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

__device__ __forceinline__ void load2(const __nv_bfloat16* p, float (&v)[2]) {
  const uint32_t w = *reinterpret_cast<const uint32_t*>(p);
  v[0] = __uint_as_float(w << 16);
  v[1] = __uint_as_float(w & 0xffff0000u);
}

// ---------------------------------------------------------------------------
// history backward
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(512, 1) mla_history_kernel(const __nv_bfloat16* __restrict__ q,
                                                             const __nv_bfloat16* __restrict__ qp,
                                                             const __nv_bfloat16* __restrict__ dy,
                                                             const __nv_bfloat16* __restrict__ k_pool,
                                                             const __nv_bfloat16* __restrict__ kp_pool,
                                                             const PagedParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  __shared__ uint64_t bar_full[2];
  __shared__ int abort_flag;
  const int page = blockIdx.x, g = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.G;
  const uint32_t q_bytes = G * kLat * 2, qp_bytes = G * kPos * 2, dy_bytes = G * kLat * 2;
  const uint32_t stage_bytes = q_bytes + qp_bytes + dy_bytes;
  const Abort ab{&abort_flag, p.err};
  if (p.listed && !p.listed[page]) return;  // compact history: a page not asked for (uniform)
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bar_full[0], 1);
    mbar_init(&bar_full[1], 1);
    mbar_fence_init();
  }
  __syncthreads();

  const int slot = page * p.page_size + warp;
  const int64_t prow = static_cast<int64_t>(slot) * p.KVH + g;
  // this slot's latent and position key, lane-distributed
  float kl[16], kpv[2];
  load16(k_pool + prow * kLat + lane * 16, kl);
  load2(kp_pool + prow * kPos + lane * 2, kpv);
  float dk[16], dkp[2];
#pragma unroll
  for (int i = 0; i < 16; ++i) dk[i] = 0.f;
  dkp[0] = dkp[1] = 0.f;
  bool any_valid = false;

  const int l0 = p.link_off[page], l1 = p.link_off[page + 1];
  // The steps are the (link, query row) pairs in link order; every thread
  // walks them identically (same number of __syncthreads).  Thread 0 stages
  // the rows of step k+1 while the warps consume step k.
  auto stage_row = [&](int r, int st) {
    mbar_arrive_expect_tx(&bar_full[st], stage_bytes);
    uint8_t* buf = sm + st * stage_bytes;
    const int64_t base = static_cast<int64_t>(r) * p.H + g * G;
    bulk_g2s(buf, q + base * kLat, q_bytes, &bar_full[st]);
    bulk_g2s(buf + q_bytes, qp + base * kPos, qp_bytes, &bar_full[st]);
    bulk_g2s(buf + q_bytes + qp_bytes, dy + base * kLat, dy_bytes, &bar_full[st]);
  };
  // first step: the first link whose sequence has rows
  auto first_row = [&](int li, int* r_out) {
    for (; li < l1; ++li) {
      const int s = p.links[li] / p.max_pages;
      if (row_end_of(p, s) > row_begin_of(p, s)) {
        *r_out = row_begin_of(p, s);
        return li;
      }
    }
    return l1;
  };
  int nli = 0, nr = 0;  // the step after the current one (thread 0's lookahead)
  if (threadIdx.x == 0) {
    nli = first_row(l0, &nr);
    if (nli < l1) stage_row(nr, 0);
  }
  int step = 0;
  bool ok = true;
  for (int li = l0; li < l1; ++li) {
    const int link = p.links[li];
    const int s = link / p.max_pages, lp = link - s * p.max_pages;
    const int len = seq_len_of(p, s);
    const int tok = lp * p.page_size + warp;
    const bool tok_ok = tok < len;
    any_valid |= tok_ok;
    const int rb = row_begin_of(p, s), re = row_end_of(p, s);
    for (int r = rb; r < re; ++r, ++step) {
      const int st = step & 1;
      uint8_t* buf = sm + st * stage_bytes;
      __syncthreads();  // every warp is done with the buffer the next copy reuses
      if (threadIdx.x == 0 && !abort_flag && nli < l1) {
        // advance the lookahead past the current step and stage it
        if (nr + 1 < row_end_of(p, p.links[nli] / p.max_pages)) {
          ++nr;
        } else {
          nli = first_row(nli + 1, &nr);
        }
        if (nli < l1) stage_row(nr, st ^ 1);
      }
      const int pos = p.causal ? p.q_pos[r] : 0x7fffffff;
      const bool vis = tok_ok && tok <= pos;
      if (!mbar_wait_warp(&bar_full[st], (step >> 1) & 1, ab)) {
        ok = false;  // aborting: keep the loop shape, skip the work
        continue;
      }
      if (!vis || !ok) continue;
      const __nv_bfloat16* qs = reinterpret_cast<const __nv_bfloat16*>(buf);
      const __nv_bfloat16* qps = reinterpret_cast<const __nv_bfloat16*>(buf + q_bytes);
      const __nv_bfloat16* dys = reinterpret_cast<const __nv_bfloat16*>(buf + q_bytes + qp_bytes);
      for (int hh = 0; hh < G; ++hh) {
        const int64_t sidx = static_cast<int64_t>(r) * p.H + g * G + hh;
        const float lse = p.lse[sidx];
        if (lse == -__int_as_float(0x7f800000)) continue;  // row with no visible token
        float qv[16], qpv[2], gv[16];
        load16(qs + hh * kLat + lane * 16, qv);
        load2(qps + hh * kPos + lane * 2, qpv);
        load16(dys + hh * kLat + lane * 16, gv);
        float sc = qpv[0] * kpv[0] + qpv[1] * kpv[1], dpv = 0.f;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          sc = fmaf(qv[i], kl[i], sc);
          dpv = fmaf(gv[i], kl[i], dpv);
        }
        sc = warp_sum(sc);
        dpv = warp_sum(dpv);
        const float pr = ex2_approx((sc * p.scale - lse) * 1.4426950408889634f);
        const float ds = pr * (dpv - p.delta[sidx]) * p.scale;
#pragma unroll
        for (int i = 0; i < 16; ++i) dk[i] = fmaf(ds, qv[i], fmaf(pr, gv[i], dk[i]));
        dkp[0] = fmaf(ds, qpv[0], dkp[0]);
        dkp[1] = fmaf(ds, qpv[1], dkp[1]);
      }
    }
  }
  // every staged copy was waited for in the loop (the lookahead never runs past
  // the last step); store this slot once, zero if no link made it valid
  __syncthreads();
  if (!ok || abort_flag) return;
  (void)any_valid;
  if (p.wrt & 2u) {
    uint32_t w[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) w[i] = pack_bf16x2(dk[2 * i], dk[2 * i + 1]);
    uint4* o = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.dk_pool) + prow * kLat + lane * 16);
    o[0] = make_uint4(w[0], w[1], w[2], w[3]);
    o[1] = make_uint4(w[4], w[5], w[6], w[7]);
  }
  if (p.wrt & 8u)
    *reinterpret_cast<uint32_t*>(reinterpret_cast<__nv_bfloat16*>(p.dkp_pool) + prow * kPos + lane * 2) =
        pack_bf16x2(dkp[0], dkp[1]);
}

// ---------------------------------------------------------------------------
// row statistics
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(1024, 1) mla_stats_kernel(const __nv_bfloat16* __restrict__ q,
                                                            const __nv_bfloat16* __restrict__ qp,
                                                            const __nv_bfloat16* __restrict__ dy,
                                                            const __nv_bfloat16* __restrict__ k_pool,
                                                            const __nv_bfloat16* __restrict__ kp_pool,
                                                            const PagedParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  __shared__ uint64_t bar_full[2];
  __shared__ int abort_flag;
  __shared__ int seq_sh;
  const int r = blockIdx.x, g = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.G;
  const int ps = p.page_size;
  const uint32_t kl_bytes = ps * kLat * 2, kp_bytes = ps * kPos * 2;
  const uint32_t stage_bytes = kl_bytes + kp_bytes;
  const Abort ab{&abort_flag, p.err};
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bar_full[0], 1);
    mbar_init(&bar_full[1], 1);
    mbar_fence_init();
    // sequence of row r: the last s with q_start[s] <= r (binary search)
    int lo = 0, hi = p.S - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (p.q_start[mid] <= r) lo = mid; else hi = mid - 1;
    }
    seq_sh = lo;
  }
  __syncthreads();
  const int s = seq_sh;
  const int len = seq_len_of(p, s);
  const int pos = p.causal ? p.q_pos[r] : len - 1;
  const int last = min(len - 1, pos);
  const int npages = last < 0 ? 0 : last / ps + 1;
  const bool active = warp < G;
  const int hh = g * G + warp;
  float qv[16], qpv[2];
  if (active) {
    const int64_t row = static_cast<int64_t>(r) * p.H + hh;
    load16(q + row * kLat + lane * 16, qv);
    load2(qp + row * kPos + lane * 2, qpv);
  }
  float m = -__int_as_float(0x7f800000), l = 0.f, o[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) o[i] = 0.f;
  __shared__ int page_ok[2];
  bool ok = true;
  // Thread 0 stages page pg+1 while the warps consume page pg; every thread
  // runs the same number of iterations (same number of __syncthreads).
  auto stage_page = [&](int pg, int st) {
    const int ph = p.page_table[static_cast<int64_t>(s) * p.max_pages + pg];
    uint8_t* buf = sm + st * stage_bytes;
    if (ph < 0 || ph >= p.num_pages) {  // malformed table entry: read nothing
      page_ok[st] = 0;
      mbar_arrive(&bar_full[st]);
      return;
    }
    page_ok[st] = 1;
    mbar_arrive_expect_tx(&bar_full[st], stage_bytes);
    // a page's slots hold rows (slot, kv head): with KVH > 1 they are not
    // contiguous per head, so copy slot by slot
    for (int t = 0; t < ps; ++t) {
      const int64_t prow = (static_cast<int64_t>(ph) * ps + t) * p.KVH + g;
      bulk_g2s(buf + t * kLat * 2, k_pool + prow * kLat, kLat * 2, &bar_full[st]);
      bulk_g2s(buf + kl_bytes + t * kPos * 2, kp_pool + prow * kPos, kPos * 2, &bar_full[st]);
    }
  };
  if (threadIdx.x == 0 && npages > 0) stage_page(0, 0);
  for (int pg = 0; pg < npages; ++pg) {
    const int st = pg & 1;
    uint8_t* buf = sm + st * stage_bytes;
    __syncthreads();
    if (threadIdx.x == 0 && pg + 1 < npages && !abort_flag) stage_page(pg + 1, st ^ 1);
    if (!mbar_wait_warp(&bar_full[st], (pg >> 1) & 1, ab)) {
      ok = false;
      continue;
    }
    if (!active || !ok || !page_ok[st]) continue;
    const __nv_bfloat16* kls = reinterpret_cast<const __nv_bfloat16*>(buf);
    const __nv_bfloat16* kps = reinterpret_cast<const __nv_bfloat16*>(buf + kl_bytes);
    for (int t = 0; t < ps; ++t) {
      const int tok = pg * ps + t;
      if (tok > last) break;
      float kv[16], kpv[2];
      load16(kls + t * kLat + lane * 16, kv);
      load2(kps + t * kPos + lane * 2, kpv);
      float sc = qpv[0] * kpv[0] + qpv[1] * kpv[1];
#pragma unroll
      for (int i = 0; i < 16; ++i) sc = fmaf(qv[i], kv[i], sc);
      sc = warp_sum(sc) * p.scale;
      if (sc > m) {
        const float a = __expf(m - sc);
        l *= a;
#pragma unroll
        for (int i = 0; i < 16; ++i) o[i] *= a;
        m = sc;
      }
      const float e = __expf(sc - m);
      l += e;
#pragma unroll
      for (int i = 0; i < 16; ++i) o[i] = fmaf(e, kv[i], o[i]);
    }
  }
  __syncthreads();
  if (!ok || !active || abort_flag) return;
  float gv[16];
  load16(dy + (static_cast<int64_t>(r) * p.H + hh) * kLat + lane * 16, gv);
  float dl = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) dl = fmaf(gv[i], o[i], dl);
  dl = warp_sum(dl);
  if (lane == 0) {
    const int64_t idx = static_cast<int64_t>(r) * p.H + hh;
    p.lse_out[idx] = l > 0.f ? m + __logf(l) : -__int_as_float(0x7f800000);
    p.delta_out[idx] = l > 0.f ? dl / l : 0.f;
  }
}

}  // namespace

cudaError_t launch_paged_mla_history(const PagedParams& p, const void* q, const void* qp, const void* dy,
                                     const void* k_pool, const void* kp_pool, cudaStream_t s) {
  if (p.num_pages == 0) return cudaSuccess;
  const int smem = 2 * p.G * (kLat + kPos + kLat) * 2 + 128;
  cudaError_t e = cudaFuncSetAttribute(mla_history_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  dim3 grid(p.num_pages, p.KVH);
  mla_history_kernel<<<grid, 32 * p.page_size, smem, s>>>(
      static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(qp),
      static_cast<const __nv_bfloat16*>(dy), static_cast<const __nv_bfloat16*>(k_pool),
      static_cast<const __nv_bfloat16*>(kp_pool), p);
  return cudaGetLastError();
}

cudaError_t launch_paged_mla_stats(const PagedParams& p, const void* q, const void* qp, const void* dy,
                                   const void* k_pool, const void* kp_pool, cudaStream_t s) {
  if (p.Nq == 0 || p.S == 0) return cudaSuccess;
  const int smem = 2 * p.page_size * (kLat + kPos) * 2 + 128;
  cudaError_t e = cudaFuncSetAttribute(mla_stats_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int threads = 32 * (p.G < 1 ? 1 : p.G);
  dim3 grid(p.Nq, p.KVH);
  mla_stats_kernel<<<grid, threads, smem, s>>>(
      static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(qp),
      static_cast<const __nv_bfloat16*>(dy), static_cast<const __nv_bfloat16*>(k_pool),
      static_cast<const __nv_bfloat16*>(kp_pool), p);
  return cudaGetLastError();
}

}  // namespace attn
