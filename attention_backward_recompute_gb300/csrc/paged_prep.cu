// Paged prep: the inverse of the page table (links of every physical page in
// a fixed order) and the zero store of pool rows no valid token owns.
//
// ruDNN src/paged_attention/ordered_kernel.rs builds the same inverse on the
// host (per-page link ranges, link = (sequence, logical page)); here it is
// built on the device from the caller's page table so the call stays
// asynchronous:
//   count  : links per physical page (integer atomics; the counts are exact)
//   scan   : exclusive prefix sum -> link_off
//   fill   : each link takes a slot of its page's segment
//   order  : each segment is sorted by link id, which fixes the traversal
//            order independently of the atomics above
// and "inactive pages/tail slots also store zero": pages with no link get
// zero dK/dV/dKp rows here; tail slots of linked pages get zero from their
// owner CTA.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "paged_common.cuh"
#include "paged_launch.h"

namespace attn {
namespace {

__global__ void count_links_kernel(PagedParams p) {
  const int64_t n = static_cast<int64_t>(p.S) * p.max_pages;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int s = static_cast<int>(i / p.max_pages), lp = static_cast<int>(i % p.max_pages);
    if (lp >= pages_of(seq_len_of(p, s), p.page_size)) continue;
    const int page = p.page_table[i];
    if (page < 0 || page >= p.num_pages) {
      atomicOr(p.err, kErrBadPage);
      continue;
    }
    atomicAdd(&p.link_count[page], 1);
  }
}

// single-CTA exclusive scan of link_count into link_off[0..num_pages]: each
// thread scans kScanPer consecutive counts in registers, the block scans the
// thread totals, one chunk of 1024 x kScanPer pages after another
constexpr int kScanPer = 16;
__global__ void __launch_bounds__(1024) scan_links_kernel(PagedParams p) {
  __shared__ int warp_sums[32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int carry = 0;  // sum of the chunks before (the same in every thread)
  for (int base = 0; base < p.num_pages; base += 1024 * kScanPer) {
    const int i0 = base + static_cast<int>(threadIdx.x) * kScanPer;
    int v[kScanPer];
    if (i0 + kScanPer <= p.num_pages) {  // 64-byte aligned: the workspace arrays are 256-byte aligned
      const int4* src = reinterpret_cast<const int4*>(p.link_count + i0);
#pragma unroll
      for (int k = 0; k < kScanPer / 4; ++k) {
        const int4 w = src[k];
        v[4 * k] = w.x;
        v[4 * k + 1] = w.y;
        v[4 * k + 2] = w.z;
        v[4 * k + 3] = w.w;
      }
    } else {
#pragma unroll
      for (int k = 0; k < kScanPer; ++k) v[k] = i0 + k < p.num_pages ? p.link_count[i0 + k] : 0;
    }
    int tot = 0;
#pragma unroll
    for (int k = 0; k < kScanPer; ++k) tot += v[k];
    int x = tot;  // inclusive scan of the thread totals within the warp
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) warp_sums[warp] = x;
    __syncthreads();
    if (warp == 0) {
      int w = warp_sums[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += y;
      }
      warp_sums[lane] = w;
    }
    __syncthreads();
    int run = carry + x - tot + (warp > 0 ? warp_sums[warp - 1] : 0);  // exclusive prefix of this thread
#pragma unroll
    for (int k = 0; k < kScanPer; ++k) {
      if (i0 + k < p.num_pages) p.link_off[i0 + k] = run;
      run += v[k];
    }
    carry += warp_sums[31];
    __syncthreads();  // warp_sums is rewritten by the next chunk
  }
  if (threadIdx.x == 0) p.link_off[p.num_pages] = carry;
}

__global__ void fill_links_kernel(PagedParams p) {
  const int64_t n = static_cast<int64_t>(p.S) * p.max_pages;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int s = static_cast<int>(i / p.max_pages), lp = static_cast<int>(i % p.max_pages);
    if (lp >= pages_of(seq_len_of(p, s), p.page_size)) continue;
    const int page = p.page_table[i];
    if (page < 0 || page >= p.num_pages) continue;
    const int slot = atomicAdd(&p.link_fill[page], 1);
    p.links[p.link_off[page] + slot] = static_cast<int32_t>(i);
  }
}

// insertion sort of each page's (short) link segment
__global__ void order_links_kernel(PagedParams p) {
  for (int page = blockIdx.x * blockDim.x + threadIdx.x; page < p.num_pages; page += gridDim.x * blockDim.x) {
    const int a = p.link_off[page], b = p.link_off[page + 1];
    for (int i = a + 1; i < b; ++i) {
      const int32_t key = p.links[i];
      int j = i - 1;
      while (j >= a && p.links[j] > key) {
        p.links[j + 1] = p.links[j];
        --j;
      }
      p.links[j + 1] = key;
    }
  }
}

// zero the rows of pages that no link references: one block per page (of
// the pool, or of the compact-history list), 16 bytes per thread
__global__ void zero_unlinked_kernel(PagedParams p, void* pool, int dim, const int32_t* list, int nlist) {
  const int per_page = p.page_size * p.KVH * (dim / 8);  // 16-byte vectors per page (bf16 rows)
  const int npg = list ? nlist : p.num_pages;
  const uint4 z = make_uint4(0u, 0u, 0u, 0u);
  for (int i = blockIdx.x; i < npg; i += gridDim.x) {
    const int page = list ? list[i] : i;
    if (page < 0 || page >= p.num_pages || p.link_count[page] != 0) continue;  // uniform over the block
    uint4* dst = reinterpret_cast<uint4*>(pool) + static_cast<int64_t>(page) * per_page;
    for (int v = threadIdx.x; v < per_page; v += blockDim.x) dst[v] = z;
  }
}

// compact history: mark the listed pages (an entry outside the pool raises
// kErrBadPage and is skipped)
__global__ void mark_listed_kernel(PagedParams p, const int32_t* pages, int64_t n) {
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int page = pages[i];
    if (page < 0 || page >= p.num_pages) {
      atomicOr(p.err, kErrBadPage);
      continue;
    }
    p.listed[page] = 1;
  }
}

// Query-side dispatch order: order[rank] = s, ranked by decreasing sequence
// length (ties by index), one thread per sequence (S^2 reads of the lengths).
__global__ void seq_order_kernel(PagedParams p) {
  for (int s = blockIdx.x * blockDim.x + threadIdx.x; s < p.S; s += gridDim.x * blockDim.x) {
    const int len = seq_len_of(p, s);
    int rank = 0;
    for (int o = 0; o < p.S; ++o) {
      const int lo = seq_len_of(p, o);
      rank += (lo > len || (lo == len && o < s)) ? 1 : 0;
    }
    p.order[rank] = s;
  }
}

}  // namespace

cudaError_t launch_paged_seq_order(const PagedParams& p, cudaStream_t s) {
  if (p.S <= 0) return cudaSuccess;
  const int blocks = (p.S + 255) / 256 < 1024 ? (p.S + 255) / 256 : 1024;
  seq_order_kernel<<<blocks, 256, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_paged_listed(const PagedParams& p, const int32_t* pages, int64_t n, cudaStream_t s) {
  cudaError_t e;
  if ((e = cudaMemsetAsync(p.listed, 0, p.num_pages, s)) != cudaSuccess) return e;
  if (n <= 0) return cudaSuccess;
  const int64_t blocks = (n + 255) / 256 < 1024 ? (n + 255) / 256 : 1024;
  mark_listed_kernel<<<static_cast<int>(blocks), 256, 0, s>>>(p, pages, n);
  return cudaGetLastError();
}

cudaError_t launch_paged_prep(const PagedParams& p, cudaStream_t s) {
  cudaError_t e;
  if ((e = cudaMemsetAsync(p.link_count, 0, sizeof(int32_t) * p.num_pages, s)) != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(p.link_fill, 0, sizeof(int32_t) * p.num_pages, s)) != cudaSuccess) return e;
  const int64_t nl = static_cast<int64_t>(p.S) * p.max_pages;
  const int gl = static_cast<int>((nl + 255) / 256 < 4096 ? (nl + 255) / 256 : 4096);
  count_links_kernel<<<gl > 0 ? gl : 1, 256, 0, s>>>(p);
  scan_links_kernel<<<1, 1024, 0, s>>>(p);
  fill_links_kernel<<<gl > 0 ? gl : 1, 256, 0, s>>>(p);
  const int gp = (p.num_pages + 255) / 256;
  order_links_kernel<<<gp > 0 ? gp : 1, 256, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_paged_zero_unlinked(const PagedParams& p, const int32_t* list, int64_t nlist, cudaStream_t s) {
  const int64_t npg = list ? nlist : p.num_pages;
  if (npg <= 0) return cudaSuccess;
  const int blocks = static_cast<int>(npg < 152 * 8 ? npg : 152 * 8);
  const int n = static_cast<int>(npg);
  if ((p.wrt & 2u) && p.dk_pool) zero_unlinked_kernel<<<blocks, 256, 0, s>>>(p, p.dk_pool, p.Dk, list, n);
  if ((p.wrt & 4u) && p.dv_pool && p.Dp == 0) zero_unlinked_kernel<<<blocks, 256, 0, s>>>(p, p.dv_pool, p.Dv, list, n);
  if ((p.wrt & 8u) && p.dkp_pool && p.Dp > 0) zero_unlinked_kernel<<<blocks, 256, 0, s>>>(p, p.dkp_pool, p.Dp, list, n);
  return cudaGetLastError();
}

}  // namespace attn
