// Shared definitions of the paged-KV history kernels.
//
// Work decomposition (ruDNN src/paged_attention/ordered_kernel.rs,
// history_backward: one owner per physical token x KV head, fixed traversal,
// one final store): a CTA owns 128 consecutive history tokens (eight 16-token
// pages) of one sequence for one KV head and accumulates their dK/dV in
// tensor memory.  A physical page referenced by several (sequence, logical
// page) links is stored only by the CTA of its FIRST link (smallest
// sequence * max_pages + logical page); that CTA adds the other links'
// contributions in increasing link order, so the sum is atomic-free and
// bit-stable.
#pragma once

#include <cstdint>

namespace attn {

struct PagedParams {
  int Nq, S, H, KVH, G;        // query rows, sequences, heads, KV heads, heads per KV head
  int page_size;               // tokens per page (16)
  int num_pages, max_pages;    // pool pages, page-table row length
  int Dk, Dv, Dp;              // key, value, position dims (Dp = 0 for GQA)
  int causal;
  float scale, scale_log2;
  const int32_t* page_table;   // [S, max_pages]
  const int32_t* seq_len;      // [S]
  const int32_t* q_start;      // [S + 1]
  const int32_t* q_pos;        // [Nq]
  const float* lse;            // [Nq, H] natural log (input) or output of the row-stat kernel
  const float* delta;          // [Nq, H]
  float* lse_out;              // row-stat kernel outputs
  float* delta_out;
  void* dk_pool;               // [slots, KVH, Dk]
  void* dv_pool;               // [slots, KVH, Dv]
  void* dkp_pool;              // [slots, KVH, Dp]
  void* dq;                    // query side: [Nq, H, Dk]
  void* dqp;                   // query side, MLA: [Nq, H, Dp]
  unsigned wrt;
  // workspace (link structure of the pool)
  int32_t* link_count;         // [num_pages]
  int32_t* link_off;           // [num_pages + 1]
  int32_t* link_fill;          // [num_pages]
  int32_t* links;              // [S * max_pages]: link ids s*max_pages+lp grouped by page
  int32_t* heavy;              // [S, ceil(max_pages / 8), KVH]: MLA blocks left to the split kernel (tile count; 0: not flagged)
  uint8_t* listed;             // [num_pages] compact history: 1 = compute and store the page; null = all
  int32_t* order;              // [S] sequences by decreasing length (ties by index): query-side dispatch order
  // MLA history counters, zeroed by the plan kernel: [0, 2) the grid kernel's
  // next unit per part, [2, 4) the split kernel's next item per part, then
  // [part][unit][cluster rank] the chunks of a unit reduced so far
  int32_t* work;               // [kMlaWorkInts]
  float* split_part;           // MLA split chunk partials: part 0 [kMlaSplitSlots][128][256], then part 1 [..][128][320]
  uint32_t* err;
};

// The MLA split kernel cuts a flagged block into chunks when few blocks are
// flagged; at most this many chunk partials are open per part.
constexpr int kMlaSplitSlots = 128;
constexpr int kMlaSplitRanks = 8;  // CTAs of a split cluster
constexpr int kMlaWorkInts = 4 + 2 * kMlaSplitSlots * kMlaSplitRanks;
constexpr size_t kMlaSplitFloats = static_cast<size_t>(kMlaSplitSlots) * 128 * (256 + 320);

// device error codes of the paged prep (OR-ed into the error word)
constexpr uint32_t kErrBadPage = 4u;   // a page-table entry outside [0, num_pages)

__host__ __device__ inline int pages_of(int len, int page_size) { return (len + page_size - 1) / page_size; }

#ifdef __CUDACC__
// Metadata read through clamps, so that malformed sequence lengths or query
// ranges can never index outside the caller's arrays.
__device__ __forceinline__ int seq_len_of(const PagedParams& p, int s) {
  return min(max(p.seq_len[s], 0), p.max_pages * p.page_size);
}
__device__ __forceinline__ int row_begin_of(const PagedParams& p, int s) { return min(max(p.q_start[s], 0), p.Nq); }
__device__ __forceinline__ int row_end_of(const PagedParams& p, int s) {
  return min(max(p.q_start[s + 1], row_begin_of(p, s)), p.Nq);
}
// The idx-th tile of rt query rows, counting the row tiles of the sequences
// in p.order (the longest sequences first, so that the CTAs with the longest
// sweeps start first): its sequence and first row; sq = -1 past the last.
// Called by a whole warp (every lane gets the result): the lanes take 32
// sequences of the order at a time and find the tile's sequence by a prefix
// sum of their tile counts.
__device__ inline void row_tile_at_warp(const PagedParams& p, int idx, int rt, int* sq, int* r0) {
  const int lane = threadIdx.x & 31;
  int base = 0;
  for (int c0 = 0; c0 < p.S; c0 += 32) {  // warp-uniform
    const int k = c0 + lane;
    int s = 0, rb = 0, tiles = 0;
    if (k < p.S) {
      s = p.order[k];
      rb = row_begin_of(p, s);
      tiles = (row_end_of(p, s) - rb + rt - 1) / rt;
    }
    int x = tiles;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    const int excl = base + x - tiles;
    const unsigned hit = __ballot_sync(0xffffffffu, idx >= excl && idx < excl + tiles);
    if (hit) {
      const int l = __ffs(hit) - 1;
      *sq = __shfl_sync(0xffffffffu, s, l);
      *r0 = __shfl_sync(0xffffffffu, rb + (idx - excl) * rt, l);
      return;
    }
    base += __shfl_sync(0xffffffffu, x, 31);
  }
  *sq = -1;
  *r0 = 0;
}
#endif

}  // namespace attn
