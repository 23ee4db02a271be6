// Host-side launchers of the paged kernels (called from paged_api.cu).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "paged_common.cuh"

namespace attn {

// TMA descriptors of one paged call: q/dy (and qp) as 3-D [Nq, H, D] tensors
// addressed (d, h, r), pools as 3-D [slots, KVH, D] tensors addressed (d, g, slot).
struct PagedMaps {
  CUtensorMap q, dy, qp;         // box (64, G, 64/G) for the history kernel
  CUtensorMap q_stats, dy_stats; // box (64, G, 128/G) for the row-statistics kernel
  CUtensorMap k, v, kp;          // box (64, 1, page_size)
};

cudaError_t launch_paged_prep(const PagedParams& p, cudaStream_t s);
// p.order: the sequences by decreasing length (the query-side kernels take
// their row tiles in that order)
cudaError_t launch_paged_seq_order(const PagedParams& p, cudaStream_t s);
// zero the pool rows of pages no link references: every page (list null) or
// the n listed ones (compact history)
cudaError_t launch_paged_zero_unlinked(const PagedParams& p, const int32_t* list, int64_t n, cudaStream_t s);
cudaError_t launch_paged_history(const PagedMaps& m, const PagedParams& p, cudaStream_t s);
cudaError_t launch_paged_row_stats(const PagedMaps& m, const PagedParams& p, cudaStream_t s);
// query side (GQA): row statistics and dQ in one kernel; q_stats/dy_stats maps
cudaError_t launch_paged_query(const PagedMaps& m, const PagedParams& p, cudaStream_t s);
// rows outside every sequence's range: dq (and dqp) = 0, lse = -inf, delta = 0
cudaError_t launch_paged_query_outside(const PagedParams& p, cudaStream_t s);
// MLA (key_dim 512 latent + position_dim 64; the latent is also the value):
// q, qp, dy as [Nq, H, D] addressed (d, h, r) with box (64, G, rows);
// latent and position pools as [slots, KVH, D] with box (64, 1, 16).
struct PagedMlaMaps {
  CUtensorMap q, qp, dy, k, kp;
};
// compact history: p.listed[page] = 1 for the n listed pages (zero otherwise)
cudaError_t launch_paged_listed(const PagedParams& p, const int32_t* pages, int64_t n, cudaStream_t s);
// MLA history on tcgen05 (two CTAs per 128-token block, each accumulating
// half of the dims); maps with 64-column boxes (64/G rows).  Blocks the plan
// flagged (p.heavy, when not null) are left to the split kernel; after_split:
// that kernel was launched just before (the first part then starts as its
// programmatic dependent)
bool mla_tc_supported(const PagedParams& p);
cudaError_t launch_paged_mla_tc(const PagedMlaMaps& m, const PagedParams& p, bool after_split, cudaStream_t s);
// flags the 128-token MLA history blocks whose shared pages carry many link
// tiles (p.heavy [S, ceil(max_pages / 8), KVH]: their tile counts) and zeroes
// the MLA work counters
cudaError_t launch_paged_mla_tc_plan(const PagedParams& p, cudaStream_t s);
// the flagged blocks, by persistent clusters of 8 CTAs on tcgen05, cut into
// chunks when few are flagged (the same maps as launch_paged_mla_tc)
cudaError_t launch_paged_mla_tc_split(const PagedMlaMaps& m, const PagedParams& p, cudaStream_t s);
// MLA row statistics on tcgen05; maps with 128-column boxes (128/G rows)
bool mla_stats_tc_supported(const PagedParams& p);
cudaError_t launch_paged_mla_stats_tc(const PagedMlaMaps& m, const PagedParams& p, cudaStream_t s);
// MLA query side (dQ, dQp) on tcgen05 from lse / delta; maps with 64-column boxes
bool mla_query_tc_supported(const PagedParams& p);
cudaError_t launch_paged_mla_query_tc(const PagedMlaMaps& m, const PagedParams& p, cudaStream_t s);

}  // namespace attn
