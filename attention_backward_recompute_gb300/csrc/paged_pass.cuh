// Pass structure of a paged history block, shared by the GQA and MLA
// history kernels.
//
// A CTA owns 128 consecutive history tokens (eight 16-token pages) of one
// sequence and one KV head.  It runs passes: the owning sequence's own rows
// first, then, for link index li = 1, 2, ..., the li-th links of the pages it
// stores (ruDNN src/paged_attention/ordered_kernel.rs, history_backward:
// every link of a physical page contributes, in link order, to the one owner
// that stores it).
#pragma once

#include "paged_common.cuh"

namespace attn {

struct PageInfo {
  int phys[8];    // physical page (or -1)
  int off[8];     // first index of the page's link segment
  int cnt[8];     // links of the page
  int store[8];   // this CTA stores the page
};

// One pass = one (sequence, token mapping, live row range); the passes of a CTA
// are enumerated identically by every role.  After the own pass come, for link
// index li = 1, 2, ..., the li-th links of the pages this CTA stores; a run of
// consecutive stored pages whose li-th links are consecutive logical pages of
// one sequence (a shared prefix) is one pass with all their rows live.  Every
// page still sees its links in increasing order.
struct PassIter {
  const PagedParams* p;
  const PageInfo* pi;
  int s0, tb;
  int j, jn, li, lmax;               // j = -1: own pass; else pages [j, jn) at link index li
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
  // advance to the next pass that has at least one tile; false when done
  __device__ bool next_pass(int rt) {
    while (true) {
      if (j < 0) {
        j = 0;
        li = 1;
      } else {
        j = jn;
      }
      while (true) {
        while (j < 8 && !(pi->store[j] && li < pi->cnt[j])) ++j;
        if (j < 8) break;
        if (++li >= lmax) return false;
        j = 0;
      }
      const int link = p->links[pi->off[j] + li];
      const int s2 = link / p->max_pages, lp2 = link - s2 * p->max_pages;
      jn = j + 1;
      while (jn < 8 && pi->store[jn] && li < pi->cnt[jn] && lp2 + (jn - j) < p->max_pages &&
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
    for (int k = 0; k < 8; ++k)
      if (pi->store[k] && pi->cnt[k] > lmax) lmax = pi->cnt[k];
    load(s0, tb * 128, 0, 128, rt);
    if (ntiles > 0) return true;
    return next_pass(rt);
  }
  __device__ bool advance(int rt) {
    if (++tile < ntiles) return true;
    return next_pass(rt);
  }
};


// Page j of token block tb of sequence s0 (npg pages in the sequence):
// physical page, link segment, and whether this block stores the page (its
// first link is this one and, in compact history, it is listed).  Returns
// whether the block stores it.
__device__ inline int fill_page_entry(const PagedParams& p, int s0, int tb, int npg, int j, PageInfo* pi) {
  const int lp = tb * 8 + j;
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
  return st;
}

// The eight pages of the block (see fill_page_entry); returns whether the
// block stores any page.
__device__ inline int fill_page_info(const PagedParams& p, int s0, int tb, int npg, PageInfo* pi) {
  int any = 0;
  for (int j = 0; j < 8; ++j) any |= fill_page_entry(p, s0, tb, npg, j, pi);
  return any;
}

}  // namespace attn
