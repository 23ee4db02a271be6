/*
 * attn_bwd.h -- C ABI of libattnbwd, an sm_103a (GB300) library for the
 * backward pass of scaled dot-product attention with recomputed scores and
 * softmax, dense and over a paged KV history.
 *
 * What is computed (dense), per batch b and head h, following rlx-cpu
 * src/attention_bwd.rs (fn backward_dense_head_all, fn apply_synthetic_mask)
 * and rlx-wgpu src/kernels/attention_bwd.wgsl (fn mask_score):
 *
 *   S   = scale * Q K^T                                    [Sq, Sk]
 *   S  += bias[b,h]                          (ATTN_MASK_BIAS)
 *   S[:, k] = mask_neg where key_mask[b,k] < mask_thr      (ATTN_MASK_KEY)
 *   structural masks, bottom-right aligned, q_off = max(Sk - Sq, 0) (0 with
 *   ATTN_MASK_TOP_LEFT),
 *   abs_q = q_off + q:   causal hides k > abs_q;  window w hides
 *   k < abs_q - w (saturating at 0) or k > abs_q.  Hidden entries get P = 0.
 *   P   = softmax over the visible keys of each row        (a row with no
 *                                                          visible key: P = 0)
 *   dV  = P^T dY
 *   dP  = dY V^T
 *   dS  = P * (dP - rowsum(P * dP)) * scale
 *   dQ  = dS K
 *   dK  = dS^T Q
 *
 * Paged (ruDNN src/paged_attention/ordered_kernel.rs, fn history_backward):
 * the same backward for packed query rows against a KV history stored in
 * pages of a pool, producing dK, dV (GQA) or dK_latent, dKp (MLA) for every
 * pool row with no floating-point atomics and a fixed summation order.
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers on the current CUDA device,
 *     owned by the caller; the library never allocates on the call path.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls are
 *     asynchronous on that stream; only attn_check_device_error synchronises.
 *   - Every call validates its arguments first and returns a status; nothing
 *     is launched when the status is not ATTN_OK.  There is no silent no-op
 *     and no CPU fallback: an unsupported case returns ATTN_ERR_UNSUPPORTED.
 *   - attn_last_error() returns a human-readable reason for the last non-OK
 *     status returned on the calling host thread.
 */
#ifndef ATTN_BWD_H
#define ATTN_BWD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define ATTN_API __attribute__((visibility("default")))
#else
#define ATTN_API
#endif

typedef int32_t attn_status_t;
#define ATTN_OK 0
#define ATTN_ERR_INVALID_ARG 1 /* null pointer, negative size, bad enum, ... */
#define ATTN_ERR_UNSUPPORTED 2 /* valid request the library does not implement */
#define ATTN_ERR_ALIAS 3       /* an output overlaps an input or another output */
#define ATTN_ERR_WORKSPACE 4   /* workspace missing, too small or misaligned */
#define ATTN_ERR_CUDA 5        /* a CUDA runtime/driver call or launch failed */
#define ATTN_ERR_TIMEOUT 6     /* a device-side bounded wait expired */

/* Storage types of q, k, v, dy, o, bias and of the gradients. */
#define ATTN_DTYPE_F32 0  /* fp32 in and out; every operand split into hi + lo bf16 and each
                            product taken as hi*hi + hi*lo + lo*hi on bf16 tensor cores */
#define ATTN_DTYPE_BF16 1 /* bf16 in and out; bf16 tensor cores, fp32 accumulation */

/* Dense layouts (rlx-cpu attention_bwd.rs, fn attention_backward: `bhsd`). */
#define ATTN_LAYOUT_BSHD 0 /* [B, S, H, D], D contiguous */
#define ATTN_LAYOUT_BHSD 1 /* [B, H, S, D], D contiguous */

/* Dense mask flags (combinable). */
#define ATTN_MASK_CAUSAL 1u /* hide k > abs_q */
#define ATTN_MASK_WINDOW 2u /* hide k < abs_q - window and k > abs_q */
#define ATTN_MASK_KEY 4u    /* custom per-key mask key_mask[B, Sk] (fp32) */
#define ATTN_MASK_BIAS 8u   /* additive bias[B, H, Sq, Sk] in the storage type */
/* align the causal and window masks top-left instead: abs_q = q (q_off = 0),
 * as rlx-wgpu attention_bwd.wgsl mask_score does (causal hides k > q) */
#define ATTN_MASK_TOP_LEFT 16u
/* per-element custom mask elem_mask[B, H, Sq, Sk] (fp32, contiguous): the
 * score of a pair whose value is < mask_thr is replaced by mask_neg, as
 * rlx-wgpu attention_bwd.wgsl mask_score does for its mask kind 2; combines
 * with ATTN_MASK_KEY.  Taken by attn_bwd_dense_strided (bf16 storage);
 * attn_bwd_dense has no argument for it (ATTN_ERR_INVALID_ARG) and the
 * forward export returns ATTN_ERR_UNSUPPORTED */
#define ATTN_MASK_ELEM 32u

/* Gradient selection (enum order of the pages: Query = 0, Key = 1, Value = 2). */
#define ATTN_WRT_DQ 1u
#define ATTN_WRT_DK 2u
#define ATTN_WRT_DV 4u
#define ATTN_WRT_DKP 8u /* paged MLA: gradient of the position keys */

typedef struct attn_dense_desc {
  int64_t batch;      /* B  >= 0 */
  int64_t heads;      /* H  >= 0 */
  int64_t seq_q;      /* Sq >= 0 */
  int64_t seq_k;      /* Sk >= 0 */
  int64_t head_dim;   /* D: 8, 16, 32, 64 or 128 for bf16; 8, 16, 32 or 64 for fp32 */
  int32_t dtype;      /* ATTN_DTYPE_* */
  int32_t layout;     /* ATTN_LAYOUT_* */
  uint32_t mask_flags;/* OR of ATTN_MASK_* */
  int32_t window;     /* window w >= 0 when ATTN_MASK_WINDOW is set */
  float mask_thr;     /* key masked when key_mask[b,k] < mask_thr (default 0.5) */
  float mask_neg;     /* masked score value, finite and < 0 (default -1e9) */
  float scale;        /* softmax scale; 0 means 1/sqrt(head_dim) */
  uint32_t options;   /* OR of ATTN_OPT_* (0: none) */
} attn_dense_desc;

/*
 * Backward option: store dS once instead of recomputing it for dQ.  The dK/dV
 * kernel writes every dS tile it forms (bf16) to the workspace and dQ is one
 * product, dQ = scale * dS K, over those tiles: 14 * D flops per visible pair
 * instead of 18 * D, for a workspace larger by
 * 16384 * batch * heads * ceil(seq_k / 128) * ceil(seq_q / 64) bytes
 * (attn_bwd_dense_workspace_bytes counts it).  Results stay deterministic:
 * dK and dV are bit-identical to the call without the option; dQ differs
 * only by rounding (dS enters it as the same bf16 values the dK product
 * uses).  bf16 storage only (fp32: ATTN_ERR_UNSUPPORTED); ignored by the
 * forward export; refused by attn_bwd_dense_noalloc.
 */
#define ATTN_OPT_STORE_DS 1u

/* Fill `d` with defaults: zeros, BSHD, bf16, mask_thr 0.5, mask_neg -1e9. */
ATTN_API void attn_dense_desc_init(attn_dense_desc* d);

/* Bytes of workspace attn_bwd_dense needs for `d` (row statistics: three fp32
 * values per (b, h, query row), each array 256-byte aligned; plus the split
 * copies of fp32 storage, the bits of a per-element mask and the stored dS of
 * ATTN_OPT_STORE_DS when those apply).  Returns 0 for an invalid descriptor. */
ATTN_API size_t attn_bwd_dense_workspace_bytes(const attn_dense_desc* d);

/*
 * Dense backward: dQ, dK, dV from Q, K, V, dY (and optionally O, LSE).
 *
 *   q, dy   [B,Sq,H,D] or [B,H,Sq,D] (layout), storage type `dtype`
 *   k, v    [B,Sk,H,D] or [B,H,Sk,D]
 *   key_mask fp32 [B, Sk], required iff ATTN_MASK_KEY (else must be NULL)
 *   bias    [B, H, Sq, Sk] in `dtype`, required iff ATTN_MASK_BIAS (else NULL);
 *           Sk * element size must be a multiple of 16 bytes
 *   o, lse  optional forward output [layout of q] and fp32 log-sum-exp
 *           [B, H, Sq] (natural log).  Both NULL: the library recomputes the
 *           row statistics with a forward sweep (self-contained mode).  Both
 *           given: only rowsum(dY * O) is computed.  One without the other is
 *           ATTN_ERR_INVALID_ARG.
 *   dq, dk, dv outputs in the layout of q / k / v; a gradient not selected in
 *           `wrt_mask` is not written and its pointer may be NULL.  Selected
 *           gradients are bit-identical to those of a call with all three.
 *   workspace device memory of at least attn_bwd_dense_workspace_bytes(d),
 *           256-byte aligned, not shared with a concurrently running call.
 *
 * All tensor pointers must be 16-byte aligned.  No output may overlap any
 * input, the workspace or another output (ATTN_ERR_ALIAS); in particular the
 * outputs may not alias v (the hazard rlx-cpu attention_backward_all guards).
 * A zero-size dimension writes zeros to the selected gradients that have
 * elements and returns ATTN_OK.
 */
ATTN_API attn_status_t attn_bwd_dense(const attn_dense_desc* d, const void* q, const void* k, const void* v,
                                      const void* dy, const float* key_mask, const void* bias, const void* o,
                                      const float* lse, void* dq, void* dk, void* dv, unsigned wrt_mask,
                                      void* workspace, size_t workspace_bytes, void* stream);

/*
 * Dense backward that allocates nothing and takes no workspace.  (The pages
 * have no counterpart: this entry point exists for callers of this library.)
 *
 * Some callers cannot call cudaMalloc: plugin code running inside a host
 * framework whose device memory belongs to that framework's allocator, or a
 * serving loop that forbids allocation on its hot path.  For them the row
 * statistics live in a scratch array owned by the library: a file-scope
 * device array of ATTN_NOALLOC_MAX_ROWS * 12 bytes (about 12 MiB), which every
 * GPU that loads the library holds until the process exits.  The caller still
 * passes every input and output; arguments, layouts and results are those of
 * attn_bwd_dense, whose outputs this call reproduces.
 *
 *   - batch * heads * seq_q above ATTN_NOALLOC_MAX_ROWS is rejected with
 *     ATTN_ERR_UNSUPPORTED (use attn_bwd_dense with a workspace instead), and
 *     so are fp32 storage (its split input copies do not fit the scratch),
 *     ATTN_OPT_STORE_DS (the stored dS tiles do not fit either) and
 *     ATTN_MASK_ELEM (the packed mask bits do not fit either).
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress; it allocates nothing) with that device current;
 *     make that first call before any stream capture.  The address is cached
 *     for the life of the process: after cudaDeviceReset on a device, do not
 *     call this entry point on that device again.
 *   - All calls share the one array and it keeps the last call's contents.
 *     Calls whose kernels overlap on the GPU (other streams, other host
 *     threads) race on it: serialise them.
 *   - No cudaMalloc, cudaFree or allocating library routine is called.
 */
#define ATTN_NOALLOC_MAX_ROWS 1048576
ATTN_API attn_status_t attn_bwd_dense_noalloc(const attn_dense_desc* d, const void* q, const void* k, const void* v,
                                              const void* dy, const float* key_mask, const void* bias,
                                              const void* o, const float* lse, void* dq, void* dk, void* dv,
                                              unsigned wrt_mask, void* stream);

/*
 * Paged KV history.
 *
 * Pools hold `num_pages * page_size` slots; slot = page * page_size + offset,
 * and pool row (slot, g) for KV head g is at element offset
 * (slot * kv_heads + g) * dim.  Logical page p of sequence s lives in physical
 * page page_table[s * max_pages_per_seq + p].  A physical page may be mapped
 * by several (sequence, logical page) links (prefix sharing); its gradient is
 * then the sum over its links, taken in increasing (sequence, logical page)
 * order.
 *
 * seq_meta is one int32 array:  seq_len[num_seqs] | q_start[num_seqs + 1] |
 * q_pos[num_queries].  Query rows of sequence s are rows q_start[s] ..
 * q_start[s+1]-1 of q/dy (packed, sequence-major); q_pos[r] is the absolute
 * position of row r.  With `causal`, row r sees history tokens t <= q_pos[r].
 *
 * GQA (position_dim == 0): query head h reads KV head h / (heads / kv_heads).
 * MLA (position_dim > 0): the score is q.k_latent + qp.k_position, the latent
 * is both key and value (value_dim == key_dim, v_pool unused), and the
 * gradients are dK_latent = dS^T Q + P^T dY and dKp = dS^T Qp.
 */
typedef struct attn_paged_desc {
  int64_t num_queries;       /* Nq: packed query rows */
  int64_t num_seqs;          /* S */
  int64_t heads;             /* query heads H */
  int64_t kv_heads;          /* KV heads; H % kv_heads == 0 */
  int64_t page_size;         /* tokens per page: 16 */
  int64_t num_pages;         /* physical pages in the pool */
  int64_t max_pages_per_seq; /* row length of page_table */
  int64_t key_dim;           /* 128 (GQA) or 512 (MLA latent) */
  int64_t value_dim;         /* == key_dim */
  int64_t position_dim;      /* 0 (GQA) or 64 (MLA) */
  int32_t dtype;             /* ATTN_DTYPE_BF16 */
  int32_t causal;            /* 0 or 1 */
  float scale;               /* 0 means 1/sqrt(key_dim + position_dim) */
  int32_t reserved;          /* must be 0 */
} attn_paged_desc;

/* Bytes of workspace attn_bwd_paged / attn_paged_row_stats need (the link
 * structure of the pool and counters; for MLA also 36 MiB of fp32 partial
 * sums of the shared-page blocks that are cut into chunks). */
ATTN_API size_t attn_bwd_paged_workspace_bytes(const attn_paged_desc* d);

/*
 * Paged history backward (gradients of the pool rows).
 *   q [Nq, H, key_dim], qp [Nq, H, position_dim] (MLA, else NULL),
 *   dy [Nq, H, value_dim]; k_pool, v_pool (GQA), kp_pool (MLA) as above;
 *   page_table int32 [num_seqs, max_pages_per_seq]; seq_meta as above;
 *   lse, delta fp32 [Nq, H]: row statistics (natural-log LSE and
 *   rowsum(P * dP)), e.g. from attn_paged_row_stats.  lse = -inf marks a row
 *   with no visible token; it contributes nothing.
 *   dk_pool, dv_pool (GQA) / dk_pool, dkp_pool (MLA): outputs shaped like the
 *   pools.  EVERY pool row is written exactly once: rows of slots that hold no
 *   valid token (unreferenced pages, tail slots past a sequence's length) get
 *   zero, so no clearing pass is needed.  wrt_mask selects among ATTN_WRT_DK,
 *   ATTN_WRT_DV (GQA) and ATTN_WRT_DKP (MLA).
 * The result is bit-identical from run to run: no floating-point atomics,
 * every sum in a fixed order (integer counters only hand out work).
 */
ATTN_API attn_status_t attn_bwd_paged(const attn_paged_desc* d, const void* q, const void* qp, const void* k_pool,
                                      const void* v_pool, const void* kp_pool, const void* dy,
                                      const int32_t* page_table, const int32_t* seq_meta, const float* lse,
                                      const float* delta, void* dk_pool, void* dv_pool, void* dkp_pool,
                                      unsigned wrt_mask, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Compact history: attn_bwd_paged restricted to the physical pages listed in
 * history_pages (int32 [num_history_pages], any order, repeats allowed), as
 * ruDNN src/paged_attention/ordered_kernel.rs does when its compact_history
 * flag maps the launch grid through a history_pages list.  Every pool row of
 * a listed page is written exactly once, with the same values as the full
 * call (zeros for slots no valid token owns; bit-identical except in MLA
 * blocks split over a cluster, whose partial sums may group differently when
 * pages of the block are not listed); rows of pages not listed are
 * not written, and the work of the pages not listed (their link passes and
 * the zero store of unreferenced ones) is skipped.  An entry outside
 * [0, num_pages) is skipped and reported by attn_check_device_error
 * (ATTN_ERR_CUDA).  num_history_pages = 0 writes nothing; a negative count
 * means every page (attn_bwd_paged).  history_pages is read on the device
 * (4-byte aligned) and may not overlap an output.  The page map lives in the
 * workspace (attn_bwd_paged_workspace_bytes covers it).
 */
ATTN_API attn_status_t attn_bwd_paged_compact(const attn_paged_desc* d, const void* q, const void* qp,
                                              const void* k_pool, const void* v_pool, const void* kp_pool,
                                              const void* dy, const int32_t* page_table, const int32_t* seq_meta,
                                              const float* lse, const float* delta, const int32_t* history_pages,
                                              int64_t num_history_pages, void* dk_pool, void* dv_pool,
                                              void* dkp_pool, unsigned wrt_mask, void* workspace,
                                              size_t workspace_bytes, void* stream);

/*
 * Row statistics for the paged path by a forward sweep over each sequence's
 * pages: lse[r, h] = log sum_t exp(s_rt) over visible tokens (-inf if none)
 * and delta[r, h] = rowsum(P * dP) = dY . O.  Same arguments as
 * attn_bwd_paged; lse and delta are fp32 [Nq, H] outputs.  The workspace
 * (as for attn_bwd_paged, else ATTN_ERR_WORKSPACE) holds the order in which
 * the row tiles are dispatched (longest sequences first).
 */
ATTN_API attn_status_t attn_paged_row_stats(const attn_paged_desc* d, const void* q, const void* qp,
                                            const void* k_pool, const void* v_pool, const void* kp_pool,
                                            const void* dy, const int32_t* page_table, const int32_t* seq_meta,
                                            float* lse, float* delta, void* workspace, size_t workspace_bytes,
                                            void* stream);

/*
 * General strides.  Element strides of the batch, sequence and head
 * dimensions of one [B, S, H, D] tensor (any order in memory); its head_dim
 * dimension is contiguous.  Strides are non-negative multiples of 16 bytes;
 * an output's strides must not make two (batch, seq, head) rows share bytes
 * (an input's may, e.g. a key tensor shared by all heads with head stride 0).
 * rlx-wgpu attention_bwd.wgsl passes per-tensor batch, head and sequence
 * strides in its Params block; this is the same freedom.
 */
typedef struct attn_strides3 {
  int64_t batch, seq, head;
} attn_strides3;

typedef struct attn_dense_strides {
  attn_strides3 q, k, v, dy, o, dq, dk, dv;  /* o: the O input (backward) or output (forward) */
} attn_dense_strides;

/* The strides of the descriptor's layout (what attn_bwd_dense uses). */
ATTN_API void attn_dense_strides_from_layout(const attn_dense_desc* d, attn_dense_strides* st);

/*
 * attn_bwd_dense and attn_fwd_dense with explicit strides (the descriptor's
 * layout field is then ignored for addressing; st NULL means the layout's
 * strides).  attn_bwd_dense_strided also takes the per-element mask
 * (ATTN_MASK_ELEM; NULL otherwise): bf16 storage only, and the workspace
 * then also holds the mask as bits (attn_bwd_dense_workspace_bytes counts
 * it when the flag is set).  fp32 storage needs q, k, v
 * and dy in the descriptor's layout (ATTN_ERR_UNSUPPORTED otherwise); bf16
 * takes any valid strides.  Results are bit-identical to the layout call on
 * the same values.
 */
ATTN_API attn_status_t attn_bwd_dense_strided(const attn_dense_desc* d, const attn_dense_strides* st, const void* q,
                                              const void* k, const void* v, const void* dy, const float* key_mask,
                                              const float* elem_mask, const void* bias, const void* o,
                                              const float* lse, void* dq, void* dk, void* dv, unsigned wrt_mask,
                                              void* workspace, size_t workspace_bytes, void* stream);
ATTN_API attn_status_t attn_fwd_dense_strided(const attn_dense_desc* d, const attn_dense_strides* st, const void* q,
                                              const void* k, const void* v, const float* key_mask, const void* bias,
                                              void* o, float* lse, void* workspace, size_t workspace_bytes,
                                              void* stream);

/*
 * Dense forward export: O and the LSE of the same attention the backward
 * differentiates (same descriptor, masks and bias), by the forward sweep of
 * the backward's row-statistics prologue (rlx-cpu src/attention_bwd.rs,
 * backward_dense_head_all: scores, masks and max-subtracted softmax; O = P V).
 *   q [.., Sq, .., D], k, v [.., Sk, .., D] in the descriptor's layout and
 *   dtype; key_mask / bias as for attn_bwd_dense (required iff flagged);
 *   o: output shaped and typed like q, O = softmax(S) V (0 for a row with no
 *   visible key);
 *   lse: fp32 [B, H, Sq] output, natural-log log-sum-exp of the row's scores
 *   (-inf for a row with no visible key).
 * The pair (o, lse) is what attn_bwd_dense takes in its O-and-LSE mode.
 * Workspace as attn_bwd_dense (attn_bwd_dense_workspace_bytes).  Errors as
 * attn_bwd_dense; an output overlapping an input or the workspace gives
 * ATTN_ERR_ALIAS.  Asynchronous on `stream`.
 */
ATTN_API attn_status_t attn_fwd_dense(const attn_dense_desc* d, const void* q, const void* k, const void* v,
                                      const float* key_mask, const void* bias, void* o, float* lse, void* workspace,
                                      size_t workspace_bytes, void* stream);

/*
 * Query side of the paged backward: the row statistics and the query
 * gradient of every packed query row in one call.  ruDNN
 * src/paged_attention/ordered_kernel.rs (history_backward) reads per (row,
 * head) statistics "computed once by the query kernel"; this is that kernel,
 * with dQ added.  Same arguments as attn_paged_row_stats, plus
 *   dq [Nq, H, key_dim] (storage dtype): output,
 *   dq[r, h] = scale * sum_t dS_rt k_t over the row's visible tokens t, with
 *   dS = P (dP - delta) and P, dP, delta as in attn_bwd_paged;
 *   dqp [Nq, H, position_dim] (MLA): output of the position part.
 * lse and delta (fp32 [Nq, H]) are written as by attn_paged_row_stats.  Every
 * row is written exactly once: a row with no visible token, or outside every
 * sequence's query range, gets dq = 0, lse = -inf and delta = 0.  Tokens are
 * visited in a fixed order, so the result is bit-identical from run to run.
 * MLA (position_dim > 0) needs heads / kv_heads dividing 64 and page size 16
 * (else ATTN_ERR_UNSUPPORTED); qp, kp_pool and dqp are then required.
 * The workspace is that of attn_bwd_paged (at least
 * attn_bwd_paged_workspace_bytes(d) bytes, 256-byte aligned, else
 * ATTN_ERR_WORKSPACE): it holds the order in which the row tiles are
 * dispatched (longest sequences first).
 */
ATTN_API attn_status_t attn_bwd_paged_query(const attn_paged_desc* d, const void* q, const void* qp,
                                            const void* k_pool, const void* v_pool, const void* kp_pool,
                                            const void* dy, const int32_t* page_table, const int32_t* seq_meta,
                                            float* lse, float* delta, void* dq, void* dqp, void* workspace,
                                            size_t workspace_bytes, void* stream);

/* Reason for the last non-OK status on this host thread ("" if none). */
ATTN_API const char* attn_last_error(void);

/* Name of a status code. */
ATTN_API const char* attn_status_string(attn_status_t s);

/*
 * Synchronise `stream` and report device-side errors raised since the last
 * check by kernels of this library on the current device: ATTN_ERR_TIMEOUT if
 * a bounded wait expired (the kernel stopped early and its outputs are
 * invalid), ATTN_ERR_CUDA if the stream itself failed or a kernel raised
 * another device error (the message gives the error word: 0x4 a page-table
 * entry outside [0, num_pages), skipped; 0x8 dynamic shared memory not at the
 * 1024-byte alignment a kernel's layout needs, the kernel did nothing), else
 * ATTN_OK.  Clears the device error word.
 */
ATTN_API attn_status_t attn_check_device_error(void* stream);

/*
 * Self-test of the failure detection above (no counterpart on the pages: it
 * checks this library's own bounded waits).  Launches on `stream` one warp
 * that waits on an mbarrier nothing ever arrives on; the wait gives up after
 * the library's bounded-wait limit (one second), sets the device error word
 * and the kernel returns.  A following attn_check_device_error(stream) must
 * report ATTN_ERR_TIMEOUT (and clear the word); the CUDA context stays usable.
 * Returns ATTN_ERR_CUDA if the launch fails, else ATTN_OK.
 */
ATTN_API attn_status_t attn_selftest_wait_timeout(void* stream);

/*
 * Per-kernel timing hook.  When `events` is non-NULL, the next dense or paged
 * call made on this host thread records events[0] on its stream before its
 * first kernel and events[i] after its i-th kernel (events are cudaEvent_t
 * handles created by the caller; `count` must cover every kernel of the call
 * plus one, else the call records nothing).  The hook applies to ONE call and
 * is then cleared.  The dense call launches, in order: (ATTN_MASK_ELEM only)
 * the kernel that packs the mask into row and column bits; (fp32 storage
 * only) one kernel that splits q, dy, k and v into bf16 hi + lo; the
 * row-statistics prologue (the delta-only kernel when O and LSE are given);
 * the dK/dV kernel (if dK or dV is requested, or dS is stored for dQ); the dQ
 * kernel (if dQ is requested).  The
 * paged backward launches its link preparation, the zero store of unlinked
 * pages and the history kernel (MLA: a plan kernel that flags the blocks whose
 * shared pages carry many links, the cluster-split kernel of those blocks,
 * then the history kernel of the others; the compact call marks its page list
 * before events[0]); the paged row statistics one kernel.
 */
ATTN_API void attn_set_timing_events(void* const* events, int count);

/* Library version, major * 10000 + minor * 100 + patch. */
ATTN_API int attn_version(void);

#ifdef __cplusplus
} /* extern "C" */
#endif

#endif /* ATTN_BWD_H */
