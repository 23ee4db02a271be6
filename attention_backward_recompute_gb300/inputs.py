"""Seeded synthetic inputs shared by the tests, the smoke check and the bench.

This module draws random numbers and builds shapes only; it holds none of the
attention arithmetic, so both the CPU oracle and the CUDA path can take their
inputs from it without sharing any of the method.

Generator: numpy's PCG64 (``np.random.default_rng(seed)``), normals from its
``standard_normal``.  Every floating-point tensor is returned as float32 whose
values are exactly representable in the requested storage type: for ``bf16``
the float32 draw is rounded to bfloat16 (round to nearest, ties to even) here,
before either side sees it, so the oracle and the GPU read identical numbers.

Workloads (shapes and value distributions of the five configurations the
attention-backward pages are measured on):

* ``dense_small_f32``    f32, B=1 H=2 Sq=Sk=16 D=16, [B,S,H,D], N(0,1), no mask
* ``dense_f32_causal``   f32, B=2 H=8 Sq=Sk=512 D=64, N(0,1), causal
* ``dense_f32_window``   same, sliding window w=128
* ``dense_bf16_s2048``   bf16, B=4 H=16 Sq=Sk=2048 D=128, N(0,1)*0.5, causal +
                          per-key mask (0 with probability 0.1, else 1) +
                          additive bias [B,H,Sq,Sk] ~ N(0,1) in bf16
* ``dense_bf16_cross``   bf16, B=8 H=16 Sq=256 Sk=4096 D=128, N(0,1)*0.5,
                          causal bottom-right aligned
* paged history: see :func:`paged_case`.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np


def bf16_round(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even); float32 out."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) >> 16) & 0xFFFF
    out = (r << 16).astype(np.uint32).view(np.float32)
    # NaN/inf never occur in these draws; keep them untouched if they did.
    bad = ~np.isfinite(x)
    if bad.any():
        out = out.copy()
        out[bad] = x[bad]
    return out.reshape(x.shape)


def store(x: np.ndarray, dtype: str) -> np.ndarray:
    """Return float32 values representable in ``dtype`` ('f32' or 'bf16')."""
    x = np.asarray(x, dtype=np.float32)
    if dtype == "bf16":
        return bf16_round(x)
    if dtype == "f32":
        return x
    raise ValueError(f"unknown storage dtype {dtype!r}")


def normal(rng: np.random.Generator, shape, scale: float, dtype: str) -> np.ndarray:
    return store(rng.standard_normal(size=shape, dtype=np.float32) * np.float32(scale), dtype)


@dataclasses.dataclass
class DenseCase:
    """One dense attention-backward problem (host arrays, float32 storage)."""
    name: str
    batch: int
    heads: int
    seq_q: int
    seq_k: int
    head_dim: int
    dtype: str                 # 'f32' | 'bf16'
    layout: str                # 'bshd' | 'bhsd'
    causal: bool
    window: int | None
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    dy: np.ndarray
    key_mask: np.ndarray | None   # [B, Sk] float32 or None
    bias: np.ndarray | None       # [B, H, Sq, Sk] float32 (bf16 values) or None
    mask_thr: float = 0.5
    mask_neg: float = -1e9

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)


def dense_inputs(*, name="custom", batch, heads, seq_q, seq_k, head_dim, dtype="bf16",
                 layout="bshd", seed=0, scale=1.0, causal=False, window=None,
                 key_mask_zero_frac=None, bias=False, bias_scale=1.0) -> DenseCase:
    """Draw Q, K, V, dY (and optional key mask / bias) for one dense case.

    Order of draws is fixed: q, k, v, dy, key mask, bias.  The key mask holds
    values in {0, 1} (0 with probability ``key_mask_zero_frac``)."""
    rng = np.random.default_rng(seed)
    if layout == "bshd":
        qs, ks = (batch, seq_q, heads, head_dim), (batch, seq_k, heads, head_dim)
    elif layout == "bhsd":
        qs, ks = (batch, heads, seq_q, head_dim), (batch, heads, seq_k, head_dim)
    else:
        raise ValueError(layout)
    q = normal(rng, qs, scale, dtype)
    k = normal(rng, ks, scale, dtype)
    v = normal(rng, ks, scale, dtype)
    dy = normal(rng, qs, scale, dtype)
    km = None
    if key_mask_zero_frac is not None:
        km = (rng.random(size=(batch, seq_k)) >= key_mask_zero_frac).astype(np.float32)
    b = None
    if bias:
        b = normal(rng, (batch, heads, seq_q, seq_k), bias_scale, dtype)
    return DenseCase(name=name, batch=batch, heads=heads, seq_q=seq_q, seq_k=seq_k,
                     head_dim=head_dim, dtype=dtype, layout=layout, causal=causal,
                     window=window, q=q, k=k, v=v, dy=dy, key_mask=km, bias=b)


def elem_mask_inputs(*, batch, heads, seq_q, seq_k, seed=0, kind="random", masked_frac=0.3, doc_lo=16,
                     doc_hi=160, full_rows=0, full_cols=0) -> np.ndarray:
    """A per-element custom mask [B, H, Sq, Sk] (float32; a pair whose value is
    below 0.5 is masked).

    kind 'random': uniform values in [0, 1) shifted so that a pair is masked
    with probability ``masked_frac``.  kind 'docs': queries and keys are cut
    into documents of lengths drawn uniformly in [doc_lo, doc_hi] (the same
    cut positions for both sides, per batch), and a pair across documents is
    masked (values 0 / 1).  Then ``full_rows`` query rows and ``full_cols``
    key columns per head are masked entirely (value 0)."""
    rng = np.random.default_rng(seed)
    shape = (batch, heads, seq_q, seq_k)
    if kind == "random":
        m = rng.random(size=shape, dtype=np.float64) + (0.5 - masked_frac)
    elif kind == "docs":
        m = np.zeros(shape)
        n = max(seq_q, seq_k)
        for b in range(batch):
            doc = np.empty(n, dtype=np.int64)
            pos, d = 0, 0
            while pos < n:
                ln = int(rng.integers(doc_lo, doc_hi + 1))
                doc[pos:pos + ln] = d
                pos, d = pos + ln, d + 1
            m[b] = (doc[:seq_q, None] == doc[None, :seq_k])
    else:
        raise ValueError(kind)
    for b in range(batch):
        for h in range(heads):
            if full_rows and seq_q:
                m[b, h, rng.choice(seq_q, size=min(full_rows, seq_q), replace=False), :] = 0.0
            if full_cols and seq_k:
                m[b, h, :, rng.choice(seq_k, size=min(full_cols, seq_k), replace=False)] = 0.0
    return m.astype(np.float32)


# The five measured configurations (dense part), by name.  Seeds follow the
# configuration order (1..5).
DENSE_CONFIGS = {
    "dense_small_f32": dict(batch=1, heads=2, seq_q=16, seq_k=16, head_dim=16, dtype="f32",
                            seed=1, scale=1.0),
    "dense_f32_causal": dict(batch=2, heads=8, seq_q=512, seq_k=512, head_dim=64, dtype="f32",
                             seed=2, scale=1.0, causal=True),
    "dense_f32_window": dict(batch=2, heads=8, seq_q=512, seq_k=512, head_dim=64, dtype="f32",
                             seed=2, scale=1.0, window=128),
    "dense_bf16_s2048": dict(batch=4, heads=16, seq_q=2048, seq_k=2048, head_dim=128,
                             dtype="bf16", seed=3, scale=0.5, causal=True,
                             key_mask_zero_frac=0.1, bias=True),
    "dense_bf16_cross": dict(batch=8, heads=16, seq_q=256, seq_k=4096, head_dim=128,
                             dtype="bf16", seed=4, scale=0.5, causal=True),
}


def dense_config(name: str, **overrides) -> DenseCase:
    kw = dict(DENSE_CONFIGS[name])
    kw.update(overrides)
    return dense_inputs(name=name, **kw)


def p1_hash_values(n: int, seed: int) -> np.ndarray:
    """Deterministic inputs of the rlx-cpu fused-backward unit test
    (rlx-cpu attention_bwd.rs, test ``all_matches_three_separate``):
    x_i = ((i * 2654435761 + seed) mod 1000) / 500 - 1, as float32."""
    i = np.arange(n, dtype=np.uint64)
    r = (i * np.uint64(2654435761) + np.uint64(seed)) % np.uint64(1000)
    return (r.astype(np.float32) / np.float32(500.0)) - np.float32(1.0)


# ----------------------------------------------------------------------------
# Paged KV history
# ----------------------------------------------------------------------------

@dataclasses.dataclass
class PagedCase:
    """Paged-KV history backward problem (host arrays).

    Pools are indexed by physical slot = page * page_size + offset and hold
    ``kv_heads`` rows per slot: pool[slot, g, :].  Slots that no sequence owns
    and tail slots past a sequence's length are filled with NaN so that any
    read of them poisons the result."""
    name: str
    heads: int
    kv_heads: int
    page_size: int
    num_pages: int
    key_dim: int
    value_dim: int
    position_dim: int          # 0 for GQA, >0 for MLA (V is the latent key)
    dtype: str
    causal: bool
    seq_len: np.ndarray        # [S] int32
    q_start: np.ndarray        # [S+1] int32 (packed query rows, sequence-major)
    q_pos: np.ndarray          # [Nq] int32 absolute position of each query row
    page_table: np.ndarray     # [S, max_pages] int32 (-1 where unused)
    q: np.ndarray              # [Nq, H, key_dim]
    qp: np.ndarray | None      # [Nq, H, position_dim]
    dy: np.ndarray             # [Nq, H, value_dim]
    k_pool: np.ndarray         # [slots, kv_heads, key_dim]
    v_pool: np.ndarray | None  # [slots, kv_heads, value_dim] (None for MLA)
    kp_pool: np.ndarray | None # [slots, kv_heads, position_dim]

    @property
    def num_seqs(self) -> int:
        return int(self.seq_len.shape[0])

    @property
    def num_queries(self) -> int:
        return int(self.q_pos.shape[0])

    @property
    def mla(self) -> bool:
        return self.position_dim > 0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.key_dim + self.position_dim)


def paged_case(*, name="paged", seed=5, num_seqs=64, len_lo=128, len_hi=4096, queries_per_seq=64,
               heads=32, kv_heads=8, page_size=16, key_dim=128, value_dim=128, position_dim=0,
               pool_factor=1.25, dtype="bf16", scale=0.5, causal=True,
               shared_prefix_pages=0) -> PagedCase:
    """Draw a paged history problem.

    Sequence lengths ~ U[len_lo, len_hi] (integers, inclusive); each sequence's
    queries are its last ``queries_per_seq`` tokens (positions len-n .. len-1,
    packed sequence-major).  The pool holds ceil(pool_factor * needed) pages;
    logical pages map to a seeded random permutation of the pool.  With
    ``shared_prefix_pages = p > 0`` every sequence's first p logical pages map
    to the same physical pages as sequence 0's (prefix sharing); those pages
    then carry one link per sequence."""
    rng = np.random.default_rng(seed)
    lens = rng.integers(len_lo, len_hi, size=num_seqs, endpoint=True).astype(np.int32)
    if shared_prefix_pages:
        lens = np.maximum(lens, shared_prefix_pages * page_size + 1).astype(np.int32)
    pages_per_seq = (lens + page_size - 1) // page_size
    own = pages_per_seq.copy()
    if shared_prefix_pages:
        own[1:] -= shared_prefix_pages
    needed = int(own.sum())
    num_pages = int(math.ceil(pool_factor * needed))
    perm = rng.permutation(num_pages).astype(np.int32)
    max_pages = int(pages_per_seq.max())
    table = np.full((num_seqs, max_pages), -1, dtype=np.int32)
    cursor = 0
    for s in range(num_seqs):
        start = 0
        if shared_prefix_pages and s > 0:
            table[s, :shared_prefix_pages] = table[0, :shared_prefix_pages]
            start = shared_prefix_pages
        n = int(pages_per_seq[s]) - start
        table[s, start:start + n] = perm[cursor:cursor + n]
        cursor += n
    nq = np.minimum(lens, queries_per_seq).astype(np.int32)
    q_start = np.zeros(num_seqs + 1, dtype=np.int32)
    q_start[1:] = np.cumsum(nq)
    q_pos = np.concatenate([np.arange(L - n, L, dtype=np.int32) for L, n in zip(lens, nq)])
    Nq = int(q_start[-1])
    slots = num_pages * page_size
    q = normal(rng, (Nq, heads, key_dim), scale, dtype)
    qp = normal(rng, (Nq, heads, position_dim), scale, dtype) if position_dim else None
    dy = normal(rng, (Nq, heads, value_dim), scale, dtype)
    k_pool = normal(rng, (slots, kv_heads, key_dim), scale, dtype)
    v_pool = normal(rng, (slots, kv_heads, value_dim), scale, dtype) if not position_dim else None
    kp_pool = normal(rng, (slots, kv_heads, position_dim), scale, dtype) if position_dim else None
    # Poison every slot that holds no valid token.
    valid = np.zeros(slots, dtype=bool)
    for s in range(num_seqs):
        for t in range(int(lens[s])):
            valid[int(table[s, t // page_size]) * page_size + t % page_size] = True
    for pool in (k_pool, v_pool, kp_pool):
        if pool is not None:
            pool[~valid] = np.nan
    return PagedCase(name=name, heads=heads, kv_heads=kv_heads, page_size=page_size,
                     num_pages=num_pages, key_dim=key_dim, value_dim=value_dim,
                     position_dim=position_dim, dtype=dtype, causal=causal, seq_len=lens,
                     q_start=q_start, q_pos=q_pos, page_table=table, q=q, qp=qp, dy=dy,
                     k_pool=k_pool, v_pool=v_pool, kp_pool=kp_pool)


PAGED_CONFIGS = {
    "paged_gqa": dict(seed=5, heads=32, kv_heads=8, key_dim=128, value_dim=128, position_dim=0),
    "paged_mla": dict(seed=5, heads=32, kv_heads=1, key_dim=512, value_dim=512, position_dim=64),
}


def paged_config(name: str, **overrides) -> PagedCase:
    kw = dict(PAGED_CONFIGS[name])
    kw.update(overrides)
    return paged_case(name=name, **kw)
