"""Paged-KV history backward by dense re-expansion, float64.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Restates ruDNN ``src/paged_attention/ordered_kernel.rs`` (``history_backward``):
for each sequence, the history tokens 0..len-1 are gathered from the pool
through the page table; each packed query row r of the sequence sees token t
when t <= pos(r) (causal) or always (non-causal); query head h reads KV head
g = h // (H / kv_heads).  The gradient of every physical pool row is the sum
over all (sequence, logical page) links that map to it, over the visible query
rows and over the query heads of its group.  Slots that no valid token owns,
and tail slots past a sequence's length, get zero.

The query side (the "query kernel" the page names, which computes the row
statistics once): dQ[r, h] = scale * sum_t dS_t k_t over the row's visible
tokens, and for MLA dQp[r, h] = scale * sum_t dS_t kp_t; a row that belongs to
no sequence, or sees no token, gets zero.

MLA (``position_dim > 0``): the score is q.k_latent + qp.k_position; the latent
is both key and value, so dK_latent = dS^T Q + P^T dY and dKp = dS^T Qp, with
no separate dV.  Here this is the dense backward on Q' = [q | qp],
K' = [k_latent | k_position], V = k_latent, then dK_latent = dK'[:, :Dk] + dV.
"""
from __future__ import annotations

import math

import numpy as np

from .dense import head_backward


def _slots_of(page_table_row, length, page_size):
    t = np.arange(length)
    return page_table_row[t // page_size].astype(np.int64) * page_size + t % page_size


def attn_bwd_paged(q, dy, k_pool, page_table, seq_len, q_start, q_pos, *, page_size, kv_heads,
                   v_pool=None, qp=None, kp_pool=None, causal=True, scale=None,
                   return_stats=False, return_dq=False):
    """q: [Nq, H, Dk]; dy: [Nq, H, Dv]; pools: [slots, kv_heads, dim].

    Returns float64 (dk_pool, dv_pool) for GQA or (dk_pool, dkp_pool) for MLA,
    plus lse, delta [Nq, H] when ``return_stats``, plus dq [Nq, H, Dk] (and
    dqp [Nq, H, Dp] for MLA) when ``return_dq``."""
    q = np.asarray(q, dtype=np.float64)
    dy = np.asarray(dy, dtype=np.float64)
    Nq, H, Dk = q.shape
    mla = qp is not None
    group = H // kv_heads
    if scale is None:
        scale = 1.0 / math.sqrt(Dk + (qp.shape[2] if mla else 0))
    slots = k_pool.shape[0]
    dk_pool = np.zeros((slots, kv_heads, Dk))
    if mla:
        Dp = qp.shape[2]
        dkp_pool = np.zeros((slots, kv_heads, Dp))
    else:
        dv_pool = np.zeros((slots, kv_heads, v_pool.shape[2]))
    lse = np.full((Nq, H), -np.inf)
    delta = np.zeros((Nq, H))
    dq = np.zeros((Nq, H, Dk))
    dqp = np.zeros((Nq, H, qp.shape[2])) if mla else None
    for s in range(len(seq_len)):
        L = int(seq_len[s])
        r0, r1 = int(q_start[s]), int(q_start[s + 1])
        if L == 0 or r1 == r0:
            continue
        sl = _slots_of(page_table[s], L, page_size)
        pos = np.asarray(q_pos[r0:r1])
        t = np.arange(L)
        vis = (t[None, :] <= pos[:, None]) if causal else np.ones((r1 - r0, L), dtype=bool)
        for h in range(H):
            g = h // group
            K = np.asarray(k_pool[sl, g], dtype=np.float64)
            if mla:
                Qc = np.concatenate([q[r0:r1, h], np.asarray(qp[r0:r1, h], dtype=np.float64)], axis=1)
                Kc = np.concatenate([K, np.asarray(kp_pool[sl, g], dtype=np.float64)], axis=1)
                r = head_backward(Qc, Kc, K, dy[r0:r1, h], vis, scale)
                np.add.at(dk_pool[:, g], sl, r["dk"][:, :Dk] + r["dv"])
                np.add.at(dkp_pool[:, g], sl, r["dk"][:, Dk:])
                dq[r0:r1, h] = r["dq"][:, :Dk]
                dqp[r0:r1, h] = r["dq"][:, Dk:]
            else:
                V = np.asarray(v_pool[sl, g], dtype=np.float64)
                r = head_backward(q[r0:r1, h], K, V, dy[r0:r1, h], vis, scale)
                np.add.at(dk_pool[:, g], sl, r["dk"])
                np.add.at(dv_pool[:, g], sl, r["dv"])
                dq[r0:r1, h] = r["dq"]
            lse[r0:r1, h] = r["lse"]
            delta[r0:r1, h] = r["delta"]
    out = (dk_pool, dkp_pool) if mla else (dk_pool, dv_pool)
    if return_stats:
        out = out + (lse, delta)
    if return_dq:
        out = out + ((dq, dqp) if mla else (dq,))
    return out


def paged_row_stats(q, dy, k_pool, page_table, seq_len, q_start, q_pos, *, page_size, kv_heads,
                    v_pool=None, qp=None, kp_pool=None, causal=True, scale=None):
    """Row statistics (lse, delta) per (query row, head), [Nq, H] float64:
    lse = log sum_t exp(s_t) over visible tokens, delta = sum_t P_t dP_t."""
    r = attn_bwd_paged(q, dy, k_pool, page_table, seq_len, q_start, q_pos, page_size=page_size,
                       kv_heads=kv_heads, v_pool=v_pool, qp=qp, kp_pool=kp_pool, causal=causal,
                       scale=scale, return_stats=True)
    return r[-2], r[-1]


def paged_query_backward(q, dy, k_pool, page_table, seq_len, q_start, q_pos, *, page_size, kv_heads,
                         v_pool=None, qp=None, kp_pool=None, causal=True, scale=None):
    """Query side of the paged backward, float64: (lse, delta, dq) for GQA or
    (lse, delta, dq, dqp) for MLA; lse, delta [Nq, H], dq [Nq, H, Dk],
    dqp [Nq, H, Dp]."""
    r = attn_bwd_paged(q, dy, k_pool, page_table, seq_len, q_start, q_pos, page_size=page_size,
                       kv_heads=kv_heads, v_pool=v_pool, qp=qp, kp_pool=kp_pool, causal=causal,
                       scale=scale, return_stats=True, return_dq=True)
    return r[2:]
