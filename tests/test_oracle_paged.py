"""Pins for the paged CPU oracle.

* a brute-force per-physical-slot evaluation (loops over the slot's links, the
  sequence's query rows and the heads of the KV group, with row statistics from
  explicit per-row loops), compared with the oracle's dense re-expansion;
* finite differences of the loss with respect to the pool entries, for GQA and
  for MLA (where the latent is both key and value);
* unowned and tail slots come out exactly zero;
* the query side (dQ, and dQp for MLA): per-(row, head) loops over the visible
  tokens, and finite differences of the loss with respect to q and qp.
"""
import math

import numpy as np
import pytest

from attention_backward_recompute_gb300 import inputs
from oracle import attn_bwd_paged, paged_query_backward


def tiny_case(mla=False, shared=0, seed=11, causal=True):
    return inputs.paged_case(seed=seed, num_seqs=3, len_lo=5, len_hi=14, queries_per_seq=4,
                             heads=4, kv_heads=2 if not mla else 1, page_size=4,
                             key_dim=8 if not mla else 6, value_dim=8 if not mla else 6,
                             position_dim=0 if not mla else 3, pool_factor=1.5, dtype="f32",
                             scale=1.0, causal=causal, shared_prefix_pages=shared)


def _links(c):
    """physical page -> list of (sequence, logical page), in sequence order."""
    links = {}
    for s in range(c.num_seqs):
        npg = (int(c.seq_len[s]) + c.page_size - 1) // c.page_size
        for lp in range(npg):
            links.setdefault(int(c.page_table[s, lp]), []).append((s, lp))
    return links


def brute_force(c):
    """Per-slot loops: one owner per (physical slot, KV head)."""
    H, G = c.heads, c.kv_heads
    group = H // G
    scale = c.scale
    slots = c.num_pages * c.page_size
    q = c.q.astype(np.float64)
    dy = c.dy.astype(np.float64)
    qp = None if c.qp is None else c.qp.astype(np.float64)

    def key_of(slot, g):
        return c.k_pool[slot, g].astype(np.float64)

    def score(row, h, slot, g):
        s = float(q[row, h] @ key_of(slot, g))
        if c.mla:
            s += float(qp[row, h] @ c.kp_pool[slot, g].astype(np.float64))
        return s * scale

    def value_of(slot, g):
        return key_of(slot, g) if c.mla else c.v_pool[slot, g].astype(np.float64)

    # row statistics by explicit loops over the sequence's visible tokens
    lse = np.full((c.num_queries, H), -np.inf)
    delta = np.zeros((c.num_queries, H))
    for s in range(c.num_seqs):
        L = int(c.seq_len[s])
        for row in range(int(c.q_start[s]), int(c.q_start[s + 1])):
            for h in range(H):
                g = h // group
                toks = [t for t in range(L) if (not c.causal) or t <= int(c.q_pos[row])]
                sl = [int(c.page_table[s, t // c.page_size]) * c.page_size + t % c.page_size for t in toks]
                sc = [score(row, h, x, g) for x in sl]
                if not sc:
                    continue
                m = max(sc)
                z = sum(math.exp(a - m) for a in sc)
                lse[row, h] = m + math.log(z)
                p = [math.exp(a - lse[row, h]) for a in sc]
                delta[row, h] = sum(pi * float(dy[row, h] @ value_of(x, g)) for pi, x in zip(p, sl))
    links = _links(c)
    Dk, Dv, Dp = c.key_dim, c.value_dim, c.position_dim
    dk = np.zeros((slots, G, Dk))
    dv = np.zeros((slots, G, Dv))
    dkp = np.zeros((slots, G, max(Dp, 1)))
    for slot in range(slots):
        page, off = divmod(slot, c.page_size)
        for g in range(G):
            for s, lp in links.get(page, []):
                t = lp * c.page_size + off
                if t >= int(c.seq_len[s]):
                    continue
                for row in range(int(c.q_start[s]), int(c.q_start[s + 1])):
                    if c.causal and t > int(c.q_pos[row]):
                        continue
                    for h in range(g * group, (g + 1) * group):
                        p = math.exp(score(row, h, slot, g) - lse[row, h])
                        dpv = float(dy[row, h] @ value_of(slot, g))
                        ds = p * (dpv - delta[row, h]) * scale
                        dk[slot, g] += ds * q[row, h]
                        if c.mla:
                            dk[slot, g] += p * dy[row, h]
                            dkp[slot, g] += ds * qp[row, h]
                        else:
                            dv[slot, g] += p * dy[row, h]
    return dk, (dkp if c.mla else dv), lse, delta


def run_oracle(c):
    return attn_bwd_paged(c.q, c.dy, c.k_pool, c.page_table, c.seq_len, c.q_start, c.q_pos,
                          page_size=c.page_size, kv_heads=c.kv_heads, v_pool=c.v_pool, qp=c.qp,
                          kp_pool=c.kp_pool, causal=c.causal, return_stats=True)


@pytest.mark.parametrize("mla", [False, True])
@pytest.mark.parametrize("shared", [0, 1])
@pytest.mark.parametrize("causal", [True, False])
def test_paged_oracle_matches_brute_force(mla, shared, causal):
    c = tiny_case(mla=mla, shared=shared, causal=causal)
    a0, a1, lse, delta = run_oracle(c)
    b0, b1, blse, bdelta = brute_force(c)
    np.testing.assert_allclose(lse, blse, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(delta, bdelta, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(a0, b0, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(a1, b1, rtol=1e-10, atol=1e-12)


def test_unowned_and_tail_slots_are_zero():
    c = tiny_case(shared=1)
    dk, dv = run_oracle(c)[:2]
    valid = np.zeros(c.num_pages * c.page_size, bool)
    for s in range(c.num_seqs):
        for t in range(int(c.seq_len[s])):
            valid[int(c.page_table[s, t // c.page_size]) * c.page_size + t % c.page_size] = True
    assert (~valid).sum() > 0
    assert np.all(dk[~valid] == 0) and np.all(dv[~valid] == 0)
    # pool poisoning never leaks: the valid part is finite
    assert np.all(np.isfinite(dk)) and np.all(np.isfinite(dv))


def _paged_loss(c, k_pool, v_pool, kp_pool):
    """sum(dY * O) with O the attention output, by direct loops per row/head."""
    H, group = c.heads, c.heads // c.kv_heads
    tot = 0.0
    for s in range(c.num_seqs):
        L = int(c.seq_len[s])
        for row in range(int(c.q_start[s]), int(c.q_start[s + 1])):
            for h in range(H):
                g = h // group
                sc, vals = [], []
                for t in range(L):
                    if c.causal and t > int(c.q_pos[row]):
                        continue
                    slot = int(c.page_table[s, t // c.page_size]) * c.page_size + t % c.page_size
                    a = float(c.q[row, h] @ k_pool[slot, g])
                    if c.mla:
                        a += float(c.qp[row, h] @ kp_pool[slot, g])
                    sc.append(a * c.scale)
                    vals.append(k_pool[slot, g] if c.mla else v_pool[slot, g])
                m = max(sc)
                w = [math.exp(a - m) for a in sc]
                z = sum(w)
                out = sum((wi / z) * vi for wi, vi in zip(w, vals))
                tot += float(c.dy[row, h] @ out)
    return tot


@pytest.mark.parametrize("mla", [False, True])
def test_paged_fd(mla):
    c = tiny_case(mla=mla, seed=13)
    c.num_seqs  # noqa: B018
    kpool = np.nan_to_num(c.k_pool.astype(np.float64))
    vpool = None if c.v_pool is None else np.nan_to_num(c.v_pool.astype(np.float64))
    kppool = None if c.kp_pool is None else np.nan_to_num(c.kp_pool.astype(np.float64))
    c.q = c.q.astype(np.float64)
    c.dy = c.dy.astype(np.float64)
    if c.qp is not None:
        c.qp = c.qp.astype(np.float64)
    d0, d1 = attn_bwd_paged(c.q, c.dy, kpool, c.page_table, c.seq_len, c.q_start, c.q_pos,
                            page_size=c.page_size, kv_heads=c.kv_heads, v_pool=vpool, qp=c.qp,
                            kp_pool=kppool, causal=c.causal)
    f = lambda: _paged_loss(c, kpool, vpool, kppool)
    # check a sample of slots (every valid slot of sequence 0 and the first of others)
    h = 1e-6
    checked = 0
    for s in range(c.num_seqs):
        for t in range(int(c.seq_len[s])):
            slot = int(c.page_table[s, t // c.page_size]) * c.page_size + t % c.page_size
            for g in range(c.kv_heads):
                for pool, grad in ((kpool, d0), ((kppool if c.mla else vpool), d1)):
                    for d in range(pool.shape[2]):
                        old = pool[slot, g, d]
                        pool[slot, g, d] = old + h
                        fp = f()
                        pool[slot, g, d] = old - h
                        fm = f()
                        pool[slot, g, d] = old
                        num = (fp - fm) / (2 * h)
                        assert abs(num - grad[slot, g, d]) <= 1e-6 * max(1.0, abs(num)), (slot, g, d)
                        checked += 1
            if s > 0:
                break
    assert checked > 0


def brute_force_dq(c):
    """dQ (and dQp) by loops over each row's visible tokens, with the row
    statistics of the slot brute force."""
    _, _, lse, delta = brute_force(c)
    H, group = c.heads, c.heads // c.kv_heads
    q = c.q.astype(np.float64)
    dy = c.dy.astype(np.float64)
    dq = np.zeros(q.shape)
    dqp = None if c.qp is None else np.zeros(c.qp.shape)
    for s in range(c.num_seqs):
        for row in range(int(c.q_start[s]), int(c.q_start[s + 1])):
            for h in range(H):
                g = h // group
                for t in range(int(c.seq_len[s])):
                    if c.causal and t > int(c.q_pos[row]):
                        continue
                    slot = int(c.page_table[s, t // c.page_size]) * c.page_size + t % c.page_size
                    k = c.k_pool[slot, g].astype(np.float64)
                    a = float(q[row, h] @ k)
                    if c.mla:
                        a += float(c.qp[row, h].astype(np.float64) @ c.kp_pool[slot, g].astype(np.float64))
                    p = math.exp(a * c.scale - lse[row, h])
                    v = k if c.mla else c.v_pool[slot, g].astype(np.float64)
                    ds = p * (float(dy[row, h] @ v) - delta[row, h]) * c.scale
                    dq[row, h] += ds * k
                    if c.mla:
                        dqp[row, h] += ds * c.kp_pool[slot, g].astype(np.float64)
    return dq, dqp, lse, delta


def run_query_oracle(c):
    return paged_query_backward(c.q, c.dy, c.k_pool, c.page_table, c.seq_len, c.q_start, c.q_pos,
                                page_size=c.page_size, kv_heads=c.kv_heads, v_pool=c.v_pool, qp=c.qp,
                                kp_pool=c.kp_pool, causal=c.causal)


@pytest.mark.parametrize("mla", [False, True])
@pytest.mark.parametrize("causal", [True, False])
def test_paged_query_oracle_matches_brute_force(mla, causal):
    c = tiny_case(mla=mla, shared=1, causal=causal)
    got = run_query_oracle(c)
    want_dq, want_dqp, want_lse, want_delta = brute_force_dq(c)
    np.testing.assert_allclose(got[0], want_lse, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(got[1], want_delta, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(got[2], want_dq, rtol=1e-10, atol=1e-12)
    if mla:
        np.testing.assert_allclose(got[3], want_dqp, rtol=1e-10, atol=1e-12)


@pytest.mark.parametrize("mla", [False, True])
def test_paged_query_fd(mla):
    c = tiny_case(mla=mla, seed=17)
    kpool = np.nan_to_num(c.k_pool.astype(np.float64))
    vpool = None if c.v_pool is None else np.nan_to_num(c.v_pool.astype(np.float64))
    kppool = None if c.kp_pool is None else np.nan_to_num(c.kp_pool.astype(np.float64))
    c.q = c.q.astype(np.float64)
    c.dy = c.dy.astype(np.float64)
    if c.qp is not None:
        c.qp = c.qp.astype(np.float64)
    r = paged_query_backward(c.q, c.dy, kpool, c.page_table, c.seq_len, c.q_start, c.q_pos,
                             page_size=c.page_size, kv_heads=c.kv_heads, v_pool=vpool, qp=c.qp,
                             kp_pool=kppool, causal=c.causal)
    f = lambda: _paged_loss(c, kpool, vpool, kppool)
    h = 1e-6
    checked = 0
    targets = [(c.q, r[2])] + ([(c.qp, r[3])] if mla else [])
    for x, grad in targets:
        for row in (0, int(c.q_start[1]), c.num_queries - 1):
            for hh in range(c.heads):
                for d in range(x.shape[2]):
                    old = x[row, hh, d]
                    x[row, hh, d] = old + h
                    fp = f()
                    x[row, hh, d] = old - h
                    fm = f()
                    x[row, hh, d] = old
                    num = (fp - fm) / (2 * h)
                    assert abs(num - grad[row, hh, d]) <= 1e-6 * max(1.0, abs(num)), (row, hh, d)
                    checked += 1
    assert checked > 0
