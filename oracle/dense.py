"""Dense attention backward, float64, one (batch, head) at a time.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Restates rlx-cpu ``src/attention_bwd.rs`` (``backward_dense_head_all`` and its
driver ``attention_backward_all``) with numpy matmuls as the only library
primitive.  Readings taken where the pages are silent or disagree:

* structural masks (causal, window) are hard: an excluded entry gets P = 0;
  a row with no structurally visible key gets P = 0 (it contributes nothing);
* masks compose as: add bias, then replace custom-masked scores by
  ``mask_neg`` (-1e9), then exclude structurally masked entries;
* the custom mask is one value per key, [B, Sk], masked when value < thr;
* dS = P * (dP - rowsum(P * dP)) * scale on every visible entry (the pages
  apply it uniformly, including custom-masked entries).
"""
from __future__ import annotations

import math

import numpy as np


def visibility(seq_q: int, seq_k: int, causal: bool, window: int | None, top_left: bool = False) -> np.ndarray:
    """Structurally visible (query, key) pairs, bottom-right aligned.

    rlx-cpu attention_bwd.rs, ``apply_synthetic_mask``: q_offset = Sk - Sq
    (saturating at 0), abs_q = q_offset + qi; causal excludes ki > abs_q; the
    sliding window w excludes ki < abs_q - w (saturating) or ki > abs_q.
    ``top_left``: the alignment of rlx-wgpu attention_bwd.wgsl ``mask_score``
    (causal hides ki > qi), i.e. q_offset = 0."""
    q_off = 0 if top_left else max(seq_k - seq_q, 0)
    abs_q = q_off + np.arange(seq_q)[:, None]
    ki = np.arange(seq_k)[None, :]
    vis = np.ones((seq_q, seq_k), dtype=bool)
    if causal or window is not None:
        vis &= ki <= abs_q
    if window is not None:
        lo = np.maximum(abs_q - int(window), 0)
        vis &= ki >= lo
    return vis


def head_backward(q, k, v, dy, vis, scale, key_masked=None, bias=None, mask_neg=-1e9, elem_masked=None):
    """Backward of one head.  q, dy: [Sq, D]; k, v: [Sk, D]; vis: [Sq, Sk] bool;
    key_masked: [Sk] bool (custom mask hit) or None; bias: [Sq, Sk] or None;
    elem_masked: [Sq, Sk] bool (per-element custom mask hit, rlx-wgpu
    attention_bwd.wgsl ``mask_score`` kind 2) or None.

    Steps (rlx-cpu attention_bwd.rs, ``backward_dense_head_all``):
      S  = scale * Q K^T            (score product)
      S += bias                     (additive bias mask)
      S[:, masked keys] = mask_neg  (custom mask; per element likewise)
      P  = softmax over visible keys, max-subtracted
      dV = P^T dY
      dP = dY V^T
      dS = P * (dP - rowsum(P * dP)) * scale
      dQ = dS K
      dK = dS^T Q
    Returns a dict with dq, dk, dv and the intermediates p, ds, lse, delta."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    dy = np.asarray(dy, dtype=np.float64)
    s = scale * (q @ k.T)
    if bias is not None:
        s = s + np.asarray(bias, dtype=np.float64)
    if key_masked is not None:
        s[:, np.asarray(key_masked, dtype=bool)] = mask_neg
    if elem_masked is not None:
        s = np.where(np.asarray(elem_masked, dtype=bool), mask_neg, s)
    s = np.where(vis, s, -np.inf)
    m = s.max(axis=1, initial=-np.inf)
    has = np.isfinite(m)
    m_safe = np.where(has, m, 0.0)
    e = np.where(vis, np.exp(s - m_safe[:, None]), 0.0)
    l = e.sum(axis=1)
    p = np.zeros_like(e)
    p[has] = e[has] / l[has, None]
    dv = p.T @ dy
    dp = dy @ v.T
    delta = (p * dp).sum(axis=1)
    ds = p * (dp - delta[:, None]) * scale
    dq = ds @ k
    dk = ds.T @ q
    lse = np.full(m.shape, -np.inf)
    lse[has] = m_safe[has] + np.log(l[has])
    return dict(dq=dq, dk=dk, dv=dv, p=p, ds=ds, lse=lse, delta=delta)


def _heads(x, layout):
    """View [B,S,H,D] or [B,H,S,D] as [B,H,S,D]."""
    if layout == "bshd":
        return np.transpose(x, (0, 2, 1, 3))
    if layout == "bhsd":
        return x
    raise ValueError(layout)


def attn_bwd_dense(q, k, v, dy, *, layout="bshd", causal=False, window=None, key_mask=None,
                   bias=None, mask_thr=0.5, mask_neg=-1e9, scale=None, heads_subset=None,
                   return_stats=False, top_left=False, elem_mask=None):
    """Full-tensor dense backward (rlx-cpu attention_bwd.rs, ``attention_backward_all``).

    q, dy: [B,Sq,H,D] ('bshd') or [B,H,Sq,D] ('bhsd'); k, v likewise with Sk.
    key_mask: [B, Sk] (masked where value < mask_thr); bias: [B, H, Sq, Sk].
    ``heads_subset``: optional list of (b, h) to evaluate (others stay zero).
    ``top_left``: causal / window masks aligned top-left (see ``visibility``).
    ``elem_mask``: [B, H, Sq, Sk] per-element custom mask (masked where value
    < mask_thr), alone or together with ``key_mask``.
    Returns float64 dq, dk, dv in the input layout (and lse, delta [B,H,Sq]
    when ``return_stats``)."""
    qh, kh, vh, dyh = (_heads(np.asarray(x), layout) for x in (q, k, v, dy))
    B, H, Sq, D = qh.shape
    Sk = kh.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    vis = visibility(Sq, Sk, causal, window, top_left)
    dq = np.zeros((B, H, Sq, D))
    dk = np.zeros((B, H, Sk, D))
    dv = np.zeros((B, H, Sk, D))
    lse = np.full((B, H, Sq), -np.inf)
    delta = np.zeros((B, H, Sq))
    pairs = heads_subset if heads_subset is not None else [(b, h) for b in range(B) for h in range(H)]
    for b, h in pairs:
        km = None if key_mask is None else (np.asarray(key_mask[b]) < mask_thr)
        bi = None if bias is None else bias[b, h]
        em = None if elem_mask is None else (np.asarray(elem_mask[b, h]) < mask_thr)
        r = head_backward(qh[b, h], kh[b, h], vh[b, h], dyh[b, h], vis, scale,
                          key_masked=km, bias=bi, mask_neg=mask_neg, elem_masked=em)
        dq[b, h], dk[b, h], dv[b, h] = r["dq"], r["dk"], r["dv"]
        lse[b, h], delta[b, h] = r["lse"], r["delta"]
    if layout == "bshd":
        dq, dk, dv = (np.transpose(x, (0, 2, 1, 3)) for x in (dq, dk, dv))
    if return_stats:
        return dq, dk, dv, lse, delta
    return dq, dk, dv


def attn_fwd_dense(q, k, v, *, layout="bshd", causal=False, window=None, key_mask=None, bias=None,
                   mask_thr=0.5, mask_neg=-1e9, scale=None, top_left=False, elem_mask=None):
    """Forward output O = P V and lse = log-sum-exp of the masked scores, float64.

    The probabilities are those of the backward (same masks, same softmax); a
    row with no visible key has O = 0 and lse = -inf.  Returns (o in the input
    layout, lse [B, H, Sq]).  ``top_left`` as for ``attn_bwd_dense``."""
    qh, kh, vh = (_heads(np.asarray(x), layout) for x in (q, k, v))
    B, H, Sq, D = qh.shape
    Sk = kh.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    vis = visibility(Sq, Sk, causal, window, top_left)
    o = np.zeros((B, H, Sq, vh.shape[3]))
    lse = np.full((B, H, Sq), -np.inf)
    for b in range(B):
        for h in range(H):
            km = None if key_mask is None else (np.asarray(key_mask[b]) < mask_thr)
            bi = None if bias is None else bias[b, h]
            em = None if elem_mask is None else (np.asarray(elem_mask[b, h]) < mask_thr)
            # the backward's P with a zero upstream gradient
            r = head_backward(qh[b, h], kh[b, h], vh[b, h], np.zeros((Sq, vh.shape[3])), vis, scale,
                              key_masked=km, bias=bi, mask_neg=mask_neg, elem_masked=em)
            o[b, h] = r["p"] @ np.asarray(vh[b, h], dtype=np.float64)
            lse[b, h] = r["lse"]
    if layout == "bshd":
        o = np.transpose(o, (0, 2, 1, 3))
    return o, lse
