"""Pins for the dense CPU oracle that do not reuse its formulas.

* central finite differences of L = sum(dY * softmax(mask(scale*QK^T + bias)) V)
  with respect to every entry of Q, K and V (the loss is evaluated here with
  explicit per-row loops, not with the oracle);
* invariants: rowsum(dS) = 0, sum_k dV_k = sum_q dY_q, sum_k dK_k = 0 and
  sum(Q*dQ) = sum(K*dK);
* closed forms (V = 0, Q = 0, a single key, the first causal row, a fully
  custom-masked row);
* the structural masks against a loop restatement and against the visible
  fractions that follow from counting.
"""
import math

import numpy as np
import pytest

from attention_backward_recompute_gb300 import inputs
from oracle import attn_bwd_dense, head_backward, visibility


# ---------------------------------------------------------------------------
# an independent forward: per-row loops over keys, float64
# ---------------------------------------------------------------------------

def _loop_visible(qi, ki, sq, sk, causal, window):
    q_off = sk - sq if sk > sq else 0
    abs_q = q_off + qi
    if causal or window is not None:
        if ki > abs_q:
            return False
    if window is not None:
        lo = abs_q - window if abs_q > window else 0
        if ki < lo:
            return False
    return True


def loop_loss(q, k, v, dy, causal=False, window=None, key_mask=None, bias=None, thr=0.5,
              neg=-1e9, layout="bshd", elem_mask=None):
    """L = sum over b,h,q,d of dY * O with O the attention output (loops)."""
    if layout == "bshd":
        B, Sq, H, D = q.shape
        Sk = k.shape[1]
        get = lambda x, b, s, h: x[b, s, h]
    else:
        B, H, Sq, D = q.shape
        Sk = k.shape[2]
        get = lambda x, b, s, h: x[b, h, s]
    scale = 1.0 / math.sqrt(D)
    total = 0.0
    for b in range(B):
        for h in range(H):
            for qi in range(Sq):
                scores = []
                for ki in range(Sk):
                    if not _loop_visible(qi, ki, Sq, Sk, causal, window):
                        continue
                    s = scale * float(np.dot(get(q, b, qi, h), get(k, b, ki, h)))
                    if bias is not None:
                        s += float(bias[b, h, qi, ki])
                    if key_mask is not None and key_mask[b, ki] < thr:
                        s = neg
                    if elem_mask is not None and elem_mask[b, h, qi, ki] < thr:
                        s = neg
                    scores.append((ki, s))
                if not scores:
                    continue
                mx = max(s for _, s in scores)
                w = [(ki, math.exp(s - mx)) for ki, s in scores]
                z = sum(e for _, e in w)
                out = np.zeros(D)
                for ki, e in w:
                    out += (e / z) * get(v, b, ki, h)
                total += float(np.dot(get(dy, b, qi, h), out))
    return total


def fd_grad(f, x, h=1e-6):
    g = np.zeros_like(x)
    it = np.nditer(x, flags=["multi_index"])
    for _ in it:
        idx = it.multi_index
        old = x[idx]
        x[idx] = old + h
        fp = f()
        x[idx] = old - h
        fm = f()
        x[idx] = old
        g[idx] = (fp - fm) / (2 * h)
    return g


def _rel(a, b):
    return np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300)


TINY = [
    # (Sq, Sk, causal, window, key mask, bias)
    (3, 5, False, None, False, False),
    (5, 3, True, None, False, False),
    (5, 8, True, None, False, False),
    (8, 8, False, 2, False, False),
    (8, 5, False, 1, False, False),
    (5, 5, False, None, True, False),
    (4, 6, True, None, True, True),
    (6, 6, False, None, False, True),
]


@pytest.mark.parametrize("sq,sk,causal,window,use_km,use_bias", TINY)
@pytest.mark.parametrize("layout", ["bshd", "bhsd"])
def test_fd_tiny(sq, sk, causal, window, use_km, use_bias, layout):
    rng = np.random.default_rng(sq * 100 + sk * 10 + int(causal))
    B, H, D = 1, 2, 4
    if layout == "bshd":
        qs, ks = (B, sq, H, D), (B, sk, H, D)
    else:
        qs, ks = (B, H, sq, D), (B, H, sk, D)
    q, k, v, dy = (rng.standard_normal(s) for s in (qs, ks, ks, qs))
    km = None
    if use_km:
        km = np.ones((B, sk))
        km[0, sk - 2] = 0.0      # mask a late key: every row keeps an unmasked key
    bias = rng.standard_normal((B, H, sq, sk)) if use_bias else None
    dq, dk, dv = attn_bwd_dense(q, k, v, dy, layout=layout, causal=causal, window=window,
                                key_mask=km, bias=bias)
    f = lambda: loop_loss(q, k, v, dy, causal, window, km, bias, layout=layout)
    for x, g in ((q, dq), (k, dk), (v, dv)):
        num = fd_grad(f, x)
        assert _rel(g, num) < 1e-6, _rel(g, num)


def test_fd_small_f32_config():
    c = inputs.dense_config("dense_small_f32")
    q, k, v, dy = (x.astype(np.float64) for x in (c.q, c.k, c.v, c.dy))
    dq, dk, dv = attn_bwd_dense(q, k, v, dy)
    f = lambda: loop_loss(q, k, v, dy)
    for x, g in ((q, dq), (k, dk), (v, dv)):
        num = fd_grad(f, x)
        assert _rel(g, num) < 1e-6


def _read_fixture():
    kv = {}
    with open(__file__.replace("test_oracle_dense.py", "golden/p1_hash_fixture.txt")) as fh:
        for line in fh:
            line = line.strip()
            if line and not line.startswith("#"):
                a, b = line.split()
                kv[a] = b
    return kv


def test_fd_p1_hash_fixture():
    fx = _read_fixture()
    b, nh, s, dh = (int(fx[n]) for n in ("batch", "heads", "seq", "head_dim"))
    n = b * s * nh * dh
    arrs = [inputs.p1_hash_values(n, int(fx[f"seed_{t}"])).reshape(b, s, nh, dh).astype(np.float64)
            for t in ("q", "k", "v", "dy")]
    q, k, v, dy = arrs
    dq, dk, dv = attn_bwd_dense(q, k, v, dy, causal=True)
    f = lambda: loop_loss(q, k, v, dy, causal=True)
    for x, g in ((q, dq), (k, dk), (v, dv)):
        num = fd_grad(f, x)
        assert _rel(g, num) < 1e-6
    # the fused result equals one-gradient-at-a-time evaluation (the unit test's
    # property): evaluating each head separately reproduces the same numbers.
    for bi in range(b):
        for hi in range(nh):
            one = attn_bwd_dense(q, k, v, dy, causal=True, heads_subset=[(bi, hi)])
            for full, part in zip((dq, dk, dv), one):
                np.testing.assert_array_equal(full[bi, :, hi], part[bi, :, hi])


# ---------------------------------------------------------------------------
# invariants
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("causal,window,use_km,use_bias", [
    (False, None, False, False), (True, None, False, False), (False, 7, False, False),
    (True, None, True, True), (False, None, True, False), (False, 3, False, True)])
@pytest.mark.parametrize("sq,sk", [(24, 24), (16, 40), (40, 16)])
def test_invariants(causal, window, use_km, use_bias, sq, sk):
    rng = np.random.default_rng(7)
    D = 8
    q, dy = rng.standard_normal((sq, D)), rng.standard_normal((sq, D))
    k, v = rng.standard_normal((sk, D)), rng.standard_normal((sk, D))
    vis = visibility(sq, sk, causal, window)
    km = None
    if use_km:
        km = rng.random(sk) < 0.3
    bias = rng.standard_normal((sq, sk)) if use_bias else None
    r = head_backward(q, k, v, dy, vis, 1 / math.sqrt(D), key_masked=km, bias=bias)
    nonempty = vis.any(axis=1)
    # rowsum(dS) = 0 for every row
    assert np.max(np.abs(r["ds"].sum(axis=1))) < 1e-12
    # sum_k dK_k = sum_q (rowsum dS_q) Q_q = 0
    assert np.max(np.abs(r["dk"].sum(axis=0))) < 1e-11
    # sum_k dV_k = sum_q dY_q over rows whose probabilities sum to one
    np.testing.assert_allclose(r["dv"].sum(axis=0), dy[nonempty].sum(axis=0), atol=1e-11)
    # sum(Q * dQ) = sum(dS * QK^T) = sum(K * dK)
    assert abs(np.sum(q * r["dq"]) - np.sum(k * r["dk"])) < 1e-10
    # probabilities: non-negative, rows sum to one (or zero for empty rows)
    assert np.all(r["p"] >= 0)
    np.testing.assert_allclose(r["p"].sum(axis=1), nonempty.astype(float), atol=1e-13)
    assert np.all(r["p"][~vis] == 0)


# ---------------------------------------------------------------------------
# closed forms
# ---------------------------------------------------------------------------

def test_zero_v_gives_zero_dq_dk():
    rng = np.random.default_rng(3)
    q, k, dy = rng.standard_normal((1, 9, 2, 8)), rng.standard_normal((1, 11, 2, 8)), rng.standard_normal((1, 9, 2, 8))
    v = np.zeros((1, 11, 2, 8))
    dq, dk, dv = attn_bwd_dense(q, k, v, dy, causal=True)
    assert np.all(dq == 0) and np.all(dk == 0)
    assert np.any(dv != 0)


def test_zero_q_uniform_attention():
    rng = np.random.default_rng(4)
    Sq, Sk, D = 6, 10, 8
    q = np.zeros((Sq, D))
    k, v, dy = rng.standard_normal((Sk, D)), rng.standard_normal((Sk, D)), rng.standard_normal((Sq, D))
    scale = 1 / math.sqrt(D)
    r = head_backward(q, k, v, dy, np.ones((Sq, Sk), bool), scale)
    np.testing.assert_allclose(r["p"], np.full((Sq, Sk), 1 / Sk), rtol=1e-14)
    # dV_k = (1/Sk) sum_q dY_q for every key
    np.testing.assert_allclose(r["dv"], np.tile(dy.sum(0) / Sk, (Sk, 1)), rtol=1e-12, atol=1e-14)
    assert np.max(np.abs(r["dk"])) < 1e-14
    vbar = v.mean(0)
    expect = np.zeros((Sq, D))
    for i in range(Sq):
        for j in range(Sk):
            expect[i] += scale / Sk * (dy[i] @ v[j] - dy[i] @ vbar) * k[j]
    np.testing.assert_allclose(r["dq"], expect, rtol=1e-11, atol=1e-13)


def test_single_key_and_first_causal_row():
    rng = np.random.default_rng(5)
    q, k, v, dy = (rng.standard_normal(s) for s in ((1, 4, 1, 8), (1, 1, 1, 8), (1, 1, 1, 8), (1, 4, 1, 8)))
    dq, dk, dv = attn_bwd_dense(q, k, v, dy)
    assert np.max(np.abs(dq)) < 1e-15 and np.max(np.abs(dk)) < 1e-15
    np.testing.assert_allclose(dv[0, 0, 0], dy[0, :, 0].sum(0), rtol=1e-14)
    # causal, Sq = Sk: row 0 sees only key 0, so its dS row is zero and dQ_0 = 0
    q, k, v, dy = (rng.standard_normal((1, 7, 2, 8)) for _ in range(4))
    dq, _, _ = attn_bwd_dense(q, k, v, dy, causal=True)
    assert np.max(np.abs(dq[0, 0])) < 1e-15


def test_fully_custom_masked_row_is_uniform():
    """A row whose visible keys are all custom-masked: every visible score is
    -1e9, so the softmax is uniform over the visible keys and the pages' dS
    formula applies to it like any other row."""
    rng = np.random.default_rng(6)
    Sq, Sk, D = 4, 4, 8
    q, k, v, dy = (rng.standard_normal((n, D)) for n in (Sq, Sk, Sk, Sq))
    vis = visibility(Sq, Sk, True, None)
    km = np.array([True, True, False, False])      # row 0 and row 1 fully masked
    r = head_backward(q, k, v, dy, vis, 1 / math.sqrt(D), key_masked=km)
    np.testing.assert_allclose(r["p"][0], [1, 0, 0, 0])
    np.testing.assert_allclose(r["p"][1], [0.5, 0.5, 0, 0])
    assert r["p"][2, 0] == 0 and r["p"][2, 1] == 0 and r["p"][2, 2] == 1.0
    dp1 = dy[1] @ v[:2].T
    ds1 = 0.5 * (dp1 - 0.5 * dp1.sum()) / math.sqrt(D)
    np.testing.assert_allclose(r["ds"][1, :2], ds1, rtol=1e-12)


def test_layouts_agree():
    c = inputs.dense_inputs(batch=2, heads=3, seq_q=9, seq_k=13, head_dim=8, dtype="f32", seed=9,
                            causal=True, key_mask_zero_frac=0.2, bias=True)
    a = attn_bwd_dense(c.q, c.k, c.v, c.dy, causal=True, key_mask=c.key_mask, bias=c.bias)
    t = lambda x: np.ascontiguousarray(np.transpose(x, (0, 2, 1, 3)))
    b = attn_bwd_dense(t(c.q), t(c.k), t(c.v), t(c.dy), layout="bhsd", causal=True,
                       key_mask=c.key_mask, bias=c.bias)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, t(y))


# ---------------------------------------------------------------------------
# structural masks
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("sq,sk,causal,window", [(5, 9, True, None), (9, 5, True, None),
                                                 (7, 7, False, 2), (4, 10, False, 3),
                                                 (10, 4, False, 1), (6, 6, False, None)])
def test_visibility_matches_loops(sq, sk, causal, window):
    vis = visibility(sq, sk, causal, window)
    for qi in range(sq):
        for ki in range(sk):
            assert vis[qi, ki] == _loop_visible(qi, ki, sq, sk, causal, window)


def test_visible_fractions_by_counting():
    # causal S x S: S(S+1)/2 pairs
    v = visibility(2048, 2048, True, None)
    assert v.sum() == 2048 * 2049 // 2
    # bottom-right causal, Sq=256, Sk=4096: row i sees 3840 + i + 1 keys
    v = visibility(256, 4096, True, None)
    assert v.sum() == sum(3841 + i for i in range(256))
    # window 128 on 512: row i sees min(i, 128) + 1 keys
    v = visibility(512, 512, False, 128)
    assert v.sum() == sum(min(i, 128) + 1 for i in range(512))
    assert abs(v.sum() / 512 ** 2 - 0.220459) < 1e-6


def test_forward_output_by_loops():
    """O from the oracle's forward equals the loop forward's attention output:
    sum(dY * O) must equal the loop loss for any dY."""
    from oracle import attn_fwd_dense
    rng = np.random.default_rng(12)
    q, k, v = rng.standard_normal((1, 6, 2, 4)), rng.standard_normal((1, 9, 2, 4)), rng.standard_normal((1, 9, 2, 4))
    km = np.ones((1, 9)); km[0, 5] = 0
    bias = rng.standard_normal((1, 2, 6, 9))
    o, lse = attn_fwd_dense(q, k, v, causal=True, key_mask=km, bias=bias)
    for _ in range(3):
        dy = rng.standard_normal(q.shape)
        assert abs(np.sum(dy * o) - loop_loss(q, k, v, dy, True, None, km, bias)) < 1e-12
    # lse: exp(lse) is the softmax normaliser, so sum_k exp(s - lse) = 1 per row
    assert np.all(np.isfinite(lse))


# ---------------------------------------------------------------------------
# top-left alignment (rlx-wgpu attention_bwd.wgsl, mask_score: causal hides
# ki > qi): each row is plain attention over a key prefix
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("sq,sk", [(5, 9), (9, 5), (6, 6)])
def test_top_left_causal_is_prefix_attention(sq, sk):
    """With top-left causal alignment row q sees keys 0..min(q, Sk-1); its
    gradients equal those of an unmasked single-row problem on that key
    prefix, summed over rows for dK and dV."""
    rng = np.random.default_rng(71)
    D = 4
    q, k, v, dy = (rng.standard_normal(s) for s in ((1, sq, 1, D), (1, sk, 1, D), (1, sk, 1, D), (1, sq, 1, D)))
    dq, dk, dv = attn_bwd_dense(q, k, v, dy, causal=True, top_left=True)
    want_dq = np.zeros_like(dq)
    want_dk = np.zeros_like(dk)
    want_dv = np.zeros_like(dv)
    for qi in range(sq):
        n = min(qi, sk - 1) + 1
        r = attn_bwd_dense(q[:, qi:qi + 1], k[:, :n], v[:, :n], dy[:, qi:qi + 1], causal=False,
                           scale=1.0 / math.sqrt(D))
        want_dq[:, qi] = r[0][:, 0]
        want_dk[:, :n] += r[1]
        want_dv[:, :n] += r[2]
    np.testing.assert_allclose(dq, want_dq, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(dk, want_dk, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(dv, want_dv, rtol=1e-12, atol=1e-12)
    if sq < sk:  # differs from the bottom-right default there
        assert not np.allclose(dq, attn_bwd_dense(q, k, v, dy, causal=True)[0])


def test_top_left_window_is_band_attention():
    """Top-left window w: row q sees keys max(q - w, 0)..q (a band of plain
    attention over that key range)."""
    rng = np.random.default_rng(72)
    sq, sk, D, w = 7, 11, 4, 2
    q, k, v, dy = (rng.standard_normal(s) for s in ((1, sq, 1, D), (1, sk, 1, D), (1, sk, 1, D), (1, sq, 1, D)))
    dq = attn_bwd_dense(q, k, v, dy, window=w, top_left=True)[0]
    for qi in range(sq):
        lo, hi = max(qi - w, 0), qi + 1
        r = attn_bwd_dense(q[:, qi:qi + 1], k[:, lo:hi], v[:, lo:hi], dy[:, qi:qi + 1], scale=1.0 / math.sqrt(D))
        np.testing.assert_allclose(dq[:, qi], r[0][:, 0], rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------------------
# per-element custom mask (rlx-wgpu attention_bwd.wgsl, mask_score kind 2)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("causal,use_bias", [(False, False), (True, True)])
def test_fd_element_mask(causal, use_bias):
    """Finite differences of the looped loss with a per-element mask (each row
    keeps an unmasked visible key)."""
    rng = np.random.default_rng(91)
    B, H, sq, sk, D = 1, 2, 5, 6, 4
    q, k, v, dy = (rng.standard_normal(x) for x in ((B, sq, H, D), (B, sk, H, D), (B, sk, H, D), (B, sq, H, D)))
    em = (rng.random((B, H, sq, sk)) > 0.3).astype(np.float64)
    em[..., 0] = 1.0  # key 0 is visible to every row under either mask
    bias = rng.standard_normal((B, H, sq, sk)) if use_bias else None
    dq, dk, dv = attn_bwd_dense(q, k, v, dy, causal=causal, bias=bias, elem_mask=em)
    f = lambda: loop_loss(q, k, v, dy, causal, None, None, bias, elem_mask=em)
    for x, g in ((q, dq), (k, dk), (v, dv)):
        assert _rel(g, fd_grad(f, x)) < 1e-6


def test_element_mask_repeating_a_key_mask_is_the_key_mask():
    """An element mask equal to a key mask on every row gives the key mask's
    gradients (and statistics), including rows whose keys are all masked."""
    rng = np.random.default_rng(92)
    B, H, sq, sk, D = 2, 2, 6, 7, 4
    q, k, v, dy = (rng.standard_normal(x) for x in ((B, sq, H, D), (B, sk, H, D), (B, sk, H, D), (B, sq, H, D)))
    km = (rng.random((B, sk)) > 0.4).astype(np.float64)
    km[:, 0] = 0.0  # under causal alignment the first row sees only masked keys
    em = np.broadcast_to(km[:, None, None, :], (B, H, sq, sk)).copy()
    a = attn_bwd_dense(q, k, v, dy, causal=True, key_mask=km, return_stats=True)
    b = attn_bwd_dense(q, k, v, dy, causal=True, elem_mask=em, return_stats=True)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)
