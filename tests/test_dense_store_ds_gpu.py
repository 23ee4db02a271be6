"""GPU parity of the dense backward with ATTN_OPT_STORE_DS (the dK/dV kernel
stores every dS tile it forms and dQ = scale * dS K is one product over those
tiles) against the CPU oracle, and against the default call: dK and dV are
bit-identical (same kernel, same arithmetic), dQ agrees within tolerance.

Tolerance as for the other dense cases: per output tensor,
max|gpu - oracle| <= 2e-2 * max|oracle| (bf16 storage).
"""
import numpy as np
import pytest

from attention_backward_recompute_gb300 import inputs

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

TOL = 2e-2


@pytest.fixture(scope="module")
def bd():
    from attention_backward_recompute_gb300 import binding, build
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    binding.lib()
    return binding


def _dev(x, dtype=torch.bfloat16):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda().to(dtype)


def _close(res, ref):
    scale = max(float(np.max(np.abs(w))) for w in ref)
    for n, g, w in zip(("dq", "dk", "dv"), res, ref):
        got = g.float().cpu().numpy().astype(np.float64)
        err = float(np.max(np.abs(got - w)))
        assert err <= TOL * max(float(np.max(np.abs(w))), 1e-3 * scale), (n, err, float(np.max(np.abs(w))))


# (B, H, Sq, Sk, D, causal, window, key-mask zero fraction, bias, layout, top_left)
CASES = [
    (2, 3, 200, 328, 128, True, None, 0.1, True, "bshd", False),
    (2, 3, 200, 328, 128, False, None, None, False, "bshd", False),
    (1, 2, 330, 200, 128, True, None, None, False, "bshd", False),
    (1, 2, 300, 300, 128, False, 37, None, False, "bshd", False),
    (1, 2, 256, 456, 128, False, 100, None, True, "bhsd", False),
    (2, 2, 192, 192, 64, True, None, 0.2, False, "bhsd", False),
    (1, 3, 130, 264, 64, False, None, None, True, "bshd", False),
    (1, 2, 77, 513, 32, True, None, None, False, "bshd", False),
    (2, 2, 200, 456, 128, True, None, 0.1, True, "bshd", True),
    (1, 1, 5, 700, 128, True, None, None, False, "bhsd", False),
]


def _run(bd, c, top_left, store_ds, wrt=7, elem=None):
    q, k, v, dy = (_dev(x) for x in (c.q, c.k, c.v, c.dy))
    km = None if c.key_mask is None else torch.from_numpy(c.key_mask).cuda()
    bi = None if c.bias is None else _dev(c.bias)
    res = bd.dense_backward(q, k, v, dy, layout=c.layout, causal=c.causal, window=c.window, key_mask=km, bias=bi,
                            top_left=top_left, store_ds=store_ds, wrt=wrt, elem_mask=elem)
    bd.check_device_error()
    return res


@pytest.mark.parametrize("case", CASES, ids=lambda c: "q%dk%dD%d_c%d_w%s_km%s_b%d_%s_tl%d" % (
    c[2], c[3], c[4], c[5], c[6], c[7], c[8], c[9], c[10]))
def test_store_ds_parity(bd, case):
    from oracle import attn_bwd_dense
    B, H, Sq, Sk, D, causal, window, kmz, bias, layout, top_left = case
    c = inputs.dense_inputs(batch=B, heads=H, seq_q=Sq, seq_k=Sk, head_dim=D, layout=layout,
                            seed=800 + CASES.index(case), scale=0.5, causal=causal, window=window,
                            key_mask_zero_frac=kmz, bias=bias)
    res = _run(bd, c, top_left, True)
    ref = attn_bwd_dense(c.q, c.k, c.v, c.dy, layout=layout, causal=causal, window=window, key_mask=c.key_mask,
                         bias=c.bias, top_left=top_left)
    _close(res, ref)
    base = _run(bd, c, top_left, False)
    assert torch.equal(res[1], base[1]) and torch.equal(res[2], base[2])


def test_store_ds_dq_only_and_elem_mask(bd):
    """dQ alone still runs the dK/dV kernel (it forms dS) and stores no dK/dV;
    with a per-element mask the stored tiles carry it."""
    from oracle import attn_bwd_dense
    c = inputs.dense_inputs(batch=1, heads=2, seq_q=256, seq_k=384, head_dim=128, seed=830, scale=0.5, causal=True,
                            bias=True)
    em = inputs.elem_mask_inputs(batch=1, heads=2, seq_q=256, seq_k=384, seed=830, kind="docs", doc_lo=30,
                                 doc_hi=120, full_rows=2)
    emt = torch.from_numpy(em).cuda()
    full = _run(bd, c, False, True, elem=emt)
    dq_only = _run(bd, c, False, True, wrt=1, elem=emt)
    assert dq_only[1] is None and dq_only[2] is None
    assert torch.equal(dq_only[0], full[0])
    _close(full, attn_bwd_dense(c.q, c.k, c.v, c.dy, causal=True, bias=c.bias, elem_mask=em))


def test_store_ds_full_size_sampled(bd):
    """The headline shape with the option, in the launch configuration the
    bench times; the oracle evaluates three (batch, head) pairs."""
    from oracle import attn_bwd_dense
    c = inputs.dense_config("dense_bf16_s2048")
    res = _run(bd, c, False, True)
    heads = [(0, 0), (1, 7), (3, 15)]
    ref = attn_bwd_dense(c.q, c.k, c.v, c.dy, layout=c.layout, causal=c.causal, window=c.window,
                         key_mask=c.key_mask, bias=c.bias, heads_subset=heads)
    for b, h in heads:
        _close([x[b, :, h] for x in res], [x[b, :, h] for x in ref])
    again = _run(bd, c, False, True)
    assert all(torch.equal(x, y) for x, y in zip(res, again))


def test_store_ds_with_o_lse_and_strided_views(bd):
    """O and LSE supplied (delta from dY . O) with stored dS, and the same call
    on q, k, v and dq, dk, dv as interleaved views of fused [B, S, 3, H, D]
    tensors: the strided call matches the contiguous one bit for bit, and both
    match the oracle."""
    from oracle import attn_bwd_dense, attn_fwd_dense
    c = inputs.dense_inputs(batch=2, heads=2, seq_q=256, seq_k=256, head_dim=128, seed=840, scale=0.5, causal=True,
                            key_mask_zero_frac=0.1, bias=True)
    o, lse = attn_fwd_dense(c.q, c.k, c.v, causal=True, key_mask=c.key_mask, bias=c.bias)
    q, k, v, dy = (_dev(x) for x in (c.q, c.k, c.v, c.dy))
    km = torch.from_numpy(c.key_mask).cuda()
    bi = _dev(c.bias)
    o_t = _dev(o.astype(np.float32))
    lse_t = torch.from_numpy(lse.astype(np.float32)).cuda().contiguous()
    a = bd.dense_backward(q, k, v, dy, causal=True, key_mask=km, bias=bi, o=o_t, lse=lse_t, store_ds=True)
    fused = torch.stack([q, k, v], dim=2).contiguous()  # [B, S, 3, H, D]
    grads = torch.empty_like(fused)
    outs = (grads[:, :, 0], grads[:, :, 1], grads[:, :, 2])
    b = bd.dense_backward(fused[:, :, 0], fused[:, :, 1], fused[:, :, 2], dy, causal=True, key_mask=km, bias=bi,
                          o=o_t, lse=lse_t, store_ds=True, outputs=outs)
    bd.check_device_error()
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    _close(a, attn_bwd_dense(c.q, c.k, c.v, c.dy, causal=True, key_mask=c.key_mask, bias=c.bias))


@pytest.mark.parametrize("window", [None, 128])
def test_many_items_per_cta(bd, window):
    """40 heads x 9 key tiles = 360 items for the persistent dK/dV kernel's
    152 CTAs, so each CTA walks two or three items (its producer, statistics
    and compute warps in step across item switches); with the window, the six
    key tiles before the window hold no visible query (items with no tile).
    Ragged Sq and Sk (a bias needs Sk * 2 bytes to be a multiple of 16), key
    mask and bias; both dQ paths against the oracle, dK and dV
    bit-identical between them."""
    from oracle import attn_bwd_dense
    c = inputs.dense_inputs(batch=2, heads=20, seq_q=200, seq_k=1096, head_dim=128, layout="bshd", seed=870,
                            scale=0.5, causal=True, window=window, key_mask_zero_frac=0.1, bias=True)
    ref = attn_bwd_dense(c.q, c.k, c.v, c.dy, layout="bshd", causal=True, window=window, key_mask=c.key_mask,
                         bias=c.bias)
    res = _run(bd, c, False, True)
    _close(res, ref)
    base = _run(bd, c, False, False)
    _close(base, ref)
    assert torch.equal(res[1], base[1]) and torch.equal(res[2], base[2])
