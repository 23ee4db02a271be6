"""GPU parity of the dense backward with a per-element custom mask (the
attention_bwd.wgsl page's mask kind 2: a (query, key) pair whose mask value is
below the threshold has its score replaced by the masked value), alone and
with the per-key mask, causal / window masks and the additive bias, against
the CPU oracle.

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


# (B, H, Sq, Sk, D, causal, window, key-mask zero fraction, bias, layout, mask kind, full rows, full cols)
CASES = [
    (2, 3, 200, 328, 128, True, None, 0.1, True, "bshd", "random", 3, 3),
    (1, 2, 130, 264, 64, False, None, None, False, "bhsd", "random", 5, 0),
    (2, 2, 384, 384, 128, True, None, None, True, "bshd", "docs", 0, 0),
    (1, 3, 100, 200, 128, False, 60, 0.2, False, "bshd", "random", 0, 7),
    (1, 2, 256, 256, 64, False, None, None, True, "bshd", "docs", 2, 2),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "q%dk%dD%d_c%d_w%s_km%s_b%d_%s_%s_r%dc%d" % (
    c[2], c[3], c[4], c[5], c[6], c[7], c[8], c[9], c[10], c[11], c[12]))
def test_elem_mask_parity(bd, case):
    from oracle import attn_bwd_dense
    B, H, Sq, Sk, D, causal, window, kmz, bias, layout, kind, fr, fc = case
    seed = 700 + CASES.index(case)
    c = inputs.dense_inputs(batch=B, heads=H, seq_q=Sq, seq_k=Sk, head_dim=D, layout=layout, seed=seed, scale=0.5,
                            causal=causal, window=window, key_mask_zero_frac=kmz, bias=bias)
    em = inputs.elem_mask_inputs(batch=B, heads=H, seq_q=Sq, seq_k=Sk, seed=seed, kind=kind, full_rows=fr,
                                 full_cols=fc)
    q, k, v, dy = (_dev(x) for x in (c.q, c.k, c.v, c.dy))
    km = None if c.key_mask is None else torch.from_numpy(c.key_mask).cuda()
    bi = None if c.bias is None else _dev(c.bias)
    res = bd.dense_backward(q, k, v, dy, layout=layout, causal=causal, window=window, key_mask=km, bias=bi,
                            elem_mask=torch.from_numpy(em).cuda())
    bd.check_device_error()
    ref = attn_bwd_dense(c.q, c.k, c.v, c.dy, layout=layout, causal=causal, window=window, key_mask=c.key_mask,
                         bias=c.bias, elem_mask=em)
    _close(res, ref)


def test_elem_mask_all_ones_is_no_mask(bd):
    """A mask that masks nothing gives bit-identical gradients to no mask."""
    c = inputs.dense_inputs(batch=1, heads=2, seq_q=192, seq_k=320, head_dim=128, seed=710, scale=0.5, causal=True,
                            key_mask_zero_frac=0.1, bias=True)
    q, k, v, dy = (_dev(x) for x in (c.q, c.k, c.v, c.dy))
    km = torch.from_numpy(c.key_mask).cuda()
    bi = _dev(c.bias)
    ones = torch.ones(1, 2, 192, 320, device="cuda")
    a = bd.dense_backward(q, k, v, dy, causal=True, key_mask=km, bias=bi, elem_mask=ones)
    b = bd.dense_backward(q, k, v, dy, causal=True, key_mask=km, bias=bi)
    bd.check_device_error()
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_elem_mask_equals_key_mask(bd):
    """A per-element mask that repeats the per-key mask on every query row gives
    the per-key mask's gradients bit for bit."""
    c = inputs.dense_inputs(batch=2, heads=2, seq_q=160, seq_k=200, head_dim=64, seed=711, scale=0.5,
                            key_mask_zero_frac=0.3)
    q, k, v, dy = (_dev(x) for x in (c.q, c.k, c.v, c.dy))
    km = torch.from_numpy(c.key_mask).cuda()
    em = km[:, None, None, :].expand(2, 2, 160, 200).contiguous()
    a = bd.dense_backward(q, k, v, dy, elem_mask=em)
    b = bd.dense_backward(q, k, v, dy, key_mask=km)
    bd.check_device_error()
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_elem_mask_with_given_o_lse(bd):
    """O and LSE of the masked forward (from the oracle), given to the backward
    in its O-and-LSE mode."""
    from oracle import attn_bwd_dense, attn_fwd_dense
    c = inputs.dense_inputs(batch=1, heads=2, seq_q=256, seq_k=256, head_dim=128, seed=712, scale=0.5, causal=True)
    em = inputs.elem_mask_inputs(batch=1, heads=2, seq_q=256, seq_k=256, seed=712, kind="docs", doc_lo=20, doc_hi=90)
    o_ref, lse_ref = attn_fwd_dense(c.q, c.k, c.v, causal=True, elem_mask=em)
    q, k, v, dy = (_dev(x) for x in (c.q, c.k, c.v, c.dy))
    res = bd.dense_backward(q, k, v, dy, causal=True, elem_mask=torch.from_numpy(em).cuda(), o=_dev(o_ref),
                            lse=torch.from_numpy(lse_ref.astype(np.float32)).cuda())
    bd.check_device_error()
    _close(res, attn_bwd_dense(c.q, c.k, c.v, c.dy, causal=True, elem_mask=em))
