"""GPU parity of the dense forward export (attn_fwd_dense: O and LSE) with the
CPU oracle's forward, and its use as the O-and-LSE input of the backward.

Tolerances: O within 2e-2 * max|O| for bf16 storage (O is rounded to bf16) and
2e-4 * max|O| for fp32 storage; the LSE (fp32 in both) within 1e-3 + 1e-6 *
|lse|: a row whose visible keys are all custom-masked has lse = mask_neg +
log(count) = -1e9 + O(1), where fp32 spacing is 64.
"""
import numpy as np
import pytest

from attention_backward_recompute_gb300 import inputs

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def bd():
    from attention_backward_recompute_gb300 import binding, build
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    binding.lib()
    return binding


def _dev(x, dtype):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda().to(dtype)


# (B, H, Sq, Sk, D, causal, window, key-mask zero fraction, bias, layout, dtype, top_left)
CASES = [
    (2, 3, 200, 328, 128, True, None, 0.1, True, "bshd", "bf16", False),
    (1, 2, 256, 456, 128, False, 100, None, True, "bhsd", "bf16", False),
    (1, 3, 130, 264, 64, False, None, None, True, "bshd", "bf16", False),
    (2, 2, 200, 456, 128, True, None, 0.1, True, "bshd", "bf16", True),
    (1, 2, 330, 200, 128, True, None, None, False, "bshd", "bf16", False),
    (2, 4, 192, 192, 64, True, None, 0.2, False, "bshd", "f32", False),
    (1, 2, 150, 96, 16, False, 30, 0.5, False, "bhsd", "f32", False),
]


def _case(case, seed):
    B, H, Sq, Sk, D, causal, window, kmz, bias, layout, dtype, top_left = case
    c = inputs.dense_inputs(batch=B, heads=H, seq_q=Sq, seq_k=Sk, head_dim=D, dtype=dtype, layout=layout, seed=seed,
                            scale=0.5, causal=causal, window=window, key_mask_zero_frac=kmz, bias=bias)
    return c, top_left


@pytest.mark.parametrize("case", CASES, ids=lambda c: "q%dk%dD%d_c%d_w%s_km%s_b%d_%s_%s_tl%d" % (
    c[2], c[3], c[4], c[5], c[6], c[7], c[8], c[9], c[10], c[11]))
def test_forward_parity(bd, case):
    from oracle import attn_fwd_dense
    c, top_left = _case(case, 300 + CASES.index(case))
    dt = torch.float32 if c.dtype == "f32" else torch.bfloat16
    q, k, v = (_dev(x, dt) for x in (c.q, c.k, c.v))
    km = None if c.key_mask is None else torch.from_numpy(c.key_mask).cuda()
    bias = None if c.bias is None else _dev(c.bias, dt)
    o, lse = bd.dense_forward(q, k, v, layout=c.layout, causal=c.causal, window=c.window, key_mask=km, bias=bias,
                              top_left=top_left)
    bd.check_device_error()
    o_ref, lse_ref = attn_fwd_dense(c.q, c.k, c.v, layout=c.layout, causal=c.causal, window=c.window,
                                    key_mask=c.key_mask, bias=c.bias, top_left=top_left)
    tol = 2e-4 if c.dtype == "f32" else 2e-2
    g = o.float().cpu().numpy().astype(np.float64)
    assert np.max(np.abs(g - o_ref)) <= tol * np.max(np.abs(o_ref))
    got = lse.cpu().numpy()
    fin = np.isfinite(lse_ref)
    assert np.all(np.abs(got[fin] - lse_ref[fin]) <= 1e-3 + 1e-6 * np.abs(lse_ref[fin]))
    assert np.all(np.isneginf(got[~fin]))


def test_forward_feeds_the_backward(bd):
    """O and LSE from the forward export, given to the backward in its
    O-and-LSE mode, reproduce the self-contained backward within tolerance."""
    c = inputs.dense_inputs(batch=2, heads=2, seq_q=256, seq_k=320, head_dim=128, dtype="bf16", seed=311,
                            scale=0.5, causal=True, key_mask_zero_frac=0.1, bias=True)
    q, k, v, dy = (_dev(x, torch.bfloat16) for x in (c.q, c.k, c.v, c.dy))
    km = torch.from_numpy(c.key_mask).cuda()
    bias = _dev(c.bias, torch.bfloat16)
    o, lse = bd.dense_forward(q, k, v, causal=True, key_mask=km, bias=bias)
    a = bd.dense_backward(q, k, v, dy, causal=True, key_mask=km, bias=bias, o=o, lse=lse)
    b = bd.dense_backward(q, k, v, dy, causal=True, key_mask=km, bias=bias)
    bd.check_device_error()
    for x, y in zip(a, b):
        xf, yf = x.float(), y.float()
        assert float((xf - yf).abs().max()) <= 2e-2 * float(yf.abs().max())


def test_forward_without_keys(bd):
    q = torch.randn(1, 64, 2, 64, device="cuda").to(torch.bfloat16)
    k = torch.zeros(1, 0, 2, 64, device="cuda", dtype=torch.bfloat16)
    o = torch.full_like(q, 7.0)
    lse = torch.zeros(1, 2, 64, device="cuda")
    bd.dense_forward(q, k, k.clone(), outputs=(o, lse))
    bd.check_device_error()
    assert torch.all(o == 0) and torch.all(torch.isneginf(lse))
