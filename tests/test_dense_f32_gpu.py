"""GPU parity of the dense backward for fp32 storage (operands split into
hi + lo bf16, three products per GEMM) with the CPU oracle.  Tolerance
(stated by the method's acceptance criterion for f32): per output tensor,
max|gpu - oracle| <= 2e-4 * max|oracle|."""
import numpy as np
import pytest

from attention_backward_recompute_gb300 import inputs

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

TOL_F32 = 2e-4


@pytest.fixture(scope="module")
def bd():
    from attention_backward_recompute_gb300 import binding, build
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    binding.lib()
    return binding


def run(bd, c, o=None, lse=None):
    t = lambda x: torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).cuda()
    km = None if c.key_mask is None else t(c.key_mask)
    res = bd.dense_backward(t(c.q), t(c.k), t(c.v), t(c.dy), layout=c.layout, causal=c.causal, window=c.window,
                            key_mask=km, o=o, lse=lse)
    bd.check_device_error()
    return res


def oracle(c):
    from oracle import attn_bwd_dense
    return attn_bwd_dense(c.q, c.k, c.v, c.dy, layout=c.layout, causal=c.causal, window=c.window,
                          key_mask=c.key_mask)


def check(res, ref, tol=TOL_F32):
    # An exactly-zero reference (e.g. dQ with a single key, where dS = P (dP - delta)
    # cancels exactly) is measured against the largest gradient of the same call.
    scale = max(float(np.max(np.abs(w))) for w in ref)
    for n, g, w in zip(("dq", "dk", "dv"), res, ref):
        g = g.cpu().numpy().astype(np.float64)
        den = np.max(np.abs(w)) if np.max(np.abs(w)) > 0 else scale
        e = np.max(np.abs(g - w)) / den
        assert e <= tol, f"{n}: max-abs-err / max|ref| = {e:.3e} > {tol}"


@pytest.mark.parametrize("name", ["dense_small_f32", "dense_f32_causal", "dense_f32_window"])
def test_f32_configs(bd, name):
    c = inputs.dense_config(name)
    check(run(bd, c), oracle(c))


@pytest.mark.parametrize("kw", [
    dict(batch=2, heads=3, seq_q=130, seq_k=200, head_dim=64, causal=True, key_mask_zero_frac=0.2),
    dict(batch=1, heads=2, seq_q=200, seq_k=70, head_dim=32, window=20, layout="bhsd"),
    dict(batch=1, heads=2, seq_q=64, seq_k=96, head_dim=8),
    dict(batch=1, heads=1, seq_q=1, seq_k=1, head_dim=16),
], ids=["causal_km_d64", "window_bhsd_d32", "d8", "single"])
def test_f32_shapes(bd, kw):
    c = inputs.dense_inputs(dtype="f32", seed=91, **kw)
    check(run(bd, c), oracle(c))


def test_f32_o_lse_supplied(bd):
    from oracle import attn_fwd_dense
    c = inputs.dense_inputs(batch=1, heads=2, seq_q=256, seq_k=256, head_dim=64, dtype="f32", seed=93, causal=True)
    o, lse = attn_fwd_dense(c.q, c.k, c.v, causal=True)
    check(run(bd, c, o=torch.from_numpy(np.ascontiguousarray(o, dtype=np.float32)).cuda(),
              lse=torch.from_numpy(np.ascontiguousarray(lse, dtype=np.float32)).cuda()), oracle(c))
