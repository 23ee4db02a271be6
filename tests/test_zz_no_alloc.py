"""attn_bwd_dense_noalloc: the dense backward for callers that cannot
allocate device memory (plugins inside a framework that owns the device
memory, serving loops that forbid allocation on the hot path).  It keeps its
row statistics in a library-owned device array instead of a workspace.

Checked through the C ABI against attn_bwd_dense (which takes a caller
workspace) on the same inputs, for two calls in a row (the second call finds
the previous call's contents in the shared array): both run the same kernels
on the same inputs, so the outputs must be bit-identical.  One case is also
compared with the CPU oracle, within the parity tolerance of the dense tests.  This file is collected last so that a run that
stops at the first failure has already run every other test; it also passes
alone in a fresh process.
"""
import ctypes

import numpy as np
import pytest

from attention_backward_recompute_gb300 import inputs
from oracle import attn_bwd_dense as oracle_bwd

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

TOL_BF16 = 2e-2


@pytest.fixture(scope="module")
def bd():
    from attention_backward_recompute_gb300 import binding, build
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    binding.lib()
    return binding


def _dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda().to(torch.bfloat16)


def _rel(a, b):
    a = a.float().cpu().numpy().astype(np.float64)
    b = b.float().cpu().numpy().astype(np.float64)
    return np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-30)


@pytest.mark.parametrize("seed,causal,kmz,bias", [(71, True, 0.1, True), (72, False, None, False)])
def test_noalloc_matches_workspace_entry_point(bd, seed, causal, kmz, bias):
    c = inputs.dense_inputs(batch=2, heads=3, seq_q=200, seq_k=264, head_dim=128, dtype="bf16", seed=seed,
                            scale=0.5, causal=causal, key_mask_zero_frac=kmz, bias=bias)
    q, k, v, dy = (_dev(x) for x in (c.q, c.k, c.v, c.dy))
    km = None if c.key_mask is None else torch.from_numpy(c.key_mask).cuda()
    bb = None if c.bias is None else _dev(c.bias)
    P = bd._ptr
    stream = bd._stream_handle(None)
    desc = bd.make_dense_desc(batch=2, heads=3, seq_q=200, seq_k=264, head_dim=128, causal=causal,
                              key_mask=km is not None, bias=bb is not None)
    # reference: the entry point with a caller workspace
    ref = [torch.empty_like(t) for t in (q, k, v)]
    ws = torch.empty(bd.attn_bwd_dense_workspace_bytes(desc), dtype=torch.uint8, device="cuda")
    st = bd.attn_bwd_dense(desc, P(q), P(k), P(v), P(dy), P(km), P(bb), None, None, P(ref[0]), P(ref[1]),
                           P(ref[2]), 7, P(ws), ws.numel(), stream)
    assert st == bd.ATTN_OK, bd.last_error()
    for call in range(2):
        out = [torch.full_like(t, float("nan")) for t in (q, k, v)]
        st = bd.attn_bwd_dense_noalloc(desc, P(q), P(k), P(v), P(dy), P(km), P(bb), None, None, P(out[0]),
                                       P(out[1]), P(out[2]), 7, stream)
        assert st == bd.ATTN_OK, bd.last_error()
        torch.cuda.synchronize()
        assert bd.attn_check_device_error(stream) == bd.ATTN_OK
        for name, a, b in zip(("dq", "dk", "dv"), out, ref):
            assert torch.equal(a, b), (f"call {call}: {name} differs from the workspace entry point "
                                       f"(max rel {_rel(a, b):.3e})")
    if seed == 71:
        want = oracle_bwd(c.q, c.k, c.v, c.dy, causal=causal, key_mask=c.key_mask, bias=c.bias)
        for name, a, w in zip(("dq", "dk", "dv"), out, want):
            g = a.float().cpu().numpy().astype(np.float64)
            e = np.max(np.abs(g - w)) / max(np.max(np.abs(w)), 1e-30)
            assert e <= TOL_BF16, f"{name} differs from the oracle by {e:.3e}"


def test_noalloc_rejects_oversized_problem(bd):
    # batch * heads * seq_q above the scratch limit is refused before any launch
    desc = bd.make_dense_desc(batch=64, heads=64, seq_q=4096, seq_k=64, head_dim=64)
    fake = ctypes.c_void_p(1 << 40)
    st = bd.attn_bwd_dense_noalloc(desc, fake, fake, fake, fake, None, None, None, None, fake, fake, fake, 7, None)
    assert st == bd.ATTN_ERR_UNSUPPORTED
    assert "scratch" in bd.last_error()
