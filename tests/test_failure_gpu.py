"""Failure detection on the GPU without a fault.

Every spin of the library's kernels on an mbarrier is bounded: when a wait runs
out it sets the device error word and the kernel returns, so the host sees
ATTN_ERR_TIMEOUT instead of a hung GPU.  attn_selftest_wait_timeout launches
one warp whose wait can never complete (nothing arrives on its barrier); the
test checks that the host reads the timeout, that the check clears it, and that
the context still runs a dense backward that matches the oracle.
"""
import time

import numpy as np
import pytest

from attention_backward_recompute_gb300 import inputs

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


def test_bounded_wait_reports_timeout_and_context_survives(bd):
    stream = torch.cuda.current_stream().cuda_stream
    assert bd.attn_check_device_error(stream) == bd.ATTN_OK  # start clean

    t0 = time.monotonic()
    assert bd.attn_selftest_wait_timeout(stream) == bd.ATTN_OK
    assert bd.attn_check_device_error(stream) == bd.ATTN_ERR_TIMEOUT
    elapsed = time.monotonic() - t0
    assert 0.5 < elapsed < 30.0, elapsed  # one bounded wait (about a second), not a hang
    assert bd.attn_check_device_error(stream) == bd.ATTN_OK  # the check cleared the word

    # the context is still usable: a small dense backward matches the oracle
    from oracle import attn_bwd_dense
    c = inputs.dense_inputs(batch=1, heads=2, seq_q=80, seq_k=96, head_dim=64, seed=11, scale=0.5,
                            causal=True, key_mask_zero_frac=0.2, bias=True)
    dev = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda().to(torch.bfloat16)
    km = torch.from_numpy(c.key_mask).cuda()
    res = bd.dense_backward(dev(c.q), dev(c.k), dev(c.v), dev(c.dy), causal=True, key_mask=km, bias=dev(c.bias))
    bd.check_device_error()
    ref = attn_bwd_dense(c.q, c.k, c.v, c.dy, causal=True, key_mask=c.key_mask, bias=c.bias)
    for got, want in zip(res, ref):
        err = np.max(np.abs(got.float().cpu().numpy().astype(np.float64) - want)) / np.max(np.abs(want))
        assert err <= TOL_BF16, err
