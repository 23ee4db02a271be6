"""GPU parity of the dense backward (C ABI -> sm_103a kernels) with the CPU oracle.

Tolerance (stated by the method's acceptance criterion): per output tensor,
max|gpu - oracle| <= 2e-2 * max|oracle| for bf16 storage.  Inputs are the
seeded synthetic draws of ``attention_backward_recompute_gb300.inputs``; the
oracle reads exactly the bf16-rounded values the GPU reads.
"""
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


def _dev(x, dtype=torch.bfloat16):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda().to(dtype)


def run_gpu(bd, c, wrt=7, o=None, lse=None, outputs=None):
    q, k, v, dy = (_dev(x) for x in (c.q, c.k, c.v, c.dy))
    km = None if c.key_mask is None else torch.from_numpy(c.key_mask).cuda()
    bias = None if c.bias is None else _dev(c.bias)
    res = bd.dense_backward(q, k, v, dy, layout=c.layout, causal=c.causal, window=c.window, key_mask=km,
                            bias=bias, o=o, lse=lse, wrt=wrt, outputs=outputs)
    bd.check_device_error()
    return res


def oracle(c, heads=None):
    from oracle import attn_bwd_dense
    return attn_bwd_dense(c.q, c.k, c.v, c.dy, layout=c.layout, causal=c.causal, window=c.window,
                          key_mask=c.key_mask, bias=c.bias, heads_subset=heads)


def rel_err(got, want, floor=0.0):
    g = got.float().cpu().numpy().astype(np.float64)
    return np.max(np.abs(g - want)) / max(np.max(np.abs(want)), floor, 1e-30)


def assert_close(res, ref, tol=TOL_BF16, names=("dq", "dk", "dv")):
    # An exactly-zero reference (e.g. dQ with a single key, where dS = P (dP - delta)
    # cancels exactly) is measured against the largest gradient of the same call.
    scale = max(float(np.max(np.abs(w))) if w.size else 0.0 for w in ref)
    for n, g, w in zip(names, res, ref):
        if g is None:
            continue
        e = rel_err(g, w, scale if np.max(np.abs(w)) == 0 else 0.0)
        assert e <= tol, f"{n}: max-abs-err / max|ref| = {e:.3e} > {tol}"


# (B, H, Sq, Sk, D, causal, window, key-mask zero fraction, bias, layout)
CASES = [
    (2, 3, 200, 328, 128, False, None, None, False, "bshd"),
    (2, 3, 200, 328, 128, True, None, None, False, "bshd"),
    (1, 2, 330, 200, 128, True, None, None, False, "bshd"),
    (2, 2, 256, 256, 128, True, None, 0.3, True, "bshd"),
    (1, 2, 300, 300, 128, False, 37, None, False, "bshd"),
    (1, 2, 256, 456, 128, False, 100, None, True, "bhsd"),
    (2, 2, 192, 192, 64, True, None, 0.2, False, "bhsd"),
    (1, 3, 130, 264, 64, False, None, None, True, "bshd"),
    (1, 2, 77, 513, 32, True, None, None, False, "bshd"),
    (1, 2, 150, 96, 16, False, None, 0.5, False, "bhsd"),
    (1, 1, 1, 1, 128, False, None, None, False, "bshd"),
    (1, 1, 5, 700, 128, True, None, None, False, "bhsd"),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B%dH%dq%dk%dD%d_c%d_w%s_km%s_b%d_%s" % (
    c[0], c[1], c[2], c[3], c[4], c[5], c[6], c[7], c[8], c[9]))
def test_parity_small(bd, case):
    B, H, Sq, Sk, D, causal, window, kmz, bias, layout = case
    c = inputs.dense_inputs(batch=B, heads=H, seq_q=Sq, seq_k=Sk, head_dim=D, dtype="bf16", layout=layout,
                            seed=100 + CASES.index(case), scale=0.5, causal=causal, window=window,
                            key_mask_zero_frac=kmz, bias=bias)
    assert_close(run_gpu(bd, c), oracle(c))


@pytest.mark.parametrize("name,heads", [
    ("dense_bf16_s2048", [(0, 0), (1, 7), (3, 15)]),
    ("dense_bf16_cross", [(0, 0), (5, 9), (7, 15)]),
])
def test_parity_full_size_sampled_heads(bd, name, heads):
    """Full-size configurations, in the launch configuration the bench times;
    the oracle evaluates a sample of (batch, head) pairs."""
    c = inputs.dense_config(name)
    res = run_gpu(bd, c)
    ref = oracle(c, heads=heads)
    for b, h in heads:
        got = [x[b, :, h] for x in res]
        want = [x[b, :, h] for x in ref]
        assert_close(got, want)


def test_wrt_subsets_bit_identical(bd):
    c = inputs.dense_inputs(batch=1, heads=2, seq_q=200, seq_k=264, head_dim=128, dtype="bf16", seed=21,
                            scale=0.5, causal=True, key_mask_zero_frac=0.1, bias=True)
    full = run_gpu(bd, c, wrt=7)
    for wrt in (1, 2, 4, 3, 5, 6):
        part = run_gpu(bd, c, wrt=wrt)
        for i, bit in enumerate((1, 2, 4)):
            if wrt & bit:
                assert torch.equal(part[i], full[i]), (wrt, i)
            else:
                assert part[i] is None


def test_deterministic(bd):
    c = inputs.dense_config("dense_bf16_s2048", batch=1, heads=4)
    a = run_gpu(bd, c)
    b = run_gpu(bd, c)
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_o_lse_supplied_mode(bd):
    """With O (bf16) and LSE from a forward, only rowsum(dY * O) is recomputed."""
    from oracle import attn_fwd_dense
    c = inputs.dense_inputs(batch=2, heads=2, seq_q=256, seq_k=320, head_dim=128, dtype="bf16", seed=31,
                            scale=0.5, causal=True, key_mask_zero_frac=0.1, bias=True)
    o, lse = attn_fwd_dense(c.q, c.k, c.v, causal=True, key_mask=c.key_mask, bias=c.bias)
    o_t = _dev(o.astype(np.float32))
    lse_t = torch.from_numpy(lse.astype(np.float32)).cuda().contiguous()
    assert_close(run_gpu(bd, c, o=o_t, lse=lse_t), oracle(c))


@pytest.mark.parametrize("n_masked,bias", [(5, False), (40, True), (130, True)])
def test_fully_custom_masked_rows(bd, n_masked, bias):
    """The first keys are custom-masked, so under the causal mask the first
    rows see only masked keys: their softmax is uniform over the visible keys
    (whatever the bias).  40 and 130 masked keys span several column groups
    and a whole 128-key tile."""
    c = inputs.dense_inputs(batch=1, heads=2, seq_q=256, seq_k=256, head_dim=128, dtype="bf16", seed=41,
                            scale=0.5, causal=True, key_mask_zero_frac=0.0, bias=bias)
    c.key_mask[0, :n_masked] = 0.0
    assert_close(run_gpu(bd, c), oracle(c))


def test_rows_without_visible_keys(bd):
    """Sq > Sk with a narrow window: rows q >= Sk + w see no key; their dQ is 0."""
    c = inputs.dense_inputs(batch=1, heads=2, seq_q=300, seq_k=96, head_dim=64, dtype="bf16", seed=51,
                            scale=0.5, window=10)
    res = run_gpu(bd, c)
    assert_close(res, oracle(c))
    assert torch.all(res[0][:, 110:] == 0)


def test_zero_size_dims(bd):
    for sq, sk in ((0, 64), (64, 0)):
        c = inputs.dense_inputs(batch=1, heads=2, seq_q=sq, seq_k=sk, head_dim=64, dtype="bf16", seed=1)
        q = torch.zeros((1, sq, 2, 64), dtype=torch.bfloat16, device="cuda")
        k = torch.zeros((1, sk, 2, 64), dtype=torch.bfloat16, device="cuda")
        outs = (torch.full_like(q, 7.0), torch.full_like(k, 7.0), torch.full_like(k, 7.0))
        bd.dense_backward(q, k, k.clone(), q.clone(), outputs=outs)
        bd.check_device_error()
        for t in outs:
            assert t.numel() == 0 or torch.all(t == 0)


def test_guard_bands_untouched(bd):
    """Outputs live inside larger buffers whose margins hold a NaN pattern;
    the kernels must write exactly the output elements."""
    c = inputs.dense_inputs(batch=1, heads=2, seq_q=200, seq_k=136, head_dim=64, dtype="bf16", seed=61,
                            scale=0.5, causal=True)
    pad = 4096
    outs, views = [], []
    for shape in ((1, 200, 2, 64), (1, 136, 2, 64), (1, 136, 2, 64)):
        n = int(np.prod(shape))
        buf = torch.full((n + 2 * pad,), float("nan"), dtype=torch.bfloat16, device="cuda")
        outs.append(buf)
        views.append(buf[pad:pad + n].view(shape))
    res = run_gpu(bd, c, outputs=tuple(views))
    assert_close(res, oracle(c))
    for buf in outs:
        assert torch.all(torch.isnan(buf[:pad])) and torch.all(torch.isnan(buf[-pad:]))


def test_error_word_clear_after_normal_runs(bd):
    c = inputs.dense_inputs(batch=1, heads=1, seq_q=64, seq_k=64, head_dim=64, dtype="bf16", seed=3)
    run_gpu(bd, c)
    assert bd.attn_check_device_error(None) == bd.ATTN_OK


@pytest.mark.parametrize("sq,sk,causal,window,dim", [(200, 456, True, None, 128), (330, 200, True, None, 128),
                                                       (190, 296, False, 40, 64)])
def test_top_left_alignment(bd, sq, sk, causal, window, dim):
    """ATTN_MASK_TOP_LEFT: causal / window masks aligned top-left (row q sees
    keys <= q); Sq < Sk leaves keys that no query sees, whose dK, dV are 0."""
    from oracle import attn_bwd_dense
    c = inputs.dense_inputs(batch=2, heads=2, seq_q=sq, seq_k=sk, head_dim=dim, dtype="bf16", seed=81,
                            scale=0.5, causal=causal, window=window, key_mask_zero_frac=0.1, bias=True)
    q, k, v, dy = (_dev(x) for x in (c.q, c.k, c.v, c.dy))
    km = torch.from_numpy(c.key_mask).cuda()
    res = bd.dense_backward(q, k, v, dy, layout=c.layout, causal=causal, window=window, key_mask=km,
                            bias=_dev(c.bias), top_left=True)
    bd.check_device_error()
    ref = attn_bwd_dense(c.q, c.k, c.v, c.dy, layout=c.layout, causal=causal, window=window,
                         key_mask=c.key_mask, bias=c.bias, top_left=True)
    assert_close(res, ref)
    if sq < sk and window is None:
        assert torch.all(res[1][:, sq:] == 0) and torch.all(res[2][:, sq:] == 0)


def test_strided_views_match_contiguous(bd):
    """q, k, v as views of one fused [B, S, 3, H, D] tensor and dq, dk, dv
    written into one fused gradient tensor give bit-identical results to the
    contiguous call (attn_bwd_dense_strided)."""
    c = inputs.dense_inputs(batch=2, heads=3, seq_q=320, seq_k=320, head_dim=128, dtype="bf16", seed=91,
                            scale=0.5, causal=True, key_mask_zero_frac=0.1, bias=True)
    qkv = torch.stack([_dev(c.q), _dev(c.k), _dev(c.v)], dim=2)  # [B, S, 3, H, D]
    q, k, v = qkv[:, :, 0], qkv[:, :, 1], qkv[:, :, 2]
    assert not q.is_contiguous()
    dy = _dev(c.dy)
    km = torch.from_numpy(c.key_mask).cuda()
    bias = _dev(c.bias)
    grads = torch.full_like(qkv, float("nan"))
    outs = (grads[:, :, 0], grads[:, :, 1], grads[:, :, 2])
    bd.dense_backward(q, k, v, dy, causal=True, key_mask=km, bias=bias, outputs=outs)
    ref = bd.dense_backward(q.contiguous(), k.contiguous(), v.contiguous(), dy, causal=True, key_mask=km, bias=bias)
    bd.check_device_error()
    for a, b in zip(outs, ref):
        assert torch.equal(a, b)
    # the forward export through the same views, O into a strided slice
    obuf = torch.full((2, 320, 2, 3, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    o, lse = bd.dense_forward(q, k, v, causal=True, key_mask=km, bias=bias,
                              outputs=(obuf[:, :, 1], torch.empty(2, 3, 320, device="cuda")))
    o2, lse2 = bd.dense_forward(q.contiguous(), k.contiguous(), v.contiguous(), causal=True, key_mask=km, bias=bias)
    bd.check_device_error()
    assert torch.equal(o, o2) and torch.equal(lse, lse2)
    assert torch.isnan(obuf[:, :, 0]).all()  # the other slice is untouched


@pytest.mark.parametrize("dtype,store_ds", [("bf16", False), ("bf16", True), ("f32", False)],
                         ids=["bf16", "bf16_store_ds", "f32"])
def test_outputs_at_16_byte_offsets(bd, dtype, store_ds):
    """dq, dk, dv written into views whose rows start 16 bytes past a 32-byte
    boundary (the epilogues then take their 16-byte store path instead of the
    32-byte one) are bit-identical to the contiguous call; the padding in
    front of every row is untouched."""
    bf16 = dtype == "bf16"  # (fp32 storage: head_dim <= 64, no bias)
    c = inputs.dense_inputs(batch=2, heads=3, seq_q=200, seq_k=328, head_dim=128 if bf16 else 64, dtype=dtype,
                            seed=93, scale=0.5, causal=True, key_mask_zero_frac=0.1, bias=bf16)
    tdt = torch.bfloat16 if bf16 else torch.float32
    pad = 16 // torch.tensor([], dtype=tdt).element_size()
    q, k, v, dy = (_dev(x, tdt) for x in (c.q, c.k, c.v, c.dy))
    bias = _dev(c.bias, tdt) if bf16 else None
    km = torch.from_numpy(c.key_mask).cuda()
    bufs = [torch.full(x.shape[:-1] + (x.shape[-1] + pad,), float("nan"), dtype=tdt, device="cuda")
            for x in (q, k, v)]
    outs = tuple(b[..., pad:] for b in bufs)
    assert all(o.data_ptr() % 32 == 16 for o in outs)
    bd.dense_backward(q, k, v, dy, causal=True, key_mask=km, bias=bias, outputs=outs, store_ds=store_ds)
    ref = bd.dense_backward(q, k, v, dy, causal=True, key_mask=km, bias=bias, store_ds=store_ds)
    bd.check_device_error()
    for a, b in zip(outs, ref):
        assert torch.equal(a, b)
    for b in bufs:
        assert torch.isnan(b[..., :pad]).all()


def test_strided_head_broadcast_keys(bd):
    """One key/value head shared by all query heads through a head stride of 0
    (inputs may overlap), against the materialised copy."""
    c = inputs.dense_inputs(batch=1, heads=4, seq_q=256, seq_k=384, head_dim=64, dtype="bf16", seed=92,
                            scale=0.5, causal=True)
    q, dy = _dev(c.q), _dev(c.dy)
    k1, v1 = _dev(c.k[:, :, :1]), _dev(c.v[:, :, :1])
    k, v = k1.expand(-1, -1, 4, -1), v1.expand(-1, -1, 4, -1)
    assert k.stride(2) == 0
    a = bd.dense_backward(q, k, v, dy, causal=True)
    b = bd.dense_backward(q, k.contiguous(), v.contiguous(), dy, causal=True)
    bd.check_device_error()
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_strided_overlapping_output_refused(bd):
    c = inputs.dense_inputs(batch=1, heads=2, seq_q=64, seq_k=64, head_dim=64, dtype="bf16", seed=93, scale=0.5)
    q, k, v, dy = (_dev(x) for x in (c.q, c.k, c.v, c.dy))
    dq = torch.empty(1, 1, 2, 64, dtype=torch.bfloat16, device="cuda").expand(1, 64, 2, 64)  # seq stride 0
    with pytest.raises(bd.AttnError):
        bd.dense_backward(q, k, v, dy, outputs=(dq, torch.empty_like(k), torch.empty_like(v)))
