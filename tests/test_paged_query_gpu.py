"""GPU parity of the query side of the paged backward (row statistics and dQ,
plus dQp for MLA, in one call) with the CPU oracle (dense re-expansion), plus bit
stability, rows outside every sequence and the full GQA configuration on
sampled sequences.  Tolerance: 2e-2 * max|ref| (bf16 dQ), 2e-2 absolute on
the LSE."""
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


def to_dev(c, bd, q=None, dy=None, q_start=None, q_pos=None):
    t = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda().to(torch.bfloat16)
    dev = dict(q=t(c.q if q is None else q), dy=t(c.dy if dy is None else dy), k=t(c.k_pool), v=t(c.v_pool))
    dev["table"] = torch.from_numpy(c.page_table).cuda().contiguous()
    dev["meta"] = bd.seq_meta_tensor(c.seq_len, c.q_start if q_start is None else q_start,
                                     c.q_pos if q_pos is None else q_pos, "cuda")
    return dev


def gpu_query(bd, c, dv):
    return bd.paged_query_backward(dv["q"], dv["k"], dv["v"], dv["dy"], dv["table"], dv["meta"], heads=c.heads,
                                   kv_heads=c.kv_heads, page_size=c.page_size, causal=c.causal)


def oracle(c, q=None, dy=None, q_start=None, q_pos=None):
    from oracle import paged_query_backward
    return paged_query_backward(c.q if q is None else q, c.dy if dy is None else dy, c.k_pool, c.page_table,
                                c.seq_len, c.q_start if q_start is None else q_start,
                                c.q_pos if q_pos is None else q_pos, page_size=c.page_size, kv_heads=c.kv_heads,
                                v_pool=c.v_pool, causal=c.causal)


def rel(got, want):
    g = got.float().cpu().numpy().astype(np.float64)
    return np.max(np.abs(g - want)) / max(np.max(np.abs(want)), 1e-30)


def check(lse, delta, dq, ref):
    lse_ref, delta_ref, dq_ref = ref
    fin = np.isfinite(lse_ref)
    got_lse = lse.cpu().numpy()
    assert np.max(np.abs(got_lse[fin] - lse_ref[fin])) < 2e-2
    assert np.all(np.isneginf(got_lse[~fin]))
    assert rel(delta, delta_ref) < TOL
    assert rel(dq, dq_ref) < TOL
    assert torch.isfinite(dq).all()


CASES = [
    dict(seed=41, num_seqs=5, len_lo=20, len_hi=300, queries_per_seq=40, heads=8, kv_heads=2, key_dim=128,
         value_dim=128, causal=True),
    dict(seed=42, num_seqs=4, len_lo=100, len_hi=520, queries_per_seq=64, heads=32, kv_heads=8, key_dim=128,
         value_dim=128, causal=True),
    dict(seed=43, num_seqs=3, len_lo=5, len_hi=200, queries_per_seq=20, heads=4, kv_heads=4, key_dim=64,
         value_dim=64, causal=False),
    dict(seed=44, num_seqs=4, len_lo=40, len_hi=260, queries_per_seq=24, heads=8, kv_heads=2, key_dim=128,
         value_dim=128, causal=True, shared_prefix_pages=3),
    # short sequences: one partial 64-token tile, ragged last page
    dict(seed=45, num_seqs=6, len_lo=9, len_hi=40, queries_per_seq=8, heads=16, kv_heads=4, key_dim=128,
         value_dim=128, causal=True),
]


@pytest.mark.parametrize("kw", CASES, ids=lambda k: f"seed{k['seed']}")
def test_paged_query_parity(bd, kw):
    c = inputs.paged_case(name="t", scale=0.5, **kw)
    dv = to_dev(c, bd)
    lse, delta, dq = gpu_query(bd, c, dv)
    bd.check_device_error()
    check(lse, delta, dq, oracle(c))


def test_paged_query_matches_row_stats(bd):
    """The statistics of the query-side call equal those of the row-statistics
    call bit for bit (same sweep, same order)."""
    c = inputs.paged_case(name="t", seed=46, num_seqs=4, len_lo=30, len_hi=400, queries_per_seq=32, heads=8,
                          kv_heads=2, key_dim=128, value_dim=128, scale=0.5)
    dv = to_dev(c, bd)
    lse, delta, _ = gpu_query(bd, c, dv)
    lse2, delta2 = bd.paged_row_stats(dv["q"], dv["k"], dv["v"], dv["dy"], dv["table"], dv["meta"],
                                      heads=c.heads, kv_heads=c.kv_heads, page_size=c.page_size, causal=c.causal)
    bd.check_device_error()
    assert torch.equal(lse, lse2) and torch.equal(delta, delta2)


def test_paged_query_rows_outside_sequences(bd):
    """Rows before the first sequence's rows and after the last one get dQ = 0,
    lse = -inf and delta = 0; the others match the oracle."""
    c = inputs.paged_case(name="t", seed=47, num_seqs=3, len_lo=20, len_hi=150, queries_per_seq=10, heads=8,
                          kv_heads=2, key_dim=128, value_dim=128, scale=0.5)
    pre, post = 3, 2
    rng = np.random.default_rng(5)
    pad = lambda x: np.concatenate([rng.standard_normal((pre,) + x.shape[1:]).astype(x.dtype), x,
                                    rng.standard_normal((post,) + x.shape[1:]).astype(x.dtype)])
    q, dy = pad(c.q), pad(c.dy)
    q_start = (c.q_start + pre).astype(np.int32)
    q_pos = np.concatenate([np.zeros(pre, np.int32), c.q_pos, np.zeros(post, np.int32)]).astype(np.int32)
    dv = to_dev(c, bd, q=q, dy=dy, q_start=q_start, q_pos=q_pos)
    lse, delta, dq = bd.paged_query_backward(dv["q"], dv["k"], dv["v"], dv["dy"], dv["table"], dv["meta"],
                                             heads=c.heads, kv_heads=c.kv_heads, page_size=c.page_size,
                                             causal=c.causal)
    bd.check_device_error()
    outside = np.r_[0:pre, q.shape[0] - post:q.shape[0]]
    assert torch.all(dq[outside] == 0)
    assert torch.all(torch.isneginf(lse[outside])) and torch.all(delta[outside] == 0)
    check(lse, delta, dq, oracle(c, q=q, dy=dy, q_start=q_start, q_pos=q_pos))


def test_paged_query_bit_stable(bd):
    c = inputs.paged_case(name="t", seed=48, num_seqs=6, len_lo=50, len_hi=700, queries_per_seq=64, heads=32,
                          kv_heads=8, key_dim=128, value_dim=128, scale=0.5, shared_prefix_pages=2)
    dv = to_dev(c, bd)
    first = gpu_query(bd, c, dv)
    for _ in range(3):
        again = gpu_query(bd, c, dv)
        for a, b in zip(first, again):
            assert torch.equal(a, b)
    bd.check_device_error()


MLA_CASES = [
    dict(seed=51, num_seqs=4, len_lo=20, len_hi=300, queries_per_seq=16, heads=8, kv_heads=1, causal=True),
    dict(seed=52, num_seqs=3, len_lo=30, len_hi=200, queries_per_seq=12, heads=8, kv_heads=2, causal=False),
    dict(seed=53, num_seqs=4, len_lo=40, len_hi=200, queries_per_seq=8, heads=32, kv_heads=1, causal=True,
         shared_prefix_pages=2),
    dict(seed=54, num_seqs=5, len_lo=9, len_hi=45, queries_per_seq=5, heads=16, kv_heads=1, causal=True),
]


def mla_dev(c, bd):
    t = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda().to(torch.bfloat16)
    dev = dict(q=t(c.q), qp=t(c.qp), dy=t(c.dy), k=t(c.k_pool), kp=t(c.kp_pool))
    dev["table"] = torch.from_numpy(c.page_table).cuda().contiguous()
    dev["meta"] = bd.seq_meta_tensor(c.seq_len, c.q_start, c.q_pos, "cuda")
    return dev


@pytest.mark.parametrize("kw", MLA_CASES, ids=lambda k: f"seed{k['seed']}")
def test_paged_query_mla_parity(bd, kw):
    from oracle import paged_query_backward
    c = inputs.paged_case(name="t", scale=0.5, key_dim=512, value_dim=512, position_dim=64, **kw)
    dv = mla_dev(c, bd)
    lse, delta, dq, dqp = bd.paged_query_backward(dv["q"], dv["k"], None, dv["dy"], dv["table"], dv["meta"],
                                                  heads=c.heads, kv_heads=c.kv_heads, page_size=c.page_size,
                                                  causal=c.causal, qp=dv["qp"], kp_pool=dv["kp"])
    bd.check_device_error()
    ref = paged_query_backward(c.q, c.dy, c.k_pool, c.page_table, c.seq_len, c.q_start, c.q_pos,
                               page_size=c.page_size, kv_heads=c.kv_heads, qp=c.qp, kp_pool=c.kp_pool,
                               causal=c.causal)
    check(lse, delta, dq, ref[:3])
    assert rel(dqp, ref[3]) < TOL
    assert torch.isfinite(dqp).all()
    again = bd.paged_query_backward(dv["q"], dv["k"], None, dv["dy"], dv["table"], dv["meta"], heads=c.heads,
                                    kv_heads=c.kv_heads, page_size=c.page_size, causal=c.causal, qp=dv["qp"],
                                    kp_pool=dv["kp"])
    for a, b in zip((lse, delta, dq, dqp), again):
        assert torch.equal(a, b)


def test_paged_query_mla_unsupported_group(bd):
    """MLA head groups outside {4, 8, 16, 32} are refused, not computed."""
    c = inputs.paged_case(name="t", seed=49, num_seqs=2, len_lo=20, len_hi=60, queries_per_seq=4, heads=6,
                          kv_heads=1, key_dim=512, value_dim=512, position_dim=64, scale=0.5)
    dv = mla_dev(c, bd)
    with pytest.raises(bd.AttnError):
        bd.paged_query_backward(dv["q"], dv["k"], None, dv["dy"], dv["table"], dv["meta"], heads=c.heads,
                                kv_heads=c.kv_heads, page_size=c.page_size, causal=c.causal, qp=dv["qp"],
                                kp_pool=dv["kp"])


def test_paged_query_full_size_mla_sampled(bd):
    """The full MLA configuration; sampled sequences against the oracle."""
    c = inputs.paged_config("paged_mla")
    dv = mla_dev(c, bd)
    lse, delta, dq, dqp = bd.paged_query_backward(dv["q"], dv["k"], None, dv["dy"], dv["table"], dv["meta"],
                                                  heads=c.heads, kv_heads=c.kv_heads, page_size=c.page_size,
                                                  causal=True, qp=dv["qp"], kp_pool=dv["kp"])
    bd.check_device_error()
    from oracle import paged_query_backward
    pick = [5, 50]
    qs = [np.arange(c.q_start[s], c.q_start[s + 1]) for s in pick]
    rows = np.concatenate(qs)
    sub_start = np.concatenate([[0], np.cumsum([len(x) for x in qs])]).astype(np.int32)
    ref = paged_query_backward(c.q[rows], c.dy[rows], c.k_pool, c.page_table[pick], c.seq_len[pick], sub_start,
                               c.q_pos[rows], page_size=c.page_size, kv_heads=c.kv_heads, qp=c.qp[rows],
                               kp_pool=c.kp_pool, causal=True)
    check(lse[rows], delta[rows], dq[rows], ref[:3])
    assert rel(dqp[rows], ref[3]) < TOL


def test_paged_query_full_size_gqa_sampled(bd):
    """The full GQA configuration (64 sequences, lengths U[128,4096]); the
    oracle re-expands a sample of sequences and their rows are compared."""
    c = inputs.paged_config("paged_gqa")
    dv = to_dev(c, bd)
    lse, delta, dq = gpu_query(bd, c, dv)
    bd.check_device_error()
    from oracle import paged_query_backward
    pick = [0, 29, 63]
    qs = [np.arange(c.q_start[s], c.q_start[s + 1]) for s in pick]
    rows = np.concatenate(qs)
    sub_start = np.concatenate([[0], np.cumsum([len(x) for x in qs])]).astype(np.int32)
    ref = paged_query_backward(c.q[rows], c.dy[rows], c.k_pool, c.page_table[pick], c.seq_len[pick], sub_start,
                               c.q_pos[rows], page_size=c.page_size, kv_heads=c.kv_heads, v_pool=c.v_pool,
                               causal=True)
    check(lse[rows], delta[rows], dq[rows], ref)
