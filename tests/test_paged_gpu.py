"""GPU parity of the paged history backward and the paged row statistics with
the CPU oracle (dense re-expansion), plus bit stability and the zero store of
slots no valid token owns.  Tolerance: 2e-2 * max|ref| per output (bf16)."""
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


def to_dev(c, bd):
    t = lambda x: None if x is None else torch.from_numpy(np.ascontiguousarray(x)).cuda().to(torch.bfloat16)
    dev = dict(q=t(c.q), dy=t(c.dy), k=t(c.k_pool), v=t(c.v_pool), qp=t(c.qp), kp=t(c.kp_pool))
    dev["table"] = torch.from_numpy(c.page_table).cuda().contiguous()
    dev["meta"] = bd.seq_meta_tensor(c.seq_len, c.q_start, c.q_pos, "cuda")
    return dev


def gpu_stats(bd, c, dv):
    return bd.paged_row_stats(dv["q"], dv["k"], dv["v"], dv["dy"], dv["table"], dv["meta"], heads=c.heads,
                              kv_heads=c.kv_heads, page_size=c.page_size, causal=c.causal, qp=dv["qp"],
                              kp_pool=dv["kp"])


def gpu_bwd(bd, c, dv, lse, delta, outputs=None):
    return bd.paged_backward(dv["q"], dv["k"], dv["v"], dv["dy"], dv["table"], dv["meta"], lse, delta,
                             heads=c.heads, kv_heads=c.kv_heads, page_size=c.page_size, causal=c.causal,
                             outputs=outputs, qp=dv["qp"], kp_pool=dv["kp"])


def oracle(c):
    from oracle import attn_bwd_paged
    return attn_bwd_paged(c.q, c.dy, c.k_pool, c.page_table, c.seq_len, c.q_start, c.q_pos,
                          page_size=c.page_size, kv_heads=c.kv_heads, v_pool=c.v_pool, qp=c.qp,
                          kp_pool=c.kp_pool, causal=c.causal, return_stats=True)


def rel(got, want, mask=None):
    g = got.float().cpu().numpy().astype(np.float64)
    if mask is not None:
        g, want = g[mask], want[mask]
    return np.max(np.abs(g - want)) / max(np.max(np.abs(want)), 1e-30)


CASES = [
    dict(seed=21, num_seqs=5, len_lo=20, len_hi=300, queries_per_seq=40, heads=8, kv_heads=2, key_dim=128,
         value_dim=128, causal=True),
    dict(seed=22, num_seqs=4, len_lo=100, len_hi=520, queries_per_seq=64, heads=32, kv_heads=8, key_dim=128,
         value_dim=128, causal=True),
    dict(seed=23, num_seqs=3, len_lo=5, len_hi=200, queries_per_seq=20, heads=4, kv_heads=4, key_dim=64,
         value_dim=64, causal=False),
    dict(seed=24, num_seqs=4, len_lo=40, len_hi=260, queries_per_seq=24, heads=8, kv_heads=2, key_dim=128,
         value_dim=128, causal=True, shared_prefix_pages=3),
    # MLA: latent 512 (also the value) + position 64
    dict(seed=25, num_seqs=4, len_lo=20, len_hi=300, queries_per_seq=16, heads=8, kv_heads=1, key_dim=512,
         value_dim=512, position_dim=64, causal=True),
    dict(seed=26, num_seqs=3, len_lo=30, len_hi=200, queries_per_seq=12, heads=8, kv_heads=2, key_dim=512,
         value_dim=512, position_dim=64, causal=False),
    dict(seed=27, num_seqs=4, len_lo=40, len_hi=200, queries_per_seq=8, heads=32, kv_heads=1, key_dim=512,
         value_dim=512, position_dim=64, causal=True, shared_prefix_pages=2),
    # long shared prefixes: 20 pages (2.5 blocks of 8 pages) and 9 pages (1.1
    # blocks) shared by every sequence
    dict(seed=28, num_seqs=12, len_lo=330, len_hi=700, queries_per_seq=32, heads=16, kv_heads=4, key_dim=128,
         value_dim=128, causal=True, shared_prefix_pages=20),
    dict(seed=29, num_seqs=10, len_lo=150, len_hi=400, queries_per_seq=6, heads=16, kv_heads=1, key_dim=512,
         value_dim=512, position_dim=64, causal=True, shared_prefix_pages=9),
    # MLA blocks whose shared pages carry more than 64 link tiles go to the
    # cluster-split kernel: 11 other sequences x 12 (resp. 6) tiles each; few
    # such blocks, so each is cut into chunks summed through the workspace
    dict(seed=30, num_seqs=12, len_lo=150, len_hi=300, queries_per_seq=24, heads=32, kv_heads=1, key_dim=512,
         value_dim=512, position_dim=64, causal=True, shared_prefix_pages=9),
    dict(seed=32, num_seqs=12, len_lo=150, len_hi=300, queries_per_seq=24, heads=32, kv_heads=2, key_dim=512,
         value_dim=512, position_dim=64, causal=False, shared_prefix_pages=5),
    # a pool of ~28,800 pages, almost all unreferenced: the link build and the
    # zero store over a pool far larger than the pages in use
    dict(seed=37, num_seqs=4, len_lo=60, len_hi=200, queries_per_seq=16, heads=4, kv_heads=1, key_dim=64,
         value_dim=64, causal=True, pool_factor=800),
    # 72 flagged (block, KV head) units (9 blocks of a 72-page prefix shared by
    # 40 sequences, 8 KV heads, 39 x 2 link tiles each): enough units that the
    # split kernel takes them whole instead of cutting them into chunks, and
    # more than it lists up front (units past the 64th are found by search)
    dict(seed=34, num_seqs=40, len_lo=1160, len_hi=1230, queries_per_seq=32, heads=32, kv_heads=8, key_dim=512,
         value_dim=512, position_dim=64, causal=True, shared_prefix_pages=72),
]


@pytest.mark.parametrize("kw", CASES, ids=lambda k: f"seed{k['seed']}")
def test_paged_parity(bd, kw):
    c = inputs.paged_case(name="t", scale=0.5, **kw)
    dv = to_dev(c, bd)
    dk_ref, dv_ref, lse_ref, delta_ref = oracle(c)
    lse, delta = gpu_stats(bd, c, dv)
    bd.check_device_error()
    fin = np.isfinite(lse_ref)
    assert np.max(np.abs(lse.cpu().numpy()[fin] - lse_ref[fin])) < 2e-2
    assert rel(delta, delta_ref) < TOL
    dk, dvv = gpu_bwd(bd, c, dv, lse, delta)
    bd.check_device_error()
    assert rel(dk, dk_ref) < TOL
    assert rel(dvv, dv_ref) < TOL
    # rows of slots no valid token owns are exactly zero (pools are NaN there)
    valid = np.zeros(c.num_pages * c.page_size, bool)
    for s in range(c.num_seqs):
        for t in range(int(c.seq_len[s])):
            valid[int(c.page_table[s, t // c.page_size]) * c.page_size + t % c.page_size] = True
    assert torch.all(dk[torch.from_numpy(~valid).cuda()] == 0)
    assert torch.all(dvv[torch.from_numpy(~valid).cuda()] == 0)
    assert torch.isfinite(dk).all() and torch.isfinite(dvv).all()


@pytest.mark.parametrize("mla", [False, True], ids=["gqa", "mla"])
def test_paged_shared_at_offsets(bd, mla):
    """Shared pages at other logical positions: sequence 2 maps its logical
    pages 0..P-2 to sequence 0's physical pages 1..P-1 (links that follow one
    another at an offset) and its page P-1 to a free page; sequence 3 swaps two
    of its shared pages (links that do not follow one another)."""
    P = 11
    kw = dict(seed=41 + int(mla), num_seqs=5, len_lo=240, len_hi=420, causal=True, shared_prefix_pages=P)
    if mla:
        kw.update(queries_per_seq=6, heads=16, kv_heads=1, key_dim=512, value_dim=512, position_dim=64)
    else:
        kw.update(queries_per_seq=24, heads=8, kv_heads=2, key_dim=128, value_dim=128)
    c = inputs.paged_case(name="t", scale=0.5, **kw)
    t = c.page_table.copy()
    used = {int(t[s, lp]) for s in range(c.num_seqs) for lp in range(-(-int(c.seq_len[s]) // c.page_size))}
    free = [q for q in range(c.num_pages) if q not in used]
    t[2, :P - 1] = c.page_table[0, 1:P]
    t[2, P - 1] = free[0]
    t[3, [1, 3]] = t[3, [3, 1]]
    c.page_table = t
    src, ps = int(c.page_table[0, 0]), c.page_size  # the free page's rows: finite values of another page
    for pool in (c.k_pool, c.v_pool, c.kp_pool):
        if pool is not None:
            pool[free[0] * ps:(free[0] + 1) * ps] = pool[src * ps:(src + 1) * ps]
    dv = to_dev(c, bd)
    dk_ref, dv_ref, lse_ref, delta_ref = oracle(c)
    lse, delta = gpu_stats(bd, c, dv)
    dk, dvv = gpu_bwd(bd, c, dv, lse, delta)
    bd.check_device_error()
    assert rel(dk, dk_ref) < TOL
    assert rel(dvv, dv_ref) < TOL
    again = gpu_bwd(bd, c, dv, lse, delta)
    assert all(torch.equal(a, b) for a, b in zip((dk, dvv), again))


def test_paged_mla_split_irregular_links(bd):
    """Cluster-split MLA blocks over links that do not follow one another:
    sequence 2 maps its logical pages 0..P-2 to sequence 0's pages 1..P-1 and
    sequence 3 swaps two shared pages, so the split kernel's tile counts (taken
    by link index in the plan) meet runs of pages that break and shift."""
    P = 11
    c = inputs.paged_case(name="t", seed=36, num_seqs=12, len_lo=200, len_hi=320, queries_per_seq=24, heads=32,
                          kv_heads=1, key_dim=512, value_dim=512, position_dim=64, scale=0.5, causal=True,
                          shared_prefix_pages=P)
    t = c.page_table.copy()
    used = {int(t[s, lp]) for s in range(c.num_seqs) for lp in range(-(-int(c.seq_len[s]) // c.page_size))}
    free = [q for q in range(c.num_pages) if q not in used]
    t[2, :P - 1] = c.page_table[0, 1:P]
    t[2, P - 1] = free[0]
    t[3, [1, 3]] = t[3, [3, 1]]
    c.page_table = t
    src, ps = int(c.page_table[0, 0]), c.page_size
    for pool in (c.k_pool, c.kp_pool):
        pool[free[0] * ps:(free[0] + 1) * ps] = pool[src * ps:(src + 1) * ps]
    dv = to_dev(c, bd)
    dk_ref, dkp_ref, lse_ref, delta_ref = oracle(c)
    lse, delta = gpu_stats(bd, c, dv)
    dk, dkp = gpu_bwd(bd, c, dv, lse, delta)
    bd.check_device_error()
    assert rel(dk, dk_ref) < TOL
    assert rel(dkp, dkp_ref) < TOL
    again = gpu_bwd(bd, c, dv, lse, delta)
    assert all(torch.equal(a, b) for a, b in zip((dk, dkp), again))


def test_paged_mla_split_bit_stable(bd):
    """The cluster-split MLA blocks (8-CTA clusters on tcgen05, each block
    cut into chunks) sum their partials in a fixed order."""
    c = inputs.paged_case(name="t", seed=33, num_seqs=12, len_lo=150, len_hi=300, queries_per_seq=24, heads=32,
                          kv_heads=1, key_dim=512, value_dim=512, position_dim=64, scale=0.5, shared_prefix_pages=6)
    dv = to_dev(c, bd)
    lse, delta = gpu_stats(bd, c, dv)
    first = gpu_bwd(bd, c, dv, lse, delta)
    for _ in range(3):
        again = gpu_bwd(bd, c, dv, lse, delta)
        for a, b in zip(first, again):
            assert torch.equal(a, b)
    bd.check_device_error()


@pytest.mark.parametrize("mla", [False, True], ids=["gqa", "mla"])
def test_paged_compact_history(bd, mla):
    """Compact history: listed pages (owned, shared, unreferenced, repeated,
    in any order) get exactly the full call's rows; the other rows keep the
    caller's values."""
    kw = dict(seed=51 + int(mla), num_seqs=6, len_lo=60, len_hi=500, causal=True, shared_prefix_pages=3)
    if mla:
        kw.update(queries_per_seq=8, heads=16, kv_heads=1, key_dim=512, value_dim=512, position_dim=64)
    else:
        kw.update(queries_per_seq=32, heads=8, kv_heads=2, key_dim=128, value_dim=128)
    c = inputs.paged_case(name="t", scale=0.5, **kw)
    dv = to_dev(c, bd)
    lse, delta = gpu_stats(bd, c, dv)
    full = gpu_bwd(bd, c, dv, lse, delta)
    rng = np.random.default_rng(7)
    pages = rng.permutation(c.num_pages)[: c.num_pages // 2].astype(np.int32)
    pages = np.concatenate([pages, pages[:3], [int(c.page_table[0, 0])]]).astype(np.int32)  # repeats, a shared page
    hist = torch.from_numpy(pages).cuda()
    outs = tuple(torch.full_like(x, 3.0) for x in full)
    res = bd.paged_backward(dv["q"], dv["k"], dv["v"], dv["dy"], dv["table"], dv["meta"], lse, delta,
                            heads=c.heads, kv_heads=c.kv_heads, page_size=c.page_size, causal=c.causal,
                            qp=dv["qp"], kp_pool=dv["kp"], history_pages=hist,
                            outputs=(outs[0], None, outs[1]) if mla else (outs[0], outs[1], None))
    bd.check_device_error()
    listed = np.zeros(c.num_pages * c.page_size, bool)
    for pg in set(int(x) for x in pages):
        listed[pg * c.page_size:(pg + 1) * c.page_size] = True
    sel = torch.from_numpy(listed).cuda()
    for a, b in zip(res, full):
        assert torch.equal(a[sel], b[sel])
        assert torch.all(a[~sel] == 3.0)


def test_paged_bit_stable(bd):
    c = inputs.paged_case(name="t", seed=31, num_seqs=6, len_lo=50, len_hi=700, queries_per_seq=64, heads=32,
                          kv_heads=8, key_dim=128, value_dim=128, scale=0.5, shared_prefix_pages=2)
    dv = to_dev(c, bd)
    lse, delta = gpu_stats(bd, c, dv)
    first = gpu_bwd(bd, c, dv, lse, delta)
    for _ in range(5):
        again = gpu_bwd(bd, c, dv, lse, delta)
        for a, b in zip(first, again):
            assert torch.equal(a, b)
    bd.check_device_error()


def test_paged_full_size_gqa_sampled(bd):
    """The full GQA configuration (64 sequences, lengths U[128,4096]); the
    oracle re-expands a sample of sequences and the slots they own are
    compared.  The whole pool is bit-identical over five runs (one owner per
    physical token and KV head, a fixed traversal order, no atomics)."""
    c = inputs.paged_config("paged_gqa")
    dv = to_dev(c, bd)
    lse, delta = gpu_stats(bd, c, dv)
    dk, dvv = gpu_bwd(bd, c, dv, lse, delta)
    bd.check_device_error()
    for _ in range(4):
        dk2, dvv2 = gpu_bwd(bd, c, dv, lse, delta)
        assert torch.equal(dk, dk2) and torch.equal(dvv, dvv2)
    bd.check_device_error()
    from oracle import attn_bwd_paged
    pick = [0, 17, 63]
    qs = [np.arange(c.q_start[s], c.q_start[s + 1]) for s in pick]
    rows = np.concatenate(qs)
    sub_start = np.concatenate([[0], np.cumsum([len(x) for x in qs])]).astype(np.int32)
    ref_dk, ref_dv, ref_lse, ref_delta = attn_bwd_paged(
        c.q[rows], c.dy[rows], c.k_pool, c.page_table[pick], c.seq_len[pick], sub_start, c.q_pos[rows],
        page_size=c.page_size, kv_heads=c.kv_heads, v_pool=c.v_pool, causal=True, return_stats=True)
    owned = np.zeros(c.num_pages * c.page_size, bool)
    for s in pick:
        for t in range(int(c.seq_len[s])):
            owned[int(c.page_table[s, t // c.page_size]) * c.page_size + t % c.page_size] = True
    assert rel(dk, ref_dk, owned) < TOL
    assert rel(dvv, ref_dv, owned) < TOL
    assert np.max(np.abs(lse.cpu().numpy()[rows] - ref_lse)) < 2e-2


def test_paged_full_size_mla_sampled(bd):
    """The full MLA configuration (latent 512 + position 64, 32 heads, one
    latent head, the same 64 sequences); sampled sequences against the oracle,
    and bit stability across five runs."""
    c = inputs.paged_config("paged_mla")
    dv = to_dev(c, bd)
    lse, delta = gpu_stats(bd, c, dv)
    dk, dkp = gpu_bwd(bd, c, dv, lse, delta)
    for _ in range(4):
        dk2, dkp2 = gpu_bwd(bd, c, dv, lse, delta)
        assert torch.equal(dk, dk2) and torch.equal(dkp, dkp2)
    bd.check_device_error()
    from oracle import attn_bwd_paged
    pick = [3, 40]
    qs = [np.arange(c.q_start[s], c.q_start[s + 1]) for s in pick]
    rows = np.concatenate(qs)
    sub_start = np.concatenate([[0], np.cumsum([len(x) for x in qs])]).astype(np.int32)
    ref_dk, ref_dkp, ref_lse, _ = attn_bwd_paged(
        c.q[rows], c.dy[rows], c.k_pool, c.page_table[pick], c.seq_len[pick], sub_start, c.q_pos[rows],
        page_size=c.page_size, kv_heads=c.kv_heads, qp=c.qp[rows], kp_pool=c.kp_pool, causal=True,
        return_stats=True)
    owned = np.zeros(c.num_pages * c.page_size, bool)
    for s in pick:
        for t in range(int(c.seq_len[s])):
            owned[int(c.page_table[s, t // c.page_size]) * c.page_size + t % c.page_size] = True
    assert rel(dk, ref_dk, owned) < TOL
    assert rel(dkp, ref_dkp, owned) < TOL
    assert np.max(np.abs(lse.cpu().numpy()[rows] - ref_lse)) < 2e-2
