"""The C-ABI library builds, loads and exports every symbol the header
declares; host-side validation returns the documented status codes without
touching a GPU."""
import ctypes

import pytest

from attention_backward_recompute_gb300 import binding as bd
from attention_backward_recompute_gb300 import build as bld


@pytest.fixture(scope="module")
def lib():
    bld.build()
    return bd.lib()


def test_exports_every_declared_symbol(lib):
    names = bd.header_symbols()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/attn_bwd.h but not exported"


def test_version_and_status_strings(lib):
    assert bd.attn_version() >= 100
    assert bd.status_string(bd.ATTN_ERR_ALIAS) == "ATTN_ERR_ALIAS"


def _desc(**kw):
    base = dict(batch=2, heads=2, seq_q=64, seq_k=64, head_dim=128)
    base.update(kw)
    return bd.make_dense_desc(**base)


FAKE = 1 << 40          # 16-byte-aligned fake device addresses; never dereferenced
MB = 1 << 20


def _call(desc, q=FAKE, k=FAKE + 4 * MB, v=FAKE + 8 * MB, dy=FAKE + 12 * MB, km=None, bias=None, o=None,
          lse=None, dq=FAKE + 16 * MB, dk=FAKE + 20 * MB, dv=FAKE + 24 * MB, wrt=7, ws=FAKE + 28 * MB,
          ws_bytes=1 << 20):
    return bd.attn_bwd_dense(desc, q, k, v, dy, km, bias, o, lse, dq, dk, dv, wrt, ws, ws_bytes, None)


def test_workspace_query(lib):
    d = _desc()
    n = bd.attn_bwd_dense_workspace_bytes(d)
    assert n >= 3 * 2 * 2 * 64 * 4 and n % 256 == 0
    assert bd.attn_bwd_dense_workspace_bytes(_desc(head_dim=0)) == 0


@pytest.mark.parametrize("kw,status", [
    (dict(head_dim=96), bd.ATTN_ERR_UNSUPPORTED),
    (dict(head_dim=-1), bd.ATTN_ERR_INVALID_ARG),
    (dict(batch=-2), bd.ATTN_ERR_INVALID_ARG),
    (dict(dtype=7), bd.ATTN_ERR_INVALID_ARG),
    (dict(layout=3), bd.ATTN_ERR_INVALID_ARG),
    (dict(window=-5), bd.ATTN_ERR_INVALID_ARG),
])
def test_bad_descriptors(lib, kw, status):
    d = _desc(**{k: v for k, v in kw.items() if k != "window"})
    if "window" in kw:
        d.mask_flags |= bd.ATTN_MASK_WINDOW
        d.window = kw["window"]
    assert _call(d) == status
    assert bd.last_error() != ""


def test_null_descriptor(lib):
    st = lib.attn_bwd_dense(None, None, None, None, None, None, None, None, None, None, None, None, 7, None, 0, None)
    assert st == bd.ATTN_ERR_INVALID_ARG


def test_argument_errors(lib):
    d = _desc()
    assert _call(d, wrt=0) == bd.ATTN_ERR_INVALID_ARG
    assert _call(d, wrt=16) == bd.ATTN_ERR_INVALID_ARG
    assert _call(d, dq=None) == bd.ATTN_ERR_INVALID_ARG
    assert _call(d, q=FAKE + 8) == bd.ATTN_ERR_INVALID_ARG           # misaligned
    assert _call(d, km=FAKE + 40 * MB) == bd.ATTN_ERR_INVALID_ARG     # key mask without the flag
    dk = _desc(key_mask=True)
    assert _call(dk) == bd.ATTN_ERR_INVALID_ARG                      # flag without the key mask
    assert _call(d, o=FAKE + 40 * MB) == bd.ATTN_ERR_INVALID_ARG      # o without lse


def test_alias_detection(lib):
    d = _desc()
    # dv overlaps v (the arena hazard of the CPU reference)
    assert _call(d, dv=FAKE + 8 * MB + 4096) == bd.ATTN_ERR_ALIAS
    # dq overlaps dk
    assert _call(d, dq=FAKE + 20 * MB) == bd.ATTN_ERR_ALIAS
    # output overlaps the workspace
    assert _call(d, dk=FAKE + 28 * MB) == bd.ATTN_ERR_ALIAS


def test_workspace_errors(lib):
    d = _desc()
    assert _call(d, ws_bytes=16) == bd.ATTN_ERR_WORKSPACE
    assert _call(d, ws=FAKE + 28 * MB + 16) == bd.ATTN_ERR_WORKSPACE


def _strided_call(desc, sts, q, k, v, dy, dq, dk, dv, elem=None, ws=None, ws_bytes=0):
    return int(bd.lib().attn_bwd_dense_strided(ctypes.byref(desc), sts if sts is None else ctypes.byref(sts),
                                               ctypes.c_void_p(q), ctypes.c_void_p(k), ctypes.c_void_p(v),
                                               ctypes.c_void_p(dy), None, elem and ctypes.c_void_p(elem), None,
                                               None, None, ctypes.c_void_p(dq), ctypes.c_void_p(dk),
                                               ctypes.c_void_p(dv), 7, ws and ctypes.c_void_p(ws), ws_bytes, None))


def test_elem_mask_checks(lib):
    """The per-element mask: flag and pointer go together, fp32 storage and the
    forward export refuse it, and the workspace grows by its row and column
    bits (Sk and Sq rounded up to 64 bits per row/column)."""
    B, H, Sq, Sk, D = 2, 3, 100, 130, 64
    d = _desc(batch=B, heads=H, seq_q=Sq, seq_k=Sk, head_dim=D)
    base = bd.attn_bwd_dense_workspace_bytes(d)
    de = _desc(batch=B, heads=H, seq_q=Sq, seq_k=Sk, head_dim=D)
    de.mask_flags |= bd.ATTN_MASK_ELEM
    ew_q, ew_k = 6, 4  # ceil(130/32) = 5 -> 6 words, ceil(100/32) = 4
    a256 = lambda x: (x + 255) // 256 * 256
    assert bd.attn_bwd_dense_workspace_bytes(de) == base + a256(B * H * Sq * ew_q * 4) + a256(B * H * Sk * ew_k * 4)
    qb, kb = FAKE, FAKE + 8 * MB
    args = (qb, kb, kb + 2 * MB, qb + 2 * MB, FAKE + 16 * MB, FAKE + 18 * MB, FAKE + 20 * MB)
    # flag without the pointer, pointer without the flag
    assert _strided_call(de, None, *args) == bd.ATTN_ERR_INVALID_ARG
    assert _strided_call(d, None, *args, elem=FAKE + 32 * MB) == bd.ATTN_ERR_INVALID_ARG
    # with both the call reaches the workspace check
    assert _strided_call(de, None, *args, elem=FAKE + 32 * MB) == bd.ATTN_ERR_WORKSPACE
    # an output on the mask is refused
    assert _strided_call(de, None, *args[:4], FAKE + 32 * MB, args[5], args[6],
                         elem=FAKE + 32 * MB) == bd.ATTN_ERR_ALIAS
    df = _desc(batch=B, heads=H, seq_q=Sq, seq_k=Sk, head_dim=D, dtype=bd.ATTN_DTYPE_F32)
    df.mask_flags |= bd.ATTN_MASK_ELEM
    assert bd.attn_bwd_dense_workspace_bytes(df) == 0
    assert _strided_call(df, None, *args, elem=FAKE + 32 * MB) == bd.ATTN_ERR_UNSUPPORTED
    st = bd.attn_fwd_dense(de, ctypes.c_void_p(qb), ctypes.c_void_p(kb), ctypes.c_void_p(kb + 2 * MB), None, None,
                           ctypes.c_void_p(FAKE + 16 * MB), ctypes.c_void_p(FAKE + 18 * MB), None, 0, None)
    assert st == bd.ATTN_ERR_UNSUPPORTED
    # the layout call has no argument for it
    assert _call(de) == bd.ATTN_ERR_INVALID_ARG


def test_strided_fused_views(lib):
    """q, k, v and dq, dk, dv as interleaved views of fused [B, S, 3, H, D]
    tensors pass the overlap checks (the call stops at the missing workspace);
    the same views with one gradient aliasing another are refused."""
    B, S, H, D = 2, 64, 2, 128
    desc = _desc(batch=B, heads=H, seq_q=S, seq_k=S, head_dim=D)
    sts = bd.attn_dense_strides()
    bd.lib().attn_dense_strides_from_layout(ctypes.byref(desc), ctypes.byref(sts))
    fused = bd.attn_strides3(S * 3 * H * D, 3 * H * D, D)
    for n in ("q", "k", "v", "dq", "dk", "dv"):
        setattr(sts, n, fused)
    es = 2
    x, g = FAKE, FAKE + 64 * MB
    st = _strided_call(desc, sts, x, x + H * D * es, x + 2 * H * D * es, FAKE + 32 * MB,
                       g, g + H * D * es, g + 2 * H * D * es)
    assert st == bd.ATTN_ERR_WORKSPACE
    st = _strided_call(desc, sts, x, x + H * D * es, x + 2 * H * D * es, FAKE + 32 * MB,
                       g, g + H * D * es, g + H * D * es + 64)
    assert st == bd.ATTN_ERR_ALIAS
    # an output whose own rows overlap (sequence stride below the head span)
    sts.dq = bd.attn_strides3(S * H * D, D, D)
    st = _strided_call(desc, sts, x, x + H * D * es, x + 2 * H * D * es, FAKE + 32 * MB,
                       g, g + H * D * es, g + 2 * H * D * es)
    assert st == bd.ATTN_ERR_INVALID_ARG


def _compact_call(d, hist, n, dk=FAKE + 40 * MB, ws=None, ws_bytes=0):
    return int(bd.lib().attn_bwd_paged_compact(
        ctypes.byref(d), ctypes.c_void_p(FAKE), None, ctypes.c_void_p(FAKE + 8 * MB), ctypes.c_void_p(FAKE + 16 * MB),
        None, ctypes.c_void_p(FAKE + 24 * MB), ctypes.c_void_p(FAKE + 30 * MB), ctypes.c_void_p(FAKE + 31 * MB),
        ctypes.c_void_p(FAKE + 32 * MB), ctypes.c_void_p(FAKE + 33 * MB), hist and ctypes.c_void_p(hist), n,
        ctypes.c_void_p(dk), ctypes.c_void_p(FAKE + 48 * MB), None, bd.ATTN_WRT_DK | bd.ATTN_WRT_DV,
        ws and ctypes.c_void_p(ws), ws_bytes, None))


def test_paged_compact_checks(lib):
    """Compact history: a list pointer is needed when pages are listed, it is
    4-byte aligned and no output may overlap it; an empty list writes nothing
    (the call returns before any device work); the workspace covers the page
    map (one byte per pool page)."""
    d = bd.make_paged_desc(num_queries=64, num_seqs=4, heads=8, kv_heads=2, page_size=16, num_pages=100,
                           max_pages_per_seq=10, key_dim=128, value_dim=128)
    d0 = bd.make_paged_desc(num_queries=64, num_seqs=4, heads=8, kv_heads=2, page_size=16, num_pages=0,
                            max_pages_per_seq=10, key_dim=128, value_dim=128)
    assert bd.attn_bwd_paged_workspace_bytes(d) >= 100 + (4 + 101 + 100 + 40) * 4
    assert _compact_call(d, None, 5) == bd.ATTN_ERR_INVALID_ARG
    assert _compact_call(d, FAKE + 34 * MB + 2, 5) == bd.ATTN_ERR_INVALID_ARG
    assert _compact_call(d, FAKE + 40 * MB, 5) == bd.ATTN_ERR_ALIAS
    assert _compact_call(d, FAKE + 34 * MB, 0) == bd.ATTN_OK
    assert _compact_call(d, None, 0) == bd.ATTN_OK
    # a list with pages needs the workspace
    assert _compact_call(d, FAKE + 34 * MB, 5) == bd.ATTN_ERR_WORKSPACE
    assert _compact_call(d0, FAKE + 34 * MB, 5) == bd.ATTN_OK


def test_paged_mla_workspace_holds_split_partials(lib):
    """MLA: the workspace also holds the split kernel's fp32 chunk partials
    (128 slots of 128 tokens x (256 + 320) dims) next to the GQA layout."""
    kw = dict(num_queries=64, num_seqs=4, heads=8, kv_heads=1, page_size=16, num_pages=100, max_pages_per_seq=10,
              key_dim=512, value_dim=512)
    mla = bd.attn_bwd_paged_workspace_bytes(bd.make_paged_desc(position_dim=64, **kw))
    gqa_layout = bd.attn_bwd_paged_workspace_bytes(bd.make_paged_desc(**dict(kw, key_dim=128, value_dim=128)))
    assert mla == gqa_layout + 128 * 128 * (256 + 320) * 4


def test_paged_query_side_needs_workspace(lib):
    """The row-statistics and query-side calls keep their dispatch order (the
    sequences by length) in the paged workspace: a missing, short or
    misaligned one is refused before any device work."""
    d = bd.make_paged_desc(num_queries=64, num_seqs=4, heads=8, kv_heads=2, page_size=16, num_pages=100,
                           max_pages_per_seq=10, key_dim=128, value_dim=128)
    n = bd.attn_bwd_paged_workspace_bytes(d)
    assert n >= 100 + (4 + 101 + 100 + 40 + 4) * 4
    L = bd.lib()
    args = [ctypes.c_void_p(FAKE), None, ctypes.c_void_p(FAKE + 8 * MB), ctypes.c_void_p(FAKE + 16 * MB), None,
            ctypes.c_void_p(FAKE + 24 * MB), ctypes.c_void_p(FAKE + 30 * MB), ctypes.c_void_p(FAKE + 31 * MB),
            ctypes.c_void_p(FAKE + 32 * MB), ctypes.c_void_p(FAKE + 33 * MB)]
    for ws, nb in ((None, 0), (FAKE + 40 * MB, n - 1), (FAKE + 40 * MB + 16, n)):
        w = ws and ctypes.c_void_p(ws)
        assert int(L.attn_paged_row_stats(ctypes.byref(d), *args, w, nb, None)) == bd.ATTN_ERR_WORKSPACE
        assert int(L.attn_bwd_paged_query(ctypes.byref(d), *args, ctypes.c_void_p(FAKE + 34 * MB), None, w, nb,
                                          None)) == bd.ATTN_ERR_WORKSPACE


def test_store_ds_option_checks(lib):
    """ATTN_OPT_STORE_DS grows the workspace by one 128 x 64 bf16 dS tile per
    (batch, head, key tile of 128, query tile of 64); fp32 storage and unknown
    option bits are refused; the no-allocation entry point refuses it."""
    d = _desc(batch=2, heads=3, seq_q=200, seq_k=300, head_dim=128)
    base = bd.attn_bwd_dense_workspace_bytes(d)
    d.options = bd.ATTN_OPT_STORE_DS
    a256 = lambda x: (x + 255) // 256 * 256
    assert bd.attn_bwd_dense_workspace_bytes(d) == base + a256(2 * 3 * 3 * 4 * 16384)
    d.options = 2
    assert bd.attn_bwd_dense_workspace_bytes(d) == 0
    assert _call(d) == bd.ATTN_ERR_INVALID_ARG
    df = _desc(dtype=bd.ATTN_DTYPE_F32, head_dim=64)
    df.options = bd.ATTN_OPT_STORE_DS
    assert _call(df) == bd.ATTN_ERR_UNSUPPORTED
    d.options = bd.ATTN_OPT_STORE_DS
    st = int(bd.lib().attn_bwd_dense_noalloc(ctypes.byref(d), ctypes.c_void_p(FAKE), ctypes.c_void_p(FAKE + 4 * MB),
                                             ctypes.c_void_p(FAKE + 8 * MB), ctypes.c_void_p(FAKE + 12 * MB), None,
                                             None, None, None, ctypes.c_void_p(FAKE + 16 * MB),
                                             ctypes.c_void_p(FAKE + 20 * MB), ctypes.c_void_p(FAKE + 24 * MB), 7,
                                             None))
    assert st == bd.ATTN_ERR_UNSUPPORTED


def test_noalloc_refuses_elem_mask(lib):
    """The no-allocation entry point refuses the per-element mask by name (its
    packed bits would need workspace) before touching any pointer."""
    d = _desc(batch=1, heads=2, seq_q=64, seq_k=64, head_dim=64)
    d.mask_flags |= bd.ATTN_MASK_ELEM
    st = int(bd.lib().attn_bwd_dense_noalloc(ctypes.byref(d), ctypes.c_void_p(FAKE), ctypes.c_void_p(FAKE + 4 * MB),
                                             ctypes.c_void_p(FAKE + 8 * MB), ctypes.c_void_p(FAKE + 12 * MB), None,
                                             None, None, None, ctypes.c_void_p(FAKE + 16 * MB),
                                             ctypes.c_void_p(FAKE + 20 * MB), ctypes.c_void_p(FAKE + 24 * MB), 7,
                                             None))
    assert st == bd.ATTN_ERR_UNSUPPORTED
    assert "per-element" in bd.last_error()


def test_paged_mla_shape_checks(lib):
    """MLA (latent 512 + position 64) takes any number of heads per KV head
    that divides 64 (a 64-column tile holds whole query rows) and refuses the
    others, and other latent / position sizes, before any device work; the
    workspace query returns 0 for a refused descriptor."""
    ok = bd.make_paged_desc(num_queries=64, num_seqs=4, heads=16, kv_heads=1, page_size=16, num_pages=100,
                            max_pages_per_seq=10, key_dim=512, value_dim=512, position_dim=64)
    assert bd.attn_bwd_paged_workspace_bytes(ok) > 0
    for heads, kv, kd, pd in ((12, 4, 512, 64), (40, 1, 512, 64), (16, 1, 256, 64), (16, 1, 512, 32)):
        d = bd.make_paged_desc(num_queries=64, num_seqs=4, heads=heads, kv_heads=kv, page_size=16, num_pages=100,
                               max_pages_per_seq=10, key_dim=kd, value_dim=kd, position_dim=pd)
        assert bd.attn_bwd_paged_workspace_bytes(d) == 0, (heads, kv, kd, pd)
