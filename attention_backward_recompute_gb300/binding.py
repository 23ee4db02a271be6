"""ctypes binding of libattnbwd (include/attn_bwd.h).

The functions named like the C entry points take raw integers (device pointers,
sizes, a cudaStream_t handle) and return the status code unchanged.  The
torch-tensor helpers (:func:`dense_backward`, :func:`paged_backward`,
:func:`paged_row_stats`) only marshal arguments: they check shapes, allocate the
outputs and the workspace with torch, pass ``data_ptr()`` values and the current
stream, and raise on a non-OK status.  Every step of the computation runs in the
library's CUDA kernels; there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import re

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libattnbwd.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "attn_bwd.h")

ATTN_OK = 0
ATTN_ERR_INVALID_ARG = 1
ATTN_ERR_UNSUPPORTED = 2
ATTN_ERR_ALIAS = 3
ATTN_ERR_WORKSPACE = 4
ATTN_ERR_CUDA = 5
ATTN_ERR_TIMEOUT = 6

ATTN_DTYPE_F32 = 0
ATTN_DTYPE_BF16 = 1
ATTN_LAYOUT_BSHD = 0
ATTN_LAYOUT_BHSD = 1
ATTN_MASK_CAUSAL = 1
ATTN_MASK_WINDOW = 2
ATTN_MASK_KEY = 4
ATTN_MASK_BIAS = 8
ATTN_MASK_TOP_LEFT = 16
ATTN_MASK_ELEM = 32
ATTN_OPT_STORE_DS = 1
ATTN_WRT_DQ = 1
ATTN_WRT_DK = 2
ATTN_WRT_DV = 4
ATTN_WRT_DKP = 8


class AttnError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{status_string(status)}: {message}")
        self.status = status


class attn_dense_desc(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int64), ("heads", ctypes.c_int64), ("seq_q", ctypes.c_int64),
                ("seq_k", ctypes.c_int64), ("head_dim", ctypes.c_int64), ("dtype", ctypes.c_int32),
                ("layout", ctypes.c_int32), ("mask_flags", ctypes.c_uint32), ("window", ctypes.c_int32),
                ("mask_thr", ctypes.c_float), ("mask_neg", ctypes.c_float), ("scale", ctypes.c_float),
                ("options", ctypes.c_uint32)]


class attn_strides3(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int64), ("seq", ctypes.c_int64), ("head", ctypes.c_int64)]


class attn_dense_strides(ctypes.Structure):
    _fields_ = [(n, attn_strides3) for n in ("q", "k", "v", "dy", "o", "dq", "dk", "dv")]


class attn_paged_desc(ctypes.Structure):
    _fields_ = [("num_queries", ctypes.c_int64), ("num_seqs", ctypes.c_int64), ("heads", ctypes.c_int64),
                ("kv_heads", ctypes.c_int64), ("page_size", ctypes.c_int64), ("num_pages", ctypes.c_int64),
                ("max_pages_per_seq", ctypes.c_int64), ("key_dim", ctypes.c_int64),
                ("value_dim", ctypes.c_int64), ("position_dim", ctypes.c_int64), ("dtype", ctypes.c_int32),
                ("causal", ctypes.c_int32), ("scale", ctypes.c_float), ("reserved", ctypes.c_int32)]


_lib = None
_P = ctypes.c_void_p
_SIG = {
    "attn_dense_desc_init": (None, [ctypes.POINTER(attn_dense_desc)]),
    "attn_bwd_dense_workspace_bytes": (ctypes.c_size_t, [ctypes.POINTER(attn_dense_desc)]),
    "attn_bwd_dense": (ctypes.c_int32, [ctypes.POINTER(attn_dense_desc), _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                        _P, ctypes.c_uint, _P, ctypes.c_size_t, _P]),
    "attn_bwd_dense_noalloc": (ctypes.c_int32, [ctypes.POINTER(attn_dense_desc), _P, _P, _P, _P, _P, _P, _P, _P,
                                                _P, _P, _P, ctypes.c_uint, _P]),
    "attn_dense_strides_from_layout": (None, [ctypes.POINTER(attn_dense_desc), ctypes.POINTER(attn_dense_strides)]),
    "attn_bwd_dense_strided": (ctypes.c_int32, [ctypes.POINTER(attn_dense_desc), ctypes.POINTER(attn_dense_strides),
                                                _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_uint, _P,
                                                ctypes.c_size_t, _P]),
    "attn_fwd_dense_strided": (ctypes.c_int32, [ctypes.POINTER(attn_dense_desc), ctypes.POINTER(attn_dense_strides),
                                                _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "attn_fwd_dense": (ctypes.c_int32, [ctypes.POINTER(attn_dense_desc), _P, _P, _P, _P, _P, _P, _P, _P,
                                        ctypes.c_size_t, _P]),
    "attn_bwd_paged_workspace_bytes": (ctypes.c_size_t, [ctypes.POINTER(attn_paged_desc)]),
    "attn_bwd_paged": (ctypes.c_int32, [ctypes.POINTER(attn_paged_desc), _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                        _P, _P, _P, ctypes.c_uint, _P, ctypes.c_size_t, _P]),
    "attn_bwd_paged_compact": (ctypes.c_int32, [ctypes.POINTER(attn_paged_desc), _P, _P, _P, _P, _P, _P, _P, _P,
                                                _P, _P, _P, ctypes.c_int64, _P, _P, _P, ctypes.c_uint, _P,
                                                ctypes.c_size_t, _P]),
    "attn_paged_row_stats": (ctypes.c_int32, [ctypes.POINTER(attn_paged_desc), _P, _P, _P, _P, _P, _P, _P, _P,
                                              _P, _P, _P, ctypes.c_size_t, _P]),
    "attn_bwd_paged_query": (ctypes.c_int32, [ctypes.POINTER(attn_paged_desc), _P, _P, _P, _P, _P, _P, _P, _P,
                                              _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "attn_last_error": (ctypes.c_char_p, []),
    "attn_status_string": (ctypes.c_char_p, [ctypes.c_int32]),
    "attn_check_device_error": (ctypes.c_int32, [_P]),
    "attn_selftest_wait_timeout": (ctypes.c_int32, [_P]),
    "attn_version": (ctypes.c_int, []),
    "attn_set_timing_events": (None, [ctypes.POINTER(ctypes.c_void_p), ctypes.c_int]),
}


def lib() -> ctypes.CDLL:
    """Load libattnbwd.so from the package directory (raises if it is absent)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it first "
                               "(python -c 'import __graft_entry__ as g; g.build()')")
        l = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIG.items():
            if hasattr(l, name):
                f = getattr(l, name)
                f.restype = res
                f.argtypes = args
        _lib = l
    return _lib


def header_symbols() -> list[str]:
    """Names of the functions include/attn_bwd.h declares with ATTN_API."""
    with open(HEADER) as fh:
        text = fh.read()
    return re.findall(r"ATTN_API\s+[\w\s\*]+?\b(attn_\w+)\s*\(", text)


def status_string(st: int) -> str:
    return lib().attn_status_string(st).decode()


def last_error() -> str:
    return lib().attn_last_error().decode()


# ---- raw entry points (same names as the C ABI) ----------------------------

def attn_dense_desc_init(desc: attn_dense_desc) -> None:
    lib().attn_dense_desc_init(ctypes.byref(desc))


def attn_bwd_dense_workspace_bytes(desc: attn_dense_desc) -> int:
    return int(lib().attn_bwd_dense_workspace_bytes(ctypes.byref(desc)))


def attn_bwd_dense(desc, q, k, v, dy, key_mask, bias, o, lse, dq, dk, dv, wrt_mask, workspace,
                   workspace_bytes, stream) -> int:
    return int(lib().attn_bwd_dense(ctypes.byref(desc), q, k, v, dy, key_mask, bias, o, lse, dq, dk, dv,
                                    wrt_mask, workspace, workspace_bytes, stream))


def attn_bwd_dense_noalloc(desc, q, k, v, dy, key_mask, bias, o, lse, dq, dk, dv, wrt_mask, stream) -> int:
    """Dense backward with the library-owned scratch (no workspace argument)."""
    return int(lib().attn_bwd_dense_noalloc(ctypes.byref(desc), q, k, v, dy, key_mask, bias, o, lse, dq, dk, dv,
                                            wrt_mask, stream))


def attn_bwd_paged_workspace_bytes(desc: attn_paged_desc) -> int:
    return int(lib().attn_bwd_paged_workspace_bytes(ctypes.byref(desc)))


def attn_bwd_paged(desc, q, qp, k_pool, v_pool, kp_pool, dy, page_table, seq_meta, lse, delta, dk_pool, dv_pool,
                   dkp_pool, wrt_mask, workspace, workspace_bytes, stream) -> int:
    return int(lib().attn_bwd_paged(ctypes.byref(desc), q, qp, k_pool, v_pool, kp_pool, dy, page_table, seq_meta,
                                    lse, delta, dk_pool, dv_pool, dkp_pool, wrt_mask, workspace, workspace_bytes,
                                    stream))


def attn_paged_row_stats(desc, q, qp, k_pool, v_pool, kp_pool, dy, page_table, seq_meta, lse, delta, workspace,
                         workspace_bytes, stream) -> int:
    return int(lib().attn_paged_row_stats(ctypes.byref(desc), q, qp, k_pool, v_pool, kp_pool, dy, page_table,
                                          seq_meta, lse, delta, workspace, workspace_bytes, stream))


def attn_bwd_paged_query(desc, q, qp, k_pool, v_pool, kp_pool, dy, page_table, seq_meta, lse, delta, dq, dqp,
                         workspace, workspace_bytes, stream) -> int:
    return int(lib().attn_bwd_paged_query(ctypes.byref(desc), q, qp, k_pool, v_pool, kp_pool, dy, page_table,
                                          seq_meta, lse, delta, dq, dqp, workspace, workspace_bytes, stream))


def attn_check_device_error(stream) -> int:
    return int(lib().attn_check_device_error(stream))


def attn_selftest_wait_timeout(stream) -> int:
    return int(lib().attn_selftest_wait_timeout(stream))


def attn_set_timing_events(events) -> None:
    """Record cudaEvent handles (ints) around the kernels of the next call."""
    if events is None:
        lib().attn_set_timing_events(None, 0)
        return
    arr = (ctypes.c_void_p * len(events))(*events)
    attn_set_timing_events._keep = arr  # the library reads the array during the next call
    lib().attn_set_timing_events(arr, len(events))


def attn_version() -> int:
    return int(lib().attn_version())


# ---- torch helpers (argument marshalling only) ------------------------------

def _ptr(t):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors passed to libattnbwd must be contiguous (the ABI takes dense layouts)")
    return ctypes.c_void_p(t.data_ptr())


def _vptr(t):
    """Pointer of a tensor whose strides are passed alongside (views allowed)."""
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check(st: int):
    if st != ATTN_OK:
        raise AttnError(st, last_error())


def _dtype_code(t):
    import torch
    if t.dtype == torch.bfloat16:
        return ATTN_DTYPE_BF16
    if t.dtype == torch.float32:
        return ATTN_DTYPE_F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def make_dense_desc(*, batch, heads, seq_q, seq_k, head_dim, dtype=ATTN_DTYPE_BF16, layout=ATTN_LAYOUT_BSHD,
                    causal=False, window=None, key_mask=False, bias=False, mask_thr=0.5, mask_neg=-1e9,
                    scale=0.0, top_left=False, elem_mask=False, store_ds=False) -> attn_dense_desc:
    d = attn_dense_desc()
    attn_dense_desc_init(d)
    d.batch, d.heads, d.seq_q, d.seq_k, d.head_dim = batch, heads, seq_q, seq_k, head_dim
    d.dtype, d.layout = dtype, layout
    flags = 0
    if causal:
        flags |= ATTN_MASK_CAUSAL
    if window is not None:
        flags |= ATTN_MASK_WINDOW
        d.window = int(window)
    if key_mask:
        flags |= ATTN_MASK_KEY
    if bias:
        flags |= ATTN_MASK_BIAS
    if top_left:
        flags |= ATTN_MASK_TOP_LEFT
    if elem_mask:
        flags |= ATTN_MASK_ELEM
    d.mask_flags = flags
    d.mask_thr, d.mask_neg, d.scale = mask_thr, mask_neg, scale
    d.options = ATTN_OPT_STORE_DS if store_ds else 0
    return d


def dense_backward(q, k, v, dy, *, layout="bshd", causal=False, window=None, key_mask=None, bias=None, o=None,
                   lse=None, wrt=ATTN_WRT_DQ | ATTN_WRT_DK | ATTN_WRT_DV, scale=0.0, mask_thr=0.5, mask_neg=-1e9,
                   outputs=None, workspace=None, stream=None, top_left=False, elem_mask=None, store_ds=False):
    """dQ, dK, dV for CUDA tensors q, k, v, dy ([B,S,H,D] or [B,H,S,D]).

    ``elem_mask`` is the optional per-element mask [B, H, Sq, Sk] (fp32,
    contiguous; a pair below ``mask_thr`` is masked).  ``store_ds`` selects
    ATTN_OPT_STORE_DS (dQ from the stored dS tiles; larger workspace).
    Returns (dq, dk, dv) with None for gradients not selected in ``wrt``."""
    import torch
    lay = {"bshd": ATTN_LAYOUT_BSHD, "bhsd": ATTN_LAYOUT_BHSD}[layout]
    if lay == ATTN_LAYOUT_BSHD:
        B, Sq, H, D = q.shape
        Sk = k.shape[1]
    else:
        B, H, Sq, D = q.shape
        Sk = k.shape[2]
    desc = make_dense_desc(batch=B, heads=H, seq_q=Sq, seq_k=Sk, head_dim=D, dtype=_dtype_code(q), layout=lay,
                           causal=causal, window=window, key_mask=key_mask is not None, bias=bias is not None,
                           mask_thr=mask_thr, mask_neg=mask_neg, scale=scale, top_left=top_left,
                           elem_mask=elem_mask is not None, store_ds=store_ds)
    if elem_mask is not None and not elem_mask.is_contiguous():
        raise ValueError("elem_mask must be contiguous")
    if outputs is None:
        dq = torch.empty_like(q) if wrt & ATTN_WRT_DQ else None
        dk = torch.empty_like(k) if wrt & ATTN_WRT_DK else None
        dv = torch.empty_like(v) if wrt & ATTN_WRT_DV else None
    else:
        dq, dk, dv = outputs
    nbytes = attn_bwd_dense_workspace_bytes(desc)
    if workspace is None:
        workspace = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=q.device)
    tensors = dict(q=q, k=k, v=v, dy=dy, o=o, dq=dq, dk=dk, dv=dv)
    if elem_mask is None and all(t is None or t.is_contiguous() for t in tensors.values()):
        st = attn_bwd_dense(desc, _ptr(q), _ptr(k), _ptr(v), _ptr(dy), _ptr(key_mask), _ptr(bias), _ptr(o),
                            _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv), wrt, _ptr(workspace), workspace.numel(),
                            _stream_handle(stream))
    else:  # non-contiguous views or a per-element mask: the strided entry point
        sts = _dense_strides(desc, layout, tensors)
        st = int(lib().attn_bwd_dense_strided(ctypes.byref(desc), ctypes.byref(sts), _vptr(q), _vptr(k), _vptr(v),
                                              _vptr(dy), _ptr(key_mask), _ptr(elem_mask), _ptr(bias), _vptr(o),
                                              _ptr(lse), _vptr(dq),
                                              _vptr(dk), _vptr(dv), wrt, _ptr(workspace), workspace.numel(),
                                              _stream_handle(stream)))
    _check(st)
    return dq, dk, dv


def _dense_strides(desc, layout, tensors):
    """attn_dense_strides from torch tensors' strides (the layout's own for a
    tensor that is None)."""
    sts = attn_dense_strides()
    lib().attn_dense_strides_from_layout(ctypes.byref(desc), ctypes.byref(sts))
    for name, t in tensors.items():
        if t is None:
            continue
        if t.stride(3) != 1:
            raise ValueError(f"{name}: the head_dim dimension must be contiguous")
        st3 = getattr(sts, name)
        if layout == "bshd":
            st3.batch, st3.seq, st3.head = t.stride(0), t.stride(1), t.stride(2)
        else:
            st3.batch, st3.head, st3.seq = t.stride(0), t.stride(1), t.stride(2)
    return sts


def attn_fwd_dense(desc, q, k, v, key_mask, bias, o, lse, workspace, workspace_bytes, stream) -> int:
    return int(lib().attn_fwd_dense(ctypes.byref(desc), q, k, v, key_mask, bias, o, lse, workspace, workspace_bytes,
                                    stream))


def dense_forward(q, k, v, *, layout="bshd", causal=False, window=None, key_mask=None, bias=None, scale=0.0,
                  mask_thr=0.5, mask_neg=-1e9, top_left=False, outputs=None, workspace=None, stream=None):
    """(o, lse) for CUDA tensors q, k, v ([B,S,H,D] or [B,H,S,D]): o like q,
    lse fp32 [B, H, Sq] (natural log)."""
    import torch
    lay = {"bshd": ATTN_LAYOUT_BSHD, "bhsd": ATTN_LAYOUT_BHSD}[layout]
    if lay == ATTN_LAYOUT_BSHD:
        B, Sq, H, D = q.shape
        Sk = k.shape[1]
    else:
        B, H, Sq, D = q.shape
        Sk = k.shape[2]
    desc = make_dense_desc(batch=B, heads=H, seq_q=Sq, seq_k=Sk, head_dim=D, dtype=_dtype_code(q), layout=lay,
                           causal=causal, window=window, key_mask=key_mask is not None, bias=bias is not None,
                           mask_thr=mask_thr, mask_neg=mask_neg, scale=scale, top_left=top_left)
    if outputs is None:
        o = torch.empty_like(q)
        lse = torch.empty((B, H, Sq), dtype=torch.float32, device=q.device)
    else:
        o, lse = outputs
    nbytes = attn_bwd_dense_workspace_bytes(desc)
    if workspace is None:
        workspace = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=q.device)
    tensors = dict(q=q, k=k, v=v, o=o)
    if all(t.is_contiguous() for t in tensors.values()):
        st = attn_fwd_dense(desc, _ptr(q), _ptr(k), _ptr(v), _ptr(key_mask), _ptr(bias), _ptr(o), _ptr(lse),
                            _ptr(workspace), workspace.numel(), _stream_handle(stream))
    else:
        sts = _dense_strides(desc, layout, tensors)
        st = int(lib().attn_fwd_dense_strided(ctypes.byref(desc), ctypes.byref(sts), _vptr(q), _vptr(k), _vptr(v),
                                              _ptr(key_mask), _ptr(bias), _vptr(o), _ptr(lse), _ptr(workspace),
                                              workspace.numel(), _stream_handle(stream)))
    _check(st)
    return o, lse


def check_device_error(stream=None) -> None:
    _check(attn_check_device_error(_stream_handle(stream)))


def make_paged_desc(*, num_queries, num_seqs, heads, kv_heads, page_size, num_pages, max_pages_per_seq, key_dim,
                    value_dim, position_dim=0, causal=True, scale=0.0, dtype=ATTN_DTYPE_BF16) -> attn_paged_desc:
    d = attn_paged_desc()
    d.num_queries, d.num_seqs, d.heads, d.kv_heads = num_queries, num_seqs, heads, kv_heads
    d.page_size, d.num_pages, d.max_pages_per_seq = page_size, num_pages, max_pages_per_seq
    d.key_dim, d.value_dim, d.position_dim = key_dim, value_dim, position_dim
    d.dtype, d.causal, d.scale, d.reserved = dtype, int(bool(causal)), scale, 0
    return d


def seq_meta_tensor(seq_len, q_start, q_pos, device):
    """Pack seq_len | q_start | q_pos into the single int32 array the ABI takes."""
    import torch
    parts = [torch.as_tensor(x, dtype=torch.int32).reshape(-1) for x in (seq_len, q_start, q_pos)]
    return torch.cat(parts).to(device).contiguous()


def _paged_desc_for(q, dy, k_pool, page_table, seq_meta, heads, kv_heads, page_size, causal, scale, qp, kp_pool):
    num_seqs = page_table.shape[0]
    return make_paged_desc(num_queries=q.shape[0], num_seqs=num_seqs, heads=heads, kv_heads=kv_heads,
                           page_size=page_size, num_pages=k_pool.shape[0] // page_size,
                           max_pages_per_seq=page_table.shape[1], key_dim=q.shape[2], value_dim=dy.shape[2],
                           position_dim=0 if qp is None else qp.shape[2], causal=causal, scale=scale)


def paged_row_stats(q, k_pool, v_pool, dy, page_table, seq_meta, *, heads, kv_heads, page_size=16, causal=True,
                    scale=0.0, qp=None, kp_pool=None, workspace=None, stream=None):
    """lse, delta [Nq, H] (fp32) for CUDA tensors: q [Nq,H,Dk], pools [slots,KVH,D]."""
    import torch
    d = _paged_desc_for(q, dy, k_pool, page_table, seq_meta, heads, kv_heads, page_size, causal, scale, qp, kp_pool)
    lse = torch.empty((q.shape[0], heads), dtype=torch.float32, device=q.device)
    delta = torch.empty_like(lse)
    n = attn_bwd_paged_workspace_bytes(d)
    if workspace is None:
        workspace = torch.empty(max(n, 256), dtype=torch.uint8, device=q.device)
    st = attn_paged_row_stats(d, _ptr(q), _ptr(qp), _ptr(k_pool), _ptr(v_pool), _ptr(kp_pool), _ptr(dy),
                              _ptr(page_table), _ptr(seq_meta), _ptr(lse), _ptr(delta), _ptr(workspace),
                              workspace.numel(), _stream_handle(stream))
    _check(st)
    return lse, delta


def paged_query_backward(q, k_pool, v_pool, dy, page_table, seq_meta, *, heads, kv_heads, page_size=16,
                         causal=True, scale=0.0, qp=None, kp_pool=None, outputs=None, workspace=None, stream=None):
    """Query side: (lse, delta, dq) for GQA or (lse, delta, dq, dqp) for MLA
    (qp, kp_pool given), for CUDA tensors; lse/delta [Nq, H] fp32, dq shaped
    like q, dqp like qp."""
    import torch
    d = _paged_desc_for(q, dy, k_pool, page_table, seq_meta, heads, kv_heads, page_size, causal, scale, qp, kp_pool)
    mla = qp is not None
    if outputs is None:
        lse = torch.empty((q.shape[0], heads), dtype=torch.float32, device=q.device)
        delta = torch.empty_like(lse)
        dq = torch.empty_like(q)
        dqp = torch.empty_like(qp) if mla else None
    else:
        lse, delta, dq = outputs[:3]
        dqp = outputs[3] if mla else None
    n = attn_bwd_paged_workspace_bytes(d)
    if workspace is None:
        workspace = torch.empty(max(n, 256), dtype=torch.uint8, device=q.device)
    st = attn_bwd_paged_query(d, _ptr(q), _ptr(qp), _ptr(k_pool), _ptr(v_pool), _ptr(kp_pool), _ptr(dy),
                              _ptr(page_table), _ptr(seq_meta), _ptr(lse), _ptr(delta), _ptr(dq), _ptr(dqp),
                              _ptr(workspace), workspace.numel(), _stream_handle(stream))
    _check(st)
    return (lse, delta, dq, dqp) if mla else (lse, delta, dq)


def paged_backward(q, k_pool, v_pool, dy, page_table, seq_meta, lse, delta, *, heads, kv_heads, page_size=16,
                   causal=True, scale=0.0, qp=None, kp_pool=None, wrt=None, outputs=None, workspace=None,
                   stream=None, history_pages=None):
    """Pool gradients (dk_pool, dv_pool) for GQA or (dk_pool, dkp_pool) for MLA.

    ``history_pages`` (int32 CUDA tensor of physical page indices) selects the
    compact history call: only the listed pages' rows are computed and
    written, the others are left as they are in ``outputs``."""
    import torch
    d = _paged_desc_for(q, dy, k_pool, page_table, seq_meta, heads, kv_heads, page_size, causal, scale, qp, kp_pool)
    mla = qp is not None
    if wrt is None:
        wrt = (ATTN_WRT_DK | ATTN_WRT_DKP) if mla else (ATTN_WRT_DK | ATTN_WRT_DV)
    if outputs is None:
        dk = torch.empty_like(k_pool) if wrt & ATTN_WRT_DK else None
        dv = torch.empty_like(v_pool) if (not mla and wrt & ATTN_WRT_DV) else None
        dkp = torch.empty_like(kp_pool) if (mla and wrt & ATTN_WRT_DKP) else None
    else:
        dk, dv, dkp = outputs
    n = attn_bwd_paged_workspace_bytes(d)
    if workspace is None:
        workspace = torch.empty(max(n, 256), dtype=torch.uint8, device=q.device)
    if history_pages is None:
        st = attn_bwd_paged(d, _ptr(q), _ptr(qp), _ptr(k_pool), _ptr(v_pool), _ptr(kp_pool), _ptr(dy),
                            _ptr(page_table), _ptr(seq_meta), _ptr(lse), _ptr(delta), _ptr(dk), _ptr(dv), _ptr(dkp),
                            wrt, _ptr(workspace), workspace.numel(), _stream_handle(stream))
    else:
        if history_pages.dtype != torch.int32 or not history_pages.is_contiguous():
            raise ValueError("history_pages must be a contiguous int32 tensor")
        st = int(lib().attn_bwd_paged_compact(ctypes.byref(d), _ptr(q), _ptr(qp), _ptr(k_pool), _ptr(v_pool),
                                              _ptr(kp_pool), _ptr(dy), _ptr(page_table), _ptr(seq_meta), _ptr(lse),
                                              _ptr(delta), _ptr(history_pages), history_pages.numel(), _ptr(dk),
                                              _ptr(dv), _ptr(dkp), wrt, _ptr(workspace), workspace.numel(),
                                              _stream_handle(stream)))
    _check(st)
    return (dk, dkp) if mla else (dk, dv)
