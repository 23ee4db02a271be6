"""CPU oracle for attention backward with recomputed scores and softmax.

TEST INFRASTRUCTURE ONLY.  This package is a plain, slow, float64 restatement
of what the pages define; it exists so that the CUDA library can be checked
against something obviously correct.  Only ``tests/``, ``__graft_entry__.smoke``
and the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import
it.  The product path (the C-ABI library and its Python binding) never calls
it, shares no code with it, and fails loudly when the CUDA extension is absent.

Sources restated (page title, section):

* rlx-cpu ``src/attention_bwd.rs``: ``apply_synthetic_mask`` (causal and
  sliding-window masks, bottom-right aligned), ``backward_dense_head_all``
  (scores, custom/bias masks, softmax, the five products dV, dP, dS, dQ, dK)
  and ``attention_backward_all`` (per batch x head driver, [B,S,H,D] and
  [B,H,S,D] layouts).
* rlx-wgpu ``src/kernels/attention_bwd.wgsl``: ``mask_score`` (custom mask
  threshold 0.5 and -1e9) and ``softmax_row``.
* ruDNN ``src/paged_attention/ordered_kernel.rs``: ``history_backward``
  (paged GQA/MLA history backward producing dK, dV, dKp; row statistics;
  MLA latent that is both key and value).

Every function here has pins in ``tests/test_oracle_*.py`` that do not reuse its
formulas: central finite differences of the loss, invariants, closed forms and
brute force on tiny inputs.
"""
from .dense import attn_bwd_dense, attn_fwd_dense, head_backward, visibility  # noqa: F401
from .paged import attn_bwd_paged, paged_query_backward, paged_row_stats  # noqa: F401
