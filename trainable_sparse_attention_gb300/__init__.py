"""trainable_sparse_attention_gb300 -- GB300 (sm_103a) hot path of trainable
sparse attention: indexer score -> deterministic exact top-k -> sparse
attention forward/backward (absorbed MLA and block Sparse-GQA), and the
indexer's training step on the selected slots (sparse KL, indexer backward).

The compute lives in ``libtsa.so`` (hand-written CUDA, C ABI in
``include/tsa.h``); this package only marshals arguments to it.
"""
from ._binding import (FLAG_INDEX_RANGE, FLAG_TIMEOUT, LIB_PATH, SIGNATURES, TsaError, kernel_launches,
                       load_library, max_seqlen, qsa_indexer_bwd, qsa_indexer_bwd_workspace_size, qsa_indexer_kl, qsa_indexer_scores, qsa_topk,
                       qsa_topk_from_scores, qsa_topk_workspace_size, read_flags, selftest_bounded_wait,
                       sparse_gqa_bwd, sparse_gqa_bwd_workspace_size, sparse_gqa_fwd, sparse_gqa_fwd_workspace_size,
                       sparse_mla_bwd,
                       sparse_mla_bwd_workspace_size, sparse_mla_fwd)

__all__ = ["qsa_indexer_scores", "qsa_topk", "qsa_topk_from_scores", "qsa_topk_workspace_size",
           "sparse_mla_fwd", "sparse_mla_bwd", "sparse_mla_bwd_workspace_size", "sparse_gqa_fwd",
           "sparse_gqa_fwd_workspace_size", "sparse_gqa_bwd", "sparse_gqa_bwd_workspace_size", "qsa_indexer_kl", "qsa_indexer_bwd", "qsa_indexer_bwd_workspace_size",
           "read_flags", "selftest_bounded_wait", "kernel_launches", "load_library", "TsaError",
           "FLAG_INDEX_RANGE", "FLAG_TIMEOUT", "max_seqlen", "build"]


def build(force: bool = False) -> str:
    from .builder import build as _build
    return _build(force=force)
