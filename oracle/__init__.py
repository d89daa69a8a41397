"""CPU oracle for the trainable sparse-attention hot path.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, by the package's ``smoke()``
check and by the bench's CPU-baseline / reference arm, never by the product
path.  See ``reference.py`` for the definitions and their sources.
"""
from .reference import *  # noqa: F401,F403
from .reference import (indexer_token_scores, indexer_block_scores, topk_lex, topk_rows, qsa_topk,
                        sparse_mla_row, sparse_gqa_row,
                        sparse_mla_fwd_dense, sparse_mla_fwd, sparse_mla_bwd, mla_bwd_delta,
                        indexer_scores_at, mla_teacher, sparse_kl, indexer_bwd,
                        sparse_gqa_fwd, sparse_gqa_bwd, pad_nope, pad_topk, seq_bounds, max_seqlen,
                        as_f64, as_i64)
