"""C-ABI checks that need no GPU: the library loads, exports every symbol that
include/tsa.h declares, and rejects bad arguments on the host (no launch)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "tsa.h")


@pytest.fixture(scope="module")
def lib():
    import trainable_sparse_attention_gb300 as tsa
    tsa.build()
    return tsa.load_library()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?(?:int|size_t|unsigned long long|char\s*\*|const char\s*\*)\s*\**\s*(\w+)\s*\(",
                       src, re.M)
    return sorted(set(names))


def test_header_declares_entry_points():
    names = declared_functions()
    for n in ("qsa_indexer_scores", "qsa_topk", "qsa_topk_from_scores", "sparse_mla_fwd", "sparse_mla_bwd",
              "sparse_gqa_fwd", "sparse_gqa_bwd", "tsa_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    from trainable_sparse_attention_gb300 import SIGNATURES
    for n in declared_functions():
        assert hasattr(lib, n), f"{n} not exported"
        assert n in SIGNATURES, f"{n} has no binding signature"


def _cu(vals):
    return (ctypes.c_int32 * len(vals))(*vals)


def test_status_strings(lib):
    for code in range(7):
        assert lib.tsa_status_string(code).decode().startswith("TSA_")


def test_host_validation_errors(lib):
    cu = _cu([0, 8])
    fake = ctypes.c_void_p(16)
    # unsupported head dim
    assert lib.sparse_mla_fwd(fake, fake, fake, cu, 1, 8, 100, 64, 0.1, fake, fake, None) == 2
    # too many heads
    assert lib.sparse_mla_fwd(fake, fake, fake, cu, 1, 129, 576, 64, 0.1, fake, fake, None) == 2
    # bad cu_seqlens
    assert lib.sparse_mla_fwd(fake, fake, fake, _cu([1, 8]), 1, 8, 576, 64, 0.1, fake, fake, None) == 1
    assert lib.sparse_mla_fwd(fake, fake, fake, _cu([0, 8, 4]), 2, 8, 576, 64, 0.1, fake, fake, None) == 1
    assert lib.sparse_mla_fwd(fake, fake, fake, None, 1, 8, 576, 64, 0.1, fake, fake, None) == 1
    # null tensor
    assert lib.sparse_mla_fwd(None, fake, fake, cu, 1, 8, 576, 64, 0.1, fake, fake, None) == 1
    # topk range
    assert lib.qsa_topk_from_scores(fake, 4, 16, 16, 0, fake, None) == 2
    assert lib.qsa_topk_from_scores(fake, 4, 16, 16, 5000, fake, None) == 2
    assert lib.qsa_topk_from_scores(fake, 4, 16, 8, 4, fake, None) == 1
    # indexer shapes
    assert lib.qsa_indexer_scores(fake, fake, fake, cu, 1, 6, 64, 1, 1, 1.0, 0, 8, fake, 8, None) == 2
    assert lib.qsa_indexer_scores(fake, fake, fake, cu, 1, 8, 96, 1, 1, 1.0, 0, 8, fake, 8, None) == 2
    assert lib.qsa_indexer_scores(fake, fake, fake, cu, 1, 8, 64, 8, 1, 1.0, 0, 8, fake, 8, None) == 2
    assert lib.qsa_indexer_scores(fake, fake, fake, cu, 1, 8, 64, 1, 3, 1.0, 0, 8, fake, 8, None) == 2
    assert lib.qsa_indexer_scores(fake, fake, fake, cu, 1, 8, 64, 1, 1, 1.0, 4, 8, fake, 8, None) == 1
    assert lib.qsa_indexer_scores(fake, fake, fake, cu, 1, 8, 64, 1, 1, 1.0, 0, 8, fake, 7, None) == 1
    # workspace too small
    assert lib.qsa_topk(fake, fake, fake, cu, 1, 8, 64, 1, 1, 1.0, 4, fake, fake, 1, None) == 3
    assert lib.sparse_mla_bwd(fake, fake, fake, fake, fake, fake, cu, 1, 8, 576, 64, 0.1, fake, fake,
                              None, fake, 16, None) == 3
    # GQA shapes
    assert lib.sparse_gqa_fwd(fake, fake, fake, fake, cu, 1, 32, 3, 128, 64, 4, 0.1, fake, fake, fake, 1 << 40, None) == 2
    assert lib.sparse_gqa_fwd(fake, fake, fake, fake, cu, 1, 32, 4, 96, 64, 4, 0.1, fake, fake, fake, 1 << 40, None) == 2
    assert lib.sparse_gqa_fwd(fake, fake, fake, fake, cu, 1, 32, 4, 128, 16, 4, 0.1, fake, fake, fake, 1 << 40, None) == 2
    assert lib.sparse_gqa_fwd(fake, fake, fake, fake, cu, 1, 32, 4, 128, 64, 4, 0.1, fake, fake, fake, 16, None) == 3
    assert "d_qk" in lib.tsa_last_error().decode() or lib.tsa_last_error().decode()


def test_empty_inputs_are_noops(lib):
    cu = _cu([0, 0])
    fake = ctypes.c_void_p(16)
    assert lib.sparse_mla_fwd(None, None, None, cu, 1, 8, 576, 64, 0.1, None, None, None) == 0
    assert lib.qsa_topk_from_scores(None, 0, 16, 16, 4, None, None) == 0
    assert lib.qsa_topk(None, None, None, cu, 1, 8, 64, 1, 1, 1.0, 4, None, None, 0, None) == 0


def test_workspace_sizes_are_bounded(lib):
    # streaming top-k scratch stays bounded by two query chunks (one being
    # scored while the other is selected), far below T x T
    cu = _cu([0, 65536])
    ws = lib.qsa_topk_workspace_size(cu, 1, 1, 1)
    assert 0 < ws <= 2 * 512 * 2 ** 20 and ws < 65536 * 65536 * 4 // 15
    assert lib.sparse_mla_bwd_workspace_size(1000, 16, 576, 2048) >= 1000 * 576 * 4 + 1000 * 16 * 4
    # the 128-head P/dS staging is one bounded chunk of queries, not T x topk
    big = lib.sparse_mla_bwd_workspace_size(65536, 128, 576, 2048)
    assert big <= 65536 * 576 * 4 + 65536 * 128 * 4 + 4 * 2 ** 30 + 1024
    assert lib.sparse_mla_bwd_workspace_size(64, 128, 576, 100) >= 64 * 128 * 128 * 4
    # fp32 dQ, dK, dV accumulators and the inverted selections (1000 x 4 x 32 entries)
    assert lib.sparse_gqa_bwd_workspace_size(1000, 32, 4, 128, 32) >= (1000 * 32 * 128 + 2 * 1000 * 4 * 128) * 4 \
        + 1000 * 4 * 32 * 4


def test_binding_refuses_cpu_tensors():
    import torch
    import trainable_sparse_attention_gb300 as tsa
    q = torch.zeros(4, 2, 576, dtype=torch.bfloat16)
    kv = torch.zeros(4, 576, dtype=torch.bfloat16)
    idx = torch.zeros(4, 64, dtype=torch.int32)
    with pytest.raises(ValueError, match="CUDA"):
        tsa.sparse_mla_fwd(q, kv, idx, [0, 4], 0.1)


def test_explicit_library_path_serves_later_calls(lib):
    """A build loaded from an explicit path is the one every later call uses."""
    import trainable_sparse_attention_gb300 as tsa
    from trainable_sparse_attention_gb300 import _binding
    try:
        other = tsa.load_library(_binding.LIB_PATH)
        assert tsa.load_library() is other
    finally:
        _binding._lib = lib


def test_backward_and_sequence_table_validation(lib):
    """More refusals decided on the host before any launch: the backward entry
    points, the sequence table's size limit and the GQA selection width."""
    cu = _cu([0, 8])
    fake = ctypes.c_void_p(16)
    # MLA backward: a null gradient pointer, an unsupported width
    assert lib.sparse_mla_bwd(fake, fake, fake, fake, fake, None, cu, 1, 8, 576, 64, 0.1, fake, fake,
                              None, fake, 1 << 30, None) == 1
    assert lib.sparse_mla_bwd(fake, fake, fake, fake, fake, fake, cu, 1, 8, 320, 64, 0.1, fake, fake,
                              None, fake, 1 << 30, None) == 2
    # indexer training: d_I other than 128, topk beyond 4096, null loss, workspace too small
    assert lib.qsa_indexer_kl(fake, fake, fake, cu, 1, 64, 64, 1.0, fake, 64, fake, fake, fake, None) == 2
    assert lib.qsa_indexer_kl(fake, fake, fake, cu, 1, 64, 128, 1.0, fake, 5000, fake, fake, fake, None) == 2
    assert lib.qsa_indexer_kl(fake, fake, fake, cu, 1, 64, 128, 1.0, fake, 64, fake, None, fake, None) == 1
    assert lib.qsa_indexer_bwd_workspace_size(8, 128) == 4096
    assert lib.qsa_indexer_bwd(fake, fake, fake, cu, 1, 64, 128, 1.0, fake, 64, fake, fake, fake, fake,
                               fake, 16, None) == 3
    # GQA backward: group size above 16, zero selected blocks, workspace too small, null dq
    args = lambda Hq, Hkv, nsel, dq, ws_bytes: (fake, fake, fake, fake, fake, fake, fake, cu, 1, Hq, Hkv, 128,
                                               64, nsel, 0.1, dq, fake, fake, fake, ws_bytes, None)
    assert lib.sparse_gqa_bwd(*args(64, 2, 4, fake, 1 << 30)) == 2
    assert lib.sparse_gqa_bwd(*args(32, 4, 0, fake, 1 << 30)) == 1
    assert lib.sparse_gqa_bwd(*args(32, 4, 4, fake, 16)) == 3
    assert lib.sparse_gqa_bwd(*args(32, 4, 4, None, 1 << 30)) == 1
    # more sequences than the kernels' sequence table holds
    n = 1025
    many = _cu(list(range(n + 1)))
    assert lib.sparse_mla_fwd(fake, fake, fake, many, n, 8, 576, 64, 0.1, fake, fake, None) == 1
