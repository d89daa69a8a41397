"""qsa_topk_no_alloc: the allocation-free streaming indexer + top-k.

This entry point serves callers that cannot give the library device memory
for scratch (hosts with a fixed memory budget, allocation-free serving loops,
plugin interfaces that pass only inputs and outputs).  It keeps its scratch
in a fixed device array inside the library.  The test calls it through the
C ABI, twice in a row (the second call reuses the array the first one left
behind), and checks that its indices equal those of qsa_topk, the entry point
that takes a caller-provided workspace.  It also checks the host-side refusal
of a problem whose score row does not fit the fixed array.

Kept in a file that pytest collects last, so that a run stopping at the first
failure has already run every other test; it passes alone in a fresh process
as well (the first call on the device performs the one-time address lookup).
"""
import ctypes

import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def tsa():
    import trainable_sparse_attention_gb300 as m
    m.build()
    m.load_library()
    return m


def _cu(vals):
    return (ctypes.c_int32 * len(vals))(*vals), len(vals) - 1


def _no_alloc(lib, x, cu_list, H_I, d_I, groups, bs, topk, out):
    cu, nseq = _cu(cu_list)
    rc = lib.qsa_topk_no_alloc(x["q_idx"].data_ptr(), x["k_idx"].data_ptr(), x["w"].data_ptr(), cu, nseq,
                               H_I, d_I, groups, bs, 1.0, topk, out.data_ptr(),
                               torch.cuda.current_stream().cuda_stream)
    return rc


@pytest.mark.parametrize("H_I,d_I,groups,bs,topk,lengths", [
    (8, 128, 1, 1, 2048, [9000]),            # many chunks: a row of 9000 scores, ~466 rows per chunk
    (64, 128, 1, 1, 256, [3000, 20000]),     # long sequence: ~209 rows per chunk
    (8, 128, 4, 64, 32, [4096, 8192, 300]),  # block scores, 4 groups
])
def test_no_alloc_matches_workspace_entry_point(tsa, H_I, d_I, groups, bs, topk, lengths):
    lib = tsa.load_library()
    cu = synth.cu_seqlens_thd(lengths)
    T = cu[-1]
    x = {k: v.to(DEV) for k, v in synth.indexer_inputs(T, H_I, d_I, seed=T + groups, zero_key_frac=0.3).items()}
    ref = tsa.qsa_topk(x["q_idx"], x["k_idx"], x["w"], cu, topk, groups=groups, block_size=bs)
    tsa.read_flags(clear=True)
    for call in range(2):
        out = torch.full((T, groups, topk), -7, dtype=torch.int32, device=DEV)
        rc = _no_alloc(lib, x, cu, H_I, d_I, groups, bs, topk, out)
        assert rc == 0, lib.tsa_last_error().decode()
        torch.cuda.synchronize()
        # no bounded wait gave up (a timeout would raise FLAG_TIMEOUT here)
        assert tsa.read_flags() == 0, f"call {call}: device flags raised"
        assert torch.equal(out, ref), f"call {call}: indices differ from qsa_topk"


def test_no_alloc_second_problem_after_first(tsa):
    """A smaller problem right after a larger one: leftovers in the shared
    array must not leak into the result."""
    lib = tsa.load_library()
    for T in (5000, 700):
        cu = [0, T]
        x = {k: v.to(DEV) for k, v in synth.indexer_inputs(T, 8, 128, seed=T).items()}
        ref = tsa.qsa_topk(x["q_idx"], x["k_idx"], x["w"], cu, 512)
        out = torch.empty((T, 1, 512), dtype=torch.int32, device=DEV)
        assert _no_alloc(lib, x, cu, 8, 128, 1, 1, 512, out) == 0
        torch.cuda.synchronize()
        assert tsa.read_flags() == 0
        assert torch.equal(out, ref)


def test_no_alloc_refuses_rows_beyond_scratch(tsa):
    lib = tsa.load_library()
    fake = ctypes.c_void_p(256)
    cu, nseq = _cu([0, 5_000_000])          # 20 MB of scores for one row > 16 MiB
    rc = lib.qsa_topk_no_alloc(fake, fake, fake, cu, nseq, 8, 128, 1, 1, 1.0, 64, fake, None)
    assert rc == 2
    assert "fixed scratch" in lib.tsa_last_error().decode()
