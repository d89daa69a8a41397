"""GPU parity: block Sparse-GQA forward/backward against the CPU oracle."""
import math

import numpy as np
import pytest
import torch

import oracle as O
import synth
from _util import check_grad, check_out_lse

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def tsa():
    import trainable_sparse_attention_gb300 as m
    m.build()
    m.load_library()
    return m


@pytest.mark.parametrize("Hq,Hkv,d,bs,nsel,lengths", [
    (8, 2, 128, 64, 4, [100, 300, 64]),
    (32, 4, 128, 64, 32, [700, 1300]),
    (4, 4, 64, 32, 5, [33, 250]),
    (16, 1, 64, 64, 3, [500]),
    (12, 2, 128, 32, 7, [129, 64, 400]),
    (8, 2, 128, 64, 1, [300, 90]),         # one selected block per query and group
    (8, 4, 64, 64, 3, [1, 3, 70]),         # sequences of 1 and 3 tokens
])
def test_gqa_fwd_bwd(tsa, Hq, Hkv, d, bs, nsel, lengths):
    cu = synth.cu_seqlens_thd(lengths)
    T = cu[-1]
    g = synth.gqa_inputs(T, Hq, Hkv, d, seed=Hq + d + bs, with_grad_out=True)
    blk = synth.random_block_indices(cu, Hkv, nsel, bs, seed=nsel)
    blk[min(5, T - 1)] = -1                    # an empty row
    scale = 1 / math.sqrt(d)
    q, k, v, dO = (g[n].to(DEV) for n in ("q", "k", "v", "dout"))
    out, lse = tsa.sparse_gqa_fwd(q, k, v, blk.to(DEV), cu, bs, scale)
    dq, dk, dv = tsa.sparse_gqa_bwd(q, k, v, blk.to(DEV), out, lse, dO, cu, bs, scale)
    torch.cuda.synchronize()
    o_r, l_r = O.sparse_gqa_fwd(g["q"], g["k"], g["v"], blk, cu, bs, scale)
    check_out_lse(out, lse, o_r, l_r)
    dq_r, dk_r, dv_r = O.sparse_gqa_bwd(g["q"], g["k"], g["v"], blk, cu, bs, scale, g["dout"])
    for name, got, ref in (("dq", dq, dq_r), ("dk", dk, dk_r), ("dv", dv, dv_r)):
        check_grad(got, ref, name)
    assert torch.all(out[min(5, T - 1)] == 0)


def test_gqa_bwd_lists_longer_than_a_chunk(tsa):
    """Every query selects block 0 (plus two others), so the inverted list of
    block 0 holds all 1300 queries of the sequence: the backward splits it over
    several CTAs whose dK/dV partial sums meet in the fp32 workspace."""
    cu = [0, 1300]
    T, Hq, Hkv, d, bs, nsel = 1300, 8, 1, 64, 64, 3
    g = synth.gqa_inputs(T, Hq, Hkv, d, seed=31, with_grad_out=True)
    blk = synth.random_block_indices(cu, Hkv, nsel, bs, seed=31)
    has0 = (blk == 0).any(dim=2, keepdim=True)
    blk[:, :, :1] = torch.where(has0, blk[:, :, :1], torch.zeros_like(blk[:, :, :1]))
    assert bool((blk == 0).any(dim=2).all())
    scale = 1 / math.sqrt(d)
    q, k, v, dO = (g[n].to(DEV) for n in ("q", "k", "v", "dout"))
    out, lse = tsa.sparse_gqa_fwd(q, k, v, blk.to(DEV), cu, bs, scale)
    dq, dk, dv = tsa.sparse_gqa_bwd(q, k, v, blk.to(DEV), out, lse, dO, cu, bs, scale)
    torch.cuda.synchronize()
    dq_r, dk_r, dv_r = O.sparse_gqa_bwd(g["q"], g["k"], g["v"], blk, cu, bs, scale, g["dout"])
    for name, got, ref in (("dq", dq, dq_r), ("dk", dk, dk_r), ("dv", dv, dv_r)):
        check_grad(got, ref, name)


def test_gqa_forward_deterministic(tsa):
    cu = [0, 900]
    g = synth.gqa_inputs(900, 16, 2, 128, seed=3)
    blk = synth.random_block_indices(cu, 2, 8, 64, seed=3).to(DEV)
    q, k, v = (g[n].to(DEV) for n in ("q", "k", "v"))
    a = tsa.sparse_gqa_fwd(q, k, v, blk, cu, 64, 0.1)
    b = tsa.sparse_gqa_fwd(q, k, v, blk, cu, 64, 0.1)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


@pytest.mark.slow
def test_gqa_thd32768_sampled(tsa):
    """Packed THD of 4 sequences (4096/8192/12288/8192), Hq=32, Hkv=4, d=128,
    block_size 64, 32 blocks per (query, group); sampled rows vs the oracle."""
    cu = synth.cu_seqlens_thd([4096, 8192, 12288, 8192])
    T = cu[-1]
    g = synth.gqa_inputs(T, 32, 4, 128, seed=8, device=DEV, with_grad_out=True)
    blk = synth.spread_block_indices(cu, 4, 32, 64, seed=20, device=DEV)
    rows = [0, 63, 64, 4095, 4096, 4160, 12287, 12288, 24576, 32767] + list(range(777, T, 3331))
    mask = torch.zeros(T, dtype=torch.bool, device=DEV)
    mask[rows] = True
    g["dout"] = torch.where(mask[:, None, None], g["dout"], torch.zeros_like(g["dout"]))
    scale = 1 / math.sqrt(128)
    out, lse = tsa.sparse_gqa_fwd(g["q"], g["k"], g["v"], blk, cu, 64, scale)
    dq, dk, dv = tsa.sparse_gqa_bwd(g["q"], g["k"], g["v"], blk, out, lse, g["dout"], cu, 64, scale)
    torch.cuda.synchronize()
    o_r, l_r = O.sparse_gqa_fwd(g["q"], g["k"], g["v"], blk, cu, 64, scale, rows=rows)
    check_out_lse(out, lse, o_r, l_r, rows=rows)
    dq_r, dk_r, dv_r = O.sparse_gqa_bwd(g["q"], g["k"], g["v"], blk, cu, 64, scale, g["dout"], rows=rows)
    check_grad(dq[rows], dq_r, "dq")
    check_grad(dk, dk_r, "dk")
    check_grad(dv, dv_r, "dv")

