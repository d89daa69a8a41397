"""GPU parity: sparse MLA forward/backward against the CPU oracle (fp64),
through the C ABI; exactness of the NoPE and top-k paddings; determinism."""
import functools
import math

import numpy as np
import pytest
import torch

import oracle as O
import synth
from _util import TOL_GRAD, TOL_OUT, check_grad, check_out_lse, rel_l2

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def tsa():
    import trainable_sparse_attention_gb300 as m
    m.build()
    m.load_library()
    return m


def _run_fwd_bwd(tsa, m, idx, cu, scale, bwd=True):
    q, kv = m["q"].to(DEV), m["kv"].to(DEV)
    ids = idx.to(DEV)
    out, lse = tsa.sparse_mla_fwd(q, kv, ids, cu, scale)
    res = {"out": out, "lse": lse}
    if bwd:
        dq, dkv = tsa.sparse_mla_bwd(q, kv, ids, out, lse, m["dout"].to(DEV), cu, scale)
        res.update(dq=dq, dkv=dkv)
    torch.cuda.synchronize()
    return res


def test_mla_t256_h8_forward():
    """T=256, H=8, 576 channels, scale 1/sqrt(576); indices = the oracle's top-64 of
    the indexer (4 heads, d_I=64); forward only."""
    import trainable_sparse_attention_gb300 as tsa
    tsa.build()
    cu = [0, 256]
    x = synth.indexer_inputs(256, 4, 64, seed=0)
    idx = torch.from_numpy(O.qsa_topk(x["q_idx"], x["k_idx"], x["w"], cu, range(256), 64)[:, 0, :].copy())
    m = synth.mla_inputs(256, 8, 576, seed=0)
    scale = 1 / math.sqrt(576)
    r = _run_fwd_bwd(tsa, m, idx, cu, scale, bwd=False)
    o_ref, l_ref = O.sparse_mla_fwd(m["q"], m["kv"], idx, cu, scale)
    check_out_lse(r["out"], r["lse"], o_ref, l_ref)
    # dense-masked definition agrees too
    o_d, l_d = O.sparse_mla_fwd_dense(m["q"], m["kv"], idx, cu, scale)
    check_out_lse(r["out"], r["lse"], o_d, l_d)


@functools.lru_cache(maxsize=None)
def _sweep_indices(topk: int):
    """Indices of the shape-edge sweep: the oracle's top-k of the indexer at seed 1
    (4 heads, d_I = 64), T = 2048; all -1 rows at {0, 97, 1000, 2047} and 1% random."""
    cu = [0, 2048]
    x = synth.indexer_inputs(2048, 4, 64, seed=1)
    idx = O.qsa_topk(x["q_idx"], x["k_idx"], x["w"], cu, range(2048), topk)[:, 0, :].copy()
    g = torch.Generator().manual_seed(1)
    extra = (torch.rand(2048, generator=g) < 0.01).nonzero().flatten().tolist()
    for r in [0, 97, 1000, 2047] + extra:
        idx[r] = -1
    return idx


@pytest.mark.parametrize("D", [512, 576])
@pytest.mark.parametrize("topk", [64, 65, 127])
@pytest.mark.parametrize("H", [8, 16, 32])
def test_mla_shape_sweep_t2048(tsa, D, topk, H):
    cu = [0, 2048]
    idx = torch.from_numpy(_sweep_indices(topk))
    m = synth.mla_inputs(2048, H, D, seed=1 + H + D + topk, with_grad_out=True)
    scale = 1 / math.sqrt(D)
    r = _run_fwd_bwd(tsa, m, idx, cu, scale)
    rows = list(range(0, 2048, 3)) + [97, 1000, 2047]
    o_ref, l_ref = O.sparse_mla_fwd(m["q"], m["kv"], idx, cu, scale, rows=rows)
    check_out_lse(r["out"], r["lse"], o_ref, l_ref, rows=rows)
    dq_ref, dkv_ref = O.sparse_mla_bwd(m["q"], m["kv"], idx, cu, scale, m["dout"])
    check_grad(r["dq"], dq_ref, "dq")
    check_grad(r["dkv"], dkv_ref, "dkv")
    # all-invalid rows: zero output, -inf lse, zero dq
    for row in (0, 97, 1000, 2047):
        assert torch.all(r["out"][row] == 0) and torch.all(torch.isneginf(r["lse"][row]))
        assert torch.all(r["dq"][row] == 0)


def test_mla_nope_and_topk_padding_are_exact(tsa):
    """512-wide NoPE inputs equal their zero-padded 576 form; an unaligned top-k
    equals the same indices -1-padded to a multiple of 64 (bit for bit)."""
    cu = [0, 700]
    m = synth.mla_inputs(700, 16, 512, seed=3, with_grad_out=True)
    idx = synth.random_topk_indices(cu, 65, seed=3)
    scale = 1 / math.sqrt(512)
    a = _run_fwd_bwd(tsa, m, idx, cu, scale)
    pad = {"q": torch.nn.functional.pad(m["q"], (0, 64)), "kv": torch.nn.functional.pad(m["kv"], (0, 64)),
           "dout": m["dout"]}
    idx_p = torch.nn.functional.pad(idx, (0, 63), value=-1)
    b = _run_fwd_bwd(tsa, pad, idx_p, cu, scale)
    assert torch.equal(a["out"], b["out"]) and torch.equal(a["lse"], b["lse"])
    assert torch.equal(a["dq"], b["dq"][..., :512])
    # dKV is accumulated with atomics (summation order not fixed): equal up to
    # fp32 reordering and the final bf16 rounding
    assert rel_l2(a["dkv"], b["dkv"][..., :512]) <= 1e-3
    assert torch.all(b["dq"][..., 512:] == 0) and torch.all(b["dkv"][..., 512:] == 0)
    o_ref, l_ref = O.sparse_mla_fwd(m["q"], m["kv"], idx, cu, scale)
    check_out_lse(a["out"], a["lse"], o_ref, l_ref)
    dq_ref, dkv_ref = O.sparse_mla_bwd(m["q"], m["kv"], idx, cu, scale, m["dout"])
    check_grad(a["dq"], dq_ref, "dq")
    check_grad(a["dkv"], dkv_ref, "dkv")


def test_mla_forward_deterministic_under_contention(tsa):
    cu = [0, 1500]
    m = synth.mla_inputs(1500, 32, 576, seed=4)
    idx = synth.random_topk_indices(cu, 256, seed=4).to(DEV)
    q, kv = m["q"].to(DEV), m["kv"].to(DEV)
    o1, l1 = tsa.sparse_mla_fwd(q, kv, idx, cu, 0.04)
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        big = torch.randn(4096, 4096, device=DEV)
        for _ in range(4):
            big = big @ big.T
            big = big / big.norm()
    o2, l2 = tsa.sparse_mla_fwd(q, kv, idx, cu, 0.04)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_mla_thd_and_index_range_flag(tsa):
    cu = [0, 100, 101, 500]
    m = synth.mla_inputs(500, 8, 576, seed=5, with_grad_out=True)
    idx = synth.random_topk_indices(cu, 64, seed=5)
    scale = 0.05
    tsa.read_flags(clear=True)
    r = _run_fwd_bwd(tsa, m, idx, cu, scale)
    assert tsa.read_flags() == 0
    o_ref, l_ref = O.sparse_mla_fwd(m["q"], m["kv"], idx, cu, scale)
    check_out_lse(r["out"], r["lse"], o_ref, l_ref)
    dq_ref, dkv_ref = O.sparse_mla_bwd(m["q"], m["kv"], idx, cu, scale, m["dout"])
    check_grad(r["dq"], dq_ref, "dq")
    check_grad(r["dkv"], dkv_ref, "dkv")
    # an index beyond its sequence is treated as -1 and raises the flag (no fault)
    bad = idx.clone()
    bad[50, 3] = 100          # sequence 0 has 100 tokens: position 100 is outside it
    o_bad, _ = tsa.sparse_mla_fwd(m["q"].to(DEV), m["kv"].to(DEV), bad.to(DEV), cu, scale)
    assert tsa.read_flags() & tsa.FLAG_INDEX_RANGE
    fixed = bad.clone()
    fixed[50, 3] = -1
    o_fix, _ = tsa.sparse_mla_fwd(m["q"].to(DEV), m["kv"].to(DEV), fixed.to(DEV), cu, scale)
    assert torch.equal(o_bad, o_fix)


@pytest.mark.slow
def test_mla_t4096_h16_topk2048(tsa):
    """T=4096, H=16, 576 channels, top-2048; fwd on sampled rows, bwd exact for dO
    restricted to those rows."""
    cu = [0, 4096]
    m = synth.mla_inputs(4096, 16, 576, seed=6, with_grad_out=True)
    idx = synth.random_topk_indices(cu, 2048, seed=6)
    scale = 1 / math.sqrt(576)
    rows = sorted(set([0, 1, 2047, 2048, 4095] + list(range(3, 4096, 61))))
    mask = torch.zeros(4096, dtype=torch.bool)
    mask[rows] = True
    m["dout"] = torch.where(mask[:, None, None], m["dout"], torch.zeros_like(m["dout"]))
    r = _run_fwd_bwd(tsa, m, idx, cu, scale)
    o_ref, l_ref = O.sparse_mla_fwd(m["q"], m["kv"], idx, cu, scale, rows=rows)
    check_out_lse(r["out"], r["lse"], o_ref, l_ref, rows=rows)
    dq_ref, dkv_ref = O.sparse_mla_bwd(m["q"], m["kv"], idx, cu, scale, m["dout"], rows=rows)
    check_grad(r["dq"].cpu()[rows], dq_ref, "dq")
    check_grad(r["dkv"], dkv_ref, "dkv")


@pytest.mark.slow
def test_mla_t65536_h128_sampled(tsa):
    """T=65536, H=128, 576 channels, top-2048, scale 1/sqrt(192): the bench's
    launch configuration; sampled rows vs the oracle (which widens only the
    rows it needs)."""
    T = 65536
    cu = [0, T]
    m = synth.mla_inputs(T, 128, 576, seed=7, device=DEV, with_grad_out=True)
    idx = synth.spread_topk_indices(cu, 2048, seed=7, device=DEV)
    rows = [0, 1, 2047, 2048, 40000, 65535]
    mask = torch.zeros(T, dtype=torch.bool, device=DEV)
    mask[rows] = True
    m["dout"] = torch.where(mask[:, None, None], m["dout"], torch.zeros_like(m["dout"]))
    scale = 1 / math.sqrt(192)
    out, lse = tsa.sparse_mla_fwd(m["q"], m["kv"], idx, cu, scale)
    dq, dkv = tsa.sparse_mla_bwd(m["q"], m["kv"], idx, out, lse, m["dout"], cu, scale)
    # the bench's launch configuration replays bit-identically (dq has no atomics)
    dq2, _ = tsa.sparse_mla_bwd(m["q"], m["kv"], idx, out, lse, m["dout"], cu, scale)
    torch.cuda.synchronize()
    assert torch.equal(dq, dq2)
    del dq2
    o_ref, l_ref = O.sparse_mla_fwd(m["q"], m["kv"], idx, cu, scale, rows=rows)
    check_out_lse(out, lse, o_ref, l_ref, rows=rows)
    dq_ref, dkv_ref = O.sparse_mla_bwd(m["q"], m["kv"], idx, cu, scale, m["dout"], rows=rows)
    check_grad(dq[rows], dq_ref, "dq")
    check_grad(dkv, dkv_ref, "dkv")


@pytest.mark.parametrize("D,topk,lengths", [
    (576, 64, [300]),            # first 63 rows have fewer than 64 candidates
    (576, 65, [130, 200]),       # ragged last tile, THD
    (576, 1000, [700]),          # top-k wider than the sequence: -1 tails
    (512, 96, [257]),            # NoPE layout
    (576, 2048, [2100]),         # 64 tiles of 32 keys
    (576, 4096, [4200]),         # the widest top-k: 128 tiles
    (576, 1, [200]),             # one slot: a single 32-key tile, 31 slots past topk
    (512, 17, [100, 50]),        # NoPE, a partial first tile, THD
])
def test_mla_h128_forward(tsa, D, topk, lengths):
    """H = 128 (the tcgen05 cluster path): parity with the oracle on sampled rows,
    all-invalid rows exact, bit-identical replay."""
    cu = synth.cu_seqlens_thd(lengths)
    T = cu[-1]
    m = synth.mla_inputs(T, 128, D, seed=T + topk + D)
    idx = synth.random_topk_indices(cu, topk, seed=topk, invalid_rows=[3, T - 1])
    scale = 1 / math.sqrt(D)
    q, kv, ids = m["q"].to(DEV), m["kv"].to(DEV), idx.to(DEV)
    out, lse = tsa.sparse_mla_fwd(q, kv, ids, cu, scale)
    out2, lse2 = tsa.sparse_mla_fwd(q, kv, ids, cu, scale)
    torch.cuda.synchronize()
    assert torch.equal(out, out2) and torch.equal(lse, lse2)
    rows = sorted(set([0, 1, 2, 3, 63, 64, T - 1] + list(range(5, T, max(1, T // 40)))))
    o_ref, l_ref = O.sparse_mla_fwd(m["q"], m["kv"], idx, cu, scale, rows=rows)
    check_out_lse(out, lse, o_ref, l_ref, rows=rows)
    for r in (3, T - 1):
        assert torch.all(out[r] == 0) and torch.all(torch.isneginf(lse[r]))


def test_mla_h128_tiny_sequences(tsa):
    """H = 128 on sequences of 1, 2 and 5 tokens (THD): most slots are -1, the
    first query of each sequence has one valid key; forward and backward on every
    row against the oracle."""
    cu = synth.cu_seqlens_thd([1, 2, 5])
    T = cu[-1]
    m = synth.mla_inputs(T, 128, 576, seed=21, with_grad_out=True)
    idx = synth.random_topk_indices(cu, 64, seed=21)
    scale = 1 / math.sqrt(576)
    q, kv, ids, dO = m["q"].to(DEV), m["kv"].to(DEV), idx.to(DEV), m["dout"].to(DEV)
    out, lse = tsa.sparse_mla_fwd(q, kv, ids, cu, scale)
    dq, dkv = tsa.sparse_mla_bwd(q, kv, ids, out, lse, dO, cu, scale)
    torch.cuda.synchronize()
    o_ref, l_ref = O.sparse_mla_fwd(m["q"], m["kv"], idx, cu, scale)
    check_out_lse(out, lse, o_ref, l_ref)
    dq_ref, dkv_ref = O.sparse_mla_bwd(m["q"], m["kv"], idx, cu, scale, m["dout"])
    check_grad(dq, dq_ref, "dq")
    check_grad(dkv, dkv_ref, "dkv")


def test_mla_h128_large_logits_rescale(tsa):
    """Large, growing logits force the lazy running-max rescale of the output
    accumulator; compare with the oracle."""
    cu = [0, 600]
    m = synth.mla_inputs(600, 128, 576, seed=11)
    m["q"] = (m["q"].float() * 4).to(torch.bfloat16)
    idx = synth.random_topk_indices(cu, 512, seed=11)
    out, lse = tsa.sparse_mla_fwd(m["q"].to(DEV), m["kv"].to(DEV), idx.to(DEV), cu, 0.2)
    rows = list(range(0, 600, 7)) + [599]
    o_ref, l_ref = O.sparse_mla_fwd(m["q"], m["kv"], idx, cu, 0.2, rows=rows)
    check_out_lse(out, lse, o_ref, l_ref, rows=rows)


@pytest.mark.parametrize("D,topk,lengths", [
    (576, 64, [300]),            # short rows: fewer candidates than slots
    (576, 65, [130, 200]),       # THD; slots padded from 65 to 128 for the dKV GEMM
    (576, 1000, [700]),          # -1 tails
    (512, 96, [257]),            # NoPE layout: four 128-channel dKV blocks
    (576, 2048, [2100]),         # 33 tiles of 64 slots
    (576, 4000, [2100, 300]),    # kp = 4096: 2048-query P/dS chunks, a boundary inside sequence 0
    (576, 1, [200]),             # one slot
    (512, 17, [100, 50]),        # NoPE, 17 slots padded to 128
])
def test_mla_h128_backward(tsa, D, topk, lengths):
    """H = 128 backward (recompute of P/dS + tcgen05 dKV GEMM): dO is kept on
    sampled rows only, so the oracle's dq of those rows and its full dkv are
    exact references; dq of the other rows must be zero."""
    cu = synth.cu_seqlens_thd(lengths)
    T = cu[-1]
    m = synth.mla_inputs(T, 128, D, seed=3 * T + topk + D, with_grad_out=True)
    idx = synth.random_topk_indices(cu, topk, seed=topk + 1, invalid_rows=[3, T - 1])
    scale = 1 / math.sqrt(D)
    rows = sorted(set([0, 1, 3, 63, 64, T - 1] + list(range(5, T, max(1, T // 24)))))
    mask = torch.zeros(T, dtype=torch.bool)
    mask[rows] = True
    m["dout"] = torch.where(mask[:, None, None], m["dout"], torch.zeros_like(m["dout"]))
    r = _run_fwd_bwd(tsa, m, idx, cu, scale)
    # dq has no atomics: a second call on the same inputs is bit-identical
    dq2, _ = tsa.sparse_mla_bwd(m["q"].to(DEV), m["kv"].to(DEV), idx.to(DEV), r["out"], r["lse"],
                                m["dout"].to(DEV), cu, scale)
    assert torch.equal(dq2, r["dq"])
    dq_ref, dkv_ref = O.sparse_mla_bwd(m["q"], m["kv"], idx, cu, scale, m["dout"], rows=rows)
    dq = r["dq"].cpu()
    check_grad(dq[rows], dq_ref, "dq")
    check_grad(r["dkv"], dkv_ref, "dkv")
    others = torch.ones(T, dtype=torch.bool)
    others[rows] = False
    assert torch.all(dq[others] == 0)
    untouched = torch.from_numpy(np.abs(np.asarray(dkv_ref)).sum(1) == 0)
    assert torch.all(r["dkv"].cpu()[untouched] == 0)


def test_mla_h128_index_range_flag(tsa):
    """H = 128 (the tcgen05 forward and backward): an index beyond its sequence
    is treated as -1 and raises FLAG_INDEX_RANGE; out, lse and dq equal those
    of the run with the bad slots set to -1 bit for bit (dkv up to the order of
    its atomic sums), and that run matches the oracle."""
    cu = [0, 300, 700]
    T = cu[-1]
    m = synth.mla_inputs(T, 128, 576, seed=21, with_grad_out=True)
    idx = synth.random_topk_indices(cu, 256, seed=21)
    bad = idx.clone()
    bad[50, 3] = 300          # sequence 0 holds local positions 0..299
    bad[400, 0] = 400         # sequence 1 holds local positions 0..399
    bad[650, 255] = 1 << 20
    fixed = bad.clone()
    fixed[50, 3] = fixed[400, 0] = fixed[650, 255] = -1
    scale = 1 / math.sqrt(576)
    tsa.read_flags(clear=True)
    rf = _run_fwd_bwd(tsa, m, fixed, cu, scale)
    assert tsa.read_flags() == 0
    rb = _run_fwd_bwd(tsa, m, bad, cu, scale)
    assert tsa.read_flags() & tsa.FLAG_INDEX_RANGE
    assert torch.equal(rb["out"], rf["out"]) and torch.equal(rb["lse"], rf["lse"])
    assert torch.equal(rb["dq"], rf["dq"])
    assert rel_l2(rb["dkv"], rf["dkv"]) <= 1e-3
    rows = [0, 49, 50, 51, 299, 300, 399, 400, 401, 650, 699]
    o_ref, l_ref = O.sparse_mla_fwd(m["q"], m["kv"], fixed, cu, scale, rows=rows)
    check_out_lse(rf["out"], rf["lse"], o_ref, l_ref, rows=rows)


@pytest.mark.parametrize("H", [48, 64, 96])
def test_mla_tp_head_counts_fwd_bwd(tsa, H):
    """Head counts of a tensor-parallel slice of 128 heads (64), a count that is
    not a power of two (96) and one that splits a warp of rows (48): the forward
    runs on the tcgen05 kernel with the heads padded to 128 rows.  Forward on
    sampled rows (and bit-identical on replay), dq of those rows and the full
    dkv with dO kept on them only."""
    cu = [0, 900, 1500]
    T = cu[-1]
    m = synth.mla_inputs(T, H, 576, seed=H, with_grad_out=True)
    idx = synth.random_topk_indices(cu, 512, seed=H, invalid_rows=[3, T - 1])
    scale = 1 / math.sqrt(576)
    rows = sorted(set([0, 1, 3, 511, 512, 899, 900, 901, T - 1] + list(range(7, T, 97))))
    mask = torch.zeros(T, dtype=torch.bool)
    mask[rows] = True
    m["dout"] = torch.where(mask[:, None, None], m["dout"], torch.zeros_like(m["dout"]))
    r = _run_fwd_bwd(tsa, m, idx, cu, scale)
    out2, lse2 = tsa.sparse_mla_fwd(m["q"].to(DEV), m["kv"].to(DEV), idx.to(DEV), cu, scale)
    torch.cuda.synchronize()
    assert torch.equal(out2, r["out"]) and torch.equal(lse2, r["lse"])
    o_ref, l_ref = O.sparse_mla_fwd(m["q"], m["kv"], idx, cu, scale, rows=rows)
    check_out_lse(r["out"], r["lse"], o_ref, l_ref, rows=rows)
    dq_ref, dkv_ref = O.sparse_mla_bwd(m["q"], m["kv"], idx, cu, scale, m["dout"], rows=rows)
    check_grad(r["dq"].cpu()[rows], dq_ref, "dq")
    check_grad(r["dkv"], dkv_ref, "dkv")
    for row in (3, T - 1):
        assert torch.all(r["out"][row] == 0) and torch.all(torch.isneginf(r["lse"][row]))
