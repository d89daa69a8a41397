"""GPU parity: indexer scores, exact top-k and the streaming indexer + top-k,
against the CPU oracle, through the C ABI."""
import math

import numpy as np
import pytest
import torch

import oracle as O
import synth
from _util import compare_topk_rows, indexer_score_bound

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tsa():
    import trainable_sparse_attention_gb300 as m
    m.build()
    m.load_library()
    return m


DEV = "cuda"


# ------------------------------------------------------------ top-k from scores

@pytest.mark.parametrize("rows,L,k", [(64, 50, 7), (64, 333, 64), (32, 4096, 2048), (16, 5000, 65),
                                      (8, 20011, 2048), (4, 65536, 2048), (8, 70000, 4096), (3, 9000, 1),
                                      (128, 256, 64), (40, 129, 200), (9, 31, 31), (5, 1, 3)])
def test_topk_from_scores_bit_exact(tsa, rows, L, k):
    """Tie-stress rows (+-0, -inf, repeated values) of every length class: one
    warp per row up to 256 entries, one CTA per row beyond; k above the row
    length pads with -1."""
    s = synth.tie_stress_scores(rows, L, seed=rows + L + k)
    got = tsa.qsa_topk_from_scores(s.to(DEV), k).cpu().numpy()
    ref = O.topk_rows(s.numpy(), k)
    np.testing.assert_array_equal(got, ref)


def test_topk_from_scores_all_masked_and_tiny_rows(tsa):
    s = torch.full((5, 10), -math.inf)
    s[1, 3] = 0.0
    s[2, :] = -0.0
    s[3, 9] = -1.0
    s[4, ::2] = 2.0
    got = tsa.qsa_topk_from_scores(s.to(DEV), 4).cpu().numpy()
    np.testing.assert_array_equal(got, O.topk_rows(s.numpy(), 4))
    assert np.all(got[0] == -1)


def test_topk_from_scores_distinct_random(tsa):
    g = torch.Generator().manual_seed(5)
    s = torch.randn((12, 30000), generator=g)
    got = tsa.qsa_topk_from_scores(s.to(DEV), 1000).cpu().numpy()
    np.testing.assert_array_equal(got, O.topk_rows(s.numpy(), 1000))


@pytest.mark.parametrize("L,k", [(20000, 2048), (9000, 1), (12000, 300), (15000, 700), (70000, 4096),
                                 (5000, 4096), (65536, 2048)])
def test_topk_from_scores_selection_branches(tsa, L, k):
    """Long rows through each branch of the selection: distinct values (the
    threshold bin fits the key buffer), a tie level of 5000 equal scores at the
    threshold (it does not: the exact three-digit search), and rows with fewer
    finite entries than k (all kept)."""
    g = torch.Generator().manual_seed(L + k)
    distinct = torch.randn((2, L), generator=g)
    ties = torch.randn((2, L), generator=g) * 0.1
    ties[:, torch.randperm(L, generator=g)[:5000]] = 1.0    # 5000 exact ties just below the top
    ties[:, torch.randperm(L, generator=g)[:k // 2]] = 5.0   # k/2 clear winners (also tied)
    sparse = torch.full((2, L), -math.inf)
    keep = torch.randperm(L, generator=g)[:max(1, k - 7)]
    sparse[:, keep] = torch.randn((2, keep.numel()), generator=g).abs().round()  # few distinct values, +0.0 ties
    s = torch.cat([distinct, ties, sparse]).contiguous()
    got = tsa.qsa_topk_from_scores(s.to(DEV), k).cpu().numpy()
    np.testing.assert_array_equal(got, O.topk_rows(s.numpy(), k))


def test_topk_from_scores_bucket_ranking_and_its_fallback(tsa):
    """Long rows whose guided candidates are ranked by buckets of their order
    key: distinct scores packed into a narrow range (small buckets), 200 exact
    ties inside the top k (one bucket over its limit: the sort instead), and
    one huge outlier that squeezes every other candidate into a few buckets."""
    g = torch.Generator().manual_seed(77)
    L, k = 30000, 2048
    tight = (1.0 + 1e-7 * torch.arange(L, dtype=torch.float64))[torch.randperm(L, generator=g)].float()
    tied = torch.randn(L, generator=g)
    tied[torch.randperm(L, generator=g)[:200]] = 2.0           # inside the top 2048 of N(0, 1)
    outlier = torch.randn(L, generator=g)
    outlier[123] = 1e30
    s = torch.stack([tight, tied, outlier, torch.randn(L, generator=g)]).contiguous()
    got = tsa.qsa_topk_from_scores(s.to(DEV), k).cpu().numpy()
    np.testing.assert_array_equal(got, O.topk_rows(s.numpy(), k))


def test_topk_deterministic_replay_under_contention(tsa):
    s = synth.tie_stress_scores(256, 12000, seed=9).to(DEV)
    a = tsa.qsa_topk_from_scores(s, 2048)
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        big = torch.randn(4096, 4096, device=DEV)
        for _ in range(4):
            big = big @ big.T
            big = big / big.norm()
    b = tsa.qsa_topk_from_scores(s, 2048)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


# ------------------------------------------------------------ indexer scores

@pytest.mark.parametrize("H_I,d_I,groups,cu", [(4, 64, 1, [0, 256]), (8, 128, 1, [0, 300, 1000]),
                                               (8, 128, 4, [0, 130, 700]), (64, 128, 1, [0, 520]),
                                               (16, 64, 2, [0, 1, 257, 390])])
def test_indexer_scores_exact_inputs_bit_exact(tsa, H_I, d_I, groups, cu):
    T = cu[-1]
    x = synth.indexer_inputs(T, H_I, d_I, seed=H_I + d_I + groups, integer=True)
    got = tsa.qsa_indexer_scores(x["q_idx"].to(DEV), x["k_idx"].to(DEV), x["w"].to(DEV), cu,
                                 groups=groups).cpu().numpy()
    ref = O.indexer_token_scores(x["q_idx"], x["k_idx"], x["w"], cu, range(T), groups)
    np.testing.assert_array_equal(got, ref)


@pytest.mark.parametrize("H_I,d_I,groups,bs,cu", [(4, 64, 1, 1, [0, 256]), (8, 128, 4, 64, [0, 300, 1000]),
                                                  (64, 128, 1, 1, [0, 700]), (8, 128, 1, 32, [0, 450])])
def test_indexer_scores_randn_within_bound(tsa, H_I, d_I, groups, bs, cu):
    T = cu[-1]
    x = synth.indexer_inputs(T, H_I, d_I, seed=3, zero_key_frac=0.3)
    got = tsa.qsa_indexer_scores(x["q_idx"].to(DEV), x["k_idx"].to(DEV), x["w"].to(DEV), cu, groups=groups,
                                 block_size=bs, score_scale=0.5).cpu().numpy()
    if bs == 1:
        ref = O.indexer_token_scores(x["q_idx"], x["k_idx"], x["w"], cu, range(T), groups, 0.5)
    else:
        ref = O.indexer_block_scores(x["q_idx"], x["k_idx"], x["w"], cu, range(T), bs, groups, 0.5)
    assert np.array_equal(np.isneginf(got), np.isneginf(ref)), "candidate pattern differs"
    fin = np.isfinite(ref)
    for t in range(0, T, 37):
        tol = 0.5 * indexer_score_bound(x["q_idx"], x["k_idx"], x["w"], cu, t, groups)
        for g in range(groups):
            f = fin[t, g]
            err = np.max(np.abs(got[t, g][f].astype(np.float64) - ref[t, g][f])) if f.any() else 0.0
            assert err <= tol[g] + 1e-30, (t, g, err, tol[g])
    # exact zeros (zero keys) are exact on both sides
    assert np.array_equal(got[fin] == 0, ref[fin] == 0)


# ------------------------------------------------------------ streaming indexer + top-k

@pytest.mark.parametrize("H_I,d_I,groups,bs,topk,cu", [
    (4, 64, 1, 1, 64, [0, 256]),
    (8, 128, 1, 1, 2048, [0, 700, 2600]),
    (64, 128, 1, 1, 128, [0, 1100]),
    (8, 128, 4, 64, 32, [0, 900, 3000]),
    (8, 128, 1, 1, 65, [0, 5, 300]),
])
def test_qsa_topk_exact_inputs_bit_exact(tsa, H_I, d_I, groups, bs, topk, cu):
    T = cu[-1]
    x = synth.indexer_inputs(T, H_I, d_I, seed=11, integer=True)
    got = tsa.qsa_topk(x["q_idx"].to(DEV), x["k_idx"].to(DEV), x["w"].to(DEV), cu, topk, groups=groups,
                       block_size=bs).cpu().numpy()
    ref = O.qsa_topk(x["q_idx"], x["k_idx"], x["w"], cu, range(T), topk, groups, bs)
    np.testing.assert_array_equal(got, ref)


def test_qsa_topk_zero_tie_stress_t4096(tsa):
    """T=4096, 8 indexer heads, d_I=128, 30% zero keys, 16 dead queries, k=2048."""
    cu = [0, 4096]
    x = synth.indexer_inputs(4096, 8, 128, seed=2, zero_key_frac=0.3, dead_queries=16)
    got = tsa.qsa_topk(x["q_idx"].to(DEV), x["k_idx"].to(DEV), x["w"].to(DEV), cu, 2048).cpu().numpy()
    dead = np.nonzero(np.all(x["q_idx"].float().numpy() == 0, axis=(1, 2)))[0]
    rows = sorted(set(list(range(0, 4096, 97)) + [0, 1, 2047, 2048, 4095] + dead.tolist()))
    sc = O.indexer_token_scores(x["q_idx"], x["k_idx"], x["w"], cu, rows)
    mism = 0
    for i, t in enumerate(rows):
        tol = indexer_score_bound(x["q_idx"], x["k_idx"], x["w"], cu, t)[0]
        mism += compare_topk_rows(got[t, 0], sc[i, 0], 2048, tol)
    for t in dead:  # all-zero rows: pure index order
        want = np.arange(min(t + 1, 2048))
        np.testing.assert_array_equal(got[t, 0, :want.size], want)
    assert mism <= 0.001 * len(rows) * 2048


@pytest.mark.parametrize("H_I,d_I,groups,bs,topk,cu", [
    (8, 128, 1, 1, 2048, [0, 4096]),
    (64, 128, 1, 1, 512, [0, 1000, 3000]),
    (8, 128, 4, 64, 32, [0, 1000, 4096]),
    (16, 64, 2, 32, 20, [0, 77, 2000]),
])
def test_qsa_topk_equals_topk_of_its_own_scores(tsa, H_I, d_I, groups, bs, topk, cu):
    """On N(0,1) inputs (scores are not exact in fp32), the fused streaming
    qsa_topk selects exactly the top-k of the fp32 scores that qsa_indexer_scores
    produces, byte for byte: the selection itself adds no error."""
    T = cu[-1]
    x = {k: v.to(DEV) for k, v in synth.indexer_inputs(T, H_I, d_I, seed=T + bs, zero_key_frac=0.3).items()}
    got = tsa.qsa_topk(x["q_idx"], x["k_idx"], x["w"], cu, topk, groups=groups, block_size=bs)
    sc = tsa.qsa_indexer_scores(x["q_idx"], x["k_idx"], x["w"], cu, groups=groups, block_size=bs)
    sel = tsa.qsa_topk_from_scores(sc, topk)
    assert torch.equal(sel, got)
    # and those scores select, on the CPU, what the GPU selects (the oracle's
    # exact top-k of the same fp32 buffer)
    scn = sc.cpu().numpy()
    for t in range(0, T, max(1, T // 64)):
        for g in range(groups):
            np.testing.assert_array_equal(got[t, g].cpu().numpy(), O.topk_lex(scn[t, g], topk))


def test_qsa_topk_deterministic(tsa):
    cu = [0, 3000]
    x = synth.indexer_inputs(3000, 8, 128, seed=4, zero_key_frac=0.3)
    args = (x["q_idx"].to(DEV), x["k_idx"].to(DEV), x["w"].to(DEV), cu, 512)
    a = tsa.qsa_topk(*args)
    b = tsa.qsa_topk(*args)
    assert torch.equal(a, b)


def test_qsa_topk_on_a_side_stream(tsa):
    """The streamed runner forks from and joins back into the caller's stream:
    called on a side stream (several chunks: two score buffers reused), its
    indices are complete once that stream is, and equal the default stream's;
    work queued on the side stream after the call sees the finished indices."""
    T = 24000
    cu = [0, 3000, T]  # 512 MB score chunks of 6272 rows: one chunk, then four
    x = synth.indexer_inputs(T, 64, 128, seed=8)
    args = (x["q_idx"].to(DEV), x["k_idx"].to(DEV), x["w"].to(DEV), cu, 1024)
    ref = tsa.qsa_topk(*args)
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        got = tsa.qsa_topk(*args, stream=side)
        total = got.to(torch.int64).sum()          # ordered after the call on the side stream
    side.synchronize()
    assert torch.equal(got, ref)
    assert total.item() == ref.to(torch.int64).sum().item()


@pytest.mark.slow
def test_qsa_topk_t65536_sampled(tsa):
    """T=65536, 64 indexer heads, d_I=128, k=2048; sampled rows vs the oracle."""
    T = 65536
    cu = [0, T]
    x = synth.indexer_inputs(T, 64, 128, seed=5, device=DEV)
    got = tsa.qsa_topk(x["q_idx"], x["k_idx"], x["w"], cu, 2048)
    rows = [0, 1, 2046, 2047, 2048, 30000, 65535] + list(range(1000, T, 9973))
    xc = {k: v.cpu() for k, v in x.items()}
    sc = O.indexer_token_scores(xc["q_idx"], xc["k_idx"], xc["w"], cu, rows)
    g = got.cpu().numpy()
    mism = 0
    for i, t in enumerate(rows):
        tol = indexer_score_bound(xc["q_idx"], xc["k_idx"], xc["w"], cu, t)[0]
        mism += compare_topk_rows(g[t, 0], sc[i, 0], 2048, tol)
    print(f"T=65536 top-2048: {mism} of {len(rows) * 2048} sampled slots differ from the oracle "
          "(each within the fp32 score bound)")
    assert mism <= 0.001 * len(rows) * 2048
    # the fused streaming call selects exactly the top-k of its own fp32 scores:
    # one 512-query chunk through qsa_indexer_scores + qsa_topk_from_scores
    q0, nq = 40000, 512
    sc_gpu = tsa.qsa_indexer_scores(x["q_idx"], x["k_idx"], x["w"], cu, q_begin=q0, q_count=nq)
    sel = tsa.qsa_topk_from_scores(sc_gpu, 2048)
    assert torch.equal(sel, got[q0:q0 + nq])


@pytest.mark.slow
def test_qsa_topk_block_thd32768_sampled(tsa):
    """Packed THD of 4 sequences (4096/8192/12288/8192), 8 heads in 4 groups,
    block_size 64, top-32 blocks; sampled rows vs the oracle."""
    cu = synth.cu_seqlens_thd([4096, 8192, 12288, 8192])
    T = cu[-1]
    x = synth.indexer_inputs(T, 8, 128, seed=6, device=DEV)
    got = tsa.qsa_topk(x["q_idx"], x["k_idx"], x["w"], cu, 32, groups=4, block_size=64).cpu().numpy()
    rows = [0, 63, 64, 4095, 4096, 4097, 12287, 12288, 24575, 24576, 32767] + list(range(500, T, 1999))
    xc = {k: v.cpu() for k, v in x.items()}
    sc = O.indexer_block_scores(xc["q_idx"], xc["k_idx"], xc["w"], cu, rows, 64, 4)
    mism = 0
    for i, t in enumerate(rows):
        tol = indexer_score_bound(xc["q_idx"], xc["k_idx"], xc["w"], cu, t, 4)
        for g in range(4):
            mism += compare_topk_rows(got[t, g], sc[i, g], 32, tol[g])
    print(f"THD 32768 block top-32: {mism} of {len(rows) * 4 * 32} sampled slots differ from the oracle "
          "(each within the fp32 score bound)")
    assert mism <= 0.001 * len(rows) * 4 * 32
    # fused call == exact top-k of its own block scores, for every query (bit for bit)
    sc_gpu = tsa.qsa_indexer_scores(x["q_idx"], x["k_idx"], x["w"], cu, groups=4, block_size=64)
    sel = tsa.qsa_topk_from_scores(sc_gpu, 32).cpu().numpy()
    np.testing.assert_array_equal(sel, got)
