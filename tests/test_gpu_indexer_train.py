"""GPU parity: the indexer's training step on the selected slots -- the
attention teacher (head mean of P, an output of the MLA backward), the sparse
KL of the student scores against it, and the indexer backward -- against the
CPU oracle, through the C ABI."""
import math

import numpy as np
import pytest
import torch

import oracle as O
import synth
from _util import TOL_GRAD, TOL_OUT, check_grad, check_rows, rel_l2

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def tsa():
    import trainable_sparse_attention_gb300 as m
    m.build()
    m.load_library()
    return m


def _teacher_case(tsa, T, H, topk, cu, seed, rows, D=576):
    m = synth.mla_inputs(T, H, D, seed=seed, with_grad_out=True)
    idx = synth.random_topk_indices(cu, topk, seed=seed, invalid_rows=[3])
    scale = 1 / math.sqrt(D)
    q, kv, ids, dO = m["q"].to(DEV), m["kv"].to(DEV), idx.to(DEV), m["dout"].to(DEV)
    out, lse = tsa.sparse_mla_fwd(q, kv, ids, cu, scale)
    dq, dkv, teacher = tsa.sparse_mla_bwd(q, kv, ids, out, lse, dO, cu, scale, want_teacher=True)
    torch.cuda.synchronize()
    ref = O.mla_teacher(m["q"], m["kv"], idx, cu, scale, rows=rows)
    return teacher.cpu(), ref, idx


@pytest.mark.parametrize("H,topk,lengths,D", [(8, 64, [300], 576), (16, 200, [130, 400], 576),
                                              (64, 96, [500], 576), (128, 256, [700], 576),
                                              (128, 65, [130, 200], 576), (128, 200, [400], 512)])
def test_teacher_from_mla_backward(tsa, H, topk, lengths, D):
    """The teacher output of sparse_mla_bwd equals the oracle's head-averaged
    attention probabilities on the selected slots (rows: rel-L2 within the
    output tolerance; -1 slots exactly 0; every valid row sums to 1).  H = 128
    with 576 channels takes it from the dKV GEMM, with 512 from the staged P,
    H < 128 from the head blocks of the small-H kernel."""
    cu = synth.cu_seqlens_thd(lengths)
    T = cu[-1]
    rows = sorted(set([0, 1, 3, 63, 64, T - 1] + list(range(5, T, max(1, T // 40)))))
    got, ref, idx = _teacher_case(tsa, T, H, topk, cu, H + topk, rows, D)
    g = got[rows].double().numpy()
    check_rows(g, ref, TOL_OUT, "teacher rows")
    assert rel_l2(g, ref) <= TOL_OUT
    inval = (idx[rows] < 0).numpy()
    assert np.all(g[inval] == 0)
    sums = g.sum(axis=1)
    has = (~inval).any(axis=1)
    np.testing.assert_allclose(sums[has], 1.0, atol=1e-2)
    assert np.all(g[~has] == 0)


@pytest.mark.parametrize("H_I,topk,lengths,scale", [(8, 2048, [4096], 1.0), (64, 512, [700, 1300], 0.5),
                                                    (64, 130, [300], 1.0), (128, 256, [600], 0.25),
                                                    (16, 65, [5, 300], 1.0)])
def test_indexer_kl_and_backward(tsa, H_I, topk, lengths, scale):
    """qsa_indexer_kl (student scores at the selected slots, KL against the
    teacher, dI = p - a) and qsa_indexer_bwd (dq_I, dk_I, dw for that dI) vs the
    oracle; indices from the streaming top-k (30% zero keys: ReLU ties), the
    teacher from the oracle; dI is kept on sampled rows only so that the
    oracle's dk_I is exact."""
    cu = synth.cu_seqlens_thd(lengths)
    T = cu[-1]
    x = synth.indexer_inputs(T, H_I, 128, seed=H_I + topk, zero_key_frac=0.3)
    xd = {k: v.to(DEV) for k, v in x.items()}
    sel = tsa.qsa_topk(xd["q_idx"], xd["k_idx"], xd["w"], cu, topk, score_scale=scale)[:, 0, :].contiguous()
    idx = sel.cpu()
    idx[min(3, T - 1)] = -1                                   # an all-invalid row
    sel = idx.to(DEV)
    rows = sorted(set([0, 1, min(3, T - 1), T // 2, T - 1] + list(range(7, T, max(1, T // 24)))))
    # teacher: any distribution over the valid slots; the oracle's attention
    # teacher of a small MLA problem on the same indices
    m = synth.mla_inputs(T, 4, 64, seed=topk)
    tea = np.zeros((T, topk))
    tea[rows] = O.mla_teacher(m["q"], m["kv"], idx, cu, 0.125, rows=rows)
    teacher = torch.from_numpy(tea).float().to(DEV)
    tsa.read_flags(clear=True)
    loss, dscore = tsa.qsa_indexer_kl(xd["q_idx"], xd["k_idx"], xd["w"], cu, sel, teacher, score_scale=scale)
    torch.cuda.synchronize()
    assert tsa.read_flags() == 0
    sc_ref = O.indexer_scores_at(x["q_idx"], x["k_idx"], x["w"], cu, idx[:, None, :], score_scale=scale,
                                 rows=rows)[:, 0, :]
    loss_ref, g_ref = O.sparse_kl(sc_ref, tea[rows])
    g_gpu = dscore.cpu().double().numpy()[rows]
    check_rows(g_gpu, g_ref, TOL_OUT, "dI rows")
    l_gpu = loss.cpu().double().numpy()[rows]
    assert np.max(np.abs(l_gpu - loss_ref)) <= TOL_OUT * max(1.0, float(np.max(np.abs(loss_ref))))
    assert loss[min(3, T - 1)].item() == 0 and torch.all(dscore[min(3, T - 1)] == 0)
    # backward of the indexer for dI kept on the sampled rows
    keep = torch.zeros(T, dtype=torch.bool, device=DEV)
    keep[rows] = True
    dI = torch.where(keep[:, None], dscore, torch.zeros_like(dscore))
    dq, dk, dw = tsa.qsa_indexer_bwd(xd["q_idx"], xd["k_idx"], xd["w"], cu, sel, dI, score_scale=scale)
    torch.cuda.synchronize()
    dI_h = dI.cpu().double().numpy()
    dq_r, dk_r, dw_r = O.indexer_bwd(x["q_idx"], x["k_idx"], x["w"], cu, idx[:, None, :], dI_h[:, None, :],
                                     score_scale=scale, rows=rows)
    check_grad(dq.cpu()[rows], dq_r, "dq_I")
    check_grad(dk, dk_r, "dk_I")
    check_grad(dw.cpu()[rows][:, None, :], dw_r[:, None, :], "dw")
    others = torch.ones(T, dtype=torch.bool)
    others[rows] = False
    assert torch.all(dq.cpu()[others] == 0) and torch.all(dw.cpu()[others] == 0)


def test_indexer_backward_replays_dq_dw(tsa):
    """dq_I and dw have no atomics: a second call is bit-identical."""
    cu = [0, 900]
    x = {k: v.to(DEV) for k, v in synth.indexer_inputs(900, 64, 128, seed=3).items()}
    sel = tsa.qsa_topk(x["q_idx"], x["k_idx"], x["w"], cu, 256)[:, 0, :].contiguous()
    g = torch.Generator(device=DEV).manual_seed(1)
    dI = torch.randn((900, 256), generator=g, device=DEV)
    a = tsa.qsa_indexer_bwd(x["q_idx"], x["k_idx"], x["w"], cu, sel, dI)
    b = tsa.qsa_indexer_bwd(x["q_idx"], x["k_idx"], x["w"], cu, sel, dI)
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0]) and torch.equal(a[2], b[2])
    assert rel_l2(a[1], b[1]) <= 1e-3


def test_indexer_kl_index_range_flag(tsa):
    """An index beyond its sequence is treated as -1 (no gradient) and raises
    FLAG_INDEX_RANGE."""
    cu = [0, 200, 500]
    x = {k: v.to(DEV) for k, v in synth.indexer_inputs(500, 64, 128, seed=9).items()}
    sel = tsa.qsa_topk(x["q_idx"], x["k_idx"], x["w"], cu, 128)[:, 0, :].contiguous()
    teacher = torch.zeros((500, 128), device=DEV)
    teacher[:, 0] = 1.0
    bad = sel.clone()
    bad[300, 5] = 400                         # sequence 1 holds local positions 0..299
    fixed = bad.clone()
    fixed[300, 5] = -1
    tsa.read_flags(clear=True)
    l1, g1 = tsa.qsa_indexer_kl(x["q_idx"], x["k_idx"], x["w"], cu, fixed, teacher)
    assert tsa.read_flags() == 0
    l2, g2 = tsa.qsa_indexer_kl(x["q_idx"], x["k_idx"], x["w"], cu, bad, teacher)
    assert tsa.read_flags() & tsa.FLAG_INDEX_RANGE
    assert torch.equal(l1, l2) and torch.equal(g1, g2)


@pytest.mark.slow
def test_indexer_train_t65536_sampled(tsa):
    """T=65536, 64 indexer heads, d_I=128, top-2048 (the bench's workload): KL
    and backward on sampled rows against the oracle."""
    T = 65536
    cu = [0, T]
    x = synth.indexer_inputs(T, 64, 128, seed=5, device=DEV)
    sel = tsa.qsa_topk(x["q_idx"], x["k_idx"], x["w"], cu, 2048)[:, 0, :].contiguous()
    rows = [0, 1, 2047, 2048, 40000, 65535]
    idx = sel.cpu()
    xc = {k: v.cpu() for k, v in x.items()}
    m = synth.mla_inputs(T, 2, 64, seed=6)
    tea = torch.zeros((T, 2048), dtype=torch.float32)
    tea[rows] = torch.from_numpy(O.mla_teacher(m["q"], m["kv"], idx, cu, 0.125, rows=rows)).float()
    loss, dscore = tsa.qsa_indexer_kl(x["q_idx"], x["k_idx"], x["w"], cu, sel, tea.to(DEV))
    keep = torch.zeros(T, dtype=torch.bool, device=DEV)
    keep[rows] = True
    dI = torch.where(keep[:, None], dscore, torch.zeros_like(dscore))
    dq, dk, dw = tsa.qsa_indexer_bwd(x["q_idx"], x["k_idx"], x["w"], cu, sel, dI)
    torch.cuda.synchronize()
    sc_ref = O.indexer_scores_at(xc["q_idx"], xc["k_idx"], xc["w"], cu, idx[:, None, :], rows=rows)[:, 0, :]
    loss_ref, g_ref = O.sparse_kl(sc_ref, tea[rows].double().numpy())
    check_rows(dscore.cpu().double().numpy()[rows], g_ref, TOL_OUT, "dI rows")
    assert np.max(np.abs(loss.cpu().double().numpy()[rows] - loss_ref)) <= TOL_OUT * max(1.0, loss_ref.max())
    dq_r, dk_r, dw_r = O.indexer_bwd(xc["q_idx"], xc["k_idx"], xc["w"], cu, idx[:, None, :],
                                     dI.cpu().double().numpy()[:, None, :], rows=rows)
    check_grad(dq.cpu()[rows], dq_r, "dq_I")
    check_grad(dk, dk_r, "dk_I")
    check_grad(dw.cpu()[rows][:, None, :], dw_r[:, None, :], "dw")
