"""Pins for the CPU oracle: each check compares it with something other than
itself -- hand-derived golden rows, closed forms, textbook dense attention,
brute force on tiny inputs, invariants the pages state (exact paddings,
all-invalid rows) and central finite differences.  CPU only."""
import json
import math
import os

import numpy as np
import pytest
import torch
from scipy.special import softmax as sp_softmax, logsumexp

import oracle as O
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _num(x):
    if isinstance(x, str):
        return float(x)  # "-inf", "-0.0"
    return float(x)


def _arr(nested):
    return np.vectorize(_num, otypes=[np.float64])(np.array(nested, dtype=object))


# ---------------------------------------------------------------- indexer

def test_indexer_golden_hand_derived():
    g = json.load(open(os.path.join(GOLDEN, "indexer_small.json")))
    q, k, w, cu = np.array(g["q_idx"], float), np.array(g["k_idx"], float), np.array(g["w"]), g["cu_seqlens"]
    s1 = O.indexer_token_scores(q, k, w, cu, range(3), groups=1)
    np.testing.assert_array_equal(s1[:, 0, :], _arr(g["scores_groups1"]).astype(np.float32))
    s2 = O.indexer_token_scores(q, k, w, cu, range(3), groups=2)
    np.testing.assert_array_equal(s2, _arr(g["scores_groups2"]).astype(np.float32))
    b = O.indexer_block_scores(q, k, w, cu, range(3), block_size=2, groups=1)
    np.testing.assert_array_equal(b[:, 0, :], _arr(g["block2_groups1"]).astype(np.float32))
    top = O.qsa_topk(q, k, w, cu, range(3), topk=2)
    np.testing.assert_array_equal(top[:, 0, :], np.array(g["top2_groups1"]))


def test_indexer_one_hot_closed_form():
    # q_I[t,h] = e_{j(t,h)}  =>  q.k_I[s] = k_I[s, j(t,h)]  (no dot product needed)
    rng = np.random.default_rng(0)
    T, H, d = 9, 3, 5
    j = rng.integers(0, d, size=(T, H))
    q = np.zeros((T, H, d))
    q[np.arange(T)[:, None], np.arange(H)[None, :], j] = 1.0
    k = rng.integers(-4, 5, size=(T, d)).astype(float)
    w = rng.integers(0, 8, size=(T, H)) / 8.0
    cu = [0, 4, 9]
    got = O.indexer_token_scores(q, k, w, cu, range(T), groups=1, score_scale=2.0)
    for t in range(T):
        s0, n = O.seq_bounds(cu, t)
        for s in range(n):
            if s > t - s0:
                assert got[t, 0, s] == -np.inf
            else:
                want = 2.0 * sum(w[t, h] * max(k[s0 + s, j[t, h]], 0.0) for h in range(H))
                assert got[t, 0, s] == np.float32(want)


def test_indexer_groups_sum_to_shared_score():
    x = synth.indexer_inputs(40, 8, 16, seed=3, integer=True)
    cu = [0, 17, 40]
    g4 = O.indexer_token_scores(x["q_idx"], x["k_idx"], x["w"], cu, range(40), groups=4)
    g1 = O.indexer_token_scores(x["q_idx"], x["k_idx"], x["w"], cu, range(40), groups=1)
    fin = np.isfinite(g1[:, 0])
    # dyadic/integer inputs: every partial sum is exact in fp32, so the sum is exact
    np.testing.assert_array_equal(g4.sum(axis=1)[fin], g1[:, 0][fin])
    assert np.all(np.isinf(g4.sum(axis=1)[~fin]))


def test_indexer_causal_self_included_and_sequence_local():
    x = synth.indexer_inputs(12, 2, 8, seed=4)
    cu = [0, 5, 12]
    s = O.indexer_token_scores(x["q_idx"], x["k_idx"], x["w"], cu, range(12))
    for t in range(12):
        s0, n = O.seq_bounds(cu, t)
        p = t - s0
        assert np.all(np.isfinite(s[t, 0, :p + 1]))
        assert np.all(s[t, 0, p + 1:] == -np.inf)
    # row 5 is the first token of sequence 2: exactly one candidate (itself)
    assert np.isfinite(s[5, 0, 0]) and np.all(s[5, 0, 1:] == -np.inf)


def test_block_scores_brute_force():
    x = synth.indexer_inputs(23, 4, 8, seed=5)
    cu = [0, 9, 23]
    bs = 4
    tok = O.indexer_token_scores(x["q_idx"], x["k_idx"], x["w"], cu, range(23), groups=2)
    blk = O.indexer_block_scores(x["q_idx"], x["k_idx"], x["w"], cu, range(23), bs, groups=2)
    for t in range(23):
        s0, n = O.seq_bounds(cu, t)
        p = t - s0
        for g in range(2):
            for b in range(blk.shape[2]):
                vals = [tok[t, g, s] for s in range(n) if s // bs == b and s <= p]
                want = max(vals) if vals else -np.inf
                assert blk[t, g, b] == np.float32(want)


# ---------------------------------------------------------------- top-k

def test_topk_golden_ties():
    g = json.load(open(os.path.join(GOLDEN, "topk_ties.json")))
    for c in g["cases"]:
        row = np.array([_num(v) for v in c["scores"]], dtype=np.float32)
        np.testing.assert_array_equal(O.topk_lex(row, c["k"]), np.array(c["expect"]))


def _brute_topk(row, k):
    # independent formulation: Python's sorted() with a tuple key
    cands = [(float(v), i) for i, v in enumerate(row) if v != -np.inf]
    cands.sort(key=lambda p: (-p[0], p[1]))
    out = [i for _, i in cands[:k]]
    return out + [-1] * (k - len(out))


def test_topk_brute_force_tie_heavy():
    s = synth.tie_stress_scores(64, 50, seed=6).numpy()
    for r in s:
        for k in (1, 7, 50, 64):
            assert O.topk_lex(r, k).tolist() == _brute_topk(r, k)


def test_topk_properties():
    rng = np.random.default_rng(7)
    # all-equal row gives 0..k-1
    np.testing.assert_array_equal(O.topk_lex(np.zeros(100, np.float32), 10), np.arange(10))
    # k >= candidates: every candidate then -1
    row = rng.standard_normal(20).astype(np.float32)
    out = O.topk_lex(row, 32)
    assert sorted(out[:20].tolist()) == list(range(20)) and np.all(out[20:] == -1)
    # permuting equal scores leaves the output unchanged (index-ascending inside ties)
    row = np.array([1, 0, 1, 0, 1, 0, 2], np.float32)
    np.testing.assert_array_equal(O.topk_lex(row, 5), [6, 0, 2, 4, 1])


# ---------------------------------------------------------------- sparse MLA

def _mla(T, H, D, seed, cu=None):
    x = synth.mla_inputs(T, H, D, seed, with_grad_out=True)
    return O.as_f64(x["q"]), O.as_f64(x["kv"]), O.as_f64(x["dout"])


def test_mla_single_key_closed_form():
    q, kv, _ = _mla(6, 3, 576, 10)
    scale = 0.07
    idx = np.full((6, 4), -1)
    j = [0, 1, 0, 2, 4, 3]
    idx[np.arange(6), 2] = j                      # one valid slot, not in slot 0
    o, lse = O.sparse_mla_fwd(q, kv, idx, [0, 6], scale)
    for t in range(6):
        np.testing.assert_allclose(o[t], np.broadcast_to(kv[j[t], :512], (3, 512)), rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse[t], scale * (q[t] @ kv[j[t]]), rtol=1e-13)


def test_mla_two_keys_closed_form():
    q, kv, _ = _mla(4, 2, 576, 11)
    scale = 0.05
    idx = np.array([[0, -1], [1, 0], [2, 0], [-1, 3]])
    o, lse = O.sparse_mla_fwd(q, kv, idx, [0, 4], scale)
    t, a, b = 2, 2, 0
    xa, xb = scale * (q[t] @ kv[a]), scale * (q[t] @ kv[b])
    wa = 1.0 / (1.0 + np.exp(xb - xa))
    np.testing.assert_allclose(o[t], wa[:, None] * kv[a, :512] + (1 - wa)[:, None] * kv[b, :512], atol=1e-12)
    np.testing.assert_allclose(lse[t], np.logaddexp(xa, xb), rtol=1e-13)


def test_mla_all_invalid_row():
    q, kv, _ = _mla(5, 2, 576, 12)
    idx = np.array([[0, -1], [-1, -1], [2, 1], [-1, -1], [4, 0]])
    for fn in (O.sparse_mla_fwd, O.sparse_mla_fwd_dense):
        o, lse = fn(q, kv, idx, [0, 5], 0.1)
        assert np.all(o[1] == 0) and np.all(o[3] == 0)
        assert np.all(lse[1] == -np.inf) and np.all(lse[3] == -np.inf)
        assert np.all(np.isfinite(lse[[0, 2, 4]]))


def _dense_causal_attention(q, kv, cu, scale, d_v):
    # textbook: full [H, n, n] causal-masked softmax per sequence (scipy softmax)
    T, H, _ = q.shape
    o = np.zeros((T, H, d_v))
    lse = np.zeros((T, H))
    for b in range(len(cu) - 1):
        s0, s1 = cu[b], cu[b + 1]
        n = s1 - s0
        logits = scale * np.einsum("thd,sd->hts", q[s0:s1], kv[s0:s1])
        logits = np.where(np.tril(np.ones((n, n), bool))[None], logits, -np.inf)
        o[s0:s1] = np.einsum("hts,sc->thc", sp_softmax(logits, axis=-1), kv[s0:s1, :d_v])
        lse[s0:s1] = logsumexp(logits, axis=-1).T
    return o, lse


@pytest.mark.parametrize("D", [576, 512])
def test_mla_topk_ge_T_is_dense_causal(D):
    cu = [0, 7, 19]
    q, kv, _ = _mla(19, 4, D, 13)
    T = 19
    rng = np.random.default_rng(1)
    idx = np.full((T, 16), -1)
    for t in range(T):
        s0, _ = O.seq_bounds(cu, t)
        p = t - s0
        idx[t, :p + 1] = rng.permutation(p + 1)   # every causal key, shuffled slots
    o, lse = O.sparse_mla_fwd(q, kv, idx, cu, 0.04)
    od, lsed = O.sparse_mla_fwd_dense(q, kv, idx, cu, 0.04)
    ot, lset = _dense_causal_attention(q, kv, cu, 0.04, 512)
    np.testing.assert_allclose(o, ot, atol=1e-12)
    np.testing.assert_allclose(lse, lset, rtol=1e-12)
    np.testing.assert_allclose(od, ot, atol=1e-12)
    np.testing.assert_allclose(lsed, lset, rtol=1e-12)


def test_mla_thd_equals_separate_sequences():
    cu = [0, 6, 10, 17]
    q, kv, dO = _mla(17, 2, 576, 14)
    idx = synth.random_topk_indices(cu, 5, seed=2).numpy()
    o, lse = O.sparse_mla_fwd(q, kv, idx, cu, 0.05)
    dq, dkv = O.sparse_mla_bwd(q, kv, idx, cu, 0.05, dO)
    for b in range(3):
        s0, s1 = cu[b], cu[b + 1]
        ob, lb = O.sparse_mla_fwd(q[s0:s1], kv[s0:s1], idx[s0:s1], [0, s1 - s0], 0.05)
        np.testing.assert_array_equal(o[s0:s1], ob)
        np.testing.assert_array_equal(lse[s0:s1], lb)
        dqb, dkvb = O.sparse_mla_bwd(q[s0:s1], kv[s0:s1], idx[s0:s1], [0, s1 - s0], 0.05, dO[s0:s1])
        np.testing.assert_allclose(dq[s0:s1], dqb, atol=1e-13)
        np.testing.assert_allclose(dkv[s0:s1], dkvb, atol=1e-13)


def test_mla_nope_zero_pad_and_topk_pad_are_exact():
    cu = [0, 12]
    q, kv, dO = _mla(12, 3, 512, 15)
    idx = synth.random_topk_indices(cu, 5, seed=3).numpy()
    o, lse = O.sparse_mla_fwd(q, kv, idx, cu, 0.1)
    op, lsep = O.sparse_mla_fwd(O.pad_nope(q), O.pad_nope(kv), O.pad_topk(idx), cu, 0.1)
    assert O.pad_topk(idx).shape[1] == 64
    np.testing.assert_array_equal(o, op)
    np.testing.assert_array_equal(lse, lsep)
    dq, dkv = O.sparse_mla_bwd(q, kv, idx, cu, 0.1, dO)
    dqp, dkvp = O.sparse_mla_bwd(O.pad_nope(q), O.pad_nope(kv), O.pad_topk(idx), cu, 0.1, dO)
    np.testing.assert_allclose(dqp[..., :512], dq, atol=1e-13)
    np.testing.assert_allclose(dkvp[..., :512], dkv, atol=1e-13)


def _fd_check(loss, x, grad, n_probe=40, eps=1e-6, seed=0):
    rng = np.random.default_rng(seed)
    flat = x.reshape(-1)
    g = grad.reshape(-1)
    for i in rng.choice(flat.size, size=min(n_probe, flat.size), replace=False):
        old = flat[i]
        flat[i] = old + eps
        lp = loss()
        flat[i] = old - eps
        lm = loss()
        flat[i] = old
        fd = (lp - lm) / (2 * eps)
        assert abs(fd - g[i]) <= 1e-6 * max(1.0, abs(fd)), (i, fd, g[i])


def test_mla_backward_finite_differences():
    cu = [0, 5, 9]
    rng = np.random.default_rng(16)
    T, H, D, dv = 9, 2, 12, 8
    q, kv, dO = rng.standard_normal((T, H, D)), rng.standard_normal((T, D)), rng.standard_normal((T, H, dv))
    idx = synth.random_topk_indices(cu, 3, seed=4).numpy()
    idx[4] = -1
    scale = 0.3

    def loss():
        o, _ = O.sparse_mla_fwd(q, kv, idx, cu, scale, d_v=dv)
        return float((o * dO).sum())

    dq, dkv = O.sparse_mla_bwd(q, kv, idx, cu, scale, dO, d_v=dv)
    _fd_check(loss, q, dq, seed=1)
    _fd_check(loss, kv, dkv, seed=2)
    assert np.all(dq[4] == 0)


def test_mla_backward_single_key_value_path():
    # one valid key: o = v, so dS = 0, dQ = 0 and dKV[:, :512] gets sum_h dO
    q, kv, dO = _mla(4, 3, 576, 17)
    idx = np.array([[0, -1], [-1, 1], [-1, -1], [2, -1]])
    dq, dkv = O.sparse_mla_bwd(q, kv, idx, [0, 4], 0.2, dO)
    np.testing.assert_allclose(dq, 0, atol=1e-12)
    np.testing.assert_allclose(dkv[[0, 1, 2], :512], dO[[0, 1, 3]].sum(axis=1), atol=1e-12)
    np.testing.assert_allclose(dkv[:, 512:], 0, atol=1e-12)
    assert np.all(dkv[3] == 0)


def test_mla_delta_matches_p_dot_dp():
    cu = [0, 10]
    q, kv, dO = _mla(10, 2, 576, 18)
    idx = synth.random_topk_indices(cu, 4, seed=5).numpy()
    o, lse = O.sparse_mla_fwd(q, kv, idx, cu, 0.05)
    dlt = O.mla_bwd_delta(o, dO)
    for t in range(10):
        sel = idx[t][idx[t] >= 0]
        K = kv[sel]
        P = np.exp(0.05 * q[t] @ K.T - lse[t][:, None])
        np.testing.assert_allclose(dlt[t], ((dO[t] @ K[:, :512].T) * P).sum(axis=1), rtol=1e-10, atol=1e-10)


# ---------------------------------------------------------------- sparse GQA

def _dense_causal_gqa(q, k, v, cu, scale):
    T, Hq, d = q.shape
    G = Hq // k.shape[1]
    kk, vv = np.repeat(k, G, axis=1), np.repeat(v, G, axis=1)   # textbook GQA head expansion
    o = np.zeros_like(q)
    for b in range(len(cu) - 1):
        s0, s1 = cu[b], cu[b + 1]
        n = s1 - s0
        logits = scale * np.einsum("thd,shd->hts", q[s0:s1], kk[s0:s1])
        logits = np.where(np.tril(np.ones((n, n), bool))[None], logits, -np.inf)
        o[s0:s1] = np.einsum("hts,shd->thd", sp_softmax(logits, axis=-1), vv[s0:s1])
    return o


def test_gqa_block1_all_selected_is_dense_causal():
    cu = [0, 6, 15]
    x = synth.gqa_inputs(15, 4, 2, 8, seed=20)
    q, k, v = (O.as_f64(x[n]) for n in ("q", "k", "v"))
    idx = np.full((15, 2, 16), -1)
    for t in range(15):
        s0, _ = O.seq_bounds(cu, t)
        p = t - s0
        idx[t, :, :p + 1] = np.arange(p + 1)[::-1]
    o, lse = O.sparse_gqa_fwd(q, k, v, idx, cu, 1, 0.2)
    np.testing.assert_allclose(o, _dense_causal_gqa(q, k, v, cu, 0.2), atol=1e-12)


def test_gqa_block_causal_inside_own_block():
    # block size 4, query at local position 5 selecting block 1 sees tokens 4, 5 only
    x = synth.gqa_inputs(8, 2, 1, 4, seed=21)
    q, k, v = (O.as_f64(x[n]) for n in ("q", "k", "v"))
    idx = np.full((8, 1, 2), -1)
    idx[5, 0, 0] = 1
    o, lse = O.sparse_gqa_fwd(q, k, v, idx, [0, 8], 4, 0.5)
    S = 0.5 * q[5] @ k[[4, 5], 0].T
    np.testing.assert_allclose(o[5], sp_softmax(S, axis=1) @ v[[4, 5], 0], atol=1e-12)
    np.testing.assert_allclose(lse[5], logsumexp(S, axis=1), rtol=1e-13)
    assert np.all(lse[[0, 1, 2, 3, 4, 6, 7]] == -np.inf)


def test_gqa_backward_finite_differences():
    cu = [0, 7, 13]
    rng = np.random.default_rng(22)
    T, Hq, Hkv, d = 13, 4, 2, 6
    q, k, v, dO = (rng.standard_normal(s) for s in [(T, Hq, d), (T, Hkv, d), (T, Hkv, d), (T, Hq, d)])
    idx = synth.random_block_indices(cu, Hkv, 2, 2, seed=6).numpy()
    scale = 0.4

    def loss():
        o, _ = O.sparse_gqa_fwd(q, k, v, idx, cu, 2, scale)
        return float((o * dO).sum())

    dq, dk, dv = O.sparse_gqa_bwd(q, k, v, idx, cu, 2, scale, dO)
    _fd_check(loss, q, dq, seed=3)
    _fd_check(loss, k, dk, seed=4)
    _fd_check(loss, v, dv, seed=5)


def test_synth_is_seeded():
    a = synth.mla_inputs(8, 2, 576, seed=1)
    b = synth.mla_inputs(8, 2, 576, seed=1)
    assert torch.equal(a["q"], b["q"]) and torch.equal(a["kv"], b["kv"])


# ---------------------------------------------------------------- indexer training (sparse KL, indexer backward)

def test_sparse_kl_closed_form():
    # student softmax(0, ln 3) = (1/4, 3/4) against teacher (1/2, 1/2):
    # KL = 1/2 ln(2) + 1/2 ln(2/3) = 1/2 ln(4/3); gradient p - a = (-1/4, 1/4)
    loss, grad = O.sparse_kl([[0.0, math.log(3.0)]], [[0.5, 0.5]])
    assert loss[0] == pytest.approx(0.5 * math.log(4.0 / 3.0), rel=1e-14)
    np.testing.assert_allclose(grad[0], [-0.25, 0.25], atol=1e-15)
    # a -inf slot (not a candidate) takes no part; a row without candidates gives 0
    loss, grad = O.sparse_kl([[0.0, -np.inf, math.log(3.0)], [-np.inf] * 3], [[0.5, 0.0, 0.5], [0.0] * 3])
    assert loss[0] == pytest.approx(0.5 * math.log(4.0 / 3.0), rel=1e-14) and loss[1] == 0.0
    np.testing.assert_allclose(grad, [[-0.25, 0.0, 0.25], [0.0, 0.0, 0.0]], atol=1e-15)


def test_sparse_kl_properties():
    rng = np.random.default_rng(30)
    S = rng.standard_normal((6, 9)) * 3
    S[2, 4:] = -np.inf
    A = rng.random((6, 9)) ** 3
    A[~np.isfinite(S)] = 0.0
    A /= A.sum(axis=1, keepdims=True)
    loss, grad = O.sparse_kl(S, A)
    assert np.all(loss >= 0)                                        # Gibbs' inequality
    np.testing.assert_allclose(grad.sum(axis=1), 0.0, atol=1e-12)   # both sides are distributions
    l2, g2 = O.sparse_kl(S + 7.25, A)                               # a softmax ignores a shift
    np.testing.assert_allclose(l2, loss, rtol=1e-12)
    np.testing.assert_allclose(g2, grad, atol=1e-13)
    # a teacher equal to the student's own softmax costs nothing
    P = np.zeros_like(S)
    for r in range(S.shape[0]):
        ok = np.isfinite(S[r])
        P[r, ok] = sp_softmax(S[r, ok])
    l0, g0 = O.sparse_kl(S, P)
    np.testing.assert_allclose(l0, 0.0, atol=1e-12)
    np.testing.assert_allclose(g0, 0.0, atol=1e-12)


def test_sparse_kl_gradient_finite_differences():
    rng = np.random.default_rng(31)
    S = rng.standard_normal((3, 7))
    S[1, 5:] = -np.inf
    A = rng.random((3, 7))
    A[~np.isfinite(S)] = 0.0
    A /= A.sum(axis=1, keepdims=True)
    _, grad = O.sparse_kl(S, A)
    fin = np.isfinite(S)
    x = np.where(fin, S, 0.0)

    def loss():
        return float(O.sparse_kl(np.where(fin, x, -np.inf), A)[0].sum())

    _fd_check(loss, x, np.where(fin, grad, 0.0), n_probe=21)


def test_mla_teacher_single_head_is_the_attention_row():
    # H = 1: the teacher is the attention probability exp(scale q.k - lse), with lse
    # from the dense-masked forward definition
    cu = [0, 6, 11]
    q, kv, _ = _mla(11, 1, 576, 32)
    idx = synth.random_topk_indices(cu, 4, seed=6, invalid_rows=[7]).numpy()
    scale = 0.06
    _, lse = O.sparse_mla_fwd_dense(q, kv, idx, cu, scale)
    a = O.mla_teacher(q, kv, idx, cu, scale)
    for t in range(11):
        s0, n = O.seq_bounds(cu, t)
        for j, s in enumerate(idx[t]):
            want = 0.0 if s < 0 else math.exp(scale * float(q[t, 0] @ kv[s0 + s]) - lse[t, 0])
            assert a[t, j] == pytest.approx(want, rel=1e-12, abs=1e-300)
    assert np.all(a[7] == 0)
    valid = (idx >= 0).any(axis=1)
    np.testing.assert_allclose(a[valid].sum(axis=1), 1.0, rtol=1e-12)


def test_mla_teacher_two_heads_closed_form():
    # head 0 has q = 0 (uniform over the two slots); head 1 puts sigma(delta) on the
    # second slot with delta = scale q1 . (k1 - k0); the teacher is their average
    rng = np.random.default_rng(33)
    kv = rng.standard_normal((3, 576))
    q = np.zeros((3, 2, 576))
    q[2, 1] = rng.standard_normal(576) * 0.1
    idx = np.array([[0, -1], [1, 0], [0, 1]])
    scale = 0.3
    a = O.mla_teacher(q, kv, idx, [0, 3], scale, rows=[2])
    delta = scale * float(q[2, 1] @ (kv[1] - kv[0]))
    p1 = 1.0 / (1.0 + math.exp(-delta))
    np.testing.assert_allclose(a[0], [0.5 * (0.5 + 1 - p1), 0.5 * (0.5 + p1)], rtol=1e-12)
    np.testing.assert_allclose(O.mla_teacher(q, kv, idx, [0, 3], scale, rows=[0])[0], [1.0, 0.0])


def _indexer_case(seed, T_cu=(0, 5, 9), H_I=4, d_I=6, groups=2, k=3):
    cu = list(T_cu)
    rng = np.random.default_rng(seed)
    T = cu[-1]
    qI = rng.standard_normal((T, H_I, d_I))
    kI = rng.standard_normal((T, d_I))
    w = rng.random((T, H_I)) + 0.1
    idx = np.stack([synth.random_topk_indices(cu, k, seed=seed + g).numpy() for g in range(groups)], axis=1)
    return cu, qI, kI, w, idx


def test_indexer_scores_at_gathers_the_token_scores():
    cu, qI, kI, w, idx = _indexer_case(34)
    S = O.indexer_scores_at(qI, kI, w, cu, idx, groups=2, score_scale=0.5)
    full = O.indexer_token_scores(qI, kI, w, cu, range(cu[-1]), groups=2, score_scale=0.5)
    for t in range(cu[-1]):
        for g in range(2):
            for j, s in enumerate(idx[t, g]):
                if s < 0:
                    assert S[t, g, j] == -np.inf
                else:   # the token scores are the same values rounded once to fp32
                    assert np.float32(S[t, g, j]) == full[t, g, s] or (S[t, g, j] == 0 and full[t, g, s] == 0)


def test_indexer_bwd_one_pair_closed_form():
    q = np.array([[[1.0, 2.0]]])
    k = np.array([[0.5, 0.25]])        # q . k = 1 > 0
    w = np.array([[3.0]])
    idx = np.array([[[0]]])
    dq, dk, dw = O.indexer_bwd(q, k, w, [0, 1], idx, np.array([[[2.0]]]), score_scale=0.5)
    c = 0.5 * 2.0
    np.testing.assert_allclose(dw, [[c * 1.0]])
    np.testing.assert_allclose(dq, [[[c * 3.0 * 0.5, c * 3.0 * 0.25]]])
    np.testing.assert_allclose(dk, [[c * 3.0 * 1.0, c * 3.0 * 2.0]])
    # a negative dot is cut by the ReLU: no gradient anywhere
    dq, dk, dw = O.indexer_bwd(-q, k, w, [0, 1], idx, np.array([[[2.0]]]), score_scale=0.5)
    assert not dq.any() and not dk.any() and not dw.any()


def test_indexer_bwd_finite_differences():
    cu, qI, kI, w, idx = _indexer_case(35)
    rng = np.random.default_rng(36)
    G = rng.standard_normal(idx.shape)
    valid = idx >= 0
    # away from the ReLU kink, so that central differences see one branch
    for t in range(cu[-1]):
        s0, _ = O.seq_bounds(cu, t)
        for g in range(2):
            for s in idx[t, g][idx[t, g] >= 0]:
                assert np.all(np.abs(qI[t, 2 * g:2 * g + 2] @ kI[s0 + s]) > 1e-4)

    def loss():
        S = O.indexer_scores_at(qI, kI, w, cu, idx, groups=2, score_scale=0.7)
        return float((G * np.where(valid, S, 0.0)).sum())

    dq, dk, dw = O.indexer_bwd(qI, kI, w, cu, idx, G, groups=2, score_scale=0.7)
    _fd_check(loss, qI, dq, seed=3)
    _fd_check(loss, kI, dk, seed=4)
    _fd_check(loss, w, dw, seed=5)


def test_indexer_kl_chain_finite_differences():
    """The sparse KL of the indexer against a fixed teacher, differentiated
    through the indexer backward, matches central differences of the loss."""
    cu, qI, kI, w, idx = _indexer_case(37, groups=1, k=4)
    rng = np.random.default_rng(38)
    A = rng.random(idx.shape)
    A[idx < 0] = 0.0
    A /= np.maximum(A.sum(axis=2, keepdims=True), 1e-300)

    def loss():
        S = O.indexer_scores_at(qI, kI, w, cu, idx, groups=1, score_scale=0.4)
        return float(O.sparse_kl(S[:, 0], A[:, 0])[0].sum())

    S = O.indexer_scores_at(qI, kI, w, cu, idx, groups=1, score_scale=0.4)
    _, gS = O.sparse_kl(S[:, 0], A[:, 0])
    dq, dk, dw = O.indexer_bwd(qI, kI, w, cu, idx, gS[:, None, :], groups=1, score_scale=0.4)
    _fd_check(loss, qI, dq, seed=6)
    _fd_check(loss, kI, dk, seed=7)
    _fd_check(loss, w, dw, seed=8)
