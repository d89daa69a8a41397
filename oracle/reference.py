"""Plain, slow CPU oracle for the trainable sparse-attention hot path.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import, call or
execute this module: only the tests, the package's ``smoke()`` check and the
bench's CPU-baseline / reference arm use it.  It shares no code with the CUDA
library (no kernels, headers, tables or helpers); both sides are fed from the
seeded generators in ``synth``.

Everything is computed in float64 from the exact values of the bf16 inputs.
The one place where floating point decides an integer (which keys the top-k
selects) is taken in fp32, the precision the kernels decide in: each indexer
score is computed in fp64 and rounded to fp32 once.

Sources (web pages, cited by title and section):
  [QSA]  Megatron-LM issue #7060 "Add trainable QSA sparse attention with a
         TileLang backend" -- indexer, exact block top-k with a lexicographic
         (score, block_id) key, Sparse-GQA, bounded-memory streaming, BSHD/THD.
  [DSA]  Megatron-LM PR #3674 "Enable DSA CP/absorbed/THD paths with TileLang
         fused ops" -- absorbed MLA, sparse MLA fwd/bwd kernels, indexer kernels,
         logits cleaning, packed THD masking.
  [NOPE] Megatron-LM PR #7617 "Support NoPE shapes and unaligned top-k in
         TileLang sparse MLA" -- q [T,H,576], kv latent with values in the first
         512 channels, -1 invalid sentinel, explicit softmax scale, the dense
         [b, heads, sq, sk] masked-softmax fallback, all-invalid rows.

Readings where the pages are silent (each is also listed in the design notes):
  * indexer score = score_scale * sum_h w[t,h] * ReLU(q_I[t,h] . k_I[s]); the
    candidate keys of query t are s <= t inside t's sequence (self included);
  * indexer heads are split into ``groups`` contiguous sets (one per kv group);
  * a block's score is the max over its causal tokens; future blocks are not
    candidates; masked entries are never selected, even when fewer than k;
  * -0.0 equals +0.0; rows come out sorted by (score desc, index asc), -1 last;
  * indices are positions local to their sequence;
  * LSE is the natural log; an all-invalid row gives o = 0 and lse = -inf;
  * sparse MLA does not re-mask the indices it is given (no causal test);
    sparse GQA keeps only tokens s <= t of the selected blocks;
  * the indexer's sparse KL: teacher = the attention probabilities averaged
    over heads on the selected slots, student = softmax of the indexer scores
    on the same slots, loss = KL(teacher || student) per query row.

Parity pins: every function here is checked in ``tests/test_oracle_pins.py``
against closed forms, textbook dense attention, brute force, hand-derived
golden rows and finite differences.
"""
from __future__ import annotations

import math
from typing import Iterable, List, Optional, Sequence

import numpy as np

NEG_INF = -math.inf


# --------------------------------------------------------------------------
# small helpers (shapes and sequence bookkeeping only)
# --------------------------------------------------------------------------

def as_f64(x) -> np.ndarray:
    """Widen an array-like (numpy, or a CPU torch tensor of any float dtype) to fp64 exactly."""
    if hasattr(x, "detach"):
        import torch  # local import: only for tensor inputs
        x = x.detach().to("cpu", torch.float64).numpy()
    return np.asarray(x, dtype=np.float64)


def as_i64(x) -> np.ndarray:
    if hasattr(x, "detach"):
        x = x.detach().cpu().numpy()
    return np.asarray(x, dtype=np.int64)


def seq_bounds(cu_seqlens: Sequence[int], t: int):
    """(start, length) of the sequence that holds packed token row t."""
    cu = list(cu_seqlens)
    for b in range(len(cu) - 1):
        if cu[b] <= t < cu[b + 1]:
            return cu[b], cu[b + 1] - cu[b]
    raise IndexError(f"token {t} outside cu_seqlens {cu}")


def max_seqlen(cu_seqlens: Sequence[int]) -> int:
    cu = list(cu_seqlens)
    return max(cu[b + 1] - cu[b] for b in range(len(cu) - 1))


# --------------------------------------------------------------------------
# indexer score  ([QSA] "Describe the solution": trainable indexer, ReLU scores;
# [DSA] "Changes": fused indexer forward + logits cleaning)
# --------------------------------------------------------------------------

def indexer_token_scores(q_idx, k_idx, w, cu_seqlens, rows: Iterable[int], groups: int = 1,
                         score_scale: float = 1.0, width: Optional[int] = None) -> np.ndarray:
    """Token-level indexer scores for the query rows ``rows``.

    I_g[t, s] = score_scale * sum_{h in group g} w[t,h] * max(q_I[t,h,:] . k_I[s,:], 0)
    for local key positions s <= p(t) of t's sequence, computed in fp64 and
    rounded once to fp32; every other column is -inf (a "cleaned" logit that can
    never be selected).  -0.0 is canonicalised to +0.0.

    Returns float32 [len(rows), groups, width], width defaulting to the longest
    sequence.
    """
    kI = as_f64(k_idx)
    H_I = q_idx.shape[1]
    if H_I % groups:
        raise ValueError("H_I must be a multiple of groups")
    hg = H_I // groups
    rows = list(rows)
    width = max_seqlen(cu_seqlens) if width is None else width
    out = np.full((len(rows), groups, width), -np.inf, dtype=np.float32)
    for i, t in enumerate(rows):
        s0, n = seq_bounds(cu_seqlens, t)
        p = t - s0
        dots = as_f64(q_idx[t]) @ kI[s0:s0 + p + 1].T      # [H_I, p+1]
        relu = np.maximum(dots, 0.0)
        w_t = as_f64(w[t])
        for g in range(groups):
            hs = slice(g * hg, (g + 1) * hg)
            acc = w_t[hs] @ relu[hs]                           # [p+1], fp64
            sc = (score_scale * acc).astype(np.float32)
            sc[sc == 0] = np.float32(0.0)                      # -0.0 -> +0.0
            out[i, g, :p + 1] = sc
    return out


def indexer_block_scores(q_idx, k_idx, w, cu_seqlens, rows: Iterable[int], block_size: int,
                         groups: int = 1, score_scale: float = 1.0,
                         width: Optional[int] = None) -> np.ndarray:
    """Block-level scores ([QSA] "Describe the solution": exact block top-k over a
    [sequence, sequence/block_size] score matrix).

    B_g[t, b] = max over local tokens s in block b with s <= p(t) of I_g[t, s]
    (the fp32 token scores above).  Blocks that start after p(t) are -inf.
    """
    Lmax = max_seqlen(cu_seqlens)
    nblk = -(-Lmax // block_size) if width is None else width
    tok = indexer_token_scores(q_idx, k_idx, w, cu_seqlens, rows, groups, score_scale, Lmax)
    out = np.full((tok.shape[0], groups, nblk), -np.inf, dtype=np.float32)
    for i, t in enumerate(rows):
        s0, _ = seq_bounds(cu_seqlens, t)
        p = t - s0
        for b in range(p // block_size + 1):
            lo, hi = b * block_size, min((b + 1) * block_size, p + 1)
            out[i, :, b] = tok[i, :, lo:hi].max(axis=1)
    return out


# --------------------------------------------------------------------------
# deterministic exact top-k ([QSA] "Describe the solution": lexicographic
# (score, block_id) key; "Additional context": deterministic tie-breaking)
# --------------------------------------------------------------------------

def topk_lex(row, k: int) -> np.ndarray:
    """The k best finite entries of one fp32 row under the total order
    (score descending, index ascending); -inf entries are not candidates.
    Output int32 [k], sorted in that order, -1 after the last candidate."""
    r = np.asarray(row, dtype=np.float32)
    cand = np.nonzero(r != -np.inf)[0]
    vals = r[cand]
    order = np.lexsort((cand, -vals))        # primary: -score ascending; then index ascending
    sel = cand[order[:k]]
    out = np.full(k, -1, dtype=np.int32)
    out[:sel.size] = sel
    return out


def topk_rows(scores, k: int) -> np.ndarray:
    """topk_lex applied to every row of a [..., L] fp32 array."""
    s = np.asarray(scores, dtype=np.float32)
    flat = s.reshape(-1, s.shape[-1])
    out = np.stack([topk_lex(r, k) for r in flat]) if flat.shape[0] else np.zeros((0, k), np.int32)
    return out.reshape(s.shape[:-1] + (k,))


def qsa_topk(q_idx, k_idx, w, cu_seqlens, rows: Iterable[int], topk: int, groups: int = 1,
             block_size: int = 1, score_scale: float = 1.0) -> np.ndarray:
    """Indexer then top-k, per query row: int32 [len(rows), groups, topk]."""
    rows = list(rows)
    if block_size == 1:
        sc = indexer_token_scores(q_idx, k_idx, w, cu_seqlens, rows, groups, score_scale)
    else:
        sc = indexer_block_scores(q_idx, k_idx, w, cu_seqlens, rows, block_size, groups, score_scale)
    return topk_rows(sc, topk)


# --------------------------------------------------------------------------
# sparse MLA ([DSA] "Changes": sparse MLA forward/backward over the absorbed
# latent; [NOPE] "What does this PR do?" and the backport's "Why"/"Change":
# q [T,H,576], kv latent, value = key[..., :512], -1 slots masked)
# --------------------------------------------------------------------------

def _valid_rows(idx_row: np.ndarray, n: int) -> np.ndarray:
    sel = idx_row[idx_row >= 0]
    if sel.size and sel.max() >= n:
        raise IndexError("index beyond its sequence")
    return sel


def sparse_mla_fwd_dense(q, kv, idx, cu_seqlens, scale: float, d_v: int = 512):
    """Dense-masked definition (the [b, heads, sq, sk] masked softmax fallback of
    [NOPE]): for every (t, h) a logit row over all keys of t's sequence that is
    -inf except at t's selected indices; softmax in fp64; o = P @ kv[:, :d_v];
    lse = log(sum exp) (natural log).  All-invalid rows give o = 0, lse = -inf.
    Returns (o [T,H,d_v], lse [T,H]) in float64."""
    Q, KV, I = as_f64(q), as_f64(kv), as_i64(idx)
    T, H, _ = Q.shape
    o = np.zeros((T, H, d_v))
    lse = np.full((T, H), -np.inf)
    for t in range(T):
        s0, n = seq_bounds(cu_seqlens, t)
        sel = _valid_rows(I[t], n)
        if sel.size == 0:
            continue
        mask = np.zeros(n, dtype=bool)
        mask[sel] = True
        logits = np.full((H, n), -np.inf)
        full = scale * (Q[t] @ KV[s0:s0 + n].T)
        logits[:, mask] = full[:, mask]
        m = logits.max(axis=1, keepdims=True)
        e = np.exp(logits - m)
        l = e.sum(axis=1, keepdims=True)
        o[t] = (e / l) @ KV[s0:s0 + n, :d_v]
        lse[t] = (m + np.log(l))[:, 0]
    return o, lse


def sparse_mla_row(q_t, kv, idx_t, s0: int, n: int, scale: float, d_v: int = 512):
    """One query row of the gather form: softmax over the valid slots of idx_t
    (slot order as given) of scale * q_t . kv[s0 + idx]; returns (o [H, d_v], lse [H])."""
    Qt, I = as_f64(q_t), as_i64(idx_t)
    H = Qt.shape[0]
    sel = _valid_rows(I, n)
    if sel.size == 0:
        return np.zeros((H, d_v)), np.full(H, -np.inf)
    K = as_f64(kv[s0 + sel]) if not isinstance(kv, np.ndarray) else kv[s0 + sel]   # [nk, D]
    S = scale * (Qt @ K.T)                                 # [H, nk]
    m = S.max(axis=1, keepdims=True)
    e = np.exp(S - m)
    l = e.sum(axis=1, keepdims=True)
    return (e / l) @ K[:, :d_v], (m + np.log(l))[:, 0]


def sparse_mla_fwd(q, kv, idx, cu_seqlens, scale: float, d_v: int = 512,
                   rows: Optional[Iterable[int]] = None):
    """Gather form of the same forward, equal to the dense-masked form when a
    row holds no duplicate index.  Returns (o [T,H,d_v], lse [T,H]) float64, or
    for ``rows`` the compact (o [len(rows),H,d_v], lse [len(rows),H])."""
    KV = as_f64(kv)
    T, H = q.shape[0], q.shape[1]
    rr = range(T) if rows is None else list(rows)
    o = np.zeros((len(rr), H, d_v))
    lse = np.full((len(rr), H), -np.inf)
    for i, t in enumerate(rr):
        s0, n = seq_bounds(cu_seqlens, t)
        o[i], lse[i] = sparse_mla_row(q[t], KV, idx[t], s0, n, scale, d_v)
    return o, lse


def sparse_mla_bwd(q, kv, idx, cu_seqlens, scale: float, dout, d_v: int = 512,
                   rows: Optional[Iterable[int]] = None):
    """Analytic gradient of the sparse MLA forward, in fp64.

    With P = exp(scale*S - lse), dP = dO . V^T, Dlt = sum_c dO*o,
    dS = P * (dP - Dlt):  dQ = scale * dS . K;
    dKV[idx] += scale * dS^T . Q  (all channels)  +  P^T . dO  (first d_v channels).
    Gradients reaching -1 slots are dropped.  ``rows`` restricts the sum to some
    query rows (exact whenever dO is zero on every other row) and makes dq
    compact [len(rows), H, D].  Returns (dq, dkv [T_kv, D]) float64."""
    KV = as_f64(kv)
    T, H, D = q.shape
    rr = list(range(T)) if rows is None else list(rows)
    dq = np.zeros((len(rr), H, D))
    dkv = np.zeros_like(KV)
    for i, t in enumerate(rr):
        s0, n = seq_bounds(cu_seqlens, t)
        sel = _valid_rows(as_i64(idx[t]), n)
        if sel.size == 0:
            continue
        Qt, dOt = as_f64(q[t]), as_f64(dout[t])
        o_t, lse_t = sparse_mla_row(Qt, KV, idx[t], s0, n, scale, d_v)
        g = s0 + sel
        K = KV[g]
        S = scale * (Qt @ K.T)
        P = np.exp(S - lse_t[:, None])
        dP = dOt @ K[:, :d_v].T
        Dlt = (dOt * o_t).sum(axis=1)
        dS = P * (dP - Dlt[:, None])
        dq[i] = scale * (dS @ K)
        np.add.at(dkv, g, scale * (dS.T @ Qt))
        np.add.at(dkv[:, :d_v], g, P.T @ dOt)
    return dq, dkv


def mla_bwd_delta(o, dout) -> np.ndarray:
    """Dlt[t,h] = sum_c dO[t,h,c] * o[t,h,c] (the backward's preprocess)."""
    return (as_f64(o) * as_f64(dout)).sum(axis=-1)


# --------------------------------------------------------------------------
# indexer training: sparse KL against the attention teacher, and the indexer
# backward ([QSA] "Describe the problem": sparse KL supervision for training
# the indexer; "Describe the solution you'd like": sparse Stage-2 teacher/KL
# loss for indexer training; [DSA] "Changes": sparse-KL streaming for the
# indexer loss; file table: fused indexer backward kernel).  The pages print
# no formula; the reading taken here:
#   teacher a[t, j]  = the sparse attention probabilities of query t averaged
#                      over its heads, on t's selected slots j (a distribution,
#                      since every head's probabilities sum to 1 over them);
#   student p[t, j]  = softmax over the same slots of the indexer scores;
#   loss_t           = KL(a_t || p_t) = sum_j a log(a / p), 0 log 0 = 0;
#   d loss_t / d I   = p - a on the selected slots (the teacher is a target).
# --------------------------------------------------------------------------

def _selected(idx_t: np.ndarray, n: int) -> np.ndarray:
    """Mask of the slots of one index row that name a key of the sequence."""
    return (idx_t >= 0) & (idx_t < n)


def indexer_scores_at(q_idx, k_idx, w, cu_seqlens, idx, groups: int = 1,
                      score_scale: float = 1.0, rows: Optional[Iterable[int]] = None) -> np.ndarray:
    """The indexer score of every selected slot, in fp64 (not rounded to fp32):
    S[t, g, j] = score_scale * sum_{h in g} w[t,h] * max(q_I[t,h] . k_I[s0 + idx[t,g,j]], 0),
    -inf at slots that are -1 or outside t's sequence.  idx: int [T, groups, k].
    ``rows``: only those query rows, compact [len(rows), groups, k].  Row
    inputs (q_I, w, idx) are read one row at a time."""
    K = as_f64(k_idx)
    T, H_I = q_idx.shape[0], q_idx.shape[1]
    hg = H_I // groups
    rr = range(T) if rows is None else list(rows)
    out = np.full((len(rr),) + tuple(idx.shape[1:]), -np.inf)
    for i, t in enumerate(rr):
        s0, n = seq_bounds(cu_seqlens, t)
        Qt, Wt, It = as_f64(q_idx[t]), as_f64(w[t]), as_i64(idx[t])
        for g in range(groups):
            hs = slice(g * hg, (g + 1) * hg)
            for j, s in enumerate(It[g]):
                if 0 <= s < n:
                    dots = Qt[hs] @ K[s0 + s]                 # [hg]
                    out[i, g, j] = score_scale * float(Wt[hs] @ np.maximum(dots, 0.0))
    return out


def mla_teacher(q, kv, idx, cu_seqlens, scale: float, rows: Optional[Iterable[int]] = None) -> np.ndarray:
    """The indexer's teacher on the selected slots of each query row: the sparse
    MLA attention probabilities exp(scale q[t,h] . kv[s] - lse[t,h]) averaged over
    the heads.  0 at -1 slots; all 0 for a row without a valid slot.
    Returns float64 [len(rows), topk].  q and idx are read one row at a time."""
    KV = as_f64(kv)
    T = q.shape[0]
    rr = range(T) if rows is None else list(rows)
    out = np.zeros((len(rr), idx.shape[1]))
    for i, t in enumerate(rr):
        s0, n = seq_bounds(cu_seqlens, t)
        It = as_i64(idx[t])
        ok = _selected(It, n)
        if not ok.any():
            continue
        S = scale * (as_f64(q[t]) @ KV[s0 + It[ok]].T)     # [H, valid slots]
        P = np.exp(S - S.max(axis=1, keepdims=True))
        P /= P.sum(axis=1, keepdims=True)
        out[i, ok] = P.mean(axis=0)
    return out


def sparse_kl(scores, teacher):
    """KL(teacher || softmax(scores)) per row over the slots whose score is
    finite, and its gradient with respect to the scores, softmax(scores) -
    teacher (0 at the other slots).  A row without a finite score gives 0, 0.
    scores, teacher: [R, k]; returns (loss float64 [R], grad float64 [R, k])."""
    S, A = as_f64(scores), as_f64(teacher)
    loss = np.zeros(S.shape[0])
    grad = np.zeros_like(S)
    for r in range(S.shape[0]):
        ok = np.isfinite(S[r])
        if not ok.any():
            continue
        z = S[r, ok]
        log_p = z - z.max() - math.log(np.exp(z - z.max()).sum())
        a = A[r, ok]
        pos = a > 0
        loss[r] = float((a[pos] * (np.log(a[pos]) - log_p[pos])).sum())
        grad[r, ok] = np.exp(log_p) - a
    return loss, grad


def indexer_bwd(q_idx, k_idx, w, cu_seqlens, idx, dscore, groups: int = 1, score_scale: float = 1.0,
                rows: Optional[Iterable[int]] = None):
    """Gradient of sum_{t,g,j} dscore[t,g,j] * I_g[t, s0 + idx[t,g,j]] (the indexer
    score definition above, taken in fp64) with respect to q_I, k_I and w:
      dw[t,h]   = score_scale * sum_j dscore * max(d, 0)
      dq_I[t,h] = score_scale * sum_j dscore * w[t,h] * [d > 0] * k_I[s]
      dk_I[s]   = score_scale * sum_{t,j} dscore * sum_h w[t,h] * [d > 0] * q_I[t,h]
    with d = q_I[t,h] . k_I[s]; slots that are -1 or outside the sequence carry
    no gradient.  ``rows`` restricts the sum to those query rows (exact when
    dscore is zero on every other row) and makes dq_I and dw compact.  Row
    inputs (q_I, w, idx, dscore) are read one row at a time.
    Returns float64 (dq_I [T,H_I,d_I], dk_I [T,d_I], dw [T,H_I])."""
    K = as_f64(k_idx)
    T, H_I, d_I = q_idx.shape
    hg = H_I // groups
    rr = list(range(T)) if rows is None else list(rows)
    dq, dk, dw = np.zeros((len(rr), H_I, d_I)), np.zeros_like(K), np.zeros((len(rr), H_I))
    for i, t in enumerate(rr):
        s0, n = seq_bounds(cu_seqlens, t)
        Qt, Wt, It, Gt = as_f64(q_idx[t]), as_f64(w[t]), as_i64(idx[t]), as_f64(dscore[t])
        for g in range(groups):
            hs = slice(g * hg, (g + 1) * hg)
            for j, s in enumerate(It[g]):
                if not (0 <= s < n) or Gt[g, j] == 0.0:
                    continue
                c = score_scale * Gt[g, j]
                d = Qt[hs] @ K[s0 + s]                       # [hg]
                on = (d > 0).astype(np.float64)
                dw[i, hs] += c * np.maximum(d, 0.0)
                dq[i, hs] += c * (Wt[hs] * on)[:, None] * K[s0 + s][None, :]
                dk[s0 + s] += c * ((Wt[hs] * on) @ Qt[hs])
    return dq, dk, dw


# --------------------------------------------------------------------------
# block Sparse-GQA ([QSA] "Describe the solution": Sparse-GQA forward and
# backward over exact block top-k selections; BSHD and packed THD)
# --------------------------------------------------------------------------

def _gqa_tokens(blk_row: np.ndarray, p: int, n: int, block_size: int) -> np.ndarray:
    """Local token positions attended by a query at local position p: every
    token s <= p inside a selected block (a set; duplicates count once)."""
    sel = blk_row[blk_row >= 0]
    if sel.size and (sel.max() * block_size >= n):
        raise IndexError("block beyond its sequence")
    mask = np.zeros(n, dtype=bool)
    for b in sel:
        mask[b * block_size: min((b + 1) * block_size, p + 1)] = True
    return np.nonzero(mask)[0]


def sparse_gqa_row(q_t, K, V, blk_t, s0: int, p: int, n: int, block_size: int, scale: float):
    """One query row: per kv group g, softmax over the attended tokens of
    scale * q[h] . k[., g] for the group's heads, times v.  Returns (o [Hq,d], lse [Hq])."""
    Qt, I = as_f64(q_t), as_i64(blk_t)
    Hq = Qt.shape[0]
    Hkv = K.shape[1]
    G = Hq // Hkv
    o = np.zeros((Hq, V.shape[2]))
    lse = np.full(Hq, -np.inf)
    for g in range(Hkv):
        tok = _gqa_tokens(I[g], p, n, block_size)
        if tok.size == 0:
            continue
        Kg, Vg = K[s0 + tok, g], V[s0 + tok, g]
        hs = slice(g * G, (g + 1) * G)
        S = scale * (Qt[hs] @ Kg.T)
        m = S.max(axis=1, keepdims=True)
        e = np.exp(S - m)
        l = e.sum(axis=1, keepdims=True)
        o[hs] = (e / l) @ Vg
        lse[hs] = (m + np.log(l))[:, 0]
    return o, lse


def sparse_gqa_fwd(q, k, v, blk_idx, cu_seqlens, block_size: int, scale: float,
                   rows: Optional[Iterable[int]] = None):
    """o[t,h] = softmax over the tokens of the selected blocks of group g(h) =
    h // (Hq/Hkv) (causal inside the query's own block) of scale * q.k, times v.
    Returns (o [T,Hq,d], lse [T,Hq]) float64 (compact for ``rows``); empty
    selections give 0 / -inf."""
    K, V = as_f64(k), as_f64(v)
    T, Hq = q.shape[0], q.shape[1]
    rr = range(T) if rows is None else list(rows)
    o = np.zeros((len(rr), Hq, V.shape[2]))
    lse = np.full((len(rr), Hq), -np.inf)
    for i, t in enumerate(rr):
        s0, n = seq_bounds(cu_seqlens, t)
        o[i], lse[i] = sparse_gqa_row(q[t], K, V, blk_idx[t], s0, t - s0, n, block_size, scale)
    return o, lse


def sparse_gqa_bwd(q, k, v, blk_idx, cu_seqlens, block_size: int, scale: float, dout,
                   rows: Optional[Iterable[int]] = None):
    """Analytic gradient of sparse_gqa_fwd (fp64): dq (compact for ``rows``),
    dk, dv, with dk/dv summed over all query heads of the group and all queries
    that attend a token (exact for ``rows`` when dO is zero elsewhere)."""
    K, V = as_f64(k), as_f64(v)
    T, Hq, d = q.shape
    Hkv = K.shape[1]
    G = Hq // Hkv
    rr = list(range(T)) if rows is None else list(rows)
    dq = np.zeros((len(rr), Hq, d))
    dk, dv = np.zeros_like(K), np.zeros_like(V)
    for i, t in enumerate(rr):
        s0, n = seq_bounds(cu_seqlens, t)
        p = t - s0
        Qt, dOt, I = as_f64(q[t]), as_f64(dout[t]), as_i64(blk_idx[t])
        o_t, lse_t = sparse_gqa_row(Qt, K, V, I, s0, p, n, block_size, scale)
        for g in range(Hkv):
            tok = _gqa_tokens(I[g], p, n, block_size)
            if tok.size == 0:
                continue
            gi = s0 + tok
            Kg, Vg = K[gi, g], V[gi, g]
            hs = slice(g * G, (g + 1) * G)
            S = scale * (Qt[hs] @ Kg.T)
            P = np.exp(S - lse_t[hs][:, None])
            dP = dOt[hs] @ Vg.T
            Dlt = (dOt[hs] * o_t[hs]).sum(axis=1)
            dS = P * (dP - Dlt[:, None])
            dq[i, hs] = scale * (dS @ Kg)
            dk[gi, g] += scale * (dS.T @ Qt[hs])
            dv[gi, g] += P.T @ dOt[hs]
    return dq, dk, dv


# --------------------------------------------------------------------------
# the two exact paddings of [NOPE] ("What does this PR do?"; backport "Change")
# --------------------------------------------------------------------------

def pad_nope(x, width: int = 576) -> np.ndarray:
    """Zero-pad the last (channel) axis of a 512-wide NoPE tensor to ``width``."""
    X = as_f64(x)
    pad = [(0, 0)] * (X.ndim - 1) + [(0, width - X.shape[-1])]
    return np.pad(X, pad)


def pad_topk(idx, multiple: int = 64) -> np.ndarray:
    """Pad the slot axis to a multiple of ``multiple`` with the -1 sentinel."""
    I = as_i64(idx)
    k = I.shape[-1]
    kp = -(-k // multiple) * multiple
    pad = [(0, 0)] * (I.ndim - 1) + [(0, kp - k)]
    return np.pad(I, pad, constant_values=-1)
