"""Comparison helpers shared by the parity tests (no method arithmetic)."""
from __future__ import annotations

import numpy as np
import torch

import oracle as O

# Tolerances of the parity contract: bf16 inputs, fp32 accumulation.
TOL_OUT = 1e-2       # rel-L2, outputs and LSE
TOL_GRAD = 2e-2      # rel-L2, gradients
TOL_LSE_ABS = 1e-2   # max-abs, LSE
U32 = 2.0 ** -24     # unit roundoff of fp32


def f64(x) -> np.ndarray:
    return O.as_f64(x)


def rel_l2(got, ref) -> float:
    g, r = f64(got), f64(ref)
    den = np.linalg.norm(r.ravel())
    num = np.linalg.norm((g - r).ravel())
    return float(num / den) if den > 0 else float(num)


# Per-row bounds: besides the whole-tensor rel-L2, every row (a (query, head)
# output or gradient row, a key row of dK / dV / dKV) is bounded, so that a
# defect confined to a few rows cannot hide in the global norm:
#   ||got_i - ref_i|| <= tol * max(||ref_i||, ROW_FLOOR * med) + abs_frac * med,
# med = the median nonzero reference row norm.  Outputs use abs_frac = 0.
# Gradients add GRAD_ROW_ABS: the backward's Delta = rowsum(dO * out) is taken
# from the forward's bf16 output, whose rounding (and the bf16 P of the
# forward's P.V) moves Delta by ~2^-9 sqrt(d_v) |dO| |o| whatever the row, and
# that error reaches dq as scale * dDelta * (the attention-weighted mean key):
# an absolute error of a few percent of a typical row on rows whose own dq
# nearly cancels (one dominant key).  A wrong tile of a row (a sixth of its
# slots) moves it by ~40 % of a typical row and still fails by a wide margin.
ROW_FLOOR = 0.05
GRAD_ROW_ABS = 0.1


def row_errors(got, ref, tol, abs_frac=0.0):
    """Per-row error divided by its bound (<= 1 passes), rows = last axis."""
    g, r = f64(got), f64(ref)
    c = r.shape[-1]
    g, r = g.reshape(-1, c), r.reshape(-1, c)
    rn = np.linalg.norm(r, axis=1)
    nz = rn[rn > 0]
    med = float(np.median(nz)) if nz.size else 1.0
    bound = tol * np.maximum(rn, ROW_FLOOR * med) + abs_frac * med
    return np.linalg.norm(g - r, axis=1) / bound, rn / med


def check_rows(got, ref, tol, what="rows", abs_frac=0.0):
    """Assert the per-row bound; prints and returns the worst row's error / bound."""
    e, rel = row_errors(got, ref, tol, abs_frac)
    worst = float(e.max()) if e.size else 0.0
    i = int(e.argmax()) if e.size else 0
    print(f"[rows] {what}: worst row {i} at {worst:.3f} of its bound (row norm {rel[i] if e.size else 0:.3f} x median)")
    assert worst <= 1.0, f"{what}: row {i} error {worst:.3f} x its bound ({int((e > 1).sum())} rows over)"
    return worst


def check_grad(got, ref, what="grad", tol=TOL_GRAD):
    """Gradient parity: whole-tensor rel-L2 and every row within its bound."""
    e = rel_l2(got, ref)
    assert e <= tol, f"{what}: rel-L2 {e:.3e} > {tol}"
    check_rows(got, ref, tol, what, GRAD_ROW_ABS)
    return e


def check_out_lse(o_gpu, lse_gpu, o_ref, lse_ref, rows=None, tol=TOL_OUT):
    """Compare GPU (out, lse) with the oracle's; with ``rows`` the oracle arrays
    are the compact per-row outputs and the GPU arrays are full."""
    if rows is not None:
        o_gpu, lse_gpu = o_gpu[rows], lse_gpu[rows]
    o_g, l_g = f64(o_gpu), f64(lse_gpu)
    o_r, l_r = np.asarray(o_ref), np.asarray(lse_ref)
    inf_r = np.isneginf(l_r)
    assert np.array_equal(np.isneginf(l_g), inf_r), "empty-row pattern differs"
    assert np.all(o_g[inf_r] == 0), "empty rows must give exactly zero output"
    e_o = rel_l2(o_g, o_r)
    assert e_o <= tol, f"out rel-L2 {e_o:.3e} > {tol}"
    check_rows(o_g, o_r, tol, "out rows")
    fin = ~inf_r
    if fin.any():
        e_l = rel_l2(l_g[fin], l_r[fin])
        m_l = float(np.max(np.abs(l_g[fin] - l_r[fin])))
        assert e_l <= tol, f"lse rel-L2 {e_l:.3e} > {tol}"
        assert m_l <= TOL_LSE_ABS, f"lse max-abs {m_l:.3e} > {TOL_LSE_ABS}"
    return e_o


def indexer_score_bound(q_idx, k_idx, w, cu_seqlens, t, groups=1):
    """Forward error bound of fp32 recursive summation for the indexer score of
    row t: (d_I + H_I/groups + 4) * u * max_s sum_h |w| sum_d |q k|, per group."""
    q, k, W = f64(q_idx[t]), f64(k_idx), f64(w[t])
    s0, n = O.seq_bounds(cu_seqlens, t)
    p = t - s0
    H, d = q.shape
    hg = H // groups
    absdot = np.abs(q) @ np.abs(k[s0:s0 + p + 1]).T    # [H, p+1]
    out = []
    for g in range(groups):
        m = (np.abs(W[g * hg:(g + 1) * hg]) @ absdot[g * hg:(g + 1) * hg]).max()
        out.append((d + hg + 4) * U32 * m)
    return np.array(out)


def compare_topk_rows(gpu_idx: np.ndarray, oracle_scores: np.ndarray, k: int, tol: float):
    """Check one GPU top-k row against the oracle's fp32 scores.

    Exact equality is required unless the oracle's scores at the selection
    boundary lie within `tol` (the fp32 error bound) of each other; then the
    GPU row must still be a valid selection: distinct candidates, right count,
    every swapped index within tol of the oracle's k-th score, ordered up to tol.
    Returns the number of slots that differ from the oracle row.
    """
    ref = O.topk_lex(oracle_scores, k)
    if np.array_equal(gpu_idx, ref):
        return 0
    cand = np.nonzero(oracle_scores != -np.inf)[0]
    nsel = min(k, cand.size)
    sel = gpu_idx[:nsel]
    assert np.all(gpu_idx[nsel:] == -1), "padding must be -1"
    assert np.all(sel >= 0) and len(set(sel.tolist())) == nsel, "duplicate or missing index"
    assert np.all(oracle_scores[sel] != -np.inf), "selected a non-candidate"
    tau = oracle_scores[ref[nsel - 1]]
    diff = set(sel.tolist()) ^ set(ref[:nsel].tolist())
    for i in diff:
        assert abs(float(oracle_scores[i]) - float(tau)) <= tol, f"index {i} swapped beyond tolerance"
    s = oracle_scores[sel].astype(np.float64)
    assert np.all(s[:-1] >= s[1:] - 2 * tol), "order violated beyond tolerance"
    return int(np.sum(gpu_idx != ref))
