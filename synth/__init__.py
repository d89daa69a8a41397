"""Seeded synthetic inputs for the sparse-attention hot path.

This module only draws random numbers and shapes them; it holds none of the
method's arithmetic (no scores, no softmax, no selection).  Both the CUDA path
and the CPU oracle are fed from here, never from each other.

Every generator takes an explicit ``seed`` and ``device``; values depend on the
(seed, device) pair because torch's CPU and CUDA generators differ.  bf16
tensors are drawn in fp32 and rounded once with round-to-nearest-even.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Dict, List, Optional

import torch

__all__ = [
    "gen", "randn_bf16", "uniform_f32", "cu_seqlens_bshd", "cu_seqlens_thd",
    "mla_inputs", "indexer_inputs", "gqa_inputs", "random_topk_indices",
    "random_block_indices", "tie_stress_scores", "Workload", "WORKLOADS",
]


def gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=torch.device(device))
    g.manual_seed(int(seed))
    return g


def randn_bf16(shape, g: torch.Generator, device) -> torch.Tensor:
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)


def uniform_f32(shape, g: torch.Generator, device) -> torch.Tensor:
    return torch.rand(shape, generator=g, device=device, dtype=torch.float32)


def small_int_bf16(shape, g: torch.Generator, device, lo: int = -3, hi: int = 3) -> torch.Tensor:
    """Integers in [lo, hi]: exact in bf16, so dot products are exact in fp32."""
    return torch.randint(lo, hi + 1, shape, generator=g, device=device).to(torch.bfloat16)


def dyadic_unit_f32(shape, g: torch.Generator, device, bits: int = 6) -> torch.Tensor:
    """Multiples of 2**-bits in [0, 1): few mantissa bits, so products stay exact."""
    n = 1 << bits
    return torch.randint(0, n, shape, generator=g, device=device).to(torch.float32) / n


def cu_seqlens_bshd(batch: int, seqlen: int) -> List[int]:
    return [i * seqlen for i in range(batch + 1)]


def cu_seqlens_thd(lengths) -> List[int]:
    out = [0]
    for n in lengths:
        out.append(out[-1] + int(n))
    return out


def mla_inputs(T: int, H: int, D: int, seed: int, device="cpu", with_grad_out: bool = False,
               d_v: int = 512) -> Dict[str, torch.Tensor]:
    """Absorbed-MLA tensors: q [T,H,D], kv [T,D] (D = 576 or NoPE 512), dO [T,H,d_v]."""
    g = gen(seed, device)
    out = {"q": randn_bf16((T, H, D), g, device), "kv": randn_bf16((T, D), g, device)}
    if with_grad_out:
        out["dout"] = randn_bf16((T, H, d_v), g, device)
    return out


def indexer_inputs(T: int, H_I: int, d_I: int, seed: int, device="cpu", zero_key_frac: float = 0.0,
                   dead_queries: int = 0, integer: bool = False) -> Dict[str, torch.Tensor]:
    """Indexer tensors q_I [T,H_I,d_I] bf16, k_I [T,d_I] bf16, w [T,H_I] fp32.

    ``zero_key_frac``: a seeded Bernoulli mask of key rows is set to exactly 0,
    so every score against those keys is exactly 0 (the zero-tie stress case).
    ``dead_queries``: that many seeded query rows get q_I = 0 (all-zero rows).
    ``integer``: small-integer q_I/k_I and dyadic w, so every score is exact in fp32.
    """
    g = gen(seed, device)
    if integer:
        qI = small_int_bf16((T, H_I, d_I), g, device)
        kI = small_int_bf16((T, d_I), g, device)
        w = dyadic_unit_f32((T, H_I), g, device)
    else:
        qI = randn_bf16((T, H_I, d_I), g, device)
        kI = randn_bf16((T, d_I), g, device)
        w = uniform_f32((T, H_I), g, device)
    if zero_key_frac > 0:
        mask = torch.rand((T,), generator=g, device=device) < zero_key_frac
        kI[mask] = 0
    if dead_queries > 0:
        rows = torch.randperm(T, generator=g, device=device)[:dead_queries]
        qI[rows] = 0
    return {"q_idx": qI, "k_idx": kI, "w": w}


def gqa_inputs(T: int, Hq: int, Hkv: int, d: int, seed: int, device="cpu",
               with_grad_out: bool = False) -> Dict[str, torch.Tensor]:
    g = gen(seed, device)
    out = {"q": randn_bf16((T, Hq, d), g, device), "k": randn_bf16((T, Hkv, d), g, device),
           "v": randn_bf16((T, Hkv, d), g, device)}
    if with_grad_out:
        out["dout"] = randn_bf16((T, Hq, d), g, device)
    return out


def random_topk_indices(cu_seqlens, topk: int, seed: int, device="cpu", causal: bool = True,
                        invalid_rows=(), invalid_frac: float = 0.0) -> torch.Tensor:
    """Distinct local key positions per query, -1 where a row has fewer candidates.

    Rows listed in ``invalid_rows`` (and a seeded ``invalid_frac`` of the rest)
    are entirely -1.
    """
    g = gen(seed, "cpu")
    T = cu_seqlens[-1]
    idx = torch.full((T, topk), -1, dtype=torch.int32)
    for b in range(len(cu_seqlens) - 1):
        s0, s1 = cu_seqlens[b], cu_seqlens[b + 1]
        n = s1 - s0
        for p in range(n):
            ncand = p + 1 if causal else n
            m = min(topk, ncand)
            perm = torch.randperm(ncand, generator=g)[:m]
            idx[s0 + p, :m] = perm.to(torch.int32)
    if invalid_frac > 0:
        extra = (torch.rand((T,), generator=g) < invalid_frac).nonzero().flatten().tolist()
    else:
        extra = []
    for r in list(invalid_rows) + extra:
        if 0 <= r < T:
            idx[r] = -1
    return idx.to(device)


def random_block_indices(cu_seqlens, Hkv: int, nsel: int, block_size: int, seed: int,
                         device="cpu") -> torch.Tensor:
    """Distinct causal local block ids per (query, kv group), -1 padded."""
    g = gen(seed, "cpu")
    T = cu_seqlens[-1]
    idx = torch.full((T, Hkv, nsel), -1, dtype=torch.int32)
    for b in range(len(cu_seqlens) - 1):
        s0, s1 = cu_seqlens[b], cu_seqlens[b + 1]
        for p in range(s1 - s0):
            nb = p // block_size + 1
            m = min(nsel, nb)
            for h in range(Hkv):
                idx[s0 + p, h, :m] = torch.randperm(nb, generator=g)[:m].to(torch.int32)
    return idx.to(device)


def tie_stress_scores(rows: int, L: int, seed: int, device="cpu", n_levels: int = 8,
                      neg_inf_tail: bool = True) -> torch.Tensor:
    """fp32 score rows drawn from a few repeated levels (heavy exact ties), with
    +0/-0 mixed in and an -inf (non-candidate) tail of random length per row."""
    g = gen(seed, device)
    levels = torch.randn((n_levels,), generator=g, device=device)
    levels[0] = 0.0
    levels[1] = -0.0
    pick = torch.randint(0, n_levels, (rows, L), generator=g, device=device)
    s = levels[pick]
    # some genuinely distinct values too
    noise_mask = torch.rand((rows, L), generator=g, device=device) < 0.25
    s = torch.where(noise_mask, torch.randn((rows, L), generator=g, device=device), s)
    if neg_inf_tail:
        n_valid = torch.randint(0, L + 1, (rows,), generator=g, device=device)
        col = torch.arange(L, device=device)[None, :]
        s = torch.where(col < n_valid[:, None], s, torch.full_like(s, -math.inf))
    return s.contiguous()


@dataclass
class Workload:
    """A named synthetic workload (shapes and recipe only)."""
    name: str
    kind: str                  # "mla" or "gqa"
    lengths: List[int]
    H: int = 0
    D: int = 576
    topk: int = 0
    scale: float = 0.0
    H_I: int = 0
    d_I: int = 0
    groups: int = 1
    block_size: int = 1
    Hkv: int = 0
    d: int = 0
    backward: bool = True
    zero_key_frac: float = 0.0
    dead_queries: int = 0
    extra: dict = field(default_factory=dict)

    @property
    def T(self) -> int:
        return sum(self.lengths)

    @property
    def cu_seqlens(self) -> List[int]:
        return cu_seqlens_thd(self.lengths)


WORKLOADS: Dict[str, Workload] = {
    # tiny absorbed MLA, forward only
    "mla_t256_h8": Workload("mla_t256_h8", "mla", [256], H=8, D=576, topk=64, scale=1 / math.sqrt(576),
                            H_I=4, d_I=64, backward=False),
    # DSA-style absorbed MLA with zero-tie stress in the indexer
    "mla_t4096_h16": Workload("mla_t4096_h16", "mla", [4096], H=16, D=576, topk=2048,
                              scale=1 / math.sqrt(576), H_I=8, d_I=128, zero_key_frac=0.3,
                              dead_queries=16),
    # QSA block sparse GQA over four packed sequences
    "gqa_thd32768": Workload("gqa_thd32768", "gqa", [4096, 8192, 12288, 8192], Hkv=4, H=32, d=128,
                             topk=32, scale=1 / math.sqrt(128), H_I=8, d_I=128, groups=4,
                             block_size=64),
    # long-context absorbed MLA
    "mla_t65536_h128": Workload("mla_t65536_h128", "mla", [65536], H=128, D=576, topk=2048,
                                scale=1 / math.sqrt(192), H_I=64, d_I=128),
}


def spread_topk_indices(cu_seqlens, topk: int, seed: int, device="cpu") -> torch.Tensor:
    """Distinct causal local indices spread over each query's range, built with
    tensor ops (fast at T = 65536 on the device).

    Query at local position p: if p+1 <= topk every key 0..p appears once (in a
    rotated order) and the rest is -1; otherwise slot j holds
    (floor(j*(p+1)/topk) + r_t) mod (p+1) with a seeded per-row rotation r_t.
    """
    g = gen(seed, device)
    T = cu_seqlens[-1]
    cu = torch.tensor(cu_seqlens, device=device, dtype=torch.int64)
    t = torch.arange(T, device=device, dtype=torch.int64)
    seq = torch.searchsorted(cu, t, right=True) - 1
    n_cand = t - cu[seq] + 1                                   # p + 1
    rot = (torch.rand((T,), generator=g, device=device) * n_cand.to(torch.float32)).to(torch.int64)
    rot = torch.minimum(rot, n_cand - 1)
    j = torch.arange(topk, device=device, dtype=torch.int64)[None, :]
    wide = n_cand[:, None] > topk
    base = torch.where(wide, (j * n_cand[:, None]) // topk, j)
    idx = (base + rot[:, None]) % n_cand[:, None]
    idx = torch.where(wide | (j < n_cand[:, None]), idx, torch.full_like(idx, -1))
    return idx.to(torch.int32).contiguous()


def spread_block_indices(cu_seqlens, Hkv: int, nsel: int, block_size: int, seed: int,
                         device="cpu") -> torch.Tensor:
    """Causal distinct local block ids per (query, kv group), spread over the
    query's causal blocks with a seeded per-row rotation; -1 padded.
    int32 [T, Hkv, nsel], built with tensor ops."""
    g = gen(seed, device)
    T = cu_seqlens[-1]
    cu = torch.tensor(cu_seqlens, device=device, dtype=torch.int64)
    t = torch.arange(T, device=device, dtype=torch.int64)
    seq = torch.searchsorted(cu, t, right=True) - 1
    nb = (t - cu[seq]) // block_size + 1                      # causal blocks of each query
    rot = (torch.rand((T, Hkv), generator=g, device=device) * nb[:, None].to(torch.float32)).to(torch.int64)
    rot = torch.minimum(rot, nb[:, None] - 1)
    j = torch.arange(nsel, device=device, dtype=torch.int64)[None, None, :]
    nbb = nb[:, None, None]
    wide = nbb > nsel
    base = torch.where(wide, (j * nbb) // nsel, j)
    b = (base + rot[:, :, None]) % nbb
    b = torch.where(wide | (j < nbb), b, torch.full_like(b, -1))
    return b.to(torch.int32).contiguous()
