"""ctypes binding of libtsa: argument marshalling only.

Every computation runs in the library's CUDA kernels.  PyTorch is used for
device memory (outputs and caller-owned workspaces) and streams.  If the
library is missing or a tensor is not on a CUDA device, the call raises: there
is no CPU path.
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional, Sequence, Tuple

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_lib", "libtsa.so")

_lib = None

c_void_p, c_int, c_int64, c_float, c_size_t = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64,
                                               ctypes.c_float, ctypes.c_size_t)
c_i32p = ctypes.POINTER(ctypes.c_int32)

# name -> (restype, argtypes); mirrors include/tsa.h
SIGNATURES = {
    "tsa_status_string": (ctypes.c_char_p, [c_int]),
    "tsa_last_error": (ctypes.c_char_p, []),
    "tsa_version": (c_int, []),
    "tsa_kernel_launches": (ctypes.c_ulonglong, []),
    "tsa_read_flags": (c_int, [ctypes.POINTER(ctypes.c_uint32), c_int, c_void_p]),
    "tsa_selftest_bounded_wait": (c_int, [c_void_p]),
    "qsa_indexer_scores": (c_int, [c_void_p, c_void_p, c_void_p, c_i32p, c_int, c_int, c_int, c_int, c_int,
                                   c_float, c_int64, c_int64, c_void_p, c_int64, c_void_p]),
    "qsa_topk_from_scores": (c_int, [c_void_p, c_int64, c_int64, c_int64, c_int, c_void_p, c_void_p]),
    "qsa_topk_workspace_size": (c_size_t, [c_i32p, c_int, c_int, c_int]),
    "qsa_topk": (c_int, [c_void_p, c_void_p, c_void_p, c_i32p, c_int, c_int, c_int, c_int, c_int, c_float,
                         c_int, c_void_p, c_void_p, c_size_t, c_void_p]),
    "qsa_topk_no_alloc": (c_int, [c_void_p, c_void_p, c_void_p, c_i32p, c_int, c_int, c_int, c_int, c_int,
                                  c_float, c_int, c_void_p, c_void_p]),
    "sparse_mla_fwd": (c_int, [c_void_p, c_void_p, c_void_p, c_i32p, c_int, c_int, c_int, c_int, c_float,
                               c_void_p, c_void_p, c_void_p]),
    "sparse_mla_bwd_workspace_size": (c_size_t, [c_int64, c_int, c_int, c_int]),
    "sparse_mla_bwd": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_i32p, c_int,
                               c_int, c_int, c_int, c_float, c_void_p, c_void_p, c_void_p, c_void_p, c_size_t,
                               c_void_p]),
    "qsa_indexer_kl": (c_int, [c_void_p, c_void_p, c_void_p, c_i32p, c_int, c_int, c_int, c_float, c_void_p, c_int,
                               c_void_p, c_void_p, c_void_p, c_void_p]),
    "qsa_indexer_bwd_workspace_size": (c_size_t, [c_int64, c_int]),
    "qsa_indexer_bwd": (c_int, [c_void_p, c_void_p, c_void_p, c_i32p, c_int, c_int, c_int, c_float, c_void_p, c_int,
                                c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_size_t, c_void_p]),
    "sparse_gqa_fwd_workspace_size": (c_size_t, [c_int64, c_int, c_int, c_int, c_int]),
    "sparse_gqa_fwd": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_i32p, c_int, c_int, c_int, c_int,
                               c_int, c_int, c_float, c_void_p, c_void_p, c_void_p, c_size_t, c_void_p]),
    "sparse_gqa_bwd_workspace_size": (c_size_t, [c_int64, c_int, c_int, c_int, c_int]),
    "sparse_gqa_bwd": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_i32p,
                               c_int, c_int, c_int, c_int, c_int, c_int, c_float, c_void_p, c_void_p, c_void_p,
                               c_void_p, c_size_t, c_void_p]),
}


class TsaError(RuntimeError):
    def __init__(self, fn: str, code: int):
        lib = load_library()
        msg = lib.tsa_status_string(code).decode()
        detail = lib.tsa_last_error().decode()
        super().__init__(f"{fn}: {msg} ({detail})")
        self.code = code


def load_library(path: Optional[str] = None):
    """Load libtsa.so (built in-tree by ``build()``; or the build at ``path``,
    which then serves every later call of this module); raises if it is absent."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"libtsa.so not found at {p}: run __graft_entry__.build() first "
                           "(there is no fallback implementation)")
    lib = ctypes.CDLL(p)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _check(fn: str, rc: int):
    if rc != 0:
        raise TsaError(fn, rc)


def _stream(stream=None) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _cu(cu_seqlens) -> Tuple[ctypes.Array, int]:
    vals = [int(v) for v in (cu_seqlens.tolist() if hasattr(cu_seqlens, "tolist") else cu_seqlens)]
    arr = (ctypes.c_int32 * len(vals))(*vals)
    return arr, len(vals) - 1


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _req(t: torch.Tensor, name: str, dtype: torch.dtype, ndim: Optional[int] = None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be on a CUDA device (libtsa has no CPU path)")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {tuple(t.shape)}")


def max_seqlen(cu_seqlens) -> int:
    vals = [int(v) for v in (cu_seqlens.tolist() if hasattr(cu_seqlens, "tolist") else cu_seqlens)]
    return max(b - a for a, b in zip(vals[:-1], vals[1:]))


# ------------------------------------------------------------------ indexer / top-k

def qsa_indexer_scores(q_idx, k_idx, w, cu_seqlens, groups: int = 1, block_size: int = 1,
                       score_scale: float = 1.0, q_begin: int = 0, q_count: Optional[int] = None,
                       width: Optional[int] = None, stream=None) -> torch.Tensor:
    """fp32 [q_count, groups, width] indexer scores (-inf = not a candidate)."""
    _req(q_idx, "q_idx", torch.bfloat16, 3)
    _req(k_idx, "k_idx", torch.bfloat16, 2)
    _req(w, "w", torch.float32, 2)
    T, H_I, d_I = q_idx.shape
    cu, nseq = _cu(cu_seqlens)
    L = max_seqlen(cu_seqlens)
    if width is None:
        width = L if block_size == 1 else -(-L // block_size)
    if q_count is None:
        q_count = T - q_begin
    out = torch.empty((q_count, groups, width), dtype=torch.float32, device=q_idx.device)
    lib = load_library()
    _check("qsa_indexer_scores", lib.qsa_indexer_scores(
        _ptr(q_idx), _ptr(k_idx), _ptr(w), cu, nseq, H_I, d_I, groups, block_size, score_scale,
        q_begin, q_count, _ptr(out), width, _stream(stream)))
    return out


def qsa_topk_from_scores(scores: torch.Tensor, topk: int, stream=None) -> torch.Tensor:
    """Deterministic exact top-k of each row of an fp32 [..., L] tensor -> int32 [..., topk]."""
    _req(scores, "scores", torch.float32)
    L = scores.shape[-1]
    rows = scores.numel() // max(L, 1) if L else 0
    out = torch.empty(scores.shape[:-1] + (topk,), dtype=torch.int32, device=scores.device)
    lib = load_library()
    _check("qsa_topk_from_scores", lib.qsa_topk_from_scores(_ptr(scores), rows, L, L, topk, _ptr(out),
                                                             _stream(stream)))
    return out


def qsa_topk_workspace_size(cu_seqlens, groups: int = 1, block_size: int = 1) -> int:
    cu, nseq = _cu(cu_seqlens)
    return int(load_library().qsa_topk_workspace_size(cu, nseq, groups, block_size))


def qsa_topk(q_idx, k_idx, w, cu_seqlens, topk: int, groups: int = 1, block_size: int = 1,
             score_scale: float = 1.0, workspace: Optional[torch.Tensor] = None, out: Optional[torch.Tensor] = None,
             stream=None) -> torch.Tensor:
    """Streaming indexer + exact top-k: int32 [T, groups, topk] (groups axis kept)."""
    _req(q_idx, "q_idx", torch.bfloat16, 3)
    _req(k_idx, "k_idx", torch.bfloat16, 2)
    _req(w, "w", torch.float32, 2)
    T, H_I, d_I = q_idx.shape
    cu, nseq = _cu(cu_seqlens)
    lib = load_library()
    need = int(lib.qsa_topk_workspace_size(cu, nseq, groups, block_size))
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q_idx.device)
    if out is None:
        out = torch.empty((T, groups, topk), dtype=torch.int32, device=q_idx.device)
    _check("qsa_topk", lib.qsa_topk(_ptr(q_idx), _ptr(k_idx), _ptr(w), cu, nseq, H_I, d_I, groups, block_size,
                                    score_scale, topk, _ptr(out), _ptr(workspace), workspace.numel(),
                                    _stream(stream)))
    return out


# ------------------------------------------------------------------ sparse MLA

def sparse_mla_fwd(q, kv, indices, cu_seqlens, softmax_scale: float, out=None, lse=None,
                   stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """out bf16 [T, H, 512], lse fp32 [T, H] (natural log)."""
    _req(q, "q", torch.bfloat16, 3)
    _req(kv, "kv", torch.bfloat16, 2)
    _req(indices, "indices", torch.int32, 2)
    T, H, D = q.shape
    topk = indices.shape[1]
    cu, nseq = _cu(cu_seqlens)
    if out is None:
        out = torch.empty((T, H, 512), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((T, H), dtype=torch.float32, device=q.device)
    lib = load_library()
    _check("sparse_mla_fwd", lib.sparse_mla_fwd(_ptr(q), _ptr(kv), _ptr(indices), cu, nseq, H, D, topk,
                                                softmax_scale, _ptr(out), _ptr(lse), _stream(stream)))
    return out, lse


def sparse_mla_bwd_workspace_size(T: int, H: int, d_qk: int, topk: int) -> int:
    return int(load_library().sparse_mla_bwd_workspace_size(T, H, d_qk, topk))


def sparse_mla_bwd(q, kv, indices, out, lse, dout, cu_seqlens, softmax_scale: float, workspace=None,
                   dq=None, dkv=None, teacher=None, want_teacher: bool = False, stream=None):
    """dq bf16 [T, H, D], dkv bf16 [T, D]; with ``want_teacher`` (or a given
    fp32 [T, topk] ``teacher`` buffer) also the indexer's KL teacher, the head
    mean of the attention probabilities at every slot: (dq, dkv, teacher)."""
    for t, n, dt in ((q, "q", torch.bfloat16), (kv, "kv", torch.bfloat16), (indices, "indices", torch.int32),
                     (out, "out", torch.bfloat16), (lse, "lse", torch.float32), (dout, "dout", torch.bfloat16)):
        _req(t, n, dt)
    T, H, D = q.shape
    topk = indices.shape[1]
    cu, nseq = _cu(cu_seqlens)
    lib = load_library()
    need = int(lib.sparse_mla_bwd_workspace_size(T, H, D, topk))
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    if dq is None:
        dq = torch.empty_like(q)
    if dkv is None:
        dkv = torch.empty_like(kv)
    if teacher is None and want_teacher:
        teacher = torch.empty((T, topk), dtype=torch.float32, device=q.device)
    if teacher is not None:
        _req(teacher, "teacher", torch.float32)
    _check("sparse_mla_bwd", lib.sparse_mla_bwd(_ptr(q), _ptr(kv), _ptr(indices), _ptr(out), _ptr(lse), _ptr(dout),
                                                cu, nseq, H, D, topk, softmax_scale, _ptr(dq), _ptr(dkv),
                                                _ptr(teacher), _ptr(workspace), workspace.numel(),
                                                _stream(stream)))
    return (dq, dkv, teacher) if teacher is not None else (dq, dkv)


# ------------------------------------------------------------------ indexer training

def _sel_indices(indices) -> Tuple[torch.Tensor, int]:
    _req(indices, "indices", torch.int32)
    return indices, indices.shape[-1]


def qsa_indexer_kl(q_idx, k_idx, w, cu_seqlens, indices, teacher, score_scale: float = 1.0, loss=None,
                   dscore=None, stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Sparse KL of the indexer against the teacher on the selected slots:
    (loss fp32 [T], dscore fp32 [T, topk] = softmax(student) - teacher)."""
    _req(q_idx, "q_idx", torch.bfloat16, 3)
    _req(k_idx, "k_idx", torch.bfloat16, 2)
    _req(w, "w", torch.float32, 2)
    indices, topk = _sel_indices(indices)
    _req(teacher, "teacher", torch.float32)
    T, H_I, d_I = q_idx.shape
    cu, nseq = _cu(cu_seqlens)
    if loss is None:
        loss = torch.empty((T,), dtype=torch.float32, device=q_idx.device)
    if dscore is None:
        dscore = torch.empty((T, topk), dtype=torch.float32, device=q_idx.device)
    _check("qsa_indexer_kl", load_library().qsa_indexer_kl(
        _ptr(q_idx), _ptr(k_idx), _ptr(w), cu, nseq, H_I, d_I, score_scale, _ptr(indices), topk, _ptr(teacher),
        _ptr(loss), _ptr(dscore), _stream(stream)))
    return loss, dscore


def qsa_indexer_bwd_workspace_size(T: int, d_I: int) -> int:
    return int(load_library().qsa_indexer_bwd_workspace_size(T, d_I))


def qsa_indexer_bwd(q_idx, k_idx, w, cu_seqlens, indices, dscore, score_scale: float = 1.0, workspace=None,
                    dq=None, dk=None, dw=None, stream=None):
    """Backward of the indexer score on the selected slots: (dq_idx bf16
    [T, H_I, d_I], dk_idx bf16 [T, d_I], dw fp32 [T, H_I])."""
    _req(q_idx, "q_idx", torch.bfloat16, 3)
    _req(k_idx, "k_idx", torch.bfloat16, 2)
    _req(w, "w", torch.float32, 2)
    indices, topk = _sel_indices(indices)
    _req(dscore, "dscore", torch.float32)
    T, H_I, d_I = q_idx.shape
    cu, nseq = _cu(cu_seqlens)
    lib = load_library()
    need = int(lib.qsa_indexer_bwd_workspace_size(T, d_I))
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q_idx.device)
    dq = torch.empty_like(q_idx) if dq is None else dq
    dk = torch.empty_like(k_idx) if dk is None else dk
    dw = torch.empty_like(w) if dw is None else dw
    _check("qsa_indexer_bwd", lib.qsa_indexer_bwd(
        _ptr(q_idx), _ptr(k_idx), _ptr(w), cu, nseq, H_I, d_I, score_scale, _ptr(indices), topk, _ptr(dscore),
        _ptr(dq), _ptr(dk), _ptr(dw), _ptr(workspace), workspace.numel(), _stream(stream)))
    return dq, dk, dw


# ------------------------------------------------------------------ sparse GQA

def sparse_gqa_fwd_workspace_size(T: int, Hq: int, Hkv: int, d: int, nsel: int) -> int:
    return int(load_library().sparse_gqa_fwd_workspace_size(T, Hq, Hkv, d, nsel))


def sparse_gqa_fwd(q, k, v, block_indices, cu_seqlens, block_size: int, softmax_scale: float, out=None,
                   lse=None, workspace=None, stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """out bf16 [T, Hq, d], lse fp32 [T, Hq]."""
    _req(q, "q", torch.bfloat16, 3)
    _req(k, "k", torch.bfloat16, 3)
    _req(v, "v", torch.bfloat16, 3)
    _req(block_indices, "block_indices", torch.int32, 3)
    T, Hq, d = q.shape
    Hkv = k.shape[1]
    nsel = block_indices.shape[2]
    cu, nseq = _cu(cu_seqlens)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((T, Hq), dtype=torch.float32, device=q.device)
    lib = load_library()
    need = int(lib.sparse_gqa_fwd_workspace_size(T, Hq, Hkv, d, nsel))
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    _check("sparse_gqa_fwd", lib.sparse_gqa_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(block_indices), cu, nseq, Hq, Hkv,
                                                d, block_size, nsel, softmax_scale, _ptr(out), _ptr(lse),
                                                _ptr(workspace), workspace.numel(), _stream(stream)))
    return out, lse


def sparse_gqa_bwd_workspace_size(T: int, Hq: int, Hkv: int, d: int, nsel: int) -> int:
    return int(load_library().sparse_gqa_bwd_workspace_size(T, Hq, Hkv, d, nsel))


def sparse_gqa_bwd(q, k, v, block_indices, out, lse, dout, cu_seqlens, block_size: int, softmax_scale: float,
                   workspace=None, stream=None):
    """(dq, dk, dv) bf16."""
    for t, n, dt in ((q, "q", torch.bfloat16), (k, "k", torch.bfloat16), (v, "v", torch.bfloat16),
                     (block_indices, "block_indices", torch.int32), (out, "out", torch.bfloat16),
                     (lse, "lse", torch.float32), (dout, "dout", torch.bfloat16)):
        _req(t, n, dt)
    T, Hq, d = q.shape
    Hkv = k.shape[1]
    nsel = block_indices.shape[2]
    cu, nseq = _cu(cu_seqlens)
    lib = load_library()
    need = int(lib.sparse_gqa_bwd_workspace_size(T, Hq, Hkv, d, nsel))
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    _check("sparse_gqa_bwd", lib.sparse_gqa_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(block_indices), _ptr(out),
                                                _ptr(lse), _ptr(dout), cu, nseq, Hq, Hkv, d, block_size, nsel,
                                                softmax_scale, _ptr(dq), _ptr(dk), _ptr(dv), _ptr(workspace),
                                                workspace.numel(), _stream(stream)))
    return dq, dk, dv


def kernel_launches() -> int:
    """Kernels libtsa has launched since it was loaded."""
    return int(load_library().tsa_kernel_launches())


def read_flags(clear: bool = True, stream=None) -> int:
    """Device error flags raised since the last clear (TSA_FLAG_* bits)."""
    v = ctypes.c_uint32(0)
    _check("tsa_read_flags", load_library().tsa_read_flags(ctypes.byref(v), int(clear), _stream(stream)))
    return int(v.value)


def selftest_bounded_wait(stream=None) -> None:
    """Launch the library's bounded-wait self-test (a wait that nothing
    satisfies gives up after 2 s and raises FLAG_TIMEOUT); read the flag with
    read_flags()."""
    _check("tsa_selftest_bounded_wait", load_library().tsa_selftest_bounded_wait(_stream(stream)))


FLAG_INDEX_RANGE = 0x1
FLAG_TIMEOUT = 0x2
