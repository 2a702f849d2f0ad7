"""GB300-native (sm_103a) DeepSeek Sparse Attention hot path.

Thin Python binding over the C ABI of ``libdsa.so`` (see ``include/dsa.h``).
The functions carry the C entry points' names and only marshal arguments:
torch supplies device memory and the current CUDA stream; every step of the
computation runs in the library's CUDA kernels.  There is no CPU fallback: if
the library is missing or the device is not sm_103, the calls raise.
"""
from __future__ import annotations

import ctypes
import math
import os
import re
import threading

import torch

from .build_ext import LIB as _LIB_PATH
from .build_ext import INCLUDE as _INCLUDE

__all__ = [
    "DsaError",
    "load_library",
    "declared_symbols",
    "dsa_packed_metadata",
    "dsa_packed_metadata_cp",
    "dsa_indexer_topk",
    "dsa_indexer_topk_cp",
    "dsa_indexer_topk_with_scores",
    "dsa_indexer_topk_scored",
    "dsa_indexer_kl",
    "dsa_kpool_metadata",
    "dsa_kpool_pool",
    "dsa_kpool_topk",
    "dsa_kpool_unpool_grad",
    "dsa_sparse_mla_fwd",
    "dsa_sparse_mla_bwd",
    "dsa_sparse_mla_bwd_noalloc",
    "dsa_sparse_mla_bwd_noalloc_read_status",
    "dsa_read_device_status",
    "dsa_set_wait_limit_cycles",
    "workspace_size",
]

DSA_OK = 0
STATUS_NAMES = {
    0: "DSA_OK",
    1: "DSA_ERR_UNSUPPORTED",
    2: "DSA_ERR_DTYPE",
    3: "DSA_ERR_INVALID_ARGUMENT",
    4: "DSA_ERR_WORKSPACE",
    5: "DSA_ERR_CUDA",
    6: "DSA_ERR_DEVICE_INDEX",
    7: "DSA_ERR_TIMEOUT",
}


class DsaError(RuntimeError):
    def __init__(self, status: int, where: str, message: str):
        self.status = status
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}: {message}")


_lib = None
_lock = threading.Lock()
_P = ctypes.c_void_p
_I = ctypes.c_int32
_SZ = ctypes.c_size_t
_F = ctypes.c_float


def declared_symbols() -> list[str]:
    """Function names declared in include/*.h (the ABI surface)."""
    names = []
    for fn in sorted(os.listdir(_INCLUDE)):
        if fn.endswith(".h"):
            text = open(os.path.join(_INCLUDE, fn)).read()
            names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*(dsa_[a-z0-9_]+)\s*\(", text, re.M)
    return sorted(set(names))


def load_library(path: str | None = None):
    """Load libdsa.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = path or _LIB_PATH
        if not os.path.exists(path):
            raise RuntimeError(
                f"{path} not found: build the CUDA library first "
                "(python -m sparse_attention_mla_gb300.build_ext, or __graft_entry__.build())")
        lib = ctypes.CDLL(path)
        lib.dsa_status_string.restype = ctypes.c_char_p
        lib.dsa_status_string.argtypes = [ctypes.c_int]
        lib.dsa_last_error_message.restype = ctypes.c_char_p
        lib.dsa_last_error_message.argtypes = []
        lib.dsa_abi_version.restype = _I
        lib.dsa_packed_metadata.argtypes = [_P, _I, _I, _P, _P, _P, _P, _P]
        lib.dsa_packed_metadata_cp.argtypes = [_P, _P, _I, _I, _P, _P, _I, _P, _P, _P, _P, _P]
        lib.dsa_indexer_topk_workspace_size.argtypes = [_I, _I]
        lib.dsa_indexer_topk_workspace_size.restype = _SZ
        lib.dsa_indexer_topk.argtypes = [_P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _SZ, _P]
        lib.dsa_indexer_topk_cp.argtypes = [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _SZ, _P]
        lib.dsa_indexer_topk_scored.argtypes = [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _SZ, _P]
        lib.dsa_indexer_topk_with_scores.argtypes = [_P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _I, _I, _P,
                                                     _SZ, _P]
        lib.dsa_sparse_mla_fwd_workspace_size.argtypes = [_I, _I]
        lib.dsa_sparse_mla_fwd_workspace_size.restype = _SZ
        lib.dsa_sparse_mla_fwd.argtypes = [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _P, _P, _P, _P, _P, _SZ, _P]
        lib.dsa_sparse_mla_bwd_workspace_size.argtypes = [_I, _I, _I]
        lib.dsa_sparse_mla_bwd_workspace_size.restype = _SZ
        lib.dsa_sparse_mla_bwd.argtypes = [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _P, _P, _P, _P, _P, _P, _P,
                                           _P, _P, _I, _P, _P, _SZ, _P]
        lib.dsa_read_device_status.argtypes = [_P, _P, _P]
        lib.dsa_indexer_kl_workspace_size.argtypes = [_I, _I]
        lib.dsa_indexer_kl_workspace_size.restype = _SZ
        lib.dsa_indexer_kl.argtypes = [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _P, _P, _P, _P, _I, _P,
                                       _SZ, _P]
        lib.dsa_indexer_kl.restype = ctypes.c_int
        lib.dsa_set_wait_limit_cycles.argtypes = [ctypes.c_int64]
        lib.dsa_set_wait_limit_cycles.restype = ctypes.c_int64
        lib.dsa_sparse_mla_bwd_noalloc_max_topk.restype = _I
        lib.dsa_sparse_mla_bwd_noalloc_max_topk.argtypes = []
        lib.dsa_sparse_mla_bwd_noalloc.argtypes = [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _P, _P, _P, _P, _P,
                                                   _P, _P, _P, _P, _I, _P, _P]
        lib.dsa_sparse_mla_bwd_noalloc.restype = ctypes.c_int
        lib.dsa_sparse_mla_bwd_noalloc_read_status.argtypes = [_P, _P]
        lib.dsa_sparse_mla_bwd_noalloc_read_status.restype = ctypes.c_int
        lib.dsa_kpool_metadata.argtypes = [_P, _I, _I, _I, _P, _P, _P, _P, _P, _P]
        lib.dsa_kpool_pool.argtypes = [_P, _I, _I, _P, _P, _I, _I, _I, _P, _P]
        lib.dsa_kpool_topk_workspace_size.argtypes = [_I, _I]
        lib.dsa_kpool_topk_workspace_size.restype = _SZ
        lib.dsa_kpool_topk.argtypes = [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P, _P, _SZ, _P]
        lib.dsa_kpool_unpool_grad.argtypes = [_P, _I, _I, _P, _P, _I, _I, _I, _P, _P]
        for name in ("dsa_kpool_metadata", "dsa_kpool_pool", "dsa_kpool_topk", "dsa_kpool_unpool_grad"):
            getattr(lib, name).restype = ctypes.c_int
        for name in ("dsa_packed_metadata", "dsa_indexer_topk", "dsa_indexer_topk_with_scores", "dsa_indexer_topk_scored",
                     "dsa_indexer_topk_cp",
                     "dsa_sparse_mla_fwd", "dsa_sparse_mla_bwd", "dsa_read_device_status"):
            getattr(lib, name).restype = ctypes.c_int
        _lib = lib
        return lib


def _check(status: int, where: str):
    if status != DSA_OK:
        lib = load_library()
        raise DsaError(status, where, lib.dsa_last_error_message().decode())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _need(t, name, dtype, ndim=None, device=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got shape {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def workspace_size(kind: str, T: int, H_or_K: int, K: int | None = None) -> int:
    """Workspace bytes: ("fwd", T, H), ("indexer", T, K) or ("bwd", T, H, K)."""
    lib = load_library()
    if kind == "bwd":
        if K is None:
            raise ValueError('workspace_size("bwd", T, H, K) needs the top-k width K')
        return int(lib.dsa_sparse_mla_bwd_workspace_size(int(T), int(H_or_K), int(K)))
    fn = {"fwd": lib.dsa_sparse_mla_fwd_workspace_size, "indexer": lib.dsa_indexer_topk_workspace_size}[kind]
    return int(fn(int(T), int(H_or_K)))


def _workspace(kind, T, x, device, workspace, K=None):
    need = workspace_size(kind, T, x, K)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=device)
    return workspace, workspace.numel()


def dsa_packed_metadata(cu_seqlens: torch.Tensor, total_tokens: int):
    """cu_seqlens int32 [nseq+1] (CUDA) -> (seq_start [T], causal_len [T], max_seqlen, all_rows_nonempty)."""
    lib = load_library()
    _need(cu_seqlens, "cu_seqlens", torch.int32, 1)
    dev = cu_seqlens.device
    T = int(total_tokens)
    start = torch.empty(T, dtype=torch.int32, device=dev)
    clen = torch.empty(T, dtype=torch.int32, device=dev)
    mx = ctypes.c_int32(0)
    ne = ctypes.c_int32(0)
    _check(lib.dsa_packed_metadata(_ptr(cu_seqlens), cu_seqlens.numel() - 1, T, _ptr(start), _ptr(clen),
                                   ctypes.byref(mx), ctypes.byref(ne), _stream(dev)), "dsa_packed_metadata")
    return start, clen, mx.value, ne.value


def dsa_packed_metadata_cp(cu_seqlens: torch.Tensor, total_key_tokens: int, query_indices=None,
                           cu_seqlens_padded=None, padding_mask=None, T_q: int | None = None):
    """Context-parallel metadata: rank-local query rows (global padded coordinates `query_indices`,
    identity when None) against gathered global keys -> (seq_start [T_q], causal_len [T_q],
    max_seqlen, all_rows_nonempty).  padding_mask: bool/uint8 [T_q], True marks a padding row."""
    lib = load_library()
    _need(cu_seqlens, "cu_seqlens", torch.int32, 1)
    dev = cu_seqlens.device
    if cu_seqlens_padded is not None:
        _need(cu_seqlens_padded, "cu_seqlens_padded", torch.int32, 1, dev)
        if cu_seqlens_padded.numel() != cu_seqlens.numel():
            raise ValueError("cu_seqlens_padded must have as many entries as cu_seqlens")
    if query_indices is not None:
        _need(query_indices, "query_indices", torch.int32, 1, dev)
    if T_q is None:
        T_q = query_indices.numel() if query_indices is not None else int(total_key_tokens)
    T_q = int(T_q)
    if query_indices is not None and query_indices.numel() != T_q:
        raise ValueError("query_indices must have T_q entries")
    if padding_mask is not None:
        if padding_mask.dtype == torch.bool:
            padding_mask = padding_mask.view(torch.uint8)
        _need(padding_mask, "padding_mask", torch.uint8, 1, dev)
        if padding_mask.numel() != T_q:
            raise ValueError("padding_mask must have T_q entries")
    start = torch.empty(T_q, dtype=torch.int32, device=dev)
    clen = torch.empty(T_q, dtype=torch.int32, device=dev)
    mx = ctypes.c_int32(0)
    ne = ctypes.c_int32(0)
    _check(lib.dsa_packed_metadata_cp(_ptr(cu_seqlens), _ptr(cu_seqlens_padded), cu_seqlens.numel() - 1,
                                      int(total_key_tokens), _ptr(query_indices), _ptr(padding_mask), T_q, _ptr(start),
                                      _ptr(clen), ctypes.byref(mx), ctypes.byref(ne), _stream(dev)),
           "dsa_packed_metadata_cp")
    return start, clen, mx.value, ne.value


def dsa_indexer_topk_cp(q_idx, k_idx, head_weights, seq_start, causal_len, K: int, topk_idx=None, topk_len=None,
                        workspace=None):
    """Indexer top-k for rank-local rows against gathered global keys: row r's window is
    [seq_start[r], seq_start[r] + causal_len[r] - 1] -> (topk_idx int32 [T_q, K], topk_len int32 [T_q])."""
    lib = load_library()
    _need(q_idx, "q_idx", torch.bfloat16, 3)
    dev = q_idx.device
    _need(k_idx, "k_idx", torch.bfloat16, 2, dev)
    _need(head_weights, "head_weights", torch.float32, 2, dev)
    _need(seq_start, "seq_start", torch.int32, 1, dev)
    _need(causal_len, "causal_len", torch.int32, 1, dev)
    T, Hi, Di = q_idx.shape
    Tk = k_idx.shape[0]
    if topk_idx is None:
        topk_idx = torch.empty(T, K, dtype=torch.int32, device=dev)
    if topk_len is None:
        topk_len = torch.empty(T, dtype=torch.int32, device=dev)
    ws, wsb = _workspace("indexer", T, K, dev, workspace)
    _check(lib.dsa_indexer_topk_cp(_ptr(q_idx), _ptr(k_idx), _ptr(head_weights), _ptr(seq_start), _ptr(causal_len),
                                   T, Tk, Hi, Di, int(K), _ptr(topk_idx), _ptr(topk_len), _ptr(ws), wsb,
                                   _stream(dev)),
           "dsa_indexer_topk_cp")
    return topk_idx, topk_len


def dsa_indexer_topk(q_idx, k_idx, head_weights, seq_start, K: int, topk_idx=None, topk_len=None,
                     workspace=None, with_len: bool = True):
    """Fused indexer score + causal top-k -> (topk_idx int32 [T,K], topk_len int32 [T] or None)."""
    lib = load_library()
    _need(q_idx, "q_idx", torch.bfloat16, 3)
    dev = q_idx.device
    _need(k_idx, "k_idx", torch.bfloat16, 2, dev)
    _need(head_weights, "head_weights", torch.float32, 2, dev)
    _need(seq_start, "seq_start", torch.int32, 1, dev)
    T, Hi, Di = q_idx.shape
    Tk = k_idx.shape[0]
    if topk_idx is None:
        topk_idx = torch.empty(T, K, dtype=torch.int32, device=dev)
    if topk_len is None and with_len:
        topk_len = torch.empty(T, dtype=torch.int32, device=dev)
    ws, wsb = _workspace("indexer", T, K, dev, workspace)
    _check(lib.dsa_indexer_topk(_ptr(q_idx), _ptr(k_idx), _ptr(head_weights), _ptr(seq_start), T, Tk, Hi, Di,
                                int(K), _ptr(topk_idx), _ptr(topk_len), _ptr(ws), wsb, _stream(dev)),
           "dsa_indexer_topk")
    return topk_idx, topk_len


def dsa_indexer_topk_scored(q_idx, k_idx, head_weights, seq_start, K: int, causal_len=None, topk_idx=None,
                            topk_len=None, topk_score=None, workspace=None):
    """dsa_indexer_topk (causal_len None) or dsa_indexer_topk_cp that also returns each selected slot's fp32
    score -> (topk_idx int32 [T,K], topk_len int32 [T], topk_score fp32 [T,K], -inf after the prefix)."""
    lib = load_library()
    _need(q_idx, "q_idx", torch.bfloat16, 3)
    dev = q_idx.device
    _need(k_idx, "k_idx", torch.bfloat16, 2, dev)
    _need(head_weights, "head_weights", torch.float32, 2, dev)
    _need(seq_start, "seq_start", torch.int32, 1, dev)
    if causal_len is not None:
        _need(causal_len, "causal_len", torch.int32, 1, dev)
    T, Hi, Di = q_idx.shape
    Tk = k_idx.shape[0]
    if topk_idx is None:
        topk_idx = torch.empty(T, K, dtype=torch.int32, device=dev)
    if topk_len is None:
        topk_len = torch.empty(T, dtype=torch.int32, device=dev)
    if topk_score is None:
        topk_score = torch.empty(T, K, dtype=torch.float32, device=dev)
    _need(topk_score, "topk_score", torch.float32, 2, dev)
    ws, wsb = _workspace("indexer", T, K, dev, workspace)
    _check(lib.dsa_indexer_topk_scored(_ptr(q_idx), _ptr(k_idx), _ptr(head_weights), _ptr(seq_start),
                                       _ptr(causal_len), T, Tk, Hi, Di, int(K), _ptr(topk_idx), _ptr(topk_len),
                                       _ptr(topk_score), _ptr(ws), wsb, _stream(dev)),
           "dsa_indexer_topk_scored")
    return topk_idx, topk_len, topk_score


def dsa_indexer_topk_with_scores(q_idx, k_idx, head_weights, seq_start, K: int, score_row0: int,
                                 score_rows: int, workspace=None):
    """Diagnostic form of dsa_indexer_topk -> (topk_idx, topk_len, scores fp32 [score_rows, T_k]): the
    fp32 score of every window key of rows score_row0 .. score_row0 + score_rows - 1 (NaN elsewhere)."""
    lib = load_library()
    _need(q_idx, "q_idx", torch.bfloat16, 3)
    dev = q_idx.device
    _need(k_idx, "k_idx", torch.bfloat16, 2, dev)
    _need(head_weights, "head_weights", torch.float32, 2, dev)
    _need(seq_start, "seq_start", torch.int32, 1, dev)
    T, Hi, Di = q_idx.shape
    Tk = k_idx.shape[0]
    topk_idx = torch.empty(T, K, dtype=torch.int32, device=dev)
    topk_len = torch.empty(T, dtype=torch.int32, device=dev)
    scores = torch.full((score_rows, Tk), float("nan"), dtype=torch.float32, device=dev)
    ws, wsb = _workspace("indexer", T, K, dev, workspace)
    _check(lib.dsa_indexer_topk_with_scores(_ptr(q_idx), _ptr(k_idx), _ptr(head_weights), _ptr(seq_start), T, Tk,
                                            Hi, Di, int(K), _ptr(topk_idx), _ptr(topk_len), _ptr(scores),
                                            int(score_row0), int(score_rows), _ptr(ws), wsb, _stream(dev)),
           "dsa_indexer_topk_with_scores")
    return topk_idx, topk_len, scores


def dsa_indexer_kl(q_idx, k_idx, head_weights, topk_idx, attn_prob, coeff: float, topk_len=None, kl=None,
                   dq_idx=None, dw=None, dk_idx_accum=None, accumulate: bool = False, workspace=None,
                   topk_score=None):
    """Indexer KL auxiliary loss over each row's selected slots and its gradient -> (kl fp32 [T],
    dq_idx bf16 [T,Hi,Di], dw fp32 [T,Hi], dk_idx_accum fp32 [T_k,Di]); the gradients are those of
    coeff * sum_t kl[t].  attn_prob: fp32 [T, K], e.g. from dsa_sparse_mla_bwd(attn_prob=True).
    topk_score: fp32 [T, K] or None, the slots' indexer scores (dsa_indexer_topk_scored), read instead
    of formed again."""
    lib = load_library()
    _need(q_idx, "q_idx", torch.bfloat16, 3)
    dev = q_idx.device
    _need(k_idx, "k_idx", torch.bfloat16, 2, dev)
    _need(head_weights, "head_weights", torch.float32, 2, dev)
    _need(topk_idx, "topk_idx", torch.int32, 2, dev)
    _need(attn_prob, "attn_prob", torch.float32, 2, dev)
    if topk_len is not None:
        _need(topk_len, "topk_len", torch.int32, 1, dev)
    T, Hi, Di = q_idx.shape
    Tk = k_idx.shape[0]
    K = topk_idx.shape[1]
    if attn_prob.shape != topk_idx.shape:
        raise ValueError("attn_prob must have the shape of topk_idx")
    if topk_score is not None:
        _need(topk_score, "topk_score", torch.float32, 2, dev)
        if topk_score.shape != topk_idx.shape:
            raise ValueError("topk_score must have the shape of topk_idx")
    kl = torch.empty(T, dtype=torch.float32, device=dev) if kl is None else kl
    dq_idx = torch.empty(T, Hi, Di, dtype=torch.bfloat16, device=dev) if dq_idx is None else dq_idx
    dw = torch.empty(T, Hi, dtype=torch.float32, device=dev) if dw is None else dw
    if dk_idx_accum is None:
        if accumulate:
            raise ValueError("accumulate=True needs an existing dk_idx_accum")
        dk_idx_accum = torch.empty(Tk, Di, dtype=torch.float32, device=dev)
    for t_, n_, dt_ in ((kl, "kl", torch.float32), (dq_idx, "dq_idx", torch.bfloat16), (dw, "dw", torch.float32),
                        (dk_idx_accum, "dk_idx_accum", torch.float32)):
        _need(t_, n_, dt_, None, dev)
    if workspace is None:
        workspace = torch.empty(max(int(lib.dsa_indexer_kl_workspace_size(T, K)), 256), dtype=torch.uint8,
                                device=dev)
    _check(lib.dsa_indexer_kl(_ptr(q_idx), _ptr(k_idx), _ptr(head_weights), _ptr(topk_idx), _ptr(topk_len),
                              _ptr(attn_prob), _ptr(topk_score), T, Tk, Hi, Di, K, float(coeff), _ptr(kl), _ptr(dq_idx), _ptr(dw),
                              _ptr(dk_idx_accum), 1 if accumulate else 0, _ptr(workspace), workspace.numel(),
                              _stream(dev)),
           "dsa_indexer_kl")
    return kl, dq_idx, dw, dk_idx_accum


class KPoolMeta:
    """Pool coordinates of a packed batch (dsa_kpool_metadata): pool size, per-sequence pool
    offsets (device int32 [nseq+1]), per-token pool_start / n_pools / tail_start (device int32 [T])
    and the total number of pools."""

    def __init__(self, cu_seqlens, pool, pool_cu, pool_start, n_pools, tail_start, total_pools):
        self.cu_seqlens, self.pool, self.pool_cu = cu_seqlens, pool, pool_cu
        self.pool_start, self.n_pools, self.tail_start, self.total_pools = pool_start, n_pools, tail_start, total_pools

    @property
    def num_seqs(self) -> int:
        return self.cu_seqlens.numel() - 1

    @property
    def total_tokens(self) -> int:
        return self.pool_start.numel()


def dsa_kpool_metadata(cu_seqlens: torch.Tensor, total_tokens: int, pool: int = 4) -> KPoolMeta:
    """k-pool coordinates: pools of `pool` consecutive tokens of each packed sequence (GLM-5.3-Flash)."""
    lib = load_library()
    _need(cu_seqlens, "cu_seqlens", torch.int32, 1)
    dev = cu_seqlens.device
    T = int(total_tokens)
    pool_cu = torch.empty(cu_seqlens.numel(), dtype=torch.int32, device=dev)
    ps = torch.empty(T, dtype=torch.int32, device=dev)
    npl = torch.empty(T, dtype=torch.int32, device=dev)
    ts = torch.empty(T, dtype=torch.int32, device=dev)
    total = ctypes.c_int32(0)
    _check(lib.dsa_kpool_metadata(_ptr(cu_seqlens), cu_seqlens.numel() - 1, T, int(pool), _ptr(pool_cu), _ptr(ps),
                                  _ptr(npl), _ptr(ts), ctypes.byref(total), _stream(dev)), "dsa_kpool_metadata")
    return KPoolMeta(cu_seqlens, int(pool), pool_cu, ps, npl, ts, total.value)


def dsa_kpool_pool(x: torch.Tensor, meta: KPoolMeta, out=None):
    """Pooled rows of x (bf16 [T, D]) -> bf16 [total_pools, D]: the mean of each pool's token rows."""
    lib = load_library()
    _need(x, "x", torch.bfloat16, 2)
    dev = x.device
    T, D = x.shape
    if out is None:
        out = torch.empty(meta.total_pools, D, dtype=torch.bfloat16, device=dev)
    _need(out, "out", torch.bfloat16, 2, dev)
    _check(lib.dsa_kpool_pool(_ptr(x), T, D, _ptr(meta.cu_seqlens), _ptr(meta.pool_cu), meta.num_seqs, meta.pool,
                              meta.total_pools, _ptr(out), _stream(dev)), "dsa_kpool_pool")
    return out


def dsa_kpool_topk(q_idx, k_pool, head_weights, meta: KPoolMeta, K: int = 2048, topk_idx=None, topk_len=None,
                   workspace=None):
    """k-pool selection -> (topk_idx int32 [T, K + pool - 1], topk_len int32 [T]): the K best complete pools
    of each row's sequence (rows 0 .. total_pools - 1), then its incomplete pool's tokens (rows
    total_pools + s), ascending, -1 suffix."""
    lib = load_library()
    _need(q_idx, "q_idx", torch.bfloat16, 3)
    dev = q_idx.device
    _need(k_pool, "k_pool", torch.bfloat16, 2, dev)
    _need(head_weights, "head_weights", torch.float32, 2, dev)
    T, Hi, Di = q_idx.shape
    W = int(K) + meta.pool - 1
    if topk_idx is None:
        topk_idx = torch.empty(T, W, dtype=torch.int32, device=dev)
    if topk_len is None:
        topk_len = torch.empty(T, dtype=torch.int32, device=dev)
    need = int(lib.dsa_kpool_topk_workspace_size(T, int(K)))
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    _check(lib.dsa_kpool_topk(_ptr(q_idx), _ptr(k_pool), _ptr(head_weights), _ptr(meta.pool_start),
                              _ptr(meta.n_pools), _ptr(meta.tail_start), T, meta.total_pools, Hi, Di, int(K),
                              meta.pool, _ptr(topk_idx), _ptr(topk_len), _ptr(workspace), workspace.numel(),
                              _stream(dev)), "dsa_kpool_topk")
    return topk_idx, topk_len


def dsa_kpool_unpool_grad(dcat: torch.Tensor, meta: KPoolMeta, dx=None):
    """Token key gradient fp32 [T, D] from the gradient of the attended rows fp32 [total_pools + T, D]."""
    lib = load_library()
    _need(dcat, "dcat", torch.float32, 2)
    dev = dcat.device
    D = dcat.shape[1]
    T = meta.total_tokens
    if dx is None:
        dx = torch.empty(T, D, dtype=torch.float32, device=dev)
    _need(dx, "dx", torch.float32, 2, dev)
    _check(lib.dsa_kpool_unpool_grad(_ptr(dcat), T, D, _ptr(meta.cu_seqlens), _ptr(meta.pool_cu), meta.num_seqs,
                                     meta.pool, meta.total_pools, _ptr(dx), _stream(dev)), "dsa_kpool_unpool_grad")
    return dx


def dsa_sparse_mla_fwd(q, kv, topk_idx, softmax_scale: float, topk_len=None, out=None, lse=None,
                       workspace=None, Dv: int = 512, out_lo=None, attn_sink=None):
    """Sparse MLA forward -> (out bf16 [T,H,Dv], lse fp32 [T,H]), or (out, lse, out_lo) when
    out_lo is a tensor or True (the bf16 rounding residual of out, for an exact backward D).
    kv may be [T_k, Dqk] or [T_k, 1, Dqk]; attn_sink: fp32 [H] per-head sink logits or None."""
    lib = load_library()
    _need(q, "q", torch.bfloat16, 3)
    dev = q.device
    if kv.dim() == 3:
        kv = kv.reshape(kv.shape[0], kv.shape[2])
    _need(kv, "kv", torch.bfloat16, 2, dev)
    if topk_idx.dim() == 3:
        topk_idx = topk_idx.reshape(topk_idx.shape[0], topk_idx.shape[2])
    _need(topk_idx, "topk_idx", torch.int32, 2, dev)
    if topk_len is not None:
        _need(topk_len, "topk_len", torch.int32, 1, dev)
    T, H, Dqk = q.shape
    K = topk_idx.shape[1]
    if attn_sink is not None:
        _need(attn_sink, "attn_sink", torch.float32, 1, dev)
        if attn_sink.numel() != H:
            raise ValueError(f"attn_sink must have H = {H} entries")
    if out is None:
        out = torch.empty(T, H, Dv, dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty(T, H, dtype=torch.float32, device=dev)
    want_lo = out_lo is not None and out_lo is not False
    if out_lo is True:
        out_lo = torch.empty(T, H, Dv, dtype=torch.bfloat16, device=dev)
    lo = out_lo if want_lo else None
    ws, wsb = _workspace("fwd", T, H, dev, workspace)
    _check(lib.dsa_sparse_mla_fwd(_ptr(q), _ptr(kv), _ptr(topk_idx), _ptr(topk_len), T, kv.shape[0], H, Dqk, Dv,
                                  K, float(softmax_scale), _ptr(attn_sink), _ptr(out), _ptr(lo), _ptr(lse), _ptr(ws),
                                  wsb, _stream(dev)),
           "dsa_sparse_mla_fwd")
    return (out, lse, lo) if want_lo else (out, lse)


def dsa_sparse_mla_bwd(q, kv, topk_idx, softmax_scale: float, out, lse, dout, topk_len=None, dq=None,
                       dkv_accum=None, accumulate: bool = False, dkv_bf16=None, workspace=None, out_lo=None,
                       attn_sink=None, d_sink=None, attn_prob=None):
    """Sparse MLA backward -> (dq bf16 [T,H,Dqk], dkv_accum fp32 [T_k,Dqk], dkv_bf16 or None), and
    d_sink fp32 [H] as a fourth result when attn_sink is given (d_sink: an existing tensor to fill,
    or to add to with accumulate=True).
    out_lo: the forward's residual of O (D then uses the fp32 output).
    attn_prob: fp32 [T, K] tensor (or True to allocate one) that receives the head-averaged
    attention probability of every slot; it is then returned as the last result."""
    lib = load_library()
    _need(q, "q", torch.bfloat16, 3)
    dev = q.device
    if kv.dim() == 3:
        kv = kv.reshape(kv.shape[0], kv.shape[2])
    _need(kv, "kv", torch.bfloat16, 2, dev)
    if topk_idx.dim() == 3:
        topk_idx = topk_idx.reshape(topk_idx.shape[0], topk_idx.shape[2])
    _need(topk_idx, "topk_idx", torch.int32, 2, dev)
    _need(out, "out", torch.bfloat16, 3, dev)
    _need(lse, "lse", torch.float32, 2, dev)
    _need(dout, "dout", torch.bfloat16, 3, dev)
    if topk_len is not None:
        _need(topk_len, "topk_len", torch.int32, 1, dev)
    if out_lo is not None:
        _need(out_lo, "out_lo", torch.bfloat16, 3, dev)
    T, H, Dqk = q.shape
    Dv = out.shape[2]
    K = topk_idx.shape[1]
    Tk = kv.shape[0]
    if dq is None:
        dq = torch.empty(T, H, Dqk, dtype=torch.bfloat16, device=dev)
    if dkv_accum is None:
        if accumulate:
            raise ValueError("accumulate=True needs an existing dkv_accum")
        dkv_accum = torch.empty(Tk, Dqk, dtype=torch.float32, device=dev)
    _need(dkv_accum, "dkv_accum", torch.float32, 2, dev)
    if attn_sink is not None:
        _need(attn_sink, "attn_sink", torch.float32, 1, dev)
        if d_sink is None:
            if accumulate:
                raise ValueError("accumulate=True needs an existing d_sink")
            d_sink = torch.empty(H, dtype=torch.float32, device=dev)
        _need(d_sink, "d_sink", torch.float32, 1, dev)
    want_prob = attn_prob is not None and attn_prob is not False
    if attn_prob is True:
        attn_prob = torch.empty(T, K, dtype=torch.float32, device=dev)
    if want_prob:
        _need(attn_prob, "attn_prob", torch.float32, 2, dev)
    ws, wsb = _workspace("bwd", T, H, dev, workspace, K)
    _check(lib.dsa_sparse_mla_bwd(_ptr(q), _ptr(kv), _ptr(topk_idx), _ptr(topk_len), T, Tk, H, Dqk, Dv, K,
                                  float(softmax_scale), _ptr(attn_sink), _ptr(out), _ptr(out_lo), _ptr(lse),
                                  _ptr(dout), _ptr(dq), _ptr(dkv_accum), _ptr(d_sink),
                                  _ptr(attn_prob if want_prob else None), 1 if accumulate else 0, _ptr(dkv_bf16),
                                  _ptr(ws), wsb, _stream(dev)),
           "dsa_sparse_mla_bwd")
    res = (dq, dkv_accum, dkv_bf16) if attn_sink is None else (dq, dkv_accum, dkv_bf16, d_sink)
    return res + (attn_prob,) if want_prob else res


def dsa_sparse_mla_bwd_noalloc(q, kv, topk_idx, softmax_scale: float, out, lse, dout, topk_len=None, dq=None,
                               dkv_accum=None, accumulate: bool = False, dkv_bf16=None, out_lo=None):
    """dsa_sparse_mla_bwd with the library's built-in scratch instead of a workspace (for callers
    that cannot allocate device memory; see include/dsa.h) -> (dq, dkv_accum, dkv_bf16).
    Output tensors the caller does not pass are allocated here by torch, as in the other calls."""
    lib = load_library()
    _need(q, "q", torch.bfloat16, 3)
    dev = q.device
    if kv.dim() == 3:
        kv = kv.reshape(kv.shape[0], kv.shape[2])
    _need(kv, "kv", torch.bfloat16, 2, dev)
    _need(topk_idx, "topk_idx", torch.int32, 2, dev)
    _need(out, "out", torch.bfloat16, 3, dev)
    _need(lse, "lse", torch.float32, 2, dev)
    _need(dout, "dout", torch.bfloat16, 3, dev)
    if topk_len is not None:
        _need(topk_len, "topk_len", torch.int32, 1, dev)
    if out_lo is not None:
        _need(out_lo, "out_lo", torch.bfloat16, 3, dev)
    T, H, Dqk = q.shape
    Tk = kv.shape[0]
    if dq is None:
        dq = torch.empty(T, H, Dqk, dtype=torch.bfloat16, device=dev)
    if dkv_accum is None:
        if accumulate:
            raise ValueError("accumulate=True needs an existing dkv_accum")
        dkv_accum = torch.empty(Tk, Dqk, dtype=torch.float32, device=dev)
    _need(dkv_accum, "dkv_accum", torch.float32, 2, dev)
    _check(lib.dsa_sparse_mla_bwd_noalloc(_ptr(q), _ptr(kv), _ptr(topk_idx), _ptr(topk_len), T, Tk, H, Dqk,
                                          out.shape[2], topk_idx.shape[1], float(softmax_scale), None, _ptr(out),
                                          _ptr(out_lo), _ptr(lse), _ptr(dout), _ptr(dq), _ptr(dkv_accum), None, None,
                                          1 if accumulate else 0, _ptr(dkv_bf16), _stream(dev)),
           "dsa_sparse_mla_bwd_noalloc")
    return dq, dkv_accum, dkv_bf16


def dsa_sparse_mla_bwd_noalloc_read_status(device=None) -> int:
    """Synchronise the current stream, read and clear the no-alloc backward's device error word."""
    lib = load_library()
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    st = ctypes.c_int32(0)
    _check(lib.dsa_sparse_mla_bwd_noalloc_read_status(_stream(dev), ctypes.byref(st)),
           "dsa_sparse_mla_bwd_noalloc_read_status")
    return st.value


def dsa_set_wait_limit_cycles(cycles: int) -> int:
    """Cycle limit of the kernels' bounded waits for later launches (negative: the default, 2^31);
    returns the previous limit."""
    return int(load_library().dsa_set_wait_limit_cycles(int(cycles)))


def dsa_read_device_status(workspace: torch.Tensor) -> int:
    """Synchronise the current stream, read and clear the device error word of ``workspace``."""
    lib = load_library()
    st = ctypes.c_int32(0)
    _check(lib.dsa_read_device_status(_ptr(workspace), _stream(workspace.device), ctypes.byref(st)),
           "dsa_read_device_status")
    return st.value
