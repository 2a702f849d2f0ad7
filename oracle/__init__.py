"""fp64 CPU oracle of the DSA hot path -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never calls it, and it
shares no code with the CUDA library: the arithmetic lives in ``dsa_oracle.c``
(plain C, fp64, OpenMP), this module only marshals numpy arrays.

Every function takes tensors/arrays that hold the exact values given to the GPU
(bf16 or fp32) and widens them to float64 before the call.

Pins (what checks this oracle against something other than itself) live in
``tests/test_oracle_pins.py``; every oracle function is pinned, none is
"parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dsa_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libdsa_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile dsa_oracle.c into a shared library with gcc (-O2, OpenMP)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", _SRC, "-o", tmp, "-lm"]
        )
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            I = ctypes.c_int
            lib.oracle_packed_metadata.argtypes = [P, I, I, P, P, P, P]
            lib.oracle_packed_metadata.restype = I
            lib.oracle_packed_metadata_cp.argtypes = [P, P, I, I, P, P, I, P, P, P, P]
            lib.oracle_packed_metadata_cp.restype = I
            lib.oracle_indexer_scores.argtypes = [P, P, P, I, I, P, P, ctypes.c_int64, P, P]
            lib.oracle_indexer_scores.restype = None
            lib.oracle_indexer_topk.argtypes = [P, P, P, P, P, I, I, I, I, P, P, P]
            lib.oracle_indexer_topk.restype = None
            lib.oracle_indexer_topk_window.argtypes = [P, P, P, P, P, I, I, I, I, P, P, P]
            lib.oracle_indexer_topk_window.restype = None
            lib.oracle_sparse_mla_fwd.argtypes = [P, P, P, P, I, I, I, I, I, I, ctypes.c_double, P, P, P]
            lib.oracle_sparse_mla_fwd.restype = None
            lib.oracle_sparse_mla_bwd.argtypes = [P, P, P, P, I, I, I, I, I, I, ctypes.c_double, P, P, P, P, P, P]
            lib.oracle_sparse_mla_bwd.restype = None
            lib.oracle_attn_slot_prob.argtypes = [P, P, P, P, I, I, I, I, I, I, ctypes.c_double, P, P]
            lib.oracle_attn_slot_prob.restype = None
            lib.oracle_indexer_kl.argtypes = [P, P, P, P, P, P, I, I, I, I, I, ctypes.c_double, P, P, P, P]
            lib.oracle_indexer_kl.restype = None
            lib.oracle_kpool_metadata.argtypes = [P, I, I, I, P, P, P, P]
            lib.oracle_kpool_metadata.restype = I
            lib.oracle_kpool_pool.argtypes = [P, I, P, I, I, I, P]
            lib.oracle_kpool_pool.restype = None
            lib.oracle_kpool_compose_row.argtypes = [P, I, I, I, I, I, P]
            lib.oracle_kpool_compose_row.restype = I
            lib.oracle_kpool_unpool_grad.argtypes = [P, I, P, I, I, I, P]
            lib.oracle_kpool_unpool_grad.restype = None
            _lib = lib
    return _lib


def _f64(x) -> np.ndarray:
    """Widen a torch tensor (any float dtype, any device) or array to C-contiguous float64."""
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(x, dtype=np.float64)


def _i32(x) -> np.ndarray:
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").numpy()
    return np.ascontiguousarray(x, dtype=np.int32)


def _i64(x) -> np.ndarray:
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").numpy()
    return np.ascontiguousarray(x, dtype=np.int64)


def _p(a: np.ndarray | None):
    return None if a is None else a.ctypes.data


def packed_metadata(cu_seqlens, total_tokens: int):
    """cu_seqlens [nseq+1] -> (seq_start[T], causal_len[T], max_seqlen, all_rows_nonempty)."""
    cu = _i32(cu_seqlens)
    T = int(total_tokens)
    start = np.zeros(max(T, 1), np.int32)
    clen = np.zeros(max(T, 1), np.int32)
    mx = np.zeros(1, np.int32)
    ne = np.zeros(1, np.int32)
    rc = _load().oracle_packed_metadata(_p(cu), len(cu) - 1, T, _p(start), _p(clen), _p(mx), _p(ne))
    if rc != 0:
        raise ValueError("cu_seqlens must be a non-decreasing cover of [0, T]")
    return start[:T], clen[:T], int(mx[0]), int(ne[0])


def packed_metadata_cp(cu_seqlens, total_key_tokens: int, query_indices=None, cu_seqlens_padded=None,
                       padding_mask=None, T_q: int | None = None):
    """Context-parallel form: local query rows (global padded coordinates `query_indices`,
    identity when absent) against gathered global keys.  Returns (seq_start[T_q],
    causal_len[T_q], max_seqlen, all_rows_nonempty); raises ValueError on invalid input."""
    cu = _i32(cu_seqlens)
    cp = None if cu_seqlens_padded is None else _i32(cu_seqlens_padded)
    qi = None if query_indices is None else _i32(query_indices)
    pm = None if padding_mask is None else np.ascontiguousarray(
        padding_mask.detach().to("cpu").numpy() if hasattr(padding_mask, "detach") else padding_mask, dtype=np.uint8)
    if T_q is None:
        T_q = len(qi) if qi is not None else int(total_key_tokens)
    n = int(T_q)
    start = np.zeros(max(n, 1), np.int32)
    clen = np.zeros(max(n, 1), np.int32)
    mx = np.zeros(1, np.int32)
    ne = np.zeros(1, np.int32)
    rc = _load().oracle_packed_metadata_cp(_p(cu), _p(cp), len(cu) - 1, int(total_key_tokens), _p(qi), _p(pm), n,
                                           _p(start), _p(clen), _p(mx), _p(ne))
    if rc != 0:
        raise ValueError("invalid sequence boundaries or query coordinates")
    return start[:n], clen[:n], int(mx[0]), int(ne[0])


def indexer_scores(q_idx_rows, k_idx, w_rows, pair_row, pair_key, with_magnitude: bool = False):
    """fp64 indexer scores for explicit pairs (pair_row indexes q_idx_rows/w_rows)."""
    q = _f64(q_idx_rows)
    k = _f64(k_idx)
    w = _f64(w_rows)
    Hi, Di = q.shape[1], q.shape[2]
    pr, pk = _i64(pair_row), _i64(pair_key)
    out = np.zeros(len(pr), np.float64)
    mag = np.zeros(len(pr), np.float64) if with_magnitude else None
    _load().oracle_indexer_scores(_p(q), _p(k), _p(w), Hi, Di, _p(pr), _p(pk), len(pr), _p(out), _p(mag))
    return (out, mag) if with_magnitude else out


def indexer_topk(q_idx_rows, k_idx, w_rows, seq_start, row_t, K: int):
    """Causal top-k for the given rows.

    q_idx_rows [n, Hi, Di] and w_rows [n, Hi] hold only the requested rows,
    row_t [n] their global token ids, seq_start [T] the per-token sequence
    start.  Returns (idx [n, K] int32 ascending + -1 suffix, len [n], kth score [n]).
    """
    q = _f64(q_idx_rows)
    k = _f64(k_idx)
    w = _f64(w_rows)
    n, Hi, Di = q.shape
    st = _i32(seq_start)
    rt = _i64(row_t)
    idx = np.zeros((n, K), np.int32)
    ln = np.zeros(n, np.int32)
    kth = np.zeros(n, np.float64)
    _load().oracle_indexer_topk(_p(q), _p(k), _p(w), _p(st), _p(rt), n, Hi, Di, int(K), _p(idx), _p(ln), _p(kth))
    return idx, ln, kth


def indexer_topk_window(q_idx_rows, k_idx, w_rows, win_start, win_len, K: int):
    """Top-k of each given row over its explicit key window [win_start, win_start + win_len - 1]
    (none when win_len = 0).  Returns (idx [n, K], len [n], kth score [n]) as indexer_topk."""
    q = _f64(q_idx_rows)
    k = _f64(k_idx)
    w = _f64(w_rows)
    n, Hi, Di = q.shape
    ws, wl = _i32(win_start), _i32(win_len)
    idx = np.zeros((n, K), np.int32)
    ln = np.zeros(n, np.int32)
    kth = np.zeros(n, np.float64)
    _load().oracle_indexer_topk_window(_p(q), _p(k), _p(w), _p(ws), _p(wl), n, Hi, Di, int(K), _p(idx), _p(ln),
                                       _p(kth))
    return idx, ln, kth


def sparse_mla_fwd(q_rows, kv, idx_rows, scale: float, Dv: int = 512, len_rows=None, sink=None):
    """Sparse MLA forward for the given query rows -> (out [n,H,Dv], lse [n,H]) in fp64.
    sink: per-head sink logits [H] (one more logit per row with no value row), or None."""
    q = _f64(q_rows)
    kvf = _f64(kv).reshape(kv.shape[0], -1)
    idx = _i32(idx_rows)
    ln = None if len_rows is None else _i32(len_rows)
    n, H, Dqk = q.shape
    K = idx.shape[1]
    out = np.zeros((n, H, Dv), np.float64)
    lse = np.zeros((n, H), np.float64)
    sk = None if sink is None else _f64(sink).reshape(H)
    _load().oracle_sparse_mla_fwd(_p(q), _p(kvf), _p(idx), _p(ln), n, kvf.shape[0], H, Dqk, Dv, K,
                                  float(scale), _p(sk), _p(out), _p(lse))
    return out, lse


def sparse_mla_bwd(q_rows, kv, idx_rows, dout_rows, scale: float, Dv: int = 512, len_rows=None, dkv=None,
                   with_dq_magnitude: bool = False, sink=None, d_sink=None):
    """Sparse MLA backward for the given rows -> (dq [n,H,Dqk], dkv [Tk,Dqk]) in fp64, and with
    with_dq_magnitude also dq_mag [n,H,Dqk] = scale * sum_j |dS_j| |kv[idx_j, :]| (the scale of
    the error of a dq formed from dS rounded to a 16-bit float).  With a sink [H], d_sink [H] (fp64,
    created when None) receives -sum_t P_sink D and is returned after dkv.

    dkv accumulates the contributions of exactly these rows (pass an existing
    array to keep adding, as query chunks do)."""
    q = _f64(q_rows)
    kvf = _f64(kv).reshape(kv.shape[0], -1)
    idx = _i32(idx_rows)
    ln = None if len_rows is None else _i32(len_rows)
    do = _f64(dout_rows)
    n, H, Dqk = q.shape
    K = idx.shape[1]
    dq = np.zeros((n, H, Dqk), np.float64)
    mag = np.zeros((n, H, Dqk), np.float64) if with_dq_magnitude else None
    sk = None if sink is None else _f64(sink).reshape(H)
    if sk is not None and d_sink is None:
        d_sink = np.zeros(H, np.float64)
    if dkv is None:
        dkv = np.zeros((kvf.shape[0], Dqk), np.float64)
    assert dkv.dtype == np.float64 and dkv.flags.c_contiguous
    _load().oracle_sparse_mla_bwd(_p(q), _p(kvf), _p(idx), _p(ln), n, kvf.shape[0], H, Dqk, Dv, K,
                                  float(scale), _p(sk), _p(do), _p(dq), _p(dkv), _p(None if sk is None else d_sink),
                                  _p(mag))
    res = (dq, dkv) + ((d_sink,) if sk is not None else ()) + ((mag,) if with_dq_magnitude else ())
    return res


def attn_slot_prob(q_rows, kv, idx_rows, scale: float, Dv: int = 512, len_rows=None, sink=None):
    """Head-averaged sparse-MLA softmax weight of every slot of the given rows -> prob [n, K] (fp64)."""
    q = _f64(q_rows)
    kvf = _f64(kv).reshape(kv.shape[0], -1)
    idx = _i32(idx_rows)
    ln = None if len_rows is None else _i32(len_rows)
    n, H, Dqk = q.shape
    K = idx.shape[1]
    sk = None if sink is None else _f64(sink).reshape(H)
    prob = np.zeros((n, K), np.float64)
    _load().oracle_attn_slot_prob(_p(q), _p(kvf), _p(idx), _p(ln), n, kvf.shape[0], H, Dqk, Dv, K, float(scale),
                                  _p(sk), _p(prob))
    return prob


def indexer_kl(q_idx_rows, k_idx, w_rows, idx_rows, prob_rows, coeff: float, len_rows=None, dk=None):
    """Indexer KL loss of the given rows over their selected slots -> (kl [n], dq_idx [n,Hi,Di], dw [n,Hi],
    dk [Tk,Di]) in fp64; prob_rows [n, K] is the attention's slot probability (normalised per row here).
    dk accumulates the contributions of exactly these rows (pass an existing array to keep adding)."""
    q = _f64(q_idx_rows)
    k = _f64(k_idx)
    w = _f64(w_rows)
    idx = _i32(idx_rows)
    pr = _f64(prob_rows)
    ln = None if len_rows is None else _i32(len_rows)
    n, Hi, Di = q.shape
    K = idx.shape[1]
    kl = np.zeros(n, np.float64)
    dq = np.zeros((n, Hi, Di), np.float64)
    dw = np.zeros((n, Hi), np.float64)
    if dk is None:
        dk = np.zeros((k.shape[0], Di), np.float64)
    assert dk.dtype == np.float64 and dk.flags.c_contiguous
    _load().oracle_indexer_kl(_p(q), _p(k), _p(w), _p(idx), _p(ln), _p(pr), n, k.shape[0], Hi, Di, K, float(coeff),
                              _p(kl), _p(dq), _p(dw), _p(dk))
    return kl, dq, dw, dk


# ---------------------------------------------------------------------------
# k-pool selection (GLM-5.3-Flash): pools of P consecutive tokens of a packed
# sequence, the query's top-K complete pools by the indexer score against the
# pooled keys, then the tokens of its incomplete pool; attention over
# [pooled rows; token rows].  The readings are written in dsa_oracle.c.
# ---------------------------------------------------------------------------
def kpool_metadata(cu_seqlens, total_tokens: int, P: int):
    """Returns (pool_cu [nseq+1], pool_start [T], n_pools [T], tail_start [T], total_pools)."""
    cu = _i32(cu_seqlens)
    T, nseq = int(total_tokens), len(cu) - 1
    pool_cu = np.zeros(nseq + 1, np.int32)
    ps = np.zeros(max(T, 1), np.int32)
    npl = np.zeros(max(T, 1), np.int32)
    ts = np.zeros(max(T, 1), np.int32)
    total = _load().oracle_kpool_metadata(_p(cu), nseq, T, int(P), _p(pool_cu), _p(ps), _p(npl), _p(ts))
    if total < 0:
        raise ValueError("cu_seqlens must be a non-decreasing cover of [0, T] and P >= 1")
    return pool_cu, ps[:T], npl[:T], ts[:T], int(total)


def kpool_pool(x, cu_seqlens, P: int, round_to_bf16: bool = True):
    """Pooled rows [total_pools, D] (fp64 values; bf16-rounded means unless round_to_bf16 is False)."""
    xv = _f64(x)
    cu = _i32(cu_seqlens)
    nseq = len(cu) - 1
    total = sum((int(cu[i + 1]) - int(cu[i])) // int(P) for i in range(nseq))
    D = xv.shape[1]
    out = np.zeros((max(total, 1), D), np.float64)
    _load().oracle_kpool_pool(_p(xv), D, _p(cu), nseq, int(P), 1 if round_to_bf16 else 0, _p(out))
    return out[:total]


def kpool_topk(q_idx_rows, k_pool, w_rows, row_t, pool_start_rows, n_pools_rows, tail_start_rows,
               total_pools: int, K: int, P: int):
    """Selection of the given rows: the K best complete pools (window [pool_start, pool_start + n_pools - 1]
    of the pooled keys), then the tail tokens as rows total_pools + s.  Returns (idx [n, K + P - 1]
    ascending with -1 suffix, len [n], the K-th best pool score [n])."""
    pidx, plen, kth = indexer_topk_window(q_idx_rows, k_pool, w_rows, pool_start_rows, n_pools_rows, K)
    lib = _load()
    n = pidx.shape[0]
    W = int(K) + int(P) - 1
    out = np.zeros((n, W), np.int32)
    ln = np.zeros(n, np.int32)
    rt, ts = _i64(row_t), _i32(tail_start_rows)
    for r in range(n):
        row = np.ascontiguousarray(pidx[r])
        o = np.zeros(W, np.int32)
        ln[r] = lib.oracle_kpool_compose_row(_p(row), int(plen[r]), int(ts[r]), int(rt[r]), int(total_pools), W, _p(o))
        out[r] = o
    return out, ln, kth


def kpool_unpool_grad(dcat, cu_seqlens, P: int, total_pools: int):
    """Token key gradient [T, D] from the gradient of the attended rows [total_pools + T, D]."""
    d = _f64(dcat)
    cu = _i32(cu_seqlens)
    T = int(cu[-1])
    D = d.shape[1]
    out = np.zeros((max(T, 1), D), np.float64)
    _load().oracle_kpool_unpool_grad(_p(d), D, _p(cu), len(cu) - 1, int(P), int(total_pools), _p(out))
    return out[:T]
