"""Indexer score + causal top-k: CUDA path (through the C ABI) vs the fp64 oracle.

The GPU scores in fp32 (bf16 products, fp32 sums); the oracle in fp64.  Index
sets must be equal except where two keys' scores are within the rounding
bound of an fp32 evaluation: an index may differ only if its fp64 score and
the oracle's n-th best score are within eps_s + eps_kth, with
eps = GAMMA * sum_h |w| sum_d |q k| (GAMMA generous for ~200-term fp32 sums).
Structure (ascending prefix, -1 suffix, lengths) must match exactly.
"""
import numpy as np
import pytest
import torch

import oracle
import sparse_attention_mla_gb300 as dsa
from sparse_attention_mla_gb300 import synth

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
GAMMA = 200 * 2.0 ** -24


def oracle_start(cu, T, gpu_start=None):
    """The oracle's own window starts for cu_seqlens; the GPU's metadata, when given, must equal them
    exactly (it is checked here, never handed to the oracle)."""
    st = oracle.packed_metadata(np.asarray(cu.cpu() if torch.is_tensor(cu) else cu, np.int32), T)[0]
    if gpu_start is not None:
        assert np.array_equal(gpu_start.cpu().numpy(), st[:T]), "seq_start differs from the oracle's"
    return st


def run_gpu(q_idx, k_idx, w, cu, K):
    T = q_idx.shape[0]
    start, _, _, _ = dsa.dsa_packed_metadata(cu.to(DEV), T)
    ws = torch.zeros(4096, dtype=torch.uint8, device=DEV)
    idx, ln = dsa.dsa_indexer_topk(q_idx.to(DEV), k_idx.to(DEV), w.to(DEV), start, K, workspace=ws)
    assert dsa.dsa_read_device_status(ws) == 0
    return idx.cpu().numpy(), ln.cpu().numpy(), oracle_start(cu, T, start)


def check_rows(gidx, glen, q_idx, k_idx, w, start, rows, K, ref_out=None):
    """The GPU rows against the oracle's own top-k of the same rows (lengths, order and -1 suffix
    exact; sets equal but for keys inside the fp32 tie band).  Returns the number of swapped pairs;
    with a dict ref_out, also hands back the oracle's selection of the rows (keys "idx", "len")."""
    ref_idx, ref_len, kth = oracle.indexer_topk(q_idx[rows], k_idx, w[rows], start, rows, K)
    if ref_out is not None:
        ref_out["idx"], ref_out["len"] = ref_idx, ref_len
    swaps = 0
    for r, t in enumerate(rows):
        n = int(ref_len[r])
        assert glen[t] == n, (t, glen[t], n)
        g = gidx[t]
        assert np.all(g[n:] == -1), t
        sel = g[:n]
        assert np.all(np.diff(sel) > 0), f"row {t} not strictly ascending"
        assert sel.min(initial=start[t]) >= start[t] and sel.max(initial=t) <= t, t
        diff = sorted(set(sel.tolist()) ^ set(ref_idx[r, :n].tolist()))
        if diff:
            swaps += len(diff) // 2
            qt, wt = q_idx[[t]], w[[t]]  # this row only
            sc, mag = oracle.indexer_scores(qt, k_idx, wt, np.zeros(len(diff), np.int64), np.array(diff),
                                            with_magnitude=True)
            # magnitude of the n-th best key's score (the lowest-scoring key the oracle selects)
            sel_ref = np.asarray(ref_idx[r, :n])
            kth_sc, kth_mag = oracle.indexer_scores(qt, k_idx, wt, np.zeros(n, np.int64), sel_ref,
                                                    with_magnitude=True)
            j = int(np.argmin(kth_sc))
            for d in range(len(diff)):
                assert abs(sc[d] - kth[r]) <= GAMMA * (mag[d] + kth_mag[j]), \
                    f"row {t}: key {diff[d]} differs outside the fp32 tie band"
    return swaps


def test_indexer_single_sequence_small():
    T, K = 300, 64
    x = synth.indexer_inputs(T, 64, 128, seed=0)
    cu = torch.tensor([0, T], dtype=torch.int32)
    gidx, glen, start = run_gpu(x["q_idx"], x["k_idx"], x["w"], cu, K)
    swaps = check_rows(gidx, glen, x["q_idx"], x["k_idx"], x["w"], start, np.arange(T), K)
    assert swaps <= 2


def test_indexer_packed_thd_and_short_windows():
    T, K = 600, 200
    x = synth.indexer_inputs(T, 64, 128, seed=1)
    cu = torch.tensor([0, 100, 350, 353, 600], dtype=torch.int32)
    gidx, glen, start = run_gpu(x["q_idx"], x["k_idx"], x["w"], cu, K)
    check_rows(gidx, glen, x["q_idx"], x["k_idx"], x["w"], start, np.arange(T), K)


def test_indexer_long_windows_trigger_compaction():
    # windows up to 5000 keys with K = 2048: the candidate buffer fills and is compacted
    T, K = 5000, 2048
    x = synth.indexer_inputs(T, 64, 128, seed=2)
    cu = torch.tensor([0, T], dtype=torch.int32)
    gidx, glen, start = run_gpu(x["q_idx"], x["k_idx"], x["w"], cu, K)
    rows = np.concatenate([np.arange(0, 8), np.arange(2040, 2060), np.arange(2900, 2910), np.arange(4980, 5000)])
    check_rows(gidx, glen, x["q_idx"], x["k_idx"], x["w"], start, rows, K)


def test_indexer_fewer_heads_and_small_k():
    T, K = 257, 5
    x = synth.indexer_inputs(T, 16, 128, seed=3)
    cu = torch.tensor([0, 130, T], dtype=torch.int32)
    gidx, glen, start = run_gpu(x["q_idx"], x["k_idx"], x["w"], cu, K)
    check_rows(gidx, glen, x["q_idx"], x["k_idx"], x["w"], start, np.arange(T), K)


def test_indexer_all_ties_take_lowest_indices():
    T, K = 700, 300
    x = synth.indexer_inputs(T, 64, 128, seed=4)
    w = torch.zeros_like(x["w"])
    cu = torch.tensor([0, 450, T], dtype=torch.int32)
    gidx, glen, start = run_gpu(x["q_idx"], x["k_idx"], w, cu, K)
    for t in range(T):
        n = min(K, t - start[t] + 1)
        assert glen[t] == n
        assert gidx[t, :n].tolist() == list(range(start[t], start[t] + n)), t
        assert np.all(gidx[t, n:] == -1)


def test_indexer_increasing_scores_pick_window_end():
    T, K = 200, 16
    k_idx = torch.zeros(T, 128)
    k_idx[:, 0] = torch.arange(1, T + 1, dtype=torch.float32)  # exact in bf16 up to 256
    q_idx = torch.zeros(T, 64, 128)
    q_idx[:, :, 0] = 1.0
    w = torch.full((T, 64), 0.125)
    cu = torch.tensor([0, T], dtype=torch.int32)
    gidx, glen, _ = run_gpu(q_idx.bfloat16(), k_idx.bfloat16(), w, cu, K)
    for t in range(T):
        n = min(K, t + 1)
        assert gidx[t, :n].tolist() == list(range(t - n + 1, t + 1))


def _exact_topk(scores_row, lo, hi, K):
    """The selection rule on given fp32 values: score descending, ties to the lower index; ascending output."""
    keys = np.arange(lo, hi + 1)
    sc = scores_row[lo:hi + 1].astype(np.float64)  # fp32 values, widened exactly
    order = np.lexsort((keys, -sc))
    return np.sort(keys[order[:min(K, len(keys))]])


@pytest.mark.parametrize("T,K,cut,row0,nrows", [(700, 200, [0, 100, 350, 353, 700], 0, 700),
                                                (5000, 2048, [0, 5000], 3800, 1200)])
def test_indexer_selection_is_exact_on_its_own_scores(T, K, cut, row0, nrows):
    # Consistency of the selection stage: the kernel's own fp32 scores, ranked by the rule, give
    # exactly its indices (candidate buffer, approximate and exact compactions, tie-breaking).
    # Independent of fp32 rounding; the set parity against the fp64 oracle is checked above.
    x = synth.indexer_inputs(T, 64, 128, seed=21)
    x["w"][:, 7] = 0.0  # a zero-weight head: its ReLU terms drop out exactly
    cu = torch.tensor(cut, dtype=torch.int32)
    start, _, _, _ = dsa.dsa_packed_metadata(cu.to(DEV), T)
    q, k, w = x["q_idx"].to(DEV), x["k_idx"].to(DEV), x["w"].to(DEV)
    ws = torch.zeros(4096, dtype=torch.uint8, device=DEV)
    idx, ln, sc = dsa.dsa_indexer_topk_with_scores(q, k, w, start, K, row0, nrows, workspace=ws)
    assert dsa.dsa_read_device_status(ws) == 0
    idx0, ln0 = dsa.dsa_indexer_topk(q, k, w, start, K)  # the production kernel selects the same
    assert torch.equal(idx0, idx) and torch.equal(ln0, ln)
    idx, ln, sc, st = idx.cpu().numpy(), ln.cpu().numpy(), sc.cpu().numpy(), oracle_start(cu, T, start)
    for r in range(nrows):
        t = row0 + r
        want = _exact_topk(sc[r], st[t], t, K)
        n = len(want)
        assert ln[t] == n
        assert np.array_equal(idx[t, :n], want), f"row {t}"
        assert np.all(idx[t, n:] == -1)
        assert np.all(np.isfinite(sc[r, st[t]:t + 1]))  # every window key was scored
