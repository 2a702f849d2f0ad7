"""Context-parallel metadata and indexer (rank-local queries, gathered global keys): CUDA path
through the C ABI vs the fp64 oracle, and vs the CP=1 path on the compact layout.

The layout is padded THD storage: every sequence's real tokens followed by padding rows, plus
trailing pack padding; ranks hold load-balanced contiguous chunks of the storage rows
(2R chunks, rank r holds chunks r and 2R-1-r), as the cuDNN DSA API page describes
query_indices ("global padded-storage coordinates for the local query rows").
"""
import numpy as np
import pytest
import torch

import oracle
import sparse_attention_mla_gb300 as dsa
from sparse_attention_mla_gb300 import synth

from test_gpu_indexer import GAMMA

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def layout(lens, pads, trailing):
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    P = np.concatenate([[0], np.cumsum(np.asarray(lens) + np.asarray(pads))]).astype(np.int32)
    return cu, P, int(P[-1]) + int(trailing)


def cp_split(total, ranks, rank):
    edges = np.linspace(0, total, 2 * ranks + 1).astype(np.int64)
    a, b = rank, 2 * ranks - 1 - rank
    return np.concatenate([np.arange(edges[a], edges[a + 1]), np.arange(edges[b], edges[b + 1])]).astype(np.int32)


def t32(a):
    return torch.as_tensor(np.asarray(a, dtype=np.int32)).to(DEV)


@pytest.mark.parametrize("ranks,padded,masked", [(1, False, False), (2, True, False), (3, True, True), (4, True, True)])
def test_metadata_cp_matches_oracle(ranks, padded, masked):
    rng = np.random.default_rng(40 + ranks)
    lens = rng.integers(0, 700, 7)
    lens[2] = 0  # an empty sequence
    pads = rng.integers(0, 50, 7) if padded else np.zeros(7, np.int64)
    cu, P, total = layout(lens, pads, 33 if padded else 0)
    for r in range(ranks):
        qi = cp_split(total, ranks, r)
        pm = (rng.random(len(qi)) < 0.05).astype(np.uint8) if masked else None
        got = dsa.dsa_packed_metadata_cp(t32(cu), total, query_indices=t32(qi),
                                         cu_seqlens_padded=t32(P) if padded else None,
                                         padding_mask=None if pm is None else torch.as_tensor(pm).to(DEV))
        ref = oracle.packed_metadata_cp(cu, total, query_indices=qi, cu_seqlens_padded=P if padded else None,
                                        padding_mask=pm)
        assert np.array_equal(got[0].cpu().numpy(), ref[0]) and np.array_equal(got[1].cpu().numpy(), ref[1])
        assert got[2:] == ref[2:]


def test_metadata_cp_identity_and_bool_mask():
    cu = np.array([0, 5, 5, 12], np.int32)
    st, cl, mx, ne = dsa.dsa_packed_metadata_cp(t32(cu), 12)
    ref = oracle.packed_metadata(cu, 12)
    assert np.array_equal(st.cpu().numpy(), ref[0]) and np.array_equal(cl.cpu().numpy(), ref[1])
    assert (mx, ne) == ref[2:]
    mask = torch.zeros(12, dtype=torch.bool, device=DEV)
    mask[7] = True
    _, cl, _, ne = dsa.dsa_packed_metadata_cp(t32(cu), 12, padding_mask=mask)
    assert cl[7].item() == 0 and ne == 0


def test_metadata_cp_rejects_inconsistent_layouts():
    cu = t32([0, 6, 9])
    with pytest.raises(dsa.DsaError):  # sequence 0 has 6 real tokens in 4 storage rows
        dsa.dsa_packed_metadata_cp(cu, 16, query_indices=t32([0, 1]), cu_seqlens_padded=t32([0, 4, 9]))
    with pytest.raises(dsa.DsaError):  # a coordinate outside the key tokens
        dsa.dsa_packed_metadata_cp(cu, 9, query_indices=t32([0, 9]))
    with pytest.raises(dsa.DsaError):  # storage beyond the key tokens
        dsa.dsa_packed_metadata_cp(cu, 8, query_indices=t32([0]))


def check_window_rows(gidx, glen, q_rows, k, w_rows, ws, wl, K):
    """Rows vs the oracle's top-k over the same windows: lengths exact; index sets equal except
    where keys sit inside the fp32 tie band of the n-th best score."""
    ref_idx, ref_len, kth = oracle.indexer_topk_window(q_rows, k, w_rows, ws, wl, K)
    for r in range(len(ws)):
        n = int(ref_len[r])
        assert glen[r] == n, (r, glen[r], n)
        assert np.all(gidx[r, n:] == -1)
        sel = gidx[r, :n]
        assert np.all(np.diff(sel) > 0)
        if n:
            assert sel.min() >= ws[r] and sel.max() <= ws[r] + wl[r] - 1
        diff = sorted(set(sel.tolist()) ^ set(ref_idx[r, :n].tolist()))
        if diff:
            sc, mag = oracle.indexer_scores(q_rows, k, w_rows, np.full(len(diff), r), np.array(diff),
                                            with_magnitude=True)
            ksc, kmag = oracle.indexer_scores(q_rows, k, w_rows, np.full(n, r), ref_idx[r, :n], with_magnitude=True)
            j = int(np.argmin(ksc))
            for d in range(len(diff)):
                assert abs(sc[d] - kth[r]) <= GAMMA * (mag[d] + kmag[j]), f"row {r}: key {diff[d]}"


def test_indexer_cp_ranks_equal_cp1_and_oracle():
    # three sequences in padded storage (one long enough for candidate compactions at K = 2048),
    # two CP ranks, a few real rows masked as padding on each rank
    lens, pads, K = [5000, 300, 1300], [37, 0, 91], 2048
    cu, P, total = layout(lens, pads, 40)
    x = synth.indexer_inputs(total, 64, 128, seed=44)  # every storage row, padding included
    q_all, k_all, w_all = x["q_idx"], x["k_idx"], x["w"]
    # CP=1 reference on the compact layout (real rows only), mapped back to storage coordinates
    real = np.concatenate([np.arange(P[i], P[i] + lens[i]) for i in range(len(lens))]).astype(np.int64)
    seq_of = np.concatenate([np.full(lens[i], i) for i in range(len(lens))])
    shift = (P[:-1] - cu[:-1])[seq_of]  # storage = compact + shift
    st_c, _, _, _ = dsa.dsa_packed_metadata(t32(cu), int(cu[-1]))
    ws = torch.zeros(4096, dtype=torch.uint8, device=DEV)
    idx_c, len_c = dsa.dsa_indexer_topk(q_all[real].to(DEV), k_all[real].to(DEV), w_all[real].to(DEV), st_c, K,
                                        workspace=ws)
    assert dsa.dsa_read_device_status(ws) == 0
    idx_c, len_c = idx_c.cpu().numpy(), len_c.cpu().numpy()
    ref_storage = np.where(idx_c >= 0, idx_c + shift[np.clip(idx_c, 0, None)], -1)
    compact_of = {int(g): c for c, g in enumerate(real)}
    rng = np.random.default_rng(45)
    k_dev = k_all.to(DEV)
    for r in range(2):
        qi = cp_split(total, 2, r)
        pm = np.zeros(len(qi), np.uint8)
        pm[rng.choice(len(qi), 5, replace=False)] = 1
        st, cl, _, ne = dsa.dsa_packed_metadata_cp(t32(cu), total, query_indices=t32(qi), cu_seqlens_padded=t32(P),
                                                   padding_mask=torch.as_tensor(pm).to(DEV))
        assert ne == 0
        qi64 = qi.astype(np.int64)
        idx, ln = dsa.dsa_indexer_topk_cp(q_all[qi64].to(DEV), k_dev, w_all[qi64].to(DEV), st, cl, K, workspace=ws)
        assert dsa.dsa_read_device_status(ws) == 0
        # the oracle's own window metadata for these rows; the GPU's must equal it
        st_ref, cl_ref, _, _ = oracle.packed_metadata_cp(cu, total, query_indices=qi, cu_seqlens_padded=P,
                                                         padding_mask=pm)
        assert np.array_equal(st.cpu().numpy(), st_ref) and np.array_equal(cl.cpu().numpy(), cl_ref)
        idx, ln, st, cl = idx.cpu().numpy(), ln.cpu().numpy(), st_ref, cl_ref
        for j, g in enumerate(qi.tolist()):
            c = compact_of.get(g)
            if c is None or pm[j]:  # a padding row: empty window, empty selection
                assert cl[j] == 0 and ln[j] == 0 and np.all(idx[j] == -1), (r, g)
                continue
            assert ln[j] == len_c[c] and np.array_equal(idx[j], ref_storage[c]), (r, g)
        # oracle on sampled rows: both chunk boundaries, the sequence ends, random rows
        pick = np.unique(np.concatenate([[0, len(qi) // 2 - 1, len(qi) // 2, len(qi) - 1],
                                         rng.choice(len(qi), 40, replace=False)]))
        check_window_rows(idx[pick], ln[pick], q_all[qi64[pick]], k_all, w_all[qi64[pick]], st[pick], cl[pick], K)


def test_cp_ranks_through_fwd_bwd_equal_one_shot():
    # One rank's half of context parallelism end to end: metadata -> indexer -> sparse MLA forward ->
    # backward on the rank's local rows against all keys, the key gradient accumulated over the ranks.
    # Rows (indices, out, lse, dq) equal the one-shot run's rows; the summed dkv equals its dkv up to
    # the order of the fp32 reductions.
    lens, pads, K, H = [1500, 700], [20, 12], 256, 16
    cu, P, total = layout(lens, pads, 8)
    ind = synth.indexer_inputs(total, 64, 128, seed=46)
    x = synth.mla_inputs(total, H, 576, 512, seed=47)
    q, kv, dout = x["q"].to(DEV), x["kv"].to(DEV), x["dout"].to(DEV)
    qx, kx, wx = ind["q_idx"].to(DEV), ind["k_idx"].to(DEV), ind["w"].to(DEV)
    scale = 192 ** -0.5
    wi = torch.zeros(4096, dtype=torch.uint8, device=DEV)
    wf = torch.zeros(dsa.workspace_size("fwd", total, H), dtype=torch.uint8, device=DEV)
    wb = torch.zeros(dsa.workspace_size("bwd", total, H, K), dtype=torch.uint8, device=DEV)

    def rank_pass(rows, dkv, accumulate):
        st, cl, _, _ = dsa.dsa_packed_metadata_cp(t32(cu), total, query_indices=rows, cu_seqlens_padded=t32(P))
        r64 = rows.long()
        idx, ln = dsa.dsa_indexer_topk_cp(qx[r64].contiguous(), kx, wx[r64].contiguous(), st, cl, K, workspace=wi)
        out, lse, lo = dsa.dsa_sparse_mla_fwd(q[r64].contiguous(), kv, idx, scale, topk_len=ln, out_lo=True,
                                              workspace=wf)
        dq, dkv, _ = dsa.dsa_sparse_mla_bwd(q[r64].contiguous(), kv, idx, scale, out, lse, dout[r64].contiguous(),
                                            topk_len=ln, out_lo=lo, dkv_accum=dkv, accumulate=accumulate,
                                            workspace=wb)
        for w_ in (wi, wf, wb):
            assert dsa.dsa_read_device_status(w_) == 0
        return idx, ln, out, lse, dq, dkv

    one = rank_pass(t32(np.arange(total)), torch.empty(total, 576, dtype=torch.float32, device=DEV), False)
    dkv = torch.empty(total, 576, dtype=torch.float32, device=DEV)
    for r in range(2):
        rows = t32(cp_split(total, 2, r))
        idx, ln, out, lse, dq, dkv = rank_pass(rows, dkv, r > 0)
        r64 = rows.long()
        assert torch.equal(idx, one[0][r64]) and torch.equal(ln, one[1][r64])
        assert torch.equal(out, one[2][r64]) and torch.equal(lse, one[3][r64]) and torch.equal(dq, one[4][r64])
    err = (dkv - one[5]).norm() / one[5].norm()
    assert err.item() <= 1e-6, err.item()
    # padding rows (storage slots past a sequence's real tokens, trailing pack padding) are empty
    pad = np.setdiff1d(np.arange(total), np.concatenate([np.arange(P[i], P[i] + lens[i]) for i in range(2)]))
    assert torch.all(one[1][torch.as_tensor(pad).to(DEV)] == 0)
    assert torch.all(one[2][torch.as_tensor(pad).to(DEV)] == 0)


def test_indexer_cp_with_scores():
    # the context-parallel indexer through the scored entry: the same selection as dsa_indexer_topk_cp,
    # and each selected slot's score against the oracle's fp64 score of its own selection (rows whose
    # selection equals the oracle's), -inf past the prefix
    lens, pads, K = [1500, 400], [10, 3], 256
    cu, P, total = layout(lens, pads, 6)
    x = synth.indexer_inputs(total, 64, 128, seed=48)
    qi = cp_split(total, 2, 1)
    st, cl, _, _ = dsa.dsa_packed_metadata_cp(t32(cu), total, query_indices=t32(qi), cu_seqlens_padded=t32(P))
    st_ref, cl_ref, _, _ = oracle.packed_metadata_cp(cu, total, query_indices=qi, cu_seqlens_padded=P)
    assert np.array_equal(st.cpu().numpy(), st_ref) and np.array_equal(cl.cpu().numpy(), cl_ref)
    qi64 = qi.astype(np.int64)
    q, k, w = x["q_idx"][qi64].to(DEV), x["k_idx"].to(DEV), x["w"][qi64].to(DEV)
    idx, ln, sc = dsa.dsa_indexer_topk_scored(q, k, w, st, K, causal_len=cl)
    idx0, ln0 = dsa.dsa_indexer_topk_cp(q, k, w, st, cl, K)
    assert torch.equal(idx, idx0) and torch.equal(ln, ln0)
    rows = np.unique(np.concatenate([[0, 1, len(qi) // 2, len(qi) - 1],
                                     np.random.default_rng(49).choice(len(qi), 60, replace=False)]))
    ref_idx, ref_len, _ = oracle.indexer_topk_window(x["q_idx"][qi64[rows]], x["k_idx"], x["w"][qi64[rows]],
                                                      st_ref[rows], cl_ref[rows], K)
    gi, gl, gs = idx.cpu().numpy()[rows], ln.cpu().numpy()[rows], sc.cpu().double().numpy()[rows]
    same = np.all(gi == ref_idx, axis=1) & (gl == ref_len)
    assert same.mean() >= 0.9
    for i in np.nonzero(same)[0]:
        n = int(ref_len[i])
        assert np.all(gs[i, n:] == -np.inf)
        if n:
            rs, mag = oracle.indexer_scores(x["q_idx"][[int(qi64[rows[i]])]], x["k_idx"], x["w"][[int(qi64[rows[i]])]],
                                            np.zeros(n, np.int64), ref_idx[i, :n], with_magnitude=True)
            assert np.all(np.abs(gs[i, :n] - rs) <= GAMMA * mag), f"row {rows[i]}: scores"
