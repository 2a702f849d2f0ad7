"""Pins of the fp64 CPU oracle against things other than itself.

Each test checks one oracle function against an independent library routine
(numpy / torch fp64), brute force on tiny inputs, a closed form, a finite
difference, an invariant stated on the pages, or a hand-derived example.
All of these run on the CPU (no GPU marker).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from sparse_attention_mla_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# --------------------------------------------------------------------------
# helpers (independent re-statements used only as checks)
# --------------------------------------------------------------------------
def numpy_indexer_scores(q, k, w):
    """Library route: einsum -> ReLU -> weighted head sum, all rows x all keys."""
    dots = np.einsum("thd,sd->ths", q, k)
    return np.einsum("th,ths->ts", w, np.maximum(dots, 0.0))


def dense_masked_attention(q, kv, mask, scale, Dv):
    """torch fp64 textbook masked softmax attention (MQA over one kv)."""
    q = torch.as_tensor(q, dtype=torch.float64)
    kv = torch.as_tensor(kv, dtype=torch.float64)
    s = scale * torch.einsum("thd,sd->ths", q, kv)  # [T,H,Tk]
    m = torch.as_tensor(mask)[:, None, :]
    s = s.masked_fill(~m, float("-inf"))
    lse = torch.logsumexp(s, dim=-1)
    p = torch.softmax(s, dim=-1)
    p = torch.nan_to_num(p, nan=0.0)
    out = torch.einsum("ths,sv->thv", p, kv[:, :Dv])
    return out, lse


def mask_from_idx(idx, Tk):
    T, K = idx.shape
    mask = np.zeros((T, Tk), bool)
    for t in range(T):
        for j in range(K):
            if 0 <= idx[t, j] < Tk:
                mask[t, idx[t, j]] = True
    return mask


def rand_case(T=24, H=3, Dqk=16, Dv=8, K=6, seed=0, holes=True):
    g = synth.generator(seed)
    q = torch.randn(T, H, Dqk, generator=g, dtype=torch.float64)
    kv = torch.randn(T, Dqk, generator=g, dtype=torch.float64)
    dout = torch.randn(T, H, Dv, generator=g, dtype=torch.float64)
    start = torch.zeros(T, dtype=torch.int32)
    idx = synth.random_causal_topk(start, K, g)
    if holes:  # move some -1 into the middle of rows (masked wherever they are)
        idx[K + 3, 1] = -1
        idx[T - 1, 0] = -1
    return q.numpy(), kv.numpy(), dout.numpy(), idx.numpy()


# --------------------------------------------------------------------------
# packed THD metadata
# --------------------------------------------------------------------------
def test_packed_metadata_by_hand():
    cu = np.array([0, 3, 3, 7], np.int32)  # includes an empty sequence
    st, cl, mx, ne = oracle.packed_metadata(cu, 7)
    assert st.tolist() == [0, 0, 0, 3, 3, 3, 3]
    assert cl.tolist() == [1, 2, 3, 1, 2, 3, 4]
    assert mx == 4 and ne == 1


def test_packed_metadata_rejects_bad_cover():
    with pytest.raises(ValueError):
        oracle.packed_metadata(np.array([0, 5, 3], np.int32), 3)
    with pytest.raises(ValueError):
        oracle.packed_metadata(np.array([0, 2, 4], np.int32), 5)


# --------------------------------------------------------------------------
# packed THD metadata with context parallelism (local queries, global keys)
# --------------------------------------------------------------------------
def cp_split(total, ranks, rank):
    """Load-balanced contiguous chunks: 2 * ranks chunks, rank r holds chunks r and 2R-1-r."""
    edges = np.linspace(0, total, 2 * ranks + 1).astype(np.int64)
    a, b = rank, 2 * ranks - 1 - rank
    return np.concatenate([np.arange(edges[a], edges[a + 1]), np.arange(edges[b], edges[b + 1])]).astype(np.int32)


def test_packed_metadata_cp_golden_two_ranks():
    with open(os.path.join(GOLDEN, "cp_metadata_two_ranks.json")) as f:
        g = json.load(f)
    for rk in g["ranks"]:
        st, cl, mx, ne = oracle.packed_metadata_cp(
            np.array(g["cu_seqlens"]), g["total_key_tokens"], query_indices=np.array(rk["query_indices"]),
            cu_seqlens_padded=np.array(g["cu_seqlens_padded"]), padding_mask=np.array(rk["padding_mask"]))
        assert st.tolist() == rk["seq_start"] and cl.tolist() == rk["causal_len"]
        assert mx == g["max_seqlen"] and ne == g["all_rows_nonempty"]


def test_packed_metadata_cp_identity_is_the_cp1_form():
    rng = np.random.default_rng(21)
    for _ in range(20):
        lens = rng.integers(0, 9, rng.integers(1, 6))
        cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
        T = int(cu[-1])
        a = oracle.packed_metadata_cp(cu, T)
        b = oracle.packed_metadata(cu, T)
        assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1]) and a[2:] == b[2:]


@pytest.mark.parametrize("ranks", [1, 2, 3])
def test_packed_metadata_cp_shards_keep_every_real_token(ranks):
    # Padded storage with a random pad after every sequence, split over CP ranks: every real
    # token shows up on exactly one rank, with the start of its sequence's storage and the
    # causal length the CP=1 metadata gives it in the compact layout; padding rows get length 0.
    rng = np.random.default_rng(22 + ranks)
    lens = rng.integers(0, 12, 5)
    pads = rng.integers(0, 4, 5)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    P = np.concatenate([[0], np.cumsum(lens + pads)]).astype(np.int32)
    total = int(P[-1]) + 2  # two rows of trailing pack padding
    _, ref_len, ref_mx, _ = oracle.packed_metadata(cu, int(cu[-1]))
    seen = {}
    for r in range(ranks):
        qi = cp_split(total, ranks, r)
        st, cl, mx, _ = oracle.packed_metadata_cp(cu, total, query_indices=qi, cu_seqlens_padded=P)
        assert mx == ref_mx
        for g, s, c in zip(qi.tolist(), st.tolist(), cl.tolist()):
            assert g not in seen
            seen[g] = (s, c)
    assert sorted(seen) == list(range(total))
    for i in range(len(lens)):
        for p in range(int(P[i + 1] - P[i])):
            s, c = seen[int(P[i]) + p]
            assert s == P[i]
            assert c == (ref_len[cu[i] + p] if p < lens[i] else 0)
    for g in range(int(P[-1]), total):
        assert seen[g][1] == 0


def test_packed_metadata_cp_mask_is_authoritative_and_bad_input_rejected():
    cu, P = np.array([0, 4], np.int32), np.array([0, 4], np.int32)
    qi = np.array([0, 1, 2, 3], np.int32)
    _, cl, _, ne = oracle.packed_metadata_cp(cu, 4, query_indices=qi, cu_seqlens_padded=P,
                                             padding_mask=np.array([0, 0, 1, 1]))
    assert cl.tolist() == [1, 2, 0, 0] and ne == 0
    with pytest.raises(ValueError):  # a real length larger than its storage
        oracle.packed_metadata_cp(np.array([0, 5]), 8, cu_seqlens_padded=np.array([0, 4]), T_q=4)
    with pytest.raises(ValueError):  # a coordinate outside the key tokens
        oracle.packed_metadata_cp(cu, 4, query_indices=np.array([0, 4]))
    with pytest.raises(ValueError):  # storage beyond the key tokens
        oracle.packed_metadata_cp(cu, 3, query_indices=np.array([0]))


# --------------------------------------------------------------------------
# indexer score
# --------------------------------------------------------------------------
def test_indexer_scores_match_numpy_einsum():
    rng = np.random.default_rng(1)
    T, Hi, Di = 9, 4, 16
    q = rng.standard_normal((T, Hi, Di))
    k = rng.standard_normal((T, Di))
    w = rng.uniform(-0.5, 1.0, (T, Hi))  # signed weights too
    pr, pk = np.meshgrid(np.arange(T), np.arange(T), indexing="ij")
    got = oracle.indexer_scores(q, k, w, pr.ravel(), pk.ravel()).reshape(T, T)
    ref = numpy_indexer_scores(q, k, w)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_indexer_special_cases():
    rng = np.random.default_rng(2)
    q = rng.standard_normal((5, 1, 8))
    k = rng.standard_normal((5, 8))
    pr, pk = np.meshgrid(np.arange(5), np.arange(5), indexing="ij")
    got = oracle.indexer_scores(q, k, np.ones((5, 1)), pr.ravel(), pk.ravel()).reshape(5, 5)
    np.testing.assert_allclose(got, np.maximum(q[:, 0, :] @ k.T, 0.0), rtol=1e-13, atol=1e-13)
    got0 = oracle.indexer_scores(q, k, np.zeros((5, 1)), pr.ravel(), pk.ravel())
    assert np.all(got0 == 0.0)


def test_indexer_score_magnitude_matches_numpy():
    # the magnitude the tie band is built from: sum_h |w[t,h]| sum_d |q[t,h,d] k[s,d]| (library route,
    # numpy), and a closed form: with q, k, w all positive no ReLU cuts and no term cancels, so the
    # magnitude equals the score itself
    rng = np.random.default_rng(21)
    T, Hi, Di = 7, 5, 12
    q = rng.standard_normal((T, Hi, Di))
    k = rng.standard_normal((T, Di))
    w = rng.uniform(-0.5, 1.0, (T, Hi))
    pr, pk = np.meshgrid(np.arange(T), np.arange(T), indexing="ij")
    _, mag = oracle.indexer_scores(q, k, w, pr.ravel(), pk.ravel(), with_magnitude=True)
    ref = np.einsum("th,thsd->ts", np.abs(w), np.abs(np.einsum("thd,sd->thsd", q, k)))
    np.testing.assert_allclose(mag.reshape(T, T), ref, rtol=1e-13, atol=1e-13)
    qp, kp, wp = np.abs(q), np.abs(k), np.abs(w)
    sc, magp = oracle.indexer_scores(qp, kp, wp, pr.ravel(), pk.ravel(), with_magnitude=True)
    np.testing.assert_allclose(magp, sc, rtol=1e-13, atol=0)


# --------------------------------------------------------------------------
# causal top-k
# --------------------------------------------------------------------------
def brute_topk(scores_row, b, t, K):
    cand = sorted(range(b, t + 1), key=lambda s: (-scores_row[s], s))
    n = min(K, t - b + 1)
    sel = sorted(cand[:n])
    return sel + [-1] * (K - n), n


@pytest.mark.parametrize("K", [1, 5, 40])
def test_topk_brute_force_packed(K):
    rng = np.random.default_rng(3)
    cu = np.array([0, 17, 40], np.int32)
    T, Hi, Di = 40, 3, 8
    q = rng.standard_normal((T, Hi, Di))
    k = rng.standard_normal((T, Di))
    w = rng.uniform(0, 1, (T, Hi))
    st, _, _, _ = oracle.packed_metadata(cu, T)
    idx, ln, kth = oracle.indexer_topk(q, k, w, st, np.arange(T), K)
    S = numpy_indexer_scores(q, k, w)
    for t in range(T):
        ref, n = brute_topk(S[t], st[t], t, K)
        assert idx[t].tolist() == ref, t
        assert ln[t] == n
        sel = [s for s in ref if s >= 0]
        assert kth[t] == pytest.approx(min(S[t, s] for s in sel), rel=1e-12, abs=1e-12)


def test_topk_all_ties_take_lowest_indices():
    rng = np.random.default_rng(4)
    T, K = 30, 7
    q = rng.standard_normal((T, 2, 4))
    k = rng.standard_normal((T, 4))
    st = np.zeros(T, np.int32)
    idx, ln, _ = oracle.indexer_topk(q, k, np.zeros((T, 2)), st, np.arange(T), K)
    for t in range(T):
        n = min(K, t + 1)
        assert idx[t, :n].tolist() == list(range(n)) and np.all(idx[t, n:] == -1)


def test_topk_strictly_increasing_scores_pick_the_window_end():
    T, Di, K = 50, 4, 6
    k = np.zeros((T, Di))
    k[:, 0] = 0.5 * (np.arange(T) + 1)          # k[s] = alpha (s+1) e0
    q = np.abs(np.random.default_rng(5).standard_normal((T, 2, Di))) + 0.1  # q[...,0] > 0
    w = np.full((T, 2), 0.25)
    st = np.zeros(T, np.int32)
    idx, ln, _ = oracle.indexer_topk(q, k, w, st, np.arange(T), K)
    for t in range(T):
        n = min(K, t + 1)
        assert idx[t, :n].tolist() == list(range(t - n + 1, t + 1))


def test_topk_subset_of_rows_matches_all_rows():
    rng = np.random.default_rng(6)
    T, K = 33, 4
    q = rng.standard_normal((T, 2, 4))
    k = rng.standard_normal((T, 4))
    w = rng.uniform(0, 1, (T, 2))
    st = np.zeros(T, np.int32)
    full, _, _ = oracle.indexer_topk(q, k, w, st, np.arange(T), K)
    rows = np.array([32, 0, 17])
    part, _, _ = oracle.indexer_topk(q[rows], k, w[rows], st, rows, K)
    assert np.array_equal(part, full[rows])


def test_topk_window_is_the_causal_form_on_causal_windows():
    rng = np.random.default_rng(7)
    cu = np.array([0, 11, 30], np.int32)
    T, K = 30, 5
    q = rng.standard_normal((T, 2, 4))
    k = rng.standard_normal((T, 4))
    w = rng.uniform(0, 1, (T, 2))
    st, cl, _, _ = oracle.packed_metadata(cu, T)
    a = oracle.indexer_topk(q, k, w, st, np.arange(T), K)
    b = oracle.indexer_topk_window(q, k, w, st, cl, K)
    assert all(np.array_equal(x, y) for x, y in zip(a, b))


def test_topk_window_brute_force_arbitrary_and_empty_windows():
    rng = np.random.default_rng(8)
    n, Tk, K = 12, 25, 6
    q = rng.standard_normal((n, 3, 5))
    k = rng.standard_normal((Tk, 5))
    w = rng.uniform(-0.2, 1, (n, 3))
    ws = rng.integers(0, Tk, n).astype(np.int32)
    wl = np.minimum(rng.integers(0, 12, n), Tk - ws).astype(np.int32)
    wl[3] = 0
    idx, ln, _ = oracle.indexer_topk_window(q, k, w, ws, wl, K)
    S = numpy_indexer_scores(q, k, w)
    for r in range(n):
        if wl[r] == 0:
            assert ln[r] == 0 and np.all(idx[r] == -1)
            continue
        ref, m = brute_topk(S[r], ws[r], ws[r] + wl[r] - 1, K)
        assert idx[r].tolist() == ref and ln[r] == m


# --------------------------------------------------------------------------
# sparse MLA forward
# --------------------------------------------------------------------------
def test_fwd_golden_two_slot_example():
    with open(os.path.join(GOLDEN, "fwd_two_slot.json")) as f:
        gd = json.load(f)
    out, lse = oracle.sparse_mla_fwd(np.array(gd["q"]), np.array(gd["kv"]), np.array(gd["idx"]),
                                     gd["scale"], Dv=gd["Dv"])
    np.testing.assert_allclose(out, np.array(gd["out"]), rtol=1e-14, atol=1e-14)
    np.testing.assert_allclose(lse, np.array(gd["lse"]), rtol=1e-14, atol=1e-14)


def test_fwd_matches_dense_masked_softmax():
    q, kv, _, idx = rand_case()
    scale = 0.37
    out, lse = oracle.sparse_mla_fwd(q, kv, idx, scale, Dv=8)
    ref_o, ref_l = dense_masked_attention(q, kv, mask_from_idx(idx, kv.shape[0]), scale, 8)
    np.testing.assert_allclose(out, ref_o.numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse, ref_l.numpy(), rtol=1e-12, atol=1e-12)


def test_fwd_full_prefix_equals_causal_sdpa():
    T, H, Dqk, Dv = 20, 2, 12, 8
    g = synth.generator(7)
    q = torch.randn(T, H, Dqk, generator=g, dtype=torch.float64)
    kv = torch.randn(T, Dqk, generator=g, dtype=torch.float64)
    idx = synth.random_causal_topk(torch.zeros(T, dtype=torch.int32), T, g)  # K >= c: whole prefix
    out, _ = oracle.sparse_mla_fwd(q, kv, idx, 0.5, Dv=Dv)
    ref = torch.nn.functional.scaled_dot_product_attention(
        q.transpose(0, 1), kv[None].expand(H, T, Dqk), kv[None, :, :Dv].expand(H, T, Dv),
        is_causal=True, scale=0.5).transpose(0, 1)
    np.testing.assert_allclose(out, ref.numpy(), rtol=1e-12, atol=1e-12)


def test_fwd_closed_forms():
    rng = np.random.default_rng(8)
    H, Dqk, Dv, Tk = 3, 10, 6, 12
    q = rng.standard_normal((2, H, Dqk))
    kv = rng.standard_normal((Tk, Dqk))
    # one valid slot: O = kv[i, :Dv], LSE = z
    idx = np.array([[-1, 5, -1], [-1, -1, -1]], np.int32)
    out, lse = oracle.sparse_mla_fwd(q, kv, idx, 0.3, Dv=Dv)
    for h in range(H):
        np.testing.assert_allclose(out[0, h], kv[5, :Dv], rtol=1e-14)
        assert lse[0, h] == pytest.approx(0.3 * q[0, h] @ kv[5], rel=1e-13)
    # empty row: O = 0, LSE = -inf
    assert np.all(out[1] == 0.0) and np.all(np.isneginf(lse[1]))
    # identical selected rows: O = that row, LSE = z + ln n
    kv2 = np.tile(kv[3], (Tk, 1))
    idx2 = np.array([[0, 2, 4, 6, 8]], np.int32)
    out2, lse2 = oracle.sparse_mla_fwd(q[:1], kv2, idx2, 0.3, Dv=Dv)
    for h in range(H):
        np.testing.assert_allclose(out2[0, h], kv[3, :Dv], rtol=1e-13)
        assert lse2[0, h] == pytest.approx(0.3 * q[0, h] @ kv[3] + math.log(5), rel=1e-13)


def test_fwd_invariants_permutation_padding_chunking_length():
    q, kv, _, idx = rand_case(T=30, K=8, holes=False)
    scale = 0.21
    out, lse = oracle.sparse_mla_fwd(q, kv, idx, scale, Dv=8)
    # slot permutation (moves the -1 suffix into the middle as well)
    perm = np.random.default_rng(9).permutation(idx.shape[1])
    o2, l2 = oracle.sparse_mla_fwd(q, kv, idx[:, perm], scale, Dv=8)
    np.testing.assert_allclose(o2, out, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(l2, lse, rtol=1e-12, atol=1e-13)
    # NoPE: zero-padding q and kv channels (the RoPE slot) changes nothing
    pad = lambda a: np.concatenate([a, np.zeros(a.shape[:-1] + (8,))], axis=-1)
    o3, l3 = oracle.sparse_mla_fwd(pad(q), pad(kv), idx, scale, Dv=8)
    np.testing.assert_allclose(o3, out, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(l3, lse, rtol=1e-13, atol=1e-14)
    # query chunks are independent
    o4, _ = oracle.sparse_mla_fwd(q[11:23], kv, idx[11:23], scale, Dv=8)
    np.testing.assert_allclose(o4, out[11:23], rtol=0, atol=0)
    # topk_len bounds the prefix: equal to writing -1 after it
    ln = np.minimum(np.arange(30), 5).astype(np.int32)
    cut = idx.copy()
    for t in range(30):
        cut[t, ln[t]:] = -1
    o5, l5 = oracle.sparse_mla_fwd(q, kv, idx, scale, Dv=8, len_rows=ln)
    o6, l6 = oracle.sparse_mla_fwd(q, kv, cut, scale, Dv=8)
    np.testing.assert_array_equal(o5, o6)
    np.testing.assert_array_equal(l5, l6)


# --------------------------------------------------------------------------
# sparse MLA backward
# --------------------------------------------------------------------------
def test_bwd_central_finite_differences():
    q, kv, dout, idx = rand_case(T=7, H=2, Dqk=6, Dv=4, K=4, seed=10, holes=False)
    idx[5, 2] = -1
    scale = 0.45
    dq, dkv = oracle.sparse_mla_bwd(q, kv, idx, dout, scale, Dv=4)

    def loss(qq, kk):
        o, _ = oracle.sparse_mla_fwd(qq, kk, idx, scale, Dv=4)
        return float(np.sum(o * dout))

    eps = 1e-6
    fq = np.zeros_like(q)
    for i in np.ndindex(q.shape):
        a, b = q.copy(), q.copy()
        a[i] += eps
        b[i] -= eps
        fq[i] = (loss(a, kv) - loss(b, kv)) / (2 * eps)
    fk = np.zeros_like(kv)
    for i in np.ndindex(kv.shape):
        a, b = kv.copy(), kv.copy()
        a[i] += eps
        b[i] -= eps
        fk[i] = (loss(q, a) - loss(q, b)) / (2 * eps)
    np.testing.assert_allclose(dq, fq, rtol=1e-6, atol=1e-8)
    np.testing.assert_allclose(dkv, fk, rtol=1e-6, atol=1e-8)


def test_bwd_matches_torch_autograd_dense():
    q, kv, dout, idx = rand_case(seed=11)
    scale = 0.3
    dq, dkv = oracle.sparse_mla_bwd(q, kv, idx, dout, scale, Dv=8)
    qt = torch.tensor(q, requires_grad=True)
    kt = torch.tensor(kv, requires_grad=True)
    o, _ = dense_masked_attention(qt, kt, mask_from_idx(idx, kv.shape[0]), scale, 8)
    o.backward(torch.tensor(dout))
    np.testing.assert_allclose(dq, qt.grad.numpy(), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(dkv, kt.grad.numpy(), rtol=1e-11, atol=1e-12)


def test_bwd_dkv_column_sums_property():
    # sum_j dS_j = 0 and sum_j P_j = 1 per (t, h) give, for every channel c,
    # sum_k dkv[k, c] = sum_{t,h nonempty} dO[t,h,c] (c < Dv) and 0 (c >= Dv).
    q, kv, dout, idx = rand_case(T=26, Dqk=12, Dv=8, seed=12)
    idx[4, :] = -1  # an empty row contributes nothing
    dq, dkv = oracle.sparse_mla_bwd(q, kv, idx, dout, 0.25, Dv=8)
    nonempty = (idx >= 0).any(axis=1)
    colsum = dkv.sum(axis=0)
    np.testing.assert_allclose(colsum[:8], dout[nonempty].sum(axis=(0, 1)), rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(colsum[8:], 0.0, atol=1e-11)
    assert np.all(dq[4] == 0.0)


def test_bwd_query_chunks_sum_to_one_shot():
    q, kv, dout, idx = rand_case(T=31, seed=13)
    dq, dkv = oracle.sparse_mla_bwd(q, kv, idx, dout, 0.2, Dv=8)
    acc = np.zeros_like(dkv)
    parts = []
    for a, b in [(0, 9), (9, 20), (20, 31)]:
        d, _ = oracle.sparse_mla_bwd(q[a:b], kv, idx[a:b], dout[a:b], 0.2, Dv=8, dkv=acc)
        parts.append(d)
    np.testing.assert_allclose(np.concatenate(parts), dq, rtol=0, atol=0)
    np.testing.assert_allclose(acc, dkv, rtol=1e-12, atol=1e-12)


def test_bwd_dq_magnitude_bounds_dq_and_is_tight_on_two_mirrored_slots():
    # dq_mag = scale sum_j |dS_j| |kv[idx_j]| bounds |dq| (triangle inequality) on any input; with two
    # valid slots whose kv rows are negatives of each other dS_2 = -dS_1 (sum_j dS_j = 0) and
    # dq = scale dS_1 (kv_1 - kv_2) = 2 scale dS_1 kv_1, so |dq| equals the magnitude exactly
    q, kv, dout, idx = rand_case(T=20, seed=16)
    dq, _, mag = oracle.sparse_mla_bwd(q, kv, idx, dout, 0.3, Dv=8, with_dq_magnitude=True)
    assert np.all(np.abs(dq) <= mag * (1 + 1e-12) + 1e-300)
    rng = np.random.default_rng(17)
    H, Dqk, Dv = 3, 10, 6
    kv2 = np.zeros((2, Dqk))
    kv2[0] = rng.uniform(0.5, 2.0, Dqk)
    kv2[1] = -kv2[0]
    q2 = rng.standard_normal((1, H, Dqk))
    do2 = rng.standard_normal((1, H, Dv))
    idx2 = np.array([[0, 1]], dtype=np.int32)
    dq2, _, mag2 = oracle.sparse_mla_bwd(q2, kv2, idx2, do2, 0.7, Dv=Dv, with_dq_magnitude=True)
    assert np.all(mag2 > 0)
    np.testing.assert_allclose(np.abs(dq2), mag2, rtol=1e-12, atol=0)


def test_oracle_takes_bf16_tensors_exactly():
    # bf16 inputs are widened exactly: bf16 -> float64 of the same value
    x = synth.randn_bf16((3, 2, 8), synth.generator(14))
    kv = synth.randn_bf16((3, 8), synth.generator(15))
    idx = torch.tensor([[0, -1], [0, 1], [2, 1]], dtype=torch.int32)
    o1, _ = oracle.sparse_mla_fwd(x, kv, idx, 0.5, Dv=4)
    o2, _ = oracle.sparse_mla_fwd(x.double().numpy(), kv.double().numpy(), idx.numpy(), 0.5, Dv=4)
    np.testing.assert_array_equal(o1, o2)


# --------------------------------------------------------------------------
# attention sink (per-head logit with no value row)
# --------------------------------------------------------------------------
def dense_attention_with_sink(q, kv, mask, scale, Dv, sink):
    """torch fp64: the masked score matrix with one more column per head holding the sink logit,
    softmax over keys + sink, the sink's weight multiplying a zero value row."""
    s = scale * torch.einsum("thd,sd->ths", q, kv)
    s = s.masked_fill(~torch.as_tensor(mask)[:, None, :], float("-inf"))
    col = sink[None, :, None].expand(s.shape[0], s.shape[1], 1)
    s = torch.cat([s, col], dim=-1)
    lse = torch.logsumexp(s, dim=-1)
    p = torch.softmax(s, dim=-1)[..., :-1]
    return torch.einsum("ths,sv->thv", p, kv[:, :Dv]), lse


def test_sink_matches_dense_softmax_with_a_sink_column_and_autograd():
    q, kv, dout, idx = rand_case(seed=31)
    idx[2, :] = -1  # an empty row: only the sink remains
    sink = np.array([0.7, -1.3, 2.1])
    scale = 0.35
    out, lse = oracle.sparse_mla_fwd(q, kv, idx, scale, Dv=8, sink=sink)
    dq, dkv, dsink = oracle.sparse_mla_bwd(q, kv, idx, dout, scale, Dv=8, sink=sink)
    qt = torch.tensor(q, requires_grad=True)
    kt = torch.tensor(kv, requires_grad=True)
    st = torch.tensor(sink, requires_grad=True)
    o, l = dense_attention_with_sink(qt, kt, mask_from_idx(idx, kv.shape[0]), scale, 8, st)
    np.testing.assert_allclose(out, o.detach().numpy(), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse, l.detach().numpy(), rtol=1e-12, atol=1e-13)
    o.backward(torch.tensor(dout))
    np.testing.assert_allclose(dq, qt.grad.numpy(), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(dkv, kt.grad.numpy(), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(dsink, st.grad.numpy(), rtol=1e-11, atol=1e-12)
    assert np.all(out[2] == 0.0) and np.allclose(lse[2], sink, rtol=0, atol=0)


def test_sink_closed_forms_and_minus_infinity():
    # one valid slot with score z: lse = log(e^z + e^s), O = sigmoid(z - s) kv_row
    rng = np.random.default_rng(32)
    q = rng.standard_normal((1, 2, 6))
    kv = rng.standard_normal((3, 6))
    idx = np.array([[1, -1, -1]], dtype=np.int32)
    sink = np.array([0.4, -0.9])
    out, lse = oracle.sparse_mla_fwd(q, kv, idx, 0.5, Dv=4, sink=sink)
    z = 0.5 * q[0] @ kv[1]
    np.testing.assert_allclose(lse[0], np.logaddexp(z, sink), rtol=1e-14)
    np.testing.assert_allclose(out[0], (1.0 / (1.0 + np.exp(sink - z)))[:, None] * kv[1, :4][None, :], rtol=1e-13)
    # a sink of -inf is no sink at all, gradients included
    q, kv, dout, idx = rand_case(seed=33)
    o0, l0 = oracle.sparse_mla_fwd(q, kv, idx, 0.3, Dv=8)
    o1, l1 = oracle.sparse_mla_fwd(q, kv, idx, 0.3, Dv=8, sink=np.full(3, -np.inf))
    np.testing.assert_array_equal(o0, o1)
    np.testing.assert_array_equal(l0, l1)
    dq0, dkv0 = oracle.sparse_mla_bwd(q, kv, idx, dout, 0.3, Dv=8)
    dq1, dkv1, ds1 = oracle.sparse_mla_bwd(q, kv, idx, dout, 0.3, Dv=8, sink=np.full(3, -np.inf))
    np.testing.assert_array_equal(dq0, dq1)
    np.testing.assert_array_equal(dkv0, dkv1)
    assert np.all(ds1 == 0.0)


def test_sink_gradient_central_finite_differences():
    q, kv, dout, idx = rand_case(T=9, H=3, Dqk=6, Dv=4, K=4, seed=34, holes=False)
    sink = np.array([0.2, -0.5, 1.1])
    _, _, dsink = oracle.sparse_mla_bwd(q, kv, idx, dout, 0.45, Dv=4, sink=sink)
    eps = 1e-6
    for h in range(3):
        a, b = sink.copy(), sink.copy()
        a[h] += eps
        b[h] -= eps
        fa = np.sum(oracle.sparse_mla_fwd(q, kv, idx, 0.45, Dv=4, sink=a)[0] * dout)
        fb = np.sum(oracle.sparse_mla_fwd(q, kv, idx, 0.45, Dv=4, sink=b)[0] * dout)
        np.testing.assert_allclose(dsink[h], (fa - fb) / (2 * eps), rtol=1e-6, atol=1e-9)


# --------------------------------------------------------------------------
# attention slot probability and the indexer KL loss (reading: see the oracle)
# --------------------------------------------------------------------------
def test_attn_slot_prob_is_the_head_mean_of_the_dense_softmax():
    q, kv, dout, idx = rand_case(seed=41)
    prob = oracle.attn_slot_prob(q, kv, idx, 0.3, Dv=8)
    qt, kt = torch.tensor(q), torch.tensor(kv)
    s = 0.3 * torch.einsum("thd,sd->ths", qt, kt)
    mask = torch.as_tensor(mask_from_idx(idx, kv.shape[0]))
    p = torch.softmax(s.masked_fill(~mask[:, None, :], float("-inf")), dim=-1).nan_to_num(0.0).mean(dim=1)
    ref = np.zeros_like(prob)
    for t in range(idx.shape[0]):
        for j in range(idx.shape[1]):
            if idx[t, j] >= 0:
                ref[t, j] = float(p[t, idx[t, j]])
    np.testing.assert_allclose(prob, ref, rtol=1e-12, atol=1e-14)
    rows = (idx >= 0).any(axis=1)
    np.testing.assert_allclose(prob[rows].sum(axis=1), 1.0, rtol=1e-12)
    # with a sink every row's probabilities sum to below 1 (the sink takes the rest)
    ps = oracle.attn_slot_prob(q, kv, idx, 0.3, Dv=8, sink=np.array([0.5, 1.0, -0.5]))
    assert np.all(ps[rows].sum(axis=1) < 1.0)


def kl_case(seed, T=12, Hi=3, Di=10, Tk=30, K=7):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((T, Hi, Di))
    k = rng.standard_normal((Tk, Di))
    w = rng.uniform(-0.3, 1.0, (T, Hi))
    idx = np.stack([np.sort(rng.choice(Tk, K, replace=False)) for _ in range(T)]).astype(np.int32)
    idx[2, 4:] = -1  # fewer valid slots
    idx[5, 0] = -1   # a hole
    prob = rng.uniform(0.0, 1.0, (T, K)) * (idx >= 0)
    return q, k, w, idx, prob


def test_indexer_kl_matches_torch_autograd_of_the_dense_definition():
    q, k, w, idx, prob = kl_case(51)
    coeff = 0.37
    kl, dq, dw, dk = oracle.indexer_kl(q, k, w, idx, prob, coeff)
    qt = torch.tensor(q, requires_grad=True)
    kt = torch.tensor(k, requires_grad=True)
    wt = torch.tensor(w, requires_grad=True)
    valid = torch.as_tensor(idx >= 0)
    gidx = torch.as_tensor(np.where(idx >= 0, idx, 0)).long()
    kg = kt[gidx]                                                      # [T, K, Di]
    s = torch.einsum("thd,tjd->thj", qt, kg)
    I = torch.einsum("th,thj->tj", wt, torch.relu(s))
    logq = torch.log_softmax(I.masked_fill(~valid, float("-inf")), dim=1)
    p = torch.tensor(prob) / torch.tensor(prob).sum(dim=1, keepdim=True)
    terms = torch.where(p > 0, p * (torch.log(torch.where(p > 0, p, 1.0)) - logq), torch.zeros_like(p))
    kl_t = terms.sum(dim=1)
    (coeff * kl_t.sum()).backward()
    np.testing.assert_allclose(kl, kl_t.detach().numpy(), rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(dq, qt.grad.numpy(), rtol=1e-10, atol=1e-13)
    np.testing.assert_allclose(dw, wt.grad.numpy(), rtol=1e-10, atol=1e-13)
    np.testing.assert_allclose(dk, kt.grad.numpy(), rtol=1e-10, atol=1e-13)


def test_indexer_kl_closed_forms():
    q, k, w, idx, _ = kl_case(52)
    # the attention's distribution equal to the indexer's (softmax of the numpy scores): zero loss and gradient
    I = np.einsum("th,thj->tj", w, np.maximum(np.einsum("thd,tjd->thj", q, k[np.where(idx >= 0, idx, 0)]), 0.0))
    e = np.where(idx >= 0, np.exp(I - I.max(axis=1, keepdims=True)), 0.0)
    kl, dq, dw, dk = oracle.indexer_kl(q, k, w, idx, e / e.sum(axis=1, keepdims=True), 1.0)
    np.testing.assert_allclose(kl, 0.0, atol=1e-12)
    for g in (dq, dw, dk):
        np.testing.assert_allclose(g, 0.0, atol=1e-12)
    # one valid slot: p = q = 1, nothing to learn; an empty row: zero
    idx1 = np.full_like(idx, -1)
    idx1[:, 3] = idx[:, 3].clip(min=0)
    idx1[4, :] = -1
    kl1, dq1, dw1, dk1 = oracle.indexer_kl(q, k, w, idx1, np.ones(idx.shape), 1.0)
    assert np.all(kl1 == 0.0) and np.all(dq1 == 0.0) and np.all(dw1 == 0.0) and np.all(dk1 == 0.0)


def test_indexer_kl_gradient_central_finite_differences_in_w():
    q, k, w, idx, prob = kl_case(53, T=6)
    _, _, dw, _ = oracle.indexer_kl(q, k, w, idx, prob, 0.5)
    eps = 1e-6
    for t in range(6):
        for h in range(3):
            a, b = w.copy(), w.copy()
            a[t, h] += eps
            b[t, h] -= eps
            fa = 0.5 * oracle.indexer_kl(q, k, a, idx, prob, 1.0)[0].sum()
            fb = 0.5 * oracle.indexer_kl(q, k, b, idx, prob, 1.0)[0].sum()
            np.testing.assert_allclose(dw[t, h], (fa - fb) / (2 * eps), rtol=1e-6, atol=1e-9)


# ---------------------------------------------------------------------------
# k-pool selection (GLM-5.3-Flash; readings in the oracle source)
# ---------------------------------------------------------------------------
def enumerate_pools(cu, P):
    """Independent route: list every complete pool (sequence, first token) in order."""
    pools = []
    for i in range(len(cu) - 1):
        a, b = int(cu[i]), int(cu[i + 1])
        for f in range(a, b - P + 1, P):
            pools.append((i, f))
    return pools


@pytest.mark.parametrize("P", [1, 3, 4])
def test_kpool_metadata_by_enumeration(P):
    cu = np.array([0, 9, 9, 11, 30, 34], np.int32)  # an empty sequence, one shorter than a pool
    T = int(cu[-1])
    pool_cu, ps, npl, ts, total = oracle.kpool_metadata(cu, T, P)
    pools = enumerate_pools(cu, P)
    assert total == len(pools)
    for i in range(len(cu) - 1):
        assert pool_cu[i] == sum(1 for (j, _) in pools if j < i)
    for t in range(T):
        i = int(np.searchsorted(cu, t, side="right")) - 1
        mine = [g for g, (j, f) in enumerate(pools) if j == i and f + P - 1 <= t]
        assert npl[t] == len(mine)
        assert ps[t] == sum(1 for (j, _) in pools if j < i)
        if mine:
            assert mine == list(range(ps[t], ps[t] + npl[t]))
        # the tail: tokens of t's sequence after its last complete pool, up to t
        last_end = pools[mine[-1]][1] + P if mine else int(cu[i])
        assert ts[t] == last_end and 0 <= t + 1 - ts[t] <= P - 1


def test_kpool_metadata_rejects_bad_input():
    with pytest.raises(ValueError):
        oracle.kpool_metadata(np.array([0, 5, 4], np.int32), 4, 4)
    with pytest.raises(ValueError):
        oracle.kpool_metadata(np.array([0, 4], np.int32), 4, 0)


def test_kpool_pool_is_the_numpy_mean_and_the_bf16_rounding_of_torch():
    cu = np.array([0, 10, 10, 23], np.int32)
    P, D = 4, 6
    x = torch.randn(23, D, generator=torch.Generator().manual_seed(41)).to(torch.bfloat16)
    xf = x.double().numpy()
    ref = []
    for i in range(len(cu) - 1):
        a, b = int(cu[i]), int(cu[i + 1])
        n = (b - a) // P
        if n:
            ref.append(xf[a:a + n * P].reshape(n, P, D).mean(axis=1))
    ref = np.concatenate(ref)
    exact = oracle.kpool_pool(x, cu, P, round_to_bf16=False)
    assert np.array_equal(exact, ref)
    rounded = oracle.kpool_pool(x, cu, P)
    assert np.array_equal(rounded, torch.from_numpy(ref).float().to(torch.bfloat16).double().numpy())
    # a pool of identical rows is that row
    same = np.repeat(xf[:1], 8, axis=0)
    assert np.array_equal(oracle.kpool_pool(same, np.array([0, 8], np.int32), 4), same[:2])


def test_kpool_unpool_grad_is_the_adjoint_of_pooling():
    # x -> [pool(x); x] is linear; the key gradient must be its transpose: <A x, y> = <x, A^T y>
    rng = np.random.default_rng(42)
    cu = np.array([0, 13, 13, 30, 33], np.int32)
    T, D, P = 33, 5, 4
    x = rng.standard_normal((T, D))
    pooled = oracle.kpool_pool(x, cu, P, round_to_bf16=False)
    total = pooled.shape[0]
    y = rng.standard_normal((total + T, D))
    lhs = float(np.sum(np.concatenate([pooled, x]) * y))
    rhs = float(np.sum(x * oracle.kpool_unpool_grad(y, cu, P, total)))
    assert lhs == pytest.approx(rhs, rel=1e-13, abs=1e-13)


def test_kpool_topk_with_pools_of_one_token_is_the_token_indexer():
    rng = np.random.default_rng(43)
    cu = np.array([0, 19, 40], np.int32)
    T, K = 40, 6
    q = torch.randn(T, 3, 8, generator=torch.Generator().manual_seed(44)).to(torch.bfloat16)
    k = torch.randn(T, 8, generator=torch.Generator().manual_seed(45)).to(torch.bfloat16)
    w = rng.uniform(0, 1, (T, 3))
    _, ps, npl, ts, total = oracle.kpool_metadata(cu, T, 1)
    kp = oracle.kpool_pool(k, cu, 1)
    assert total == T and np.array_equal(kp, k.double().numpy())
    idx, ln, _ = oracle.kpool_topk(q, kp, w, np.arange(T), ps, npl, ts, total, K, 1)
    st, _, _, _ = oracle.packed_metadata(cu, T)
    ref, rln, _ = oracle.indexer_topk(q, k, w, st, np.arange(T), K)
    assert np.array_equal(idx, ref) and np.array_equal(ln, rln)


def test_kpool_topk_increasing_pool_scores_pick_the_latest_pools_and_the_tail():
    cu = np.array([0, 23, 41], np.int32)
    T, Di, K, P = 41, 4, 3, 4
    k = np.zeros((T, Di))
    for i in range(len(cu) - 1):  # every token of pool p (in its sequence) = alpha (p+1) e0
        for t in range(int(cu[i]), int(cu[i + 1])):
            k[t, 0] = 0.5 * ((t - int(cu[i])) // P + 1)
    q = np.abs(np.random.default_rng(46).standard_normal((T, 2, Di))) + 0.1
    w = np.full((T, 2), 0.25)
    _, ps, npl, ts, total = oracle.kpool_metadata(cu, T, P)
    kp = oracle.kpool_pool(k, cu, P)
    idx, ln, _ = oracle.kpool_topk(q, kp, w, np.arange(T), ps, npl, ts, total, K, P)
    for t in range(T):
        n = min(K, int(npl[t]))
        pools = list(range(ps[t] + npl[t] - n, ps[t] + npl[t]))
        tail = [total + s for s in range(ts[t], t + 1)]
        want = pools + tail
        assert idx[t].tolist() == want + [-1] * (K + P - 1 - len(want)), t
        assert ln[t] == len(want)


def test_kpool_topk_brute_force():
    rng = np.random.default_rng(47)
    cu = np.array([0, 30, 37, 64], np.int32)
    T, Hi, Di, K, P = 64, 3, 6, 4, 4
    q = rng.standard_normal((T, Hi, Di))
    k = rng.standard_normal((T, Di))
    w = rng.uniform(-0.1, 1, (T, Hi))
    _, ps, npl, ts, total = oracle.kpool_metadata(cu, T, P)
    kp = oracle.kpool_pool(k, cu, P, round_to_bf16=False)
    idx, ln, _ = oracle.kpool_topk(q, kp, w, np.arange(T), ps, npl, ts, total, K, P)
    S = numpy_indexer_scores(q, kp, w)
    for t in range(T):
        cand = sorted(range(ps[t], ps[t] + npl[t]), key=lambda p: (-S[t, p], p))
        sel = sorted(cand[:K]) + [total + s for s in range(ts[t], t + 1)]
        assert idx[t].tolist() == sel + [-1] * (K + P - 1 - len(sel)), t
