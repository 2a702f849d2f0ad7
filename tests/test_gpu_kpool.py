"""GPU parity of the k-pool selection (GLM-5.3-Flash) against the fp64 oracle.

Pool coordinates and pooled rows bit for bit; the selected pools as index sets
equal to the oracle's except inside the fp32 tie band of the K-th best pool (as
for the token indexer), the tail tokens exactly; then the whole path -- pooled
kv, sparse MLA forward and backward over [pooled rows; token rows] at width
K + 3, and the key gradient back to the tokens -- element by element."""
import numpy as np
import pytest
import torch

import oracle
import sparse_attention_mla_gb300 as dsa
from sparse_attention_mla_gb300 import synth

from _cmp import assert_close, assert_lse
from test_gpu_indexer import GAMMA

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def t32(a):
    return torch.as_tensor(np.asarray(a), dtype=torch.int32)


@pytest.mark.parametrize("P", [1, 3, 4])
def test_kpool_metadata_and_pooling_match_the_oracle(P):
    cu = t32([0, 9, 9, 11, 300, 301, 517])  # an empty sequence, ones shorter than a pool
    T = int(cu[-1])
    meta = dsa.dsa_kpool_metadata(cu.to(DEV), T, P)
    pool_cu, ps, npl, ts, total = oracle.kpool_metadata(cu, T, P)
    assert meta.total_pools == total
    for got, ref in ((meta.pool_cu, pool_cu), (meta.pool_start, ps), (meta.n_pools, npl), (meta.tail_start, ts)):
        assert np.array_equal(got.cpu().numpy(), ref)
    g = synth.generator(70 + P)
    for D in (128, 576, 512):
        x = synth.randn_bf16((T, D), g)
        got = dsa.dsa_kpool_pool(x.to(DEV), meta)
        ref = oracle.kpool_pool(x, cu, P)
        # the fp32 sum of P bf16 values of these magnitudes is exact, so both round the same mean
        assert np.array_equal(got.cpu().double().numpy(), ref), D


def test_kpool_topk_matches_the_oracle():
    cu = t32([0, 700, 703, 2900])
    T, Hi, K, P = 2900, 64, 128, 4
    g = synth.generator(74)
    q_idx = synth.randn_bf16((T, Hi, 128), g)
    k_idx = synth.randn_bf16((T, 128), g)
    w = torch.rand(T, Hi, generator=g) * 0.1
    meta = dsa.dsa_kpool_metadata(cu.to(DEV), T, P)
    k_pool = dsa.dsa_kpool_pool(k_idx.to(DEV), meta)
    ws = torch.zeros(dsa.load_library().dsa_kpool_topk_workspace_size(T, K), dtype=torch.uint8, device=DEV)
    idx, ln = dsa.dsa_kpool_topk(q_idx.to(DEV), k_pool, w.to(DEV), meta, K, workspace=ws)
    assert dsa.dsa_read_device_status(ws) == 0
    assert idx.shape == (T, K + P - 1)
    gidx, glen = idx.cpu().numpy(), ln.cpu().numpy()
    _, ps, npl, ts, total = oracle.kpool_metadata(cu, T, P)
    kp = oracle.kpool_pool(k_idx, cu, P)
    ref_idx, ref_len, kth = oracle.kpool_topk(q_idx, kp, w, np.arange(T), ps, npl, ts, total, K, P)
    swaps = 0
    for t in range(T):
        n = int(ref_len[t])
        assert glen[t] == n, (t, glen[t], n)
        assert np.all(gidx[t, n:] == -1)
        ntail = t + 1 - int(ts[t])
        npool = n - ntail
        assert np.array_equal(gidx[t, npool:n], ref_idx[t, npool:n]), f"row {t}: tail"  # exact
        sel = gidx[t, :npool]
        assert np.all(np.diff(gidx[t, :n]) > 0), f"row {t} not ascending"
        if npool:
            assert sel.min() >= ps[t] and sel.max() <= ps[t] + npl[t] - 1, t
        diff = sorted(set(sel.tolist()) ^ set(ref_idx[t, :npool].tolist()))
        if diff:
            swaps += len(diff) // 2
            sc, mag = oracle.indexer_scores(q_idx[[t]], kp, w[[t]], np.zeros(len(diff), np.int64), np.array(diff),
                                            with_magnitude=True)
            ksc, kmag = oracle.indexer_scores(q_idx[[t]], kp, w[[t]], np.zeros(npool, np.int64),
                                              ref_idx[t, :npool], with_magnitude=True)
            j = int(np.argmin(ksc))
            for d in range(len(diff)):
                assert abs(sc[d] - kth[t]) <= GAMMA * (mag[d] + kmag[j]), f"row {t}: pool {diff[d]}"
    assert swaps <= T // 50


def test_kpool_path_through_fwd_bwd_and_the_key_gradient():
    # NoPE width 512 (GLM-5.3-Flash), a few heads, pools of 4, K pools + the tail
    cu = t32([0, 190, 193, 620])
    T, H, D, Hi, K, P = 620, 16, 512, 64, 40, 4
    scale = D ** -0.5
    g = synth.generator(75)
    q_idx = synth.randn_bf16((T, Hi, 128), g)
    k_idx = synth.randn_bf16((T, 128), g)
    w = torch.rand(T, Hi, generator=g) * 0.1
    q = synth.randn_bf16((T, H, D), g)
    kv = synth.randn_bf16((T, D), g)
    dout = synth.randn_bf16((T, H, 512), g)
    # GPU path
    meta = dsa.dsa_kpool_metadata(cu.to(DEV), T, P)
    k_pool = dsa.dsa_kpool_pool(k_idx.to(DEV), meta)
    kv_cat = torch.empty(meta.total_pools + T, D, dtype=torch.bfloat16, device=DEV)
    dsa.dsa_kpool_pool(kv.to(DEV), meta, out=kv_cat[:meta.total_pools])
    kv_cat[meta.total_pools:] = kv.to(DEV)
    idx, ln = dsa.dsa_kpool_topk(q_idx.to(DEV), k_pool, w.to(DEV), meta, K)
    wf = torch.zeros(dsa.workspace_size("fwd", T, H), dtype=torch.uint8, device=DEV)
    wb = torch.zeros(dsa.workspace_size("bwd", T, H, K + P - 1), dtype=torch.uint8, device=DEV)
    out, lse, lo = dsa.dsa_sparse_mla_fwd(q.to(DEV), kv_cat, idx, scale, topk_len=ln, out_lo=True, workspace=wf)
    dq, dcat, _ = dsa.dsa_sparse_mla_bwd(q.to(DEV), kv_cat, idx, scale, out, lse, dout.to(DEV), topk_len=ln,
                                          out_lo=lo, workspace=wb)
    dkv = dsa.dsa_kpool_unpool_grad(dcat, meta)
    assert dsa.dsa_read_device_status(wf) == 0 and dsa.dsa_read_device_status(wb) == 0
    # oracle path, from its own pooling and selection
    _, ps, npl, ts, total = oracle.kpool_metadata(cu, T, P)
    kp = oracle.kpool_pool(k_idx, cu, P)
    ref_idx, ref_len, _ = oracle.kpool_topk(q_idx, kp, w, np.arange(T), ps, npl, ts, total, K, P)
    same = np.all(idx.cpu().numpy() == ref_idx, axis=1)
    assert same.mean() > 0.98  # rows that differ only inside the tie band are compared by the test above
    kv_cat_ref = np.concatenate([oracle.kpool_pool(kv, cu, P), kv.double().numpy()])
    ref_o, ref_l = oracle.sparse_mla_fwd(q, kv_cat_ref, ref_idx, scale, Dv=512, len_rows=ref_len)
    rows = np.nonzero(same)[0]
    assert_close(out.cpu()[rows], ref_o[rows], "out")
    assert_lse(lse.cpu()[rows], ref_l[rows])
    if same.all():
        ref_dq, ref_dcat = oracle.sparse_mla_bwd(q, kv_cat_ref, ref_idx, dout, scale, Dv=512, len_rows=ref_len)
        assert_close(dq.cpu(), ref_dq, "dq")
        assert_close(dcat.cpu(), ref_dcat, "dkv over the attended rows")
        ref_dkv = oracle.kpool_unpool_grad(ref_dcat, cu, P, total)
        assert_close(dkv.cpu(), ref_dkv, "token dkv")


@pytest.mark.parametrize("P", [3, 4])
def test_kpool_unpool_grad_matches_the_oracle(P):
    # the gradient step alone on seeded fp32 rows (a + b / P: one or two fp32 roundings per element)
    cu = t32([0, 41, 41, 44, 200])
    T, D = 200, 576
    meta = dsa.dsa_kpool_metadata(cu.to(DEV), T, P)
    dcat = torch.randn(meta.total_pools + T, D, generator=synth.generator(77))
    got = dsa.dsa_kpool_unpool_grad(dcat.to(DEV), meta).cpu().double().numpy()
    ref = oracle.kpool_unpool_grad(dcat, cu, P, meta.total_pools)
    assert np.max(np.abs(got - ref) / (1.0 + np.abs(ref))) <= 2.0 ** -22


def test_kpool_rows_without_complete_pools_and_empty_calls():
    # sequences shorter than a pool: no pool at all, every row is its tail only
    cu = t32([0, 3, 5, 8])
    T, Hi, K, P = 8, 4, 16, 4
    g = synth.generator(76)
    q_idx = synth.randn_bf16((T, Hi, 128), g)
    w = torch.rand(T, Hi, generator=g)
    meta = dsa.dsa_kpool_metadata(cu.to(DEV), T, P)
    assert meta.total_pools == 0
    k_pool = torch.empty(0, 128, dtype=torch.bfloat16, device=DEV)
    idx, ln = dsa.dsa_kpool_topk(q_idx.to(DEV), k_pool, w.to(DEV), meta, K)
    _, ps, npl, ts, total = oracle.kpool_metadata(cu, T, P)
    ref_idx, ref_len, _ = oracle.kpool_topk(q_idx, np.zeros((0, 128)), w, np.arange(T), ps, npl, ts, total, K, P)
    assert np.array_equal(idx.cpu().numpy(), ref_idx) and np.array_equal(ln.cpu().numpy(), ref_len)
    # the gradient step with no pool is the identity on the token rows
    dcat = torch.randn(T, 64, device=DEV)
    assert torch.equal(dsa.dsa_kpool_unpool_grad(dcat, meta), dcat)
