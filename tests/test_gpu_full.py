"""Full-size checks: the pages' workloads at their full sizes, in the launch
configuration the benchmark times (the forward's residual of O passed to the
backward), against the fp64 oracle.

  * V3.2 layout and NoPE: dq of every query row and dkv of every key row,
    element by element (the oracle runs every row, in chunks whose key
    gradients accumulate, as query chunks do);
  * the 32k indexer -> MLA path and the THD IndexShare layers, where the
    oracle cannot run every row: out / lse / dq on sampled rows the oracle
    computes one by one (query rows are independent), dkv restricted to a
    chunk of rows (a call on those rows) against the oracle's dkv of exactly
    those rows at full T_k and K, and the dkv column sums
    sum_k dkv[k,c] = sum_{t,h nonempty} dO[t,h,c] (c < 512), 0 for RoPE;
  * query chunks give the same outputs as one shot.
Inputs are drawn on the GPU with the seeded recipe (sparse_attention_mla_gb300.synth).  Where the
index sets come from the GPU indexer, the oracle computes its own selection of the rows it checks
and runs the attention on its own indices, on the rows whose selection equals the GPU's.
"""
import numpy as np
import pytest
import torch

import oracle
import sparse_attention_mla_gb300 as dsa
from sparse_attention_mla_gb300 import synth

from _cmp import assert_close, assert_lse
from test_gpu_indexer import check_rows, oracle_start

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
ORACLE_CHUNK_BYTES = 6e8  # the oracle keeps P and dS (fp64) of the rows of one chunk


def causal_idx_gpu(seq_start, K, seed, T):
    """Random causal index sets drawn on the GPU: uniform n-subset of [start, t], ascending, -1 suffix."""
    g = torch.Generator(device=DEV)
    g.manual_seed(seed)
    st = seq_start.to(DEV).long()
    idx = torch.full((T, K), -1, dtype=torch.int32, device=DEV)
    for a in range(0, T, 1024):
        b = min(T, a + 1024)
        t = torch.arange(a, b, device=DEV)
        c = t - st[a:b] + 1
        cmax = int(c.max())
        r = torch.rand(b - a, cmax, generator=g, device=DEV)
        r.masked_fill_(torch.arange(cmax, device=DEV)[None, :] >= c[:, None], -1.0)
        kk = min(K, cmax)
        v, i = r.topk(kk, dim=1)
        i = torch.where(v >= 0, i + st[a:b, None], torch.full_like(i, 1 << 30)).sort(dim=1).values
        i = torch.where(i == (1 << 30), torch.full_like(i, -1), i)
        idx[a:b, :kk] = i.to(torch.int32)
    return idx


def sample_rows(T, starts_of_interest, n_random=12, seed=0):
    g = np.random.default_rng(seed)
    rows = set(int(x) for x in starts_of_interest if 0 <= x < T)
    rows |= set(g.integers(0, T, n_random).tolist())
    return np.array(sorted(rows))


def matching_rows(idx, ln, rows, sel):
    """Rows whose GPU selection equals the oracle's own (sel = (idx, len) of `rows`), with the
    oracle's indices of those rows."""
    ridx, rlen = sel
    g = idx[torch.as_tensor(rows)].cpu().numpy()
    gl = ln[torch.as_tensor(rows)].cpu().numpy()
    same = np.all(g == ridx, axis=1) & (gl == rlen)
    assert same.mean() >= 0.9, f"only {same.sum()} of {len(rows)} rows select as the oracle does"
    return np.asarray(rows)[same], torch.as_tensor(ridx[same]), torch.as_tensor(rlen[same])


def mla_full_check(q, kv, dout, idx, scale, ln=None, rows=None, chunk=(0, 64), Dv=512, every_row=False,
                   ref_sel=None, chunk_sel=None):
    """fwd+bwd of the whole problem as the benchmark runs it, then out/lse on the sampled rows and
    either (every_row) dq of every row and the whole dkv element by element, or dq on the sampled
    rows, the dkv column sums and the exact dkv of one chunk of rows.  When the index sets come
    from the GPU indexer, ref_sel / chunk_sel carry the oracle's own selection of `rows` / of the
    chunk's rows: the oracle then runs on its own indices, on the rows where they equal the GPU's."""
    T, H = q.shape[0], q.shape[1]
    K = idx.shape[1]
    wf = torch.zeros(dsa.workspace_size("fwd", T, H), dtype=torch.uint8, device=DEV)
    wb = torch.zeros(dsa.workspace_size("bwd", T, H, K), dtype=torch.uint8, device=DEV)
    out, lse, lo = dsa.dsa_sparse_mla_fwd(q, kv, idx, scale, topk_len=ln, out_lo=True, workspace=wf)
    dq, dkv, _ = dsa.dsa_sparse_mla_bwd(q, kv, idx, scale, out, lse, dout, topk_len=ln, out_lo=lo, workspace=wb)
    assert dsa.dsa_read_device_status(wf) == 0 and dsa.dsa_read_device_status(wb) == 0
    kvc = kv.cpu()
    if ref_sel is not None:
        rows, ridx, rlen = matching_rows(idx, ln, rows, ref_sel)
    r = torch.as_tensor(rows)
    if ref_sel is None:  # seeded index sets: the same input on both sides
        ridx, rlen = idx[r].cpu(), None if ln is None else ln[r].cpu()
    ln_r = rlen
    ref_o, ref_l = oracle.sparse_mla_fwd(q[r].cpu(), kvc, ridx, scale, len_rows=ln_r)
    assert_close(out[r].cpu(), ref_o, "out (sampled rows)")
    assert_lse(lse[r].cpu(), ref_l)
    if every_row:
        ref_dkv = np.zeros((kv.shape[0], kv.shape[1]), np.float64)
        step = max(1, int(ORACLE_CHUNK_BYTES // (H * K * 16)))
        for a in range(0, T, step):
            b = min(T, a + step)
            ref_dq, _ = oracle.sparse_mla_bwd(q[a:b].cpu(), kvc, idx[a:b].cpu(), dout[a:b].cpu(), scale,
                                              len_rows=None if ln is None else ln[a:b].cpu(), dkv=ref_dkv)
            assert_close(dq[a:b].cpu(), ref_dq, f"dq rows {a}:{b}")
        assert_close(dkv.cpu(), ref_dkv, "dkv (every key row)")
        return out, lse, lo, dq, dkv
    ref_dq, _ = oracle.sparse_mla_bwd(q[r].cpu(), kvc, ridx, dout[r].cpu(), scale, len_rows=ln_r)
    assert_close(dq[r].cpu(), ref_dq, "dq (sampled rows)")
    # column sums of the full dkv
    valid = (idx >= 0) if ln is None else ((idx >= 0) & (torch.arange(K, device=DEV)[None, :] < ln[:, None]))
    nonempty = valid.any(dim=1)
    col = dkv.double().sum(0).cpu().numpy()
    ref = torch.zeros(dout.shape[-1], dtype=torch.float64, device=DEV)
    for a in range(0, dout.shape[0], 4096):
        ref += dout[a:a + 4096][nonempty[a:a + 4096]].double().sum((0, 1))
    ref = ref.cpu().numpy()
    scale_ref = max(1.0, float(np.abs(ref).max()))
    assert np.max(np.abs(col[:Dv] - ref)) <= 2e-2 * scale_ref, "dkv column sums (value channels)"
    assert np.max(np.abs(col[Dv:])) <= 2e-2 * scale_ref if col.shape[0] > Dv else True
    # exact dkv of a chunk of rows, at full T_k and K
    a, b = chunk
    if chunk_sel is None:
        cr, cidx, clen = torch.arange(a, b), idx[a:b].cpu(), None if ln is None else ln[a:b].cpu()
    else:
        crows, cidx, clen = matching_rows(idx, ln, np.arange(a, b), chunk_sel)
        cr = torch.as_tensor(crows)
    g = lambda x: x[cr.to(x.device)].contiguous()
    _, dkv_c, _ = dsa.dsa_sparse_mla_bwd(g(q), kv, g(idx), scale, g(out), g(lse), g(dout),
                                         topk_len=None if ln is None else g(ln), out_lo=g(lo), workspace=wb)
    assert dsa.dsa_read_device_status(wb) == 0
    _, ref_c = oracle.sparse_mla_bwd(q[cr.to(q.device)].cpu(), kvc, cidx, dout[cr.to(q.device)].cpu(), scale,
                                     len_rows=clen)
    assert_close(dkv_c.cpu(), ref_c, f"dkv of rows {a}:{b}")
    return out, lse, lo, dq, dkv


def test_full_v32_layout_S4096_H128_K2048():
    # DeepSeek-V3.2 layout: 1 sequence, S=4096, H=128, width 576, K=2048 random causal, scale 192^-0.5
    c = synth.WORKLOADS["v32"]
    T = c["T"]
    x = synth.mla_inputs(T, c["H"], c["Dqk"], c["Dv"], seed=2, device=DEV)
    idx = causal_idx_gpu(torch.zeros(T, dtype=torch.int32), c["K"], 2, T)
    rows = np.union1d(sample_rows(T, [0, 1, 2, 63, 2047, 2048, 2049, T - 1], n_random=0, seed=2),
                      np.random.default_rng(2).choice(T, 2048, replace=False))  # >= 2048 distinct rows
    mla_full_check(x["q"], x["kv"], x["dout"], idx, c["scale"], rows=rows, every_row=True)


def test_full_indexer_32k_then_sparse_mla_H64():
    # the benchmark's workload: S=32768, indexer 64x128, K=2048, then H=64 sparse MLA fwd+bwd at width 576
    c = synth.WORKLOADS["idx32k"]
    T, K = c["T"], c["K"]
    ind = synth.indexer_inputs(T, c["Hi"], c["Di"], seed=3, device=DEV)
    cu = torch.tensor([0, T], dtype=torch.int32, device=DEV)
    start, _, _, _ = dsa.dsa_packed_metadata(cu, T)
    ws = torch.zeros(dsa.workspace_size("indexer", T, K), dtype=torch.uint8, device=DEV)
    idx, ln = dsa.dsa_indexer_topk(ind["q_idx"], ind["k_idx"], ind["w"], start, K, workspace=ws)
    assert dsa.dsa_read_device_status(ws) == 0
    # >= 2048 distinct rows of the indexer against the oracle's full-window top-k; the MLA checks run
    # on a subset of them with the oracle's own selection
    rows = sample_rows(T, [0, 1, 2047, 2048, 2049, 16383, T - 2, T - 1], n_random=24, seed=3)
    mla_rows = np.union1d(rows, np.random.default_rng(33).choice(T, 512, replace=False))  # oracle time bounds this
    chunk_rows = np.arange(T - 32, T)
    all_rows = np.union1d(np.union1d(mla_rows, chunk_rows), np.random.default_rng(3).choice(T, 2048, replace=False))
    qi = ind["q_idx"].cpu()
    ref = {}
    check_rows(idx.cpu().numpy(), ln.cpu().numpy(), qi, ind["k_idx"].cpu(), ind["w"].cpu(),
               oracle_start(cu, T, start), all_rows, K, ref_out=ref)
    pick = lambda rr: (ref["idx"][np.searchsorted(all_rows, rr)], ref["len"][np.searchsorted(all_rows, rr)])
    x = synth.mla_inputs(T, c["H"], c["Dqk"], c["Dv"], seed=4, device=DEV)
    mla_full_check(x["q"], x["kv"], x["dout"], idx, c["scale"], ln=ln, rows=mla_rows, chunk=(T - 32, T),
                   ref_sel=pick(mla_rows), chunk_sel=pick(chunk_rows))


def test_full_nope_S16384_H8_K2051_and_query_chunks():
    # GLM-5.3-Flash NoPE: S=16384, H=8, width 512, unaligned K=2051, scale 512^-0.5; 4096-token chunks = one shot
    c = synth.WORKLOADS["nope"]
    T, K = c["T"], c["K"]
    x = synth.mla_inputs(T, c["H"], c["Dqk"], c["Dv"], seed=5, device=DEV)
    idx = causal_idx_gpu(torch.zeros(T, dtype=torch.int32), K, 5, T)
    rows = np.union1d(sample_rows(T, [0, 1, 2050, 2051, 2052, T - 1], n_random=0, seed=5),
                      np.random.default_rng(5).choice(T, 2048, replace=False))
    out, lse, lo, dq, dkv = mla_full_check(x["q"], x["kv"], x["dout"], idx, c["scale"], rows=rows, every_row=True)
    acc = None
    for a in range(0, T, 4096):
        b = min(T, a + 4096)
        o_c, l_c, lo_c = dsa.dsa_sparse_mla_fwd(x["q"][a:b], x["kv"], idx[a:b], c["scale"], out_lo=True)
        assert torch.equal(o_c, out[a:b]) and torch.equal(l_c, lse[a:b])
        dq_c, acc, _ = dsa.dsa_sparse_mla_bwd(x["q"][a:b], x["kv"], idx[a:b], c["scale"], o_c, l_c, x["dout"][a:b],
                                              dkv_accum=acc, accumulate=acc is not None, out_lo=lo_c)
        assert torch.equal(dq_c, dq[a:b])
    assert_close(acc.cpu(), dkv.cpu().double(), "chunked dkv", max_abs=1e-3, rel_fro=1e-5)


def test_full_thd_packed_indexshare_4_layers():
    # 8 sequences, lengths U[4096, 32768] rescaled to 131072 tokens; indexer once, its top-k reused by 4 layers
    c = synth.WORKLOADS["thd"]
    T, K = c["T"], c["K"]
    lens = synth.thd_lengths(c["nseq"], c["lo"], c["hi"], T, synth.generator(6))
    cu = synth.cu_seqlens_from_lengths(lens)
    start, clen, mx, ne = dsa.dsa_packed_metadata(cu.to(DEV), T)
    st_ref, cl_ref, mx_ref, _ = oracle.packed_metadata(cu.numpy(), T)
    assert np.array_equal(start.cpu().numpy(), st_ref) and np.array_equal(clen.cpu().numpy(), cl_ref)
    assert mx == mx_ref == max(lens) and ne == 1
    ind = synth.indexer_inputs(T, c["Hi"], c["Di"], seed=6, device=DEV)
    ws = torch.zeros(dsa.workspace_size("indexer", T, K), dtype=torch.uint8, device=DEV)
    idx, ln = dsa.dsa_indexer_topk(ind["q_idx"], ind["k_idx"], ind["w"], start, K, workspace=ws)
    assert dsa.dsa_read_device_status(ws) == 0
    cuts = cu.tolist()
    rows = sample_rows(T, [cuts[1] - 1, cuts[1], cuts[1] + 1, cuts[4] + 2047, cuts[4] + 2048, T - 1], n_random=6,
                       seed=6)
    chunk_rows = np.arange(cuts[5] - 16, cuts[5] + 16)
    all_rows = np.union1d(rows, chunk_rows)
    ref = {}
    check_rows(idx.cpu().numpy(), ln.cpu().numpy(), ind["q_idx"].cpu(), ind["k_idx"].cpu(), ind["w"].cpu(),
               st_ref, all_rows, K, ref_out=ref)
    pick = lambda rr: (ref["idx"][np.searchsorted(all_rows, rr)], ref["len"][np.searchsorted(all_rows, rr)])
    # packing is exact: one sequence run alone gives the same indices (shifted by its offset)
    a, b = cuts[2], cuts[3]
    cu1 = torch.tensor([0, b - a], dtype=torch.int32, device=DEV)
    s1, _, _, _ = dsa.dsa_packed_metadata(cu1, b - a)
    idx1, ln1 = dsa.dsa_indexer_topk(ind["q_idx"][a:b], ind["k_idx"][a:b], ind["w"][a:b], s1, K)
    shifted = torch.where(idx1 >= 0, idx1 + a, idx1)
    assert torch.equal(shifted, idx[a:b]) and torch.equal(ln1, ln[a:b])
    # IndexShare: the same index tensor drives 4 layers with independent q / kv / dO
    idx_before = idx.clone()
    for layer in range(c["layers"]):
        x = synth.mla_inputs(T, c["H"], c["Dqk"], 512, seed=100 + layer, device=DEV)
        mla_full_check(x["q"], x["kv"], x["dout"], idx, c["scale"], ln=ln, rows=rows[::3],
                       chunk=(cuts[5] - 16, cuts[5] + 16), ref_sel=pick(rows[::3]), chunk_sel=pick(chunk_rows))
        del x
        torch.cuda.empty_cache()
    assert torch.equal(idx, idx_before)


def test_full_indexer_kl_32k_after_the_backward():
    # the indexer KL loss on the 32k workload: indexer -> sparse MLA fwd -> bwd (slot probabilities) -> KL.
    # Sampled rows against the oracle (slot probability, kl, dq_idx, dw), and dk_idx of a chunk of rows
    # exactly (a call on those rows)
    c = synth.WORKLOADS["idx32k"]
    T, K = c["T"], c["K"]
    ind = synth.indexer_inputs(T, c["Hi"], c["Di"], seed=8, device=DEV)
    cu = torch.tensor([0, T], dtype=torch.int32, device=DEV)
    start, _, _, _ = dsa.dsa_packed_metadata(cu, T)
    idx, ln, isc = dsa.dsa_indexer_topk_scored(ind["q_idx"], ind["k_idx"], ind["w"], start, K)
    x = synth.mla_inputs(T, c["H"], c["Dqk"], c["Dv"], seed=9, device=DEV)
    out, lse, lo = dsa.dsa_sparse_mla_fwd(x["q"], x["kv"], idx, c["scale"], topk_len=ln, out_lo=True)
    wb = torch.zeros(dsa.workspace_size("bwd", T, c["H"], K), dtype=torch.uint8, device=DEV)
    *_, prob = dsa.dsa_sparse_mla_bwd(x["q"], x["kv"], idx, c["scale"], out, lse, x["dout"], topk_len=ln,
                                      out_lo=lo, workspace=wb, attn_prob=True)
    assert dsa.dsa_read_device_status(wb) == 0
    del wb, out, lo
    ws = torch.zeros(4096, dtype=torch.uint8, device=DEV)
    # the KL twice: forming the slots' indexer scores itself, and reading the selection's own scores
    runs = [dsa.dsa_indexer_kl(ind["q_idx"], ind["k_idx"], ind["w"], idx, prob, 1.0, topk_len=ln, workspace=ws,
                               topk_score=s_) for s_ in (None, isc)]
    assert dsa.dsa_read_device_status(ws) == 0
    del isc
    # the oracle's own chain for the checked rows: its selection, its slot probabilities, its loss
    rows = sample_rows(T, [0, 1, 2047, 2048, T - 1], n_random=43, seed=8)
    chunk_rows = np.arange(T - 40, T)
    all_rows = np.union1d(rows, chunk_rows)
    ref = {}
    check_rows(idx.cpu().numpy(), ln.cpu().numpy(), ind["q_idx"].cpu(), ind["k_idx"].cpu(), ind["w"].cpu(),
               oracle_start(cu, T, start), all_rows, K, ref_out=ref)
    pick = lambda rr: (ref["idx"][np.searchsorted(all_rows, rr)], ref["len"][np.searchsorted(all_rows, rr)])
    rows, ridx, rlen = matching_rows(idx, ln, rows, pick(rows))
    r = torch.as_tensor(rows)
    ref_p = oracle.attn_slot_prob(x["q"][r].cpu(), x["kv"].cpu(), ridx, c["scale"], len_rows=rlen)
    assert np.max(np.abs(prob[r].cpu().double().numpy() - ref_p)) <= 1e-5, "slot probability (sampled rows)"
    rkl, rdq, rdw, _ = oracle.indexer_kl(ind["q_idx"][r].cpu(), ind["k_idx"].cpu(), ind["w"][r].cpu(), ridx,
                                         ref_p, 1.0, len_rows=rlen)
    for how, (kl, dq, dw, _) in zip(("formed scores", "read scores"), runs):
        assert np.max(np.abs(kl[r].cpu().double().numpy() - rkl) / np.maximum(1.0, np.abs(rkl))) <= 1e-4, how
        assert_close(dq[r].cpu(), rdq, f"dq_idx (sampled rows, {how})", max_abs=2e-3 * float(np.abs(rdq).max()))
        assert_close(dw[r].cpu(), rdw, f"dw (sampled rows, {how})", max_abs=2e-3 * float(np.abs(rdw).max()),
                     rel_fro=1e-4)
    del runs
    # dk_idx of the chunk's rows whose selection matches, each side from its own probabilities
    crows, cidx, clen = matching_rows(idx, ln, chunk_rows, pick(chunk_rows))
    cr = torch.as_tensor(crows)
    g = lambda t_: t_[cr.to(t_.device)].contiguous()
    _, _, _, dk_c = dsa.dsa_indexer_kl(g(ind["q_idx"]), ind["k_idx"], g(ind["w"]), g(idx), g(prob), 1.0,
                                       topk_len=g(ln), workspace=ws)
    assert dsa.dsa_read_device_status(ws) == 0
    cp_ref = oracle.attn_slot_prob(g(x["q"]).cpu(), x["kv"].cpu(), cidx, c["scale"], len_rows=clen)
    _, _, _, ref_c = oracle.indexer_kl(g(ind["q_idx"]).cpu(), ind["k_idx"].cpu(), g(ind["w"]).cpu(), cidx, cp_ref,
                                       1.0, len_rows=clen)
    assert_close(dk_c.cpu(), ref_c, f"dk_idx of rows {chunk_rows[0]}:{chunk_rows[-1] + 1}",
                 max_abs=2e-3 * float(np.abs(ref_c).max()), rel_fro=1e-4)


def test_full_kpool_glm_flash_S16384_H8_K2048_plus_tail():
    """GLM-5.3-Flash k-pool selection at full size (the kpool workload of the benchmark): NoPE
    width 512, H = 8, 4096 pools of 4 tokens, K = 2048 pools + the 3-token tail.  The oracle makes
    its own pooling and selection for the rows it checks (sampled rows and a chunk of 64 rows);
    rows whose selection equals the GPU's are compared element by element with the oracle's own
    indices (out, lse, dq, and the chunk's dkv over [pooled rows; token rows]), and every checked
    row's pool set must match within the indexer's fp32 tie band."""
    c = synth.WORKLOADS["kpool"]
    T, H, D, P = c["T"], c["H"], c["Dqk"], c["pool"]
    Kp = c["K"] - P + 1
    scale = c["scale"]
    cu = torch.tensor([0, T], dtype=torch.int32)
    ind = synth.indexer_inputs(T, c["Hi"], c["Di"], seed=0, device=DEV)
    x = synth.mla_inputs(T, H, D, c["Dv"], seed=1000, device=DEV)
    meta = dsa.dsa_kpool_metadata(cu.to(DEV), T, P)
    k_pool = dsa.dsa_kpool_pool(ind["k_idx"], meta)
    kv_cat = torch.empty(meta.total_pools + T, D, dtype=torch.bfloat16, device=DEV)
    dsa.dsa_kpool_pool(x["kv"], meta, out=kv_cat[:meta.total_pools])
    kv_cat[meta.total_pools:] = x["kv"]
    idx, ln = dsa.dsa_kpool_topk(ind["q_idx"], k_pool, ind["w"], meta, Kp)
    W = idx.shape[1]
    wf = torch.zeros(dsa.workspace_size("fwd", T, H), dtype=torch.uint8, device=DEV)
    wb = torch.zeros(dsa.workspace_size("bwd", T, H, W), dtype=torch.uint8, device=DEV)
    out, lse, lo = dsa.dsa_sparse_mla_fwd(x["q"], kv_cat, idx, scale, topk_len=ln, out_lo=True, workspace=wf)
    dq, dcat, _ = dsa.dsa_sparse_mla_bwd(x["q"], kv_cat, idx, scale, out, lse, x["dout"], topk_len=ln, out_lo=lo,
                                          workspace=wb)
    dkv = dsa.dsa_kpool_unpool_grad(dcat, meta)
    assert dsa.dsa_read_device_status(wf) == 0 and dsa.dsa_read_device_status(wb) == 0
    # the oracle's own pooling and selection for the checked rows
    _, ps, npl, ts, total = oracle.kpool_metadata(cu, T, P)
    assert total == meta.total_pools
    kp = oracle.kpool_pool(ind["k_idx"].cpu(), cu, P)
    kv_cat_ref = np.concatenate([oracle.kpool_pool(x["kv"].cpu(), cu, P), x["kv"].cpu().double().numpy()])
    a = T - 64
    rows = np.unique(np.concatenate([sample_rows(T, [0, 2, 3, 4, 7, 8190, 8191, T - 1], n_random=16, seed=11),
                                     np.arange(a, T)]))
    qi, wr = ind["q_idx"][torch.as_tensor(rows)].cpu(), ind["w"][torch.as_tensor(rows)].cpu()
    ref_idx, ref_len, kth = oracle.kpool_topk(qi, kp, wr, rows, ps[rows], npl[rows], ts[rows], total, Kp, P)
    gidx, glen = idx[torch.as_tensor(rows)].cpu().numpy(), ln[torch.as_tensor(rows)].cpu().numpy()
    same = np.zeros(len(rows), bool)
    for k, t in enumerate(rows):
        n = int(ref_len[k])
        assert glen[k] == n and np.all(gidx[k, n:] == -1), t
        ntail = t + 1 - int(ts[t])
        assert np.array_equal(gidx[k, n - ntail:n], ref_idx[k, n - ntail:n]), f"row {t}: tail"
        npool = n - ntail
        diff = sorted(set(gidx[k, :npool].tolist()) ^ set(ref_idx[k, :npool].tolist()))
        same[k] = not diff
        if diff:
            sc, mag = oracle.indexer_scores(qi[[k]], kp, wr[[k]], np.zeros(len(diff), np.int64), np.array(diff),
                                            with_magnitude=True)
            ksc, kmag = oracle.indexer_scores(qi[[k]], kp, wr[[k]], np.zeros(npool, np.int64), ref_idx[k, :npool],
                                              with_magnitude=True)
            j = int(np.argmin(ksc))
            for d in range(len(diff)):
                assert abs(sc[d] - kth[k]) <= 200 * 2.0 ** -24 * (mag[d] + kmag[j]), f"row {t}: pool {diff[d]}"
    assert same.mean() >= 0.9
    ok = rows[same]
    r = torch.as_tensor(ok)
    ref_o, ref_l = oracle.sparse_mla_fwd(x["q"][r].cpu(), kv_cat_ref, ref_idx[same], scale, Dv=512,
                                         len_rows=ref_len[same])
    assert_close(out[r].cpu(), ref_o, "out (checked rows)")
    assert_lse(lse[r].cpu(), ref_l)
    ref_dq, _ = oracle.sparse_mla_bwd(x["q"][r].cpu(), kv_cat_ref, ref_idx[same], x["dout"][r].cpu(), scale,
                                      Dv=512, len_rows=ref_len[same])
    assert_close(dq[r].cpu(), ref_dq, "dq (checked rows)")
    # dkv over [pooled rows; token rows] from the chunk's rows whose selection matched, and the
    # token gradient through the pooling
    cr = torch.as_tensor(ok[ok >= a])
    _, dcat_c, _ = dsa.dsa_sparse_mla_bwd(x["q"][cr].contiguous(), kv_cat, idx[cr].contiguous(), scale,
                                          out[cr].contiguous(), lse[cr].contiguous(), x["dout"][cr].contiguous(),
                                          topk_len=ln[cr].contiguous(), out_lo=lo[cr].contiguous(), workspace=wb)
    assert dsa.dsa_read_device_status(wb) == 0
    sel = np.isin(rows, ok[ok >= a])
    _, ref_dcat = oracle.sparse_mla_bwd(x["q"][cr].cpu(), kv_cat_ref, ref_idx[sel], x["dout"][cr].cpu(), scale,
                                        Dv=512, len_rows=ref_len[sel])
    assert_close(dcat_c.cpu(), ref_dcat, "dkv of the chunk's rows over [pooled; token] rows")
    assert_close(dsa.dsa_kpool_unpool_grad(dcat_c, meta).cpu(), oracle.kpool_unpool_grad(ref_dcat, cu, P, total),
                 "token dkv of the chunk's rows")
    assert dkv.shape == (T, D)
