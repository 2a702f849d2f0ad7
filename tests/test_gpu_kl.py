"""Indexer KL auxiliary loss: the backward's head-averaged slot probability and
dsa_indexer_kl (loss per row and its gradients) against the fp64 oracle.

Reading (the pages give only the intent; see the oracle): per row over its
selected slots, p = the attention's slot probability averaged over heads and
normalised, q = softmax of the indexer scores, kl = sum p (log p - log q),
gradients of coeff * sum kl back through the indexer score.  The tests use
coeff = 1 so that the gradients are of unit-test size; the kernel's
arithmetic does not depend on it."""
import numpy as np
import pytest
import torch

import oracle
import sparse_attention_mla_gb300 as dsa
from sparse_attention_mla_gb300 import synth

from _cmp import assert_close, errors, storage_half_ulp, to64
from test_gpu_fwd import make_case

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def gpu_prob(q, kv, dout, idx, scale, ln=None, sink=None):
    qd, kvd, idd, dod = q.to(DEV), kv.to(DEV), idx.to(DEV), dout.to(DEV)
    lnd = None if ln is None else ln.to(DEV)
    sd = None if sink is None else sink.to(DEV)
    out, lse, lo = dsa.dsa_sparse_mla_fwd(qd, kvd, idd, scale, topk_len=lnd, out_lo=True, attn_sink=sd)
    ws = torch.zeros(dsa.workspace_size("bwd", q.shape[0], q.shape[1], idx.shape[1]), dtype=torch.uint8, device=DEV)
    res = dsa.dsa_sparse_mla_bwd(qd, kvd, idd, scale, out, lse, dod, topk_len=lnd, out_lo=lo, attn_sink=sd,
                                 workspace=ws, attn_prob=True)
    assert dsa.dsa_read_device_status(ws) == 0
    return res[-1]


@pytest.mark.parametrize("H,Dqk,K,with_sink", [(64, 576, 300, False), (128, 512, 261, True), (16, 576, 64, False)])
def test_backward_slot_probability_matches_oracle(H, Dqk, K, with_sink):
    q, kv, dout, idx = make_case(40, 500, H, Dqk, K, 61)
    idx[3, 7] = -1
    idx[5, :] = -1  # empty row: all zero
    sink = (torch.randn(H, generator=torch.Generator().manual_seed(61)) if with_sink else None)
    prob = gpu_prob(q, kv, dout, idx, 192 ** -0.5, sink=sink)
    ref = oracle.attn_slot_prob(q, kv, idx, 192 ** -0.5, Dv=512, sink=sink)
    g = to64(prob)
    assert np.max(np.abs(g - ref)) <= 1e-5, np.max(np.abs(g - ref))
    assert np.all(g[5] == 0.0)
    if not with_sink:
        rows = (idx >= 0).any(dim=1).numpy()
        np.testing.assert_allclose(g[rows].sum(axis=1), 1.0, atol=1e-5)


def kl_inputs(T, Tk, K, Hi, seed, ln_frac=None):
    x = synth.indexer_inputs(Tk, Hi, 128, seed=seed)
    g = synth.generator(seed + 1)
    q_idx, w = x["q_idx"][:T].contiguous(), x["w"][:T].contiguous()
    idx = torch.stack([torch.randperm(Tk, generator=g)[:K].sort().values for _ in range(T)]).to(torch.int32)
    prob = torch.rand(T, K, generator=g, dtype=torch.float64)
    prob = (prob ** 4).float()  # a peaked target
    ln = None
    if ln_frac is not None:
        ln = (torch.rand(T, generator=g) * (K + 1) * ln_frac).to(torch.int32)
    return q_idx, x["k_idx"], w, idx, prob, ln


def check_kl(q_idx, k_idx, w, idx, prob, coeff=1.0, ln=None, topk_score=None, ref=None):
    """The GPU's KL on (idx, prob, ln[, topk_score]) against the oracle's on ref = (idx, prob, ln): the
    same seeded inputs by default, or the oracle's own selection and target where the GPU's come from
    GPU kernels (they must then name the same slots)."""
    ws = torch.zeros(4096, dtype=torch.uint8, device=DEV)
    dev = lambda t_: None if t_ is None else t_.to(DEV)
    kl, dq, dw, dk = dsa.dsa_indexer_kl(dev(q_idx), dev(k_idx), dev(w), dev(idx), dev(prob), coeff, topk_len=dev(ln),
                                        workspace=ws, topk_score=dev(topk_score))
    assert dsa.dsa_read_device_status(ws) == 0
    r_idx, r_prob, r_ln = (idx, prob, ln) if ref is None else ref
    rkl, rdq, rdw, rdk = oracle.indexer_kl(q_idx, k_idx, w, r_idx, r_prob, coeff, len_rows=r_ln)
    gkl = to64(kl)
    assert np.max(np.abs(gkl - rkl) / np.maximum(1.0, np.abs(rkl))) <= 1e-4, "kl"
    for got, ref, name in ((dq, rdq, "dq_idx"), (dw, rdw, "dw"), (dk, rdk, "dk_idx")):
        scale = max(float(np.max(np.abs(ref))), 1e-30)
        d = np.abs(to64(got) - ref) - storage_half_ulp(got)
        assert float(np.max(d)) <= 2e-3 * scale, f"{name}: max error {float(np.max(d)):.3e} vs scale {scale:.3e}"
        _, rf = errors(got, ref)
        assert rf <= (5e-3 if name == "dq_idx" else 1e-4), f"{name}: rel_fro={rf:.3e}"
    return kl, dq, dw, dk


def test_kl_several_tiles_ragged_holes_and_special_rows():
    q_idx, k_idx, w, idx, prob, _ = kl_inputs(24, 900, 300, 64, 71)
    idx[2, 10] = -1          # a hole
    idx[4, :] = -1           # empty row: kl = 0, no gradient
    idx[6, 1:] = -1          # one valid slot: p = q = 1
    prob[8] = 0.0            # target sums to 0: kl = 0, no gradient
    kl, dq, dw, _ = check_kl(q_idx, k_idx, w, idx, prob)
    for r in (4, 6, 8):
        assert float(kl[r]) == 0.0 or abs(float(kl[r])) < 1e-6
        assert torch.all(dw[r] == 0)


def _slot_scores_fp32(q_idx, k_idx, w, idx):
    # the slots' indexer scores in fp64 by torch (not the oracle), stored as fp32 like the indexer's output;
    # holes and slots past a row's prefix get NaN, which the kernel must never read
    qd, kd, wd = q_idx.double(), k_idx.double(), w.double()
    safe = idx.clamp(min=0).long()
    I = torch.einsum("th,thj->tj", wd, torch.relu(torch.einsum("thd,tjd->thj", qd, kd[safe])))
    return torch.where(idx >= 0, I, torch.full_like(I, float("nan"))).float()


@pytest.mark.parametrize("T,K,use_len,Hi", [(24, 300, False, 64), (400, 300, True, 64), (400, 301, False, 64),
                                              (300, 300, True, 16)])
def test_kl_reading_scores_special_rows_and_many_rows_per_cta(T, K, use_len, Hi):
    # the score-reading kernel walks several rows per CTA (T = 400 over at most one CTA per SM): rows
    # without tiles (empty, zero target) between rows with tiles, holes, one valid slot, prefixes; rows
    # of K = 300 slots start on 16-byte boundaries (vector loads), rows of K = 301 do not
    q_idx, k_idx, w, idx, prob, ln = kl_inputs(T, 900, K, Hi, 76, ln_frac=1.0 if use_len else None)
    idx[2, 10] = -1
    idx[4, :] = -1
    idx[6, 1:] = -1
    prob[8] = 0.0
    idx[T - 1, :] = -1
    if ln is not None:
        ln[11] = 0
        idx = torch.where(torch.arange(idx.shape[1])[None, :] < ln[:, None].long(), idx, torch.full_like(idx, -1))
    sc = _slot_scores_fp32(q_idx, k_idx, w, idx)
    kl, dq, dw, _ = check_kl(q_idx, k_idx, w, idx, prob, ln=ln, topk_score=sc)
    for r in (4, 6, 8, T - 1):
        assert abs(float(kl[r])) < 1e-6
        assert torch.all(dw[r] == 0)


def test_kl_fewer_heads_topk_len_and_coefficient():
    q_idx, k_idx, w, idx, prob, ln = kl_inputs(20, 700, 261, 16, 72, ln_frac=1.0)
    check_kl(q_idx, k_idx, w, idx, prob, coeff=0.001, ln=ln)


def test_kl_target_equal_to_indexer_distribution_gives_zero():
    # p proportional to exp(I) of the indexer's own scores (computed in fp64 here): kl ~ 0, gradients ~ 0
    q_idx, k_idx, w, idx, _, _ = kl_inputs(8, 500, 130, 64, 73)
    qd, kd, wd = q_idx.double(), k_idx.double(), w.double()
    I = torch.einsum("th,thj->tj", wd, torch.relu(torch.einsum("thd,tjd->thj", qd, kd[idx.long()])))
    prob = torch.softmax(I, dim=1).float()
    ws = torch.zeros(4096, dtype=torch.uint8, device=DEV)
    run = lambda p: dsa.dsa_indexer_kl(q_idx.to(DEV), k_idx.to(DEV), w.to(DEV), idx.to(DEV), p.to(DEV), 1.0,
                                       workspace=ws)
    # the scale of each gradient for a generic target, then the matching target
    scale = [float(g.float().abs().max()) for g in run(torch.rand(prob.shape, generator=synth.generator(75)))[1:]]
    kl, dq, dw, dk = run(prob)
    assert dsa.dsa_read_device_status(ws) == 0
    # the exact values are 0; what remains is the fp32 rounding of q - p (about 1e-7 per slot)
    assert float(kl.abs().max()) < 1e-5
    for g, sc, name in zip((dq, dw, dk), scale, ("dq_idx", "dw", "dk_idx")):
        assert float(g.float().abs().max()) <= 1e-3 * sc, name


def test_kl_chained_after_the_sparse_mla_backward():
    # the backward's attn_prob feeds the KL kernel directly (the training order); the oracle chains its
    # own slot probabilities into its own loss
    T, Tk, K = 64, 700, 200
    q, kv, dout, idx = make_case(T, Tk - T, 64, 576, K, 74)
    x = synth.indexer_inputs(Tk, 64, 128, seed=74)
    prob = gpu_prob(q, kv, dout, idx, 192 ** -0.5)
    ref_prob = torch.as_tensor(oracle.attn_slot_prob(q, kv, idx, 192 ** -0.5, Dv=512))
    check_kl(x["q_idx"][Tk - T:].contiguous(), x["k_idx"], x["w"][Tk - T:].contiguous(), idx, prob,
             ref=(idx, ref_prob, None))


@pytest.mark.parametrize("T,K,cut,nrows", [(900, 256, [0, 300, 303, 900], 900), (2300, 2048, [0, 2300], 160)])
def test_kl_reading_the_selection_scores(T, K, cut, nrows):
    # indexer with its scores -> KL reading them (no second gather or S product for the scores).  The
    # scores against the oracle's fp64 scores of its own selection; the loss and gradients against the
    # oracle on the rows whose selection equals the oracle's, with the oracle's own indices
    from test_gpu_indexer import GAMMA, check_rows, oracle_start
    x = synth.indexer_inputs(T, 64, 128, seed=79)
    cu = torch.tensor(cut, dtype=torch.int32)
    start, _, _, _ = dsa.dsa_packed_metadata(cu.to(DEV), T)
    q, k, w = x["q_idx"].to(DEV), x["k_idx"].to(DEV), x["w"].to(DEV)
    idx, ln, sc = dsa.dsa_indexer_topk_scored(q, k, w, start, K)
    idx0, ln0 = dsa.dsa_indexer_topk(q, k, w, start, K)
    assert torch.equal(idx, idx0) and torch.equal(ln, ln0)  # the same kernel selects the same
    # checked rows: all, or a sample with the first and last rows and those around K
    chk = np.arange(T) if nrows >= T else np.union1d([0, 1, K - 1, K, K + 1, T - 1],
                                                     np.random.default_rng(81).choice(T, nrows, replace=False))
    ref = {}
    check_rows(idx.cpu().numpy(), ln.cpu().numpy(), x["q_idx"], x["k_idx"], x["w"], oracle_start(cu, T, start),
               chk, K, ref_out=ref)
    gi, gl, gs = idx.cpu().numpy()[chk], ln.cpu().numpy()[chk], sc.cpu().double().numpy()[chk]
    same = np.all(gi == ref["idx"], axis=1) & (gl == ref["len"])
    assert same.mean() >= 0.95
    for i in np.nonzero(same)[0][:: max(1, int(same.sum()) // 200)]:
        t, n = int(chk[i]), int(ref["len"][i])
        assert np.all(gs[i, n:] == -np.inf), t
        rs, mag = oracle.indexer_scores(x["q_idx"][[t]], x["k_idx"], x["w"][[t]], np.zeros(n, np.int64),
                                        ref["idx"][i, :n], with_magnitude=True)
        assert np.all(np.abs(gs[i, :n] - rs) <= GAMMA * mag), f"row {t}: scores"
    prob = (torch.rand(T, K, generator=synth.generator(80), dtype=torch.float64) ** 4).float()
    rows = chk[same]
    r = torch.as_tensor(rows)
    ref_idx, ref_ln = torch.as_tensor(ref["idx"][same]), torch.as_tensor(ref["len"][same])
    g = lambda t_: t_[r.to(t_.device)].contiguous()
    check_kl(g(x["q_idx"]), x["k_idx"], g(x["w"]), g(idx), g(prob), ln=g(ln), topk_score=g(sc),
             ref=(ref_idx, g(prob), ref_ln))
