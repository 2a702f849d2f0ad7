"""Edge cases of the CUDA path against the fp64 oracle: top-k of one, scores
that grow across tiles (the forward's lazy rescale of the running max), kv
longer than the queries with non-causal index sets, empty calls, and the
indexer at the smallest and largest K.

Every case passes the forward's residual of O to the backward, so D is
accurate to about fp32.  On stress inputs (far outside unit scale) out, lse
and dkv meet the pages' bounds element by element.  dq is formed from dS rounded to bf16 (unit
roundoff 2^-8) before the dq product, so where large terms cancel its error
is bounded by 2^-8 scale sum_j |dS_j| |kv[idx_j, c]| (the oracle's dq
magnitude), not by |dq|: dq is checked against that bound plus the pages'
2e-2, and in relative Frobenius norm."""
import numpy as np
import pytest
import torch

import oracle
import sparse_attention_mla_gb300 as dsa
from sparse_attention_mla_gb300 import synth

from _cmp import MAX_ABS, REL_FRO, assert_close, assert_lse, errors, storage_half_ulp, to64
from test_gpu_fwd import make_case
from test_gpu_indexer import check_rows, oracle_start

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def fwd_bwd_vs_oracle(q, kv, dout, idx, scale, ln=None, stress=False):
    qd, kvd, idd, dod = q.to(DEV), kv.to(DEV), idx.to(DEV), dout.to(DEV)
    lnd = None if ln is None else ln.to(DEV)
    wf = torch.zeros(dsa.workspace_size("fwd", q.shape[0], q.shape[1]), dtype=torch.uint8, device=DEV)
    wb = torch.zeros(dsa.workspace_size("bwd", q.shape[0], q.shape[1], idx.shape[1]), dtype=torch.uint8, device=DEV)
    out, lse, lo = dsa.dsa_sparse_mla_fwd(qd, kvd, idd, scale, topk_len=lnd, out_lo=True, workspace=wf)
    dq, dkv, _ = dsa.dsa_sparse_mla_bwd(qd, kvd, idd, scale, out, lse, dod, topk_len=lnd, out_lo=lo, workspace=wb)
    assert dsa.dsa_read_device_status(wf) == 0 and dsa.dsa_read_device_status(wb) == 0
    ref_o, ref_l = oracle.sparse_mla_fwd(q, kv, idx, scale, len_rows=ln)
    ref_dq, ref_dkv, dq_mag = oracle.sparse_mla_bwd(q, kv, idx, dout, scale, len_rows=ln, with_dq_magnitude=True)
    assert_close(out.cpu(), ref_o, "out")
    assert_lse(lse.cpu(), ref_l)
    assert_close(dkv.cpu(), ref_dkv, "dkv")
    if not stress:
        assert_close(dq.cpu(), ref_dq, "dq")
    else:
        g = dq.cpu()
        excess = np.abs(to64(g) - ref_dq) - storage_half_ulp(g) - 2.0 ** -8 * dq_mag
        assert float(np.max(excess)) <= MAX_ABS, f"dq: {float(np.max(excess)):.3e} beyond the bf16-dS bound"
        _, rf = errors(g, ref_dq)
        assert rf <= REL_FRO, f"dq: rel_fro={rf:.3e}"


@pytest.mark.parametrize("H", [64, 16])  # the 64-head forward and the few-heads one (H <= 16)
def test_topk_one(H):
    # K = 1: each row attends to exactly one key (P = 1, dS = 0, dkv = dO on that row)
    q, kv, dout, idx = make_case(40, 100, H, 576, 1, 11)
    fwd_bwd_vs_oracle(q, kv, dout, idx, 192 ** -0.5)


@pytest.mark.parametrize("H,D", [(64, 576), (8, 576), (8, 512)])  # 64-head forward; few heads, ring of 2 / 3 tiles
def test_growing_scores_rescale_running_max(H, D):
    # kv rows scaled up with the key index, slots ascending: every new tile raises the running max by
    # far more than the lazy-rescale threshold, so O is rescaled tile after tile
    q, kv, dout, idx = make_case(24, 700, H, D, 600, 12)
    ramp = (1.0 + torch.arange(kv.shape[0], dtype=torch.float32) / 120.0)[:, None]
    kv = (kv.float() * ramp).to(torch.bfloat16)
    fwd_bwd_vs_oracle(q, kv, dout, idx, 0.25, stress=True)


def test_peaky_softmax_large_scale():
    # one dominant key per row: exp2 arguments span a wide range, most P round to tiny values
    q, kv, dout, idx = make_case(32, 400, 16, 576, 260, 13)
    fwd_bwd_vs_oracle(q, kv, dout, idx, 1.0, stress=True)


def test_kv_longer_than_queries_non_causal_indices():
    # the MLA kernels take any index set: rows pick keys anywhere in a kv 3x longer than the queries
    T, Tk, H, K = 48, 3000, 64, 333
    g = synth.generator(14)
    q = synth.randn_bf16((T, H, 576), g)
    kv = synth.randn_bf16((Tk, 576), g)
    dout = synth.randn_bf16((T, H, 512), g)
    idx = torch.stack([torch.randperm(Tk, generator=g)[:K].sort().values for _ in range(T)]).to(torch.int32)
    fwd_bwd_vs_oracle(q, kv, dout, idx, 192 ** -0.5)


def test_empty_calls_leave_outputs_consistent():
    # T = 0: nothing is launched; the backward still zeroes dkv (accumulate = 0)
    kv = synth.randn_bf16((16, 576), synth.generator(15)).to(DEV)
    q = torch.empty(0, 64, 576, dtype=torch.bfloat16, device=DEV)
    idx = torch.empty(0, 32, dtype=torch.int32, device=DEV)
    out, lse = dsa.dsa_sparse_mla_fwd(q, kv, idx, 0.1)
    assert out.shape == (0, 64, 512) and lse.shape == (0, 64)
    dout = torch.empty(0, 64, 512, dtype=torch.bfloat16, device=DEV)
    dkv = torch.full((16, 576), 7.0, dtype=torch.float32, device=DEV)
    dq, dkv, _ = dsa.dsa_sparse_mla_bwd(q, kv, idx, 0.1, out, lse, dout, dkv_accum=dkv)
    torch.cuda.synchronize()
    assert dq.shape == (0, 64, 576) and torch.all(dkv == 0)
    qi = torch.empty(0, 64, 128, dtype=torch.bfloat16, device=DEV)
    ki = synth.randn_bf16((16, 128), synth.generator(16)).to(DEV)
    w = torch.empty(0, 64, dtype=torch.float32, device=DEV)
    st = torch.empty(0, dtype=torch.int32, device=DEV)
    ti, tl = dsa.dsa_indexer_topk(qi, ki, w, st, 8)
    assert ti.shape == (0, 8) and tl.shape == (0,)


def test_indexer_k_one_and_k_2048_boundaries():
    # K = 1 picks the single best key; K = 2048 (the largest) on windows just above and below it;
    # sets equal the oracle's except inside the fp32 tie band (check_rows)
    T = 2300
    x = synth.indexer_inputs(T, 64, 128, seed=17)
    cu = torch.tensor([0, T], dtype=torch.int32)
    start, _, _, _ = dsa.dsa_packed_metadata(cu.to(DEV), T)
    rows = np.array([0, 1, 2, 1000, 2046, 2047, 2048, 2049, 2050, T - 2, T - 1])
    for K in (1, 2048):
        ws = torch.zeros(4096, dtype=torch.uint8, device=DEV)
        idx, ln = dsa.dsa_indexer_topk(x["q_idx"].to(DEV), x["k_idx"].to(DEV), x["w"].to(DEV), start, K, workspace=ws)
        assert dsa.dsa_read_device_status(ws) == 0
        check_rows(idx.cpu().numpy(), ln.cpu().numpy(), x["q_idx"], x["k_idx"], x["w"], oracle_start(cu, T, start),
                   rows, K)
