"""The bounded device-side waits: a wait that runs past its limit records
DSA_ERR_TIMEOUT in the device error word, every role of the CTA leaves its
loop and reaches the teardown (no barrier is left waiting), and the next call
with the default limit runs normally.

The limit is set to 0 cycles, so each kernel gives up at its first wait whose
phase has not completed (the first gathered tile, the first k_idx tile): the
timeout is certain and no fault or hang is involved.  The outputs of the
timed-out calls are not defined and are not checked; the calls that follow
are checked against the oracle."""
import numpy as np
import pytest
import torch

import oracle
import sparse_attention_mla_gb300 as dsa
from sparse_attention_mla_gb300 import synth

from _cmp import assert_close, assert_lse
from test_gpu_fwd import make_case
from test_gpu_indexer import check_rows, oracle_start

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
DSA_ERR_TIMEOUT = 7


@pytest.fixture
def zero_wait_limit():
    dsa.dsa_set_wait_limit_cycles(0)
    try:
        yield
    finally:
        dsa.dsa_set_wait_limit_cycles(-1)


def run_all(q, kv, dout, idx, scale, ind, start, K):
    wi = torch.zeros(4096, dtype=torch.uint8, device=DEV)
    wf = torch.zeros(4096, dtype=torch.uint8, device=DEV)
    wb = torch.zeros(dsa.workspace_size("bwd", q.shape[0], q.shape[1], idx.shape[1]), dtype=torch.uint8, device=DEV)
    ti, tl = dsa.dsa_indexer_topk(ind["q_idx"].to(DEV), ind["k_idx"].to(DEV), ind["w"].to(DEV), start, K, workspace=wi)
    out, lse, lo = dsa.dsa_sparse_mla_fwd(q.to(DEV), kv.to(DEV), idx.to(DEV), scale, out_lo=True, workspace=wf)
    dq, dkv, _ = dsa.dsa_sparse_mla_bwd(q.to(DEV), kv.to(DEV), idx.to(DEV), scale, out, lse, dout.to(DEV), out_lo=lo,
                                        workspace=wb)
    status = (dsa.dsa_read_device_status(wi), dsa.dsa_read_device_status(wf), dsa.dsa_read_device_status(wb))
    return status, (ti, tl), (out, lse), (dq, dkv)


def test_wait_limit_expiry_is_reported_and_the_next_call_is_clean(zero_wait_limit):
    q, kv, dout, idx = make_case(12, 600, 64, 576, 400, 51)  # 4 tiles of slots per row
    T, K = 700, 64
    ind = synth.indexer_inputs(T, 64, 128, seed=51)
    start, _, _, _ = dsa.dsa_packed_metadata(torch.tensor([0, T], dtype=torch.int32, device=DEV), T)
    status, _, _, _ = run_all(q, kv, dout, idx, 0.1, ind, start, K)
    assert status == (DSA_ERR_TIMEOUT,) * 3, status
    # default limit again: every kernel runs normally and matches the oracle
    dsa.dsa_set_wait_limit_cycles(-1)
    status, (ti, tl), (out, lse), (dq, dkv) = run_all(q, kv, dout, idx, 0.1, ind, start, K)
    assert status == (0, 0, 0), status
    check_rows(ti.cpu().numpy(), tl.cpu().numpy(), ind["q_idx"], ind["k_idx"], ind["w"], oracle_start([0, T], T, start),
               np.array([0, 1, 63, 64, 350, T - 1]), K)
    ref_o, ref_l = oracle.sparse_mla_fwd(q, kv, idx, 0.1)
    ref_dq, ref_dkv = oracle.sparse_mla_bwd(q, kv, idx, dout, 0.1)
    assert_close(out.cpu(), ref_o, "out")
    assert_lse(lse.cpu(), ref_l)
    assert_close(dq.cpu(), ref_dq, "dq")
    assert_close(dkv.cpu(), ref_dkv, "dkv")



def test_wait_limit_expiry_in_the_few_heads_forward_and_the_kl_kernels(zero_wait_limit):
    # The few-heads forward (its gather, S^T and P.V warps) and both KL kernels (forming the slots'
    # scores, and reading them with one CTA per SM walking the rows): each reports DSA_ERR_TIMEOUT with
    # a zero limit, and the same calls with the default limit match the oracle.
    from test_gpu_kl import _slot_scores_fp32, check_kl, kl_inputs
    q, kv, dout, idx = make_case(12, 600, 8, 512, 400, 53)  # 7 tiles of 64 keys: the ring turns over
    q_idx, k_idx, w, kidx, prob, _ = kl_inputs(200, 900, 300, 64, 78)  # 200 rows: several per CTA
    sc = _slot_scores_fp32(q_idx, k_idx, w, kidx)

    def fwd():
        ws = torch.zeros(4096, dtype=torch.uint8, device=DEV)
        out, lse = dsa.dsa_sparse_mla_fwd(q.to(DEV), kv.to(DEV), idx.to(DEV), 0.1, workspace=ws)
        return dsa.dsa_read_device_status(ws), out, lse

    def kl(score):
        ws = torch.zeros(4096, dtype=torch.uint8, device=DEV)
        dsa.dsa_indexer_kl(q_idx.to(DEV), k_idx.to(DEV), w.to(DEV), kidx.to(DEV), prob.to(DEV), 1.0, workspace=ws,
                           topk_score=None if score is None else score.to(DEV))
        return dsa.dsa_read_device_status(ws)

    assert fwd()[0] == DSA_ERR_TIMEOUT
    assert kl(None) == DSA_ERR_TIMEOUT
    assert kl(sc) == DSA_ERR_TIMEOUT
    dsa.dsa_set_wait_limit_cycles(-1)
    status, out, lse = fwd()
    assert status == 0
    ref_o, ref_l = oracle.sparse_mla_fwd(q, kv, idx, 0.1)
    assert_close(out.cpu(), ref_o, "out")
    assert_lse(lse.cpu(), ref_l)
    check_kl(q_idx, k_idx, w, kidx, prob)
    check_kl(q_idx, k_idx, w, kidx, prob, topk_score=sc)
