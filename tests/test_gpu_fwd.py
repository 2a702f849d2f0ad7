"""Sparse MLA forward: CUDA path (through the C ABI) vs the fp64 oracle.

Every case runs with and without the request for O's residual (out_lo);
the residual request must not change out or lse."""
import numpy as np
import pytest
import torch

import oracle
import sparse_attention_mla_gb300 as dsa
from sparse_attention_mla_gb300 import synth

from _cmp import assert_close, assert_lse

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def make_case(nrows, pos0, H, Dqk, K, seed, Tk=None):
    """Rows are query positions pos0 .. pos0+nrows-1 of one sequence starting at 0."""
    Tk = Tk or (pos0 + nrows)
    g = synth.generator(seed)
    q = synth.randn_bf16((nrows, H, Dqk), g)
    kv = synth.randn_bf16((Tk, Dqk), g)
    dout = synth.randn_bf16((nrows, H, 512), g)
    start = torch.zeros(pos0 + nrows, dtype=torch.int32)
    idx = synth.random_causal_topk(start, K, g, rows=torch.arange(pos0, pos0 + nrows))
    return q, kv, dout, idx


def run_fwd(q, kv, idx, scale, ln=None, with_lo=False):
    ws = torch.zeros(1 << 12, dtype=torch.uint8, device=DEV)
    res = dsa.dsa_sparse_mla_fwd(q.to(DEV), kv.to(DEV), idx.to(DEV), scale,
                                 topk_len=None if ln is None else ln.to(DEV), workspace=ws,
                                 out_lo=True if with_lo else None)
    status = dsa.dsa_read_device_status(ws)
    return res[0].cpu(), res[1].cpu(), status


def check(q, kv, idx, scale, ln=None, expect_status=0):
    ref_o, ref_l = oracle.sparse_mla_fwd(q, kv, idx, scale, len_rows=ln)
    res = []
    for with_lo in (False, True):
        out, lse, status = run_fwd(q, kv, idx, scale, ln, with_lo)
        assert status == expect_status
        assert_close(out, ref_o, f"out (with_lo={with_lo})")
        assert_lse(lse, ref_l)
        res.append((out, lse))
    assert torch.equal(res[0][0], res[1][0]) and torch.equal(res[0][1], res[1][1])
    return out, lse


def test_fwd_tiny_config():
    # 1 sequence, T=256, H=16, width 576, K=64, random causal indices, seed 0
    c = synth.WORKLOADS["tiny"]
    q, kv, _, idx = make_case(c["T"], 0, c["H"], c["Dqk"], c["K"], 0)
    check(q, kv, idx, c["scale"])


def test_fwd_multi_tile_ragged_64_heads():
    # 3 tiles of 128 slots (128, 128, 44), K not a multiple of 4 or 64
    q, kv, _, idx = make_case(96, 700, 64, 576, 300, 1)
    check(q, kv, idx, 192 ** -0.5)


def test_fwd_causal_prefix_rows_with_minus_one_suffix():
    # early rows have fewer valid slots than K (c_t < K): -1 suffix of every length
    q, kv, _, idx = make_case(160, 0, 64, 576, 150, 2)
    check(q, kv, idx, 192 ** -0.5)


def test_fwd_two_head_groups_nope_topk_len_holes():
    q, kv, _, idx = make_case(40, 400, 128, 512, 261, 3)
    idx[3, 5] = -1
    idx[7, :17] = -1  # holes at the front
    g = synth.generator(33)
    ln = torch.randint(0, 262, (40,), generator=g, dtype=torch.int32)
    ln[0] = 0
    check(q, kv, idx, 512 ** -0.5, ln=ln)


@pytest.mark.parametrize("H,D", [(8, 512), (3, 576), (12, 512)])  # 8 and 16 heads per CTA, padded in smem
def test_fwd_few_heads_padded_in_smem(H, D):
    q, kv, _, idx = make_case(50, 300, H, D, 259, 4)
    check(q, kv, idx, D ** -0.5)


def test_fwd_empty_rows_and_single_slot():
    q, kv, _, idx = make_case(12, 100, 16, 576, 40, 5)
    idx[0, :] = -1
    idx[1, :] = -1
    idx[1, 39] = 17      # single valid slot at the end of the row
    idx[2, 1:] = -1      # single valid slot at the front
    out, lse = check(q, kv, idx, 0.1)
    assert torch.all(out[0] == 0) and torch.all(torch.isneginf(lse[0]))


def test_fwd_out_of_range_index_is_masked_and_reported():
    q, kv, _, idx = make_case(8, 200, 16, 576, 64, 6)
    idx[2, 3] = 10_000   # >= T_k
    idx[5, 0] = -7       # < -1
    check(q, kv, idx, 0.1, expect_status=6)  # DSA_ERR_DEVICE_INDEX; the oracle masks them too


def test_fwd_query_chunks_equal_one_shot():
    q, kv, _, idx = make_case(64, 500, 64, 576, 200, 7)
    full, lfull, _ = run_fwd(q, kv, idx, 0.07)
    parts = [run_fwd(q[a:b], kv, idx[a:b], 0.07) for a, b in [(0, 21), (21, 40), (40, 64)]]
    assert torch.equal(torch.cat([p[0] for p in parts]), full)
    assert torch.equal(torch.cat([p[1] for p in parts]), lfull)


def test_fwd_nope_zero_pad_matches_576():
    q, kv, _, idx = make_case(32, 300, 64, 512, 130, 8)
    pad = lambda x: torch.cat([x, torch.zeros(*x.shape[:-1], 64, dtype=x.dtype)], dim=-1)
    o512, l512, _ = run_fwd(q, kv, idx, 0.05)
    o576, l576, _ = run_fwd(pad(q), pad(kv), idx, 0.05)
    assert_close(o576, o512.double(), "pad vs nope", max_abs=1e-6, rel_fro=1e-6)
    assert torch.allclose(l512, l576, atol=1e-5, rtol=0)
