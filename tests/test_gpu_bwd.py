"""Sparse MLA backward: CUDA path (through the C ABI) vs the fp64 oracle.

The backward gets the forward's residual of O (as the benchmark runs it), so
that D = <dO, O> uses the fp32 O; one case takes D from the rounded output."""
import numpy as np
import pytest
import torch

import oracle
import sparse_attention_mla_gb300 as dsa
from sparse_attention_mla_gb300 import synth

from _cmp import assert_close
from test_gpu_fwd import make_case

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def gpu_fwd_bwd(q, kv, dout, idx, scale, ln=None, dkv=None, accumulate=False, want_bf16=False, use_lo=True):
    dq_, kv_, i_, do_ = q.to(DEV), kv.to(DEV), idx.to(DEV), dout.to(DEV)
    ln_ = None if ln is None else ln.to(DEV)
    ws = torch.zeros(dsa.workspace_size("bwd", q.shape[0], q.shape[1], idx.shape[1]) + 256, dtype=torch.uint8, device=DEV)
    out, lse, lo = dsa.dsa_sparse_mla_fwd(dq_, kv_, i_, scale, topk_len=ln_, out_lo=True)
    lo = lo if use_lo else None
    kb = torch.empty_like(kv_) if want_bf16 else None
    dq, dkv, kb = dsa.dsa_sparse_mla_bwd(dq_, kv_, i_, scale, out, lse, do_, topk_len=ln_, dkv_accum=dkv,
                                         accumulate=accumulate, dkv_bf16=kb, workspace=ws, out_lo=lo)
    assert dsa.dsa_read_device_status(ws) == 0
    return dq, dkv, kb


def check(q, kv, dout, idx, scale, ln=None, use_lo=True):
    dq, dkv, _ = gpu_fwd_bwd(q, kv, dout, idx, scale, ln, use_lo=use_lo)
    ref_dq, ref_dkv = oracle.sparse_mla_bwd(q, kv, idx, dout, scale, len_rows=ln)
    assert_close(dq.cpu(), ref_dq, "dq")
    assert_close(dkv.cpu(), ref_dkv, "dkv")
    return dq, dkv


def test_bwd_tiny_config():
    c = synth.WORKLOADS["tiny"]
    q, kv, dout, idx = make_case(c["T"], 0, c["H"], c["Dqk"], c["K"], 0)
    check(q, kv, dout, idx, c["scale"])


def test_bwd_multi_tile_ragged_64_heads():
    q, kv, dout, idx = make_case(64, 700, 64, 576, 300, 1)
    check(q, kv, dout, idx, 192 ** -0.5)


def test_bwd_prefix_rows_64_heads():
    q, kv, dout, idx = make_case(160, 0, 64, 576, 150, 2)
    check(q, kv, dout, idx, 192 ** -0.5)


def test_bwd_two_head_groups_nope_topk_len_holes():
    q, kv, dout, idx = make_case(32, 400, 128, 512, 261, 3)
    idx[3, 5] = -1
    idx[7, :17] = -1
    g = synth.generator(33)
    ln = torch.randint(0, 262, (32,), generator=g, dtype=torch.int32)
    ln[0] = 0
    check(q, kv, dout, idx, 512 ** -0.5, ln=ln)


def test_bwd_without_residual_many_keys():
    # D from the rounded output only: fine when every row has many keys
    q, kv, dout, idx = make_case(32, 400, 128, 512, 261, 3)
    check(q, kv, dout, idx, 512 ** -0.5, use_lo=False)


def test_bwd_few_heads_padded_and_empty_rows():
    q, kv, dout, idx = make_case(40, 300, 8, 512, 259, 4)
    idx[0, :] = -1
    idx[5, 1:] = -1
    dq, _ = check(q, kv, dout, idx, 512 ** -0.5)
    assert torch.all(dq[0].cpu() == 0)


def test_bwd_query_chunks_accumulate_to_one_shot():
    q, kv, dout, idx = make_case(48, 500, 64, 576, 200, 7)
    dq, dkv, _ = gpu_fwd_bwd(q, kv, dout, idx, 0.07)
    acc = None
    parts = []
    for a, b in [(0, 17), (17, 30), (30, 48)]:
        d, acc, _ = gpu_fwd_bwd(q[a:b], kv, dout[a:b], idx[a:b], 0.07, dkv=acc, accumulate=acc is not None)
        parts.append(d)
    assert torch.equal(torch.cat(parts), dq)
    # key gradients sum; only the fp32 summation order differs
    assert_close(acc.cpu(), dkv.cpu().double(), "chunked dkv", max_abs=1e-4, rel_fro=1e-5)


def test_bwd_dkv_bf16_copy_is_rounded_accumulator():
    q, kv, dout, idx = make_case(24, 200, 16, 576, 64, 9)
    _, dkv, kb = gpu_fwd_bwd(q, kv, dout, idx, 0.1, want_bf16=True)
    assert torch.equal(kb, dkv.to(torch.bfloat16))


def test_bwd_dkv_column_sums_equal_dout_sums():
    # property at any size: sum_k dkv[k, c] = sum_{t,h nonempty} dO[t,h,c] (c < 512), 0 for RoPE channels.
    # It rests on sum_j dS_j = 0, i.e. on D = <dO, O> with the fp32 O (the forward's residual)
    q, kv, dout, idx = make_case(256, 1000, 64, 576, 700, 10)
    _, dkv, _ = gpu_fwd_bwd(q, kv, dout, idx, 192 ** -0.5)
    col = dkv.double().sum(0).cpu().numpy()
    ref = dout.double().sum((0, 1)).numpy()
    assert np.max(np.abs(col[:512] - ref)) < 2e-2
    assert np.max(np.abs(col[512:])) < 2e-2
