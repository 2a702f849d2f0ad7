"""Attention sink in sparse MLA forward and backward: CUDA path (through the C
ABI) vs the fp64 oracle.  The reading (NeMo AutoModel cudnn_dsa,
_pad_attention_heads pads a sink [H] together with q; no formula is printed):
one more logit per row of head h, in the units of the scaled scores, with no
value row; lse includes it, an empty row gets lse = sink and out = 0, and
d_sink[h] = -sum_t exp(sink[h] - lse[t,h]) <dO, O>[t,h]."""
import numpy as np
import pytest
import torch

import oracle
import sparse_attention_mla_gb300 as dsa
from sparse_attention_mla_gb300 import synth

from _cmp import assert_close, assert_lse
from test_gpu_fwd import make_case

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def sink_values(H, seed):
    g = torch.Generator().manual_seed(seed)
    s = torch.randn(H, generator=g, dtype=torch.float32) * 2.0
    s[H // 3] = -float("inf")  # one head without a sink
    return s


def run(q, kv, dout, idx, scale, sink, ln=None, chunks=None):
    qd, kvd, idd, dod, sd = q.to(DEV), kv.to(DEV), idx.to(DEV), dout.to(DEV), sink.to(DEV)
    lnd = None if ln is None else ln.to(DEV)
    wf = torch.zeros(dsa.workspace_size("fwd", q.shape[0], q.shape[1]), dtype=torch.uint8, device=DEV)
    wb = torch.zeros(dsa.workspace_size("bwd", q.shape[0], q.shape[1], idx.shape[1]), dtype=torch.uint8, device=DEV)
    out, lse, lo = dsa.dsa_sparse_mla_fwd(qd, kvd, idd, scale, topk_len=lnd, out_lo=True, workspace=wf, attn_sink=sd)
    assert dsa.dsa_read_device_status(wf) == 0
    T = q.shape[0]
    chunks = chunks or [(0, T)]
    dq = torch.empty_like(qd)
    dkv, dsink = None, None
    for a, b in chunks:
        dq_c, dkv, _, dsink = dsa.dsa_sparse_mla_bwd(
            qd[a:b], kvd, idd[a:b], scale, out[a:b], lse[a:b], dod[a:b], topk_len=None if lnd is None else lnd[a:b],
            out_lo=lo[a:b], workspace=wb, attn_sink=sd, dkv_accum=dkv, d_sink=dsink, accumulate=dkv is not None)
        dq[a:b] = dq_c
        assert dsa.dsa_read_device_status(wb) == 0
    return out, lse, dq, dkv, dsink


def check(q, kv, dout, idx, scale, sink, ln=None, chunks=None):
    out, lse, dq, dkv, dsink = run(q, kv, dout, idx, scale, sink, ln, chunks)
    ref_o, ref_l = oracle.sparse_mla_fwd(q, kv, idx, scale, len_rows=ln, sink=sink)
    ref_dq, ref_dkv, ref_ds = oracle.sparse_mla_bwd(q, kv, idx, dout, scale, len_rows=ln, sink=sink)
    assert_close(out.cpu(), ref_o, "out")
    assert_lse(lse.cpu(), ref_l)
    assert_close(dq.cpu(), ref_dq, "dq")
    assert_close(dkv.cpu(), ref_dkv, "dkv")
    assert_close(dsink.cpu(), ref_ds, "d_sink")
    return out, lse


def test_sink_multi_tile_64_heads_with_empty_rows():
    q, kv, dout, idx = make_case(40, 600, 64, 576, 300, 41)
    idx[5, :] = -1                      # empty row: lse = sink, out = 0
    idx[9, 1:] = -1                     # one valid slot
    out, lse = check(q, kv, dout, idx, 192 ** -0.5, sink_values(64, 41))
    s = sink_values(64, 41)
    fin = torch.isfinite(s)
    assert torch.all(out[5] == 0)
    assert torch.allclose(lse[5].cpu()[fin], s[fin], atol=1e-6, rtol=0)


def test_sink_two_head_groups_nope_topk_len():
    q, kv, dout, idx = make_case(24, 400, 128, 512, 261, 42)
    ln = torch.randint(0, 262, (24,), generator=torch.Generator().manual_seed(42), dtype=torch.int32)
    check(q, kv, dout, idx, 512 ** -0.5, sink_values(128, 42), ln=ln)


def test_sink_few_heads_nope_empty_rows_and_topk_len():
    # the few-heads forward at 8 heads per CTA (NoPE width): the sink starts the running max, an empty
    # row has lse = sink and out = 0, prefixes of random length
    q, kv, dout, idx = make_case(30, 500, 8, 512, 259, 45)
    idx[3, :] = -1
    ln = torch.randint(0, 260, (30,), generator=torch.Generator().manual_seed(45), dtype=torch.int32)
    s = sink_values(8, 45)
    out, lse = check(q, kv, dout, idx, 512 ** -0.5, s, ln=ln)
    fin = torch.isfinite(s)
    assert torch.all(out[3] == 0)
    assert torch.allclose(lse[3].cpu()[fin], s[fin], atol=1e-6, rtol=0)


def test_sink_dominant_and_query_chunks_accumulate():
    # sinks far above the scores take most of the mass; d_sink and dkv accumulate over query chunks
    q, kv, dout, idx = make_case(48, 500, 16, 576, 200, 43)
    sink = sink_values(16, 43) + 6.0
    check(q, kv, dout, idx, 192 ** -0.5, sink, chunks=[(0, 17), (17, 30), (30, 48)])


def test_sink_of_minus_infinity_equals_no_sink():
    q, kv, dout, idx = make_case(16, 300, 64, 576, 150, 44)
    qd, kvd, idd = q.to(DEV), kv.to(DEV), idx.to(DEV)
    o0, l0 = dsa.dsa_sparse_mla_fwd(qd, kvd, idd, 0.1)
    o1, l1 = dsa.dsa_sparse_mla_fwd(qd, kvd, idd, 0.1, attn_sink=torch.full((64,), -float("inf"), device=DEV))
    assert torch.equal(o0, o1) and torch.equal(l0, l1)
