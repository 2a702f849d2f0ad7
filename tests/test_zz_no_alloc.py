"""dsa_sparse_mla_bwd_noalloc: the backward for callers that cannot allocate
device memory (runtimes that own all device memory through their own pool,
plug-ins whose host program owns every allocation).  It takes its scratch from
a device array built into the library instead of a caller workspace.

The GPU tests call it through the C ABI and check it against
dsa_sparse_mla_bwd (caller workspace) on calls in a row with different inputs,
so that a result left in the shared array by one call cannot pass for the
next; after every call the array's device error word is read back and must be
clear, except in the case that plants an out-of-range index.  The sizes cover
the array's largest top-k (its dS scratch is full) and the NoPE width with a
topk_len prefix.  The file is collected last and needs nothing from the other
tests; the rejection test runs on the host only.
"""
import ctypes

import pytest
import torch

import sparse_attention_mla_gb300 as dsa
from sparse_attention_mla_gb300 import synth

from _cmp import assert_close

DEV = "cuda:0"
DSA_ERR_WORKSPACE = 4
DSA_ERR_DEVICE_INDEX = 6


def _case(seed, T=48, pos0=500, H=64, Dqk=576, K=200):
    g = synth.generator(seed)
    q = synth.randn_bf16((T, H, Dqk), g).to(DEV)
    kv = synth.randn_bf16((pos0 + T, Dqk), g).to(DEV)
    dout = synth.randn_bf16((T, H, 512), g).to(DEV)
    idx = synth.random_causal_topk(torch.zeros(pos0 + T, dtype=torch.int32), K, g,
                                   rows=torch.arange(pos0, pos0 + T)).to(DEV)
    return q, kv, dout, idx


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _noalloc_call(lib, q, kv, idx, scale, out, out_lo, lse, dout, ln=None):
    T, H, Dqk = q.shape
    dq = torch.empty_like(q)
    dkv = torch.empty(kv.shape[0], Dqk, dtype=torch.float32, device=DEV)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = lib.dsa_sparse_mla_bwd_noalloc(_p(q), _p(kv), _p(idx), _p(ln), T, kv.shape[0], H, Dqk, 512, idx.shape[1],
                                        ctypes.c_float(scale), None, _p(out), _p(out_lo), _p(lse), _p(dout), _p(dq),
                                        _p(dkv), None, None, 0, None, stream)
    assert st == 0, lib.dsa_last_error_message().decode()
    dev_status = ctypes.c_int32(-1)
    assert lib.dsa_sparse_mla_bwd_noalloc_read_status(stream, ctypes.byref(dev_status)) == 0
    return dq, dkv, dev_status.value


def _check_against_workspace_bwd(lib, seed, scale, ln_frac=None, **shape):
    q, kv, dout, idx = _case(seed, **shape)
    ln = None
    if ln_frac is not None:  # a valid prefix shorter than the index row
        ln = ((idx >= 0).sum(1).float() * ln_frac).to(torch.int32)
    out, lse, out_lo = dsa.dsa_sparse_mla_fwd(q, kv, idx, scale, topk_len=ln, out_lo=True)
    dq_ref, dkv_ref, _ = dsa.dsa_sparse_mla_bwd(q, kv, idx, scale, out, lse, dout, topk_len=ln, out_lo=out_lo)
    dq, dkv, status = _noalloc_call(lib, q, kv, idx, scale, out, out_lo, lse, dout, ln)
    assert status == 0, f"device status {status} (call seed {seed})"
    assert_close(dq.cpu(), dq_ref.cpu().double(), f"dq (call seed {seed})")
    assert_close(dkv.cpu(), dkv_ref.cpu().double(), f"dkv (call seed {seed})")


@pytest.mark.gpu
def test_noalloc_bwd_matches_workspace_bwd_on_two_calls():
    lib = dsa.load_library()
    for seed, scale in [(101, 192 ** -0.5), (202, 0.05)]:
        _check_against_workspace_bwd(lib, seed, scale)


@pytest.mark.gpu
def test_noalloc_bwd_at_its_largest_topk_and_nope_width():
    # K = the array's limit (17 dS tiles per slot: the scratch layout at its edge), then the NoPE
    # width 512 with a topk_len prefix, one call after the other
    lib = dsa.load_library()
    kmax = lib.dsa_sparse_mla_bwd_noalloc_max_topk()
    _check_against_workspace_bwd(lib, 303, 192 ** -0.5, T=6, pos0=kmax + 40, K=kmax)
    _check_against_workspace_bwd(lib, 404, 512 ** -0.5, ln_frac=0.75, T=20, pos0=700, Dqk=512, K=333)


@pytest.mark.gpu
def test_noalloc_bwd_reports_a_bad_index_through_its_status():
    # an index below -1 is masked (no read) and flagged in the array's error word; the next call
    # on good input clears the word and reports nothing
    lib = dsa.load_library()
    q, kv, dout, idx = _case(505, T=8)
    out, lse = dsa.dsa_sparse_mla_fwd(q, kv, idx, 0.1)
    bad = idx.clone()
    bad[3, 0] = -2
    _, _, status = _noalloc_call(lib, q, kv, bad, 0.1, out, None, lse, dout)
    assert status == DSA_ERR_DEVICE_INDEX
    _, _, status = _noalloc_call(lib, q, kv, idx, 0.1, out, None, lse, dout)
    assert status == 0


def test_noalloc_bwd_rejects_topk_beyond_its_scratch():
    # host-side check: K one past the array's limit is rejected before any device call
    lib = dsa.load_library()
    K = lib.dsa_sparse_mla_bwd_noalloc_max_topk() + 1
    fake = ctypes.c_void_p(0x10000)
    st = lib.dsa_sparse_mla_bwd_noalloc(fake, fake, fake, None, 4, 4, 64, 576, 512, K, ctypes.c_float(0.1), None,
                                        fake, None, fake, fake, fake, fake, None, None, 0, None, None)
    assert st == DSA_ERR_WORKSPACE
    assert "scratch limit" in lib.dsa_last_error_message().decode()


@pytest.mark.gpu
def test_noalloc_bwd_splits_rows_beyond_its_d_array_into_chunks():
    # T * H above the array's 4 Mi (row, head) pairs: rows run in two chunks whose key gradients sum;
    # dq must equal the workspace backward's bit for bit, dkv within fp32 reduction-order rounding
    lib = dsa.load_library()
    T, H, K = 33000, 128, 64
    g = synth.generator(606)
    q = synth.randn_bf16((T, H, 576), g).to(DEV)
    kv = synth.randn_bf16((T, 576), g).to(DEV)
    dout = synth.randn_bf16((T, H, 512), g).to(DEV)
    idx = torch.randint(0, T, (T, K), dtype=torch.int32, device=DEV)
    out, lse, out_lo = dsa.dsa_sparse_mla_fwd(q, kv, idx, 0.05, out_lo=True)
    dq_ref, dkv_ref, _ = dsa.dsa_sparse_mla_bwd(q, kv, idx, 0.05, out, lse, dout, out_lo=out_lo)
    dq, dkv, status = _noalloc_call(lib, q, kv, idx, 0.05, out, out_lo, lse, dout)
    assert status == 0
    assert torch.equal(dq, dq_ref)
    assert_close(dkv.cpu(), dkv_ref.cpu().double(), "dkv (two row chunks)", max_abs=1e-3, rel_fro=1e-5)
