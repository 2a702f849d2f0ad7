"""dsa_sparse_mla_bwd_noalloc: the backward for callers that cannot allocate
device memory (runtimes that own all device memory through their own pool,
plug-ins whose host program owns every allocation).  It takes its scratch from
a device array built into the library instead of a caller workspace.

The test calls it through the C ABI and checks it against dsa_sparse_mla_bwd
(caller workspace) on two calls in a row with different inputs, so that a
result left in the shared array by the first call cannot pass for the second.
It is collected last (file name) and needs nothing from the other tests.
"""
import ctypes

import pytest
import torch

import sparse_attention_mla_gb300 as dsa
from sparse_attention_mla_gb300 import synth

from _cmp import assert_close

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


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


def _noalloc_call(lib, q, kv, idx, scale, out, out_lo, lse, dout):
    T, H, Dqk = q.shape
    dq = torch.empty_like(q)
    dkv = torch.empty(kv.shape[0], Dqk, dtype=torch.float32, device=DEV)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = lib.dsa_sparse_mla_bwd_noalloc(_p(q), _p(kv), _p(idx), None, T, kv.shape[0], H, Dqk, 512, idx.shape[1],
                                        ctypes.c_float(scale), _p(out), _p(out_lo), _p(lse), _p(dout), _p(dq), _p(dkv),
                                        0, None, stream)
    assert st == 0, lib.dsa_last_error_message().decode()
    torch.cuda.synchronize()
    return dq, dkv


def test_noalloc_bwd_matches_workspace_bwd_on_two_calls():
    lib = dsa.load_library()
    for seed, scale in [(101, 192 ** -0.5), (202, 0.05)]:
        q, kv, dout, idx = _case(seed)
        out, lse, out_lo = dsa.dsa_sparse_mla_fwd(q, kv, idx, scale, out_lo=True)
        dq_ref, dkv_ref, _ = dsa.dsa_sparse_mla_bwd(q, kv, idx, scale, out, lse, dout, out_lo=out_lo)
        dq, dkv = _noalloc_call(lib, q, kv, idx, scale, out, out_lo, lse, dout)
        assert_close(dq.cpu(), dq_ref.cpu().double(), f"dq (call seed {seed})")
        assert_close(dkv.cpu(), dkv_ref.cpu().double(), f"dkv (call seed {seed})")


def test_noalloc_bwd_rejects_rows_beyond_its_scratch():
    lib = dsa.load_library()
    max_rows = lib.dsa_sparse_mla_bwd_noalloc_max_rows()
    H = 64
    T = max_rows // H + 1  # one row too many; rejected on the host before any launch
    fake = ctypes.c_void_p(0x10000)
    st = lib.dsa_sparse_mla_bwd_noalloc(fake, fake, fake, None, T, T, H, 576, 512, 64, ctypes.c_float(0.1), fake,
                                        None, fake, fake, fake, fake, 0, None, None)
    assert st == 4  # DSA_ERR_WORKSPACE
    assert "scratch limit" in lib.dsa_last_error_message().decode()


def test_noalloc_bwd_rejects_topk_beyond_its_scratch():
    lib = dsa.load_library()
    K = lib.dsa_sparse_mla_bwd_noalloc_max_topk() + 1  # rejected on the host before any launch
    fake = ctypes.c_void_p(0x10000)
    st = lib.dsa_sparse_mla_bwd_noalloc(fake, fake, fake, None, 4, 4, 64, 576, 512, K, ctypes.c_float(0.1), fake,
                                        None, fake, fake, fake, fake, 0, None, None)
    assert st == 4  # DSA_ERR_WORKSPACE
    assert "scratch limit" in lib.dsa_last_error_message().decode()
