"""CPU checks of the C ABI: the library loads, exports every declared symbol,
and rejects bad arguments on the host before touching a device."""
import ctypes

import pytest

import sparse_attention_mla_gb300 as dsa
from sparse_attention_mla_gb300 import build_ext


@pytest.fixture(scope="module")
def lib():
    build_ext.build()
    return dsa.load_library()


def test_every_declared_symbol_is_exported(lib):
    names = dsa.declared_symbols()
    expected = {"dsa_packed_metadata", "dsa_packed_metadata_cp", "dsa_indexer_topk", "dsa_indexer_topk_cp",
                "dsa_sparse_mla_fwd", "dsa_sparse_mla_bwd", "dsa_sparse_mla_bwd_noalloc",
                "dsa_sparse_mla_bwd_noalloc_read_status", "dsa_sparse_mla_bwd_noalloc_max_topk",
                "dsa_status_string", "dsa_last_error_message", "dsa_read_device_status"}
    assert expected <= set(names)
    for n in names:
        assert hasattr(lib, n), n


def test_abi_version_and_status_strings(lib):
    assert lib.dsa_abi_version() == 3
    for code in range(8):
        s = lib.dsa_status_string(code).decode()
        assert s.startswith(dsa.STATUS_NAMES[code])


P = ctypes.c_void_p
FAKE = P(0x10000)  # never dereferenced: validation fails before any device use


def fwd(lib, **kw):
    a = dict(q=FAKE, kv=FAKE, idx=FAKE, ln=None, T=4, Tk=8, H=16, Dqk=576, Dv=512, K=64, scale=0.1, sink=None,
             out=FAKE, lse=FAKE, ws=P(0x100000), wsb=1 << 20, stream=None)
    a.update(kw)
    return lib.dsa_sparse_mla_fwd(a["q"], a["kv"], a["idx"], a["ln"], a["T"], a["Tk"], a["H"], a["Dqk"], a["Dv"],
                                  a["K"], ctypes.c_float(a["scale"]), a["sink"], a["out"], None, a["lse"], a["ws"],
                                  a["wsb"], a["stream"])


@pytest.mark.parametrize("bad", [dict(Dqk=500), dict(Dv=256), dict(K=0), dict(H=0), dict(Tk=0), dict(T=-1),
                                 dict(scale=0.0), dict(scale=float("nan")), dict(scale=-1.0), dict(q=None),
                                 dict(q=P(0x10002))])
def test_fwd_rejects_invalid_arguments(lib, bad):
    assert fwd(lib, **bad) == 3  # DSA_ERR_INVALID_ARGUMENT
    assert lib.dsa_last_error_message().decode().startswith("dsa_sparse_mla_fwd")


@pytest.mark.parametrize("bad", [dict(ws=None), dict(ws=P(0x100010)), dict(wsb=16)])
def test_fwd_rejects_bad_workspace(lib, bad):
    assert fwd(lib, **bad) == 4  # DSA_ERR_WORKSPACE


def test_metadata_rejects_invalid_arguments(lib):
    assert lib.dsa_packed_metadata(None, 1, 4, FAKE, FAKE, None, None, None) == 3
    assert lib.dsa_packed_metadata(FAKE, 0, 4, FAKE, FAKE, None, None, None) == 3


def meta_cp(lib, **kw):
    a = dict(cu=FAKE, cup=None, n=2, Tk=16, qi=FAKE, pm=None, Tq=4, st=FAKE, cl=FAKE)
    a.update(kw)
    return lib.dsa_packed_metadata_cp(a["cu"], a["cup"], a["n"], a["Tk"], a["qi"], a["pm"], a["Tq"], a["st"], a["cl"],
                                      None, None, None)


@pytest.mark.parametrize("bad", [dict(cu=None), dict(n=0), dict(Tq=-1), dict(Tk=-1), dict(st=None), dict(cl=None),
                                 dict(qi=None, Tq=17)])
def test_metadata_cp_rejects_invalid_arguments(lib, bad):
    assert meta_cp(lib, **bad) == 3  # DSA_ERR_INVALID_ARGUMENT, before any device access
    assert lib.dsa_last_error_message().decode().startswith("dsa_packed_metadata_cp")


def bwd(lib, **kw):
    a = dict(q=FAKE, kv=FAKE, idx=FAKE, ln=None, T=4, Tk=8, H=16, Dqk=576, Dv=512, K=64, scale=0.1, sink=None,
             out=FAKE, out_lo=None, lse=FAKE, dout=FAKE, dq=FAKE, dkv=FAKE, dsink=None, prob=None, acc=0,
             dkv_bf16=None, ws=P(0x100000), wsb=1 << 30, stream=None)
    a.update(kw)
    return lib.dsa_sparse_mla_bwd(a["q"], a["kv"], a["idx"], a["ln"], a["T"], a["Tk"], a["H"], a["Dqk"], a["Dv"],
                                  a["K"], ctypes.c_float(a["scale"]), a["sink"], a["out"], a["out_lo"], a["lse"],
                                  a["dout"], a["dq"], a["dkv"], a["dsink"], a["prob"], a["acc"], a["dkv_bf16"], a["ws"],
                                  a["wsb"], a["stream"])


@pytest.mark.parametrize("bad", [dict(Dqk=500), dict(Dv=256), dict(K=0), dict(H=0), dict(Tk=0), dict(T=-1),
                                 dict(acc=2), dict(scale=0.0), dict(scale=float("inf")), dict(kv=None),
                                 dict(dkv=None), dict(dq=None), dict(q=P(0x10002)), dict(out_lo=P(0x10008)),
                                 dict(dkv_bf16=P(0x10002)), dict(dsink=FAKE)])
def test_bwd_rejects_invalid_arguments(lib, bad):
    assert bwd(lib, **bad) == 3  # DSA_ERR_INVALID_ARGUMENT
    assert lib.dsa_last_error_message().decode().startswith("dsa_sparse_mla_bwd")


def test_bwd_workspace_grows_with_rows_heads_and_topk(lib):
    lib.dsa_sparse_mla_bwd_workspace_size.restype = ctypes.c_size_t
    base = lib.dsa_sparse_mla_bwd_workspace_size(4, 16, 64)
    assert lib.dsa_sparse_mla_bwd_workspace_size(4096, 16, 64) > base          # D per (row, head)
    assert lib.dsa_sparse_mla_bwd_workspace_size(4, 16, 2051) > base           # dS scratch per 128-slot tile
    assert bwd(lib, wsb=base - 256) == 4                                         # DSA_ERR_WORKSPACE
    assert bwd(lib, ws=P(0x100010)) == 4                                         # not 256-byte aligned


def idxr(lib, **kw):
    a = dict(q=FAKE, k=FAKE, w=FAKE, st=FAKE, T=4, Tk=8, Hi=64, Di=128, K=64, idx=FAKE, ln=None, ws=P(0x100000),
             wsb=1 << 20, stream=None)
    a.update(kw)
    return lib.dsa_indexer_topk(a["q"], a["k"], a["w"], a["st"], a["T"], a["Tk"], a["Hi"], a["Di"], a["K"], a["idx"],
                                a["ln"], a["ws"], a["wsb"], a["stream"])


@pytest.mark.parametrize("bad", [dict(Tk=3), dict(T=-1), dict(Hi=0), dict(Hi=65), dict(Di=64), dict(K=0),
                                 dict(K=2049), dict(k=None), dict(w=None), dict(st=None), dict(idx=None),
                                 dict(q=P(0x10002))])
def test_indexer_rejects_invalid_arguments(lib, bad):
    assert idxr(lib, **bad) == 3  # DSA_ERR_INVALID_ARGUMENT
    assert lib.dsa_last_error_message().decode().startswith("dsa_indexer_topk")


def idxr_cp(lib, **kw):
    a = dict(q=FAKE, k=FAKE, w=FAKE, st=FAKE, cl=FAKE, T=4, Tk=8, Hi=64, Di=128, K=64, idx=FAKE, ln=None,
             ws=P(0x100000), wsb=1 << 20, stream=None)
    a.update(kw)
    return lib.dsa_indexer_topk_cp(a["q"], a["k"], a["w"], a["st"], a["cl"], a["T"], a["Tk"], a["Hi"], a["Di"],
                                   a["K"], a["idx"], a["ln"], a["ws"], a["wsb"], a["stream"])


@pytest.mark.parametrize("bad", [dict(cl=None), dict(T=-1), dict(Hi=65), dict(Di=64), dict(K=2049), dict(k=None),
                                 dict(st=None), dict(q=P(0x10002))])
def test_indexer_cp_rejects_invalid_arguments(lib, bad):
    assert idxr_cp(lib, **bad) == 3
    assert lib.dsa_last_error_message().decode().startswith("dsa_indexer_topk_cp")


def test_indexer_scored_rejects_invalid_arguments(lib):
    def call(**kw):
        a = dict(q=FAKE, k=FAKE, w=FAKE, st=FAKE, cl=None, T=4, Tk=8, Hi=64, Di=128, K=64, idx=FAKE, ln=None,
                 sc=FAKE, ws=P(0x100000), wsb=1 << 20, stream=None)
        a.update(kw)
        return lib.dsa_indexer_topk_scored(a["q"], a["k"], a["w"], a["st"], a["cl"], a["T"], a["Tk"], a["Hi"],
                                           a["Di"], a["K"], a["idx"], a["ln"], a["sc"], a["ws"], a["wsb"],
                                           a["stream"])
    for bad in (dict(sc=None), dict(Tk=3), dict(K=2049), dict(Hi=65), dict(q=P(0x10002))):
        assert call(**bad) == 3, bad
        assert lib.dsa_last_error_message().decode().startswith("dsa_indexer_topk_scored")
    assert call(ws=None) == 4


def test_indexer_rejects_bad_workspace(lib):
    assert idxr(lib, ws=None) == 4
    assert idxr(lib, wsb=16) == 4


def test_wait_limit_setter_returns_the_previous_value(lib):
    lib.dsa_set_wait_limit_cycles.argtypes = [ctypes.c_int64]
    lib.dsa_set_wait_limit_cycles.restype = ctypes.c_int64
    prev = lib.dsa_set_wait_limit_cycles(12345)
    try:
        assert lib.dsa_set_wait_limit_cycles(-1) == 12345
        assert lib.dsa_set_wait_limit_cycles(-1) == 1 << 31  # negative: the default
    finally:
        lib.dsa_set_wait_limit_cycles(prev)


def test_kpool_entries_reject_invalid_arguments(lib):
    I = ctypes.c_int32
    m = lib.dsa_kpool_metadata
    assert m(FAKE, 2, 16, 0, FAKE, FAKE, FAKE, FAKE, None, None) == 3      # pool < 1
    assert m(None, 2, 16, 4, FAKE, FAKE, FAKE, FAKE, None, None) == 3      # no cu_seqlens
    assert m(FAKE, 0, 16, 4, FAKE, FAKE, FAKE, FAKE, None, None) == 3      # no sequence
    assert m(FAKE, 2, 16, 4, FAKE, None, FAKE, FAKE, None, None) == 3      # no output
    assert lib.dsa_last_error_message().decode().startswith("dsa_kpool_metadata")
    pl = lib.dsa_kpool_pool
    assert pl(FAKE, 16, 12, FAKE, FAKE, 2, 4, 4, FAKE, None) == 3           # D not a multiple of 8
    assert pl(FAKE, 16, 128, FAKE, FAKE, 2, 4, 5, FAKE, None) == 3          # more pools than tokens / P
    assert pl(P(0x10002), 16, 128, FAKE, FAKE, 2, 4, 4, FAKE, None) == 3    # misaligned rows
    assert lib.dsa_last_error_message().decode().startswith("dsa_kpool_pool")
    tk = lib.dsa_kpool_topk
    tk.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, P, P, P, ctypes.c_size_t, P]

    def topk(**kw):
        a = dict(T=8, pools=2, Hi=64, Di=128, K=2048, pool=4, ws=P(0x100000), wsb=1 << 20)
        a.update(kw)
        return tk(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, a["T"], a["pools"], a["Hi"], a["Di"], a["K"], a["pool"], FAKE,
                  FAKE, a["ws"], a["wsb"], None)

    for bad in [dict(K=0), dict(K=2049), dict(Hi=65), dict(Di=64), dict(pool=0), dict(T=-1)]:
        assert topk(**bad) == 3, bad
    assert topk(ws=None) == 4 and topk(wsb=64) == 4
    assert lib.dsa_kpool_topk_workspace_size(8, 2048) >= 8 * 2048 * 4 + 8 * 4
    ug = lib.dsa_kpool_unpool_grad
    assert ug(FAKE, 16, 6, FAKE, FAKE, 2, 4, 4, FAKE, None) == 3            # D not a multiple of 4
    assert ug(P(0x100000), 16, 8, FAKE, FAKE, 2, 4, 4, P(0x100040), None) == 3  # dx overlaps dcat
    assert lib.dsa_last_error_message().decode().startswith("dsa_kpool_unpool_grad")
