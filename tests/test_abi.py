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
    expected = {"dsa_packed_metadata", "dsa_indexer_topk", "dsa_sparse_mla_fwd", "dsa_sparse_mla_bwd",
                "dsa_status_string", "dsa_last_error_message", "dsa_read_device_status"}
    assert expected <= set(names)
    for n in names:
        assert hasattr(lib, n), n


def test_abi_version_and_status_strings(lib):
    assert lib.dsa_abi_version() == 1
    for code in range(8):
        s = lib.dsa_status_string(code).decode()
        assert s.startswith(dsa.STATUS_NAMES[code])


P = ctypes.c_void_p
FAKE = P(0x10000)  # never dereferenced: validation fails before any device use


def fwd(lib, **kw):
    a = dict(q=FAKE, kv=FAKE, idx=FAKE, ln=None, T=4, Tk=8, H=16, Dqk=576, Dv=512, K=64, scale=0.1, out=FAKE,
             lse=FAKE, ws=P(0x100000), wsb=1 << 20, stream=None)
    a.update(kw)
    return lib.dsa_sparse_mla_fwd(a["q"], a["kv"], a["idx"], a["ln"], a["T"], a["Tk"], a["H"], a["Dqk"], a["Dv"],
                                  a["K"], ctypes.c_float(a["scale"]), a["out"], None, a["lse"], a["ws"], a["wsb"],
                                  a["stream"])


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
