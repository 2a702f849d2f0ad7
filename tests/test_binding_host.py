"""CPU checks of the Python binding: it only marshals arguments, and it refuses tensors the
library cannot take (host memory, wrong dtypes or shapes, mismatched lengths) with an error
before any call reaches the library."""
import pytest
import torch

import sparse_attention_mla_gb300 as dsa
from sparse_attention_mla_gb300 import build_ext


@pytest.fixture(autouse=True, scope="module")
def _library():
    build_ext.build()
    dsa.load_library()


def test_binding_names_match_the_c_abi():
    for name in ("dsa_packed_metadata", "dsa_packed_metadata_cp", "dsa_indexer_topk", "dsa_indexer_topk_cp",
                 "dsa_indexer_topk_with_scores", "dsa_indexer_topk_scored", "dsa_indexer_kl", "dsa_kpool_metadata",
                 "dsa_kpool_pool", "dsa_kpool_topk", "dsa_kpool_unpool_grad", "dsa_sparse_mla_fwd",
                 "dsa_sparse_mla_bwd"):
        assert callable(getattr(dsa, name)), name
        assert name in dsa.declared_symbols(), name


def test_host_tensors_are_refused():
    cu = torch.tensor([0, 4], dtype=torch.int32)  # host memory: the library takes device pointers
    with pytest.raises(ValueError, match="CUDA"):
        dsa.dsa_packed_metadata(cu, 4)
    with pytest.raises(ValueError, match="CUDA"):
        dsa.dsa_packed_metadata_cp(cu, 4)
    q = torch.zeros(2, 64, 576, dtype=torch.bfloat16)
    kv = torch.zeros(4, 576, dtype=torch.bfloat16)
    idx = torch.zeros(2, 8, dtype=torch.int32)
    with pytest.raises(ValueError, match="CUDA"):
        dsa.dsa_sparse_mla_fwd(q, kv, idx, 0.1)


def test_wrong_dtypes_are_refused():
    with pytest.raises(TypeError):
        dsa.dsa_packed_metadata(torch.tensor([0, 4], dtype=torch.int64), 4)
    q = torch.zeros(2, 64, 576, dtype=torch.float32)
    with pytest.raises(TypeError):
        dsa.dsa_sparse_mla_fwd(q, q[0], torch.zeros(2, 8, dtype=torch.int32), 0.1)
    with pytest.raises(TypeError):
        dsa.dsa_indexer_topk_cp(q, q[0], q[:, 0], torch.zeros(2, dtype=torch.int32),
                                torch.zeros(2, dtype=torch.int32), 8)


def test_indexer_scored_and_kl_refuse_host_tensors():
    q_idx = torch.zeros(2, 64, 128, dtype=torch.bfloat16)
    k_idx = torch.zeros(4, 128, dtype=torch.bfloat16)
    w = torch.zeros(2, 64, dtype=torch.float32)
    st = torch.zeros(2, dtype=torch.int32)
    with pytest.raises(ValueError, match="CUDA"):
        dsa.dsa_indexer_topk_scored(q_idx, k_idx, w, st, 8)
    idx = torch.zeros(2, 8, dtype=torch.int32)
    prob = torch.zeros(2, 8, dtype=torch.float32)
    with pytest.raises(ValueError, match="CUDA"):
        dsa.dsa_indexer_kl(q_idx, k_idx, w, idx, prob, 0.001, topk_score=prob)
