"""csa_index_topk_static: the indexer + top-k for callers that cannot
allocate device memory (their own pool already holds the GPU's memory, or
cudaMalloc's host blocking / device synchronisation is not allowed where they
call).  Its scratch is libcsa's fixed device array instead of a workspace.

Checked through the C ABI against csa_index_topk with a workspace, on two
calls in a row after a larger call with other keys (the array keeps the
previous call's contents).  This file is
collected last so that a run stopping at the first failure has already run
every other test; it also passes alone in a fresh process.
"""
import numpy as np
import pytest
import torch

import synthetic as syn

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def csa():
    import compressed_sparse_attention_02_gb300 as m
    return m


def test_static_scratch_matches_workspace_entry_point_on_two_calls(csa):
    B, n_cap, k = 8, 65536, 512          # rows of 65536 visible entries, 2 MiB of scores
    t = 4 * n_cap - 1
    p = csa.csa_default_params(topk=k)
    assert csa.csa_workspace_size(csa.CSA_OP_INDEX_TOPK, p, B, 1, n_cap) <= csa.STATIC_SCRATCH_BYTES
    x = syn.indexer_query(60, B, 1, device=DEV)
    kI = syn.indexer_keys(60, B, n_cap, device=DEV)
    pos = torch.full((B, 1), t, dtype=torch.int32, device=DEV)

    idx_ref = torch.empty(B, 1, k, dtype=torch.int32, device=DEV)
    sc_ref = torch.empty(B, 1, k, dtype=torch.float32, device=DEV)
    ws = csa.workspace(csa.CSA_OP_INDEX_TOPK, p, B, 1, n_cap)
    csa.csa_index_topk(p, B, 1, pos, x["qI"], x["wI"], kI, n_cap, idx_ref, sc_ref, ws)
    assert csa.csa_check_status() == 0

    # a larger call with other keys first: longer rows and more sequences
    # leave scores, candidate lists and tie bits in the shared array that the
    # calls below must not pick up
    B2, n2 = 12, 98304
    assert csa.csa_workspace_size(csa.CSA_OP_INDEX_TOPK, p, B2, 1, n2) <= csa.STATIC_SCRATCH_BYTES
    x2 = syn.indexer_query(61, B2, 1, device=DEV)
    kI2 = syn.indexer_keys(61, B2, n2, device=DEV)
    pos2 = torch.full((B2, 1), 4 * n2 - 1, dtype=torch.int32, device=DEV)
    idx2 = torch.empty(B2, 1, k, dtype=torch.int32, device=DEV)
    csa.csa_index_topk_static(p, B2, 1, pos2, x2["qI"], x2["wI"], kI2, n2, idx2, None)
    assert csa.csa_check_status() == 0

    for call in range(2):
        idx = torch.full((B, 1, k), -7, dtype=torch.int32, device=DEV)
        sc = torch.empty(B, 1, k, dtype=torch.float32, device=DEV)
        csa.csa_index_topk_static(p, B, 1, pos, x["qI"], x["wI"], kI, n_cap, idx, sc)
        assert csa.csa_check_status() == 0
        np.testing.assert_array_equal(idx.cpu().numpy(), idx_ref.cpu().numpy(), err_msg="call %d" % call)
        np.testing.assert_allclose(sc.cpu().numpy(), sc_ref.cpu().numpy(), rtol=1e-6, atol=1e-7)


def test_static_scratch_rejects_sizes_beyond_its_maximum(csa):
    """64 sequences x 262144 entries need 64 MiB of scratch: refused before any
    launch (the small buffers passed are never read)."""
    p = csa.csa_default_params(topk=512)
    need = csa.csa_workspace_size(csa.CSA_OP_INDEX_TOPK, p, 64, 1, 262144)
    assert need > csa.STATIC_SCRATCH_BYTES
    small = torch.zeros(4096, dtype=torch.uint8, device=DEV)
    with pytest.raises(csa.CsaError) as e:
        csa.csa_index_topk_static(p, 64, 1, small, small, small, small, 262144, small, None)
    assert e.value.status == 6  # CSA_ERR_WORKSPACE
