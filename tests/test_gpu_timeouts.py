"""Failure detection: every device wait of the library's kernels is bounded.

With the test-only switch csa_test_set_wait_fault (a short wait limit, and
one signal withheld so that a wait must run out) each kernel family's waits
give up, the kernels finish (tensor memory released, copies in flight
waited for), the call reports CSA_ERR_TIMEOUT, and the very next normal call
on the same stream is parity-green against the oracle.  Families: the
lightning indexer (contiguous key tiles, and the Reindex form that gathers
pool blocks), the cluster top-k, and the sparse attention in its cluster and
split-KV forms."""
import contextlib

import numpy as np
import pytest
import torch

import oracle
import synthetic as syn
from _util import assert_close, bits, check_topk

pytestmark = pytest.mark.gpu
DEV = "cuda"
LIMIT_US = 200
TIMEOUT = 4  # CSA_ERR_TIMEOUT


@pytest.fixture(scope="module")
def csa():
    import compressed_sparse_attention_02_gb300 as m
    return m


@contextlib.contextmanager
def faulted(csa, fault):
    csa.csa_test_set_wait_fault(LIMIT_US, fault)
    try:
        yield
    finally:
        csa.csa_test_set_wait_fault(0, 0)


def run_index_topk(csa, p, x, kI, pos, n_cap):
    B, Q = pos.shape
    idx = torch.full((B, Q, p.topk), -7, dtype=torch.int32, device=DEV)
    sc = torch.empty((B, Q, p.topk), dtype=torch.float32, device=DEV)
    ws = csa.workspace(csa.CSA_OP_INDEX_TOPK, p, B, Q, n_cap)
    csa.csa_index_topk(p, B, Q, pos.to(DEV), x["qI"].to(DEV), x["wI"].to(DEV), kI.to(DEV), n_cap, idx, sc, ws)
    return csa.csa_check_status(), idx.cpu().numpy(), sc.cpu().numpy()


@pytest.mark.parametrize("fault,n_cap", [("indexer", 1000), ("topk", 20000)])
def test_indexer_and_topk_waits_give_up(csa, fault, n_cap):
    """A row of 1000 entries (indexer fault) and one of 20000 (five chunks: a
    cluster of five top-k CTAs, top-k fault)."""
    p = csa.csa_default_params(topk=64)
    x = syn.indexer_query(91, 1, 1)
    kI = syn.indexer_keys(91, 1, n_cap)
    t = 4 * n_cap - 1
    pos = torch.tensor([[t]], dtype=torch.int32)
    bit = {"indexer": csa.CSA_TEST_FAULT_INDEXER, "topk": csa.CSA_TEST_FAULT_TOPK}[fault]
    with faulted(csa, bit):
        st, _, _ = run_index_topk(csa, p, x, kI, pos, n_cap)
    assert st == TIMEOUT, csa.csa_status_string(st)
    st, idx, sc = run_index_topk(csa, p, x, kI, pos, n_cap)
    assert st == 0, csa.csa_status_string(st)
    V = oracle.visible(t)
    scores = oracle.index_scores(bits(x["qI"][0, 0]), bits(x["wI"][0, 0]), bits(kI[0])[:V])
    check_topk(idx[0, 0], scores, p.topk, "after the timeout")
    ref = scores[idx[0, 0]]
    assert np.all(np.abs(sc[0, 0] - ref) <= 1e-4 * np.abs(scores).max() + 1e-4 * np.abs(ref))


def test_reindex_waits_give_up(csa):
    """The Reindex form (pool blocks gathered by the indexer's lane-parallel
    producer)."""
    n_cap, nb = 4096, 16
    p = csa.csa_default_params(topk=32)
    x = syn.indexer_query(92, 1, 1)
    kI = syn.indexer_keys(92, 1, n_cap)
    t = 4 * n_cap - 1
    pos = torch.tensor([[t]], dtype=torch.int32, device=DEV)
    pool = torch.arange(0, 2 * nb, 2, dtype=torch.int32, device=DEV).view(1, 1, nb)

    def run():
        idx = torch.full((1, 1, p.topk), -7, dtype=torch.int32, device=DEV)
        sc = torch.empty((1, 1, p.topk), dtype=torch.float32, device=DEV)
        ws = csa.workspace(csa.CSA_OP_REINDEX_TOPK, p, 1, 1, n_cap)
        csa.csa_reindex_topk(p, 1, 1, pos, x["qI"].to(DEV), x["wI"].to(DEV), kI.to(DEV), n_cap, pool, nb, idx, sc, ws)
        return csa.csa_check_status(), idx.cpu().numpy(), sc.cpu().numpy()
    with faulted(csa, csa.CSA_TEST_FAULT_INDEXER):
        st, _, _ = run()
    assert st == TIMEOUT, csa.csa_status_string(st)
    st, idx, sc = run()
    assert st == 0, csa.csa_status_string(st)
    V = oracle.visible(t)
    _, ent, esc = oracle.reindex_topk(bits(x["qI"][0, 0]), bits(x["wI"][0, 0]), bits(kI[0]), pool[0, 0].cpu().numpy(),
                                      V, p.topk)
    slots = np.searchsorted(ent, idx[0, 0])
    assert np.all(np.isin(idx[0, 0], ent))
    check_topk(slots, esc, p.topk, "reindex after the timeout")


@pytest.mark.parametrize("form", ["split-kv", "cluster"])
def test_attention_waits_give_up(csa, form):
    """Four queries over 640 rows each: with a full workspace the split-KV
    form (slices merged by a second kernel), with one too small for any slice
    the cluster form (slices merged through distributed shared memory)."""
    n_cap, k, B = 4096, 512, 4
    t = 4 * n_cap - 1
    x = syn.decode_inputs(syn.Workload("timeout-attn", 93, "decode", B=B, t=t, topk=k, n_cap=n_cap))
    p = csa.csa_default_params(topk=k)
    g = torch.Generator().manual_seed(93)
    idx = torch.stack([torch.sort(torch.randperm(n_cap, generator=g)[:k])[0] for _ in range(B)]).to(torch.int32)
    idx = idx.view(B, 1, k)
    slice_bytes = (64 * 512 + 2 * 64) * 4
    ws = (csa.workspace(csa.CSA_OP_SPARSE_ATTN, p, B, 1, n_cap) if form == "split-kv"
          else torch.empty(B * slice_bytes, dtype=torch.uint8, device=DEV))
    g_in = {kk: x[kk].to(DEV) for kk in ("q", "kv", "swa", "sink")}

    def run():
        out = torch.empty(B, 1, 64, 512, dtype=torch.bfloat16, device=DEV)
        lse = torch.empty(B, 1, 64, dtype=torch.float32, device=DEV)
        csa.csa_sparse_attn(p, B, 1, torch.full((B, 1), t, dtype=torch.int32, device=DEV), g_in["q"], g_in["kv"],
                            n_cap, idx.to(DEV), g_in["swa"], 0, 128, None, g_in["sink"], out, lse, ws)
        return csa.csa_check_status(), out.float().cpu().numpy(), lse.cpu().numpy()
    with faulted(csa, csa.CSA_TEST_FAULT_ATTN):
        st, _, _ = run()
    assert st == TIMEOUT, csa.csa_status_string(st)
    st, out, lse = run()
    assert st == 0, csa.csa_status_string(st)
    W = p.swa_window
    for b in (0, B - 1):
        ring = bits(x["swa"][b])
        o, l = oracle.attend_query(t, bits(x["q"][b, 0]), idx[b, 0].numpy(), bits(x["kv"][b]), lambda u: ring[u % W],
                                   bits(x["sink"]), W=W)
        assert_close(out[b, 0], o, "%s b=%d after the timeout" % (form, b))
        np.testing.assert_allclose(lse[b, 0], l, rtol=1e-3, atol=1e-3)


def test_switch_refuses_bad_arguments(csa):
    """Unknown fault bits, or a fault without a wait limit, are refused; the
    switch is off afterwards (a normal call is clean)."""
    import ctypes
    raw = ctypes.CDLL(csa.LIBRARY_PATH)
    raw.csa_test_set_wait_fault.restype = ctypes.c_int
    assert raw.csa_test_set_wait_fault(ctypes.c_uint32(100), ctypes.c_uint32(8)) == 1
    assert raw.csa_test_set_wait_fault(ctypes.c_uint32(0), ctypes.c_uint32(1)) == 1
    assert raw.csa_test_set_wait_fault(ctypes.c_uint32(0), ctypes.c_uint32(0)) == 0
