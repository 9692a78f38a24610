"""Hierarchical indexer parity ("DeepSeek-V4 CSA/HCA 与 DeepSeek-V4.1 CSA2"
§11): the Full layer's candidate pool (csa_index_topk_pool) and a Reindex
layer's top-k over it (csa_reindex_topk), against the oracle."""
import numpy as np
import pytest
import torch

import oracle
import synthetic as syn
from _util import bits, check_topk

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def csa():
    import compressed_sparse_attention_02_gb300 as m
    return m


def full_layer(csa, p, x, kI, pos, n_cap, nb):
    B, Q = pos.shape
    idx = torch.full((B, Q, p.topk), -7, dtype=torch.int32, device=DEV)
    sc = torch.empty((B, Q, p.topk), dtype=torch.float32, device=DEV)
    pool = torch.full((B, Q, nb), -7, dtype=torch.int32, device=DEV)
    ws = csa.workspace(csa.CSA_OP_INDEX_TOPK_POOL, p, B, Q, n_cap)
    csa.csa_index_topk_pool(p, B, Q, pos.to(DEV), x["qI"].to(DEV), x["wI"].to(DEV), kI.to(DEV), n_cap, idx, sc, nb,
                            pool, ws)
    st = csa.csa_check_status()
    assert st == 0, csa.csa_status_string(st)
    return idx.cpu().numpy(), sc.cpu().numpy(), pool


def reindex(csa, p, x, kI, pos, n_cap, pool, nb):
    B, Q = pos.shape
    idx = torch.full((B, Q, p.topk), -7, dtype=torch.int32, device=DEV)
    sc = torch.empty((B, Q, p.topk), dtype=torch.float32, device=DEV)
    ws = csa.workspace(csa.CSA_OP_REINDEX_TOPK, p, B, Q, n_cap)
    csa.csa_reindex_topk(p, B, Q, pos.to(DEV), x["qI"].to(DEV), x["wI"].to(DEV), kI.to(DEV), n_cap,
                         torch.as_tensor(pool, dtype=torch.int32).to(DEV), nb, idx, sc, ws)
    st = csa.csa_check_status()
    assert st == 0, csa.csa_status_string(st)
    return idx.cpu().numpy(), sc.cpu().numpy()


def check_full_row(idx, sc, pool, qI, wI, kI, t, k, nb, what):
    V = oracle.visible(t)
    scores = oracle.index_scores(bits(qI), bits(wI), bits(kI)[:V])
    check_topk(idx, scores, k, what + " top-k")
    n = min(k, V)
    if n:
        ref = scores[idx[:n]]
        assert np.all(np.abs(sc[:n] - ref) <= 1e-4 * np.abs(scores).max() + 1e-4 * np.abs(ref)), what + ": scores"
    assert np.all(np.isneginf(sc[n:]))
    check_topk(pool, oracle.block_scores(scores), nb, what + " pool")


def check_reindex_row(idx, sc, pool, qI, wI, kI, t, k, what):
    """The GPU's entries, turned into positions in the pool's entry list, must
    be a valid top-k of the oracle's scores of the pool's entries."""
    V = oracle.visible(t)
    want, ent, esc = oracle.reindex_topk(bits(qI), bits(wI), bits(kI), pool, V, k)
    n = min(k, ent.size)
    assert np.all(idx[n:] == -1), what + ": padding"
    assert np.all(np.isin(idx[:n], ent)), what + ": an entry outside the pool"
    slots = np.searchsorted(ent, idx[:n])
    got = np.full(k, -1, np.int64)
    got[:n] = slots
    check_topk(got, esc, k, what)
    tol = 1e-4 * (np.abs(esc).max() if esc.size else 0.0) + 1e-4 * np.abs(esc[slots])
    assert np.all(np.abs(sc[:n] - esc[slots]) <= tol), what + ": selected scores"
    assert np.all(np.isneginf(sc[n:]))
    return want


@pytest.mark.parametrize("t", [4 * 4096 - 1, 4 * 4093 - 1, 4 * 517 - 1, 4 * 300 - 1, 2, 4 * 9 - 1])
def test_full_layer_pool_and_reindex(csa, t):
    """V = 4096, 4093 (the pool can hold a partial last block), 517, 300 (the
    pool holds every block), 0 and 9 visible entries; pool of 64 blocks."""
    n_cap, nb, k = 4096, 64, 64
    x = syn.indexer_query(30, 2, 1)
    x2 = syn.indexer_query(31, 2, 1)
    kI = syn.indexer_keys(30, 2, n_cap)
    p = csa.csa_default_params(topk=k)
    pos = torch.tensor([[t], [t]], dtype=torch.int32)
    idx, sc, pool = full_layer(csa, p, x, kI, pos, n_cap, nb)
    pool_np = pool.cpu().numpy()
    for b in range(2):
        check_full_row(idx[b, 0], sc[b, 0], pool_np[b, 0], x["qI"][b, 0], x["wI"][b, 0], kI[b], t, k, nb,
                       "t=%d b=%d" % (t, b))
    # the Reindex layer over the GPU's own pool, with another layer's query
    ridx, rsc = reindex(csa, p, x2, kI, pos, n_cap, pool_np, nb)
    for b in range(2):
        check_reindex_row(ridx[b, 0], rsc[b, 0], pool_np[b, 0], x2["qI"][b, 0], x2["wI"][b, 0], kI[b], t, k,
                          "reindex t=%d b=%d" % (t, b))


def test_partial_last_block_in_the_pool(csa):
    """V = 8*40 + 3 (41 visible blocks): a pool of 16 blocks ending with the
    partial block 40 (entries 320..322); the Reindex layer must score those
    three and nothing past V."""
    n_cap, nb, k = 1024, 16, 128
    V = 8 * 40 + 3
    t = 4 * V + 2
    assert oracle.visible(t) == V
    x = syn.indexer_query(32, 1, 1)
    kI = syn.indexer_keys(32, 1, n_cap)
    pool = np.array([[[0, 3, 5, 8, 13, 21, 22, 23, 24, 25, 26, 27, 28, 34, 39, 40]]], dtype=np.int32)
    pos = torch.tensor([[t]], dtype=torch.int32)
    p = csa.csa_default_params(topk=k)
    ridx, rsc = reindex(csa, p, x, kI, pos, n_cap, pool, nb)
    want = check_reindex_row(ridx[0, 0], rsc[0, 0], pool[0, 0], x["qI"][0, 0], x["wI"][0, 0], kI[0], t, k, "partial")
    assert np.array_equal(ridx[0, 0], want)  # k covers the whole pool: 15*8 + 3 entries
    assert (ridx[0, 0] >= 0).sum() == 15 * 8 + 3


def test_a_foreign_pool_never_yields_an_invisible_entry(csa):
    """A pool with fewer blocks than the Full layer would write (and a block
    id past the cache) is outside the contract; the selection may then hold
    -1 slots, but every entry it returns is a visible entry of the pool, and
    the id past the cache is reported."""
    n_cap, nb, k = 1024, 16, 128
    V = 8 * 40 + 3
    t = 4 * V + 2
    x = syn.indexer_query(37, 1, 1)
    kI = syn.indexer_keys(37, 1, n_cap)
    pool = np.array([[[0, 3, 5, 8, 13, 21, 34, 40] + [-1] * 8]], dtype=np.int32)
    pos = torch.tensor([[t]], dtype=torch.int32)
    p = csa.csa_default_params(topk=k)
    ridx, _ = reindex(csa, p, x, kI, pos, n_cap, pool, nb)
    got = ridx[0, 0][ridx[0, 0] >= 0]
    assert set(got) <= set(oracle.pool_entries(pool[0, 0], V)) and len(got) == 7 * 8 + 3
    pool[0, 0, 8] = 5000  # block 5000 starts past the 1024-entry cache
    idx = torch.empty((1, 1, k), dtype=torch.int32, device=DEV)
    ws = csa.workspace(csa.CSA_OP_REINDEX_TOPK, p, 1, 1, n_cap)
    csa.csa_reindex_topk(p, 1, 1, pos.to(DEV), x["qI"].to(DEV), x["wI"].to(DEV), kI.to(DEV), n_cap,
                         torch.as_tensor(pool).to(DEV), nb, idx, None, ws)
    assert csa.csa_check_status() == 5  # CSA_ERR_INDEX_RANGE
    got = idx.cpu().numpy()[0, 0]
    assert set(got[got >= 0]) <= set(oracle.pool_entries(pool[0, 0], V))


def test_reindex_with_the_full_layers_query_gives_the_full_topk(csa):
    """With the Full layer's own q^I / w^I, the Reindex top-k over a pool of
    at least k blocks is the Full layer's top-k (ties aside)."""
    n_cap, nb, k = 8192, 128, 128
    t = 4 * n_cap - 1
    x = syn.indexer_query(33, 2, 1)
    kI = syn.indexer_keys(33, 2, n_cap)
    p = csa.csa_default_params(topk=k)
    pos = torch.tensor([[t], [t - 4 * 77]], dtype=torch.int32)
    idx, sc, pool = full_layer(csa, p, x, kI, pos, n_cap, nb)
    ridx, rsc = reindex(csa, p, x, kI, pos, n_cap, pool.cpu().numpy(), nb)
    for b in range(2):
        assert np.array_equal(ridx[b, 0], idx[b, 0]), "b=%d" % b
        np.testing.assert_array_equal(rsc[b, 0], sc[b, 0])


def test_many_queries_prefill_shaped(csa):
    """2 sequences x 6 queries with their own visible counts: the Full layer
    runs the four-queries-per-tile indexer, the Reindex layer one query per
    tile (a pool belongs to one query)."""
    B, Q, n_cap, nb, k = 2, 6, 3000, 32, 96
    x = syn.indexer_query(34, B, Q)
    x2 = syn.indexer_query(35, B, Q)
    kI = syn.indexer_keys(34, B, n_cap)
    pos = torch.tensor([[4 * (700 + 389 * j) + b for j in range(Q)] for b in range(B)], dtype=torch.int32)
    p = csa.csa_default_params(topk=k)
    idx, sc, pool = full_layer(csa, p, x, kI, pos, n_cap, nb)
    pool_np = pool.cpu().numpy()
    ridx, rsc = reindex(csa, p, x2, kI, pos, n_cap, pool_np, nb)
    for b in range(B):
        for j in range(Q):
            tt = int(pos[b, j])
            check_full_row(idx[b, j], sc[b, j], pool_np[b, j], x["qI"][b, j], x["wI"][b, j], kI[b], tt, k, nb,
                           "b=%d q=%d" % (b, j))
            check_reindex_row(ridx[b, j], rsc[b, j], pool_np[b, j], x2["qI"][b, j], x2["wI"][b, j], kI[b], tt, k,
                              "reindex b=%d q=%d" % (b, j))


def test_equal_block_scores_take_the_smaller_blocks(csa):
    """Every key equal: every block score ties, so the pool is blocks 0..nb-1
    and the Reindex layer (all scores equal too) takes the k lowest entries."""
    n_cap, nb, k = 5000, 48, 200
    t = 4 * n_cap - 1
    x = syn.indexer_query(36, 1, 1)
    one = syn.indexer_keys(36, 1, 1)
    kI = one.view(torch.uint8)[:, torch.zeros(n_cap, dtype=torch.long)].contiguous().view(torch.float8_e4m3fn)
    p = csa.csa_default_params(topk=k)
    pos = torch.tensor([[t]], dtype=torch.int32)
    idx, sc, pool = full_layer(csa, p, x, kI, pos, n_cap, nb)
    assert np.array_equal(pool.cpu().numpy()[0, 0], np.arange(nb))
    ridx, rsc = reindex(csa, p, x, kI, pos, n_cap, pool.cpu().numpy(), nb)
    assert np.array_equal(ridx[0, 0], np.arange(k))


@pytest.mark.parametrize("cfg,samples", [(2, [0, 37]), (3, [6])])
def test_full_size_pool_of_2048_blocks_sampled(csa, cfg, samples):
    """The pages' sizes: 2048 blocks (16384 candidates) from the 32768 and
    262144 entries of the 128K and 1M decode configurations, every sequence
    run, sampled sequences checked."""
    w = syn.WORKLOADS[cfg]
    nb = 2048
    x = syn.indexer_query(cfg, w.B, 1, device=DEV)
    x2 = syn.indexer_query(40 + cfg, w.B, 1, device=DEV)
    kI = syn.indexer_keys(cfg, w.B, w.n_cap, device=DEV, hadamard_rows=w.hadamard_kI)
    p = csa.csa_default_params(topk=w.topk)
    pos = torch.full((w.B, 1), w.t, dtype=torch.int32)
    idx, sc, pool = full_layer(csa, p, x, kI, pos, w.n_cap, nb)
    pool_np = pool.cpu().numpy()
    ridx, rsc = reindex(csa, p, x2, kI, pos, w.n_cap, pool_np, nb)
    for b in samples:
        check_full_row(idx[b, 0], sc[b, 0], pool_np[b, 0], x["qI"][b, 0], x["wI"][b, 0], kI[b], w.t, w.topk, nb,
                       "c%d b=%d" % (cfg, b))
        check_reindex_row(ridx[b, 0], rsc[b, 0], pool_np[b, 0], x2["qI"][b, 0], x2["wI"][b, 0], kI[b], w.t, w.topk,
                          "reindex c%d b=%d" % (cfg, b))
