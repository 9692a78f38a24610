"""Lightning indexer + top-k parity (csa_index_topk) against the oracle."""
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


def run(csa, p, qI, wI, kI, q_pos, n_cap):
    B, Q = q_pos.shape
    idx = torch.full((B, Q, p.topk), -7, dtype=torch.int32, device=DEV)
    sc = torch.empty((B, Q, p.topk), dtype=torch.float32, device=DEV)
    ws = csa.workspace(csa.CSA_OP_INDEX_TOPK, p, B, Q, n_cap)
    csa.csa_index_topk(p, B, Q, q_pos.to(DEV), qI.to(DEV), wI.to(DEV), kI.to(DEV), n_cap, idx, sc, ws)
    st = csa.csa_check_status()
    assert st == 0, csa.csa_status_string(st)
    return idx.cpu().numpy(), sc.cpu().numpy()


def check_row(idx, sc, qI, wI, kI, t, k, m=4, what=""):
    V = oracle.visible(t, m)
    scores = oracle.index_scores(bits(qI), bits(wI), bits(kI)[:V])
    check_topk(idx, scores, k, what)
    n = min(k, V)
    sel = idx[:n]
    ref = scores[sel]
    tol = 1e-4 * (np.abs(scores).max() if V else 0.0) + 1e-4 * np.abs(ref)
    assert np.all(np.abs(sc[:n] - ref) <= tol), what + ": selected scores"
    assert np.all(np.isneginf(sc[n:]))


def test_tiny_decode_config(csa):
    w = syn.WORKLOADS[0]
    x = syn.indexer_query(0, 1, 1)
    kI = syn.indexer_keys(0, 1, w.n_cap)
    p = csa.csa_default_params(topk=w.topk)
    idx, sc = run(csa, p, x["qI"], x["wI"], kI, torch.tensor([[w.t]], dtype=torch.int32), w.n_cap)
    check_row(idx[0, 0], sc[0, 0], x["qI"][0, 0], x["wI"][0, 0], kI[0], w.t, w.topk, what="c0")


@pytest.mark.parametrize("t", [2, 3, 17, 259, 1023])
def test_visible_count_below_and_at_k(csa, t):
    """V(t) = 0, 1, 4, 65 and 256 entries with k = 64 (the -1 padding and the
    'k covers every visible entry' case)."""
    x = syn.indexer_query(1, 1, 1)
    kI = syn.indexer_keys(1, 1, 256)
    p = csa.csa_default_params(topk=64)
    idx, sc = run(csa, p, x["qI"], x["wI"], kI, torch.tensor([[t]], dtype=torch.int32), 256)
    check_row(idx[0, 0], sc[0, 0], x["qI"][0, 0], x["wI"][0, 0], kI[0], t, 64, what="t=%d" % t)


def test_exact_ties_go_to_the_smaller_index(csa):
    """Keys repeat with period 37: every score occurs several times exactly."""
    n_cap = 1000
    x = syn.indexer_query(2, 1, 1)
    base = syn.indexer_keys(2, 1, 37)
    kI = base.view(torch.uint8)[:, torch.arange(n_cap) % 37].contiguous().view(torch.float8_e4m3fn)
    p = csa.csa_default_params(topk=100)
    t = 4 * n_cap - 1
    idx, sc = run(csa, p, x["qI"], x["wI"], kI, torch.tensor([[t]], dtype=torch.int32), n_cap)
    check_row(idx[0, 0], sc[0, 0], x["qI"][0, 0], x["wI"][0, 0], kI[0], t, 100, what="ties")


def test_all_negative_head_weights(csa):
    n_cap = 700
    x = syn.indexer_query(3, 1, 1)
    wI = (-x["wI"].float().abs()).to(torch.bfloat16)
    kI = syn.indexer_keys(3, 1, n_cap)
    p = csa.csa_default_params(topk=64)
    t = 4 * n_cap - 1
    idx, sc = run(csa, p, x["qI"], wI, kI, torch.tensor([[t]], dtype=torch.int32), n_cap)
    check_row(idx[0, 0], sc[0, 0], x["qI"][0, 0], wI[0, 0], kI[0], t, 64, what="negative w")


def test_many_queries_causal(csa):
    """Prefill-shaped call: 2 sequences x 37 queries (a ragged group of the
    4-queries-per-CTA kernel), each with its own visible count."""
    B, Q, n_cap = 2, 37, 420
    x = syn.indexer_query(4, B, Q)
    kI = syn.indexer_keys(4, B, n_cap)
    pos = torch.tensor([[300 + 37 * j + b for j in range(Q)] for b in range(B)], dtype=torch.int32)
    p = csa.csa_default_params(topk=128)
    idx, sc = run(csa, p, x["qI"], x["wI"], kI, pos, n_cap)
    for b in range(B):
        for j in range(Q):
            check_row(idx[b, j], sc[b, j], x["qI"][b, j], x["wI"][b, j], kI[b], int(pos[b, j]), 128,
                      what="b=%d q=%d" % (b, j))


def test_position_beyond_cache_is_reported(csa):
    x = syn.indexer_query(5, 1, 1)
    kI = syn.indexer_keys(5, 1, 100)
    p = csa.csa_default_params(topk=16)
    idx = torch.empty((1, 1, 16), dtype=torch.int32, device=DEV)
    ws = csa.workspace(csa.CSA_OP_INDEX_TOPK, p, 1, 1, 100)
    csa.csa_index_topk(p, 1, 1, torch.tensor([[4000]], dtype=torch.int32, device=DEV), x["qI"].to(DEV),
                       x["wI"].to(DEV), kI.to(DEV), 100, idx, None, ws)
    assert csa.csa_check_status() == 5  # CSA_ERR_INDEX_RANGE; V clamped to the cache
    check_topk(idx[0, 0].cpu().numpy(), oracle.index_scores(bits(x["qI"][0, 0]), bits(x["wI"][0, 0]),
                                                             bits(kI[0])), 16)


@pytest.mark.parametrize("cfg,samples", [(1, [0, 31]), (2, [0, 29, 63]), (3, [5, 7])])
def test_full_size_decode_configs_sampled(csa, cfg, samples):
    """The decode configurations at full size in the launch configuration the
    benchmark times; every sequence runs, sampled sequences are checked."""
    w = syn.WORKLOADS[cfg]
    x = syn.indexer_query(cfg, w.B, 1, device=DEV)
    kI = syn.indexer_keys(cfg, w.B, w.n_cap, device=DEV, hadamard_rows=w.hadamard_kI)
    p = csa.csa_default_params(topk=w.topk)
    pos = torch.full((w.B, 1), w.t, dtype=torch.int32)
    idx, sc = run(csa, p, x["qI"], x["wI"], kI, pos, w.n_cap)
    for b in samples:
        check_row(idx[b, 0], sc[b, 0], x["qI"][b, 0], x["wI"][b, 0], kI[b], w.t, w.topk, what="c%d b=%d" % (cfg, b))


def periodic_keys(seed, n_cap, period):
    base = syn.indexer_keys(seed, 1, period)
    return base.view(torch.uint8)[:, torch.arange(n_cap) % period].contiguous().view(torch.float8_e4m3fn)


@pytest.mark.parametrize("period,k", [(1, 512), (5, 700), (37, 300)])
def test_repeated_scores_over_a_long_row(csa, period, k):
    """20000 visible entries (five 4096-entry chunks) whose keys repeat with a
    short period, so each score occurs 20000/period times exactly: with period
    1 every score is equal (the whole row competes in one digit, past every
    candidate buffer, and the k lowest positions win); periods 5 and 37 put
    thousands or hundreds of equal keys at the threshold across chunk
    boundaries."""
    n_cap = 20000
    x = syn.indexer_query(6, 1, 1)
    kI = periodic_keys(6, n_cap, period)
    p = csa.csa_default_params(topk=k)
    t = 4 * n_cap - 1
    idx, sc = run(csa, p, x["qI"], x["wI"], kI, torch.tensor([[t]], dtype=torch.int32), n_cap)
    check_row(idx[0, 0], sc[0, 0], x["qI"][0, 0], x["wI"][0, 0], kI[0], t, k, what="period %d" % period)
    if period == 1:
        assert np.array_equal(idx[0, 0], np.arange(k)), "equal scores: the k lowest positions"


def test_selection_is_exactly_the_keys_of_one_score(csa):
    """Two distinct keys over 20000 entries: the higher-scoring one at every
    16th position (1250 entries) and k = 1250, so the selection is exactly
    those positions and nothing at the threshold is left over."""
    n_cap, k = 20000, 1250
    x = syn.indexer_query(7, 1, 1)
    two = syn.indexer_keys(7, 1, 2)
    s2 = oracle.index_scores(bits(x["qI"][0, 0]), bits(x["wI"][0, 0]), bits(two[0]))
    assert s2[0] != s2[1]
    hi, lo = (0, 1) if s2[0] > s2[1] else (1, 0)
    pick = torch.full((n_cap,), lo, dtype=torch.long)
    pick[::16] = hi
    kI = two.view(torch.uint8)[:, pick].contiguous().view(torch.float8_e4m3fn)
    p = csa.csa_default_params(topk=k)
    t = 4 * n_cap - 1
    idx, sc = run(csa, p, x["qI"], x["wI"], kI, torch.tensor([[t]], dtype=torch.int32), n_cap)
    assert np.array_equal(idx[0, 0], np.arange(0, n_cap, 16))
    check_row(idx[0, 0], sc[0, 0], x["qI"][0, 0], x["wI"][0, 0], kI[0], t, k, what="one score")


@pytest.mark.parametrize("period,k", [(100, 1500), (80, 1000), (600, 2000), (15, 2048)])
def test_long_candidate_list_read_from_global_memory(csa, period, k):
    """80000 visible entries whose keys repeat with a period: with periods
    100, 80 and 600 the crossing digit holds 3200, 4000 and 2532 candidates,
    more than a finish stages in shared memory (2048) but within the row's
    list (5120), so every pass reads them from global memory (period 100: 800
    equal keys at the threshold, 500 of them taken; period 80: the 1000 equal
    keys at the threshold are exactly the keys still needed).  Period 37 puts
    6486 candidates in the digit, past the list: the row is resolved from its
    scores."""
    n_cap = 80000
    x = syn.indexer_query(8, 1, 1)
    kI = periodic_keys(8, n_cap, period)
    p = csa.csa_default_params(topk=k)
    t = 4 * n_cap - 1
    idx, sc = run(csa, p, x["qI"], x["wI"], kI, torch.tensor([[t]], dtype=torch.int32), n_cap)
    check_row(idx[0, 0], sc[0, 0], x["qI"][0, 0], x["wI"][0, 0], kI[0], t, k, what="period %d" % period)


def check_row_bf16(idx, sc, qI, wI, kI, t, k, what):
    """bf16 scores: the returned scores are bf16 values within one bf16 step
    of the oracle's; every entry left out scores (in bf16) at most the
    lowest selected one, up to that step; ascending, -1 padded."""
    V = oracle.visible(t)
    s = oracle.index_scores(bits(qI), bits(wI), bits(kI)[:V])
    r = oracle.bf16_to_f64(oracle.f64_to_bf16_bits(s))
    n = min(k, V)
    sel = idx[:n]
    assert np.all(idx[n:] == -1), what + ": padding"
    assert np.all(np.diff(sel) > 0) and (n == 0 or (sel.min() >= 0 and sel.max() < V)), what + ": order / range"
    got = sc[:n].astype(np.float64)
    assert np.array_equal(oracle.bf16_to_f64(oracle.f64_to_bf16_bits(got)), got), what + ": not bf16 values"
    step = 2.0 ** -7 * np.abs(r[sel]) + 1e-30
    assert np.all(np.abs(got - r[sel]) <= step), what + ": scores"
    if n < V and n > 0:
        kth = got.min()
        out = np.setdiff1d(np.arange(V), sel)
        assert np.all(r[out] <= kth + 2.0 ** -7 * abs(kth)), what + ": a left-out entry outranks the selection"
    assert np.all(np.isneginf(sc[n:]))


@pytest.mark.parametrize("cfg,samples", [(2, [0, 40]), (3, [1])])
def test_bf16_scores_full_size(csa, cfg, samples):
    w = syn.WORKLOADS[cfg]
    x = syn.indexer_query(cfg, w.B, 1, device=DEV)
    kI = syn.indexer_keys(cfg, w.B, w.n_cap, device=DEV, hadamard_rows=w.hadamard_kI)
    p = csa.csa_default_params(topk=w.topk, bf16_scores=1)
    idx, sc = run(csa, p, x["qI"], x["wI"], kI, torch.full((w.B, 1), w.t, dtype=torch.int32), w.n_cap)
    for b in samples:
        check_row_bf16(idx[b, 0], sc[b, 0], x["qI"][b, 0], x["wI"][b, 0], kI[b], w.t, w.topk, "c%d b=%d" % (cfg, b))


@pytest.mark.parametrize("period,k,t", [(37, 700, 4 * 20000 - 1), (1, 512, 4 * 20000 - 1), (5, 64, 4 * 1000 - 1),
                                        (600, 2048, 4 * 80000 - 1)])
def test_bf16_scores_with_ties_go_to_the_smaller_entries(csa, period, k, t):
    """Repeated keys: every bf16 score occurs many times, so the tie rule
    decides most of the selection; the k lowest positions among equal scores
    win (period 1: exactly 0..k-1)."""
    n_cap = (t + 1) // 4
    x = syn.indexer_query(9, 1, 1)
    kI = periodic_keys(9, n_cap, period)
    p = csa.csa_default_params(topk=k, bf16_scores=1)
    idx, sc = run(csa, p, x["qI"], x["wI"], kI, torch.tensor([[t]], dtype=torch.int32), n_cap)
    check_row_bf16(idx[0, 0], sc[0, 0], x["qI"][0, 0], x["wI"][0, 0], kI[0], t, k, "period %d" % period)
    V = oracle.visible(t)
    r = oracle.bf16_to_f64(oracle.f64_to_bf16_bits(oracle.index_scores(bits(x["qI"][0, 0]), bits(x["wI"][0, 0]),
                                                                       bits(kI[0])[:V])))
    want = oracle.topk(r, k)  # ties toward the smaller entry on the bf16 values
    assert np.array_equal(idx[0, 0], want), "tie order"
    if period == 1:
        assert np.array_equal(idx[0, 0], np.arange(k))
