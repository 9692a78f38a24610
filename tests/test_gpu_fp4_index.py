"""FP4 indexer (index_format = 1; "DeepSeek-V4 CSA/HCA 与 DeepSeek-V4.1 CSA2"
§16.2, "DeepSeek-V4 的 KV 压缩" §7.2): the key and query quantizers bit for
bit against the oracle, and the block-scaled tensor-core indexer + top-k
against the oracle's scores over the oracle's own FP4 rows."""
import numpy as np
import pytest
import torch

import oracle
import synthetic as syn
from _util import (bits, check_topk, pack_index_keys_fp4, pack_index_query_fp4, unpack_index_keys_fp4,
                   unpack_index_query_fp4)

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def csa():
    import compressed_sparse_attention_02_gb300 as m
    return m


def plant_edges(x):
    """Edge rows for the quantizer (x: fp32 [n][128], n >= 8)."""
    x[0] = 0.0                                                  # zero blocks: scale byte 0, codes 0
    x[1, :32] = -1e-3                                           # a block of one tiny negative value
    x[1, 32:64] = torch.tensor([6.0, 5.0, 2.5, 0.25, 0.75, 1.25, 1.75, 3.5] * 4)  # ties of x/s at s = 1
    x[2] = 3.0e38                                               # near the largest bf16: scale 2^126
    x[3, :32] = 1e-39                                           # bf16 subnormals: the smallest scale
    x[3, 32:64] = 0.75                                          # amax = 6 * 2^-3 exactly
    x[3, 64:96] = 0.75390625                                    # the next bf16 above it
    x[4, ::2] = -x[4, ::2]
    x[5] = x[5] * torch.exp2(torch.arange(-64, 64, dtype=torch.float32))  # magnitudes across the range
    return x


def test_key_quantizer_matches_the_oracle_bit_for_bit(csa):
    B, n_cap, entry0, n_new = 2, 333, 5, 300
    x = syn.indexer_keys_bf16(40, B, n_new).float()
    x = x * torch.exp2(torch.randint(-12, 12, (B, n_new, 4), generator=torch.Generator().manual_seed(40)).float()
                       ).repeat_interleave(32, dim=2)
    plant_edges(x[0])
    rows = x.to(torch.bfloat16)
    kI = torch.full((csa.index_keys_fp4_bytes(B, n_cap),), 0xAB, dtype=torch.uint8, device=DEV)
    csa.csa_quantize_index_keys_fp4(B, n_new, entry0, rows.to(DEV), n_new * 128, kI, n_cap)
    assert csa.csa_check_status() == 0
    got = kI.cpu().numpy()
    codes, scales = unpack_index_keys_fp4(got, B, n_cap)
    want_c, want_s = oracle.quantize_index_fp4(bits(rows))
    np.testing.assert_array_equal(codes[:, entry0:entry0 + n_new], want_c)
    np.testing.assert_array_equal(scales[:, entry0:entry0 + n_new], want_s)
    # nothing else is written: other entries' codes, other scale bytes
    assert np.all(codes[:, :entry0] == 0xAB) and np.all(codes[:, entry0 + n_new:] == 0xAB)
    assert np.count_nonzero(got[B * n_cap * 64:] != 0xAB) <= B * n_new * 4
    assert np.all(scales[:, :entry0] == 0xAB) and np.all(scales[:, entry0 + n_new:] == 0xAB)


def test_query_quantizer_matches_the_oracle_bit_for_bit(csa):
    n_q = 5
    x = syn.indexer_query_bf16(41, 1, n_q)["qI"].float().view(n_q * 64, 128)
    plant_edges(x)
    rows = x.view(n_q, 64, 128).to(torch.bfloat16)
    qI = torch.full((csa.index_query_fp4_bytes(n_q),), 0xAB, dtype=torch.uint8, device=DEV)
    csa.csa_quantize_index_query_fp4(n_q, rows.to(DEV), qI)
    assert csa.csa_check_status() == 0
    codes, scales, pad = unpack_index_query_fp4(qI.cpu().numpy(), n_q)
    want_c, want_s = oracle.quantize_index_fp4(bits(rows))
    np.testing.assert_array_equal(codes, want_c)
    np.testing.assert_array_equal(scales, want_s)
    assert not pad.any()


class Fp4Inputs:
    """Indexer inputs quantized by the oracle and packed into the device layouts."""

    def __init__(self, seed, B, Q, n_cap, key_seed=None):
        q = syn.indexer_query_bf16(seed, B, Q)
        self.wI = q["wI"]
        self.qc, self.qs = oracle.quantize_index_fp4(bits(q["qI"]))      # [B][Q][64][64], [B][Q][64][4]
        ks = seed if key_seed is None else key_seed
        self.kc, self.ks = oracle.quantize_index_fp4(bits(syn.indexer_keys_bf16(ks, B, n_cap)))
        self.kI = torch.from_numpy(pack_index_keys_fp4(self.kc, self.ks, n_cap))
        self.qI = torch.from_numpy(pack_index_query_fp4(self.qc.reshape(B * Q, 64, 64), self.qs.reshape(B * Q, 64, 4)))
        self.n_cap = n_cap

    def scores(self, b, q, t, m=4):
        V = min(oracle.visible(t, m), self.n_cap)
        return oracle.index_scores_fp4(self.qc[b, q], self.qs[b, q], bits(self.wI[b, q]), self.kc[b, :V],
                                       self.ks[b, :V])


def run(csa, p, x, q_pos):
    B, Q = q_pos.shape
    idx = torch.full((B, Q, p.topk), -7, dtype=torch.int32, device=DEV)
    sc = torch.empty((B, Q, p.topk), dtype=torch.float32, device=DEV)
    ws = csa.workspace(csa.CSA_OP_INDEX_TOPK, p, B, Q, x.n_cap)
    csa.csa_index_topk(p, B, Q, q_pos.to(DEV), x.qI.to(DEV), x.wI.to(DEV), x.kI.to(DEV), x.n_cap, idx, sc, ws)
    st = csa.csa_check_status()
    assert st == 0, csa.csa_status_string(st)
    return idx.cpu().numpy(), sc.cpu().numpy()


def check_row(idx, sc, scores, k, what):
    """The selection is a valid top-k of the oracle's scores; the returned
    scores match within fp32 accumulation error (the FP4 products and each
    32-value block sum are exact, blocks are scaled by powers of two)."""
    V = len(scores)
    check_topk(idx, scores, k, what)
    n = min(k, V)
    ref = scores[idx[:n]]
    tol = 1e-5 * (np.abs(scores).max() if V else 0.0) + 1e-5 * np.abs(ref)
    assert np.all(np.abs(sc[:n] - ref) <= tol), what + ": selected scores"
    assert np.all(np.isneginf(sc[n:]))


def test_decode_rows_over_several_tiles(csa):
    """Three sequences, 2000 entries (15 tiles and a ragged one), each query
    with its own visible count; one query per CTA."""
    x = Fp4Inputs(42, 3, 1, 2000)
    p = csa.csa_default_params(topk=256, index_format=1)
    pos = torch.tensor([[4 * 2000 - 1], [4 * 777 + 2], [130]], dtype=torch.int32)
    idx, sc = run(csa, p, x, pos)
    for b in range(3):
        check_row(idx[b, 0], sc[b, 0], x.scores(b, 0, int(pos[b, 0])), 256, "b=%d" % b)


@pytest.mark.parametrize("t", [2, 3, 17, 259, 1023])
def test_visible_count_below_and_at_k(csa, t):
    x = Fp4Inputs(43, 1, 1, 256)
    p = csa.csa_default_params(topk=64, index_format=1)
    idx, sc = run(csa, p, x, torch.tensor([[t]], dtype=torch.int32))
    check_row(idx[0, 0], sc[0, 0], x.scores(0, 0, t), 64, "t=%d" % t)


def test_prefill_three_queries_per_cta(csa):
    """2 sequences x 7 queries: groups of three queries (the last one ragged),
    one block-scaled MMA per query on a shared key tile."""
    B, Q, n_cap = 2, 7, 900
    x = Fp4Inputs(44, B, Q, n_cap)
    pos = torch.tensor([[1500 + 290 * j + b for j in range(Q)] for b in range(B)], dtype=torch.int32)
    p = csa.csa_default_params(topk=128, index_format=1)
    idx, sc = run(csa, p, x, pos)
    for b in range(B):
        for j in range(Q):
            check_row(idx[b, j], sc[b, j], x.scores(b, j, int(pos[b, j])), 128, "b=%d q=%d" % (b, j))


def test_fp4_queries_with_bf16_scores(csa):
    """The combination the pages report for the selector: FP4 QK path, scores
    rounded to bf16 before the top-k."""
    x = Fp4Inputs(45, 2, 1, 3000)
    p = csa.csa_default_params(topk=512, index_format=1, bf16_scores=1)
    t = 4 * 3000 - 1
    idx, sc = run(csa, p, x, torch.full((2, 1), t, dtype=torch.int32))
    for b in range(2):
        s = x.scores(b, 0, t)
        r = oracle.bf16_to_f64(oracle.f64_to_bf16_bits(s))
        sel = idx[b, 0]
        got = sc[b, 0].astype(np.float64)
        assert np.all(np.diff(sel) > 0) and sel.min() >= 0 and sel.max() < len(s)
        assert np.array_equal(oracle.bf16_to_f64(oracle.f64_to_bf16_bits(got)), got)
        assert np.all(np.abs(got - r[sel]) <= 2.0 ** -7 * np.abs(r[sel]) + 1e-30)
        out = np.setdiff1d(np.arange(len(s)), sel)
        kth = got.min()
        assert np.all(r[out] <= kth + 2.0 ** -7 * abs(kth)), "a left-out entry outranks the selection"


@pytest.mark.parametrize("cfg,samples", [(2, (0, 63)), (3, (5,))])
def test_full_size_decode_sampled_rows(csa, cfg, samples):
    """decode-b64-128k and v4pro-decode-b8-1m with FP4 keys and queries
    (quantized on the device by the library's own quantizers); sampled rows
    against the oracle, which quantizes those sequences' bf16 rows itself."""
    w = syn.WORKLOADS[cfg]
    B, n_cap, k, t = w.B, w.n_cap, w.topk, w.t
    q = syn.indexer_query_bf16(w.config, B, 1, device=DEV)
    keys = syn.indexer_keys_bf16(w.config, B, n_cap, device=DEV)
    kI = torch.empty(csa.index_keys_fp4_bytes(B, n_cap), dtype=torch.uint8, device=DEV)
    qI = torch.empty(csa.index_query_fp4_bytes(B), dtype=torch.uint8, device=DEV)
    csa.csa_quantize_index_keys_fp4(B, n_cap, 0, keys, n_cap * 128, kI, n_cap)
    csa.csa_quantize_index_query_fp4(B, q["qI"], qI)
    p = csa.csa_default_params(topk=k, index_format=1)
    idx = torch.empty((B, 1, k), dtype=torch.int32, device=DEV)
    sc = torch.empty((B, 1, k), dtype=torch.float32, device=DEV)
    ws = csa.workspace(csa.CSA_OP_INDEX_TOPK, p, B, 1, n_cap)
    csa.csa_index_topk(p, B, 1, torch.full((B, 1), t, dtype=torch.int32, device=DEV), qI, q["wI"], kI, n_cap, idx,
                       sc, ws)
    assert csa.csa_check_status() == 0
    idx, sc = idx.cpu().numpy(), sc.cpu().numpy()
    for b in samples:
        qc, qs = oracle.quantize_index_fp4(bits(q["qI"][b, 0]))
        kc, ks = oracle.quantize_index_fp4(bits(keys[b]))
        V = oracle.visible(t)
        s = oracle.index_scores_fp4(qc, qs, bits(q["wI"][b, 0]), kc[:V], ks[:V])
        check_row(idx[b, 0], sc[b, 0], s, k, "b=%d" % b)


def test_full_layer_pool_on_fp4_keys(csa):
    """The Full layer of the hierarchical indexer on FP4 keys: the same top-k
    as the plain call, and a pool that is the oracle's candidate pool of the
    oracle's FP4 scores."""
    B, n_cap, k, blocks = 2, 6000, 256, 256
    x = Fp4Inputs(46, B, 1, n_cap)
    t = 4 * n_cap - 1
    p = csa.csa_default_params(topk=k, index_format=1)
    idx = torch.empty((B, 1, k), dtype=torch.int32, device=DEV)
    pool = torch.empty((B, 1, blocks), dtype=torch.int32, device=DEV)
    ws = csa.workspace(csa.CSA_OP_INDEX_TOPK_POOL, p, B, 1, n_cap)
    q_pos = torch.full((B, 1), t, dtype=torch.int32, device=DEV)
    csa.csa_index_topk_pool(p, B, 1, q_pos, x.qI.to(DEV), x.wI.to(DEV), x.kI.to(DEV), n_cap, idx, None, blocks,
                            pool, ws)
    assert csa.csa_check_status() == 0
    plain, _ = run(csa, p, x, q_pos.cpu())
    np.testing.assert_array_equal(idx.cpu().numpy(), plain)
    pool = pool.cpu().numpy()
    for b in range(B):  # the pool is a valid top-`blocks` of the oracle's block scores
        check_topk(pool[b, 0], oracle.block_scores(x.scores(b, 0, t)), blocks, "pool b=%d" % b)


def reindex_fp4(csa, p, x, pos, pool, nb):
    B, Q = pos.shape
    idx = torch.full((B, Q, p.topk), -7, dtype=torch.int32, device=DEV)
    sc = torch.empty((B, Q, p.topk), dtype=torch.float32, device=DEV)
    ws = csa.workspace(csa.CSA_OP_REINDEX_TOPK, p, B, Q, x.n_cap)
    csa.csa_reindex_topk(p, B, Q, pos.to(DEV), x.qI.to(DEV), x.wI.to(DEV), x.kI.to(DEV), x.n_cap,
                         torch.as_tensor(pool, dtype=torch.int32).to(DEV), nb, idx, sc, ws)
    return idx.cpu().numpy(), sc.cpu().numpy()


def check_reindex_row(idx, sc, pool, x, b, t, k, what):
    """The Reindex selection over FP4 keys, as positions in the pool's entry
    list, is a valid top-k of the oracle's FP4 scores of the pool's entries
    (the pool's visible entries, then the scores of those entries only)."""
    V = oracle.visible(t)
    ent = oracle.pool_entries(pool, V)
    esc = oracle.index_scores_fp4(x.qc[b, 0], x.qs[b, 0], bits(x.wI[b, 0]), x.kc[b, ent], x.ks[b, ent])
    n = min(k, ent.size)
    assert np.all(idx[n:] == -1), what + ": padding"
    assert np.all(np.isin(idx[:n], ent)), what + ": an entry outside the pool"
    slots = np.searchsorted(ent, idx[:n])
    got = np.full(k, -1, np.int64)
    got[:n] = slots
    check_topk(got, esc, k, what)
    tol = 1e-5 * (np.abs(esc).max() if esc.size else 0.0) + 1e-5 * np.abs(esc[slots])
    assert np.all(np.abs(sc[:n] - esc[slots]) <= tol), what + ": selected scores"
    assert np.all(np.isneginf(sc[n:]))
    return ent[np.sort(oracle.topk(esc, k)[:n])] if n else np.empty(0, np.int64)


@pytest.mark.parametrize("t", [4 * 6000 - 1, 2047])
def test_reindex_on_fp4_keys(csa, t):
    """A Reindex layer on FP4 keys: the pool comes from the Full layer of
    another FP4 query set over the same keys (its slots gathered 16 blocks to
    a tile, with the scale words assembled in the producer), and the Reindex
    top-k is checked against the oracle's FP4 scores of the pool's entries.
    t = 2047: 64 visible blocks for 256 pool slots (-1 slots)."""
    B, n_cap, k, nb = 3, 6000, 256, 256
    xf = Fp4Inputs(47, B, 1, n_cap)
    xr = Fp4Inputs(48, B, 1, n_cap, key_seed=47)
    p = csa.csa_default_params(topk=k, index_format=1)
    q_pos = torch.full((B, 1), t, dtype=torch.int32, device=DEV)
    idx = torch.empty((B, 1, k), dtype=torch.int32, device=DEV)
    pool = torch.empty((B, 1, nb), dtype=torch.int32, device=DEV)
    csa.csa_index_topk_pool(p, B, 1, q_pos, xf.qI.to(DEV), xf.wI.to(DEV), xf.kI.to(DEV), n_cap, idx, None, nb, pool,
                            csa.workspace(csa.CSA_OP_INDEX_TOPK_POOL, p, B, 1, n_cap))
    assert csa.csa_check_status() == 0
    pool = pool.cpu().numpy()
    ridx, rsc = reindex_fp4(csa, p, xr, q_pos.cpu(), pool, nb)
    assert csa.csa_check_status() == 0
    for b in range(B):
        check_reindex_row(ridx[b, 0], rsc[b, 0], pool[b, 0], xr, b, t, k, "reindex b=%d" % b)


def test_reindex_on_fp4_keys_partial_block_and_foreign_ids(csa):
    """The partial last block (V = 8*40 + 3) is scored up to V only; a block
    id past the cache is reported and nothing invisible is returned."""
    n_cap, nb, k = 1024, 16, 128
    V = 8 * 40 + 3
    t = 4 * V + 2
    x = Fp4Inputs(49, 1, 1, n_cap)
    p = csa.csa_default_params(topk=k, index_format=1)
    pool = np.array([[[0, 3, 5, 8, 13, 21, 22, 23, 24, 25, 26, 27, 28, 34, 39, 40]]], dtype=np.int32)
    pos = torch.tensor([[t]], dtype=torch.int32)
    ridx, rsc = reindex_fp4(csa, p, x, pos, pool, nb)
    assert csa.csa_check_status() == 0
    want = check_reindex_row(ridx[0, 0], rsc[0, 0], pool[0, 0], x, 0, t, k, "partial")
    assert np.array_equal(ridx[0, 0][:len(want)], want) and (ridx[0, 0] >= 0).sum() == 15 * 8 + 3
    pool[0, 0, 8] = 5000  # past the 1024-entry cache
    ridx, _ = reindex_fp4(csa, p, x, pos, pool, nb)
    assert csa.csa_check_status() == 5  # CSA_ERR_INDEX_RANGE
    got = ridx[0, 0]
    assert set(got[got >= 0]) <= set(oracle.pool_entries(pool[0, 0], V))


def gpu_fp4_rows(csa, config, B, Q, n_cap):
    """FP4 key cache and query records quantized on the device."""
    q = syn.indexer_query_bf16(config, B, Q, device=DEV)
    kI = torch.empty(csa.index_keys_fp4_bytes(B, n_cap), dtype=torch.uint8, device=DEV)
    qI = torch.empty(csa.index_query_fp4_bytes(B * Q), dtype=torch.uint8, device=DEV)
    csa.csa_quantize_index_keys_fp4(B, n_cap, 0, syn.indexer_keys_bf16(config, B, n_cap, device=DEV), n_cap * 128,
                                    kI, n_cap)
    csa.csa_quantize_index_query_fp4(B * Q, q["qI"], qI)
    return kI, qI, q["wI"]


@pytest.mark.parametrize("B", [3, 40])
def test_layer_decode_with_the_fp4_indexer(csa, B):
    """A decode step with index_format = 1 selects what the plain FP4 call
    selects, and outputs the attention over those entries bit for bit."""
    n_cap, k = 2048, 512
    t = 4 * n_cap - 1
    x = syn.decode_inputs(syn.Workload("fp4-index-layer", 97, "decode", B=B, t=t, topk=k, n_cap=n_cap), device=DEV)
    kI, qI, wI = gpu_fp4_rows(csa, 97, B, 1, n_cap)
    p = csa.csa_default_params(topk=k, index_format=1)
    cache = x["kv"].clone()
    idx = torch.empty(B, k, dtype=torch.int32, device=DEV)
    out = torch.empty(B, 64, 512, dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(B, 64, dtype=torch.float32, device=DEV)
    csa.csa_layer_decode(p, B, x["q_pos"], x["ring_Ca"], x["ring_Za"], x["ring_Cb"], x["ring_Zb"], x["Ba"], x["Bb"],
                         x["rms_w"], cache, n_cap, kI, qI, wI, x["q"], x["swa"], x["sink"], idx, out, lse,
                         csa.workspace(csa.CSA_OP_LAYER_DECODE, p, B, 1, n_cap))
    assert csa.csa_check_status() == 0
    plain = torch.empty(B, 1, k, dtype=torch.int32, device=DEV)
    csa.csa_index_topk(p, B, 1, x["q_pos"].view(B, 1), qI, wI, kI, n_cap, plain, None,
                       csa.workspace(csa.CSA_OP_INDEX_TOPK, p, B, 1, n_cap))
    assert torch.equal(idx, plain.view(B, k))
    o = torch.empty(B, 1, 64, 512, dtype=torch.bfloat16, device=DEV)
    l = torch.empty(B, 1, 64, dtype=torch.float32, device=DEV)
    csa.csa_sparse_attn(p, B, 1, x["q_pos"].view(B, 1), x["q"].view(B, 1, 64, 512), cache, n_cap, idx.view(B, 1, k),
                        x["swa"], 0, 128, None, x["sink"], o, l, csa.workspace(csa.CSA_OP_SPARSE_ATTN, p, B, 1, n_cap))
    assert csa.csa_check_status() == 0
    assert torch.equal(out.view(B, 1, 64, 512), o) and torch.equal(lse.view(B, 1, 64), l)


def test_layer_prefill_with_the_fp4_indexer(csa):
    """A prefill chunk with index_format = 1 (three queries per indexer CTA)
    selects what the plain FP4 call selects for the chunk's positions."""
    B, Q, pos0, k = 2, 64, 512, 64
    w = syn.Workload("fp4-index-prefill", 98, "prefill", B=B, t=pos0 + Q - 1, topk=k, n_cap=(pos0 + Q) // 4 + 8, Q=Q,
                     pos0=pos0)
    x = syn.prefill_inputs(w, device=DEV)
    n_cap = x["n_cap"]
    kI, qI, wI = gpu_fp4_rows(csa, 98, B, Q, n_cap)
    p = csa.csa_default_params(topk=k, index_format=1)
    idx = torch.empty(B, Q, k, dtype=torch.int32, device=DEV)
    out = torch.empty(B, Q, 64, 512, dtype=torch.bfloat16, device=DEV)
    csa.csa_layer_prefill(p, B, Q, pos0, x["Ca"], x["Za"], x["Cb"], x["Zb"], x["Cb_prev"], x["Zb_prev"], x["Ba"],
                          x["Bb"], x["rms_w"], x["kv"].clone(), n_cap, kI, qI, wI, x["q"], x["swa"], x["sink"], idx,
                          out, None, csa.workspace(csa.CSA_OP_LAYER_PREFILL, p, B, Q, n_cap))
    assert csa.csa_check_status() == 0
    q_pos = (pos0 + torch.arange(Q, dtype=torch.int32, device=DEV)).view(1, Q).repeat(B, 1).contiguous()
    plain = torch.empty(B, Q, k, dtype=torch.int32, device=DEV)
    csa.csa_index_topk(p, B, Q, q_pos, qI, wI, kI, n_cap, plain, None,
                       csa.workspace(csa.CSA_OP_INDEX_TOPK, p, B, Q, n_cap))
    assert csa.csa_check_status() == 0
    assert torch.equal(idx, plain)
