"""Whole-layer parity (csa_layer_decode / csa_layer_prefill) against the
oracle's composition of the same steps, on every workload of the pages'
configurations (full size; sampled sequences / queries where the oracle
would take too long)."""
import numpy as np
import pytest
import torch

import oracle
import synthetic as syn
from _util import assert_close, bits, check_key_codes, check_topk

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def csa():
    import compressed_sparse_attention_02_gb300 as m
    return m


def run_decode(csa, p, w, g, kv):
    B = w.B
    idx = torch.empty(B, p.topk, dtype=torch.int32, device=DEV)
    out = torch.empty(B, 64, 512, dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(B, 64, dtype=torch.float32, device=DEV)
    ws = csa.workspace(csa.CSA_OP_LAYER_DECODE, p, B, 1, w.n_cap)
    csa.csa_layer_decode(p, B, g["q_pos"], g["ring_Ca"], g["ring_Za"], g["ring_Cb"], g["ring_Zb"], g["Ba"], g["Bb"],
                         g["rms_w"], kv, w.n_cap, g["kI"], g["qI"], g["wI"], g["q"], g["swa"], g["sink"], idx, out, lse,
                         ws)
    st = csa.csa_check_status()
    assert st == 0, csa.csa_status_string(st)
    return idx.cpu().numpy(), out.float().cpu().numpy(), lse.cpu().numpy()


def check_decode_seq(w, x, b, kv_in, kv_gpu, idx, out, lse):
    """Oracle decode step of sequence b (its own emission, selection and
    attention) against the GPU results."""
    kv_o, idx_o, out_o, lse_o = oracle.layer_decode_one(
        w.t, bits(x["ring_Ca"][b]), bits(x["ring_Za"][b]), bits(x["ring_Cb"][b]), bits(x["ring_Zb"][b]),
        bits(x["Ba"]), bits(x["Bb"]), bits(x["rms_w"]), kv_in, bits(x["kI"][b]), bits(x["qI"][b, 0]),
        bits(x["wI"][b, 0]), bits(x["q"][b, 0]), bits(x["swa"][b]), bits(x["sink"]), m=w.m, topk_k=w.topk, W=w.W)
    if (w.t + 1) % w.m == 0:
        i = (w.t + 1) // w.m - 1
        assert_close(kv_gpu[i], oracle.bf16_to_f64(kv_o[i]), "emitted entry b=%d" % b)
    V = oracle.visible(w.t, w.m)
    scores = oracle.index_scores(bits(x["qI"][b, 0]), bits(x["wI"][b, 0]), bits(x["kI"][b])[:V])
    n_diff = check_topk(idx, scores, w.topk, "b=%d" % b)
    # the attention is judged over the GPU's own selection (a legal near-tie
    # swap changes the rows, not the kernel's correctness) ...
    swa = bits(x["swa"][b])
    out_g, lse_g = oracle.attend_query(w.t, bits(x["q"][b, 0]), idx, kv_o, lambda u: swa[u % w.W], bits(x["sink"]),
                                       W=w.W)
    assert_close(out, out_g, "out b=%d" % b)
    np.testing.assert_allclose(lse, lse_g, rtol=1e-3, atol=1e-3)
    # ... and the whole step against the oracle's own composition when the
    # selections agree
    if n_diff == 0:
        assert_close(out, out_o, "layer step b=%d" % b)
        np.testing.assert_allclose(lse, lse_o, rtol=1e-3, atol=1e-3)


@pytest.mark.parametrize("cfg,samples", [(0, [0]), (2, [0, 41, 63]), (3, [3])])
def test_layer_decode(csa, cfg, samples):
    w = syn.WORKLOADS[cfg]
    x = syn.decode_inputs(w, device=DEV)
    p = csa.csa_default_params(topk=w.topk)
    kv = x["kv"].clone()
    idx, out, lse = run_decode(csa, p, w, x, kv)
    for b in samples:
        check_decode_seq(w, x, b, bits(x["kv"][b]), kv[b].float().cpu().numpy(), idx[b], out[b], lse[b])


@pytest.mark.parametrize("m,t", [(1, 299), (2, 599), (8, 2399), (8, 2395), (4, 3)])
def test_layer_decode_other_compression_ratios(csa, m, t):
    """Decode steps for m = 1, 2 and 8 (the emitted entry is computed inside
    the top-k launch for m <= 4 and by its own kernel for m = 8), a step that
    emits nothing (t+1 not a multiple of m) and one at the very first block
    (no previous block, fewer visible entries than k)."""
    w = syn.Workload("decode-m%d" % m, 0, "decode", B=3, t=t, topk=64, n_cap=400, m=m)
    x = syn.decode_inputs(w, device=DEV)
    p = csa.csa_default_params(topk=w.topk, m=m)
    kv = x["kv"].clone()
    idx, out, lse = run_decode(csa, p, w, x, kv)
    for b in range(w.B):
        check_decode_seq(w, x, b, bits(x["kv"][b]), kv[b].float().cpu().numpy(), idx[b], out[b], lse[b])


@pytest.mark.parametrize("t,with_key", [(1023, True), (1022, True), (1023, False)])
def test_layer_decode_append_stores_the_new_rows(csa, t, with_key):
    """csa_layer_decode_append: the new window row and the completing entry's
    indexer key, stored by the step's first kernel, give the same step (bit
    for bit) as storing them first and calling csa_layer_decode; the caches
    hold them afterwards; a sequence at position -1 stores nothing; at
    t = 1022 no entry completes and kI is left as it was; without kI_new only
    the window row is stored."""
    w = syn.Workload("decode-append", 0, "decode", B=3, t=t, topk=64, n_cap=400, m=4)
    x = syn.decode_inputs(w, device=DEV)
    x["q_pos"][2] = -1
    p = csa.csa_default_params(topk=w.topk)
    swa_new = x["swa"][:, 5].roll(1, dims=0).contiguous()   # bf16 rows unlike the slots they go to
    kI_new = x["kI"][:, 17].view(torch.uint8).roll(1, dims=0).contiguous()  # valid e4m3 rows
    ref = {k: x[k].clone() for k in ("kv", "swa", "kI")}
    for b in range(2):
        ref["swa"][b, t % w.W] = swa_new[b]
        if with_key and (t + 1) % w.m == 0:
            ref["kI"][b, (t + 1) // w.m - 1].view(torch.uint8).copy_(kI_new[b])
    got = {k: x[k].clone() for k in ("kv", "swa", "kI")}
    res = []
    for form, c in (("plain", ref), ("append", got)):
        idx = torch.empty(w.B, p.topk, dtype=torch.int32, device=DEV)
        out = torch.empty(w.B, 64, 512, dtype=torch.bfloat16, device=DEV)
        lse = torch.empty(w.B, 64, dtype=torch.float32, device=DEV)
        ws = csa.workspace(csa.CSA_OP_LAYER_DECODE, p, w.B, 1, w.n_cap)
        common = (x["Ba"], x["Bb"], x["rms_w"], c["kv"], w.n_cap, c["kI"], x["qI"], x["wI"], x["q"], c["swa"],
                  x["sink"], idx, out, lse, ws)
        rings = (x["ring_Ca"], x["ring_Za"], x["ring_Cb"], x["ring_Zb"])
        if form == "plain":
            csa.csa_layer_decode(p, w.B, x["q_pos"], *rings, *common)
        else:
            csa.csa_layer_decode_append(p, w.B, x["q_pos"], swa_new, kI_new if with_key else None, *rings, *common)
        st = csa.csa_check_status()
        assert st == 0, csa.csa_status_string(st)
        res.append((idx.cpu(), bits(out), lse.cpu()))
    for k in ("kv", "swa", "kI"):
        assert torch.equal(got[k].view(torch.uint8), ref[k].view(torch.uint8)), k
    assert torch.equal(res[0][0], res[1][0])
    assert np.array_equal(res[0][1], res[1][1])
    assert torch.equal(res[0][2], res[1][2])


def test_layer_decode_v4flash_cache_from_the_compressor(csa):
    """Batch 32 x 8192 tokens: the cache is built by the bulk compressor over
    the whole context, then one decode step at t = 8191 re-emits the last
    entry from the staging ring."""
    w = syn.WORKLOADS[1]
    T = w.t + 1
    rows = syn.compressor_rows(1, w.B, T, device=DEV)
    x = syn.decode_inputs(w, device=DEV)
    p = csa.csa_default_params(topk=w.topk)
    kv = torch.zeros(w.B, w.n_cap, 512, dtype=torch.bfloat16, device=DEV)
    csa.csa_compress(p, w.B, w.n_cap, 0, rows["Ca"], rows["Za"], rows["Cb"], rows["Zb"], None, None, x["Ba"], x["Bb"],
                     x["rms_w"], kv, w.n_cap * 512)
    for k in ("Ca", "Za", "Cb", "Zb"):  # the ring holds the last 2m tokens' rows
        u = torch.arange(T - 2 * w.m, T, device=DEV)
        x["ring_" + k] = torch.empty_like(x["ring_" + k])
        x["ring_" + k][:, u % (2 * w.m)] = rows[k][:, u]
    idx, out, lse = run_decode(csa, p, w, x, kv)
    for b in (0, 17):
        kv_o = oracle.compress(0, w.n_cap, bits(rows["Ca"][b]), bits(rows["Za"][b]), bits(rows["Cb"][b]),
                               bits(rows["Zb"][b]), None, None, bits(x["Ba"]), bits(x["Bb"]), bits(x["rms_w"]))
        kv_g = kv[b].float().cpu().numpy()
        assert_close(kv_g, kv_o, "bulk cache b=%d" % b)
        check_decode_seq(w, x, b, oracle.f64_to_bf16_bits(kv_o), kv_g, idx[b], out[b], lse[b])


def run_prefill(csa, p, w, x):
    B, Q = w.B, w.Q
    g = x
    kv = x["kv"].clone()
    idx = torch.empty(B, Q, p.topk, dtype=torch.int32, device=DEV)
    out = torch.empty(B, Q, 64, 512, dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(B, Q, 64, dtype=torch.float32, device=DEV)
    ws = csa.workspace(csa.CSA_OP_LAYER_PREFILL, p, B, Q, x["n_cap"])
    prev = w.pos0 > 0
    csa.csa_layer_prefill(p, B, Q, w.pos0, g["Ca"], g["Za"], g["Cb"], g["Zb"], g["Cb_prev"] if prev else None,
                          g["Zb_prev"] if prev else None, g["Ba"], g["Bb"], g["rms_w"], kv, x["n_cap"], g["kI"],
                          g["qI"], g["wI"], g["q"], g["swa"], g["sink"], idx, out, lse, ws)
    st = csa.csa_check_status()
    assert st == 0, csa.csa_status_string(st)
    return kv, idx.cpu().numpy(), out, lse.cpu().numpy()


def check_prefill(w, x, kv_gpu, idx, out, lse, b, queries):
    m, W, Q, pos0 = w.m, w.W, w.Q, w.pos0
    e0 = pos0 // m
    n_new = (pos0 + Q) // m - e0
    prev = pos0 > 0
    new = oracle.compress(e0, n_new, bits(x["Ca"][b])[: m * n_new], bits(x["Za"][b])[: m * n_new],
                          bits(x["Cb"][b])[: m * n_new], bits(x["Zb"][b])[: m * n_new],
                          bits(x["Cb_prev"][b]) if prev else None, bits(x["Zb_prev"][b]) if prev else None,
                          bits(x["Ba"]), bits(x["Bb"]), bits(x["rms_w"]), m=m)
    kv_g = kv_gpu[b].float().cpu().numpy()
    assert_close(kv_g[e0:e0 + n_new], new, "prefill entries b=%d" % b)
    kv_o = bits(x["kv"][b]).copy()
    kv_o[e0:e0 + n_new] = oracle.f64_to_bf16_bits(new)
    lin = bits(x["swa"][b])
    kI = bits(x["kI"][b])
    for j in queries:
        t = pos0 + j
        V = oracle.visible(t, m)
        scores = oracle.index_scores(bits(x["qI"][b, j]), bits(x["wI"][b, j]), kI[:V])
        n_diff = check_topk(idx[b, j], scores, w.topk, "q=%d" % j)
        # attention over the GPU's selection; the oracle's own when they agree
        sels = [idx[b, j]] + ([oracle.topk(scores, w.topk)] if n_diff == 0 else [])
        for sel in sels:
            o, l = oracle.attend_query(t, bits(x["q"][b, j]), sel, kv_o, lambda u: lin[u - (pos0 - (W - 1))],
                                       bits(x["sink"]), W=W)
            assert_close(out[b, j].float().cpu().numpy(), o, "prefill out q=%d" % j)
            np.testing.assert_allclose(lse[b, j], l, rtol=1e-3, atol=1e-3)


@pytest.mark.parametrize("B,Q,pos0,k", [(2, 64, 512, 64), (1, 70, 0, 16), (1, 45, 8, 32)])
def test_layer_prefill_small(csa, B, Q, pos0, k):
    """Every query checked; includes a chunk at position 0 (no previous block)
    and ragged chunks whose trailing partial block yields no entry."""
    w = syn.Workload("prefill-small", 50 + Q, "prefill", B=B, t=pos0 + Q - 1, topk=k, n_cap=0, Q=Q, pos0=pos0)
    x = syn.prefill_inputs(w, device=DEV)
    p = csa.csa_default_params(topk=k)
    kv, idx, out, lse = run_prefill(csa, p, w, x)
    for b in range(B):
        check_prefill(w, x, kv, idx, out, lse, b, range(Q))


def test_layer_prefill_chunk_of_4096_at_61440(csa):
    """The chunked-prefill configuration at full size; queries sampled: the
    first and last 8 and every 256th."""
    w = syn.WORKLOADS[4]
    x = syn.prefill_inputs(w, device=DEV)
    p = csa.csa_default_params(topk=w.topk)
    kv, idx, out, lse = run_prefill(csa, p, w, x)
    qs = sorted(set(list(range(8)) + list(range(w.Q - 8, w.Q)) + list(range(0, w.Q, 256))))
    check_prefill(w, x, kv, idx, out, lse, 0, qs)


def decode_keys_src(csa, x):
    return csa.index_key_src(x["ring_CIa"], x["ring_ZIa"], x["ring_CIb"], x["ring_ZIb"], x["BIa"], x["BIb"],
                             x["rms_wI"])


def oracle_ring_key(x, b, t, m):
    """The oracle's indexer key of the entry completing at t, from sequence
    b's staging ring (slot u mod 2m holds token u)."""
    i = (t + 1) // m - 1
    sa = [(m * i + r) % (2 * m) for r in range(m)]
    sb = [(m * (i - 1) + r) % (2 * m) for r in range(m)]
    return oracle.index_key_entry(i, bits(x["ring_CIa"][b])[sa], bits(x["ring_ZIa"][b])[sa],
                                  bits(x["ring_CIb"][b])[sb], bits(x["ring_ZIb"][b])[sb], bits(x["BIa"]),
                                  bits(x["BIb"]), bits(x["rms_wI"]))


@pytest.mark.parametrize("cfg,m,t", [(0, 4, 1023), (None, 8, 2399), (None, 2, 598), (None, 1, 0)])
def test_layer_decode_with_keys(csa, cfg, m, t):
    """csa_layer_decode_with_keys computes the step's indexer key from the key
    compressor's staging ring: the kI row it writes matches the oracle's key
    (E4M3 codes equal but at rounding midpoints); no other row changes (and
    none at a step that completes no block, or for a sequence at position
    -1); the rest of the step is bit for bit csa_layer_decode over the kI and
    window ring so written; and the step is the oracle's layer step over the
    written keys (emission, selection, attention)."""
    if cfg is not None:
        w = syn.WORKLOADS[cfg]
    else:
        w = syn.Workload("decode-keys-m%d" % m, 30 + m, "decode", B=3, t=t, topk=32, n_cap=300 if m > 1 else 64, m=m)
    x = syn.decode_inputs(w, device=DEV)
    if w.B > 2:
        x["q_pos"][2] = -1
    p = csa.csa_default_params(topk=w.topk, m=w.m)
    swa_new = x["swa"][:, 7].roll(1, dims=0).contiguous()
    keys = decode_keys_src(csa, x)
    kv, kI, swa = x["kv"].clone(), x["kI"].clone(), x["swa"].clone()
    B = w.B
    idx = torch.empty(B, p.topk, dtype=torch.int32, device=DEV)
    out = torch.empty(B, 64, 512, dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(B, 64, dtype=torch.float32, device=DEV)
    ws = csa.workspace(csa.CSA_OP_LAYER_DECODE, p, B, 1, w.n_cap)
    csa.csa_layer_decode_with_keys(p, B, x["q_pos"], swa_new, keys, x["ring_Ca"], x["ring_Za"], x["ring_Cb"],
                                   x["ring_Zb"], x["Ba"], x["Bb"], x["rms_w"], kv, w.n_cap, kI, x["qI"], x["wI"],
                                   x["q"], swa, x["sink"], idx, out, lse, ws)
    st = csa.csa_check_status()
    assert st == 0, csa.csa_status_string(st)
    kI_g = kI.view(torch.uint8).cpu().numpy()
    kI_0 = x["kI"].view(torch.uint8).cpu().numpy()
    qp = x["q_pos"].view(-1).cpu().numpy()
    for b in range(B):
        others = np.ones(w.n_cap, bool)
        if qp[b] >= 0 and (qp[b] + 1) % w.m == 0:
            i = (qp[b] + 1) // w.m - 1
            pre, codes = oracle_ring_key(x, b, int(qp[b]), w.m)
            check_key_codes(kI_g[b, i], pre, codes, "decode key b=%d" % b)
            others[i] = False
        assert np.array_equal(kI_g[b, others], kI_0[b, others]), "kI rows other than the step's, b=%d" % b
    # the same step through csa_layer_decode over the caches as written
    kv2 = x["kv"].clone()
    idx2, out2, lse2 = torch.empty_like(idx), torch.empty_like(out), torch.empty_like(lse)
    csa.csa_layer_decode(p, B, x["q_pos"], x["ring_Ca"], x["ring_Za"], x["ring_Cb"], x["ring_Zb"], x["Ba"], x["Bb"],
                         x["rms_w"], kv2, w.n_cap, kI, x["qI"], x["wI"], x["q"], swa, x["sink"], idx2, out2, lse2, ws)
    assert csa.csa_check_status() == 0
    assert torch.equal(idx, idx2) and torch.equal(out.view(torch.int16), out2.view(torch.int16))
    assert torch.equal(lse, lse2) and torch.equal(kv.view(torch.int16), kv2.view(torch.int16))
    # the layer step against the oracle's, over the keys and window as written
    xo = dict(x)
    xo["kI"], xo["swa"] = kI, swa
    idx_c, out_c, lse_c = idx.cpu().numpy(), out.float().cpu().numpy(), lse.cpu().numpy()
    kv_c = kv.float().cpu().numpy()
    for b in range(min(B, 2)):
        check_decode_seq(w, xo, b, bits(x["kv"][b]), kv_c[b], idx_c[b], out_c[b], lse_c[b])


def run_prefill_with_keys(csa, p, w, x):
    B, Q = w.B, w.Q
    prev = w.pos0 > 0
    keys = csa.index_key_src(x["CIa"], x["ZIa"], x["CIb"], x["ZIb"], x["BIa"], x["BIb"], x["rms_wI"],
                             x["CIb_prev"] if prev else None, x["ZIb_prev"] if prev else None)
    kv, kI = x["kv"].clone(), x["kI"].clone()
    e0 = w.pos0 // w.m
    kI[:, e0:] = 0  # the call writes the chunk's keys
    idx = torch.empty(B, Q, p.topk, dtype=torch.int32, device=DEV)
    out = torch.empty(B, Q, 64, 512, dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(B, Q, 64, dtype=torch.float32, device=DEV)
    ws = csa.workspace(csa.CSA_OP_LAYER_PREFILL, p, B, Q, x["n_cap"])
    csa.csa_layer_prefill_with_keys(p, B, Q, w.pos0, x["Ca"], x["Za"], x["Cb"], x["Zb"],
                                    x["Cb_prev"] if prev else None, x["Zb_prev"] if prev else None, x["Ba"],
                                    x["Bb"], x["rms_w"], keys, kv, x["n_cap"], kI, x["qI"], x["wI"], x["q"],
                                    x["swa"], x["sink"], idx, out, lse, ws)
    st = csa.csa_check_status()
    assert st == 0, csa.csa_status_string(st)
    return kv, kI, idx, out, lse, ws


def check_prefill_keys(csa, p, w, x, kv, kI, idx, out, lse, ws):
    """The chunk's keys against the oracle's; rows before the chunk kept; the
    step bit for bit csa_layer_prefill over the keys as written."""
    m, Q, pos0, B = w.m, w.Q, w.pos0, w.B
    e0, n_new = pos0 // m, (pos0 + Q) // m - pos0 // m
    prev = pos0 > 0
    kI_g = kI.view(torch.uint8).cpu().numpy()
    kI_0 = x["kI"].view(torch.uint8).cpu().numpy()
    near = 0
    for b in range(B):
        pre, codes = oracle.index_keys(e0, n_new, bits(x["CIa"][b])[: m * n_new], bits(x["ZIa"][b])[: m * n_new],
                                       bits(x["CIb"][b])[: m * n_new], bits(x["ZIb"][b])[: m * n_new],
                                       bits(x["CIb_prev"][b]) if prev else None,
                                       bits(x["ZIb_prev"][b]) if prev else None, bits(x["BIa"]), bits(x["BIb"]),
                                       bits(x["rms_wI"]), m=m)
        near += check_key_codes(kI_g[b, e0:e0 + n_new], pre, codes, "prefill keys b=%d" % b)
        assert np.array_equal(kI_g[b, :e0], kI_0[b, :e0]), "rows before the chunk b=%d" % b
    assert near <= 0.01 * B * n_new * 128 + 1
    kv2 = x["kv"].clone()
    idx2, out2, lse2 = torch.empty_like(idx), torch.empty_like(out), torch.empty_like(lse)
    csa.csa_layer_prefill(p, B, Q, pos0, x["Ca"], x["Za"], x["Cb"], x["Zb"], x["Cb_prev"] if prev else None,
                          x["Zb_prev"] if prev else None, x["Ba"], x["Bb"], x["rms_w"], kv2, x["n_cap"], kI, x["qI"],
                          x["wI"], x["q"], x["swa"], x["sink"], idx2, out2, lse2, ws)
    assert csa.csa_check_status() == 0
    assert torch.equal(idx, idx2) and torch.equal(out.view(torch.int16), out2.view(torch.int16))
    assert torch.equal(lse, lse2) and torch.equal(kv.view(torch.int16), kv2.view(torch.int16))


@pytest.mark.parametrize("B,Q,pos0,k", [(2, 64, 512, 64), (1, 70, 0, 16), (3, 45, 8, 32)])
def test_layer_prefill_with_keys_small(csa, B, Q, pos0, k):
    """Small chunks (the first block, and ragged chunks computed sequence by
    sequence): the chunk's keys, then every query's selection and attention
    against the oracle over the keys as written."""
    w = syn.Workload("prefill-keys", 70 + Q, "prefill", B=B, t=pos0 + Q - 1, topk=k, n_cap=0, Q=Q, pos0=pos0)
    x = syn.prefill_inputs(w, device=DEV)
    p = csa.csa_default_params(topk=k)
    kv, kI, idx, out, lse, ws = run_prefill_with_keys(csa, p, w, x)
    check_prefill_keys(csa, p, w, x, kv, kI, idx, out, lse, ws)
    xo = dict(x)
    xo["kI"] = kI
    idx_c, lse_c = idx.cpu().numpy(), lse.cpu().numpy()
    for b in range(B):
        check_prefill(w, xo, kv, idx_c, out, lse_c, b, range(Q))


def test_layer_prefill_with_keys_chunk_of_4096_at_61440(csa):
    """The chunked-prefill configuration at full size with the chunk's 1024
    indexer keys computed by the call."""
    w = syn.WORKLOADS[4]
    x = syn.prefill_inputs(w, device=DEV)
    p = csa.csa_default_params(topk=w.topk)
    kv, kI, idx, out, lse, ws = run_prefill_with_keys(csa, p, w, x)
    check_prefill_keys(csa, p, w, x, kv, kI, idx, out, lse, ws)
    xo = dict(x)
    xo["kI"] = kI
    qs = [0, 1, 2047, 4095]
    check_prefill(w, xo, kv, idx.cpu().numpy(), out, lse.cpu().numpy(), 0, qs)


def test_two_decode_steps_replayed_as_a_cuda_graph_match_eager_launches(csa):
    """Two consecutive self-contained decode steps (positions t and t+1)
    captured in one CUDA graph and replayed give, bit for bit, what the same
    two calls give launched eagerly: outputs, selections, lse and every cache
    they write.  (The benchmark replays such graphs; inside a graph the step's
    kernels keep their programmatic launch edges, across the two steps as
    well, and each kernel's reads before its dependency wait see the same
    data as in a stream.)"""
    n_cap, k = 4096, 512
    t = 4 * n_cap - 2  # step A completes no block, step B (t + 1) completes the last one
    w = syn.Workload("decode-graph", 83, "decode", B=8, t=t, topk=k, n_cap=n_cap)
    x = syn.decode_inputs(w, device=DEV)
    p = csa.csa_default_params(topk=k)
    B = w.B
    keys = decode_keys_src(csa, x)
    pos_a = x["q_pos"].clone()
    pos_b = (x["q_pos"] + 1).contiguous()
    row_a = x["swa"][:, 3].contiguous()
    row_b = x["swa"][:, 5].contiguous()
    ws = csa.workspace(csa.CSA_OP_LAYER_DECODE, p, B, 1, n_cap)

    def buffers():
        return {"kv": x["kv"].clone(), "kI": x["kI"].clone(), "swa": x["swa"].clone(),
                "idx": torch.empty(B, k, dtype=torch.int32, device=DEV),
                "out": torch.empty(B, 64, 512, dtype=torch.bfloat16, device=DEV),
                "lse": torch.empty(B, 64, dtype=torch.float32, device=DEV)}

    def two_steps(o):
        for pos, row in ((pos_a, row_a), (pos_b, row_b)):
            csa.csa_layer_decode_with_keys(p, B, pos, row, keys, x["ring_Ca"], x["ring_Za"], x["ring_Cb"],
                                           x["ring_Zb"], x["Ba"], x["Bb"], x["rms_w"], o["kv"], n_cap, o["kI"],
                                           x["qI"], x["wI"], x["q"], o["swa"], x["sink"], o["idx"], o["out"],
                                           o["lse"], ws)

    eager = buffers()
    two_steps(eager)
    torch.cuda.synchronize()
    assert csa.csa_check_status() == 0

    replayed = buffers()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        two_steps(replayed)
    graph.replay()
    torch.cuda.synchronize()
    assert csa.csa_check_status() == 0
    for name in ("idx", "out", "lse", "kv", "kI", "swa"):
        assert torch.equal(eager[name].view(torch.uint8), replayed[name].view(torch.uint8)), name
