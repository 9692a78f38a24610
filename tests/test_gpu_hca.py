"""HCA / CSA2 path parity: the single-stream compressor (csa_compress_single,
csa_compress_single_step) and dense attention over every visible compressed
entry (csa_sparse_attn with idx = NULL), against the oracle."""
import numpy as np
import pytest
import torch

import oracle
import synthetic as syn
from _util import assert_close, bits

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def csa():
    import compressed_sparse_attention_02_gb300 as m
    return m


def params(csa, m):
    return csa.csa_default_params(m=m)


@pytest.mark.parametrize("m,with_bias,B,n_new,entry0", [(128, True, 2, 3, 0), (128, True, 1, 2, 61),
                                                        (2, False, 3, 37, 5), (1, False, 2, 9, 100),
                                                        (4, True, 2, 17, 0), (16, False, 1, 5, 2)])
def test_bulk_single_stream_compressor(csa, m, with_bias, B, n_new, entry0):
    """HCA (m = 128 with its slot bias), CSA2 (m = 2, no bias), ratio 1 and
    other block sizes; entries past entry0 so the RoPE positions are m*i."""
    x = syn.single_stream_inputs(50 + m, B, m * n_new, m, with_bias)
    bias, w = x["B"], x["rms_w"]
    p = params(csa, m)
    n_cap = entry0 + n_new
    kv = torch.zeros(B, n_cap, 512, dtype=torch.bfloat16, device=DEV)
    csa.csa_compress_single(p, B, n_new, entry0, x["C"].to(DEV), x["Z"].to(DEV),
                            None if bias is None else bias.to(DEV), w.to(DEV), kv, n_cap * 512)
    assert csa.csa_check_status() == 0
    got = kv.float().cpu().numpy()
    for b in range(B):
        want = oracle.compress_single(entry0, n_new, bits(x["C"][b]), bits(x["Z"][b]),
                                      None if bias is None else bits(bias), bits(w), m=m)
        assert_close(got[b, entry0:], want, "m=%d b=%d" % (m, b))
        assert not got[b, :entry0].any(), "rows before entry0 untouched"


@pytest.mark.parametrize("m,with_bias", [(128, True), (8, False), (1, True)])
def test_decode_steps_with_online_state(csa, m, with_bias):
    """Three sequences stepped token by token from different block starts
    over two blocks and a bit: each completed block's entry equals the bulk
    definition; nothing is written between block ends."""
    B, cfg = 3, 70 + m
    starts = [0, m * 5, m * 11]
    n_steps = 2 * m + m // 2 + 1
    x = syn.single_stream_inputs(cfg, B, n_steps, m, with_bias)
    bias, w = x["B"], x["rms_w"]
    p = params(csa, m)
    n_cap = starts[-1] // m + 4
    kv = torch.full((B, n_cap, 512), 7.0, dtype=torch.bfloat16, device=DEV)
    state = torch.empty(B, 3, 512, dtype=torch.float32, device=DEV)
    C, Z = x["C"].to(DEV), x["Z"].to(DEV)
    bd = None if bias is None else bias.to(DEV)
    wd = w.to(DEV)
    for s in range(n_steps):
        pos = torch.tensor([st + s for st in starts], dtype=torch.int32, device=DEV)
        csa.csa_compress_single_step(p, B, pos, C[:, s].contiguous(), Z[:, s].contiguous(), bd, wd, state, kv,
                                     n_cap * 512, n_cap)
    assert csa.csa_check_status() == 0
    got = kv.float().cpu().numpy()
    done = n_steps // m  # complete blocks per sequence
    for b in range(B):
        i0 = starts[b] // m
        for k in range(done):
            want = oracle.compress_single_entry(i0 + k, bits(x["C"][b, k * m:(k + 1) * m]),
                                                bits(x["Z"][b, k * m:(k + 1) * m]),
                                                None if bias is None else bits(bias), bits(w))
            assert_close(got[b, i0 + k], want, "m=%d b=%d entry %d" % (m, b, i0 + k))
        untouched = [j for j in range(n_cap) if not (i0 <= j < i0 + done)]
        assert np.all(got[b, untouched] == 7.0), "no write outside completed blocks"


def dense_inputs(cfg, B, n_cap, W=128):
    return {"q": syn.main_query(cfg, B, 1), "kv": syn.cache_rows(cfg, B, n_cap),
            "swa": syn.cache_rows(cfg, B, W, name="swa"),
            "sink": syn.normal((64,), 1000 * cfg, "sink", "cpu").float()}


def run_dense(csa, p, x, pos, n_cap, split_ws=True):
    """split_ws: pass the workspace, so few queries take the split-KV path."""
    B = x["q"].shape[0]
    out = torch.empty(B, 1, 64, 512, dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(B, 1, 64, dtype=torch.float32, device=DEV)
    ws = csa.workspace(csa.CSA_OP_SPARSE_ATTN, p, B, 1, n_cap) if split_ws else None
    csa.csa_sparse_attn(p, B, 1, torch.tensor(pos, dtype=torch.int32, device=DEV).view(B, 1), x["q"].to(DEV),
                        x["kv"].to(DEV), n_cap, None, x["swa"].to(DEV), 0, p.swa_window, None, x["sink"].to(DEV),
                        out, lse, ws)
    return out.float().cpu().numpy(), lse.cpu().numpy()


def oracle_dense(p, x, b, t, m, n_cap):
    V = min((t + 1) // m, n_cap)
    ring = bits(x["swa"][b])
    return oracle.attend_query(t, bits(x["q"][b, 0]), np.arange(V, dtype=np.int32), bits(x["kv"][b]),
                               lambda u: ring[u % 128], bits(x["sink"]), W=128, sm_scale=p.sm_scale)


@pytest.mark.parametrize("split_ws", [True, False])
@pytest.mark.parametrize("m,ts", [(128, [131071, 128 * 700 + 5]), (128, [100, 127]), (2, [999, 1500]),
                                  (16, [16 * 333 - 1, 40])])
def test_dense_attention_over_every_visible_entry(csa, m, ts, split_ws):
    """HCA's read path: window rows + all floor((t+1)/m) entries + sink;
    at m = 128, V = 1024 and 700, then V = 0 (t = 100: the window alone) and
    V = 1 (t = 127); the CSA2 block size 2 and 16."""
    B = len(ts)
    n_cap = max((t + 1) // m for t in ts) + 3
    x = dense_inputs(80 + m, B, n_cap)
    p = params(csa, m)
    out, lse = run_dense(csa, p, x, ts, n_cap, split_ws)
    assert csa.csa_check_status() == 0
    for b, t in enumerate(ts):
        o, l = oracle_dense(p, x, b, t, m, n_cap)
        assert_close(out[b, 0], o, "dense m=%d t=%d split=%s" % (m, t, split_ws))
        np.testing.assert_allclose(lse[b, 0], l, rtol=1e-3, atol=1e-3)


def test_dense_attention_equals_the_sparse_call_with_every_entry_listed(csa):
    m, t = 128, 128 * 300 + 77
    V = (t + 1) // m
    x = dense_inputs(91, 1, V)
    p = params(csa, m)
    dense, _ = run_dense(csa, p, x, [t], V, split_ws=False)
    pk = csa.csa_default_params(m=m, topk=512)
    idx = torch.cat([torch.arange(V, dtype=torch.int32), torch.full((512 - V,), -1, dtype=torch.int32)]).view(1, 1, -1)
    out = torch.empty(1, 1, 64, 512, dtype=torch.bfloat16, device=DEV)
    csa.csa_sparse_attn(pk, 1, 1, torch.tensor([[t]], dtype=torch.int32, device=DEV), x["q"].to(DEV),
                        x["kv"].to(DEV), V, idx.to(DEV), x["swa"].to(DEV), 0, 128, None, x["sink"].to(DEV), out, None)
    assert csa.csa_check_status() == 0
    np.testing.assert_array_equal(dense, out.float().cpu().numpy())


def test_dense_position_past_the_cache_is_reported(csa):
    m, n_cap = 128, 50
    x = dense_inputs(92, 1, n_cap)
    p = params(csa, m)
    t = 128 * 80
    out, _ = run_dense(csa, p, x, [t], n_cap)
    assert csa.csa_check_status() == 5  # CSA_ERR_INDEX_RANGE; V clamped to the cache
    o, _ = oracle_dense(p, x, 0, t, m, n_cap)
    assert_close(out[0, 0], o, "clamped")


def test_hca_decode_at_1m_context_sampled(csa):
    """The million-token HCA decode: 8 sequences, 8192 entries each (m = 128),
    window 128; sequences 0 and 5 checked."""
    m, B, t = 128, 8, 1048575
    n_cap = (t + 1) // m
    x = {"q": syn.main_query(93, B, 1, device=DEV), "kv": syn.cache_rows(93, B, n_cap, device=DEV),
         "swa": syn.cache_rows(93, B, 128, device=DEV, name="swa"),
         "sink": syn.normal((64,), 93000, "sink", DEV).float()}
    p = params(csa, m)
    out, lse = run_dense(csa, p, x, [t] * B, n_cap)
    assert csa.csa_check_status() == 0
    for b in (0, 5):
        o, l = oracle_dense(p, x, b, t, m, n_cap)
        assert_close(out[b, 0], o, "1m b=%d" % b)


@pytest.mark.parametrize("inverse_rope", [0, 1])
def test_split_kv_path_with_inverse_rope_and_sparse_selection(csa, inverse_rope):
    """Few queries with a sparse selection (the 1M CSA shape: k = 1024 of
    262144 entries, 8 sequences) through the split-KV path, with and without
    the inverse RoPE epilogue (applied by the merge kernel)."""
    B, n_cap, k, t = 8, 262144, 1024, 1048575
    x = {"q": syn.main_query(94, B, 1), "kv": syn.cache_rows(94, B, n_cap, device=DEV),
         "swa": syn.cache_rows(94, B, 128, name="swa"), "sink": syn.normal((64,), 94000, "sink", "cpu").float()}
    g = torch.Generator().manual_seed(94)
    sel = torch.stack([torch.sort(torch.randperm(n_cap, generator=g)[:k])[0] for _ in range(B)]).to(torch.int32)
    p = csa.csa_default_params(topk=k, inverse_rope=inverse_rope)
    out = torch.empty(B, 1, 64, 512, dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(B, 1, 64, dtype=torch.float32, device=DEV)
    ws = csa.workspace(csa.CSA_OP_SPARSE_ATTN, p, B, 1, n_cap)
    csa.csa_sparse_attn(p, B, 1, torch.full((B, 1), t, dtype=torch.int32, device=DEV), x["q"].to(DEV), x["kv"],
                        n_cap, sel.view(B, 1, k).to(DEV), x["swa"].to(DEV), 0, 128, None, x["sink"].to(DEV), out, lse,
                        ws)
    assert csa.csa_check_status() == 0
    for b in (0, 7):
        ring = bits(x["swa"][b])
        o, l = oracle.attend_query(t, bits(x["q"][b, 0]), sel[b].numpy(), bits(x["kv"][b]), lambda u: ring[u % 128],
                                   bits(x["sink"]), W=128, sm_scale=p.sm_scale, inverse_rope_out=bool(inverse_rope))
        assert_close(out[b, 0].float().cpu().numpy(), o, "split-kv b=%d" % b)
        np.testing.assert_allclose(lse[b, 0].cpu().numpy(), l, rtol=1e-3, atol=1e-3)


@pytest.mark.parametrize("m,B,steps,check_every", [(8, 2, 20, 1), (128, 3, 130, 43)])
def test_hca_layer_decode_steps(csa, m, B, steps, check_every):
    """csa_hca_layer_decode stepped from a block start over a block boundary:
    each completed block's entry equals the bulk definition, and every
    step's output is the oracle's attention over the ring window and all
    entries visible at that step (the one just completed included)."""
    cfg = 120 + m
    i0 = 5                      # entries 0..4 exist before the first step
    t0 = m * i0                 # the first token of block 5
    n_cap = i0 + steps // m + 2
    x = syn.single_stream_inputs(cfg, B, steps, m, True)
    kv = syn.cache_rows(cfg, B, n_cap)
    kv[:, i0:] = 0
    ring = syn.cache_rows(cfg, B, 128, name="swa")
    sink = syn.normal((64,), 1000 * cfg, "sink", "cpu").float()
    q = syn.main_query(cfg, B, steps)
    p = params(csa, m)
    kvd, ringd, sinkd = kv.to(DEV), ring.to(DEV), sink.to(DEV)
    C, Z, bias, w = x["C"].to(DEV), x["Z"].to(DEV), x["B"].to(DEV), x["rms_w"].to(DEV)
    state = torch.empty(B, 3, 512, dtype=torch.float32, device=DEV)
    ws = csa.workspace(csa.CSA_OP_HCA_LAYER_DECODE, p, B, 1, n_cap)
    out = torch.empty(B, 1, 64, 512, dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(B, 1, 64, dtype=torch.float32, device=DEV)
    kv_host = bits(kv).copy()
    for s in range(steps):
        t = t0 + s
        pos = torch.full((B, 1), t, dtype=torch.int32, device=DEV)
        csa.csa_hca_layer_decode(p, B, pos, C[:, s].contiguous(), Z[:, s].contiguous(), bias, w, state, kvd, n_cap,
                                 q[:, s:s + 1].contiguous().to(DEV), ringd, sinkd, out, lse, ws)
        if (t + 1) % m == 0:  # the oracle's cache gains the block's entry
            e = (t + 1) // m - 1
            blk = slice(s + 1 - m, s + 1)
            for b in range(B):
                ent = oracle.compress_single_entry(e, bits(x["C"][b, blk]), bits(x["Z"][b, blk]), bits(x["B"]),
                                                   bits(x["rms_w"]))
                got = kvd[b, e].float().cpu().numpy()
                assert_close(got, ent, "entry %d b=%d" % (e, b))
                kv_host[b, e] = bits(kvd[b, e])  # the attention reads the stored bf16 entry
        if s % check_every == 0 or s == steps - 1:
            assert csa.csa_check_status() == 0
            V = (t + 1) // m
            for b in range(B):
                rb = bits(ring[b])
                o, l = oracle.attend_query(t, bits(q[b, s]), np.arange(V, dtype=np.int32), kv_host[b],
                                           lambda u: rb[u % 128], bits(sink), W=128, sm_scale=p.sm_scale)
                assert_close(out[b, 0].float().cpu().numpy(), o, "step t=%d b=%d" % (t, b))
    assert csa.csa_check_status() == 0
