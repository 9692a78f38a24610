"""Sparse attention parity (csa_sparse_attn) against the oracle."""
import math

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


def run_ring(csa, p, q, kv, idx, swa, sink, pos, lse=True):
    """Decode form: q [B,1,64,512], ring window [B,W,512]."""
    B = q.shape[0]
    out = torch.empty(B, 1, 64, 512, dtype=torch.bfloat16, device=DEV)
    l = torch.empty(B, 1, 64, dtype=torch.float32, device=DEV) if lse else None
    csa.csa_sparse_attn(p, B, 1, torch.tensor(pos, dtype=torch.int32, device=DEV).view(B, 1), q.to(DEV),
                        kv.to(DEV), kv.shape[1], idx.to(DEV), swa.to(DEV), 0, p.swa_window, None, sink.to(DEV), out,
                        l)
    return out, l


def oracle_ring(p, q, kv, idx, swa, sink, t):
    W = p.swa_window
    ring = bits(swa)
    return oracle.attend_query(t, bits(q), np.asarray(idx), bits(kv), lambda u: ring[u % W], bits(sink), W=W,
                               sm_scale=p.sm_scale, inverse_rope_out=bool(p.inverse_rope), theta=p.rope_theta)


def test_tiny_decode_config_with_oracle_selection(csa):
    w = syn.WORKLOADS[0]
    x = syn.decode_inputs(w)
    p = csa.csa_default_params(topk=w.topk)
    V = oracle.visible(w.t)
    sel = oracle.topk(oracle.index_scores(bits(x["qI"][0, 0]), bits(x["wI"][0, 0]), bits(x["kI"][0])[:V]), w.topk)
    idx = torch.from_numpy(sel).view(1, 1, -1)
    out, lse = run_ring(csa, p, x["q"], x["kv"], idx, x["swa"], x["sink"], [w.t])
    assert csa.csa_check_status() == 0
    o, l = oracle_ring(p, x["q"][0, 0], x["kv"][0], sel, x["swa"][0], x["sink"], w.t)
    assert_close(out[0, 0].float().cpu().numpy(), o, "attn c0")
    np.testing.assert_allclose(lse[0, 0].cpu().numpy(), l, rtol=1e-3, atol=1e-3)


@pytest.mark.parametrize("sink_kind", ["none", "large", "mixed"])
def test_sink_limits(csa, sink_kind):
    w = syn.WORKLOADS[0]
    x = syn.decode_inputs(w)
    p = csa.csa_default_params(topk=w.topk)
    sink = {"none": torch.full((64,), -math.inf), "large": torch.full((64,), 30.0),
            "mixed": torch.linspace(-30, 30, 64)}[sink_kind].float()
    sel = np.arange(0, 256, 4, dtype=np.int32)[: w.topk]
    out, _ = run_ring(csa, p, x["q"], x["kv"], torch.from_numpy(sel).view(1, 1, -1), x["swa"], sink, [w.t])
    assert csa.csa_check_status() == 0
    o, _ = oracle_ring(p, x["q"][0, 0], x["kv"][0], sel, x["swa"][0], sink, w.t)
    assert_close(out[0, 0].float().cpu().numpy(), o, "sink " + sink_kind)
    if sink_kind == "large":
        assert float(out.float().abs().max()) < 1e-6


def test_every_visible_entry_selected_equals_dense(csa):
    """k >= V(t): the sparse result is full attention over window + all entries."""
    n_cap, t, k = 200, 799, 256
    x = syn.decode_inputs(syn.Workload("dense", 7, "decode", B=1, t=t, topk=k, n_cap=n_cap))
    p = csa.csa_default_params(topk=k)
    sel = np.concatenate([np.arange(n_cap), -np.ones(k - n_cap)]).astype(np.int32)
    out, _ = run_ring(csa, p, x["q"], x["kv"], torch.from_numpy(sel).view(1, 1, -1), x["swa"], x["sink"], [t])
    rows = np.concatenate([bits(x["swa"][0])[[u % 128 for u in range(t - 127, t + 1)]], bits(x["kv"][0])])
    o, _ = oracle.attend(bits(x["q"][0, 0]), rows, bits(x["sink"]), p.sm_scale)
    assert_close(out[0, 0].float().cpu().numpy(), o, "dense")


def test_early_queries_and_unsorted_holes(csa):
    """Queries with fewer than W window rows, selections with -1 holes in any
    order; B = 4 sequences at different positions."""
    pos = [0, 5, 126, 400]
    B, n_cap, k = 4, 120, 64
    x = syn.decode_inputs(syn.Workload("early", 8, "decode", B=B, t=0, topk=k, n_cap=n_cap))
    rng = np.random.default_rng(8)
    sel = np.full((B, 1, k), -1, np.int32)
    for b, t in enumerate(pos):
        V = min(n_cap, (t + 1) // 4)
        n = min(V, int(rng.integers(0, k)))
        slots = rng.choice(k, size=n, replace=False)
        sel[b, 0, slots] = rng.choice(V, size=n, replace=False) if n else []
    p = csa.csa_default_params(topk=k)
    out, _ = run_ring(csa, p, x["q"], x["kv"], torch.from_numpy(sel), x["swa"], x["sink"], pos)
    assert csa.csa_check_status() == 0
    for b, t in enumerate(pos):
        o, _ = oracle_ring(p, x["q"][b, 0], x["kv"][b], sel[b, 0], x["swa"][b], x["sink"], t)
        assert_close(out[b, 0].float().cpu().numpy(), o, "t=%d" % t)


def test_out_of_range_index_is_reported_and_skipped(csa):
    n_cap, t, k = 64, 400, 16
    x = syn.decode_inputs(syn.Workload("bad", 9, "decode", B=1, t=t, topk=k, n_cap=n_cap))
    sel = np.arange(k, dtype=np.int32)
    bad = sel.copy()
    bad[3] = n_cap + 5
    p = csa.csa_default_params(topk=k)
    out, _ = run_ring(csa, p, x["q"], x["kv"], torch.from_numpy(bad).view(1, 1, -1), x["swa"], x["sink"], [t])
    assert csa.csa_check_status() == 5
    keep = np.delete(sel, 3)
    o, _ = oracle_ring(p, x["q"][0, 0], x["kv"][0], keep, x["swa"][0], x["sink"], t)
    assert_close(out[0, 0].float().cpu().numpy(), o, "skip bad index")


def test_many_tiles_and_a_late_dominant_row(csa):
    """W = 128 plus k = 2048 rows (17 tiles); one row in a late tile has a
    logit far above the rest for half of the heads, which moves the running
    reference maximum and rescales the accumulated output."""
    n_cap, k = 3000, 2048
    t = 4 * n_cap - 1
    x = syn.decode_inputs(syn.Workload("long", 10, "decode", B=1, t=t, topk=k, n_cap=n_cap))
    sel = np.sort(np.random.default_rng(10).choice(n_cap, size=k, replace=False)).astype(np.int32)
    kv = x["kv"].clone()
    q = x["q"].clone()
    target = int(sel[1900])
    q[0, 0, :32] = 0.0
    q[0, 0, :32, 7] = 16.0                   # heads 0..31 look along channel 7
    kv[0, target] = 0.0
    kv[0, target, 7] = 64.0                  # logit 1024/sqrt(512) ~ 45 for those heads
    kv[0, target, 9] = -3.0
    p = csa.csa_default_params(topk=k)
    out, lse = run_ring(csa, p, q, kv, torch.from_numpy(sel).view(1, 1, -1), x["swa"], x["sink"], [t])
    assert csa.csa_check_status() == 0
    o, l = oracle_ring(p, q[0, 0], kv[0], sel, x["swa"][0], x["sink"], t)
    assert_close(out[0, 0].float().cpu().numpy(), o, "many tiles")
    np.testing.assert_allclose(lse[0, 0].cpu().numpy(), l, rtol=1e-3, atol=1e-3)


def test_linear_window_many_queries(csa):
    """Prefill form: B = 2 sequences, Q = 6 queries each, linear window buffer
    whose row 0 is position pos0 - 127."""
    B, Q, pos0, k, n_cap = 2, 6, 300, 32, 90
    W = 128
    x = syn.prefill_inputs(syn.Workload("lin", 11, "prefill", B=B, t=pos0 + Q - 1, topk=k, n_cap=n_cap, Q=Q,
                                        pos0=pos0))
    n_cap = x["n_cap"]
    rng = np.random.default_rng(11)
    sel = np.full((B, Q, k), -1, np.int32)
    for b in range(B):
        for j in range(Q):
            V = (pos0 + j + 1) // 4
            sel[b, j] = np.sort(rng.choice(V, size=k, replace=False))
    p = csa.csa_default_params(topk=k)
    out = torch.empty(B, Q, 64, 512, dtype=torch.bfloat16, device=DEV)
    pos = torch.tensor([[pos0 + j for j in range(Q)]] * B, dtype=torch.int32, device=DEV)
    pos0s = torch.full((B,), pos0 - (W - 1), dtype=torch.int32, device=DEV)
    csa.csa_sparse_attn(p, B, Q, pos, x["q"].to(DEV), x["kv"].to(DEV), n_cap, torch.from_numpy(sel).to(DEV),
                        x["swa"].to(DEV), 1, W - 1 + Q, pos0s, x["sink"].to(DEV), out)
    assert csa.csa_check_status() == 0
    for b in range(B):
        lin = bits(x["swa"][b])
        for j in range(Q):
            o, _ = oracle.attend_query(pos0 + j, bits(x["q"][b, j]), sel[b, j], bits(x["kv"][b]),
                                       lambda u: lin[u - (pos0 - (W - 1))], bits(x["sink"]), W=W,
                                       sm_scale=p.sm_scale)
            assert_close(out[b, j].float().cpu().numpy(), o, "b=%d q=%d" % (b, j))


@pytest.mark.parametrize("B", [2, 96])
def test_inverse_rope_epilogue(csa, B):
    """The output's last 64 channels turned back by the query position: B = 2
    runs the rows of a query over a cluster (the rotation is applied by the
    CTA owning those channels), B = 96 one CTA per query; positions up to
    2^20 - 1 exercise the angle reduction."""
    n_cap, k = 300, 64
    w = syn.Workload("inv-rope", 11, "decode", B=B, t=1199, topk=k, n_cap=n_cap)
    x = syn.decode_inputs(w)
    p = csa.csa_default_params(topk=k)
    p.inverse_rope = 1
    pos = [1199 if b % 2 == 0 else (1 << 20) - 1 - 7 * b for b in range(B)]
    rng = np.random.default_rng(3)
    sel = np.stack([np.sort(rng.choice(n_cap, k, replace=False)).astype(np.int32) for _ in range(B)])
    out, lse = run_ring(csa, p, x["q"], x["kv"], torch.from_numpy(sel).view(B, 1, k), x["swa"], x["sink"], pos)
    assert csa.csa_check_status() == 0
    for b in sorted({0, 1, B - 1}):
        o, l = oracle_ring(p, x["q"][b, 0], x["kv"][b], sel[b], x["swa"][b], x["sink"], pos[b])
        assert_close(out[b, 0].float().cpu().numpy(), o, "inverse rope b=%d" % b)
        np.testing.assert_allclose(lse[b, 0].cpu().numpy(), l, rtol=1e-3, atol=1e-3)


def test_inverse_rope_flag_is_validated(csa):
    p = csa.csa_default_params()
    p.inverse_rope = 2
    out = torch.empty(1, 1, 64, 512, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(csa.CsaError):
        csa.csa_sparse_attn(p, 1, 1, torch.zeros(1, 1, dtype=torch.int32, device=DEV),
                            torch.zeros(1, 1, 64, 512, dtype=torch.bfloat16, device=DEV),
                            torch.zeros(1, 16, 512, dtype=torch.bfloat16, device=DEV), 16,
                            torch.full((1, 1, p.topk), -1, dtype=torch.int32, device=DEV),
                            torch.zeros(1, 128, 512, dtype=torch.bfloat16, device=DEV), 0, 128, None,
                            torch.zeros(64, device=DEV), out)


def test_split_kv_slices_follow_the_workspace(csa):
    """The split-KV form takes as many slices per query as the workspace
    holds: a workspace for 2 slices (where the GPU alone would take 16), one
    sized by csa_workspace_size, and one too small for any (the cluster form)
    all give the oracle's result, and the split forms agree with each other
    to fp32 summation order."""
    n_cap, k, B = 4096, 512, 4
    t = 4 * n_cap - 1
    x = syn.decode_inputs(syn.Workload("split-ws", 71, "decode", B=B, t=t, topk=k, n_cap=n_cap))
    p = csa.csa_default_params(topk=k)
    g = torch.Generator().manual_seed(71)
    idx = torch.stack([torch.sort(torch.randperm(n_cap, generator=g)[:k])[0] for _ in range(B)]).to(torch.int32)
    idx = idx.view(B, 1, k)
    slice_bytes = (64 * 512 + 2 * 64) * 4
    full = csa.workspace(csa.CSA_OP_SPARSE_ATTN, p, B, 1, n_cap)
    two = torch.empty(B * 2 * slice_bytes, dtype=torch.uint8, device=DEV)
    small = torch.empty(B * slice_bytes, dtype=torch.uint8, device=DEV)
    outs = {}
    for name, ws in (("full", full), ("two", two), ("small", small)):
        out = torch.empty(B, 1, 64, 512, dtype=torch.bfloat16, device=DEV)
        csa.csa_sparse_attn(p, B, 1, torch.full((B, 1), t, dtype=torch.int32, device=DEV), x["q"].to(DEV),
                            x["kv"].to(DEV), n_cap, idx.to(DEV), x["swa"].to(DEV), 0, 128, None, x["sink"].to(DEV),
                            out, None, ws)
        assert csa.csa_check_status() == 0
        outs[name] = out.float().cpu().numpy()
    for b in (0, B - 1):
        o, _ = oracle_ring(p, x["q"][b, 0], x["kv"][b], idx[b, 0].numpy(), x["swa"][b], x["sink"], t)
        for name in outs:
            assert_close(outs[name][b, 0], o, "%s b=%d" % (name, b))
    np.testing.assert_allclose(outs["two"], outs["full"], rtol=2e-2, atol=2e-3)
