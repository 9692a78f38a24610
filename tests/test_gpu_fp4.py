"""FP4 cache entries ("DeepSeek-V4 CSA/HCA 与 DeepSeek-V4.1 CSA2" §16.1):
the quantizer (csa_quantize_kv_fp4, bit-exact against the oracle) and the
attention reading the FP4 cache (kv_format = 1)."""
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


def quantize(csa, rows):
    """rows: [n, 512] bf16 (any device) -> [n, 288] uint8 on the device."""
    n = rows.shape[0]
    out = torch.full((n, 288), 0xAB, dtype=torch.uint8, device=DEV)
    csa.csa_quantize_kv_fp4(n, rows.to(DEV).contiguous(), 512, out, 288)
    assert csa.csa_check_status() == 0
    return out


@pytest.mark.parametrize("kind", ["normal", "scaled", "edges"])
def test_quantizer_matches_the_oracle_bit_for_bit(csa, kind):
    g = torch.Generator().manual_seed({"normal": 1, "scaled": 2, "edges": 3}[kind])
    n = 300
    x = torch.randn(n, 512, generator=g)
    if kind == "scaled":  # groups spanning many magnitudes, past the E4M3 scale range too
        x = x * torch.exp2(torch.randint(-20, 14, (n, 32), generator=g).float()).repeat_interleave(16, dim=1)
    if kind == "edges":
        x[0] = 0.0                            # all-zero entry: zero scales and codes
        x[1, :16] = -1e-3                     # tiny negatives next to larger values
        x[1, 16:32] = torch.tensor([6.0, 3.0, 2.5, 1.75, 1.25, 0.75, 0.25, -5.0] * 2)  # ties of x/s
        x[2] = 1e5                            # past 448 * 6: saturating scale and codes
        x[3, ::2] = -x[3, ::2]
    rows = x.to(torch.bfloat16)
    got = quantize(csa, rows).cpu().numpy()
    want = oracle.quantize_kv_fp4(bits(rows))
    bad = np.argwhere(got != want)
    assert bad.size == 0, "first mismatch at %s: got %#x want %#x" % (bad[0], got[tuple(bad[0])], want[tuple(bad[0])])


def dequantized_bf16(entries):
    """Exact bf16 rows of FP4 entries (value * scale is exact in bf16)."""
    vals = oracle.dequantize_kv_fp4(entries)
    b = oracle.f64_to_bf16_bits(vals)
    assert np.array_equal(oracle.bf16_to_f64(b), vals)
    return torch.from_numpy(b.view(np.int16)).view(torch.bfloat16)


def run_attn(csa, p, q, kv_any, n_cap, idx, swa, sink, pos, ws=None):
    B = q.shape[0]
    out = torch.empty(B, 1, 64, 512, dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(B, 1, 64, dtype=torch.float32, device=DEV)
    csa.csa_sparse_attn(p, B, 1, torch.tensor(pos, dtype=torch.int32, device=DEV).view(B, 1), q.to(DEV),
                        kv_any.to(DEV), n_cap, None if idx is None else idx.to(DEV), swa.to(DEV), 0, 128, None,
                        sink.to(DEV), out, lse, ws)
    assert csa.csa_check_status() == 0
    return out.float().cpu().numpy(), lse.cpu().numpy()


@pytest.mark.parametrize("B,split_ws,dense", [(64, False, False), (3, True, False), (2, True, True),
                                              (2, False, True)])
def test_attention_over_the_fp4_cache(csa, B, split_ws, dense):
    """The FP4 cache gives the bf16 result of its dequantized rows bit for bit
    (the expansion on chip is exact), and matches the oracle over those rows;
    64 queries take the cluster path, 2-3 the split-KV path, dense is HCA's."""
    n_cap, k = 2048, 512
    t = 4 * n_cap - 1
    m = 4
    x = syn.decode_inputs(syn.Workload("fp4", 95, "decode", B=B, t=t, topk=k, n_cap=n_cap), device=DEV)
    fp4 = quantize(csa, x["kv"].view(-1, 512)).view(B, n_cap, 288)
    deq = dequantized_bf16(fp4.cpu().numpy()).view(B, n_cap, 512)
    g = torch.Generator().manual_seed(95)
    idx = None if dense else torch.stack(
        [torch.sort(torch.randperm(n_cap, generator=g)[:k])[0] for _ in range(B)]).to(torch.int32).view(B, 1, k)
    p4 = csa.csa_default_params(topk=k, kv_format=1, m=m)
    p16 = csa.csa_default_params(topk=k, m=m)
    ws = csa.workspace(csa.CSA_OP_SPARSE_ATTN, p4, B, 1, n_cap) if split_ws else None
    o4, l4 = run_attn(csa, p4, x["q"], fp4, n_cap, idx, x["swa"], x["sink"], [t] * B, ws)
    o16, l16 = run_attn(csa, p16, x["q"], deq, n_cap, idx, x["swa"], x["sink"], [t] * B, ws)
    np.testing.assert_array_equal(o4, o16)
    np.testing.assert_array_equal(l4, l16)
    for b in sorted({0, B - 1}):
        ring = bits(x["swa"][b])
        sel = np.arange(oracle.visible(t, m), dtype=np.int32) if dense else idx[b, 0].numpy()
        o, l = oracle.attend_query(t, bits(x["q"][b, 0]), sel, bits(deq[b]), lambda u: ring[u % 128],
                                   bits(x["sink"]), W=128, sm_scale=p4.sm_scale)
        assert_close(o4[b, 0], o, "fp4 attention b=%d" % b)
        np.testing.assert_allclose(l4[b, 0], l, rtol=1e-3, atol=1e-3)


def test_bulk_compressor_refuses_the_fp4_cache(csa):
    p4 = csa.csa_default_params(kv_format=1)
    with pytest.raises(csa.CsaError) as e:
        csa.csa_compress(p4, 1, 1, 0, *([torch.zeros(4, 512, dtype=torch.bfloat16, device=DEV)] * 4), None, None,
                         torch.zeros(4, 512, dtype=torch.bfloat16, device=DEV),
                         torch.zeros(4, 512, dtype=torch.bfloat16, device=DEV),
                         torch.ones(512, dtype=torch.bfloat16, device=DEV),
                         torch.zeros(1, 512, dtype=torch.bfloat16, device=DEV), 512)
    assert e.value.status == 2


@pytest.mark.parametrize("B", [3, 40])
def test_layer_decode_on_the_fp4_cache(csa, B):
    """A decode step on the FP4 cache leaves exactly the FP4 entries of the
    bf16 step's cache (the emitted entry included), selects the same entries,
    and outputs exactly the bf16 attention over the dequantized cache."""
    n_cap, k = 2048, 512
    t = 4 * n_cap - 1  # the step emits entry n_cap - 1
    w = syn.Workload("fp4-layer", 96, "decode", B=B, t=t, topk=k, n_cap=n_cap)
    x = syn.decode_inputs(w, device=DEV)
    p16 = csa.csa_default_params(topk=k)
    p4 = csa.csa_default_params(topk=k, kv_format=1)
    outs = {}
    for name, p, cache in (("bf16", p16, x["kv"].clone()), ("fp4", p4, quantize(csa, x["kv"].view(-1, 512)))):
        idx = torch.empty(B, k, dtype=torch.int32, device=DEV)
        out = torch.empty(B, 64, 512, dtype=torch.bfloat16, device=DEV)
        lse = torch.empty(B, 64, dtype=torch.float32, device=DEV)
        ws = csa.workspace(csa.CSA_OP_LAYER_DECODE, p, B, 1, n_cap)
        csa.csa_layer_decode(p, B, x["q_pos"], x["ring_Ca"], x["ring_Za"], x["ring_Cb"], x["ring_Zb"], x["Ba"],
                             x["Bb"], x["rms_w"], cache, n_cap, x["kI"], x["qI"], x["wI"], x["q"], x["swa"],
                             x["sink"], idx, out, lse, ws)
        assert csa.csa_check_status() == 0
        outs[name] = (cache, idx, out, lse)
    kv16, idx16, _, _ = outs["bf16"]
    kv4, idx4, out4, lse4 = outs["fp4"]
    assert torch.equal(idx4, idx16)
    want4 = quantize(csa, kv16.view(-1, 512)).view(B, n_cap, 288)
    assert torch.equal(kv4.view(B, n_cap, 288), want4), "the FP4 cache after the step"
    deq = dequantized_bf16(kv4.view(B, n_cap, 288).cpu().numpy()).view(B, n_cap, 512)
    o16, l16 = run_attn(csa, p16, x["q"].view(B, 1, 64, 512), deq, n_cap, idx4.view(B, 1, k), x["swa"], x["sink"],
                        [t] * B, csa.workspace(csa.CSA_OP_SPARSE_ATTN, p16, B, 1, n_cap))
    np.testing.assert_array_equal(out4.view(B, 1, 64, 512).float().cpu().numpy(), o16)
    np.testing.assert_array_equal(lse4.view(B, 1, 64).cpu().numpy(), l16)


def test_layer_prefill_on_the_fp4_cache(csa):
    """A prefill chunk on the FP4 cache writes exactly the FP4 entries of the
    bf16 chunk's new entries and leaves the others as they were."""
    B, Q, pos0, k = 2, 64, 512, 64
    w = syn.Workload("fp4-prefill", 97, "prefill", B=B, t=pos0 + Q - 1, topk=k, n_cap=(pos0 + Q) // 4 + 8, Q=Q,
                     pos0=pos0)
    x = syn.prefill_inputs(w, device=DEV)
    n_cap = x["n_cap"]
    p16 = csa.csa_default_params(topk=k)
    p4 = csa.csa_default_params(topk=k, kv_format=1)
    res = {}
    for name, p, cache in (("bf16", p16, x["kv"].clone()), ("fp4", p4, quantize(csa, x["kv"].view(-1, 512)))):
        idx = torch.empty(B, Q, k, dtype=torch.int32, device=DEV)
        out = torch.empty(B, Q, 64, 512, dtype=torch.bfloat16, device=DEV)
        ws = csa.workspace(csa.CSA_OP_LAYER_PREFILL, p, B, Q, n_cap)
        csa.csa_layer_prefill(p, B, Q, pos0, x["Ca"], x["Za"], x["Cb"], x["Zb"], x["Cb_prev"], x["Zb_prev"],
                              x["Ba"], x["Bb"], x["rms_w"], cache, n_cap, x["kI"], x["qI"], x["wI"], x["q"], x["swa"],
                              x["sink"], idx, out, None, ws)
        assert csa.csa_check_status() == 0
        res[name] = (cache, idx, out)
    kv16, idx16, out16 = res["bf16"]
    kv4, idx4, out4 = res["fp4"]
    assert torch.equal(idx4, idx16)
    assert torch.equal(kv4.view(B, n_cap, 288), quantize(csa, kv16.view(-1, 512)).view(B, n_cap, 288))
    # the output is the bf16 attention over the dequantized cache, bit for bit
    deq = dequantized_bf16(kv4.view(B, n_cap, 288).cpu().numpy()).view(B, n_cap, 512).to(DEV)
    W = p16.swa_window
    q_pos = (pos0 + torch.arange(Q, dtype=torch.int32, device=DEV)).view(1, Q).repeat(B, 1).contiguous()
    swa_pos0 = torch.full((B,), pos0 - (W - 1), dtype=torch.int32, device=DEV)
    o16 = torch.empty(B, Q, 64, 512, dtype=torch.bfloat16, device=DEV)
    csa.csa_sparse_attn(p16, B, Q, q_pos, x["q"], deq, n_cap, idx4, x["swa"], 1, W - 1 + Q, swa_pos0, x["sink"], o16,
                        None, csa.workspace(csa.CSA_OP_SPARSE_ATTN, p16, B, Q, n_cap))
    assert csa.csa_check_status() == 0
    assert torch.equal(out4, o16)
