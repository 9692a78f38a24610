"""Compressor parity (csa_compress / decode emission) against the oracle."""
import numpy as np
import pytest
import torch

import oracle
import synthetic as syn
from _util import assert_close, bits, check_key_codes

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def csa():
    import compressed_sparse_attention_02_gb300 as m
    return m


def run_bulk(csa, p, x, B, n_new, entry0, prev, n_cap):
    kv = torch.zeros(B, n_cap, 512, dtype=torch.bfloat16, device=DEV)
    g = {k: v.to(DEV) for k, v in x.items()}
    csa.csa_compress(p, B, n_new, entry0, g["Ca"], g["Za"], g["Cb"], g["Zb"],
                     prev["Cb_prev"].to(DEV) if prev else None, prev["Zb_prev"].to(DEV) if prev else None,
                     g["Ba"], g["Bb"], g["rms_w"], kv, n_cap * 512)
    assert csa.csa_check_status() == 0
    return kv.float().cpu().numpy()


def oracle_bulk(x, b, n_new, entry0, prev, m=4):
    return oracle.compress(entry0, n_new, bits(x["Ca"][b]), bits(x["Za"][b]), bits(x["Cb"][b]), bits(x["Zb"][b]),
                           bits(prev["Cb_prev"][b]) if prev else None, bits(prev["Zb_prev"][b]) if prev else None,
                           bits(x["Ba"]), bits(x["Bb"]), bits(x["rms_w"]), m=m)


def test_bulk_compress_tiny_decode_config(csa):
    """1024 tokens -> 256 entries (the tiny decode case's compressor inputs)."""
    x = syn.compressor_rows(0, 1, 1024)
    x.update({k: syn.shared_params(0)[k] for k in ("Ba", "Bb", "rms_w")})
    p = csa.csa_default_params()
    got = run_bulk(csa, p, x, 1, 256, 0, None, 256)
    assert_close(got[0], oracle_bulk(x, 0, 256, 0, None), "compress c0")


def test_chunk_after_previous_block_ragged_batch(csa):
    """entry0 > 0 takes block entry0-1 from the previous-block rows."""
    B, n_new, entry0 = 3, 37, 5
    x = syn.compressor_rows(11, B, 4 * n_new)
    x.update({k: syn.shared_params(11)[k] for k in ("Ba", "Bb", "rms_w")})
    prev = syn.compressor_rows(12, B, 4, names=("Cb_prev", "Zb_prev"))
    p = csa.csa_default_params()
    got = run_bulk(csa, p, x, B, n_new, entry0, prev, entry0 + n_new + 3)
    for b in range(B):
        assert_close(got[b, entry0:entry0 + n_new], oracle_bulk(x, b, n_new, entry0, prev), "compress b=%d" % b)
        assert np.all(got[b, :entry0] == 0) and np.all(got[b, entry0 + n_new:] == 0)


@pytest.mark.parametrize("m,entry0", [(4, 0), (4, 7), (8, 7), (1, 3)])
def test_staged_form_from_2048_entries(csa, m, entry0):
    """Launches of at least 2048 entries stage each entry's rows in shared
    memory by bulk copies (fewer use the register form): every entry of two
    sequences of 1100, with and without a previous block."""
    B, n_new = 2, 1100
    x = syn.compressor_rows(21 + m, B, m * n_new)
    x.update({k: syn.shared_params(21 + m, m)[k] for k in ("Ba", "Bb", "rms_w")})
    prev = syn.compressor_rows(31 + m, B, m, names=("Cb_prev", "Zb_prev")) if entry0 else None
    p = csa.csa_default_params(m=m)
    got = run_bulk(csa, p, x, B, n_new, entry0, prev, entry0 + n_new + 2)
    for b in range(B):
        assert_close(got[b, entry0:entry0 + n_new], oracle_bulk(x, b, n_new, entry0, prev, m=m), "b=%d" % b)
        assert np.all(got[b, :entry0] == 0) and np.all(got[b, entry0 + n_new:] == 0)


@pytest.mark.parametrize("m", [1, 2, 8])
def test_other_ratios(csa, m):
    n_new = 9
    x = syn.compressor_rows(20 + m, 1, m * n_new)
    sp = syn.shared_params(20 + m, m=m)
    x.update({k: sp[k] for k in ("Ba", "Bb", "rms_w")})
    p = csa.csa_default_params(m=m)
    got = run_bulk(csa, p, x, 1, n_new, 0, None, n_new)
    assert_close(got[0], oracle_bulk(x, 0, n_new, 0, None, m=m), "compress m=%d" % m)


def test_rope_at_million_token_positions(csa):
    """Entries near 2^18 (positions near 2^20): the rotation angle must stay
    accurate (it is formed in fp64 on the device)."""
    n_new, entry0 = 8, 262136
    x = syn.compressor_rows(30, 1, 4 * n_new)
    x.update({k: syn.shared_params(30)[k] for k in ("Ba", "Bb", "rms_w")})
    prev = syn.compressor_rows(31, 1, 4, names=("Cb_prev", "Zb_prev"))
    p = csa.csa_default_params()
    got = run_bulk(csa, p, x, 1, n_new, entry0, prev, entry0 + n_new)
    assert_close(got[0, entry0:], oracle_bulk(x, 0, n_new, entry0, prev), "compress at 1M")


def test_decode_emission_from_ring(csa):
    """Sequences at different positions: an entry is emitted only when a block
    completes, from the staged rows of blocks i and i-1."""
    m, n_cap = 4, 300
    pos = [3, 7, 1023, 130, 1199]
    B = len(pos)
    ring = syn.compressor_rows(40, B, 2 * m, names=("ring_Ca", "ring_Za", "ring_Cb", "ring_Zb"))
    sp = syn.shared_params(40)
    kv0 = syn.cache_rows(40, B, n_cap)
    g = {k: v.to(DEV) for k, v in ring.items()}
    kv = kv0.to(DEV).clone()
    q_pos = torch.tensor(pos, dtype=torch.int32, device=DEV)
    # the emission is the first stage of a decode step through the C ABI
    x = syn.decode_inputs(syn.Workload("emit", 40, "decode", B=B, t=0, topk=8, n_cap=n_cap), device="cpu")
    gx = {k: (v.to(DEV) if torch.is_tensor(v) else v) for k, v in x.items()}
    p = csa.csa_default_params(topk=8)
    idx = torch.empty(B, 8, dtype=torch.int32, device=DEV)
    out = torch.empty(B, 64, 512, dtype=torch.bfloat16, device=DEV)
    ws = csa.workspace(csa.CSA_OP_LAYER_DECODE, p, B, 1, n_cap)
    csa.csa_layer_decode(p, B, q_pos, g["ring_Ca"], g["ring_Za"], g["ring_Cb"], g["ring_Zb"], sp["Ba"].to(DEV),
                         sp["Bb"].to(DEV), sp["rms_w"].to(DEV), kv, n_cap, gx["kI"], gx["qI"], gx["wI"], gx["q"],
                         gx["swa"], sp["sink"].to(DEV), idx, out, None, ws)
    status = csa.csa_check_status()
    # position 1199 emits entry 299 (inside n_cap); every position is valid
    assert status == 0, csa.csa_status_string(status)
    got = kv.float().cpu().numpy()
    ref = kv0.float().numpy()
    for b, t in enumerate(pos):
        if (t + 1) % m:
            np.testing.assert_array_equal(got[b], ref[b])
            continue
        i = (t + 1) // m - 1
        sa = [(m * i + r) % (2 * m) for r in range(m)]
        sb = [(m * (i - 1) + r) % (2 * m) for r in range(m)]
        want = oracle.compress_entry(i, bits(ring["ring_Ca"][b])[sa], bits(ring["ring_Za"][b])[sa],
                                     bits(ring["ring_Cb"][b])[sb], bits(ring["ring_Zb"][b])[sb], bits(sp["Ba"]),
                                     bits(sp["Bb"]), bits(sp["rms_w"]))
        assert_close(got[b, i], want, "emission t=%d" % t)
        others = np.ones(n_cap, bool)
        others[i] = False
        np.testing.assert_array_equal(got[b, others], ref[b, others])


@pytest.mark.parametrize("m,B,n_new,entry0", [(4, 2, 37, 0), (4, 3, 29, 1021), (8, 1, 9, 3), (1, 2, 50, 7)])
def test_indexer_key_compressor_bulk(csa, m, B, n_new, entry0):
    """Ragged entry counts (CTAs of four entries), the first block (no previous
    rows) and a chunk far into the sequence (RoPE angles near 4100 rad)."""
    x = syn.indexer_compressor_inputs(20 + m, B, m * n_new, m=m)
    p = csa.csa_default_params(m=m)
    n_cap = entry0 + n_new + 3
    kI = torch.full((B, n_cap, 128), 0x55, dtype=torch.uint8, device=DEV)
    prev = entry0 > 0
    g = {k: v.to(DEV) for k, v in x.items()}
    csa.csa_compress_indexer_keys(p, B, n_new, entry0, g["CIa"], g["ZIa"], g["CIb"], g["ZIb"],
                                  g["CIb_prev"] if prev else None, g["ZIb_prev"] if prev else None, g["BIa"],
                                  g["BIb"], g["rms_wI"], kI, n_cap * 128)
    assert csa.csa_check_status() == 0
    kI = kI.cpu().numpy()
    near = 0
    for b in range(B):
        pre, codes = oracle.index_keys(entry0, n_new, bits(x["CIa"][b]), bits(x["ZIa"][b]), bits(x["CIb"][b]),
                                       bits(x["ZIb"][b]), bits(x["CIb_prev"][b]) if prev else None,
                                       bits(x["ZIb_prev"][b]) if prev else None, bits(x["BIa"]), bits(x["BIb"]),
                                       bits(x["rms_wI"]), m=m)
        near += check_key_codes(kI[b, entry0:entry0 + n_new], pre, codes, "keys b=%d" % b)
        assert np.all(kI[b, :entry0] == 0x55) and np.all(kI[b, entry0 + n_new:] == 0x55), "rows outside the chunk"
    assert near <= 0.01 * B * n_new * 128
