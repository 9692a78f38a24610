"""Pins of the CPU oracle to facts the pages and the mathematics fix.

Each test checks the oracle against something other than itself: the storage
formats as decoded by PyTorch, hand-derived closed forms stored under
tests/golden/ (each with its citation), the pages' worked block-structure
example, textbook special cases (mean pooling, plain softmax attention via
scipy, unit RMS, rotation algebra), brute force on tiny inputs, and the top-k
error bound of "DeepSeek-V4 的 KV 压缩：从删 token 误解到预算检索" §2.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

import oracle

RNG = np.random.default_rng(12345)


def bf16_bits(x):
    t = torch.tensor(np.asarray(x, dtype=np.float64), dtype=torch.float64).to(torch.bfloat16)
    back = t.to(torch.float64).numpy()
    assert np.array_equal(back, np.asarray(x, dtype=np.float64)), "value not exact in bf16"
    return t.view(torch.int16).numpy().view(np.uint16)


def e4m3_bits(x):
    t = torch.tensor(np.asarray(x, dtype=np.float32)).to(torch.float8_e4m3fn)
    back = t.to(torch.float64).numpy()
    assert np.array_equal(back, np.asarray(x, dtype=np.float64)), "value not exact in e4m3"
    return t.view(torch.uint8).numpy()


def rand_bf16(shape, scale=1.0):
    return bf16_bits(torch.tensor(RNG.standard_normal(shape) * scale).to(torch.bfloat16).double().numpy())


def rand_e4m3(shape):
    return torch.tensor(RNG.standard_normal(shape), dtype=torch.float32).to(torch.float8_e4m3fn) \
        .view(torch.uint8).numpy()


def closed_form(expr):
    return float(eval(expr, {"__builtins__": {}},
                      {"e": math.e, "exp": math.exp, "log": math.log, "sqrt": math.sqrt, "cos": math.cos,
                       "sin": math.sin}))


def load(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


# ---- storage formats ------------------------------------------------------

def test_e4m3_decoder_matches_torch_on_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = oracle.e4m3_to_f64(codes)
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    ok = ~np.isnan(ref)
    assert np.array_equal(ref[ok], got[ok])
    assert got[0x38] == 1.0 and got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9


def test_bf16_decoder_matches_torch_on_all_codes():
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(codes.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    got = oracle.bf16_to_f64(codes)
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    ok = ~np.isnan(ref)
    assert np.array_equal(ref[ok], got[ok])


def test_bf16_store_rounding_matches_torch():
    x = RNG.standard_normal(50000) * np.exp(RNG.uniform(-30, 30, 50000))
    ref = torch.tensor(x, dtype=torch.float64).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.f64_to_bf16_bits(x), ref)


# ---- compressor -----------------------------------------------------------

def test_golden_compressor_tiny(golden_dir):
    g = load(golden_dir, "compressor_tiny_m2.json")
    m, D = g["m"], g["D"]
    tok = {k: bf16_bits(v) for k, v in g["tokens"].items()}
    Ba, Bb, w = bf16_bits(g["Ba"]), bf16_bits(g["Bb"]), bf16_bits(g["rms_w"])
    n = len(g["expected"])
    got = oracle.compress(0, n, tok["Ca"], tok["Za"], tok["Cb"], tok["Zb"], None, None, Ba, Bb, w, m=m,
                          rope_dim=g["rope_dim"], theta=g["theta"], eps=g["eps"])
    for i in range(n):
        want = [closed_form(e) for e in g["expected"]["entry%d" % i]]
        np.testing.assert_allclose(got[i], want, rtol=1e-13, atol=1e-13)


def test_golden_block_structure_of_worked_example(golden_dir):
    """Perturbing one token row changes exactly the entries the page's
    flowchart connects it to (pins the block / stream index arithmetic)."""
    g = load(golden_dir, "block_structure_m4.json")
    m, T, n = g["m"], g["n_tokens"], g["n_entries"]
    D = 8
    base = {k: rand_bf16((T, D)) for k in ("Ca", "Za", "Cb", "Zb")}
    Ba, Bb, w = rand_bf16((m, D)), rand_bf16((m, D)), bf16_bits(np.ones(D))

    def run(t):
        return oracle.compress(0, n, t["Ca"], t["Za"], t["Cb"], t["Zb"], None, None, Ba, Bb, w, m=m, rope_dim=2)

    ref = run(base)
    for feed in g["feeds"]:
        for tok in feed["tokens"]:
            for which in ("C", "Z"):
                t = {k: v.copy() for k, v in base.items()}
                name = which + feed["stream"]
                t[name][tok] = rand_bf16(D, scale=3.0)
                changed = [i for i in range(n) if not np.array_equal(run(t)[i], ref[i])]
                assert changed == feed["entries"], (name, tok, changed)


def test_pool_with_flat_logits_is_mean_pooling():
    """Constant Z and B make every per-channel softmax flat: the entry is the
    mean of its 2m rows (m rows for entry 0, whose b slots are -inf)."""
    m, D = 4, 32
    Ca, Cb = rand_bf16((m, D)), rand_bf16((m, D))
    Z = bf16_bits(np.full((m, D), 0.75))
    B0 = bf16_bits(np.zeros((m, D)))
    dec = oracle.bf16_to_f64
    x = oracle.compress_pool(Ca, Z, Cb, Z, B0, B0)
    np.testing.assert_allclose(x, np.concatenate([dec(Ca), dec(Cb)]).mean(0), rtol=1e-14, atol=1e-15)
    x0 = oracle.compress_pool(Ca, Z, None, None, B0, B0)
    np.testing.assert_allclose(x0, dec(Ca).mean(0), rtol=1e-14, atol=1e-15)


def test_pool_dominant_bias_selects_its_slot():
    """A block-slot bias 100 above every other logit puts all weight on that
    slot's row (B^a / B^b are added to Z before the softmax)."""
    m, D = 4, 16
    Ca, Za, Cb, Zb = (rand_bf16((m, D)) for _ in range(4))
    dec = oracle.bf16_to_f64
    for stream, r in (("a", 2), ("b", 1)):
        Ba, Bb = bf16_bits(np.zeros((m, D))), bf16_bits(np.zeros((m, D)))
        (Ba if stream == "a" else Bb)[r] = bf16_bits(np.full(D, 100.0))
        x = oracle.compress_pool(Ca, Za, Cb, Zb, Ba, Bb)
        want = dec(Ca)[r] if stream == "a" else dec(Cb)[r]
        np.testing.assert_allclose(x, want, rtol=1e-12, atol=1e-12)


def test_pool_weights_are_per_channel():
    """Channel d's weights depend only on channel d's logits: perturbing Z in
    one channel leaves every other channel unchanged."""
    m, D = 4, 16
    Ca, Za, Cb, Zb, Ba, Bb = (rand_bf16((m, D)) for _ in range(6))
    x = oracle.compress_pool(Ca, Za, Cb, Zb, Ba, Bb)
    Za2 = Za.copy()
    Za2[:, 5] = rand_bf16(m, scale=4.0)
    y = oracle.compress_pool(Ca, Za2, Cb, Zb, Ba, Bb)
    keep = np.arange(D) != 5
    assert np.array_equal(x[keep], y[keep]) and x[5] != y[5]


def test_rmsnorm_gives_unit_rms_and_applies_weight():
    x = RNG.standard_normal(512) * 3.7
    ones = bf16_bits(np.ones(512))
    y = oracle.rmsnorm(x, ones, 0.0)
    assert abs(np.sqrt(np.mean(y ** 2)) - 1.0) < 1e-14
    np.testing.assert_allclose(oracle.rmsnorm(5.0 * x, ones, 0.0), y, rtol=1e-14)
    w = rand_bf16(512)
    np.testing.assert_allclose(oracle.rmsnorm(x, w, 0.0), y * oracle.bf16_to_f64(w), rtol=1e-14, atol=1e-15)
    # eps enters under the square root with the mean square
    y_eps = oracle.rmsnorm(np.full(4, 1.0), bf16_bits(np.ones(4)), 3.0)
    np.testing.assert_allclose(y_eps, np.full(4, 0.5), rtol=1e-15)


def test_rope_rotation_algebra():
    D, R, theta = 512, 64, 1e4
    y = RNG.standard_normal(D)
    np.testing.assert_array_equal(oracle.rope(y, R, theta, 0.0), y)
    p1, p2 = 37.0, 1000.0
    a = oracle.rope(oracle.rope(y, R, theta, p1), R, theta, p2)
    np.testing.assert_allclose(a, oracle.rope(y, R, theta, p1 + p2), rtol=1e-9, atol=1e-9)
    z = oracle.rope(y, R, theta, 123.0)
    np.testing.assert_array_equal(z[: D - R], y[: D - R])
    pairs = lambda v: np.hypot(v[D - R::2], v[D - R + 1::2])
    np.testing.assert_allclose(pairs(z), pairs(y), rtol=1e-13)
    # (1, 0) in pair j at position 1 turns counter-clockwise by theta^(-2j/R)
    for j in (0, 1, 7, 31):
        e = np.zeros(D)
        e[D - R + 2 * j] = 1.0
        r = oracle.rope(e, R, theta, 1.0)
        ang = math.atan2(r[D - R + 2 * j + 1], r[D - R + 2 * j])
        assert abs(ang - theta ** (-2.0 * j / R)) < 1e-13


def test_compress_entry_is_rope_of_norm_of_pool_at_block_start():
    m, D, R = 4, 64, 16
    Ca, Za, Cb, Zb, Ba, Bb = (rand_bf16((m, D)) for _ in range(6))
    w = rand_bf16(D)
    i = 11
    x = oracle.compress_pool(Ca, Za, Cb, Zb, Ba, Bb)
    want = oracle.rope(oracle.rmsnorm(x, w, 1e-6), R, 1e4, m * i)
    got = oracle.compress_entry(i, Ca, Za, Cb, Zb, Ba, Bb, w, rope_dim=R, theta=1e4, eps=1e-6)
    np.testing.assert_array_equal(got, want)


# ---- visibility, indexer, top-k -------------------------------------------

def test_visibility_matches_last_covered_token_reading():
    """'DeepSeek-V4 的 KV 压缩' §9.8: with m = 4 entry j is readable at t >= 4j+3."""
    for t in range(0, 300):
        brute = sum(1 for j in range(200) if t >= 4 * j + 3)
        assert oracle.visible(t, 4) == brute
    for m in (1, 2, 8, 128):
        for t in (0, m - 2, m - 1, m, 5 * m - 1, 5 * m):
            if t >= 0:
                assert oracle.visible(t, m) == sum(1 for j in range(10) if t >= m * j + m - 1)


def test_golden_indexer_tiny(golden_dir):
    g = load(golden_dir, "indexer_tiny.json")
    q, w, k = e4m3_bits(g["qI"]), bf16_bits(g["wI"]), e4m3_bits(g["kI"])
    s = oracle.index_scores(q, w, k)
    np.testing.assert_array_equal(s, g["expected_scores"])
    for kk, want in g["expected_topk"].items():
        np.testing.assert_array_equal(oracle.topk(s, int(kk)), want)


def test_indexer_single_head_unit_query_reads_one_key_channel():
    V, Dk = 50, 128
    k = rand_e4m3((V, Dk))
    for c in (0, 17, 127):
        q = np.zeros((1, Dk), np.uint8)
        q[0, c] = 0x38  # 1.0
        s = oracle.index_scores(q, bf16_bits([1.0]), k)
        np.testing.assert_array_equal(s, np.maximum(0.0, oracle.e4m3_to_f64(k[:, c])))


def test_indexer_relu_per_head_then_weighted_sum():
    """Two heads with opposite queries: ReLU keeps exactly one of q.k and -q.k,
    so with weights (1, 1) the score is |q.k| and with (1, -1) it is q.k."""
    V, Dk = 40, 128
    k = rand_e4m3((V, Dk))
    q1 = rand_e4m3((1, Dk))
    q = np.concatenate([q1, q1 ^ 0x80])  # sign flip of every e4m3 code
    dots = oracle.e4m3_to_f64(k) @ oracle.e4m3_to_f64(q1[0])
    np.testing.assert_allclose(oracle.index_scores(q, bf16_bits([1.0, 1.0]), k), np.abs(dots), rtol=1e-15)
    np.testing.assert_allclose(oracle.index_scores(q, bf16_bits([1.0, -1.0]), k), dots, rtol=1e-15)


def test_topk_matches_exhaustive_subset_search():
    """Brute force: among all k-subsets whose every member scores >= every
    non-member, the answer is the lexicographically smallest (ties toward the
    smaller index), listed ascending."""
    for trial in range(200):
        V = int(RNG.integers(1, 9))
        k = int(RNG.integers(1, 10))
        scores = RNG.integers(-2, 3, V).astype(np.float64)  # many ties
        kk = min(k, V)
        best = None
        for sub in itertools.combinations(range(V), kk):
            inside = scores[list(sub)]
            outside = np.delete(scores, list(sub))
            if outside.size == 0 or inside.min() >= outside.max():
                if best is None or sub < best:
                    best = sub
        want = list(best) + [-1] * (k - kk)
        np.testing.assert_array_equal(oracle.topk(scores, k), want)


# ---- attention ------------------------------------------------------------

def test_golden_attention_tiny(golden_dir):
    g = load(golden_dir, "attention_tiny.json")
    sink = np.array([float(s) for s in g["sink"]], np.float32)
    out, lse = oracle.attend(bf16_bits(g["q"]), bf16_bits(g["rows"]), sink, g["sm_scale"])
    want = np.array([[closed_form(e) for e in row] for row in g["expected_out"]])
    np.testing.assert_allclose(out, want, rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(lse, [closed_form(e) for e in g["expected_lse"]], rtol=1e-14)


def test_attention_without_sink_is_plain_softmax_attention():
    H, D, n = 4, 64, 23
    q, rows = rand_bf16((H, D)), rand_bf16((n, D))
    scale = 1 / math.sqrt(D)
    out, _ = oracle.attend(q, rows, np.full(H, -np.inf, np.float32), scale)
    Q, K = oracle.bf16_to_f64(q), oracle.bf16_to_f64(rows)
    want = scipy.special.softmax(scale * Q @ K.T, axis=1) @ K
    np.testing.assert_allclose(out, want, rtol=1e-12, atol=1e-14)


def test_attention_sink_limits_and_single_row():
    H, D = 3, 32
    q, rows = rand_bf16((H, D)), rand_bf16((5, D))
    out, _ = oracle.attend(q, rows, np.full(H, 1e4, np.float32), 0.1)
    assert np.all(out == 0.0)  # all weight leaks to the sink
    one = rows[2:3]
    out1, lse1 = oracle.attend(q, one, np.full(H, -np.inf, np.float32), 0.1)
    np.testing.assert_array_equal(out1, np.broadcast_to(oracle.bf16_to_f64(one[0]), (H, D)))
    # a finite sink scales a single row by e^l / (e^l + e^s)
    s = np.array([0.0, 1.0, -2.0], np.float32)
    out2, _ = oracle.attend(q, one, s, 0.1)
    l = 0.1 * oracle.bf16_to_f64(q) @ oracle.bf16_to_f64(one[0])
    frac = 1.0 / (1.0 + np.exp(s.astype(np.float64) - l))
    np.testing.assert_allclose(out2, frac[:, None] * oracle.bf16_to_f64(one[0])[None, :], rtol=1e-13)


def test_attention_is_invariant_to_row_order():
    H, D, n = 2, 32, 9
    q, rows = rand_bf16((H, D)), rand_bf16((n, D))
    sink = np.array([0.3, -1.0], np.float32)
    a, la = oracle.attend(q, rows, sink, 0.2)
    b, lb = oracle.attend(q, rows[RNG.permutation(n)], sink, 0.2)
    np.testing.assert_allclose(a, b, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(la, lb, rtol=1e-14)


def test_attention_topk_error_bound():
    """'DeepSeek-V4 的 KV 压缩' §2: ||o - o_S|| <= 2 V R_t(S), V the largest value
    norm and R_t(S) the full-attention mass outside S (sink kept on both sides
    as a member of S with a zero value row)."""
    H, D, n = 4, 64, 60
    for trial in range(20):
        q, rows = rand_bf16((H, D), scale=2.0), rand_bf16((n, D))
        sink = RNG.standard_normal(H).astype(np.float32)
        scale = 1 / math.sqrt(D)
        full, lse = oracle.attend(q, rows, sink, scale)
        S = np.sort(RNG.choice(n, size=int(RNG.integers(1, n)), replace=False))
        sparse, _ = oracle.attend(q, rows[S], sink, scale)
        K = oracle.bf16_to_f64(rows)
        logits = scale * oracle.bf16_to_f64(q) @ K.T
        alpha = np.exp(logits - lse[:, None])
        outside = np.setdiff1d(np.arange(n), S)
        R = alpha[:, outside].sum(1)
        Vmax = np.linalg.norm(K, axis=1).max()
        err = np.linalg.norm(full - sparse, axis=1)
        assert np.all(err <= 2 * Vmax * R + 1e-12)


def test_dense_selection_equals_full_attention_over_visible_entries():
    """When k covers every visible entry the sparse path is full attention over
    the window rows plus all V(t) entries."""
    W, D, H, n_cap, m = 8, 32, 2, 12, 4
    t = 37                      # V(t) = 9
    kv = rand_bf16((n_cap, D))
    swa_ring = rand_bf16((W, D))
    q, sink = rand_bf16((H, D)), np.array([0.1, -0.4], np.float32)
    V = oracle.visible(t, m)
    idx = oracle.topk(RNG.standard_normal(V), 16)
    out, _ = oracle.attend_query(t, q, idx, kv, lambda u: swa_ring[u % W], sink, W=W, sm_scale=0.3)
    rows = np.concatenate([swa_ring[[u % W for u in range(t - W + 1, t + 1)]], kv[:V]])
    want, _ = oracle.attend(q, rows, sink, 0.3)
    np.testing.assert_allclose(out, want, rtol=1e-13, atol=1e-15)
    # the window of an early query starts at position 0
    assert list(oracle.window_positions(3, 128)) == [0, 1, 2, 3]
    assert list(oracle.window_positions(200, 128)) == list(range(73, 201))


def test_decode_emission_reads_the_staged_rows_of_blocks_i_and_i_minus_1():
    """The decode ring (slot u mod 2m) reproduces the bulk compressor's entry."""
    m, D, T = 4, 64, 24
    rows = {k: rand_bf16((T, D)) for k in ("Ca", "Za", "Cb", "Zb")}
    Ba, Bb, w = rand_bf16((m, D)), rand_bf16((m, D)), rand_bf16(D)
    bulk = oracle.compress(0, T // m, rows["Ca"], rows["Za"], rows["Cb"], rows["Zb"], None, None, Ba, Bb, w,
                           m=m, rope_dim=16)
    for t in (3, 7, 23):
        ring = {k: np.zeros((2 * m, D), np.uint16) for k in rows}
        for u in range(max(0, t - 2 * m + 1), t + 1):
            for k in rows:
                ring[k][u % (2 * m)] = rows[k][u]
        n_cap, H = T // m, 2
        kv = np.zeros((n_cap, D), np.uint16)
        kI = rand_e4m3((n_cap, 128))
        kv_after, _, _, _ = oracle.layer_decode_one(
            t, ring["Ca"], ring["Za"], ring["Cb"], ring["Zb"], Ba, Bb, w, kv, kI, rand_e4m3((H, 128)),
            rand_bf16(H), rand_bf16((H, D)), rand_bf16((8, D)), np.zeros(H, np.float32), m=m, topk_k=4, W=8,
            rope_dim=16)
        i = (t + 1) // m - 1
        np.testing.assert_array_equal(kv_after[i], oracle.f64_to_bf16_bits(bulk[i]))


# ---- inverse partial RoPE ([CSA2 详解] §12.1) -----------------------------------

@pytest.mark.parametrize("t", [0, 1, 777, 131071, 1 << 20])
def test_inverse_rope_undoes_rope_at_the_same_position(t):
    rng = np.random.default_rng(5 + t % 97)
    x = rng.standard_normal((3, 512))
    rotated = np.stack([oracle.rope(r, 64, 1e4, t) for r in x])
    back = oracle.inverse_rope(rotated, t)
    np.testing.assert_allclose(back, x, rtol=0, atol=1e-9)


def test_inverse_rope_keeps_the_plain_channels_and_the_pair_norms():
    rng = np.random.default_rng(6)
    x = rng.standard_normal((2, 512))
    y = oracle.inverse_rope(x, 4321)
    np.testing.assert_array_equal(y[:, :448], x[:, :448])
    n0 = x[:, 448:].reshape(2, 32, 2)
    n1 = y[:, 448:].reshape(2, 32, 2)
    np.testing.assert_allclose(np.hypot(n1[..., 0], n1[..., 1]), np.hypot(n0[..., 0], n0[..., 1]), atol=1e-12)
    assert not np.allclose(y[:, 448:], x[:, 448:])


def test_inverse_rope_recovers_the_output_of_unrotated_rows():
    """The page's reason for the step: rows all rotated to the query's
    position t and summed with any weights give, after the inverse rotation,
    the same weighted sum of the unrotated rows."""
    rng = np.random.default_rng(7)
    t = 90001
    rows = rng.standard_normal((40, 512))
    wts = rng.random((64, 40))
    wts /= wts.sum(1, keepdims=True)
    rotated = np.stack([oracle.rope(r, 64, 1e4, t) for r in rows])
    np.testing.assert_allclose(oracle.inverse_rope(wts @ rotated, t), wts @ rows, rtol=0, atol=1e-9)


# ---- indexer keys ([hca_csa] "CSA：轻压缩 + 稀疏选择") --------------------------

def test_hadamard_matches_the_kronecker_construction_and_is_an_involution():
    import synthetic as syn
    rng = np.random.default_rng(8)
    x = rng.standard_normal(128)
    H = syn.hadamard(128).double().numpy() / np.sqrt(128.0)  # H_2k = [[H_k, H_k], [H_k, -H_k]] built by blocks
    np.testing.assert_allclose(oracle.hadamard(x), H @ x, atol=1e-12)
    np.testing.assert_allclose(oracle.hadamard(oracle.hadamard(x)), x, atol=1e-12)
    assert np.linalg.norm(oracle.hadamard(x)) == pytest.approx(np.linalg.norm(x), rel=1e-12)


def test_e4m3_encoding_round_trips_and_agrees_with_torch_in_range():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    vals = oracle.e4m3_to_f64(codes)
    back = oracle.to_e4m3(vals)
    assert np.array_equal(back[codes != 0x80], codes[codes != 0x80])  # -0 and +0 decode alike
    rng = np.random.default_rng(9)
    x = np.concatenate([rng.standard_normal(4000) * s for s in (1e-3, 0.05, 1.0, 30.0, 140.0)])
    x = x[np.abs(x) <= 448].astype(np.float32)
    want = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.to_e4m3(x.astype(np.float64)), want)


def test_e4m3_ties_go_to_the_even_code_and_large_values_saturate():
    pos = np.arange(1, 0x7E, dtype=np.uint8)  # neighbouring finite positive codes c, c+1
    lo, hi = oracle.e4m3_to_f64(pos), oracle.e4m3_to_f64(pos + 1)
    got = oracle.to_e4m3((lo + hi) / 2)
    want = np.where(pos % 2 == 0, pos, pos + 1)
    assert np.array_equal(got, want)
    assert list(oracle.to_e4m3(np.array([1e4, -1e4, 449.0]))) == [0x7E, 0xFE, 0x7E]
    assert oracle.to_e4m3(np.array([np.nan]))[0] == 0x7F


def test_index_key_entry_is_the_compressor_entry_at_width_128_rotated_then_rounded():
    m, D = 4, 128
    Ca, Za, Cb, Zb, Ba, Bb = (rand_bf16((m, D)) for _ in range(6))
    w = bf16_bits(torch.tensor(1 + 0.1 * RNG.standard_normal(D)).to(torch.bfloat16).double().numpy())
    for i in (0, 5, 70000):
        pre, codes = oracle.index_key_entry(i, Ca, Za, Cb, Zb, Ba, Bb, w)
        ent = oracle.compress_entry(i, Ca, Za, Cb, Zb, Ba, Bb, w)
        np.testing.assert_allclose(pre, oracle.hadamard(ent), atol=1e-12)
        assert np.array_equal(codes, oracle.to_e4m3(pre))


# ---- hierarchical indexer ([CSA2 详解] §11) ------------------------------------

def test_block_scores_worked_example():
    """21 entries in blocks of 8: blocks {0..7}, {8..15}, {16..20}.  Rising
    scores put each block's maximum on its last visible entry, falling scores
    on its first one (values written out by hand)."""
    rising = np.arange(21, dtype=np.float64)
    np.testing.assert_array_equal(oracle.block_scores(rising), [7.0, 15.0, 20.0])
    np.testing.assert_array_equal(oracle.block_scores(rising[::-1].copy()), [20.0, 12.0, 4.0])
    np.testing.assert_array_equal(oracle.block_scores(np.array([3.0])), [3.0])
    assert oracle.block_scores(np.zeros(0)).size == 0


def test_candidate_pool_separates_chosen_from_unchosen_entries():
    """Every entry of an unchosen block scores at most the smallest chosen
    block's best entry; pools are ascending, unique and -1 padded; when every
    visible block fits, the pool is all of them."""
    for trial in range(100):
        V = int(RNG.integers(1, 200))
        nb = int(RNG.integers(1, 30))
        s = RNG.integers(-5, 6, V).astype(np.float64)  # many ties
        pool = oracle.candidate_pool(s, nb)
        n_vis = (V + 7) // 8
        n = min(nb, n_vis)
        assert pool.shape == (nb,)
        assert np.all(pool[n:] == -1)
        chosen = pool[:n]
        assert np.all(np.diff(chosen) > 0) and chosen.min() >= 0 and chosen.max() < n_vis
        if n == n_vis:
            np.testing.assert_array_equal(chosen, np.arange(n_vis))
            continue
        best_in = [s[8 * b:min(V, 8 * b + 8)].max() for b in chosen]
        out_entries = [s[e] for e in range(V) if e // 8 not in set(chosen.tolist())]
        assert min(best_in) >= max(out_entries)
        # ties between a chosen and an unchosen block: the chosen one is smaller
        floor = min(best_in)
        tied_out = [b for b in range(n_vis) if b not in set(chosen.tolist()) and s[8 * b:min(V, 8 * b + 8)].max() == floor]
        tied_in = [b for b in chosen if s[8 * b:min(V, 8 * b + 8)].max() == floor]
        if tied_out:
            assert max(tied_in) < min(tied_out)


def test_pool_entries_drop_the_invisible_tail_of_the_last_block():
    # V = 59: block 7 holds entries 56..58 only
    np.testing.assert_array_equal(oracle.pool_entries([2, 7, -1], 59), list(range(16, 24)) + [56, 57, 58])
    assert oracle.pool_entries([-1, -1], 59).size == 0


def test_reindex_with_the_full_layers_query_reproduces_the_full_topk():
    """A position of the full top-k has a block score at least its own score,
    and at most k blocks can score above it, so with n_blocks >= k the pool
    holds the whole full top-k: a Reindex layer using the Full layer's own
    q^I / w^I must then return exactly the full top-k."""
    V, k, nb = 2000, 64, 64
    q, w, kI = rand_e4m3((64, 128)), rand_bf16(64, 1 / 90.0), rand_e4m3((V, 128))
    full = oracle.index_scores(q, w, kI)
    top = np.sort(full)[::-1][:k + 1]
    assert np.all(np.diff(top) < 0), "the seed must give distinct leading scores"
    pool = oracle.candidate_pool(full, nb)
    assert (pool >= 0).sum() == nb and oracle.pool_entries(pool, V).size == 8 * nb < V
    idx, ent, sc = oracle.reindex_topk(q, w, kI, pool, V, k)
    np.testing.assert_array_equal(idx, oracle.topk(full, k))


def test_reindex_equals_masking_the_full_scores_outside_the_pool():
    """Scoring the gathered pool equals scoring every entry and masking the
    entries outside the pool to -inf before the top-k (the two forms of
    [CSA2 详解] §20.1), with a second layer's own query."""
    V, k, nb = 777, 40, 12
    q1, w1 = rand_e4m3((64, 128)), rand_bf16(64, 1 / 90.0)
    q2, w2 = rand_e4m3((64, 128)), rand_bf16(64, 1 / 90.0)
    kI = rand_e4m3((V, 128))
    pool = oracle.candidate_pool(oracle.index_scores(q1, w1, kI), nb)
    idx, ent, sc = oracle.reindex_topk(q2, w2, kI, pool, V, k)
    masked = np.full(V, -np.inf)
    keep = oracle.pool_entries(pool, V)
    masked[keep] = oracle.index_scores(q2, w2, kI)[keep]
    np.testing.assert_array_equal(idx, oracle.topk(masked, k)[:k])
    np.testing.assert_array_equal(sc, masked[ent])


def test_reindex_returns_the_whole_pool_when_k_covers_it():
    V = 59
    kI = rand_e4m3((V, 128))
    q, w = rand_e4m3((64, 128)), rand_bf16(64, 1 / 90.0)
    idx, ent, sc = oracle.reindex_topk(q, w, kI, [0, 7, -1, -1], V, 16)
    np.testing.assert_array_equal(idx, list(range(8)) + [56, 57, 58] + [-1] * 5)


# ---- non-overlapped compressor (HCA, CSA2) ----------------------------------

def test_single_stream_entry_zero_is_the_overlapped_entry_zero():
    """[hca_csa]: HCA is the CSA compressor with one stream and no block i-1;
    the overlapped entry 0 has no block i-1 either, so the two agree exactly."""
    m, D = 4, 512
    C, Z, B = rand_bf16((m, D)), rand_bf16((m, D)), rand_bf16((m, D))
    w = bf16_bits(torch.tensor(1 + 0.1 * RNG.standard_normal(D)).to(torch.bfloat16).double().numpy())
    junk = rand_bf16((m, D))
    want = oracle.compress_entry(0, C, Z, junk, junk, B, junk, w)
    np.testing.assert_array_equal(oracle.compress_single_entry(0, C, Z, B, w), want)


def test_single_stream_flat_logits_and_no_bias_are_mean_pooling():
    m, D = 128, 512
    C = rand_bf16((m, D))
    Z = np.full((m, D), bf16_bits([0.75])[0], np.uint16)
    w = bf16_bits(np.ones(D))
    mean = oracle.bf16_to_f64(C).mean(axis=0)
    want = oracle.rope(oracle.rmsnorm(mean, w, 1e-6), 64, 1e4, 128 * 3)
    np.testing.assert_allclose(oracle.compress_single_entry(3, C, Z, None, w), want, rtol=1e-12, atol=1e-12)


def test_single_stream_ratio_one_is_norm_of_the_row():
    """[CSA2 详解] §7.5: with one token per group the softmax weight is 1, so
    the entry is RoPE(Norm(C)) of that token's row."""
    D = 512
    C, Z, B = rand_bf16((1, D)), rand_bf16((1, D)), rand_bf16((1, D))
    w = bf16_bits(torch.tensor(1 + 0.1 * RNG.standard_normal(D)).to(torch.bfloat16).double().numpy())
    want = oracle.rope(oracle.rmsnorm(oracle.bf16_to_f64(C[0]), w, 1e-6), 64, 1e4, 37)
    np.testing.assert_array_equal(oracle.compress_single_entry(37, C, Z, B, w), want)
    np.testing.assert_array_equal(oracle.compress_single_entry(37, C, Z, None, w), want)


def test_single_stream_dominant_logit_selects_its_row_per_channel():
    """A logit 60 above the others takes the whole softmax weight of its
    channel: channel d picks row d % m."""
    m, D = 128, 512
    C = rand_bf16((m, D))
    Z = np.zeros((m, D), np.uint16)
    hot = bf16_bits([60.0])[0]
    for d in range(D):
        Z[d % m, d] = hot
    w = bf16_bits(np.ones(D))
    Cf = oracle.bf16_to_f64(C)
    picked = np.array([Cf[d % m, d] for d in range(D)])
    want = oracle.rope(oracle.rmsnorm(picked, w, 1e-6), 64, 1e4, 0)
    np.testing.assert_allclose(oracle.compress_single_entry(0, C, Z, None, w), want, rtol=1e-12, atol=1e-12)


def test_single_stream_rope_position_is_m_times_i():
    """The same rows as entry i or entry 0 differ only by RoPE at m*i."""
    m, D, i = 128, 512, 77
    C, Z, B = rand_bf16((m, D)), rand_bf16((m, D)), rand_bf16((m, D))
    w = bf16_bits(np.ones(D))
    e0 = oracle.compress_single_entry(0, C, Z, B, w)
    ei = oracle.compress_single_entry(i, C, Z, B, w)
    np.testing.assert_allclose(oracle.rope(e0, 64, 1e4, m * i), ei, rtol=1e-9, atol=1e-12)
    np.testing.assert_array_equal(ei[:448], e0[:448])


# ---- FP4 cache entries ([CSA2 详解] §16.1) ------------------------------------

def test_e2m1_values_of_all_codes():
    """The E2M1 grid (sign, 2 exponent bits with bias 1, 1 mantissa bit)."""
    mags = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    np.testing.assert_array_equal(oracle.e2m1_to_f64(np.arange(8)), mags)
    np.testing.assert_array_equal(oracle.e2m1_to_f64(np.arange(8, 16)), [-m for m in mags])
    assert math.copysign(1.0, oracle.e2m1_to_f64(np.array([8]))[0]) == -1.0


def test_e2m1_rounding_is_nearest_with_ties_to_even_and_saturates():
    codes = np.arange(16, dtype=np.uint8)
    np.testing.assert_array_equal(oracle.to_e2m1(oracle.e2m1_to_f64(codes))[1:], codes[1:])  # round trip (+0 / -0 apart)
    ties = {0.25: 0.0, 0.75: 1.0, 1.25: 1.0, 1.75: 2.0, 2.5: 2.0, 3.5: 4.0, 5.0: 4.0}
    for x, want in ties.items():
        assert oracle.e2m1_to_f64(oracle.to_e2m1(np.array([x])))[0] == want, x
        assert oracle.e2m1_to_f64(oracle.to_e2m1(np.array([-x])))[0] == -want, -x
    np.testing.assert_array_equal(oracle.e2m1_to_f64(oracle.to_e2m1(np.array([6.5, 100.0, -7.0]))), [6.0, 6.0, -6.0])
    grid = oracle.e2m1_to_f64(np.arange(16))
    x = RNG.uniform(-7, 7, 2000)
    got = oracle.e2m1_to_f64(oracle.to_e2m1(x))
    err = np.abs(got - x)
    assert np.all(err <= np.min(np.abs(grid[None, :] - x[:, None]), axis=1) + 1e-15)  # nearest by brute force


def test_fp4_entry_layout_worked_example():
    """Group 0 holds 6, -0.5, 3, 0 ... (scale E4M3(6/6) = 1.0, code 0x38): byte 0
    = (code(-0.5) << 4) | code(6) = 0x97, byte 1 = 0x05 (3, then +0); other
    groups are zero (scale code 0, zero codes)."""
    x = np.zeros(512)
    x[:4] = [6.0, -0.5, 3.0, 0.0]
    e = oracle.quantize_kv_fp4(bf16_bits(x))
    assert e.shape == (288,)
    assert e[0] == 0x97 and e[1] == 0x05 and not e[2:256].any()
    assert e[256] == 0x38 and not e[257:].any()
    np.testing.assert_array_equal(oracle.dequantize_kv_fp4(e), x)


def test_fp4_entries_on_the_grid_round_trip_and_others_round_to_the_nearest_code():
    # rows that are exactly s * e2m1 with amax = 6 s round-trip
    s = oracle.e4m3_to_f64(np.array([0x30, 0x38, 0x41, 0x2A], np.uint8))  # 0.5, 1, 2.25, 0.3125
    vals = oracle.e2m1_to_f64(RNG.integers(0, 16, 512).astype(np.uint8))
    vals[::16] = 6.0
    x = vals * np.repeat(np.resize(s, 32), 16)
    np.testing.assert_array_equal(oracle.dequantize_kv_fp4(oracle.quantize_kv_fp4(bf16_bits(x))), x)
    # general rows: the scale is E4M3(amax/6), each code the nearest grid point of x/s
    x = oracle.bf16_to_f64(rand_bf16(512, 2.0))
    e = oracle.quantize_kv_fp4(bf16_bits(x))
    deq = oracle.dequantize_kv_fp4(e)
    grid = oracle.e2m1_to_f64(np.arange(16))
    for g in range(32):
        sc = oracle.e4m3_to_f64(e[256 + g:257 + g])[0]
        amax = np.abs(x[16 * g:16 * g + 16]).max()
        assert abs(sc - amax / 6) <= 0.0625 * amax / 6 + 1e-12  # E4M3: 3 mantissa bits
        q = x[16 * g:16 * g + 16] / sc
        best = np.min(np.abs(grid[None, :] - q[:, None]), axis=1)
        assert np.all(np.abs(deq[16 * g:16 * g + 16] / sc - q) <= best + 1e-9)


def test_fp4_entry_binary32_quotients_choose_the_fp64_codes_on_every_input():
    """The FP4 entry's two quotients (amax/6 for the scale, x/s for a code) are
    formed in binary32, the kernel's precision; the pages fix no rounding.
    This reading is harmless: for every bf16 amax and every (bf16 x, E4M3
    scale s) pair the binary32 and fp64 quotients have no E2M1 / E4M3 rounding
    midpoint between them (an exact midpoint is representable in binary32 and
    is then the same in both), so both readings give the same codes; and the
    oracle's entries equal the ones built from fp64 quotients."""
    u = np.arange(1, 0x7F80, dtype=np.uint32)                      # every positive finite bf16
    x = (u << 16).view(np.float32).astype(np.float64)
    e4 = oracle.e4m3_to_f64(np.arange(0, 127, dtype=np.uint8))     # 0 .. 448, ascending
    mid4 = (e4[:-1] + e4[1:]) / 2
    mid2 = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])        # between E2M1 magnitudes

    def crossing(q64, q32, mids):
        lo, hi = np.minimum(q64, q32), np.maximum(q64, q32)
        k = np.searchsorted(mids, lo, side="left")                  # first midpoint >= lo
        return (q64 != q32) & (k < len(mids)) & (mids[np.minimum(k, len(mids) - 1)] <= hi)

    # the scale quotient, every bf16 amax
    q64 = x / 6.0
    q32 = (x.astype(np.float32) / np.float32(6.0)).astype(np.float64)
    assert not crossing(q64, q32, mid4).any()
    # the code quotient, every bf16 x against every non-zero E4M3 scale
    for s in e4[1:]:
        q64 = x / s
        q32 = (x.astype(np.float32) / np.float32(s)).astype(np.float64)
        assert not crossing(q64, q32, mid2).any(), s
    # the oracle's entries equal those of the fp64 reading (random rows and
    # groups whose amax sits at E4M3 midpoints times 6)
    rows = oracle.bf16_to_f64(rand_bf16((24, 512), 2.0))
    rows[:, ::16] = np.resize(oracle.bf16_to_f64(bf16_bits(mid4[40:100] * 6.0)), (24, 32))
    for r in rows:
        e = oracle.quantize_kv_fp4(bf16_bits(r))
        rb = oracle.bf16_to_f64(bf16_bits(r))
        for g in range(32):
            grp = rb[16 * g:16 * g + 16]
            sc = oracle.to_e4m3(np.array([np.abs(grp).max() / 6.0]))[0]
            assert e[256 + g] == sc
            sv = oracle.e4m3_to_f64(np.array([sc], np.uint8))[0]
            codes = oracle.to_e2m1(grp / sv) if sv != 0 else np.zeros(16, np.uint8)
            want = (codes[0::2] | (codes[1::2] << 4)).astype(np.uint8)
            np.testing.assert_array_equal(e[8 * g:8 * g + 8], want)


# ---- FP4 indexer keys and queries ------------------------------------------

def test_e8m0_scale_bytes_worked_by_hand():
    """Smallest 2^e with 6 * 2^e >= amax, byte e + 127: 6 = 6 * 2^0 -> 127;
    the next bf16 above 6 needs 2^1 -> 128; 1 lies in (6 * 2^-3, 6 * 2^-2] ->
    125; 0.75 = 6 * 2^-3 -> 124; 3 = 6 * 2^-1 -> 126; 1e38 in
    (6 * 2^123, 6 * 2^124] -> 251; the largest bf16 (about 3.39e38) in
    (6 * 2^125, 6 * 2^126] -> 253; zero and anything at or below
    6 * 2^-127 -> 0 (the format's smallest scale)."""
    cases = {6.0: 127, 6.0234375: 128, 1.0: 125, 0.75: 124, 3.0: 126, 1e38: 251, 3.3895313892515355e38: 253,
             0.0: 0, 2.0 ** -133: 0, 6.0 * 2.0 ** -127: 0, 2.0 ** -124: 1}
    for amax, want in cases.items():
        assert oracle.e8m0_scale(amax) == want, amax
    np.testing.assert_array_equal(oracle.e8m0_to_f64(np.array([0, 126, 127, 128, 254], np.uint8)),
                                  [2.0 ** -127, 0.5, 1.0, 2.0, 2.0 ** 127])


def test_fp4_index_row_layout_worked_example():
    """Block 0 = [2.5, 5, 0.25, 0.75, -2.5, 1.25, 1.75, 3.5, 6, 0 ...] has amax 6,
    scale byte 127 (s = 1); the codes by hand (ties to the even code):
    2.5 -> 2 (0x4), 5 -> 4 (0x6), 0.25 -> 0 (0x0), 0.75 -> 1 (0x2),
    -2.5 -> -2 (0xC), 1.25 -> 1 (0x2), 1.75 -> 2 (0x4), 3.5 -> 4 (0x6), 6 (0x7);
    byte j = code(2j) | code(2j+1) << 4.  Block 1 = 12 at channel 32: scale
    2 (byte 128), code 6 (0x7).  Blocks 2, 3 are zero: byte 0, zero codes."""
    x = np.zeros(128)
    x[:9] = [2.5, 5.0, 0.25, 0.75, -2.5, 1.25, 1.75, 3.5, 6.0]
    x[32] = 12.0
    codes, scales = oracle.quantize_index_fp4(bf16_bits(x))
    assert codes.shape == (64,) and scales.shape == (4,)
    assert list(codes[:5]) == [0x64, 0x20, 0x2C, 0x64, 0x07]
    assert not codes[5:16].any() and codes[16] == 0x07 and not codes[17:].any()
    assert list(scales) == [127, 128, 0, 0]
    np.testing.assert_array_equal(oracle.dequantize_index_fp4(codes, scales)[:9],
                                  [2.0, 4.0, 0.0, 1.0, -2.0, 1.0, 2.0, 4.0, 6.0])


def test_fp4_index_rows_on_the_grid_round_trip_and_others_round_to_the_nearest_code():
    # a block of e2m1 values times 2^k with amax 6 * 2^k or 4 * 2^k has scale 2^k and round-trips
    for top in (6.0, 4.0):
        k = RNG.integers(-20, 20, 4)
        vals = oracle.e2m1_to_f64(RNG.integers(0, 16, 128).astype(np.uint8))
        vals = np.clip(vals, -top, top)
        vals[::32] = top
        x = vals * np.repeat(2.0 ** k, 32)
        codes, scales = oracle.quantize_index_fp4(bf16_bits(x))
        np.testing.assert_array_equal(scales, k + 127)
        np.testing.assert_array_equal(oracle.dequantize_index_fp4(codes, scales), x)
    # general rows: |x| / s within E2M1's range, each value the nearest grid point of x / s
    grid = oracle.e2m1_to_f64(np.arange(16))
    for scale in (1e-3, 1.0, 300.0):
        x = oracle.bf16_to_f64(rand_bf16(128, scale))
        codes, scales = oracle.quantize_index_fp4(bf16_bits(x))
        deq = oracle.dequantize_index_fp4(codes, scales)
        for g in range(4):
            s = 2.0 ** (int(scales[g]) - 127)
            blk = x[32 * g:32 * g + 32]
            assert 3 * s < np.abs(blk).max() <= 6 * s  # the smallest power of two that fits
            q = blk / s
            best = np.min(np.abs(grid[None, :] - q[:, None]), axis=1)
            assert np.all(np.abs(deq[32 * g:32 * g + 32] / s - q) <= best + 1e-12)


def test_fp4_index_scores_equal_the_e4m3_scores_of_the_same_values():
    """Values e2m1 * 2^k with k in -6..4 are exact in E4M3 too: the FP4 scorer
    (E8M0 scales per 32 channels, nibble codes) and the E4M3 scorer must give
    the same scores, block scales differing across a row."""
    H, V = 8, 40
    def rows(n):
        codes = RNG.integers(0, 256, (n, 64)).astype(np.uint8)
        scales = RNG.integers(121, 132, (n, 4)).astype(np.uint8)
        return codes, scales
    qc, qs = rows(H)
    kc, ks = rows(V)
    w = rand_bf16(H)
    fp4 = oracle.index_scores_fp4(qc, qs, w, kc, ks)
    q8 = e4m3_bits(oracle.dequantize_index_fp4(qc, qs))
    k8 = e4m3_bits(oracle.dequantize_index_fp4(kc, ks))
    np.testing.assert_array_equal(fp4, oracle.index_scores(q8, w, k8))
    assert np.count_nonzero(fp4) > V // 2
