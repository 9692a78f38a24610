"""Shared helpers of the parity tests (comparison rules, device moves)."""
import numpy as np
import torch

# Floating-point tolerance for compressor and attention outputs: an element
# passes when |gpu - oracle| <= ATOL + RTOL * |oracle| (bf16 inputs, fp32
# accumulation, bf16 output).
ATOL, RTOL = 2e-2, 1e-2
# Near-tie band of the top-k comparison, relative to the k-th oracle score.
TIE_REL = 1e-3


def to_dev(x: dict, dev) -> dict:
    return {k: (v.to(dev) if torch.is_tensor(v) else v) for k, v in x.items()}


def assert_close(got, want, what="output", atol=ATOL, rtol=RTOL):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape, (got.shape, want.shape)
    err = np.abs(got - want)
    bad = err > atol + rtol * np.abs(want)
    if bad.any():
        i = np.unravel_index(np.argmax(err - (atol + rtol * np.abs(want))), err.shape)
        raise AssertionError("%s: %d/%d elements out of tolerance; worst at %s: got %r want %r"
                             % (what, bad.sum(), bad.size, i, got[i], want[i]))


def check_topk(got_idx, scores, k, what="top-k"):
    """The GPU selection must be a valid top-k of the exact oracle scores:
    ascending, unique, min(k, V) entries then -1; equal to the oracle's set
    unless the oracle's k-th and (k+1)-th scores lie within TIE_REL of each
    other, and then every differing entry lies within TIE_REL of the k-th."""
    import oracle
    got_idx = np.asarray(got_idx)
    V = len(scores)
    n = min(k, V)
    assert got_idx.shape == (k,)
    valid = got_idx[:n]
    assert np.all(got_idx[n:] == -1), "%s: padding is not -1" % what
    assert np.all((valid >= 0) & (valid < V)), "%s: index out of range" % what
    assert np.all(np.diff(valid) > 0), "%s: not strictly ascending" % what
    want = oracle.topk(scores, k)[:n]
    if np.array_equal(valid, want):
        return 0
    order = np.sort(scores)[::-1]
    ok_ = order[n - 1]
    band = TIE_REL * abs(ok_)
    assert n < V and abs(order[n - 1] - order[n]) <= band, \
        "%s: sets differ outside a near tie (k-th %r, k+1-th %r)" % (what, order[n - 1], order[n] if n < V else None)
    diff = np.setxor1d(valid, want)
    assert np.all(np.abs(scores[diff] - ok_) <= band), "%s: differing entries not near the k-th score" % what
    return len(diff)


def bits(t):
    import synthetic
    return synthetic.bits(t)


# ---- FP4 indexer layouts (include/csa.h, csa_quantize_index_keys_fp4) -------
# Pure byte placement: codes planes first, then the E8M0 scales in 512-byte
# atoms (entry e of a key sequence at 16*(e%32) + 4*((e%128)/32) + block of
# atom e/128; head h of a query record at 16*(h%32) + 4*(h/32) + block).

def pack_index_keys_fp4(codes, scales, n_cap):
    """codes [B][n][64] u8, scales [B][n][4] u8 (n <= n_cap) -> FP4 key cache
    bytes; entries n.. are zero."""
    codes, scales = np.asarray(codes, np.uint8), np.asarray(scales, np.uint8)
    B, n = codes.shape[:2]
    A = (n_cap + 127) // 128
    buf = np.zeros(B * (n_cap * 64 + A * 512), np.uint8)
    buf[:B * n_cap * 64].reshape(B, n_cap, 64)[:, :n] = codes
    sp = buf[B * n_cap * 64:].reshape(B, A, 32, 4, 4)
    e = np.arange(n)
    for b in range(B):
        sp[b, e // 128, e % 32, (e % 128) // 32, :] = scales[b]
    return buf


def unpack_index_keys_fp4(buf, B, n_cap):
    """FP4 key cache bytes -> (codes [B][n_cap][64], scales [B][n_cap][4])."""
    buf = np.asarray(buf, np.uint8).reshape(-1)
    A = (n_cap + 127) // 128
    codes = buf[:B * n_cap * 64].reshape(B, n_cap, 64)
    sp = buf[B * n_cap * 64:B * (n_cap * 64 + A * 512)].reshape(B, A, 32, 4, 4)
    e = np.arange(n_cap)
    return codes, np.stack([sp[b, e // 128, e % 32, (e % 128) // 32, :] for b in range(B)])


def pack_index_query_fp4(codes, scales):
    """codes [n_q][64][64] u8, scales [n_q][64][4] u8 -> FP4 query records."""
    codes, scales = np.asarray(codes, np.uint8), np.asarray(scales, np.uint8)
    nq = codes.shape[0]
    buf = np.zeros(nq * 4608, np.uint8)
    buf[:nq * 4096] = codes.reshape(-1)
    sp = buf[nq * 4096:].reshape(nq, 32, 16)
    sp[:, :, 0:4] = scales[:, :32]
    sp[:, :, 4:8] = scales[:, 32:]
    return buf


def unpack_index_query_fp4(buf, nq):
    """FP4 query records -> (codes [n_q][64][64], scales [n_q][64][4], the
    unused bytes 8..15 of every line [n_q][32][8])."""
    buf = np.asarray(buf, np.uint8).reshape(-1)
    codes = buf[:nq * 4096].reshape(nq, 64, 64)
    sp = buf[nq * 4096:nq * 4608].reshape(nq, 32, 16)
    return codes, np.concatenate([sp[:, :, 0:4], sp[:, :, 4:8]], axis=1), sp[:, :, 8:]


def check_key_codes(got, pre, codes, what):
    """Equal E4M3 codes, except where the oracle's value sits within a relative
    1e-4 of the midpoint between two neighbouring codes: there the kernel's
    fp32 rounding may land on either side (both codes are then accepted)."""
    import oracle
    got = np.asarray(got, dtype=np.uint8).ravel()
    codes = np.asarray(codes, dtype=np.uint8).ravel()
    pre = np.asarray(pre, dtype=np.float64).ravel()
    diff = np.nonzero(got != codes)[0]
    for j in diff:
        a, b = oracle.e4m3_to_f64(np.array([got[j], codes[j]], dtype=np.uint8))
        mid = (a + b) / 2
        assert abs(int(got[j] & 0x7F) - int(codes[j] & 0x7F)) <= 1 and (got[j] & 0x80) == (codes[j] & 0x80), \
            "%s: element %d code %#x vs %#x" % (what, j, got[j], codes[j])
        assert abs(pre[j] - mid) <= 1e-4 * abs(mid) + 1e-9, "%s: element %d not at a rounding midpoint" % (what, j)
    return len(diff)
