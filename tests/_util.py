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
