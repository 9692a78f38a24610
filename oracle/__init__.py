"""CSA oracle — TEST INFRASTRUCTURE ONLY.

Plain fp64 CPU statement of one CSA layer's hot path (compressor, visibility,
lightning indexer, top-k, joint softmax with sink), used to check the CUDA
library.  Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU
baseline / reference arm may import this package.  It shares no code with the
CUDA path: the arithmetic lives in ``csa_oracle.c`` (double precision,
single-threaded); this module only marshals numpy arrays and composes the
per-query steps in the order the pages give them ("DeepSeek-V4 的 KV 压缩：
从删 token 误解到预算检索" §9.9: window indices, indexer top-k, compressed
cache write at block boundaries, gather + attention).

Every array argument holds raw storage bits: bf16 as ``np.uint16``, FP8 E4M3
as ``np.uint8``; the attention sink is ``np.float32``.

Parity pins for every function live in ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "csa_oracle.c")
_LIB = os.path.join(_HERE, "liboracle_csa.so")
_lib = None

_u8p = ctypes.POINTER(ctypes.c_uint8)
_u16p = ctypes.POINTER(ctypes.c_uint16)
_i32p = ctypes.POINTER(ctypes.c_int32)
_f32p = ctypes.POINTER(ctypes.c_float)
_f64p = ctypes.POINTER(ctypes.c_double)


def build(force: bool = False) -> str:
    """Compile csa_oracle.c into liboracle_csa.so next to it (gcc, no FMA
    contraction so that the rounding order is the one written)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(
            ["gcc", "-O2", "-ffp-contract=off", "-std=c11", "-fPIC", "-shared",
             _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        lib.orc_bf16.restype = ctypes.c_double
        lib.orc_bf16.argtypes = [ctypes.c_uint16]
        lib.orc_e4m3.restype = ctypes.c_double
        lib.orc_e4m3.argtypes = [ctypes.c_uint8]
        lib.orc_compress_pool.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int] + [_u16p] * 6 + [_f64p]
        lib.orc_rmsnorm.argtypes = [ctypes.c_int, _f64p, _u16p, ctypes.c_double, _f64p]
        lib.orc_rope.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_double, _f64p]
        lib.orc_compress_entry.argtypes = ([ctypes.c_int] * 3 + [ctypes.c_double] * 2 + [ctypes.c_int64]
                                           + [_u16p] * 7 + [_f64p])
        lib.orc_compress_single_entry.argtypes = ([ctypes.c_int] * 3 + [ctypes.c_double] * 2 + [ctypes.c_int64]
                                                  + [_u16p] * 4 + [_f64p])
        lib.orc_hadamard.argtypes = [ctypes.c_int, _f64p, _f64p]
        lib.orc_to_e4m3.restype = ctypes.c_uint8
        lib.orc_to_e4m3.argtypes = [ctypes.c_double]
        lib.orc_index_key_entry.argtypes = ([ctypes.c_int] * 3 + [ctypes.c_double] * 2 + [ctypes.c_int64]
                                            + [_u16p] * 7 + [_f64p, _u8p])
        lib.orc_e2m1.restype = ctypes.c_double
        lib.orc_e2m1.argtypes = [ctypes.c_uint8]
        lib.orc_to_e2m1.restype = ctypes.c_uint8
        lib.orc_to_e2m1.argtypes = [ctypes.c_double]
        lib.orc_quantize_kv_fp4.argtypes = [ctypes.c_int, _u16p, _u8p]
        lib.orc_dequantize_kv_fp4.argtypes = [ctypes.c_int, _u8p, _f64p]
        lib.orc_e8m0_scale.restype = ctypes.c_uint8
        lib.orc_e8m0_scale.argtypes = [ctypes.c_double]
        lib.orc_e8m0.restype = ctypes.c_double
        lib.orc_e8m0.argtypes = [ctypes.c_uint8]
        lib.orc_quantize_index_fp4.argtypes = [ctypes.c_int, _u16p, _u8p, _u8p]
        lib.orc_dequantize_index_fp4.argtypes = [ctypes.c_int, _u8p, _u8p, _f64p]
        lib.orc_quantize_index_fp4_rows.argtypes = [ctypes.c_int64, ctypes.c_int, _u16p, _u8p, _u8p]
        lib.orc_dequantize_index_fp4_rows.argtypes = [ctypes.c_int64, ctypes.c_int, _u8p, _u8p, _f64p]
        lib.orc_index_scores_f64.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int64, _f64p, _u16p, _f64p,
                                             _f64p]
        lib.orc_visible.restype = ctypes.c_int64
        lib.orc_visible.argtypes = [ctypes.c_int64, ctypes.c_int]
        lib.orc_index_scores.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int64, _u8p, _u16p, _u8p, _f64p]
        lib.orc_topk.restype = ctypes.c_int
        lib.orc_topk.argtypes = [ctypes.c_int64, ctypes.c_int, _f64p, _i32p]
        lib.orc_attend.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, _u16p, _u16p, _f32p,
                                   ctypes.c_double, _f64p, _f64p]
        lib.orc_decode_bf16.argtypes = [ctypes.c_int64, _u16p, _f64p]
        lib.orc_decode_e4m3.argtypes = [ctypes.c_int64, _u8p, _f64p]
        _lib = lib
    return _lib


def _ptr(a: np.ndarray | None, ctype):
    if a is None:
        return ctypes.cast(None, ctype)
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctype)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ---- storage formats ------------------------------------------------------

def bf16_to_f64(bits) -> np.ndarray:
    bits = _c(bits, np.uint16)
    out = np.empty(bits.shape, np.float64)
    _load().orc_decode_bf16(bits.size, _ptr(bits, _u16p), _ptr(out, _f64p))
    return out


def e4m3_to_f64(bits) -> np.ndarray:
    bits = _c(bits, np.uint8)
    out = np.empty(bits.shape, np.float64)
    _load().orc_decode_e4m3(bits.size, _ptr(bits, _u8p), _ptr(out, _f64p))
    return out


# ---- compressor -----------------------------------------------------------

def compress_pool(Ca, Za, Cb, Zb, Ba, Bb) -> np.ndarray:
    """Per-channel softmax pooling of one entry before Norm/RoPE.  Ca/Za are
    the m rows of block i; Cb/Zb the m rows of block i-1 or None for i = 0."""
    Ca, Za, Ba, Bb = (_c(a, np.uint16) for a in (Ca, Za, Ba, Bb))
    m, D = Ca.shape
    has_prev = Cb is not None
    Cb = _c(Cb, np.uint16) if has_prev else None
    Zb = _c(Zb, np.uint16) if has_prev else None
    x = np.empty(D, np.float64)
    _load().orc_compress_pool(m, D, int(has_prev), _ptr(Ca, _u16p), _ptr(Za, _u16p), _ptr(Cb, _u16p),
                              _ptr(Zb, _u16p), _ptr(Ba, _u16p), _ptr(Bb, _u16p), _ptr(x, _f64p))
    return x


def rmsnorm(x, w, eps) -> np.ndarray:
    x = _c(x, np.float64)
    w = _c(w, np.uint16)
    y = np.empty_like(x)
    _load().orc_rmsnorm(x.size, _ptr(x, _f64p), _ptr(w, _u16p), eps, _ptr(y, _f64p))
    return y


def rope(y, rope_dim, theta, pos) -> np.ndarray:
    y = np.array(y, dtype=np.float64, copy=True)
    _load().orc_rope(y.size, rope_dim, theta, float(pos), _ptr(y, _f64p))
    return y


def compress_entry(i, Ca, Za, Cb, Zb, Ba, Bb, w, *, rope_dim=64, theta=1e4, eps=1e-6) -> np.ndarray:
    """Entry i = RoPE(Norm(pool)); Cb/Zb are block i-1's rows (ignored for i = 0)."""
    Ca, Za, Ba, Bb, w = (_c(a, np.uint16) for a in (Ca, Za, Ba, Bb, w))
    m, D = Ca.shape
    if i > 0:
        Cb, Zb = _c(Cb, np.uint16), _c(Zb, np.uint16)
    else:
        Cb = Zb = None
    out = np.empty(D, np.float64)
    _load().orc_compress_entry(m, D, rope_dim, theta, eps, int(i), _ptr(Ca, _u16p), _ptr(Za, _u16p),
                               _ptr(Cb, _u16p), _ptr(Zb, _u16p), _ptr(Ba, _u16p), _ptr(Bb, _u16p),
                               _ptr(w, _u16p), _ptr(out, _f64p))
    return out


def compress_single_entry(i, C, Z, B, w, *, rope_dim=64, theta=1e4, eps=1e-6) -> np.ndarray:
    """Non-overlapped compressor ([hca_csa] "HCA：同一个算子，关掉重叠"; [CSA2
    详解] §7.2, §7.5): entry i from the m rows C/Z of its own block, B the
    [m, D] position bias or None (CSA2 has none); RoPE(Norm(pool)) at m*i."""
    C, Z, w = (_c(a, np.uint16) for a in (C, Z, w))
    B = None if B is None else _c(B, np.uint16)
    m, D = C.shape
    out = np.empty(D, np.float64)
    _load().orc_compress_single_entry(m, D, rope_dim, theta, eps, int(i), _ptr(C, _u16p), _ptr(Z, _u16p),
                                      _ptr(B, _u16p), _ptr(w, _u16p), _ptr(out, _f64p))
    return out


def compress_single(entry0, n_new, C, Z, B, w, *, m, rope_dim=64, theta=1e4, eps=1e-6) -> np.ndarray:
    """Bulk non-overlapped form for one sequence: C/Z hold the chunk's m*n_new
    token rows (row j is token m*entry0 + j); returns entries entry0.. as
    [n_new, D] doubles."""
    C, Z = _c(C, np.uint16), _c(Z, np.uint16)
    D = C.shape[1]
    out = np.empty((n_new, D), np.float64)
    for e in range(n_new):
        rows = slice(m * e, m * (e + 1))
        out[e] = compress_single_entry(entry0 + e, C[rows], Z[rows], B, w, rope_dim=rope_dim, theta=theta, eps=eps)
    return out


def compress(entry0, n_new, Ca, Za, Cb, Zb, Cb_prev, Zb_prev, Ba, Bb, w, *, m=4, rope_dim=64,
             theta=1e4, eps=1e-6) -> np.ndarray:
    """Bulk form for one sequence: Ca/Za/Cb/Zb hold the chunk's m*n_new token
    rows (row j = token m*entry0 + j); Cb_prev/Zb_prev the m rows before the
    chunk (None iff entry0 == 0).  Returns [n_new, D]."""
    D = Ca.shape[-1]
    out = np.empty((n_new, D), np.float64)
    for e in range(n_new):
        i = entry0 + e
        blk = slice(m * e, m * e + m)
        if i == 0:
            cb = zb = None
        elif e == 0:
            cb, zb = Cb_prev, Zb_prev
        else:
            prev = slice(m * (e - 1), m * e)
            cb, zb = Cb[prev], Zb[prev]
        out[e] = compress_entry(i, Ca[blk], Za[blk], cb, zb, Ba, Bb, w, rope_dim=rope_dim, theta=theta,
                                eps=eps)
    return out


# ---- visibility, indexer, top-k -------------------------------------------

def visible(t: int, m: int = 4) -> int:
    return int(_load().orc_visible(int(t), int(m)))


def index_scores(qI, wI, kI) -> np.ndarray:
    """qI [H, Dk] e4m3, wI [H] bf16, kI [V, Dk] e4m3 -> scores [V] (fp64)."""
    qI, kI = _c(qI, np.uint8), _c(kI, np.uint8)
    wI = _c(wI, np.uint16)
    H, Dk = qI.shape
    V = kI.shape[0]
    out = np.empty(V, np.float64)
    _load().orc_index_scores(H, Dk, V, _ptr(qI, _u8p), _ptr(wI, _u16p), _ptr(kI, _u8p), _ptr(out, _f64p))
    return out


def topk(scores, k: int) -> np.ndarray:
    scores = _c(scores, np.float64)
    idx = np.empty(k, np.int32)
    _load().orc_topk(scores.size, k, _ptr(scores, _f64p), _ptr(idx, _i32p))
    return idx


# ---- hierarchical indexer ---------------------------------------------------
# [CSA2 详解] §11 "Hierarchical Sparse Indexer": the Full layer scores every
# visible entry; entries are grouped in blocks of 8 consecutive ones, a
# block's score is the largest score among its entries, and at most 2048
# blocks with the largest block scores form the candidate pool (at most 16384
# entries).  A Reindex layer scores only the pool's entries with its own q^I
# and head weights and takes its own top-k among them (§11.1; §20.1: the
# candidates are gathered first, so the cost is fixed by the pool size).

POOL_BLOCK = 8


def block_scores(scores, block: int = POOL_BLOCK) -> np.ndarray:
    """Scores of the ceil(V/block) blocks of V visible entries: block j holds
    entries j*block .. j*block+block-1 below V, its score is their largest."""
    s = np.asarray(scores, dtype=np.float64)
    V = s.size
    nb = (V + block - 1) // block
    out = np.empty(nb, np.float64)
    for j in range(nb):
        out[j] = s[j * block:min(V, (j + 1) * block)].max()
    return out


def candidate_pool(scores, n_blocks: int = 2048, block: int = POOL_BLOCK) -> np.ndarray:
    """The Full layer's pool: the min(n_blocks, ceil(V/block)) blocks with the
    largest block scores (equal scores: the smaller block first), in
    ascending block order, then -1 up to n_blocks slots."""
    return topk(block_scores(scores, block), n_blocks)


def pool_entries(pool, V: int, block: int = POOL_BLOCK) -> np.ndarray:
    """Entries of the pool's blocks (-1 slots skipped) that are visible
    (below V), in ascending order."""
    out = [b * block + r for b in np.asarray(pool) if b >= 0 for r in range(block) if b * block + r < V]
    return np.asarray(out, dtype=np.int64)


def reindex_topk(qI, wI, kI, pool, V: int, k: int, block: int = POOL_BLOCK):
    """A Reindex layer over the pool: its own scores I_s for the pool's
    entries s only, then the min(k, |pool|) largest (equal scores: the
    smaller entry first), returned as entry indices in ascending order and
    -1 up to k slots.  Returns (idx [k], the pool's entries, their scores)."""
    ent = pool_entries(pool, V, block)
    kI = np.asarray(kI)
    sc = index_scores(qI, wI, kI[ent]) if ent.size else np.empty(0, np.float64)
    slots = topk(sc, k)
    idx = np.full(k, -1, np.int32)
    n = int((slots >= 0).sum())
    idx[:n] = ent[slots[:n]]
    return idx, ent, sc


# ---- attention ------------------------------------------------------------

def attend(q, rows, sink, sm_scale):
    """q [H, D] bf16, rows [n, D] bf16, sink [H] fp32 -> (out [H, D], lse [H])."""
    q, rows = _c(q, np.uint16), _c(rows, np.uint16)
    sink = _c(sink, np.float32)
    H, D = q.shape
    out = np.empty((H, D), np.float64)
    lse = np.empty(H, np.float64)
    _load().orc_attend(H, D, rows.shape[0], _ptr(q, _u16p), _ptr(rows, _u16p), _ptr(sink, _f32p),
                       float(sm_scale), _ptr(out, _f64p), _ptr(lse, _f64p))
    return out, lse


def hadamard(x) -> np.ndarray:
    """H_n x / sqrt(n), Sylvester H_n (n = len(x), a power of two)."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    y = np.empty_like(x)
    _load().orc_hadamard(x.size, _ptr(x, _f64p), _ptr(y, _f64p))
    return y


def to_e4m3(x) -> np.ndarray:
    """Nearest E4M3 codes (ties to even, saturating at +-448) of doubles."""
    x = np.asarray(x, dtype=np.float64)
    lib = _load()
    return np.array([lib.orc_to_e4m3(float(v)) for v in x.ravel()], dtype=np.uint8).reshape(x.shape)


def e2m1_to_f64(codes) -> np.ndarray:
    """Values of E2M1 codes (the low 4 bits of each element)."""
    codes = np.asarray(codes, dtype=np.uint8)
    lib = _load()
    return np.array([lib.orc_e2m1(int(c) & 0xF) for c in codes.ravel()], np.float64).reshape(codes.shape)


def to_e2m1(x) -> np.ndarray:
    """Nearest E2M1 codes (ties to even, saturating at +-6, sign kept) of doubles."""
    x = np.asarray(x, dtype=np.float64)
    lib = _load()
    return np.array([lib.orc_to_e2m1(float(v)) for v in x.ravel()], np.uint8).reshape(x.shape)


def quantize_kv_fp4(rows) -> np.ndarray:
    """bf16 rows [n, D] -> FP4 entries [n, D/2 + D/16] bytes ([CSA2 详解] §16.1)."""
    rows = _c(rows, np.uint16)
    rows2 = rows.reshape(-1, rows.shape[-1])
    D = rows2.shape[1]
    out = np.empty((rows2.shape[0], D // 2 + D // 16), np.uint8)
    for i in range(rows2.shape[0]):
        r = np.ascontiguousarray(rows2[i])
        o = np.empty(D // 2 + D // 16, np.uint8)
        _load().orc_quantize_kv_fp4(D, _ptr(r, _u16p), _ptr(o, _u8p))
        out[i] = o
    return out.reshape(rows.shape[:-1] + (D // 2 + D // 16,))


def dequantize_kv_fp4(entries, D: int = 512) -> np.ndarray:
    """FP4 entries [n, D/2 + D/16] bytes -> their values [n, D] (doubles)."""
    entries = _c(entries, np.uint8)
    e2 = entries.reshape(-1, entries.shape[-1])
    out = np.empty((e2.shape[0], D), np.float64)
    for i in range(e2.shape[0]):
        r = np.ascontiguousarray(e2[i])
        o = np.empty(D, np.float64)
        _load().orc_dequantize_kv_fp4(D, _ptr(r, _u8p), _ptr(o, _f64p))
        out[i] = o
    return out.reshape(entries.shape[:-1] + (D,))


# ---- FP4 indexer keys and queries ([CSA2 详解] §16.2) -----------------------
# 128 E2M1 values and one E8M0 scale per 32 of them.  Scale rounding (the
# pages leave it open): the smallest power of two s with 6 * s >= the block's
# largest magnitude; see orc_e8m0_scale.

def e8m0_scale(amax: float) -> int:
    """E8M0 byte of a block whose largest magnitude is ``amax``."""
    return int(_load().orc_e8m0_scale(float(amax)))


def e8m0_to_f64(b) -> np.ndarray:
    b = np.asarray(b, dtype=np.uint8)
    lib = _load()
    return np.array([lib.orc_e8m0(int(v)) for v in b.ravel()], np.float64).reshape(b.shape)


def quantize_index_fp4(rows):
    """bf16 rows [..., D] -> (codes [..., D/2] u8, scales [..., D/32] u8): per
    row, channel 2j in the low nibble of code byte j, scale g for channels
    32g .. 32g+31."""
    rows = _c(rows, np.uint16)
    r2 = np.ascontiguousarray(rows.reshape(-1, rows.shape[-1]))
    D = r2.shape[1]
    codes = np.empty((r2.shape[0], D // 2), np.uint8)
    scales = np.empty((r2.shape[0], D // 32), np.uint8)
    _load().orc_quantize_index_fp4_rows(r2.shape[0], D, _ptr(r2, _u16p), _ptr(codes, _u8p), _ptr(scales, _u8p))
    lead = rows.shape[:-1]
    return codes.reshape(lead + (D // 2,)), scales.reshape(lead + (D // 32,))


def dequantize_index_fp4(codes, scales) -> np.ndarray:
    """(codes [..., D/2], scales [..., D/32]) -> values [..., D] (doubles)."""
    codes, scales = _c(codes, np.uint8), _c(scales, np.uint8)
    D = codes.shape[-1] * 2
    c2 = np.ascontiguousarray(codes.reshape(-1, D // 2))
    s2 = np.ascontiguousarray(scales.reshape(-1, D // 32))
    out = np.empty((c2.shape[0], D), np.float64)
    if c2.shape[0]:
        _load().orc_dequantize_index_fp4_rows(c2.shape[0], D, _ptr(c2, _u8p), _ptr(s2, _u8p), _ptr(out, _f64p))
    return out.reshape(codes.shape[:-1] + (D,))


def index_scores_fp4(q_codes, q_scales, wI, k_codes, k_scales) -> np.ndarray:
    """The indexer score over FP4 queries and keys: q [H, Dk/2] + [H, Dk/32],
    wI [H] bf16, k [V, Dk/2] + [V, Dk/32] -> scores [V] (fp64); the products
    of the decoded values, as index_scores forms them for E4M3."""
    q = np.ascontiguousarray(dequantize_index_fp4(q_codes, q_scales))
    k = np.ascontiguousarray(dequantize_index_fp4(k_codes, k_scales)) if len(k_codes) else np.empty((0, q.shape[1]))
    wI = _c(wI, np.uint16)
    H, Dk = q.shape
    V = k.shape[0]
    out = np.empty(V, np.float64)
    if V:
        _load().orc_index_scores_f64(H, Dk, V, _ptr(q, _f64p), _ptr(wI, _u16p), _ptr(k, _f64p), _ptr(out, _f64p))
    return out


def index_key_entry(i, Ca, Za, Cb, Zb, Ba, Bb, w, *, rope_dim=64, theta=1e4, eps=1e-6):
    """Indexer key entry i ([hca_csa] "CSA：轻压缩 + 稀疏选择"): the compressor's
    steps at width 128, then H_128/sqrt(128), then E4M3.  Returns (values
    before rounding [128] f64, codes [128] u8)."""
    Ca, Za, Ba, Bb, w = (_c(a, np.uint16) for a in (Ca, Za, Ba, Bb, w))
    m, D = Ca.shape
    if i > 0:
        Cb, Zb = _c(Cb, np.uint16), _c(Zb, np.uint16)
    else:
        Cb = Zb = None
    pre = np.empty(D, np.float64)
    codes = np.empty(D, np.uint8)
    _load().orc_index_key_entry(m, D, rope_dim, theta, eps, int(i), _ptr(Ca, _u16p), _ptr(Za, _u16p),
                                _ptr(Cb, _u16p), _ptr(Zb, _u16p), _ptr(Ba, _u16p), _ptr(Bb, _u16p), _ptr(w, _u16p),
                                _ptr(pre, _f64p), _ptr(codes, _u8p))
    return pre, codes


def index_keys(entry0, n_new, Ca, Za, Cb, Zb, Cb_prev, Zb_prev, Ba, Bb, w, *, m=4, rope_dim=64, theta=1e4,
               eps=1e-6):
    """Indexer keys of entries entry0 .. entry0+n_new-1 from a chunk's rows
    (layout as compress()): (values before rounding [n_new,128], codes)."""
    pre = np.empty((n_new, Ca.shape[-1]), np.float64)
    codes = np.empty((n_new, Ca.shape[-1]), np.uint8)
    for e in range(n_new):
        i = entry0 + e
        a_rows = slice(m * e, m * e + m)
        if e > 0:
            b_rows = slice(m * (e - 1), m * e)
            cb, zb = Cb[b_rows], Zb[b_rows]
        else:
            cb, zb = Cb_prev, Zb_prev
        pre[e], codes[e] = index_key_entry(i, Ca[a_rows], Za[a_rows], cb, zb, Ba, Bb, w, rope_dim=rope_dim,
                                           theta=theta, eps=eps)
    return pre, codes


def inverse_rope(o, t, *, rope_dim=64, theta=1e4) -> np.ndarray:
    """Inverse partial RoPE of attention outputs ([CSA2 详解] §12.1 "Partial
    RoPE 与 inverse RoPE"; [KV 压缩] §9.6, the note after the kernel path): the
    rows carry RoPE on their last rope_dim channels, so a weighted sum of them
    carries the rotations too; each head's output is turned back by the angle
    of the query position t, i.e. RoPE at position -t with the same pairs and
    frequencies.  o [H, D] -> [H, D] float64."""
    o = np.array(o, dtype=np.float64, copy=True)
    for h in range(o.shape[0]):
        o[h] = rope(o[h], rope_dim, theta, -float(t))
    return o


def window_positions(t: int, W: int) -> np.ndarray:
    """Raw window of the query at t: positions max(0, t-W+1) .. t.  The pages
    do not say whether the window holds the current token; it is read as
    included (W positions ending at t)."""
    return np.arange(max(0, t - W + 1), t + 1, dtype=np.int64)


def gather_rows(t, idx, kv_comp, swa_row_of, W):
    """Row set of the query at t: its window rows, then kv_comp[idx] for idx != -1."""
    pos = window_positions(t, W)
    swa_rows = np.stack([swa_row_of(int(u)) for u in pos]) if len(pos) else np.zeros((0, kv_comp.shape[1]), np.uint16)
    sel = idx[idx >= 0]
    return np.concatenate([swa_rows, kv_comp[sel]], axis=0)


def attend_query(t, q, idx, kv_comp, swa_row_of, sink, *, W=128, sm_scale=1.0 / np.sqrt(512.0),
                 inverse_rope_out=False, rope_dim=64, theta=1e4):
    rows = gather_rows(t, np.asarray(idx), kv_comp, swa_row_of, W)
    out, lse = attend(q, rows, sink, sm_scale)
    if inverse_rope_out:
        out = inverse_rope(out, t, rope_dim=rope_dim, theta=theta)
    return out, lse


# ---- layer compositions -----------------------------------------------------

def layer_decode_one(t, ring_Ca, ring_Za, ring_Cb, ring_Zb, Ba, Bb, rms_w, kv_comp, kI, qI, wI, q, swa_ring,
                     sink, *, m=4, topk_k=512, W=128, rope_dim=64, theta=1e4, eps=1e-6,
                     sm_scale=1.0 / np.sqrt(512.0)):
    """One decode step of one sequence (the query at position t).

    kv_comp [n_cap, D] is copied; if (t+1) % m == 0 entry (t+1)/m - 1 is
    compressed from the staged ring rows (slot u mod 2m holds token u) and
    stored in the copy.  Returns (kv_comp_after, idx [topk], out [H, D], lse [H]).
    """
    kv = np.array(kv_comp, copy=True)
    if (t + 1) % m == 0:
        i = (t + 1) // m - 1
        slots_a = [(m * i + r) % (2 * m) for r in range(m)]
        slots_b = [(m * (i - 1) + r) % (2 * m) for r in range(m)]
        entry = compress_entry(i, ring_Ca[slots_a], ring_Za[slots_a], ring_Cb[slots_b], ring_Zb[slots_b],
                               Ba, Bb, rms_w, rope_dim=rope_dim, theta=theta, eps=eps)
        kv[i] = f64_to_bf16_bits(entry)
    V = visible(t, m)
    scores = index_scores(qI, wI, kI[:V])
    idx = topk(scores, topk_k)
    out, lse = attend_query(t, q, idx, kv, lambda u: swa_ring[u % W], sink, W=W, sm_scale=sm_scale)
    return kv, idx, out, lse


def f64_to_bf16_bits(x) -> np.ndarray:
    """Round-to-nearest-even of doubles to bf16 bits, used where the path
    stores a bf16 result that a later step reads (the compressed cache).
    Rounds to binary32 with round-to-odd first, which makes the second
    rounding (binary32 -> bf16, nearest-even) the correctly rounded result."""
    x = np.asarray(x, dtype=np.float64)
    f = x.astype(np.float32)
    u = f.view(np.uint32).astype(np.int64)
    inexact = f.astype(np.float64) != x
    overshoot = np.abs(f.astype(np.float64)) > np.abs(x)
    u = np.where(inexact & overshoot, u - 1, u)      # truncate toward zero
    u = np.where(inexact, u | 1, u)                  # sticky bit: round to odd
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)
