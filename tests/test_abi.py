"""The C-ABI library loads on a machine without a GPU, exports every entry
point include/csa.h declares, and rejects bad arguments on the host before any
launch."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "csa.h")


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__._load_builder().build()
    import compressed_sparse_attention_02_gb300 as csa
    return csa


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(csa_[a-z_]+)\s*\(", text)))


def test_every_declared_entry_point_is_exported(lib):
    names = declared_functions()
    assert {"csa_compress", "csa_index_topk", "csa_sparse_attn", "csa_layer_decode", "csa_layer_prefill",
            "csa_check_status", "csa_workspace_size"} <= set(names)
    raw = ctypes.CDLL(lib.LIBRARY_PATH)
    for n in names:
        assert hasattr(raw, n), n


def test_default_params_and_status_strings(lib):
    p = lib.csa_default_params()
    assert (p.m, p.n_heads, p.head_dim, p.rope_dim, p.idx_heads, p.idx_dim, p.topk, p.swa_window) == \
        (4, 64, 512, 64, 64, 128, 512, 128)
    assert abs(p.sm_scale - 512 ** -0.5) < 1e-7 and p.rope_theta == 1e4
    assert p.inverse_rope == 0 and p.kv_format == 0 and p.bf16_scores == 0 and p.index_format == 0
    assert ctypes.sizeof(p) == 15 * 4
    for s in range(7):
        assert lib.csa_status_string(s).startswith(lib.STATUS_NAMES[s])


def test_workspace_sizes(lib):
    p = lib.csa_default_params()
    n = lib.csa_workspace_size(lib.CSA_OP_LAYER_DECODE, p, 64, 1, 32768)
    assert n >= 64 * 32768 * 4
    assert lib.csa_workspace_size(lib.CSA_OP_INDEX_TOPK, p, 8, 1, 262144) >= 8 * 262144 * 4
    bad = lib.csa_default_params(head_dim=256)
    assert lib.csa_workspace_size(lib.CSA_OP_INDEX_TOPK, bad, 1, 1, 1024) == 0
    bad = lib.csa_default_params(inverse_rope=2)  # a flag: 0 or 1
    assert lib.csa_workspace_size(lib.CSA_OP_INDEX_TOPK, bad, 1, 1, 1024) == 0


def _call_raw(lib, fn, *args):
    return getattr(ctypes.CDLL(lib.LIBRARY_PATH), fn)(*args)


def test_host_validation_rejects_before_launch(lib):
    raw = ctypes.CDLL(lib.LIBRARY_PATH)
    raw.csa_index_topk.restype = ctypes.c_int
    raw.csa_compress.restype = ctypes.c_int
    raw.csa_layer_decode.restype = ctypes.c_int
    p = lib.csa_default_params()
    P = ctypes.byref(p)
    fake = ctypes.c_void_p(0x10000)       # aligned, never dereferenced: rejected first
    odd = ctypes.c_void_p(0x10008)        # 8-byte aligned only
    i64 = ctypes.c_int64
    # null pointers
    assert raw.csa_index_topk(P, 1, 1, None, None, None, None, i64(1024), None, None, None, ctypes.c_size_t(0),
                              None) == 1
    # misaligned pointer
    assert raw.csa_compress(P, 1, 4, i64(0), odd, fake, fake, fake, None, None, fake, fake, fake, fake, i64(4096),
                            None) == 1
    # previous-block rows must be given iff entry0 > 0
    assert raw.csa_compress(P, 1, 4, i64(3), fake, fake, fake, fake, None, None, fake, fake, fake, fake,
                            i64(8 * 512), None) == 1
    # unsupported dimensions
    p2 = lib.csa_default_params(n_heads=128)
    assert raw.csa_compress(ctypes.byref(p2), 1, 4, i64(0), fake, fake, fake, fake, None, None, fake, fake, fake,
                            fake, i64(4096), None) == 2
    p3 = lib.csa_default_params(topk=4096)
    assert raw.csa_index_topk(ctypes.byref(p3), 1, 1, fake, fake, fake, fake, i64(1024), fake, None, fake,
                              ctypes.c_size_t(1 << 30), None) == 2
    # workspace too small
    assert raw.csa_index_topk(P, 1, 1, fake, fake, fake, fake, i64(1024), fake, None, fake, ctypes.c_size_t(16),
                              None) == 6
    # empty batch is a no-op
    assert raw.csa_compress(P, 0, 4, i64(0), None, None, None, None, None, None, None, None, None, None, i64(0),
                            None) == 0


def test_pool_calls_validate_and_size_their_workspace(lib):
    raw = ctypes.CDLL(lib.LIBRARY_PATH)
    raw.csa_index_topk_pool.restype = ctypes.c_int
    raw.csa_reindex_topk.restype = ctypes.c_int
    p = lib.csa_default_params()
    P = ctypes.byref(p)
    fake = ctypes.c_void_p(0x10000)
    i64, sz = ctypes.c_int64, ctypes.c_size_t
    big = sz(1 << 40)
    # pool_blocks: 16..2048, a multiple of 16
    for nb in (0, 8, 24, 2064):
        assert raw.csa_index_topk_pool(P, 1, 1, fake, fake, fake, fake, i64(4096), fake, None, nb, fake, fake, big,
                                       None) == 2
        assert raw.csa_reindex_topk(P, 1, 1, fake, fake, fake, fake, i64(4096), fake, nb, fake, None, fake, big,
                                    None) == 2
    # a missing pool / pool output is an argument error
    assert raw.csa_index_topk_pool(P, 1, 1, fake, fake, fake, fake, i64(4096), fake, None, 64, None, fake, big,
                                   None) == 1
    assert raw.csa_reindex_topk(P, 1, 1, fake, fake, fake, fake, i64(4096), None, 64, fake, None, fake, big,
                                None) == 1
    # workspace too small
    assert raw.csa_index_topk_pool(P, 1, 1, fake, fake, fake, fake, i64(4096), fake, None, 64, fake, fake, sz(16),
                                   None) == 6
    assert raw.csa_reindex_topk(P, 1, 1, fake, fake, fake, fake, i64(4096), fake, 64, fake, None, fake, sz(16),
                                None) == 6
    # the Full layer's scratch holds the entries' and the blocks' selections
    full = lib.csa_workspace_size(lib.CSA_OP_INDEX_TOPK, p, 64, 1, 32768)
    pool = lib.csa_workspace_size(lib.CSA_OP_INDEX_TOPK_POOL, p, 64, 1, 32768)
    assert pool > full + 64 * (32768 // 8) * 4
    # the Reindex layer's scratch holds 16384 slot scores per query
    assert lib.csa_workspace_size(lib.CSA_OP_REINDEX_TOPK, p, 64, 1, 32768) >= 64 * 16384 * 4


def test_block_sizes_and_single_stream_calls_validate(lib):
    raw = ctypes.CDLL(lib.LIBRARY_PATH)
    for n in ("csa_compress", "csa_compress_single", "csa_compress_single_step", "csa_layer_decode"):
        getattr(raw, n).restype = ctypes.c_int
    fake = ctypes.c_void_p(0x10000)
    i64 = ctypes.c_int64
    # m: a power of two up to 128
    for m in (3, 256, 0):
        p = lib.csa_default_params(m=m)
        assert raw.csa_compress_single(ctypes.byref(p), 1, 1, i64(0), fake, fake, None, fake, fake, i64(512),
                                       None) == 2
    p128 = lib.csa_default_params(m=128)
    # the overlapped compressor and the layer calls stop at 8
    assert raw.csa_compress(ctypes.byref(p128), 1, 4, i64(0), fake, fake, fake, fake, None, None, fake, fake, fake,
                            fake, i64(4096), None) == 2
    # single stream: bias optional, state required for the step form
    assert raw.csa_compress_single(ctypes.byref(p128), 1, 1, i64(0), fake, None, None, fake, fake, i64(512),
                                   None) == 1
    assert raw.csa_compress_single_step(ctypes.byref(p128), 1, fake, fake, fake, None, fake, None, fake, i64(512),
                                        i64(1), None) == 1
    assert raw.csa_compress_single(ctypes.byref(p128), 0, 1, i64(0), None, None, None, None, None, i64(0),
                                   None) == 0


def test_layer_decode_append_argument_checks(lib):
    """The append form refuses on the host, before any launch: swa_new missing
    or misaligned, kI_new misaligned, kI_new with FP4 index keys."""
    raw = ctypes.CDLL(lib.LIBRARY_PATH)
    raw.csa_layer_decode_append.restype = ctypes.c_int
    fake, odd = ctypes.c_void_p(0x10000), ctypes.c_void_p(0x10008)

    def call(p, swa_new, kI_new):
        return raw.csa_layer_decode_append(ctypes.byref(p), 1, fake, swa_new, kI_new, *([fake] * 8),
                                           ctypes.c_int64(4096), *([fake] * 9), fake, ctypes.c_size_t(1 << 30), None)
    p = lib.csa_default_params()
    assert call(p, None, fake) == 1
    assert call(p, odd, fake) == 1
    assert call(p, fake, odd) == 1
    assert call(lib.csa_default_params(index_format=1), fake, fake) == 2


def test_layer_calls_with_keys_argument_checks(lib):
    """The layer calls that compute their own indexer keys refuse on the host,
    before any launch: no key source, a null or misaligned array in it, the
    previous-block rows not given exactly when the chunk does not start the
    sequence, FP4 index keys; the size of the source struct is nine pointers."""
    raw = ctypes.CDLL(lib.LIBRARY_PATH)
    raw.csa_layer_decode_with_keys.restype = ctypes.c_int
    raw.csa_layer_prefill_with_keys.restype = ctypes.c_int
    assert ctypes.sizeof(lib.CsaIndexKeySrc) == 9 * ctypes.sizeof(ctypes.c_void_p)
    fake, odd = 0x10000, 0x10008
    i64 = ctypes.c_int64

    def src(**kw):
        f = {n: fake for n in ("CIa", "ZIa", "CIb", "ZIb", "BIa", "BIb", "rms_wI")}
        f.update(kw)
        return lib.CsaIndexKeySrc(**f)

    def dec(p, keys):
        return raw.csa_layer_decode_with_keys(ctypes.byref(p), 1, ctypes.c_void_p(fake), None,
                                              None if keys is None else ctypes.byref(keys),
                                              *([ctypes.c_void_p(fake)] * 7), i64(4096),
                                              *([ctypes.c_void_p(fake)] * 9), ctypes.c_void_p(fake),
                                              ctypes.c_size_t(1 << 30), None)

    def pre(p, keys, pos0):
        prev = [ctypes.c_void_p(fake) if pos0 else None] * 2
        return raw.csa_layer_prefill_with_keys(ctypes.byref(p), 1, 16, i64(pos0), *([ctypes.c_void_p(fake)] * 4),
                                               *prev, *([ctypes.c_void_p(fake)] * 3),
                                               None if keys is None else ctypes.byref(keys), ctypes.c_void_p(fake),
                                               i64(4096), *([ctypes.c_void_p(fake)] * 9), ctypes.c_void_p(fake),
                                               ctypes.c_size_t(1 << 30), None)
    p = lib.csa_default_params()
    assert dec(p, None) == 1
    assert dec(p, src(CIa=None)) == 1
    assert dec(p, src(rms_wI=odd)) == 1
    assert dec(lib.csa_default_params(index_format=1), src()) == 2
    assert pre(p, None, 0) == 1
    assert pre(p, src(BIb=None), 0) == 1
    assert pre(p, src(CIb_prev=fake, ZIb_prev=fake), 0) == 1  # block -1 does not exist
    assert pre(p, src(), 64) == 1  # its rows are needed past the first chunk
    assert pre(lib.csa_default_params(index_format=1), src(), 0) == 2


def test_fp4_indexer_argument_checks(lib):
    """FP4 indexer rows: sizes of the layouts, and host-side refusals (no launch)."""
    assert lib.index_keys_fp4_bytes(2, 300) == 2 * (300 * 64 + 3 * 512)
    assert lib.index_query_fp4_bytes(5) == 5 * (64 * 64 + 512)
    raw = ctypes.CDLL(lib.LIBRARY_PATH)
    for fn in ("csa_quantize_index_keys_fp4", "csa_quantize_index_query_fp4", "csa_compress_indexer_keys"):
        getattr(raw, fn).restype = ctypes.c_int
    fake = ctypes.c_void_p(0x10000)
    i64 = ctypes.c_int64
    # entries past the cache, a stride that is not a multiple of 8, a null input
    assert raw.csa_quantize_index_keys_fp4(1, 8, i64(100), fake, i64(1024), fake, i64(104), None) == 1
    assert raw.csa_quantize_index_keys_fp4(2, 8, i64(0), fake, i64(1028), fake, i64(104), None) == 1
    assert raw.csa_quantize_index_query_fp4(i64(3), None, fake, None) == 1
    assert raw.csa_quantize_index_query_fp4(i64(0), None, None, None) == 0  # nothing to do
    # formats: only 0 and 1; the E4M3 key compressor takes no FP4
    assert lib.csa_workspace_size(lib.CSA_OP_INDEX_TOPK, lib.csa_default_params(index_format=2), 1, 1, 1024) == 0
    p4 = lib.csa_default_params(index_format=1)
    assert raw.csa_compress_indexer_keys(ctypes.byref(p4), 1, 4, i64(0), *([fake] * 4), None, None,
                                         *([fake] * 4), i64(512), None) == 2


def test_fp4_layouts_give_the_890_bytes_per_token_of_the_csa2_accounting():
    """[CSA2 详解] §16: a Main KV entry is 288 B and an indexer key 68 B; at
    2.5 entries per token (three ratio-2 encoder sources, one ratio-1 decoder
    source) that is 890 B per token.  The library's layouts take exactly those
    bytes per entry (the scale atoms of 128 keys amortised)."""
    import re as _re
    text = open(HEADER).read()
    main = int(_re.search(r"#define CSA_FP4_ENTRY_BYTES (\d+)", text).group(1))
    import compressed_sparse_attention_02_gb300 as csa
    key = csa.index_keys_fp4_bytes(1, 128 * 1000) / (128 * 1000)
    assert (main, key) == (288, 68)
    assert (main + key) * (3 * 0.5 + 1 * 1.0) == 890
