"""Python binding of libcsa, the GB300 (sm_103a) CSA layer hot path.

Argument marshalling only: every function below forwards to the C entry point
of the same name in ``libcsa.so`` (declared in ``include/csa.h``), passing
device pointers (``tensor.data_ptr()``), sizes, and the current CUDA stream.
All computation runs in the library's CUDA kernels; there is no fallback, and
importing this package fails if the library has not been built
(``python compressed_sparse_attention_02_gb300/build.py``).

Tensor conventions: bf16 tensors are ``torch.bfloat16``, FP8 E4M3 tensors are
``torch.float8_e4m3fn`` (or uint8 holding the same bits), positions and
indices ``torch.int32``, the sink ``torch.float32``; every tensor is
contiguous and on the current CUDA device.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIBRARY_PATH = os.path.join(_HERE, "libcsa.so")

if not os.path.exists(LIBRARY_PATH):
    raise ImportError(
        "libcsa.so is not built (expected at %s); run python compressed_sparse_attention_02_gb300/build.py"
        % LIBRARY_PATH)

_lib = ctypes.CDLL(LIBRARY_PATH)

CSA_OK = 0
STATUS_NAMES = {0: "CSA_OK", 1: "CSA_ERR_INVALID_ARG", 2: "CSA_ERR_UNSUPPORTED", 3: "CSA_ERR_CUDA",
                4: "CSA_ERR_TIMEOUT", 5: "CSA_ERR_INDEX_RANGE", 6: "CSA_ERR_WORKSPACE"}
(CSA_OP_COMPRESS, CSA_OP_INDEX_TOPK, CSA_OP_SPARSE_ATTN, CSA_OP_LAYER_DECODE, CSA_OP_LAYER_PREFILL,
 CSA_OP_INDEX_TOPK_POOL, CSA_OP_REINDEX_TOPK, CSA_OP_HCA_LAYER_DECODE) = range(8)
CSA_POOL_BLOCK = 8
CSA_FP4_ENTRY_BYTES = 288


class CsaParams(ctypes.Structure):
    """Mirror of ``csa_params``."""
    _fields_ = [("m", ctypes.c_int32), ("n_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("rope_dim", ctypes.c_int32), ("idx_heads", ctypes.c_int32), ("idx_dim", ctypes.c_int32),
                ("topk", ctypes.c_int32), ("swa_window", ctypes.c_int32), ("rope_theta", ctypes.c_float),
                ("rms_eps", ctypes.c_float), ("sm_scale", ctypes.c_float), ("inverse_rope", ctypes.c_int32),
                ("kv_format", ctypes.c_int32), ("bf16_scores", ctypes.c_int32), ("index_format", ctypes.c_int32)]


class CsaIndexKeySrc(ctypes.Structure):
    """Mirror of ``csa_index_key_src`` (device pointers)."""
    _fields_ = [(n, ctypes.c_void_p) for n in ("CIa", "ZIa", "CIb", "ZIb", "CIb_prev", "ZIb_prev", "BIa", "BIb",
                                                "rms_wI")]


def index_key_src(CIa, ZIa, CIb, ZIb, BIa, BIb, rms_wI, CIb_prev=None, ZIb_prev=None) -> CsaIndexKeySrc:
    """A ``csa_index_key_src`` over device tensors (which the caller keeps alive)."""
    return CsaIndexKeySrc(*[None if t is None else t.data_ptr()
                            for t in (CIa, ZIa, CIb, ZIb, CIb_prev, ZIb_prev, BIa, BIb, rms_wI)])


class CsaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__("%s returned %s: %s" % (where, STATUS_NAMES.get(status, status),
                                                  csa_status_string(status)))


_vp = ctypes.c_void_p
_i32, _i64, _sz = ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
_P = ctypes.POINTER(CsaParams)

_lib.csa_default_params.argtypes = [_P]
_lib.csa_default_params.restype = None
_lib.csa_workspace_size.argtypes = [_i32, _P, _i32, _i32, _i64]
_lib.csa_workspace_size.restype = _sz
_lib.csa_compress.argtypes = [_P, _i32, _i32, _i64] + [_vp] * 9 + [_vp, _i64, _vp]
_lib.csa_compress_indexer_keys.argtypes = [_P, _i32, _i32, _i64] + [_vp] * 9 + [_vp, _i64, _vp]
_lib.csa_index_topk.argtypes = [_P, _i32, _i32, _vp, _vp, _vp, _vp, _i64, _vp, _vp, _vp, _sz, _vp]
_lib.csa_index_topk_static.argtypes = [_P, _i32, _i32, _vp, _vp, _vp, _vp, _i64, _vp, _vp, _vp]
_lib.csa_index_topk_static.restype = ctypes.c_int
_lib.csa_compress_single.argtypes = [_P, _i32, _i32, _i64, _vp, _vp, _vp, _vp, _vp, _i64, _vp]
_lib.csa_compress_single.restype = ctypes.c_int
_lib.csa_compress_single_step.argtypes = [_P, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _vp]
_lib.csa_compress_single_step.restype = ctypes.c_int
_lib.csa_hca_layer_decode.argtypes = [_P, _i32] + [_vp] * 6 + [_vp, _i64] + [_vp] * 5 + [_vp, _sz, _vp]
_lib.csa_hca_layer_decode.restype = ctypes.c_int
_lib.csa_quantize_kv_fp4.argtypes = [_i64, _vp, _i64, _vp, _i64, _vp]
_lib.csa_quantize_kv_fp4.restype = ctypes.c_int
_lib.csa_quantize_index_keys_fp4.argtypes = [_i32, _i32, _i64, _vp, _i64, _vp, _i64, _vp]
_lib.csa_quantize_index_keys_fp4.restype = ctypes.c_int
_lib.csa_quantize_index_query_fp4.argtypes = [_i64, _vp, _vp, _vp]
_lib.csa_quantize_index_query_fp4.restype = ctypes.c_int
_lib.csa_index_topk_pool.argtypes = [_P, _i32, _i32, _vp, _vp, _vp, _vp, _i64, _vp, _vp, _i32, _vp, _vp, _sz, _vp]
_lib.csa_index_topk_pool.restype = ctypes.c_int
_lib.csa_reindex_topk.argtypes = [_P, _i32, _i32, _vp, _vp, _vp, _vp, _i64, _vp, _i32, _vp, _vp, _vp, _sz, _vp]
_lib.csa_reindex_topk.restype = ctypes.c_int
_lib.csa_sparse_attn.argtypes = [_P, _i32, _i32, _vp, _vp, _vp, _i64, _vp, _vp, _i32, _i64, _vp, _vp, _vp, _vp,
                                 _vp, _sz, _vp]
_lib.csa_layer_decode.argtypes = [_P, _i32, _vp] + [_vp] * 7 + [_vp, _i64] + [_vp] * 9 + [_vp, _sz, _vp]
_lib.csa_layer_decode_append.argtypes = [_P, _i32, _vp] + [_vp] * 9 + [_vp, _i64] + [_vp] * 9 + [_vp, _sz, _vp]
_lib.csa_layer_prefill.argtypes = [_P, _i32, _i32, _i64] + [_vp] * 9 + [_vp, _i64] + [_vp] * 9 + [_vp, _sz, _vp]
_K = ctypes.POINTER(CsaIndexKeySrc)
_lib.csa_layer_decode_with_keys.argtypes = ([_P, _i32, _vp, _vp, _K] + [_vp] * 7 + [_vp, _i64] + [_vp] * 9 +
                                            [_vp, _sz, _vp])
_lib.csa_layer_prefill_with_keys.argtypes = ([_P, _i32, _i32, _i64] + [_vp] * 9 + [_K, _vp, _i64] + [_vp] * 9 +
                                             [_vp, _sz, _vp])
for _f in ("csa_compress", "csa_compress_indexer_keys", "csa_index_topk", "csa_sparse_attn", "csa_layer_decode",
           "csa_layer_decode_append", "csa_layer_prefill", "csa_layer_decode_with_keys",
           "csa_layer_prefill_with_keys"):
    getattr(_lib, _f).restype = ctypes.c_int
_lib.csa_set_trace_events.argtypes = [ctypes.POINTER(_vp), _i32]
_lib.csa_set_trace_events.restype = ctypes.c_int
_lib.csa_launch_count.argtypes = []
_lib.csa_launch_count.restype = ctypes.c_uint64
_lib.csa_check_status.argtypes = [_vp]
_lib.csa_check_status.restype = ctypes.c_int
_lib.csa_status_string.argtypes = [ctypes.c_int]
_lib.csa_status_string.restype = ctypes.c_char_p


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(stream=None):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _check(status: int, where: str):
    if status != CSA_OK:
        raise CsaError(status, where)


def csa_default_params(**overrides) -> CsaParams:
    """The V4-Flash CSA parameters (m=4, 64x512 heads, top-k 512, window 128,
    theta 1e4, eps 1e-6, scale 1/sqrt(512)), with any field overridden."""
    p = CsaParams()
    _lib.csa_default_params(ctypes.byref(p))
    for k, v in overrides.items():
        setattr(p, k, v)
    return p


def csa_status_string(status: int) -> str:
    return _lib.csa_status_string(int(status)).decode()


def csa_workspace_size(op: int, params: CsaParams, B: int, Q: int, n_cap: int) -> int:
    return int(_lib.csa_workspace_size(op, ctypes.byref(params), B, Q, n_cap))


def workspace(op: int, params: CsaParams, B: int, Q: int, n_cap: int, device=None) -> torch.Tensor:
    """Allocates (through torch) a workspace of csa_workspace_size() bytes."""
    n = csa_workspace_size(op, params, B, Q, n_cap)
    if n == 0:
        raise CsaError(2, "csa_workspace_size")
    return torch.empty(n, dtype=torch.uint8, device=device or "cuda")


def csa_compress(params, B, n_new, entry0, Ca, Za, Cb, Zb, Cb_prev, Zb_prev, Ba, Bb, rms_w, kv_out, kv_stride_b,
                 stream=None):
    _check(_lib.csa_compress(ctypes.byref(params), B, n_new, entry0, _ptr(Ca), _ptr(Za), _ptr(Cb), _ptr(Zb),
                             _ptr(Cb_prev), _ptr(Zb_prev), _ptr(Ba), _ptr(Bb), _ptr(rms_w), _ptr(kv_out),
                             kv_stride_b, _stream(stream)), "csa_compress")


def csa_compress_indexer_keys(params, B, n_new, entry0, CIa, ZIa, CIb, ZIb, CIb_prev, ZIb_prev, BIa, BIb, rms_wI,
                              kI_out, kI_stride_b, stream=None):
    _check(_lib.csa_compress_indexer_keys(ctypes.byref(params), B, n_new, entry0, _ptr(CIa), _ptr(ZIa), _ptr(CIb),
                                          _ptr(ZIb), _ptr(CIb_prev), _ptr(ZIb_prev), _ptr(BIa), _ptr(BIb),
                                          _ptr(rms_wI), _ptr(kI_out), kI_stride_b, _stream(stream)),
           "csa_compress_indexer_keys")


def csa_compress_single(params, B, n_new, entry0, C, Z, bias, rms_w, kv_out, kv_stride_b, stream=None):
    _check(_lib.csa_compress_single(ctypes.byref(params), B, n_new, entry0, _ptr(C), _ptr(Z), _ptr(bias), _ptr(rms_w),
                                    _ptr(kv_out), kv_stride_b, _stream(stream)), "csa_compress_single")


def csa_compress_single_step(params, B, q_pos, C, Z, bias, rms_w, state, kv_out, kv_stride_b, n_cap, stream=None):
    _check(_lib.csa_compress_single_step(ctypes.byref(params), B, _ptr(q_pos), _ptr(C), _ptr(Z), _ptr(bias),
                                         _ptr(rms_w), _ptr(state), _ptr(kv_out), kv_stride_b, n_cap, _stream(stream)),
           "csa_compress_single_step")


def csa_index_topk(params, B, Q, q_pos, qI, wI, kI, n_cap, idx_out, score_out, ws, stream=None):
    _check(_lib.csa_index_topk(ctypes.byref(params), B, Q, _ptr(q_pos), _ptr(qI), _ptr(wI), _ptr(kI), n_cap,
                               _ptr(idx_out), _ptr(score_out), _ptr(ws), 0 if ws is None else ws.numel(),
                               _stream(stream)), "csa_index_topk")


def csa_hca_layer_decode(params, B, q_pos, C, Z, bias, rms_w, state, kv_comp, n_cap, q, swa_ring, sink, out, lse,
                         ws, stream=None):
    _check(_lib.csa_hca_layer_decode(ctypes.byref(params), B, _ptr(q_pos), _ptr(C), _ptr(Z), _ptr(bias), _ptr(rms_w),
                                     _ptr(state), _ptr(kv_comp), n_cap, _ptr(q), _ptr(swa_ring), _ptr(sink), _ptr(out),
                                     _ptr(lse), _ptr(ws), 0 if ws is None else ws.numel(), _stream(stream)),
           "csa_hca_layer_decode")


def csa_quantize_kv_fp4(n_rows, inp, in_stride, out, out_stride, stream=None):
    _check(_lib.csa_quantize_kv_fp4(n_rows, _ptr(inp), in_stride, _ptr(out), out_stride, _stream(stream)),
           "csa_quantize_kv_fp4")


def csa_quantize_index_keys_fp4(B, n_new, entry0, inp, in_stride_b, kI, n_cap, stream=None):
    _check(_lib.csa_quantize_index_keys_fp4(B, n_new, entry0, _ptr(inp), in_stride_b, _ptr(kI), n_cap,
                                            _stream(stream)), "csa_quantize_index_keys_fp4")


def csa_quantize_index_query_fp4(n_q, inp, qI, stream=None):
    _check(_lib.csa_quantize_index_query_fp4(n_q, _ptr(inp), _ptr(qI), _stream(stream)),
           "csa_quantize_index_query_fp4")


def index_keys_fp4_bytes(B: int, n_cap: int) -> int:
    """Bytes of an FP4 indexer key cache (CSA_FP4_INDEX_KEYS_BYTES)."""
    return B * (n_cap * 64 + (n_cap + 127) // 128 * 512)


def index_query_fp4_bytes(n_q: int) -> int:
    """Bytes of n_q FP4 indexer query records (CSA_FP4_INDEX_QUERY_BYTES)."""
    return n_q * 4608


def csa_index_topk_pool(params, B, Q, q_pos, qI, wI, kI, n_cap, idx_out, score_out, pool_blocks, pool_out, ws,
                        stream=None):
    _check(_lib.csa_index_topk_pool(ctypes.byref(params), B, Q, _ptr(q_pos), _ptr(qI), _ptr(wI), _ptr(kI), n_cap,
                                    _ptr(idx_out), _ptr(score_out), pool_blocks, _ptr(pool_out), _ptr(ws),
                                    0 if ws is None else ws.numel(), _stream(stream)), "csa_index_topk_pool")


def csa_reindex_topk(params, B, Q, q_pos, qI, wI, kI, n_cap, pool, pool_blocks, idx_out, score_out, ws,
                     stream=None):
    _check(_lib.csa_reindex_topk(ctypes.byref(params), B, Q, _ptr(q_pos), _ptr(qI), _ptr(wI), _ptr(kI), n_cap,
                                 _ptr(pool), pool_blocks, _ptr(idx_out), _ptr(score_out), _ptr(ws),
                                 0 if ws is None else ws.numel(), _stream(stream)), "csa_reindex_topk")


STATIC_SCRATCH_BYTES = 16 << 20


def csa_index_topk_static(params, B, Q, q_pos, qI, wI, kI, n_cap, idx_out, score_out, stream=None):
    """csa_index_topk with its scratch in libcsa's fixed 16 MiB device array
    instead of a caller-provided workspace, for callers that cannot allocate
    device memory at the call (their own pool holds the GPU's memory, or they
    must not risk cudaMalloc blocking the host and synchronising the device).
    The first call on a device should come before any stream capture; calls
    that can overlap on the GPU race on the shared array."""
    _check(_lib.csa_index_topk_static(ctypes.byref(params), B, Q, _ptr(q_pos), _ptr(qI), _ptr(wI), _ptr(kI), n_cap,
                                      _ptr(idx_out), _ptr(score_out), _stream(stream)), "csa_index_topk_static")


def csa_sparse_attn(params, B, Q, q_pos, q, kv_comp, n_cap, idx, swa, swa_mode, swa_len, swa_pos0, sink, out,
                    lse=None, ws=None, stream=None):
    _check(_lib.csa_sparse_attn(ctypes.byref(params), B, Q, _ptr(q_pos), _ptr(q), _ptr(kv_comp), n_cap, _ptr(idx),
                                _ptr(swa), swa_mode, swa_len, _ptr(swa_pos0), _ptr(sink), _ptr(out), _ptr(lse),
                                _ptr(ws), 0 if ws is None else ws.numel(), _stream(stream)), "csa_sparse_attn")


def csa_layer_decode(params, B, q_pos, ring_Ca, ring_Za, ring_Cb, ring_Zb, Ba, Bb, rms_w, kv_comp, n_cap, kI, qI,
                     wI, q, swa_ring, sink, idx_out, out, lse, ws, stream=None):
    _check(_lib.csa_layer_decode(ctypes.byref(params), B, _ptr(q_pos), _ptr(ring_Ca), _ptr(ring_Za),
                                 _ptr(ring_Cb), _ptr(ring_Zb), _ptr(Ba), _ptr(Bb), _ptr(rms_w), _ptr(kv_comp),
                                 n_cap, _ptr(kI), _ptr(qI), _ptr(wI), _ptr(q), _ptr(swa_ring), _ptr(sink),
                                 _ptr(idx_out), _ptr(out), _ptr(lse), _ptr(ws), 0 if ws is None else ws.numel(),
                                 _stream(stream)), "csa_layer_decode")


def csa_layer_decode_append(params, B, q_pos, swa_new, kI_new, ring_Ca, ring_Za, ring_Cb, ring_Zb, Ba, Bb, rms_w,
                            kv_comp, n_cap, kI, qI, wI, q, swa_ring, sink, idx_out, out, lse, ws, stream=None):
    _check(_lib.csa_layer_decode_append(ctypes.byref(params), B, _ptr(q_pos), _ptr(swa_new), _ptr(kI_new),
                                        _ptr(ring_Ca), _ptr(ring_Za), _ptr(ring_Cb), _ptr(ring_Zb), _ptr(Ba),
                                        _ptr(Bb), _ptr(rms_w), _ptr(kv_comp), n_cap, _ptr(kI), _ptr(qI), _ptr(wI),
                                        _ptr(q), _ptr(swa_ring), _ptr(sink), _ptr(idx_out), _ptr(out), _ptr(lse),
                                        _ptr(ws), 0 if ws is None else ws.numel(), _stream(stream)),
           "csa_layer_decode_append")


def csa_layer_decode_with_keys(params, B, q_pos, swa_new, keys, ring_Ca, ring_Za, ring_Cb, ring_Zb, Ba, Bb, rms_w,
                               kv_comp, n_cap, kI, qI, wI, q, swa_ring, sink, idx_out, out, lse, ws, stream=None):
    """``keys``: a CsaIndexKeySrc (see index_key_src) over the key compressor's staging rings."""
    _check(_lib.csa_layer_decode_with_keys(ctypes.byref(params), B, _ptr(q_pos), _ptr(swa_new),
                                           None if keys is None else ctypes.byref(keys), _ptr(ring_Ca),
                                           _ptr(ring_Za), _ptr(ring_Cb), _ptr(ring_Zb), _ptr(Ba), _ptr(Bb),
                                           _ptr(rms_w), _ptr(kv_comp), n_cap, _ptr(kI), _ptr(qI), _ptr(wI), _ptr(q),
                                           _ptr(swa_ring), _ptr(sink), _ptr(idx_out), _ptr(out), _ptr(lse),
                                           _ptr(ws), 0 if ws is None else ws.numel(), _stream(stream)),
           "csa_layer_decode_with_keys")


def csa_layer_prefill_with_keys(params, B, Q, pos0, Ca, Za, Cb, Zb, Cb_prev, Zb_prev, Ba, Bb, rms_w, keys, kv_comp,
                                n_cap, kI, qI, wI, q, swa, sink, idx_out, out, lse, ws, stream=None):
    """``keys``: a CsaIndexKeySrc (see index_key_src) over the chunk's key compressor rows."""
    _check(_lib.csa_layer_prefill_with_keys(ctypes.byref(params), B, Q, pos0, _ptr(Ca), _ptr(Za), _ptr(Cb),
                                            _ptr(Zb), _ptr(Cb_prev), _ptr(Zb_prev), _ptr(Ba), _ptr(Bb), _ptr(rms_w),
                                            None if keys is None else ctypes.byref(keys), _ptr(kv_comp), n_cap,
                                            _ptr(kI), _ptr(qI), _ptr(wI), _ptr(q), _ptr(swa), _ptr(sink),
                                            _ptr(idx_out), _ptr(out), _ptr(lse), _ptr(ws),
                                            0 if ws is None else ws.numel(), _stream(stream)),
           "csa_layer_prefill_with_keys")


def csa_layer_prefill(params, B, Q, pos0, Ca, Za, Cb, Zb, Cb_prev, Zb_prev, Ba, Bb, rms_w, kv_comp, n_cap, kI, qI,
                      wI, q, swa, sink, idx_out, out, lse, ws, stream=None):
    _check(_lib.csa_layer_prefill(ctypes.byref(params), B, Q, pos0, _ptr(Ca), _ptr(Za), _ptr(Cb), _ptr(Zb),
                                  _ptr(Cb_prev), _ptr(Zb_prev), _ptr(Ba), _ptr(Bb), _ptr(rms_w), _ptr(kv_comp),
                                  n_cap, _ptr(kI), _ptr(qI), _ptr(wI), _ptr(q), _ptr(swa), _ptr(sink),
                                  _ptr(idx_out), _ptr(out), _ptr(lse), _ptr(ws), 0 if ws is None else ws.numel(),
                                  _stream(stream)), "csa_layer_prefill")


CSA_TEST_FAULT_INDEXER, CSA_TEST_FAULT_TOPK, CSA_TEST_FAULT_ATTN = 1, 2, 4
_lib.csa_test_set_wait_fault.argtypes = [ctypes.c_uint32, ctypes.c_uint32]
_lib.csa_test_set_wait_fault.restype = ctypes.c_int


def csa_test_set_wait_fault(wait_limit_us, faults):
    """Test-only: device wait limit (us, 0 = default) and withheld signals (CSA_TEST_FAULT_*)."""
    _check(_lib.csa_test_set_wait_fault(wait_limit_us, faults), "csa_test_set_wait_fault")


def csa_check_status(stream=None) -> int:
    """Synchronises the stream and returns (and clears) the device status."""
    return int(_lib.csa_check_status(_stream(stream)))


def csa_set_trace_events(events) -> None:
    """Record the five stage-boundary events (torch.cuda.Event, timing
    enabled) in every following layer call; None turns tracing off."""
    if events is None:
        _check(_lib.csa_set_trace_events(None, 0), "csa_set_trace_events")
        return
    for e in events:
        if not e.cuda_event:  # torch creates the CUDA event at its first record
            e.record()
    arr = (_vp * len(events))(*[e.cuda_event for e in events])
    _check(_lib.csa_set_trace_events(arr, len(events)), "csa_set_trace_events")


def csa_launch_count() -> int:
    """Kernels launched by libcsa in this process so far."""
    return int(_lib.csa_launch_count())
