"""ctypes declarations of librq's C ABI (include/rq.h, include/rq_synth.h, include/rq_test.h,
include/rq_ablation.h).

Loading fails loudly: there is no fallback implementation of any entry point.
"""

import ctypes
import os

RQ_MAX_LOOPS = 16
LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "librq.so")

STATUS = {0: "RQ_OK", 1: "RQ_ERR_INVALID_ARG", 2: "RQ_ERR_UNSUPPORTED",
          3: "RQ_ERR_WORKSPACE", 4: "RQ_ERR_CUDA", 5: "RQ_ERR_INTERNAL"}

EXPORTS = ("rq_cache_bytes", "rq_record_bytes", "rq_encode_append", "rq_decode_workspace_bytes",
           "rq_decode_attention", "rq_bf16_decode_attention", "rq_status_str",
           "rq_synth_states", "rq_synth_queries", "rq_decode_noalloc_scratch_bytes",
           "rq_decode_attention_noalloc", "rq_paged_cache_bytes", "rq_paged_encode_append",
           "rq_paged_decode_attention", "rq_advance_ctx",
           "rq_test_decode_attention_wait_runs_out", "rq_ablation_encode_append",
           "rq_ablation_decode_attention")


class RqShape(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("n_q_heads", ctypes.c_int32),
                ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("n_loops", ctypes.c_int32), ("group", ctypes.c_int32),
                ("capacity", ctypes.c_int32), ("res_bits", ctypes.c_int8 * RQ_MAX_LOOPS),
                ("softmax_scale", ctypes.c_float)]


_P = ctypes.c_void_p


class RqCache(ctypes.Structure):
    _fields_ = [("data", _P), ("rot_signs", _P * 2)]


class RqPaging(ctypes.Structure):
    _fields_ = [("block_table", _P), ("max_pages", ctypes.c_int32), ("n_pages", ctypes.c_int32)]


class RqSynthParams(ctypes.Structure):
    _fields_ = [("seed", ctypes.c_uint64), ("layer", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32),
                ("dist", ctypes.c_int32), ("sigma", ctypes.c_float * RQ_MAX_LOOPS),
                ("outlier_mult", ctypes.c_float), ("n_outliers", ctypes.c_int32),
                ("outlier_table", _P)]


class RqError(RuntimeError):
    def __init__(self, fn, status):
        super().__init__("%s returned %s" % (fn, STATUS.get(status, status)))
        self.status = status


_lib = None


def lib():
    """The loaded librq.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError("librq.so is not built: run looped_transformer_kv_gb300.build.build() "
                           "(the CUDA extension is required; there is no CPU fallback)")
    L = ctypes.CDLL(LIB_PATH)
    i32, i64, sz = ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    S, C = ctypes.POINTER(RqShape), ctypes.POINTER(RqCache)
    L.rq_cache_bytes.argtypes = [S]
    L.rq_cache_bytes.restype = sz
    L.rq_record_bytes.argtypes = [S]
    L.rq_record_bytes.restype = sz
    L.rq_encode_append.argtypes = [S, C, _P, ctypes.POINTER(i64), _P, i32, i32, _P]
    L.rq_encode_append.restype = i32
    L.rq_decode_workspace_bytes.argtypes = [S, i32, i32]
    L.rq_decode_workspace_bytes.restype = sz
    L.rq_decode_attention.argtypes = [S, C, _P, i32, i32, _P, _P, i32, _P, _P, sz, _P]
    L.rq_decode_attention.restype = i32
    L.rq_bf16_decode_attention.argtypes = [S, _P, _P, _P, i32, i32, _P, _P, i32, _P, _P, sz, _P]
    L.rq_bf16_decode_attention.restype = i32
    L.rq_decode_noalloc_scratch_bytes.argtypes = []
    L.rq_decode_noalloc_scratch_bytes.restype = sz
    L.rq_decode_attention_noalloc.argtypes = [S, C, _P, i32, i32, _P, _P, i32, _P, _P]
    L.rq_decode_attention_noalloc.restype = i32
    G = ctypes.POINTER(RqPaging)
    L.rq_paged_cache_bytes.argtypes = [S, i32]
    L.rq_paged_cache_bytes.restype = sz
    L.rq_paged_encode_append.argtypes = [S, C, G, _P, ctypes.POINTER(i64), _P, i32, i32, _P]
    L.rq_paged_encode_append.restype = i32
    L.rq_paged_decode_attention.argtypes = [S, C, G, _P, i32, i32, _P, _P, i32, _P, _P, sz, _P]
    L.rq_paged_decode_attention.restype = i32
    L.rq_test_decode_attention_wait_runs_out.argtypes = [S, C, _P, i32, i32, _P, _P, i32, _P,
                                                         _P, sz, ctypes.c_uint64, _P]
    L.rq_test_decode_attention_wait_runs_out.restype = i32
    L.rq_ablation_encode_append.argtypes = [S, C, _P, ctypes.POINTER(i64), _P, i32, i32, i32, _P]
    L.rq_ablation_encode_append.restype = i32
    L.rq_ablation_decode_attention.argtypes = [S, C, i32, _P, i32, _P, _P, i32, _P, _P, sz, _P]
    L.rq_ablation_decode_attention.restype = i32
    L.rq_advance_ctx.argtypes = [_P, i32, i32, i32, _P]
    L.rq_advance_ctx.restype = i32
    L.rq_status_str.argtypes = [i32]
    L.rq_status_str.restype = ctypes.c_char_p
    P = ctypes.POINTER(RqSynthParams)
    L.rq_synth_states.argtypes = [P, _P, ctypes.POINTER(i64), i32, i32, i32, i32, i32, i32, _P]
    L.rq_synth_states.restype = i32
    L.rq_synth_queries.argtypes = [P, _P, i32, i32, i32, i32, i32, i32, _P]
    L.rq_synth_queries.restype = i32
    _lib = L
    return L


def check(fn, status):
    if status != 0:
        raise RqError(fn, status)
