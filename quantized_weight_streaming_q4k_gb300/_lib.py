"""ctypes loader for libqws.so (built in-tree by build.py).

Loading fails loudly: there is no CPU path behind these calls.
"""
from __future__ import annotations

import ctypes as C
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libqws.so")

QWS_OK = 0
STATUS_NAMES = {
    0: "QWS_OK", 1: "QWS_ERR_NULL", 2: "QWS_ERR_SHAPE", 3: "QWS_ERR_ALIGN",
    4: "QWS_ERR_FORMAT", 5: "QWS_ERR_WORKSPACE", 6: "QWS_ERR_CUDA", 7: "QWS_ERR_TIMEOUT",
}
Q4_0, Q8_0, Q4_K, Q6_K = 2, 8, 12, 14
OP_MATVEC, OP_FFN, OP_DECODE_CHAIN, OP_PREFILL, OP_KV_ATTENTION = 0, 1, 2, 3, 4


class QwsLayer(C.Structure):
    _fields_ = [
        ("Wq", C.c_void_p), ("Wk", C.c_void_p), ("Wv", C.c_void_p), ("Wo", C.c_void_p),
        ("Wg", C.c_void_p), ("Wu", C.c_void_p), ("Wd", C.c_void_p),
        ("fmt_qkv", C.c_int), ("fmt_o", C.c_int), ("fmt_gu", C.c_int), ("fmt_down", C.c_int),
        ("w_in", C.c_void_p), ("w_post_attn", C.c_void_p), ("w_pre_ffn", C.c_void_p),
        ("w_post_ffn", C.c_void_p),
    ]


class QwsDims(C.Structure):
    _fields_ = [
        ("hidden", C.c_int64), ("inter", C.c_int64),
        ("n_q_heads", C.c_int), ("n_kv_heads", C.c_int), ("head_dim", C.c_int),
        ("eps", C.c_float), ("post_norms", C.c_int),
    ]


class QwsKv(C.Structure):
    _fields_ = [
        ("k_caches", C.c_void_p), ("v_caches", C.c_void_p), ("max_seq", C.c_int64),
        ("pos", C.c_int64), ("rot_dim", C.c_int), ("rope_base", C.c_double),
        ("attn_scale", C.c_float), ("softcap", C.c_float),
    ]


# name -> (restype, argtypes); mirrors include/qws.h
P, F, I64, I, SZ, U = C.c_void_p, C.c_void_p, C.c_int64, C.c_int, C.c_size_t, C.c_uint
SIGNATURES = {
    "qws_q4k_matvec": (I, [P, F, F, I64, I64, I, P]),
    "qws_q6k_matvec": (I, [P, F, F, I64, I64, I, P]),
    "qws_q4_0_matvec": (I, [P, F, F, I64, I64, I, I, P, SZ, P]),
    "qws_matvec": (I, [I, P, F, F, I64, I64, I, I, P, SZ, P]),
    "qws_q4k_qkv_proj": (I, [P, P, P, F, F, F, F, I64, I64, I64, P]),
    "qws_q4k_ffn_gate_up_geglu_down": (I, [P, P, P, I, F, F, I64, I64, P, SZ, P]),
    "qws_q4k_ffn_gate_up_geglu": (I, [P, P, F, F, I64, I64, P]),
    "qws_q4k_ffn_gate_up_geglu_down_noalloc": (I, [P, P, P, I, F, F, I64, I64, P]),
    "qws_q4k_ffn_gate_up_silu_down": (I, [P, P, P, I, F, F, I64, I64, P, SZ, P]),
    "qws_q4k_ffn_gate_up_silu": (I, [P, P, F, F, I64, I64, P]),
    "qws_residual_rms_norm": (I, [F, F, F, F, I64, C.c_float, I, P]),
    "qws_quantize_q8_0": (I, [F, P, I64, I, P]),
    "qws_q4k_prefill_matmul": (I, [P, F, F, I64, I64, I64, P, SZ, P]),
    "qws_rope_at_pos": (I, [F, I, I, I, I64, C.c_double, P]),
    "qws_kv_append": (I, [F, F, F, F, I, I, I64, I64, P]),
    "qws_kv_attention": (I, [F, F, F, F, I, I, I, I64, I64, C.c_float, C.c_float, P, SZ, P]),
    "qws_q8_matvec": (I, [I, P, P, F, I64, I64, I, P]),
    "qws_rms_norm_q8": (I, [F, F, P, I64, C.c_float, I, P]),
    "qws_residual_rms_norm_q8": (I, [F, F, F, P, I64, C.c_float, I, P]),
    "qws_q8_qkv_proj": (I, [I, P, P, P, P, F, F, F, I64, I64, I64, P]),
    "qws_rms_norm": (I, [F, F, F, I64, C.c_float, I, P]),
    "qws_residual_add": (I, [F, F, I64, I, P]),
    "qws_decode_chain": (I, [C.POINTER(QwsLayer), I, F, C.POINTER(QwsDims), P, SZ, P]),
    "qws_decode_chain_final_norm": (I, [C.POINTER(QwsLayer), I, F, F, F, C.POINTER(QwsDims), P,
                                        SZ, P]),
    "qws_workspace_bytes": (SZ, [I, I64, I64, I64, I, I]),
    "qws_last_error": (C.c_char_p, []),
    "qws_device_error": (I, [C.POINTER(U)]),
    "qws_version": (C.c_char_p, []),
    "qws_selftest_wait_timeout": (I, [C.c_int, C.c_longlong, C.c_void_p, C.c_void_p]),
    "qws_decode_kv_workspace_bytes": (SZ, [C.POINTER(QwsDims), I64]),
    "qws_decode_kv": (I, [C.POINTER(QwsLayer), I, F, C.POINTER(QwsDims), C.POINTER(QwsKv), P,
                          SZ, P]),
}

_lib = None
_lock = threading.Lock()


class QwsError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


def lib():
    """The loaded library.  Raises if libqws.so has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build it with "
                    "`python -m quantized_weight_streaming_q4k_gb300.build`")
            h = C.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(h, name)
                fn.restype = res
                fn.argtypes = args
            _lib = h
        return _lib


def check(status: int) -> None:
    if status != QWS_OK:
        msg = lib().qws_last_error()
        raise QwsError(status, msg.decode() if msg else "")
