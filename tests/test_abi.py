"""C-ABI checks that need no GPU: the library loads, exports every function
include/qws.h declares, and rejects bad arguments on the host before any CUDA
call (every case below returns before the first CUDA runtime call)."""
import ctypes as C
import os
import re

import pytest

from quantized_weight_streaming_q4k_gb300 import _lib, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qws.h")

OK, NULL, SHAPE, ALIGN, FORMAT, WORKSPACE = 0, 1, 2, 3, 4, 5
A = 0x10000          # a 16-byte-aligned fake device address (never dereferenced)


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.lib()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(qws_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_expected_calls():
    names = declared_functions()
    for n in ["qws_q4k_matvec", "qws_q6k_matvec", "qws_q4_0_matvec", "qws_q4k_qkv_proj",
              "qws_q4k_ffn_gate_up_geglu_down", "qws_rms_norm", "qws_residual_add",
              "qws_decode_chain", "qws_decode_chain_final_norm", "qws_workspace_bytes", "qws_last_error", "qws_device_error",
              "qws_quantize_q8_0", "qws_q8_matvec", "qws_q8_qkv_proj",
              "qws_q4k_prefill_matmul", "qws_rope_at_pos", "qws_kv_append",
              "qws_kv_attention"]:
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing
    # and the Python binding covers them all
    assert set(declared_functions()) <= set(_lib.SIGNATURES)


def test_version(lib):
    assert b"sm_103a" in lib.qws_version()


def _err(lib):
    return lib.qws_last_error().decode()


def test_matvec_null_pointers(lib):
    assert lib.qws_q4k_matvec(None, A, A, 10, 256, 1, None) == NULL
    assert "W is NULL" in _err(lib)
    assert lib.qws_q4k_matvec(A, None, A, 10, 256, 1, None) == NULL
    assert lib.qws_q6k_matvec(A, A, None, 10, 256, 1, None) == NULL


def test_matvec_shapes(lib):
    assert lib.qws_q4k_matvec(A, A, A, -1, 256, 1, None) == SHAPE
    assert lib.qws_q4k_matvec(A, A, A, 10, 0, 1, None) == SHAPE
    assert lib.qws_q4k_matvec(A, A, A, 10, 300, 1, None) == SHAPE
    assert lib.qws_q4_0_matvec(A, A, A, 10, 96, 1, 1, None, 0, None) == SHAPE
    assert lib.qws_q4k_matvec(A, A, A, 10, 256, 0, None) == SHAPE
    assert lib.qws_q4k_matvec(A, A, A, 10, 40960, 1, None) == SHAPE     # one pass <= 20480
    assert lib.qws_q4k_matvec(A, A, A, 10, 2560, 9, None) == SHAPE      # 9 * 40 > 320 lanes
    assert "320" in _err(lib)


def test_q6k_lane_limit(lib):
    # lanes own 64 columns: batch 9 x 2560 columns needs 360 lanes, and a
    # column split of a 10-block Q6_K row (2100 B) is not 16-byte aligned
    assert lib.qws_q6k_matvec(A, A, A, 10, 2560, 9, None) == SHAPE


def test_matvec_alignment(lib):
    assert lib.qws_q4k_matvec(A + 8, A, A, 10, 256, 1, None) == ALIGN
    assert lib.qws_q4k_matvec(A, A + 2, A, 10, 256, 1, None) == ALIGN
    assert lib.qws_q4k_matvec(A, A, A + 1, 10, 256, 1, None) == ALIGN


def test_matvec_format_and_zero_rows(lib):
    assert lib.qws_matvec(7, A, A, A, 10, 256, 1, 1, None, 0, None) == FORMAT
    # zero rows: valid, nothing enqueued (no CUDA call happens)
    assert lib.qws_q4k_matvec(A, A, A, 0, 256, 1, None) == OK


def test_decode_once_batch_has_no_lane_limit(lib):
    # Q4_0 / Q4_K with 2..8 vectors, hidden % 256 == 0 and <= 3072, split_k 0
    # or 1: the decode-once kernel (no 320-lane limit, no workspace); zero
    # rows keep every call launch-free
    assert lib.qws_q4_0_matvec(A, A, A, 0, 3072, 8, 1, None, 0, None) == OK
    assert lib.qws_q4_0_matvec(A, A, A, 0, 3072, 8, 0, None, 0, None) == OK
    assert lib.qws_matvec(12, A, A, A, 0, 3072, 8, 1, None, 0, None) == OK
    # Q6_K has no decode-once kernel: 48 * 8 lanes is refused in one pass
    assert lib.qws_matvec(14, A, A, A, 10, 3072, 8, 1, None, 0, None) == SHAPE
    # nine vectors: the lane-unit engine, where 48 * 9 = 432 lanes do not fit one pass
    assert lib.qws_q4_0_matvec(A, A, A, 10, 3072, 9, 1, None, 0, None) == SHAPE


def test_splitk_workspace_checks(lib):
    need = lib.qws_workspace_bytes(_lib.OP_MATVEC, 1000, 2560, 0, 1, 5)
    assert need >= 5 * 1000 * 4
    assert lib.qws_q4_0_matvec(A, A, A, 1000, 2560, 1, 5, None, 0, None) == WORKSPACE
    assert lib.qws_q4_0_matvec(A, A, A, 1000, 2560, 1, 5, A, need - 1, None) == WORKSPACE
    assert lib.qws_q4_0_matvec(A, A, A, 1000, 2560, 1, 3, A, need, None) == SHAPE   # 3 !| 10
    assert lib.qws_q4_0_matvec(A, A, A, 1000, 2560, 1, -1, A, need, None) == SHAPE
    assert lib.qws_workspace_bytes(_lib.OP_MATVEC, 1000, 2560, 0, 1, 1) == 0
    # large hidden needs a split: library choice picks one that fits 320 lanes
    assert lib.qws_workspace_bytes(_lib.OP_MATVEC, 10, 40960, 0, 1, 0) >= 2 * 10 * 4


def test_qkv_and_ffn_checks(lib):
    assert lib.qws_q4k_qkv_proj(A, A, None, A, A, A, A, 2560, 2048, 1024, None) == NULL
    assert lib.qws_q4k_qkv_proj(A, A, A, A, A, A, A, 2500, 2048, 1024, None) == SHAPE
    assert lib.qws_q4k_qkv_proj(A, A, A, A, A, A, A, 2560, 0, 0, None) == OK
    need = lib.qws_workspace_bytes(_lib.OP_FFN, 0, 2560, 10240, 1, 0)
    assert need >= 10240 * 4
    assert lib.qws_q4k_ffn_gate_up_geglu_down(A, A, A, 2, A, A, 2560, 10240, A, need,
                                              None) == FORMAT
    assert lib.qws_q4k_ffn_gate_up_geglu_down(A, A, A, 14, A, A, 2560, 10240, A, need - 4,
                                              None) == WORKSPACE
    assert lib.qws_q4k_ffn_gate_up_geglu_down(A, A, A, 14, A, A, 2560, 1000, A, need,
                                              None) == SHAPE
    assert lib.qws_q4k_ffn_gate_up_geglu(A, A, A, None, 2560, 10240, None) == NULL


def test_silu_ffn_and_residual_norm_checks(lib):
    need = lib.qws_workspace_bytes(_lib.OP_FFN, 0, 2560, 10240, 1, 0)
    assert lib.qws_q4k_ffn_gate_up_silu_down(A, A, A, 2, A, A, 2560, 10240, A, need, None) == FORMAT
    assert lib.qws_q4k_ffn_gate_up_silu_down(A, A, A, 14, A, A, 2560, 10240, A, need - 4,
                                             None) == WORKSPACE
    assert lib.qws_q4k_ffn_gate_up_silu_down(A, A, A, 14, A, A, 2560, 1000, A, need,
                                             None) == SHAPE
    assert lib.qws_q4k_ffn_gate_up_silu(A, A, A, None, 2560, 10240, None) == NULL
    assert lib.qws_residual_rms_norm(A, A, None, A, 10, C.c_float(1e-6), 1, None) == NULL
    assert lib.qws_residual_rms_norm(A, A, A, A, 0, C.c_float(1e-6), 1, None) == SHAPE
    assert lib.qws_residual_rms_norm(A, A, A, A, 10, C.c_float(-1.0), 1, None) == SHAPE


def test_q8_path_checks(lib):
    Q40, Q80, Q4K = 2, 8, 12
    assert lib.qws_quantize_q8_0(None, A, 64, 1, None) == NULL
    assert lib.qws_quantize_q8_0(A, None, 64, 1, None) == NULL
    assert lib.qws_quantize_q8_0(A, A, 48, 1, None) == SHAPE
    assert lib.qws_quantize_q8_0(A, A, 0, 1, None) == SHAPE
    assert lib.qws_quantize_q8_0(A, A, 64, 0, None) == SHAPE
    assert lib.qws_quantize_q8_0(A + 2, A, 64, 1, None) == ALIGN
    assert lib.qws_quantize_q8_0(A, A + 1, 64, 1, None) == ALIGN
    assert lib.qws_q8_matvec(Q4K, A, A, A, 10, 2560, 1, None) == FORMAT
    assert "Q4_0 or Q8_0" in _err(lib)
    assert lib.qws_q8_matvec(Q40, None, A, A, 10, 2560, 1, None) == NULL
    assert lib.qws_q8_matvec(Q40, A + 4, A, A, 10, 2560, 1, None) == ALIGN
    assert lib.qws_q8_matvec(Q80, A, A + 2, A, 10, 2560, 1, None) == ALIGN
    assert lib.qws_q8_matvec(Q40, A, A, A, 10, 2592, 1, None) == SHAPE      # not % 64
    assert lib.qws_q8_matvec(Q40, A, A, A, 10, 20480 + 64, 1, None) == SHAPE
    assert lib.qws_q8_matvec(Q40, A, A, A, 10, 2560, 9, None) == SHAPE      # 40 * 9 > 320
    assert lib.qws_q8_matvec(Q40, A, A, A, -1, 2560, 1, None) == SHAPE
    assert lib.qws_q8_matvec(Q80, A, A, A, 0, 2560, 8, None) == OK
    # 2..8 vectors at hidden % 256 == 0, <= 3072 take the decode-once kernel,
    # which has no lane limit: 48 * 8 = 384 lanes is accepted there (zero
    # rows: no launch), and refused where the lane-unit engine would run
    assert lib.qws_q8_matvec(Q40, A, A, A, 0, 3072, 8, None) == OK
    assert lib.qws_q8_matvec(Q80, A, A, A, 0, 3072, 8, None) == OK
    assert lib.qws_q8_matvec(Q40, A, A, A, 0, 3072 + 64, 8, None) == SHAPE    # not % 256
    assert lib.qws_q8_matvec(Q40, A, A, A, 0, 3328, 8, None) == SHAPE         # above 3072
    assert lib.qws_q8_matvec(Q40, A, A, A, 0, 1536, 14, None) == SHAPE        # 9+ vectors: 336
    assert lib.qws_q8_qkv_proj(Q40, A, A, None, A, A, A, A, 2560, 2048, 1024, None) == NULL
    assert lib.qws_q8_qkv_proj(Q4K, A, A, A, A, A, A, A, 2560, 2048, 1024, None) == FORMAT
    assert lib.qws_q8_qkv_proj(Q80, A, A, A, A, A, A, A, 2560, 0, 0, None) == OK
    assert lib.qws_rms_norm_q8(A, A, None, 64, C.c_float(1e-6), 1, None) == NULL
    assert lib.qws_rms_norm_q8(A, A, A, 48, C.c_float(1e-6), 1, None) == SHAPE
    assert lib.qws_rms_norm_q8(A, A, A + 1, 64, C.c_float(1e-6), 1, None) == ALIGN
    assert lib.qws_residual_rms_norm_q8(A, None, A, A, 64, C.c_float(1e-6), 1, None) == NULL
    assert lib.qws_residual_rms_norm_q8(A, A, A, A, 64, C.c_float(-1.0), 1, None) == SHAPE
    # the f32-activation entry points do not take Q8_0 weights
    assert lib.qws_matvec(Q80, A, A, A, 10, 2560, 1, 1, None, 0, None) == FORMAT


def test_prefill_checks(lib):
    need = lib.qws_workspace_bytes(_lib.OP_PREFILL, 0, 2560, 0, 512, 0)
    # f16 hi and lo tiles of 256 tokens, then one f32 scale per padded token
    assert need == 512 * 2560 * 2 * 2 + 512 * 4
    assert lib.qws_workspace_bytes(_lib.OP_PREFILL, 0, 2560, 0, 1, 0) == 256 * 2560 * 4 + 256 * 4
    assert lib.qws_workspace_bytes(_lib.OP_PREFILL, 0, 2500, 0, 8, 0) == 0
    assert lib.qws_q4k_prefill_matmul(None, A, A, 10, 2560, 8, A, need, None) == NULL
    assert lib.qws_q4k_prefill_matmul(A, A + 4, A, 10, 2560, 8, A, need, None) == ALIGN
    assert lib.qws_q4k_prefill_matmul(A, A, A, 10, 2500, 8, A, need, None) == SHAPE
    assert lib.qws_q4k_prefill_matmul(A, A, A, 10, 20480 + 256, 8, A, need, None) == SHAPE
    assert lib.qws_q4k_prefill_matmul(A, A, A, 10, 2560, 0, A, need, None) == SHAPE
    assert lib.qws_q4k_prefill_matmul(A, A, A, -1, 2560, 8, A, need, None) == SHAPE
    small = lib.qws_workspace_bytes(_lib.OP_PREFILL, 0, 2560, 0, 8, 0)
    assert lib.qws_q4k_prefill_matmul(A, A, A, 10, 2560, 8, A, small - 16, None) == WORKSPACE
    assert lib.qws_q4k_prefill_matmul(A, A, A, 10, 2560, 8, A + 8, small, None) == ALIGN
    assert lib.qws_q4k_prefill_matmul(A, A, A, 0, 2560, 8, A, small, None) == OK


def test_attention_checks(lib):
    ws = lib.qws_workspace_bytes(_lib.OP_KV_ATTENTION, 4096, 256, 8, 4, 0)
    assert ws > 0
    assert lib.qws_workspace_bytes(_lib.OP_KV_ATTENTION, 4096, 256, 6, 4, 0) == 0
    f, d = C.c_float, C.c_double
    assert lib.qws_rope_at_pos(None, 8, 256, 256, 5, d(1e4), None) == NULL
    assert lib.qws_rope_at_pos(A, 8, 256, 255, 5, d(1e4), None) == SHAPE
    assert lib.qws_rope_at_pos(A, 8, 256, 258, 5, d(1e4), None) == SHAPE
    assert lib.qws_rope_at_pos(A, 2, 1024, 514, 5, d(1e4), None) == SHAPE   # rot_dim > 512
    assert lib.qws_rope_at_pos(A, 8, 256, 256, -1, d(1e4), None) == SHAPE
    assert lib.qws_rope_at_pos(A, 8, 256, 256, 5, d(0.0), None) == SHAPE
    assert lib.qws_kv_append(A, A, A, None, 4, 256, 100, 5, None) == NULL
    assert lib.qws_kv_append(A, A, A, A, 4, 256, 100, 100, None) == SHAPE
    assert lib.qws_kv_attention(A, A, A, A, 8, 4, 200, 4096, 4096, f(0.0625), f(0.0), A, ws,
                                None) == SHAPE
    assert lib.qws_kv_attention(A, A, A, A, 10, 2, 256, 4096, 4096, f(0.0625), f(0.0), A, ws,
                                None) == SHAPE                       # group 5 > 4
    assert lib.qws_kv_attention(A, A, A, A, 8, 4, 256, 4096, 4097, f(0.0625), f(0.0), A, ws,
                                None) == SHAPE
    assert lib.qws_kv_attention(A, A, A, A, 8, 4, 256, 4096, 4096, f(0.0625), f(-1.0), A, ws,
                                None) == SHAPE
    assert lib.qws_kv_attention(A, A, A, A, 8, 4, 256, 4096, 4096, f(0.0625), f(0.0), A, 16,
                                None) == WORKSPACE
    assert lib.qws_kv_attention(A + 4, A, A, A, 8, 4, 256, 4096, 4096, f(0.0625), f(0.0), A, ws,
                                None) == ALIGN


def test_vector_op_checks(lib):
    assert lib.qws_rms_norm(A, None, A, 10, C.c_float(1e-6), 1, None) == NULL
    assert lib.qws_rms_norm(A, A, A, 0, C.c_float(1e-6), 1, None) == SHAPE
    assert lib.qws_rms_norm(A, A, A, 10, C.c_float(-1.0), 1, None) == SHAPE
    assert lib.qws_residual_add(A, A, -1, 1, None) == SHAPE
    assert lib.qws_residual_add(A, A, 0, 1, None) == OK


def test_device_error_null(lib):
    assert lib.qws_device_error(None) == NULL


def test_selftest_wait_timeout_checks_arguments(lib):
    # refused on the host, nothing launched
    assert lib.qws_selftest_wait_timeout(2, 1000, None, None) == SHAPE
    assert lib.qws_selftest_wait_timeout(0, 0, None, None) == SHAPE
    assert lib.qws_selftest_wait_timeout(0, 3_000_000_000, None, None) == SHAPE
    assert lib.qws_selftest_wait_timeout(1, 1000, None, None) == NULL
    assert lib.qws_selftest_wait_timeout(1, 1000, C.c_void_p(0x10004), None) == ALIGN


def _layers(n, **over):
    """n qws_layer structs of fake aligned addresses, Gemma-3 formats (Q4_K,
    Q6_K down); keyword arguments override fields of layer 0."""
    arr = (_lib.QwsLayer * n)()
    for i in range(n):
        L = arr[i]
        for f in ("Wq", "Wk", "Wv", "Wo", "Wg", "Wu", "Wd"):
            setattr(L, f, A)
        L.fmt_qkv = L.fmt_o = L.fmt_gu = 12
        L.fmt_down = 14
        for f in ("w_in", "w_post_attn", "w_pre_ffn", "w_post_ffn"):
            setattr(L, f, A)
    for k, v in over.items():
        setattr(arr[0], k, v)
    return arr


def _dims(**over):
    d = dict(hidden=2560, inter=10240, n_q_heads=8, n_kv_heads=4, head_dim=256, eps=1e-6,
             post_norms=1)
    d.update(over)
    return _lib.QwsDims(d["hidden"], d["inter"], d["n_q_heads"], d["n_kv_heads"],
                        d["head_dim"], d["eps"], d["post_norms"])


def test_decode_chain_checks(lib):
    need = lib.qws_workspace_bytes(_lib.OP_DECODE_CHAIN, 0, 2560, 10240, 1, 0)
    assert need > 0

    def call(layers=None, n=2, h=A, dims=None, ws=A, ws_bytes=need):
        layers = _layers(n) if layers is None else layers
        D = _dims() if dims is None else dims
        return lib.qws_decode_chain(layers, n, h, C.byref(D), ws, ws_bytes, None)

    assert lib.qws_decode_chain(None, 2, A, C.byref(_dims()), A, need, None) == NULL
    assert call(h=None) == NULL
    assert call(ws=None) == NULL
    assert call(n=0) == SHAPE
    assert call(layers=_layers(65), n=65) == SHAPE          # one parameter block: <= 64
    assert call(dims=_dims(n_q_heads=6)) == SHAPE          # 6 % 4 != 0
    assert call(dims=_dims(hidden=2500)) == SHAPE
    assert call(dims=_dims(inter=10000)) == SHAPE
    assert call(dims=_dims(hidden=6144, inter=12288)) == SHAPE   # > 5120
    assert call(dims=_dims(eps=-1.0)) == SHAPE
    assert call(h=A + 2) == ALIGN
    assert call(ws=A + 8) == ALIGN
    assert call(ws_bytes=need - 8) == WORKSPACE
    assert call(layers=_layers(2, Wd=None)) == NULL
    assert call(layers=_layers(2, Wo=A + 8)) == ALIGN
    assert call(layers=_layers(2, w_pre_ffn=None)) == NULL
    assert call(layers=_layers(2, w_post_attn=None)) == NULL     # sandwich norms need it
    assert call(layers=_layers(2, w_in=A + 2)) == ALIGN
    assert call(layers=_layers(2, fmt_qkv=14)) == FORMAT
    assert call(layers=_layers(2, fmt_down=2)) == FORMAT
    assert call(layers=_layers(2, fmt_down=12)) == FORMAT        # differs from layer 1
    # without the post norms their weights may be NULL: the call gets as far
    # as the format check
    assert call(layers=_layers(2, w_post_attn=None, fmt_down=2),
                dims=_dims(post_norms=0)) == FORMAT
    assert b"qws_decode_chain" in lib.qws_last_error()

    def fcall(w_final=A + 0x40000, hn=A + 0x80000, h=A, dims=None, ws_bytes=need):
        D = _dims() if dims is None else dims
        return lib.qws_decode_chain_final_norm(_layers(2), 2, h, w_final, hn, C.byref(D), A,
                                               ws_bytes, None)

    assert fcall(w_final=None) == NULL
    assert fcall(hn=None) == NULL
    assert fcall(hn=A + 0x80002) == ALIGN
    assert fcall(w_final=A + 0x40001) == ALIGN
    assert fcall(hn=A) == SHAPE                       # hn = h
    assert fcall(hn=A + 4 * 2559) == SHAPE            # last element of h
    # adjacent but not overlapping: passes, and the workspace check comes next
    assert fcall(h=A + 4 * 2560, hn=A, ws_bytes=need - 8) == WORKSPACE
    assert fcall(dims=_dims(hidden=2500)) == SHAPE    # the chain's own checks follow
    assert fcall(ws_bytes=need - 8) == WORKSPACE
    assert b"qws_decode_chain_final_norm" in lib.qws_last_error()


def test_decode_kv_checks(lib):
    D0 = _dims()
    need = lib.qws_decode_kv_workspace_bytes(C.byref(D0), 2048)
    assert need > 0
    caches = (C.c_void_p * 2)(A, A)

    def kv(**over):
        k = dict(k_caches=C.cast(caches, C.c_void_p), v_caches=C.cast(caches, C.c_void_p),
                 max_seq=2048, pos=1024, rot_dim=256, rope_base=1e6, attn_scale=0.0625,
                 softcap=0.0)
        k.update(over)
        return _lib.QwsKv(k["k_caches"], k["v_caches"], k["max_seq"], k["pos"], k["rot_dim"],
                          k["rope_base"], k["attn_scale"], k["softcap"])

    def call(layers=None, n=2, h=A, dims=None, K=None, ws=A, ws_bytes=need):
        layers = _layers(n) if layers is None else layers
        D = _dims() if dims is None else dims
        K = kv() if K is None else K
        return lib.qws_decode_kv(layers, n, h, C.byref(D), C.byref(K), ws, ws_bytes, None)

    assert lib.qws_decode_kv(_layers(2), 2, A, C.byref(D0), None, A, need, None) == NULL
    assert call(h=None) == NULL
    assert call(n=0) == SHAPE
    assert call(dims=_dims(n_q_heads=8, n_kv_heads=1)) == SHAPE    # group of 8 > 4
    assert call(dims=_dims(n_q_heads=6)) == SHAPE
    assert call(dims=_dims(head_dim=96, n_q_heads=8, n_kv_heads=8, hidden=768,
                           inter=2048)) == SHAPE
    assert call(dims=_dims(inter=1000)) == SHAPE
    assert call(dims=_dims(eps=-1.0)) == SHAPE
    assert call(K=kv(k_caches=None)) == NULL
    assert call(K=kv(pos=2048)) == SHAPE
    assert call(K=kv(pos=-1)) == SHAPE
    assert call(K=kv(max_seq=0, pos=0)) == SHAPE
    assert call(K=kv(rot_dim=255)) == SHAPE
    assert call(K=kv(rot_dim=512)) == SHAPE
    assert call(K=kv(rot_dim=0)) == SHAPE
    assert call(K=kv(rope_base=0.0)) == SHAPE
    assert call(K=kv(attn_scale=float("inf"))) == SHAPE
    assert call(K=kv(softcap=-1.0)) == SHAPE
    assert call(h=A + 4) == ALIGN
    assert call(ws=A + 8) == ALIGN
    assert call(ws_bytes=need - 8) == WORKSPACE
    assert call(layers=_layers(2, Wk=None)) == NULL
    assert call(layers=_layers(2, Wg=A + 4)) == ALIGN
    assert call(layers=_layers(2, w_in=None)) == NULL
    assert call(layers=_layers(2, fmt_o=2)) == FORMAT
    bad = (C.c_void_p * 2)(None, A)
    assert call(K=kv(v_caches=C.cast(bad, C.c_void_p))) == NULL
    mis = (C.c_void_p * 2)(A + 4, A)
    assert call(K=kv(k_caches=C.cast(mis, C.c_void_p))) == ALIGN
    assert b"qws_decode_kv" in lib.qws_last_error()
