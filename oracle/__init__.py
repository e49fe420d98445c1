"""f64 CPU oracle for the quantized weight-streaming decode path.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  It shares no code
with the CUDA library and never imports it.

The arithmetic lives in ``oracle.c`` (plain C, every value in f64, sums in
index order); this module only marshals numpy arrays through ctypes.  The
shared object is compiled on first use with gcc (``build()``); the build flags
keep IEEE f64 semantics (no fast-math, no FMA contraction).
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

Q4_0, Q8_0, Q4_K, Q6_K = 2, 8, 12, 14
BLOCK_WEIGHTS = {Q4_0: 32, Q8_0: 32, Q4_K: 256, Q6_K: 256}
BLOCK_BYTES = {Q4_0: 18, Q8_0: 34, Q4_K: 144, Q6_K: 210}

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (gcc, no fast-math)."""
    if force or not os.path.exists(_LIB_PATH) or (
        os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)
    ):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-D_DEFAULT_SOURCE", "-fPIC", "-shared",
             "-ffp-contract=off", "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
        )
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Layer(C.Structure):
    _fields_ = [
        ("fmt_qkv", C.c_int), ("fmt_o", C.c_int), ("fmt_gu", C.c_int), ("fmt_down", C.c_int),
        ("Wq", C.c_void_p), ("Wk", C.c_void_p), ("Wv", C.c_void_p), ("Wo", C.c_void_p),
        ("Wg", C.c_void_p), ("Wu", C.c_void_p), ("Wd", C.c_void_p),
        ("w_in", C.c_void_p), ("w_post_attn", C.c_void_p), ("w_pre_ffn", C.c_void_p),
        ("w_post_ffn", C.c_void_p),
    ]


class _Dims(C.Structure):
    _fields_ = [
        ("hidden", C.c_int64), ("inter", C.c_int64),
        ("n_q_heads", C.c_int), ("n_kv_heads", C.c_int), ("head_dim", C.c_int),
        ("eps", C.c_double), ("post_norms", C.c_int),
    ]


_TRACE_FIELDS = ["n1", "q", "k", "v", "attn", "o", "h1", "n2", "g", "u", "m", "f", "bound_f"]


class _Trace(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in _TRACE_FIELDS]


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = C.CDLL(build())
        P, I64, I = C.c_void_p, C.c_int64, C.c_int
        lib.qo_half.restype = C.c_double
        lib.qo_half.argtypes = [C.c_uint16]
        lib.qo_rope.restype = I
        lib.qo_rope.argtypes = [P, I, I, I, I64, C.c_double]
        lib.qo_kv_append.restype = I
        lib.qo_kv_append.argtypes = [P, P, P, P, I, I, I64, I64]
        lib.qo_kv_attention.restype = I
        lib.qo_kv_attention.argtypes = [P, P, P, I, I, I, I64, I64, C.c_double, C.c_double,
                                        P, P, P]
        lib.qo_half_bits.restype = C.c_uint16
        lib.qo_half_bits.argtypes = [C.c_float]
        lib.qo_quantize_q8_0.restype = I
        lib.qo_quantize_q8_0.argtypes = [P, I64, P]
        lib.qo_matvec_q8.restype = I
        lib.qo_matvec_q8.argtypes = [I, P, I64, I64, P, I, I64, I64, P, P]
        for name in ("qo_dequant_q4_0", "qo_dequant_q8_0", "qo_dequant_q4_k",
                     "qo_dequant_q6_k"):
            getattr(lib, name).restype = None
            getattr(lib, name).argtypes = [P, P]
        lib.qo_q4_k_scale_min.restype = None
        lib.qo_q4_k_scale_min.argtypes = [P, I, P, P]
        lib.qo_dequant_rows.restype = I
        lib.qo_dequant_rows.argtypes = [I, P, I64, I64, P]
        lib.qo_matvec.restype = I
        lib.qo_matvec.argtypes = [I, P, I64, I64, P, I, I64, I64, P, P]
        lib.qo_gelu_tanh.restype = C.c_double
        lib.qo_gelu_tanh.argtypes = [C.c_double]
        lib.qo_rms_norm.restype = None
        lib.qo_rms_norm.argtypes = [P, P, I64, C.c_double, P]
        lib.qo_residual_add.restype = None
        lib.qo_residual_add.argtypes = [P, P, I64]
        lib.qo_attn_seq1.restype = I
        lib.qo_attn_seq1.argtypes = [P, I, I, I, P]
        lib.qo_ffn.restype = I
        lib.qo_ffn.argtypes = [I, P, P, I, P, I64, I64, P, P, P, P, P, P]
        lib.qo_ffn_act.restype = I
        lib.qo_ffn_act.argtypes = [I, I, P, P, I, P, I64, I64, P, P, P, P, P, P]
        lib.qo_silu.restype = C.c_double
        lib.qo_silu.argtypes = [C.c_double]
        lib.qo_residual_rms_norm.restype = None
        lib.qo_residual_rms_norm.argtypes = [P, P, P, I64, C.c_double, P]
        lib.qo_layer_forward.restype = I
        lib.qo_layer_forward.argtypes = [C.POINTER(_Layer), C.POINTER(_Dims), P, P,
                                         C.POINTER(_Trace)]
        lib.qo_topk.restype = I
        lib.qo_topk.argtypes = [P, I64, I, P]
        _lib = lib
        return lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _u8(W) -> np.ndarray:
    a = np.ascontiguousarray(np.asarray(W), dtype=np.uint8).reshape(-1)
    return a


def _f64(x) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def half(bits: int) -> float:
    """binary16 bit pattern -> value (f64)."""
    return _load().qo_half(int(bits) & 0xFFFF)


def dequant_block(fmt: int, blk) -> np.ndarray:
    b = _u8(blk)
    assert b.size == BLOCK_BYTES[fmt]
    out = np.empty(BLOCK_WEIGHTS[fmt], dtype=np.float64)
    name = {Q4_0: "qo_dequant_q4_0", Q8_0: "qo_dequant_q8_0", Q4_K: "qo_dequant_q4_k",
            Q6_K: "qo_dequant_q6_k"}[fmt]
    getattr(_load(), name)(_ptr(b), _ptr(out))
    return out


def q4_k_scale_min(sc12, s: int) -> tuple[int, int]:
    b = _u8(sc12)
    assert b.size == 12
    a, m = C.c_int(), C.c_int()
    _load().qo_q4_k_scale_min(_ptr(b), int(s), C.addressof(a), C.addressof(m))
    return a.value, m.value


def dequant(fmt: int, W, rows: int, hidden: int) -> np.ndarray:
    """Dense f64 [rows, hidden] copy of a quantized row-major matrix."""
    w = _u8(W)
    assert w.size == rows * (hidden // BLOCK_WEIGHTS[fmt]) * BLOCK_BYTES[fmt]
    out = np.empty((rows, hidden), dtype=np.float64)
    rc = _load().qo_dequant_rows(fmt, _ptr(w), rows, hidden, _ptr(out))
    if rc:
        raise ValueError(f"qo_dequant_rows failed ({rc})")
    return out


def matvec(fmt: int, W, rows: int, hidden: int, x, threads: int = 1,
           row_begin: int = 0, row_end: int | None = None):
    """y[b, r] = sum_i w[r, i] x[b, i] and bound[b, r] = sum_i |w x| (f64).

    ``x`` is [hidden] or [batch, hidden].  Rows are split across ``threads``
    host threads; every row is still computed by the same plain loop.
    Only rows in [row_begin, row_end) are computed; the rest of y/bound is NaN.
    """
    w = _u8(W)
    assert w.size == rows * (hidden // BLOCK_WEIGHTS[fmt]) * BLOCK_BYTES[fmt]
    xs = _f64(x)
    squeeze = xs.ndim == 1
    xs = xs.reshape(-1, hidden)
    batch = xs.shape[0]
    row_end = rows if row_end is None else row_end
    y = np.full((batch, rows), np.nan)
    bound = np.full((batch, rows), np.nan)
    lib = _load()

    def run(a: int, b: int) -> int:
        return lib.qo_matvec(fmt, _ptr(w), rows, hidden, _ptr(xs), batch, a, b,
                             _ptr(y), _ptr(bound))

    n = row_end - row_begin
    threads = max(1, min(int(threads), n if n > 0 else 1))
    if threads == 1:
        rcs = [run(row_begin, row_end)]
    else:
        edges = [row_begin + (n * t) // threads for t in range(threads + 1)]
        with ThreadPoolExecutor(threads) as ex:
            rcs = list(ex.map(lambda t: run(edges[t], edges[t + 1]), range(threads)))
    if any(rcs):
        raise ValueError(f"qo_matvec failed ({rcs})")
    if squeeze:
        return y[0], bound[0]
    return y, bound


def half_bits(f) -> int:
    """f32 value -> binary16 bit pattern (nearest, ties to even)."""
    return int(_load().qo_half_bits(float(np.float32(f))))


def quantize_q8_0(x) -> np.ndarray:
    """f32 activations [..., n] (n % 32 == 0) -> Q8_0 blocks, uint8
    [..., n / 32 * 34]; the decisions are taken in f32."""
    xs = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    n = xs.shape[-1]
    out = np.empty(xs.shape[:-1] + (n // 32 * 34,), dtype=np.uint8)
    rc = _load().qo_quantize_q8_0(_ptr(xs), xs.size, _ptr(out))
    if rc or n % 32:
        raise ValueError(f"qo_quantize_q8_0 failed ({rc})")
    return out


def rms_norm_q8(x, w, eps: float) -> np.ndarray:
    """rms_norm_q8 ([compute] §Shaders "Fused ops"): the f64 rms_norm of each
    row of x, rounded to f32 (the activation type), then quantize_q8_0."""
    xs = _f64(x)
    rows = xs.reshape(-1, xs.shape[-1])
    y = np.stack([rms_norm(r, w, eps) for r in rows]).astype(np.float32)
    return quantize_q8_0(y.reshape(xs.shape))


def residual_rms_norm_q8(h, y, w, eps: float):
    """residual_norm_q8: h + y (f64), then rms_norm_q8 of the sum.  Returns
    (h + y, blocks)."""
    hs = _f64(h) + _f64(y)
    return hs, rms_norm_q8(hs, w, eps)


def matvec_q8(wfmt: int, W, rows: int, hidden: int, xq, threads: int = 1,
              row_begin: int = 0, row_end: int | None = None):
    """Q4_0 / Q8_0 weights times Q8_0 activations ``xq`` ([hidden / 32 * 34]
    or [batch, hidden / 32 * 34] bytes): y[b, r] and bound[b, r] in f64.
    Rows outside [row_begin, row_end) are NaN."""
    w = _u8(W)
    assert w.size == rows * (hidden // 32) * BLOCK_BYTES[wfmt]
    xb = np.ascontiguousarray(np.asarray(xq, dtype=np.uint8))
    squeeze = xb.ndim == 1
    xb = xb.reshape(-1, hidden // 32 * 34)
    batch = xb.shape[0]
    row_end = rows if row_end is None else row_end
    y = np.full((batch, rows), np.nan)
    bound = np.full((batch, rows), np.nan)
    lib = _load()

    def run(a: int, b: int) -> int:
        return lib.qo_matvec_q8(wfmt, _ptr(w), rows, hidden, _ptr(xb), batch, a, b,
                                _ptr(y), _ptr(bound))

    n = row_end - row_begin
    threads = max(1, min(int(threads), n if n > 0 else 1))
    if threads == 1:
        rcs = [run(row_begin, row_end)]
    else:
        edges = [row_begin + (n * t) // threads for t in range(threads + 1)]
        with ThreadPoolExecutor(threads) as ex:
            rcs = list(ex.map(lambda t: run(edges[t], edges[t + 1]), range(threads)))
    if any(rcs):
        raise ValueError(f"qo_matvec_q8 failed ({rcs})")
    if squeeze:
        return y[0], bound[0]
    return y, bound


def gelu_tanh(t):
    lib = _load()
    arr = np.asarray(t, dtype=np.float64)
    out = np.array([lib.qo_gelu_tanh(float(v)) for v in arr.reshape(-1)], dtype=np.float64)
    return out.reshape(arr.shape) if arr.ndim else float(out[0])


def rms_norm(x, w, eps: float) -> np.ndarray:
    xs, ws = _f64(x).reshape(-1), _f64(w).reshape(-1)
    assert xs.size == ws.size
    out = np.empty_like(xs)
    _load().qo_rms_norm(_ptr(xs), _ptr(ws), xs.size, float(eps), _ptr(out))
    return out


def residual_add(h, y) -> np.ndarray:
    hs = _f64(h).reshape(-1).copy()
    ys = _f64(y).reshape(-1)
    assert hs.size == ys.size
    _load().qo_residual_add(_ptr(hs), _ptr(ys), hs.size)
    return hs


def attn_seq1(v, n_q_heads: int, n_kv_heads: int, head_dim: int) -> np.ndarray:
    vs = _f64(v).reshape(-1)
    assert vs.size == n_kv_heads * head_dim
    out = np.empty(n_q_heads * head_dim)
    rc = _load().qo_attn_seq1(_ptr(vs), n_q_heads, n_kv_heads, head_dim, _ptr(out))
    if rc:
        raise ValueError("bad head counts")
    return out


def rope(x, n_heads: int, head_dim: int, rot_dim: int, pos: int, base: float) -> np.ndarray:
    """Rotary embedding of [n_heads, head_dim] at position pos (half-split pairs)."""
    xs = _f64(x).reshape(-1).copy()
    assert xs.size == n_heads * head_dim
    rc = _load().qo_rope(_ptr(xs), n_heads, head_dim, rot_dim, int(pos), float(base))
    if rc:
        raise ValueError("bad rope arguments")
    return xs.reshape(n_heads, head_dim)


def kv_append(kc, vc, k, v, n_kv_heads: int, head_dim: int, max_seq: int, pos: int):
    """Returns copies of the caches with k, v written at position pos."""
    kc2, vc2 = _f64(kc).reshape(-1).copy(), _f64(vc).reshape(-1).copy()
    ks, vs = _f64(k).reshape(-1), _f64(v).reshape(-1)
    rc = _load().qo_kv_append(_ptr(kc2), _ptr(vc2), _ptr(ks), _ptr(vs), n_kv_heads, head_dim,
                              max_seq, int(pos))
    if rc:
        raise ValueError("bad position")
    shape = (n_kv_heads, max_seq, head_dim)
    return kc2.reshape(shape), vc2.reshape(shape)


def kv_attention(q, kc, vc, n_q_heads: int, n_kv_heads: int, head_dim: int, max_seq: int,
                 n_ctx: int, scale: float, softcap: float = 0.0):
    """One query token over the first n_ctx cache positions.  Returns
    (out, bound, smax): out and bound [n_q, hd], smax [n_q]."""
    qs = _f64(q).reshape(-1)
    ks, vs = _f64(kc).reshape(-1), _f64(vc).reshape(-1)
    assert qs.size == n_q_heads * head_dim and ks.size == n_kv_heads * max_seq * head_dim
    out = np.empty(n_q_heads * head_dim)
    bound = np.empty(n_q_heads * head_dim)
    smax = np.empty(n_q_heads)
    rc = _load().qo_kv_attention(_ptr(qs), _ptr(ks), _ptr(vs), n_q_heads, n_kv_heads, head_dim,
                                 max_seq, int(n_ctx), float(scale), float(softcap), _ptr(out),
                                 _ptr(bound), _ptr(smax))
    if rc:
        raise ValueError(f"qo_kv_attention failed ({rc})")
    return out.reshape(n_q_heads, head_dim), bound.reshape(n_q_heads, head_dim), smax


ACT_GELU_TANH, ACT_SILU = 0, 1


def silu(t):
    lib = _load()
    arr = np.asarray(t, dtype=np.float64)
    out = np.array([lib.qo_silu(float(v)) for v in arr.reshape(-1)], dtype=np.float64)
    return out.reshape(arr.shape) if arr.ndim else float(out[0])


def residual_rms_norm(h, y, w, eps: float):
    """h + y and rms_norm(h + y, w): returns (h_new, x)."""
    hs = _f64(h).reshape(-1).copy()
    ys, ws = _f64(y).reshape(-1), _f64(w).reshape(-1)
    assert hs.size == ys.size == ws.size
    x = np.empty_like(hs)
    _load().qo_residual_rms_norm(_ptr(hs), _ptr(ys), _ptr(ws), hs.size, float(eps), _ptr(x))
    return hs, x


def ffn(fmt_gu: int, Wg, Wu, fmt_d: int, Wd, hidden: int, inter: int, x,
        act: int = ACT_GELU_TANH) -> dict:
    """Gated FFN; returns dict with g, u, m (= act(g) u), y and bound_y."""
    wg, wu, wd = _u8(Wg), _u8(Wu), _u8(Wd)
    xs = _f64(x).reshape(-1)
    assert xs.size == hidden
    out = {k: np.empty(inter) for k in ("g", "u", "m")}
    out["y"] = np.empty(hidden)
    out["bound_y"] = np.empty(hidden)
    rc = _load().qo_ffn_act(act, fmt_gu, _ptr(wg), _ptr(wu), fmt_d, _ptr(wd), hidden, inter,
                            _ptr(xs), _ptr(out["g"]), _ptr(out["u"]), _ptr(out["m"]),
                            _ptr(out["y"]), _ptr(out["bound_y"]))
    if rc:
        raise ValueError(f"qo_ffn failed ({rc})")
    return out


def layer_forward(layer: dict, dims: dict, h, trace: bool = False):
    """One decoder layer (see qo_layer_forward in oracle.c).

    ``layer`` holds numpy arrays: Wq, Wk, Wv, Wo, Wg, Wu, Wd (uint8 blocks),
    w_in, w_post_attn, w_pre_ffn, w_post_ffn (float arrays) and the formats
    fmt_qkv, fmt_o, fmt_gu, fmt_down.  ``dims`` holds hidden, inter, n_q_heads,
    n_kv_heads, head_dim, eps and post_norms.  Returns h_out, or
    (h_out, trace_dict) when ``trace`` is true.
    """
    keep = []

    def u8(a):
        a = _u8(a)
        keep.append(a)
        return _ptr(a)

    def f64(a):
        a = _f64(a).reshape(-1)
        keep.append(a)
        return _ptr(a)

    L = _Layer(layer["fmt_qkv"], layer["fmt_o"], layer["fmt_gu"], layer["fmt_down"],
               u8(layer["Wq"]), u8(layer["Wk"]), u8(layer["Wv"]), u8(layer["Wo"]),
               u8(layer["Wg"]), u8(layer["Wu"]), u8(layer["Wd"]),
               f64(layer["w_in"]), f64(layer["w_post_attn"]), f64(layer["w_pre_ffn"]),
               f64(layer["w_post_ffn"]))
    D = _Dims(dims["hidden"], dims["inter"], dims["n_q_heads"], dims["n_kv_heads"],
              dims["head_dim"], float(dims["eps"]), int(dims["post_norms"]))
    H, I = dims["hidden"], dims["inter"]
    qd = dims["n_q_heads"] * dims["head_dim"]
    kd = dims["n_kv_heads"] * dims["head_dim"]
    hs = _f64(h).reshape(-1)
    assert hs.size == H
    out = np.empty(H)
    tr = None
    tptr = None
    if trace:
        sizes = dict(n1=H, q=qd, k=kd, v=kd, attn=qd, o=H, h1=H, n2=H, g=I, u=I, m=I, f=H,
                     bound_f=H)
        tr = {k: np.empty(sizes[k]) for k in _TRACE_FIELDS}
        T = _Trace(*[_ptr(tr[k]) for k in _TRACE_FIELDS])
        tptr = C.pointer(T)
    rc = _load().qo_layer_forward(C.pointer(L), C.pointer(D), _ptr(hs), _ptr(out), tptr)
    if rc:
        raise ValueError(f"qo_layer_forward failed ({rc})")
    return (out, tr) if trace else out


class _KV(C.Structure):
    _fields_ = [("k_cache", C.c_void_p), ("v_cache", C.c_void_p), ("max_seq", C.c_int64),
                ("pos", C.c_int64), ("rot_dim", C.c_int), ("rope_base", C.c_double),
                ("scale", C.c_double), ("softcap", C.c_double)]


def layer_forward_kv(layer: dict, dims: dict, kv: dict, h, trace: bool = False):
    """One decoder layer at position kv["pos"] with a KV cache (see
    qo_layer_forward_kv in oracle.c).  ``kv`` holds k_cache and v_cache (f64
    arrays [n_kv_heads, max_seq, head_dim], updated in place at pos), max_seq,
    pos, rot_dim, rope_base, scale and softcap.  Returns h_out, or
    (h_out, trace_dict) when ``trace`` is true (q and k after the rotation)."""
    keep = []

    def u8(a):
        a = _u8(a)
        keep.append(a)
        return _ptr(a)

    def f64(a):
        a = _f64(a).reshape(-1)
        keep.append(a)
        return _ptr(a)

    for name in ("k_cache", "v_cache"):
        arr = kv[name]
        if not (isinstance(arr, np.ndarray) and arr.dtype == np.float64 and arr.flags.c_contiguous):
            raise TypeError(f"kv[{name!r}] must be a C-contiguous float64 array (updated in place)")
    L = _Layer(layer["fmt_qkv"], layer["fmt_o"], layer["fmt_gu"], layer["fmt_down"],
               u8(layer["Wq"]), u8(layer["Wk"]), u8(layer["Wv"]), u8(layer["Wo"]),
               u8(layer["Wg"]), u8(layer["Wu"]), u8(layer["Wd"]),
               f64(layer["w_in"]), f64(layer["w_post_attn"]), f64(layer["w_pre_ffn"]),
               f64(layer["w_post_ffn"]))
    D = _Dims(dims["hidden"], dims["inter"], dims["n_q_heads"], dims["n_kv_heads"],
              dims["head_dim"], float(dims["eps"]), int(dims["post_norms"]))
    K = _KV(_ptr(kv["k_cache"]), _ptr(kv["v_cache"]), int(kv["max_seq"]), int(kv["pos"]),
            int(kv["rot_dim"]), float(kv["rope_base"]), float(kv["scale"]),
            float(kv.get("softcap", 0.0)))
    H, I = dims["hidden"], dims["inter"]
    qd = dims["n_q_heads"] * dims["head_dim"]
    kd = dims["n_kv_heads"] * dims["head_dim"]
    assert kv["k_cache"].size == dims["n_kv_heads"] * int(kv["max_seq"]) * dims["head_dim"]
    assert kv["v_cache"].size == kv["k_cache"].size
    hs = _f64(h).reshape(-1)
    assert hs.size == H
    out = np.empty(H)
    tr = None
    tptr = None
    if trace:
        sizes = dict(n1=H, q=qd, k=kd, v=kd, attn=qd, o=H, h1=H, n2=H, g=I, u=I, m=I, f=H,
                     bound_f=H)
        tr = {k: np.empty(sizes[k]) for k in _TRACE_FIELDS}
        T = _Trace(*[_ptr(tr[k]) for k in _TRACE_FIELDS])
        tptr = C.pointer(T)
    rc = _load().qo_layer_forward_kv(C.pointer(L), C.pointer(D), C.pointer(K), _ptr(hs),
                                     _ptr(out), tptr)
    if rc:
        raise ValueError(f"qo_layer_forward_kv failed ({rc})")
    return (out, tr) if trace else out


def topk(v, k: int) -> np.ndarray:
    vs = _f64(v).reshape(-1)
    idx = np.empty(k, dtype=np.int64)
    rc = _load().qo_topk(_ptr(vs), vs.size, int(k), _ptr(idx))
    if rc:
        raise ValueError("bad k")
    return idx
