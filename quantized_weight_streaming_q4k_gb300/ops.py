"""Thin torch-facing binding over the C ABI (include/qws.h).

Argument marshalling only: every function passes device pointers, sizes and
the current CUDA stream to libqws.so; all arithmetic runs in its kernels.
Outputs are allocated with torch when ``out`` is not given (PyTorch is the
allocator, the library allocates nothing).
"""
from __future__ import annotations

import ctypes as C

import torch

from . import _lib
from ._lib import (OP_DECODE_CHAIN, OP_FFN, OP_KV_ATTENTION, OP_MATVEC, OP_PREFILL, Q4_0,
                   Q4_K, Q6_K, Q8_0,
                   QwsError, check, lib)

__all__ = [
    "Q4_0", "Q4_K", "Q6_K", "Q8_0", "QwsError", "q4k_matvec", "q6k_matvec", "q4_0_matvec",
    "matvec", "quantize_q8_0", "q8_matvec", "q8_qkv_proj", "q4k_prefill_matmul",
    "rope_at_pos", "kv_append", "kv_attention", "rms_norm_q8", "residual_rms_norm_q8",
    "q4k_qkv_proj", "q4k_ffn_gate_up_geglu", "q4k_ffn_gate_up_geglu_down", "rms_norm",
    "residual_add", "decode_chain", "decode_kv", "decode_kv_workspace_bytes", "workspace_bytes",
    "device_error", "Layer", "Dims",
    "stream_handle",
]


def stream_handle(stream: torch.cuda.Stream | None = None) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _dev(t: torch.Tensor, name: str, dtype: torch.dtype | None = None) -> int:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _out(out, shape, like: torch.Tensor) -> torch.Tensor:
    if out is None:
        return torch.empty(shape, dtype=torch.float32, device=like.device)
    return out


def workspace_bytes(op: int, rows: int = 0, hidden: int = 0, inter: int = 0, batch: int = 1,
                    split_k: int = 0) -> int:
    return int(lib().qws_workspace_bytes(op, rows, hidden, inter, batch, split_k))


def _mv(name: str, W, x, rows: int, hidden: int, batch: int, out, stream):
    y = _out(out, (batch, rows) if batch > 1 else (rows,), x)
    fn = getattr(lib(), name)
    check(fn(_dev(W, "W", torch.uint8), _dev(x, "x", torch.float32),
             _dev(y, "y", torch.float32), rows, hidden, batch, stream_handle(stream)))
    return y


def q4k_matvec(W, x, rows: int, hidden: int, batch: int = 1, out=None, stream=None):
    """y = dequant_Q4_K(W) @ x; x [batch, hidden] (or [hidden]), y [batch, rows]."""
    return _mv("qws_q4k_matvec", W, x, rows, hidden, batch, out, stream)


def q6k_matvec(W, x, rows: int, hidden: int, batch: int = 1, out=None, stream=None):
    return _mv("qws_q6k_matvec", W, x, rows, hidden, batch, out, stream)


def matvec(fmt: int, W, x, rows: int, hidden: int, batch: int = 1, split_k: int = 1,
           workspace=None, out=None, stream=None):
    y = _out(out, (batch, rows) if batch > 1 else (rows,), x)
    ws_ptr, ws_bytes = (0, 0) if workspace is None else (_dev(workspace, "workspace"),
                                                          workspace.numel() * workspace.element_size())
    check(lib().qws_matvec(fmt, _dev(W, "W", torch.uint8), _dev(x, "x", torch.float32),
                           _dev(y, "y", torch.float32), rows, hidden, batch, split_k,
                           ws_ptr or None, ws_bytes, stream_handle(stream)))
    return y


def q4_0_matvec(W, x, rows: int, hidden: int, batch: int = 1, split_k: int = 1, workspace=None,
                out=None, stream=None):
    y = _out(out, (batch, rows) if batch > 1 else (rows,), x)
    ws_ptr, ws_bytes = (0, 0) if workspace is None else (_dev(workspace, "workspace"),
                                                          workspace.numel() * workspace.element_size())
    check(lib().qws_q4_0_matvec(_dev(W, "W", torch.uint8), _dev(x, "x", torch.float32),
                                _dev(y, "y", torch.float32), rows, hidden, batch, split_k,
                                ws_ptr or None, ws_bytes, stream_handle(stream)))
    return y


def q4k_qkv_proj(Wq, Wk, Wv, x, hidden: int, q_dim: int, kv_dim: int, out=None, stream=None):
    if out is None:
        q = torch.empty(q_dim, dtype=torch.float32, device=x.device)
        k = torch.empty(kv_dim, dtype=torch.float32, device=x.device)
        v = torch.empty(kv_dim, dtype=torch.float32, device=x.device)
    else:
        q, k, v = out
    check(lib().qws_q4k_qkv_proj(_dev(Wq, "Wq", torch.uint8), _dev(Wk, "Wk", torch.uint8),
                                 _dev(Wv, "Wv", torch.uint8), _dev(x, "x", torch.float32),
                                 _dev(q, "q", torch.float32), _dev(k, "k", torch.float32),
                                 _dev(v, "v", torch.float32), hidden, q_dim, kv_dim,
                                 stream_handle(stream)))
    return q, k, v


def quantize_q8_0(x, n: int, batch: int = 1, out=None, stream=None):
    """x [batch, n] (or [n]) f32 -> Q8_0 blocks, uint8 [batch, n / 32 * 34] (or flat)."""
    nbytes = n // 32 * 34
    if out is None:
        out = torch.empty((batch, nbytes) if batch > 1 else (nbytes,), dtype=torch.uint8,
                          device=x.device)
    check(lib().qws_quantize_q8_0(_dev(x, "x", torch.float32), _dev(out, "xq", torch.uint8), n,
                                  batch, stream_handle(stream)))
    return out


def _xq_out(out, n: int, batch: int, like):
    if out is not None:
        return out
    nbytes = n // 32 * 34
    return torch.empty((batch, nbytes) if batch > 1 else (nbytes,), dtype=torch.uint8,
                       device=like.device)


def rms_norm_q8(x, w, eps: float, n: int, batch: int = 1, out=None, stream=None):
    """Q8_0 blocks of rms_norm(x, w) ([batch, n] or [n] f32 -> uint8 [.., n / 32 * 34])."""
    xq = _xq_out(out, n, batch, x)
    check(lib().qws_rms_norm_q8(_dev(x, "x", torch.float32), _dev(w, "w", torch.float32),
                                _dev(xq, "xq", torch.uint8), n, eps, batch,
                                stream_handle(stream)))
    return xq


def residual_rms_norm_q8(h, y, w, eps: float, n: int, batch: int = 1, out=None, stream=None):
    """h += y (in place), then the Q8_0 blocks of rms_norm(h, w)."""
    xq = _xq_out(out, n, batch, h)
    check(lib().qws_residual_rms_norm_q8(_dev(h, "h", torch.float32), _dev(y, "y", torch.float32),
                                         _dev(w, "w", torch.float32), _dev(xq, "xq", torch.uint8),
                                         n, eps, batch, stream_handle(stream)))
    return xq


def q8_matvec(wfmt: int, W, xq, rows: int, hidden: int, batch: int = 1, out=None, stream=None):
    """y = W @ xq for Q4_0 / Q8_0 weights and Q8_0 activations xq."""
    y = _out(out, (batch, rows) if batch > 1 else (rows,), xq)
    check(lib().qws_q8_matvec(wfmt, _dev(W, "W", torch.uint8), _dev(xq, "xq", torch.uint8),
                              _dev(y, "y", torch.float32), rows, hidden, batch,
                              stream_handle(stream)))
    return y


def q8_qkv_proj(wfmt: int, Wq, Wk, Wv, xq, hidden: int, q_dim: int, kv_dim: int, out=None,
                stream=None):
    if out is None:
        q = torch.empty(q_dim, dtype=torch.float32, device=xq.device)
        k = torch.empty(kv_dim, dtype=torch.float32, device=xq.device)
        v = torch.empty(kv_dim, dtype=torch.float32, device=xq.device)
    else:
        q, k, v = out
    check(lib().qws_q8_qkv_proj(wfmt, _dev(Wq, "Wq", torch.uint8), _dev(Wk, "Wk", torch.uint8),
                                _dev(Wv, "Wv", torch.uint8), _dev(xq, "xq", torch.uint8),
                                _dev(q, "q", torch.float32), _dev(k, "k", torch.float32),
                                _dev(v, "v", torch.float32), hidden, q_dim, kv_dim,
                                stream_handle(stream)))
    return q, k, v


def q4k_prefill_matmul(W, X, rows: int, hidden: int, n_tokens: int, workspace=None, out=None,
                       stream=None):
    """Y [n_tokens, rows] = X [n_tokens, hidden] @ dequant_Q4_K(W)^T on the tensor cores
    (f16 operands, f32 accumulation)."""
    Y = _out(out, (n_tokens, rows), X)
    need = workspace_bytes(OP_PREFILL, 0, hidden, 0, n_tokens, 0)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=X.device)
    check(lib().qws_q4k_prefill_matmul(
        _dev(W, "W", torch.uint8), _dev(X, "X", torch.float32), _dev(Y, "Y", torch.float32),
        rows, hidden, n_tokens, _dev(workspace, "workspace"),
        workspace.numel() * workspace.element_size(), stream_handle(stream)))
    return Y


def rope_at_pos(x, n_heads: int, head_dim: int, rot_dim: int, pos: int, base: float,
                stream=None):
    """Rotates x [n_heads, head_dim] in place at position pos; returns x."""
    check(lib().qws_rope_at_pos(_dev(x, "x", torch.float32), n_heads, head_dim, rot_dim, pos,
                                float(base), stream_handle(stream)))
    return x


def kv_append(k_cache, v_cache, k, v, n_kv_heads: int, head_dim: int, max_seq: int, pos: int,
              stream=None):
    check(lib().qws_kv_append(_dev(k_cache, "k_cache", torch.float32),
                              _dev(v_cache, "v_cache", torch.float32),
                              _dev(k, "k", torch.float32), _dev(v, "v", torch.float32),
                              n_kv_heads, head_dim, max_seq, pos, stream_handle(stream)))


def kv_attention(q, k_cache, v_cache, n_q_heads: int, n_kv_heads: int, head_dim: int,
                 max_seq: int, n_ctx: int, scale: float, softcap: float = 0.0, workspace=None,
                 out=None, stream=None):
    """One query token q [n_q_heads, head_dim] over cache positions 0 .. n_ctx-1."""
    y = out if out is not None else torch.empty((n_q_heads, head_dim), dtype=torch.float32,
                                                device=q.device)
    need = workspace_bytes(OP_KV_ATTENTION, n_ctx, head_dim, n_q_heads, n_kv_heads)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    check(lib().qws_kv_attention(
        _dev(q, "q", torch.float32), _dev(k_cache, "k_cache", torch.float32),
        _dev(v_cache, "v_cache", torch.float32), _dev(y, "out", torch.float32), n_q_heads,
        n_kv_heads, head_dim, max_seq, n_ctx, float(scale), float(softcap),
        _dev(workspace, "workspace"), workspace.numel() * workspace.element_size(),
        stream_handle(stream)))
    return y


def q4k_ffn_gate_up_geglu(Wg, Wu, x, hidden: int, inter: int, out=None, stream=None):
    m = _out(out, (inter,), x)
    check(lib().qws_q4k_ffn_gate_up_geglu(_dev(Wg, "Wg", torch.uint8), _dev(Wu, "Wu", torch.uint8),
                                          _dev(x, "x", torch.float32), _dev(m, "m", torch.float32),
                                          hidden, inter, stream_handle(stream)))
    return m


def q4k_ffn_gate_up_geglu_down(Wg, Wu, Wd, wd_fmt: int, x, hidden: int, inter: int,
                               workspace=None, out=None, stream=None):
    y = _out(out, (hidden,), x)
    need = workspace_bytes(OP_FFN, 0, hidden, inter, 1, 0)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    check(lib().qws_q4k_ffn_gate_up_geglu_down(
        _dev(Wg, "Wg", torch.uint8), _dev(Wu, "Wu", torch.uint8), _dev(Wd, "Wd", torch.uint8),
        wd_fmt, _dev(x, "x", torch.float32), _dev(y, "y", torch.float32), hidden, inter,
        _dev(workspace, "workspace"), workspace.numel() * workspace.element_size(),
        stream_handle(stream)))
    return y


def q4k_ffn_gate_up_silu(Wg, Wu, x, hidden: int, inter: int, out=None, stream=None):
    m = _out(out, (inter,), x)
    check(lib().qws_q4k_ffn_gate_up_silu(_dev(Wg, "Wg", torch.uint8), _dev(Wu, "Wu", torch.uint8),
                                         _dev(x, "x", torch.float32), _dev(m, "m", torch.float32),
                                         hidden, inter, stream_handle(stream)))
    return m


def q4k_ffn_gate_up_silu_down(Wg, Wu, Wd, wd_fmt: int, x, hidden: int, inter: int,
                              workspace=None, out=None, stream=None):
    y = _out(out, (hidden,), x)
    need = workspace_bytes(OP_FFN, 0, hidden, inter, 1, 0)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    check(lib().qws_q4k_ffn_gate_up_silu_down(
        _dev(Wg, "Wg", torch.uint8), _dev(Wu, "Wu", torch.uint8), _dev(Wd, "Wd", torch.uint8),
        wd_fmt, _dev(x, "x", torch.float32), _dev(y, "y", torch.float32), hidden, inter,
        _dev(workspace, "workspace"), workspace.numel() * workspace.element_size(),
        stream_handle(stream)))
    return y


def residual_rms_norm(h, y, w, eps: float, batch: int = 1, out=None, stream=None):
    """h += y (in place), returns x = rms_norm(h, w)."""
    n = h.numel() // batch
    x = _out(out, tuple(h.shape), h)
    check(lib().qws_residual_rms_norm(_dev(h, "h", torch.float32), _dev(y, "y", torch.float32),
                                      _dev(w, "w", torch.float32), _dev(x, "x", torch.float32), n,
                                      float(eps), batch, stream_handle(stream)))
    return x


def rms_norm(x, w, eps: float, batch: int = 1, out=None, stream=None):
    y = _out(out, tuple(x.shape), x)
    n = x.numel() // batch
    check(lib().qws_rms_norm(_dev(x, "x", torch.float32), _dev(w, "w", torch.float32),
                             _dev(y, "y", torch.float32), n, float(eps), batch,
                             stream_handle(stream)))
    return y


def residual_add(h, y, batch: int = 1, stream=None):
    n = h.numel() // batch
    check(lib().qws_residual_add(_dev(h, "h", torch.float32), _dev(y, "y", torch.float32), n,
                                 batch, stream_handle(stream)))
    return h


Layer = _lib.QwsLayer
Dims = _lib.QwsDims


def make_layer(t: dict) -> Layer:
    """qws_layer from a dict of device tensors (Wq..Wd uint8, w_* float32) and formats."""
    return Layer(
        _dev(t["Wq"], "Wq", torch.uint8), _dev(t["Wk"], "Wk", torch.uint8),
        _dev(t["Wv"], "Wv", torch.uint8), _dev(t["Wo"], "Wo", torch.uint8),
        _dev(t["Wg"], "Wg", torch.uint8), _dev(t["Wu"], "Wu", torch.uint8),
        _dev(t["Wd"], "Wd", torch.uint8),
        int(t["fmt_qkv"]), int(t["fmt_o"]), int(t["fmt_gu"]), int(t["fmt_down"]),
        _dev(t["w_in"], "w_in", torch.float32), _dev(t["w_post_attn"], "w_post_attn", torch.float32),
        _dev(t["w_pre_ffn"], "w_pre_ffn", torch.float32),
        _dev(t["w_post_ffn"], "w_post_ffn", torch.float32))


def make_dims(d: dict) -> Dims:
    return Dims(int(d["hidden"]), int(d["inter"]), int(d["n_q_heads"]), int(d["n_kv_heads"]),
                int(d["head_dim"]), float(d["eps"]), int(d["post_norms"]))


def decode_chain(layers, h, dims: dict, workspace=None, stream=None, w_final=None, hn=None):
    """Runs len(layers) decoder layers on h (in place).  layers: list of dicts
    of device tensors (see make_layer) or prepared Layer structs.  With
    w_final and hn (qws_decode_chain_final_norm) the same launch also writes
    hn = rms_norm(h, w_final) after the last layer."""
    n = len(layers)
    arr = (Layer * n)(*[L if isinstance(L, Layer) else make_layer(L) for L in layers])
    D = make_dims(dims)
    # the kernel reads / writes `hidden` values of each: a shorter tensor
    # would be overrun on the device, so refuse it here
    for name, t in (("h", h), ("w_final", w_final), ("hn", hn)):
        if isinstance(t, torch.Tensor) and t.numel() < int(dims["hidden"]):
            raise ValueError(f"{name} has {t.numel()} elements, hidden is {dims['hidden']}")
    need = workspace_bytes(OP_DECODE_CHAIN, 0, dims["hidden"], dims["inter"], 1, 0)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=h.device)
    nbytes = workspace.numel() * workspace.element_size()
    if w_final is None and hn is None:
        check(lib().qws_decode_chain(arr, n, _dev(h, "h", torch.float32), C.byref(D),
                                     _dev(workspace, "workspace"), nbytes,
                                     stream_handle(stream)))
        return h
    check(lib().qws_decode_chain_final_norm(
        arr, n, _dev(h, "h", torch.float32), _dev(w_final, "w_final", torch.float32),
        _dev(hn, "hn", torch.float32), C.byref(D), _dev(workspace, "workspace"), nbytes,
        stream_handle(stream)))
    return h


def decode_kv_workspace_bytes(dims: dict, max_seq: int) -> int:
    D = make_dims(dims)
    return int(lib().qws_decode_kv_workspace_bytes(C.byref(D), int(max_seq)))


def decode_kv(layers, h, dims: dict, k_caches, v_caches, max_seq: int, pos: int, rot_dim: int,
              rope_base: float, attn_scale: float, softcap: float = 0.0, workspace=None,
              stream=None):
    """One decode step at position pos over len(layers) layers with KV caches
    (qws_decode_kv): h in place; k_caches[l] / v_caches[l] are f32 device
    tensors [n_kv_heads, max_seq, head_dim], position pos is written."""
    n = len(layers)
    if len(k_caches) != n or len(v_caches) != n:
        raise ValueError("one k and one v cache per layer")
    # the kernels read / write these extents: refuse shorter tensors here
    if h.numel() < int(dims["hidden"]):
        raise ValueError(f"h has {h.numel()} elements, hidden is {dims['hidden']}")
    cache = int(dims["n_kv_heads"]) * int(max_seq) * int(dims["head_dim"])
    for t in list(k_caches) + list(v_caches):
        if isinstance(t, torch.Tensor) and t.numel() < cache:
            raise ValueError(f"a cache has {t.numel()} elements, needs {cache}")
    arr = (Layer * n)(*[L if isinstance(L, Layer) else make_layer(L) for L in layers])
    D = make_dims(dims)
    kp = (C.c_void_p * n)(*[_dev(t, "k_cache", torch.float32) for t in k_caches])
    vp = (C.c_void_p * n)(*[_dev(t, "v_cache", torch.float32) for t in v_caches])
    kv = _lib.QwsKv(C.cast(kp, C.c_void_p), C.cast(vp, C.c_void_p), int(max_seq), int(pos),
                    int(rot_dim), float(rope_base), float(attn_scale), float(softcap))
    need = decode_kv_workspace_bytes(dims, max_seq)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=h.device)
    check(lib().qws_decode_kv(arr, n, _dev(h, "h", torch.float32), C.byref(D), C.byref(kv),
                              _dev(workspace, "workspace"),
                              workspace.numel() * workspace.element_size(),
                              stream_handle(stream)))
    return h


def device_error() -> int:
    """Waits for the device; returns (and clears) the kernels' error code (0 = none)."""
    code = C.c_uint(0)
    lib().qws_device_error(C.byref(code))
    return int(code.value)
