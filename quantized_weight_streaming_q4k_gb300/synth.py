"""Seeded synthetic inputs for the decode path (host numpy arrays).

This module only draws random numbers and places them in the block fields.  It
holds none of the path's arithmetic: no dequantization, no product, no norm.
It feeds both the CUDA path and the oracle, so both see identical bytes.

Distributions (Gemma-3-4B shapes; infer-inference PERFORMANCE.md §GPU Decode
Path runs the same shapes with random weights):

* Q4_K super-block (144 B): d, dmin = f16(U(0.001, 0.02)); the 12 packed
  scale/min bytes and the 128 nibble bytes are uniform random bytes.  Every one
  of the 96 bits of the 12 scale bytes belongs to exactly one of the sixteen
  6-bit fields, so uniform bytes give sixteen independent U{0..63} scales and
  mins; uniform nibble bytes give U{0..15} quants.
* Q6_K super-block (210 B): ql and qh are uniform random bytes (6-bit quants
  ~U{0..63}); the sixteen int8 scales are U{scale_lo..scale_hi} (default
  U{0..63}); d = f16(U(0.001, 0.02)).
* Q4_0 block (18 B): d = f16(U(0.001, 0.02)); 16 uniform nibble bytes.
* Q8_0 block (34 B): d = f16(U(0.001, 0.02)); 32 uniform bytes read as int8
  (every code -128..127, including -128, which a quantizer never writes).
* Activations: x ~ N(0, 1) f32.  A "unit-RMS" vector is a uniform random point
  on the sphere of radius sqrt(n) (a normal draw divided by its RMS), the
  distribution of an RMS-normalised normal vector with unit weights.
* Norm weights ~ N(1, 0.1) f32.

Seeds: every tensor draws from ``numpy.random.default_rng(SeedSequence([0x5EED,
*key]))`` where ``key`` names the workload, tensor and layer.
"""
from __future__ import annotations

import numpy as np

BASE_SEED = 0x5EED
Q4_0, Q8_0, Q4_K, Q6_K = 2, 8, 12, 14
BLOCK_WEIGHTS = {Q4_0: 32, Q8_0: 32, Q4_K: 256, Q6_K: 256}
BLOCK_BYTES = {Q4_0: 18, Q8_0: 34, Q4_K: 144, Q6_K: 210}


def rng(*key: int) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence([BASE_SEED, *[int(k) for k in key]]))


def _random_bytes(g: np.random.Generator, n: int) -> np.ndarray:
    return np.frombuffer(g.bytes(n), dtype=np.uint8).copy()


def _f16_bytes(g: np.random.Generator, n: int, lo: float, hi: float) -> np.ndarray:
    v = g.uniform(lo, hi, size=n).astype(np.float16)
    return v.view(np.uint8).reshape(n, 2)


def n_blocks(fmt: int, rows: int, hidden: int) -> int:
    assert hidden % BLOCK_WEIGHTS[fmt] == 0
    return rows * (hidden // BLOCK_WEIGHTS[fmt])


def q4_k_matrix(g: np.random.Generator, rows: int, hidden: int,
                d_range=(0.001, 0.02), dmin_range=(0.001, 0.02)) -> np.ndarray:
    nb = n_blocks(Q4_K, rows, hidden)
    b = _random_bytes(g, nb * 144).reshape(nb, 144)
    b[:, 0:2] = _f16_bytes(g, nb, *d_range)
    b[:, 2:4] = _f16_bytes(g, nb, *dmin_range)
    return b.reshape(-1)


def q6_k_matrix(g: np.random.Generator, rows: int, hidden: int, scale_lo: int = 0,
                scale_hi: int = 63, d_range=(0.001, 0.02)) -> np.ndarray:
    nb = n_blocks(Q6_K, rows, hidden)
    b = _random_bytes(g, nb * 210).reshape(nb, 210)
    sc = g.integers(scale_lo, scale_hi + 1, size=(nb, 16)).astype(np.int8)
    b[:, 192:208] = sc.view(np.uint8)
    b[:, 208:210] = _f16_bytes(g, nb, *d_range)
    return b.reshape(-1)


def q4_0_matrix(g: np.random.Generator, rows: int, hidden: int,
                d_range=(0.001, 0.02)) -> np.ndarray:
    nb = n_blocks(Q4_0, rows, hidden)
    b = _random_bytes(g, nb * 18).reshape(nb, 18)
    b[:, 0:2] = _f16_bytes(g, nb, *d_range)
    return b.reshape(-1)


def q8_0_matrix(g: np.random.Generator, rows: int, hidden: int,
                d_range=(0.001, 0.02)) -> np.ndarray:
    nb = n_blocks(Q8_0, rows, hidden)
    b = _random_bytes(g, nb * 34).reshape(nb, 34)
    b[:, 0:2] = _f16_bytes(g, nb, *d_range)
    return b.reshape(-1)


def matrix(fmt: int, g: np.random.Generator, rows: int, hidden: int) -> np.ndarray:
    if fmt == Q4_K:
        return q4_k_matrix(g, rows, hidden)
    if fmt == Q6_K:
        return q6_k_matrix(g, rows, hidden)
    if fmt == Q4_0:
        return q4_0_matrix(g, rows, hidden)
    if fmt == Q8_0:
        return q8_0_matrix(g, rows, hidden)
    raise ValueError(f"unknown format {fmt}")


def normal_vector(g: np.random.Generator, n: int, batch: int | None = None) -> np.ndarray:
    shape = (n,) if batch is None else (batch, n)
    return g.standard_normal(size=shape).astype(np.float32)


def unit_rms_vector(g: np.random.Generator, n: int) -> np.ndarray:
    z = g.standard_normal(size=n)
    return (z / np.sqrt(np.mean(z * z))).astype(np.float32)


def norm_weights(g: np.random.Generator, n: int) -> np.ndarray:
    return g.normal(1.0, 0.1, size=n).astype(np.float32)


# --------------------------------------------------------------------------
# Workloads (Gemma-3-4B shapes)
# --------------------------------------------------------------------------
GEMMA3_4B = dict(hidden=2560, inter=10240, n_q_heads=8, n_kv_heads=4, head_dim=256,
                 eps=1e-6, post_norms=1)

# workload ids used in seeds
W_MATVEC, W_QKV, W_FFN, W_CHAIN, W_LM_HEAD = 0, 1, 2, 3, 4
# tensor ids used in seeds
T_WQ, T_WK, T_WV, T_WO, T_WG, T_WU, T_WD, T_NIN, T_NPA, T_NPF, T_NPFF, T_X, T_W, T_NFINAL = \
    range(14)


def chain_layer(layer: int, dims: dict = GEMMA3_4B, fmt_down: int = Q6_K,
                workload: int = W_CHAIN) -> dict:
    """All tensors of one decoder layer of the chain workload."""
    H, I = dims["hidden"], dims["inter"]
    qd = dims["n_q_heads"] * dims["head_dim"]
    kd = dims["n_kv_heads"] * dims["head_dim"]
    L = dict(fmt_qkv=Q4_K, fmt_o=Q4_K, fmt_gu=Q4_K, fmt_down=fmt_down)
    L["Wq"] = q4_k_matrix(rng(workload, T_WQ, layer), qd, H)
    L["Wk"] = q4_k_matrix(rng(workload, T_WK, layer), kd, H)
    L["Wv"] = q4_k_matrix(rng(workload, T_WV, layer), kd, H)
    L["Wo"] = q4_k_matrix(rng(workload, T_WO, layer), H, qd)
    L["Wg"] = q4_k_matrix(rng(workload, T_WG, layer), I, H)
    L["Wu"] = q4_k_matrix(rng(workload, T_WU, layer), I, H)
    L["Wd"] = matrix(fmt_down, rng(workload, T_WD, layer), H, I)
    L["w_in"] = norm_weights(rng(workload, T_NIN, layer), H)
    L["w_post_attn"] = norm_weights(rng(workload, T_NPA, layer), H)
    L["w_pre_ffn"] = norm_weights(rng(workload, T_NPF, layer), H)
    L["w_post_ffn"] = norm_weights(rng(workload, T_NPFF, layer), H)
    return L
