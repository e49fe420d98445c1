"""GPU parity for decode attention over a KV cache (infer-compute README
§Shaders rows "RoPE" and "Attention"; infer-inference README §BLAS-Fused
Attention), through the C ABI, against the oracle.

Tolerances, derived from the arithmetic:
  rope       : the GPU rotates in f64 and rounds once, so |y - ref| <=
               2^-24 |ref| + 2^-40 (|a| + |b|) (f64 differences in sin/cos).
  kv_append  : bit-exact.
  attention  : each score is an f32 sum of head_dim products and a shuffle
               tree: |ds| <= (hd + 32) 2^-24 smax, smax = max_t sum_i |scale q k|;
               exp turns it into a relative weight error ~2 |ds| (plus a few
               ulp of expf), and the online rescaling and the merges add
               O(2^-20) relative; so per element
                 |out - ref| <= (8 (hd + 32) 2^-24 smax + 1e-5) * sum_t p_t |v_t|.
"""
import numpy as np
import pytest
import torch

import oracle
from quantized_weight_streaming_q4k_gb300 import build, ops, synth

pytestmark = pytest.mark.gpu
W_ATT = 60         # workload id of this file's seeds


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    torch.cuda.set_device(0)
    yield
    assert ops.device_error() == 0


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def host(t):
    return t.detach().cpu().numpy().astype(np.float64)


# ------------------------------------------------------------------ rope
@pytest.mark.parametrize("hd,rot", [(256, 256), (256, 64), (128, 128), (64, 16)])
@pytest.mark.parametrize("pos,base", [(0, 10000.0), (1, 10000.0), (4095, 10000.0),
                                      (131071, 1e6), (1000, 500.0)])
def test_rope_parity(hd, rot, pos, base):
    g = synth.rng(W_ATT, 1, hd, rot, pos)
    x = g.standard_normal((8, hd)).astype(np.float32)
    y = host(ops.rope_at_pos(dev(x), 8, hd, rot, pos, base))
    ref = oracle.rope(x, 8, hd, rot, pos, base)
    half = rot // 2
    ab = np.abs(x).astype(np.float64)
    scale = np.concatenate([ab[:, :half] + ab[:, half:rot]] * 2 + [ab[:, rot:]], axis=1)
    assert np.all(np.abs(y - ref) <= 2.0 ** -24 * np.abs(ref) + 2.0 ** -40 * scale + 1e-30)
    assert np.array_equal(y[:, rot:], x[:, rot:].astype(np.float64))


# ------------------------------------------------------------------ kv_append
def test_kv_append_bit_exact():
    g = synth.rng(W_ATT, 2)
    nkv, hd, L = 4, 256, 64
    kc, vc = g.standard_normal((2, nkv, L, hd)).astype(np.float32)
    k, v = g.standard_normal((2, nkv, hd)).astype(np.float32)
    kcd, vcd = dev(kc), dev(vc)
    ops.kv_append(kcd, vcd, dev(k), dev(v), nkv, hd, L, 37)
    rk, rv = oracle.kv_append(kc, vc, k, v, nkv, hd, L, 37)
    assert np.array_equal(host(kcd), rk) and np.array_equal(host(vcd), rv)


# ------------------------------------------------------------------ attention
def check_attention(nq, nkv, hd, L, n_ctx, scale, softcap, seed):
    g = synth.rng(W_ATT, 3, seed)
    kc = g.standard_normal((nkv, L, hd)).astype(np.float32)
    vc = g.standard_normal((nkv, L, hd)).astype(np.float32)
    q = g.standard_normal((nq, hd)).astype(np.float32)
    out = host(ops.kv_attention(dev(q), dev(kc), dev(vc), nq, nkv, hd, L, n_ctx, scale, softcap))
    ref, bound, smax = oracle.kv_attention(q, kc, vc, nq, nkv, hd, L, n_ctx, scale, softcap)
    tol = (8 * (hd + 32) * 2.0 ** -24 * smax[:, None] + 1e-5) * bound
    err = np.abs(out - ref)
    assert np.all(err <= tol), (f"worst err/bound {np.max(err / bound):.3e}, "
                                f"tol/bound {np.max(tol / bound):.3e}")
    return out


@pytest.mark.parametrize("n_ctx", [1, 2, 7, 128, 129, 1000, 4097])
def test_attention_lengths_gemma_heads(n_ctx):
    check_attention(8, 4, 256, 4100, n_ctx, 1.0 / 16, 0.0, n_ctx)


@pytest.mark.parametrize("nq,nkv,hd", [(4, 4, 128), (8, 2, 64), (6, 3, 32), (16, 4, 128)])
def test_attention_head_layouts(nq, nkv, hd):
    check_attention(nq, nkv, hd, 700, 613, hd ** -0.5, 0.0, nq * 100 + hd)


@pytest.mark.parametrize("softcap", [50.0, 1.5])
def test_attention_softcap(softcap):
    check_attention(8, 4, 256, 900, 900, 0.2, softcap, int(softcap * 10))


def test_attention_full_context_gemma():
    # 32768 cached positions: 268 MB of f32 K and V
    check_attention(8, 4, 256, 32768, 32768, 1.0 / 16, 0.0, 99)


def test_attention_is_run_to_run_identical():
    g = synth.rng(W_ATT, 4)
    kc = dev(g.standard_normal((4, 3000, 128)))
    vc = dev(g.standard_normal((4, 3000, 128)))
    q = dev(g.standard_normal((8, 128)))
    a = host(ops.kv_attention(q, kc, vc, 8, 4, 128, 3000, 2999, 0.088))
    b = host(ops.kv_attention(q, kc, vc, 8, 4, 128, 3000, 2999, 0.088))
    assert np.array_equal(a, b)


def test_decode_step_rope_append_attend():
    # one decode step at position pos: RoPE on q and k, append k and v, attend
    nq, nkv, hd, L, pos, base = 8, 4, 256, 512, 300, 10000.0
    g = synth.rng(W_ATT, 5)
    kc = g.standard_normal((nkv, L, hd)).astype(np.float32)
    vc = g.standard_normal((nkv, L, hd)).astype(np.float32)
    q = g.standard_normal((nq, hd)).astype(np.float32)
    k = g.standard_normal((nkv, hd)).astype(np.float32)
    v = g.standard_normal((nkv, hd)).astype(np.float32)
    qd, kd, kcd, vcd = dev(q), dev(k), dev(kc), dev(vc)
    ops.rope_at_pos(qd, nq, hd, hd, pos, base)
    ops.rope_at_pos(kd, nkv, hd, hd, pos, base)
    ops.kv_append(kcd, vcd, kd, dev(v), nkv, hd, L, pos)
    out = host(ops.kv_attention(qd, kcd, vcd, nq, nkv, hd, L, pos + 1, 1.0 / 16))
    qr = oracle.rope(q, nq, hd, hd, pos, base)
    kr = oracle.rope(k, nkv, hd, hd, pos, base)
    kc2, vc2 = oracle.kv_append(kc, vc, kr, v, nkv, hd, L, pos)
    ref, bound, smax = oracle.kv_attention(qr, kc2, vc2, nq, nkv, hd, L, pos + 1, 1.0 / 16)
    # the GPU's rotated q and k differ from the oracle's by one f32 rounding:
    # a relative score change of ~2^-23, folded into the attention tolerance
    tol = (8 * (hd + 32) * 2.0 ** -24 * smax[:, None] + 2.0 ** -20 * smax[:, None] + 1e-5) * bound
    assert np.all(np.abs(out - ref) <= tol)
