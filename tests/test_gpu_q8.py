"""GPU parity for the 8-bit path (infer-compute README §Shaders rows "Q8" and
"Element-wise"; §Architecture "Q4_0 through legacy Q8 path"), through the C
ABI, against the oracle.

  quantize_q8          : bit-exact bytes (codes and binary16 scales); both
                         sides take every decision in f32 with correctly
                         rounded operations.
  Q4_0 / Q8_0 x Q8_0   : |y - y_ref| <= 1e-5 * bound per row, bound =
                         sum_k |dw dx| sum_j |qw qx| (the integer sums are
                         exact on both sides; only the f32 scaling and the
                         f32 accumulation over blocks round).
  rms_norm_q8 /        : the GPU's f32 norm may differ from the oracle's in the
  residual_norm_q8       last bit, so a binary16 scale may differ by one step
                         and a code by one near a rounding half; every block
                         must still quantize the oracle's norm to within
                         0.57 steps (half a step plus the binary16 rounding of
                         d times 127) and 99.9 % of the bytes must agree.
"""
import os

import numpy as np
import pytest
import torch

import oracle
from quantized_weight_streaming_q4k_gb300 import build, ops, synth

pytestmark = pytest.mark.gpu
THREADS = max(1, min(16, os.cpu_count() or 1))
W_Q8 = 40          # workload id of this file's seeds


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    torch.cuda.set_device(0)
    yield
    assert ops.device_error() == 0


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    return t.detach().cpu().numpy()


def assert_bound(y, ref, bound, tol=1e-5, what=""):
    err = np.abs(y.astype(np.float64) - ref)
    ok = err <= tol * bound
    assert ok.all(), (f"{what}: {np.count_nonzero(~ok)} of {ok.size} outside {tol}*bound; "
                      f"worst err/bound {np.max(err / np.maximum(bound, 1e-300)):.3e}")


# ------------------------------------------------------------------ quantize
@pytest.mark.parametrize("n,batch", [(32, 1), (96, 1), (2560, 1), (2560, 8), (10240, 3)])
def test_quantize_bit_exact(n, batch):
    g = synth.rng(W_Q8, 1, n, batch)
    x = synth.normal_vector(g, n, batch if batch > 1 else None)
    got = host(ops.quantize_q8_0(dev(x), n, batch))
    want = oracle.quantize_q8_0(x)
    assert got.shape == want.shape
    assert np.array_equal(got, want), np.argwhere(got != want)[:8]


def test_quantize_special_blocks_bit_exact():
    # exact unit scale with halfway codes, a zero block, tiny (binary16
    # subnormal scale), huge, one-hot and sign-mixed blocks
    blocks = [
        np.concatenate([[127.0], np.arange(31) - 15.5]),
        np.zeros(32),
        np.linspace(-1e-6, 1e-6, 32),
        np.linspace(-3e4, 5e4, 32),
        np.eye(32)[7] * -2.5,
        np.tile([1.0, -1.0], 16) * (np.arange(32) + 0.5),
    ]
    x = np.concatenate(blocks).astype(np.float32)
    got = host(ops.quantize_q8_0(dev(x), x.size))
    assert np.array_equal(got, oracle.quantize_q8_0(x))


def test_quantize_random_scales_bit_exact():
    g = synth.rng(W_Q8, 2)
    scale = np.exp(g.uniform(-12, 12, size=(4096, 1)))
    x = (g.standard_normal((4096, 32)) * scale).astype(np.float32).reshape(-1)
    got = host(ops.quantize_q8_0(dev(x), x.size))
    assert np.array_equal(got, oracle.quantize_q8_0(x))


# ------------------------------------------------------------------ matvec
SHAPES = [(1, 64), (5, 192), (33, 512), (300, 2560), (129, 10240), (77, 20480)]


@pytest.mark.parametrize("wfmt", [oracle.Q4_0, oracle.Q8_0])
@pytest.mark.parametrize("rows,hidden", SHAPES)
def test_q8_matvec_parity_shapes(wfmt, rows, hidden):
    g = synth.rng(W_Q8, 3, wfmt, rows, hidden)
    W = synth.matrix(wfmt, g, rows, hidden)
    xq = oracle.quantize_q8_0(synth.normal_vector(g, hidden))
    y = host(ops.q8_matvec(wfmt, dev(W), dev(xq), rows, hidden))
    ref, bound = oracle.matvec_q8(wfmt, W, rows, hidden, xq, threads=THREADS)
    assert_bound(y, ref, bound, what=f"fmt {wfmt} {rows}x{hidden}")


@pytest.mark.parametrize("wfmt", [oracle.Q4_0, oracle.Q8_0])
@pytest.mark.parametrize("batch", [2, 3, 8])
def test_q8_matvec_batch(wfmt, batch):
    rows, hidden = 1000, 2560
    g = synth.rng(W_Q8, 4, wfmt, batch)
    W = synth.matrix(wfmt, g, rows, hidden)
    xq = oracle.quantize_q8_0(synth.normal_vector(g, hidden, batch))
    y = host(ops.q8_matvec(wfmt, dev(W), dev(xq), rows, hidden, batch)).reshape(batch, rows)
    ref, bound = oracle.matvec_q8(wfmt, W, rows, hidden, xq, threads=THREADS)
    assert_bound(y, ref, bound, what=f"fmt {wfmt} batch {batch}")


@pytest.mark.parametrize("wfmt", [oracle.Q4_0, oracle.Q8_0])
@pytest.mark.parametrize("rows,hidden,batch", [
    (17, 256, 8),      # smallest hidden of the decode-once kernel; one full tile + 1 row
    (333, 3072, 8),    # largest hidden: Q8_0 rows leave room for two ring stages only
    (16, 512, 5),      # exactly one tile
    (1, 768, 2),       # one row: the tile is almost all tail
    (250, 2624, 4),    # hidden % 256 != 0: the lane-unit engine instead
    (40, 3584, 2),     # hidden > 3072: the lane-unit engine instead
])
def test_q8_matvec_batch_kernel_edges(wfmt, rows, hidden, batch):
    g = synth.rng(W_Q8, 10, wfmt, rows, hidden, batch)
    W = synth.matrix(wfmt, g, rows, hidden)
    xq = oracle.quantize_q8_0(synth.normal_vector(g, hidden, batch))
    y = host(ops.q8_matvec(wfmt, dev(W), dev(xq), rows, hidden, batch)).reshape(batch, rows)
    ref, bound = oracle.matvec_q8(wfmt, W, rows, hidden, xq)
    assert_bound(y, ref, bound, what=f"fmt {wfmt} {rows}x{hidden} batch {batch}")


def test_q8_matvec_batch_extreme_codes():
    # every weight code -128 / 127 and every activation code +-127 at batch 8:
    # the per-block integer products reach 32 * 128 * 127 in the tensor-core sum
    rows, hidden, batch = 24, 1024, 8
    g = synth.rng(W_Q8, 11)
    W = synth.q8_0_matrix(g, rows, hidden).reshape(-1, 34)
    W[0::2, 2:] = 0x80
    W[1::2, 2:] = 0x7F
    sign = np.where(np.arange(hidden) % 2 == 0, 1.0, -1.0)
    x = np.stack([sign * (n + 1) * (-1.0) ** n for n in range(batch)]).astype(np.float32)
    xq = oracle.quantize_q8_0(x)
    assert np.all(np.abs(xq.reshape(-1, 34)[:, 2:].view(np.int8)) == 127)
    y = host(ops.q8_matvec(oracle.Q8_0, dev(W.reshape(-1)), dev(xq), rows, hidden, batch))
    ref, bound = oracle.matvec_q8(oracle.Q8_0, W.reshape(-1), rows, hidden, xq)
    assert_bound(y.reshape(batch, rows), ref, bound, what="batch extreme codes")


def test_q8_matvec_batch_is_run_to_run_identical():
    rows, hidden, batch = 4099, 2560, 8
    g = synth.rng(W_Q8, 12)
    W = dev(synth.matrix(oracle.Q4_0, g, rows, hidden))
    xq = dev(oracle.quantize_q8_0(synth.normal_vector(g, hidden, batch)))
    a = host(ops.q8_matvec(oracle.Q4_0, W, xq, rows, hidden, batch))
    b = host(ops.q8_matvec(oracle.Q4_0, W, xq, rows, hidden, batch))
    assert np.array_equal(a, b)


def test_q8_matvec_lane_limit_batch_at_maximum_hidden():
    # batch * hidden / 64 == 320: every consumer lane holds one unit
    rows, hidden, batch = 97, 5120, 4
    g = synth.rng(W_Q8, 5)
    W = synth.matrix(oracle.Q4_0, g, rows, hidden)
    xq = oracle.quantize_q8_0(synth.normal_vector(g, hidden, batch))
    y = host(ops.q8_matvec(oracle.Q4_0, dev(W), dev(xq), rows, hidden, batch))
    ref, bound = oracle.matvec_q8(oracle.Q4_0, W, rows, hidden, xq)
    assert_bound(y.reshape(batch, rows), ref, bound, what="lane limit")


def test_q8_matvec_extreme_codes():
    # Q8_0 weights with every code -128 / 127 against activations at +-127:
    # the integer sums reach their largest magnitude
    rows, hidden = 8, 256
    g = synth.rng(W_Q8, 6)
    W = synth.q8_0_matrix(g, rows, hidden).reshape(-1, 34)
    W[0::2, 2:] = 0x80
    W[1::2, 2:] = 0x7F
    x = np.where(np.arange(hidden) % 2 == 0, 1.0, -1.0).astype(np.float32) * 3.0
    xq = oracle.quantize_q8_0(x)
    y = host(ops.q8_matvec(oracle.Q8_0, dev(W.reshape(-1)), dev(xq), rows, hidden))
    ref, bound = oracle.matvec_q8(oracle.Q8_0, W.reshape(-1), rows, hidden, xq)
    assert_bound(y, ref, bound, what="extreme codes")


def test_q8_matvec_is_run_to_run_identical():
    rows, hidden = 4099, 2560
    g = synth.rng(W_Q8, 7)
    W = dev(synth.matrix(oracle.Q4_0, g, rows, hidden))
    xq = dev(oracle.quantize_q8_0(synth.normal_vector(g, hidden)))
    a = host(ops.q8_matvec(oracle.Q4_0, W, xq, rows, hidden))
    b = host(ops.q8_matvec(oracle.Q4_0, W, xq, rows, hidden))
    assert np.array_equal(a, b)


def test_quantize_then_matvec_on_device():
    # the whole 8-bit path on the GPU: quantize_q8 then the Q4_0 x Q8_0 matvec
    rows, hidden = 2560, 10240
    g = synth.rng(W_Q8, 8)
    W = synth.matrix(oracle.Q4_0, g, rows, hidden)
    x = synth.normal_vector(g, hidden)
    xq_d = ops.quantize_q8_0(dev(x), hidden)
    y = host(ops.q8_matvec(oracle.Q4_0, dev(W), xq_d, rows, hidden))
    xq = oracle.quantize_q8_0(x)
    assert np.array_equal(host(xq_d), xq)
    ref, bound = oracle.matvec_q8(oracle.Q4_0, W, rows, hidden, xq, threads=THREADS)
    assert_bound(y, ref, bound, what="quantize + matvec")


@pytest.mark.parametrize("wfmt", [oracle.Q4_0, oracle.Q8_0])
def test_q8_qkv_proj_gemma_shapes(wfmt):
    hidden, q_dim, kv_dim = 2560, 2048, 1024
    g = synth.rng(W_Q8, 9, wfmt)
    Wq = synth.matrix(wfmt, g, q_dim, hidden)
    Wk = synth.matrix(wfmt, g, kv_dim, hidden)
    Wv = synth.matrix(wfmt, g, kv_dim, hidden)
    xq = oracle.quantize_q8_0(synth.unit_rms_vector(g, hidden))
    q, k, v = ops.q8_qkv_proj(wfmt, dev(Wq), dev(Wk), dev(Wv), dev(xq), hidden, q_dim, kv_dim)
    for name, W, rows, out in (("q", Wq, q_dim, q), ("k", Wk, kv_dim, k), ("v", Wv, kv_dim, v)):
        ref, bound = oracle.matvec_q8(wfmt, W, rows, hidden, xq)
        assert_bound(host(out), ref, bound, what=name)


@pytest.mark.parametrize("batch", [1, 8])
def test_q8_lm_head_full_size(batch):
    # the 262144 x 2560 Q4_0 lm_head through the 8-bit path; all rows checked
    V, H = 262144, 2560
    g = synth.rng(synth.W_LM_HEAD, W_Q8, batch)
    W = synth.q4_0_matrix(g, V, H)
    x = synth.normal_vector(g, H, batch if batch > 1 else None)
    xq_d = ops.quantize_q8_0(dev(x), H, batch)
    y = host(ops.q8_matvec(oracle.Q4_0, dev(W), xq_d, V, H, batch)).reshape(batch, V)
    xq = oracle.quantize_q8_0(x).reshape(batch, -1)
    assert np.array_equal(host(xq_d).reshape(batch, -1), xq)
    ref, bound = oracle.matvec_q8(oracle.Q4_0, W, V, H, xq, threads=THREADS)
    assert_bound(y, ref.reshape(batch, V), bound.reshape(batch, V), what=f"lm_head q8 b{batch}")


# ------------------------------------------------------------------ fused norm + quantize
def check_norm_q8(got, y_ref, want):
    """got / want: Q8_0 blocks of the GPU and the oracle; y_ref: the oracle's
    f64 normalised values.  The GPU's norm differs from the oracle's in the
    last f32 bit, so a scale may differ by one binary16 step and a code by
    one where x * id falls within rounding of a half; every block must still
    be a valid quantization of y_ref and almost all bytes must agree."""
    g2, w2 = got.reshape(-1, 34), want.reshape(-1, 34)
    y = y_ref.reshape(-1, 32)
    for blk_g, blk_w, yb in zip(g2, w2, y):
        dg, dw = int(blk_g[0]) | int(blk_g[1]) << 8, int(blk_w[0]) | int(blk_w[1]) << 8
        assert abs(dg - dw) <= 1
        d = oracle.half(dg)
        q = blk_g[2:].view(np.int8).astype(np.int64)
        assert np.all(np.abs(yb - d * q) <= 0.57 * d + 1e-30)
    assert np.mean(got == want) >= 0.999


@pytest.mark.parametrize("n,batch", [(32, 1), (2560, 1), (2560, 3), (10240, 1)])
def test_rms_norm_q8(n, batch):
    g = synth.rng(W_Q8, 10, n, batch)
    x = synth.normal_vector(g, n, batch if batch > 1 else None)
    w = synth.norm_weights(g, n)
    got = host(ops.rms_norm_q8(dev(x), dev(w), 1e-6, n, batch))
    want = oracle.rms_norm_q8(x, w, 1e-6)
    xs = np.asarray(x, dtype=np.float64).reshape(-1, n)
    y_ref = np.stack([oracle.rms_norm(r, w, 1e-6) for r in xs])
    check_norm_q8(got, y_ref, want)


@pytest.mark.parametrize("n,batch", [(2560, 1), (512, 4)])
def test_residual_rms_norm_q8(n, batch):
    g = synth.rng(W_Q8, 11, n, batch)
    h = synth.normal_vector(g, n, batch if batch > 1 else None)
    y = synth.normal_vector(g, n, batch if batch > 1 else None)
    w = synth.norm_weights(g, n)
    hd = dev(h)
    got = host(ops.residual_rms_norm_q8(hd, dev(y), dev(w), 1e-6, n, batch))
    hs, want = oracle.residual_rms_norm_q8(h, y, w, 1e-6)
    # the residual sum is one f32 rounding of the exact sum on both sides
    assert np.array_equal(host(hd), hs.astype(np.float32))
    y_ref = np.stack([oracle.rms_norm(r, w, 1e-6) for r in hs.astype(np.float32).astype(np.float64).reshape(-1, n)])
    check_norm_q8(got, y_ref, oracle.rms_norm_q8(hs.astype(np.float32), w, 1e-6))
