"""GPU parity: the CUDA path (through the C ABI) against the f64 oracle.

Tolerances (stated by the workload definition):
  matvec / QKV / lm_head : |y - y_ref| <= 1e-5 * sum_i |w_i x_i|       per row
  gated FFN output       : |y - y_ref| <= 1e-4 * |y_ref|, or, where y_ref
                           nearly cancels, <= 1e-4 * sum_j |wd_j m_j|
  GEGLU intermediate m   : first-order propagation of the matvec bound
  rms_norm               : relative 1e-5 per element (f32 arithmetic)
"""
import os

import numpy as np
import pytest
import torch

import oracle
from quantized_weight_streaming_q4k_gb300 import build, ops, synth

pytestmark = pytest.mark.gpu
THREADS = max(1, min(16, os.cpu_count() or 1))


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    torch.cuda.set_device(0)
    yield
    assert ops.device_error() == 0


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    return t.detach().cpu().numpy().astype(np.float64)


def assert_bound(y, ref, bound, tol=1e-5, what=""):
    err = np.abs(y - ref)
    ok = err <= tol * bound
    assert ok.all(), (f"{what}: {np.count_nonzero(~ok)} of {ok.size} outside {tol}*bound; "
                      f"worst err/bound {np.max(err / np.maximum(bound, 1e-300)):.3e}")


FMT_NAME = {oracle.Q4_0: "q4_0", oracle.Q4_K: "q4_k", oracle.Q6_K: "q6_k"}


def run_matvec(fmt, W, x, rows, hidden, batch=1, split_k=1):
    Wd, xd = dev(W), dev(x)
    if fmt == oracle.Q4_K and split_k == 1:
        return host(ops.q4k_matvec(Wd, xd, rows, hidden, batch))
    if fmt == oracle.Q6_K and split_k == 1:
        return host(ops.q6k_matvec(Wd, xd, rows, hidden, batch))
    ws = None
    if split_k != 1:
        nbytes = ops.workspace_bytes(ops._lib.OP_MATVEC, rows, hidden, 0, batch, split_k)
        ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device="cuda")
    if fmt == oracle.Q4_0:
        return host(ops.q4_0_matvec(Wd, xd, rows, hidden, batch, split_k, ws))
    return host(ops.matvec(fmt, Wd, xd, rows, hidden, batch, split_k, ws))


# (65, 20480): the widest single pass (320 lane units of 64 columns, one row
# slot per tile round)
SHAPES = [(1, 256), (3, 256), (33, 512), (300, 2560), (129, 10240), (77, 2048), (65, 20480)]


@pytest.mark.parametrize("fmt", [oracle.Q4_K, oracle.Q6_K, oracle.Q4_0])
@pytest.mark.parametrize("rows,hidden", SHAPES)
def test_matvec_parity_shapes(fmt, rows, hidden):
    g = synth.rng(1000, fmt, rows, hidden)
    W = synth.matrix(fmt, g, rows, hidden)
    x = synth.normal_vector(g, hidden)
    y = run_matvec(fmt, W, x, rows, hidden)
    ref, bound = oracle.matvec(fmt, W, rows, hidden, x, threads=THREADS)
    assert_bound(y, ref, bound, what=f"{FMT_NAME[fmt]} {rows}x{hidden}")


@pytest.mark.parametrize("fmt", [oracle.Q4_K, oracle.Q6_K, oracle.Q4_0])
def test_matvec_full_size_cfg0_shape(fmt):
    rows, hidden = 2560, 2560
    g = synth.rng(1001, fmt)
    W = synth.matrix(fmt, g, rows, hidden)
    x = synth.normal_vector(g, hidden)
    y = run_matvec(fmt, W, x, rows, hidden)
    ref, bound = oracle.matvec(fmt, W, rows, hidden, x, threads=THREADS)
    assert_bound(y, ref, bound, what=f"{FMT_NAME[fmt]} 2560x2560")


def test_q6k_down_projection_full_size():
    rows, hidden = 2560, 10240
    g = synth.rng(1002)
    W = synth.q6_k_matrix(g, rows, hidden)
    x = synth.normal_vector(g, hidden)
    y = run_matvec(oracle.Q6_K, W, x, rows, hidden)
    ref, bound = oracle.matvec(oracle.Q6_K, W, rows, hidden, x, threads=THREADS)
    assert_bound(y, ref, bound, what="q6_k 2560x10240")


def test_q6k_signed_scales_full_range():
    rows, hidden = 200, 2048
    g = synth.rng(1003)
    W = synth.q6_k_matrix(g, rows, hidden, scale_lo=-128, scale_hi=127)
    x = synth.normal_vector(g, hidden)
    y = run_matvec(oracle.Q6_K, W, x, rows, hidden)
    ref, bound = oracle.matvec(oracle.Q6_K, W, rows, hidden, x)
    assert_bound(y, ref, bound, what="q6_k signed scales")


@pytest.mark.parametrize("fmt", [oracle.Q4_K, oracle.Q6_K, oracle.Q4_0])
@pytest.mark.parametrize("dbits", [0x0001, 0x03FF, 0x8400, 0x0000, 0xBC00, 0x7800])
def test_special_scale_values(fmt, dbits):
    """binary16 subnormal, negative, zero and large d (and dmin for Q4_K)."""
    rows, hidden = 40, 512
    g = synth.rng(1004, fmt, dbits)
    W = synth.matrix(fmt, g, rows, hidden).reshape(-1, synth.BLOCK_BYTES[fmt])
    d = np.array([dbits & 0xFF, dbits >> 8], dtype=np.uint8)
    if fmt == oracle.Q4_K:
        W[::2, 0:2] = d
        W[1::3, 2:4] = d
    elif fmt == oracle.Q6_K:
        W[::2, 208:210] = d
    else:
        W[::2, 0:2] = d
    W = W.reshape(-1)
    x = synth.normal_vector(g, hidden)
    y = run_matvec(fmt, W, x, rows, hidden)
    ref, bound = oracle.matvec(fmt, W, rows, hidden, x)
    assert_bound(y, ref, bound, what=f"{FMT_NAME[fmt]} d=0x{dbits:04x}")


@pytest.mark.parametrize("scale", [1e-2, 1e3, 2.0 ** -40, 2.0 ** 30])
def test_activation_magnitudes(scale):
    rows, hidden = 64, 2560
    g = synth.rng(1005)
    W = synth.q4_k_matrix(g, rows, hidden)
    x = (synth.normal_vector(g, hidden) * np.float32(scale)).astype(np.float32)
    y = run_matvec(oracle.Q4_K, W, x, rows, hidden)
    ref, bound = oracle.matvec(oracle.Q4_K, W, rows, hidden, x)
    assert_bound(y, ref, bound, what=f"x*{scale}")


def test_zero_activation_gives_zero():
    rows, hidden = 50, 512
    W = synth.q4_k_matrix(synth.rng(1006), rows, hidden)
    y = run_matvec(oracle.Q4_K, W, np.zeros(hidden, np.float32), rows, hidden)
    assert np.all(y == 0)


@pytest.mark.parametrize("fmt,batch", [(oracle.Q4_K, 2), (oracle.Q4_K, 3), (oracle.Q4_K, 8),
                                       (oracle.Q4_0, 2), (oracle.Q4_0, 8), (oracle.Q6_K, 2),
                                       (oracle.Q6_K, 4), (oracle.Q6_K, 8)])
def test_batched_matvec(fmt, batch):
    rows, hidden = 333, 2560
    g = synth.rng(1007, fmt, batch)
    W = synth.matrix(fmt, g, rows, hidden)
    x = synth.normal_vector(g, hidden, batch=batch)
    y = run_matvec(fmt, W, x, rows, hidden, batch=batch)
    ref, bound = oracle.matvec(fmt, W, rows, hidden, x, threads=THREADS)
    assert y.shape == (batch, rows)
    assert_bound(y, ref, bound, what=f"{FMT_NAME[fmt]} batch {batch}")


@pytest.mark.parametrize("fmt", [oracle.Q4_K, oracle.Q4_0])
@pytest.mark.parametrize("hidden", [256, 768, 3072])
def test_batched_matvec_hidden_sizes(fmt, hidden):
    """Batch 8 on the decode-once kernel at hidden sizes whose column slices
    do not split evenly: at 256 most warps take no block, at 768 and 3072
    slices are odd and some start on an odd sub-block."""
    rows = 100
    g = synth.rng(1009, fmt, hidden)
    W = synth.matrix(fmt, g, rows, hidden)
    x = synth.normal_vector(g, hidden, batch=8)
    y = run_matvec(fmt, W, x, rows, hidden, batch=8)
    ref, bound = oracle.matvec(fmt, W, rows, hidden, x, threads=THREADS)
    assert y.shape == (8, rows)
    assert_bound(y, ref, bound, what=f"{FMT_NAME[fmt]} batch 8 hidden {hidden}")


@pytest.mark.parametrize("split_k", [2, 5, 10])
@pytest.mark.parametrize("batch", [1, 8])
def test_q4_0_split_k(split_k, batch):
    rows, hidden = 1000, 2560
    g = synth.rng(1008, split_k, batch)
    W = synth.q4_0_matrix(g, rows, hidden)
    x = synth.normal_vector(g, hidden, batch=batch if batch > 1 else None)
    y = run_matvec(oracle.Q4_0, W, x, rows, hidden, batch=batch, split_k=split_k)
    ref, bound = oracle.matvec(oracle.Q4_0, W, rows, hidden, x, threads=THREADS)
    assert_bound(y, ref, bound, what=f"q4_0 split {split_k} batch {batch}")
    # deterministic: run-to-run identical
    y2 = run_matvec(oracle.Q4_0, W, x, rows, hidden, batch=batch, split_k=split_k)
    assert np.array_equal(y, y2)


def test_large_hidden_needs_split():
    rows, hidden = 64, 40960
    g = synth.rng(1009)
    W = synth.q4_k_matrix(g, rows, hidden)
    x = synth.normal_vector(g, hidden)
    y = run_matvec(oracle.Q4_K, W, x, rows, hidden, split_k=0)
    ref, bound = oracle.matvec(oracle.Q4_K, W, rows, hidden, x)
    assert_bound(y, ref, bound, what="q4_k hidden 40960 auto split")


def test_qkv_projection_full_size():
    H, qd, kd = 2560, 2048, 1024
    g = synth.rng(1010)
    Wq, Wk, Wv = (synth.q4_k_matrix(g, r, H) for r in (qd, kd, kd))
    x = synth.unit_rms_vector(g, H)
    q, k, v = ops.q4k_qkv_proj(dev(Wq), dev(Wk), dev(Wv), dev(x), H, qd, kd)
    for name, W, r, t in (("q", Wq, qd, q), ("k", Wk, kd, k), ("v", Wv, kd, v)):
        ref, bound = oracle.matvec(oracle.Q4_K, W, r, H, x, threads=THREADS)
        assert_bound(host(t), ref, bound, what=f"qkv {name}")


def test_qkv_ragged_segments():
    H, qd, kd = 512, 40, 24
    g = synth.rng(1011)
    Wq, Wk, Wv = (synth.q4_k_matrix(g, r, H) for r in (qd, kd, kd))
    x = synth.normal_vector(g, H)
    q, k, v = ops.q4k_qkv_proj(dev(Wq), dev(Wk), dev(Wv), dev(x), H, qd, kd)
    for W, r, t in ((Wq, qd, q), (Wk, kd, k), (Wv, kd, v)):
        ref, bound = oracle.matvec(oracle.Q4_K, W, r, H, x)
        assert_bound(host(t), ref, bound, what="qkv ragged")


def test_o_projection_full_size():
    rows, hidden = 2560, 2048
    g = synth.rng(1012)
    W = synth.q4_k_matrix(g, rows, hidden)
    x = synth.normal_vector(g, hidden)
    y = run_matvec(oracle.Q4_K, W, x, rows, hidden)
    ref, bound = oracle.matvec(oracle.Q4_K, W, rows, hidden, x, threads=THREADS)
    assert_bound(y, ref, bound, what="o proj")


def _geglu_tolerance(g_ref, bg, u_ref, bu):
    # m = gelu(g) u;  |gelu'| <= 1.13;  first-order propagation of 1e-5 * bound
    gel = oracle.gelu_tanh(g_ref)
    return 1e-4 * np.abs(gel * u_ref) + 1e-5 * (1.13 * bg * np.abs(u_ref) + np.abs(gel) * bu)


@pytest.mark.parametrize("hidden,inter,scale", [(2560, 10240, 1.0), (512, 768, 1.0),
                                                (2560, 10240, 1e-2)])
def test_gate_up_geglu(hidden, inter, scale):
    g = synth.rng(1013, hidden, inter, int(scale * 100))
    Wg = synth.q4_k_matrix(g, inter, hidden)
    Wu = synth.q4_k_matrix(g, inter, hidden)
    x = (synth.unit_rms_vector(g, hidden) * np.float32(scale)).astype(np.float32)
    m = host(ops.q4k_ffn_gate_up_geglu(dev(Wg), dev(Wu), dev(x), hidden, inter))
    gr, bg = oracle.matvec(oracle.Q4_K, Wg, inter, hidden, x, threads=THREADS)
    ur, bu = oracle.matvec(oracle.Q4_K, Wu, inter, hidden, x, threads=THREADS)
    mref = oracle.gelu_tanh(gr) * ur
    tol = _geglu_tolerance(gr, bg, ur, bu)
    err = np.abs(m - mref)
    assert np.all(err <= tol), f"worst err/tol {np.max(err / tol):.3e}"


def _ffn_check(y, out, what):
    ref, bnd = out["y"], out["bound_y"]
    err = np.abs(y - ref)
    rel_ok = err <= 1e-4 * np.abs(ref)
    ok = rel_ok | (err <= 1e-4 * bnd)
    assert ok.all(), f"{what}: {np.count_nonzero(~ok)} outside; worst {np.max(err / bnd):.3e}"
    return int(np.count_nonzero(~rel_ok))


@pytest.mark.parametrize("fmt_d", [oracle.Q6_K, oracle.Q4_K])
@pytest.mark.parametrize("scale", [1.0, 1e-2])
def test_ffn_full_size(fmt_d, scale):
    H, I = 2560, 10240
    g = synth.rng(1014, fmt_d, int(scale * 100))
    Wg = synth.q4_k_matrix(g, I, H)
    Wu = synth.q4_k_matrix(g, I, H)
    Wd = synth.matrix(fmt_d, g, H, I)
    x = (synth.unit_rms_vector(g, H) * np.float32(scale)).astype(np.float32)
    y = host(ops.q4k_ffn_gate_up_geglu_down(dev(Wg), dev(Wu), dev(Wd), fmt_d, dev(x), H, I))
    out = oracle.ffn(oracle.Q4_K, Wg, Wu, fmt_d, Wd, H, I, x)
    n_second = _ffn_check(y, out, f"ffn down={FMT_NAME[fmt_d]} x*{scale}")
    print(f"ffn: {n_second} of {H} elements passed on the cancellation clause")


@pytest.mark.parametrize("hidden,inter,scale", [(2560, 10240, 1.0), (2560, 10240, 1e-2)])
def test_gate_up_silu(hidden, inter, scale):
    g = synth.rng(1018, hidden, inter, int(scale * 100))
    Wg = synth.q4_k_matrix(g, inter, hidden)
    Wu = synth.q4_k_matrix(g, inter, hidden)
    x = (synth.unit_rms_vector(g, hidden) * np.float32(scale)).astype(np.float32)
    m = host(ops.q4k_ffn_gate_up_silu(dev(Wg), dev(Wu), dev(x), hidden, inter))
    gr, bg = oracle.matvec(oracle.Q4_K, Wg, inter, hidden, x, threads=THREADS)
    ur, bu = oracle.matvec(oracle.Q4_K, Wu, inter, hidden, x, threads=THREADS)
    act = oracle.silu(gr)
    # m = silu(g) u;  |silu'| <= 1.1;  first-order propagation of 1e-5 * bound
    tol = 1e-4 * np.abs(act * ur) + 1e-5 * (1.1 * bg * np.abs(ur) + np.abs(act) * bu)
    err = np.abs(m - act * ur)
    assert np.all(err <= tol), f"worst err/tol {np.max(err / tol):.3e}"


@pytest.mark.parametrize("scale", [1.0, 1e-2])
def test_ffn_silu_full_size(scale):
    H, I = 2560, 10240
    g = synth.rng(1019, int(scale * 100))
    Wg = synth.q4_k_matrix(g, I, H)
    Wu = synth.q4_k_matrix(g, I, H)
    Wd = synth.q6_k_matrix(g, H, I)
    x = (synth.unit_rms_vector(g, H) * np.float32(scale)).astype(np.float32)
    y = host(ops.q4k_ffn_gate_up_silu_down(dev(Wg), dev(Wu), dev(Wd), ops.Q6_K, dev(x), H, I))
    out = oracle.ffn(oracle.Q4_K, Wg, Wu, oracle.Q6_K, Wd, H, I, x, act=oracle.ACT_SILU)
    _ffn_check(y, out, f"silu ffn x*{scale}")


@pytest.mark.parametrize("n,batch", [(2560, 1), (10240, 1), (2560, 3), (7, 2)])
def test_residual_rms_norm(n, batch):
    g = synth.rng(1020, n, batch)
    h = synth.normal_vector(g, n, batch)
    y = synth.normal_vector(g, n, batch)
    w = synth.norm_weights(g, n)
    hd = dev(h)
    x = host(ops.residual_rms_norm(hd, dev(y), dev(w), 1e-6, batch=batch))
    hb = host(hd).reshape(batch, n)
    for b in range(batch):
        h_ref, x_ref = oracle.residual_rms_norm(h.reshape(batch, n)[b], y.reshape(batch, n)[b], w,
                                                1e-6)
        # the add is exact in f32 rounding; the norm within 1e-5 relative
        assert np.array_equal(hb[b], h_ref.astype(np.float32).astype(np.float64))
        assert np.all(np.abs(x.reshape(batch, n)[b] - x_ref) <= 1e-5 * np.abs(x_ref) + 1e-30)


@pytest.mark.parametrize("n,batch", [(2560, 1), (10240, 1), (2560, 3), (7, 2)])
def test_rms_norm(n, batch):
    g = synth.rng(1015, n, batch)
    x = synth.normal_vector(g, n, batch=batch)
    w = synth.norm_weights(g, n)
    y = host(ops.rms_norm(dev(x), dev(w), 1e-6, batch=batch)).reshape(batch, n)
    for b in range(batch):
        ref = oracle.rms_norm(x.reshape(batch, n)[b], w, 1e-6)
        assert np.all(np.abs(y[b] - ref) <= 1e-5 * np.abs(ref) + 1e-30)


def test_back_to_back_dependent_launches():
    """Kernels overlap their start with the previous kernel's tail; each must
    still see the previous output (read after write) and must not overwrite
    a buffer the previous kernel is still reading (write after read).  Four
    matvecs ping-pong between two vectors, a norm and a residual add in
    between, with no host synchronisation."""
    g = synth.rng(1017)
    n = 2560
    Ws = [synth.q4_k_matrix(g, n, n) for _ in range(4)]
    w = synth.norm_weights(g, n)
    x0 = synth.normal_vector(g, n)
    Wd = [dev(W) for W in Ws]
    a, b = dev(x0), torch.empty(n, device="cuda")
    wd = dev(w)
    ops.q4k_matvec(Wd[0], a, n, n, out=b)       # b = W0 a
    ops.q4k_matvec(Wd[1], b, n, n, out=a)       # a = W1 b   (a was read by the previous)
    ops.rms_norm(a, wd, 1e-6, out=b)            # b = norm(a)
    ops.q4k_matvec(Wd[2], b, n, n, out=a)       # a = W2 b
    ops.residual_add(a, b)                      # a += b
    ops.q4k_matvec(Wd[3], a, n, n, out=b)       # b = W3 a
    got = host(b)
    r = x0.astype(np.float64)
    r, _ = oracle.matvec(oracle.Q4_K, Ws[0], n, n, r)
    r, _ = oracle.matvec(oracle.Q4_K, Ws[1], n, n, r)
    nb = oracle.rms_norm(r, w, 1e-6)
    r, _ = oracle.matvec(oracle.Q4_K, Ws[2], n, n, nb)
    r = r + nb
    ref, bound = oracle.matvec(oracle.Q4_K, Ws[3], n, n, r)
    # errors of the earlier steps propagate: compare against the oracle run
    # on the GPU's own input to the last step as well
    last_in = host(a)
    ref_tf, bound_tf = oracle.matvec(oracle.Q4_K, Ws[3], n, n, last_in)
    assert_bound(got, ref_tf, bound_tf, what="last step, teacher-forced")
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert rel < 1e-4, f"chain of launches: relative L2 error {rel:.2e}"


def test_residual_add_exact():
    g = synth.rng(1016)
    h = synth.normal_vector(g, 2560)
    y = synth.normal_vector(g, 2560)
    hd = dev(h)
    ops.residual_add(hd, dev(y))
    ref = oracle.residual_add(h, y)
    assert np.array_equal(host(hd), ref.astype(np.float32).astype(np.float64))


def _top5_check(logits, ref, bound, what):
    idx_ref = oracle.topk(ref, 6)
    idx = np.argsort(-logits, kind="stable")[:5]
    gaps = -np.diff(ref[idx_ref])
    tol = 2e-5 * np.max(bound[idx_ref])
    if np.all(gaps[:5] > tol):
        assert list(idx) == list(idx_ref[:5]), what
    else:  # near-tie: the sets must agree up to the tied ranks
        assert set(idx[:4]) <= set(idx_ref)
    return float(np.min(gaps[:5]))


@pytest.mark.parametrize("fmt", [oracle.Q4_0, oracle.Q4_K])
@pytest.mark.parametrize("batch", [1, 8])
def test_lm_head_full_size(fmt, batch):
    V, H = 262144, 2560
    g = synth.rng(synth.W_LM_HEAD, fmt, batch)
    W = synth.matrix(fmt, g, V, H)
    x = synth.normal_vector(g, H, batch=batch if batch > 1 else None)
    split = 1 if fmt == oracle.Q4_K else 0
    y = run_matvec(fmt, W, x, V, H, batch=batch, split_k=split).reshape(batch, V)
    ref, bound = oracle.matvec(fmt, W, V, H, x, threads=THREADS)
    ref, bound = ref.reshape(batch, V), bound.reshape(batch, V)
    assert_bound(y, ref, bound, what=f"lm_head {FMT_NAME[fmt]} b{batch}")
    for b in range(batch):
        gap = _top5_check(y[b], ref[b], bound[b], f"top5 b{b}")
        print(f"lm_head {FMT_NAME[fmt]} b{b}: min top-6 gap {gap:.3f}")


def test_lm_head_split_k_matches_single_pass():
    V, H = 262144, 2560
    g = synth.rng(synth.W_LM_HEAD, 99)
    W = synth.q4_0_matrix(g, V, H)
    x = synth.normal_vector(g, H)
    y1 = run_matvec(oracle.Q4_0, W, x, V, H, split_k=1)
    y5 = run_matvec(oracle.Q4_0, W, x, V, H, split_k=5)
    rows = np.arange(0, V, 997)
    ref, bound = oracle.matvec(oracle.Q4_0, W, V, H, x, threads=THREADS)
    assert_bound(y1[rows], ref[rows], bound[rows], what="split 1")
    assert_bound(y5[rows], ref[rows], bound[rows], what="split 5")
    assert np.all(np.abs(y1 - y5) <= 2e-5 * bound)


# Q4_0 and Q4_K at 2..8 vectors take the decode-once kernel (mma.sync on the
# codes and an f16 hi + lo split of x scaled by a power of two); the
# tolerance is the matvec's 1e-5 * sum |w x|.
@pytest.mark.parametrize("fmt", [oracle.Q4_0, oracle.Q4_K])
@pytest.mark.parametrize("rows,hidden,batch", [(37, 256, 2), (1000, 2560, 8), (4099, 3072, 5),
                                               (16, 512, 3), (17, 1024, 7), (300, 3328, 4),
                                               (333, 3072, 8)])   # 384 lanes: decode-once only
def test_q4_batched_decode_once(fmt, rows, hidden, batch):
    g = synth.rng(1010, fmt, rows, hidden, batch)
    W = synth.matrix(fmt, g, rows, hidden)
    x = synth.normal_vector(g, hidden, batch=batch)
    y = run_matvec(fmt, W, x, rows, hidden, batch=batch, split_k=0)
    ref, bound = oracle.matvec(fmt, W, rows, hidden, x, threads=THREADS)
    assert_bound(y, ref, bound, what=f"{FMT_NAME[fmt]} {rows}x{hidden} batch {batch}")


@pytest.mark.parametrize("fmt", [oracle.Q4_0, oracle.Q4_K])
def test_q4_batched_scales_and_dynamic_range(fmt):
    # vectors at very different magnitudes (each gets its own power-of-two
    # scale), one all-zero vector and wide dynamic range inside a vector
    rows, hidden, batch = 500, 2560, 6
    g = synth.rng(1011, fmt)
    W = synth.matrix(fmt, g, rows, hidden)
    x = synth.normal_vector(g, hidden, batch=batch)
    x[0] *= 1e-20
    x[1] *= 3e15
    x[2] = 0.0
    x[3] *= np.exp(g.uniform(-8, 8, hidden)).astype(np.float32)
    x[4, :7] = 65504.0 * 4
    y = run_matvec(fmt, W, x, rows, hidden, batch=batch, split_k=0)
    ref, bound = oracle.matvec(fmt, W, rows, hidden, x)
    assert np.all(y[2] == 0.0)
    assert_bound(y, ref, bound, what="scales")


def test_q4_0_batched_is_run_to_run_identical():
    rows, hidden, batch = 2049, 2560, 8
    g = synth.rng(1012)
    Wd = dev(synth.q4_0_matrix(g, rows, hidden))
    xd = dev(synth.normal_vector(g, hidden, batch=batch))
    a = host(ops.q4_0_matvec(Wd, xd, rows, hidden, batch, 0))
    b = host(ops.q4_0_matvec(Wd, xd, rows, hidden, batch, 0))
    assert np.array_equal(a, b)
