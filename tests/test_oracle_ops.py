"""Pins for the oracle's matvec, activation, norm, attention, FFN, layer and
top-k functions (CPU only).  Each check uses something other than the oracle
itself: closed forms, library routines on special cases, exact identities or
brute force on tiny inputs."""
import math

import numpy as np
import pytest

import oracle
from quantized_weight_streaming_q4k_gb300 import synth

FMTS = [oracle.Q4_0, oracle.Q4_K, oracle.Q6_K]


def kahan_sum(terms):
    s, c = 0.0, 0.0
    for t in terms:
        y = t - c
        u = s + y
        c = (u - s) - y
        s = u
    return s


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("rows,hidden", [(1, 256), (4, 512)])
def test_matvec_brute_force(fmt, rows, hidden):
    g = synth.rng(7, fmt, rows)
    W = synth.matrix(fmt, g, rows, hidden)
    x = synth.normal_vector(g, hidden)
    y, bound = oracle.matvec(fmt, W, rows, hidden, x)
    dense = oracle.dequant(fmt, W, rows, hidden)
    for r in range(rows):
        terms = [float(dense[r, i]) * float(x[i]) for i in range(hidden)]
        ref = kahan_sum(terms)
        mag = kahan_sum([abs(t) for t in terms])
        assert abs(y[r] - ref) <= 1e-13 * mag
        assert abs(bound[r] - mag) <= 1e-13 * mag


@pytest.mark.parametrize("fmt", FMTS)
def test_matvec_equals_dense_matmul(fmt):
    rows, hidden = 37, 1024
    g = synth.rng(8, fmt)
    W = synth.matrix(fmt, g, rows, hidden)
    x = synth.normal_vector(g, hidden, batch=3)
    y, bound = oracle.matvec(fmt, W, rows, hidden, x)
    dense = oracle.dequant(fmt, W, rows, hidden)
    ref = x.astype(np.float64) @ dense.T
    assert np.all(np.abs(y - ref) <= 1e-12 * bound)
    assert np.allclose(bound, np.abs(x.astype(np.float64)) @ np.abs(dense.T), rtol=1e-12)


@pytest.mark.parametrize("fmt", FMTS)
def test_matvec_one_hot_picks_a_column(fmt):
    rows, hidden = 5, 512
    W = synth.matrix(fmt, synth.rng(9, fmt), rows, hidden)
    dense = oracle.dequant(fmt, W, rows, hidden)
    for i in (0, 1, 31, 32, 255, 256, 511):
        x = np.zeros(hidden, dtype=np.float32)
        x[i] = 1.0
        y, _ = oracle.matvec(fmt, W, rows, hidden, x)
        assert np.array_equal(y, dense[:, i])


def test_matvec_row_split_threads_identical():
    rows, hidden = 64, 512
    W = synth.q4_k_matrix(synth.rng(10), rows, hidden)
    x = synth.normal_vector(synth.rng(11), hidden)
    y1, b1 = oracle.matvec(oracle.Q4_K, W, rows, hidden, x, threads=1)
    y4, b4 = oracle.matvec(oracle.Q4_K, W, rows, hidden, x, threads=4)
    assert np.array_equal(y1, y4) and np.array_equal(b1, b4)


def test_q4_k_closed_form_constant_quants():
    # all nibbles = c: y = sum_s (d*sc_s*c - dmin*m_s) * sum(x over sub-block s)
    scales = [63, 0, 33, 17, 48, 21, 62, 5]
    mins = [5, 63, 16, 47, 32, 9, 60, 1]
    b = np.zeros(144, dtype=np.uint8)
    b[0:2] = np.array([0.0078125], dtype=np.float16).view(np.uint8)      # d = 2^-7
    b[2:4] = np.array([0.01171875], dtype=np.float16).view(np.uint8)     # dmin = 3*2^-8
    b[4:16] = np.frombuffer(bytes.fromhex("ff40e111853fd02f0095ce15"), dtype=np.uint8)
    c = 11
    b[16:] = c | (c << 4)
    x = synth.normal_vector(synth.rng(12), 256).astype(np.float64)
    y, _ = oracle.matvec(oracle.Q4_K, b, 1, 256, x)
    # sub-block s covers weights 64*(s//2) + 32*(s%2) + [0, 32)
    ref = 0.0
    for s in range(8):
        lo = 64 * (s // 2) + 32 * (s % 2)
        ref += (0.0078125 * scales[s] * c - 0.01171875 * mins[s]) * math.fsum(x[lo:lo + 32])
    assert abs(y[0] - ref) <= 1e-13 * np.sum(np.abs(x)) * 10


def test_q4_k_textbook_dot_special_case():
    # scales 1, mins 0 -> y = d * sum(q * x): a plain dot product
    g = synth.rng(13)
    b = synth.q4_k_matrix(g, 1, 256).reshape(144)
    b[4:8] = 1
    b[8:12] = 0
    b[12:16] = 1
    q = np.empty(256)
    for c in range(4):
        for l in range(32):
            q[64 * c + l] = b[16 + 32 * c + l] & 15
            q[64 * c + 32 + l] = b[16 + 32 * c + l] >> 4
    x = synth.normal_vector(g, 256).astype(np.float64)
    d = float(b[0:2].view(np.float16)[0])
    y, _ = oracle.matvec(oracle.Q4_K, b, 1, 256, x)
    assert abs(y[0] - d * np.dot(q, x)) <= 1e-13 * d * np.dot(q, np.abs(x))


def test_q4_0_offset_eight_is_zero():
    W = np.tile(np.r_[np.frombuffer(np.float16(1.5).tobytes(), dtype=np.uint8),
                      np.full(16, 0x88, dtype=np.uint8)], 8)
    x = synth.normal_vector(synth.rng(14), 256)
    y, b = oracle.matvec(oracle.Q4_0, W, 1, 256, x)
    assert y[0] == 0.0 and b[0] == 0.0


# ---------------------------------------------------------------- GELU (tanh)
def test_gelu_tanh_identities():
    assert oracle.gelu_tanh(0.0) == 0.0
    for t in (0.1, 0.5, 1.0, 2.5, 7.0, 30.0):
        # tanh is odd  =>  gelu(t) - gelu(-t) = t exactly (up to f64 rounding)
        assert abs(oracle.gelu_tanh(t) - oracle.gelu_tanh(-t) - t) <= 4e-16 * max(1.0, t)
    assert oracle.gelu_tanh(40.0) == 40.0
    assert oracle.gelu_tanh(-40.0) == 0.0 or abs(oracle.gelu_tanh(-40.0)) < 1e-300


def test_gelu_tanh_close_to_erf_gelu():
    # The tanh form approximates x*Phi(x); its largest error is a few 1e-4.
    ts = np.linspace(-8, 8, 4001)
    got = oracle.gelu_tanh(ts)
    ref = np.array([0.5 * t * (1.0 + math.erf(t / math.sqrt(2.0))) for t in ts])
    err = np.max(np.abs(got - ref))
    assert err < 1e-3
    assert err > 1e-5   # and it is the tanh form, not the erf form itself


def test_gelu_tanh_matches_independent_tanh_gelu():
    # Pins both constants (sqrt(2/pi) and 0.044715) of the tanh form.  The
    # oracle is compared at 241 points of [-6, 6] (the curved region included)
    # with two implementations written elsewhere: torch's float64
    # gelu(approximate="tanh"), and the logistic identity
    # 0.5 (1 + tanh z) = 1 / (1 + exp(-2 z)) evaluated with Python's math.
    # The bound is relative to |t| (|gelu(t)| <= |t|): in the negative tail the
    # output is a difference of nearly equal terms, where libm rounding, not
    # the constants, sets its relative error.  A change of either constant in
    # its 4th significant digit moves gelu by > 1e-6 |t| near |t| = 2.
    torch = pytest.importorskip("torch")
    ts = np.linspace(-6.0, 6.0, 241)
    got = oracle.gelu_tanh(ts)
    ref_torch = torch.nn.functional.gelu(torch.from_numpy(ts), approximate="tanh").numpy()
    k = math.sqrt(2.0 / math.pi)
    ref_logistic = np.array([t / (1.0 + math.exp(-2.0 * k * (t + 0.044715 * t ** 3))) for t in ts])
    scale = np.maximum(np.abs(ts), 1e-300)
    assert np.max(np.abs(got - ref_torch) / scale) <= 1e-14
    assert np.max(np.abs(got - ref_logistic) / scale) <= 1e-14


def test_gelu_tanh_derivative_at_zero_is_half():
    h = 1e-6
    assert abs((oracle.gelu_tanh(h) - oracle.gelu_tanh(-h)) / (2 * h) - 0.5) < 1e-9


def test_silu_identities_and_logistic():
    # silu(t) = t * logistic(t): silu(t) - silu(-t) = t; silu(0) = 0; slope 1/2 at 0
    from scipy.special import expit
    assert oracle.silu(0.0) == 0.0
    for t in (0.1, 0.5, 1.0, 2.5, 7.0, 30.0):
        assert abs(oracle.silu(t) - oracle.silu(-t) - t) <= 4e-16 * max(1.0, t)
    ts = np.linspace(-30, 30, 601)
    assert np.allclose(oracle.silu(ts), ts * expit(ts), rtol=1e-14, atol=1e-300)
    h = 1e-6
    assert abs((oracle.silu(h) - oracle.silu(-h)) / (2 * h) - 0.5) < 1e-9
    assert oracle.silu(-800.0) == 0.0 or abs(oracle.silu(-800.0)) < 1e-300


def test_ffn_silu_matches_dense_composition():
    hidden, inter = 256, 512
    g = synth.rng(22)
    Wg = synth.q4_k_matrix(g, inter, hidden)
    Wu = synth.q4_k_matrix(g, inter, hidden)
    Wd = synth.q6_k_matrix(g, hidden, inter)
    x = synth.unit_rms_vector(g, hidden).astype(np.float64)
    out = oracle.ffn(oracle.Q4_K, Wg, Wu, oracle.Q6_K, Wd, hidden, inter, x, act=oracle.ACT_SILU)
    gd = oracle.dequant(oracle.Q4_K, Wg, inter, hidden) @ x
    ud = oracle.dequant(oracle.Q4_K, Wu, inter, hidden) @ x
    m = gd / (1.0 + np.exp(-gd)) * ud
    Dd = oracle.dequant(oracle.Q6_K, Wd, hidden, inter)
    assert np.allclose(out["m"], m, rtol=1e-12, atol=1e-300)
    assert np.all(np.abs(out["y"] - Dd @ m) <= 1e-11 * (np.abs(Dd) @ np.abs(m)))


def test_residual_rms_norm_is_add_then_norm():
    n, eps = 2560, 1e-6
    g = synth.rng(23)
    h = synth.normal_vector(g, n).astype(np.float64)
    y = synth.normal_vector(g, n).astype(np.float64)
    w = synth.norm_weights(g, n).astype(np.float64)
    h2, x = oracle.residual_rms_norm(h, y, w, eps)
    assert np.array_equal(h2, h + y)
    r = h + y
    assert np.allclose(x, r / np.sqrt(np.mean(r * r) + eps) * w, rtol=1e-14)


# ---------------------------------------------------------------- rms_norm
def test_rms_norm_one_hot_and_constant():
    n, eps = 2560, 1e-6
    w = synth.norm_weights(synth.rng(15), n).astype(np.float64)
    x = np.zeros(n)
    x[17] = 3.0
    y = oracle.rms_norm(x, w, eps)
    assert abs(y[17] - 3.0 / math.sqrt(9.0 / n + eps) * w[17]) <= 1e-15 * abs(y[17])
    assert np.count_nonzero(y) == 1
    # eps shifts it by a relative eps*n/(2*9) = 1.4e-4
    assert abs(y[17] / w[17] / math.sqrt(n) - 1.0) < 2e-4
    c = -0.25
    y = oracle.rms_norm(np.full(n, c), w, eps)
    assert np.allclose(y, -w * 0.25 / math.sqrt(0.0625 + eps), rtol=1e-15, atol=0)


def test_rms_norm_scale_invariance_and_unit_rms():
    n = 1000
    x = synth.normal_vector(synth.rng(16), n).astype(np.float64)
    ones = np.ones(n)
    y = oracle.rms_norm(x, ones, 0.0)
    assert abs(np.sqrt(np.mean(y * y)) - 1.0) < 1e-14
    y2 = oracle.rms_norm(1024.0 * x, ones, 0.0)
    assert np.allclose(y, y2, rtol=1e-14, atol=0)
    assert np.array_equal(oracle.rms_norm(np.zeros(8), np.ones(8), 1e-6), np.zeros(8))


def test_residual_add_exact():
    h = synth.normal_vector(synth.rng(17), 300).astype(np.float64)
    y = synth.normal_vector(synth.rng(18), 300).astype(np.float64)
    assert np.array_equal(oracle.residual_add(h, y), h + y)


# ---------------------------------------------------------------- attention
def test_attention_seq1_equals_single_key_softmax_attention():
    nq, nkv, hd = 8, 4, 256
    g = synth.rng(19)
    q = g.standard_normal(nq * hd)
    k = g.standard_normal(nkv * hd)
    v = g.standard_normal(nkv * hd)
    got = oracle.attn_seq1(v, nq, nkv, hd)
    ref = np.empty(nq * hd)
    for h in range(nq):
        kv = h // (nq // nkv)
        score = np.array([np.dot(q[h * hd:(h + 1) * hd], k[kv * hd:(kv + 1) * hd]) / math.sqrt(hd)])
        p = np.exp(score - score.max())
        p /= p.sum()
        ref[h * hd:(h + 1) * hd] = p[0] * v[kv * hd:(kv + 1) * hd]
    assert np.array_equal(got, ref)


def test_attention_seq1_grouping_is_contiguous():
    v = np.arange(4 * 3, dtype=np.float64)
    got = oracle.attn_seq1(v, 8, 4, 3)
    assert list(got[:6]) == [0, 1, 2, 0, 1, 2] and list(got[6:12]) == [3, 4, 5, 3, 4, 5]


# ---------------------------------------------------------------- FFN
def test_ffn_matches_dense_composition():
    hidden, inter = 256, 512
    g = synth.rng(20)
    Wg = synth.q4_k_matrix(g, inter, hidden)
    Wu = synth.q4_k_matrix(g, inter, hidden)
    Wd = synth.q6_k_matrix(g, hidden, inter)
    x = synth.unit_rms_vector(g, hidden).astype(np.float64)
    out = oracle.ffn(oracle.Q4_K, Wg, Wu, oracle.Q6_K, Wd, hidden, inter, x)
    gd = oracle.dequant(oracle.Q4_K, Wg, inter, hidden) @ x
    ud = oracle.dequant(oracle.Q4_K, Wu, inter, hidden) @ x
    m = 0.5 * gd * (1 + np.tanh(math.sqrt(2 / math.pi) * (gd + 0.044715 * gd ** 3))) * ud
    Dd = oracle.dequant(oracle.Q6_K, Wd, hidden, inter)
    y = Dd @ m
    assert np.allclose(out["g"], gd, rtol=1e-12, atol=0)
    assert np.allclose(out["u"], ud, rtol=1e-12, atol=0)
    assert np.all(np.abs(out["y"] - y) <= 1e-11 * (np.abs(Dd) @ np.abs(m)))
    assert np.allclose(out["bound_y"], np.abs(Dd) @ np.abs(out["m"]), rtol=1e-12)


def test_ffn_zero_up_gives_zero():
    hidden, inter = 256, 256
    g = synth.rng(21)
    Wg = synth.q4_k_matrix(g, inter, hidden)
    Wu = synth.q4_k_matrix(g, inter, hidden, d_range=(0, 0), dmin_range=(0, 0))
    Wd = synth.q6_k_matrix(g, hidden, inter)
    out = oracle.ffn(oracle.Q4_K, Wg, Wu, oracle.Q6_K, Wd, hidden, inter,
                     synth.normal_vector(g, hidden))
    assert np.all(out["m"] == 0) and np.all(out["y"] == 0)


# ---------------------------------------------------------------- layer
SMALL = dict(hidden=512, inter=1024, n_q_heads=4, n_kv_heads=2, head_dim=128, eps=1e-6,
             post_norms=1)


def _zero_layer(dims):
    L = synth.chain_layer(0, dims)
    z = dict(d_range=(0, 0), dmin_range=(0, 0))
    H, I = dims["hidden"], dims["inter"]
    qd, kd = dims["n_q_heads"] * dims["head_dim"], dims["n_kv_heads"] * dims["head_dim"]
    g = synth.rng(22)
    L.update(Wq=synth.q4_k_matrix(g, qd, H, **z), Wk=synth.q4_k_matrix(g, kd, H, **z),
             Wv=synth.q4_k_matrix(g, kd, H, **z), Wo=synth.q4_k_matrix(g, H, qd, **z),
             Wg=synth.q4_k_matrix(g, I, H, **z), Wu=synth.q4_k_matrix(g, I, H, **z),
             Wd=synth.q6_k_matrix(g, H, I, d_range=(0, 0)))
    return L


@pytest.mark.parametrize("post_norms", [0, 1])
def test_layer_with_zero_weights_is_identity(post_norms):
    dims = dict(SMALL, post_norms=post_norms)
    h = synth.normal_vector(synth.rng(23), dims["hidden"])
    out = oracle.layer_forward(_zero_layer(dims), dims, h)
    assert np.array_equal(out, h.astype(np.float64))


@pytest.mark.parametrize("post_norms", [0, 1])
def test_layer_matches_dense_composition(post_norms):
    dims = dict(SMALL, post_norms=post_norms)
    H, I = dims["hidden"], dims["inter"]
    nq, nkv, hd = dims["n_q_heads"], dims["n_kv_heads"], dims["head_dim"]
    L = synth.chain_layer(1, dims)
    h = synth.normal_vector(synth.rng(24), H).astype(np.float64)
    out, tr = oracle.layer_forward(L, dims, h, trace=True)

    def rms(x, w):
        return x / np.sqrt(np.mean(x * x) + dims["eps"]) * w

    def dq(name, rows, cols):
        return oracle.dequant(oracle.Q4_K if name != "Wd" else oracle.Q6_K, L[name], rows, cols)

    n1 = rms(h, L["w_in"])
    v = dq("Wv", nkv * hd, H) @ n1
    a = np.concatenate([v[(i // (nq // nkv)) * hd:(i // (nq // nkv) + 1) * hd] for i in range(nq)])
    o = dq("Wo", H, nq * hd) @ a
    h1 = h + (rms(o, L["w_post_attn"]) if post_norms else o)
    n2 = rms(h1, L["w_pre_ffn"])
    gg, uu = dq("Wg", I, H) @ n2, dq("Wu", I, H) @ n2
    m = 0.5 * gg * (1 + np.tanh(math.sqrt(2 / math.pi) * (gg + 0.044715 * gg ** 3))) * uu
    f = dq("Wd", H, I) @ m
    ref = h1 + (rms(f, L["w_post_ffn"]) if post_norms else f)
    assert np.allclose(tr["o"], o, rtol=1e-10, atol=1e-12)
    assert np.allclose(tr["m"], m, rtol=1e-9, atol=1e-12)
    assert np.allclose(out, ref, rtol=1e-9, atol=1e-9)


# ---------------------------------------------------------------- top-k
def test_topk_matches_stable_argsort_with_ties():
    g = synth.rng(25)
    v = np.round(g.standard_normal(5000) * 3.0, 1)   # many exact ties
    for k in (1, 5, 17):
        ref = np.argsort(-v, kind="stable")[:k]
        assert list(oracle.topk(v, k)) == list(ref)
