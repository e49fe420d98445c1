"""GPU parity for the prefill product (infer-compute README §Architecture,
prefill_q4: seq > 1) on the tensor cores, through the C ABI, against the
oracle's batch matvec (the same definition, y[n][r] = sum_k w[r][k] x[n][k],
in f64).

Tolerance: the matvecs' bound, |y - y_ref| <= 1e-5 * sum_k |w x| per output.
The kernel splits each operand into two f16 parts (the weight scaled by 2^10,
each token by its own power of two), so each operand keeps 22 bits and each
product is within ~3 * 2^-22 of exact, plus one f32 rounding per 16-column MMA
in the two tensor-memory accumulators: far inside the bound.
"""
import os

import numpy as np
import pytest
import torch

import oracle
from quantized_weight_streaming_q4k_gb300 import build, ops, synth

pytestmark = pytest.mark.gpu
THREADS = max(1, min(16, os.cpu_count() or 1))
W_PF = 50          # workload id of this file's seeds


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    torch.cuda.set_device(0)
    yield
    assert ops.device_error() == 0


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def check_prefill(W, X, rows, K, N, rows_sel=None):
    Y = ops.q4k_prefill_matmul(dev(W), dev(X), rows, K, N).cpu().numpy().astype(np.float64)
    assert Y.shape == (N, rows)
    if rows_sel is None:
        ref, bound = oracle.matvec(oracle.Q4_K, W, rows, K, X, threads=THREADS)
        sel = np.arange(rows)
    else:
        sel = np.asarray(rows_sel)
        ref = np.full((N, rows), np.nan)
        bound = np.full((N, rows), np.nan)
        for a in sel:
            r1, b1 = oracle.matvec(oracle.Q4_K, W, rows, K, X, row_begin=int(a), row_end=int(a) + 1)
            ref[:, a] = r1.reshape(N, rows)[:, a]
            bound[:, a] = b1.reshape(N, rows)[:, a]
    ref, bound = ref.reshape(N, rows)[:, sel], bound.reshape(N, rows)[:, sel]
    tol = 1e-5 * bound
    err = np.abs(Y[:, sel] - ref)
    bad = err > tol
    assert not bad.any(), (f"{np.count_nonzero(bad)} of {bad.size} outside; worst err/bound "
                           f"{np.max(err / np.maximum(bound, 1e-300)):.3e}; first "
                           f"{np.argwhere(bad)[:4].tolist()}")
    return Y


@pytest.mark.parametrize("rows,K,N", [(128, 256, 1), (128, 256, 8), (128, 512, 256),
                                      (300, 512, 300), (77, 2560, 33), (1000, 1024, 513)])
def test_prefill_parity_small(rows, K, N):
    g = synth.rng(W_PF, 1, rows, K, N)
    W = synth.q4_k_matrix(g, rows, K)
    X = synth.normal_vector(g, K, N)
    check_prefill(W, X, rows, K, N)


def test_prefill_gemma_gate_shape_sampled_rows():
    # gate/up shape of the Gemma-3-4B FFN at 512 prompt tokens
    rows, K, N = 10240, 2560, 512
    g = synth.rng(W_PF, 2)
    W = synth.q4_k_matrix(g, rows, K)
    X = synth.normal_vector(g, K, N)
    sel = np.concatenate([np.arange(0, 130), np.arange(5000, 5040), np.arange(rows - 130, rows)])
    check_prefill(W, X, rows, K, N, rows_sel=sel)


def test_prefill_odd_token_tiles_sampled_rows():
    # 76 row tiles x 3 token tiles, the last one mostly padding
    rows, K, N = 76 * 128, 1024, 600
    g = synth.rng(W_PF, 5)
    W = synth.q4_k_matrix(g, rows, K)
    X = synth.normal_vector(g, K, N)
    sel = np.concatenate([np.arange(0, 140), np.arange(4800, 4900), np.arange(rows - 140, rows)])
    check_prefill(W, X, rows, K, N, rows_sel=sel)


@pytest.mark.parametrize("scale", [1e-6, 1e-2, 37.0, 1e4])
def test_prefill_activation_scales(scale):
    # the per-token power-of-two scaling keeps the split exact at any
    # activation magnitude
    rows, K, N = 256, 1024, 20
    g = synth.rng(W_PF, 6, int(np.log10(scale) + 10))
    W = synth.q4_k_matrix(g, rows, K)
    X = (synth.normal_vector(g, K, N) * np.float32(scale)).astype(np.float32)
    check_prefill(W, X, rows, K, N)


def test_prefill_tokens_of_very_different_magnitudes():
    # one tile of tokens whose magnitudes span 2^-40 .. 2^30: each token keeps
    # its own scale
    rows, K, N = 256, 512, 64
    g = synth.rng(W_PF, 7)
    W = synth.q4_k_matrix(g, rows, K)
    X = synth.normal_vector(g, K, N)
    X *= np.float32(2.0) ** np.linspace(-40, 30, N, dtype=np.float32)[:, None].astype(np.float32)
    X[5] = 0.0          # an all-zero token
    check_prefill(W, X.astype(np.float32), rows, K, N)


def test_prefill_flags_weights_outside_the_split_range():
    # |w| >= 64 cannot be split into f16 after the 2^10 pre-scale: the kernel
    # records the range error (code 256) instead of returning silently
    rows, K, N = 128, 256, 4
    g = synth.rng(W_PF, 8)
    W = synth.q4_k_matrix(g, rows, K, d_range=(8.0, 8.0))   # d * sc * q up to 8 * 63 * 15
    X = synth.normal_vector(g, K, N)
    ops.q4k_prefill_matmul(dev(W), dev(X), rows, K, N)
    torch.cuda.synchronize()
    assert ops.device_error() & 256


def test_prefill_matches_matvec_per_token():
    # every token of the prefill equals the batch-1 matvec of that token within
    # the sum of their tolerances (a property at any size)
    rows, K, N = 512, 2560, 40
    g = synth.rng(W_PF, 3)
    W = synth.q4_k_matrix(g, rows, K)
    X = synth.normal_vector(g, K, N)
    Wd, Xd = dev(W), dev(X)
    Y = ops.q4k_prefill_matmul(Wd, Xd, rows, K, N).cpu().numpy()
    for n in (0, 17, N - 1):
        y1 = ops.q4k_matvec(Wd, Xd[n].contiguous(), rows, K).cpu().numpy()
        _, bound = oracle.matvec(oracle.Q4_K, W, rows, K, X[n])
        assert np.all(np.abs(Y[n] - y1) <= 2e-5 * bound)


def test_prefill_is_run_to_run_identical():
    rows, K, N = 384, 1024, 300
    g = synth.rng(W_PF, 4)
    W, X = dev(synth.q4_k_matrix(g, rows, K)), dev(synth.normal_vector(g, K, N))
    a = ops.q4k_prefill_matmul(W, X, rows, K, N).cpu().numpy()
    b = ops.q4k_prefill_matmul(W, X, rows, K, N).cpu().numpy()
    assert np.array_equal(a, b)
