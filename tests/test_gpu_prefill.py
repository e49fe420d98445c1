"""GPU parity for the prefill product (infer-compute README §Architecture,
prefill_q4: seq > 1) on the tensor cores, through the C ABI, against the
oracle's batch matvec (the same definition, y[n][r] = sum_k w[r][k] x[n][k],
in f64).

Tolerance, derived from the arithmetic: each weight (after its f32
dequantization) and each activation is rounded once to f16 (relative error
<= 2^-11 each for normal values, absolute <= 2^-25 in the f16 subnormal
range); the products are exact in f32 and summed in f32 (<= K * 2^-24
relative to sum |w x|).  So per output
  |y - y_ref| <= (2^-10 + 2^-21 + K * 2^-24) * sum_k |w x|
                 + 2^-25 * (sum_k |w| * max|x|... bounded here by
                   2^-25 * (sum_k |w| + sum_k |x|) * max(|w|, |x|))
and the tests use (2^-10 + K * 2^-24 + 2^-20) * bound + 2^-24 * (sum|w| + sum|x|) * 64.
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
    wabs = np.abs(oracle.dequant(oracle.Q4_K, W, rows, K)[sel]).sum(axis=1)      # [sel]
    xabs = np.abs(X.astype(np.float64)).reshape(N, K).sum(axis=1)              # [N]
    tol = (2.0 ** -10 + K * 2.0 ** -24 + 2.0 ** -20) * bound \
        + 2.0 ** -24 * 64 * (wabs[None, :] + xabs[:, None])
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


def test_prefill_two_accumulators_odd_token_tiles():
    # 76 row tiles x 3 token tiles: on 152 SMs the two-accumulator kernel
    # (two token tiles per CTA) saves a wave, and its second pair is half
    # padding (a zero token tile)
    rows, K, N = 76 * 128, 1024, 600
    g = synth.rng(W_PF, 5)
    W = synth.q4_k_matrix(g, rows, K)
    X = synth.normal_vector(g, K, N)
    sel = np.concatenate([np.arange(0, 140), np.arange(4800, 4900), np.arange(rows - 140, rows)])
    check_prefill(W, X, rows, K, N, rows_sel=sel)


def test_prefill_matches_matvec_per_token_within_f16_rounding():
    # every token of the prefill equals the batch-1 matvec of that token up to
    # the f16 operand rounding (a property at any size)
    rows, K, N = 512, 2560, 40
    g = synth.rng(W_PF, 3)
    W = synth.q4_k_matrix(g, rows, K)
    X = synth.normal_vector(g, K, N)
    Wd, Xd = dev(W), dev(X)
    Y = ops.q4k_prefill_matmul(Wd, Xd, rows, K, N).cpu().numpy()
    for n in (0, 17, N - 1):
        y1 = ops.q4k_matvec(Wd, Xd[n].contiguous(), rows, K).cpu().numpy()
        _, bound = oracle.matvec(oracle.Q4_K, W, rows, K, X[n])
        assert np.all(np.abs(Y[n] - y1) <= 2.0 ** -9 * bound + 1e-6)


def test_prefill_is_run_to_run_identical():
    rows, K, N = 384, 1024, 300
    g = synth.rng(W_PF, 4)
    W, X = dev(synth.q4_k_matrix(g, rows, K)), dev(synth.normal_vector(g, K, N))
    a = ops.q4k_prefill_matmul(W, X, rows, K, N).cpu().numpy()
    b = ops.q4k_prefill_matmul(W, X, rows, K, N).cpu().numpy()
    assert np.array_equal(a, b)
