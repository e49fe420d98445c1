"""GPU parity of the decode chain (qws_decode_chain) against the oracle.

Layer tolerance, from the step tolerances: a layer adds two branches to h,
a = post-attention branch and b = post-FFN branch, each an RMS-normalised
matvec output.  A branch's matvec output carries at most the FFN's 1e-4
relative error per element (the plain projections' 1e-5 * sum|w x| is
smaller); the RMS norm divides by rms(.) of the whole vector, so a relative
error e in every element moves the normalised element by at most e * |a_i|
plus e * rms(a) through the scale; the input norms feed the next matvec with
1e-5 relative error, inside the same budget; the two f32 residual adds round
by 2^-24 (|h| + |a| + |b|) at most.  Per element:
    |h'_gpu - h'_ref| <= 1e-4 * (|h| + |a| + |b|) + 1e-4 * (rms(a) + rms(b))
checked teacher-forced: the oracle runs each layer on the GPU's input to that
layer.  One launch over L layers must equal L single-layer launches bit for bit
(the kernel is deterministic), and the end-to-end relative L2 error against the
oracle is reported and bounded.
"""
import os

import numpy as np
import pytest
import torch

import oracle
from quantized_weight_streaming_q4k_gb300 import build, ops, synth

pytestmark = pytest.mark.gpu

SMALL = dict(hidden=512, inter=1024, n_q_heads=4, n_kv_heads=2, head_dim=128, eps=1e-6,
             post_norms=1)


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    torch.cuda.set_device(0)
    yield
    assert ops.device_error() == 0


def to_dev(L):
    out = {}
    for k, v in L.items():
        out[k] = torch.from_numpy(np.ascontiguousarray(v)).cuda() if isinstance(v, np.ndarray) else v
    return out


def check_layer(h_in, h_gpu, L, dims):
    ref, tr = oracle.layer_forward(L, dims, h_in, trace=True)
    h = h_in.astype(np.float64)
    a = tr["h1"] - h                      # post-attention branch (normed o, or o)
    b = ref - tr["h1"]                    # post-FFN branch
    tol = 1e-4 * (np.abs(h) + np.abs(a) + np.abs(b)) + 1e-4 * (
        np.sqrt(np.mean(a * a)) + np.sqrt(np.mean(b * b)))
    err = np.abs(h_gpu.astype(np.float64) - ref)
    assert np.all(err <= tol), f"worst err/tol {np.max(err / tol):.3e}"
    return float(np.max(err / tol)), ref


def run_chain(layers_dev, h0, dims):
    h = torch.from_numpy(h0.copy()).cuda()
    ops.decode_chain(layers_dev, h, dims)
    torch.cuda.synchronize()
    return h.cpu().numpy()


@pytest.mark.parametrize("post_norms", [1, 0])
@pytest.mark.parametrize("fmt_down", [oracle.Q6_K, oracle.Q4_K])
def test_chain_small_teacher_forced(post_norms, fmt_down):
    dims = dict(SMALL, post_norms=post_norms)
    n = 3
    layers = [synth.chain_layer(l, dims, fmt_down=fmt_down, workload=50 + post_norms) for l in range(n)]
    ldev = [to_dev(L) for L in layers]
    h0 = synth.normal_vector(synth.rng(51, post_norms), dims["hidden"])
    h = h0
    outs = []
    for l in range(n):
        hg = run_chain([ldev[l]], h, dims)
        check_layer(h, hg, layers[l], dims)
        outs.append(hg)
        h = hg
    # one launch over n layers == n single-layer launches, bit for bit
    hall = run_chain(ldev, h0, dims)
    assert np.array_equal(hall, outs[-1])
    # run-to-run identical
    assert np.array_equal(run_chain(ldev, h0, dims), hall)


# hidden above 8 * 320 takes the wide prologue (16 values per thread in the
# residual / norm step), a separate kernel instantiation.
WIDE = dict(hidden=4096, inter=4096, n_q_heads=8, n_kv_heads=4, head_dim=256, eps=1e-6,
            post_norms=1)


def test_chain_wide_hidden_teacher_forced():
    dims = WIDE
    n = 2
    layers = [synth.chain_layer(l, dims, fmt_down=oracle.Q6_K, workload=56) for l in range(n)]
    ldev = [to_dev(L) for L in layers]
    h0 = synth.normal_vector(synth.rng(57), dims["hidden"])
    h = h0
    outs = []
    for l in range(n):
        hg = run_chain([ldev[l]], h, dims)
        check_layer(h, hg, layers[l], dims)
        outs.append(hg)
        h = hg
    assert np.array_equal(run_chain(ldev, h0, dims), outs[-1])


# Fewer 16-byte row groups than CTAs in the down phase (Q6_K rows of 256
# columns are 210 B: 8-row groups, 32 of them): most CTAs own no rows there and
# still take part in every phase's synchronisation.
TINY = dict(hidden=256, inter=256, n_q_heads=2, n_kv_heads=1, head_dim=128, eps=1e-6,
            post_norms=1)


def test_chain_tiny_idle_ctas():
    dims = TINY
    n = 5
    layers = [synth.chain_layer(l, dims, fmt_down=oracle.Q6_K, workload=54) for l in range(n)]
    ldev = [to_dev(L) for L in layers]
    h0 = synth.normal_vector(synth.rng(55), dims["hidden"])
    h = h0
    outs = []
    for l in range(n):
        hg = run_chain([ldev[l]], h, dims)
        check_layer(h, hg, layers[l], dims)
        outs.append(hg)
        h = hg
    hall = run_chain(ldev, h0, dims)
    assert np.array_equal(hall, outs[-1])


def test_chain_64_layers_one_launch():
    """The most layers one launch takes (64: stamps up to 4 * 64, one
    prologue counter per phase): equal bit for bit to 64 single-layer
    launches, and close to the oracle end to end."""
    dims = TINY
    n = 64
    layers = [synth.chain_layer(l, dims, fmt_down=oracle.Q6_K, workload=61) for l in range(n)]
    ldev = [to_dev(L) for L in layers]
    h0 = synth.normal_vector(synth.rng(62), dims["hidden"])
    h = h0
    for l in range(n):
        h = run_chain([ldev[l]], h, dims)
    hall = run_chain(ldev, h0, dims)
    assert np.array_equal(hall, h)
    ref = h0.astype(np.float64)
    for L in layers:
        ref = oracle.layer_forward(L, dims, ref)
    rel = np.linalg.norm(hall - ref) / np.linalg.norm(ref)
    print(f"chain tiny 64 layers: relative L2 error {rel:.2e}")
    assert rel < 1e-3


def test_chain_small_end_to_end():
    dims = SMALL
    n = 4
    layers = [synth.chain_layer(l, dims, workload=52) for l in range(n)]
    ldev = [to_dev(L) for L in layers]
    h0 = synth.normal_vector(synth.rng(53), dims["hidden"])
    hg = run_chain(ldev, h0, dims)
    ref = h0.astype(np.float64)
    for L in layers:
        ref = oracle.layer_forward(L, dims, ref)
    rel = np.linalg.norm(hg - ref) / np.linalg.norm(ref)
    print(f"chain small 4 layers: relative L2 error {rel:.2e}")
    assert rel < 1e-4


def test_chain_full_size_gemma3_4b():
    """34 Gemma-3-4B-shaped layers: teacher-forced parity on layers 0, 1, 33,
    bit-exact equality of one 34-layer launch with 34 single-layer launches,
    and end-to-end relative L2 error against the oracle."""
    dims = synth.GEMMA3_4B
    n = 34
    layers = [synth.chain_layer(l, dims) for l in range(n)]
    ldev = [to_dev(L) for L in layers]
    h0 = synth.normal_vector(synth.rng(synth.W_CHAIN, 99), dims["hidden"])
    hs = [h0]
    for l in range(n):
        hs.append(run_chain([ldev[l]], hs[-1], dims))
    worst = []
    for l in (0, 1, n - 1):
        w, _ = check_layer(hs[l], hs[l + 1], layers[l], dims)
        worst.append(w)
    hall = run_chain(ldev, h0, dims)
    assert np.array_equal(hall, hs[-1])
    ref = h0.astype(np.float64)
    for L in layers:
        ref = oracle.layer_forward(L, dims, ref)
    rel = np.linalg.norm(hall - ref) / np.linalg.norm(ref)
    print(f"chain 34 layers: worst teacher-forced err/tol {max(worst):.3e}, "
          f"end-to-end relative L2 {rel:.2e}")
    assert rel < 1e-3


@pytest.mark.parametrize("shape", ["small", "small_pre_norms", "wide", "gemma3_4b"])
def test_chain_final_norm(shape):
    """qws_decode_chain_final_norm: h bit-identical to qws_decode_chain's, and
    hn = rms_norm(h, w_final) within the norm's 1e-5 relative bound against the
    oracle's norm of the GPU's h (the narrow and the wide keeper step, without
    the post norms, and the Gemma-3-4B hidden size)."""
    dims, n = {"small": (SMALL, 3), "small_pre_norms": (dict(SMALL, post_norms=0), 2),
               "wide": (WIDE, 2), "gemma3_4b": (synth.GEMMA3_4B, 2)}[shape]
    fmt = oracle.Q4_K if shape == "small_pre_norms" else oracle.Q6_K
    layers = [synth.chain_layer(l, dims, fmt_down=fmt, workload=58) for l in range(n)]
    ldev = [to_dev(L) for L in layers]
    H = dims["hidden"]
    h0 = synth.normal_vector(synth.rng(59, H), H)
    w = synth.norm_weights(synth.rng(60, H), H)
    plain = run_chain(ldev, h0, dims)
    h = torch.from_numpy(h0.copy()).cuda()
    hn = torch.full((H,), float("nan"), device="cuda")
    ops.decode_chain(ldev, h, dims, w_final=torch.from_numpy(w).cuda(), hn=hn)
    torch.cuda.synchronize()
    hg, hng = h.cpu().numpy(), hn.cpu().numpy()
    assert np.array_equal(hg, plain)
    ref = oracle.rms_norm(hg, w, dims["eps"])
    assert np.all(np.abs(hng - ref) <= 1e-5 * np.abs(ref) + 1e-30)


def test_chain_then_dependent_matvec_without_sync():
    """The chain lets the next kernel start as its CTAs exit; a Q4_0 matvec
    launched right after it (no host synchronisation) must read the final
    norm the chain wrote: its logits equal, bit for bit, those of the same
    matvec run after a device synchronise, over several back-to-back steps
    with different inputs."""
    dims = SMALL
    n = 2
    H = dims["hidden"]
    layers = [to_dev(synth.chain_layer(l, dims, workload=63)) for l in range(n)]
    w = torch.from_numpy(synth.norm_weights(synth.rng(64), H)).cuda()
    V = 4096
    W = torch.from_numpy(synth.q4_0_matrix(synth.rng(65), V, H)).cuda()
    hs = [torch.from_numpy(synth.normal_vector(synth.rng(66, i), H)).cuda() for i in range(3)]
    hn = torch.empty(H, device="cuda")
    outs = []
    for h0 in hs:
        h = h0.clone()
        ops.decode_chain(layers, h, dims, w_final=w, hn=hn)
        outs.append(ops.q4_0_matvec(W, hn, V, H))
    torch.cuda.synchronize()
    for h0, y in zip(hs, outs):
        h = h0.clone()
        hn2 = torch.empty(H, device="cuda")
        ops.decode_chain(layers, h, dims, w_final=w, hn=hn2)
        torch.cuda.synchronize()
        y2 = ops.q4_0_matvec(W, hn2, V, H)
        torch.cuda.synchronize()
        assert torch.equal(y, y2)


def test_chain_rejects_bad_arguments():
    dims = dict(SMALL)
    L = to_dev(synth.chain_layer(0, dims))
    h = torch.zeros(dims["hidden"], device="cuda")
    with pytest.raises(ops.QwsError):
        ops.decode_chain([L], h, dict(dims, hidden=500))
    with pytest.raises(ops.QwsError):
        ops.decode_chain([dict(L, fmt_qkv=oracle.Q6_K)], h, dims)
    with pytest.raises(ops.QwsError):
        ops.decode_chain([L], h, dict(dims, n_q_heads=3))
