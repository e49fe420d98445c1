"""GPU parity of the decode step over a KV cache (qws_decode_kv) against the
oracle's qo_layer_forward_kv.

Checked teacher-forced, one layer at a time: the oracle runs layer l on the
GPU's input to layer l and on the same cache contents (positions 0..pos-1
filled with seeded values, the same numbers in f32 and f64).

Layer tolerance, from the step tolerances: the layer adds two branches to h,
a = h1 - h (post-attention) and b = h' - h1 (post-FFN), each an RMS-normalised
matvec output.  The attention output carries the matvec error of q, k, v
(1e-5 * sum|w x|) plus its own (the score and softmax roundings, a few 2^-24
times the score magnitude, which is O(1) here: the q and k projections are
drawn with small block scales so the softmax mixes many positions); the O
projection adds 1e-5 * sum|w a|.  All of it stays inside the FFN's 1e-4
relative budget that the chain's tolerance carries through both branches:
    |h'_gpu - h'_ref| <= 1e-4 * (|h| + |a| + |b|) + 1e-4 * (rms(a) + rms(b)).
The caches: every position but pos is untouched (bit for bit), and position
pos holds the step's v (within the matvec tolerance of the oracle's).
One launch over L layers equals L single-layer launches bit for bit.  Shapes
that fit the decode chain run on it: with head_dim 256 and at most 2 query
heads per kv head, or head_dim 128 and 1, 2 or 4, the attention runs inside
the chain kernel (every layer in one launch); other head shapes take one
chain launch per layer between the standalone attention launches.  Layers
with mixed down-projection formats take the launch sequence of standalone
kernels.  Each path is tested here.
"""
import numpy as np
import pytest
import torch

import oracle
from quantized_weight_streaming_q4k_gb300 import build, ops, synth

pytestmark = pytest.mark.gpu

SMALL = dict(hidden=512, inter=1024, n_q_heads=4, n_kv_heads=2, head_dim=64, eps=1e-6,
             post_norms=1)
# (n_q_heads, n_kv_heads, head_dim): standalone attention launches between
# chain launches, then the three shapes of the in-kernel attention
HEADS = [(4, 2, 64), (4, 2, 128), (4, 1, 128), (2, 2, 256)]


def _layer(l, dims, workload, fmt_down=synth.Q6_K):
    L = synth.chain_layer(l, dims, fmt_down=fmt_down, workload=workload)
    g = synth.rng(workload, 77, l)
    small = dict(d_range=(2e-5, 4e-5), dmin_range=(2e-5, 4e-5))
    L["Wq"] = synth.q4_k_matrix(g, dims["n_q_heads"] * dims["head_dim"], dims["hidden"], **small)
    L["Wk"] = synth.q4_k_matrix(g, dims["n_kv_heads"] * dims["head_dim"], dims["hidden"], **small)
    return L


def _caches(dims, max_seq, pos, seed):
    g = synth.rng(950, seed)
    shape = (dims["n_kv_heads"], max_seq, dims["head_dim"])
    kc = (0.5 * g.standard_normal(shape)).astype(np.float32)
    vc = g.standard_normal(shape).astype(np.float32)
    kc[:, pos:] = 0.0
    vc[:, pos:] = 0.0
    return kc, vc


def _dev(L):
    return {k: (torch.from_numpy(np.ascontiguousarray(v)).cuda() if isinstance(v, np.ndarray)
                else v) for k, v in L.items()}


def _tol(h_in, tr, ref):
    hb = np.asarray(h_in, np.float64)
    a = tr["h1"] - hb
    b = ref - tr["h1"]
    return 1e-4 * (np.abs(hb) + np.abs(a) + np.abs(b)) + 1e-4 * (
        np.sqrt(np.mean(a * a)) + np.sqrt(np.mean(b * b)))


def _run_layers(dims, layers, n_layers, max_seq, pos, h0, workload, rot_dim=None, softcap=0.0):
    build.build()
    torch.cuda.set_device(0)
    hd = dims["head_dim"]
    rot = hd if rot_dim is None else rot_dim
    scale = 1.0 / np.sqrt(hd)
    ldev = [_dev(L) for L in layers]
    caches = [_caches(dims, max_seq, pos, workload * 10 + l) for l in range(n_layers)]
    h_in = h0.copy()
    worst = 0.0
    for l in range(n_layers):
        kc, vc = caches[l]
        kd, vd = torch.from_numpy(kc.copy()).cuda(), torch.from_numpy(vc.copy()).cuda()
        h = torch.from_numpy(h_in.copy()).cuda()
        ops.decode_kv([ldev[l]], h, dims, [kd], [vd], max_seq, pos, rot, 10000.0, scale, softcap)
        torch.cuda.synchronize()
        hg = h.cpu().numpy()
        kv = dict(k_cache=kc.astype(np.float64), v_cache=vc.astype(np.float64), max_seq=max_seq,
                  pos=pos, rot_dim=rot, rope_base=10000.0, scale=scale, softcap=softcap)
        ref, tr = oracle.layer_forward_kv(layers[l], dims, kv, h_in, trace=True)
        tol = _tol(h_in, tr, ref)
        err = np.abs(hg.astype(np.float64) - ref)
        assert np.all(err <= tol), f"layer {l}: max err/tol {np.max(err / tol):.3g}"
        worst = max(worst, float(np.max(err / tol)))
        # caches: only position pos changed; v at pos is the step's v
        kg, vg = kd.cpu().numpy(), vd.cpu().numpy()
        keep = np.ones(max_seq, bool)
        keep[pos] = False
        assert np.array_equal(kg[:, keep], kc[:, keep]) and np.array_equal(vg[:, keep], vc[:, keep])
        v_ref = tr["v"].reshape(dims["n_kv_heads"], hd)
        k_ref = tr["k"].reshape(dims["n_kv_heads"], hd)
        vmag = np.max(np.abs(v_ref)) + 1e-30
        kmag = np.max(np.abs(k_ref)) + 1e-30
        assert np.max(np.abs(vg[:, pos] - v_ref)) <= 1e-4 * vmag
        assert np.max(np.abs(kg[:, pos] - k_ref)) <= 1e-4 * kmag
        h_in = hg
    assert ops.device_error() == 0
    return h_in, caches, worst


@pytest.mark.parametrize("heads", HEADS)
@pytest.mark.parametrize("post_norms,pos,rot_dim,softcap",
                         [(1, 37, None, 0.0), (0, 5, 32, 0.0), (1, 0, None, 0.0),
                          (1, 63, None, 30.0)])
def test_decode_kv_small(post_norms, pos, rot_dim, softcap, heads):
    nq, nkv, hd = heads
    dims = dict(SMALL, post_norms=post_norms, n_q_heads=nq, n_kv_heads=nkv, head_dim=hd)
    layers = [_layer(l, dims, 960 + post_norms) for l in range(2)]
    h0 = synth.normal_vector(synth.rng(961, pos), dims["hidden"])
    _run_layers(dims, layers, 2, 64, pos, h0, 960, rot_dim, softcap)


@pytest.mark.parametrize("shape,pos,max_seq", [
    # 4001 cached positions over 2 kv heads: 76 chunks of 53 positions, so
    # every warp of the in-kernel attention takes three rounds of rows
    (dict(n_q_heads=4, n_kv_heads=2, head_dim=128), 4000, 4096),
    (dict(n_q_heads=2, n_kv_heads=2, head_dim=256), 4000, 4096),
    # 3 kv heads: 51 chunks each, 153 items on 152 CTAs (one CTA takes two)
    (dict(n_q_heads=6, n_kv_heads=3, head_dim=128), 2000, 2048),
    # 64 query heads of 128: 8192 outputs, 54 per CTA, merged in two rounds;
    # 32 kv heads x 5 chunks = 160 items
    (dict(hidden=2048, inter=2048, n_q_heads=64, n_kv_heads=32, head_dim=128), 200, 256),
])
def test_decode_kv_long_cache(shape, pos, max_seq):
    dims = dict(SMALL, **shape)
    layers = [_layer(l, dims, 972) for l in range(2)]
    h0 = synth.normal_vector(synth.rng(973), dims["hidden"])
    _run_layers(dims, layers, 2, max_seq, pos, h0, 972)


def test_decode_kv_launch_sequence_path():
    """Layers whose down projections differ in format take the launch
    sequence (the chain kernel takes one down format): same parity bar."""
    dims = SMALL
    layers = [_layer(0, dims, 966, synth.Q6_K), _layer(1, dims, 966, synth.Q4_K)]
    h0 = synth.normal_vector(synth.rng(967), dims["hidden"])
    _run_layers(dims, layers, 2, 48, 21, h0, 966)


@pytest.mark.parametrize("heads", [HEADS[0], HEADS[1]])
def test_decode_kv_multi_layer_launch_equals_single_layer_launches(heads):
    build.build()
    torch.cuda.set_device(0)
    nq, nkv, hd = heads
    dims = dict(SMALL, n_q_heads=nq, n_kv_heads=nkv, head_dim=hd)
    max_seq, pos = 32, 9
    layers = [_layer(l, dims, 962) for l in range(3)]
    ldev = [_dev(L) for L in layers]
    h0 = synth.normal_vector(synth.rng(963), dims["hidden"])
    base = [_caches(dims, max_seq, pos, 970 + l) for l in range(3)]
    scale = 1.0 / np.sqrt(dims["head_dim"])

    def fresh():
        return ([torch.from_numpy(k.copy()).cuda() for k, _ in base],
                [torch.from_numpy(v.copy()).cuda() for _, v in base])

    ks, vs = fresh()
    h = torch.from_numpy(h0.copy()).cuda()
    ops.decode_kv(ldev, h, dims, ks, vs, max_seq, pos, 64, 10000.0, scale)
    ks1, vs1 = fresh()
    h1 = torch.from_numpy(h0.copy()).cuda()
    for l in range(3):
        ops.decode_kv([ldev[l]], h1, dims, [ks1[l]], [vs1[l]], max_seq, pos, 64, 10000.0, scale)
    torch.cuda.synchronize()
    assert torch.equal(h, h1)
    for l in range(3):
        assert torch.equal(ks[l], ks1[l]) and torch.equal(vs[l], vs1[l])
    assert ops.device_error() == 0


@pytest.mark.parametrize("heads", [HEADS[0], HEADS[1]])
def test_decode_kv_more_layers_than_one_chain_launch_holds(heads):
    """70 layers run as a group of 64 and a group of 6 (chain launches per
    group); the result equals 70 one-layer calls bit for bit (h and every
    cache)."""
    build.build()
    torch.cuda.set_device(0)
    nq, nkv, hd = heads
    dims = dict(SMALL, hidden=256, inter=512, n_q_heads=nq, n_kv_heads=nkv, head_dim=hd)
    n, max_seq, pos = 70, 16, 3
    layers = [_dev(_layer(l, dims, 968)) for l in range(n)]
    h0 = synth.normal_vector(synth.rng(969), dims["hidden"])
    base = [_caches(dims, max_seq, pos, 980 + l) for l in range(n)]
    scale = 1.0 / np.sqrt(dims["head_dim"])

    def fresh():
        return ([torch.from_numpy(k.copy()).cuda() for k, _ in base],
                [torch.from_numpy(v.copy()).cuda() for _, v in base])

    ks, vs = fresh()
    h = torch.from_numpy(h0.copy()).cuda()
    ops.decode_kv(layers, h, dims, ks, vs, max_seq, pos, 64, 10000.0, scale)
    ks1, vs1 = fresh()
    h1 = torch.from_numpy(h0.copy()).cuda()
    for l in range(n):
        ops.decode_kv([layers[l]], h1, dims, [ks1[l]], [vs1[l]], max_seq, pos, 64, 10000.0,
                      scale)
    torch.cuda.synchronize()
    assert torch.isfinite(h).all()
    assert torch.equal(h, h1)
    for l in range(n):
        assert torch.equal(ks[l], ks1[l]) and torch.equal(vs[l], vs1[l])
    assert ops.device_error() == 0


def test_decode_kv_gemma3_4b_1024_cached_positions():
    dims = synth.GEMMA3_4B
    pos, max_seq = 1024, 1088
    layers = [_layer(0, dims, 964)]
    h0 = synth.normal_vector(synth.rng(965), dims["hidden"])
    _, _, worst = _run_layers(dims, layers, 1, max_seq, pos, h0, 964)
    print(f"decode_kv Gemma-3-4B, 1025 positions: max err/tol {worst:.3g}")
