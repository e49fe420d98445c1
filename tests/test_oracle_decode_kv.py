"""Pins of the oracle's decoder layer with a KV cache (qo_layer_forward_kv).

It is pinned against things other than itself:
  * at position 0 (empty cache) it equals the sequence-1 layer
    (qo_layer_forward) bit for bit: the rotation angle is 0 and the softmax
    runs over a single key;
  * at any position it equals the composition of the separately pinned steps
    (rms_norm, matvec, rope, kv_append, kv_attention, ffn), run here one by
    one through their own oracle entry points;
  * it writes the rotated k and the plain v at position pos of the caches and
    nothing else;
  * consecutive positions see every earlier key (position 1 attends over the
    key written at position 0).
"""
import numpy as np
import pytest

import oracle
from quantized_weight_streaming_q4k_gb300 import synth

DIMS = dict(hidden=512, inter=1024, n_q_heads=4, n_kv_heads=2, head_dim=64, eps=1e-6,
            post_norms=1)


def _layer(seed, dims=DIMS):
    return synth.chain_layer(seed, dims, workload=930)


def _kv(dims, max_seq, pos, seed, rot_dim=None, base=10000.0, softcap=0.0):
    g = synth.rng(931, seed)
    shape = (dims["n_kv_heads"], max_seq, dims["head_dim"])
    kc = g.standard_normal(shape)
    vc = g.standard_normal(shape)
    kc[:, pos:] = 0.0
    vc[:, pos:] = 0.0
    return dict(k_cache=kc, v_cache=vc, max_seq=max_seq, pos=pos,
                rot_dim=dims["head_dim"] if rot_dim is None else rot_dim, rope_base=base,
                scale=1.0 / np.sqrt(dims["head_dim"]), softcap=softcap)


@pytest.mark.parametrize("post_norms", [1, 0])
def test_position_zero_equals_sequence_one_layer(post_norms):
    dims = dict(DIMS, post_norms=post_norms)
    L = _layer(1)
    h = synth.normal_vector(synth.rng(932, post_norms), dims["hidden"]).astype(np.float64)
    kv = _kv(dims, 16, 0, 1)
    got = oracle.layer_forward_kv(L, dims, kv, h)
    ref = oracle.layer_forward(L, dims, h)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("pos,rot_dim,softcap", [(5, None, 0.0), (37, 32, 0.0), (20, None, 8.0)])
def test_equals_composition_of_pinned_steps(pos, rot_dim, softcap):
    dims = DIMS
    H, I = dims["hidden"], dims["inter"]
    nq, nkv, hd = dims["n_q_heads"], dims["n_kv_heads"], dims["head_dim"]
    L = _layer(2)
    h = synth.normal_vector(synth.rng(933, pos), H).astype(np.float64)
    kv = _kv(dims, 64, pos, 3, rot_dim=rot_dim, softcap=softcap)
    kc0, vc0 = kv["k_cache"].copy(), kv["v_cache"].copy()
    got, tr = oracle.layer_forward_kv(L, dims, kv, h, trace=True)

    eps = dims["eps"]
    n1 = oracle.rms_norm(h, L["w_in"], eps)
    q, _ = oracle.matvec(oracle.Q4_K, L["Wq"], nq * hd, H, n1)
    k, _ = oracle.matvec(oracle.Q4_K, L["Wk"], nkv * hd, H, n1)
    v, _ = oracle.matvec(oracle.Q4_K, L["Wv"], nkv * hd, H, n1)
    q = oracle.rope(q, nq, hd, kv["rot_dim"], pos, kv["rope_base"])
    k = oracle.rope(k, nkv, hd, kv["rot_dim"], pos, kv["rope_base"])
    kc, vc = oracle.kv_append(kc0, vc0, k, v, nkv, hd, 64, pos)
    a, _, _ = oracle.kv_attention(q, kc, vc, nq, nkv, hd, 64, pos + 1, kv["scale"], softcap)
    o, _ = oracle.matvec(oracle.Q4_K, L["Wo"], H, nq * hd, a.reshape(-1))
    h1 = h + oracle.rms_norm(o, L["w_post_attn"], eps)
    n2 = oracle.rms_norm(h1, L["w_pre_ffn"], eps)
    f = oracle.ffn(oracle.Q4_K, L["Wg"], L["Wu"], oracle.Q6_K, L["Wd"], H, I, n2)["y"]
    ref = h1 + oracle.rms_norm(f, L["w_post_ffn"], eps)

    np.testing.assert_allclose(tr["q"], q.reshape(-1), rtol=0, atol=0)
    np.testing.assert_allclose(tr["attn"], a.reshape(-1), rtol=1e-13, atol=1e-300)
    scale = np.abs(h1) + np.abs(ref - h1) + 1.0
    assert np.max(np.abs(got - ref) / scale) <= 1e-12
    # the caches: rotated k and plain v at pos, everything else untouched
    np.testing.assert_array_equal(kv["k_cache"], np.asarray(kc).reshape(kc0.shape))
    np.testing.assert_array_equal(kv["v_cache"], np.asarray(vc).reshape(vc0.shape))
    mask = np.ones(kc0.shape[1], bool)
    mask[pos] = False
    np.testing.assert_array_equal(kv["k_cache"][:, mask], kc0[:, mask])
    np.testing.assert_array_equal(kv["v_cache"][:, pos].reshape(-1), v.reshape(-1))


def test_consecutive_positions_see_earlier_keys():
    dims = DIMS
    L = _layer(4)
    # small q and k projections keep the scores moderate, so the softmax mixes
    # the two keys instead of picking one
    gq = synth.rng(935, 0)
    small = dict(d_range=(2e-5, 4e-5), dmin_range=(2e-5, 4e-5))
    L["Wq"] = synth.q4_k_matrix(gq, dims["n_q_heads"] * dims["head_dim"], dims["hidden"], **small)
    L["Wk"] = synth.q4_k_matrix(gq, dims["n_kv_heads"] * dims["head_dim"], dims["hidden"], **small)
    h0 = synth.normal_vector(synth.rng(934, 0), dims["hidden"]).astype(np.float64)
    kv = _kv(dims, 8, 0, 5)
    h1 = oracle.layer_forward_kv(L, dims, kv, h0)
    assert np.any(kv["k_cache"][:, 0] != 0.0)
    kv["pos"] = 1
    h2, tr = oracle.layer_forward_kv(L, dims, kv, h1, trace=True)
    # position 1 attends over two keys: the output is a convex mix of the two
    # value rows of each kv head, and differs from attending to the new key alone
    nq, nkv, hd = dims["n_q_heads"], dims["n_kv_heads"], dims["head_dim"]
    a = tr["attn"].reshape(nq, hd)
    group = nq // nkv
    for hq in range(nq):
        g = hq // group
        v0, v1 = kv["v_cache"][g, 0], kv["v_cache"][g, 1]
        lam = np.dot(a[hq] - v1, v0 - v1) / np.dot(v0 - v1, v0 - v1)
        assert 1e-3 < lam < 1 - 1e-3           # both keys carry weight
        np.testing.assert_allclose(a[hq], lam * v0 + (1 - lam) * v1, rtol=0,
                                   atol=1e-9 * np.max(np.abs(v0 - v1)))
