"""Pins for the oracle's KV-cache attention pieces (CPU only): RoPE at a
position, kv_append and one query token's attention over the cache
(infer-compute README §Shaders rows "Attention" and "RoPE"; infer-inference
README §BLAS-Fused Attention).

What pins each function:
* rope: position 0 is the identity; the defining property of a rotary
  embedding -- the dot product of a rotated query and a rotated key depends
  only on the difference of their positions; rotations compose additively in
  the position; norms are kept; unit vectors land on cos / sin of the
  textbook angles (cos 1, sin 1, cos 3, sin 3), which fixes the pairing of
  dimension i with i + r/2, the sign and the frequency base^(-2i/r); the
  dimensions past rot_dim are untouched.
* kv_append: the written slot reads back, every other slot is unchanged.
* kv_attention: one position gives that position's value; equal scores give
  the mean of the values; a common shift of every score changes nothing;
  scipy's softmax on small inputs (brute force); softcap -> infinity is no
  softcap and softcap bounds every score; GQA grouping; the returned bound
  dominates |out|.
"""

import numpy as np
import pytest

import oracle

scipy_special = pytest.importorskip("scipy.special")


# ------------------------------------------------------------------ rope
def test_rope_position_zero_is_identity():
    x = np.random.default_rng(1).standard_normal((3, 8))
    assert np.array_equal(oracle.rope(x, 3, 8, 8, 0, 10000.0), x)


def test_rope_unit_vectors_land_on_textbook_angles():
    # r = 4, base 10000: theta_0 = pos, theta_1 = pos / 100
    e0 = np.array([[1.0, 0.0, 0.0, 0.0]])
    got = oracle.rope(e0, 1, 4, 4, 3, 10000.0)
    assert np.allclose(got, [[-0.9899924966004454, 0.0, 0.1411200080598672, 0.0]], atol=1e-15)
    e1 = np.array([[0.0, 1.0, 0.0, 0.0]])
    got = oracle.rope(e1, 1, 4, 4, 100, 10000.0)
    assert np.allclose(got, [[0.0, 0.5403023058681398, 0.0, 0.8414709848078965]], atol=1e-13)
    # the partner dimension rotates the other way: e2 -> (-sin, cos) on (0, 2)
    e2 = np.array([[0.0, 0.0, 1.0, 0.0]])
    got = oracle.rope(e2, 1, 4, 4, 3, 10000.0)
    assert np.allclose(got, [[-0.1411200080598672, 0.0, -0.9899924966004454, 0.0]], atol=1e-15)


@pytest.mark.parametrize("rot", [8, 4, 2])
def test_rope_dot_depends_only_on_position_difference(rot):
    g = np.random.default_rng(2)
    q, k = g.standard_normal((1, 8)), g.standard_normal((1, 8))
    for m, n, d in ((5, 2, 7), (100, 40, 1000), (3, 9, 12)):
        a = np.dot(oracle.rope(q, 1, 8, rot, m, 500.0)[0], oracle.rope(k, 1, 8, rot, n, 500.0)[0])
        b = np.dot(oracle.rope(q, 1, 8, rot, m + d, 500.0)[0],
                   oracle.rope(k, 1, 8, rot, n + d, 500.0)[0])
        assert a == pytest.approx(b, rel=1e-9, abs=1e-9)


def test_rope_composes_additively_and_keeps_norms():
    g = np.random.default_rng(3)
    x = g.standard_normal((4, 16))
    a = oracle.rope(oracle.rope(x, 4, 16, 16, 37, 1e6), 4, 16, 16, 1000, 1e6)
    b = oracle.rope(x, 4, 16, 16, 1037, 1e6)
    assert np.allclose(a, b, atol=1e-9)
    assert np.allclose(np.linalg.norm(b, axis=1), np.linalg.norm(x, axis=1), rtol=1e-13)


def test_rope_partial_leaves_the_tail_alone():
    g = np.random.default_rng(4)
    x = g.standard_normal((2, 16))
    y = oracle.rope(x, 2, 16, 4, 77, 10000.0)
    assert np.array_equal(y[:, 4:], x[:, 4:])
    assert not np.allclose(y[:, :4], x[:, :4])
    with pytest.raises(ValueError):
        oracle.rope(x, 2, 16, 5, 1, 10000.0)
    with pytest.raises(ValueError):
        oracle.rope(x, 2, 16, 18, 1, 10000.0)


# ------------------------------------------------------------------ kv_append
def test_kv_append_writes_one_slot():
    g = np.random.default_rng(5)
    kc, vc = g.standard_normal((2, 6, 4)), g.standard_normal((2, 6, 4))
    k, v = g.standard_normal((2, 4)), g.standard_normal((2, 4))
    kc2, vc2 = oracle.kv_append(kc, vc, k, v, 2, 4, 6, 3)
    assert np.array_equal(kc2[:, 3], k) and np.array_equal(vc2[:, 3], v)
    mask = np.ones(6, bool)
    mask[3] = False
    assert np.array_equal(kc2[:, mask], kc[:, mask]) and np.array_equal(vc2[:, mask], vc[:, mask])
    with pytest.raises(ValueError):
        oracle.kv_append(kc, vc, k, v, 2, 4, 6, 6)


# ------------------------------------------------------------------ attention
def _cache(g, nkv, L, hd):
    return g.standard_normal((nkv, L, hd)), g.standard_normal((nkv, L, hd))


def test_attention_one_position_returns_its_value():
    g = np.random.default_rng(6)
    kc, vc = _cache(g, 2, 5, 8)
    q = g.standard_normal((4, 8))
    out, _, _ = oracle.kv_attention(q, kc, vc, 4, 2, 8, 5, 1, 0.3)
    assert np.array_equal(out, vc[[0, 0, 1, 1], 0])


def test_attention_equal_scores_average_the_values():
    g = np.random.default_rng(7)
    kc, vc = _cache(g, 1, 9, 8)
    kc[:] = kc[:, :1]                      # every key the same
    q = g.standard_normal((2, 8))
    out, _, _ = oracle.kv_attention(q, kc, vc, 2, 1, 8, 9, 7, 0.5)
    assert np.allclose(out, np.broadcast_to(vc[0, :7].mean(axis=0), (2, 8)), atol=1e-14)
    out0, _, _ = oracle.kv_attention(np.zeros((2, 8)), g.standard_normal((1, 9, 8)), vc, 2, 1, 8,
                                     9, 9, 0.5)
    assert np.allclose(out0, np.broadcast_to(vc[0].mean(axis=0), (2, 8)), atol=1e-14)


def test_attention_common_score_shift_changes_nothing():
    g = np.random.default_rng(8)
    kc, vc = _cache(g, 1, 12, 8)
    q = g.standard_normal((1, 8))
    base, _, _ = oracle.kv_attention(q, kc, vc, 1, 1, 8, 12, 12, 0.25)
    shifted = kc + 3.0 * q[0] / np.dot(q[0], q[0])     # q . k_t grows by 3 for every t
    out, _, _ = oracle.kv_attention(q, shifted, vc, 1, 1, 8, 12, 12, 0.25)
    assert np.allclose(out, base, atol=1e-13)


@pytest.mark.parametrize("softcap", [0.0, 2.5])
def test_attention_brute_force_small(softcap):
    g = np.random.default_rng(9)
    nq, nkv, hd, L, n = 6, 2, 8, 10, 7
    kc, vc = _cache(g, nkv, L, hd)
    q = g.standard_normal((nq, hd)) * 2.0
    out, bound, _ = oracle.kv_attention(q, kc, vc, nq, nkv, hd, L, n, 0.7, softcap)
    for h in range(nq):
        grp = h // (nq // nkv)
        s = 0.7 * kc[grp, :n] @ q[h]
        if softcap:
            s = softcap * np.tanh(s / softcap)
            assert np.all(np.abs(s) <= softcap)
        p = scipy_special.softmax(s)
        assert np.allclose(out[h], p @ vc[grp, :n], atol=1e-13)
        assert np.all(bound[h] >= np.abs(out[h]) - 1e-15)


def test_attention_large_softcap_is_no_softcap():
    g = np.random.default_rng(10)
    kc, vc = _cache(g, 1, 6, 4)
    q = g.standard_normal((1, 4))
    a, _, _ = oracle.kv_attention(q, kc, vc, 1, 1, 4, 6, 6, 0.5, 0.0)
    b, _, _ = oracle.kv_attention(q, kc, vc, 1, 1, 4, 6, 6, 0.5, 1e9)
    assert np.allclose(a, b, atol=1e-12)


def test_attention_gqa_grouping():
    g = np.random.default_rng(11)
    kc, vc = _cache(g, 2, 8, 4)
    q = g.standard_normal((4, 4))
    q[1] = q[0]
    out, _, _ = oracle.kv_attention(q, kc, vc, 4, 2, 4, 8, 8, 1.0)
    assert np.array_equal(out[0], out[1])
    kc2 = kc.copy()
    kc2[0] = g.standard_normal((8, 4))     # kv head 0 only feeds query heads 0 and 1
    out2, _, _ = oracle.kv_attention(q, kc2, vc, 4, 2, 4, 8, 8, 1.0)
    assert np.array_equal(out2[2:], out[2:]) and not np.allclose(out2[:2], out[:2])


def test_attention_dominant_key():
    g = np.random.default_rng(12)
    kc, vc = _cache(g, 1, 5, 8)
    u = kc[0, 2] / np.linalg.norm(kc[0, 2])
    kc[0, 2] = 20.0 * u                    # score 100 against at most ~5 |k_t| for the rest
    out, _, _ = oracle.kv_attention(5.0 * u[None, :], kc, vc, 1, 1, 8, 5, 5, 1.0)
    assert np.allclose(out[0], vc[0, 2], atol=1e-12)


def test_attention_rejects_bad_arguments():
    kc = np.zeros((1, 4, 2))
    with pytest.raises(ValueError):
        oracle.kv_attention(np.zeros((3, 2)), np.zeros((2, 4, 2)), np.zeros((2, 4, 2)), 3, 2, 2,
                            4, 2, 1.0)
    with pytest.raises(ValueError):
        oracle.kv_attention(np.zeros((1, 2)), kc, kc, 1, 1, 2, 4, 5, 1.0)
