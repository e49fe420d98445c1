"""Pins for the oracle's 8-bit path (CPU only): the binary16 encoder, the Q8_0
decoder, activation quantization (quantize_q8) and the matvec over Q8_0
activations (infer-compute README §Shaders rows "Q8" and "Element-wise";
§Architecture "Q4_0 through legacy Q8 path").

What pins each function:
* binary16 encoder: numpy's float16 conversion (an independent library
  routine, round to nearest even) on random, subnormal, overflow and tie
  values, and the round trip of every finite binary16 pattern.
* Q8_0 decoder: hand-decoded byte fixtures in tests/golden/q8_0_blocks.json.
* quantize_q8: hand-derived blocks (exact unit scale with ties, a zero block,
  a negative maximum) and invariants on random data: the largest magnitude
  maps to +-127, codes keep the sign, the reconstruction error is at most half
  a step, and a power-of-two scaling of x leaves the codes unchanged.
* matvec over Q8_0 activations: the dense f64 product of the separately
  dequantized weights and activations (decoders pinned above and in
  test_oracle_formats.py), and a brute-force integer loop on tiny inputs.
"""
import json
import os

import numpy as np
import pytest

import oracle
from quantized_weight_streaming_q4k_gb300 import synth


def _load(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


def _s8(b):
    return np.asarray(b, dtype=np.uint8).view(np.int8).astype(np.int64)


def _d_bits(blk):
    return int(blk[0]) | (int(blk[1]) << 8)


# ---------------------------------------------------------------- binary16
def test_half_bits_matches_numpy_float16_on_random_f32():
    g = np.random.default_rng(11)
    vals = np.concatenate([
        g.standard_normal(20000).astype(np.float32),
        (g.standard_normal(5000) * 1e-6).astype(np.float32),      # subnormal range
        (g.standard_normal(5000) * 1e-8).astype(np.float32),      # underflow to 0
        (g.standard_normal(5000) * 3e4).astype(np.float32),       # near overflow
        g.uniform(65000, 70000, 1000).astype(np.float32),
    ])
    for v in vals:
        with np.errstate(over="ignore"):
            want = int(np.float32(v).astype(np.float16).view(np.uint16))
        assert oracle.half_bits(v) == want, (v, hex(want))


def test_half_bits_ties_go_to_even():
    # 1 + 2^-11 is halfway between 1 and 1 + 2^-10: even significand is 1.0
    assert oracle.half_bits(1.0 + 2.0 ** -11) == 0x3C00
    # 1 + 3 * 2^-11 is halfway between 1 + 2^-10 (odd) and 1 + 2^-9 (even)
    assert oracle.half_bits(1.0 + 3 * 2.0 ** -11) == 0x3C02
    # 2^-25 is halfway between 0 and the smallest subnormal 2^-24: rounds to 0
    assert oracle.half_bits(2.0 ** -25) == 0x0000
    assert oracle.half_bits(3 * 2.0 ** -25) == 0x0002
    # 65520 is halfway between 65504 and 2^16 (out of range): infinity
    assert oracle.half_bits(65519.0) == 0x7BFF
    assert oracle.half_bits(65520.0) == 0x7C00
    assert oracle.half_bits(-0.0) == 0x8000


def test_half_bits_round_trips_every_finite_half():
    for h in range(1 << 16):
        if (h & 0x7C00) == 0x7C00:
            continue
        assert oracle.half_bits(np.float32(oracle.half(h))) == h, hex(h)


# ---------------------------------------------------------------- Q8_0 decode
def test_q8_0_hand_decoded_blocks(golden_dir):
    for entry in _load(golden_dir, "q8_0_blocks.json")["blocks"]:
        b = np.zeros(34, dtype=np.uint8)
        b[0:2] = np.frombuffer(bytes.fromhex(entry["d_bits"]), dtype=np.uint8)[::-1]
        b[2:34] = np.frombuffer(bytes.fromhex(entry["qs_hex"]), dtype=np.uint8)
        got = oracle.dequant_block(oracle.Q8_0, b)
        assert np.array_equal(got, np.array(entry["expected"], dtype=float)), entry["name"]


# ---------------------------------------------------------------- quantize_q8
def test_quantize_hand_derived_blocks(golden_dir):
    for entry in _load(golden_dir, "q8_0_blocks.json")["quantize"]:
        out = oracle.quantize_q8_0(np.array(entry["x"], dtype=np.float32))
        assert out.shape == (34,)
        assert _d_bits(out) == int(entry["d_bits"], 16), entry["name"]
        assert np.array_equal(_s8(out[2:]), np.array(entry["q"])), entry["name"]


def _quantize_checks(x):
    x = np.asarray(x, dtype=np.float32).reshape(-1, 32)
    out = oracle.quantize_q8_0(x.reshape(-1)).reshape(-1, 34)
    for blk, xb in zip(out, x):
        q = _s8(blk[2:])
        amax = np.float32(np.max(np.abs(xb)))
        d32 = np.float32(amax / np.float32(127))
        # stored scale: d rounded to binary16 (numpy's conversion)
        assert _d_bits(blk) == int(d32.astype(np.float16).view(np.uint16))
        assert np.all(np.abs(q) <= 127)
        if amax == 0:
            assert np.all(q == 0)
            continue
        j = int(np.argmax(np.abs(xb)))
        assert abs(q[j]) == 127 and np.sign(q[j]) == np.sign(xb[j])
        assert np.all((q == 0) | (np.sign(q) == np.sign(xb)))
        # reconstruction with the f32 step: at most half a step (+ f32 slack)
        err = np.abs(xb.astype(np.float64) - float(d32) * q)
        assert np.all(err <= float(d32) * (0.5 + 1e-5)), err.max() / float(d32)
    return out


def test_quantize_invariants_on_random_blocks():
    g = np.random.default_rng(5)
    x = np.concatenate([
        g.standard_normal(32 * 200),
        g.standard_normal(32 * 50) * 1e-3,
        g.uniform(-1, 1, 32 * 50) * 200.0,
    ]).astype(np.float32)
    _quantize_checks(x)


def test_quantize_is_invariant_under_power_of_two_scaling():
    g = np.random.default_rng(6)
    x = g.standard_normal(32 * 64).astype(np.float32)
    base = oracle.quantize_q8_0(x).reshape(-1, 34)
    for k in (-6, -1, 1, 5):
        out = oracle.quantize_q8_0(x * np.float32(2.0 ** k)).reshape(-1, 34)
        assert np.array_equal(out[:, 2:], base[:, 2:]), k
        d0 = np.array([oracle.half(_d_bits(b)) for b in base])
        dk = np.array([oracle.half(_d_bits(b)) for b in out])
        assert np.array_equal(dk, d0 * 2.0 ** k), k


def test_quantize_rejects_ragged_length():
    with pytest.raises(ValueError):
        oracle.quantize_q8_0(np.zeros(48, dtype=np.float32))


def test_quantize_batch_rows_are_independent():
    g = np.random.default_rng(7)
    x = g.standard_normal((3, 128)).astype(np.float32)
    out = oracle.quantize_q8_0(x)
    assert out.shape == (3, 4 * 34)
    for b in range(3):
        assert np.array_equal(out[b], oracle.quantize_q8_0(x[b]))


# ---------------------------------------------------------------- matvec
def _dequant_q8_vector(xq, hidden):
    return oracle.dequant(oracle.Q8_0, xq, 1, hidden)[0]


@pytest.mark.parametrize("wfmt", [oracle.Q4_0, oracle.Q8_0])
@pytest.mark.parametrize("batch", [1, 3])
def test_matvec_q8_equals_dense_product_of_dequantized_operands(wfmt, batch):
    rows, hidden = 37, 192
    W = synth.matrix(wfmt, synth.rng(70, wfmt), rows, hidden)
    x = synth.normal_vector(synth.rng(71), hidden, batch)
    xq = oracle.quantize_q8_0(x)
    y, bound = oracle.matvec_q8(wfmt, W, rows, hidden, xq)
    Wd = oracle.dequant(wfmt, W, rows, hidden)
    for b in range(batch):
        xd = _dequant_q8_vector(xq[b], hidden)
        ref = Wd @ xd
        mag = np.abs(Wd) @ np.abs(xd)
        assert np.allclose(y[b], ref, rtol=0, atol=1e-12 * mag.max())
        assert np.allclose(bound[b], mag, rtol=1e-12, atol=0)


@pytest.mark.parametrize("wfmt", [oracle.Q4_0, oracle.Q8_0])
def test_matvec_q8_brute_force_integer_sums(wfmt):
    rows, hidden = 2, 64
    W = synth.matrix(wfmt, synth.rng(72, wfmt), rows, hidden)
    xq = oracle.quantize_q8_0(synth.normal_vector(synth.rng(73), hidden))
    y, _ = oracle.matvec_q8(wfmt, W, rows, hidden, xq)
    bb = oracle.BLOCK_BYTES[wfmt]
    for r in range(rows):
        total = 0.0
        for k in range(hidden // 32):
            wb = W[(r * 2 + k) * bb:(r * 2 + k + 1) * bb]
            xb = xq[k * 34:(k + 1) * 34]
            if wfmt == oracle.Q4_0:
                codes = [int(wb[2 + j % 16] >> (4 * (j // 16)) & 15) - 8 for j in range(32)]
            else:
                codes = [int(v) for v in _s8(wb[2:])]
            isum = sum(c * int(a) for c, a in zip(codes, _s8(xb[2:])))
            total += oracle.half(_d_bits(wb)) * oracle.half(_d_bits(xb)) * isum
        assert y[r] == pytest.approx(total, rel=1e-14, abs=1e-14)


def test_matvec_q8_all_eight_q4_0_weights_give_zero():
    rows, hidden = 3, 64
    W = synth.q4_0_matrix(synth.rng(74), rows, hidden).reshape(-1, 18)
    W[:, 2:] = 0x88
    xq = oracle.quantize_q8_0(synth.normal_vector(synth.rng(75), hidden))
    y, bound = oracle.matvec_q8(oracle.Q4_0, W.reshape(-1), rows, hidden, xq)
    assert np.array_equal(y, np.zeros(rows)) and np.array_equal(bound, np.zeros(rows))


def test_matvec_q8_row_window_and_threads():
    rows, hidden = 50, 128
    W = synth.matrix(oracle.Q8_0, synth.rng(76), rows, hidden)
    xq = oracle.quantize_q8_0(synth.normal_vector(synth.rng(77), hidden))
    y, _ = oracle.matvec_q8(oracle.Q8_0, W, rows, hidden, xq)
    y2, _ = oracle.matvec_q8(oracle.Q8_0, W, rows, hidden, xq, threads=4)
    y3, _ = oracle.matvec_q8(oracle.Q8_0, W, rows, hidden, xq, row_begin=10, row_end=20)
    assert np.array_equal(y, y2)
    assert np.array_equal(y3[10:20], y[10:20]) and np.all(np.isnan(y3[:10]))


def test_matvec_f32_path_accepts_q8_0_weights():
    # the plain f64 matvec decodes Q8_0 weights like the other formats
    rows, hidden = 5, 64
    W = synth.matrix(oracle.Q8_0, synth.rng(78), rows, hidden)
    x = synth.normal_vector(synth.rng(79), hidden)
    y, _ = oracle.matvec(oracle.Q8_0, W, rows, hidden, x)
    ref = oracle.dequant(oracle.Q8_0, W, rows, hidden) @ x.astype(np.float64)
    assert np.allclose(y, ref, rtol=1e-13, atol=1e-13)


# ---------------------------------------------------------------- fused norm + quantize
def test_rms_norm_q8_constant_and_one_hot():
    # a constant vector normalises to +-1 (to within eps): every code is +-127
    x = np.full(64, -3.0, dtype=np.float32)
    out = oracle.rms_norm_q8(x, np.ones(64), 1e-6).reshape(-1, 34)
    assert np.all(_s8(out[:, 2:]) == -127)
    # a one-hot vector: sqrt(n) * w_0 at index 0, zeros elsewhere
    x = np.zeros(64, dtype=np.float32)
    x[0] = 5.0
    out = oracle.rms_norm_q8(x, np.ones(64), 0.0).reshape(-1, 34)
    q = _s8(out[0, 2:])
    assert q[0] == 127 and np.all(q[1:] == 0)
    assert np.all(out[1] == 0)                      # second block all zero: d = 0, codes 0
    assert oracle.half(_d_bits(out[0])) == pytest.approx(8.0 / 127, rel=2.0 ** -11)


def test_rms_norm_q8_reconstructs_the_norm():
    g = np.random.default_rng(21)
    x = g.standard_normal((2, 256)).astype(np.float32)
    w = g.normal(1.0, 0.1, 256)
    out = oracle.rms_norm_q8(x, w, 1e-6).reshape(2, -1, 34)
    for b in range(2):
        y = oracle.rms_norm(x[b], w, 1e-6)
        for k in range(8):
            d = oracle.half(_d_bits(out[b, k]))
            rec = d * _s8(out[b, k, 2:])
            assert np.all(np.abs(rec - y[32 * k:32 * k + 32]) <= d * 0.57)


def test_residual_rms_norm_q8_adds_then_normalises():
    g = np.random.default_rng(22)
    h = g.standard_normal(128).astype(np.float32)
    y = g.standard_normal(128).astype(np.float32)
    w = g.normal(1.0, 0.1, 128)
    hs, out = oracle.residual_rms_norm_q8(h, y, w, 1e-6)
    assert np.array_equal(hs, h.astype(np.float64) + y.astype(np.float64))
    assert np.array_equal(out, oracle.rms_norm_q8(hs, w, 1e-6))
