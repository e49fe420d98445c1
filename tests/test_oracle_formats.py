"""Pins for the oracle's block decoders (CPU only).

Each decoder is checked against hand-packed byte fixtures in tests/golden/
whose expected weights were derived by hand from the literal field values, and
the binary16 decoder against numpy's float16 for every bit pattern.
"""
import json
import os

import numpy as np
import pytest

import oracle


def _load(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


def test_half_all_patterns_match_numpy_float16():
    # numpy's float16 -> float64 conversion is exact, so it pins every pattern
    # (normals, subnormals, signed zeros, infinities, NaNs).
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.half(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # sign of zero
    assert np.signbit(oracle.half(0x8000)) and not np.signbit(oracle.half(0x0000))


@pytest.mark.parametrize("bits,value", [
    (0x3C00, 1.0), (0x3800, 0.5), (0xC000, -2.0), (0x0001, 2.0 ** -24),
    (0x03FF, 1023 * 2.0 ** -24), (0x0400, 2.0 ** -14), (0x7BFF, 65504.0),
    (0x0200, 2.0 ** -15), (0xB400, -0.25),
])
def test_half_textbook_values(bits, value):
    assert oracle.half(bits) == value


def _q4k_block(entry):
    b = np.zeros(144, dtype=np.uint8)
    b[0:2] = np.frombuffer(bytes.fromhex(entry["d_bits"]), dtype=np.uint8)[::-1]
    b[2:4] = np.frombuffer(bytes.fromhex(entry["dmin_bits"]), dtype=np.uint8)[::-1]
    b[4:16] = np.frombuffer(bytes.fromhex(entry["sc12_hex"].replace(" ", "")), dtype=np.uint8)
    for c in range(4):
        for l in range(32):
            if entry["name"] == "small_fields":
                lo, hi = l & 15, 15 - (l & 15)
            else:
                lo, hi = (3 * l + c) & 15, (7 * l + 5 * c) & 15
            b[16 + 32 * c + l] = lo | (hi << 4)
    return b


def _q4k_expected(entry):
    d, dmin = entry["d"], entry["dmin"]
    sc, mn = entry["scales"], entry["mins"]
    w = np.empty(256)
    for c in range(4):
        for l in range(32):
            if entry["name"] == "small_fields":
                lo, hi = l & 15, 15 - (l & 15)
            else:
                lo, hi = (3 * l + c) & 15, (7 * l + 5 * c) & 15
            w[64 * c + l] = d * sc[2 * c] * lo - dmin * mn[2 * c]
            w[64 * c + 32 + l] = d * sc[2 * c + 1] * hi - dmin * mn[2 * c + 1]
    return w


def test_q4_k_scale_min_unpacking(golden_dir):
    for entry in _load(golden_dir, "q4_k_blocks.json")["blocks"]:
        sc12 = np.frombuffer(bytes.fromhex(entry["sc12_hex"].replace(" ", "")), dtype=np.uint8)
        got = [oracle.q4_k_scale_min(sc12, s) for s in range(8)]
        assert [g[0] for g in got] == entry["scales"], entry["name"]
        assert [g[1] for g in got] == entry["mins"], entry["name"]


def test_q4_k_hand_decoded_blocks(golden_dir):
    for entry in _load(golden_dir, "q4_k_blocks.json")["blocks"]:
        got = oracle.dequant_block(oracle.Q4_K, _q4k_block(entry))
        # every expected value is exact in f64 (11-bit d x 6-bit scale x 4-bit q)
        assert np.array_equal(got, _q4k_expected(entry)), entry["name"]


def test_q4_k_d_and_dmin_positions():
    # d only: scales 1, mins 0 -> w = d*q ; dmin only: q = 0 -> w = -dmin*min
    b = np.zeros(144, dtype=np.uint8)
    b[0:2] = [0x00, 0x40]          # d = 2.0
    b[2:4] = [0x00, 0x3C]          # dmin = 1.0
    b[4:8] = 1                     # scale[0..3] = 1, mins[0..3] = 0
    b[12:16] = 0x01                # scale[4..7] = 1, mins[4..7] = 0
    b[16:] = 0x21                  # lo nibble 1, hi nibble 2
    w = oracle.dequant_block(oracle.Q4_K, b)
    assert np.array_equal(w, np.tile(np.r_[np.full(32, 2.0), np.full(32, 4.0)], 4))
    b[4:16] = 0
    b[8:12] = 9                    # min[0..3] = 9, scales 0
    b[16:] = 0
    w = oracle.dequant_block(oracle.Q4_K, b)
    assert np.array_equal(w[:128], np.full(128, -9.0)) and np.array_equal(w[128:], np.zeros(128))


def _q6k_block(entry):
    b = np.zeros(210, dtype=np.uint8)
    if entry["ql"] == "ramp":
        b[0:128] = np.arange(128, dtype=np.uint8)
    if "qh_byte" in entry:
        b[128:192] = entry["qh_byte"]
    elif entry.get("qh") == "ramp":
        b[128:192] = np.arange(64, dtype=np.uint8)
    b[192:208] = np.array(entry["sc"], dtype=np.int8).view(np.uint8)
    b[208:210] = np.frombuffer(bytes.fromhex(entry["d_bits"]), dtype=np.uint8)[::-1]
    return b


def _q6k_expected(entry):
    w = np.empty(256)
    for h in range(2):
        for k in range(4):
            for l in range(32):
                i = 128 * h + 32 * k + l
                if entry["name"] == "ql_ramp_qh_const":
                    q = [(l & 15) - 32, (l & 15) - 16, 4 * h + (l >> 4), 4 * h + 18 + (l >> 4)][k]
                elif entry["name"] == "qh_ramp":
                    q = 16 * (((32 * h + l) >> (2 * k)) & 3) - 32
                else:
                    q = 0
                w[i] = entry["d"] * entry["sc"][i // 16] * q
    return w


def test_q6_k_hand_decoded_blocks(golden_dir):
    for entry in _load(golden_dir, "q6_k_blocks.json")["blocks"]:
        got = oracle.dequant_block(oracle.Q6_K, _q6k_block(entry))
        assert np.array_equal(got, _q6k_expected(entry)), entry["name"]


def test_q6_k_signed_scale_cases():
    # one scale byte at a time: -128, -1, 127 with q = 31 (max) in its 16 weights
    for val in (-128, -1, 127):
        for slot in (0, 7, 15):
            b = np.zeros(210, dtype=np.uint8)
            b[0:128] = 0xFF                 # nibbles 15
            b[128:192] = 0x55               # high bits 1 everywhere -> q6 = 31 -> q = -1
            b[192 + slot] = np.int8(val).view(np.uint8)
            b[208:210] = [0x00, 0x3C]       # d = 1
            w = oracle.dequant_block(oracle.Q6_K, b)
            expect = np.zeros(256)
            expect[16 * slot:16 * slot + 16] = -1.0 * val
            assert np.array_equal(w, expect), (val, slot)


def test_q4_0_hand_decoded_blocks(golden_dir):
    for entry in _load(golden_dir, "q4_0_blocks.json")["blocks"]:
        b = np.zeros(18, dtype=np.uint8)
        b[0:2] = np.frombuffer(bytes.fromhex(entry["d_bits"]), dtype=np.uint8)[::-1]
        b[2:18] = np.frombuffer(bytes.fromhex(entry["qs_hex"]), dtype=np.uint8)
        got = oracle.dequant_block(oracle.Q4_0, b)
        assert np.array_equal(got[:16], np.array(entry["expected_lo"], dtype=float))
        assert np.array_equal(got[16:], np.array(entry["expected_hi"], dtype=float))


def test_dequant_rows_concatenates_blocks_row_major():
    from quantized_weight_streaming_q4k_gb300 import synth
    for fmt in (oracle.Q4_0, oracle.Q4_K, oracle.Q6_K):
        qk, bb = oracle.BLOCK_WEIGHTS[fmt], oracle.BLOCK_BYTES[fmt]
        rows, hidden = 3, 2 * qk
        W = synth.matrix(fmt, synth.rng(99, fmt), rows, hidden)
        dense = oracle.dequant(fmt, W, rows, hidden)
        for r in range(rows):
            for b in range(2):
                blk = W[(r * 2 + b) * bb:(r * 2 + b + 1) * bb]
                assert np.array_equal(dense[r, b * qk:(b + 1) * qk], oracle.dequant_block(fmt, blk))
