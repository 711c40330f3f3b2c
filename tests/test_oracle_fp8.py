"""The oracle's e4m3 decoding, pinned to the format's definition (OCP 8-bit
floating point, E4M3: bias 7, 3 mantissa bits, no infinities, S.1111.111 is
NaN) by values it fixes, and checked against the input generator's encoder
(written separately) by a round trip over every finite code."""

from __future__ import annotations

import numpy as np

import oracle
from ragged_paged_attention_rpa_gb300 import workloads

ANCHORS = {
    0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x38: 1.0,
    0x3C: 1.5, 0x40: 2.0, 0x7E: 448.0, 0x77: 240.0, 0xB8: -1.0, 0xFE: -448.0, 0x81: -(2.0 ** -9),
}


def test_anchor_values():
    codes = np.array(sorted(ANCHORS), dtype=np.uint8)
    got = oracle.decode_e4m3(codes)
    want = np.array([ANCHORS[c] for c in sorted(ANCHORS)], dtype=np.float32)
    assert np.array_equal(got, want)


def test_nan_codes_and_negative_zero():
    got = oracle.decode_e4m3(np.array([0x7F, 0xFF, 0x80], dtype=np.uint8))
    assert np.isnan(got[0]) and np.isnan(got[1])
    assert got[2] == 0.0 and np.signbit(got[2])


def test_positive_codes_increase_and_negatives_mirror():
    pos = oracle.decode_e4m3(np.arange(0x00, 0x7F, dtype=np.uint8))
    assert np.all(np.diff(pos) > 0)
    neg = oracle.decode_e4m3(np.arange(0x80, 0xFF, dtype=np.uint8))
    assert np.array_equal(neg, -pos)


def test_round_trip_through_the_generator_encoder():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF, 0x80)], dtype=np.uint8)
    vals = oracle.decode_e4m3(codes)
    assert np.array_equal(workloads.e4m3_encode(vals), codes)


def test_dequantize_applies_the_head_scale():
    codes = np.full((2, 4, 3, 8), 0x38, dtype=np.uint8)   # 1.0 everywhere
    scale = np.array([0.5, 2.0, 3.0], dtype=np.float32)
    v = oracle.dequantize_kv(codes, scale)
    for g in range(3):
        assert np.all(v[:, :, g, :] == scale[g])
