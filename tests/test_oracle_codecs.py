"""Pins of the oracle's number codecs against independent definitions.

Each check restates the format from its bit fields (or searches the value
grid exhaustively) in Python; none re-calls the oracle's own tables.
"""
import math
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_pairs(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            a, b = line.split()
            rows.append((int(a), float(b)))
    return rows


def _e2m1_from_bits(code):
    s, e, m = (code >> 3) & 1, (code >> 1) & 3, code & 1
    mag = (2.0 ** (e - 1)) * (1 + m / 2) if e > 0 else m / 2
    return -mag if s else mag


def test_e2m1_table_matches_golden_and_bitfields():
    golden = _read_pairs("e2m1_values.txt")
    assert [c for c, _ in golden] == list(range(16))
    for code, val in golden:
        got = oracle.e2m1_value(code)
        assert got == val and math.copysign(1, got) == math.copysign(1, val), code
        assert got == _e2m1_from_bits(code)
    # code 8 is negative zero
    assert math.copysign(1.0, oracle.e2m1_value(8)) == -1.0


def test_e8m0_closed_form():
    for byte, val in _read_pairs("e8m0_examples.txt"):
        assert oracle.e8m0_value(byte) == val
    for b in range(1, 255):
        assert oracle.e8m0_value(b) == math.ldexp(1.0, b - 127) == 2.0 ** (b - 127)


def _e4m3_from_bits(code):
    s, e, m = (code >> 7) & 1, (code >> 3) & 15, code & 7
    if e == 15 and m == 7:
        return float("nan")
    mag = m * 2.0 ** -9 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7)
    return -mag if s else mag


def test_e4m3_decode_all_codes():
    for code in range(256):
        ref = _e4m3_from_bits(code)
        got = oracle.e4m3_value(code)
        if math.isnan(ref):
            assert math.isnan(got)
        else:
            assert got == ref and math.copysign(1, got) == math.copysign(1, ref), hex(code)
    assert oracle.e4m3_value(0x7E) == 448.0
    assert oracle.e4m3_value(0x01) == 2.0 ** -9


def _bf16_values(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def test_bf16_to_e4m3_exhaustive_nearest_even():
    """All 65,536 bf16 inputs against an exhaustive nearest search over the
    finite e4m3 grid (ties to the even code, saturation at 448, sign kept)."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    x = _bf16_values(bits)
    finite = np.isfinite(x)
    got = oracle.bf16_to_e4m3(bits)

    codes = np.array([c for c in range(128) if c != 0x7F], dtype=np.int64)  # + magnitudes
    vals = np.array([_e4m3_from_bits(c) for c in codes])
    ax = np.abs(x[finite])
    big = ax >= 448.0            # satfinite: everything at or past the top saturates
    ax = np.where(big, 448.0, ax)
    dist = np.abs(ax[:, None] - vals[None, :])
    best = dist.min(axis=1, keepdims=True)
    cand = dist == best
    # among ties pick the even code; adjacent codes differ in their lowest bit
    n_c = cand.sum(axis=1)
    assert n_c.max() <= 2
    even = cand & ((codes[None, :] & 1) == 0)
    pick = np.where(n_c == 1, np.argmax(cand, axis=1), np.argmax(even, axis=1))
    ref_mag = codes[pick]
    sign = np.signbit(x[finite]).astype(np.int64) << 7
    ref = (ref_mag | sign).astype(np.uint8)
    np.testing.assert_array_equal(got[finite], ref)

    # infinities saturate like any |x| >= 448
    inf_idx = np.where(np.isinf(x))[0]
    for i in inf_idx:
        assert got[i] == (0xFE if x[i] < 0 else 0x7E)


def test_e4m3_rounding_spot_values():
    # ties: 1 + 1/16 lies halfway between 1 (code 0x38) and 1.125 (0x39) -> even 0x38
    assert oracle.e4m3_from_double(1.0625) == 0x38
    # 1.1875 halfway between 1.125 (0x39) and 1.25 (0x3A) -> even 0x3A
    assert oracle.e4m3_from_double(1.1875) == 0x3A
    # subnormal tie 0.5 * 2^-9 -> +0; 1.5 * 2^-9 -> 2 * 2^-9
    assert oracle.e4m3_from_double(2.0 ** -10) == 0x00
    assert oracle.e4m3_from_double(-(2.0 ** -10)) == 0x80
    assert oracle.e4m3_from_double(1.5 * 2.0 ** -9) == 0x02
    assert oracle.e4m3_from_double(1000.0) == 0x7E
    assert oracle.e4m3_from_double(-464.0) == 0xFE
