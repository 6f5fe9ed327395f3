"""Pins for the oracle's E4M3FN decode / encode (CPU only).

The checks do not reuse the oracle's formulas: decode is pinned by format
facts and by structure (monotone, symmetric, 254 finite codes); encode is
pinned by the tie values printed in sglang PR #33533 (Motivation) and by a
brute-force nearest-value
search over the decoded grid, run exhaustively over every fp32 input in the
range where rounding happens.
"""
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "e4m3_pins.txt")


def _load_pins():
    rows = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                a, b = line.split()
                rows.append((int(a, 16), int(b, 16)))
    return rows


def test_decode_format_facts():
    codes = np.arange(256, dtype=np.uint8)
    v = oracle.e4m3_decode(codes)
    assert v[0x7E] == 448.0 and v[0xFE] == -448.0
    assert v[0x38] == 1.0 and v[0xB8] == -1.0
    assert v[0x01] == 2.0 ** -9 and v[0x07] == 7 * 2.0 ** -9 and v[0x08] == 2.0 ** -6
    assert v[0x00] == 0.0 and np.signbit(v[0x80])
    assert np.isnan(v[0x7F]) and np.isnan(v[0xFF])
    assert np.isfinite(v).sum() == 254
    # positive codes 0..126 are strictly increasing; the sign bit mirrors them
    pos = v[:127]
    assert np.all(np.diff(pos) > 0)
    assert np.array_equal(v[128:255], -pos)
    # each binade holds 8 evenly spaced values: (8+m) * 2^(e-10)
    for e in range(1, 16):
        for m in range(8):
            c = (e << 3) | m
            if c == 0x7F:
                continue
            assert v[c] == (8 + m) * 2.0 ** (e - 10)


def test_encode_golden_pins():
    pins = _load_pins()
    x = np.array([p[0] for p in pins], np.uint32).view(np.float32)
    want = np.array([p[1] for p in pins], np.uint8)
    got = oracle.e4m3_encode(x)
    bad = [(hex(p[0]), hex(p[1]), hex(int(g))) for p, g in zip(pins, got) if p[1] != g]
    assert not bad, bad


def test_encode_roundtrip_all_finite_codes():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    vals = oracle.e4m3_decode(codes).astype(np.float32)
    assert np.array_equal(oracle.e4m3_encode(vals), codes)


def _brute_force_encode(x32: np.ndarray) -> np.ndarray:
    """Nearest finite E4M3 value by search over the decoded grid; ties to
    the code with an even last bit; magnitudes beyond 448 saturate."""
    grid = oracle.e4m3_decode(np.arange(127, dtype=np.uint8))     # 0 .. 448, increasing
    a = np.abs(x32.astype(np.float64))
    a = np.minimum(a, 448.0)
    hi = np.searchsorted(grid, a, side="left")                     # grid[hi] >= a
    hi = np.minimum(hi, 126)
    lo = np.maximum(hi - 1, 0)
    d_lo = a - grid[lo]
    d_hi = grid[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    exact = grid[hi] == a
    code = np.where(exact | pick_hi, hi, lo).astype(np.uint8)
    return code | np.where(np.signbit(x32), 0x80, 0).astype(np.uint8)


def test_encode_exhaustive_positive_rounding_range():
    # every positive fp32 in [2^-11, 2^10): all rounding and saturation cases
    for biased in range(127 - 11, 127 + 10):
        bits = (np.uint32(biased) << np.uint32(23)) | np.arange(1 << 23, dtype=np.uint32)
        x = bits.view(np.float32)
        got = oracle.e4m3_encode(x)
        want = _brute_force_encode(x)
        n_bad = int(np.count_nonzero(got != want))
        assert n_bad == 0, (biased, n_bad)


def test_encode_negative_and_extremes_sampled():
    rng = np.random.default_rng(7)
    # negative binades around the top of the range, and random bit patterns
    parts = []
    for biased in (127 - 10, 127 + 2, 127 + 8, 127 + 9):
        bits = (np.uint32(0x100 | biased) << np.uint32(23)) | np.arange(1 << 23, dtype=np.uint32)
        parts.append(bits)
    parts.append(rng.integers(0, 2 ** 32, size=4_000_000, dtype=np.uint64).astype(np.uint32))
    bits = np.concatenate(parts)
    x = bits.view(np.float32)
    x = x[~np.isnan(x)]
    got = oracle.e4m3_encode(x)
    want = _brute_force_encode(x)
    assert np.array_equal(got, want)
