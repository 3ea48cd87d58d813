"""Pins for the oracle's E4M3FN codec, each independent of the oracle's own code.

* hand-written reference points from the OCP 8-bit floating point specification
  (tests/golden/e4m3fn_points.txt);
* the exhaustive 256-code round trip and ordering of the code table;
* a brute-force encoder (nearest of the 254 finite values by exhaustive comparison,
  ties to the even code, clamp to 448) over sweeps of binary32 values;
* an independent library: torch's float8_e4m3fn cast, on |y| <= 448.
"""
import os

import numpy as np
import pytest
import torch

from oracle.fp8_oracle import e4m3_decode, e4m3_encode

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "e4m3fn_points.txt")


def _read_golden():
    dec, enc, sect = [], [], None
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        if line.startswith("["):
            sect = line.strip("[]")
            continue
        a, b = line.split()
        if sect == "decode":
            dec.append((int(a, 16), b))
        else:
            enc.append((a, int(b, 16)))
    return dec, enc


def _parse_value(s):
    if s == "nan":
        return float("nan")
    if "p" in s or s.startswith("0x") or s.startswith("-0x"):
        return float.fromhex(s)
    return float(s)


def test_golden_decode_points():
    dec, _ = _read_golden()
    for code, sval in dec:
        v = float(e4m3_decode(np.array([code], np.uint8))[0])
        want = _parse_value(sval)
        if np.isnan(want):
            assert np.isnan(v), hex(code)
        else:
            assert v == want, (hex(code), v, want)
            assert np.signbit(v) == np.signbit(want), hex(code)


def test_golden_encode_points():
    _, enc = _read_golden()
    for sval, code in enc:
        y = np.array([_parse_value(sval)], np.float32)
        assert int(e4m3_encode(y)[0]) == code, (sval, hex(int(e4m3_encode(y)[0])), hex(code))


def test_code_table_round_trip_and_order():
    codes = np.arange(256, dtype=np.uint8)
    v = e4m3_decode(codes)
    nan = np.isnan(v)
    assert set(np.nonzero(nan)[0].tolist()) == {0x7F, 0xFF}
    finite = ~nan
    assert np.array_equal(e4m3_encode(v[finite].astype(np.float32)), codes[finite])
    pos = v[:0x7F]
    assert np.all(np.diff(pos) > 0)                       # strictly increasing magnitudes
    assert np.array_equal(v[0x80:0xFF], -pos)             # sign bit mirrors the table
    assert pos.max() == 448.0 and pos[1] == 2.0 ** -9 and pos[8] == 2.0 ** -6
    # spacing: 2^-9 through the subnormals and the first normal binade, then doubling per binade
    assert np.all(np.diff(pos[:16]) == 2.0 ** -9)
    for e in range(1, 16):
        lo = 8 * e
        hi = min(lo + 8, 0x7F)
        assert np.all(np.diff(pos[lo:hi]) == 2.0 ** (e - 10))


def _brute_force_encode(y):
    """Nearest of the 127 non-negative finite values by direct comparison, ties to the
    even code, values above 448 clamp to 448, sign copied."""
    table = e4m3_decode(np.arange(0x7F, dtype=np.uint8))   # 0x00..0x7E, increasing
    y = np.asarray(y, np.float32)
    a = np.abs(y.astype(np.float64))
    hi = np.clip(np.searchsorted(table, a, side="left"), 1, 0x7E)
    lo = hi - 1
    d_lo = a - table[lo]
    d_hi = table[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo)
    code = np.where(a >= table[-1], 0x7E, code)
    return (code | np.where(np.signbit(y), 0x80, 0)).astype(np.uint8)


def _sweep_values():
    parts = []
    # every binary32 pattern below 2^9 at a prime stride (covers all binades of E4M3)
    parts.append(np.arange(0, 0x44000000, 1009, dtype=np.uint32))
    # every pattern within +-300 ulps of each non-negative E4M3 value and midpoint
    table = e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    pts = np.concatenate([table, (table[1:] + table[:-1]) / 2, [464.0, 480.0, 2.0 ** -10]])
    base = pts.astype(np.float32).view(np.uint32).astype(np.int64)
    win = np.arange(-300, 301, dtype=np.int64)
    around = (base[:, None] + win[None, :]).ravel()
    parts.append(around[(around >= 0) & (around < 0x7F800000)].astype(np.uint32))
    u = np.concatenate(parts)
    y = u.view(np.float32)
    return np.concatenate([y, -y])


def test_encoder_matches_brute_force_on_sweep():
    y = _sweep_values()
    got = e4m3_encode(y)
    want = _brute_force_encode(y)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, [(float(y[i]), hex(got[i]), hex(want[i])) for i in bad[:10]]


def test_encoder_saturates_large_values():
    y = np.array([448.0, 448.00003, 463.99997, 464.0, 464.00003, 479.0, 480.0, 1e4, 3e38], np.float32)
    assert np.all(e4m3_encode(y) == 0x7E)
    assert np.all(e4m3_encode(-y) == 0xFE)


def test_encoder_agrees_with_torch_float8_in_range():
    rng = np.random.default_rng(123)
    y = np.concatenate([
        rng.uniform(-448, 448, 200_000),
        rng.standard_normal(200_000) * 0.01,
        np.ldexp(rng.uniform(-1, 1, 200_000), rng.integers(-14, 9, 200_000)),
    ]).astype(np.float32)
    y = y[np.abs(y) <= 448]
    t = torch.from_numpy(y).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(e4m3_encode(y), t)


def test_encoder_rejects_non_finite():
    with pytest.raises(ValueError):
        e4m3_encode(np.array([np.inf], np.float32))
    with pytest.raises(ValueError):
        e4m3_encode(np.array([np.nan], np.float32))
