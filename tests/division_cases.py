"""Activation tiles on which dividing by the scale and multiplying by its binary32
reciprocal give different E4M3 codes.

The cast reads q = E4M3(fl32(x / s)). fl32(x * fl32(1 / s)) differs from fl32(x / s) by
at most a couple of binary32 units, which changes the E4M3 code only when the quotient
sits next to a rounding midpoint of E4M3; random data almost never does that. These
tiles are built to hit it, so that a check that passes on them fixes the division
reading. The search uses plain numpy binary32 arithmetic and a nearest-value rounding
written here, not the oracle.
"""
import numpy as np


def _nearest_e4m3_magnitude(y):
    # non-negative finite E4M3FN values from the field definition, increasing
    vals = [m / 512.0 if e == 0 else (1 + m / 8.0) * 2.0 ** (e - 7) for e in range(16) for m in range(8)][:127]
    t = np.array(vals)
    a = np.abs(np.asarray(y, np.float64))
    hi = np.clip(np.searchsorted(t, a), 1, 126)
    lo = hi - 1
    dl, dh = a - t[lo], t[hi] - a
    idx = np.where((dh < dl) | ((dh == dl) & (hi % 2 == 0)), hi, lo)
    return np.where(a >= 448.0, 126, idx)


def division_sensitive_tiles(n_tiles=16, seed=2024):
    """float32 array [n_tiles, 128] of bf16 values; element 0 of each tile is its amax."""
    rng = np.random.default_rng(seed)
    bf16 = (np.arange(0x0080, 0x7F80, dtype=np.uint32) << 16).view(np.float32)
    pool = bf16[(bf16 > 2.0 ** -12) & (bf16 < 2.0 ** 12)]
    tiles = []
    while len(tiles) < n_tiles:
        amax = np.float32(rng.choice(pool))
        s = np.float32(amax / np.float32(448.0))
        if s == 0:
            continue
        x = pool[pool <= amax]
        yd = (x / s).astype(np.float32)
        ym = (x * np.float32(np.float32(1.0) / s)).astype(np.float32)
        hits = x[_nearest_e4m3_magnitude(yd) != _nearest_e4m3_magnitude(ym)]
        if hits.size == 0:
            continue
        hits = hits[:63]
        fill = rng.standard_normal(127 - 2 * hits.size).astype(np.float32) * np.float32(amax) * np.float32(0.3)
        body = np.concatenate([hits, -hits, fill]).astype(np.float32)
        rng.shuffle(body)
        tiles.append(np.concatenate([[amax], body]).astype(np.float32))
    out = np.stack(tiles)
    # round the filler to bf16 values (hits and amax already are)
    u = out.view(np.uint32)
    u = ((u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000).astype(np.uint32)
    return u.view(np.float32)
