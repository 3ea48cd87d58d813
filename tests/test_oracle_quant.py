"""Pins for the oracle's quantizers (1x128 activation tiles, 128x128 weight blocks,
token-dimension tiles stored transposed).

Independent references: an exact rational restatement (tests/exact_ref.py) on small
tensors, and invariants that hold at any size: the amax element encodes to +-448, no
code exceeds 448 in magnitude, the per-element error is within half an E4M3 spacing
plus the binary32 rounding of the quotient, s * 448 reproduces amax within one binary32
rounding, all-zero tiles give s = 0 and zero codes, and the tile layout is the one the
indices say (a tile only sees its own 128 elements).
"""
import numpy as np
import pytest
import torch

from oracle.fp8_oracle import (
    e4m3_decode, quant_act_1x128, quant_act_1x128_transposed, quant_w_128x128,
)
from tests.exact_ref import quantize_group


def bf16_values(a):
    return torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16).float().numpy()


def special_rows():
    """Rows of 128-element tiles exercising edge cases (all bf16 values)."""
    rng = np.random.default_rng(7)
    t = []
    t.append(rng.standard_normal(128))                                  # plain
    r = rng.standard_normal(128); r[17] = 60.0; t.append(r)             # outlier
    t.append(np.zeros(128))                                             # all-zero tile
    r = np.zeros(128); r[::2] = -0.0; r[5] = 3.0; r[6] = -0.0; t.append(r)  # signed zeros
    r = rng.standard_normal(128) * 1e-3; r[0] = 100.0; t.append(r)      # many E4M3 subnormals
    r = -np.abs(rng.standard_normal(128)); t.append(r)                  # amax from a negative value
    r = rng.standard_normal(128) * 1e30; t.append(r)                    # huge magnitudes
    r = rng.standard_normal(128) * 1e-36; t.append(r)                   # s is a binary32 subnormal
    r = np.full(128, 2.5); t.append(r)                                  # constant tile
    r = np.linspace(-7.0, 7.0, 128); t.append(r)                        # many rounding ties
    return bf16_values(np.array(t))


def test_act_quant_matches_exact_rational_restatement():
    x = special_rows().reshape(2, 5 * 128)
    q, s = quant_act_1x128(x)
    for m in range(x.shape[0]):
        for tcol in range(x.shape[1] // 128):
            tile = x[m, 128 * tcol:128 * tcol + 128]
            codes, scale = quantize_group(tile)
            assert np.float32(scale) == s[m, tcol] or (scale == 0 and s[m, tcol] == 0)
            assert q[m, 128 * tcol:128 * tcol + 128].tolist() == codes, (m, tcol)


def test_weight_quant_matches_exact_rational_restatement():
    rng = np.random.default_rng(11)
    w = rng.standard_normal((128, 256)) * 0.02
    w[3, 200] = 0.9       # outlier in block (0, 1)
    w = bf16_values(w)
    q, s = quant_w_128x128(w)
    assert q.shape == (128, 256) and s.shape == (1, 2)
    for j in range(2):
        blk = w[:, 128 * j:128 * j + 128]
        codes, scale = quantize_group(blk.ravel())
        assert np.float32(scale) == s[0, j]
        assert q[:, 128 * j:128 * j + 128].ravel().tolist() == codes


def test_transposed_quant_matches_exact_rational_restatement():
    rng = np.random.default_rng(12)
    x = rng.standard_normal((256, 8))
    x[130, 3] = 40.0
    x[:128, 5] = 0.0      # an all-zero token tile of feature 5
    x = bf16_values(x)
    q, s = quant_act_1x128_transposed(x)
    assert q.shape == (8, 256) and s.shape == (8, 2)
    for d in range(8):
        for tb in range(2):
            col = x[128 * tb:128 * tb + 128, d]
            codes, scale = quantize_group(col)
            assert np.float32(scale) == s[d, tb] or (scale == 0 and s[d, tb] == 0)
            assert q[d, 128 * tb:128 * tb + 128].tolist() == codes


def _check_invariants(x, q, s, groups_x, groups_q):
    """groups_*: arrays [..., G] of the same grouping of x and q; s[...] the group scale."""
    gx = groups_x.astype(np.float64)
    dq = e4m3_decode(groups_q)
    assert not np.any(np.isnan(dq))
    assert np.all(np.abs(dq) <= 448.0)
    amax = np.max(np.abs(gx), axis=-1)
    s64 = s.astype(np.float64)
    nz = amax > 0
    # s * 448 reproduces amax within one binary32 rounding of the quotient
    assert np.all(np.abs(s64[nz] * 448.0 - amax[nz]) <= amax[nz] * 2.0 ** -24)
    # zero groups: s = 0 and codes 0
    assert np.all(s64[~nz] == 0.0)
    assert np.all(groups_q[~nz] == 0)
    # the amax element encodes to +-448
    idx = np.argmax(np.abs(gx), axis=-1)
    top = np.take_along_axis(dq, idx[..., None], axis=-1)[..., 0]
    topx = np.take_along_axis(gx, idx[..., None], axis=-1)[..., 0]
    assert np.all(np.abs(top[nz]) == 448.0)
    assert np.all(np.sign(top[nz]) == np.sign(topx[nz]))
    # per-element error: half an E4M3 spacing at the quotient, plus its binary32 rounding
    y = np.where(nz[..., None], gx / np.where(nz, s64, 1.0)[..., None], 0.0)
    expo = np.floor(np.log2(np.maximum(np.abs(y), 2.0 ** -6)))
    half_spacing = np.exp2(expo - 4.0)
    bound = (half_spacing + np.abs(y) * 2.0 ** -23) * s64[..., None]
    err = np.abs(gx - dq * s64[..., None])
    assert np.all(err[nz] <= bound[nz] * (1 + 1e-12))


def _random_activation(M, K, seed):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((M, K))
    pos = rng.choice(M * K, size=max(1, (M * K) // 1000), replace=False)
    x.flat[pos] *= 100.0
    x[3, 256:384] = 0.0
    return bf16_values(x)


def test_act_quant_invariants_random():
    x = _random_activation(256, 1024, 3)
    q, s = quant_act_1x128(x)
    _check_invariants(x, q, s, x.reshape(256, 8, 128), q.reshape(256, 8, 128))
    assert s[3, 2] == 0.0


def test_weight_quant_invariants_random():
    rng = np.random.default_rng(4)
    w = bf16_values(rng.standard_normal((384, 512)) * 0.02)
    w[128:256, 0:128] = 0.0
    q, s = quant_w_128x128(w)
    gx = w.reshape(3, 128, 4, 128).transpose(0, 2, 1, 3).reshape(3, 4, -1)
    gq = q.reshape(3, 128, 4, 128).transpose(0, 2, 1, 3).reshape(3, 4, -1)
    _check_invariants(w, q, s, gx, gq)
    assert s[1, 0] == 0.0


def test_transposed_quant_invariants_random():
    x = _random_activation(512, 256, 5)
    q, s = quant_act_1x128_transposed(x)
    gx = x.T.reshape(256, 4, 128)
    _check_invariants(x, q, s, gx, q.reshape(256, 4, 128))


def test_tiles_are_independent():
    """Changing one tile changes exactly that tile's codes and scale."""
    x = _random_activation(128, 512, 6)
    q0, s0 = quant_act_1x128(x)
    x2 = x.copy()
    x2[77, 130] = 5000.0
    q1, s1 = quant_act_1x128(x2)
    diff_s = np.argwhere(s0 != s1)
    assert diff_s.tolist() == [[77, 1]]
    dq = np.argwhere(q0 != q1)
    assert np.all(dq[:, 0] == 77) and np.all((dq[:, 1] >= 128) & (dq[:, 1] < 256))


def test_shape_rules():
    with pytest.raises(ValueError):
        quant_act_1x128(np.zeros((2, 100), np.float32))
    with pytest.raises(ValueError):
        quant_w_128x128(np.zeros((100, 128), np.float32))
    with pytest.raises(ValueError):
        quant_act_1x128_transposed(np.zeros((100, 128), np.float32))


def test_deterministic():
    x = _random_activation(128, 256, 9)
    a = quant_act_1x128(x)
    b = quant_act_1x128(x.copy())
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_quotient_is_a_division_not_a_reciprocal_product():
    """Tiles where x / s and x * (1/s) round to different codes (tests/division_cases.py):
    the oracle must agree with the exact rational restatement of fl32(x / s)."""
    from tests.division_cases import division_sensitive_tiles
    tiles = division_sensitive_tiles(8)
    q, s = quant_act_1x128(tiles)
    for i in range(tiles.shape[0]):
        codes, scale = quantize_group(tiles[i])
        assert np.float32(scale) == s[i, 0]
        assert q[i].tolist() == codes, i


def test_weight_blocks_transpose_symmetric():
    """A 128x128 block holds the same elements in either orientation, so quantizing W^T
    gives the transposed codes and scales (the data-gradient operand W^T needs no second
    quantization); a block index swapped anywhere breaks this on a non-square grid."""
    rng = np.random.default_rng(12)
    w = bf16_values(rng.standard_normal((384, 640)) * 0.02)
    sr = special_rows()
    w[:128, 128:256] = np.stack([np.roll(sr[i % len(sr)], i) for i in range(128)])
    w[256:384, 512:640] = 0.0
    q, s = quant_w_128x128(w)
    qt, st = quant_w_128x128(np.ascontiguousarray(w.T))
    assert np.array_equal(qt, q.T) and np.array_equal(st.view(np.uint32), s.T.view(np.uint32))
    assert st.shape == (5, 3) and s[2, 4] == 0.0
