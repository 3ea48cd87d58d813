"""Pins for the oracle's delayed (history-based) scaling.

Independent references: the exact rational restatement (tests/exact_ref.py: binary32
and E4M3 rounding written out from their definitions) element by element; the special
case of a history holding exactly this tensor's maximum, which reduces to quantizing the
whole tensor as one group; saturation of every value beyond 448 s; the history shift.
"""
from fractions import Fraction
import math

import numpy as np

from oracle.fp8_oracle import e4m3_decode, quant_act_delayed
from tests.exact_ref import quantize_group, round_to_e4m3_code, round_to_f32


def bf16_values(a):
    import torch
    return torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16).float().numpy()


def exact_codes(x, hmax):
    s = round_to_f32(Fraction(float(hmax)) / 448) if hmax > 0 else Fraction(1)
    out = []
    for v in x.ravel():
        y = round_to_f32(Fraction(float(v)) / s)
        neg_zero = y == 0 and math.copysign(1.0, float(v)) < 0
        out.append(round_to_e4m3_code(y, negative_zero=neg_zero))
    return np.array(out, np.uint8).reshape(x.shape), float(s)


def test_delayed_matches_exact_restatement_with_saturation():
    rng = np.random.default_rng(40)
    x = bf16_values(rng.standard_normal((2, 256)) * 3.0)
    x[0, 5] = -0.0
    x[1, 7] = 50.0                                   # far beyond the history's maximum
    hist = np.array([2.0, 0.5, 4.0], np.float32)     # max 4 < max |x|: saturation happens
    q, s, h = quant_act_delayed(x, hist)
    want, s_exact = exact_codes(x, 4.0)
    assert np.array_equal(q, want)
    assert (s == np.float32(s_exact)).all() and s.shape == (2, 2)
    assert q[1, 7] == 0x7E and q[0, 5] == 0x80
    beyond = np.abs(x) >= 448 * s_exact
    assert beyond.any() and set(q[beyond].tolist()) <= {0x7E, 0xFE}


def test_history_equal_to_the_tensor_maximum_is_one_group_quantization():
    """With the history holding max |x| the scale is amax / 448 of the whole tensor: the
    result is the quantization of the tensor as a single group."""
    rng = np.random.default_rng(41)
    x = bf16_values(rng.standard_normal((3, 128)))
    amax = np.float32(np.abs(x).max())
    q, s, _ = quant_act_delayed(x, np.array([amax, 0.0], np.float32))
    codes, scale = quantize_group(x.ravel())
    assert np.array_equal(q.ravel(), np.array(codes, np.uint8)) and (s == np.float32(scale)).all()


def test_empty_history_uses_unit_scale():
    rng = np.random.default_rng(42)
    x = bf16_values(rng.standard_normal((1, 128)) * 100.0)
    q, s, h = quant_act_delayed(x, np.zeros(4, np.float32))
    want, s_exact = exact_codes(x, 0.0)
    assert s_exact == 1.0 and (s == 1.0).all() and np.array_equal(q, want)
    assert h[0] == np.abs(x).max() and (h[1:] == 0).all()


def test_history_shift_over_calls():
    rng = np.random.default_rng(43)
    hist = np.zeros(3, np.float32)
    seen = []
    for i in range(5):
        x = bf16_values(rng.standard_normal((1, 128)) * (i + 1))
        _, s, hist = quant_act_delayed(x, hist)
        seen.insert(0, np.float32(np.abs(x).max()))
        assert np.array_equal(hist, np.array((seen + [0, 0, 0])[:3], np.float32))


def test_dequantized_error_within_half_step_unless_saturated():
    rng = np.random.default_rng(44)
    x = bf16_values(rng.standard_normal((4, 256)))
    q, s, _ = quant_act_delayed(x, np.array([2.5], np.float32))
    d = e4m3_decode(q) * s[0, 0].astype(np.float64)
    ok = np.abs(x) < 448 * s[0, 0]
    y = np.abs(x[ok]) / s[0, 0]
    step = np.where(y < 2.0 ** -6, 2.0 ** -9, 2.0 ** (np.floor(np.log2(np.maximum(y, 2.0 ** -6))) - 3))
    assert np.all(np.abs(d[ok] - x[ok]) <= (0.5 * step + y * 2.0 ** -24) * s[0, 0] * (1 + 1e-12))
