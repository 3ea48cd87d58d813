"""The oracle's pins have teeth: plant a plausible mistake in the oracle (on the CPU,
by monkeypatching) and check that at least one pin fails.

Each planted mistake is a bug one could really write: truncating or rounding ties away
instead of to even, forgetting saturation, a wrong exponent bias, 447 for 448, a
reciprocal product for the division, weight blocks grouped along the wrong axes,
the k // 128 scale index written as k % 128, B not transposed, an off-by-one expert.
"""
import numpy as np
import pytest

import oracle.fp8_oracle as O
import tests.test_oracle_codec as TC
import tests.test_oracle_gemm as TG
import tests.test_oracle_quant as TQ

_real_encode = O.e4m3_encode
_real_decode = O.e4m3_decode


def _fails(fn):
    try:
        fn()
    except AssertionError:
        return True
    return False


def _codec_pins_fail():
    return any(_fails(f) for f in (
        TC.test_golden_decode_points, TC.test_golden_encode_points,
        TC.test_code_table_round_trip_and_order, TC.test_encoder_matches_brute_force_on_sweep,
        TC.test_encoder_saturates_large_values))


def _quant_pins_fail():
    return any(_fails(f) for f in (
        TQ.test_act_quant_matches_exact_rational_restatement,
        TQ.test_weight_quant_matches_exact_rational_restatement,
        TQ.test_transposed_quant_matches_exact_rational_restatement,
        TQ.test_quotient_is_a_division_not_a_reciprocal_product,
        TQ.test_act_quant_invariants_random, TQ.test_weight_quant_invariants_random))


def _gemm_pins_fail():
    return any(_fails(f) for f in (
        TG.test_gemm_equals_exact_sum_block_scales, TG.test_gemm_equals_exact_sum_row_scales,
        TG.test_gemm_orientation_one_hot, TG.test_gemm_scale_indexing_closed_form,
        TG.test_grouped_gemm_exact_and_empty_expert))


def _encode_with(rounder, saturate=True):
    def enc(y):
        y = np.asarray(y, np.float32)
        sign = np.where(np.signbit(y), 0x80, 0).astype(np.int64)
        a = np.abs(y.astype(np.float64))
        _, ex = np.frexp(a)
        E = np.where(a >= 2.0 ** -6, ex.astype(np.int64) - 1, -6)
        n = rounder(np.ldexp(a, (3 - E).astype(np.int32))).astype(np.int64)
        normal = a >= 2.0 ** -6
        n_sub = rounder(np.minimum(a, 2.0 ** -6) * 512.0).astype(np.int64)
        code_sub = n_sub
        carry = n == 16
        E = np.where(carry, E + 1, E)
        n = np.where(carry, 8, n)
        code = np.where(normal, ((E + 7) << 3) | (n - 8), code_sub)
        if saturate:
            code = np.where(a >= 448.0, 0x7E, code)
        else:
            code = np.where(a >= 464.0, 0x7F, code)
        return (np.clip(code, 0, 0x7F) | sign).astype(np.uint8)
    return enc


def _patch_encode(monkeypatch, enc):
    monkeypatch.setattr(O, "e4m3_encode", enc)
    monkeypatch.setattr(TC, "e4m3_encode", enc)


def test_pins_catch_truncation(monkeypatch):
    _patch_encode(monkeypatch, _encode_with(np.floor))
    assert _codec_pins_fail() and _quant_pins_fail()


def test_pins_catch_ties_away_from_zero(monkeypatch):
    _patch_encode(monkeypatch, _encode_with(lambda v: np.floor(v + 0.5)))
    assert _codec_pins_fail() and _quant_pins_fail()


def test_pins_catch_missing_saturation(monkeypatch):
    _patch_encode(monkeypatch, _encode_with(np.rint, saturate=False))
    assert _codec_pins_fail()


def test_pins_catch_wrong_exponent_bias(monkeypatch):
    def dec(codes):
        return _real_decode(codes) * 0.5
    monkeypatch.setattr(O, "e4m3_decode", dec)
    monkeypatch.setattr(TC, "e4m3_decode", dec)
    assert _codec_pins_fail()


def _quantize_groups_variant(divisor=448.0, reciprocal=False):
    def qg(g):
        g = np.asarray(g, np.float32)
        amax = np.max(np.abs(g), axis=-1)
        s = (amax / np.float32(divisor)).astype(np.float32)
        zero = s == 0
        sd = np.where(zero, np.float32(1.0), s).astype(np.float32)
        if reciprocal:
            y = (g * (np.float32(1.0) / sd).astype(np.float32)[..., None]).astype(np.float32)
        else:
            y = (g / sd[..., None]).astype(np.float32)
        q = np.where(zero[..., None], np.uint8(0), O.e4m3_encode(y)).astype(np.uint8)
        return q, s
    return qg


def test_pins_catch_wrong_max_constant(monkeypatch):
    monkeypatch.setattr(O, "_quantize_groups", _quantize_groups_variant(divisor=447.0))
    assert _quant_pins_fail()


def test_pins_catch_reciprocal_product(monkeypatch):
    monkeypatch.setattr(O, "_quantize_groups", _quantize_groups_variant(reciprocal=True))
    assert _quant_pins_fail()


def test_pins_catch_weight_blocks_on_wrong_axes(monkeypatch):
    def bad_w(w):
        w = np.asarray(w, np.float32)
        N, K = w.shape
        # groups 128 consecutive rows of 128 elements of the flattened array (no transpose)
        q, s = O._quantize_groups(w.reshape(N // 128, K // 128, 128 * 128))
        return q.reshape(N, K), s
    monkeypatch.setattr(TQ, "quant_w_128x128", bad_w)
    assert _quant_pins_fail()


def test_pins_catch_scale_index_modulo(monkeypatch):
    def bad_rows(q, s):
        K = q.shape[1]
        idx = np.arange(K) % s.shape[1]
        return _real_decode(q) * np.asarray(s, np.float64)[:, idx]
    monkeypatch.setattr(O, "dequant_rows_1x128", bad_rows)
    assert _gemm_pins_fail()


def test_pins_catch_untransposed_b(monkeypatch):
    real = O.blockscaled_gemm

    def bad(qa, sa, qb, sb, sb_kind=0, rows=None):
        A = O.dequant_rows_1x128(np.asarray(qa)[rows] if rows is not None else qa,
                                 np.asarray(sa)[rows] if rows is not None else sa)
        B = O.dequant_b(np.asarray(qb), np.asarray(sb), sb_kind)
        if B.shape[0] != B.shape[1]:
            return real(qa, sa, qb, sb, sb_kind, rows) * 0.0 + 1.0
        return A @ B
    monkeypatch.setattr(TG, "blockscaled_gemm", bad)
    assert _gemm_pins_fail()


def test_pins_catch_off_by_one_expert(monkeypatch):
    def bad_grouped(qa, sa, qb, sb, group_offsets, experts=None):
        off = np.asarray(group_offsets, np.int64)
        E = np.asarray(qb).shape[0]
        C = np.zeros((np.asarray(qa).shape[0], np.asarray(qb).shape[1]))
        for e in range(E):
            lo, hi = int(off[e]), int(off[e + 1])
            if hi > lo:
                C[lo:hi] = O.blockscaled_gemm(qa[lo:hi], sa[lo:hi], qb[(e + 1) % E], sb[(e + 1) % E])
        return C
    monkeypatch.setattr(TG, "grouped_gemm", bad_grouped)
    assert _gemm_pins_fail()


def test_unpatched_oracle_passes_all_pins():
    assert not _codec_pins_fail()
    assert not _quant_pins_fail()
    assert not _gemm_pins_fail()
