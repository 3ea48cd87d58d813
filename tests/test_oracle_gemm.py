"""Pins for the oracle's block-scaled GEMM and grouped GEMM.

* exact rational sums (tests/exact_ref.py) on small random operands, both scale kinds;
* orientation (C = A . B^T, both operands K-contiguous) with one-hot A rows;
* scale indexing with all-one codes and distinct power-of-two scales (closed form);
* grouped GEMM: exact sums per expert, an empty expert, and padding rows giving 0.
"""
from fractions import Fraction

import numpy as np

from oracle.fp8_oracle import (
    SB_BLOCK_128x128, SB_ROW_1x128, blockscaled_gemm, e4m3_decode, grouped_gemm, relative_error,
)
from tests.exact_ref import exact_gemm_entry


def random_codes(rng, shape):
    c = rng.integers(0, 256, size=shape, dtype=np.int64).astype(np.uint8)
    nan = (c & 0x7F) == 0x7F
    c[nan] = 0x7E
    return c


def random_scales(rng, shape):
    # positive binary32 scales spanning a few binades, as amax / 448 would be
    return (rng.uniform(0.5, 2.0, shape) * 2.0 ** rng.integers(-8, 3, shape)).astype(np.float32)


def _sum_abs_terms(qa_row, sa_row, qb_row, sbk):
    a = np.abs(e4m3_decode(qa_row)) * np.repeat(sa_row.astype(np.float64), 128)
    b = np.abs(e4m3_decode(qb_row)) * np.repeat(np.array([sbk(i) for i in range(len(sa_row))], np.float64), 128)
    return float(np.sum(a * b))


def test_gemm_equals_exact_sum_block_scales():
    rng = np.random.default_rng(21)
    M, N, K = 3, 256, 256
    qa, qb = random_codes(rng, (M, K)), random_codes(rng, (N, K))
    sa, sb = random_scales(rng, (M, K // 128)), random_scales(rng, (N // 128, K // 128))
    C = blockscaled_gemm(qa, sa, qb, sb, SB_BLOCK_128x128)
    assert C.shape == (M, N) and C.dtype == np.float64
    for m in range(M):
        for n in (0, 1, 127, 128, 200, 255):
            sbk = lambda kb, n=n: sb[n // 128, kb]
            exact = exact_gemm_entry(qa[m], sa[m], qb[n], sbk)
            bound = K * 2.0 ** -53 * _sum_abs_terms(qa[m], sa[m], qb[n], sbk)
            assert abs(Fraction(float(C[m, n])) - exact) <= Fraction(bound), (m, n)


def test_gemm_equals_exact_sum_row_scales():
    rng = np.random.default_rng(22)
    M, N, K = 2, 5, 384
    qa, qb = random_codes(rng, (M, K)), random_codes(rng, (N, K))
    sa, sb = random_scales(rng, (M, K // 128)), random_scales(rng, (N, K // 128))
    C = blockscaled_gemm(qa, sa, qb, sb, SB_ROW_1x128)
    for m in range(M):
        for n in range(N):
            sbk = lambda kb, n=n: sb[n, kb]
            exact = exact_gemm_entry(qa[m], sa[m], qb[n], sbk)
            bound = K * 2.0 ** -53 * _sum_abs_terms(qa[m], sa[m], qb[n], sbk)
            assert abs(Fraction(float(C[m, n])) - exact) <= Fraction(bound), (m, n)


def test_gemm_orientation_one_hot():
    """A row m = e_m (code 1.0 at k = m, scale 1) picks column m of B: C[m, n] = B[n, m]."""
    rng = np.random.default_rng(23)
    M, N, K = 6, 128, 256
    qa = np.zeros((M, K), np.uint8)
    for m in range(M):
        qa[m, 130 + m] = 0x38
    sa = np.ones((M, 2), np.float32)
    qb = random_codes(rng, (N, K))
    sb = random_scales(rng, (1, 2))
    C = blockscaled_gemm(qa, sa, qb, sb, SB_BLOCK_128x128)
    for m in range(M):
        for n in range(N):
            assert C[m, n] == float(e4m3_decode(qb[n:n + 1, 130 + m])[0]) * float(sb[0, 1])


def test_gemm_scale_indexing_closed_form():
    """All codes 1.0: C[m, n] = 128 * sum_kb sa[m, kb] * sb(n, kb), exact for powers of two."""
    M, N, K = 4, 256, 384
    qa = np.full((M, K), 0x38, np.uint8)
    qb = np.full((N, K), 0x38, np.uint8)
    sa = np.array([[2.0 ** (m + 3 * kb) for kb in range(3)] for m in range(M)], np.float32)
    sb_blk = np.array([[2.0 ** (-kb - 5 * nb) for kb in range(3)] for nb in range(2)], np.float32)
    C = blockscaled_gemm(qa, sa, qb, sb_blk, SB_BLOCK_128x128)
    for m in range(M):
        for n in (0, 127, 128, 255):
            want = 128.0 * sum(float(sa[m, kb]) * float(sb_blk[n // 128, kb]) for kb in range(3))
            assert C[m, n] == want
    sb_row = np.array([[2.0 ** (-(n % 7) - kb) for kb in range(3)] for n in range(N)], np.float32)
    C = blockscaled_gemm(qa, sa, qb, sb_row, SB_ROW_1x128)
    for m in range(M):
        for n in (0, 1, 6, 200):
            want = 128.0 * sum(float(sa[m, kb]) * float(sb_row[n, kb]) for kb in range(3))
            assert C[m, n] == want


def test_gemm_row_subset_matches_full():
    rng = np.random.default_rng(24)
    qa, qb = random_codes(rng, (256, 256)), random_codes(rng, (128, 256))
    sa, sb = random_scales(rng, (256, 2)), random_scales(rng, (1, 2))
    full = blockscaled_gemm(qa, sa, qb, sb)
    rows = np.array([0, 5, 255, 128])
    # same entries up to the float64 summation order the matrix-product library picks
    assert relative_error(blockscaled_gemm(qa, sa, qb, sb, rows=rows), full[rows]) <= 1e-13


def test_grouped_gemm_exact_and_empty_expert():
    rng = np.random.default_rng(25)
    E, N, K = 3, 128, 256
    off = np.array([0, 128, 128, 256], np.int32)          # expert 1 has no rows
    qa = random_codes(rng, (256, K))
    qa[200:] = 0                                            # padding rows of expert 2
    sa = random_scales(rng, (256, 2))
    sa[200:] = 0.0
    qb = random_codes(rng, (E, N, K))
    sb = random_scales(rng, (E, 1, 2))
    C = grouped_gemm(qa, sa, qb, sb, off)
    assert C.shape == (256, N)
    assert np.all(C[200:] == 0.0)
    for m, e in ((0, 0), (127, 0), (128, 2), (199, 2)):
        for n in (0, 77, 127):
            sbk = lambda kb, e=e: sb[e, 0, kb]
            exact = exact_gemm_entry(qa[m], sa[m], qb[e, n], sbk)
            bound = K * 2.0 ** -53 * _sum_abs_terms(qa[m], sa[m], qb[e, n], sbk)
            assert abs(Fraction(float(C[m, n])) - exact) <= Fraction(bound), (m, n)
    only2 = grouped_gemm(qa, sa, qb, sb, off, experts=[2])
    assert np.all(only2[:128] == 0.0) and relative_error(only2[128:], C[128:]) <= 1e-13


def test_relative_error_measure():
    ref = np.array([[1.0, -4.0], [2.0, 0.5]])
    assert relative_error(ref, ref) == 0.0
    assert relative_error(ref + np.array([[0.0, 0.0], [0.0, 0.25]]), ref) == 0.25 / 4.0
    assert relative_error(np.zeros((0, 3)), np.zeros((0, 3))) == 0.0
    assert relative_error(np.ones(2), np.zeros(2)) == float("inf")


def test_gemm_e4m3_output_closed_form():
    """A = ones (code 0x38, scale 1), K = 128, B row n constant with value v_n, so
    C[m, n] = 128 v_n sb_n exactly; with v_n = k n / 8 patterns the tile maxima and
    quotients are known rationals and the codes are checked against the exact
    restatement (rational arithmetic, nearest E4M3 value by table search).
    v_n = ((n mod 13) - 6) / 2 are E4M3 values (at most 3 significant bits)."""
    from oracle.fp8_oracle import blockscaled_gemm_e4m3, e4m3_encode
    from tests.exact_ref import quantize_group
    M, N, K = 3, 256, 128
    qa = np.full((M, K), 0x38, np.uint8)
    sa = np.ones((M, 1), np.float32)
    vals = np.array([((n % 13) - 6) / 2.0 for n in range(N)], np.float32)
    codes = e4m3_encode(vals)
    qb = np.repeat(codes[:, None], K, axis=1)
    sb = np.array([[0.5], [4.0]], np.float32)                                 # 128x128 blocks of B
    q, s, c32 = blockscaled_gemm_e4m3(qa, sa, qb, sb)
    dec = np.array([float(v) for v in vals])
    for n in range(N):
        assert c32[0, n] == np.float32(128.0 * dec[n] * sb[n // 128, 0])
    for t in range(2):
        want_codes, want_s = quantize_group(c32[1, 128 * t:128 * t + 128])
        assert np.float32(want_s) == s[1, t]
        assert q[1, 128 * t:128 * t + 128].tolist() == want_codes
    # the tile maximum |C| = 128 * 3 * sb sets the scale, and its elements encode to +-448
    assert s[0, 0] == np.float32(128 * 3 * 0.5 / 448) and s[0, 1] == np.float32(128 * 3 * 4.0 / 448)
    assert set(q[0][np.abs(c32[0]) == np.abs(c32[0]).max()].tolist()) <= {0x7E, 0xFE}


def test_quantizer_on_binary32_values_matches_exact_restatement():
    """The GEMM epilogue quantizes FP32 (not bf16) values: tiles of random binary32
    values, values placed on and next to E4M3 rounding midpoints of x / s, signed zeros
    and tiny magnitudes, against the exact rational restatement."""
    from oracle.fp8_oracle import quant_act_1x128
    from tests.exact_ref import quantize_group
    rng = np.random.default_rng(21)
    rows = [rng.standard_normal(128).astype(np.float32) * np.float32(3.7)]
    r = rng.standard_normal(128).astype(np.float32); r[0] = np.float32(448.0)   # s = 1: midpoints exact
    r[1:20] = np.float32(1.0625); r[20:40] = np.nextafter(np.float32(1.0625), np.float32(2)); r[40] = -0.0
    r[41] = np.float32(-2 ** -10); r[42] = np.float32(2 ** -10); r[43] = np.float32(3 * 2 ** -11)
    rows.append(r)
    rows.append((rng.random(128) * 1e-30).astype(np.float32))
    rows.append((rng.standard_normal(128) * 1e20).astype(np.float32))
    x = np.array(rows, np.float32)
    q, s = quant_act_1x128(x)
    for m in range(x.shape[0]):
        codes, scale = quantize_group(x[m])
        assert np.float32(scale) == s[m, 0]
        assert q[m].tolist() == codes, m
