"""Plain CPU oracle for fine-grained FP8 quantization and the block-scaled FP8 GEMM.

TEST INFRASTRUCTURE. This module is the slow, obviously correct statement of what
the hot path computes. Only the test suite, ``__graft_entry__.smoke()`` and the CPU
baseline / reference arm of ``bench.py`` may import it. The product (the CUDA
library and its Python binding) never imports, calls or links anything here, and
this module imports nothing from the product.

What it computes, with the passages it follows (the five knowledge-base pages on
DeepSeek-V3 FP8 training; each is cited by its title and section):

* "Online quantization vs delayed quantization in DeepSeek-V3" (Russian page),
  item 1: a scaling factor is computed dynamically for every 1x128 activation tile
  and every 128x128 weight block from the data being processed (items 2-3: no
  history of maxima is kept).
* "Unified E4M3 format in DeepSeek-V3" (Arabic page), section
  "fine-grained quantization strategy": activations are grouped and scaled per
  1x128 tile, weights per 128x128 block, and E4M3 is used in every pass (forward
  and backward).
* "Advantages of using FP8 for GEMM operations in DeepSeek-V3" (Italian page),
  item 5: partial
  sums of the tensor-core accumulation are promoted to FP32 at fixed intervals;
  item 6: one E4M3 format for all tensors, the per-group scale acting as a shared
  exponent; item 8: a dense and a MoE (grouped) FP8 GEMM.

Readings where the pages are silent (each also listed in the design notes):

* scale s = fl32(amax / 448), 448 being the largest finite E4M3FN value; the
  element is divided by s in IEEE binary32 (round to nearest even) and the fp32
  quotient is then rounded to E4M3FN (round to nearest, ties to even, saturating
  to +-448, sign kept, so a negative value that rounds to zero gives 0x80);
* a tile whose amax is 0 gets s = +0.0 and all-zero codes (0x00);
* the GEMM result is C[m,n] = sum_k dec(qa[m,k]) sa[m,k/128] dec(qb[n,k]) sb(n,k),
  accumulated in float64 (the FP32 promotion of the pages reaches the same value up
  to fp32 rounding); C = A . B^T with both operands K-contiguous;
* the grouped GEMM is the dense GEMM applied to each expert's contiguous rows;
* delayed scaling (the contrast of the Russian page, items 2-3) keeps one scale per
  tensor from the maxima of earlier calls: s = fl32(max(history) / 448), s = 1 for an
  empty history, codes E4M3(fl32(x / s)) saturating, and this call's max |x| enters
  the history;
* a GEMM whose output stays in FP8 (the Arabic page's memory section: activations
  stored in FP8) quantizes its FP32 result in 1x128 tiles along N with the activation
  quantizer, without rounding to BF16 first; the oracle's FP32 result is the float64
  sum rounded once to binary32.

E4M3FN is the OCP 8-bit floating point format "E4M3": bit layout s.eeee.mmm,
exponent bias 7, subnormals at e = 0 (value m * 2^-9), no infinities, NaN only at
s.1111.111, largest finite value 448 (0.1111.110).

Parity pins: every function here is pinned in ``tests/test_oracle_*.py`` against
closed forms, exhaustive code tables, exact rational arithmetic and brute force.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0       # largest finite E4M3FN value, 0x7E
TILE = 128             # 1x128 activation tiles, 128x128 weight blocks, 128-deep K chunks


# --------------------------------------------------------------------------- codec


def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    """Value of each E4M3FN byte as float64 (NaN for the two NaN codes).

    Field definition: sign s = bit 7, exponent e = bits 6..3, mantissa m = bits 2..0;
    e == 0 -> (-1)^s * m * 2^-9; e == 15 and m == 7 -> NaN; else (-1)^s * (1 + m/8) * 2^(e-7).
    """
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    s = (c >> 7) & 1
    e = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    val = np.where(s == 1, -mag, mag)
    return np.where((e == 15) & (m == 7), np.nan, val)


def e4m3_encode(y: np.ndarray) -> np.ndarray:
    """Round binary32 values to E4M3FN bytes: nearest, ties to even, saturate to +-448.

    Works on the value, not on bit patterns: in the normal range [2^-6, 448) the
    spacing of E4M3FN numbers in the binade [2^E, 2^(E+1)) is 2^(E-3); below 2^-6
    the spacing is the subnormal quantum 2^-9. The value divided by its spacing is
    rounded to the nearest integer with ties to even (np.rint, exact in float64
    because the division is by a power of two). Inputs must be finite.
    """
    y = np.asarray(y, dtype=np.float32)
    if not np.all(np.isfinite(y)):
        raise ValueError("e4m3_encode: inputs must be finite")
    sign = np.where(np.signbit(y), 0x80, 0x00).astype(np.int64)
    a = np.abs(y.astype(np.float64))

    # binade exponent E with 2^E <= a < 2^(E+1); frexp gives a = f * 2^ex, f in [0.5, 1)
    _, ex = np.frexp(a)
    E = ex.astype(np.int64) - 1
    normal = a >= 2.0 ** -6

    # subnormal range: spacing 2^-9, n in 0..8 (8 means the smallest normal 2^-6)
    n_sub = np.rint(np.minimum(a, 2.0 ** -6) * 2.0 ** 9).astype(np.int64)
    code_sub = np.where(n_sub == 8, 0x08, n_sub)

    # normal range: spacing 2^(E-3), n in 8..16 (16 carries into the next binade)
    En = np.where(normal, E, -6)
    n_nrm = np.rint(np.ldexp(a, (3 - En).astype(np.int32))).astype(np.int64)
    carry = n_nrm == 16
    En = np.where(carry, En + 1, En)
    n_nrm = np.where(carry, 8, n_nrm)
    code_nrm = ((En + 7) << 3) | (n_nrm - 8)

    code = np.where(normal, code_nrm, code_sub)
    # saturation: 448 is the largest finite value; every a >= 448 rounds (or clamps) to it
    code = np.where(a >= E4M3_MAX, 0x7E, code)
    return (code | sign).astype(np.uint8)


# --------------------------------------------------------------------------- quantizers


def _quantize_groups(g: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """Quantize groups laid out as g[..., group_elements] (float32 values).

    Per group: amax = max |x| (exact), s = fl32(amax / 448), q = E4M3(fl32(x / s)).
    A group with amax == 0 gets s = 0 and codes 0x00.
    """
    g = np.asarray(g, dtype=np.float32)
    amax = np.max(np.abs(g), axis=-1)                           # float32, exact
    s = (amax / np.float32(E4M3_MAX)).astype(np.float32)        # IEEE binary32 division
    zero = s == np.float32(0.0)
    s_div = np.where(zero, np.float32(1.0), s).astype(np.float32)
    y = (g / s_div[..., None]).astype(np.float32)               # IEEE binary32 division
    q = e4m3_encode(y)
    q = np.where(zero[..., None], np.uint8(0), q).astype(np.uint8)
    return q, s


def quant_act_1x128(x: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """Activation quantization in 1x128 tiles along the last (K) dimension.

    x: float32 [M, K] (bf16 values for activations; any binary32 values work), K % 128 == 0.
    Returns q uint8 [M, K] (E4M3FN codes) and s float32 [M, K/128], s[m, t] being the
    scale of columns 128t .. 128t+127 of row m; x[m, k] ~= dec(q[m, k]) * s[m, k // 128].
    Follows the Russian page, item 1, and the Arabic page, "fine-grained strategy".
    """
    x = np.asarray(x, dtype=np.float32)
    M, K = x.shape
    if K % TILE:
        raise ValueError("K must be a multiple of 128")
    q, s = _quantize_groups(x.reshape(M, K // TILE, TILE))
    return q.reshape(M, K), s


def quant_act_1x128_transposed(x: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """Activation quantization in 1x128 tiles along the first (token) dimension.

    x: float32 [T, D] (T tokens, D features), T % 128 == 0. Each tile is 128
    consecutive tokens of one feature column. The result is stored transposed, so
    that the token dimension is contiguous: q uint8 [D, T], s float32 [D, T/128],
    x[t, d] ~= dec(q[d, t]) * s[d, t // 128]. This is the operand layout of a
    weight-gradient GEMM dW = dY^T X, in which the token dimension is the reduction;
    the Arabic page says E4M3 with 1x128 activation tiles is used in the backward
    pass as well.
    """
    x = np.asarray(x, dtype=np.float32)
    if x.shape[0] % TILE:
        raise ValueError("T must be a multiple of 128")
    return quant_act_1x128(np.ascontiguousarray(x.T))


def quant_act_delayed(x: np.ndarray, history: np.ndarray):
    """Delayed (history-based) scaling of a tensor, the contrast to online scaling.

    x: float32 [M, K] (bf16 values), K % 128 == 0; history: float32 [H], the per-tensor
    maxima of the H previous calls, most recent first.
    s = fl32(max(history) / 448), or 1 when that maximum is 0; q = E4M3(fl32(x / s)),
    saturating (a quotient beyond the binary32 range is infinite and saturates too).
    Returns q uint8 [M, K], the tile scales float32 [M, K/128] (all equal to s) and the
    new history [H]: max |x| first, the oldest entry dropped.
    Follows the Russian page, items 2-3 (delayed quantization relies on historical
    maxima that have to be stored).
    """
    x = np.asarray(x, dtype=np.float32)
    history = np.asarray(history, dtype=np.float32)
    M, K = x.shape
    if K % TILE:
        raise ValueError("K must be a multiple of 128")
    hmax = np.float32(history.max()) if history.size else np.float32(0.0)
    s = (hmax / np.float32(E4M3_MAX)).astype(np.float32) if hmax > 0 else np.float32(1.0)
    with np.errstate(over="ignore"):
        y = (x / s).astype(np.float32)                            # IEEE binary32 division
    # an infinite quotient lies beyond 448 like any other overflowing one: saturate it
    y = np.where(np.isinf(y), np.copysign(np.float32(2 * E4M3_MAX), y), y).astype(np.float32)
    q = e4m3_encode(y)
    tiles = np.full((M, K // TILE), s, np.float32)
    amax = np.float32(np.max(np.abs(x))) if x.size else np.float32(0.0)
    new_history = np.concatenate([[amax], history[:-1]]).astype(np.float32)
    return q, tiles, new_history


def quant_w_128x128(w: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """Weight quantization in 128x128 blocks.

    w: float32 [N, K] holding bf16 values, N % 128 == 0, K % 128 == 0.
    Returns q uint8 [N, K] and s float32 [N/128, K/128], s[i, j] the scale of rows
    128i.. and columns 128j.. ; w[n, k] ~= dec(q[n, k]) * s[n // 128, k // 128].
    Follows the Russian page, item 1, and the Arabic page, "fine-grained strategy".
    """
    w = np.asarray(w, dtype=np.float32)
    N, K = w.shape
    if N % TILE or K % TILE:
        raise ValueError("N and K must be multiples of 128")
    blocks = w.reshape(N // TILE, TILE, K // TILE, TILE).transpose(0, 2, 1, 3)
    q, s = _quantize_groups(blocks.reshape(N // TILE, K // TILE, TILE * TILE))
    q = q.reshape(N // TILE, K // TILE, TILE, TILE).transpose(0, 2, 1, 3).reshape(N, K)
    return np.ascontiguousarray(q), s


# --------------------------------------------------------------------------- GEMM


SB_BLOCK_128x128 = 0   # B scales sb[N/128, K/128] (weights)
SB_ROW_1x128 = 1       # B scales sb[N, K/128]     (activations, e.g. a weight-gradient GEMM)


def dequant_rows_1x128(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    """float64 dec(q[m, k]) * s[m, k // 128] (exact: 4-bit by 24-bit significands)."""
    return e4m3_decode(q) * np.repeat(np.asarray(s, np.float64), TILE, axis=1)


def dequant_blocks_128x128(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    """float64 dec(q[n, k]) * s[n // 128, k // 128]."""
    s64 = np.asarray(s, np.float64)
    return e4m3_decode(q) * np.repeat(np.repeat(s64, TILE, axis=0), TILE, axis=1)


def dequant_b(qb: np.ndarray, sb: np.ndarray, sb_kind: int) -> np.ndarray:
    if sb_kind == SB_BLOCK_128x128:
        return dequant_blocks_128x128(qb, sb)
    if sb_kind == SB_ROW_1x128:
        return dequant_rows_1x128(qb, sb)
    raise ValueError("sb_kind must be 0 (128x128 blocks) or 1 (1x128 rows)")


def blockscaled_gemm(qa, sa, qb, sb, sb_kind: int = SB_BLOCK_128x128, rows=None) -> np.ndarray:
    """C = A . B^T over block-scaled E4M3 operands, float64 result.

    A [M, K] codes qa with 1x128 scales sa [M, K/128]; B [N, K] codes qb with scales sb
    (sb_kind 0: 128x128 blocks [N/128, K/128]; 1: 1x128 rows [N, K/128]).
    C[m, n] = sum_k dec(qa[m,k]) sa[m,k/128] * dec(qb[n,k]) sb(n,k), every term exact
    in float64 and the sum accumulated in float64 (a float64 matrix product).
    ``rows`` restricts the result to a subset of output rows (for sampled checks of
    large problems); the arithmetic per entry is unchanged.
    Follows the Italian page, items 1, 5 and 8.
    """
    qa = np.asarray(qa)
    sa = np.asarray(sa)
    if rows is not None:
        qa = qa[rows]
        sa = sa[rows]
    A = dequant_rows_1x128(qa, sa)
    B = dequant_b(np.asarray(qb), np.asarray(sb), sb_kind)
    return A @ B.T


def blockscaled_gemm_e4m3(qa, sa, qb, sb, sb_kind: int = SB_BLOCK_128x128, rows=None):
    """The block-scaled GEMM with its output quantized in 1x128 tiles along N.

    C = blockscaled_gemm(...) (float64) is rounded once to binary32 and quantized by
    quant_act_1x128: returns (codes uint8 [M, N], scales float32 [M, N/128], C32).
    Follows the Arabic page, memory section (activations kept in FP8), with the
    quantization of the Russian page, item 1.
    """
    c32 = blockscaled_gemm(qa, sa, qb, sb, sb_kind, rows=rows).astype(np.float32)
    q, s = quant_act_1x128(c32)
    return q, s, c32


def grouped_gemm(qa, sa, qb, sb, group_offsets, experts=None) -> np.ndarray:
    """Grouped (MoE) block-scaled GEMM, float64 result [Mtot, N].

    qa [Mtot, K] / sa [Mtot, K/128]: the rows of expert e are offsets[e] .. offsets[e+1]-1.
    qb [E, N, K] / sb [E, N/128, K/128]: expert e's weight and its 128x128 block scales.
    Rows of expert e: C = blockscaled_gemm(qa[rows], sa[rows], qb[e], sb[e]).
    ``experts`` restricts the computation to a subset of experts (other rows stay 0).
    Follows the Italian page, item 8 (the MoE GEMM of DeepGEMM).
    """
    qb = np.asarray(qb)
    off = np.asarray(group_offsets, dtype=np.int64)
    E = qb.shape[0]
    C = np.zeros((np.asarray(qa).shape[0], qb.shape[1]), np.float64)
    for e in (range(E) if experts is None else experts):
        lo, hi = int(off[e]), int(off[e + 1])
        if hi > lo:
            C[lo:hi] = blockscaled_gemm(qa[lo:hi], sa[lo:hi], qb[e], sb[e], SB_BLOCK_128x128)
    return C


def relative_error(c_test: np.ndarray, c_ref: np.ndarray) -> float:
    """max |C_test - C_ref| / max |C_ref| (the GEMM parity measure), in float64."""
    c_test = np.asarray(c_test, np.float64)
    c_ref = np.asarray(c_ref, np.float64)
    den = float(np.max(np.abs(c_ref))) if c_ref.size else 0.0
    num = float(np.max(np.abs(c_test - c_ref))) if c_ref.size else 0.0
    if den == 0.0:
        return 0.0 if num == 0.0 else float("inf")
    return num / den
