"""GPU parity of the block-scaled FP8 GEMM against the oracle, through the C ABI.

Tolerance (fixed by the method's acceptance bar): max|C_gpu - C_oracle| / max|C_oracle|
<= 1e-4 for FP32 output and <= 8e-3 for BF16 output, C_oracle being the float64 sum of
the dequantized operands. Operands come from the oracle's quantizer (or from the GPU
quantizer after checking it is bit-identical), so both sides multiply the same codes.
An exact-sum case (one 128-deep chunk, codes in [1, 2), power-of-two scales) must
match exactly: every partial sum is representable in FP32.
"""
import numpy as np
import pytest
import torch

from fp8_fine_grained_cast_b300 import inputs, ops
from oracle import fp8_oracle as O

pytestmark = pytest.mark.gpu

TOL = {torch.float32: 1e-4, torch.bfloat16: 8e-3}


def f32(t):
    return t.detach().float().cpu().numpy()


def dev(a, device, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    return t.to(device) if dtype is None else t.to(dtype).to(device)


def random_quantized(rng, M, N, K, sb_kind):
    """Operands produced by the oracle's quantizers from bf16-valued random data."""
    xa = torch.from_numpy(rng.standard_normal((M, K)).astype(np.float32)).to(torch.bfloat16).float().numpy()
    xa[rng.random((M, K)) < 0.001] *= 50.0
    qa, sa = O.quant_act_1x128(xa)
    xb = torch.from_numpy((rng.standard_normal((N, K)) * 0.02).astype(np.float32)).to(torch.bfloat16).float().numpy()
    if sb_kind == O.SB_BLOCK_128x128:
        qb, sb = O.quant_w_128x128(xb)
    else:
        qb, sb = O.quant_act_1x128(xb)
    return qa, sa, qb, sb


def run_gemm(qa, sa, qb, sb, sb_kind, out_dtype, device):
    c = ops.blockscaled_gemm(dev(qa, device), dev(sa, device), dev(qb, device), dev(sb, device), sb_kind, out_dtype)
    ops.sync_status()
    return c


@pytest.mark.parametrize("sb_kind", [O.SB_BLOCK_128x128, O.SB_ROW_1x128])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("M,N,K", [(128, 128, 128), (300, 384, 640), (1, 256, 256), (520, 1024, 1152),
                                   (200, 768, 384)])
def test_gemm_matches_oracle(cuda_device, sb_kind, out_dtype, M, N, K):
    rng = np.random.default_rng(M * 7 + N * 3 + K)
    qa, sa, qb, sb = random_quantized(rng, M, N, K, sb_kind)
    c = run_gemm(qa, sa, qb, sb, sb_kind, out_dtype, cuda_device)
    ref = O.blockscaled_gemm(qa, sa, qb, sb, sb_kind)
    err = O.relative_error(f32(c), ref)
    assert err <= TOL[out_dtype], err


def test_gemm_exact_single_chunk(cuda_device):
    """K = 128, codes in [1, 2) with random signs, power-of-two scales: products carry
    at most 8 significant bits and the sum of 128 of them at most 15, so FP32 holds
    every partial sum exactly and the result must equal the oracle bit for bit."""
    rng = np.random.default_rng(3)
    M, N, K = 256, 512, 128
    qa = (0x38 + rng.integers(0, 8, (M, K))).astype(np.uint8) | (rng.integers(0, 2, (M, K)) << 7).astype(np.uint8)
    qb = (0x38 + rng.integers(0, 8, (N, K))).astype(np.uint8) | (rng.integers(0, 2, (N, K)) << 7).astype(np.uint8)
    sa = np.exp2(rng.integers(-6, 6, (M, 1))).astype(np.float32)
    for sb_kind, sb in ((O.SB_BLOCK_128x128, np.exp2(rng.integers(-6, 6, (N // 128, 1))).astype(np.float32)),
                        (O.SB_ROW_1x128, np.exp2(rng.integers(-6, 6, (N, 1))).astype(np.float32))):
        c = run_gemm(qa, sa, qb, sb, sb_kind, torch.float32, cuda_device)
        ref = O.blockscaled_gemm(qa, sa, qb, sb, sb_kind)
        assert np.array_equal(f32(c), ref.astype(np.float32)), O.relative_error(f32(c), ref)


def test_gemm_exact_chunk_promotion(cuda_device):
    """Four chunks, codes in {1, 2, 4}, scales in {1/2, 1, 2}: a chunk sum is an
    integer below 2^11, a promoted term a multiple of 1/4 below 2^13 and the total below
    2^15, so FP32 is exact throughout and per-chunk scaling must reproduce the oracle
    exactly; a mis-indexed scale would not."""
    rng = np.random.default_rng(4)
    M, N, K = 128, 256, 512
    qa = (0x38 + 8 * rng.integers(0, 3, (M, K))).astype(np.uint8)      # 1, 2, 4
    qb = (0x38 + 8 * rng.integers(0, 3, (N, K))).astype(np.uint8)
    sa = np.exp2(rng.integers(-1, 2, (M, K // 128))).astype(np.float32)
    sb = np.exp2(rng.integers(-1, 2, (N // 128, K // 128))).astype(np.float32)
    c = run_gemm(qa, sa, qb, sb, O.SB_BLOCK_128x128, torch.float32, cuda_device)
    ref = O.blockscaled_gemm(qa, sa, qb, sb, O.SB_BLOCK_128x128)
    assert np.array_equal(f32(c), ref.astype(np.float32))


def test_tiny_config_end_to_end(cuda_device):
    t = inputs.tiny(cuda_device)
    qx, sx = ops.quant_act_1x128(t.x)
    qw, sw = ops.quant_w_128x128(t.w)
    c = ops.blockscaled_gemm(qx, sx, qw, sw, ops.SB_BLOCK_128x128, torch.float32)
    ops.sync_status()
    rq, rs = O.quant_act_1x128(f32(t.x))
    wq, ws = O.quant_w_128x128(f32(t.w))
    assert np.array_equal(qx.cpu().numpy(), rq) and np.array_equal(sx.cpu().numpy(), rs)
    assert np.array_equal(qw.cpu().numpy(), wq) and np.array_equal(sw.cpu().numpy(), ws)
    ref = O.blockscaled_gemm(rq, rs, wq, ws)
    assert O.relative_error(f32(c), ref) <= 1e-4


def _sample_rows(M, rng, must=()):
    rows = set(rng.choice(M, size=min(M, 192), replace=False).tolist()) | set(must) | {0, M - 1}
    return np.array(sorted(rows))


def test_dense_projection_config_full(cuda_device):
    """X [4096, 7168] 1x128, W [18432, 7168] 128x128, C [4096, 18432] BF16, in the same
    launch configuration the benchmark times; oracle on sampled rows, including every
    row holding an all-zero tile."""
    d = inputs.dense(cuda_device)
    qx, sx = ops.quant_act_1x128(d.x)
    qw, sw = ops.quant_w_128x128(d.w)
    c = ops.blockscaled_gemm(qx, sx, qw, sw, ops.SB_BLOCK_128x128, torch.bfloat16)
    ops.sync_status()
    xh = f32(d.x)
    rq, rs = O.quant_act_1x128(xh)
    wq, ws = O.quant_w_128x128(f32(d.w))
    assert np.array_equal(qx.cpu().numpy(), rq) and np.array_equal(sw.cpu().numpy(), ws)
    assert np.array_equal(qw.cpu().numpy(), wq)
    zero_rows = np.nonzero((rs == 0).any(axis=1))[0]
    rows = _sample_rows(4096, np.random.default_rng(0), zero_rows)
    ref = O.blockscaled_gemm(rq, rs, wq, ws, rows=rows)
    assert O.relative_error(f32(c[torch.from_numpy(rows).to(cuda_device)]), ref) <= 8e-3


def test_wgrad_config_full(cuda_device):
    """dW [2048, 7168] = dY^T X, both quantized in 1x128 tiles along tokens (transposed),
    FP32 out; oracle on sampled rows."""
    w = inputs.wgrad(cuda_device)
    qdy, sdy = ops.quant_act_1x128(w.dy, transposed=True)      # [2048, 4096]
    qx, sx = ops.quant_act_1x128(w.x, transposed=True)         # [7168, 4096]
    c = ops.blockscaled_gemm(qdy, sdy, qx, sx, ops.SB_ROW_1x128, torch.float32)
    ops.sync_status()
    rdq, rds = O.quant_act_1x128_transposed(f32(w.dy))
    rxq, rxs = O.quant_act_1x128_transposed(f32(w.x))
    assert np.array_equal(qdy.cpu().numpy(), rdq) and np.array_equal(qx.cpu().numpy(), rxq)
    rows = _sample_rows(2048, np.random.default_rng(1))
    ref = O.blockscaled_gemm(rdq, rds, rxq, rxs, O.SB_ROW_1x128, rows=rows)
    assert O.relative_error(f32(c[torch.from_numpy(rows).to(cuda_device)]), ref) <= 1e-4


def test_gemm_k_zero_and_empty(cuda_device):
    qa = torch.empty((4, 0), dtype=torch.uint8, device=cuda_device)
    sa = torch.empty((4, 0), dtype=torch.float32, device=cuda_device)
    qb = torch.empty((128, 0), dtype=torch.uint8, device=cuda_device)
    sb = torch.empty((1, 0), dtype=torch.float32, device=cuda_device)
    c = torch.full((4, 128), 7.0, dtype=torch.float32, device=cuda_device)
    ops.blockscaled_gemm(qa, sa, qb, sb, ops.SB_BLOCK_128x128, torch.float32, c=c)
    assert torch.count_nonzero(c).item() == 0
    e = ops.blockscaled_gemm(torch.empty((0, 128), dtype=torch.uint8, device=cuda_device),
                             torch.empty((0, 1), dtype=torch.float32, device=cuda_device),
                             torch.zeros((128, 128), dtype=torch.uint8, device=cuda_device),
                             torch.ones((1, 1), dtype=torch.float32, device=cuda_device))
    assert e.shape == (0, 128)


def test_gemm_deterministic(cuda_device):
    rng = np.random.default_rng(9)
    qa, sa, qb, sb = random_quantized(rng, 384, 512, 1024, O.SB_BLOCK_128x128)
    a = run_gemm(qa, sa, qb, sb, O.SB_BLOCK_128x128, torch.float32, cuda_device)
    b = run_gemm(qa, sa, qb, sb, O.SB_BLOCK_128x128, torch.float32, cuda_device)
    assert torch.equal(a, b)
