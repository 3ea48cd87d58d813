"""GPU parity of the dual-output quantizers and of the data-gradient GEMM, through the C
ABI.

- fp8_quant_act_1x128_dual: both outputs must equal the oracle's 1x128 quantization
  along K and along M (stored transposed) bit for bit.
- fp8_quant_w_128x128_dual: q and s must equal the oracle's 128x128 quantization of W,
  and qt and st must equal the oracle's quantization of W^T (which is the transpose).
- dX = dY . W: the GEMM fed with q(dY) and the transposed weight copy must agree with
  the oracle's float64 product of the dequantized operands within the GEMM tolerance:
  max|C_gpu - C_oracle| / max|C_oracle| <= 1e-4 (FP32 out) and <= 8e-3 (BF16 out).
"""
import numpy as np
import pytest
import torch

from fp8_fine_grained_cast_b300 import _lib, inputs, ops
from oracle import fp8_oracle as O
from tests.division_cases import division_sensitive_tiles
from tests.test_gpu_quant import assert_same_quant, bf16_dev, edge_rows, f32

pytestmark = pytest.mark.gpu

TOL = {torch.float32: 1e-4, torch.bfloat16: 8e-3}


def check_act_dual(x: torch.Tensor):
    q, s, qt, st = ops.quant_act_1x128_dual(x)
    ops.sync_status()
    xh = f32(x)
    assert_same_quant(q, s, *O.quant_act_1x128(xh))
    assert_same_quant(qt, st, *O.quant_act_1x128_transposed(xh))


def check_w_dual(w: torch.Tensor):
    q, s, qt, st = ops.quant_w_128x128_dual(w)
    ops.sync_status()
    wh = f32(w)
    q_ref, s_ref = O.quant_w_128x128(wh)
    assert_same_quant(q, s, q_ref, s_ref)
    assert_same_quant(qt, st, np.ascontiguousarray(q_ref.T), np.ascontiguousarray(s_ref.T))
    return q_ref, s_ref


def random_bf16(rng, shape, sigma=1.0, outliers=0.001, scale=50.0):
    x = (rng.standard_normal(shape) * sigma).astype(np.float32)
    x[rng.random(shape) < outliers] *= scale
    return x


@pytest.mark.parametrize("M,K", [(128, 128), (256, 384), (384, 1024), (1280, 256)])
def test_act_dual_small(cuda_device, M, K):
    rng = np.random.default_rng(M + 3 * K)
    check_act_dual(bf16_dev(random_bf16(rng, (M, K)), cuda_device))


def test_act_dual_edge_tiles_both_orientations(cuda_device):
    """Edge-case and division-sensitive tiles laid along rows (1x128 tiles along K) and,
    in a second matrix, along columns (tiles along M)."""
    rows = np.concatenate([edge_rows(), division_sensitive_tiles(4)])    # 16 tiles of 128
    a = np.zeros((256, 1024), np.float32)
    for r in range(256):
        for t in range(8):
            a[r, 128 * t:128 * t + 128] = np.roll(rows[(r + t) % 16], r)
    check_act_dual(bf16_dev(a, cuda_device))
    check_act_dual(bf16_dev(np.ascontiguousarray(a[:, :256].T.copy()), cuda_device))
    b = np.zeros((1024, 256), np.float32)
    for j in range(256):
        b[:, j] = np.concatenate([np.roll(rows[(j + u) % 16], j) for u in range(8)])
    check_act_dual(bf16_dev(b, cuda_device))


def test_act_dual_padded_stride(cuda_device):
    base = inputs.quant_only(cuda_device, rows=512, cols=1152)
    check_act_dual(base[:, :768])


def test_act_dual_quantize_only_config_full(cuda_device):
    check_act_dual(inputs.quant_only(cuda_device))                      # [16384, 7168]


def test_act_dual_dense_activations_full(cuda_device):
    check_act_dual(inputs.dense(cuda_device).x)                          # [4096, 7168]


def test_act_dual_matches_single_calls(cuda_device):
    x = inputs.wgrad(cuda_device).x                                      # [4096, 7168]
    q, s, qt, st = ops.quant_act_1x128_dual(x)
    q1, s1 = ops.quant_act_1x128(x)
    q2, s2 = ops.quant_act_1x128(x, transposed=True)
    ops.sync_status()
    for a, b in ((q, q1), (s, s1), (qt, q2), (st, s2)):
        assert torch.equal(a, b)


@pytest.mark.parametrize("N,K", [(128, 128), (256, 384), (384, 256), (640, 1152)])
def test_w_dual_small(cuda_device, N, K):
    rng = np.random.default_rng(N * 5 + K)
    check_w_dual(bf16_dev(random_bf16(rng, (N, K), 0.02), cuda_device))


def test_w_dual_edge_blocks(cuda_device):
    rows = np.concatenate([edge_rows(), division_sensitive_tiles(4)])
    e = np.zeros((512, 512), np.float32)
    for b in range(16):
        br, bc = divmod(b, 4)
        e[128 * br:128 * br + 128, 128 * bc:128 * bc + 128] = np.stack([np.roll(rows[b], i) for i in range(128)])
    check_w_dual(bf16_dev(e, cuda_device))


def test_w_dual_padded_stride(cuda_device):
    base = inputs.gaussian_bf16((384, 896), 0.02, cuda_device, 9, 6)
    check_w_dual(base[:, :640])


def test_w_dual_dense_config_full(cuda_device):
    check_w_dual(inputs.dense(cuda_device).w)                            # [18432, 7168]


def run_dgrad(dy: torch.Tensor, w: torch.Tensor, out_dtype):
    qdy, sdy = ops.quant_act_1x128(dy)
    _, _, qwt, swt = ops.quant_w_128x128_dual(w)
    dx = ops.blockscaled_gemm(qdy, sdy, qwt, swt, ops.SB_BLOCK_128x128, out_dtype)
    ops.sync_status()
    return qdy, sdy, qwt, swt, dx


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("T,Dout,Din", [(128, 128, 128), (300, 384, 640), (1, 256, 256), (520, 1152, 1024)])
def test_dgrad_small(cuda_device, out_dtype, T, Dout, Din):
    rng = np.random.default_rng(T + Dout + Din)
    dy = bf16_dev(random_bf16(rng, (T, Dout), 1e-3), cuda_device)
    w = bf16_dev(random_bf16(rng, (Dout, Din), 0.02), cuda_device)
    qdy, sdy, qwt, swt, dx = run_dgrad(dy, w, out_dtype)
    rq, rs = O.quant_act_1x128(f32(dy))
    wq, ws = O.quant_w_128x128(f32(w))
    assert np.array_equal(qdy.cpu().numpy(), rq) and np.array_equal(qwt.cpu().numpy(), wq.T)
    ref = O.blockscaled_gemm(rq, rs, np.ascontiguousarray(wq.T), np.ascontiguousarray(ws.T))
    # the same product written as dY . W from the untransposed weight codes
    ref2 = O.dequant_rows_1x128(rq, rs) @ O.dequant_blocks_128x128(wq, ws)
    assert np.allclose(ref, ref2, rtol=0, atol=1e-12 * max(1.0, np.abs(ref2).max()))
    assert O.relative_error(f32(dx), ref) <= TOL[out_dtype]


def test_dgrad_config_full(cuda_device):
    """dX [4096, 7168] = dY [4096, 18432] . W [18432, 7168], BF16 out, in the launch
    configuration the benchmark times; oracle on sampled rows."""
    d = inputs.dgrad(cuda_device)
    qdy, sdy, qwt, swt, dx = run_dgrad(d.dy, d.w, torch.bfloat16)
    rq, rs = O.quant_act_1x128(f32(d.dy))
    wq, ws = O.quant_w_128x128(f32(d.w))
    assert np.array_equal(qdy.cpu().numpy(), rq)
    assert np.array_equal(qwt.cpu().numpy(), wq.T) and np.array_equal(swt.cpu().numpy(), ws.T)
    rows = np.array(sorted(set(np.random.default_rng(2).choice(4096, 192, replace=False).tolist()) | {0, 4095}))
    ref = O.blockscaled_gemm(rq, rs, np.ascontiguousarray(wq.T), np.ascontiguousarray(ws.T), rows=rows)
    assert O.relative_error(f32(dx[torch.from_numpy(rows).to(cuda_device)]), ref) <= 8e-3


def test_dual_rejects_bad_shapes(cuda_device):
    x = torch.zeros((200, 256), dtype=torch.bfloat16, device=cuda_device)
    with pytest.raises(_lib.Fp8fgError) as ei:
        ops.quant_act_1x128_dual(x)
    assert ei.value.code == _lib.FP8FG_ERR_ARG
    w = torch.zeros((256, 200), dtype=torch.bfloat16, device=cuda_device)
    with pytest.raises(_lib.Fp8fgError) as ei:
        ops.quant_w_128x128_dual(w)
    assert ei.value.code == _lib.FP8FG_ERR_ARG
