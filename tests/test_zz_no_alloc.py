"""The stream-K GEMM entry point that allocates nothing (fp8_blockscaled_gemm_sk_static,
a library-owned static workspace): two calls in a row must equal the data-parallel
fp8_blockscaled_gemm and the caller-workspace fp8_blockscaled_gemm_ws bit for bit (the
second call also shows that the first left the release flags cleared). The file name
sorts last so that it also runs after every other test; it passes on its own too."""
import numpy as np
import pytest
import torch

from fp8_fine_grained_cast_b300 import _lib, ops
from oracle import fp8_oracle as O

pytestmark = pytest.mark.gpu


def _dev(a, device):
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def _static(qa, sa, qb, sb, sb_kind, c):
    M, K = qa.shape
    N = qb.shape[0]
    c_dtype = _lib.FP8FG_OUT_BF16 if c.dtype == torch.bfloat16 else _lib.FP8FG_OUT_F32
    _lib.fp8_blockscaled_gemm_sk_static(qa.data_ptr(), sa.data_ptr(), qb.data_ptr(), sb.data_ptr(), sb_kind,
                                        c.data_ptr(), c_dtype, M, N, K, torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("sb_kind,out_dtype", [(O.SB_BLOCK_128x128, torch.bfloat16), (O.SB_ROW_1x128, torch.float32)])
def test_static_workspace_gemm_matches_existing_entry_points(cuda_device, sb_kind, out_dtype):
    # 160 x 2 tiles of 128 x 256 on 148 SMs: a partial last wave, so tiles are cut
    M, N, K = 20480, 512, 1152
    rng = np.random.default_rng(77 + sb_kind)
    xa = torch.from_numpy(rng.standard_normal((M, K)).astype(np.float32)).to(torch.bfloat16).to(cuda_device)
    xb = torch.from_numpy((rng.standard_normal((N, K)) * 0.02).astype(np.float32)).to(torch.bfloat16).to(cuda_device)
    qa, sa = ops.quant_act_1x128(xa)
    qb, sb = ops.quant_w_128x128(xb) if sb_kind == O.SB_BLOCK_128x128 else ops.quant_act_1x128(xb)
    ref = ops.blockscaled_gemm(qa, sa, qb, sb, sb_kind, out_dtype)
    ws = ops.gemm_workspace(cuda_device)
    ref_ws = ops.blockscaled_gemm(qa, sa, qb, sb, sb_kind, out_dtype, workspace=ws)
    outs = []
    for _ in range(2):
        c = torch.full((M, N), 3.0, dtype=out_dtype, device=cuda_device)
        _static(qa, sa, qb, sb, sb_kind, c)
        outs.append(c)
    ops.sync_status()
    assert torch.equal(ref, ref_ws)
    assert torch.equal(outs[0], ref) and torch.equal(outs[1], ref)


def test_static_workspace_gemm_small_problem(cuda_device):
    """Fewer tiles than SMs: the plain schedule, same result."""
    rng = np.random.default_rng(78)
    qa = (0x30 + rng.integers(0, 16, (300, 384))).astype(np.uint8)
    qb = (0x30 + rng.integers(0, 16, (256, 384))).astype(np.uint8)
    sa = np.exp2(rng.integers(-3, 3, (300, 3))).astype(np.float32)
    sb = np.exp2(rng.integers(-3, 3, (2, 3))).astype(np.float32)
    a, b, s1, s2 = _dev(qa, cuda_device), _dev(qb, cuda_device), _dev(sa, cuda_device), _dev(sb, cuda_device)
    ref = ops.blockscaled_gemm(a, s1, b, s2, O.SB_BLOCK_128x128, torch.float32)
    c = torch.empty_like(ref)
    _static(a, s1, b, s2, O.SB_BLOCK_128x128, c)
    ops.sync_status()
    assert torch.equal(c, ref)


def test_static_workspace_after_a_recorded_timeout(cuda_device):
    """A device-side wait that ran out (the self-test kernel) is reported once; the
    static-workspace GEMM then still equals the data-parallel GEMM on two calls in a row."""
    _lib.fp8fg_selftest_wait_timeout(torch.cuda.current_stream().cuda_stream)
    with pytest.raises(_lib.Fp8fgError) as ei:
        ops.sync_status()
    assert ei.value.code == _lib.FP8FG_ERR_TIMEOUT
    M, N, K = 20480, 512, 1152
    rng = np.random.default_rng(79)
    xa = torch.from_numpy(rng.standard_normal((M, K)).astype(np.float32)).to(torch.bfloat16).to(cuda_device)
    xb = torch.from_numpy((rng.standard_normal((N, K)) * 0.02).astype(np.float32)).to(torch.bfloat16).to(cuda_device)
    qa, sa = ops.quant_act_1x128(xa)
    qb, sb = ops.quant_w_128x128(xb)
    ref = ops.blockscaled_gemm(qa, sa, qb, sb, O.SB_BLOCK_128x128, torch.float32)
    for _ in range(2):
        c = torch.full((M, N), 5.0, dtype=torch.float32, device=cuda_device)
        _static(qa, sa, qb, sb, O.SB_BLOCK_128x128, c)
        ops.sync_status()
        assert torch.equal(c, ref)
