"""Host-side argument checks of the tensor-level binding (no GPU needed): the C ABI
receives raw pointers only, so a scale matrix or output of the wrong shape, dtype or
layout must be refused in Python before any launch. The GEMM operand checks run here
on host tensors; the same function guards every GEMM call on the device."""
import pytest
import torch

from fp8_fine_grained_cast_b300 import ops


def operands(M=256, N=384, K=512, sb_kind=ops.SB_BLOCK_128x128):
    qa = torch.zeros((M, K), dtype=torch.uint8)
    sa = torch.ones((M, K // 128), dtype=torch.float32)
    qb = torch.zeros((N, K), dtype=torch.uint8)
    rows = N // 128 if sb_kind == ops.SB_BLOCK_128x128 else N
    sb = torch.ones((rows, K // 128), dtype=torch.float32)
    return qa, sa, qb, sb


@pytest.mark.parametrize("sb_kind", [ops.SB_BLOCK_128x128, ops.SB_ROW_1x128])
def test_valid_operands_pass(sb_kind):
    assert ops._gemm_operands(*operands(sb_kind=sb_kind), sb_kind, cuda=False) == (256, 384, 512)


def test_sb_layout_must_match_sb_kind():
    qa, sa, qb, sb = operands(sb_kind=ops.SB_BLOCK_128x128)
    with pytest.raises(ValueError, match="sb must have shape"):
        ops._gemm_operands(qa, sa, qb, sb, ops.SB_ROW_1x128, cuda=False)
    qa, sa, qb, sb = operands(sb_kind=ops.SB_ROW_1x128)
    with pytest.raises(ValueError, match="sb must have shape"):
        ops._gemm_operands(qa, sa, qb, sb, ops.SB_BLOCK_128x128, cuda=False)


@pytest.mark.parametrize("bad", ["sa_rows", "sa_cols", "sb_cols", "sa_dtype", "sa_strided", "qb_k", "sb_kind"])
def test_mismatched_operands_are_refused(bad):
    qa, sa, qb, sb = operands()
    sb_kind = ops.SB_BLOCK_128x128
    if bad == "sa_rows":
        sa = torch.ones((255, 4), dtype=torch.float32)
    elif bad == "sa_cols":
        sa = torch.ones((256, 3), dtype=torch.float32)
    elif bad == "sb_cols":
        sb = torch.ones((3, 5), dtype=torch.float32)
    elif bad == "sa_dtype":
        sa = sa.double()
    elif bad == "sa_strided":
        sa = torch.ones((4, 256), dtype=torch.float32).t()
    elif bad == "qb_k":
        qb = torch.zeros((384, 384), dtype=torch.uint8)
    elif bad == "sb_kind":
        sb_kind = 7
    with pytest.raises((ValueError, TypeError)):
        ops._gemm_operands(qa, sa, qb, sb, sb_kind, cuda=False)


@pytest.mark.parametrize("bad", ["shape", "dtype", "strided"])
def test_outputs_must_match(bad):
    good = torch.empty((256, 384), dtype=torch.bfloat16)
    ops._exact(good, (256, 384), torch.bfloat16, good.device, "c", cuda=False)
    t = {"shape": torch.empty((256, 383), dtype=torch.bfloat16),
         "dtype": torch.empty((256, 384), dtype=torch.float32),
         "strided": torch.empty((384, 256), dtype=torch.bfloat16).t()}[bad]
    with pytest.raises((ValueError, TypeError)):
        ops._exact(t, (256, 384), torch.bfloat16, good.device, "c", cuda=False)


def test_host_tensors_are_refused_by_the_public_calls():
    qa, sa, qb, sb = operands()
    with pytest.raises(TypeError, match="CUDA tensor"):
        ops.blockscaled_gemm(qa, sa, qb, sb)
