"""Maximum-size edge cases: tensors with more than 2^31 elements (byte offsets beyond 4 GB
in the codes and beyond 2^32 in the bf16 inputs), through the C ABI, checked against the
oracle on sampled rows, blocks and columns at the far end of the tensors."""
import numpy as np
import pytest
import torch

from fp8_fine_grained_cast_b300 import ops
from oracle import fp8_oracle as O
from tests.test_gpu_quant import f32

pytestmark = pytest.mark.gpu


def big_bf16(rows, cols, device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    x = torch.randn((rows, cols), generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)
    return x


def test_row_and_transposed_quantizers_beyond_2_31_elements(cuda_device):
    M, K = 4096 * 9, 65536                       # 2.42e9 elements, 4.8 GB of bf16
    x = big_bf16(M, K, cuda_device, 1)
    q, s = ops.quant_act_1x128(x)
    torch.cuda.synchronize()
    for r in (0, 12345, M - 129, M - 1):
        qr, sr = O.quant_act_1x128(f32(x[r:r + 1]))
        assert np.array_equal(q[r].cpu().numpy(), qr[0]) and np.array_equal(s[r].cpu().numpy(), sr[0])
    del q, s
    qt, st = ops.quant_act_1x128(x, transposed=True)                    # [K][M] codes: 2.4 GB
    torch.cuda.synchronize()
    for c in (0, 777, K - 8, K - 1):
        qc, sc = O.quant_act_1x128_transposed(f32(x[:, c:c + 1]))
        assert np.array_equal(qt[c].cpu().numpy(), qc[0]) and np.array_equal(st[c].cpu().numpy(), sc[0])


def test_weight_quantizer_beyond_2_31_elements(cuda_device):
    N, K = 36864, 65536                          # 2.42e9 elements
    w = big_bf16(N, K, cuda_device, 2)
    q, s = ops.quant_w_128x128(w)
    torch.cuda.synchronize()
    for br, bc in ((0, 0), (N // 128 - 1, K // 128 - 1), (200, 300)):
        blk = f32(w[128 * br:128 * br + 128, 128 * bc:128 * bc + 128])
        qb, sb = O.quant_w_128x128(blk)
        assert np.array_equal(q[128 * br:128 * br + 128, 128 * bc:128 * bc + 128].cpu().numpy(), qb)
        assert s[br, bc].item() == sb[0, 0]


def test_gemm_output_beyond_2_31_elements(cuda_device):
    M, N, K = 65536, 40960, 256                  # C has 2.7e9 elements (5.4 GB of bf16)
    rng = np.random.default_rng(9)
    qa = torch.from_numpy((0x30 + rng.integers(0, 24, (M, K))).astype(np.uint8)).to(cuda_device)
    qb = torch.from_numpy((0x30 + rng.integers(0, 24, (N, K))).astype(np.uint8)).to(cuda_device)
    sa = torch.from_numpy(np.exp2(rng.integers(-3, 3, (M, K // 128))).astype(np.float32)).to(cuda_device)
    sb = torch.from_numpy(np.exp2(rng.integers(-3, 3, (N // 128, K // 128))).astype(np.float32)).to(cuda_device)
    c = ops.blockscaled_gemm(qa, sa, qb, sb, ops.SB_BLOCK_128x128, torch.bfloat16)
    ops.sync_status()
    rows = np.array([0, 1, 40000, M - 2, M - 1])
    ref = O.blockscaled_gemm(qa.cpu().numpy(), sa.cpu().numpy(), qb.cpu().numpy(), sb.cpu().numpy(), rows=rows)
    got = c[torch.from_numpy(rows).to(cuda_device)].float().cpu().numpy()
    assert O.relative_error(got, ref) <= 8e-3
