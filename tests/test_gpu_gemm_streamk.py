"""GPU checks of the stream-K schedule (fp8_blockscaled_gemm_ws): its result must be
bit-identical to the data-parallel fp8_blockscaled_gemm (the chunk order of every element
is the same), on shapes whose tiles leave a partial last wave (cut tiles, several chunk
groups per cut, one-chunk groups when K / 128 is not a multiple of the group), on the
full dgrad and wgrad workloads, over repeated calls on one workspace (the flags are left
cleared), over dozens of launches queued back to back on one workspace, and within the
oracle tolerance; a too small workspace is refused."""
import numpy as np
import pytest
import torch

from fp8_fine_grained_cast_b300 import _lib, inputs, ops
from oracle import fp8_oracle as O
from tests.test_gpu_gemm import dev, f32, random_quantized

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ws(cuda_device):
    return ops.gemm_workspace(cuda_device)


def both(qa, sa, qb, sb, sb_kind, out_dtype, ws):
    c_dp = ops.blockscaled_gemm(qa, sa, qb, sb, sb_kind, out_dtype)
    c_sk = ops.blockscaled_gemm(qa, sa, qb, sb, sb_kind, out_dtype, workspace=ws)
    ops.sync_status()
    return c_dp, c_sk


@pytest.mark.parametrize("sb_kind", [O.SB_BLOCK_128x128, O.SB_ROW_1x128])
@pytest.mark.parametrize("M,N,K", [(20480, 256, 512), (2000, 7168, 384), (19200, 512, 1152)])
def test_streamk_bit_identical_and_oracle(cuda_device, ws, sb_kind, M, N, K):
    rng = np.random.default_rng(M + N + K + sb_kind)
    qa, sa, qb, sb = random_quantized(rng, M, N, K, sb_kind)
    args = (dev(qa, cuda_device), dev(sa, cuda_device), dev(qb, cuda_device), dev(sb, cuda_device))
    c_dp, c_sk = both(*args, sb_kind, torch.float32, ws)
    assert torch.equal(c_dp, c_sk)
    rows = np.array(sorted(set(rng.choice(M, 160, replace=False).tolist()) | {0, M - 1}))
    ref = O.blockscaled_gemm(qa, sa, qb, sb, sb_kind, rows=rows)
    assert O.relative_error(f32(c_sk[torch.from_numpy(rows).to(cuda_device)]), ref) <= 1e-4
    sm = torch.cuda.get_device_properties(cuda_device).multi_processor_count
    flags = ws[sm * 128 * 256 * 4: sm * 128 * 256 * 4 + 4 * sm]
    assert int(flags.count_nonzero()) == 0                      # every release flag cleared again
    c_again = ops.blockscaled_gemm(*args, sb_kind, torch.float32, workspace=ws)
    ops.sync_status()
    assert torch.equal(c_again, c_sk)


def test_streamk_dgrad_and_wgrad_full(cuda_device, ws):
    g = inputs.dgrad(cuda_device)
    qdy, sdy = ops.quant_act_1x128(g.dy)
    _, _, qwt, swt = ops.quant_w_128x128_dual(g.w)
    del g
    c_dp, c_sk = both(qdy, sdy, qwt, swt, ops.SB_BLOCK_128x128, torch.bfloat16, ws)
    assert torch.equal(c_dp, c_sk)
    del qdy, sdy, qwt, swt, c_dp, c_sk
    w = inputs.wgrad(cuda_device)
    a, sa = ops.quant_act_1x128(w.dy, transposed=True)
    b, sb = ops.quant_act_1x128(w.x, transposed=True)
    c_dp, c_sk = both(a, sa, b, sb, ops.SB_ROW_1x128, torch.float32, ws)
    assert torch.equal(c_dp, c_sk)


def test_streamk_dense_full(cuda_device, ws):
    d = inputs.dense(cuda_device)
    qx, sx = ops.quant_act_1x128(d.x)
    qw, sw = ops.quant_w_128x128(d.w)
    del d
    c_dp, c_sk = both(qx, sx, qw, sw, ops.SB_BLOCK_128x128, torch.bfloat16, ws)
    assert torch.equal(c_dp, c_sk)


def test_streamk_refuses_small_workspace(cuda_device):
    small = torch.zeros(1024, dtype=torch.uint8, device=cuda_device)
    qa = torch.zeros((128, 128), dtype=torch.uint8, device=cuda_device)
    s = torch.ones((128, 1), dtype=torch.float32, device=cuda_device)
    with pytest.raises(_lib.Fp8fgError) as ei:
        ops.blockscaled_gemm(qa, s, qa, s[:1], ops.SB_BLOCK_128x128, torch.float32, workspace=small)
    assert ei.value.code == _lib.FP8FG_ERR_ARG


@pytest.mark.parametrize("stale", [1, -1])
def test_streamk_ignores_flags_left_by_an_earlier_launch(cuda_device, stale):
    """A launch whose tail gave up (a bounded wait that ran out) leaves its release flag
    set. Planting such flags on the host (the value 1, which an earlier launch of this
    process used as its epoch, and -1) must not change the result: a tail accepts only
    its own launch's epoch."""
    rng = np.random.default_rng(404)
    M, N, K = 20480, 256, 512
    qa, sa, qb, sb = random_quantized(rng, M, N, K, O.SB_BLOCK_128x128)
    args = (dev(qa, cuda_device), dev(sa, cuda_device), dev(qb, cuda_device), dev(sb, cuda_device))
    ws = ops.gemm_workspace(cuda_device)
    c_dp = ops.blockscaled_gemm(*args, O.SB_BLOCK_128x128, torch.float32)
    for _ in range(2):                          # this process's epochs are past 1 from here on
        ops.blockscaled_gemm(*args, O.SB_BLOCK_128x128, torch.float32, workspace=ws)
    ops.sync_status()
    sm = torch.cuda.get_device_properties(cuda_device).multi_processor_count
    flags = ws[sm * 128 * 256 * 4: sm * 128 * 256 * 4 + 4 * sm].view(torch.int32)
    ws[: sm * 128 * 256 * 4].view(torch.float32).fill_(1.0e30)    # garbage partial sums
    flags.fill_(stale)
    c_sk = ops.blockscaled_gemm(*args, O.SB_BLOCK_128x128, torch.float32, workspace=ws)
    ops.sync_status()
    assert torch.equal(c_sk, c_dp)


# Shapes whose 128 x 256 tiles overfill whole waves of 148 CTAs by varying amounts, with
# chunk counts K / 128 that are odd (one-chunk loader groups), even but not a multiple of
# the loader group, or small (a head and a tail in the same tile).
SWEEP = [(19328, 512, 640), (4096, 1536, 896), (2000, 4864, 256), (640, 7936, 1024), (300, 36864, 384),
         (38000, 256, 128)]


@pytest.mark.parametrize("sb_kind", [O.SB_BLOCK_128x128, O.SB_ROW_1x128])
@pytest.mark.parametrize("M,N,K", SWEEP)
def test_streamk_shape_sweep_bit_identical(cuda_device, ws, sb_kind, M, N, K):
    rng = np.random.default_rng(M * 3 + N + K + sb_kind)
    qa, sa, qb, sb = random_quantized(rng, M, N, K, sb_kind)
    args = (dev(qa, cuda_device), dev(sa, cuda_device), dev(qb, cuda_device), dev(sb, cuda_device))
    out_dtype = torch.bfloat16 if (M + K) % 2 else torch.float32
    c_dp, c_sk = both(*args, sb_kind, out_dtype, ws)
    assert torch.equal(c_dp, c_sk)
    rows = np.array(sorted(set(rng.choice(M, 48, replace=False).tolist()) | {0, M - 1}))
    ref = O.blockscaled_gemm(qa, sa, qb, sb, sb_kind, rows=rows)
    tol = 1e-4 if out_dtype == torch.float32 else 8e-3
    assert O.relative_error(f32(c_sk[torch.from_numpy(rows).to(cuda_device)]), ref) <= tol


@pytest.mark.parametrize("M,N,K,sb_kind", [(2000, 4864, 256, O.SB_ROW_1x128), (2048, 7168, 4096, O.SB_ROW_1x128),
                                           (4096, 1536, 896, O.SB_BLOCK_128x128)])
def test_streamk_back_to_back_launches_stay_bit_identical(cuda_device, ws, M, N, K, sb_kind):
    # Many launches on one workspace with no host synchronisation in between: every cut
    # tile's partial sums must be visible to the CTA that finishes the tile in every
    # launch (one thread per CTA fences before setting the release flag).
    rng = np.random.default_rng(M + 7 * N + K)
    qa, sa, qb, sb = random_quantized(rng, M, N, K, sb_kind)
    args = (dev(qa, cuda_device), dev(sa, cuda_device), dev(qb, cuda_device), dev(sb, cuda_device))
    c_dp = ops.blockscaled_gemm(*args, sb_kind, torch.float32)
    outs = [torch.empty_like(c_dp) for _ in range(24)]
    for rep in range(2):
        for c in outs:
            ops.blockscaled_gemm(*args, sb_kind, torch.float32, c=c, workspace=ws)
        ops.sync_status()
        bad = [i for i, c in enumerate(outs) if not torch.equal(c, c_dp)]
        assert not bad, f"launches {bad} of repetition {rep} differ from the data-parallel result"
