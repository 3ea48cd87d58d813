"""GPU parity of the quantization kernels against the oracle: E4M3 codes and FP32 scales
must match bit for bit, through the C ABI, on the seeded workloads at full size and on
edge cases (all-zero tiles, signed zeros, rounding ties, division-sensitive tiles,
binary32-subnormal scales, huge magnitudes, ragged row counts, padded row strides)."""
import numpy as np
import pytest
import torch

from fp8_fine_grained_cast_b300 import _lib, inputs, ops
from oracle import fp8_oracle as O
from tests.division_cases import division_sensitive_tiles

pytestmark = pytest.mark.gpu


def f32(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy()


def assert_same_quant(q_gpu, s_gpu, q_ref, s_ref):
    qg = q_gpu.cpu().numpy()
    sg = s_gpu.cpu().numpy()
    assert qg.shape == q_ref.shape and sg.shape == s_ref.shape
    bad_s = np.argwhere(sg.view(np.uint32) != s_ref.view(np.uint32))
    assert bad_s.size == 0, f"{len(bad_s)} scales differ, first {bad_s[:5].tolist()}"
    bad_q = np.argwhere(qg != q_ref)
    assert bad_q.size == 0, (f"{len(bad_q)} codes differ, first at {bad_q[:5].tolist()}: "
                             f"gpu {[hex(qg[tuple(i)]) for i in bad_q[:5]]} "
                             f"ref {[hex(q_ref[tuple(i)]) for i in bad_q[:5]]}")


def bf16_dev(a: np.ndarray, dev) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(torch.bfloat16).to(dev)


def edge_rows():
    rng = np.random.default_rng(7)
    t = [rng.standard_normal(128)]
    r = rng.standard_normal(128); r[17] = 60.0; t.append(r)
    t.append(np.zeros(128))
    r = np.zeros(128); r[::2] = -0.0; r[5] = 3.0; r[6] = -0.0; t.append(r)
    r = rng.standard_normal(128) * 1e-3; r[0] = 100.0; t.append(r)
    t.append(-np.abs(rng.standard_normal(128)))
    t.append(rng.standard_normal(128) * 1e30)
    t.append(rng.standard_normal(128) * 1e-36)       # binary32-subnormal scale
    t.append(rng.standard_normal(128) * 1e-25)       # scale ~1e-28: plain-division range
    t.append(np.full(128, 2.5))
    t.append(np.linspace(-7.0, 7.0, 128))
    r = rng.standard_normal(128); r[3] = -1e-40; r[4] = 1e-40; t.append(r)   # bf16 subnormals
    return np.array(t, dtype=np.float32)


def test_act_rows_tiny(cuda_device):
    x = inputs.tiny(cuda_device).x
    q, s = ops.quant_act_1x128(x)
    q_ref, s_ref = O.quant_act_1x128(f32(x))
    assert_same_quant(q, s, q_ref, s_ref)


def test_act_rows_edge_cases_and_ragged_rows(cuda_device):
    rows = np.concatenate([edge_rows(), division_sensitive_tiles(24)])   # 36 tiles
    x = rows.reshape(9, 4 * 128)                                         # M = 9: ragged
    xd = bf16_dev(x, cuda_device)
    q, s = ops.quant_act_1x128(xd)
    q_ref, s_ref = O.quant_act_1x128(f32(xd))
    assert_same_quant(q, s, q_ref, s_ref)


@pytest.mark.parametrize("M", [1, 3, 17, 255])
def test_act_rows_small_ragged(cuda_device, M):
    x = inputs.activation_bf16(M, 384, 100.0, 0.01, 0, cuda_device, 9, M)
    q, s = ops.quant_act_1x128(x)
    assert_same_quant(q, s, *O.quant_act_1x128(f32(x)))


def test_act_rows_padded_stride(cuda_device):
    base = inputs.activation_bf16(200, 1024, 100.0, 0.001, 64, cuda_device, 9, 99)
    x = base[:, :768]                                                    # ldx = 1024 > K = 768
    q, s = ops.quant_act_1x128(x)
    assert_same_quant(q, s, *O.quant_act_1x128(f32(x)))


def test_act_rows_quantize_only_config_full(cuda_device):
    x = inputs.quant_only(cuda_device)                                   # [16384, 7168]
    q, s = ops.quant_act_1x128(x)
    xh = f32(x)
    q_ref, s_ref = O.quant_act_1x128(xh)
    assert_same_quant(q, s, q_ref, s_ref)
    assert int((s_ref == 0).sum()) == 16                                 # one zero tile per 1024 rows


def test_all_bf16_quotients(cuda_device):
    """Every finite bf16 x with |x| <= amax for 48 amax values spread over the binades:
    each tile holds amax first and 127 further values, covering the quotient x / s."""
    bits = (np.arange(0x0001, 0x7F80, dtype=np.uint32) << 16).view(np.float32)
    rng = np.random.default_rng(5)
    amaxes = np.sort(rng.choice(bits[(bits > 1e-30) & (bits < 1e30)], 48, replace=False))
    tiles = []
    for a in amaxes:
        xs = bits[bits <= a]
        xs = np.concatenate([xs, -xs])
        pad = (-len(xs)) % 127
        xs = np.concatenate([xs, np.zeros(pad, np.float32)]).reshape(-1, 127)
        tiles.append(np.concatenate([np.full((xs.shape[0], 1), a, np.float32), xs], axis=1))
    x = np.concatenate(tiles)
    x = x[: (x.shape[0] // 4) * 4].reshape(-1, 512)
    xd = bf16_dev(x, cuda_device)
    q, s = ops.quant_act_1x128(xd)
    assert_same_quant(q, s, *O.quant_act_1x128(f32(xd)))


def test_weight_blocks_tiny_and_edges(cuda_device):
    w = inputs.tiny(cuda_device).w
    q, s = ops.quant_w_128x128(w)
    assert_same_quant(q, s, *O.quant_w_128x128(f32(w)))
    # a 4 x 4 grid of 128x128 blocks, each built from one edge-case or division-sensitive
    # row by rolling it down the block, so that each block keeps that row's amax
    rows = np.concatenate([edge_rows(), division_sensitive_tiles(4)])   # 16 rows
    e = np.zeros((512, 512), np.float32)
    for b in range(16):
        br, bc = divmod(b, 4)
        blk = np.stack([np.roll(rows[b], i) for i in range(128)])
        e[128 * br:128 * br + 128, 128 * bc:128 * bc + 128] = blk
    ed = bf16_dev(e, cuda_device)
    q, s = ops.quant_w_128x128(ed)
    assert_same_quant(q, s, *O.quant_w_128x128(f32(ed)))


def test_weight_blocks_dense_config_full(cuda_device):
    w = inputs.dense(cuda_device).w                                      # [18432, 7168]
    q, s = ops.quant_w_128x128(w)
    assert_same_quant(q, s, *O.quant_w_128x128(f32(w)))


def test_weight_blocks_padded_stride(cuda_device):
    base = inputs.gaussian_bf16((256, 640), 0.02, cuda_device, 9, 5)
    w = base[:, :512]
    q, s = ops.quant_w_128x128(w)
    assert_same_quant(q, s, *O.quant_w_128x128(f32(w)))


def test_transposed_wgrad_config_full(cuda_device):
    wg = inputs.wgrad(cuda_device)
    for t in (wg.dy, wg.x):                                              # [4096, 2048], [4096, 7168]
        q, s = ops.quant_act_1x128(t, transposed=True)
        assert_same_quant(q, s, *O.quant_act_1x128_transposed(f32(t)))


@pytest.mark.parametrize("K", [8, 136, 264])
def test_transposed_ragged_columns_and_edges(cuda_device, K):
    rows = np.concatenate([edge_rows(), division_sensitive_tiles(4)])    # 16 tiles of 128
    x = np.zeros((256, K), np.float32)
    for j in range(K):
        x[:, j] = rows[(2 * j) % 16].tolist() + rows[(2 * j + 1) % 16].tolist()
    xd = bf16_dev(x, cuda_device)
    q, s = ops.quant_act_1x128(xd, transposed=True)
    assert_same_quant(q, s, *O.quant_act_1x128_transposed(f32(xd)))


def test_deterministic_and_empty(cuda_device):
    x = inputs.quant_only(cuda_device, rows=1024, cols=1024)
    a = ops.quant_act_1x128(x)
    b = ops.quant_act_1x128(x)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    e = torch.empty((0, 256), dtype=torch.bfloat16, device=cuda_device)
    q, s = ops.quant_act_1x128(e)
    assert q.shape == (0, 256) and s.shape == (0, 2)


def test_gpu_call_rejects_bad_shape(cuda_device):
    x = torch.zeros((4, 200), dtype=torch.bfloat16, device=cuda_device)
    with pytest.raises(_lib.Fp8fgError) as ei:
        ops.quant_act_1x128(x)
    assert ei.value.code == _lib.FP8FG_ERR_ARG


def test_transposed_many_blocks_and_ragged_columns(cuda_device):
    """The persistent transposed quantizer with about two, and more than two, blocks per
    CTA, and with a ragged last column block over many row blocks, against the oracle."""
    sm = torch.cuda.get_device_properties(cuda_device).multi_processor_count
    rng = np.random.default_rng(33)
    for mb, K in ((4 * sm // 8, 1024), (4 * sm // 8 + 1, 1024), (300, 264)):
        x = rng.standard_normal((128 * mb, K)).astype(np.float32)
        x[rng.random(x.shape) < 0.001] *= 40.0
        x[128:256, 3] = 0.0                                               # an all-zero tile (tokens 128-255)
        x[5:133, 5] = 0.0                                                 # zeros straddling two tiles
        xd = bf16_dev(x, cuda_device)
        q, s = ops.quant_act_1x128(xd, transposed=True)
        assert_same_quant(q, s, *O.quant_act_1x128_transposed(f32(xd)))


def test_transposed_pair_wgrad_operands(cuda_device):
    """Both weight-gradient operands (dY [4096, 2048], X [4096, 7168]) in one launch:
    bit-identical to two single calls, which the oracle pins at full size above; and a
    ragged second tensor (K = 264, padded row stride) against the oracle directly."""
    w = inputs.wgrad(cuda_device)
    q0, s0, q1, s1 = ops.quant_act_1x128_transposed_pair(w.dy, w.x)
    r0 = ops.quant_act_1x128(w.dy, transposed=True)
    r1 = ops.quant_act_1x128(w.x, transposed=True)
    ops.sync_status()
    assert torch.equal(q0, r0[0]) and torch.equal(s0.view(torch.int32), r0[1].view(torch.int32))
    assert torch.equal(q1, r1[0]) and torch.equal(s1.view(torch.int32), r1[1].view(torch.int32))
    rng = np.random.default_rng(41)
    a = rng.standard_normal((512, 384)).astype(np.float32)
    b = rng.standard_normal((512, 272)).astype(np.float32) * 3.0
    b[rng.random(b.shape) < 0.002] *= 60.0
    b[128:256, 7] = 0.0                                                    # an all-zero tile
    xa = bf16_dev(a, cuda_device)
    xb = bf16_dev(b, cuda_device)[:, :264]                                 # row stride 272
    q0, s0, q1, s1 = ops.quant_act_1x128_transposed_pair(xa, xb)
    ops.sync_status()
    assert_same_quant(q0, s0, *O.quant_act_1x128_transposed(f32(xa)))
    assert_same_quant(q1, s1, *O.quant_act_1x128_transposed(f32(xb)))


def test_transposed_pair_with_an_empty_tensor(cuda_device):
    x = bf16_dev(np.random.default_rng(42).standard_normal((256, 128)).astype(np.float32), cuda_device)
    e = torch.empty((256, 0), dtype=torch.bfloat16, device=cuda_device)
    q0, s0, q1, s1 = ops.quant_act_1x128_transposed_pair(e, x)
    ops.sync_status()
    assert q0.shape == (0, 256)
    assert_same_quant(q1, s1, *O.quant_act_1x128_transposed(f32(x)))
