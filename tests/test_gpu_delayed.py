"""GPU parity of delayed (history-based) scaling against the oracle, bit for bit: codes,
tile scales and the history state after each call of a sequence whose magnitude grows
(so that the delayed scale lags and values saturate), at small and full size."""
import numpy as np
import pytest
import torch

from fp8_fine_grained_cast_b300 import _lib, inputs, ops
from oracle import fp8_oracle as O
from tests.test_gpu_quant import bf16_dev, f32

pytestmark = pytest.mark.gpu


def run_sequence(xs, H, device, hist0=None):
    hist = ops.new_amax_history(H, device)
    ref_hist = np.zeros(H, np.float32)
    if hist0 is not None:
        hist[:H] = torch.from_numpy(hist0).to(device)
        ref_hist = hist0.copy()
    for x in xs:
        q, s = ops.quant_act_delayed(x, hist)
        ops.sync_status()
        q_ref, s_ref, ref_hist = O.quant_act_delayed(f32(x), ref_hist)
        assert np.array_equal(q.cpu().numpy(), q_ref), np.argwhere(q.cpu().numpy() != q_ref)[:5]
        assert np.array_equal(s.cpu().numpy().view(np.uint32), s_ref.view(np.uint32))
        h = hist.cpu().numpy()
        assert np.array_equal(h[:H].view(np.uint32), ref_hist.view(np.uint32)), (h, ref_hist)
        assert h[H] == 0.0 and not np.signbit(h[H])


@pytest.mark.parametrize("H", [1, 4, 1024])
def test_delayed_growing_sequence(cuda_device, H):
    rng = np.random.default_rng(50 + H)
    xs = []
    for i in range(5):
        a = rng.standard_normal((384, 512)).astype(np.float32) * (1.6 ** i)
        a[rng.random(a.shape) < 0.001] *= 30.0
        a[7, :128] = 0.0
        a[8, 3] = -0.0
        xs.append(bf16_dev(a, cuda_device))
    run_sequence(xs, H, cuda_device)


def test_delayed_ragged_rows_padded_stride_and_extremes(cuda_device):
    rng = np.random.default_rng(51)
    base = bf16_dev(rng.standard_normal((300, 768)).astype(np.float32), cuda_device)
    x = base[:, :640]                                                    # ldx 768 > K 640
    big = rng.standard_normal((128, 256)).astype(np.float32) * 1e30     # far beyond a tiny history
    tiny = rng.standard_normal((128, 256)).astype(np.float32) * 1e-30
    run_sequence([x, bf16_dev(big, cuda_device), bf16_dev(tiny, cuda_device), x], 2, cuda_device,
                 hist0=np.array([1e-20, 3.0], np.float32))


def test_delayed_quantize_only_config_full(cuda_device):
    """X [16384, 7168] with a history whose maximum is half of the tensor's: every
    outlier above that saturates."""
    x = inputs.quant_only(cuda_device)
    amax = float(x.abs().max().float())
    run_sequence([x, x], 16, cuda_device, hist0=np.full(16, amax / 2, np.float32))


def test_delayed_empty_tensor_pushes_zero(cuda_device):
    hist = ops.new_amax_history(3, cuda_device)
    hist[:3] = torch.tensor([5.0, 6.0, 7.0], device=cuda_device)
    e = torch.empty((0, 256), dtype=torch.bfloat16, device=cuda_device)
    q, s = ops.quant_act_delayed(e, hist)
    ops.sync_status()
    assert hist.cpu().tolist() == [0.0, 5.0, 6.0, 0.0]


def test_delayed_rejects_bad_history_length(cuda_device):
    x = torch.zeros((4, 128), dtype=torch.bfloat16, device=cuda_device)
    with pytest.raises(_lib.Fp8fgError) as ei:
        ops.quant_act_delayed(x, torch.zeros(1, dtype=torch.float32, device=cuda_device))   # H = 0
    assert ei.value.code == _lib.FP8FG_ERR_ARG
