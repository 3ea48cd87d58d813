"""GPU parity of the grouped (MoE) block-scaled GEMM against the oracle, through the C
ABI: small cases with empty experts and padding rows, the full MoE workload (256
experts, Zipf routing) on sampled experts, agreement with the dense kernel on each
expert's rows, and device-side rejection of invalid group offsets."""
import numpy as np
import pytest
import torch

from fp8_fine_grained_cast_b300 import _lib, inputs, ops
from oracle import fp8_oracle as O

pytestmark = pytest.mark.gpu


def f32(t):
    return t.detach().float().cpu().numpy()


def dev(a, device):
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def small_case(rng, counts, N, K):
    E = len(counts)
    padded = [((c + 127) // 128) * 128 for c in counts]
    off = np.concatenate([[0], np.cumsum(padded)]).astype(np.int32)
    Mtot = int(off[-1])
    xa = np.zeros((Mtot, K), np.float32)
    for e, c in enumerate(counts):
        xa[off[e]:off[e] + c] = rng.standard_normal((c, K))
    xa = torch.from_numpy(xa).to(torch.bfloat16).float().numpy()
    qa, sa = O.quant_act_1x128(xa)
    xb = torch.from_numpy((rng.standard_normal((E * N, K)) * 0.02).astype(np.float32)).to(torch.bfloat16).float().numpy()
    qb, sb = O.quant_w_128x128(xb)
    return qa, sa, qb.reshape(E, N, K), sb.reshape(E, N // 128, K // 128), off


@pytest.mark.parametrize("out_dtype,tol", [(torch.float32, 1e-4), (torch.bfloat16, 8e-3)])
@pytest.mark.parametrize("counts,N,K", [([130, 0, 5, 256], 256, 256), ([1, 300], 384, 640),
                                        ([0, 0, 128], 128, 128), ([77] * 9, 512, 384)])
def test_grouped_matches_oracle(cuda_device, out_dtype, tol, counts, N, K):
    rng = np.random.default_rng(sum(counts) + N + K)
    qa, sa, qb, sb, off = small_case(rng, counts, N, K)
    c = ops.grouped_gemm(dev(qa, cuda_device), dev(sa, cuda_device), dev(qb, cuda_device), dev(sb, cuda_device),
                         dev(off, cuda_device), out_dtype)
    ops.sync_status()
    ref = O.grouped_gemm(qa, sa, qb, sb, off)
    assert O.relative_error(f32(c), ref) <= tol
    for e, cnt in enumerate(counts):        # padding rows are exact zeros
        assert np.all(f32(c)[off[e] + cnt:off[e + 1]] == 0.0)


def test_grouped_equals_dense_per_expert(cuda_device):
    rng = np.random.default_rng(11)
    qa, sa, qb, sb, off = small_case(rng, [200, 128, 50], 256, 512)
    c = ops.grouped_gemm(dev(qa, cuda_device), dev(sa, cuda_device), dev(qb, cuda_device), dev(sb, cuda_device),
                         dev(off, cuda_device), torch.float32)
    for e in range(3):
        lo, hi = int(off[e]), int(off[e + 1])
        d = ops.blockscaled_gemm(dev(qa[lo:hi], cuda_device), dev(sa[lo:hi], cuda_device),
                                 dev(qb[e], cuda_device), dev(sb[e], cuda_device), ops.SB_BLOCK_128x128,
                                 torch.float32)
        assert torch.equal(c[lo:hi], d), e
    ops.sync_status()


def test_moe_config_full(cuda_device):
    """256 experts x [2048, 7168], ~32.8k routed rows padded per expert, BF16 out, in
    the launch configuration the benchmark times; oracle on the largest, the smallest
    and two other experts."""
    m = inputs.moe(cuda_device)
    E, N, K = m.w.shape
    qa, sa = ops.quant_act_1x128(m.a)
    qw, sw = ops.quant_w_128x128(m.w.view(E * N, K))
    c = ops.grouped_gemm(qa, sa, qw.view(E, N, K), sw.view(E, N // 128, K // 128), m.offsets, torch.bfloat16)
    ops.sync_status()
    counts = np.array(m.rows_per_expert)
    picks = sorted({int(np.argmax(counts)), int(np.argmin(counts)), 17, 200})
    off = m.offsets_host
    for e in picks:
        lo, hi = off[e], off[e + 1]
        rq, rs = O.quant_act_1x128(f32(m.a[lo:hi]))
        assert np.array_equal(qa[lo:hi].cpu().numpy(), rq) and np.array_equal(sa[lo:hi].cpu().numpy(), rs)
        wq, ws = O.quant_w_128x128(f32(m.w[e]))
        assert np.array_equal(qw[e * N:(e + 1) * N].cpu().numpy(), wq)
        ref = O.blockscaled_gemm(rq, rs, wq, ws)
        assert O.relative_error(f32(c[lo:hi]), ref) <= 8e-3, e
        assert np.all(f32(c[lo + counts[e]:hi]) == 0.0)


def test_moe_config_every_expert(cuda_device):
    """The full MoE workload, every one of the 256 experts: its first and last routed
    rows against the oracle on one 128-column block of the output (the oracle quantizes
    only that block's 128 weight rows, which the 128x128 blocks keep independent), and
    every padding row of every expert exactly zero."""
    m = inputs.moe(cuda_device)
    E, N, K = m.w.shape
    qa, sa = ops.quant_act_1x128(m.a)
    qw, sw = ops.quant_w_128x128(m.w.view(E * N, K))
    c = ops.grouped_gemm(qa, sa, qw.view(E, N, K), sw.view(E, N // 128, K // 128), m.offsets, torch.bfloat16)
    ops.sync_status()
    counts = np.array(m.rows_per_expert)
    off = m.offsets_host
    pad_rows = [np.arange(off[e] + counts[e], off[e + 1]) for e in range(E)]
    pad_rows = torch.from_numpy(np.concatenate(pad_rows)).to(cuda_device)
    assert pad_rows.numel() == int(off[E]) - int(counts.sum())
    assert torch.count_nonzero(c[pad_rows]).item() == 0
    checked = 0
    for e in range(E):
        if counts[e] == 0:
            continue
        rows = np.unique([off[e], off[e] + counts[e] - 1])
        nb = e % (N // 128)
        x_rows = f32(m.a[torch.from_numpy(rows).to(cuda_device)])
        rq, rs = O.quant_act_1x128(x_rows)
        wq, ws = O.quant_w_128x128(f32(m.w[e, 128 * nb:128 * (nb + 1)]))
        ref = O.blockscaled_gemm(rq, rs, wq, ws)
        got = f32(c[torch.from_numpy(rows).to(cuda_device), 128 * nb:128 * (nb + 1)])
        assert O.relative_error(got, ref) <= 8e-3, e
        checked += 1
    assert checked == int((counts > 0).sum())


def test_bad_offsets_are_reported(cuda_device):
    rng = np.random.default_rng(2)
    qa, sa, qb, sb, off = small_case(rng, [128, 128], 128, 128)
    bad = off.copy()
    bad[1] = 100                                               # not a multiple of 128
    ops.grouped_gemm(dev(qa, cuda_device), dev(sa, cuda_device), dev(qb, cuda_device), dev(sb, cuda_device),
                     dev(bad, cuda_device), torch.float32)
    with pytest.raises(_lib.Fp8fgError) as ei:
        ops.sync_status()
    assert ei.value.code == _lib.FP8FG_ERR_DEVICE_ARG
    ops.sync_status()                                          # the status word was cleared
