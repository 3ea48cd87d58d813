"""GPU parity of the GEMM whose output is quantized to E4M3 in 1x128 tiles, through the
C ABI, against the oracle (float64 product rounded once to binary32, then the 1x128
activation quantizer).

Where the tensor-core sums are exact (the exact-sum constructions below) the GPU's FP32
accumulators equal the oracle's binary32 values, so codes and scales must match bit for
bit. Elsewhere the two FP32 results differ by accumulation rounding (the FP32 GEMM
tolerance is 1e-4 of max|C|); then
  - every scale must agree within a relative 1e-5 (a tile maximum moves by that much
    at most), zero tiles exactly;
  - a code may differ only by one E4M3 step, and only where the oracle's quotient
    C / s lies within 2e-5 * 448 of the rounding midpoint between the two codes;
  - at most 0.5 % of the codes may differ on the small random cases, and on the full
    dense projection at most the cap below, about twice the count observed there.
"""
import numpy as np
import pytest
import torch

from fp8_fine_grained_cast_b300 import inputs, ops
from oracle import fp8_oracle as O
from tests.test_gpu_gemm import dev, f32, random_quantized

pytestmark = pytest.mark.gpu

# Codes of the full dense test (98 sampled rows x 18432 columns = 1.8M codes) that may
# differ from the oracle by one step next to a rounding midpoint: 7 were observed on a
# B300, the cap is about twice that.
DENSE_FULL_MAX_DIFFERING = 16


def run(qa, sa, qb, sb, sb_kind, device):
    q, s = ops.blockscaled_gemm_e4m3(dev(qa, device), dev(sa, device), dev(qb, device), dev(sb, device), sb_kind)
    ops.sync_status()
    return q.cpu().numpy(), s.cpu().numpy()


def assert_exact(q, s, q_ref, s_ref):
    assert np.array_equal(s.view(np.uint32), s_ref.view(np.uint32)), np.argwhere(s != s_ref)[:5]
    bad = np.argwhere(q != q_ref)
    assert bad.size == 0, (bad[:5].tolist(), q[tuple(bad[0])], q_ref[tuple(bad[0])])


def assert_close(q, s, q_ref, s_ref, c_ref):
    zero = s_ref == 0
    assert np.array_equal(s[zero], s_ref[zero])
    rel = np.abs(s[~zero].astype(np.float64) / s_ref[~zero] - 1.0)
    assert rel.size == 0 or rel.max() <= 1e-5, rel.max()
    bad = np.argwhere(q != q_ref)
    assert len(bad) <= 0.005 * q.size, f"{len(bad)} of {q.size} codes differ"
    print(f"e4m3-out codes differing from the oracle: {len(bad)} of {q.size}")
    if len(bad):
        m, n = bad[:, 0], bad[:, 1]
        dg = O.e4m3_decode(q[m, n])
        dr = O.e4m3_decode(q_ref[m, n])
        y = c_ref[m, n].astype(np.float64) / s_ref[m, n // 128]
        # adjacent codes: same sign (or a zero), one step apart in magnitude order
        ag, ar = q[m, n].astype(int) & 0x7F, q_ref[m, n].astype(int) & 0x7F
        assert np.all(np.abs(ag - ar) <= 1), "codes more than one step apart"
        mid = (dg + dr) / 2.0
        assert np.all(np.abs(y - mid) <= 2e-5 * 448), np.max(np.abs(y - mid))
    return len(bad)


@pytest.mark.parametrize("sb_kind", [O.SB_BLOCK_128x128, O.SB_ROW_1x128])
def test_e4m3_out_exact_single_chunk(cuda_device, sb_kind):
    """K = 128, codes in [1, 2), power-of-two scales: C is exact in FP32."""
    rng = np.random.default_rng(31)
    M, N, K = 256, 512, 128
    qa = (0x38 + rng.integers(0, 8, (M, K))).astype(np.uint8) | (rng.integers(0, 2, (M, K)) << 7).astype(np.uint8)
    qb = (0x38 + rng.integers(0, 8, (N, K))).astype(np.uint8) | (rng.integers(0, 2, (N, K)) << 7).astype(np.uint8)
    sa = np.exp2(rng.integers(-6, 6, (M, 1))).astype(np.float32)
    rows_b = N // 128 if sb_kind == O.SB_BLOCK_128x128 else N
    sb = np.exp2(rng.integers(-6, 6, (rows_b, 1))).astype(np.float32)
    q, s = run(qa, sa, qb, sb, sb_kind, cuda_device)
    q_ref, s_ref, _ = O.blockscaled_gemm_e4m3(qa, sa, qb, sb, sb_kind)
    assert_exact(q, s, q_ref, s_ref)


def test_e4m3_out_exact_chunk_promotion(cuda_device):
    """Four chunks, codes in {1, 2, 4}, scales in {1/2, 1, 2}: FP32 is exact throughout
    (sums below 2^15 in steps of 1/4), so the quantized output must match exactly."""
    rng = np.random.default_rng(32)
    M, N, K = 200, 384, 512
    qa = (0x38 + 8 * rng.integers(0, 3, (M, K))).astype(np.uint8)
    qb = (0x38 + 8 * rng.integers(0, 3, (N, K))).astype(np.uint8)
    qb[rng.random((N, K)) < 0.3] |= 0x80                                  # mixed signs
    sa = np.exp2(rng.integers(-1, 2, (M, K // 128))).astype(np.float32)
    sb = np.exp2(rng.integers(-1, 2, (N // 128, K // 128))).astype(np.float32)
    qa[7] = 0                                                              # an all-zero row of C
    q, s = run(qa, sa, qb, sb, O.SB_BLOCK_128x128, cuda_device)
    q_ref, s_ref, _ = O.blockscaled_gemm_e4m3(qa, sa, qb, sb)
    assert (s_ref[7] == 0).all()
    assert_exact(q, s, q_ref, s_ref)


@pytest.mark.parametrize("sb_kind", [O.SB_BLOCK_128x128, O.SB_ROW_1x128])
@pytest.mark.parametrize("M,N,K", [(128, 128, 128), (300, 384, 640), (1, 256, 256), (520, 1024, 1152)])
def test_e4m3_out_matches_oracle(cuda_device, sb_kind, M, N, K):
    rng = np.random.default_rng(M + 5 * N + 7 * K)
    qa, sa, qb, sb = random_quantized(rng, M, N, K, sb_kind)
    q, s = run(qa, sa, qb, sb, sb_kind, cuda_device)
    q_ref, s_ref, c_ref = O.blockscaled_gemm_e4m3(qa, sa, qb, sb, sb_kind)
    assert_close(q, s, q_ref, s_ref, c_ref)


def test_e4m3_out_dense_projection_full(cuda_device):
    """X [4096, 7168] . W^T [18432, 7168] with the output quantized, in the launch
    configuration the benchmark times; oracle on sampled rows."""
    d = inputs.dense(cuda_device)
    qx, sx = ops.quant_act_1x128(d.x)
    qw, sw = ops.quant_w_128x128(d.w)
    cq, cs = ops.blockscaled_gemm_e4m3(qx, sx, qw, sw)
    ops.sync_status()
    rq, rs = O.quant_act_1x128(f32(d.x))
    wq, ws = O.quant_w_128x128(f32(d.w))
    assert np.array_equal(qx.cpu().numpy(), rq) and np.array_equal(qw.cpu().numpy(), wq)
    rows = np.array(sorted(set(np.random.default_rng(3).choice(4096, 96, replace=False).tolist()) | {0, 4095}))
    q_ref, s_ref, c_ref = O.blockscaled_gemm_e4m3(rq, rs, wq, ws, rows=rows)
    sel = torch.from_numpy(rows).to(cuda_device)
    n_bad = assert_close(cq[sel].cpu().numpy(), cs[sel].cpu().numpy(), q_ref, s_ref, c_ref)
    assert n_bad <= DENSE_FULL_MAX_DIFFERING, n_bad


def test_e4m3_out_k_zero_and_empty(cuda_device):
    q = torch.full((4, 256), 0x55, dtype=torch.uint8, device=cuda_device)
    s = torch.full((4, 2), 7.0, dtype=torch.float32, device=cuda_device)
    ops.blockscaled_gemm_e4m3(torch.empty((4, 0), dtype=torch.uint8, device=cuda_device),
                              torch.empty((4, 0), dtype=torch.float32, device=cuda_device),
                              torch.empty((256, 0), dtype=torch.uint8, device=cuda_device),
                              torch.empty((2, 0), dtype=torch.float32, device=cuda_device), out=(q, s))
    ops.sync_status()
    assert torch.count_nonzero(q).item() == 0 and torch.count_nonzero(s).item() == 0
