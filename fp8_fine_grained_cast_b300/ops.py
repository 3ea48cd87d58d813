"""Tensor-level calls of the C ABI: torch supplies device memory and the stream.

Each function allocates its outputs with torch (device memory is PyTorch's job here),
then makes exactly one library call on the current CUDA stream; all arithmetic runs
in the library's kernels. Inputs must be CUDA tensors of the documented dtype and
layout; anything else raises before the call.
"""
from __future__ import annotations

import torch

from . import _lib

OUT_F32 = _lib.FP8FG_OUT_F32
OUT_BF16 = _lib.FP8FG_OUT_BF16
SB_BLOCK_128x128 = _lib.FP8FG_SB_BLOCK_128x128
SB_ROW_1x128 = _lib.FP8FG_SB_ROW_1x128


def _stream() -> int:
    return torch.cuda.current_stream().cuda_stream


def _need(t: torch.Tensor, dtype, name: str, ndim: int, cuda: bool = True):
    if not isinstance(t, torch.Tensor) or (cuda and not t.is_cuda):
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dimensions, got shape {tuple(t.shape)}")


def _rows_contiguous(t: torch.Tensor, name: str):
    if t.stride(-1) != 1:
        raise ValueError(f"{name}: the last dimension must be contiguous")


def _exact(t: torch.Tensor, shape, dtype, device, name: str, cuda: bool = True):
    """A tensor the library reads or writes as a dense row-major array of `shape`: the
    C ABI sees only its pointer, so every property it relies on is checked here."""
    if not isinstance(t, torch.Tensor) or (cuda and not t.is_cuda):
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, the operands on {device}")
    return t


def _out_or_new(t, shape, dtype, device, name: str):
    if t is None:
        return torch.empty(shape, dtype=dtype, device=device)
    return _exact(t, shape, dtype, device, name)


def quant_act_1x128(x: torch.Tensor, transposed: bool = False, q=None, s=None):
    """x bf16 [M, K] (row stride may exceed K) -> (q uint8, s float32).

    transposed=False: q [M, K], s [M, K/128] (tiles along K).
    transposed=True:  q [K, M], s [K, M/128] (tiles along M, stored transposed).
    """
    _need(x, torch.bfloat16, "x", 2)
    _rows_contiguous(x, "x")
    M, K = x.shape
    if transposed:
        q = _out_or_new(q, (K, M), torch.uint8, x.device, "q")
        s = _out_or_new(s, (K, M // 128), torch.float32, x.device, "s")
    else:
        q = _out_or_new(q, (M, K), torch.uint8, x.device, "q")
        s = _out_or_new(s, (M, K // 128), torch.float32, x.device, "s")
    _lib.fp8_quant_act_1x128(x.data_ptr(), M, K, x.stride(0), int(transposed), q.data_ptr(), s.data_ptr(),
                             _stream())
    return q, s


def quant_act_1x128_transposed_pair(x0: torch.Tensor, x1: torch.Tensor, out=None):
    """Tiles along M of two bf16 tensors with the same M ([M, K0] and [M, K1]) in one
    launch: returns (q0 [K0, M], s0 [K0, M/128], q1 [K1, M], s1 [K1, M/128]), the results of
    quant_act_1x128(x0, transposed=True) and quant_act_1x128(x1, transposed=True)."""
    for t, n in ((x0, "x0"), (x1, "x1")):
        _need(t, torch.bfloat16, n, 2)
        _rows_contiguous(t, n)
    if x0.device != x1.device:
        raise ValueError("x0 and x1 must be on the same device")
    M, K0 = x0.shape
    if x1.shape[0] != M:
        raise ValueError("x0 and x1 must have the same number of rows")
    K1 = x1.shape[1]
    q0, s0, q1, s1 = (None,) * 4 if out is None else out
    dev = x0.device
    q0 = _out_or_new(q0, (K0, M), torch.uint8, dev, "q0")
    s0 = _out_or_new(s0, (K0, M // 128), torch.float32, dev, "s0")
    q1 = _out_or_new(q1, (K1, M), torch.uint8, dev, "q1")
    s1 = _out_or_new(s1, (K1, M // 128), torch.float32, dev, "s1")
    _lib.fp8_quant_act_1x128_transposed_pair(x0.data_ptr(), K0, x0.stride(0), q0.data_ptr(), s0.data_ptr(),
                                             x1.data_ptr(), K1, x1.stride(0), q1.data_ptr(), s1.data_ptr(), M,
                                             _stream())
    return q0, s0, q1, s1


def new_amax_history(H: int, device) -> torch.Tensor:
    """Zero-initialized history state for quant_act_delayed: float32 [H + 1]."""
    return torch.zeros(H + 1, dtype=torch.float32, device=device)


def quant_act_delayed(x: torch.Tensor, amax_history: torch.Tensor, q=None, s=None):
    """Delayed scaling of x bf16 [M, K] with the per-tensor scale from amax_history
    (float32 [H + 1], updated in place): returns (q uint8 [M, K], s float32 [M, K/128])."""
    _need(x, torch.bfloat16, "x", 2)
    _rows_contiguous(x, "x")
    _need(amax_history, torch.float32, "amax_history", 1)
    if not amax_history.is_contiguous():
        raise ValueError("amax_history must be contiguous")
    if amax_history.device != x.device:
        raise ValueError("amax_history must be on the device of x")
    M, K = x.shape
    q = _out_or_new(q, (M, K), torch.uint8, x.device, "q")
    s = _out_or_new(s, (M, K // 128), torch.float32, x.device, "s")
    _lib.fp8_quant_act_delayed(x.data_ptr(), M, K, x.stride(0), amax_history.data_ptr(), amax_history.numel() - 1,
                               q.data_ptr(), s.data_ptr(), _stream())
    return q, s


def quant_w_128x128(w: torch.Tensor, q=None, s=None):
    """w bf16 [N, K] -> (q uint8 [N, K], s float32 [N/128, K/128])."""
    _need(w, torch.bfloat16, "w", 2)
    _rows_contiguous(w, "w")
    N, K = w.shape
    q = _out_or_new(q, (N, K), torch.uint8, w.device, "q")
    s = _out_or_new(s, (N // 128, K // 128), torch.float32, w.device, "s")
    _lib.fp8_quant_w_128x128(w.data_ptr(), N, K, w.stride(0), q.data_ptr(), s.data_ptr(), _stream())
    return q, s


def quant_act_1x128_dual(x: torch.Tensor, out=None):
    """x bf16 [M, K] -> (q [M, K], s [M, K/128], qt [K, M], st [K, M/128]) from one read of x:
    the results of quant_act_1x128(x) and quant_act_1x128(x, transposed=True)."""
    _need(x, torch.bfloat16, "x", 2)
    _rows_contiguous(x, "x")
    M, K = x.shape
    if out is None:
        dev = x.device
        out = (torch.empty((M, K), dtype=torch.uint8, device=dev),
               torch.empty((M, K // 128), dtype=torch.float32, device=dev),
               torch.empty((K, M), dtype=torch.uint8, device=dev),
               torch.empty((K, M // 128), dtype=torch.float32, device=dev))
    q, s, qt, st = out
    for t, shape, dt, n in ((q, (M, K), torch.uint8, "q"), (s, (M, K // 128), torch.float32, "s"),
                            (qt, (K, M), torch.uint8, "qt"), (st, (K, M // 128), torch.float32, "st")):
        _exact(t, shape, dt, x.device, n)
    _lib.fp8_quant_act_1x128_dual(x.data_ptr(), M, K, x.stride(0), q.data_ptr(), s.data_ptr(), qt.data_ptr(),
                                  st.data_ptr(), _stream())
    return q, s, qt, st


def quant_w_128x128_dual(w: torch.Tensor, out=None):
    """w bf16 [N, K] -> (q [N, K], s [N/128, K/128], qt [K, N], st [K/128, N/128]): the 128x128
    block quantization of w and its transpose (the B operand of dX = dY . W)."""
    _need(w, torch.bfloat16, "w", 2)
    _rows_contiguous(w, "w")
    N, K = w.shape
    if out is None:
        dev = w.device
        out = (torch.empty((N, K), dtype=torch.uint8, device=dev),
               torch.empty((N // 128, K // 128), dtype=torch.float32, device=dev),
               torch.empty((K, N), dtype=torch.uint8, device=dev),
               torch.empty((K // 128, N // 128), dtype=torch.float32, device=dev))
    q, s, qt, st = out
    for t, shape, dt, n in ((q, (N, K), torch.uint8, "q"), (s, (N // 128, K // 128), torch.float32, "s"),
                            (qt, (K, N), torch.uint8, "qt"), (st, (K // 128, N // 128), torch.float32, "st")):
        _exact(t, shape, dt, w.device, n)
    _lib.fp8_quant_w_128x128_dual(w.data_ptr(), N, K, w.stride(0), q.data_ptr(), s.data_ptr(), qt.data_ptr(),
                                  st.data_ptr(), _stream())
    return q, s, qt, st


def gemm_workspace(device) -> torch.Tensor:
    """A zero-filled workspace for the stream-K GEMM on `device` (reusable across calls)."""
    with torch.cuda.device(device):
        n = _lib.fp8_blockscaled_gemm_workspace_bytes()
    return torch.zeros(n, dtype=torch.uint8, device=device)


def _gemm_operands(qa, sa, qb, sb, sb_kind, cuda: bool = True):
    """Checks the operands of a dense GEMM against each other; returns (M, N, K).
    (cuda=False runs the same checks on host tensors, for testing without a GPU.)"""
    _need(qa, torch.uint8, "qa", 2, cuda)
    _need(qb, torch.uint8, "qb", 2, cuda)
    M, K = qa.shape
    N = qb.shape[0]
    if qb.shape[1] != K:
        raise ValueError("qa and qb disagree on K")
    if sb_kind not in (SB_BLOCK_128x128, SB_ROW_1x128):
        raise ValueError(f"unknown sb_kind {sb_kind}")
    dev = qa.device
    _exact(qa, (M, K), torch.uint8, dev, "qa", cuda)
    _exact(qb, (N, K), torch.uint8, dev, "qb", cuda)
    _exact(sa, (M, K // 128), torch.float32, dev, "sa", cuda)
    sb_rows = N // 128 if sb_kind == SB_BLOCK_128x128 else N
    _exact(sb, (sb_rows, K // 128), torch.float32, dev, "sb", cuda)
    return M, N, K


def blockscaled_gemm(qa, sa, qb, sb, sb_kind: int = SB_BLOCK_128x128, out_dtype=torch.bfloat16, c=None,
                     workspace=None):
    """C = A . B^T from E4M3 codes and scales; C [M, N] in bf16 or float32. With a
    workspace (see gemm_workspace) the stream-K schedule runs; the result is the same."""
    M, N, K = _gemm_operands(qa, sa, qb, sb, sb_kind)
    if out_dtype not in (torch.bfloat16, torch.float32):
        raise TypeError("out_dtype must be torch.bfloat16 or torch.float32")
    c_dtype = OUT_BF16 if out_dtype == torch.bfloat16 else OUT_F32
    c = _out_or_new(c, (M, N), out_dtype, qa.device, "c")
    if workspace is None:
        _lib.fp8_blockscaled_gemm(qa.data_ptr(), sa.data_ptr(), qb.data_ptr(), sb.data_ptr(), sb_kind, c.data_ptr(),
                                  c_dtype, M, N, K, _stream())
    else:
        _need(workspace, torch.uint8, "workspace", 1)
        if not workspace.is_contiguous() or workspace.device != qa.device:
            raise ValueError("workspace must be contiguous and on the device of the operands")
        _lib.fp8_blockscaled_gemm_ws(qa.data_ptr(), sa.data_ptr(), qb.data_ptr(), sb.data_ptr(), sb_kind,
                                     c.data_ptr(), c_dtype, M, N, K, workspace.data_ptr(), workspace.numel(),
                                     _stream())
    return c


def blockscaled_gemm_e4m3(qa, sa, qb, sb, sb_kind: int = SB_BLOCK_128x128, out=None):
    """C = A . B^T quantized in 1x128 tiles from the FP32 accumulators:
    returns (c_q uint8 [M, N], c_s float32 [M, N/128])."""
    M, N, K = _gemm_operands(qa, sa, qb, sb, sb_kind)
    c_q, c_s = (None, None) if out is None else out
    c_q = _out_or_new(c_q, (M, N), torch.uint8, qa.device, "c_q")
    c_s = _out_or_new(c_s, (M, N // 128), torch.float32, qa.device, "c_s")
    _lib.fp8_blockscaled_gemm_e4m3(qa.data_ptr(), sa.data_ptr(), qb.data_ptr(), sb.data_ptr(), sb_kind,
                                   c_q.data_ptr(), c_s.data_ptr(), M, N, K, _stream())
    return c_q, c_s


def grouped_gemm(qa, sa, qb, sb, group_offsets, out_dtype=torch.bfloat16, c=None):
    """Grouped GEMM: qa [Mtot, K], qb [E, N, K], sb [E, N/128, K/128], offsets int32 [E+1]."""
    _need(qa, torch.uint8, "qa", 2)
    _need(sa, torch.float32, "sa", 2)
    _need(qb, torch.uint8, "qb", 3)
    _need(sb, torch.float32, "sb", 3)
    _need(group_offsets, torch.int32, "group_offsets", 1)
    for t, n in ((qa, "qa"), (sa, "sa"), (qb, "qb"), (sb, "sb"), (group_offsets, "group_offsets")):
        if not t.is_contiguous():
            raise ValueError(f"{n} must be contiguous")
    Mtot, K = qa.shape
    E, N, _ = qb.shape
    if group_offsets.numel() != E + 1:
        raise ValueError("group_offsets must have E + 1 entries")
    dev = qa.device
    _exact(qb, (E, N, K), torch.uint8, dev, "qb")
    _exact(sa, (Mtot, K // 128), torch.float32, dev, "sa")
    _exact(sb, (E, N // 128, K // 128), torch.float32, dev, "sb")
    _exact(group_offsets, (E + 1,), torch.int32, dev, "group_offsets")
    if out_dtype not in (torch.bfloat16, torch.float32):
        raise TypeError("out_dtype must be torch.bfloat16 or torch.float32")
    c_dtype = OUT_BF16 if out_dtype == torch.bfloat16 else OUT_F32
    c = _out_or_new(c, (Mtot, N), out_dtype, dev, "c")
    _lib.fp8_grouped_gemm(qa.data_ptr(), sa.data_ptr(), qb.data_ptr(), sb.data_ptr(), group_offsets.data_ptr(), E,
                          Mtot, c.data_ptr(), c_dtype, N, K, _stream())
    return c


def sync_status():
    """Synchronize the current stream and raise if a kernel reported a device-side error."""
    _lib.fp8fg_sync_status(_stream())
