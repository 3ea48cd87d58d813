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


def _need(t: torch.Tensor, dtype, name: str, ndim: int):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dimensions, got shape {tuple(t.shape)}")


def _rows_contiguous(t: torch.Tensor, name: str):
    if t.stride(-1) != 1:
        raise ValueError(f"{name}: the last dimension must be contiguous")


def quant_act_1x128(x: torch.Tensor, transposed: bool = False, q=None, s=None):
    """x bf16 [M, K] (row stride may exceed K) -> (q uint8, s float32).

    transposed=False: q [M, K], s [M, K/128] (tiles along K).
    transposed=True:  q [K, M], s [K, M/128] (tiles along M, stored transposed).
    """
    _need(x, torch.bfloat16, "x", 2)
    _rows_contiguous(x, "x")
    M, K = x.shape
    if transposed:
        q = torch.empty((K, M), dtype=torch.uint8, device=x.device) if q is None else q
        s = torch.empty((K, M // 128), dtype=torch.float32, device=x.device) if s is None else s
    else:
        q = torch.empty((M, K), dtype=torch.uint8, device=x.device) if q is None else q
        s = torch.empty((M, K // 128), dtype=torch.float32, device=x.device) if s is None else s
    _lib.fp8_quant_act_1x128(x.data_ptr(), M, K, x.stride(0), int(transposed), q.data_ptr(), s.data_ptr(),
                             _stream())
    return q, s


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
    M, K = x.shape
    q = torch.empty((M, K), dtype=torch.uint8, device=x.device) if q is None else q
    s = torch.empty((M, K // 128), dtype=torch.float32, device=x.device) if s is None else s
    _lib.fp8_quant_act_delayed(x.data_ptr(), M, K, x.stride(0), amax_history.data_ptr(), amax_history.numel() - 1,
                               q.data_ptr(), s.data_ptr(), _stream())
    return q, s


def quant_w_128x128(w: torch.Tensor, q=None, s=None):
    """w bf16 [N, K] -> (q uint8 [N, K], s float32 [N/128, K/128])."""
    _need(w, torch.bfloat16, "w", 2)
    _rows_contiguous(w, "w")
    N, K = w.shape
    q = torch.empty((N, K), dtype=torch.uint8, device=w.device) if q is None else q
    s = torch.empty((N // 128, K // 128), dtype=torch.float32, device=w.device) if s is None else s
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
    _lib.fp8_quant_w_128x128_dual(w.data_ptr(), N, K, w.stride(0), q.data_ptr(), s.data_ptr(), qt.data_ptr(),
                                  st.data_ptr(), _stream())
    return q, s, qt, st


def gemm_workspace(device) -> torch.Tensor:
    """A zero-filled workspace for the stream-K GEMM on `device` (reusable across calls)."""
    with torch.cuda.device(device):
        n = _lib.fp8_blockscaled_gemm_workspace_bytes()
    return torch.zeros(n, dtype=torch.uint8, device=device)


def blockscaled_gemm(qa, sa, qb, sb, sb_kind: int = SB_BLOCK_128x128, out_dtype=torch.bfloat16, c=None,
                     workspace=None):
    """C = A . B^T from E4M3 codes and scales; C [M, N] in bf16 or float32. With a
    workspace (see gemm_workspace) the stream-K schedule runs; the result is the same."""
    for t, n, dt, nd in ((qa, "qa", torch.uint8, 2), (sa, "sa", torch.float32, 2), (qb, "qb", torch.uint8, 2),
                         (sb, "sb", torch.float32, 2)):
        _need(t, dt, n, nd)
        if not t.is_contiguous():
            raise ValueError(f"{n} must be contiguous")
    M, K = qa.shape
    N = qb.shape[0]
    if qb.shape[1] != K:
        raise ValueError("qa and qb disagree on K")
    c_dtype = OUT_BF16 if out_dtype == torch.bfloat16 else OUT_F32
    if out_dtype not in (torch.bfloat16, torch.float32):
        raise TypeError("out_dtype must be torch.bfloat16 or torch.float32")
    c = torch.empty((M, N), dtype=out_dtype, device=qa.device) if c is None else c
    if workspace is None:
        _lib.fp8_blockscaled_gemm(qa.data_ptr(), sa.data_ptr(), qb.data_ptr(), sb.data_ptr(), sb_kind, c.data_ptr(),
                                  c_dtype, M, N, K, _stream())
    else:
        _need(workspace, torch.uint8, "workspace", 1)
        _lib.fp8_blockscaled_gemm_ws(qa.data_ptr(), sa.data_ptr(), qb.data_ptr(), sb.data_ptr(), sb_kind,
                                     c.data_ptr(), c_dtype, M, N, K, workspace.data_ptr(), workspace.numel(),
                                     _stream())
    return c


def blockscaled_gemm_e4m3(qa, sa, qb, sb, sb_kind: int = SB_BLOCK_128x128, out=None):
    """C = A . B^T quantized in 1x128 tiles from the FP32 accumulators:
    returns (c_q uint8 [M, N], c_s float32 [M, N/128])."""
    for t, n, dt, nd in ((qa, "qa", torch.uint8, 2), (sa, "sa", torch.float32, 2), (qb, "qb", torch.uint8, 2),
                         (sb, "sb", torch.float32, 2)):
        _need(t, dt, n, nd)
        if not t.is_contiguous():
            raise ValueError(f"{n} must be contiguous")
    M, K = qa.shape
    N = qb.shape[0]
    if qb.shape[1] != K:
        raise ValueError("qa and qb disagree on K")
    if out is None:
        out = (torch.empty((M, N), dtype=torch.uint8, device=qa.device),
               torch.empty((M, N // 128), dtype=torch.float32, device=qa.device))
    c_q, c_s = out
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
    if out_dtype not in (torch.bfloat16, torch.float32):
        raise TypeError("out_dtype must be torch.bfloat16 or torch.float32")
    c_dtype = OUT_BF16 if out_dtype == torch.bfloat16 else OUT_F32
    c = torch.empty((Mtot, N), dtype=out_dtype, device=qa.device) if c is None else c
    _lib.fp8_grouped_gemm(qa.data_ptr(), sa.data_ptr(), qb.data_ptr(), sb.data_ptr(), group_offsets.data_ptr(), E,
                          Mtot, c.data_ptr(), c_dtype, N, K, _stream())
    return c


def sync_status():
    """Synchronize the current stream and raise if a kernel reported a device-side error."""
    _lib.fp8fg_sync_status(_stream())
