"""Seeded synthetic inputs with the shapes and value distributions of the DeepSeek-V3
FP8 workloads. Input generation only: nothing here quantizes or multiplies.

Every tensor is drawn with torch's generator on the requested device, seeded from
(configuration seed, tensor id), sampled in float32 and rounded once to bf16 (round to
nearest even). The same call on the same device and software returns the same bytes;
the CPU and CUDA generators produce different streams, so a check always feeds the
very same tensors (copied to the host when needed) to both sides.

Workloads (one scale group = 1x128 activation tile or 128x128 weight block):
  tiny        X [128, 512] ~ N(0, 1) with round(0.001 * numel) entries x50,
              W [128, 512] ~ N(0, 0.02)                                 (seed 0)
  quant       X [16384, 7168] ~ N(0, 1), 0.1% entries x100, one all-zero 1x128
              tile per 1024 rows (seeded row and tile column)          (seed 1)
  dense       X [4096, 7168] as `quant`, W [18432, 7168] ~ N(0, 0.02)    (seed 2)
  moe         4096 tokens x 7168 as `quant`; each token picks 8 distinct experts of
              256 by Gumbel-top-k on log p(e), p(e) ~ (e + 1)^-1.1; each expert's rows
              are its tokens in token order, zero-padded to a multiple of 128 rows;
              W [256, 2048, 7168] ~ N(0, 0.02)                            (seed 3)
  wgrad       dY [4096, 2048] ~ N(0, 1e-3), X [4096, 7168] ~ N(0, 1)     (seed 4)
  dgrad       backward of the dense projection: dY [4096, 18432] ~ N(0, 1e-3),
              W [18432, 7168] ~ N(0, 0.02); dX = dY . W [4096, 7168]      (seed 5)
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

CONFIG_SEEDS = {"tiny": 0, "quant": 1, "dense": 2, "moe": 3, "wgrad": 4, "dgrad": 5}


def _gen(device, seed: int, tensor_id: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed * 1_000_003 + tensor_id)
    return g


def gaussian_bf16(shape, sigma: float, device, seed: int, tensor_id: int) -> torch.Tensor:
    g = _gen(device, seed, tensor_id)
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if sigma != 1.0:
        x.mul_(sigma)
    return x.to(torch.bfloat16)


def activation_bf16(rows: int, cols: int, outlier_scale: float, outlier_frac: float, zero_tile_every: int,
                    device, seed: int, tensor_id: int) -> torch.Tensor:
    """N(0, 1) activations with exactly round(outlier_frac * numel) entries (chosen
    uniformly without replacement) multiplied by outlier_scale, and, if
    zero_tile_every > 0, one all-zero 1x128 tile per block of that many rows."""
    g = _gen(device, seed, tensor_id)
    x = torch.randn((rows, cols), generator=g, device=device, dtype=torch.float32)
    n = x.numel()
    count = int(round(outlier_frac * n))
    if count:
        pos = torch.randperm(n, generator=g, device=device)[:count]
        x.view(-1)[pos] *= outlier_scale
    if zero_tile_every > 0 and cols >= 128:
        blocks = (rows + zero_tile_every - 1) // zero_tile_every
        r_in = torch.randint(0, zero_tile_every, (blocks,), generator=g, device=device).cpu()
        t_col = torch.randint(0, cols // 128, (blocks,), generator=g, device=device).cpu()
        for b in range(blocks):
            r = b * zero_tile_every + int(r_in[b])
            if r < rows:
                c = int(t_col[b]) * 128
                x[r, c:c + 128] = 0.0
    return x.to(torch.bfloat16)


@dataclass
class Tiny:
    x: torch.Tensor
    w: torch.Tensor


def tiny(device="cpu") -> Tiny:
    s = CONFIG_SEEDS["tiny"]
    return Tiny(x=activation_bf16(128, 512, 50.0, 0.001, 0, device, s, 0),
                w=gaussian_bf16((128, 512), 0.02, device, s, 1))


def quant_only(device="cpu", rows: int = 16384, cols: int = 7168) -> torch.Tensor:
    return activation_bf16(rows, cols, 100.0, 0.001, 1024, device, CONFIG_SEEDS["quant"], 0)


@dataclass
class Dense:
    x: torch.Tensor
    w: torch.Tensor


def dense(device="cpu", M: int = 4096, N: int = 18432, K: int = 7168) -> Dense:
    s = CONFIG_SEEDS["dense"]
    return Dense(x=activation_bf16(M, K, 100.0, 0.001, 1024, device, s, 0),
                 w=gaussian_bf16((N, K), 0.02, device, s, 1))


@dataclass
class MoE:
    a: torch.Tensor              # bf16 [Mtot, K]: gathered token rows, zero padding rows
    w: torch.Tensor              # bf16 [E, N, K]
    offsets: torch.Tensor        # int32 [E + 1] on the same device, multiples of 128
    offsets_host: list           # the same offsets as Python ints
    rows_per_expert: list        # real (unpadded) rows per expert
    token_of_row: torch.Tensor   # int64 [Mtot]: source token of each row, -1 for padding
    real_rows: int


def zipf_topk_routing(tokens: int, experts: int, top_k: int, exponent: float, device, seed: int,
                      tensor_id: int) -> torch.Tensor:
    """[tokens, top_k] distinct expert ids per token: Gumbel-top-k sampling without
    replacement from p(e) proportional to (e + 1)^-exponent."""
    g = _gen(device, seed, tensor_id)
    logp = -exponent * torch.log(torch.arange(1, experts + 1, device=device, dtype=torch.float64))
    u = torch.rand((tokens, experts), generator=g, device=device, dtype=torch.float64)
    u = u.clamp_min(1e-300)
    gumbel = -torch.log(-torch.log(u))
    return torch.topk(logp[None, :] + gumbel, top_k, dim=1).indices


def moe(device="cpu", tokens: int = 4096, hidden: int = 7168, experts: int = 256, inter: int = 2048,
        top_k: int = 8, exponent: float = 1.1) -> MoE:
    s = CONFIG_SEEDS["moe"]
    x = activation_bf16(tokens, hidden, 100.0, 0.001, 1024, device, s, 0)
    route = zipf_topk_routing(tokens, experts, top_k, exponent, device, s, 1).cpu()
    flat_e = route.reshape(-1)
    flat_t = torch.arange(tokens).repeat_interleave(top_k)
    order = torch.argsort(flat_e * tokens + flat_t)          # by expert, then token id
    flat_e, flat_t = flat_e[order], flat_t[order]
    counts = torch.bincount(flat_e, minlength=experts)
    padded = ((counts + 127) // 128) * 128
    offsets = torch.zeros(experts + 1, dtype=torch.int64)
    offsets[1:] = torch.cumsum(padded, 0)
    mtot = int(offsets[-1])
    token_of_row = torch.full((mtot,), -1, dtype=torch.int64)
    starts = torch.zeros(experts, dtype=torch.int64)
    starts[1:] = torch.cumsum(counts, 0)[:-1]
    pos_in_expert = torch.arange(flat_e.numel()) - starts[flat_e]
    token_of_row[offsets[:-1][flat_e] + pos_in_expert] = flat_t
    a = torch.zeros((mtot, hidden), dtype=torch.bfloat16, device=device)
    real = token_of_row >= 0
    a[real.to(device)] = x[token_of_row[real].to(device)]
    w = torch.empty((experts, inter, hidden), dtype=torch.bfloat16, device=device)
    for e in range(experts):
        w[e] = gaussian_bf16((inter, hidden), 0.02, device, s, 100 + e)
    return MoE(a=a, w=w, offsets=offsets.to(torch.int32).to(device), offsets_host=offsets.tolist(),
               rows_per_expert=counts.tolist(), token_of_row=token_of_row, real_rows=int(counts.sum()))


@dataclass
class WGrad:
    dy: torch.Tensor
    x: torch.Tensor


def wgrad(device="cpu", T: int = 4096, dout: int = 2048, din: int = 7168) -> WGrad:
    s = CONFIG_SEEDS["wgrad"]
    return WGrad(dy=gaussian_bf16((T, dout), 1e-3, device, s, 0), x=gaussian_bf16((T, din), 1.0, device, s, 1))


@dataclass
class DGrad:
    dy: torch.Tensor
    w: torch.Tensor


def dgrad(device="cpu", T: int = 4096, dout: int = 18432, din: int = 7168) -> DGrad:
    s = CONFIG_SEEDS["dgrad"]
    return DGrad(dy=gaussian_bf16((T, dout), 1e-3, device, s, 0), w=gaussian_bf16((dout, din), 0.02, device, s, 1))


def gemm_flops(M: int, N: int, K: int) -> float:
    return 2.0 * M * N * K


def moe_real_flops(m: MoE, inter: int, hidden: int) -> float:
    return 2.0 * m.real_rows * inter * hidden


__all__ = ["CONFIG_SEEDS", "tiny", "quant_only", "dense", "moe", "wgrad", "dgrad", "gaussian_bf16", "activation_bf16",
           "zipf_topk_routing", "gemm_flops", "moe_real_flops"]
