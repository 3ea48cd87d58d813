"""Benchmark of the fine-grained FP8 hot path on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--no-rows]

Step (the timed unit): the dense-projection workload — X bf16 [4096, 7168] quantized in
1x128 tiles, W bf16 [18432, 7168] quantized in 128x128 blocks, then the block-scaled
FP8 GEMM C [4096, 18432] = X . W^T with BF16 output: three library calls through the C
ABI, inputs resident in HBM. `value` is the step's GEMM FLOPs over the step time
(TFLOP/s). The inputs (322 MB) exceed the 126 MB L2, so no flush is needed between
steps. `e2e` repeats the step through the same calls with the inputs in pinned host
memory: host-to-device copies of X and W and the device-to-host copy of C are inside
the timed region. `rows` times every other kernel of the path alone (quantize-only
1x128 [16384, 7168], transposed quantization and the weight-gradient GEMM, and the
grouped MoE GEMM), each against its roofline; L2 is flushed between those runs.

Under torchrun (N > 1) every rank runs the same step on its own GPU with its own data
(weak scaling, no collective on the data path); the time is the max over ranks and
`value` counts the work of all ranks.

--impl reference times the CPU oracle on a bounded sample of the same workload on the
host cores (rank 0 only).
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "block-scaled FP8 GEMM TFLOP/s (% FP8 peak); 1x128 quantize GB/s (% HBM)"
WORKLOAD = "dense projection: X bf16 [4096,7168] 1x128 + W bf16 [18432,7168] 128x128 quantize, block-scaled GEMM C[4096,18432] BF16"
M, N, K = 4096, 18432, 7168
GEMM_FLOPS = 2.0 * M * N * K
FP8_OVER_BF16 = 2.0          # nominal dense FP8 / BF16 tensor rate of the part (4.5 / 2.25 PFLOP/s)
GEMM_KERNEL_NAME = "blockscaled_gemm_kernel<256,4,0,bf16>"
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}


# ----------------------------------------------------------------------------- helpers


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def _code_only(text: str) -> str:
    """Source text without comments and blank space, so that the hash follows the code."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "".join(text.split())


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for f in ("gemm.cu", "gemm_sched.cuh", "quant.cu", "common.cuh", "e4m3.cuh"):
        h.update(_code_only(open(os.path.join(ROOT, "fp8_fine_grained_cast_b300", "csrc", f)).read()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(kernel: str):
    """DRAM bytes per launch recorded from an ncu capture (profiles/dram_traffic.txt),
    or None when absent or taken on other kernel sources."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(p):
        return None
    for line in open(p):
        parts = line.split("#", 1)[0].split()          # a trailing comment names the case
        if len(parts) == 3 and parts[0] == kernel:
            return int(parts[2]) if parts[1] == kernel_source_hash() else None
    return None


class ClockSampler:
    """nvidia-smi clock and throttle-reason samples (every 50 ms) during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"fp8fg_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax, "samples": len(sm),
                "reasons": sorted(reasons)}


# ----------------------------------------------------------------------------- distributed


def dist_setup():
    """(rank, world, local_rank) from the torchrun environment; a process group (NCCL
    on GPUs, gloo otherwise) only when world > 1."""
    import torch
    import torch.distributed as dist
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1 and not dist.is_initialized():
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    return rank, world, local


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def max_over_ranks(value: float, device=None) -> float:
    """Maximum of a per-rank scalar (the elapsed time) over all ranks."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_throughput(units_per_rank: float, world: int, max_elapsed_s: float) -> float:
    """Whole-job throughput: the units of all ranks over the slowest rank's time."""
    return units_per_rank * world / max_elapsed_s


# ----------------------------------------------------------------------------- our arm


def run_ours(args, rank, world, local):
    import torch
    from fp8_fine_grained_cast_b300 import inputs, ops

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    peaks, peak_kind = load_peaks()
    fp8_peak = FP8_OVER_BF16 * peaks["bf16_tflops"]
    fp8_peak_sus = FP8_OVER_BF16 * peaks["bf16_tflops_sustained"]
    hbm_peak = peaks["hbm_gbs"]

    d = inputs.dense(dev)
    x, w = d.x, d.w
    qx = torch.empty((M, K), dtype=torch.uint8, device=dev)
    sx = torch.empty((M, K // 128), dtype=torch.float32, device=dev)
    qw = torch.empty((N, K), dtype=torch.uint8, device=dev)
    sw = torch.empty((N // 128, K // 128), dtype=torch.float32, device=dev)
    c = torch.empty((M, N), dtype=torch.bfloat16, device=dev)

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        ops.quant_act_1x128(x, q=qx, s=sx)
        if ev is not None:
            ev[1].record(stream)
        ops.quant_w_128x128(w, q=qw, s=sw)
        if ev is not None:
            ev[2].record(stream)
        ops.blockscaled_gemm(qx, sx, qw, sw, ops.SB_BLOCK_128x128, torch.bfloat16, c=c)
        if ev is not None:
            ev[3].record(stream)

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clocks:
        # the warm-up steps run after the sampler has started (starting it leaves the GPU
        # idle for a moment), directly before the timed steps
        for _ in range(args.warmup):
            step()
        ops.sync_status()
        barrier()
        torch.cuda.synchronize()
        start.record(stream)
        for i in range(args.steps):
            step(evs[i])
        stop.record(stream)
        torch.cuda.synchronize()
    barrier()
    ops.sync_status()
    elapsed_ms = start.elapsed_time(stop)
    elapsed_ms = max_over_ranks(elapsed_ms, dev)
    ms_per_step = elapsed_ms / args.steps
    value = aggregate_throughput(GEMM_FLOPS, world, ms_per_step / 1e3) / 1e12
    t_qx = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
    t_qw = statistics.mean(e[1].elapsed_time(e[2]) for e in evs)
    t_gemm = statistics.mean(e[2].elapsed_time(e[3]) for e in evs)
    gemm_tflops = GEMM_FLOPS / (t_gemm / 1e3) / 1e12
    qx_bytes = M * K * 2 + M * K + M * (K // 128) * 4
    qw_bytes = N * K * 2 + N * K + (N // 128) * (K // 128) * 4
    clk = clocks.summary()

    # ------------------------------------------------------------------ end to end
    # Every step copies its inputs X and W from pinned host memory and reads its result C
    # back, through the public ops. The copies run on their own streams (one per
    # direction, double-buffered on the device), so that step i+1's upload and step
    # i-1's download overlap step i's kernels; events order every buffer reuse.
    xh = x.cpu().pin_memory()
    wh = w.cpu().pin_memory()
    chs = [torch.empty((M, N), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    xds = [torch.empty_like(x) for _ in range(2)]
    wds = [torch.empty_like(w) for _ in range(2)]
    cds = [torch.empty_like(c) for _ in range(2)]
    s_h2d, s_d2h = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = {k: [torch.cuda.Event() for _ in range(2)] for k in ("in", "used", "out", "read")}
    for k in ev:                                  # every event recorded once: waits are then well defined
        for e_ in ev[k]:
            e_.record(stream)

    def e2e_step(i):
        j = i % 2
        with torch.cuda.stream(s_h2d):
            s_h2d.wait_event(ev["used"][j])       # step i-2 has finished reading these inputs
            xds[j].copy_(xh, non_blocking=True)
            wds[j].copy_(wh, non_blocking=True)
            ev["in"][j].record(s_h2d)
        stream.wait_event(ev["in"][j])
        stream.wait_event(ev["read"][j])          # step i-2's result has been downloaded
        ops.quant_act_1x128(xds[j], q=qx, s=sx)
        ops.quant_w_128x128(wds[j], q=qw, s=sw)
        ev["used"][j].record(stream)
        ops.blockscaled_gemm(qx, sx, qw, sw, ops.SB_BLOCK_128x128, torch.bfloat16, c=cds[j])
        ev["out"][j].record(stream)
        with torch.cuda.stream(s_d2h):
            s_d2h.wait_event(ev["out"][j])
            chs[j].copy_(cds[j], non_blocking=True)
            ev["read"][j].record(s_d2h)

    for i in range(2):
        e2e_step(i)
    torch.cuda.synchronize()
    e2e_steps = max(3, min(args.steps, 10))
    barrier()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(s_h2d)
    for i in range(e2e_steps):
        e2e_step(i)
    b.record(s_d2h)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(a.elapsed_time(b), dev) / e2e_steps
    e2e_value = aggregate_throughput(GEMM_FLOPS, world, e2e_ms / 1e3) / 1e12
    assert torch.equal(chs[(e2e_steps - 1) % 2], c.cpu()), "end-to-end result differs from the device-resident step"
    ops.sync_status()

    rows = {} if args.no_rows else bench_rows(dev, stream, hbm_peak, fp8_peak, args)

    # The FP8 denominators: 2 x the measured BF16 rates, or the measured plain FP8 GEMM
    # where that is higher. Measured last: its loop at the full tensor rate leaves the
    # part power-capped for a while, which would slow whatever runs next.
    fp8_check = plain_fp8_gemm_check(dev)
    if fp8_check["burst_tflops"] > fp8_peak:
        rescale_tensor_fracs(rows, fp8_check["burst_tflops"])
    fp8_peak = max(fp8_peak, fp8_check["burst_tflops"])
    fp8_peak_sus = max(fp8_peak_sus, fp8_check["sustained_tflops"])
    fp8_check["gemm_in_step_vs_sustained"] = round(gemm_tflops / fp8_check["sustained_tflops"], 4)
    launches = 3 * args.steps

    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "e4m3 x e4m3 -> f32 (bf16 in, bf16 out)",
        "data": "synthetic (seeded N(0,1) activations with 0.1% x100 outliers and zero tiles; N(0,0.02) weights)",
        "config": {"workload": WORKLOAD, "M": M, "N": N, "K": K, "l2": "inputs 322 MB > 126 MB L2, no flush",
                   "parallelism": f"replicas x{world} (weak, no data-path collective)"},
        "frac_of_fp8_peak": round(value / fp8_peak, 4),
        # the timed region lasts milliseconds, not seconds, so the denominator is the
        # burst tensor rate (2 x the measured burst BF16 rate); the sustained figure is
        # reported beside it
        "roofline": {"bound": "tensor", "kernel": GEMM_KERNEL_NAME,
                     "achieved": round(gemm_tflops, 2), "peak": round(fp8_peak, 1), "unit": "TFLOP/s",
                     "frac": round(gemm_tflops / fp8_peak, 4),
                     "peak_source": (f"{peak_kind}: 2 x bf16 burst {peaks['bf16_tflops']} TFLOP/s "
                                     "(nominal FP8/BF16 ratio) or the measured plain FP8 GEMM if higher; "
                                     f"timed region {args.steps} steps = {elapsed_ms:.1f} ms"),
                     "plain_fp8_gemm": fp8_check,
                     "peak_sustained": round(fp8_peak_sus, 1),
                     "frac_of_sustained": round(gemm_tflops / fp8_peak_sus, 4),
                     "traffic": profiled_traffic("blockscaled_gemm_dense"),
                     "algorithmic_flops_per_launch": GEMM_FLOPS, "avg_launch_ms": round(t_gemm, 4)},
        "step_kernels_ms": {"quant_act_1x128": round(t_qx, 4), "quant_w_128x128": round(t_qw, 4),
                            "blockscaled_gemm": round(t_gemm, 4)},
        "quantize": {"act_1x128_GBps": round(qx_bytes / (t_qx / 1e3) / 1e9, 1),
                     "act_frac_hbm": round(qx_bytes / (t_qx / 1e3) / 1e9 / hbm_peak, 4),
                     "w_128x128_GBps": round(qw_bytes / (t_qw / 1e3) / 1e9, 1),
                     "w_frac_hbm": round(qw_bytes / (t_qw / 1e3) / 1e9 / hbm_peak, 4),
                     "hbm_peak_GBps": hbm_peak,
                     "note": ("in-step figures: the X quantizer follows the previous step's GEMM, whose "
                              "C (151 MB) is still partly dirty in L2 and is written back during it; "
                              "the quantizers alone are in rows")},
        "e2e": {"value": round(e2e_value, 3), "unit": "TFLOP/s", "ms_per_step": round(e2e_ms, 3),
                "h2d_bytes_per_step": x.numel() * 2 + w.numel() * 2, "d2h_bytes_per_step": c.numel() * 2,
                "pipelining": "uploads, kernels and downloads of consecutive steps on three streams"},
        "gpu_launches": launches,
        "clocks": clk,
        "rows": rows,
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.cpu_sample_rows, args.cpu_sample_wrows, args.cpu_sample_qrows)
    return line


def flush_l2(flush):
    """Evict L2 before a timed launch: write a buffer larger than L2 (512 MB), then read
    half of it, so that the write-back of the flush's own dirty lines happens here and
    not inside the timed kernel (ncu's cache-controlled durations agree with this)."""
    flush.zero_()
    flush[: flush.numel() // 2].max()


def timed(fn, stream, iters, warm, flush):
    """Median device time (ms) of fn over `iters` runs, L2 flushed before each run (the
    median keeps a rare host-side stall between the events from skewing a short kernel)."""
    import torch
    for _ in range(warm):
        fn()
    ts = []
    for _ in range(iters):
        flush_l2(flush)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b))
    return statistics.median(ts)


def rescale_tensor_fracs(rows, peak):
    """Recompute the tensor-bound rows' fractions (and their stream-K entries) against
    another FP8 peak."""
    for row in rows.values():
        if not (isinstance(row, dict) and row.get("bound") == "tensor"):
            continue
        for d in (row, row.get("stream_k")):
            if isinstance(d, dict) and "TFLOPs" in d and "frac" in d:
                d["frac"] = round(d["TFLOPs"] / peak, 4)


def plain_fp8_gemm_check(dev, m=M, n=N, k=K, secs=1.5, flush=None):
    """Measured confirmation of the FP8 denominator: the library's plain FP8 GEMM
    (cuBLASLt through torch._scaled_mm, one scale per tensor, no fine-grained scaling) on
    a GEMM shape (the dense projection by default), as a burst (median of single launches)
    and, if `secs` > 0, as a loop of about `secs` seconds. A loop at the full tensor rate
    leaves the part power-capped for a while, so the rows take the burst only. Used only
    as a reference rate, outside every timed region. With `flush`, L2 is flushed before
    each burst launch, as for the rows."""
    import torch
    a = torch.randn(m, k, device=dev).to(torch.float8_e4m3fn)
    b = torch.randn(n, k, device=dev).to(torch.float8_e4m3fn)
    one = torch.tensor(1.0, device=dev)
    flops = 2.0 * m * n * k

    def f():
        return torch._scaled_mm(a, b.t(), scale_a=one, scale_b=one, out_dtype=torch.bfloat16)
    for _ in range(5):
        f()
    torch.cuda.synchronize()
    ts = []
    for _ in range(10):
        if flush is not None:
            flush_l2(flush)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        f()
        e1.record()
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1))
    t_burst = statistics.median(ts)
    out = {"kernel": f"cuBLASLt per-tensor FP8 GEMM (torch._scaled_mm) {m}x{n}x{k}, bf16 out",
           "burst_tflops": round(flops / (t_burst * 1e-3) / 1e12, 1)}
    if secs <= 0:
        return out
    reps = max(1, int(secs / (t_burst * 1e-3)))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        f()
    e1.record()
    torch.cuda.synchronize()
    t_loop = e0.elapsed_time(e1) / reps
    out["sustained_tflops"] = round(flops / (t_loop * 1e-3) / 1e12, 1)
    return out


def bench_rows(dev, stream, hbm_peak, fp8_peak, args):
    """Each remaining kernel of the path alone, against its roofline."""
    import torch
    from fp8_fine_grained_cast_b300 import inputs, ops

    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    iters, warm = max(5, min(args.steps, 20)), 3
    out = {}
    gemm_ws = ops.gemm_workspace(dev)

    # The fixed cost of one launch under this protocol (L2 flushed, two events): each
    # quantizer on a single 128 x 128 tile. It bounds the fraction that the small
    # tensors below can reach, whatever the streaming rate.
    x1 = inputs.gaussian_bf16((128, 128), 1.0, dev, 0, 99)
    o_r, o_t, o_d, o_w = (ops.quant_act_1x128(x1), ops.quant_act_1x128(x1, transposed=True),
                          ops.quant_act_1x128_dual(x1), ops.quant_w_128x128(x1))
    floor = {"events_only": timed(lambda: None, stream, iters, warm, flush),
             "quant_act_1x128": timed(lambda: ops.quant_act_1x128(x1, q=o_r[0], s=o_r[1]), stream, iters, warm,
                                      flush),
             "quant_act_1x128 transposed": timed(lambda: ops.quant_act_1x128(x1, True, o_t[0], o_t[1]), stream, iters,
                                                 warm, flush),
             "quant_act_1x128_dual": timed(lambda: ops.quant_act_1x128_dual(x1, out=o_d), stream, iters, warm, flush),
             "quant_w_128x128": timed(lambda: ops.quant_w_128x128(x1, q=o_w[0], s=o_w[1]), stream, iters, warm,
                                      flush)}
    out["launch floor: one 128x128 tile per call"] = {k: round(v * 1e3, 2) for k, v in floor.items()}
    out["launch floor: one 128x128 tile per call"]["unit"] = "us"
    del x1

    xq = inputs.quant_only(dev)
    nb = xq.numel() * 3 + xq.numel() // 128 * 4
    o_q = ops.quant_act_1x128(xq)
    t = timed(lambda: ops.quant_act_1x128(xq, q=o_q[0], s=o_q[1]), stream, iters, warm, flush)
    out["quant_act_1x128 [16384,7168]"] = {"bound": "hbm", "ms": round(t, 4), "GBps": round(nb / t / 1e6, 1),
                                          "frac": round(nb / t / 1e6 / hbm_peak, 4), "algorithmic_bytes": nb}
    del xq

    # delayed (history) scaling on the same tensor, and its accuracy contrast with online
    # 1x128 scaling when the data grow by 1.5x over the recorded maxima
    xq = inputs.quant_only(dev)
    hist = ops.new_amax_history(16, dev)
    amax0 = xq.abs().max().float()
    hist[:16] = amax0
    nb = xq.numel() * 3 + xq.numel() // 128 * 4

    # every run quantizes the same tensor, whose max |x| equals the recorded maxima, so the
    # history's maximum (hence the scale) stays the same from run to run without a reset
    o_q = ops.quant_act_1x128(xq)
    t = timed(lambda: ops.quant_act_delayed(xq, hist, q=o_q[0], s=o_q[1]), stream, iters, warm, flush)
    x2 = (xq.float() * 1.5).to(torch.bfloat16)
    qd, sd = ops.quant_act_delayed(x2, hist)
    qo, so = ops.quant_act_1x128(x2)
    ref = x2.float()

    def deq(q, sc):
        return q.view(torch.float8_e4m3fn).float() * sc.repeat_interleave(128, dim=1)
    err_d = ((deq(qd, sd) - ref).abs().sum() / ref.abs().sum()).item()
    err_o = ((deq(qo, so) - ref).abs().sum() / ref.abs().sum()).item()
    # values beyond 448 s are clipped to +-448 s (online scaling clips nothing by construction)
    clip_d = (ref.abs() > 448.0 * sd.repeat_interleave(128, dim=1)).float().mean().item()
    clip_o = (ref.abs() > 448.0 * so.repeat_interleave(128, dim=1)).float().mean().item()
    out["quant_act_delayed [16384,7168] H16"] = {
        "bound": "hbm", "ms": round(t, 4), "GBps": round(nb / t / 1e6, 1), "frac": round(nb / t / 1e6 / hbm_peak, 4),
        "algorithmic_bytes": nb,
        "contrast_x1.5_growth": {"rel_l1_err_delayed": round(err_d, 5), "rel_l1_err_online": round(err_o, 5),
                                 "clipped_frac_delayed": round(clip_d, 7), "clipped_frac_online": round(clip_o, 7)}}
    del xq, x2, qd, sd, qo, so, ref

    wg = inputs.wgrad(dev)
    for name, tsr in (("dY [4096,2048]", wg.dy), ("X [4096,7168]", wg.x)):
        nb = tsr.numel() * 3 + tsr.numel() // 128 * 4
        o_t = ops.quant_act_1x128(tsr, transposed=True)
        t = timed(lambda: ops.quant_act_1x128(tsr, True, o_t[0], o_t[1]), stream, iters, warm, flush)
        out[f"quant_act_1x128 transposed {name}"] = {"bound": "hbm", "ms": round(t, 4),
                                                     "GBps": round(nb / t / 1e6, 1),
                                                     "frac": round(nb / t / 1e6 / hbm_peak, 4),
                                                     "algorithmic_bytes": nb}
    # both operands of the weight-gradient GEMM in one launch
    nb = sum(t_.numel() * 3 + t_.numel() // 128 * 4 for t_ in (wg.dy, wg.x))
    o_p = ops.quant_act_1x128_transposed_pair(wg.dy, wg.x)
    t = timed(lambda: ops.quant_act_1x128_transposed_pair(wg.dy, wg.x, out=o_p), stream, iters, warm, flush)
    out["quant_act_1x128_transposed_pair dY [4096,2048] + X [4096,7168]"] = {
        "bound": "hbm", "ms": round(t, 4), "GBps": round(nb / t / 1e6, 1), "frac": round(nb / t / 1e6 / hbm_peak, 4),
        "algorithmic_bytes": nb}
    qdy, sdy, qxt, sxt = o_p
    fl = 2.0 * 2048 * 7168 * 4096
    cw = torch.empty((2048, 7168), dtype=torch.float32, device=dev)
    t = timed(lambda: ops.blockscaled_gemm(qdy, sdy, qxt, sxt, ops.SB_ROW_1x128, torch.float32, c=cw), stream, iters,
              warm, flush)
    t_sk = timed(lambda: ops.blockscaled_gemm(qdy, sdy, qxt, sxt, ops.SB_ROW_1x128, torch.float32, c=cw,
                                              workspace=gemm_ws), stream, iters, warm, flush)
    out["blockscaled_gemm wgrad 2048x7168x4096 f32"] = {"bound": "tensor", "ms": round(t, 4),
                                                        "TFLOPs": round(fl / t / 1e9, 1),
                                                        "frac": round(fl / t / 1e9 / fp8_peak, 4),
                                                        "stream_k": {"ms": round(t_sk, 4),
                                                                     "TFLOPs": round(fl / t_sk / 1e9, 1),
                                                                     "frac": round(fl / t_sk / 1e9 / fp8_peak, 4)}}
    ref = plain_fp8_gemm_check(dev, 2048, 7168, 4096, secs=0, flush=flush)
    out["blockscaled_gemm wgrad 2048x7168x4096 f32"]["plain_fp8_same_shape"] = {
        "kernel": ref["kernel"], "TFLOPs": ref["burst_tflops"], "ours_stream_k_over_it": round(fl / t_sk / 1e9 / ref["burst_tflops"], 4)}
    del wg, qdy, sdy, qxt, sxt

    # the dense projection with its output kept in FP8 (codes + 1x128 scales)
    d = inputs.dense(dev)
    qx, sx = ops.quant_act_1x128(d.x)
    qw, sw = ops.quant_w_128x128(d.w)
    del d
    cq = torch.empty((M, N), dtype=torch.uint8, device=dev)
    cs = torch.empty((M, N // 128), dtype=torch.float32, device=dev)
    t = timed(lambda: ops.blockscaled_gemm_e4m3(qx, sx, qw, sw, ops.SB_BLOCK_128x128, out=(cq, cs)), stream, iters,
              warm, flush)
    out["blockscaled_gemm dense 4096x18432x7168 e4m3 out"] = {"bound": "tensor", "ms": round(t, 4),
                                                              "TFLOPs": round(GEMM_FLOPS / t / 1e9, 1),
                                                              "frac": round(GEMM_FLOPS / t / 1e9 / fp8_peak, 4)}
    del qx, sx, qw, sw, cq, cs

    # both orientations of X from one read (fprop 1x128 along K + wgrad tiles along M)
    xd = inputs.dense(dev, N=128).x                                          # [4096, 7168]
    nb = xd.numel() * 4 + 2 * (xd.numel() // 128) * 4
    o_d = ops.quant_act_1x128_dual(xd)
    t = timed(lambda: ops.quant_act_1x128_dual(xd, out=o_d), stream, iters, warm, flush)
    t2 = timed(lambda: (ops.quant_act_1x128(xd, False, o_d[0], o_d[1]), ops.quant_act_1x128(xd, True, o_d[2], o_d[3])),
               stream, iters, warm,
               flush)
    out["quant_act_1x128_dual X [4096,7168]"] = {"bound": "hbm", "ms": round(t, 4), "GBps": round(nb / t / 1e6, 1),
                                                 "frac": round(nb / t / 1e6 / hbm_peak, 4), "algorithmic_bytes": nb,
                                                 "ms_two_single_calls": round(t2, 4)}
    del xd

    # dX = dY . W of the dense projection: W quantized once in both orientations
    dg = inputs.dgrad(dev)                                                   # dY [4096,18432], W [18432,7168]
    nb = dg.w.numel() * 4 + 2 * (dg.w.numel() // 16384) * 4
    o_w = ops.quant_w_128x128_dual(dg.w)
    t = timed(lambda: ops.quant_w_128x128_dual(dg.w, out=o_w), stream, iters, warm, flush)
    out["quant_w_128x128_dual W [18432,7168]"] = {"bound": "hbm", "ms": round(t, 4), "GBps": round(nb / t / 1e6, 1),
                                                  "frac": round(nb / t / 1e6 / hbm_peak, 4), "algorithmic_bytes": nb}
    qdy, sdy = ops.quant_act_1x128(dg.dy)
    _, _, qwt, swt = ops.quant_w_128x128_dual(dg.w)
    del dg
    dx = torch.empty((4096, 7168), dtype=torch.bfloat16, device=dev)
    fl = 2.0 * 4096 * 7168 * 18432
    t = timed(lambda: ops.blockscaled_gemm(qdy, sdy, qwt, swt, ops.SB_BLOCK_128x128, torch.bfloat16, c=dx), stream,
              iters, warm, flush)
    t_sk = timed(lambda: ops.blockscaled_gemm(qdy, sdy, qwt, swt, ops.SB_BLOCK_128x128, torch.bfloat16, c=dx,
                                              workspace=gemm_ws), stream, iters, warm, flush)
    out["blockscaled_gemm dgrad 4096x7168x18432 bf16"] = {"bound": "tensor", "ms": round(t, 4),
                                                          "TFLOPs": round(fl / t / 1e9, 1),
                                                          "frac": round(fl / t / 1e9 / fp8_peak, 4),
                                                          "stream_k": {"ms": round(t_sk, 4),
                                                                       "TFLOPs": round(fl / t_sk / 1e9, 1),
                                                                       "frac": round(fl / t_sk / 1e9 / fp8_peak, 4)}}
    ref = plain_fp8_gemm_check(dev, 4096, 7168, 18432, secs=0, flush=flush)
    out["blockscaled_gemm dgrad 4096x7168x18432 bf16"]["plain_fp8_same_shape"] = {
        "kernel": ref["kernel"], "TFLOPs": ref["burst_tflops"], "ours_stream_k_over_it": round(fl / t_sk / 1e9 / ref["burst_tflops"], 4)}
    del qdy, sdy, qwt, swt, dx

    m = inputs.moe(dev)
    E, Ni, Kh = m.w.shape
    qa, sa = ops.quant_act_1x128(m.a)
    wflat = m.w.view(E * Ni, Kh)
    nb = wflat.numel() * 3 + wflat.numel() // 16384 * 4
    o_w = ops.quant_w_128x128(wflat)
    t = timed(lambda: ops.quant_w_128x128(wflat, q=o_w[0], s=o_w[1]), stream, max(3, iters // 4), 1, flush)
    out["quant_w_128x128 moe [256x2048,7168]"] = {"bound": "hbm", "ms": round(t, 4), "GBps": round(nb / t / 1e6, 1),
                                                  "frac": round(nb / t / 1e6 / hbm_peak, 4), "algorithmic_bytes": nb}
    qw, sw = ops.quant_w_128x128(wflat)
    qw3, sw3 = qw.view(E, Ni, Kh), sw.view(E, Ni // 128, Kh // 128)
    mtot = m.a.shape[0]
    c = torch.empty((mtot, Ni), dtype=torch.bfloat16, device=dev)
    t = timed(lambda: ops.grouped_gemm(qa, sa, qw3, sw3, m.offsets, torch.bfloat16, c=c), stream, iters, warm, flush)
    nb = qw.numel() + sw.numel() * 4 + qa.numel() + sa.numel() * 4 + c.numel() * 2
    real_fl = 2.0 * m.real_rows * Ni * Kh
    pad_fl = 2.0 * mtot * Ni * Kh
    out["grouped_gemm moe 256 experts N2048 K7168 bf16"] = {
        "bound": "hbm", "ms": round(t, 4), "GBps": round(nb / t / 1e6, 1), "frac": round(nb / t / 1e6 / hbm_peak, 4),
        "algorithmic_bytes": nb, "TFLOPs_real_rows": round(real_fl / t / 1e9, 1),
        "TFLOPs_padded_rows": round(pad_fl / t / 1e9, 1), "real_rows": m.real_rows, "padded_rows": mtot}
    ops.sync_status()
    return out


# ----------------------------------------------------------------------------- oracle arm


def _host_cores():
    """The cores this process may run on (its CPU affinity set)."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def _openblas_threads(n):
    """Without threadpoolctl: the OpenBLAS library numpy loaded, found in this process's
    memory map and called through its exported thread-count functions. n=None reads the
    count; otherwise sets it to n and returns a function that restores the old count
    (None if no OpenBLAS was found)."""
    import ctypes
    paths = set()
    try:
        for line in open("/proc/self/maps"):
            part = line.split()[-1]
            if "openblas" in part and ".so" in part:
                paths.add(part)
    except OSError:
        return None
    for path in sorted(paths):
        lib = ctypes.CDLL(path)
        for prefix in ("scipy_openblas", "openblas"):
            for suffix in ("64_", ""):
                get = getattr(lib, f"{prefix}_get_num_threads{suffix}", None)
                put = getattr(lib, f"{prefix}_set_num_threads{suffix}", None)
                if get is None or put is None:
                    continue
                get.restype = ctypes.c_int
                put.argtypes = [ctypes.c_int]
                if n is None:
                    return int(get())
                old = int(get())
                put(int(n))
                return lambda: put(old)
    return None


class OracleThreads:
    """Runs the oracle on every host core: BLAS (the float64 GEMM) limited to exactly
    `n` threads through threadpoolctl, and the numpy quantizers applied to row blocks
    of the sample by `n` worker threads (numpy releases the GIL inside its array
    loops). The oracle's code is unchanged; only the work is divided. `blas_threads`
    reports what BLAS actually runs with inside the block."""

    def __init__(self, n):
        self.n = n
        self.blas_threads = None
        self._limits = None

    def __enter__(self):
        from concurrent.futures import ThreadPoolExecutor

        import numpy  # noqa: F401  (loads the BLAS library, so that it can be found and limited)
        try:
            from threadpoolctl import threadpool_info, threadpool_limits
        except ImportError:
            self._restore = _openblas_threads(self.n)
            self.blas_threads = _openblas_threads(None)
        else:
            limits = threadpool_limits(limits=self.n, user_api="blas")
            self._restore = limits.restore_original_limits
            info = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
            self.blas_threads = max(info) if info else None
        self.pool = ThreadPoolExecutor(self.n)
        return self

    def __exit__(self, *exc):
        self.pool.shutdown()
        if callable(self._restore):
            self._restore()

    def rows(self, fn, x, unit=128):
        """fn over row blocks of x (block boundaries on multiples of `unit` rows),
        results concatenated along the rows."""
        import numpy as np
        m = x.shape[0]
        step = max(unit, (m // self.n + unit - 1) // unit * unit)
        parts = list(self.pool.map(fn, [x[i:i + step] for i in range(0, m, step)]))
        return tuple(np.concatenate([p[j] for p in parts]) for j in range(len(parts[0])))


def oracle_sample_step(x_rows, w_rows, threads):
    """One oracle pass over a sample of the dense-projection step: 1x128 quantization
    of x_rows rows of X, 128x128 quantization of w_rows rows of W, and the float64 GEMM
    of those rows, on all host cores (see OracleThreads). Returns (seconds, GEMM FLOPs
    of the sample)."""
    import numpy as np
    from fp8_fine_grained_cast_b300 import inputs
    from oracle import fp8_oracle as O

    d = inputs.dense("cpu", M=x_rows, N=w_rows)
    xh = d.x.float().numpy()
    wh = d.w.float().numpy()
    t0 = time.perf_counter()
    qx, sx = threads.rows(O.quant_act_1x128, xh, unit=1)       # 1x128 tiles: any row split
    qw, sw = threads.rows(O.quant_w_128x128, wh)                # 128x128 blocks: whole row blocks
    c = O.blockscaled_gemm(qx, sx, qw, sw)
    dt = time.perf_counter() - t0
    assert np.isfinite(c).all()
    return dt, 2.0 * x_rows * w_rows * K


def oracle_quantize_rate(rows, threads):
    """GB/s of the oracle's 1x128 quantizer (algorithmic bytes: 2 read + 1 written per
    element + 4 per 128-element scale) on the first `rows` rows of the quantize-only
    workload [16384, 7168], on all host cores."""
    from fp8_fine_grained_cast_b300 import inputs
    from oracle import fp8_oracle as O
    x = inputs.quant_only("cpu", rows=rows).float().numpy()
    t0 = time.perf_counter()
    threads.rows(O.quant_act_1x128, x, unit=1)
    dt = time.perf_counter() - t0
    nb = x.size * 3 + x.size // 128 * 4
    return nb / dt / 1e9, dt


def cpu_baseline(x_rows, w_rows, q_rows):
    n = _host_cores()
    with OracleThreads(n) as th:
        dt, fl = oracle_sample_step(x_rows, w_rows, th)
        q_gbps, q_dt = oracle_quantize_rate(q_rows, th)
        blas = th.blas_threads
    return {"value": round(fl / dt / 1e12, 6), "unit": "TFLOP/s", "cores": n, "kind": "oracle",
            "quantize_GBps": round(q_gbps, 3),
            "sample": (f"X[:{x_rows}] 1x128 + W[:{w_rows}] 128x128 quantization and their float64 GEMM of the "
                       f"dense projection: {dt:.2f} s for {fl:.3e} FLOP; quantize_GBps: 1x128 quantization of "
                       f"rows [:{q_rows}] of the quantize-only tensor [16384,7168], {q_dt:.2f} s. "
                       f"{n} threads (the process's CPU affinity set), BLAS limited to {blas} threads")}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    cores = _host_cores()
    times = []
    fl = 0.0
    with OracleThreads(cores) as th:
        for _ in range(args.warmup):
            oracle_sample_step(args.ref_rows, args.ref_wrows, th)
        for _ in range(args.steps):
            dt, fl = oracle_sample_step(args.ref_rows, args.ref_wrows, th)
            times.append(dt)
    sec = sum(times) / len(times)
    value = fl / sec / 1e12
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(sec * 1e3, 1), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64 (oracle)", "data": "synthetic",
        "config": {"workload": WORKLOAD, "M": M, "N": N, "K": K},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": (f"per step X[:{args.ref_rows}] and W[:{args.ref_wrows}] of the workload, "
                                    f"{cores} threads (the process's CPU affinity set)")},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# ----------------------------------------------------------------------------- single-kernel cases


def run_case(args):
    """One kernel on its workload, `--iters` launches after 3 warm-up launches, for
    profiling (ncu -k) and quick timing. Prints one JSON line with the mean time.
    The MoE case uses 64 experts and 1024 tokens so that a profiler capture holds a few
    GB at most (the full MoE workload holds about 12 GB)."""
    import torch
    from fp8_fine_grained_cast_b300 import inputs, ops

    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream()
    case = args.case
    ws = ops.gemm_workspace(dev) if args.sk else None     # stream-K schedule for the dense GEMMs
    if case == "qrow":
        x = inputs.quant_only(dev)
        fn = lambda: ops.quant_act_1x128(x)
        work = {"bytes": x.numel() * 3 + x.numel() // 128 * 4}
    elif case == "qcol":
        x = inputs.wgrad(dev).x
        fn = lambda: ops.quant_act_1x128(x, transposed=True)
        work = {"bytes": x.numel() * 3 + x.numel() // 128 * 4}
    elif case == "qcolpair":
        wg = inputs.wgrad(dev)
        o_p = ops.quant_act_1x128_transposed_pair(wg.dy, wg.x)
        fn = lambda: ops.quant_act_1x128_transposed_pair(wg.dy, wg.x, out=o_p)
        work = {"bytes": sum(t_.numel() * 3 + t_.numel() // 128 * 4 for t_ in (wg.dy, wg.x))}
    elif case == "qw":
        w = inputs.dense(dev, M=128).w
        fn = lambda: ops.quant_w_128x128(w)
        work = {"bytes": w.numel() * 3 + w.numel() // 16384 * 4}
    elif case == "gemm":
        d = inputs.dense(dev)
        qx, sx = ops.quant_act_1x128(d.x)
        qw, sw = ops.quant_w_128x128(d.w)
        del d
        c = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        fn = lambda: ops.blockscaled_gemm(qx, sx, qw, sw, ops.SB_BLOCK_128x128, torch.bfloat16, c=c, workspace=ws)
        work = {"flops": GEMM_FLOPS}
    elif case == "wgrad":
        wg = inputs.wgrad(dev)
        a, sa = ops.quant_act_1x128(wg.dy, transposed=True)
        b, sb = ops.quant_act_1x128(wg.x, transposed=True)
        del wg
        cw = torch.empty((2048, 7168), dtype=torch.float32, device=dev)
        fn = lambda: ops.blockscaled_gemm(a, sa, b, sb, ops.SB_ROW_1x128, torch.float32, c=cw, workspace=ws)
        work = {"flops": 2.0 * 2048 * 7168 * 4096}
    elif case == "gemm_e4m3":
        d = inputs.dense(dev)
        qx, sx = ops.quant_act_1x128(d.x)
        qw, sw = ops.quant_w_128x128(d.w)
        del d
        cq = torch.empty((M, N), dtype=torch.uint8, device=dev)
        cs = torch.empty((M, N // 128), dtype=torch.float32, device=dev)
        fn = lambda: ops.blockscaled_gemm_e4m3(qx, sx, qw, sw, ops.SB_BLOCK_128x128, out=(cq, cs))
        work = {"flops": GEMM_FLOPS}
    elif case == "qdelayed":
        x = inputs.quant_only(dev)
        hist = ops.new_amax_history(16, dev)
        hist[:16] = x.abs().max().float()
        fn = lambda: ops.quant_act_delayed(x, hist)
        work = {"bytes": x.numel() * 3 + x.numel() // 128 * 4}
    elif case == "qdual":
        x = inputs.dense(dev, N=128).x
        fn = lambda: ops.quant_act_1x128_dual(x)
        work = {"bytes": x.numel() * 4 + 2 * (x.numel() // 128) * 4}
    elif case == "wdual":
        w = inputs.dense(dev, M=128).w
        fn = lambda: ops.quant_w_128x128_dual(w)
        work = {"bytes": w.numel() * 4 + 2 * (w.numel() // 16384) * 4}
    elif case == "dgrad":
        dg = inputs.dgrad(dev)
        a, sa = ops.quant_act_1x128(dg.dy)
        _, _, b, sb = ops.quant_w_128x128_dual(dg.w)
        del dg
        c = torch.empty((4096, 7168), dtype=torch.bfloat16, device=dev)
        fn = lambda: ops.blockscaled_gemm(a, sa, b, sb, ops.SB_BLOCK_128x128, torch.bfloat16, c=c, workspace=ws)
        work = {"flops": 2.0 * 4096 * 7168 * 18432}
    elif case == "grouped":
        m = inputs.moe(dev, tokens=1024, experts=64)
        E, Ni, Kh = m.w.shape
        qa, sa = ops.quant_act_1x128(m.a)
        qw, sw = ops.quant_w_128x128(m.w.view(E * Ni, Kh))
        off = m.offsets
        del m
        qw3, sw3 = qw.view(E, Ni, Kh), sw.view(E, Ni // 128, Kh // 128)
        c = torch.empty((qa.shape[0], Ni), dtype=torch.bfloat16, device=dev)
        fn = lambda: ops.grouped_gemm(qa, sa, qw3, sw3, off, torch.bfloat16, c=c)
        work = {"bytes": qw.numel() + sw.numel() * 4 + qa.numel() + sa.numel() * 4 + c.numel() * 2}
    else:
        raise SystemExit(f"unknown case {case}")
    torch.cuda.empty_cache()
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    t = timed(fn, stream, args.iters, 3, flush)
    ops.sync_status()
    out = {"case": case, "stream_k": bool(args.sk), "iters": args.iters, "ms": round(t, 4)}
    if "bytes" in work:
        out["GBps"] = round(work["bytes"] / t / 1e6, 1)
    if "flops" in work:
        out["TFLOPs"] = round(work["flops"] / t / 1e9, 1)
    print(json.dumps(out), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-rows", action="store_true", help="skip the per-kernel rows")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-sample-rows", type=int, default=1024)
    ap.add_argument("--cpu-sample-wrows", type=int, default=4608)
    ap.add_argument("--cpu-sample-qrows", type=int, default=4096)
    ap.add_argument("--ref-rows", type=int, default=256)
    ap.add_argument("--ref-wrows", type=int, default=2048)
    ap.add_argument("--case", choices=["qrow", "qcol", "qcolpair", "qw", "gemm", "wgrad", "grouped", "qdual", "wdual", "dgrad", "gemm_e4m3", "qdelayed"],
                    help="time one kernel on its workload instead of the step (for profiling)")
    ap.add_argument("--iters", type=int, default=3)
    ap.add_argument("--sk", action="store_true", help="--case gemm/wgrad/dgrad: the stream-K schedule")
    args = ap.parse_args()
    if args.case:
        run_case(args)
        return
    args.warmup = max(3, args.warmup)      # at least three untimed warm-up steps
    args.steps = max(1, args.steps)
    rank, world, local = dist_setup()
    if args.impl == "reference":
        line = run_reference(args, rank, world)
    else:
        line = run_ours(args, rank, world, local)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
