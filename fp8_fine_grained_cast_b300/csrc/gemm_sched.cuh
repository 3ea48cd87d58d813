// Work schedule of the block-scaled GEMM kernels (gemm.cu): data-parallel tiles, and the
// stream-K split of a partial last wave with the hand-off of a cut tile's FP32 partial
// sums. Also small helpers of those kernels (vector scale loads, BF16 packing).
#pragma once

#include <cuda_bf16.h>

#include "common.cuh"

namespace fp8fg {
namespace {

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// G consecutive floats (16-, 8- or 4-byte aligned) or zeros.
template <int G>
struct Vec;
template <>
struct Vec<1> {
  float v[1];
  __device__ __forceinline__ void load(const float* p, bool ok) { v[0] = ok ? __ldg(p) : 0.0f; }
};
template <>
struct Vec<2> {
  float v[2];
  __device__ __forceinline__ void load(const float* p, bool ok) {
    const float2 t = ok ? __ldg(reinterpret_cast<const float2*>(p)) : make_float2(0.0f, 0.0f);
    v[0] = t.x;
    v[1] = t.y;
  }
};
template <>
struct Vec<4> {
  float v[4];
  __device__ __forceinline__ void load(const float* p, bool ok) {
    const float4 t = ok ? __ldg(reinterpret_cast<const float4*>(p)) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    v[0] = t.x;
    v[1] = t.y;
    v[2] = t.z;
    v[3] = t.w;
  }
};

// Work schedule of a launch over G workers (CTAs) c = 0 .. G-1.
// Data-parallel: worker c takes tiles c, c + G, ... Stream-K (sk_tiles > 0): the first
// dp_tiles tiles (a multiple of G) go data-parallel, and the chunks of the last sk_tiles
// tiles (G <= sk_tiles < 2G) are divided into G contiguous ranges of whole loader groups
// (grp chunks), one per worker, in (tile, chunk) order. A range is at least one tile
// long, so a tile is cut at most once: the worker whose range ends inside it computes
// its head and leaves the FP32 partial sums in its workspace slot with a release flag;
// the next worker, whose range starts there, computes the tail last, starting its
// accumulators from that partial. The chunk order of every element is unchanged, so the
// result is bit-identical to the data-parallel schedule.
struct Schedule {
  int dp_tiles;       // tiles scheduled data-parallel (all of them when sk_tiles == 0)
  int sk_tiles;       // tiles in the stream-K region, 0 for none
  int grp;            // chunks per loader group; range boundaries are multiples of it
  int64_t sk_groups;  // sk_tiles * KB / grp
};

enum UnitKind { kWhole = 0, kHead = 1, kTail = 2 };

struct Unit {
  int tile, kb0, kb1, kind;
};

// The units of worker c, in processing order: its head piece (so that the partial is
// ready early), whole stream-K tiles, data-parallel tiles, its tail piece (last, so that
// the previous worker's partial has long been written). One thread derives the
// description once into shared memory; the roles read it there, so that none keeps it
// (or the 64-bit arithmetic behind it) in registers.
struct WorkDesc {
  int n_units, n_head, head_tile, head_kb1, n_whole, whole0, n_dp, tail_tile, tail_kb0;
};

__device__ __forceinline__ void work_desc_init(const Schedule& s, int num_tiles, int KB, int c, int G, WorkDesc* wd) {
  WorkDesc d{};
  if (s.sk_tiles == 0) {
    d.n_dp = c < num_tiles ? (num_tiles - 1 - c) / G + 1 : 0;
  } else {
    const int64_t g0 = (static_cast<int64_t>(c) * s.sk_groups) / G * s.grp;
    const int64_t g1 = (static_cast<int64_t>(c + 1) * s.sk_groups) / G * s.grp;
    d.n_head = (g1 % KB) != 0;
    d.head_tile = s.dp_tiles + static_cast<int>(g1 / KB);
    d.head_kb1 = static_cast<int>(g1 % KB);
    d.whole0 = s.dp_tiles + static_cast<int>((g0 + KB - 1) / KB);
    d.n_whole = s.dp_tiles + static_cast<int>(g1 / KB) - d.whole0;
    d.n_dp = s.dp_tiles / G;
    d.tail_tile = s.dp_tiles + static_cast<int>(g0 / KB);
    d.tail_kb0 = static_cast<int>(g0 % KB);
    d.n_units = (g0 % KB) != 0;  // the tail, counted below
  }
  d.n_units += d.n_head + d.n_whole + d.n_dp;
  *wd = d;
}

template <bool SK>
__device__ __forceinline__ Unit unit_get(const WorkDesc* wd, int KB, int u, int c, int G) {
  if constexpr (!SK) return {c + u * G, 0, KB, kWhole};
  if (u < wd->n_head) return {wd->head_tile, 0, wd->head_kb1, kHead};
  u -= wd->n_head;
  if (u < wd->n_whole) return {wd->whole0 + u, 0, KB, kWhole};
  u -= wd->n_whole;
  if (u < wd->n_dp) return {c + u * G, 0, KB, kWhole};
  return {wd->tail_tile, wd->tail_kb0, KB, kTail};
}

// Bounded wait until a flag that another CTA sets with release semantics holds this
// launch's epoch; the same limit and abort protocol as the mbarrier waits. A value left
// by an earlier launch that gave up before its tail read it (another epoch) is ignored.
__device__ __forceinline__ bool flag_wait(const int* flag, int epoch, volatile int* abort_flag, unsigned* status) {
  const uint64_t t0 = global_timer_ns();
  for (;;) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(flag) : "memory");
    if (v == epoch) return true;
    if (*abort_flag) return false;
    if (global_timer_ns() - t0 > kWaitLimitNs) {
      atomicOr(status, kStatusTimeout);
      *abort_flag = 1;
      return false;
    }
  }
}

}  // namespace
}  // namespace fp8fg
