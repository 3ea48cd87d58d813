// Block-scaled FP8 GEMM (dense and grouped) for sm_103a: TMA -> shared memory ->
// tcgen05.mma (E4M3 x E4M3 -> FP32 in TMEM) per 128-deep K chunk, with the chunk's
// partial sum promoted into FP32 registers with the product of its two scales
// ("Advantages of using FP8 for GEMM operations in DeepSeek-V3", item 5: partial sums
// promoted to FP32 at fixed intervals; item 8: dense and MoE GEMMs).
//
// C = A . B^T, A [M][K] E4M3 with scales sa[M][K/128]; B [N][K] E4M3 with scales per
// 128x128 block (sb[N/128][K/128]) or per 1x128 tile (sb[N][K/128]).
//
// Kernel structure (one persistent CTA per SM, three warpgroups = 12 warps):
//   warp 0     TMA producer: per K chunk, the A tile (128 x 128 B) and the B tile
//              (BN x 128 B), 128-byte swizzled, into a STAGES-deep ring.
//   warp 1     TMEM owner and MMA issuer: per chunk, 4 x tcgen05.mma (K = 32 each) into
//              one of two TMEM accumulators (BN columns each), the first with the
//              accumulate flag cleared, so that each accumulator holds exactly one
//              chunk's partial sum P[m][n] = sum_{k in chunk} qa[m][k] qb[n][k]; one
//              commit per chunk tells both the producer (stage free) and the
//              promotion warps (accumulator complete).
//   warps 2-3  scale loaders: per chunk, the 128 row scales of A and the column (or
//              column-block) scales of B into a shared-memory ring, alternate groups of
//              chunks per warp
//   warps 4-11 promotion and epilogue: two warpgroups; warpgroup g owns columns
//              [g BN/2, (g+1) BN/2) of the tile and warp (w % 4) owns TMEM lanes (rows)
//              32 (w % 4) .. +31. Per chunk: tcgen05.ld the partial sums in rounds of 32
//              columns (the next round's load issued before this round's arithmetic),
//              release the accumulator once the last round has arrived, and
//              C_acc += P * (sa[m][kb] * sb(n, kb)) in FP32 registers. While they
//              promote chunk kb the tensor cores already
//              compute chunk kb+1 into the other accumulator. After the last chunk the
//              accumulators are rounded to the output type, transposed through a small
//              swizzled shared-memory buffer per warp and written with coalesced 16-byte
//              stores (the TMA unit stays free for the operand loads). The output can
//              also be E4M3 codes with 1x128 scales: each promotion thread holds exactly
//              one 1x128 tile of C.
// Schedules: data-parallel (CTA c takes tiles c, c + G, ...) or, with a workspace,
// stream-K for a partial last wave (see Schedule below), as separate instantiations.
// Every mbarrier wait is bounded (about one second); a wait that runs out raises a
// CTA-wide abort flag and records a timeout in the device status word, every role
// leaves its loop, in-flight copies and MMAs are drained (bounded) and TMEM is freed.
#include <cuda_bf16.h>

#include <atomic>

#include "common.cuh"
#include "e4m3.cuh"
#include "gemm_sched.cuh"
#include "internal.h"

namespace fp8fg {

// Status word of the GEMM kernels, one per device; read and cleared by fp8fg_sync_status.
__device__ unsigned int g_gemm_status = 0;

__device__ __forceinline__ void record_status(unsigned bits) { atomicOr(&g_gemm_status, bits); }

__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
  return mbar_wait(bar, parity, abort_flag, &g_gemm_status);
}

namespace {

constexpr int kBM = 128;
constexpr int kBK = 128;
constexpr int kFirstPromoWarp = 4;
constexpr int kStagingPerWarp = 4096;

// Layout by tile width BN. Warpgroup 0 holds the TMA producer, the MMA issuer and the two
// scale loaders; two promotion warpgroups follow, each owning kCols = BN / 2 columns.
// Register split: the block is launched with kLaunchRegs per thread (384 threads x 168 =
// 64512); warpgroup 0 then drops to 40 and the promotion warpgroups rise to 232, which
// sums to the same 4 x 32 x 40 + 8 x 32 x 232 = 64512. Per SM sub-partition the lanes of
// its three warps get 40 + 232 + 232 = 504 registers, within its 16K register file.
// (A three-warpgroup layout with 192-column tiles, one TMEM round trip per chunk and
// warp, measured slower on the dense workload and is not built.)
template <int BN>
struct WarpLayout {
  static_assert(BN == 128 || BN == 256, "tile width");
  static constexpr int kPWG = 2;
  static constexpr int kCols = BN / kPWG;
  static constexpr int kPromoWarps = 4 * kPWG;
  static constexpr int kThreads = 128 * (1 + kPWG);
  static constexpr int kLaunchRegs = (65536 / kThreads) / 8 * 8;
  static constexpr uint32_t kRegsControl = 40;
  static constexpr uint32_t kRegsPromo = 232;
  static_assert(4 * 32 * kRegsControl + kPromoWarps * 32 * kRegsPromo <= kThreads * kLaunchRegs, "register split");
  // chunk accumulators in TMEM (512 columns): two of 256 columns or four of 128, so that
  // the MMA can run up to kNumAcc - 1 chunks ahead of the promotion warps
  static constexpr uint32_t kNumAcc = 512 / BN;
  static constexpr uint32_t kTmemBuf = BN;  // column stride of the chunk accumulators
  static constexpr uint32_t kTmemCols = kNumAcc * kTmemBuf;
};

template <int BN, int STAGES, int SB_KIND, int OUT, bool GROUPED>
struct GemmCfg : WarpLayout<BN> {
  using L = WarpLayout<BN>;
  static constexpr int kStageA = kBM * kBK;
  static constexpr int kStageB = BN * kBK;
  // scale ring: per chunk, sa for the tile's 128 rows and the B scales: one per column
  // (1x128 scales of B) or one per promotion warpgroup (128x128 scales of B; a
  // warpgroup's columns lie in a single 128-column block)
  static constexpr int kSlots = (BN == 256 && SB_KIND == 0 && STAGES >= 4) ? 4 : 8;  // 4: shared memory is full
  static constexpr int kGroup = kSlots / 2;  // chunks per scale-loader group (two groups in flight)
  static constexpr int kSbPerSlot = SB_KIND == 1 ? BN : 4;
  static constexpr int kSlotFloats = kBM + kSbPerSlot;
  static constexpr int kOffB = STAGES * kStageA;
  static constexpr int kOffStaging = kOffB + STAGES * kStageB;
  static constexpr int kOffRing = kOffStaging + L::kPromoWarps * kStagingPerWarp;
  static constexpr int kOffBar = kOffRing + kSlots * kSlotFloats * 4;
  // full[STAGES], done[STAGES], tmem_empty[kNumAcc], scale_full[kSlots],
  // scale_empty[kSlots], drain, head_written, tail_read
  static constexpr int kNumBars = 2 * STAGES + L::kNumAcc + 2 * kSlots + 3;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kOffWork = kOffMisc + 16;  // WorkDesc of this CTA
  static constexpr int kOffOffsets = kOffWork + 48;
  static size_t smem_bytes(int E) { return kOffOffsets + (GROUPED ? 4 * (3 * E + 2) : 0); }
  // epilogue box: 32 rows x 128 bytes of FP32 (OUT 0), BF16 (OUT 1) or E4M3 codes (OUT 2)
  static constexpr int kBoxCols = OUT == 0 ? 32 : OUT == 1 ? 64 : 128;
  static_assert(OUT != 2 || L::kCols == 128, "an E4M3 output row slice is one 1x128 tile");
  static_assert(L::kCols % kBoxCols == 0, "epilogue boxes");
};

// Scale-loader loop of loader warp `li` (0 or 1): groups of G chunks, alternate groups
// per warp; slot of chunk c is c % kSlots (kSlots >= 2 G). Requires KB % G == 0 and unit
// boundaries at multiples of G, so that a group never straddles two units.
template <int G, typename Cfg, bool GROUPED, int SB_KIND, bool SK, typename Coords>
__device__ __forceinline__ void load_scales_impl(int li, int lane, int KB, int M, int N, int num_tiles,
                                                 const Coords& tile_coords, const WorkDesc* wd,
                                                 const float* __restrict__ sa, const float* __restrict__ sb,
                                                 float* ring, uint64_t* sfull, uint64_t* sempty,
                                                 volatile int* abort_flag) {
  constexpr int kSlots = Cfg::kSlots;
  constexpr int BN = Cfg::kStageB / kBK;
  uint32_t it = 0;
  const int n_units = wd->n_units;
  for (int u = 0; u < n_units; ++u) {
    const Unit w = unit_get<SK>(wd, KB, u, static_cast<int>(blockIdx.x), static_cast<int>(gridDim.x));
    int m_blk, n_blk, e;
    tile_coords(w.tile, m_blk, n_blk, e);
    const int m0 = m_blk * kBM;
    const int n0 = n_blk * BN;
    const int64_t step32 = static_cast<int64_t>(32) * KB;  // 32 rows of a scale matrix
    const float* sa_col = sa + static_cast<int64_t>(m0 + lane) * KB;
    const float* sb_col =
        SB_KIND == 1 ? sb + static_cast<int64_t>(n0 + lane) * KB
                     : sb + (static_cast<int64_t>(GROUPED ? e * (N / kBM) : 0) + (n0 + lane * Cfg::kCols) / kBM) * KB;
    for (int kb0 = w.kb0; kb0 < w.kb1; kb0 += G, it += G) {
      if (static_cast<int>((it / G) & 1u) != li) continue;
      for (int g = 0; g < G; ++g) {
        const uint32_t c = it + g;
        if (!mbar_wait(&sempty[c % kSlots], ((c / kSlots) & 1u) ^ 1u, abort_flag)) return;
      }
#pragma unroll
      for (int i = 0; i < kBM / 32; ++i) {
        const int r = lane + 32 * i;
        Vec<G> x;
        x.load(sa_col + i * step32 + kb0, m0 + r < M);
#pragma unroll
        for (int g = 0; g < G; ++g) ring[((it + g) % kSlots) * Cfg::kSlotFloats + r] = x.v[g];
      }
      if constexpr (SB_KIND == 0) {
        if (lane < Cfg::kPWG) {  // the 128x128 block of promotion warpgroup `lane`'s columns
          Vec<G> x;
          x.load(sb_col + kb0, (n0 + lane * Cfg::kCols) / kBM < N / kBM);
#pragma unroll
          for (int g = 0; g < G; ++g) ring[((it + g) % kSlots) * Cfg::kSlotFloats + kBM + lane] = x.v[g];
        }
      } else {
#pragma unroll
        for (int i = 0; i < BN / 32; ++i) {
          Vec<G> x;
          x.load(sb_col + i * step32 + kb0, n0 + lane + 32 * i < N);
#pragma unroll
          for (int g = 0; g < G; ++g) ring[((it + g) % kSlots) * Cfg::kSlotFloats + kBM + lane + 32 * i] = x.v[g];
        }
      }
#pragma unroll
      for (int g = 0; g < G; ++g) mbar_arrive(&sfull[(it + g) % kSlots]);  // each lane its own writes
    }
  }
}

template <int BN, int STAGES, int SB_KIND, int OUT, bool GROUPED, bool SK>
__global__ void __launch_bounds__(WarpLayout<BN>::kThreads, 1)
    blockscaled_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                            void* __restrict__ c_out, float* __restrict__ c_scale, const float* __restrict__ sa,
                            const float* __restrict__ sb, const int32_t* __restrict__ offsets, int E, int M, int N,
                            int K, int num_m_tiles, int num_n_tiles, int m_group,
                            const __grid_constant__ Schedule sched,
                            float* __restrict__ ws_partial, int* __restrict__ ws_flags, int sk_epoch) {
  using Cfg = GemmCfg<BN, STAGES, SB_KIND, OUT, GROUPED>;
  constexpr int kSlots = Cfg::kSlots;
  constexpr int kPromoWarps = Cfg::kPromoWarps;
  constexpr int kGroup = Cfg::kGroup;
  // The dynamic shared window starts 1024-byte aligned (checked below); the swizzled
  // TMA tiles and the UMMA descriptors rely on it.
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::kOffBar);
  uint64_t* full = bars;
  // done[s]: the MMAs of the chunk in stage s have completed, so the stage may be refilled
  // and that chunk's accumulator read (one commit per chunk serves both)
  uint64_t* done = bars + STAGES;
  constexpr uint32_t kNumAcc = Cfg::kNumAcc;
  uint64_t* tempty = bars + 2 * STAGES;
  uint64_t* sfull = tempty + kNumAcc;
  uint64_t* sempty = sfull + kSlots;
  uint64_t* drain = sempty + kSlots;
  uint64_t* head_written = drain + 1;  // stream-K: the promotion threads' partial sums are stored
  uint64_t* tail_read = drain + 2;     // stream-K: the promotion threads have read the previous partial
  float* ring = reinterpret_cast<float*>(smem + Cfg::kOffRing);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Cfg::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Cfg::kOffMisc + 4);
  volatile int* bad_args = reinterpret_cast<volatile int*>(smem + Cfg::kOffMisc + 8);
  int32_t* s_off = reinterpret_cast<int32_t*>(smem + Cfg::kOffOffsets);
  WorkDesc* wd = reinterpret_cast<WorkDesc*>(smem + Cfg::kOffWork);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int KB = K / kBK;
  const int num_tiles = num_m_tiles * num_n_tiles;

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&done[i], 1);
    }
    for (uint32_t i = 0; i < kNumAcc; ++i) mbar_init(&tempty[i], kPromoWarps);
    for (int i = 0; i < kSlots; ++i) {
      mbar_init(&sfull[i], 32);
      mbar_init(&sempty[i], SB_KIND == 0 ? kPromoWarps : kPromoWarps * 32);
    }
    mbar_init(drain, 1);
    mbar_init(head_written, kPromoWarps * 32);
    mbar_init(tail_read, kPromoWarps * 32);
    work_desc_init(sched, num_tiles, KB, static_cast<int>(blockIdx.x), static_cast<int>(gridDim.x), wd);
    *abort_flag = 0;
    *bad_args = (smem_u32(smem) & 1023u) != 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, Cfg::kTmemCols);
    tmem_relinquish();
  }
  if constexpr (GROUPED) {
    for (int i = threadIdx.x; i <= E; i += blockDim.x) s_off[i] = offsets[i];
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if constexpr (GROUPED) {
    if (threadIdx.x == 0) {
      bool ok = s_off[0] == 0 && s_off[E] == M;
      for (int i = 0; ok && i < E; ++i) ok = (s_off[i + 1] >= s_off[i]) && (s_off[i + 1] % kBM == 0);
      if (!ok) {
        *bad_args = 1;
        if (blockIdx.x == 0) record_status(kStatusBadOffsets);
      }
    }
    __syncthreads();
  }
  // grouped: row tiles in an order that alternates between the largest and the smallest
  // experts (s_sorted: experts by size, descending, by an O(E^2) rank count for E <= 512,
  // else in index order; s_cum: their row-tile prefix sums)
  int32_t* s_sorted = s_off + E + 1;
  int32_t* s_cum = s_sorted + E;
  if constexpr (GROUPED) {
    if (E <= 512) {
      for (int i = threadIdx.x; i < E; i += blockDim.x) {
        const int si = s_off[i + 1] - s_off[i];
        int rank = 0;
        for (int j = 0; j < E; ++j) {
          const int sj = s_off[j + 1] - s_off[j];
          rank += (sj > si) || (sj == si && j < i);
        }
        s_sorted[rank] = i;
      }
    } else {
      for (int i = threadIdx.x; i < E; i += blockDim.x) s_sorted[i] = i;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      s_cum[0] = 0;
      for (int q = 0; q < E; ++q) s_cum[q + 1] = s_cum[q] + (s_off[s_sorted[q] + 1] - s_off[s_sorted[q]]) / kBM;
    }
    __syncthreads();
  }
  const uint32_t tmem_base = *tmem_slot;
  const bool run = !*bad_args;

  // tile t -> (m block, n block, expert). Dense: groups of m_group row blocks, the rows of
  // a group fastest, so that the CTAs working at the same time share B tiles and the
  // group's band of A (m_group x 128 rows x K bytes, kept within about 40 MB by the host)
  // stays in L2 while the group's column tiles stream past; when all of A fits in that
  // budget the group is all of M (m fastest). Grouped: n fastest, so that
  // consecutive tiles share an expert's rows and concurrent tiles share its weights; the
  // row tiles themselves alternate between the largest and the smallest experts, so that
  // weight streaming (small experts) and tensor work (large experts reusing their weights
  // from L2) overlap across the SMs instead of coming in separate phases.
  auto tile_coords = [&](int t, int& m_blk, int& n_blk, int& e) {
    if constexpr (GROUPED) {
      n_blk = t % num_n_tiles;
      const int pos = t / num_n_tiles;
      // alternate: even positions from the front of the size-sorted row tiles, odd from the back
      const int a = (pos & 1) ? num_m_tiles - 1 - (pos >> 1) : (pos >> 1);
      int lo = 0, hi = E - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_cum[mid] <= a) lo = mid; else hi = mid - 1;
      }
      e = s_sorted[lo];
      m_blk = s_off[e] / kBM + (a - s_cum[lo]);
    } else {
      const int span = m_group * num_n_tiles;
      const int grp = t / span;
      const int in = t - grp * span;
      const int m_first = grp * m_group;
      const int gm = min(m_group, num_m_tiles - m_first);
      m_blk = m_first + in % gm;
      n_blk = in / gm;
      e = 0;
    }
  };

  if (warp < kFirstPromoWarp) {
    regs_decrease<Cfg::kRegsControl>();
    if (warp == 0) {
      // ---------------------------------------------------------- TMA producer
      if (lane == 0 && run) {
        tma_prefetch_map(&tmA);
        tma_prefetch_map(&tmB);
        uint32_t it = 0;
        bool ok = true;
        for (int u = 0; ok && u < wd->n_units; ++u) {
          const Unit w = unit_get<SK>(wd, KB, u, static_cast<int>(blockIdx.x), static_cast<int>(gridDim.x));
          int m_blk, n_blk, e;
          tile_coords(w.tile, m_blk, n_blk, e);
          const int a_row = m_blk * kBM;
          const int b_row = (GROUPED ? e * N : 0) + n_blk * BN;
          for (int kb = w.kb0; kb < w.kb1; ++kb) {
            const uint32_t st = it % STAGES;
            if (!mbar_wait(&done[st], ((it / STAGES) & 1u) ^ 1u, abort_flag)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&full[st], Cfg::kStageA + Cfg::kStageB);
            tma_load_2d(smem + st * Cfg::kStageA, &tmA, &full[st], kb * kBK, a_row);
            tma_load_2d(smem + Cfg::kOffB + st * Cfg::kStageB, &tmB, &full[st], kb * kBK, b_row);
            ++it;
          }
        }
        if (!ok) {  // let the loads still in flight land before the CTA can exit
          for (uint32_t j = it > STAGES ? it - STAGES : 0; j < it; ++j) {
            mbar_wait_drain(&full[j % STAGES], (j / STAGES) & 1u);
          }
        }
      }
    } else if (warp == 1) {
      // ---------------------------------------------------------- MMA issuer
      if (lane == 0 && run) {
        constexpr uint32_t idesc = idesc_e4m3_f32(kBM, BN);
        uint32_t it = 0;
        bool ok = true;
        for (int u = 0; ok && u < wd->n_units; ++u) {
          const Unit w = unit_get<SK>(wd, KB, u, static_cast<int>(blockIdx.x), static_cast<int>(gridDim.x));
          for (int kb = w.kb0; kb < w.kb1; ++kb) {
            const uint32_t st = it % STAGES;
            const uint32_t buf = it % kNumAcc;
            if (!mbar_wait(&full[st], (it / STAGES) & 1u, abort_flag) ||
                !mbar_wait(&tempty[buf], ((it / kNumAcc) & 1u) ^ 1u, abort_flag)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t d = tmem_base + buf * Cfg::kTmemBuf;
            const uint64_t a0 = sdesc_kmajor_sw128(smem_u32(smem + st * Cfg::kStageA));
            const uint64_t b0 = sdesc_kmajor_sw128(smem_u32(smem + Cfg::kOffB + st * Cfg::kStageB));
#pragma unroll
            for (int k = 0; k < kBK / 32; ++k) {
              // advance 32 bytes (= 32 E4M3 values) along K inside the swizzle atom
              mma_f8f6f4(d, a0 + 2u * k, b0 + 2u * k, idesc, k > 0 ? 1u : 0u);
            }
            mma_commit(&done[st]);
            ++it;
          }
        }
        mma_commit(drain);
        mbar_wait_drain(drain, 0);
      }
      __syncwarp();
    } else if (run) {
      // ---------------------------------------------------------- scale loaders
      // Warps 2 and 3 fill the scale ring ahead of the promotion warps, so that no
      // global load sits on their critical path: per chunk, sa[m0 .. m0+127][kb] and the
      // B scales of the tile's columns (1x128) or column blocks (128x128). Chunks go in
      // groups of kGroup, fetched with one vector load per scale row; the two warps take
      // alternate groups, so two groups of loads are in flight while the promotion warps
      // consume a third.
      const int li = warp - 2;
      if (KB % kGroup == 0) {
        load_scales_impl<kGroup, Cfg, GROUPED, SB_KIND, SK>(li, lane, KB, M, N, num_tiles, tile_coords, wd, sa, sb, ring,
                                                        sfull, sempty, abort_flag);
      } else {
        load_scales_impl<1, Cfg, GROUPED, SB_KIND, SK>(li, lane, KB, M, N, num_tiles, tile_coords, wd, sa, sb, ring, sfull,
                                                   sempty, abort_flag);
      }
    }
  } else {
    regs_increase<Cfg::kRegsPromo>();
    if (run) {
      // ---------------------------------------------------------- promotion + epilogue
      constexpr int kCols = Cfg::kCols;
      const int pw = warp - kFirstPromoWarp;
      const int g = pw >> 2;
      const int qd = warp & 3;
      const int row = 32 * qd + lane;
      uint8_t* stg = smem + Cfg::kOffStaging + pw * kStagingPerWarp;
      const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(32 * qd) << 16);
      // Stream-K partial sums of CTA c: float4 i of row r of warpgroup g's columns at
      // ((c * (BN / kCols) + g) * (kCols / 4) + i) * kBM + r, so that the 32 rows of a warp
      // move 512 contiguous bytes per instruction (a row-major tile would scatter each
      // instruction over 32 lines)
      auto partial_offset = [&](int cta, int grp, int r) -> size_t {
        return (static_cast<size_t>(cta) * (BN / kCols) + grp) * (kCols / 4) * kBM + r;
      };
      uint32_t it = 0;
      bool ok = true;
      for (int u = 0; ok && u < wd->n_units; ++u) {
        const Unit w = unit_get<SK>(wd, KB, u, static_cast<int>(blockIdx.x), static_cast<int>(gridDim.x));
        int m_blk, n_blk, e;
        tile_coords(w.tile, m_blk, n_blk, e);
        const int m0 = m_blk * kBM;
        const int col0 = n_blk * BN + g * kCols;

        // FP32 accumulators of this thread's row, in pairs for the packed FMAs: zero, plus
        // for the tail of a cut tile the head's partial sums (left by the previous CTA)
        float2 acc2[kCols / 2];
        float* acc = reinterpret_cast<float*>(acc2);
#pragma unroll
        for (int i = 0; i < kCols / 2; ++i) acc2[i] = make_float2(0.0f, 0.0f);
        if (w.kind == kTail) {
          // every promotion thread adds its row's part of the previous CTA's partial sums
          // (once that CTA's release flag holds this launch's epoch) to its zeroed
          // accumulators: exact, since sums that start from +0 are never -0; one thread
          // then clears the flag, after all have read. Each CTA has at most one tail
          // unit, so the barrier completes at most once (phase 0). (Loading the partial
          // into the accumulators directly made the compiler spill them.)
          ok = flag_wait(ws_flags + blockIdx.x - 1, sk_epoch, abort_flag, &g_gemm_status);
          if (ok) {
            const float4* src = reinterpret_cast<const float4*>(ws_partial) + partial_offset(blockIdx.x - 1, g, row);
#pragma unroll
            for (int i = 0; i < kCols / 4; ++i) {
              const float4 v = __ldcg(src + i * kBM);
              acc2[2 * i].x += v.x;
              acc2[2 * i].y += v.y;
              acc2[2 * i + 1].x += v.z;
              acc2[2 * i + 1].y += v.w;
            }
          }
          mbar_arrive(tail_read);
          if (threadIdx.x == kFirstPromoWarp * 32 && ok && mbar_wait(tail_read, 0, abort_flag)) {
            ws_flags[blockIdx.x - 1] = 0;
          }
          if (!ok) break;
        }

        for (int kb = w.kb0; kb < w.kb1; ++kb) {
          const uint32_t slot = it % kSlots;
          const uint32_t buf = it % kNumAcc;
          if (!mbar_wait(&sfull[slot], (it / kSlots) & 1u, abort_flag)) {
            ok = false;
            break;
          }
          const float* sa_s = ring + slot * Cfg::kSlotFloats;
          const float* sb_s = sa_s + kBM + g * kCols;
          const float sa_v = sa_s[row];
          float sc = 0.0f;
          if constexpr (SB_KIND == 0) {
            sc = sa_v * sa_s[kBM + g];
            // Both scales of this chunk are now in registers: release the slot. The
            // warp-wide reduction makes lane 0's arrive wait until every lane's scale
            // product (hence its two shared-memory reads) has completed.
            const uint32_t dep = __reduce_or_sync(0xFFFFFFFFu, __float_as_uint(sc));
            if (lane == 0) mbar_arrive_after(&sempty[slot], dep);
          }
          // the chunk's accumulator is complete: its stage's done barrier (the MMA warp
          // runs at most kNumAcc chunks ahead, fewer than STAGES, so no phase is skipped)
          if (!mbar_wait(&done[it % STAGES], (it / STAGES) & 1u, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t t_col = t_lane + buf * Cfg::kTmemBuf + g * kCols;
          // rounds of 32 columns with two register buffers: the load of round p + 1 is
          // issued before the arithmetic of round p, so that its latency overlaps it; the
          // accumulator goes back to the MMA warp once the last round's load has arrived
          const float2 sa2 = make_float2(sa_v, sa_v);
          const float2 sc2 = make_float2(sc, sc);
          uint32_t wa[32], wb[32];
          tmem_ld_32x32b_x32(t_col, wa);
#pragma unroll
          for (int p = 0; p < kCols / 32; ++p) {
            uint32_t(&cur)[32] = (p & 1) ? wb : wa;
            uint32_t(&nxt)[32] = (p & 1) ? wa : wb;
            tmem_wait_ld_tied(cur);
            if (p + 1 < kCols / 32) {
              tmem_ld_32x32b_x32(t_col + 32 * (p + 1), nxt);
            } else {  // this warp has read its whole chunk slice
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(&tempty[buf]);
            }
            float2* acp = acc2 + 16 * p;
            if constexpr (SB_KIND == 0) {
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                acp[j] = __ffma2_rn(make_float2(__uint_as_float(cur[2 * j]), __uint_as_float(cur[2 * j + 1])), sc2, acp[j]);
              }
            } else {
#pragma unroll
              for (int j = 0; j < 16; j += 2) {
                const float4 s4 = *reinterpret_cast<const float4*>(sb_s + 32 * p + 2 * j);
                const float2 t0 = __fmul2_rn(make_float2(s4.x, s4.y), sa2);
                const float2 t1 = __fmul2_rn(make_float2(s4.z, s4.w), sa2);
                acp[j] = __ffma2_rn(make_float2(__uint_as_float(cur[2 * j]), __uint_as_float(cur[2 * j + 1])), t0, acp[j]);
                acp[j + 1] = __ffma2_rn(make_float2(__uint_as_float(cur[2 * j + 2]), __uint_as_float(cur[2 * j + 3])), t1,
                                        acp[j + 1]);
              }
            }
          }
          if constexpr (SB_KIND == 1) {
            // each thread releases the scale slot once the values it read from it have
            // been used (its last accumulator depends on them)
            mbar_arrive_after(&sempty[slot], __float_as_uint(acc[kCols - 1]));
          }
          ++it;
        }
        if (w.kind == kHead) {
          // the head of a cut tile: leave the partial sums in slot blockIdx.x; once every
          // promotion thread has stored its part (at most one head unit per CTA: phase 0),
          // one thread releases them to the CTA that computes the tail. The arrive (release,
          // CTA scope) and that thread's wait (acquire, CTA scope) order every thread's
          // stores before its GPU-scope fence and release store, so only that thread waits
          // for the stores to become visible and the others go on with their next unit.
          // A thread that has given up still arrives, so the waiter never waits for it; no
          // flag is set then.
          if (ok) {
            float4* dst = reinterpret_cast<float4*>(ws_partial) + partial_offset(blockIdx.x, g, row);
#pragma unroll
            for (int i = 0; i < kCols / 4; ++i) {
              __stcg(dst + i * kBM, make_float4(acc2[2 * i].x, acc2[2 * i].y, acc2[2 * i + 1].x, acc2[2 * i + 1].y));
            }
          }
          mbar_arrive(head_written);
          if (threadIdx.x == kFirstPromoWarp * 32 && ok && mbar_wait(head_written, 0, abort_flag) && !*abort_flag) {
            __threadfence();
            asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(ws_flags + blockIdx.x), "r"(sk_epoch) : "memory");
          }
          if (!ok) break;
          continue;
        }
        if (!ok) break;

        // ------------------------------------------------------ epilogue
        // Per box of 32 rows x 128 bytes: each lane writes its row into the warp's
        // staging buffer (16-byte chunk c of row r at chunk position c ^ (r % 8), so
        // that both the row-wise writes and the column-wise reads below hit all 32
        // banks), then the warp reads it back four rows per instruction and stores
        // four full 128-byte lines per instruction to C. The stores go through the
        // load/store path, not the TMA unit, which is busy with the operand loads.
        // E4M3 output (OUT 2): this thread's 128 columns of row m0 + row are one 1x128
        // tile of C, quantized like an activation tile (scale fl32(amax / 448), codes
        // E4M3(fl32(c / s))) straight from the FP32 accumulators.
        constexpr int kBoxCols = Cfg::kBoxCols;
        uint8_t* c_bytes = reinterpret_cast<uint8_t*>(c_out);
        constexpr int kEsize = OUT == 0 ? 4 : OUT == 1 ? 2 : 1;
        Scale osc;
        if constexpr (OUT == 2) {
          float am0 = 0.0f, am1 = 0.0f;
#pragma unroll
          for (int i = 0; i < kCols; i += 2) {
            am0 = fmaxf(am0, fabsf(acc[i]));
            am1 = fmaxf(am1, fabsf(acc[i + 1]));
          }
          osc = make_scale(fmaxf(am0, am1));
          if (col0 < N && m0 + row < M) c_scale[static_cast<int64_t>(m0 + row) * (N / 128) + col0 / 128] = osc.s;
        }
#pragma unroll
        for (int h = 0; h < kCols / kBoxCols; ++h) {
          const int box_col = col0 + h * kBoxCols;
          if (box_col >= N) break;
#pragma unroll
          for (int ch = 0; ch < 8; ++ch) {
            uint4 w;
            if constexpr (OUT == 2) {
              const float* a = acc + 16 * ch;
              w = make_uint4(quantize4(a[0], a[1], a[2], a[3], osc), quantize4(a[4], a[5], a[6], a[7], osc),
                             quantize4(a[8], a[9], a[10], a[11], osc), quantize4(a[12], a[13], a[14], a[15], osc));
            } else if constexpr (OUT == 1) {
              const float* a = acc + h * 64 + 8 * ch;
              w = make_uint4(pack_bf16x2(a[0], a[1]), pack_bf16x2(a[2], a[3]), pack_bf16x2(a[4], a[5]),
                             pack_bf16x2(a[6], a[7]));
            } else {
              const float* a = acc + h * 32 + 4 * ch;
              w = make_uint4(__float_as_uint(a[0]), __float_as_uint(a[1]), __float_as_uint(a[2]),
                             __float_as_uint(a[3]));
            }
            *reinterpret_cast<uint4*>(stg + lane * 128 + ((ch ^ (lane & 7)) << 4)) = w;
          }
          __syncwarp();
          const int ch = lane & 7;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int r = 4 * i + (lane >> 3);
            const uint4 w = *reinterpret_cast<const uint4*>(stg + r * 128 + ((ch ^ (r & 7)) << 4));
            const int64_t grow = static_cast<int64_t>(m0) + 32 * qd + r;
            if (grow < M) {
              *reinterpret_cast<uint4*>(c_bytes + (grow * N + box_col) * kEsize + ch * 16) = w;
            }
          }
          __syncwarp();
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, Cfg::kTmemCols);
  }
}

// ------------------------------------------------------------------ host side

// Stream-K workspace: one FP32 partial tile (128 x 256) per CTA, then one flag per CTA.
constexpr size_t kPartialTileBytes = static_cast<size_t>(kBM) * 256 * 4;
size_t gemm_partial_bytes(int ctas) { return static_cast<size_t>(ctas) * kPartialTileBytes; }

template <int BN, int STAGES, int SB_KIND, int OUT, bool GROUPED, bool SK = false>
LaunchResult run_gemm(const uint8_t* qa, const float* sa, const uint8_t* qb, const float* sb,
                      const int32_t* offsets, int E, int64_t M, int64_t N, int64_t K, int64_t b_rows, void* c,
                      float* c_scale, cudaStream_t stream, int sm_count, void* workspace = nullptr) {
  using Cfg = GemmCfg<BN, STAGES, SB_KIND, OUT, GROUPED>;
  auto kernel = blockscaled_gemm_kernel<BN, STAGES, SB_KIND, OUT, GROUPED, SK>;
  const size_t smem = Cfg::smem_bytes(E);
  cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (err != cudaSuccess) return {err, "cudaFuncSetAttribute(max dynamic shared memory)"};
  // The in-kernel register split assumes the block starts with kLaunchRegs per thread;
  // with fewer, the promotion warpgroups could never obtain their registers.
  cudaFuncAttributes fa;
  err = cudaFuncGetAttributes(&fa, kernel);
  if (err != cudaSuccess) return {err, "cudaFuncGetAttributes"};
  if (fa.numRegs != Cfg::kLaunchRegs) return {cudaErrorInvalidConfiguration, "register count of the GEMM kernel"};

  CUtensorMap tmA, tmB;
  if (!encode_2d(&tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, qa, K, M, K, kBK, kBM, true))
    return {cudaErrorInvalidValue, "cuTensorMapEncodeTiled(A)"};
  if (!encode_2d(&tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, qb, K, b_rows, K, kBK, BN, true))
    return {cudaErrorInvalidValue, "cuTensorMapEncodeTiled(B)"};

  const int num_m = static_cast<int>((M + kBM - 1) / kBM);
  const int num_n = static_cast<int>((N + BN - 1) / BN);
  // dense raster: row-block groups whose band of A stays within about 40 MB of L2
  const int64_t band = (int64_t(40) << 20) / (kBM * K);
  const int m_group = static_cast<int>(band < 1 ? 1 : band > num_m ? num_m : band);
  const int64_t tiles = static_cast<int64_t>(num_m) * num_n;
  const int grid = static_cast<int>(tiles < sm_count ? tiles : sm_count);
  Schedule sched{static_cast<int>(tiles), 0, 1, 0};
  float* ws_partial = nullptr;
  int* ws_flags = nullptr;
  int epoch = 0;
  const int KB = static_cast<int>(K / kBK);
  if (SK && workspace && tiles > grid && tiles % grid != 0) {
    // stream-K over the last one to two waves' worth of tiles (see Schedule)
    const int grp = KB % Cfg::kGroup == 0 ? Cfg::kGroup : 1;
    sched.dp_tiles = static_cast<int>((tiles / grid - 1) * grid);
    sched.sk_tiles = static_cast<int>(tiles) - sched.dp_tiles;
    sched.grp = grp;
    sched.sk_groups = static_cast<int64_t>(sched.sk_tiles) * KB / grp;
    ws_partial = static_cast<float*>(workspace);
    ws_flags = reinterpret_cast<int*>(static_cast<char*>(workspace) + gemm_partial_bytes(sm_count));
    epoch = next_streamk_epoch();
  }
  kernel<<<grid, Cfg::kThreads, smem, stream>>>(tmA, tmB, c, c_scale, sa, sb, offsets, E, static_cast<int>(M),
                                           static_cast<int>(N), static_cast<int>(K), num_m, num_n, m_group, sched,
                                           ws_partial, ws_flags, epoch);
  err = cudaGetLastError();
  if (err != cudaSuccess) return {err, "kernel launch"};
  return {cudaSuccess, nullptr};
}

}  // namespace

// Epoch of a stream-K launch: a head CTA releases its partial sums by writing the epoch
// into its flag, the tail CTA waits for exactly that value and then clears the flag.
// Distinct launches get distinct epochs (1 .. 2^31 - 1, cycling), so a flag left set
// by a launch whose tail gave up (a bounded wait that ran out) cannot release a later
// launch's tail early.
namespace {
std::atomic<uint32_t> g_streamk_epoch{0};
}  // namespace

int next_streamk_epoch() {
  return static_cast<int>(g_streamk_epoch.fetch_add(1, std::memory_order_relaxed) % 0x7FFFFFFFu) + 1;
}

// Library-owned stream-K workspace for fp8_blockscaled_gemm_sk_static: room for the
// partial tiles and flags of a device with up to kStaticScratchSms SMs (about 20 MB). One
// copy per device; calls that use it must not overlap.
constexpr int kStaticScratchSms = 160;
constexpr size_t kStaticScratchBytes =
    (static_cast<size_t>(kStaticScratchSms) * (kPartialTileBytes + sizeof(int)) + 255) / 256 * 256;
static __device__ __align__(256) uint8_t g_gemm_scratch[kStaticScratchBytes];

cudaError_t gemm_static_scratch(void** ptr, size_t* bytes) {
  *bytes = kStaticScratchBytes;
  return cudaGetSymbolAddress(ptr, g_gemm_scratch);
}

size_t gemm_workspace_bytes(int sm_count) {
  return (gemm_partial_bytes(sm_count) + static_cast<size_t>(sm_count) * sizeof(int) + 255) / 256 * 256;
}

LaunchResult launch_blockscaled_gemm(const uint8_t* qa, const float* sa, const uint8_t* qb, const float* sb,
                                     int sb_kind, void* c, float* c_scale, int c_kind, int64_t M, int64_t N,
                                     int64_t K, cudaStream_t stream, int sm_count, void* workspace) {
  // 128 x 256 tiles throughout: 128-column tiles (with two or with four TMEM
  // accumulators, on one CTA or on a CTA pair with cta_group::2 MMAs), tried for the
  // weight-gradient shape whose 256-column tiles leave a nearly empty last wave, measured
  // slower on every workload. The stream-K variants (with a workspace) are separate
  // instantiations, so that the data-parallel kernel carries none of their code.
  const bool sk = workspace != nullptr;
  if (sb_kind == 0) {
    if (c_kind == 2) return run_gemm<256, 4, 0, 2, false>(qa, sa, qb, sb, nullptr, 0, M, N, K, N, c, c_scale, stream, sm_count);
    if (c_kind == 1) {
      return sk ? run_gemm<256, 4, 0, 1, false, true>(qa, sa, qb, sb, nullptr, 0, M, N, K, N, c, nullptr, stream, sm_count, workspace)
                : run_gemm<256, 4, 0, 1, false>(qa, sa, qb, sb, nullptr, 0, M, N, K, N, c, nullptr, stream, sm_count);
    }
    return sk ? run_gemm<256, 4, 0, 0, false, true>(qa, sa, qb, sb, nullptr, 0, M, N, K, N, c, nullptr, stream, sm_count, workspace)
              : run_gemm<256, 4, 0, 0, false>(qa, sa, qb, sb, nullptr, 0, M, N, K, N, c, nullptr, stream, sm_count);
  }
  if (c_kind == 2) return run_gemm<256, 3, 1, 2, false>(qa, sa, qb, sb, nullptr, 0, M, N, K, N, c, c_scale, stream, sm_count);
  if (c_kind == 1) {
    return sk ? run_gemm<256, 3, 1, 1, false, true>(qa, sa, qb, sb, nullptr, 0, M, N, K, N, c, nullptr, stream, sm_count, workspace)
              : run_gemm<256, 3, 1, 1, false>(qa, sa, qb, sb, nullptr, 0, M, N, K, N, c, nullptr, stream, sm_count);
  }
  return sk ? run_gemm<256, 3, 1, 0, false, true>(qa, sa, qb, sb, nullptr, 0, M, N, K, N, c, nullptr, stream, sm_count, workspace)
            : run_gemm<256, 3, 1, 0, false>(qa, sa, qb, sb, nullptr, 0, M, N, K, N, c, nullptr, stream, sm_count);
}

LaunchResult launch_grouped_gemm(const uint8_t* qa, const float* sa, const uint8_t* qb, const float* sb,
                                 const int32_t* offsets, int E, int64_t Mtot, void* c, int c_bf16, int64_t N,
                                 int64_t K, cudaStream_t stream, int sm_count) {
  if (c_bf16)
    return run_gemm<256, 3, 0, 1, true>(qa, sa, qb, sb, offsets, E, Mtot, N, K, N * E, c, nullptr, stream, sm_count);
  return run_gemm<256, 3, 0, 0, true>(qa, sa, qb, sb, offsets, E, Mtot, N, K, N * E, c, nullptr, stream, sm_count);
}

namespace {

// One thread waits on a barrier that never completes; the bounded wait gives up after
// kWaitLimitNs and records kStatusTimeout in the GEMM status word.
__global__ void wait_timeout_selftest_kernel() {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) (void)mbar_wait(&bar, 0, &abort_flag);
}

}  // namespace

cudaError_t launch_wait_timeout_selftest(cudaStream_t stream) {
  wait_timeout_selftest_kernel<<<1, 32, 0, stream>>>();
  return cudaGetLastError();
}

cudaError_t read_and_clear_gemm_status(unsigned* out) {
  cudaError_t err = cudaMemcpyFromSymbol(out, g_gemm_status, sizeof(unsigned));
  if (err != cudaSuccess) return err;
  if (*out) {
    const unsigned zero = 0;
    err = cudaMemcpyToSymbol(g_gemm_status, &zero, sizeof(unsigned));
  }
  return err;
}

}  // namespace fp8fg
