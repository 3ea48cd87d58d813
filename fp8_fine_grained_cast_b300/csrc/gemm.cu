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
//              chunk's partial sum P[m][n] = sum_{k in chunk} qa[m][k] qb[n][k].
//   warps 2-3  idle (they complete the first warpgroup, which gives its registers up)
//   warps 4-11 promotion and epilogue: two warpgroups; warpgroup g owns columns
//              [g BN/2, (g+1) BN/2) of the tile and warp (w % 4) owns TMEM lanes (rows)
//              32 (w % 4) .. +31. Per chunk: tcgen05.ld the partial sums, release the
//              accumulator to the MMA warp, then C_acc += P * (sa[m][kb] * sb(n, kb)) in
//              FP32 registers. While they promote chunk kb the tensor cores already
//              compute chunk kb+1 into the other accumulator. After the last chunk the
//              accumulators are rounded to the output type, staged in shared memory with
//              the 128-byte swizzle and written by TMA stores.
// Every mbarrier wait is bounded (about one second); a wait that runs out raises a
// CTA-wide abort flag and records a timeout in the device status word, every role
// leaves its loop, in-flight copies and MMAs are drained (bounded) and TMEM is freed.
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace fp8fg {

// One status word per device; read and cleared by fp8fg_sync_status.
__device__ unsigned int g_status = 0;

enum : unsigned {
  kStatusTimeout = 1u,
  kStatusBadOffsets = 2u,
};

__device__ __forceinline__ void record_status(unsigned bits) { atomicOr(&g_status, bits); }

// Bounded wait for the phase of `bar` with parity `parity`. Returns false if the
// CTA's abort flag is raised or the time limit runs out (then it raises the flag and
// records a timeout).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 0) {
      if (*abort_flag) return false;
      if (global_timer_ns() - t0 > kWaitLimitNs) {
        *abort_flag = 1;
        record_status(kStatusTimeout);
        return false;
      }
    }
  }
}

namespace {

constexpr int kBM = 128;
constexpr int kBK = 128;
constexpr int kThreads = 384;
constexpr int kPromoWarps = 8;
constexpr int kFirstPromoWarp = 4;
constexpr int kStagingPerWarp = 4096;
// Register split: the block is launched with kLaunchRegs per thread (384 x 168 =
// 64512); warpgroup 0 (TMA, MMA) drops to 56 and the two promotion warpgroups rise to
// 224, which sums to the same 4 x 32 x 56 + 8 x 32 x 224 = 64512. Per SM sub-partition
// that is 56 + 224 + 224 registers for its three warps' lanes, within its 16K file.
constexpr int kLaunchRegs = 168;
constexpr uint32_t kRegsControl = 56;
constexpr uint32_t kRegsPromo = 224;
static_assert(4 * 32 * kRegsControl + 8 * 32 * kRegsPromo <= kThreads * kLaunchRegs, "register split");

template <int BN, int STAGES, int SB_KIND, bool OUT_BF16, bool GROUPED>
struct GemmCfg {
  static_assert(BN == 128 || BN == 256, "tile width");
  static constexpr int kHalf = BN / 2;
  static constexpr uint32_t kTmemCols = 2 * BN;
  static constexpr int kStageA = kBM * kBK;
  static constexpr int kStageB = BN * kBK;
  static constexpr int kOffB = STAGES * kStageA;
  static constexpr int kOffStaging = kOffB + STAGES * kStageB;
  static constexpr int kOffSb = kOffStaging + kPromoWarps * kStagingPerWarp;
  static constexpr int kSbBytes = SB_KIND == 1 ? kPromoWarps * kHalf * 4 : 0;
  static constexpr int kOffBar = kOffSb + kSbBytes;
  // full[STAGES], empty[STAGES], tmem_full[2], tmem_empty[2], drain
  static constexpr int kNumBars = 2 * STAGES + 5;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kOffOffsets = kOffMisc + 16;
  static size_t smem_bytes(int E) { return 1024 + kOffOffsets + (GROUPED ? 4 * (E + 1) : 0); }
  // output box: 128 bytes of one row x 32 rows
  static constexpr int kBoxCols = OUT_BF16 ? 64 : 32;
};

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

template <int BN, int STAGES, int SB_KIND, bool OUT_BF16, bool GROUPED>
__global__ void __launch_bounds__(kThreads, 1)
    blockscaled_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                            const __grid_constant__ CUtensorMap tmC, const float* __restrict__ sa,
                            const float* __restrict__ sb, const int32_t* __restrict__ offsets, int E, int M, int N,
                            int K, int num_m_tiles, int num_n_tiles) {
  using Cfg = GemmCfg<BN, STAGES, SB_KIND, OUT_BF16, GROUPED>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::kOffBar);
  uint64_t* full = bars;
  uint64_t* empty = bars + STAGES;
  uint64_t* tfull = bars + 2 * STAGES;
  uint64_t* tempty = bars + 2 * STAGES + 2;
  uint64_t* drain = bars + 2 * STAGES + 4;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Cfg::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Cfg::kOffMisc + 4);
  volatile int* bad_args = reinterpret_cast<volatile int*>(smem + Cfg::kOffMisc + 8);
  int32_t* s_off = reinterpret_cast<int32_t*>(smem + Cfg::kOffOffsets);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int KB = K / kBK;
  const int num_tiles = num_m_tiles * num_n_tiles;

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], kPromoWarps);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    *bad_args = 0;
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
  const uint32_t tmem_base = *tmem_slot;
  const bool run = !*bad_args;

  // tile t -> (m block, n block, expert)
  auto tile_coords = [&](int t, int& m_blk, int& n_blk, int& e) {
    if constexpr (GROUPED) {
      n_blk = t % num_n_tiles;
      m_blk = t / num_n_tiles;
      const int m0 = m_blk * kBM;
      int lo = 0, hi = E - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_off[mid] <= m0) lo = mid; else hi = mid - 1;
      }
      e = lo;
    } else {
      m_blk = t % num_m_tiles;
      n_blk = t / num_m_tiles;
      e = 0;
    }
  };

  if (warp < kFirstPromoWarp) {
   regs_decrease<kRegsControl>();
   if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0 && run) {
      tma_prefetch_map(&tmA);
      tma_prefetch_map(&tmB);
      uint32_t it = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < num_tiles; t += gridDim.x) {
        int m_blk, n_blk, e;
        tile_coords(t, m_blk, n_blk, e);
        const int a_row = m_blk * kBM;
        const int b_row = (GROUPED ? e * N : 0) + n_blk * BN;
        for (int kb = 0; kb < KB; ++kb) {
          const uint32_t st = it % STAGES;
          const uint32_t use = it / STAGES;
          if (!mbar_wait(&empty[st], (use & 1u) ^ 1u, abort_flag)) {
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
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && run) {
      constexpr uint32_t idesc = idesc_e4m3_f32(kBM, BN);
      uint32_t it = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < num_tiles; t += gridDim.x) {
        for (int kb = 0; kb < KB; ++kb) {
          const uint32_t st = it % STAGES;
          const uint32_t use = it / STAGES;
          const uint32_t buf = it & 1u;
          const uint32_t buse = it >> 1;
          if (!mbar_wait(&full[st], use & 1u, abort_flag) ||
              !mbar_wait(&tempty[buf], (buse & 1u) ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d = tmem_base + buf * BN;
          const uint64_t a0 = sdesc_kmajor_sw128(smem_u32(smem + st * Cfg::kStageA));
          const uint64_t b0 = sdesc_kmajor_sw128(smem_u32(smem + Cfg::kOffB + st * Cfg::kStageB));
#pragma unroll
          for (int k = 0; k < kBK / 32; ++k) {
            // advance 32 bytes (= 32 E4M3 values) along K inside the swizzle atom
            mma_f8f6f4(d, a0 + 2u * k, b0 + 2u * k, idesc, k > 0 ? 1u : 0u);
          }
          mma_commit(&empty[st]);
          mma_commit(&tfull[buf]);
          ++it;
        }
      }
      mma_commit(drain);
      mbar_wait_drain(drain, 0);
    }
    __syncwarp();
   }
  } else {
   regs_increase<kRegsPromo>();
   if (run) {
    // ------------------------------------------------------------ promotion + epilogue
    constexpr int kHalf = Cfg::kHalf;
    const int pw = warp - kFirstPromoWarp;
    const int g = pw >> 2;
    const int qd = warp & 3;
    const int row = 32 * qd + lane;
    uint8_t* stg = smem + Cfg::kOffStaging + pw * kStagingPerWarp;
    float* sbs = reinterpret_cast<float*>(smem + Cfg::kOffSb) + pw * kHalf;
    const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(32 * qd) << 16);
    uint32_t it = 0;
    bool ok = true;
    for (int t = blockIdx.x; ok && t < num_tiles; t += gridDim.x) {
      int m_blk, n_blk, e;
      tile_coords(t, m_blk, n_blk, e);
      const int m0 = m_blk * kBM;
      const int col0 = n_blk * BN + g * kHalf;
      const int64_t grow = static_cast<int64_t>(m0) + row;
      const bool row_ok = grow < M;
      const float* sa_row = sa + grow * KB;
      const float* sb_blk = sb;
      bool sb_ok = col0 < N;
      if constexpr (SB_KIND == 0) {
        sb_blk = sb + (static_cast<int64_t>(GROUPED ? e * (N / kBM) : 0) + col0 / kBM) * KB;
      }

      float acc[kHalf];
#pragma unroll
      for (int i = 0; i < kHalf; ++i) acc[i] = 0.0f;

      for (int kb = 0; kb < KB; ++kb) {
        const float sa_v = row_ok ? __ldg(sa_row + kb) : 0.0f;
        float sb_v = 0.0f;
        if constexpr (SB_KIND == 0) {
          sb_v = sb_ok ? __ldg(sb_blk + kb) : 0.0f;
        } else {
          __syncwarp();
#pragma unroll
          for (int i = 0; i < kHalf / 32; ++i) {
            const int n = col0 + 32 * i + lane;
            sbs[32 * i + lane] = n < N ? __ldg(sb + static_cast<int64_t>(n) * KB + kb) : 0.0f;
          }
          __syncwarp();
        }
        const uint32_t buf = it & 1u;
        const uint32_t buse = it >> 1;
        if (!mbar_wait(&tfull[buf], buse & 1u, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const float sc = sa_v * sb_v;
#pragma unroll
        for (int c = 0; c < kHalf / 32; ++c) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(t_lane + buf * BN + g * kHalf + 32 * c, v);
          tmem_wait_ld();
          if (c == kHalf / 32 - 1) {  // all of this warp's reads of the accumulator are done
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[buf]);
          }
          if constexpr (SB_KIND == 0) {
#pragma unroll
            for (int j = 0; j < 32; ++j) acc[32 * c + j] = fmaf(__uint_as_float(v[j]), sc, acc[32 * c + j]);
          } else {
#pragma unroll
            for (int j4 = 0; j4 < 8; ++j4) {
              const float4 s4 = reinterpret_cast<const float4*>(sbs + 32 * c)[j4];
              acc[32 * c + 4 * j4 + 0] = fmaf(__uint_as_float(v[4 * j4 + 0]), sa_v * s4.x, acc[32 * c + 4 * j4 + 0]);
              acc[32 * c + 4 * j4 + 1] = fmaf(__uint_as_float(v[4 * j4 + 1]), sa_v * s4.y, acc[32 * c + 4 * j4 + 1]);
              acc[32 * c + 4 * j4 + 2] = fmaf(__uint_as_float(v[4 * j4 + 2]), sa_v * s4.z, acc[32 * c + 4 * j4 + 2]);
              acc[32 * c + 4 * j4 + 3] = fmaf(__uint_as_float(v[4 * j4 + 3]), sa_v * s4.w, acc[32 * c + 4 * j4 + 3]);
            }
          }
        }
        ++it;
      }
      if (!ok) break;

      // -------------------------------------------------------- epilogue
      constexpr int kBoxCols = Cfg::kBoxCols;
#pragma unroll
      for (int h = 0; h < kHalf / kBoxCols; ++h) {
        if (col0 + h * kBoxCols >= N) break;
        if (lane == 0) bulk_wait_group_read0();  // staging buffer free again
        __syncwarp();
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          uint4 w;
          if constexpr (OUT_BF16) {
            const float* a = acc + h * 64 + 8 * c;
            w = make_uint4(pack_bf16x2(a[0], a[1]), pack_bf16x2(a[2], a[3]), pack_bf16x2(a[4], a[5]),
                           pack_bf16x2(a[6], a[7]));
          } else {
            const float* a = acc + h * 32 + 4 * c;
            w = make_uint4(__float_as_uint(a[0]), __float_as_uint(a[1]), __float_as_uint(a[2]),
                           __float_as_uint(a[3]));
          }
          // 128-byte swizzle: 16-byte chunk c of row r sits at chunk position c ^ (r % 8)
          *reinterpret_cast<uint4*>(stg + lane * 128 + ((c ^ (lane & 7)) << 4)) = w;
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_2d(&tmC, stg, col0 + h * kBoxCols, m0 + 32 * qd);
          bulk_commit_group();
        }
      }
    }
    if (lane == 0) bulk_wait_group0();
    __syncwarp();
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

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess) {
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
  });
  return fn;
}

// 2D row-major tensor [rows][cols] with the given row pitch, box = box_cols x box_rows,
// 128-byte swizzle, out-of-range elements read as zero.
bool encode_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t cols, uint64_t rows,
               uint64_t row_bytes, uint32_t box_cols, uint32_t box_rows) {
  auto fn = tensor_map_encoder();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t elem_strides[2] = {1, 1};
  const CUresult r = fn(map, dtype, 2, const_cast<void*>(base), dims, strides, box, elem_strides,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int BN, int STAGES, int SB_KIND, bool OUT_BF16, bool GROUPED>
LaunchResult run_gemm(const uint8_t* qa, const float* sa, const uint8_t* qb, const float* sb,
                      const int32_t* offsets, int E, int64_t M, int64_t N, int64_t K, int64_t b_rows, void* c,
                      cudaStream_t stream, int sm_count) {
  using Cfg = GemmCfg<BN, STAGES, SB_KIND, OUT_BF16, GROUPED>;
  auto kernel = blockscaled_gemm_kernel<BN, STAGES, SB_KIND, OUT_BF16, GROUPED>;
  const size_t smem = Cfg::smem_bytes(E);
  cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (err != cudaSuccess) return {err, "cudaFuncSetAttribute(max dynamic shared memory)"};
  // The in-kernel register split assumes the block starts with kLaunchRegs per thread;
  // with fewer, the promotion warpgroups could never obtain their registers.
  cudaFuncAttributes fa;
  err = cudaFuncGetAttributes(&fa, kernel);
  if (err != cudaSuccess) return {err, "cudaFuncGetAttributes"};
  if (fa.numRegs != kLaunchRegs) return {cudaErrorInvalidConfiguration, "register count of the GEMM kernel"};

  CUtensorMap tmA, tmB, tmC;
  if (!encode_2d(&tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, qa, K, M, K, kBK, kBM))
    return {cudaErrorInvalidValue, "cuTensorMapEncodeTiled(A)"};
  if (!encode_2d(&tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, qb, K, b_rows, K, kBK, BN))
    return {cudaErrorInvalidValue, "cuTensorMapEncodeTiled(B)"};
  const uint64_t esize = OUT_BF16 ? 2 : 4;
  if (!encode_2d(&tmC, OUT_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, c, N, M,
                 N * esize, Cfg::kBoxCols, 32))
    return {cudaErrorInvalidValue, "cuTensorMapEncodeTiled(C)"};

  const int num_m = static_cast<int>((M + kBM - 1) / kBM);
  const int num_n = static_cast<int>((N + BN - 1) / BN);
  const int64_t tiles = static_cast<int64_t>(num_m) * num_n;
  const int grid = static_cast<int>(tiles < sm_count ? tiles : sm_count);
  kernel<<<grid, kThreads, smem, stream>>>(tmA, tmB, tmC, sa, sb, offsets, E, static_cast<int>(M),
                                           static_cast<int>(N), static_cast<int>(K), num_m, num_n);
  err = cudaGetLastError();
  if (err != cudaSuccess) return {err, "kernel launch"};
  return {cudaSuccess, nullptr};
}

}  // namespace

LaunchResult launch_blockscaled_gemm(const uint8_t* qa, const float* sa, const uint8_t* qb, const float* sb,
                                     int sb_kind, void* c, int c_bf16, int64_t M, int64_t N, int64_t K,
                                     cudaStream_t stream, int sm_count) {
  if (sb_kind == 0) {
    if (c_bf16) return run_gemm<256, 4, 0, true, false>(qa, sa, qb, sb, nullptr, 0, M, N, K, N, c, stream, sm_count);
    return run_gemm<256, 4, 0, false, false>(qa, sa, qb, sb, nullptr, 0, M, N, K, N, c, stream, sm_count);
  }
  if (c_bf16) return run_gemm<256, 3, 1, true, false>(qa, sa, qb, sb, nullptr, 0, M, N, K, N, c, stream, sm_count);
  return run_gemm<256, 3, 1, false, false>(qa, sa, qb, sb, nullptr, 0, M, N, K, N, c, stream, sm_count);
}

LaunchResult launch_grouped_gemm(const uint8_t* qa, const float* sa, const uint8_t* qb, const float* sb,
                                 const int32_t* offsets, int E, int64_t Mtot, void* c, int c_bf16, int64_t N,
                                 int64_t K, cudaStream_t stream, int sm_count) {
  if (c_bf16)
    return run_gemm<256, 3, 0, true, true>(qa, sa, qb, sb, offsets, E, Mtot, N, K, N * E, c, stream, sm_count);
  return run_gemm<256, 3, 0, false, true>(qa, sa, qb, sb, offsets, E, Mtot, N, K, N * E, c, stream, sm_count);
}

// Host access to the status word for fp8fg_sync_status.
cudaError_t read_and_clear_status(unsigned* out) {
  cudaError_t err = cudaMemcpyFromSymbol(out, g_status, sizeof(unsigned));
  if (err != cudaSuccess) return err;
  if (*out) {
    const unsigned zero = 0;
    err = cudaMemcpyToSymbol(g_status, &zero, sizeof(unsigned));
  }
  return err;
}

}  // namespace fp8fg
