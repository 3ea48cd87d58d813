// Launchers shared between the kernel files and the C ABI layer. Arguments have been
// validated by the caller (abi.cu) before any of these is called.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace fp8fg {

cudaError_t launch_quant_act_rows(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, uint8_t* q, float* s,
                                  cudaStream_t stream, int sm_count);
cudaError_t launch_quant_act_cols(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, uint8_t* q, float* s,
                                  cudaStream_t stream, int sm_count);
// Tiles along M for two tensors with the same M in one launch: x0 [M][K0] -> q0[K0][M],
// s0[K0][M/128] and x1 [M][K1] -> q1[K1][M], s1[K1][M/128]; M % 128 == 0.
cudaError_t launch_quant_act_cols_pair(const uint16_t* x0, int64_t K0, int64_t ldx0, uint8_t* q0, float* s0,
                                       const uint16_t* x1, int64_t K1, int64_t ldx1, uint8_t* q1, float* s1,
                                       int64_t M, cudaStream_t stream, int sm_count);
// Both orientations from one read: q[M][K], s[M][K/128] (tiles along K) and
// qt[K][M], st[K][M/128] (tiles along M); M and K multiples of 128.
cudaError_t launch_quant_act_dual(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, uint8_t* q, float* s,
                                  uint8_t* qt, float* st, cudaStream_t stream, int sm_count);
// Delayed scaling: one scale from history[0..H-1], history[H] the max |x| accumulator
// (zero on entry and on return); pushes this call's max |x| into the history.
cudaError_t launch_quant_act_delayed(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, float* history, int H,
                                     uint8_t* q, float* s, cudaStream_t stream, int sm_count);
// 2D row-major tensor [rows][cols] with the given row pitch in bytes; box = box_cols x
// box_rows elements; optional 128-byte swizzle; out-of-range elements read as zero.
bool encode_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t cols, uint64_t rows,
               uint64_t row_bytes, uint32_t box_cols, uint32_t box_rows, bool swizzle128);

// Status words of the kernel files (timeouts, invalid device-side arguments).
cudaError_t read_and_clear_gemm_status(unsigned* out);
cudaError_t read_and_clear_quant_status(unsigned* out);
cudaError_t launch_wait_timeout_selftest(cudaStream_t stream);

cudaError_t launch_quant_w_blocks(const uint16_t* w, int64_t N, int64_t K, int64_t ldw, uint8_t* q, float* s,
                                  cudaStream_t stream);
// Both orientations of the 128x128 block quantization: q[N][K], s[N/128][K/128] and
// qt[K][N], st[K/128][N/128].
cudaError_t launch_quant_w_dual(const uint16_t* w, int64_t N, int64_t K, int64_t ldw, uint8_t* q, float* s,
                                uint8_t* qt, float* st, cudaStream_t stream);

// Status of a GEMM launch: cudaSuccess, or the failing CUDA call's error; `what`
// names the failing step.
struct LaunchResult {
  cudaError_t err;
  const char* what;
};

// c_kind: 0 FP32 C, 1 BF16 C, 2 E4M3 codes of C with 1x128 scales c_scale[M][N/128].
// workspace: null for the data-parallel schedule, else at least gemm_workspace_bytes(sm_count)
// bytes (zero-initialized before first use) for the stream-K schedule.
LaunchResult launch_blockscaled_gemm(const uint8_t* qa, const float* sa, const uint8_t* qb, const float* sb,
                                     int sb_kind, void* c, float* c_scale, int c_kind, int64_t M, int64_t N,
                                     int64_t K, cudaStream_t stream, int sm_count, void* workspace = nullptr);
size_t gemm_workspace_bytes(int sm_count);
// Epoch of a stream-K launch (1 .. 2^31 - 1, cycling; distinct for consecutive launches).
int next_streamk_epoch();
// Address (current device) and size of the library-owned static stream-K workspace.
cudaError_t gemm_static_scratch(void** ptr, size_t* bytes);

LaunchResult launch_grouped_gemm(const uint8_t* qa, const float* sa, const uint8_t* qb, const float* sb,
                                 const int32_t* offsets, int E, int64_t Mtot, void* c, int c_bf16, int64_t N,
                                 int64_t K, cudaStream_t stream, int sm_count);

}  // namespace fp8fg
