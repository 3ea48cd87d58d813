// C ABI of libfp8fg.so (declared in include/fp8fg.h): host-side argument validation,
// device capability checks, per-thread error messages and the device status word.
// No entry point allocates or frees memory.
#include <cstdarg>
#include <cstdio>
#include <mutex>

#include "../../include/fp8fg.h"
#include "internal.h"

namespace {

thread_local char g_last_error[512] = "";

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return code;
}

int cuda_fail(cudaError_t err, const char* what) {
  return fail(FP8FG_ERR_CUDA, "%s failed: %s (%s)", what, cudaGetErrorName(err), cudaGetErrorString(err));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct DeviceInfo {
  int sm_count = 0;
  int supported = 0;
  int known = 0;
  void* scratch = nullptr;  // static stream-K workspace, set up on first use
};

constexpr int kMaxDevices = 64;
DeviceInfo g_devices[kMaxDevices];
std::mutex g_devices_mutex;

// Looks up (once per device) the SM count and whether the current device is an
// sm_103 GPU, the only architecture this library is built for.
int current_device(DeviceInfo* out) {
  int dev = -1;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return cuda_fail(err, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(FP8FG_ERR_UNSUPPORTED, "device index %d out of range", dev);
  std::lock_guard<std::mutex> lock(g_devices_mutex);
  DeviceInfo& d = g_devices[dev];
  if (!d.known) {
    int major = 0, minor = 0, sms = 0;
    if ((err = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (err = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
        (err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) {
      return cuda_fail(err, "cudaDeviceGetAttribute");
    }
    d.sm_count = sms;
    d.supported = (major == 10 && minor == 3);
    d.known = 1;
  }
  if (!d.supported) return fail(FP8FG_ERR_UNSUPPORTED, "device %d is not an sm_103 (B300) GPU", dev);
  *out = d;
  return FP8FG_OK;
}

constexpr int64_t kMaxDim = (int64_t(1) << 31) - 1;

// Address of the current device's static stream-K workspace, found once per device
// with cudaGetSymbolAddress (the array's host-side name is not a device address). The
// first call on a device also zero-fills the array with an asynchronous memset on the
// caller's stream, ordered before the GEMM launched next on that stream; make that
// first call outside stream capture. The release flags need no further clearing: a
// launch only accepts its own epoch (see next_streamk_epoch), and its tails clear the
// flags they consumed.
int static_scratch(void** out, cudaStream_t stream) {
  int dev = -1;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return cuda_fail(err, "cudaGetDevice");
  DeviceInfo info;
  if (int rc = current_device(&info)) return rc;
  std::lock_guard<std::mutex> lock(g_devices_mutex);
  DeviceInfo& d = g_devices[dev];
  if (!d.scratch) {
    void* p = nullptr;
    size_t bytes = 0;
    if ((err = fp8fg::gemm_static_scratch(&p, &bytes)) != cudaSuccess) return cuda_fail(err, "cudaGetSymbolAddress");
    if (fp8fg::gemm_workspace_bytes(d.sm_count) > bytes) {
      return fail(FP8FG_ERR_UNSUPPORTED, "static GEMM workspace holds %zu bytes, %zu needed for %d SMs", bytes,
                  fp8fg::gemm_workspace_bytes(d.sm_count), d.sm_count);
    }
    if ((err = cudaMemsetAsync(p, 0, bytes, stream)) != cudaSuccess) return cuda_fail(err, "cudaMemsetAsync");
    d.scratch = p;
  }
  *out = d.scratch;
  return FP8FG_OK;
}



}  // namespace

namespace {

// Validation and launch shared by fp8_blockscaled_gemm and fp8_blockscaled_gemm_ws.
int gemm_checked(const uint8_t* qa, const float* sa, const uint8_t* qb, const float* sb, int sb_kind, void* c,
                 int c_dtype, int64_t M, int64_t N, int64_t K, void* workspace, fp8fg_stream_t stream,
                 const char* name) {
  if (M < 0 || N < 0 || K < 0) return fail(FP8FG_ERR_ARG, "%s: negative size", name);
  if (sb_kind != FP8FG_SB_BLOCK_128x128 && sb_kind != FP8FG_SB_ROW_1x128) return fail(FP8FG_ERR_ARG, "%s: unknown sb_kind %d", name, sb_kind);
  if (c_dtype != FP8FG_OUT_F32 && c_dtype != FP8FG_OUT_BF16) return fail(FP8FG_ERR_ARG, "%s: unknown c_dtype %d", name, c_dtype);
  if (K % 128 || N % 128) return fail(FP8FG_ERR_ARG, "%s: K=%lld and N=%lld must be multiples of 128", name, (long long)K, (long long)N);
  if (M > kMaxDim || N > kMaxDim || K > kMaxDim) return fail(FP8FG_ERR_ARG, "%s: dimension too large", name);
  if (M == 0 || N == 0) return FP8FG_OK;
  if (!c) return fail(FP8FG_ERR_ARG, "%s: null output pointer", name);
  if (!aligned16(c)) return fail(FP8FG_ERR_ARG, "%s: pointers must be 16-byte aligned", name);
  const size_t esize = c_dtype == FP8FG_OUT_BF16 ? 2 : 4;
  if (K == 0) {
    DeviceInfo dev;
    if (int rc = current_device(&dev)) return rc;
    cudaError_t err = cudaMemsetAsync(c, 0, static_cast<size_t>(M) * N * esize, reinterpret_cast<cudaStream_t>(stream));
    return err == cudaSuccess ? FP8FG_OK : cuda_fail(err, "cudaMemsetAsync");
  }
  if (!qa || !sa || !qb || !sb) return fail(FP8FG_ERR_ARG, "%s: null pointer", name);
  if (!aligned16(qa) || !aligned16(sa) || !aligned16(qb) || !aligned16(sb)) return fail(FP8FG_ERR_ARG, "%s: pointers must be 16-byte aligned", name);
  DeviceInfo dev;
  if (int rc = current_device(&dev)) return rc;
  fp8fg::LaunchResult r = fp8fg::launch_blockscaled_gemm(qa, sa, qb, sb, sb_kind, c, nullptr,
                                                         c_dtype == FP8FG_OUT_BF16 ? 1 : 0, M, N, K,
                                                         reinterpret_cast<cudaStream_t>(stream), dev.sm_count,
                                                         workspace);
  if (r.err != cudaSuccess) return cuda_fail(r.err, r.what);
  return FP8FG_OK;
}

}  // namespace

extern "C" {

const char* fp8fg_last_error(void) { return g_last_error; }

int fp8fg_version(void) { return 100; }

int fp8_quant_act_1x128(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, int transposed, uint8_t* q, float* s,
                        fp8fg_stream_t stream) {
  g_last_error[0] = '\0';
  if (M < 0 || K < 0) return fail(FP8FG_ERR_ARG, "fp8_quant_act_1x128: negative size M=%lld K=%lld", (long long)M, (long long)K);
  if (transposed != 0 && transposed != 1) return fail(FP8FG_ERR_ARG, "fp8_quant_act_1x128: transposed must be 0 or 1");
  if (ldx < K) return fail(FP8FG_ERR_ARG, "fp8_quant_act_1x128: ldx=%lld < K=%lld", (long long)ldx, (long long)K);
  if (ldx % 8) return fail(FP8FG_ERR_ARG, "fp8_quant_act_1x128: ldx must be a multiple of 8 elements");
  if (transposed == 0 && K % 128) return fail(FP8FG_ERR_ARG, "fp8_quant_act_1x128: K=%lld is not a multiple of 128", (long long)K);
  if (transposed == 1 && M % 128) return fail(FP8FG_ERR_ARG, "fp8_quant_act_1x128 (transposed): M=%lld is not a multiple of 128", (long long)M);
  if (transposed == 1 && K % 8) return fail(FP8FG_ERR_ARG, "fp8_quant_act_1x128 (transposed): K=%lld is not a multiple of 8", (long long)K);
  if (M > kMaxDim || K > kMaxDim) return fail(FP8FG_ERR_ARG, "fp8_quant_act_1x128: dimension too large");
  if (M == 0 || K == 0) return FP8FG_OK;
  if (!x || !q || !s) return fail(FP8FG_ERR_ARG, "fp8_quant_act_1x128: null pointer");
  if (!aligned16(x) || !aligned16(q) || !aligned16(s)) return fail(FP8FG_ERR_ARG, "fp8_quant_act_1x128: pointers must be 16-byte aligned");
  DeviceInfo dev;
  if (int rc = current_device(&dev)) return rc;
  cudaError_t err = transposed
                        ? fp8fg::launch_quant_act_cols(x, M, K, ldx, q, s, reinterpret_cast<cudaStream_t>(stream),
                                                       dev.sm_count)
                        : fp8fg::launch_quant_act_rows(x, M, K, ldx, q, s, reinterpret_cast<cudaStream_t>(stream),
                                                       dev.sm_count);
  if (err != cudaSuccess) return cuda_fail(err, "fp8_quant_act_1x128 launch");
  return FP8FG_OK;
}

int fp8_quant_act_1x128_transposed_pair(const uint16_t* x0, int64_t K0, int64_t ldx0, uint8_t* q0, float* s0,
                                        const uint16_t* x1, int64_t K1, int64_t ldx1, uint8_t* q1, float* s1,
                                        int64_t M, fp8fg_stream_t stream) {
  g_last_error[0] = '\0';
  const char* name = "fp8_quant_act_1x128_transposed_pair";
  if (M < 0 || K0 < 0 || K1 < 0) return fail(FP8FG_ERR_ARG, "%s: negative size", name);
  if (M % 128) return fail(FP8FG_ERR_ARG, "%s: M=%lld is not a multiple of 128", name, (long long)M);
  if (K0 % 8 || K1 % 8) return fail(FP8FG_ERR_ARG, "%s: K0=%lld and K1=%lld must be multiples of 8", name, (long long)K0, (long long)K1);
  if ((K0 > 0 && (ldx0 < K0 || ldx0 % 8)) || (K1 > 0 && (ldx1 < K1 || ldx1 % 8))) {
    return fail(FP8FG_ERR_ARG, "%s: row strides must be >= K and multiples of 8", name);
  }
  if (M > kMaxDim || K0 > kMaxDim || K1 > kMaxDim) return fail(FP8FG_ERR_ARG, "%s: dimension too large", name);
  const bool use0 = M > 0 && K0 > 0, use1 = M > 0 && K1 > 0;
  if ((use0 && (!x0 || !q0 || !s0)) || (use1 && (!x1 || !q1 || !s1))) return fail(FP8FG_ERR_ARG, "%s: null pointer", name);
  if ((use0 && (!aligned16(x0) || !aligned16(q0) || !aligned16(s0))) ||
      (use1 && (!aligned16(x1) || !aligned16(q1) || !aligned16(s1)))) {
    return fail(FP8FG_ERR_ARG, "%s: pointers must be 16-byte aligned", name);
  }
  if (!use0 && !use1) return FP8FG_OK;
  DeviceInfo dev;
  if (int rc = current_device(&dev)) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t err;
  if (use0 && use1) {
    err = fp8fg::launch_quant_act_cols_pair(x0, K0, ldx0, q0, s0, x1, K1, ldx1, q1, s1, M, st, dev.sm_count);
  } else if (use0) {
    err = fp8fg::launch_quant_act_cols(x0, M, K0, ldx0, q0, s0, st, dev.sm_count);
  } else {
    err = fp8fg::launch_quant_act_cols(x1, M, K1, ldx1, q1, s1, st, dev.sm_count);
  }
  if (err != cudaSuccess) return cuda_fail(err, "fp8_quant_act_1x128_transposed_pair launch");
  return FP8FG_OK;
}

int fp8_quant_act_delayed(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, float* amax_history, int H,
                          uint8_t* q, float* s, fp8fg_stream_t stream) {
  g_last_error[0] = '\0';
  if (M < 0 || K < 0) return fail(FP8FG_ERR_ARG, "fp8_quant_act_delayed: negative size");
  if (K % 128) return fail(FP8FG_ERR_ARG, "fp8_quant_act_delayed: K=%lld is not a multiple of 128", (long long)K);
  if (ldx < K || ldx % 8) return fail(FP8FG_ERR_ARG, "fp8_quant_act_delayed: ldx=%lld must be >= K and a multiple of 8", (long long)ldx);
  if (H < 1 || H > 1024) return fail(FP8FG_ERR_ARG, "fp8_quant_act_delayed: history length %d outside 1..1024", H);
  if (M > kMaxDim || K > kMaxDim) return fail(FP8FG_ERR_ARG, "fp8_quant_act_delayed: dimension too large");
  if (!amax_history) return fail(FP8FG_ERR_ARG, "fp8_quant_act_delayed: null history");
  if (!aligned16(amax_history)) return fail(FP8FG_ERR_ARG, "fp8_quant_act_delayed: pointers must be 16-byte aligned");
  if (M > 0 && K > 0) {
    if (!x || !q || !s) return fail(FP8FG_ERR_ARG, "fp8_quant_act_delayed: null pointer");
    if (!aligned16(x) || !aligned16(q) || !aligned16(s)) return fail(FP8FG_ERR_ARG, "fp8_quant_act_delayed: pointers must be 16-byte aligned");
  }
  DeviceInfo dev;
  if (int rc = current_device(&dev)) return rc;
  cudaError_t err;
  if (M == 0 || K == 0) {  // nothing to quantize: max |x| = 0 still enters the history
    err = fp8fg::launch_quant_act_delayed(nullptr, 0, 128, 128, amax_history, H, nullptr, nullptr,
                                          reinterpret_cast<cudaStream_t>(stream), dev.sm_count);
  } else {
    err = fp8fg::launch_quant_act_delayed(x, M, K, ldx, amax_history, H, q, s, reinterpret_cast<cudaStream_t>(stream),
                                          dev.sm_count);
  }
  if (err != cudaSuccess) return cuda_fail(err, "fp8_quant_act_delayed launch");
  return FP8FG_OK;
}

int fp8_quant_w_128x128(const uint16_t* w, int64_t N, int64_t K, int64_t ldw, uint8_t* q, float* s,
                        fp8fg_stream_t stream) {
  g_last_error[0] = '\0';
  if (N < 0 || K < 0) return fail(FP8FG_ERR_ARG, "fp8_quant_w_128x128: negative size");
  if (N % 128 || K % 128) return fail(FP8FG_ERR_ARG, "fp8_quant_w_128x128: N=%lld and K=%lld must be multiples of 128", (long long)N, (long long)K);
  if (ldw < K || ldw % 8) return fail(FP8FG_ERR_ARG, "fp8_quant_w_128x128: ldw=%lld must be >= K and a multiple of 8", (long long)ldw);
  if (N > kMaxDim || K > kMaxDim) return fail(FP8FG_ERR_ARG, "fp8_quant_w_128x128: dimension too large");
  if (N == 0 || K == 0) return FP8FG_OK;
  if (!w || !q || !s) return fail(FP8FG_ERR_ARG, "fp8_quant_w_128x128: null pointer");
  if (!aligned16(w) || !aligned16(q) || !aligned16(s)) return fail(FP8FG_ERR_ARG, "fp8_quant_w_128x128: pointers must be 16-byte aligned");
  DeviceInfo dev;
  if (int rc = current_device(&dev)) return rc;
  cudaError_t err = fp8fg::launch_quant_w_blocks(w, N, K, ldw, q, s, reinterpret_cast<cudaStream_t>(stream));
  if (err != cudaSuccess) return cuda_fail(err, "fp8_quant_w_128x128 launch");
  return FP8FG_OK;
}

int fp8_quant_act_1x128_dual(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, uint8_t* q, float* s,
                             uint8_t* qt, float* st, fp8fg_stream_t stream) {
  g_last_error[0] = '\0';
  if (M < 0 || K < 0) return fail(FP8FG_ERR_ARG, "fp8_quant_act_1x128_dual: negative size");
  if (M % 128 || K % 128) return fail(FP8FG_ERR_ARG, "fp8_quant_act_1x128_dual: M=%lld and K=%lld must be multiples of 128", (long long)M, (long long)K);
  if (ldx < K || ldx % 8) return fail(FP8FG_ERR_ARG, "fp8_quant_act_1x128_dual: ldx=%lld must be >= K and a multiple of 8", (long long)ldx);
  if (M > kMaxDim || K > kMaxDim) return fail(FP8FG_ERR_ARG, "fp8_quant_act_1x128_dual: dimension too large");
  if (M == 0 || K == 0) return FP8FG_OK;
  if (!x || !q || !s || !qt || !st) return fail(FP8FG_ERR_ARG, "fp8_quant_act_1x128_dual: null pointer");
  if (!aligned16(x) || !aligned16(q) || !aligned16(s) || !aligned16(qt) || !aligned16(st)) {
    return fail(FP8FG_ERR_ARG, "fp8_quant_act_1x128_dual: pointers must be 16-byte aligned");
  }
  DeviceInfo dev;
  if (int rc = current_device(&dev)) return rc;
  cudaError_t err = fp8fg::launch_quant_act_dual(x, M, K, ldx, q, s, qt, st, reinterpret_cast<cudaStream_t>(stream),
                                                 dev.sm_count);
  if (err != cudaSuccess) return cuda_fail(err, "fp8_quant_act_1x128_dual launch");
  return FP8FG_OK;
}

int fp8_quant_w_128x128_dual(const uint16_t* w, int64_t N, int64_t K, int64_t ldw, uint8_t* q, float* s,
                             uint8_t* qt, float* st, fp8fg_stream_t stream) {
  g_last_error[0] = '\0';
  if (N < 0 || K < 0) return fail(FP8FG_ERR_ARG, "fp8_quant_w_128x128_dual: negative size");
  if (N % 128 || K % 128) return fail(FP8FG_ERR_ARG, "fp8_quant_w_128x128_dual: N=%lld and K=%lld must be multiples of 128", (long long)N, (long long)K);
  if (ldw < K || ldw % 8) return fail(FP8FG_ERR_ARG, "fp8_quant_w_128x128_dual: ldw=%lld must be >= K and a multiple of 8", (long long)ldw);
  if (N > kMaxDim || K > kMaxDim) return fail(FP8FG_ERR_ARG, "fp8_quant_w_128x128_dual: dimension too large");
  if (N == 0 || K == 0) return FP8FG_OK;
  if (!w || !q || !s || !qt || !st) return fail(FP8FG_ERR_ARG, "fp8_quant_w_128x128_dual: null pointer");
  if (!aligned16(w) || !aligned16(q) || !aligned16(s) || !aligned16(qt) || !aligned16(st)) {
    return fail(FP8FG_ERR_ARG, "fp8_quant_w_128x128_dual: pointers must be 16-byte aligned");
  }
  DeviceInfo dev;
  if (int rc = current_device(&dev)) return rc;
  cudaError_t err = fp8fg::launch_quant_w_dual(w, N, K, ldw, q, s, qt, st, reinterpret_cast<cudaStream_t>(stream));
  if (err != cudaSuccess) return cuda_fail(err, "fp8_quant_w_128x128_dual launch");
  return FP8FG_OK;
}

int fp8_blockscaled_gemm(const uint8_t* qa, const float* sa, const uint8_t* qb, const float* sb, int sb_kind,
                         void* c, int c_dtype, int64_t M, int64_t N, int64_t K, fp8fg_stream_t stream) {
  g_last_error[0] = '\0';
  return gemm_checked(qa, sa, qb, sb, sb_kind, c, c_dtype, M, N, K, nullptr, stream, "fp8_blockscaled_gemm");
}

int64_t fp8_blockscaled_gemm_workspace_bytes(void) {
  g_last_error[0] = '\0';
  DeviceInfo dev;
  if (int rc = current_device(&dev)) return rc;
  return static_cast<int64_t>(fp8fg::gemm_workspace_bytes(dev.sm_count));
}

int fp8_blockscaled_gemm_ws(const uint8_t* qa, const float* sa, const uint8_t* qb, const float* sb, int sb_kind,
                            void* c, int c_dtype, int64_t M, int64_t N, int64_t K, void* workspace,
                            int64_t workspace_bytes, fp8fg_stream_t stream) {
  g_last_error[0] = '\0';
  if (!workspace) return fail(FP8FG_ERR_ARG, "fp8_blockscaled_gemm_ws: null workspace");
  if (!aligned16(workspace)) return fail(FP8FG_ERR_ARG, "fp8_blockscaled_gemm_ws: workspace must be 16-byte aligned");
  DeviceInfo dev;
  if (int rc = current_device(&dev)) return rc;
  const int64_t need = static_cast<int64_t>(fp8fg::gemm_workspace_bytes(dev.sm_count));
  if (workspace_bytes < need) {
    return fail(FP8FG_ERR_ARG, "fp8_blockscaled_gemm_ws: workspace of %lld bytes, %lld needed", (long long)workspace_bytes,
                (long long)need);
  }
  return gemm_checked(qa, sa, qb, sb, sb_kind, c, c_dtype, M, N, K, workspace, stream, "fp8_blockscaled_gemm_ws");
}

int fp8_blockscaled_gemm_sk_static(const uint8_t* qa, const float* sa, const uint8_t* qb, const float* sb,
                                   int sb_kind, void* c, int c_dtype, int64_t M, int64_t N, int64_t K,
                                   fp8fg_stream_t stream) {
  g_last_error[0] = '\0';
  void* scratch = nullptr;
  if (int rc = static_scratch(&scratch, reinterpret_cast<cudaStream_t>(stream))) return rc;
  return gemm_checked(qa, sa, qb, sb, sb_kind, c, c_dtype, M, N, K, scratch, stream, "fp8_blockscaled_gemm_sk_static");
}

int fp8_blockscaled_gemm_e4m3(const uint8_t* qa, const float* sa, const uint8_t* qb, const float* sb, int sb_kind,
                              uint8_t* c_q, float* c_s, int64_t M, int64_t N, int64_t K, fp8fg_stream_t stream) {
  g_last_error[0] = '\0';
  if (M < 0 || N < 0 || K < 0) return fail(FP8FG_ERR_ARG, "fp8_blockscaled_gemm_e4m3: negative size");
  if (sb_kind != FP8FG_SB_BLOCK_128x128 && sb_kind != FP8FG_SB_ROW_1x128) return fail(FP8FG_ERR_ARG, "fp8_blockscaled_gemm_e4m3: unknown sb_kind %d", sb_kind);
  if (K % 128 || N % 128) return fail(FP8FG_ERR_ARG, "fp8_blockscaled_gemm_e4m3: K=%lld and N=%lld must be multiples of 128", (long long)K, (long long)N);
  if (M > kMaxDim || N > kMaxDim || K > kMaxDim) return fail(FP8FG_ERR_ARG, "fp8_blockscaled_gemm_e4m3: dimension too large");
  if (M == 0 || N == 0) return FP8FG_OK;
  if (!c_q || !c_s) return fail(FP8FG_ERR_ARG, "fp8_blockscaled_gemm_e4m3: null output pointer");
  if (!aligned16(c_q) || !aligned16(c_s)) return fail(FP8FG_ERR_ARG, "fp8_blockscaled_gemm_e4m3: pointers must be 16-byte aligned");
  if (K == 0) {  // C = 0: every tile is all-zero, scale +0 and codes 0x00
    DeviceInfo dev;
    if (int rc = current_device(&dev)) return rc;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t err = cudaMemsetAsync(c_q, 0, static_cast<size_t>(M) * N, st);
    if (err == cudaSuccess) err = cudaMemsetAsync(c_s, 0, static_cast<size_t>(M) * (N / 128) * sizeof(float), st);
    return err == cudaSuccess ? FP8FG_OK : cuda_fail(err, "cudaMemsetAsync");
  }
  if (!qa || !sa || !qb || !sb) return fail(FP8FG_ERR_ARG, "fp8_blockscaled_gemm_e4m3: null pointer");
  if (!aligned16(qa) || !aligned16(sa) || !aligned16(qb) || !aligned16(sb)) return fail(FP8FG_ERR_ARG, "fp8_blockscaled_gemm_e4m3: pointers must be 16-byte aligned");
  DeviceInfo dev;
  if (int rc = current_device(&dev)) return rc;
  fp8fg::LaunchResult r = fp8fg::launch_blockscaled_gemm(qa, sa, qb, sb, sb_kind, c_q, c_s, 2, M, N, K,
                                                         reinterpret_cast<cudaStream_t>(stream), dev.sm_count);
  if (r.err != cudaSuccess) return cuda_fail(r.err, r.what);
  return FP8FG_OK;
}

int fp8_grouped_gemm(const uint8_t* qa, const float* sa, const uint8_t* qb, const float* sb,
                     const int32_t* group_offsets, int E, int64_t Mtot, void* c, int c_dtype, int64_t N, int64_t K,
                     fp8fg_stream_t stream) {
  g_last_error[0] = '\0';
  if (E < 1 || E > 1024) return fail(FP8FG_ERR_ARG, "fp8_grouped_gemm: E=%d must be in 1..1024", E);
  if (Mtot < 0 || N < 0 || K < 0) return fail(FP8FG_ERR_ARG, "fp8_grouped_gemm: negative size");
  if (c_dtype != FP8FG_OUT_F32 && c_dtype != FP8FG_OUT_BF16) return fail(FP8FG_ERR_ARG, "fp8_grouped_gemm: unknown c_dtype %d", c_dtype);
  if (Mtot % 128 || N % 128 || K % 128) return fail(FP8FG_ERR_ARG, "fp8_grouped_gemm: Mtot=%lld, N=%lld and K=%lld must be multiples of 128", (long long)Mtot, (long long)N, (long long)K);
  if (Mtot > kMaxDim || N * E > kMaxDim || K > kMaxDim) return fail(FP8FG_ERR_ARG, "fp8_grouped_gemm: dimension too large");
  if (Mtot == 0 || N == 0) return FP8FG_OK;
  if (K == 0) return fail(FP8FG_ERR_ARG, "fp8_grouped_gemm: K must be positive");
  if (!qa || !sa || !qb || !sb || !group_offsets || !c) return fail(FP8FG_ERR_ARG, "fp8_grouped_gemm: null pointer");
  if (!aligned16(qa) || !aligned16(sa) || !aligned16(qb) || !aligned16(sb) || !aligned16(c) ||
      (reinterpret_cast<uintptr_t>(group_offsets) & 3u))
    return fail(FP8FG_ERR_ARG, "fp8_grouped_gemm: misaligned pointer");
  DeviceInfo dev;
  if (int rc = current_device(&dev)) return rc;
  fp8fg::LaunchResult r = fp8fg::launch_grouped_gemm(qa, sa, qb, sb, group_offsets, E, Mtot, c,
                                                     c_dtype == FP8FG_OUT_BF16, N, K,
                                                     reinterpret_cast<cudaStream_t>(stream), dev.sm_count);
  if (r.err != cudaSuccess) return cuda_fail(r.err, r.what);
  return FP8FG_OK;
}

int fp8fg_selftest_wait_timeout(fp8fg_stream_t stream) {
  g_last_error[0] = '\0';
  DeviceInfo dev;
  if (int rc = current_device(&dev)) return rc;
  cudaError_t err = fp8fg::launch_wait_timeout_selftest(reinterpret_cast<cudaStream_t>(stream));
  if (err != cudaSuccess) return cuda_fail(err, "fp8fg_selftest_wait_timeout launch");
  return FP8FG_OK;
}

int fp8fg_sync_status(fp8fg_stream_t stream) {
  g_last_error[0] = '\0';
  cudaError_t err = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  if (err != cudaSuccess) return cuda_fail(err, "cudaStreamSynchronize");
  unsigned st = 0, st_q = 0;
  err = fp8fg::read_and_clear_gemm_status(&st);
  if (err == cudaSuccess) err = fp8fg::read_and_clear_quant_status(&st_q);
  if (err != cudaSuccess) return cuda_fail(err, "reading the device status words");
  st |= st_q;
  if (st & 1u) return fail(FP8FG_ERR_TIMEOUT, "a device-side wait ran out of time (status 0x%x)", st);
  if (st & 2u) return fail(FP8FG_ERR_DEVICE_ARG, "invalid group offsets on the device (status 0x%x)", st);
  return FP8FG_OK;
}

}  // extern "C"
