/*
 * fp8fg — fine-grained FP8 (E4M3) quantization and block-scaled FP8 GEMM on B300 (sm_103a).
 *
 * C ABI of the shared library libfp8fg.so. Every entry point takes plain device
 * pointers and sizes; no PyTorch or C++ type crosses this boundary.
 *
 * What the operations are (knowledge-base pages on DeepSeek-V3 FP8 training):
 *  - "Online quantization vs delayed quantization in DeepSeek-V3", item 1, and
 *    "Unified E4M3 format in DeepSeek-V3", section on the fine-grained quantization
 *    strategy: a scaling factor is computed on the fly for every 1x128 activation
 *    tile and every 128x128 weight block, and all tensors use E4M3.
 *  - "Advantages of using FP8 for GEMM operations in DeepSeek-V3", item 5: the FP8
 *    GEMM promotes the tensor-core partial sums to FP32 at fixed intervals; item 8:
 *    dense and MoE (grouped) FP8 GEMMs.
 *
 * Numerical definition (identical for every quantizer; a "group" is one 1x128 tile
 * or one 128x128 block):
 *    amax = max |x| over the group (exact)
 *    s    = amax / 448          IEEE binary32 division, round to nearest even
 *    q    = E4M3FN( x / s )     binary32 division, then round to nearest even into
 *                               E4M3FN, saturating to +-448; the sign is kept, so a
 *                               negative value that rounds to zero gives 0x80
 *    a group with amax == 0 gets s = +0.0f and codes 0x00.
 * E4M3FN is the OCP 8-bit float "E4M3" (bias 7, max 448, no infinities, NaN 0x7F/0xFF);
 * codes are passed as uint8_t. Inputs are bfloat16 given as raw 16-bit words; NaN or
 * infinite inputs give unspecified codes.
 *
 * Conventions shared by all entry points:
 *  - Pointers are CUDA device pointers owned by the caller. The library never
 *    allocates or frees memory. Outputs are overwritten, never accumulated into.
 *  - Every data pointer must be 16-byte aligned; leading dimensions are in elements.
 *  - Calls are asynchronous on `stream` (NULL = the legacy default stream) and do not
 *    synchronize. They return FP8FG_OK (0) on success or a negative error code; on
 *    error nothing has been launched and fp8fg_last_error() describes the problem.
 *  - The pipelined kernels (the GEMMs and the transposed quantizer) bound every
 *    device-side wait. A wait that runs out (about one second) makes the kernel record
 *    a timeout in a device status word and return; fp8fg_sync_status() reports it as
 *    FP8FG_ERR_TIMEOUT. Invalid group offsets found on the
 *    device are reported the same way (FP8FG_ERR_DEVICE_ARG).
 *  - Empty problems (a zero dimension) return FP8FG_OK without launching.
 */
#ifndef FP8FG_H
#define FP8FG_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st *fp8fg_stream_t;

enum fp8fg_status {
    FP8FG_OK = 0,
    FP8FG_ERR_ARG = -1,        /* invalid argument detected on the host; nothing launched */
    FP8FG_ERR_CUDA = -2,       /* a CUDA runtime or driver call failed */
    FP8FG_ERR_TIMEOUT = -3,    /* a device-side wait ran out (from fp8fg_sync_status) */
    FP8FG_ERR_DEVICE_ARG = -4, /* invalid device-resident argument (from fp8fg_sync_status) */
    FP8FG_ERR_UNSUPPORTED = -5 /* the current device is not an sm_103 (B300) GPU */
};

enum fp8fg_out_dtype { FP8FG_OUT_F32 = 0, FP8FG_OUT_BF16 = 1 };

enum fp8fg_sb_kind {
    FP8FG_SB_BLOCK_128x128 = 0, /* sb[N/128][K/128]: one scale per 128x128 block of B */
    FP8FG_SB_ROW_1x128 = 1      /* sb[N][K/128]:     one scale per 1x128 tile of B   */
};

/*
 * Activation quantization in 1x128 tiles ("Online quantization vs delayed
 * quantization in DeepSeek-V3", item 1; "Unified E4M3 format in DeepSeek-V3",
 * fine-grained quantization strategy).
 *
 * x: bf16 [M][K], row stride ldx >= K elements (ldx % 8 == 0).
 * transposed == 0: tiles run along K (a row's 128 consecutive columns).
 *     Requires K % 128 == 0. Outputs q[M][K] (row stride K) and s[M][K/128].
 *     x[m][k] ~= dec(q[m][k]) * s[m][k/128].
 * transposed == 1: tiles run along M (128 consecutive rows of one column, e.g. 128
 *     tokens of one feature, the reduction dimension of a weight-gradient GEMM; the
 *     E4M3 page says the backward pass uses E4M3 too). Requires M % 128 == 0 and
 *     K % 8 == 0. The result is stored transposed so that M is contiguous: q[K][M]
 *     (row stride M) and s[K][M/128]; x[m][k] ~= dec(q[k][m]) * s[k][m/128].
 * Returns FP8FG_ERR_ARG for a null pointer, misalignment or a shape rule broken.
 */
int fp8_quant_act_1x128(const uint16_t *x, int64_t M, int64_t K, int64_t ldx, int transposed,
                        uint8_t *q, float *s, fp8fg_stream_t stream);

/*
 * The tiles-along-M quantization (fp8_quant_act_1x128 with transposed == 1) of two
 * tensors that share M, in one launch: typically the two operands of a weight-gradient
 * GEMM dW = dY^T . X, whose reduction runs over the tokens ("Unified E4M3 format in
 * DeepSeek-V3": E4M3 with 1x128 tiles in the backward pass as well). One launch instead
 * of two saves a launch's fixed cost and spreads the blocks of both tensors over all SMs.
 *
 * x0: bf16 [M][K0], row stride ldx0 >= K0; x1: bf16 [M][K1], row stride ldx1 >= K1
 * (strides and K0, K1 multiples of 8; M % 128 == 0).
 * Outputs, bit-identical to two calls of fp8_quant_act_1x128(.., transposed = 1, ..):
 *     q0[K0][M], s0[K0][M/128] and q1[K1][M], s1[K1][M/128].
 * A tensor with K = 0 is skipped (its pointers and row stride are not used).
 * Returns FP8FG_ERR_ARG for a null pointer, misalignment or a shape rule broken.
 */
int fp8_quant_act_1x128_transposed_pair(const uint16_t *x0, int64_t K0, int64_t ldx0, uint8_t *q0, float *s0,
                                        const uint16_t *x1, int64_t K1, int64_t ldx1, uint8_t *q1, float *s1,
                                        int64_t M, fp8fg_stream_t stream);

/*
 * Delayed (history-based) quantization, the contrast to the online scaling above
 * ("Online quantization vs delayed quantization in DeepSeek-V3", items 2-3: delayed
 * quantization derives the scale from maximum values recorded in earlier iterations
 * and has to keep that history).
 *
 * x: bf16 [M][K], row stride ldx >= K (ldx % 8 == 0); K % 128 == 0; any M >= 0.
 * amax_history: DEVICE float [H + 1], 1 <= H <= 1024, caller-owned state that lives
 *     across calls: entries 0..H-1 are the per-tensor maxima max |x| of the H most
 *     recent calls, most recent first; entry H must be +0 (the library leaves it +0).
 *     Zero-initialize all H + 1 floats before the first call.
 * One scale for the whole tensor: s = fl32(max(amax_history[0..H-1]) / 448), or s = 1
 * when that maximum is 0 (no history yet). Codes q[M][K] = E4M3FN(fl32(x / s)),
 * saturating to +-448 (values beyond 448 s saturate; online scaling never does), and
 * s[M][K/128] = s for every 1x128 tile, so (q, s) can be the A operand of
 * fp8_blockscaled_gemm. Then the history shifts by one: amax_history[0] = max |x| of
 * this call (exact), the oldest entry drops out.
 * Two kernels on `stream`: the quantization (which also accumulates max |x| into entry
 * H) and a one-block history update. Calls that share a history must be ordered.
 * Returns FP8FG_ERR_ARG for a null pointer, misalignment or a shape rule broken.
 */
int fp8_quant_act_delayed(const uint16_t *x, int64_t M, int64_t K, int64_t ldx, float *amax_history, int H,
                          uint8_t *q, float *s, fp8fg_stream_t stream);

/*
 * Weight quantization in 128x128 blocks (same passages as above).
 *
 * w: bf16 [N][K], row stride ldw >= K (ldw % 8 == 0); N % 128 == 0, K % 128 == 0.
 * Outputs q[N][K] (row stride K) and s[N/128][K/128];
 * w[n][k] ~= dec(q[n][k]) * s[n/128][k/128].
 */
int fp8_quant_w_128x128(const uint16_t *w, int64_t N, int64_t K, int64_t ldw,
                        uint8_t *q, float *s, fp8fg_stream_t stream);

/*
 * Both orientations of the 1x128 activation quantization from one read of x (the
 * transposed copy feeds the weight-gradient GEMM; "Unified E4M3 format in DeepSeek-V3":
 * E4M3 in the backward pass too, and fine-grained quantization strategy).
 *
 * x: bf16 [M][K], row stride ldx >= K (ldx % 8 == 0); M % 128 == 0 and K % 128 == 0.
 * Outputs, bit-identical to fp8_quant_act_1x128 with transposed = 0 and = 1:
 *     q[M][K], s[M][K/128]   tiles along K;
 *     qt[K][M], st[K][M/128] tiles along M, stored transposed.
 * Reads x once (2 bytes per element) instead of twice.
 * Returns FP8FG_ERR_ARG for a null pointer, misalignment or a shape rule broken.
 */
int fp8_quant_act_1x128_dual(const uint16_t *x, int64_t M, int64_t K, int64_t ldx, uint8_t *q, float *s,
                             uint8_t *qt, float *st, fp8fg_stream_t stream);

/*
 * Both orientations of the 128x128 weight quantization from one read of w (same
 * passages). A 128x128 block holds the same elements, hence the same scale and codes, in
 * either orientation, so the transposed copy is the B operand of the data-gradient GEMM
 * dX = dY . W, computed as fp8_blockscaled_gemm(q(dY), s(dY), qt, st, 128x128, ...).
 *
 * w: bf16 [N][K], row stride ldw >= K (ldw % 8 == 0); N % 128 == 0 and K % 128 == 0.
 * Outputs: q[N][K], s[N/128][K/128], bit-identical to fp8_quant_w_128x128, and
 *     qt[K][N] = q transposed, st[K/128][N/128] = s transposed.
 * Returns FP8FG_ERR_ARG for a null pointer, misalignment or a shape rule broken.
 */
int fp8_quant_w_128x128_dual(const uint16_t *w, int64_t N, int64_t K, int64_t ldw, uint8_t *q, float *s,
                             uint8_t *qt, float *st, fp8fg_stream_t stream);

/*
 * Block-scaled FP8 GEMM C = A . B^T ("Advantages of using FP8 for GEMM operations in
 * DeepSeek-V3", items 1, 5 and 8).
 *
 * qa: E4M3 [M][K] (row stride K), sa: f32 [M][K/128] (1x128 tiles of A).
 * qb: E4M3 [N][K] (row stride K), sb: f32 scales of B, layout by sb_kind
 *     (FP8FG_SB_BLOCK_128x128: [N/128][K/128]; FP8FG_SB_ROW_1x128: [N][K/128]).
 * c:  [M][N] row-major, c_dtype FP8FG_OUT_F32 or FP8FG_OUT_BF16 (round to nearest even).
 * For every 128-deep K chunk kb the tensor cores form the chunk's partial sum P in
 * FP32, and C_acc[m][n] += P[m][n] * (sa[m][kb] * sb(n, kb)) is added in FP32.
 * Requires K % 128 == 0 and N % 128 == 0; any M >= 0. K == 0 writes zeros.
 */
int fp8_blockscaled_gemm(const uint8_t *qa, const float *sa, const uint8_t *qb, const float *sb,
                         int sb_kind, void *c, int c_dtype, int64_t M, int64_t N, int64_t K,
                         fp8fg_stream_t stream);

/*
 * The same GEMM as fp8_blockscaled_gemm, scheduled stream-K with a caller-owned
 * workspace (no counterpart on the pages: a scheduling choice for this GPU). When the
 * tiles do not fill whole waves of CTAs, the chunks of the last one to two waves' worth
 * of tiles are divided evenly over the CTAs; a tile cut between two CTAs has its head's
 * FP32 partial sums passed through the workspace, and the tail continues from them in the
 * same chunk order, so C is bit-identical to fp8_blockscaled_gemm.
 *
 * workspace: DEVICE memory of at least fp8_blockscaled_gemm_workspace_bytes() bytes,
 *     16-byte aligned, zero-filled before its first use. The library leaves it ready for
 *     the next call, also after a call that reported FP8FG_ERR_TIMEOUT: a cut tile's
 *     partial sums are released by a flag holding a value unique to the launch, so a
 *     flag left set by a launch that gave up is ignored by later launches. Calls that
 *     share a workspace must not run concurrently (order them on one stream).
 * Other arguments, layouts and errors as fp8_blockscaled_gemm; FP8FG_ERR_ARG for a null,
 * misaligned or too small workspace.
 */
int fp8_blockscaled_gemm_ws(const uint8_t *qa, const float *sa, const uint8_t *qb, const float *sb, int sb_kind,
                            void *c, int c_dtype, int64_t M, int64_t N, int64_t K, void *workspace,
                            int64_t workspace_bytes, fp8fg_stream_t stream);

/*
 * fp8_blockscaled_gemm_ws with a library-owned workspace: the call allocates nothing
 * (no counterpart on the pages; it makes the stream-K schedule available to callers that
 * cannot hand over device memory). The workspace is one file-scope static device array
 * per device, sized for devices with up to 160 SMs (about 20 MB; FP8FG_ERR_UNSUPPORTED
 * beyond that). Its address is looked up, and the array zero-filled by an asynchronous
 * memset on `stream`, on the first call on each device, so make that first call before
 * capturing a stream into a graph. Its release flags stay valid after a call that
 * reported FP8FG_ERR_TIMEOUT (see fp8_blockscaled_gemm_ws), so the array never needs to
 * be cleared again. Every call on a device uses the same array: calls that overlap in
 * time (on different streams, or from different threads without ordering) race on it and
 * give undefined results; order them on one stream. Arguments, results (bit-identical to
 * fp8_blockscaled_gemm) and errors otherwise as fp8_blockscaled_gemm.
 */
int fp8_blockscaled_gemm_sk_static(const uint8_t *qa, const float *sa, const uint8_t *qb, const float *sb,
                                   int sb_kind, void *c, int c_dtype, int64_t M, int64_t N, int64_t K,
                                   fp8fg_stream_t stream);

/* Workspace size for fp8_blockscaled_gemm_ws on the current device (about 128 KB per SM);
 * a negative error code if the device is unsupported. */
int64_t fp8_blockscaled_gemm_workspace_bytes(void);

/*
 * Block-scaled FP8 GEMM whose output is quantized to E4M3 in 1x128 tiles (activations
 * kept in FP8 between layers: "Unified E4M3 format in DeepSeek-V3", memory section; the
 * quantization is the one of fp8_quant_act_1x128).
 *
 * C = A . B^T is formed exactly as by fp8_blockscaled_gemm (same operands, layouts and
 * per-chunk FP32 promotion); then every 1x128 tile of C (row m, columns 128 t .. 128 t
 * + 127) is quantized from the FP32 accumulators, without rounding to BF16 first:
 *     c_s[m][t] = fl32(max |C| over the tile / 448),
 *     c_q[m][n] = E4M3FN(fl32(C[m][n] / c_s[m][n / 128])), RNE, saturating;
 *     an all-zero tile gets scale +0 and codes 0x00.
 * c_q: [M][N] uint8 (row stride N), c_s: [M][N/128] float; (c_q, c_s) can be the A
 * operand of a following GEMM. Requires K % 128 == 0 and N % 128 == 0; any M >= 0.
 * K == 0 gives C = 0: all scales +0 and all codes 0x00.
 */
int fp8_blockscaled_gemm_e4m3(const uint8_t *qa, const float *sa, const uint8_t *qb, const float *sb,
                              int sb_kind, uint8_t *c_q, float *c_s, int64_t M, int64_t N, int64_t K,
                              fp8fg_stream_t stream);

/*
 * Grouped (MoE expert) block-scaled FP8 GEMM ("Advantages of using FP8 for GEMM
 * operations in DeepSeek-V3", item 8: the MoE variant).
 *
 * qa: E4M3 [Mtot][K], sa: f32 [Mtot][K/128]. The rows of expert e are
 *     group_offsets[e] .. group_offsets[e+1]-1 (contiguous, padded by the caller).
 * group_offsets: DEVICE int32 [E+1], non-decreasing multiples of 128,
 *     group_offsets[0] == 0 and group_offsets[E] == Mtot. Checked on the device: a
 *     violation writes nothing useful and is reported by fp8fg_sync_status().
 * qb: E4M3 [E][N][K], sb: f32 [E][N/128][K/128] (128x128 blocks per expert).
 * c:  [Mtot][N]; row m of expert e is A[m] . B_e^T with the same per-chunk promotion
 *     as fp8_blockscaled_gemm. Requires Mtot % 128 == 0, N % 128 == 0, K % 128 == 0.
 */
int fp8_grouped_gemm(const uint8_t *qa, const float *sa, const uint8_t *qb, const float *sb,
                     const int32_t *group_offsets, int E, int64_t Mtot, void *c, int c_dtype,
                     int64_t N, int64_t K, fp8fg_stream_t stream);

/* Message for the last nonzero return on the calling thread ("" if none). */
const char *fp8fg_last_error(void);

/*
 * Synchronize `stream`, then read and clear the current device's status words.
 * Returns FP8FG_OK, FP8FG_ERR_TIMEOUT, FP8FG_ERR_DEVICE_ARG, or FP8FG_ERR_CUDA when
 * the stream reports a CUDA error.
 */
int fp8fg_sync_status(fp8fg_stream_t stream);

/*
 * Self-test of the device-side failure detection (no counterpart on the pages: it
 * exercises this library's own safety mechanism). Launches one small kernel that waits,
 * with the bounded wait every pipelined kernel here uses, on a shared-memory barrier
 * nothing ever arrives at. After about one second the wait gives up and records a
 * timeout in the device status word; the kernel then returns normally, so the context
 * stays usable. A following fp8fg_sync_status(stream) returns FP8FG_ERR_TIMEOUT and
 * clears the word. Returns FP8FG_OK when the launch succeeded.
 */
int fp8fg_selftest_wait_timeout(fp8fg_stream_t stream);

/* Library version, e.g. 100 for 0.1.0. */
int fp8fg_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FP8FG_H */
