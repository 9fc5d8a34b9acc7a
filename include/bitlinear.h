/*
 * bitlinear.h -- C ABI of the B300 BitLinear W1.58A8 forward library.
 *
 * The operation (BitNet b1.58 BitLinear, weights 1.58-bit, activations 8-bit):
 *
 *   gamma   = mean(|W|)                                   per tensor, fp32
 *   code    = clip(rint(W / (gamma + 1e-5)), -1, 1)       ternary weight codes
 *   Wp      = four codes per byte                         packed weights
 *   s_m     = 127 / max(max_k |x[m][k]|, 1e-5)            per-token scale, fp32
 *   x_q     = clip(rint(x * s_m), -128, 127)              int8 activations
 *   acc     = sum_k code[n][k] * x_q[m][k]                exact int32
 *   y[m][n] = acc * gamma / s_m                           fp32 output
 *
 * Sources (web pages, cited by title and section):
 *   "BitNet 1-bit LLM 的混合精度微调技术：渐进量化策略" (blog.hotdry.top), body,
 *     the quantisation-function paragraph (weight absmean = mean(|W|),
 *     activation absmax = max(|X|, eps = 1e-5)) and the forward-pass sentence
 *     (divide by the absmean factor, round, limit to [-1, 1], multiply back;
 *     activations absmax-quantised per token to 8 bits).
 *   "穿越1比特的奇幻旅程：高效语言模型的未来之谜" (summary of the BitNet b1.58
 *     2B4T Technical Report), section "架构创新：量化魔法的背后" (absmean
 *     ternary weights, per-token absmax INT8 activations, no bias) and section
 *     "GPU端：CUDA内核的定制魔法" (W1.58A8 matmul; four ternary weights packed
 *     into one 8-bit value: pack, store, load, unpack, compute).
 *   "BitNet 中使用直通估计器工程化三元权重训练" (blog.hotdry.top), section
 *     "STE 机制在三元训练中的作用" (torch.round: ties to even).
 *
 * Numerical contract (every step is deterministic and bit-reproducible):
 *   - gamma is the exact mean of |W| rounded once to fp32, ties to even;
 *   - d = fp32(gamma + 1e-5f); code = clip(rint(fp32(W / d)), -1, 1);
 *   - s_m = fp32(127 / fp32 max(absmax, 1e-5f)); x_q = clip(rint(fp32(x * s_m)));
 *   - y = fp32(fp32((float)acc * gamma) / s_m);
 *   - every rounding is round-to-nearest, ties to even.
 *
 * Packed layout: Wp is uint8 [N][K/4], row-major. Byte j of row n holds the
 * codes of k = 4j .. 4j+3; the code of k = 4j+i sits in bits 2i..2i+1 as the
 * field value code + 1 (0 -> -1, 1 -> 0, 2 -> +1; 3 never occurs).
 *
 * Conventions for every entry point:
 *   - Pointers are device pointers unless stated otherwise; the caller owns
 *     and allocates every buffer. The library never allocates device memory
 *     on the compute path.
 *   - All work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and is asynchronous: nothing synchronises the host.
 *   - Argument errors are detected on the host before any launch and return
 *     a non-zero status with nothing enqueued. Launch errors return
 *     BL_ERR_CUDA. Errors while kernels run surface at the caller's next
 *     synchronisation, as for any CUDA work.
 *   - x, W, Wp, x_q and y must be 16-byte aligned. M, N, K > 0, K % 4 == 0,
 *     N * K < 2^32 and K <= 65536 (the int32 accumulator of |acc| <= 127*K).
 *   - Inputs must be finite; NaN or Inf inputs give unspecified codes.
 *   - Several host threads may call the library, on one device or on
 *     several; the last error message is thread-local. Each kernel's
 *     shared-memory limit is raised once per (device, kernel), on the device
 *     current in the calling thread, in a table guarded by a mutex, so first
 *     calls may happen concurrently and one process may drive several GPUs.
 */
#ifndef BITLINEAR_H
#define BITLINEAR_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define BL_API __attribute__((visibility("default")))
#else
#define BL_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    BL_OK = 0,
    BL_ERR_INVALID_ARG = 1,   /* a pointer, size, alignment or dtype is invalid */
    BL_ERR_UNSUPPORTED = 2,   /* valid arguments this build does not handle */
    BL_ERR_CUDA = 3,          /* a CUDA call failed; see bitlinear_last_error() */
    BL_ERR_WORKSPACE = 4      /* workspace missing, misaligned or too small */
} bl_status;

typedef enum {
    BL_F32 = 0,               /* activations are fp32 */
    BL_BF16 = 1               /* activations are bf16 (widened exactly to fp32) */
} bl_dtype;

/* Same type as cudaStream_t, declared without including CUDA headers. */
typedef struct CUstream_st* bl_stream_t;

/* ---------------------------------------------------------------------------
 * Weight quantisation and packing (absmean, ternary codes, 4 codes per byte).
 * Passages: the quantisation-function paragraph and forward-pass sentence of
 * "BitNet 1-bit LLM 的混合精度微调技术"; sections "架构创新" and "GPU端" of the
 * 2B4T summary.
 *
 * W         fp32 [N][K] row-major (nn.Linear layout: out x in), read only.
 * Wp        uint8 [N][K/4], written.
 * gamma     one fp32, written (device pointer).
 * workspace at least bitlinear_pack_workspace_bytes(N, K) bytes, 256-byte
 *           aligned, used as scratch for the exact sum; no initial contents
 *           are needed and none survive the call.
 * ------------------------------------------------------------------------- */
BL_API size_t bitlinear_pack_workspace_bytes(int64_t N, int64_t K);

BL_API bl_status bitlinear_pack_weights(const float* W, int64_t N, int64_t K,
                                 uint8_t* Wp, float* gamma,
                                 void* workspace, size_t ws_bytes,
                                 bl_stream_t stream);

/* The two halves of bitlinear_pack_weights, for callers that need gamma alone
 * or time the steps separately.
 *
 * bitlinear_absmean: gamma = mean(|W|), exact sum rounded once to fp32.
 *   workspace: at least bitlinear_pack_workspace_bytes(N, K) bytes, 256-byte
 *   aligned, scratch only.
 * bitlinear_quantize_pack: codes clip(rint(W / (gamma + 1e-5)), -1, 1) packed
 *   four per byte into Wp, with gamma read from device memory (as written by
 *   bitlinear_absmean, or any fp32 value >= 0). */
BL_API bl_status bitlinear_absmean(const float* W, int64_t N, int64_t K, float* gamma,
                                   void* workspace, size_t ws_bytes, bl_stream_t stream);

BL_API bl_status bitlinear_quantize_pack(const float* W, int64_t N, int64_t K, const float* gamma,
                                         uint8_t* Wp, bl_stream_t stream);

/* ---------------------------------------------------------------------------
 * Weight packing by one of the quantisers the pages describe. The packed
 * layout and the forward are unchanged: pass `scale` to bitlinear_forward in
 * place of gamma (y = acc * scale / s).
 *
 *   BL_QUANT_ABSMEAN      the default rule, exactly bitlinear_pack_weights
 *                         (factor is ignored; scale = gamma).
 *   BL_QUANT_ALPHA_ROUND  alpha = fp32(factor x mean|W|);
 *                         code = clip(rint(fp32(W / alpha)), -1, 1); scale = alpha.
 *                         "BitNet 中使用直通估计器工程化三元权重训练", sections
 *                         "STE 机制在三元训练中的作用" and "工程化训练流程与参数配置"
 *                         (factor 0.7; its zero threshold tau = 0.1 alpha changes
 *                         no code, since |W| < tau already rounds to 0). An
 *                         all-zero W gives alpha = 0 and all codes 0.
 *   BL_QUANT_THRESHOLD    delta = fp32(factor x mean|W|); code = sign(W) where
 *                         |W| > delta, else 0; scale = exact sum of |W| over the
 *                         kept weights / (N*K), rounded once to fp32.
 *                         "BitNet 三元权重阈值优化工程实践", section
 *                         "三元权重阈值优化的核心原理" and its threshold module
 *                         (factor 0.7; 0.75 for attention, 0.6 for FFN layers).
 *
 * mean|W| is gamma of the default rule (the exact mean rounded once to fp32).
 * factor: positive and finite (the pages use 0.6, 0.7 and 0.75).
 * Wp, scale, workspace: as Wp, gamma and workspace of bitlinear_pack_weights.
 * The threshold rule reads W three times and uses *scale for gamma until its
 * last kernel writes the scale.
 * ------------------------------------------------------------------------- */
typedef enum {
    BL_QUANT_ABSMEAN = 0,
    BL_QUANT_ALPHA_ROUND = 1,
    BL_QUANT_THRESHOLD = 2
} bl_quantizer;

BL_API bl_status bitlinear_pack_weights_quantizer(const float* W, int64_t N, int64_t K,
                                                  bl_quantizer quantizer, float factor,
                                                  uint8_t* Wp, float* scale,
                                                  void* workspace, size_t ws_bytes,
                                                  bl_stream_t stream);

/* bitlinear_pack_weights_noalloc: the same packing as bitlinear_pack_weights,
 * for callers that cannot allocate device memory and so cannot pass a
 * workspace: a plugin running inside another framework whose caching
 * allocator owns the device and must not be bypassed, or a runtime that
 * reserved all device memory up front, where a cudaMalloc would fail or
 * fragment memory the host framework manages. The pages have no counterpart
 * of this call; it is an interface convenience.
 *
 * Scratch: a static device array of 75,776 bytes (bitlinear_pack_workspace_bytes
 * of any shape) inside the library, which every GPU that loads the library
 * holds until the process exits. No cudaMalloc, cudaFree or other allocating
 * call is made. W, Wp and gamma are as for bitlinear_pack_weights.
 *
 * Every call looks up the array's device address on the current device
 * (cudaGetSymbolAddress); the first call on a device may load the library's
 * device code there, so make it before any stream capture begins. Because the
 * address is not cached, calls after a cudaDeviceReset use the reloaded
 * array. Every call on a device shares the one
 * array: calls whose work overlaps on the GPU (different streams, no ordering
 * between them) race and give wrong results; calls ordered on one stream are
 * safe. Nothing in the array needs to start at zero: each call writes every
 * slot it reads.
 *
 * Returns BL_ERR_UNSUPPORTED (with a message) if the shape needs more scratch
 * than the array holds, and the statuses of bitlinear_pack_weights otherwise. */
BL_API bl_status bitlinear_pack_weights_noalloc(const float* W, int64_t N, int64_t K,
                                                uint8_t* Wp, float* gamma, bl_stream_t stream);

/* ---------------------------------------------------------------------------
 * Per-token absmax int8 activation quantisation.
 * Passages: "activation absmax = max(|X|, eps=1e-5)" and per-token 8-bit
 * quantisation in "BitNet 1-bit LLM 的混合精度微调技术"; INT8 per-token absmax in
 * section "架构创新" of the 2B4T summary.
 *
 * x      [M][K] row-major, fp32 or bf16 per `dt`, read only.
 * xq     int8 [M][K] row-major, written.
 * scale  fp32 [M], written: s_m = 127 / max(max|x_m|, 1e-5).
 * ------------------------------------------------------------------------- */
BL_API bl_status bitlinear_quant_act(const void* x, bl_dtype dt, int64_t M, int64_t K,
                              int8_t* xq, float* scale, bl_stream_t stream);

/* ---------------------------------------------------------------------------
 * The forward: activation quantisation, ternary x int8 contraction with an
 * exact int32 accumulator and the fp32 rescale y = acc * gamma / s.
 * Passages: section "GPU端：CUDA内核的定制魔法" of the 2B4T summary (W1.58A8
 * matmul over packed weights); "multiply back by the factor" in the
 * forward-pass sentence of "BitNet 1-bit LLM 的混合精度微调技术".
 *
 * x          [M][K] row-major activations, fp32 or bf16 per `dt`.
 * Wp, gamma  from bitlinear_pack_weights.
 * y          fp32 [M][N] row-major, written.
 * xq_out     optional int8 [M][K]: if non-NULL the quantised activations are
 *            also written there.
 * scale_out  optional fp32 [M]: if non-NULL the per-token scales are written.
 * workspace  at least bitlinear_forward_workspace_bytes(M, N, K) bytes,
 *            256-byte aligned (may be NULL when that size is 0). Scratch:
 *            its contents need no initialisation and are overwritten. The
 *            size depends on the current device's SM count (the tensor-core
 *            path keeps a split-tile buffer there), so query it on the device
 *            that runs the call.
 *
 * The kernels are chosen by M and K: with K % 64 == 0, a dp4a GEMV with the
 * activation pass ahead of it for M <= 4, a fused mma.sync kernel for
 * M <= 8, activation quantisation plus mma.sync for M <= 16, and the tcgen05
 * tensor-core path for M >= 17; K % 64 != 0 takes the activation pass plus a
 * dp4a kernel. Calls that share a workspace must not overlap on the GPU.
 * ------------------------------------------------------------------------- */
BL_API size_t bitlinear_forward_workspace_bytes(int64_t M, int64_t N, int64_t K);

BL_API bl_status bitlinear_forward(const void* x, bl_dtype dt, int64_t M,
                            const uint8_t* Wp, const float* gamma,
                            int64_t N, int64_t K, float* y,
                            int8_t* xq_out, float* scale_out,
                            void* workspace, size_t ws_bytes,
                            bl_stream_t stream);

/* ---------------------------------------------------------------------------
 * The contraction and rescale on already-quantised activations:
 * y[m][n] = fp32(fp32(acc[m][n] * gamma) / scale[m]).
 * Passages: as for bitlinear_forward.
 *
 * xq         int8 [M][K] row-major, scale fp32 [M] (from bitlinear_quant_act).
 * workspace  at least bitlinear_gemm_workspace_bytes(M, N, K) bytes, 256-byte
 *            aligned (may be NULL when that size is 0).
 * ------------------------------------------------------------------------- */
BL_API size_t bitlinear_gemm_workspace_bytes(int64_t M, int64_t N, int64_t K);

BL_API bl_status bitlinear_gemm(const int8_t* xq, const float* scale, int64_t M,
                                const uint8_t* Wp, const float* gamma, int64_t N, int64_t K,
                                float* y, void* workspace, size_t ws_bytes, bl_stream_t stream);

/* ---------------------------------------------------------------------------
 * The bare contraction acc[m][n] = sum_k code[n][k] * xq[m][k] (exact int32),
 * for checking the accumulator bit for bit.
 * Passage: section "GPU端：CUDA内核的定制魔法" of the 2B4T summary.
 *
 * xq   int8 [M][K] row-major; Wp uint8 [N][K/4]; acc int32 [M][N], written.
 * workspace at least bitlinear_gemm_i32_workspace_bytes(M, N, K) bytes.
 * ------------------------------------------------------------------------- */
BL_API size_t bitlinear_gemm_i32_workspace_bytes(int64_t M, int64_t N, int64_t K);

BL_API bl_status bitlinear_gemm_i32(const int8_t* xq, const uint8_t* Wp,
                             int64_t M, int64_t N, int64_t K, int32_t* acc,
                             void* workspace, size_t ws_bytes,
                             bl_stream_t stream);

/* ---------------------------------------------------------------------------
 * The forward for one token by table lookup: the table idea of bitnet.cpp's
 * TL1 kernel ("部署 BitNet 1-bit LLM：三元权重边缘推理优化", kernel types; TL1
 * uses a lookup table), as an alternative to the dp4a GEMV of
 * bitlinear_forward, with the same result bit for bit. For every pair of
 * consecutive inputs the kernel tabulates the nine partial sums
 * (f0 - 1) x_q[2p] + (f1 - 1) x_q[2p + 1] once per call; each 4-bit nibble
 * of a packed row then selects one entry.
 *
 * x      [1][K] fp32 or bf16 per `dt`, 16-byte aligned; M must be 1.
 * Wp, gamma from bitlinear_pack_weights; K % 64 == 0, K <= 16384.
 * y      fp32 [1][N], 4-byte aligned, written: fp32(fp32(acc * gamma) / s).
 * No workspace. Errors: BL_ERR_UNSUPPORTED for M != 1 or K > 16384;
 * otherwise as for bitlinear_forward.
 * ------------------------------------------------------------------------- */
BL_API bl_status bitlinear_forward_lut(const void* x, bl_dtype dt, int64_t M,
                                       const uint8_t* Wp, const float* gamma,
                                       int64_t N, int64_t K, float* y,
                                       bl_stream_t stream);

/* ---------------------------------------------------------------------------
 * Per-group weight quantisation, groups of 64.
 * Passage: "BitNet 1-bit LLM 的混合精度微调技术：渐进量化策略", body: per-group
 * quantisation with a group size of 64. The page names the group size only;
 * here a group is 64 consecutive k of one row, and each group takes the
 * absmean rule of bitlinear_pack_weights on its own:
 *   gamma[n][g] = exact mean of |W[n][64g .. 64g + 63]|, rounded once to fp32;
 *   code = clip(rint(fp32(W / fp32(gamma[n][k / 64] + 1e-5))), -1, 1).
 *
 * W       fp32 [N][K] row-major, 16-byte aligned, finite, read only; K % 64 == 0.
 * Wp      uint8 [N][K/4], 16-byte aligned, written: the per-tensor packing
 *         layout (code of k = 4j + i in bits 2i..2i+1 of byte j of the row,
 *         field = code + 1).
 * gammas  fp32 [N][K/64] row-major, 4-byte aligned, written.
 * No workspace; W is read once. Errors: BL_ERR_INVALID_ARG for null or
 * misaligned pointers, non-positive sizes or K % 64 != 0; BL_ERR_UNSUPPORTED
 * for K > 65536 or N*K >= 2^32; BL_ERR_CUDA if the launch fails.
 * ------------------------------------------------------------------------- */
BL_API bl_status bitlinear_pack_weights_grouped(const float* W, int64_t N, int64_t K,
                                                uint8_t* Wp, float* gammas, bl_stream_t stream);

/* ---------------------------------------------------------------------------
 * The forward over per-group scales:
 *   y[m][n] = sum_g gammas[n][g] * acc[m][n][g] / s_m,
 *   acc[m][n][g] = sum over group g of code * x_q (exact integers),
 * with x_q and s_m the per-token absmax codes and scales of bitlinear_quant_act.
 * Passages: as for bitlinear_pack_weights_grouped and bitlinear_forward.
 *
 * x          [M][K] row-major, fp32 or bf16 per `dt`, 16-byte aligned.
 * Wp, gammas from bitlinear_pack_weights_grouped (K % 64 == 0).
 * y          fp32 [M][N] row-major, 4-byte aligned, written. Each product
 *            gamma * acc is exact in fp64; the K/64 products of a row are
 *            added in fp64, divided by s_m in fp64 and rounded to fp32, so
 *            |y - RN(exact / s_m)| <= ulp(y) + (K/64) 2^-52 sum_g |gamma * acc| / s_m.
 * xq_out     optional int8 [M][K] (16-byte aligned) and scale_out optional
 *            fp32 [M]: the quantised activations and scales, bit for bit those
 *            of bitlinear_quant_act.
 * workspace  at least bitlinear_forward_grouped_workspace_bytes(M, N, K)
 *            bytes, 256-byte aligned; scratch. Calls that share a workspace
 *            must not overlap on the GPU.
 * Errors: as for bitlinear_forward, plus BL_ERR_INVALID_ARG for K % 64 != 0
 * and BL_ERR_UNSUPPORTED for M > 65535.
 * ------------------------------------------------------------------------- */
BL_API size_t bitlinear_forward_grouped_workspace_bytes(int64_t M, int64_t N, int64_t K);

BL_API bl_status bitlinear_forward_grouped(const void* x, bl_dtype dt, int64_t M,
                                           const uint8_t* Wp, const float* gammas,
                                           int64_t N, int64_t K, float* y,
                                           int8_t* xq_out, float* scale_out,
                                           void* workspace, size_t ws_bytes,
                                           bl_stream_t stream);

/* ---------------------------------------------------------------------------
 * Schedule of the tensor-core contraction (the path of bitlinear_forward,
 * bitlinear_gemm and bitlinear_gemm_i32 for M >= 17 and K % 64 == 0), as a
 * test hook: host arithmetic only, no CUDA call, so it runs on any machine.
 * It lists the work the persistent kernel's CTAs would do for M tokens, N
 * weight rows and K inputs on `sms` multiprocessors, so that a test can check
 * that every output tile's k-stages are covered exactly once.
 *
 * Output tiles are 128 weight rows x BN tokens; tile t covers weight rows
 * from 128 (t % R) and tokens from BN (t / R), R = ceil(N / 128), and has
 * K / 64 k-stages. Tiles below D are computed whole; tiles D .. D + S - 1 are
 * split by k-stages over several CTAs whose partial sums are added in an
 * fp32 buffer.
 *
 * plan      int32 [9], written: BN, grid (CTAs), R, k-stages per tile, D, S,
 *           CTAs that take a run of split stages, token tiles ceil(M / BN),
 *           bytes of the split-tile buffer and counters in the workspace.
 * n_items   int32 [grid] or NULL: the number of work items of each CTA.
 * items     int32 [grid][max_items][3] or NULL: item i of CTA b is
 *           (tile, k0, k1), the tile and its k-stage range [k0, k1), in the
 *           order the CTA computes them. Caller-owned host memory.
 * Errors: BL_ERR_INVALID_ARG for sizes bitlinear_forward rejects, K not a
 * multiple of 64, sms outside 1..4096, a NULL plan, or (with items) a CTA
 * with more than max_items items; n_items is complete in that last case.
 * ------------------------------------------------------------------------- */
BL_API bl_status bitlinear_tc_schedule(int64_t M, int64_t N, int64_t K, int sms,
                                       int32_t* plan, int32_t* n_items, int32_t* items,
                                       int max_items);

/* ---------------------------------------------------------------------------
 * Diagnostics.
 * ------------------------------------------------------------------------- */
BL_API const char* bitlinear_strerror(bl_status status);   /* static string */
BL_API const char* bitlinear_last_error(void);             /* thread-local detail of the last failure */
BL_API int bitlinear_version(void);                        /* ABI version, currently 1 */

/* Reads and clears the library's device-side error word of the current
 * device into *flag (host pointer): non-zero if, since the last call, a
 * kernel gave up a bounded wait for its own asynchronous copies (its outputs
 * are then unspecified). Synchronises with the device. */
BL_API bl_status bitlinear_device_error(int* flag);

#ifdef __cplusplus
}
#endif

#endif /* BITLINEAR_H */
