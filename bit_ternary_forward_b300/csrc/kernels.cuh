// Kernel declarations shared by the C-ABI layer and the kernel sources.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "bitlinear.h"

namespace bl {

// Launches `kern` as a programmatic dependent of the previous work in `s`
// (see pdl_wait in common.cuh): it may start before that work ends.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// Records `msg` as the calling thread's last error and returns `st` (abi.cu).
bl_status record_error(bl_status st, const char* msg);

// Per-device kernel set-up (setup.cu), thread-safe: raise `func`'s dynamic
// shared-memory limit on the current device to at least `bytes` (a no-op up
// to the default 48 KB), and the resident CTAs per SM of `func` with
// `threads` threads and `bytes` of dynamic shared memory (0 if it cannot run).
cudaError_t ensure_smem(const void* func, size_t bytes);
int resident_ctas(const void* func, int threads, size_t bytes);

// ---- weight packing (pack.cu)
// Both weight-pass kernels stream W through a ring of shared-memory stages
// filled by bulk copies: consumer threads plus one producer warp.
constexpr int kAbsumThreads = 256;          // consumers of the exact-sum kernel
constexpr int kPackThreads = 256;           // consumers of the packing kernel
constexpr int kRingStageF4 = 1024;          // float4 per stage (16 KB)
constexpr int kRingStages = 4;              // stages in flight per CTA (64 KB)
constexpr uint32_t kRingSmem = kRingStages * kRingStageF4 * 16;
// Bytes of W the exact-sum pass marks to stay in L2 for the packing pass
// (three quarters of a 126 MB L2).
constexpr uint64_t kL2KeepBytes = 96ull << 20;
constexpr int kPartialWords = 16;          // one 64-byte exact partial per CTA (12 limbs used)
constexpr int kMaxAbsumCtas = 1184;        // 8 per SM on 148 SMs

// Rules of the packing pass (how gamma becomes the code threshold and scale).
constexpr int kRuleAbsmean = 0;      // codes of W / (gamma + 1e-5), scale gamma
constexpr int kRuleAlphaRound = 1;   // codes of W / alpha, alpha = fp32(factor x gamma), scale alpha
constexpr int kRuleThreshold = 2;    // codes sign(W) [|W| > fp32(factor x gamma)], scale from a masked sum
// Exact-sum partials of |W| (n4 float4) into `partials` on `grid` CTAs; with
// mask_gamma, only weights with |w| > fp32(factor x *mask_gamma) count.
cudaError_t launch_absum(const float4* w4, uint64_t n4, uint32_t* partials, const float* mask_gamma, float factor,
                         unsigned grid, cudaStream_t s);
int absum_ctas_per_sm(bool masked);   // 0: the shared memory cannot be reserved
cudaError_t take_pack_wait_error(int* flag);
__global__ void bl_gamma_finalize(const uint32_t* __restrict__ partials, int n_partials, uint64_t count,
                                  float* __restrict__ gamma);
// Codes and packing of W (n_bytes = N*K/4 output bytes) on a one-wave grid,
// by `rule` (kRule*). With partials (the fused form) every CTA combines gamma
// from the exact-sum partials; otherwise gamma is read from *gamma_in. If
// scale_out is not null, CTA 0 writes the forward's scale there (gamma or
// alpha; never for kRuleThreshold).
cudaError_t launch_quant_pack(const float4* w4, uint64_t n_bytes, const float* gamma_in, const uint32_t* partials,
                              int n_partials, float* scale_out, uint32_t* wp_words, int rule, float factor, int sms,
                              cudaStream_t s);

// ---- activation quantisation (act_quant.cu)
constexpr int kActThreads = 256;
// x is fp32 (bf16 == false) or bf16 bits (bf16 == true); one CTA per token.
cudaError_t launch_act_quant(const void* x, bool bf16, int M, int K, int8_t* xq, float* scale, cudaStream_t s);

// ---- decode GEMV (gemv.cu)
constexpr int kGemvThreads = 512;          // 16 warps, one output row per warp at a time

enum class GemvOut { kY = 0, kAcc = 1 };

// out is fp32 y [M][N] (kY) or int32 acc [M][N] (kAcc); scale/gamma unused for kAcc.
// vec selects 16-byte weight loads (K % 64 == 0, 16-byte aligned rows); mt is
// the number of tokens per CTA (1, 2 or 4); grid_x CTAs of kGemvThreads.
cudaError_t launch_gemv(const uint8_t* wp, const int8_t* xq, const float* scale, const float* gamma, void* out,
                        int M, int N, int K, GemvOut mode, bool vec, int mt, int grid_x, cudaStream_t s);

// ---- decode / skinny contraction on mma.sync (decode.cu)
constexpr int kDecodeThreads = 512;
constexpr int kXinF32 = 0, kXinBF16 = 1, kXinI8 = 2;   // activation input kinds
constexpr size_t kMaxSmemPerCta = 227 * 1024;
constexpr size_t kOneCtaPerSmSmem = 120 * 1024;   // > half of the 228 KB an SM holds

// Dynamic shared memory of bl_decode_mma for a block of rows_per_cta rows.
size_t decode_smem_bytes(int rows_per_cta, int K);

// x is fp32 / bf16 (quantised in the kernel; xq_out and scale_out optional) or
// int8 x_q with scale_in (xin == kXinI8). out is fp32 y or int32 acc [M][N].
// Needs K % 64 == 0 and 16-byte aligned wp, x.
cudaError_t launch_decode(const uint8_t* wp, const void* x, int xin, const float* scale_in, const float* gamma,
                          void* out, bool out_acc, int8_t* xq_out, float* scale_out, int M, int N, int K,
                          int rows_per_cta, cudaStream_t s);

// Reads and clears the device word set when a bounded wait gave up (synchronous).
cudaError_t take_wait_error(int* flag);

// ---- decode GEMV for M <= 4: per-token activation pass + contraction (gemv_fused.cu)
constexpr int kGemvFusedThreads = 512;
constexpr int kActTqThreads = 256;
constexpr int kGemvFusedMaxM = 4;
// Chooses rows per CTA and the number of k-parts for M x N x K on `sms` SMs;
// returns the contraction's dynamic shared memory in bytes (never 0), or 0 if
// the path does not take the shape (M > 4, K % 64 != 0, K too long).
size_t gemv_fused_plan(int M, int N, int K, int sms, int* rows_per_cta, int* parts);
// Launches both kernels. workspace: the transposed codes (M*K bytes, rounded up
// to 256), then int token sums [M] (rounded up to 256), then fp32 scales [M]
// (used when scale_out is NULL). With xin == kXinI8, x is x_q and scale_in its
// scales; out is fp32 y or int32 acc (out_acc).
cudaError_t launch_gemv_fused(const uint8_t* wp, const void* x, int xin, const float* scale_in, const float* gamma,
                              void* out, bool out_acc, int8_t* xq_out, float* scale_out, int M, int N, int K,
                              int rows_per_cta, int parts, size_t smem, void* workspace, cudaStream_t s);
cudaError_t take_gemv_wait_error(int* flag);

// ---- decode GEMV for M <= 4 in one kernel: activation pass + dp4a contraction (gemv_dp4a.cu)
constexpr int kGemvDp4aThreads = 512;
constexpr int kGemvDp4aMaxM = 4;
constexpr size_t kGemvDp4aMaxAct = 65536;          // bytes of quantised activations (tokens rounded to 1, 2, 4) x K
constexpr size_t kGemvDp4aMaxSmem = 110 * 1024;    // two CTAs fit on an SM: this one and the next kernel's
// Rows of W per CTA for M x N x K on `sms` SMs; returns the dynamic shared
// memory in bytes, or 0 if the kernel does not take the shape (M > 4,
// K % 64 != 0, or the activations do not fit).
size_t gemv_dp4a_plan(int M, int N, int K, int sms, int* rows_per_cta);
// x is fp32 / bf16 (quantised in the kernel; xq_out and scale_out optional) or
// int8 x_q with scale_in (xin == kXinI8). out is fp32 y or int32 acc (out_acc,
// int8 input only). No workspace.
cudaError_t launch_gemv_dp4a(const uint8_t* wp, const void* x, int xin, const float* scale_in, const float* gamma,
                             void* out, bool out_acc, int8_t* xq_out, float* scale_out, int M, int N, int K,
                             int rows_per_cta, size_t smem, cudaStream_t s);
cudaError_t take_dp4a_wait_error(int* flag);

// ---- lookup-table decode GEMV, one token (gemv_lut.cu)
constexpr int kLutMaxK = 16384;
size_t gemv_lut_smem(int K);
cudaError_t launch_gemv_lut(const uint8_t* wp, const void* x, bool bf16, const float* gamma, float* y, int N, int K,
                            int sms, cudaStream_t s);

// ---- per-group (64) packing and forward (grouped.cu)
cudaError_t launch_pack_grouped(const float* W, int64_t N, int64_t K, uint8_t* wp, float* gam, int sms,
                                cudaStream_t s);
// Workspace of the grouped forward: transposed codes, group code sums, scales.
size_t forward_grouped_workspace(int64_t M, int64_t K);
cudaError_t launch_forward_grouped(const void* x, bool bf16, int M, int N, int K, const uint8_t* wp, const float* gam,
                                   float* y, int8_t* xq_out, float* scale_out, void* ws, cudaStream_t s);

// ---- prefill contraction on tcgen05 (prefill.cu)
constexpr int kTcMinM = 17;   // smallest M routed to the tensor-core kernel (below it the
                              // mma.sync decode kernel is faster on B300)
// Launch plan of the tensor-core contraction (tc_plan, prefill.cu): token-tile
// width, grid, whole tiles and split ("stream-K") tiles, and the bytes of its
// split-tile workspace (an fp32 buffer of sk_buf_bytes, then int counters),
// which must be zero when the contraction starts.
struct TcPlan {
  int bn = 256, grid = 1, n_tiles_n = 1, k_iters = 1, dp_tiles = 0, sk_tiles = 0, sk_ctas = 0;
  size_t sk_buf_bytes = 0, sk_bytes = 0;
};
TcPlan tc_plan(int M, int N, int K, int sms);
// Work items of CTA b of the plan's grid, in the order the kernel computes
// them: (tile, k0, k1) triples into out[3 i ..] for i < max_items (host
// arithmetic only). Returns the number of items.
int tc_items(const TcPlan& plan, int b, int max_items, int32_t* out);
// x (fp32 / bf16, or int8 x_q with xin == kXinI8) -> fp16 operand xperm [M][K]
// (transposed 16-code blocks scaled by 4^-i), token sums rowsum [M], and for
// float input the scales scale_out [M] and optionally int8 codes xq_out; also
// zeroes zero_bytes (a multiple of 16) at `zero`.
cudaError_t launch_act_perm(const void* x, int xin, const float* scale_in, int M, int K, int8_t* xq_out,
                            float* scale_out, void* xperm, int* rowsum, void* zero, size_t zero_bytes,
                            cudaStream_t s);
// y (or int32 acc when out_acc) from xperm, rowsum, scale and packed weights;
// needs K % 64 == 0; sk_ws is the plan's zeroed split-tile workspace. Returns
// cudaErrorNotSupported if tensor maps cannot be made.
cudaError_t launch_gemm_tc(const void* xperm, const uint8_t* wp, const float* scale, const int* rowsum,
                           const float* gamma, void* out, bool out_acc, int M, int N, int K, const TcPlan& plan,
                           void* sk_ws, cudaStream_t s);
cudaError_t take_tc_wait_error(int* flag);

}  // namespace bl
