// C-ABI entry points: argument validation, kernel choice and launches.
// Every function validates on the host before enqueueing anything, launches
// on the caller's stream and never synchronises.

#include <cstdio>
#include <cstdarg>
#include <string>

#include "bitlinear.h"
#include "common.cuh"
#include "kernels.cuh"

namespace {

thread_local std::string g_last_error;

bl_status fail(bl_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

constexpr int64_t kMaxK = 65536;

bl_status check_dims(int64_t M, int64_t N, int64_t K, bool need_m) {
  if ((need_m && M <= 0) || N <= 0 || K <= 0)
    return fail(BL_ERR_INVALID_ARG, "dimensions must be positive (M=%lld N=%lld K=%lld)",
                (long long)M, (long long)N, (long long)K);
  if (K % 4) return fail(BL_ERR_INVALID_ARG, "K=%lld is not a multiple of 4", (long long)K);
  if (K > kMaxK) return fail(BL_ERR_UNSUPPORTED, "K=%lld exceeds %lld", (long long)K, (long long)kMaxK);
  if (N * K >= (int64_t(1) << 32))
    return fail(BL_ERR_UNSUPPORTED, "N*K=%lld must be below 2^32", (long long)(N * K));
  if (need_m && M > (int64_t(1) << 31) - 1) return fail(BL_ERR_UNSUPPORTED, "M=%lld too large", (long long)M);
  return BL_OK;
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 148;
  return n;
}

// ---- GEMV / small-M contraction launcher (any M; tokens in groups of mt per CTA)
bl_status launch_gemv(const uint8_t* wp, const int8_t* xq, const float* scale, const float* gamma, void* out,
                      int64_t M, int64_t N, int64_t K, bl::GemvOut mode, cudaStream_t s) {
  const bool vec = (K % 64 == 0) && aligned(wp, 16) && aligned(xq, 16);
  const int64_t Kp = (K + 63) / 64 * 64;
  int mt = M == 1 ? 1 : (M == 2 ? 2 : 4);
  while (mt > 1 && mt * Kp > 200 * 1024) mt >>= 1;
  const int warps_per_cta = bl::kGemvThreads / 32;
  const int64_t want = (N + warps_per_cta - 1) / warps_per_cta;
  const int64_t cap = static_cast<int64_t>(sm_count()) * 4;
  const int gx = static_cast<int>(want < cap ? want : cap);
  if ((M + mt - 1) / mt > 65535) return fail(BL_ERR_UNSUPPORTED, "M=%lld too large for the GEMV grid", (long long)M);
  cudaError_t e = bl::launch_gemv(wp, xq, scale, gamma, out, static_cast<int>(M), static_cast<int>(N),
                                  static_cast<int>(K), mode, vec, mt, gx, s);
  if (e != cudaSuccess) return fail(BL_ERR_CUDA, "bl_gemv_w2a8: %s", cudaGetErrorString(e));
  return BL_OK;
}

bl_status launch_act_quant(const void* x, bl_dtype dt, int64_t M, int64_t K, int8_t* xq, float* scale,
                           cudaStream_t s) {
  cudaError_t e = bl::launch_act_quant(x, dt == BL_BF16, static_cast<int>(M), static_cast<int>(K), xq, scale, s);
  if (e != cudaSuccess) return fail(BL_ERR_CUDA, "bl_act_quant: %s", cudaGetErrorString(e));
  return BL_OK;
}

// Rows of W per CTA for the mma.sync contraction (bl_decode_mma), or 0 when it
// does not take this shape (K % 64 != 0, or the shared-memory block is too big).
int decode_rows(int64_t N, int64_t K) {
  if (K % 64 != 0) return 0;
  const int sms = sm_count();
  int64_t rows = (N + sms - 1) / sms;
  while (rows > 16 && bl::decode_smem_bytes(static_cast<int>(rows), static_cast<int>(K)) > bl::kMaxSmemPerCta)
    rows = (rows + 1) / 2;
  if (bl::decode_smem_bytes(static_cast<int>(rows), static_cast<int>(K)) > bl::kMaxSmemPerCta) return 0;
  return static_cast<int>(rows);
}

bl_status launch_decode(const uint8_t* wp, const void* x, int xin, const float* scale_in, const float* gamma,
                        void* out, bool out_acc, int8_t* xq_out, float* scale_out, int64_t M, int64_t N, int64_t K,
                        int rows, cudaStream_t s) {
  cudaError_t e = bl::launch_decode(wp, x, xin, scale_in, gamma, out, out_acc, xq_out, scale_out, static_cast<int>(M),
                                    static_cast<int>(N), static_cast<int>(K), rows, s);
  if (e != cudaSuccess) return fail(BL_ERR_CUDA, "bl_decode_mma: %s", cudaGetErrorString(e));
  return BL_OK;
}

// Largest M that the forward quantises inside the contraction kernel.
constexpr int64_t kFusedMaxM = 8;

bool use_tc(int64_t M, int64_t K) { return M >= bl::kTcMinM && K % 64 == 0; }

// Workspace of the CUDA-core paths: int8 codes (caller layout or transposed
// blocks) [M][K], then int token sums [M], then fp32 scales [M].
size_t small_workspace_bytes(int64_t M, int64_t K) {
  return align_up(static_cast<size_t>(M) * static_cast<size_t>(K), 256) + 2 * align_up(static_cast<size_t>(M) * 4, 256);
}

// Workspace of the tensor-core path: fp16 operand, token sums, scales, then
// the contraction's split-tile buffer and counters.
struct TcWorkspace {
  void* xperm;
  int* rowsum;
  float* scale;
  void* sk;
};

bl::TcPlan tc_plan_for(int64_t M, int64_t N, int64_t K) {
  return bl::tc_plan(static_cast<int>(M), static_cast<int>(N), static_cast<int>(K), sm_count());
}

size_t tc_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  return align_up(static_cast<size_t>(M) * static_cast<size_t>(K) * 2, 256) +
         2 * align_up(static_cast<size_t>(M) * 4, 256) + tc_plan_for(M, N, K).sk_bytes;
}

TcWorkspace tc_workspace(void* ws, int64_t M, int64_t K) {
  uint8_t* b = static_cast<uint8_t*>(ws);
  TcWorkspace t;
  t.xperm = b;
  b += align_up(static_cast<size_t>(M) * static_cast<size_t>(K) * 2, 256);
  t.rowsum = reinterpret_cast<int*>(b);
  b += align_up(static_cast<size_t>(M) * 4, 256);
  t.scale = reinterpret_cast<float*>(b);
  b += align_up(static_cast<size_t>(M) * 4, 256);
  t.sk = b;
  return t;
}

bl_status run_tc(const void* x, int xin, const float* scale_in, const uint8_t* Wp, const float* gamma, void* out,
                 bool out_acc, int8_t* xq_out, float* scale_out, int64_t M, int64_t N, int64_t K, void* ws,
                 cudaStream_t s) {
  TcWorkspace t = tc_workspace(ws, M, K);
  const bl::TcPlan plan = tc_plan_for(M, N, K);
  float* sc = xin == bl::kXinI8 ? const_cast<float*>(scale_in) : (scale_out ? scale_out : t.scale);
  cudaError_t e = bl::launch_act_perm(x, xin, scale_in, static_cast<int>(M), static_cast<int>(K), xq_out,
                                      xin == bl::kXinI8 ? nullptr : sc, t.xperm, t.rowsum, t.sk, plan.sk_bytes, s);
  if (e != cudaSuccess) return fail(BL_ERR_CUDA, "bl_act_perm: %s", cudaGetErrorString(e));
  e = bl::launch_gemm_tc(t.xperm, Wp, sc, t.rowsum, gamma, out, out_acc, static_cast<int>(M), static_cast<int>(N),
                         static_cast<int>(K), plan, t.sk, s);
  if (e != cudaSuccess) return fail(BL_ERR_CUDA, "bl_gemm_tc: %s", cudaGetErrorString(e));
  return BL_OK;
}

// Launch plan of the one-kernel dp4a GEMV (M <= 4); smem == 0 when it does not apply.
struct Dp4aPlan {
  int rows = 0;
  size_t smem = 0;
};

Dp4aPlan dp4a_plan(int64_t M, int64_t N, int64_t K) {
  Dp4aPlan p;
  if (M > bl::kGemvDp4aMaxM) return p;
  p.smem = bl::gemv_dp4a_plan(static_cast<int>(M), static_cast<int>(N), static_cast<int>(K), sm_count(), &p.rows);
  return p;
}

bl_status launch_dp4a(const uint8_t* wp, const void* x, int xin, const float* scale_in, const float* gamma, void* out,
                      bool out_acc, int8_t* xq_out, float* scale_out, int64_t M, int64_t N, int64_t K,
                      const Dp4aPlan& p, cudaStream_t s) {
  cudaError_t e = bl::launch_gemv_dp4a(wp, x, xin, scale_in, gamma, out, out_acc, xq_out, scale_out,
                                       static_cast<int>(M), static_cast<int>(N), static_cast<int>(K), p.rows, p.smem, s);
  if (e != cudaSuccess) return fail(BL_ERR_CUDA, "bl_gemv_dp4a: %s", cudaGetErrorString(e));
  return BL_OK;
}

// Launch plan of the two-kernel dp4a GEMV (M <= 4, shapes the one-kernel form
// does not take); smem == 0 when it does not apply.
struct GemvPlan {
  int rows = 0, parts = 0;
  size_t smem = 0;
};

GemvPlan gemv_plan(int64_t M, int64_t N, int64_t K) {
  GemvPlan p;
  if (M > bl::kGemvFusedMaxM) return p;
  p.smem = bl::gemv_fused_plan(static_cast<int>(M), static_cast<int>(N), static_cast<int>(K), sm_count(), &p.rows,
                               &p.parts);
  return p;
}

bl_status launch_gemv_fused(const uint8_t* wp, const void* x, int xin, const float* scale_in, const float* gamma,
                            void* out, bool out_acc, int8_t* xq_out, float* scale_out, int64_t M, int64_t N,
                            int64_t K, const GemvPlan& p, void* workspace, cudaStream_t s) {
  cudaError_t e = bl::launch_gemv_fused(wp, x, xin, scale_in, gamma, out, out_acc, xq_out, scale_out,
                                        static_cast<int>(M), static_cast<int>(N), static_cast<int>(K), p.rows, p.parts,
                                        p.smem, workspace, s);
  if (e != cudaSuccess) return fail(BL_ERR_CUDA, "bl_act_tq + bl_gemv_w: %s", cudaGetErrorString(e));
  return BL_OK;
}

}  // namespace

namespace bl {
// Lets entry points defined in other files record their thread-local message.
bl_status record_error(bl_status st, const char* msg) { return fail(st, "%s", msg); }
}  // namespace bl

extern "C" {

const char* bitlinear_strerror(bl_status st) {
  switch (st) {
    case BL_OK: return "ok";
    case BL_ERR_INVALID_ARG: return "invalid argument";
    case BL_ERR_UNSUPPORTED: return "unsupported arguments";
    case BL_ERR_CUDA: return "CUDA error";
    case BL_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
  }
  return "unknown status";
}

const char* bitlinear_last_error(void) { return g_last_error.c_str(); }

int bitlinear_version(void) { return 1; }

bl_status bitlinear_device_error(int* flag) {
  g_last_error.clear();
  if (!flag) return fail(BL_ERR_INVALID_ARG, "null pointer (flag)");
  int a = 0, b = 0, c = 0, d = 0, f = 0;
  cudaError_t e = bl::take_wait_error(&a);
  if (e == cudaSuccess) e = bl::take_gemv_wait_error(&b);
  if (e == cudaSuccess) e = bl::take_tc_wait_error(&c);
  if (e == cudaSuccess) e = bl::take_pack_wait_error(&d);
  if (e == cudaSuccess) e = bl::take_dp4a_wait_error(&f);
  if (e != cudaSuccess) return fail(BL_ERR_CUDA, "bitlinear_device_error: %s", cudaGetErrorString(e));
  *flag = a | b | c | d | f;
  return BL_OK;
}

bl_status bitlinear_tc_schedule(int64_t M, int64_t N, int64_t K, int sms, int32_t* plan, int32_t* n_items,
                                int32_t* items, int max_items) {
  g_last_error.clear();
  if (bl_status st = check_dims(M, N, K, true)) return st;
  if (K % 64) return fail(BL_ERR_INVALID_ARG, "K=%lld is not a multiple of 64", (long long)K);
  if (sms < 1 || sms > 4096) return fail(BL_ERR_INVALID_ARG, "sms=%d out of range 1..4096", sms);
  if (!plan) return fail(BL_ERR_INVALID_ARG, "null pointer (plan)");
  if (items && max_items < 1) return fail(BL_ERR_INVALID_ARG, "max_items=%d must be positive with items", max_items);
  const bl::TcPlan p = bl::tc_plan(static_cast<int>(M), static_cast<int>(N), static_cast<int>(K), sms);
  const int32_t vals[9] = {p.bn,       p.grid,     p.n_tiles_n,
                           p.k_iters,  p.dp_tiles, p.sk_tiles,
                           p.sk_ctas,  static_cast<int32_t>((M + p.bn - 1) / p.bn),
                           static_cast<int32_t>(p.sk_bytes)};
  for (int i = 0; i < 9; ++i) plan[i] = vals[i];
  int most = 0;
  for (int b = 0; b < p.grid; ++b) {
    const int n = bl::tc_items(p, b, items ? max_items : 0,
                               items ? items + static_cast<size_t>(b) * max_items * 3 : nullptr);
    if (n_items) n_items[b] = n;
    most = n > most ? n : most;
  }
  if (items && most > max_items)
    return fail(BL_ERR_INVALID_ARG, "a CTA has %d work items, more than max_items=%d", most, max_items);
  return BL_OK;
}

size_t bitlinear_pack_workspace_bytes(int64_t N, int64_t K) {
  (void)N;
  (void)K;
  return static_cast<size_t>(bl::kMaxAbsumCtas) * bl::kPartialWords * sizeof(uint32_t);
}

namespace {

bl_status check_pack_args(const float* W, int64_t N, int64_t K, const void* Wp_or_null, const void* gamma) {
  if (bl_status st = check_dims(1, N, K, false)) return st;
  if (!W || !gamma) return fail(BL_ERR_INVALID_ARG, "null pointer (W or gamma)");
  if (!aligned(W, 16)) return fail(BL_ERR_INVALID_ARG, "W must be 16-byte aligned");
  if (Wp_or_null && !aligned(Wp_or_null, 16)) return fail(BL_ERR_INVALID_ARG, "Wp must be 16-byte aligned");
  if (!aligned(gamma, 4)) return fail(BL_ERR_INVALID_ARG, "gamma must be 4-byte aligned");
  return BL_OK;
}

// One wave of ring CTAs, each with at least one stage of work.
uint64_t ring_grid(uint64_t stages, int per_sm) {
  const uint64_t wave = static_cast<uint64_t>(sm_count()) * static_cast<uint64_t>(per_sm);
  uint64_t g = stages < wave ? stages : wave;
  return g < 1 ? 1 : g;
}

// Exact-sum partials of |W| into `partials`; returns their count in
// *n_partials. With mask_gamma, only |w| > fp32(factor x *mask_gamma) count.
bl_status run_absum(const float* W, int64_t N, int64_t K, uint32_t* partials, int* n_partials,
                    const float* mask_gamma, float factor, cudaStream_t s) {
  const int per_sm = bl::absum_ctas_per_sm(mask_gamma != nullptr);
  if (per_sm <= 0) return fail(BL_ERR_CUDA, "bl_absum_partials: cannot reserve %u bytes of shared memory", bl::kRingSmem);
  const uint64_t n4 = static_cast<uint64_t>(N) * static_cast<uint64_t>(K) / 4;
  uint64_t ga = ring_grid((n4 + bl::kRingStageF4 - 1) / bl::kRingStageF4, per_sm);
  if (ga > static_cast<uint64_t>(bl::kMaxAbsumCtas)) ga = bl::kMaxAbsumCtas;
  cudaError_t e = bl::launch_absum(reinterpret_cast<const float4*>(W), n4, partials, mask_gamma, factor,
                                   static_cast<unsigned>(ga), s);
  if (e != cudaSuccess) return fail(BL_ERR_CUDA, "bl_absum_partials: %s", cudaGetErrorString(e));
  *n_partials = static_cast<int>(ga);
  return BL_OK;
}

bl_status run_finalize(const uint32_t* partials, int n_partials, int64_t N, int64_t K, float* out, cudaStream_t s) {
  const uint64_t nk = static_cast<uint64_t>(N) * static_cast<uint64_t>(K);
  cudaError_t e = bl::launch_pdl(bl::bl_gamma_finalize, dim3(1), dim3(256), 0, s, partials, n_partials, nk, out);
  if (e != cudaSuccess) return fail(BL_ERR_CUDA, "bl_gamma_finalize: %s", cudaGetErrorString(e));
  return BL_OK;
}

bl_status run_absmean(const float* W, int64_t N, int64_t K, float* gamma, void* workspace, cudaStream_t s) {
  uint32_t* partials = static_cast<uint32_t*>(workspace);
  int n_partials = 0;
  if (bl_status st = run_absum(W, N, K, partials, &n_partials, nullptr, 0.f, s)) return st;
  return run_finalize(partials, n_partials, N, K, gamma, s);
}

// Codes and packing (see launch_quant_pack).
bl_status run_quantize_pack(const float* W, int64_t N, int64_t K, const float* gamma_in, const uint32_t* partials,
                            int n_partials, float* scale_out, uint8_t* Wp, int rule, float factor, cudaStream_t s) {
  const uint64_t n_bytes = static_cast<uint64_t>(N) * static_cast<uint64_t>(K) / 4;
  cudaError_t e = bl::launch_quant_pack(reinterpret_cast<const float4*>(W), n_bytes, gamma_in, partials, n_partials,
                                        scale_out, reinterpret_cast<uint32_t*>(Wp), rule, factor, sm_count(), s);
  if (e != cudaSuccess) return fail(BL_ERR_CUDA, "bl_quant_pack: %s", cudaGetErrorString(e));
  return BL_OK;
}

// The whole packing by one rule. absmean and alpha-round: the exact sum, then
// the packing pass, which combines gamma itself and writes the scale. The
// threshold rule: gamma into *scale, the masked exact sum (reading gamma
// there), the packing pass (reading it too), and last the masked mean into
// *scale; each kernel reads gamma only after its dependency wait, so the
// final write cannot overtake a read.
bl_status run_pack(const float* W, int64_t N, int64_t K, int rule, float factor, uint8_t* Wp, float* scale,
                   void* workspace, cudaStream_t s) {
  uint32_t* partials = static_cast<uint32_t*>(workspace);
  int n_partials = 0;
  if (bl_status st = run_absum(W, N, K, partials, &n_partials, nullptr, 0.f, s)) return st;
  if (rule != bl::kRuleThreshold)
    return run_quantize_pack(W, N, K, nullptr, partials, n_partials, scale, Wp, rule, factor, s);
  if (bl_status st = run_finalize(partials, n_partials, N, K, scale, s)) return st;
  if (bl_status st = run_absum(W, N, K, partials, &n_partials, scale, factor, s)) return st;
  if (bl_status st = run_quantize_pack(W, N, K, scale, nullptr, 0, nullptr, Wp, rule, factor, s)) return st;
  return run_finalize(partials, n_partials, N, K, scale, s);
}

bl_status check_pack_workspace(int64_t N, int64_t K, const void* workspace, size_t ws_bytes) {
  if (!workspace || !aligned(workspace, 256) || ws_bytes < bitlinear_pack_workspace_bytes(N, K))
    return fail(BL_ERR_WORKSPACE, "pack workspace needs %zu bytes, 256-byte aligned",
                bitlinear_pack_workspace_bytes(N, K));
  return BL_OK;
}

}  // namespace

bl_status bitlinear_absmean(const float* W, int64_t N, int64_t K, float* gamma, void* workspace, size_t ws_bytes,
                            bl_stream_t stream) {
  g_last_error.clear();
  if (bl_status st = check_pack_args(W, N, K, nullptr, gamma)) return st;
  if (bl_status st = check_pack_workspace(N, K, workspace, ws_bytes)) return st;
  return run_absmean(W, N, K, gamma, workspace, reinterpret_cast<cudaStream_t>(stream));
}

bl_status bitlinear_quantize_pack(const float* W, int64_t N, int64_t K, const float* gamma, uint8_t* Wp,
                                  bl_stream_t stream) {
  g_last_error.clear();
  if (bl_status st = check_pack_args(W, N, K, Wp, gamma)) return st;
  if (!Wp) return fail(BL_ERR_INVALID_ARG, "null pointer (Wp)");
  return run_quantize_pack(W, N, K, gamma, nullptr, 0, nullptr, Wp, bl::kRuleAbsmean, 0.f,
                           reinterpret_cast<cudaStream_t>(stream));
}

bl_status bitlinear_pack_weights(const float* W, int64_t N, int64_t K, uint8_t* Wp, float* gamma,
                                 void* workspace, size_t ws_bytes, bl_stream_t stream) {
  g_last_error.clear();
  if (bl_status st = check_pack_args(W, N, K, Wp, gamma)) return st;
  if (!Wp) return fail(BL_ERR_INVALID_ARG, "null pointer (Wp)");
  if (bl_status st = check_pack_workspace(N, K, workspace, ws_bytes)) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // gamma is combined inside the packing kernel, which starts streaming W
  // while the exact sum finishes
  return run_pack(W, N, K, bl::kRuleAbsmean, 0.f, Wp, gamma, workspace, s);
}

bl_status bitlinear_pack_weights_quantizer(const float* W, int64_t N, int64_t K, bl_quantizer quantizer, float factor,
                                           uint8_t* Wp, float* scale, void* workspace, size_t ws_bytes,
                                           bl_stream_t stream) {
  g_last_error.clear();
  if (bl_status st = check_pack_args(W, N, K, Wp, scale)) return st;
  if (!Wp) return fail(BL_ERR_INVALID_ARG, "null pointer (Wp)");
  int rule = bl::kRuleAbsmean;
  switch (quantizer) {
    case BL_QUANT_ABSMEAN: rule = bl::kRuleAbsmean; break;
    case BL_QUANT_ALPHA_ROUND: rule = bl::kRuleAlphaRound; break;
    case BL_QUANT_THRESHOLD: rule = bl::kRuleThreshold; break;
    default: return fail(BL_ERR_INVALID_ARG, "unknown quantizer %d", static_cast<int>(quantizer));
  }
  if (rule != bl::kRuleAbsmean && !(factor > 0.f && factor < 3.4e38f))
    return fail(BL_ERR_INVALID_ARG, "factor must be positive and finite (got %g)", static_cast<double>(factor));
  if (bl_status st = check_pack_workspace(N, K, workspace, ws_bytes)) return st;
  return run_pack(W, N, K, rule, factor, Wp, scale, workspace, reinterpret_cast<cudaStream_t>(stream));
}

bl_status bitlinear_quant_act(const void* x, bl_dtype dt, int64_t M, int64_t K, int8_t* xq, float* scale,
                              bl_stream_t stream) {
  g_last_error.clear();
  if (bl_status st = check_dims(M, 1, K, true)) return st;
  if (dt != BL_F32 && dt != BL_BF16) return fail(BL_ERR_INVALID_ARG, "unknown dtype %d", (int)dt);
  if (!x || !xq || !scale) return fail(BL_ERR_INVALID_ARG, "null pointer (x, xq or scale)");
  if (!aligned(x, 16) || !aligned(xq, 16) || !aligned(scale, 4))
    return fail(BL_ERR_INVALID_ARG, "x and xq must be 16-byte aligned, scale 4-byte aligned");
  return launch_act_quant(x, dt, M, K, xq, scale, reinterpret_cast<cudaStream_t>(stream));
}

size_t bitlinear_forward_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  if (M <= 0 || N <= 0 || K <= 0) return 0;
  if (use_tc(M, K)) return tc_workspace_bytes(M, N, K);
  if (dp4a_plan(M, N, K).smem) return 0;
  return small_workspace_bytes(M, K);
}

bl_status bitlinear_forward(const void* x, bl_dtype dt, int64_t M, const uint8_t* Wp, const float* gamma,
                            int64_t N, int64_t K, float* y, int8_t* xq_out, float* scale_out, void* workspace,
                            size_t ws_bytes, bl_stream_t stream) {
  g_last_error.clear();
  if (bl_status st = check_dims(M, N, K, true)) return st;
  if (dt != BL_F32 && dt != BL_BF16) return fail(BL_ERR_INVALID_ARG, "unknown dtype %d", (int)dt);
  if (!x || !Wp || !gamma || !y) return fail(BL_ERR_INVALID_ARG, "null pointer (x, Wp, gamma or y)");
  if (!aligned(x, 16) || !aligned(Wp, 16) || !aligned(y, 16) || !aligned(gamma, 4))
    return fail(BL_ERR_INVALID_ARG, "x, Wp and y must be 16-byte aligned, gamma 4-byte aligned");
  if (xq_out && !aligned(xq_out, 16)) return fail(BL_ERR_INVALID_ARG, "xq_out must be 16-byte aligned");
  if (scale_out && !aligned(scale_out, 4)) return fail(BL_ERR_INVALID_ARG, "scale_out must be 4-byte aligned");
  const size_t need = bitlinear_forward_workspace_bytes(M, N, K);
  if (need && (!workspace || !aligned(workspace, 256) || ws_bytes < need))
    return fail(BL_ERR_WORKSPACE, "forward workspace needs %zu bytes, 256-byte aligned", need);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int8_t* xq = xq_out ? xq_out : reinterpret_cast<int8_t*>(ws);
  float* sc = scale_out ? scale_out
                        : reinterpret_cast<float*>(ws + align_up(static_cast<size_t>(M) * static_cast<size_t>(K), 256));
  const int xin = dt == BL_BF16 ? bl::kXinBF16 : bl::kXinF32;
  if (use_tc(M, K)) return run_tc(x, xin, nullptr, Wp, gamma, y, false, xq_out, scale_out, M, N, K, workspace, s);
  const Dp4aPlan dp = dp4a_plan(M, N, K);
  if (dp.smem) return launch_dp4a(Wp, x, xin, nullptr, gamma, y, false, xq_out, scale_out, M, N, K, dp, s);
  const GemvPlan gp = gemv_plan(M, N, K);
  if (gp.smem)
    return launch_gemv_fused(Wp, x, xin, nullptr, gamma, y, false, xq_out, scale_out, M, N, K, gp, workspace, s);
  const int rows = decode_rows(N, K);
  if (rows && M <= kFusedMaxM)
    return launch_decode(Wp, x, dt == BL_BF16 ? bl::kXinBF16 : bl::kXinF32, nullptr, gamma, y, false, xq_out,
                         scale_out, M, N, K, rows, s);
  if (bl_status st = launch_act_quant(x, dt, M, K, xq, sc, s)) return st;
  if (rows) return launch_decode(Wp, xq, bl::kXinI8, sc, gamma, y, false, nullptr, nullptr, M, N, K, rows, s);
  return launch_gemv(Wp, xq, sc, gamma, y, M, N, K, bl::GemvOut::kY, s);
}

bl_status bitlinear_forward_lut(const void* x, bl_dtype dt, int64_t M, const uint8_t* Wp, const float* gamma,
                                int64_t N, int64_t K, float* y, bl_stream_t stream) {
  g_last_error.clear();
  if (bl_status st = check_dims(M, N, K, true)) return st;
  if (M != 1) return fail(BL_ERR_UNSUPPORTED, "the lookup-table GEMV takes one token (M=%lld)", (long long)M);
  if (K % 64) return fail(BL_ERR_INVALID_ARG, "K=%lld is not a multiple of 64", (long long)K);
  if (K > bl::kLutMaxK) return fail(BL_ERR_UNSUPPORTED, "K=%lld exceeds %d for the lookup-table GEMV", (long long)K, bl::kLutMaxK);
  if (dt != BL_F32 && dt != BL_BF16) return fail(BL_ERR_INVALID_ARG, "unknown dtype %d", (int)dt);
  if (!x || !Wp || !gamma || !y) return fail(BL_ERR_INVALID_ARG, "null pointer (x, Wp, gamma or y)");
  if (!aligned(x, 16) || !aligned(Wp, 16) || !aligned(y, 4) || !aligned(gamma, 4))
    return fail(BL_ERR_INVALID_ARG, "x and Wp must be 16-byte aligned, y and gamma 4-byte aligned");
  const cudaError_t e = bl::launch_gemv_lut(Wp, x, dt == BL_BF16, gamma, y, static_cast<int>(N), static_cast<int>(K),
                                            sm_count(), reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(BL_ERR_CUDA, "bl_gemv_lut: %s", cudaGetErrorString(e));
  return BL_OK;
}

bl_status bitlinear_pack_weights_grouped(const float* W, int64_t N, int64_t K, uint8_t* Wp, float* gammas,
                                         bl_stream_t stream) {
  g_last_error.clear();
  if (bl_status st = check_dims(1, N, K, false)) return st;
  if (K % 64) return fail(BL_ERR_INVALID_ARG, "K=%lld is not a multiple of 64 (the group size)", (long long)K);
  if (!W || !Wp || !gammas) return fail(BL_ERR_INVALID_ARG, "null pointer (W, Wp or gammas)");
  if (!aligned(W, 16) || !aligned(Wp, 16) || !aligned(gammas, 4))
    return fail(BL_ERR_INVALID_ARG, "W and Wp must be 16-byte aligned, gammas 4-byte aligned");
  const cudaError_t e =
      bl::launch_pack_grouped(W, N, K, Wp, gammas, sm_count(), reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(BL_ERR_CUDA, "bl_pack_grouped: %s", cudaGetErrorString(e));
  return BL_OK;
}

size_t bitlinear_forward_grouped_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  (void)N;
  if (M <= 0 || K <= 0) return 0;
  return bl::forward_grouped_workspace(M, K);
}

bl_status bitlinear_forward_grouped(const void* x, bl_dtype dt, int64_t M, const uint8_t* Wp, const float* gammas,
                                    int64_t N, int64_t K, float* y, int8_t* xq_out, float* scale_out, void* workspace,
                                    size_t ws_bytes, bl_stream_t stream) {
  g_last_error.clear();
  if (bl_status st = check_dims(M, N, K, true)) return st;
  if (K % 64) return fail(BL_ERR_INVALID_ARG, "K=%lld is not a multiple of 64 (the group size)", (long long)K);
  if (dt != BL_F32 && dt != BL_BF16) return fail(BL_ERR_INVALID_ARG, "unknown dtype %d", (int)dt);
  if (M > 65535) return fail(BL_ERR_UNSUPPORTED, "M=%lld exceeds 65535 for the grouped forward", (long long)M);
  if (!x || !Wp || !gammas || !y) return fail(BL_ERR_INVALID_ARG, "null pointer (x, Wp, gammas or y)");
  if (!aligned(x, 16) || !aligned(Wp, 16) || !aligned(y, 4) || !aligned(gammas, 4))
    return fail(BL_ERR_INVALID_ARG, "x and Wp must be 16-byte aligned, y and gammas 4-byte aligned");
  if (xq_out && !aligned(xq_out, 16)) return fail(BL_ERR_INVALID_ARG, "xq_out must be 16-byte aligned");
  if (scale_out && !aligned(scale_out, 4)) return fail(BL_ERR_INVALID_ARG, "scale_out must be 4-byte aligned");
  const size_t need = bitlinear_forward_grouped_workspace_bytes(M, N, K);
  if (!workspace || !aligned(workspace, 256) || ws_bytes < need)
    return fail(BL_ERR_WORKSPACE, "grouped forward workspace needs %zu bytes, 256-byte aligned", need);
  const cudaError_t e =
      bl::launch_forward_grouped(x, dt == BL_BF16, static_cast<int>(M), static_cast<int>(N), static_cast<int>(K), Wp,
                                 gammas, y, xq_out, scale_out, workspace, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(BL_ERR_CUDA, "grouped forward: %s", cudaGetErrorString(e));
  return BL_OK;
}

size_t bitlinear_gemm_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  if (M <= 0 || N <= 0 || K <= 0) return 0;
  if (use_tc(M, K)) return tc_workspace_bytes(M, N, K);
  if (dp4a_plan(M, N, K).smem) return 0;
  if (gemv_plan(M, N, K).smem) return small_workspace_bytes(M, K);
  return 0;
}

bl_status bitlinear_gemm(const int8_t* xq, const float* scale, int64_t M, const uint8_t* Wp, const float* gamma,
                         int64_t N, int64_t K, float* y, void* workspace, size_t ws_bytes, bl_stream_t stream) {
  g_last_error.clear();
  if (bl_status st = check_dims(M, N, K, true)) return st;
  if (!xq || !scale || !Wp || !gamma || !y) return fail(BL_ERR_INVALID_ARG, "null pointer (xq, scale, Wp, gamma or y)");
  if (!aligned(xq, 16) || !aligned(Wp, 16) || !aligned(y, 16) || !aligned(scale, 4) || !aligned(gamma, 4))
    return fail(BL_ERR_INVALID_ARG, "xq, Wp and y must be 16-byte aligned, scale and gamma 4-byte aligned");
  const size_t need = bitlinear_gemm_workspace_bytes(M, N, K);
  if (need && (!workspace || !aligned(workspace, 256) || ws_bytes < need))
    return fail(BL_ERR_WORKSPACE, "gemm workspace needs %zu bytes, 256-byte aligned", need);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (use_tc(M, K)) return run_tc(xq, bl::kXinI8, scale, Wp, gamma, y, false, nullptr, nullptr, M, N, K, workspace, s);
  const Dp4aPlan dp = dp4a_plan(M, N, K);
  if (dp.smem) return launch_dp4a(Wp, xq, bl::kXinI8, scale, gamma, y, false, nullptr, nullptr, M, N, K, dp, s);
  const GemvPlan gp = gemv_plan(M, N, K);
  if (gp.smem) return launch_gemv_fused(Wp, xq, bl::kXinI8, scale, gamma, y, false, nullptr, nullptr, M, N, K, gp, workspace, s);
  if (const int rows = decode_rows(N, K))
    return launch_decode(Wp, xq, bl::kXinI8, scale, gamma, y, false, nullptr, nullptr, M, N, K, rows, s);
  return launch_gemv(Wp, xq, scale, gamma, y, M, N, K, bl::GemvOut::kY, s);
}

size_t bitlinear_gemm_i32_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  return bitlinear_gemm_workspace_bytes(M, N, K);
}

bl_status bitlinear_gemm_i32(const int8_t* xq, const uint8_t* Wp, int64_t M, int64_t N, int64_t K, int32_t* acc,
                             void* workspace, size_t ws_bytes, bl_stream_t stream) {
  g_last_error.clear();
  if (bl_status st = check_dims(M, N, K, true)) return st;
  if (!xq || !Wp || !acc) return fail(BL_ERR_INVALID_ARG, "null pointer (xq, Wp or acc)");
  if (!aligned(xq, 16) || !aligned(Wp, 16) || !aligned(acc, 16))
    return fail(BL_ERR_INVALID_ARG, "xq, Wp and acc must be 16-byte aligned");
  const size_t need = bitlinear_gemm_i32_workspace_bytes(M, N, K);
  if (need && (!workspace || !aligned(workspace, 256) || ws_bytes < need))
    return fail(BL_ERR_WORKSPACE, "gemm_i32 workspace needs %zu bytes, 256-byte aligned", need);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (use_tc(M, K)) return run_tc(xq, bl::kXinI8, nullptr, Wp, nullptr, acc, true, nullptr, nullptr, M, N, K, workspace, s);
  const Dp4aPlan dp = dp4a_plan(M, N, K);
  if (dp.smem) return launch_dp4a(Wp, xq, bl::kXinI8, nullptr, nullptr, acc, true, nullptr, nullptr, M, N, K, dp, s);
  const GemvPlan gp = gemv_plan(M, N, K);
  if (gp.smem) return launch_gemv_fused(Wp, xq, bl::kXinI8, nullptr, nullptr, acc, true, nullptr, nullptr, M, N, K, gp, workspace, s);
  if (const int rows = decode_rows(N, K))
    return launch_decode(Wp, xq, bl::kXinI8, nullptr, nullptr, acc, true, nullptr, nullptr, M, N, K, rows, s);
  return launch_gemv(Wp, xq, nullptr, nullptr, acc, M, N, K, bl::GemvOut::kAcc, s);
}

}  // extern "C"
