// Shared device helpers for the BitLinear W1.58A8 kernels (sm_103a).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "bitlinear.h"

#define BL_DEVICE __device__ __forceinline__
#define BL_HOST_DEVICE __host__ __device__ __forceinline__

namespace bl {

constexpr float kEpsGamma = 1e-5f;    // added to gamma in the quantisation divisor
constexpr float kEpsAbsmax = 1e-5f;   // floor on the per-token absmax

// Packed field of a ternary code: field = code + 1.
//   code = 0  <=>  |w| <= d/2   (w/d rounds to a value <= 0.5, and rint(0.5) = 0)
//   code = +-1 otherwise, with the sign of w.
// For a normal fp32 divisor d the two predicates agree bit for bit with
// clip(rint(RN(w/d)), -1, 1): the fp32 quotient of a value just above d/2 is
// at least 0.5 + 2^-24, because w = d/2 + ulp(d/2) gives w/d = 0.5 + 1/(2M)
// with M < 2^24 the significand of d, which lies above the midpoint
// 0.5 + 2^-25 between 0.5 and its successor.
BL_DEVICE uint32_t ternary_field(float w, float half_d) {
  return fabsf(w) > half_d ? (w > 0.f ? 2u : 0u) : 1u;
}

BL_DEVICE int dp4a_us(uint32_t a_u8x4, int b_s8x4, int c) {
  int d;
  asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a_u8x4), "r"(b_s8x4), "r"(c));
  return d;
}

BL_DEVICE int dp4a_ss(int a, int b, int c) {
  int d;
  asm("dp4a.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// 4x4 byte transpose of a 16-byte block: out word i, byte j = in word j, byte i.
BL_DEVICE void transpose4x4_bytes(uint32_t a, uint32_t b, uint32_t c, uint32_t d,
                                  uint32_t& o0, uint32_t& o1, uint32_t& o2, uint32_t& o3) {
  // pairs first: (a,b) -> bytes {a0 b0 a1 b1}, {a2 b2 a3 b3}
  uint32_t ab_lo = __byte_perm(a, b, 0x5140);
  uint32_t ab_hi = __byte_perm(a, b, 0x7362);
  uint32_t cd_lo = __byte_perm(c, d, 0x5140);
  uint32_t cd_hi = __byte_perm(c, d, 0x7362);
  o0 = __byte_perm(ab_lo, cd_lo, 0x5410);   // a0 b0 c0 d0
  o1 = __byte_perm(ab_lo, cd_lo, 0x7632);   // a1 b1 c1 d1
  o2 = __byte_perm(ab_hi, cd_hi, 0x5410);   // a2 b2 c2 d2
  o3 = __byte_perm(ab_hi, cd_hi, 0x7632);   // a3 b3 c3 d3
}

BL_DEVICE float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

BL_DEVICE int warp_sum(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Per-token scale and code, as fp32 operations with round-to-nearest-even.
BL_DEVICE float token_scale(float absmax) {
  return __fdiv_rn(127.0f, fmaxf(absmax, kEpsAbsmax));
}

BL_DEVICE int quant_code(float x, float s) {
  int q = __float2int_rn(__fmul_rn(x, s));
  return min(127, max(-128, q));
}

BL_DEVICE float bf16_to_f32(uint16_t b) { return __uint_as_float(static_cast<uint32_t>(b) << 16); }

BL_DEVICE float rescale(int acc, float gamma, float s) {
  return __fdiv_rn(__fmul_rn(static_cast<float>(acc), gamma), s);
}

// The reciprocal div_rn_recip takes: fp32(1/s) for s inside 2^-96..2^96, and
// 0 otherwise (such scales take the IEEE division).
BL_DEVICE float recip_for_div(float s) { return (s > 0x1p-96f && s < 0x1p96f) ? __frcp_rn(s) : 0.f; }

// fp32(t / s) rounded to nearest even, from r = recip_for_div(s), by
// Markstein's correction step (P. Markstein, "Computation of elementary
// functions on the IBM RISC System/6000 processor", IBM J. Res. Dev. 34(1),
// 1990): q = RN(t * r), the residual e = RN(t - q * s) in one FMA, and
// RN(q + e * r) is the correctly rounded quotient. It is taken only where
// nothing leaves the normal range: |t| inside 2^-96..2^96 (the residual keeps
// every bit) and |q| inside 2^-100..2^126 (a normal quotient whose correction
// cannot overflow). A zero t gives q, which carries the sign of t / s. Every
// other case (overflowing or underflowing quotients, scales outside
// 2^-96..2^96) takes the IEEE division.
// The IEEE division out of line, so that the unrolled loops that may need it
// keep their code small.
static __device__ __noinline__ float div_ieee(float t, float s) { return __fdiv_rn(t, s); }

BL_DEVICE float div_rn_recip(float t, float s, float r) {
  const float q = __fmul_rn(t, r);
  const float at = fabsf(t), aq = fabsf(q);
  if (r != 0.f) {
    if (t == 0.f) return q;
    if (at > 0x1p-96f && at < 0x1p96f && aq > 0x1p-100f && aq < 0x1p126f)
      return __fmaf_rn(__fmaf_rn(-q, s, t), r, q);
  }
  return div_ieee(t, s);
}

// Programmatic dependent launch. Every kernel of this library runs
//   prologue (no global reads) -> pdl_wait() -> pdl_launch_dependents() -> body
// so a grid may become resident before its predecessor ends, no read of the
// body can see a partial write of the predecessor (pdl_wait returns once the
// predecessor has completed and its memory is visible), and the dependent
// grid, released only after this grid's own wait, cannot overtake writes of
// anything earlier. Both are no-ops for a grid launched without the attribute.
BL_DEVICE void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
BL_DEVICE void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// The same pointer, opaque to the compiler: loads through it cannot be hoisted
// above the asm (read-only loads could otherwise move above pdl_wait()).
template <typename T>
BL_DEVICE T* launder(T* p) {
  T* q;
  asm volatile("mov.b64 %0, %1;" : "=l"(q) : "l"(p) : "memory");
  return q;
}

}  // namespace bl
