// Weight quantisation and packing: exact absmean gamma, ternary codes,
// four codes per byte.
//
// Passages: "BitNet 1-bit LLM 的混合精度微调技术：渐进量化策略", body, the
// quantisation-function paragraph (weight absmean = mean(|W|)) and the
// forward-pass sentence (divide by the absmean factor, round, limit to
// [-1, 1]); "穿越1比特的奇幻旅程" (2B4T summary), sections "架构创新：量化魔法的
// 背后" (absmean to {-1, 0, +1}) and "GPU端：CUDA内核的定制魔法" (four ternary
// weights per 8-bit value).
//
// gamma is the exact mean of |W| rounded once to fp32. Every finite fp32 value
// is an integer multiple of 2^-149, so sum |W| is an exact integer in those
// units (below 2^309 for N*K < 2^32); the kernels below compute it without any
// rounding, in an order-independent way, then divide by N*K and round once.
//
//   1. bl_absum_partials: each CTA sums its share of |W| exactly. A thread
//      keeps a 128-bit accumulator for the 32 binades below (and 4 above) the
//      CTA's sampled maximum; elements outside that window go to 254
//      per-exponent 64-bit bins in shared memory. The CTA folds both into a
//      384-bit fixed-point partial (12 x 32-bit limbs).
//   2. bl_gamma_finalize: one CTA adds the partials, divides by N*K and rounds
//      the quotient to fp32, ties to even.
//   3. bl_quant_pack: codes and packing. code = 0 iff |w| <= d/2 with
//      d = fp32(gamma + 1e-5), which equals clip(rint(fp32(w/d)), -1, 1) for
//      every finite w (see ternary_field in common.cuh).

#include "common.cuh"
#include "kernels.cuh"

namespace bl {

namespace {

constexpr int kLimbs = 12;            // 384-bit fixed point, units of 2^-149
constexpr int kSmemLimbs = 16;        // headroom for shifted pieces
constexpr int kBins = 256;

// |w| = m * 2^e1 in units of 2^-149 (e1 in [0, 253]).
BL_DEVICE void decompose_abs(float w, uint32_t& m, int& e1) {
  uint32_t b = __float_as_uint(w) & 0x7fffffffu;
  uint32_t e = b >> 23;
  m = (b & 0x7fffffu) | (e ? 0x800000u : 0u);
  e1 = e ? static_cast<int>(e) - 1 : 0;
}

// Adds v * 2^shift to 64-bit shared limbs holding 32 bits of value each.
BL_DEVICE void add_shifted_u64(unsigned long long* limbs, unsigned long long v, int shift) {
  if (v == 0) return;
  const int q = shift >> 5, r = shift & 31;
  const uint32_t w[2] = {static_cast<uint32_t>(v), static_cast<uint32_t>(v >> 32)};
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    unsigned long long piece = static_cast<unsigned long long>(w[i]) << r;   // < 2^63
    if (piece == 0) continue;
    atomicAdd(&limbs[q + i], piece & 0xffffffffull);
    if (piece >> 32) atomicAdd(&limbs[q + i + 1], piece >> 32);
  }
}

struct Acc128 {
  unsigned long long lo, hi;
};

BL_DEVICE void acc_add(Acc128& a, unsigned long long v) {
  unsigned long long s = a.lo + v;
  a.hi += (s < a.lo) ? 1ull : 0ull;
  a.lo = s;
}

BL_DEVICE void acc_add(Acc128& a, const Acc128& b) {
  unsigned long long s = a.lo + b.lo;
  a.hi += b.hi + ((s < a.lo) ? 1ull : 0ull);
  a.lo = s;
}

}  // namespace

__global__ void __launch_bounds__(kAbsumThreads)
bl_absum_partials(const float4* __restrict__ w4, uint64_t n4, uint32_t* __restrict__ partials) {
  __shared__ unsigned long long s_bins[kBins];
  __shared__ unsigned long long s_limbs[kSmemLimbs];
  __shared__ int s_emax;

  const int tid = threadIdx.x;
  for (int i = tid; i < kBins; i += blockDim.x) s_bins[i] = 0ull;
  if (tid < kSmemLimbs) s_limbs[tid] = 0ull;
  if (tid == 0) s_emax = 0;
  __syncthreads();

  const uint64_t stride = static_cast<uint64_t>(gridDim.x) * blockDim.x;
  const uint64_t first = static_cast<uint64_t>(blockIdx.x) * blockDim.x + tid;

  // Window base from a sample: the largest exponent among this CTA's first float4s.
  {
    int e_loc = 0;
    if (first < n4) {
      float4 v = w4[first];
      uint32_t m; int e1;
      decompose_abs(v.x, m, e1); e_loc = max(e_loc, e1);
      decompose_abs(v.y, m, e1); e_loc = max(e_loc, e1);
      decompose_abs(v.z, m, e1); e_loc = max(e_loc, e1);
      decompose_abs(v.w, m, e1); e_loc = max(e_loc, e1);
    }
    atomicMax(&s_emax, e_loc);
  }
  __syncthreads();
  // window [base, base + 31]: 4 binades above the sample maximum, 27 below
  const int base = max(0, min(s_emax + 4, 253) - 31);

  Acc128 acc{0ull, 0ull};
  auto take = [&](float x) {
    uint32_t m; int e1;
    decompose_abs(x, m, e1);
    const unsigned d = static_cast<unsigned>(e1 - base);
    if (d < 32u) {
      acc_add(acc, static_cast<unsigned long long>(m) << d);
    } else if (m) {
      atomicAdd(&s_bins[e1], static_cast<unsigned long long>(m));
    }
  };

  uint64_t i = first;
  for (; i + 3 * stride < n4; i += 4 * stride) {
    float4 v0 = w4[i], v1 = w4[i + stride], v2 = w4[i + 2 * stride], v3 = w4[i + 3 * stride];
    take(v0.x); take(v0.y); take(v0.z); take(v0.w);
    take(v1.x); take(v1.y); take(v1.z); take(v1.w);
    take(v2.x); take(v2.y); take(v2.z); take(v2.w);
    take(v3.x); take(v3.y); take(v3.z); take(v3.w);
  }
  for (; i < n4; i += stride) {
    float4 v = w4[i];
    take(v.x); take(v.y); take(v.z); take(v.w);
  }

  // warp-reduce the 128-bit window accumulators
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    Acc128 other;
    other.lo = __shfl_down_sync(0xffffffffu, acc.lo, o);
    other.hi = __shfl_down_sync(0xffffffffu, acc.hi, o);
    acc_add(acc, other);
  }
  __syncthreads();   // bins complete
  if ((tid & 31) == 0) {
    add_shifted_u64(s_limbs, acc.lo, base);
    add_shifted_u64(s_limbs, acc.hi, base + 64);
  }
  for (int e = tid; e < kBins; e += blockDim.x) add_shifted_u64(s_limbs, s_bins[e], e);
  __syncthreads();
  if (tid == 0) {
    unsigned long long carry = 0;
    uint32_t* out = partials + static_cast<size_t>(blockIdx.x) * kPartialWords;
    for (int l = 0; l < kLimbs; ++l) {
      unsigned long long v = s_limbs[l] + carry;
      out[l] = static_cast<uint32_t>(v);
      carry = v >> 32;
    }
    // (the total is below 2^309 for N*K < 2^32, so no carry leaves limb 11)
  }
}

namespace {

BL_DEVICE uint32_t get_bit(const uint32_t* q, int pos) { return (q[pos >> 5] >> (pos & 31)) & 1u; }

BL_DEVICE bool any_below(const uint32_t* q, int pos) {   // any bit in [0, pos)
  const int li = pos >> 5, r = pos & 31;
  for (int l = 0; l < li; ++l)
    if (q[l]) return true;
  return r ? (q[li] & ((1u << r) - 1u)) != 0u : false;
}

}  // namespace

__global__ void __launch_bounds__(256)
bl_gamma_finalize(const uint32_t* __restrict__ partials, int n_partials, uint64_t count,
                  float* __restrict__ gamma) {
  __shared__ unsigned long long s_sum[kLimbs];
  const int tid = threadIdx.x;
  if (tid < kLimbs) s_sum[tid] = 0ull;
  __syncthreads();
  unsigned long long loc[kLimbs];
#pragma unroll
  for (int l = 0; l < kLimbs; ++l) loc[l] = 0ull;
  for (int c = tid; c < n_partials; c += blockDim.x) {
    const uint32_t* p = partials + static_cast<size_t>(c) * kPartialWords;
#pragma unroll
    for (int l = 0; l < kLimbs; ++l) loc[l] += p[l];
  }
#pragma unroll
  for (int l = 0; l < kLimbs; ++l)
    if (loc[l]) atomicAdd(&s_sum[l], loc[l]);
  __syncthreads();
  if (tid != 0) return;

  // normalise the exact sum S into 32-bit limbs (S < 2^309 fits in 10 limbs)
  uint32_t S[kLimbs + 1];
  unsigned long long carry = 0;
  for (int l = 0; l < kLimbs; ++l) {
    unsigned long long v = s_sum[l] + carry;
    S[l] = static_cast<uint32_t>(v);
    carry = v >> 32;
  }
  S[kLimbs] = static_cast<uint32_t>(carry);

  // Q = floor(S / count), R = S mod count (count < 2^32)
  const unsigned long long D = count;
  uint32_t Q[kLimbs + 1];
  unsigned long long rem = 0;
  for (int l = kLimbs; l >= 0; --l) {
    unsigned long long cur = (rem << 32) | S[l];
    Q[l] = static_cast<uint32_t>(cur / D);
    rem = cur % D;
  }

  // mean = (Q + rem/D) * 2^-149: round to fp32, ties to even
  int top = kLimbs;
  while (top >= 0 && Q[top] == 0u) --top;
  const int p = top < 0 ? 0 : 32 * top + (32 - __clz(Q[top]));   // bit length of Q
  const int shift = p > 24 ? p - 24 : 0;
  uint32_t mant;
  {
    const int li = shift >> 5, r = shift & 31;
    unsigned long long two = Q[li];
    if (li + 1 <= kLimbs) two |= static_cast<unsigned long long>(Q[li + 1]) << 32;
    mant = static_cast<uint32_t>(two >> r) & 0xffffffu;
  }
  bool up;
  if (shift == 0) {
    const unsigned long long twice = rem * 2ull;
    up = twice > D || (twice == D && (mant & 1u));
  } else {
    const bool guard = get_bit(Q, shift - 1);
    const bool sticky = any_below(Q, shift - 1) || rem != 0ull;
    up = guard && (sticky || (mant & 1u));
  }
  unsigned long long bits = (static_cast<unsigned long long>(shift) << 23) + mant + (up ? 1u : 0u);
  if (bits >= 0x7f800000ull) bits = 0x7f800000ull;   // unreachable for finite inputs
  *gamma = __uint_as_float(static_cast<uint32_t>(bits));
}

// 16 weights -> 4 packed bytes (one 32-bit word).
BL_DEVICE uint32_t pack16(const float4& a, const float4& b, const float4& c, const float4& d, float h) {
  uint32_t r = 0;
  r |= ternary_field(a.x, h) << 0;  r |= ternary_field(a.y, h) << 2;
  r |= ternary_field(a.z, h) << 4;  r |= ternary_field(a.w, h) << 6;
  r |= ternary_field(b.x, h) << 8;  r |= ternary_field(b.y, h) << 10;
  r |= ternary_field(b.z, h) << 12; r |= ternary_field(b.w, h) << 14;
  r |= ternary_field(c.x, h) << 16; r |= ternary_field(c.y, h) << 18;
  r |= ternary_field(c.z, h) << 20; r |= ternary_field(c.w, h) << 22;
  r |= ternary_field(d.x, h) << 24; r |= ternary_field(d.y, h) << 26;
  r |= ternary_field(d.z, h) << 28; r |= ternary_field(d.w, h) << 30;
  return r;
}

__global__ void __launch_bounds__(256)
bl_quant_pack(const float4* __restrict__ w4, uint64_t n_bytes, const float* __restrict__ gamma,
              uint32_t* __restrict__ wp_words) {
  const float d = __fadd_rn(*gamma, kEpsGamma);
  const float h = 0.5f * d;                 // exact: d is a normal fp32
  const uint64_t n_words = n_bytes >> 2;
  const uint64_t stride = static_cast<uint64_t>(gridDim.x) * blockDim.x;
  for (uint64_t i = static_cast<uint64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n_words; i += stride) {
    const float4* src = w4 + 4 * i;
    float4 a = __ldcs(src), b = __ldcs(src + 1), c = __ldcs(src + 2), e = __ldcs(src + 3);
    wp_words[i] = pack16(a, b, c, e, h);
  }
  // tail: up to three bytes when N*K/4 is not a multiple of 4
  const uint64_t t = (static_cast<uint64_t>(blockIdx.x) * blockDim.x + threadIdx.x);
  const uint64_t tb = n_words * 4 + t;
  if (tb < n_bytes) {
    float4 v = w4[tb];
    uint8_t* wp = reinterpret_cast<uint8_t*>(wp_words);
    wp[tb] = static_cast<uint8_t>(ternary_field(v.x, h) | (ternary_field(v.y, h) << 2) |
                                  (ternary_field(v.z, h) << 4) | (ternary_field(v.w, h) << 6));
  }
}

}  // namespace bl
