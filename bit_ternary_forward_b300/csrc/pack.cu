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
// Both weight passes stream W through four 16 KB shared-memory stages that
// one producer thread fills with bulk asynchronous copies (ring_produce in
// async.cuh); the consumer warps sleep on the stage barriers.
//
//   1. bl_absum_partials: each CTA sums its share of |W| exactly. Each warp
//      picks a window of 32 binades from the largest exponent among its first
//      128 weights (4 binades above it, 27 below). For a weight in the window,
//      at distance d binades above its bottom, |w| = m * 2^d window units (m
//      the 24-bit significand), which one wide multiply-add (mad.wide.u32)
//      adds to a 64-bit register accumulator; 2^d comes from a wrapping
//      funnel shift, so the sign bit needs no masking (it adds 256, a
//      multiple of 32, to the shift amount). One OR over the four shift
//      amounts of a float4 finds the weights outside the window (zeros,
//      subnormals, stragglers far from the warp's scale); their terms are
//      taken back and they go to 254 per-exponent 64-bit bins in shared
//      memory. The accumulators are folded into 96 bits after every stage,
//      and the CTA folds everything into a 384-bit fixed-point partial
//      (12 x 32-bit limbs). The masked form sums only |w| > delta (the
//      threshold quantiser's scale).
//   2. The combine adds the partials (shuffle reductions), then one thread
//      divides the top 64 bits of the exact sum by N*K and rounds the quotient
//      to fp32, ties to even, with the dropped bits and the remainder as the
//      sticky bit: inside every CTA of the fused packing pass, or in the
//      one-CTA bl_gamma_finalize.
//   3. bl_quant_pack: codes and packing. code = 0 iff |w| <= h, else the sign
//      of w, with h = fp32(gamma + 1e-5) / 2 for the absmean rule, which equals
//      clip(rint(fp32(w/d)), -1, 1) with d = fp32(gamma + 1e-5) for every
//      finite w (see ternary_field in common.cuh); the variant rules change h
//      (see the kernel).

#include "async.cuh"
#include "common.cuh"
#include "kernels.cuh"

namespace bl {

namespace {

constexpr int kLimbs = 12;            // 384-bit fixed point, units of 2^-149
constexpr int kSmemLimbs = 16;        // headroom for shifted pieces
constexpr int kBins = 256;

// (a2:a1:a0) += (hi:lo), 96-bit, carries through the flag register.
BL_DEVICE void add96(uint32_t& a0, uint32_t& a1, uint32_t& a2, uint32_t lo, uint32_t hi) {
  asm("add.cc.u32 %0, %0, %3;\n\t"
      "addc.cc.u32 %1, %1, %4;\n\t"
      "addc.u32 %2, %2, 0;"
      : "+r"(a0), "+r"(a1), "+r"(a2) : "r"(lo), "r"(hi));
}

BL_DEVICE void add96(uint32_t& a0, uint32_t& a1, uint32_t& a2, uint32_t b0, uint32_t b1, uint32_t b2) {
  asm("add.cc.u32 %0, %0, %3;\n\t"
      "addc.cc.u32 %1, %1, %4;\n\t"
      "addc.u32 %2, %2, %5;"
      : "+r"(a0), "+r"(a1), "+r"(a2) : "r"(b0), "r"(b1), "r"(b2));
}

// Adds the little-endian 32-bit words w[0..n) times 2^shift to shared limbs
// that hold 32 bits of value each in 64-bit cells (carries settle later).
template <int NW>
BL_DEVICE void add_words_shifted(unsigned long long* limbs, const uint32_t (&w)[NW], int shift) {
  const int q = shift >> 5, r = shift & 31;
  uint32_t prev = 0u;
#pragma unroll
  for (int i = 0; i <= NW; ++i) {
    const uint32_t cur = i < NW ? w[i] : 0u;
    // word i of (w << r): the high half of (cur:prev) << r
    const uint32_t piece = r ? __funnelshift_l(prev, cur, r) : cur;
    if (piece) atomicAdd(&limbs[q + i], static_cast<unsigned long long>(piece));
    prev = cur;
  }
}

BL_DEVICE int exp_field(float x) { return static_cast<int>((__float_as_uint(x) >> 23) & 0xffu); }

// a * b + c with a 64-bit addend and result (exact while it stays below 2^64).
BL_DEVICE unsigned long long mad_wide_u32(uint32_t a, uint32_t b, unsigned long long c) {
  unsigned long long r;
  asm("mad.wide.u32 %0, %1, %2, %3;" : "=l"(r) : "r"(a), "r"(b), "l"(c));
  return r;
}

}  // namespace

// Set (never cleared by a kernel) when a bounded mbarrier wait gave up.
__device__ int g_pack_wait_error;

// 1 << (s mod 32): funnel shift of (1:0) with wrap-around shift amounts.
BL_DEVICE uint32_t pow2_wrap(uint32_t s) {
  uint32_t r;
  asm("shf.l.wrap.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(0u), "r"(1u), "r"(s));
  return r;
}

// MASKED: only weights with |w| > delta = fp32(factor x gamma) are summed
// (gamma read from *gamma_in), for the threshold quantiser's scale.
template <bool MASKED>
__global__ void __launch_bounds__(kAbsumThreads + 32, 2)
bl_absum_partials(const float4* __restrict__ w4, uint64_t n4, uint32_t* __restrict__ partials,
                  const float* __restrict__ gamma_in, float factor) {
  extern __shared__ __align__(128) float4 s_ring[];        // kRingStages x kRingStageF4
  __shared__ unsigned long long s_bins[kBins];
  __shared__ unsigned long long s_limbs[kSmemLimbs];
  __shared__ __align__(8) uint64_t s_full[kRingStages], s_empty[kRingStages];
  constexpr int kConsumerWarps = kAbsumThreads / 32;
  constexpr int kPer = kRingStageF4 / kAbsumThreads;      // float4 per consumer thread and stage
  // a fold adds kPer * 4 window terms below 2^55 each: far below 2^64
  static_assert(kPer * kAbsumThreads == kRingStageF4 && kPer * 4 <= 256, "fold bound");

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int i = tid; i < kBins; i += blockDim.x) s_bins[i] = 0ull;
  if (tid < kSmemLimbs) s_limbs[tid] = 0ull;
  if (tid == 0) {
    for (int s = 0; s < kRingStages; ++s) {
      mbar_init(&s_full[s], 1);
      mbar_init(&s_empty[s], kConsumerWarps);
    }
    mbar_init_fence();
  }
  // this CTA's share: the contiguous float4 range [f0, f1), in stages of
  // kRingStageF4 (the last one shorter)
  const uint64_t f0 = n4 * blockIdx.x / gridDim.x, f1 = n4 * (blockIdx.x + 1) / gridDim.x;
  const int n_stages = static_cast<int>((f1 - f0 + kRingStageF4 - 1) / kRingStageF4);
  __syncthreads();   // barriers initialised, bins and limbs cleared
  pdl_wait();
  pdl_launch_dependents();
  w4 = launder(w4);
  bool ok = true;

  uint32_t a0 = 0u, a1 = 0u, a2 = 0u;      // 96-bit total of this thread
  int base = 0;                            // warp-uniform window bottom, units of 2^-149

  if (warp == kConsumerWarps) {
    // ---- producer: one thread keeps kRingStages bulk copies in flight
    // W is read again by the packing pass: the first kL2KeepBytes of it stay
    // in L2 at high priority, the rest streams through
    if (lane == 0)
      ok = ring_produce(s_ring, kRingStageF4 * 16u, kRingStages, w4 + f0, (f1 - f0) * 16u, s_full, s_empty,
                        f0 * 16u < kL2KeepBytes ? l2_evict_last() : l2_evict_first());
    __syncwarp();
  } else {
    // ---- consumers: thread t sums float4 t, t + kAbsumThreads, ... of every stage
    uint32_t bias = 0u;
    // the mask threshold as bits: for non-negative floats the bit patterns
    // order like the values
    const uint32_t dbits = MASKED ? __float_as_uint(__fmul_rn(factor, *launder(gamma_in))) : 0u;
    auto kept = [&](uint32_t abs_bits) { return !MASKED || abs_bits > dbits; };
    // out-of-window weights of a float4 (rare): exact per-exponent bins
    auto rare = [&](float x) {
      const uint32_t b = __float_as_uint(x) & 0x7fffffffu;
      const uint32_t e = b >> 23;
      if ((e - bias) >= 32u && b != 0u && kept(b)) {
        const uint32_t m = e ? ((b & 0x7fffffu) | 0x800000u) : b;
        atomicAdd(&s_bins[e ? e - 1u : 0u], static_cast<unsigned long long>(m));
      }
    };
    // Window terms of a float4 into acc. With the sign bit left in, the shift
    // amount (bits >> 23) - bias is the binade distance plus 256 for a
    // negative weight; 256 is a multiple of 32, so the wrapping shift gives
    // the same power of two, and a weight lies in the window iff bits 5..7
    // of that amount are clear (for either sign, and for any wrapped value).
    auto take4 = [&](const float4& v, unsigned long long& acc) {
      const uint32_t b0 = __float_as_uint(v.x), b1 = __float_as_uint(v.y);
      const uint32_t b2 = __float_as_uint(v.z), b3 = __float_as_uint(v.w);
      const uint32_t d0 = (b0 >> 23) - bias, d1 = (b1 >> 23) - bias, d2 = (b2 >> 23) - bias, d3 = (b3 >> 23) - bias;
      const uint32_t m0 = kept(b0 & 0x7fffffffu) ? (b0 & 0x7fffffu) | 0x800000u : 0u;
      const uint32_t m1 = kept(b1 & 0x7fffffffu) ? (b1 & 0x7fffffu) | 0x800000u : 0u;
      const uint32_t m2 = kept(b2 & 0x7fffffffu) ? (b2 & 0x7fffffu) | 0x800000u : 0u;
      const uint32_t m3 = kept(b3 & 0x7fffffffu) ? (b3 & 0x7fffffu) | 0x800000u : 0u;
      acc = mad_wide_u32(m0, pow2_wrap(d0), acc);
      acc = mad_wide_u32(m1, pow2_wrap(d1), acc);
      acc = mad_wide_u32(m2, pow2_wrap(d2), acc);
      acc = mad_wide_u32(m3, pow2_wrap(d3), acc);
      if ((d0 | d1 | d2 | d3) & 0xe0u) {
        // the four window terms above are exact only for in-window weights:
        // take back those of the others and bin them instead
        const uint32_t dd[4] = {d0, d1, d2, d3};
        const uint32_t mm[4] = {m0, m1, m2, m3};
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if (dd[q] & 0xe0u) acc -= static_cast<unsigned long long>(mm[q]) << (dd[q] & 31u);
        rare(v.x); rare(v.y); rare(v.z); rare(v.w);
      }
    };
    for (int j = 0; j < n_stages; ++j) {
      const int s = j % kRingStages;
      // warp-uniform verdict, so a timed-out lane cannot split the warp
      if (!__all_sync(0xffffffffu, mbar_wait_sleep(&s_full[s], (j / kRingStages) & 1))) {
        ok = false;
        break;
      }
      const float4* st = s_ring + s * kRingStageF4;
      const uint64_t lo = f0 + static_cast<uint64_t>(j) * kRingStageF4;
      const int cnt = static_cast<int>(min(f1 - lo, static_cast<uint64_t>(kRingStageF4)));
      if (j == 0) {
        // Warp-uniform window [base, base + 31] from the largest exponent
        // among the warp's first 128 weights; a normal weight with exponent
        // field e and significand m (implicit bit included) is m * 2^(e - 1)
        // in units of 2^-149, so its distance above the bottom is e - 1 - base.
        const float4 v0 = tid < cnt ? st[tid] : make_float4(0.f, 0.f, 0.f, 0.f);
        int e_loc = max(max(exp_field(v0.x), exp_field(v0.y)), max(exp_field(v0.z), exp_field(v0.w)));
        e_loc = min(e_loc, 254);
        const int e_max = static_cast<int>(__reduce_max_sync(0xffffffffu, static_cast<unsigned>(e_loc)));
        const int top = min(max(e_max - 1, 0) + 4, 253);
        base = max(0, top - 31);
        bias = static_cast<uint32_t>(base) + 1u;
      }
      unsigned long long acc[kPer];
#pragma unroll
      for (int k = 0; k < kPer; ++k) acc[k] = 0ull;
      if (cnt == kRingStageF4) {
        float4 v[kPer];
#pragma unroll
        for (int k = 0; k < kPer; ++k) v[k] = st[tid + k * kAbsumThreads];
#pragma unroll
        for (int k = 0; k < kPer; ++k) take4(v[k], acc[k]);
      } else {
#pragma unroll
        for (int k = 0; k < kPer; ++k)
          if (tid + k * kAbsumThreads < cnt) take4(st[tid + k * kAbsumThreads], acc[k]);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_empty[s]);
      unsigned long long t = acc[0];
#pragma unroll
      for (int k = 1; k < kPer; ++k) t += acc[k];
      add96(a0, a1, a2, static_cast<uint32_t>(t), static_cast<uint32_t>(t >> 32));
    }
  }
  if (!ok) atomicExch(&g_pack_wait_error, 1);

  // warp sum of the 96-bit accumulators (all lanes of a warp share `base`)
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const uint32_t b0 = __shfl_down_sync(0xffffffffu, a0, o);
    const uint32_t b1 = __shfl_down_sync(0xffffffffu, a1, o);
    const uint32_t b2 = __shfl_down_sync(0xffffffffu, a2, o);
    add96(a0, a1, a2, b0, b1, b2);
  }
  __syncthreads();   // every bin update done
  if (lane == 0 && warp < kConsumerWarps) {
    const uint32_t w[3] = {a0, a1, a2};
    add_words_shifted(s_limbs, w, base);
  }
  for (int e = tid; e < kBins; e += blockDim.x) {
    const unsigned long long v = s_bins[e];
    if (v) {
      const uint32_t w[2] = {static_cast<uint32_t>(v), static_cast<uint32_t>(v >> 32)};
      add_words_shifted(s_limbs, w, e);
    }
  }
  __syncthreads();
  if (tid == 0) {
    unsigned long long carry = 0;
    uint32_t* out = partials + static_cast<size_t>(blockIdx.x) * kPartialWords;
    for (int l = 0; l < kLimbs; ++l) {
      const unsigned long long v = s_limbs[l] + carry;
      out[l] = static_cast<uint32_t>(v);
      carry = v >> 32;
    }
    // (the total is below 2^309 for N*K < 2^32, so no carry leaves limb 11)
  }
}

cudaError_t take_pack_wait_error(int* flag) {
  int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(flag, g_pack_wait_error, sizeof(int));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_pack_wait_error, &zero, sizeof(int));
}

namespace {

constexpr int kFinalThreads = 256;      // threads that combine the partials

struct FinalSmem {
  unsigned long long part[kFinalThreads / 32][kLimbs];
  unsigned long long lo[kLimbs], hi[kLimbs];
  float gamma;
};

// Exact sum S (32-bit limbs, units of 2^-149) divided by count and rounded
// once to fp32, ties to even.
BL_DEVICE float round_mean(const uint32_t (&S)[kLimbs + 1], uint64_t count) {
  // T = the top 64 bits of S (all of S when it is shorter), sh = bits dropped
  int topl = kLimbs;
  while (topl > 0 && S[topl] == 0u) --topl;
  const int P = S[topl] ? 32 * topl + (32 - __clz(S[topl])) : 0;   // bit length of S
  const int sh = P > 64 ? P - 64 : 0;
  unsigned long long T;
  bool low_nonzero = false;
  {
    const int li = sh >> 5, r = sh & 31;
    const unsigned long long w01 =
        static_cast<unsigned long long>(S[li]) | (static_cast<unsigned long long>(li + 1 <= kLimbs ? S[li + 1] : 0u) << 32);
    const uint32_t w2 = li + 2 <= kLimbs ? S[li + 2] : 0u;
    T = r ? ((w01 >> r) | (static_cast<unsigned long long>(w2) << (64 - r))) : w01;
    for (int l = 0; l < li; ++l) low_nonzero |= S[l] != 0u;
    if (r) low_nonzero |= (S[li] & ((1u << r) - 1u)) != 0u;
  }
  // mean = (q + f) * 2^sh units of 2^-149, f in [0, 1), f > 0 iff rem or low bits
  const unsigned long long q = T / count;
  const unsigned long long rem = T - q * count;
  const int p = q ? 64 - __clzll(static_cast<long long>(q)) : 0;   // bit length of q
  const int E = p - 1 + sh;                                        // top bit position of the mean
  const int t = E > 23 ? E - 23 : 0;                               // fp32 spacing 2^t units
  const int drop = t - sh;                                         // low bits of q to round away
  unsigned long long mant;
  bool up;
  if (drop <= 0) {
    // sh == 0 here: round q + rem/count to an integer
    mant = q;
    const unsigned long long twice = rem * 2ull;
    up = twice > count || (twice == count && (q & 1ull));
  } else {
    mant = q >> drop;
    const bool guard = (q >> (drop - 1)) & 1ull;
    const bool sticky = (drop > 1 && (q & ((1ull << (drop - 1)) - 1ull)) != 0ull) || rem != 0ull || low_nonzero;
    up = guard && (sticky || (mant & 1ull));
  }
  unsigned long long bits = (static_cast<unsigned long long>(t) << 23) + mant + (up ? 1ull : 0ull);
  if (bits >= 0x7f800000ull) bits = 0x7f800000ull;   // unreachable for finite inputs
  return __uint_as_float(static_cast<uint32_t>(bits));
}

// gamma from the exact per-CTA partials, run by threads 0 .. kFinalThreads - 1
// of the CTA; sync() is a barrier over exactly those threads. Every caller
// thread gets gamma.
template <typename Sync>
BL_DEVICE float gamma_from_partials(const uint32_t* partials, int n_partials, uint64_t count, FinalSmem& sm,
                                    Sync sync) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  unsigned long long loc[kLimbs];
#pragma unroll
  for (int l = 0; l < kLimbs; ++l) loc[l] = 0ull;
  for (int c = tid; c < n_partials; c += kFinalThreads) {
    const uint4* p = reinterpret_cast<const uint4*>(partials + static_cast<size_t>(c) * kPartialWords);
    const uint4 q0 = p[0], q1 = p[1], q2 = p[2];
    loc[0] += q0.x; loc[1] += q0.y; loc[2] += q0.z; loc[3] += q0.w;
    loc[4] += q1.x; loc[5] += q1.y; loc[6] += q1.z; loc[7] += q1.w;
    loc[8] += q2.x; loc[9] += q2.y; loc[10] += q2.z; loc[11] += q2.w;
  }
#pragma unroll
  for (int l = 0; l < kLimbs; ++l) {
    unsigned long long v = loc[l];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_down_sync(0xffffffffu, v, o);
    if (lane == 0) sm.part[warp][l] = v;
  }
  sync();
  // limb l summed over the warps by thread l: 32-bit halves kept apart so no
  // 64-bit sum can wrap (each warp value is below 2^32 * n_partials)
  if (tid < kLimbs) {
    unsigned long long lo = 0, hi = 0;
#pragma unroll
    for (int w = 0; w < kFinalThreads / 32; ++w) {
      lo += sm.part[w][tid] & 0xffffffffull;
      hi += sm.part[w][tid] >> 32;
    }
    sm.lo[tid] = lo;
    sm.hi[tid] = hi;
  }
  sync();
  if (tid == 0) {
    // exact sum S in 32-bit limbs (S < 2^309)
    uint32_t S[kLimbs + 1];
    unsigned long long carry = 0;
#pragma unroll
    for (int l = 0; l < kLimbs; ++l) {
      const unsigned long long v = carry + sm.lo[l];
      S[l] = static_cast<uint32_t>(v);
      carry = (v >> 32) + sm.hi[l];
    }
    S[kLimbs] = static_cast<uint32_t>(carry);
    sm.gamma = round_mean(S, count);
  }
  sync();
  return sm.gamma;
}

}  // namespace

__global__ void __launch_bounds__(kFinalThreads)
bl_gamma_finalize(const uint32_t* __restrict__ partials, int n_partials, uint64_t count,
                  float* __restrict__ gamma) {
  __shared__ FinalSmem sm;
  pdl_wait();
  pdl_launch_dependents();
  partials = launder(partials);
  const float g = gamma_from_partials(partials, n_partials, count, sm, [] { __syncthreads(); });
  if (threadIdx.x == 0) *gamma = g;
}

// Four weights -> one packed byte (fields in bits 0-1, 2-3, 4-5, 6-7).
BL_DEVICE uint32_t pack4(const float4& v, float h) {
  return ternary_field(v.x, h) | (ternary_field(v.y, h) << 2) | (ternary_field(v.z, h) << 4) |
         (ternary_field(v.w, h) << 6);
}

// Code of one weight by the exact quotient: clip(rint(fp32(w / a)), -1, 1)
// as a packed field (code + 1), for a subnormal divisor a > 0.
BL_DEVICE uint32_t field_by_division(float w, float a) {
  const float q = rintf(__fdiv_rn(w, a));
  return q > 0.f ? 2u : (q < 0.f ? 0u : 1u);
}

BL_DEVICE uint32_t pack4_division(const float4& v, float a) {
  return field_by_division(v.x, a) | (field_by_division(v.y, a) << 2) | (field_by_division(v.z, a) << 4) |
         (field_by_division(v.w, a) << 6);
}

template <bool FUSED>
__global__ void __launch_bounds__(kPackThreads + 32, 2)
bl_quant_pack(const float4* __restrict__ w4, uint64_t n_bytes, const float* __restrict__ gamma_in,
              const uint32_t* __restrict__ partials, int n_partials, float* __restrict__ gamma_out,
              uint32_t* __restrict__ wp_words, int rule, float factor) {
  extern __shared__ __align__(128) float4 s_ring[];        // kRingStages x kRingStageF4
  __shared__ __align__(8) uint64_t s_full[kRingStages], s_empty[kRingStages];
  __shared__ FinalSmem s_fin;
  constexpr int kConsumerWarps = kPackThreads / 32;
  constexpr int kStageWords = kRingStageF4 / 4;            // packed words per stage
  static_assert(kStageWords == kPackThreads, "one packed word per consumer thread and stage");
  static_assert(kPackThreads == kFinalThreads, "the consumers combine the partials");

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    for (int s = 0; s < kRingStages; ++s) {
      mbar_init(&s_full[s], 1);
      mbar_init(&s_empty[s], kConsumerWarps);
    }
    mbar_init_fence();
  }
  // this CTA's share: the contiguous word range [q0, q1); word q packs the 16
  // weights of float4 4q .. 4q + 3
  const uint64_t n_words = n_bytes >> 2;
  const uint64_t q0 = n_words * blockIdx.x / gridDim.x, q1 = n_words * (blockIdx.x + 1) / gridDim.x;
  const int n_stages = static_cast<int>((q1 - q0 + kStageWords - 1) / kStageWords);
  __syncthreads();
  bool ok = true;

  if (warp == kConsumerWarps) {
    // The producer of the fused form streams W before the dependency wait:
    // its predecessor is the exact-sum kernel of the same W, which reads W
    // only and released this grid after its own dependency wait, so every
    // earlier write of W is complete and visible by now. The stand-alone
    // form cannot know who wrote W last and waits first.
    if (!FUSED) pdl_wait();
    if (lane == 0)
      ok = ring_produce(s_ring, kRingStageF4 * 16u, kRingStages, launder(w4) + 4 * q0, (q1 - q0) * 64u, s_full,
                        s_empty, l2_evict_first());   // the last read of W
    __syncwarp();
  } else {
    pdl_wait();
    pdl_launch_dependents();
    float g;
    if (FUSED) {
      // every CTA combines the partials itself (while its first stages are in
      // flight)
      g = gamma_from_partials(launder(partials), n_partials, n_bytes * 4, s_fin,
                              [] { asm volatile("bar.sync 1, %0;" ::"n"(kPackThreads) : "memory"); });
    } else {
      g = *launder(gamma_in);
    }
    // code = 0 iff |w| <= h, else the sign of w (see ternary_field):
    //   absmean      h = fp32(gamma + 1e-5) / 2   (exact: a normal fp32 halved)
    //   alpha-round  h = alpha / 2, alpha = fp32(factor x gamma); below 2^-125
    //                alpha / 2 may not be exact, so the codes are taken from
    //                the exact quotient instead; alpha = 0 (an all-zero W)
    //                gives h = infinity, all codes 0
    //   threshold    h = delta = fp32(factor x gamma)  (strict |w| > delta)
    // CTA 0 writes the forward's scale: gamma or alpha (the threshold rule's
    // scale comes from the masked exact sum).
    float h, alpha = 0.f;
    bool divide = false;
    if (rule == kRuleAlphaRound) {
      alpha = __fmul_rn(factor, g);
      divide = alpha > 0.f && alpha < 0x1p-125f;
      h = alpha > 0.f ? 0.5f * alpha : __int_as_float(0x7f800000);
    } else if (rule == kRuleThreshold) {
      h = __fmul_rn(factor, g);
    } else {
      h = 0.5f * __fadd_rn(g, kEpsGamma);
    }
    if (gamma_out && blockIdx.x == 0 && tid == 0 && rule != kRuleThreshold)
      *gamma_out = rule == kRuleAlphaRound ? alpha : g;
    // Thread t packs word t of each stage from float4 4t .. 4t + 3, taking
    // them in the rotated order (k + t/2) mod 4, so that the eight threads of
    // each quarter-warp read eight different 16-byte bank groups.
    const int rot = (tid >> 1) & 3;
    for (int j = 0; j < n_stages; ++j) {
      const int s = j % kRingStages;
      if (!__all_sync(0xffffffffu, mbar_wait_sleep(&s_full[s], (j / kRingStages) & 1))) {
        ok = false;
        break;
      }
      const uint64_t w0 = q0 + static_cast<uint64_t>(j) * kStageWords;
      const bool mine = w0 + tid < q1;
      const float4* st = s_ring + s * kRingStageF4 + 4 * tid;
      uint32_t r = 0u;
      if (mine) {
        if (!divide) {
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int q = (k + rot) & 3;
            r |= pack4(st[q], h) << (8 * q);
          }
        } else {
          for (int q = 0; q < 4; ++q) r |= pack4_division(st[q], alpha) << (8 * q);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_empty[s]);
      if (mine) wp_words[w0 + tid] = r;
    }
    // tail: up to three bytes when N*K/4 is not a multiple of 4
    const uint64_t tb = n_words * 4 + static_cast<uint64_t>(blockIdx.x) * kPackThreads + tid;
    if (tb < n_bytes) {
      const float4 v = launder(w4)[tb];
      reinterpret_cast<uint8_t*>(wp_words)[tb] =
          static_cast<uint8_t>(divide ? pack4_division(v, alpha) : pack4(v, h));
    }
  }
  if (!ok) atomicExch(&g_pack_wait_error, 1);
}

cudaError_t launch_quant_pack(const float4* w4, uint64_t n_bytes, const float* gamma_in, const uint32_t* partials,
                              int n_partials, float* scale_out, uint32_t* wp_words, int rule, float factor, int sms,
                              cudaStream_t s) {
  const bool fused = partials != nullptr;
  auto kern = fused ? bl_quant_pack<true> : bl_quant_pack<false>;
  // resident CTAs per SM (0: the shared memory cannot be reserved)
  const int per_sm = resident_ctas(reinterpret_cast<const void*>(kern), kPackThreads + 32, kRingSmem);
  if (per_sm <= 0) return cudaErrorInvalidConfiguration;
  const uint64_t n_words = n_bytes / 4;
  const uint64_t stages = (n_words + kRingStageF4 / 4 - 1) / (kRingStageF4 / 4);
  const uint64_t wave = static_cast<uint64_t>(sms) * static_cast<uint64_t>(per_sm);
  uint64_t grid = stages < wave ? stages : wave;
  if (grid < 1) grid = 1;
  return launch_pdl(kern, dim3(static_cast<unsigned>(grid)), dim3(kPackThreads + 32), kRingSmem, s, w4, n_bytes,
                    gamma_in, partials, n_partials, scale_out, wp_words, rule, factor);
}

int absum_ctas_per_sm(bool masked) {
  const void* k = masked ? reinterpret_cast<const void*>(bl_absum_partials<true>)
                         : reinterpret_cast<const void*>(bl_absum_partials<false>);
  return resident_ctas(k, kAbsumThreads + 32, kRingSmem);
}

cudaError_t launch_absum(const float4* w4, uint64_t n4, uint32_t* partials, const float* mask_gamma, float factor,
                         unsigned grid, cudaStream_t s) {
  if (mask_gamma)
    return launch_pdl(bl_absum_partials<true>, dim3(grid), dim3(kAbsumThreads + 32), kRingSmem, s, w4, n4, partials,
                      mask_gamma, factor);
  return launch_pdl(bl_absum_partials<false>, dim3(grid), dim3(kAbsumThreads + 32), kRingSmem, s, w4, n4, partials,
                    static_cast<const float*>(nullptr), 0.f);
}

}  // namespace bl
