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
//   1. bl_absum_partials: each CTA sums its share of |W| exactly. Each warp
//      picks a window of 32 binades from the largest exponent among its first
//      128 weights (4 binades above it, 27 below). For a weight in the window,
//      at distance d binades above its bottom, |w| = m * 2^d window units (m
//      the 24-bit significand), which one wide multiply-add (mad.wide.u32)
//      adds to a 64-bit register accumulator; 2^d comes from a shift that
//      gives 0 for any d outside 0..31, so out-of-window weights add nothing
//      there. One OR over the four shift amounts of a float4 finds those
//      weights (zeros, subnormals, stragglers far from the warp's scale);
//      they go to 254 per-exponent 64-bit bins in shared memory. The 64-bit
//      accumulator is folded into 96 bits after every 16 weights, and the CTA
//      folds everything into a 384-bit fixed-point partial (12 x 32-bit limbs).
//   2. bl_gamma_finalize: one CTA adds the partials (shuffle reductions), then
//      one thread divides the top 64 bits of the exact sum by N*K and rounds
//      the quotient to fp32, ties to even, with the dropped bits and the
//      remainder as the sticky bit.
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

// Streaming 16-byte load that does not allocate in L1.
BL_DEVICE float4 ld_f4_stream(const float4* p) {
  float4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.f32 {%0,%1,%2,%3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "l"(p));
  return v;
}

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

// a << s with PTX semantics: shift amounts of 32 or more give 0.
BL_DEVICE uint32_t shl_clamped(uint32_t a, uint32_t s) {
  uint32_t r;
  asm("shl.b32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(s));
  return r;
}

// a * b + c with a 64-bit addend and result (exact while it stays below 2^64).
BL_DEVICE unsigned long long mad_wide_u32(uint32_t a, uint32_t b, unsigned long long c) {
  unsigned long long r;
  asm("mad.wide.u32 %0, %1, %2, %3;" : "=l"(r) : "r"(a), "r"(b), "l"(c));
  return r;
}

}  // namespace

__global__ void __launch_bounds__(kAbsumThreads)
bl_absum_partials(const float4* __restrict__ w4, uint64_t n4, uint32_t* __restrict__ partials) {
  __shared__ unsigned long long s_bins[kBins];
  __shared__ unsigned long long s_limbs[kSmemLimbs];

  const int tid = threadIdx.x;
  for (int i = tid; i < kBins; i += blockDim.x) s_bins[i] = 0ull;
  if (tid < kSmemLimbs) s_limbs[tid] = 0ull;

  const uint64_t stride = static_cast<uint64_t>(gridDim.x) * blockDim.x;
  const uint64_t first = static_cast<uint64_t>(blockIdx.x) * blockDim.x + tid;
  auto ld_stream_f4 = [](const float4* p) { return ld_f4_stream(p); };
  pdl_wait();
  pdl_launch_dependents();
  w4 = launder(w4);

  // Warp-uniform window [base, base + 31] in units of 2^-149; a normal weight
  // with exponent field e and significand m (implicit bit included) is
  // m * 2^(e - 1) in those units, so d = e - 1 - base.
  float4 v0 = make_float4(0.f, 0.f, 0.f, 0.f);
  if (first < n4) v0 = ld_stream_f4(w4 + first);
  int e_loc = max(max(exp_field(v0.x), exp_field(v0.y)), max(exp_field(v0.z), exp_field(v0.w)));
  e_loc = min(e_loc, 254);
  const int e_max = static_cast<int>(__reduce_max_sync(0xffffffffu, static_cast<unsigned>(e_loc)));
  const int top = min(max(e_max - 1, 0) + 4, 253);
  const int base = max(0, top - 31);
  const uint32_t bias = static_cast<uint32_t>(base) + 1u;
  __syncthreads();   // bins and limbs cleared

  uint32_t a0 = 0u, a1 = 0u, a2 = 0u;      // 96-bit total
  unsigned long long acc = 0ull;           // at most 16 window terms below 2^55 each

  // out-of-window weights of a float4 (rare): exact per-exponent bins
  auto rare = [&](float x) {
    const uint32_t b = __float_as_uint(x) & 0x7fffffffu;
    const uint32_t e = b >> 23;
    if ((e - bias) >= 32u && b != 0u) {
      const uint32_t m = e ? ((b & 0x7fffffu) | 0x800000u) : b;
      atomicAdd(&s_bins[e ? e - 1u : 0u], static_cast<unsigned long long>(m));
    }
  };
  auto take4 = [&](const float4& v) {
    const uint32_t b0 = __float_as_uint(v.x) & 0x7fffffffu, b1 = __float_as_uint(v.y) & 0x7fffffffu;
    const uint32_t b2 = __float_as_uint(v.z) & 0x7fffffffu, b3 = __float_as_uint(v.w) & 0x7fffffffu;
    const uint32_t d0 = (b0 >> 23) - bias, d1 = (b1 >> 23) - bias, d2 = (b2 >> 23) - bias, d3 = (b3 >> 23) - bias;
    acc = mad_wide_u32((b0 & 0x7fffffu) | 0x800000u, shl_clamped(1u, d0), acc);
    acc = mad_wide_u32((b1 & 0x7fffffu) | 0x800000u, shl_clamped(1u, d1), acc);
    acc = mad_wide_u32((b2 & 0x7fffffu) | 0x800000u, shl_clamped(1u, d2), acc);
    acc = mad_wide_u32((b3 & 0x7fffffu) | 0x800000u, shl_clamped(1u, d3), acc);
    if ((d0 | d1 | d2 | d3) >= 32u) {
      rare(v.x); rare(v.y); rare(v.z); rare(v.w);
    }
  };
  auto fold = [&]() {
    add96(a0, a1, a2, static_cast<uint32_t>(acc), static_cast<uint32_t>(acc >> 32));
    acc = 0ull;
  };

  if (first < n4) {
    take4(v0);
    fold();
  }
  // software pipeline: the next four float4 of this thread are in flight while
  // the current four are summed
  uint64_t i = first + stride;
  float4 c0 = make_float4(0.f, 0.f, 0.f, 0.f), c1 = c0, c2 = c0, c3 = c0;
  bool have = i + 3 * stride < n4;
  if (have) {
    c0 = ld_stream_f4(w4 + i); c1 = ld_stream_f4(w4 + i + stride);
    c2 = ld_stream_f4(w4 + i + 2 * stride); c3 = ld_stream_f4(w4 + i + 3 * stride);
  }
  while (have) {
    const uint64_t nxt = i + 4 * stride;
    const bool more = nxt + 3 * stride < n4;
    float4 p0 = c0, p1 = c1, p2 = c2, p3 = c3;
    if (more) {
      p0 = ld_stream_f4(w4 + nxt); p1 = ld_stream_f4(w4 + nxt + stride);
      p2 = ld_stream_f4(w4 + nxt + 2 * stride); p3 = ld_stream_f4(w4 + nxt + 3 * stride);
    }
    take4(c0); take4(c1); take4(c2); take4(c3);
    fold();
    c0 = p0; c1 = p1; c2 = p2; c3 = p3;
    i = nxt;
    have = more;
  }
  for (; i < n4; i += stride) {
    take4(ld_stream_f4(w4 + i));
    fold();
  }

  // warp sum of the 96-bit accumulators (all lanes share `base`)
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const uint32_t b0 = __shfl_down_sync(0xffffffffu, a0, o);
    const uint32_t b1 = __shfl_down_sync(0xffffffffu, a1, o);
    const uint32_t b2 = __shfl_down_sync(0xffffffffu, a2, o);
    add96(a0, a1, a2, b0, b1, b2);
  }
  __syncthreads();   // every bin update done
  if ((tid & 31) == 0) {
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

__global__ void __launch_bounds__(256)
bl_gamma_finalize(const uint32_t* __restrict__ partials, int n_partials, uint64_t count,
                  float* __restrict__ gamma) {
  __shared__ unsigned long long s_part[256 / 32][kLimbs];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  pdl_wait();
  pdl_launch_dependents();
  partials = launder(partials);
  unsigned long long loc[kLimbs];
#pragma unroll
  for (int l = 0; l < kLimbs; ++l) loc[l] = 0ull;
  for (int c = tid; c < n_partials; c += blockDim.x) {
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
    if (lane == 0) s_part[warp][l] = v;
  }
  __syncthreads();
  // limb l summed over the warps by thread l: 32-bit halves kept apart so no
  // 64-bit sum can wrap (each warp value is below 2^32 * n_partials)
  __shared__ unsigned long long s_lo[kLimbs], s_hi[kLimbs];
  if (tid < kLimbs) {
    unsigned long long lo = 0, hi = 0;
#pragma unroll
    for (int w = 0; w < 256 / 32; ++w) {
      lo += s_part[w][tid] & 0xffffffffull;
      hi += s_part[w][tid] >> 32;
    }
    s_lo[tid] = lo;
    s_hi[tid] = hi;
  }
  __syncthreads();
  if (tid != 0) return;

  // exact sum S in 32-bit limbs (S < 2^309)
  uint32_t S[kLimbs + 1];
  unsigned long long carry = 0;
#pragma unroll
  for (int l = 0; l < kLimbs; ++l) {
    const unsigned long long v = carry + s_lo[l];
    S[l] = static_cast<uint32_t>(v);
    carry = (v >> 32) + s_hi[l];
  }
  S[kLimbs] = static_cast<uint32_t>(carry);

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
  const uint64_t n_words = n_bytes >> 2;
  const uint64_t stride = static_cast<uint64_t>(gridDim.x) * blockDim.x;
  uint64_t i = static_cast<uint64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  pdl_wait();
  pdl_launch_dependents();
  w4 = launder(w4);
  gamma = launder(gamma);
  // software pipeline: the next word's 16 weights load while this one packs,
  // and the first loads are in flight before gamma arrives
  float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a, c = a, e = a;
  if (i < n_words) {
    const float4* src = w4 + 4 * i;
    a = ld_f4_stream(src); b = ld_f4_stream(src + 1);
    c = ld_f4_stream(src + 2); e = ld_f4_stream(src + 3);
  }
  const float d = __fadd_rn(*gamma, kEpsGamma);
  const float h = 0.5f * d;                 // exact: d is a normal fp32
  while (i < n_words) {
    const uint64_t nxt = i + stride;
    float4 na = a, nb = b, nc = c, ne = e;
    if (nxt < n_words) {
      const float4* src = w4 + 4 * nxt;
      na = ld_f4_stream(src); nb = ld_f4_stream(src + 1);
      nc = ld_f4_stream(src + 2); ne = ld_f4_stream(src + 3);
    }
    wp_words[i] = pack16(a, b, c, e, h);
    a = na; b = nb; c = nc; e = ne;
    i = nxt;
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
