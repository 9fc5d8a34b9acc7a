// Per-group weight quantisation (groups of 64 consecutive k of one row) and
// the forward over per-group scales.
//
// Passage: "BitNet 1-bit LLM 的混合精度微调技术：渐进量化策略", body: per-group
// quantisation with a group size of 64, so that each scale covers a small
// block of weights. The page gives the group size only; this library takes
// the group as 64 consecutive input features of one weight row (the axis the
// dot product sums over), applies the per-tensor absmean rule to each group,
// and multiplies every group's partial sum by its own scale:
//   gamma[n][g] = exact mean of |W[n][64g .. 64g+63]|, rounded once to fp32
//   code[n][k]  = clip(rint(fp32(W[n][k] / fp32(gamma[n][k/64] + 1e-5))), -1, 1)
//   y[m][n]     = sum_g gamma[n][g] * acc[m][n][g] / s_m,
//   acc[m][n][g] = sum over the group of code * x_q (exact integers).
// The packed codes keep the per-tensor layout (four per byte, code of k = 4j
// + i in bits 2i..2i+1 of byte j of the row).
//
// Packing reads W once: a half-warp holds one group (a float4 per lane), so
// the group's scale needs no second pass. The exact sum: every finite fp32
// value is m * 2^(f - 150) (m its 24-bit significand, f = max(exponent
// field, 1)). With F the largest f of the group, each weight within 33
// binades of F is m * 2^(f - F + 33) units of 2^(F - 183): below 2^57, so
// the 64 of them add up exactly in 64 bits. A group with a nonzero weight
// further below (rare: a spread of more than 2^33 inside 64 weights) is
// summed instead by one lane in a 288-bit fixed-point number in units of
// 2^-149. Either sum times the unit over 64 is rounded once to fp32 (ties to
// even), with every dropped bit kept as a sticky bit.
//
// The forward: per-token absmax codes (as in the per-tensor forward, stored
// in the transposed block layout with the code sum of every group), then a
// contraction over tiles of 32 weight rows x up to 8 tokens with the tile's
// codes staged in shared memory: per group, the four packed words meet the
// four activation blocks plane by plane in dp4a (fields are codes + 1, so the
// group's code sum is taken off), and the group sum times its scale is
// accumulated in fp64: each product is exact (24-bit scale times a sum below
// 2^14), and the fp64 sum over the K/64 groups of a row carries a relative
// error below (K/64) 2^-53 of sum_g |gamma * acc|. y is the fp64 sum divided
// by s_m in fp64 and rounded to fp32.

#include "async.cuh"
#include "common.cuh"
#include "kernels.cuh"

namespace bl {

namespace {

constexpr int kGpThreads = 256;             // packing: 8 warps, two groups per warp at a time
constexpr int kSlowLimbs = 9;               // 288 bits of 2^-149 units: 64 weights below 2^128 each

// The fp32 value nearest to T * 2^e (ties to even). A caller that dropped
// nonzero bits below T has set T's lowest bit and kept T >= 2^62, so that bit
// lies below the rounding position and only breaks ties.
BL_DEVICE float round_scaled_u64(unsigned long long T, int e) {
  if (T == 0ull) return 0.f;
  const int p = 63 - __clzll(static_cast<long long>(T));
  int ex = p + e;                                      // exponent of the top bit
  const bool normal = ex >= -126;
  const int shift = normal ? p - 23 : -149 - e;        // bits of T below the kept significand
  unsigned long long mant;
  if (shift <= 0) {
    mant = T << (-shift);
  } else if (shift >= 64) {
    mant = (shift == 64 && T > (1ull << 63)) ? 1ull : 0ull;
  } else {
    mant = T >> shift;
    const unsigned long long rem = T & ((1ull << shift) - 1ull), half = 1ull << (shift - 1);
    if (rem > half || (rem == half && (mant & 1ull))) ++mant;
  }
  if (!normal) return __uint_as_float(static_cast<uint32_t>(mant));   // 2^23 is the smallest normal
  if (mant == (1ull << 24)) {
    mant >>= 1;
    ++ex;
  }
  return __uint_as_float((static_cast<uint32_t>(ex + 127) << 23) | (static_cast<uint32_t>(mant) & 0x7fffffu));
}

// Significand and effective exponent field of |v| (finite): |v| = m 2^(f - 150).
BL_DEVICE void split_f32(uint32_t bits, uint32_t& m, int& f) {
  const uint32_t fe = (bits >> 23) & 0xffu;
  m = (bits & 0x7fffffu) | (fe ? 0x800000u : 0u);
  f = fe ? static_cast<int>(fe) : 1;
}

// Exact mean of the 64 |w| of this half-warp's group (four per lane), rounded
// once to fp32; every lane of the warp must call it (shuffles over the warp).
BL_DEVICE float group_gamma(const float4& v, int lane) {
  const uint32_t b[4] = {__float_as_uint(v.x), __float_as_uint(v.y), __float_as_uint(v.z), __float_as_uint(v.w)};
  uint32_t m[4];
  int f[4];
  int F = 1;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    split_f32(b[i], m[i], f[i]);
    if (m[i]) F = max(F, f[i]);
  }
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) F = max(F, __shfl_xor_sync(0xffffffffu, F, o));   // within each half
  const int B = F - 33;
  bool far = false;
#pragma unroll
  for (int i = 0; i < 4; ++i) far = far || (m[i] != 0u && f[i] < B);
  if (!__any_sync(0xffffffffu, far)) {
    unsigned long long t = 0ull;
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (m[i]) t += static_cast<unsigned long long>(m[i]) << (f[i] - B);
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
    // sum * 2^(B - 150) / 64, rounded by the first lane of each half only
    const float g = (lane & 15) == 0 ? round_scaled_u64(t, B - 156) : 0.f;
    return __shfl_sync(0xffffffffu, g, lane & 16);
  }
  // rare: a weight more than 33 binades below the group's largest. Lane 0 of
  // each half adds the group's 64 weights into 288-bit fixed point.
  uint32_t limb[kSlowLimbs];
#pragma unroll
  for (int j = 0; j < kSlowLimbs; ++j) limb[j] = 0u;
  const int base = lane & 16;
  for (int src = 0; src < 16; ++src) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t mi = __shfl_sync(0xffffffffu, m[i], base + src);
      const int fi = __shfl_sync(0xffffffffu, f[i], base + src);
      if ((lane & 15) == 0 && mi) {
        const int pos = fi - 1;                        // bit position of m's lowest bit in 2^-149 units
        const int q = pos >> 5, r = pos & 31;
        const unsigned long long piece = static_cast<unsigned long long>(mi) << r;   // below 2^55
        uint32_t carry = 0u;
#pragma unroll
        for (int j = 0; j < kSlowLimbs; ++j) {
          const uint32_t add = j == q ? static_cast<uint32_t>(piece) : (j == q + 1 ? static_cast<uint32_t>(piece >> 32) : 0u);
          const unsigned long long s = static_cast<unsigned long long>(limb[j]) + add + carry;
          limb[j] = static_cast<uint32_t>(s);
          carry = static_cast<uint32_t>(s >> 32);
        }
      }
    }
  }
  float g = 0.f;
  if ((lane & 15) == 0) {
    int top = kSlowLimbs - 1;
    while (top > 0 && limb[top] == 0u) --top;
    if (top <= 1) {
      g = round_scaled_u64((static_cast<unsigned long long>(limb[1]) << 32) | limb[0], -155);
    } else {
      // the top 64 bits (limbs top, top - 1) and a sticky bit for everything below,
      // normalised so the window's top bit is bit 63
      const int lz = __clz(static_cast<int>(limb[top]));
      unsigned long long T = (static_cast<unsigned long long>(limb[top]) << 32) | limb[top - 1];
      const uint32_t next = limb[top - 2];
      if (lz) T = (T << lz) | (next >> (32 - lz));
      bool sticky = (lz ? (next << lz) : next) != 0u;
      for (int j = top - 3; j >= 0; --j) sticky = sticky || limb[j] != 0u;
      if (sticky) T |= 1ull;
      // T's lowest bit is 2^(32 (top - 1) - lz) units of 2^-149, and 64 divides out
      g = round_scaled_u64(T, 32 * (top - 1) - lz - 149 - 6);
    }
  }
  return __shfl_sync(0xffffffffu, g, base);
}

}  // namespace

// gamma[n][g] and the packed codes of W [N][K] (K % 64 == 0): two groups per
// warp per step (one per half), a float4 per lane, one packed byte per lane.
__global__ void __launch_bounds__(kGpThreads)
bl_pack_grouped(const float4* __restrict__ w4, uint64_t n_groups, uint8_t* __restrict__ wp,
                float* __restrict__ gam) {
  pdl_wait();
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31;
  const uint64_t warps = static_cast<uint64_t>(gridDim.x) * (kGpThreads / 32);
  const uint64_t wid = static_cast<uint64_t>(blockIdx.x) * (kGpThreads / 32) + (threadIdx.x >> 5);
  auto load = [&](uint64_t pair) {
    const uint64_t g = pair + (lane >> 4);
    return g < n_groups ? __ldcs(w4 + g * 16 + (lane & 15)) : make_float4(0.f, 0.f, 0.f, 0.f);
  };
  // the next pair's weights are loaded before this pair's arithmetic
  float4 next = load(2 * wid);
  for (uint64_t pair0 = 2 * wid; pair0 < n_groups; pair0 += 2 * warps) {
    const uint64_t g = pair0 + (lane >> 4);
    const bool live = g < n_groups;                     // the last pair may hold one group
    const float4 v = next;
    next = load(pair0 + 2 * warps);
    const float gamma = group_gamma(v, lane);
    if (!live) continue;
    const float h = __fmul_rn(__fadd_rn(gamma, kEpsGamma), 0.5f);   // d / 2, d = fp32(gamma + 1e-5) >= 1e-5
    wp[g * 16 + (lane & 15)] = static_cast<uint8_t>(ternary_field(v.x, h) | (ternary_field(v.y, h) << 2) |
                                                    (ternary_field(v.z, h) << 4) | (ternary_field(v.w, h) << 6));
    if ((lane & 15) == 0) gam[g] = gamma;
  }
}

cudaError_t launch_pack_grouped(const float* W, int64_t N, int64_t K, uint8_t* wp, float* gam, int sms,
                                cudaStream_t s) {
  const uint64_t n_groups = static_cast<uint64_t>(N) * static_cast<uint64_t>(K / 64);
  const uint64_t need = (n_groups + 2 * (kGpThreads / 32) - 1) / (2 * (kGpThreads / 32));
  const unsigned grid = static_cast<unsigned>(std::min<uint64_t>(need, static_cast<uint64_t>(sms) * 8));
  return launch_pdl(bl_pack_grouped, dim3(grid), dim3(kGpThreads), 0, s, reinterpret_cast<const float4*>(W), n_groups,
                    wp, gam);
}

// ---- forward

namespace {

constexpr int kGaThreads = 512;             // activation pass: one CTA per token
constexpr int kGThreads = 256;              // contraction: 8 warps (k-slices) x 32 rows
constexpr size_t kGMaxSmem = 200 * 1024;

// Loads through L2 (not L1): the data may have been written by the grid this
// one waited for.
BL_DEVICE uint4 ldg_cg_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p) : "memory");
  return v;
}

BL_DEVICE uint32_t low4(uint32_t b0, uint32_t b1, uint32_t b2, uint32_t b3) {
  return __byte_perm(__byte_perm(b0, b1, 0x0040), __byte_perm(b2, b3, 0x0040), 0x5410);
}

template <typename T> struct Block16;
template <> struct Block16<float> {
  static BL_DEVICE void load(const float* row, int b, float (&f)[16]) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 v = ldg_cg_v4(row + 16 * b + 4 * i);
      f[4 * i] = __uint_as_float(v.x);
      f[4 * i + 1] = __uint_as_float(v.y);
      f[4 * i + 2] = __uint_as_float(v.z);
      f[4 * i + 3] = __uint_as_float(v.w);
    }
  }
};
template <> struct Block16<uint16_t> {   // bf16 bits
  static BL_DEVICE void load(const uint16_t* row, int b, float (&f)[16]) {
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const uint4 v = ldg_cg_v4(row + 16 * b + 8 * i);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        f[8 * i + 2 * j] = __uint_as_float(w[j] << 16);
        f[8 * i + 2 * j + 1] = __uint_as_float(w[j] & 0xffff0000u);
      }
    }
  }
};

}  // namespace

// Per-token absmax codes of x [M][K] in the transposed block layout the
// contraction reads (block b of token m at byte 16 (m K/16 + b); its word i
// holds the codes of k = 16b + 4j + i as bytes j), the code sum of every
// group of 64, the scales, and optionally the codes in row order.
template <typename T>
__global__ void __launch_bounds__(kGaThreads)
bl_act_quant_grouped(const T* __restrict__ x, int K, uint4* __restrict__ xt, int* __restrict__ gsum,
                     float* __restrict__ scale, int8_t* __restrict__ xq_out, float* __restrict__ scale_out) {
  __shared__ float s_red[kGaThreads / 32];
  pdl_wait();
  pdl_launch_dependents();
  x = launder(x);
  const int m = blockIdx.x, tid = threadIdx.x, lane = tid & 31;
  const T* row = x + static_cast<size_t>(m) * K;
  const int nblk = K >> 4;
  float amax = 0.f;
  for (int b = tid; b < nblk; b += kGaThreads) {
    float f[16];
    Block16<T>::load(row, b, f);
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(f[i]));
  }
  amax = warp_max(amax);
  if (lane == 0) s_red[tid >> 5] = amax;
  __syncthreads();
  const float s = token_scale(warp_max(lane < kGaThreads / 32 ? s_red[lane] : 0.f));
  if (tid == 0) {
    scale[m] = s;
    if (scale_out) scale_out[m] = s;
  }
  // blocks 4g .. 4g + 3 (one group) are taken by four consecutive threads
  const int nb_pad = (nblk + kGaThreads - 1) / kGaThreads * kGaThreads;
  for (int b = tid; b < nb_pad; b += kGaThreads) {
    int bs = 0;
    if (b < nblk) {
      float f[16];
      Block16<T>::load(row, b, f);
      uint32_t c[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) c[i] = static_cast<uint32_t>(quant_code(f[i], s)) & 0xffu;
      uint4 t;
      t.x = low4(c[0], c[4], c[8], c[12]);
      t.y = low4(c[1], c[5], c[9], c[13]);
      t.z = low4(c[2], c[6], c[10], c[14]);
      t.w = low4(c[3], c[7], c[11], c[15]);
      xt[static_cast<size_t>(m) * nblk + b] = t;
      bs = dp4a_ss(static_cast<int>(t.w), 0x01010101,
                   dp4a_ss(static_cast<int>(t.z), 0x01010101,
                           dp4a_ss(static_cast<int>(t.y), 0x01010101, dp4a_ss(static_cast<int>(t.x), 0x01010101, 0))));
      if (xq_out) {
        uint4 o;
        o.x = low4(c[0], c[1], c[2], c[3]);
        o.y = low4(c[4], c[5], c[6], c[7]);
        o.z = low4(c[8], c[9], c[10], c[11]);
        o.w = low4(c[12], c[13], c[14], c[15]);
        reinterpret_cast<uint4*>(xq_out + static_cast<size_t>(m) * K)[b] = o;
      }
    }
    bs += __shfl_xor_sync(0xffffffffu, bs, 1);
    bs += __shfl_xor_sync(0xffffffffu, bs, 2);
    if ((b & 3) == 0 && b < nblk) gsum[static_cast<size_t>(m) * (nblk >> 2) + (b >> 2)] = bs;
  }
}

// y[m][n] for a tile of 32 weight rows x TM tokens. The tile's transposed
// codes and group code sums are staged in shared memory once; warp w takes
// the groups g = w, w + 8, ... and lane l the row n0 + l, so the 32 lanes of
// a read of the activations read the same word (a broadcast). Per group the
// four packed words of the row (one 16-byte load) meet the four activation
// blocks plane by plane (dp4a), the group's code sum is taken off, and
// gamma[n][g] * acc is added in fp64 (exact product). The eight warps'
// partial sums of a (row, token) are added in a fixed order, then divided
// by s_m in fp64 and rounded to fp32.
constexpr int kGRows = 32;
constexpr int kGSlices = kGThreads / 32;

size_t gemm_grouped_smem(int K, int tm) {
  return static_cast<size_t>(tm) * K + static_cast<size_t>(tm) * (K / 64) * 4 +
         static_cast<size_t>(kGSlices) * kGRows * tm * 8 + 16;
}

// The contraction of a staged tile (codes s_x [tm][K/16], group code sums
// s_gs [tm][G]) against weight rows blockIdx.x * 32 .., and y = sum / sc[t]
// for its tm tokens m0 ...; ends with a CTA barrier before the stores.
template <int TM>
BL_DEVICE void grouped_tile(const uint4* s_x, const int* s_gs, double* s_part, const uint8_t* __restrict__ wp,
                            const float* __restrict__ gam, const float* sc, float* __restrict__ y, int m0, int tm,
                            int N, int K) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = K >> 6, nblk = K >> 4;
  const int n = blockIdx.x * kGRows + lane;
  double acc[TM];
#pragma unroll
  for (int t = 0; t < TM; ++t) acc[t] = 0.0;
  if (n < N) {
    const uint4* wrow = reinterpret_cast<const uint4*>(wp + static_cast<size_t>(n) * (K >> 2));
    const float* grow = gam + static_cast<size_t>(n) * G;
    // the next group's packed words and scale are loaded before this group's arithmetic
    uint4 wn = warp < G ? __ldg(wrow + warp) : make_uint4(0u, 0u, 0u, 0u);
    float gn = warp < G ? __ldg(grow + warp) : 0.f;
    for (int g = warp; g < G; g += kGSlices) {
      const uint4 w = wn;
      const double gm = static_cast<double>(gn);
      if (g + kGSlices < G) {
        wn = __ldg(wrow + g + kGSlices);
        gn = __ldg(grow + g + kGSlices);
      }
      const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
      uint32_t pl[4][4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        pl[j][0] = wv[j] & 0x03030303u;
        pl[j][1] = wv[j] & 0x0c0c0c0cu;
        pl[j][2] = wv[j] & 0x30303030u;
        pl[j][3] = wv[j] & 0xc0c0c0c0u;
      }
#pragma unroll
      for (int t = 0; t < TM; ++t) {
        if (t < tm) {
          const uint4* xb = s_x + t * nblk + 4 * g;
          int a0 = 0, a1 = 0, a2 = 0, a3 = 0;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint4 a = xb[j];
            a0 = dp4a_us(pl[j][0], static_cast<int>(a.x), a0);
            a1 = dp4a_us(pl[j][1], static_cast<int>(a.y), a1);
            a2 = dp4a_us(pl[j][2], static_cast<int>(a.z), a2);
            a3 = dp4a_us(pl[j][3], static_cast<int>(a.w), a3);
          }
          const int ag = a0 + (a1 >> 2) + (a2 >> 4) + (a3 >> 6) - s_gs[t * G + g];
          acc[t] = fma(gm, static_cast<double>(ag), acc[t]);   // the product is exact
        }
      }
    }
  }
#pragma unroll
  for (int t = 0; t < TM; ++t) s_part[(warp * kGRows + lane) * TM + t] = acc[t];
  __syncthreads();
  for (int i = tid; i < kGRows * tm; i += kGThreads) {
    const int r = i / tm, t = i - r * tm;
    const int nn = blockIdx.x * kGRows + r;
    if (nn < N) {
      double v = 0.0;
      for (int sl = 0; sl < kGSlices; ++sl) v += s_part[(sl * kGRows + r) * TM + t];
      y[static_cast<size_t>(m0 + t) * N + nn] = __double2float_rn(v / static_cast<double>(sc[t]));
    }
  }
}

template <int TM>
__global__ void __launch_bounds__(kGThreads)
bl_gemm_grouped(const uint8_t* __restrict__ wp, const float* __restrict__ gam, const uint4* __restrict__ xt,
                const int* __restrict__ gsum, const float* __restrict__ scale, float* __restrict__ y, int M, int N,
                int K) {
  extern __shared__ __align__(16) uint8_t smem[];
  pdl_wait();
  pdl_launch_dependents();
  xt = launder(xt);
  gsum = launder(gsum);
  scale = launder(scale);
  const int tid = threadIdx.x;
  const int G = K >> 6, nblk = K >> 4;
  const int m0 = blockIdx.y * TM;
  const int tm = min(TM, M - m0);
  uint4* s_x = reinterpret_cast<uint4*>(smem);                                   // [TM][K/16]
  int* s_gs = reinterpret_cast<int*>(smem + static_cast<size_t>(TM) * K);        // [TM][G]
  double* s_part = reinterpret_cast<double*>(
      (reinterpret_cast<uintptr_t>(s_gs + TM * G) + 7) & ~uintptr_t(7));         // [slices][rows][TM]
  for (int i = tid; i < tm * nblk; i += kGThreads) s_x[i] = ldg_cg_v4(xt + static_cast<size_t>(m0) * nblk + i);
  for (int i = tid; i < tm * G; i += kGThreads) s_gs[i] = __ldcg(gsum + static_cast<size_t>(m0) * G + i);
  __syncthreads();
  grouped_tile<TM>(s_x, s_gs, s_part, wp, gam, scale + m0, y, m0, tm, N, K);
}

// One token (M = 1) in one kernel: every CTA quantises the token itself
// (the same absmax, codes and group sums as bl_act_quant_grouped, into shared
// memory), then contracts its 32 weight rows as bl_gemm_grouped does. The
// rows' packed words start moving into L2 before the dependency
// wait (a prefetch cannot change what later loads see). CTA 0 also writes
// the optional scale and codes.
template <typename T>
__global__ void __launch_bounds__(kGThreads)
bl_gemv_grouped(const T* __restrict__ x, const uint8_t* __restrict__ wp, const float* __restrict__ gam,
                float* __restrict__ y, int8_t* __restrict__ xq_out, float* __restrict__ scale_out, int N, int K) {
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ float s_red[kGThreads / 32];
  __shared__ float s_scale;
  const int tid = threadIdx.x, lane = tid & 31;
  const int G = K >> 6, nblk = K >> 4;
  if (tid == 0) {
    // 16-byte aligned, a multiple of 16 bytes: K / 4 is a multiple of 16
    const int r0 = blockIdx.x * kGRows, rows = min(kGRows, N - r0);
    prefetch_l2_range(wp + static_cast<size_t>(r0) * (K >> 2), static_cast<uint64_t>(rows) * (K >> 2));
  }
  pdl_wait();
  pdl_launch_dependents();
  x = launder(x);
  wp = launder(wp);
  gam = launder(gam);
  uint4* s_x = reinterpret_cast<uint4*>(smem);                                   // [K/16]
  int* s_gs = reinterpret_cast<int*>(smem + static_cast<size_t>(K));             // [G]
  double* s_part = reinterpret_cast<double*>(
      (reinterpret_cast<uintptr_t>(s_gs + G) + 7) & ~uintptr_t(7));              // [slices][rows]
  float amax = 0.f;
  for (int b = tid; b < nblk; b += kGThreads) {
    float f[16];
    Block16<T>::load(x, b, f);
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(f[i]));
  }
  amax = warp_max(amax);
  if (lane == 0) s_red[tid >> 5] = amax;
  __syncthreads();
  const float s = token_scale(warp_max(lane < kGThreads / 32 ? s_red[lane] : 0.f));
  if (tid == 0) {
    s_scale = s;
    if (scale_out && blockIdx.x == 0) scale_out[0] = s;
  }
  // blocks 4g .. 4g + 3 (one group) are taken by four consecutive threads
  const int nb_pad = (nblk + kGThreads - 1) / kGThreads * kGThreads;
  for (int b = tid; b < nb_pad; b += kGThreads) {
    int bs = 0;
    if (b < nblk) {
      float f[16];
      Block16<T>::load(x, b, f);
      uint32_t c[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) c[i] = static_cast<uint32_t>(quant_code(f[i], s)) & 0xffu;
      uint4 t;
      t.x = low4(c[0], c[4], c[8], c[12]);
      t.y = low4(c[1], c[5], c[9], c[13]);
      t.z = low4(c[2], c[6], c[10], c[14]);
      t.w = low4(c[3], c[7], c[11], c[15]);
      s_x[b] = t;
      bs = dp4a_ss(static_cast<int>(t.w), 0x01010101,
                   dp4a_ss(static_cast<int>(t.z), 0x01010101,
                           dp4a_ss(static_cast<int>(t.y), 0x01010101, dp4a_ss(static_cast<int>(t.x), 0x01010101, 0))));
      if (xq_out && blockIdx.x == 0) {
        uint4 o;
        o.x = low4(c[0], c[1], c[2], c[3]);
        o.y = low4(c[4], c[5], c[6], c[7]);
        o.z = low4(c[8], c[9], c[10], c[11]);
        o.w = low4(c[12], c[13], c[14], c[15]);
        reinterpret_cast<uint4*>(xq_out)[b] = o;
      }
    }
    bs += __shfl_xor_sync(0xffffffffu, bs, 1);
    bs += __shfl_xor_sync(0xffffffffu, bs, 2);
    if ((b & 3) == 0 && b < nblk) s_gs[b >> 2] = bs;
  }
  __syncthreads();
  grouped_tile<1>(s_x, s_gs, s_part, wp, gam, &s_scale, y, 0, 1, N, K);
}

size_t forward_grouped_workspace(int64_t M, int64_t K) {
  const size_t a = (static_cast<size_t>(M) * static_cast<size_t>(K) + 255) / 256 * 256;
  const size_t b = (static_cast<size_t>(M) * static_cast<size_t>(K / 64) * 4 + 255) / 256 * 256;
  return a + b + (static_cast<size_t>(M) * 4 + 255) / 256 * 256;
}

cudaError_t launch_forward_grouped(const void* x, bool bf16, int M, int N, int K, const uint8_t* wp, const float* gam,
                                   float* y, int8_t* xq_out, float* scale_out, void* ws, cudaStream_t s) {
  if (M == 1) {
    // one token: one kernel, every CTA quantising the token itself
    const size_t smem = gemm_grouped_smem(K, 1);
    const dim3 grid((N + kGRows - 1) / kGRows);
    auto go1 = [&](auto kern, auto xp) -> cudaError_t {
      const cudaError_t e1 = ensure_smem(reinterpret_cast<const void*>(kern), smem);
      if (e1 != cudaSuccess) return e1;
      return launch_pdl(kern, grid, dim3(kGThreads), smem, s, xp, wp, gam, y, xq_out, scale_out, N, K);
    };
    return bf16 ? go1(bl_gemv_grouped<uint16_t>, static_cast<const uint16_t*>(x))
                : go1(bl_gemv_grouped<float>, static_cast<const float*>(x));
  }
  uint8_t* base = static_cast<uint8_t*>(ws);
  uint4* xt = reinterpret_cast<uint4*>(base);
  base += (static_cast<size_t>(M) * K + 255) / 256 * 256;
  int* gs = reinterpret_cast<int*>(base);
  base += (static_cast<size_t>(M) * (K / 64) * 4 + 255) / 256 * 256;
  float* sc = reinterpret_cast<float*>(base);
  cudaError_t e = bf16 ? launch_pdl(bl_act_quant_grouped<uint16_t>, dim3(M), dim3(kGaThreads), 0, s,
                                    static_cast<const uint16_t*>(x), K, xt, gs, sc, xq_out, scale_out)
                       : launch_pdl(bl_act_quant_grouped<float>, dim3(M), dim3(kGaThreads), 0, s,
                                    static_cast<const float*>(x), K, xt, gs, sc, xq_out, scale_out);
  if (e != cudaSuccess) return e;
  // token tile: as many tokens as M needs (1, 2, 4 or 8) while the staged codes fit
  int tm = M <= 1 ? 1 : (M <= 2 ? 2 : (M <= 4 ? 4 : 8));
  while (tm > 1 && gemm_grouped_smem(K, tm) > kGMaxSmem) tm >>= 1;
  const size_t smem = gemm_grouped_smem(K, tm);
  const dim3 grid((N + kGRows - 1) / kGRows, (M + tm - 1) / tm);
  auto go = [&](auto kern) -> cudaError_t {
    const cudaError_t e2 = ensure_smem(reinterpret_cast<const void*>(kern), smem);
    if (e2 != cudaSuccess) return e2;
    return launch_pdl(kern, grid, dim3(kGThreads), smem, s, wp, gam, xt, gs, sc, y, M, N, K);
  };
  if (tm == 1) return go(bl_gemm_grouped<1>);
  if (tm == 2) return go(bl_gemm_grouped<2>);
  if (tm == 4) return go(bl_gemm_grouped<4>);
  return go(bl_gemm_grouped<8>);
}

}  // namespace bl
