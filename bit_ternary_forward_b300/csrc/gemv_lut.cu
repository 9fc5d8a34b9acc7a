// Lookup-table decode GEMV (one token): the table idea of bitnet.cpp's TL1
// kernel, on the GPU, as an alternative to the dp4a GEMV.
//
// Passages: "部署 BitNet 1-bit LLM：三元权重边缘推理优化", the kernel types
// (TL1 uses a lookup table); "BitNet 三元权重阈值优化工程实践", the bitnet.cpp
// kernels; "穿越1比特的奇幻旅程" (2B4T summary), section "GPU端：CUDA内核的定制
// 魔法" (W1.58A8 over four-per-byte packed weights); "BitNet 1-bit LLM 的混合
// 精度微调技术：渐进量化策略", body, quantisation functions.
//
// Two consecutive weights k = 2p, 2p + 1 sit in one 4-bit nibble of a packed
// byte (fields f0 | f1 << 2, f = code + 1). For each pair p the kernel
// tabulates the nine possible partial sums
//     T_p[f0 + 4 f1] = (f0 - 1) x_q[2p] + (f1 - 1) x_q[2p + 1]
// once per call, and the contraction is one table read and one add per two
// weights: acc = sum_p T_p[nibble p of the row]. Every entry and every sum is
// an exact integer, so y = fp32(fp32(acc * gamma) / s) is the same as the
// other paths'.
//
// Layout of the table (int16, in shared memory): entry (nibble v, pair p)
// with p = 8 w + q (packed word w of the row, nibble q of it) at index
// (8 v + q) L + w, L = K/16 rounded up to a multiple of 64. In one read a
// warp's lanes take words w = l + 32t at the same q, so lane l's entry sits
// in bank (w / 2) mod 32 whatever its nibble v (8 v L is a multiple of 64
// slots, 32 banks): lanes 2i and 2i + 1 share a bank, and a read costs one
// wavefront when their nibbles agree and two when they differ. Nibble values
// above 10 never occur in packed data.
//
// Per two weights the table form costs a shift, a mask, an address, a shared
// load and an add; the dp4a form costs half an instruction per weight. It is
// kept for the comparison.

#include "common.cuh"
#include "kernels.cuh"

namespace bl {

namespace {

constexpr int kLutThreads = 512;
constexpr int kLutWarps = kLutThreads / 32;
constexpr int kLutRows = 11;                    // nibble values 0..10

BL_DEVICE uint4 ldcg_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p) : "memory");
  return v;
}

BL_DEVICE int lut_stride(int K) { return (K / 16 + 63) / 64 * 64; }

// Widens 8 raw activations (bf16 or fp32) starting at element e to fp32.
template <int XIN>
BL_DEVICE void load8(const void* x, int e, float (&f)[8]) {
  if constexpr (XIN == kXinBF16) {
    const uint4 v = ldcg_v4(static_cast<const uint16_t*>(x) + e);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = __uint_as_float(w[i] << 16);
      f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  } else {
    const uint4 a = ldcg_v4(static_cast<const float*>(x) + e);
    const uint4 b = ldcg_v4(static_cast<const float*>(x) + e + 4);
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) f[i] = __uint_as_float(w[i]);
  }
}

}  // namespace

// Dynamic shared memory: the table [11 * 8][L] int16, the codes x_q [K] int8,
// then warp maxima [16].
template <int XIN>
__global__ void __launch_bounds__(kLutThreads, 1)
bl_gemv_lut(const uint8_t* __restrict__ wp, const void* __restrict__ x, const float* __restrict__ gamma,
            float* __restrict__ y, int N, int K) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int L = lut_stride(K);
  int16_t* s_t = reinterpret_cast<int16_t*>(smem);
  int8_t* s_xq = reinterpret_cast<int8_t*>(smem + static_cast<size_t>(kLutRows) * 8 * L * 2);
  float* s_red = reinterpret_cast<float*>(s_xq + ((K + 15) & ~15));
  pdl_wait();
  pdl_launch_dependents();
  x = launder(x);
  wp = launder(wp);
  gamma = launder(gamma);

  // ---- per-token absmax and codes (8 values per thread per step)
  float amax = 0.f;
  for (int e = 8 * tid; e < K; e += 8 * kLutThreads) {
    float f[8];
    load8<XIN>(x, e, f);
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(f[i]));
  }
  amax = warp_max(amax);
  if (lane == 0) s_red[warp] = amax;
  __syncthreads();
  const float s = token_scale(warp_max(lane < kLutWarps ? s_red[lane] : 0.f));
  const float rc = recip_for_div(s);
  for (int e = 8 * tid; e < K; e += 8 * kLutThreads) {
    float f[8];
    load8<XIN>(x, e, f);
    uint32_t c[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) c[i] = static_cast<uint32_t>(quant_code(f[i], s)) & 0xffu;
    uint2 o;
    o.x = c[0] | (c[1] << 8) | (c[2] << 16) | (c[3] << 24);
    o.y = c[4] | (c[5] << 8) | (c[6] << 16) | (c[7] << 24);
    *reinterpret_cast<uint2*>(s_xq + e) = o;
  }
  __syncthreads();

  // ---- the table: pair p = 8w + q, entries for nibbles 0..10
  const int P = K >> 1;
  for (int p = tid; p < P; p += kLutThreads) {
    const int x0 = s_xq[2 * p], x1 = s_xq[2 * p + 1];
    const int w = p >> 3, q = p & 7;
#pragma unroll
    for (int v = 0; v < kLutRows; ++v) {
      const int f0 = v & 3, f1 = v >> 2;
      const int t = (f0 < 3 && f1 < 3) ? (f0 - 1) * x0 + (f1 - 1) * x1 : 0;
      s_t[(8 * v + q) * L + w] = static_cast<int16_t>(t);
    }
  }
  __syncthreads();

  // ---- rows: one warp per row at a time, lanes over the row's packed words
  const float gm = __ldg(gamma);
  const int W = K >> 4;                           // packed words per row
  const uint32_t t32 = static_cast<uint32_t>(__cvta_generic_to_shared(s_t));
  const uint32_t row_bytes16 = 16u * static_cast<uint32_t>(L);   // bytes between nibble values (8 L slots)
  for (int n = blockIdx.x * kLutWarps + warp; n < N; n += gridDim.x * kLutWarps) {
    const uint32_t* wrow = reinterpret_cast<const uint32_t*>(wp + static_cast<size_t>(n) * (K >> 2));
    int acc = 0;
    for (int w0 = 0; w0 < W; w0 += 128) {
      uint32_t wv[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int w = w0 + lane + 32 * j;
        wv[j] = w < W ? __ldg(wrow + w) : 0x55555555u;          // fields 1: code 0, table entry 0
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t w = static_cast<uint32_t>(w0 + lane + 32 * j);
        if (static_cast<int>(w) < W) {
          // slot (8 v + q) L + w, two bytes each: base 2 (q L + w), plus v * 16 L
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const uint32_t v = (wv[j] >> (4 * q)) & 15u;
            const uint32_t a = t32 + 2u * (static_cast<uint32_t>(q) * static_cast<uint32_t>(L) + w) + v * row_bytes16;
            int16_t e;
            asm volatile("ld.shared.s16 %0, [%1];" : "=h"(e) : "r"(a));
            acc += e;
          }
        }
      }
    }
    acc = __reduce_add_sync(0xffffffffu, acc);
    if (lane == 0) y[n] = div_rn_recip(__fmul_rn(static_cast<float>(acc), gm), s, rc);
  }
}

size_t gemv_lut_smem(int K) {
  const size_t L = static_cast<size_t>((K / 16 + 63) / 64 * 64);
  return static_cast<size_t>(kLutRows) * 8 * L * 2 + ((static_cast<size_t>(K) + 15) & ~size_t(15)) + kLutWarps * 4;
}

cudaError_t launch_gemv_lut(const uint8_t* wp, const void* x, bool bf16, const float* gamma, float* y, int N, int K,
                            int sms, cudaStream_t s) {
  const size_t smem = gemv_lut_smem(K);
  const int grid = N < sms ? N : sms;
  if (bf16) {
    const cudaError_t e = ensure_smem(reinterpret_cast<const void*>(bl_gemv_lut<kXinBF16>), smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(bl_gemv_lut<kXinBF16>, dim3(grid), dim3(kLutThreads), smem, s, wp, x, gamma, y, N, K);
  }
  const cudaError_t e = ensure_smem(reinterpret_cast<const void*>(bl_gemv_lut<kXinF32>), smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(bl_gemv_lut<kXinF32>, dim3(grid), dim3(kLutThreads), smem, s, wp, x, gamma, y, N, K);
}

}  // namespace bl
