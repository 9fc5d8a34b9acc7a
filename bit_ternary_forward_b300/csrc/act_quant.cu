// Per-token absmax int8 activation quantisation.
//
// Passages: "BitNet 1-bit LLM 的混合精度微调技术：渐进量化策略", body, quantisation
// functions (activation absmax = max(|X|, eps = 1e-5); per-token 8-bit
// absmax); "穿越1比特的奇幻旅程" (2B4T summary), section "架构创新：量化魔法的
// 背后" (INT8 activations, absmax per token).
//
// One CTA per token. Pass 1 reads the row with 8- or 16-byte vector loads and
// reduces max|x| with warp shuffles; pass 2 re-reads the row (now in L1/L2),
// computes x_q = clip(rint(fp32(x * s)), -128, 127) and stores four codes per
// 32-bit word.

#include "common.cuh"
#include "kernels.cuh"

namespace bl {

namespace {

template <typename T> struct Vec4;
template <> struct Vec4<float> {
  using type = float4;
  static BL_DEVICE void unpack(const float4& v, float (&f)[4]) { f[0] = v.x; f[1] = v.y; f[2] = v.z; f[3] = v.w; }
};
template <> struct Vec4<uint16_t> {   // bf16 bits
  using type = uint2;
  static BL_DEVICE void unpack(const uint2& v, float (&f)[4]) {
    f[0] = __uint_as_float(v.x << 16); f[1] = __uint_as_float(v.x & 0xffff0000u);
    f[2] = __uint_as_float(v.y << 16); f[3] = __uint_as_float(v.y & 0xffff0000u);
  }
};

}  // namespace

template <typename T>
__global__ void __launch_bounds__(kActThreads)
bl_act_quant(const T* __restrict__ x, int K, int8_t* __restrict__ xq, float* __restrict__ scale) {
  using V = typename Vec4<T>::type;
  __shared__ float s_red[kActThreads / 32];
  pdl_wait();
  pdl_launch_dependents();
  x = launder(x);
  const int m = blockIdx.x;
  const V* row = reinterpret_cast<const V*>(x + static_cast<size_t>(m) * K);
  const int nv = K >> 2;   // K % 4 == 0

  float amax = 0.f;
  for (int i = threadIdx.x; i < nv; i += blockDim.x) {
    float f[4];
    Vec4<T>::unpack(row[i], f);
    amax = fmaxf(amax, fmaxf(fmaxf(fabsf(f[0]), fabsf(f[1])), fmaxf(fabsf(f[2]), fabsf(f[3]))));
  }
  amax = warp_max(amax);
  if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = amax;
  __syncthreads();
  if (threadIdx.x < 32) {
    float v = threadIdx.x < (blockDim.x >> 5) ? s_red[threadIdx.x] : 0.f;
    v = warp_max(v);
    if (threadIdx.x == 0) s_red[0] = v;
  }
  __syncthreads();
  const float s = token_scale(s_red[0]);
  if (threadIdx.x == 0) scale[m] = s;

  uint32_t* out = reinterpret_cast<uint32_t*>(xq + static_cast<size_t>(m) * K);
  for (int i = threadIdx.x; i < nv; i += blockDim.x) {
    float f[4];
    Vec4<T>::unpack(row[i], f);
    const uint32_t q0 = static_cast<uint32_t>(quant_code(f[0], s)) & 0xffu;
    const uint32_t q1 = static_cast<uint32_t>(quant_code(f[1], s)) & 0xffu;
    const uint32_t q2 = static_cast<uint32_t>(quant_code(f[2], s)) & 0xffu;
    const uint32_t q3 = static_cast<uint32_t>(quant_code(f[3], s)) & 0xffu;
    out[i] = q0 | (q1 << 8) | (q2 << 16) | (q3 << 24);
  }
}

cudaError_t launch_act_quant(const void* x, bool bf16, int M, int K, int8_t* xq, float* scale, cudaStream_t s) {
  if (bf16) return launch_pdl(bl_act_quant<uint16_t>, dim3(M), dim3(kActThreads), 0, s,
                              static_cast<const uint16_t*>(x), K, xq, scale);
  return launch_pdl(bl_act_quant<float>, dim3(M), dim3(kActThreads), 0, s, static_cast<const float*>(x), K, xq, scale);
}

}  // namespace bl
