// Decode GEMV for one to four tokens: a per-token activation kernel and a
// packed-ternary x int8 contraction on dp4a, chained with programmatic
// dependent launch.
//
// Passages: "穿越1比特的奇幻旅程" (2B4T summary), section "GPU端：CUDA内核的定制
// 魔法" (W1.58A8 matmul over four-per-byte packed weights: pack, store, load,
// unpack, compute); "BitNet 1-bit LLM 的混合精度微调技术：渐进量化策略", body,
// quantisation functions (per-token absmax, eps = 1e-5) and the forward-pass
// sentence (multiply back by the factors).
//
// At M <= 4 the work is one stream of the packed weights (N*K/4 bytes) against
// a few KB of activations; a 2B-class projection (4.4 MB) lasts about as long
// as one HBM round trip, so the path is shaped to overlap everything with
// that round trip:
//   1. bl_act_tq (one CTA per token) quantises x once: scale s, optional
//      int8 codes in the caller's layout, the token sum of the codes, and the
//      codes again with each 16-code block transposed as a 4x4 byte matrix
//      (word i of a block holds the codes of k = 16b + 4j + i, j = 0..3).
//      Both kernels are launched as programmatic dependents: each first waits
//      for the grid before it (griddepcontrol.wait) and only then lets its
//      own dependent start, so a kernel can be resident before its
//      predecessor ends, while no early read can overtake a write of any
//      kernel but the one it waits for.
//   2. bl_gemv_w starts while (1) runs: every warp issues the loads of all its
//      weight words straight into registers (L1-bypassing, 128 contiguous
//      bytes per warp instruction), and only then waits for (1). The weights
//      are never written by (1), and (1) let this grid start only after its
//      own wait, so the early loads see every earlier write; everything (1)
//      writes is read after the wait.
//   3. Each warp owns whole rows of one k-part (the row is split into P parts
//      only when a lane's share would not fit in registers). Lane l takes
//      words l, l + 32, ... of the part and loads the matching transposed
//      activation words once for all its rows. A packed word masked into its
//      four field planes, (word & 0x03030303 << 2i), is multiplied by word i
//      of the activation block with dp4a:
//        sum_k field * x = acc0 + acc1/4 + acc2/16 + acc3/64   (each exact)
//      and field = code + 1, so sum_k code * x = that - sum_k x.
//   4. One shuffle reduction per row; lane 0 writes y = fp32(fp32(acc *
//      gamma) / s) directly (P = 1) or adds into shared memory for a final
//      pass (P > 1; integer atomics, so the order does not matter).
// There is no shared memory and no block barrier on the P = 1 path.

#include "common.cuh"
#include "kernels.cuh"

namespace bl {

namespace {

constexpr int kWarps = kGemvFusedThreads / 32;
// weight words a lane holds in registers (fewer when more tokens need accumulators)
constexpr int word_regs(int mt) { return mt == 1 ? 48 : (mt == 2 ? 36 : 24); }
// rows per warp: as many as the word registers allow, at most 16 (unrolled code size)
constexpr int rows_per_warp(int mt, int kw) { return word_regs(mt) / kw < 16 ? word_regs(mt) / kw : 16; }

BL_DEVICE uint32_t ld_stream_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}

// Coherent loads that the compiler keeps after pdl_wait(): data written by the
// grid this kernel depends on must not come through the read-only path or be
// hoisted above the wait.
BL_DEVICE uint4 ld_after_wait_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p) : "memory");
  return v;
}
BL_DEVICE int ld_after_wait_s32(const int* p) {
  int v;
  asm volatile("ld.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
BL_DEVICE float ld_after_wait_f32(const float* p) {
  float v;
  asm volatile("ld.global.f32 %0, [%1];" : "=f"(v) : "l"(p) : "memory");
  return v;
}

// 16 activations starting at `off`, widened exactly to fp32.
template <int XIN>
BL_DEVICE void load16(const void* x, size_t off, float (&f)[16]) {
  if constexpr (XIN == kXinF32) {
    const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(x) + off);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float4 v = __ldg(p + i);
      f[4 * i] = v.x; f[4 * i + 1] = v.y; f[4 * i + 2] = v.z; f[4 * i + 3] = v.w;
    }
  } else {
    const uint4* p = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(x) + off);
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const uint4 v = __ldg(p + i);
      const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        f[8 * i + 2 * j] = __uint_as_float(u[j] << 16);
        f[8 * i + 2 * j + 1] = __uint_as_float(u[j] & 0xffff0000u);
      }
    }
  }
}

// Code of one activation, clip(rint(fp32(x * s)), -128, 127), returned in the
// low byte (two's complement). Rounding uses the classic 1.5 * 2^23 addition:
// for |v| <= 2^22, fp32 v + 12582912 lies in [2^23, 2^24) where the spacing is
// 1, so the round-to-nearest-even addition lands on 12582912 + rint(v) and the
// integer sits in the low mantissa bits (0x4B400000 has a zero low byte). The
// clamp comes first; it is exact and leaves integers in range unchanged.
BL_DEVICE uint32_t code_byte(float x, float s) {
  const float v = fminf(fmaxf(__fmul_rn(x, s), -128.f), 127.f);
  return __float_as_uint(__fadd_rn(v, 12582912.f));
}

BL_DEVICE uint32_t pack4(uint32_t b0, uint32_t b1, uint32_t b2, uint32_t b3) {
  return __byte_perm(__byte_perm(b0, b1, 0x0040), __byte_perm(b2, b3, 0x0040), 0x5410);
}

BL_DEVICE int sum16(const uint32_t (&w)[4]) {
  int s = dp4a_ss(static_cast<int>(w[0]), 0x01010101, 0);
  s = dp4a_ss(static_cast<int>(w[1]), 0x01010101, s);
  s = dp4a_ss(static_cast<int>(w[2]), 0x01010101, s);
  return dp4a_ss(static_cast<int>(w[3]), 0x01010101, s);
}

}  // namespace

// ---- 1. per-token activation pass (one CTA of kActTqThreads per token)
template <int XIN>
__global__ void __launch_bounds__(kActTqThreads)
bl_act_tq(const void* __restrict__ x, const float* __restrict__ scale_in, int K, int8_t* __restrict__ xq_out,
          float* __restrict__ scale_out, uint8_t* __restrict__ xt, int* __restrict__ rowsum) {
  __shared__ float s_red[kActTqThreads / 32];
  __shared__ int s_sum[kActTqThreads / 32];
  // Wait for the previous grid (it may have produced x) before anything else,
  // and only then let the contraction start: its early weight loads must not
  // overtake writes of the kernels before this one.
  pdl_wait();
  pdl_launch_dependents();
  const int m = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nblk = K >> 4;
  const size_t row = static_cast<size_t>(m) * K;
  int part = 0;
  if constexpr (XIN == kXinI8) {
    for (int b = tid; b < nblk; b += blockDim.x) {
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(static_cast<const int8_t*>(x) + row) + b);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
      part += sum16(w);
      uint4 t;
      transpose4x4_bytes(w[0], w[1], w[2], w[3], t.x, t.y, t.z, t.w);
      *reinterpret_cast<uint4*>(xt + row + 16 * b) = t;
    }
    if (tid == 0 && scale_out) scale_out[m] = __ldg(scale_in + m);
  } else {
    float f0[16];                                   // the first block of each thread stays in registers
    if (tid < nblk) load16<XIN>(x, row + 16 * tid, f0);
    float amax = 0.f;
    for (int b = tid; b < nblk; b += blockDim.x) {
      float f[16];
      if (b == tid) {
#pragma unroll
        for (int j = 0; j < 16; ++j) f[j] = f0[j];
      } else {
        load16<XIN>(x, row + 16 * b, f);
      }
#pragma unroll
      for (int j = 0; j < 16; ++j) amax = fmaxf(amax, fabsf(f[j]));
    }
    amax = warp_max(amax);
    if (lane == 0) s_red[warp] = amax;
    __syncthreads();
    float a = 0.f;
#pragma unroll
    for (int w = 0; w < kActTqThreads / 32; ++w) a = fmaxf(a, s_red[w]);
    const float s = token_scale(a);
    if (tid == 0) scale_out[m] = s;
    for (int b = tid; b < nblk; b += blockDim.x) {
      float f[16];
      if (b == tid) {
#pragma unroll
        for (int j = 0; j < 16; ++j) f[j] = f0[j];
      } else {
        load16<XIN>(x, row + 16 * b, f);
      }
      uint32_t w[4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
        w[i] = pack4(code_byte(f[4 * i], s), code_byte(f[4 * i + 1], s), code_byte(f[4 * i + 2], s),
                     code_byte(f[4 * i + 3], s));
      if (xq_out) *reinterpret_cast<uint4*>(xq_out + row + 16 * b) = make_uint4(w[0], w[1], w[2], w[3]);
      part += sum16(w);
      uint4 t;
      transpose4x4_bytes(w[0], w[1], w[2], w[3], t.x, t.y, t.z, t.w);
      *reinterpret_cast<uint4*>(xt + row + 16 * b) = t;
    }
  }
  part = warp_sum(part);
  if (lane == 0) s_sum[warp] = part;
  __syncthreads();
  if (tid == 0) {
    int t = 0;
#pragma unroll
    for (int w = 0; w < kActTqThreads / 32; ++w) t += s_sum[w];
    rowsum[m] = t;
  }
}

// ---- 2..4. the contraction (KW = words per lane per part, exact for this
// shape; RW = rows per warp; P divides kWarps, so warp w works on part w % P)
template <int MT, int KW, bool OUT_ACC>
__global__ void __launch_bounds__(kGemvFusedThreads, 1)
bl_gemv_w(const uint8_t* __restrict__ wp, const uint8_t* xt, const int* rowsum, const float* scale,
          const float* gamma, void* __restrict__ out, int M, int N, int K, int rows_per_cta, int P) {
  constexpr int kRW = rows_per_warp(MT, KW);
  extern __shared__ __align__(16) int s_acc[];      // [rows][MT], only when P > 1
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n0 = blockIdx.x * rows_per_cta;
  const int R = min(rows_per_cta, N - n0);
  if (R <= 0) return;
  const int words = K >> 4;                         // packed 32-bit words per row = 16-code blocks per token
  const int part = warp % P;
  const int w_lo = part * 32 * KW;
  const int row_step = kWarps / P;

  // weight words straight into registers, before waiting for the activations
  uint32_t wr[kRW][KW];
  const uint32_t* wbase = reinterpret_cast<const uint32_t*>(wp) + static_cast<size_t>(n0) * words + w_lo + lane;
#pragma unroll
  for (int i = 0; i < kRW; ++i) {
    const int r = warp / P + row_step * i;
    if (r < R) {                                    // warp-uniform
      const uint32_t* rp = wbase + static_cast<size_t>(r) * words;
#pragma unroll
      for (int j = 0; j < KW; ++j) wr[i][j] = (w_lo + lane + 32 * j < words) ? ld_stream_u32(rp + 32 * j) : 0u;
    }
  }
  if (P > 1)
    for (int i = tid; i < R * MT; i += blockDim.x) s_acc[i] = 0;
  pdl_wait();                                       // the activation pass has finished
  pdl_launch_dependents();                          // the next grid waits for this one before its own reads

  uint4 xr[KW][MT];
#pragma unroll
  for (int j = 0; j < KW; ++j) {
    const int wd = w_lo + lane + 32 * j;
#pragma unroll
    for (int m = 0; m < MT; ++m)
      xr[j][m] = (wd < words && m < M) ? ld_after_wait_v4(xt + static_cast<size_t>(m) * K + 16 * static_cast<size_t>(wd))
                                       : make_uint4(0u, 0u, 0u, 0u);
  }
  int rs[MT];
  float sc[MT], rc[MT];
#pragma unroll
  for (int m = 0; m < MT; ++m) {
    rs[m] = m < M ? ld_after_wait_s32(rowsum + m) : 0;
    sc[m] = (!OUT_ACC && m < M) ? ld_after_wait_f32(scale + m) : 1.f;
    rc[m] = recip_for_div(sc[m]);
  }
  const float gm = OUT_ACC ? 0.f : ld_after_wait_f32(gamma);
  if (P > 1) __syncthreads();                       // s_acc cleared

  int vsum[kRW][MT];
#pragma unroll
  for (int i = 0; i < kRW; ++i) {
    const int r = warp / P + row_step * i;
#pragma unroll
    for (int m = 0; m < MT; ++m) vsum[i][m] = 0;
    if (r < R) {                                    // warp-uniform
      int acc[MT][4];
#pragma unroll
      for (int m = 0; m < MT; ++m) acc[m][0] = acc[m][1] = acc[m][2] = acc[m][3] = 0;
#pragma unroll
      for (int j = 0; j < KW; ++j) {
        const uint32_t wv = wr[i][j];
        const uint32_t a0 = wv & 0x03030303u, a1 = wv & 0x0c0c0c0cu, a2 = wv & 0x30303030u, a3 = wv & 0xc0c0c0c0u;
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          acc[m][0] = dp4a_us(a0, static_cast<int>(xr[j][m].x), acc[m][0]);
          acc[m][1] = dp4a_us(a1, static_cast<int>(xr[j][m].y), acc[m][1]);
          acc[m][2] = dp4a_us(a2, static_cast<int>(xr[j][m].z), acc[m][2]);
          acc[m][3] = dp4a_us(a3, static_cast<int>(xr[j][m].w), acc[m][3]);
        }
      }
#pragma unroll
      for (int m = 0; m < MT; ++m) vsum[i][m] = acc[m][0] + (acc[m][1] >> 2) + (acc[m][2] >> 4) + (acc[m][3] >> 6);
    }
  }
  // reductions of all rows together (independent shuffle chains)
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
    for (int i = 0; i < kRW; ++i) {
      if (warp / P + row_step * i < R) {
#pragma unroll
        for (int m = 0; m < MT; ++m) vsum[i][m] += __shfl_xor_sync(0xffffffffu, vsum[i][m], o);
      }
    }
  }
  if (lane == 0) {
#pragma unroll
    for (int i = 0; i < kRW; ++i) {
      const int r = warp / P + row_step * i;
      if (r < R) {
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          if (m < M) {
            if (P > 1) {
              atomicAdd(&s_acc[r * MT + m], vsum[i][m]);
            } else {
              const size_t o = static_cast<size_t>(m) * N + n0 + r;
              if constexpr (OUT_ACC) {
                static_cast<int32_t*>(out)[o] = vsum[i][m] - rs[m];
              } else {
                static_cast<float*>(out)[o] =
                    div_rn_recip(__fmul_rn(static_cast<float>(vsum[i][m] - rs[m]), gm), sc[m], rc[m]);
              }
            }
          }
        }
      }
    }
  }
  if (P > 1) {
    __syncthreads();
    for (int i = tid; i < M * R; i += blockDim.x) {
      const int m = i / R, r = i - m * R;
      int rsm = 0;
      float scm = 1.f, rcm = 0.f;
#pragma unroll
      for (int mm = 0; mm < MT; ++mm) {
        if (mm == m) {
          rsm = rs[mm];
          scm = sc[mm];
          rcm = rc[mm];
        }
      }
      const int a = s_acc[r * MT + m] - rsm;
      const size_t o = static_cast<size_t>(m) * N + n0 + r;
      if constexpr (OUT_ACC) {
        static_cast<int32_t*>(out)[o] = a;
      } else {
        static_cast<float*>(out)[o] = div_rn_recip(__fmul_rn(static_cast<float>(a), gm), scm, rcm);
      }
    }
  }
}

size_t gemv_fused_plan(int M, int N, int K, int sms, int* rows_per_cta, int* parts) {
  if (M < 1 || M > kGemvFusedMaxM || K % 64 != 0 || N < 1) return 0;
  const int mt = M <= 1 ? 1 : (M <= 2 ? 2 : 4);
  const int kw_max = 8 / mt;
  const int words = K / 16;
  int P = 1;
  while (P < kWarps && (words + 32 * P - 1) / (32 * P) > kw_max) P *= 2;
  const int kw = (words + 32 * P - 1) / (32 * P);
  if (kw > kw_max) return 0;
  int rows = (N + sms - 1) / sms;
  const int max_rows = rows_per_warp(mt, kw) * (kWarps / P);
  if (rows > max_rows) rows = max_rows;
  *rows_per_cta = rows;
  *parts = P;
  // dynamic shared memory: the cross-part accumulators (P > 1) plus one int so
  // the size is never zero
  return static_cast<size_t>(P > 1 ? rows * mt * 4 : 0) + 16;
}

namespace {

template <int MT, int KW, bool OUT_ACC>
cudaError_t launch_w(const uint8_t* wp, const uint8_t* xt, const int* rowsum, const float* scale, const float* gamma,
                     void* out, int M, int N, int K, int rows, int P, size_t smem, cudaStream_t s) {
  const int grid = (N + rows - 1) / rows;
  return launch_pdl(bl_gemv_w<MT, KW, OUT_ACC>, dim3(grid), dim3(kGemvFusedThreads), smem, s, wp, xt, rowsum,
                          scale, gamma, out, M, N, K, rows, P);
}

template <int MT, int KW>
cudaError_t pick_kw(int kw, bool out_acc, const uint8_t* wp, const uint8_t* xt, const int* rowsum,
                    const float* scale, const float* gamma, void* out, int M, int N, int K, int rows, int P,
                    size_t smem, cudaStream_t s) {
  if constexpr (KW > 1) {
    if (kw < KW)
      return pick_kw<MT, KW - 1>(kw, out_acc, wp, xt, rowsum, scale, gamma, out, M, N, K, rows, P, smem, s);
  }
  if (out_acc) return launch_w<MT, KW, true>(wp, xt, rowsum, scale, gamma, out, M, N, K, rows, P, smem, s);
  return launch_w<MT, KW, false>(wp, xt, rowsum, scale, gamma, out, M, N, K, rows, P, smem, s);
}

}  // namespace

cudaError_t launch_gemv_fused(const uint8_t* wp, const void* x, int xin, const float* scale_in, const float* gamma,
                              void* out, bool out_acc, int8_t* xq_out, float* scale_out, int M, int N, int K,
                              int rows_per_cta, int parts, size_t smem, void* workspace, cudaStream_t s) {
  uint8_t* xt = static_cast<uint8_t*>(workspace);
  uint8_t* b = xt + ((static_cast<size_t>(M) * K + 255) & ~size_t(255));
  int* rowsum = reinterpret_cast<int*>(b);
  float* sc = reinterpret_cast<float*>(b + ((static_cast<size_t>(M) * 4 + 255) & ~size_t(255)));
  if (scale_out) sc = scale_out;
  cudaError_t e;
  if (xin == kXinF32)
    e = launch_pdl(bl_act_tq<kXinF32>, dim3(M), dim3(kActTqThreads), 0, s, x, scale_in, K, xq_out, sc, xt,
                         rowsum);
  else if (xin == kXinBF16)
    e = launch_pdl(bl_act_tq<kXinBF16>, dim3(M), dim3(kActTqThreads), 0, s, x, scale_in, K, xq_out, sc, xt,
                         rowsum);
  else
    e = launch_pdl(bl_act_tq<kXinI8>, dim3(M), dim3(kActTqThreads), 0, s, x, scale_in, K,
                         static_cast<int8_t*>(nullptr), static_cast<float*>(nullptr), xt, rowsum);
  if (e != cudaSuccess) return e;
  const float* scale = (xin == kXinI8) ? scale_in : sc;
  const int words = K / 16;
  const int kw = (words + 32 * parts - 1) / (32 * parts);
  if (M <= 1) return pick_kw<1, 8>(kw, out_acc, wp, xt, rowsum, scale, gamma, out, M, N, K, rows_per_cta, parts, smem, s);
  if (M <= 2) return pick_kw<2, 4>(kw, out_acc, wp, xt, rowsum, scale, gamma, out, M, N, K, rows_per_cta, parts, smem, s);
  return pick_kw<4, 2>(kw, out_acc, wp, xt, rowsum, scale, gamma, out, M, N, K, rows_per_cta, parts, smem, s);
}

cudaError_t take_gemv_wait_error(int* flag) {
  *flag = 0;   // this path has no asynchronous copies to wait for
  return cudaSuccess;
}

}  // namespace bl
