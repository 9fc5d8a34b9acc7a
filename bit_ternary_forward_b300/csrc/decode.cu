// Decode and skinny contraction: packed ternary weights x int8 activations on
// the warp-level integer tensor-core MMA, for a few tokens (5 <= M <= 16 with
// K % 64 == 0; from M = 17 the tcgen05 path of prefill.cu is faster).
//
// Passages: "穿越1比特的奇幻旅程" (2B4T summary), section "GPU端：CUDA内核的定制
// 魔法" (W1.58A8 matmul over four-per-byte packed weights: pack, store, load,
// unpack, compute); "BitNet 1-bit LLM 的混合精度微调技术：渐进量化策略", body,
// quantisation functions (per-token absmax with eps = 1e-5) and the
// forward-pass sentence (multiply back by the factors).
//
// Work split. Each CTA owns a contiguous block of weight rows [n0, n0 + R).
// Before its dependency wait, thread 0 prefetches the block into L2 (a hint
// that cannot change what later loads see). After the wait,
// one thread copies the block into shared memory with one bulk async copy
// per row (rows padded by 16 bytes so that the MMA fragment loads are free of
// bank conflicts), one mbarrier per 16-row tile; meanwhile all threads
// quantise (or stage) the activations of up to 8 tokens. The contraction
// runs on mma.sync.m16n8k32 (u8 x s8 -> s32): weight rows are the MMA's M
// dimension (16 per tile), tokens its N dimension (8), and warp w takes the
// k-steps w, w + 16, ... of every tile, so the activation fragment of a
// k-step is loaded once for all tiles. Partial sums meet in shared memory
// (integer atomics, so the order does not matter) and the epilogue writes
// y = fp32(fp32(acc * gamma) / s) or the int32 accumulator.
//
// Fragment mapping. A packed 32-bit word holds 16 codes of one row: byte j
// carries k = 16w + 4j .. 16w + 4j + 3, the code of k = 16w + 4j + i in bits
// 2i..2i+1 as the field value code + 1. Thread (g, t) of the MMA (g = lane/4,
// t = lane%4) owns A-fragment slots 4t..4t+3 of rows g and g+8; it fills them
// with plane t of the word, (word >> 2t) & 0x03030303, whose byte j is the
// field of k = 16w + 4j + t. So slot 4t + j stands for k = 16w + 4j + t, and
// the B fragment (the activations) must hold x[16w + 4j + t] in byte j: word
// t of the 16-byte activation block transposed as a 4x4 byte matrix. Slots
// 16..31 do the same for the next word. The MMA then gives
//   sum_k field * x = sum_k code * x + sum_k x,
// and the epilogue subtracts the per-token sum of x_q.

#include "async.cuh"
#include "common.cuh"
#include "kernels.cuh"

namespace bl {

namespace {

constexpr int kWarps = kDecodeThreads / 32;
constexpr int kTok = 8;                 // tokens per MMA column block
// Set (never cleared by a kernel) when a bounded mbarrier wait gave up.
__device__ int g_wait_error;

BL_DEVICE void mma_u8s8(int (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.s32.u8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+r"(c[0]), "+r"(c[1]), "+r"(c[2]), "+r"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Byte offset, inside one token's staged row, of word t of transposed block b:
// the two blocks of a 32-k step sit side by side per t (8 bytes), so the B
// fragment of thread t is one 64-bit load.
BL_DEVICE int xoff(int block, int t) { return 32 * (block >> 1) + 8 * t + 4 * (block & 1); }

// Stages 16 codes (q[0..15] = x_q[16b .. 16b+15]) of one token, transposed.
BL_DEVICE void stage_block(uint8_t* xrow, int block, const uint32_t (&w)[4]) {
  uint32_t t0, t1, t2, t3;
  transpose4x4_bytes(w[0], w[1], w[2], w[3], t0, t1, t2, t3);
  *reinterpret_cast<uint32_t*>(xrow + xoff(block, 0)) = t0;
  *reinterpret_cast<uint32_t*>(xrow + xoff(block, 1)) = t1;
  *reinterpret_cast<uint32_t*>(xrow + xoff(block, 2)) = t2;
  *reinterpret_cast<uint32_t*>(xrow + xoff(block, 3)) = t3;
}

template <int XIN> struct XLoad;
template <> struct XLoad<kXinF32> {   // 16 fp32 values
  static BL_DEVICE void load(const void* x, size_t off, float (&f)[16]) {
    const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(x) + off);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float4 v = __ldg(p + i);
      f[4 * i] = v.x; f[4 * i + 1] = v.y; f[4 * i + 2] = v.z; f[4 * i + 3] = v.w;
    }
  }
};
template <> struct XLoad<kXinBF16> {  // 16 bf16 values, widened exactly
  static BL_DEVICE void load(const void* x, size_t off, float (&f)[16]) {
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
};

}  // namespace

// Dynamic shared memory layout (bytes):
//   [0, wbytes)              weight rows, R_pad rows of wstride bytes
//   [wbytes, +8*xstride)     activations of 8 tokens, transposed blocks
//   then int32 acc[R_pad][8], int32 rowsum[8], float scale[8], float red[kWarps][8],
//   uint64 mbarrier[n_tiles]
template <int XIN, bool OUT_ACC>
__global__ void __launch_bounds__(kDecodeThreads, 1)
bl_decode_mma(const uint8_t* __restrict__ wp, const void* __restrict__ x, const float* __restrict__ scale_in,
              const float* __restrict__ gamma, void* __restrict__ out, int8_t* __restrict__ xq_out,
              float* __restrict__ scale_out, int M, int N, int K, int rows_per_cta) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, t = lane & 3;

  const int n0 = blockIdx.x * rows_per_cta;
  const int R = min(rows_per_cta, N - n0);
  if (R <= 0) return;
  const int n_tiles = (R + 15) >> 4;
  const int rp = (rows_per_cta + 15) & ~15;
  const int rowbytes = K >> 2;
  const int wstride = rowbytes + 16;
  const int xstride = K + 32;
  const int nblk = K >> 4;
  const int ksteps = K >> 5;

  uint8_t* s_w = smem;
  uint8_t* s_x = smem + static_cast<size_t>(rp) * wstride;
  int* s_acc = reinterpret_cast<int*>(s_x + static_cast<size_t>(kTok) * xstride);
  int* s_rowsum = s_acc + rp * kTok;
  float* s_scale = reinterpret_cast<float*>(s_rowsum + kTok);
  float* s_red = s_scale + kTok;
  uint64_t* s_bar = reinterpret_cast<uint64_t*>((reinterpret_cast<uintptr_t>(s_red + kWarps * kTok) + 7) & ~uintptr_t(7));

  // the block's packed rows start moving into L2 while the previous kernel ends
  if (tid == 0) prefetch_l2_range(wp + static_cast<size_t>(n0) * rowbytes, static_cast<uint64_t>(R) * rowbytes);
  pdl_wait();
  pdl_launch_dependents();
  x = launder(x);
  scale_in = launder(scale_in);
  gamma = launder(gamma);
  // ---- issue the weight copies (one thread), one mbarrier per 16-row tile
  if (tid == 0) {
    for (int tl = 0; tl < n_tiles; ++tl) mbar_init(&s_bar[tl], 1);
    mbar_init_fence();
    for (int tl = 0; tl < n_tiles; ++tl) {
      const int r_lo = tl * 16, r_hi = min(R, r_lo + 16);
      mbar_expect_tx(&s_bar[tl], static_cast<uint32_t>((r_hi - r_lo) * rowbytes));
      for (int r = r_lo; r < r_hi; ++r)
        bulk_copy_g2s(s_w + static_cast<size_t>(r) * wstride, wp + static_cast<size_t>(n0 + r) * rowbytes,
                      static_cast<uint32_t>(rowbytes), &s_bar[tl]);
    }
  }

  const float gm = OUT_ACC ? 0.f : __ldg(gamma);
  bool ok = true;

  for (int m0 = 0; m0 < M; m0 += kTok) {
    const int mt = min(kTok, M - m0);
    // ---- stage the activations of tokens m0 .. m0+mt-1 (zeros for the rest)
    for (int i = tid; i < kTok * rp; i += blockDim.x) s_acc[i] = 0;
    if constexpr (XIN == kXinI8) {
      int part[kTok];
#pragma unroll
      for (int m = 0; m < kTok; ++m) part[m] = 0;
      for (int i = tid; i < kTok * nblk; i += blockDim.x) {
        const int m = i / nblk, b = i - m * nblk;
        uint32_t w[4] = {0u, 0u, 0u, 0u};
        if (m < mt) {
          const uint4 v = __ldg(reinterpret_cast<const uint4*>(static_cast<const int8_t*>(x) +
                                                              static_cast<size_t>(m0 + m) * K) + b);
          w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
        }
        int s = 0;
        s = dp4a_ss(static_cast<int>(w[0]), 0x01010101, s);
        s = dp4a_ss(static_cast<int>(w[1]), 0x01010101, s);
        s = dp4a_ss(static_cast<int>(w[2]), 0x01010101, s);
        s = dp4a_ss(static_cast<int>(w[3]), 0x01010101, s);
#pragma unroll
        for (int mm = 0; mm < kTok; ++mm) part[mm] += (mm == m) ? s : 0;
        stage_block(s_x + static_cast<size_t>(m) * xstride, b, w);
      }
#pragma unroll
      for (int m = 0; m < kTok; ++m) {
        const int v = warp_sum(part[m]);
        if (lane == 0) reinterpret_cast<int*>(s_red)[warp * kTok + m] = v;
      }
      __syncthreads();
      if (tid < kTok) {
        int s = 0;
        for (int w = 0; w < kWarps; ++w) s += reinterpret_cast<int*>(s_red)[w * kTok + tid];
        s_rowsum[tid] = s;
        s_scale[tid] = (OUT_ACC || tid >= mt) ? 1.f : __ldg(scale_in + m0 + tid);
      }
    } else {
      // pass 1: per-token absmax
      float amax[kTok];
#pragma unroll
      for (int m = 0; m < kTok; ++m) amax[m] = 0.f;
      for (int i = tid; i < mt * nblk; i += blockDim.x) {
        const int m = i / nblk, b = i - m * nblk;
        float f[16];
        XLoad<XIN>::load(x, static_cast<size_t>(m0 + m) * K + 16 * b, f);
        float a = 0.f;
#pragma unroll
        for (int j = 0; j < 16; ++j) a = fmaxf(a, fabsf(f[j]));
#pragma unroll
        for (int mm = 0; mm < kTok; ++mm) amax[mm] = (mm == m) ? fmaxf(amax[mm], a) : amax[mm];
      }
#pragma unroll
      for (int m = 0; m < kTok; ++m) {
        const float v = warp_max(amax[m]);
        if (lane == 0) s_red[warp * kTok + m] = v;
      }
      __syncthreads();
      if (tid < kTok) {
        float a = 0.f;
        for (int w = 0; w < kWarps; ++w) a = fmaxf(a, s_red[w * kTok + tid]);
        const float s = token_scale(a);
        s_scale[tid] = s;
        if (scale_out && blockIdx.x == 0 && tid < mt) scale_out[m0 + tid] = s;
      }
      __syncthreads();
      // pass 2: codes, transposed into shared memory, and per-token sums
      int part[kTok];
#pragma unroll
      for (int m = 0; m < kTok; ++m) part[m] = 0;
      for (int i = tid; i < kTok * nblk; i += blockDim.x) {
        const int m = i / nblk, b = i - m * nblk;
        uint32_t w[4] = {0u, 0u, 0u, 0u};
        if (m < mt) {
          float f[16];
          XLoad<XIN>::load(x, static_cast<size_t>(m0 + m) * K + 16 * b, f);
          const float s = s_scale[m];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint32_t q0 = static_cast<uint32_t>(quant_code(f[4 * j], s)) & 0xffu;
            const uint32_t q1 = static_cast<uint32_t>(quant_code(f[4 * j + 1], s)) & 0xffu;
            const uint32_t q2 = static_cast<uint32_t>(quant_code(f[4 * j + 2], s)) & 0xffu;
            const uint32_t q3 = static_cast<uint32_t>(quant_code(f[4 * j + 3], s)) & 0xffu;
            w[j] = q0 | (q1 << 8) | (q2 << 16) | (q3 << 24);
          }
          if (xq_out && blockIdx.x == 0)
            *reinterpret_cast<uint4*>(xq_out + static_cast<size_t>(m0 + m) * K + 16 * b) = make_uint4(w[0], w[1], w[2], w[3]);
        }
        int s = 0;
        s = dp4a_ss(static_cast<int>(w[0]), 0x01010101, s);
        s = dp4a_ss(static_cast<int>(w[1]), 0x01010101, s);
        s = dp4a_ss(static_cast<int>(w[2]), 0x01010101, s);
        s = dp4a_ss(static_cast<int>(w[3]), 0x01010101, s);
#pragma unroll
        for (int mm = 0; mm < kTok; ++mm) part[mm] += (mm == m) ? s : 0;
        stage_block(s_x + static_cast<size_t>(m) * xstride, b, w);
      }
      __syncthreads();   // s_red reads of pass 1 are done before it is reused
#pragma unroll
      for (int m = 0; m < kTok; ++m) {
        const int v = warp_sum(part[m]);
        if (lane == 0) reinterpret_cast<int*>(s_red)[warp * kTok + m] = v;
      }
      __syncthreads();
      if (tid < kTok) {
        int s = 0;
        for (int w = 0; w < kWarps; ++w) s += reinterpret_cast<int*>(s_red)[w * kTok + tid];
        s_rowsum[tid] = s;
      }
    }
    __syncthreads();

    // ---- contraction: warp w takes k-steps w, w + kWarps, ... of every tile
    int acc[6][4];
#pragma unroll
    for (int i = 0; i < 6; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0;
    const uint8_t* xrow = s_x + static_cast<size_t>(g) * xstride + 8 * t;
    const int shift = 2 * t;
    for (int tl0 = 0; tl0 < n_tiles; tl0 += 6) {
      const int nt = min(6, n_tiles - tl0);
      if (m0 == 0) {
        for (int i = 0; i < nt; ++i) ok = mbar_wait_sleep(&s_bar[tl0 + i], 0u) && ok;
      }
      for (int ks = warp; ks < ksteps; ks += kWarps) {
        const uint2 bv = *reinterpret_cast<const uint2*>(xrow + 32 * ks);
#pragma unroll
        for (int i = 0; i < 6; ++i) {
          if (i < nt) {
            const uint8_t* wr = s_w + static_cast<size_t>((tl0 + i) * 16 + g) * wstride + 8 * ks;
            const uint2 lo = *reinterpret_cast<const uint2*>(wr);
            const uint2 hi = *reinterpret_cast<const uint2*>(wr + 8 * wstride);
            const uint32_t a0 = (lo.x >> shift) & 0x03030303u;
            const uint32_t a2 = (lo.y >> shift) & 0x03030303u;
            const uint32_t a1 = (hi.x >> shift) & 0x03030303u;
            const uint32_t a3 = (hi.y >> shift) & 0x03030303u;
            mma_u8s8(acc[i], a0, a1, a2, a3, bv.x, bv.y);
          }
        }
      }
#pragma unroll
      for (int i = 0; i < 6; ++i) {
        if (i < nt) {
          const int r = (tl0 + i) * 16 + g;
          int* row0 = s_acc + r * kTok + 2 * t;
          int* row8 = s_acc + (r + 8) * kTok + 2 * t;
          atomicAdd(row0, acc[i][0]);
          atomicAdd(row0 + 1, acc[i][1]);
          atomicAdd(row8, acc[i][2]);
          atomicAdd(row8 + 1, acc[i][3]);
          acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0;
        }
      }
    }
    __syncthreads();

    // ---- epilogue: subtract the token sums, rescale, store (rows fastest)
    for (int i = tid; i < mt * R; i += blockDim.x) {
      const int m = i / R, r = i - m * R;
      const int a = s_acc[r * kTok + m] - s_rowsum[m];
      const size_t o = static_cast<size_t>(m0 + m) * N + n0 + r;
      if constexpr (OUT_ACC) {
        static_cast<int32_t*>(out)[o] = a;
      } else {
        static_cast<float*>(out)[o] = rescale(a, gm, s_scale[m]);
      }
    }
    __syncthreads();
  }
  if (!ok) atomicExch(&g_wait_error, 1);
}

size_t decode_smem_bytes(int rows_per_cta, int K) {
  const size_t rp = static_cast<size_t>((rows_per_cta + 15) & ~15);
  const size_t n_tiles = rp / 16;
  size_t b = rp * static_cast<size_t>(K / 4 + 16) + static_cast<size_t>(kTok) * (K + 32);
  b += rp * kTok * 4 + kTok * 4 + kTok * 4 + (kWarps * kTok + 1) * 4;
  b = (b + 7) & ~size_t(7);
  b += n_tiles * 8;
  // more than half an SM's shared memory: one CTA (one row block) per SM
  return b < kOneCtaPerSmSmem ? kOneCtaPerSmSmem : b;
}

template <int XIN, bool OUT_ACC>
cudaError_t launch_decode_t(const uint8_t* wp, const void* x, const float* scale_in, const float* gamma, void* out,
                            int8_t* xq_out, float* scale_out, int M, int N, int K, int rows_per_cta, cudaStream_t s) {
  const size_t smem = decode_smem_bytes(rows_per_cta, K);
  cudaError_t e = ensure_smem(reinterpret_cast<const void*>(bl_decode_mma<XIN, OUT_ACC>), smem);
  if (e != cudaSuccess) return e;
  const int grid = (N + rows_per_cta - 1) / rows_per_cta;
  return launch_pdl(bl_decode_mma<XIN, OUT_ACC>, dim3(grid), dim3(kDecodeThreads), smem, s, wp, x, scale_in, gamma,
                    out, xq_out, scale_out, M, N, K, rows_per_cta);
}

cudaError_t launch_decode(const uint8_t* wp, const void* x, int xin, const float* scale_in, const float* gamma,
                          void* out, bool out_acc, int8_t* xq_out, float* scale_out, int M, int N, int K,
                          int rows_per_cta, cudaStream_t s) {
  if (out_acc) {
    if (xin == kXinF32) return launch_decode_t<kXinF32, true>(wp, x, scale_in, gamma, out, xq_out, scale_out, M, N, K, rows_per_cta, s);
    if (xin == kXinBF16) return launch_decode_t<kXinBF16, true>(wp, x, scale_in, gamma, out, xq_out, scale_out, M, N, K, rows_per_cta, s);
    return launch_decode_t<kXinI8, true>(wp, x, scale_in, gamma, out, xq_out, scale_out, M, N, K, rows_per_cta, s);
  }
  if (xin == kXinF32) return launch_decode_t<kXinF32, false>(wp, x, scale_in, gamma, out, xq_out, scale_out, M, N, K, rows_per_cta, s);
  if (xin == kXinBF16) return launch_decode_t<kXinBF16, false>(wp, x, scale_in, gamma, out, xq_out, scale_out, M, N, K, rows_per_cta, s);
  return launch_decode_t<kXinI8, false>(wp, x, scale_in, gamma, out, xq_out, scale_out, M, N, K, rows_per_cta, s);
}

cudaError_t take_wait_error(int* flag) {
  int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(flag, g_wait_error, sizeof(int));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_wait_error, &zero, sizeof(int));
}

}  // namespace bl
