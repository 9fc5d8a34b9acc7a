// Decode GEMV for one to four tokens in one kernel: per-token activation
// quantisation and the packed-ternary x int8 contraction on dp4a.
//
// Passages: "穿越1比特的奇幻旅程" (2B4T summary), section "GPU端：CUDA内核的定制
// 魔法" (W1.58A8 matmul over four-per-byte packed weights: pack, store, load,
// unpack, compute); "BitNet 1-bit LLM 的混合精度微调技术：渐进量化策略", body,
// quantisation functions (per-token absmax, eps = 1e-5) and the forward-pass
// sentence (multiply back by the factors).
//
// A decode projection streams N*K/4 bytes of packed weights against a few KB
// of activations, so its time is that stream plus the latency around it. The
// kernel starts the stream as early as the launch protocol allows:
//
//   * Before its dependency wait (griddepcontrol.wait), thread 0 of each CTA
//     issues L2 prefetches of the CTA's block of packed rows
//     (cp.async.bulk.prefetch.L2). A prefetch only moves lines into L2, which
//     is the point of coherence, so it cannot change what any later load
//     returns and may run while the previous kernel is still writing. Each
//     CTA leaves room on its SM for a CTA of the next kernel (at most 64
//     registers per thread and under half the shared memory) and releases the
//     next grid right after its own wait, so the next forward's CTAs become
//     resident early and prefetch their weights while this one computes.
//   * After the wait, thread 0 copies the CTA's rows into shared memory with
//     one bulk copy per group of rows (one mbarrier each), while all threads
//     quantise the activations into shared memory: the absmax of each token
//     (warp shuffles, one block barrier), s = 127 / max(absmax, 1e-5), the
//     codes clip(rint(fp32(x * s)), -128, 127), their token sums, and each
//     16-code block transposed as a 4x4 byte matrix (word i holds the codes
//     of k = 16b + 4j + i, j = 0..3).
//   * Warp w takes rows w, w + 16, ..., RB of them at a time; lane l takes the
//     16-code blocks l, l + 32, ... of each row: one 16-byte shared load of the
//     transposed activation block, reused for the RB rows, and one 4-byte
//     shared load of each row's packed word. The four field planes of the
//     word, (word & 0x03030303 << 2i), meet word i of the activation block in
//     one dp4a each:
//        sum_k field * x = acc0 + acc1/4 + acc2/16 + acc3/64   (each exact)
//     and field = code + 1, so sum_k code * x = that - sum_k x.
//   * One redux.sync per (row, token); lane m writes token m's output
//     y = fp32(fp32(acc * gamma) / s), or the int32 accumulator.

#include "async.cuh"
#include "common.cuh"
#include "kernels.cuh"

namespace bl {

namespace {

constexpr int kThreads = kGemvDp4aThreads;
constexpr int kWarps = kThreads / 32;
constexpr uint32_t kGroupBytes = 16384;     // packed bytes per bulk copy and mbarrier (at least one row)
// 16-value blocks per thread kept in registers between the two passes over x
template <int XIN>
constexpr int cache_blocks() { return XIN == kXinF32 ? 1 : 2; }
// Set (never cleared by a kernel) when a bounded mbarrier wait gave up.
__device__ int g_dp4a_wait_error;

// Rows a warp works on at once: 4 accumulators per (row, token) stay in registers.
template <int MT>
constexpr int rows_per_batch() { return MT == 1 ? 6 : (MT == 2 ? 3 : 1); }

// Loads through L2 (not L1), issued after the dependency wait: the data may
// have been written by the grid this one waited for.
BL_DEVICE uint4 ld_cg_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p) : "memory");
  return v;
}
BL_DEVICE float ld_cg_f32(const float* p) {
  float v;
  asm volatile("ld.global.cg.f32 %0, [%1];" : "=f"(v) : "l"(p) : "memory");
  return v;
}

// Shared-memory loads by 32-bit shared address.
BL_DEVICE uint32_t lds_u32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}
BL_DEVICE uint4 lds_v4(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
  return v;
}

// One 16-activation block in its raw form: 2 (bf16) or 4 (fp32) 16-byte words.
template <int XIN>
struct XBlock {
  static constexpr int kVec = XIN == kXinF32 ? 4 : 2;
  uint4 v[kVec];
  BL_DEVICE void load(const void* x, size_t off) {
    const uint4* p = XIN == kXinF32 ? reinterpret_cast<const uint4*>(static_cast<const float*>(x) + off)
                                    : reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(x) + off);
#pragma unroll
    for (int i = 0; i < kVec; ++i) v[i] = ld_cg_v4(p + i);
  }
  BL_DEVICE void widen(float (&f)[16]) const {
#pragma unroll
    for (int i = 0; i < kVec; ++i) {
      const uint32_t u[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if constexpr (XIN == kXinF32) {
          f[4 * i + j] = __uint_as_float(u[j]);
        } else {
          f[8 * i + 2 * j] = __uint_as_float(u[j] << 16);
          f[8 * i + 2 * j + 1] = __uint_as_float(u[j] & 0xffff0000u);
        }
      }
    }
  }
};

// Code of one activation, clip(rint(fp32(x * s)), -128, 127), in the low byte
// (two's complement): after the exact clamp, adding 1.5 * 2^23 rounds to the
// nearest integer, ties to even (the sum lies in [2^23, 2^24), spacing 1), and
// leaves it in the low mantissa bits (0x4B400000 has a zero low byte).
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

// The transposed activation block `blk` (16 codes) of token m sits at byte
// 16 * (m * nblk + blk): lanes reading consecutive blocks read consecutive
// 16-byte words.
BL_DEVICE void store_block(uint8_t* s_act, int m, int blk, int nblk, const uint32_t (&w)[4]) {
  uint4 t;
  transpose4x4_bytes(w[0], w[1], w[2], w[3], t.x, t.y, t.z, t.w);
  *reinterpret_cast<uint4*>(s_act + 16 * (static_cast<size_t>(m) * nblk + blk)) = t;
}

}  // namespace

// Dynamic shared memory (bytes): packed rows [rows_per_cta][K/4] (rounded up
// to 16), transposed activation blocks [MT][K/16][16], warp partials
// float [16][MT] and int [16][MT], then one mbarrier per row group.
template <int XIN, int MT, bool OUT_ACC>
__global__ void __launch_bounds__(kThreads, 2)
bl_gemv_dp4a(const uint8_t* __restrict__ wp, const void* __restrict__ x, const float* __restrict__ scale_in,
             const float* __restrict__ gamma, void* __restrict__ out, int8_t* __restrict__ xq_out,
             float* __restrict__ scale_out, int M, int N, int K, int rows_per_cta) {
  constexpr int RB = rows_per_batch<MT>();
  extern __shared__ __align__(128) uint8_t smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int rowbytes = K >> 2;
  const int nblk = K >> 4;                       // 16-code blocks per token
  const int n0 = blockIdx.x * rows_per_cta;
  const int R = min(rows_per_cta, N - n0);       // at least 1: the grid is ceil(N / rows_per_cta)
  const int rpg = max(1, static_cast<int>(kGroupBytes) / rowbytes);
  const int n_groups = (R + rpg - 1) / rpg;
  uint8_t* s_w = smem;
  uint8_t* s_act = smem + ((static_cast<size_t>(rows_per_cta) * rowbytes + 15) & ~size_t(15));
  float* s_red = reinterpret_cast<float*>(s_act + static_cast<size_t>(MT) * K);
  int* s_sum = reinterpret_cast<int*>(s_red + kWarps * MT);
  uint64_t* s_bar = reinterpret_cast<uint64_t*>(
      (reinterpret_cast<uintptr_t>(s_sum + kWarps * MT) + 7) & ~uintptr_t(7));

  const uint8_t* wblk = wp + static_cast<size_t>(n0) * rowbytes;
  const uint32_t wbytes = static_cast<uint32_t>(R) * static_cast<uint32_t>(rowbytes);   // N*K < 2^32
  if (tid == 0) {
    prefetch_l2_range(wblk, wbytes);
    for (int g = 0; g < n_groups; ++g) mbar_init(&s_bar[g], 1);
    mbar_init_fence();
  } else if (tid == 32) {
    // this CTA's share of the activations (every CTA reads all of x); x may
    // still be being written by the previous grid, which a prefetch cannot
    // disturb
    const uint32_t xbytes = static_cast<uint32_t>(M) * static_cast<uint32_t>(K) *
                            (XIN == kXinF32 ? 4u : (XIN == kXinBF16 ? 2u : 1u));
    const uint32_t share = ((xbytes + gridDim.x - 1) / gridDim.x + 15u) & ~15u;
    const uint32_t lo = blockIdx.x * share;
    if (lo < xbytes) prefetch_l2(static_cast<const uint8_t*>(x) + lo, min(share, xbytes - lo));
  }
  pdl_wait();                                    // everything this grid reads is written and visible
  pdl_launch_dependents();
  wblk = launder(wblk);
  x = launder(x);
  scale_in = launder(scale_in);
  gamma = launder(gamma);
  if (tid == 0) {
    for (int g = 0; g < n_groups; ++g) {
      const int r0 = g * rpg, r1 = min(R, r0 + rpg);
      const uint32_t b = static_cast<uint32_t>(r1 - r0) * static_cast<uint32_t>(rowbytes);
      mbar_expect_tx(&s_bar[g], b);
      bulk_copy_g2s(s_w + static_cast<size_t>(r0) * rowbytes, wblk + static_cast<size_t>(r0) * rowbytes, b,
                    &s_bar[g]);
    }
  }

  // ---- activations: scale, codes, token sums, transposed blocks in shared memory
  float sc[MT];
  int part[MT];
#pragma unroll
  for (int m = 0; m < MT; ++m) {
    sc[m] = 1.f;
    part[m] = 0;
  }
  const int total = M * nblk;
  if constexpr (XIN == kXinI8) {
    for (int q = tid; q < total; q += kThreads) {
      const int m = q / nblk, blk = q - m * nblk;
      const uint4 v = ld_cg_v4(static_cast<const int8_t*>(x) + static_cast<size_t>(m) * K + 16 * blk);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
      const int s16 = sum16(w);
#pragma unroll
      for (int mm = 0; mm < MT; ++mm) part[mm] += mm == m ? s16 : 0;
      store_block(s_act, m, blk, nblk, w);
    }
    if constexpr (!OUT_ACC) {
#pragma unroll
      for (int m = 0; m < MT; ++m) sc[m] = m < M ? ld_cg_f32(scale_in + m) : 1.f;
    }
  } else {
    constexpr int kCacheBlocks = cache_blocks<XIN>();
    XBlock<XIN> cache[kCacheBlocks];
    float amax[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) amax[m] = 0.f;
    auto absmax_of = [&](const XBlock<XIN>& xb, int m) {
      float f[16];
      xb.widen(f);
      float a = 0.f;
#pragma unroll
      for (int j = 0; j < 16; ++j) a = fmaxf(a, fabsf(f[j]));
#pragma unroll
      for (int mm = 0; mm < MT; ++mm) amax[mm] = mm == m ? fmaxf(amax[mm], a) : amax[mm];
    };
#pragma unroll
    for (int u = 0; u < kCacheBlocks; ++u) {
      const int q = tid + kThreads * u;
      if (q < total) {
        const int m = q / nblk;
        cache[u].load(x, static_cast<size_t>(m) * K + 16 * (q - m * nblk));
        absmax_of(cache[u], m);
      }
    }
    for (int q = tid + kThreads * kCacheBlocks; q < total; q += kThreads) {
      const int m = q / nblk;
      XBlock<XIN> xb;
      xb.load(x, static_cast<size_t>(m) * K + 16 * (q - m * nblk));
      absmax_of(xb, m);
    }
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      const float v = warp_max(amax[m]);
      if (lane == 0) s_red[warp * MT + m] = v;
    }
    __syncthreads();
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      float a = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) a = fmaxf(a, s_red[w * MT + m]);
      sc[m] = token_scale(a);
    }
    if (blockIdx.x == 0 && tid < M && scale_out) {
#pragma unroll
      for (int m = 0; m < MT; ++m)
        if (m == tid) scale_out[m] = sc[m];
    }
    auto quantise = [&](const XBlock<XIN>& xb, int q) {
      const int m = q / nblk, blk = q - m * nblk;
      float s = 1.f;
#pragma unroll
      for (int mm = 0; mm < MT; ++mm) s = mm == m ? sc[mm] : s;
      float f[16];
      xb.widen(f);
      uint32_t w[4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
        w[i] = pack4(code_byte(f[4 * i], s), code_byte(f[4 * i + 1], s), code_byte(f[4 * i + 2], s),
                     code_byte(f[4 * i + 3], s));
      if (xq_out && blockIdx.x == 0)
        *reinterpret_cast<uint4*>(xq_out + static_cast<size_t>(m) * K + 16 * blk) = make_uint4(w[0], w[1], w[2], w[3]);
      const int s16 = sum16(w);
#pragma unroll
      for (int mm = 0; mm < MT; ++mm) part[mm] += mm == m ? s16 : 0;
      store_block(s_act, m, blk, nblk, w);
    };
#pragma unroll
    for (int u = 0; u < kCacheBlocks; ++u) {
      const int q = tid + kThreads * u;
      if (q < total) quantise(cache[u], q);
    }
    for (int q = tid + kThreads * kCacheBlocks; q < total; q += kThreads) {
      const int m = q / nblk;
      XBlock<XIN> xb;
      xb.load(x, static_cast<size_t>(m) * K + 16 * (q - m * nblk));
      quantise(xb, q);
    }
  }
#pragma unroll
  for (int m = 0; m < MT; ++m) {
    const int v = warp_sum(part[m]);
    if (lane == 0) s_sum[warp * MT + m] = v;
  }
  __syncthreads();                               // codes, token sums and mbarrier set-up complete

  int rsum[MT];
  float rc[MT];
#pragma unroll
  for (int m = 0; m < MT; ++m) {
    int t = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) t += s_sum[w * MT + m];
    rsum[m] = t;
    rc[m] = OUT_ACC ? 0.f : recip_for_div(sc[m]);
  }
  const float gm = OUT_ACC ? 0.f : ld_cg_f32(gamma);

  // ---- contraction: warp w takes rows w, w + 16, ..., RB at a time; lane l
  // the 16-code blocks l, l + 32, ... of each row (one packed word each)
  bool ok = true;
  const int nrw = warp < R ? (R - warp + kWarps - 1) / kWarps : 0;
  const uint32_t s_w32 = smem_u32(s_w), s_act32 = smem_u32(s_act);
  for (int t0 = 0; t0 < nrw; t0 += RB) {
    int acc[RB][MT][4];
#pragma unroll
    for (int i = 0; i < RB; ++i) {
#pragma unroll
      for (int m = 0; m < MT; ++m) acc[i][m][0] = acc[i][m][1] = acc[i][m][2] = acc[i][m][3] = 0;
      if (t0 + i < nrw) ok = mbar_wait_sleep(&s_bar[(warp + kWarps * (t0 + i)) / rpg], 0u) && ok;
    }
    // shared address of word `lane` of the batch's first row; row i is i * rstride further
    const uint32_t rstride = static_cast<uint32_t>(kWarps) * static_cast<uint32_t>(rowbytes);
    uint32_t wa = s_w32 + static_cast<uint32_t>(warp + kWarps * t0) * static_cast<uint32_t>(rowbytes) + 4u * lane;
    for (int b = lane; b < nblk; b += 32, wa += 128u) {
      uint32_t wv[RB];
#pragma unroll
      for (int i = 0; i < RB; ++i) wv[i] = t0 + i < nrw ? lds_u32(wa + i * rstride) : 0u;
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        if (m < M) {
          const uint4 a = lds_v4(s_act32 + 16u * static_cast<uint32_t>(m * nblk + b));
#pragma unroll
          for (int i = 0; i < RB; ++i) {
            if (t0 + i < nrw) {                  // warp-uniform
              const uint32_t w = wv[i];
              acc[i][m][0] = dp4a_us(w & 0x03030303u, static_cast<int>(a.x), acc[i][m][0]);
              acc[i][m][1] = dp4a_us(w & 0x0c0c0c0cu, static_cast<int>(a.y), acc[i][m][1]);
              acc[i][m][2] = dp4a_us(w & 0x30303030u, static_cast<int>(a.z), acc[i][m][2]);
              acc[i][m][3] = dp4a_us(w & 0xc0c0c0c0u, static_cast<int>(a.w), acc[i][m][3]);
            }
          }
        }
      }
    }
#pragma unroll
    for (int i = 0; i < RB; ++i) {
      if (t0 + i < nrw) {                        // warp-uniform
        const int r = warp + kWarps * (t0 + i);
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          if (m < M) {
            const int v = __reduce_add_sync(0xffffffffu, acc[i][m][0] + (acc[i][m][1] >> 2) +
                                                             (acc[i][m][2] >> 4) + (acc[i][m][3] >> 6));
            if (lane == m) {
              const size_t o = static_cast<size_t>(m) * N + n0 + r;
              if constexpr (OUT_ACC) {
                static_cast<int32_t*>(out)[o] = v - rsum[m];
              } else {
                static_cast<float*>(out)[o] =
                    div_rn_recip(__fmul_rn(static_cast<float>(v - rsum[m]), gm), sc[m], rc[m]);
              }
            }
          }
        }
      }
    }
  }
  // every bulk copy has landed before the CTA exits (warps without rows did not wait)
  if (tid == 0)
    for (int g = 0; g < n_groups; ++g) ok = mbar_wait_sleep(&s_bar[g], 0u) && ok;
  if (!ok) atomicExch(&g_dp4a_wait_error, 1);
}

namespace {

size_t align16(size_t v) { return (v + 15) & ~size_t(15); }

size_t dp4a_smem(int rows, int K, int mt) {
  const size_t rowbytes = static_cast<size_t>(K) / 4;
  const int rpg = rowbytes >= kGroupBytes ? 1 : static_cast<int>(kGroupBytes / rowbytes);
  const size_t groups = (static_cast<size_t>(rows) + rpg - 1) / rpg;
  return align16(static_cast<size_t>(rows) * rowbytes) + static_cast<size_t>(mt) * K +
         static_cast<size_t>(kWarps) * mt * 8 + 8 + 8 * groups;
}

template <int XIN, int MT, bool OUT_ACC>
cudaError_t launch_t(const uint8_t* wp, const void* x, const float* scale_in, const float* gamma, void* out,
                     int8_t* xq_out, float* scale_out, int M, int N, int K, int rows, size_t smem, cudaStream_t s) {
  auto kern = bl_gemv_dp4a<XIN, MT, OUT_ACC>;
  const cudaError_t e = ensure_smem(reinterpret_cast<const void*>(kern), smem);
  if (e != cudaSuccess) return e;
  const int grid = (N + rows - 1) / rows;
  return launch_pdl(kern, dim3(grid), dim3(kThreads), smem, s, wp, x, scale_in, gamma, out, xq_out, scale_out, M, N,
                    K, rows);
}

template <int MT>
cudaError_t launch_mt(const uint8_t* wp, const void* x, int xin, const float* scale_in, const float* gamma, void* out,
                      bool out_acc, int8_t* xq_out, float* scale_out, int M, int N, int K, int rows, size_t smem,
                      cudaStream_t s) {
  if (xin == kXinF32)
    return launch_t<kXinF32, MT, false>(wp, x, nullptr, gamma, out, xq_out, scale_out, M, N, K, rows, smem, s);
  if (xin == kXinBF16)
    return launch_t<kXinBF16, MT, false>(wp, x, nullptr, gamma, out, xq_out, scale_out, M, N, K, rows, smem, s);
  if (out_acc)
    return launch_t<kXinI8, MT, true>(wp, x, nullptr, nullptr, out, nullptr, nullptr, M, N, K, rows, smem, s);
  return launch_t<kXinI8, MT, false>(wp, x, scale_in, gamma, out, nullptr, nullptr, M, N, K, rows, smem, s);
}

}  // namespace

size_t gemv_dp4a_plan(int M, int N, int K, int sms, int* rows_per_cta) {
  if (M < 1 || M > kGemvDp4aMaxM || N < 1 || K < 64 || K % 64 != 0 || sms < 1) return 0;
  const int mt = M == 1 ? 1 : (M == 2 ? 2 : 4);
  if (static_cast<size_t>(mt) * K > kGemvDp4aMaxAct) return 0;
  int rows = (N + sms - 1) / sms;
  while (rows > 1 && dp4a_smem(rows, K, mt) > kGemvDp4aMaxSmem) rows = (rows + 1) / 2;
  const size_t smem = dp4a_smem(rows, K, mt);
  if (smem > kGemvDp4aMaxSmem) return 0;
  *rows_per_cta = rows;
  return smem;
}

cudaError_t launch_gemv_dp4a(const uint8_t* wp, const void* x, int xin, const float* scale_in, const float* gamma,
                             void* out, bool out_acc, int8_t* xq_out, float* scale_out, int M, int N, int K,
                             int rows_per_cta, size_t smem, cudaStream_t s) {
  if (M <= 1)
    return launch_mt<1>(wp, x, xin, scale_in, gamma, out, out_acc, xq_out, scale_out, M, N, K, rows_per_cta, smem, s);
  if (M <= 2)
    return launch_mt<2>(wp, x, xin, scale_in, gamma, out, out_acc, xq_out, scale_out, M, N, K, rows_per_cta, smem, s);
  return launch_mt<4>(wp, x, xin, scale_in, gamma, out, out_acc, xq_out, scale_out, M, N, K, rows_per_cta, smem, s);
}

cudaError_t take_dp4a_wait_error(int* flag) {
  int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(flag, g_dp4a_wait_error, sizeof(int));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_dp4a_wait_error, &zero, sizeof(int));
}

}  // namespace bl
