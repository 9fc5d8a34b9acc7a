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
// kernel starts the stream as early as the launch protocol allows and keeps
// every warp's instruction chains short:
//
//   * Before its dependency wait (griddepcontrol.wait), each CTA issues L2
//     prefetches of its block of packed rows and of its share of x
//     (cp.async.bulk.prefetch.L2). A prefetch only moves lines into L2, which
//     is the point of coherence, so it cannot change what any later load
//     returns and may run while the previous kernel is still writing. Each
//     CTA leaves room on its SM for a CTA of the next kernel (at most 64
//     registers per thread and under half the shared memory) and releases the
//     next grid right after its own wait, so the next forward's CTAs become
//     resident early and prefetch their weights while this one computes.
//   * After the wait, thread 0 copies the CTA's rows into shared memory with
//     one bulk copy per group of rows (one mbarrier each), while all threads
//     quantise the activations, one 4-code word per thread at a time: the
//     absmax of each token (warp shuffles, one block barrier), s = 127 /
//     max(absmax, 1e-5), the codes rint(fp32(x * s)) (within +-127, so the
//     clip never acts), their token sums, and each code stored as one byte of
//     the 16-code block transposed as a 4x4 byte matrix (word i of block b
//     holds the codes of k = 16b + 4j + i, j = 0..3).
//   * The contraction is cut into equal shares per warp: rows are taken RB at
//     a time, and the (row batch, 16-code block) pairs of the CTA are split
//     into 16 contiguous ranges. Over its range a lane takes blocks l, l + 32,
//     ...: one 16-byte shared load of the transposed activation block, reused
//     for the RB rows, and one 4-byte shared load of each row's packed word.
//     The four field planes of the word, (word & 0x03030303 << 2i), meet word
//     i of the activation block in one dp4a each:
//        sum_k field * x = acc0 + acc1/4 + acc2/16 + acc3/64   (each exact)
//     and field = code + 1, so sum_k code * x = that - sum_k x.
//   * Partial sums of a row (a range may cover part of a row) meet in shared
//     memory through integer atomics, so their order does not matter; after a
//     block barrier the threads write y = fp32(fp32(acc * gamma) / s) (or the
//     int32 accumulator), coalesced along the rows.

#include "async.cuh"
#include "common.cuh"
#include "kernels.cuh"

namespace bl {

namespace {

constexpr int kThreads = kGemvDp4aThreads;
constexpr int kWarps = kThreads / 32;
constexpr uint32_t kGroupBytes = 16384;     // packed bytes per bulk copy and mbarrier (at least one row)
constexpr int kCacheWords = 4;              // 4-value words per thread kept in registers between the two passes
// Set (never cleared by a kernel) when a bounded mbarrier wait gave up.
__device__ int g_dp4a_wait_error;

// Rows a warp works on at once: 4 accumulators per (row, token) stay in registers.
template <int MT>
constexpr int rows_per_batch() { return MT == 1 ? 4 : (MT == 2 ? 2 : 1); }

// Loads through L2 (not L1), issued after the dependency wait: the data may
// have been written by the grid this one waited for.
BL_DEVICE uint4 ld_cg_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p) : "memory");
  return v;
}
BL_DEVICE uint2 ld_cg_v2(const void* p) {
  uint2 v;
  asm volatile("ld.global.cg.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p) : "memory");
  return v;
}
BL_DEVICE uint32_t ld_cg_u32(const void* p) {
  uint32_t v;
  asm volatile("ld.global.cg.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
BL_DEVICE float ld_cg_f32(const float* p) {
  float v;
  asm volatile("ld.global.cg.f32 %0, [%1];" : "=f"(v) : "l"(p) : "memory");
  return v;
}

// Shared-memory access by 32-bit shared address.
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
BL_DEVICE void sts_u8(uint32_t a, uint32_t v) { asm volatile("st.shared.u8 [%0], %1;" ::"r"(a), "r"(v)); }

// One 4-activation word in its raw form: 8 bytes (bf16), 16 bytes (fp32) or
// 4 bytes (int8 codes), widened exactly to fp32 for the float kinds.
template <int XIN> struct XWord;
template <> struct XWord<kXinBF16> {
  uint2 v;
  BL_DEVICE void load(const void* x, size_t word) { v = ld_cg_v2(static_cast<const uint16_t*>(x) + 4 * word); }
  BL_DEVICE void widen(float (&f)[4]) const {
    f[0] = __uint_as_float(v.x << 16);
    f[1] = __uint_as_float(v.x & 0xffff0000u);
    f[2] = __uint_as_float(v.y << 16);
    f[3] = __uint_as_float(v.y & 0xffff0000u);
  }
};
template <> struct XWord<kXinF32> {
  uint4 v;
  BL_DEVICE void load(const void* x, size_t word) { v = ld_cg_v4(static_cast<const float*>(x) + 4 * word); }
  BL_DEVICE void widen(float (&f)[4]) const {
    f[0] = __uint_as_float(v.x);
    f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z);
    f[3] = __uint_as_float(v.w);
  }
};

// Code of one activation, rint(fp32(x * s)), in the low byte (two's
// complement). |x| <= absmax makes |x * s| at most 127 (1 + 2^-23), so the
// clip to [-128, 127] never acts and the sum with 1.5 * 2^23 (which lies in
// [2^23, 2^24), spacing 1) rounds to the nearest integer, ties to even, and
// leaves it in the low mantissa bits (0x4B400000 has a zero low byte).
BL_DEVICE uint32_t code_byte(float x, float s) { return __float_as_uint(__fadd_rn(__fmul_rn(x, s), 12582912.f)); }

BL_DEVICE uint32_t pack4(uint32_t b0, uint32_t b1, uint32_t b2, uint32_t b3) {
  return __byte_perm(__byte_perm(b0, b1, 0x0040), __byte_perm(b2, b3, 0x0040), 0x5410);
}

// Places the four codes of word j of token m (k = 4j .. 4j + 3) into the
// transposed block layout: the code of k = 16b + 4jj + i is byte jj of word i
// of block b, at byte 16 (m nblk + b) + 4 i + jj of the activation area.
BL_DEVICE void store_word(uint32_t s_act32, int m, int j, int nblk, uint32_t w) {
  const uint32_t base = s_act32 + 16u * static_cast<uint32_t>(m * nblk + (j >> 2)) + static_cast<uint32_t>(j & 3);
  sts_u8(base, w & 0xffu);
  sts_u8(base + 4u, (w >> 8) & 0xffu);
  sts_u8(base + 8u, (w >> 16) & 0xffu);
  sts_u8(base + 12u, w >> 24);
}

}  // namespace

// Dynamic shared memory (bytes): packed rows [rows_per_cta][K/4] (rounded up
// to 16), transposed activation blocks [MT][K/16][16], warp partials
// float [16][MT] and int [16][MT], row accumulators int [rows, rounded up to
// RB][MT], then one mbarrier per row group.
template <int XIN, int MT, bool OUT_ACC>
__global__ void __launch_bounds__(kThreads, 2)
bl_gemv_dp4a(const uint8_t* __restrict__ wp, const void* __restrict__ x, const float* __restrict__ scale_in,
             const float* __restrict__ gamma, void* __restrict__ out, int8_t* __restrict__ xq_out,
             float* __restrict__ scale_out, int M, int N, int K, int rows_per_cta) {
  constexpr int RB = rows_per_batch<MT>();
  extern __shared__ __align__(128) uint8_t smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int rowbytes = K >> 2;
  const int nblk = K >> 4;                       // 16-code blocks per token (packed words per row)
  const int nw = K >> 2;                         // 4-value activation words per token
  const int n0 = blockIdx.x * rows_per_cta;
  const int R = min(rows_per_cta, N - n0);       // at least 1: the grid is ceil(N / rows_per_cta)
  const int n_batches = (R + RB - 1) / RB;
  const int rows_pad = (rows_per_cta + RB - 1) / RB * RB;
  const int rpg = max(1, static_cast<int>(kGroupBytes) / rowbytes);
  const int n_groups = (R + rpg - 1) / rpg;
  uint8_t* s_w = smem;
  uint8_t* s_act = smem + ((static_cast<size_t>(rows_per_cta) * rowbytes + 15) & ~size_t(15));
  float* s_red = reinterpret_cast<float*>(s_act + static_cast<size_t>(MT) * K);
  int* s_sum = reinterpret_cast<int*>(s_red + kWarps * MT);
  int* s_acc = s_sum + kWarps * MT;
  uint64_t* s_bar = reinterpret_cast<uint64_t*>((reinterpret_cast<uintptr_t>(s_acc + rows_pad * MT) + 7) & ~uintptr_t(7));

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
  for (int i = tid; i < rows_pad * MT; i += kThreads) s_acc[i] = 0;
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

  // gamma now: its load latency hides under the activation pass
  const float gm = OUT_ACC ? 0.f : ld_cg_f32(gamma);

  // ---- activations: scale, codes, token sums, transposed blocks in shared memory
  const uint32_t s_act32 = smem_u32(s_act);
  const int total = M * nw;                      // words over all tokens
  float sc[MT], rc[MT];                          // scales and recip_for_div of them
  int part[MT];
#pragma unroll
  for (int m = 0; m < MT; ++m) {
    sc[m] = 1.f;
    rc[m] = 0.f;
    part[m] = 0;
  }
  // token and word index of flat word q
  auto split = [&](int q, int& m, int& j) {
    if constexpr (MT == 1) {
      m = 0;
      j = q;
    } else {
      m = q / nw;
      j = q - m * nw;
    }
  };
  if constexpr (XIN == kXinI8) {
    for (int q = tid; q < total; q += kThreads) {
      int m, j;
      split(q, m, j);
      const uint32_t w = ld_cg_u32(static_cast<const int8_t*>(x) + static_cast<size_t>(m) * K + 4 * j);
      const int s4 = dp4a_ss(static_cast<int>(w), 0x01010101, 0);
#pragma unroll
      for (int mm = 0; mm < MT; ++mm) part[mm] += mm == m ? s4 : 0;
      store_word(s_act32, m, j, nblk, w);
    }
    if constexpr (!OUT_ACC) {
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        sc[m] = m < M ? ld_cg_f32(scale_in + m) : 1.f;
        rc[m] = recip_for_div(sc[m]);
      }
    }
  } else {
    XWord<XIN> cache[kCacheWords];
    float amax[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) amax[m] = 0.f;
    auto absmax_of = [&](const XWord<XIN>& xw, int m) {
      float f[4];
      xw.widen(f);
      const float a = fmaxf(fmaxf(fabsf(f[0]), fabsf(f[1])), fmaxf(fabsf(f[2]), fabsf(f[3])));
#pragma unroll
      for (int mm = 0; mm < MT; ++mm) amax[mm] = mm == m ? fmaxf(amax[mm], a) : amax[mm];
    };
#pragma unroll
    for (int u = 0; u < kCacheWords; ++u) {
      const int q = tid + kThreads * u;
      if (q < total) {
        int m, j;
        split(q, m, j);
        cache[u].load(x, static_cast<size_t>(m) * nw + j);
      }
    }
#pragma unroll
    for (int u = 0; u < kCacheWords; ++u) {
      const int q = tid + kThreads * u;
      if (q < total) {
        int m, j;
        split(q, m, j);
        absmax_of(cache[u], m);
      }
    }
    for (int q = tid + kThreads * kCacheWords; q < total; q += kThreads) {
      int m, j;
      split(q, m, j);
      XWord<XIN> xw;
      xw.load(x, static_cast<size_t>(m) * nw + j);
      absmax_of(xw, m);
    }
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      const float v = warp_max(amax[m]);
      if (lane == 0) s_red[warp * MT + m] = v;
    }
    __syncthreads();
    // each warp reduces the per-warp maxima itself: one load per lane, then shuffles
#pragma unroll
    for (int m = 0; m < MT; ++m) sc[m] = token_scale(warp_max(lane < kWarps ? s_red[lane * MT + m] : 0.f));
    // the reciprocals of the rescale, off the critical path of the output
#pragma unroll
    for (int m = 0; m < MT; ++m) rc[m] = recip_for_div(sc[m]);
    if (blockIdx.x == 0 && tid < M && scale_out) {
#pragma unroll
      for (int m = 0; m < MT; ++m)
        if (m == tid) scale_out[m] = sc[m];
    }
    auto quantise = [&](const XWord<XIN>& xw, int q) {
      int m, j;
      split(q, m, j);
      float s = 1.f;
#pragma unroll
      for (int mm = 0; mm < MT; ++mm) s = mm == m ? sc[mm] : s;
      float f[4];
      xw.widen(f);
      const uint32_t w = pack4(code_byte(f[0], s), code_byte(f[1], s), code_byte(f[2], s), code_byte(f[3], s));
      if (xq_out && blockIdx.x == 0) *reinterpret_cast<uint32_t*>(xq_out + static_cast<size_t>(m) * K + 4 * j) = w;
      const int s4 = dp4a_ss(static_cast<int>(w), 0x01010101, 0);
#pragma unroll
      for (int mm = 0; mm < MT; ++mm) part[mm] += mm == m ? s4 : 0;
      store_word(s_act32, m, j, nblk, w);
    };
#pragma unroll
    for (int u = 0; u < kCacheWords; ++u) {
      const int q = tid + kThreads * u;
      if (q < total) quantise(cache[u], q);
    }
    for (int q = tid + kThreads * kCacheWords; q < total; q += kThreads) {
      int m, j;
      split(q, m, j);
      XWord<XIN> xw;
      xw.load(x, static_cast<size_t>(m) * nw + j);
      quantise(xw, q);
    }
  }
#pragma unroll
  for (int m = 0; m < MT; ++m) {
    const int v = warp_sum(part[m]);
    if (lane == 0) s_sum[warp * MT + m] = v;
  }
  __syncthreads();                               // codes, token sums, zeroed accumulators and mbarriers ready

  // ---- contraction: the (row batch, block) pairs split into equal ranges per warp
  bool ok = true;
  const uint32_t s_w32 = smem_u32(s_w);
  const int work = n_batches * nblk;
  int f = static_cast<int>(static_cast<long long>(work) * warp / kWarps);
  const int f_end = static_cast<int>(static_cast<long long>(work) * (warp + 1) / kWarps);
  while (f < f_end) {
    const int bt = f / nblk, b0 = f - bt * nblk;
    const int b1 = min(nblk, b0 + (f_end - f));
    const int r0 = bt * RB;
    const int r_last = min(r0 + RB, R) - 1;
    for (int g = r0 / rpg; g <= r_last / rpg; ++g) ok = mbar_wait_sleep(&s_bar[g], 0u) && ok;
    uint32_t ra[RB];                             // shared address of word `lane` of each row of the batch
    bool rv[RB];
#pragma unroll
    for (int i = 0; i < RB; ++i) {
      rv[i] = r0 + i < R;
      ra[i] = s_w32 + static_cast<uint32_t>(min(r0 + i, R - 1)) * static_cast<uint32_t>(rowbytes) + 4u * lane;
    }
    int acc[RB][MT][4];
#pragma unroll
    for (int i = 0; i < RB; ++i)
#pragma unroll
      for (int m = 0; m < MT; ++m) acc[i][m][0] = acc[i][m][1] = acc[i][m][2] = acc[i][m][3] = 0;
    // two blocks per iteration (b and b + 32) for independent loads; a block
    // past the range reads block b again with its weights taken as zero
    for (int b = b0 + lane; b < b1; b += 64) {
      const bool two = b + 32 < b1;
      const int b2 = two ? b + 32 : b;
      const uint32_t off = 4u * static_cast<uint32_t>(b - lane);
      const uint32_t off2 = 4u * static_cast<uint32_t>(b2 - lane);
      uint32_t wv[RB], wv2[RB];
#pragma unroll
      for (int i = 0; i < RB; ++i) {
        const uint32_t w = lds_u32(ra[i] + off);
        const uint32_t w2 = lds_u32(ra[i] + off2);
        wv[i] = rv[i] ? w : 0u;
        wv2[i] = rv[i] && two ? w2 : 0u;
      }
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        if (m < M) {
          const uint4 a = lds_v4(s_act32 + 16u * static_cast<uint32_t>(m * nblk + b));
          const uint4 a2 = lds_v4(s_act32 + 16u * static_cast<uint32_t>(m * nblk + b2));
#pragma unroll
          for (int i = 0; i < RB; ++i) {
            acc[i][m][0] = dp4a_us(wv[i] & 0x03030303u, static_cast<int>(a.x), acc[i][m][0]);
            acc[i][m][1] = dp4a_us(wv[i] & 0x0c0c0c0cu, static_cast<int>(a.y), acc[i][m][1]);
            acc[i][m][2] = dp4a_us(wv[i] & 0x30303030u, static_cast<int>(a.z), acc[i][m][2]);
            acc[i][m][3] = dp4a_us(wv[i] & 0xc0c0c0c0u, static_cast<int>(a.w), acc[i][m][3]);
            acc[i][m][0] = dp4a_us(wv2[i] & 0x03030303u, static_cast<int>(a2.x), acc[i][m][0]);
            acc[i][m][1] = dp4a_us(wv2[i] & 0x0c0c0c0cu, static_cast<int>(a2.y), acc[i][m][1]);
            acc[i][m][2] = dp4a_us(wv2[i] & 0x30303030u, static_cast<int>(a2.z), acc[i][m][2]);
            acc[i][m][3] = dp4a_us(wv2[i] & 0xc0c0c0c0u, static_cast<int>(a2.w), acc[i][m][3]);
          }
        }
      }
    }
#pragma unroll
    for (int i = 0; i < RB; ++i) {
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        const int v = __reduce_add_sync(0xffffffffu, acc[i][m][0] + (acc[i][m][1] >> 2) + (acc[i][m][2] >> 4) +
                                                         (acc[i][m][3] >> 6));
        if (lane == 0 && rv[i] && m < M) atomicAdd(&s_acc[(r0 + i) * MT + m], v);
      }
    }
    f += b1 - b0;
  }
  __syncthreads();                               // every partial sum is in s_acc

  // ---- outputs, coalesced along the rows
#pragma unroll
  for (int m = 0; m < MT; ++m) {
    if (m < M) {
      const int rs = __reduce_add_sync(0xffffffffu, lane < kWarps ? s_sum[lane * MT + m] : 0);
      for (int r = tid; r < R; r += kThreads) {
        const int a = s_acc[r * MT + m] - rs;
        const size_t o = static_cast<size_t>(m) * N + n0 + r;
        if constexpr (OUT_ACC) {
          static_cast<int32_t*>(out)[o] = a;
        } else {
          static_cast<float*>(out)[o] = div_rn_recip(__fmul_rn(static_cast<float>(a), gm), sc[m], rc[m]);
        }
      }
    }
  }
  // every bulk copy has landed before the CTA exits (a warp whose wait gave up
  // left its copy in flight)
  if (tid == 0)
    for (int g = 0; g < n_groups; ++g) ok = mbar_wait_sleep(&s_bar[g], 0u) && ok;
  if (!ok) atomicExch(&g_dp4a_wait_error, 1);
}

namespace {

size_t align16(size_t v) { return (v + 15) & ~size_t(15); }

size_t dp4a_smem(int rows, int K, int mt) {
  const int rb = mt == 1 ? 4 : (mt == 2 ? 2 : 1);   // rows_per_batch
  const size_t rowbytes = static_cast<size_t>(K) / 4;
  const int rpg = rowbytes >= kGroupBytes ? 1 : static_cast<int>(kGroupBytes / rowbytes);
  const size_t groups = (static_cast<size_t>(rows) + rpg - 1) / rpg;
  const size_t rows_pad = (static_cast<size_t>(rows) + rb - 1) / rb * rb;
  return align16(static_cast<size_t>(rows) * rowbytes) + static_cast<size_t>(mt) * K +
         static_cast<size_t>(kWarps) * mt * 8 + rows_pad * mt * 4 + 8 + 8 * groups;
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
