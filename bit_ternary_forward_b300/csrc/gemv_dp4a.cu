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
// of activations. The weight stream overlaps the previous kernel (below), so
// what is left after the dependency wait is a chain of short phases, and the
// kernel keeps each one to few instructions with no per-element control flow:
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
//   * After the wait every thread loads its 16-value blocks of x (16-byte
//     loads); then one thread copies the CTA's rows into shared memory, one
//     bulk copy per group of row batches (one mbarrier each).
//   * Activations, per 16-value block: the absmax in integer form (the
//     magnitude bits of finite floats order like the values, so the max of
//     |x| is an unsigned max of bits with the sign cleared: three-way 16x2 and
//     32-bit max instructions, then a warp max reduction and one block
//     barrier), s = 127 / max(absmax, 1e-5), the codes rint(fp32(x * s))
//     (a rounded multiply, then a rounded add that leaves the nearest integer
//     in the low byte), their token sum (dp4a with ones), and the block stored as
//     one 16-byte word in the transposed layout the contraction reads: word i
//     holds the codes of k = 16b + 4j + i, j = 0..3, as its bytes j.
//     |x| <= absmax keeps |x * s| <= 127 (1 + 2^-23), so the clip never acts.
//   * Contraction: rows are taken RB at a time and each row's 16-code blocks
//     in chunks of 32, one block per lane; a unit is (row batch, chunk) and
//     each warp owns an equal contiguous range of units, in row-batch-major
//     order, so its accumulators carry over chunks and are reduced only when
//     the batch changes. Per unit a lane loads one 4-byte packed word per row
//     and one 16-byte activation word per token, and the four field planes of
//     each packed word, (word & 0x03030303 << 2i), meet word i of the
//     activation block in one dp4a each:
//        sum_k field * x = acc0 + acc1/4 + acc2/16 + acc3/64   (each exact)
//     and field = code + 1, so sum_k code * x = that - sum_k x. The activation
//     area of each token is zero-padded to whole chunks, so the lanes past
//     the end of a row contribute nothing whatever bytes they read.
//   * Partial sums of a row meet in shared memory through integer atomics
//     (their order does not matter); after a block barrier the threads write
//     y = fp32(fp32(acc * gamma) / s) (or the int32 accumulator), coalesced
//     along the rows.

#include "async.cuh"
#include "common.cuh"
#include "kernels.cuh"

namespace bl {

namespace {

constexpr int kThreads = kGemvDp4aThreads;
constexpr int kWarps = kThreads / 32;
constexpr int kChunk = 32;                  // 16-code blocks per contraction unit: one per lane
constexpr uint32_t kGroupBytes = 16384;     // packed bytes per bulk copy and mbarrier (at least one row batch)
constexpr int kCopyThread = kThreads - 32;  // issues the weight copies (lane 0 of the last warp)
// Set (never cleared by a kernel) when a bounded mbarrier wait gave up.
__device__ int g_dp4a_wait_error;

// Rows a warp works on at once (4 accumulators per (row, token) in registers;
// two rows keep the units small, so the warps' shares balance).
template <int MT>
constexpr int rows_per_batch() { return MT == 4 ? 1 : 2; }

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
BL_DEVICE void sts_v4(uint32_t a, uint32_t x, uint32_t y, uint32_t z, uint32_t w) {
  asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(a), "r"(x), "r"(y), "r"(z), "r"(w));
}

// Code of one activation, rint(fp32(x * s)), in the low byte (two's
// complement): RN(RN(x * s) + 1.5 * 2^23) leaves it there (ties to even),
// because RN(x * s) lies within +-127 (1 + 2^-23) and 1.5 * 2^23 + [-128, 128]
// stays in [2^23, 2^24), where the spacing is 1; 0x4B400000 has a zero low
// byte. Two separately rounded operations: a fused multiply-add would round
// only once and differ at products just below a half.
BL_DEVICE uint32_t code_byte(uint32_t xbits, float s) {
  return __float_as_uint(__fadd_rn(__fmul_rn(__uint_as_float(xbits), s), 12582912.f));
}

// Low bytes of four registers as one word (byte j from register j).
BL_DEVICE uint32_t pack4(uint32_t b0, uint32_t b1, uint32_t b2, uint32_t b3) {
  return __byte_perm(__byte_perm(b0, b1, 0x0040), __byte_perm(b2, b3, 0x0040), 0x5410);
}

// One 16-value block of activations in its raw form: bf16 (two 16-byte
// words), fp32 (four) or int8 codes (one).
template <int XIN> struct XBlock;
template <> struct XBlock<kXinBF16> {
  uint4 v[2];
  BL_DEVICE void load(const void* x, size_t blk) {
    const uint16_t* p = static_cast<const uint16_t*>(x) + 16 * blk;
    v[0] = ld_cg_v4(p);
    v[1] = ld_cg_v4(p + 8);
  }
  BL_DEVICE void zero() { v[0] = v[1] = make_uint4(0u, 0u, 0u, 0u); }
  // max of the magnitude bits, as two 16-bit lanes
  BL_DEVICE uint32_t mag_max(uint32_t run) const {
    constexpr uint32_t m = 0x7fff7fffu;
    const uint32_t a = __vimax3_u16x2(v[0].x & m, v[0].y & m, v[0].z & m);
    const uint32_t b = __vimax3_u16x2(v[0].w & m, v[1].x & m, v[1].y & m);
    const uint32_t c = __vimax3_u16x2(v[1].z & m, v[1].w & m, a);
    return __vimax3_u16x2(b, c, run);
  }
  // the largest magnitude of the two lanes (taken before any reduction across
  // threads, which compares whole words) and its value
  static BL_DEVICE uint32_t mag_scalar(uint32_t run) { return max(run & 0xffffu, run >> 16); }
  static BL_DEVICE float mag_to_float(uint32_t mag) { return __uint_as_float(mag << 16); }
  // codes of the 16 values, value j in the low byte of c[j]
  BL_DEVICE void codes(float s, uint32_t (&c)[16]) const {
    const uint32_t w[8] = {v[0].x, v[0].y, v[0].z, v[0].w, v[1].x, v[1].y, v[1].z, v[1].w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      c[2 * i] = code_byte(w[i] << 16, s);
      c[2 * i + 1] = code_byte(w[i] & 0xffff0000u, s);
    }
  }
};
template <> struct XBlock<kXinF32> {
  uint4 v[4];
  BL_DEVICE void load(const void* x, size_t blk) {
    const float* p = static_cast<const float*>(x) + 16 * blk;
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = ld_cg_v4(p + 4 * i);
  }
  BL_DEVICE void zero() {
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = make_uint4(0u, 0u, 0u, 0u);
  }
  BL_DEVICE uint32_t mag_max(uint32_t run) const {
    constexpr uint32_t m = 0x7fffffffu;
    uint32_t r[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) r[i] = __vimax3_u32(v[i].x & m, v[i].y & m, max(v[i].z & m, v[i].w & m));
    return __vimax3_u32(__vimax3_u32(r[0], r[1], r[2]), r[3], run);
  }
  static BL_DEVICE uint32_t mag_scalar(uint32_t run) { return run; }
  static BL_DEVICE float mag_to_float(uint32_t mag) { return __uint_as_float(mag); }
  BL_DEVICE void codes(float s, uint32_t (&c)[16]) const {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      c[4 * i] = code_byte(v[i].x, s);
      c[4 * i + 1] = code_byte(v[i].y, s);
      c[4 * i + 2] = code_byte(v[i].z, s);
      c[4 * i + 3] = code_byte(v[i].w, s);
    }
  }
};

}  // namespace

// Dynamic shared memory (bytes): packed rows [rows_per_cta][K/4] (rounded up
// to 16), transposed activation blocks [MT][nchunk * 32][16] (zero past K),
// warp maxima [16][MT], warp token sums [16][MT], row accumulators
// [rows rounded up to RB][MT], then one mbarrier per row group.
template <int XIN, int MT, bool OUT_ACC>
__global__ void __launch_bounds__(kThreads, 2)
bl_gemv_dp4a(const uint8_t* __restrict__ wp, const void* __restrict__ x, const float* __restrict__ scale_in,
             const float* __restrict__ gamma, void* __restrict__ out, int8_t* __restrict__ xq_out,
             float* __restrict__ scale_out, int M, int N, int K, int rows_per_cta) {
  constexpr int RB = rows_per_batch<MT>();
  constexpr int CB = XIN == kXinBF16 ? 2 : 1;   // blocks per thread kept in registers between the two passes
  extern __shared__ __align__(128) uint8_t smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int rowbytes = K >> 2;
  const int nblk = K >> 4;                       // 16-code blocks per token (packed words per row)
  const int nchunk = (nblk + kChunk - 1) / kChunk;
  const int nblk_pad = nchunk * kChunk;
  const int n0 = blockIdx.x * rows_per_cta;
  const int R = min(rows_per_cta, N - n0);       // at least 1: the grid is ceil(N / rows_per_cta)
  const int n_batches = (R + RB - 1) / RB;
  const int rows_pad = (rows_per_cta + RB - 1) / RB * RB;
  const int bpg = max(1, static_cast<int>(kGroupBytes) / (RB * rowbytes));   // row batches per copy group
  const int rpg = bpg * RB;
  const int n_groups = (R + rpg - 1) / rpg;
  uint8_t* s_w = smem;
  uint8_t* s_act = smem + ((static_cast<size_t>(rows_per_cta) * rowbytes + 15) & ~size_t(15));
  uint32_t* s_red = reinterpret_cast<uint32_t*>(s_act + static_cast<size_t>(MT) * nblk_pad * 16);
  int* s_sum = reinterpret_cast<int*>(s_red + kWarps * MT);
  int* s_acc = s_sum + kWarps * MT;
  uint64_t* s_bar = reinterpret_cast<uint64_t*>((reinterpret_cast<uintptr_t>(s_acc + rows_pad * MT) + 7) & ~uintptr_t(7));

  const uint8_t* wblk = wp + static_cast<size_t>(n0) * rowbytes;
  const uint32_t wbytes = static_cast<uint32_t>(R) * static_cast<uint32_t>(rowbytes);   // N*K < 2^32
  if (tid == kCopyThread) {                      // the thread that will issue the copies owns the barriers
    prefetch_l2_range(wblk, wbytes);
    for (int g = 0; g < n_groups; ++g) mbar_init(&s_bar[g], 1);
    mbar_init_fence();
  } else if (tid == 0) {
    // this CTA's share of the activations (every CTA reads all of x); x may
    // still be being written by the previous grid, which a prefetch cannot
    // disturb
    const uint32_t xbytes = static_cast<uint32_t>(M) * static_cast<uint32_t>(K) *
                            (XIN == kXinF32 ? 4u : (XIN == kXinBF16 ? 2u : 1u));
    const uint32_t share = ((xbytes + gridDim.x - 1) / gridDim.x + 15u) & ~15u;
    const uint32_t lo = blockIdx.x * share;
    if (lo < xbytes) prefetch_l2(static_cast<const uint8_t*>(x) + lo, min(share, xbytes - lo));
  }
  __shared__ int s_fail[1];                      // a contraction warp's weight wait gave up
  if (tid == 0) s_fail[0] = 0;
  for (int i = tid; i < rows_pad * MT; i += kThreads) s_acc[i] = 0;
  pdl_wait();                                    // everything this grid reads is written and visible
  pdl_launch_dependents();
  wblk = launder(wblk);
  x = launder(x);
  scale_in = launder(scale_in);
  gamma = launder(gamma);

  // ---- activations: blocks q = tid, tid + 512, ... of the flat [MT][nblk_pad] space
  const uint32_t s_act32 = smem_u32(s_act);
  const int total = M * nblk_pad;
  // token and block of flat block q (M <= 4: comparisons, no division)
  auto split = [&](int q, int& m, int& b) {
    m = 0;
    if constexpr (MT > 1) {
#pragma unroll
      for (int mm = 1; mm < MT; ++mm) m += q >= mm * nblk_pad ? 1 : 0;
    }
    b = q - m * nblk_pad;
  };
  float sc[MT], rc[MT];                          // scales and recip_for_div of them
  int part[MT];                                  // this thread's token sums
#pragma unroll
  for (int m = 0; m < MT; ++m) {
    sc[m] = 1.f;
    rc[m] = 0.f;
    part[m] = 0;
  }
  auto add_part = [&](int m, int v) {
#pragma unroll
    for (int mm = 0; mm < MT; ++mm) part[mm] += mm == m ? v : 0;
  };
  // stores block b of token m (transposed words t0..t3) and adds its token sum
  auto put = [&](int m, int b, uint32_t t0, uint32_t t1, uint32_t t2, uint32_t t3) {
    sts_v4(s_act32 + 16u * static_cast<uint32_t>(m * nblk_pad + b), t0, t1, t2, t3);
    add_part(m, dp4a_ss(static_cast<int>(t3), 0x01010101,
                        dp4a_ss(static_cast<int>(t2), 0x01010101,
                                dp4a_ss(static_cast<int>(t1), 0x01010101, dp4a_ss(static_cast<int>(t0), 0x01010101, 0)))));
  };

  if constexpr (XIN == kXinI8) {
    if (tid == kCopyThread) {
      for (int g = 0; g < n_groups; ++g) {
        const int r0 = g * rpg, r1 = min(R, r0 + rpg);
        const uint32_t bytes = static_cast<uint32_t>(r1 - r0) * static_cast<uint32_t>(rowbytes);
        mbar_expect_tx(&s_bar[g], bytes);
        bulk_copy_g2s(s_w + static_cast<size_t>(r0) * rowbytes, wblk + static_cast<size_t>(r0) * rowbytes, bytes,
                      &s_bar[g]);
      }
    }
    for (int q = tid; q < total; q += kThreads) {
      int m, b;
      split(q, m, b);
      uint32_t t0 = 0u, t1 = 0u, t2 = 0u, t3 = 0u;
      if (b < nblk) {
        const uint4 v = ld_cg_v4(static_cast<const int8_t*>(x) + static_cast<size_t>(m) * K + 16 * b);
        transpose4x4_bytes(v.x, v.y, v.z, v.w, t0, t1, t2, t3);
      }
      put(m, b, t0, t1, t2, t3);
    }
    if constexpr (!OUT_ACC) {
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        sc[m] = m < M ? ld_cg_f32(scale_in + m) : 1.f;
        rc[m] = recip_for_div(sc[m]);
      }
    }
  } else {
    XBlock<XIN> cache[CB];
#pragma unroll
    for (int u = 0; u < CB; ++u) {
      const int q = tid + kThreads * u;
      cache[u].zero();
      if (q < total) {
        int m, b;
        split(q, m, b);
        if (b < nblk) cache[u].load(x, static_cast<size_t>(m) * nblk + b);
      }
    }
    if (tid == kCopyThread) {                    // after this thread's own x loads are in flight
      for (int g = 0; g < n_groups; ++g) {
        const int r0 = g * rpg, r1 = min(R, r0 + rpg);
        const uint32_t bytes = static_cast<uint32_t>(r1 - r0) * static_cast<uint32_t>(rowbytes);
        mbar_expect_tx(&s_bar[g], bytes);
        bulk_copy_g2s(s_w + static_cast<size_t>(r0) * rowbytes, wblk + static_cast<size_t>(r0) * rowbytes, bytes,
                      &s_bar[g]);
      }
    }
    uint32_t amax[MT];                           // running max of magnitude bits per token
#pragma unroll
    for (int m = 0; m < MT; ++m) amax[m] = 0u;
    auto add_max = [&](const XBlock<XIN>& blk, int m) {
#pragma unroll
      for (int mm = 0; mm < MT; ++mm) amax[mm] = mm == m ? blk.mag_max(amax[mm]) : amax[mm];
    };
#pragma unroll
    for (int u = 0; u < CB; ++u) {
      const int q = tid + kThreads * u;
      if (q < total) {
        int m, b;
        split(q, m, b);
        add_max(cache[u], m);
      }
    }
    for (int q = tid + kThreads * CB; q < total; q += kThreads) {
      int m, b;
      split(q, m, b);
      if (b < nblk) {
        XBlock<XIN> blk;
        blk.load(x, static_cast<size_t>(m) * nblk + b);
        add_max(blk, m);
      }
    }
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      const uint32_t v = __reduce_max_sync(0xffffffffu, XBlock<XIN>::mag_scalar(amax[m]));
      if (lane == 0) s_red[warp * MT + m] = v;
    }
    __syncthreads();
    // each warp reduces the per-warp maxima itself: one load per lane, then one reduction
#pragma unroll
    for (int m = 0; m < MT; ++m)
      sc[m] = token_scale(XBlock<XIN>::mag_to_float(__reduce_max_sync(0xffffffffu, lane < kWarps ? s_red[lane * MT + m] : 0u)));
    // the reciprocals of the rescale, off the critical path of the output
#pragma unroll
    for (int m = 0; m < MT; ++m) rc[m] = recip_for_div(sc[m]);
    if (blockIdx.x == 0 && tid < M && scale_out) {
#pragma unroll
      for (int m = 0; m < MT; ++m)
        if (m == tid) scale_out[m] = sc[m];
    }
    auto quantise = [&](const XBlock<XIN>& blk, int q) {
      int m, b;
      split(q, m, b);
      float s = sc[0];
#pragma unroll
      for (int mm = 1; mm < MT; ++mm) s = mm == m ? sc[mm] : s;
      uint32_t c[16];
      blk.codes(s, c);
      // word i of the transposed block: the codes of values i, 4 + i, 8 + i, 12 + i
      put(m, b, pack4(c[0], c[4], c[8], c[12]), pack4(c[1], c[5], c[9], c[13]), pack4(c[2], c[6], c[10], c[14]),
          pack4(c[3], c[7], c[11], c[15]));
      if (xq_out && blockIdx.x == 0 && b < nblk) {
        uint4 o;
        o.x = pack4(c[0], c[1], c[2], c[3]);
        o.y = pack4(c[4], c[5], c[6], c[7]);
        o.z = pack4(c[8], c[9], c[10], c[11]);
        o.w = pack4(c[12], c[13], c[14], c[15]);
        *reinterpret_cast<uint4*>(xq_out + static_cast<size_t>(m) * K + 16 * b) = o;
      }
    };
#pragma unroll
    for (int u = 0; u < CB; ++u) {
      const int q = tid + kThreads * u;
      if (q < total) quantise(cache[u], q);       // a padding block is zero and gives zero codes
    }
    for (int q = tid + kThreads * CB; q < total; q += kThreads) {
      int m, b;
      split(q, m, b);
      XBlock<XIN> blk;
      blk.zero();
      if (b < nblk) blk.load(x, static_cast<size_t>(m) * nblk + b);
      quantise(blk, q);
    }
  }
  const float gm = OUT_ACC ? 0.f : ld_cg_f32(gamma);
#pragma unroll
  for (int m = 0; m < MT; ++m) {
    const int v = __reduce_add_sync(0xffffffffu, part[m]);
    if (lane == 0) s_sum[warp * MT + m] = v;
  }
  __syncthreads();                               // codes, token sums, zeroed accumulators and mbarriers ready

  // ---- contraction over units (row batch, chunk), an equal contiguous range per warp
  bool ok = true;
  const int units = n_batches * nchunk;
  int u = units * warp / kWarps;
  const int u_end = units * (warp + 1) / kWarps;
  if (u < u_end) {
    // the CTA's rows are all needed: lane g waits for copy group g
    for (int g = lane; g < n_groups; g += 32) ok = mbar_wait_sleep(&s_bar[g], 0u) && ok;
    if (!__all_sync(0xffffffffu, ok) && lane == 0) s_fail[0] = 1;
    __syncwarp();
    const uint32_t s_w32 = smem_u32(s_w) + 4u * lane;
    const uint32_t a32 = s_act32 + 16u * lane;
    int bt = u / nchunk;
    int c = u - bt * nchunk;
    uint32_t ra[RB];                             // shared address of word `lane` of each row of the batch
    auto rows_of = [&](int batch) {
#pragma unroll
      for (int i = 0; i < RB; ++i)
        ra[i] = s_w32 + static_cast<uint32_t>(min(batch * RB + i, R - 1)) * static_cast<uint32_t>(rowbytes);
    };
    rows_of(bt);
    int acc[RB][MT][4];
#pragma unroll
    for (int i = 0; i < RB; ++i)
#pragma unroll
      for (int m = 0; m < MT; ++m) acc[i][m][0] = acc[i][m][1] = acc[i][m][2] = acc[i][m][3] = 0;
    while (true) {
      const uint32_t wo = 128u * static_cast<uint32_t>(c);     // byte offset of the chunk in a row
      uint32_t wv[RB];
#pragma unroll
      for (int i = 0; i < RB; ++i) wv[i] = lds_u32(ra[i] + wo);
      uint4 a[MT];
#pragma unroll
      for (int m = 0; m < MT; ++m)
        a[m] = m < M ? lds_v4(a32 + 16u * static_cast<uint32_t>(m * nblk_pad + kChunk * c)) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int i = 0; i < RB; ++i) {
        const uint32_t p0 = wv[i] & 0x03030303u, p1 = wv[i] & 0x0c0c0c0cu;
        const uint32_t p2 = wv[i] & 0x30303030u, p3 = wv[i] & 0xc0c0c0c0u;
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          acc[i][m][0] = dp4a_us(p0, static_cast<int>(a[m].x), acc[i][m][0]);
          acc[i][m][1] = dp4a_us(p1, static_cast<int>(a[m].y), acc[i][m][1]);
          acc[i][m][2] = dp4a_us(p2, static_cast<int>(a[m].z), acc[i][m][2]);
          acc[i][m][3] = dp4a_us(p3, static_cast<int>(a[m].w), acc[i][m][3]);
        }
      }
      ++u;
      ++c;
      if (c == nchunk || u == u_end) {
        // the batch's partial sums (this warp's chunks of it) into the row accumulators
#pragma unroll
        for (int i = 0; i < RB; ++i) {
#pragma unroll
          for (int m = 0; m < MT; ++m) {
            const int v = __reduce_add_sync(0xffffffffu, acc[i][m][0] + (acc[i][m][1] >> 2) + (acc[i][m][2] >> 4) +
                                                             (acc[i][m][3] >> 6));
            if (lane == 0 && bt * RB + i < R && m < M) atomicAdd(&s_acc[(bt * RB + i) * MT + m], v);
            acc[i][m][0] = acc[i][m][1] = acc[i][m][2] = acc[i][m][3] = 0;
          }
        }
        if (u == u_end) break;
        c = 0;
        rows_of(++bt);
      }
    }
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
  // every bulk copy has landed before the CTA exits: each warp with units
  // waited for every group, so only after a wait that gave up (its copy may
  // still be in flight) does thread 0 wait again
  if (tid == 0 && s_fail[0])
    for (int g = 0; g < n_groups; ++g) ok = mbar_wait_sleep(&s_bar[g], 0u) && ok;
  if (!ok) atomicExch(&g_dp4a_wait_error, 1);
}

namespace {

size_t align16(size_t v) { return (v + 15) & ~size_t(15); }

size_t dp4a_act_bytes(int K, int mt) {
  const size_t nblk_pad = (static_cast<size_t>(K) / 16 + kChunk - 1) / kChunk * kChunk;
  return static_cast<size_t>(mt) * nblk_pad * 16;
}

size_t dp4a_smem(int rows, int K, int mt) {
  const int rb = mt == 4 ? 1 : 2;   // rows_per_batch
  const size_t rowbytes = static_cast<size_t>(K) / 4;
  const size_t bpg = rb * rowbytes >= kGroupBytes ? 1 : kGroupBytes / (rb * rowbytes);
  const size_t rpg = bpg * rb;
  const size_t groups = (static_cast<size_t>(rows) + rpg - 1) / rpg;
  const size_t rows_pad = (static_cast<size_t>(rows) + rb - 1) / rb * rb;
  return align16(static_cast<size_t>(rows) * rowbytes) + dp4a_act_bytes(K, mt) +
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
  if (dp4a_act_bytes(K, mt) > kGemvDp4aMaxAct) return 0;
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
