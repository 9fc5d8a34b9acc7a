// Prefill contraction on the 5th-generation tensor cores (tcgen05, TMEM, TMA).
//
// Passages: "穿越1比特的奇幻旅程" (2B4T summary), section "GPU端：CUDA内核的定制
// 魔法" (W1.58A8 matmul over four-per-byte packed weights: pack, store, load,
// unpack, compute); "BitNet 1-bit LLM 的混合精度微调技术：渐进量化策略", body,
// quantisation functions and forward-pass sentence (per-token absmax int8
// activations, rescale by the factors).
//
// sm_103a has no integer kind for tcgen05.mma, so the contraction runs as
// kind::f16 (fp16 x fp16 -> fp32) and is made exact:
//
//   * Weights. A packed byte holds the fields f = code + 1 of k = 4j .. 4j+3
//     at bits 2i. Spreading two bytes of a word into the low bytes of two
//     16-bit lanes and masking plane i (0x0003 << 2i) leaves 4^i * f in each
//     lane; read as an fp16 bit pattern that is the subnormal 4^i * f * 2^-24.
//     Two byte permutes and eight masks expand 16 codes.
//   * Activations. The matching slot holds x_q * 4^-i, also exact in fp16
//     (|x_q| <= 127, 4^-i >= 2^-6). Slot 16q + 4i + j of a 64-wide k-stage
//     stands for k = 16q + 4j + i: within each 16-code block the activations
//     are stored transposed as a 4 x 4 matrix, matching the plane order.
//   * Every product is then f * x_q * 2^-24 exactly, and every partial sum is
//     an integer times 2^-24 of magnitude at most 2 * 128 * K * 2^-24 <= 1
//     for K <= 65536, so the fp32 accumulator holds it exactly (as long as
//     the tensor core adds such multiples of 2^-24 without loss; the GPU
//     parity tests drive the sum to that bound at K = 65536, on whole and on
//     split tiles, and compare bit for bit). The epilogue subtracts the
//     token sum of x_q times 2^-24 (field = code + 1), which leaves
//     acc * 2^-24 exactly, and applies y = fp32(fp32(acc * gamma) / s),
//     taking acc * gamma as (acc * 2^-24) * (gamma * 2^24).
//
// Kernel shape: persistent, one CTA per SM, tiles of 128 weight rows x BN
// tokens, 448 threads. Whole tiles are dealt round-robin; when the last
// round would leave most SMs idle, the k-stages of its tiles are instead
// split evenly over the CTAs ("stream-K"): each CTA adds its partial sum of
// such a tile into an fp32 buffer with atomic adds, which are exact here
// (every partial is an integer multiple of 2^-24 below 1 in magnitude), and
// the CTA whose contribution completes the tile's k-count applies the
// epilogue from the buffer. The roles:
//   warp 0      TMA producer: activation tile [BN][64] fp16 (128-byte
//               swizzle) and packed weight tile [128][16] bytes per stage,
//               as many stages as fit (6 at BN = 256, 10 at BN = 128: about
//               the latency-bandwidth product of one SM's share of L2);
//   warp 1      allocates the 512 TMEM columns and issues tcgen05.mma
//               (M = 128 weight rows, N = BN tokens, K = 16) from lane 0;
//               TMEM holds two accumulators and the expanded weight stages
//               beside them, or for the 256-token tile one accumulator and
//               four weight stages;
//   warps 2..5  expand each packed stage into the fp16 operand in TMEM
//               (tcgen05.st; a row per thread, warp w holds TMEM lanes
//               32 (w % 4) ..) and arrive at the stage's named barrier,
//               where the MMA warp syncs;
//   warps 6..13 epilogue of the previous tile while the MMA fills the other
//               accumulator; two warps share each TMEM lane quarter, taking
//               alternate 32-token chunks: tcgen05.ld 32x32b (TMEM lane =
//               weight row), stores coalesced along the rows. With one
//               accumulator each warp first parks half of its chunks in
//               the TMEM columns the weight stages leave free and hands
//               the accumulator back before any arithmetic.
// Every wait on the full / empty stage barriers and on the accumulator
// barriers is bounded; the named barriers are matched by construction (both
// sides walk the same schedule). The expansion and epilogue warps sleep
// until the phase completes instead of polling: polling warps take issue
// slots from the MMA warp (measured 4-6 % slower). The TMA producer polls its
// free-stage barrier (no measurable difference).

#include <cuda.h>
#include <cuda_fp16.h>
#include <mutex>

#include "async.cuh"
#include "common.cuh"
#include "kernels.cuh"

namespace bl {

namespace {

constexpr int kBM = 128;                    // weight rows per tile: the MMA's M
constexpr int kBK = 64;                     // k per stage (one 128-byte fp16 swizzle atom)
constexpr int kExpWarps = 4;                 // expansion: one warp per TMEM lane quarter, a row per thread
constexpr int kEpiWarps = 8;                 // epilogue: two warps per TMEM lane quarter
constexpr int kEpiWarp0 = 2 + kExpWarps;     // first epilogue warp
constexpr int kEpiThreads = 32 * kEpiWarps;
constexpr int kThreads = 32 * (kEpiWarp0 + kEpiWarps);   // producer, MMA, expansion, epilogue
constexpr int kMaxBN = 256;                 // tokens per tile at most: the MMA's N
constexpr int kMaxStages = 10;
constexpr int kPrefetchStages = 32;         // weight boxes a CTA prefetches into L2 before its dependency wait
constexpr uint32_t kTmemCols = 512;         // two accumulators of up to 256 columns
constexpr uint32_t kWpBytes = kBM * kBK / 4;    // 2048
// barriers (256 B), then per-token epilogue data for two tiles: scale,
// reciprocal, token sum (fp32) and per-chunk flags
constexpr uint32_t kEpiBytes = 3 * kMaxBN * 4 + 64;
constexpr uint32_t kMiscBytes = 256 + 2 * kEpiBytes;
constexpr uint32_t kSmemBudget = 232448;    // opt-in shared memory per CTA
// The expanded weights (the MMA's A operand) live in tensor memory, in
// 32-column slots of one 64-k stage (128 rows x 64 fp16) each: for tiles of
// up to 224 tokens at the top of each 256-column half, beside two
// accumulators (columns [0, BN) and [256, 256 + BN)); for the 256-token tile
// in the upper half, beside one accumulator. The expansion warps write them
// with tcgen05.st, which the MMA may read right after the handoff. Weights
// written to shared memory instead would need a generic-to-async proxy fence
// before the MMA reads them, and that fence, issued while MMAs are in flight,
// costs the tensor pipe about 40 % (measured: 225 against 128 cycles per
// 128 x 256 x 16 MMA with the stage handoff alone).
// Accumulators: two (the MMA fills one while the epilogue drains the other),
// except for the 256-token tile, whose one accumulator takes [0, 256).
constexpr int acc_bufs(int bn) { return bn == 256 ? 1 : 2; }
// expanded-weight stages in TMEM
constexpr int a_stages(int bn) {
  return bn == 256 ? 4 : (2 * ((256 - bn) / 32) < 4 ? 2 * ((256 - bn) / 32) : 4);
}
// TMA stage: activation tile [BN][64] fp16, then packed weights [128][16] bytes
// (a multiple of 1024 bytes, so every swizzled tile stays 1024-aligned).
constexpr uint32_t stage_bytes(int bn) { return static_cast<uint32_t>(bn) * kBK * 2 + kWpBytes; }
// As many TMA stages as fit: the ring should hold about one latency's worth
// of the SM's operand stream whatever the tile width.
constexpr int stages_for(int bn) {
  return static_cast<int>((kSmemBudget - 1024 - kMiscBytes) / stage_bytes(bn)) < kMaxStages
             ? static_cast<int>((kSmemBudget - 1024 - kMiscBytes) / stage_bytes(bn))
             : kMaxStages;
}
constexpr uint32_t smem_for(int bn) {
  return static_cast<uint32_t>(stages_for(bn)) * stage_bytes(bn) + kMiscBytes + 1024;
}
// barriers: full and empty per TMA stage, efree per expanded stage, tfull and
// tempty per accumulator, then the TMEM base and a flag
static_assert(8 * (2 * kMaxStages + 4 + 4) + 8 <= 256, "barrier area");
__device__ int g_tc_wait_error;

// L2 prefetch of one box of a tensor map.
BL_DEVICE void tma_prefetch_2d(const CUtensorMap* map, int c0, int c1) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(reinterpret_cast<uint64_t>(map)),
               "r"(c0), "r"(c1)
               : "memory");
}

BL_DEVICE void tma_load_2d(void* dst, const CUtensorMap* map, int c0, int c1, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
      : "memory");
}

// Shared-memory matrix descriptor of a K-major operand in the 128-byte
// swizzled layout: 128-byte rows, 8-row groups 1024 bytes apart.
BL_DEVICE uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3fffu);          // start address
  d |= static_cast<uint64_t>(1u) << 16;                        // leading byte offset (unused for this layout)
  d |= static_cast<uint64_t>(1024u >> 4) << 32;                // stride byte offset: 8-row group pitch
  d |= static_cast<uint64_t>(1u) << 46;                        // descriptor version
  d |= static_cast<uint64_t>(2u) << 61;                        // 128-byte swizzle
  return d;
}

// Instruction descriptor, kind::f16: fp32 accumulator, fp16 A and B, both
// K-major, M = 128, N = BN.
template <int BN>
constexpr uint32_t idesc_f16() {
  return (1u << 4) | (0u << 7) | (0u << 10) | (static_cast<uint32_t>(BN >> 3) << 17) |
         (static_cast<uint32_t>(kBM >> 4) << 24);
}

// D (+)= A B^T on the tensor core, A (the weights, 128 rows x 16 k of fp16)
// from tensor memory (lane = row, two consecutive k per 32-bit column, the
// lower k in the low half), B (BN tokens x 16 k) from shared memory.
template <int BN>
BL_DEVICE void umma_f16_ts(uint32_t tmem_d, uint32_t tmem_a, uint64_t bdesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(tmem_d),
      "r"(tmem_a), "l"(bdesc), "r"(idesc_f16<BN>()), "r"(accumulate)
      : "memory");
}

BL_DEVICE void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

BL_DEVICE void named_bar(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
BL_DEVICE void named_arrive(int id, int count) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(count) : "memory");
}
// Named barriers 2 .. 2 + a_stages(BN) - 1 (at most 2 .. 5): expanded stage e
// is ready (the expansion warps arrive, the MMA warp syncs).
constexpr int kExpdBar = 2;
constexpr int kExpdCount = 32 * (kExpWarps + 1);

BL_DEVICE void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
BL_DEVICE void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

BL_DEVICE void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Stores 32 consecutive 32-bit columns of this thread's TMEM lane and waits
// until they are written.
BL_DEVICE void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
      "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
      "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Four fp32 reductions into 16-byte aligned global memory in one request.
BL_DEVICE void red_add_v4(float* p, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// TMEM column of expanded weight stage e (0 <= e < a_stages(BN)): the free
// columns at the top of each accumulator's 256-column half, or the upper half
// when one accumulator takes the lower.
template <int BN>
BL_DEVICE uint32_t a_col(uint32_t e) {
  if constexpr (acc_bufs(BN) == 1) return 256u + 32u * e;
  constexpr uint32_t kHalf = a_stages(BN) >= 2 ? static_cast<uint32_t>(a_stages(BN) / 2) : 1u;
  return (e / kHalf) * 256u + (256u - 32u * kHalf) + 32u * (e % kHalf);
}

}  // namespace

// Work of CTA b (of G): first a run of the k-stages of the split tiles
// [dp_tiles, dp_tiles + sk_tiles) (their sk_tiles * k_iters stages are cut
// into sk_ctas runs of equal length to within one stage, run b for CTA
// b < sk_ctas; the part of a run inside one tile is one item, so a run is
// the end of one tile, any whole tiles, then the start of another), then
// whole tiles b, b + G, ... below dp_tiles. Split work first: its atomic
// partials and the final epilogue of a completed split tile then overlap the
// MMA of the next whole tile instead of ending the kernel. The same code
// runs on the host to list the schedule (tc_items).
struct TcSched {
  int n_tiles_n;   // tiles along the weight rows
  int k_iters;     // k-stages per tile
  int dp_tiles;    // tiles computed whole
  int sk_tiles;    // tiles split over the CTAs
  int sk_ctas;     // CTAs that take a run of split-tile stages

  BL_HOST_DEVICE void run(int b, long long& u0, long long& u1) const {
    u0 = u1 = 0;
    if (b < sk_ctas) {
      const long long U = static_cast<long long>(sk_tiles) * k_iters;
      u0 = U * b / sk_ctas;
      u1 = U * (b + 1) / sk_ctas;
    }
  }
  BL_HOST_DEVICE int split_items(int b) const {
    long long u0, u1;
    run(b, u0, u1);
    return u1 > u0 ? static_cast<int>((u1 - 1) / k_iters - u0 / k_iters) + 1 : 0;
  }
  BL_HOST_DEVICE int items(int b, int G) const {
    const int dp = b < dp_tiles ? (dp_tiles - b + G - 1) / G : 0;
    return split_items(b) + dp;
  }
  // item i of CTA b: tile and k-stage range [k0, k1)
  BL_HOST_DEVICE void item(int b, int G, int i, int& tile, int& k0, int& k1) const {
    const int ns = split_items(b);
    if (i >= ns) {
      tile = b + (i - ns) * G;
      k0 = 0;
      k1 = k_iters;
      return;
    }
    long long u0, u1;
    run(b, u0, u1);
    const long long t = u0 / k_iters + i;
    const long long lo = t * k_iters;
    k0 = static_cast<int>(u0 > lo ? u0 - lo : 0);
    k1 = static_cast<int>(u1 - lo < k_iters ? u1 - lo : k_iters);
    tile = dp_tiles + static_cast<int>(t);
  }
};

template <int BN, bool OUT_ACC>
__global__ void __launch_bounds__(kThreads, 1)
bl_gemm_tc(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
           const float* __restrict__ scale, const int* __restrict__ rowsum, const float* __restrict__ gamma,
           void* __restrict__ out, int M, int N, int K, TcSched sch, float* __restrict__ sk_buf,
           int* __restrict__ sk_cnt) {
  constexpr int kStages = stages_for(BN);
  constexpr uint32_t kStageBytes = stage_bytes(BN);
  constexpr uint32_t kXBytes = static_cast<uint32_t>(BN) * kBK * 2;
  constexpr uint32_t kAcc = acc_bufs(BN);       // TMEM accumulators
  constexpr bool kNarrowSplit = BN <= 64;       // split-tile buffer [row][token] (else [token][row])
  constexpr int kES = a_stages(BN);              // expanded-weight stages (TMEM)
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* misc = smem + kStages * kStageBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(misc);            // TMA stage landed
  uint64_t* empty = full + kStages;                              // TMA stage consumed by the MMA
  uint64_t* efree = empty + kStages;                             // expanded buffer consumed
  uint64_t* tfull = efree + kES;                                 // accumulator b holds a finished tile
  uint64_t* tempty = tfull + 2;                                  // accumulator b has been read out
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 2);
  int* s_last = reinterpret_cast<int*>(tmem_slot + 1);         // this CTA completes a split tile

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_tiles_n = sch.n_tiles_n;
  const int n_items = sch.items(blockIdx.x, gridDim.x);
  (void)K;
  bool ok = true;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int e = 0; e < kES; ++e) mbar_init(&efree[e], 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], kEpiWarps);
    }
    mbar_init_fence();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // The packed weights of this CTA's first k-stages start moving into L2
  // while the grid before ends (a prefetch cannot change what later loads
  // see); the activation operand is written by that grid, so it waits.
  if (warp == 0 && lane == 0) {
    int done = 0;
    for (int item = 0; item < n_items && done < kPrefetchStages; ++item) {
      int tile, k0, k1;
      sch.item(blockIdx.x, gridDim.x, item, tile, k0, k1);
      const int n0 = (tile % n_tiles_n) * kBM;
      for (int it = k0; it < k1 && done < kPrefetchStages; ++it, ++done) tma_prefetch_2d(&tm_w, it * (kBK / 4), n0);
    }
  }
  pdl_wait();                                    // inputs come from the grid before (TMA reads after this)
  pdl_launch_dependents();
  scale = launder(scale);
  rowsum = launder(rowsum);
  gamma = launder(gamma);

  if (warp == 0) {
    // ---- TMA producer
    if (lane == 0) {
      uint32_t g = 0;
      for (int item = 0; item < n_items; ++item) {
        int tile, k0, k1;
        sch.item(blockIdx.x, gridDim.x, item, tile, k0, k1);
        const int n0 = (tile % n_tiles_n) * kBM, m0 = (tile / n_tiles_n) * BN;
        for (int it = k0; it < k1; ++it, ++g) {
          const uint32_t s = g % kStages, ph = (g / kStages) & 1u;
          if (g >= kStages) ok = mbar_wait(&empty[s], ph ^ 1u) && ok;   // polls (one thread)
          uint8_t* st = smem + s * kStageBytes;
          mbar_expect_tx(&full[s], kXBytes + kWpBytes);
          tma_load_2d(st, &tm_x, it * kBK, m0, &full[s]);
          tma_load_2d(st + kXBytes, &tm_w, it * (kBK / 4), n0, &full[s]);
        }
      }
    }
  } else if (warp == 1) {
    // ---- MMA issuer: the whole warp runs the loop, lane 0 issues. It learns
    // that an expanded stage is ready (which also means that its TMA stage
    // has landed) at a named barrier, not by polling an mbarrier: a shared
    // memory access by the thread right after its tcgen05.commit stalls for
    // about 120 cycles, which at four MMAs per stage cost a fifth of the
    // tensor pipe. The barrier cannot hang: the expansion warps arrive once
    // for every stage of the same schedule, whatever their own waits return.
    uint32_t g = 0, tcount = 0;
    for (int item = 0; item < n_items; ++item, ++tcount) {
      int tile, k0, k1;
      sch.item(blockIdx.x, gridDim.x, item, tile, k0, k1);
      // accumulator b's use u of this tile waits for the epilogue of use u - 1
      const uint32_t b = tcount % kAcc, u = tcount / kAcc;
      if (u >= 1) ok = mbar_wait_sleep(&tempty[b], (u & 1u) ^ 1u) && ok;
      const uint32_t d = tmem + b * 256u;
      for (int it = k0; it < k1; ++it, ++g) {
        const uint32_t s = g % kStages, e = g % kES;
        named_bar(kExpdBar + static_cast<int>(e), kExpdCount);
        tc_fence_after();
        if (lane == 0) {
          const uint64_t bdesc = sw128_desc(smem_u32(smem + s * kStageBytes));   // activations [BN][64]
          const uint32_t a = tmem + a_col<BN>(e);                               // weights, TMEM lanes 0..127
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
            umma_f16_ts<BN>(d, a + 8u * kk, bdesc + 2u * kk, (it != k0 || kk != 0) ? 1u : 0u);
          umma_commit(&empty[s]);
          umma_commit(&efree[e]);
        }
        __syncwarp();
      }
      if (lane == 0) umma_commit(&tfull[b]);
      __syncwarp();
    }
  } else if (warp < kEpiWarp0) {
    // ---- weight expansion into TMEM: warp w reaches TMEM lanes 32 (w % 4) ..
    // 32 (w % 4) + 31 only, so lane l expands row 32 (w % 4) + l, all 64
    // codes of the stage (32 columns).
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    uint32_t g = 0;
    for (int item = 0; item < n_items; ++item) {
      int tile, k0, k1;
      sch.item(blockIdx.x, gridDim.x, item, tile, k0, k1);
      for (int it = k0; it < k1; ++it, ++g) {
        const uint32_t s = g % kStages, ph = (g / kStages) & 1u;
        const uint32_t e = g % kES, eph = (g / kES) & 1u;
        ok = mbar_wait_sleep(&full[s], ph) && ok;
        if (g >= static_cast<uint32_t>(kES)) ok = mbar_wait_sleep(&efree[e], eph ^ 1u) && ok;
        tc_fence_after();
        const uint4 pw = *reinterpret_cast<const uint4*>(smem + s * kStageBytes + kXBytes + r * 16);
        const uint32_t words[4] = {pw.x, pw.y, pw.z, pw.w};
        uint32_t v[32];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          // column 8 q + c holds slots 16 q + 2c (low half) and 16 q + 2c + 1
          const uint32_t lo = __byte_perm(words[q], 0u, 0x4140);   // bytes 0, 1 -> 16-bit lanes
          const uint32_t hi = __byte_perm(words[q], 0u, 0x4342);   // bytes 2, 3
          v[8 * q + 0] = lo & 0x00030003u;
          v[8 * q + 1] = hi & 0x00030003u;
          v[8 * q + 2] = lo & 0x000c000cu;
          v[8 * q + 3] = hi & 0x000c000cu;
          v[8 * q + 4] = lo & 0x00300030u;
          v[8 * q + 5] = hi & 0x00300030u;
          v[8 * q + 6] = lo & 0x00c000c0u;
          v[8 * q + 7] = hi & 0x00c000c0u;
        }
        tmem_st32(lane_base + a_col<BN>(e), v);
        tc_fence_before();
        named_arrive(kExpdBar + static_cast<int>(e), kExpdCount);
      }
    }
  } else {
    // ---- epilogue: TMEM lane = weight row, column = token.
    // D = (sum_k field * x_q) * 2^-24 exactly; every value below is an
    // integer smaller than 2^24 in magnitude times 2^-24 (or an integer), so
    // the fp32 arithmetic is exact up to the rescale, which rounds as
    // fp32(fp32(acc * gamma) / s).
    // The reciprocal-and-correction division is exact when t = acc * gamma
    // and the quotient stay in the normal range. With gamma inside
    // 2^-72..2^72, every nonzero |t| lies in gamma..2^24 gamma, inside
    // 2^-96..2^96, and a zero t (acc = 0, so t = +0) gives +0 either way; so a
    // 32-token chunk takes the branch-free form when every scale lies in
    // 2^-96..2^96 and 2^24 gamma max(1/s) < 2^125 and gamma min(1/s) > 2^-99
    // (no quotient can leave the normal range). Other chunks take
    // div_rn_recip, which checks each output.
    const int et = tid - 32 * kEpiWarp0;         // 0 .. kEpiThreads - 1
    const int quarter = warp & 3;
    // the two warps of a lane quarter take alternate 32-token chunks of each tile
    const int chunk0 = 32 * ((warp - kEpiWarp0) >> 2);
    const float gm = OUT_ACC ? 0.f : __ldg(gamma);
    const bool gamma_fast = OUT_ACC || (gm > 0x1p-72f && gm < 0x1p72f);
    const float gm24 = __fmul_rn(gm, 16777216.f);   // exact whenever the branch-free form is taken
    uint32_t tcount = 0;
    for (int item = 0; item < n_items; ++item, ++tcount) {
      int tile, k0, k1;
      sch.item(blockIdx.x, gridDim.x, item, tile, k0, k1);
      const int n0 = (tile % n_tiles_n) * kBM, m0 = (tile / n_tiles_n) * BN;
      const uint32_t b = tcount & 1u;               // per-token data buffer
      const uint32_t bacc = tcount % kAcc;          // accumulator
      float* s_scale = reinterpret_cast<float*>(misc + 256 + b * kEpiBytes);
      float* s_rcp = s_scale + kMaxBN;           // recip_for_div(s): fp32(1/s), or 0 outside 2^-96..2^96
      float* s_rowsum = s_rcp + kMaxBN;          // token sums of x_q times 2^-24 (exact) as fp32
      int* s_fast = reinterpret_cast<int*>(s_rowsum + kMaxBN);   // per 32-token chunk: the branch-free form is exact
      for (int i = et; i < BN; i += kEpiThreads) {
        const int m = m0 + i;
        const float sc = (!OUT_ACC && m < M) ? __ldg(scale + m) : 1.f;
        s_scale[i] = sc;
        s_rcp[i] = recip_for_div(sc);
        // |sum| <= 128 K <= 2^23: exact, and so is the scaling by 2^-24
        s_rowsum[i] = __fmul_rn(static_cast<float>(m < M ? __ldg(rowsum + m) : 0), 0x1p-24f);
      }
      for (int c = warp - kEpiWarp0; c < BN / 32; c += kEpiWarps) {
        const int m = m0 + c * 32 + lane;
        const float sc = (!OUT_ACC && m < M) ? __ldg(scale + m) : 1.f;
        const float r = recip_for_div(sc);
        float rmax = r, rmin = r;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          rmax = fmaxf(rmax, __shfl_xor_sync(0xffffffffu, rmax, o));
          rmin = fminf(rmin, __shfl_xor_sync(0xffffffffu, rmin, o));
        }
        const bool fast = OUT_ACC || (gamma_fast && rmin != 0.f && __fmul_rn(__fmul_rn(gm, 0x1p24f), rmax) < 0x1p125f &&
                                      __fmul_rn(gm, rmin) > 0x1p-99f);
        if (lane == 0) s_fast[c] = fast;
      }
      named_bar(1, kEpiThreads);                 // the per-token data is complete
      ok = mbar_wait_sleep(&tfull[bacc], (tcount / kAcc) & 1u) && ok;
      tc_fence_after();
      const int n = n0 + quarter * 32 + lane;
      float* yrow = OUT_ACC ? nullptr : static_cast<float*>(out) + static_cast<size_t>(m0) * N + n;
      int32_t* arow = OUT_ACC ? static_cast<int32_t*>(out) + static_cast<size_t>(m0) * N + n : nullptr;
      // y (or acc) of tokens m0 + c0 .. m0 + c0 + 31 of row n from the sums D.
      // D - rowsum 2^-24 = acc 2^-24 exactly (both multiples of 2^-24, the
      // difference below 2^23 2^-24); acc 2^-24 times gamma 2^24 is the real
      // number acc gamma, so t rounds as fp32(acc * gamma).
      auto emit = [&](int c0, const float (&dv)[32]) {
        const bool full_chunk = m0 + c0 + 32 <= M;
        if (full_chunk && s_fast[c0 >> 5]) {
#pragma unroll
          for (int j4 = 0; j4 < 32; j4 += 4) {
            const float4 rs = *reinterpret_cast<const float4*>(s_rowsum + c0 + j4);   // 16-byte aligned
            const float rsv[4] = {rs.x, rs.y, rs.z, rs.w};
            if constexpr (OUT_ACC) {
#pragma unroll
              for (int jj = 0; jj < 4; ++jj)
                arow[static_cast<size_t>(c0 + j4 + jj) * N] =
                    static_cast<int>(__fmul_rn(__fsub_rn(dv[j4 + jj], rsv[jj]), 16777216.f));
            } else {
              const float4 rc = *reinterpret_cast<const float4*>(s_rcp + c0 + j4);
              const float4 sc = *reinterpret_cast<const float4*>(s_scale + c0 + j4);
              const float rcv[4] = {rc.x, rc.y, rc.z, rc.w}, scv[4] = {sc.x, sc.y, sc.z, sc.w};
#pragma unroll
              for (int jj = 0; jj < 4; ++jj) {
                const float t = __fmul_rn(__fsub_rn(dv[j4 + jj], rsv[jj]), gm24);
                const float q = __fmul_rn(t, rcv[jj]);
                yrow[static_cast<size_t>(c0 + j4 + jj) * N] = __fmaf_rn(__fmaf_rn(-q, scv[jj], t), rcv[jj], q);
              }
            }
          }
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            if (m0 + c0 + j < M) {
              const float acc = __fmul_rn(__fsub_rn(dv[j], s_rowsum[c0 + j]), 16777216.f);
              const size_t o = static_cast<size_t>(c0 + j) * N;
              if constexpr (OUT_ACC) {
                arow[o] = static_cast<int>(acc);
              } else {
                yrow[o] = div_rn_recip(__fmul_rn(acc, gm), s_scale[c0 + j], s_rcp[c0 + j]);
              }
            }
          }
        }
      };
      // The accumulator goes back to the MMA as early as possible. With two
      // accumulators the MMA fills the other one meanwhile, so the warp reads
      // its chunks one at a time and hands the accumulator back right after
      // its last TMEM load. With one (the 256-token tile) the MMA waits for
      // it: the warp first moves its first two chunks into the free TMEM
      // columns above the weight stages ([384, 512), 64 per warp of a lane
      // quarter) and loads its last two into registers, hands the
      // accumulator back after those four loads and two stores, and only then
      // does the arithmetic and the memory traffic of all four.
      const uint32_t lane_q = static_cast<uint32_t>(quarter * 32) << 16;
      const uint32_t acc_base = tmem + bacc * 256u + lane_q;
      auto release = [&]() {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[bacc]);
      };
      auto drain = [&](auto&& consume) {
        if constexpr (kAcc == 1) {
          const uint32_t spare = tmem + lane_q + 384u + 64u * static_cast<uint32_t>((warp - kEpiWarp0) >> 2);
          uint32_t v[32], w[32];
          tmem_ld32(acc_base + static_cast<uint32_t>(chunk0), v);
          tmem_st32(spare, v);
          tmem_ld32(acc_base + static_cast<uint32_t>(chunk0 + 64), v);
          tmem_st32(spare + 32u, v);
          tmem_ld32(acc_base + static_cast<uint32_t>(chunk0 + 128), v);
          tmem_ld32(acc_base + static_cast<uint32_t>(chunk0 + 192), w);
          release();
          consume(chunk0 + 128, v);
          consume(chunk0 + 192, w);
          tmem_ld32(spare, v);
          consume(chunk0, v);
          tmem_ld32(spare + 32u, v);
          consume(chunk0 + 64, v);
        } else {
          bool released = false;
#pragma unroll 1
          for (int c0 = chunk0; c0 < BN; c0 += 64) {
            uint32_t v[32];
            tmem_ld32(acc_base + static_cast<uint32_t>(c0), v);
            if (c0 + 64 >= BN) {
              release();
              released = true;
            }
            consume(c0, v);
          }
          if (!released) release();
        }
      };
      if (tile < sch.dp_tiles) {
        // a whole tile: y straight from the accumulator
        drain([&](int c0, const uint32_t (&v)[32]) {
          if (n >= N) return;
          float dv[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) dv[j] = __uint_as_float(v[j]);
          emit(c0, dv);
        });
      } else {
        // part of a split tile: add the partial into the tile's buffer.
        // Narrow tiles (BN <= 64, every tile split over all SMs) keep it
        // [row][token] and add four consecutive tokens per vector reduction:
        // a quarter of the reduction instructions. Wider tiles keep it
        // [token][row], where the 32 lanes of a warp add 32 consecutive
        // floats; there the vector form (32 lines per instruction) made the
        // 2048 x 6912 -> 2560 forward 16 % slower. Tokens past M read zero
        // operand rows, so their sums are 0 and may be added (the buffer
        // holds BN tokens per row).
        const int sk = tile - sch.dp_tiles;
        float* buf = sk_buf + static_cast<size_t>(sk) * BN * kBM +
                     (kNarrowSplit ? static_cast<size_t>(quarter * 32 + lane) * BN : static_cast<size_t>(quarter * 32 + lane));
        const int m_left = M - m0;
        drain([&](int c0, const uint32_t (&v)[32]) {
          if (n >= N) return;
          if constexpr (kNarrowSplit) {
#pragma unroll
            for (int j = 0; j < 32; j += 4) red_add_v4(buf + c0 + j, v[j], v[j + 1], v[j + 2], v[j + 3]);
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (c0 + j < m_left) atomicAdd(buf + static_cast<size_t>(c0 + j) * kBM, __uint_as_float(v[j]));
          }
        });
        // the CTA whose stages complete the tile's k-count writes it
        __threadfence();
        named_bar(1, kEpiThreads);
        if (et == 0) *s_last = atomicAdd(sk_cnt + sk, k1 - k0) + (k1 - k0) == sch.k_iters;
        named_bar(1, kEpiThreads);
        if (*s_last) {
          __threadfence();
#pragma unroll 1
          for (int c0 = chunk0; c0 < BN; c0 += 64) {
            if (n >= N) break;
            float dv[32];
            if constexpr (kNarrowSplit) {
#pragma unroll
              for (int j = 0; j < 32; j += 4) {
                const float4 q = __ldcg(reinterpret_cast<const float4*>(buf + c0 + j));
                dv[j] = q.x;
                dv[j + 1] = q.y;
                dv[j + 2] = q.z;
                dv[j + 3] = q.w;
              }
            } else {
#pragma unroll
              for (int j = 0; j < 32; ++j)
                dv[j] = c0 + j < m_left ? __ldcg(buf + static_cast<size_t>(c0 + j) * kBM) : 0.f;
            }
            emit(c0, dv);
          }
        }
        named_bar(1, kEpiThreads);               // s_last is read before the next split tile sets it
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
  if (!ok) atomicExch(&g_tc_wait_error, 1);
}

// Per-token activation pass for the tensor-core path: the scale, optional
// int8 codes, the token sum of the codes, and the fp16 operand (transposed
// 16-code blocks, slot 16q + 4i + j = x_q[16q + 4j + i] * 4^-i).
//
// One CTA of kPermThreads per token. Thread t takes 16-code blocks t,
// t + kPermThreads, ...; the first kPermCache of them (every block up to
// K = 8192) stay in registers between the absmax reduction (warp shuffles,
// then one CTA barrier) and the quantisation, so x is read from memory once.
// For bf16 input the absmax is the unsigned max of the magnitude bits, taken
// without widening (for finite values the bits order like the magnitudes).
// Codes are rounded with the 1.5 * 2^23 addition (exact round-to-nearest-even
// for |v| <= 2^22 after the clamp), which also leaves the code in the low
// mantissa byte.
namespace {

constexpr int kPermThreads = 128;            // threads per token
constexpr int kPermCache = 4;                // 16-code blocks per thread kept in registers

// Raw 16-activation block: 2 (bf16) or 4 (fp32) 16-byte vectors.
template <int XIN> struct Raw16 {
  static constexpr int kVec = XIN == kXinF32 ? 4 : 2;
  uint4 v[kVec];
  BL_DEVICE void load(const void* x, size_t off) {
    const uint4* p = XIN == kXinF32 ? reinterpret_cast<const uint4*>(static_cast<const float*>(x) + off)
                                    : reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(x) + off);
#pragma unroll
    for (int i = 0; i < kVec; ++i) v[i] = __ldg(p + i);
  }
  // Folds max|x| of the 16 values into the running maximum: for bf16 as the
  // unsigned max of the magnitude bits (two 16-bit lanes in `mag`; for
  // finite values they order like the magnitudes), for fp32 in floats.
  BL_DEVICE void max_abs(float& amax, uint32_t& mag) const {
    if constexpr (XIN == kXinBF16) {
      constexpr uint32_t m = 0x7fff7fffu;
      const uint32_t a = __vimax3_u16x2(v[0].x & m, v[0].y & m, v[0].z & m);
      const uint32_t b = __vimax3_u16x2(v[0].w & m, v[1].x & m, v[1].y & m);
      const uint32_t c = __vimax3_u16x2(v[1].z & m, v[1].w & m, a);
      mag = __vimax3_u16x2(b, c, mag);
    } else {
      float f[16];
      widen(f);
#pragma unroll
      for (int j = 0; j < 16; ++j) amax = fmaxf(amax, fabsf(f[j]));
    }
  }
  // The larger magnitude of the two 16-bit lanes as an fp32 value.
  static BL_DEVICE float mag_to_float(uint32_t mag) { return __uint_as_float(max(mag & 0xffffu, mag >> 16) << 16); }
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

// Codes of one 16-block and its fp16 operand block, from the biased codes
// e[j] = 1.5 * 2^23 + x_q[16b + j] (exact floats whose low mantissa byte is
// the code in two's complement).
BL_DEVICE void emit_block(const float (&e)[16], int8_t* xq_row, __half* xp_row, int b, bool write_xq, int& sum) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t b0 = __float_as_uint(e[4 * i]);
    const uint32_t b1 = __float_as_uint(e[4 * i + 1]);
    const uint32_t b2 = __float_as_uint(e[4 * i + 2]);
    const uint32_t b3 = __float_as_uint(e[4 * i + 3]);
    w[i] = __byte_perm(__byte_perm(b0, b1, 0x0040), __byte_perm(b2, b3, 0x0040), 0x5410);
  }
  if (write_xq) *reinterpret_cast<uint4*>(xq_row + 16 * b) = make_uint4(w[0], w[1], w[2], w[3]);
  sum = dp4a_ss(static_cast<int>(w[0]), 0x01010101, sum);
  sum = dp4a_ss(static_cast<int>(w[1]), 0x01010101, sum);
  sum = dp4a_ss(static_cast<int>(w[2]), 0x01010101, sum);
  sum = dp4a_ss(static_cast<int>(w[3]), 0x01010101, sum);
  // slot 4i + j holds x_q[4j + i] * 4^-i: e * 4^-i - 1.5 * 2^23 * 4^-i in one
  // fused multiply-add, exact (both products are exact and so is their
  // difference, a small integer times a power of two), then to fp16 (exact)
  uint32_t h[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float sc = i == 0 ? 1.f : (i == 1 ? 0.25f : (i == 2 ? 0.0625f : 0.015625f));
    const float off = -12582912.f * sc;
    const __half2 lo = __floats2half2_rn(__fmaf_rn(e[i], sc, off), __fmaf_rn(e[4 + i], sc, off));
    const __half2 hi = __floats2half2_rn(__fmaf_rn(e[8 + i], sc, off), __fmaf_rn(e[12 + i], sc, off));
    h[2 * i] = *reinterpret_cast<const uint32_t*>(&lo);
    h[2 * i + 1] = *reinterpret_cast<const uint32_t*>(&hi);
  }
  uint4* dst = reinterpret_cast<uint4*>(xp_row + 16 * b);
  dst[0] = make_uint4(h[0], h[1], h[2], h[3]);
  dst[1] = make_uint4(h[4], h[5], h[6], h[7]);
}

// The code of x, clip(rint(fp32(x * s)), -128, 127), biased: 1.5 * 2^23 +
// the code (the addition rounds the clamped product to the nearest integer,
// ties to even, and is exact for it).
BL_DEVICE float code_biased(float x, float s) {
  const float v = fminf(fmaxf(__fmul_rn(x, s), -128.f), 127.f);
  return __fadd_rn(v, 12582912.f);
}

}  // namespace

template <int XIN>
__global__ void __launch_bounds__(kPermThreads)
bl_act_perm(const void* __restrict__ x, const float* __restrict__ scale_in, int M, int K,
            int8_t* __restrict__ xq_out, float* __restrict__ scale_out, __half* __restrict__ xperm,
            int* __restrict__ rowsum, uint4* __restrict__ zero, size_t zero_n16) {
  __shared__ float s_max[kPermThreads / 32];
  __shared__ int s_sum[kPermThreads / 32];
  pdl_wait();
  pdl_launch_dependents();
  x = launder(x);
  scale_in = launder(scale_in);
  // the contraction's split-tile buffer and counters start from zero (after
  // the wait: the contraction before this one may still have used them)
  for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < zero_n16;
       i += static_cast<size_t>(gridDim.x) * blockDim.x)
    zero[i] = make_uint4(0u, 0u, 0u, 0u);
  const int m = blockIdx.x;                      // one CTA per token
  if (m >= M) return;                            // uniform over the CTA
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nblk = K >> 4;
  const size_t row = static_cast<size_t>(m) * K;
  __half* xp_row = xperm + row;
  int sum = 0;
  if constexpr (XIN == kXinI8) {
    const int8_t* xr = static_cast<const int8_t*>(x) + row;
    for (int b = tid; b < nblk; b += kPermThreads) {
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(xr) + b);
      const uint32_t u[4] = {v.x, v.y, v.z, v.w};
      float q[16];
#pragma unroll
      for (int j = 0; j < 16; ++j)
        q[j] = __fadd_rn(static_cast<float>(static_cast<int8_t>((u[j >> 2] >> (8 * (j & 3))) & 0xffu)), 12582912.f);
      emit_block(q, nullptr, xp_row, b, false, sum);
    }
  } else {
    Raw16<XIN> cache[kPermCache];
    float amax = 0.f;                            // fp32 input: the running max|x|
    uint32_t mrun = 0u;                          // bf16 input: running max of the magnitude bits
#pragma unroll
    for (int c = 0; c < kPermCache; ++c) {
      const int b = tid + kPermThreads * c;
      if (b < nblk) {
        cache[c].load(x, row + 16 * b);
        cache[c].max_abs(amax, mrun);
      }
    }
    for (int b = tid + kPermThreads * kPermCache; b < nblk; b += kPermThreads) {
      Raw16<XIN> r;
      r.load(x, row + 16 * b);
      r.max_abs(amax, mrun);
    }
    if constexpr (XIN == kXinBF16) amax = Raw16<XIN>::mag_to_float(mrun);
    amax = warp_max(amax);
    if (lane == 0) s_max[warp] = amax;
    __syncthreads();
    float a = 0.f;
#pragma unroll
    for (int w = 0; w < kPermThreads / 32; ++w) a = fmaxf(a, s_max[w]);
    const float s = token_scale(a);
    if (tid == 0 && scale_out) scale_out[m] = s;
    int8_t* xq_row = xq_out ? xq_out + row : nullptr;
#pragma unroll
    for (int c = 0; c < kPermCache; ++c) {
      const int b = tid + kPermThreads * c;
      if (b < nblk) {
        float f[16], q[16];
        cache[c].widen(f);
#pragma unroll
        for (int j = 0; j < 16; ++j) q[j] = code_biased(f[j], s);
        emit_block(q, xq_row, xp_row, b, xq_out != nullptr, sum);
      }
    }
    for (int b = tid + kPermThreads * kPermCache; b < nblk; b += kPermThreads) {
      Raw16<XIN> r;
      r.load(x, row + 16 * b);
      float f[16], q[16];
      r.widen(f);
#pragma unroll
      for (int j = 0; j < 16; ++j) q[j] = code_biased(f[j], s);
      emit_block(q, xq_row, xp_row, b, xq_out != nullptr, sum);
    }
  }
  sum = warp_sum(sum);
  if (lane == 0) s_sum[warp] = sum;
  __syncthreads();
  if (tid == 0) {
    int t = 0;
#pragma unroll
    for (int w = 0; w < kPermThreads / 32; ++w) t += s_sum[w];
    rowsum[m] = t;
  }
}

namespace {

using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                 const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encode_fn() {
  static EncodeTiled fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiled>(p);
  });
  return fn;
}

}  // namespace

// Time of one k-stage of a tile, in units of the 256-token stage with the
// weights in shared memory, measured on B300 over the 2B and 7B projection
// shapes at M = 512-2048. The tiles with their weights in TMEM take 0.62
// (256 tokens, one accumulator) to 0.76; the 32- and 64-token tiles keep
// the earlier estimate. (The 256-token tile's figure was measured before its
// epilogue handed the accumulator back early, which made it 1-4 % faster.)
constexpr double stage_cost(int bn) {
  return bn == 256 ? 0.62 : bn == 224 ? 0.76 : bn == 192 ? 0.72 : bn == 160 ? 0.70 : bn == 128 ? 0.67 : 0.78;
}

// Launch plan: token-tile width BN, grid and work split. For each BN the
// tiles are dealt round-robin to the SMs; a last round that would occupy at
// most a tenth of the SMs is split by k-stages instead (stream-K), costed as
// the fraction of a round it fills plus a fixed 12 k-stages for the partial
// sums and the final epilogue. (Every contributing CTA adds a whole 128 x BN
// fp32 partial with atomics; with more split tiles that traffic costs more
// than the idle SMs it saves.) A narrow tile that holds every token
// (M <= BN <= 64) has small partials, so when there are fewer such tiles
// than SMs they are always split. A plan's cost is its rounds times
// stage_cost(BN); among equal costs the plan with fewer token tiles, then
// the narrower tile, wins.
TcPlan tc_plan(int M, int N, int K, int sms) {
  const int cands[7] = {256, 224, 192, 160, 128, 64, 32};
  const int tn = (N + kBM - 1) / kBM;
  const int k_iters = K / kBK;
  TcPlan best;
  double best_cost = -1.0;
  int best_tm = 0;
  for (int bn : cands) {
    // the 256-token tile has one accumulator, so the MMA still waits for
    // part of each epilogue: it needs tiles long in k and nearly full in tokens
    if (bn == 256 && (M <= 192 || k_iters < 16)) continue;
    const int tm = (M + bn - 1) / bn;
    const int tiles = tn * tm;
    const int full = tiles / sms, r = tiles % sms;
    const bool sk = r > 0 && (10 * r <= sms || (full == 0 && bn <= 64 && tm == 1));
    const double rounds =
        r == 0 ? full : (sk ? full + static_cast<double>(r) / sms + 12.0 / k_iters : full + 1.0);
    const double cost = rounds * stage_cost(bn);
    if (best_cost >= 0.0 && (cost > best_cost || (cost == best_cost && tm > best_tm))) continue;
    best_cost = cost;
    best_tm = tm;
    TcPlan p;
    p.bn = bn;
    p.n_tiles_n = tn;
    p.k_iters = k_iters;
    p.dp_tiles = sk ? full * sms : tiles;
    p.sk_tiles = sk ? r : 0;
    long long ctas = sk ? static_cast<long long>(r) * k_iters / 4 : 0;   // runs of at least 4 stages
    if (ctas > sms) ctas = sms;
    if (sk && ctas < 1) ctas = 1;
    p.sk_ctas = static_cast<int>(ctas);
    p.grid = full > 0 ? sms : (sk ? p.sk_ctas : tiles);
    const size_t buf = static_cast<size_t>(p.sk_tiles) * bn * kBM * 4;
    p.sk_buf_bytes = (buf + 255) / 256 * 256;
    p.sk_bytes = p.sk_buf_bytes + (static_cast<size_t>(p.sk_tiles) * 4 + 255) / 256 * 256;
    best = p;
  }
  return best;
}

namespace {

TcSched sched_of(const TcPlan& p) {
  TcSched sch;
  sch.n_tiles_n = p.n_tiles_n;
  sch.k_iters = p.k_iters;
  sch.dp_tiles = p.dp_tiles;
  sch.sk_tiles = p.sk_tiles;
  sch.sk_ctas = p.sk_ctas;
  return sch;
}

}  // namespace

int tc_items(const TcPlan& p, int b, int max_items, int32_t* out) {
  const TcSched sch = sched_of(p);
  const int n = sch.items(b, p.grid);
  for (int i = 0; i < n && i < max_items; ++i) {
    int tile, k0, k1;
    sch.item(b, p.grid, i, tile, k0, k1);
    out[3 * i] = tile;
    out[3 * i + 1] = k0;
    out[3 * i + 2] = k1;
  }
  return n;
}

namespace {

template <int BN, bool OUT_ACC>
cudaError_t launch_tc_t(const CUtensorMap& tm_x, const CUtensorMap& tm_w, const float* scale, const int* rowsum,
                        const float* gamma, void* out, int M, int N, int K, const TcPlan& p, void* sk_ws,
                        cudaStream_t s) {
  constexpr size_t smem = smem_for(BN);
  static_assert(smem <= kSmemBudget, "shared memory budget");
  static_assert(stages_for(BN) >= 4, "pipeline depth");
  const cudaError_t e = ensure_smem(reinterpret_cast<const void*>(bl_gemm_tc<BN, OUT_ACC>), smem);
  if (e != cudaSuccess) return e;
  const TcSched sch = sched_of(p);
  float* sk_buf = static_cast<float*>(sk_ws);
  int* sk_cnt = reinterpret_cast<int*>(static_cast<uint8_t*>(sk_ws) + p.sk_buf_bytes);
  return launch_pdl(bl_gemm_tc<BN, OUT_ACC>, dim3(p.grid), dim3(kThreads), smem, s, tm_x, tm_w, scale, rowsum, gamma,
                    out, M, N, K, sch, sk_buf, sk_cnt);
}

template <bool OUT_ACC>
cudaError_t launch_tc_bn(const TcPlan& p, const CUtensorMap& tm_x, const CUtensorMap& tm_w, const float* scale,
                         const int* rowsum, const float* gamma, void* out, int M, int N, int K, void* sk_ws,
                         cudaStream_t s) {
  switch (p.bn) {
    case 224: return launch_tc_t<224, OUT_ACC>(tm_x, tm_w, scale, rowsum, gamma, out, M, N, K, p, sk_ws, s);
    case 192: return launch_tc_t<192, OUT_ACC>(tm_x, tm_w, scale, rowsum, gamma, out, M, N, K, p, sk_ws, s);
    case 160: return launch_tc_t<160, OUT_ACC>(tm_x, tm_w, scale, rowsum, gamma, out, M, N, K, p, sk_ws, s);
    case 128: return launch_tc_t<128, OUT_ACC>(tm_x, tm_w, scale, rowsum, gamma, out, M, N, K, p, sk_ws, s);
    case 64: return launch_tc_t<64, OUT_ACC>(tm_x, tm_w, scale, rowsum, gamma, out, M, N, K, p, sk_ws, s);
    case 32: return launch_tc_t<32, OUT_ACC>(tm_x, tm_w, scale, rowsum, gamma, out, M, N, K, p, sk_ws, s);
    default: return launch_tc_t<256, OUT_ACC>(tm_x, tm_w, scale, rowsum, gamma, out, M, N, K, p, sk_ws, s);
  }
}

}  // namespace

cudaError_t launch_act_perm(const void* x, int xin, const float* scale_in, int M, int K, int8_t* xq_out,
                            float* scale_out, void* xperm, int* rowsum, void* zero, size_t zero_bytes,
                            cudaStream_t s) {
  __half* xp = static_cast<__half*>(xperm);
  uint4* z = static_cast<uint4*>(zero);
  const size_t n16 = zero_bytes / 16;
  const int grid = M;
  if (xin == kXinF32)
    return launch_pdl(bl_act_perm<kXinF32>, dim3(grid), dim3(kPermThreads), 0, s, x, scale_in, M, K, xq_out, scale_out, xp,
                      rowsum, z, n16);
  if (xin == kXinBF16)
    return launch_pdl(bl_act_perm<kXinBF16>, dim3(grid), dim3(kPermThreads), 0, s, x, scale_in, M, K, xq_out, scale_out, xp,
                      rowsum, z, n16);
  return launch_pdl(bl_act_perm<kXinI8>, dim3(grid), dim3(kPermThreads), 0, s, x, scale_in, M, K, xq_out, scale_out, xp, rowsum,
                    z, n16);
}

cudaError_t launch_gemm_tc(const void* xperm, const uint8_t* wp, const float* scale, const int* rowsum,
                           const float* gamma, void* out, bool out_acc, int M, int N, int K, const TcPlan& plan,
                           void* sk_ws, cudaStream_t s) {
  EncodeTiled enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  const int bn = plan.bn;
  CUtensorMap tm_x, tm_w;
  {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(M)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
    const cuuint32_t box[2] = {kBK, static_cast<cuuint32_t>(bn)};
    const cuuint32_t es[2] = {1, 1};
    if (enc(&tm_x, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(xperm), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K / 4), static_cast<cuuint64_t>(N)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K / 4)};
    const cuuint32_t box[2] = {kBK / 4, kBM};
    const cuuint32_t es[2] = {1, 1};
    if (enc(&tm_w, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(wp), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  if (out_acc) return launch_tc_bn<true>(plan, tm_x, tm_w, scale, rowsum, gamma, out, M, N, K, sk_ws, s);
  return launch_tc_bn<false>(plan, tm_x, tm_w, scale, rowsum, gamma, out, M, N, K, sk_ws, s);
}

cudaError_t take_tc_wait_error(int* flag) {
  int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(flag, g_tc_wait_error, sizeof(int));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_tc_wait_error, &zero, sizeof(int));
}

}  // namespace bl
