// GEMV for any K % 4 == 0: packed-ternary weights x int8 activations, the
// path for shapes the other contraction kernels do not take (K % 64 != 0).
//
// Passages: "穿越1比特的奇幻旅程" (2B4T summary), section "GPU端：CUDA内核的定制
// 魔法" (W1.58A8 matmul over four-per-byte packed weights: pack, store, load,
// unpack, compute); "BitNet 1-bit LLM 的混合精度微调技术：渐进量化策略", body,
// forward-pass sentence (multiply back by the factors).
//
// Layout trick. A 32-bit word of a packed row holds 16 codes; byte j carries
// k = 4j..4j+3 with the code of k = 4j+i in bits 2i..2i+1 as code+1. Masking
// the word with 0x03030303 << 2i gives, in byte j, 4^i * field(4j+i): four
// unsigned bytes that dp4a can multiply with four signed activations
// x[i], x[4+i], x[8+i], x[12+i]. So the activations are staged in shared
// memory with each 16-byte block transposed as a 4x4 byte matrix, and the
// field planes go straight into dp4a.u32.s32 with no shifts:
//   sum_k field*x = acc0 + acc1/4 + acc2/16 + acc3/64   (exact: each acc_i is a
//   multiple of 4^i)
// and since field = code + 1, sum_k code*x = that - sum_k x.
//
// One warp per output row at a time; each lane streams 16-byte chunks of the
// row with L1-bypassing loads, the warp reduces with shuffles, and lane m
// writes token m's output.

#include "common.cuh"
#include "kernels.cuh"

namespace bl {

namespace {

BL_DEVICE uint4 ld_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

// index of activation k inside the transposed staging buffer
BL_DEVICE int perm_index(int k) { return (k & ~15) | ((k & 3) << 2) | ((k >> 2) & 3); }

}  // namespace

template <int MT, bool VEC, GemvOut OUT>
__global__ void __launch_bounds__(kGemvThreads)
bl_gemv_w2a8(const uint8_t* __restrict__ wp, const int8_t* __restrict__ xq,
             const float* __restrict__ scale, const float* __restrict__ gamma,
             void* __restrict__ out, int M, int N, int K) {
  extern __shared__ __align__(16) uint8_t s_x[];          // MT x Kp transposed activations
  __shared__ int s_rowsum[MT];
  pdl_wait();
  pdl_launch_dependents();
  wp = launder(wp);
  xq = launder(xq);
  scale = launder(scale);
  gamma = launder(gamma);
  const int Kp = (K + 63) & ~63;                          // staging row length, zero padded
  const int m0 = blockIdx.y * MT;
  const int mcount = min(MT, M - m0);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  if (tid < MT) s_rowsum[tid] = 0;
  __syncthreads();

  // ---- stage x_q (transposed per 16-byte block) and its row sums
  for (int m = 0; m < MT; ++m) {
    const int8_t* src = xq + static_cast<size_t>(m0 + m) * K;
    int part = 0;
    for (int b = tid; b < Kp / 16; b += blockDim.x) {
      uint32_t w[4] = {0u, 0u, 0u, 0u};
      if (m < mcount) {
        if (VEC) {
          if (16 * b < K) {
            const uint4 v = *reinterpret_cast<const uint4*>(src + 16 * b);
            w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
          }
        } else {
#pragma unroll
          for (int j = 0; j < 4; ++j)
            if (16 * b + 4 * j < K) w[j] = *reinterpret_cast<const uint32_t*>(src + 16 * b + 4 * j);
        }
      }
      part = dp4a_ss(static_cast<int>(w[0]), 0x01010101, part);
      part = dp4a_ss(static_cast<int>(w[1]), 0x01010101, part);
      part = dp4a_ss(static_cast<int>(w[2]), 0x01010101, part);
      part = dp4a_ss(static_cast<int>(w[3]), 0x01010101, part);
      uint4 t;
      transpose4x4_bytes(w[0], w[1], w[2], w[3], t.x, t.y, t.z, t.w);
      *reinterpret_cast<uint4*>(s_x + static_cast<size_t>(m) * Kp + 16 * b) = t;
    }
    part = warp_sum(part);
    if (lane == 0 && part) atomicAdd(&s_rowsum[m], part);
  }
  __syncthreads();

  const float g = (OUT == GemvOut::kY) ? *gamma : 0.f;
  const int warps_total = gridDim.x * (blockDim.x >> 5);
  const int rowbytes = K >> 2;

  for (int n = blockIdx.x * (blockDim.x >> 5) + warp; n < N; n += warps_total) {
    int acc[MT][4];
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[m][i] = 0;

    const uint8_t* row = wp + static_cast<size_t>(n) * rowbytes;
    if (VEC) {
      const uint4* row4 = reinterpret_cast<const uint4*>(row);
      const int nchunk = rowbytes >> 4;                  // K % 64 == 0 on this path
      for (int c = lane; c < nchunk; c += 32) {
        const uint4 wv = ld_stream(row4 + c);
        const uint32_t words[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const uint32_t f0 = words[t] & 0x03030303u, f1 = words[t] & 0x0c0c0c0cu;
          const uint32_t f2 = words[t] & 0x30303030u, f3 = words[t] & 0xc0c0c0c0u;
#pragma unroll
          for (int m = 0; m < MT; ++m) {
            const uint4 xv = *reinterpret_cast<const uint4*>(s_x + static_cast<size_t>(m) * Kp + 64 * c + 16 * t);
            acc[m][0] = dp4a_us(f0, static_cast<int>(xv.x), acc[m][0]);
            acc[m][1] = dp4a_us(f1, static_cast<int>(xv.y), acc[m][1]);
            acc[m][2] = dp4a_us(f2, static_cast<int>(xv.z), acc[m][2]);
            acc[m][3] = dp4a_us(f3, static_cast<int>(xv.w), acc[m][3]);
          }
        }
      }
    } else {
      // any K % 4 == 0: one packed byte (4 codes) at a time
      for (int j = lane; j < rowbytes; j += 32) {
        const uint32_t byte = row[j];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int f = static_cast<int>((byte >> (2 * i)) & 3u);
          const int pk = perm_index(4 * j + i);
#pragma unroll
          for (int m = 0; m < MT; ++m)
            acc[m][0] += f * static_cast<int>(static_cast<int8_t>(s_x[static_cast<size_t>(m) * Kp + pk]));
        }
      }
    }

    int tot[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      int v = acc[m][0] + (acc[m][1] >> 2) + (acc[m][2] >> 4) + (acc[m][3] >> 6);
      tot[m] = warp_sum(v);
    }
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      if (lane == m && m < mcount) {
        const int a = tot[m] - s_rowsum[m];
        const size_t o = static_cast<size_t>(m0 + m) * N + n;
        if (OUT == GemvOut::kY) {
          static_cast<float*>(out)[o] = rescale(a, g, scale[m0 + m]);
        } else {
          static_cast<int32_t*>(out)[o] = a;
        }
      }
    }
  }
}

cudaError_t launch_gemv(const uint8_t* wp, const int8_t* xq, const float* scale, const float* gamma, void* out,
                        int M, int N, int K, GemvOut mode, bool vec, int mt, int grid_x, cudaStream_t s) {
  using Fn = void (*)(const uint8_t*, const int8_t*, const float*, const float*, void*, int, int, int);
  Fn fn = nullptr;
#define BL_PICK(MT)                                                                                   \
  if (mode == GemvOut::kY) fn = vec ? bl_gemv_w2a8<MT, true, GemvOut::kY> : bl_gemv_w2a8<MT, false, GemvOut::kY>; \
  else fn = vec ? bl_gemv_w2a8<MT, true, GemvOut::kAcc> : bl_gemv_w2a8<MT, false, GemvOut::kAcc>;
  if (mt == 1) { BL_PICK(1) } else if (mt == 2) { BL_PICK(2) } else { BL_PICK(4) }
#undef BL_PICK
  const int Kp = (K + 63) & ~63;
  const size_t smem = static_cast<size_t>(mt) * Kp;
  const cudaError_t e = ensure_smem(reinterpret_cast<const void*>(fn), smem);
  if (e != cudaSuccess) return e;
  dim3 grid(grid_x, (M + mt - 1) / mt);
  return launch_pdl(fn, grid, dim3(kGemvThreads), smem, s, wp, xq, scale, gamma, out, M, N, K);
}

}  // namespace bl
