// mbarrier and bulk asynchronous copy helpers (sm_90 and later PTX), shared by
// the kernels that stage global memory through shared memory.
//
// Every wait is bounded: a kernel that gives up records it in its own error
// word, which the host reads through bitlinear_device_error().
#pragma once

#include <cstdint>

#include "common.cuh"

namespace bl {

// Number of suspended try_wait calls before a wait gives up. Each call ends by
// itself after a hardware time limit, so the bound is in time, not in polls.
constexpr uint32_t kWaitTries = 1u << 16;

BL_DEVICE uint32_t smem_u32(const void* p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }

BL_DEVICE void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// Makes barrier initialisation visible to the async proxy (bulk copies).
BL_DEVICE void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

BL_DEVICE void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}

BL_DEVICE void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// One suspended wait on the phase of the given parity.
BL_DEVICE bool mbar_try(uint64_t* bar, uint32_t phase) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(phase)
      : "memory");
  return ok != 0u;
}

// Bounded wait: true once the phase completed, false after kWaitTries
// suspended waits, so a lost arrival cannot hang the kernel.
BL_DEVICE bool mbar_wait(uint64_t* bar, uint32_t phase) {
  for (uint32_t i = 0; i < kWaitTries; ++i)
    if (mbar_try(bar, phase)) return true;
  return false;
}

// One wait that may suspend the thread for up to kSleepNs before it gives up
// (it resumes as soon as the phase completes), for consumers that would
// otherwise poll for a long time while a copy is in flight.
constexpr uint32_t kSleepNs = 20000;
constexpr uint32_t kSleepTries = 1u << 14;   // a wait gives up after at most ~0.33 s
BL_DEVICE bool mbar_try_sleep(uint64_t* bar, uint32_t phase) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(phase), "n"(kSleepNs)
      : "memory");
  return ok != 0u;
}
BL_DEVICE bool mbar_wait_sleep(uint64_t* bar, uint32_t phase) {
  for (uint32_t i = 0; i < kSleepTries; ++i)
    if (mbar_try_sleep(bar, phase)) return true;
  return false;
}

// Global -> shared bulk copy completing on an mbarrier (both addresses 16-byte
// aligned, bytes a multiple of 16).
BL_DEVICE void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Moves `bytes` (a multiple of 16, 16-byte aligned source) of global memory
// into L2 ahead of use. A prefetch returns no data and L2 is the point of
// coherence, so it cannot change what a later load sees: a kernel may issue it
// before its dependency wait, while the kernel before it is still writing.
BL_DEVICE void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// L2 prefetches of [p, p + bytes) in pieces of at most 32 KB.
BL_DEVICE void prefetch_l2_range(const void* p, uint64_t bytes) {
  const uint8_t* b = static_cast<const uint8_t*>(p);
  for (uint64_t off = 0; off < bytes; off += 32768)
    prefetch_l2(b + off, static_cast<uint32_t>(bytes - off < 32768 ? bytes - off : 32768));
}

// L2 eviction-priority policies for cache-hinted copies.
BL_DEVICE uint64_t l2_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
BL_DEVICE uint64_t l2_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// bulk_copy_g2s with an L2 eviction-priority policy for the source lines.
BL_DEVICE void bulk_copy_g2s_hint(void* dst, const void* src, uint32_t bytes, uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// Producer of a ring of `stages` shared-memory stages of `stage_bytes` each,
// run by one thread: streams `bytes` (a multiple of 16) from `src`, stage j of
// the stream into slot j % stages once the consumers have released the
// slot's previous use (empty[slot] completes on one arrival per consumer
// warp); the copy completes full[slot]. Consumers wait on full[j % stages]
// with parity (j / stages) & 1. Returns false if a wait gave up; every copy
// issued has landed when it returns, so the CTA may then exit. The source
// lines are read with the L2 policy `policy`.
BL_DEVICE bool ring_produce(void* ring, uint32_t stage_bytes, int stages, const void* src, uint64_t bytes,
                            uint64_t* full, uint64_t* empty, uint64_t policy) {
  const int n = static_cast<int>((bytes + stage_bytes - 1) / stage_bytes);
  uint8_t* dst = static_cast<uint8_t*>(ring);
  const uint8_t* from = static_cast<const uint8_t*>(src);
  bool ok = true;
  int j = 0;
  for (; j < n; ++j) {
    const int s = j % stages;
    if (j >= stages && !mbar_wait(&empty[s], ((j / stages) - 1) & 1)) {
      ok = false;
      break;
    }
    const uint64_t off = static_cast<uint64_t>(j) * stage_bytes;
    const uint32_t len = static_cast<uint32_t>(min(bytes - off, static_cast<uint64_t>(stage_bytes)));
    mbar_expect_tx(&full[s], len);
    bulk_copy_g2s_hint(dst + static_cast<size_t>(s) * stage_bytes, from + off, len, &full[s], policy);
  }
  for (int k = max(0, j - stages); k < j; ++k)
    if (!mbar_wait(&full[k % stages], (k / stages) & 1)) ok = false;
  return ok;
}

}  // namespace bl
