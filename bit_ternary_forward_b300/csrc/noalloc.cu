// Weight packing for callers that cannot allocate device memory.
//
// bitlinear_pack_weights needs a small scratch buffer for the exact absmean
// (one fixed-point partial sum per CTA). Some callers have no way to provide
// one: code that runs where cudaMalloc is forbidden or unavailable, such as a
// plugin inside a host framework whose caching allocator owns all device
// memory and must not be bypassed, or a runtime that has reserved the whole
// device up front. For them this file keeps the scratch in a
// file-scope __device__ array that the CUDA module holds from the moment the
// library is loaded on a device until the process exits, and passes its
// device address to the ordinary packing path.

#include <cstdio>

#include "bitlinear.h"
#include "kernels.cuh"

namespace {

// Scratch of the exact-sum partials: one 64-byte slot per CTA of the absmean
// kernel, at most bl::kMaxAbsumCtas slots (75,776 bytes).
constexpr size_t kScratchWords = static_cast<size_t>(bl::kMaxAbsumCtas) * bl::kPartialWords;
__device__ __align__(256) uint32_t g_pack_scratch[kScratchWords];

// Device address of g_pack_scratch on the current device. In host code the
// name g_pack_scratch is only a host-side shadow, so the address must come
// from cudaGetSymbolAddress with the device current. It is looked up on every
// call (a cheap table lookup in the runtime once the module is loaded), so no
// address outlives a device reset and nothing is shared between host threads.
bl_status scratch_address(void** out, const char** why) {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_pack_scratch);
  if (e != cudaSuccess || !p) {
    *why = e != cudaSuccess ? cudaGetErrorString(e) : "cudaGetSymbolAddress returned NULL";
    return BL_ERR_CUDA;
  }
  *out = p;
  return BL_OK;
}

}  // namespace

extern "C" bl_status bitlinear_pack_weights_noalloc(const float* W, int64_t N, int64_t K, uint8_t* Wp,
                                                    float* gamma, bl_stream_t stream) {
  const size_t need = bitlinear_pack_workspace_bytes(N, K);
  if (need > sizeof(g_pack_scratch)) {
    char msg[256];
    snprintf(msg, sizeof(msg),
             "bitlinear_pack_weights_noalloc: N=%lld K=%lld needs %zu bytes of scratch, more than the "
             "%zu-byte static array holds; use bitlinear_pack_weights with a workspace",
             (long long)N, (long long)K, need, sizeof(g_pack_scratch));
    return bl::record_error(BL_ERR_UNSUPPORTED, msg);
  }
  void* scratch = nullptr;
  const char* why = nullptr;
  if (bl_status st = scratch_address(&scratch, &why)) return bl::record_error(st, why);
  // Every partial slot the kernels read is written earlier in the same call,
  // so the array needs no clearing between calls.
  return bitlinear_pack_weights(W, N, K, Wp, gamma, scratch, sizeof(g_pack_scratch), stream);
}
