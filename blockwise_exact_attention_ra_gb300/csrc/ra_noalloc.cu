// ra_ring_fwd_noalloc: the ring forward for callers that cannot allocate
// device memory (see include/ra.h).  The scratch that ra_ring_fwd takes as a
// caller workspace (its unit counter and, for bf16 inputs, the fp16 copy of
// V) lives here in a fixed, file-scope device array instead.
#include <cuda_runtime.h>
#include <stdio.h>

#include <mutex>

#include "ra_internal.h"

namespace {

constexpr size_t kVBytes = size_t(32) << 20;         // room for the fp16 V copy
constexpr size_t kScratchBytes = 256 + kVBytes;       // + the unit counter, per device

// One copy per device that loads the library; it lives until the process
// exits.  In host code `g_noalloc_scratch` names a host-side stand-in, not a
// device address: only the pointer from cudaGetSymbolAddress may be passed
// to kernels.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

}  // namespace

extern "C" {
#pragma GCC visibility push(default)

int ra_ring_fwd_noalloc(const void* q, const void* k, const void* v, ra_dtype dtype,
                        ra_shape shape, int P, int flags, float scale, void* o,
                        ra_dtype o_dtype, float* lse, void* stream) {
  // The extents are checked before the scratch size is formed from them, so
  // that no product of out-of-range extents can wrap around to a small size.
  if (shape.B < 1 || shape.N_kv < 1 || shape.Hkv < 1 || shape.d < 1 || shape.N_kv >= (1 << 30) ||
      shape.Hkv > 4096 || shape.d > 4096)
    return ra::set_error(RA_ERR_INVALID_ARG, "ra_ring_fwd_noalloc: key/value extents out of range");
  // B * N_kv * Hkv * d * 2 bytes, compared without overflow: B < 2^31 and
  // N_kv * Hkv * d * 2 < 2^55
  const unsigned long long per_batch = (unsigned long long)shape.N_kv * shape.Hkv * shape.d * 2ull;
  const bool too_big = dtype == RA_BF16 && (unsigned long long)shape.B > kVBytes / per_batch;
  const size_t need = too_big ? 0 : ra_ring_fwd_workspace_bytes(dtype, shape, P);
  if (too_big || need > kScratchBytes) {
    char msg[256];
    if (too_big)
      snprintf(msg, sizeof msg,
               "ra_ring_fwd_noalloc: this shape needs more scratch than the built-in buffer holds "
               "(%zu bytes); call ra_ring_fwd with a workspace instead",
               kScratchBytes);  // only bf16 shapes need more than the counter
    else
      snprintf(msg, sizeof msg,
               "ra_ring_fwd_noalloc: this shape needs %zu bytes of scratch but the built-in buffer "
               "holds %zu; call ra_ring_fwd with a workspace instead",
               need, kScratchBytes);
    return ra::set_error(RA_ERR_INVALID_ARG, msg);
  }
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return ra::set_error(RA_ERR_CUDA, "ra_ring_fwd_noalloc: no usable current device");
  void* scratch = nullptr;
  {
    // set-up, once per device, with that device current
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_scratch_ptr[dev]) {
      void* p = nullptr;
      const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
      if (e != cudaSuccess || !p) {
        char msg[256];
        snprintf(msg, sizeof msg, "ra_ring_fwd_noalloc: cudaGetSymbolAddress(scratch) failed: %s",
                 cudaGetErrorString(e));
        return ra::set_error(RA_ERR_CUDA, msg);
      }
      g_scratch_ptr[dev] = p;
    }
    scratch = g_scratch_ptr[dev];
  }
  return ra_ring_fwd(q, k, v, dtype, shape, P, flags, scale, o, o_dtype, lse, scratch,
                     kScratchBytes, stream);
}

#pragma GCC visibility pop
}  // extern "C"
