// Allocation-free split-KV forward.
//
// attn_fwd_split needs a scratch buffer for the partial results of its key
// ranges, which the caller normally allocates.  Some callers cannot allocate
// device memory at the moment they call us -- for example a plugin running
// inside a host application that manages all device memory through its own
// pool and hands plugins no allocator, or a latency-critical loop that cannot
// afford cudaMalloc's implicit device synchronisation and unbounded cost.
// attn_fwd_split_noalloc serves them: its scratch is the fixed array below,
// which the library declares in device memory, so a call allocates nothing.
//
// Limits and sharing rules (also stated in include/attn_fa2.h):
//  * the array holds kNoAllocScratchBytes (64 MiB); larger plans are rejected;
//  * CUDA loads this file's device code onto a device lazily, so the first
//    call on a device is what commits the array there (and can fail with out
//    of memory); it also looks up the array's device address, once per device,
//    with that device current -- make that first call at set-up time, before
//    any stream capture; the device then keeps the array until exit;
//  * the address is cached per device ordinal, so cudaDeviceReset on a device
//    while the library is in use there is not supported;
//  * all calls share the array and it keeps the last call's contents; every
//    byte a call reads it has written first, so nothing needs clearing; calls
//    whose work overlaps on the GPU race on the array and must be serialised.
#include <cstddef>
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "attn_fa2.h"

namespace attn {
int set_last_error(int status, const char* msg);  // attn_api.cu
}

namespace {

constexpr size_t kNoAllocScratchBytes = static_cast<size_t>(64) << 20;

// Split-KV partial O / L of attn_fwd_split_noalloc (see the file comment).
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of g_noalloc_scratch on the current device.  In host code the
// name g_noalloc_scratch is only a host-side stand-in, never a device address.
int scratch_address(void** out) {
  constexpr int kMaxDev = 64;
  static void* cache[kMaxDev] = {};
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return attn::set_last_error(ATTN_ERR_CUDA, cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDev) return attn::set_last_error(ATTN_ERR_UNSUPPORTED, "device ordinal out of range");
  std::lock_guard<std::mutex> lock(mu);
  if (!cache[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return attn::set_last_error(ATTN_ERR_CUDA, cudaGetErrorString(e));
    cache[dev] = p;
  }
  *out = cache[dev];
  return ATTN_OK;
}

}  // namespace

extern "C" int attn_fwd_split_noalloc(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                                      int N, int d, float scale, float q_descale, float k_descale, float v_descale,
                                      int causal, int dtype, int n_splits, void* stream) {
  int splits = 0;
  size_t need = 0;
  int st = attn_fwd_split_plan(B, H, N, d, n_splits, &splits, &need);
  if (st != ATTN_OK) return st;
  if (need > kNoAllocScratchBytes)
    return attn::set_last_error(ATTN_ERR_UNSUPPORTED,
                                "this split needs more scratch than the built-in 64 MiB array holds; "
                                "use fewer splits or attn_fwd_split with your own workspace");
  void* scratch = nullptr;
  if ((st = scratch_address(&scratch)) != ATTN_OK) return st;
  return attn_fwd_split(q, k, v, o, lse, B, H, N, d, scale, q_descale, k_descale, v_descale, causal, dtype,
                        n_splits, scratch, kNoAllocScratchBytes, stream);
}
