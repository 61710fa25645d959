// fa_bwd_noalloc: the backward for callers that cannot allocate device
// memory.  Its scratch is a fixed array in this translation unit alone: the
// library is built without relocatable device code, so this file is a module
// of its own, which the CUDA runtime loads (and whose array it reserves on a
// device) only when a process first looks the array up, i.e. on its first
// fa_bwd_noalloc call.  Processes that never call it do not hold the array.
#include <mutex>

#include <cuda_runtime.h>

#include "fa.h"

namespace fa {
namespace {

// The backward's D and fp32 dQ accumulator for callers that cannot allocate.
// Fixed size, one per device, shared by every call.
static __device__ __align__(256) unsigned char g_noalloc_scratch[FA_NOALLOC_SCRATCH_BYTES];

// Device address of g_noalloc_scratch for the current device.  Host code may
// not pass the array's name to a kernel (on the host it names a host-side
// stand-in), so the address is looked up once per device, with that device
// current, and cached.
void* noalloc_scratch_ptr() {
  static std::mutex mu;
  static void* ptrs[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!ptrs[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
    ptrs[dev] = p;
  }
  return ptrs[dev];
}

}  // namespace
}  // namespace fa

extern "C" int fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                              const float* lse, const void* dout, void* dq, void* dk, void* dv,
                              int B, int H, int N, int d, float scale, int causal, void* stream) {
  // 0 bytes: an empty problem (a no-op) or an invalid or unsupported shape;
  // fa_bwd returns the matching status without touching any workspace.
  const size_t need = fa_bwd_workspace_bytes(B, H, N, d);
  if (need == 0)
    return fa_bwd(q, k, v, o, lse, dout, dq, dk, dv, B, H, N, d, scale, causal, nullptr, 0,
                  stream);
  if (need > FA_NOALLOC_SCRATCH_BYTES) return FA_ERR_TOO_LARGE;
  if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv) return FA_ERR_INVALID_ARG;
  void* scratch = fa::noalloc_scratch_ptr();
  if (!scratch) return FA_ERR_CUDA;
  // fa_bwd's first kernel zeroes the dQ accumulator and overwrites D, so the
  // previous call's contents of the scratch do not matter.
  return fa_bwd(q, k, v, o, lse, dout, dq, dk, dv, B, H, N, d, scale, causal, scratch,
                FA_NOALLOC_SCRATCH_BYTES, stream);
}
