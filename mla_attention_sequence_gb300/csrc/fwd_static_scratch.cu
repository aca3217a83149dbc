// laga_mla_fwd_noalloc: the forward pass for callers that cannot allocate
// device memory (and so cannot hand the library a workspace).
//
// Some callers cannot call cudaMalloc or reach an allocator: a plug-in whose
// host framework owns every byte of device memory through its own pool, a
// runtime with a fixed memory budget set before it starts, a C caller with no
// allocator of its own. For them this entry point keeps the forward's scratch
// -- the per-head K_nope and V the reconstruction GEMM writes and the
// attention kernel reads back -- in one file-scope device array instead of a
// caller workspace.
//
// The array is a module global: every GPU that loads the library holds
// kNoallocScratchBytes of it until the process exits. All calls on a device
// share it and it keeps the last call's contents; nothing in it needs to start
// at zero, because the reconstruction GEMM writes every row the attention
// kernel reads. Calls whose kernels overlap on the GPU (different streams, or
// different host threads) race on it; serialise them.
#include "../../include/laga_mla.h"
#include "internal.h"

#include <cstdio>
#include <mutex>

namespace laga {
namespace {

constexpr size_t kNoallocScratchBytes = static_cast<size_t>(LAGA_NOALLOC_SCRATCH_BYTES);

__device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

// Device address of g_noalloc_scratch on the current device. In host code the
// symbol's name is only a host-side handle, so the address is looked up once
// per device (with that device current) and cached together with the context
// it was looked up in: should the caller reset the device, the new primary
// context loads the module afresh and the array may sit elsewhere, so the
// address is looked up again.
cudaError_t scratch_address(void** out) {
  static void* addr[64] = {};
  static void* ctxs[64] = {};
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  void* ctx = current_context();
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev] || ctxs[dev] != ctx) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    addr[dev] = p;
    ctxs[dev] = ctx;
  }
  *out = addr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace laga

extern "C" laga_status laga_mla_fwd_noalloc(const laga_mla_desc* desc, const void* q, const void* c_kv,
                                            const void* k_rope, const void* W_UK, const void* W_UV, void* out,
                                            float* lse, laga_stream_t stream) {
  const size_t need = laga_mla_fwd_workspace_size(desc);
  if (need > laga::kNoallocScratchBytes) {
    // laga_mla_fwd reports its own argument errors; this one is the size limit.
    char msg[160];
    std::snprintf(msg, sizeof(msg), "scratch for this problem is %zu bytes, above the %zu-byte static array",
                  need, laga::kNoallocScratchBytes);
    laga::set_last_error(msg);
    return LAGA_ERR_WORKSPACE;
  }
  void* scratch = nullptr;
  if (need > 0) {
    const cudaError_t e = laga::scratch_address(&scratch);
    if (e != cudaSuccess) {
      char msg[160];
      std::snprintf(msg, sizeof(msg), "cudaGetSymbolAddress(static scratch): %s", cudaGetErrorString(e));
      laga::set_last_error(msg);
      return LAGA_ERR_CUDA;
    }
  }
  return laga_mla_fwd(desc, q, c_kv, k_rope, W_UK, W_UV, out, lse, scratch, need, stream);
}
