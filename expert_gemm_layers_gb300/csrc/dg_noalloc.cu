// dg_tp_swiglu_noalloc: the SwiGLU pair for callers that cannot allocate
// device memory (see include/dg.h).  Its scratch -- the h activations
// between the two GEMMs -- lives in a fixed-size array compiled into the
// library, so the call needs no workspace argument and never allocates.
// Argument checks and the two GEMM launches are those of dg_tp_swiglu.
#include <cuda_runtime.h>

#include <mutex>

#include "dg_internal.h"

namespace dg {
namespace {

// Upper bound on h = [rows, ffn] bf16 for this entry point: 32 MiB.
constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;

// The scratch itself.  Every device that loads the library holds one copy
// until the process exits.  In host code this name is only a stand-in for the
// device object; kernels get its device address from cudaGetSymbolAddress.
__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
struct ScratchSlot {
  std::once_flag once;
  void* ptr = nullptr;
  cudaError_t status = cudaSuccess;
};
ScratchSlot g_scratch[kMaxDevices];

// Device address of this device's scratch array, looked up once per device
// with that device current.
dg_status scratch_address(const DeviceInfo& dev, void** out) {
  ScratchSlot& slot = g_scratch[dev.device];
  std::call_once(slot.once, [&] { slot.status = cudaGetSymbolAddress(&slot.ptr, g_noalloc_scratch); });
  if (slot.status != cudaSuccess)
    return fail(DG_ERR_CUDA, "tp_swiglu_noalloc: cudaGetSymbolAddress failed: %s", cudaGetErrorString(slot.status));
  *out = slot.ptr;
  return DG_OK;
}

}  // namespace
}  // namespace dg

using namespace dg;

extern "C" dg_status dg_tp_swiglu_noalloc(int64_t S, int64_t d, int64_t ffn, int32_t W, int32_t bsz,
                                          const void* x_shards, const void* w13, const void* w2, void* y_shards,
                                          void* stream) {
  dg_status st = tp_swiglu_check_sizes(S, d, ffn, W, bsz, "tp_swiglu_noalloc");
  if (st != DG_OK) return st;
  // S*bsz and ffn are below 2^31 here, so the product is exact in 64 bits
  const uint64_t need = static_cast<uint64_t>(S) * static_cast<uint64_t>(bsz) * static_cast<uint64_t>(ffn) * 2u;
  if (need > kNoAllocScratchBytes)
    return fail(DG_ERR_UNSUPPORTED,
                "tp_swiglu_noalloc: h = S*bsz x ffn bf16 needs %llu bytes, more than the built-in %zu-byte scratch; "
                "use dg_tp_swiglu with a caller-provided workspace",
                static_cast<unsigned long long>(need), kNoAllocScratchBytes);
  DeviceInfo dev;
  if ((st = device_info(&dev)) != DG_OK) return st;
  void* h = nullptr;
  if ((st = scratch_address(dev, &h)) != DG_OK) return st;
  // The scratch must not alias a caller tensor (it cannot, being library
  // memory, unless a caller passes pointers into it).
  if ((st = tp_swiglu_check(S, d, ffn, W, bsz, x_shards, w13, w2, y_shards, h, kNoAllocScratchBytes,
                            "tp_swiglu_noalloc")) != DG_OK)
    return st;
  dev.err = dev.builtin_err;  // failures go to the library's own error word
  return tp_swiglu_enqueue(S, d, ffn, W, bsz, x_shards, w13, w2, y_shards, h, dev, static_cast<cudaStream_t>(stream),
                           false);
}
