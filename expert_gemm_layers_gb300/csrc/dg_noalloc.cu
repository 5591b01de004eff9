// dg_tp_swiglu_noalloc: the SwiGLU pair for callers that cannot allocate
// device memory (see include/dg.h).  Its scratch -- the h activations
// between the two GEMMs -- lives in a fixed-size array compiled into the
// library, so the call needs no workspace argument and never allocates.
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

// One launch of a GEMM variant without the tracing hook (tracing records CUDA
// events, which this entry point must not create).
dg_status launch_untraced(GemmVariant v, const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& d,
                          GemmParams p, const DeviceInfo& dev, cudaStream_t s) {
  p.tiles_m = (p.M + gemm_tile_m() - 1) / gemm_tile_m();
  p.tiles_n = (p.N + gemm_tile_n(v) - 1) / gemm_tile_n(v);
  p.err = dev.err;
  const int64_t tiles = static_cast<int64_t>(p.G) * p.tiles_m * p.tiles_n;
  if (tiles == 0) return DG_OK;
  cudaError_t e = v == GV_BF16_KK_SWIGLU ? launch_gemm_bf16_kk_swiglu(a, b, d, d, p, dev.num_sms, s)
                                         : launch_gemm_bf16_kk_store(a, b, d, d, p, dev.num_sms, s);
  if (e != cudaSuccess) return fail(DG_ERR_CUDA, "tp_swiglu_noalloc: GEMM launch: %s", cudaGetErrorString(e));
  return DG_OK;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace dg

using namespace dg;

extern "C" dg_status dg_tp_swiglu_noalloc(int64_t S, int64_t d, int64_t ffn, int32_t W, int32_t bsz,
                                          const void* x_shards, const void* w13, const void* w2, void* y_shards,
                                          void* stream) {
  if (S < 1 || d < 1 || ffn < 1 || W < 1 || bsz < 1)
    return fail(DG_ERR_INVALID_ARGUMENT, "tp_swiglu_noalloc: S, d, ffn, W, bsz must be >= 1");
  if (S % W || ffn % W) return fail(DG_ERR_INVALID_ARGUMENT, "tp_swiglu_noalloc: S and ffn must be divisible by W");
  const int64_t F = ffn / W;
  if (d % 8 || F % 8) return fail(DG_ERR_INVALID_ARGUMENT, "tp_swiglu_noalloc: d and ffn/W must be multiples of 8");
  const int64_t rows = S * bsz;
  const double need = static_cast<double>(rows) * static_cast<double>(ffn) * 2.0;
  if (need > static_cast<double>(kNoAllocScratchBytes))
    return fail(DG_ERR_UNSUPPORTED,
                "tp_swiglu_noalloc: h = S*bsz x ffn bf16 needs %.0f bytes, more than the built-in %zu-byte scratch; "
                "use dg_tp_swiglu with a caller-provided workspace",
                need, kNoAllocScratchBytes);
  if (!x_shards || !w13 || !w2 || !y_shards)
    return fail(DG_ERR_INVALID_ARGUMENT, "tp_swiglu_noalloc: NULL tensor pointer");
  if (!aligned16(x_shards) || !aligned16(w13) || !aligned16(w2) || !aligned16(y_shards))
    return fail(DG_ERR_INVALID_ARGUMENT, "tp_swiglu_noalloc: tensors must be 16-byte aligned");
  const size_t act = static_cast<size_t>(rows) * d * 2;
  const uintptr_t xa = reinterpret_cast<uintptr_t>(x_shards), ya = reinterpret_cast<uintptr_t>(y_shards);
  if (xa < ya + act && ya < xa + act) return fail(DG_ERR_INVALID_ARGUMENT, "tp_swiglu_noalloc: y_shards overlaps x_shards");
  DeviceInfo dev;
  dg_status st = device_info(&dev);
  if (st != DG_OK) return st;
  void* h = nullptr;
  if ((st = scratch_address(dev, &h)) != DG_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const uint64_t R = rows, Dm = d, Fu = F, Wu = W, FF = ffn;

  // GEMM1 over all shards into h (the scratch array): h[:, s*F + c] = silu(X w1_s[c]) * (X w3_s[c]).
  CUtensorMap mx, mw13, mh;
  if ((st = make_map_3d(&mx, true, x_shards, Dm, R, 1, Dm * 2, R * Dm * 2, 64, 128, 1, "x_shards")) != DG_OK) return st;
  if ((st = make_map_3d(&mw13, true, w13, Dm, Fu, 2 * Wu, Dm * 2, Fu * Dm * 2, 64, 128, 1, "w13")) != DG_OK) return st;
  if ((st = make_map_3d(&mh, true, h, Fu, Wu, R, Fu * 2, FF * 2, 64, 1, 32, "h")) != DG_OK) return st;
  GemmParams p{};
  p.G = W;
  p.M = static_cast<int32_t>(R);
  p.N = static_cast<int32_t>(F);
  p.K = static_cast<int32_t>(d);
  p.a_g = G_NONE;
  p.b_g = G_OUTER;
  p.d_g = G_MID;
  if ((st = launch_untraced(GV_BF16_KK_SWIGLU, mx, mw13, mh, p, dev, s)) != DG_OK) return st;

  // GEMM2: y = h @ w2^T, the shard sum being the K loop.
  CUtensorMap mh_k, mw2, my;
  if ((st = make_map_3d(&mh_k, true, h, FF, R, 1, FF * 2, R * FF * 2, 64, 128, 1, "h (A)")) != DG_OK) return st;
  if ((st = make_map_3d(&mw2, true, w2, FF, Dm, 1, FF * 2, Dm * FF * 2, 64, kKMajorBRows, 1, "w2")) != DG_OK) return st;
  if ((st = make_map_3d(&my, true, y_shards, Dm, R, 1, Dm * 2, R * Dm * 2, 64, 32, 1, "y_shards")) != DG_OK) return st;
  p = GemmParams{};
  p.G = 1;
  p.M = static_cast<int32_t>(R);
  p.N = static_cast<int32_t>(d);
  p.K = static_cast<int32_t>(ffn);
  p.a_g = G_OUTER;
  p.b_g = G_OUTER;
  p.d_g = G_OUTER;
  return launch_untraced(GV_BF16_KK_STORE, mh_k, mw2, my, p, dev, s);
}
