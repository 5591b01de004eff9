// The C ABI of libdg (include/dg.h): argument validation, TMA tensor maps,
// scratch carving and the launch sequence of each operation.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdarg.h>
#include <stdio.h>

#include <mutex>
#include <string>
#include <string.h>
#include <vector>

#include "dg_internal.h"

namespace dg {

// The library's own error word, one per device.  Only the call that takes no
// workspace (dg_tp_swiglu_noalloc) records its failures here; every other call
// uses the error block at the start of its caller's workspace.
__device__ uint32_t g_builtin_error_word;

namespace {

thread_local char t_last_error[512] = "";

constexpr int kMaxDevices = 64;
struct DeviceSlot {
  std::once_flag once;
  DeviceInfo info;
  dg_status status;
};
DeviceSlot g_devices[kMaxDevices];

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

inline size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

dg_status cuda_fail(cudaError_t e, const char* what) {
  return fail(DG_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

}  // namespace

dg_status fail(dg_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(t_last_error, sizeof(t_last_error), fmt, ap);
  va_end(ap);
  return s;
}

namespace {
struct TraceRecord {
  const char* name;
  double flops, bytes;
  cudaEvent_t e0, e1;
};
std::mutex g_trace_mu;
bool g_tracing = false;
std::string g_trace_only;  // record only launches of this name (empty: all)
std::vector<TraceRecord> g_trace;
}  // namespace

TraceScope::TraceScope(const char* name, cudaStream_t s, double flops, double bytes)
    : stream_(s), name_(name), flops_(flops), bytes_(bytes) {
  if (name == nullptr) return;
  {
    std::lock_guard<std::mutex> g(g_trace_mu);
    if (!g_tracing) return;
    if (!g_trace_only.empty() && g_trace_only != name) return;
  }
  if (cudaEventCreate(&e0_) != cudaSuccess) return;
  if (cudaEventCreate(&e1_) != cudaSuccess) {
    cudaEventDestroy(e0_);
    return;
  }
  cudaEventRecord(e0_, stream_);
  active_ = true;
}

TraceScope::~TraceScope() {
  if (!active_) return;
  cudaEventRecord(e1_, stream_);
  std::lock_guard<std::mutex> g(g_trace_mu);
  g_trace.push_back(TraceRecord{name_, flops_, bytes_, e0_, e1_});
}

dg_status device_info(DeviceInfo* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(DG_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
  // Bind the device's primary context to this thread: driver-API calls such as
  // tensor-map encoding need a current context, which a fresh thread (an
  // autograd worker, say) does not have until a runtime call creates it.
  e = cudaSetDevice(dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaSetDevice");
  DeviceSlot& slot = g_devices[dev];
  std::call_once(slot.once, [&] {
    slot.status = DG_OK;
    slot.info.device = dev;
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&slot.info.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      slot.status = DG_ERR_CUDA;
      return;
    }
    if (major != 10 || minor != 3) {
      slot.status = DG_ERR_UNSUPPORTED;
      return;
    }
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_builtin_error_word) != cudaSuccess) {
      slot.status = DG_ERR_CUDA;
      return;
    }
    slot.info.builtin_err = static_cast<uint32_t*>(p);
    slot.info.err = nullptr;
  });
  if (slot.status == DG_ERR_UNSUPPORTED)
    return fail(DG_ERR_UNSUPPORTED, "device %d is not sm_103 (this library is built for sm_103a only)", dev);
  if (slot.status != DG_OK) return fail(slot.status, "device %d: attribute or symbol query failed", dev);
  *out = slot.info;
  return DG_OK;
}

dg_status device_info_ws(DeviceInfo* dev, void* ws, size_t ws_bytes, const char* what) {
  dg_status st = check_error_block(ws, ws_bytes, what);
  if (st != DG_OK) return st;
  if ((st = device_info(dev)) != DG_OK) return st;
  dev->err = static_cast<uint32_t*>(ws);
  return DG_OK;
}

dg_status check_error_block(const void* ws, size_t ws_bytes, const char* what) {
  if (!ws)
    return fail(DG_ERR_WORKSPACE, "%s: ws is NULL (its first %d bytes are the call's error block)", what,
                DG_ERROR_BLOCK_BYTES);
  if (!aligned16(ws)) return fail(DG_ERR_INVALID_ARGUMENT, "%s: ws is not 16-byte aligned", what);
  if (ws_bytes < static_cast<size_t>(DG_ERROR_BLOCK_BYTES))
    return fail(DG_ERR_WORKSPACE, "%s: workspace has %zu bytes, less than the %d-byte error block", what, ws_bytes,
                DG_ERROR_BLOCK_BYTES);
  return DG_OK;
}

dg_status make_map_3d(CUtensorMap* map, bool is_bf16, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                      uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t b0, uint32_t b1, uint32_t b2,
                      const char* what) {
  return make_map_3d_sw(map, is_bf16, base, d0, d1, d2, stride1_bytes, stride2_bytes, b0, b1, b2, 128, what);
}

dg_status make_map_3d_sw(CUtensorMap* map, bool is_bf16, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                         uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t b0, uint32_t b1, uint32_t b2,
                         int swizzle_bytes, const char* what) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return fail(DG_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  if (!aligned16(base)) return fail(DG_ERR_INVALID_ARGUMENT, "%s: base address must be 16-byte aligned", what);
  if ((stride1_bytes & 15u) || (stride2_bytes & 15u))
    return fail(DG_ERR_INVALID_ARGUMENT, "%s: row strides must be multiples of 16 bytes", what);
  if (d0 == 0 || d1 == 0 || d2 == 0) return fail(DG_ERR_INVALID_ARGUMENT, "%s: empty dimension", what);
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {stride1_bytes, stride2_bytes};
  const cuuint32_t box[3] = {b0, b1, b2};
  const cuuint32_t estr[3] = {1, 1, 1};
  if (swizzle_bytes != 64 && swizzle_bytes != 128) return fail(DG_ERR_INVALID_ARGUMENT, "%s: swizzle", what);
  CUresult r = enc(map, is_bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 3,
                   const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   swizzle_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(DG_ERR_INVALID_ARGUMENT, "%s: tensor map rejected (CUresult %d)", what, (int)r);
  return DG_OK;
}

dg_status make_map_mn(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                      uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t b1, uint32_t b2, uint32_t blocks,
                      int32_t* mn4, const char* what) {
  *mn4 = 0;
  if (d0 % 64 == 0 && d1 > 0 && d2 > 0 && aligned16(base) && !(stride1_bytes & 15u) && !(stride2_bytes & 15u)) {
    EncodeTiledFn enc = encode_fn();
    if (enc) {
      const cuuint64_t dims[4] = {64, d1, d2, d0 / 64};
      const cuuint64_t strides[3] = {stride1_bytes, stride2_bytes, 128};
      const cuuint32_t box[4] = {64, b1, b2, blocks};
      const cuuint32_t estr[4] = {1, 1, 1, 1};
      CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
                       CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
      if (r == CUDA_SUCCESS) {
        *mn4 = 1;
        return DG_OK;
      }
    }
  }
  return make_map_3d(map, true, base, d0, d1, d2, stride1_bytes, stride2_bytes, 64, b1, b2, what);
}

int gemm_tile_m() { return kUsePairs ? 256 : 128; }

int gemm_tile_n(GemmVariant v) { return v == GV_BF16_KK_SWIGLU ? 128 : v == GV_FP8_KK_N224 ? 224 : 256; }

dg_status run_gemm(GemmVariant v, const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& d,
                   const CUtensorMap& c, GemmParams p, const DeviceInfo& dev, cudaStream_t s, const char* name,
                   double bytes) {
  p.tiles_m = (p.M + gemm_tile_m() - 1) / gemm_tile_m();
  p.tiles_n = (p.N + gemm_tile_n(v) - 1) / gemm_tile_n(v);
  // Tile order within a problem: along the longer side fastest, so the tiles
  // that share a panel of the larger operand run on neighbouring CTA pairs at
  // the same time (measured on every FFN and TP launch of the benchmark).
  p.n_fastest = p.tiles_n < p.tiles_m ? 1 : 0;
  if (dev.err == nullptr) return fail(DG_ERR_INVALID_ARGUMENT, "internal: GEMM launch without an error word");
  p.err = dev.err;
  const int64_t tiles = static_cast<int64_t>(p.G) * p.tiles_m * p.tiles_n;
  if (tiles == 0) return DG_OK;
  if (tiles > 0x7fffffff) return fail(DG_ERR_UNSUPPORTED, "too many output tiles (%lld)", (long long)tiles);
  const int grid = dev.num_sms;
  const double n_mma = v == GV_BF16_KK_SWIGLU ? 2.0 * p.N : static_cast<double>(p.N);
  TraceScope trace(name, s, 2.0 * p.G * static_cast<double>(p.M) * n_mma * p.K, bytes);
  cudaError_t e;
  switch (v) {
    case GV_FP8_KK: e = launch_gemm_fp8_kk(a, b, d, c, p, grid, s); break;
    case GV_BF16_KK_STORE: e = launch_gemm_bf16_kk_store(a, b, d, c, p, grid, s); break;
    case GV_BF16_KM_BIAS: e = launch_gemm_bf16_km_bias(a, b, d, c, p, grid, s); break;
    case GV_BF16_MM_STORE: e = launch_gemm_bf16_mm_store(a, b, d, c, p, grid, s); break;
    case GV_BF16_KK_SWIGLU: e = launch_gemm_bf16_kk_swiglu(a, b, d, c, p, grid, s); break;
    case GV_BF16_KM_LNSTATS: e = launch_gemm_bf16_km_lnstats(a, b, d, c, p, grid, s); break;
    case GV_BF16_KM_STORE: e = launch_gemm_bf16_km_store(a, b, d, c, p, grid, s); break;
    case GV_FP8_KK_N224: e = launch_gemm_fp8_kk_n224(a, b, d, c, p, grid, s); break;
    case GV_BF16_KK_BIAS: e = launch_gemm_bf16_kk_bias(a, b, d, c, p, grid, s); break;
    case GV_FP8_KK_LNSTATS: e = launch_gemm_fp8_kk_lnstats(a, b, d, c, p, grid, s); break;
    case GV_FP8_KK_BIAS: e = launch_gemm_fp8_kk_bias(a, b, d, c, p, grid, s); break;
    default: return fail(DG_ERR_UNSUPPORTED, "unknown GEMM variant");
  }
  if (e != cudaSuccess) return cuda_fail(e, "GEMM launch");
  return DG_OK;
}

dg_status run_gemm_gated(const CUtensorMap& b, const CUtensorMap& d, const CUtensorMap& z, GemmParams p,
                         const GateSrc& q, const DeviceInfo& dev, cudaStream_t s, const char* name, double bytes) {
  p.tiles_m = (p.M + gemm_tile_m() - 1) / gemm_tile_m();
  p.tiles_n = (p.N + gemm_gated_tile_n() - 1) / gemm_gated_tile_n();
  // The column passes of one row block on neighbouring pairs: they read the
  // same rows of Z at about the same time.
  p.n_fastest = 1;
  if (dev.err == nullptr) return fail(DG_ERR_INVALID_ARGUMENT, "internal: GEMM launch without an error word");
  p.err = dev.err;
  const int64_t tiles = static_cast<int64_t>(p.G) * p.tiles_m * p.tiles_n;
  if (tiles == 0) return DG_OK;
  if (tiles > 0x7fffffff) return fail(DG_ERR_UNSUPPORTED, "too many output tiles (%lld)", (long long)tiles);
  TraceScope trace(name, s, 2.0 * p.G * static_cast<double>(p.M) * p.N * p.K, bytes);
  cudaError_t e = launch_gemm_gated(b, d, z, p, q, dev.num_sms, s);
  if (e != cudaSuccess) return cuda_fail(e, "gated GEMM launch");
  return DG_OK;
}

}  // namespace dg

using namespace dg;

namespace {

struct FfnDims {
  int64_t P, B, T, D, k, H, L, M;
};

dg_status check_ffn_shape(const dg_ffn_shape* sh, FfnDims* o) {
  if (!sh) return fail(DG_ERR_INVALID_ARGUMENT, "shape is NULL");
  if (sh->P < 1 || sh->B < 1 || sh->T < 1 || sh->D < 1 || sh->k < 1)
    return fail(DG_ERR_INVALID_ARGUMENT, "shape: P, B, T, D, k must all be >= 1 (got %d, %d, %d, %d, %d)", sh->P,
                sh->B, sh->T, sh->D, sh->k);
  if (sh->T % sh->P) return fail(DG_ERR_INVALID_ARGUMENT, "shape: T %% P != 0 (T=%d, P=%d)", sh->T, sh->P);
  if (sh->D % 8) return fail(DG_ERR_INVALID_ARGUMENT, "shape: D must be a multiple of 8 (16-byte rows), got %d", sh->D);
  if (!(sh->eps > 0.0f)) return fail(DG_ERR_INVALID_ARGUMENT, "shape: eps must be > 0");
  o->P = sh->P; o->B = sh->B; o->T = sh->T; o->D = sh->D; o->k = sh->k;
  o->H = o->D * o->k;
  o->L = o->T / o->P;
  o->M = o->P * o->B;
  if (o->H > kMaxFfnH)
    return fail(DG_ERR_UNSUPPORTED, "shape: H = D*k = %lld exceeds %d", (long long)o->H, kMaxFfnH);
  if (o->M > (1 << 30)) return fail(DG_ERR_UNSUPPORTED, "shape: P*B too large");
  return DG_OK;
}

// Carving of the forward's `saved` buffer: Z [T,M,2H] bf16, Hl [T,M,H] bf16,
// stats [T,M] float4, and the per-tile LayerNorm partials [T,tiles_n,M] float4.
struct SavedLayout {
  size_t z, hl, stats, part, total;
  int tiles_n;
};
SavedLayout saved_layout(const FfnDims& f) {
  SavedLayout l;
  const size_t rows = static_cast<size_t>(f.T) * f.M;
  l.tiles_n = static_cast<int>((2 * f.H + gemm_tile_n(GV_BF16_KM_LNSTATS) - 1) / gemm_tile_n(GV_BF16_KM_LNSTATS));
  l.z = 0;
  l.hl = round_up(l.z + rows * 2 * f.H * 2, 256);
  l.stats = round_up(l.hl + rows * f.H * 2, 256);
  l.part = round_up(l.stats + rows * 16, 256);
  l.total = round_up(l.part + rows * l.tiles_n * 16, 256);
  return l;
}

// Carving of the backward's workspace: the error block, then
// (DG_FFN_COMP_ONLY) the rank/slice-swapped inputs, dY and d_inputs, then
// dHl [T,M,H] bf16, dZ [T,M,2H] bf16, the per-row coefficient records
// [T,M] x 32 bytes and the column partials [T,nsplit,6,H] fp32.
struct BwdLayout {
  size_t perm_x, perm_dy, perm_dx, dhl, dz, rowcoef, part, total;
  int nsplit;
};
BwdLayout bwd_layout(const FfnDims& f, uint32_t flags) {
  BwdLayout l{};
  const size_t rows = static_cast<size_t>(f.T) * f.M;
  const size_t act = static_cast<size_t>(f.P) * f.B * f.T * f.D * 2;
  l.nsplit = ffn_bwd_row_splits(static_cast<int>(f.T), static_cast<int>(f.M), static_cast<int>(f.H));
  size_t off = DG_ERROR_BLOCK_BYTES;
  if (flags & DG_FFN_COMP_ONLY) {
    l.perm_x = off;
    off = round_up(off + act, 256);
    l.perm_dy = off;
    off = round_up(off + act, 256);
    l.perm_dx = off;
    off = round_up(off + act, 256);
  }
  l.dhl = off;
  l.dz = round_up(l.dhl + rows * f.H * 2, 256);
  l.rowcoef = round_up(l.dz + rows * 2 * f.H * 2, 256);
  l.part = round_up(l.rowcoef + rows * 32, 256);
  l.total = round_up(l.part + static_cast<size_t>(f.T) * l.nsplit * 6 * f.H * 4, 256);
  return l;
}

inline const char* ptr_name_null(const void* const* ptrs, const char* const* names, int n) {
  for (int i = 0; i < n; ++i)
    if (!ptrs[i]) return names[i];
  return nullptr;
}

inline const char* ptr_name_unaligned(const void* const* ptrs, const char* const* names, int n) {
  for (int i = 0; i < n; ++i)
    if (!aligned16(ptrs[i])) return names[i];
  return nullptr;
}

}  // namespace

extern "C" {

const char* dg_last_error(void) { return t_last_error; }

const char* dg_version(void) { return "dg 0.1 (sm_103a)"; }

dg_status dg_workspace_init(void* ws, size_t ws_bytes, void* stream) {
  DeviceInfo dev;
  dg_status st = device_info_ws(&dev, ws, ws_bytes, "workspace_init");
  if (st != DG_OK) return st;
  cudaError_t e = cudaMemsetAsync(ws, 0, DG_ERROR_BLOCK_BYTES, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? DG_OK : cuda_fail(e, "workspace_init: clearing the error block");
}

dg_status dg_check_device_error(void* ws, void* stream, uint32_t* site) {
  DeviceInfo dev;
  dg_status st = device_info(&dev);
  if (st != DG_OK) return st;
  uint32_t* word = ws ? static_cast<uint32_t*>(ws) : dev.builtin_err;
  if (ws && !aligned16(ws)) return fail(DG_ERR_INVALID_ARGUMENT, "check_device_error: ws is not 16-byte aligned");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t value = 0;
  cudaError_t e = cudaMemcpyAsync(&value, word, sizeof(value), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "check_device_error: reading the error word");
  if (value == 0) return DG_OK;
  e = cudaMemsetAsync(word, 0, sizeof(uint32_t), s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "check_device_error: clearing the error word");
  if (site) *site = value;
  if (value & kErrTimeout)
    return fail(DG_ERR_TIMEOUT, "a device-side wait exceeded its limit (site %u)", value & 0xffu);
  return fail(DG_ERR_DEVICE_CHECK, "device-side check failed (code 0x%x)", value);
}

dg_status dg_debug_wait_timeout(void* ws, size_t ws_bytes, uint32_t limit_us, void* stream) {
  DeviceInfo dev;
  dg_status st = device_info_ws(&dev, ws, ws_bytes, "debug_wait_timeout");
  if (st != DG_OK) return st;
  if (limit_us == 0 || limit_us > 10u * 1000u * 1000u)
    return fail(DG_ERR_INVALID_ARGUMENT, "limit_us must be in (0, 10 s]");
  cudaError_t e = launch_debug_wait(dev.err, static_cast<uint64_t>(limit_us) * 1000u, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "debug wait launch");
  return DG_OK;
}

// ------------------------------------------------------------------ FP8 GEMM

size_t dg_gemm_fp8_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  (void)M;
  (void)N;
  (void)K;
  return DG_ERROR_BLOCK_BYTES;
}

dg_status dg_gemm_fp8(int64_t M, int64_t N, int64_t K, const void* A, const void* B, const void* C, void* D,
                      float alpha, float beta, void* ws, size_t ws_bytes, void* stream) {
  if (M < 0 || N < 0 || K < 0) return fail(DG_ERR_INVALID_ARGUMENT, "gemm_fp8: negative size");
  if (M == 0 || N == 0) return DG_OK;
  if (M > 0x7fffffff || N > 0x7fffffff || K > 0x7fffffff)
    return fail(DG_ERR_UNSUPPORTED, "gemm_fp8: sizes beyond 2^31-1");
  if (K % 16) return fail(DG_ERR_INVALID_ARGUMENT, "gemm_fp8: K must be a multiple of 16 (16-byte rows), got %lld",
                          (long long)K);
  if (N % 8) return fail(DG_ERR_INVALID_ARGUMENT, "gemm_fp8: N must be a multiple of 8 (16-byte rows), got %lld",
                         (long long)N);
  if (!D) return fail(DG_ERR_INVALID_ARGUMENT, "gemm_fp8: D is NULL");
  if (K > 0 && (!A || !B)) return fail(DG_ERR_INVALID_ARGUMENT, "gemm_fp8: A or B is NULL");
  const bool has_c = beta != 0.0f;
  if (has_c && !C) return fail(DG_ERR_INVALID_ARGUMENT, "gemm_fp8: C is NULL but beta != 0");
  const size_t dbytes = static_cast<size_t>(M) * N * 2;
  if (overlaps(D, dbytes, A, static_cast<size_t>(M) * K) || overlaps(D, dbytes, B, static_cast<size_t>(N) * K) ||
      (has_c && overlaps(D, dbytes, C, dbytes)) || overlaps(D, dbytes, ws, DG_ERROR_BLOCK_BYTES))
    return fail(DG_ERR_INVALID_ARGUMENT, "gemm_fp8: D overlaps an input or the workspace");
  DeviceInfo dev;
  dg_status st = device_info_ws(&dev, ws, ws_bytes, "gemm_fp8");
  if (st != DG_OK) return st;
  // Tile width: 224 columns where that needs fewer (wave x width) column
  // steps than 256 across the co-resident CTA pairs (e.g. 4096 x 4096:
  // 304 tiles = 4 full waves of 76 pairs instead of 256 tiles = 3.4 waves).
  int units = 0;
  cudaError_t ce = gemm_fp8_units(dev.num_sms, &units);
  if (ce != cudaSuccess) return cuda_fail(ce, "gemm_fp8: occupancy query");
  const int64_t tiles_m = (M + gemm_tile_m() - 1) / gemm_tile_m();
  auto wave_cost = [&](int64_t bn) {
    const int64_t tiles = tiles_m * ((N + bn - 1) / bn);
    return ((tiles + units - 1) / units) * bn;
  };
  const GemmVariant v = wave_cost(224) < wave_cost(256) ? GV_FP8_KK_N224 : GV_FP8_KK;
  const uint32_t b_rows = static_cast<uint32_t>(gemm_tile_n(v) / (kUsePairs ? 2 : 1));
  CUtensorMap ma, mb, md, mc;
  // K == 0: the maps still need a valid (non-empty) tensor; the kernel loads nothing.
  const uint64_t kd = K > 0 ? static_cast<uint64_t>(K) : 16u;
  const void* a_ptr = K > 0 ? A : D;
  const void* b_ptr = K > 0 ? B : D;
  const uint64_t am = K > 0 ? static_cast<uint64_t>(M) : 1u, bn = K > 0 ? static_cast<uint64_t>(N) : 1u;
  if ((st = make_map_3d(&ma, false, a_ptr, kd, am, 1, kd, kd * am, 128, 128, 1, "A")) != DG_OK) return st;
  if ((st = make_map_3d(&mb, false, b_ptr, kd, bn, 1, kd, kd * bn, 128, b_rows, 1, "B")) != DG_OK) return st;
  if ((st = make_map_3d(&md, true, D, N, M, 1, N * 2, N * 2 * M, 64, 32, 1, "D")) != DG_OK) return st;
  if (has_c) {
    if ((st = make_map_3d(&mc, true, C, N, M, 1, N * 2, N * 2 * M, 64, 32, 1, "C")) != DG_OK) return st;
  } else {
    mc = md;
  }
  GemmParams p{};
  p.G = 1;
  p.M = static_cast<int32_t>(M);
  p.N = static_cast<int32_t>(N);
  p.K = static_cast<int32_t>(K);
  p.a_g = p.b_g = p.d_g = G_OUTER;
  p.alpha = alpha;
  p.beta = beta;
  p.has_c = has_c ? 1 : 0;
  p.c_ptr = static_cast<const __nv_bfloat16*>(has_c ? C : D);
  p.d_ptr = static_cast<__nv_bfloat16*>(D);
  const double bytes = static_cast<double>(M) * K + static_cast<double>(N) * K + (has_c ? 2.0 : 1.0) * 2.0 * M * N;
  return run_gemm(v, ma, mb, md, mc, p, dev, static_cast<cudaStream_t>(stream),
                  v == GV_FP8_KK_N224 ? "gemm_fp8_n224" : "gemm_fp8", bytes);
}

// ------------------------------------------------------------------ A2A FFN

namespace {

constexpr uint32_t kFfnFlagsKnown = DG_FFN_COMP_ONLY | DG_FFN_FUSED_GATE | DG_FFN_SEPARATE_GATE;

dg_status check_ffn_flags(const FfnDims& f, uint32_t flags, uint32_t allowed, const char* what) {
  if (flags & ~allowed) return fail(DG_ERR_INVALID_ARGUMENT, "%s: unknown flags 0x%x", what, flags & ~allowed);
  if ((flags & DG_FFN_FUSED_GATE) && (flags & DG_FFN_SEPARATE_GATE))
    return fail(DG_ERR_INVALID_ARGUMENT, "%s: DG_FFN_FUSED_GATE and DG_FFN_SEPARATE_GATE exclude each other", what);
  (void)f;
  return DG_OK;
}

// The normalise-and-gate runs inside GEMM2 unless the separate pass is asked for.
inline bool ffn_fused_gate(uint32_t flags) { return !(flags & DG_FFN_SEPARATE_GATE); }

// The forward's workspace: the error block, then (DG_FFN_COMP_ONLY) the
// rank/slice-swapped input and output, then (inference, saved == NULL) the
// Z, statistics and per-tile partials that would otherwise live in `saved`,
// and Hl unless the gated GEMM covers all of D in one column pass.
struct FwdWsLayout {
  size_t perm_in, perm_out, z, stats, part, hl, total;
};
FwdWsLayout fwd_ws_layout(const FfnDims& f, bool inference, uint32_t flags) {
  FwdWsLayout l{};
  const size_t rows = static_cast<size_t>(f.T) * f.M;
  const size_t act = static_cast<size_t>(f.P) * f.B * f.T * f.D * 2;
  const int tiles_n = static_cast<int>((2 * f.H + gemm_tile_n(GV_BF16_KM_LNSTATS) - 1) / gemm_tile_n(GV_BF16_KM_LNSTATS));
  size_t off = DG_ERROR_BLOCK_BYTES;
  if (flags & DG_FFN_COMP_ONLY) {
    l.perm_in = off;
    off = round_up(off + act, 256);
    l.perm_out = off;
    off = round_up(off + act, 256);
  }
  if (inference) {
    l.z = off;
    off = round_up(off + rows * 2 * f.H * 2, 256);
    l.stats = off;
    off = round_up(off + rows * 16, 256);
    l.part = off;
    off = round_up(off + rows * tiles_n * 16, 256);
    if (!ffn_fused_gate(flags) || f.D > gemm_gated_tile_n()) {
      l.hl = off;
      off = round_up(off + rows * f.H * 2, 256);
    }
  }
  l.total = off;
  return l;
}

}  // namespace

size_t dg_a2a_ffn_saved_bytes(const dg_ffn_shape* shape) {
  FfnDims f{};
  if (check_ffn_shape(shape, &f) != DG_OK) return 0;
  return saved_layout(f).total;
}

size_t dg_a2a_ffn_fwd_workspace_bytes(const dg_ffn_shape* shape, int32_t inference, uint32_t flags) {
  FfnDims f{};
  if (check_ffn_shape(shape, &f) != DG_OK || (flags & ~kFfnFlagsKnown) ||
      ((flags & DG_FFN_FUSED_GATE) && (flags & DG_FFN_SEPARATE_GATE)))
    return 0;
  return fwd_ws_layout(f, inference != 0, flags).total;
}

size_t dg_a2a_ffn_bwd_workspace_bytes(const dg_ffn_shape* shape, uint32_t flags) {
  FfnDims f{};
  if (check_ffn_shape(shape, &f) != DG_OK || (flags & ~kFfnFlagsKnown)) return 0;
  if ((flags & DG_FFN_FUSED_GATE) && (flags & DG_FFN_SEPARATE_GATE)) return 0;
  return bwd_layout(f, flags).total;
}

dg_status dg_a2a_ffn_fwd(const dg_ffn_shape* shape, const void* inputs, const void* w1, const void* b1,
                         const void* wout, const void* bout, const void* nx_w, const void* nx_b, const void* ng_w,
                         const void* ng_b, void* output, void* saved, size_t saved_bytes, void* ws, size_t ws_bytes,
                         uint32_t flags, void* stream) {
  FfnDims f{};
  dg_status st = check_ffn_shape(shape, &f);
  if (st != DG_OK) return st;
  if ((st = check_ffn_flags(f, flags, kFfnFlagsKnown, "a2a_ffn_fwd")) != DG_OK) return st;
  const void* ptrs[] = {inputs, w1, b1, wout, bout, nx_w, nx_b, ng_w, ng_b, output};
  const char* names[] = {"inputs", "w1", "b1", "wout", "bout", "nx_w", "nx_b", "ng_w", "ng_b", "output"};
  if (const char* n = ptr_name_null(ptrs, names, 10)) return fail(DG_ERR_INVALID_ARGUMENT, "a2a_ffn_fwd: %s is NULL", n);
  if (const char* n = ptr_name_unaligned(ptrs, names, 10))
    return fail(DG_ERR_INVALID_ARGUMENT, "a2a_ffn_fwd: %s is not 16-byte aligned", n);
  const bool inference = saved == nullptr;
  if (!inference && !aligned16(saved)) return fail(DG_ERR_INVALID_ARGUMENT, "a2a_ffn_fwd: saved is not 16-byte aligned");
  const SavedLayout sl = saved_layout(f);
  if (!inference && saved_bytes < sl.total)
    return fail(DG_ERR_WORKSPACE, "a2a_ffn_fwd: saved buffer has %zu bytes, needs %zu", saved_bytes, sl.total);
  const FwdWsLayout wl = fwd_ws_layout(f, inference, flags);
  if (ws_bytes < wl.total && ws != nullptr)
    return fail(DG_ERR_WORKSPACE, "a2a_ffn_fwd: workspace has %zu bytes, needs %zu", ws_bytes, wl.total);
  const size_t act = static_cast<size_t>(f.P) * f.B * f.T * f.D * 2;
  const size_t svb = inference ? 0 : sl.total;
  if (overlaps(output, act, inputs, act) || overlaps(output, act, saved, svb) || overlaps(saved, svb, inputs, act) ||
      overlaps(ws, wl.total, inputs, act) || overlaps(ws, wl.total, output, act) || overlaps(ws, wl.total, saved, svb))
    return fail(DG_ERR_INVALID_ARGUMENT, "a2a_ffn_fwd: output / saved / workspace / inputs overlap");
  DeviceInfo dev;
  if ((st = device_info_ws(&dev, ws, ws_bytes, "a2a_ffn_fwd")) != DG_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* w = static_cast<uint8_t*>(ws);
  uint8_t* sv = static_cast<uint8_t*>(saved);
  void* Z = inference ? w + wl.z : sv + sl.z;
  void* stats = inference ? w + wl.stats : sv + sl.stats;
  void* part = inference ? w + wl.part : sv + sl.part;
  void* Hl = inference ? (ffn_fused_gate(flags) && f.D <= gemm_gated_tile_n() ? nullptr : w + wl.hl)
                       : sv + sl.hl;
  const uint64_t T = f.T, M = f.M, D = f.D, H = f.H;
  const double rows = static_cast<double>(T) * M;
  cudaError_t e;

  // comp_only: no exchange.  Rank r's own [B, T, D] rows, viewed as
  // [B, P, L, D], feed its L problems; that is the exchange with the roles of
  // rank and slice swapped, so the inputs are swapped into the workspace, the
  // layer runs as usual, and its output is swapped back.
  const void* x_in = inputs;
  void* y_out = output;
  if (flags & DG_FFN_COMP_ONLY) {
    TraceScope trace("ffn_comp_only_swap", s, 0.0, 2.0 * act);
    e = launch_swap_rank_slice(inputs, w + wl.perm_in, static_cast<int>(f.P), static_cast<int>(f.B),
                               static_cast<int>(T), static_cast<int>(D), dev, s);
    if (e != cudaSuccess) return cuda_fail(e, "comp_only input swap launch");
    x_in = w + wl.perm_in;
    y_out = w + wl.perm_out;
  }

  // GEMM1: Z_t = Xlocal_t @ w1_t + b1_t.  Xlocal_t row n is inputs row n*T + t (dispatch).
  // The epilogue also writes each row's per-tile mean and M2 of its U and G columns.
  CUtensorMap mx, mw1, mz;
  if ((st = make_map_3d(&mx, true, x_in, D, T, M, D * 2, T * D * 2, 64, 1, 128, "inputs")) != DG_OK) return st;
  int32_t w1_mn4 = 0;
  if ((st = make_map_mn(&mw1, w1, 2 * H, D, T, 2 * H * 2, D * 2 * H * 2, 64, 1, kMnBlocksB, &w1_mn4, "w1")) != DG_OK)
    return st;
  if ((st = make_map_3d(&mz, true, Z, 2 * H, M, T, 2 * H * 2, M * 2 * H * 2, 64, 32, 1, "Z")) != DG_OK) return st;
  GemmParams p1{};
  p1.G = static_cast<int32_t>(T);
  p1.M = static_cast<int32_t>(M);
  p1.N = static_cast<int32_t>(2 * H);
  p1.K = static_cast<int32_t>(D);
  p1.a_g = G_MID;
  p1.b_g = G_OUTER;
  p1.d_g = G_OUTER;
  p1.bias = static_cast<const __nv_bfloat16*>(b1);
  p1.bias_g_stride = static_cast<int64_t>(2 * H);
  p1.ln_part = static_cast<float4*>(part);
  p1.ln_H = static_cast<int32_t>(H);
  p1.b_mn4 = w1_mn4;
  if ((st = run_gemm(GV_BF16_KM_LNSTATS, mx, mw1, mz, mz, p1, dev, s, "ffn_gemm1",
                     2.0 * (rows * D + static_cast<double>(T) * D * 2 * H + rows * 2 * H) +
                         rows * sl.tiles_n * 16.0)) != DG_OK)
    return st;

  // Per-row statistics of U and G.
  {
    TraceScope trace("ffn_ln_stats", s, 0.0, rows * sl.tiles_n * 16.0 + rows * 16.0);
    e = launch_ln_stats_finalize(static_cast<const float4*>(part), stats, static_cast<int>(T), static_cast<int>(M),
                                 static_cast<int>(H), gemm_tile_n(GV_BF16_KM_LNSTATS), sl.tiles_n, shape->eps, dev, s);
  }
  if (e != cudaSuccess) return cuda_fail(e, "LayerNorm statistics launch");

  // GEMM2: output rows (s, b, t) = Hl_t @ wout_t + bout_t at the combine offsets,
  // with Hl = LN_x(U) * silu(LN_g(G)) computed by the GEMM's own producer
  // warps from Z (the default) or, with DG_FFN_SEPARATE_GATE, by a separate
  // pass through HBM.  The gated GEMM covers the first column pass (up to
  // gemm_gated_tile_n() output columns) and stores Hl as it goes; a plain
  // GEMM2 on that Hl computes the remaining columns, so the gate is computed
  // once, not once per column pass.
  CUtensorMap mwo, mo;
  int32_t wo_mn4 = 0;
  if ((st = make_map_mn(&mwo, wout, D, H, T, D * 2, H * D * 2, 64, 1, kMnBlocksB, &wo_mn4, "wout")) != DG_OK)
    return st;
  if ((st = make_map_3d(&mo, true, y_out, D, T, M, D * 2, T * D * 2, 64, 1, 32, "output")) != DG_OK) return st;
  GemmParams p2{};
  p2.b_mn4 = wo_mn4;
  p2.G = static_cast<int32_t>(T);
  p2.M = static_cast<int32_t>(M);
  p2.N = static_cast<int32_t>(D);
  p2.K = static_cast<int32_t>(H);
  p2.a_g = G_OUTER;
  p2.b_g = G_OUTER;
  p2.d_g = G_MID;
  p2.bias = static_cast<const __nv_bfloat16*>(bout);
  p2.bias_g_stride = static_cast<int64_t>(D);
  if (ffn_fused_gate(flags)) {
    GateSrc q{};
    q.Z = static_cast<const __nv_bfloat16*>(Z);
    q.stats = static_cast<const float4*>(stats);
    q.gx = static_cast<const __nv_bfloat16*>(nx_w);
    q.bx = static_cast<const __nv_bfloat16*>(nx_b);
    q.gg = static_cast<const __nv_bfloat16*>(ng_w);
    q.bg = static_cast<const __nv_bfloat16*>(ng_b);
    q.Hl = static_cast<__nv_bfloat16*>(Hl);
    q.H = static_cast<int32_t>(H);
    q.L = static_cast<int32_t>(f.L);
    const int64_t n_fused = D < gemm_gated_tile_n() ? D : gemm_gated_tile_n();
    const double bytes = rows * (2.0 * 2 * H + 16.0 + 2.0 * n_fused) + 2.0 * static_cast<double>(T) * H * n_fused +
                         (Hl ? rows * 2.0 * H : 0.0);
    // Z by rows, U at x = k and G at x = H + k, and wout, in boxes of the gated
    // GEMM's K block (BK columns of Z with a 2*BK-byte swizzle; BK rows of wout)
    const uint32_t bk = static_cast<uint32_t>(gemm_gated_bk());
    CUtensorMap mzk, mwok;
    if ((st = make_map_3d_sw(&mzk, true, Z, 2 * H, M, T, 2 * H * 2, M * 2 * H * 2, bk, 128, 1,
                             static_cast<int>(2 * bk), "Z (gate)")) != DG_OK)
      return st;
    if ((st = make_map_mn(&mwok, wout, D, H, T, D * 2, H * D * 2, bk, 1, kMnBlocksB, &p2.b_mn4, "wout")) != DG_OK)
      return st;
    mwo = mwok;
    GemmParams pf = p2;
    pf.N = static_cast<int32_t>(n_fused);
    if ((st = run_gemm_gated(mwo, mo, mzk, pf, q, dev, s, "ffn_gemm2_gated", bytes)) != DG_OK) return st;
    if (D > n_fused) {
      // columns [n_fused, D): a plain GEMM2 on the Hl the gated pass stored
      const int64_t rest = D - n_fused;
      CUtensorMap mh, mwor, mor;
      GemmParams pr = p2;
      pr.N = static_cast<int32_t>(rest);
      pr.bias = static_cast<const __nv_bfloat16*>(bout) + n_fused;
      const __nv_bfloat16* wout_r = static_cast<const __nv_bfloat16*>(wout) + n_fused;
      __nv_bfloat16* y_r = static_cast<__nv_bfloat16*>(y_out) + n_fused;
      if ((st = make_map_3d(&mh, true, Hl, H, M, T, H * 2, M * H * 2, 64, 128, 1, "Hl")) != DG_OK) return st;
      if ((st = make_map_mn(&mwor, wout_r, rest, H, T, D * 2, H * D * 2, 64, 1, kMnBlocksB, &pr.b_mn4,
                            "wout (remaining columns)")) != DG_OK)
        return st;
      if ((st = make_map_3d(&mor, true, y_r, rest, T, M, D * 2, T * D * 2, 64, 1, 32, "output (remaining columns)")) !=
          DG_OK)
        return st;
      if ((st = run_gemm(GV_BF16_KM_BIAS, mh, mwor, mor, mor, pr, dev, s, "ffn_gemm2_rest",
                         2.0 * (rows * H + static_cast<double>(T) * H * rest + rows * rest))) != DG_OK)
        return st;
    }
  } else {
    {
      TraceScope trace("ffn_ln_gate_fwd", s, 0.0, rows * (2.0 * 2 * H + 2.0 * H + 16.0));
      e = launch_ln_gate_fwd(Z, stats, nx_w, nx_b, ng_w, ng_b, Hl, nullptr, nullptr, static_cast<int>(f.P),
                             static_cast<int>(M), static_cast<int>(f.L), static_cast<int>(H), dev, s);
    }
    if (e != cudaSuccess) return cuda_fail(e, "LayerNorm-gate launch");
    CUtensorMap mh;
    if ((st = make_map_3d(&mh, true, Hl, H, M, T, H * 2, M * H * 2, 64, 128, 1, "Hl")) != DG_OK) return st;
    if ((st = run_gemm(GV_BF16_KM_BIAS, mh, mwo, mo, mo, p2, dev, s, "ffn_gemm2",
                       2.0 * (rows * H + static_cast<double>(T) * H * D + rows * D))) != DG_OK)
      return st;
  }

  if (flags & DG_FFN_COMP_ONLY) {
    TraceScope trace("ffn_comp_only_swap", s, 0.0, 2.0 * act);
    e = launch_swap_rank_slice(y_out, output, static_cast<int>(f.P), static_cast<int>(f.B), static_cast<int>(T),
                               static_cast<int>(D), dev, s);
    if (e != cudaSuccess) return cuda_fail(e, "comp_only output swap launch");
  }
  return DG_OK;
}

dg_status dg_a2a_ffn_bwd(const dg_ffn_shape* shape, const void* inputs, const void* w1, const void* b1,
                         const void* wout, const void* bout, const void* nx_w, const void* nx_b, const void* ng_w,
                         const void* ng_b, const void* saved, size_t saved_bytes, const void* dY, void* d_inputs,
                         void* d_w1, void* d_b1, void* d_wout, void* d_bout, void* d_nx_w, void* d_nx_b,
                         void* d_ng_w, void* d_ng_b, void* ws, size_t ws_bytes, uint32_t flags, void* stream) {
  FfnDims f{};
  dg_status st = check_ffn_shape(shape, &f);
  if (st != DG_OK) return st;
  // The forward's flags: comp_only applies; the gate flags are checked the
  // same way but leave the backward unchanged (its row sums are a pass of
  // their own either way).
  if ((st = check_ffn_flags(f, flags, kFfnFlagsKnown, "a2a_ffn_bwd")) != DG_OK) return st;
  (void)b1;
  (void)bout;
  // What each requested gradient needs: dZ (from dHl and the LayerNorm-gate
  // backward) feeds d_inputs, d_w1, d_b1 and the norm gradients; d_wout needs
  // Hl; d_bout needs only dY.
  const bool want_norm = d_nx_w || d_nx_b || d_ng_w || d_ng_b;
  const bool need_dz = d_inputs || d_w1 || d_b1 || want_norm;
  const void* ptrs[] = {inputs, w1, wout, nx_w, nx_b, ng_w, ng_b, saved, dY};
  const char* names[] = {"inputs", "w1", "wout", "nx_w", "nx_b", "ng_w", "ng_b", "saved", "dY"};
  const bool needed[] = {d_w1 != nullptr, d_inputs != nullptr, need_dz, need_dz, need_dz, need_dz, need_dz,
                         need_dz || d_wout != nullptr, true};
  for (int i = 0; i < 9; ++i) {
    if (needed[i] && !ptrs[i])
      return fail(DG_ERR_INVALID_ARGUMENT, "a2a_ffn_bwd: %s is NULL but a requested gradient needs it", names[i]);
    if (ptrs[i] && !aligned16(ptrs[i]))
      return fail(DG_ERR_INVALID_ARGUMENT, "a2a_ffn_bwd: %s is not 16-byte aligned", names[i]);
  }
  void* outs[] = {d_inputs, d_w1, d_b1, d_wout, d_bout, d_nx_w, d_nx_b, d_ng_w, d_ng_b};
  const char* onames[] = {"d_inputs", "d_w1", "d_b1", "d_wout", "d_bout", "d_nx_w", "d_nx_b", "d_ng_w", "d_ng_b"};
  for (int i = 0; i < 9; ++i)
    if (outs[i] && !aligned16(outs[i]))
      return fail(DG_ERR_INVALID_ARGUMENT, "a2a_ffn_bwd: %s is not 16-byte aligned", onames[i]);
  const SavedLayout sl = saved_layout(f);
  if (saved && saved_bytes < sl.total)
    return fail(DG_ERR_WORKSPACE, "a2a_ffn_bwd: saved buffer has %zu bytes, needs %zu", saved_bytes, sl.total);
  const BwdLayout bl = bwd_layout(f, flags);
  if (ws && ws_bytes < bl.total)
    return fail(DG_ERR_WORKSPACE, "a2a_ffn_bwd: workspace has %zu bytes, needs %zu", ws_bytes, bl.total);
  // Every written region (the gradients and the workspace) must be disjoint
  // from every other region, read or written.
  const size_t act = static_cast<size_t>(f.P) * f.B * f.T * f.D * 2;
  const size_t w1b = static_cast<size_t>(f.T) * f.D * 2 * f.H * 2, b1b = static_cast<size_t>(f.T) * 2 * f.H * 2;
  const size_t wob = static_cast<size_t>(f.T) * f.H * f.D * 2, bob = static_cast<size_t>(f.T) * f.D * 2;
  const size_t nb = static_cast<size_t>(f.P) * f.H * 2;
  const void* wr[] = {d_inputs, d_w1, d_b1, d_wout, d_bout, d_nx_w, d_nx_b, d_ng_w, d_ng_b, ws};
  const size_t wr_n[] = {act, w1b, b1b, wob, bob, nb, nb, nb, nb, bl.total};
  const void* rd[] = {inputs, w1, wout, nx_w, nx_b, ng_w, ng_b, saved, dY};
  const size_t rd_n[] = {act, w1b, wob, nb, nb, nb, nb, sl.total, act};
  for (int i = 0; i < 10; ++i) {
    for (int j = 0; j < 10; ++j)
      if (j != i && overlaps(wr[i], wr_n[i], wr[j], wr_n[j]))
        return fail(DG_ERR_INVALID_ARGUMENT, "a2a_ffn_bwd: written buffers overlap");
    for (int j = 0; j < 9; ++j)
      if (overlaps(wr[i], wr_n[i], rd[j], rd_n[j]))
        return fail(DG_ERR_INVALID_ARGUMENT, "a2a_ffn_bwd: a written buffer overlaps %s", names[j]);
  }
  DeviceInfo dev;
  if ((st = device_info_ws(&dev, ws, ws_bytes, "a2a_ffn_bwd")) != DG_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const uint8_t* sv = static_cast<const uint8_t*>(saved);
  const void* Z = sv ? sv + sl.z : nullptr;
  const void* Hl = sv ? sv + sl.hl : nullptr;
  const void* stats = sv ? sv + sl.stats : nullptr;
  uint8_t* w = static_cast<uint8_t*>(ws);
  void* dHl = w + bl.dhl;
  void* dZ = w + bl.dz;
  void* rowcoef = w + bl.rowcoef;
  float* part = reinterpret_cast<float*>(w + bl.part);
  const uint64_t T = f.T, M = f.M, D = f.D, H = f.H;
  const double rows = static_cast<double>(T) * M;
  cudaError_t e;

  // comp_only: the same backward on the rank/slice-swapped tensors (see the forward).
  const void* x_in = inputs;
  const void* dy_in = dY;
  void* dx_out = d_inputs;
  if (flags & DG_FFN_COMP_ONLY) {
    TraceScope trace("ffn_comp_only_swap", s, 0.0, 2.0 * act);
    if (inputs && d_w1) {
      e = launch_swap_rank_slice(inputs, w + bl.perm_x, static_cast<int>(f.P), static_cast<int>(f.B),
                                 static_cast<int>(T), static_cast<int>(D), dev, s);
      if (e != cudaSuccess) return cuda_fail(e, "comp_only input swap launch");
      x_in = w + bl.perm_x;
    }
    e = launch_swap_rank_slice(dY, w + bl.perm_dy, static_cast<int>(f.P), static_cast<int>(f.B), static_cast<int>(T),
                               static_cast<int>(D), dev, s);
    if (e != cudaSuccess) return cuda_fail(e, "comp_only dY swap launch");
    dy_in = w + bl.perm_dy;
    if (d_inputs) dx_out = w + bl.perm_dx;
  }

  if (need_dz) {
    // (1) dHl_t = dY_t @ wout_t^T      (dY_t: the dispatched rows of dY)
    CUtensorMap mdy_k, mwo_k, mdh;
    if ((st = make_map_3d(&mdy_k, true, dy_in, D, T, M, D * 2, T * D * 2, 64, 1, 128, "dY")) != DG_OK) return st;
    if ((st = make_map_3d(&mwo_k, true, wout, D, H, T, D * 2, H * D * 2, 64, kKMajorBRows, 1, "wout")) != DG_OK)
      return st;
    if ((st = make_map_3d(&mdh, true, dHl, H, M, T, H * 2, M * H * 2, 64, 32, 1, "dHl")) != DG_OK) return st;
    GemmParams p{};
    p.G = static_cast<int32_t>(T);
    p.M = static_cast<int32_t>(M);
    p.N = static_cast<int32_t>(H);
    p.K = static_cast<int32_t>(D);
    p.a_g = G_MID;
    p.b_g = G_OUTER;
    p.d_g = G_OUTER;
    if ((st = run_gemm(GV_BF16_KK_STORE, mdy_k, mwo_k, mdh, mdh, p, dev, s, "ffn_bwd_dhl",
                       2.0 * (rows * D + static_cast<double>(T) * H * D + rows * H))) != DG_OK)
      return st;
  }

  if (d_wout) {
    // (2) dwout_t = Hl_t^T @ dY_t     [H, D], contraction over the M rows
    CUtensorMap mhl_t, mdy_n, mdwo;
    int32_t hl_mn4 = 0, dyn_mn4 = 0;
    if ((st = make_map_mn(&mhl_t, Hl, H, M, T, H * 2, M * H * 2, 64, 1, kMnBlocksA, &hl_mn4, "Hl^T")) != DG_OK)
      return st;
    if ((st = make_map_mn(&mdy_n, dy_in, D, T, M, D * 2, T * D * 2, 1, 64, kMnBlocksB, &dyn_mn4, "dY (N-major)")) !=
        DG_OK)
      return st;
    if ((st = make_map_3d(&mdwo, true, d_wout, D, H, T, D * 2, H * D * 2, 64, 32, 1, "d_wout")) != DG_OK) return st;
    GemmParams p{};
    p.G = static_cast<int32_t>(T);
    p.M = static_cast<int32_t>(H);
    p.N = static_cast<int32_t>(D);
    p.K = static_cast<int32_t>(M);
    p.a_g = G_OUTER;
    p.b_g = G_MID;
    p.d_g = G_OUTER;
    p.a_mn4 = hl_mn4;
    p.b_mn4 = dyn_mn4;
    if ((st = run_gemm(GV_BF16_MM_STORE, mhl_t, mdy_n, mdwo, mdwo, p, dev, s, "ffn_bwd_dwout",
                       2.0 * (rows * H + rows * D + static_cast<double>(T) * H * D))) != DG_OK)
      return st;
  }

  if (d_bout) {
    // (3) dbout_t = sum_n dY_t[n, :]
    TraceScope trace("ffn_bwd_dbout", s, 0.0, rows * D * 2.0 + static_cast<double>(T) * D * 2.0);
    e = launch_column_sum(dy_in, d_bout, static_cast<int>(T), static_cast<int>(M), static_cast<int>(D),
                          static_cast<int64_t>(D), static_cast<int64_t>(T * D), dev, s);
    if (e != cudaSuccess) return cuda_fail(e, "column-sum launch");
  }

  if (need_dz) {
    // (4) gate + LayerNorm backward: per-row sums, then dZ with db1 and the norm column sums
    {
      TraceScope trace("ffn_bwd_ln_rowsum", s, 0.0, rows * (2.0 * 2 * H + 2.0 * H + 16.0 + 32.0));
      e = launch_ln_gate_bwd_rowsum(Z, stats, dHl, nx_w, nx_b, ng_w, ng_b, rowcoef, static_cast<int>(T),
                                    static_cast<int>(M), static_cast<int>(f.L), static_cast<int>(H), dev, s);
    }
    if (e != cudaSuccess) return cuda_fail(e, "LayerNorm-gate backward (row sums) launch");
    {
      TraceScope trace("ffn_bwd_ln_apply", s, 0.0,
                       rows * (2.0 * 2 * H + 2.0 * H + 32.0 + 2.0 * 2 * H) +
                           static_cast<double>(T) * bl.nsplit * 6 * H * 4);
      e = launch_ln_gate_bwd_apply(Z, rowcoef, dHl, nx_w, nx_b, ng_w, ng_b, dZ, part, static_cast<int>(T),
                                   static_cast<int>(M), static_cast<int>(f.L), static_cast<int>(H), bl.nsplit, dev, s);
    }
    if (e != cudaSuccess) return cuda_fail(e, "LayerNorm-gate backward (apply) launch");
  }

  if (d_b1 || want_norm) {
    // (5) db1, d(norm_x), d(norm_gate): partial sums added in a fixed order
    TraceScope trace("ffn_bwd_grad_reduce", s, 0.0,
                     static_cast<double>(T) * bl.nsplit * 6 * H * 4 + static_cast<double>(T) * 2 * H * 2 +
                         static_cast<double>(f.P) * 4 * H * 2);
    e = launch_grad_reduce(part, d_b1, d_nx_w, d_nx_b, d_ng_w, d_ng_b, static_cast<int>(f.P), static_cast<int>(f.L),
                           static_cast<int>(H), bl.nsplit, dev, s);
    if (e != cudaSuccess) return cuda_fail(e, "gradient reduction launch");
  }

  if (d_inputs) {
    // (6) dX_t = dZ_t @ w1_t^T, stored at the rows dispatch read from (inverse permutation)
    CUtensorMap mdz_k, mw1_k, mdx;
    if ((st = make_map_3d(&mdz_k, true, dZ, 2 * H, M, T, 2 * H * 2, M * 2 * H * 2, 64, 128, 1, "dZ")) != DG_OK)
      return st;
    if ((st = make_map_3d(&mw1_k, true, w1, 2 * H, D, T, 2 * H * 2, D * 2 * H * 2, 64, kKMajorBRows, 1,
                          "w1 (K-major)")) != DG_OK)
      return st;
    if ((st = make_map_3d(&mdx, true, dx_out, D, T, M, D * 2, T * D * 2, 64, 1, 32, "d_inputs")) != DG_OK) return st;
    GemmParams p{};
    p.G = static_cast<int32_t>(T);
    p.M = static_cast<int32_t>(M);
    p.N = static_cast<int32_t>(D);
    p.K = static_cast<int32_t>(2 * H);
    p.a_g = G_OUTER;
    p.b_g = G_OUTER;
    p.d_g = G_MID;
    if ((st = run_gemm(GV_BF16_KK_STORE, mdz_k, mw1_k, mdx, mdx, p, dev, s, "ffn_bwd_dx",
                       2.0 * (rows * 2 * H + static_cast<double>(T) * D * 2 * H + rows * D))) != DG_OK)
      return st;
  }

  if (d_w1) {
    // (7) dw1_t = Xlocal_t^T @ dZ_t   [D, 2H], contraction over the M rows
    CUtensorMap mx_t, mdz_n, mdw1;
    int32_t xt_mn4 = 0, dzn_mn4 = 0;
    if ((st = make_map_mn(&mx_t, x_in, D, T, M, D * 2, T * D * 2, 1, 64, kMnBlocksA, &xt_mn4, "inputs^T")) != DG_OK)
      return st;
    if ((st = make_map_mn(&mdz_n, dZ, 2 * H, M, T, 2 * H * 2, M * 2 * H * 2, 64, 1, kMnBlocksB, &dzn_mn4,
                          "dZ (N-major)")) != DG_OK)
      return st;
    if ((st = make_map_3d(&mdw1, true, d_w1, 2 * H, D, T, 2 * H * 2, D * 2 * H * 2, 64, 32, 1, "d_w1")) != DG_OK)
      return st;
    GemmParams p{};
    p.G = static_cast<int32_t>(T);
    p.M = static_cast<int32_t>(D);
    p.N = static_cast<int32_t>(2 * H);
    p.K = static_cast<int32_t>(M);
    p.a_g = G_MID;
    p.b_g = G_OUTER;
    p.d_g = G_OUTER;
    p.a_mn4 = xt_mn4;
    p.b_mn4 = dzn_mn4;
    if ((st = run_gemm(GV_BF16_MM_STORE, mx_t, mdz_n, mdw1, mdw1, p, dev, s, "ffn_bwd_dw1",
                       2.0 * (rows * D + rows * 2 * H + static_cast<double>(T) * D * 2 * H))) != DG_OK)
      return st;
  }

  if ((flags & DG_FFN_COMP_ONLY) && d_inputs) {
    TraceScope trace("ffn_comp_only_swap", s, 0.0, 2.0 * act);
    e = launch_swap_rank_slice(dx_out, d_inputs, static_cast<int>(f.P), static_cast<int>(f.B), static_cast<int>(T),
                               static_cast<int>(D), dev, s);
    if (e != cudaSuccess) return cuda_fail(e, "comp_only d_inputs swap launch");
  }
  return DG_OK;
}

dg_status dg_a2a_dispatch(int32_t P, int32_t B, int32_t T, int32_t D, const void* inputs, void* xlocal,
                          void* stream) {
  if (P < 1 || B < 1 || T < 1 || D < 1 || T % P || D % 8)
    return fail(DG_ERR_INVALID_ARGUMENT, "a2a_dispatch: need P,B,T,D >= 1, T %% P == 0, D %% 8 == 0");
  if (!inputs || !xlocal || !aligned16(inputs) || !aligned16(xlocal))
    return fail(DG_ERR_INVALID_ARGUMENT, "a2a_dispatch: NULL or unaligned pointer");
  const size_t bytes = static_cast<size_t>(P) * B * T * D * 2;
  if (overlaps(inputs, bytes, xlocal, bytes)) return fail(DG_ERR_INVALID_ARGUMENT, "a2a_dispatch: in-place not supported");
  DeviceInfo dev;
  dg_status st = device_info(&dev);
  if (st != DG_OK) return st;
  TraceScope trace("a2a_dispatch", static_cast<cudaStream_t>(stream), 0.0, 2.0 * bytes);
  cudaError_t e = launch_dispatch(inputs, xlocal, P, B, T, D, dev, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? DG_OK : cuda_fail(e, "dispatch launch");
}

dg_status dg_a2a_combine(int32_t P, int32_t B, int32_t T, int32_t D, const void* ylocal, void* output,
                         void* stream) {
  if (P < 1 || B < 1 || T < 1 || D < 1 || T % P || D % 8)
    return fail(DG_ERR_INVALID_ARGUMENT, "a2a_combine: need P,B,T,D >= 1, T %% P == 0, D %% 8 == 0");
  if (!ylocal || !output || !aligned16(ylocal) || !aligned16(output))
    return fail(DG_ERR_INVALID_ARGUMENT, "a2a_combine: NULL or unaligned pointer");
  const size_t bytes = static_cast<size_t>(P) * B * T * D * 2;
  if (overlaps(ylocal, bytes, output, bytes)) return fail(DG_ERR_INVALID_ARGUMENT, "a2a_combine: in-place not supported");
  DeviceInfo dev;
  dg_status st = device_info(&dev);
  if (st != DG_OK) return st;
  TraceScope trace("a2a_combine", static_cast<cudaStream_t>(stream), 0.0, 2.0 * bytes);
  cudaError_t e = launch_combine(ylocal, output, P, B, T, D, dev, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? DG_OK : cuda_fail(e, "combine launch");
}

// ------------------------------------------------------------------ A2A FFN, FP8 GEMMs (forward)

namespace {

// e4m3 copy of the weights: w1 codes [T][2H][D] and scales [T][2H], wout codes
// [T][D][H] and scales [T][D] (codes K-major for the GEMMs' B operands).
struct Fp8WeightsLayout {
  size_t w1q, s1, woq, so, i1, io, total;
};
Fp8WeightsLayout fp8_weights_layout(const FfnDims& f) {
  Fp8WeightsLayout l;
  const size_t T = f.T, D = f.D, H = f.H;
  l.w1q = 0;
  l.s1 = round_up(T * 2 * H * D, 256);
  l.woq = round_up(l.s1 + T * 2 * H * 4, 256);
  l.so = round_up(l.woq + T * D * H, 256);
  l.i1 = round_up(l.so + T * D * 4, 256);  // inverse scales, used while packing
  l.io = round_up(l.i1 + T * 2 * H * 4, 256);
  l.total = round_up(l.io + T * D * 4, 256);
  return l;
}

// Forward workspace: the error block; input codes [P,B,T,D] and row scales [T,M]; Z [T,M,2H]
// bf16, the per-tile LayerNorm partials and the row statistics (as in the
// bf16 forward); Hl codes [T,M,H] and row scales [T,M].
struct Fp8FwdLayout {
  size_t xq, sx, z, part, stats, hq, sh, total;
  int tiles_n;
};
Fp8FwdLayout fp8_fwd_layout(const FfnDims& f) {
  Fp8FwdLayout l;
  const size_t rows = static_cast<size_t>(f.T) * f.M;
  l.tiles_n = static_cast<int>((2 * f.H + gemm_tile_n(GV_FP8_KK_LNSTATS) - 1) / gemm_tile_n(GV_FP8_KK_LNSTATS));
  l.xq = DG_ERROR_BLOCK_BYTES;
  l.sx = round_up(l.xq + rows * f.D, 256);
  l.z = round_up(l.sx + rows * 4, 256);
  l.part = round_up(l.z + rows * 2 * f.H * 2, 256);
  l.stats = round_up(l.part + rows * l.tiles_n * 16, 256);
  l.hq = round_up(l.stats + rows * 16, 256);
  l.sh = round_up(l.hq + rows * f.H, 256);
  l.total = round_up(l.sh + rows * 4, 256);
  return l;
}

dg_status check_fp8_shape(const dg_ffn_shape* shape, FfnDims* f, const char* what) {
  dg_status st = check_ffn_shape(shape, f);
  if (st != DG_OK) return st;
  if (f->D % 16 || f->H % 16)
    return fail(DG_ERR_INVALID_ARGUMENT, "%s: D and H = D*k must be multiples of 16 (16-byte e4m3 rows)", what);
  if (f->H > 8192) return fail(DG_ERR_UNSUPPORTED, "%s: H = %lld > 8192 (an e4m3 Hl row is scaled in one CTA)", what,
                               (long long)f->H);
  return DG_OK;
}

}  // namespace

size_t dg_a2a_ffn_fp8_weights_bytes(const dg_ffn_shape* shape) {
  FfnDims f{};
  if (check_fp8_shape(shape, &f, "a2a_ffn_fp8_weights_bytes") != DG_OK) return 0;
  return fp8_weights_layout(f).total;
}

size_t dg_a2a_ffn_fp8_workspace_bytes(const dg_ffn_shape* shape) {
  FfnDims f{};
  if (check_fp8_shape(shape, &f, "a2a_ffn_fp8_workspace_bytes") != DG_OK) return 0;
  return fp8_fwd_layout(f).total;
}

dg_status dg_a2a_ffn_fp8_pack_weights(const dg_ffn_shape* shape, const void* w1, const void* wout, void* packed,
                                      size_t packed_bytes, void* stream) {
  FfnDims f{};
  dg_status st = check_fp8_shape(shape, &f, "a2a_ffn_fp8_pack_weights");
  if (st != DG_OK) return st;
  const void* ptrs[] = {w1, wout, packed};
  const char* names[] = {"w1", "wout", "packed"};
  if (const char* n = ptr_name_null(ptrs, names, 3))
    return fail(DG_ERR_INVALID_ARGUMENT, "a2a_ffn_fp8_pack_weights: %s is NULL", n);
  if (const char* n = ptr_name_unaligned(ptrs, names, 3))
    return fail(DG_ERR_INVALID_ARGUMENT, "a2a_ffn_fp8_pack_weights: %s is not 16-byte aligned", n);
  const Fp8WeightsLayout wl = fp8_weights_layout(f);
  if (packed_bytes < wl.total)
    return fail(DG_ERR_WORKSPACE, "a2a_ffn_fp8_pack_weights: packed buffer has %zu bytes, needs %zu", packed_bytes,
                wl.total);
  const size_t wbytes = static_cast<size_t>(f.T) * f.D * 2 * f.H * 2, wobytes = static_cast<size_t>(f.T) * f.H * f.D * 2;
  if (overlaps(packed, wl.total, w1, wbytes) || overlaps(packed, wl.total, wout, wobytes))
    return fail(DG_ERR_INVALID_ARGUMENT, "a2a_ffn_fp8_pack_weights: packed overlaps a weight");
  DeviceInfo dev;
  if ((st = device_info(&dev)) != DG_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* pk = static_cast<uint8_t*>(packed);
  cudaError_t e;
  {
    TraceScope trace("ffn_fp8_pack_w1", s, 0.0, 2.0 * wbytes);
    e = launch_quant_weight(w1, reinterpret_cast<float*>(pk + wl.s1), reinterpret_cast<float*>(pk + wl.i1),
                            pk + wl.w1q, static_cast<int>(f.T), static_cast<int>(f.D), static_cast<int>(2 * f.H), dev, s);
  }
  if (e != cudaSuccess) return cuda_fail(e, "w1 quantisation launch");
  {
    TraceScope trace("ffn_fp8_pack_wout", s, 0.0, 2.0 * wobytes);
    e = launch_quant_weight(wout, reinterpret_cast<float*>(pk + wl.so), reinterpret_cast<float*>(pk + wl.io),
                            pk + wl.woq, static_cast<int>(f.T), static_cast<int>(f.H), static_cast<int>(f.D), dev, s);
  }
  return e == cudaSuccess ? DG_OK : cuda_fail(e, "wout quantisation launch");
}

dg_status dg_a2a_ffn_fwd_fp8(const dg_ffn_shape* shape, const void* inputs, const void* packed, size_t packed_bytes,
                             const void* b1, const void* bout, const void* nx_w, const void* nx_b, const void* ng_w,
                             const void* ng_b, void* output, void* ws, size_t ws_bytes, void* stream) {
  FfnDims f{};
  dg_status st = check_fp8_shape(shape, &f, "a2a_ffn_fwd_fp8");
  if (st != DG_OK) return st;
  const void* ptrs[] = {inputs, packed, b1, bout, nx_w, nx_b, ng_w, ng_b, output, ws};
  const char* names[] = {"inputs", "packed", "b1", "bout", "nx_w", "nx_b", "ng_w", "ng_b", "output", "ws"};
  if (const char* n = ptr_name_null(ptrs, names, 10))
    return fail(DG_ERR_INVALID_ARGUMENT, "a2a_ffn_fwd_fp8: %s is NULL", n);
  if (const char* n = ptr_name_unaligned(ptrs, names, 10))
    return fail(DG_ERR_INVALID_ARGUMENT, "a2a_ffn_fwd_fp8: %s is not 16-byte aligned", n);
  const Fp8WeightsLayout wl = fp8_weights_layout(f);
  const Fp8FwdLayout fl = fp8_fwd_layout(f);
  if (packed_bytes < wl.total)
    return fail(DG_ERR_WORKSPACE, "a2a_ffn_fwd_fp8: packed weights have %zu bytes, need %zu", packed_bytes, wl.total);
  if (ws_bytes < fl.total)
    return fail(DG_ERR_WORKSPACE, "a2a_ffn_fwd_fp8: workspace has %zu bytes, needs %zu", ws_bytes, fl.total);
  const size_t act = static_cast<size_t>(f.P) * f.B * f.T * f.D * 2;
  if (overlaps(output, act, inputs, act) || overlaps(output, act, ws, fl.total) || overlaps(ws, fl.total, inputs, act) ||
      overlaps(ws, fl.total, packed, wl.total) || overlaps(output, act, packed, wl.total))
    return fail(DG_ERR_INVALID_ARGUMENT, "a2a_ffn_fwd_fp8: output / workspace / inputs / packed weights overlap");
  DeviceInfo dev;
  if ((st = device_info_ws(&dev, ws, ws_bytes, "a2a_ffn_fwd_fp8")) != DG_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const uint8_t* pk = static_cast<const uint8_t*>(packed);
  uint8_t* w = static_cast<uint8_t*>(ws);
  const uint64_t T = f.T, M = f.M, D = f.D, H = f.H;
  const double rows = static_cast<double>(T) * M;
  cudaError_t e;

  // e4m3 input rows, one scale per row
  {
    TraceScope trace("ffn_fp8_quant_inputs", s, 0.0, rows * D * 2.0 + rows * D + rows * 4.0);
    e = launch_quant_rows(inputs, w + fl.xq, reinterpret_cast<float*>(w + fl.sx), static_cast<int64_t>(T * M),
                          static_cast<int>(D), static_cast<int>(T), static_cast<int>(M), dev, s);
  }
  if (e != cudaSuccess) return cuda_fail(e, "input quantisation launch");

  // GEMM1 on e4m3 operands (dispatch folded into the input map), dequantised in
  // the epilogue, + b1, LayerNorm partial statistics, bf16 Z.
  CUtensorMap mx, mw1, mz;
  if ((st = make_map_3d(&mx, false, w + fl.xq, D, T, M, D, T * D, 128, 1, 128, "input codes")) != DG_OK) return st;
  if ((st = make_map_3d(&mw1, false, pk + wl.w1q, D, 2 * H, T, D, 2 * H * D, 128, kKMajorBRows, 1, "w1 codes")) != DG_OK)
    return st;
  if ((st = make_map_3d(&mz, true, w + fl.z, 2 * H, M, T, 2 * H * 2, M * 2 * H * 2, 64, 32, 1, "Z")) != DG_OK) return st;
  GemmParams p1{};
  p1.G = static_cast<int32_t>(T);
  p1.M = static_cast<int32_t>(M);
  p1.N = static_cast<int32_t>(2 * H);
  p1.K = static_cast<int32_t>(D);
  p1.a_g = G_MID;
  p1.b_g = G_OUTER;
  p1.d_g = G_OUTER;
  p1.bias = static_cast<const __nv_bfloat16*>(b1);
  p1.bias_g_stride = static_cast<int64_t>(2 * H);
  p1.ln_part = reinterpret_cast<float4*>(w + fl.part);
  p1.ln_H = static_cast<int32_t>(H);
  p1.row_scale = reinterpret_cast<const float*>(w + fl.sx);
  p1.row_scale_g = static_cast<int64_t>(M);
  p1.col_scale = reinterpret_cast<const float*>(pk + wl.s1);
  p1.col_scale_g = static_cast<int64_t>(2 * H);
  if ((st = run_gemm(GV_FP8_KK_LNSTATS, mx, mw1, mz, mz, p1, dev, s, "ffn_fp8_gemm1",
                     rows * D + static_cast<double>(T) * D * 2 * H + rows * 2 * H * 2 + rows * 4 +
                         rows * fl.tiles_n * 16.0)) != DG_OK)
    return st;

  {
    TraceScope trace("ffn_fp8_ln_stats", s, 0.0, rows * fl.tiles_n * 16.0 + rows * 16.0);
    e = launch_ln_stats_finalize(reinterpret_cast<const float4*>(w + fl.part), w + fl.stats, static_cast<int>(T),
                                 static_cast<int>(M), static_cast<int>(H), gemm_tile_n(GV_FP8_KK_LNSTATS), fl.tiles_n,
                                 shape->eps, dev, s);
  }
  if (e != cudaSuccess) return cuda_fail(e, "LayerNorm statistics launch");
  {
    TraceScope trace("ffn_fp8_ln_gate", s, 0.0, rows * (2.0 * 2 * H + H + 16.0 + 4.0));
    e = launch_ln_gate_fwd(w + fl.z, w + fl.stats, nx_w, nx_b, ng_w, ng_b, nullptr, w + fl.hq,
                           reinterpret_cast<float*>(w + fl.sh), static_cast<int>(f.P), static_cast<int>(M),
                           static_cast<int>(f.L), static_cast<int>(H), dev, s);
  }
  if (e != cudaSuccess) return cuda_fail(e, "LayerNorm-gate launch");

  // GEMM2 on e4m3 operands, dequantised, + bout, stored at the combine offsets.
  CUtensorMap mh, mwo, mo;
  if ((st = make_map_3d(&mh, false, w + fl.hq, H, M, T, H, M * H, 128, 128, 1, "Hl codes")) != DG_OK) return st;
  if ((st = make_map_3d(&mwo, false, pk + wl.woq, H, D, T, H, D * H, 128, kKMajorBRows, 1, "wout codes")) != DG_OK)
    return st;
  if ((st = make_map_3d(&mo, true, output, D, T, M, D * 2, T * D * 2, 64, 1, 32, "output")) != DG_OK) return st;
  GemmParams p2{};
  p2.G = static_cast<int32_t>(T);
  p2.M = static_cast<int32_t>(M);
  p2.N = static_cast<int32_t>(D);
  p2.K = static_cast<int32_t>(H);
  p2.a_g = G_OUTER;
  p2.b_g = G_OUTER;
  p2.d_g = G_MID;
  p2.bias = static_cast<const __nv_bfloat16*>(bout);
  p2.bias_g_stride = static_cast<int64_t>(D);
  p2.row_scale = reinterpret_cast<const float*>(w + fl.sh);
  p2.row_scale_g = static_cast<int64_t>(M);
  p2.col_scale = reinterpret_cast<const float*>(pk + wl.so);
  p2.col_scale_g = static_cast<int64_t>(D);
  return run_gemm(GV_FP8_KK_BIAS, mh, mwo, mo, mo, p2, dev, s, "ffn_fp8_gemm2",
                  rows * H + static_cast<double>(T) * H * D + rows * D * 2.0 + rows * 4);
}

// ------------------------------------------------------------------ TP SwiGLU

size_t dg_tp_swiglu_workspace_bytes(int64_t S, int64_t d, int64_t ffn, int32_t W, int32_t bsz) {
  if (S < 1 || d < 1 || ffn < 1 || W < 1 || bsz < 1 || S % W || ffn % W) return 0;
  // the error block, then h [S*bsz, ffn] bf16
  return DG_ERROR_BLOCK_BYTES + round_up(static_cast<size_t>(S) * bsz * ffn * 2, 256);
}

}  // extern "C"

namespace dg {

dg_status tp_swiglu_check_sizes(int64_t S, int64_t d, int64_t ffn, int32_t W, int32_t bsz, const char* what) {
  if (S < 1 || d < 1 || ffn < 1 || W < 1 || bsz < 1)
    return fail(DG_ERR_INVALID_ARGUMENT, "%s: S, d, ffn, W, bsz must be >= 1", what);
  if (S % W || ffn % W) return fail(DG_ERR_INVALID_ARGUMENT, "%s: S and ffn must be divisible by W", what);
  const int64_t F = ffn / W;
  if (d % 8 || F % 8) return fail(DG_ERR_INVALID_ARGUMENT, "%s: d and ffn/W must be multiples of 8", what);
  if (S > 0x7fffffff || ffn > 0x7fffffff || d > 0x7fffffff || S > 0x7fffffff / bsz)
    return fail(DG_ERR_UNSUPPORTED, "%s: sizes beyond 2^31-1", what);
  return DG_OK;
}

dg_status tp_swiglu_check(int64_t S, int64_t d, int64_t ffn, int32_t W, int32_t bsz, const void* x_shards,
                          const void* w13, const void* w2, const void* y_shards, const void* scratch,
                          size_t scratch_bytes, const char* what) {
  dg_status st = tp_swiglu_check_sizes(S, d, ffn, W, bsz, what);
  if (st != DG_OK) return st;
  const int64_t rows = S * bsz;
  const void* ptrs[] = {x_shards, w13, w2, y_shards};
  const char* names[] = {"x_shards", "w13", "w2", "y_shards"};
  if (const char* n = ptr_name_null(ptrs, names, 4)) return fail(DG_ERR_INVALID_ARGUMENT, "%s: %s is NULL", what, n);
  if (const char* n = ptr_name_unaligned(ptrs, names, 4))
    return fail(DG_ERR_INVALID_ARGUMENT, "%s: %s is not 16-byte aligned", what, n);
  const size_t act = static_cast<size_t>(rows) * d * 2;
  const size_t wb = static_cast<size_t>(2) * ffn * d * 2, w2b = static_cast<size_t>(ffn) * d * 2;
  if (overlaps(y_shards, act, x_shards, act) || overlaps(y_shards, act, w13, wb) || overlaps(y_shards, act, w2, w2b))
    return fail(DG_ERR_INVALID_ARGUMENT, "%s: y_shards overlaps an input", what);
  if (overlaps(scratch, scratch_bytes, y_shards, act) || overlaps(scratch, scratch_bytes, x_shards, act) ||
      overlaps(scratch, scratch_bytes, w13, wb) || overlaps(scratch, scratch_bytes, w2, w2b))
    return fail(DG_ERR_INVALID_ARGUMENT, "%s: the workspace overlaps a tensor", what);
  return DG_OK;
}

}  // namespace dg

extern "C" {

dg_status dg_tp_swiglu(int64_t S, int64_t d, int64_t ffn, int32_t W, int32_t bsz, const void* x_shards,
                       const void* w13, const void* w2, void* y_shards, void* ws, size_t ws_bytes, void* stream) {
  const size_t need = dg_tp_swiglu_workspace_bytes(S, d, ffn, W, bsz);
  dg_status st = tp_swiglu_check(S, d, ffn, W, bsz, x_shards, w13, w2, y_shards, ws, need, "tp_swiglu");
  if (st != DG_OK) return st;
  if (!ws) return fail(DG_ERR_WORKSPACE, "tp_swiglu: ws is NULL");
  if (!aligned16(ws)) return fail(DG_ERR_INVALID_ARGUMENT, "tp_swiglu: ws is not 16-byte aligned");
  if (ws_bytes < need) return fail(DG_ERR_WORKSPACE, "tp_swiglu: workspace has %zu bytes, needs %zu", ws_bytes, need);
  DeviceInfo dev;
  if ((st = device_info_ws(&dev, ws, ws_bytes, "tp_swiglu")) != DG_OK) return st;
  return tp_swiglu_enqueue(S, d, ffn, W, bsz, x_shards, w13, w2, y_shards,
                           static_cast<uint8_t*>(ws) + DG_ERROR_BLOCK_BYTES, dev, static_cast<cudaStream_t>(stream),
                           true);
}

}  // extern "C"

namespace dg {

dg_status tp_swiglu_enqueue(int64_t S, int64_t d, int64_t ffn, int32_t W, int32_t bsz, const void* x_shards,
                            const void* w13, const void* w2, void* y_shards, void* h, const DeviceInfo& dev,
                            cudaStream_t s, bool traced) {
  dg_status st;
  const int64_t F = ffn / W;
  const uint64_t R = static_cast<uint64_t>(S) * bsz, Dm = d, Fu = F, Wu = W, FF = ffn;

  // GEMM1 over all shards: h[:, s*F + c] = silu(X w1_s[c]) * (X w3_s[c]).  The
  // gathered X is the rows of x_shards in memory order (rank, batch, seq_local).
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
  p.b_g = G_OUTER;  // unused: the paired load addresses w13 directly
  p.d_g = G_MID;
  if ((st = run_gemm(GV_BF16_KK_SWIGLU, mx, mw13, mh, mh, p, dev, s, traced ? "tp_gemm1_swiglu" : nullptr,
                     2.0 * (static_cast<double>(R) * Dm + 2.0 * FF * Dm + static_cast<double>(R) * FF))) != DG_OK)
    return st;

  // GEMM2: y = sum_s h_s @ w2_s^T = h @ w2^T; the shard sum is the K loop.
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
  return run_gemm(GV_BF16_KK_STORE, mh_k, mw2, my, my, p, dev, s, traced ? "tp_gemm2" : nullptr,
                  2.0 * (static_cast<double>(R) * FF + static_cast<double>(Dm) * FF + static_cast<double>(R) * Dm));
}

}  // namespace dg

extern "C" {

size_t dg_tp_swiglu_bwd_workspace_bytes(int64_t S, int64_t d, int64_t ffn, int32_t W, int32_t bsz) {
  if (S < 1 || d < 1 || ffn < 1 || W < 1 || bsz < 1 || S % W || ffn % W) return 0;
  // the error block; [a|b] (later [da|db]) is [rows, 2*ffn]; dh (later h) is [rows, ffn].
  return DG_ERROR_BLOCK_BYTES + 3 * round_up(static_cast<size_t>(S) * bsz * ffn * 2, 256);
}

dg_status dg_tp_swiglu_bwd(int64_t S, int64_t d, int64_t ffn, int32_t W, int32_t bsz, const void* x_shards,
                           const void* w13, const void* w2, const void* dy_shards, void* dx_shards, void* d_w13,
                           void* d_w2, void* ws, size_t ws_bytes, void* stream) {
  if (S < 1 || d < 1 || ffn < 1 || W < 1 || bsz < 1)
    return fail(DG_ERR_INVALID_ARGUMENT, "tp_swiglu_bwd: S, d, ffn, W, bsz must be >= 1");
  if (S % W || ffn % W) return fail(DG_ERR_INVALID_ARGUMENT, "tp_swiglu_bwd: S and ffn must be divisible by W");
  const int64_t F = ffn / W;
  if (d % 8 || F % 8) return fail(DG_ERR_INVALID_ARGUMENT, "tp_swiglu_bwd: d and ffn/W must be multiples of 8");
  const int64_t rows = S * bsz;
  if (rows > 0x7fffffff || 2 * ffn > 0x7fffffff || d > 0x7fffffff)
    return fail(DG_ERR_UNSUPPORTED, "tp_swiglu_bwd: sizes beyond 2^31-1");
  const void* ptrs[] = {x_shards, w13, w2, dy_shards, dx_shards, d_w13, d_w2, ws};
  const char* names[] = {"x_shards", "w13", "w2", "dy_shards", "dx_shards", "d_w13", "d_w2", "ws"};
  if (const char* n = ptr_name_null(ptrs, names, 8))
    return fail(DG_ERR_INVALID_ARGUMENT, "tp_swiglu_bwd: %s is NULL", n);
  if (const char* n = ptr_name_unaligned(ptrs, names, 8))
    return fail(DG_ERR_INVALID_ARGUMENT, "tp_swiglu_bwd: %s is not 16-byte aligned", n);
  const size_t need = dg_tp_swiglu_bwd_workspace_bytes(S, d, ffn, W, bsz);
  if (ws_bytes < need)
    return fail(DG_ERR_WORKSPACE, "tp_swiglu_bwd: workspace has %zu bytes, needs %zu", ws_bytes, need);
  const size_t act = static_cast<size_t>(rows) * d * 2;
  const size_t wbytes = static_cast<size_t>(2) * ffn * d * 2, w2bytes = static_cast<size_t>(ffn) * d * 2;
  // Every written region (dx, d_w13, d_w2, ws) must be disjoint from every
  // other region, read or written.
  const void* wr[] = {dx_shards, d_w13, d_w2, ws};
  const size_t wr_n[] = {act, wbytes, w2bytes, need};
  const void* all[] = {x_shards, w13, w2, dy_shards, dx_shards, d_w13, d_w2, ws};
  const size_t all_n[] = {act, wbytes, w2bytes, act, act, wbytes, w2bytes, need};
  for (int i = 0; i < 4; ++i)
    for (int j = 0; j < 8; ++j)
      if (j != 4 + i && overlaps(wr[i], wr_n[i], all[j], all_n[j]))
        return fail(DG_ERR_INVALID_ARGUMENT, "tp_swiglu_bwd: %s overlaps %s", names[4 + i], names[j]);
  DeviceInfo dev;
  dg_status st = device_info_ws(&dev, ws, ws_bytes, "tp_swiglu_bwd");
  if (st != DG_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const uint64_t R = rows, Dm = d, FF = ffn, F2 = 2 * ffn;
  const size_t ab_bytes = round_up(static_cast<size_t>(rows) * ffn * 2, 256) * 2;
  void* ab = static_cast<unsigned char*>(ws) + DG_ERROR_BLOCK_BYTES;  // [R, W, 2F]: (a_s | b_s), then (da_s | db_s)
  void* dh = static_cast<unsigned char*>(ab) + ab_bytes;              // [R, ffn]: dh, then h
  const double r = static_cast<double>(R), dd = static_cast<double>(Dm), ff = static_cast<double>(FF);

  // 1. Recompute the gate inputs of all shards at once: [a | b] = X [w1_s ; w3_s]^T,
  //    w13 read as one [2*ffn, d] matrix whose rows are ordered (shard, w1|w3, c).
  CUtensorMap mx_k, mw13_k, mab;
  if ((st = make_map_3d(&mx_k, true, x_shards, Dm, R, 1, Dm * 2, R * Dm * 2, 64, 128, 1, "x_shards")) != DG_OK) return st;
  if ((st = make_map_3d(&mw13_k, true, w13, Dm, F2, 1, Dm * 2, F2 * Dm * 2, 64, kKMajorBRows, 1, "w13")) != DG_OK)
    return st;
  if ((st = make_map_3d(&mab, true, ab, F2, R, 1, F2 * 2, R * F2 * 2, 64, 32, 1, "[a|b]")) != DG_OK) return st;
  GemmParams p{};
  p.G = 1;
  p.M = static_cast<int32_t>(R);
  p.N = static_cast<int32_t>(F2);
  p.K = static_cast<int32_t>(d);
  p.a_g = p.b_g = p.d_g = G_OUTER;
  if ((st = run_gemm(GV_BF16_KK_STORE, mx_k, mw13_k, mab, mab, p, dev, s, "tp_bwd_ab",
                     2.0 * (r * dd + 2.0 * ff * dd + 2.0 * r * ff))) != DG_OK)
    return st;

  // 2. dh = dY w2 (w2 [d, ffn] read N-major: the gradient of y = h w2^T w.r.t. h).
  CUtensorMap mdy_k, mw2_n, mdh;
  if ((st = make_map_3d(&mdy_k, true, dy_shards, Dm, R, 1, Dm * 2, R * Dm * 2, 64, 128, 1, "dy_shards")) != DG_OK)
    return st;
  int32_t w2n_mn4 = 0;
  if ((st = make_map_mn(&mw2_n, w2, FF, Dm, 1, FF * 2, Dm * FF * 2, 64, 1, kMnBlocksB, &w2n_mn4, "w2 (N-major)")) != DG_OK)
    return st;
  if ((st = make_map_3d(&mdh, true, dh, FF, R, 1, FF * 2, R * FF * 2, 64, 32, 1, "dh")) != DG_OK) return st;
  p = GemmParams{};
  p.G = 1;
  p.M = static_cast<int32_t>(R);
  p.N = static_cast<int32_t>(ffn);
  p.K = static_cast<int32_t>(d);
  p.a_g = p.b_g = p.d_g = G_OUTER;
  p.b_mn4 = w2n_mn4;
  if ((st = run_gemm(GV_BF16_KM_STORE, mdy_k, mw2_n, mdh, mdh, p, dev, s, "tp_bwd_dh",
                     2.0 * (r * dd + ff * dd + r * ff))) != DG_OK)
    return st;

  // 3. Gate backward, in place: [a|b] -> [da|db], dh -> h.
  {
    TraceScope trace("tp_bwd_gate", s, 0.0, 12.0 * r * ff);
    cudaError_t e = launch_swiglu_gate_bwd(ab, dh, rows, W, static_cast<int>(F), dev, s);
    if (e != cudaSuccess) return cuda_fail(e, "tp_bwd_gate launch");
  }

  // 4. d_w2 = dY^T h: [d, ffn], contraction over the gathered rows.
  CUtensorMap mdy_t, mh_n, mdw2;
  int32_t dyt_mn4 = 0, hn_mn4 = 0;
  if ((st = make_map_mn(&mdy_t, dy_shards, Dm, R, 1, Dm * 2, R * Dm * 2, 64, 1, kMnBlocksA, &dyt_mn4, "dy^T")) != DG_OK)
    return st;
  if ((st = make_map_mn(&mh_n, dh, FF, R, 1, FF * 2, R * FF * 2, 64, 1, kMnBlocksB, &hn_mn4, "h (N-major)")) != DG_OK)
    return st;
  if ((st = make_map_3d(&mdw2, true, d_w2, FF, Dm, 1, FF * 2, Dm * FF * 2, 64, 32, 1, "d_w2")) != DG_OK) return st;
  p = GemmParams{};
  p.G = 1;
  p.M = static_cast<int32_t>(d);
  p.N = static_cast<int32_t>(ffn);
  p.K = static_cast<int32_t>(R);
  p.a_g = p.b_g = p.d_g = G_OUTER;
  p.a_mn4 = dyt_mn4;
  p.b_mn4 = hn_mn4;
  if ((st = run_gemm(GV_BF16_MM_STORE, mdy_t, mh_n, mdw2, mdw2, p, dev, s, "tp_bwd_dw2",
                     2.0 * (r * dd + r * ff + dd * ff))) != DG_OK)
    return st;

  // 5. dX = [da|db] [w1_s ; w3_s] over all shards at once: one product with
  //    K = 2*ffn, so the shard sum (the row-parallel reduction) is the K loop.
  CUtensorMap mdab_k, mw13_n, mdx;
  if ((st = make_map_3d(&mdab_k, true, ab, F2, R, 1, F2 * 2, R * F2 * 2, 64, 128, 1, "[da|db]")) != DG_OK) return st;
  int32_t w13n_mn4 = 0;
  if ((st = make_map_mn(&mw13_n, w13, Dm, F2, 1, Dm * 2, F2 * Dm * 2, 64, 1, kMnBlocksB, &w13n_mn4, "w13 (N-major)")) !=
      DG_OK)
    return st;
  if ((st = make_map_3d(&mdx, true, dx_shards, Dm, R, 1, Dm * 2, R * Dm * 2, 64, 32, 1, "dx_shards")) != DG_OK) return st;
  p = GemmParams{};
  p.G = 1;
  p.M = static_cast<int32_t>(R);
  p.N = static_cast<int32_t>(d);
  p.K = static_cast<int32_t>(F2);
  p.a_g = p.b_g = p.d_g = G_OUTER;
  p.b_mn4 = w13n_mn4;
  if ((st = run_gemm(GV_BF16_KM_STORE, mdab_k, mw13_n, mdx, mdx, p, dev, s, "tp_bwd_dx",
                     2.0 * (2.0 * r * ff + 2.0 * ff * dd + r * dd))) != DG_OK)
    return st;

  // 6. d_w13 = [da|db]^T X: [2*ffn, d] in w13's own row order.
  CUtensorMap mdab_t, mx_n, mdw13;
  int32_t dabt_mn4 = 0, xn_mn4 = 0;
  if ((st = make_map_mn(&mdab_t, ab, F2, R, 1, F2 * 2, R * F2 * 2, 64, 1, kMnBlocksA, &dabt_mn4, "[da|db]^T")) != DG_OK)
    return st;
  if ((st = make_map_mn(&mx_n, x_shards, Dm, R, 1, Dm * 2, R * Dm * 2, 64, 1, kMnBlocksB, &xn_mn4, "x (N-major)")) != DG_OK)
    return st;
  if ((st = make_map_3d(&mdw13, true, d_w13, Dm, F2, 1, Dm * 2, F2 * Dm * 2, 64, 32, 1, "d_w13")) != DG_OK) return st;
  p = GemmParams{};
  p.G = 1;
  p.M = static_cast<int32_t>(F2);
  p.N = static_cast<int32_t>(d);
  p.K = static_cast<int32_t>(R);
  p.a_g = p.b_g = p.d_g = G_OUTER;
  p.a_mn4 = dabt_mn4;
  p.b_mn4 = xn_mn4;
  return run_gemm(GV_BF16_MM_STORE, mdab_t, mx_n, mdw13, mdw13, p, dev, s, "tp_bwd_dw13",
                  2.0 * (2.0 * r * ff + r * dd + 2.0 * ff * dd));
}

// ------------------------------------------------------------------ TP linear (attention projections)

namespace {

dg_status check_linear(int64_t rows, int64_t in_f, int64_t out_f, const char* what) {
  if (rows < 1 || in_f < 1 || out_f < 1)
    return fail(DG_ERR_INVALID_ARGUMENT, "%s: rows, in_features, out_features must be >= 1", what);
  if (in_f % 8 || out_f % 8)
    return fail(DG_ERR_INVALID_ARGUMENT, "%s: in_features and out_features must be multiples of 8", what);
  if (rows > 0x7fffffff || in_f > 0x7fffffff || out_f > 0x7fffffff)
    return fail(DG_ERR_UNSUPPORTED, "%s: sizes beyond 2^31-1", what);
  return DG_OK;
}

}  // namespace

dg_status dg_tp_linear_fwd(int64_t rows, int64_t in_f, int64_t out_f, const void* x, const void* weight,
                           const void* bias, void* y, void* ws, size_t ws_bytes, void* stream) {
  dg_status st = check_linear(rows, in_f, out_f, "tp_linear_fwd");
  if (st != DG_OK) return st;
  const void* ptrs[] = {x, weight, y};
  const char* names[] = {"x", "weight", "y"};
  if (const char* n = ptr_name_null(ptrs, names, 3)) return fail(DG_ERR_INVALID_ARGUMENT, "tp_linear_fwd: %s is NULL", n);
  if (const char* n = ptr_name_unaligned(ptrs, names, 3))
    return fail(DG_ERR_INVALID_ARGUMENT, "tp_linear_fwd: %s is not 16-byte aligned", n);
  if (bias && !aligned16(bias)) return fail(DG_ERR_INVALID_ARGUMENT, "tp_linear_fwd: bias is not 16-byte aligned");
  const size_t xb = static_cast<size_t>(rows) * in_f * 2, wb = static_cast<size_t>(out_f) * in_f * 2;
  const size_t yb = static_cast<size_t>(rows) * out_f * 2;
  if (overlaps(y, yb, x, xb) || overlaps(y, yb, weight, wb) || (bias && overlaps(y, yb, bias, out_f * 2)) ||
      overlaps(y, yb, ws, DG_ERROR_BLOCK_BYTES))
    return fail(DG_ERR_INVALID_ARGUMENT, "tp_linear_fwd: y overlaps an input or the workspace");
  DeviceInfo dev;
  if ((st = device_info_ws(&dev, ws, ws_bytes, "tp_linear_fwd")) != DG_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const uint64_t R = rows, I = in_f, O = out_f;
  // y = x weight^T (+ bias): one K/K GEMM; every rank's feature block (column
  // parallel) or every rank's partial product (row parallel, summed in the K
  // loop) is part of it.
  CUtensorMap mx, mw, my;
  if ((st = make_map_3d(&mx, true, x, I, R, 1, I * 2, R * I * 2, 64, 128, 1, "x")) != DG_OK) return st;
  if ((st = make_map_3d(&mw, true, weight, I, O, 1, I * 2, O * I * 2, 64, kKMajorBRows, 1, "weight")) != DG_OK)
    return st;
  if ((st = make_map_3d(&my, true, y, O, R, 1, O * 2, R * O * 2, 64, 32, 1, "y")) != DG_OK) return st;
  GemmParams p{};
  p.G = 1;
  p.M = static_cast<int32_t>(rows);
  p.N = static_cast<int32_t>(out_f);
  p.K = static_cast<int32_t>(in_f);
  p.a_g = p.b_g = p.d_g = G_OUTER;
  p.bias = static_cast<const __nv_bfloat16*>(bias);
  p.bias_g_stride = 0;
  const double bytes = static_cast<double>(xb) + wb + yb + (bias ? 2.0 * out_f : 0.0);
  return run_gemm(bias ? GV_BF16_KK_BIAS : GV_BF16_KK_STORE, mx, mw, my, my, p, dev, s, "tp_linear_fwd", bytes);
}

size_t dg_tp_linear_workspace_bytes(int64_t rows, int64_t in_features, int64_t out_features) {
  (void)rows;
  (void)in_features;
  (void)out_features;
  return DG_ERROR_BLOCK_BYTES;
}

dg_status dg_tp_linear_bwd(int64_t rows, int64_t in_f, int64_t out_f, const void* x, const void* weight,
                           const void* dy, void* dx, void* d_weight, void* d_bias, void* ws, size_t ws_bytes,
                           void* stream) {
  dg_status st = check_linear(rows, in_f, out_f, "tp_linear_bwd");
  if (st != DG_OK) return st;
  const void* ptrs[] = {x, weight, dy};
  const char* names[] = {"x", "weight", "dy"};
  if (const char* n = ptr_name_null(ptrs, names, 3)) return fail(DG_ERR_INVALID_ARGUMENT, "tp_linear_bwd: %s is NULL", n);
  if (const char* n = ptr_name_unaligned(ptrs, names, 3))
    return fail(DG_ERR_INVALID_ARGUMENT, "tp_linear_bwd: %s is not 16-byte aligned", n);
  if ((dx && !aligned16(dx)) || (d_weight && !aligned16(d_weight)) || (d_bias && !aligned16(d_bias)))
    return fail(DG_ERR_INVALID_ARGUMENT, "tp_linear_bwd: an output is not 16-byte aligned");
  const size_t xb = static_cast<size_t>(rows) * in_f * 2, wb = static_cast<size_t>(out_f) * in_f * 2;
  const size_t yb = static_cast<size_t>(rows) * out_f * 2, bb = static_cast<size_t>(out_f) * 2;
  const void* outs[] = {dx, d_weight, d_bias, ws};
  const size_t outs_n[] = {xb, wb, bb, static_cast<size_t>(DG_ERROR_BLOCK_BYTES)};
  const void* all[] = {x, weight, dy, dx, d_weight, d_bias, ws};
  const size_t all_n[] = {xb, wb, yb, xb, wb, bb, static_cast<size_t>(DG_ERROR_BLOCK_BYTES)};
  for (int i = 0; i < 4; ++i)
    for (int j = 0; j < 7; ++j)
      if (outs[i] && all[j] && j != 3 + i && overlaps(outs[i], outs_n[i], all[j], all_n[j]))
        return fail(DG_ERR_INVALID_ARGUMENT, "tp_linear_bwd: outputs, workspace and inputs overlap");
  DeviceInfo dev;
  if ((st = device_info_ws(&dev, ws, ws_bytes, "tp_linear_bwd")) != DG_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const uint64_t R = rows, I = in_f, O = out_f;
  const double r = static_cast<double>(rows), fi = static_cast<double>(in_f), fo = static_cast<double>(out_f);
  if (dx) {
    // dx = dy weight: B = weight read N-major ([out, in], in contiguous)
    CUtensorMap mdy, mw, mdx;
    if ((st = make_map_3d(&mdy, true, dy, O, R, 1, O * 2, R * O * 2, 64, 128, 1, "dy")) != DG_OK) return st;
    int32_t w_mn4 = 0;
    if ((st = make_map_mn(&mw, weight, I, O, 1, I * 2, O * I * 2, 64, 1, kMnBlocksB, &w_mn4, "weight (N-major)")) !=
        DG_OK)
      return st;
    if ((st = make_map_3d(&mdx, true, dx, I, R, 1, I * 2, R * I * 2, 64, 32, 1, "dx")) != DG_OK) return st;
    GemmParams p{};
    p.G = 1;
    p.M = static_cast<int32_t>(rows);
    p.N = static_cast<int32_t>(in_f);
    p.K = static_cast<int32_t>(out_f);
    p.a_g = p.b_g = p.d_g = G_OUTER;
    p.b_mn4 = w_mn4;
    if ((st = run_gemm(GV_BF16_KM_STORE, mdy, mw, mdx, mdx, p, dev, s, "tp_linear_bwd_dx",
                       2.0 * (r * fo + fo * fi + r * fi))) != DG_OK)
      return st;
  }
  if (d_weight) {
    // d_weight = dy^T x: both operands MN-major, the contraction over rows
    CUtensorMap mdy_t, mx_n, mdw;
    int32_t dyt_mn4 = 0, xn_mn4 = 0;
    if ((st = make_map_mn(&mdy_t, dy, O, R, 1, O * 2, R * O * 2, 64, 1, kMnBlocksA, &dyt_mn4, "dy^T")) != DG_OK)
      return st;
    if ((st = make_map_mn(&mx_n, x, I, R, 1, I * 2, R * I * 2, 64, 1, kMnBlocksB, &xn_mn4, "x (N-major)")) != DG_OK)
      return st;
    if ((st = make_map_3d(&mdw, true, d_weight, I, O, 1, I * 2, O * I * 2, 64, 32, 1, "d_weight")) != DG_OK)
      return st;
    GemmParams p{};
    p.G = 1;
    p.M = static_cast<int32_t>(out_f);
    p.N = static_cast<int32_t>(in_f);
    p.K = static_cast<int32_t>(rows);
    p.a_g = p.b_g = p.d_g = G_OUTER;
    p.a_mn4 = dyt_mn4;
    p.b_mn4 = xn_mn4;
    if ((st = run_gemm(GV_BF16_MM_STORE, mdy_t, mx_n, mdw, mdw, p, dev, s, "tp_linear_bwd_dw",
                       2.0 * (r * fo + r * fi + fo * fi))) != DG_OK)
      return st;
  }
  if (d_bias) {
    TraceScope trace("tp_linear_bwd_db", s, 0.0, r * fo * 2.0 + fo * 2.0);
    cudaError_t e = launch_column_sum(dy, d_bias, 1, static_cast<int>(rows), static_cast<int>(out_f), 0,
                                      static_cast<int64_t>(out_f), dev, s);
    if (e != cudaSuccess) return cuda_fail(e, "tp_linear_bwd: column-sum launch");
  }
  return DG_OK;
}

dg_status dg_trace_begin(void) { return dg_trace_begin_only(nullptr); }

dg_status dg_trace_begin_only(const char* name) {
  std::lock_guard<std::mutex> g(g_trace_mu);
  g_trace_only = name ? name : "";
  g_tracing = true;
  return DG_OK;
}

int32_t dg_trace_end(dg_trace_entry* out, int32_t max_entries) {
  std::vector<TraceRecord> recs;
  {
    std::lock_guard<std::mutex> g(g_trace_mu);
    g_tracing = false;
    recs.swap(g_trace);
  }
  std::vector<dg_trace_entry> agg;
  bool ok = true;
  for (const TraceRecord& r : recs) {
    float ms = 0.0f;
    if (cudaEventSynchronize(r.e1) != cudaSuccess || cudaEventElapsedTime(&ms, r.e0, r.e1) != cudaSuccess) ok = false;
    cudaEventDestroy(r.e0);
    cudaEventDestroy(r.e1);
    size_t i = 0;
    while (i < agg.size() && strncmp(agg[i].name, r.name, sizeof(agg[i].name)) != 0) ++i;
    if (i == agg.size()) {
      dg_trace_entry e{};
      strncpy(e.name, r.name, sizeof(e.name) - 1);
      agg.push_back(e);
    }
    agg[i].launches += 1;
    agg[i].total_ms += ms;
    agg[i].flops += r.flops;
    agg[i].bytes += r.bytes;
  }
  if (!ok) {
    fail(DG_ERR_CUDA, "dg_trace_end: event timing failed");
    return -1;
  }
  const int32_t n = static_cast<int32_t>(agg.size());
  for (int32_t i = 0; i < n && i < max_entries; ++i) out[i] = agg[i];
  return n;
}

}  // extern "C"
