// Host-side internals shared by the translation units of libdg.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <utility>

#include "../../include/dg.h"
#include "dg_gemm.cuh"

namespace dg {

// Records a thread-local message and returns `s`.
dg_status fail(dg_status s, const char* fmt, ...);

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// True if [a, a+na) and [b, b+nb) overlap (a NULL or empty range overlaps nothing).
inline bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  if (!a || !b || na == 0 || nb == 0) return false;
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

// Per-device facts, cached on first use of each device.  `err` is the
// error word the kernels of one call record a failed wait in: each entry point
// points it at the error block of its caller's workspace (device_info leaves
// it NULL).  `builtin_err` is the library's own word, which only the call
// that takes no workspace (dg_tp_swiglu_noalloc) uses.
struct DeviceInfo {
  int device;
  int num_sms;
  uint32_t* err;
  uint32_t* builtin_err;
};
dg_status device_info(DeviceInfo* out);

// Checks that `ws` holds at least the error block (DG_ERROR_BLOCK_BYTES,
// 16-byte aligned), before any device call.
dg_status check_error_block(const void* ws, size_t ws_bytes, const char* what);
// check_error_block, then device_info, with dev->err pointed at the first word of `ws`.
dg_status device_info_ws(DeviceInfo* dev, void* ws, size_t ws_bytes, const char* what);

// A 3-D TMA tensor map over a row-major tensor.  dims are in elements,
// innermost first; strides (bytes) are those of dims 1 and 2; box in
// elements.  Swizzle is 128 B, out-of-bounds elements read as zero.
dg_status make_map_3d(CUtensorMap* map, bool is_bf16, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                      uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t b0, uint32_t b1, uint32_t b2,
                      const char* what);

// make_map_3d with a 64- or 128-byte swizzle (the box's inner extent must not
// exceed it).
dg_status make_map_3d_sw(CUtensorMap* map, bool is_bf16, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                         uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t b0, uint32_t b1, uint32_t b2,
                         int swizzle_bytes, const char* what);

// The map of an MN-major GEMM operand (MN = d0, the contiguous dimension;
// d1, d2, strides and the box's b1, b2 as for make_map_3d with b0 = 64).
// When MN is a multiple of 64 the map is 4-D, (mn % 64, d1, d2, mn / 64)
// with a last stride of 128 bytes, and its box (64, b1, b2, blocks) fetches
// `blocks` 64-element MN blocks in one copy, stacked in shared memory
// exactly like `blocks` separate 3-D boxes; *mn4 is set to 1.  Otherwise (or
// if the driver rejects the 4-D form) it is the 3-D map and *mn4 = 0.
dg_status make_map_mn(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                      uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t b1, uint32_t b2, uint32_t blocks,
                      int32_t* mn4, const char* what);

enum GemmVariant : int {
  GV_FP8_KK = 0,        // e4m3, A and B K-major, alpha/beta/C epilogue
  GV_BF16_KK_STORE = 1, // bf16, A and B K-major, plain store
  GV_BF16_KM_BIAS = 2,  // bf16, A K-major, B MN-major, bias epilogue
  GV_BF16_MM_STORE = 3, // bf16, A and B MN-major, plain store
  GV_BF16_KK_SWIGLU = 4, // bf16, A and B K-major, paired silu(a)*b epilogue
  GV_BF16_KM_LNSTATS = 5, // bf16, A K-major, B MN-major, bias + per-tile LayerNorm statistics
  GV_BF16_KM_STORE = 6,   // bf16, A K-major, B MN-major, plain store
  GV_FP8_KK_N224 = 7,     // GV_FP8_KK with 224-column tiles
  GV_BF16_KK_BIAS = 8,    // bf16, A and B K-major, bias epilogue
  GV_FP8_KK_LNSTATS = 9,  // e4m3, A and B K-major, dequantise + bias + per-tile LayerNorm statistics
  GV_FP8_KK_BIAS = 10     // e4m3, A and B K-major, dequantise + bias
};

// Tiles along N of one problem for this variant (output columns per tile).
int gemm_tile_n(GemmVariant v);
int gemm_tile_m();

// Enqueue one persistent GEMM launch.  `p.tiles_*` and the grid are filled in
// here.  `name` and `bytes` (algorithmic HBM bytes) label the launch for
// tracing; a NULL name launches it untraced (no events are created).
dg_status run_gemm(GemmVariant v, const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& d,
                   const CUtensorMap& c, GemmParams p, const DeviceInfo& dev, cudaStream_t s, const char* name,
                   double bytes);

// The FFN's second GEMM with the normalise-and-gate folded into its A operand
// (launch_gemm_gated), traced like run_gemm.
struct GateSrc;
dg_status run_gemm_gated(const CUtensorMap& b, const CUtensorMap& d, const CUtensorMap& z, GemmParams p,
                         const GateSrc& q, const DeviceInfo& dev, cudaStream_t s, const char* name, double bytes);

// Argument checks of the TP SwiGLU pair (sizes, NULL, alignment, overlaps of
// the output and of the scratch region [scratch, scratch + scratch_bytes)
// with the tensors); the same for every entry point of the pair.
dg_status tp_swiglu_check_sizes(int64_t S, int64_t d, int64_t ffn, int32_t W, int32_t bsz, const char* what);
dg_status tp_swiglu_check(int64_t S, int64_t d, int64_t ffn, int32_t W, int32_t bsz, const void* x_shards,
                          const void* w13, const void* w2, const void* y_shards, const void* scratch,
                          size_t scratch_bytes, const char* what);

// The two GEMMs of the TP SwiGLU pair with h [S*bsz, ffn] bf16 at `h`; the
// arguments have been validated by the caller.  traced = false creates no
// events (the entry point that must not allocate anything).
dg_status tp_swiglu_enqueue(int64_t S, int64_t d, int64_t ffn, int32_t W, int32_t bsz, const void* x_shards,
                            const void* w13, const void* w2, void* y_shards, void* h, const DeviceInfo& dev,
                            cudaStream_t s, bool traced);

// Brackets one kernel launch with CUDA events while tracing is on (dg_trace_begin).
class TraceScope {
 public:
  TraceScope(const char* name, cudaStream_t s, double flops, double bytes);
  ~TraceScope();
  TraceScope(const TraceScope&) = delete;
  TraceScope& operator=(const TraceScope&) = delete;

 private:
  bool active_ = false;
  cudaStream_t stream_;
  const char* name_;
  double flops_, bytes_;
  cudaEvent_t e0_{}, e1_{};
};

// Launchers, one per translation unit.
cudaError_t launch_gemm_fp8_kk(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                               const GemmParams&, int num_sms, cudaStream_t);
cudaError_t launch_gemm_bf16_kk_store(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                      const CUtensorMap&, const GemmParams&, int num_sms, cudaStream_t);
cudaError_t launch_gemm_bf16_km_bias(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                     const CUtensorMap&, const GemmParams&, int num_sms, cudaStream_t);
cudaError_t launch_gemm_bf16_mm_store(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                      const CUtensorMap&, const GemmParams&, int num_sms, cudaStream_t);
cudaError_t launch_gemm_bf16_kk_swiglu(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                       const CUtensorMap&, const GemmParams&, int num_sms, cudaStream_t);
cudaError_t launch_gemm_bf16_km_lnstats(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                        const CUtensorMap&, const GemmParams&, int num_sms, cudaStream_t);
cudaError_t launch_gemm_bf16_km_store(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                      const CUtensorMap&, const GemmParams&, int num_sms, cudaStream_t);
cudaError_t launch_gemm_bf16_kk_bias(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                     const CUtensorMap&, const GemmParams&, int num_sms, cudaStream_t);
cudaError_t launch_gemm_fp8_kk_lnstats(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                       const GemmParams&, int num_sms, cudaStream_t);
cudaError_t launch_gemm_fp8_kk_bias(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                    const GemmParams&, int num_sms, cudaStream_t);
cudaError_t launch_gemm_fp8_kk_n224(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                    const GemmParams&, int num_sms, cudaStream_t);
// Co-resident CTA pairs (or CTAs) of the e4m3 GEMM on the current device.
cudaError_t gemm_fp8_units(int num_sms, int* units);

// Sources of the normalise-and-gate folded into the A operand of the FFN's
// second GEMM (dg_gemm_gated.cu): A[m, k] = LN_x(U)[m, k] * silu(LN_g(G))[m, k]
// of problem g, computed from Z and the row statistics.
struct GateSrc {
  const __nv_bfloat16* Z;                  // [G][M][2H]: U = columns [0, H), G = [H, 2H)
  const float4* stats;                     // [G][M]: (mean_u, rstd_u, mean_g, rstd_g)
  const __nv_bfloat16 *gx, *bx, *gg, *bg;  // [P][H]: LayerNorm weight and bias of U and of G
  __nv_bfloat16* Hl;                       // [G][M][H], written by the units of column pass 0; or NULL
  int32_t H, L;                            // half width of Z; problems per rank (rank of problem g = g / L)
};
// Output columns per work unit of the gated GEMM (two 256-column UMMAs), and
// the K elements of one of its pipeline stages (32 or 64).
int gemm_gated_tile_n();
int gemm_gated_bk();
// One persistent launch of the gated GEMM: B = wout (MN-major map, p.b_mn4),
// D = the output map with p.d_g, Z = the map of q.Z ([G][M][2H], box 64 x 128
// rows), p.bias [G][N] with p.bias_g_stride.
cudaError_t launch_gemm_gated(const CUtensorMap& b, const CUtensorMap& d, const CUtensorMap& z, const GemmParams& p,
                              const GateSrc& q, int num_sms, cudaStream_t s);

// Widest FFN hidden size H = D*k accepted (GEMM N = 2H stays far inside int32
// tile arithmetic; the row kernels split wider rows into column blocks).
constexpr int kMaxFfnH = 65536;

// The GEMMs run as CTA pairs (cta_group::2, 256-row tiles, clusters of 2).
constexpr bool kUsePairs = true;

// Rows of a K-major B tile each CTA loads (the TMA box height of such B maps).
constexpr int kKMajorBRows = kUsePairs ? 128 : 256;
// 64-element MN blocks per stage of an MN-major operand: A (128 rows a CTA)
// and B (a CTA's share of the tile's columns).
constexpr uint32_t kMnBlocksA = 2;
constexpr uint32_t kMnBlocksB = kKMajorBRows / 64;

// Per device, once: the kernel's shared-memory attribute and the number of
// co-resident CTA pairs (CTAs) -- host-side work kept off the launch path.
template <bool kFp8, bool kAMN, bool kBMN, int kEpi, int kBN = 256>
cudaError_t gemm_units_t(int num_sms, int* out) {
  using Cfg = GemmCfg<kFp8, kAMN, kBMN, kEpi, kUsePairs, kBN>;
  auto kern = gemm_tc_kernel<kFp8, kAMN, kBMN, kEpi, kUsePairs, kBN>;
  static std::atomic<int> units_cache[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  int units = units_cache[dev].load(std::memory_order_relaxed);
  if (units == 0) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    units = num_sms;
    if (kUsePairs) {
      cudaLaunchConfig_t cfg = {};
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = 2;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      cfg.blockDim = dim3(Cfg::NUM_THREADS);
      cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
      cfg.gridDim = dim3(2);
      int clusters = 0;
      e = cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg);
      if (e != cudaSuccess) return e;
      units = clusters > 0 ? clusters : 1;
    }
    units_cache[dev].store(units, std::memory_order_relaxed);
  }
  *out = units;
  return cudaSuccess;
}

// Host launcher body shared by the instantiation units: one persistent launch,
// one CTA (or CTA pair) per SM (pair of SMs) up to the number of tiles.
template <bool kFp8, bool kAMN, bool kBMN, int kEpi, int kBN = 256>
cudaError_t launch_gemm_t(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& d, const CUtensorMap& c,
                          const GemmParams& p, int num_sms, cudaStream_t s) {
  using Cfg = GemmCfg<kFp8, kAMN, kBMN, kEpi, kUsePairs, kBN>;
  auto kern = gemm_tc_kernel<kFp8, kAMN, kBMN, kEpi, kUsePairs, kBN>;
  int units = 0;
  cudaError_t e = gemm_units_t<kFp8, kAMN, kBMN, kEpi, kBN>(num_sms, &units);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  cfg.blockDim = dim3(Cfg::NUM_THREADS);
  cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
  cfg.stream = s;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (kUsePairs) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 2;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.numAttrs = 2;
  }
  const int64_t tiles = static_cast<int64_t>(p.G) * p.tiles_m * p.tiles_n;
  if (tiles < units) units = static_cast<int>(tiles);
  cfg.gridDim = dim3(units * Cfg::CTAS);
  return cudaLaunchKernelEx(&cfg, kern, a, b, d, c, p);
}

// One launch with programmatic stream serialisation: the kernel may begin
// while the preceding kernel of the stream finishes, and waits for it
// (griddep_wait) before reading anything that kernel may have written.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// ---------------------------------------------------------------- row kernels (dg_rowops.cu)

// Per-row LayerNorm statistics stats [T*M] (mean_u, rstd_u, mean_g, rstd_g) from the
// per-tile (mean, M2) pairs part [T][tiles_n][M] the GEMM1 epilogue wrote.
cudaError_t launch_ln_stats_finalize(const float4* part, void* stats, int T, int M, int H, int tile_n, int tiles_n,
                                     float eps, const DeviceInfo& dev, cudaStream_t s);

// Normalise and gate: Hl [rows, H] = LN_x(U) * silu(LN_g(G)) from Z [rows, 2H] and stats.
cudaError_t launch_ln_gate_fwd(const void* Z, const void* stats, const void* nx_w, const void* nx_b, const void* ng_w,
                               const void* ng_b, void* Hl, uint8_t* hq, float* hs, int P, int M, int L, int H,
                               const DeviceInfo& dev, cudaStream_t s);

// e4m3 operands of the FP8 path (per row or output column: scale = amax / 448,
// code = e4m3(x * 448 / amax)): input rows [P*B*T, D] -> codes in place of
// each row and scale[t*M + s*B + b]; weight [G][K][N] -> scale and inverse
// scale [G][N] and codes [G][N][K] (K-major).
cudaError_t launch_quant_rows(const void* x, void* q, float* scale, int64_t rows, int D, int T, int M,
                              const DeviceInfo& dev, cudaStream_t s);
cudaError_t launch_quant_weight(const void* w, float* scale, float* inv, void* q, int G, int K, int N,
                                const DeviceInfo& dev, cudaStream_t s);


// Backward of the gate and both LayerNorms, pass 1: per row, the sums of
// dx_u, dx_u*x_u, dx_g and dx_g*x_g over its H columns, stored with the row's
// statistics as a coefficient record rc[2*row], rc[2*row+1] (two float4: see
// store_row_coef).
cudaError_t launch_ln_gate_bwd_rowsum(const void* Z, const void* stats, const void* dHl, const void* nx_w,
                                      const void* nx_b, const void* ng_w, const void* ng_b, void* rc, int T, int M,
                                      int L, int H, const DeviceInfo& dev, cudaStream_t s);

// Pass 2: dZ [rows, 2H] from the records and per-(t, row range) column partial
// sums part [T, nsplit, 6, H] fp32 (dU, dG, da*x_u, da, ds*x_g, ds).
cudaError_t launch_ln_gate_bwd_apply(const void* Z, const void* rc, const void* dHl, const void* nx_w,
                                     const void* nx_b, const void* ng_w, const void* ng_b, void* dZ, float* part, int T,
                                     int M, int L, int H, int nsplit, const DeviceInfo& dev, cudaStream_t s);

// Row ranges per token position used by pass 2.
int ffn_bwd_row_splits(int T, int M, int H);

// db1 [T, 2H] and d_nx_w, d_nx_b, d_ng_w, d_ng_b [P, H] from the partials, in a
// fixed order; a NULL output is skipped.
cudaError_t launch_grad_reduce(const float* part, void* d_b1, void* d_nx_w, void* d_nx_b, void* d_ng_w, void* d_ng_b,
                               int P, int L, int H, int nsplit, const DeviceInfo& dev, cudaStream_t s);

// out[g, c] = sum_n src[g*g_stride + n*row_stride + c] (bf16 in, fp32 sum, bf16 out [G, ncols]).
cudaError_t launch_column_sum(const void* src, void* out, int G, int rows, int ncols, int64_t g_stride,
                              int64_t row_stride, const DeviceInfo& dev, cudaStream_t s);

// Backward of the SwiGLU gate, in place: ab [rows, W, 2F] holds (a_s | b_s)
// and becomes (da_s | db_s); dh [rows, W*F] becomes h = silu(a)*b.
cudaError_t launch_swiglu_gate_bwd(void* ab, void* dh_h, int64_t rows, int W, int F, const DeviceInfo& dev,
                                   cudaStream_t s);

// comp_only layout: out[p][b][r*L + l] = in[r][b][p*L + l] for tensors
// [P, B, T, D] with T = P*L (an involution; 16-byte vector copies).
cudaError_t launch_swap_rank_slice(const void* in, void* out, int P, int B, int T, int D, const DeviceInfo& dev,
                                   cudaStream_t s);

// Row permutations of the exchange (16-byte vector copies).
cudaError_t launch_dispatch(const void* in, void* out, int P, int B, int T, int D, const DeviceInfo& dev,
                            cudaStream_t s);
cudaError_t launch_combine(const void* in, void* out, int P, int B, int T, int D, const DeviceInfo& dev,
                           cudaStream_t s);

cudaError_t launch_debug_wait(uint32_t* err, uint64_t limit_ns, cudaStream_t s);

}  // namespace dg
