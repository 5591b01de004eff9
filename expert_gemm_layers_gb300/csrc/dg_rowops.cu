// HBM-bound kernels of the A2A FFN layer: the LayerNorm-and-gate pass
// (forward and backward), deterministic column reductions, and the two
// exchange permutations as explicit copies.
//
// Source of the arithmetic: the A2A-FFN project statement (problems/p04),
// "Computation and communication example": (U, G) are the two H-wide halves
// of Z, LN(z) = (z - mean z) / sqrt(mean((z - mean z)^2) + eps) * gamma + beta,
// Hl = LN_x(U) * silu(LN_gate(G)).  Statistics come from the stored bf16 Z
// (what the page's bmm path normalises), two passes over registers.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include <mutex>
#include <vector>

#include "dg_gate.cuh"
#include "dg_internal.h"

namespace dg {

namespace {

constexpr int kMaxRowWarps = 16;  // row kernels use up to 512 threads

__device__ __forceinline__ void unpack8(const uint4 v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 t = unpack_bf16x2(w[e]);
    f[2 * e] = t.x;
    f[2 * e + 1] = t.y;
  }
}


// True if the call's error word records a failure.  A kernel without bounded
// waits may be given no error word (NULL), which reads as no failure.
__device__ __forceinline__ bool err_set(const uint32_t* err) { return err != nullptr && ld_volatile_u32(err) != 0u; }

// Warp-uniform read of the error word (these kernels use full-warp barriers
// and shuffles, so a warp must not split on it).
__device__ __forceinline__ bool warp_aborted(const uint32_t* err) {
  return __shfl_sync(0xffffffffu, err_set(err) ? 1u : 0u, 0) != 0u;
}

// Block-uniform read of the error word (a divergent early return ahead of a
// barrier would be undefined).
__device__ __forceinline__ bool block_aborted(const uint32_t* err) {
  __shared__ uint32_t flag;
  if (threadIdx.x == 0) flag = err_set(err) ? 1u : 0u;
  __syncthreads();
  return flag != 0u;
}

// e4m3 code of x * inv (inv = 448 / amax): binary32 product, round to
// nearest even, saturating at +-448 (the code decision of the per-row /
// per-column quantisation).
__device__ __forceinline__ uint32_t e4m3_code(float x, float inv) {
  return static_cast<uint32_t>(__nv_cvt_float_to_fp8(__fmul_rn(x, inv), __NV_SATFINITE, __NV_E4M3));
}

// Four e4m3 codes packed little-endian into a word: the binary32 values a.x,
// a.y, b.x, b.y rounded to nearest even, saturating (cvt ... e4m3x2 puts its
// first source operand in the upper byte of its 16-bit result).
__device__ __forceinline__ uint32_t e4m3x4(float2 a, float2 b) {
  uint32_t r;
  asm("{\n\t.reg .b16 lo, hi;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 lo, %2, %1;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 hi, %4, %3;\n\t"
      "mov.b32 %0, {lo, hi};\n\t}"
      : "=r"(r)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return r;
}

// Codes of eight values, packed little-endian into two words: the same
// binary32 products and round-to-nearest-even saturating conversions as
// e4m3_code, two values per multiply and per conversion.
__device__ __forceinline__ uint2 e4m3_code8(const float (&x)[8], float inv) {
  const float2 iv = make_float2(inv, inv);
  float2 p[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) p[e] = mul2(make_float2(x[2 * e], x[2 * e + 1]), iv);
  return make_uint2(e4m3x4(p[0], p[1]), e4m3x4(p[2], p[3]));
}

// Scale (amax / 448) and inverse scale (448 / amax) of a vector whose largest
// magnitude is amax; both 1 for an all-zero vector.
__device__ __forceinline__ float e4m3_scale(float amax) { return amax > 0.0f ? __fdiv_rn(amax, 448.0f) : 1.0f; }
__device__ __forceinline__ float e4m3_inv(float amax) { return amax > 0.0f ? __fdiv_rn(448.0f, amax) : 1.0f; }

// Per-thread asynchronous copies into shared memory (cp.async): a thread
// copies exactly the bytes it will read back itself, so a multi-stage ring
// needs no barrier for the copies, only cp.async.wait_group.
__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src),
               "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// ------------------------------------------------------------------ forward
//
// The row statistics come from the GEMM that produced Z: its epilogue
// writes, per row and per 256-column tile, the mean and centred second
// moment of the tile's U and G columns; ln_stats_finalize merges the tiles
// of a row (Chan's pairwise formula) into (mean_u, rstd_u, mean_g, rstd_g).
// The normalise-and-gate pass is then a pure map: a CTA walks rows of ONE
// rank (so each thread keeps the affines of its columns in fp32 registers),
// staging rows through a shared-memory ring with per-thread cp.async.

__global__ void ln_stats_finalize_kernel(const float4* __restrict__ part, float4* __restrict__ stats, int T, int M,
                                         int H, int tile_n, int tiles_n, float eps, const uint32_t* err) {
  griddep_wait();
  if (err_set(err)) return;
  const int64_t rows = static_cast<int64_t>(T) * M;
  const int N = 2 * H;
  for (int64_t row = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; row < rows;
       row += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int t = static_cast<int>(row / M), n = static_cast<int>(row - static_cast<int64_t>(t) * M);
    MeanM2 su{0.0f, 0.0f, 0.0f}, sg{0.0f, 0.0f, 0.0f};
    for (int nt = 0; nt < tiles_n; ++nt) {
      const int c0 = nt * tile_n, cend = min(c0 + tile_n, N);
      const int nu = min(max(H - c0, 0), cend - c0), ng = cend - c0 - nu;
      const float4 q = part[(static_cast<int64_t>(t) * tiles_n + nt) * M + n];
      su.merge(static_cast<float>(nu), q.x, q.y);
      sg.merge(static_cast<float>(ng), q.z, q.w);
    }
    const float inv_h = 1.0f / static_cast<float>(H);
    stats[row] = make_float4(su.mean, rsqrtf(su.m2 * inv_h + eps), sg.mean, rsqrtf(sg.m2 * inv_h + eps));
  }
}

constexpr int kFwdStages = 4;

// kFp8Out: instead of bf16 Hl, write each row as e4m3 codes with one scale per
// row (row amax / 448) for an e4m3 GEMM2; the whole row is in one CTA.  The
// row amax is a lagged block reduction: each warp publishes its share of row
// i through one of four mbarrier-guarded slots and meanwhile quantises row
// i - 1, whose shares are complete by then (a slot is reused four rows later,
// after every warp has published row i - 2, so it has read row i - 4).
template <int NT, int VPT, bool kFp8Out>
__global__ void __launch_bounds__(NT, 512 / NT) ln_gate_fwd_kernel(
    const __nv_bfloat16* __restrict__ Z, const float4* __restrict__ stats, const __nv_bfloat16* __restrict__ gx,
    const __nv_bfloat16* __restrict__ bx, const __nv_bfloat16* __restrict__ gg, const __nv_bfloat16* __restrict__ bg,
    __nv_bfloat16* __restrict__ Hl, uint8_t* __restrict__ hq, float* __restrict__ hs, int M, int L, int H,
    int ctas_per_rank, int col_blocks, uint32_t* err) {
  __shared__ float red_max[4][kMaxRowWarps];
  __shared__ uint64_t rbar[4];
  if (kFp8Out && threadIdx.x == 0) {
    for (int b = 0; b < 4; ++b) mbar_init(&rbar[b], NT / 32);
    fence_mbar_init();
  }
  extern __shared__ uint4 ring[];  // [kFwdStages][VPT][2][NT]
  griddep_wait();
  if (block_aborted(err)) return;
  // CTA -> (rank, slot within the rank, column block); a column block is
  // NT*VPT 8-column vectors of U (and the same columns of G)
  const int cb = blockIdx.x % col_blocks;
  const int cta = blockIdx.x / col_blocks;
  const int nvec = H >> 3;
  const int vbase = cb * NT * VPT;
  const int64_t zstride = 2 * static_cast<int64_t>(H);
  const int r = cta / ctas_per_rank;
  const int64_t rank_rows = static_cast<int64_t>(L) * M;
  const int64_t stride = ctas_per_rank;
  const int64_t n_mine = (rank_rows - (cta % ctas_per_rank) + stride - 1) / stride;
  const int64_t row0 = static_cast<int64_t>(r) * rank_rows + (cta % ctas_per_rank);

  float2 wx[VPT][4], cx[VPT][4], wg[VPT][4], cg[VPT][4];
#pragma unroll
  for (int j = 0; j < VPT; ++j) {
    const int v = vbase + threadIdx.x + NT * j;
    const Affine8 a = load_affine8(gx, bx, gg, bg, static_cast<int64_t>(r) * H + 8 * (v < nvec ? v : 0));
    const uint32_t w0[4] = {a.wx.x, a.wx.y, a.wx.z, a.wx.w}, w1[4] = {a.cx.x, a.cx.y, a.cx.z, a.cx.w};
    const uint32_t w2[4] = {a.wg.x, a.wg.y, a.wg.z, a.wg.w}, w3[4] = {a.cg.x, a.cg.y, a.cg.z, a.cg.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      wx[j][e] = unpack_bf16x2(w0[e]);
      cx[j][e] = unpack_bf16x2(w1[e]);
      // the gate norm's affine halved (exact): h = s/2 = x_g*(gg/2) + bg/2
      // rounds to exactly half of fma(x_g, gg, bg), so Hl is unchanged
      wg[j][e] = mul2(unpack_bf16x2(w2[e]), splat2(0.5f));
      cg[j][e] = mul2(unpack_bf16x2(w3[e]), splat2(0.5f));
    }
  }
  auto issue = [&](int64_t i) {
    if (i < n_mine) {
      const __nv_bfloat16* zu = Z + (row0 + i * stride) * zstride;
      uint4* st = ring + (i % kFwdStages) * (VPT * 2 * NT);
#pragma unroll
      for (int j = 0; j < VPT; ++j) {
        const int v = vbase + threadIdx.x + NT * j;
        const bool ok = v < nvec;
        cp_async16(st + (2 * j) * NT + threadIdx.x, zu + 8 * (ok ? v : 0), ok);
        cp_async16(st + (2 * j + 1) * NT + threadIdx.x, zu + H + 8 * (ok ? v : 0), ok);
      }
    }
    cp_async_commit();
  };
#pragma unroll
  for (int i = 0; i < kFwdStages - 1; ++i) issue(i);
  float4 st_next = n_mine > 0 ? stats[row0] : make_float4(0.f, 0.f, 0.f, 0.f);
  // e4m3 output: the previous row's values wait in the other of two arrays
  // (the rows alternate between them) for that row's amax
  float oa[VPT][8], ob[VPT][8];
  int64_t prev_row = 0;
  auto finish_row = [&](int64_t k, int64_t krow, const float (&o_prev)[VPT][8]) -> bool {
    const int slot = static_cast<int>(k & 3);
    const uint32_t parity = static_cast<uint32_t>(k >> 2) & 1u;
    if (!__all_sync(0xffffffffu, mbar_wait(&rbar[slot], parity, err, 0x41u))) return false;  // warp-uniform
    float m = (threadIdx.x & 31) < NT / 32 ? red_max[slot][threadIdx.x & 31] : 0.0f;
#pragma unroll
    for (int o2 = 16; o2 > 0; o2 >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o2));
    const float inv = e4m3_inv(m);
    uint8_t* qrow = hq + krow * static_cast<int64_t>(H);
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
      const int v = vbase + threadIdx.x + NT * j;
      if (v < nvec) {
        *reinterpret_cast<uint2*>(qrow + 8 * v) = e4m3_code8(o_prev[j], inv);
      }
    }
    if (threadIdx.x == 0) hs[krow] = e4m3_scale(m);
    return true;
  };
  auto do_row = [&](int64_t i, float (&o)[VPT][8], const float (&o_prev)[VPT][8]) -> bool {
    issue(i + kFwdStages - 1);
    const int64_t row = row0 + i * stride;
    const float4 sr = st_next;
    if (i + 1 < n_mine) st_next = stats[row + stride];
    cp_async_wait<kFwdStages - 1>();
    const uint4* st = ring + (i % kFwdStages) * (VPT * 2 * NT);
    const float2 rsu = make_float2(sr.y, sr.y), cu = make_float2(-sr.x * sr.y, -sr.x * sr.y);
    const float2 rsg = make_float2(sr.w, sr.w), cgs = make_float2(-sr.z * sr.w, -sr.z * sr.w);
    float amax = 0.0f;
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
      const int v = vbase + threadIdx.x + NT * j;
      if (v < nvec) {
        const uint4 pu = st[(2 * j) * NT + threadIdx.x], pg = st[(2 * j + 1) * NT + threadIdx.x];
        const uint32_t uw[4] = {pu.x, pu.y, pu.z, pu.w}, gw[4] = {pg.x, pg.y, pg.z, pg.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 a = fma2(fma2(unpack_bf16x2(uw[e]), rsu, cu), wx[j][e], cx[j][e]);
          const float2 h = fma2(fma2(unpack_bf16x2(gw[e]), rsg, cgs), wg[j][e], cg[j][e]);
          const float2 silu = fma2(h, make_float2(tanh_fast(h.x), tanh_fast(h.y)), h);
          const float2 ov = mul2(a, silu);
          o[j][2 * e] = ov.x;
          o[j][2 * e + 1] = ov.y;
          amax = fmaxf(amax, fmaxf(fabsf(ov.x), fabsf(ov.y)));
        }
      }
    }
    if (!kFp8Out) {
      __nv_bfloat16* hrow = Hl + row * static_cast<int64_t>(H);
#pragma unroll
      for (int j = 0; j < VPT; ++j) {
        const int v = vbase + threadIdx.x + NT * j;
        if (v < nvec)
          __stcs(reinterpret_cast<uint4*>(hrow + 8 * v),
                 make_uint4(pack_bf16x2(o[j][0], o[j][1]), pack_bf16x2(o[j][2], o[j][3]),
                            pack_bf16x2(o[j][4], o[j][5]), pack_bf16x2(o[j][6], o[j][7])));
      }
    } else {
      float wmax = amax;
#pragma unroll
      for (int o2 = 16; o2 > 0; o2 >>= 1) wmax = fmaxf(wmax, __shfl_xor_sync(0xffffffffu, wmax, o2));
      const int slot = static_cast<int>(i & 3);
      if ((threadIdx.x & 31) == 0) {
        red_max[slot][threadIdx.x >> 5] = wmax;
        mbar_arrive(&rbar[slot]);
      }
      if (i > 0 && !finish_row(i - 1, prev_row, o_prev)) return false;
      prev_row = row;
    }
    return true;
  };
  if (kFp8Out) {
    for (int64_t i = 0; i < n_mine; i += 2) {
      if (!do_row(i, oa, ob)) return;
      if (i + 1 < n_mine && !do_row(i + 1, ob, oa)) return;
    }
  } else {
    for (int64_t i = 0; i < n_mine; ++i) do_row(i, oa, ob);
  }
  if (kFp8Out && n_mine > 0 && !finish_row(n_mine - 1, prev_row, ((n_mine - 1) & 1) ? ob : oa)) return;
  cp_async_wait<0>();
}

// The e4m3 gate pass for rows of up to 7680 columns as a bulk-copy
// pipeline: one producer thread streams whole rows of Z (U | G, 4H bytes)
// and their statistics into a ring of shared-memory slots with
// cp.async.bulk; fifteen consumer warps take two 8-column vectors a thread
// (affines in fp32 registers), compute the row's values and its largest
// magnitude, park the values in one of kGfVbuf fp32 row buffers in shared
// memory (each thread its own columns) and release the slot.  The row amax
// is a lagged block reduction: each warp publishes its share of row i
// through one of kGfSlots mbarrier-guarded slots and then quantises row
// i - kGfLag, whose shares are complete by then unless a warp is more than
// kGfLag rows behind (two rows of lag instead of one measured 11 % faster:
// the warps drift apart by about a row).  A slot is rewritten kGfSlots rows
// later; a warp publishing row j has seen every warp publish row
// j - 1 - kGfLag, so every warp has quantised row j - 2 - 2 * kGfLag, which
// kGfSlots >= 2 + 2 * kGfLag makes old enough.  The warp and block maxima
// are taken by redux.sync on the bit patterns: the per-thread amax is a
// non-negative float that is never NaN (fmaxf drops NaNs), and for those
// the unsigned order of the bits is the order of the values.  Values and
// codes are those of ln_gate_fwd_kernel<..., true>.  Each CTA takes a
// contiguous range of rows.
#ifndef DG_GF_LAG
#define DG_GF_LAG 2
#endif
constexpr int kGfLag = DG_GF_LAG;                  // rows between computing a row and quantising it
constexpr int kGfRing = kGfLag == 1 ? 5 : 4;       // Z row slots
constexpr int kGfVbuf = kGfLag + 1;                // parked rows of fp32 values
constexpr int kGfSlots = 8;                        // amax slots (at least 2 + 2 * kGfLag)
static_assert(kGfSlots >= 2 + 2 * kGfLag, "amax slots");
constexpr int kGfConsumers = 15;
constexpr int kGfVec = 2;
constexpr int kGfMaxH = 8 * 32 * kGfConsumers * kGfVec;
constexpr int kGfThreads = 32 * (kGfConsumers + 1);

template <bool kFull>  // kFull: H == kGfMaxH, so every consumer thread owns two whole vectors
__global__ void __launch_bounds__(kGfThreads, 1) ln_gate_fwd_fp8_bulk_kernel(
    const __nv_bfloat16* __restrict__ Z, const float4* __restrict__ stats, const __nv_bfloat16* __restrict__ gx,
    const __nv_bfloat16* __restrict__ bx, const __nv_bfloat16* __restrict__ gg, const __nv_bfloat16* __restrict__ bg,
    uint8_t* __restrict__ hq, float* __restrict__ hs, int64_t rows, int M, int L, int H, int slot_bytes,
    uint32_t* err) {
  extern __shared__ __align__(128) uint8_t gf_smem[];
  float* vbuf = reinterpret_cast<float*>(gf_smem + kGfRing * slot_bytes);  // [kGfVbuf][H] row values
  uint64_t* full = reinterpret_cast<uint64_t*>(vbuf + kGfVbuf * H);
  uint64_t* empty = full + kGfRing;
  uint64_t* rbar = empty + kGfRing;                            // [kGfSlots]
  uint32_t* red = reinterpret_cast<uint32_t*>(rbar + kGfSlots);  // [kGfSlots][kGfConsumers]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kGfRing; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kGfConsumers);
    }
    for (int b = 0; b < kGfSlots; ++b) mbar_init(&rbar[b], kGfConsumers);
    fence_mbar_init();
  }
  griddep_wait();
  if (block_aborted(err)) return;  // (its barrier also publishes the barrier initialisation)
  const int64_t per = (rows + gridDim.x - 1) / gridDim.x;
  const int64_t r0 = min(rows, static_cast<int64_t>(blockIdx.x) * per);
  const int n = static_cast<int>(min(rows, r0 + per) - r0);
  const uint32_t zbytes = 4u * H;
  const int nvec = H >> 3;

  if (warp == kGfConsumers) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      int issued = 0;
      for (int i = 0; i < n; ++i) {
        const int s = i % kGfRing;
        if (i >= kGfRing && !mbar_wait(&empty[s], static_cast<uint32_t>(i / kGfRing - 1) & 1u, err, 0x42u)) break;
        uint8_t* slot = gf_smem + s * slot_bytes;
        const int64_t row = r0 + i;
        mbar_arrive_expect_tx(&full[s], zbytes + 16u);
        bulk_load(slot, Z + row * 2 * static_cast<int64_t>(H), zbytes, &full[s]);
        bulk_load(slot + zbytes, stats + row, 16u, &full[s]);
        issued = i + 1;
      }
      // every copy issued has landed before the CTA may exit
      for (int i = max(0, issued - kGfRing); i < issued; ++i) {
        uint32_t dummy = 0;
        if (!mbar_try_wait(&full[i % kGfRing], static_cast<uint32_t>(i / kGfRing) & 1u))
          mbar_wait_slow(&full[i % kGfRing], static_cast<uint32_t>(i / kGfRing) & 1u, &dummy, 0x43u, kWaitLimitNs);
      }
    }
    return;
  }

  // ---------------------------------------------------------------- consumers
  const int64_t rank_rows = static_cast<int64_t>(L) * M;
  int rank = static_cast<int>(r0 / rank_rows);
  int next_rank_at = static_cast<int>(min(static_cast<int64_t>(n), (rank + 1) * rank_rows - r0));
  bool reload = true;
  AffineF af[kGfVec];
  // this thread's vectors: v0 + 32 * kGfConsumers * j
  const int v0 = warp * 32 + lane;
  int s = 0;           // ring slot of the row being computed
  uint32_t ph = 0;     // and its phase parity
  uint8_t* qrow = hq + r0 * static_cast<int64_t>(H);  // code row of the row being quantised
  // quantise row k (local index) once every warp's share of its amax is in
  auto finish_row = [&](int k) -> bool {
    const int slot = k % kGfSlots;
    if (!__all_sync(0xffffffffu, mbar_wait(&rbar[slot], static_cast<uint32_t>(k / kGfSlots) & 1u, err, 0x44u)))
      return false;
    const uint32_t mb = __reduce_max_sync(0xffffffffu, lane < kGfConsumers ? red[slot * kGfConsumers + lane] : 0u);
    const float m = __uint_as_float(mb);
    const float inv = e4m3_inv(m);
    const float* vrow = vbuf + (k % kGfVbuf) * H;
#pragma unroll
    for (int j = 0; j < kGfVec; ++j) {
      const int v = v0 + 32 * kGfConsumers * j;
      if (kFull || v < nvec) {
        const float4 x0 = reinterpret_cast<const float4*>(vrow)[2 * v];
        const float4 x1 = reinterpret_cast<const float4*>(vrow)[2 * v + 1];
        const float x[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
        *reinterpret_cast<uint2*>(qrow + 8 * v) = e4m3_code8(x, inv);
      }
    }
    if (warp == 0 && lane == 0) hs[r0 + k] = e4m3_scale(m);
    qrow += H;
    return true;
  };
  auto do_row = [&](int i) -> bool {
    if (!__all_sync(0xffffffffu, mbar_wait(&full[s], ph, err, 0x45u))) return false;
    if (i == next_rank_at) {
      ++rank;
      next_rank_at = static_cast<int>(min(static_cast<int64_t>(n), next_rank_at + rank_rows));
      reload = true;
    }
    if (reload) {
      reload = false;
#pragma unroll
      for (int j = 0; j < kGfVec; ++j) {
        const int v = v0 + 32 * kGfConsumers * j;
        if (kFull || v < nvec) {
          af[j] = load_affine_f(gx, bx, gg, bg, static_cast<int64_t>(rank) * H + 8 * v);
          halve_gate_affine(af[j]);  // h = s/2 from one fma, exactly as in ln_gate_fwd_kernel
        }
      }
    }
    const uint8_t* slot = gf_smem + s * slot_bytes;
    const uint4* zrow = reinterpret_cast<const uint4*>(slot);
    const float4 sr = *reinterpret_cast<const float4*>(slot + zbytes);
    const float2 rsu = splat2(sr.y), cu = splat2(-sr.x * sr.y), rsg = splat2(sr.w), cgs = splat2(-sr.z * sr.w);
    float* vrow = vbuf + (i % kGfVbuf) * H;
    float amax = 0.0f;
#pragma unroll
    for (int j = 0; j < kGfVec; ++j) {
      const int v = v0 + 32 * kGfConsumers * j;
      if (kFull || v < nvec) {
        const uint4 pu = zrow[v], pg = zrow[nvec + v];
        const uint32_t uw[4] = {pu.x, pu.y, pu.z, pu.w}, gw[4] = {pg.x, pg.y, pg.z, pg.w};
        float o[8];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 a = fma2(fma2(unpack_bf16x2(uw[e]), rsu, cu), af[j].wx[e], af[j].cx[e]);
          const float2 h = fma2(fma2(unpack_bf16x2(gw[e]), rsg, cgs), af[j].wg[e], af[j].cg[e]);
          const float2 silu = fma2(h, make_float2(tanh_fast(h.x), tanh_fast(h.y)), h);
          const float2 ov = mul2(a, silu);
          o[2 * e] = ov.x;
          o[2 * e + 1] = ov.y;
          amax = fmaxf(amax, fmaxf(fabsf(ov.x), fabsf(ov.y)));
        }
        reinterpret_cast<float4*>(vrow)[2 * v] = make_float4(o[0], o[1], o[2], o[3]);
        reinterpret_cast<float4*>(vrow)[2 * v + 1] = make_float4(o[4], o[5], o[6], o[7]);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);  // the slot has been read
    if (++s == kGfRing) {
      s = 0;
      ph ^= 1u;
    }
    const uint32_t wmax = __reduce_max_sync(0xffffffffu, __float_as_uint(amax));
    if (lane == 0) {
      red[(i % kGfSlots) * kGfConsumers + warp] = wmax;
      mbar_arrive(&rbar[i % kGfSlots]);
    }
    return i < kGfLag || finish_row(i - kGfLag);
  };
  for (int i = 0; i < n; ++i)
    if (!do_row(i)) return;
  for (int k = max(0, n - kGfLag); k < n; ++k)
    if (!finish_row(k)) return;
}

// ------------------------------------------------------------------ e4m3 operands
// Quantisation for the FP8 GEMMs of the layer: scale = amax / 448 per row of
// an activation or per output column of a weight, code = the e4m3 value
// nearest to x / scale (binary32 division, ties to even, saturating).

// inputs [P*B*T rows of D] -> codes in the same layout, one scale per row,
// stored per problem: scale[t*M + n] for input row (s, b, t), n = s*B + b.
// One warp per row.
__global__ void quant_rows_kernel(const __nv_bfloat16* __restrict__ x, uint8_t* __restrict__ q,
                                  float* __restrict__ scale, int64_t rows, int D, int T, int M,
                                  const uint32_t* err) {
  griddep_wait();
  if (warp_aborted(err)) return;
  const int lane = threadIdx.x & 31;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  for (int64_t row = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); row < rows;
       row += warps) {
    const __nv_bfloat16* xr = x + row * D;
    float amax = 0.0f;
    for (int c = 8 * lane; c < D; c += 256) {
      float f[8];
      unpack8(__ldg(reinterpret_cast<const uint4*>(xr + c)), f);
#pragma unroll
      for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(f[e]));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float inv = e4m3_inv(amax);
    uint8_t* qr = q + row * D;
    for (int c = 8 * lane; c < D; c += 256) {
      float f[8];
      unpack8(__ldg(reinterpret_cast<const uint4*>(xr + c)), f);
      *reinterpret_cast<uint2*>(qr + c) = e4m3_code8(f, inv);
    }
    if (lane == 0) {
      const int64_t sb = row / T;  // s*B + b
      const int t = static_cast<int>(row - sb * T);
      scale[static_cast<int64_t>(t) * M + sb] = e4m3_scale(amax);
    }
  }
}

// Weight [G][K][N] (N contiguous): scale[g][n] = amax over k / 448 and
// inv[g][n] = 448 / amax.
__global__ void col_scale_kernel(const __nv_bfloat16* __restrict__ w, float* __restrict__ scale,
                                 float* __restrict__ inv, int K, int N, const uint32_t* err) {
  griddep_wait();
  if (err_set(err)) return;
  const int g = blockIdx.y;
  const int n = blockIdx.x * blockDim.x + threadIdx.x;
  if (n >= N) return;
  const __nv_bfloat16* p = w + static_cast<int64_t>(g) * K * N + n;
  float amax = 0.0f;
  for (int k = 0; k < K; ++k) amax = fmaxf(amax, fabsf(__bfloat162float(p[static_cast<int64_t>(k) * N])));
  scale[static_cast<int64_t>(g) * N + n] = e4m3_scale(amax);
  inv[static_cast<int64_t>(g) * N + n] = e4m3_inv(amax);
}

// Weight [G][K][N] -> codes [G][N][K] (K contiguous: the K-major B operand of
// an e4m3 GEMM), through a 64 x 64 shared-memory tile.  256 threads.
__global__ void transpose_quant_kernel(const __nv_bfloat16* __restrict__ w, const float* __restrict__ inv,
                                       uint8_t* __restrict__ q, int K, int N, const uint32_t* err) {
  __shared__ float tile[64][65];
  griddep_wait();
  if (block_aborted(err)) return;
  const int g = blockIdx.z;
  const int k0 = blockIdx.y * 64, n0 = blockIdx.x * 64;
  const __nv_bfloat16* wg = w + static_cast<int64_t>(g) * K * N;
  {
    // load: 64 k-rows of 64 n-columns, 16 values per thread
    const int kr = threadIdx.x >> 2, nc = (threadIdx.x & 3) * 16;
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const int k = k0 + kr, n = n0 + nc + e;
      tile[kr][nc + e] = (k < K && n < N) ? __bfloat162float(wg[static_cast<int64_t>(k) * N + n]) : 0.0f;
    }
  }
  __syncthreads();
  {
    // store: 64 n-rows of 64 k-codes, 16 per thread
    const int nr = threadIdx.x >> 2, kc = (threadIdx.x & 3) * 16;
    const int n = n0 + nr;
    if (n < N) {
      const float iv = inv[static_cast<int64_t>(g) * N + n];
      uint8_t* qn = q + (static_cast<int64_t>(g) * N + n) * K;
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const int k = k0 + kc + e;
        if (k < K) qn[k] = static_cast<uint8_t>(e4m3_code(tile[kc + e][nr], iv));
      }
    }
  }
}

// ------------------------------------------------------------------ backward
//
// With x_u = (U - mu_u) * rstd_u, a = x_u*gx + bx, x_g likewise, s = x_g*gg + bg,
// q = silu(s), Hl = a*q:  da = dHl*q, ds = dHl*a*silu'(s) with
// silu'(s) = sig(s) + s*sig(s)*(1 - sig(s)), dx_u = da*gx,
// dU = rstd_u * (dx_u - mean(dx_u) - x_u*mean(dx_u*x_u)), and the same for G.
//
// Pass 1 (row sums): per row, the sums of dx_u, dx_u*x_u, dx_g and dx_g*x_g,
// stored with the row's statistics as a 32-byte coefficient record.
// Pass 2 (apply): a CTA owns a column block of one token position t and a
// range of its rows: it writes dZ and sums, per column, dU, dG (db1),
// da*x_u, da (norm_x grads), ds*x_g, ds (norm_gate grads) in registers; the
// per-(t, row range) partial sums are added in a fixed order afterwards.

// Pass 1 for rows wider than 7680 columns: one warp per row, no block barrier.  The warp walks the row in
// 256-column steps (8 columns per lane), two steps in flight, and reduces
// the four sums with shuffles.  The affines come through L1 (a CTA's warps
// work on consecutive rows, hence mostly on one rank).
constexpr int kRowsumThreads = 256;

__global__ void __launch_bounds__(kRowsumThreads, 2) ln_gate_bwd_rowsum_kernel(
    const __nv_bfloat16* __restrict__ Z, const float4* __restrict__ stats, const __nv_bfloat16* __restrict__ dHl,
    const __nv_bfloat16* __restrict__ gx, const __nv_bfloat16* __restrict__ bx, const __nv_bfloat16* __restrict__ gg,
    const __nv_bfloat16* __restrict__ bg, float4* __restrict__ rc, int64_t rows, int M, int L, int H,
    const uint32_t* err) {
  griddep_wait();
  if (warp_aborted(err)) return;
  const float inv_h = 1.0f / static_cast<float>(H);
  const int lane = threadIdx.x & 31;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (kRowsumThreads / 32);
  const int64_t zstride = 2 * static_cast<int64_t>(H);
  for (int64_t row = static_cast<int64_t>(blockIdx.x) * (kRowsumThreads / 32) + (threadIdx.x >> 5); row < rows;
       row += warps) {
    const int r = static_cast<int>(row / M) / L;
    const float4 sr = stats[row];
    const float2 rsu = splat2(sr.y), cu = splat2(-sr.x * sr.y), rsg = splat2(sr.w), cgs = splat2(-sr.z * sr.w);
    const __nv_bfloat16* zu = Z + row * zstride;
    const __nv_bfloat16* dh = dHl + row * static_cast<int64_t>(H);
    const int64_t pr = static_cast<int64_t>(r) * H;
    float2 s1u = splat2(0.f), s2u = splat2(0.f), s1g = splat2(0.f), s2g = splat2(0.f);
#pragma unroll 2
    for (int c = 8 * lane; c < H; c += 256) {
      const uint4 pu = __ldcs(reinterpret_cast<const uint4*>(zu + c));
      const uint4 pg = __ldcs(reinterpret_cast<const uint4*>(zu + H + c));
      const uint4 ph = __ldcs(reinterpret_cast<const uint4*>(dh + c));
      const AffineF af = load_affine_f(gx, bx, gg, bg, pr + c);
      const uint32_t uw[4] = {pu.x, pu.y, pu.z, pu.w}, gw[4] = {pg.x, pg.y, pg.z, pg.w};
      const uint32_t hw[4] = {ph.x, ph.y, ph.z, ph.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const GatePair gp = gate_pair(unpack_bf16x2(uw[e]), unpack_bf16x2(gw[e]), rsu, cu, rsg, cgs, af.wx[e],
                                      af.cx[e], af.wg[e], af.cg[e]);
        const float2 d = unpack_bf16x2(hw[e]);
        const float2 dxu = mul2(mul2(d, gp.q), af.wx[e]);
        const float2 dxg = mul2(mul2(mul2(d, gp.a), gp.dsil), af.wg[e]);
        s1u = add2(s1u, dxu);
        s2u = fma2(dxu, gp.xu, s2u);
        s1g = add2(s1g, dxg);
        s2g = fma2(dxg, gp.xg, s2g);
      }
    }
    float acc[4] = {s1u.x + s1u.y, s2u.x + s2u.y, s1g.x + s1g.y, s2g.x + s2g.y};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) acc[i] += __shfl_xor_sync(0xffffffffu, acc[i], o);
    }
    if (lane == 0) store_row_coef(rc + 2 * row, sr, make_float4(acc[0], acc[1], acc[2], acc[3]), inv_h);
  }
}

// Pass 1 for rows of up to 7680 columns, as a bulk-copy pipeline: one
// producer warp streams whole rows (the U|G row of Z, the dHl row, the row's
// statistics) into a ring of shared-memory slots with cp.async.bulk; fifteen
// consumer warps each take every fifteenth 8-column vector of the row (two
// vectors a thread, their affines held in fp32 registers) and publish each
// lane's four partial sums; when the producer warp recycles a slot its lanes
// add the partials of their lane position over the warps in a fixed order,
// reduce the four sums over the lanes, and lane 0 writes the row's
// coefficient record (store_row_coef).  The producer warp, which otherwise
// only issues copies, thus does the row reduction the consumers would each
// have done.  Each CTA takes a contiguous range of rows (so the rank, and
// with it the affines, change at most a few times).
constexpr int kRsRing = 4;
// Sixteen warps in all: four per SM sub-partition leave 128 registers a thread.
constexpr int kRsConsumers = 15;
constexpr int kRsVec = 2;  // 8-column vectors per consumer thread: 15 * 32 * 2 * 8 = 7680 columns
constexpr int kRsMaxH = 8 * 32 * kRsConsumers * kRsVec;
constexpr int kRsThreads = 32 * (kRsConsumers + 1);

__global__ void __launch_bounds__(kRsThreads, 1) ln_gate_bwd_rowsum_bulk_kernel(
    const __nv_bfloat16* __restrict__ Z, const float4* __restrict__ stats, const __nv_bfloat16* __restrict__ dHl,
    const __nv_bfloat16* __restrict__ gx, const __nv_bfloat16* __restrict__ bx, const __nv_bfloat16* __restrict__ gg,
    const __nv_bfloat16* __restrict__ bg, float4* __restrict__ rc, int64_t rows, int M, int L, int H,
    int slot_bytes, uint32_t* err) {
  extern __shared__ __align__(128) uint8_t rs_smem[];
  float4* part = reinterpret_cast<float4*>(rs_smem + kRsRing * slot_bytes);  // [kRsRing][kRsConsumers][32]
  uint64_t* full = reinterpret_cast<uint64_t*>(part + kRsRing * kRsConsumers * 32);
  uint64_t* empty = full + kRsRing;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kRsRing; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kRsConsumers);  // one release per consumer warp
    }
    fence_mbar_init();
  }
  griddep_wait();
  if (block_aborted(err)) return;  // (its barrier also publishes the barrier initialisation)
  const int64_t per = (rows + gridDim.x - 1) / gridDim.x;
  const int64_t r0 = min(rows, static_cast<int64_t>(blockIdx.x) * per);
  const int n = static_cast<int>(min(rows, r0 + per) - r0);
  const uint32_t zbytes = 4u * H, hbytes = 2u * H;
  const int nvec = H >> 3;
  const float inv_h = 1.0f / static_cast<float>(H);

  if (warp == kRsConsumers) {
    // ---------------------------------------------------------------- producer
    // The whole warp: lane 0 issues the copies, every lane takes part in the
    // reduction of a recycled row.  The row's four sums: each lane adds the
    // partials of its lane position over the consumer warps in warp order,
    // then a reduce-scatter over the lanes (after the xor-16 step a lane keeps
    // two of the sums, after the xor-8 step one; lanes 0, 8, 16 and 24 end
    // with sums 0 to 3), and lane 0 writes the record; the slot still holds
    // the row's statistics.
    const bool hi = (lane & 16) != 0, mid = (lane & 8) != 0;
    auto finish = [&](int i) {
      const int sl = i % kRsRing;
      const float4* pp = part + sl * kRsConsumers * 32 + lane;
      float4 a = pp[0];
      for (int w = 1; w < kRsConsumers; ++w) {
        const float4 b = pp[32 * w];
        a.x += b.x;
        a.y += b.y;
        a.z += b.z;
        a.w += b.w;
      }
      const float k0 = (hi ? a.z : a.x) + __shfl_xor_sync(0xffffffffu, hi ? a.x : a.z, 16);
      const float k1 = (hi ? a.w : a.y) + __shfl_xor_sync(0xffffffffu, hi ? a.y : a.w, 16);
      float t = (mid ? k1 : k0) + __shfl_xor_sync(0xffffffffu, mid ? k0 : k1, 8);
#pragma unroll
      for (int o = 4; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
      const float t1 = __shfl_sync(0xffffffffu, t, 8), t2 = __shfl_sync(0xffffffffu, t, 16);
      const float t3 = __shfl_sync(0xffffffffu, t, 24);
      if (lane == 0) {
        const float4 sr = *reinterpret_cast<const float4*>(rs_smem + sl * slot_bytes + zbytes + hbytes);
        store_row_coef(rc + 2 * (r0 + i), sr, make_float4(t, t1, t2, t3), inv_h);
      }
      __syncwarp();
    };
    bool ok = true;
    int issued = 0;
    for (int i = 0; i < n && ok; ++i) {
      const int s = i % kRsRing;
      if (i >= kRsRing) {
        if (!__all_sync(0xffffffffu, mbar_wait(&empty[s], static_cast<uint32_t>(i / kRsRing - 1) & 1u, err, 0x50u))) {
          ok = false;
          break;
        }
        finish(i - kRsRing);
      }
      if (lane == 0) {
        uint8_t* slot = rs_smem + s * slot_bytes;
        const int64_t row = r0 + i;
        mbar_arrive_expect_tx(&full[s], zbytes + hbytes + 16u);
        bulk_load(slot, Z + row * 2 * static_cast<int64_t>(H), zbytes, &full[s]);
        bulk_load(slot + zbytes, dHl + row * static_cast<int64_t>(H), hbytes, &full[s]);
        bulk_load(slot + zbytes + hbytes, stats + row, 16u, &full[s]);
      }
      __syncwarp();
      issued = i + 1;
    }
    for (int i = max(0, issued - kRsRing); i < issued && ok; ++i) {
      if (!__all_sync(0xffffffffu,
                      mbar_wait(&empty[i % kRsRing], static_cast<uint32_t>(i / kRsRing) & 1u, err, 0x51u))) {
        ok = false;
        break;
      }
      finish(i);
    }
    // every copy issued has landed before the CTA may exit
    if (lane == 0) {
      for (int i = max(0, issued - kRsRing); i < issued; ++i) {
        uint32_t dummy = 0;
        if (!mbar_try_wait(&full[i % kRsRing], static_cast<uint32_t>(i / kRsRing) & 1u))
          mbar_wait_slow(&full[i % kRsRing], static_cast<uint32_t>(i / kRsRing) & 1u, &dummy, 0x52u, kWaitLimitNs);
      }
    }
  } else {
    // ---------------------------------------------------------------- consumers
    // rank of the current row, and the local index of the first row of the next rank
    const int64_t rank_rows = static_cast<int64_t>(L) * M;
    int rank = static_cast<int>(r0 / rank_rows);
    int next_rank_at = static_cast<int>(min(static_cast<int64_t>(n), (rank + 1) * rank_rows - r0));
    bool reload = true;
    AffineF af[kRsVec];
    for (int i = 0; i < n; ++i) {
      const int s = i % kRsRing;
      const bool ok = mbar_wait(&full[s], static_cast<uint32_t>(i / kRsRing) & 1u, err, 0x53u);
      if (!__all_sync(0xffffffffu, ok)) break;
      if (i == next_rank_at) {
        ++rank;
        next_rank_at = static_cast<int>(min(static_cast<int64_t>(n), next_rank_at + rank_rows));
        reload = true;
      }
      if (reload) {
        reload = false;
#pragma unroll
        for (int j = 0; j < kRsVec; ++j) {
          const int v = warp * 32 + lane + 32 * kRsConsumers * j;
          if (v < nvec) {
            af[j] = load_affine_f(gx, bx, gg, bg, static_cast<int64_t>(rank) * H + 8 * v);
            halve_gate_affine(af[j]);
          }
        }
      }
      const uint8_t* slot = rs_smem + s * slot_bytes;
      const uint4* zrow = reinterpret_cast<const uint4*>(slot);
      const uint4* hrow = reinterpret_cast<const uint4*>(slot + zbytes);
      const float4 sr = *reinterpret_cast<const float4*>(slot + zbytes + hbytes);
      const float2 rsu = splat2(sr.y), cu = splat2(-sr.x * sr.y), rsg = splat2(sr.w), cgs = splat2(-sr.z * sr.w);
      // the four sums start from the first column pair's terms (no zeroing and
      // no first additions); a thread without any vector of this row holds zeros
      float2 s1u, s2u, s1g, s2g;
#pragma unroll
      for (int j = 0; j < kRsVec; ++j) {
        const int v = warp * 32 + lane + 32 * kRsConsumers * j;
        if (j == 0 && v >= nvec) s1u = s2u = s1g = s2g = splat2(0.f);
        if (v < nvec) {
          const uint4 pu = zrow[v], pg = zrow[nvec + v], ph = hrow[v];
          const uint32_t uw[4] = {pu.x, pu.y, pu.z, pu.w}, gw[4] = {pg.x, pg.y, pg.z, pg.w};
          const uint32_t hw[4] = {ph.x, ph.y, ph.z, ph.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 wx = af[j].wx[e], wg2 = af[j].wg[e];
            const GatePairH gp = gate_pair_h(unpack_bf16x2(uw[e]), unpack_bf16x2(gw[e]), rsu, cu, rsg, cgs, wx,
                                             af[j].cx[e], wg2, af[j].cg[e]);
            const float2 d = unpack_bf16x2(hw[e]);
            const float2 dxu = mul2(mul2(d, gp.q), wx);
            const float2 dxg = mul2(mul2(mul2(d, gp.a), gp.dsil2), wg2);
            if (j == 0 && e == 0) {
              s1u = dxu;
              s2u = mul2(dxu, gp.xu);
              s1g = dxg;
              s2g = mul2(dxg, gp.xg);
            } else {
              s1u = add2(s1u, dxu);
              s2u = fma2(dxu, gp.xu, s2u);
              s1g = add2(s1g, dxg);
              s2g = fma2(dxg, gp.xg, s2g);
            }
          }
        }
      }
      // this lane's four partial sums, for the producer warp to reduce
      part[(s * kRsConsumers + warp) * 32 + lane] =
          make_float4(s1u.x + s1u.y, s2u.x + s2u.y, s1g.x + s1g.y, s2g.x + s2g.y);
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
  }
}

// Pass 2 as a bulk-copy pipeline: one producer thread streams, per row, the
// CTA's column segments of U, G and dHl plus the row's coefficient record
// into a ring of shared-memory stages with cp.async.bulk; three consumer
// warps (8 columns a thread) hold the fp32 affines and the six column sums in
// registers, write dZ, and release each row's stage (one arrival a warp) at
// the start of the next row.  Four warps a CTA keep the SM's four
// sub-partitions evenly loaded.
constexpr int kApConsumers = 3;
constexpr int kApCols = 8 * 32 * kApConsumers;  // columns of one CTA: 768
constexpr int kApThreads = 32 * (kApConsumers + 1);
constexpr int kApRing = 8;
constexpr int kApSeg = 2 * kApCols;                 // bytes of one bf16 row segment
constexpr int kApStageBytes = 3 * kApSeg + 32;      // U, G, dHl segments, the row's coefficient record
constexpr int kApSmem = kApRing * kApStageBytes + 2 * kApRing * 8;

// grid: (column blocks of kApCols, T, row splits).
__global__ void __launch_bounds__(kApThreads, 4) ln_gate_bwd_apply_kernel(
    const __nv_bfloat16* __restrict__ Z, const float4* __restrict__ rc, const __nv_bfloat16* __restrict__ dHl,
    const __nv_bfloat16* __restrict__ gx, const __nv_bfloat16* __restrict__ bx, const __nv_bfloat16* __restrict__ gg,
    const __nv_bfloat16* __restrict__ bg, __nv_bfloat16* __restrict__ dZ, float* __restrict__ part, int M, int L, int H,
    uint32_t* err) {
  extern __shared__ __align__(128) uint8_t ap_smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(ap_smem + kApRing * kApStageBytes);
  uint64_t* empty = full + kApRing;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kApRing; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kApConsumers);
    }
    fence_mbar_init();
  }
  griddep_wait();
  if (block_aborted(err)) return;  // (its barrier also publishes the barrier initialisation)
  const int t = blockIdx.y, rsp = blockIdx.z, nsplit = gridDim.z;
  const int col0 = blockIdx.x * kApCols;
  const int wc = min(kApCols, H - col0);  // columns of this block, a multiple of 8
  const int rows_per = (M + nsplit - 1) / nsplit;
  const int n_begin = min(M, rsp * rows_per), n_end = min(M, n_begin + rows_per);
  const int n_rows = n_end - n_begin;
  const int64_t rowbase = static_cast<int64_t>(t) * M + n_begin;
  const int64_t zstride = 2 * static_cast<int64_t>(H);

  if (warp == kApConsumers) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      const uint32_t seg = 2u * static_cast<uint32_t>(wc);
      const __nv_bfloat16* zp = Z + rowbase * zstride + col0;
      const __nv_bfloat16* hp = dHl + rowbase * H + col0;
      int stage = 0, issued = 0;
      uint32_t phase = 0;
      for (int i = 0; i < n_rows; ++i) {
        // stage reuse waits for the consumers' release of row i - kApRing
        if (i >= kApRing && !mbar_wait(&empty[stage], phase ^ 1u, err, 0x54u)) break;
        uint8_t* slot = ap_smem + stage * kApStageBytes;
        mbar_arrive_expect_tx(&full[stage], 3u * seg + 32u);
        bulk_load(slot, zp, seg, &full[stage]);
        bulk_load(slot + kApSeg, zp + H, seg, &full[stage]);
        bulk_load(slot + 2 * kApSeg, hp, seg, &full[stage]);
        bulk_load(slot + 3 * kApSeg, rc + 2 * (rowbase + i), 32u, &full[stage]);
        zp += zstride;
        hp += H;
        issued = i + 1;
        if (++stage == kApRing) {
          stage = 0;
          phase ^= 1u;
        }
      }
      // every copy issued has landed before the CTA may exit
      for (int i = max(0, issued - kApRing); i < issued; ++i) {
        uint32_t dummy = 0;
        if (!mbar_try_wait(&full[i % kApRing], static_cast<uint32_t>(i / kApRing) & 1u))
          mbar_wait_slow(&full[i % kApRing], static_cast<uint32_t>(i / kApRing) & 1u, &dummy, 0x55u, kWaitLimitNs);
      }
    }
    return;
  }

  // ---------------------------------------------------------------- consumers
  const int v = warp * 32 + lane;
  const bool active = 8 * v < wc;
  const int c0 = col0 + (active ? 8 * v : 0);
  AffineF aff = load_affine_f(gx, bx, gg, bg, static_cast<int64_t>(t / L) * H + c0);
  halve_gate_affine(aff);
  float2 s_du[4], s_dg[4], s_gx[4], s_bx[4], s_gg[4], s_bg[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) s_du[e] = s_dg[e] = s_gx[e] = s_bx[e] = s_gg[e] = s_bg[e] = splat2(0.0f);
  __nv_bfloat16* dzp = dZ + rowbase * zstride + c0;
  int stage = 0;
  uint32_t phase = 0;
  for (int i = 0; i < n_rows; ++i) {
    const bool ok = mbar_wait(&full[stage], phase, err, 0x56u);
    if (!__all_sync(0xffffffffu, ok)) break;
    // Release the previous row's stage: every lane has issued that row's
    // stores (this warp-wide vote follows them), and they need values
    // computed from every load of the stage that is used, so those loads have
    // returned.  (Released right after its loads, a stage could be refilled
    // while a load of it was still being served, and the next row's copy
    // overwrote part of what it read.)  The last row's stage is never
    // released; nothing waits for it.
    if (i > 0 && lane == 0) mbar_arrive(&empty[stage == 0 ? kApRing - 1 : stage - 1]);
    const uint8_t* slot = ap_smem + stage * kApStageBytes;
    uint4 pu = make_uint4(0u, 0u, 0u, 0u), pg = pu, ph = pu;
    if (active) {
      pu = reinterpret_cast<const uint4*>(slot)[v];
      pg = reinterpret_cast<const uint4*>(slot + kApSeg)[v];
      ph = reinterpret_cast<const uint4*>(slot + 2 * kApSeg)[v];
    }
    const float4* rcs = reinterpret_cast<const float4*>(slot + 3 * kApSeg);
    const float4 cst = rcs[0], csum = rcs[1];
    if (++stage == kApRing) {
      stage = 0;
      phase ^= 1u;
    }
    if (active) {
      const float2 rsu = splat2(cst.x), cu = splat2(cst.y), rsg = splat2(cst.z), cgs = splat2(cst.w);
      const float2 m1u = splat2(csum.x), m2u = splat2(csum.y), m1g = splat2(csum.z), m2g = splat2(csum.w);
      const uint32_t uw[4] = {pu.x, pu.y, pu.z, pu.w}, gw[4] = {pg.x, pg.y, pg.z, pg.w}, hw[4] = {ph.x, ph.y, ph.z, ph.w};
      uint32_t ou[4], og[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const GatePairH gp = gate_pair_h(unpack_bf16x2(uw[e]), unpack_bf16x2(gw[e]), rsu, cu, rsg, cgs, aff.wx[e],
                                         aff.cx[e], aff.wg[e], aff.cg[e]);
        const float2 dh = unpack_bf16x2(hw[e]);
        const float2 da = mul2(dh, gp.q);
        const float2 ds = mul2(mul2(dh, gp.a), gp.dsil2);  // twice ds: aff.wg is halved, ds*gg = this*wg
        // dU = rstd_u * (da*gx - mean(dx_u) - x_u*mean(dx_u*x_u)); same for dG
        const float2 du = mul2(rsu, fma2(gp.xu, m2u, fma2(da, aff.wx[e], m1u)));
        const float2 dg = mul2(rsg, fma2(gp.xg, m2g, fma2(ds, aff.wg[e], m1g)));
        s_du[e] = add2(s_du[e], du);
        s_dg[e] = add2(s_dg[e], dg);
        s_gx[e] = fma2(da, gp.xu, s_gx[e]);
        s_bx[e] = add2(s_bx[e], da);
        s_gg[e] = fma2(ds, gp.xg, s_gg[e]);
        s_bg[e] = add2(s_bg[e], ds);
        ou[e] = pack_bf16x2(du.x, du.y);
        og[e] = pack_bf16x2(dg.x, dg.y);
      }
      __stcs(reinterpret_cast<uint4*>(dzp), make_uint4(ou[0], ou[1], ou[2], ou[3]));
      __stcs(reinterpret_cast<uint4*>(dzp + H), make_uint4(og[0], og[1], og[2], og[3]));
    }
    dzp += zstride;
  }
  if (!active) return;
  // part[t][split][q][c], q: dU, dG, da*x_u, da, ds*x_g, ds (the last two were summed twice over)
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    s_gg[e] = mul2(s_gg[e], splat2(0.5f));
    s_bg[e] = mul2(s_bg[e], splat2(0.5f));
  }
  float* pp = part + (static_cast<int64_t>(t) * nsplit + rsp) * 6 * H + c0;
  const float2* src[6] = {s_du, s_dg, s_gx, s_bx, s_gg, s_bg};
#pragma unroll
  for (int q = 0; q < 6; ++q) {
    float4* d4 = reinterpret_cast<float4*>(pp + q * static_cast<int64_t>(H));
    d4[0] = make_float4(src[q][0].x, src[q][0].y, src[q][1].x, src[q][1].y);
    d4[1] = make_float4(src[q][2].x, src[q][2].y, src[q][3].x, src[q][3].y);
  }
}

// db1 [T, 2H] and the norm gradients [P, H] from the partials, summed in a
// fixed order (row splits, then the rank's slices): reruns are bit-identical.
__global__ void grad_reduce_kernel(const float* __restrict__ part, __nv_bfloat16* __restrict__ d_b1,
                                   __nv_bfloat16* __restrict__ d_nx_w, __nv_bfloat16* __restrict__ d_nx_b,
                                   __nv_bfloat16* __restrict__ d_ng_w, __nv_bfloat16* __restrict__ d_ng_b, int P,
                                   int L, int H, int nsplit, const uint32_t* err) {
  griddep_wait();
  if (err_set(err)) return;
  const int T = P * L;
  const int64_t n_b1 = static_cast<int64_t>(T) * 2 * H;
  const int64_t n_norm = static_cast<int64_t>(P) * 4 * H;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n_b1 + n_norm;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    if (i < n_b1) {
      if (d_b1 == nullptr) continue;
      const int t = static_cast<int>(i / (2 * H));
      const int c2 = static_cast<int>(i - static_cast<int64_t>(t) * 2 * H);
      const int q = c2 >= H ? 1 : 0;
      const int c = c2 - q * H;
      float s = 0.0f;
      for (int k = 0; k < nsplit; ++k) s += part[((static_cast<int64_t>(t) * nsplit + k) * 6 + q) * H + c];
      d_b1[i] = __float2bfloat16_rn(s);
    } else {
      const int64_t j = i - n_b1;
      const int r = static_cast<int>(j / (4 * H));
      const int q = static_cast<int>((j / H) % 4);  // 0: nx_w, 1: nx_b, 2: ng_w, 3: ng_b
      const int c = static_cast<int>(j % H);
      if ((q == 0 ? d_nx_w : q == 1 ? d_nx_b : q == 2 ? d_ng_w : d_ng_b) == nullptr) continue;
      float s = 0.0f;
      for (int l = 0; l < L; ++l)
        for (int k = 0; k < nsplit; ++k)
          s += part[((static_cast<int64_t>(r * L + l) * nsplit + k) * 6 + 2 + q) * H + c];
      __nv_bfloat16* out = q == 0 ? d_nx_w : q == 1 ? d_nx_b : q == 2 ? d_ng_w : d_ng_b;
      if (out != nullptr) out[static_cast<int64_t>(r) * H + c] = __float2bfloat16_rn(s);
    }
  }
}

// out[g, c] = sum over rows n of src[g*g_stride + n*row_stride + c] for a slab
// of 256 columns per CTA: each lane owns 8 columns (one 16-byte load a row),
// the CTA's warps take interleaved rows, and their fp32 partials are added in
// warp order through shared memory.  Columns and row stride multiples of 8.
constexpr int kColSumWarps = 16;
__global__ void __launch_bounds__(32 * kColSumWarps) column_sum_slab_kernel(
    const __nv_bfloat16* __restrict__ src, __nv_bfloat16* __restrict__ out, int rows, int ncols, int64_t g_stride,
    int64_t row_stride, const uint32_t* err) {
  __shared__ float part[kColSumWarps][256 + 4];
  griddep_wait();
  if (err_set(err)) return;
  const int g = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.x * 256 + 8 * lane;
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  if (c < ncols) {
    const __nv_bfloat16* p = src + g * g_stride + c;
    int n = warp;
    for (; n + 3 * kColSumWarps < rows; n += 4 * kColSumWarps) {
      uint4 v[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) v[i] = __ldcs(reinterpret_cast<const uint4*>(p + (n + i * kColSumWarps) * row_stride));
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = unpack_bf16x2(w[e]);
          acc[2 * e] += f.x;
          acc[2 * e + 1] += f.y;
        }
      }
    }
    for (; n < rows; n += kColSumWarps) {
      const uint4 v = __ldcs(reinterpret_cast<const uint4*>(p + n * row_stride));
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = unpack_bf16x2(w[e]);
        acc[2 * e] += f.x;
        acc[2 * e + 1] += f.y;
      }
    }
  }
#pragma unroll
  for (int e = 0; e < 8; ++e) part[warp][8 * lane + e] = acc[e];
  __syncthreads();
  if (threadIdx.x < 128) {
    const int cc = blockIdx.x * 256 + 2 * threadIdx.x;
    float s0 = 0.f, s1 = 0.f;
#pragma unroll
    for (int w = 0; w < kColSumWarps; ++w) {
      s0 += part[w][2 * threadIdx.x];
      s1 += part[w][2 * threadIdx.x + 1];
    }
    if (cc < ncols) *reinterpret_cast<uint32_t*>(out + static_cast<int64_t>(g) * ncols + cc) = pack_bf16x2(s0, s1);
  }
}

// out[g, c] = sum over rows n of src[g*g_stride + n*row_stride + c]; two columns per thread.
__global__ void column_sum_kernel(const __nv_bfloat16* __restrict__ src, __nv_bfloat16* __restrict__ out, int rows,
                                  int ncols, int64_t g_stride, int64_t row_stride, const uint32_t* err) {
  griddep_wait();
  if (err_set(err)) return;
  const int g = blockIdx.y;
  const int c = 2 * (blockIdx.x * blockDim.x + threadIdx.x);
  if (c >= ncols) return;
  const __nv_bfloat16* p = src + g * g_stride + c;
  float s0 = 0.0f, s1 = 0.0f;
  int n = 0;
  for (; n + 4 <= rows; n += 4) {
    float2 v[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
      v[i] = unpack_bf16x2(__ldcs(reinterpret_cast<const uint32_t*>(p + (n + i) * row_stride)));
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      s0 += v[i].x;
      s1 += v[i].y;
    }
  }
  for (; n < rows; ++n) {
    const float2 v = unpack_bf16x2(__ldcs(reinterpret_cast<const uint32_t*>(p + n * row_stride)));
    s0 += v.x;
    s1 += v.y;
  }
  *reinterpret_cast<uint32_t*>(out + static_cast<int64_t>(g) * ncols + c) = pack_bf16x2(s0, s1);
}

// Backward of the SwiGLU gate h = silu(a) * b for the column-parallel pair:
// with sig = sigmoid(a),  da = dh * b * (sig + a*sig*(1 - sig)),  db = dh * a * sig,
// and h itself (needed for w2's gradient).  In place: (a, b) -> (da, db),
// dh -> h; 8 columns per thread.
__global__ void swiglu_gate_bwd_kernel(__nv_bfloat16* __restrict__ ab, __nv_bfloat16* __restrict__ dh_h, int64_t rows,
                                       int W, int F, const uint32_t* err) {
  griddep_wait();
  if (err_set(err)) return;
  const int fv = F / 8;
  const int64_t total = rows * W * fv;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t n = i / (static_cast<int64_t>(W) * fv);
    const int rem = static_cast<int>(i - n * W * fv);
    const int sh = rem / fv, c = 8 * (rem - sh * fv);
    __nv_bfloat16* pa = ab + (n * W + sh) * 2 * static_cast<int64_t>(F) + c;
    __nv_bfloat16* pb = pa + F;
    __nv_bfloat16* ph = dh_h + (n * W + sh) * static_cast<int64_t>(F) + c;
    const uint4 va = *reinterpret_cast<const uint4*>(pa), vb = *reinterpret_cast<const uint4*>(pb);
    const uint4 vh = *reinterpret_cast<const uint4*>(ph);
    const uint32_t aw[4] = {va.x, va.y, va.z, va.w}, bw[4] = {vb.x, vb.y, vb.z, vb.w};
    const uint32_t hw[4] = {vh.x, vh.y, vh.z, vh.w};
    uint32_t oa[4], ob[4], oh[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 a = unpack_bf16x2(aw[e]), b = unpack_bf16x2(bw[e]), d = unpack_bf16x2(hw[e]);
      const float2 half_a = mul2(a, splat2(0.5f));
      const float2 sig = fma2(make_float2(tanh_fast(half_a.x), tanh_fast(half_a.y)), splat2(0.5f), splat2(0.5f));
      const float2 as = mul2(a, sig);                                         // silu(a)
      const float2 dsil = fma2(as, fma2(sig, splat2(-1.0f), splat2(1.0f)), sig);  // silu'(a)
      const float2 da = mul2(mul2(d, b), dsil);
      const float2 db = mul2(d, as);
      const float2 h = mul2(as, b);
      oa[e] = pack_bf16x2(da.x, da.y);
      ob[e] = pack_bf16x2(db.x, db.y);
      oh[e] = pack_bf16x2(h.x, h.y);
    }
    *reinterpret_cast<uint4*>(pa) = make_uint4(oa[0], oa[1], oa[2], oa[3]);
    *reinterpret_cast<uint4*>(pb) = make_uint4(ob[0], ob[1], ob[2], ob[3]);
    *reinterpret_cast<uint4*>(ph) = make_uint4(oh[0], oh[1], oh[2], oh[3]);
  }
}

// Exchange permutations, 16 bytes per thread.  A NULL error word (the explicit
// permutation calls, which have no workspace) is not read.
__global__ void dispatch_kernel(const uint4* __restrict__ in, uint4* __restrict__ out, int P, int B, int T,
                                int vec_per_row, const uint32_t* err) {
  griddep_wait();
  if (err_set(err)) return;
  const int L = T / P, PB = P * B;
  const int64_t total = static_cast<int64_t>(P) * PB * L * vec_per_row;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t q = i / vec_per_row;  // destination row (r, n, l)
    const int c = static_cast<int>(i - q * vec_per_row);
    const int r = static_cast<int>(q / (static_cast<int64_t>(PB) * L));
    const int rem = static_cast<int>(q - static_cast<int64_t>(r) * PB * L);
    const int n = rem / L, l = rem - (rem / L) * L;
    const int64_t src_row = static_cast<int64_t>(n) * T + r * L + l;  // inputs[s][b][r*L+l], n = s*B+b
    out[i] = in[src_row * vec_per_row + c];
  }
}

__global__ void combine_kernel(const uint4* __restrict__ in, uint4* __restrict__ out, int P, int B, int T,
                               int vec_per_row, const uint32_t* err) {
  griddep_wait();
  if (err_set(err)) return;
  const int L = T / P, PB = P * B;
  const int64_t total = static_cast<int64_t>(PB) * T * vec_per_row;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t q = i / vec_per_row;  // destination row (s, b, t)
    const int c = static_cast<int>(i - q * vec_per_row);
    const int n = static_cast<int>(q / T), t = static_cast<int>(q - (q / T) * T);
    const int r = t / L, l = t - (t / L) * L;
    const int64_t src_row = (static_cast<int64_t>(r) * PB + n) * L + l;  // Ylocal[r][n][l]
    out[i] = in[src_row * vec_per_row + c];
  }
}

// comp_only layout (the exchange with the roles of rank and slice swapped):
// out row (p, b, r*L + l) = in row (r, b, p*L + l) of [P, B, T, D] tensors.
__global__ void swap_rank_slice_kernel(const uint4* __restrict__ in, uint4* __restrict__ out, int P, int B, int T,
                                       int vec_per_row, const uint32_t* err) {
  griddep_wait();
  if (err_set(err)) return;
  const int L = T / P;
  const int64_t total = static_cast<int64_t>(P) * B * T * vec_per_row;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t q = i / vec_per_row;  // destination row (p, b, t)
    const int c = static_cast<int>(i - q * vec_per_row);
    const int t = static_cast<int>(q % T);
    const int64_t pb = q / T;
    const int b = static_cast<int>(pb % B), p = static_cast<int>(pb / B);
    const int r = t / L, l = t - (t / L) * L;
    const int64_t src_row = (static_cast<int64_t>(r) * B + b) * T + static_cast<int64_t>(p) * L + l;
    out[i] = in[src_row * vec_per_row + c];
  }
}

// Waits, with the library's bounded wait, on a barrier nobody arrives at.
__global__ void debug_wait_kernel(uint32_t* err, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  griddep_wait();
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(&bar, 0u, err, 0x7fu, limit_ns);
}

}  // namespace

// The dynamic shared-memory limit of a kernel, raised once per device and
// kernel (a host-side attribute: kept off the launch path, and out of the way
// of stream capture).
static cudaError_t smem_attr_once(const void* kern, int bytes) {
  struct Entry {
    const void* kern;
    int device, bytes;
  };
  static std::mutex mu;
  static std::vector<Entry> done;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> g(mu);
  for (const Entry& x : done)
    if (x.kern == kern && x.device == dev && x.bytes >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done.push_back(Entry{kern, dev, bytes});
  return e;
}

// CTAs per rank so that the row kernels fill every SM (each CTA stays on one rank).
static int ctas_per_rank(const DeviceInfo& dev, const void* kernel, int threads, size_t smem, int P,
                         int64_t rank_rows) {
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, smem) != cudaSuccess || per_sm < 1)
    per_sm = 1;
  int64_t c = (static_cast<int64_t>(per_sm) * dev.num_sms + P - 1) / P;
  if (c > rank_rows) c = rank_rows;
  return static_cast<int>(c < 1 ? 1 : c);
}

// Block shape of the normalise-and-gate pass: NT threads x VPT 8-column
// vectors per CTA, and the number of CTAs (column blocks) one row is split
// over when it is wider than 8192 columns.
static void row_shape(int H, int* nt, int* vpt, int* col_blocks) {
  const int nvec = H / 8;
  *col_blocks = 1;
  if (nvec <= 256) { *nt = 256; *vpt = 1; return; }
  if (nvec <= 512) { *nt = 256; *vpt = 2; return; }
  *nt = 512;
  *vpt = 2;
  *col_blocks = (nvec + 1023) / 1024;
}

cudaError_t launch_ln_stats_finalize(const float4* part, void* stats, int T, int M, int H, int tile_n, int tiles_n,
                                     float eps, const DeviceInfo& dev, cudaStream_t s) {
  const int64_t rows = static_cast<int64_t>(T) * M;
  int64_t blocks = (rows + 255) / 256;
  if (blocks > 16 * dev.num_sms) blocks = 16 * dev.num_sms;
  return launch_pdl(ln_stats_finalize_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, s, part,
                    static_cast<float4*>(stats), T, M, H, tile_n, tiles_n, eps, dev.err);
}

cudaError_t launch_ln_gate_fwd(const void* Z, const void* stats, const void* nx_w, const void* nx_b, const void* ng_w,
                               const void* ng_b, void* Hl, uint8_t* hq, float* hs, int P, int M, int L, int H,
                               const DeviceInfo& dev, cudaStream_t s) {
  int nt = 0, vpt = 0, cb = 1;
  row_shape(H, &nt, &vpt, &cb);
  if (hq && cb != 1) return cudaErrorInvalidValue;  // e4m3 rows need the whole row in one CTA
  auto run = [&](auto kern) {
    const size_t smem = static_cast<size_t>(kFwdStages) * vpt * 2 * nt * 16;
    cudaError_t e = smem_attr_once(reinterpret_cast<const void*>(kern), static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    // CTAs per rank and column block, so that the grid fills every SM
    const int cpr =
        ctas_per_rank(dev, reinterpret_cast<const void*>(kern), nt, smem, P * cb, static_cast<int64_t>(L) * M);
    return launch_pdl(kern, dim3(P * cpr * cb), dim3(nt), smem, s, static_cast<const __nv_bfloat16*>(Z),
                      static_cast<const float4*>(stats), static_cast<const __nv_bfloat16*>(nx_w),
                      static_cast<const __nv_bfloat16*>(nx_b), static_cast<const __nv_bfloat16*>(ng_w),
                      static_cast<const __nv_bfloat16*>(ng_b), static_cast<__nv_bfloat16*>(Hl), hq, hs, M, L, H, cpr,
                      cb, dev.err);
  };
  if (hq && H <= kGfMaxH) {
    // bulk-copy pipeline: kGfRing slots of a Z row and its statistics
    const int64_t rows = static_cast<int64_t>(P) * L * M;
    if (rows == 0) return cudaSuccess;
    const int slot_bytes = (4 * H + 16 + 127) / 128 * 128;
    const int smem = kGfRing * slot_bytes + kGfVbuf * H * 4 + (2 * kGfRing + kGfSlots) * 8 + kGfSlots * kGfConsumers * 4;
    auto kern = H == kGfMaxH ? ln_gate_fwd_fp8_bulk_kernel<true> : ln_gate_fwd_fp8_bulk_kernel<false>;
    cudaError_t e = smem_attr_once(reinterpret_cast<const void*>(kern), smem);
    if (e != cudaSuccess) return e;
    int64_t blocks = dev.num_sms;
    if (blocks > rows) blocks = rows;
    return launch_pdl(kern, dim3(static_cast<unsigned>(blocks)), dim3(kGfThreads),
                      static_cast<size_t>(smem), s, static_cast<const __nv_bfloat16*>(Z),
                      static_cast<const float4*>(stats), static_cast<const __nv_bfloat16*>(nx_w),
                      static_cast<const __nv_bfloat16*>(nx_b), static_cast<const __nv_bfloat16*>(ng_w),
                      static_cast<const __nv_bfloat16*>(ng_b), hq, hs, rows, M, L, H, slot_bytes, dev.err);
  }
  if (hq) {
    if (nt == 256 && vpt == 1) return run(ln_gate_fwd_kernel<256, 1, true>);
    if (nt == 256) return run(ln_gate_fwd_kernel<256, 2, true>);
    return run(ln_gate_fwd_kernel<512, 2, true>);
  }
  if (nt == 256 && vpt == 1) return run(ln_gate_fwd_kernel<256, 1, false>);
  if (nt == 256) return run(ln_gate_fwd_kernel<256, 2, false>);
  return run(ln_gate_fwd_kernel<512, 2, false>);
}

cudaError_t launch_quant_rows(const void* x, void* q, float* scale, int64_t rows, int D, int T, int M,
                              const DeviceInfo& dev, cudaStream_t s) {
  int64_t blocks = (rows + 7) / 8;
  if (blocks > 16 * dev.num_sms) blocks = 16 * dev.num_sms;
  return launch_pdl(quant_rows_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, s,
                    static_cast<const __nv_bfloat16*>(x), static_cast<uint8_t*>(q), scale, rows, D, T, M, dev.err);
}

cudaError_t launch_quant_weight(const void* w, float* scale, float* inv, void* q, int G, int K, int N,
                                const DeviceInfo& dev, cudaStream_t s) {
  cudaError_t e = launch_pdl(col_scale_kernel, dim3((N + 255) / 256, G), dim3(256), 0, s,
                             static_cast<const __nv_bfloat16*>(w), scale, inv, K, N, dev.err);
  if (e != cudaSuccess) return e;
  return launch_pdl(transpose_quant_kernel, dim3((N + 63) / 64, (K + 63) / 64, G), dim3(256), 0, s,
                    static_cast<const __nv_bfloat16*>(w), static_cast<const float*>(inv), static_cast<uint8_t*>(q), K,
                    N, dev.err);
}

cudaError_t launch_ln_gate_bwd_rowsum(const void* Z, const void* stats, const void* dHl, const void* nx_w,
                                      const void* nx_b, const void* ng_w, const void* ng_b, void* rc, int T, int M,
                                      int L, int H, const DeviceInfo& dev, cudaStream_t s) {
  const int64_t rows = static_cast<int64_t>(T) * M;
  if (H <= kRsMaxH) {
    // bulk-copy pipeline: kRsRing row slots of the U|G row, the dHl row and the statistics
    const int slot_bytes = (6 * H + 16 + 127) / 128 * 128;
    const int smem = kRsRing * slot_bytes + kRsRing * kRsConsumers * 32 * 16 + 2 * kRsRing * 8;
    cudaError_t e = smem_attr_once(reinterpret_cast<const void*>(ln_gate_bwd_rowsum_bulk_kernel), smem);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, ln_gate_bwd_rowsum_bulk_kernel, kRsThreads, smem) !=
            cudaSuccess ||
        per_sm < 1)
      per_sm = 1;
    int64_t blocks = static_cast<int64_t>(per_sm) * dev.num_sms;
    if (blocks > rows) blocks = rows;
    return launch_pdl(ln_gate_bwd_rowsum_bulk_kernel, dim3(static_cast<unsigned>(blocks)), dim3(kRsThreads),
                      static_cast<size_t>(smem), s, static_cast<const __nv_bfloat16*>(Z),
                      static_cast<const float4*>(stats), static_cast<const __nv_bfloat16*>(dHl),
                      static_cast<const __nv_bfloat16*>(nx_w), static_cast<const __nv_bfloat16*>(nx_b),
                      static_cast<const __nv_bfloat16*>(ng_w), static_cast<const __nv_bfloat16*>(ng_b),
                      static_cast<float4*>(rc), rows, M, L, H, slot_bytes, dev.err);
  }
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, ln_gate_bwd_rowsum_kernel, kRowsumThreads, 0) !=
          cudaSuccess ||
      per_sm < 1)
    per_sm = 1;
  int64_t blocks = static_cast<int64_t>(per_sm) * dev.num_sms;
  const int64_t need = (rows + kRowsumThreads / 32 - 1) / (kRowsumThreads / 32);
  if (blocks > need) blocks = need;
  return launch_pdl(ln_gate_bwd_rowsum_kernel, dim3(static_cast<unsigned>(blocks)), dim3(kRowsumThreads), 0, s,
      static_cast<const __nv_bfloat16*>(Z), static_cast<const float4*>(stats), static_cast<const __nv_bfloat16*>(dHl),
      static_cast<const __nv_bfloat16*>(nx_w), static_cast<const __nv_bfloat16*>(nx_b),
      static_cast<const __nv_bfloat16*>(ng_w), static_cast<const __nv_bfloat16*>(ng_b), static_cast<float4*>(rc),
      rows, M, L, H, dev.err);
}

int ffn_bwd_row_splits(int T, int M, int H) {
  // about sixteen waves of (t, column block, row range) items at four CTAs per
  // SM, and no fewer than 128 rows an item where M allows
  const int blocks = (H + kApCols - 1) / kApCols;
  int splits = (10240 + T * blocks - 1) / (T * blocks);
  const int cap = (M + 127) / 128;
  if (splits > cap) splits = cap;
  return splits < 1 ? 1 : splits;
}

cudaError_t launch_ln_gate_bwd_apply(const void* Z, const void* rc, const void* dHl, const void* nx_w,
                                     const void* nx_b, const void* ng_w, const void* ng_b, void* dZ, float* part, int T,
                                     int M, int L, int H, int nsplit, const DeviceInfo& dev, cudaStream_t s) {
  dim3 grid((H + kApCols - 1) / kApCols, T, nsplit);
  cudaError_t e = smem_attr_once(reinterpret_cast<const void*>(ln_gate_bwd_apply_kernel), kApSmem);
  if (e != cudaSuccess) return e;
  return launch_pdl(ln_gate_bwd_apply_kernel, grid, dim3(kApThreads), kApSmem, s,
      static_cast<const __nv_bfloat16*>(Z), static_cast<const float4*>(rc), static_cast<const __nv_bfloat16*>(dHl),
      static_cast<const __nv_bfloat16*>(nx_w), static_cast<const __nv_bfloat16*>(nx_b),
      static_cast<const __nv_bfloat16*>(ng_w), static_cast<const __nv_bfloat16*>(ng_b),
      static_cast<__nv_bfloat16*>(dZ), part, M, L, H, dev.err);
}

cudaError_t launch_grad_reduce(const float* part, void* d_b1, void* d_nx_w, void* d_nx_b, void* d_ng_w, void* d_ng_b,
                               int P, int L, int H, int nsplit, const DeviceInfo& dev, cudaStream_t s) {
  const int64_t n = static_cast<int64_t>(P) * L * 2 * H + static_cast<int64_t>(P) * 4 * H;
  int64_t blocks = (n + 255) / 256;
  if (blocks > 8 * dev.num_sms) blocks = 8 * dev.num_sms;
  return launch_pdl(grad_reduce_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, s,
      part, static_cast<__nv_bfloat16*>(d_b1), static_cast<__nv_bfloat16*>(d_nx_w), static_cast<__nv_bfloat16*>(d_nx_b),
      static_cast<__nv_bfloat16*>(d_ng_w), static_cast<__nv_bfloat16*>(d_ng_b), P, L, H, nsplit, dev.err);
}

cudaError_t launch_column_sum(const void* src, void* out, int G, int rows, int ncols, int64_t g_stride,
                              int64_t row_stride, const DeviceInfo& dev, cudaStream_t s) {
  if (ncols % 8 == 0 && row_stride % 8 == 0 && g_stride % 8 == 0 && (reinterpret_cast<uintptr_t>(src) & 15u) == 0)
    return launch_pdl(column_sum_slab_kernel, dim3((ncols + 255) / 256, G), dim3(32 * kColSumWarps), 0, s,
                      static_cast<const __nv_bfloat16*>(src), static_cast<__nv_bfloat16*>(out), rows, ncols, g_stride,
                      row_stride, dev.err);
  const int threads = 128;
  dim3 grid((ncols / 2 + threads - 1) / threads, G);
  return launch_pdl(column_sum_kernel, grid, dim3(threads), 0, s, static_cast<const __nv_bfloat16*>(src),
                    static_cast<__nv_bfloat16*>(out), rows, ncols, g_stride, row_stride, dev.err);
}

cudaError_t launch_swiglu_gate_bwd(void* ab, void* dh_h, int64_t rows, int W, int F, const DeviceInfo& dev,
                                   cudaStream_t s) {
  const int64_t total = rows * W * (F / 8);
  int64_t blocks = (total + 255) / 256;
  if (blocks > 16 * dev.num_sms) blocks = 16 * dev.num_sms;
  return launch_pdl(swiglu_gate_bwd_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, s,
                    static_cast<__nv_bfloat16*>(ab), static_cast<__nv_bfloat16*>(dh_h), rows, W, F, dev.err);
}

cudaError_t launch_dispatch(const void* in, void* out, int P, int B, int T, int D, const DeviceInfo& dev,
                            cudaStream_t s) {
  const int64_t total = static_cast<int64_t>(P) * B * T * (D / 8);
  int64_t blocks = (total + 255) / 256;
  if (blocks > 16 * dev.num_sms) blocks = 16 * dev.num_sms;
  return launch_pdl(dispatch_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, s,
                    static_cast<const uint4*>(in), static_cast<uint4*>(out), P, B, T, D / 8, dev.err);
}

cudaError_t launch_combine(const void* in, void* out, int P, int B, int T, int D, const DeviceInfo& dev,
                           cudaStream_t s) {
  const int64_t total = static_cast<int64_t>(P) * B * T * (D / 8);
  int64_t blocks = (total + 255) / 256;
  if (blocks > 16 * dev.num_sms) blocks = 16 * dev.num_sms;
  return launch_pdl(combine_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, s,
                    static_cast<const uint4*>(in), static_cast<uint4*>(out), P, B, T, D / 8, dev.err);
}

cudaError_t launch_swap_rank_slice(const void* in, void* out, int P, int B, int T, int D, const DeviceInfo& dev,
                                   cudaStream_t s) {
  const int64_t total = static_cast<int64_t>(P) * B * T * (D / 8);
  int64_t blocks = (total + 255) / 256;
  if (blocks > 16 * dev.num_sms) blocks = 16 * dev.num_sms;
  return launch_pdl(swap_rank_slice_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, s,
                    static_cast<const uint4*>(in), static_cast<uint4*>(out), P, B, T, D / 8, dev.err);
}

cudaError_t launch_debug_wait(uint32_t* err, uint64_t limit_ns, cudaStream_t s) {
  return launch_pdl(debug_wait_kernel, dim3(1), dim3(32), 0, s, err, limit_ns);
}

}  // namespace dg
