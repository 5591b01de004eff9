// Persistent, warp-specialised tcgen05 GEMM for sm_103a.
//
// One CTA per SM walks a static tile schedule.  Per CTA:
//   warp 0   TMA producer: fills a STAGES-deep ring of (A, B) K-blocks in
//            shared memory, 128-byte swizzled, signalling `full[s]`.
//   warp 1   allocates TMEM (two 128 x BN fp32 accumulators) and one lane
//            issues tcgen05.mma for every K-block, releasing smem stages
//            through tcgen05.commit -> `empty[s]` and handing a finished
//            accumulator to the epilogue through `tfull[a]`.
//   warps 2-5 epilogue: tcgen05.ld the accumulator (32 rows per warp),
//            apply the fused epilogue, round to bf16, write 32x64 sub-tiles
//            into swizzled staging buffers and TMA-store them.  The two
//            accumulators let the epilogue of tile i overlap the mainloop
//            of tile i+1.
//
// Operands are described by 3-D TMA tensor maps whose coordinates are
// (x, y, g) or (x, g, y): x is the contiguous dimension, y the other matrix
// dimension and g the problem ("group") index.  A problem whose rows are
// strided through a larger tensor -- the dispatched rows of the A2A layer --
// is therefore just another tensor map: the exchange costs no data movement.
//
// Operand majorness: K-major tiles are [rows][64 bf16 | 128 e4m3] (one
// 128-byte swizzle row per tile row); MN-major tiles are [64 k-rows][64 mn]
// boxes stacked along MN.  The UMMA smem descriptors below encode those two
// canonical layouts.
#pragma once

#include "dg_gate.cuh"
#include "dg_ptx.cuh"

namespace dg {

enum GMode : int32_t { G_OUTER = 0, G_MID = 1, G_NONE = 2 };
enum Epi : int32_t {
  EPI_STORE = 0,         // D = acc
  EPI_BIAS = 1,          // D = acc + bias
  EPI_FP8 = 2,           // D = alpha*acc + beta*C
  EPI_SWIGLU = 3,        // D = silu(acc[:, :BN/2]) * acc[:, BN/2:]
  EPI_BIAS_LNSTATS = 4   // D = acc + bias, and per-tile (mean, M2) of each row's U and G columns
};

// Wait-site codes recorded with a timeout.
enum WaitSite : uint32_t {
  SITE_EMPTY = 1, SITE_FULL = 2, SITE_TEMPTY = 3, SITE_TFULL = 4, SITE_CLOAD = 5, SITE_DRAIN = 6, SITE_PARAM = 7
};

struct GemmParams {
  int32_t G, M, N, K;        // problems; rows, output columns, contraction of each problem
  int32_t tiles_m, tiles_n;  // tiles per problem
  int32_t n_fastest;         // tile order within a problem: 0 = row tiles fastest, 1 = column tiles fastest
  int32_t a_g, b_g, d_g;     // GMode of the group coordinate of A, B and D (C follows D)
  const __nv_bfloat16* bias; // EPI_BIAS: bias[g * bias_g_stride + n]
  int64_t bias_g_stride;
  float alpha, beta;         // EPI_FP8
  int32_t has_c;             // EPI_FP8: read C
  float4* ln_part;           // EPI_BIAS_LNSTATS: [G][tiles_n][M] (mean_u, M2_u, mean_g, M2_g) per tile
  int32_t ln_H;              // EPI_BIAS_LNSTATS: columns [0, ln_H) are U, [ln_H, N) are G
  uint32_t* err;             // device error word
  const __nv_bfloat16* c_ptr; // narrow tiles: C and D as row-major [G][M][N] for the last 32-column chunk
  __nv_bfloat16* d_ptr;
  // e4m3 variants other than EPI_FP8: acc is dequantised as
  // acc * row_scale[g*row_scale_g + m] * col_scale[g*col_scale_g + n] before the bias
  const float* row_scale;
  const float* col_scale;
  int64_t row_scale_g, col_scale_g;
  // MN-major A / B described by a 4-D map (mn mod 64, the two other
  // coordinates, mn / 64): one copy fetches all 64-wide MN blocks of a stage.
  // Set only when the operand's MN extent is a multiple of 64.
  int32_t a_mn4, b_mn4;
};

// Running (count, mean, M2) of a set of values; merge() is the pairwise
// combination of Chan, Golub & LeVeque ("Updating formulae and a pairwise
// algorithm for computing sample variances").
struct MeanM2 {
  float n, mean, m2;
  __device__ __forceinline__ void merge(float nb, float mean_b, float m2_b) {
    if (nb <= 0.0f) return;
    const float nn = n + nb;
    const float d = mean_b - mean;
    const float f = nb / nn;
    mean = fmaf(d, f, mean);
    m2 = m2 + m2_b + d * d * n * f;
    n = nn;
  }
};

// Two-pass (mean, M2) of v[lo, hi) -- values held in registers.
template <int K>
static __device__ __forceinline__ void chunk_mean_m2(const float (&v)[K], int lo, int hi, float& mean, float& m2) {
  float s = 0.0f;
#pragma unroll
  for (int i = 0; i < K; ++i) s += (i >= lo && i < hi) ? v[i] : 0.0f;
  const float n = static_cast<float>(hi - lo);
  mean = s / n;
  float q = 0.0f;
#pragma unroll
  for (int i = 0; i < K; ++i) {
    const float d = v[i] - mean;
    q = (i >= lo && i < hi) ? fmaf(d, d, q) : q;
  }
  m2 = q;
}

template <bool kFp8, bool kAMN, bool kBMN, int kEpi, bool kPair, int kBN = 256>
struct GemmCfg {
  static constexpr int CTAS = kPair ? 2 : 1;          // CTAs sharing one UMMA (cta_group)
  static constexpr int BM = 128;                      // rows per CTA (one TMEM lane per row)
  static constexpr int UMMA_M = BM * CTAS;            // rows per MMA tile
  static constexpr int BN = kBN;                      // UMMA N = accumulator columns
  static constexpr int ACC_STRIDE = 256;              // TMEM columns between the two accumulators
  static constexpr int BN_OUT = (kEpi == EPI_SWIGLU) ? BN / 2 : BN;
  static constexpr int B_ROWS = BN / CTAS;            // B rows each CTA stages per K-block
  static constexpr int ROW_BYTES = 128;               // K-block = one 128-byte swizzle row
  static constexpr int BK = kFp8 ? 128 : 64;          // K elements per stage
  static constexpr int K_STEPS = 4;                   // UMMA K = 32 bytes: 16 bf16 / 32 e4m3
  // per-tile epilogue parameters staged in shared memory (bias, e4m3 column scales)
  static constexpr bool HAS_BIAS = kEpi == EPI_BIAS || kEpi == EPI_BIAS_LNSTATS;
  static constexpr bool HAS_SCALES = kFp8 && kEpi != EPI_FP8;
  static constexpr int STAGES = kPair ? (HAS_SCALES ? 5 : 6) : 4;
  static constexpr int A_BYTES = BM * ROW_BYTES;      // 16 KB
  static constexpr int B_BYTES = B_ROWS * ROW_BYTES;  // 16 KB (pair) or 32 KB
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int MN_BOX_BYTES = 64 * 64 * 2;    // MN-major box: 64 k-rows x 64 bf16
  static constexpr int EPI_WARPS = 4;
  static constexpr int EPI_BUF_BYTES = 32 * 128;      // 32 rows x 64 bf16
  static constexpr int EPI_BYTES = EPI_WARPS * 2 * EPI_BUF_BYTES;
  static constexpr int NUM_THREADS = 64 + EPI_WARPS * 32;
  static constexpr int NACC = 2;                      // TMEM accumulators (double buffered)
  static constexpr uint32_t TMEM_COLS = NACC * ACC_STRIDE;
  static constexpr bool HALF_CHUNK = (BN_OUT % 64) == 32;  // a last 32-column chunk per tile
  static constexpr int BIAS_BYTES = HAS_BIAS ? BN_OUT * 2 : 0;    // one tile's bias, bf16
  static constexpr int SCALE_BYTES = HAS_SCALES ? BN_OUT * 4 : 0; // one tile's column scales, f32
  static constexpr int PARAM_BYTES = 2 * (BIAS_BYTES + SCALE_BYTES);  // double buffered
  static constexpr int NUM_BARS = 2 * STAGES + 4 + 2 * EPI_WARPS + 1 + 2;
  static constexpr int BAR_BYTES = 256;
  static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + EPI_BYTES + PARAM_BYTES + BAR_BYTES;
  static constexpr uint32_t IDESC = umma_idesc(kFp8 ? 0u : 1u, kAMN, kBMN, BN, UMMA_M);
  static_assert(NUM_BARS * 8 + 4 <= BAR_BYTES, "barrier area");
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
  static_assert(!(kFp8 && (kAMN || kBMN)), "e4m3 operands are K-major here");
  static_assert(!kFp8 || kEpi == EPI_FP8 || kEpi == EPI_BIAS || kEpi == EPI_BIAS_LNSTATS, "e4m3 epilogues");
  static_assert(kBN <= ACC_STRIDE && kBN % 32 == 0 && (kBN / CTAS) % 8 == 0, "tile width");
  static_assert(kBN == 256 || kEpi == EPI_FP8, "narrow tiles: the alpha/beta/C epilogue only");
};

static __device__ __forceinline__ void tma_load_op(void* dst, const CUtensorMap* map, uint64_t* bar, int32_t x,
                                                   int32_t y, int32_t g, int32_t mode) {
  if (mode == G_MID) {
    tma_load_3d(dst, map, bar, x, g, y);
  } else if (mode == G_OUTER) {
    tma_load_3d(dst, map, bar, x, y, g);
  } else {
    tma_load_3d(dst, map, bar, x, y, 0);
  }
}

static __device__ __forceinline__ void tma_store_op(const CUtensorMap* map, const void* src, int32_t x, int32_t y,
                                                    int32_t g, int32_t mode) {
  if (mode == G_MID) {
    tma_store_3d(map, src, x, g, y);
  } else if (mode == G_OUTER) {
    tma_store_3d(map, src, x, y, g);
  } else {
    tma_store_3d(map, src, x, y, 0);
  }
}

static __device__ __forceinline__ float silu_f(float x) { return x / (1.0f + __expf(-x)); }

// (row tile, column tile) of the rem-th tile of a problem in the launch's order.
static __device__ __forceinline__ void tile_coords(const GemmParams& p, int rem, int& mt, int& nt) {
  if (p.n_fastest) {
    mt = rem / p.tiles_n;
    nt = rem - mt * p.tiles_n;
  } else {
    nt = rem / p.tiles_m;
    mt = rem - nt * p.tiles_m;
  }
}

template <bool kFp8, bool kAMN, bool kBMN, int kEpi, bool kPair, int kBN>
__global__ void __launch_bounds__(GemmCfg<kFp8, kAMN, kBMN, kEpi, kPair, kBN>::NUM_THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmD, const __grid_constant__ CUtensorMap tmC,
                   const GemmParams p) {
  using Cfg = GemmCfg<kFp8, kAMN, kBMN, kEpi, kPair, kBN>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint32_t s_abort;

  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  uint8_t* stage_base = smem;
  uint8_t* epi_base = smem + Cfg::STAGES * Cfg::STAGE_BYTES;
  uint8_t* param_base = epi_base + Cfg::EPI_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(param_base + Cfg::PARAM_BYTES);
  uint64_t* full = bars;
  uint64_t* empty = bars + Cfg::STAGES;
  uint64_t* tfull = bars + 2 * Cfg::STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* cbar = tempty + 2;
  uint64_t* drain = cbar + 2 * Cfg::EPI_WARPS;
  uint64_t* pready = drain + 1;  // [2]: a tile's epilogue parameters are in shared memory
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(pready + 2);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  const uint32_t rank = kPair ? cluster_ctarank() : 0u;  // position in the CTA pair
  const bool leader = rank == 0u;

  // Prologue: barriers and descriptor prefetch touch nothing a preceding
  // kernel writes, so with programmatic launch they overlap its tail.
  if (warp == 0 && lane == 0) {
    for (int s = 0; s < Cfg::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], Cfg::EPI_WARPS * Cfg::CTAS);
    }
    for (int i = 0; i < 2 * Cfg::EPI_WARPS; ++i) mbar_init(&cbar[i], 1);
    mbar_init(drain, 1);
    mbar_init(&pready[0], Cfg::EPI_WARPS);
    mbar_init(&pready[1], Cfg::EPI_WARPS);
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmD);
    if (kEpi == EPI_FP8 && p.has_c) tma_prefetch_desc(&tmC);
  }
  if (kPair) cluster_sync_all();  // both CTAs run before any access to the peer's shared memory
  griddep_wait();                 // inputs and the error word may come from the preceding kernel

  // A sticky device error from an earlier failure: do nothing.  In a CTA pair
  // the leader decides for both, so the pair's control flow stays uniform
  // (the value is published by the barrier after the TMEM allocation).
  if (threadIdx.x == 0) {
    const uint32_t v = ld_volatile_u32(p.err);
    if (kPair) {
      if (leader) {
        st_cluster_u32(mapa_shared(smem_u32(&s_abort), 0), v);
        st_cluster_u32(mapa_shared(smem_u32(&s_abort), 1), v);
      }
    } else {
      s_abort = v;
    }
  }
  if (warp == 1) {
    if (kPair) {
      tmem_alloc_pair(tmem_holder, Cfg::TMEM_COLS);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(tmem_holder, Cfg::TMEM_COLS);
      tmem_relinquish();
    }
  }
  tc_fence_before_sync();
  if (kPair)
    cluster_sync_all();
  else
    __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_holder;
  const bool aborted = s_abort != 0u;

  const int tiles_per_group = p.tiles_m * p.tiles_n;
  const int total_tiles = p.G * tiles_per_group;
  const int num_kb = (p.K + Cfg::BK - 1) / Cfg::BK;
  const int unit = static_cast<int>(blockIdx.x) / Cfg::CTAS;  // this CTA's (pair's) slot in the schedule
  const int num_units = static_cast<int>(gridDim.x) / Cfg::CTAS;

  if (aborted) {
    // nothing to do: straight to the teardown (TMEM is freed there)
  } else if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t armed = 0, armed_parity = 0;
      bool ok = true;
      for (int tile = unit; tile < total_tiles && ok; tile += num_units) {
        const int g = tile / tiles_per_group;
        const int rem = tile - g * tiles_per_group;
        int mt, nt;
        tile_coords(p, rem, mt, nt);
        const int m0 = mt * Cfg::UMMA_M + static_cast<int>(rank) * Cfg::BM;
        const int n0 = nt * Cfg::BN_OUT;
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, p.err, SITE_EMPTY)) {
            ok = false;
            break;
          }
          // The pair's loads all complete on the leader's full barrier.
          if (leader) mbar_arrive_expect_tx(&full[stage], Cfg::STAGE_BYTES * Cfg::CTAS);
          const uint32_t bar_c = kPair ? mapa_shared(smem_u32(&full[stage]), 0) : smem_u32(&full[stage]);
          uint8_t* sa = stage_base + stage * Cfg::STAGE_BYTES;
          uint8_t* sb = sa + Cfg::A_BYTES;
          const int k0 = kb * Cfg::BK;
          auto load = [&](void* dst, const CUtensorMap* map, int32_t x, int32_t y, int32_t g3, int32_t mode) {
            int32_t c1 = y, c2 = g3;
            if (mode == G_MID) {
              c1 = g3;
              c2 = y;
            } else if (mode == G_NONE) {
              c2 = 0;
            }
            if (kPair)
              tma_load_3d_pair(dst, map, bar_c, x, c1, c2);
            else
              tma_load_3d(dst, map, &full[stage], x, c1, c2);
          };
          // MN-major, one copy: coordinates (0, k, g, mn/64) in the map's order
          auto load_mn4 = [&](void* dst, const CUtensorMap* map, int32_t k, int32_t mn_blk, int32_t g3,
                              int32_t mode) {
            int32_t c1 = k, c2 = g3;
            if (mode == G_MID) {
              c1 = g3;
              c2 = k;
            } else if (mode == G_NONE) {
              c2 = 0;
            }
            if (kPair)
              tma_load_4d_pair(dst, map, bar_c, 0, c1, c2, mn_blk);
            else
              tma_load_4d(dst, map, &full[stage], 0, c1, c2, mn_blk);
          };
          if (!kAMN) {
            load(sa, &tmA, k0, m0, g, p.a_g);
          } else if (p.a_mn4) {
            load_mn4(sa, &tmA, k0, m0 / 64, g, p.a_g);
          } else {
#pragma unroll
            for (int i = 0; i < Cfg::BM / 64; ++i) load(sa + i * Cfg::MN_BOX_BYTES, &tmA, m0 + 64 * i, k0, g, p.a_g);
          }
          if (kEpi == EPI_SWIGLU) {
            // rows [c0, c0+BN/2) of w1_g, then the same rows of w3_g (one plane per CTA of a pair)
            if (kPair) {
              load(sb, &tmB, k0, n0, 2 * g + static_cast<int>(rank), G_OUTER);
            } else {
              load(sb, &tmB, k0, n0, 2 * g, G_OUTER);
              load(sb + (Cfg::BN / 2) * Cfg::ROW_BYTES, &tmB, k0, n0, 2 * g + 1, G_OUTER);
            }
          } else if (!kBMN) {
            load(sb, &tmB, k0, n0 + static_cast<int>(rank) * Cfg::B_ROWS, g, p.b_g);
          } else if (p.b_mn4) {
            load_mn4(sb, &tmB, k0, (n0 + static_cast<int>(rank) * Cfg::B_ROWS) / 64, g, p.b_g);
          } else {
#pragma unroll
            for (int i = 0; i < Cfg::B_ROWS / 64; ++i)
              load(sb + i * Cfg::MN_BOX_BYTES, &tmB, n0 + static_cast<int>(rank) * Cfg::B_ROWS + 64 * i, k0, g,
                   p.b_g);
          }
          armed |= 1u << stage;
          armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == Cfg::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // Every load issued must land before the CTA exits (the leader's full
      // barriers count the loads of both CTAs of a pair).
      for (int s = 0; s < Cfg::STAGES; ++s)
        if (leader && (armed & (1u << s))) {
          if (!mbar_try_wait(&full[s], (armed_parity >> s) & 1u)) {
            uint32_t dummy = 0;
            mbar_wait_slow(&full[s], (armed_parity >> s) & 1u, &dummy, SITE_DRAIN, kWaitLimitNs);
          }
        }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (pair leader)
    if (lane == 0 && leader) {
      int stage = 0;
      uint32_t phase = 0, tphase = 0;
      bool ok = true;
      int local = 0;
      for (int tile = unit; tile < total_tiles && ok; tile += num_units, ++local) {
        const int acc = local & (Cfg::NACC - 1);
        if (!mbar_wait(&tempty[acc], ((tphase >> acc) & 1u) ^ 1u, p.err, SITE_TEMPTY)) {
          ok = false;
          break;
        }
        tphase ^= 1u << acc;
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * Cfg::ACC_STRIDE);
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(&full[stage], phase, p.err, SITE_FULL)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t sa = smem_u32(stage_base + stage * Cfg::STAGE_BYTES);
          const uint32_t sb = sa + Cfg::A_BYTES;
#pragma unroll
          for (int j = 0; j < Cfg::K_STEPS; ++j) {
            // K-major: advance 32 bytes inside the swizzle row; 8-row groups 1024 B apart.
            // MN-major: advance 16 k-rows (2048 B); 8-k-row groups 1024 B apart,
            //           64-wide MN boxes MN_BOX_BYTES apart.
            const uint64_t ad = kAMN ? smem_desc_sw128(sa + j * 2048, Cfg::MN_BOX_BYTES, 1024)
                                     : smem_desc_sw128(sa + j * 32, 16, 1024);
            const uint64_t bd = kBMN ? smem_desc_sw128(sb + j * 2048, Cfg::MN_BOX_BYTES, 1024)
                                     : smem_desc_sw128(sb + j * 32, 16, 1024);
            const uint32_t accum = (kb > 0 || j > 0) ? 1u : 0u;
            if (kPair) {
              if (kFp8)
                umma_f8_pair(d_tmem, ad, bd, Cfg::IDESC, accum);
              else
                umma_bf16_pair(d_tmem, ad, bd, Cfg::IDESC, accum);
            } else {
              if (kFp8)
                umma_f8(d_tmem, ad, bd, Cfg::IDESC, accum);
              else
                umma_bf16(d_tmem, ad, bd, Cfg::IDESC, accum);
            }
          }
          if (kPair)
            tc_commit_pair_mc(&empty[stage], 0x3);
          else
            tc_commit(&empty[stage]);
          if (++stage == Cfg::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        if (kPair)
          tc_commit_pair_mc(&tfull[acc], 0x3);
        else
          tc_commit(&tfull[acc]);
      }
      // Every MMA this thread issued must complete before TMEM is released.
      if (kPair)
        tc_commit_pair_mc(drain, 0x1);
      else
        tc_commit(drain);
      if (!mbar_try_wait(drain, 0)) {
        uint32_t dummy = 0;
        mbar_wait_slow(drain, 0, &dummy, SITE_DRAIN, kWaitLimitNs);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int ew = warp - 2;  // staging-buffer owner index
    const int lg = warp & 3;  // TMEM lane quarter this warp may access
    uint8_t* stg = epi_base + ew * 2 * Cfg::EPI_BUF_BYTES;
    uint64_t* my_cbar = cbar + 2 * ew;
    const bool use_c = (kEpi == EPI_FP8) && (p.has_c != 0);
    uint32_t tphase = 0, cphase = 0, chunk_ctr = 0;
    uint32_t pending = 0, pending_parity = 0;  // async loads in flight, per staging buffer
    bool ok = true;
    const uint32_t lane_addr = tmem_base + (static_cast<uint32_t>(32 * lg) << 16);
    // Epilogue parameters of one tile held by this thread: its part of the
    // bias and of the e4m3 column scales, and its row's e4m3 scale.
    struct TileParams {
      uint4 b;
      float4 sc;
      float rs;
    };
    const int et = static_cast<int>(threadIdx.x) - 64;  // epilogue thread 0..127
    auto fetch_params = [&](int t, TileParams& q) {
      q.b = make_uint4(0u, 0u, 0u, 0u);
      q.sc = make_float4(0.f, 0.f, 0.f, 0.f);
      q.rs = 0.0f;
      if (t >= total_tiles) return;
      const int g = t / tiles_per_group;
      int mt, nt;
      tile_coords(p, t - g * tiles_per_group, mt, nt);
      const int n0 = nt * Cfg::BN_OUT;
      if (Cfg::HAS_BIAS && et < Cfg::BN_OUT / 8) {
        const int c = n0 + 8 * et;
        if (c < p.N) q.b = __ldg(reinterpret_cast<const uint4*>(p.bias + static_cast<int64_t>(g) * p.bias_g_stride + c));
      }
      if (Cfg::HAS_SCALES) {
        if (et < Cfg::BN_OUT / 4) {
          const int c = n0 + 4 * et;
          if (c < p.N)
            q.sc = __ldg(reinterpret_cast<const float4*>(p.col_scale + static_cast<int64_t>(g) * p.col_scale_g + c));
        }
        const int row = mt * Cfg::UMMA_M + static_cast<int>(rank) * Cfg::BM + 32 * lg + lane;
        if (row < p.M) q.rs = __ldg(p.row_scale + static_cast<int64_t>(g) * p.row_scale_g + row);
      }
    };
    auto publish_params = [&](const TileParams& q, int buf) {
      if (Cfg::HAS_BIAS && et < Cfg::BN_OUT / 8)
        reinterpret_cast<uint4*>(param_base + buf * Cfg::BIAS_BYTES)[et] = q.b;
      if (Cfg::HAS_SCALES && et < Cfg::BN_OUT / 4)
        reinterpret_cast<float4*>(param_base + 2 * Cfg::BIAS_BYTES + buf * Cfg::SCALE_BYTES)[et] = q.sc;
      __syncwarp();
      if (lane == 0) mbar_arrive(&pready[buf]);
    };
    TileParams prm;
    if (Cfg::HAS_BIAS || Cfg::HAS_SCALES) {
      fetch_params(unit, prm);
      publish_params(prm, 0);
    }
    int local = 0;
    for (int tile = unit; tile < total_tiles && ok; tile += num_units, ++local) {
      const int g = tile / tiles_per_group;
      const int rem = tile - g * tiles_per_group;
      int mt, nt;
      tile_coords(p, rem, mt, nt);
      const int m0 = mt * Cfg::UMMA_M + static_cast<int>(rank) * Cfg::BM;
      const int n0 = nt * Cfg::BN_OUT;
      const int acc = local & (Cfg::NACC - 1);
      const int row0 = m0 + 32 * lg;
      int nchunks = (p.N - n0 + 63) / 64;
      if (nchunks > Cfg::BN_OUT / 64) nchunks = Cfg::BN_OUT / 64;
      if (row0 >= p.M) nchunks = 0;

      // C (FP8 epilogue) of chunk j into staging buffer buf
      auto issue_load = [&](int j, int buf) {
        if (lane == 0) {
          bulk_wait_group_read<0>();
          mbar_arrive_expect_tx(&my_cbar[buf], Cfg::EPI_BUF_BYTES);
          tma_load_op(stg + buf * Cfg::EPI_BUF_BYTES, &tmC, &my_cbar[buf], n0 + 64 * j, row0, g, p.d_g);
        }
        pending |= 1u << buf;
        pending_parity = (pending_parity & ~(1u << buf)) | (((cphase >> buf) & 1u) << buf);
        __syncwarp();
      };
      if (use_c && nchunks > 0) issue_load(0, static_cast<int>(chunk_ctr & 1u));

      // This tile's bias and column scales sit in shared-memory buffer
      // `local & 1`, published by pready at the end of the previous tile (or
      // before the first); the next tile's are fetched into registers now and
      // published once this tile's chunks are done.  A buffer is rewritten
      // two tiles later, after every warp has passed the next tile's pready,
      // i.e. finished reading it.
      const int pb = local & 1;
      const uint4* sbias = reinterpret_cast<const uint4*>(param_base + pb * Cfg::BIAS_BYTES);
      const float4* sscale = reinterpret_cast<const float4*>(param_base + 2 * Cfg::BIAS_BYTES + pb * Cfg::SCALE_BYTES);
      const float rsc = prm.rs;
      TileParams nxt;
      if (Cfg::HAS_BIAS || Cfg::HAS_SCALES) {
        fetch_params(tile + num_units, nxt);
        if (!mbar_wait(&pready[pb], static_cast<uint32_t>(local >> 1) & 1u, p.err, SITE_PARAM)) {
          ok = false;
          break;
        }
      }

      if (!mbar_wait(&tfull[acc], (tphase >> acc) & 1u, p.err, SITE_TFULL)) {
        ok = false;
        break;
      }
      tphase ^= 1u << acc;
      tc_fence_after_sync();

      // The accumulator goes back to the MMA warp as soon as this warp's last
      // TMEM load of the tile has completed (the rest of the tile's epilogue
      // works from registers and shared memory).
      bool released = false;
      auto release_acc = [&]() {
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) {
          if (kPair)
            mbar_arrive_cluster(mapa_shared(smem_u32(&tempty[acc]), 0));
          else
            mbar_arrive(&tempty[acc]);
        }
        released = true;
      };
      const bool last_ld_in_loop = !Cfg::HALF_CHUNK || !(row0 < p.M && n0 + Cfg::BN_OUT - 32 < p.N);

      MeanM2 st_u{0.0f, 0.0f, 0.0f}, st_g{0.0f, 0.0f, 0.0f};
      for (int j = 0; j < nchunks; ++j) {
        const int buf = static_cast<int>((chunk_ctr + j) & 1u);
        if (use_c && j + 1 < nchunks) issue_load(j + 1, buf ^ 1);

        float v[64];
        if (kEpi == EPI_SWIGLU) {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            uint32_t ra[32], rb[32];
            const uint32_t col = static_cast<uint32_t>(acc * Cfg::ACC_STRIDE + 64 * j + 32 * h);
            tmem_ld_32x32b_x32(lane_addr + col, ra);
            tmem_ld_32x32b_x32(lane_addr + col + Cfg::BN / 2, rb);
            tmem_ld_wait();
            tmem_regs_after_wait(ra);
            tmem_regs_after_wait(rb);
            if (h == 1 && j + 1 == nchunks && last_ld_in_loop) release_acc();
#pragma unroll
            for (int i = 0; i < 32; ++i)
              v[32 * h + i] = silu_f(__uint_as_float(ra[i])) * __uint_as_float(rb[i]);
          }
        } else {
          uint32_t r0[32], r1[32];
          const uint32_t col = static_cast<uint32_t>(acc * Cfg::ACC_STRIDE + 64 * j);
          tmem_ld_32x32b_x32(lane_addr + col, r0);
          tmem_ld_32x32b_x32(lane_addr + col + 32, r1);
          tmem_ld_wait();
          tmem_regs_after_wait(r0);
          tmem_regs_after_wait(r1);
          if (j + 1 == nchunks && last_ld_in_loop) release_acc();
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            v[i] = __uint_as_float(r0[i]);
            v[32 + i] = __uint_as_float(r1[i]);
          }
        }
        if (num_kb == 0) {
#pragma unroll
          for (int i = 0; i < 64; ++i) v[i] = 0.0f;
        }

        uint8_t* sbuf = stg + buf * Cfg::EPI_BUF_BYTES;
        if (use_c) {
          if (!mbar_wait(&my_cbar[buf], (cphase >> buf) & 1u, p.err, SITE_CLOAD)) {
            ok = false;
            break;
          }
          cphase ^= 1u << buf;
          pending &= ~(1u << buf);
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const uint4 cv =
                *reinterpret_cast<const uint4*>(sbuf + lane * 128 + ((q ^ (lane & 7)) << 4));
            const uint32_t cw[4] = {cv.x, cv.y, cv.z, cv.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 c2 = unpack_bf16x2(cw[e]);
              v[8 * q + 2 * e] = p.alpha * v[8 * q + 2 * e] + p.beta * c2.x;
              v[8 * q + 2 * e + 1] = p.alpha * v[8 * q + 2 * e + 1] + p.beta * c2.y;
            }
          }
        } else {
          if (kEpi == EPI_FP8) {
#pragma unroll
            for (int i = 0; i < 64; ++i) v[i] *= p.alpha;
          }
          if (Cfg::HAS_SCALES) {
            // per-row scale of the e4m3 A rows, per-column scale of the e4m3 B rows
            const float2 rs2 = make_float2(rsc, rsc);
#pragma unroll
            for (int q = 0; q < 16; ++q) {
              {
                const float4 c4 = sscale[16 * j + q];
                const float2 a = mul2(mul2(make_float2(v[4 * q], v[4 * q + 1]), rs2), make_float2(c4.x, c4.y));
                const float2 b = mul2(mul2(make_float2(v[4 * q + 2], v[4 * q + 3]), rs2), make_float2(c4.z, c4.w));
                v[4 * q] = a.x;
                v[4 * q + 1] = a.y;
                v[4 * q + 2] = b.x;
                v[4 * q + 3] = b.y;
              }
            }
          }
          if (Cfg::HAS_BIAS) {
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              {
                const uint4 bv = sbias[8 * j + q];
                const uint32_t bw[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  const float2 sum = add2(make_float2(v[8 * q + 2 * e], v[8 * q + 2 * e + 1]), unpack_bf16x2(bw[e]));
                  v[8 * q + 2 * e] = sum.x;
                  v[8 * q + 2 * e + 1] = sum.y;
                }
              }
            }
          }
          // the store that last read this buffer (two chunks ago) must be done
          if (lane == 0) bulk_wait_group_read<1>();
          __syncwarp();
        }
        if (kEpi == EPI_BIAS_LNSTATS) {
          // statistics of this row's valid columns of the chunk, split at ln_H
          const int c0 = n0 + 64 * j;
          const int cend = min(c0 + 64, p.N);
          const int nvalid = cend - c0;
          const int usplit = min(max(p.ln_H - c0, 0), nvalid);  // columns [0, usplit) are U
          float mean, m2;
          if (nvalid == 64 && (usplit == 0 || usplit == 64)) {
            // two passes over the chunk, each with four independent packed
            // accumulators (short dependency chains)
            float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                             make_float2(0.f, 0.f)};
#pragma unroll
            for (int i = 0; i < 32; ++i) acc[i & 3] = add2(acc[i & 3], make_float2(v[2 * i], v[2 * i + 1]));
            const float2 s01 = add2(acc[0], acc[1]), s23 = add2(acc[2], acc[3]);
            const float2 s4 = add2(s01, s23);
            mean = (s4.x + s4.y) * (1.0f / 64.0f);
            const float2 nm = make_float2(-mean, -mean);
            float2 sq[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                            make_float2(0.f, 0.f)};
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const float2 d = add2(make_float2(v[2 * i], v[2 * i + 1]), nm);
              sq[i & 3] = fma2(d, d, sq[i & 3]);
            }
            const float2 q01 = add2(sq[0], sq[1]), q23 = add2(sq[2], sq[3]);
            const float2 q4 = add2(q01, q23);
            const float q = q4.x + q4.y;
            (usplit == 64 ? st_u : st_g).merge(64.0f, mean, q);
          } else {
            if (usplit > 0) {
              chunk_mean_m2<64>(v, 0, usplit, mean, m2);
              st_u.merge(static_cast<float>(usplit), mean, m2);
            }
            if (nvalid > usplit) {
              chunk_mean_m2<64>(v, usplit, nvalid, mean, m2);
              st_g.merge(static_cast<float>(nvalid - usplit), mean, m2);
            }
          }
        }
        uint32_t packed[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) packed[i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          *reinterpret_cast<uint4*>(sbuf + lane * 128 + ((q ^ (lane & 7)) << 4)) =
              make_uint4(packed[4 * q], packed[4 * q + 1], packed[4 * q + 2], packed[4 * q + 3]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_op(&tmD, sbuf, n0 + 64 * j, row0, g, p.d_g);
          bulk_commit_group();
        }
      }
      if (!ok) break;
      if (Cfg::HALF_CHUNK) {
        // Columns [BN_OUT - 32, BN_OUT) of the tile: one 32-column TMEM load,
        // then plain 16-byte global loads/stores per row (a 64-wide TMA box
        // would reach into the next tile's columns).
        const int c0 = n0 + Cfg::BN_OUT - 32;
        if (row0 < p.M && c0 < p.N) {
          uint32_t r0[32];
          tmem_ld_32x32b_x32(lane_addr + static_cast<uint32_t>(acc * Cfg::ACC_STRIDE + Cfg::BN_OUT - 32), r0);
          tmem_ld_wait();
          tmem_regs_after_wait(r0);
          release_acc();
          const int row = row0 + lane;
          if (row < p.M) {
            const int64_t off = (static_cast<int64_t>(g) * p.M + row) * p.N + c0;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              if (c0 + 8 * q < p.N) {
                float v[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) v[i] = num_kb == 0 ? 0.0f : p.alpha * __uint_as_float(r0[8 * q + i]);
                if (use_c) {
                  const uint4 cv = __ldg(reinterpret_cast<const uint4*>(p.c_ptr + off + 8 * q));
                  const uint32_t cw[4] = {cv.x, cv.y, cv.z, cv.w};
#pragma unroll
                  for (int e = 0; e < 4; ++e) {
                    const float2 c2 = unpack_bf16x2(cw[e]);
                    v[2 * e] = fmaf(p.beta, c2.x, v[2 * e]);
                    v[2 * e + 1] = fmaf(p.beta, c2.y, v[2 * e + 1]);
                  }
                }
                *reinterpret_cast<uint4*>(p.d_ptr + off + 8 * q) =
                    make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                               pack_bf16x2(v[6], v[7]));
              }
            }
          }
        }
      }
      if (kEpi == EPI_BIAS_LNSTATS && nchunks > 0 && row0 + lane < p.M) {
        p.ln_part[(static_cast<int64_t>(g) * p.tiles_n + nt) * p.M + row0 + lane] =
            make_float4(st_u.mean, st_u.m2, st_g.mean, st_g.m2);
      }
      chunk_ctr += static_cast<uint32_t>(nchunks);
      if (Cfg::HAS_BIAS || Cfg::HAS_SCALES) {
        publish_params(nxt, pb ^ 1);
        prm = nxt;
      }
      if (!released) release_acc();
    }
    // Outstanding copies of this warp must finish before the CTA exits.
    if (lane == 0) bulk_wait_group<0>();
    for (int b2 = 0; b2 < 2; ++b2) {
      if ((pending >> b2) & 1u) {
        const uint32_t par = (pending_parity >> b2) & 1u;
        if (!mbar_try_wait(&my_cbar[b2], par)) {
          uint32_t dummy = 0;
          mbar_wait_slow(&my_cbar[b2], par, &dummy, SITE_DRAIN, kWaitLimitNs);
        }
      }
    }
    __syncwarp();
  }

  // This CTA's work is issued: the next kernel may start launching.
  griddep_launch_dependents();
  tc_fence_before_sync();
  if (kPair)
    cluster_sync_all();
  else
    __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    if (kPair)
      tmem_dealloc_pair(tmem_base, Cfg::TMEM_COLS);
    else
      tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
  }
}

}  // namespace dg
