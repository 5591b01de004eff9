// The A2A FFN's second GEMM with the normalise-and-gate folded into the
// production of its A operand (sm_103a, tcgen05, CTA pairs).
//
// Source of the arithmetic: the A2A-FFN project statement (problems/p04),
// "Computation and communication example": with (U, G) the two H-wide halves
// of Z and LN(z) = (z - mean z) / sqrt(var z + eps) * gamma + beta,
//   Ylocal = (LN_x(U) * silu(LN_gate(G))) @ wout + bout.
// The per-row statistics come from GEMM1's epilogue (finalised beforehand);
// what is folded here is the map Hl = LN_x(U) * silu(LN_g(G)) itself.
//
// Per CTA pair and work unit: a 256-row block of one problem times a column
// pass of up to 512 output columns (two 256-column UMMAs per K step into one
// 512-column TMEM accumulator).  Five column tiles of 256 would recompute
// every Hl element five times; passes of 512 recompute it ceil(N / 512)
// times, and the passes of one row block run on neighbouring pairs at the
// same time, so Z is read from HBM about once.
//
// Warp roles (512 threads):
//   warp 0      Z producer: per K block (64 columns, or 32 when built with
//               DG_GATED_BK=32), this CTA's 128 rows of the U and G columns
//               of Z (two boxes swizzled at the K block's row width, 128 or
//               64 bytes, the U box landing in the stage's A tile), on a
//               per-CTA barrier
//   warp 14     B producer: the CTA's half of the block's B (wout, MN-major)
//               columns, on the pair leader's barrier
//   warp 15     parameter producer: the block's LayerNorm weights and biases
//               (four bulk copies) on the per-CTA barrier of the Z boxes
//               (three producers, because one thread issuing all of a
//               stage's copies took longer than the stage's MMAs)
//   warp 1      MMA issuer (pair leader, one lane)
//   warps 2-5   epilogue: TMEM -> + bout -> bf16 -> TMA store at the combine offsets
//   warps 6-13  transform: for four rows each (two with 32-wide K blocks), read a U and a G vector from
//               shared memory, compute Hl in fp32, and write it as bf16 over
//               the U vector (the same swizzled position, which is where the
//               MMA reads A).  With a non-NULL Hl pointer the units of column
//               pass 0 also store Hl (the backward's dwout needs it).
// A stage is full when the B copies of both CTAs have landed and the eight
// transform warps of both CTAs have arrived on the leader's barrier (after a
// generic-to-async proxy fence; the arrive is a CTA-scope release, which a
// cluster-scope one would stall for up to a microsecond per stage).  Each stage therefore passes through copy,
// transform and MMA in turn; three stages of 64 K values (six of 32) keep
// enough of them in flight for that chain.  The arithmetic is that of the separate
// normalise-and-gate pass (that pass folds the 1/2 of h = s/2 into the gate
// norm's affine instead of multiplying by 0.5, which rounds to the same
// value), so the A operand equals that pass's Hl bit for bit.
#include "dg_internal.h"

#ifndef DG_GATED_BK
#define DG_GATED_BK 64
#endif

namespace dg {

namespace {

struct GatedCfg {
  static constexpr int CTAS = 2;
  static constexpr int BM = 128;                 // A rows per CTA (TMEM lanes)
  static constexpr int UMMA_M = 256;
  static constexpr int SUB_N = 256;              // columns per UMMA
  static constexpr int NSUB = 2;                 // UMMAs per K step
  static constexpr int BN_OUT = SUB_N * NSUB;    // columns per pass
  static constexpr int B_ROWS = SUB_N / CTAS;    // B columns each CTA stages per UMMA
  static constexpr int BK = DG_GATED_BK;         // K elements per stage: one 64- or 128-byte swizzle row
  static constexpr int ROW_BYTES = BK * 2;       // A and G rows (bf16), also their swizzle width
  static constexpr int K_STEPS = BK / 16;        // UMMA K = 16
  static constexpr int VECS = BK / 8;            // 16-byte vectors per row
  static constexpr int A_BYTES = BM * BK * 2;    // U on arrival, Hl (the A operand) after the transform
  static constexpr int G_BYTES = BM * BK * 2;    // G
  static constexpr int MN_BOX_BYTES = 64 * BK * 2;       // one 64-column MN-major box of B
  static constexpr int SUB_B_BYTES = B_ROWS * BK * 2;    // 8 KB
  static constexpr int B_BYTES = NSUB * SUB_B_BYTES;
  static constexpr int STAGE_BYTES = A_BYTES + G_BYTES + B_BYTES;
  static constexpr int STAGES = BK == 32 ? 6 : 3;
  static constexpr int PRM_BYTES = 4 * BK * 2;   // the K block's LayerNorm weights and biases, bf16
  static constexpr int EPI_WARPS = 4;
  static constexpr int XF_WARPS = 8;
  static constexpr int XF_ROWS_PER_WARP = BM / XF_WARPS;
  static constexpr int XF_ROWS = BM * VECS / (XF_WARPS * 32);   // rows per transform thread
  static constexpr int EPI_BUF_BYTES = 32 * 128; // 32 rows x 64 bf16, one per epilogue warp
  static constexpr int EPI_BYTES = EPI_WARPS * EPI_BUF_BYTES;
  static constexpr int NUM_THREADS = 64 + 32 * (EPI_WARPS + XF_WARPS) + 64;  // + the B and parameter producers
  static constexpr int B_WARP = 2 + EPI_WARPS + XF_WARPS;
  static constexpr int PRM_WARP = B_WARP + 1;
  static constexpr uint32_t TMEM_COLS = BN_OUT;
  static constexpr int BIAS_BYTES = BN_OUT * 2;
  static constexpr int PARAM_BYTES = 2 * BIAS_BYTES;
  static constexpr int NUM_BARS = 3 * STAGES + 3 + 2;
  static constexpr int BAR_BYTES = 256;
  static constexpr int SMEM_BYTES =
      1024 + STAGES * STAGE_BYTES + STAGES * PRM_BYTES + EPI_BYTES + PARAM_BYTES + BAR_BYTES;
  static constexpr uint32_t IDESC = umma_idesc(1u, false, true, SUB_N, UMMA_M);
  static_assert(NUM_BARS * 8 + 4 <= BAR_BYTES, "barrier area");
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
  static_assert(XF_ROWS * XF_WARPS * (32 / VECS) == BM && XF_ROWS * (32 / VECS) == XF_ROWS_PER_WARP,
                "transform warps cover the A rows");
  static_assert(BK == 32 || BK == 64, "K block of 32 or 64");
  static_assert(STAGE_BYTES % 1024 == 0 && EPI_BUF_BYTES % 1024 == 0, "swizzled regions stay 1024-byte aligned");
};

// Arrive once on an mbarrier of the peer CTA (shared::cluster address) with
// the default release at CTA scope, after a proxy fence of this thread's
// shared-memory writes: the peer's MMA then reads them.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// Shared-memory descriptor of a 64-byte-swizzled K-major tile (8-row groups
// `sbo` bytes apart); the layout code of that swizzle is 4.
__device__ __forceinline__ uint64_t smem_desc_sw64(uint32_t start, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((start >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1u) << 46;
  d |= static_cast<uint64_t>(4u) << 61;
  return d;
}

// Bounded wait for a long-pending phase (the epilogue waits a whole mainloop
// for its accumulator): polls with short sleeps in between, so the waiting
// warps do not take issue slots from the transform warps on the same SM.
__device__ __noinline__ bool mbar_wait_sleepy(uint64_t* bar, uint32_t parity, uint32_t* err, uint32_t site) {
  const uint64_t t0 = global_timer_ns();
  uint32_t n = 0;
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    __nanosleep(256);
    if ((++n & 63u) == 0u) {
      if (ld_volatile_u32(err) != 0u) return false;
      if (global_timer_ns() - t0 > kWaitLimitNs) {
        atomicCAS(err, 0u, kErrTimeout | (site & 0xffu));
        return false;
      }
    }
  }
}

__global__ void __launch_bounds__(GatedCfg::NUM_THREADS, 1)
    gemm_gated_kernel(const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmD,
                      const __grid_constant__ CUtensorMap tmZ, const GemmParams p, const GateSrc q) {
  using Cfg = GatedCfg;
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint32_t s_abort;

  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  // The operand tiles and the epilogue's staging buffers come first: TMA and
  // the MMA compute the 128-byte swizzle from address bits, so those regions
  // stay 1024-byte aligned; the small parameter ring follows them.
  uint8_t* stage_base = smem;
  uint8_t* epi_base = smem + Cfg::STAGES * Cfg::STAGE_BYTES;
  uint8_t* prm_base = epi_base + Cfg::EPI_BYTES;  // [STAGES][4][BK] bf16
  uint8_t* param_base = prm_base + Cfg::STAGES * Cfg::PRM_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(param_base + Cfg::PARAM_BYTES);
  uint64_t* full = bars;                        // leader: B landed + transform warps of both CTAs
  uint64_t* empty = bars + Cfg::STAGES;         // both CTAs: the MMAs of the stage are done
  uint64_t* zfull = bars + 2 * Cfg::STAGES;     // per CTA: its U and G boxes landed
  uint64_t* tfull = bars + 3 * Cfg::STAGES;
  uint64_t* tempty = tfull + 1;
  uint64_t* drain = tempty + 1;
  uint64_t* pready = drain + 1;  // [2]
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(pready + 2);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0u;

  if (warp == 0 && lane == 0) {
    for (int s = 0; s < Cfg::STAGES; ++s) {
      mbar_init(&full[s], 1 + Cfg::CTAS * Cfg::XF_WARPS);
      mbar_init(&empty[s], 1);
      mbar_init(&zfull[s], 1);
    }
    mbar_init(tfull, 1);
    mbar_init(tempty, Cfg::EPI_WARPS * Cfg::CTAS);
    mbar_init(drain, 1);
    mbar_init(&pready[0], Cfg::EPI_WARPS);
    mbar_init(&pready[1], Cfg::EPI_WARPS);
    fence_mbar_init();
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmD);
    tma_prefetch_desc(&tmZ);
  }
  cluster_sync_all();
  griddep_wait();  // Z, the statistics and the error word come from the preceding kernels

  if (threadIdx.x == 0 && leader) {
    const uint32_t v = ld_volatile_u32(p.err);
    st_cluster_u32(mapa_shared(smem_u32(&s_abort), 0), v);
    st_cluster_u32(mapa_shared(smem_u32(&s_abort), 1), v);
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_holder, Cfg::TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before_sync();
  cluster_sync_all();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_holder;
  const bool aborted = s_abort != 0u;

  const int tiles_per_group = p.tiles_m * p.tiles_n;
  const int total_tiles = p.G * tiles_per_group;
  const int num_kb = (p.K + Cfg::BK - 1) / Cfg::BK;
  const int unit = static_cast<int>(blockIdx.x) / Cfg::CTAS;
  const int num_units = static_cast<int>(gridDim.x) / Cfg::CTAS;
  auto nsub_of = [&](int n0) { return p.N - n0 > Cfg::SUB_N ? 2 : 1; };

  if (aborted) {
    // straight to the teardown
  } else if (warp == 0 || warp == Cfg::B_WARP || warp == Cfg::PRM_WARP) {
    // ------------------------------------------------------------ producers
    // warp 0: this CTA's U and G boxes of Z; B_WARP: its half of the B columns;
    // PRM_WARP: the K block's LayerNorm parameters.  Each walks the same ring.
    if (lane == 0) {
      const int role = warp == 0 ? 0 : (warp == Cfg::B_WARP ? 1 : 2);
      int stage = 0;
      uint32_t phase = 0, armed = 0, armed_parity = 0;
      bool ok = true;
      for (int tile = unit; tile < total_tiles && ok; tile += num_units) {
        const int g = tile / tiles_per_group;
        int mt, nt;
        tile_coords(p, tile - g * tiles_per_group, mt, nt);
        const int m0 = mt * Cfg::UMMA_M + static_cast<int>(rank) * Cfg::BM;
        const int n0 = nt * Cfg::BN_OUT;
        const int nsub = nsub_of(n0);
        const int64_t prm0 = static_cast<int64_t>(g / q.L) * q.H;
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, p.err, SITE_EMPTY)) {
            ok = false;
            break;
          }
          uint8_t* sa = stage_base + stage * Cfg::STAGE_BYTES;
          const int k0 = kb * Cfg::BK;
          // the K block's parameter columns below H (none past it)
          const int pcols = k0 < q.H ? min(Cfg::BK, q.H - k0) : 0;
          const uint32_t pbytes = static_cast<uint32_t>(pcols) * 2u;
          if (role == 0) {
            // U into the A tile and G, plus the parameters' bytes, on this CTA's barrier
            mbar_arrive_expect_tx(&zfull[stage], Cfg::A_BYTES + Cfg::G_BYTES + 4u * pbytes);
            tma_load_3d(sa, &tmZ, &zfull[stage], k0, m0, g);
            tma_load_3d(sa + Cfg::A_BYTES, &tmZ, &zfull[stage], q.H + k0, m0, g);
          } else if (role == 1) {
            // this CTA's half of the B columns, completing on the leader's barrier
            uint8_t* sb = sa + Cfg::A_BYTES + Cfg::G_BYTES;
            if (leader) mbar_arrive_expect_tx(&full[stage], nsub * Cfg::SUB_B_BYTES * Cfg::CTAS);
            const uint32_t bar_c = mapa_shared(smem_u32(&full[stage]), 0);
            for (int j = 0; j < nsub; ++j) {
              const int nb = n0 + Cfg::SUB_N * j + static_cast<int>(rank) * Cfg::B_ROWS;
              if (p.b_mn4) {
                tma_load_4d_pair(sb + j * Cfg::SUB_B_BYTES, &tmB, bar_c, 0, k0, g, nb / 64);
              } else {
                tma_load_3d_pair(sb + j * Cfg::SUB_B_BYTES, &tmB, bar_c, nb, k0, g);
                tma_load_3d_pair(sb + j * Cfg::SUB_B_BYTES + Cfg::MN_BOX_BYTES, &tmB, bar_c, nb + 64, k0, g);
              }
            }
          } else if (pcols > 0) {
            uint8_t* sp = prm_base + stage * Cfg::PRM_BYTES;
            const int64_t po = prm0 + k0;
            bulk_load(sp + 0 * Cfg::BK * 2, q.gx + po, pbytes, &zfull[stage]);
            bulk_load(sp + 1 * Cfg::BK * 2, q.bx + po, pbytes, &zfull[stage]);
            bulk_load(sp + 2 * Cfg::BK * 2, q.gg + po, pbytes, &zfull[stage]);
            bulk_load(sp + 3 * Cfg::BK * 2, q.bg + po, pbytes, &zfull[stage]);
          }
          armed |= 1u << stage;
          armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == Cfg::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // Every copy issued must land before the CTA exits: the Z producer waits
      // for each armed phase of its barrier (which also counts the parameter
      // copies), the leader's B producer for each armed phase of the pair's.
      for (int s = 0; s < Cfg::STAGES; ++s)
        if (armed & (1u << s)) {
          const uint32_t par = (armed_parity >> s) & 1u;
          uint32_t dummy = 0;
          if (role == 0 && !mbar_try_wait(&zfull[s], par))
            mbar_wait_slow(&zfull[s], par, &dummy, SITE_DRAIN, kWaitLimitNs);
          if (role == 1 && leader && !mbar_try_wait(&full[s], par))
            mbar_wait_slow(&full[s], par, &dummy, SITE_DRAIN, kWaitLimitNs);
        }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && leader) {
      int stage = 0;
      uint32_t phase = 0, tphase = 0;
      bool ok = true;
      for (int tile = unit; tile < total_tiles && ok; tile += num_units) {
        const int g = tile / tiles_per_group;
        int mt, nt;
        tile_coords(p, tile - g * tiles_per_group, mt, nt);
        const int nsub = nsub_of(nt * Cfg::BN_OUT);
        if (!mbar_wait(tempty, tphase ^ 1u, p.err, SITE_TEMPTY)) {
          ok = false;
          break;
        }
        tphase ^= 1u;
        tc_fence_after_sync();
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(&full[stage], phase, p.err, SITE_FULL)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t sa = smem_u32(stage_base + stage * Cfg::STAGE_BYTES);
          const uint32_t sb = sa + Cfg::A_BYTES + Cfg::G_BYTES;
#pragma unroll
          for (int j = 0; j < Cfg::K_STEPS; ++j) {
            // K-major A, 64-byte rows: the 16-element K step advances 32 bytes
            // inside the swizzle row; 8-row groups are 512 bytes apart
            const uint64_t ad = Cfg::BK == 32 ? smem_desc_sw64(sa + j * 32, 16, 512) : smem_desc_sw128(sa + j * 32, 16, 1024);
            const uint32_t accum = (kb > 0 || j > 0) ? 1u : 0u;
            for (int s = 0; s < nsub; ++s) {
              const uint64_t bd = smem_desc_sw128(sb + s * Cfg::SUB_B_BYTES + j * 2048, Cfg::MN_BOX_BYTES, 1024);
              umma_bf16_pair(tmem_base + static_cast<uint32_t>(s * Cfg::SUB_N), ad, bd, Cfg::IDESC, accum);
            }
          }
          tc_commit_pair_mc(&empty[stage], 0x3);
          if (++stage == Cfg::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit_pair_mc(tfull, 0x3);
      }
      tc_commit_pair_mc(drain, 0x1);
      if (!mbar_try_wait(drain, 0)) {
        uint32_t dummy = 0;
        mbar_wait_slow(drain, 0, &dummy, SITE_DRAIN, kWaitLimitNs);
      }
    }
  } else if (warp < 2 + Cfg::EPI_WARPS) {
    // ------------------------------------------------------------ epilogue
    const int ew = warp - 2;
    const int lg = warp & 3;  // TMEM lane quarter this warp may access
    uint8_t* stg = epi_base + ew * Cfg::EPI_BUF_BYTES;
    uint32_t tphase = 0;
    bool ok = true;
    const uint32_t lane_addr = tmem_base + (static_cast<uint32_t>(32 * lg) << 16);
    const int et = static_cast<int>(threadIdx.x) - 64;  // 0..127
    auto fetch_bias = [&](int t) {
      uint4 b = make_uint4(0u, 0u, 0u, 0u);
      if (t < total_tiles && et < Cfg::BN_OUT / 8) {
        const int g = t / tiles_per_group;
        int mt, nt;
        tile_coords(p, t - g * tiles_per_group, mt, nt);
        const int c = nt * Cfg::BN_OUT + 8 * et;
        if (c < p.N) b = __ldg(reinterpret_cast<const uint4*>(p.bias + static_cast<int64_t>(g) * p.bias_g_stride + c));
      }
      return b;
    };
    auto publish_bias = [&](uint4 b, int buf) {
      if (et < Cfg::BN_OUT / 8) reinterpret_cast<uint4*>(param_base + buf * Cfg::BIAS_BYTES)[et] = b;
      __syncwarp();
      if (lane == 0) mbar_arrive(&pready[buf]);
    };
    publish_bias(fetch_bias(unit), 0);
    int local = 0;
    for (int tile = unit; tile < total_tiles && ok; tile += num_units, ++local) {
      const int g = tile / tiles_per_group;
      int mt, nt;
      tile_coords(p, tile - g * tiles_per_group, mt, nt);
      const int m0 = mt * Cfg::UMMA_M + static_cast<int>(rank) * Cfg::BM;
      const int n0 = nt * Cfg::BN_OUT;
      const int row0 = m0 + 32 * lg;
      int nchunks = (p.N - n0 + 63) / 64;
      if (nchunks > Cfg::BN_OUT / 64) nchunks = Cfg::BN_OUT / 64;
      if (row0 >= p.M) nchunks = 0;
      const int pb = local & 1;
      const uint4* sbias = reinterpret_cast<const uint4*>(param_base + pb * Cfg::BIAS_BYTES);
      const uint4 nxt = fetch_bias(tile + num_units);
      if (!__all_sync(0xffffffffu, mbar_wait(&pready[pb], static_cast<uint32_t>(local >> 1) & 1u, p.err,
                                              SITE_PARAM))) {
        ok = false;
        break;
      }
      if (!__all_sync(0xffffffffu, mbar_wait_sleepy(tfull, tphase, p.err, SITE_TFULL))) {
        ok = false;
        break;
      }
      tphase ^= 1u;
      tc_fence_after_sync();
      bool released = false;
      auto release_acc = [&]() {
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(tempty), 0));
        released = true;
      };
      for (int j = 0; j < nchunks; ++j) {
        // the previous chunk's store must have read the staging buffer
        if (lane == 0) bulk_wait_group_read<0>();
        __syncwarp();
        // two 32-column halves (one TMEM load each, to keep few registers live)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t r[32];
          tmem_ld_32x32b_x32(lane_addr + static_cast<uint32_t>(64 * j + 32 * h), r);
          tmem_ld_wait();
          tmem_regs_after_wait(r);
          if (h == 1 && j + 1 == nchunks) release_acc();
          uint32_t packed[16];
#pragma unroll
          for (int qq = 0; qq < 4; ++qq) {
            const uint4 bv = sbias[8 * j + 4 * h + qq];
            const uint32_t bw[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              float2 a = make_float2(__uint_as_float(r[8 * qq + 2 * e]), __uint_as_float(r[8 * qq + 2 * e + 1]));
              if (num_kb == 0) a = make_float2(0.0f, 0.0f);
              const float2 sum = add2(a, unpack_bf16x2(bw[e]));
              packed[4 * qq + e] = pack_bf16x2(sum.x, sum.y);
            }
          }
#pragma unroll
          for (int qq = 0; qq < 4; ++qq) {
            const int c = 4 * h + qq;  // 16-byte vector of the 128-byte staging row
            *reinterpret_cast<uint4*>(stg + lane * 128 + ((c ^ (lane & 7)) << 4)) =
                make_uint4(packed[4 * qq], packed[4 * qq + 1], packed[4 * qq + 2], packed[4 * qq + 3]);
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_op(&tmD, stg, n0 + 64 * j, row0, g, p.d_g);
          bulk_commit_group();
        }
      }
      publish_bias(nxt, pb ^ 1);
      if (!released) release_acc();
    }
    if (lane == 0) bulk_wait_group<0>();
    __syncwarp();
  } else {
    // ------------------------------------------------------------ transform (normalise and gate)
    const int xw = warp - 2 - Cfg::EPI_WARPS;  // 0..XF_WARPS-1
    const int q4 = lane & (Cfg::VECS - 1);     // 8-column vector of the K block
    const int rs = lane / Cfg::VECS;           // row within the warp's group of 32 / VECS
    const float2 half2 = make_float2(0.5f, 0.5f);
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int tile = unit; tile < total_tiles && ok; tile += num_units) {
      const int g = tile / tiles_per_group;
      int mt, nt;
      tile_coords(p, tile - g * tiles_per_group, mt, nt);
      const int m0 = mt * Cfg::UMMA_M + static_cast<int>(rank) * Cfg::BM;
      // this thread's rows: r_i = XF_ROWS_PER_WARP*xw + (32 / VECS)*i + rs
      constexpr int RSTEP = 32 / Cfg::VECS;
      bool valid[Cfg::XF_ROWS];
      float2 rsu[Cfg::XF_ROWS], cu[Cfg::XF_ROWS], rsg[Cfg::XF_ROWS], cgs[Cfg::XF_ROWS];
#pragma unroll
      for (int i = 0; i < Cfg::XF_ROWS; ++i) {
        const int row = m0 + Cfg::XF_ROWS_PER_WARP * xw + RSTEP * i + rs;
        valid[i] = row < p.M;
        const float4 sr = valid[i] ? q.stats[static_cast<int64_t>(g) * p.M + row] : make_float4(0.f, 1.f, 0.f, 1.f);
        rsu[i] = make_float2(sr.y, sr.y);
        cu[i] = make_float2(-sr.x * sr.y, -sr.x * sr.y);
        rsg[i] = make_float2(sr.w, sr.w);
        cgs[i] = make_float2(-sr.z * sr.w, -sr.z * sr.w);
      }
      __nv_bfloat16* hl_row0 =
          (q.Hl != nullptr && nt == 0)
              ? q.Hl + (static_cast<int64_t>(g) * p.M + m0 + Cfg::XF_ROWS_PER_WARP * xw + rs) * static_cast<int64_t>(q.H)
              : nullptr;
      for (int kb = 0; kb < num_kb; ++kb) {
        const int k = kb * Cfg::BK + 8 * q4;
        const bool kv = k < q.H;
        // every lane waits (each must observe the copies' completion); the warp
        // leaves together if any lane's wait gave up
        if (!__all_sync(0xffffffffu, mbar_wait(&zfull[stage], phase, p.err, SITE_CLOAD))) {
          ok = false;
          break;
        }
        // this vector's LayerNorm weights and biases, from the stage's parameter slot
        const uint8_t* sp = prm_base + stage * Cfg::PRM_BYTES + q4 * 16;
        float2 wx[4], cx[4], wg[4], cg[4];
        {
          const uint4 a0 = *reinterpret_cast<const uint4*>(sp + 0 * Cfg::BK * 2);
          const uint4 a1 = *reinterpret_cast<const uint4*>(sp + 1 * Cfg::BK * 2);
          const uint4 a2 = *reinterpret_cast<const uint4*>(sp + 2 * Cfg::BK * 2);
          const uint4 a3 = *reinterpret_cast<const uint4*>(sp + 3 * Cfg::BK * 2);
          const uint32_t w0[4] = {a0.x, a0.y, a0.z, a0.w}, w1[4] = {a1.x, a1.y, a1.z, a1.w};
          const uint32_t w2[4] = {a2.x, a2.y, a2.z, a2.w}, w3[4] = {a3.x, a3.y, a3.z, a3.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            wx[e] = unpack_bf16x2(w0[e]);
            cx[e] = unpack_bf16x2(w1[e]);
            wg[e] = unpack_bf16x2(w2[e]);
            cg[e] = unpack_bf16x2(w3[e]);
          }
        }
        uint8_t* sa = stage_base + stage * Cfg::STAGE_BYTES;
        const uint8_t* sg = sa + Cfg::A_BYTES;
        uint4 outv[Cfg::XF_ROWS];
#pragma unroll
        for (int i = 0; i < Cfg::XF_ROWS; ++i) {
          // the 16-byte vector q of row r sits at vector q ^ ((r / 2) % 4) (64-byte
          // swizzle) or q ^ (r % 8) (128-byte swizzle)
          const int r = Cfg::XF_ROWS_PER_WARP * xw + RSTEP * i + rs;
          const int sw = Cfg::BK == 32 ? ((r >> 1) & 3) : (r & 7);
          const int off = r * Cfg::ROW_BYTES + ((q4 ^ sw) << 4);
          const uint4 pu = *reinterpret_cast<const uint4*>(sa + off);
          const uint4 pg = *reinterpret_cast<const uint4*>(sg + off);
          const uint32_t uw[4] = {pu.x, pu.y, pu.z, pu.w};
          const uint32_t gw[4] = {pg.x, pg.y, pg.z, pg.w};
          uint32_t o[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 a = fma2(fma2(unpack_bf16x2(uw[e]), rsu[i], cu[i]), wx[e], cx[e]);
            const float2 sv = fma2(fma2(unpack_bf16x2(gw[e]), rsg[i], cgs[i]), wg[e], cg[e]);
            const float2 h = mul2(sv, half2);
            const float2 silu = fma2(h, make_float2(tanh_fast(h.x), tanh_fast(h.y)), h);
            const float2 ov = mul2(a, silu);
            o[e] = pack_bf16x2(ov.x, ov.y);
          }
          // rows past M and columns past H (G columns in the U box's tail) are zero
          outv[i] = (valid[i] && kv) ? make_uint4(o[0], o[1], o[2], o[3]) : make_uint4(0u, 0u, 0u, 0u);
          *reinterpret_cast<uint4*>(sa + off) = outv[i];
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          if (leader)
            mbar_arrive(&full[stage]);
          else
            mbar_arrive_remote(mapa_shared(smem_u32(&full[stage]), 0));
        }
        // Hl goes out after the arrive: a cluster-scope release-arrive would
        // otherwise wait for these stores to complete
        if (hl_row0 != nullptr && kv) {
#pragma unroll
          for (int i = 0; i < Cfg::XF_ROWS; ++i)
            if (valid[i]) __stcs(reinterpret_cast<uint4*>(hl_row0 + static_cast<int64_t>(RSTEP * i) * q.H + k), outv[i]);
        }
        if (++stage == Cfg::STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  }

  griddep_launch_dependents();
  tc_fence_before_sync();
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc_pair(tmem_base, Cfg::TMEM_COLS);
  }
}

}  // namespace

int gemm_gated_tile_n() { return GatedCfg::BN_OUT; }
int gemm_gated_bk() { return GatedCfg::BK; }

cudaError_t launch_gemm_gated(const CUtensorMap& b, const CUtensorMap& d, const CUtensorMap& z, const GemmParams& p,
                              const GateSrc& q, int num_sms, cudaStream_t s) {
  using Cfg = GatedCfg;
  static std::atomic<int> units_cache[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  int units = units_cache[dev].load(std::memory_order_relaxed);
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(Cfg::NUM_THREADS);
  cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (units == 0) {
    e = cudaFuncSetAttribute(gemm_gated_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    cfg.gridDim = dim3(2);
    int clusters = 0;
    e = cudaOccupancyMaxActiveClusters(&clusters, gemm_gated_kernel, &cfg);
    if (e != cudaSuccess) return e;
    units = clusters > 0 ? clusters : 1;
    units_cache[dev].store(units, std::memory_order_relaxed);
  }
  (void)num_sms;
  const int64_t tiles = static_cast<int64_t>(p.G) * p.tiles_m * p.tiles_n;
  if (tiles < units) units = static_cast<int>(tiles);
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.numAttrs = 2;
  cfg.stream = s;
  cfg.gridDim = dim3(units * Cfg::CTAS);
  return cudaLaunchKernelEx(&cfg, gemm_gated_kernel, b, d, z, p, q);
}

}  // namespace dg
