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

#include "dg_internal.h"

namespace dg {

namespace {

constexpr int kMaxRowWarps = 16;  // row kernels use up to 512 threads
constexpr int kRowThreads = 256;  // threads of the per-row kernels

__device__ __forceinline__ void unpack8(const uint4 v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 t = unpack_bf16x2(w[e]);
    f[2 * e] = t.x;
    f[2 * e + 1] = t.y;
  }
}

__device__ __forceinline__ void load8(const __nv_bfloat16* p, float (&f)[8]) {
  const uint4 v = __ldg(reinterpret_cast<const uint4*>(p));
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 t = unpack_bf16x2(w[e]);
    f[2 * e] = t.x;
    f[2 * e + 1] = t.y;
  }
}

__device__ __forceinline__ void load8_stream(const __nv_bfloat16* p, float (&f)[8]) {
  const uint4 v = __ldcs(reinterpret_cast<const uint4*>(p));
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 t = unpack_bf16x2(w[e]);
    f[2 * e] = t.x;
    f[2 * e + 1] = t.y;
  }
}

__device__ __forceinline__ void load4(const __nv_bfloat16* p, float (&f)[4]) {
  const uint2 v = __ldg(reinterpret_cast<const uint2*>(p));
  const float2 a = unpack_bf16x2(v.x), b = unpack_bf16x2(v.y);
  f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
}


__device__ __forceinline__ void store8(__nv_bfloat16* p, const float (&f)[8]) {
  uint4 v;
  v.x = pack_bf16x2(f[0], f[1]);
  v.y = pack_bf16x2(f[2], f[3]);
  v.z = pack_bf16x2(f[4], f[5]);
  v.w = pack_bf16x2(f[6], f[7]);
  *reinterpret_cast<uint4*>(p) = v;
}

__device__ __forceinline__ void store8_stream(__nv_bfloat16* p, const float (&f)[8]) {
  uint4 v;
  v.x = pack_bf16x2(f[0], f[1]);
  v.y = pack_bf16x2(f[2], f[3]);
  v.z = pack_bf16x2(f[4], f[5]);
  v.w = pack_bf16x2(f[6], f[7]);
  __stcs(reinterpret_cast<uint4*>(p), v);
}

__device__ __forceinline__ float sigmoid_f(float x) { return 1.0f / (1.0f + __expf(-x)); }

// Block-uniform read of the error word (a divergent early return ahead of a
// barrier would be undefined).
__device__ __forceinline__ bool block_aborted(const uint32_t* err) {
  __shared__ uint32_t flag;
  if (threadIdx.x == 0) flag = ld_volatile_u32(err);
  __syncthreads();
  return flag != 0u;
}

// Block-wide sums of N values; consecutive calls must alternate `slot`,
// which makes a trailing barrier unnecessary.
template <int N>
__device__ __forceinline__ void block_sum(float (&v)[N], float (*sm)[kMaxRowWarps][4], int slot) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nwarps = blockDim.x >> 5;
#pragma unroll
  for (int i = 0; i < N; ++i) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v[i] += __shfl_xor_sync(0xffffffffu, v[i], o);
  }
  if (lane == 0) {
#pragma unroll
    for (int i = 0; i < N; ++i) sm[slot][warp][i] = v[i];
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < N; ++i) {
    float t = 0.0f;
    for (int w = 0; w < nwarps; ++w) t += sm[slot][w][i];
    v[i] = t;
  }
}

// ------------------------------------------------------------------ forward
//
// One 256-thread CTA per row (grid-stride), several CTAs per SM.  Thread i
// keeps 8-column vectors i, i + 256, ... of U and G as packed bf16 in
// registers: mean, then the centred second moment (two passes, no
// cancellation), then the affine and the gate.

template <int VPT>
__global__ void __launch_bounds__(kRowThreads, 2) ln_gate_fwd_kernel(
    const __nv_bfloat16* __restrict__ Z, const __nv_bfloat16* __restrict__ gx, const __nv_bfloat16* __restrict__ bx,
    const __nv_bfloat16* __restrict__ gg, const __nv_bfloat16* __restrict__ bg, __nv_bfloat16* __restrict__ Hl,
    float4* __restrict__ stats, int64_t rows, int M, int L, int H, float eps, const uint32_t* err) {
  __shared__ float sm[2][kMaxRowWarps][4];
  if (block_aborted(err)) return;
  const int nvec = H >> 3;
  const float inv_h = 1.0f / static_cast<float>(H);
  for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
    const int r = static_cast<int>(row / M) / L;
    const __nv_bfloat16* zu = Z + row * (2 * static_cast<int64_t>(H));
    const __nv_bfloat16* zg = zu + H;
    uint4 pu[VPT], pg[VPT];
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
      const int v = threadIdx.x + kRowThreads * j;
      if (v < nvec) {
        pu[j] = __ldcs(reinterpret_cast<const uint4*>(zu + 8 * v));
        pg[j] = __ldcs(reinterpret_cast<const uint4*>(zg + 8 * v));
      } else {
        pu[j] = pg[j] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
    float s[2] = {0.0f, 0.0f};
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
      float u[8], g[8];
      unpack8(pu[j], u);
      unpack8(pg[j], g);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        s[0] += u[e];
        s[1] += g[e];
      }
    }
    block_sum<2>(s, sm, 0);
    const float mu_u = s[0] * inv_h, mu_g = s[1] * inv_h;
    float q[2] = {0.0f, 0.0f};
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
      if (threadIdx.x + kRowThreads * j < nvec) {
        float u[8], g[8];
        unpack8(pu[j], u);
        unpack8(pg[j], g);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float du = u[e] - mu_u, dg = g[e] - mu_g;
          q[0] += du * du;
          q[1] += dg * dg;
        }
      }
    }
    block_sum<2>(q, sm, 1);
    const float rs_u = rsqrtf(q[0] * inv_h + eps), rs_g = rsqrtf(q[1] * inv_h + eps);
    __nv_bfloat16* hrow = Hl + row * static_cast<int64_t>(H);
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
      const int v = threadIdx.x + kRowThreads * j;
      if (v < nvec) {
        float u[8], g[8], wx[8], cx[8], wg[8], cg[8], h[8];
        unpack8(pu[j], u);
        unpack8(pg[j], g);
        const int64_t po = static_cast<int64_t>(r) * H + 8 * v;
        load8(gx + po, wx);
        load8(bx + po, cx);
        load8(gg + po, wg);
        load8(bg + po, cg);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float a = (u[e] - mu_u) * rs_u * wx[e] + cx[e];
          const float sg = (g[e] - mu_g) * rs_g * wg[e] + cg[e];
          h[e] = a * (sg * sigmoid_f(sg));
        }
        store8_stream(hrow + 8 * v, h);
      }
    }
    if (threadIdx.x == 0) stats[row] = make_float4(mu_u, rs_u, mu_g, rs_g);
  }
}

// ------------------------------------------------------------------ backward
//
// With x_u = (U - mu_u) * rstd_u, a = x_u*gx + bx, x_g likewise, s = x_g*gg + bg,
// q = silu(s), Hl = a*q:  da = dHl*q, ds = dHl*a*sigmoid(s)*(1 + s*(1 - sigmoid(s))),
// dx_u = da*gx, dU = rstd_u * (dx_u - mean(dx_u) - x_u*mean(dx_u*x_u)), and the
// same for G with ds and gg.
//
// Pass 1 (row sums): one CTA per row computes sum(dx_u), sum(dx_u*x_u),
// sum(dx_g), sum(dx_g*x_g) -> rowsum[row].
// Pass 2 (apply): a CTA owns 8*128 columns of one token position t and walks
// all M rows of t: it writes dZ and keeps the column sums of dU, dG (db1),
// da*x_u, da (norm_x grads), ds*x_g, ds (norm_gate grads) in registers, so
// every column sum is complete in one CTA (fixed order, deterministic).

template <int VPT>
__global__ void __launch_bounds__(kRowThreads, 2) ln_gate_bwd_rowsum_kernel(
    const __nv_bfloat16* __restrict__ Z, const float4* __restrict__ stats, const __nv_bfloat16* __restrict__ dHl,
    const __nv_bfloat16* __restrict__ gx, const __nv_bfloat16* __restrict__ bx, const __nv_bfloat16* __restrict__ gg,
    const __nv_bfloat16* __restrict__ bg, float4* __restrict__ rowsum, int64_t rows, int M, int L, int H,
    const uint32_t* err) {
  __shared__ float sm[2][kMaxRowWarps][4];
  if (block_aborted(err)) return;
  const int nvec = H >> 3;
  int slot = 0;
  for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
    const int r = static_cast<int>(row / M) / L;
    const float4 st = stats[row];
    const __nv_bfloat16* zu = Z + row * (2 * static_cast<int64_t>(H));
    const __nv_bfloat16* zg = zu + H;
    const __nv_bfloat16* dh = dHl + row * static_cast<int64_t>(H);
    uint4 pu[VPT], pg[VPT], ph[VPT];
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
      const int v = threadIdx.x + kRowThreads * j;
      if (v < nvec) {
        pu[j] = __ldcs(reinterpret_cast<const uint4*>(zu + 8 * v));
        pg[j] = __ldcs(reinterpret_cast<const uint4*>(zg + 8 * v));
        ph[j] = __ldcs(reinterpret_cast<const uint4*>(dh + 8 * v));
      }
    }
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
      const int v = threadIdx.x + kRowThreads * j;
      if (v < nvec) {
        float u[8], g[8], hv[8], wx[8], cx[8], wg[8], cg[8];
        unpack8(pu[j], u);
        unpack8(pg[j], g);
        unpack8(ph[j], hv);
        const int64_t po = static_cast<int64_t>(r) * H + 8 * v;
        load8(gx + po, wx);
        load8(bx + po, cx);
        load8(gg + po, wg);
        load8(bg + po, cg);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float xu = (u[e] - st.x) * st.y, xg = (g[e] - st.z) * st.w;
          const float a = xu * wx[e] + cx[e], sv = xg * wg[e] + cg[e];
          const float sgm = sigmoid_f(sv);
          const float dxu = hv[e] * (sv * sgm) * wx[e];
          const float dxg = hv[e] * a * (sgm * (1.0f + sv * (1.0f - sgm))) * wg[e];
          acc[0] += dxu;
          acc[1] += dxu * xu;
          acc[2] += dxg;
          acc[3] += dxg * xg;
        }
      }
    }
    block_sum<4>(acc, sm, slot);
    slot ^= 1;
    if (threadIdx.x == 0) rowsum[row] = make_float4(acc[0], acc[1], acc[2], acc[3]);
  }
}

constexpr int kApplyThreads = 128;
constexpr int kApplyCols = 8 * kApplyThreads;

__global__ void __launch_bounds__(kApplyThreads) ln_gate_bwd_apply_kernel(
    const __nv_bfloat16* __restrict__ Z, const float4* __restrict__ stats, const float4* __restrict__ rowsum,
    const __nv_bfloat16* __restrict__ dHl, const __nv_bfloat16* __restrict__ gx, const __nv_bfloat16* __restrict__ bx,
    const __nv_bfloat16* __restrict__ gg, const __nv_bfloat16* __restrict__ bg, __nv_bfloat16* __restrict__ dZ,
    __nv_bfloat16* __restrict__ d_b1, float* __restrict__ norm_part, int M, int L, int H, const uint32_t* err) {
  if (ld_volatile_u32(err) != 0u) return;
  const int t = blockIdx.y;
  const int r = t / L;
  const int c0 = blockIdx.x * kApplyCols + 8 * threadIdx.x;
  if (c0 >= H) return;
  const float inv_h = 1.0f / static_cast<float>(H);
  float wx[8], cx[8], wg[8], cg[8];
  {
    const int64_t po = static_cast<int64_t>(r) * H + c0;
    load8(gx + po, wx);
    load8(bx + po, cx);
    load8(gg + po, wg);
    load8(bg + po, cg);
  }
  float s_du[8], s_dg[8], s_gx[8], s_bx[8], s_gg[8], s_bg[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) s_du[e] = s_dg[e] = s_gx[e] = s_bx[e] = s_gg[e] = s_bg[e] = 0.0f;
  const int64_t row0 = static_cast<int64_t>(t) * M;
  const int64_t zstride = 2 * static_cast<int64_t>(H);
  constexpr int U = 2;  // rows in flight per thread
  for (int n = 0; n < M; n += U) {
    uint4 pu[U], pg[U], ph[U];
    float4 st[U], rs[U];
#pragma unroll
    for (int i = 0; i < U; ++i) {
      if (n + i < M) {
        const int64_t row = row0 + n + i;
        pu[i] = __ldcs(reinterpret_cast<const uint4*>(Z + row * zstride + c0));
        pg[i] = __ldcs(reinterpret_cast<const uint4*>(Z + row * zstride + H + c0));
        ph[i] = __ldcs(reinterpret_cast<const uint4*>(dHl + row * H + c0));
        st[i] = stats[row];
        rs[i] = rowsum[row];
      }
    }
#pragma unroll
    for (int i = 0; i < U; ++i) {
      if (n + i < M) {
        const int64_t row = row0 + n + i;
        float u[8], g[8], hv[8], du[8], dg[8];
        unpack8(pu[i], u);
        unpack8(pg[i], g);
        unpack8(ph[i], hv);
        const float m1u = rs[i].x * inv_h, m2u = rs[i].y * inv_h;
        const float m1g = rs[i].z * inv_h, m2g = rs[i].w * inv_h;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float xu = (u[e] - st[i].x) * st[i].y, xg = (g[e] - st[i].z) * st[i].w;
          const float a = xu * wx[e] + cx[e], sv = xg * wg[e] + cg[e];
          const float sgm = sigmoid_f(sv);
          const float da = hv[e] * (sv * sgm);
          const float ds = hv[e] * a * (sgm * (1.0f + sv * (1.0f - sgm)));
          du[e] = st[i].y * (da * wx[e] - m1u - xu * m2u);
          dg[e] = st[i].w * (ds * wg[e] - m1g - xg * m2g);
          s_du[e] += du[e];
          s_dg[e] += dg[e];
          s_gx[e] += da * xu;
          s_bx[e] += da;
          s_gg[e] += ds * xg;
          s_bg[e] += ds;
        }
        store8_stream(dZ + row * zstride + c0, du);
        store8_stream(dZ + row * zstride + H + c0, dg);
      }
    }
  }
  store8(d_b1 + static_cast<int64_t>(t) * 2 * H + c0, s_du);
  store8(d_b1 + static_cast<int64_t>(t) * 2 * H + H + c0, s_dg);
  float* np = norm_part + static_cast<int64_t>(t) * 4 * H + c0;
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    np[e] = s_gx[e];
    np[H + e] = s_bx[e];
    np[2 * H + e] = s_gg[e];
    np[3 * H + e] = s_bg[e];
  }
}

// Norm gradients of rank r: sum of its L slices' column sums, in slice order.
__global__ void norm_reduce_kernel(const float* __restrict__ norm_part, __nv_bfloat16* __restrict__ d_nx_w,
                                   __nv_bfloat16* __restrict__ d_nx_b, __nv_bfloat16* __restrict__ d_ng_w,
                                   __nv_bfloat16* __restrict__ d_ng_b, int P, int L, int H, const uint32_t* err) {
  if (ld_volatile_u32(err) != 0u) return;
  const int64_t n = static_cast<int64_t>(P) * 4 * H;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int r = static_cast<int>(i / (4 * H));
    const int q = static_cast<int>((i / H) % 4);  // 0: nx_w, 1: nx_b, 2: ng_w, 3: ng_b
    const int c = static_cast<int>(i % H);
    float s = 0.0f;
    for (int l = 0; l < L; ++l) s += norm_part[(static_cast<int64_t>(r * L + l) * 4 + q) * H + c];
    __nv_bfloat16* out = q == 0 ? d_nx_w : q == 1 ? d_nx_b : q == 2 ? d_ng_w : d_ng_b;
    out[static_cast<int64_t>(r) * H + c] = __float2bfloat16_rn(s);
  }
}

// out[g, c] = sum over rows n of src[g*g_stride + n*row_stride + c]; two columns per thread.
__global__ void column_sum_kernel(const __nv_bfloat16* __restrict__ src, __nv_bfloat16* __restrict__ out, int rows,
                                  int ncols, int64_t g_stride, int64_t row_stride, const uint32_t* err) {
  if (ld_volatile_u32(err) != 0u) return;
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

// Exchange permutations, 16 bytes per thread.
__global__ void dispatch_kernel(const uint4* __restrict__ in, uint4* __restrict__ out, int P, int B, int T,
                                int vec_per_row, const uint32_t* err) {
  if (ld_volatile_u32(err) != 0u) return;
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
  if (ld_volatile_u32(err) != 0u) return;
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

// Waits, with the library's bounded wait, on a barrier nobody arrives at.
__global__ void debug_wait_kernel(uint32_t* err, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(&bar, 0u, err, 0x7fu, limit_ns);
}

int grid_for(const DeviceInfo& dev, const void* kernel, int threads, size_t smem, int64_t work_items) {
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, smem) != cudaSuccess || per_sm < 1)
    per_sm = 1;
  int64_t g = static_cast<int64_t>(per_sm) * dev.num_sms;
  if (work_items < g) g = work_items;
  return static_cast<int>(g < 1 ? 1 : g);
}

}  // namespace

cudaError_t launch_ln_gate_fwd(const void* Z, const void* nx_w, const void* nx_b, const void* ng_w,
                               const void* ng_b, void* Hl, void* stats, int64_t rows, int M, int L, int H,
                               float eps, const DeviceInfo& dev, cudaStream_t s) {
  const int vpt = (H / 8 + kRowThreads - 1) / kRowThreads;
  auto run = [&](auto kern) {
    const int grid = grid_for(dev, reinterpret_cast<const void*>(kern), kRowThreads, 0, rows);
    kern<<<grid, kRowThreads, 0, s>>>(static_cast<const __nv_bfloat16*>(Z), static_cast<const __nv_bfloat16*>(nx_w),
                                      static_cast<const __nv_bfloat16*>(nx_b), static_cast<const __nv_bfloat16*>(ng_w),
                                      static_cast<const __nv_bfloat16*>(ng_b), static_cast<__nv_bfloat16*>(Hl),
                                      static_cast<float4*>(stats), rows, M, L, H, eps, dev.err);
    return cudaGetLastError();
  };
  if (vpt <= 1) return run(ln_gate_fwd_kernel<1>);
  if (vpt <= 2) return run(ln_gate_fwd_kernel<2>);
  if (vpt <= 4) return run(ln_gate_fwd_kernel<4>);
  return cudaErrorInvalidValue;
}

cudaError_t launch_ln_gate_bwd_rowsum(const void* Z, const void* stats, const void* dHl, const void* nx_w,
                                      const void* nx_b, const void* ng_w, const void* ng_b, void* rowsum, int T, int M,
                                      int L, int H, const DeviceInfo& dev, cudaStream_t s) {
  const int64_t rows = static_cast<int64_t>(T) * M;
  const int vpt = (H / 8 + kRowThreads - 1) / kRowThreads;
  auto run = [&](auto kern) {
    const int grid = grid_for(dev, reinterpret_cast<const void*>(kern), kRowThreads, 0, rows);
    kern<<<grid, kRowThreads, 0, s>>>(static_cast<const __nv_bfloat16*>(Z), static_cast<const float4*>(stats),
                                      static_cast<const __nv_bfloat16*>(dHl), static_cast<const __nv_bfloat16*>(nx_w),
                                      static_cast<const __nv_bfloat16*>(nx_b), static_cast<const __nv_bfloat16*>(ng_w),
                                      static_cast<const __nv_bfloat16*>(ng_b), static_cast<float4*>(rowsum), rows, M,
                                      L, H, dev.err);
    return cudaGetLastError();
  };
  if (vpt <= 1) return run(ln_gate_bwd_rowsum_kernel<1>);
  if (vpt <= 2) return run(ln_gate_bwd_rowsum_kernel<2>);
  if (vpt <= 4) return run(ln_gate_bwd_rowsum_kernel<4>);
  return cudaErrorInvalidValue;
}

cudaError_t launch_ln_gate_bwd_apply(const void* Z, const void* stats, const void* rowsum, const void* dHl,
                                     const void* nx_w, const void* nx_b, const void* ng_w, const void* ng_b, void* dZ,
                                     void* d_b1, float* norm_part, int T, int M, int L, int H, const DeviceInfo& dev,
                                     cudaStream_t s) {
  dim3 grid((H + kApplyCols - 1) / kApplyCols, T);
  ln_gate_bwd_apply_kernel<<<grid, kApplyThreads, 0, s>>>(
      static_cast<const __nv_bfloat16*>(Z), static_cast<const float4*>(stats), static_cast<const float4*>(rowsum),
      static_cast<const __nv_bfloat16*>(dHl), static_cast<const __nv_bfloat16*>(nx_w),
      static_cast<const __nv_bfloat16*>(nx_b), static_cast<const __nv_bfloat16*>(ng_w),
      static_cast<const __nv_bfloat16*>(ng_b), static_cast<__nv_bfloat16*>(dZ), static_cast<__nv_bfloat16*>(d_b1),
      norm_part, M, L, H, dev.err);
  return cudaGetLastError();
}

cudaError_t launch_norm_reduce(const float* norm_part, void* d_nx_w, void* d_nx_b, void* d_ng_w, void* d_ng_b, int P,
                               int L, int H, const DeviceInfo& dev, cudaStream_t s) {
  const int64_t n = static_cast<int64_t>(P) * 4 * H;
  int64_t blocks = (n + 255) / 256;
  if (blocks > 8 * dev.num_sms) blocks = 8 * dev.num_sms;
  norm_reduce_kernel<<<static_cast<int>(blocks), 256, 0, s>>>(
      norm_part, static_cast<__nv_bfloat16*>(d_nx_w), static_cast<__nv_bfloat16*>(d_nx_b),
      static_cast<__nv_bfloat16*>(d_ng_w), static_cast<__nv_bfloat16*>(d_ng_b), P, L, H, dev.err);
  return cudaGetLastError();
}

cudaError_t launch_column_sum(const void* src, void* out, int G, int rows, int ncols, int64_t g_stride,
                              int64_t row_stride, const DeviceInfo& dev, cudaStream_t s) {
  const int threads = 128;
  dim3 grid((ncols / 2 + threads - 1) / threads, G);
  column_sum_kernel<<<grid, threads, 0, s>>>(static_cast<const __nv_bfloat16*>(src), static_cast<__nv_bfloat16*>(out),
                                            rows, ncols, g_stride, row_stride, dev.err);
  return cudaGetLastError();
}

cudaError_t launch_dispatch(const void* in, void* out, int P, int B, int T, int D, const DeviceInfo& dev,
                            cudaStream_t s) {
  const int64_t total = static_cast<int64_t>(P) * B * T * (D / 8);
  int64_t blocks = (total + 255) / 256;
  if (blocks > 16 * dev.num_sms) blocks = 16 * dev.num_sms;
  dispatch_kernel<<<static_cast<int>(blocks), 256, 0, s>>>(static_cast<const uint4*>(in), static_cast<uint4*>(out), P,
                                                            B, T, D / 8, dev.err);
  return cudaGetLastError();
}

cudaError_t launch_combine(const void* in, void* out, int P, int B, int T, int D, const DeviceInfo& dev,
                           cudaStream_t s) {
  const int64_t total = static_cast<int64_t>(P) * B * T * (D / 8);
  int64_t blocks = (total + 255) / 256;
  if (blocks > 16 * dev.num_sms) blocks = 16 * dev.num_sms;
  combine_kernel<<<static_cast<int>(blocks), 256, 0, s>>>(static_cast<const uint4*>(in), static_cast<uint4*>(out), P,
                                                           B, T, D / 8, dev.err);
  return cudaGetLastError();
}

cudaError_t launch_debug_wait(uint32_t* err, uint64_t limit_ns, cudaStream_t s) {
  debug_wait_kernel<<<1, 32, 0, s>>>(err, limit_ns);
  return cudaGetLastError();
}

}  // namespace dg
