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


__device__ __forceinline__ void store8_stream(__nv_bfloat16* p, const float (&f)[8]) {
  uint4 v;
  v.x = pack_bf16x2(f[0], f[1]);
  v.y = pack_bf16x2(f[2], f[3]);
  v.z = pack_bf16x2(f[4], f[5]);
  v.w = pack_bf16x2(f[6], f[7]);
  __stcs(reinterpret_cast<uint4*>(p), v);
}

// sigmoid(x) = (1 + tanh(x/2)) / 2, with the hardware tanh approximation
// (tanh.approx.f32, relative error about 2^-11): one MUFU operation instead of
// an exponential and a division.
__device__ __forceinline__ float tanh_fast(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float sigmoid_fast(float x) { return fmaf(0.5f, tanh_fast(0.5f * x), 0.5f); }

// silu(x) = x * sigmoid(x) = h + h * tanh(h) with h = x/2.
__device__ __forceinline__ float silu_fast(float x) {
  const float h = 0.5f * x;
  return fmaf(h, tanh_fast(h), h);
}

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
// One CTA per row (grid-stride).  Thread i keeps 8-column vectors
// i, i + blockDim, ... of U and G as packed bf16 in registers, and loads the
// CTA's next row while it finishes the current one.  The row statistics use
// the shifted-data single pass (Chan, Golub & LeVeque, "Algorithms for
// computing the sample variance"): with K the row's first element,
// mean = K + S1/H and var = S2/H - (S1/H)^2 where S1 = sum(x-K),
// S2 = sum((x-K)^2); K is a sample of the row, so the subtraction does not
// cancel catastrophically, and a constant row gives exactly var = 0.

template <int VPT>
struct RowFrag {
  uint4 u[VPT], g[VPT];
  float ku, kg;
};

template <int VPT>
__device__ __forceinline__ void load_zrow(RowFrag<VPT>& f, const __nv_bfloat16* zu, int H, int nvec) {
  const __nv_bfloat16* zg = zu + H;
#pragma unroll
  for (int j = 0; j < VPT; ++j) {
    const int v = threadIdx.x + blockDim.x * j;
    if (v < nvec) {
      f.u[j] = __ldcs(reinterpret_cast<const uint4*>(zu + 8 * v));
      f.g[j] = __ldcs(reinterpret_cast<const uint4*>(zg + 8 * v));
    } else {
      f.u[j] = f.g[j] = make_uint4(0u, 0u, 0u, 0u);
    }
  }
  f.ku = __bfloat162float(zu[0]);
  f.kg = __bfloat162float(zg[0]);
}

template <int VPT>
__global__ void __launch_bounds__(kRowThreads, 2) ln_gate_fwd_kernel(
    const __nv_bfloat16* __restrict__ Z, const __nv_bfloat16* __restrict__ gx, const __nv_bfloat16* __restrict__ bx,
    const __nv_bfloat16* __restrict__ gg, const __nv_bfloat16* __restrict__ bg, __nv_bfloat16* __restrict__ Hl,
    float4* __restrict__ stats, int64_t rows, int M, int L, int H, float eps, const uint32_t* err) {
  __shared__ float sm[2][kMaxRowWarps][4];
  if (block_aborted(err)) return;
  const int nvec = H >> 3;
  const float inv_h = 1.0f / static_cast<float>(H);
  const int64_t zstride = 2 * static_cast<int64_t>(H);
  RowFrag<VPT> cur, nxt;
  int64_t row = blockIdx.x;
  if (row < rows) load_zrow(cur, Z + row * zstride, H, nvec);
  int slot = 0;
  for (; row < rows; row += gridDim.x) {
    const int64_t next = row + gridDim.x;
    if (next < rows) load_zrow(nxt, Z + next * zstride, H, nvec);
    const int r = static_cast<int>(row / M) / L;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
      if (threadIdx.x + blockDim.x * j < nvec) {
        float u[8], g[8];
        unpack8(cur.u[j], u);
        unpack8(cur.g[j], g);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float du = u[e] - cur.ku, dg = g[e] - cur.kg;
          acc[0] += du;
          acc[1] = fmaf(du, du, acc[1]);
          acc[2] += dg;
          acc[3] = fmaf(dg, dg, acc[3]);
        }
      }
    }
    block_sum<4>(acc, sm, slot);
    slot ^= 1;
    const float m1u = acc[0] * inv_h, m1g = acc[2] * inv_h;
    const float mu_u = cur.ku + m1u, mu_g = cur.kg + m1g;
    const float rs_u = rsqrtf(fmaxf(acc[1] * inv_h - m1u * m1u, 0.0f) + eps);
    const float rs_g = rsqrtf(fmaxf(acc[3] * inv_h - m1g * m1g, 0.0f) + eps);
    const float cu = -mu_u * rs_u, cgg = -mu_g * rs_g;
    __nv_bfloat16* hrow = Hl + row * static_cast<int64_t>(H);
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
      const int v = threadIdx.x + blockDim.x * j;
      if (v < nvec) {
        float u[8], g[8], wx[8], cx[8], wg[8], cg[8], h[8];
        unpack8(cur.u[j], u);
        unpack8(cur.g[j], g);
        const int64_t po = static_cast<int64_t>(r) * H + 8 * v;
        load8(gx + po, wx);
        load8(bx + po, cx);
        load8(gg + po, wg);
        load8(bg + po, cg);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float a = fmaf(fmaf(u[e], rs_u, cu), wx[e], cx[e]);
          const float sg = fmaf(fmaf(g[e], rs_g, cgg), wg[e], cg[e]);
          h[e] = a * silu_fast(sg);
        }
        store8_stream(hrow + 8 * v, h);
      }
    }
    if (threadIdx.x == 0) stats[row] = make_float4(mu_u, rs_u, mu_g, rs_g);
    cur = nxt;
  }
}

// ------------------------------------------------------------------ backward
//
// With x_u = (U - mu_u) * rstd_u, a = x_u*gx + bx, x_g likewise, s = x_g*gg + bg,
// q = silu(s), Hl = a*q:  da = dHl*q, ds = dHl*a*silu'(s) with
// silu'(s) = sig(s) + s*sig(s)*(1 - sig(s)), dx_u = da*gx,
// dU = rstd_u * (dx_u - mean(dx_u) - x_u*mean(dx_u*x_u)), and the same for G.
//
// Pass 1 (row sums): one CTA per row computes sum(dx_u), sum(dx_u*x_u),
// sum(dx_g), sum(dx_g*x_g) -> rowsum[row], loading the next row early.
// Pass 2 (apply): a CTA owns a column block of one token position t and a
// range of its rows: it writes dZ and sums, per column, dU, dG (db1),
// da*x_u, da (norm_x grads), ds*x_g, ds (norm_gate grads) in registers; the
// per-(t, row range) partial sums are added in a fixed order afterwards.

template <int VPT>
struct GradFrag {
  uint4 u[VPT], g[VPT], h[VPT];
  float4 st;
};

template <int VPT>
__device__ __forceinline__ void load_grow(GradFrag<VPT>& f, const __nv_bfloat16* zu, const __nv_bfloat16* dh,
                                          const float4* st, int H, int nvec) {
  const __nv_bfloat16* zg = zu + H;
#pragma unroll
  for (int j = 0; j < VPT; ++j) {
    const int v = threadIdx.x + blockDim.x * j;
    if (v < nvec) {
      f.u[j] = __ldcs(reinterpret_cast<const uint4*>(zu + 8 * v));
      f.g[j] = __ldcs(reinterpret_cast<const uint4*>(zg + 8 * v));
      f.h[j] = __ldcs(reinterpret_cast<const uint4*>(dh + 8 * v));
    }
  }
  f.st = *st;
}

template <int VPT>
__global__ void __launch_bounds__(512, 1) ln_gate_bwd_rowsum_kernel(
    const __nv_bfloat16* __restrict__ Z, const float4* __restrict__ stats, const __nv_bfloat16* __restrict__ dHl,
    const __nv_bfloat16* __restrict__ gx, const __nv_bfloat16* __restrict__ bx, const __nv_bfloat16* __restrict__ gg,
    const __nv_bfloat16* __restrict__ bg, float4* __restrict__ rowsum, int64_t rows, int M, int L, int H,
    const uint32_t* err) {
  __shared__ float sm[2][kMaxRowWarps][4];
  if (block_aborted(err)) return;
  const int nvec = H >> 3;
  const int64_t zstride = 2 * static_cast<int64_t>(H);
  GradFrag<VPT> cur, nxt;
  int64_t row = blockIdx.x;
  if (row < rows) load_grow(cur, Z + row * zstride, dHl + row * H, stats + row, H, nvec);
  int slot = 0;
  for (; row < rows; row += gridDim.x) {
    const int64_t next = row + gridDim.x;
    if (next < rows) load_grow(nxt, Z + next * zstride, dHl + next * H, stats + next, H, nvec);
    const int r = static_cast<int>(row / M) / L;
    const float4 st = cur.st;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
      const int v = threadIdx.x + blockDim.x * j;
      if (v < nvec) {
        float u[8], g[8], hv[8], wx[8], cx[8], wg[8], cg[8];
        unpack8(cur.u[j], u);
        unpack8(cur.g[j], g);
        unpack8(cur.h[j], hv);
        const int64_t po = static_cast<int64_t>(r) * H + 8 * v;
        load8(gx + po, wx);
        load8(bx + po, cx);
        load8(gg + po, wg);
        load8(bg + po, cg);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float xu = (u[e] - st.x) * st.y, xg = (g[e] - st.z) * st.w;
          const float a = fmaf(xu, wx[e], cx[e]), sv = fmaf(xg, wg[e], cg[e]);
          const float sg = sigmoid_fast(sv);
          const float dxu = hv[e] * (sv * sg) * wx[e];
          const float dxg = hv[e] * a * fmaf(sv * sg, 1.0f - sg, sg) * wg[e];
          acc[0] += dxu;
          acc[1] = fmaf(dxu, xu, acc[1]);
          acc[2] += dxg;
          acc[3] = fmaf(dxg, xg, acc[3]);
        }
      }
    }
    block_sum<4>(acc, sm, slot);
    slot ^= 1;
    if (threadIdx.x == 0) rowsum[row] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    cur = nxt;
  }
}

constexpr int kApplyVec = 4;   // columns per thread
constexpr int kApplyRows = 4;  // rows in flight per thread

__device__ __forceinline__ void unpack4(const uint2 v, float (&f)[4]) {
  const float2 a = unpack_bf16x2(v.x), b = unpack_bf16x2(v.y);
  f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
}

__device__ __forceinline__ uint2 pack4(const float (&f)[4]) {
  return make_uint2(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]));
}

// grid: (column blocks, T, row splits); block: cols_per_block / 4 threads.
__global__ void __launch_bounds__(256) ln_gate_bwd_apply_kernel(
    const __nv_bfloat16* __restrict__ Z, const float4* __restrict__ stats, const float4* __restrict__ rowsum,
    const __nv_bfloat16* __restrict__ dHl, const __nv_bfloat16* __restrict__ gx, const __nv_bfloat16* __restrict__ bx,
    const __nv_bfloat16* __restrict__ gg, const __nv_bfloat16* __restrict__ bg, __nv_bfloat16* __restrict__ dZ,
    float* __restrict__ part, int M, int L, int H, int cols_per_block, const uint32_t* err) {
  if (ld_volatile_u32(err) != 0u) return;
  const int t = blockIdx.y, rs = blockIdx.z, nsplit = gridDim.z;
  const int r = t / L;
  const int c0 = blockIdx.x * cols_per_block + kApplyVec * threadIdx.x;
  if (kApplyVec * threadIdx.x >= cols_per_block || c0 >= H) return;
  const float inv_h = 1.0f / static_cast<float>(H);
  float wx[4], cx[4], wg[4], cg[4];
  {
    const int64_t po = static_cast<int64_t>(r) * H + c0;
    unpack4(__ldg(reinterpret_cast<const uint2*>(gx + po)), wx);
    unpack4(__ldg(reinterpret_cast<const uint2*>(bx + po)), cx);
    unpack4(__ldg(reinterpret_cast<const uint2*>(gg + po)), wg);
    unpack4(__ldg(reinterpret_cast<const uint2*>(bg + po)), cg);
  }
  float s_du[4], s_dg[4], s_gx[4], s_bx[4], s_gg[4], s_bg[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) s_du[e] = s_dg[e] = s_gx[e] = s_bx[e] = s_gg[e] = s_bg[e] = 0.0f;
  const int rows_per = (M + nsplit - 1) / nsplit;
  const int n_begin = rs * rows_per, n_end = min(M, n_begin + rows_per);
  const int64_t row0 = static_cast<int64_t>(t) * M;
  const int64_t zstride = 2 * static_cast<int64_t>(H);
  for (int n = n_begin; n < n_end; n += kApplyRows) {
    uint2 pu[kApplyRows], pg[kApplyRows], ph[kApplyRows];
    float4 st[kApplyRows], rsm[kApplyRows];
#pragma unroll
    for (int i = 0; i < kApplyRows; ++i) {
      if (n + i < n_end) {
        const int64_t row = row0 + n + i;
        pu[i] = __ldcs(reinterpret_cast<const uint2*>(Z + row * zstride + c0));
        pg[i] = __ldcs(reinterpret_cast<const uint2*>(Z + row * zstride + H + c0));
        ph[i] = __ldcs(reinterpret_cast<const uint2*>(dHl + row * H + c0));
        st[i] = stats[row];
        rsm[i] = rowsum[row];
      }
    }
#pragma unroll
    for (int i = 0; i < kApplyRows; ++i) {
      if (n + i < n_end) {
        const int64_t row = row0 + n + i;
        float u[4], g[4], hv[4], du[4], dg[4];
        unpack4(pu[i], u);
        unpack4(pg[i], g);
        unpack4(ph[i], hv);
        const float m1u = rsm[i].x * inv_h, m2u = rsm[i].y * inv_h;
        const float m1g = rsm[i].z * inv_h, m2g = rsm[i].w * inv_h;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float xu = (u[e] - st[i].x) * st[i].y, xg = (g[e] - st[i].z) * st[i].w;
          const float a = fmaf(xu, wx[e], cx[e]), sv = fmaf(xg, wg[e], cg[e]);
          const float sg = sigmoid_fast(sv);
          const float da = hv[e] * (sv * sg);
          const float ds = hv[e] * a * fmaf(sv * sg, 1.0f - sg, sg);
          du[e] = st[i].y * (fmaf(da, wx[e], -m1u) - xu * m2u);
          dg[e] = st[i].w * (fmaf(ds, wg[e], -m1g) - xg * m2g);
          s_du[e] += du[e];
          s_dg[e] += dg[e];
          s_gx[e] = fmaf(da, xu, s_gx[e]);
          s_bx[e] += da;
          s_gg[e] = fmaf(ds, xg, s_gg[e]);
          s_bg[e] += ds;
        }
        __stcs(reinterpret_cast<uint2*>(dZ + row * zstride + c0), pack4(du));
        __stcs(reinterpret_cast<uint2*>(dZ + row * zstride + H + c0), pack4(dg));
      }
    }
  }
  // part[t][rs][q][c], q: dU, dG, da*x_u, da, ds*x_g, ds
  float* pp = part + (static_cast<int64_t>(t) * nsplit + rs) * 6 * H + c0;
  *reinterpret_cast<float4*>(pp + 0 * static_cast<int64_t>(H)) = make_float4(s_du[0], s_du[1], s_du[2], s_du[3]);
  *reinterpret_cast<float4*>(pp + 1 * static_cast<int64_t>(H)) = make_float4(s_dg[0], s_dg[1], s_dg[2], s_dg[3]);
  *reinterpret_cast<float4*>(pp + 2 * static_cast<int64_t>(H)) = make_float4(s_gx[0], s_gx[1], s_gx[2], s_gx[3]);
  *reinterpret_cast<float4*>(pp + 3 * static_cast<int64_t>(H)) = make_float4(s_bx[0], s_bx[1], s_bx[2], s_bx[3]);
  *reinterpret_cast<float4*>(pp + 4 * static_cast<int64_t>(H)) = make_float4(s_gg[0], s_gg[1], s_gg[2], s_gg[3]);
  *reinterpret_cast<float4*>(pp + 5 * static_cast<int64_t>(H)) = make_float4(s_bg[0], s_bg[1], s_bg[2], s_bg[3]);
}

// db1 [T, 2H] and the norm gradients [P, H] from the partials, summed in a
// fixed order (row splits, then the rank's slices): reruns are bit-identical.
__global__ void grad_reduce_kernel(const float* __restrict__ part, __nv_bfloat16* __restrict__ d_b1,
                                   __nv_bfloat16* __restrict__ d_nx_w, __nv_bfloat16* __restrict__ d_nx_b,
                                   __nv_bfloat16* __restrict__ d_ng_w, __nv_bfloat16* __restrict__ d_ng_b, int P,
                                   int L, int H, int nsplit, const uint32_t* err) {
  if (ld_volatile_u32(err) != 0u) return;
  const int T = P * L;
  const int64_t n_b1 = static_cast<int64_t>(T) * 2 * H;
  const int64_t n_norm = static_cast<int64_t>(P) * 4 * H;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n_b1 + n_norm;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    if (i < n_b1) {
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
      float s = 0.0f;
      for (int l = 0; l < L; ++l)
        for (int k = 0; k < nsplit; ++k)
          s += part[((static_cast<int64_t>(r * L + l) * nsplit + k) * 6 + 2 + q) * H + c];
      __nv_bfloat16* out = q == 0 ? d_nx_w : q == 1 ? d_nx_b : q == 2 ? d_ng_w : d_ng_b;
      out[static_cast<int64_t>(r) * H + c] = __float2bfloat16_rn(s);
    }
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
  const int nvec = H / 8;
  // VPT vectors per thread, at most 512 threads
  const int vpt = nvec <= 512 ? 1 : nvec <= 1024 ? 2 : nvec <= 2048 ? 4 : 0;
  if (vpt == 0) return cudaErrorInvalidValue;
  int threads = (nvec + vpt - 1) / vpt;
  threads = ((threads + 31) / 32) * 32;
  auto run = [&](auto kern) {
    const int grid = grid_for(dev, reinterpret_cast<const void*>(kern), threads, 0, rows);
    kern<<<grid, threads, 0, s>>>(static_cast<const __nv_bfloat16*>(Z), static_cast<const float4*>(stats),
                                  static_cast<const __nv_bfloat16*>(dHl), static_cast<const __nv_bfloat16*>(nx_w),
                                  static_cast<const __nv_bfloat16*>(nx_b), static_cast<const __nv_bfloat16*>(ng_w),
                                  static_cast<const __nv_bfloat16*>(ng_b), static_cast<float4*>(rowsum), rows, M, L,
                                  H, dev.err);
    return cudaGetLastError();
  };
  if (vpt == 1) return run(ln_gate_bwd_rowsum_kernel<1>);
  if (vpt == 2) return run(ln_gate_bwd_rowsum_kernel<2>);
  return run(ln_gate_bwd_rowsum_kernel<4>);
}

int ffn_bwd_row_splits(int T, int M) {
  // enough (t, column block, row range) items to fill the GPU several times over
  int splits = (2048 + T - 1) / T;
  const int cap = (M + 63) / 64;
  if (splits > cap) splits = cap;
  return splits < 1 ? 1 : splits;
}

cudaError_t launch_ln_gate_bwd_apply(const void* Z, const void* stats, const void* rowsum, const void* dHl,
                                     const void* nx_w, const void* nx_b, const void* ng_w, const void* ng_b, void* dZ,
                                     float* part, int T, int M, int L, int H, int nsplit, const DeviceInfo& dev,
                                     cudaStream_t s) {
  // balanced column blocks of at most 1024 columns (256 threads x 4 columns)
  const int nblk = (H + 1023) / 1024;
  int cols = (H + nblk - 1) / nblk;
  cols = ((cols + 4 * 32 - 1) / (4 * 32)) * (4 * 32);
  const int threads = cols / kApplyVec;
  dim3 grid(nblk, T, nsplit);
  ln_gate_bwd_apply_kernel<<<grid, threads, 0, s>>>(
      static_cast<const __nv_bfloat16*>(Z), static_cast<const float4*>(stats), static_cast<const float4*>(rowsum),
      static_cast<const __nv_bfloat16*>(dHl), static_cast<const __nv_bfloat16*>(nx_w),
      static_cast<const __nv_bfloat16*>(nx_b), static_cast<const __nv_bfloat16*>(ng_w),
      static_cast<const __nv_bfloat16*>(ng_b), static_cast<__nv_bfloat16*>(dZ), part, M, L, H, cols, dev.err);
  return cudaGetLastError();
}

cudaError_t launch_grad_reduce(const float* part, void* d_b1, void* d_nx_w, void* d_nx_b, void* d_ng_w, void* d_ng_b,
                               int P, int L, int H, int nsplit, const DeviceInfo& dev, cudaStream_t s) {
  const int64_t n = static_cast<int64_t>(P) * L * 2 * H + static_cast<int64_t>(P) * 4 * H;
  int64_t blocks = (n + 255) / 256;
  if (blocks > 8 * dev.num_sms) blocks = 8 * dev.num_sms;
  grad_reduce_kernel<<<static_cast<int>(blocks), 256, 0, s>>>(
      part, static_cast<__nv_bfloat16*>(d_b1), static_cast<__nv_bfloat16*>(d_nx_w), static_cast<__nv_bfloat16*>(d_nx_b),
      static_cast<__nv_bfloat16*>(d_ng_w), static_cast<__nv_bfloat16*>(d_ng_b), P, L, H, nsplit, dev.err);
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
