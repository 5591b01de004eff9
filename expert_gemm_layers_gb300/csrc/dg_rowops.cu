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

__device__ __forceinline__ void load4_stream(const __nv_bfloat16* p, float (&f)[4]) {
  const uint2 v = __ldcs(reinterpret_cast<const uint2*>(p));
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
// One CTA per row (grid-stride).  Thread i holds 8-column vectors
// i, i + blockDim, ... of U and G in registers: mean, then the centred
// second moment (two passes, no cancellation), then the affine and the gate.

template <int VPT>
__global__ void __launch_bounds__(512) ln_gate_fwd_kernel(
    const __nv_bfloat16* __restrict__ Z, const __nv_bfloat16* __restrict__ gx, const __nv_bfloat16* __restrict__ bx,
    const __nv_bfloat16* __restrict__ gg, const __nv_bfloat16* __restrict__ bg, __nv_bfloat16* __restrict__ Hl,
    float4* __restrict__ stats, int64_t rows, int M, int L, int H, float eps, const uint32_t* err) {
  __shared__ float sm[2][kMaxRowWarps][4];
  if (block_aborted(err)) return;
  const int nvec = H >> 3;
  const int nt = blockDim.x;
  const float inv_h = 1.0f / static_cast<float>(H);
  for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
    const int r = static_cast<int>(row / M) / L;
    const __nv_bfloat16* zu = Z + row * (2 * static_cast<int64_t>(H));
    const __nv_bfloat16* zg = zu + H;
    float u[VPT][8], g[VPT][8];
    float s[2] = {0.0f, 0.0f};
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
      const int v = threadIdx.x + nt * j;
      if (v < nvec) {
        load8_stream(zu + 8 * v, u[j]);
        load8_stream(zg + 8 * v, g[j]);
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) u[j][e] = g[j][e] = 0.0f;
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        s[0] += u[j][e];
        s[1] += g[j][e];
      }
    }
    block_sum<2>(s, sm, 0);
    const float mu_u = s[0] * inv_h, mu_g = s[1] * inv_h;
    float q[2] = {0.0f, 0.0f};
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
      if (threadIdx.x + nt * j < nvec) {
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float du = u[j][e] - mu_u, dg = g[j][e] - mu_g;
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
      const int v = threadIdx.x + nt * j;
      if (v < nvec) {
        float wx[8], cx[8], wg[8], cg[8], h[8];
        const int64_t po = static_cast<int64_t>(r) * H + 8 * v;
        load8(gx + po, wx);
        load8(bx + po, cx);
        load8(gg + po, wg);
        load8(bg + po, cg);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float a = (u[j][e] - mu_u) * rs_u * wx[e] + cx[e];
          const float sg = (g[j][e] - mu_g) * rs_g * wg[e] + cg[e];
          h[e] = a * (sg * sigmoid_f(sg));
        }
        store8(hrow + 8 * v, h);
      }
    }
    if (threadIdx.x == 0) stats[row] = make_float4(mu_u, rs_u, mu_g, rs_g);
  }
}

// ------------------------------------------------------------------ backward
//
// One CTA per work item (t, chunk) handles rows [chunk*R, chunk*R + R) of
// token position t.  Per row it recomputes x_hat, the affines and the gate
// from Z and the saved statistics, forms da, ds, the two row reductions of
// the LayerNorm backward and writes dZ.  Column partials of
// (dU, dG, da*xu, da, ds*xg, ds) accumulate in shared memory (each thread
// owns fixed 4-column vectors, so no atomics) and are written once per item.

template <int VPT4>
__global__ void __launch_bounds__(512) ln_gate_bwd_kernel(
    const __nv_bfloat16* __restrict__ Z, const float4* __restrict__ stats, const __nv_bfloat16* __restrict__ dHl,
    const __nv_bfloat16* __restrict__ gx, const __nv_bfloat16* __restrict__ bx, const __nv_bfloat16* __restrict__ gg,
    const __nv_bfloat16* __restrict__ bg, __nv_bfloat16* __restrict__ dZ, float* __restrict__ part, int T, int M,
    int L, int H, int nchunk, const uint32_t* err) {
  extern __shared__ float4 acc4[];  // [6][H/4]
  __shared__ float sm[2][kMaxRowWarps][4];
  if (block_aborted(err)) return;
  const int nv4 = H >> 2;
  const int nt = blockDim.x;
  const float inv_h = 1.0f / static_cast<float>(H);
  const int R = (M + nchunk - 1) / nchunk;
  const int items = T * nchunk;
  for (int item = blockIdx.x; item < items; item += gridDim.x) {
    const int t = item / nchunk, chunk = item - t * nchunk;
    const int r = t / L;
    const int64_t pr = static_cast<int64_t>(r) * H;
    for (int i = threadIdx.x; i < 6 * nv4; i += nt) acc4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    __syncthreads();
    const int n_end = min(M, (chunk + 1) * R);
    int slot = 0;
    for (int n = chunk * R; n < n_end; ++n) {
      const int64_t row = static_cast<int64_t>(t) * M + n;
      const float4 st = stats[row];
      const __nv_bfloat16* zu = Z + row * (2 * static_cast<int64_t>(H));
      const __nv_bfloat16* zg = zu + H;
      const __nv_bfloat16* dh = dHl + row * static_cast<int64_t>(H);
      float xu[VPT4][4], xg[VPT4][4], da[VPT4][4], ds[VPT4][4];
      float rsum[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int j = 0; j < VPT4; ++j) {
        const int v = threadIdx.x + nt * j;
        if (v < nv4) {
          float uv[4], gv[4], hv[4], wx[4], cx[4], wg[4], cg[4];
          load4_stream(zu + 4 * v, uv);
          load4_stream(zg + 4 * v, gv);
          load4_stream(dh + 4 * v, hv);
          load4(gx + pr + 4 * v, wx);
          load4(bx + pr + 4 * v, cx);
          load4(gg + pr + 4 * v, wg);
          load4(bg + pr + 4 * v, cg);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float x_u = (uv[e] - st.x) * st.y;
            const float x_g = (gv[e] - st.z) * st.w;
            const float a = x_u * wx[e] + cx[e];
            const float s = x_g * wg[e] + cg[e];
            const float sg = sigmoid_f(s);
            const float d_a = hv[e] * (s * sg);
            const float d_s = hv[e] * a * (sg * (1.0f + s * (1.0f - sg)));
            xu[j][e] = x_u;
            xg[j][e] = x_g;
            da[j][e] = d_a;
            ds[j][e] = d_s;
            const float dxu = d_a * wx[e], dxg = d_s * wg[e];
            rsum[0] += dxu;
            rsum[1] += dxu * x_u;
            rsum[2] += dxg;
            rsum[3] += dxg * x_g;
          }
        } else {
#pragma unroll
          for (int e = 0; e < 4; ++e) xu[j][e] = xg[j][e] = da[j][e] = ds[j][e] = 0.0f;
        }
      }
      block_sum<4>(rsum, sm, slot);
      slot ^= 1;
      const float m1u = rsum[0] * inv_h, m2u = rsum[1] * inv_h;
      const float m1g = rsum[2] * inv_h, m2g = rsum[3] * inv_h;
      __nv_bfloat16* dzu = dZ + row * (2 * static_cast<int64_t>(H));
      __nv_bfloat16* dzg = dzu + H;
#pragma unroll
      for (int j = 0; j < VPT4; ++j) {
        const int v = threadIdx.x + nt * j;
        if (v < nv4) {
          float wx[4], wg[4], du[4], dg[4];
          load4(gx + pr + 4 * v, wx);
          load4(gg + pr + 4 * v, wg);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            du[e] = st.y * (da[j][e] * wx[e] - m1u - xu[j][e] * m2u);
            dg[e] = st.w * (ds[j][e] * wg[e] - m1g - xg[j][e] * m2g);
          }
          uint2 o;
          o.x = pack_bf16x2(du[0], du[1]);
          o.y = pack_bf16x2(du[2], du[3]);
          *reinterpret_cast<uint2*>(dzu + 4 * v) = o;
          o.x = pack_bf16x2(dg[0], dg[1]);
          o.y = pack_bf16x2(dg[2], dg[3]);
          *reinterpret_cast<uint2*>(dzg + 4 * v) = o;
          float4* a0 = acc4 + v;
          float4 q;
          q = a0[0 * nv4]; q.x += du[0]; q.y += du[1]; q.z += du[2]; q.w += du[3]; a0[0 * nv4] = q;
          q = a0[1 * nv4]; q.x += dg[0]; q.y += dg[1]; q.z += dg[2]; q.w += dg[3]; a0[1 * nv4] = q;
          q = a0[2 * nv4];
          q.x += da[j][0] * xu[j][0]; q.y += da[j][1] * xu[j][1]; q.z += da[j][2] * xu[j][2]; q.w += da[j][3] * xu[j][3];
          a0[2 * nv4] = q;
          q = a0[3 * nv4]; q.x += da[j][0]; q.y += da[j][1]; q.z += da[j][2]; q.w += da[j][3]; a0[3 * nv4] = q;
          q = a0[4 * nv4];
          q.x += ds[j][0] * xg[j][0]; q.y += ds[j][1] * xg[j][1]; q.z += ds[j][2] * xg[j][2]; q.w += ds[j][3] * xg[j][3];
          a0[4 * nv4] = q;
          q = a0[5 * nv4]; q.x += ds[j][0]; q.y += ds[j][1]; q.z += ds[j][2]; q.w += ds[j][3]; a0[5 * nv4] = q;
        }
      }
    }
    __syncthreads();
    float4* dst = reinterpret_cast<float4*>(part + static_cast<int64_t>(item) * 6 * H);
    for (int i = threadIdx.x; i < 6 * nv4; i += nt) dst[i] = acc4[i];
    __syncthreads();
  }
}

// db1[t, c] (c < 2H) and the four norm gradients [P, H], summing the
// partials in a fixed order (chunks, then slices), so reruns are bit-identical.
__global__ void reduce_partials_kernel(const float* __restrict__ part, __nv_bfloat16* __restrict__ d_b1,
                                       __nv_bfloat16* __restrict__ d_nx_w, __nv_bfloat16* __restrict__ d_nx_b,
                                       __nv_bfloat16* __restrict__ d_ng_w, __nv_bfloat16* __restrict__ d_ng_b, int P,
                                       int L, int H, int nchunk, const uint32_t* err) {
  if (ld_volatile_u32(err) != 0u) return;
  const int T = P * L;
  const int64_t n_b1 = static_cast<int64_t>(T) * 2 * H;
  const int64_t n_norm = static_cast<int64_t>(P) * 4 * H;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n_b1 + n_norm;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    if (i < n_b1) {
      const int t = static_cast<int>(i / (2 * H));
      const int c2 = static_cast<int>(i - static_cast<int64_t>(t) * 2 * H);
      const int which = c2 >= H ? 1 : 0;
      const int c = c2 - which * H;
      float s = 0.0f;
      for (int k = 0; k < nchunk; ++k)
        s += part[((static_cast<int64_t>(t) * nchunk + k) * 6 + which) * H + c];
      d_b1[i] = __float2bfloat16_rn(s);
    } else {
      const int64_t j = i - n_b1;
      const int r = static_cast<int>(j / (4 * H));
      const int q = static_cast<int>((j / H) % 4);  // 0: nx_w, 1: nx_b, 2: ng_w, 3: ng_b
      const int c = static_cast<int>(j % H);
      float s = 0.0f;
      for (int l = 0; l < L; ++l)
        for (int k = 0; k < nchunk; ++k)
          s += part[((static_cast<int64_t>(r * L + l) * nchunk + k) * 6 + 2 + q) * H + c];
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

int ffn_bwd_chunks(int T, int M) {
  int want = (1024 + T - 1) / T;
  int cap = (M + 31) / 32;
  if (want > cap) want = cap;
  return want < 1 ? 1 : want;
}

// Smallest VPT in {1,2,4,8} whose block (rounded to warps) has at most 512 threads.
static bool row_block(int nvec, int* vpt, int* threads) {
  for (int v = 1; v <= 8; v *= 2) {
    int t = (nvec + v - 1) / v;
    t = ((t + 31) / 32) * 32;
    if (t <= 512) {
      *vpt = v;
      *threads = t < 32 ? 32 : t;
      return true;
    }
  }
  return false;
}

cudaError_t launch_ln_gate_fwd(const void* Z, const void* nx_w, const void* nx_b, const void* ng_w,
                               const void* ng_b, void* Hl, void* stats, int64_t rows, int M, int L, int H,
                               float eps, const DeviceInfo& dev, cudaStream_t s) {
  int vpt = 0, threads = 0;
  if (!row_block(H / 8, &vpt, &threads)) return cudaErrorInvalidValue;
  auto run = [&](auto kern) {
    const int grid = grid_for(dev, reinterpret_cast<const void*>(kern), threads, 0, rows);
    kern<<<grid, threads, 0, s>>>(static_cast<const __nv_bfloat16*>(Z), static_cast<const __nv_bfloat16*>(nx_w),
                                  static_cast<const __nv_bfloat16*>(nx_b), static_cast<const __nv_bfloat16*>(ng_w),
                                  static_cast<const __nv_bfloat16*>(ng_b), static_cast<__nv_bfloat16*>(Hl),
                                  static_cast<float4*>(stats), rows, M, L, H, eps, dev.err);
    return cudaGetLastError();
  };
  if (vpt == 1) return run(ln_gate_fwd_kernel<1>);
  if (vpt == 2) return run(ln_gate_fwd_kernel<2>);
  if (vpt == 4) return run(ln_gate_fwd_kernel<4>);
  return run(ln_gate_fwd_kernel<8>);
}

size_t ln_gate_bwd_smem(int H) { return static_cast<size_t>(6) * H * sizeof(float); }

cudaError_t launch_ln_gate_bwd(const void* Z, const void* stats, const void* dHl, const void* nx_w,
                               const void* nx_b, const void* ng_w, const void* ng_b, void* dZ, float* part,
                               int T, int M, int L, int H, int nchunk, const DeviceInfo& dev, cudaStream_t s) {
  int vpt = 0, threads = 0;
  if (!row_block(H / 4, &vpt, &threads)) return cudaErrorInvalidValue;
  const size_t smem = ln_gate_bwd_smem(H);
  auto run = [&](auto kern) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    const int grid = grid_for(dev, reinterpret_cast<const void*>(kern), threads, smem,
                              static_cast<int64_t>(T) * nchunk);
    kern<<<grid, threads, smem, s>>>(
        static_cast<const __nv_bfloat16*>(Z), static_cast<const float4*>(stats),
        static_cast<const __nv_bfloat16*>(dHl), static_cast<const __nv_bfloat16*>(nx_w),
        static_cast<const __nv_bfloat16*>(nx_b), static_cast<const __nv_bfloat16*>(ng_w),
        static_cast<const __nv_bfloat16*>(ng_b), static_cast<__nv_bfloat16*>(dZ), part, T, M, L, H, nchunk, dev.err);
    return cudaGetLastError();
  };
  if (vpt == 1) return run(ln_gate_bwd_kernel<1>);
  if (vpt == 2) return run(ln_gate_bwd_kernel<2>);
  if (vpt == 4) return run(ln_gate_bwd_kernel<4>);
  return run(ln_gate_bwd_kernel<8>);
}

cudaError_t launch_reduce_partials(const float* part, void* d_b1, void* d_nx_w, void* d_nx_b, void* d_ng_w,
                                   void* d_ng_b, int P, int L, int H, int nchunk, const DeviceInfo& dev,
                                   cudaStream_t s) {
  const int64_t n = static_cast<int64_t>(P) * L * 2 * H + static_cast<int64_t>(P) * 4 * H;
  int64_t blocks = (n + 255) / 256;
  if (blocks > 8 * dev.num_sms) blocks = 8 * dev.num_sms;
  reduce_partials_kernel<<<static_cast<int>(blocks), 256, 0, s>>>(
      part, static_cast<__nv_bfloat16*>(d_b1), static_cast<__nv_bfloat16*>(d_nx_w),
      static_cast<__nv_bfloat16*>(d_nx_b), static_cast<__nv_bfloat16*>(d_ng_w), static_cast<__nv_bfloat16*>(d_ng_b), P,
      L, H, nchunk, dev.err);
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
