// Elementwise math of the LayerNorm-gated SiLU, shared by the row kernels
// and the GEMM epilogues: packed two-lane fp32 arithmetic (the .f32x2 forms
// of fma/mul/add issue two lanes per instruction) and the gate's forward
// quantities recomputed from Z.
#pragma once

#include "dg_ptx.cuh"

namespace dg {

// sigmoid(x) = (1 + tanh(x/2)) / 2, with the hardware tanh approximation
// (tanh.approx.f32, relative error about 2^-11): one MUFU operation instead of
// an exponential and a division.
static __device__ __forceinline__ float tanh_fast(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

static __device__ __forceinline__ float sigmoid_fast(float x) { return fmaf(0.5f, tanh_fast(0.5f * x), 0.5f); }

// silu(x) = x * sigmoid(x) = h + h * tanh(h) with h = x/2.
static __device__ __forceinline__ float silu_fast(float x) {
  const float h = 0.5f * x;
  return fmaf(h, tanh_fast(h), h);
}


// Packed two-lane fp32 arithmetic (fma/mul .f32x2): one issue slot for two lanes.
static __device__ __forceinline__ unsigned long long f2u(float2 a) { return *reinterpret_cast<unsigned long long*>(&a); }
static __device__ __forceinline__ float2 u2f(unsigned long long a) { return *reinterpret_cast<float2*>(&a); }
static __device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  unsigned long long d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(f2u(a)), "l"(f2u(b)), "l"(f2u(c)));
  return u2f(d);
}
static __device__ __forceinline__ float2 mul2(float2 a, float2 b) {
  unsigned long long d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(f2u(a)), "l"(f2u(b)));
  return u2f(d);
}
static __device__ __forceinline__ float2 add2(float2 a, float2 b) {
  unsigned long long d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(f2u(a)), "l"(f2u(b)));
  return u2f(d);
}
static __device__ __forceinline__ float2 sub2(float2 a, float2 b) {
  unsigned long long d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(f2u(a)), "l"(f2u(b)));
  return u2f(d);
}
static __device__ __forceinline__ float2 splat2(float x) { return make_float2(x, x); }


// Forward quantities of the gate at one column pair, recomputed from Z:
// x_u, x_g (normalised), a = LN_x(U), s = LN_g(G), q = silu(s), silu'(s).
struct GatePair {
  float2 xu, xg, a, q, dsil;
};

static __device__ __forceinline__ GatePair gate_pair(float2 u, float2 g, float2 rsu, float2 cu, float2 rsg, float2 cg_,
                                              float2 wx, float2 cx, float2 wg, float2 cgb) {
  GatePair r;
  r.xu = fma2(u, rsu, cu);
  r.xg = fma2(g, rsg, cg_);
  r.a = fma2(r.xu, wx, cx);
  const float2 sv = fma2(r.xg, wg, cgb);
  const float2 h = mul2(sv, splat2(0.5f));
  const float2 sig = fma2(make_float2(tanh_fast(h.x), tanh_fast(h.y)), splat2(0.5f), splat2(0.5f));
  r.q = mul2(sv, sig);
  // silu'(s) = sig + s*sig*(1 - sig) = q*(1 - sig) + sig
  r.dsil = fma2(r.q, fma2(sig, splat2(-1.0f), splat2(1.0f)), sig);
  return r;
}


// The same quantities with the gate norm's affine pre-halved (wg2 = gg/2,
// cg2 = bg/2), so that h = s/2 comes out of one fma.  With t = tanh(h):
// q = silu(s) = h*(1 + t), and silu'(s) = sig*(1 + s*(1 - sig)) with
// sig = (1 + t)/2 gives dsil2 = 2*silu'(s) = (1 + t)*w, w = 1 + h*(1 - t),
// which needs the single constant 1 (a register pair the loops keep).
// Callers use dsil2 with the halved gg, so d*a*dsil2*wg2 = d*a*silu'(s)*gg.
struct GatePairH {
  float2 xu, xg, a, q, dsil2;
};

static __device__ __forceinline__ GatePairH gate_pair_h(float2 u, float2 g, float2 rsu, float2 cu, float2 rsg,
                                                       float2 cg_, float2 wx, float2 cx, float2 wg2, float2 cg2) {
  GatePairH r;
  r.xu = fma2(u, rsu, cu);
  r.xg = fma2(g, rsg, cg_);
  r.a = fma2(r.xu, wx, cx);
  const float2 h = fma2(r.xg, wg2, cg2);
  const float2 t = make_float2(tanh_fast(h.x), tanh_fast(h.y));
  r.q = fma2(h, t, h);
  const float2 one = splat2(1.0f);
  const float2 w = fma2(h, sub2(one, t), one);
  r.dsil2 = fma2(t, w, w);
  return r;
}

// Per-row coefficients of the backward, stored by the row-sum pass as two
// float4: (rstd_u, -mean_u*rstd_u, rstd_g, -mean_g*rstd_g) and
// (-mean(dx_u), -mean(dx_u*x_u), -mean(dx_g), -mean(dx_g*x_g)), the means
// over the row's H columns.
static __device__ __forceinline__ void store_row_coef(float4* rc, float4 stats, float4 sums, float inv_h) {
  rc[0] = make_float4(stats.y, -stats.x * stats.y, stats.w, -stats.z * stats.w);
  rc[1] = make_float4(-sums.x * inv_h, -sums.y * inv_h, -sums.z * inv_h, -sums.w * inv_h);
}


// bf16x2-packed affine parameters of one 8-column vector (held for all rows).
struct Affine8 {
  uint4 wx, cx, wg, cg;
};

static __device__ __forceinline__ Affine8 load_affine8(const __nv_bfloat16* gx, const __nv_bfloat16* bx,
                                                const __nv_bfloat16* gg, const __nv_bfloat16* bg, int64_t off) {
  Affine8 a;
  a.wx = __ldg(reinterpret_cast<const uint4*>(gx + off));
  a.cx = __ldg(reinterpret_cast<const uint4*>(bx + off));
  a.wg = __ldg(reinterpret_cast<const uint4*>(gg + off));
  a.cg = __ldg(reinterpret_cast<const uint4*>(bg + off));
  return a;
}

// Affine parameters of one 8-column vector as four fp32 pairs each.
struct AffineF {
  float2 wx[4], cx[4], wg[4], cg[4];
};

static __device__ __forceinline__ AffineF load_affine_f(const __nv_bfloat16* gx, const __nv_bfloat16* bx,
                                                 const __nv_bfloat16* gg, const __nv_bfloat16* bg, int64_t off) {
  const Affine8 a = load_affine8(gx, bx, gg, bg, off);
  const uint32_t w0[4] = {a.wx.x, a.wx.y, a.wx.z, a.wx.w}, w1[4] = {a.cx.x, a.cx.y, a.cx.z, a.cx.w};
  const uint32_t w2[4] = {a.wg.x, a.wg.y, a.wg.z, a.wg.w}, w3[4] = {a.cg.x, a.cg.y, a.cg.z, a.cg.w};
  AffineF f;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    f.wx[e] = unpack_bf16x2(w0[e]);
    f.cx[e] = unpack_bf16x2(w1[e]);
    f.wg[e] = unpack_bf16x2(w2[e]);
    f.cg[e] = unpack_bf16x2(w3[e]);
  }
  return f;
}

// The gate norm's affine halved (exact), for gate_pair_h.
static __device__ __forceinline__ void halve_gate_affine(AffineF& f) {
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    f.wg[e] = mul2(f.wg[e], splat2(0.5f));
    f.cg[e] = mul2(f.cg[e], splat2(0.5f));
  }
}

}  // namespace dg
