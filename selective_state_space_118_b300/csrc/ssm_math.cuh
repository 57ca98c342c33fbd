// ssm_math.cuh -- the per-token arithmetic of the selective scan, shared by the
// prefill kernels and the decode kernel so that both perform the same fp32
// operations in the same order (explicit __f*_rn intrinsics: no contraction or
// reassociation by the compiler).
//
// One token of channel c (the layer of "【大模型】- Jamba 混合 SSM-Transformer",
// section "实现 > Mamba 层", with the read-out y = C h of the lesson's
// "Um SSM em uma pagina"):
//   pre = conv_b + w0 x[t-3] + w1 x[t-2] + w2 x[t-1] + w3 x[t]
//   u   = silu(pre);   dt = softplus(dt_raw);   dtu = dt * u
//   h_n = 2^(dt * A2_n) * h_n + dtu * B_n,      A2_n = -exp(A_log_n) * log2(e)
//   y   = (sum_n C_n h_n + D u) * silu(z)
// The 16 states of a channel are split over 4 lanes (4 states each, lanes
// g = lane & 3); the read-out sum is ((p0 + p2) + (p1 + p3)) over the lanes'
// partial sums p_g.
#pragma once
#include <cuda_bf16.h>

#include "ptx.cuh"

namespace mamba {

constexpr float kLog2e = 1.44269504088896340736f;
constexpr float kLn2 = 0.69314718055994530942f;

// ---------------------------------------------------------------- I/O types
__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T>
__device__ __forceinline__ T from_f32(float v);
template <>
__device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}

// ---------------------------------------------------------------- activations
// silu(v) = v / (1 + e^-v), the exponential as 2^(-v log2 e).
__device__ __forceinline__ float silu(float v) {
  const float e = ex2_approx(__fmul_rn(v, -kLog2e));
  return __fmul_rn(v, rcp_approx(__fadd_rn(1.0f, e)));
}

// softplus(v) = log(1 + e^v), and v itself above 20 (beta 1, threshold 20).
// Two regions of e = e^v:
//   e < 1/8:  log1p(e) = e * P(e), P a degree-5 polynomial fitted to
//             log1p(e)/e on [0, 1/8] by least squares (fit_log1p.py; max
//             relative error 9e-8 evaluated in fp32).  This keeps full
//             relative accuracy for the small dt of the layer, where
//             log2(1 + e) would lose it, and needs no reciprocal.
//   e >= 1/8: log2(1 + e) ln 2, with 1 + e >= 1.125, where the approximate
//             log2's absolute error stays ~1e-6 relative to the result.
// softplus() evaluates both and selects (straight-line code); the scan calls
// softplus_small() directly when a whole warp's values lie in the first
// region -- the same formula, hence the same bits.
__device__ __forceinline__ float softplus_e(float v) { return ex2_approx(__fmul_rn(v, kLog2e)); }

__device__ __forceinline__ float softplus_small(float e) {
  float p = __fmaf_rn(e, -0.12255968898534775f, 0.19420583546161652f);
  p = __fmaf_rn(e, p, -0.24963703751564026f);
  p = __fmaf_rn(e, p, 0.3333229124546051f);
  p = __fmaf_rn(e, p, -0.49999988079071045f);
  p = __fmaf_rn(e, p, 1.0f);
  return __fmul_rn(e, p);
}

constexpr float kSoftplusSmallE = 0.125f;

__device__ __forceinline__ float softplus_large(float v, float e) {
  const float r = __fmul_rn(lg2_approx(__fadd_rn(1.0f, e)), kLn2);
  return v > 20.0f ? v : r;
}

__device__ __forceinline__ float softplus(float v) {
  const float e = softplus_e(v);
  return e < kSoftplusSmallE ? softplus_small(e) : softplus_large(v, e);
}

// ---------------------------------------------------------------- conv
// Causal depthwise cross-correlation of width 4: w.w multiplies the current
// input (PyTorch Conv1d with padding 3, first L outputs kept).
__device__ __forceinline__ float conv4(float4 w, float bias, float xm3, float xm2, float xm1,
                                       float x0) {
  float a = __fmaf_rn(w.x, xm3, bias);
  a = __fmaf_rn(w.y, xm2, a);
  a = __fmaf_rn(w.z, xm1, a);
  return __fmaf_rn(w.w, x0, a);
}

// A2 = A * log2(e) with A = -exp(A_log): the state decay exponent in base 2.
__device__ __forceinline__ float a2_from_log(float a_log) { return __fmul_rn(-expf(a_log), kLog2e); }

// ---------------------------------------------------------------- state
// Four states of one channel (h01 = states 4g, 4g+1; h23 = 4g+2, 4g+3).
struct State4 {
  float2 h01, h23;
};

// One token on four states; returns this lane's read-out partial
// (C0 h0 + C2 h2) + (C1 h1 + C3 h3).
__device__ __forceinline__ float state4_step(State4& s, float2 a01, float2 a23, float dt, float dtu,
                                             float4 B, float4 C) {
  const float2 dt2 = make_float2(dt, dt);
  const float2 x01 = __fmul2_rn(dt2, a01);
  const float2 x23 = __fmul2_rn(dt2, a23);
  const float2 dA01 = make_float2(ex2_approx(x01.x), ex2_approx(x01.y));
  const float2 dA23 = make_float2(ex2_approx(x23.x), ex2_approx(x23.y));
  const float2 u2 = make_float2(dtu, dtu);
  const float2 b01 = __fmul2_rn(u2, make_float2(B.x, B.y));
  const float2 b23 = __fmul2_rn(u2, make_float2(B.z, B.w));
  s.h01 = __ffma2_rn(dA01, s.h01, b01);
  s.h23 = __ffma2_rn(dA23, s.h23, b23);
  float2 p = __fmul2_rn(make_float2(C.x, C.y), s.h01);
  p = __ffma2_rn(make_float2(C.z, C.w), s.h23, p);
  return __fadd_rn(p.x, p.y);
}

// State update without the read-out (the chunk-summary pass).
__device__ __forceinline__ void state4_advance(State4& s, float2 a01, float2 a23, float dt, float dtu,
                                               float4 B) {
  const float2 dt2 = make_float2(dt, dt);
  const float2 x01 = __fmul2_rn(dt2, a01);
  const float2 x23 = __fmul2_rn(dt2, a23);
  const float2 dA01 = make_float2(ex2_approx(x01.x), ex2_approx(x01.y));
  const float2 dA23 = make_float2(ex2_approx(x23.x), ex2_approx(x23.y));
  const float2 u2 = make_float2(dtu, dtu);
  s.h01 = __ffma2_rn(dA01, s.h01, __fmul2_rn(u2, make_float2(B.x, B.y)));
  s.h23 = __ffma2_rn(dA23, s.h23, __fmul2_rn(u2, make_float2(B.z, B.w)));
}

// Sum of the four lanes' partials of one channel, ((p0 + p2) + (p1 + p3)),
// returned on all four lanes.
__device__ __forceinline__ float group4_sum(float p) {
  p = __fadd_rn(p, __shfl_xor_sync(0xffffffffu, p, 2));
  return __fadd_rn(p, __shfl_xor_sync(0xffffffffu, p, 1));
}

// Four tokens at once: lane g holds its partials p[0..3] of tokens t0..t0+3
// and receives the full sum of token t0 + g, in the same association as
// group4_sum.
__device__ __forceinline__ float group4_reduce_scatter(const float p[4], int g) {
  const bool hi = (g & 2) != 0;
  const float send0 = hi ? p[0] : p[2];
  const float send1 = hi ? p[1] : p[3];
  const float keep0 = hi ? p[2] : p[0];
  const float keep1 = hi ? p[3] : p[1];
  const float q0 = __fadd_rn(keep0, __shfl_xor_sync(0xffffffffu, send0, 2));
  const float q1 = __fadd_rn(keep1, __shfl_xor_sync(0xffffffffu, send1, 2));
  const bool lo = (g & 1) != 0;
  const float keep = lo ? q1 : q0;
  const float send = lo ? q0 : q1;
  return __fadd_rn(keep, __shfl_xor_sync(0xffffffffu, send, 1));
}

// y = (S + D u) * gz with gz = silu(z)
__device__ __forceinline__ float gate_out(float S, float Dc, float u, float gz) {
  return __fmul_rn(__fmaf_rn(Dc, u, S), gz);
}

}  // namespace mamba
