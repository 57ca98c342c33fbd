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
// The prefill kernels keep all 16 states of a channel in one lane, as 8
// float2 pairs (h[k] = states 2k, 2k+1) advanced with packed f32x2
// arithmetic; the decode kernel splits them over two lanes.  The read-out
// sum is fixed so that both layouts produce the same bits: two packed
// accumulation chains, p_lo over the pairs of states 0-7 and p_hi over those
// of states 8-15 (each one packed multiply, then three packed fmas in pair
// order), v = p_lo + p_hi (packed), and sum_n C_n h_n = v.x + v.y.
#pragma once
#include <cuda_bf16.h>

#include "ptx.cuh"

namespace mamba {

constexpr int kN = 16;  // d_state
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
//             relative error 1.2e-7 evaluated in fp32).  This keeps full
//             relative accuracy for the small dt of the layer, where
//             log2(1 + e) would lose it, and needs no reciprocal.
//   e >= 1/8: log2(1 + e) ln 2, with 1 + e >= 1.125, where the approximate
//             log2's absolute error stays ~1e-6 relative to the result.
// softplus() selects per value.  The scan kernels check a whole tile first
// and, when every value lies below kSoftplusSmallRaw (so that e < 1/8 for
// sure: 2^(-2.08 log2 e) = 0.12493), take softplus_small(softplus_e(v))
// directly -- the formula softplus() selects there, hence the same bits.
__device__ __forceinline__ float softplus_e(float v) { return ex2_approx(__fmul_rn(v, kLog2e)); }

// P evaluated in Estrin's scheme (depth 4 instead of Horner's 6):
// P = (1 + a1 e) + e^2 ((a2 + a3 e) + e^2 (a4 + a5 e)).
constexpr float kLp1 = -0.49999988079071045f;  // coefficients a1..a5 of P (fit_log1p.py)
constexpr float kLp2 = 0.3333229124546051f;
constexpr float kLp3 = -0.24963703751564026f;
constexpr float kLp4 = 0.19420583546161652f;
constexpr float kLp5 = -0.12255968898534775f;

__device__ __forceinline__ float softplus_small(float e) {
  const float e2 = __fmul_rn(e, e);
  const float q0 = __fmaf_rn(e, kLp1, 1.0f);
  const float q1 = __fmaf_rn(e, kLp3, kLp2);
  const float q2 = __fmaf_rn(e, kLp5, kLp4);
  const float p = __fmaf_rn(__fmaf_rn(q2, e2, q1), e2, q0);
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

constexpr float kSoftplusSmallRaw = -2.08f;

// softplus(v) for v < kSoftplusSmallRaw (the caller guarantees it).
__device__ __forceinline__ float softplus_small_raw(float v) { return softplus_small(softplus_e(v)); }

// The same three functions on two values at once with packed f32x2
// operations: each lane of a packed operation performs the scalar
// operation above, in the same order, so the results are the same bits.
__device__ __forceinline__ float2 silu_x2(float2 v) {
  const float2 m = __fmul2_rn(v, make_float2(-kLog2e, -kLog2e));
  const float2 d = __fadd2_rn(make_float2(1.0f, 1.0f), make_float2(ex2_approx(m.x), ex2_approx(m.y)));
  return __fmul2_rn(v, make_float2(rcp_approx(d.x), rcp_approx(d.y)));
}

// softplus of two raw values both below kSoftplusSmallRaw (the caller
// guarantees it): softplus_small(softplus_e(v)) on each.
__device__ __forceinline__ float2 softplus_small_raw_x2(float2 v) {
  const float2 m = __fmul2_rn(v, make_float2(kLog2e, kLog2e));
  const float2 e = make_float2(ex2_approx(m.x), ex2_approx(m.y));
  const float2 e2 = __fmul2_rn(e, e);
  const float2 q0 = __ffma2_rn(e, make_float2(kLp1, kLp1), make_float2(1.0f, 1.0f));
  const float2 q1 = __ffma2_rn(e, make_float2(kLp3, kLp3), make_float2(kLp2, kLp2));
  const float2 q2 = __ffma2_rn(e, make_float2(kLp5, kLp5), make_float2(kLp4, kLp4));
  const float2 p = __ffma2_rn(__ffma2_rn(q2, e2, q1), e2, q0);
  return __fmul2_rn(e, p);
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

// conv4 for two consecutive tokens t, t+1 (inputs x[t-3..t+1]).
__device__ __forceinline__ float2 conv4_x2(float4 w, float bias, float xm3, float xm2, float xm1, float x0,
                                           float x1) {
  float2 a = __ffma2_rn(make_float2(w.x, w.x), make_float2(xm3, xm2), make_float2(bias, bias));
  a = __ffma2_rn(make_float2(w.y, w.y), make_float2(xm2, xm1), a);
  a = __ffma2_rn(make_float2(w.z, w.z), make_float2(xm1, x0), a);
  return __ffma2_rn(make_float2(w.w, w.w), make_float2(x0, x1), a);
}

// gate_out for two tokens.
__device__ __forceinline__ float2 gate_out_x2(float2 S, float Dc, float2 u, float2 gz) {
  return __fmul2_rn(__ffma2_rn(make_float2(Dc, Dc), u, S), gz);
}

// ---------------------------------------------------------------- parameters
// A2 = A * log2(e) with A = -exp(A_log) = -2^(A_log log2 e): the state decay
// exponent in base 2.
__device__ __forceinline__ float a2_from_log(float a_log) {
  return __fmul_rn(-ex2_approx(__fmul_rn(a_log, kLog2e)), kLog2e);
}

// The per-channel constants one lane keeps in registers.
struct Channel {
  float2 a2[8];  // A2 of states (2k, 2k+1)
  float4 w;      // conv taps
  float bias;    // conv bias
  float Dc;      // skip weight
};

__device__ __forceinline__ void load_channel(Channel& ch, const float* __restrict__ A_log,
                                             const float* __restrict__ conv_w,
                                             const float* __restrict__ conv_b,
                                             const float* __restrict__ Dskip, int c) {
  const float4* al = reinterpret_cast<const float4*>(A_log + (size_t)c * kN);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float4 v = __ldg(al + q);
    ch.a2[2 * q] = make_float2(a2_from_log(v.x), a2_from_log(v.y));
    ch.a2[2 * q + 1] = make_float2(a2_from_log(v.z), a2_from_log(v.w));
  }
  ch.w = __ldg(reinterpret_cast<const float4*>(conv_w + (size_t)c * 4));
  ch.bias = conv_b ? __ldg(conv_b + c) : 0.0f;
  ch.Dc = __ldg(Dskip + c);
}

// ---------------------------------------------------------------- state
struct State16 {
  float2 h[8];  // states (2k, 2k+1)
};

__device__ __forceinline__ void state16_zero(State16& s) {
#pragma unroll
  for (int k = 0; k < 8; ++k) s.h[k] = make_float2(0.0f, 0.0f);
}

__device__ __forceinline__ void state16_load(State16& s, const float* p) {
  const float4* q = reinterpret_cast<const float4*>(p);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float4 v = q[k];
    s.h[2 * k] = make_float2(v.x, v.y);
    s.h[2 * k + 1] = make_float2(v.z, v.w);
  }
}

__device__ __forceinline__ void state16_store(const State16& s, float* p) {
  float4* q = reinterpret_cast<float4*>(p);
#pragma unroll
  for (int k = 0; k < 4; ++k)
    q[k] = make_float4(s.h[2 * k].x, s.h[2 * k].y, s.h[2 * k + 1].x, s.h[2 * k + 1].y);
}

// The state-independent half of one token's update: the decays 2^(dt A2) and
// the inputs dtu B of all 16 states.
struct Drive16 {
  float2 dA[8];
  float2 bu[8];
};

// From widened B/C rows in pair-quad layout: Q[k] = (B_2k, B_2k+1, C_2k,
// C_2k+1); only the B halves are used here.
__device__ __forceinline__ void drive16_q(Drive16& d, const float2 (&a2)[8], float dt, float dtu,
                                          const float4 (&Q)[8]) {
  const float2 d2 = make_float2(dt, dt);
  const float2 u2 = make_float2(dtu, dtu);
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const float2 x = __fmul2_rn(d2, a2[k]);
    d.dA[k] = make_float2(ex2_approx(x.x), ex2_approx(x.y));
    d.bu[k] = __fmul2_rn(u2, make_float2(Q[k].x, Q[k].y));
  }
}

// The state-dependent half: h <- dA h + bu.
__device__ __forceinline__ void state16_apply(State16& s, const Drive16& d) {
#pragma unroll
  for (int k = 0; k < 8; ++k) s.h[k] = __ffma2_rn(d.dA[k], s.h[k], d.bu[k]);
}

// Half of the read-out: the 8 states of pairs h[0..3] (C values C[0..1]) as
// one packed chain, p = C01 h01; p += C23 h23; p += C45 h45; p += C67 h67.
__device__ __forceinline__ float2 readout_half(const float2* h, const float4* C) {
  float2 p = __fmul2_rn(make_float2(C[0].x, C[0].y), h[0]);
  p = __ffma2_rn(make_float2(C[0].z, C[0].w), h[1], p);
  p = __ffma2_rn(make_float2(C[1].x, C[1].y), h[2], p);
  return __ffma2_rn(make_float2(C[1].z, C[1].w), h[3], p);
}

// The two halves combined: v = p_lo + p_hi, sum_n C_n h_n = v.x + v.y.
__device__ __forceinline__ float readout_join(float2 lo, float2 hi) {
  const float2 v = __fadd2_rn(lo, hi);
  return __fadd_rn(v.x, v.y);
}

// sum_n C_n h_n in the fixed order described at the top of the file.
__device__ __forceinline__ float state16_readout(const State16& s, const float4 (&C)[4]) {
  return readout_join(readout_half(&s.h[0], &C[0]), readout_half(&s.h[4], &C[2]));
}

// The same with C taken from pair quads (the C halves of Q[k]).
__device__ __forceinline__ float2 readout_half_q(const float2* h, const float4* Q) {
  float2 p = __fmul2_rn(make_float2(Q[0].z, Q[0].w), h[0]);
  p = __ffma2_rn(make_float2(Q[1].z, Q[1].w), h[1], p);
  p = __ffma2_rn(make_float2(Q[2].z, Q[2].w), h[2], p);
  return __ffma2_rn(make_float2(Q[3].z, Q[3].w), h[3], p);
}

__device__ __forceinline__ float state16_readout_q(const State16& s, const float4 (&Q)[8]) {
  return readout_join(readout_half_q(&s.h[0], &Q[0]), readout_half_q(&s.h[4], &Q[4]));
}

// Carry fold: h <- 2^(A2 S) h + hl, S the summed dt of a span of tokens and
// hl that span's end state from zero.
__device__ __forceinline__ void state16_fold(State16& s, const float2 (&a2)[8], float S,
                                             const State16& hl) {
  const float2 S2 = make_float2(S, S);
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const float2 x = __fmul2_rn(S2, a2[k]);
    s.h[k] = __ffma2_rn(make_float2(ex2_approx(x.x), ex2_approx(x.y)), s.h[k], hl.h[k]);
  }
}

// y = (S + D u) * gz with gz = silu(z)
__device__ __forceinline__ float gate_out(float S, float Dc, float u, float gz) {
  return __fmul_rn(__fmaf_rn(Dc, u, S), gz);
}

}  // namespace mamba
