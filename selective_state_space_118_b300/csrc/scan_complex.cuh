// scan_complex.cuh -- the complex-valued selective scan (the Mamba-3 state
// update of "Jamba -- SSM-Transformer Hibrido", section "Mamba-3: a linha de
// base de SSM puro em 2026", items 1 and 2).
//
// Per channel, 8 complex modes (16 fp32 numbers: the real scan's state size)
// with lambda_n = -exp(A_log[c,n]) + i theta[c,n].  One token:
//   u = silu(conv(x)), dt = softplus(dt_raw)      (as in the real scan)
//   alpha_n = exp(dt lambda_n) = 2^(dt A2_n) (cos(dt theta_n) + i sin(dt theta_n))
//   v_n = B_n u                                   (B_n complex: (re, im))
//   Euler:        h_n = alpha_n h_n + dt v_n
//   trapezoidal:  h_n = alpha_n (h_n + dt/2 vprev_n) + dt/2 v_n,  vprev = v
//   y = (Re(sum_n C_n h_n) + D u) silu(z)
// The approximate sine and cosine hold their error bound on [-pi, pi].  A
// token whose dt keeps every turn dt theta_n of the channel within it (dt <=
// pi / max |theta_n|, the common case) takes the angle as it is; any other
// takes it in whole turns first (t = dt theta_n / 2pi, reduced to
// [-1/2, 1/2] by subtracting the nearest integer).  So that a turn of many
// revolutions per token keeps its fraction to fp32 precision, theta / 2pi is
// then formed as two fp32 parts (hi + lo) and the product dt * hi carries its
// exact rounding error (an fma) into the fraction.
//
// Decomposition: as the real scan's main pass -- a CTA is one warp, lane i
// owns channel c0 + i with all 16 numbers of its state in registers, tiles of
// 16 tokens of x, z, dt_raw and the widened B/C rows arrive by TMA through a
// two-stage mbarrier ring.  The modes are advanced two at a time with packed
// fp32 pair arithmetic: the state is held as (Re, Im) pairs across modes 2q,
// 2q+1, and the widened row of a token holds, per mode pair q, the quads
// (Re B_2q, Re B_2q+1, Im B_2q, Im B_2q+1) and (Re C_2q, ..., Im C_2q+1).
//
// Chunked mode (batch 1 needs it to fill the GPU): three exact passes, no
// term dropped.  (1) Each chunk but the last runs the recurrence from a zero
// state (with the true state input of the token before it, which depends on
// the inputs only) and stores its end state hloc_j and its dt sum S_j; the
// end state of chunk j is then W_j h_in_j + hloc_j with W_j = exp(lambda S_j)
// (the product of the chunk's alphas).  (2) One thread per channel folds
// them in chunk order into the state entering every chunk.  (3) The main
// pass runs every chunk from its entering state.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>

#include <cstdint>

#include "params.h"
#include "ptx.cuh"
#include "scan_fwd.cuh"
#include "ssm_math.cuh"

namespace mamba {

constexpr int kModes = 8;
constexpr int kPairs = kModes / 2;  // modes are advanced two at a time (packed fp32 pairs)
constexpr float kInvTwoPi = 0.15915494309189533577f;
constexpr float kTwoPi = 6.28318530717958647693f;
constexpr float kPi = 3.14159265358979323846f;

__device__ __forceinline__ float sin_approx(float x) {
  float y;
  asm("sin.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float cos_approx(float x) {
  float y;
  asm("cos.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// theta / 2pi as hi + lo: hi = fl(theta * (1/2pi)_hi), lo the rest of
// theta * ((1/2pi)_hi + (1/2pi)_lo) (the product's rounding error from an
// fma, plus theta times the low part of 1/2pi).
constexpr float kInvTwoPiLo = 6.4206382e-09f;  // 1/2pi - kInvTwoPi, rounded to fp32

__device__ __forceinline__ void turns_of(float theta, float& hi, float& lo) {
  hi = __fmul_rn(theta, kInvTwoPi);
  lo = __fmaf_rn(theta, kInvTwoPiLo, __fmaf_rn(theta, kInvTwoPi, -hi));
}

// The turn s theta of one mode reduced to [-pi, pi]: the turn count
// t = s theta / 2pi = s (hi + lo) less its nearest integer, formed as
// (t - rint(t)) + (the rounding error of t = s hi) + s lo.  Subtracting the
// nearest integer is exact, so the fraction keeps fp32's relative precision
// however many whole turns t holds.
__device__ __forceinline__ float turn_angle(float theta, float s) {
  float hi, lo;
  turns_of(theta, hi, lo);
  const float t = __fmul_rn(s, hi);
  const float e = __fmaf_rn(s, hi, -t);
  const float f = __fadd_rn(__fsub_rn(t, rintf(t)), __fmaf_rn(s, lo, e));
  return __fmul_rn(f, kTwoPi);
}

// The per-channel constants of one lane, by mode pair: element 0 of pair q
// belongs to mode 2q, element 1 to mode 2q + 1.
struct CChannel {
  float2 a2[kPairs];  // A2 = -exp(A_log) log2(e)
  float2 th[kPairs];  // theta
  float thr;          // steps s up to this keep every turn s theta within [-pi, pi]
  float4 w;
  float bias;
  float Dc;
};

__device__ __forceinline__ void load_cchannel(CChannel& ch, const ComplexParams& p, int c) {
  float tmax = 0.0f;
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const float4 al = __ldg(reinterpret_cast<const float4*>(p.A_log + (size_t)c * kModes) + q);
    const float4 th = __ldg(reinterpret_cast<const float4*>(p.theta + (size_t)c * kModes) + q);
    ch.a2[2 * q] = make_float2(a2_from_log(al.x), a2_from_log(al.y));
    ch.a2[2 * q + 1] = make_float2(a2_from_log(al.z), a2_from_log(al.w));
    ch.th[2 * q] = make_float2(th.x, th.y);
    ch.th[2 * q + 1] = make_float2(th.z, th.w);
    tmax = fmaxf(tmax, fmaxf(fmaxf(fabsf(th.x), fabsf(th.y)), fmaxf(fabsf(th.z), fabsf(th.w))));
  }
  // s <= fl(pi / tmax) keeps |fl(s theta)| within pi up to a rounding
  ch.thr = tmax > 0.0f ? __fdiv_rn(kPi, tmax) : __int_as_float(0x7f800000);
  ch.w = __ldg(reinterpret_cast<const float4*>(p.conv_w + (size_t)c * 4));
  ch.bias = p.conv_b ? __ldg(p.conv_b + c) : 0.0f;
  ch.Dc = __ldg(p.Dskip + c);
}

// exp(s lambda) for the first NP mode pairs at a step s (a dt or a dt sum):
// magnitude 2^(s A2), angle s theta -- taken as it is when s <= thr (every
// turn within [-pi, pi]), else reduced by turn_angle -- as (re, im) pairs.
template <int NP>
__device__ __forceinline__ void calphas(const CChannel& ch, float s, float2 (&are)[NP], float2 (&aim)[NP]) {
  const float2 s2 = make_float2(s, s);
  float2 r[NP];
  if (s <= ch.thr) {
#pragma unroll
    for (int q = 0; q < NP; ++q) r[q] = __fmul2_rn(s2, ch.th[q]);
  } else {
#pragma unroll
    for (int q = 0; q < NP; ++q) r[q] = make_float2(turn_angle(ch.th[q].x, s), turn_angle(ch.th[q].y, s));
  }
#pragma unroll
  for (int q = 0; q < NP; ++q) {
    const float2 e = __fmul2_rn(s2, ch.a2[q]);
    const float2 m = make_float2(ex2_approx(e.x), ex2_approx(e.y));
    are[q] = __fmul2_rn(m, make_float2(cos_approx(r[q].x), cos_approx(r[q].y)));
    aim[q] = __fmul2_rn(m, make_float2(sin_approx(r[q].x), sin_approx(r[q].y)));
  }
}

// (are + i aim)(gre + i gim) + (addre + i addim) for a mode pair, into
// (gre, gim): re = are gre + (-aim gim + addre), im = are gim + (aim gre + addim).
__device__ __forceinline__ void cmad2(float2 are, float2 aim, float2& gre, float2& gim, float2 addre,
                                      float2 addim) {
  const float2 re = __ffma2_rn(are, gre, __ffma2_rn(make_float2(-aim.x, -aim.y), gim, addre));
  const float2 im = __ffma2_rn(are, gim, __ffma2_rn(aim, gre, addim));
  gre = re;
  gim = im;
}

// A complex state (or state input) of one lane, by mode pair.  In memory it
// is (re, im) per mode in mode order, 16 floats.
struct CState {
  float2 re[kPairs];
  float2 im[kPairs];
};

// Four floats (re_2q, im_2q, re_2q+1, im_2q+1) of memory into pair q.
__device__ __forceinline__ void cstate_set(CState& s, int q, float4 v) {
  s.re[q] = make_float2(v.x, v.z);
  s.im[q] = make_float2(v.y, v.w);
}

// One token of one lane: the state advanced, and Re(sum_n C_n h_n) returned
// (per mode pair, Re C Re h and Im C Im h accumulated as packed pairs over
// the pairs in order, then the halves summed and the two parts subtracted).
// Q: the token's widened B/C row, per mode pair q the quads Q[2q] =
// (Re B_2q, Re B_2q+1, Im B_2q, Im B_2q+1) and Q[2q+1] the same of C.
// vp: the previous token's state input (trapezoidal only).
// NP < kPairs: only pairs 0..NP-1 advance (the carry walk's modes whose
// weight to the boundary is still above the drop bound; the others stay).
template <bool kTrap, bool kRead, int NP = kPairs>
__device__ __forceinline__ float ctoken(const CChannel& ch, CState& st, CState& vp, float u, float dt,
                                        const float4 (&Q)[kModes]) {
  float2 are[NP], aim[NP];
  calphas<NP>(ch, dt, are, aim);
  const float2 u2 = make_float2(u, u);
  const float h = kTrap ? __fmul_rn(0.5f, dt) : dt;  // the input's weight: dt/2 (trapezoidal) or dt
  const float2 h2 = make_float2(h, h);
  float2 accre = make_float2(0.0f, 0.0f), accim = make_float2(0.0f, 0.0f);
#pragma unroll
  for (int q = 0; q < NP; ++q) {
    const float2 vre = __fmul2_rn(make_float2(Q[2 * q].x, Q[2 * q].y), u2);
    const float2 vim = __fmul2_rn(make_float2(Q[2 * q].z, Q[2 * q].w), u2);
    if (kTrap) {
      st.re[q] = __ffma2_rn(h2, vp.re[q], st.re[q]);
      st.im[q] = __ffma2_rn(h2, vp.im[q], st.im[q]);
      vp.re[q] = vre;
      vp.im[q] = vim;
    }
    cmad2(are[q], aim[q], st.re[q], st.im[q], __fmul2_rn(h2, vre), __fmul2_rn(h2, vim));
    if (kRead) {
      accre = __ffma2_rn(make_float2(Q[2 * q + 1].x, Q[2 * q + 1].y), st.re[q], accre);
      accim = __ffma2_rn(make_float2(Q[2 * q + 1].z, Q[2 * q + 1].w), st.im[q], accim);
    }
  }
  return __fsub_rn(__fadd_rn(accre.x, accre.y), __fadd_rn(accim.x, accim.y));
}

// acc += exp(s lambda) h, every mode (a carry weight times a state).
__device__ __forceinline__ void cstate_add_weighted(const CChannel& ch, float s, const CState& h, CState& acc) {
  float2 are[kPairs], aim[kPairs];
  calphas<kPairs>(ch, s, are, aim);
#pragma unroll
  for (int q = 0; q < kPairs; ++q) {
    float2 re = h.re[q], im = h.im[q];
    cmad2(are[q], aim[q], re, im, acc.re[q], acc.im[q]);
    acc.re[q] = re;
    acc.im[q] = im;
  }
}

__device__ __forceinline__ void cstate_zero(CState& s) {
#pragma unroll
  for (int q = 0; q < kPairs; ++q) {
    s.re[q] = make_float2(0.0f, 0.0f);
    s.im[q] = make_float2(0.0f, 0.0f);
  }
}

__device__ __forceinline__ void cstate_load(CState& s, const float* p) {
#pragma unroll
  for (int q = 0; q < kPairs; ++q) cstate_set(s, q, reinterpret_cast<const float4*>(p)[q]);
}

__device__ __forceinline__ void cstate_store(const CState& s, float* p) {
#pragma unroll
  for (int q = 0; q < kPairs; ++q)
    reinterpret_cast<float4*>(p)[q] = make_float4(s.re[q].x, s.im[q].x, s.re[q].y, s.im[q].y);
}

// The state input v = B u of a token from its widened B/C row (global).
__device__ __forceinline__ void cinput_from_row(CState& v, const float* row, float u) {
  const float2 u2 = make_float2(u, u);
#pragma unroll
  for (int q = 0; q < kPairs; ++q) {
    const float4 b = __ldg(reinterpret_cast<const float4*>(row) + 2 * q);
    v.re[q] = __fmul2_rn(make_float2(b.x, b.y), u2);
    v.im[q] = __fmul2_rn(make_float2(b.z, b.w), u2);
  }
}

// Raw input of channel c at token tau (tau < 0: conv_state0, or zero).
template <typename IO>
__device__ __forceinline__ float cinput_at(const ComplexParams& p, int b, long tau, int c) {
  if (tau >= 0) return to_f32(reinterpret_cast<const IO*>(p.x)[((size_t)b * p.seqlen + tau) * p.d_inner + c]);
  if (p.conv_state0 == nullptr) return 0.0f;
  return to_f32(reinterpret_cast<const IO*>(p.conv_state0)[((size_t)b * 3 + (3 + tau)) * p.d_inner + c]);
}

// The state input v of the token before t0 (trapezoidal rule): v0 (or zero)
// before the first token, else B_{t0-1} u_{t0-1} from the inputs (xm3..xm1
// are the inputs at t0-3..t0-1).
template <typename IO>
__device__ __forceinline__ void cvprev_at(CState& vp, const ComplexParams& p, const CChannel& ch, int b, int t0,
                                          int cl, float xm3, float xm2, float xm1) {
  if (t0 == 0) {
    if (p.v0)
      cstate_load(vp, p.v0 + ((size_t)b * p.d_inner + cl) * 16);
    else
      cstate_zero(vp);
    return;
  }
  const float xm4 = cinput_at<IO>(p, b, (long)t0 - 4, cl);
  const float u = silu(conv4(ch.w, ch.bias, xm4, xm3, xm2, xm1));
  cinput_from_row(vp, p.bc + ((size_t)b * p.seqlen + t0 - 1) * kBC, u);
}

// One chunk of one channel group (lane = channel) of one batch row.  kSummary
// (the exact chunked mode's first pass): chunks 0..n-2 from a zero state, no
// z and no y; stores hloc_j and S_j.  Otherwise the main pass: the chunk from
// its entering state, y written.  fused (the walked chunked mode, one launch
// with the carry walks): the state entering chunk j > 0 is awaited (bounded)
// on its flag; chunk 0's warp and boundary 1's walk, the readers of h0, v0
// and conv_state0, count themselves done on the group's chunk-0 flag, which
// the last chunk's warp checks before it writes the final states that may
// alias them.
// Token r of a staged tile (x, dt_raw, B/C rows; z when kY): the state
// advanced, y stored where wy holds (kY), dt summed into sdt (kSum).
// kSmall: the tile's dt_raw all lie in softplus's small region.
template <typename IO, typename Stage, bool kTrap, bool kY, bool kSum, int NP, bool kSmall>
__device__ __forceinline__ void ctoken_one(const Stage& S, int r, int lane, const CChannel& ch, CState& st,
                                           CState& vp, float& sdt, float& xm3, float& xm2, float& xm1, bool wy,
                                           IO* ytile, int D) {
  const float xv = to_f32(S.x[r][lane]);
  const float u = silu(conv4(ch.w, ch.bias, xm3, xm2, xm1, xv));
  xm3 = xm2;
  xm2 = xm1;
  xm1 = xv;
  const float dt = softplus_sel<kSmall>(to_f32(S.dt[r][lane]));
  float4 Q[kModes];
  load_quads(&S.bc[r][0], Q);
  const float yss = ctoken<kTrap, kY, NP>(ch, st, vp, u, dt, Q);
  if (kSum) sdt = __fadd_rn(sdt, dt);
  if constexpr (kY) {
    const float gz = silu(to_f32(S.z[r][lane]));
    st_global_if(wy, ytile + (size_t)r * D, from_f32<IO>(gate_out(yss, ch.Dc, u, gz)));
  }
}

// Tokens r and r+1 of a tile whose dt_raw all lie in softplus's small
// region: as ctoken_one on each, with the per-token scalar work (conv, SiLU,
// softplus, SiLU(z), gate) of the two as packed f32x2 operations -- the same
// operations on each token, so the same bits.
template <typename IO, typename Stage, bool kTrap, bool kY, bool kSum, int NP>
__device__ __forceinline__ void ctoken_two(const Stage& S, int r, int lane, const CChannel& ch, CState& st,
                                           CState& vp, float& sdt, float& xm3, float& xm2, float& xm1, bool wy,
                                           IO* ytile, int D) {
  const float x0 = to_f32(S.x[r][lane]);
  const float x1 = to_f32(S.x[r + 1][lane]);
  const float2 u = silu_x2(conv4_x2(ch.w, ch.bias, xm3, xm2, xm1, x0, x1));
  xm3 = xm1;
  xm2 = x0;
  xm1 = x1;
  const float2 dt = softplus_small_raw_x2(make_float2(to_f32(S.dt[r][lane]), to_f32(S.dt[r + 1][lane])));
  float4 Q[kModes];
  load_quads(&S.bc[r][0], Q);
  const float y0 = ctoken<kTrap, kY, NP>(ch, st, vp, u.x, dt.x, Q);
  load_quads(&S.bc[r + 1][0], Q);
  const float y1 = ctoken<kTrap, kY, NP>(ch, st, vp, u.y, dt.y, Q);
  if (kSum) sdt = __fadd_rn(__fadd_rn(sdt, dt.x), dt.y);
  if constexpr (kY) {
    const float2 gz = silu_x2(make_float2(to_f32(S.z[r][lane]), to_f32(S.z[r + 1][lane])));
    const float2 yv = gate_out_x2(make_float2(y0, y1), ch.Dc, u, gz);
    st_global_if(wy, ytile + (size_t)r * D, from_f32<IO>(yv.x));
    st_global_if(wy, ytile + (size_t)(r + 1) * D, from_f32<IO>(yv.y));
  }
}

// One staged tile of `rows` tokens, token pairs in tiles whose dt_raw all
// lie in softplus's small region (checked over the warp's active lanes).
// Euler unrolls two token pairs (the next pair's angles and inputs overlap
// the current pair's state updates: 2.66 -> 2.56 ms at 32k x 8192, 164
// registers, still three warps per scheduler); the trapezoidal rule, whose
// previous inputs take 16 more registers, measured slower so (2.66 -> 2.70).
template <typename IO, typename Stage, bool kTrap, bool kY, bool kSum, int NP>
__device__ __forceinline__ void ctile(const Stage& S, int rows, int lane, bool active, const CChannel& ch,
                                      CState& st, CState& vp, float& sdt, float& xm3, float& xm2, float& xm1,
                                      bool wy, IO* ytile, int D) {
  if (small_dt_tile<IO>(S.dt, rows, lane, active)) {
    int r = 0;
#pragma unroll(kTrap ? 1 : 2)
    for (; r + 1 < rows; r += 2)
      ctoken_two<IO, Stage, kTrap, kY, kSum, NP>(S, r, lane, ch, st, vp, sdt, xm3, xm2, xm1, wy, ytile, D);
    if (r < rows)
      ctoken_one<IO, Stage, kTrap, kY, kSum, NP, true>(S, r, lane, ch, st, vp, sdt, xm3, xm2, xm1, wy, ytile, D);
  } else {
#pragma unroll 2
    for (int r = 0; r < rows; ++r)
      ctoken_one<IO, Stage, kTrap, kY, kSum, NP, false>(S, r, lane, ch, st, vp, sdt, xm3, xm2, xm1, wy, ytile, D);
  }
}

template <typename IO, bool kTrap, bool kSummary>
__device__ __forceinline__ void complex_pass(const CUtensorMap& tm_x, const CUtensorMap& tm_z,
                                             const CUtensorMap& tm_dt, const CUtensorMap& tm_bc,
                                             const ComplexParams& p, MainSmem<IO>& sm, int g, int b, int j,
                                             bool fused) {
  constexpr bool kY = !kSummary;
  const int lane = threadIdx.x;
  const int c0 = g * kLanes;
  const int D = p.d_inner;
  const int c = c0 + lane;
  const bool active = c < D;
  const int cl = active ? c : D - 1;
  const int t_begin = j * p.chunk_tiles * kT;
  const int t_end = min(t_begin + p.chunk_tiles * kT, p.seqlen);
  const int n_tiles = (t_end - t_begin + kT - 1) / kT;

  if (lane == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(smem_u32(&sm.full[s]), 1);
    fence_mbar_init();
    prefetch_tensormap(&tm_x);
    if (kY) prefetch_tensormap(&tm_z);
    prefetch_tensormap(&tm_dt);
    prefetch_tensormap(&tm_bc);
  }
  __syncwarp();

  constexpr uint32_t kBytes = (kY ? 3 : 2) * kT * kLanes * sizeof(IO) + kT * kBC * sizeof(float);
  if (lane == 0) {
    for (int k = 0; k < kStages && k < n_tiles; ++k) {
      const uint32_t bar = smem_u32(&sm.full[k]);
      const int tt = t_begin + k * kT;
      mbar_arrive_expect_tx(bar, kBytes);
      tma_load_3d(smem_u32(&sm.stage[k].x[0][0]), &tm_x, c0, tt, b, bar);
      if (kY) tma_load_3d(smem_u32(&sm.stage[k].z[0][0]), &tm_z, c0, tt, b, bar);
      tma_load_3d(smem_u32(&sm.stage[k].dt[0][0]), &tm_dt, c0, tt, b, bar);
      tma_load_3d(smem_u32(&sm.stage[k].bc[0][0]), &tm_bc, 0, tt, b, bar);
    }
  }

  CChannel ch;
  load_cchannel(ch, p, cl);
  const size_t sidx = ((size_t)b * D + cl) * 16;  // this channel's 16 numbers in (B, D, 16)
  // In the exact chunked mode the fold (an earlier launch) copied h0 into the
  // carry's chunk-0 slot and v0 into the unused last slot of hloc, so that no
  // CTA of the main launch reads h0 or v0, which the last chunk's final_h
  // and final_v may alias.
  const bool folded = !kSummary && !fused && p.n_chunks > 1;
  CState st, vp;
  if (fused && j > 0) {
    bool have = true;
    if (lane == 0) {
      const unsigned* ready = p.counters + 1 + ((size_t)b * p.n_groups + g) * p.n_chunks;
      const uint64_t t_start = globaltimer_ns();
      while (atomicAdd(const_cast<unsigned*>(ready + j), 0u) == 0u) {
        if (globaltimer_ns() - t_start > p.timeout_ns) {
          have = false;
          break;
        }
      }
    }
    have = __shfl_sync(0xffffffffu, have, 0);
    __threadfence();
    if (!have) {
      if (lane == 0) report_error(4u);  // MAMBA_ERR_TIMEOUT
      cstate_zero(st);
    } else {
      const float4* src = reinterpret_cast<const float4*>(p.carry + (((size_t)b * p.n_chunks + j) * D + cl) * 16);
#pragma unroll
      for (int q = 0; q < kPairs; ++q) cstate_set(st, q, __ldcg(src + q));  // from L2: written by another SM during this launch
    }
  } else if (kSummary || (j == 0 && !folded && p.h0 == nullptr)) {
    cstate_zero(st);
  } else if (j == 0 && !folded) {
    cstate_load(st, p.h0 + sidx);
  } else {
    cstate_load(st, p.carry + (((size_t)b * p.n_chunks + j) * D + cl) * 16);
  }

  if (!kTrap) cstate_zero(vp);
  float xm3 = cinput_at<IO>(p, b, (long)t_begin - 3, cl);
  float xm2 = cinput_at<IO>(p, b, (long)t_begin - 2, cl);
  float xm1 = cinput_at<IO>(p, b, (long)t_begin - 1, cl);
  if (kTrap) {  // the state input of the token before the chunk
    if (j == 0 && folded) {
      if (p.v0 == nullptr)
        cstate_zero(vp);
      else
        cstate_load(vp, p.hloc + (((size_t)b * p.n_chunks + p.n_chunks - 1) * D + cl) * 16);
    } else {
      cvprev_at<IO>(vp, p, ch, b, t_begin, cl, xm3, xm2, xm1);
    }
  }
  if (kY && !fused && j == 0 && p.final_conv_state != nullptr) {
    // the one CTA of these channels in this launch that reads conv_state0,
    // which the final conv state may alias: read before written
    const float f0 = cinput_at<IO>(p, b, (long)p.seqlen - 3, cl);
    const float f1 = cinput_at<IO>(p, b, (long)p.seqlen - 2, cl);
    const float f2 = cinput_at<IO>(p, b, (long)p.seqlen - 1, cl);
    __syncwarp();
    if (active) {
      IO* fcs = reinterpret_cast<IO*>(p.final_conv_state) + (size_t)b * 3 * D + c;
      fcs[0] = from_f32<IO>(f0);
      fcs[D] = from_f32<IO>(f1);
      fcs[2 * (size_t)D] = from_f32<IO>(f2);
    }
  }
  if (fused && j == 0) {  // h0, v0 and conv_state0 read
    __syncwarp();
    if (lane == 0) {
      __threadfence();
      atomicAdd(p.counters + 1 + ((size_t)b * p.n_groups + g) * p.n_chunks, 1u);
    }
  }
  // the fused launch's last chunk writes the final conv state at its end
  float f0 = 0.0f, f1 = 0.0f, f2 = 0.0f;
  if (kY && fused && j == p.n_chunks - 1 && p.final_conv_state != nullptr) {
    f0 = cinput_at<IO>(p, b, (long)p.seqlen - 3, cl);
    f1 = cinput_at<IO>(p, b, (long)p.seqlen - 2, cl);
    f2 = cinput_at<IO>(p, b, (long)p.seqlen - 1, cl);
  }

  const bool wy = kY && active;
  IO* yrow = kY ? reinterpret_cast<IO*>(p.y) + ((size_t)b * p.seqlen + t_begin) * D + cl : nullptr;
  float sdt = 0.0f;
  bool ok = true;
  int k = 0;
  for (; k < n_tiles; ++k) {
    const int s = k % kStages;
    const MainStage<IO>& S = sm.stage[s];
    const int rows = min(kT, t_end - (t_begin + k * kT));
    const bool mine = mbar_wait_bounded(smem_u32(&sm.full[s]), (k / kStages) & 1, p.timeout_ns);
    ok = __all_sync(0xffffffffu, mine);
    if (!ok) break;
    IO* ytile = kY ? yrow + (size_t)k * kT * D : nullptr;
    ctile<IO, MainStage<IO>, kTrap, kY, kSummary, kPairs>(S, rows, lane, active, ch, st, vp, sdt, xm3, xm2, xm1,
                                                          wy, ytile, D);
    __syncwarp();  // every lane is done with stage s
    if (lane == 0 && k + kStages < n_tiles) {
      const uint32_t bar = smem_u32(&sm.full[s]);
      const int tt = t_begin + (k + kStages) * kT;
      mbar_arrive_expect_tx(bar, kBytes);
      tma_load_3d(smem_u32(&sm.stage[s].x[0][0]), &tm_x, c0, tt, b, bar);
      if (kY) tma_load_3d(smem_u32(&sm.stage[s].z[0][0]), &tm_z, c0, tt, b, bar);
      tma_load_3d(smem_u32(&sm.stage[s].dt[0][0]), &tm_dt, c0, tt, b, bar);
      tma_load_3d(smem_u32(&sm.stage[s].bc[0][0]), &tm_bc, 0, tt, b, bar);
    }
  }

  if (!ok) {
    if (lane == 0) {
      report_error(4u);  // MAMBA_ERR_TIMEOUT
      drain_ring(sm.full, k, n_tiles, p.timeout_ns);
    }
    return;
  }
  const bool finals = !kSummary && j == p.n_chunks - 1;
  if (finals && fused) {  // the readers of h0, v0 and conv_state0 are done (bounded)
    if (lane == 0) {
      const unsigned* readers = p.counters + 1 + ((size_t)b * p.n_groups + g) * p.n_chunks;
      const uint64_t t_start = globaltimer_ns();
      while (ld_relaxed_gpu(readers) < 2u) {
        if (globaltimer_ns() - t_start > p.timeout_ns) {
          report_error(4u);  // MAMBA_ERR_TIMEOUT
          break;
        }
      }
    }
    __syncwarp();  // the other lanes' stores come after lane 0's check
  }
  if (!active) return;
  if (kSummary) {
    cstate_store(st, p.hloc + (((size_t)b * p.n_chunks + j) * D + c) * 16);
    p.sdt[((size_t)b * p.n_chunks + j) * D + c] = sdt;
  } else if (finals) {
    if (p.final_h) cstate_store(st, p.final_h + sidx);
    if (p.final_v) {
      if (!kTrap) {  // Euler keeps no previous input: the last token's, from its inputs
        const float u =
            silu(conv4(ch.w, ch.bias, cinput_at<IO>(p, b, (long)p.seqlen - 4, c), xm3, xm2, xm1));
        cinput_from_row(vp, p.bc + ((size_t)b * p.seqlen + p.seqlen - 1) * kBC, u);
      }
      cstate_store(vp, p.final_v + sidx);
    }
    if (fused && p.final_conv_state != nullptr) {
      IO* fcs = reinterpret_cast<IO*>(p.final_conv_state) + (size_t)b * 3 * D + c;
      fcs[0] = from_f32<IO>(f0);
      fcs[D] = from_f32<IO>(f1);
      fcs[2 * (size_t)D] = from_f32<IO>(f2);
    }
  }
}

// grid (n_groups, batch, chunks), 32 threads: one pass, or a pass of the
// exact chunked mode.
template <typename IO, bool kTrap, bool kSummary>
__global__ void __launch_bounds__(kLanes)
    complex_scan_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_z,
                        const __grid_constant__ CUtensorMap tm_dt, const __grid_constant__ CUtensorMap tm_bc,
                        const __grid_constant__ ComplexParams p) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  complex_pass<IO, kTrap, kSummary>(tm_x, tm_z, tm_dt, tm_bc, p,
                                    *reinterpret_cast<MainSmem<IO>*>(smem_raw + smem_pad128(smem_raw)), blockIdx.x,
                                    blockIdx.y, blockIdx.z, false);
}

// One full tile of a carry piece: mode pairs 0..NP-1 advanced, the dt summed.
template <typename IO, bool kTrap, int NP>
__device__ __forceinline__ void ccarry_tile(const SummaryStage<IO>& S, int lane, bool active, const CChannel& ch,
                                            CState& st, CState& vp, float& sdt, float& xm3, float& xm2,
                                            float& xm1) {
  ctile<IO, SummaryStage<IO>, kTrap, false, true, NP>(S, kT, lane, active, ch, st, vp, sdt, xm3, xm2, xm1, false,
                                                      static_cast<IO*>(nullptr), 0);
}

// The walked chunked mode's carry walk: one warp per (chunk boundary j =
// 1..n_chunks-1, channel group, batch row), taken in ticket order, computes
// the state entering chunk j from chunk j-1's tokens as the real scan's walk
// does, with complex weights: chunk j-1's pieces are walked backwards, each
// scanned forward from zero (hloc_q), and
//   carry_j = sum_q W_q hloc_q + W_start carry_{j-1},
// W_q = exp(lambda * (dt summed from the end of piece q to the boundary)),
// the product of the alphas over those tokens.  The walk stops once every
// mode of every lane has decayed below 2^-32 (|W| = 2^(A2 s) with the
// slowest A2) from the current piece's start to the boundary; otherwise it
// waits (bounded) for carry_{j-1}, published by boundary j-1's warp (an
// earlier ticket), and folds it in.  Trapezoidal: each piece starts from the
// state input of the token before it (from the inputs; v0 before token 0).
template <typename IO, bool kTrap>
__device__ __forceinline__ void ccarry_warp(const CUtensorMap& tm_x, const CUtensorMap& tm_dt,
                                            const CUtensorMap& tm_bc, const ComplexParams& p, CarrySmem<IO>& sm,
                                            unsigned ticket) {
  const int lane = threadIdx.x;
  if (lane == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(smem_u32(&sm.full[s]), 1);
    fence_mbar_init();
    prefetch_tensormap(&tm_x);
    prefetch_tensormap(&tm_dt);
    prefetch_tensormap(&tm_bc);
  }
  __syncwarp();
  const int per = p.n_chunks - 1;
  const int j = (int)(ticket % per) + 1;  // boundary: the state entering chunk j
  const int gb = (int)(ticket / per);
  const int g = gb % p.n_groups;
  const int b = gb / p.n_groups;
  const int D = p.d_inner;
  const int c0 = g * kLanes;
  const int c = c0 + lane;
  const bool active = c < D;
  const int cl = active ? c : D - 1;
  unsigned* ready = p.counters + 1 + ((size_t)b * p.n_groups + g) * p.n_chunks;

  PieceWalk wk;  // chunk j-1 is never the last chunk: whole tiles
  wk.first_tile = (j - 1) * p.chunk_tiles;
  wk.C = p.chunk_tiles;
  wk.P = p.piece_tiles;
  wk.m = p.pieces;
  wk.len_last = p.chunk_tiles - (p.pieces - 1) * p.piece_tiles;
  const int n_tiles = wk.C;
  if (lane == 0)
    for (int k = 0; k < kStages && k < n_tiles; ++k)
      issue_carry_tile<IO>(sm, k, &tm_x, &tm_dt, &tm_bc, c0, wk.tile_of(k), b);

  CChannel ch;
  load_cchannel(ch, p, cl);
  float a2max = fmaxf(ch.a2[0].x, ch.a2[0].y);  // the slowest decay of this channel
#pragma unroll
  for (int q = 1; q < kPairs; ++q) a2max = fmaxf(a2max, fmaxf(ch.a2[q].x, ch.a2[q].y));
  CState acc, st, vp;
  cstate_zero(acc);
  cstate_zero(st);
  float s_after = 0.0f;  // dt summed from the current piece's end to the boundary
  float sdt = 0.0f;
  int left = wk.piece_len(wk.piece_of(0));  // tiles left in the current piece
  int t0 = wk.tile_of(0) * kT;
  float xm3 = cinput_at<IO>(p, b, (long)t0 - 3, cl);
  float xm2 = cinput_at<IO>(p, b, (long)t0 - 2, cl);
  float xm1 = cinput_at<IO>(p, b, (long)t0 - 1, cl);
  if (kTrap) cvprev_at<IO>(vp, p, ch, b, t0, cl, xm3, xm2, xm1);
  else cstate_zero(vp);

  int n_pairs = kPairs;  // leading mode pairs the current piece advances
  bool ok = true, done = false;
  int k = 0;
  for (; k < n_tiles; ++k) {
    const int s = k % kStages;
    const SummaryStage<IO>& S = sm.stage[s];
    const bool mine = mbar_wait_bounded(smem_u32(&sm.full[s]), (k / kStages) & 1, p.timeout_ns);
    ok = __all_sync(0xffffffffu, mine);
    if (!ok) break;
    if (n_pairs == 1)
      ccarry_tile<IO, kTrap, 1>(S, lane, active, ch, st, vp, sdt, xm3, xm2, xm1);
    else if (n_pairs == 2)
      ccarry_tile<IO, kTrap, 2>(S, lane, active, ch, st, vp, sdt, xm3, xm2, xm1);
    else
      ccarry_tile<IO, kTrap, 4>(S, lane, active, ch, st, vp, sdt, xm3, xm2, xm1);
    __syncwarp();  // every lane is done with stage s
    if (lane == 0 && k + kStages < n_tiles)
      issue_carry_tile<IO>(sm, s, &tm_x, &tm_dt, &tm_bc, c0, wk.tile_of(k + kStages), b);
    if (--left == 0) {  // piece done: acc += W hloc, W from the piece's end to the boundary
      cstate_add_weighted(ch, s_after, st, acc);
      s_after = __fadd_rn(s_after, sdt);
      if ((p.flags & kFlagExactCarry) == 0 &&
          __all_sync(0xffffffffu, !active || __fmul_rn(a2max, s_after) < kCarryDropLog2)) {
        done = true;
        ++k;
        break;
      }
      if (k + 1 < n_tiles) {  // the next (earlier) piece, from zero
        left = wk.piece_len(wk.piece_of(k + 1));
        cstate_zero(st);
        sdt = 0.0f;
        // modes whose weight to the boundary fell below the drop bound add
        // nothing from here on: the piece advances the leading pairs up to
        // the last pair with a mode still above it
        if ((p.flags & kFlagExactCarry) == 0) {
          int last = -1;
#pragma unroll
          for (int q = 0; q < kPairs; ++q)
            if (__fmul_rn(fmaxf(ch.a2[q].x, ch.a2[q].y), s_after) >= kCarryDropLog2) last = q;
          n_pairs = __reduce_max_sync(0xffffffffu, active ? last + 1 : 0);
        }
        t0 = wk.tile_of(k + 1) * kT;
        xm3 = cinput_at<IO>(p, b, (long)t0 - 3, cl);
        xm2 = cinput_at<IO>(p, b, (long)t0 - 2, cl);
        xm1 = cinput_at<IO>(p, b, (long)t0 - 1, cl);
        if (kTrap) cvprev_at<IO>(vp, p, ch, b, t0, cl, xm3, xm2, xm1);
      }
    }
  }
  if (lane == 0) {  // copies still in flight land before shared memory goes away
    for (int kk = k; kk < n_tiles && kk < k + kStages; ++kk)
      (void)mbar_wait_bounded(smem_u32(&sm.full[kk % kStages]), (kk / kStages) & 1, p.timeout_ns);
  }
  if (!ok && lane == 0) report_error(4u);  // MAMBA_ERR_TIMEOUT

  if (ok && !done) {  // the whole chunk matters: fold in the state entering it
    CState prev;
    if (j - 1 == 0) {
      if (p.h0)
        cstate_load(prev, p.h0 + ((size_t)b * D + cl) * 16);
      else
        cstate_zero(prev);
    } else {
      bool have = true;
      if (lane == 0) {
        const uint64_t t_start = globaltimer_ns();
        while (atomicAdd(ready + (j - 1), 0u) == 0u) {
          if (globaltimer_ns() - t_start > p.timeout_ns) {
            have = false;
            break;
          }
        }
      }
      have = __shfl_sync(0xffffffffu, have, 0);
      __threadfence();
      if (!have) {
        if (lane == 0) report_error(4u);
        cstate_zero(prev);
      } else {
        const float4* src = reinterpret_cast<const float4*>(p.carry + (((size_t)b * p.n_chunks + (j - 1)) * D + cl) * 16);
#pragma unroll
        for (int q = 0; q < kPairs; ++q) cstate_set(prev, q, __ldcg(src + q));
      }
    }
    cstate_add_weighted(ch, s_after, prev, acc);
  }

  // publish carry_j (also after a failure, so that no later boundary waits in vain)
  if (active) cstate_store(acc, p.carry + (((size_t)b * p.n_chunks + j) * D + c) * 16);
  __threadfence();
  __syncwarp();
  if (lane == 0) {
    atomicExch(ready + j, 1u);
    if (j == 1) atomicAdd(ready, 1u);  // boundary 1's walk is done with h0, v0 and conv_state0
  }
}

// The walked chunked mode in one launch of (n_chunks - 1) * n_groups * batch
// carry warps and n_chunks * n_groups * batch main warps, ticket-ordered as
// the real scan's fused launch.
template <typename IO, bool kTrap>
__global__ void __launch_bounds__(kLanes)
    complex_fused_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_z,
                         const __grid_constant__ CUtensorMap tm_dt, const __grid_constant__ CUtensorMap tm_bc,
                         const __grid_constant__ ComplexParams p) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  unsigned char* base = smem_raw + smem_pad128(smem_raw);
  unsigned ticket = 0;
  if (threadIdx.x == 0) ticket = atomicAdd(p.counters, 1u);
  ticket = __shfl_sync(0xffffffffu, ticket, 0);
  const unsigned per = (unsigned)p.n_groups * (unsigned)p.batch;
  const unsigned n_carry = (unsigned)(p.n_chunks - 1) * per;
  if (ticket < n_carry) {
    ccarry_warp<IO, kTrap>(tm_x, tm_dt, tm_bc, p, *reinterpret_cast<CarrySmem<IO>*>(base), ticket);
  } else {
    const unsigned t = ticket - n_carry;
    const int j = (int)(t / per), gb = (int)(t % per);
    complex_pass<IO, kTrap, false>(tm_x, tm_z, tm_dt, tm_bc, p, *reinterpret_cast<MainSmem<IO>*>(base),
                                   gb % p.n_groups, gb / p.n_groups, j, true);
  }
}

// The fold: one thread per (batch row, channel); h_in_{j+1} = W_j h_in_j +
// hloc_j in chunk order, h_in_0 = h0 (or zero); W_j = exp(lambda S_j).
// h_in_0 goes to the carry's chunk-0 slot and v0 to hloc's last slot (the
// summary pass leaves it unused), from which the main pass reads them.
__global__ void __launch_bounds__(256) complex_fold_kernel(const __grid_constant__ ComplexParams p) {
  const long i = (long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (long)p.batch * p.d_inner) return;
  const int b = (int)(i / p.d_inner), c = (int)(i % p.d_inner);
  const int D = p.d_inner;
  CChannel ch;
  load_cchannel(ch, p, c);
  CState h;
  if (p.h0)
    cstate_load(h, p.h0 + ((size_t)b * D + c) * 16);
  else
    cstate_zero(h);
  cstate_store(h, p.carry + ((size_t)b * p.n_chunks * D + c) * 16);
  if (p.v0) {
    CState v;
    cstate_load(v, p.v0 + ((size_t)b * D + c) * 16);
    cstate_store(v, p.hloc + (((size_t)b * p.n_chunks + p.n_chunks - 1) * D + c) * 16);
  }
  for (int j = 0; j + 1 < p.n_chunks; ++j) {
    const size_t cj = ((size_t)b * p.n_chunks + j) * D + c;
    CState hl;
    cstate_load(hl, p.hloc + cj * 16);
    const float S = p.sdt[cj];
    cstate_add_weighted(ch, S, h, hl);  // hl = W_j h_in_j + hloc_j
    h = hl;
    cstate_store(h, p.carry + (((size_t)b * p.n_chunks + j + 1) * D + c) * 16);
  }
}

}  // namespace mamba
