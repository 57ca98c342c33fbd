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
// The turn dt theta_n is taken in whole turns first (t = dt theta_n / 2pi,
// reduced to [-1/2, 1/2] by subtracting the nearest integer) and then fed to
// the approximate sine and cosine, whose error bound holds on [-pi, pi].  So
// that a turn of many revolutions per token keeps its fraction to fp32
// precision, theta / 2pi is held as two fp32 parts (hi + lo) and the product
// dt * hi carries its exact rounding error (an fma) into the fraction.
//
// Decomposition: as the real scan's main pass -- a CTA is one warp, lane i
// owns channel c0 + i with all 16 numbers of its state in registers, tiles of
// 16 tokens of x, z, dt_raw and the widened B/C rows arrive by TMA through a
// two-stage mbarrier ring.  The widened row of a token holds, per mode n,
// the quad (Re B_n, Im B_n, Re C_n, Im C_n).
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
constexpr float kInvTwoPi = 0.15915494309189533577f;
constexpr float kTwoPi = 6.28318530717958647693f;

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

// The per-channel constants of one lane.
struct CChannel {
  float a2[kModes];  // A2 = -exp(A_log) log2(e)
  float tu[kModes];  // theta / 2pi (turns per unit of dt), rounded to fp32 ...
  float tl[kModes];  // ... and the rest: theta / 2pi = tu + tl to ~2^-48
  float4 w;
  float bias;
  float Dc;
};

__device__ __forceinline__ void load_cchannel(CChannel& ch, const ComplexParams& p, int c) {
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const float4 al = __ldg(reinterpret_cast<const float4*>(p.A_log + (size_t)c * kModes) + q);
    const float4 th = __ldg(reinterpret_cast<const float4*>(p.theta + (size_t)c * kModes) + q);
    ch.a2[4 * q + 0] = a2_from_log(al.x);
    ch.a2[4 * q + 1] = a2_from_log(al.y);
    ch.a2[4 * q + 2] = a2_from_log(al.z);
    ch.a2[4 * q + 3] = a2_from_log(al.w);
    const float thv[4] = {th.x, th.y, th.z, th.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) turns_of(thv[i], ch.tu[4 * q + i], ch.tl[4 * q + i]);
  }
  ch.w = __ldg(reinterpret_cast<const float4*>(p.conv_w + (size_t)c * 4));
  ch.bias = p.conv_b ? __ldg(p.conv_b + c) : 0.0f;
  ch.Dc = __ldg(p.Dskip + c);
}

// exp(s lambda) for a dt (or dt sum) s: magnitude 2^(s A2), turn
// s theta / 2pi = s (tu + tl), whose fraction is formed as (t - rint(t)) +
// (the rounding error of t = s tu) + s tl: the subtraction of the nearest
// integer is exact, so the fraction keeps fp32's relative precision however
// many whole turns t holds.
__device__ __forceinline__ float2 cexp_step(float a2, float tu, float tl, float s) {
  const float m = ex2_approx(__fmul_rn(s, a2));
  const float t = __fmul_rn(s, tu);
  const float e = __fmaf_rn(s, tu, -t);
  const float f = __fadd_rn(__fsub_rn(t, rintf(t)), __fmaf_rn(s, tl, e));
  const float r = __fmul_rn(f, kTwoPi);
  return make_float2(__fmul_rn(m, cos_approx(r)), __fmul_rn(m, sin_approx(r)));
}

// (a + ib)(x + iy) + (bx' + i by')
__device__ __forceinline__ float2 cmul_add(float2 a, float2 g, float2 add) {
  return make_float2(__fmaf_rn(a.x, g.x, __fmaf_rn(-a.y, g.y, add.x)), __fmaf_rn(a.x, g.y, __fmaf_rn(a.y, g.x, add.y)));
}

struct CState {
  float2 h[kModes];
};

// One token of one lane: the state advanced, and Re(sum_n C_n h_n) returned
// (read-out accumulated in a fixed order: (Re C Re h, Im C Im h) summed over
// n as a packed pair, then the two parts subtracted).  vp: the previous
// token's state input (trapezoidal only).
template <bool kTrap, bool kRead>
__device__ __forceinline__ float ctoken(const CChannel& ch, CState& st, CState& vp, float u, float dt,
                                        const float4 (&Q)[kModes]) {
  const float hdt = __fmul_rn(0.5f, dt);
  float2 acc = make_float2(0.0f, 0.0f);
#pragma unroll
  for (int n = 0; n < kModes; ++n) {
    const float2 al = cexp_step(ch.a2[n], ch.tu[n], ch.tl[n], dt);
    const float2 v = make_float2(__fmul_rn(Q[n].x, u), __fmul_rn(Q[n].y, u));
    if (kTrap) {
      const float2 g = make_float2(__fmaf_rn(hdt, vp.h[n].x, st.h[n].x), __fmaf_rn(hdt, vp.h[n].y, st.h[n].y));
      st.h[n] = cmul_add(al, g, make_float2(__fmul_rn(hdt, v.x), __fmul_rn(hdt, v.y)));
      vp.h[n] = v;
    } else {
      st.h[n] = cmul_add(al, st.h[n], make_float2(__fmul_rn(dt, v.x), __fmul_rn(dt, v.y)));
    }
    if (kRead) acc = __ffma2_rn(make_float2(Q[n].z, Q[n].w), st.h[n], acc);
  }
  return __fsub_rn(acc.x, acc.y);
}

__device__ __forceinline__ void cstate_zero(CState& s) {
#pragma unroll
  for (int n = 0; n < kModes; ++n) s.h[n] = make_float2(0.0f, 0.0f);
}

__device__ __forceinline__ void cstate_load(CState& s, const float* p) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float4 v = reinterpret_cast<const float4*>(p)[q];
    s.h[2 * q] = make_float2(v.x, v.y);
    s.h[2 * q + 1] = make_float2(v.z, v.w);
  }
}

__device__ __forceinline__ void cstate_store(const CState& s, float* p) {
#pragma unroll
  for (int q = 0; q < 4; ++q)
    reinterpret_cast<float4*>(p)[q] = make_float4(s.h[2 * q].x, s.h[2 * q].y, s.h[2 * q + 1].x, s.h[2 * q + 1].y);
}

// Raw input of channel c at token tau (tau < 0: conv_state0, or zero).
template <typename IO>
__device__ __forceinline__ float cinput_at(const ComplexParams& p, int b, long tau, int c) {
  if (tau >= 0) return to_f32(reinterpret_cast<const IO*>(p.x)[((size_t)b * p.seqlen + tau) * p.d_inner + c]);
  if (p.conv_state0 == nullptr) return 0.0f;
  return to_f32(reinterpret_cast<const IO*>(p.conv_state0)[((size_t)b * 3 + (3 + tau)) * p.d_inner + c]);
}

// grid (n_groups, batch, chunks), 32 threads.  kSummary: chunks 0..n-2 from
// a zero state, no z and no y; stores hloc_j and S_j.  Otherwise: the main
// pass, every chunk from its entering state, y written.
template <typename IO, bool kTrap, bool kSummary>
__global__ void __launch_bounds__(kLanes)
    complex_scan_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_z,
                        const __grid_constant__ CUtensorMap tm_dt, const __grid_constant__ CUtensorMap tm_bc,
                        const __grid_constant__ ComplexParams p) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  MainSmem<IO>& sm = *reinterpret_cast<MainSmem<IO>*>(smem_raw + smem_pad128(smem_raw));
  constexpr bool kY = !kSummary;

  const int lane = threadIdx.x;
  const int c0 = blockIdx.x * kLanes;
  const int b = blockIdx.y;
  const int j = blockIdx.z;
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
  // In the chunked mode the fold (an earlier launch) copied h0 into the
  // carry's chunk-0 slot and v0 into the unused last slot of hloc, so that
  // no CTA of this launch reads h0 or v0, which the last chunk's final_h and
  // final_v may alias.
  const bool folded = !kSummary && p.n_chunks > 1;
  CState st, vp;
  if (kSummary || (j == 0 && !folded && p.h0 == nullptr))
    cstate_zero(st);
  else if (j == 0 && !folded)
    cstate_load(st, p.h0 + sidx);
  else
    cstate_load(st, p.carry + (((size_t)b * p.n_chunks + j) * D + cl) * 16);

  if (!kTrap) cstate_zero(vp);
  float xm3 = cinput_at<IO>(p, b, (long)t_begin - 3, cl);
  float xm2 = cinput_at<IO>(p, b, (long)t_begin - 2, cl);
  float xm1 = cinput_at<IO>(p, b, (long)t_begin - 1, cl);
  if (kTrap) {  // the state input of the token before the chunk
    if (j == 0) {
      if (p.v0 == nullptr)
        cstate_zero(vp);
      else if (folded)
        cstate_load(vp, p.hloc + (((size_t)b * p.n_chunks + p.n_chunks - 1) * D + cl) * 16);
      else
        cstate_load(vp, p.v0 + sidx);
    } else {
      const float xm4 = cinput_at<IO>(p, b, (long)t_begin - 4, cl);
      const float u = silu(conv4(ch.w, ch.bias, xm4, xm3, xm2, xm1));
      const float4* row = reinterpret_cast<const float4*>(p.bc + ((size_t)b * p.seqlen + t_begin - 1) * kBC);
#pragma unroll
      for (int n = 0; n < kModes; ++n) {
        const float4 q = __ldg(row + n);
        vp.h[n] = make_float2(__fmul_rn(q.x, u), __fmul_rn(q.y, u));
      }
    }
  }
  if (kY && j == 0 && p.final_conv_state != nullptr) {
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
#pragma unroll 2
    for (int r = 0; r < rows; ++r) {
      const float xv = to_f32(S.x[r][lane]);
      const float u = silu(conv4(ch.w, ch.bias, xm3, xm2, xm1, xv));
      xm3 = xm2;
      xm2 = xm1;
      xm1 = xv;
      const float dt = softplus(to_f32(S.dt[r][lane]));
      float4 Q[kModes];
      load_quads(&S.bc[r][0], Q);
      const float yss = ctoken<kTrap, kY>(ch, st, vp, u, dt, Q);
      if (kSummary) sdt = __fadd_rn(sdt, dt);
      if (kY) {
        const float gz = silu(to_f32(S.z[r][lane]));
        st_global_if(wy, ytile + (size_t)r * D, from_f32<IO>(gate_out(yss, ch.Dc, u, gz)));
      }
    }
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
  if (!active) return;
  if (kSummary) {
    cstate_store(st, p.hloc + (((size_t)b * p.n_chunks + j) * D + c) * 16);
    p.sdt[((size_t)b * p.n_chunks + j) * D + c] = sdt;
  } else if (j == p.n_chunks - 1) {
    if (p.final_h) cstate_store(st, p.final_h + sidx);
    if (p.final_v) {
      if (!kTrap) {  // Euler keeps no previous input: the last token's, from its inputs
        const float u =
            silu(conv4(ch.w, ch.bias, cinput_at<IO>(p, b, (long)p.seqlen - 4, c), xm3, xm2, xm1));
        const float4* row = reinterpret_cast<const float4*>(p.bc + ((size_t)b * p.seqlen + p.seqlen - 1) * kBC);
#pragma unroll
        for (int n = 0; n < kModes; ++n) {
          const float4 q = __ldg(row + n);
          vp.h[n] = make_float2(__fmul_rn(q.x, u), __fmul_rn(q.y, u));
        }
      }
      cstate_store(vp, p.final_v + sidx);
    }
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
#pragma unroll
    for (int n = 0; n < kModes; ++n) h.h[n] = cmul_add(cexp_step(ch.a2[n], ch.tu[n], ch.tl[n], S), h.h[n], hl.h[n]);
    cstate_store(h, p.carry + (((size_t)b * p.n_chunks + j + 1) * D + c) * 16);
  }
}

}  // namespace mamba
