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
// NM < kModes: only modes 0..NM-1 advance (the carry walk's modes whose
// weight to the boundary is still above the drop bound; the others stay).
template <bool kTrap, bool kRead, int NM = kModes>
__device__ __forceinline__ float ctoken(const CChannel& ch, CState& st, CState& vp, float u, float dt,
                                        const float4 (&Q)[kModes]) {
  const float hdt = __fmul_rn(0.5f, dt);
  float2 acc = make_float2(0.0f, 0.0f);
#pragma unroll
  for (int n = 0; n < NM; ++n) {
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
  const float4* row = reinterpret_cast<const float4*>(p.bc + ((size_t)b * p.seqlen + t0 - 1) * kBC);
#pragma unroll
  for (int n = 0; n < kModes; ++n) {
    const float4 q = __ldg(row + n);
    vp.h[n] = make_float2(__fmul_rn(q.x, u), __fmul_rn(q.y, u));
  }
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
      for (int q = 0; q < 4; ++q) {  // from L2: written by another SM during this launch
        const float4 v = __ldcg(src + q);
        st.h[2 * q] = make_float2(v.x, v.y);
        st.h[2 * q + 1] = make_float2(v.z, v.w);
      }
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
        const float4* row = reinterpret_cast<const float4*>(p.bc + ((size_t)b * p.seqlen + p.seqlen - 1) * kBC);
#pragma unroll
        for (int n = 0; n < kModes; ++n) {
          const float4 q = __ldg(row + n);
          vp.h[n] = make_float2(__fmul_rn(q.x, u), __fmul_rn(q.y, u));
        }
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

// One full tile of a carry piece: modes 0..NM-1 advanced, the dt summed.
template <typename IO, bool kTrap, int NM>
__device__ __forceinline__ void ccarry_tile(const SummaryStage<IO>& S, int lane, const CChannel& ch, CState& st,
                                            CState& vp, float& sdt, float& xm3, float& xm2, float& xm1) {
#pragma unroll 2
  for (int r = 0; r < kT; ++r) {
    const float xv = to_f32(S.x[r][lane]);
    const float u = silu(conv4(ch.w, ch.bias, xm3, xm2, xm1, xv));
    xm3 = xm2;
    xm2 = xm1;
    xm1 = xv;
    const float dt = softplus(to_f32(S.dt[r][lane]));
    float4 Q[kModes];
    load_quads(&S.bc[r][0], Q);
    (void)ctoken<kTrap, false, NM>(ch, st, vp, u, dt, Q);
    sdt = __fadd_rn(sdt, dt);
  }
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
  float a2max = ch.a2[0];  // the slowest decay of this channel
#pragma unroll
  for (int n = 1; n < kModes; ++n) a2max = fmaxf(a2max, ch.a2[n]);
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

  int n_modes = kModes;  // leading modes the current piece advances
  bool ok = true, done = false;
  int k = 0;
  for (; k < n_tiles; ++k) {
    const int s = k % kStages;
    const SummaryStage<IO>& S = sm.stage[s];
    const bool mine = mbar_wait_bounded(smem_u32(&sm.full[s]), (k / kStages) & 1, p.timeout_ns);
    ok = __all_sync(0xffffffffu, mine);
    if (!ok) break;
    if (n_modes == 1)
      ccarry_tile<IO, kTrap, 1>(S, lane, ch, st, vp, sdt, xm3, xm2, xm1);
    else if (n_modes == 2)
      ccarry_tile<IO, kTrap, 2>(S, lane, ch, st, vp, sdt, xm3, xm2, xm1);
    else if (n_modes <= 4)
      ccarry_tile<IO, kTrap, 4>(S, lane, ch, st, vp, sdt, xm3, xm2, xm1);
    else
      ccarry_tile<IO, kTrap, 8>(S, lane, ch, st, vp, sdt, xm3, xm2, xm1);
    __syncwarp();  // every lane is done with stage s
    if (lane == 0 && k + kStages < n_tiles)
      issue_carry_tile<IO>(sm, s, &tm_x, &tm_dt, &tm_bc, c0, wk.tile_of(k + kStages), b);
    if (--left == 0) {  // piece done: acc += W hloc, W from the piece's end to the boundary
#pragma unroll
      for (int n = 0; n < kModes; ++n)
        acc.h[n] = cmul_add(cexp_step(ch.a2[n], ch.tu[n], ch.tl[n], s_after), st.h[n], acc.h[n]);
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
        // nothing from here on: the piece advances the leading ones up to
        // the last mode still above it
        if ((p.flags & kFlagExactCarry) == 0) {
          int last = -1;
#pragma unroll
          for (int n = 0; n < kModes; ++n)
            if (__fmul_rn(ch.a2[n], s_after) >= kCarryDropLog2) last = n;
          n_modes = __reduce_max_sync(0xffffffffu, active ? last + 1 : 0);
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
        for (int q = 0; q < 4; ++q) {
          const float4 v = __ldcg(src + q);
          prev.h[2 * q] = make_float2(v.x, v.y);
          prev.h[2 * q + 1] = make_float2(v.z, v.w);
        }
      }
    }
#pragma unroll
    for (int n = 0; n < kModes; ++n)
      acc.h[n] = cmul_add(cexp_step(ch.a2[n], ch.tu[n], ch.tl[n], s_after), prev.h[n], acc.h[n]);
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
#pragma unroll
    for (int n = 0; n < kModes; ++n) h.h[n] = cmul_add(cexp_step(ch.a2[n], ch.tu[n], ch.tl[n], S), h.h[n], hl.h[n]);
    cstate_store(h, p.carry + (((size_t)b * p.n_chunks + j + 1) * D + c) * 16);
  }
}

}  // namespace mamba
