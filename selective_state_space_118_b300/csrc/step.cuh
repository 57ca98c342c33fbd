// step.cuh -- decode: one token through the layer, state updated in place.
//
// The constant-memory recurrence of the lesson's "Um SSM em uma pagina":
// y_t needs only h_{t-1}, the last three inputs and x_t.  Four lanes serve one
// channel, each holding four of its 16 fp32 states (one 16-byte load and one
// 16-byte store of h per lane, so a warp moves 8 channels x 64 B of h
// contiguously).  The per-token arithmetic is ssm_math.cuh's, in the same
// order as one token of scan_fwd_kernel, so a sequence of steps reproduces a
// single-pass scan bit for bit.  The step is HBM-bound: h is 128 of the ~144
// bytes moved per channel.
#pragma once
#include <cuda_bf16.h>

#include "params.h"
#include "ssm_math.cuh"

namespace mamba {

constexpr int kStepThreads = 256;

template <typename IO>
__device__ __forceinline__ float4 load4_io(const IO* p) {
  return make_float4(to_f32(p[0]), to_f32(p[1]), to_f32(p[2]), to_f32(p[3]));
}

template <typename IO>
__global__ void __launch_bounds__(kStepThreads) step_kernel(const __grid_constant__ StepParams p) {
  const long gtid = (long)blockIdx.x * kStepThreads + threadIdx.x;
  const long ch = gtid >> 2;  // flattened (b, c); B*D is a multiple of 16, so whole warps exit together
  if (ch >= (long)p.batch * p.d_inner) return;
  const int g = threadIdx.x & 3;
  const int D = p.d_inner;
  const int b = (int)(ch / D);
  const int c = (int)(ch - (long)b * D);

  float* hp = p.h + ch * kN + 4 * g;
  const float4 h = *reinterpret_cast<const float4*>(hp);
  IO* cs = reinterpret_cast<IO*>(p.conv_state);
  const size_t cs0 = ((size_t)b * 3) * D + c;
  const IO r0 = cs[cs0], r1 = cs[cs0 + D], r2 = cs[cs0 + 2 * (size_t)D];
  const IO rx = reinterpret_cast<const IO*>(p.x_t)[ch];
  const float zv = to_f32(reinterpret_cast<const IO*>(p.z_t)[ch]);
  const float dr = to_f32(reinterpret_cast<const IO*>(p.dt_raw_t)[ch]);
  const float4 w = *reinterpret_cast<const float4*>(p.conv_w + (size_t)c * 4);
  const float bias = p.conv_b ? p.conv_b[c] : 0.0f;
  const float Dc = p.Dskip[c];
  const float4 al = *reinterpret_cast<const float4*>(p.A_log + (size_t)c * kN + 4 * g);
  const float4 Bv = load4_io(reinterpret_cast<const IO*>(p.B_t) + (size_t)b * kN + 4 * g);
  const float4 Cv = load4_io(reinterpret_cast<const IO*>(p.C_t) + (size_t)b * kN + 4 * g);

  const float x0 = to_f32(rx);
  const float u = silu(conv4(w, bias, to_f32(r0), to_f32(r1), to_f32(r2), x0));
  const float dt = softplus(dr);
  const float dtu = __fmul_rn(dt, u);
  const float2 a01 = make_float2(a2_from_log(al.x), a2_from_log(al.y));
  const float2 a23 = make_float2(a2_from_log(al.z), a2_from_log(al.w));
  State4 st;
  st.h01 = make_float2(h.x, h.y);
  st.h23 = make_float2(h.z, h.w);
  const float part = state4_step(st, a01, a23, dt, dtu, Bv, Cv);
  const float S = group4_sum(part);
  *reinterpret_cast<float4*>(hp) = make_float4(st.h01.x, st.h01.y, st.h23.x, st.h23.y);
  if (g == 0) {
    reinterpret_cast<IO*>(p.y_t)[ch] = from_f32<IO>(gate_out(S, Dc, u, silu(zv)));
    cs[cs0] = r1;
    cs[cs0 + D] = r2;
    cs[cs0 + 2 * (size_t)D] = rx;
  }
}

}  // namespace mamba
