// step.cuh -- decode: one token through the layer, state updated in place.
//
// The constant-memory recurrence of the lesson's "Um SSM em uma pagina":
// y_t needs only h_{t-1}, the last three inputs and x_t.  One thread serves
// one (batch row, channel) and holds its 16 fp32 states in registers: it reads
// and writes its 64 bytes of h as four 16-byte accesses (a warp moves 32
// channels x 64 B contiguously).  The per-token arithmetic is ssm_math.cuh's,
// in the same order as one token of scan_fwd_kernel, so a sequence of steps
// reproduces a single-pass scan bit for bit.  The step is HBM-bound: h is 128
// of the ~144 bytes moved per channel.
#pragma once
#include <cuda_bf16.h>

#include "params.h"
#include "ssm_math.cuh"

namespace mamba {

constexpr int kStepThreads = 128;

template <typename IO>
__device__ __forceinline__ void load16_io(const IO* p, float4 (&v)[4]) {
#pragma unroll
  for (int q = 0; q < 4; ++q)
    v[q] = make_float4(to_f32(p[4 * q]), to_f32(p[4 * q + 1]), to_f32(p[4 * q + 2]), to_f32(p[4 * q + 3]));
}

// grid (ceil(D / 128), batch), 128 threads: thread = channel of one batch row.
template <typename IO>
__global__ void __launch_bounds__(kStepThreads) step_kernel(const __grid_constant__ StepParams p) {
  const int D = p.d_inner;
  const int c = blockIdx.x * kStepThreads + threadIdx.x;
  const int b = blockIdx.y;
  if (c >= D) return;
  const size_t ch = (size_t)b * D + c;

  float* hp = p.h + ch * kN;
  State16 st;
  state16_load(st, hp);
  IO* cs = reinterpret_cast<IO*>(p.conv_state) + (size_t)b * 3 * D + c;
  const IO r0 = cs[0], r1 = cs[D], r2 = cs[2 * (size_t)D];
  const IO rx = reinterpret_cast<const IO*>(p.x_t)[ch];
  const float zv = to_f32(reinterpret_cast<const IO*>(p.z_t)[ch]);
  const float dr = to_f32(reinterpret_cast<const IO*>(p.dt_raw_t)[ch]);
  float4 Bv[4], Cv[4];
  load16_io(reinterpret_cast<const IO*>(p.B_t) + (size_t)b * kN, Bv);
  load16_io(reinterpret_cast<const IO*>(p.C_t) + (size_t)b * kN, Cv);
  Channel chn;
  load_channel(chn, p.A_log, p.conv_w, p.conv_b, p.Dskip, c);

  const float u = silu(conv4(chn.w, chn.bias, to_f32(r0), to_f32(r1), to_f32(r2), to_f32(rx)));
  const float dt = softplus(dr);
  const float gz = silu(zv);
  state16_advance(st, chn.a2, dt, __fmul_rn(dt, u), Bv);
  const float yv = gate_out(state16_readout(st, Cv), chn.Dc, u, gz);
  state16_store(st, hp);
  reinterpret_cast<IO*>(p.y_t)[ch] = from_f32<IO>(yv);
  cs[0] = r1;
  cs[D] = r2;
  cs[2 * (size_t)D] = rx;
}

}  // namespace mamba
