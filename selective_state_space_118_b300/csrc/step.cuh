// step.cuh -- decode: one token through the layer, state updated in place.
//
// The constant-memory recurrence of the lesson's "Um SSM em uma pagina":
// y_t needs only h_{t-1}, the last three inputs and x_t.  Two lanes serve one
// (batch row, channel), lane q holding states 8q..8q+7, each reading and
// writing its half of h with one 32-byte access, so that a warp instruction
// moves a contiguous 1 KB of h (a lane-per-channel layout touches 16 cache
// lines per instruction and throttles the load/store unit; four lanes per
// channel issue more instructions and measured slower).  The lanes of a channel all compute its
// conv, SiLU, softplus and gate (cheap: the step is HBM-bound, not
// arithmetic-bound); their read-out chains (p_lo on lane 0, p_hi on lane 1)
// meet through one exchange in the fixed order of state16_readout.  The arithmetic is ssm_math.cuh's, in the
// same order as one token of scan_fwd_kernel, so a sequence of steps
// reproduces a single-pass scan bit for bit.  h is 128 of the ~144 bytes
// moved per channel and row: a CTA's block of h (64 channels of one row,
// 4 KB contiguous) comes in by one bulk copy and leaves by one bulk store,
// which keeps more bytes in flight per SM than per-lane loads do.
#pragma once
#include <cuda_bf16.h>

#include "params.h"
#include "ptx.cuh"
#include "scan_fwd.cuh"
#include "ssm_math.cuh"

namespace mamba {

constexpr int kStepThreads = 128;
constexpr int kLPC = 2;                       // lanes per (row, channel)
constexpr int kLS = kN / kLPC;                // states per lane: 8
constexpr int kStepChannels = kStepThreads / kLPC;

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// kLS consecutive I/O values (part of a B or C row) as fp32.
__device__ __forceinline__ void load_part(const float* p, float4 (&v)[kLS / 4]) {
#pragma unroll
  for (int q = 0; q < kLS / 4; ++q) v[q] = __ldg(reinterpret_cast<const float4*>(p) + q);
}

__device__ __forceinline__ void load_part(const __nv_bfloat16* p, float4 (&v)[kLS / 4]) {
  if constexpr (kLS == 8) {
    const uint4 a = __ldg(reinterpret_cast<const uint4*>(p));
    v[0] = make_float4(bf16_lo(a.x), bf16_hi(a.x), bf16_lo(a.y), bf16_hi(a.y));
    v[1] = make_float4(bf16_lo(a.z), bf16_hi(a.z), bf16_lo(a.w), bf16_hi(a.w));
  } else {
    const uint2 a = __ldg(reinterpret_cast<const uint2*>(p));
    v[0] = make_float4(bf16_lo(a.x), bf16_hi(a.x), bf16_lo(a.y), bf16_hi(a.y));
  }
}

// grid (ceil(D / kStepChannels), batch), kStepThreads threads: kLPC
// consecutive threads = one channel of one batch row.
template <typename IO>
__global__ void __launch_bounds__(kStepThreads) step_kernel(const __grid_constant__ StepParams p) {
  __shared__ __align__(128) float hs[kStepChannels * kN];
  __shared__ __align__(8) uint64_t hbar;
  griddep_wait();
  griddep_launch_dependents();
  const int D = p.d_inner;
  const int q = threadIdx.x % kLPC;
  const int c0 = blockIdx.x * kStepChannels;
  const int c = c0 + threadIdx.x / kLPC;
  const int b = blockIdx.y;
  const bool valid = c < D;  // the lanes of a channel share it
  const int cl = valid ? c : D - 1;
  const size_t ch = (size_t)b * D + cl;
  const uint32_t hbytes = (uint32_t)min(kStepChannels, D - c0) * kN * 4;  // this block's channels of h
  float* hblk = p.h + ((size_t)b * D + c0) * kN;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&hbar), 1);
    fence_mbar_init();
    mbar_arrive_expect_tx(smem_u32(&hbar), hbytes);
    bulk_load(smem_u32(hs), hblk, hbytes, smem_u32(&hbar));
  }
  __syncthreads();

  float4 hv[kLS / 4], Bv[kLS / 4], Cv[kLS / 4];
  const IO* cs = reinterpret_cast<const IO*>(p.conv_state) + (size_t)b * 3 * D + cl;
  const IO r0 = cs[0], r1 = cs[D], r2 = cs[2 * (size_t)D];
  const IO rx = __ldg(reinterpret_cast<const IO*>(p.x_t) + ch);
  const float zv = to_f32(__ldg(reinterpret_cast<const IO*>(p.z_t) + ch));
  const float dr = to_f32(__ldg(reinterpret_cast<const IO*>(p.dt_raw_t) + ch));
  load_part(reinterpret_cast<const IO*>(p.B_t) + (size_t)b * kN + kLS * q, Bv);
  load_part(reinterpret_cast<const IO*>(p.C_t) + (size_t)b * kN + kLS * q, Cv);
  float4 al[kLS / 4];
  load_part(p.A_log + (size_t)cl * kN + kLS * q, al);
  const float4 w = __ldg(reinterpret_cast<const float4*>(p.conv_w + (size_t)cl * 4));
  const float bias = p.conv_b ? __ldg(p.conv_b + cl) : 0.0f;
  const float Dc = __ldg(p.Dskip + cl);
  if (!__syncthreads_and(mbar_wait_bounded(smem_u32(&hbar), 0, p.timeout_ns))) {
    if (threadIdx.x == 0) report_error(4u);  // MAMBA_ERR_TIMEOUT
    return;
  }
  {
    const float4* hp4 = reinterpret_cast<const float4*>(hs + (threadIdx.x / kLPC) * kN + kLS * q);
#pragma unroll
    for (int k = 0; k < kLS / 4; ++k) hv[k] = hp4[k];
  }

  const float u = silu(conv4(w, bias, to_f32(r0), to_f32(r1), to_f32(r2), to_f32(rx)));
  const float dt = softplus(dr);
  const float gz = silu(zv);
  const float2 d2 = make_float2(dt, dt);
  const float dtu = __fmul_rn(dt, u);
  const float2 u2 = make_float2(dtu, dtu);
  float2 hp[kLS / 2];
#pragma unroll
  for (int k = 0; k < kLS / 4; ++k) {  // one group of 4 states: pairs h01, h23
    const float2 a01 = make_float2(a2_from_log(al[k].x), a2_from_log(al[k].y));
    const float2 a23 = make_float2(a2_from_log(al[k].z), a2_from_log(al[k].w));
    const float2 x01 = __fmul2_rn(d2, a01), x23 = __fmul2_rn(d2, a23);
    const float2 e01 = make_float2(ex2_approx(x01.x), ex2_approx(x01.y));
    const float2 e23 = make_float2(ex2_approx(x23.x), ex2_approx(x23.y));
    float2 h01 = make_float2(hv[k].x, hv[k].y), h23 = make_float2(hv[k].z, hv[k].w);
    h01 = __ffma2_rn(e01, h01, __fmul2_rn(u2, make_float2(Bv[k].x, Bv[k].y)));
    h23 = __ffma2_rn(e23, h23, __fmul2_rn(u2, make_float2(Bv[k].z, Bv[k].w)));
    hv[k] = make_float4(h01.x, h01.y, h23.x, h23.y);
    hp[2 * k] = h01;
    hp[2 * k + 1] = h23;
  }
  // this lane's half of the read-out, then T_lo + T_hi
  const float2 pr = readout_half(hp, Cv);
  const float2 po = make_float2(__shfl_xor_sync(0xffffffffu, pr.x, 1), __shfl_xor_sync(0xffffffffu, pr.y, 1));
  const float ss = q == 0 ? readout_join(pr, po) : readout_join(po, pr);
  {
    float4* hp4 = reinterpret_cast<float4*>(hs + (threadIdx.x / kLPC) * kN + kLS * q);
#pragma unroll
    for (int k = 0; k < kLS / 4; ++k) hp4[k] = hv[k];
  }
  fence_proxy_async_smem();
  __syncthreads();
  if (threadIdx.x == 0) {
    bulk_store(hblk, smem_u32(hs), hbytes);
    bulk_commit();
  }
  if (valid) {
    if (q == 0) {
      reinterpret_cast<IO*>(p.y_t)[ch] = from_f32<IO>(gate_out(ss, Dc, u, gz));
      IO* csw = reinterpret_cast<IO*>(p.conv_state) + (size_t)b * 3 * D + c;
      csw[0] = r1;
      csw[D] = r2;
      csw[2 * (size_t)D] = rx;
    }
  }
  if (threadIdx.x == 0) bulk_wait_read<0>();  // the block of h has left shared memory
}

}  // namespace mamba
