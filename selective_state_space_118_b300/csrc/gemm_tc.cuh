// gemm_tc.cuh -- bf16 GEMM on the 5th-generation tensor cores (tcgen05):
// row-major C (M x N) = A (M x K) * W^T (W: N x K, the nn.Linear weight
// layout) [+ bias (N)], fp32 accumulation in tensor memory, bf16 out.
//
// Work decomposition.  Output tiles of 128 x 256, taken by a persistent grid
// (one CTA per SM) in row-block order, so that the CTAs running at once share
// A's row block and walk W, which stays in L2.  Per CTA, six warps with fixed
// roles:
//   warp 0     the producer: one lane issues the TMA loads of A and W tiles
//              (64 columns of K, 128 B rows, 128-byte swizzle) into a ring of
//              4 shared-memory stages, each released by the MMA that read it;
//   warp 1     owns the tensor memory (512 columns: two accumulators of 256)
//              and one lane issues the MMAs: per stage four 128 x 256 x 16
//              tcgen05.mma, then a commit that frees the stage; per tile a
//              commit that hands the accumulator to the epilogue;
//   warps 2-5  the epilogue: each reads its 32 TMEM lanes (tile rows) 32
//              columns at a time, adds the bias, rounds to bf16 and stores
//              64 contiguous bytes per row, then frees the accumulator; the
//              next tile's MMAs run meanwhile in the other accumulator.
// Every wait on an mbarrier is bounded (wait_timeout_ns); a wait that gives
// up records MAMBA_ERR_TIMEOUT and its role stops, the others give up in
// turn, and the tensor memory is always released.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>

#include <cstdint>

#include "params.h"
#include "ptx.cuh"
#include "scan_fwd.cuh"

namespace mamba {

constexpr int kGemmBM = 128;
constexpr int kGemmBN = 256;
constexpr int kGemmBK = 64;  // one 128-byte swizzle row of bf16
constexpr int kGemmStages = 4;
constexpr int kGemmThreads = 192;
constexpr uint32_t kGemmTmemCols = 2 * kGemmBN;

struct GemmSmem {
  __nv_bfloat16 a[kGemmStages][kGemmBM * kGemmBK];  // 16 KB per stage
  __nv_bfloat16 b[kGemmStages][kGemmBN * kGemmBK];  // 32 KB per stage
  uint64_t full[kGemmStages];
  uint64_t empty[kGemmStages];
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint32_t tmem_base;
};

// Shared-memory matrix descriptor of a K-major tile written by TMA with the
// 128-byte swizzle: rows of 128 bytes, 8-row swizzle atoms 1024 bytes apart
// (the stride byte offset); the leading byte offset is unused in this mode.
__device__ __forceinline__ uint64_t smem_desc_k128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);  // start address, 16-byte units
  d |= (uint64_t)1 << 16;                   // leading byte offset (unused)
  d |= (uint64_t)(1024 >> 4) << 32;         // stride byte offset
  d |= (uint64_t)1 << 46;                   // descriptor version
  d |= (uint64_t)2 << 61;                   // 128-byte swizzle
  return d;
}

// Instruction descriptor, kind::f16: fp32 accumulator (bits 4-5 = 1), A and
// B bf16 (bits 7-9, 10-12 = 1), both K-major (bits 15, 16 = 0), N / 8 at
// bits 17-22, M / 16 at bits 24-28.
constexpr uint32_t kGemmIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kGemmBN >> 3) << 17) |
                                ((uint32_t)(kGemmBM >> 4) << 24);

__device__ __forceinline__ uint32_t smem_pad1024(const void* base) {
  return (1024u - (smem_u32(base) & 1023u)) & 1023u;
}

__device__ __forceinline__ uint32_t pack2_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_w,
                   const __grid_constant__ GemmParams p) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  GemmSmem& sm = *reinterpret_cast<GemmSmem*>(smem_raw + smem_pad1024(smem_raw));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int tiles_n = (p.N + kGemmBN - 1) / kGemmBN;
  const long tiles = ((p.M + kGemmBM - 1) / kGemmBM) * (long)tiles_n;
  const int nk = p.K / kGemmBK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kGemmStages; ++s) {
      mbar_init(smem_u32(&sm.full[s]), 1);
      mbar_init(smem_u32(&sm.empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&sm.acc_full[b]), 1);
      mbar_init(smem_u32(&sm.acc_empty[b]), 4);  // one arrival per epilogue warp
    }
    fence_mbar_init();
    prefetch_tensormap(&tm_a);
    prefetch_tensormap(&tm_w);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&sm.tmem_base), kGemmTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  bool ok = true;

  if (warp == 0) {
    if (lane == 0) {  // producer
      uint32_t it = 0;
      for (long t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
        const int m0 = (int)(t / tiles_n) * kGemmBM;
        const int n0 = (int)(t % tiles_n) * kGemmBN;
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int s = (int)(it % kGemmStages);
          const uint32_t ph = (it / kGemmStages) & 1u;
          if (!mbar_wait_bounded(smem_u32(&sm.empty[s]), ph ^ 1u, p.timeout_ns)) {
            ok = false;
            break;
          }
          const uint32_t bar = smem_u32(&sm.full[s]);
          mbar_arrive_expect_tx(bar, (kGemmBM + kGemmBN) * kGemmBK * 2);
          tma_load_2d(smem_u32(&sm.a[s][0]), &tm_a, kb * kGemmBK, m0, bar);
          tma_load_2d(smem_u32(&sm.b[s][0]), &tm_w, kb * kGemmBK, n0, bar);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {  // MMA issuer
      uint32_t it = 0, i = 0;
      for (long t = blockIdx.x; t < tiles && ok; t += gridDim.x, ++i) {
        const uint32_t buf = i & 1u;
        if (!mbar_wait_bounded(smem_u32(&sm.acc_empty[buf]), ((i >> 1) & 1u) ^ 1u, p.timeout_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem + buf * kGemmBN;
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int s = (int)(it % kGemmStages);
          if (!mbar_wait_bounded(smem_u32(&sm.full[s]), (it / kGemmStages) & 1u, p.timeout_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t ad = smem_desc_k128(smem_u32(&sm.a[s][0]));
          const uint64_t bd = smem_desc_k128(smem_u32(&sm.b[s][0]));
#pragma unroll
          for (int kk = 0; kk < kGemmBK / 16; ++kk)  // 16 elements = 32 bytes further along the row
            tc_mma_f16(d, ad + 2 * kk, bd + 2 * kk, kGemmIdesc, (kb | kk) != 0);
          tc_commit(smem_u32(&sm.empty[s]));
        }
        if (!ok) break;
        tc_commit(smem_u32(&sm.acc_full[buf]));
      }
    }
  } else {  // epilogue, warps 2..5: warp w reads TMEM lanes 32 (w % 4) .. + 31
    const int q = warp & 3;
    uint32_t i = 0;
    for (long t = blockIdx.x; t < tiles; t += gridDim.x, ++i) {
      const uint32_t buf = i & 1u;
      const bool mine = mbar_wait_bounded(smem_u32(&sm.acc_full[buf]), (i >> 1) & 1u, p.timeout_ns);
      if (!__all_sync(0xffffffffu, mine)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const long row = (t / tiles_n) * kGemmBM + 32 * q + lane;
      const int n0 = (int)(t % tiles_n) * kGemmBN;
      __nv_bfloat16* crow = static_cast<__nv_bfloat16*>(p.C) + row * (long)p.ldc;
      const __nv_bfloat16* bias = static_cast<const __nv_bfloat16*>(p.bias);
#pragma unroll 1
      for (int c = 0; c < kGemmBN / 32; ++c) {
        const int col0 = n0 + 32 * c;
        if (col0 >= p.N) break;  // warp-uniform
        uint32_t r[32];
        tmem_ld_32cols(tmem + ((uint32_t)(32 * q) << 16) + buf * kGemmBN + 32 * c, r);
        float v[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
        if (bias) {
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (col0 + j < p.N) v[j] = __fadd_rn(v[j], __bfloat162float(bias[col0 + j]));
        }
        if (row < p.M) {
          if (col0 + 32 <= p.N) {
#pragma unroll
            for (int g = 0; g < 4; ++g)
              reinterpret_cast<uint4*>(crow + col0)[g] =
                  make_uint4(pack2_bf16(v[8 * g], v[8 * g + 1]), pack2_bf16(v[8 * g + 2], v[8 * g + 3]),
                             pack2_bf16(v[8 * g + 4], v[8 * g + 5]), pack2_bf16(v[8 * g + 6], v[8 * g + 7]));
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (col0 + j < p.N) crow[col0 + j] = __float2bfloat16_rn(v[j]);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sm.acc_empty[buf]));
    }
  }

  if (!ok) report_error(4u);  // MAMBA_ERR_TIMEOUT
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();  // the warp-wide tcgen05 operations need the whole warp converged
    tc_fence_after();
    tmem_dealloc(tmem, kGemmTmemCols);
  }
}

}  // namespace mamba
