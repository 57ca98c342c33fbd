// gemm_tc.cuh -- bf16 GEMM on the 5th-generation tensor cores (tcgen05):
// row-major C (M x N) = A (M x K) * W^T (W: N x K, the nn.Linear weight
// layout) [+ bias (N)], fp32 accumulation in tensor memory, bf16 out.
//
// Work decomposition.  Output tiles of 256 x bn (bn: the N extent divided
// evenly into tiles of at most 256, rounded up to 32), each taken by a
// cluster of two CTAs (one per SM; a persistent grid) that compute its two
// 128-row halves: each CTA loads its own rows of A and half of W's bn rows,
// multicast to both, so that a W tile crosses from L2 once per pair.  Tiles
// are taken in row-block order, so that the clusters running at once share
// A's rows and walk W, which stays in L2.  Per CTA, six warps with fixed
// roles:
//   warp 0     the producer: one lane issues the TMA loads of A and W tiles
//              (64 columns of K, 128 B rows, 128-byte swizzle) into a ring of
//              4 shared-memory stages, each released when the MMAs of both
//              CTAs have read it;
//   warp 1     owns the tensor memory (512 columns: two accumulators of 256)
//              and one lane issues the MMAs: per stage four 128 x 256 x 16
//              tcgen05.mma, then a commit that frees the stage (arriving in
//              both CTAs); per tile a commit that hands the accumulator to
//              the epilogue;
//   warps 2-5  the epilogue: each reads its 32 TMEM lanes (tile rows) 32
//              columns at a time, adds the bias, rounds to bf16, writes the
//              32 x 32 chunk into one of two staging buffers of its own and
//              stores it with one TMA store; the accumulator is freed after
//              its last load, and the next tile's MMAs run meanwhile in the
//              other accumulator.
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
  // per epilogue warp, two staging buffers of 32 rows x 32 columns (64-byte
  // rows, 64-byte swizzle) for the TMA stores of C
  __nv_bfloat16 cst[4][2][32 * 32];
  uint64_t full[kGemmStages];
  uint64_t empty[kGemmStages];
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint32_t tmem_base;
};

// Shared-memory matrix descriptor of a K-major tile written by TMA with the
// 128-byte swizzle: rows of 128 bytes, 8-row swizzle atoms 1024 bytes apart
// (the stride byte offset); the leading byte offset is unused in this mode.
__device__ __forceinline__ uint64_t smem_desc_k128(uint32_t saddr) { return umma_desc(saddr, 1024, 2); }

// Instruction descriptor, kind::f16: fp32 accumulator (bits 4-5 = 1), A and
// B bf16 (bits 7-9, 10-12 = 1), both K-major (bits 15, 16 = 0), N / 8 at
// bits 17-22, M / 16 at bits 24-28.
__device__ __forceinline__ uint32_t gemm_idesc(int bn) { return umma_idesc_bf16(kGemmBM, bn, false); }

__device__ __forceinline__ uint32_t smem_pad1024(const void* base) {
  return (1024u - (smem_u32(base) & 1023u)) & 1023u;
}

__device__ __forceinline__ uint32_t pack2_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_w,
                   const __grid_constant__ CUtensorMap tm_c, const __grid_constant__ GemmParams p) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  GemmSmem& sm = *reinterpret_cast<GemmSmem*>(smem_raw + smem_pad1024(smem_raw));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int bn = p.bn;  // the N tile: a multiple of 32, at most kGemmBN
  const int tiles_n = (p.N + bn - 1) / bn;
  // the CTA pair of a cluster takes the two 128-row halves of 256-row tiles
  const uint32_t rank = cluster_ctarank();
  const long tiles = ((p.M + 2 * kGemmBM - 1) / (2 * kGemmBM)) * (long)tiles_n;
  const long first = cluster_id_x(), step = cluster_count_x();
  const int nk = (p.K + kGemmBK - 1) / kGemmBK;  // the loads fill zeros past K
  const uint32_t idesc = gemm_idesc(bn);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kGemmStages; ++s) {
      mbar_init(smem_u32(&sm.full[s]), 1);
      mbar_init(smem_u32(&sm.empty[s]), 2);  // the MMAs of both CTAs of the pair
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&sm.acc_full[b]), 1);
      mbar_init(smem_u32(&sm.acc_empty[b]), 4);  // one arrival per epilogue warp
    }
    fence_mbar_init();
    prefetch_tensormap(&tm_a);
    prefetch_tensormap(&tm_w);
    prefetch_tensormap(&tm_c);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&sm.tmem_base), kGemmTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  cluster_sync();  // both CTAs' barriers are initialised before either multicasts
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  bool ok = true;

  if (warp == 0) {
    if (lane == 0) {  // producer
      const uint64_t keep = l2_policy_evict_last();  // W: read by every row block
      uint32_t it = 0;
      for (long t = first; t < tiles && ok; t += step) {
        const int m0 = (int)(t / tiles_n) * 2 * kGemmBM + (int)rank * kGemmBM;
        const int n0 = (int)(t % tiles_n) * bn;
        const int half = bn / 2;  // the W rows this CTA loads for both
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int s = (int)(it % kGemmStages);
          const uint32_t ph = (it / kGemmStages) & 1u;
          // stage s is free in both CTAs (its empty barrier counts both MMAs)
          if (!mbar_wait_bounded(smem_u32(&sm.empty[s]), ph ^ 1u, p.timeout_ns)) {
            ok = false;
            break;
          }
          const uint32_t bar = smem_u32(&sm.full[s]);
          mbar_arrive_expect_tx(bar, (kGemmBM + bn) * kGemmBK * 2);  // own A, both halves of W
          tma_load_2d(smem_u32(&sm.a[s][0]), &tm_a, kb * kGemmBK, m0, bar);  // A: reused by the row block's tiles
          tma_load_2d_mc(smem_u32(&sm.b[s][(size_t)rank * half * kGemmBK]), &tm_w, kb * kGemmBK, n0 + (int)rank * half,
                         bar, 0x3, keep);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {  // MMA issuer
      uint32_t it = 0, i = 0;
      for (long t = first; t < tiles && ok; t += step, ++i) {
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
            tc_mma_f16(d, ad + 2 * kk, bd + 2 * kk, idesc, (kb | kk) != 0);
          tc_commit_mc(smem_u32(&sm.empty[s]), 0x3);  // frees stage s in both CTAs
        }
        if (!ok) break;
        tc_commit(smem_u32(&sm.acc_full[buf]));
      }
    }
  } else {  // epilogue, warps 2..5: warp w reads TMEM lanes 32 (w % 4) .. + 31
    const int q = warp & 3;
    const __nv_bfloat16* bias = static_cast<const __nv_bfloat16*>(p.bias);
    const uint64_t out_policy = l2_policy_evict_first();  // C: written once
    uint32_t i = 0, sb = 0;
    for (long t = first; t < tiles; t += step, ++i) {
      const uint32_t buf = i & 1u;
      const bool mine = mbar_wait_bounded(smem_u32(&sm.acc_full[buf]), (i >> 1) & 1u, p.timeout_ns);
      if (!__all_sync(0xffffffffu, mine)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int m0 = (int)(t / tiles_n) * 2 * kGemmBM + (int)rank * kGemmBM;
      const int n0 = (int)(t % tiles_n) * bn;
      const uint32_t tbase = tmem + ((uint32_t)(32 * q) << 16) + buf * kGemmBN;
      const int chunks = min(bn, p.N - n0 + 31) / 32;  // 32-column chunks holding valid columns
#pragma unroll 1
      for (int c = 0; c < chunks; ++c) {
        uint32_t r[32];
        tmem_ld_32cols(tbase + 32 * c, r);
        if (c == chunks - 1) {  // the accumulator is in registers: hand it back to the MMAs
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&sm.acc_empty[buf]));
        }
        const int col0 = n0 + 32 * c;
        // the chunk's 32 bias values (the same for every lane: broadcast
        // loads), four 16-byte vectors where the chunk lies inside N
        uint32_t bw[16];
#pragma unroll
        for (int g = 0; g < 16; ++g) bw[g] = 0u;
        if (bias) {
          if (col0 + 32 <= p.N) {
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              const uint4 b4 = __ldg(reinterpret_cast<const uint4*>(bias + col0) + v);
              bw[4 * v] = b4.x;
              bw[4 * v + 1] = b4.y;
              bw[4 * v + 2] = b4.z;
              bw[4 * v + 3] = b4.w;
            }
          } else {
#pragma unroll
            for (int g = 0; g < 16; ++g) {
              const uint32_t lo = col0 + 2 * g < p.N ? __bfloat16_as_ushort(bias[col0 + 2 * g]) : 0u;
              const uint32_t hi = col0 + 2 * g + 1 < p.N ? __bfloat16_as_ushort(bias[col0 + 2 * g + 1]) : 0u;
              bw[g] = lo | (hi << 16);
            }
          }
        }
        uint32_t pk[16];
#pragma unroll
        for (int g = 0; g < 16; ++g) {
          float lo = __uint_as_float(r[2 * g]), hi = __uint_as_float(r[2 * g + 1]);
          if (bias) {
            lo = __fadd_rn(lo, __uint_as_float(bw[g] << 16));
            hi = __fadd_rn(hi, __uint_as_float(bw[g] & 0xffff0000u));
          }
          pk[g] = pack2_bf16(lo, hi);
        }
        // this lane's row of the chunk into the staging buffer (64-byte
        // swizzle: the 16-byte piece j of row r sits at piece j ^ ((r / 2) % 4)),
        // then one TMA store of the 32 x 32 chunk (clipped at the matrix edge)
        const uint32_t st = smem_u32(&sm.cst[q][sb][0]);
        if (lane == 0) bulk_wait_read<1>();  // the store that last read this buffer is done reading
        __syncwarp();
#pragma unroll
        for (int j = 0; j < 4; ++j)
          st_shared_v4(st + lane * 64 + 16 * (j ^ ((lane >> 1) & 3)), pk[4 * j], pk[4 * j + 1], pk[4 * j + 2],
                       pk[4 * j + 3]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_2d(&tm_c, col0, m0 + 32 * q, st, out_policy);
          bulk_commit();
        }
        sb ^= 1u;
      }
    }
    if (lane == 0) bulk_wait_all();  // every store has left shared memory before the CTA ends
  }

  if (!ok) report_error(4u);  // MAMBA_ERR_TIMEOUT
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();  // the warp-wide tcgen05 operations need the whole warp converged
    tc_fence_after();
    tmem_dealloc(tmem, kGemmTmemCols);
  }
  cluster_sync();  // the peer's last arrivals on this CTA's barriers have landed
}

}  // namespace mamba
