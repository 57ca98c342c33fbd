// gemm_tc.cuh -- bf16 GEMM on the 5th-generation tensor cores (tcgen05):
// row-major C (M x N) = A (M x K) * W^T (W: N x K, the nn.Linear weight
// layout) [+ bias (N)], fp32 accumulation in tensor memory, bf16 out.
//
// Work decomposition.  Output tiles of 256 x bn (bn: the N extent divided
// evenly into tiles of at most 256, rounded up to 32), each taken by a
// cluster of two CTAs (one per SM; a persistent grid) acting as one pair MMA
// (cta_group::2, M = 256): each CTA loads its own 128 rows of A and half of
// W's bn rows, and the tensor cores of both SMs read both halves, so a stage
// holds 32 KB per CTA and six stages fit.  Tiles are taken in groups of 8
// row blocks, column by column within a group: the ~74 pairs running at once
// cover 8 row blocks x ~9 column tiles, so each slice of W they load is read
// by ~8 pairs at about the same time, and W comes from DRAM once per group
// rather than relying on all of it staying in L2.  Per CTA, ten warps with
// fixed roles:
//   warp 0     the producer: one lane issues the TMA loads of A and W tiles
//              (64 columns of K, 128 B rows, 128-byte swizzle) into a ring of
//              6 shared-memory stages; both CTAs' loads of a stage complete on
//              rank 0's barrier, and a stage is released in both CTAs when
//              the MMAs have read it;
//   warp 1     owns the tensor memory (512 columns in each SM: two
//              accumulators of 256); in rank 0 one lane issues the MMAs: per
//              stage four 256 x bn x 16 pair MMAs, then a commit that frees
//              the stage (arriving in both CTAs); per tile a commit that hands
//              the accumulator to both CTAs' epilogues;
//   warps 2-9  the epilogue, two warps per quarter of the TMEM lanes (tile
//              rows) taking alternate 32-column chunks: each reads a chunk,
//              adds the bias, rounds to bf16, writes the 32 x 32 chunk into
//              one of two staging buffers of its own and stores it with one
//              TMA store; the accumulator is freed (an arrival on rank 0's
//              barrier) after the last loads, and the next tile's MMAs run
//              meanwhile in the other accumulator.  (Four epilogue warps
//              measured the same on the large shapes and 1.5 times slower at
//              K = 256, where the epilogue sets the pace.)
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

constexpr int kGemmBM = 128;  // rows per CTA: a pair MMA covers 256
constexpr int kGemmBN = 256;
constexpr int kGemmBK = 64;  // one 128-byte swizzle row of bf16
constexpr int kGemmStages = 6;
constexpr int kGemmEpiWarps = 8;
constexpr int kGemmThreads = 32 * (2 + kGemmEpiWarps);
constexpr uint32_t kGemmTmemCols = 2 * kGemmBN;

struct GemmSmem {
  __nv_bfloat16 a[kGemmStages][kGemmBM * kGemmBK];      // 16 KB per stage
  __nv_bfloat16 b[kGemmStages][kGemmBN / 2 * kGemmBK];  // this CTA's half of W: 16 KB per stage
  // per epilogue warp, two staging buffers of 32 rows x 32 columns (64-byte
  // rows, 64-byte swizzle) for the TMA stores of C
  __nv_bfloat16 cst[kGemmEpiWarps][2][32 * 32];
  uint64_t full[kGemmStages];   // rank 0's count both CTAs' loads
  uint64_t empty[kGemmStages];  // arrived by the MMA commit in both CTAs
  uint64_t acc_full[2];         // arrived by the MMA commit in both CTAs
  uint64_t acc_empty[2];        // rank 0's count both CTAs' epilogue warps
  uint32_t tmem_base;
};

// Shared-memory matrix descriptor of a K-major tile written by TMA with the
// 128-byte swizzle: rows of 128 bytes, 8-row swizzle atoms 1024 bytes apart
// (the stride byte offset); the leading byte offset is unused in this mode.
__device__ __forceinline__ uint64_t smem_desc_k128(uint32_t saddr) { return umma_desc(saddr, 1024, 2); }

// Instruction descriptor, kind::f16: fp32 accumulator (bits 4-5 = 1), A and
// B bf16 (bits 7-9, 10-12 = 1), both K-major (bits 15, 16 = 0), N / 8 at
// bits 17-22, M / 16 at bits 24-28; M = 256 over the pair.
__device__ __forceinline__ uint32_t gemm_idesc(int bn) { return umma_idesc_bf16(2 * kGemmBM, bn, false); }

__device__ __forceinline__ uint32_t smem_pad1024(const void* base) {
  return (1024u - (smem_u32(base) & 1023u)) & 1023u;
}

__device__ __forceinline__ uint32_t pack2_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

constexpr int kGemmGroupRows = 8;  // row blocks of 256 per raster group

// Row block and column tile of tile t (grouped raster order, above).
__device__ __forceinline__ void gemm_tile(long t, int tiles_m, int tiles_n, int& mb, int& nb) {
  const long per_group = (long)kGemmGroupRows * tiles_n;
  const int g = (int)(t / per_group);
  const int w = (int)(t - g * per_group);
  const int rows = min(kGemmGroupRows, tiles_m - g * kGemmGroupRows);
  nb = w / rows;
  mb = g * kGemmGroupRows + (w - nb * rows);
}

__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_w,
                   const __grid_constant__ CUtensorMap tm_c, const __grid_constant__ GemmParams p) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  GemmSmem& sm = *reinterpret_cast<GemmSmem*>(smem_raw + smem_pad1024(smem_raw));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int bn = p.bn;  // the N tile: a multiple of 32, at most kGemmBN
  const int half = bn / 2;  // the W rows this CTA holds
  const int tiles_n = (p.N + bn - 1) / bn;
  // the CTA pair of a cluster takes the two 128-row halves of 256-row tiles
  const uint32_t rank = cluster_ctarank();
  const int tiles_m = (int)((p.M + 2 * kGemmBM - 1) / (2 * kGemmBM));
  const long tiles = (long)tiles_m * tiles_n;
  const long first = cluster_id_x(), step = cluster_count_x();
  const int nk = (p.K + kGemmBK - 1) / kGemmBK;  // the loads fill zeros past K
  const uint32_t idesc = gemm_idesc(bn);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kGemmStages; ++s) {
      mbar_init(smem_u32(&sm.full[s]), 1);   // rank 0's producer, plus both CTAs' bytes
      mbar_init(smem_u32(&sm.empty[s]), 1);  // the MMA commit
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&sm.acc_full[b]), 1);
      mbar_init(smem_u32(&sm.acc_empty[b]), 2 * kGemmEpiWarps);  // the epilogue warps of both CTAs
    }
    fence_mbar_init();
    prefetch_tensormap(&tm_a);
    prefetch_tensormap(&tm_w);
    prefetch_tensormap(&tm_c);
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(&sm.tmem_base), kGemmTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync();  // both CTAs' barriers are initialised before either signals the other's
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  bool ok = true;

  if (warp == 0) {
    if (lane == 0) {  // producer
      const uint64_t keep = l2_policy_evict_last();  // W: read by every row block
      uint32_t it = 0;
      for (long t = first; t < tiles && ok; t += step) {
        int mb, nb;
        gemm_tile(t, tiles_m, tiles_n, mb, nb);
        const int m0 = mb * 2 * kGemmBM + (int)rank * kGemmBM;
        const int n0 = nb * bn + (int)rank * half;
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int s = (int)(it % kGemmStages);
          const uint32_t ph = (it / kGemmStages) & 1u;
          // stage s of this CTA has been read by the MMAs of its last round
          if (!mbar_wait_bounded(smem_u32(&sm.empty[s]), ph ^ 1u, p.timeout_ns)) {
            ok = false;
            break;
          }
          const uint32_t bar = mapa_shared(smem_u32(&sm.full[s]), 0);  // rank 0's barrier
          if (rank == 0) mbar_arrive_expect_tx(smem_u32(&sm.full[s]), 2 * (kGemmBM + half) * kGemmBK * 2);
          tma_load_2d_pair(smem_u32(&sm.a[s][0]), &tm_a, kb * kGemmBK, m0, bar);  // reused by the row block's tiles
          tma_load_2d_pair(smem_u32(&sm.b[s][0]), &tm_w, kb * kGemmBK, n0, bar, keep);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {  // MMA issuer
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
            tc_mma_f16_pair(d, ad + 2 * kk, bd + 2 * kk, idesc, (kb | kk) != 0);
          tc_commit_pair_mc(smem_u32(&sm.empty[s]), 0x3);  // frees stage s in both CTAs
        }
        if (!ok) break;
        tc_commit_pair_mc(smem_u32(&sm.acc_full[buf]), 0x3);
      }
    }
  } else {  // epilogue: warp w reads TMEM lanes 32 (w % 4) .. + 31
    const int q = warp & 3;
    const int e = warp - 2;    // staging buffers
    const int h = e >> 2;      // chunks h, h + kGemmEpiWarps / 4, ...
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
      int mb, nb;
      gemm_tile(t, tiles_m, tiles_n, mb, nb);
      const int m0 = mb * 2 * kGemmBM + (int)rank * kGemmBM;
      const int n0 = nb * bn;
      const uint32_t tbase = tmem + ((uint32_t)(32 * q) << 16) + buf * kGemmBN;
      const int chunks = min(bn, p.N - n0 + 31) / 32;  // 32-column chunks holding valid columns
      const uint32_t acc_empty = mapa_shared(smem_u32(&sm.acc_empty[buf]), 0);
      if (h >= chunks) {  // nothing of this tile for this warp
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(acc_empty);
      }
#pragma unroll 1
      for (int c = h; c < chunks; c += kGemmEpiWarps / 4) {
        const int col0 = n0 + 32 * c;
        // the chunk's 32 bias values (the same for every lane: broadcast
        // loads), four 16-byte vectors where the chunk lies inside N, issued
        // before the chunk's TMEM load so that the two latencies overlap
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
        uint32_t r[32];
        tmem_ld_32cols(tbase + 32 * c, r);
        if (c + kGemmEpiWarps / 4 >= chunks) {  // this warp's share is in registers: hand it back
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(acc_empty);
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
        const uint32_t st = smem_u32(&sm.cst[e][sb][0]);
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
  // both CTAs are done with the tensor memory and with each other's barriers
  // (a peer's last arrivals have landed) before the pair frees it
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  if (warp == 1) {
    __syncwarp();  // the warp-wide tcgen05 operations need the whole warp converged
    tc_fence_after();
    tmem_dealloc_pair(tmem, kGemmTmemCols);
  }
  cluster_sync();
}

}  // namespace mamba
