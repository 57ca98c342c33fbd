// ssd.cuh -- Mamba-2's scan in its chunked matrix form on the tensor cores.
//
// The structure of "Jamba -- SSM-Transformer Hibrido" (ai-engineering.academy),
// section "Mamba-3: a linha de base de SSM puro em 2026", items 1 and 2: the
// state matrix is a scaled identity, discretised with Euler's method.  Heads of
// P = 64 channels share dt and A, so the decay from token s to token t,
// exp(A (cum_t - cum_s)), is one number per (t, s) for the whole head, and
// within a chunk of Q = 128 tokens the scan is a few small matrix products:
//   Y_diag = (mask(t >= s) * exp(A (cum_t - cum_s)) * dt_s * (C B^T)) X
//   Y_off  = exp(A cum_t) (C S_in)          (S_in: the state entering the chunk)
//   S_end  = (exp(A (cum_last - cum_s)) dt_s B_s)^T X + exp(A cum_last) S_in
// Three kernels: ssd_states_kernel (each chunk's end state from zero, the
// transposed 64 x 16 product on tcgen05), ssd_pass_kernel (the states
// entering the chunks, serially per head, in fp32) and ssd_output_kernel
// (Y_diag + Y_off + D x, gated) on tcgen05.  The first and the last are
// persistent, warp-specialised pipelines: tiles brought in by TMA, 128- or
// 64-row MMAs with the accumulators in tensor memory.  fp32 quantities
// entering a product (the decay-weighted B rows and C B^T entries, the
// entering state) go in as two bf16 terms (hi + lo, ~16 significant bits).
#pragma once
#include <cuda_bf16.h>

#include <cstdint>

#include "params.h"
#include "ptx.cuh"
#include "scan_fwd.cuh"
#include "ssm_math.cuh"

namespace mamba {

constexpr int kSsdQ = 128;         // tokens per chunk
constexpr int kSsdP = 64;          // channels per head
constexpr int kSsdN = 16;          // d_state

// two floats as a bf16 pair (lo in the low half: the smaller column)
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

__device__ __forceinline__ float2 unpack_bf16(uint32_t v) {
  return make_float2(__uint_as_float(v << 16), __uint_as_float(v & 0xffff0000u));
}

// 16-byte piece `piece` of row `row` in a 128-byte-swizzled tile of 128-byte
// rows (the tile 1024-byte aligned).
__device__ __forceinline__ uint32_t sw128(uint32_t base, int row, int piece) {
  return base + row * 128 + ((piece ^ (row & 7)) << 4);
}

struct SsdTileId {
  int h, c, b;
};

// (the host keeps the tile count below 2^31)
__device__ __forceinline__ SsdTileId ssd_tile(uint32_t t, uint32_t H, uint32_t nC) {
  SsdTileId id;
  const uint32_t hc = t / H;
  id.h = (int)(t - hc * H);
  id.b = (int)(hc / nC);
  id.c = (int)(hc - (uint32_t)id.b * nC);
  return id;
}

// v (two fp32 values) as hi + lo bf16 pairs, packed arithmetic.
__device__ __forceinline__ void split_bf16_x2(float2 v, uint32_t& hi, uint32_t& lo) {
  hi = pack_bf16(v.x, v.y);
  const float2 h = unpack_bf16(hi);
  const float2 d = __ffma2_rn(h, make_float2(-1.0f, -1.0f), v);  // v - h, exactly rounded
  lo = pack_bf16(d.x, d.y);
}

// ---------------------------------------------------------------- chunk end states
// S_c[n][p] = sum_j 2^(acum_last - acum_j) dt_j B_j[n] x_j[p], each chunk's end
// state from zero, as the transposed product S_c^T = X^T (w o B): M = 64
// channels, N = 16 states, K = 128 tokens on tcgen05 (M = 64: accumulator row
// m in tensor-memory lane 32 (m / 16) + m % 16), the weights w_j =
// 2^(acum_last - acum_j) dt_j applied to the B rows, which enter as hi + lo
// bf16 terms.  A persistent kernel, two CTAs per SM, tiles (head, chunk,
// batch row) with the head fastest:
//   warp 0      loads x (128 tokens x 64 channels, 128-byte swizzle: the
//               MN-major A operand) and B (128 x 16, 32-byte swizzle) of tile
//               k into stage k % 3 by TMA;
//   warp 1      issues the 16 MMAs of tile k into accumulator k % 4 once its
//               weighted-B operand is written, freeing the stage;
//   warps 4-11  two groups of four warps, group g taking the tiles k with
//               k % 2 = g (the per-tile work is a chain of dependent steps:
//               two chains in flight per CTA).  Thread j = token j:
//               softplus(dt), the chunk's decay prefix (warp scans, then the
//               earlier warps' totals), the weight, w_j B_j as hi + lo into
//               the K-major operand, the chunk's (prefix, dt) pairs and total
//               for the later kernels; then the accumulator of the group's
//               previous tile out of tensor memory into S_c.
constexpr int kStStages = 3;
constexpr int kStGroups = 2;
constexpr int kStThreads = 128 + 128 * kStGroups;
constexpr int kStBufs = 2 * kStGroups;  // weighted-B operands and accumulators (16 columns each)

struct StStage {
  __nv_bfloat16 x[kSsdQ * kSsdP];  // rows of 128 bytes
  __nv_bfloat16 b[kSsdQ * kSsdN];  // rows of 32 bytes
  unsigned char pad[3072];         // keeps the next stage's x 1024-byte aligned
};
static_assert(sizeof(StStage) % 1024 == 0, "stage alignment");

struct StSmem {
  StStage st[kStStages];
  __nv_bfloat16 whi[kStBufs][2][kSsdN * 64];  // [buffer][K half]: rows n of 64 tokens (128 bytes)
  __nv_bfloat16 wlo[kStBufs][2][kSsdN * 64];
  float wsum[kStGroups][4];                   // per group: its warps' dt A totals
  uint64_t full[kStStages], empty[kStStages];
  uint64_t wb_full[kStBufs], wb_empty[kStBufs], acc_full[kStBufs], acc_empty[kStBufs];
  uint32_t tmem_base;
};

// The 128 threads of compute group g (named barrier 1 + g) agree on a predicate.
__device__ __forceinline__ bool group_all(int g, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, %2, 128, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v), "r"(1 + g)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ void group_sync(int g) { asm volatile("bar.sync %0, 128;" ::"r"(1 + g) : "memory"); }

// 32-byte-swizzled tile of 32-byte rows: 16-byte chunk c of row r.
__device__ __forceinline__ uint32_t sw32(uint32_t base, int r, int c) {
  return base + r * 32 + ((c ^ ((r >> 2) & 1)) << 4);
}

__global__ void __launch_bounds__(kStThreads, 2)
    ssd_states_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_b,
                      const __grid_constant__ SsdParams p) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  StSmem& sm = *reinterpret_cast<StSmem*>(smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int H = p.heads, nC = p.n_chunks, L = p.seqlen;
  const uint32_t tiles = (uint32_t)H * nC * p.batch;
  const uint32_t n_mine = (tiles - blockIdx.x + gridDim.x - 1) / gridDim.x;

  if (tid == 0) {
    for (int s = 0; s < kStStages; ++s) {
      mbar_init(smem_u32(&sm.full[s]), 1);
      mbar_init(smem_u32(&sm.empty[s]), 1);
    }
    for (int w = 0; w < kStBufs; ++w) {
      mbar_init(smem_u32(&sm.wb_full[w]), 4);  // one arrival per warp of the group
      mbar_init(smem_u32(&sm.wb_empty[w]), 1);
      mbar_init(smem_u32(&sm.acc_full[w]), 1);
      mbar_init(smem_u32(&sm.acc_empty[w]), 4);
    }
    fence_mbar_init();
    prefetch_tensormap(&tm_x);
    prefetch_tensormap(&tm_b);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&sm.tmem_base), 16 * kStBufs);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // a programmatic dependent: the kernel before it (the previous call's
  // output kernel reads the chunk states and prefixes this one writes) has
  // completed before any global memory is touched; the pass may launch now
  griddep_wait();
  griddep_launch_dependents();
  const uint32_t tmem = sm.tmem_base;
  bool ok = true;

  if (warp == 0) {
    if (lane == 0) {  // producer
      uint32_t k = 0;
      for (; k < n_mine; ++k) {
        const int s = (int)(k % kStStages);
        if (!mbar_wait_bounded(smem_u32(&sm.empty[s]), ((k / kStStages) & 1u) ^ 1u, p.timeout_ns)) {
          ok = false;
          break;
        }
        const SsdTileId id = ssd_tile(blockIdx.x + k * gridDim.x, H, nC);
        const int g = id.h / (H / p.groups), t0 = id.c * kSsdQ;
        const uint32_t bar = smem_u32(&sm.full[s]);
        mbar_arrive_expect_tx(bar, kSsdQ * kSsdP * 2 + kSsdQ * kSsdN * 2);
        tma_load_4d(smem_u32(sm.st[s].x), &tm_x, 0, id.h, t0, id.b, bar);
        tma_load_4d(smem_u32(sm.st[s].b), &tm_b, 0, g, t0, id.b, bar);
      }
      for (uint32_t j = k > kStStages ? k - kStStages : 0; j < k; ++j)
        if (!mbar_wait_bounded(smem_u32(&sm.full[j % kStStages]), (j / kStStages) & 1u, p.timeout_ns)) ok = false;
    }
  } else if (warp == 1) {
    if (lane == 0) {  // MMA issuer
      const uint32_t idesc = umma_idesc_bf16(64, 16, false) | (1u << 15);  // A (x^T) MN-major, B K-major
      for (uint32_t k = 0; k < n_mine; ++k) {
        const int s = (int)(k % kStStages);
        const uint32_t w = k % kStBufs, ph = (k / kStBufs) & 1u;
        if (!mbar_wait_bounded(smem_u32(&sm.wb_full[w]), ph, p.timeout_ns) ||
            !mbar_wait_bounded(smem_u32(&sm.full[s]), (k / kStStages) & 1u, p.timeout_ns) ||
            !mbar_wait_bounded(smem_u32(&sm.acc_empty[w]), ph ^ 1u, p.timeout_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem + w * 16;
#pragma unroll
        for (int part = 0; part < 2; ++part)
#pragma unroll
          for (int kh = 0; kh < 2; ++kh)
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
              const uint64_t ad = umma_desc(smem_u32(sm.st[s].x) + (kh * 64 + ks * 16) * 128, 1024, 2);  // 16 tokens
              const uint32_t wb = smem_u32(part == 0 ? sm.whi[w][kh] : sm.wlo[w][kh]);
              tc_mma_f16(d, ad, umma_desc(wb + 32 * ks, 1024, 2), idesc, (part | kh | ks) != 0);
            }
        tc_commit(smem_u32(&sm.acc_full[w]));
        tc_commit(smem_u32(&sm.wb_empty[w]));
        tc_commit(smem_u32(&sm.empty[s]));
      }
    }
  } else if (warp >= 4) {  // compute groups
    const int grp = (warp - 4) >> 2, cw = warp & 3;
    const int j = 32 * cw + lane;  // token of the chunk
    const unsigned short* dtr16 = static_cast<const unsigned short*>(p.dt_raw);
    // this thread's dt_raw (bf16 bits, converted at use) and the head's
    // A_log of tile k: plain loads, no select on their values (which would
    // wait for them here); tokens past the sequence's end read the last one
    // and are masked at use
    auto inputs_of = [&](uint32_t k) -> uint2 {
      const SsdTileId id = ssd_tile(blockIdx.x + (k < n_mine ? k : 0) * gridDim.x, H, nC);
      const int t = min(id.c * kSsdQ + j, L - 1);
      return make_uint2((uint32_t)__ldg(dtr16 + ((size_t)id.b * L + t) * H + id.h),
                        __float_as_uint(__ldg(p.A_log + id.h)));
    };
    // the accumulator of tile kk out of tensor memory into S_c: lanes 0..15
    // of warp q hold channels 16 q .. + 15, 16 states each
    auto drain = [&](uint32_t kk) -> bool {
      const uint32_t w = kk % kStBufs;
      if (!group_all(grp, mbar_wait_bounded(smem_u32(&sm.acc_full[w]), (kk / kStBufs) & 1u, p.timeout_ns)))
        return false;
      tc_fence_after();
      uint32_t r[16];
      tmem_ld_16cols(tmem + ((uint32_t)(32 * cw) << 16) + w * 16, r);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sm.acc_empty[w]));
      if (lane < 16) {
        const SsdTileId id = ssd_tile(blockIdx.x + kk * gridDim.x, H, nC);
        const int col = 16 * cw + lane;  // channel
        float* dst = p.S_c + (((size_t)id.b * H + id.h) * nC + id.c) * (kSsdN * kSsdP) + col;
#pragma unroll
        for (int n = 0; n < kSsdN; ++n) dst[n * kSsdP] = __uint_as_float(r[n]);
      }
      return true;
    };
    uint2 in = inputs_of(grp);
    uint32_t k = grp;
    for (; k < n_mine; k += kStGroups) {
      const int s = (int)(k % kStStages);
      const uint32_t w = k % kStBufs;
      const SsdTileId id = ssd_tile(blockIdx.x + k * gridDim.x, H, nC);
      const uint2 in_next = inputs_of(k + kStGroups);  // in flight through this tile
      const bool mine = mbar_wait_bounded(smem_u32(&sm.full[s]), (k / kStStages) & 1u, p.timeout_ns) &&
                        mbar_wait_bounded(smem_u32(&sm.wb_empty[w]), ((k / kStBufs) & 1u) ^ 1u, p.timeout_ns);
      if (!group_all(grp, mine)) {
        ok = false;
        break;
      }
      // dt and the inclusive prefix of dt A (base 2) over the chunk: per
      // warp, then each warp adds the totals of the warps before it
      const float A2 = a2_from_log(__uint_as_float(in.y));
      const int t = id.c * kSsdQ + j;
      const float dt = t < L ? softplus(__uint_as_float(in.x << 16)) : 0.0f;
      float v = __fmul_rn(dt, A2);
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float u = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v = __fadd_rn(v, u);
      }
      if (lane == 31) sm.wsum[grp][cw] = v;
      group_sync(grp);
      float off = 0.0f;
#pragma unroll
      for (int q = 0; q < 3; ++q)
        if (q < cw) off = __fadd_rn(off, sm.wsum[grp][q]);
      const float acum = cw > 0 ? __fadd_rn(v, off) : v;
      // the last token's prefix, by the same sums in the same order as its
      // own: warp 3's scan plus the totals of warps 0..2
      float last = 0.0f;
#pragma unroll
      for (int q = 0; q < 3; ++q) last = __fadd_rn(last, sm.wsum[grp][q]);
      last = __fadd_rn(sm.wsum[grp][3], last);
      const float wj = __fmul_rn(ex2_approx(__fsub_rn(last, acum)), dt);
      const size_t chunk = ((size_t)id.b * H + id.h) * nC + id.c;
      reinterpret_cast<float2*>(p.cum)[chunk * kSsdQ + j] = make_float2(acum, dt);
      if (j == kSsdQ - 1) p.totals[chunk] = acum;
      // w_j B_j (16 states) as hi + lo into the K-major operand: row n, token j
      {
        const StStage& st = sm.st[s];
        uint4 b0, b1;
        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(b0.x), "=r"(b0.y), "=r"(b0.z), "=r"(b0.w)
                     : "r"(sw32(smem_u32(st.b), j, 0)));
        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(b1.x), "=r"(b1.y), "=r"(b1.z), "=r"(b1.w)
                     : "r"(sw32(smem_u32(st.b), j, 1)));
        const uint32_t bw[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
        const int kh = j >> 6, jj = j & 63;
        const uint32_t hb = smem_u32(sm.whi[w][kh]), lb = smem_u32(sm.wlo[w][kh]);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float2 bv = unpack_bf16(bw[e]);
          uint32_t hi, lo;
          split_bf16_x2(__fmul2_rn(bv, make_float2(wj, wj)), hi, lo);
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int n = 2 * e + u;
            const uint32_t off16 = sw128(0, n, jj >> 3) + (jj & 7) * 2;
            const uint16_t hv = (uint16_t)(u ? hi >> 16 : hi & 0xffffu);
            const uint16_t lv = (uint16_t)(u ? lo >> 16 : lo & 0xffffu);
            asm volatile("st.shared.b16 [%0], %1;" ::"r"(hb + off16), "h"(hv) : "memory");
            asm volatile("st.shared.b16 [%0], %1;" ::"r"(lb + off16), "h"(lv) : "memory");
          }
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sm.wb_full[w]));
      in = in_next;
      if (k >= (uint32_t)kStGroups && !drain(k - kStGroups)) {  // the group's previous tile
        ok = false;
        break;
      }
    }
    if (ok && k >= (uint32_t)kStGroups && !drain(k - kStGroups)) ok = false;  // the group's last tile
  }

  if (!ok) report_error(4u);  // MAMBA_ERR_TIMEOUT
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 16 * kStBufs);
  }
}

// ---------------------------------------------------------------- state passing
// The state entering chunk c: S_in[0] = h0 (or 0), S_in[c + 1] = 2^(total_c)
// S_in[c] + S_c[c], in fp32.  Two CTAs per (batch row, head), each walking
// the chunks in order over half of the head's 16 x 64 state, one thread per
// value.  The halves of S_c come in by bulk copies, kPassRing chunks ahead
// (the per-SM limit on outstanding cache misses would hold plain loads to a
// fraction of the bandwidth), and S_in leaves by bulk stores from a staging
// ring, kPassGroup chunks per step; the chain itself is one fma per value and
// chunk.  The chunks' decay factors 2^(total) are staged in shared memory,
// kPassBlock at a time.
constexpr int kPassThreads = kSsdN * kSsdP / 2;
constexpr int kPassRing = 32;
constexpr int kPassGroup = 4;                 // chunks per step (one barrier, one bulk group)
constexpr int kPassStage = 3 * kPassGroup;    // staging slots: three steps' worth
constexpr int kPassBlock = 1024;

struct PassSmem {
  float ring[kPassRing][kPassThreads];
  float out[kPassStage][kPassThreads];
  float fac[kPassBlock];
  uint64_t full[kPassRing];
};

__global__ void __launch_bounds__(kPassThreads) ssd_pass_kernel(const __grid_constant__ SsdParams p) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  PassSmem& sm = *reinterpret_cast<PassSmem*>(smem_raw + smem_pad128(smem_raw));
  const int half = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x;
  const size_t bh = (size_t)b * p.heads + h;
  const int nC = p.n_chunks;
  constexpr int kStep = kSsdN * kSsdP;  // floats per chunk state
  constexpr uint32_t kBytes = kPassThreads * 4;
  const float* src = p.S_c + bh * nC * kStep + half * kPassThreads;
  float* dst = p.S_in + bh * nC * kStep + half * kPassThreads;
  const float* tot = p.totals + bh * nC;
  griddep_wait();  // the states kernel's chunk states are complete
  griddep_launch_dependents();
  if (tid == 0) {
    for (int r = 0; r < kPassRing; ++r) mbar_init(smem_u32(&sm.full[r]), 1);
    fence_mbar_init();
    for (int c = 0; c < kPassRing && c < nC; ++c) {
      mbar_arrive_expect_tx(smem_u32(&sm.full[c]), kBytes);
      bulk_load(smem_u32(sm.ring[c]), src + (size_t)c * kStep, kBytes, smem_u32(&sm.full[c]));
    }
  }
  __syncthreads();
  float S = p.h0 ? p.h0[bh * kStep + half * kPassThreads + tid] : 0.0f;
  bool ok = true;
  int c0 = 0;
  for (int step = 0; c0 < nC; ++step, c0 += kPassGroup) {
    if (c0 % kPassBlock == 0) {  // the next block of decay factors (the last block's reads are behind a barrier)
      for (int i = tid; i < kPassBlock && c0 + i < nC; i += kPassThreads) sm.fac[i] = ex2_approx(__ldg(tot + c0 + i));
      __syncthreads();
    }
    bool mine = true;
#pragma unroll
    for (int u = 0; u < kPassGroup; ++u) {
      const int c = c0 + u;
      if (c < nC) mine = mine && mbar_wait_bounded(smem_u32(&sm.full[c % kPassRing]), (c / kPassRing) & 1u, p.timeout_ns);
    }
    if (!__syncthreads_and(mine)) {
      ok = false;
      break;
    }
    const int o0 = (step % 3) * kPassGroup;
#pragma unroll
    for (int u = 0; u < kPassGroup; ++u) {
      const int c = c0 + u;
      if (c < nC) {
        const float v = sm.ring[c % kPassRing][tid];
        sm.out[o0 + u][tid] = S;
        S = __fmaf_rn(sm.fac[c % kPassBlock], S, v);
      }
    }
    fence_proxy_async_smem();
    __syncthreads();  // the ring slots are read and the staging slots written by every thread
    if (tid == 0) {
#pragma unroll
      for (int u = 0; u < kPassGroup; ++u) {
        const int c = c0 + u;
        if (c < nC) bulk_store(dst + (size_t)c * kStep, smem_u32(sm.out[o0 + u]), kBytes);
      }
      bulk_commit();
#pragma unroll
      for (int u = 0; u < kPassGroup; ++u) {
        const int c = c0 + u;
        if (c + kPassRing < nC) {
          mbar_arrive_expect_tx(smem_u32(&sm.full[c % kPassRing]), kBytes);
          bulk_load(smem_u32(sm.ring[c % kPassRing]), src + (size_t)(c + kPassRing) * kStep, kBytes,
                    smem_u32(&sm.full[c % kPassRing]));
        }
      }
      // the stores of the step before have left shared memory: their staging
      // slots are written two steps on, after the next step's barrier
      bulk_wait_read<1>();
    }
  }
  if (tid == 0) {
    bulk_wait_all();
    if (!ok) report_error(4u);  // MAMBA_ERR_TIMEOUT
    // every load issued has landed before the CTA may end: chunks below
    // min(nC, c0 + kPassRing), the last of each ring slot
    const int issued = min(nC, c0 + kPassRing);
    for (int cc = issued > kPassRing ? issued - kPassRing : 0; cc < issued; ++cc)
      mbar_wait_bounded(smem_u32(&sm.full[cc % kPassRing]), (cc / kPassRing) & 1u, p.timeout_ns);
  }
  if (ok && p.final_state) p.final_state[bh * kStep + half * kPassThreads + tid] = S;
}

// ---------------------------------------------------------------- output
// A persistent kernel, one CTA per SM, walking tiles t = (head, chunk, batch
// row) with the head fastest (the SMs at work at one time share a chunk's B
// and C rows and read its x, z rows whole).  Warp roles, linked by mbarriers:
//   warp 0      loads tile k into stage k % 5 by TMA: x (128 tokens x 64
//               channels, 128-byte swizzle), B, C (128 x 16, 32-byte
//               swizzle), the entering state (fp32, 4 KB) and the chunk's
//               (decay prefix, dt) pairs by bulk copies; z, read only by the
//               epilogue, into a ring of its own of three tiles;
//   warp 1      issues the MMAs, each as soon as its inputs are ready:
//               G = C B^T (128 x 128, K = 16) into score buffer k % 2 of
//               tensor memory; then Y = G' X (128 x 64), G' read from tensor
//               memory (hi and lo terms accumulated), in two halves of K =
//               64, each once the converter has written its half of G', into
//               accumulator buffer k % 4 (64 columns); with the second half
//               the entering state's term (e C) S_in (K = 16, e_i =
//               2^(acum_i); hi + lo products) accumulated into the same Y;
//   warps 4-11  warp w reads rows 32 (w % 4) .. + 31 of G and columns
//               64 h .. + 63 (h = (w - 4) / 4, the K half), masks them to
//               s <= t, scales them by the decay 2^(acum_i - acum_j) dt_j and
//               writes them back in place as hi + lo bf16 terms (G' = G_hi +
//               G_lo, ~16 significant bits: each 32-column group's 32 fp32
//               columns become 16 columns of hi pairs and 16 of lo pairs), the
//               A operand of the Y product; the h = 1 warps also write the
//               entering state (hi + lo, MN-major) into shared memory, and
//               the rows e_i C_i (hi + lo) over the stage's B and C tiles,
//               dead once G is formed;
//   warps 12-15 y = Y + D x, times silu(z) (through tanh), written over the
//               stage's x rows and stored by TMA (32 rows per warp), which
//               frees the stage.
// Tensor memory holds two score buffers (2 x 128 columns) and four
// accumulator buffers (4 x 64): a score buffer is free again once the Y
// product has read it, so G of tile k + 2 needs only tile k's Y product, and
// the epilogue runs up to four tiles behind the MMAs.
// The decay factor of an entry is taken relative to the first token of its
// 32-column group, 2^(acum_i - acum_r) * (2^(acum_r - acum_j) dt_j): both
// factors stay in range while the decay across the 32 tokens is at most
// 2^60; beyond that (very fast decay) the entry's factor is computed whole.
constexpr int kSsdStages = 5;
constexpr int kSsdZ = 3;  // the gate's ring
constexpr int kSsdAcc = 4;
constexpr int kSsdOutThreads = 512;
constexpr int kSsdTmemCols = 512;  // score buffers at columns 0, 128; accumulators at 256 + 64 j

struct SsdStage {
  __nv_bfloat16 x[kSsdQ * kSsdP];  // 16 KB, rows of 128 bytes; then y
  __nv_bfloat16 b[kSsdQ * kSsdN];  // rows of 32 bytes; then the e C rows' hi terms
  __nv_bfloat16 c[kSsdQ * kSsdN];  // then their lo terms
  float s[kSsdN * kSsdP];          // the entering state, row n of 64 channels
  float2 cum[kSsdQ];               // (decay prefix, dt) per token
};
static_assert(sizeof(SsdStage) % 1024 == 0, "stages keep the 1024-byte alignment of the swizzled tiles");

struct SsdOutSmem {
  SsdStage st[kSsdStages];
  __nv_bfloat16 z[kSsdZ][kSsdQ * kSsdP];  // the gate's ring
  __nv_bfloat16 shi[2][kSsdN * kSsdP];    // the entering state: rows n of 64 channels
  __nv_bfloat16 slo[2][kSsdN * kSsdP];
  float fdt[8][64];                       // per converter warp: 2^(acum_r - acum_j) dt_j for its columns
  uint64_t full[kSsdStages], empty[kSsdStages];
  uint64_t zfull[kSsdZ], zempty[kSsdZ];
  uint64_t gfull[2], aempty[2];  // score buffers: G formed; read by the Y product
  uint64_t opfull[2][2];         // [score buffer][K half]: G' written
  uint64_t yfull[kSsdAcc], yempty[kSsdAcc];  // accumulator buffers
  uint32_t tmem_base;
};

// silu(z) = z sigmoid(z) = h + h tanh(h), h = z / 2: one MUFU operation per
// value (tanh.approx, relative error about 2^-11, which moves silu by at most
// about |h| 2^-11 -- below a bf16 output's half ulp relative to the gated
// output's scale).
__device__ __forceinline__ float tanh_approx(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float2 silu_tanh_x2(float2 z) {
  const float2 h = __fmul2_rn(z, make_float2(0.5f, 0.5f));
  return __ffma2_rn(h, make_float2(tanh_approx(h.x), tanh_approx(h.y)), h);
}

// The Y half kh of a tile (and, with the second half, the entering state's
// term): MMAs with G' from score buffer column ga into accumulator column dy.
__device__ __forceinline__ void ssd_issue_y(const SsdOutSmem& sm, const SsdStage& st, uint32_t ga, uint32_t dy,
                                            int kh, int sb) {
  const uint32_t iy = umma_idesc_bf16(128, 64, true);  // B operand (x rows, S rows) MN-major
#pragma unroll
  for (int ks = 0; ks < 4; ++ks) {
    // 16 columns of G': group ks / 2 of the half, its hi pairs at +0, lo at +16
    const uint32_t a = ga + 64 * kh + 32 * (ks >> 1) + 8 * (ks & 1);
    const uint64_t bd = umma_desc(smem_u32(st.x) + (kh * 64 + ks * 16) * 128, 1024, 2);  // 16 rows of x
    tc_mma_f16_ta(dy, a, bd, iy, kh > 0 || ks > 0);
    tc_mma_f16_ta(dy, a + 16, bd, iy, true);
  }
  if (kh == 1) {  // + (e C) S_in: (e C)_hi S_hi + (e C)_hi S_lo + (e C)_lo S_hi
    const uint64_t ehi = umma_desc(smem_u32(st.b), 256, 6), elo = umma_desc(smem_u32(st.c), 256, 6);
    const uint64_t shi = umma_desc(smem_u32(sm.shi[sb]), 1024, 2), slo = umma_desc(smem_u32(sm.slo[sb]), 1024, 2);
    tc_mma_f16(dy, ehi, shi, iy, true);
    tc_mma_f16(dy, ehi, slo, iy, true);
    tc_mma_f16(dy, elo, shi, iy, true);
  }
}

__global__ void __launch_bounds__(kSsdOutThreads, 1)
    ssd_output_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_z,
                      const __grid_constant__ CUtensorMap tm_b, const __grid_constant__ CUtensorMap tm_c,
                      const __grid_constant__ CUtensorMap tm_y, const __grid_constant__ SsdParams p) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  SsdOutSmem& sm = *reinterpret_cast<SsdOutSmem*>(smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int H = p.heads, nC = p.n_chunks, L = p.seqlen;
  const uint32_t tiles = (uint32_t)H * nC * p.batch;
  const uint32_t n_mine = (tiles - blockIdx.x + gridDim.x - 1) / gridDim.x;  // this CTA's tiles
  const bool gate = p.z != nullptr;

  if (tid == 0) {
    for (int s = 0; s < kSsdStages; ++s) {
      mbar_init(smem_u32(&sm.full[s]), 1);
      mbar_init(smem_u32(&sm.empty[s]), 4);  // one arrival per epilogue warp
    }
    for (int z = 0; z < kSsdZ; ++z) {
      mbar_init(smem_u32(&sm.zfull[z]), 1);
      mbar_init(smem_u32(&sm.zempty[z]), 4);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(smem_u32(&sm.gfull[a]), 1);
      mbar_init(smem_u32(&sm.aempty[a]), 1);
      mbar_init(smem_u32(&sm.opfull[a][0]), 4);  // one arrival per converter warp of the half
      mbar_init(smem_u32(&sm.opfull[a][1]), 4);
    }
    for (int e = 0; e < kSsdAcc; ++e) {
      mbar_init(smem_u32(&sm.yfull[e]), 1);
      mbar_init(smem_u32(&sm.yempty[e]), 4);
    }
    fence_mbar_init();
    prefetch_tensormap(&tm_x);
    prefetch_tensormap(&tm_z);
    prefetch_tensormap(&tm_b);
    prefetch_tensormap(&tm_c);
    prefetch_tensormap(&tm_y);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&sm.tmem_base), kSsdTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  griddep_wait();  // the pass's entering states are complete
  griddep_launch_dependents();
  const uint32_t tmem = sm.tmem_base;
  bool ok = true;

  if (warp == 0) {
    if (lane == 0) {  // producer: the stages, and the gate's ring
      const uint32_t bytes = kSsdQ * kSsdP * 2 + 2 * kSsdQ * kSsdN * 2 + kSsdN * kSsdP * 4 + kSsdQ * 8;
      uint32_t k = 0, kz = 0;
      uint64_t idle_since = globaltimer_ns();
      while (k < n_mine || (gate && kz < n_mine)) {
        bool moved = false;
        if (k < n_mine && mbar_test_wait(smem_u32(&sm.empty[k % kSsdStages]), ((k / kSsdStages) & 1u) ^ 1u)) {
          const int s = (int)(k % kSsdStages);
          const SsdTileId id = ssd_tile(blockIdx.x + k * gridDim.x, H, nC);
          const int g = id.h / (H / p.groups), t0 = id.c * kSsdQ;
          const size_t chunk = ((size_t)id.b * H + id.h) * nC + id.c;
          SsdStage& st = sm.st[s];
          const uint32_t bar = smem_u32(&sm.full[s]);
          if (gate) tma_prefetch_4d(&tm_z, 0, id.h, t0, id.b);  // into L2, for the gate's ring
          mbar_arrive_expect_tx(bar, bytes);
          tma_load_4d(smem_u32(st.x), &tm_x, 0, id.h, t0, id.b, bar);
          tma_load_4d(smem_u32(st.b), &tm_b, 0, g, t0, id.b, bar);
          tma_load_4d(smem_u32(st.c), &tm_c, 0, g, t0, id.b, bar);
          bulk_load(smem_u32(st.s), p.S_in + chunk * (kSsdN * kSsdP), kSsdN * kSsdP * 4, bar);
          bulk_load(smem_u32(st.cum), p.cum + chunk * (2 * kSsdQ), kSsdQ * 8, bar);
          ++k;
          moved = true;
        }
        if (gate && kz < k && mbar_test_wait(smem_u32(&sm.zempty[kz % kSsdZ]), ((kz / kSsdZ) & 1u) ^ 1u)) {
          const SsdTileId id = ssd_tile(blockIdx.x + kz * gridDim.x, H, nC);
          const uint32_t bar = smem_u32(&sm.zfull[kz % kSsdZ]);
          mbar_arrive_expect_tx(bar, kSsdQ * kSsdP * 2);
          tma_load_4d(smem_u32(sm.z[kz % kSsdZ]), &tm_z, 0, id.h, id.c * kSsdQ, id.b, bar);
          ++kz;
          moved = true;
        }
        if (moved) {
          idle_since = globaltimer_ns();
        } else {
          if (globaltimer_ns() - idle_since > p.timeout_ns) {
            ok = false;
            break;
          }
        }
      }
      // the copies issued last have landed before the CTA may end
      for (uint32_t j = k > kSsdStages ? k - kSsdStages : 0; j < k; ++j)
        if (!mbar_wait_bounded(smem_u32(&sm.full[j % kSsdStages]), (j / kSsdStages) & 1u, p.timeout_ns)) ok = false;
      for (uint32_t j = kz > kSsdZ ? kz - kSsdZ : 0; j < kz; ++j)
        if (!mbar_wait_bounded(smem_u32(&sm.zfull[j % kSsdZ]), (j / kSsdZ) & 1u, p.timeout_ns)) ok = false;
    }
  } else if (warp == 1) {
    if (lane == 0) {  // MMA issuer: G of tile kg, Y halves of tiles ky0, ky1, each as soon as it may go
      // (polled without sleeping, the Y halves first: they gate the epilogue)
      const uint32_t ig = umma_idesc_bf16(128, 128, false);  // G = C B^T: both K-major
      uint32_t kg = 0, ky0 = 0, ky1 = 0;
      uint64_t idle_since = globaltimer_ns();
      while (ky1 < n_mine) {
        bool moved = false;
        if (ky1 < ky0 && mbar_test_wait(smem_u32(&sm.opfull[ky1 & 1u][1]), (ky1 >> 1) & 1u)) {
          tc_fence_after();
          const uint32_t a = ky1 & 1u, e = ky1 % kSsdAcc;
          ssd_issue_y(sm, sm.st[ky1 % kSsdStages], tmem + 128 * a, tmem + 256 + 64 * e, 1, (int)a);
          tc_commit(smem_u32(&sm.aempty[a]));
          tc_commit(smem_u32(&sm.yfull[e]));
          ++ky1;
          moved = true;
        }
        if (ky0 < kg && mbar_test_wait(smem_u32(&sm.opfull[ky0 & 1u][0]), (ky0 >> 1) & 1u) &&
            mbar_test_wait(smem_u32(&sm.yempty[ky0 % kSsdAcc]), ((ky0 / kSsdAcc) & 1u) ^ 1u)) {
          tc_fence_after();
          const uint32_t a = ky0 & 1u, e = ky0 % kSsdAcc;
          ssd_issue_y(sm, sm.st[ky0 % kSsdStages], tmem + 128 * a, tmem + 256 + 64 * e, 0, (int)a);
          ++ky0;
          moved = true;
        }
        if (kg < n_mine && mbar_test_wait(smem_u32(&sm.full[kg % kSsdStages]), (kg / kSsdStages) & 1u) &&
            mbar_test_wait(smem_u32(&sm.aempty[kg & 1u]), ((kg >> 1) & 1u) ^ 1u)) {
          tc_fence_after();
          const SsdStage& st = sm.st[kg % kSsdStages];
          tc_mma_f16(tmem + 128 * (kg & 1u), umma_desc(smem_u32(st.c), 256, 6), umma_desc(smem_u32(st.b), 256, 6),
                     ig, false);
          tc_commit(smem_u32(&sm.gfull[kg & 1u]));
          ++kg;
          moved = true;
        }
        if (moved) {
          idle_since = globaltimer_ns();
        } else {
          if (globaltimer_ns() - idle_since > p.timeout_ns) {
            ok = false;
            break;
          }
        }
      }
    }
  } else if (warp >= 4 && warp < 12) {  // G -> G' in place
    const int q4 = warp & 3, kh = (warp - 4) >> 2, cw = warp - 4;
    const int i = 32 * q4 + lane;  // this thread's row (token of the chunk)
    const uint32_t lanes = (uint32_t)(32 * q4) << 16;
    float* fd = sm.fdt[cw];
    for (uint32_t k = 0; k < n_mine; ++k) {
      const int s = (int)(k % kSsdStages);
      const uint32_t a = k & 1u;
      // G formed in score buffer a (which also means tile k - 2's Y product,
      // and with it its reads of the state operand's buffer a, are done)
      const bool mine = mbar_wait_bounded(smem_u32(&sm.full[s]), (k / kSsdStages) & 1u, p.timeout_ns) &&
                        mbar_wait_bounded(smem_u32(&sm.gfull[a]), (k >> 1) & 1u, p.timeout_ns);
      if (!__all_sync(0xffffffffu, mine)) {
        ok = false;
        break;
      }
      tc_fence_after();
      SsdStage& st = sm.st[s];
      const float ai = st.cum[i].x;
      const uint32_t gbuf = tmem + lanes + 128 * a;
#pragma unroll
      for (int gq = 0; gq < 2; ++gq) {
        const int col0 = 64 * kh + 32 * gq;  // the group's first column (token r)
        uint32_t hi[16], lo[16];
        if (col0 > 32 * q4) {  // above the diagonal for the whole warp: zero
#pragma unroll
          for (int e = 0; e < 16; ++e) hi[e] = lo[e] = 0u;
        } else {
          const float ar = st.cum[col0].x;
          const bool fast = __fsub_rn(ar, st.cum[col0 + 31].x) <= 60.0f;  // the group's decay span
          {
            const float2 v = st.cum[col0 + lane];
            fd[32 * gq + lane] = __fmul_rn(ex2_approx(__fsub_rn(ar, v.x)), v.y);
          }
          __syncwarp();
          const float ri = ex2_approx(__fsub_rn(ai, ar));
          const float2 ri2 = make_float2(ri, ri);
          uint32_t graw[32];
          tmem_ld_32cols(gbuf + col0, graw);
          const bool diag = col0 == 32 * q4;
#pragma unroll
          for (int e4 = 0; e4 < 8; ++e4) {
            float2 f01, f23;
            if (fast) {
              const float4 fv = *reinterpret_cast<const float4*>(fd + 32 * gq + 4 * e4);
              f01 = __fmul2_rn(ri2, make_float2(fv.x, fv.y));
              f23 = __fmul2_rn(ri2, make_float2(fv.z, fv.w));
            } else {
              float f[4];
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                const float2 v = st.cum[col0 + 4 * e4 + u];
                f[u] = __fmul_rn(ex2_approx(__fsub_rn(ai, v.x)), v.y);
              }
              f01 = make_float2(f[0], f[1]);
              f23 = make_float2(f[2], f[3]);
            }
            float2 v01 = __fmul2_rn(make_float2(__uint_as_float(graw[4 * e4]), __uint_as_float(graw[4 * e4 + 1])), f01);
            float2 v23 =
                __fmul2_rn(make_float2(__uint_as_float(graw[4 * e4 + 2]), __uint_as_float(graw[4 * e4 + 3])), f23);
            if (diag) {
              const int j = col0 + 4 * e4;
              if (j > i) v01.x = 0.0f;
              if (j + 1 > i) v01.y = 0.0f;
              if (j + 2 > i) v23.x = 0.0f;
              if (j + 3 > i) v23.y = 0.0f;
            }
            split_bf16_x2(v01, hi[2 * e4], lo[2 * e4]);
            split_bf16_x2(v23, hi[2 * e4 + 1], lo[2 * e4 + 1]);
          }
          __syncwarp();  // fd is read before the next group overwrites it
        }
        // in place: the group's 32 fp32 columns become 16 columns of hi pairs, 16 of lo pairs
        tmem_st_16cols(gbuf + col0, hi);
        tmem_st_16cols(gbuf + col0 + 16, lo);
      }
      if (kh == 1) {  // the entering state: row n, 8 channels (one 16-byte piece) per thread
        const int n = i >> 3, piece = i & 7;
        const float4 v0 = *reinterpret_cast<const float4*>(st.s + n * kSsdP + 8 * piece);
        const float4 v1 = *reinterpret_cast<const float4*>(st.s + n * kSsdP + 8 * piece + 4);
        uint32_t h[4], l[4];
        split_bf16_x2(make_float2(v0.x, v0.y), h[0], l[0]);
        split_bf16_x2(make_float2(v0.z, v0.w), h[1], l[1]);
        split_bf16_x2(make_float2(v1.x, v1.y), h[2], l[2]);
        split_bf16_x2(make_float2(v1.z, v1.w), h[3], l[3]);
        st_shared_v4(sw128(smem_u32(sm.shi[a]), n, piece), h[0], h[1], h[2], h[3]);
        st_shared_v4(sw128(smem_u32(sm.slo[a]), n, piece), l[0], l[1], l[2], l[3]);
        // row i of C times e_i = 2^(acum_i), as hi + lo over the stage's B
        // and C tiles (read by the G product, which is done)
        const float ei = ex2_approx(ai);
        const float2 ei2 = make_float2(ei, ei);
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          uint4 cv;
          asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                       : "=r"(cv.x), "=r"(cv.y), "=r"(cv.z), "=r"(cv.w)
                       : "r"(sw32(smem_u32(st.c), i, q)));
          const uint32_t cw4[4] = {cv.x, cv.y, cv.z, cv.w};
          uint32_t eh[4], el[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) split_bf16_x2(__fmul2_rn(unpack_bf16(cw4[e]), ei2), eh[e], el[e]);
          st_shared_v4(sw32(smem_u32(st.b), i, q), eh[0], eh[1], eh[2], eh[3]);
          st_shared_v4(sw32(smem_u32(st.c), i, q), el[0], el[1], el[2], el[3]);
        }
      }
      fence_proxy_async_smem();  // the shared-memory operands, visible to the tensor core
      tc_fence_before();         // and G' in tensor memory, written, before the MMAs read it
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sm.opfull[a][kh]));
    }
  } else if (warp >= 12) {  // epilogue
    const int q4 = warp & 3;
    const int i = 32 * q4 + lane;
    const uint32_t lanes = (uint32_t)(32 * q4) << 16;
    for (uint32_t k = 0; k < n_mine; ++k) {
      const int s = (int)(k % kSsdStages);
      const uint32_t e = k % kSsdAcc;
      const SsdTileId id = ssd_tile(blockIdx.x + k * gridDim.x, H, nC);
      const float Dh = __ldg(p.Dskip + id.h);  // in flight while the accumulators are waited for
      const bool mine = mbar_wait_bounded(smem_u32(&sm.yfull[e]), (k / kSsdAcc) & 1u, p.timeout_ns) &&
                        mbar_wait_bounded(smem_u32(&sm.full[s]), (k / kSsdStages) & 1u, p.timeout_ns) &&
                        (!gate || mbar_wait_bounded(smem_u32(&sm.zfull[k % kSsdZ]), (k / kSsdZ) & 1u, p.timeout_ns));
      if (!__all_sync(0xffffffffu, mine)) {
        ok = false;
        break;
      }
      tc_fence_after();
      SsdStage& st = sm.st[s];
      const float2 Dh2 = make_float2(Dh, Dh);
      const uint32_t xb = smem_u32(st.x), zb = smem_u32(sm.z[k % kSsdZ]);
      const uint32_t ybuf = tmem + lanes + 256 + 64 * e;
#pragma unroll
      for (int r = 0; r < 4; ++r) {  // 16 channels at a time
        uint32_t yv[16];
        tmem_ld_16cols(ybuf + 16 * r, yv);
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const uint32_t xa = sw128(xb, i, 2 * r + q);
          uint4 xv;
          asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                       : "=r"(xv.x), "=r"(xv.y), "=r"(xv.z), "=r"(xv.w)
                       : "r"(xa));
          const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
          uint4 zv = make_uint4(0u, 0u, 0u, 0u);
          if (gate)
            asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(zv.x), "=r"(zv.y), "=r"(zv.z), "=r"(zv.w)
                         : "r"(sw128(zb, i, 2 * r + q)));
          const uint32_t zw[4] = {zv.x, zv.y, zv.z, zv.w};
          uint32_t out[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int kk = 8 * q + 2 * u;
            float2 y2 = __ffma2_rn(Dh2, unpack_bf16(xw[u]),
                                   make_float2(__uint_as_float(yv[kk]), __uint_as_float(yv[kk + 1])));
            if (gate) y2 = __fmul2_rn(y2, silu_tanh_x2(unpack_bf16(zw[u])));
            out[u] = pack_bf16(y2.x, y2.y);
          }
          st_shared_v4(xa, out[0], out[1], out[2], out[3]);
        }
      }
      tc_fence_before();  // the accumulator is read: accumulator buffer e is free
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(smem_u32(&sm.yempty[e]));
        if (gate) mbar_arrive(smem_u32(&sm.zempty[k % kSsdZ]));  // this warp's rows of z are read
        if (id.c * kSsdQ + 32 * q4 < L) {  // rows past the sequence's end are clipped (or all of them)
          tma_store_4d(&tm_y, 0, id.h, id.c * kSsdQ + 32 * q4, id.b, xb + 32 * q4 * 128);
          bulk_commit();
          bulk_wait_read<0>();  // the rows have left shared memory: this warp's share of the stage is free
        }
        mbar_arrive(smem_u32(&sm.empty[s]));
      }
      __syncwarp();
    }
    if (lane == 0) bulk_wait_all();
  }

  if (!ok) report_error(4u);  // MAMBA_ERR_TIMEOUT
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kSsdTmemCols);
  }
}

}  // namespace mamba
