// scan_fwd.cuh -- prefill kernels of the selective scan.
//
// Work decomposition.  A CTA of 64 threads owns one tile of 16 channels of one
// batch row and one chunk of the sequence (the whole sequence when n_chunks is
// 1), and walks it in tiles of 64 tokens.  Each tile of x, z, dt_raw
// (64 tokens x 16 channels, I/O dtype) and of the token rows of B and C
// (64 x 32 fp32, widened and interleaved beforehand by bc_widen_kernel) is
// brought into shared memory by TMA bulk-tensor copies through a ring of
// three mbarrier-tracked stages, so every input byte is read from HBM once.
//
// Lanes.  Thread (ci = tid >> 2, g = tid & 3) owns states 4g..4g+3 of
// channel ci in registers (fp32).  Tokens go eight at a time; in each step
// lane g first runs the per-token prologue (causal conv, SiLU, softplus,
// silu(z)) of its own two tokens t0+g and t0+4+g, shares (dt, dt*u) with the
// three other lanes of its channel through an 8-entry warp-private buffer,
// advances its four states through the eight tokens, combines the four
// lanes' read-out partials (shuffle reduce-scatter) and finishes its two
// tokens, y = (C.h + D u) silu(z), u and silu(z) still in its registers.  All
// exponentials and products of a step are independent of the state, so they
// are issued ahead of the eight dependent state updates.
//
// The ring is refilled one tile late (the stage of tile k-1 after tile k is
// done), so the previous tile's x rows are still resident and give the conv
// its three earlier inputs; before the first tile those rows of the spare
// stage hold conv_state0 (or the inputs before the chunk).  y leaves through
// a double-buffered shared tile and a TMA store, which clips rows past the end
// of the sequence.  Padding tokens past the end carry dt = dt*u = 0, which
// leaves the state bit-for-bit unchanged (2^0 = 1, fma(1, h, 0) = h).
//
// Chunked mode (n_chunks > 1, chunks a multiple of 64 tokens) is two passes:
// scan_chunk_summary_kernel computes, for every chunk but the last, the end
// state hloc_j of the chunk started from zero and S_j = sum of dt over the
// chunk; the last CTA to finish for a (channel tile, batch row) folds them in
// chunk order into the carried-in state of every chunk,
//   carry_0 = h0,   carry_{j+1} = 2^(A2 S_j) * carry_j + hloc_j,
// and scan_fwd_kernel then runs each chunk from its carry (the "chunked scan
// equals the sequential scan" identity of the oracle).
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>

#include <cstdint>

#include "params.h"
#include "ptx.cuh"
#include "ssm_math.cuh"

namespace mamba {

constexpr int kScanThreads = 64;
constexpr int kT = 64;       // tokens per tile
constexpr int kCT = 16;      // channels per CTA
constexpr int kN = 16;       // d_state
constexpr int kBC = 2 * kN;  // widened B and C per token
constexpr int kStages = 3;   // TMA ring depth

// Sticky device error word (MAMBA_ERR_* code of the first failure).
__device__ unsigned int g_mamba_error;

__device__ __forceinline__ void report_error(unsigned code) { atomicCAS(&g_mamba_error, 0u, code); }

// Bytes to skip from the dynamic shared-memory base to a 128-byte boundary
// (offsetting the __shared__ array itself keeps accesses in the shared space).
__device__ __forceinline__ uint32_t smem_pad128(const void* base) {
  return (128u - (smem_u32(base) & 127u)) & 127u;
}

// Raw input of channel c at token tau of batch row b (tau < 0: conv_state0,
// or zero).
template <typename IO>
__device__ __forceinline__ IO input_raw(const ScanParams& p, int b, long tau, int c) {
  if (tau >= 0) return reinterpret_cast<const IO*>(p.x)[((size_t)b * p.seqlen + tau) * p.d_inner + c];
  if (p.conv_state0 == nullptr) return from_f32<IO>(0.0f);
  return reinterpret_cast<const IO*>(p.conv_state0)[((size_t)b * 3 + (3 + tau)) * p.d_inner + c];
}

// ---------------------------------------------------------------- B, C widening
// bc[row][0..15] = B[row][:], bc[row][16..31] = C[row][:] in fp32, for the
// B*L token rows (64 bytes per token read in bf16), so that the scan's TMA
// brings both rows in one box and the lanes read fp32 directly.
template <typename IO>
__global__ void __launch_bounds__(256) bc_widen_kernel(const IO* __restrict__ Bm, const IO* __restrict__ Cm,
                                                       float* __restrict__ bc, long rows) {
  const long n = rows * 8;  // 8 groups of 4 values per row (4 of B, then 4 of C)
  for (long i = (long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long)gridDim.x * blockDim.x) {
    const long r = i >> 3;
    const int q = (int)(i & 7);
    const IO* src = (q < 4 ? Bm : Cm) + r * kN + (q & 3) * 4;
    const float4 v = make_float4(to_f32(src[0]), to_f32(src[1]), to_f32(src[2]), to_f32(src[3]));
    *reinterpret_cast<float4*>(bc + r * kBC + q * 4) = v;
  }
}

// ---------------------------------------------------------------- shared layout
template <typename IO>
struct ScanStage {
  IO x[kT][kCT];
  IO z[kT][kCT];
  IO dt[kT][kCT];
  float bc[kT][kBC];
};

template <typename IO>
struct ScanSmem {
  ScanStage<IO> stage[kStages];
  IO y[2][kT][kCT];
  float2 dtb[2][kCT][8];  // (dt, dt*u) of a step's 8 tokens per channel, double-buffered
  uint64_t full[kStages];
};

// Issues the copies of one tile; with_z = false skips z (the summary pass).
template <typename IO, bool kWithZ>
__device__ __forceinline__ void issue_tile(ScanStage<IO>& S, uint64_t* bar_ptr, const CUtensorMap* tx,
                                           const CUtensorMap* tz, const CUtensorMap* tdt,
                                           const CUtensorMap* tbc, int c0, int tt, int b) {
  constexpr uint32_t kBytes =
      (kWithZ ? 3 : 2) * kT * kCT * sizeof(IO) + kT * kBC * sizeof(float);
  const uint32_t bar = smem_u32(bar_ptr);
  mbar_arrive_expect_tx(bar, kBytes);
  tma_load_3d(smem_u32(&S.x[0][0]), tx, c0, tt, b, bar);
  if (kWithZ) tma_load_3d(smem_u32(&S.z[0][0]), tz, c0, tt, b, bar);
  tma_load_3d(smem_u32(&S.dt[0][0]), tdt, c0, tt, b, bar);
  tma_load_3d(smem_u32(&S.bc[0][0]), tbc, 0, tt, b, bar);
}

// x of channel ci at tile row r in [-3, 63]: rows < 0 are the previous tile's
// rows 61..63, still resident in the previous stage.
template <typename IO>
__device__ __forceinline__ float x_at(const ScanStage<IO>& S, const ScanStage<IO>& P, int r, int ci) {
  const IO* row = r >= 0 ? &S.x[r][0] : &P.x[kT + r][0];
  return to_f32(row[ci]);
}

// Conv + SiLU of the token at tile row r of channel ci.
template <typename IO>
__device__ __forceinline__ float conv_silu_at(const ScanStage<IO>& S, const ScanStage<IO>& P, int r,
                                              int ci, float4 w, float bias) {
  return silu(conv4(w, bias, x_at<IO>(S, P, r - 3, ci), x_at<IO>(S, P, r - 2, ci),
                    x_at<IO>(S, P, r - 1, ci), x_at<IO>(S, P, r, ci)));
}

// softplus of two dt_raw values; the warp takes the small-dt formula alone
// when all its values allow it (the same formula softplus() selects there).
__device__ __forceinline__ void softplus2(float v0, float v1, float& d0, float& d1) {
  const float e0 = softplus_e(v0), e1 = softplus_e(v1);
  const bool small = (e0 < kSoftplusSmallE) && (e1 < kSoftplusSmallE);
  if (__all_sync(0xffffffffu, small)) {
    d0 = softplus_small(e0);
    d1 = softplus_small(e1);
  } else {
    d0 = e0 < kSoftplusSmallE ? softplus_small(e0) : softplus_large(v0, e0);
    d1 = e1 < kSoftplusSmallE ? softplus_small(e1) : softplus_large(v1, e1);
  }
}

// Writes the raw inputs of tokens t_begin-3 .. t_begin-1 into rows 61..63 of
// the spare stage (the conv's earlier inputs for the first tile) and, from
// chunk 0 only, final_conv_state = the last three inputs of the sequence.
// Chunk 0 is the one CTA of these channels that reads conv_state0, so the
// final state may alias it: everything is read before the barrier.
template <typename IO>
__device__ __forceinline__ void init_halo(const ScanParams& p, ScanStage<IO>& spare, int b, int c0,
                                          int t_begin, bool write_final) {
  const int tid = threadIdx.x;
  const int k = tid >> 4, cc = tid & 15;  // tid < 48: k = 0..2
  IO fv = from_f32<IO>(0.0f);
  const bool fin = write_final && p.final_conv_state != nullptr && tid < 48;
  if (tid < 48) {
    spare.x[kT - 3 + k][cc] = input_raw<IO>(p, b, (long)t_begin - 3 + k, c0 + cc);
    if (fin) fv = input_raw<IO>(p, b, (long)p.seqlen - 3 + k, c0 + cc);
    fence_proxy_async_smem();  // these rows are later overwritten by TMA
  }
  __syncthreads();
  if (fin) reinterpret_cast<IO*>(p.final_conv_state)[((size_t)b * 3 + k) * p.d_inner + c0 + cc] = fv;
}

template <typename IO>
__global__ void __launch_bounds__(kScanThreads)
    scan_fwd_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_z,
                    const __grid_constant__ CUtensorMap tm_dt, const __grid_constant__ CUtensorMap tm_bc,
                    const __grid_constant__ CUtensorMap tm_y, const __grid_constant__ ScanParams p) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  ScanSmem<IO>& sm = *reinterpret_cast<ScanSmem<IO>*>(smem_raw + smem_pad128(smem_raw));

  const int tid = threadIdx.x;
  const int c0 = blockIdx.x * kCT;
  const int b = blockIdx.y;
  const int j = blockIdx.z;
  const int D = p.d_inner;
  const int t_begin = j * p.chunk_len;
  const int t_end = min(t_begin + p.chunk_len, p.seqlen);
  const int n_tiles = (t_end - t_begin + kT - 1) / kT;
  const int ci = tid >> 2, g = tid & 3;
  const int c = c0 + ci;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(smem_u32(&sm.full[s]), 1);
    fence_mbar_init();
    prefetch_tensormap(&tm_x);
    prefetch_tensormap(&tm_z);
    prefetch_tensormap(&tm_dt);
    prefetch_tensormap(&tm_bc);
    prefetch_tensormap(&tm_y);
  }

  // ---- per-thread parameters and initial state
  const float4 w = *reinterpret_cast<const float4*>(p.conv_w + (size_t)c * 4);
  const float bias = p.conv_b ? p.conv_b[c] : 0.0f;
  const float Dc = p.Dskip[c];
  const float4 al = *reinterpret_cast<const float4*>(p.A_log + (size_t)c * kN + 4 * g);
  const float2 a01 = make_float2(a2_from_log(al.x), a2_from_log(al.y));
  const float2 a23 = make_float2(a2_from_log(al.z), a2_from_log(al.w));
  State4 st;
  {
    const float* src = nullptr;
    if (p.n_chunks > 1)
      src = p.carry + (((size_t)b * p.n_chunks + j) * D + c) * kN + 4 * g;
    else if (p.h0)
      src = p.h0 + ((size_t)b * D + c) * kN + 4 * g;
    const float4 h = src ? *reinterpret_cast<const float4*>(src) : make_float4(0.f, 0.f, 0.f, 0.f);
    st.h01 = make_float2(h.x, h.y);
    st.h23 = make_float2(h.z, h.w);
  }
  init_halo<IO>(p, sm.stage[kStages - 1], b, c0, t_begin, j == 0);

  // ---- fill the ring (the last stage is refilled after tile 0)
  const bool stall_test = (p.flags & 1u) != 0;
  if (tid == 0) {
    for (int k = 0; k < kStages - 1 && k < n_tiles; ++k) {
      if (stall_test && k == 0) continue;  // test switch: this stage never completes
      issue_tile<IO, true>(sm.stage[k], &sm.full[k], &tm_x, &tm_z, &tm_dt, &tm_bc, c0, t_begin + k * kT, b);
    }
  }

  bool ok = true;
  int k = 0;
  for (; k < n_tiles; ++k) {
    const int s = k % kStages;
    const int sp = (k + kStages - 1) % kStages;
    const ScanStage<IO>& S = sm.stage[s];
    const ScanStage<IO>& P = sm.stage[sp];
    const int tile_t0 = t_begin + k * kT;
    const int t_valid = min(kT, t_end - tile_t0);
    IO(*ytile)[kCT] = sm.y[k & 1];

    bool mine = mbar_wait_bounded(smem_u32(&sm.full[s]), (k / kStages) & 1, p.timeout_ns);
    mine = __all_sync(0xffffffffu, mine);
    if (mine) {
      const int n_steps = (t_valid + 7) >> 3;
#pragma unroll 1
      for (int oc = 0; oc < n_steps; ++oc) {
        const int t0 = oc * 8;
        const int ra = t0 + g, rb = t0 + 4 + g;
        // prologue of this lane's two tokens
        float da, db;
        softplus2(to_f32(S.dt[ra][ci]), to_f32(S.dt[rb][ci]), da, db);
        const float ua = conv_silu_at<IO>(S, P, ra, ci, w, bias);
        const float ub = conv_silu_at<IO>(S, P, rb, ci, w, bias);
        const float gza = silu(to_f32(S.z[ra][ci]));
        const float gzb = silu(to_f32(S.z[rb][ci]));
        if (ra >= t_valid) da = 0.0f;
        if (rb >= t_valid) db = 0.0f;
        float2(*dtb)[8] = sm.dtb[oc & 1];
        dtb[ci][g] = make_float2(da, __fmul_rn(da, ua));
        dtb[ci][4 + g] = make_float2(db, __fmul_rn(db, ub));
        __syncwarp();
        float dts[8], dtus[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float4 v = *reinterpret_cast<const float4*>(&dtb[ci][2 * i]);
          dts[2 * i] = v.x;
          dtus[2 * i] = v.y;
          dts[2 * i + 1] = v.z;
          dtus[2 * i + 1] = v.w;
        }
        // eight tokens through this lane's four states
        float part[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const float4 Bv = *reinterpret_cast<const float4*>(&S.bc[t0 + q][4 * g]);
          const float4 Cv = *reinterpret_cast<const float4*>(&S.bc[t0 + q][kN + 4 * g]);
          part[q] = state4_step(st, a01, a23, dts[q], dtus[q], Bv, Cv);
        }
        const float Sa = group4_reduce_scatter(part, g);
        const float Sb = group4_reduce_scatter(part + 4, g);
        ytile[ra][ci] = from_f32<IO>(gate_out(Sa, Dc, ua, gza));
        ytile[rb][ci] = from_f32<IO>(gate_out(Sb, Dc, ub, gzb));
      }
      fence_proxy_async_smem();  // y tile -> TMA store
    }
    if (tid == 0) bulk_wait_read<0>();  // tile k-1's store has read the buffer tile k+1 reuses
    ok = __syncthreads_and(mine) != 0;
    if (!ok) break;
    if (tid == 0) {
      tma_store_3d(&tm_y, c0, tile_t0, b, smem_u32(&ytile[0][0]));
      bulk_commit();
      const int kn = k + kStages - 1;  // refill the previous tile's stage
      if (kn < n_tiles)
        issue_tile<IO, true>(sm.stage[sp], &sm.full[sp], &tm_x, &tm_z, &tm_dt, &tm_bc, c0, t_begin + kn * kT, b);
    }
  }

  if (!ok) {
    if (tid == 0) {
      report_error(4u);  // MAMBA_ERR_TIMEOUT
      // let the copies already issued land (bounded) before shared memory goes away
      for (int kk = k; kk < n_tiles && kk < k + kStages - 1; ++kk)
        (void)mbar_wait_bounded(smem_u32(&sm.full[kk % kStages]), (kk / kStages) & 1, p.timeout_ns);
      bulk_wait_all();
    }
    return;
  }
  if (tid == 0) bulk_wait_all();

  if (j == p.n_chunks - 1 && p.final_h) {
    float* dst = p.final_h + ((size_t)b * D + c) * kN + 4 * g;
    *reinterpret_cast<float4*>(dst) = make_float4(st.h01.x, st.h01.y, st.h23.x, st.h23.y);
  }
}

// ---------------------------------------------------------------- chunk summary
// For chunk j < n_chunks-1: the chunk's end state from h = 0 (hloc_j) and the
// sum of its dt (S_j); then the fold of all chunks by the last CTA to finish.
template <typename IO>
struct SummarySmem {
  ScanStage<IO> stage[kStages];  // z unused
  float2 dtb[2][kCT][8];
  uint64_t full[kStages];
  int last;
};

template <typename IO>
__global__ void __launch_bounds__(kScanThreads)
    scan_chunk_summary_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_dt,
                              const __grid_constant__ CUtensorMap tm_bc, const __grid_constant__ ScanParams p) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  SummarySmem<IO>& sm = *reinterpret_cast<SummarySmem<IO>*>(smem_raw + smem_pad128(smem_raw));

  const int tid = threadIdx.x;
  const int c0 = blockIdx.x * kCT;
  const int b = blockIdx.y;
  const int j = blockIdx.z;  // 0 .. n_chunks-2: always full chunks
  const int D = p.d_inner;
  const int t_begin = j * p.chunk_len;
  const int n_tiles = p.chunk_len / kT;
  const int ci = tid >> 2, g = tid & 3;
  const int c = c0 + ci;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(smem_u32(&sm.full[s]), 1);
    fence_mbar_init();
    prefetch_tensormap(&tm_x);
    prefetch_tensormap(&tm_dt);
    prefetch_tensormap(&tm_bc);
  }
  const float4 w = *reinterpret_cast<const float4*>(p.conv_w + (size_t)c * 4);
  const float bias = p.conv_b ? p.conv_b[c] : 0.0f;
  const float4 al = *reinterpret_cast<const float4*>(p.A_log + (size_t)c * kN + 4 * g);
  const float2 a01 = make_float2(a2_from_log(al.x), a2_from_log(al.y));
  const float2 a23 = make_float2(a2_from_log(al.z), a2_from_log(al.w));
  State4 st;
  st.h01 = make_float2(0.f, 0.f);
  st.h23 = make_float2(0.f, 0.f);
  float sdt = 0.0f;
  init_halo<IO>(p, sm.stage[kStages - 1], b, c0, t_begin, false);

  if (tid == 0) {
    for (int k = 0; k < kStages - 1 && k < n_tiles; ++k)
      issue_tile<IO, false>(sm.stage[k], &sm.full[k], &tm_x, nullptr, &tm_dt, &tm_bc, c0, t_begin + k * kT, b);
  }

  bool ok = true;
  int k = 0;
  for (; k < n_tiles; ++k) {
    const int s = k % kStages;
    const int sp = (k + kStages - 1) % kStages;
    const ScanStage<IO>& S = sm.stage[s];
    const ScanStage<IO>& P = sm.stage[sp];
    bool mine = mbar_wait_bounded(smem_u32(&sm.full[s]), (k / kStages) & 1, p.timeout_ns);
    mine = __all_sync(0xffffffffu, mine);
    if (mine) {
#pragma unroll 1
      for (int oc = 0; oc < kT / 8; ++oc) {
        const int t0 = oc * 8;
        const int ra = t0 + g, rb = t0 + 4 + g;
        float da, db;
        softplus2(to_f32(S.dt[ra][ci]), to_f32(S.dt[rb][ci]), da, db);
        const float ua = conv_silu_at<IO>(S, P, ra, ci, w, bias);
        const float ub = conv_silu_at<IO>(S, P, rb, ci, w, bias);
        float2(*dtb)[8] = sm.dtb[oc & 1];
        dtb[ci][g] = make_float2(da, __fmul_rn(da, ua));
        dtb[ci][4 + g] = make_float2(db, __fmul_rn(db, ub));
        __syncwarp();
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float4 v = *reinterpret_cast<const float4*>(&dtb[ci][2 * i]);
          const float4 B0 = *reinterpret_cast<const float4*>(&S.bc[t0 + 2 * i][4 * g]);
          const float4 B1 = *reinterpret_cast<const float4*>(&S.bc[t0 + 2 * i + 1][4 * g]);
          state4_advance(st, a01, a23, v.x, v.y, B0);
          state4_advance(st, a01, a23, v.z, v.w, B1);
          sdt = __fadd_rn(__fadd_rn(sdt, v.x), v.z);
        }
      }
    }
    ok = __syncthreads_and(mine) != 0;
    if (!ok) break;
    if (tid == 0) {
      const int kn = k + kStages - 1;
      if (kn < n_tiles)
        issue_tile<IO, false>(sm.stage[sp], &sm.full[sp], &tm_x, nullptr, &tm_dt, &tm_bc, c0,
                              t_begin + kn * kT, b);
    }
  }
  if (!ok) {
    if (tid == 0) {
      report_error(4u);
      for (int kk = k; kk < n_tiles && kk < k + kStages - 1; ++kk)
        (void)mbar_wait_bounded(smem_u32(&sm.full[kk % kStages]), (kk / kStages) & 1, p.timeout_ns);
    }
    return;
  }

  // ---- publish this chunk's summary
  const int nsum = p.n_chunks - 1;
  {
    const size_t o = ((size_t)b * nsum + j) * D + c;
    *reinterpret_cast<float4*>(p.hloc + o * kN + 4 * g) = make_float4(st.h01.x, st.h01.y, st.h23.x, st.h23.y);
    if (g == 0) p.sum_dt[o] = sdt;
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    unsigned* cnt = p.counters + (size_t)b * (D / kCT) + blockIdx.x;
    const unsigned prev = atomicAdd(cnt, 1u);
    sm.last = (prev == (unsigned)(nsum - 1));
    if (sm.last) *cnt = 0u;  // every chunk of this tile has arrived: reset for the next call
  }
  __syncthreads();
  if (!sm.last) return;
  __threadfence();

  // ---- fold in chunk order: carry_0 = h0, carry_{j+1} = 2^(A2 S_j) carry_j + hloc_j
  float4 h = make_float4(0.f, 0.f, 0.f, 0.f);
  if (p.h0) h = *reinterpret_cast<const float4*>(p.h0 + ((size_t)b * D + c) * kN + 4 * g);
  float* carry = p.carry + ((size_t)b * p.n_chunks * D + c) * kN + 4 * g;
  const size_t cstride = (size_t)D * kN;
  *reinterpret_cast<float4*>(carry) = h;
  for (int jj = 0; jj < nsum; ++jj) {
    const size_t o = ((size_t)b * nsum + jj) * D + c;
    const float4 hl = __ldcg(reinterpret_cast<const float4*>(p.hloc + o * kN + 4 * g));
    const float S = __ldcg(p.sum_dt + o);
    const float2 S2 = make_float2(S, S);
    const float2 x01 = __fmul2_rn(S2, a01), x23 = __fmul2_rn(S2, a23);
    h.x = __fmaf_rn(ex2_approx(x01.x), h.x, hl.x);
    h.y = __fmaf_rn(ex2_approx(x01.y), h.y, hl.y);
    h.z = __fmaf_rn(ex2_approx(x23.x), h.z, hl.z);
    h.w = __fmaf_rn(ex2_approx(x23.y), h.w, hl.w);
    *reinterpret_cast<float4*>(carry + (size_t)(jj + 1) * cstride) = h;
  }
}

}  // namespace mamba
