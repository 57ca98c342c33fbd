// scan_fwd.cuh -- prefill kernels of the selective scan.
//
// Work decomposition.  A CTA is one warp.  Lane i owns channel c0 + i of a
// group of 32 channels of one batch row, with all 16 of its fp32 states in
// registers, and walks one chunk of the sequence in tiles of 32 tokens.  Each
// tile of x, z, dt_raw (32 tokens x 32 channels, I/O dtype) and of the token
// rows of B and C (32 x 32 fp32, widened and interleaved beforehand by
// bc_widen_kernel) is brought into shared memory by TMA bulk-tensor copies
// through a ring of two mbarrier-tracked stages, so every input byte is read
// from HBM once.  B and C are the same for every channel: all lanes read the
// same row, so their 128-bit shared loads are broadcasts.  Nothing is
// exchanged between lanes; the only serial dependence is each state's
// recurrence, and a lane has 16 independent ones plus all the per-token
// exponentials, which do not depend on the state, to overlap with it.
//
// The conv's three earlier inputs travel in registers from token to token
// (loaded from x, or conv_state0, at the chunk start).  y is stored straight
// from registers (a warp writes 32 consecutive channels of one token).
//
// Chunked mode.  At batch 1 the groups alone cannot fill the GPU, so the
// sequence is cut into n_chunks chunks that run in parallel, each starting
// from its carried-in state.  Those carries come from a first pass,
// scan_piece_summary_kernel: every chunk but the last is cut into pieces; for
// each piece it computes the end state hloc of the piece started from zero and
// S = sum of dt over the piece; the last CTA to finish for a (group, batch
// row) folds the pieces in order,
//   carry <- h0;   for each piece: carry <- 2^(A2 S) carry + hloc
// writing the carry at every chunk boundary (the "chunked scan equals the
// sequential scan" identity of the oracle).  The fold order is fixed, so the
// result does not depend on timing.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>

#include <cstdint>

#include "params.h"
#include "ptx.cuh"
#include "ssm_math.cuh"

namespace mamba {

constexpr int kLanes = 32;   // channels per CTA (one warp)
constexpr int kT = kTileTokens;
constexpr int kBC = 2 * kN;  // widened B and C per token
constexpr int kStages = 2;   // TMA ring depth
constexpr int kScanUnroll = 4;  // tokens unrolled in the tile loops

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
__device__ __forceinline__ float input_at(const ScanParams& p, int b, long tau, int c) {
  if (tau >= 0) return to_f32(reinterpret_cast<const IO*>(p.x)[((size_t)b * p.seqlen + tau) * p.d_inner + c]);
  if (p.conv_state0 == nullptr) return 0.0f;
  return to_f32(reinterpret_cast<const IO*>(p.conv_state0)[((size_t)b * 3 + (3 + tau)) * p.d_inner + c]);
}

// ---------------------------------------------------------------- B, C widening
// bc[row][0..15] = B[row][:], bc[row][16..31] = C[row][:] in fp32, for the
// B*L token rows (64 bytes per token read in bf16), so that one TMA box
// carries both rows and the lanes read fp32 directly.
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
struct MainStage {
  IO x[kT][kLanes];
  IO z[kT][kLanes];
  IO dt[kT][kLanes];
  float bc[kT][kBC];
};

template <typename IO>
struct MainSmem {
  MainStage<IO> stage[kStages];
  uint64_t full[kStages];
};

template <typename IO>
struct SummaryStage {
  IO x[kT][kLanes];
  IO dt[kT][kLanes];
  float b[kT][kN];
};

template <typename IO>
struct SummarySmem {
  SummaryStage<IO> stage[kStages];
  uint64_t full[kStages];
  int last;
};

__device__ __forceinline__ void load_bc4(const float* row, float4 (&v)[4]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) v[q] = *reinterpret_cast<const float4*>(row + 4 * q);
}

// Lets the copies already issued land (bounded) before shared memory goes away.
__device__ __forceinline__ void drain_ring(uint64_t* full, int k, int n_tiles, uint64_t timeout_ns) {
  for (int kk = k; kk < n_tiles && kk < k + kStages; ++kk)
    (void)mbar_wait_bounded(smem_u32(&full[kk % kStages]), (kk / kStages) & 1, timeout_ns);
}

// True when every dt_raw of the tile's first `rows` rows (over the active
// lanes) lies in softplus's small-e region, checked on the raw value.
template <typename IO>
__device__ __forceinline__ bool small_dt_tile(const IO (&dt)[kT][kLanes], int rows, int lane, bool active) {
  float m = -3.0e38f;
#pragma unroll 8
  for (int r = 0; r < rows; ++r) m = fmaxf(m, to_f32(dt[r][lane]));
  return __all_sync(0xffffffffu, !active || m < kSoftplusSmallRaw);
}

template <bool kSmall>
__device__ __forceinline__ float softplus_sel(float v) {
  return kSmall ? softplus_small_raw(v) : softplus(v);
}

// One tile of the main pass, `rows` tokens, straight-line per token.
template <typename IO, bool kSmall>
__device__ __forceinline__ void main_tile(const MainStage<IO>& S, int rows, int lane, bool active,
                                          const Channel& ch, State16& st, float& xm3, float& xm2, float& xm1,
                                          IO* ytile, int D) {
#pragma unroll(kScanUnroll)
  for (int r = 0; r < rows; ++r) {
    const float xv = to_f32(S.x[r][lane]);
    const float u = silu(conv4(ch.w, ch.bias, xm3, xm2, xm1, xv));
    xm3 = xm2;
    xm2 = xm1;
    xm1 = xv;
    const float dt = softplus_sel<kSmall>(to_f32(S.dt[r][lane]));
    const float gz = silu(to_f32(S.z[r][lane]));
    float4 Bv[4], Cv[4];
    load_bc4(&S.bc[r][0], Bv);
    load_bc4(&S.bc[r][kN], Cv);
    state16_advance(st, ch.a2, dt, __fmul_rn(dt, u), Bv);
    const float yv = gate_out(state16_readout(st, Cv), ch.Dc, u, gz);
    st_global_if(active, ytile + (size_t)r * D, from_f32<IO>(yv));
  }
}

// One full tile of the summary pass.
template <typename IO, bool kSmall>
__device__ __forceinline__ void summary_tile(const SummaryStage<IO>& S, int lane, const Channel& ch, State16& st,
                                             float& sdt, float& xm3, float& xm2, float& xm1) {
#pragma unroll(kScanUnroll)
  for (int r = 0; r < kT; ++r) {
    const float xv = to_f32(S.x[r][lane]);
    const float u = silu(conv4(ch.w, ch.bias, xm3, xm2, xm1, xv));
    xm3 = xm2;
    xm2 = xm1;
    xm1 = xv;
    const float dt = softplus_sel<kSmall>(to_f32(S.dt[r][lane]));
    float4 Bv[4];
    load_bc4(&S.b[r][0], Bv);
    state16_advance(st, ch.a2, dt, __fmul_rn(dt, u), Bv);
    sdt = __fadd_rn(sdt, dt);
  }
}

// ---------------------------------------------------------------- main pass
// grid (n_groups, batch, n_chunks), 32 threads.
template <typename IO>
__global__ void __launch_bounds__(kLanes)
    scan_fwd_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_z,
                    const __grid_constant__ CUtensorMap tm_dt, const __grid_constant__ CUtensorMap tm_bc,
                    const __grid_constant__ ScanParams p) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  MainSmem<IO>& sm = *reinterpret_cast<MainSmem<IO>*>(smem_raw + smem_pad128(smem_raw));

  const int lane = threadIdx.x;
  const int c0 = blockIdx.x * kLanes;
  const int b = blockIdx.y;
  const int j = blockIdx.z;
  const int D = p.d_inner;
  const int c = c0 + lane;
  const bool active = c < D;
  const int cl = active ? c : D - 1;  // channel whose parameters an idle lane reads
  const int t_begin = j * p.chunk_tiles * kT;
  const int t_end = min(t_begin + p.chunk_tiles * kT, p.seqlen);
  const int n_tiles = (t_end - t_begin + kT - 1) / kT;

  if (lane == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(smem_u32(&sm.full[s]), 1);
    fence_mbar_init();
    prefetch_tensormap(&tm_x);
    prefetch_tensormap(&tm_z);
    prefetch_tensormap(&tm_dt);
    prefetch_tensormap(&tm_bc);
  }
  __syncwarp();

  const bool stall_test = (p.flags & 1u) != 0;
  if (lane == 0) {
    constexpr uint32_t kBytes = 3 * kT * kLanes * sizeof(IO) + kT * kBC * sizeof(float);
    for (int k = 0; k < kStages && k < n_tiles; ++k) {
      if (stall_test && k == 0) continue;  // test switch: this stage never completes
      const uint32_t bar = smem_u32(&sm.full[k]);
      const int tt = t_begin + k * kT;
      mbar_arrive_expect_tx(bar, kBytes);
      tma_load_3d(smem_u32(&sm.stage[k].x[0][0]), &tm_x, c0, tt, b, bar);
      tma_load_3d(smem_u32(&sm.stage[k].z[0][0]), &tm_z, c0, tt, b, bar);
      tma_load_3d(smem_u32(&sm.stage[k].dt[0][0]), &tm_dt, c0, tt, b, bar);
      tma_load_3d(smem_u32(&sm.stage[k].bc[0][0]), &tm_bc, 0, tt, b, bar);
    }
  }

  Channel ch;
  load_channel(ch, p.A_log, p.conv_w, p.conv_b, p.Dskip, cl);
  State16 st;
  if (j > 0)
    state16_load(st, p.carry + (((size_t)b * p.n_chunks + j) * D + cl) * kN);
  else if (p.h0)
    state16_load(st, p.h0 + ((size_t)b * D + cl) * kN);
  else
    state16_zero(st);

  // the conv's earlier inputs; chunk 0 also writes the final conv state (it
  // is the one CTA of these channels that reads conv_state0, which the final
  // state may alias: everything is read before anything is written)
  float xm3 = input_at<IO>(p, b, (long)t_begin - 3, cl);
  float xm2 = input_at<IO>(p, b, (long)t_begin - 2, cl);
  float xm1 = input_at<IO>(p, b, (long)t_begin - 1, cl);
  if (j == 0 && p.final_conv_state != nullptr) {
    const float f0 = input_at<IO>(p, b, (long)p.seqlen - 3, cl);
    const float f1 = input_at<IO>(p, b, (long)p.seqlen - 2, cl);
    const float f2 = input_at<IO>(p, b, (long)p.seqlen - 1, cl);
    __syncwarp();
    if (active) {
      IO* fcs = reinterpret_cast<IO*>(p.final_conv_state) + (size_t)b * 3 * D + c;
      fcs[0] = from_f32<IO>(f0);
      fcs[D] = from_f32<IO>(f1);
      fcs[2 * (size_t)D] = from_f32<IO>(f2);
    }
  }

  IO* yrow = reinterpret_cast<IO*>(p.y) + ((size_t)b * p.seqlen + t_begin) * D + cl;
  bool ok = true;
  int k = 0;
  for (; k < n_tiles; ++k) {
    const int s = k % kStages;
    const MainStage<IO>& S = sm.stage[s];
    const int t_valid = min(kT, t_end - (t_begin + k * kT));
    bool mine = mbar_wait_bounded(smem_u32(&sm.full[s]), (k / kStages) & 1, p.timeout_ns);
    ok = __all_sync(0xffffffffu, mine);
    if (!ok) break;
    if (small_dt_tile<IO>(S.dt, t_valid, lane, active))
      main_tile<IO, true>(S, t_valid, lane, active, ch, st, xm3, xm2, xm1, yrow + (size_t)k * kT * D, D);
    else
      main_tile<IO, false>(S, t_valid, lane, active, ch, st, xm3, xm2, xm1, yrow + (size_t)k * kT * D, D);
    __syncwarp();  // every lane is done with stage s
    if (lane == 0 && k + kStages < n_tiles) {
      constexpr uint32_t kBytes = 3 * kT * kLanes * sizeof(IO) + kT * kBC * sizeof(float);
      const uint32_t bar = smem_u32(&sm.full[s]);
      const int tt = t_begin + (k + kStages) * kT;
      mbar_arrive_expect_tx(bar, kBytes);
      tma_load_3d(smem_u32(&sm.stage[s].x[0][0]), &tm_x, c0, tt, b, bar);
      tma_load_3d(smem_u32(&sm.stage[s].z[0][0]), &tm_z, c0, tt, b, bar);
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
  if (j == p.n_chunks - 1 && p.final_h && active) state16_store(st, p.final_h + ((size_t)b * D + c) * kN);
}

// ---------------------------------------------------------------- piece summaries
// grid (n_groups, batch, (n_chunks - 1) * pieces), 32 threads.  Piece q of
// chunk jc covers tiles [jc*C + q*P, min(jc*C + (q+1)*P, (jc+1)*C)).
template <typename IO>
__global__ void __launch_bounds__(kLanes)
    scan_piece_summary_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_dt,
                              const __grid_constant__ CUtensorMap tm_b, const __grid_constant__ ScanParams p) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  SummarySmem<IO>& sm = *reinterpret_cast<SummarySmem<IO>*>(smem_raw + smem_pad128(smem_raw));

  const int lane = threadIdx.x;
  const int c0 = blockIdx.x * kLanes;
  const int b = blockIdx.y;
  const int piece = blockIdx.z;  // 0 .. (n_chunks-1)*pieces - 1
  const int jc = piece / p.pieces;
  const int q = piece - jc * p.pieces;
  const int D = p.d_inner;
  const int c = c0 + lane;
  const bool active = c < D;
  const int cl = active ? c : D - 1;
  const int tile0 = jc * p.chunk_tiles + q * p.piece_tiles;
  const int tile1 = min(tile0 + p.piece_tiles, (jc + 1) * p.chunk_tiles);
  const int t_begin = tile0 * kT;
  const int n_tiles = tile1 - tile0;  // >= 1: chunks before the last are full

  if (lane == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(smem_u32(&sm.full[s]), 1);
    fence_mbar_init();
    prefetch_tensormap(&tm_x);
    prefetch_tensormap(&tm_dt);
    prefetch_tensormap(&tm_b);
  }
  __syncwarp();
  constexpr uint32_t kBytes = 2 * kT * kLanes * sizeof(IO) + kT * kN * sizeof(float);
  if (lane == 0) {
    for (int k = 0; k < kStages && k < n_tiles; ++k) {
      const uint32_t bar = smem_u32(&sm.full[k]);
      const int tt = t_begin + k * kT;
      mbar_arrive_expect_tx(bar, kBytes);
      tma_load_3d(smem_u32(&sm.stage[k].x[0][0]), &tm_x, c0, tt, b, bar);
      tma_load_3d(smem_u32(&sm.stage[k].dt[0][0]), &tm_dt, c0, tt, b, bar);
      tma_load_3d(smem_u32(&sm.stage[k].b[0][0]), &tm_b, 0, tt, b, bar);
    }
  }

  Channel ch;
  load_channel(ch, p.A_log, p.conv_w, p.conv_b, p.Dskip, cl);
  State16 st;
  state16_zero(st);
  float sdt = 0.0f;
  float xm3 = input_at<IO>(p, b, (long)t_begin - 3, cl);
  float xm2 = input_at<IO>(p, b, (long)t_begin - 2, cl);
  float xm1 = input_at<IO>(p, b, (long)t_begin - 1, cl);

  bool ok = true;
  int k = 0;
  for (; k < n_tiles; ++k) {
    const int s = k % kStages;
    const SummaryStage<IO>& S = sm.stage[s];
    bool mine = mbar_wait_bounded(smem_u32(&sm.full[s]), (k / kStages) & 1, p.timeout_ns);
    ok = __all_sync(0xffffffffu, mine);
    if (!ok) break;
    if (small_dt_tile<IO>(S.dt, kT, lane, active))
      summary_tile<IO, true>(S, lane, ch, st, sdt, xm3, xm2, xm1);
    else
      summary_tile<IO, false>(S, lane, ch, st, sdt, xm3, xm2, xm1);
    __syncwarp();
    if (lane == 0 && k + kStages < n_tiles) {
      const uint32_t bar = smem_u32(&sm.full[s]);
      const int tt = t_begin + (k + kStages) * kT;
      mbar_arrive_expect_tx(bar, kBytes);
      tma_load_3d(smem_u32(&sm.stage[s].x[0][0]), &tm_x, c0, tt, b, bar);
      tma_load_3d(smem_u32(&sm.stage[s].dt[0][0]), &tm_dt, c0, tt, b, bar);
      tma_load_3d(smem_u32(&sm.stage[s].b[0][0]), &tm_b, 0, tt, b, bar);
    }
  }
  if (!ok) {
    if (lane == 0) {
      report_error(4u);
      drain_ring(sm.full, k, n_tiles, p.timeout_ns);
    }
    return;
  }

  // ---- publish this piece's summary
  const int npieces = (p.n_chunks - 1) * p.pieces;
  const size_t o = ((size_t)b * npieces + piece) * D + cl;
  if (active) {
    state16_store(st, p.hloc + o * kN);
    p.sum_dt[o] = sdt;
  }
  __threadfence();
  __syncwarp();
  if (lane == 0) {
    unsigned* cnt = p.counters + (size_t)b * p.n_groups + blockIdx.x;
    const unsigned prev = atomicAdd(cnt, 1u);
    sm.last = (prev == (unsigned)(npieces - 1));
    if (sm.last) *cnt = 0u;  // every piece of this group has arrived: reset for the next call
  }
  __syncwarp();
  if (!sm.last) return;
  __threadfence();

  // ---- fold in piece order; the carry at the end of chunk jc is chunk jc+1's start
  if (!active) return;
  State16 h;
  if (p.h0)
    state16_load(h, p.h0 + ((size_t)b * D + c) * kN);
  else
    state16_zero(h);
  for (int pc = 0; pc < npieces; ++pc) {
    const size_t oo = ((size_t)b * npieces + pc) * D + c;
    State16 hl;
    const float4* src = reinterpret_cast<const float4*>(p.hloc + oo * kN);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      const float4 v = __ldcg(src + kk);
      hl.h[2 * kk] = make_float2(v.x, v.y);
      hl.h[2 * kk + 1] = make_float2(v.z, v.w);
    }
    state16_fold(h, ch.a2, __ldcg(p.sum_dt + oo), hl);
    if ((pc + 1) % p.pieces == 0) {
      const int jn = (pc + 1) / p.pieces;  // the chunk this carry starts
      state16_store(h, p.carry + (((size_t)b * p.n_chunks + jn) * D + c) * kN);
    }
  }
}

}  // namespace mamba
