// scan_fwd.cuh -- prefill kernels of the selective scan.
//
// Work decomposition.  A CTA is one warp.  Lane i owns channel c0 + i of a
// group of 32 channels of one batch row, with all 16 of its fp32 states in
// registers, and walks one chunk of the sequence in tiles of 16 tokens.  Each
// tile of x, z, dt_raw (16 tokens x 32 channels, I/O dtype) and of the token
// rows of B and C (16 x 32 fp32, widened and interleaved beforehand by
// bc_widen_kernel) is brought into shared memory by TMA bulk-tensor copies
// through a ring of two mbarrier-tracked stages, so every input byte is read
// from HBM once.  B and C are the same for every channel: all lanes read the
// same row, so their 128-bit shared loads are broadcasts.  Nothing is
// exchanged between lanes; the only serial dependence is each state's
// recurrence, and a lane has 16 independent ones plus all the per-token
// exponentials, which do not depend on the state, to overlap with it.  In
// tiles whose dt_raw all lie in softplus's small region (the common case),
// the per-token scalar work of two consecutive tokens runs as packed f32x2
// operations.
//
// The conv's three earlier inputs travel in registers from token to token
// (loaded from x, or conv_state0, at the chunk start).  y is stored straight
// from registers (a warp writes 32 consecutive channels of one token).
//
// Chunked mode.  At batch 1 the groups alone cannot fill the GPU, so the
// sequence is cut into n_chunks chunks that run in parallel, each starting
// from its carried-in state.  Those carries come from carry walks
// (carry_warp, described with it below) that run in the same launch as the
// main pass (scan_fused_kernel, at the end): one warp per chunk boundary
// and channel group walks the previous chunk backwards in pieces and stops
// where the decay to the boundary makes earlier tokens negligible (below
// 2^-32 for every state), or else chains onto the previous boundary's carry;
// on the way, each piece advances only the state pairs whose decay to the
// boundary is not yet below that bound.
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

// The chunk-carry walks drop terms whose weight to the boundary is below
// 2^-32 of their own size.
constexpr float kCarryDropLog2 = -32.0f;
constexpr float kCarryDropWeight = 2.3283064365386963e-10f;  // 2^-32

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
// B and C rows widened to fp32 in pair-quad layout: bc[row][4k .. 4k+3] =
// (B_2k, B_2k+1, C_2k, C_2k+1) for the state pairs k = 0..7, for the B*L
// token rows (64 bytes per token read in bf16).  One TMA box carries both
// rows; one 128-bit shared load gives a lane the B and C values of one state
// pair as two aligned register pairs.
// ld: elements from one token's row of B (and of C) to the next (16 when
// they are (B, L, 16) tensors; more when they are columns of a wider
// projection output).
//
// kModePairs (the complex scan, whose rows hold 8 complex numbers (re, im)):
// per pair of modes q = 0..3 the quads bc[row][8q .. 8q+3] = (Re B_2q,
// Re B_2q+1, Im B_2q, Im B_2q+1) and bc[row][8q+4 .. 8q+7] the same of C, so
// that each quad gives a lane two aligned register pairs across two modes.
//
// Launched as a programmatic dependent (the forward's chunked mode) it waits
// for the kernel before it (the previous call's scan, which reads bc) before
// touching memory, then lets the scan after it launch; block 0 also zeroes
// that scan's ticket counter and flags (n_counters words, when given).
template <typename IO, bool kModePairs>
__global__ void __launch_bounds__(256) bc_widen_kernel(const IO* __restrict__ Bm, const IO* __restrict__ Cm,
                                                       float* __restrict__ bc, long rows, int ld,
                                                       unsigned* __restrict__ counters, int n_counters) {
  griddep_wait();
  griddep_launch_dependents();
  if (blockIdx.x == 0)
    for (int i = threadIdx.x; i < n_counters; i += blockDim.x) counters[i] = 0u;
  const long n = rows * 8;  // 8 quads per row
  for (long i = (long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long)gridDim.x * blockDim.x) {
    const long r = i >> 3;
    const int k = (int)(i & 7);
    float4 v;
    if (kModePairs) {
      const IO* s = ((k & 1) ? Cm : Bm) + r * ld + 4 * (k >> 1);
      v = make_float4(to_f32(s[0]), to_f32(s[2]), to_f32(s[1]), to_f32(s[3]));
    } else {
      const IO* b = Bm + r * ld + 2 * k;
      const IO* c = Cm + r * ld + 2 * k;
      v = make_float4(to_f32(b[0]), to_f32(b[1]), to_f32(c[0]), to_f32(c[1]));
    }
    *reinterpret_cast<float4*>(bc + r * kBC + 4 * k) = v;
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
  float bc[kT][kBC];  // B and C (only B is used: the quads interleave them)
};


__device__ __forceinline__ void load_quads(const float* row, float4 (&Q)[8]) {
#pragma unroll
  for (int k = 0; k < 8; ++k) Q[k] = *reinterpret_cast<const float4*>(row + 4 * k);
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

// One token r of a tile of the main pass; y is stored where wy holds.  kY
// false: the states alone (z, the read-out and y are skipped).
template <typename IO, bool kSmall, bool kY>
__device__ __forceinline__ void main_token(const MainStage<IO>& S, int r, int lane, bool wy, const Channel& ch,
                                           State16& st, float& xm3, float& xm2, float& xm1, IO* ytile, int D) {
  const float xv = to_f32(S.x[r][lane]);
  const float u = silu(conv4(ch.w, ch.bias, xm3, xm2, xm1, xv));
  xm3 = xm2;
  xm2 = xm1;
  xm1 = xv;
  const float dt = softplus_sel<kSmall>(to_f32(S.dt[r][lane]));
  float4 Q[8];
  load_quads(&S.bc[r][0], Q);
  Drive16 d;
  drive16_q(d, ch.a2, dt, __fmul_rn(dt, u), Q);
  state16_apply(st, d);
  if (kY) {
    const float gz = silu(to_f32(S.z[r][lane]));
    const float yv = gate_out(state16_readout_q(st, Q), ch.Dc, u, gz);
    st_global_if(wy, ytile + (size_t)r * D, from_f32<IO>(yv));
  }
}

// Tokens r and r+1, both with dt_raw in softplus's small region: the
// per-token scalar work (conv, SiLU, softplus, dt*u, SiLU(z), gate) of the
// two tokens runs as packed f32x2 operations, the same operations as
// main_token's on each (the same bits), in about half the instructions.
template <typename IO, bool kY>
__device__ __forceinline__ void main_token_pair(const MainStage<IO>& S, int r, int lane, bool wy,
                                                const Channel& ch, State16& st, float& xm3, float& xm2, float& xm1,
                                                IO* ytile, int D) {
  const float x0 = to_f32(S.x[r][lane]);
  const float x1 = to_f32(S.x[r + 1][lane]);
  const float2 u = silu_x2(conv4_x2(ch.w, ch.bias, xm3, xm2, xm1, x0, x1));
  xm3 = xm1;
  xm2 = x0;
  xm1 = x1;
  const float2 dt = softplus_small_raw_x2(make_float2(to_f32(S.dt[r][lane]), to_f32(S.dt[r + 1][lane])));
  const float2 dtu = __fmul2_rn(dt, u);
  float2 ss = make_float2(0.0f, 0.0f);
  {
    float4 Q[8];
    load_quads(&S.bc[r][0], Q);
    Drive16 d;
    drive16_q(d, ch.a2, dt.x, dtu.x, Q);
    state16_apply(st, d);
    if (kY) ss.x = state16_readout_q(st, Q);
  }
  {
    float4 Q[8];
    load_quads(&S.bc[r + 1][0], Q);
    Drive16 d;
    drive16_q(d, ch.a2, dt.y, dtu.y, Q);
    state16_apply(st, d);
    if (kY) ss.y = state16_readout_q(st, Q);
  }
  if (kY) {
    const float2 gz = silu_x2(make_float2(to_f32(S.z[r][lane]), to_f32(S.z[r + 1][lane])));
    const float2 yv = gate_out_x2(ss, ch.Dc, u, gz);
    st_global_if(wy, ytile + (size_t)r * D, from_f32<IO>(yv.x));
    st_global_if(wy, ytile + (size_t)(r + 1) * D, from_f32<IO>(yv.y));
  }
}

// One tile of the main pass, `rows` tokens, straight-line per token (per
// token pair in small-dt tiles).  kFull: rows == kT, unrolled completely.
template <typename IO, bool kSmall, bool kFull, bool kY>
__device__ __forceinline__ void main_tile(const MainStage<IO>& S, int rows, int lane, bool wy,
                                          const Channel& ch, State16& st, float& xm3, float& xm2, float& xm1,
                                          IO* ytile, int D) {
  if (kFull) rows = kT;
  if (kSmall) {
    int r = 0;
#pragma unroll(kFull ? kT / 2 : kScanUnroll / 2)
    for (; r + 1 < rows; r += 2)
      main_token_pair<IO, kY>(S, r, lane, wy, ch, st, xm3, xm2, xm1, ytile, D);
    if (!kFull && r < rows) main_token<IO, true, kY>(S, r, lane, wy, ch, st, xm3, xm2, xm1, ytile, D);
  } else {
#pragma unroll(kFull ? kT : kScanUnroll)
    for (int r = 0; r < rows; ++r) main_token<IO, false, kY>(S, r, lane, wy, ch, st, xm3, xm2, xm1, ytile, D);
  }
}

// One full tile of a carry piece (state and dt sum only), advancing the
// first kPairs state pairs (the later ones, whose decay to the boundary is
// already below the drop bound, stay as they are: zero within the piece).
// Tiles whose dt_raw all lie in softplus's small region (kSmall) take their
// tokens two at a time, the per-token scalar work (conv, SiLU, softplus,
// dt*u) of the two as packed f32x2 operations: the same operations on each
// token, so the same bits.
template <typename IO, bool kSmall, int kPairs>
__device__ __forceinline__ void summary_tile(const SummaryStage<IO>& S, int lane, const Channel& ch, State16& st,
                                             float& sdt, float& xm3, float& xm2, float& xm1) {
  if constexpr (kSmall) {
#pragma unroll(kScanUnroll / 2)
    for (int r = 0; r < kT; r += 2) {
      const float x0 = to_f32(S.x[r][lane]);
      const float x1 = to_f32(S.x[r + 1][lane]);
      const float2 u = silu_x2(conv4_x2(ch.w, ch.bias, xm3, xm2, xm1, x0, x1));
      xm3 = xm1;
      xm2 = x0;
      xm1 = x1;
      const float2 dt = softplus_small_raw_x2(make_float2(to_f32(S.dt[r][lane]), to_f32(S.dt[r + 1][lane])));
      const float2 dtu = __fmul2_rn(dt, u);
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const float2 d2 = i ? make_float2(dt.y, dt.y) : make_float2(dt.x, dt.x);
        const float2 u2 = i ? make_float2(dtu.y, dtu.y) : make_float2(dtu.x, dtu.x);
#pragma unroll
        for (int k = 0; k < kPairs; ++k) {
          const float4 q = *reinterpret_cast<const float4*>(&S.bc[r + i][4 * k]);
          const float2 x = __fmul2_rn(d2, ch.a2[k]);
          const float2 dA = make_float2(ex2_approx(x.x), ex2_approx(x.y));
          st.h[k] = __ffma2_rn(dA, st.h[k], __fmul2_rn(u2, make_float2(q.x, q.y)));
        }
      }
      sdt = __fadd_rn(__fadd_rn(sdt, dt.x), dt.y);
    }
  } else {
#pragma unroll(kScanUnroll)
    for (int r = 0; r < kT; ++r) {
      const float xv = to_f32(S.x[r][lane]);
      const float u = silu(conv4(ch.w, ch.bias, xm3, xm2, xm1, xv));
      xm3 = xm2;
      xm2 = xm1;
      xm1 = xv;
      const float dt = softplus_sel<kSmall>(to_f32(S.dt[r][lane]));
      const float2 d2 = make_float2(dt, dt);
      const float dtu = __fmul_rn(dt, u);
      const float2 u2 = make_float2(dtu, dtu);
#pragma unroll
      for (int k = 0; k < kPairs; ++k) {  // the operations of drive16_q and state16_apply, pair by pair
        const float4 q = *reinterpret_cast<const float4*>(&S.bc[r][4 * k]);
        const float2 x = __fmul2_rn(d2, ch.a2[k]);
        const float2 dA = make_float2(ex2_approx(x.x), ex2_approx(x.y));
        st.h[k] = __ffma2_rn(dA, st.h[k], __fmul2_rn(u2, make_float2(q.x, q.y)));
      }
      sdt = __fadd_rn(sdt, dt);
    }
  }
}

template <typename IO, bool kSmall>
__device__ __forceinline__ void summary_tile_n(int n_pairs, const SummaryStage<IO>& S, int lane, const Channel& ch,
                                               State16& st, float& sdt, float& xm3, float& xm2, float& xm1) {
  if (n_pairs <= 1)
    summary_tile<IO, kSmall, 1>(S, lane, ch, st, sdt, xm3, xm2, xm1);
  else if (n_pairs <= 2)
    summary_tile<IO, kSmall, 2>(S, lane, ch, st, sdt, xm3, xm2, xm1);
  else if (n_pairs <= 4)
    summary_tile<IO, kSmall, 4>(S, lane, ch, st, sdt, xm3, xm2, xm1);
  else
    summary_tile<IO, kSmall, 8>(S, lane, ch, st, sdt, xm3, xm2, xm1);
}

// Number of leading state pairs whose weight to the boundary (wgt, over the
// active lanes) is still at or above the drop bound: 1 + the last such pair,
// 0 when none is.
__device__ __forceinline__ int live_pairs(const State16& wgt, bool active) {
  int last = -1;
#pragma unroll
  for (int k = 0; k < 8; ++k)
    if (fmaxf(wgt.h[k].x, wgt.h[k].y) >= kCarryDropWeight) last = k;
  return __reduce_max_sync(0xffffffffu, active ? last + 1 : 0);
}

// ---------------------------------------------------------------- main pass
// One warp per (channel group g, batch row b, chunk j).  kY false: no y (and
// no z): the pass only stores the states entering every tile (p.ckpt), for
// the backward.  wait_carry: the carry entering chunk j is published during
// this launch (the fused kernel below); wait (bounded) for its flag first.
template <typename IO, bool kY>
__device__ __forceinline__ void main_warp(const CUtensorMap& tm_x, const CUtensorMap& tm_z, const CUtensorMap& tm_dt,
                                          const CUtensorMap& tm_bc, const ScanParams& p, MainSmem<IO>& sm, int g,
                                          int b, int j, bool wait_carry) {
  const int lane = threadIdx.x;
  const int c0 = g * kLanes;
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

  const bool stall_test = (p.flags & kFlagTestStallFirstLoad) != 0;
  constexpr uint32_t kBytes = (kY ? 3 : 2) * kT * kLanes * sizeof(IO) + kT * kBC * sizeof(float);
  if (lane == 0) {
    for (int k = 0; k < kStages && k < n_tiles; ++k) {
      if (stall_test && k == 0) continue;  // test switch: this stage never completes
      const uint32_t bar = smem_u32(&sm.full[k]);
      const int tt = t_begin + k * kT;
      mbar_arrive_expect_tx(bar, kBytes);
      tma_load_3d(smem_u32(&sm.stage[k].x[0][0]), &tm_x, c0, tt, b, bar);
      if (kY) tma_load_3d(smem_u32(&sm.stage[k].z[0][0]), &tm_z, c0, tt, b, bar);
      tma_load_3d(smem_u32(&sm.stage[k].dt[0][0]), &tm_dt, c0, tt, b, bar);
      tma_load_3d(smem_u32(&sm.stage[k].bc[0][0]), &tm_bc, 0, tt, b, bar);
    }
  }

  Channel ch;
  load_channel(ch, p.A_log, p.conv_w, p.conv_b, p.Dskip, cl);
  State16 st;
  if (j > 0 && wait_carry) {
    bool have = true;
    if (lane == 0) {
      const unsigned* ready = p.counters + 1 + (size_t)b * p.n_groups * p.n_chunks + (size_t)g * p.n_chunks;
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
      state16_zero(st);
    } else {
      const float4* src = reinterpret_cast<const float4*>(p.carry + (((size_t)b * p.n_chunks + j) * D + cl) * kN);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {  // from L2: written by another SM during this launch
        const float4 v = __ldcg(src + kk);
        st.h[2 * kk] = make_float2(v.x, v.y);
        st.h[2 * kk + 1] = make_float2(v.z, v.w);
      }
    }
  } else if (j > 0)
    state16_load(st, p.carry + (((size_t)b * p.n_chunks + j) * D + cl) * kN);
  else if (p.h0)
    state16_load(st, p.h0 + ((size_t)b * D + cl) * kN);
  else
    state16_zero(st);

  // the conv's earlier inputs
  float xm3 = input_at<IO>(p, b, (long)t_begin - 3, cl);
  float xm2 = input_at<IO>(p, b, (long)t_begin - 2, cl);
  float xm1 = input_at<IO>(p, b, (long)t_begin - 1, cl);
  // final_h and final_conv_state may alias h0 and conv_state0.  In the one
  // launch of the chunked mode their readers are chunk 0's main warp (here)
  // and boundary 1's carry walk; each counts itself done (a fence, then an
  // atomic increment) on the group's chunk-0 flag after its last read, and
  // the last chunk's warp checks the count before it writes (below).
  if (wait_carry && p.n_chunks > 1 && j == 0) {
    __syncwarp();
    if (lane == 0) {
      __threadfence();
      atomicAdd(p.counters + 1 + ((size_t)b * p.n_groups + g) * p.n_chunks, 1u);
    }
  }

  // the final conv state (the last three inputs), read by the last chunk at
  // its start (taking them from the conv window after the loop instead
  // measured 3 % slower on the whole launch)
  float f0 = 0.0f, f1 = 0.0f, f2 = 0.0f;
  if (j == p.n_chunks - 1 && p.final_conv_state != nullptr) {
    f0 = input_at<IO>(p, b, (long)p.seqlen - 3, cl);
    f1 = input_at<IO>(p, b, (long)p.seqlen - 2, cl);
    f2 = input_at<IO>(p, b, (long)p.seqlen - 1, cl);
  }
  // y may be null (a checkpointing pass for the backward needs only the states)
  const bool wy = active && p.y != nullptr;
  IO* yrow = reinterpret_cast<IO*>(p.y) + ((size_t)b * p.seqlen + t_begin) * D + cl;
  bool ok = true;
  int k = 0;
  for (; k < n_tiles; ++k) {
    const int s = k % kStages;
    const MainStage<IO>& S = sm.stage[s];
    const int t_valid = min(kT, t_end - (t_begin + k * kT));
    if (p.ckpt != nullptr && active)
      state16_store(st, p.ckpt + (((size_t)b * p.seq_tiles + (t_begin / kT + k)) * D + c) * kN);
    bool mine = mbar_wait_bounded(smem_u32(&sm.full[s]), (k / kStages) & 1, p.timeout_ns);
    ok = __all_sync(0xffffffffu, mine);
    if (!ok) break;
    IO* ytile = yrow + (size_t)k * kT * D;
    if (small_dt_tile<IO>(S.dt, t_valid, lane, active)) {
      if (t_valid == kT)
        main_tile<IO, true, true, kY>(S, kT, lane, wy, ch, st, xm3, xm2, xm1, ytile, D);
      else
        main_tile<IO, true, false, kY>(S, t_valid, lane, wy, ch, st, xm3, xm2, xm1, ytile, D);
    } else {
      main_tile<IO, false, false, kY>(S, t_valid, lane, wy, ch, st, xm3, xm2, xm1, ytile, D);
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
  if (j == p.n_chunks - 1 && (p.final_h != nullptr || p.final_conv_state != nullptr)) {
    if (wait_carry && p.n_chunks > 1) {
      // the readers of h0 and conv_state0 are done (by the time the carry
      // chain has let this chunk start they normally are: one load); the
      // stores below are issued after, and depend on, the observed count.
      // Nothing of this is kept live across the main loop: the same check at
      // the warp's start measured 4 % slower on the whole launch.
      const unsigned* readers = p.counters + 1 + ((size_t)b * p.n_groups + g) * p.n_chunks;
      if (lane == 0) {
        const uint64_t t_start = globaltimer_ns();
        while (ld_relaxed_gpu(readers) < 2u) {
          if (globaltimer_ns() - t_start > p.timeout_ns) {
            report_error(4u);  // MAMBA_ERR_TIMEOUT
            break;
          }
        }
      }
      __syncwarp();
    }
    if (active) {
      if (p.final_h != nullptr) state16_store(st, p.final_h + ((size_t)b * D + c) * kN);
      if (p.final_conv_state != nullptr) {
        IO* fcs = reinterpret_cast<IO*>(p.final_conv_state) + (size_t)b * 3 * D + c;
        fcs[0] = from_f32<IO>(f0);
        fcs[D] = from_f32<IO>(f1);
        fcs[2 * (size_t)D] = from_f32<IO>(f2);
      }
    }
  }
}

// grid (n_groups, batch, n_chunks), 32 threads: the carries were computed by
// an earlier launch.
template <typename IO, bool kY>
__global__ void __launch_bounds__(kLanes)
    scan_fwd_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_z,
                    const __grid_constant__ CUtensorMap tm_dt, const __grid_constant__ CUtensorMap tm_bc,
                    const __grid_constant__ ScanParams p) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  main_warp<IO, kY>(tm_x, tm_z, tm_dt, tm_bc, p, *reinterpret_cast<MainSmem<IO>*>(smem_raw + smem_pad128(smem_raw)),
                    blockIdx.x, blockIdx.y, blockIdx.z, false);
}

// ---------------------------------------------------------------- chunk carries
// One warp per (chunk boundary j = 1..n_chunks-1, channel group, batch row),
// assigned in launch order from a ticket counter, so that the warp of
// boundary j-1 of the same group always started earlier.  It computes
// carry_j, the state entering chunk j, from the tokens of chunk j-1, walking
// that chunk's pieces backwards, each scanned forward from zero: with hloc_q
// and S_q the end state and dt sum of piece q, and W_q = 2^(A2 * (sum of S
// over the pieces after q)) the decay from the end of piece q to the boundary,
//   carry_j = sum_q W_q hloc_q + W_start carry_{j-1}      (per state)
// where W_start is the decay over the whole chunk.  The walk stops early once
// every state of every lane has decayed below 2^-32 from the start of the
// current piece to the boundary: the terms left out (earlier pieces and
// carry_{j-1}) then enter with weights below 2^-32 and are dropped.
// Otherwise, after the chunk's first piece, the warp waits (bounded) for
// carry_{j-1}, published by boundary j-1's warp, and folds it in.  Fast
// decay, the common case, costs a few pieces per boundary; no decay at all
// costs one pass over the earlier chunks and a chain of waits, no more than a
// full two-pass scan.

template <typename IO>
struct CarrySmem {
  SummaryStage<IO> stage[kStages];
  uint64_t full[kStages];
  unsigned ticket;
};

// Tiles of chunk jc's pieces in walk order (last piece first, each forward):
// piece q covers chunk tiles [q*P, min((q+1)*P, C)).
struct PieceWalk {
  int first_tile;  // chunk's first tile
  int C, P, m;     // chunk tiles, piece tiles, pieces
  int len_last;    // tiles of the last piece
  __device__ __forceinline__ int piece_of(int i) const {
    return i < len_last ? m - 1 : m - 2 - (i - len_last) / P;
  }
  __device__ __forceinline__ int tile_of(int i) const {
    if (i < len_last) return first_tile + (m - 1) * P + i;
    const int r = i - len_last;
    return first_tile + (m - 2 - r / P) * P + r % P;
  }
  __device__ __forceinline__ int piece_len(int q) const { return q == m - 1 ? len_last : P; }
};

template <typename IO>
__device__ __forceinline__ void issue_carry_tile(CarrySmem<IO>& sm, int s, const CUtensorMap* tx,
                                                 const CUtensorMap* tdt, const CUtensorMap* tbc, int c0, int tile,
                                                 int b) {
  constexpr uint32_t kBytes = 2 * kT * kLanes * sizeof(IO) + kT * kBC * sizeof(float);
  const uint32_t bar = smem_u32(&sm.full[s]);
  const int tt = tile * kT;
  mbar_arrive_expect_tx(bar, kBytes);
  tma_load_3d(smem_u32(&sm.stage[s].x[0][0]), tx, c0, tt, b, bar);
  tma_load_3d(smem_u32(&sm.stage[s].dt[0][0]), tdt, c0, tt, b, bar);
  tma_load_3d(smem_u32(&sm.stage[s].bc[0][0]), tbc, 0, tt, b, bar);
}

// One warp of the carry pass (in the fused launch below, or in the
// backward's launch that runs it beside the adjoint carries).
template <typename IO>
__device__ __forceinline__ void carry_warp(const CUtensorMap& tm_x, const CUtensorMap& tm_dt, const CUtensorMap& tm_bc,
                                           const ScanParams& p, CarrySmem<IO>& sm, long ticket_in = -1) {
  const int lane = threadIdx.x;
  if (lane == 0) {
    sm.ticket = ticket_in >= 0 ? (unsigned)ticket_in : atomicAdd(p.counters, 1u);
    for (int s = 0; s < kStages; ++s) mbar_init(smem_u32(&sm.full[s]), 1);
    fence_mbar_init();
    prefetch_tensormap(&tm_x);
    prefetch_tensormap(&tm_dt);
    prefetch_tensormap(&tm_bc);
  }
  __syncwarp();
  const int per = p.n_chunks - 1;
  const unsigned ticket = sm.ticket;
  const int j = (int)(ticket % per) + 1;  // boundary: carry into chunk j
  const int gb = (int)(ticket / per);
  const int g = gb % p.n_groups;
  const int b = gb / p.n_groups;
  const int D = p.d_inner;
  const int c0 = g * kLanes;
  const int c = c0 + lane;
  const bool active = c < D;
  const int cl = active ? c : D - 1;
  unsigned* ready = p.counters + 1 + (size_t)b * p.n_groups * p.n_chunks + (size_t)g * p.n_chunks;

  PieceWalk wk;
  wk.first_tile = (j - 1) * p.chunk_tiles;
  wk.C = p.chunk_tiles;
  wk.P = p.piece_tiles;
  wk.m = p.pieces;
  wk.len_last = p.chunk_tiles - (p.pieces - 1) * p.piece_tiles;
  const int n_tiles = wk.C;

  if (lane == 0)
    for (int k = 0; k < kStages && k < n_tiles; ++k)
      issue_carry_tile<IO>(sm, k, &tm_x, &tm_dt, &tm_bc, c0, wk.tile_of(k), b);

  Channel ch;
  load_channel(ch, p.A_log, p.conv_w, p.conv_b, p.Dskip, cl);
  float a2max = ch.a2[0].x;  // the slowest decay of this channel
#pragma unroll
  for (int k = 0; k < 8; ++k) a2max = fmaxf(a2max, fmaxf(ch.a2[k].x, ch.a2[k].y));
  State16 acc, wgt, st;
  state16_zero(acc);
#pragma unroll
  for (int k = 0; k < 8; ++k) wgt.h[k] = make_float2(1.0f, 1.0f);
  float s_after = 0.0f;  // dt summed from the current piece's end to the boundary
  const bool exact = (p.flags & kFlagExactCarry) != 0;  // walk the whole chunk, drop nothing
  int n_pairs = 8;  // leading state pairs the current piece advances

  bool ok = true, done = false;
  int k = 0;
  int q = wk.piece_of(0);
  int left = wk.piece_len(q);  // tiles left in the current piece
  float sdt = 0.0f, xm3 = 0.0f, xm2 = 0.0f, xm1 = 0.0f;
  state16_zero(st);
  {
    const long t0 = (long)wk.tile_of(0) * kT;
    xm3 = input_at<IO>(p, b, t0 - 3, cl);
    xm2 = input_at<IO>(p, b, t0 - 2, cl);
    xm1 = input_at<IO>(p, b, t0 - 1, cl);
  }
  for (; k < n_tiles; ++k) {
    const int s = k % kStages;
    const SummaryStage<IO>& S = sm.stage[s];
    bool mine = mbar_wait_bounded(smem_u32(&sm.full[s]), (k / kStages) & 1, p.timeout_ns);
    ok = __all_sync(0xffffffffu, mine);
    if (!ok) break;
    if (small_dt_tile<IO>(S.dt, kT, lane, active))
      summary_tile_n<IO, true>(n_pairs, S, lane, ch, st, sdt, xm3, xm2, xm1);
    else
      summary_tile_n<IO, false>(n_pairs, S, lane, ch, st, sdt, xm3, xm2, xm1);
    __syncwarp();
    if (lane == 0 && k + kStages < n_tiles)
      issue_carry_tile<IO>(sm, s, &tm_x, &tm_dt, &tm_bc, c0, wk.tile_of(k + kStages), b);
    if (--left == 0) {  // piece q done: acc += wgt hloc_q, then wgt decays over piece q
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) acc.h[kk] = __ffma2_rn(wgt.h[kk], st.h[kk], acc.h[kk]);
      State16 zero;
      state16_zero(zero);
      state16_fold(wgt, ch.a2, sdt, zero);
      s_after = __fadd_rn(s_after, sdt);
      if (!exact && __all_sync(0xffffffffu, !active || __fmul_rn(a2max, s_after) < kCarryDropLog2)) {
        done = true;
        ++k;
        break;
      }
      if (k + 1 < n_tiles) {  // next (earlier) piece: restart from zero
        q = wk.piece_of(k + 1);
        left = wk.piece_len(q);
        state16_zero(st);
        sdt = 0.0f;
        // state pairs whose weight to the boundary fell below the drop bound
        // contribute nothing from here on: the piece advances the others only
        if (!exact) n_pairs = live_pairs(wgt, active);
        const long t0 = (long)wk.tile_of(k + 1) * kT;
        xm3 = input_at<IO>(p, b, t0 - 3, cl);
        xm2 = input_at<IO>(p, b, t0 - 2, cl);
        xm1 = input_at<IO>(p, b, t0 - 1, cl);
      }
    }
  }
  if (lane == 0) {  // copies still in flight land before shared memory goes away
    for (int kk = k; kk < n_tiles && kk < k + kStages; ++kk)
      (void)mbar_wait_bounded(smem_u32(&sm.full[kk % kStages]), (kk / kStages) & 1, p.timeout_ns);
  }
  if (!ok && lane == 0) report_error(4u);  // MAMBA_ERR_TIMEOUT

  if (ok && !done) {  // the whole chunk matters: fold in the carry entering it
    State16 prev;
    bool have = true;
    if (j - 1 == 0) {
      if (p.h0)
        state16_load(prev, p.h0 + ((size_t)b * D + cl) * kN);
      else
        state16_zero(prev);
    } else {
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
        state16_zero(prev);
      } else {
        const float4* src = reinterpret_cast<const float4*>(
            p.carry + (((size_t)b * p.n_chunks + (j - 1)) * D + cl) * kN);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const float4 v = __ldcg(src + kk);
          prev.h[2 * kk] = make_float2(v.x, v.y);
          prev.h[2 * kk + 1] = make_float2(v.z, v.w);
        }
      }
    }
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) acc.h[kk] = __ffma2_rn(wgt.h[kk], prev.h[kk], acc.h[kk]);
  }

  // publish carry_j (also after a failure, so that no later boundary waits in vain)
  if (active) state16_store(acc, p.carry + (((size_t)b * p.n_chunks + j) * D + c) * kN);
  __threadfence();
  __syncwarp();
  if (lane == 0) {
    atomicExch(ready + j, 1u);
    // boundary 1's walk is done reading h0 and conv_state0 (the final states
    // may alias them): count it on the group's chunk-0 flag
    if (j == 1) atomicAdd(ready, 1u);
  }
}

// ---------------------------------------------------------------- carries and main pass in one launch
// The chunked mode's two passes as one launch of (n_chunks - 1) * n_groups *
// batch carry warps and n_chunks * n_groups * batch main warps.  Each CTA
// takes a ticket at its start: the carry tasks come first (in the carry
// kernel's order), then the main tasks chunk by chunk.  The main warp of
// chunk j > 0 waits (bounded) for carry_j's flag; its carry warp took an
// earlier ticket, so it is resident or done, and chunk 0's main warps and the
// carries run side by side instead of one pass after the other.
template <typename IO>
constexpr size_t fused_smem_bytes() {
  return sizeof(MainSmem<IO>) > sizeof(CarrySmem<IO>) ? sizeof(MainSmem<IO>) : sizeof(CarrySmem<IO>);
}

template <typename IO, bool kY>
__global__ void __launch_bounds__(kLanes)
    scan_fused_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_z,
                      const __grid_constant__ CUtensorMap tm_dt, const __grid_constant__ CUtensorMap tm_bc,
                      const __grid_constant__ ScanParams p) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  unsigned char* base = smem_raw + smem_pad128(smem_raw);
  // a programmatic dependent of the B/C widening (which zeroed the counters):
  // nothing is read before it has completed; the next call's widening may
  // launch meanwhile (it waits for this launch in turn)
  griddep_wait();
  griddep_launch_dependents();
  unsigned ticket = 0;
  if (threadIdx.x == 0) ticket = atomicAdd(p.counters, 1u);
  ticket = __shfl_sync(0xffffffffu, ticket, 0);
  const unsigned per = (unsigned)p.n_groups * (unsigned)p.batch;
  const unsigned n_carry = (unsigned)(p.n_chunks - 1) * per;
  if (ticket < n_carry) {
    carry_warp<IO>(tm_x, tm_dt, tm_bc, p, *reinterpret_cast<CarrySmem<IO>*>(base), (long)ticket);
  } else {
    const unsigned t = ticket - n_carry;
    const int j = (int)(t / per), gb = (int)(t % per);
    main_warp<IO, kY>(tm_x, tm_z, tm_dt, tm_bc, p, *reinterpret_cast<MainSmem<IO>*>(base), gb % p.n_groups,
                      gb / p.n_groups, j, true);
  }
}

}  // namespace mamba
