// scan_bwd.cuh -- backward pass of the selective scan.
//
// Gradients of a loss l with respect to every input of the prefill, given
// dy = dl/dy (and optionally dl/dfinal_h, dl/dfinal_conv_state).  The
// chain rule through one token of the recurrence (the layer of
// "【大模型】- Jamba 混合 SSM-Transformer", section "实现 > Mamba 层"), with
// lam = dl/dh_t, dA_n = 2^(dt A2_n), w_n = lam_n dA_n h_{t-1,n}:
//   dyss = dy silu(z)                      dz   = dy yss silu'(z)
//   lam += C dyss                          dC_t = sum over channels of dyss h_t
//   dB_t = sum over channels of dt u lam   ddt  = ln2 sum_n A2_n w_n + u sum_n lam_n B_n
//   dA_log_n += A_n dt w_n                 du   = D dyss + dt sum_n lam_n B_n
//   lam <- dA lam (the adjoint entering token t-1)
//   ddt_raw = ddt sigmoid(dt_raw)          dpre = du silu'(pre), then the conv's
//                                          transpose gives dx, dconv_w, dconv_b
//
// Work decomposition (the forward's: one warp = 32 channels of one batch
// row, lane = channel, all 16 states in registers, a chunk of the sequence
// per CTA) walking its chunk's tiles in reverse.  The states h_{t-1} the
// reverse step needs come from checkpoints: a checkpointing forward pass
// stores the state entering every 16-token tile.  A tile is then handled in
// 4-token sub-tiles, last first: one forward pass over the tile's first 12
// tokens leaves the states entering sub-tiles 1..3 in shared memory; each
// sub-tile is recomputed forward from its entry state keeping all five of its
// states in registers (h before each token and after the last), and walked
// backwards.  Every forward quantity is recomputed with the forward pass's
// own operations, so the states match it bit for bit.
//
// dB and dC sum over channels: per token each lane's 32 values (dB | dC of
// its channel) are summed over the warp through a padded shared-memory
// transpose in a fixed order, and the warp's sums go to a per-group partial
// buffer that a final kernel sums over the groups in a fixed order (no
// atomics: the gradients are deterministic).  The per-channel parameter
// gradients are summed over a chunk in registers and over chunks and batch
// rows by a last kernel, also in a fixed order.
//
// Chunked mode.  The reverse sweep of chunk j needs the adjoint flowing into
// its last token from the tokens after it.  That adjoint obeys the same kind
// of linear recurrence as the state, run backwards:
//   R_{t-1} = dA_t (C_t dyss_t + R_t),        R_{L-1} = dl/dfinal_h
// (dyss does not depend on the state), so the adjoint-carry warps compute the
// carries like the forward's carry walks with time reversed: one warp
// per boundary walks the next chunk forwards in pieces, each piece scanned
// backwards from zero, and stops once the decay from the boundary makes the
// rest negligible (below 2^-32), or chains onto the next boundary's carry.
// The conv couples a chunk's last three tokens to the next chunk's first
// three: those dx values are finished by a small kernel afterwards.
#pragma once
#include "scan_fwd.cuh"

namespace mamba {

constexpr int kSub = 4;             // tokens per register sub-tile
constexpr int kSubs = kT / kSub;    // sub-tiles per tile
constexpr int kParamStride = 24;    // floats per channel of the parameter partials

template <typename IO>
struct BwdStage {
  IO x[kT][kLanes];
  IO z[kT][kLanes];
  IO dt[kT][kLanes];
  IO dy[kT][kLanes];
  float bc[kT][kBC];
};

template <typename IO>
struct BwdSmem {
  BwdStage<IO> stage[kStages];
  float4 sub[kSubs - 1][4][kLanes];  // states entering sub-tiles 1..3 of the current tile
  float4 red[2][kLanes][8];          // dB | dC of two tokens, one swizzled row per lane each
  uint64_t full[kStages];
};

template <typename IO>
struct ACarryStage {
  IO z[kT][kLanes];
  IO dt[kT][kLanes];
  IO dy[kT][kLanes];
  float bc[kT][kBC];
};

template <typename IO>
struct ACarrySmem {
  ACarryStage<IO> stage[kStages];
  uint64_t full[kStages];
  unsigned ticket;
};

// One tile of an adjoint-carry piece, walked backwards from its last row
// (rows tokens): R <- dA (C dyss + R) on the first kPairs state pairs (the
// later ones, whose decay to the boundary is already below the drop bound,
// stay as they are: zero within the piece), and the dt sum.
template <typename IO, int kPairs>
__device__ __forceinline__ void adjoint_tile(const ACarryStage<IO>& S, int rows, int lane, bool active,
                                             const Channel& ch, State16& rr, float& sdt) {
#pragma unroll(kScanUnroll)
  for (int r = rows - 1; r >= 0; --r) {
    const float dt = softplus(to_f32(S.dt[r][lane]));
    const float dyv = active ? to_f32(S.dy[r][lane]) : 0.0f;
    const float dyss = __fmul_rn(dyv, silu(to_f32(S.z[r][lane])));
    const float2 d2 = make_float2(dt, dt), y2 = make_float2(dyss, dyss);
#pragma unroll
    for (int kk = 0; kk < kPairs; ++kk) {
      const float4 q = *reinterpret_cast<const float4*>(&S.bc[r][4 * kk]);
      const float2 xa = __fmul2_rn(d2, ch.a2[kk]);
      const float2 dA = make_float2(ex2_approx(xa.x), ex2_approx(xa.y));
      rr.h[kk] = __fmul2_rn(__ffma2_rn(make_float2(q.z, q.w), y2, rr.h[kk]), dA);
    }
    sdt = __fadd_rn(sdt, dt);
  }
}

// softplus(v) (the forward's bits) and its derivative sigmoid(v), which is 1
// above the threshold where softplus(v) = v.
__device__ __forceinline__ void softplus_grad(float v, float& sp, float& sig) {
  const float e = softplus_e(v);
  sp = e < kSoftplusSmallE ? softplus_small(e) : softplus_large(v, e);
  sig = v > 20.0f ? 1.0f : __fmul_rn(e, rcp_approx(__fadd_rn(1.0f, e)));
}

// silu(v) (the forward's bits) and silu'(v) = s (1 + v (1 - s)), s = sigmoid(v).
__device__ __forceinline__ void silu_grad(float v, float& sv, float& dsv) {
  const float e = ex2_approx(__fmul_rn(v, -kLog2e));
  const float s = rcp_approx(__fadd_rn(1.0f, e));
  sv = __fmul_rn(v, s);
  dsv = __fmul_rn(s, __fmaf_rn(v, __fsub_rn(1.0f, s), 1.0f));
}

// Raw conv input of channel c at position tau of batch row b (tau < 0:
// conv_state0, or zero).
template <typename IO>
__device__ __forceinline__ float conv_input_at(const void* x, const void* cs0, int seqlen, int D, int b, long tau,
                                               int c) {
  if (tau >= 0) return to_f32(reinterpret_cast<const IO*>(x)[((size_t)b * seqlen + tau) * D + c]);
  if (cs0 == nullptr) return 0.0f;
  return to_f32(reinterpret_cast<const IO*>(cs0)[((size_t)b * 3 + (3 + tau)) * D + c]);
}

__device__ __forceinline__ void state16_store_f4(float4 (&dst)[4][kLanes], int lane, const State16& s) {
#pragma unroll
  for (int q = 0; q < 4; ++q)
    dst[q][lane] = make_float4(s.h[2 * q].x, s.h[2 * q].y, s.h[2 * q + 1].x, s.h[2 * q + 1].y);
}

__device__ __forceinline__ void state16_load_f4(State16& s, const float4 (&src)[4][kLanes], int lane) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float4 v = src[q][lane];
    s.h[2 * q] = make_float2(v.x, v.y);
    s.h[2 * q + 1] = make_float2(v.z, v.w);
  }
}

// dB | dC of one token summed over the warp's 32 channels, in two steps:
// every lane writes its channel's 32 values as one row of a buffer
// (write_bc_row), then, for up to two tokens at once (reduce_bc_pair), lane
// (rg, cg) adds rows 8 rg .. 8 rg + 7 of columns 4 cg .. 4 cg + 3 in row
// order and the four row groups are combined by two exchanges (xor 8, then
// xor 16); lanes 0-7 store the first token's 32 sums (128 bytes), lanes 8-15
// the second's.  Row r keeps quad q at position q ^ (r % 8), so that both the
// row writes and the column reads of 8 consecutive lanes touch 8 different
// 16-byte bank groups.  Batching two tokens halves the warp barriers, which
// also fence the compiler's scheduling of shared-memory accesses.
__device__ __forceinline__ void write_bc_row(float4 (&red)[kLanes][8], const float2 (&dB)[8],
                                             const float2 (&dC)[8], int lane) {
  const int sw = lane & 7;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    red[lane][q ^ sw] = make_float4(dB[2 * q].x, dB[2 * q].y, dB[2 * q + 1].x, dB[2 * q + 1].y);
    red[lane][(4 + q) ^ sw] = make_float4(dC[2 * q].x, dC[2 * q].y, dC[2 * q + 1].x, dC[2 * q + 1].y);
  }
}

// Column sums of 8 rows as two interleaved chains (even and odd rows), added
// at the end: half the dependent latency of one chain, still a fixed order.
__device__ __forceinline__ void column_sums(const float4 (&red)[kLanes][8], int lane, float2& s0, float2& s1) {
  const int cg = lane & 7, rg = lane >> 3;
  float2 e0, e1, o0, o1;
#pragma unroll
  for (int m = 0; m < 8; ++m) {
    const float4 v = red[rg * 8 + m][cg ^ m];
    const float2 lo = make_float2(v.x, v.y), hi = make_float2(v.z, v.w);
    if (m == 0) {
      e0 = lo;
      e1 = hi;
    } else if (m == 1) {
      o0 = lo;
      o1 = hi;
    } else if (m & 1) {
      o0 = __fadd2_rn(o0, lo);
      o1 = __fadd2_rn(o1, hi);
    } else {
      e0 = __fadd2_rn(e0, lo);
      e1 = __fadd2_rn(e1, hi);
    }
  }
  s0 = __fadd2_rn(e0, o0);
  s1 = __fadd2_rn(e1, o1);
}

__device__ __forceinline__ void rowgroup_sums(float2& s0, float2& s1) {
#pragma unroll
  for (int m = 8; m <= 16; m <<= 1) {
    const float2 o0 = make_float2(__shfl_xor_sync(0xffffffffu, s0.x, m), __shfl_xor_sync(0xffffffffu, s0.y, m));
    const float2 o1 = make_float2(__shfl_xor_sync(0xffffffffu, s1.x, m), __shfl_xor_sync(0xffffffffu, s1.y, m));
    s0 = __fadd2_rn(s0, o0);
    s1 = __fadd2_rn(s1, o1);
  }
}

// Rows of token A in red[a], of token B (if two) in red[a ^ 1]; sums to dstA, dstB.
__device__ __forceinline__ void reduce_bc_pair(float4 (&red)[2][kLanes][8], int a, bool two, int lane,
                                               float* dstA, float* dstB) {
  __syncwarp();  // every row written
  float2 a0, a1, b0 = make_float2(0.0f, 0.0f), b1 = make_float2(0.0f, 0.0f);
  column_sums(red[a], lane, a0, a1);
  if (two) column_sums(red[a ^ 1], lane, b0, b1);
  __syncwarp();  // every row read: the buffers are free again
  rowgroup_sums(a0, a1);
  if (two) rowgroup_sums(b0, b1);
  if (lane < 8) *reinterpret_cast<float4*>(dstA + 4 * lane) = make_float4(a0.x, a0.y, a1.x, a1.y);
  if (two && lane >= 8 && lane < 16)
    *reinterpret_cast<float4*>(dstB + 4 * (lane - 8)) = make_float4(b0.x, b0.y, b1.x, b1.y);
}

// The forward quantities of one token kept for its reverse step.
struct TokFwd {
  float u, dsil, dt, dsig;
};

// Everything a lane carries through its chunk's reverse sweep.
struct BwdLane {
  State16 lam;   // dl/dh entering the token being processed from its right
  State16 Sw;    // sum over tokens of dt * w (dA_log = A * Sw)
  float dD, dbias;
  float4 dw;     // conv taps
  float dp1, dp2, dp3;  // d pre of the three tokens after the current one
};

// One sub-tile: `rq` tokens (1..4) starting at tile row r0, entering state
// hh[0].  xw[0..2] are the three inputs before row r0.
template <typename IO>
__device__ __forceinline__ void bwd_subtile(const BwdParams& p, const BwdStage<IO>& S,
                                            float4 (&red)[2][kLanes][8],
                                            int lane, bool active, int c, int b, int g, int t0, int r0, int rq,
                                            int edge_from, const Channel& ch, State16 (&hh)[kSub + 1],
                                            float (&xw)[kSub + 3], BwdLane& ln, size_t BL) {
  const int D = p.d_inner;
  TokFwd f[kSub];
#pragma unroll
  for (int i = 0; i < kSub; ++i) xw[3 + i] = to_f32(S.x[r0 + i][lane]);
  // forward: hh[i + 1] = state after token i
#pragma unroll
  for (int i = 0; i < kSub; ++i) {
    if (i < rq) {
      const int r = r0 + i;
      const float pre = conv4(ch.w, ch.bias, xw[i], xw[i + 1], xw[i + 2], xw[i + 3]);
      silu_grad(pre, f[i].u, f[i].dsil);
      softplus_grad(to_f32(S.dt[r][lane]), f[i].dt, f[i].dsig);
      float4 Q[8];
      load_quads(&S.bc[r][0], Q);
      Drive16 d;
      drive16_q(d, ch.a2, f[i].dt, __fmul_rn(f[i].dt, f[i].u), Q);
      hh[i + 1] = hh[i];
      state16_apply(hh[i + 1], d);
    }
  }
  // reverse; row0: element (b, t0 + r0, c) of the (B, L, D) outputs; part0:
  // row (g, b, t0 + r0) of the dB | dC sums
  const size_t row0 = ((size_t)b * p.seqlen + t0 + r0) * D + c;
  float* part0 = p.part_bc + ((size_t)g * BL + (size_t)b * p.seqlen + t0 + r0) * 32;
  const int cl = active ? c : D - 1;
#pragma unroll
  for (int i = kSub - 1; i >= 0; --i) {
    if (i < rq) {
      const int r = r0 + i;
      const int t = t0 + r;
      const float u = f[i].u, dt = f[i].dt;
      float4 Q[8];
      load_quads(&S.bc[r][0], Q);
      const float zv = to_f32(S.z[r][lane]);
      const float dyv = active ? to_f32(S.dy[r][lane]) : 0.0f;
      float gz, dsz;
      silu_grad(zv, gz, dsz);
      const float dyss = __fmul_rn(dyv, gz);
      const float yss = __fmaf_rn(ch.Dc, u, state16_readout_q(hh[i + 1], Q));
      const float dzv = __fmul_rn(__fmul_rn(dyv, yss), dsz);
      ln.dD = __fmaf_rn(dyss, u, ln.dD);
      const float dtu = __fmul_rn(dt, u);
      const float2 dyss2 = make_float2(dyss, dyss), dtu2 = make_float2(dtu, dtu), dt2 = make_float2(dt, dt);
      // sum_n lam_n B_n and sum_n A2_n w_n as two chains each (pairs 0-3, 4-7)
      float2 lamB[2] = {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f)};
      float2 ddtA[2] = {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f)};
      float2 dBv[8], dCv[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float2 Bk = make_float2(Q[k].x, Q[k].y), Ck = make_float2(Q[k].z, Q[k].w);
        float2 lam = __ffma2_rn(Ck, dyss2, ln.lam.h[k]);
        dCv[k] = __fmul2_rn(hh[i + 1].h[k], dyss2);
        dBv[k] = __fmul2_rn(lam, dtu2);
        lamB[k >> 2] = __ffma2_rn(lam, Bk, lamB[k >> 2]);
        const float2 xa = __fmul2_rn(dt2, ch.a2[k]);
        const float2 dA = make_float2(ex2_approx(xa.x), ex2_approx(xa.y));
        lam = __fmul2_rn(lam, dA);
        const float2 w = __fmul2_rn(lam, hh[i].h[k]);
        ddtA[k >> 2] = __ffma2_rn(ch.a2[k], w, ddtA[k >> 2]);
        ln.Sw.h[k] = __ffma2_rn(dt2, w, ln.Sw.h[k]);
        ln.lam.h[k] = lam;
      }
      const float2 lB = __fadd2_rn(lamB[0], lamB[1]), dA2 = __fadd2_rn(ddtA[0], ddtA[1]);
      const float sB = __fadd_rn(lB.x, lB.y);
      const float sA = __fadd_rn(dA2.x, dA2.y);
      const float ddt = __fmaf_rn(sA, kLn2, __fmul_rn(sB, u));
      const float du = __fmaf_rn(dyss, ch.Dc, __fmul_rn(sB, dt));
      const float dpre = __fmul_rn(du, f[i].dsil);
      ln.dbias = __fadd_rn(ln.dbias, dpre);
      ln.dw.x = __fmaf_rn(dpre, xw[i], ln.dw.x);
      ln.dw.y = __fmaf_rn(dpre, xw[i + 1], ln.dw.y);
      ln.dw.z = __fmaf_rn(dpre, xw[i + 2], ln.dw.z);
      ln.dw.w = __fmaf_rn(dpre, xw[i + 3], ln.dw.w);
      float dxv = __fmul_rn(ch.w.w, dpre);
      dxv = __fmaf_rn(ch.w.z, ln.dp1, dxv);
      dxv = __fmaf_rn(ch.w.y, ln.dp2, dxv);
      dxv = __fmaf_rn(ch.w.x, ln.dp3, dxv);
      ln.dp3 = ln.dp2;
      ln.dp2 = ln.dp1;
      ln.dp1 = dpre;
      if (p.dfinal_conv_state != nullptr && t >= p.seqlen - 3)  // the same for every lane
        dxv = __fadd_rn(dxv, to_f32(reinterpret_cast<const IO*>(p.dfinal_conv_state)
                                        [((size_t)b * 3 + (t - (p.seqlen - 3))) * D + cl]));
      const size_t o = row0 + (size_t)i * D;
      st_global_if(active, reinterpret_cast<IO*>(p.dz) + o, from_f32<IO>(dzv));
      st_global_if(active, reinterpret_cast<IO*>(p.ddt_raw) + o, from_f32<IO>(__fmul_rn(ddt, f[i].dsig)));
      if (t >= edge_from)  // the same for every lane: a chunk's last three tokens
        st_global_if(active, p.edge_dx + (((size_t)b * p.n_chunks + blockIdx.z) * 3 + (t - edge_from)) * D + c,
                     dxv);
      else
        st_global_if(active, reinterpret_cast<IO*>(p.dx) + o, from_f32<IO>(dxv));
      // tokens 3, 2 and 1, 0 of the sub-tile share one reduction
      write_bc_row(red[i & 1], dBv, dCv, lane);
      if ((i & 1) == 0) {
        float* dst = part0 + (size_t)i * 32;
        reduce_bc_pair(red, 0, i + 1 < rq, lane, dst, dst + 32);
      }
    }
  }
}

// The forward pass over a tile's rows [0, n_pre) from state st (n_pre = 4 *
// (sub-tiles - 1)), storing the state entering each later sub-tile.
template <typename IO, bool kFull>
__device__ __forceinline__ void bwd_tile_prefix(const BwdStage<IO>& S, float4 (&sub)[kSubs - 1][4][kLanes],
                                                int lane, int n_pre, const Channel& ch, State16& st, float xm3,
                                                float xm2, float xm1) {
  if (kFull) n_pre = kT - kSub;
#pragma unroll(kFull ? kT - kSub : kSub)
  for (int r = 0; r < n_pre; ++r) {
    if (r > 0 && (r % kSub) == 0) state16_store_f4(sub[r / kSub - 1], lane, st);
    const float xv = to_f32(S.x[r][lane]);
    const float u = silu(conv4(ch.w, ch.bias, xm3, xm2, xm1, xv));
    xm3 = xm2;
    xm2 = xm1;
    xm1 = xv;
    const float dt = softplus(to_f32(S.dt[r][lane]));
    float4 Q[8];
    load_quads(&S.bc[r][0], Q);
    Drive16 d;
    drive16_q(d, ch.a2, dt, __fmul_rn(dt, u), Q);
    state16_apply(st, d);
  }
  if (n_pre > 0) state16_store_f4(sub[n_pre / kSub - 1], lane, st);
}

template <typename IO>
__device__ __forceinline__ void issue_bwd_tile(BwdSmem<IO>& sm, int s, const CUtensorMap* tx, const CUtensorMap* tz,
                                               const CUtensorMap* tdt, const CUtensorMap* tdy,
                                               const CUtensorMap* tbc, int c0, int tile, int b) {
  constexpr uint32_t kBytes = 4 * kT * kLanes * sizeof(IO) + kT * kBC * sizeof(float);
  const uint32_t bar = smem_u32(&sm.full[s]);
  const int tt = tile * kT;
  mbar_arrive_expect_tx(bar, kBytes);
  tma_load_3d(smem_u32(&sm.stage[s].x[0][0]), tx, c0, tt, b, bar);
  tma_load_3d(smem_u32(&sm.stage[s].z[0][0]), tz, c0, tt, b, bar);
  tma_load_3d(smem_u32(&sm.stage[s].dt[0][0]), tdt, c0, tt, b, bar);
  tma_load_3d(smem_u32(&sm.stage[s].dy[0][0]), tdy, c0, tt, b, bar);
  tma_load_3d(smem_u32(&sm.stage[s].bc[0][0]), tbc, 0, tt, b, bar);
}

// ---------------------------------------------------------------- reverse sweep
// grid (n_groups, batch, n_chunks), 32 threads.
template <typename IO>
__global__ void __launch_bounds__(kLanes)
    scan_bwd_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_z,
                    const __grid_constant__ CUtensorMap tm_dt, const __grid_constant__ CUtensorMap tm_dy,
                    const __grid_constant__ CUtensorMap tm_bc, const __grid_constant__ BwdParams p) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  BwdSmem<IO>& sm = *reinterpret_cast<BwdSmem<IO>*>(smem_raw + smem_pad128(smem_raw));

  const int lane = threadIdx.x;
  const int g = blockIdx.x;
  const int c0 = g * kLanes;
  const int b = blockIdx.y;
  const int j = blockIdx.z;
  const int D = p.d_inner;
  const int c = c0 + lane;
  const bool active = c < D;
  const int cl = active ? c : D - 1;
  const int t_begin = j * p.chunk_tiles * kT;
  const int t_end = min(t_begin + p.chunk_tiles * kT, p.seqlen);
  const int n_tiles = (t_end - t_begin + kT - 1) / kT;
  const int tile0 = t_begin / kT;
  const bool last_chunk = j == p.n_chunks - 1;
  const int edge_from = last_chunk ? p.seqlen : t_end - 3;  // dx of later tokens is partial
  const size_t BL = (size_t)p.batch * p.seqlen;

  if (lane == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(smem_u32(&sm.full[s]), 1);
    fence_mbar_init();
    prefetch_tensormap(&tm_x);
    prefetch_tensormap(&tm_z);
    prefetch_tensormap(&tm_dt);
    prefetch_tensormap(&tm_dy);
    prefetch_tensormap(&tm_bc);
  }
  __syncwarp();
  if (lane == 0)
    for (int i = 0; i < kStages && i < n_tiles; ++i)
      issue_bwd_tile<IO>(sm, i, &tm_x, &tm_z, &tm_dt, &tm_dy, &tm_bc, c0, tile0 + n_tiles - 1 - i, b);

  Channel ch;
  load_channel(ch, p.A_log, p.conv_w, p.conv_b, p.Dskip, cl);
  BwdLane ln;
  if (!active)
    state16_zero(ln.lam);
  else if (!last_chunk)
    state16_load(ln.lam, p.acarry + (((size_t)b * p.n_chunks + j) * D + c) * kN);
  else if (p.dfinal_h)
    state16_load(ln.lam, p.dfinal_h + ((size_t)b * D + c) * kN);
  else
    state16_zero(ln.lam);
  state16_zero(ln.Sw);
  ln.dD = 0.0f;
  ln.dbias = 0.0f;
  ln.dw = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  ln.dp1 = ln.dp2 = ln.dp3 = 0.0f;

  bool ok = true;
  int i = 0;
  for (; i < n_tiles; ++i) {
    const int k = n_tiles - 1 - i;
    const int s = i % kStages;
    const BwdStage<IO>& S = sm.stage[s];
    const int t0 = t_begin + k * kT;
    const int rows = min(kT, t_end - t0);
    const int nsub = (rows + kSub - 1) / kSub;
    // the state entering the tile and the three inputs before it
    const float* ck = p.ckpt + (((size_t)b * p.seq_tiles + tile0 + k) * D + cl) * kN;
    State16 st;
    state16_load(st, ck);
    const float xp3 = conv_input_at<IO>(p.x, p.conv_state0, p.seqlen, D, b, (long)t0 - 3, cl);
    const float xp2 = conv_input_at<IO>(p.x, p.conv_state0, p.seqlen, D, b, (long)t0 - 2, cl);
    const float xp1 = conv_input_at<IO>(p.x, p.conv_state0, p.seqlen, D, b, (long)t0 - 1, cl);
    bool mine = mbar_wait_bounded(smem_u32(&sm.full[s]), (i / kStages) & 1, p.timeout_ns);
    ok = __all_sync(0xffffffffu, mine);
    if (!ok) break;
    if (rows == kT)
      bwd_tile_prefix<IO, true>(S, sm.sub, lane, kT - kSub, ch, st, xp3, xp2, xp1);
    else
      bwd_tile_prefix<IO, false>(S, sm.sub, lane, (nsub - 1) * kSub, ch, st, xp3, xp2, xp1);
    State16 hh[kSub + 1];
    for (int q = nsub - 1; q >= 0; --q) {
      const int r0 = q * kSub;
      float xw[kSub + 3];
      if (q == 0) {
        state16_load(hh[0], ck);  // the tile's entry state again (an L1/L2 hit)
        xw[0] = xp3;
        xw[1] = xp2;
        xw[2] = xp1;
      } else {
        state16_load_f4(hh[0], sm.sub[q - 1], lane);
        xw[0] = to_f32(S.x[r0 - 3][lane]);
        xw[1] = to_f32(S.x[r0 - 2][lane]);
        xw[2] = to_f32(S.x[r0 - 1][lane]);
      }
      bwd_subtile<IO>(p, S, sm.red, lane, active, c, b, g, t0, r0, min(kSub, rows - r0), edge_from, ch, hh, xw,
                      ln, BL);
    }
    __syncwarp();  // every lane is done with stage s
    if (lane == 0 && i + kStages < n_tiles)
      issue_bwd_tile<IO>(sm, s, &tm_x, &tm_z, &tm_dt, &tm_dy, &tm_bc, c0, tile0 + n_tiles - 1 - (i + kStages), b);
  }
  if (!ok) {
    if (lane == 0) {
      report_error(4u);  // MAMBA_ERR_TIMEOUT
      for (int kk = i; kk < n_tiles && kk < i + kStages; ++kk)
        (void)mbar_wait_bounded(smem_u32(&sm.full[kk % kStages]), (kk / kStages) & 1, p.timeout_ns);
    }
    return;
  }
  if (!active) return;

  // d pre of the chunk's first three tokens, for the dx of the chunk before
  if (j > 0) {
    float* e = p.edge_dpre + ((size_t)b * p.n_chunks + j) * 3 * D + c;
    e[0] = ln.dp1;
    e[D] = ln.dp2;
    e[2 * (size_t)D] = ln.dp3;
  } else {
    if (p.dh0) state16_store(ln.lam, p.dh0 + ((size_t)b * D + c) * kN);
    if (p.dconv_state0) {
      // inputs at t = -3, -2, -1 feed the conv of tokens 0..2
      float d0 = __fmul_rn(ch.w.x, ln.dp1);
      float d1 = __fmaf_rn(ch.w.x, ln.dp2, __fmul_rn(ch.w.y, ln.dp1));
      float d2 = __fmaf_rn(ch.w.x, ln.dp3, __fmaf_rn(ch.w.y, ln.dp2, __fmul_rn(ch.w.z, ln.dp1)));
      if (p.dfinal_conv_state != nullptr && p.seqlen < 3) {  // the final conv state reaches back before t = 0
        const IO* f = reinterpret_cast<const IO*>(p.dfinal_conv_state) + (size_t)b * 3 * D + c;
        float dd[3] = {d0, d1, d2};
        for (int q = 0; q < 3; ++q) {
          const int tau = p.seqlen - 3 + q;  // input position of final_conv_state[q]
          if (tau < 0) dd[3 + tau] = __fadd_rn(dd[3 + tau], to_f32(f[(size_t)q * D]));
        }
        d0 = dd[0];
        d1 = dd[1];
        d2 = dd[2];
      }
      float* o = p.dconv_state0 + (size_t)b * 3 * D + c;
      o[0] = d0;
      o[D] = d1;
      o[2 * (size_t)D] = d2;
    }
  }
  // this chunk's share of the parameter gradients
  float* pp = p.part_param + (((size_t)b * p.n_chunks + j) * D + c) * kParamStride;
  float4* pq = reinterpret_cast<float4*>(pp);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float2 s0 = __fmul2_rn(ln.Sw.h[2 * q], ch.a2[2 * q]);
    const float2 s1 = __fmul2_rn(ln.Sw.h[2 * q + 1], ch.a2[2 * q + 1]);
    pq[q] = make_float4(__fmul_rn(s0.x, kLn2), __fmul_rn(s0.y, kLn2), __fmul_rn(s1.x, kLn2), __fmul_rn(s1.y, kLn2));
  }
  pq[4] = make_float4(ln.dD, ln.dw.x, ln.dw.y, ln.dw.z);
  pq[5] = make_float4(ln.dw.w, ln.dbias, 0.0f, 0.0f);
}

// ---------------------------------------------------------------- adjoint carries
// One warp per (boundary j = 0..n_chunks-2, channel group, batch row): the
// adjoint R_j entering chunk j's last token from chunk j+1 onwards.  With the
// pieces q of chunk j+1 walked from its start, Rloc_q the adjoint piece q
// alone sends out of its first token (scanned backwards from zero), S_q its dt
// sum and W_q = 2^(A2 * (sum of S over the pieces before q)):
//   R_j = sum_q W_q Rloc_q + W_all R_{j+1},    R_{n_chunks-1} = dl/dfinal_h.
// The walk stops once every state of every lane has decayed below 2^-32;
// otherwise the warp waits (bounded) for R_{j+1}, published by boundary
// j+1's warp, which the ticket order started earlier.
template <typename IO>
__device__ __forceinline__ void issue_acarry_tile(ACarrySmem<IO>& sm, int s, const CUtensorMap* tz,
                                                  const CUtensorMap* tdt, const CUtensorMap* tdy,
                                                  const CUtensorMap* tbc, int c0, int tile, int b) {
  constexpr uint32_t kBytes = 3 * kT * kLanes * sizeof(IO) + kT * kBC * sizeof(float);
  const uint32_t bar = smem_u32(&sm.full[s]);
  const int tt = tile * kT;
  mbar_arrive_expect_tx(bar, kBytes);
  tma_load_3d(smem_u32(&sm.stage[s].z[0][0]), tz, c0, tt, b, bar);
  tma_load_3d(smem_u32(&sm.stage[s].dt[0][0]), tdt, c0, tt, b, bar);
  tma_load_3d(smem_u32(&sm.stage[s].dy[0][0]), tdy, c0, tt, b, bar);
  tma_load_3d(smem_u32(&sm.stage[s].bc[0][0]), tbc, 0, tt, b, bar);
}

// Walk order over chunk jc's tiles: pieces first to last, each piece's tiles
// last to first.
struct RevPieceWalk {
  int first_tile, C, P;
  __device__ __forceinline__ int piece_len(int q) const { return min(P, C - q * P); }
  __device__ __forceinline__ int tile_of(int i) const {
    const int q = i / P, r = i % P;
    return first_tile + q * P + (piece_len(q) - 1 - r);
  }
};

template <typename IO>
__device__ __forceinline__ void acarry_warp(const CUtensorMap& tm_z, const CUtensorMap& tm_dt, const CUtensorMap& tm_dy,
                                            const CUtensorMap& tm_bc, const BwdParams& p, ACarrySmem<IO>& sm) {
  const int lane = threadIdx.x;
  if (lane == 0) {
    sm.ticket = atomicAdd(p.counters, 1u);
    for (int s = 0; s < kStages; ++s) mbar_init(smem_u32(&sm.full[s]), 1);
    fence_mbar_init();
    prefetch_tensormap(&tm_z);
    prefetch_tensormap(&tm_dt);
    prefetch_tensormap(&tm_dy);
    prefetch_tensormap(&tm_bc);
  }
  __syncwarp();
  const int per = p.n_chunks - 1;
  const unsigned ticket = sm.ticket;
  const int j = per - 1 - (int)(ticket % per);  // boundaries in decreasing order
  const int gb = (int)(ticket / per);
  const int g = gb % p.n_groups;
  const int b = gb / p.n_groups;
  const int D = p.d_inner;
  const int c0 = g * kLanes;
  const int c = c0 + lane;
  const bool active = c < D;
  const int cl = active ? c : D - 1;
  unsigned* ready = p.counters + 1 + (size_t)b * p.n_groups * p.n_chunks + (size_t)g * p.n_chunks;

  RevPieceWalk wk;
  wk.first_tile = (j + 1) * p.chunk_tiles;
  wk.C = min(p.chunk_tiles, p.seq_tiles - wk.first_tile);
  wk.P = p.piece_tiles;
  const int n_tiles = wk.C;

  if (lane == 0)
    for (int k = 0; k < kStages && k < n_tiles; ++k)
      issue_acarry_tile<IO>(sm, k, &tm_z, &tm_dt, &tm_dy, &tm_bc, c0, wk.tile_of(k), b);

  Channel ch;
  load_channel(ch, p.A_log, p.conv_w, p.conv_b, p.Dskip, cl);
  float a2max = ch.a2[0].x;
#pragma unroll
  for (int k = 0; k < 8; ++k) a2max = fmaxf(a2max, fmaxf(ch.a2[k].x, ch.a2[k].y));
  State16 acc, wgt, rr;
  state16_zero(acc);
  state16_zero(rr);
#pragma unroll
  for (int k = 0; k < 8; ++k) wgt.h[k] = make_float2(1.0f, 1.0f);
  float s_before = 0.0f, sdt = 0.0f;
  const bool exact = (p.flags & kFlagExactCarry) != 0;  // walk the whole chunk, drop nothing
  int n_pairs = 8;  // leading state pairs the current piece advances

  bool ok = true, done = false;
  int k = 0;
  int q = 0;
  int left = wk.piece_len(0);
  for (; k < n_tiles; ++k) {
    const int s = k % kStages;
    const ACarryStage<IO>& S = sm.stage[s];
    const int tile = wk.tile_of(k);
    const int rows = min(kT, p.seqlen - tile * kT);
    bool mine = mbar_wait_bounded(smem_u32(&sm.full[s]), (k / kStages) & 1, p.timeout_ns);
    ok = __all_sync(0xffffffffu, mine);
    if (!ok) break;
    if (n_pairs <= 1)
      adjoint_tile<IO, 1>(S, rows, lane, active, ch, rr, sdt);
    else if (n_pairs <= 2)
      adjoint_tile<IO, 2>(S, rows, lane, active, ch, rr, sdt);
    else if (n_pairs <= 4)
      adjoint_tile<IO, 4>(S, rows, lane, active, ch, rr, sdt);
    else
      adjoint_tile<IO, 8>(S, rows, lane, active, ch, rr, sdt);
    __syncwarp();
    if (lane == 0 && k + kStages < n_tiles)
      issue_acarry_tile<IO>(sm, s, &tm_z, &tm_dt, &tm_dy, &tm_bc, c0, wk.tile_of(k + kStages), b);
    if (--left == 0) {  // piece q done: acc += wgt Rloc_q, then wgt decays over piece q
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) acc.h[kk] = __ffma2_rn(wgt.h[kk], rr.h[kk], acc.h[kk]);
      State16 zero;
      state16_zero(zero);
      state16_fold(wgt, ch.a2, sdt, zero);
      s_before = __fadd_rn(s_before, sdt);
      if (!exact && __all_sync(0xffffffffu, !active || __fmul_rn(a2max, s_before) < kCarryDropLog2)) {
        done = true;
        ++k;
        break;
      }
      ++q;
      if (k + 1 < n_tiles) {
        left = wk.piece_len(q);
        state16_zero(rr);
        sdt = 0.0f;
        // state pairs whose weight to the boundary fell below the drop bound
        // contribute nothing from here on: the piece advances the others only
        if (!exact) n_pairs = live_pairs(wgt, active);
      }
    }
  }
  if (lane == 0) {  // copies still in flight land before shared memory goes away
    for (int kk = k; kk < n_tiles && kk < k + kStages; ++kk)
      (void)mbar_wait_bounded(smem_u32(&sm.full[kk % kStages]), (kk / kStages) & 1, p.timeout_ns);
  }
  if (!ok && lane == 0) report_error(4u);  // MAMBA_ERR_TIMEOUT

  if (ok && !done) {  // the whole next chunk matters: fold in the adjoint entering it
    State16 prev;
    if (j + 1 == p.n_chunks - 1) {
      if (p.dfinal_h)
        state16_load(prev, p.dfinal_h + ((size_t)b * D + cl) * kN);
      else
        state16_zero(prev);
    } else {
      bool have = true;
      if (lane == 0) {
        const uint64_t t_start = globaltimer_ns();
        while (atomicAdd(ready + (j + 1), 0u) == 0u) {
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
        const float4* src = reinterpret_cast<const float4*>(p.acarry + (((size_t)b * p.n_chunks + (j + 1)) * D + cl) * kN);
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

  // publish R_j (also after a failure, so that no earlier boundary waits in vain)
  if (active) state16_store(acc, p.acarry + (((size_t)b * p.n_chunks + j) * D + c) * kN);
  __threadfence();
  __syncwarp();
  if (lane == 0) atomicExch(ready + j, 1u);
}

// Both carry passes of the backward in one launch (they are independent, and
// each alone leaves most of the GPU idle): CTAs [0, n_fwd) run the forward's
// chunk carries, the rest the adjoint carries.  Each kind takes its tickets
// from its own counter and waits only on earlier tickets of its own kind, so
// every awaited warp has started.  grid (n_fwd + n_adj), 32 threads.
template <typename IO>
union CarriesSmem {
  CarrySmem<IO> fwd;
  ACarrySmem<IO> adj;
};

template <typename IO>
__global__ void __launch_bounds__(kLanes)
    scan_carries_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_z,
                        const __grid_constant__ CUtensorMap tm_dt, const __grid_constant__ CUtensorMap tm_dy,
                        const __grid_constant__ CUtensorMap tm_bc, const __grid_constant__ ScanParams fp,
                        const __grid_constant__ BwdParams bp, unsigned n_fwd) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  CarriesSmem<IO>& sm = *reinterpret_cast<CarriesSmem<IO>*>(smem_raw + smem_pad128(smem_raw));
  if (blockIdx.x < n_fwd)
    carry_warp<IO>(tm_x, tm_dt, tm_bc, fp, sm.fwd);
  else
    acarry_warp<IO>(tm_z, tm_dt, tm_dy, tm_bc, bp, sm.adj);
}

// ---------------------------------------------------------------- finishing
// dx of every chunk's last three tokens (chunks 0..n_chunks-2): the partial
// from the chunk itself plus the conv terms of the next chunk's first three
// tokens.  One thread per (batch row, boundary, channel).
template <typename IO>
__global__ void __launch_bounds__(256) bwd_edges_kernel(const __grid_constant__ BwdParams p) {
  const int D = p.d_inner;
  const long n = (long)p.batch * (p.n_chunks - 1) * D;
  for (long id = (long)blockIdx.x * blockDim.x + threadIdx.x; id < n; id += (long)gridDim.x * blockDim.x) {
    const int c = (int)(id % D);
    const int j = (int)((id / D) % (p.n_chunks - 1));
    const int b = (int)(id / ((long)D * (p.n_chunks - 1)));
    const int t_end = (j + 1) * p.chunk_tiles * kT;
    const float4 w = __ldg(reinterpret_cast<const float4*>(p.conv_w + (size_t)c * 4));
    const float* e = p.edge_dx + ((size_t)b * p.n_chunks + j) * 3 * D + c;
    const float* dn = p.edge_dpre + ((size_t)b * p.n_chunks + j + 1) * 3 * D + c;
    const float q0 = dn[0], q1 = dn[D], q2 = dn[2 * (size_t)D];  // d pre at t_end, t_end+1, t_end+2
    const float v0 = __fmaf_rn(w.x, q0, e[0]);
    const float v1 = __fmaf_rn(w.x, q1, __fmaf_rn(w.y, q0, e[D]));
    const float v2 = __fmaf_rn(w.x, q2, __fmaf_rn(w.y, q1, __fmaf_rn(w.z, q0, e[2 * (size_t)D])));
    IO* dx = reinterpret_cast<IO*>(p.dx) + ((size_t)b * p.seqlen + t_end - 3) * D + c;
    dx[0] = from_f32<IO>(v0);
    dx[D] = from_f32<IO>(v1);
    dx[2 * (size_t)D] = from_f32<IO>(v2);
  }
}

// dB and dC: the per-group sums added over the groups in group order.  One
// thread per (token row, 4 of the 32 values).
__global__ void __launch_bounds__(256) bwd_reduce_bc_kernel(const float* __restrict__ part, int groups, long rows,
                                                             float* __restrict__ dB, float* __restrict__ dC) {
  const long n = rows * 8;
  for (long id = (long)blockIdx.x * blockDim.x + threadIdx.x; id < n; id += (long)gridDim.x * blockDim.x) {
    const long r = id >> 3;
    const int q = (int)(id & 7);
    const float4* src = reinterpret_cast<const float4*>(part + r * 32) + q;
    const size_t step = (size_t)rows * 8;  // float4s per group
    float4 s = __ldcs(src);
    for (int g = 1; g < groups; ++g) {
      const float4 v = __ldcs(src + g * step);
      s.x = __fadd_rn(s.x, v.x);
      s.y = __fadd_rn(s.y, v.y);
      s.z = __fadd_rn(s.z, v.z);
      s.w = __fadd_rn(s.w, v.w);
    }
    float* dst = q < 4 ? dB + r * kN + 4 * q : dC + r * kN + 4 * (q - 4);
    *reinterpret_cast<float4*>(dst) = s;
  }
}

// dA_log, dD, dconv_w, dconv_b: the per-(batch row, chunk) partials added in
// that order.  One thread per (channel, value).
__global__ void __launch_bounds__(256) bwd_reduce_param_kernel(const float* __restrict__ part, int parts, int D,
                                                                float* __restrict__ dA_log, float* __restrict__ dD,
                                                                float* __restrict__ dconv_w, float* __restrict__ dconv_b) {
  const long n = (long)D * 22;
  for (long id = (long)blockIdx.x * blockDim.x + threadIdx.x; id < n; id += (long)gridDim.x * blockDim.x) {
    const int c = (int)(id / 22);
    const int e = (int)(id % 22);
    const float* src = part + (size_t)c * kParamStride + e;
    const size_t step = (size_t)D * kParamStride;
    float s = src[0];
    for (int r = 1; r < parts; ++r) s = __fadd_rn(s, src[r * step]);
    if (e < 16)
      dA_log[(size_t)c * kN + e] = s;
    else if (e == 16)
      dD[c] = s;
    else if (e < 21)
      dconv_w[(size_t)c * 4 + (e - 17)] = s;
    else if (dconv_b)
      dconv_b[c] = s;
  }
}

// I/O-dtype values to fp32 (the gradient of conv_state0 when seqlen is 0).
template <typename IO>
__global__ void __launch_bounds__(256) io_to_f32_kernel(const IO* __restrict__ src, float* __restrict__ dst, long n) {
  for (long i = (long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long)gridDim.x * blockDim.x)
    dst[i] = to_f32(src[i]);
}

}  // namespace mamba
